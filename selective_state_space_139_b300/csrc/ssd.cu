// Mamba-2 state space duality (SSD) forward, chunked block form on the tensor cores
// ("Mamba и State Space Models", "Mamba-2: State Space Duality (SSD)": a scalar A per head,
// d_state 128, the SSM as a product with a semi-separable matrix; "Модуль 8. Альтернативы
// Transformer", §7: M_ij = C_i·B_j Π_{r=j+1..i} a_r, computed inside a chunk as a masked matrix
// product with only the state passed between chunks; §14: state [batch, nheads, headdim, d_state]
// and the input term Δ·B·x).
//
// Per batch b and head h (group g), with a_t = exp(Δ_t A_h), cum_i = Σ_{r≤i} Δ_r A_h inside a chunk
// of Q = 64 steps, and H the (headdim 64 x d_state 128) state entering the chunk:
//   y_i = Σ_{j≤i} (C_i·B_j) e^{cum_i − cum_j} Δ_j x_j  +  e^{cum_i} C_i·H  +  D_h x_i
//   H  <- e^{cum_end} H + Σ_j e^{cum_end − cum_j} Δ_j x_j B_j^T
// One CTA (4 warps) per (b, h) walks the chunks in order; the fp32 state lives in the MMA
// accumulators of the warps (warp w owns state rows p = 16w..16w+15).  Per chunk:
//   G = C B^T (exact bf16 products, fp32 sums), kept in registers: the m16n8 accumulator layout of G
//       is the m16k16 A-operand layout of M = G ∘ e^{cum_i − cum_j} Δ_j (causal), so M never touches
//       shared memory;
//   Y = (e^{cum_i} C H^T) + M X;  H = e^{cum_end} H + (w ∘ X)^T B.
// The tensor-core operands x, B, C are exact bf16 inputs.  The computed operands (M, H, w ∘ x) are
// fp32 values split into bf16 hi + lo (about 16 significant bits), one MMA each, so that the result
// keeps float32-level accuracy rather than bf16's 8 bits.  mma.sync m16n8k16 bf16 with fp32 accumulate;
// fragments loaded with ldmatrix from padded (bank-conflict free) shared tiles filled by cp.async.
#include "internal.h"
#include "ssm_device.cuh"

#ifndef SSM_SSD_TCGEN05
#define SSM_SSD_TCGEN05 1   // 1: the tcgen05 kernel (ssd_tc.cu); 0: this mma.sync kernel
#endif

namespace ssm {
namespace {

constexpr int kQ = 64;         // chunk length
constexpr int kHd = 64;        // head dim
constexpr int kNs = 128;       // d_state
constexpr int kThreads = 128;  // 4 warps
constexpr int kXPitch = kHd * 2 + 16;   // bytes per row of x / (w ∘ x) tiles
constexpr int kBPitch = kNs * 2 + 16;   // bytes per row of B, C and H tiles

struct SsdSmem {
  static constexpr int kX = 0;                          // x chunk [j][p] bf16
  static constexpr int kB = kX + kQ * kXPitch;          // B chunk [j][n] bf16
  static constexpr int kC = kB + kQ * kBPitch;          // C chunk [i][n] bf16
  static constexpr int kWh = kC + kQ * kBPitch;         // (w ∘ x) hi [j][p]
  static constexpr int kWl = kWh + kQ * kXPitch;        // (w ∘ x) lo
  static constexpr int kHh = kWl + kQ * kXPitch;        // H hi [p][n]
  static constexpr int kHl = kHh + kHd * kBPitch;       // H lo
  static constexpr int kDl = kHl + kHd * kBPitch;       // Δ_i (float)
  static constexpr int kCum = kDl + kQ * 4;             // cum_i in log2 units (float)
  static constexpr int kTot = kCum + kQ * 4 + 16;       // + the warp-0 scan total
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
// D += A B, m16n8k16, bf16 inputs, fp32 accumulate
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// 16-byte global -> shared copy; src_bytes = 0 fills zeros
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// fp32 pair -> bf16x2 hi part and the bf16x2 of the remainders (a in the low half)
__device__ __forceinline__ void split2(float a, float b, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16x2(a, b);
  lo = pack_bf16x2(a - bf16lo_to_f32(hi), b - bf16hi_to_f32(hi));
}

// Lane addresses of the four 8x8 matrices an x4 ldmatrix reads (byte offsets in a row-major tile).
// A operand (16 x 16 at rows r0, cols c0), non-transposed storage [m][k].
__device__ __forceinline__ uint32_t a_addr(uint32_t base, int pitch, int r0, int c0, int lane) {
  return base + (r0 + (lane & 7) + ((lane >> 3) & 1) * 8) * pitch + (c0 + (lane >> 4) * 8) * 2;
}
// A operand stored transposed [k][m] (tile: A rows m0.., A cols k0..)
__device__ __forceinline__ uint32_t a_addr_t(uint32_t base, int pitch, int m0, int k0, int lane) {
  return base + (k0 + (lane & 7) + ((lane >> 4) & 1) * 8) * pitch + (m0 + ((lane >> 3) & 1) * 8) * 2;
}
// B operands of two n8 tiles (n0, n0 + 8) and one k16 step, storage [n][k] (non-transposed)
__device__ __forceinline__ uint32_t b_addr(uint32_t base, int pitch, int n0, int k0, int lane) {
  return base + (n0 + (lane & 7) + ((lane >> 4) & 1) * 8) * pitch + (k0 + ((lane >> 3) & 1) * 8) * 2;
}
// B operands of two n8 tiles and one k16 step, storage [k][n] (transposed load)
__device__ __forceinline__ uint32_t b_addr_t(uint32_t base, int pitch, int n0, int k0, int lane) {
  return base + (k0 + (lane & 7) + ((lane >> 3) & 1) * 8) * pitch + (n0 + ((lane >> 4) & 1) * 8) * 2;
}

__global__ void __launch_bounds__(kThreads, 2) ssd_chunk_kernel(const SsdParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sb = smem_u32(smem);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t4 = lane & 3;
  const int h = blockIdx.x, b = blockIdx.y;
  const int grp = h / (p.nheads / p.ngroups);
  float* s_dl = reinterpret_cast<float*>(smem + SsdSmem::kDl);
  float* s_cum = reinterpret_cast<float*>(smem + SsdSmem::kCum);
  float* s_tot = reinterpret_cast<float*>(smem + SsdSmem::kCum + kQ * 4);
  const float A2 = p.A[h] * kLog2e;
  const float bias = p.dt_bias ? p.dt_bias[h] : 0.0f;
  const float Dh = p.D ? p.D[h] : 0.0f;
  const int64_t L = p.L;
  const __nv_bfloat16* xg = static_cast<const __nv_bfloat16*>(p.x);
  const __nv_bfloat16* dtg = static_cast<const __nv_bfloat16*>(p.dt);
  const __nv_bfloat16* Bg = static_cast<const __nv_bfloat16*>(p.B);
  const __nv_bfloat16* Cg = static_cast<const __nv_bfloat16*>(p.C);
  __nv_bfloat16* yg = static_cast<__nv_bfloat16*>(p.y);

  // the state: warp w owns rows p = 16w..16w+15 over 16 n8 tiles
  float hacc[16][4];
  bool have_state = p.h0 != nullptr;
  {
    const float* h0 = p.h0 ? p.h0 + (static_cast<int64_t>(b) * p.nheads + h) * kHd * kNs : nullptr;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      const int n = nt * 8 + 2 * t4;
      const int r0 = warp * 16 + g, r1 = r0 + 8;
      hacc[nt][0] = h0 ? h0[r0 * kNs + n] : 0.0f;
      hacc[nt][1] = h0 ? h0[r0 * kNs + n + 1] : 0.0f;
      hacc[nt][2] = h0 ? h0[r1 * kNs + n] : 0.0f;
      hacc[nt][3] = h0 ? h0[r1 * kNs + n + 1] : 0.0f;
      uint32_t hi, lo;
      split2(hacc[nt][0], hacc[nt][1], hi, lo);
      *reinterpret_cast<uint32_t*>(smem + SsdSmem::kHh + r0 * kBPitch + n * 2) = hi;
      *reinterpret_cast<uint32_t*>(smem + SsdSmem::kHl + r0 * kBPitch + n * 2) = lo;
      split2(hacc[nt][2], hacc[nt][3], hi, lo);
      *reinterpret_cast<uint32_t*>(smem + SsdSmem::kHh + r1 * kBPitch + n * 2) = hi;
      *reinterpret_cast<uint32_t*>(smem + SsdSmem::kHl + r1 * kBPitch + n * 2) = lo;
    }
  }

  // chunk loads: x (64 rows x 128 B) and C, B (64 rows x 256 B); rows past L are zero-filled.  x and C
  // of the next chunk are issued while the state update of the current one runs (they are free by
  // then); B is used by that update and is loaded at the top of the next iteration.
  auto load_x = [&](int64_t t0) {
    for (int i = tid; i < kQ * 8; i += kThreads) {
      const int j = i >> 3, q = i & 7;
      const bool ok = t0 + j < L;
      const __nv_bfloat16* src = xg + ((static_cast<int64_t>(b) * L + (ok ? t0 + j : 0)) * p.nheads + h) * kHd + q * 8;
      cp_async16(sb + SsdSmem::kX + j * kXPitch + q * 16, src, ok ? 16 : 0);
    }
  };
  auto load_bc = [&](int64_t t0, int off) {
    const __nv_bfloat16* base = off == SsdSmem::kB ? Bg : Cg;
    for (int i = tid; i < kQ * 16; i += kThreads) {
      const int j = i >> 4, q = i & 15;
      const bool ok = t0 + j < L;
      const int64_t row = (static_cast<int64_t>(b) * L + (ok ? t0 + j : 0)) * p.ngroups + grp;
      cp_async16(sb + off + j * kBPitch + q * 16, base + row * kNs + q * 8, ok ? 16 : 0);
    }
  };
  const int nchunks = static_cast<int>((L + kQ - 1) / kQ);
  load_x(0);
  load_bc(0, SsdSmem::kC);
  for (int c = 0; c < nchunks; ++c) {
    const int64_t t0 = static_cast<int64_t>(c) * kQ;
    load_bc(t0, SsdSmem::kB);
    // ---- Δ and the inclusive prefix of Δ·A (log2 units) over the chunk: warps 0 and 1
    if (tid < kQ) {
      const int64_t t = t0 + tid;
      float dl = 0.0f;
      if (t < L) {
        const float v = __bfloat162float(dtg[(static_cast<int64_t>(b) * L + t) * p.nheads + h]) + bias;
        dl = p.softplus ? softplus_fast(v) : v;
      }
      float s = dl * A2;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float u = __shfl_up_sync(0xffffffffu, s, o);
        if (lane >= o) s += u;
      }
      s_dl[tid] = dl;
      s_cum[tid] = s;
      if (tid == 31) s_tot[0] = s;
    }
    cp_async_wait_all();
    __syncthreads();
    if (tid >= 32 && tid < kQ) s_cum[tid] += s_tot[0];
    __syncthreads();

    // ---- outputs of the chunk: warp w computes rows i = 16w..16w+15
    const int ri0 = warp * 16 + g, ri1 = ri0 + 8;
    const float cum_r0 = s_cum[ri0], cum_r1 = s_cum[ri1];
    float acc[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.0f;
    float gacc[8][4];
#pragma unroll
    for (int jt = 0; jt < 8; ++jt) gacc[jt][0] = gacc[jt][1] = gacc[jt][2] = gacc[jt][3] = 0.0f;
#pragma unroll
    for (int ks = 0; ks < kNs / 16; ++ks) {
      uint32_t a[4];
      ldsm_x4(a_addr(sb + SsdSmem::kC, kBPitch, warp * 16, ks * 16, lane), a[0], a[1], a[2], a[3]);
      // e^{cum_i} C H^T (the state entering the chunk), hi and lo parts of H
      if (have_state) {
        // all fragments first, then the MMAs cycling over the eight accumulators (no back-to-back
        // dependent MMAs)
        uint32_t bh[4][4], bl[4][4];
#pragma unroll
        for (int pt = 0; pt < 4; ++pt) {
          ldsm_x4(b_addr(sb + SsdSmem::kHh, kBPitch, pt * 16, ks * 16, lane), bh[pt][0], bh[pt][1], bh[pt][2], bh[pt][3]);
          ldsm_x4(b_addr(sb + SsdSmem::kHl, kBPitch, pt * 16, ks * 16, lane), bl[pt][0], bl[pt][1], bl[pt][2], bl[pt][3]);
        }
#pragma unroll
        for (int pt = 0; pt < 4; ++pt) {
          mma16816(acc[2 * pt], a, bh[pt][0], bh[pt][1]);
          mma16816(acc[2 * pt + 1], a, bh[pt][2], bh[pt][3]);
        }
#pragma unroll
        for (int pt = 0; pt < 4; ++pt) {
          mma16816(acc[2 * pt], a, bl[pt][0], bl[pt][1]);
          mma16816(acc[2 * pt + 1], a, bl[pt][2], bl[pt][3]);
        }
      }
      // G = C B^T for the causal j tiles 0 .. 2w+1
#pragma unroll
      for (int jp = 0; jp < 4; ++jp) {
        if (jp <= warp) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(b_addr(sb + SsdSmem::kB, kBPitch, jp * 16, ks * 16, lane), b0, b1, b2, b3);
          mma16816(gacc[2 * jp], a, b0, b1);
          mma16816(gacc[2 * jp + 1], a, b2, b3);
        }
      }
    }
    {
      const float e0 = ex2_approx(cum_r0), e1 = ex2_approx(cum_r1);
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        acc[nt][0] *= e0;
        acc[nt][1] *= e0;
        acc[nt][2] *= e1;
        acc[nt][3] *= e1;
      }
    }
    // M = G ∘ e^{cum_i − cum_j} Δ_j (j ≤ i) as A fragments, times X
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      if (s <= warp) {
        float m[8];   // (r0, c), (r0, c+1), (r1, c), (r1, c+1), then the same at c + 8
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int jt = 2 * s + half;
          const int c0 = jt * 8 + 2 * t4;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int r = e < 2 ? ri0 : ri1;
            const int cc = c0 + (e & 1);
            const float cum_r = e < 2 ? cum_r0 : cum_r1;
            float v = 0.0f;
            if (cc <= r) v = gacc[jt][e] * ex2_approx(cum_r - s_cum[cc]) * s_dl[cc];
            m[half * 4 + e] = v;
          }
        }
        uint32_t ah[4], al[4];
        split2(m[0], m[1], ah[0], al[0]);
        split2(m[2], m[3], ah[1], al[1]);
        split2(m[4], m[5], ah[2], al[2]);
        split2(m[6], m[7], ah[3], al[3]);
        uint32_t bx[4][4];
#pragma unroll
        for (int pt = 0; pt < 4; ++pt)
          ldsm_x4_t(b_addr_t(sb + SsdSmem::kX, kXPitch, pt * 16, s * 16, lane), bx[pt][0], bx[pt][1], bx[pt][2], bx[pt][3]);
#pragma unroll
        for (int pt = 0; pt < 4; ++pt) {
          mma16816(acc[2 * pt], ah, bx[pt][0], bx[pt][1]);
          mma16816(acc[2 * pt + 1], ah, bx[pt][2], bx[pt][3]);
        }
#pragma unroll
        for (int pt = 0; pt < 4; ++pt) {
          mma16816(acc[2 * pt], al, bx[pt][0], bx[pt][1]);
          mma16816(acc[2 * pt + 1], al, bx[pt][2], bx[pt][3]);
        }
      }
    }
    // y = acc + D x, rounded to bf16
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const int pc = nt * 8 + 2 * t4;
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int r = hr ? ri1 : ri0;
        if (t0 + r < L) {
          const uint32_t xw = *reinterpret_cast<const uint32_t*>(smem + SsdSmem::kX + r * kXPitch + pc * 2);
          const float y0 = acc[nt][2 * hr] + Dh * bf16lo_to_f32(xw);
          const float y1 = acc[nt][2 * hr + 1] + Dh * bf16hi_to_f32(xw);
          *reinterpret_cast<uint32_t*>(yg + ((static_cast<int64_t>(b) * L + t0 + r) * p.nheads + h) * kHd + pc) =
              pack_bf16x2(y0, y1);
        }
      }
    }

    // ---- the state at the chunk end
    const float cum_end = s_cum[kQ - 1];
    {
      // (w ∘ x)[j][p] with w_j = e^{cum_end − cum_j} Δ_j, split into hi and lo: thread -> row j, 32 p
      const int j = tid >> 1, p0 = (tid & 1) * 32;
      const float wj = ex2_approx(cum_end - s_cum[j]) * s_dl[j];
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const uint32_t xw = *reinterpret_cast<const uint32_t*>(smem + SsdSmem::kX + j * kXPitch + (p0 + 2 * q) * 2);
        uint32_t hi, lo;
        split2(wj * bf16lo_to_f32(xw), wj * bf16hi_to_f32(xw), hi, lo);
        *reinterpret_cast<uint32_t*>(smem + SsdSmem::kWh + j * kXPitch + (p0 + 2 * q) * 2) = hi;
        *reinterpret_cast<uint32_t*>(smem + SsdSmem::kWl + j * kXPitch + (p0 + 2 * q) * 2) = lo;
      }
    }
    __syncthreads();   // (w ∘ x) complete; every warp is done reading H, x and C for the outputs
    if (c + 1 < nchunks) {
      load_x(t0 + kQ);
      load_bc(t0 + kQ, SsdSmem::kC);
    }
    {
      const float eE = ex2_approx(cum_end);
#pragma unroll
      for (int nt = 0; nt < 16; ++nt) {
        hacc[nt][0] *= eE;
        hacc[nt][1] *= eE;
        hacc[nt][2] *= eE;
        hacc[nt][3] *= eE;
      }
    }
#pragma unroll
    for (int ks = 0; ks < kQ / 16; ++ks) {
      uint32_t ah[4], al[4];
      ldsm_x4_t(a_addr_t(sb + SsdSmem::kWh, kXPitch, warp * 16, ks * 16, lane), ah[0], ah[1], ah[2], ah[3]);
      ldsm_x4_t(a_addr_t(sb + SsdSmem::kWl, kXPitch, warp * 16, ks * 16, lane), al[0], al[1], al[2], al[3]);
#pragma unroll
      for (int half = 0; half < 2; ++half) {   // 4 n-tile pairs at a time: hi MMAs over 8 accumulators, then lo
        uint32_t bb[4][4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
          ldsm_x4_t(b_addr_t(sb + SsdSmem::kB, kBPitch, (half * 4 + q) * 16, ks * 16, lane), bb[q][0], bb[q][1],
                    bb[q][2], bb[q][3]);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          mma16816(hacc[2 * (half * 4 + q)], ah, bb[q][0], bb[q][1]);
          mma16816(hacc[2 * (half * 4 + q) + 1], ah, bb[q][2], bb[q][3]);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          mma16816(hacc[2 * (half * 4 + q)], al, bb[q][0], bb[q][1]);
          mma16816(hacc[2 * (half * 4 + q) + 1], al, bb[q][2], bb[q][3]);
        }
      }
    }
    // the new state as the hi/lo B operand of the next chunk
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      const int n = nt * 8 + 2 * t4;
      const int r0 = warp * 16 + g, r1 = r0 + 8;
      uint32_t hi, lo;
      split2(hacc[nt][0], hacc[nt][1], hi, lo);
      *reinterpret_cast<uint32_t*>(smem + SsdSmem::kHh + r0 * kBPitch + n * 2) = hi;
      *reinterpret_cast<uint32_t*>(smem + SsdSmem::kHl + r0 * kBPitch + n * 2) = lo;
      split2(hacc[nt][2], hacc[nt][3], hi, lo);
      *reinterpret_cast<uint32_t*>(smem + SsdSmem::kHh + r1 * kBPitch + n * 2) = hi;
      *reinterpret_cast<uint32_t*>(smem + SsdSmem::kHl + r1 * kBPitch + n * 2) = lo;
    }
    have_state = true;
    __syncthreads();   // H written; x, B, C, Δ free for the next chunk
  }
  if (p.hT) {
    float* hT = p.hT + (static_cast<int64_t>(b) * p.nheads + h) * kHd * kNs;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      const int n = nt * 8 + 2 * t4;
      const int r0 = warp * 16 + g, r1 = r0 + 8;
      *reinterpret_cast<float2*>(hT + r0 * kNs + n) = make_float2(hacc[nt][0], hacc[nt][1]);
      *reinterpret_cast<float2*>(hT + r1 * kNs + n) = make_float2(hacc[nt][2], hacc[nt][3]);
    }
  }
}

}  // namespace

int ssd_head_dim() { return kHd; }
int ssd_state_dim() { return kNs; }

cudaError_t ssd_fwd_launch(const SsdParams& p, cudaStream_t stream) {
  if (SSM_SSD_TCGEN05) return ssd_tc_launch(p, stream);
  cudaError_t e = cudaFuncSetAttribute(ssd_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SsdSmem::kTot);
  if (e != cudaSuccess) return e;
  ssd_chunk_kernel<<<dim3(p.nheads, p.batch), kThreads, SsdSmem::kTot, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace ssm
