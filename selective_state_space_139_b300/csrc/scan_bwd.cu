// Backward of the selective scan (reverse-mode differentiation of the forward recurrence), with
// the states recomputed from checkpoints instead of stored: the training half of the
// hardware-aware scan that keeps intermediate states out of HBM ("Mamba: линейная альтернатива
// трансформеру", "Почему selectivity ломает старый трюк со свёрткой"; the ai.pinkoculture.com concept
// page, 硬件感知的实现: recomputation to save memory).  The pages give only the forward recurrence;
// the derivatives below are its chain rule.
//
// Forward (per channel): v_t = Δ_raw_t + bias, Δ_t = softplus(v_t), Ā = exp(Δ A), h_t = Ā ⊙ h_{t-1} +
// Δ_t B_t x_t, s_t = C_t·h_t + D x_t, y_t = s_t SiLU(z_t).  Backward from dy:
//   ds_t = dy_t SiLU(z_t);  dz_t = dy_t s_t SiLU'(z_t)
//   dh_t = ds_t C_t + Ā_{t+1} ⊙ dh_{t+1}
//   dC_t = Σ_channels ds_t h_t;  dB_t = Σ_channels dh_t Δ_t x_t
//   dΔ_t = Σ_n dh_{t,n} (h_{t-1,n} Ā_{t,n} A_n + B_{t,n} x_t);  dA_n = Σ_{batch, t} dh_{t,n} h_{t-1,n} Ā_{t,n} Δ_t
//   dx_t = ds_t D + Σ_n dh_{t,n} Δ_t B_{t,n};  dD = Σ ds_t x_t;  dΔ_raw_t = dΔ_t σ(v_t);  dbias = Σ dΔ_raw
//
// Two kernels.  (1) A forward pass (one thread per channel) writes the state at the start of every
// 8-step segment.  (2) The backward pass walks the segments from the last to the first: it
// recomputes the segment's 8 states from its checkpoint into shared memory (layout [step][state]
// [thread], conflict free), then runs the 8 steps backwards.  dB and dC sum over the channels of a
// batch row: per step a warp transpose-reduces its 32 values (16 of dB, 16 of dC), the four warps'
// partials are added in shared memory and one global atomic per (step, state) and CTA adds them.
// dA, dD and dbias accumulate per thread and are added once per channel.  bf16 io computes in
// float32 with the MUFU approximations of the forward; float32 io computes in double and
// accumulates its cross-channel sums in double (the same reasoning as the forward).
#include <cstring>

#include "internal.h"
#include "ssm_device.cuh"

namespace ssm {
namespace {

constexpr int kThreads = 128;   // channels per CTA
constexpr int kSeg = 8;         // steps per segment
constexpr int kN = 16;

template <typename CT>
struct Smem {
  // B and C of the segment [step][B0..15 | C0..15] (float), the recomputed states, and the dB/dC
  // partials of the four warps
  static constexpr int kBC = kSeg * 32 * 4;
  static constexpr int kH = kSeg * kN * kThreads * static_cast<int>(sizeof(CT));
  static constexpr int kRed = 4 * kSeg * 32 * static_cast<int>(sizeof(CT));
  static constexpr int kTotal = kBC + kH + kRed;
};

template <typename CT>
__device__ __forceinline__ CT sp(CT v, bool fast) {
  if constexpr (sizeof(CT) == 4) {
    return fast ? softplus_fast(v) : (v > 0.f ? v + log1pf(expf(-v)) : log1pf(expf(v)));
  } else {
    return v > 0.0 ? v + log1p(exp(-v)) : log1p(exp(v));
  }
}

template <typename CT>
__device__ __forceinline__ CT expo(CT x) {
  if constexpr (sizeof(CT) == 4) return ex2_approx(x * kLog2e);
  else return exp(x);
}

template <typename CT>
__device__ __forceinline__ CT sigm(CT x) {
  if constexpr (sizeof(CT) == 4) return rcp_approx(1.0f + ex2_approx(-x * kLog2e));
  else return 1.0 / (1.0 + exp(-x));
}

template <typename IO>
__device__ __forceinline__ float ld(const void* p, int64_t i) {
  return IoTraits<IO>::to_f32(static_cast<const IO*>(p)[i]);
}

// widen B and C of steps [t0, t0 + nk) of batch row b into the shared table (zeros past dstate / L)
template <typename IO>
__device__ __forceinline__ void load_bc(float* bc, const BwdParams& p, int b, int64_t t0, int nk) {
  for (int i = threadIdx.x; i < kSeg * 32; i += kThreads) {
    const int k = i / 32, col = i % 32, arr = col / 16, n = col % 16;
    float v = 0.0f;
    if (k < nk && n < p.N) v = ld<IO>(arr ? p.C : p.B, (static_cast<int64_t>(b) * p.N + n) * p.L + t0 + k);
    bc[i] = v;
  }
}

// (1) forward with checkpoints: ckpt[(b, d), seg, :] = state entering segment seg
template <typename IO, typename CT>
__global__ void __launch_bounds__(kThreads) bwd_ckpt_kernel(const BwdParams p) {
  __shared__ float bc[kSeg * 32];
  constexpr bool kFast = sizeof(CT) == 4;
  const int b = blockIdx.y;
  const int d = blockIdx.x * kThreads + threadIdx.x;
  const bool valid = d < p.dim;
  const int dd = valid ? d : 0;
  const int64_t row = static_cast<int64_t>(b) * p.dim + dd;
  CT A[kN], h[kN];
#pragma unroll
  for (int n = 0; n < kN; ++n) {
    A[n] = n < p.N ? p.A[static_cast<int64_t>(dd) * p.N + n] : 0.0f;
    h[n] = 0;
  }
  const CT bias = p.bias ? p.bias[dd] : 0.0f;
  const int64_t nseg = (p.L + kSeg - 1) / kSeg;
  CT* ck = static_cast<CT*>(p.ckpt) + row * nseg * kN;
  for (int64_t s = 0; s < nseg; ++s) {
    const int64_t t0 = s * kSeg;
    const int nk = static_cast<int>(p.L - t0 < kSeg ? p.L - t0 : kSeg);
    __syncthreads();
    load_bc<IO>(bc, p, b, t0, nk);
    __syncthreads();
    if (valid) {
#pragma unroll
      for (int n = 0; n < kN; ++n) ck[s * kN + n] = h[n];
    }
    for (int k = 0; k < nk; ++k) {
      const CT x = ld<IO>(p.u, row * p.L + t0 + k);
      const CT v = ld<IO>(p.delta, row * p.L + t0 + k) + bias;
      const CT dl = p.softplus ? sp<CT>(v, kFast) : v;
#pragma unroll
      for (int n = 0; n < kN; ++n) h[n] = expo<CT>(dl * A[n]) * h[n] + dl * static_cast<CT>(bc[k * 32 + n]) * x;
    }
  }
}

// warp transpose-reduce: lane i returns the sum over the warp's lanes of v[i] (32 values)
template <typename CT>
__device__ __forceinline__ CT warp_transpose_sum(CT (&v)[32]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) {
    const bool upper = (lane & w) != 0;
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const CT send = upper ? v[i] : v[i + w];
      const CT keep = upper ? v[i + w] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, w);
    }
  }
  return v[0];
}

// (2) backward over segments in reverse
template <typename IO, typename CT>
__global__ void __launch_bounds__(kThreads) bwd_kernel(const BwdParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  float* bc = reinterpret_cast<float*>(smem);
  CT* hbuf = reinterpret_cast<CT*>(smem + Smem<CT>::kBC);                  // [k][n][thread]
  CT* red = reinterpret_cast<CT*>(smem + Smem<CT>::kBC + Smem<CT>::kH);    // [warp][k][32]
  constexpr bool kFast = sizeof(CT) == 4;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.y;
  const int d = blockIdx.x * kThreads + tid;
  const bool valid = d < p.dim;
  const int dd = valid ? d : 0;
  const int64_t row = static_cast<int64_t>(b) * p.dim + dd;
  CT A[kN], dh[kN], dA[kN];
#pragma unroll
  for (int n = 0; n < kN; ++n) {
    A[n] = n < p.N ? p.A[static_cast<int64_t>(dd) * p.N + n] : 0.0f;
    dh[n] = 0;
    dA[n] = 0;
  }
  const CT bias = p.bias ? p.bias[dd] : 0.0f;
  const CT Dd = p.D ? p.D[dd] : 0.0f;
  CT dD = 0, dbias = 0;
  const int64_t nseg = (p.L + kSeg - 1) / kSeg;
  const CT* ck = static_cast<const CT*>(p.ckpt) + row * nseg * kN;
  for (int64_t s = nseg - 1; s >= 0; --s) {
    const int64_t t0 = s * kSeg;
    const int nk = static_cast<int>(p.L - t0 < kSeg ? p.L - t0 : kSeg);
    __syncthreads();   // the previous segment is done with bc and red
    load_bc<IO>(bc, p, b, t0, nk);
    __syncthreads();
    // inputs of the segment and the recomputed forward
    CT x[kSeg], dl[kSeg], vv[kSeg], sv[kSeg], zz[kSeg], dyv[kSeg];
    CT h0[kN];
#pragma unroll
    for (int n = 0; n < kN; ++n) h0[n] = ck[s * kN + n];
    {
      CT h[kN];
#pragma unroll
      for (int n = 0; n < kN; ++n) h[n] = h0[n];
#pragma unroll
      for (int k = 0; k < kSeg; ++k) {
        if (k < nk) {
          const int64_t i = row * p.L + t0 + k;
          x[k] = ld<IO>(p.u, i);
          vv[k] = ld<IO>(p.delta, i) + bias;
          dl[k] = p.softplus ? sp<CT>(vv[k], kFast) : vv[k];
          zz[k] = p.z ? ld<IO>(p.z, i) : 0.0f;
          dyv[k] = ld<IO>(p.dy, i);
          CT sacc = Dd * x[k];
#pragma unroll
          for (int n = 0; n < kN; ++n) {
            h[n] = expo<CT>(dl[k] * A[n]) * h[n] + dl[k] * static_cast<CT>(bc[k * 32 + n]) * x[k];
            hbuf[(k * kN + n) * kThreads + tid] = h[n];
            sacc += static_cast<CT>(bc[k * 32 + 16 + n]) * h[n];
          }
          sv[k] = sacc;
        } else {
          x[k] = dl[k] = vv[k] = sv[k] = zz[k] = dyv[k] = 0;
        }
      }
    }
    // backward over the segment's steps
    CT gdu[kSeg], gdd[kSeg], gdz[kSeg];
#pragma unroll
    for (int k = kSeg - 1; k >= 0; --k) {
      if (k >= nk) {
        gdu[k] = gdd[k] = gdz[k] = 0;
        continue;
      }
      CT ds = dyv[k];
      gdz[k] = 0;
      if (p.z) {
        const CT sg = sigm<CT>(zz[k]);
        ds = dyv[k] * zz[k] * sg;
        gdz[k] = dyv[k] * sv[k] * sg * (static_cast<CT>(1) + zz[k] * (static_cast<CT>(1) - sg));
      }
      if (!valid) ds = 0;
      CT dx = ds * Dd;
      dD += ds * x[k];
      CT ddl = 0;
      CT vals[32];
#pragma unroll
      for (int n = 0; n < kN; ++n) {
        const CT abar = expo<CT>(dl[k] * A[n]);
        const CT bn = bc[k * 32 + n];
        const CT cn = bc[k * 32 + 16 + n];
        dh[n] += ds * cn;
        const CT hk = hbuf[(k * kN + n) * kThreads + tid];
        const CT hprev = k > 0 ? hbuf[((k - 1) * kN + n) * kThreads + tid] : h0[n];
        vals[16 + n] = ds * hk;                 // dC contribution
        vals[n] = dh[n] * dl[k] * x[k];         // dB contribution
        ddl += dh[n] * (hprev * abar * A[n] + bn * x[k]);
        dA[n] += dh[n] * hprev * abar * dl[k];
        dx += dh[n] * dl[k] * bn;
        dh[n] *= abar;
      }
      const CT dv = p.softplus ? ddl * sigm<CT>(vv[k]) : ddl;
      gdu[k] = dx;
      gdd[k] = dv;
      dbias += dv;
      const CT tot = warp_transpose_sum<CT>(vals);
      red[(warp * kSeg + k) * 32 + lane] = tot;
    }
    // outputs of the segment
    if (valid) {
#pragma unroll
      for (int k = 0; k < kSeg; ++k) {
        if (k < nk) {
          const int64_t i = row * p.L + t0 + k;
          static_cast<IO*>(p.du)[i] = IoTraits<IO>::from_f32(static_cast<float>(gdu[k]));
          static_cast<IO*>(p.ddelta)[i] = IoTraits<IO>::from_f32(static_cast<float>(gdd[k]));
          if (p.z) static_cast<IO*>(p.dz)[i] = IoTraits<IO>::from_f32(static_cast<float>(gdz[k]));
        }
      }
    }
    __syncthreads();
    // the CTA's dB/dC partials of this segment: (k, col) pairs over the threads
    for (int i = tid; i < kSeg * 32; i += kThreads) {
      const int k = i / 32, col = i % 32, arr = col / 16, n = col % 16;
      if (k < nk && n < p.N) {
        const CT v = red[(0 * kSeg + k) * 32 + col] + red[(1 * kSeg + k) * 32 + col] +
                     red[(2 * kSeg + k) * 32 + col] + red[(3 * kSeg + k) * 32 + col];
        CT* dst = static_cast<CT*>(arr ? p.acc_dC : p.acc_dB);
        atomicAdd(dst + (static_cast<int64_t>(b) * p.N + n) * p.L + t0 + k, v);
      }
    }
  }
  if (valid) {
#pragma unroll
    for (int n = 0; n < kN; ++n)
      if (n < p.N) atomicAdd(static_cast<CT*>(p.acc_dA) + static_cast<int64_t>(d) * p.N + n, dA[n]);
    if (p.acc_dD) atomicAdd(static_cast<CT*>(p.acc_dD) + d, dD);
    if (p.acc_dbias) atomicAdd(static_cast<CT*>(p.acc_dbias) + d, dbias);
  }
}

__global__ void double_to_float_kernel(const double* __restrict__ src, float* __restrict__ dst, int64_t n) {
  const int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  if (i < n) dst[i] = static_cast<float>(src[i]);
}

template <typename IO, typename CT>
cudaError_t launch(const BwdParams& p, cudaStream_t stream) {
  const dim3 grid((p.dim + kThreads - 1) / kThreads, p.batch);
  bwd_ckpt_kernel<IO, CT><<<grid, kThreads, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  auto k = bwd_kernel<IO, CT>;
  e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Smem<CT>::kTotal);
  if (e != cudaSuccess) return e;
  k<<<grid, kThreads, Smem<CT>::kTotal, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

int bwd_segment_steps() { return kSeg; }

cudaError_t scan_bwd_launch(const BwdParams& p, cudaStream_t stream) {
  // zero the accumulators (the float outputs for bf16 io, the double workspace for float32 io)
  const size_t e = p.io_bf16 ? sizeof(float) : sizeof(double);
  const size_t nA = static_cast<size_t>(p.dim) * p.N, nBC = static_cast<size_t>(p.batch) * p.N * p.L;
  cudaError_t ce;
  if ((ce = cudaMemsetAsync(p.acc_dA, 0, nA * e, stream)) != cudaSuccess) return ce;
  if ((ce = cudaMemsetAsync(p.acc_dB, 0, nBC * e, stream)) != cudaSuccess) return ce;
  if ((ce = cudaMemsetAsync(p.acc_dC, 0, nBC * e, stream)) != cudaSuccess) return ce;
  if (p.acc_dD && (ce = cudaMemsetAsync(p.acc_dD, 0, p.dim * e, stream)) != cudaSuccess) return ce;
  if (p.acc_dbias && (ce = cudaMemsetAsync(p.acc_dbias, 0, p.dim * e, stream)) != cudaSuccess) return ce;
  ce = p.io_bf16 ? launch<__nv_bfloat16, float>(p, stream) : launch<float, double>(p, stream);
  if (ce != cudaSuccess || p.io_bf16) return ce;
  // float32 io: convert the double accumulators into the float32 outputs
  struct Pair {
    const void* src;
    float* dst;
    size_t n;
  } pairs[5] = {{p.acc_dA, p.dA, nA}, {p.acc_dB, p.dB, nBC}, {p.acc_dC, p.dC, nBC},
                {p.acc_dD, p.dD, static_cast<size_t>(p.dim)}, {p.acc_dbias, p.dbias, static_cast<size_t>(p.dim)}};
  for (const Pair& q : pairs) {
    if (!q.src || !q.dst) continue;
    double_to_float_kernel<<<static_cast<unsigned>((q.n + 255) / 256), 256, 0, stream>>>(
        static_cast<const double*>(q.src), q.dst, static_cast<int64_t>(q.n));
    if ((ce = cudaGetLastError()) != cudaSuccess) return ce;
  }
  return cudaSuccess;
}

}  // namespace ssm
