// Prefill selective scan, bf16 io fast path for sm_103a.
//
// Operator ("Mamba и State Space Models", "Selective Scan (core algorithm)"; "State Space Models:
// Mamba и альтернатива Transformer", "Mamba: Selective State Space"):
//   Δ_t = softplus(Δ_raw + bias);  h_t = exp(Δ_t A) ⊙ h_{t-1} + Δ_t B_t u_t;  y_t = (C_t·h_t + D u_t)·SiLU(z_t)
//
// Layout of the work:
//  * A CTA owns 64 consecutive channels of one batch row (a "group").  kLanes adjacent lanes share a
//    channel (2 or 4; the build default is the measured faster one), lane q holding the states
//    [q·16/kLanes, (q+1)·16/kLanes) as packed f32x2 pairs.  The per-step scalars (softplus, decay
//    exponent, Δu, gate, D skip) of each step are computed once, by the lane that owns the step,
//    and broadcast to the other lanes of the channel with shuffles; each lane reduces its part of
//    the readout and a shuffle butterfly hands every lane the totals of the steps it owns, which it
//    gates, rounds and stores.
//  * u, Δ_raw, z tiles [64 channels x 64 steps] and B, C tiles [dstate x 64 steps] arrive by TMA with
//    a 128-byte swizzle through a 3-stage mbarrier pipeline (100 KB of shared memory, two CTAs per
//    SM); B and C are widened once per tile into a float32 table read with broadcast 128-bit loads.
//  * Decays: with A[d,n] = (n+1)·A[d,0] they are powers of r = exp(Δ A[d,0]); each lane needs r and
//    its base r^(8p+1) (two MUFU ex2) and builds its eight powers with a multiply tree.  General A
//    takes one ex2 per state.
//  * Scheduling: either one CTA per (group, time chunk) ("grid"), or a balanced persistent schedule
//    ("balanced"): the (group, tile) work is cut into equal contiguous ranges, one per resident CTA.
//    A range starts inside some group g0 and ends inside some group g1 >= g0.  The CTA first runs
//    the head of g1 (tiles [0, tb)) from the initial state and publishes the state at its end; then
//    every complete group in between; last, the tail of g0, whose carried-in state was published
//    by the previous CTA when it ran that head first.  Every range is at least one group long, so
//    the wait is short.  All CTAs are co-resident (cooperative launch) and the wait is bounded.
#include <cstring>

#include "internal.h"
#include "scan_walk.cuh"
#include "ssm_device.cuh"

// Build-time variants (the defaults are the measured best).
#ifndef SSM_FAST_SHFL_DIRECT
#define SSM_FAST_SHFL_DIRECT 0      // 1: fetch each step's scalars from its owner lane (no selects)
#endif
#ifndef SSM_FAST_SOFTPLUS_LOG
#define SSM_FAST_SOFTPLUS_LOG 0     // 1: ln2 * log2(1 + e^v) everywhere below v = 15 (no series branch)
#endif
#ifndef SSM_FAST_UNROLL
#define SSM_FAST_UNROLL 1           // unroll factor of the chunk-pair loop (ping-pong variant)
#endif
#ifndef SSM_FAST_LANES
#define SSM_FAST_LANES 2            // lanes per channel: 2 or 4
#endif
#ifndef SSM_FAST_PINGPONG
#define SSM_FAST_PINGPONG 0         // 1: prepare chunk c+1 while running chunk c (two Prep buffers); 0 measured faster
#endif
#ifndef SSM_FAST_STAGES
#define SSM_FAST_STAGES 3           // TMA pipeline stages
#endif
#ifndef SSM_FAST_MINB
#define SSM_FAST_MINB 2             // resident CTAs per SM the kernel is compiled for
#endif
#ifndef SSM_FAST_DECAYS_FIRST
#define SSM_FAST_DECAYS_FIRST 0     // 1: compute the chunk's decay factors before its recurrence
#endif

namespace ssm {
namespace {

__device__ unsigned int g_fast_status = 0;

constexpr int kCh = 64;    // channels per CTA
constexpr int kLanesDefault = SSM_FAST_LANES;
constexpr int kSt = SSM_FAST_STAGES;     // TMA stages
constexpr int kRow = 128;  // bytes of one tile row = 64 bf16 steps
constexpr int kT = 64;     // steps per tile
constexpr int kN = 16;     // state width
#if SSM_FAST_PINGPONG
constexpr int kUnrollChunks = SSM_FAST_UNROLL;
#endif

struct SmemF {
  static constexpr int kTileIO = kCh * kRow;                // 8 KB
  static constexpr int kTileBC = kN * kRow;                 // 2 KB
  static constexpr int kStage = 3 * kTileIO + 2 * kTileBC;  // 28 KB
  static constexpr int kBC32 = kT * 2 * kN * 4;             // 8 KB
  static constexpr int kBars = kSt * kStage + 2 * kBC32;    // 100 KB with 3 stages
  static constexpr int kTotal = kBars + 64 + 1024;
};

enum { kMain = 0, kAgg = 1 };

struct Maps {
  CUtensorMap u, dt, z, B, C;
};

__device__ __forceinline__ float prmt_half(uint32_t word, uint32_t sel) {
  return __uint_as_float(__byte_perm(word, 0u, sel));
}

// fast softplus on a packed pair (MUFU per element)
#if SSM_FAST_SOFTPLUS_LOG
__device__ __forceinline__ float softplus_log(float v) {
  const float e = ex2_approx(v * kLog2e);
  const float r = kLn2 * lg2_approx(1.0f + e);
  return v > 15.0f ? v : r;
}
#endif
__device__ __forceinline__ f2 softplus2(f2 v) {
#if SSM_FAST_SOFTPLUS_LOG
  return f2_make(softplus_log(f2_lo(v)), softplus_log(f2_hi(v)));
#else
  return f2_make(softplus_fast(f2_lo(v)), softplus_fast(f2_hi(v)));
#endif
}

__device__ __forceinline__ f2 silu2(f2 z) {
  const f2 e = f2_make(ex2_approx(-f2_lo(z) * kLog2e), ex2_approx(-f2_hi(z) * kLog2e));
  const f2 den = f2_add(e, f2_splat(1.0f));
  return f2_mul(z, f2_make(rcp_approx(f2_lo(den)), rcp_approx(f2_hi(den))));
}

template <int kNl>
struct Lane {
  float A0L2;           // A[d,0]·log2(e)
  float kb;             // q·kNl + 1: exponent multiplier of this lane's first decay
  float AL2[kNl];       // A[d, q·kNl + i]·log2(e) (general A)
  float D, bias;
};

template <int kLanes, int kMode>
__global__ void __launch_bounds__(kCh * kLanes, SSM_FAST_MINB) scan_fast_kernel(const __grid_constant__ Maps tm,
                                                                      const ScanParams p) {
  constexpr int kThr = kCh * kLanes;
  constexpr int kNh = kN / kLanes;      // states per lane
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* bc32[2] = {reinterpret_cast<float*>(smem + kSt * SmemF::kStage),
                    reinterpret_cast<float*>(smem + kSt * SmemF::kStage + SmemF::kBC32)};
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + SmemF::kBars);

  const int tid = threadIdx.x;
  const int ch = tid / kLanes;
  const int pl = tid % kLanes;                     // lane within the channel
  const uint32_t sel = pl ? 0x3244u : 0x1044u;    // (2 lanes) byte_perm selector: this lane's bf16 half -> f32
  const int sw = ch & 7;                           // 128-byte swizzle of this channel's tile row
  const int64_t Lt = (p.L + kT - 1) / kT;
  const int gpb = (p.dim + kCh - 1) / kCh;         // groups per batch row
  const bool has_z = kMode == kMain && p.z != nullptr;

  // ---- the walk of this CTA
  Walk w;
  int64_t chunk_idx = 0;
  if (p.sched_balanced) {
    w = make_walk_balanced(blockIdx.x, p.range_tiles, static_cast<int64_t>(p.batch) * gpb * Lt, Lt);
  } else {
    // one (group, chunk): a single segment started from h0 / the carried-in state
    chunk_idx = blockIdx.y;
    w = make_walk_grid(blockIdx.x, chunk_idx, (p.chunk_len + kT - 1) / kT, Lt);
  }
  const int64_t ntiles = w.total();

  const uint32_t tx_bytes = (2 + (has_z ? 1 : 0)) * SmemF::kTileIO + (kMode == kMain ? 2 : 1) * p.N * kRow;
  if (tid == 0) {
    for (int s = 0; s < kSt; ++s) mbar_init(&full[s], 1);
    fence_mbar_init();
    prefetch_tensormap(&tm.u);
    prefetch_tensormap(&tm.dt);
    prefetch_tensormap(&tm.B);
    if (has_z) prefetch_tensormap(&tm.z);
    if (kMode == kMain) prefetch_tensormap(&tm.C);
  }
  __syncthreads();

  auto issue = [&](int64_t k) {
    int64_t g, t;
    w.at(k, g, t);
    const int b = static_cast<int>(g / gpb);
    const int row = b * p.dim + static_cast<int>(g % gpb) * kCh;
    const int x = static_cast<int>(t * kT);
    uint8_t* st = smem + (k % kSt) * SmemF::kStage;
    uint64_t* bar = &full[k % kSt];
    mbar_arrive_expect_tx(bar, tx_bytes);
    tma_load_2d(st, &tm.u, bar, x, row);
    tma_load_2d(st + SmemF::kTileIO, &tm.dt, bar, x, row);
    if (has_z) tma_load_2d(st + 2 * SmemF::kTileIO, &tm.z, bar, x, row);
    tma_load_2d(st + 3 * SmemF::kTileIO, &tm.B, bar, x, b * p.N);
    if (kMode == kMain) tma_load_2d(st + 3 * SmemF::kTileIO + SmemF::kTileBC, &tm.C, bar, x, b * p.N);
  };
  if (tid == 0)
    for (int64_t k = 0; k < kSt - 1 && k < ntiles; ++k) issue(k);

  Lane<kNh> ln;
  f2 h[kNh / 2];
  float sum_delta = 0.0f;
  bool warp_structured = true;
  int64_t cur_g = -1;
  int cur_b = 0, cur_d = 0;
  bool valid = false;
  bool ok = true;
  int64_t failed_at = -1;

  // per-channel state row offset of a group
  auto state_off = [&](int b, int d) { return (static_cast<int64_t>(b) * p.dim + d) * p.N; };

  for (int64_t k = 0; k < ntiles; ++k) {
    int64_t g, t;
    w.at(k, g, t);
    const int s = static_cast<int>(k % kSt);
    uint8_t* st = smem + s * SmemF::kStage;

    // ---- segment start: load the channel constants and the initial state
    if (g != cur_g || (k == w.n_head + w.n_full && w.n_tail > 0)) {
      cur_g = g;
      cur_b = static_cast<int>(g / gpb);
      cur_d = static_cast<int>(g % gpb) * kCh + ch;
      valid = cur_d < p.dim;
      const int64_t arow = static_cast<int64_t>(valid ? cur_d : 0) * p.N;
      const float a0 = valid ? p.A[arow] : 0.0f;
      ln.A0L2 = a0 * kLog2e;
      ln.kb = static_cast<float>(kNh * pl + 1);
      bool st_ok = true;
#pragma unroll
      for (int i = 0; i < kNh; ++i) {
        const int n = kNh * pl + i;
        const float an = (valid && n < p.N) ? p.A[arow + n] : 0.0f;
        ln.AL2[i] = an * kLog2e;
        if (n < p.N && an != static_cast<float>(n + 1) * a0) st_ok = false;
      }
      ln.D = (valid && p.D) ? p.D[cur_d] : 0.0f;
      ln.bias = (valid && p.bias) ? p.bias[cur_d] : 0.0f;
      warp_structured = __all_sync(0xffffffffu, st_ok) != 0;
      sum_delta = 0.0f;
      // initial state
      float init[kNh];
#pragma unroll
      for (int i = 0; i < kNh; ++i) init[i] = 0.0f;
      const bool is_tail = (k == w.n_head + w.n_full) && w.n_tail > 0;
      if (is_tail && p.sched_balanced) {
        // carried in from the previous CTA, which ran the head of this group first
        __shared__ int carry_ok;
        if (tid == 0) {
          const unsigned* flag = p.flags + (blockIdx.x - 1);
          const uint64_t t0 = globaltimer_ns();
          int got = 0;
          while (true) {
            unsigned v;
            asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
            if (v != 0u) { got = 1; break; }
            if (globaltimer_ns() - t0 > (p.carry_wait_ns ? p.carry_wait_ns : 2000000000ull)) break;
            __nanosleep(200);
          }
          if (!got) atomicOr(&g_fast_status, kStatusTimeout);
          carry_ok = got;
        }
        __syncthreads();
        if (carry_ok) {
          const float* src = p.carry + (static_cast<int64_t>(blockIdx.x) - 1) * kCh * kN + ch * kN + kNh * pl;
#pragma unroll
          for (int i = 0; i < kNh; ++i) init[i] = __ldcg(src + i);
        }
      } else if (is_tail && p.h_in != nullptr) {
        // chunked grid schedule: the carried-in state of this chunk
        const float* src = static_cast<const float*>(p.h_in) + chunk_idx * p.h_in_chunk_stride +
                           state_off(cur_b, valid ? cur_d : 0);
#pragma unroll
        for (int i = 0; i < kNh; ++i)
          if (valid && kNh * pl + i < p.N) init[i] = src[kNh * pl + i];
      } else if (p.h0 != nullptr && t == 0) {
        const float* src = p.h0 + state_off(cur_b, valid ? cur_d : 0);
#pragma unroll
        for (int i = 0; i < kNh; ++i)
          if (valid && kNh * pl + i < p.N) init[i] = src[kNh * pl + i];
      }
#pragma unroll
      for (int i = 0; i < kNh / 2; ++i) h[i] = f2_make(init[2 * i], init[2 * i + 1]);
    }

    // ---- this tile's data
    ok = mbar_wait_bounded(&full[s], static_cast<uint32_t>((k / kSt) & 1), &g_fast_status);
    {
      // widen B and C into the float32 table [t][B0..15 | C0..15]; rows n >= dstate are zero
      float* tab = bc32[k & 1];
      const uint32_t tB = smem_u32(st + 3 * SmemF::kTileIO);
#pragma unroll
      for (int rep = 0; rep < 256 / kThr; ++rep) {
        const int job = tid + rep * kThr;
        const int arr = job >> 7;
        const int n = job & 15;
        const int c = (job >> 4) & 7;
        if (arr == 1 && kMode != kMain) continue;
        float vals[8];
        if (n < p.N) {
          unpack_chunk(lds128(tB + arr * SmemF::kTileBC + n * kRow + ((c ^ (n & 7)) << 4)), vals, __nv_bfloat16());
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j) vals[j] = 0.0f;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) tab[(c * 8 + j) * 32 + arr * 16 + n] = vals[j];
      }
    }
    ok = __syncthreads_and(ok) != 0;
    if (!ok) {
      failed_at = k;
      break;
    }
    if (tid == 0 && k + kSt - 1 < ntiles) issue(k + kSt - 1);

    const int64_t t0 = t * kT;
    const int nch = static_cast<int>(((p.L - t0 < kT) ? (p.L - t0) : kT) / 8);
    const uint32_t urow = smem_u32(st) + ch * kRow;
    const uint32_t bct = smem_u32(bc32[k & 1]) + pl * kNh * 4;
    __nv_bfloat16* yrow = (kMode == kMain && valid)
                              ? static_cast<__nv_bfloat16*>(p.y) + (static_cast<int64_t>(cur_b) * p.dim + cur_d) * p.L
                              : nullptr;

    // Per chunk of 8 steps: "prep" reads the inputs, computes the scalars of the steps this lane owns
    // and broadcasts them to the channel's lanes; "run" does the recurrence, the readout, the
    // reduction over the channel's lanes and the store.  By default they run one after the other
    // (168 registers); the ping-pong variant prepares chunk c+1 while it runs chunk c (two Prep
    // buffers, 234 registers) and measured slower.
    struct Prep {
      float qs[8], ws[8], dls[8];
      float g[8 / kLanes], du[8 / kLanes];   // SiLU(z) and D·u of this lane's own steps
    };

    auto prep = [&](auto structured_tag, int c, Prep& P) {
      constexpr bool kS = decltype(structured_tag)::value;
      const uint32_t off = (c ^ sw) << 4;
      if constexpr (kLanes == 2) {
        // own steps 2i + pl: the pl half of each 32-bit word of the 16-byte chunk
        const uint4 uw = lds128(urow + off);
        const uint4 dw = lds128(urow + SmemF::kTileIO + off);
        const f2 u01 = f2_make(prmt_half(uw.x, sel), prmt_half(uw.y, sel));
        const f2 u23 = f2_make(prmt_half(uw.z, sel), prmt_half(uw.w, sel));
        const f2 bias2 = f2_splat(ln.bias);
        f2 d01 = f2_add(f2_make(prmt_half(dw.x, sel), prmt_half(dw.y, sel)), bias2);
        f2 d23 = f2_add(f2_make(prmt_half(dw.z, sel), prmt_half(dw.w, sel)), bias2);
        if (p.softplus) {
          d01 = softplus2(d01);
          d23 = softplus2(d23);
        }
        if (kMode == kAgg) sum_delta += (f2_lo(d01) + f2_hi(d01)) + (f2_lo(d23) + f2_hi(d23));
        const f2 a0 = f2_splat(ln.A0L2);
        const f2 q01 = f2_mul(d01, a0), q23 = f2_mul(d23, a0);     // log2 of the step's base decay
        const f2 w01 = f2_mul(d01, u01), w23 = f2_mul(d23, u23);   // Δ·u
        const float qo[4] = {f2_lo(q01), f2_hi(q01), f2_lo(q23), f2_hi(q23)};
        const float wo[4] = {f2_lo(w01), f2_hi(w01), f2_lo(w23), f2_hi(w23)};
        const float dlo[4] = {f2_lo(d01), f2_hi(d01), f2_lo(d23), f2_hi(d23)};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float qx = __shfl_xor_sync(0xffffffffu, qo[i], 1);
          const float wx = __shfl_xor_sync(0xffffffffu, wo[i], 1);
          P.qs[2 * i] = pl ? qx : qo[i];
          P.qs[2 * i + 1] = pl ? qo[i] : qx;
          P.ws[2 * i] = pl ? wx : wo[i];
          P.ws[2 * i + 1] = pl ? wo[i] : wx;
          if (!kS) {
            const float dx = __shfl_xor_sync(0xffffffffu, dlo[i], 1);
            P.dls[2 * i] = pl ? dx : dlo[i];
            P.dls[2 * i + 1] = pl ? dlo[i] : dx;
          }
        }
        if (kMode == kMain) {
          f2 g01 = f2_splat(1.0f), g23 = f2_splat(1.0f);
          if (has_z) {
            const uint4 zw = lds128(urow + 2 * SmemF::kTileIO + off);
            g01 = silu2(f2_make(prmt_half(zw.x, sel), prmt_half(zw.y, sel)));
            g23 = silu2(f2_make(prmt_half(zw.z, sel), prmt_half(zw.w, sel)));
          }
          const f2 dd = f2_splat(ln.D);
          const f2 du01 = f2_mul(dd, u01), du23 = f2_mul(dd, u23);
          P.g[0] = f2_lo(g01); P.g[1] = f2_hi(g01); P.g[2] = f2_lo(g23); P.g[3] = f2_hi(g23);
          P.du[0] = f2_lo(du01); P.du[1] = f2_hi(du01); P.du[2] = f2_lo(du23); P.du[3] = f2_hi(du23);
        }
      } else {
        // own steps 2·pl and 2·pl + 1: the 32-bit word pl of the 16-byte chunk
        const uint32_t woff = off + 4 * pl;
        const uint32_t uw = lds32(urow + woff);
        const uint32_t dw = lds32(urow + SmemF::kTileIO + woff);
        const f2 u2 = f2_make(bf16lo_to_f32(uw), bf16hi_to_f32(uw));
        f2 d2 = f2_add(f2_make(bf16lo_to_f32(dw), bf16hi_to_f32(dw)), f2_splat(ln.bias));
        if (p.softplus) d2 = softplus2(d2);
        if (kMode == kAgg) sum_delta += f2_lo(d2) + f2_hi(d2);
        const f2 q2 = f2_mul(d2, f2_splat(ln.A0L2));
        const f2 w2 = f2_mul(d2, u2);
        const int quad0 = (threadIdx.x & 31) & ~3;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int src = quad0 | (j >> 1);
          P.qs[j] = __shfl_sync(0xffffffffu, (j & 1) ? f2_hi(q2) : f2_lo(q2), src);
          P.ws[j] = __shfl_sync(0xffffffffu, (j & 1) ? f2_hi(w2) : f2_lo(w2), src);
          if (!kS) P.dls[j] = __shfl_sync(0xffffffffu, (j & 1) ? f2_hi(d2) : f2_lo(d2), src);
        }
        if (kMode == kMain) {
          f2 g2 = f2_splat(1.0f);
          if (has_z) {
            const uint32_t zw = lds32(urow + 2 * SmemF::kTileIO + woff);
            g2 = silu2(f2_make(bf16lo_to_f32(zw), bf16hi_to_f32(zw)));
          }
          const f2 du2 = f2_mul(f2_splat(ln.D), u2);
          P.g[0] = f2_lo(g2); P.g[1] = f2_hi(g2);
          P.du[0] = f2_lo(du2); P.du[1] = f2_hi(du2);
        }
      }
    };

    auto run = [&](auto structured_tag, int c, const Prep& P) {
      constexpr bool kS = decltype(structured_tag)::value;
      float py[8];
#if SSM_FAST_DECAYS_FIRST
      f2 aa[8][kNh / 2];
      if (kS) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float r = ex2_approx(P.qs[j]);
          const float bse = ex2_approx(P.qs[j] * ln.kb);
          const float r2 = r * r;
          aa[j][0] = f2_make(bse, bse * r);
          aa[j][1] = f2_mul(aa[j][0], f2_splat(r2));
          if constexpr (kNh == 8) {
            const float r4 = r2 * r2;
            aa[j][2] = f2_mul(aa[j][0], f2_splat(r4));
            aa[j][3] = f2_mul(aa[j][1], f2_splat(r4));
          }
        }
      }
#endif
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        f2 a[kNh / 2];
#if SSM_FAST_DECAYS_FIRST
        if (kS) {
#pragma unroll
          for (int i = 0; i < kNh / 2; ++i) a[i] = aa[j][i];
        } else
#endif
        if (kS) {
          // powers r^(q·kNl + 1) .. r^(q·kNl + kNl) of r = exp(Δ A[d,0])
          const float r = ex2_approx(P.qs[j]);
          const float bse = ex2_approx(P.qs[j] * ln.kb);
          const float r2 = r * r;
          a[0] = f2_make(bse, bse * r);
          a[1] = f2_mul(a[0], f2_splat(r2));
          if constexpr (kNh == 8) {
            const float r4 = r2 * r2;
            a[2] = f2_mul(a[0], f2_splat(r4));
            a[3] = f2_mul(a[1], f2_splat(r4));
          }
        } else {
#pragma unroll
          for (int i = 0; i < kNh / 2; ++i)
            a[i] = f2_make(ex2_approx(P.dls[j] * ln.AL2[2 * i]), ex2_approx(P.dls[j] * ln.AL2[2 * i + 1]));
        }
        const uint32_t rowb = bct + (c * 8 + j) * 128;
        const f2 wj = f2_splat(P.ws[j]);
        f2 acc;
        if constexpr (kNh == 8) {
          const float4 b0 = lds128f(rowb), b1 = lds128f(rowb + 16);
          h[0] = f2_fma(a[0], h[0], f2_mul(wj, f2_make(b0.x, b0.y)));
          h[1] = f2_fma(a[1], h[1], f2_mul(wj, f2_make(b0.z, b0.w)));
          h[2] = f2_fma(a[2], h[2], f2_mul(wj, f2_make(b1.x, b1.y)));
          h[3] = f2_fma(a[3], h[3], f2_mul(wj, f2_make(b1.z, b1.w)));
          if (kMode == kMain) {
            const float4 c0 = lds128f(rowb + 64), c1 = lds128f(rowb + 80);
            acc = f2_mul(f2_make(c0.x, c0.y), h[0]);
            acc = f2_fma(f2_make(c0.z, c0.w), h[1], acc);
            acc = f2_fma(f2_make(c1.x, c1.y), h[2], acc);
            acc = f2_fma(f2_make(c1.z, c1.w), h[3], acc);
          }
        } else {
          const float4 b0 = lds128f(rowb);
          h[0] = f2_fma(a[0], h[0], f2_mul(wj, f2_make(b0.x, b0.y)));
          h[1] = f2_fma(a[1], h[1], f2_mul(wj, f2_make(b0.z, b0.w)));
          if (kMode == kMain) {
            const float4 c0 = lds128f(rowb + 64);
            acc = f2_mul(f2_make(c0.x, c0.y), h[0]);
            acc = f2_fma(f2_make(c0.z, c0.w), h[1], acc);
          }
        }
        if (kMode == kMain) py[j] = f2_lo(acc) + f2_hi(acc);
      }
      if (kMode != kMain) return;
      if constexpr (kLanes == 2) {
        // owner of step 2i + pl finishes it: (own half + partner half + D u) * SiLU(z)
        float yo[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float mine = pl ? py[2 * i + 1] : py[2 * i];
          const float send = pl ? py[2 * i] : py[2 * i + 1];
          const float other = __shfl_xor_sync(0xffffffffu, send, 1);
          yo[i] = (mine + other + P.du[i]) * P.g[i];
        }
        // lane 0 stores steps 0..3, lane 1 steps 4..7 of this chunk
        const float s1 = __shfl_xor_sync(0xffffffffu, pl ? yo[0] : yo[2], 1);   // lane0 gets y1, lane1 gets y4
        const float s2 = __shfl_xor_sync(0xffffffffu, pl ? yo[1] : yo[3], 1);   // lane0 gets y3, lane1 gets y6
        uint2 out;
        if (pl == 0) {
          out.x = pack_bf16x2(yo[0], s1);
          out.y = pack_bf16x2(yo[1], s2);
        } else {
          out.x = pack_bf16x2(s1, yo[2]);
          out.y = pack_bf16x2(s2, yo[3]);
        }
        if (valid) *reinterpret_cast<uint2*>(yrow + t0 + c * 8 + pl * 4) = out;
      } else {
        // butterfly over the 4 lanes: after it, lane q holds the totals of steps 2q and 2q + 1
        const bool up2 = (pl & 2) != 0;
        float k4[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float send = up2 ? py[i] : py[4 + i];
          const float keep = up2 ? py[4 + i] : py[i];
          k4[i] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
        }
        const bool up1 = (pl & 1) != 0;
        float tot[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const float send = up1 ? k4[i] : k4[2 + i];
          const float keep = up1 ? k4[2 + i] : k4[i];
          tot[i] = keep + __shfl_xor_sync(0xffffffffu, send, 1);
        }
        const f2 y2 = f2_mul(f2_add(f2_make(tot[0], tot[1]), f2_make(P.du[0], P.du[1])), f2_make(P.g[0], P.g[1]));
        if (valid) *reinterpret_cast<uint32_t*>(yrow + t0 + c * 8 + 2 * pl) = pack_bf16x2(f2_lo(y2), f2_hi(y2));
      }
    };

    auto pipeline = [&](auto tag) {
#if SSM_FAST_PINGPONG
      Prep pa, pb;
      prep(tag, 0, pa);
#pragma unroll kUnrollChunks
      for (int c = 0; c < nch; c += 2) {
        if (c + 1 < nch) prep(tag, c + 1, pb);
        run(tag, c, pa);
        if (c + 1 < nch) {
          if (c + 2 < nch) prep(tag, c + 2, pa);
          run(tag, c + 1, pb);
        }
      }
#else
      for (int c = 0; c < nch; ++c) {
        Prep pa;
        prep(tag, c, pa);
        run(tag, c, pa);
      }
#endif
    };
    if (nch > 0) {
      if (warp_structured) pipeline(std::true_type());
      else pipeline(std::false_type());
    }

    // ---- segment end
    const bool head_end = (k == w.n_head - 1) && p.sched_balanced;
    const bool group_end = (t == Lt - 1);
    const bool chunk_end = !p.sched_balanced && (k == ntiles - 1);
    if (head_end) {
      // publish the state at the end of the head for the next CTA
      float* dst = p.carry + static_cast<int64_t>(blockIdx.x) * kCh * kN + ch * kN + kNh * pl;
#pragma unroll
      for (int i = 0; i < kNh / 2; ++i) {
        dst[2 * i] = f2_lo(h[i]);
        dst[2 * i + 1] = f2_hi(h[i]);
      }
      __syncthreads();
      if (tid == 0 && static_cast<int>(blockIdx.x) != p.test_withhold_cta) {
        __threadfence();
        asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p.flags + blockIdx.x), "r"(1u) : "memory");
      }
    } else if (kMode == kMain && group_end && valid && p.last_state) {
      float* dst = p.last_state + state_off(cur_b, cur_d);
#pragma unroll
      for (int i = 0; i < kNh / 2; ++i) {
        if (kNh * pl + 2 * i < p.N) dst[kNh * pl + 2 * i] = f2_lo(h[i]);
        if (kNh * pl + 2 * i + 1 < p.N) dst[kNh * pl + 2 * i + 1] = f2_hi(h[i]);
      }
    }
    // the pair's ΣΔ (every lane takes part in the shuffle, valid or not)
    float sd = 0.0f;
    if (kMode == kAgg && chunk_end) {
      sd = sum_delta + __shfl_xor_sync(0xffffffffu, sum_delta, 1);
      if (kLanes == 4) sd += __shfl_xor_sync(0xffffffffu, sd, 2);
    }
    if (kMode == kAgg && chunk_end && valid) {
      // aggregate of this chunk: P = exp(A ΣΔ), Q = h_end from a zero state
      const int64_t cbase = chunk_idx * p.h_in_chunk_stride + state_off(cur_b, cur_d);
      float* P = static_cast<float*>(p.agg_P);
      float* Q = static_cast<float*>(p.agg_Q);
#pragma unroll
      for (int i = 0; i < kNh; ++i) {
        const int n = kNh * pl + i;
        if (n < p.N) {
          P[cbase + n] = ex2_approx(ln.AL2[i] * sd);
          Q[cbase + n] = i & 1 ? f2_hi(h[i >> 1]) : f2_lo(h[i >> 1]);
        }
      }
    }
  }

  if (failed_at >= 0 && tid == 0) {
    // a wait gave up: wait (bounded) for this CTA's copies still in flight, then leave
    const int64_t issued = failed_at + kSt - 1 < ntiles ? failed_at + kSt - 1 : ntiles;
    for (int64_t k = failed_at; k < issued; ++k)
      (void)mbar_wait_bounded(&full[k % kSt], static_cast<uint32_t>((k / kSt) & 1), &g_fast_status, 100000000ull);
  }
}

}  // namespace

int fast_channels_per_cta() { return kCh; }

int fast_resident_ctas() {
  static int cached[64] = {0};
  int occ = 0, dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return 0; }
  if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) { cudaGetLastError(); return 0; }
  auto kern = scan_fast_kernel<kLanesDefault, kMain>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SmemF::kTotal) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kCh * kLanesDefault, SmemF::kTotal) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  if (dev >= 0 && dev < 64) cached[dev] = occ * sms;
  return occ * sms;
}

cudaError_t fast_status_read_and_clear(unsigned int* out) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_fast_status, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_fast_status, &zero, sizeof(unsigned int));
}

cudaError_t scan_fast_launch(const ScanParams& p, int nchunks, int balanced_ctas, cudaStream_t stream, char* err,
                             size_t errlen) {
  constexpr int kL = kLanesDefault;
  constexpr int kThreads = kCh * kL;
  Maps tm;
  memset(&tm, 0, sizeof(tm));
  const uint64_t rows = static_cast<uint64_t>(p.batch) * p.dim;
  struct M {
    CUtensorMap* map;
    const void* ptr;
    uint64_t rows;
    uint32_t box_rows;
  } maps[5] = {{&tm.u, p.u, rows, kCh},
               {&tm.dt, p.delta, rows, kCh},
               {&tm.z, p.z ? p.z : p.u, rows, kCh},
               {&tm.B, p.B, static_cast<uint64_t>(p.batch) * p.N, static_cast<uint32_t>(p.N)},
               {&tm.C, p.C, static_cast<uint64_t>(p.batch) * p.N, static_cast<uint32_t>(p.N)}};
  for (auto& m : maps) {
    if (!encode_tensor_map_2d(m.map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<void*>(m.ptr),
                              static_cast<uint64_t>(p.L), m.rows, static_cast<uint64_t>(p.L) * 2, kT, m.box_rows, err,
                              errlen))
      return cudaErrorInvalidValue;
  }
  const int gpb = (p.dim + kCh - 1) / kCh;
  const unsigned groups = static_cast<unsigned>(p.batch) * gpb;
  auto kmain = scan_fast_kernel<kL, kMain>;
  auto kagg = scan_fast_kernel<kL, kAgg>;
  cudaError_t e;
  e = cudaFuncSetAttribute(kmain, cudaFuncAttributeMaxDynamicSharedMemorySize, SmemF::kTotal);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kagg, cudaFuncAttributeMaxDynamicSharedMemorySize, SmemF::kTotal);
  if (e != cudaSuccess) return e;
  if (balanced_ctas > 0) {
    e = cudaMemsetAsync(p.flags, 0, sizeof(unsigned) * balanced_ctas, stream);
    if (e != cudaSuccess) return e;
    void* args[] = {const_cast<Maps*>(&tm), const_cast<ScanParams*>(&p)};
    return cudaLaunchCooperativeKernel(reinterpret_cast<void*>(kmain), dim3(balanced_ctas), dim3(kThreads), args,
                                       SmemF::kTotal, stream);
  }
  if (nchunks > 1) {
    ScanParams pa = p;
    pa.h_in = nullptr;
    pa.h0 = nullptr;
    kagg<<<dim3(groups, nchunks - 1), kThreads, SmemF::kTotal, stream>>>(tm, pa);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = carry_launch_f32(p, nchunks, stream);
    if (e != cudaSuccess) return e;
  }
  kmain<<<dim3(groups, nchunks), kThreads, SmemF::kTotal, stream>>>(tm, p);
  return cudaGetLastError();
}

}  // namespace ssm
