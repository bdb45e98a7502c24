// Prefill selective scan for sm_103a.
//
// Operator ("Mamba и State Space Models", "Selective Scan (core algorithm)"; "State Space Models:
// Mamba и альтернатива Transformer", "Mamba: Selective State Space"):
//   Δ_t = softplus(Δ_raw + bias);  h_t = exp(Δ_t A) ⊙ h_{t-1} + Δ_t B_t u_t;
//   y_t = (C_t·h_t + D u_t) · SiLU(z_t)
//
// Kernel structure (one CTA = 128 consecutive channels of one batch row, one thread per channel):
//  * u, Δ_raw, z tiles [128 channels x 128 bytes of time] and B, C tiles [dstate x 128 bytes] are
//    brought into shared memory by TMA (128-byte swizzle, so that each thread reading its own row
//    is bank-conflict free) through a 3-stage mbarrier pipeline; a non-TMA variant fills the same
//    layout with plain loads for shapes TMA cannot describe (row pitch not a multiple of 16 bytes).
//  * B and C are widened once per tile to a float32 [t][B0..15, C0..15] table that every thread
//    reads with broadcast 128-bit loads.
//  * The 16 states live in registers as 8 packed f32x2 pairs; discretisation happens on the fly.
//    When A[d, n] = (n+1)·A[d, 0] (the S4D-real layout of every Mamba layer at initialisation and
//    of all workloads here) the decays are powers of r = exp(Δ A[d,0]) and cost one MUFU per step
//    instead of sixteen.
//  * Only y and the final state are written.
// Long sequences with few channels use the chunked form ("Модуль 8", §7): per-chunk affine
// aggregates (Π exp(ΔA), h_end from zero), a carry pass composing them, and a re-run of every
// chunk from its carried-in state.
#include <cstring>
#include <type_traits>

#include "internal.h"
#include "ssm_device.cuh"

namespace ssm {

namespace {

__device__ unsigned int g_device_status = 0;

constexpr int kCH = 128;        // channels (threads) per CTA
constexpr int kStages = 3;      // TMA pipeline depth
constexpr int kRowBytes = 128;  // bytes of time per tile row (the 128-byte swizzle span)
constexpr int kNmax = 16;       // register state width

enum Mode { kModeMain = 0, kModeAggregate = 1 };

// Shared memory carve-up (offsets from a 1024-byte-aligned base).
struct Smem {
  static constexpr int kTileIO = kCH * kRowBytes;          // 16 KB: u, Δ_raw or z tile
  static constexpr int kTileBC = kNmax * kRowBytes;        // 2 KB: B or C tile
  static constexpr int kStage = 3 * kTileIO + 2 * kTileBC; // 52 KB
  static constexpr int kBC32 = 64 * 2 * kNmax * 4;         // 8 KB: float32 [T][32] table (T <= 64)
  static constexpr int kBars = kStages * kStage + 2 * kBC32;
  static constexpr int kTotal = kBars + 64 + 1024;         // + barriers + alignment slack
};

template <typename IO>
struct Tile {
  static constexpr int kVec = IoTraits<IO>::kVec;          // elements per 16-byte chunk
  static constexpr int kT = kRowBytes / IoTraits<IO>::kBytes;  // steps per tile: 64 (bf16), 32 (f32)
  static constexpr int kChunks = kT / kVec;                // 8 chunks per row
};

// Per-thread view of one time step's widened B and C.
struct BC {
  f2 b[kNmax / 2];
  f2 c[kNmax / 2];
};

__device__ __forceinline__ void load_bc(uint32_t bc_row, BC& x) {
#pragma unroll
  for (int q = 0; q < kNmax / 4; ++q) {
    float4 vb = lds128f(bc_row + q * 16);
    float4 vc = lds128f(bc_row + 64 + q * 16);
    x.b[2 * q] = f2_make(vb.x, vb.y);
    x.b[2 * q + 1] = f2_make(vb.z, vb.w);
    x.c[2 * q] = f2_make(vc.x, vc.y);
    x.c[2 * q + 1] = f2_make(vc.z, vc.w);
  }
}

// Decay factors exp(Δ A[d, n]) for the 16 states, as 8 pairs.
// Structured A (A[d,n] = (n+1) A[d,0]): powers of r = exp(Δ A[d,0]) by a short multiply tree.
__device__ __forceinline__ void decays_structured(float r, f2 (&a)[kNmax / 2]) {
  const float r2 = r * r;
  const float r4 = r2 * r2;
  const float r8 = r4 * r4;
  a[0] = f2_make(r, r2);
  a[1] = f2_mul(a[0], f2_splat(r2));
  a[2] = f2_mul(a[0], f2_splat(r4));
  a[3] = f2_mul(a[1], f2_splat(r4));
#pragma unroll
  for (int i = 0; i < 4; ++i) a[4 + i] = f2_mul(a[i], f2_splat(r8));
}

// Per-channel constants.
struct Chan {
  float AL2[kNmax];   // A[d,n]·log2(e) (fast path) or A[d,n] (accurate path)
  float invA[kNmax];  // 1/A[d,n] for the ZOH input term (0 where |A| < 2^-60)
  float D, bias;
  bool structured;
};

// One time step for one channel.  Returns y_t (before the final dtype rounding) and updates h.
// kFast: MUFU approximations (bf16 io); otherwise the CUDA math library (float32 io).
template <bool kFast, bool kStructured, int kDisc, int kMode>
__device__ __forceinline__ float scan_step(const Chan& ch, float u, float draw, float z, const BC& bc,
                                           f2 (&h)[kNmax / 2], bool softplus, bool has_z, float& sum_delta) {
  const float v = draw + ch.bias;
  float dl;
  if (softplus) dl = kFast ? softplus_fast(v) : softplus_accurate(v);
  else dl = v;
  if (kMode == kModeAggregate) sum_delta += dl;
  f2 a[kNmax / 2];
  if (kStructured) {
    const float r = kFast ? ex2_approx(dl * ch.AL2[0]) : expf(dl * ch.AL2[0]);
    decays_structured(r, a);
  } else {
#pragma unroll
    for (int i = 0; i < kNmax / 2; ++i) {
      if (kFast) a[i] = f2_make(ex2_approx(dl * ch.AL2[2 * i]), ex2_approx(dl * ch.AL2[2 * i + 1]));
      else a[i] = f2_make(expf(dl * ch.AL2[2 * i]), expf(dl * ch.AL2[2 * i + 1]));
    }
  }
  if (kDisc == 0) {
    const f2 w = f2_splat(dl * u);
#pragma unroll
    for (int i = 0; i < kNmax / 2; ++i) h[i] = f2_fma(a[i], h[i], f2_mul(w, bc.b[i]));
  } else {
    // exact zero-order hold: bbar = (exp(ΔA) - 1)/A · B, with the A -> 0 limit Δ·B
#pragma unroll
    for (int i = 0; i < kNmax / 2; ++i) {
      float e[2];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int n = 2 * i + k;
        const float x = kFast ? dl * ch.AL2[n] * kLn2 : dl * ch.AL2[n];   // Δ·A[d,n]
        float em1;
        if (kFast) {
          const float ak = k == 0 ? f2_lo(a[i]) : f2_hi(a[i]);
          const float taylor = x * fmaf(x, fmaf(x, fmaf(x, 1.0f / 24.0f, 1.0f / 6.0f), 0.5f), 1.0f);
          em1 = fabsf(x) < 0.03125f ? taylor : ak - 1.0f;
        } else {
          em1 = expm1f(x);
        }
        e[k] = ch.invA[n] != 0.0f ? em1 * ch.invA[n] : dl;
      }
      const f2 bb = f2_mul(f2_make(e[0] * u, e[1] * u), bc.b[i]);
      h[i] = f2_fma(a[i], h[i], bb);
    }
  }
  if (kMode == kModeAggregate) return 0.0f;
  f2 acc = f2_mul(bc.c[0], h[0]);
#pragma unroll
  for (int i = 1; i < kNmax / 2; ++i) acc = f2_fma(bc.c[i], h[i], acc);
  float y = f2_lo(acc) + f2_hi(acc);
  y = fmaf(ch.D, u, y);
  if (has_z) y *= kFast ? silu_fast(z) : silu_accurate(z);
  return y;
}

// Float32-io step in double precision.  A float32 evaluation of the recurrence does not meet the
// 2e-5 parity bound beyond a few hundred steps (rounding of Δ, exp(ΔA) and of the state compounds),
// so the float32 io path keeps its coefficients, state and readout in double.
struct ChanD {
  double A[kNmax];
  double D, bias;
};

template <int kDisc, int kMode>
__device__ __forceinline__ double scan_step_precise(const ChanD& ch, double u, double draw, double z, uint32_t bc_row,
                                                    double (&h)[kNmax], bool softplus, bool has_z,
                                                    double& sum_delta) {
  const double v = draw + ch.bias;
  const double dl = softplus ? (v > 0.0 ? v + log1p(exp(-v)) : log1p(exp(v))) : v;
  if (kMode == kModeAggregate) sum_delta += dl;
  double y = 0.0;
#pragma unroll
  for (int q = 0; q < kNmax / 4; ++q) {
    const float4 b4 = lds128f(bc_row + q * 16);
    float4 c4 = make_float4(0.f, 0.f, 0.f, 0.f);
    if (kMode == kModeMain) c4 = lds128f(bc_row + 64 + q * 16);
    const float bb[4] = {b4.x, b4.y, b4.z, b4.w};
    const float cc[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int n = 4 * q + k;
      const double x = dl * ch.A[n];
      const double a = exp(x);
      double bbar;
      if (kDisc == 1 && ch.A[n] != 0.0) bbar = expm1(x) / ch.A[n] * bb[k];
      else bbar = dl * bb[k];
      h[n] = a * h[n] + bbar * u;
      y += cc[k] * h[n];
    }
  }
  if (kMode == kModeAggregate) return 0.0;
  y += ch.D * u;
  if (has_z) y *= z / (1.0 + exp(-z));
  return y;
}

// Widen the B and C tiles of one stage into the float32 table [t][B0..15 | C0..15].
// Rows n >= dstate are written as zeros, so the unused states stay at zero.
template <typename IO>
__device__ __forceinline__ void widen_bc(uint32_t tileB, uint32_t tileC, float* bc32, int N, int tid,
                                         bool need_c) {
  using TL = Tile<IO>;
  // 2 arrays x 16 rows x 8 chunks = 256 jobs over 128 threads
#pragma unroll
  for (int rep = 0; rep < 2; ++rep) {
    const int job = tid + rep * kCH;
    const int arr = job >> 7;            // 0: B, 1: C
    const int n = job & 15;
    const int c = (job >> 4) & 7;
    if (arr == 1 && !need_c) continue;
    float vals[TL::kVec];
    if (n < N) {
      const uint32_t base = arr == 0 ? tileB : tileC;
      const uint4 raw = lds128(base + n * kRowBytes + ((c ^ (n & 7)) << 4));
      unpack_chunk(raw, vals, IO());
    } else {
#pragma unroll
      for (int j = 0; j < TL::kVec; ++j) vals[j] = 0.0f;
    }
#pragma unroll
    for (int j = 0; j < TL::kVec; ++j) bc32[(c * TL::kVec + j) * 32 + arr * 16 + n] = vals[j];
  }
}

// Fill one stage's tiles with plain loads (used when TMA cannot describe the tensors).  The smem
// layout is the same as the TMA one (128-byte swizzle, zeros outside the tensor).
template <typename IO>
__device__ void fill_stage_plain(uint8_t* stage, const ScanParams& p, int b, int d0, int64_t t0, int tid,
                                 int mode) {
  using TL = Tile<IO>;
  const IO* srcs[3] = {static_cast<const IO*>(p.u), static_cast<const IO*>(p.delta),
                       static_cast<const IO*>(p.z)};
  const int narr = (mode == kModeAggregate || p.z == nullptr) ? 2 : 3;
  for (int a = 0; a < narr; ++a) {
    IO* tile = reinterpret_cast<IO*>(stage + a * Smem::kTileIO);
    for (int idx = tid; idx < kCH * TL::kT; idx += kCH) {
      const int r = idx / TL::kT, t = idx % TL::kT;
      const int d = d0 + r;
      const int64_t tt = t0 + t;
      IO v = IoTraits<IO>::from_f32(0.0f);
      if (d < p.dim && tt < p.L)
        v = *checked(srcs[a], (static_cast<int64_t>(b) * p.dim + d) * p.L + tt, static_cast<int64_t>(p.batch) * p.dim * p.L);
      const int chunk = t / TL::kVec, e = t % TL::kVec;
      tile[(r * kRowBytes + (((chunk ^ (r & 7)) << 4))) / IoTraits<IO>::kBytes + e] = v;
    }
  }
  const IO* bcs[2] = {static_cast<const IO*>(p.B), static_cast<const IO*>(p.C)};
  const int nbc = mode == kModeAggregate ? 1 : 2;
  for (int a = 0; a < nbc; ++a) {
    IO* tile = reinterpret_cast<IO*>(stage + 3 * Smem::kTileIO + a * Smem::kTileBC);
    for (int idx = tid; idx < p.N * TL::kT; idx += kCH) {
      const int n = idx / TL::kT, t = idx % TL::kT;
      const int64_t tt = t0 + t;
      IO v = IoTraits<IO>::from_f32(0.0f);
      if (tt < p.L) v = *checked(bcs[a], (static_cast<int64_t>(b) * p.N + n) * p.L + tt, static_cast<int64_t>(p.batch) * p.N * p.L);
      const int chunk = t / TL::kVec, e = t % TL::kVec;
      tile[(n * kRowBytes + (((chunk ^ (n & 7)) << 4))) / IoTraits<IO>::kBytes + e] = v;
    }
  }
}

struct TensorMaps {
  CUtensorMap u, dt, z, B, C;
};

// Main / aggregate pass over one (batch row, 128-channel group, time chunk).
// grid = (ceil(dim/128), batch, nchunks)
template <typename IO, bool kFast, int kDisc, int kMode, bool kTma>
__global__ void __launch_bounds__(kCH, 1)
    scan_chunk_kernel(const __grid_constant__ TensorMaps tm, const ScanParams p) {
  using TL = Tile<IO>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* bc32[2] = {reinterpret_cast<float*>(smem + kStages * Smem::kStage),
                    reinterpret_cast<float*>(smem + kStages * Smem::kStage + Smem::kBC32)};
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Smem::kBars);

  const int tid = threadIdx.x;
  const int b = blockIdx.y;
  const int d0 = blockIdx.x * kCH;
  const int d = d0 + tid;
  const bool valid = d < p.dim;
  const int chunk = blockIdx.z;
  const int64_t t_begin = static_cast<int64_t>(chunk) * p.chunk_len;
  const int64_t t_end = t_begin + p.chunk_len < p.L ? t_begin + p.chunk_len : p.L;
  const int ntiles = static_cast<int>((t_end - t_begin + TL::kT - 1) / TL::kT);
  const bool has_z = p.z != nullptr && kMode == kModeMain;
  const bool load_z = has_z;
  const int row = b * p.dim + d0;   // first tensor row of this CTA's u/Δ/z box
  uint32_t tx_bytes = (2 + (load_z ? 1 : 0)) * Smem::kTileIO +
                      (kMode == kModeMain ? 2 : 1) * p.N * kRowBytes;

  if (kTma && tid == 0) {
#pragma unroll
    for (int s = 0; s < kStages; ++s) mbar_init(&full[s], 1);
    fence_mbar_init();
    prefetch_tensormap(&tm.u);
    prefetch_tensormap(&tm.dt);
    prefetch_tensormap(&tm.B);
    if (load_z) prefetch_tensormap(&tm.z);
    if (kMode == kModeMain) prefetch_tensormap(&tm.C);
  }
  __syncthreads();

  auto issue = [&](int k) {
    uint8_t* st = smem + (k % kStages) * Smem::kStage;
    const int x = static_cast<int>(t_begin + static_cast<int64_t>(k) * TL::kT);
    mbar_arrive_expect_tx(&full[k % kStages], tx_bytes);
    tma_load_2d(st, &tm.u, &full[k % kStages], x, row);
    tma_load_2d(st + Smem::kTileIO, &tm.dt, &full[k % kStages], x, row);
    if (load_z) tma_load_2d(st + 2 * Smem::kTileIO, &tm.z, &full[k % kStages], x, row);
    tma_load_2d(st + 3 * Smem::kTileIO, &tm.B, &full[k % kStages], x, b * p.N);
    if (kMode == kModeMain)
      tma_load_2d(st + 3 * Smem::kTileIO + Smem::kTileBC, &tm.C, &full[k % kStages], x, b * p.N);
  };
  if (kTma && tid == 0) {
    for (int k = 0; k < kStages - 1 && k < ntiles; ++k) issue(k);
  }

  // per-channel constants (the float32-io path keeps them in double)
  Chan ch;
  ChanD chd;
  ch.structured = true;
  {
    const int64_t nA = static_cast<int64_t>(p.dim) * p.N;
    const float a0 = valid ? *checked(p.A, static_cast<int64_t>(d) * p.N, nA) : 0.0f;
#pragma unroll
    for (int n = 0; n < kNmax; ++n) {
      const float an = (valid && n < p.N) ? *checked(p.A, static_cast<int64_t>(d) * p.N + n, nA) : 0.0f;
      ch.AL2[n] = an * kLog2e;
      ch.invA[n] = fabsf(an) >= 0x1p-60f ? 1.0f / an : 0.0f;   // below 2^-60: the A -> 0 limit Δ·B
      chd.A[n] = an;
      if (n < p.N && an != static_cast<float>(n + 1) * a0) ch.structured = false;
    }
    ch.D = (valid && p.D) ? *checked(p.D, d, p.dim) : 0.0f;
    ch.bias = (valid && p.bias) ? *checked(p.bias, d, p.dim) : 0.0f;
    chd.D = ch.D;
    chd.bias = ch.bias;
  }
  // the decay shortcut is decided per warp
  const bool warp_structured = __all_sync(0xffffffffu, ch.structured) && kFast && kDisc == 0;

  // state: 8 packed f32x2 pairs (bf16 io) or 16 doubles (float32 io)
  f2 h[kNmax / 2];
  double hd[kNmax];
  {
    const int64_t base = (static_cast<int64_t>(b) * p.dim + d) * p.N;
    const int64_t coff = static_cast<int64_t>(chunk) * p.h_in_chunk_stride;
#pragma unroll
    for (int n = 0; n < kNmax; ++n) {
      double v = 0.0;
      if (p.h_in && valid && n < p.N) {
        // chunked schedule: nchunks carried-in states; single pass: h0 in h_in (one)
        const int64_t nh = static_cast<int64_t>(gridDim.z) * (p.h_in_chunk_stride ? p.h_in_chunk_stride : base + p.N);
        v = p.carry_f64 ? *checked(static_cast<const double*>(p.h_in), coff + base + n, nh)
                        : static_cast<double>(*checked(static_cast<const float*>(p.h_in), coff + base + n, nh));
      }
      hd[n] = v;
    }
#pragma unroll
    for (int i = 0; i < kNmax / 2; ++i) h[i] = f2_make(static_cast<float>(hd[2 * i]), static_cast<float>(hd[2 * i + 1]));
  }
  float sum_delta = 0.0f;
  double sum_delta_d = 0.0;
  bool ok = true;
  int failed_at = -1;

  IO* yrow = (kMode == kModeMain && valid)
                 ? static_cast<IO*>(p.y) + (static_cast<int64_t>(b) * p.dim + d) * p.L : nullptr;
  const bool vec_store = p.vec_ok;

  for (int k = 0; k < ntiles; ++k) {
    const int s = k % kStages;
    uint8_t* st = smem + s * Smem::kStage;
    const int64_t t0 = t_begin + static_cast<int64_t>(k) * TL::kT;
    if (kTma) {
      ok = mbar_wait_bounded(&full[s], (k / kStages) & 1, &g_device_status);
    } else {
      __syncthreads();   // everyone is done with this stage's previous contents
      fill_stage_plain<IO>(st, p, b, d0, t0, tid, kMode);
      __syncthreads();
    }
    widen_bc<IO>(smem_u32(st + 3 * Smem::kTileIO), smem_u32(st + 3 * Smem::kTileIO + Smem::kTileBC),
                 bc32[k & 1], p.N, tid, kMode == kModeMain);
    // every thread takes part, so a wait that gave up anywhere stops the whole CTA consistently
    ok = __syncthreads_and(ok) != 0;
    if (!ok) {
      failed_at = k;
      break;
    }
    if (kTma && tid == 0 && k + kStages - 1 < ntiles) issue(k + kStages - 1);

    const int steps = static_cast<int>(t_end - t0 < TL::kT ? t_end - t0 : TL::kT);
    const uint32_t urow = smem_u32(st) + tid * kRowBytes;
    const uint32_t drow = urow + Smem::kTileIO;
    const uint32_t zrow = urow + 2 * Smem::kTileIO;
    const uint32_t bcb = smem_u32(bc32[k & 1]);
    const int sw = tid & 7;

    auto one = [&](auto structured_tag, int c, int j, const float* uu, const float* dd, const float* zz) -> float {
      constexpr bool kS = decltype(structured_tag)::value;
      (void)kS;   // used by the float path only
      const uint32_t row = bcb + (c * TL::kVec + j) * 128;
      if constexpr (kFast) {
        BC x;
        load_bc(row, x);
        return scan_step<true, kS, kDisc, kMode>(ch, uu[j], dd[j], zz[j], x, h, p.softplus, has_z, sum_delta);
      } else {
        return static_cast<float>(scan_step_precise<kDisc, kMode>(chd, uu[j], dd[j], zz[j], row, hd, p.softplus,
                                                                   has_z, sum_delta_d));
      }
    };

    auto run = [&](auto structured_tag) {
#pragma unroll 1
      for (int c = 0; c < TL::kChunks; ++c) {
        if (c * TL::kVec >= steps) break;
        float uu[TL::kVec], dd[TL::kVec], zz[TL::kVec], yy[TL::kVec];
        unpack_chunk(lds128(urow + ((c ^ sw) << 4)), uu, IO());
        unpack_chunk(lds128(drow + ((c ^ sw) << 4)), dd, IO());
        if (has_z) unpack_chunk(lds128(zrow + ((c ^ sw) << 4)), zz, IO());
        else {
#pragma unroll
          for (int j = 0; j < TL::kVec; ++j) zz[j] = 0.0f;
        }
        const int nvalid = steps - c * TL::kVec;
        if (nvalid >= TL::kVec) {
#pragma unroll
          for (int j = 0; j < TL::kVec; ++j) yy[j] = one(structured_tag, c, j, uu, dd, zz);
          if (kMode == kModeMain && valid) {
            const int64_t t = t0 + c * TL::kVec;
            if (vec_store) {
              *reinterpret_cast<uint4*>(checked(yrow, t, p.L - 0, TL::kVec)) = pack_chunk(yy);
            } else {
#pragma unroll
              for (int j = 0; j < TL::kVec; ++j) *checked(yrow, t + j, p.L) = IoTraits<IO>::from_f32(yy[j]);
            }
          }
        } else {
#pragma unroll
          for (int j = 0; j < TL::kVec; ++j) {
            if (j < nvalid) {
              yy[j] = one(structured_tag, c, j, uu, dd, zz);
              if (kMode == kModeMain && valid) *checked(yrow, t0 + c * TL::kVec + j, p.L) = IoTraits<IO>::from_f32(yy[j]);
            }
          }
        }
      }
    };
    if (warp_structured) run(std::true_type());
    else run(std::false_type());
  }

  if (failed_at >= 0) {
    // a wait gave up: wait (bounded) for the copies this CTA still has in flight, then leave
    if (kTma && tid == 0) {
      const int issued = failed_at + kStages - 1 < ntiles ? failed_at + kStages - 1 : ntiles;
      for (int k = failed_at; k < issued; ++k)
        (void)mbar_wait_bounded(&full[k % kStages], (k / kStages) & 1, &g_device_status, 100000000ull);
    }
    return;
  }
  if (!valid) return;
  if constexpr (kFast) {
#pragma unroll
    for (int i = 0; i < kNmax / 2; ++i) {
      hd[2 * i] = f2_lo(h[i]);
      hd[2 * i + 1] = f2_hi(h[i]);
    }
    sum_delta_d = sum_delta;
  }
  const int64_t sbase = (static_cast<int64_t>(b) * p.dim + d) * p.N;
  if (kMode == kModeMain) {
    if (p.last_state && chunk == static_cast<int>(gridDim.z) - 1) {
#pragma unroll
      for (int n = 0; n < kNmax; ++n)
        if (n < p.N) *checked(p.last_state, sbase + n, static_cast<int64_t>(p.batch) * p.dim * p.N) = static_cast<float>(hd[n]);
    }
  } else {
    // aggregate of this chunk: P = Π exp(Δ A) = exp(A ΣΔ) (one accurate exp per state), Q = h_end
    const int64_t cbase = static_cast<int64_t>(chunk) * p.h_in_chunk_stride + sbase;
#pragma unroll
    for (int n = 0; n < kNmax; ++n) {
      if (n < p.N) {
        const float an = *checked(p.A, static_cast<int64_t>(d) * p.N + n, static_cast<int64_t>(p.dim) * p.N);
        const int64_t nagg = static_cast<int64_t>(gridDim.z) * p.h_in_chunk_stride;
        if (p.carry_f64) {
          *checked(static_cast<double*>(p.agg_P), cbase + n, nagg) = exp(static_cast<double>(an) * sum_delta_d);
          *checked(static_cast<double*>(p.agg_Q), cbase + n, nagg) = hd[n];
        } else {
          *checked(static_cast<float*>(p.agg_P), cbase + n, nagg) = expf(an * sum_delta);
          *checked(static_cast<float*>(p.agg_Q), cbase + n, nagg) = static_cast<float>(hd[n]);
        }
      }
    }
  }
}

// Carry pass: h_in[0] = h0 (or 0); h_in[k+1] = P[k] ⊙ h_in[k] + Q[k].  One thread per (b, d, n).
template <typename T>
__global__ void carry_kernel(const T* __restrict__ P, const T* __restrict__ Q, const float* __restrict__ h0,
                             T* __restrict__ h_in, int64_t per_chunk, int nchunks) {
  const int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  if (i >= per_chunk) return;
  T h = h0 ? static_cast<T>(h0[i]) : T(0);
  h_in[i] = h;
  for (int k = 0; k + 1 < nchunks; ++k) {
    h = P[k * per_chunk + i] * h + Q[k * per_chunk + i];
    h_in[(k + 1) * per_chunk + i] = h;
  }
}

template <typename IO, bool kFast, int kDisc, int kMode, bool kTma>
cudaError_t launch_one(const TensorMaps& tm, const ScanParams& p, int nchunks, cudaStream_t stream) {
  auto kern = scan_chunk_kernel<IO, kFast, kDisc, kMode, kTma>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Smem::kTotal);
  if (e != cudaSuccess) return e;
  dim3 grid((p.dim + kCH - 1) / kCH, p.batch, nchunks);
  kern<<<grid, kCH, Smem::kTotal, stream>>>(tm, p);
  return cudaGetLastError();
}

template <typename IO, bool kFast, int kMode, bool kTma>
cudaError_t launch_disc(const TensorMaps& tm, const ScanParams& p, int nchunks, cudaStream_t stream) {
  if (p.disc == 1) return launch_one<IO, kFast, 1, kMode, kTma>(tm, p, nchunks, stream);
  return launch_one<IO, kFast, 0, kMode, kTma>(tm, p, nchunks, stream);
}

template <typename IO, int kMode>
cudaError_t launch_pass(const TensorMaps& tm, const ScanParams& p, int nchunks, bool tma, cudaStream_t stream) {
  constexpr bool kFast = sizeof(IO) == 2;
  if (tma) return launch_disc<IO, kFast, kMode, true>(tm, p, nchunks, stream);
  return launch_disc<IO, kFast, kMode, false>(tm, p, nchunks, stream);
}

}  // namespace

int scan_tile_steps(int io_bytes) { return kRowBytes / io_bytes; }

cudaError_t general_check_read_and_clear(unsigned int* out) { return tu_check_read_and_clear(out); }

cudaError_t read_and_clear_device_status(unsigned int* out, cudaStream_t stream) {
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return e;
  e = cudaMemcpyFromSymbol(out, g_device_status, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  const unsigned int zero = 0;
  e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  unsigned int scaled = 0;
  e = scaled_status_read_and_clear(&scaled);
  *out |= scaled;
  if (e != cudaSuccess) return e;
  unsigned int ssd = 0;
  e = ssd_status_read_and_clear(&ssd);
  *out |= ssd;
  if (e != cudaSuccess) return e;
  unsigned int st = 0;
  e = selftest_status_read_and_clear(&st);
  *out |= st;
  if (e != cudaSuccess) return e;
  // index checks of the checked build (each reader returns 0 in the ordinary build)
  cudaError_t (*const readers[])(unsigned int*) = {general_check_read_and_clear, scaled_check_read_and_clear,
                                                    decode_check_read_and_clear,  conv1d_check_read_and_clear,
                                                    ssd_check_read_and_clear,     ssd_decode_check_read_and_clear,
                                                    bwd_check_read_and_clear};
  for (auto* r : readers) {
    unsigned int c = 0;
    e = r(&c);
    *out |= c;
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t carry_launch_f32(const ScanParams& p, int nchunks, cudaStream_t stream) {
  const int64_t per_chunk = static_cast<int64_t>(p.batch) * p.dim * p.N;
  const unsigned blocks = static_cast<unsigned>((per_chunk + 255) / 256);
  carry_kernel<float><<<blocks, 256, 0, stream>>>(static_cast<const float*>(p.agg_P),
                                                   static_cast<const float*>(p.agg_Q), p.h0,
                                                   static_cast<float*>(const_cast<void*>(p.h_in)), per_chunk,
                                                   nchunks);
  return cudaGetLastError();
}

// Builds the tensor maps (when the layout allows TMA) and launches the passes.
cudaError_t scan_fwd_launch(const ScanParams& p_in, int nchunks, cudaStream_t stream, char* err, size_t errlen) {
  ScanParams p = p_in;
  const int ebytes = p.io_bf16 ? 2 : 4;
  TensorMaps tm;
  memset(&tm, 0, sizeof(tm));
  bool tma = p.tma_ok;
  if (tma) {
    const int T = kRowBytes / ebytes;
    const CUtensorMapDataType dt = p.io_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    struct M {
      CUtensorMap* map;
      const void* ptr;
      uint64_t rows;
      uint32_t box_rows;
    } maps[5] = {{&tm.u, p.u, static_cast<uint64_t>(p.batch) * p.dim, kCH},
                 {&tm.dt, p.delta, static_cast<uint64_t>(p.batch) * p.dim, kCH},
                 {&tm.z, p.z ? p.z : p.u, static_cast<uint64_t>(p.batch) * p.dim, kCH},
                 {&tm.B, p.B, static_cast<uint64_t>(p.batch) * p.N, static_cast<uint32_t>(p.N)},
                 {&tm.C, p.C, static_cast<uint64_t>(p.batch) * p.N, static_cast<uint32_t>(p.N)}};
    for (auto& m : maps) {
      if (!encode_tensor_map_2d(m.map, dt, const_cast<void*>(m.ptr), static_cast<uint64_t>(p.L), m.rows,
                                static_cast<uint64_t>(p.L) * ebytes, static_cast<uint32_t>(T), m.box_rows,
                                err, errlen)) {
        tma = false;
        break;
      }
    }
  }
  if (nchunks > 1) {
    // 1. aggregates of chunks 0..nchunks-2, each from a zero state
    ScanParams pa = p;
    pa.h_in = nullptr;
    cudaError_t e = p.io_bf16 ? launch_pass<__nv_bfloat16, kModeAggregate>(tm, pa, nchunks - 1, tma, stream)
                              : launch_pass<float, kModeAggregate>(tm, pa, nchunks - 1, tma, stream);
    if (e != cudaSuccess) return e;
    // 2. carry
    const int64_t per_chunk = static_cast<int64_t>(p.batch) * p.dim * p.N;
    const unsigned blocks = static_cast<unsigned>((per_chunk + 255) / 256);
    if (p.carry_f64)
      carry_kernel<double><<<blocks, 256, 0, stream>>>(static_cast<const double*>(p.agg_P),
                                                        static_cast<const double*>(p.agg_Q), p.h0,
                                                        static_cast<double*>(const_cast<void*>(p.h_in)),
                                                        per_chunk, nchunks);
    else
      carry_kernel<float><<<blocks, 256, 0, stream>>>(static_cast<const float*>(p.agg_P),
                                                       static_cast<const float*>(p.agg_Q), p.h0,
                                                       static_cast<float*>(const_cast<void*>(p.h_in)),
                                                       per_chunk, nchunks);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  // 3. main pass
  return p.io_bf16 ? launch_pass<__nv_bfloat16, kModeMain>(tm, p, nchunks, tma, stream)
                   : launch_pass<float, kModeMain>(tm, p, nchunks, tma, stream);
}

}  // namespace ssm
