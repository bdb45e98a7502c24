// Prefill selective scan on a rescaled state: bf16 io, one thread per channel, sm_103a.
//
// Operator ("Mamba и State Space Models", "Selective Scan (core algorithm)"; "State Space Models:
// Mamba и альтернатива Transformer", "Mamba: Selective State Space"):
//   Δ_t = softplus(Δ_raw + bias);  h_t = exp(Δ_t A) ⊙ h_{t-1} + Δ_t B_t u_t;  y_t = (C_t·h_t + D u_t)·SiLU(z_t)
//
// Rescaled state.  Write Δ_t = ln2·ℓ_t (ℓ_t is Δ in base-2 units) and σ_t = ℓ_t u_t, so that
// Δ_t u_t = ln2·σ_t.  The kernel carries g_t = h_t / σ_t instead of h_t.  Dividing the recurrence by
// σ_t gives
//   g_t = exp(Δ_t A) ρ_t ⊙ g_{t-1} + ln2·B_t,   ρ_t = σ_{t-1}/σ_t,   y_t = σ_t (C_t·g_t) + D u_t,
// an exact rewrite of the same recurrence in which the input term needs no multiply: per state and
// step there are three float32 operations (the decay ρ_t exp(Δ_t A[d,n]), the state FMA with the
// table value ln2·B_t[n], the readout FMA) instead of four.  ρ_t folds into the decay for free: with
// A[d,n] = (n+1)·A[d,0] the decays are ρ_t r^(n+1), r = exp(Δ_t A[d,0]), a multiply tree rooted at
// ρ_t r.  The segment starts from g = h_init (σ_init = 1) and ends with h = σ_last·g.  |σ_t| below
// 1e-20 (u_t = 0, or Δ_t underflowing to 0) is replaced by 1e-20, which adds at most 1e-20·ln2·|B_t|
// to the state where the exact input term is smaller than that.
//
// Layout of the work:
//  * A CTA is 128 threads and owns 128 consecutive channels of one batch row (a "group"): one
//    channel per thread, all 16 states in registers (8 packed f32x2 pairs), one CTA per SM.
//  * u, Δ_raw, z tiles [128 channels x 64 steps] and B, C tiles [dstate x 64 steps] arrive by TMA
//    with a 128-byte swizzle through a 4-stage mbarrier pipeline.  At the start of tile k the CTA
//    widens tile k+1's B and C into a float32 table [step][ln2·B_0..15 | C_0..15], read by every
//    thread with broadcast 128-bit loads.
//  * Per 8-step chunk a thread computes the chunk's per-step scalars (ℓ, ρ, σ·SiLU(z), D u·SiLU(z))
//    one chunk ahead of the recurrence that consumes them, so that their MUFU chains overlap the
//    previous chunk's state updates.
//  * Scheduling: the balanced persistent schedule or the grid schedule of scan_walk.cuh, with the
//    CTA-to-CTA carry of the balanced schedule behind a bounded wait.
//  * Aggregate mode (chunked schedule): per (group, chunk) from a zero state, the chunk's decay
//    product exp(A ΣΔ) and end state, for the carry pass ("Модуль 8", §7).
#include <cstring>
#include <type_traits>

#include "internal.h"
#include "scan_walk.cuh"
#include "ssm_device.cuh"

#ifndef SSM_SCALED_SCALARS_AFTER
#define SSM_SCALED_SCALARS_AFTER 0    // 1: the next chunk's scalars after this chunk's recurrence in program order
#endif
#ifndef SSM_SCALED_CHUNK
#define SSM_SCALED_CHUNK 8            // steps per chunk: 8 or 4
#endif
#ifndef SSM_SCALED_LANES
#define SSM_SCALED_LANES 2            // lanes per channel: 1 (16 states per thread) or 2 (8 states each)
#endif
#ifndef SSM_SCALED_PLAIN_BC_LOADS
#define SSM_SCALED_PLAIN_BC_LOADS 0   // 1: table reads as plain C++ loads (the compiler may hoist them)
#endif

namespace ssm {
namespace {

__device__ unsigned int g_scaled_status = 0;

constexpr int kCh = 128;    // channels (threads) per CTA
constexpr int kT = 64;      // steps per tile
constexpr int kSt = 4;      // TMA stages
constexpr int kRow = 128;   // bytes of one tile row (64 bf16 steps)
constexpr int kN = 16;      // register state width
constexpr int kC = SSM_SCALED_CHUNK;   // steps per chunk
constexpr int kLanesDefault = SSM_SCALED_LANES;
constexpr int kCP = kC / 2;            // step pairs per chunk
constexpr float kSigmaMin = 1e-20f;
constexpr uint64_t kWaitNs = 2000000000ull;

struct SmemS {
  static constexpr int kTileIO = kCh * kRow;                // 16 KB: u, Δ_raw or z tile
  static constexpr int kTileBC = kN * kRow;                 // 2 KB: B or C tile
  static constexpr int kStage = 3 * kTileIO + 2 * kTileBC;  // 52 KB
  static constexpr int kTab = kT * 2 * kN * 4;              // 8 KB: float32 [step][32] table
  static constexpr int kBars = kSt * kStage + 2 * kTab;     // 224 KB
  static constexpr int kTotal = kBars + 64 + 1024;          // + mbarriers + alignment slack
};

enum { kMain = 0, kAgg = 1 };

struct MapsS {
  CUtensorMap u, dt, z, B, C;
};

// Per-step scalars of one 8-step chunk of one channel, as pairs of consecutive steps.
struct Sc {
  f2 l2[kCP];    // ℓ = Δ/ln2
  f2 rho[kCP];   // σ_{t-1}/σ_t
  f2 al[kCP];    // σ_t·SiLU(z_t)            (main mode)
  f2 be[kCP];    // D·u_t·SiLU(z_t)          (main mode)
  float sig;   // σ of the chunk's last step
  float lsum;  // Σ ℓ over the chunk       (aggregate mode)
};

// Per-channel constants of a segment.
struct Chan {
  float bias2;   // bias·log2(e)
  float D;
  float A0;      // A[d,0]
  int b, d;
  bool valid;
  bool structured;   // warp-uniform: every lane's row has A[d,n] = (n+1)·A[d,0]
};

__device__ __forceinline__ float pick(f2 v, int j) { return (j & 1) ? f2_hi(v) : f2_lo(v); }

// Scalars of chunk c of the tile whose u row (this thread's channel) starts at `urow` in shared memory.
template <int kMode>
__device__ __forceinline__ void chunk_scalars(Sc& s, uint32_t urow, int c, int sw, float bias2, float D, float sig_prev,
                                              bool softplus, bool has_z) {
  // this chunk's steps inside the 16-byte (8-step) swizzled unit of the row
  const uint32_t off = static_cast<uint32_t>((((c * kC) >> 3) ^ sw) << 4) + ((c * kC) & 7) * 2;
  uint32_t uu[kCP], dd[kCP], zz[kCP];
  if (kC == 8) {
    const uint4 uw = lds128(urow + off);
    const uint4 dw = lds128(urow + SmemS::kTileIO + off);
    uint4 zw = make_uint4(0u, 0u, 0u, 0u);
    if (kMode == kMain && has_z) zw = lds128(urow + 2 * SmemS::kTileIO + off);
    const uint32_t a[4] = {uw.x, uw.y, uw.z, uw.w}, b[4] = {dw.x, dw.y, dw.z, dw.w}, e[4] = {zw.x, zw.y, zw.z, zw.w};
#pragma unroll
    for (int q = 0; q < kCP; ++q) { uu[q] = a[q]; dd[q] = b[q]; zz[q] = e[q]; }
  } else {
    const uint2 uw = lds64(urow + off);
    const uint2 dw = lds64(urow + SmemS::kTileIO + off);
    uint2 zw = make_uint2(0u, 0u);
    if (kMode == kMain && has_z) zw = lds64(urow + 2 * SmemS::kTileIO + off);
    const uint32_t a[2] = {uw.x, uw.y}, b[2] = {dw.x, dw.y}, e[2] = {zw.x, zw.y};
#pragma unroll
    for (int q = 0; q < kCP; ++q) { uu[q] = a[q % 2]; dd[q] = b[q % 2]; zz[q] = e[q % 2]; }
  }
  f2 lsum2 = f2_splat(0.0f);
#pragma unroll
  for (int q = 0; q < kCP; ++q) {
    const f2 u2 = f2_make(bf16lo_to_f32(uu[q]), bf16hi_to_f32(uu[q]));
    const f2 v2 = f2_make(bf16lo_to_f32(dd[q]), bf16hi_to_f32(dd[q]));
    const f2 x = f2_fma(v2, f2_splat(kLog2e), f2_splat(bias2));   // (Δ_raw + bias)·log2(e)
    f2 l2 = x;
    if (softplus) {
      // ℓ = log2(1 + 2^x) = softplus(v)/ln2; max(., x) covers x > 64, where 2^x is clamped
      const f2 e = f2_make(ex2_approx(fminf(f2_lo(x), 64.0f)), ex2_approx(fminf(f2_hi(x), 64.0f)));
      const f2 w = f2_add(e, f2_splat(1.0f));
      l2 = f2_make(fmaxf(lg2_approx(f2_lo(w)), f2_lo(x)), fmaxf(lg2_approx(f2_hi(w)), f2_hi(x)));
    }
    s.l2[q] = l2;
    if (kMode == kAgg) lsum2 = f2_add(lsum2, l2);
    const f2 sg = f2_mul(l2, u2);
    float s0 = f2_lo(sg), s1 = f2_hi(sg);
    s0 = fabsf(s0) < kSigmaMin ? kSigmaMin : s0;
    s1 = fabsf(s1) < kSigmaMin ? kSigmaMin : s1;
    s.rho[q] = f2_mul(f2_make(sig_prev, s0), f2_make(rcp_approx(s0), rcp_approx(s1)));
    sig_prev = s1;
    if (kMode == kMain) {
      f2 g = f2_splat(1.0f);
      if (has_z) {
        const f2 z2 = f2_make(bf16lo_to_f32(zz[q]), bf16hi_to_f32(zz[q]));
        const f2 t = f2_mul(z2, f2_splat(-kLog2e));
        const f2 den = f2_add(f2_make(ex2_approx(f2_lo(t)), ex2_approx(f2_hi(t))), f2_splat(1.0f));
        g = f2_mul(z2, f2_make(rcp_approx(f2_lo(den)), rcp_approx(f2_hi(den))));
      }
      s.al[q] = f2_mul(f2_make(s0, s1), g);
      s.be[q] = f2_mul(f2_mul(f2_splat(D), u2), g);
    }
  }
  s.sig = sig_prev;
  if (kMode == kAgg) s.lsum = f2_lo(lsum2) + f2_hi(lsum2);
}

__device__ __forceinline__ float4 tab_load(uint32_t addr) {
#if SSM_SCALED_PLAIN_BC_LOADS
  float4 v;
  asm("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
  return v;
#else
  return lds128f(addr);
#endif
}

// The recurrence over one 8-step chunk: g ← ρ exp(ΔA) ⊙ g + ln2·B, then (main mode) the readout
// y = σ·SiLU(z)·(C·g) + D·u·SiLU(z) for each step, returned packed as eight bf16 values.
template <int kMode, bool kS>
__device__ __forceinline__ uint4 chunk_run(f2 (&h)[8], const Sc& s, uint32_t tab, const Chan& k, const float* Arow,
                                           int N) {
  float Ag[kN];
  if (!kS) {
#pragma unroll
    for (int n = 0; n < kN; ++n) Ag[n] = n < N ? __ldg(Arow + n) : 0.0f;
  }
  float y[kC];
#pragma unroll
  for (int j = 0; j < kC; ++j) {
    const float l2 = pick(s.l2[j >> 1], j);
    const float rho = pick(s.rho[j >> 1], j);
    const uint32_t row = tab + j * 128;
    f2 P[8];
    if (kS) {
      // ρ r^(n+1), n = 0..15, r = exp(Δ A[d,0]) = 2^(ℓ A[d,0])
      const float r = ex2_approx(l2 * k.A0);
      const float r2 = r * r, r4 = r2 * r2, r8 = r4 * r4;
      const float c0 = rho * r;
      P[0] = f2_make(c0, c0 * r);
      P[1] = f2_mul(P[0], f2_splat(r2));
      P[2] = f2_mul(P[0], f2_splat(r4));
      P[3] = f2_mul(P[1], f2_splat(r4));
#pragma unroll
      for (int i = 0; i < 4; ++i) P[4 + i] = f2_mul(P[i], f2_splat(r8));
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        P[i] = f2_make(rho * ex2_approx(l2 * Ag[2 * i]), rho * ex2_approx(l2 * Ag[2 * i + 1]));
    }
    const float4 b0 = tab_load(row), b1 = tab_load(row + 16), b2 = tab_load(row + 32), b3 = tab_load(row + 48);
    h[0] = f2_fma(P[0], h[0], f2_make(b0.x, b0.y));
    h[1] = f2_fma(P[1], h[1], f2_make(b0.z, b0.w));
    h[2] = f2_fma(P[2], h[2], f2_make(b1.x, b1.y));
    h[3] = f2_fma(P[3], h[3], f2_make(b1.z, b1.w));
    h[4] = f2_fma(P[4], h[4], f2_make(b2.x, b2.y));
    h[5] = f2_fma(P[5], h[5], f2_make(b2.z, b2.w));
    h[6] = f2_fma(P[6], h[6], f2_make(b3.x, b3.y));
    h[7] = f2_fma(P[7], h[7], f2_make(b3.z, b3.w));
    if (kMode == kMain) {
      const float4 c0v = tab_load(row + 64), c1v = tab_load(row + 80), c2v = tab_load(row + 96),
                   c3v = tab_load(row + 112);
      f2 a0 = f2_mul(f2_make(c0v.x, c0v.y), h[0]);
      f2 a1 = f2_mul(f2_make(c0v.z, c0v.w), h[1]);
      a0 = f2_fma(f2_make(c1v.x, c1v.y), h[2], a0);
      a1 = f2_fma(f2_make(c1v.z, c1v.w), h[3], a1);
      a0 = f2_fma(f2_make(c2v.x, c2v.y), h[4], a0);
      a1 = f2_fma(f2_make(c2v.z, c2v.w), h[5], a1);
      a0 = f2_fma(f2_make(c3v.x, c3v.y), h[6], a0);
      a1 = f2_fma(f2_make(c3v.z, c3v.w), h[7], a1);
      const f2 sum = f2_add(a0, a1);
      y[j] = fmaf(pick(s.al[j >> 1], j), f2_lo(sum) + f2_hi(sum), pick(s.be[j >> 1], j));
    }
  }
  if (kMode != kMain) return make_uint4(0u, 0u, 0u, 0u);
  if (kC == 8)
    return make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]), pack_bf16x2(y[4], y[5 % kC]),
                      pack_bf16x2(y[6 % kC], y[7 % kC]));
  return make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]), 0u, 0u);
}

// ---------------------------------------------------------------- two lanes per channel
// Lane p of a channel holds states [8p, 8p+8) and owns steps [4p, 4p+4) of every 8-step chunk: it
// computes those steps' scalars and finishes their outputs.  Each step's decay exponent and ρ reach
// both lanes by shuffles; each step's readout is the sum of the two lanes' halves.
struct Sc2 {
  float q[8];      // per step: ℓ·A[d,0] (structured A) or ℓ (general A)
  float rho[8];    // per step: σ_{t-1}/σ_t
  f2 al[2];        // own steps: σ_t·SiLU(z_t)
  f2 be[2];        // own steps: D·u_t·SiLU(z_t)
  float sig;       // σ of the chunk's last step (both lanes)
  float lsum;      // Σ ℓ over the own steps (aggregate mode)
};

template <int kMode>
__device__ __forceinline__ void chunk_scalars2(Sc2& s, uint32_t urow, int c, int sw, int pl, float bias2, float D,
                                               float qmul, float sig_prev, bool softplus, bool has_z) {
  const uint32_t off = static_cast<uint32_t>((c ^ sw) << 4) + 8u * pl;   // own 4 steps: 8 bytes of the unit
  const uint2 uw = lds64(urow + off);
  const uint2 dw = lds64(urow + SmemS::kTileIO + off);
  uint2 zw = make_uint2(0u, 0u);
  if (kMode == kMain && has_z) zw = lds64(urow + 2 * SmemS::kTileIO + off);
  const uint32_t uu[2] = {uw.x, uw.y}, dd[2] = {dw.x, dw.y}, zz[2] = {zw.x, zw.y};
  float qo[4], sg[4], rs[4];
  float lsum = 0.0f;
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const f2 u2 = f2_make(bf16lo_to_f32(uu[q]), bf16hi_to_f32(uu[q]));
    const f2 v2 = f2_make(bf16lo_to_f32(dd[q]), bf16hi_to_f32(dd[q]));
    const f2 x = f2_fma(v2, f2_splat(kLog2e), f2_splat(bias2));
    f2 l2 = x;
    if (softplus) {
      const f2 e = f2_make(ex2_approx(fminf(f2_lo(x), 64.0f)), ex2_approx(fminf(f2_hi(x), 64.0f)));
      const f2 w = f2_add(e, f2_splat(1.0f));
      l2 = f2_make(fmaxf(lg2_approx(f2_lo(w)), f2_lo(x)), fmaxf(lg2_approx(f2_hi(w)), f2_hi(x)));
    }
    if (kMode == kAgg) lsum += f2_lo(l2) + f2_hi(l2);
    const f2 qq = f2_mul(l2, f2_splat(qmul));
    qo[2 * q] = f2_lo(qq);
    qo[2 * q + 1] = f2_hi(qq);
    const f2 sgm = f2_mul(l2, u2);
    float s0 = f2_lo(sgm), s1 = f2_hi(sgm);
    s0 = fabsf(s0) < kSigmaMin ? kSigmaMin : s0;
    s1 = fabsf(s1) < kSigmaMin ? kSigmaMin : s1;
    sg[2 * q] = s0;
    sg[2 * q + 1] = s1;
    rs[2 * q] = rcp_approx(s0);
    rs[2 * q + 1] = rcp_approx(s1);
    if (kMode == kMain) {
      f2 g = f2_splat(1.0f);
      if (has_z) {
        const f2 z2 = f2_make(bf16lo_to_f32(zz[q]), bf16hi_to_f32(zz[q]));
        const f2 t = f2_mul(z2, f2_splat(-kLog2e));
        const f2 den = f2_add(f2_make(ex2_approx(f2_lo(t)), ex2_approx(f2_hi(t))), f2_splat(1.0f));
        g = f2_mul(z2, f2_make(rcp_approx(f2_lo(den)), rcp_approx(f2_hi(den))));
      }
      s.al[q] = f2_mul(f2_make(s0, s1), g);
      s.be[q] = f2_mul(f2_mul(f2_splat(D), u2), g);
    }
  }
  // σ before the first own step: lane 1 takes step 3 from lane 0; lane 0 takes the previous chunk's
  // step 7 (sig_prev), which lane 1 handed over at the end of that chunk
  const float s3x = __shfl_xor_sync(0xffffffffu, sg[3], 1);
  const float first_prev = pl ? s3x : sig_prev;
  float ro[4];
  ro[0] = first_prev * rs[0];
  ro[1] = sg[0] * rs[1];
  ro[2] = sg[1] * rs[2];
  ro[3] = sg[2] * rs[3];
  s.sig = pl ? sg[3] : s3x;
  const int base = (threadIdx.x & 31) & ~1;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    s.q[j] = __shfl_sync(0xffffffffu, qo[j & 3], base | (j >> 2));
    s.rho[j] = __shfl_sync(0xffffffffu, ro[j & 3], base | (j >> 2));
  }
  s.lsum = lsum;
}

// The recurrence of one lane's 8 states over one 8-step chunk; returns the lane's four own outputs
// packed as bf16 (main mode).
template <int kMode, bool kS>
__device__ __forceinline__ uint2 chunk_run2(f2 (&h)[4], const Sc2& s, uint32_t tab, int pl, float kb,
                                            const float* Arow, int N) {
  float Ah[8];
  if (!kS) {
#pragma unroll
    for (int i = 0; i < 8; ++i) Ah[i] = 8 * pl + i < N ? __ldg(Arow + 8 * pl + i) : 0.0f;
  }
  float part[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float q = s.q[j];
    const float rho = s.rho[j];
    const uint32_t row = tab + j * 128 + pl * 32;
    f2 a[4];
    if (kS) {
      // ρ r^(8p+1) .. ρ r^(8p+8), r = 2^q
      const float r = ex2_approx(q);
      const float c0 = rho * ex2_approx(q * kb);
      const float r2 = r * r, r4 = r2 * r2;
      a[0] = f2_make(c0, c0 * r);
      a[1] = f2_mul(a[0], f2_splat(r2));
      a[2] = f2_mul(a[0], f2_splat(r4));
      a[3] = f2_mul(a[1], f2_splat(r4));
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = f2_make(rho * ex2_approx(q * Ah[2 * i]), rho * ex2_approx(q * Ah[2 * i + 1]));
    }
    const float4 b0 = tab_load(row), b1 = tab_load(row + 16);
    h[0] = f2_fma(a[0], h[0], f2_make(b0.x, b0.y));
    h[1] = f2_fma(a[1], h[1], f2_make(b0.z, b0.w));
    h[2] = f2_fma(a[2], h[2], f2_make(b1.x, b1.y));
    h[3] = f2_fma(a[3], h[3], f2_make(b1.z, b1.w));
    if (kMode == kMain) {
      const float4 c0v = tab_load(row + 64), c1v = tab_load(row + 80);
      f2 a0 = f2_mul(f2_make(c0v.x, c0v.y), h[0]);
      f2 a1 = f2_mul(f2_make(c0v.z, c0v.w), h[1]);
      a0 = f2_fma(f2_make(c1v.x, c1v.y), h[2], a0);
      a1 = f2_fma(f2_make(c1v.z, c1v.w), h[3], a1);
      const f2 sum = f2_add(a0, a1);
      part[j] = f2_lo(sum) + f2_hi(sum);
    }
  }
  if constexpr (kMode != kMain) {
    return make_uint2(0u, 0u);
  }
  // each lane finishes its own four steps: its half plus the partner's half
  float y[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float send = pl ? part[i] : part[4 + i];
    const float mine = pl ? part[4 + i] : part[i];
    const float tot = mine + __shfl_xor_sync(0xffffffffu, send, 1);
    y[i] = fmaf(pick(s.al[i >> 1], i), tot, pick(s.be[i >> 1], i));
  }
  return make_uint2(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]));
}

template <int kMode, int kLanes>
__global__ void __launch_bounds__(kCh * kLanes, 1) scan_scaled_kernel(const __grid_constant__ MapsS tm,
                                                                        const ScanParams p) {
  constexpr int kThr = kCh * kLanes;
  constexpr int kNs = kN / kLanes;     // states per lane
  static_assert(kLanes == 1 || (kLanes == 2 && kC == 8), "two lanes per channel need 8-step chunks");
  using ScT = typename std::conditional<kLanes == 1, Sc, Sc2>::type;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // table of tile k: tab_at(k)
  auto tab_at = [&](int64_t k) { return reinterpret_cast<float*>(smem + kSt * SmemS::kStage + (k & 1) * SmemS::kTab); };
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + SmemS::kBars);
  __shared__ int s_carry_ok;

  const int tid = threadIdx.x;
  const int ch = tid / kLanes;                     // channel within the group
  const int pl = tid % kLanes;                     // lane within the channel
  const int n0 = pl * kNs;                         // this lane's first state
  const int sw = ch & 7;                           // 128-byte swizzle of this channel's tile row
  const int64_t Lt = (p.L + kT - 1) / kT;
  const int gpb = (p.dim + kCh - 1) / kCh;         // groups per batch row
  const bool has_z = kMode == kMain && p.z != nullptr;
  const bool softplus = p.softplus != 0;

  Walk w;
  int64_t chunk_idx = 0;
  if (p.sched_balanced) {
    w = make_walk_balanced(blockIdx.x, p.range_tiles, static_cast<int64_t>(p.batch) * gpb * Lt, Lt);
  } else {
    chunk_idx = blockIdx.y;
    w = make_walk_grid(blockIdx.x, chunk_idx, (p.chunk_len + kT - 1) / kT, Lt);
  }
  const int64_t ntiles = w.total();
  if (ntiles <= 0) return;

  const uint32_t tx_bytes = (2 + (has_z ? 1 : 0)) * SmemS::kTileIO + (kMode == kMain ? 2 : 1) * p.N * kRow;
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

  // thread 0's issue stream: tile `issued`, at (gi, ti)
  int64_t gi = 0, ti = 0;
  w.at(0, gi, ti);
  auto issue = [&](int64_t k) {
    const int64_t g = gi, t = ti;
    w.advance(k, gi, ti);
    const int g32 = static_cast<int>(g);
    const int b = g32 / gpb;
    const int row = b * p.dim + (g32 - b * gpb) * kCh;
    const int x = static_cast<int>(t * kT);
    uint8_t* st = smem + (k % kSt) * SmemS::kStage;
    uint64_t* bar = &full[k % kSt];
    mbar_arrive_expect_tx(bar, tx_bytes);
    tma_load_2d(st, &tm.u, bar, x, row);
    tma_load_2d(st + SmemS::kTileIO, &tm.dt, bar, x, row);
    if (has_z) tma_load_2d(st + 2 * SmemS::kTileIO, &tm.z, bar, x, row);
    tma_load_2d(st + 3 * SmemS::kTileIO, &tm.B, bar, x, b * p.N);
    if (kMode == kMain) tma_load_2d(st + 3 * SmemS::kTileIO + SmemS::kTileBC, &tm.C, bar, x, b * p.N);
  };
  int64_t issued = 0;   // tiles issued so far (thread 0)
  if (tid == 0) {
    for (int64_t k = 0; k < kSt - 1 && k < ntiles; ++k) issue(k);
    issued = ntiles < kSt - 1 ? ntiles : kSt - 1;
  }

  // Widens tile k's B and C (stage k % kSt) into table k & 1: ln2·B in columns 0..15, C in 16..31,
  // zero rows for n >= dstate.  256 jobs (array, n, 8-step chunk) over the CTA; a warp's 32 threads
  // store 32 consecutive words.
  auto widen = [&](int64_t k) {
    const uint32_t src = smem_u32(smem + (k % kSt) * SmemS::kStage + 3 * SmemS::kTileIO);
    float* tab = tab_at(k);
#pragma unroll
    for (int rep = 0; rep < 256 / kThr; ++rep) {
      const int job = tid + rep * kThr;
      const int arr = (job >> 4) & 1;
      const int n = job & 15;
      const int c = job >> 5;
      if (arr == 1 && kMode != kMain) continue;
      float vals[8];
      if (n < p.N) {
        unpack_chunk(lds128(src + arr * SmemS::kTileBC + n * kRow + ((c ^ (n & 7)) << 4)), vals, __nv_bfloat16());
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) vals[j] = 0.0f;
      }
      const float scale = arr == 0 ? kLn2 : 1.0f;
#pragma unroll
      for (int j = 0; j < 8; ++j) tab[(c * 8 + j) * 32 + arr * 16 + n] = vals[j] * scale;
    }
  };

  auto tile_chan = [&](int64_t g, Chan& cc) {
    const int g32 = static_cast<int>(g);
    cc.b = g32 / gpb;
    const int d = (g32 - cc.b * gpb) * kCh + ch;
    cc.valid = d < p.dim;
    cc.d = cc.valid ? d : 0;
    const int64_t arow = static_cast<int64_t>(cc.d) * p.N;
    cc.A0 = p.A[arow];
    bool st_ok = true;
    for (int n = 1; n < p.N; ++n)
      if (p.A[arow + n] != static_cast<float>(n + 1) * cc.A0) st_ok = false;
    cc.structured = __all_sync(0xffffffffu, st_ok) != 0;
    cc.D = p.D ? p.D[cc.d] : 0.0f;
    cc.bias2 = (p.bias ? p.bias[cc.d] : 0.0f) * kLog2e;
  };
  // scalars of chunk c of the tile in the stage whose row starts at urow; sig_prev = σ before it
  auto scalars = [&](ScT& sc, uint32_t urow, int c, const Chan& cc, float sig_prev) {
    if constexpr (kLanes == 1) {
      chunk_scalars<kMode>(sc, urow, c, sw, cc.bias2, cc.D, sig_prev, softplus, has_z);
    } else {
      chunk_scalars2<kMode>(sc, urow, c, sw, pl, cc.bias2, cc.D, cc.structured ? cc.A0 : 1.0f, sig_prev, softplus,
                            has_z);
    }
  };

  // prologue: tile 0's table and channel constants, the first chunk's scalars
  bool ok = mbar_wait_bounded(&full[0], 0u, &g_scaled_status);
  if (ok) widen(0);
  // (gk, tk): tile k; (gn, tn): tile k + 1
  int64_t gk = 0, tk = 0;
  w.at(0, gk, tk);
  Chan cur, nxt;
  tile_chan(gk, cur);
  ScT sc_a, sc_b;   // scalar buffers: sc_a holds the scalars of the next chunk to run
  const uint32_t stage0 = smem_u32(smem);
  scalars(sc_a, stage0 + ch * kRow, 0, cur, 1.0f);

  f2 h[kNs / 2];   // this lane's rescaled states
#pragma unroll
  for (int i = 0; i < kNs / 2; ++i) h[i] = f2_splat(0.0f);
  float lsum = 0.0f;
  int64_t failed_at = -1;

  bool cur_start = true;   // tile k starts a segment
  for (int64_t k = 0; k < ntiles; ++k) {
    const int64_t t = tk;
    int64_t gn = gk, tn = tk;
    w.advance(k, gn, tn);
    const bool tail_start = w.is_tail_start(k);
    if (tail_start && p.sched_balanced && tid == 0) {
      // the state carried in from the previous CTA, which ran the head of this group first
      const unsigned* flag = p.flags + (blockIdx.x - 1);
      const uint64_t limit = p.carry_wait_ns ? p.carry_wait_ns : kWaitNs;
      const uint64_t t0 = globaltimer_ns();
      int got = 0;
      while (true) {
        unsigned v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
        if (v != 0u) { got = 1; break; }
        if (globaltimer_ns() - t0 > limit) break;
        __nanosleep(256);
      }
      if (!got) atomicOr(&g_scaled_status, kStatusTimeout);
      s_carry_ok = got;
    }
    // every thread is done with tile k-1 (its stage and its table); the wait for tile k succeeded
    ok = __syncthreads_and(ok) != 0;
    if (!ok) {
      failed_at = k;
      break;
    }
    if (tid == 0 && issued < ntiles) issue(issued++);   // tile k + kSt - 1 into stage (k - 1) % kSt
    if (k + 1 < ntiles) {
      ok = mbar_wait_bounded(&full[(k + 1) % kSt], static_cast<uint32_t>(((k + 1) / kSt) & 1), &g_scaled_status);
      if (ok) widen(k + 1);
    }
    const bool next_new = k + 1 < ntiles && (gn != gk || w.is_tail_start(k + 1));
    if (next_new) tile_chan(gn, nxt);
    else nxt = cur;

    // ---- segment start: the initial state (σ_init = 1, so g = h)
    const int64_t soff = (static_cast<int64_t>(cur.b) * p.dim + cur.d) * p.N;
    if (cur_start) {
      float init[kNs];
#pragma unroll
      for (int i = 0; i < kNs; ++i) init[i] = 0.0f;
      lsum = 0.0f;
      if (tail_start && p.sched_balanced) {
        if (s_carry_ok) {
          const float4* src = reinterpret_cast<const float4*>(
              p.carry + (static_cast<int64_t>(blockIdx.x) - 1) * kCh * kN + ch * kN + n0);
#pragma unroll
          for (int i = 0; i < kNs / 4; ++i) {
            const float4 v = __ldcg(src + i);
            init[4 * i] = v.x; init[4 * i + 1] = v.y; init[4 * i + 2] = v.z; init[4 * i + 3] = v.w;
          }
        }
      } else if (tail_start && p.h_in != nullptr) {
        const float* src = static_cast<const float*>(p.h_in) + chunk_idx * p.h_in_chunk_stride + soff;
#pragma unroll
        for (int i = 0; i < kNs; ++i)
          if (n0 + i < p.N) init[i] = src[n0 + i];
      } else if (p.h0 != nullptr && t == 0) {
#pragma unroll
        for (int i = 0; i < kNs; ++i)
          if (n0 + i < p.N) init[i] = p.h0[soff + n0 + i];
      }
#pragma unroll
      for (int i = 0; i < kNs / 2; ++i) h[i] = f2_make(init[2 * i], init[2 * i + 1]);
    }

    // ---- the tile's chunks; chunk c's scalars were computed during chunk c - 1
    const int64_t t0 = t * kT;
    const int nch = static_cast<int>(((p.L - t0 < kT) ? (p.L - t0) : kT) / kC);
    const uint32_t urow = smem_u32(smem + (k % kSt) * SmemS::kStage) + ch * kRow;
    const uint32_t urow_next = smem_u32(smem + ((k + 1) % kSt) * SmemS::kStage) + ch * kRow;
    const uint32_t tab = smem_u32(tab_at(k));
    __nv_bfloat16* yrow = nullptr;
    if (kMode == kMain && cur.valid)
      yrow = static_cast<__nv_bfloat16*>(p.y) + (static_cast<int64_t>(cur.b) * p.dim + cur.d) * p.L + t0;
    const float* Arow = p.A + static_cast<int64_t>(cur.d) * p.N;
    const float kb = static_cast<float>(8 * pl + 1);
    float sig_end = 1.0f;
    // Chunks in pairs with two scalar buffers (the tile's chunk count is even): chunk c runs on the
    // buffer filled during chunk c - 1, and the other buffer takes chunk c + 1 (or the next tile's
    // first chunk), so no scalar set is copied.
    auto chunks = [&](auto tag) {
      constexpr bool kS = decltype(tag)::value;
      auto one = [&](ScT& run_sc, ScT& fill_sc, int c) {
        // the next chunk's scalars: chunk c + 1 of this tile or chunk 0 of the next tile, chosen by
        // selects so that they share one basic block with this chunk's recurrence (past the last
        // tile they are computed from a stale stage and never used)
        const bool in_tile = c + 1 < nch;
#if !SSM_SCALED_SCALARS_AFTER
        scalars(fill_sc, in_tile ? urow : urow_next, in_tile ? c + 1 : 0, in_tile ? cur : nxt,
                (in_tile || !next_new) ? run_sc.sig : 1.0f);
#endif
        if constexpr (kLanes == 1) {
          const uint4 yv = chunk_run<kMode, kS>(h, run_sc, tab + c * kC * 128, cur, Arow, p.N);
          if (kMode == kMain && yrow) {
            if (kC == 8) *reinterpret_cast<uint4*>(yrow + c * kC) = yv;
            else *reinterpret_cast<uint2*>(yrow + c * kC) = make_uint2(yv.x, yv.y);
          }
        } else {
          const uint2 yv = chunk_run2<kMode, kS>(h, run_sc, tab + c * kC * 128, pl, kb, Arow, p.N);
          if (kMode == kMain && yrow) *reinterpret_cast<uint2*>(yrow + c * kC + 4 * pl) = yv;
        }
#if SSM_SCALED_SCALARS_AFTER
        scalars(fill_sc, in_tile ? urow : urow_next, in_tile ? c + 1 : 0, in_tile ? cur : nxt,
                (in_tile || !next_new) ? run_sc.sig : 1.0f);
#endif
        if (kMode == kAgg) lsum += run_sc.lsum;
        sig_end = run_sc.sig;
      };
      for (int c = 0; c < nch; c += 2) {
        one(sc_a, sc_b, c);
        one(sc_b, sc_a, c + 1);
      }
    };
    if (cur.structured) chunks(std::true_type());
    else chunks(std::false_type());

    // ---- segment end: h = σ_last·g
    const bool seg_end = (k + 1 == ntiles) || next_new;
    if (seg_end) {
      float hv[kNs];
#pragma unroll
      for (int i = 0; i < kNs / 2; ++i) {
        const f2 v = f2_mul(f2_splat(sig_end), h[i]);
        hv[2 * i] = f2_lo(v);
        hv[2 * i + 1] = f2_hi(v);
      }
      if (p.sched_balanced && k == w.n_head - 1) {
        // publish the state at the end of the head for the next CTA, once every thread has
        // written its part
        float4* dst = reinterpret_cast<float4*>(p.carry + static_cast<int64_t>(blockIdx.x) * kCh * kN + ch * kN + n0);
#pragma unroll
        for (int i = 0; i < kNs / 4; ++i) dst[i] = make_float4(hv[4 * i], hv[4 * i + 1], hv[4 * i + 2], hv[4 * i + 3]);
        __syncthreads();
        if (tid == 0 && static_cast<int>(blockIdx.x) != p.test_withhold_cta) {
          __threadfence();
          asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p.flags + blockIdx.x), "r"(1u) : "memory");
        }
      } else if (kMode == kMain && t == Lt - 1 && cur.valid && p.last_state) {
#pragma unroll
        for (int i = 0; i < kNs; ++i)
          if (n0 + i < p.N) p.last_state[soff + n0 + i] = hv[i];
      }
      if (kMode == kAgg && !p.sched_balanced) {
        // aggregate of this chunk: P = exp(A ΣΔ) = 2^(A Σℓ), Q = h_end from a zero state
        float ls = lsum;
        if (kLanes == 2) ls += __shfl_xor_sync(0xffffffffu, ls, 1);
        if (cur.valid) {
          const int64_t cbase = chunk_idx * p.h_in_chunk_stride + soff;
          float* Pa = static_cast<float*>(p.agg_P);
          float* Qa = static_cast<float*>(p.agg_Q);
#pragma unroll
          for (int i = 0; i < kNs; ++i) {
            if (n0 + i < p.N) {
              Pa[cbase + n0 + i] = ex2_approx(p.A[static_cast<int64_t>(cur.d) * p.N + n0 + i] * ls);
              Qa[cbase + n0 + i] = hv[i];
            }
          }
        }
      }
    }
    cur = nxt;
    cur_start = next_new;
    gk = gn;
    tk = tn;
  }

  if (failed_at >= 0 && tid == 0) {
    // a wait gave up: wait (bounded) for this CTA's copies still in flight, then leave
    for (int64_t k = failed_at; k < issued; ++k)
      (void)mbar_wait_bounded(&full[k % kSt], static_cast<uint32_t>((k / kSt) & 1), &g_scaled_status, 100000000ull);
  }
}

}  // namespace

int scaled_channels_per_cta() { return kCh; }

int scaled_resident_ctas() {
  static int cached[64] = {0};
  int occ = 0, dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return 0; }
  if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) { cudaGetLastError(); return 0; }
  auto kern = scan_scaled_kernel<kMain, kLanesDefault>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SmemS::kTotal) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kCh * kLanesDefault, SmemS::kTotal) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  if (dev >= 0 && dev < 64) cached[dev] = occ * sms;
  return occ * sms;
}

cudaError_t scaled_status_read_and_clear(unsigned int* out) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_scaled_status, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_scaled_status, &zero, sizeof(unsigned int));
}

cudaError_t scan_scaled_launch(const ScanParams& p, int nchunks, int balanced_ctas, cudaStream_t stream, char* err,
                               size_t errlen) {
  MapsS tm;
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
  auto kmain = scan_scaled_kernel<kMain, kLanesDefault>;
  auto kagg = scan_scaled_kernel<kAgg, kLanesDefault>;
  constexpr int kThreads = kCh * kLanesDefault;
  cudaError_t e;
  e = cudaFuncSetAttribute(kmain, cudaFuncAttributeMaxDynamicSharedMemorySize, SmemS::kTotal);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kagg, cudaFuncAttributeMaxDynamicSharedMemorySize, SmemS::kTotal);
  if (e != cudaSuccess) return e;
  if (balanced_ctas > 0) {
    e = cudaMemsetAsync(p.flags, 0, sizeof(unsigned) * balanced_ctas, stream);
    if (e != cudaSuccess) return e;
    void* args[] = {const_cast<MapsS*>(&tm), const_cast<ScanParams*>(&p)};
    return cudaLaunchCooperativeKernel(reinterpret_cast<void*>(kmain), dim3(balanced_ctas), dim3(kThreads), args,
                                       SmemS::kTotal, stream);
  }
  if (nchunks > 1) {
    ScanParams pa = p;
    pa.h_in = nullptr;
    pa.h0 = nullptr;
    kagg<<<dim3(groups, nchunks - 1), kThreads, SmemS::kTotal, stream>>>(tm, pa);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = carry_launch_f32(p, nchunks, stream);
    if (e != cudaSuccess) return e;
  }
  kmain<<<dim3(groups, nchunks), kThreads, SmemS::kTotal, stream>>>(tm, p);
  return cudaGetLastError();
}

}  // namespace ssm
