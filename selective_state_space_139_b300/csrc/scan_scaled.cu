// Prefill selective scan on a rescaled state: bf16 io, two lanes per channel, sm_103a.
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
// ρ_t r.  A segment starts from g = h_init (σ_init = 1) and ends with h = σ_last·g.  |σ_t| below 1e-20
// (u_t = 0, or Δ_t underflowing to 0) is replaced by 1e-20, which adds at most 1e-20·ln2·|B_t| to the
// state where the exact input term is smaller than that.
//
// Exact zero-order hold ("Модуль 8", §4: the input term (exp(ΔA) - 1)/A · B u).  With
// A[d,n] = (n+1)·A[d,0] and a_n = exp(Δ_t A[d,n]) the input term is (a_n - 1)·B̃_n·u_t/A[d,0] with
// B̃_n = B_t[n]/(n+1), so the kernel takes σ_t = -u_t/A[d,0] and carries k_t = h_t/σ_t:
//   k_t = a_n ρ_t k_{t-1} + (1 - a_n) B̃_n = B̃_n - a_n·(B̃_n - ρ_t k_{t-1}),
// two FMAs per state whose addend is the same table value B̃_n (the table holds B/(n+1) instead of
// ln2·B; ρ_t and the decay powers are kept negated so that neither FMA needs a sign change).  The
// readout and the segment ends are those of the Δ·B form.  Warps whose A is not of that form, or
// whose A[d,0] is 0, carry g_t = h_t/u_t with one input coefficient per state,
// (n+1)(a_n - 1)/A[d,n], or its series in Δ A[d,n] where |Δ A[d,n]| < 1/32 (the A -> 0 limit Δ·B
// included).
//
// Layout of the work:
//  * A CTA is 256 threads and owns 128 consecutive channels of one batch row (a "group"), one CTA
//    per SM.  Two adjacent lanes share a channel: lane p holds the states n = p, p+2, .., p+14 (its
//    k-th value is state p + 2k) as four packed f32x2 pairs, so that both lanes' decays are ρ r^(p+1)
//    times powers of r^2 and need the same two numbers per step, r and ρ.
//  * u, Δ_raw, z tiles [128 channels x 64 steps] and B, C tiles [dstate x 64 steps] arrive by TMA
//    with a 128-byte swizzle through a 4-stage mbarrier pipeline.  At the start of tile k the CTA
//    widens tile k+1's B and C into a float32 table [step][ln2·B | C], each half with the even states
//    first and the odd states after, read by the two lanes of a channel with 128-bit loads.
//  * Steps are processed in chunks of 8.  Lane p owns steps 4p..4p+3 of each chunk: it computes their
//    scalars (ℓ, r or ℓ, σ, ρ, σ·SiLU(z), D u·SiLU(z)) one chunk ahead, in phases placed between the
//    steps of the current chunk's recurrence so that their load and MUFU chains overlap it; r and ρ
//    reach both lanes by shuffles; each step's readout is the sum of the two lanes' halves, and the
//    owner of the step finishes, rounds and stores it.
//  * Scheduling: the balanced persistent schedule or the grid schedule of scan_walk.cuh, with the
//    CTA-to-CTA carry of the balanced schedule behind a bounded wait.
//  * Aggregate mode (chunked schedule): per (group, chunk) from a zero state, the chunk's decay
//    product exp(A ΣΔ) and end state, for the carry pass ("Модуль 8", §7).
#include <cstring>
#include <type_traits>

#include "internal.h"
#include "scan_walk.cuh"
#include "ssm_device.cuh"

namespace ssm {
namespace {

__device__ unsigned int g_scaled_status = 0;

constexpr int kCh = 128;        // channels per CTA
constexpr int kThreads = 256;   // two lanes per channel
constexpr int kT = 64;          // steps per tile
constexpr int kC = 8;           // steps per chunk
constexpr int kSt = 4;          // TMA stages
constexpr int kRow = 128;       // bytes of one tile row (64 bf16 steps)
constexpr int kN = 16;          // state width
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

// Scalars of one 8-step chunk as one lane sees them.
struct Sc {
  float q[8];      // per step: r = 2^(ℓ·A[d,0]) (A[d,n] = (n+1)·A[d,0]) or ℓ (other A)
  float rho[8];    // per step: σ_{t-1}/σ_t (exact-ZOH mode: -σ_{t-1}/σ_t)
  f2 al[2];        // own steps: σ_t·SiLU(z_t)
  f2 be[2];        // own steps: D·u_t·SiLU(z_t)
  float sig;       // σ of the chunk's last step (both lanes)
  float lsum;      // Σ ℓ over the own steps (aggregate mode)
};

// Per-channel constants of a segment.
struct Chan {
  float bias2;   // bias·log2(e)
  float D;
  float A0;      // A[d,0]
  float sA;      // exact-ZOH mode: σ_t = sA·u_t (-1/A[d,0] for structured warps, 1 otherwise)
  int b, d;
  bool valid;
  bool structured;   // warp-uniform: every channel of the warp has A[d,n] = (n+1)·A[d,0]
};

__device__ __forceinline__ float pick(f2 v, int j) { return (j & 1) ? f2_hi(v) : f2_lo(v); }

// The scalars of a chunk (a lane's own steps 4p..4p+3, read from its channel's row of the stage),
// computed in phases: load, then for each own step pair softplus and σ (a, b), the gate (gate), and
// the exchange of r and ρ between the two lanes (exchange).
template <int kMode, bool kZoh>
struct Phases {
  uint32_t uu[2], dd[2], zz[2];
  f2 x[2], l2v[2], u2v[2];
  float qo[4], sg[4], rs[4];
  float lsum = 0.0f;

  __device__ __forceinline__ void load(uint32_t urow, int c, int sw, int pl, bool has_z) {
    const uint32_t off = static_cast<uint32_t>((c ^ sw) << 4) + 8u * pl;   // own 4 steps: 8 bytes of the unit
    const uint2 uw = lds64(urow + off);
    const uint2 dw = lds64(urow + SmemS::kTileIO + off);
    uint2 zw = make_uint2(0u, 0u);
    if (kMode == kMain && has_z) zw = lds64(urow + 2 * SmemS::kTileIO + off);
    uu[0] = uw.x; uu[1] = uw.y; dd[0] = dw.x; dd[1] = dw.y; zz[0] = zw.x; zz[1] = zw.y;
  }
  // (Δ_raw + bias)·log2(e), and 1 + 2^x for the softplus
  __device__ __forceinline__ void a(int q, float bias2, bool softplus) {
    u2v[q] = f2_make(bf16lo_to_f32(uu[q]), bf16hi_to_f32(uu[q]));
    const f2 v2 = f2_make(bf16lo_to_f32(dd[q]), bf16hi_to_f32(dd[q]));
    x[q] = f2_fma(v2, f2_splat(kLog2e), f2_splat(bias2));
    l2v[q] = x[q];
    if (softplus) {
      const f2 e = f2_make(ex2_approx(fminf(f2_lo(x[q]), 64.0f)), ex2_approx(fminf(f2_hi(x[q]), 64.0f)));
      l2v[q] = f2_add(e, f2_splat(1.0f));
    }
  }
  // ℓ = log2(1 + 2^x) = softplus(v)/ln2 (max(., x) covers x > 64, where 2^x is clamped), r, σ, 1/σ
  __device__ __forceinline__ void b(int q, float A0, float sA, bool structured, bool softplus) {
    f2 l2 = l2v[q];
    if (softplus)
      l2 = f2_make(fmaxf(lg2_approx(f2_lo(l2)), f2_lo(x[q])), fmaxf(lg2_approx(f2_hi(l2)), f2_hi(x[q])));
    if (kMode == kAgg) lsum += f2_lo(l2) + f2_hi(l2);
    const f2 qq = f2_mul(l2, f2_splat(A0));
    qo[2 * q] = structured ? ex2_approx(f2_lo(qq)) : f2_lo(l2);
    qo[2 * q + 1] = structured ? ex2_approx(f2_hi(qq)) : f2_hi(l2);
    const f2 sgm = kZoh ? f2_mul(u2v[q], f2_splat(sA)) : f2_mul(l2, u2v[q]);
    float s0 = f2_lo(sgm), s1 = f2_hi(sgm);
    s0 = fabsf(s0) < kSigmaMin ? kSigmaMin : s0;
    s1 = fabsf(s1) < kSigmaMin ? kSigmaMin : s1;
    sg[2 * q] = s0;
    sg[2 * q + 1] = s1;
    rs[2 * q] = rcp_approx(s0);
    rs[2 * q + 1] = rcp_approx(s1);
  }
  // σ·SiLU(z) and D·u·SiLU(z)
  __device__ __forceinline__ void gate(int q, Sc& ns, float D, bool has_z) {
    if (kMode != kMain) return;
    f2 g = f2_splat(1.0f);
    if (has_z) {
      const f2 z2 = f2_make(bf16lo_to_f32(zz[q]), bf16hi_to_f32(zz[q]));
      const f2 t = f2_mul(z2, f2_splat(-kLog2e));
      const f2 den = f2_add(f2_make(ex2_approx(f2_lo(t)), ex2_approx(f2_hi(t))), f2_splat(1.0f));
      g = f2_mul(z2, f2_make(rcp_approx(f2_lo(den)), rcp_approx(f2_hi(den))));
    }
    ns.al[q] = f2_mul(f2_make(sg[2 * q], sg[2 * q + 1]), g);
    ns.be[q] = f2_mul(f2_mul(f2_splat(D), u2v[q]), g);
  }
  // ρ of the own steps and the exchange: σ before the first own step is, for lane 1, step 3 from
  // lane 0 and, for lane 0, the previous chunk's step 7 (sig_prev); then r and ρ of every step reach
  // both lanes from the step's owner
  __device__ __forceinline__ void exchange(Sc& ns, int pl, float sig_prev) {
    const float s3x = __shfl_xor_sync(0xffffffffu, sg[3], 1);
    const float first_prev = pl ? s3x : sig_prev;
    float ro[4];
    ro[0] = first_prev * rs[0];
    ro[1] = sg[0] * rs[1];
    ro[2] = sg[1] * rs[2];
    ro[3] = sg[2] * rs[3];
    if (kZoh) {
#pragma unroll
      for (int i = 0; i < 4; ++i) ro[i] = -ro[i];
    }
    ns.sig = pl ? sg[3] : s3x;
    const int base = (threadIdx.x & 31) & ~1;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      ns.q[j] = __shfl_sync(0xffffffffu, qo[j & 3], base | (j >> 2));
      ns.rho[j] = __shfl_sync(0xffffffffu, ro[j & 3], base | (j >> 2));
    }
    ns.lsum = lsum;
  }
};

// One 8-step chunk of one lane: the recurrence of the current chunk (scalars in s) with the next
// chunk's scalars computed into ns in phases placed between the steps, so that their load and MUFU
// chains overlap the state updates (0.381 ms against 0.403 ms with the scalars computed as one block
// on the 2.8B layer).  urow, c, sig_prev and the channel constants describe the next chunk.  Returns
// the lane's four own outputs packed as bf16 (main mode).
template <int kMode, bool kS, bool kZoh>
__device__ __forceinline__ uint2 chunk_step(f2 (&h)[4], const Sc& s, Sc& ns, uint32_t tab, int pl,
                                            const float (&Ah)[8], const float (&Wz)[8], uint32_t urow, int c,
                                            int sw, float bias2, float D, float A0, float sA, bool structured,
                                            float sig_prev, bool softplus, bool has_z) {
  Phases<kMode, kZoh> ph;
  ph.load(urow, c, sw, pl, has_z);
  float part[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float q = s.q[j];
    const float rho = s.rho[j];
    const uint32_t row = tab + j * 128 + pl * 32;
    f2 a[4];
    if (kS) {
      const float r = q;
      const float r2 = r * r, r4 = r2 * r2;
      // Δ·B: ρ r^(p+1+2k), k = 0..7.  Exact ZOH: -r^(p+1+2k) (ρ enters through t below)
      const float c0 = kZoh ? -(pl ? r2 : r) : rho * (pl ? r2 : r);
      a[0] = f2_make(c0, c0 * r2);
      const f2 R4 = f2_splat(r4);   // one splat: the pairs are a[0]·(r^4)^i
      a[1] = f2_mul(a[0], R4);
      a[2] = f2_mul(a[1], R4);
      a[3] = f2_mul(a[2], R4);
    } else if (!kZoh) {
      const f2 q2 = f2_splat(q);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const f2 x = f2_mul(q2, f2_make(Ah[2 * i], Ah[2 * i + 1]));
        a[i] = f2_make(rho * ex2_approx(f2_lo(x)), rho * ex2_approx(f2_hi(x)));
      }
    }
    const float4 b0 = lds128f(row), b1 = lds128f(row + 16);
    const f2 bt[4] = {f2_make(b0.x, b0.y), f2_make(b0.z, b0.w), f2_make(b1.x, b1.y), f2_make(b1.z, b1.w)};
    if (!kZoh) {
#pragma unroll
      for (int i = 0; i < 4; ++i) h[i] = f2_fma(a[i], h[i], bt[i]);
    } else if (kS) {
      // k_t = B̃ - a·(B̃ - ρ k_{t-1}) with rho = -ρ, a[i] = -a
#pragma unroll
      for (int i = 0; i < 4; ++i) h[i] = f2_fma(a[i], f2_fma(f2_splat(rho), h[i], bt[i]), bt[i]);
    } else {
      // exact ZOH, any A: g_t = ρ e g_{t-1} + m B̃ with e = 2^(ℓ A[d,n]) = exp(y), y = Δ A[d,n], and
      // m = (n+1)(e - 1)/A[d,n] = Wz·(e - 1), e - 1 taken from its series y(1 + y/2 + y²/6 + y³/24)
      // where |y| < 1/32, free of the cancellation in e - 1.  |A[d,n]| < 2^-60 (zero or denormal,
      // where 1/A would overflow) is held as 2^-60 (Ah, Wz): the series then gives m = (n+1)·Δ, the
      // A -> 0 limit, and e = 1, both exact to float32 precision.
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const f2 x = f2_mul(f2_splat(q), f2_make(Ah[2 * i], Ah[2 * i + 1]));
        const f2 e = f2_make(ex2_approx(f2_lo(x)), ex2_approx(f2_hi(x)));
        const f2 y = f2_mul(x, f2_splat(kLn2));
        const f2 poly = f2_mul(y, f2_fma(y, f2_fma(y, f2_fma(y, f2_splat(1.0f / 24.0f), f2_splat(1.0f / 6.0f)),
                                                       f2_splat(0.5f)), f2_splat(1.0f)));
        const f2 em = f2_add(e, f2_splat(-1.0f));
        const f2 em1 = f2_make(fabsf(f2_lo(y)) < 0.03125f ? f2_lo(poly) : f2_lo(em),
                               fabsf(f2_hi(y)) < 0.03125f ? f2_hi(poly) : f2_hi(em));
        const f2 m = f2_mul(em1, f2_make(Wz[2 * i], Wz[2 * i + 1]));
        h[i] = f2_fma(f2_mul(f2_splat(-rho), e), h[i], f2_mul(m, bt[i]));   // rho = -ρ
      }
    }
    if (kMode == kMain) {
      const float4 c0v = lds128f(row + 64), c1v = lds128f(row + 80);
      f2 acc = f2_mul(f2_make(c0v.x, c0v.y), h[0]);
      acc = f2_fma(f2_make(c0v.z, c0v.w), h[1], acc);
      acc = f2_fma(f2_make(c1v.x, c1v.y), h[2], acc);
      acc = f2_fma(f2_make(c1v.z, c1v.w), h[3], acc);
      part[j] = f2_lo(acc) + f2_hi(acc);
    }
    // a phase of the next chunk's scalars
    if (j == 0 || j == 2) ph.a(j >> 1, bias2, softplus);
    if (j == 1 || j == 3) ph.b(j >> 1, A0, sA, structured, softplus);
    if (j == 4 || j == 5) ph.gate(j - 4, ns, D, has_z);
    if (j == 6) ph.exchange(ns, pl, sig_prev);
  }
  if constexpr (kMode != kMain) {
    return make_uint2(0u, 0u);
  } else {
    // lane p finishes steps 4p..4p+3: its half plus the partner's half
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
}

// The scalars of a chunk on their own (the first chunk of a CTA's walk).
template <int kMode, bool kZoh>
__device__ __forceinline__ void chunk_scalars(Sc& ns, uint32_t urow, int c, int sw, int pl, float bias2, float D,
                                              float A0, float sA, bool structured, float sig_prev, bool softplus,
                                              bool has_z) {
  Phases<kMode, kZoh> ph;
  ph.load(urow, c, sw, pl, has_z);
  ph.a(0, bias2, softplus);
  ph.a(1, bias2, softplus);
  ph.b(0, A0, sA, structured, softplus);
  ph.b(1, A0, sA, structured, softplus);
  ph.gate(0, ns, D, has_z);
  ph.gate(1, ns, D, has_z);
  ph.exchange(ns, pl, sig_prev);
}

// kZ (a gate z is given) and kSp (softplus on Δ) are template parameters rather than run-time flags:
// tested at run time they split each chunk's body into basic blocks that the compiler does not
// schedule across, and the next chunk's scalar phases stop overlapping the recurrence (0.369 ms
// against 0.335 ms on the 2.8B layer).
template <int kMode, bool kZoh, bool kZ, bool kSp>
__global__ void __launch_bounds__(kThreads, 1) scan_scaled_kernel(const __grid_constant__ MapsS tm, const ScanParams p) {
  constexpr int kNs = kN / 2;     // states per lane
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // table of tile k: tab_at(k)
  auto tab_at = [&](int64_t k) { return reinterpret_cast<float*>(smem + kSt * SmemS::kStage + (k & 1) * SmemS::kTab); };
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + SmemS::kBars);
  __shared__ int s_carry_ok;

  const int tid = threadIdx.x;
  const int ch = tid >> 1;                         // channel within the group
  const int pl = tid & 1;                          // lane within the channel
  auto sidx = [&](int k) { return pl + 2 * k; };   // this lane's k-th state
  const int n0 = pl * kNs;                         // this lane's slot in a CTA-to-CTA carry row
  const int sw = ch & 7;                           // 128-byte swizzle of this channel's tile row
  const int64_t Lt = (p.L + kT - 1) / kT;
  const int gpb = (p.dim + kCh - 1) / kCh;         // groups per batch row
  constexpr bool has_z = kMode == kMain && kZ;
  constexpr bool softplus = kSp;
  // buffer sizes (elements) for the index checks of checked builds
  const int64_t nA = static_cast<int64_t>(p.dim) * p.N;
  const int64_t nState = static_cast<int64_t>(p.batch) * p.dim * p.N;
  const int64_t nIO = static_cast<int64_t>(p.batch) * p.dim * p.L;
  const int64_t nCarry = static_cast<int64_t>(gridDim.x) * kCh * kN;

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

  // Widens tile k's B and C (stage k % kSt) into table k & 1: ln2·B (exact-ZOH mode: B/(n+1)) in
  // columns 0..15, C in 16..31, zero rows for n >= dstate.  256 jobs (array, n, 8-step chunk), one per thread; a warp's 32
  // threads store 32 consecutive words.
  auto widen = [&](int64_t k) {
    const uint32_t src = smem_u32(smem + (k % kSt) * SmemS::kStage + 3 * SmemS::kTileIO);
    float* tab = tab_at(k);
    {
      const int job = tid;
      const int arr = (job >> 4) & 1;
      const int n = job & 15;
      const int c = job >> 5;
      float vals[8];
      if (n < p.N && (arr == 0 || kMode == kMain)) {
        unpack_chunk(lds128(src + arr * SmemS::kTileBC + n * kRow + ((c ^ (n & 7)) << 4)), vals, __nv_bfloat16());
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) vals[j] = 0.0f;
      }
      const float scale = arr == 0 ? (kZoh ? 1.0f / static_cast<float>(n + 1) : kLn2) : 1.0f;
      // even states in columns 0..7 of each half, odd states in 8..15 (one block per lane)
      const int col = (n & 1) * 8 + (n >> 1);
#pragma unroll
      for (int j = 0; j < 8; ++j) tab[(c * 8 + j) * 32 + arr * 16 + col] = vals[j] * scale;
    }
  };

  auto tile_chan = [&](int64_t g, Chan& cc) {
    const int g32 = static_cast<int>(g);
    cc.b = g32 / gpb;
    const int d = (g32 - cc.b * gpb) * kCh + ch;
    cc.valid = d < p.dim;
    cc.d = cc.valid ? d : 0;
    const int64_t arow = static_cast<int64_t>(cc.d) * p.N;
    cc.A0 = *checked(p.A, arow, nA);
    // exact ZOH divides by A[d,0]: a row with |A[d,0]| < 2^-60 (zero or denormal, where 1/A would
    // overflow) takes the per-state path, which has the A -> 0 limit
    bool st_ok = !kZoh || fabsf(cc.A0) >= 0x1p-60f;
    for (int n = 1; n < p.N; ++n)
      if (*checked(p.A, arow + n, nA) != static_cast<float>(n + 1) * cc.A0) st_ok = false;
    cc.structured = __all_sync(0xffffffffu, st_ok) != 0;
    cc.sA = kZoh && cc.structured ? -1.0f / cc.A0 : 1.0f;
    cc.D = p.D ? *checked(p.D, cc.d, p.dim) : 0.0f;
    cc.bias2 = (p.bias ? *checked(p.bias, cc.d, p.dim) : 0.0f) * kLog2e;
  };
  // prologue: tile 0's table and channel constants, the first chunk's scalars
  bool ok = mbar_wait_bounded(&full[0], 0u, &g_scaled_status);
  if (ok) widen(0);
  // (gk, tk): tile k; (gn, tn): tile k + 1
  int64_t gk = 0, tk = 0;
  w.at(0, gk, tk);
  Chan cur, nxt;
  tile_chan(gk, cur);
  Sc sc_a, sc_b;   // scalar buffers: sc_a holds the scalars of the next chunk to run
  chunk_scalars<kMode, kZoh>(sc_a, smem_u32(smem) + ch * kRow, 0, sw, pl, cur.bias2, cur.D, cur.A0, cur.sA,
                             cur.structured, 1.0f, softplus, has_z);

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
      const unsigned* flag = checked(p.flags, static_cast<int64_t>(blockIdx.x) - 1, gridDim.x);
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
              checked(p.carry, (static_cast<int64_t>(blockIdx.x) - 1) * kCh * kN + ch * kN + n0, nCarry, 8));
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
          if (sidx(i) < p.N)
            init[i] = *checked(src, sidx(i), (static_cast<int64_t>(gridDim.y) - chunk_idx) * p.h_in_chunk_stride - soff);
      } else if (p.h0 != nullptr && t == 0) {
#pragma unroll
        for (int i = 0; i < kNs; ++i)
          if (sidx(i) < p.N) init[i] = *checked(p.h0, soff + sidx(i), nState);
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
      yrow = checked(static_cast<__nv_bfloat16*>(p.y), (static_cast<int64_t>(cur.b) * p.dim + cur.d) * p.L + t0, nIO,
                     nch * kC);
    float sig_end = 1.0f;
    // Chunks in pairs with two scalar buffers: chunk c runs on the buffer filled during chunk c - 1,
    // and the other buffer takes chunk c + 1 (or the next tile's first chunk), so no scalar set is
    // copied.  A tile with an odd chunk count (the last tile when L is an odd multiple of 8) ends
    // with one chunk on sc_a and a copy back into sc_a.
    auto chunks = [&](auto tag) {
      constexpr bool kS = decltype(tag)::value;
      float Ah[8];   // this lane's row of A (A not of the form (n+1)·A[d,0])
      float Wz[8];   // exact-ZOH mode: (n+1)/A[d,n], with |A[d,n]| < 2^-60 held as 2^-60 in Ah and Wz
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        Ah[i] = (!kS && sidx(i) < p.N) ? *checked(p.A, static_cast<int64_t>(cur.d) * p.N + sidx(i), nA) : 0.0f;
        if (kZoh && fabsf(Ah[i]) < 0x1p-60f) Ah[i] = 0x1p-60f;   // same decay and limit to float32 precision
        Wz[i] = (!kS && kZoh) ? static_cast<float>(sidx(i) + 1) / Ah[i] : 0.0f;
      }
      auto one = [&](Sc& run_sc, Sc& fill_sc, int c) {
        // the next chunk's scalars: chunk c + 1 of this tile or chunk 0 of the next tile, chosen by
        // selects so that they share one basic block with this chunk's recurrence (past the last
        // tile they are computed from a stale stage and never used)
        const bool in_tile = c + 1 < nch;
        const Chan& cc = in_tile ? cur : nxt;
        const uint2 yv = chunk_step<kMode, kS, kZoh>(h, run_sc, fill_sc, tab + c * kC * 128, pl, Ah, Wz,
                                                     in_tile ? urow : urow_next, in_tile ? c + 1 : 0, sw, cc.bias2,
                                                     cc.D, cc.A0, cc.sA, cc.structured,
                                                     (in_tile || !next_new) ? run_sc.sig : 1.0f, softplus, has_z);
        if (kMode == kMain && yrow) *reinterpret_cast<uint2*>(yrow + c * kC + 4 * pl) = yv;
        if (kMode == kAgg) lsum += run_sc.lsum;
        sig_end = run_sc.sig;
      };
      int c = 0;
      for (; c + 1 < nch; c += 2) {
        one(sc_a, sc_b, c);
        one(sc_b, sc_a, c + 1);
      }
      if (c < nch) {
        one(sc_a, sc_b, c);
        sc_a = sc_b;
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
        float4* dst = reinterpret_cast<float4*>(
            checked(p.carry, static_cast<int64_t>(blockIdx.x) * kCh * kN + ch * kN + n0, nCarry, 8));
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
          if (sidx(i) < p.N) *checked(p.last_state, soff + sidx(i), nState) = hv[i];
      }
      if (kMode == kAgg && !p.sched_balanced) {
        // aggregate of this chunk: P = exp(A ΣΔ) = 2^(A Σℓ), Q = h_end from a zero state
        float ls = lsum;
        ls += __shfl_xor_sync(0xffffffffu, ls, 1);
        if (cur.valid) {
          const int64_t cbase = chunk_idx * p.h_in_chunk_stride + soff;
          float* Pa = static_cast<float*>(p.agg_P);
          float* Qa = static_cast<float*>(p.agg_Q);
#pragma unroll
          for (int i = 0; i < kNs; ++i) {
            if (sidx(i) < p.N) {
              const int64_t nAgg = static_cast<int64_t>(gridDim.y) * p.h_in_chunk_stride;
              *checked(Pa, cbase + sidx(i), nAgg) = ex2_approx(*checked(p.A, static_cast<int64_t>(cur.d) * p.N + sidx(i), nA) * ls);
              *checked(Qa, cbase + sidx(i), nAgg) = hv[i];
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

using ScaledKernel = void (*)(MapsS, ScanParams);

template <int kMode, bool kZoh, bool kZ>
ScaledKernel pick_sp(bool sp) {
  return sp ? scan_scaled_kernel<kMode, kZoh, kZ, true> : scan_scaled_kernel<kMode, kZoh, kZ, false>;
}

// The instance for these parameters (the aggregate pass reads no z).
template <int kMode>
ScaledKernel pick_kernel(const ScanParams& p) {
  const bool z = kMode == kMain && p.z != nullptr;
  const bool sp = p.softplus != 0;
  if (p.disc == 1) return z ? pick_sp<kMode, true, kMode == kMain>(sp) : pick_sp<kMode, true, false>(sp);
  return z ? pick_sp<kMode, false, kMode == kMain>(sp) : pick_sp<kMode, false, false>(sp);
}

}  // namespace

int scaled_channels_per_cta() { return kCh; }

int scaled_resident_ctas() {
  static int cached[64] = {0};
  int occ = 0, dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return 0; }
  if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) { cudaGetLastError(); return 0; }
  auto kern = scan_scaled_kernel<kMain, false, true, true>;   // every instance has the same shared memory
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SmemS::kTotal) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kThreads, SmemS::kTotal) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  if (dev >= 0 && dev < 64) cached[dev] = occ * sms;
  return occ * sms;
}

cudaError_t scaled_check_read_and_clear(unsigned int* out) { return tu_check_read_and_clear(out); }

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
  const ScaledKernel kmain = pick_kernel<kMain>(p);
  const ScaledKernel kagg = pick_kernel<kAgg>(p);
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
