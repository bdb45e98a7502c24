// Backward of the selective scan (reverse-mode differentiation of the forward recurrence), with
// the states recomputed from checkpoints instead of stored: the training half of the
// hardware-aware scan that keeps intermediate states out of HBM ("Mamba: линейная альтернатива
// трансформеру", "Почему selectivity ломает старый трюк со свёрткой"; the ai.pinkoculture.com concept
// page, 硬件感知的实现: recomputation to save memory).  The pages give only the forward recurrence;
// the derivatives below are its chain rule.
//
// Forward (per channel): v_t = Δ_raw_t + bias, Δ_t = softplus(v_t), Ā_t = exp(Δ_t A), h_t = Ā_t ⊙ h_{t-1}
// + Δ_t B_t x_t, s_t = C_t·h_t + D x_t, y_t = s_t SiLU(z_t).  Backward from dy:
//   ds_t = dy_t SiLU(z_t);  dz_t = dy_t s_t SiLU'(z_t)
//   dh_t = ds_t C_t + Ā_{t+1} ⊙ dh_{t+1}
//   dC_t = Σ_channels ds_t h_t;  dB_t = Σ_channels dh_t Δ_t x_t
//   dΔ_t = Σ_n dh_{t,n} (h_{t-1,n} Ā_{t,n} A_n + B_{t,n} x_t);  dA_n = Σ_{batch, t} dh_{t,n} h_{t-1,n} Ā_{t,n} Δ_t
//   dx_t = ds_t D + Σ_n dh_{t,n} Δ_t B_{t,n};  dD = Σ ds_t x_t;  dΔ_raw_t = dΔ_t σ(v_t);  dbias = Σ dΔ_raw
//
// Time is cut into chunks so that (channel group, chunk) tiles run in parallel.  Both recurrences are
// affine maps of the state, so a chunk is summarised by three vectors per channel (the same
// composition as the forward's chunked schedule):
//   P = Π_chunk Ā (the decay over the chunk),  Q = the chunk's end state from a zero start,
//   G = Σ_t (Π_{r=chunk start..t} Ā_r) ⊙ C_t ds_t, the gradient reaching the state before the chunk from
//       the chunk's own outputs.
// Three kernels: (1) per tile, a forward pass from a zero state that writes P, Q, G and a
// checkpoint (the local state and the running Σ Δ) every 8 steps; (2) per channel, the carries:
// h_start(c+1) = P_c ⊙ h_start(c) + Q_c forwards, dh_in(c) = G_{c+1} + P_{c+1} ⊙ dh_in(c+1) backwards;
// (3) per tile, the reverse pass: for each 8-step segment from the last, the true state at the
// segment start is the checkpoint plus exp(A Σ Δ) ⊙ h_start, the segment's 8 states are recomputed into
// shared memory (layout [step][state][thread], conflict free), and the 8 steps run backwards starting
// from dh_in.  dB and dC sum over the channels of a batch row: per step a warp transpose-reduces its
// 32 values (16 of dB, 16 of dC), the four warps' partials are added in shared memory and the CTA adds
// them to global memory with vector atomics.  dA, dD and dbias accumulate per thread and are added
// once per tile.  bf16 io computes in float32 with the MUFU approximations of the forward and runs
// (1) and (3) with two lanes per channel ((1') and (3') below: eight states per lane, 64 channels per
// CTA); float32 io computes in double, one channel per thread, and accumulates its cross-channel sums
// in double.
#include <cstring>

#include "internal.h"
#include "ssm_device.cuh"

namespace ssm {
namespace {

#ifndef SSM_BWD_TWO_LANES
#define SSM_BWD_TWO_LANES 1   // bf16 io: local forward and reverse pass with two lanes per channel (1) or one (0)
#endif
#ifndef SSM_BWD_FWD_MINB
#define SSM_BWD_FWD_MINB 3   // resident CTAs per SM the local forward is compiled for (float state)
#endif

constexpr int kThreads = 128;   // channels per CTA
constexpr int kSeg = 8;         // steps per segment (checkpoint interval)
constexpr int kN = 16;
constexpr int kAgg = 3 * kN;    // per (channel, chunk): [Q -> h_start | P | G -> dh_in]

template <typename CT>
struct Smem {
  // B and C of the segment [step][B0..15 | C0..15] (float, two buffers), the recomputed states, the
  // dB/dC partials of the four warps (two buffers) and the chunk start states
  static constexpr int kBC = 2 * kSeg * 32 * 4;
  static constexpr int kH = kSeg * kN * kThreads * static_cast<int>(sizeof(CT));
  static constexpr int kRed = 2 * 4 * kSeg * 32 * static_cast<int>(sizeof(CT));
  static constexpr int kHs = kN * kThreads * static_cast<int>(sizeof(CT));   // chunk start states
  static constexpr int kTotal = kBC + kH + kRed + kHs;
};

template <typename CT>
__device__ __forceinline__ CT sp(CT v) {
  if constexpr (sizeof(CT) == 4) return softplus_fast(v);
  else return v > 0.0 ? v + log1p(exp(-v)) : log1p(exp(v));
}

template <typename CT>
__device__ __forceinline__ CT sigm(CT x) {
  if constexpr (sizeof(CT) == 4) return rcp_approx(1.0f + ex2_approx(-x * kLog2e));
  else return 1.0 / (1.0 + exp(-x));
}

// Two states (n, n+1) of a channel.  float: one packed f32x2 register pair, so elementwise
// arithmetic issues once per pair; double (the float32-io path): two scalars.  The exponent of Ā is
// taken base 2 for float (A pre-scaled by log2 e) and base e for double.
template <typename CT>
struct Pair;

template <>
struct Pair<float> {
  f2 v;
  static constexpr float kExpScale = kLog2e;
  __device__ static Pair make(float lo, float hi) { return {f2_make(lo, hi)}; }
  __device__ static Pair splat(float a) { return {f2_splat(a)}; }
  __device__ static Pair from_f2(f2 a) { return {a}; }
  __device__ float lo() const { return f2_lo(v); }
  __device__ float hi() const { return f2_hi(v); }
};

template <>
struct Pair<double> {
  double a, b;
  static constexpr double kExpScale = 1.0;
  __device__ static Pair make(double lo, double hi) { return {lo, hi}; }
  __device__ static Pair splat(double x) { return {x, x}; }
  __device__ static Pair from_f2(f2 x) { return {f2_lo(x), f2_hi(x)}; }
  __device__ double lo() const { return a; }
  __device__ double hi() const { return b; }
};

__device__ __forceinline__ Pair<float> pmul(Pair<float> x, Pair<float> y) { return {f2_mul(x.v, y.v)}; }
__device__ __forceinline__ Pair<float> pfma(Pair<float> x, Pair<float> y, Pair<float> z) { return {f2_fma(x.v, y.v, z.v)}; }
__device__ __forceinline__ Pair<float> padd(Pair<float> x, Pair<float> y) { return {f2_add(x.v, y.v)}; }
// exp of the pre-scaled exponent: 2^x for float
__device__ __forceinline__ Pair<float> pexp(Pair<float> x) { return Pair<float>::make(ex2_approx(x.lo()), ex2_approx(x.hi())); }

__device__ __forceinline__ Pair<double> pmul(Pair<double> x, Pair<double> y) { return {x.a * y.a, x.b * y.b}; }
__device__ __forceinline__ Pair<double> pfma(Pair<double> x, Pair<double> y, Pair<double> z) {
  return {fma(x.a, y.a, z.a), fma(x.b, y.b, z.b)};
}
__device__ __forceinline__ Pair<double> padd(Pair<double> x, Pair<double> y) { return {x.a + y.a, x.b + y.b}; }
__device__ __forceinline__ Pair<double> pexp(Pair<double> x) { return {exp(x.a), exp(x.b)}; }

constexpr int kP = kN / 2;   // state pairs per channel

// The io inputs of one 8-step segment of a channel, as raw 16-byte words: u, Δ_raw, dy, z.  Fetched
// one segment ahead (software pipeline), unpacked when the segment is processed.
template <typename IO>
struct SegRaw {
  static constexpr int kW = kSeg * static_cast<int>(sizeof(IO)) / 16;   // 16-byte words per array
  uint4 w[4][kW];
};

// vec: the row segment is 16-byte aligned and complete; otherwise scalar loads (zeros past nk)
template <typename IO>
__device__ __forceinline__ void fetch_one(const void* base, int64_t off, int nk, bool vec, uint4 (&w)[SegRaw<IO>::kW],
                                          int64_t n_total) {
  constexpr int kW = SegRaw<IO>::kW;
  const IO* p = checked(static_cast<const IO*>(base), off, n_total, nk);   // the segment's nk elements
  if (vec && nk == kSeg) {
#pragma unroll
    for (int i = 0; i < kW; ++i) w[i] = __ldg(reinterpret_cast<const uint4*>(p) + i);
  } else {
    IO e[kSeg];
#pragma unroll
    for (int k = 0; k < kSeg; ++k) e[k] = k < nk ? p[k] : IoTraits<IO>::from_f32(0.0f);
    static_assert(sizeof(e) == sizeof(w), "segment words");
    memcpy(&w, e, sizeof(e));
  }
}

template <typename IO>
__device__ __forceinline__ void fetch_seg(const BwdParams& p, int64_t off, int nk, SegRaw<IO>& r) {
  const int64_t n_io = static_cast<int64_t>(p.batch) * p.dim * p.L;
  fetch_one<IO>(p.u, off, nk, p.vec_io, r.w[0], n_io);
  fetch_one<IO>(p.delta, off, nk, p.vec_io, r.w[1], n_io);
  fetch_one<IO>(p.dy, off, nk, p.vec_io, r.w[2], n_io);
  if (p.z) fetch_one<IO>(p.z, off, nk, p.vec_io, r.w[3], n_io);
}

template <typename IO, typename CT>
__device__ __forceinline__ void unpack_one(const uint4 (&w)[SegRaw<IO>::kW], CT (&out)[kSeg]) {
  if constexpr (sizeof(IO) == 2) {
    float f[8];
    unpack_chunk(w[0], f, IO());
#pragma unroll
    for (int k = 0; k < kSeg; ++k) out[k] = f[k];
  } else {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      float f[4];
      unpack_chunk(w[i], f, IO());
#pragma unroll
      for (int k = 0; k < 4; ++k) out[4 * i + k] = f[k];
    }
  }
}

template <typename IO, typename CT>
__device__ __forceinline__ void store_seg(void* base, int64_t off, int nk, bool vec, const CT (&v)[kSeg], int64_t n_total) {
  IO* p = checked(static_cast<IO*>(base), off, n_total, nk);   // the segment's nk elements
  float f[kSeg];
#pragma unroll
  for (int k = 0; k < kSeg; ++k) f[k] = static_cast<float>(v[k]);
  if (vec && nk == kSeg) {
    if constexpr (sizeof(IO) == 2) {
      *reinterpret_cast<uint4*>(p) = pack_chunk(f);
    } else {
      const float a[4] = {f[0], f[1], f[2], f[3]}, b[4] = {f[4], f[5], f[6], f[7]};
      reinterpret_cast<uint4*>(p)[0] = pack_chunk(a);
      reinterpret_cast<uint4*>(p)[1] = pack_chunk(b);
    }
  } else {
#pragma unroll
    for (int k = 0; k < kSeg; ++k)
      if (k < nk) p[k] = IoTraits<IO>::from_f32(f[k]);
  }
}

// B and C of steps [t0, t0 + nk) of batch row b: each thread fetches 2 of the segment's 8 x 32 table
// entries ([step][B0..15 | C0..15], zeros past dstate / nk) one segment ahead and stores them, widened
// to float, when that segment starts.  The loads keep their raw bits until then (bf16: the 16-bit
// pattern), so no instruction waits for them while the current segment is computed.
__device__ __forceinline__ void fetch_bc(const BwdParams& p, int b, int64_t t0, int nk, uint32_t (&r)[2]) {
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int i = threadIdx.x + j * kThreads;
    const int k = i / 32, col = i % 32, arr = col / 16, n = col % 16;
    uint32_t v = 0u;
    if (k < nk && n < p.N) {
      const int64_t idx = (static_cast<int64_t>(b) * p.N + n) * p.L + t0 + k;
      const int64_t nbc = static_cast<int64_t>(p.batch) * p.N * p.L;
      const void* src = arr ? p.C : p.B;
      v = p.io_bf16 ? static_cast<uint32_t>(*checked(static_cast<const unsigned short*>(src), idx, nbc))
                    : *checked(static_cast<const uint32_t*>(src), idx, nbc);
    }
    r[j] = v;
  }
}

__device__ __forceinline__ void store_bc(float* bc, const uint32_t (&r)[2], bool bf16) {
  bc[threadIdx.x] = __uint_as_float(bf16 ? r[0] << 16 : r[0]);
  bc[threadIdx.x + kThreads] = __uint_as_float(bf16 ? r[1] << 16 : r[1]);
}

// The B and C rows of one 8-step segment for the two-lane (bf16) kernels.  With 16-byte rows (L a
// multiple of 8, B and C 16-byte aligned) and a full segment, thread t < 32 loads the segment's 8 steps
// of row t % 16 of B (t < 16) or C (t >= 16) in one 16-byte load; otherwise every thread fetches two
// elements as fetch_bc does (held in .x and .y).
struct BcSeg {
  uint4 v;
  bool vec;
};

__device__ __forceinline__ bool bc_rows_vec(const BwdParams& p) {
  return p.io_bf16 && p.L % kSeg == 0 &&
         ((reinterpret_cast<uintptr_t>(p.B) | reinterpret_cast<uintptr_t>(p.C)) & 15u) == 0;
}

__device__ __forceinline__ void fetch_bc2(const BwdParams& p, int b, int64_t t0, int nk, bool rows_vec, BcSeg& r) {
  r.vec = rows_vec && nk == kSeg;
  if (r.vec) {
    const int t = threadIdx.x, n = t & 15;
    r.v = make_uint4(0u, 0u, 0u, 0u);
    if (t < 32 && n < p.N) {
      const int64_t idx = (static_cast<int64_t>(b) * p.N + n) * p.L + t0;
      const int64_t nbc = static_cast<int64_t>(p.batch) * p.N * p.L;
      const unsigned short* src = static_cast<const unsigned short*>(t < 16 ? p.B : p.C);
      r.v = __ldg(reinterpret_cast<const uint4*>(checked(src, idx, nbc, kSeg)));
    }
  } else {
    uint32_t e[2];
    fetch_bc(p, b, t0, nk, e);
    r.v = make_uint4(e[0], e[1], 0u, 0u);
  }
}

__device__ __forceinline__ void store_bc2(float* bc, const BcSeg& r) {
  if (r.vec) {
    if (threadIdx.x < 32) {
      float f[kSeg];
      unpack_chunk(r.v, f, __nv_bfloat16());
#pragma unroll
      for (int k = 0; k < kSeg; ++k) bc[k * 32 + threadIdx.x] = f[k];
    }
  } else {
    const uint32_t e[2] = {r.v.x, r.v.y};
    store_bc(bc, e, true);
  }
}

// One checkpoint record: 16 states, 64 (float) or 128 (double) bytes, 16-byte aligned.
__device__ __forceinline__ void store_ckpt(float* dst, const Pair<float> (&h)[kP]) {
#pragma unroll
  for (int i = 0; i < kP / 2; ++i)
    reinterpret_cast<float4*>(dst)[i] = make_float4(h[2 * i].lo(), h[2 * i].hi(), h[2 * i + 1].lo(), h[2 * i + 1].hi());
}
__device__ __forceinline__ void store_ckpt(double* dst, const Pair<double> (&h)[kP]) {
#pragma unroll
  for (int j = 0; j < kP; ++j) reinterpret_cast<double2*>(dst)[j] = make_double2(h[j].a, h[j].b);
}
__device__ __forceinline__ void load_ckpt(const float* src, float (&r)[kN]) {
#pragma unroll
  for (int i = 0; i < kN / 4; ++i) {
    const float4 q = __ldg(reinterpret_cast<const float4*>(src) + i);
    r[4 * i] = q.x;
    r[4 * i + 1] = q.y;
    r[4 * i + 2] = q.z;
    r[4 * i + 3] = q.w;
  }
}
__device__ __forceinline__ void load_ckpt(const double* src, double (&r)[kN]) {
#pragma unroll
  for (int j = 0; j < kN / 2; ++j) {
    const double2 q = __ldg(reinterpret_cast<const double2*>(src) + j);
    r[2 * j] = q.x;
    r[2 * j + 1] = q.y;
  }
}

struct Tile {
  int b, d, dd;
  bool valid;
  int64_t row;           // b * dim + dd
  int64_t c0, c1;        // the chunk's steps [c0, c1)
  int64_t ag;            // index of the (row, chunk) aggregate
};

// element counts of the buffers, for the index checks of the checked build
struct Sizes {
  int64_t nA, nDim, nIO, nBC, nCk, nCs, nAgg;
};
__device__ __forceinline__ Sizes sizes_of(const BwdParams& p) {
  Sizes z{};
  if (!SSM_CHECK) return z;   // the ordinary build checks nothing
  const int64_t rows = static_cast<int64_t>(p.batch) * p.dim, nseg = (p.L + kSeg - 1) / kSeg;
  z.nA = static_cast<int64_t>(p.dim) * p.N;
  z.nDim = p.dim;
  z.nIO = rows * p.L;
  z.nBC = static_cast<int64_t>(p.batch) * p.N * p.L;
  z.nCk = rows * nseg * kN;
  z.nCs = rows * nseg;
  z.nAgg = rows * p.nchunks * kAgg;
  return z;
}

__device__ __forceinline__ Tile tile_of(const BwdParams& p) {
  Tile t;
  t.b = blockIdx.y;
  t.d = blockIdx.x * kThreads + threadIdx.x;
  t.valid = t.d < p.dim;
  t.dd = t.valid ? t.d : 0;
  t.row = static_cast<int64_t>(t.b) * p.dim + t.dd;
  t.c0 = static_cast<int64_t>(blockIdx.z) * p.chunk_len;
  t.c1 = t.c0 + p.chunk_len < p.L ? t.c0 + p.chunk_len : p.L;
  t.ag = (t.row * p.nchunks + blockIdx.z) * kAgg;
  return t;
}

// (1) local forward of one tile: checkpoints every 8 steps and the chunk aggregates P, Q, G.
// The next segment's inputs are fetched into registers while the current one is computed; B/C go
// through a double-buffered shared table, so each segment needs one barrier.
template <typename IO, typename CT>
__global__ void __launch_bounds__(kThreads, sizeof(CT) == 4 ? SSM_BWD_FWD_MINB : 1) bwd_chunk_fwd_kernel(const BwdParams p) {
  using P = Pair<CT>;
  __shared__ __align__(16) float bc_buf[2][kSeg * 32];
  const Tile T = tile_of(p);
  const Sizes Z = sizes_of(p);
  const int64_t nseg = (p.L + kSeg - 1) / kSeg;
  P A2[kP], h[kP], E[kP], G[kP];
  {
    const float* Ad = checked(p.A, static_cast<int64_t>(T.dd) * p.N, Z.nA, p.N);
#pragma unroll
    for (int j = 0; j < kP; ++j) {
      const CT a0 = 2 * j < p.N ? static_cast<CT>(Ad[2 * j]) : static_cast<CT>(0);
      const CT a1 = 2 * j + 1 < p.N ? static_cast<CT>(Ad[2 * j + 1]) : static_cast<CT>(0);
      A2[j] = P::make(a0 * P::kExpScale, a1 * P::kExpScale);
      h[j] = P::splat(0);
      E[j] = P::splat(1);
      G[j] = P::splat(0);
    }
  }
  const CT bias = p.bias ? *checked(p.bias, T.dd, Z.nDim) : 0.0f;
  CT S = 0;
  CT* const ck = static_cast<CT*>(p.ckpt) + T.row * nseg * kN;
  CT* const cs = static_cast<CT*>(p.ckpt_s) + T.row * nseg;
  auto seg_len = [&](int64_t t0) { return static_cast<int>(T.c1 - t0 < kSeg ? T.c1 - t0 : kSeg); };
  SegRaw<IO> raw;
  uint32_t bcr[2];
  fetch_seg<IO>(p, T.row * p.L + T.c0, seg_len(T.c0), raw);
  fetch_bc(p, T.b, T.c0, seg_len(T.c0), bcr);
  store_bc(bc_buf[0], bcr, p.io_bf16);
  __syncthreads();
  int buf = 0;
  for (int64_t t0 = T.c0; t0 < T.c1; t0 += kSeg) {
    const int nk = seg_len(t0);
    CT x[kSeg], v[kSeg], zz[kSeg], dyv[kSeg];
    unpack_one<IO, CT>(raw.w[0], x);
    unpack_one<IO, CT>(raw.w[1], v);
    unpack_one<IO, CT>(raw.w[2], dyv);
    if (p.z) unpack_one<IO, CT>(raw.w[3], zz);
    const int64_t tn = t0 + kSeg;
    const bool more = tn < T.c1;
    if (more) {
      fetch_seg<IO>(p, T.row * p.L + tn, seg_len(tn), raw);
      fetch_bc(p, T.b, tn, seg_len(tn), bcr);
    }
    if (T.valid) {
      const int64_t s = t0 / kSeg;
      store_ckpt(checked(ck, s * kN, Z.nCk - T.row * nseg * kN, kN), h);
      *checked(cs, s, Z.nCs - T.row * nseg) = S;
    }
    const f2* bc2 = reinterpret_cast<const f2*>(bc_buf[buf]);   // [k][B pairs 0..7 | C pairs 0..7]
#pragma unroll
    for (int k = 0; k < kSeg; ++k) {
      if (k < nk) {
        const CT dl = p.softplus ? sp<CT>(v[k] + bias) : v[k] + bias;
        const CT ds = p.z ? dyv[k] * zz[k] * sigm<CT>(zz[k]) : dyv[k];
        S += dl;
        const P dlp = P::splat(dl), dlx = P::splat(dl * x[k]), dsp = P::splat(ds);
#pragma unroll
        for (int j = 0; j < kP; ++j) {
          const P a = pexp(pmul(dlp, A2[j]));
          h[j] = pfma(a, h[j], pmul(dlx, P::from_f2(bc2[k * 16 + j])));
          E[j] = pmul(E[j], a);
          G[j] = pfma(E[j], pmul(P::from_f2(bc2[k * 16 + 8 + j]), dsp), G[j]);
        }
      }
    }
    if (more) store_bc(bc_buf[buf ^ 1], bcr, p.io_bf16);
    __syncthreads();
    buf ^= 1;
  }
  if (T.valid) {
    CT* const base = static_cast<CT*>(p.agg);
    CT* const aq = checked(base, T.ag, Z.nAgg, kN);
    CT* const ap = checked(base, T.ag + kN, Z.nAgg, kN);
    CT* const agg = checked(base, T.ag + 2 * kN, Z.nAgg, kN);
#pragma unroll
    for (int j = 0; j < kP; ++j) {
      aq[2 * j] = h[j].lo();
      aq[2 * j + 1] = h[j].hi();
      ap[2 * j] = E[j].lo();
      ap[2 * j + 1] = E[j].hi();
      agg[2 * j] = G[j].lo();
      agg[2 * j + 1] = G[j].hi();
    }
  }
}

// (1') local forward with two lanes per channel (bfloat16 io): lane pl of a channel runs the states
// 8pl .. 8pl + 7; both lanes evaluate the per-step scalars.  Same outputs as (1).
// kZ (a gate is given), kSp (softplus on Δ) and kFull (every 8-step segment full: L and the chunk
// length multiples of 8) are template parameters: tested at run time inside the unrolled steps they
// split the segment's body into basic blocks the compiler does not schedule across.
template <typename IO, bool kZ, bool kSp, bool kFull>
__global__ void __launch_bounds__(kThreads, 4) bwd_fwd2_kernel(const BwdParams p) {
  using P = Pair<float>;
  __shared__ __align__(16) float bc_buf[2][kSeg * 32];
  const int tid = threadIdx.x;
  const int pl = tid & 1;
  const int b = blockIdx.y;
  const int d = blockIdx.x * 64 + (tid >> 1);
  const bool valid = d < p.dim;
  const int dd = valid ? d : 0;
  const int64_t row = static_cast<int64_t>(b) * p.dim + dd;
  const int64_t c0 = static_cast<int64_t>(blockIdx.z) * p.chunk_len;
  const int64_t c1 = c0 + p.chunk_len < p.L ? c0 + p.chunk_len : p.L;
  const int64_t nseg = (p.L + kSeg - 1) / kSeg;
  const Sizes Z = sizes_of(p);
  const int n0 = 8 * pl;
  P A2[4], h[4], E[4], G[4];
  {
    const float* Ad = checked(p.A, static_cast<int64_t>(dd) * p.N, Z.nA, p.N);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + 2 * j;
      A2[j] = P::make((n < p.N ? Ad[n] : 0.0f) * kLog2e, (n + 1 < p.N ? Ad[n + 1] : 0.0f) * kLog2e);
      h[j] = P::splat(0.0f);
      E[j] = P::splat(1.0f);
      G[j] = P::splat(0.0f);
    }
  }
  const float bias = p.bias ? *checked(p.bias, dd, Z.nDim) : 0.0f;
  float S = 0.0f;
  const int64_t ck_row = row * nseg * kN + n0, cs_row = row * nseg;
  float* const ck = static_cast<float*>(p.ckpt) + ck_row;   // this lane's checkpoint row
  float* const cs = static_cast<float*>(p.ckpt_s) + cs_row;
  auto seg_len = [&](int64_t t0) { return static_cast<int>(c1 - t0 < kSeg ? c1 - t0 : kSeg); };
  SegRaw<IO> raw;
  BcSeg bcr;
  const bool rows_vec = bc_rows_vec(p);
  fetch_seg<IO>(p, row * p.L + c0, seg_len(c0), raw);
  fetch_bc2(p, b, c0, seg_len(c0), rows_vec, bcr);
  store_bc2(bc_buf[0], bcr);
  __syncthreads();
  int buf = 0;
  for (int64_t t0 = c0; t0 < c1; t0 += kSeg) {
    const int nk = kFull ? kSeg : seg_len(t0);
    float x[kSeg], v[kSeg], zz[kSeg], dyv[kSeg];
    unpack_one<IO, float>(raw.w[0], x);
    unpack_one<IO, float>(raw.w[1], v);
    unpack_one<IO, float>(raw.w[2], dyv);
    if (kZ) unpack_one<IO, float>(raw.w[3], zz);
    const int64_t tn = t0 + kSeg;
    const bool more = tn < c1;
    if (more) {
      fetch_seg<IO>(p, row * p.L + tn, seg_len(tn), raw);
      fetch_bc2(p, b, tn, seg_len(tn), rows_vec, bcr);
    }
    if (valid) {
      const int64_t sgi = t0 / kSeg;
      float4* const cq = reinterpret_cast<float4*>(checked(ck, sgi * kN, Z.nCk - ck_row, 8));
      cq[0] = make_float4(h[0].lo(), h[0].hi(), h[1].lo(), h[1].hi());
      cq[1] = make_float4(h[2].lo(), h[2].hi(), h[3].lo(), h[3].hi());
      if (pl == 0) *checked(cs, sgi, Z.nCs - cs_row) = S;
    }
    const f2* bc2 = reinterpret_cast<const f2*>(bc_buf[buf]);
#pragma unroll
    for (int k = 0; k < kSeg; ++k) {
      if (k < nk) {
        const float vb = v[k] + bias;
        const float dl = kSp ? softplus_fast(vb) : vb;
        const float ds = kZ ? dyv[k] * zz[k] * rcp_approx(1.0f + ex2_approx(-zz[k] * kLog2e)) : dyv[k];
        S += dl;
        const P dlp = P::splat(dl), dlx = P::splat(dl * x[k]), dsp = P::splat(ds);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const P a = pexp(pmul(dlp, A2[j]));
          h[j] = pfma(a, h[j], pmul(dlx, P::from_f2(bc2[k * 16 + 4 * pl + j])));
          E[j] = pmul(E[j], a);
          G[j] = pfma(E[j], pmul(P::from_f2(bc2[k * 16 + 8 + 4 * pl + j]), dsp), G[j]);
        }
      }
    }
    if (more) store_bc2(bc_buf[buf ^ 1], bcr);
    __syncthreads();
    buf ^= 1;
  }
  if (valid) {
    float* const base = static_cast<float*>(p.agg);
    const int64_t a0 = (row * p.nchunks + blockIdx.z) * kAgg + n0;
    float* const aq = checked(base, a0, Z.nAgg, 8);
    float* const ap = checked(base, a0 + kN, Z.nAgg, 8);
    float* const agg = checked(base, a0 + 2 * kN, Z.nAgg, 8);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      aq[2 * j] = h[j].lo();
      aq[2 * j + 1] = h[j].hi();
      ap[2 * j] = E[j].lo();
      ap[2 * j + 1] = E[j].hi();
      agg[2 * j] = G[j].lo();
      agg[2 * j + 1] = G[j].hi();
    }
  }
}

// (2) carries across chunks, one thread per (channel, state): Q becomes h_start, G becomes dh_in.
// The aggregates are read 8 chunks at a time ahead of the serial composition, so that the loads of
// a batch are in flight together.
template <typename CT>
__global__ void bwd_carry_kernel(const BwdParams p) {
  constexpr int kB8 = 8;
  const int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  const int64_t rows = static_cast<int64_t>(p.batch) * p.dim;
  if (i >= rows * kN) return;
  const int64_t row = i / kN;
  const int n = static_cast<int>(i % kN);
  const Sizes Z = sizes_of(p);
  CT* const base = static_cast<CT*>(p.agg);
  const int64_t a0 = row * p.nchunks * kAgg + n;
  auto ag = [&](int64_t off) -> CT& { return *checked(base, a0 + off, Z.nAgg); };
  CT h = 0;
  for (int c0 = 0; c0 < p.nchunks; c0 += kB8) {
    CT q[kB8], P[kB8];
#pragma unroll
    for (int k = 0; k < kB8; ++k) {
      const int c = c0 + k;
      q[k] = c < p.nchunks ? ag(static_cast<int64_t>(c) * kAgg) : CT(0);
      P[k] = c < p.nchunks ? ag(static_cast<int64_t>(c) * kAgg + kN) : CT(0);
    }
#pragma unroll
    for (int k = 0; k < kB8; ++k) {
      const int c = c0 + k;
      if (c < p.nchunks) {
        ag(static_cast<int64_t>(c) * kAgg) = h;
        h = P[k] * h + q[k];
      }
    }
  }
  CT g = 0;
  for (int c0 = p.nchunks - 1; c0 >= 0; c0 -= kB8) {
    CT gc[kB8], P[kB8];
#pragma unroll
    for (int k = 0; k < kB8; ++k) {
      const int c = c0 - k;
      gc[k] = c >= 0 ? ag(static_cast<int64_t>(c) * kAgg + 2 * kN) : CT(0);
      P[k] = c >= 0 ? ag(static_cast<int64_t>(c) * kAgg + kN) : CT(0);
    }
#pragma unroll
    for (int k = 0; k < kB8; ++k) {
      const int c = c0 - k;
      if (c >= 0) {
        ag(static_cast<int64_t>(c) * kAgg + 2 * kN) = g;
        g = gc[k] + P[k] * g;
      }
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

__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

// (3) reverse pass of one tile.  Pipelined like (1): the previous segment's inputs, checkpoint and
// B/C are fetched while the current one is computed; the dB/dC partials are double-buffered and
// reduced one segment later by the first two warps.
template <typename IO, typename CT>
__global__ void __launch_bounds__(kThreads) bwd_chunk_rev_kernel(const BwdParams p) {
  using P = Pair<CT>;
  extern __shared__ __align__(16) uint8_t smem[];
  float* bc_base = reinterpret_cast<float*>(smem);                                           // [2][k][32]
  P* hbuf = reinterpret_cast<P*>(smem + Smem<CT>::kBC);                                      // [k][j][thread]
  CT* red_base = reinterpret_cast<CT*>(smem + Smem<CT>::kBC + Smem<CT>::kH);                  // [2][warp][k][32]
  P* hs_s = reinterpret_cast<P*>(smem + Smem<CT>::kBC + Smem<CT>::kH + Smem<CT>::kRed);      // [j][thread]
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const Tile T = tile_of(p);
  const Sizes Z = sizes_of(p);
  const int64_t nseg = (p.L + kSeg - 1) / kSeg;
  P A2[kP], dh[kP], dA[kP];
  {
    const CT* const agb = static_cast<const CT*>(p.agg);
    const CT* const aq = checked(agb, T.ag, Z.nAgg, kN);
    const CT* const agd = checked(agb, T.ag + 2 * kN, Z.nAgg, kN);
    const float* Ad = checked(p.A, static_cast<int64_t>(T.dd) * p.N, Z.nA, p.N);
#pragma unroll
    for (int j = 0; j < kP; ++j) {
      const CT a0 = 2 * j < p.N ? static_cast<CT>(Ad[2 * j]) : static_cast<CT>(0);
      const CT a1 = 2 * j + 1 < p.N ? static_cast<CT>(Ad[2 * j + 1]) : static_cast<CT>(0);
      A2[j] = P::make(a0 * P::kExpScale, a1 * P::kExpScale);
      hs_s[j * kThreads + tid] = P::make(aq[2 * j], aq[2 * j + 1]);
      dh[j] = T.valid ? P::make(agd[2 * j], agd[2 * j + 1]) : P::splat(0);
      dA[j] = P::splat(0);
    }
  }
  const CT bias = p.bias ? *checked(p.bias, T.dd, Z.nDim) : 0.0f;
  const CT Dd = p.D ? *checked(p.D, T.dd, Z.nDim) : 0.0f;
  CT dD = 0, dbias = 0;
  const CT* const ck = static_cast<const CT*>(p.ckpt) + T.row * nseg * kN;
  const CT* const cs = static_cast<const CT*>(p.ckpt_s) + T.row * nseg;
  auto seg_len = [&](int64_t t0) { return static_cast<int>(T.c1 - t0 < kSeg ? T.c1 - t0 : kSeg); };
  // adds the CTA's dB/dC partials of the segment at t0 (buffer rb) to global memory
  auto flush_red = [&](const CT* rb, int64_t t0, int nk) {
    if (tid >= 64) return;
    const int col = tid & 31, half = tid >> 5, arr = col / 16, n = col % 16;
    const int k0 = half * 4;
    if (n >= p.N || k0 >= nk) return;
    CT s4[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      s4[i] = (rb[(0 * kSeg + k0 + i) * 32 + col] + rb[(1 * kSeg + k0 + i) * 32 + col]) +
              (rb[(2 * kSeg + k0 + i) * 32 + col] + rb[(3 * kSeg + k0 + i) * 32 + col]);
    CT* dst = checked(static_cast<CT*>(arr ? p.acc_dC : p.acc_dB), (static_cast<int64_t>(T.b) * p.N + n) * p.L + t0 + k0,
                      Z.nBC, nk - k0 < 4 ? nk - k0 : 4);
    if constexpr (sizeof(CT) == 4) {
      if (p.vec_red && k0 + 4 <= nk) {
        red_add_v4(dst, s4[0], s4[1], s4[2], s4[3]);
        return;
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (k0 + i < nk) atomicAdd(dst + i, s4[i]);
  };
  const int64_t last = T.c0 + ((T.c1 - T.c0 - 1) / kSeg) * kSeg;
  SegRaw<IO> raw;
  uint32_t bcr[2];
  CT ckr[kN], ckS;
  auto fetch_ck = [&](int64_t t0) {
    const int64_t s = t0 / kSeg;
    load_ckpt(checked(ck, s * kN, Z.nCk - T.row * nseg * kN, kN), ckr);
    ckS = *checked(cs, s, Z.nCs - T.row * nseg);
  };
  fetch_seg<IO>(p, T.row * p.L + last, seg_len(last), raw);
  fetch_bc(p, T.b, last, seg_len(last), bcr);
  fetch_ck(last);
  store_bc(bc_base, bcr, p.io_bf16);
  __syncthreads();
  int buf = 0;
  int64_t pend_t0 = -1;   // the segment whose dB/dC partials wait in the other red buffer
  int pend_nk = 0;
  for (int64_t t0 = last; t0 >= T.c0; t0 -= kSeg) {
    const int nk = seg_len(t0);
    const int64_t off = T.row * p.L + t0;
    const f2* bc2 = reinterpret_cast<const f2*>(bc_base + buf * (kSeg * 32));   // [k][B pairs | C pairs]
    CT* red = red_base + buf * (4 * kSeg * 32);
    CT x[kSeg], v[kSeg], zz[kSeg], dyv[kSeg];
    unpack_one<IO, CT>(raw.w[0], x);
    unpack_one<IO, CT>(raw.w[1], v);
    unpack_one<IO, CT>(raw.w[2], dyv);
    if (p.z) unpack_one<IO, CT>(raw.w[3], zz);
    // the true state entering the segment: local checkpoint + decayed chunk start state
    P h0[kP];
    {
      const P Sp = P::splat(ckS);
#pragma unroll
      for (int j = 0; j < kP; ++j)
        h0[j] = pfma(pexp(pmul(A2[j], Sp)), hs_s[j * kThreads + tid], P::make(ckr[2 * j], ckr[2 * j + 1]));
    }
    const int64_t tn = t0 - kSeg;
    const bool more = tn >= T.c0;
    if (more) {
      fetch_seg<IO>(p, T.row * p.L + tn, seg_len(tn), raw);
      fetch_bc(p, T.b, tn, seg_len(tn), bcr);
      fetch_ck(tn);
    }
    if (pend_t0 >= 0) flush_red(red_base + (buf ^ 1) * (4 * kSeg * 32), pend_t0, pend_nk);
    // recompute the segment forwards: states into shared memory, Δ, σ(v), ds; dz is final here
    CT dl[kSeg], sg[kSeg], ds[kSeg], gdz[kSeg];
    P hc[kP];   // the state after the step being differentiated (ends as the segment's last)
#pragma unroll
    for (int j = 0; j < kP; ++j) hc[j] = h0[j];
#pragma unroll
    for (int k = 0; k < kSeg; ++k) {
      gdz[k] = 0;
      if (k < nk) {
        const CT vb = v[k] + bias;
        dl[k] = p.softplus ? sp<CT>(vb) : vb;
        sg[k] = p.softplus ? sigm<CT>(vb) : static_cast<CT>(1);
        const P dlp = P::splat(dl[k]), dlx = P::splat(dl[k] * x[k]);
        P sa[2] = {P::make(Dd * x[k], 0), P::splat(0)};   // C·h in four partial sums
#pragma unroll
        for (int j = 0; j < kP; ++j) {
          hc[j] = pfma(pexp(pmul(dlp, A2[j])), hc[j], pmul(dlx, P::from_f2(bc2[k * 16 + j])));
          if (k < kSeg - 1) hbuf[(k * kP + j) * kThreads + tid] = hc[j];
          sa[j & 1] = pfma(P::from_f2(bc2[k * 16 + 8 + j]), hc[j], sa[j & 1]);
        }
        const P st = padd(sa[0], sa[1]);
        const CT sacc = st.lo() + st.hi();
        if (p.z) {
          const CT sz = sigm<CT>(zz[k]);
          ds[k] = dyv[k] * zz[k] * sz;
          gdz[k] = dyv[k] * sacc * sz * (static_cast<CT>(1) + zz[k] * (static_cast<CT>(1) - sz));
        } else {
          ds[k] = dyv[k];
        }
        if (!T.valid) ds[k] = 0;
      } else {
        dl[k] = sg[k] = ds[k] = 0;
      }
    }
    if (T.valid && p.z) store_seg<IO, CT>(p.dz, off, nk, p.vec_io, gdz, Z.nIO);
    // backward over the segment's steps
    CT gdu[kSeg], gdd[kSeg];
#pragma unroll
    for (int k = kSeg - 1; k >= 0; --k) {
      gdu[k] = gdd[k] = 0;
      if (k < nk) {
        dD += ds[k] * x[k];
        const P dlp = P::splat(dl[k]), dsp = P::splat(ds[k]), dlx = P::splat(dl[k] * x[k]);
        P dq[2] = {P::splat(0), P::splat(0)}, db[2] = {P::splat(0), P::splat(0)};
        CT vals[32];
#pragma unroll
        for (int j = 0; j < kP; ++j) {
          const P abar = pexp(pmul(dlp, A2[j]));
          const P bn = P::from_f2(bc2[k * 16 + j]);
          const P cn = P::from_f2(bc2[k * 16 + 8 + j]);
          dh[j] = pfma(dsp, cn, dh[j]);
          // the state after step k is hc; the one before it is h0 or recomputed in shared memory
          const P hp = k > 0 ? hbuf[((k - 1) * kP + j) * kThreads + tid] : h0[j];
          const P vc = pmul(dsp, hc[j]);            // dC contribution
          const P vb = pmul(dh[j], dlx);            // dB contribution
          vals[16 + 2 * j] = vc.lo();
          vals[16 + 2 * j + 1] = vc.hi();
          vals[2 * j] = vb.lo();
          vals[2 * j + 1] = vb.hi();
          const P w = pmul(pmul(dh[j], hp), abar);  // gradient of the exponent of Ā
          dq[j & 1] = pfma(w, A2[j], dq[j & 1]);
          dA[j] = pfma(w, dlp, dA[j]);
          db[j & 1] = pfma(dh[j], bn, db[j & 1]);
          dh[j] = pmul(dh[j], abar);
          hc[j] = hp;
        }
        const P dbt = padd(db[0], db[1]), dqt = padd(dq[0], dq[1]);
        const CT dhb = dbt.lo() + dbt.hi();
        // dq sums w·A·kExpScale: undo the exponent scale
        const CT ddl = (dqt.lo() + dqt.hi()) * (static_cast<CT>(1) / P::kExpScale) + dhb * x[k];
        const CT dv = ddl * sg[k];
        gdu[k] = ds[k] * Dd + dhb * dl[k];
        gdd[k] = dv;
        dbias += dv;
        red[(warp * kSeg + k) * 32 + lane] = warp_transpose_sum<CT>(vals);
      }
    }
    if (T.valid) {
      store_seg<IO, CT>(p.du, off, nk, p.vec_io, gdu, Z.nIO);
      store_seg<IO, CT>(p.ddelta, off, nk, p.vec_io, gdd, Z.nIO);
    }
    if (more) store_bc(bc_base + (buf ^ 1) * (kSeg * 32), bcr, p.io_bf16);
    __syncthreads();
    pend_t0 = t0;
    pend_nk = nk;
    buf ^= 1;
  }
  if (pend_t0 >= 0) flush_red(red_base + (buf ^ 1) * (4 * kSeg * 32), pend_t0, pend_nk);
  if (T.valid) {
    CT* accA = checked(static_cast<CT*>(p.acc_dA), static_cast<int64_t>(T.d) * p.N, Z.nA, p.N);
#pragma unroll
    for (int j = 0; j < kP; ++j) {
      if (2 * j < p.N) atomicAdd(accA + 2 * j, dA[j].lo());
      if (2 * j + 1 < p.N) atomicAdd(accA + 2 * j + 1, dA[j].hi());
    }
    if (p.acc_dD) atomicAdd(checked(static_cast<CT*>(p.acc_dD), T.d, Z.nDim), dD);
    if (p.acc_dbias) atomicAdd(checked(static_cast<CT*>(p.acc_dbias), T.d, Z.nDim), dbias);
  }
}

// (3') reverse pass with two lanes per channel (bfloat16 io, float32 arithmetic): lane pl of a channel
// owns the states 8pl .. 8pl + 7, so a CTA of 128 threads covers 64 channels with half the per-thread
// state of (3) and more resident warps.  The per-step scalars (Δ, σ, ds, the output gradients) are
// computed by both lanes; the partial sums over states (C·h, the two reductions of the Δ gradient) are
// completed with one lane exchange.  dB/dC: a 4-round butterfly over the 16 channels of a warp that share
// the lane parity leaves lane l with the sum of value (l >> 1) & 15 of its half.
constexpr int kCh2 = 64;       // channels per CTA of (3')
constexpr int kP2 = 4;         // state pairs per lane

struct Smem2 {
  static constexpr int kBC = 2 * kSeg * 32 * 4;                 // B/C table, two buffers
  static constexpr int kH = kSeg * kP2 * kThreads * 8;          // recomputed states [k][j/2][thread][2] (pairs)
  static constexpr int kRed = 2 * 4 * kSeg * 32 * 4;            // dB/dC partials, two buffers
  static constexpr int kHs = kP2 * kThreads * 8;                // chunk start states [j][thread]
  static constexpr int kTotal = kBC + kH + kRed + kHs;
};

template <typename IO, bool kZ, bool kSp>
__global__ void __launch_bounds__(kThreads, 3) bwd_rev2_kernel(const BwdParams p) {
  using P = Pair<float>;
  extern __shared__ __align__(16) uint8_t smem[];
  float* bc_base = reinterpret_cast<float*>(smem);
  P* hbuf = reinterpret_cast<P*>(smem + Smem2::kBC);
  float* red_base = reinterpret_cast<float*>(smem + Smem2::kBC + Smem2::kH);
  P* hs_s = reinterpret_cast<P*>(smem + Smem2::kBC + Smem2::kH + Smem2::kRed);
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int pl = tid & 1;                       // which half of the states
  const int b = blockIdx.y;
  const int d = blockIdx.x * kCh2 + (tid >> 1);
  const bool valid = d < p.dim;
  const int dd = valid ? d : 0;
  const int64_t row = static_cast<int64_t>(b) * p.dim + dd;
  const int64_t c0 = static_cast<int64_t>(blockIdx.z) * p.chunk_len;
  const int64_t c1 = c0 + p.chunk_len < p.L ? c0 + p.chunk_len : p.L;
  const int64_t nseg = (p.L + kSeg - 1) / kSeg;
  const int n0 = 8 * pl;                        // first state of this lane
  // Pair slot j of this lane holds the states n0 + 2·(j ^ pm) and the next one: the XOR with lane
  // bits 4 and 3 places the pairs that the first two rounds of the dB/dC butterfly keep in the lower
  // slots, so those rounds need no selects
  const int pm = (((lane >> 4) & 1) << 1) | ((lane >> 3) & 1);
  const Sizes Z = sizes_of(p);
  P A2[kP2], dh[kP2], dA[kP2];
  {
    const float* const agb = static_cast<const float*>(p.agg);
    const int64_t a0i = (row * p.nchunks + blockIdx.z) * kAgg;
    const float* const aq = checked(agb, a0i, Z.nAgg, kN);
    const float* const agd = checked(agb, a0i + 2 * kN, Z.nAgg, kN);
    const float* Ad = checked(p.A, static_cast<int64_t>(dd) * p.N, Z.nA, p.N);
#pragma unroll
    for (int j = 0; j < kP2; ++j) {
      const int n = n0 + 2 * (j ^ pm);
      const float a0 = n < p.N ? Ad[n] : 0.0f;
      const float a1 = n + 1 < p.N ? Ad[n + 1] : 0.0f;
      A2[j] = P::make(a0 * kLog2e, a1 * kLog2e);
      hs_s[j * kThreads + tid] = P::make(aq[n], aq[n + 1]);
      dh[j] = valid ? P::make(agd[n], agd[n + 1]) : P::splat(0.0f);
      dA[j] = P::splat(0.0f);
    }
  }
  const float bias = p.bias ? *checked(p.bias, dd, Z.nDim) : 0.0f;
  const float Dd = p.D ? *checked(p.D, dd, Z.nDim) : 0.0f;
  float dD = 0.0f, dbias = 0.0f;
  const int64_t ck_row = row * nseg * kN + n0, cs_row = row * nseg;
  const float* const ck = static_cast<const float*>(p.ckpt) + ck_row;   // this lane's checkpoint row
  const float* const cs = static_cast<const float*>(p.ckpt_s) + cs_row;
  auto seg_len = [&](int64_t t0) { return static_cast<int>(c1 - t0 < kSeg ? c1 - t0 : kSeg); };
  auto flush_red = [&](const float* rb, int64_t t0, int nk) {
    if (tid >= 64) return;
    const int col = tid & 31, half = tid >> 5, arr = col / 16, n = col % 16;
    const int k0 = half * 4;
    if (n >= p.N || k0 >= nk) return;
    float s4[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      s4[i] = (rb[(0 * kSeg + k0 + i) * 32 + col] + rb[(1 * kSeg + k0 + i) * 32 + col]) +
              (rb[(2 * kSeg + k0 + i) * 32 + col] + rb[(3 * kSeg + k0 + i) * 32 + col]);
    float* dst = checked(static_cast<float*>(arr ? p.acc_dC : p.acc_dB), (static_cast<int64_t>(b) * p.N + n) * p.L + t0 + k0,
                         Z.nBC, nk - k0 < 4 ? nk - k0 : 4);
    if (p.vec_red && k0 + 4 <= nk) {
      red_add_v4(dst, s4[0], s4[1], s4[2], s4[3]);
      return;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (k0 + i < nk) atomicAdd(dst + i, s4[i]);
  };
  const int64_t last = c0 + ((c1 - c0 - 1) / kSeg) * kSeg;
  SegRaw<IO> raw;
  BcSeg bcr;
  const bool rows_vec = bc_rows_vec(p);
  float2 ckp[kP2];   // checkpoint pairs, in slot order
  float ckS;
  auto fetch_ck = [&](int64_t t0) {
    const int64_t sgi = t0 / kSeg;
    const float2* const cq = reinterpret_cast<const float2*>(checked(ck, sgi * kN, Z.nCk - ck_row, 8));
#pragma unroll
    for (int j = 0; j < kP2; ++j) ckp[j] = __ldg(cq + (j ^ pm));
    ckS = *checked(cs, sgi, Z.nCs - cs_row);
  };
  fetch_seg<IO>(p, row * p.L + last, seg_len(last), raw);
  fetch_bc2(p, b, last, seg_len(last), rows_vec, bcr);
  fetch_ck(last);
  store_bc2(bc_base, bcr);
  __syncthreads();
  int buf = 0;
  int64_t pend_t0 = -1;
  int pend_nk = 0;
  // the column of the dB/dC table this lane's butterfly result belongs to: pair pm, dB or dC by lane
  // bit 2, low or high state of the pair by lane bit 1
  const int rcol = ((lane >> 2) & 1) * 16 + n0 + 2 * pm + ((lane >> 1) & 1);
  for (int64_t t0 = last; t0 >= c0; t0 -= kSeg) {
    const int nk = seg_len(t0);
    const int64_t off = row * p.L + t0;
    // this lane's B pairs at bcl[k * 16 + (j ^ pm)], C pairs 8 further
    const f2* bcl = reinterpret_cast<const f2*>(bc_base + buf * (kSeg * 32)) + 4 * pl;
    float* red = red_base + buf * (4 * kSeg * 32);
    float x[kSeg], v[kSeg], zz[kSeg], dyv[kSeg];
    unpack_one<IO, float>(raw.w[0], x);
    unpack_one<IO, float>(raw.w[1], v);
    unpack_one<IO, float>(raw.w[2], dyv);
    if (kZ) unpack_one<IO, float>(raw.w[3], zz);
    P h0[kP2];
    {
      const P Sp = P::splat(ckS);
#pragma unroll
      for (int j = 0; j < kP2; ++j)
        h0[j] = pfma(pexp(pmul(A2[j], Sp)), hs_s[j * kThreads + tid], P::make(ckp[j].x, ckp[j].y));
    }
    const int64_t tn = t0 - kSeg;
    const bool more = tn >= c0;
    if (more) {
      fetch_seg<IO>(p, row * p.L + tn, seg_len(tn), raw);
      fetch_bc2(p, b, tn, seg_len(tn), rows_vec, bcr);
      fetch_ck(tn);
    }
    if (pend_t0 >= 0) flush_red(red_base + (buf ^ 1) * (4 * kSeg * 32), pend_t0, pend_nk);
    // recompute the segment (this lane's 8 states), finish C·h with the partner lane
    float dl[kSeg], sg[kSeg], ds[kSeg], gdz[kSeg];
    P hc[kP2];
#pragma unroll
    for (int j = 0; j < kP2; ++j) hc[j] = h0[j];
#pragma unroll
    for (int k = 0; k < kSeg; ++k) {
      gdz[k] = 0.0f;
      if (k < nk) {
        const float vb = v[k] + bias;
        dl[k] = kSp ? softplus_fast(vb) : vb;
        sg[k] = kSp ? rcp_approx(1.0f + ex2_approx(-vb * kLog2e)) : 1.0f;
        const P dlp = P::splat(dl[k]), dlx = P::splat(dl[k] * x[k]);
        P sa = P::splat(0.0f);
#pragma unroll
        for (int j = 0; j < kP2; ++j) {
          hc[j] = pfma(pexp(pmul(dlp, A2[j])), hc[j], pmul(dlx, P::from_f2(bcl[k * 16 + (j ^ pm)])));
          sa = pfma(P::from_f2(bcl[k * 16 + 8 + (j ^ pm)]), hc[j], sa);
        }
        if (k < kSeg - 1) {
          // slots 2jj and 2jj + 1 side by side: one 16-byte store each ([k][jj][thread][2] pairs)
#pragma unroll
          for (int jj = 0; jj < 2; ++jj)
            *reinterpret_cast<float4*>(&hbuf[((k * 2 + jj) * kThreads + tid) * 2]) =
                make_float4(hc[2 * jj].lo(), hc[2 * jj].hi(), hc[2 * jj + 1].lo(), hc[2 * jj + 1].hi());
        }
        const float part = sa.lo() + sa.hi();
        const float sacc = part + __shfl_xor_sync(0xffffffffu, part, 1) + Dd * x[k];
        if (kZ) {
          const float sz = rcp_approx(1.0f + ex2_approx(-zz[k] * kLog2e));
          ds[k] = dyv[k] * zz[k] * sz;
          gdz[k] = dyv[k] * sacc * sz * (1.0f + zz[k] * (1.0f - sz));
        } else {
          ds[k] = dyv[k];
        }
        if (!valid) ds[k] = 0.0f;
      } else {
        dl[k] = sg[k] = ds[k] = 0.0f;
        // keep the partner exchange uniform: the partner lane runs the same k with the same nk
      }
    }
    if (valid && kZ && pl == 1) store_seg<IO, float>(p.dz, off, nk, p.vec_io, gdz, Z.nIO);
    float gdu[kSeg], gdd[kSeg];
#pragma unroll
    for (int k = kSeg - 1; k >= 0; --k) {
      gdu[k] = gdd[k] = 0.0f;
      if (k < nk) {
        dD += ds[k] * x[k];
        const P dlp = P::splat(dl[k]), dsp = P::splat(ds[k]), dlx = P::splat(dl[k] * x[k]);
        P dq = P::splat(0.0f), db = P::splat(0.0f);
        float vals[16];
        P hpv[kP2];   // the state before step k: h0 or recomputed in shared memory
        if (k > 0) {
#pragma unroll
          for (int jj = 0; jj < 2; ++jj) {
            const float4 v4 = *reinterpret_cast<const float4*>(&hbuf[(((k - 1) * 2 + jj) * kThreads + tid) * 2]);
            hpv[2 * jj] = P::make(v4.x, v4.y);
            hpv[2 * jj + 1] = P::make(v4.z, v4.w);
          }
        } else {
#pragma unroll
          for (int j = 0; j < kP2; ++j) hpv[j] = h0[j];
        }
#pragma unroll
        for (int j = 0; j < kP2; ++j) {
          const P abar = pexp(pmul(dlp, A2[j]));
          const P bn = P::from_f2(bcl[k * 16 + (j ^ pm)]);
          const P cn = P::from_f2(bcl[k * 16 + 8 + (j ^ pm)]);
          dh[j] = pfma(dsp, cn, dh[j]);
          const P hp = hpv[j];
          const P vc = pmul(dsp, hc[j]);
          const P vbb = pmul(dh[j], dlx);
          vals[4 * j] = vbb.lo();
          vals[4 * j + 1] = vbb.hi();
          vals[4 * j + 2] = vc.lo();
          vals[4 * j + 3] = vc.hi();
          const P w = pmul(pmul(dh[j], hp), abar);
          dq = pfma(w, A2[j], dq);
          dA[j] = pfma(w, dlp, dA[j]);
          db = pfma(dh[j], bn, db);
          dh[j] = pmul(dh[j], abar);
          hc[j] = hp;
        }
        const float dbm = db.lo() + db.hi(), dqm = dq.lo() + dq.hi();
        const float dhb = dbm + __shfl_xor_sync(0xffffffffu, dbm, 1);
        const float dqs = dqm + __shfl_xor_sync(0xffffffffu, dqm, 1);
        const float ddl = dqs * kLn2 + dhb * x[k];
        const float dv = ddl * sg[k];
        gdu[k] = ds[k] * Dd + dhb * dl[k];
        gdd[k] = dv;
        dbias += dv;
        // butterfly over the 16 channels sharing this lane's parity.  Lane bits 4 and 3: the slot
        // order already puts the kept pairs first (slots 0-1 of the partner across bit 4 hold the
        // pairs of this lane's slots 2-3, and so on); lane bit 2: dB or dC; lane bit 1: low or high
#pragma unroll
        for (int i = 0; i < 8; ++i) vals[i] += __shfl_xor_sync(0xffffffffu, vals[i + 8], 16);
#pragma unroll
        for (int i = 0; i < 4; ++i) vals[i] += __shfl_xor_sync(0xffffffffu, vals[i + 4], 8);
#pragma unroll
        for (int w = 4, half = 2; w >= 2; w >>= 1, half >>= 1) {
          const bool upper = (lane & w) != 0;
#pragma unroll
          for (int i = 0; i < half; ++i) {
            const float send = upper ? vals[i] : vals[i + half];
            const float keep = upper ? vals[i + half] : vals[i];
            vals[i] = keep + __shfl_xor_sync(0xffffffffu, send, w);
          }
        }
        red[(warp * kSeg + k) * 32 + rcol] = vals[0];
      }
    }
    if (valid && pl == 0) {
      store_seg<IO, float>(p.du, off, nk, p.vec_io, gdu, Z.nIO);
      store_seg<IO, float>(p.ddelta, off, nk, p.vec_io, gdd, Z.nIO);
    }
    if (more) store_bc2(bc_base + (buf ^ 1) * (kSeg * 32), bcr);
    __syncthreads();
    pend_t0 = t0;
    pend_nk = nk;
    buf ^= 1;
  }
  if (pend_t0 >= 0) flush_red(red_base + (buf ^ 1) * (4 * kSeg * 32), pend_t0, pend_nk);
  if (valid) {
    float* accA = checked(static_cast<float*>(p.acc_dA), static_cast<int64_t>(d) * p.N, Z.nA, p.N);
#pragma unroll
    for (int j = 0; j < kP2; ++j) {
      const int n = n0 + 2 * (j ^ pm);
      if (n < p.N) atomicAdd(accA + n, dA[j].lo());
      if (n + 1 < p.N) atomicAdd(accA + n + 1, dA[j].hi());
    }
    if (pl == 0) {
      if (p.acc_dD) atomicAdd(checked(static_cast<float*>(p.acc_dD), d, Z.nDim), dD);
      if (p.acc_dbias) atomicAdd(checked(static_cast<float*>(p.acc_dbias), d, Z.nDim), dbias);
    }
  }
}

__global__ void double_to_float_kernel(const double* __restrict__ src, float* __restrict__ dst, int64_t n) {
  const int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  if (i < n) dst[i] = static_cast<float>(src[i]);
}

using BwdKernel = void (*)(BwdParams);

template <typename IO, bool kZ, bool kSp>
BwdKernel pick_fwd2_full(const BwdParams& p) {
  const bool full = p.L % kSeg == 0 && p.chunk_len % kSeg == 0;
  return full ? bwd_fwd2_kernel<IO, kZ, kSp, true> : bwd_fwd2_kernel<IO, kZ, kSp, false>;
}

template <typename IO>
BwdKernel pick_fwd2(const BwdParams& p) {
  if (p.z) return p.softplus ? pick_fwd2_full<IO, true, true>(p) : pick_fwd2_full<IO, true, false>(p);
  return p.softplus ? pick_fwd2_full<IO, false, true>(p) : pick_fwd2_full<IO, false, false>(p);
}

template <typename IO>
BwdKernel pick_rev2(const BwdParams& p) {
  if (p.z) return p.softplus ? bwd_rev2_kernel<IO, true, true> : bwd_rev2_kernel<IO, true, false>;
  return p.softplus ? bwd_rev2_kernel<IO, false, true> : bwd_rev2_kernel<IO, false, false>;
}

template <typename IO, typename CT>
cudaError_t launch(const BwdParams& p, cudaStream_t stream) {
  const dim3 grid((p.dim + kThreads - 1) / kThreads, p.batch, p.nchunks);
  const dim3 grid2((p.dim + kCh2 - 1) / kCh2, p.batch, p.nchunks);
  bool two_lanes = false;
  if constexpr (sizeof(CT) == 4) {
    if (SSM_BWD_TWO_LANES) {
      pick_fwd2<IO>(p)<<<grid2, kThreads, 0, stream>>>(p);
      two_lanes = true;
    }
  }
  if (!two_lanes) bwd_chunk_fwd_kernel<IO, CT><<<grid, kThreads, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t carry_threads = static_cast<int64_t>(p.batch) * p.dim * kN;
  bwd_carry_kernel<CT><<<static_cast<unsigned>((carry_threads + 255) / 256), 256, 0, stream>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if constexpr (sizeof(CT) == 4) {
    if (SSM_BWD_TWO_LANES) {
      auto k2 = pick_rev2<IO>(p);
      e = cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, Smem2::kTotal);
      if (e != cudaSuccess) return e;
      k2<<<grid2, kThreads, Smem2::kTotal, stream>>>(p);
      return cudaGetLastError();
    }
  }
  auto k = bwd_chunk_rev_kernel<IO, CT>;
  e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Smem<CT>::kTotal);
  if (e != cudaSuccess) return e;
  k<<<grid, kThreads, Smem<CT>::kTotal, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

int bwd_segment_steps() { return kSeg; }

int bwd_aggregate_floats() { return kAgg; }

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
    if (!q.src || !q.dst || q.n == 0) continue;
    double_to_float_kernel<<<static_cast<unsigned>((q.n + 255) / 256), 256, 0, stream>>>(
        static_cast<const double*>(q.src), q.dst, static_cast<int64_t>(q.n));
    if ((ce = cudaGetLastError()) != cudaSuccess) return ce;
  }
  return cudaSuccess;
}

cudaError_t bwd_check_read_and_clear(unsigned int* out) { return tu_check_read_and_clear(out); }

}  // namespace ssm
