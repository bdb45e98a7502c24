// Mamba-2 SSD forward on the fifth-generation tensor cores (tcgen05, accumulators in tensor memory),
// chunked block form ("Mamba и State Space Models", "Mamba-2: State Space Duality (SSD)": a scalar A per
// head, d_state 128, the SSM as a product with a semi-separable matrix; "Модуль 8. Альтернативы
// Transformer", §7: M_ij = C_i·B_j Π_{r=j+1..i} a_r as a masked matrix product inside a chunk, only the
// state passed between chunks; §14: state [batch, nheads, headdim, d_state], input term Δ·B·x):
//   y_i = Σ_{j≤i} (C_i·B_j) e^{cum_i − cum_j} Δ_j x_j + e^{cum_i} C_i·H + D_h x_i
//   H  <- e^{cum_end} H + Σ_j e^{cum_end − cum_j} Δ_j x_j B_j^T
// over chunks of 64 steps, one CTA (8 warps) per (batch, head) or per balanced range of chunks, two CTAs
// per SM.
//
// Per chunk, four tcgen05.mma groups (bf16 operands from 128-byte-swizzled shared tiles, fp32
// accumulators in tensor memory):
//   G   = C B^T          M 64 (i) x N 64 (j) x K 128 (n)   A: C [i][n] K-major, B: B [j][n] K-major
//   Yo  = C H^T          M 64 (i) x N 128 x K 128 (n)      B: H^T hi and lo tiles [n][p] (MN-major) side by
//                                                          side as one N = 128 operand; the halves are added
//                                                          when Yo is read
//   S^T = B^T (w ∘ x)    M 128 (n) x N 64 (p) x K 64 (j)   A: the same B tile read MN-major, B: (w ∘ x) [j][p]
//   Yd  = M X            M 64 (i) x N 64 (p) x K 64 (j)    A: M [i][j] K-major (hi + lo), B: x [j][p] MN-major
// The K-major 128-byte-swizzled tile of B[j][n] is byte for byte the MN-major tile of B^T, so one copy
// serves both products and nothing is transposed.  The CUDA cores do the element-wise parts: Δ and its
// prefix sum, M = G ∘ e^{cum_i − cum_j} Δ_j (causal) from the G accumulator, w ∘ x, the state update
// H = e^{cum_end} H + S^T (threads n and n + 128 own the two halves of column n of H in registers) and the
// output y.  Warps w and w + 4 share tensor-memory lane quadrant w and split the 64 accumulator columns.
// x, B, C enter the MMAs exactly (bf16 inputs) and every computed operand (M, H, w ∘ x) is split into
// two bf16 terms (about 16 significant bits), so products keep float32-level accuracy rather than
// bf16's 8 bits.
// Tensor memory: columns [0, 64) G then Yd (M = 64 rows sit in lanes 32w .. 32w + 15 of warp w),
// [64, 192) Yo (C H_hi^T then C H_lo^T), [192, 256) S^T (row n in lane n); 256 columns are allocated
// per CTA.
// Every mbarrier wait is bounded; on a timeout the CTA records it, stops and frees its tensor memory.
#include <algorithm>
#include <cstring>

#include "internal.h"
#include "scan_walk.cuh"
#include "ssm_device.cuh"

namespace ssm {
namespace {

__device__ unsigned int g_ssd_status = 0;

constexpr int kQ = 64;         // chunk length
constexpr int kHd = 64;        // head dim
constexpr int kNs = 128;       // d_state
constexpr int kThreads = 256;
constexpr uint32_t kTmemCols = 256;

// tiles (byte offsets from a 1024-byte aligned base); every tile is 128-byte swizzled
struct TcSmem {
  static constexpr int kC = 0;        // C [i][n]: 2 atoms (n 0..63, 64..127) of 64 rows x 128 B
  static constexpr int kB = 16384;    // B [j][n]: same layout
  static constexpr int kX = 32768;    // x [j][p]: 64 rows x 128 B
  static constexpr int kWh = 40960;   // (w ∘ x) hi [j][p]
  static constexpr int kWl = 49152;   // (w ∘ x) lo
  static constexpr int kMh = 57344;   // M hi [i][j]
  static constexpr int kMl = 65536;   // M lo
  static constexpr int kHh = 73728;   // H^T hi [n][p]: 128 rows x 128 B
  static constexpr int kHl = 90112;   // H^T lo
  static constexpr int kTiles = 106496;
  static constexpr int kDynamic = kTiles + 1024;
};

// byte offset of the 16-byte chunk `c` (0..7 inside a 128-byte row) of row r in a 128-byte swizzled
// tile region (rows of 128 B, 8-row groups of 1024 B)
__device__ __forceinline__ uint32_t sw_chunk(int r, int c) {
  return static_cast<uint32_t>((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

// shared-memory matrix descriptor: start, leading and stride byte offsets, version 1, 128-byte swizzle
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFF) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFF) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46) | (2ull << 61);
}
// The descriptor of a tile `off` bytes further on: the start address field holds address >> 4 in 14 bits,
// and every tile lies below 256 KB from the 1024-byte aligned base, so the field never carries.
__device__ __forceinline__ uint64_t dadd(uint64_t base, uint32_t off) { return base + (off >> 4); }
// instruction descriptor, kind::f16: fp32 accumulate, bf16 A and B, major-ness of A and B, N, M
__device__ __forceinline__ uint32_t idesc_bf16(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(a_mn) << 15) |
         (static_cast<uint32_t>(b_mn) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}
__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// 32 consecutive fp32 columns of this thread's tensor-memory lane (warp-collective)
__device__ __forceinline__ void tc_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}

// The M = 64 accumulator rows of a warp (16 rows in lanes 32q .. 32q + 15 of its lane quadrant q) in the
// m16n8 fragment layout, 32 columns from `taddr`: with g = lane / 4 and t = lane % 4, v[4r .. 4r + 3] =
// rows (g, g, g + 8, g + 8), columns (8r + 2t, 8r + 2t + 1, 8r + 2t, 8r + 2t + 1) for r = 0..3
// (warp-collective).
__device__ __forceinline__ void tc_ld_frag32(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
}

// fp32 pair -> bf16x2 hi and bf16x2 of the remainders
__device__ __forceinline__ void split2(float a, float b, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16x2(a, b);
  lo = pack_bf16x2(a - bf16lo_to_f32(hi), b - bf16hi_to_f32(hi));
}

// 8 fp32 -> the hi and lo 16-byte chunks
__device__ __forceinline__ void split8(const float* v, uint4& hi, uint4& lo) {
  split2(v[0], v[1], hi.x, lo.x);
  split2(v[2], v[3], hi.y, lo.y);
  split2(v[4], v[5], hi.z, lo.z);
  split2(v[6], v[7], hi.w, lo.w);
}

// Tensor maps of the C, B and x tiles: (batch, L, columns) with boxes of 64 columns x 64 steps, so a
// chunk's rows past L read zeros rather than the next batch row's.
struct SsdMaps {
  CUtensorMap C, B, x;
};

constexpr int kLoader = 32;   // warp 1, lane 0 issues the tile loads (thread 0 issues the MMAs)
constexpr uint64_t kCarryWaitNs = 2000000000ull;

// A sequence (batch row b, head h) of the walk and its per-head constants.
struct SsdSeq {
  int b, h, grp;
  float A2;     // A[h]·log2(e)
  float bias;   // dt_bias[h]
  float Dh;     // D[h]
};

// One CTA walks a list of (sequence, chunk) units in order: one whole sequence (kBal false: one CTA per
// sequence), or one of the equal ranges of the balanced schedule (kBal true; scan_walk.cuh: the
// sequences' chunks laid end to end, one range per resident CTA; the head of the range's last sequence
// first, its state published for the range after it, then the complete sequences, then the tail of
// the first sequence from the state the range before it published).  512 sequences of the 4 x 128-head
// layer on 296 resident CTAs are otherwise two waves, the second 73 % full.  A CTA takes its range
// index from a counter when it starts, so the range it waits for belongs to a CTA that started earlier
// and runs its head before anything it could wait for: no deadlock, whether or not every CTA is
// resident at once.
template <bool kBal>
__global__ void __launch_bounds__(kThreads, 2) ssd_tc_kernel(const __grid_constant__ SsdMaps tm, const SsdParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bars[3];
  __shared__ uint64_t tbar[3];   // the C, B and x tiles of a chunk have landed
  __shared__ uint32_t tmem_slot;
  __shared__ int s_carry_ok;
  __shared__ int s_range;
  // Δ and its prefix sum of a unit, in two buffers by unit parity: warp 0 fills the next unit's while
  // the other warps still read this unit's (no barrier at the end of a unit)
  __shared__ __align__(16) float s_dl[2][kQ];
  __shared__ __align__(16) float s_cum[2][kQ];
  const int64_t L = p.L;
  const int nchunks = static_cast<int>((L + kQ - 1) / kQ);
  const int64_t nseq = static_cast<int64_t>(p.batch) * p.nheads;
  int range = blockIdx.x;
  if (kBal) {
    if (threadIdx.x == 0) s_range = static_cast<int>(atomicAdd(p.flags + gridDim.x, 1u));
    __syncthreads();
    range = s_range;
  }
  const Walk w = kBal ? make_walk_balanced(range, p.range, nseq * nchunks, nchunks)
                      : make_walk_grid(range, 0, nchunks, nchunks);
  if (w.total() <= 0) return;
  // 1024-byte aligned tile base, derived by pointer arithmetic on the shared array so that the compiler
  // keeps shared-space loads and stores (an integer round trip would make them generic)
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(sm);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // element counts of the buffers, for the index checks of the checked build
  const int64_t nHead = p.nheads;
  const int64_t nRowX = static_cast<int64_t>(p.batch) * L * p.nheads, nX = nRowX * kHd;
  const int64_t nState = nseq * kHd * kNs;
  const int64_t nCarry = static_cast<int64_t>(gridDim.x) * kHd * kNs;
  const int hpg = p.nheads / p.ngroups;
  const __nv_bfloat16* dtg = static_cast<const __nv_bfloat16*>(p.dt);
  __nv_bfloat16* yg = static_cast<__nv_bfloat16*>(p.y);
  auto seq_of = [&](int64_t g, SsdSeq& s) {
    s.b = static_cast<int>(g / p.nheads);
    s.h = static_cast<int>(g - static_cast<int64_t>(s.b) * p.nheads);
    s.grp = s.h / hpg;
    s.A2 = *checked(p.A, s.h, nHead) * kLog2e;
    s.bias = p.dt_bias ? *checked(p.dt_bias, s.h, nHead) : 0.0f;
    s.Dh = p.D ? *checked(p.D, s.h, nHead) : 0.0f;
  };
  // The walk as segments, each one sequence's chunks [c0, c1): the head, the complete sequences, the
  // tail (any of them may be absent).
  const int64_t n_whole = w.n_full / nchunks;
  const int64_t nseg = kBal ? (w.n_head > 0 ? 1 : 0) + n_whole + (w.n_tail > 0 ? 1 : 0) : 1;
  auto seg_at = [&](int64_t si, int64_t& gs, int& c0, int& c1) {
    if (!kBal) { gs = range; c0 = 0; c1 = nchunks; return; }
    if (w.n_head > 0) {
      if (si == 0) { gs = w.g_head; c0 = 0; c1 = static_cast<int>(w.tb); return; }
      --si;
    }
    if (si < n_whole) { gs = w.gf0 + si; c0 = 0; c1 = nchunks; return; }
    gs = w.g_tail; c0 = static_cast<int>(w.ta); c1 = nchunks;
  };
  auto is_head = [&](int64_t si) { return kBal && w.n_head > 0 && si == 0; };
  auto is_tail = [&](int64_t si) { return kBal && w.n_tail > 0 && si == nseg - 1; };
  int64_t gs = 0;   // the current segment: sequence gs, chunks [c0, c1)
  int c0 = 0, c1 = 0;
  seg_at(0, gs, c0, c1);
  SsdSeq cur;
  seq_of(gs, cur);

  if (tid == 0) {
    for (int i = 0; i < 3; ++i) mbar_init(&bars[i], 1);
    for (int i = 0; i < 3; ++i) mbar_init(&tbar[i], 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_slot)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }

  // the state: thread n (< 128) holds H[p][n] for p < 32, thread n + 128 for p >= 32, in fp32
  const int quad = warp & 3, half = warp >> 2;   // tensor-memory lane quadrant and column half
  const int n_own = tid & 127;
  const int pbase = 32 * half;
  float H[kHd / 2];
  bool ok = true;
  // The state entering segment si (sequence sg): the state the previous CTA published (the tail of a
  // balanced range; zero if that wait gives up), h0 of the sequence, or zero.
  auto init_state = [&](int64_t si, int64_t sg) {
    const float* src = nullptr;
    bool carried = false;
    if (is_tail(si)) {
      if (tid == 0) {
        const unsigned* flag = checked(p.flags, static_cast<int64_t>(range) - 1, gridDim.x);
        const uint64_t limit = p.carry_wait_ns ? p.carry_wait_ns : kCarryWaitNs;
        const uint64_t t_start = globaltimer_ns();
        int got = 0;
        while (true) {
          unsigned v;
          asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
          if (v != 0u) { got = 1; break; }
          if (globaltimer_ns() - t_start > limit) break;
          __nanosleep(256);
        }
        if (!got) atomicOr(&g_ssd_status, kStatusTimeout);
        s_carry_ok = got;
      }
      __syncthreads();
      if (s_carry_ok) {
        src = p.carry + (static_cast<int64_t>(range) - 1) * kHd * kNs;
        carried = true;
      }
    } else if (p.h0) {
      src = p.h0 + sg * kHd * kNs;
    }
#pragma unroll
    for (int q = 0; q < kHd / 2; ++q) {
      const int64_t i = (pbase + q) * kNs + n_own;
      H[q] = !src ? 0.0f
                  : carried ? __ldcg(checked(src, i, nCarry - (static_cast<int64_t>(range) - 1) * kHd * kNs))
                            : *checked(src, i, nState - sg * kHd * kNs);
    }
  };
  // The state leaving segment si (sequence sg): published for the next CTA (the head of a balanced
  // range) once every thread has written its part, or written to final_state.
  auto finish_state = [&](int64_t si, int64_t sg) {
    if (is_head(si)) {
      const int64_t base = static_cast<int64_t>(range) * kHd * kNs;
#pragma unroll
      for (int q = 0; q < kHd / 2; ++q) *checked(p.carry, base + (pbase + q) * kNs + n_own, nCarry) = H[q];
      __syncthreads();
      if (tid == 0 && range != p.test_withhold_cta) {
        __threadfence();
        asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p.flags + range), "r"(1u) : "memory");
      }
    } else if (ok && p.hT) {
#pragma unroll
      for (int q = 0; q < kHd / 2; ++q) *checked(p.hT, sg * kHd * kNs + (pbase + q) * kNs + n_own, nState) = H[q];
    }
  };
  // the state tiles H^T hi and lo [n][p] the next C·H^T product reads
  auto store_state_tiles = [&](uint32_t state_off, int s3) {
#pragma unroll
    for (int c8 = 0; c8 < 4; ++c8) {
      uint4 hi, lo;
      split8(&H[c8 * 8], hi, lo);
      const uint32_t o = state_off + ((c8 ^ s3) << 4);
      *reinterpret_cast<uint4*>(sm + TcSmem::kHh + o) = hi;
      *reinterpret_cast<uint4*>(sm + TcSmem::kHl + o) = lo;
    }
  };
  const uint32_t state_off =
      static_cast<uint32_t>((n_own >> 3) * 1024 + (n_own & 7) * 128 + (((4 * half) ^ (n_own & 4)) << 4));
  const int s3 = n_own & 3;
  init_state(0, gs);
  store_state_tiles(state_off, s3);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const uint32_t t_lane = static_cast<uint32_t>(quad * 32) << 16;   // this warp's lane quadrant

  // base descriptors of the three operand layouts, built once (the MMA issue adds constant offsets)
  const uint64_t dK = sdesc(sb, 16, 1024);          // K-major tiles: C, B, M
  const uint64_t dH = sdesc(sb, 16384, 1024);       // H^T as an MN-major operand (128 rows of n)
  const uint64_t dN = sdesc(sb, kQ * 128, 1024);    // MN-major 64-row tiles: B^T, w ∘ x, x
  const uint32_t id_g = idesc_bf16(64, 64, 0, 0);
  const uint32_t id_yo = idesc_bf16(64, 128, 0, 1);   // the H^T lo tile is the next MN atom of the hi tile
  const uint32_t id_s = idesc_bf16(128, 64, 1, 1);
  const uint32_t id_yd = idesc_bf16(64, 64, 0, 1);

  // Tile loads by TMA, issued by one thread: each tile of unit k + 1 is requested as soon as the
  // tensor cores and the threads are done with that tile of unit k.  C and B are two boxes of 64
  // columns (the two 128-byte atoms of the 128 state columns), x one box of the head's 64 columns;
  // rows past L are zero-filled by the tensor map.
  auto issue_c = [&](int grp, int b, int t0) {
    mbar_arrive_expect_tx(&tbar[0], 2 * kQ * 128);
    tma_load_3d(sm + TcSmem::kC, &tm.C, &tbar[0], grp * kNs, t0, b);
    tma_load_3d(sm + TcSmem::kC + kQ * 128, &tm.C, &tbar[0], grp * kNs + 64, t0, b);
  };
  auto issue_b = [&](int grp, int b, int t0) {
    mbar_arrive_expect_tx(&tbar[1], 2 * kQ * 128);
    tma_load_3d(sm + TcSmem::kB, &tm.B, &tbar[1], grp * kNs, t0, b);
    tma_load_3d(sm + TcSmem::kB + kQ * 128, &tm.B, &tbar[1], grp * kNs + 64, t0, b);
  };
  auto issue_x = [&](int h, int b, int t0) {
    mbar_arrive_expect_tx(&tbar[2], kQ * 128);
    tma_load_3d(sm + TcSmem::kX, &tm.x, &tbar[2], h * kHd, t0, b);
  };
  // dt of the next unit is fetched as raw bf16 bits one unit ahead and only converted (softplus)
  // when that unit starts, so the load's latency is not waited for
  const unsigned short* dtr = reinterpret_cast<const unsigned short*>(dtg);
  auto load_dt_raw = [&](int b, int h, int64_t tt) -> uint32_t {
    return tt < L ? static_cast<uint32_t>(*checked(dtr, (static_cast<int64_t>(b) * L + tt) * p.nheads + h, nRowX)) : 0u;
  };
  auto dl_of = [&](uint32_t raw, int64_t tt) -> float {
    if (tt >= L) return 0.0f;
    const float v = __uint_as_float(raw << 16) + cur.bias;
    return p.softplus ? softplus_fast(v) : v;
  };
  // tiles armed per barrier (loader thread) and units whose tiles every thread has waited for
  int armed[3] = {0, 0, 0};   // (a CTA runs fewer than 2^31 units: the host keeps ranges below that)
  int started = 0;
  if (tid == kLoader) {
    prefetch_tensormap(&tm.C);
    prefetch_tensormap(&tm.B);
    prefetch_tensormap(&tm.x);
    issue_c(cur.grp, cur.b, c0 * kQ);
    issue_b(cur.grp, cur.b, c0 * kQ);
    issue_x(cur.h, cur.b, c0 * kQ);
    armed[0] = armed[1] = armed[2] = 1;
  }
  uint32_t dt_raw0 = 0u, dt_raw1 = 0u;
  if (warp == 0) {
    dt_raw0 = load_dt_raw(cur.b, cur.h, static_cast<int64_t>(c0) * kQ + 2 * lane);
    dt_raw1 = load_dt_raw(cur.b, cur.h, static_cast<int64_t>(c0) * kQ + 2 * lane + 1);
  }
  // Shared-tile offsets that are the same in every chunk.  Row r's 16-byte chunk c sits at
  // sw_chunk(r, c); for the fragment rows ri0 = 16·quad + fg (and ri1 = ri0 + 8, 1024 bytes further) and
  // chunk 4·half + rr this is frag_off + ((rr ^ (fg & 3)) << 4), for the state row n_own and chunk
  // 4·half + c8 it is state_off + ((c8 ^ (n_own & 3)) << 4) (4·half and rr occupy disjoint bits).
  const int fg = lane >> 2, ft = lane & 3;             // fragment row and column pair of this lane
  const int ri0 = quad * 16 + fg, ri1 = ri0 + 8;       // its two rows of the M = 64 results
  const uint32_t frag_off = static_cast<uint32_t>(quad * 2048 + fg * 128 + (((4 * half) ^ (fg & 4)) << 4) + 4 * ft);
  const int f3 = fg & 3;
  const int jw = tid >> 2;                             // the w ∘ x row of this thread, chunks cw and cw + 1
  const uint32_t w_off0 = sw_chunk(jw, (tid & 3) * 2), w_off1 = sw_chunk(jw, (tid & 3) * 2 + 1);
  const int64_t y_step = static_cast<int64_t>(p.nheads) * kHd;   // elements per time step of x and y
  int k = 0;   // units (chunks) run so far: the parity of every barrier phase
  for (int64_t si = 0; si < nseg && ok; ++si) {
    // the next segment, whose first chunk is requested during this segment's last one
    const bool more_seg = si + 1 < nseg;
    int64_t gs_n = gs;
    int c0_n = 0, c1_n = 0;
    SsdSeq nx = cur;
    if (more_seg) {
      seg_at(si + 1, gs_n, c0_n, c1_n);
      seq_of(gs_n, nx);
    }
    const int64_t y_base = ((static_cast<int64_t>(cur.b) * L + ri0) * p.nheads + cur.h) * kHd;
    for (int c = c0; c < c1; ++c, ++k) {
      const int64_t t0 = static_cast<int64_t>(c) * kQ;
      float* const dlb = s_dl[k & 1];
      float* const cmb = s_cum[k & 1];
      const uint32_t par = static_cast<uint32_t>(k & 1);
      // the next unit: chunk c + 1 of this sequence, or the next segment's first chunk
      const bool last = c + 1 == c1;
      const bool more = !last || more_seg;
      const int nb = last ? nx.b : cur.b, nh = last ? nx.h : cur.h, ngrp = last ? nx.grp : cur.grp;
      const int nt0 = (last ? c0_n : c + 1) * kQ;
      // ---- P0: Δ and its inclusive prefix sum over the chunk, by warp 0 (two steps per lane); the
      // chunk's tiles were requested during the previous unit
      if (warp == 0) {
        const float d0 = dl_of(dt_raw0, t0 + 2 * lane), d1 = dl_of(dt_raw1, t0 + 2 * lane + 1);
        if (more) {
          dt_raw0 = load_dt_raw(nb, nh, nt0 + 2 * lane);   // zero past L
          dt_raw1 = load_dt_raw(nb, nh, nt0 + 2 * lane + 1);
        }
        const float a0 = d0 * cur.A2;
        float s2 = a0 + d1 * cur.A2;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float u = __shfl_up_sync(0xffffffffu, s2, o);
          if (lane >= o) s2 += u;
        }
        const float before = __shfl_up_sync(0xffffffffu, s2, 1);
        const float base = lane > 0 ? before : 0.0f;
        *reinterpret_cast<float2*>(&dlb[2 * lane]) = make_float2(d0, d1);
        *reinterpret_cast<float2*>(&cmb[2 * lane]) = make_float2(base + a0, s2);
      }
      ok = ok && mbar_wait_bounded(&tbar[0], par, &g_ssd_status);
      ok = ok && mbar_wait_bounded(&tbar[1], par, &g_ssd_status);
      ok = ok && mbar_wait_bounded(&tbar[2], par, &g_ssd_status);
      started = k + 1;
      // the tiles, Δ and the H tiles of the previous unit's P3 are in place; every thread is done with
      // the previous unit's tensor memory
      fence_async_smem();
      tc_fence_before();
      ok = __syncthreads_and(ok) != 0;
      tc_fence_after();
      if (!ok) break;
      // x at this lane's fragment positions for P4's D x, bf16 pairs [r][row half], read now so that
      // the next unit's x can be requested as soon as M X is done with the tile
      uint32_t xw[8];
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) {
        const uint32_t o0 = frag_off + ((rr ^ f3) << 4);
        xw[2 * rr] = *reinterpret_cast<const uint32_t*>(sm + TcSmem::kX + o0);
        xw[2 * rr + 1] = *reinterpret_cast<const uint32_t*>(sm + TcSmem::kX + o0 + 1024);
      }

      // ---- P1: G = C B^T and Yo = C H^T on the tensor cores; meanwhile w ∘ x on the CUDA cores
      if (tid == 0) {
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t ka = (ks >> 2) * (kQ * 128) + (ks & 3) * 32;
          tc_mma(tmem + 0, dadd(dK, TcSmem::kC + ka), dadd(dK, TcSmem::kB + ka), id_g, ks > 0);
        }
        // Yo = C H^T in every chunk, a segment's first one included (its H tiles are h0, the carried
        // state or zero): one fewer run-time branch in the issue and output phases (0.548 -> 0.540 ms,
        // outputs identical)
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t ka = (ks >> 2) * (kQ * 128) + (ks & 3) * 32;
          tc_mma(tmem + 64, dadd(dK, TcSmem::kC + ka), dadd(dH, TcSmem::kHh + ks * 2048), id_yo, ks > 0);
        }
        tc_commit(&bars[0]);
      }
      const float cum_end = cmb[kQ - 1];
      {
        const float wj = ex2_approx(cum_end - cmb[jw]) * dlb[jw];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const uint32_t o = q ? w_off1 : w_off0;
          float v[8];
          unpack_chunk(*reinterpret_cast<const uint4*>(sm + TcSmem::kX + o), v, __nv_bfloat16());
#pragma unroll
          for (int e = 0; e < 8; ++e) v[e] *= wj;
          uint4 hi, lo;
          split8(v, hi, lo);
          *reinterpret_cast<uint4*>(sm + TcSmem::kWh + o) = hi;
          *reinterpret_cast<uint4*>(sm + TcSmem::kWl + o) = lo;
        }
      }
      fence_async_smem();
      tc_fence_before();
      __syncthreads();
      tc_fence_after();

      // ---- P2: S^T = B^T (w ∘ x) on the tensor cores; M = G ∘ e^{cum_i − cum_j} Δ_j on the CUDA cores
      if (tid == 0) {
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          tc_mma(tmem + 192, dadd(dN, TcSmem::kB + ks * 2048), dadd(dN, TcSmem::kWh + ks * 2048), id_s, ks > 0);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          tc_mma(tmem + 192, dadd(dN, TcSmem::kB + ks * 2048), dadd(dN, TcSmem::kWl + ks * 2048), id_s, 1);
        tc_commit(&bars[1]);
      }
      ok = mbar_wait_bounded(&bars[0], par, &g_ssd_status);
      ok = __all_sync(0xffffffffu, ok);   // the tensor-memory loads below are warp-collective
      tc_fence_after();
      if (tid == kLoader && more) {   // G and Yo are done with C
        issue_c(ngrp, nb, nt0);
        ++armed[0];
      }
      // The element-wise phases run whether or not the wait before them succeeded: after a failed
      // wait they read allocated tensor memory and write in-bounds shared and global memory (y is
      // undefined once the status word reports a timeout), and the loop leaves at the next barrier.
      // Without the run-time branches around them: 0.540 -> 0.527 ms.
      {
        const float cr0 = cmb[ri0], cr1 = cmb[ri1];
        float gv[16];
        tc_ld_frag32(tmem + t_lane + pbase, gv);
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) {
          const int r = 4 * half + rr;                     // 16-byte column chunk of the row
          const int j = 8 * r + 2 * ft;
          const float2 cj = *reinterpret_cast<const float2*>(&cmb[j]);
          const float2 dj = *reinterpret_cast<const float2*>(&dlb[j]);
          const float m00 = j <= ri0 ? gv[4 * rr] * ex2_approx(cr0 - cj.x) * dj.x : 0.0f;
          const float m01 = j + 1 <= ri0 ? gv[4 * rr + 1] * ex2_approx(cr0 - cj.y) * dj.y : 0.0f;
          const float m10 = j <= ri1 ? gv[4 * rr + 2] * ex2_approx(cr1 - cj.x) * dj.x : 0.0f;
          const float m11 = j + 1 <= ri1 ? gv[4 * rr + 3] * ex2_approx(cr1 - cj.y) * dj.y : 0.0f;
          uint32_t hi, lo;
          const uint32_t o0 = frag_off + ((rr ^ f3) << 4), o1 = o0 + 1024;
          split2(m00, m01, hi, lo);
          *reinterpret_cast<uint32_t*>(sm + TcSmem::kMh + o0) = hi;
          *reinterpret_cast<uint32_t*>(sm + TcSmem::kMl + o0) = lo;
          split2(m10, m11, hi, lo);
          *reinterpret_cast<uint32_t*>(sm + TcSmem::kMh + o1) = hi;
          *reinterpret_cast<uint32_t*>(sm + TcSmem::kMl + o1) = lo;
        }
      }
      fence_async_smem();
      tc_fence_before();
      ok = __syncthreads_and(ok) != 0;
      tc_fence_after();
      if (!ok) break;

      // ---- P3: Yd = M X on the tensor cores; the state update on the CUDA cores
      if (tid == 0) {
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          tc_mma(tmem + 0, dadd(dK, TcSmem::kMh + ks * 32), dadd(dN, TcSmem::kX + ks * 2048),
                 id_yd, ks > 0);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          tc_mma(tmem + 0, dadd(dK, TcSmem::kMl + ks * 32), dadd(dN, TcSmem::kX + ks * 2048),
                 id_yd, 1);
        tc_commit(&bars[2]);
      }
      ok = mbar_wait_bounded(&bars[1], par, &g_ssd_status);
      ok = __all_sync(0xffffffffu, ok);   // the tensor-memory loads below are warp-collective
      tc_fence_after();
      if (tid == kLoader && more) {   // G and S^T are done with B
        issue_b(ngrp, nb, nt0);
        ++armed[1];
      }
      {
        const float eE = ex2_approx(cum_end);
        float s[32];
        tc_ld32(tmem + t_lane + 192 + pbase, s);
#pragma unroll
        for (int q = 0; q < 32; ++q) H[q] = fmaf(eE, H[q], s[q]);
      }
      store_state_tiles(state_off, s3);
      // every thread read x before P2's barrier (w ∘ x, xw); once M X is done the tile is free (a
      // failed wait leaves the next x unrequested: the next unit's tile wait then gives up)
      if (tid == kLoader && more && mbar_wait_bounded(&bars[2], par, &g_ssd_status)) {
        fence_async_smem();
        issue_x(nh, nb, nt0);
        ++armed[2];
      }

      // ---- P4: y = Yd + e^{cum_i} Yo + D x
      ok = ok && mbar_wait_bounded(&bars[2], par, &g_ssd_status);
      ok = __all_sync(0xffffffffu, ok);   // the tensor-memory loads below are warp-collective
      tc_fence_after();
      {
        const float e0 = ex2_approx(cmb[ri0]), e1 = ex2_approx(cmb[ri1]);
        float yd[16], yo[16];
        tc_ld_frag32(tmem + t_lane + pbase, yd);
        {
          float yl[16];
          tc_ld_frag32(tmem + t_lane + 64 + pbase, yo);
          tc_ld_frag32(tmem + t_lane + 128 + pbase, yl);
#pragma unroll
          for (int q = 0; q < 16; ++q) yo[q] += yl[q];
        }
        const int64_t y0 = y_base + t0 * y_step, y1 = y0 + 8 * y_step;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int pc = pbase + 8 * r + 2 * ft;
          float v00 = yd[4 * r] + cur.Dh * bf16lo_to_f32(xw[2 * r]);
          float v01 = yd[4 * r + 1] + cur.Dh * bf16hi_to_f32(xw[2 * r]);
          float v10 = yd[4 * r + 2] + cur.Dh * bf16lo_to_f32(xw[2 * r + 1]);
          float v11 = yd[4 * r + 3] + cur.Dh * bf16hi_to_f32(xw[2 * r + 1]);
          v00 = fmaf(e0, yo[4 * r], v00);
          v01 = fmaf(e0, yo[4 * r + 1], v01);
          v10 = fmaf(e1, yo[4 * r + 2], v10);
          v11 = fmaf(e1, yo[4 * r + 3], v11);
          if (t0 + ri0 < L) *reinterpret_cast<uint32_t*>(checked(yg, y0 + pc, nX, 2)) = pack_bf16x2(v00, v01);
          if (t0 + ri1 < L) *reinterpret_cast<uint32_t*>(checked(yg, y1 + pc, nX, 2)) = pack_bf16x2(v10, v11);
        }
      }
    }
    // CTA-uniform from here: the barriers of the segment switch below
    ok = __syncthreads_and(ok) != 0;
    if (!ok) break;
    // The segment ends: its state leaves, the next segment's state replaces it in the H tiles (read
    // first by the next chunk's C·H^T, after that chunk's barrier and proxy fence).  Kept out of the
    // chunk loop so that its straight-line phases are not split at a branch (CTA-uniform: every thread
    // reaches the barriers inside).
    finish_state(si, gs);
    if (more_seg) {
      init_state(si + 1, gs_n);
      store_state_tiles(state_off, s3);
    }
    gs = gs_n;
    c0 = c0_n;
    c1 = c1_n;
    cur = nx;
  }
  // every tile load the loader requested has landed before the CTA's shared memory is released (a
  // loop left after a failed wait may have loads in flight)
  if (tid == kLoader) {
    for (int i = 0; i < 3; ++i)
      for (int k = started; k < armed[i]; ++k)
        (void)mbar_wait_bounded(&tbar[i], static_cast<uint32_t>(k & 1), &g_ssd_status, 100000000ull);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
}

}  // namespace

int ssd_head_dim() { return kHd; }
int ssd_state_dim() { return kNs; }

static cudaError_t set_smem_attributes() {
  for (const void* k : {reinterpret_cast<const void*>(ssd_tc_kernel<false>),
                        reinterpret_cast<const void*>(ssd_tc_kernel<true>)}) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, TcSmem::kDynamic);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// CTAs of the SSD kernel that fit on the current device at once, from its registers, shared memory and
// threads per SM and the tensor-memory columns each CTA allocates (512 per SM).  The runtime's
// occupancy query reports one CTA per SM for this kernel (measured on a B300, even with no dynamic
// shared memory), while two run side by side (the time of 296 sequences is 1.3 times that of 148); the
// balanced schedule does not depend on the number for correctness.
int ssd_resident_ctas() {
  static int cached[64] = {0};
  int dev = 0, sms = 0, smem = 0, reserved = 0, regs = 0, threads = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return 0; }
  if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
  cudaFuncAttributes fa;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&regs, cudaDevAttrMaxRegistersPerMultiprocessor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&threads, cudaDevAttrMaxThreadsPerMultiProcessor, dev) != cudaSuccess ||
      cudaFuncGetAttributes(&fa, ssd_tc_kernel<true>) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  const int warps = kThreads / 32;
  const int regs_per_warp = (fa.numRegs * 32 + 255) / 256 * 256;   // allocated per warp in units of 256
  int per_sm = 512 / static_cast<int>(kTmemCols);
  per_sm = std::min(per_sm, smem / (TcSmem::kDynamic + static_cast<int>(fa.sharedSizeBytes) + reserved));
  per_sm = std::min(per_sm, regs / (warps * regs_per_warp));
  per_sm = std::min(per_sm, threads / kThreads);
  per_sm = std::min(per_sm, 2);   // the kernel's launch bounds
  if (per_sm < 1) per_sm = 1;
  if (dev >= 0 && dev < 64) cached[dev] = per_sm * sms;
  return per_sm * sms;
}

cudaError_t ssd_fwd_launch(const SsdParams& p, int balanced_ctas, cudaStream_t stream) {
  if (p.L > 0x7fffffffLL) return cudaErrorInvalidValue;   // TMA row coordinates are 32-bit
  SsdMaps tm;
  memset(&tm, 0, sizeof(tm));
  char err[160];
  const uint64_t L = static_cast<uint64_t>(p.L), bcw = static_cast<uint64_t>(p.ngroups) * kNs,
                 xw = static_cast<uint64_t>(p.nheads) * kHd;
  if (!encode_tensor_map_3d(&tm.C, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<void*>(p.C), bcw, L, p.batch, bcw * 2,
                            L * bcw * 2, 64, kQ, err, sizeof(err)) ||
      !encode_tensor_map_3d(&tm.B, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<void*>(p.B), bcw, L, p.batch, bcw * 2,
                            L * bcw * 2, 64, kQ, err, sizeof(err)) ||
      !encode_tensor_map_3d(&tm.x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<void*>(p.x), xw, L, p.batch, xw * 2,
                            L * xw * 2, 64, kQ, err, sizeof(err))) {
    set_last_error("ssd tensor maps: %s", err);
    return cudaErrorInvalidValue;
  }
  cudaError_t e = set_smem_attributes();
  if (e != cudaSuccess) return e;
  if (p.balanced) {
    // the publication flags and the range counter after them start at zero
    e = cudaMemsetAsync(p.flags, 0, sizeof(unsigned) * (balanced_ctas + 1), stream);
    if (e != cudaSuccess) return e;
    ssd_tc_kernel<true><<<balanced_ctas, kThreads, TcSmem::kDynamic, stream>>>(tm, p);
    return cudaGetLastError();
  }
  const int64_t nseq = static_cast<int64_t>(p.batch) * p.nheads;
  if (nseq > 0x7fffffffLL) return cudaErrorInvalidValue;
  ssd_tc_kernel<false><<<static_cast<unsigned>(nseq), kThreads, TcSmem::kDynamic, stream>>>(tm, p);
  return cudaGetLastError();
}

cudaError_t ssd_status_read_and_clear(unsigned int* out) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_ssd_status, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_ssd_status, &zero, sizeof(unsigned int));
}

cudaError_t ssd_check_read_and_clear(unsigned int* out) { return tu_check_read_and_clear(out); }

}  // namespace ssm
