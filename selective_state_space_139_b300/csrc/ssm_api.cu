// C ABI of libssm_b300.so (declared in include/ssm.h): argument checks, algorithm choice,
// workspace layout, TMA tensor-map encoding and dispatch to the kernels.  Every check runs on the
// host before anything is enqueued.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "ssm.h"

namespace {

thread_local char g_err[512] = {0};

// One-shot diagnostic of the balanced schedule's carry wait (ssm_selftest_withhold_carry).
struct Withhold {
  bool armed = false;
  int cta = -1;
  int64_t limit_ns = 0;
};
thread_local Withhold g_withhold;

ssm_status fail(ssm_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return s;
}

ssm_status cuda_fail(cudaError_t e, const char* what) {
  return fail(SSM_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#ifndef SSM_BWD_TILES_PER_SM
#define SSM_BWD_TILES_PER_SM 24   // backward: (channel group, chunk) tiles to aim for per SM
#endif

constexpr int kChannelsPerCta = 128;
constexpr int64_t kMinChunkTiles = 4;

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct Range {
  uintptr_t lo, hi;
};
Range range_of(const void* p, size_t bytes) {
  uintptr_t a = reinterpret_cast<uintptr_t>(p);
  return {a, a + bytes};
}
bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi && a.lo != a.hi && b.lo != b.hi; }

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 148;
  }
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    return 148;
  }
  return n;
}

struct Plan {
  int path = 0;           // 0: general kernel (float32 io, layouts TMA cannot describe); 1: bf16 fast path
  int nchunks = 1;
  int64_t chunk_len = 0;
  int balanced_ctas = 0;  // fast path: > 0 selects the balanced persistent schedule
  int64_t range_tiles = 0;
  size_t workspace = 0;
  size_t off_P = 0, off_Q = 0, off_hin = 0;
  size_t off_carry = 0, off_flags = 0;
};

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// The balanced schedule of the SSD forward (ssd_tc.cu) for these sizes: CTAs (0: one CTA per
// sequence, when the sequences fit in one wave of resident CTAs or no workspace is given), units of
// (sequence, 64-step chunk) per CTA, and the workspace: the ranges' carried states, then their flags
// and the range counter.
struct SsdPlan {
  int ctas = 0;
  int64_t range = 0;
  size_t carry = 0, workspace = 0;
};
SsdPlan ssd_plan(int batch, int nheads, int64_t seqlen, int ctas) {
  SsdPlan pl;
  if (seqlen <= 0) return pl;
  const int64_t nseq = static_cast<int64_t>(batch) * nheads;
  const int64_t nchunks = (seqlen + 63) / 64;
  const int64_t slots = ssm::ssd_resident_ctas();
  const int64_t G = ctas > 0 ? std::min<int64_t>(ctas, slots) : slots;
  if (G <= 0 || G >= nseq) return pl;
  // G < nseq, so every range is longer than a sequence: a CTA's tail never waits for long
  const int64_t total = nseq * nchunks;
  pl.range = (total + G - 1) / G;
  if (pl.range > (1LL << 30)) return SsdPlan();   // a CTA counts its units in 32 bits
  pl.ctas = static_cast<int>((total + pl.range - 1) / pl.range);
  pl.carry = round_up(static_cast<size_t>(pl.ctas) * ssm::ssd_head_dim() * ssm::ssd_state_dim() * sizeof(float), 256);
  pl.workspace = pl.carry + round_up(static_cast<size_t>(pl.ctas + 1) * sizeof(unsigned), 256);
  return pl;
}

// The bf16 fast path needs: bf16 io, the Δ·B or the exact-ZOH input term, rows TMA can describe (L a
// multiple of 8, at least one 64-step tile, at least 128 rows).  Pointer alignment is checked at call
// time.
bool fast_eligible(int batch, int dim, int64_t seqlen, ssm_dtype io, int disc) {
  return io == SSM_BF16 && (disc == SSM_DISC_DELTA_B || disc == SSM_DISC_ZOH) && seqlen % 8 == 0 &&
         seqlen >= 64 && static_cast<int64_t>(batch) * dim >= 128;
}

void layout_chunked(Plan* pl, int batch, int dim, int dstate, size_t carry_bytes) {
  const size_t per_chunk = static_cast<size_t>(batch) * dim * dstate * carry_bytes;
  pl->off_P = 0;
  pl->off_Q = round_up(per_chunk * (pl->nchunks - 1), 256);
  pl->off_hin = pl->off_Q + round_up(per_chunk * (pl->nchunks - 1), 256);
  pl->workspace = pl->off_hin + round_up(per_chunk * pl->nchunks, 256);
}

// The chunk length (a multiple of 64, at least 256; 0 = one pass) that minimises the estimated
// time of the grid and chunked schedules for G channel groups on `slots` co-resident CTAs: time in
// units of one CTA running one step of its group, the main pass taking ceil(G n / slots) waves of a
// chunk plus a pipeline fill of about one tile per wave, the aggregate pass (no readout, no outputs)
// about 0.6 of that.  With need_chunks, at least two chunks.
int64_t best_chunk(int64_t G, int64_t slots, int64_t seqlen, bool need_chunks) {
  const int64_t Lt = (seqlen + 63) / 64;
  double best = 0.0;
  int64_t best_c = 0;
  for (int64_t n = need_chunks ? 2 : 1; n <= Lt && n <= 65535; ++n) {
    const int64_t c = static_cast<int64_t>(round_up(static_cast<size_t>((seqlen + n - 1) / n), 64));
    const int64_t nn = (seqlen + c - 1) / c;
    if (nn != n) continue;   // the same chunk length as a smaller n
    if (nn > 1 && c < 256) break;
    const double main = static_cast<double>((G * nn + slots - 1) / slots) * (c + 64);
    const double agg = nn > 1 ? 0.6 * static_cast<double>((G * (nn - 1) + slots - 1) / slots) * (c + 64) : 0.0;
    const double t = main + agg;
    if (best_c == 0 || t < best * 0.999) {
      best = t;
      best_c = nn > 1 ? c : -1;
    }
  }
  return best_c > 0 ? best_c : 0;
}

// Decides the kernel path and schedule and lays out the workspace.  Returns false on bad options.
bool make_plan(int batch, int dim, int dstate, int64_t seqlen, ssm_dtype io, const ssm_scan_options* o, Plan* pl) {
  const int algo = o ? o->algorithm : SSM_ALGO_AUTO;
  const int disc = o ? o->discretization : SSM_DISC_DELTA_B;
  if (algo != SSM_ALGO_AUTO && algo != SSM_ALGO_SINGLE_PASS && algo != SSM_ALGO_CHUNKED) return false;
  int64_t user_chunk = 0;
  if (algo == SSM_ALGO_CHUNKED) {
    user_chunk = o->chunk_len;
    if (user_chunk < 0 || user_chunk % 64 != 0) return false;
  }
  const int sms = sm_count();
  *pl = Plan();
  if (fast_eligible(batch, dim, seqlen, io, disc)) {
    // rescaled-state kernel: the balanced schedule when there are at least as many 128-channel
    // groups as resident CTAs, otherwise one pass per group or time chunks, whichever the wave
    // count makes faster
    pl->path = 1;
    const int64_t cpc = ssm::scaled_channels_per_cta();
    const int64_t G = static_cast<int64_t>(batch) * ((dim + cpc - 1) / cpc);
    const int64_t Lt = (seqlen + 63) / 64;
    const int64_t S = ssm::scaled_resident_ctas();   // 0 when unknown (no device)
    if (algo == SSM_ALGO_AUTO && S > 0 && G >= S) {
      pl->balanced_ctas = static_cast<int>(S);
      pl->range_tiles = (G * Lt + S - 1) / S;
      pl->nchunks = 1;
      pl->chunk_len = seqlen;
      pl->off_carry = 0;
      pl->off_flags = round_up(static_cast<size_t>(S) * cpc * 16 * sizeof(float), 256);
      pl->workspace = pl->off_flags + round_up(static_cast<size_t>(S) * sizeof(unsigned), 256);
      return true;
    }
    int64_t chunk = 0;
    if (algo == SSM_ALGO_CHUNKED && user_chunk > 0) {
      chunk = user_chunk;
    } else if (algo != SSM_ALGO_SINGLE_PASS) {
      chunk = best_chunk(G, S > 0 ? S : sms, seqlen, algo == SSM_ALGO_CHUNKED);
    }
    if (chunk > 0 && (seqlen + chunk - 1) / chunk > 65535)
      chunk = round_up(static_cast<size_t>((seqlen + 65534) / 65535), 64);
    if (chunk <= 0 || chunk >= seqlen) {
      pl->nchunks = 1;
      pl->chunk_len = seqlen;
      pl->workspace = 0;
      return true;
    }
    pl->chunk_len = chunk;
    pl->nchunks = static_cast<int>((seqlen + chunk - 1) / chunk);
    layout_chunked(pl, batch, dim, dstate, sizeof(float));
    return true;
  }
  // general kernel
  pl->path = 0;
  const int T = ssm::scan_tile_steps(io == SSM_BF16 ? 2 : 4);
  const int64_t groups = static_cast<int64_t>(batch) * ((dim + kChannelsPerCta - 1) / kChannelsPerCta);
  int64_t chunk = 0;
  if (algo == SSM_ALGO_CHUNKED) {
    chunk = user_chunk;
    if (chunk == 0) {
      const int64_t target = std::max<int64_t>(2, (4 * sms + groups - 1) / groups);
      chunk = round_up(static_cast<size_t>((seqlen + target - 1) / target), 64);
    }
  } else if (algo == SSM_ALGO_AUTO) {
    if (groups < sms && seqlen >= 2 * kMinChunkTiles * T) {
      const int64_t target = (4 * sms + groups - 1) / groups;
      int64_t c = round_up(static_cast<size_t>((seqlen + target - 1) / target), 64);
      c = std::max<int64_t>(c, kMinChunkTiles * 64);
      if (c < seqlen) chunk = c;
    }
  }
  // grid.z holds the chunk index: keep the chunk count within 65535
  if (chunk > 0 && (seqlen + chunk - 1) / chunk > 65535)
    chunk = round_up(static_cast<size_t>((seqlen + 65534) / 65535), 64);
  if (chunk <= 0 || chunk >= seqlen) {
    pl->nchunks = 1;
    pl->chunk_len = seqlen;
    pl->workspace = 0;
    return true;
  }
  pl->chunk_len = chunk;
  pl->nchunks = static_cast<int>((seqlen + chunk - 1) / chunk);
  // float32 io keeps its chunk carries in double (see the float32-io note in scan_fwd.cu)
  layout_chunked(pl, batch, dim, dstate, io == SSM_F32 ? sizeof(double) : sizeof(float));
  return true;
}

bool sizes_ok(int batch, int dim, int dstate, int64_t seqlen, ssm_dtype io) {
  return batch >= 1 && dim >= 1 && dstate >= 1 && dstate <= 16 && seqlen >= 0 && (io == SSM_F32 || io == SSM_BF16);
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    else
      cudaGetLastError();
  });
  return fn;
}

}  // namespace

namespace ssm {

void set_last_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
}

bool encode_tensor_map_2d(CUtensorMap* map, CUtensorMapDataType dtype, void* base, uint64_t inner, uint64_t rows,
                          uint64_t row_pitch_bytes, uint32_t box_inner, uint32_t box_rows, char* err,
                          size_t errlen) {
  auto enc = tensor_map_encoder();
  if (!enc) {
    snprintf(err, errlen, "cuTensorMapEncodeTiled is not available");
    return false;
  }
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {row_pitch_bytes};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, dtype, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(err, errlen, "cuTensorMapEncodeTiled failed with %d", static_cast<int>(r));
    return false;
  }
  return true;
}

bool encode_tensor_map_3d(CUtensorMap* map, CUtensorMapDataType dtype, void* base, uint64_t inner, uint64_t rows,
                          uint64_t outer, uint64_t row_pitch_bytes, uint64_t outer_pitch_bytes, uint32_t box_inner,
                          uint32_t box_rows, char* err, size_t errlen) {
  auto enc = tensor_map_encoder();
  if (!enc) {
    snprintf(err, errlen, "cuTensorMapEncodeTiled is not available");
    return false;
  }
  const cuuint64_t dims[3] = {inner, rows, outer};
  const cuuint64_t strides[2] = {row_pitch_bytes, outer_pitch_bytes};
  const cuuint32_t box[3] = {box_inner, box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, dtype, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(err, errlen, "cuTensorMapEncodeTiled failed with %d", static_cast<int>(r));
    return false;
  }
  return true;
}

}  // namespace ssm

extern "C" {

int ssm_abi_version(void) { return 1; }

int ssm_checked_build(void) { return SSM_CHECK ? 1 : 0; }

const char* ssm_status_string(ssm_status s) {
  switch (s) {
    case SSM_OK: return "SSM_OK";
    case SSM_ERR_INVALID_ARG: return "SSM_ERR_INVALID_ARG";
    case SSM_ERR_UNSUPPORTED: return "SSM_ERR_UNSUPPORTED";
    case SSM_ERR_CUDA: return "SSM_ERR_CUDA";
    case SSM_ERR_TIMEOUT: return "SSM_ERR_TIMEOUT";
    case SSM_ERR_CHECK: return "SSM_ERR_CHECK";
  }
  return "SSM_ERR_UNKNOWN";
}

const char* ssm_last_error_message(void) { return g_err; }

size_t ssm_scan_fwd_workspace_size_ex(int batch, int dim, int dstate, int64_t seqlen, ssm_dtype io_dtype,
                                      const ssm_scan_options* opts) {
  if (!sizes_ok(batch, dim, dstate, seqlen, io_dtype)) return 0;
  if (opts && opts->struct_size != static_cast<int>(sizeof(ssm_scan_options))) return 0;
  Plan pl;
  if (!make_plan(batch, dim, dstate, seqlen, io_dtype, opts, &pl)) return 0;
  return pl.workspace;
}

ssm_status ssm_scan_fwd_describe(int batch, int dim, int dstate, int64_t seqlen, ssm_dtype io_dtype,
                                 const ssm_scan_options* opts, ssm_scan_plan* plan) {
  g_err[0] = 0;
  if (!plan || plan->struct_size != static_cast<int>(sizeof(ssm_scan_plan)))
    return fail(SSM_ERR_INVALID_ARG, "ssm_scan_plan.struct_size mismatch");
  if (io_dtype != SSM_F32 && io_dtype != SSM_BF16) return fail(SSM_ERR_INVALID_ARG, "unknown io_dtype %d", io_dtype);
  if (batch < 1 || dim < 1 || seqlen < 0 || dstate < 1) return fail(SSM_ERR_INVALID_ARG, "bad sizes");
  if (dstate > 16) return fail(SSM_ERR_UNSUPPORTED, "dstate=%d > 16 is not supported", dstate);
  if (opts && opts->struct_size != static_cast<int>(sizeof(ssm_scan_options)))
    return fail(SSM_ERR_INVALID_ARG, "ssm_scan_options.struct_size mismatch");
  Plan pl;
  if (!make_plan(batch, dim, dstate, seqlen, io_dtype, opts, &pl))
    return fail(SSM_ERR_INVALID_ARG, "bad algorithm or chunk_len (a multiple of 64 is required)");
  plan->path = pl.path;
  plan->nchunks = pl.nchunks;
  plan->chunk_len = pl.chunk_len;
  plan->workspace_bytes = pl.workspace;
  const int64_t cpc = pl.path == 1 ? ssm::scaled_channels_per_cta() : kChannelsPerCta;
  const int64_t groups = static_cast<int64_t>(batch) * ((dim + cpc - 1) / cpc);
  if (pl.balanced_ctas > 0) {
    plan->schedule = 1;
    plan->ctas = pl.balanced_ctas;
    plan->kernel_launches = 1;
  } else if (pl.nchunks > 1) {
    plan->schedule = 2;
    plan->ctas = static_cast<int>(groups * pl.nchunks);
    plan->kernel_launches = 3;
  } else {
    plan->schedule = 0;
    plan->ctas = static_cast<int>(groups);
    plan->kernel_launches = seqlen > 0 ? 1 : 0;
  }
  return SSM_OK;
}

size_t ssm_scan_fwd_workspace_size(int batch, int dim, int dstate, int64_t seqlen, ssm_dtype io_dtype) {
  return ssm_scan_fwd_workspace_size_ex(batch, dim, dstate, seqlen, io_dtype, nullptr);
}

ssm_status ssm_scan_fwd_ex(const void* u, const void* delta, const float* A, const void* B, const void* C,
                           const float* D, const void* z, const float* delta_bias, int softplus_flag, void* y,
                           float* last_state, int batch, int dim, int dstate, int64_t seqlen, ssm_dtype io_dtype,
                           void* workspace, size_t workspace_bytes, const ssm_scan_options* opts,
                           cudaStream_t stream) {
  g_err[0] = 0;
  if (io_dtype != SSM_F32 && io_dtype != SSM_BF16) return fail(SSM_ERR_INVALID_ARG, "unknown io_dtype %d", io_dtype);
  if (batch < 1 || dim < 1 || seqlen < 0 || dstate < 1)
    return fail(SSM_ERR_INVALID_ARG, "bad sizes batch=%d dim=%d dstate=%d seqlen=%lld", batch, dim, dstate,
                static_cast<long long>(seqlen));
  if (dstate > 16) return fail(SSM_ERR_UNSUPPORTED, "dstate=%d > 16 is not supported", dstate);
  if (seqlen > (int64_t(1) << 32)) return fail(SSM_ERR_UNSUPPORTED, "seqlen above 2^32 is not supported");
  if (batch > 65535) return fail(SSM_ERR_UNSUPPORTED, "batch=%d above 65535 is not supported", batch);
  if (opts && opts->struct_size != static_cast<int>(sizeof(ssm_scan_options)))
    return fail(SSM_ERR_INVALID_ARG, "ssm_scan_options.struct_size mismatch");
  const int disc = opts ? opts->discretization : SSM_DISC_DELTA_B;
  if (disc != SSM_DISC_DELTA_B && disc != SSM_DISC_ZOH)
    return fail(SSM_ERR_INVALID_ARG, "unknown discretization %d", disc);
  const float* h0 = opts ? opts->h0 : nullptr;
  if (seqlen > 0 && (!u || !delta || !A || !B || !C || !y))
    return fail(SSM_ERR_INVALID_ARG, "null required pointer (u, delta, A, B, C, y)");
  const size_t e = io_dtype == SSM_BF16 ? 2 : 4;
  const void* io_ptrs[] = {u, delta, z, B, C, y};
  for (const void* p : io_ptrs)
    if (p && !aligned(p, e)) return fail(SSM_ERR_INVALID_ARG, "io pointer not aligned to its element size");
  const void* f_ptrs[] = {A, D, delta_bias, last_state, h0};
  for (const void* p : f_ptrs)
    if (p && !aligned(p, 4)) return fail(SSM_ERR_INVALID_ARG, "float32 pointer not 4-byte aligned");
  Plan pl;
  if (!make_plan(batch, dim, dstate, seqlen, io_dtype, opts, &pl))
    return fail(SSM_ERR_INVALID_ARG, "bad algorithm or chunk_len (a multiple of 64 is required)");

  const size_t bdl = static_cast<size_t>(batch) * dim * seqlen * e;
  const size_t bnl = static_cast<size_t>(batch) * dstate * seqlen * e;
  const size_t st = static_cast<size_t>(batch) * dim * dstate * 4;
  const Range outs[] = {range_of(y, bdl), range_of(last_state, last_state ? st : 0)};
  const Range ins[] = {range_of(u, bdl), range_of(delta, bdl), range_of(z, z ? bdl : 0), range_of(B, bnl),
                       range_of(C, bnl), range_of(A, static_cast<size_t>(dim) * dstate * 4),
                       range_of(D, D ? dim * 4 : 0), range_of(delta_bias, delta_bias ? dim * 4 : 0),
                       range_of(h0, h0 ? st : 0)};
  for (const Range& o : outs)
    for (const Range& i : ins)
      if (overlap(o, i)) return fail(SSM_ERR_INVALID_ARG, "an output overlaps an input");
  if (y && last_state && overlap(outs[0], outs[1])) return fail(SSM_ERR_INVALID_ARG, "y overlaps last_state");
  if (pl.workspace > 0) {
    if (!workspace || workspace_bytes < pl.workspace)
      return fail(SSM_ERR_INVALID_ARG, "workspace of %zu bytes required, %zu given", pl.workspace, workspace_bytes);
    if (!aligned(workspace, 256)) return fail(SSM_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    const Range w = range_of(workspace, pl.workspace);
    for (const Range& i : ins)
      if (overlap(w, i)) return fail(SSM_ERR_INVALID_ARG, "workspace overlaps an input");
    for (const Range& o : outs)
      if (overlap(w, o)) return fail(SSM_ERR_INVALID_ARG, "workspace overlaps an output");
  }

  if (seqlen == 0) {
    // no steps: the final state is the initial state
    if (last_state) {
      cudaError_t ce = h0 ? cudaMemcpyAsync(last_state, h0, st, cudaMemcpyDeviceToDevice, stream)
                          : cudaMemsetAsync(last_state, 0, st, stream);
      if (ce != cudaSuccess) return cuda_fail(ce, "seqlen 0 state copy");
    }
    return SSM_OK;
  }

  ssm::ScanParams p;
  memset(&p, 0, sizeof(p));
  p.u = u; p.delta = delta; p.z = z; p.B = B; p.C = C; p.A = A; p.D = D; p.bias = delta_bias;
  p.y = y; p.last_state = last_state; p.h0 = h0;
  p.batch = batch; p.dim = dim; p.N = dstate; p.L = seqlen;
  p.softplus = softplus_flag != 0; p.disc = disc; p.io_bf16 = io_dtype == SSM_BF16;
  bool aligned16 = true;
  for (const void* q : {u, delta, z, B, C, static_cast<const void*>(y)})
    if (q && !aligned(q, 16)) aligned16 = false;
  p.test_withhold_cta = -1;
  p.carry_wait_ns = 0;
  if (g_withhold.armed) {
    // one-shot diagnostic armed by ssm_selftest_withhold_carry on this host thread
    p.test_withhold_cta = g_withhold.cta;
    p.carry_wait_ns = static_cast<uint64_t>(g_withhold.limit_ns);
    g_withhold.armed = false;
  }
  char err[256] = {0};
  char* ws = static_cast<char*>(workspace);
  if (pl.path == 1 && aligned16) {
    if (pl.balanced_ctas > 0) {
      p.sched_balanced = 1;
      p.range_tiles = pl.range_tiles;
      p.carry = reinterpret_cast<float*>(ws + pl.off_carry);
      p.flags = reinterpret_cast<unsigned*>(ws + pl.off_flags);
      p.chunk_len = seqlen;
    } else if (pl.nchunks > 1) {
      p.agg_P = ws + pl.off_P;
      p.agg_Q = ws + pl.off_Q;
      p.h_in = ws + pl.off_hin;
      p.h_in_chunk_stride = static_cast<int64_t>(batch) * dim * dstate;
      p.chunk_len = pl.chunk_len;
    } else {
      p.chunk_len = pl.chunk_len;
    }
    cudaError_t ce = ssm::scan_scaled_launch(p, pl.nchunks, pl.balanced_ctas, stream, err, sizeof(err));
    if (ce != cudaSuccess) return cuda_fail(ce, err[0] ? err : "scan launch");
    return SSM_OK;
  }
  // general kernel (also the fallback for buffers whose alignment TMA cannot use)
  const int T = ssm::scan_tile_steps(static_cast<int>(e));
  bool tma = ((seqlen * e) % 16 == 0) && seqlen >= T && static_cast<int64_t>(batch) * dim >= kChannelsPerCta;
  for (const void* q : {u, delta, z, B, C})
    if (q && !aligned(q, 16)) tma = false;
  p.tma_ok = tma;
  p.vec_ok = aligned(y, 16) && (seqlen * e) % 16 == 0;
  int nchunks = pl.nchunks;
  if (pl.path == 0 && nchunks > 1) {
    p.agg_P = ws + pl.off_P;
    p.agg_Q = ws + pl.off_Q;
    p.h_in = ws + pl.off_hin;
    p.h_in_chunk_stride = static_cast<int64_t>(batch) * dim * dstate;
    p.chunk_len = pl.chunk_len;
    p.carry_f64 = io_dtype == SSM_F32;
  } else {
    nchunks = 1;   // the fast plan's workspace layout does not apply here: run one pass
    p.h_in = h0;
    p.h_in_chunk_stride = 0;
    p.chunk_len = seqlen;
  }
  cudaError_t ce = ssm::scan_fwd_launch(p, nchunks, stream, err, sizeof(err));
  if (ce != cudaSuccess) return cuda_fail(ce, err[0] ? err : "scan launch");
  return SSM_OK;
}

ssm_status ssm_scan_fwd(const void* u, const void* delta, const float* A, const void* B, const void* C,
                        const float* D, const void* z, const float* delta_bias, int softplus_flag, void* y,
                        float* last_state, int batch, int dim, int dstate, int64_t seqlen, ssm_dtype io_dtype,
                        void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return ssm_scan_fwd_ex(u, delta, A, B, C, D, z, delta_bias, softplus_flag, y, last_state, batch, dim, dstate,
                         seqlen, io_dtype, workspace, workspace_bytes, nullptr, stream);
}

ssm_status ssm_state_update(const void* x_t, const void* delta_t, const float* A, const void* B_t, const void* C_t,
                            const float* D, const void* z_t, float* state, float* conv_state, const float* conv_w,
                            const float* delta_bias, int softplus_flag, void* y_t, int batch, int dim, int dstate,
                            int dconv, ssm_dtype io_dtype, cudaStream_t stream) {
  g_err[0] = 0;
  if (io_dtype != SSM_F32 && io_dtype != SSM_BF16) return fail(SSM_ERR_INVALID_ARG, "unknown io_dtype %d", io_dtype);
  if (batch < 1 || dim < 1 || dstate < 1 || dconv < 1)
    return fail(SSM_ERR_INVALID_ARG, "bad sizes batch=%d dim=%d dstate=%d dconv=%d", batch, dim, dstate, dconv);
  if (dstate > 16) return fail(SSM_ERR_UNSUPPORTED, "dstate=%d > 16 is not supported", dstate);
  if (dconv != 4) return fail(SSM_ERR_UNSUPPORTED, "d_conv=%d is not supported (only 4)", dconv);
  if (static_cast<int64_t>(batch) * dim >= (int64_t(1) << 31))
    return fail(SSM_ERR_UNSUPPORTED, "batch * dim must be below 2^31");
  if (!x_t || !delta_t || !A || !B_t || !C_t || !state || !conv_state || !conv_w || !y_t)
    return fail(SSM_ERR_INVALID_ARG, "null required pointer");
  const size_t e = io_dtype == SSM_BF16 ? 2 : 4;
  for (const void* p : {x_t, delta_t, z_t, B_t, C_t, static_cast<const void*>(y_t)})
    if (p && !aligned(p, e)) return fail(SSM_ERR_INVALID_ARG, "io pointer not aligned to its element size");
  for (const void* p : {static_cast<const void*>(A), static_cast<const void*>(D),
                        static_cast<const void*>(delta_bias), static_cast<const void*>(state),
                        static_cast<const void*>(conv_state), static_cast<const void*>(conv_w)})
    if (p && !aligned(p, 4)) return fail(SSM_ERR_INVALID_ARG, "float32 pointer not 4-byte aligned");
  const size_t bd = static_cast<size_t>(batch) * dim;
  const Range outs[] = {range_of(y_t, bd * e), range_of(state, bd * dstate * 4),
                        range_of(conv_state, bd * (dconv - 1) * 4)};
  const Range ins[] = {range_of(x_t, bd * e), range_of(delta_t, bd * e), range_of(z_t, z_t ? bd * e : 0),
                       range_of(B_t, batch * dstate * e), range_of(C_t, batch * dstate * e),
                       range_of(A, static_cast<size_t>(dim) * dstate * 4), range_of(D, D ? dim * 4 : 0),
                       range_of(delta_bias, delta_bias ? dim * 4 : 0), range_of(conv_w, dim * dconv * 4)};
  for (const Range& o : outs)
    for (const Range& i : ins)
      if (overlap(o, i)) return fail(SSM_ERR_INVALID_ARG, "an output or state overlaps an input");
  if (overlap(outs[0], outs[1]) || overlap(outs[0], outs[2]) || overlap(outs[1], outs[2]))
    return fail(SSM_ERR_INVALID_ARG, "y_t, state and conv_state overlap");
  ssm::DecodeParams p;
  memset(&p, 0, sizeof(p));
  p.x = x_t; p.delta = delta_t; p.z = z_t; p.B = B_t; p.C = C_t; p.A = A; p.D = D; p.bias = delta_bias;
  p.conv_w = conv_w; p.state = state; p.conv_state = conv_state; p.y = y_t;
  p.batch = batch; p.dim = dim; p.N = dstate; p.softplus = softplus_flag != 0; p.io_bf16 = io_dtype == SSM_BF16;
  p.vec16 = dstate == 16 && aligned(state, 16) && aligned(A, 16) && aligned(conv_w, 16) && aligned(B_t, 8) &&
            aligned(C_t, 8);
  cudaError_t ce = ssm::state_update_launch(p, stream);
  if (ce != cudaSuccess) return cuda_fail(ce, "state update launch");
  return SSM_OK;
}

ssm_status ssm_causal_conv1d_fwd(const void* x, const float* conv_w, const float* conv_state_in, void* u,
                                 float* conv_state_out, int batch, int dim, int64_t seqlen, int dconv, int apply_silu,
                                 ssm_dtype io_dtype, cudaStream_t stream) {
  g_err[0] = 0;
  if (io_dtype != SSM_F32 && io_dtype != SSM_BF16) return fail(SSM_ERR_INVALID_ARG, "unknown io_dtype %d", io_dtype);
  if (batch < 1 || dim < 1 || seqlen < 0 || dconv < 1)
    return fail(SSM_ERR_INVALID_ARG, "bad sizes batch=%d dim=%d seqlen=%lld dconv=%d", batch, dim,
                static_cast<long long>(seqlen), dconv);
  if (dconv != 4) return fail(SSM_ERR_UNSUPPORTED, "d_conv=%d is not supported (only 4)", dconv);
  if (static_cast<int64_t>(batch) * dim >= (int64_t(1) << 31))
    return fail(SSM_ERR_UNSUPPORTED, "batch * dim must be below 2^31");
  if (!conv_w || (seqlen > 0 && (!x || !u))) return fail(SSM_ERR_INVALID_ARG, "null required pointer (x, conv_w, u)");
  const size_t e = io_dtype == SSM_BF16 ? 2 : 4;
  for (const void* p : {x, static_cast<const void*>(u)})
    if (p && !aligned(p, e)) return fail(SSM_ERR_INVALID_ARG, "io pointer not aligned to its element size");
  for (const void* p : {static_cast<const void*>(conv_w), static_cast<const void*>(conv_state_in),
                        static_cast<const void*>(conv_state_out)})
    if (p && !aligned(p, 4)) return fail(SSM_ERR_INVALID_ARG, "float32 pointer not 4-byte aligned");
  const size_t bdl = static_cast<size_t>(batch) * dim * seqlen * e;
  const size_t st = static_cast<size_t>(batch) * dim * 3 * 4;
  const Range outs[] = {range_of(u, bdl), range_of(conv_state_out, conv_state_out ? st : 0)};
  const Range ins[] = {range_of(x, bdl), range_of(conv_w, static_cast<size_t>(dim) * 4 * 4),
                       range_of(conv_state_in, conv_state_in ? st : 0)};
  for (const Range& o : outs)
    for (const Range& i : ins)
      if (overlap(o, i)) return fail(SSM_ERR_INVALID_ARG, "an output overlaps an input");
  if (overlap(outs[0], outs[1])) return fail(SSM_ERR_INVALID_ARG, "u overlaps conv_state_out");
  if (seqlen == 0) {
    if (conv_state_out) {
      cudaError_t ce = conv_state_in ? cudaMemcpyAsync(conv_state_out, conv_state_in, st, cudaMemcpyDeviceToDevice, stream)
                                     : cudaMemsetAsync(conv_state_out, 0, st, stream);
      if (ce != cudaSuccess) return cuda_fail(ce, "seqlen 0 conv state copy");
    }
    return SSM_OK;
  }
  ssm::ConvParams p;
  memset(&p, 0, sizeof(p));
  p.x = x; p.w = conv_w; p.state_in = conv_state_in; p.u = u; p.state_out = conv_state_out;
  p.batch = batch; p.dim = dim; p.L = seqlen; p.silu = apply_silu != 0; p.io_bf16 = io_dtype == SSM_BF16;
  const int64_t vecn = static_cast<int64_t>(16 / e);
  // the vectorised kernel indexes chunks with 32-bit integers
  const bool vec = seqlen % vecn == 0 && aligned(x, 16) && aligned(u, 16) && aligned(conv_w, 16) &&
                   static_cast<int64_t>(batch) * dim * (seqlen / vecn) < (int64_t(1) << 31);
  cudaError_t ce = ssm::conv1d_launch(p, vec, stream);
  if (ce != cudaSuccess) return cuda_fail(ce, "conv1d launch");
  return SSM_OK;
}

ssm_status ssm_selftest_bounded_wait(int which, int64_t limit_ns, cudaStream_t stream) {
  g_err[0] = 0;
  if (which != 0 && which != 1) return fail(SSM_ERR_INVALID_ARG, "which must be 0 (mbarrier) or 1 (flag), got %d", which);
  const int64_t lim = limit_ns < 1000000 ? 1000000 : (limit_ns > 2000000000 ? 2000000000 : limit_ns);
  cudaError_t ce = ssm::selftest_bounded_wait_launch(which, static_cast<unsigned long long>(lim), stream);
  if (ce != cudaSuccess) return cuda_fail(ce, "self-test launch");
  return SSM_OK;
}

ssm_status ssm_selftest_index_check(cudaStream_t stream) {
  g_err[0] = 0;
  if (!SSM_CHECK) return fail(SSM_ERR_UNSUPPORTED, "the index check self-test needs the checked build");
  cudaError_t ce = ssm::selftest_index_check_launch(stream);
  if (ce != cudaSuccess) return cuda_fail(ce, "self-test launch");
  return SSM_OK;
}

ssm_status ssm_selftest_withhold_carry(int cta, int64_t limit_ns) {
  g_err[0] = 0;
  if (cta < 0) return fail(SSM_ERR_INVALID_ARG, "cta must be >= 0, got %d", cta);
  g_withhold.armed = true;
  g_withhold.cta = cta;
  g_withhold.limit_ns = limit_ns < 1000000 ? 1000000 : (limit_ns > 2000000000 ? 2000000000 : limit_ns);
  return SSM_OK;
}

ssm_status ssm_device_status(cudaStream_t stream) {
  unsigned int word = 0;
  cudaError_t ce = ssm::read_and_clear_device_status(&word, stream);
  if (ce != cudaSuccess) return cuda_fail(ce, "device status read");
  if (word & ssm::kStatusBounds) return fail(SSM_ERR_CHECK, "an index check failed (status word 0x%x)", word);
  if (word != 0) return fail(SSM_ERR_TIMEOUT, "a device wait gave up (status word 0x%x)", word);
  return SSM_OK;
}

}  // extern "C"

namespace {

struct BwdLayout {
  size_t ckpt = 0, ckpt_s = 0, agg = 0, acc_dA = 0, acc_dB = 0, acc_dC = 0, acc_dD = 0, acc_dbias = 0, total = 0;
  int64_t chunk_len = 0;
  int nchunks = 1;
};

// Time chunks: enough (channel group, chunk) tiles for several waves of resident CTAs, chunks a
// multiple of the segment length and at least 64 steps.
void bwd_chunks(int batch, int dim, int64_t seqlen, BwdLayout* l) {
  const int K = ssm::bwd_segment_steps();
  const int64_t groups = static_cast<int64_t>(batch) * ((dim + kChannelsPerCta - 1) / kChannelsPerCta);
  const int64_t target_tiles = static_cast<int64_t>(SSM_BWD_TILES_PER_SM) * sm_count();
  int64_t nch = std::max<int64_t>(1, (target_tiles + groups - 1) / groups);
  nch = std::min<int64_t>(nch, std::max<int64_t>(1, seqlen / 64));
  nch = std::min<int64_t>(nch, 65535);
  int64_t chunk = static_cast<int64_t>(round_up(static_cast<size_t>((seqlen + nch - 1) / nch), K));
  if (chunk <= 0) chunk = K;
  l->chunk_len = chunk;
  l->nchunks = static_cast<int>((seqlen + chunk - 1) / chunk);
}

// checkpoints (16 local states and a Δ sum per channel and segment), chunk aggregates, then for
// float32 io the double accumulators
BwdLayout bwd_layout(int batch, int dim, int dstate, int64_t seqlen, ssm_dtype io) {
  BwdLayout l;
  if (seqlen <= 0) return l;
  bwd_chunks(batch, dim, seqlen, &l);
  const size_t ce = io == SSM_BF16 ? sizeof(float) : sizeof(double);
  const int K = ssm::bwd_segment_steps();
  const size_t rows = static_cast<size_t>(batch) * dim;
  const size_t nseg = static_cast<size_t>((seqlen + K - 1) / K);
  size_t off = round_up(rows * nseg * 16 * ce, 256);
  l.ckpt_s = off;
  off += round_up(rows * nseg * ce, 256);
  l.agg = off;
  off += round_up(rows * l.nchunks * ssm::bwd_aggregate_floats() * ce, 256);
  if (io == SSM_F32) {
    l.acc_dA = off;
    off += round_up(static_cast<size_t>(dim) * dstate * 8, 256);
    l.acc_dB = off;
    off += round_up(static_cast<size_t>(batch) * dstate * seqlen * 8, 256);
    l.acc_dC = off;
    off += round_up(static_cast<size_t>(batch) * dstate * seqlen * 8, 256);
    l.acc_dD = off;
    off += round_up(static_cast<size_t>(dim) * 8, 256);
    l.acc_dbias = off;
    off += round_up(static_cast<size_t>(dim) * 8, 256);
  }
  l.total = off;
  return l;
}

}  // namespace

extern "C" {

size_t ssm_scan_bwd_workspace_size(int batch, int dim, int dstate, int64_t seqlen, ssm_dtype io_dtype) {
  if (!sizes_ok(batch, dim, dstate, seqlen, io_dtype)) return 0;
  return bwd_layout(batch, dim, dstate, seqlen, io_dtype).total;
}

ssm_status ssm_scan_bwd(const void* u, const void* delta, const float* A, const void* B, const void* C,
                        const float* D, const void* z, const float* delta_bias, int softplus_flag, const void* dy,
                        void* du, void* ddelta, void* dz, float* dA, float* dB, float* dC, float* dD,
                        float* ddelta_bias, int batch, int dim, int dstate, int64_t seqlen, ssm_dtype io_dtype,
                        void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  g_err[0] = 0;
  if (io_dtype != SSM_F32 && io_dtype != SSM_BF16) return fail(SSM_ERR_INVALID_ARG, "unknown io_dtype %d", io_dtype);
  if (batch < 1 || dim < 1 || seqlen < 0 || dstate < 1)
    return fail(SSM_ERR_INVALID_ARG, "bad sizes batch=%d dim=%d dstate=%d seqlen=%lld", batch, dim, dstate,
                static_cast<long long>(seqlen));
  if (dstate > 16) return fail(SSM_ERR_UNSUPPORTED, "dstate=%d > 16 is not supported", dstate);
  if (batch > 65535) return fail(SSM_ERR_UNSUPPORTED, "batch=%d above 65535 is not supported", batch);
  if (!A || !dA) return fail(SSM_ERR_INVALID_ARG, "null required pointer (A, dA)");
  if (seqlen > 0 && (!u || !delta || !B || !C || !dy || !du || !ddelta || !dB || !dC))
    return fail(SSM_ERR_INVALID_ARG, "null required pointer (u, delta, B, C, dy, du, ddelta, dB, dC)");
  if ((z == nullptr) != (dz == nullptr)) return fail(SSM_ERR_INVALID_ARG, "dz must be given exactly when z is");
  const size_t e = io_dtype == SSM_BF16 ? 2 : 4;
  for (const void* q : {u, delta, z, B, C, dy, static_cast<const void*>(du), static_cast<const void*>(ddelta),
                        static_cast<const void*>(dz)})
    if (q && !aligned(q, e)) return fail(SSM_ERR_INVALID_ARG, "io pointer not aligned to its element size");
  for (const void* q : {static_cast<const void*>(A), static_cast<const void*>(D), static_cast<const void*>(delta_bias),
                        static_cast<const void*>(dA), static_cast<const void*>(dB), static_cast<const void*>(dC),
                        static_cast<const void*>(dD), static_cast<const void*>(ddelta_bias)})
    if (q && !aligned(q, 4)) return fail(SSM_ERR_INVALID_ARG, "float32 pointer not 4-byte aligned");
  const size_t bdl = static_cast<size_t>(batch) * dim * seqlen * e;
  const size_t bnl = static_cast<size_t>(batch) * dstate * seqlen * e;
  const size_t bnl4 = static_cast<size_t>(batch) * dstate * seqlen * 4;
  const size_t dn4 = static_cast<size_t>(dim) * dstate * 4;
  const Range outs[] = {range_of(du, bdl), range_of(ddelta, bdl), range_of(dz, dz ? bdl : 0), range_of(dA, dn4),
                        range_of(dB, bnl4), range_of(dC, bnl4), range_of(dD, dD ? dim * 4 : 0),
                        range_of(ddelta_bias, ddelta_bias ? dim * 4 : 0)};
  const Range ins[] = {range_of(u, bdl), range_of(delta, bdl), range_of(z, z ? bdl : 0), range_of(B, bnl),
                       range_of(C, bnl), range_of(A, dn4), range_of(D, D ? dim * 4 : 0),
                       range_of(delta_bias, delta_bias ? dim * 4 : 0), range_of(dy, bdl)};
  for (const Range& o : outs)
    for (const Range& i : ins)
      if (overlap(o, i)) return fail(SSM_ERR_INVALID_ARG, "an output overlaps an input");
  const int nouts = static_cast<int>(sizeof(outs) / sizeof(outs[0]));
  for (int i = 0; i < nouts; ++i)
    for (int j = i + 1; j < nouts; ++j)
      if (overlap(outs[i], outs[j])) return fail(SSM_ERR_INVALID_ARG, "two outputs overlap");
  const BwdLayout lay = bwd_layout(batch, dim, dstate, seqlen, io_dtype);
  if (lay.total > 0) {
    if (!workspace || workspace_bytes < lay.total)
      return fail(SSM_ERR_INVALID_ARG, "workspace of %zu bytes required, %zu given", lay.total, workspace_bytes);
    if (!aligned(workspace, 256)) return fail(SSM_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    const Range w = range_of(workspace, lay.total);
    for (const Range& i : ins)
      if (overlap(w, i)) return fail(SSM_ERR_INVALID_ARG, "workspace overlaps an input");
    for (const Range& o : outs)
      if (overlap(w, o)) return fail(SSM_ERR_INVALID_ARG, "workspace overlaps an output");
  }
  if (seqlen == 0) {
    // no steps: every parameter gradient is zero
    cudaError_t ce = cudaMemsetAsync(dA, 0, dn4, stream);
    if (ce == cudaSuccess && dD) ce = cudaMemsetAsync(dD, 0, dim * 4, stream);
    if (ce == cudaSuccess && ddelta_bias) ce = cudaMemsetAsync(ddelta_bias, 0, dim * 4, stream);
    if (ce != cudaSuccess) return cuda_fail(ce, "seqlen 0 gradient clear");
    return SSM_OK;
  }
  ssm::BwdParams p;
  memset(&p, 0, sizeof(p));
  p.u = u; p.delta = delta; p.z = z; p.B = B; p.C = C; p.A = A; p.D = D; p.bias = delta_bias; p.dy = dy;
  p.du = du; p.ddelta = ddelta; p.dz = dz; p.dA = dA; p.dB = dB; p.dC = dC; p.dD = dD; p.dbias = ddelta_bias;
  p.batch = batch; p.dim = dim; p.N = dstate; p.L = seqlen;
  p.softplus = softplus_flag != 0; p.io_bf16 = io_dtype == SSM_BF16;
  p.chunk_len = lay.chunk_len;
  p.nchunks = lay.nchunks;
  bool vec_io = seqlen % 8 == 0;
  for (const void* q : {u, delta, z, dy, static_cast<const void*>(du), static_cast<const void*>(ddelta),
                        static_cast<const void*>(dz)})
    if (q && !aligned(q, 16)) vec_io = false;
  p.vec_io = vec_io;
  p.vec_red = seqlen % 4 == 0 && aligned(dB, 16) && aligned(dC, 16);
  char* ws = static_cast<char*>(workspace);
  p.ckpt = ws + lay.ckpt;
  p.ckpt_s = ws + lay.ckpt_s;
  p.agg = ws + lay.agg;
  if (io_dtype == SSM_BF16) {
    p.acc_dA = dA; p.acc_dB = dB; p.acc_dC = dC; p.acc_dD = dD; p.acc_dbias = ddelta_bias;
  } else {
    p.acc_dA = ws + lay.acc_dA; p.acc_dB = ws + lay.acc_dB; p.acc_dC = ws + lay.acc_dC;
    p.acc_dD = dD ? ws + lay.acc_dD : nullptr;
    p.acc_dbias = ddelta_bias ? ws + lay.acc_dbias : nullptr;
  }
  cudaError_t ce = ssm::scan_bwd_launch(p, stream);
  if (ce != cudaSuccess) return cuda_fail(ce, "scan backward launch");
  return SSM_OK;
}

}  // extern "C"

extern "C" {

ssm_status ssm_ssd_fwd_ex(const void* x, const void* dt, const float* A, const void* B, const void* C, const float* D,
                       const float* dt_bias, int softplus_flag, const float* h0, void* y, float* final_state,
                          int batch, int64_t seqlen, int nheads, int headdim, int dstate, int ngroups,
                          ssm_dtype io_dtype, void* workspace, size_t workspace_bytes, int ctas, cudaStream_t stream) {
  g_err[0] = 0;
  if (io_dtype != SSM_F32 && io_dtype != SSM_BF16) return fail(SSM_ERR_INVALID_ARG, "unknown io_dtype %d", io_dtype);
  if (batch < 1 || seqlen < 0 || nheads < 1 || headdim < 1 || dstate < 1 || ngroups < 1 || nheads % ngroups != 0)
    return fail(SSM_ERR_INVALID_ARG, "bad sizes batch=%d seqlen=%lld nheads=%d headdim=%d dstate=%d ngroups=%d",
                batch, static_cast<long long>(seqlen), nheads, headdim, dstate, ngroups);
  if (io_dtype != SSM_BF16) return fail(SSM_ERR_UNSUPPORTED, "the SSD path supports bf16 io only");
  if (headdim != ssm::ssd_head_dim() || dstate != ssm::ssd_state_dim())
    return fail(SSM_ERR_UNSUPPORTED, "the SSD path supports headdim %d and dstate %d only", ssm::ssd_head_dim(),
                ssm::ssd_state_dim());
  if (batch > 65535) return fail(SSM_ERR_UNSUPPORTED, "batch=%d above 65535 is not supported", batch);
  if (!A || (seqlen > 0 && (!x || !dt || !B || !C || !y)))
    return fail(SSM_ERR_INVALID_ARG, "null required pointer (x, dt, A, B, C, y)");
  for (const void* q : {x, B, C, static_cast<const void*>(y)})
    if (q && !aligned(q, 16)) return fail(SSM_ERR_INVALID_ARG, "x, B, C and y must be 16-byte aligned");
  if (dt && !aligned(dt, 2)) return fail(SSM_ERR_INVALID_ARG, "dt not aligned to its element size");
  for (const void* q : {static_cast<const void*>(A), static_cast<const void*>(D), static_cast<const void*>(dt_bias)})
    if (q && !aligned(q, 4)) return fail(SSM_ERR_INVALID_ARG, "float32 pointer not 4-byte aligned");
  for (const void* q : {static_cast<const void*>(h0), static_cast<const void*>(final_state)})
    if (q && !aligned(q, 8)) return fail(SSM_ERR_INVALID_ARG, "h0 and final_state must be 8-byte aligned");
  const size_t e = 2;
  const size_t xl = static_cast<size_t>(batch) * seqlen * nheads * headdim * e;
  const size_t bcl = static_cast<size_t>(batch) * seqlen * ngroups * dstate * e;
  const size_t st = static_cast<size_t>(batch) * nheads * headdim * dstate * 4;
  if (ctas < 0) return fail(SSM_ERR_INVALID_ARG, "ctas must be >= 0, got %d", ctas);
  const SsdPlan plan = workspace ? ssd_plan(batch, nheads, seqlen, ctas) : SsdPlan();
  if (plan.ctas > 0 && workspace_bytes < plan.workspace)
    return fail(SSM_ERR_INVALID_ARG, "workspace of %zu bytes, the balanced schedule needs %zu", workspace_bytes,
                plan.workspace);
  if (plan.ctas > 0 && !aligned(workspace, 256)) return fail(SSM_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  const Range outs[] = {range_of(y, xl), range_of(final_state, final_state ? st : 0),
                        range_of(workspace, plan.ctas > 0 ? plan.workspace : 0)};
  const Range ins[] = {range_of(x, xl), range_of(dt, static_cast<size_t>(batch) * seqlen * nheads * e),
                       range_of(B, bcl), range_of(C, bcl), range_of(A, nheads * 4), range_of(D, D ? nheads * 4 : 0),
                       range_of(dt_bias, dt_bias ? nheads * 4 : 0), range_of(h0, h0 ? st : 0)};
  for (const Range& o : outs)
    for (const Range& i : ins)
      if (overlap(o, i)) return fail(SSM_ERR_INVALID_ARG, "an output overlaps an input");
  for (int i = 0; i < 3; ++i)
    for (int j = i + 1; j < 3; ++j)
      if (overlap(outs[i], outs[j])) return fail(SSM_ERR_INVALID_ARG, "y, final_state and the workspace overlap");
  if (seqlen == 0) {
    if (final_state) {
      cudaError_t ce = h0 ? cudaMemcpyAsync(final_state, h0, st, cudaMemcpyDeviceToDevice, stream)
                          : cudaMemsetAsync(final_state, 0, st, stream);
      if (ce != cudaSuccess) return cuda_fail(ce, "seqlen 0 state copy");
    }
    return SSM_OK;
  }
  ssm::SsdParams p;
  memset(&p, 0, sizeof(p));
  p.x = x; p.dt = dt; p.A = A; p.B = B; p.C = C; p.D = D; p.dt_bias = dt_bias; p.h0 = h0; p.y = y; p.hT = final_state;
  p.batch = batch; p.nheads = nheads; p.ngroups = ngroups; p.L = seqlen; p.softplus = softplus_flag != 0;
  p.test_withhold_cta = -1;
  p.carry_wait_ns = 0;
  if (plan.ctas > 0) {
    p.balanced = 1;
    p.range = plan.range;
    p.carry = static_cast<float*>(workspace);
    p.flags = reinterpret_cast<unsigned*>(static_cast<char*>(workspace) + plan.carry);
  }
  if (g_withhold.armed) {
    // one-shot diagnostic armed by ssm_selftest_withhold_carry on this host thread
    if (plan.ctas > 0) {
      p.test_withhold_cta = g_withhold.cta;
      p.carry_wait_ns = static_cast<uint64_t>(g_withhold.limit_ns);
    }
    g_withhold.armed = false;
  }
  cudaError_t ce = ssm::ssd_fwd_launch(p, plan.ctas, stream);
  if (ce != cudaSuccess) return cuda_fail(ce, "ssd launch");
  return SSM_OK;
}


ssm_status ssm_ssd_fwd(const void* x, const void* dt, const float* A, const void* B, const void* C, const float* D,
                       const float* dt_bias, int softplus_flag, const float* h0, void* y, float* final_state,
                       int batch, int64_t seqlen, int nheads, int headdim, int dstate, int ngroups, ssm_dtype io_dtype,
                       cudaStream_t stream) {
  return ssm_ssd_fwd_ex(x, dt, A, B, C, D, dt_bias, softplus_flag, h0, y, final_state, batch, seqlen, nheads, headdim,
                        dstate, ngroups, io_dtype, nullptr, 0, 0, stream);
}

size_t ssm_ssd_fwd_workspace_size(int batch, int64_t seqlen, int nheads, int ctas) {
  if (batch < 1 || seqlen < 1 || nheads < 1 || ctas < 0) return 0;
  return ssd_plan(batch, nheads, seqlen, ctas).workspace;
}

}  // extern "C"

extern "C" {

ssm_status ssm_ssd_state_update(const void* x_t, const void* dt_t, const float* A, const void* B_t, const void* C_t,
                                const float* D, const float* dt_bias, int softplus_flag, float* state, void* y_t,
                                int batch, int nheads, int headdim, int dstate, int ngroups, ssm_dtype io_dtype,
                                cudaStream_t stream) {
  g_err[0] = 0;
  if (io_dtype != SSM_F32 && io_dtype != SSM_BF16) return fail(SSM_ERR_INVALID_ARG, "unknown io_dtype %d", io_dtype);
  if (batch < 1 || nheads < 1 || headdim < 1 || dstate < 1 || ngroups < 1 || nheads % ngroups != 0)
    return fail(SSM_ERR_INVALID_ARG, "bad sizes batch=%d nheads=%d headdim=%d dstate=%d ngroups=%d", batch, nheads,
                headdim, dstate, ngroups);
  if (io_dtype != SSM_BF16) return fail(SSM_ERR_UNSUPPORTED, "the SSD decode step supports bf16 io only");
  if (headdim != ssm::ssd_head_dim() || dstate != ssm::ssd_state_dim())
    return fail(SSM_ERR_UNSUPPORTED, "the SSD decode step supports headdim %d and dstate %d only", ssm::ssd_head_dim(),
                ssm::ssd_state_dim());
  if (batch > 65535) return fail(SSM_ERR_UNSUPPORTED, "batch=%d above 65535 is not supported", batch);
  if (!x_t || !dt_t || !A || !B_t || !C_t || !state || !y_t)
    return fail(SSM_ERR_INVALID_ARG, "null required pointer (x_t, dt_t, A, B_t, C_t, state, y_t)");
  for (const void* q : {x_t, dt_t, static_cast<const void*>(y_t)})
    if (!aligned(q, 2)) return fail(SSM_ERR_INVALID_ARG, "io pointer not aligned to its element size");
  for (const void* q : {B_t, C_t, static_cast<const void*>(state)})
    if (!aligned(q, 16)) return fail(SSM_ERR_INVALID_ARG, "B_t, C_t and state must be 16-byte aligned");
  for (const void* q : {static_cast<const void*>(A), static_cast<const void*>(D), static_cast<const void*>(dt_bias)})
    if (q && !aligned(q, 4)) return fail(SSM_ERR_INVALID_ARG, "float32 pointer not 4-byte aligned");
  const size_t bh = static_cast<size_t>(batch) * nheads;
  const size_t bg = static_cast<size_t>(batch) * ngroups;
  const Range outs[] = {range_of(y_t, bh * headdim * 2), range_of(state, bh * headdim * dstate * 4)};
  const Range ins[] = {range_of(x_t, bh * headdim * 2), range_of(dt_t, bh * 2), range_of(B_t, bg * dstate * 2),
                       range_of(C_t, bg * dstate * 2), range_of(A, nheads * 4), range_of(D, D ? nheads * 4 : 0),
                       range_of(dt_bias, dt_bias ? nheads * 4 : 0)};
  for (const Range& o : outs)
    for (const Range& i : ins)
      if (overlap(o, i)) return fail(SSM_ERR_INVALID_ARG, "an output or the state overlaps an input");
  if (overlap(outs[0], outs[1])) return fail(SSM_ERR_INVALID_ARG, "y_t overlaps the state");
  ssm::SsdDecodeParams p;
  memset(&p, 0, sizeof(p));
  p.x = x_t; p.dt = dt_t; p.A = A; p.B = B_t; p.C = C_t; p.D = D; p.dt_bias = dt_bias; p.state = state; p.y = y_t;
  p.batch = batch; p.nheads = nheads; p.ngroups = ngroups; p.softplus = softplus_flag != 0;
  cudaError_t ce = ssm::ssd_decode_launch(p, stream);
  if (ce != cudaSuccess) return cuda_fail(ce, "ssd decode launch");
  return SSM_OK;
}

}  // extern "C"
