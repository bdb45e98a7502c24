// Internal interfaces between the C-ABI layer (ssm_api.cu) and the kernel files.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#ifndef SSM_CHECK
#define SSM_CHECK 0   // 1 in the checked debug build (libssm_b300_check.so)
#endif

namespace ssm {

// Bits of the device status word read by ssm_device_status(): a bounded wait gave up; an index
// check of the checked build failed.
constexpr unsigned kStatusTimeout = 1u;
constexpr unsigned kStatusBounds = 2u;

// Everything a prefill pass needs; filled and validated by the API layer.
struct ScanParams {
  const void* u;
  const void* delta;
  const void* z;          // may be null
  const void* B;
  const void* C;
  const float* A;
  const float* D;         // may be null
  const float* bias;      // may be null
  void* y;
  float* last_state;      // may be null
  const float* h0;        // user initial state (batch, dim, N) or null
  const void* h_in;       // initial state per chunk: h_in + chunk * h_in_chunk_stride, or null
  int64_t h_in_chunk_stride;
  void* agg_P;            // chunk aggregates (workspace), chunked algorithm only
  void* agg_Q;
  int carry_f64;          // h_in / agg_P / agg_Q hold doubles (float32-io chunked), else floats
  int batch, dim, N;
  int64_t L;
  int64_t chunk_len;      // steps per chunk (== L for a single pass)
  int softplus;
  int disc;               // 0: Δ·B, 1: exact ZOH
  int io_bf16;            // 1: bfloat16 io, 0: float32 io
  int tma_ok;             // the layout allows 2D TMA tensor maps
  int vec_ok;             // y rows allow 16-byte stores
  // bf16 fast path, balanced persistent schedule
  int sched_balanced;     // 1: one range of (group, tile) work per resident CTA
  int64_t range_tiles;    // tiles per CTA range
  float* carry;           // (ctas, channels per CTA, 16) states handed from one CTA to the next
  unsigned* flags;        // (ctas) publication flags
  // Diagnostics (ssm_selftest_withhold_carry): the CTA whose carry publication is withheld (-1: none)
  // and the limit of the carry wait in ns (0: the default 2 s).
  int test_withhold_cta;
  uint64_t carry_wait_ns;
};

// Steps per time tile for an io element size (64 for bf16, 32 for float32).
int scan_tile_steps(int io_bytes);

// Launches the passes of one prefill call on `stream` (nchunks == 1: single pass).
cudaError_t scan_fwd_launch(const ScanParams& p, int nchunks, cudaStream_t stream, char* err, size_t errlen);

// Builds a 2D tiled tensor map (rows of `inner` elements, `rows` rows, 128-byte swizzle, zero fill).
bool encode_tensor_map_2d(CUtensorMap* map, CUtensorMapDataType dtype, void* base, uint64_t inner, uint64_t rows,
                          uint64_t row_pitch_bytes, uint32_t box_inner, uint32_t box_rows, char* err,
                          size_t errlen);

// Builds a 3D tiled tensor map (`outer` blocks of `rows` rows of `inner` elements, 128-byte swizzle,
// zero fill; boxes of box_inner x box_rows x 1): coordinates past `rows` read zeros instead of the
// next block's rows.
bool encode_tensor_map_3d(CUtensorMap* map, CUtensorMapDataType dtype, void* base, uint64_t inner, uint64_t rows,
                          uint64_t outer, uint64_t row_pitch_bytes, uint64_t outer_pitch_bytes, uint32_t box_inner,
                          uint32_t box_rows, char* err, size_t errlen);

struct DecodeParams {
  const void* x;
  const void* delta;
  const void* z;          // may be null
  const void* B;
  const void* C;
  const float* A;
  const float* D;         // may be null
  const float* bias;      // may be null
  const float* conv_w;
  float* state;
  float* conv_state;
  void* y;
  int batch, dim, N;
  int softplus;
  int io_bf16;
  int vec16;              // dstate == 16 and state, A, conv_w, B, C aligned for vector access
};

cudaError_t state_update_launch(const DecodeParams& p, cudaStream_t stream);

struct ConvParams {
  const void* x;          // (batch, dim, L) io dtype
  const float* w;         // (dim, 4)
  const float* state_in;  // (batch, dim, 3) or null (zeros)
  void* u;                // (batch, dim, L) io dtype
  float* state_out;       // (batch, dim, 3) or null
  int batch, dim;
  int64_t L;
  int silu;
  int io_bf16;
};

// vec: L is a multiple of the 16-byte element count and x, u, w are 16-byte aligned
cudaError_t conv1d_launch(const ConvParams& p, bool vec, cudaStream_t stream);

// Backward of the prefill scan (scan_bwd.cu).  For bfloat16 io the cross-channel sums are
// accumulated straight into the float32 outputs (acc_* == dA, dB, ...); for float32 io they are
// accumulated in double in the workspace and converted at the end.
struct BwdParams {
  const void* u;
  const void* delta;
  const void* z;          // may be null
  const void* B;
  const void* C;
  const float* A;
  const float* D;         // may be null
  const float* bias;      // may be null
  const void* dy;
  void* du;
  void* ddelta;
  void* dz;               // null iff z is null
  float* dA;              // (dim, N)
  float* dB;              // (batch, N, L)
  float* dC;              // (batch, N, L)
  float* dD;              // (dim) or null
  float* dbias;           // (dim) or null
  void* ckpt;             // (batch, dim, ceil(L / segment), 16) local states, float (bf16 io) or double (f32 io)
  void* ckpt_s;           // (batch, dim, ceil(L / segment)) running sum of Δ within the chunk, same type
  void* agg;              // (batch, dim, nchunks, 48) chunk aggregates, same type
  void* acc_dA;
  void* acc_dB;
  void* acc_dC;
  void* acc_dD;           // null when dD is null
  void* acc_dbias;        // null when dbias is null
  int batch, dim, N;
  int64_t L;
  int64_t chunk_len;      // steps per chunk, a multiple of the segment length
  int nchunks;
  int softplus;
  int io_bf16;
  int vec_io;             // L % 8 == 0 and every io row base 16-byte aligned
  int vec_red;            // dB, dC 16-byte aligned and L % 4 == 0 (vector atomics)
};

int bwd_segment_steps();
int bwd_aggregate_floats();
cudaError_t scan_bwd_launch(const BwdParams& p, cudaStream_t stream);

// Mamba-2 SSD forward (ssd_tc.cu): bf16 io, headdim 64, d_state 128.
struct SsdParams {
  const void* x;          // (batch, L, nheads, 64) bf16
  const void* dt;         // (batch, L, nheads) bf16, before bias and softplus
  const float* A;         // (nheads)
  const void* B;          // (batch, L, ngroups, 128) bf16
  const void* C;          // (batch, L, ngroups, 128) bf16
  const float* D;         // (nheads) or null
  const float* dt_bias;   // (nheads) or null
  const float* h0;        // (batch, nheads, 64, 128) or null
  void* y;                // (batch, L, nheads, 64) bf16
  float* hT;              // (batch, nheads, 64, 128) or null
  int batch, nheads, ngroups;
  int64_t L;
  int softplus;
  // balanced persistent schedule (0: one CTA per sequence)
  int balanced;
  int64_t range;            // (sequence, chunk) units per CTA
  float* carry;             // (ranges, 64, 128): each range's state at the end of its head
  unsigned* flags;          // (ranges + 1): the carry is published; then the range counter; cleared
                            // before the launch
  int test_withhold_cta;    // diagnostic: this range never publishes its carry (-1: none)
  uint64_t carry_wait_ns;   // limit of the carry wait (0: 2 s)
};

int ssd_head_dim();
int ssd_state_dim();
int ssd_resident_ctas();   // co-resident CTAs of the SSD kernel on the current device (0 if unknown)
// balanced_ctas: the ranges (and CTAs) of the balanced schedule (p.balanced), ignored otherwise
cudaError_t ssd_fwd_launch(const SsdParams& p, int balanced_ctas, cudaStream_t stream);

// Mamba-2 decode step (ssd_decode.cu): one token, state (batch, nheads, 64, 128) float32 in place.
struct SsdDecodeParams {
  const void* x;          // (batch, nheads, 64) bf16
  const void* dt;         // (batch, nheads) bf16
  const float* A;         // (nheads)
  const void* B;          // (batch, ngroups, 128) bf16
  const void* C;          // (batch, ngroups, 128) bf16
  const float* D;         // (nheads) or null
  const float* dt_bias;   // (nheads) or null
  float* state;           // (batch, nheads, 64, 128)
  void* y;                // (batch, nheads, 64) bf16
  int batch, nheads, ngroups;
  int softplus;
};
cudaError_t ssd_decode_launch(const SsdDecodeParams& p, cudaStream_t stream);
cudaError_t ssd_status_read_and_clear(unsigned int* out);

// Sets the text returned by ssm_last_error_message() on the calling host thread (ssm_api.cu).
void set_last_error(const char* fmt, ...);

// Self-test of the device failure path (selftest.cu): which 0 = an mbarrier wait, 1 = a flag poll.
cudaError_t selftest_bounded_wait_launch(int which, unsigned long long limit_ns, cudaStream_t stream);
cudaError_t selftest_status_read_and_clear(unsigned int* out);
// Checked build only: a store one past a buffer, caught by its index check (cudaErrorNotSupported in
// the ordinary build, which launches nothing).
cudaError_t selftest_index_check_launch(cudaStream_t stream);

// Device status word access (scan_fwd.cu owns the symbol).
cudaError_t read_and_clear_device_status(unsigned int* out, cudaStream_t stream);

// Index-check words of the checked build (-DSSM_CHECK=1), one per kernel file; each reads its word
// and clears it, and reports 0 in the ordinary build.
cudaError_t general_check_read_and_clear(unsigned int* out);
cudaError_t scaled_check_read_and_clear(unsigned int* out);
cudaError_t decode_check_read_and_clear(unsigned int* out);
cudaError_t conv1d_check_read_and_clear(unsigned int* out);
cudaError_t ssd_check_read_and_clear(unsigned int* out);
cudaError_t ssd_decode_check_read_and_clear(unsigned int* out);
cudaError_t bwd_check_read_and_clear(unsigned int* out);

// Carry pass of the chunked algorithm over float carries (scan_fwd.cu).
cudaError_t carry_launch_f32(const ScanParams& p, int nchunks, cudaStream_t stream);

// bf16 prefill on the rescaled state, one thread per channel (scan_scaled.cu).
int scaled_channels_per_cta();
int scaled_resident_ctas();   // co-resident CTAs on the current device (0 if unknown)
cudaError_t scaled_status_read_and_clear(unsigned int* out);
cudaError_t scan_scaled_launch(const ScanParams& p, int nchunks, int balanced_ctas, cudaStream_t stream, char* err,
                               size_t errlen);

}  // namespace ssm
