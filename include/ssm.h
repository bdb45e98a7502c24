/*
 * ssm.h -- C ABI of the B300 selective state-space scan library (libssm_b300.so).
 *
 * The operation is the Mamba-1 selective SSM ("Mamba и State Space Models", sections
 * "Mamba: Selective State Space Model" and "Selective Scan (core algorithm)"; "Модуль 8.
 * Альтернативы Transformer: SSM, Mamba и гибриды", §4 and §6; "State Space Models: Mamba и
 * альтернатива Transformer", "Mamba: Selective State Space"), per batch b and channel d:
 *
 *     Δ_t  = softplus(Δ_raw[b,d,t] + delta_bias[d])        (or Δ_raw + bias if softplus is off)
 *     h_t  = exp(Δ_t A[d,:]) ⊙ h_{t-1} + Δ_t B[b,:,t] u[b,d,t],    h_{-1} = 0
 *     y_t  = (C[b,:,t]·h_t + D[d] u[b,d,t]) · SiLU(z[b,d,t])
 *
 * Conventions shared by every entry point:
 *  - All pointers are DEVICE pointers, owned by the caller; the library never allocates or frees
 *    device memory.  Every tensor is dense and row-major (contiguous) in the layout stated.
 *  - Calls are asynchronous on `stream` (0 = legacy default stream).  Host-side argument checks run
 *    before anything is enqueued; a call that returns an error has enqueued nothing.
 *  - Inputs must not alias outputs, except the in/out state buffers of ssm_state_update.
 *  - io tensors (u, delta, z, B, C, y and the per-token decode inputs) share one dtype, `io_dtype`;
 *    A, D, delta_bias, conv weights and all states are float32.  Arithmetic is float32.
 *  - Supported sizes: 1 <= dstate <= 16, d_conv == 4; batch, dim >= 1; seqlen >= 0.
 *  - On a CUDA error the call returns SSM_ERR_CUDA; ssm_last_error_message() gives the text.
 *  - Device-side failures that are not CUDA errors (a pipeline wait that exceeded its time limit)
 *    set a device status word, read and cleared by ssm_device_status().
 */
#ifndef SSM_B300_H
#define SSM_B300_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define SSM_API __attribute__((visibility("default")))
#else
#define SSM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SSM_OK = 0,
  SSM_ERR_INVALID_ARG = 1,   /* null pointer, bad size, bad flag, aliasing, short workspace */
  SSM_ERR_UNSUPPORTED = 2,   /* valid but outside what this build implements (dstate > 16, d_conv != 4) */
  SSM_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed */
  SSM_ERR_TIMEOUT = 4,       /* reported by ssm_device_status(): a device wait gave up */
  SSM_ERR_CHECK = 5          /* reported by ssm_device_status() of the checked build: an index check failed */
} ssm_status;

typedef enum { SSM_F32 = 0, SSM_BF16 = 1 } ssm_dtype;

typedef enum {
  SSM_ALGO_AUTO = 0,         /* pick from the shape */
  SSM_ALGO_SINGLE_PASS = 1,  /* one pass over time per channel tile */
  SSM_ALGO_CHUNKED = 2       /* split time into chunks: aggregates, carry, re-run */
} ssm_algorithm;

typedef enum {
  SSM_DISC_DELTA_B = 0,      /* input term Δ·B·x (the Mamba parameterisation) */
  SSM_DISC_ZOH = 1           /* exact zero-order hold: (exp(ΔA) - 1)/A · B · x ("Модуль 8", §4) */
} ssm_discretization;

/* Options for ssm_scan_fwd_ex.  Zero-initialise, then set struct_size = sizeof(ssm_scan_options). */
typedef struct {
  int struct_size;
  int algorithm;             /* ssm_algorithm */
  int64_t chunk_len;         /* SSM_ALGO_CHUNKED: steps per chunk, a multiple of 64; 0 = choose */
  int discretization;        /* ssm_discretization */
  const float* h0;           /* initial state (batch, dim, dstate) float32, or NULL for zeros */
} ssm_scan_options;

/* ABI version of this header (increments on any signature change). */
SSM_API int ssm_abi_version(void);

/*
 * 1 for the checked debug build (libssm_b300_check.so, compiled with -DSSM_CHECK=1), 0 otherwise.
 * In the checked build every global load and store of the kernels goes through an index check
 * against the buffer's element count; an access outside it is not made (loads read a zeroed sink,
 * stores go to it), the kernel carries on, and the next ssm_device_status() returns SSM_ERR_CHECK.
 * Nothing traps.  The checks cost time: the checked build is for tests, not for measurement.
 */
SSM_API int ssm_checked_build(void);

/* Human-readable name of a status code (static string). */
SSM_API const char* ssm_status_string(ssm_status s);

/* Text of the last error raised on the calling host thread (empty if none). */
SSM_API const char* ssm_last_error_message(void);

/*
 * Bytes of caller-provided device workspace that ssm_scan_fwd needs for this shape with the
 * default algorithm choice.  0 means no workspace is needed.  Never fails; returns 0 for
 * invalid sizes (the scan call then rejects them).
 */
SSM_API size_t ssm_scan_fwd_workspace_size(int batch, int dim, int dstate, int64_t seqlen, ssm_dtype io_dtype);

/* Same, for a given option set (NULL = defaults). */
SSM_API size_t ssm_scan_fwd_workspace_size_ex(int batch, int dim, int dstate, int64_t seqlen, ssm_dtype io_dtype,
                                      const ssm_scan_options* opts);

/*
 * Prefill: the selective scan over a whole sequence.
 *   u, delta, z, y : (batch, dim, seqlen)   io_dtype.  delta holds Δ_raw.  z may be NULL (no gate).
 *   A              : (dim, dstate)          float32, diagonal real state matrix (any sign).
 *   B, C           : (batch, dstate, seqlen) io_dtype, one group shared by all channels.
 *   D, delta_bias  : (dim)                  float32, each may be NULL (treated as zero).
 *   softplus_flag  : nonzero: Δ = softplus(Δ_raw + bias); zero: Δ = Δ_raw + bias.
 *   last_state     : (batch, dim, dstate)   float32 output h at the last step, or NULL.
 *   workspace      : device buffer of at least ssm_scan_fwd_workspace_size(...) bytes, 256-byte
 *                    aligned; may be NULL when that size is 0.
 * Precision: y matches the exact recurrence to about 1e-6 relative for float32 io and to bf16
 * rounding (plus about 1e-4 relative) for bfloat16 io; the state is kept in float32 throughout.
 * y and last_state are defined once ssm_device_status() has returned SSM_OK for the stream: the
 * balanced schedule hands states from one CTA to the next behind a bounded wait, and a wait that
 * gives up (status SSM_ERR_TIMEOUT) leaves the rest of that CTA's range computed from a zero state.
 */
SSM_API ssm_status ssm_scan_fwd(const void* u, const void* delta, const float* A, const void* B, const void* C,
                        const float* D, const void* z, const float* delta_bias, int softplus_flag,
                        void* y, float* last_state, int batch, int dim, int dstate, int64_t seqlen,
                        ssm_dtype io_dtype, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ssm_scan_fwd with options (NULL = defaults): algorithm choice, chunk length, exact-ZOH input
 * term, initial state. */
SSM_API ssm_status ssm_scan_fwd_ex(const void* u, const void* delta, const float* A, const void* B, const void* C,
                           const float* D, const void* z, const float* delta_bias, int softplus_flag,
                           void* y, float* last_state, int batch, int dim, int dstate, int64_t seqlen,
                           ssm_dtype io_dtype, void* workspace, size_t workspace_bytes,
                           const ssm_scan_options* opts, cudaStream_t stream);

/*
 * Decode: one token of a Mamba-1 layer with its two caches ("Модуль 8", §6 and §14):
 *   window      = [conv_state[b,d,0..2], x_t[b,d]]
 *   u           = SiLU(Σ_k conv_w[d,k] window[k]);   conv_state[b,d,:] <- window[1..3]
 *   Δ           = softplus(delta_t + delta_bias[d])  (or without softplus)
 *   state[b,d,:] <- exp(Δ A[d,:]) ⊙ state[b,d,:] + Δ B_t[b,:] u
 *   y_t[b,d]    = (C_t[b,:]·state[b,d,:] + D[d] u) · SiLU(z_t[b,d])
 *   x_t, delta_t, z_t, y_t : (batch, dim)     io_dtype; z_t may be NULL (no gate)
 *   B_t, C_t               : (batch, dstate)  io_dtype
 *   A                      : (dim, dstate)    float32;  D, delta_bias: (dim) float32 or NULL
 *   state                  : (batch, dim, dstate) float32, updated in place
 *   conv_state             : (batch, dim, dconv-1) float32, updated in place, oldest input first
 *   conv_w                 : (dim, dconv)     float32; conv_w[d, dconv-1] multiplies x_t
 * dconv must be 4.  The conv has no bias.
 */
SSM_API ssm_status ssm_state_update(const void* x_t, const void* delta_t, const float* A, const void* B_t,
                            const void* C_t, const float* D, const void* z_t, float* state,
                            float* conv_state, const float* conv_w, const float* delta_bias,
                            int softplus_flag, void* y_t, int batch, int dim, int dstate, int dconv,
                            ssm_dtype io_dtype, cudaStream_t stream);

/*
 * Prefill scan for callers that cannot allocate device memory.  The paper has no counterpart: this
 * is a library convenience.  Some callers cannot call cudaMalloc or hand over a workspace -- code
 * running where allocation is forbidden or unavailable (a host callback, a plugin hook that must not
 * allocate, a process whose device allocator belongs to another framework, a memory-capped sandbox)
 * or code that cannot afford an allocation on its latency path.  This call allocates nothing:
 * its scratch is a fixed array of ssm_scan_fwd_noalloc_max_scratch() bytes (8 MiB) inside this
 * library's device image, which every GPU that loads the library holds until the process exits.
 *  - Arguments and results are those of ssm_scan_fwd_ex without the workspace: the caller still
 *    passes every input and output buffer.
 *  - Shapes whose schedule needs more scratch than the fixed size return SSM_ERR_UNSUPPORTED
 *    with a message naming the size; use ssm_scan_fwd with a caller workspace for those.
 *  - The first call in a CUDA context (the first on each device, and the first after a
 *    cudaDeviceReset) looks up the array's device address (cudaGetSymbolAddress) with that context
 *    current; make that first call before any stream capture.
 *  - All calls on a device share the one array and it keeps the last call's contents (each call
 *    writes the scratch words it reads, so results do not depend on them).  Two calls whose
 *    kernels overlap on the GPU (different streams, or host threads without ordering) race on
 *    the array: order them.
 */
SSM_API ssm_status ssm_scan_fwd_noalloc(const void* u, const void* delta, const float* A, const void* B,
                                        const void* C, const float* D, const void* z, const float* delta_bias,
                                        int softplus_flag, void* y, float* last_state, int batch, int dim,
                                        int dstate, int64_t seqlen, ssm_dtype io_dtype,
                                        const ssm_scan_options* opts, cudaStream_t stream);

/* Size in bytes of the fixed scratch array used by ssm_scan_fwd_noalloc. */
SSM_API size_t ssm_scan_fwd_noalloc_max_scratch(void);

/* How a prefill call with these sizes and options would run (filled by ssm_scan_fwd_describe). */
typedef struct {
  int struct_size;           /* set to sizeof(ssm_scan_plan) before the call */
  int path;                  /* 0: general kernel (float32 io, or layouts TMA cannot use);
                                1: bf16 fast path (rescaled-state kernel, two lanes per channel;
                                   Δ·B or exact-ZOH input term) */
  int schedule;              /* 0: one CTA per channel tile; 1: balanced persistent ranges; 2: chunked (aggregates, carry, re-run) */
  int nchunks;               /* time chunks (1 unless schedule 2) */
  int64_t chunk_len;         /* steps per chunk */
  int ctas;                  /* CTAs of the main pass */
  int kernel_launches;       /* kernels one call launches (memsets not counted) */
  size_t workspace_bytes;    /* same as ssm_scan_fwd_workspace_size_ex */
} ssm_scan_plan;

/* Describes the plan ssm_scan_fwd_ex would use for these sizes and options, assuming 16-byte
 * aligned buffers (a call with less aligned buffers runs the general kernel in one pass).
 * Returns SSM_ERR_INVALID_ARG / SSM_ERR_UNSUPPORTED like the scan itself; enqueues nothing. */
SSM_API ssm_status ssm_scan_fwd_describe(int batch, int dim, int dstate, int64_t seqlen, ssm_dtype io_dtype,
                                         const ssm_scan_options* opts, ssm_scan_plan* plan);

/*
 * Prefill of the short convolution that feeds the scan: causal depthwise conv1d of width dconv (4)
 * followed by SiLU ("Mamba и State Space Models", "Реализация MambaBlock"; "State Space Models: Mamba и
 * альтернатива Transformer", "Mamba: Selective State Space"; the cache of "Модуль 8", §14):
 *   u[b,d,t] = SiLU( Σ_{k<4} conv_w[d,k] · xpad[b,d,t+k] ),  xpad = [conv_state_in[b,d,0..2], x[b,d,:]]
 *   conv_state_out[b,d,:] = the last three entries of xpad (oldest first), ready for ssm_state_update
 *   x, u            : (batch, dim, seqlen) io_dtype
 *   conv_w          : (dim, dconv) float32, no bias; conv_w[d, dconv-1] multiplies the newest input
 *   conv_state_in   : (batch, dim, dconv-1) float32 or NULL (zeros: a fresh sequence)
 *   conv_state_out  : (batch, dim, dconv-1) float32 or NULL; must not alias conv_state_in
 *   apply_silu      : nonzero applies SiLU (the Mamba block does)
 * dconv must be 4.  Float32 io is computed in double.
 */
SSM_API ssm_status ssm_causal_conv1d_fwd(const void* x, const float* conv_w, const float* conv_state_in, void* u,
                                         float* conv_state_out, int batch, int dim, int64_t seqlen, int dconv,
                                         int apply_silu, ssm_dtype io_dtype, cudaStream_t stream);

/*
 * Backward of the prefill scan: the gradients of sum(dy ⊙ y) with respect to every input of
 * ssm_scan_fwd (zero initial state, Δ·B input term).  The pages define only the forward recurrence;
 * this is its chain rule, computed with the states recomputed from checkpoints every 8 steps instead
 * of stored (the recomputation of the hardware-aware scan: "Mamba: линейная альтернатива
 * трансформеру", "Почему selectivity ломает старый трюк со свёрткой"; the ai.pinkoculture.com concept
 * page, 硬件感知的实现).
 *   inputs      : as ssm_scan_fwd, plus dy (batch, dim, seqlen) io_dtype, the gradient of y
 *   du, ddelta  : (batch, dim, seqlen) io_dtype; ddelta is the gradient of the raw Δ input (before
 *                 delta_bias and softplus)
 *   dz          : (batch, dim, seqlen) io_dtype; required when z is given, NULL when z is NULL
 *   dA          : (dim, dstate) float32, summed over the batch
 *   dB, dC      : (batch, dstate, seqlen) float32, summed over the channels
 *   dD          : (dim) float32 summed over the batch, or NULL (not computed)
 *   ddelta_bias : (dim) float32 summed over the batch, or NULL (not computed)
 * All outputs are overwritten (the call zeroes the accumulated ones itself).  The cross-channel sums
 * use atomic adds, so their last bits can differ from run to run.  Float32 io is computed in double.
 * workspace: ssm_scan_bwd_workspace_size() bytes, 256-byte aligned, no initial contents required.
 */
SSM_API size_t ssm_scan_bwd_workspace_size(int batch, int dim, int dstate, int64_t seqlen, ssm_dtype io_dtype);

SSM_API ssm_status ssm_scan_bwd(const void* u, const void* delta, const float* A, const void* B, const void* C,
                                const float* D, const void* z, const float* delta_bias, int softplus_flag,
                                const void* dy, void* du, void* ddelta, void* dz, float* dA, float* dB, float* dC,
                                float* dD, float* ddelta_bias, int batch, int dim, int dstate, int64_t seqlen,
                                ssm_dtype io_dtype, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Mamba-2 state space duality (SSD) forward: a scalar decay per head and a (headdim, dstate) state per
 * head ("Mamba и State Space Models", "Mamba-2: State Space Duality (SSD)"; "Модуль 8", §7 and §14).
 * Per batch b and head h, with g = h / (nheads / ngroups) the head's B/C group:
 *     Δ_t = softplus(dt[b,t,h] + dt_bias[h])   (or dt + dt_bias when softplus_flag is 0)
 *     H_t = exp(Δ_t A[h]) H_{t-1} + Δ_t x[b,t,h,:] B[b,t,g,:]^T,   H_{-1} = h0[b,h] (or zeros)
 *     y[b,t,h,:] = H_t C[b,t,g,:] + D[h] x[b,t,h,:]
 *   x, y          : (batch, seqlen, nheads, headdim) io_dtype
 *   dt            : (batch, seqlen, nheads) io_dtype
 *   B, C          : (batch, seqlen, ngroups, dstate) io_dtype
 *   A, D, dt_bias : (nheads) float32; D and dt_bias may be NULL (zero)
 *   h0            : (batch, nheads, headdim, dstate) float32 or NULL (zeros)
 *   final_state   : (batch, nheads, headdim, dstate) float32 or NULL
 * This build implements io_dtype SSM_BF16 with headdim 64 and dstate 128 (the pages' Mamba-2
 * geometry); other values return SSM_ERR_UNSUPPORTED.  x, B, C and y must be 16-byte aligned, h0 and
 * final_state 8-byte aligned.  Accumulation and the state are float32 (tensor-core products with the
 * computed operand split into two bf16 terms).  One CTA per (batch, head) sequence, no workspace (see
 * ssm_ssd_fwd_ex for the balanced schedule).  The kernel's waits for its tensor-core results are
 * bounded: y and final_state are defined once ssm_device_status() has returned SSM_OK for the stream
 * (SSM_ERR_TIMEOUT: a wait gave up; y and final_state are then undefined, and no other memory is
 * written).
 */
SSM_API ssm_status ssm_ssd_fwd(const void* x, const void* dt, const float* A, const void* B, const void* C,
                               const float* D, const float* dt_bias, int softplus_flag, const float* h0, void* y,
                               float* final_state, int batch, int64_t seqlen, int nheads, int headdim, int dstate,
                               int ngroups, ssm_dtype io_dtype, cudaStream_t stream);

/*
 * Bytes of device workspace ssm_ssd_fwd_ex needs for its balanced schedule on the current device:
 * nonzero when there are more (batch, head) sequences than CTAs of the kernel fit on the device at
 * once (or than `ctas`, when ctas > 0), 0 when one CTA per sequence runs (the workspace is then not
 * used).  Returns 0 for invalid sizes or without a device.
 */
SSM_API size_t ssm_ssd_fwd_workspace_size(int batch, int64_t seqlen, int nheads, int ctas);

/*
 * ssm_ssd_fwd with a balanced schedule.  One CTA per sequence leaves the last wave of CTAs partly
 * empty when the sequences outnumber the co-resident CTAs (512 sequences on 296 resident CTAs: two
 * waves, the second 73 % full).  Given a workspace, the (sequence, 64-step chunk) units laid end to
 * end are cut into equal ranges, one per co-resident CTA; a sequence split between two ranges passes
 * its state from one CTA to the next through the workspace (the chunk-to-chunk state passing of
 * "Модуль 8", §7), published behind a flag and waited for with a 2 s limit (SSM_ERR_TIMEOUT from
 * ssm_device_status() if it runs out).  CTAs take their ranges in the order they start, so a CTA
 * only waits for one that is already running.
 *   workspace, workspace_bytes : NULL (one CTA per sequence, as ssm_ssd_fwd), or a device buffer of
 *                                at least ssm_ssd_fwd_workspace_size(batch, seqlen, nheads, ctas)
 *                                bytes, 256-byte aligned, no initial contents, not overlapping the
 *                                inputs or outputs; owned by the caller and not used after the
 *                                stream reaches the end of the call
 *   ctas                       : 0 = one range per co-resident CTA; > 0 = at most that many ranges
 * Results equal ssm_ssd_fwd's up to rounding order (the same arithmetic per chunk).  Other arguments,
 * the requirements and the status as ssm_ssd_fwd; SSM_ERR_INVALID_ARG also for ctas < 0, a too small
 * or misaligned workspace, or one that overlaps y or final_state.
 */
SSM_API ssm_status ssm_ssd_fwd_ex(const void* x, const void* dt, const float* A, const void* B, const void* C,
                                  const float* D, const float* dt_bias, int softplus_flag, const float* h0, void* y,
                                  float* final_state, int batch, int64_t seqlen, int nheads, int headdim, int dstate,
                                  int ngroups, ssm_dtype io_dtype, void* workspace, size_t workspace_bytes, int ctas,
                                  cudaStream_t stream);

/*
 * One-token decode step of a Mamba-2 (SSD) layer, updating its state cache in place ("Модуль 8", §14:
 * the Mamba-2 state [batch, nheads, headdim, d_state]; "Mamba и State Space Models", "Mamba-2: State
 * Space Duality (SSD)").  Per batch b and head h (B/C group g = h / (nheads / ngroups)):
 *     Δ = softplus(dt[b,h] + dt_bias[h]);   H = exp(Δ A[h]) H + Δ x[b,h,:] B[b,g,:]^T
 *     y[b,h,:] = H C[b,g,:] + D[h] x[b,h,:]
 *   x_t, y_t  : (batch, nheads, headdim) io_dtype       dt_t : (batch, nheads) io_dtype
 *   B_t, C_t  : (batch, ngroups, dstate) io_dtype       A, D, dt_bias : (nheads) float32 (D, dt_bias may be NULL)
 *   state     : (batch, nheads, headdim, dstate) float32, read and written in place
 * The same recurrence ssm_ssd_fwd computes (equal up to rounding), one step at a time, so decode steps
 * from a prefill's final state continue its sequence.  This build implements io_dtype SSM_BF16, headdim 64,
 * dstate 128 (others SSM_ERR_UNSUPPORTED); state 16-byte aligned, B_t and C_t 16-byte aligned.
 */
SSM_API ssm_status ssm_ssd_state_update(const void* x_t, const void* dt_t, const float* A, const void* B_t,
                                        const void* C_t, const float* D, const float* dt_bias, int softplus_flag,
                                        float* state, void* y_t, int batch, int nheads, int headdim, int dstate,
                                        int ngroups, ssm_dtype io_dtype, cudaStream_t stream);

/*
 * Diagnostic of the device failure path; the pages have no counterpart.  Enqueues one small kernel
 * that performs a bounded wait which nothing can satisfy and gives up after limit_ns nanoseconds
 * (clamped to 1 ms .. 2 s), recording a timeout in the device status word exactly as the library's
 * kernels do when one of their waits runs out:
 *   which = 0: an mbarrier phase that never completes (the wait of the TMA pipelines);
 *   which = 1: a global flag that nothing sets (the wait of the balanced schedule's carry).
 * The next ssm_device_status() then returns SSM_ERR_TIMEOUT and clears the word; the CUDA context
 * stays usable.  Nothing faults, traps or waits without a limit.  Returns SSM_ERR_INVALID_ARG for
 * another `which` (before enqueuing anything) and SSM_ERR_CUDA if the launch fails.
 */
SSM_API ssm_status ssm_selftest_bounded_wait(int which, int64_t limit_ns, cudaStream_t stream);

/*
 * Diagnostic of the balanced schedule's carry wait, on the real prefill and SSD kernels; the pages
 * have no counterpart.  Arms a one-shot fault for the next ssm_scan_fwd / ssm_scan_fwd_ex /
 * ssm_ssd_fwd / ssm_ssd_fwd_ex call made on the calling host thread: if that call runs a balanced
 * schedule (ssm_scan_fwd_describe: schedule 1; ssm_ssd_fwd_ex with a workspace), CTA `cta` computes
 * and writes its carry but never raises the flag that publishes it, and the carry wait of every CTA
 * is limited to limit_ns nanoseconds (clamped to 1 ms .. 2 s).  CTA cta + 1 then gives up its wait,
 * records a timeout in the device status word and finishes its range from a zero state; the next
 * ssm_device_status() returns SSM_ERR_TIMEOUT.  Nothing faults or waits without a limit, and the
 * context stays usable.  A call with another schedule consumes the arming without effect.  Returns
 * SSM_ERR_INVALID_ARG for cta < 0.
 */
SSM_API ssm_status ssm_selftest_withhold_carry(int cta, int64_t limit_ns);

/*
 * Self-test of the index checks (checked build only): enqueues on `stream` one kernel that stores to
 * the element one past a 32-element device buffer through the index check, which redirects the store
 * to a sink inside the library and records the failure; the next ssm_device_status() returns
 * SSM_ERR_CHECK and clears it.  No memory outside the library's own buffers is touched.  The ordinary
 * build returns SSM_ERR_UNSUPPORTED and enqueues nothing.
 */
SSM_API ssm_status ssm_selftest_index_check(cudaStream_t stream);

/*
 * Reads and clears the device status word (synchronises `stream`).  Returns SSM_OK, SSM_ERR_CHECK if
 * (checked build only) an index check failed since the last call, else SSM_ERR_TIMEOUT if a kernel
 * gave up a bounded wait since the last call, or SSM_ERR_CUDA.
 */
SSM_API ssm_status ssm_device_status(cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SSM_B300_H */
