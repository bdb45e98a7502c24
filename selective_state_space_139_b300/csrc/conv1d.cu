// Causal depthwise conv1d (width 4) followed by SiLU, for the prefill of a Mamba block
// ("Mamba и State Space Models", "Реализация MambaBlock": Conv1d with groups = channels and
// d_conv - 1 leading pad values, cropped to the sequence; "State Space Models: Mamba и альтернатива
// Transformer", "Mamba: Selective State Space": SiLU after the conv; "Модуль 8", §6 and §14: the
// conv cache of the last d_conv - 1 inputs).
//
//   u[b,d,t] = SiLU( Σ_{k=0..3} w[d,k] · xpad[b,d,t+k] ),  xpad = [state_in[b,d,0..2], x[b,d,0..L-1]]
//   state_out[b,d,:] = the last three entries of xpad, oldest first
//
// Memory bound (2 + 2 bytes per element for bf16).  One thread per 8-step (16-byte) chunk of a
// channel row: consecutive threads take consecutive chunks, so loads and stores are coalesced
// 128-bit accesses; the three inputs before the chunk come from the neighbouring lane by a
// shuffle (lane 0 of a warp re-reads the previous chunk), or, at t = 0, from the incoming state.
#include "internal.h"
#include "ssm_device.cuh"

namespace ssm {
namespace {

template <typename IO>
__device__ __forceinline__ float io_at(const IO* p, int64_t i) {
  return IoTraits<IO>::to_f32(p[i]);
}

// vectorised path: L % kVec == 0 and 16-byte aligned rows.  A grid of SSM_CONV_BLOCKS_PER_SM blocks per
// SM walks the flat (row, chunk) index space with a grid-sized stride; each iteration a thread issues
// the loads of kPer chunks (one stride apart) before any arithmetic: one with SiLU, whose arithmetic
// makes the kernel issue-bound (two or four chunks, requesting the next chunk before computing the
// current one, or a SiLU with one MUFU operation and a Newton reciprocal were all slower), two without
// it (59.4 us against 62.8 us for one on the 2.8B layer's x).  Consecutive lanes hold consecutive flat chunks, so the three inputs before a chunk come
// from the previous lane by a shuffle (lane 0 re-reads them).  Flat indices fit 32 bits (checked on
// the host).
#ifndef SSM_CONV_BLOCKS_PER_SM
#define SSM_CONV_BLOCKS_PER_SM 32 // blocks of the grid-stride loop per SM (8: 73.9 us, 16: 71.9, 32: 69.8, 64: 69.8)
#endif
template <bool kSilu>
__host__ __device__ constexpr int per_thread() { return kSilu ? 1 : 2; }   // chunks per thread and iteration

// kSilu is a template parameter: tested at run time inside the unrolled outputs it splits the body
// into basic blocks.
template <typename IO, bool kSilu>
__global__ void __launch_bounds__(256) conv1d_vec_kernel(const ConvParams p) {
  using T = IoTraits<IO>;
  constexpr int V = T::kVec;
  constexpr int kPer = per_thread<kSilu>();
  constexpr bool kFast = sizeof(IO) == 2;
  const uint32_t cpr = static_cast<uint32_t>(p.L / V);
  const uint32_t total = static_cast<uint32_t>(p.batch) * p.dim * cpr;
  const uint32_t stride = gridDim.x * blockDim.x;
  const int lane = threadIdx.x & 31;
  const IO* __restrict__ xg = static_cast<const IO*>(p.x);     // x and u never overlap (checked on the host)
  const int64_t nRows = static_cast<int64_t>(p.batch) * p.dim;  // buffer sizes for the checks of checked builds
  const int64_t nIO = nRows * p.L;
  IO* __restrict__ ug = static_cast<IO*>(p.u);
  for (uint32_t f0 = blockIdx.x * blockDim.x + threadIdx.x; f0 - lane < total; f0 += kPer * stride) {
    uint32_t row[kPer], c[kPer];
    bool live[kPer];
    uint4 raw[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const uint32_t f = f0 + i * stride;
      live[i] = f < total;
      const uint32_t fl = live[i] ? f : total - 1;   // lanes past the end mirror the last chunk
      row[i] = fl / cpr;
      c[i] = fl - row[i] * cpr;
      raw[i] = __ldg(reinterpret_cast<const uint4*>(checked(xg, static_cast<int64_t>(fl) * V, nIO, V)));
    }
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int64_t rbase = static_cast<int64_t>(row[i]) * p.L;
      const int d = static_cast<int>(row[i] % static_cast<uint32_t>(p.dim));
      float xv[V];
      unpack_chunk(raw[i], xv, IO());
      float up[3];
#pragma unroll
      for (int k = 0; k < 3; ++k) up[k] = __shfl_up_sync(0xffffffffu, xv[V - 3 + k], 1);
      float prev[3];
      if (c[i] > 0 && lane > 0) {
        prev[0] = up[0]; prev[1] = up[1]; prev[2] = up[2];
      } else if (c[i] > 0) {
        float pv[V];
        unpack_chunk(__ldg(reinterpret_cast<const uint4*>(checked(xg, rbase + (c[i] - 1) * V, nIO, V))), pv, IO());
        prev[0] = pv[V - 3]; prev[1] = pv[V - 2]; prev[2] = pv[V - 1];
      } else if (p.state_in) {
        const float* si = checked(p.state_in, static_cast<int64_t>(row[i]) * 3, nRows * 3, 3);
        prev[0] = si[0]; prev[1] = si[1]; prev[2] = si[2];
      } else {
        prev[0] = prev[1] = prev[2] = 0.0f;
      }
      const float4 w = *reinterpret_cast<const float4*>(checked(p.w, static_cast<int64_t>(d) * 4, static_cast<int64_t>(p.dim) * 4, 4));
      float win[V + 3];
      win[0] = prev[0]; win[1] = prev[1]; win[2] = prev[2];
#pragma unroll
      for (int j = 0; j < V; ++j) win[3 + j] = xv[j];
      float out[V];
#pragma unroll
      for (int j = 0; j < V; ++j) {
        if constexpr (kFast) {
          const float s = fmaf(w.w, win[j + 3], fmaf(w.z, win[j + 2], fmaf(w.y, win[j + 1], w.x * win[j])));
          out[j] = kSilu ? silu_fast(s) : s;
        } else {
          const double s = static_cast<double>(w.x) * win[j] + static_cast<double>(w.y) * win[j + 1] +
                           static_cast<double>(w.z) * win[j + 2] + static_cast<double>(w.w) * win[j + 3];
          out[j] = static_cast<float>(kSilu ? s / (1.0 + exp(-s)) : s);
        }
      }
      if (live[i]) {
        *reinterpret_cast<uint4*>(checked(ug, rbase + c[i] * V, nIO, V)) = pack_chunk(out);
        if (p.state_out && c[i] == cpr - 1) {
          float* so = checked(p.state_out, static_cast<int64_t>(row[i]) * 3, nRows * 3, 3);
          so[0] = xv[V - 3];
          so[1] = xv[V - 2];
          so[2] = xv[V - 1];
        }
      }
    }
  }
}

// general path: one thread per element (any L, any alignment)
template <typename IO>
__global__ void __launch_bounds__(256) conv1d_scalar_kernel(const ConvParams p) {
  constexpr bool kFast = sizeof(IO) == 2;
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t nrows = static_cast<int64_t>(p.batch) * p.dim;
  if (idx >= nrows * p.L) return;
  const int64_t row = idx / p.L;
  const int64_t t = idx % p.L;
  const int d = static_cast<int>(row % p.dim);
  const IO* xr = static_cast<const IO*>(p.x) + row * p.L;
  float win[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int64_t tt = t - 3 + k;   // position in x; negative -> the incoming state
    if (tt >= 0) win[k] = IoTraits<IO>::to_f32(*checked(static_cast<const IO*>(p.x), row * p.L + tt, nrows * p.L));
    else win[k] = p.state_in ? *checked(p.state_in, row * 3 + (tt + 3), nrows * 3) : 0.0f;
  }
  const float* w = checked(p.w, static_cast<int64_t>(d) * 4, static_cast<int64_t>(p.dim) * 4, 4);
  float o;
  if constexpr (kFast) {
    const float s = fmaf(w[3], win[3], fmaf(w[2], win[2], fmaf(w[1], win[1], w[0] * win[0])));
    o = p.silu ? silu_fast(s) : s;
  } else {
    const double s = static_cast<double>(w[0]) * win[0] + static_cast<double>(w[1]) * win[1] +
                     static_cast<double>(w[2]) * win[2] + static_cast<double>(w[3]) * win[3];
    o = static_cast<float>(p.silu ? s / (1.0 + exp(-s)) : s);
  }
  *checked(static_cast<IO*>(p.u), row * p.L + t, nrows * p.L) = IoTraits<IO>::from_f32(o);
  if (p.state_out && t >= p.L - 3) {
    // the last three entries of xpad (L >= 3 here; shorter sequences are handled by the host)
    *checked(p.state_out, row * 3 + (t - (p.L - 3)), nrows * 3) = io_at(xr, t);
  }
}

// L < 3: the outgoing state mixes the incoming state and x; one thread per row does it
__global__ void conv1d_short_state_kernel(const ConvParams p, int io_bf16) {
  const int64_t row = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (row >= static_cast<int64_t>(p.batch) * p.dim) return;
  float pad[6];
  for (int k = 0; k < 3; ++k) pad[k] = p.state_in ? p.state_in[row * 3 + k] : 0.0f;
  for (int64_t t = 0; t < p.L; ++t)
    pad[3 + t] = io_bf16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(p.x)[row * p.L + t])
                         : static_cast<const float*>(p.x)[row * p.L + t];
  for (int k = 0; k < 3; ++k) p.state_out[row * 3 + k] = pad[p.L + k];
}

template <typename IO>
cudaError_t launch(const ConvParams& p, bool vec, cudaStream_t stream) {
  const int64_t nrows = static_cast<int64_t>(p.batch) * p.dim;
  const bool short_seq = p.L < 3;
  ConvParams q = p;
  if (short_seq) q.state_out = nullptr;
  if (p.L > 0) {
    if (vec) {
      int dev = 0, sms = 148;
      if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      const int64_t total = nrows * (p.L / IoTraits<IO>::kVec);
      const int per = p.silu ? per_thread<true>() : per_thread<false>();
      const int64_t want = (total + 256 * per - 1) / (256 * per);
      const int64_t cap = static_cast<int64_t>(SSM_CONV_BLOCKS_PER_SM) * sms;
      const unsigned blocks = static_cast<unsigned>(want < cap ? want : cap);
      if (p.silu) conv1d_vec_kernel<IO, true><<<blocks, 256, 0, stream>>>(q);
      else conv1d_vec_kernel<IO, false><<<blocks, 256, 0, stream>>>(q);
    } else {
      const int64_t n = nrows * p.L;
      conv1d_scalar_kernel<IO><<<static_cast<unsigned>((n + 255) / 256), 256, 0, stream>>>(q);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (short_seq && p.state_out) {
    conv1d_short_state_kernel<<<static_cast<unsigned>((nrows + 255) / 256), 256, 0, stream>>>(p, sizeof(IO) == 2);
    return cudaGetLastError();
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t conv1d_check_read_and_clear(unsigned int* out) { return tu_check_read_and_clear(out); }

cudaError_t conv1d_launch(const ConvParams& p, bool vec, cudaStream_t stream) {
  return p.io_bf16 ? launch<__nv_bfloat16>(p, vec, stream) : launch<float>(p, vec, stream);
}

}  // namespace ssm
