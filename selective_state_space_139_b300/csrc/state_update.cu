// One-token decode step of a Mamba-1 layer with its two caches ("Модуль 8. Альтернативы
// Transformer: SSM, Mamba и гибриды", §6 and §14; conv + SiLU as in "State Space Models: Mamba и
// альтернатива Transformer", "Mamba: Selective State Space"):
//   u = SiLU(Σ_k w[d,k] · [conv_state, x_t][k]);  conv_state <- last 3 raw inputs
//   Δ = softplus(Δ_raw + bias);  h <- exp(Δ A) ⊙ h + Δ B_t u;  y = (C_t·h + D u) · SiLU(z_t)
//
// The step is bound by HBM traffic on the float32 state (read + write 64 bytes per channel for
// dstate 16).  Four lanes share a channel, each owning four consecutive states, so a warp moves
// 8 channels x 64 contiguous bytes with 128-bit accesses; the per-channel scalars are computed
// redundantly by the four lanes and the readout is reduced with two shuffles.
#include "internal.h"
#include "ssm_device.cuh"

namespace ssm {
namespace {

constexpr int kLanesPerChannel = 4;
constexpr int kThreads = 256;
constexpr int kChannelsPerBlock = kThreads / kLanesPerChannel;

template <typename IO>
__device__ __forceinline__ float ld_io(const void* p, int64_t i) {
  return IoTraits<IO>::to_f32(static_cast<const IO*>(p)[i]);
}

template <typename IO, bool kFull16>
__global__ void __launch_bounds__(kThreads) state_update_kernel(const DecodeParams p) {
  constexpr bool kFast = sizeof(IO) == 2;
  const int tid = threadIdx.x;
  // channel indices fit 32 bits (batch * dim < 2^31 is checked on the host): 32-bit division only
  const int c_raw = static_cast<int>(blockIdx.x) * kChannelsPerBlock + tid / kLanesPerChannel;
  const int j = tid % kLanesPerChannel;
  const int nchan = p.batch * p.dim;
  // lanes past the last channel still take part in the shuffles; they read a valid channel and
  // write nothing
  const bool live = c_raw < nchan;
  const int c32 = live ? c_raw : nchan - 1;
  const int b = c32 / p.dim;
  const int d = c32 - b * p.dim;
  const int64_t c = c32;
  const int N = kFull16 ? 16 : p.N;

  // conv window [cs0, cs1, cs2, x_t] and its weights
  const float x = ld_io<IO>(p.x, c);
  float* cs = p.conv_state + c * 3;
  const float cs0 = cs[0], cs1 = cs[1], cs2 = cs[2];
  float4 w;
  if (kFull16) {
    w = *reinterpret_cast<const float4*>(p.conv_w + static_cast<int64_t>(d) * 4);
  } else {
    const float* wr = p.conv_w + static_cast<int64_t>(d) * 4;
    w = make_float4(wr[0], wr[1], wr[2], wr[3]);
  }
  const float s = fmaf(w.w, x, fmaf(w.z, cs2, fmaf(w.y, cs1, w.x * cs0)));
  const float u = kFast ? silu_fast(s) : silu_accurate(s);

  const float v = ld_io<IO>(p.delta, c) + (p.bias ? p.bias[d] : 0.0f);
  const float dl = p.softplus ? (kFast ? softplus_fast(v) : softplus_accurate(v)) : v;
  const float wu = dl * u;

  float hv[4], av[4], bv[4], cv[4];
  float* srow = p.state + c * N;
  const float* arow = p.A + static_cast<int64_t>(d) * N;
  const int64_t bcrow = static_cast<int64_t>(b) * N;
  if (kFull16) {
    const float4 h4 = *reinterpret_cast<const float4*>(srow + 4 * j);
    const float4 a4 = *reinterpret_cast<const float4*>(arow + 4 * j);
    hv[0] = h4.x; hv[1] = h4.y; hv[2] = h4.z; hv[3] = h4.w;
    av[0] = a4.x; av[1] = a4.y; av[2] = a4.z; av[3] = a4.w;
    if (kFast) {
      const uint2 braw = *reinterpret_cast<const uint2*>(static_cast<const IO*>(p.B) + bcrow + 4 * j);
      const uint2 craw = *reinterpret_cast<const uint2*>(static_cast<const IO*>(p.C) + bcrow + 4 * j);
      bv[0] = bf16lo_to_f32(braw.x); bv[1] = bf16hi_to_f32(braw.x);
      bv[2] = bf16lo_to_f32(braw.y); bv[3] = bf16hi_to_f32(braw.y);
      cv[0] = bf16lo_to_f32(craw.x); cv[1] = bf16hi_to_f32(craw.x);
      cv[2] = bf16lo_to_f32(craw.y); cv[3] = bf16hi_to_f32(craw.y);
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        bv[i] = ld_io<IO>(p.B, bcrow + 4 * j + i);
        cv[i] = ld_io<IO>(p.C, bcrow + 4 * j + i);
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int n = 4 * j + i;
      const bool in = n < N;
      hv[i] = in ? srow[n] : 0.0f;
      av[i] = in ? arow[n] : 0.0f;
      bv[i] = in ? ld_io<IO>(p.B, bcrow + n) : 0.0f;
      cv[i] = in ? ld_io<IO>(p.C, bcrow + n) : 0.0f;
    }
  }

  float py = 0.0f;
  double pyd = 0.0, ud = 0.0;
  if constexpr (kFast) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float a = ex2_approx(dl * av[i] * kLog2e);
      hv[i] = fmaf(a, hv[i], wu * bv[i]);
      py = fmaf(cv[i], hv[i], py);
    }
    py += __shfl_xor_sync(0xffffffffu, py, 1);
    py += __shfl_xor_sync(0xffffffffu, py, 2);
  } else {
    // float32 io: conv, Δ, decays and readout in double; the state is stored back as float32
    const double sd = static_cast<double>(w.w) * x + static_cast<double>(w.z) * cs2 +
                      static_cast<double>(w.y) * cs1 + static_cast<double>(w.x) * cs0;
    ud = sd / (1.0 + exp(-sd));
    const double vd = static_cast<double>(ld_io<IO>(p.delta, c)) + (p.bias ? p.bias[d] : 0.0f);
    const double dld = p.softplus ? (vd > 0.0 ? vd + log1p(exp(-vd)) : log1p(exp(vd))) : vd;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const double hn = exp(dld * av[i]) * hv[i] + dld * bv[i] * ud;
      hv[i] = static_cast<float>(hn);
      pyd += cv[i] * hn;
    }
    pyd += __shfl_xor_sync(0xffffffffu, pyd, 1);
    pyd += __shfl_xor_sync(0xffffffffu, pyd, 2);
  }

  // every lane has read the old conv window before any lane overwrites it
  __syncwarp();
  if (!live) return;
  if (kFull16) {
    *reinterpret_cast<float4*>(srow + 4 * j) = make_float4(hv[0], hv[1], hv[2], hv[3]);
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (4 * j + i < N) srow[4 * j + i] = hv[i];
  }
  if (j < 3) cs[j] = j == 0 ? cs1 : (j == 1 ? cs2 : x);
  if (j == 0) {
    if constexpr (kFast) {
      float y = fmaf(p.D ? p.D[d] : 0.0f, u, py);
      if (p.z) y *= silu_fast(ld_io<IO>(p.z, c));
      static_cast<IO*>(p.y)[c] = IoTraits<IO>::from_f32(y);
    } else {
      double y = pyd + (p.D ? static_cast<double>(p.D[d]) : 0.0) * ud;
      if (p.z) {
        const double z = ld_io<IO>(p.z, c);
        y *= z / (1.0 + exp(-z));
      }
      static_cast<IO*>(p.y)[c] = IoTraits<IO>::from_f32(static_cast<float>(y));
    }
  }
}

// bf16 io, dstate 16, aligned buffers: each thread serves kPer channels (slot + 64 k of its block),
// issuing every load before any arithmetic and storing after.  One channel per thread (32
// registers, full occupancy) measured fastest: the bytes in flight come from resident warps.
#ifndef SSM_DECODE_PER
#define SSM_DECODE_PER 1   // channels per thread of the bf16 decode kernel (1 measured fastest)
#endif
constexpr int kPer = SSM_DECODE_PER;

__global__ void __launch_bounds__(kThreads) state_update_bf16_kernel(const DecodeParams p) {
  using IO = __nv_bfloat16;
  const int tid = threadIdx.x;
  const int j = tid % kLanesPerChannel;
  const int slot = tid / kLanesPerChannel;
  const int nchan = p.batch * p.dim;
  const int base = static_cast<int>(blockIdx.x) * (kChannelsPerBlock * kPer);
  int cc[kPer];
  bool live[kPer];
  float4 h4[kPer], a4[kPer], w4[kPer];
  uint2 braw[kPer], craw[kPer];
  float xv[kPer], dv[kPer], zv[kPer], c0[kPer], c1[kPer], c2[kPer], Dv[kPer], bv[kPer];
  // ---- loads
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int craw_i = base + slot + kChannelsPerBlock * k;
    live[k] = craw_i < nchan;
    const int c = live[k] ? craw_i : nchan - 1;
    const int b = c / p.dim;
    const int d = c - b * p.dim;
    cc[k] = c;
    const int64_t c64 = c;
    h4[k] = *reinterpret_cast<const float4*>(p.state + c64 * 16 + 4 * j);
    a4[k] = *reinterpret_cast<const float4*>(p.A + static_cast<int64_t>(d) * 16 + 4 * j);
    w4[k] = *reinterpret_cast<const float4*>(p.conv_w + static_cast<int64_t>(d) * 4);
    braw[k] = *reinterpret_cast<const uint2*>(static_cast<const IO*>(p.B) + static_cast<int64_t>(b) * 16 + 4 * j);
    craw[k] = *reinterpret_cast<const uint2*>(static_cast<const IO*>(p.C) + static_cast<int64_t>(b) * 16 + 4 * j);
    xv[k] = ld_io<IO>(p.x, c64);
    dv[k] = ld_io<IO>(p.delta, c64);
    zv[k] = p.z ? ld_io<IO>(p.z, c64) : 0.0f;
    c0[k] = p.conv_state[c64 * 3 + 0];
    c1[k] = p.conv_state[c64 * 3 + 1];
    c2[k] = p.conv_state[c64 * 3 + 2];
    Dv[k] = p.D ? p.D[d] : 0.0f;
    bv[k] = p.bias ? p.bias[d] : 0.0f;
  }
  // ---- arithmetic
  float yk[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const float4 w = w4[k];
    const float s = fmaf(w.w, xv[k], fmaf(w.z, c2[k], fmaf(w.y, c1[k], w.x * c0[k])));
    const float u = silu_fast(s);
    const float v = dv[k] + bv[k];
    const float dl = p.softplus ? softplus_fast(v) : v;
    const float wu = dl * u;
    const float av[4] = {a4[k].x, a4[k].y, a4[k].z, a4[k].w};
    float hv[4] = {h4[k].x, h4[k].y, h4[k].z, h4[k].w};
    const float bb[4] = {bf16lo_to_f32(braw[k].x), bf16hi_to_f32(braw[k].x), bf16lo_to_f32(braw[k].y),
                         bf16hi_to_f32(braw[k].y)};
    const float cv[4] = {bf16lo_to_f32(craw[k].x), bf16hi_to_f32(craw[k].x), bf16lo_to_f32(craw[k].y),
                         bf16hi_to_f32(craw[k].y)};
    float py = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float a = ex2_approx(dl * av[i] * kLog2e);
      hv[i] = fmaf(a, hv[i], wu * bb[i]);
      py = fmaf(cv[i], hv[i], py);
    }
    h4[k] = make_float4(hv[0], hv[1], hv[2], hv[3]);
    py += __shfl_xor_sync(0xffffffffu, py, 1);
    py += __shfl_xor_sync(0xffffffffu, py, 2);
    float y = fmaf(Dv[k], u, py);
    if (p.z) y *= silu_fast(zv[k]);
    yk[k] = y;
  }
  // ---- stores (every lane read its channel's old conv window in the load phase)
  __syncwarp();
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    if (!live[k]) continue;
    const int64_t c64 = cc[k];
    *reinterpret_cast<float4*>(p.state + c64 * 16 + 4 * j) = h4[k];
    if (j < 3) p.conv_state[c64 * 3 + j] = j == 0 ? c1[k] : (j == 1 ? c2[k] : xv[k]);
    if (j == 0) static_cast<IO*>(p.y)[c64] = IoTraits<IO>::from_f32(yk[k]);
  }
}

template <typename IO>
cudaError_t launch(const DecodeParams& p, cudaStream_t stream) {
  const int64_t nchan = static_cast<int64_t>(p.batch) * p.dim;
  if (sizeof(IO) == 2 && p.vec16) {
    const unsigned blocks =
        static_cast<unsigned>((nchan + kChannelsPerBlock * kPer - 1) / (kChannelsPerBlock * kPer));
    state_update_bf16_kernel<<<blocks, kThreads, 0, stream>>>(p);
    return cudaGetLastError();
  }
  const unsigned blocks = static_cast<unsigned>((nchan + kChannelsPerBlock - 1) / kChannelsPerBlock);
  if (p.vec16) state_update_kernel<IO, true><<<blocks, kThreads, 0, stream>>>(p);
  else state_update_kernel<IO, false><<<blocks, kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t state_update_launch(const DecodeParams& p, cudaStream_t stream) {
  return p.io_bf16 ? launch<__nv_bfloat16>(p, stream) : launch<float>(p, stream);
}

}  // namespace ssm
