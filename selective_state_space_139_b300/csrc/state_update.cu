// One-token decode step of a Mamba-1 layer with its two caches ("Модуль 8. Альтернативы
// Transformer: SSM, Mamba и гибриды", §6 and §14; conv + SiLU as in "State Space Models: Mamba и
// альтернатива Transformer", "Mamba: Selective State Space"):
//   u = SiLU(Σ_k w[d,k] · [conv_state, x_t][k]);  conv_state <- last 3 raw inputs
//   Δ = softplus(Δ_raw + bias);  h <- exp(Δ A) ⊙ h + Δ B_t u;  y = (C_t·h + D u) · SiLU(z_t)
//
// The step is bound by HBM traffic on the float32 state (read + write 64 bytes per channel for
// dstate 16).  The bf16 kernel gives each thread whole state rows (below); the general kernel (float32
// io, dstate < 16 or unaligned buffers) lets four lanes share a channel, each owning four consecutive
// states, so a warp moves 8 channels x 64 contiguous bytes, with the per-channel scalars computed by
// the four lanes and the readout reduced with two shuffles.
#include "internal.h"
#include "ssm_device.cuh"

namespace ssm {
namespace {

constexpr int kLanesPerChannel = 4;
constexpr int kThreads = 256;
constexpr int kChannelsPerBlock = kThreads / kLanesPerChannel;

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
  const float x = IoTraits<IO>::to_f32(*checked(static_cast<const IO*>(p.x), c, nchan));
  float* cs = checked(p.conv_state, c * 3, static_cast<int64_t>(nchan) * 3, 3);
  const float cs0 = cs[0], cs1 = cs[1], cs2 = cs[2];
  float4 w;
  const float* wr = checked(p.conv_w, static_cast<int64_t>(d) * 4, static_cast<int64_t>(p.dim) * 4, 4);
  if (kFull16) {
    w = *reinterpret_cast<const float4*>(wr);
  } else {
    w = make_float4(wr[0], wr[1], wr[2], wr[3]);
  }
  const float s = fmaf(w.w, x, fmaf(w.z, cs2, fmaf(w.y, cs1, w.x * cs0)));
  const float u = kFast ? silu_fast(s) : silu_accurate(s);

  const float v = IoTraits<IO>::to_f32(*checked(static_cast<const IO*>(p.delta), c, nchan)) +
                  (p.bias ? *checked(p.bias, d, p.dim) : 0.0f);
  const float dl = p.softplus ? (kFast ? softplus_fast(v) : softplus_accurate(v)) : v;
  const float wu = dl * u;

  float hv[4], av[4], bv[4], cv[4];
  float* srow = checked(p.state, c * N, static_cast<int64_t>(nchan) * N, N);
  const float* arow = checked(p.A, static_cast<int64_t>(d) * N, static_cast<int64_t>(p.dim) * N, N);
  const int64_t bcrow = static_cast<int64_t>(b) * N;
  const IO* Brow = checked(static_cast<const IO*>(p.B), bcrow, static_cast<int64_t>(p.batch) * N, N);
  const IO* Crow = checked(static_cast<const IO*>(p.C), bcrow, static_cast<int64_t>(p.batch) * N, N);
  if (kFull16) {
    const float4 h4 = *reinterpret_cast<const float4*>(srow + 4 * j);
    const float4 a4 = *reinterpret_cast<const float4*>(arow + 4 * j);
    hv[0] = h4.x; hv[1] = h4.y; hv[2] = h4.z; hv[3] = h4.w;
    av[0] = a4.x; av[1] = a4.y; av[2] = a4.z; av[3] = a4.w;
    if (kFast) {
      const uint2 braw = *reinterpret_cast<const uint2*>(Brow + 4 * j);
      const uint2 craw = *reinterpret_cast<const uint2*>(Crow + 4 * j);
      bv[0] = bf16lo_to_f32(braw.x); bv[1] = bf16hi_to_f32(braw.x);
      bv[2] = bf16lo_to_f32(braw.y); bv[3] = bf16hi_to_f32(braw.y);
      cv[0] = bf16lo_to_f32(craw.x); cv[1] = bf16hi_to_f32(craw.x);
      cv[2] = bf16lo_to_f32(craw.y); cv[3] = bf16hi_to_f32(craw.y);
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        bv[i] = IoTraits<IO>::to_f32(Brow[4 * j + i]);
        cv[i] = IoTraits<IO>::to_f32(Crow[4 * j + i]);
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int n = 4 * j + i;
      const bool in = n < N;
      hv[i] = in ? srow[n] : 0.0f;
      av[i] = in ? arow[n] : 0.0f;
      bv[i] = in ? IoTraits<IO>::to_f32(Brow[n]) : 0.0f;
      cv[i] = in ? IoTraits<IO>::to_f32(Crow[n]) : 0.0f;
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
    const double vd = static_cast<double>(IoTraits<IO>::to_f32(*checked(static_cast<const IO*>(p.delta), c, nchan))) +
                      (p.bias ? *checked(p.bias, d, p.dim) : 0.0f);
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
      float y = fmaf(p.D ? *checked(p.D, d, p.dim) : 0.0f, u, py);
      if (p.z) y *= silu_fast(IoTraits<IO>::to_f32(*checked(static_cast<const IO*>(p.z), c, nchan)));
      *checked(static_cast<IO*>(p.y), c, nchan) = IoTraits<IO>::from_f32(y);
    } else {
      double y = pyd + (p.D ? static_cast<double>(*checked(p.D, d, p.dim)) : 0.0) * ud;
      if (p.z) {
        const double z = IoTraits<IO>::to_f32(*checked(static_cast<const IO*>(p.z), c, nchan));
        y *= z / (1.0 + exp(-z));
      }
      *checked(static_cast<IO*>(p.y), c, nchan) = IoTraits<IO>::from_f32(static_cast<float>(y));
    }
  }
}

// bf16 io, dstate 16, aligned buffers: one thread per channel d and kBpt batch rows.  The thread
// issues every load first (kBpt whole 64-byte state rows, the A row once for all its rows, B/C rows,
// conv window and scalars), so a warp keeps 4 KB of state in flight, and it computes the conv,
// softplus and gate once per channel.  Measured on the 256 x 5120 decode step: 44.2 us with four
// lanes per channel (512 bytes in flight per warp), 39.5 us with one row per thread, 35.9 us with
// two, 35.4 us with three, 38.9 us with four (210 registers).
constexpr int kThreads1 = 128;
#ifndef SSM_DECODE_BPT
#define SSM_DECODE_BPT 2    // batch rows per thread
#endif
constexpr int kBpt = SSM_DECODE_BPT;

// kZ (a gate is given) and kSp (softplus on Δ) are template parameters, so the per-row arithmetic
// is one basic block.
template <bool kZ, bool kSp>
__global__ void __launch_bounds__(kThreads1) state_update_bf16_kernel(const DecodeParams p) {
  using IO = __nv_bfloat16;
  const int pairs = ((p.batch + kBpt - 1) / kBpt) * p.dim;
  const int t_raw = static_cast<int>(blockIdx.x) * kThreads1 + threadIdx.x;
  if (t_raw >= pairs) return;
  const int bq = t_raw / p.dim;
  const int d = t_raw - bq * p.dim;
  // buffer sizes (elements) for the index checks of checked builds
  const int64_t nBD = static_cast<int64_t>(p.batch) * p.dim;
  // ---- loads: every state row, the A row, conv weights, B/C rows and the per-channel scalars
  const float4* arow = reinterpret_cast<const float4*>(checked(p.A, static_cast<int64_t>(d) * 16, static_cast<int64_t>(p.dim) * 16, 16));
  float4 a4[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) a4[q] = arow[q];
  const float4 w = *reinterpret_cast<const float4*>(checked(p.conv_w, static_cast<int64_t>(d) * 4, static_cast<int64_t>(p.dim) * 4, 4));
  const float Dv = p.D ? *checked(p.D, d, p.dim) : 0.0f;
  const float bv = p.bias ? *checked(p.bias, d, p.dim) : 0.0f;
  float4 h4[kBpt][4];
  uint4 braw[kBpt][2], craw[kBpt][2];
  float xv[kBpt], dv[kBpt], zv[kBpt], c0[kBpt], c1[kBpt], c2[kBpt];
  bool live[kBpt];
  int64_t cc[kBpt];
#pragma unroll
  for (int k = 0; k < kBpt; ++k) {
    const int b0 = bq * kBpt + k;
    live[k] = b0 < p.batch;
    const int b = live[k] ? b0 : p.batch - 1;
    const int64_t c = static_cast<int64_t>(b) * p.dim + d;
    cc[k] = c;
    const float4* srow = reinterpret_cast<const float4*>(checked(p.state, c * 16, nBD * 16, 16));
#pragma unroll
    for (int q = 0; q < 4; ++q) h4[k][q] = srow[q];
    const uint4* brow = reinterpret_cast<const uint4*>(
        checked(static_cast<const IO*>(p.B), static_cast<int64_t>(b) * 16, static_cast<int64_t>(p.batch) * 16, 16));
    const uint4* crow = reinterpret_cast<const uint4*>(
        checked(static_cast<const IO*>(p.C), static_cast<int64_t>(b) * 16, static_cast<int64_t>(p.batch) * 16, 16));
    braw[k][0] = brow[0]; braw[k][1] = brow[1];
    craw[k][0] = crow[0]; craw[k][1] = crow[1];
    xv[k] = IoTraits<IO>::to_f32(*checked(static_cast<const IO*>(p.x), c, nBD));
    dv[k] = IoTraits<IO>::to_f32(*checked(static_cast<const IO*>(p.delta), c, nBD));
    zv[k] = kZ ? IoTraits<IO>::to_f32(*checked(static_cast<const IO*>(p.z), c, nBD)) : 0.0f;
    const float* cs = checked(p.conv_state, c * 3, nBD * 3, 3);
    c0[k] = cs[0]; c1[k] = cs[1]; c2[k] = cs[2];
  }
  // ---- arithmetic and stores
#pragma unroll
  for (int k = 0; k < kBpt; ++k) {
    const float s = fmaf(w.w, xv[k], fmaf(w.z, c2[k], fmaf(w.y, c1[k], w.x * c0[k])));
    const float u = silu_fast(s);
    const float v = dv[k] + bv;
    const float dl = kSp ? softplus_fast(v) : v;
    const float wu = dl * u;
    const float dl2 = dl * kLog2e;
    const uint32_t bw[8] = {braw[k][0].x, braw[k][0].y, braw[k][0].z, braw[k][0].w,
                            braw[k][1].x, braw[k][1].y, braw[k][1].z, braw[k][1].w};
    const uint32_t cw[8] = {craw[k][0].x, craw[k][0].y, craw[k][0].z, craw[k][0].w,
                            craw[k][1].x, craw[k][1].y, craw[k][1].z, craw[k][1].w};
    float py0 = 0.0f, py1 = 0.0f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float hv[4] = {h4[k][q].x, h4[k][q].y, h4[k][q].z, h4[k][q].w};
      const float av[4] = {a4[q].x, a4[q].y, a4[q].z, a4[q].w};
      const float bb[4] = {bf16lo_to_f32(bw[2 * q]), bf16hi_to_f32(bw[2 * q]), bf16lo_to_f32(bw[2 * q + 1]),
                           bf16hi_to_f32(bw[2 * q + 1])};
      const float ccv[4] = {bf16lo_to_f32(cw[2 * q]), bf16hi_to_f32(cw[2 * q]), bf16lo_to_f32(cw[2 * q + 1]),
                            bf16hi_to_f32(cw[2 * q + 1])};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        hv[i] = fmaf(ex2_approx(dl2 * av[i]), hv[i], wu * bb[i]);
        if (i & 1) py1 = fmaf(ccv[i], hv[i], py1);
        else py0 = fmaf(ccv[i], hv[i], py0);
      }
      h4[k][q] = make_float4(hv[0], hv[1], hv[2], hv[3]);
    }
    float y = fmaf(Dv, u, py0 + py1);
    if (kZ) y *= silu_fast(zv[k]);
    if (!live[k]) continue;
    const int64_t c = cc[k];
    float4* sw = reinterpret_cast<float4*>(checked(p.state, c * 16, nBD * 16, 16));
#pragma unroll
    for (int q = 0; q < 4; ++q) sw[q] = h4[k][q];
    float* cs = checked(p.conv_state, c * 3, nBD * 3, 3);
    cs[0] = c1[k];
    cs[1] = c2[k];
    cs[2] = xv[k];
    *checked(static_cast<IO*>(p.y), c, nBD) = IoTraits<IO>::from_f32(y);
  }
}

template <typename IO>
cudaError_t launch(const DecodeParams& p, cudaStream_t stream) {
  const int64_t nchan = static_cast<int64_t>(p.batch) * p.dim;
  if (sizeof(IO) == 2 && p.vec16) {
    const int64_t threads = ((p.batch + kBpt - 1) / kBpt) * static_cast<int64_t>(p.dim);
    const unsigned blocks = static_cast<unsigned>((threads + kThreads1 - 1) / kThreads1);
    if (p.z) {
      if (p.softplus) state_update_bf16_kernel<true, true><<<blocks, kThreads1, 0, stream>>>(p);
      else state_update_bf16_kernel<true, false><<<blocks, kThreads1, 0, stream>>>(p);
    } else {
      if (p.softplus) state_update_bf16_kernel<false, true><<<blocks, kThreads1, 0, stream>>>(p);
      else state_update_bf16_kernel<false, false><<<blocks, kThreads1, 0, stream>>>(p);
    }
    return cudaGetLastError();
  }
  const unsigned blocks = static_cast<unsigned>((nchan + kChannelsPerBlock - 1) / kChannelsPerBlock);
  if (p.vec16) state_update_kernel<IO, true><<<blocks, kThreads, 0, stream>>>(p);
  else state_update_kernel<IO, false><<<blocks, kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t decode_check_read_and_clear(unsigned int* out) { return tu_check_read_and_clear(out); }

cudaError_t state_update_launch(const DecodeParams& p, cudaStream_t stream) {
  return p.io_bf16 ? launch<__nv_bfloat16>(p, stream) : launch<float>(p, stream);
}

}  // namespace ssm
