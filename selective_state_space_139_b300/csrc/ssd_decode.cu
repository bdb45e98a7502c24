// One-token decode step of a Mamba-2 (SSD) layer with its state cache ("Модуль 8. Альтернативы
// Transformer", §14: the Mamba-2 state has the shape [batch, nheads, headdim, d_state] and the input
// term is Δ·B·x; "Mamba и State Space Models", "Mamba-2: State Space Duality (SSD)": a scalar A per
// head).  Per batch b and head h (B/C group g):
//   Δ = softplus(dt[b,h] + dt_bias[h]),  a = exp(Δ A[h])
//   H[p][n] <- a H[p][n] + Δ x[b,h,p] B[b,g,n];   y[b,h,p] = Σ_n C[b,g,n] H[p][n] + D[h] x[b,h,p]
// The step is bound by HBM traffic on the float32 state (32 KB read and written per head for headdim
// 64, d_state 128).  One CTA of 128 threads per (b, h): lane l of warp w holds states 4l .. 4l+3 of
// rows w, w+4, .., w+60, so every warp access moves one contiguous 512-byte row; all loads are issued
// before any arithmetic.  The 16 row readouts of a warp are summed over its lanes with one butterfly.
#include "internal.h"
#include "ssm_device.cuh"

namespace ssm {
namespace {

constexpr int kHd = 64;
constexpr int kNs = 128;
constexpr int kThreads = 128;
constexpr int kRows = kHd / 4;   // rows per warp

__global__ void __launch_bounds__(kThreads) ssd_decode_kernel(const SsdDecodeParams p) {
  const int h = blockIdx.x, b = blockIdx.y;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int grp = h / (p.nheads / p.ngroups);
  const int64_t bh = static_cast<int64_t>(b) * p.nheads + h;
  const int64_t nHead = p.nheads, nBH = static_cast<int64_t>(p.batch) * p.nheads;
  const int64_t nState4 = nBH * kHd * kNs / 4, nBC = static_cast<int64_t>(p.batch) * p.ngroups * kNs;
  float4* const st4 = reinterpret_cast<float4*>(p.state);
  const int64_t st0 = bh * kHd * kNs / 4 + lane;   // row r: st4[st0 + r * 32]
  const int64_t bg = (static_cast<int64_t>(b) * p.ngroups + grp) * kNs + 4 * lane;
  // ---- loads
  float4 hv[kRows];
#pragma unroll
  for (int i = 0; i < kRows; ++i) hv[i] = *checked(st4, st0 + (warp + 4 * i) * 32, nState4);
  const uint2 braw = __ldg(reinterpret_cast<const uint2*>(checked(static_cast<const __nv_bfloat16*>(p.B), bg, nBC, 4)));
  const uint2 craw = __ldg(reinterpret_cast<const uint2*>(checked(static_cast<const __nv_bfloat16*>(p.C), bg, nBC, 4)));
  const __nv_bfloat16* const xg = static_cast<const __nv_bfloat16*>(p.x);
  const int64_t nX = nBH * kHd;
  float xv[kRows];
#pragma unroll
  for (int i = 0; i < kRows; ++i) xv[i] = __bfloat162float(*checked(xg, bh * kHd + warp + 4 * i, nX));
  const float v = __bfloat162float(*checked(static_cast<const __nv_bfloat16*>(p.dt), bh, nBH)) +
                  (p.dt_bias ? *checked(p.dt_bias, h, nHead) : 0.0f);
  const float Ah = *checked(p.A, h, nHead);
  const float Dh = p.D ? *checked(p.D, h, nHead) : 0.0f;
  // ---- arithmetic
  const float dl = p.softplus ? softplus_fast(v) : v;
  const float a = ex2_approx(dl * Ah * kLog2e);
  const float b0 = bf16lo_to_f32(braw.x), b1 = bf16hi_to_f32(braw.x), b2 = bf16lo_to_f32(braw.y),
              b3 = bf16hi_to_f32(braw.y);
  const float c0 = bf16lo_to_f32(craw.x), c1 = bf16hi_to_f32(craw.x), c2 = bf16lo_to_f32(craw.y),
              c3 = bf16hi_to_f32(craw.y);
  float part[kRows];
#pragma unroll
  for (int i = 0; i < kRows; ++i) {
    const float dlx = dl * xv[i];
    float4& hh = hv[i];
    hh.x = fmaf(a, hh.x, dlx * b0);
    hh.y = fmaf(a, hh.y, dlx * b1);
    hh.z = fmaf(a, hh.z, dlx * b2);
    hh.w = fmaf(a, hh.w, dlx * b3);
    part[i] = fmaf(c3, hh.w, fmaf(c2, hh.z, fmaf(c1, hh.y, c0 * hh.x)));
  }
  // ---- stores of the state, then the readouts: butterfly over lane bits 4..1 (16 values -> 1) and a
  // last exchange over bit 0; lane l then holds the sum of row warp + 4 ((l >> 1) & 15)
#pragma unroll
  for (int i = 0; i < kRows; ++i) *checked(st4, st0 + (warp + 4 * i) * 32, nState4) = hv[i];
#pragma unroll
  for (int w = 16, cnt = kRows; w >= 2; w >>= 1, cnt >>= 1) {
    const bool upper = (lane & w) != 0;
    const int half = cnt / 2;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = upper ? part[i] : part[i + half];
      const float keep = upper ? part[i + half] : part[i];
      part[i] = keep + __shfl_xor_sync(0xffffffffu, send, w);
    }
  }
  part[0] += __shfl_xor_sync(0xffffffffu, part[0], 1);
  if ((lane & 1) == 0) {
    const int i = (lane >> 1) & 15;
    const int r = warp + 4 * i;
    *checked(static_cast<__nv_bfloat16*>(p.y), bh * kHd + r, nX) =
        __float2bfloat16_rn(part[0] + Dh * __bfloat162float(*checked(xg, bh * kHd + r, nX)));
  }
}

}  // namespace

cudaError_t ssd_decode_launch(const SsdDecodeParams& p, cudaStream_t stream) {
  ssd_decode_kernel<<<dim3(p.nheads, p.batch), kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t ssd_decode_check_read_and_clear(unsigned int* out) { return tu_check_read_and_clear(out); }

}  // namespace ssm
