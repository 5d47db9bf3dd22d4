// conv.cu - gdn_conv_update: varlen causal depthwise conv (4 taps) + SiLU
// with the per-slot history updated in place (page "Qwen3.8-27B: from model
// structure to vLLM inference data flow", section 01, conv row and the L00
// table's conv-history row).
//
// One thread per (request, channel) walks the request's tokens with a sliding
// window of the last three inputs in registers; a warp covers 32 consecutive
// channels, so every token row is read and written coalesced. The same thread
// reads the old history and writes the new one, so the in-place update has no
// cross-thread ordering to respect.
#include "device.cuh"
#include "launch.h"

namespace gdn {

namespace {

constexpr int kThreads = 128;

__global__ void __launch_bounds__(kThreads) conv_kernel(const ConvArgs p) {
  const int c = blockIdx.x * kThreads + threadIdx.x;
  const int n = blockIdx.y;
  if (c >= p.CH) return;
  const int slot = p.slot_idx[n];
  if (slot < 0) return;
  const int t0 = p.qsl[n], t1 = p.qsl[n + 1];
  if (t0 < 0 || t1 < t0 || t1 > p.T || (n == 0 && t0 != 0) || (n == p.N - 1 && t1 != p.T)) {
    if (c == 0) report(p.dev_err, GDN_DEVERR_OFFSETS);
    return;
  }
  if (slot >= p.Rs) {
    if (c == 0) report(p.dev_err, GDN_DEVERR_SLOT);
    return;
  }
  const int L = t1 - t0;
  if (L == 0) return;
  const bool init = p.has_init ? p.has_init[n] != 0 : true;
  const float4 w = *reinterpret_cast<const float4*>(p.conv_w + (size_t)c * kTaps);
  uint16_t* hp = p.conv_hist + ((size_t)slot * p.CH + c) * (kTaps - 1);
  uint16_t h0 = 0, h1 = 0, h2 = 0;  // oldest .. newest
  if (init) {
    h0 = hp[0];
    h1 = hp[1];
    h2 = hp[2];
  }
  const uint16_t* x = p.x + (size_t)t0 * p.CH + c;
  uint16_t* y = p.y + (size_t)t0 * p.CH + c;
#pragma unroll 4
  for (int t = 0; t < L; ++t) {
    const uint16_t xb = x[(size_t)t * p.CH];
    float pre = w.x * bf16_to_f32(xb);
    pre = fmaf(w.y, bf16_to_f32(h2), pre);
    pre = fmaf(w.z, bf16_to_f32(h1), pre);
    pre = fmaf(w.w, bf16_to_f32(h0), pre);
    y[(size_t)t * p.CH] = f32_to_bf16(silu(pre));
    h0 = h1;
    h1 = h2;
    h2 = xb;
  }
  hp[0] = h0;
  hp[1] = h1;
  hp[2] = h2;
}

}  // namespace

cudaError_t launch_conv(const ConvArgs& a, cudaStream_t stream) {
  dim3 grid((a.CH + kThreads - 1) / kThreads, a.N, 1);
  conv_kernel<<<grid, kThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace gdn
