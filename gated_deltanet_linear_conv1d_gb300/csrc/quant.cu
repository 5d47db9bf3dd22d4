// quant.cu - FP8 E4M3 block quantisation for the projections around the mixer
// core (page "Qwen3.8-27B: from model structure to vLLM inference data flow",
// section 04, precision and cache: the checkpoint's linear weights are FP8 E4M3
// with one scale per 128 x 128 weight block, and activations are quantised
// dynamically).
//
// Both kernels take the block's largest magnitude a, set the block's scale to
// s = max(a, kMinAmax) / 448 (448 is the largest finite E4M3 value) and store
// each element as E4M3(x / s), rounded to nearest even and saturated; the
// divisions are IEEE-rounded, so the codes are a pure function of the inputs.
//
//  * quant_act_kernel: activations [T][K] bf16, one scale per token and
//    128-element group of K; half a warp per (token, group), 8 elements per lane.
//  * quant_weight_kernel: weights [N][K] bf16, one scale per 128 x 128 block;
//    one 256-thread block per weight block, 64 elements per thread.
#include "device.cuh"
#include "launch.h"

namespace gdn {

namespace {

constexpr float kE4m3Max = 448.f;
constexpr float kMinAmax = 1e-12f;  // an all-zero block gets a tiny positive scale (codes all 0)

// Two fp32 values to two E4M3 codes (round to nearest even, saturate); lo lands in the low byte.
__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t quant4(const float (&v)[4], float s) {
  const uint32_t a = e4m3x2(__fdiv_rn(v[0], s), __fdiv_rn(v[1], s));
  const uint32_t b = e4m3x2(__fdiv_rn(v[2], s), __fdiv_rn(v[3], s));
  return a | (b << 16);
}

// Half a warp per (token, group): lane l of the half holds elements 8l .. 8l+7
// (one 16-byte load); each thread takes kActRounds items, loads first.
constexpr int kActRounds = 2;
constexpr int kActItemsPerBlock = 8 * 2 * kActRounds;

// Index type I: 32-bit unsigned when the item count allows (the item -> (token,
// group) split is then a 32-bit division, done once per item), else 64-bit.
template <typename I>
__global__ void __launch_bounds__(256) quant_act_kernel(const QuantActArgs p) {
  const I groups = (I)(p.K / 128);
  const I items = (I)p.T * groups;
  const int lane = threadIdx.x & 31, sub = lane & 15;
  const I base = ((I)blockIdx.x * 8 + (I)(threadIdx.x >> 5)) * (2 * kActRounds) + (I)(lane >> 4);
  uint4 raw[kActRounds];
  size_t off[kActRounds];  // element offset of this lane's 8 values; the scale index
  size_t soff[kActRounds];
#pragma unroll
  for (int r = 0; r < kActRounds; ++r) {
    const I item = base + 2 * r;
    raw[r] = make_uint4(0u, 0u, 0u, 0u);
    off[r] = 0;
    soff[r] = 0;
    if (item < items) {
      const I t = item / groups, g = item - t * groups;
      off[r] = (size_t)t * p.K + (size_t)g * 128 + sub * 8;
      soff[r] = (size_t)t * p.scale_t + (size_t)g * p.scale_g;
      raw[r] = *reinterpret_cast<const uint4*>(p.x + off[r]);
    }
  }
#pragma unroll
  for (int r = 0; r < kActRounds; ++r) {
    const I item = base + 2 * r;
    const uint32_t w4[4] = {raw[r].x, raw[r].y, raw[r].z, raw[r].w};
    float v0[4], v1[4];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      v0[2 * e] = bf16_to_f32(w4[e] & 0xffff);
      v0[2 * e + 1] = bf16_to_f32(w4[e] >> 16);
      v1[2 * e] = bf16_to_f32(w4[2 + e] & 0xffff);
      v1[2 * e + 1] = bf16_to_f32(w4[2 + e] >> 16);
    }
    float a = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) a = fmaxf(a, fmaxf(fabsf(v0[e]), fabsf(v1[e])));
#pragma unroll
    for (int m = 8; m > 0; m >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, m));  // within the half
    const float s = __fdiv_rn(fmaxf(a, kMinAmax), kE4m3Max);
    if (item < items) {
      *reinterpret_cast<uint2*>(p.x8 + off[r]) = make_uint2(quant4(v0, s), quant4(v1, s));
      if (sub == 0) p.scale[soff[r]] = s;
    }
  }
}

__global__ void __launch_bounds__(256) quant_weight_kernel(const QuantWeightArgs p) {
  __shared__ float wmax[8];
  const int kb = blockIdx.x, nb = blockIdx.y;
  const int r = threadIdx.x >> 1, half = threadIdx.x & 1;  // row r of the block, columns half*64 ..
  const int n = nb * 128 + r;
  const bool live = n < p.N;
  const size_t off = (size_t)n * p.K + (size_t)kb * 128 + half * 64;
  uint4 raw[8];
  float a = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    raw[i] = live ? reinterpret_cast<const uint4*>(p.w + off)[i] : make_uint4(0u, 0u, 0u, 0u);
    const uint32_t w4[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
#pragma unroll
    for (int j = 0; j < 4; ++j)
      a = fmaxf(a, fmaxf(fabsf(bf16_to_f32(w4[j] & 0xffff)), fabsf(bf16_to_f32(w4[j] >> 16))));
  }
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, m));
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = a;
  __syncthreads();
  a = wmax[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) a = fmaxf(a, wmax[w]);
  const float s = __fdiv_rn(fmaxf(a, kMinAmax), kE4m3Max);
  if (threadIdx.x == 0) p.scale[(size_t)nb * p.scale_n + (size_t)kb * p.scale_k] = s;
  if (!live) return;
  uint32_t q[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t w4[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
    const float v0[4] = {bf16_to_f32(w4[0] & 0xffff), bf16_to_f32(w4[0] >> 16), bf16_to_f32(w4[1] & 0xffff),
                         bf16_to_f32(w4[1] >> 16)};
    const float v1[4] = {bf16_to_f32(w4[2] & 0xffff), bf16_to_f32(w4[2] >> 16), bf16_to_f32(w4[3] & 0xffff),
                         bf16_to_f32(w4[3] >> 16)};
    q[2 * i] = quant4(v0, s);
    q[2 * i + 1] = quant4(v1, s);
  }
  uint4* dst = reinterpret_cast<uint4*>(p.w8 + off);
#pragma unroll
  for (int i = 0; i < 4; ++i) dst[i] = make_uint4(q[4 * i], q[4 * i + 1], q[4 * i + 2], q[4 * i + 3]);
}

}  // namespace

cudaError_t launch_quant_act(const QuantActArgs& a, cudaStream_t stream) {
  const long long items = (long long)a.T * (a.K / 128);
  if (items == 0) return cudaSuccess;
  const unsigned blocks = (unsigned)((items + kActItemsPerBlock - 1) / kActItemsPerBlock);
  if (items + kActItemsPerBlock < (1LL << 32))
    quant_act_kernel<uint32_t><<<blocks, 256, 0, stream>>>(a);
  else
    quant_act_kernel<unsigned long long><<<blocks, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_quant_weight(const QuantWeightArgs& a, cudaStream_t stream) {
  quant_weight_kernel<<<dim3(a.K / 128, (a.N + 127) / 128, 1), 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace gdn
