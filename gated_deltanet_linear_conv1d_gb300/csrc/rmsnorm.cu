// rmsnorm.cu - gdn_gated_rmsnorm: out = o / sqrt(mean(o^2) + eps) * gamma * SiLU(z)
// per head row (page "Qwen3.8-27B: from model structure to vLLM inference data
// flow", section 01, gate row Ogate = RMSNorm(o) (.) SiLU(Z); section 08, the
// GDN output gate is SiLU after RMSNorm).
//
// One warp per row of D values; each lane holds D/32 values (4-element, 8-byte
// vectors when D is a multiple of 128). Purely bandwidth-bound: 6 bytes in and
// 2 bytes out per element.
#include "device.cuh"
#include "launch.h"

namespace gdn {

namespace {

constexpr int kThreads = 256;
constexpr int kRowsPerBlock = kThreads / 32;
constexpr int kMaxPerLane = 32;  // D <= 1024

__global__ void __launch_bounds__(kThreads) gated_rmsnorm_kernel(const NormArgs p) {
  const int row = blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= p.rows) return;
  const uint16_t* o = p.o + (size_t)row * p.D;
  const uint16_t* z = p.z + (size_t)row * p.D;
  uint16_t* out = p.out + (size_t)row * p.D;
  // groups of 4 consecutive elements, strided over the lanes
  const int groups = p.D / 4;
  float ov[kMaxPerLane];
  float ss = 0.f;
#pragma unroll
  for (int u = 0; u < kMaxPerLane / 4; ++u) {
    const int gi = lane + 32 * u;
    if (gi < groups) {
      const uint2 raw = *reinterpret_cast<const uint2*>(o + 4 * gi);
      ov[4 * u + 0] = bf16_to_f32(raw.x & 0xffff);
      ov[4 * u + 1] = bf16_to_f32(raw.x >> 16);
      ov[4 * u + 2] = bf16_to_f32(raw.y & 0xffff);
      ov[4 * u + 3] = bf16_to_f32(raw.y >> 16);
#pragma unroll
      for (int e = 0; e < 4; ++e) ss = fmaf(ov[4 * u + e], ov[4 * u + e], ss);
    }
  }
  ss = warp_sum(ss);
  const float rinv = rsqrtf(ss / (float)p.D + p.eps);
#pragma unroll
  for (int u = 0; u < kMaxPerLane / 4; ++u) {
    const int gi = lane + 32 * u;
    if (gi < groups) {
      const uint2 zr = *reinterpret_cast<const uint2*>(z + 4 * gi);
      const float4 gm = *reinterpret_cast<const float4*>(p.gamma + 4 * gi);
      const float zf[4] = {bf16_to_f32(zr.x & 0xffff), bf16_to_f32(zr.x >> 16), bf16_to_f32(zr.y & 0xffff),
                           bf16_to_f32(zr.y >> 16)};
      const float gf[4] = {gm.x, gm.y, gm.z, gm.w};
      uint16_t r[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) r[e] = f32_to_bf16(ov[4 * u + e] * rinv * gf[e] * silu(zf[e]));
      uint2 packed;
      packed.x = (uint32_t)r[0] | ((uint32_t)r[1] << 16);
      packed.y = (uint32_t)r[2] | ((uint32_t)r[3] << 16);
      *reinterpret_cast<uint2*>(out + 4 * gi) = packed;
    }
  }
}

}  // namespace

cudaError_t launch_gated_rmsnorm(const NormArgs& a, cudaStream_t stream) {
  dim3 grid((a.rows + kRowsPerBlock - 1) / kRowsPerBlock, 1, 1);
  gated_rmsnorm_kernel<<<grid, kThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace gdn
