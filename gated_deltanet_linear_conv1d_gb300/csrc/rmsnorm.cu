// rmsnorm.cu - the two RMSNorms of the GDN layer (page "Qwen3.8-27B: from model
// structure to vLLM inference data flow", section 01 operator table):
//
//  * gdn_gated_rmsnorm: out = o / sqrt(mean(o^2) + eps) * gamma * SiLU(z) per
//    head row (gate row Ogate = RMSNorm(o) (.) SiLU(Z); section 08, the GDN
//    output gate is SiLU after RMSNorm). One warp per row of D values, each
//    lane holding 4-element (8-byte) groups, several rows per warp with all
//    their loads in flight together. 6 bytes in and 2 out per element.
//  * gdn_rmsnorm: the layer's input norm U = X / sqrt(mean(X^2) + eps) (.) gamma
//    over the hidden size, optionally with the residual add in front of it
//    (residual <- bf16(X + residual), U = RMSNorm(residual) (.) gamma), the
//    fused add-and-norm of page "DeepSeek-V3 inference pipeline walk-through" section 4.2.
//    One 128-thread block per row; each thread holds up to 8 16-byte vectors
//    of the row in registers, so every element is read once and written once.
#include "device.cuh"
#include "launch.h"

namespace gdn {

namespace {

constexpr int kThreads = 256;
constexpr int kWarpsPerBlock = kThreads / 32;

// One warp per row, R rows per warp with every load issued before any row is
// reduced (so a warp keeps 2 R rows of o and z in flight); lane l holds the
// 4-element groups l, l + 32, ... (U of them: D <= 128 U). The head dim of the
// layer (128) takes U = 1, R = 4; other sizes up to 1024 take U = 8, R = 1.
template <int U, int R>
__global__ void __launch_bounds__(kThreads) gated_rmsnorm_kernel(const NormArgs p) {
  const int row0 = (blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5)) * R;
  const int lane = threadIdx.x & 31;
  const int groups = p.D / 4;
  uint2 oraw[R][U], zraw[R][U];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int row = row0 + r;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int gi = lane + 32 * u;
      if (row < p.rows && gi < groups) {
        oraw[r][u] = *reinterpret_cast<const uint2*>(p.o + (size_t)row * p.D + 4 * gi);
        zraw[r][u] = *reinterpret_cast<const uint2*>(p.z + (size_t)row * p.D + 4 * gi);
      } else {
        oraw[r][u] = make_uint2(0u, 0u);
        zraw[r][u] = make_uint2(0u, 0u);
      }
    }
  }
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int row = row0 + r;
    if (row >= p.rows) break;  // uniform over the warp
    float ss = 0.f;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const float f[4] = {bf16_to_f32(oraw[r][u].x & 0xffff), bf16_to_f32(oraw[r][u].x >> 16),
                          bf16_to_f32(oraw[r][u].y & 0xffff), bf16_to_f32(oraw[r][u].y >> 16)};
#pragma unroll
      for (int e = 0; e < 4; ++e) ss = fmaf(f[e], f[e], ss);  // lanes past D hold zeros
    }
    ss = warp_sum(ss);
    const float rinv = rsqrtf(ss / (float)p.D + p.eps);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int gi = lane + 32 * u;
      if (gi < groups) {
        const float of[4] = {bf16_to_f32(oraw[r][u].x & 0xffff), bf16_to_f32(oraw[r][u].x >> 16),
                             bf16_to_f32(oraw[r][u].y & 0xffff), bf16_to_f32(oraw[r][u].y >> 16)};
        const float zf[4] = {bf16_to_f32(zraw[r][u].x & 0xffff), bf16_to_f32(zraw[r][u].x >> 16),
                             bf16_to_f32(zraw[r][u].y & 0xffff), bf16_to_f32(zraw[r][u].y >> 16)};
        const float4 gm = *reinterpret_cast<const float4*>(p.gamma + 4 * gi);
        const float gf[4] = {gm.x, gm.y, gm.z, gm.w};
        uint16_t q[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) q[e] = f32_to_bf16(of[e] * rinv * gf[e] * silu_tanh(zf[e]));
        *reinterpret_cast<uint2*>(p.out + (size_t)row * p.D + 4 * gi) =
            make_uint2((uint32_t)q[0] | ((uint32_t)q[1] << 16), (uint32_t)q[2] | ((uint32_t)q[3] << 16));
      }
    }
  }
}

constexpr int kRowThreads = 128;
constexpr int kMaxVec = 8;  // 16-byte vectors per thread: hidden <= 128 * 8 * 8 = 8192

__device__ __forceinline__ void unpack8(const uint4& v, float* f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

__device__ __forceinline__ uint4 pack8(const float* f) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) w[i] = (uint32_t)f32_to_bf16(f[2 * i]) | ((uint32_t)f32_to_bf16(f[2 * i + 1]) << 16);
  return make_uint4(w[0], w[1], w[2], w[3]);
}

__global__ void __launch_bounds__(kRowThreads) rmsnorm_kernel(const RmsArgs p) {
  __shared__ float part[kRowThreads / 32];
  const size_t base = (size_t)blockIdx.x * p.D;
  const uint4* x = reinterpret_cast<const uint4*>(p.x + base);
  uint4* res = p.residual ? reinterpret_cast<uint4*>(p.residual + base) : nullptr;
  uint4* out = reinterpret_cast<uint4*>(p.out + base);
  const int nv = p.D / 8;
  uint4 v[kMaxVec], r[kMaxVec];
#pragma unroll
  for (int u = 0; u < kMaxVec; ++u) {
    const int i = threadIdx.x + u * kRowThreads;
    if (i < nv) {
      v[u] = x[i];
      if (res) r[u] = res[i];
    }
  }
  float ss = 0.f;
#pragma unroll
  for (int u = 0; u < kMaxVec; ++u) {
    const int i = threadIdx.x + u * kRowThreads;
    if (i < nv) {
      float f[8];
      unpack8(v[u], f);
      if (res) {  // the sum is rounded to bf16 first: it is the residual stream the norm reads
        float g[8];
        unpack8(r[u], g);
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] += g[e];
        v[u] = pack8(f);
        res[i] = v[u];
        unpack8(v[u], f);
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) ss = fmaf(f[e], f[e], ss);
    }
  }
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < kRowThreads / 32; ++w) tot += part[w];
  const float rinv = rsqrtf(tot / (float)p.D + p.eps);
#pragma unroll
  for (int u = 0; u < kMaxVec; ++u) {
    const int i = threadIdx.x + u * kRowThreads;
    if (i < nv) {
      float f[8];
      unpack8(v[u], f);
      const float4 g0 = reinterpret_cast<const float4*>(p.gamma)[2 * i];
      const float4 g1 = reinterpret_cast<const float4*>(p.gamma)[2 * i + 1];
      const float gf[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) f[e] = f[e] * rinv * gf[e];
      out[i] = pack8(f);
    }
  }
}

}  // namespace

cudaError_t launch_rmsnorm(const RmsArgs& a, cudaStream_t stream) {
  rmsnorm_kernel<<<dim3(a.rows, 1, 1), kRowThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_gated_rmsnorm(const NormArgs& a, cudaStream_t stream) {
  if (a.D <= 128) {
    constexpr int kR = 4;
    const long long per_block = (long long)kWarpsPerBlock * kR;
    gated_rmsnorm_kernel<1, kR><<<(unsigned)((a.rows + per_block - 1) / per_block), kThreads, 0, stream>>>(a);
  } else {
    gated_rmsnorm_kernel<8, 1><<<(unsigned)((a.rows + kWarpsPerBlock - 1) / kWarpsPerBlock), kThreads, 0, stream>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace gdn
