// prefill.cu - gdn_chunk_prefill: varlen prefill through the whole mixer core
// (page "Qwen3.8-27B: from model structure to vLLM inference data flow",
// section 01 GDN operator table): conv + SiLU fused in, q/k L2 norm, the gated
// delta rule carried across the request, gated RMSNorm.
//
// This is the CUDA-core path: one CTA per (value head h, request n) with 128
// threads, thread r holding row r of the fp32 state (128 registers) for the
// whole request. Tokens are staged 32 at a time: the conv outputs of the
// CTA's q, k and v channels go to shared memory, q and k are normalised there,
// then the recurrence walks the staged tokens (every thread reads the same k
// and q vectors, a shared-memory broadcast), and the staged outputs are gated
// and written. Rows are independent given k, q, alpha, beta, so no reduction
// crosses threads inside the recurrence.
//
// The G CTAs of one key head form a cluster: all read the old conv history of
// their shared q/k channels before a cluster barrier, and the group's first CTA
// writes the new history after the request is done.
#include <cooperative_groups.h>

#include "device.cuh"
#include "launch.h"

namespace cg = cooperative_groups;

namespace gdn {

namespace {

constexpr int kThreads = kHeadDim;  // one thread per state row / channel
constexpr int kStage = 32;          // tokens staged per pass
constexpr float kInvSqrtDk = 0.08838834764831845f;

struct PfSmem {
  float q[kStage][kHeadDim];
  float k[kStage][kHeadDim];
  float v[kStage][kHeadDim];
  float o[kStage][kHeadDim];
  float a[kStage], b[kStage], kq[kStage];
};

__global__ void __launch_bounds__(kThreads, 2) prefill_kernel(const PrefillArgs p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  PfSmem& sm = *reinterpret_cast<PfSmem*>(smem_raw);
  const int h = blockIdx.x, n = blockIdx.y;
  const int g = h % p.G, j = h / p.G;
  const int r = threadIdx.x, warp = r >> 5, lane = r & 31;

  const int slot = p.slot_idx[n];
  if (slot < 0) return;  // padding (uniform over the cluster)
  const int t0 = p.qsl[n], t1 = p.qsl[n + 1];
  if (t0 < 0 || t1 < t0 || t1 > p.T || (n == 0 && t0 != 0) || (n == p.N - 1 && t1 != p.T)) {
    if (r == 0 && g == 0) report(p.dev_err, GDN_DEVERR_OFFSETS);
    return;
  }
  if (slot >= p.Rs) {
    if (r == 0 && g == 0) report(p.dev_err, GDN_DEVERR_SLOT);
    return;
  }
  if (t1 == t0) return;  // no tokens: the slot is left untouched (uniform over the cluster)
  const bool init = p.has_init ? p.has_init[n] != 0 : true;

  // channels of this thread: q head j, k head j, v head h, element r
  const int gc[3] = {j * kHeadDim + r, (p.Hk + j) * kHeadDim + r, 2 * p.Hk * kHeadDim + h * kHeadDim + r};
  float4 w[3];
  uint16_t hb[3][3];  // conv windows: oldest .. newest input, per part
#pragma unroll
  for (int u = 0; u < 3; ++u) {
    w[u] = *reinterpret_cast<const float4*>(p.conv_w + (size_t)gc[u] * kTaps);
    const uint16_t* hp = p.conv_hist + ((size_t)slot * p.CH + gc[u]) * (kTaps - 1);
    hb[u][0] = init ? hp[0] : 0;
    hb[u][1] = init ? hp[1] : 0;
    hb[u][2] = init ? hp[2] : 0;
  }
  float* Srow_g = p.state + (((size_t)slot * p.Hv + h) * kHeadDim + r) * kHeadDim;
  float S[kHeadDim];
#pragma unroll
  for (int c = 0; c < kHeadDim; c += 4) {
    float4 v4 = init ? *reinterpret_cast<const float4*>(Srow_g + c) : make_float4(0.f, 0.f, 0.f, 0.f);
    S[c] = v4.x;
    S[c + 1] = v4.y;
    S[c + 2] = v4.z;
    S[c + 3] = v4.w;
  }
  // All CTAs of the key-head group have read the old history from here on.
  cg::this_cluster().sync();

  for (int c0 = t0; c0 < t1; c0 += kStage) {
    const int L = min(kStage, t1 - c0);
    // ---- a2: conv + SiLU of the staged tokens
    for (int t = 0; t < L; ++t) {
      const size_t rowx = (size_t)(c0 + t) * p.CH;
#pragma unroll
      for (int u = 0; u < 3; ++u) {
        const uint16_t xb = p.qkv0[rowx + gc[u]];
        float pre = w[u].x * bf16_to_f32(xb);
        pre = fmaf(w[u].y, bf16_to_f32(hb[u][2]), pre);
        pre = fmaf(w[u].z, bf16_to_f32(hb[u][1]), pre);
        pre = fmaf(w[u].w, bf16_to_f32(hb[u][0]), pre);
        const float y = silu(pre);
        if (u == 0) sm.q[t][r] = y;
        else if (u == 1) sm.k[t][r] = y;
        else sm.v[t][r] = y;
        hb[u][0] = hb[u][1];
        hb[u][1] = hb[u][2];
        hb[u][2] = xb;
      }
    }
    if (r < L) {
      const size_t ai = (size_t)(c0 + r) * p.Hv + h;
      sm.a[r] = p.alpha[ai];
      sm.b[r] = p.beta[ai];
    }
    __syncthreads();
    // ---- a3: L2 norm of q and k; warp w takes tokens w, w+4, ...
    for (int t = warp; t < L; t += kThreads / 32) {
      float4 q4 = reinterpret_cast<const float4*>(sm.q[t])[lane];
      float4 k4 = reinterpret_cast<const float4*>(sm.k[t])[lane];
      const float sq = warp_sum(q4.x * q4.x + q4.y * q4.y + q4.z * q4.z + q4.w * q4.w);
      const float sk = warp_sum(k4.x * k4.x + k4.y * k4.y + k4.z * k4.z + k4.w * k4.w);
      const float iq = rsqrtf(sq + 1e-12f), ik = rsqrtf(sk + 1e-12f);
      q4.x *= iq; q4.y *= iq; q4.z *= iq; q4.w *= iq;
      k4.x *= ik; k4.y *= ik; k4.z *= ik; k4.w *= ik;
      reinterpret_cast<float4*>(sm.q[t])[lane] = q4;
      reinterpret_cast<float4*>(sm.k[t])[lane] = k4;
      const float kq = warp_sum(q4.x * k4.x + q4.y * k4.y + q4.z * k4.z + q4.w * k4.w);
      if (lane == 0) sm.kq[t] = kq;
    }
    __syncthreads();
    // ---- a4: the recurrence, row r of the state in registers
    for (int t = 0; t < L; ++t) {
      const float a = sm.a[t], b = sm.b[t];
      const float4* k4p = reinterpret_cast<const float4*>(sm.k[t]);
      const float4* q4p = reinterpret_cast<const float4*>(sm.q[t]);
      float pk0 = 0.f, pk1 = 0.f, pq0 = 0.f, pq1 = 0.f;
#pragma unroll
      for (int c = 0; c < kHeadDim; c += 8) {
        const float4 ka = k4p[c / 4], kb = k4p[c / 4 + 1];
        const float4 qa = q4p[c / 4], qb = q4p[c / 4 + 1];
        pk0 = fmaf(S[c], ka.x, pk0); pk0 = fmaf(S[c + 1], ka.y, pk0);
        pk0 = fmaf(S[c + 2], ka.z, pk0); pk0 = fmaf(S[c + 3], ka.w, pk0);
        pk1 = fmaf(S[c + 4], kb.x, pk1); pk1 = fmaf(S[c + 5], kb.y, pk1);
        pk1 = fmaf(S[c + 6], kb.z, pk1); pk1 = fmaf(S[c + 7], kb.w, pk1);
        pq0 = fmaf(S[c], qa.x, pq0); pq0 = fmaf(S[c + 1], qa.y, pq0);
        pq0 = fmaf(S[c + 2], qa.z, pq0); pq0 = fmaf(S[c + 3], qa.w, pq0);
        pq1 = fmaf(S[c + 4], qb.x, pq1); pq1 = fmaf(S[c + 5], qb.y, pq1);
        pq1 = fmaf(S[c + 6], qb.z, pq1); pq1 = fmaf(S[c + 7], qb.w, pq1);
      }
      const float sk = pk0 + pk1, sq = pq0 + pq1;
      const float e = sm.v[t][r] - a * sk;  // v - Sbar k
      const float be = b * e;
      sm.o[t][r] = fmaf(be, sm.kq[t], a * sq) * kInvSqrtDk;
#pragma unroll
      for (int c = 0; c < kHeadDim; c += 4) {
        const float4 k4 = k4p[c / 4];
        S[c] = fmaf(be, k4.x, a * S[c]);
        S[c + 1] = fmaf(be, k4.y, a * S[c + 1]);
        S[c + 2] = fmaf(be, k4.z, a * S[c + 2]);
        S[c + 3] = fmaf(be, k4.w, a * S[c + 3]);
      }
    }
    __syncthreads();
    // ---- a5: gated RMSNorm of the staged outputs; warp w takes tokens w, w+4, ...
    for (int t = warp; t < L; t += kThreads / 32) {
      const float4 o4 = reinterpret_cast<const float4*>(sm.o[t])[lane];
      const size_t base = ((size_t)(c0 + t) * p.Hv + h) * kHeadDim + lane * 4;
      if (p.o) {
        uint2 packed;
        packed.x = (uint32_t)f32_to_bf16(o4.x) | ((uint32_t)f32_to_bf16(o4.y) << 16);
        packed.y = (uint32_t)f32_to_bf16(o4.z) | ((uint32_t)f32_to_bf16(o4.w) << 16);
        *reinterpret_cast<uint2*>(p.o + base) = packed;
      }
      if (p.ogate) {
        const float ss = warp_sum(o4.x * o4.x + o4.y * o4.y + o4.z * o4.z + o4.w * o4.w);
        const float rinv = rsqrtf(ss * (1.0f / kHeadDim) + p.eps);
        const uint2 zr = *reinterpret_cast<const uint2*>(p.z + base);
        const float4 gm = reinterpret_cast<const float4*>(p.gamma)[lane];
        uint2 packed;
        packed.x = (uint32_t)f32_to_bf16(o4.x * rinv * gm.x * silu(bf16_to_f32(zr.x & 0xffff))) |
                   ((uint32_t)f32_to_bf16(o4.y * rinv * gm.y * silu(bf16_to_f32(zr.x >> 16))) << 16);
        packed.y = (uint32_t)f32_to_bf16(o4.z * rinv * gm.z * silu(bf16_to_f32(zr.y & 0xffff))) |
                   ((uint32_t)f32_to_bf16(o4.w * rinv * gm.w * silu(bf16_to_f32(zr.y >> 16))) << 16);
        *reinterpret_cast<uint2*>(p.ogate + base) = packed;
      }
    }
    __syncthreads();
  }

  // ---- a6: state and history scatter
#pragma unroll
  for (int c = 0; c < kHeadDim; c += 4)
    *reinterpret_cast<float4*>(Srow_g + c) = make_float4(S[c], S[c + 1], S[c + 2], S[c + 3]);
#pragma unroll
  for (int u = 0; u < 3; ++u) {
    if (u < 2 && g != 0) continue;  // q/k history is written by the group's first CTA
    uint16_t* hp = p.conv_hist + ((size_t)slot * p.CH + gc[u]) * (kTaps - 1);
    hp[0] = hb[u][0];
    hp[1] = hb[u][1];
    hp[2] = hb[u][2];
  }
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream) {
  const size_t smem = sizeof(PfSmem);
  cudaError_t err = ensure_dynamic_smem(reinterpret_cast<const void*>(&prefill_kernel), smem);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.Hv, a.N, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = a.G;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, prefill_kernel, a);
}

}  // namespace gdn
