// step.cu - the state-streaming recurrent kernel behind gdn_decode_step
// (one token per request, state updated in place) and gdn_spec_verify (P
// positions per request, the state after every position kept in a checkpoint
// slot), and the commit kernel behind gdn_spec_commit.
//
// Math (page "Qwen3.8-27B: from model structure to vLLM inference data flow",
// section 01 GDN operator table; section 08: decay first, then predict from the
// decayed state):
//   c = SiLU(sum_i w_i x_{t-i});  q = q/|q|,  k = k/|k|
//   Sbar = a S;  e = v - Sbar k;  S' = Sbar + b e k^T;  o = S' q / sqrt(dk)
//   Ogate = o / sqrt(mean(o^2) + eps) * gamma * SiLU(z)
// One pass over S gives both S k and S q, because
//   o = S' q / sqrt(dk) = (a (S q) + b e (k . q)) / sqrt(dk),
// so the 64 KiB state of a (request, value head) is read once and written once.
//
// Work split: one CTA per (value head h, request n), 256 threads; the CTA owns
// the state tile S[slot][h] (128 x 128 fp32). A bulk (TMA) copy stages the tile
// in shared memory while the CTA computes the conv of its q, k and v channels.
// The G = Hv/Hk CTAs that share a key head form a thread-block cluster: each
// reads the old conv history of the shared q/k channels, and only after a
// cluster barrier does the group's first CTA overwrite that history.
#include <cooperative_groups.h>

#include "device.cuh"
#include "launch.h"

namespace cg = cooperative_groups;

namespace gdn {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kTile = kHeadDim * kHeadDim;       // fp32 elements of one head state
constexpr uint32_t kTileBytes = kTile * 4;       // 64 KiB
constexpr float kInvSqrtDk = 0.08838834764831845f;  // 1/sqrt(128)

struct SmemLayout {
  // offsets in floats from the start of dynamic shared memory
  int q, k, v, o, red, ab, total;
  __host__ __device__ explicit SmemLayout(int P) {
    q = kTile;
    k = q + P * kHeadDim;
    v = k + P * kHeadDim;
    o = v + P * kHeadDim;
    red = o + kHeadDim;      // [P][16]
    ab = red + P * 16;       // [P][3]: alpha, beta, k.q
    total = ab + P * 4;
  }
};

template <bool kSpec>
__global__ void __launch_bounds__(kThreads) step_kernel(const StepArgs p) {
  extern __shared__ __align__(128) float smem[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ int wait_ok;
  const SmemLayout L(p.P);
  float* S = smem;
  float* qs = smem + L.q;
  float* ks = smem + L.k;
  float* vs = smem + L.v;
  float* os = smem + L.o;
  float* red = smem + L.red;
  float* ab = smem + L.ab;

  const int h = blockIdx.x, n = blockIdx.y;
  const int g = h % p.G, j = h / p.G;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int P = p.P;

  // ---- a1: slot gather (all CTAs of a cluster share n, so exits are uniform)
  const int slot = p.slot_idx[n];
  if (slot < 0) return;  // padding
  bool bad = slot >= p.Rs;
  if (kSpec)
    for (int q = 0; q < P; ++q) {
      const int s = p.spec_slot[n * P + q];
      bad |= (s < 0) | (s >= p.Rs);
    }
  if (bad) {
    if (tid == 0 && g == 0) report(p.dev_err, GDN_DEVERR_SLOT);
    return;
  }
  float* Sg = p.state + ((size_t)slot * p.Hv + h) * kTile;

  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    const uint64_t pol = l2_policy_evict_first();
    mbar_arrive_expect_tx(&bar, kTileBytes);
#pragma unroll
    for (int c = 0; c < 4; ++c) bulk_g2s(S + c * (kTile / 4), Sg + c * (kTile / 4), kTileBytes / 4, &bar, pol);
  }
  if (tid < P) {
    const size_t row = (size_t)(n * P + tid) * p.Hv + h;
    ab[tid * 4 + 0] = p.alpha[row];
    ab[tid * 4 + 1] = p.beta[row];
  }

  // ---- a2: conv + SiLU of the CTA's 384 channels (q head j, k head j, v head h)
  // Threads 0..127 take channels tid and tid+256, threads 128..255 take tid.
  uint16_t nh[2][3];
  int gcs[2];
  bool own[2];
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int lc = tid + u * kThreads;
    own[u] = false;
    if (lc >= 3 * kHeadDim) continue;
    const int part = lc >> 7, d = lc & 127;
    const int gc = part == 0 ? j * kHeadDim + d
                 : part == 1 ? (p.Hk + j) * kHeadDim + d
                             : 2 * p.Hk * kHeadDim + h * kHeadDim + d;
    gcs[u] = gc;
    own[u] = (part == 2) || (g == 0);
    const float4 w = *reinterpret_cast<const float4*>(p.conv_w + (size_t)gc * kTaps);
    const uint16_t* hp = p.conv_hist + ((size_t)slot * p.CH + gc) * (kTaps - 1);
    uint16_t h0 = hp[0], h1 = hp[1], h2 = hp[2];
    float* dst = (part == 0 ? qs : part == 1 ? ks : vs) + d;
    for (int q = 0; q < P; ++q) {
      const uint16_t xb = p.qkv0[(size_t)(n * P + q) * p.CH + gc];
      float pre = w.x * bf16_to_f32(xb);
      pre = fmaf(w.y, bf16_to_f32(h2), pre);
      pre = fmaf(w.z, bf16_to_f32(h1), pre);
      pre = fmaf(w.w, bf16_to_f32(h0), pre);
      dst[q * kHeadDim] = silu(pre);
      h0 = h1;
      h1 = h2;
      h2 = xb;
      if (kSpec && own[u]) {
        uint16_t* ck = p.conv_hist + ((size_t)p.spec_slot[n * P + q] * p.CH + gc) * (kTaps - 1);
        ck[0] = h0;
        ck[1] = h1;
        ck[2] = h2;
      }
    }
    nh[u][0] = h0;
    nh[u][1] = h1;
    nh[u][2] = h2;
  }
  if (!kSpec) {
    // Every CTA of the key-head group has read the old history of the shared
    // q/k channels; the owners may now overwrite it (a6 scatter).
    cg::this_cluster().sync();
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if (!own[u]) continue;
      uint16_t* hp = p.conv_hist + ((size_t)slot * p.CH + gcs[u]) * (kTaps - 1);
      hp[0] = nh[u][0];
      hp[1] = nh[u][1];
      hp[2] = nh[u][2];
    }
  }
  __syncthreads();

  // ---- a3: L2 norm of q and k for each position (warps 0-3: q, warps 4-7: k)
  for (int q = 0; q < P; ++q) {
    const float x = (warp < 4 ? qs : ks)[q * kHeadDim + (warp & 3) * 32 + lane];
    const float ss = warp_sum(x * x);
    if (lane == 0) red[q * 16 + warp] = ss;
  }
  __syncthreads();
  for (int q = 0; q < P; ++q) {
    const float* r = red + q * 16 + (warp < 4 ? 0 : 4);
    const float inv = rsqrtf(((r[0] + r[1]) + (r[2] + r[3])) + 1e-12f);
    (warp < 4 ? qs : ks)[q * kHeadDim + (warp & 3) * 32 + lane] *= inv;
  }
  __syncthreads();
  if (warp < 4)
    for (int q = 0; q < P; ++q) {
      const int i = warp * 32 + lane;
      const float kq = warp_sum(ks[q * kHeadDim + i] * qs[q * kHeadDim + i]);
      if (lane == 0) red[q * 16 + 8 + warp] = kq;
    }
  float zpre = 0.f;  // prefetch z for the gate of position 0
  if (tid < kHeadDim && p.ogate) zpre = bf16_to_f32(p.z[((size_t)(n * P) * p.Hv + h) * kHeadDim + tid]);
  __syncthreads();
  if (tid < P) {
    const float* r = red + tid * 16 + 8;
    ab[tid * 4 + 2] = (r[0] + r[1]) + (r[2] + r[3]);
  }

  // ---- wait for the state tile (bounded; a timeout is reported, never hangs)
  if (tid == 0) wait_ok = mbar_wait_bounded(&bar, 0) ? 1 : 0;
  __syncthreads();
  if (!wait_ok) {
    if (tid == 0) {
      report(p.dev_err, GDN_DEVERR_TIMEOUT);
      mbar_wait_bounded(&bar, 0);  // give the copy in flight a second bounded chance to land
    }
    return;
  }
  mbar_wait_bounded(&bar, 0);  // already complete: makes the async-proxy writes visible to this thread

  const uint64_t wpol = l2_policy_evict_first();
  for (int q = 0; q < P; ++q) {
    const float a = ab[q * 4 + 0], b = ab[q * 4 + 1], kq = ab[q * 4 + 2];
    const float4 k4 = reinterpret_cast<const float4*>(ks + q * kHeadDim)[lane];
    const float4 q4 = reinterpret_cast<const float4*>(qs + q * kHeadDim)[lane];
    const float* vq = vs + q * kHeadDim;
    float* Sout = kSpec ? p.state + ((size_t)p.spec_slot[n * P + q] * p.Hv + h) * kTile : Sg;
    const bool carry = q + 1 < P;

    // ---- a4: one gated-delta-rule step; warp w owns rows 16w .. 16w+15
#pragma unroll 4
    for (int r = 0; r < kHeadDim / kWarps; ++r) {
      const int i = warp * (kHeadDim / kWarps) + r;
      float4 s = reinterpret_cast<const float4*>(S + i * kHeadDim)[lane];
      float pk = s.x * k4.x;
      pk = fmaf(s.y, k4.y, pk);
      pk = fmaf(s.z, k4.z, pk);
      pk = fmaf(s.w, k4.w, pk);
      float pq = s.x * q4.x;
      pq = fmaf(s.y, q4.y, pq);
      pq = fmaf(s.z, q4.z, pq);
      pq = fmaf(s.w, q4.w, pq);
      pk = warp_sum(pk);  // (S k)_i
      pq = warp_sum(pq);  // (S q)_i
      const float e = vq[i] - a * pk;  // v - Sbar k
      const float be = b * e;
      float4 ns;
      ns.x = fmaf(be, k4.x, a * s.x);
      ns.y = fmaf(be, k4.y, a * s.y);
      ns.z = fmaf(be, k4.z, a * s.z);
      ns.w = fmaf(be, k4.w, a * s.w);
      // a6: state scatter (in place for decode, checkpoint slot for verify)
      st_global_v4_hint(Sout + i * kHeadDim + lane * 4, ns, wpol);
      if (carry) reinterpret_cast<float4*>(S + i * kHeadDim)[lane] = ns;
      if (lane == 0) os[i] = fmaf(be, kq, a * pq) * kInvSqrtDk;
    }
    __syncthreads();

    // ---- a5: gated RMSNorm of the head row
    float oi = 0.f;
    if (tid < kHeadDim) {
      oi = os[tid];
      const float ss = warp_sum(oi * oi);
      if (lane == 0) red[q * 16 + 12 + warp] = ss;
    }
    __syncthreads();
    if (tid < kHeadDim) {
      const float* r = red + q * 16 + 12;
      const float ms = ((r[0] + r[1]) + (r[2] + r[3])) * (1.0f / kHeadDim);
      const float rinv = rsqrtf(ms + p.eps);
      const size_t row = ((size_t)(n * P + q) * p.Hv + h) * kHeadDim + tid;
      if (p.o) p.o[row] = f32_to_bf16(oi);
      if (p.ogate) {
        const float zz = q == 0 ? zpre : bf16_to_f32(p.z[row]);
        p.ogate[row] = f32_to_bf16(oi * rinv * p.gamma[tid] * silu(zz));
      }
    }
  }
}

// Commit: copy (or repoint to) the checkpoint of the accepted position.
// grid (Hv + 1, N): block x < Hv copies head x of the state, block Hv copies
// the conv history.
__global__ void __launch_bounds__(256) commit_kernel(const CommitArgs p) {
  const int n = blockIdx.y, x = blockIdx.x;
  const int slot = p.slot_idx[n];
  if (slot < 0) return;
  const int a = p.accepted[n];
  if (a < 0 || a >= p.P) {
    if (threadIdx.x == 0 && x == 0) report(p.dev_err, GDN_DEVERR_ACCEPTED);
    return;
  }
  const int src = p.spec_slot[n * p.P + a];
  if (slot >= p.Rs || src < 0 || src >= p.Rs) {
    if (threadIdx.x == 0 && x == 0) report(p.dev_err, GDN_DEVERR_SLOT);
    return;
  }
  if (p.mode == GDN_COMMIT_REPOINT) {
    if (x == 0 && threadIdx.x == 0) p.slot_idx[n] = src;
    return;
  }
  if (x < p.Hv) {
    // 64 KiB: 16 float4 per thread, loaded four at a time before they are stored
    const float4* s = reinterpret_cast<const float4*>(p.state + ((size_t)src * p.Hv + x) * kTile);
    float4* d = reinterpret_cast<float4*>(p.state + ((size_t)slot * p.Hv + x) * kTile);
    for (int i0 = threadIdx.x; i0 < kTile / 4; i0 += 4 * blockDim.x) {
      float4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = i0 + u * blockDim.x;
        if (i < kTile / 4) v[u] = s[i];
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = i0 + u * blockDim.x;
        if (i < kTile / 4) d[i] = v[u];
      }
    }
  } else {
    const size_t nb = (size_t)p.CH * (kTaps - 1);  // uint16 per slot
    const uint16_t* s = p.conv_hist + (size_t)src * nb;
    uint16_t* d = p.conv_hist + (size_t)slot * nb;
    if (((reinterpret_cast<uintptr_t>(s) | reinterpret_cast<uintptr_t>(d)) & 15) == 0 && nb % 8 == 0) {
      const uint4* s4 = reinterpret_cast<const uint4*>(s);
      uint4* d4 = reinterpret_cast<uint4*>(d);
      for (size_t i = threadIdx.x; i < nb / 8; i += blockDim.x) d4[i] = s4[i];
    } else {
      for (size_t i = threadIdx.x; i < nb; i += blockDim.x) d[i] = s[i];
    }
  }
}

}  // namespace

size_t step_smem_bytes(int P) { return (size_t)SmemLayout(P).total * sizeof(float); }

cudaError_t launch_step(const StepArgs& a, bool spec, cudaStream_t stream) {
  const size_t smem = step_smem_bytes(a.P);
  const void* fn = spec ? reinterpret_cast<const void*>(&step_kernel<true>)
                        : reinterpret_cast<const void*>(&step_kernel<false>);
  cudaError_t err = ensure_dynamic_smem(fn, smem);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.Hv, a.N, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = spec ? 1 : a.G;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (spec) return cudaLaunchKernelEx(&cfg, step_kernel<true>, a);
  return cudaLaunchKernelEx(&cfg, step_kernel<false>, a);
}

cudaError_t launch_commit(const CommitArgs& a, cudaStream_t stream) {
  dim3 grid(a.mode == GDN_COMMIT_REPOINT ? 1 : a.Hv + 1, a.N, 1);
  commit_kernel<<<grid, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace gdn
