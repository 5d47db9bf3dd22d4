// commit.cu - the commit kernel behind gdn_spec_commit: the state and conv
// history after a request's accepted position become its live state ("Qwen3.8
// MTP" page, section 5, accept / reject: the longest accepted prefix is kept and
// the state follows it). Copy mode moves 3 MiB of state and the history per
// request; repoint mode only rewrites the slot index.
#include "device.cuh"
#include "launch.h"

namespace gdn {

namespace {

constexpr int kTile = kHeadDim * kHeadDim;  // fp32 elements of one head state (64 KiB)

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

cudaError_t launch_commit(const CommitArgs& a, cudaStream_t stream) {
  dim3 grid(a.mode == GDN_COMMIT_REPOINT ? 1 : a.Hv + 1, a.N, 1);
  commit_kernel<<<grid, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace gdn
