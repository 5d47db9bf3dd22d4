// api.cu - the extern "C" entry points of libgdn: argument validation on the
// host, then one launch on the caller's stream. Declarations and the full
// contract of every entry point are in include/gdn.h.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <mutex>
#include <unordered_map>

#include "device.cuh"
#include "gdn.h"
#include "launch.h"

namespace gdn {

cudaError_t ensure_dynamic_smem(const void* fn, size_t bytes) {
  // (function, device) -> the largest dynamic shared-memory size set so far
  static std::mutex mu;
  static std::unordered_map<const void*, std::unordered_map<int, size_t>> set_to;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  std::lock_guard<std::mutex> lock(mu);
  size_t& cur = set_to[fn][dev];
  if (bytes <= cur) return cudaSuccess;
  err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (err != cudaSuccess) return err;
  cur = bytes;
  return cudaSuccess;
}

int resident_clusters(const void* fn, int threads, size_t smem, int cluster_size) {
  struct Key {
    const void* fn;
    int dev, threads, csize;
    size_t smem;
    bool operator==(const Key& o) const {
      return fn == o.fn && dev == o.dev && threads == o.threads && csize == o.csize && smem == o.smem;
    }
  };
  struct Hash {
    size_t operator()(const Key& k) const {
      return std::hash<const void*>()(k.fn) ^ ((size_t)k.dev << 40) ^ ((size_t)k.threads << 20) ^
             ((size_t)k.csize << 12) ^ k.smem;
    }
  };
  static std::mutex mu;
  static std::unordered_map<Key, int, Hash> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  const Key key{fn, dev, threads, cluster_size, smem};
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)cluster_size, 1, 1);
  cfg.blockDim = dim3((unsigned)threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cluster_size;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    n = 0;
  }
  cache.emplace(key, n);
  return n;
}

namespace {

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Geometry check shared by every call that takes gdn_dims.
gdn_status check_dims(const gdn_dims* d) {
  if (!d) return GDN_ERR_INVALID_ARG;
  if (d->num_k_heads <= 0 || d->num_v_heads <= 0 || d->head_k_dim <= 0 || d->head_v_dim <= 0 ||
      d->conv_kernel <= 0 || d->num_slots <= 0)
    return GDN_ERR_INVALID_ARG;
  if (d->head_k_dim != kHeadDim || d->head_v_dim != kHeadDim || d->conv_kernel != kTaps)
    return GDN_ERR_UNSUPPORTED;
  if (d->num_v_heads % d->num_k_heads != 0) return GDN_ERR_UNSUPPORTED;
  if (d->num_v_heads / d->num_k_heads > kMaxGroup) return GDN_ERR_UNSUPPORTED;
  if (d->num_v_heads > 65535) return GDN_ERR_UNSUPPORTED;
  return GDN_OK;
}

int channels(const gdn_dims* d) {
  return 2 * d->num_k_heads * d->head_k_dim + d->num_v_heads * d->head_v_dim;
}

bool eps_ok(float eps) { return std::isfinite(eps) && eps >= 0.f; }

gdn_status from_cuda(cudaError_t e) { return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA; }

}  // namespace
}  // namespace gdn

using namespace gdn;

extern "C" {

size_t gdn_state_bytes(const gdn_dims* d) {
  if (!d || d->num_v_heads <= 0 || d->head_v_dim <= 0 || d->head_k_dim <= 0) return 0;
  return (size_t)d->num_v_heads * d->head_v_dim * d->head_k_dim * sizeof(float);
}

size_t gdn_conv_hist_bytes(const gdn_dims* d) {
  if (!d || d->num_k_heads <= 0 || d->num_v_heads <= 0 || d->head_k_dim <= 0 || d->head_v_dim <= 0 ||
      d->conv_kernel <= 1)
    return 0;
  return (size_t)channels(d) * (d->conv_kernel - 1) * sizeof(uint16_t);
}

// Prefill scratch: the schedule (requests, longest first) and one ticket per (request, key head).
size_t prefill_order_bytes(int32_t num_seqs) { return ((size_t)num_seqs * sizeof(int32_t) + 255) / 256 * 256; }

size_t gdn_prefill_workspace_bytes(const gdn_dims* d, int32_t num_seqs, int32_t num_tokens) {
  (void)num_tokens;
  if (check_dims(d) != GDN_OK || num_seqs <= 0) return 0;
  return prefill_order_bytes(num_seqs) +
         ((size_t)num_seqs * d->num_k_heads * sizeof(int32_t) + 255) / 256 * 256;
}

const char* gdn_status_string(gdn_status s) {
  switch (s) {
    case GDN_OK: return "GDN_OK";
    case GDN_ERR_INVALID_ARG: return "GDN_ERR_INVALID_ARG: invalid argument";
    case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED: unsupported geometry";
    case GDN_ERR_CUDA: return "GDN_ERR_CUDA: CUDA runtime or launch failure";
    case GDN_ERR_DEVICE_CHECK: return "GDN_ERR_DEVICE_CHECK: the device flagged an invalid index";
    case GDN_ERR_TIMEOUT: return "GDN_ERR_TIMEOUT: a bounded device wait ran out";
  }
  return "unknown gdn_status";
}

gdn_status gdn_read_device_error(int32_t* dev_err, int32_t* host_err, int32_t reset, void* stream) {
  if (!dev_err || !host_err) return GDN_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, dev_err, sizeof v, cudaMemcpyDeviceToHost, s) != cudaSuccess) return GDN_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return GDN_ERR_CUDA;
  if (reset && v != 0) {
    if (cudaMemsetAsync(dev_err, 0, sizeof(int32_t), s) != cudaSuccess) return GDN_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return GDN_ERR_CUDA;
  }
  *host_err = v;
  if (v == 0) return GDN_OK;
  return (v & GDN_DEVERR_TIMEOUT) ? GDN_ERR_TIMEOUT : GDN_ERR_DEVICE_CHECK;
}

gdn_status gdn_conv_update(const gdn_dims* d, const uint16_t* x, const float* conv_w, uint16_t* conv_hist,
                           const int32_t* qsl, const int32_t* slot_idx, const uint8_t* has_init,
                           int32_t num_seqs, int32_t num_tokens, uint16_t* y, int32_t* dev_err,
                           void* stream) {
  gdn_status st = check_dims(d);
  if (st != GDN_OK) return st;
  if (num_seqs < 0 || num_tokens < 0 || num_seqs > 65535) return GDN_ERR_INVALID_ARG;
  if (num_seqs == 0) return num_tokens == 0 ? GDN_OK : GDN_ERR_INVALID_ARG;
  if (!conv_w || !conv_hist || !qsl || !slot_idx) return GDN_ERR_INVALID_ARG;
  if (num_tokens > 0 && (!x || !y)) return GDN_ERR_INVALID_ARG;
  if (!aligned(conv_w, 16) || !aligned(conv_hist, 4)) return GDN_ERR_INVALID_ARG;
  if (num_tokens > 0 && (!aligned(x, 8) || !aligned(y, 8))) return GDN_ERR_INVALID_ARG;
  ConvArgs a{x, conv_w, conv_hist, qsl, slot_idx, has_init, y, dev_err, channels(d), d->num_slots, num_seqs,
             num_tokens};
  return from_cuda(launch_conv(a, static_cast<cudaStream_t>(stream)));
}

gdn_status gdn_decode_step(const gdn_dims* d, const uint16_t* qkv0, const float* conv_w, uint16_t* conv_hist,
                           float* state, const int32_t* slot_idx, const float* alpha, const float* beta,
                           const uint16_t* z, const float* gamma, float eps, uint16_t* o, uint16_t* ogate,
                           int32_t num_seqs, int32_t* dev_err, void* stream) {
  gdn_status st = check_dims(d);
  if (st != GDN_OK) return st;
  if (num_seqs < 0 || num_seqs > 65535) return GDN_ERR_INVALID_ARG;
  if (num_seqs == 0) return GDN_OK;
  if (!qkv0 || !conv_w || !conv_hist || !state || !slot_idx || !alpha || !beta) return GDN_ERR_INVALID_ARG;
  if (!o && !ogate) return GDN_ERR_INVALID_ARG;
  if (ogate && (!z || !gamma)) return GDN_ERR_INVALID_ARG;
  if (!eps_ok(eps)) return GDN_ERR_INVALID_ARG;
  if (!aligned(state, 16) || !aligned(conv_w, 16) || !aligned(qkv0, 16) || !aligned(conv_hist, 16) ||
      (ogate && !aligned(z, 16)))
    return GDN_ERR_INVALID_ARG;
  StepArgs a{qkv0, conv_w, conv_hist, state, slot_idx, nullptr, alpha, beta, z, gamma, eps, o, ogate, dev_err,
             d->num_k_heads, d->num_v_heads, d->num_v_heads / d->num_k_heads, channels(d), d->num_slots,
             num_seqs, 1};
  return from_cuda(launch_stream(a, static_cast<cudaStream_t>(stream)));
}

gdn_status gdn_spec_verify(const gdn_dims* d, const uint16_t* qkv0, const float* conv_w, uint16_t* conv_hist,
                           float* state, const int32_t* slot_idx, const int32_t* spec_slot_idx,
                           const float* alpha, const float* beta, const uint16_t* z, const float* gamma,
                           float eps, uint16_t* o, uint16_t* ogate, int32_t num_seqs, int32_t num_pos,
                           int32_t* dev_err, void* stream) {
  gdn_status st = check_dims(d);
  if (st != GDN_OK) return st;
  if (num_seqs < 0 || num_seqs > 65535 || num_pos < 1 || num_pos > 8) return GDN_ERR_INVALID_ARG;
  if (num_seqs == 0) return GDN_OK;
  if (!qkv0 || !conv_w || !conv_hist || !state || !slot_idx || !spec_slot_idx || !alpha || !beta)
    return GDN_ERR_INVALID_ARG;
  if (!o && !ogate) return GDN_ERR_INVALID_ARG;
  if (ogate && (!z || !gamma)) return GDN_ERR_INVALID_ARG;
  if (!eps_ok(eps)) return GDN_ERR_INVALID_ARG;
  if (!aligned(state, 16) || !aligned(conv_w, 16) || !aligned(qkv0, 16) || !aligned(conv_hist, 16) ||
      (ogate && !aligned(z, 16)))
    return GDN_ERR_INVALID_ARG;
  StepArgs a{qkv0, conv_w, conv_hist, state, slot_idx, spec_slot_idx, alpha, beta, z, gamma, eps, o, ogate,
             dev_err, d->num_k_heads, d->num_v_heads, d->num_v_heads / d->num_k_heads, channels(d),
             d->num_slots, num_seqs, num_pos};
  if (!stream_supported(a.G, a.P)) return GDN_ERR_UNSUPPORTED;  // never for the supported geometry
  return from_cuda(launch_stream(a, static_cast<cudaStream_t>(stream)));
}

gdn_status gdn_spec_commit(const gdn_dims* d, const int32_t* accepted, const int32_t* spec_slot_idx,
                           int32_t* slot_idx, float* state, uint16_t* conv_hist, int32_t num_seqs,
                           int32_t num_pos, int32_t mode, int32_t* dev_err, void* stream) {
  gdn_status st = check_dims(d);
  if (st != GDN_OK) return st;
  if (num_seqs < 0 || num_seqs > 65535 || num_pos < 1 || num_pos > 8) return GDN_ERR_INVALID_ARG;
  if (mode != GDN_COMMIT_COPY && mode != GDN_COMMIT_REPOINT) return GDN_ERR_INVALID_ARG;
  if (num_seqs == 0) return GDN_OK;
  if (!accepted || !spec_slot_idx || !slot_idx) return GDN_ERR_INVALID_ARG;
  if (mode == GDN_COMMIT_COPY && (!state || !conv_hist || !aligned(state, 16))) return GDN_ERR_INVALID_ARG;
  CommitArgs a{accepted, spec_slot_idx, slot_idx, state, conv_hist, dev_err, d->num_v_heads, channels(d),
               d->num_slots, num_seqs, num_pos, mode};
  return from_cuda(launch_commit(a, static_cast<cudaStream_t>(stream)));
}

gdn_status gdn_chunk_prefill(const gdn_dims* d, const uint16_t* qkv0, const float* conv_w, uint16_t* conv_hist,
                             float* state, const int32_t* qsl, const int32_t* slot_idx, const uint8_t* has_init,
                             const float* alpha, const float* beta, const uint16_t* z, const float* gamma,
                             float eps, uint16_t* o, uint16_t* ogate, int32_t num_seqs, int32_t num_tokens,
                             void* workspace, size_t workspace_bytes, int32_t* dev_err, void* stream) {
  gdn_status st = check_dims(d);
  if (st != GDN_OK) return st;
  if (num_seqs < 0 || num_tokens < 0 || num_seqs > 65535) return GDN_ERR_INVALID_ARG;
  if (num_seqs == 0) return num_tokens == 0 ? GDN_OK : GDN_ERR_INVALID_ARG;
  if (!conv_w || !conv_hist || !state || !qsl || !slot_idx) return GDN_ERR_INVALID_ARG;
  if (num_tokens == 0) return GDN_OK;  // every request is empty: nothing is read or written
  if (!qkv0 || !alpha || !beta) return GDN_ERR_INVALID_ARG;
  if (!o && !ogate) return GDN_ERR_INVALID_ARG;
  if (ogate && (!z || !gamma)) return GDN_ERR_INVALID_ARG;
  if (!eps_ok(eps)) return GDN_ERR_INVALID_ARG;
  if (!aligned(state, 16) || !aligned(conv_w, 16)) return GDN_ERR_INVALID_ARG;
  if (num_tokens > 0 && !aligned(qkv0, 16)) return GDN_ERR_INVALID_ARG;
  if ((o && !aligned(o, 8)) || (ogate && (!aligned(ogate, 16) || !aligned(z, 16) || !aligned(gamma, 16))))
    return GDN_ERR_INVALID_ARG;
  const size_t need = gdn_prefill_workspace_bytes(d, num_seqs, num_tokens);
  if (workspace_bytes < need || (need > 0 && (!workspace || !aligned(workspace, 256))))
    return GDN_ERR_INVALID_ARG;
  PrefillArgs a{qkv0, conv_w, conv_hist, state, qsl, slot_idx, has_init, alpha, beta, z, gamma, eps, o, ogate,
                dev_err, d->num_k_heads, d->num_v_heads, d->num_v_heads / d->num_k_heads, channels(d),
                d->num_slots, num_seqs, num_tokens, static_cast<int32_t*>(workspace),
                reinterpret_cast<int32_t*>(static_cast<unsigned char*>(workspace) + prefill_order_bytes(num_seqs)),
                nullptr, nullptr, 0, 0};
  return from_cuda(launch_prefill(a, static_cast<cudaStream_t>(stream)));
}

gdn_status gdn_chunk_prefill_align(const gdn_dims* d, const uint16_t* qkv0, const float* conv_w, uint16_t* conv_hist,
                                   float* state, const int32_t* qsl, const int32_t* slot_idx, const uint8_t* has_init,
                                   const float* alpha, const float* beta, const uint16_t* z, const float* gamma,
                                   float eps, uint16_t* o, uint16_t* ogate, int32_t num_seqs, int32_t num_tokens,
                                   const int32_t* prefix_len, int32_t block_tokens, const int32_t* snap_slot,
                                   int32_t max_snaps, void* workspace, size_t workspace_bytes, int32_t* dev_err,
                                   void* stream) {
  gdn_status st = check_dims(d);
  if (st != GDN_OK) return st;
  if (num_seqs < 0 || num_tokens < 0 || num_seqs > 65535) return GDN_ERR_INVALID_ARG;
  if (block_tokens <= 0 || block_tokens % 64 != 0 || max_snaps < 0 || (max_snaps > 0 && !snap_slot))
    return GDN_ERR_INVALID_ARG;
  if (num_seqs == 0) return num_tokens == 0 ? GDN_OK : GDN_ERR_INVALID_ARG;
  if (!conv_w || !conv_hist || !state || !qsl || !slot_idx) return GDN_ERR_INVALID_ARG;
  if (num_tokens == 0) return GDN_OK;  // every request is empty: nothing is read or written
  if (!qkv0 || !alpha || !beta) return GDN_ERR_INVALID_ARG;
  if (!o && !ogate) return GDN_ERR_INVALID_ARG;
  if (ogate && (!z || !gamma)) return GDN_ERR_INVALID_ARG;
  if (!eps_ok(eps)) return GDN_ERR_INVALID_ARG;
  if (!aligned(state, 16) || !aligned(conv_w, 16)) return GDN_ERR_INVALID_ARG;
  if (num_tokens > 0 && !aligned(qkv0, 16)) return GDN_ERR_INVALID_ARG;
  if ((o && !aligned(o, 8)) || (ogate && (!aligned(ogate, 16) || !aligned(z, 16) || !aligned(gamma, 16))))
    return GDN_ERR_INVALID_ARG;
  const size_t need = gdn_prefill_workspace_bytes(d, num_seqs, num_tokens);
  if (workspace_bytes < need || (need > 0 && (!workspace || !aligned(workspace, 256))))
    return GDN_ERR_INVALID_ARG;
  PrefillArgs a{qkv0, conv_w, conv_hist, state, qsl, slot_idx, has_init, alpha, beta, z, gamma, eps, o, ogate,
                dev_err, d->num_k_heads, d->num_v_heads, d->num_v_heads / d->num_k_heads, channels(d),
                d->num_slots, num_seqs, num_tokens, static_cast<int32_t*>(workspace),
                reinterpret_cast<int32_t*>(static_cast<unsigned char*>(workspace) + prefill_order_bytes(num_seqs)),
                prefix_len, max_snaps > 0 ? snap_slot : nullptr, block_tokens, max_snaps};
  return from_cuda(launch_prefill(a, static_cast<cudaStream_t>(stream)));
}

gdn_status gdn_chunk_prefill_noalloc(const gdn_dims* d, const uint16_t* qkv0, const float* conv_w,
                                     uint16_t* conv_hist, float* state, const int32_t* qsl,
                                     const int32_t* slot_idx, const uint8_t* has_init, const float* alpha,
                                     const float* beta, const uint16_t* z, const float* gamma, float eps,
                                     uint16_t* o, uint16_t* ogate, int32_t num_seqs, int32_t num_tokens,
                                     int32_t* dev_err, void* stream) {
  gdn_status st = check_dims(d);
  if (st != GDN_OK) return st;
  if (num_seqs < 0 || num_tokens < 0) return GDN_ERR_INVALID_ARG;
  if (num_seqs > gdn::kStaticPrefillMaxSeqs ||
      (long long)num_seqs * d->num_k_heads > gdn::kStaticPrefillMaxTickets)
    return GDN_ERR_INVALID_ARG;  // beyond the fixed schedule arrays
  if (num_seqs == 0) return num_tokens == 0 ? GDN_OK : GDN_ERR_INVALID_ARG;
  if (!conv_w || !conv_hist || !state || !qsl || !slot_idx) return GDN_ERR_INVALID_ARG;
  if (num_tokens == 0) return GDN_OK;  // every request is empty: nothing is read or written
  if (!qkv0 || !alpha || !beta) return GDN_ERR_INVALID_ARG;
  if (!o && !ogate) return GDN_ERR_INVALID_ARG;
  if (ogate && (!z || !gamma)) return GDN_ERR_INVALID_ARG;
  if (!eps_ok(eps)) return GDN_ERR_INVALID_ARG;
  if (!aligned(state, 16) || !aligned(conv_w, 16)) return GDN_ERR_INVALID_ARG;
  if (num_tokens > 0 && !aligned(qkv0, 16)) return GDN_ERR_INVALID_ARG;
  if ((o && !aligned(o, 8)) || (ogate && (!aligned(ogate, 16) || !aligned(z, 16) || !aligned(gamma, 16))))
    return GDN_ERR_INVALID_ARG;
  int32_t* order = nullptr;
  int32_t* tickets = nullptr;
  if (gdn::static_prefill_order(&order, &tickets) != cudaSuccess) return GDN_ERR_CUDA;
  PrefillArgs a{qkv0, conv_w, conv_hist, state, qsl, slot_idx, has_init, alpha, beta, z, gamma, eps, o, ogate,
                dev_err, d->num_k_heads, d->num_v_heads, d->num_v_heads / d->num_k_heads, channels(d),
                d->num_slots, num_seqs, num_tokens, order, tickets, nullptr, nullptr, 0, 0};
  return from_cuda(launch_prefill(a, static_cast<cudaStream_t>(stream)));
}

gdn_status gdn_out_proj(const uint16_t* ogate, const uint16_t* w, const uint16_t* residual, uint16_t* out,
                        int32_t num_tokens, int32_t in_features, int32_t out_features, int32_t* dev_err,
                        void* stream) {
  if (num_tokens < 0 || in_features <= 0 || out_features <= 0) return GDN_ERR_INVALID_ARG;
  if (in_features % 8 != 0 || out_features % 8 != 0) return GDN_ERR_UNSUPPORTED;
  if (num_tokens == 0) return GDN_OK;
  if (!ogate || !w || !out) return GDN_ERR_INVALID_ARG;
  if (!aligned(ogate, 16) || !aligned(w, 16) || !aligned(out, 16) || (residual && !aligned(residual, 16)))
    return GDN_ERR_INVALID_ARG;
  GemmOperands o{};
  o.x = ogate;
  o.T = num_tokens;
  o.K = in_features;
  o.nseg = 1;
  o.seg[0] = GemmSegOperands{w, out, residual, out_features, false};
  return from_cuda(launch_gemm(o, dev_err, static_cast<cudaStream_t>(stream)));
}

gdn_status gdn_in_proj(const gdn_dims* d, const uint16_t* hidden, int32_t hidden_size, const uint16_t* w_qkv,
                       const uint16_t* w_z, const uint16_t* w_ab, uint16_t* qkv0, uint16_t* z, float* ab,
                       int32_t num_tokens, int32_t* dev_err, void* stream) {
  gdn_status st = check_dims(d);
  if (st != GDN_OK) return st;
  if (num_tokens < 0 || hidden_size <= 0) return GDN_ERR_INVALID_ARG;
  const int CH = channels(d), NZ = d->num_v_heads * d->head_v_dim, NAB = 2 * d->num_v_heads;
  if (hidden_size % 8 != 0 || NAB % 4 != 0) return GDN_ERR_UNSUPPORTED;
  if (num_tokens == 0) return GDN_OK;
  if (!hidden || !w_qkv || !qkv0 || !w_z || !z || (!w_ab != !ab)) return GDN_ERR_INVALID_ARG;
  if (!aligned(hidden, 16) || !aligned(w_qkv, 16) || !aligned(qkv0, 16) || !aligned(w_z, 16) || !aligned(z, 16) ||
      (w_ab && (!aligned(w_ab, 16) || !aligned(ab, 16))))
    return GDN_ERR_INVALID_ARG;
  GemmOperands o{};
  o.x = hidden;
  o.T = num_tokens;
  o.K = hidden_size;
  o.seg[0] = GemmSegOperands{w_qkv, qkv0, nullptr, CH, false};
  o.seg[1] = GemmSegOperands{w_z, z, nullptr, NZ, false};
  o.nseg = 2;
  if (w_ab) {
    o.seg[2] = GemmSegOperands{w_ab, ab, nullptr, NAB, true};
    o.nseg = 3;
  }
  return from_cuda(launch_gemm(o, dev_err, static_cast<cudaStream_t>(stream)));
}

gdn_status gdn_gated_rmsnorm(const uint16_t* o, const uint16_t* z, const float* gamma, float eps, uint16_t* out,
                             int32_t num_tokens, int32_t num_heads, int32_t head_dim, void* stream) {
  if (num_tokens < 0 || num_heads <= 0 || head_dim <= 0) return GDN_ERR_INVALID_ARG;
  if (head_dim % 4 != 0 || head_dim > 1024) return GDN_ERR_UNSUPPORTED;
  if (!eps_ok(eps)) return GDN_ERR_INVALID_ARG;
  const long long rows = (long long)num_tokens * num_heads;
  if (rows == 0) return GDN_OK;
  if (rows > (1ll << 31) - 1) return GDN_ERR_INVALID_ARG;
  if (!o || !z || !gamma || !out) return GDN_ERR_INVALID_ARG;
  if (!aligned(o, 8) || !aligned(z, 8) || !aligned(out, 8) || !aligned(gamma, 16)) return GDN_ERR_INVALID_ARG;
  NormArgs a{o, z, gamma, out, eps, (int)rows, head_dim};
  return from_cuda(launch_gated_rmsnorm(a, static_cast<cudaStream_t>(stream)));
}

gdn_status gdn_rmsnorm(const uint16_t* x, uint16_t* residual, const float* gamma, float eps, uint16_t* out,
                       int32_t num_tokens, int32_t hidden_size, void* stream) {
  if (num_tokens < 0 || hidden_size <= 0) return GDN_ERR_INVALID_ARG;
  if (hidden_size % 8 != 0 || hidden_size > 8192) return GDN_ERR_UNSUPPORTED;
  if (!eps_ok(eps)) return GDN_ERR_INVALID_ARG;
  if (num_tokens == 0) return GDN_OK;
  if (!x || !gamma || !out) return GDN_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(gamma, 16) || !aligned(out, 16) || (residual && !aligned(residual, 16)))
    return GDN_ERR_INVALID_ARG;
  RmsArgs a{x, residual, gamma, out, eps, (int)num_tokens, (int)hidden_size};
  return from_cuda(launch_rmsnorm(a, static_cast<cudaStream_t>(stream)));
}

gdn_status gdn_fp8_quant_act(const uint16_t* x, uint8_t* x8, float* x_scale, int32_t num_tokens, int32_t k,
                             void* stream) {
  if (num_tokens < 0 || k <= 0) return GDN_ERR_INVALID_ARG;
  if (k % 128 != 0) return GDN_ERR_UNSUPPORTED;
  if (num_tokens == 0) return GDN_OK;
  if (!x || !x8 || !x_scale) return GDN_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(x8, 16) || !aligned(x_scale, 16)) return GDN_ERR_INVALID_ARG;
  QuantActArgs a{x, x8, x_scale, k / 128, 1, (int)num_tokens, (int)k};  // scales [T][K/128]
  return from_cuda(launch_quant_act(a, static_cast<cudaStream_t>(stream)));
}

gdn_status gdn_fp8_quant_weight(const uint16_t* w, uint8_t* w8, float* w_scale, int32_t n, int32_t k, void* stream) {
  if (n < 0 || k <= 0) return GDN_ERR_INVALID_ARG;
  if (k % 128 != 0) return GDN_ERR_UNSUPPORTED;
  if (n == 0) return GDN_OK;
  if (!w || !w8 || !w_scale) return GDN_ERR_INVALID_ARG;
  if (!aligned(w, 16) || !aligned(w8, 16) || !aligned(w_scale, 16)) return GDN_ERR_INVALID_ARG;
  QuantWeightArgs a{w, w8, w_scale, k / 128, 1, (int)n, (int)k};  // scales [ceil(N/128)][K/128]
  return from_cuda(launch_quant_weight(a, static_cast<cudaStream_t>(stream)));
}

size_t gdn_fp8_linear_workspace_bytes(int32_t num_tokens, int32_t k, int32_t n) {
  if (num_tokens <= 0 || n <= 0 || k <= 0 || k % 128 != 0) return 0;
  return fp8_gemm_workspace_bytes(num_tokens, n, k);
}

gdn_status gdn_fp8_linear(const uint8_t* x8, const float* x_scale, const uint8_t* w8, const float* w_scale,
                          const uint16_t* residual, uint16_t* out, int32_t num_tokens, int32_t k, int32_t n,
                          void* workspace, size_t workspace_bytes, int32_t* dev_err, void* stream) {
  if (num_tokens < 0 || k <= 0 || n <= 0) return GDN_ERR_INVALID_ARG;
  if (k % 128 != 0 || n % 16 != 0) return GDN_ERR_UNSUPPORTED;
  if (num_tokens == 0) return GDN_OK;
  if (!x8 || !x_scale || !w8 || !w_scale || !out) return GDN_ERR_INVALID_ARG;
  if (!aligned(x8, 16) || !aligned(x_scale, 16) || !aligned(w8, 16) || !aligned(w_scale, 16) || !aligned(out, 16) ||
      (residual && !aligned(residual, 16)))
    return GDN_ERR_INVALID_ARG;
  if (workspace_bytes > 0 && (!workspace || !aligned(workspace, 256))) return GDN_ERR_INVALID_ARG;
  Fp8Operands o{x8, x_scale, w8, w_scale, residual, out, (int)num_tokens, (int)k, (int)n};
  return from_cuda(launch_fp8_gemm(o, workspace_bytes ? workspace : nullptr, workspace_bytes, dev_err,
                                   static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
