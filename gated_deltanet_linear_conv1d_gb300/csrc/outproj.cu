// outproj.cu - the two projections around the mixer core (page "Qwen3.8-27B:
// from model structure to vLLM inference data flow", section 01 GDN operator
// table): gdn_in_proj, the rows in front of the conv ([T,5120] -> QKV0
// [T,10240], Z [T,6144] and the a, b projections [T,48] each), and
// gdn_out_proj, the Wo row ([T,6144] -> [T,5120]) with the residual add. The
// conv is fused into the mixer kernels that read QKV0 and the gated RMSNorm into
// the ones that write Ogate, so what is left on either side is a plain GEMM:
// bf16 operands, fp32 accumulation, the residual folded into the epilogue
// (D = A B + C), issued through cuBLASLt.
//
// Row-major out[T][N] = ogate[T][K] W^T (+ residual[T][N]) with W [N][K] (the
// nn.Linear layout) is, column-major, out^T (N x T) = op(W) (N x K) ogate^T (K x T)
// where W viewed column-major is K x N and op = transpose.
#include <cublasLt.h>

#include <map>
#include <mutex>
#include <tuple>

#include "launch.h"

namespace gdn {

namespace {

struct Plan {
  cublasLtMatmulDesc_t op = nullptr;
  cublasLtMatrixLayout_t a = nullptr, b = nullptr, c = nullptr;
  cublasLtMatmulAlgo_t algo{};
};

struct LtCache {
  std::mutex mu;
  std::map<int, cublasLtHandle_t> handles;                                  // per device
  std::map<std::tuple<int, int, int, int, size_t, int>, Plan> plans;        // (device, T, K, N, workspace, D type)
};

LtCache& cache() {
  static LtCache* c = new LtCache();  // lives for the process
  return *c;
}

// The device's library handle (created on first use; caller holds lc.mu).
cublasStatus_t handle_locked(LtCache& lc, int dev, cublasLtHandle_t* h_out) {
  auto hit = lc.handles.find(dev);
  if (hit == lc.handles.end()) {
    cublasLtHandle_t h = nullptr;
    const cublasStatus_t st = cublasLtCreate(&h);
    if (st != CUBLAS_STATUS_SUCCESS) return st;
    hit = lc.handles.emplace(dev, h).first;
  }
  *h_out = hit->second;
  return CUBLAS_STATUS_SUCCESS;
}

// Builds (once per shape) the descriptors and the heuristic's first algorithm.
cublasStatus_t get_plan(int dev, int T, int K, int N, size_t ws_bytes, cudaDataType_t cd_type, cublasLtHandle_t* h_out,
                        Plan* out) {
  LtCache& lc = cache();
  std::lock_guard<std::mutex> lock(lc.mu);
  cublasStatus_t st = handle_locked(lc, dev, h_out);
  if (st != CUBLAS_STATUS_SUCCESS) return st;
  const auto key = std::make_tuple(dev, T, K, N, ws_bytes, (int)cd_type);
  auto pit = lc.plans.find(key);
  if (pit != lc.plans.end()) {
    *out = pit->second;
    return CUBLAS_STATUS_SUCCESS;
  }
  Plan p;
  cublasLtMatmulPreference_t pref = nullptr;
  auto fail = [&](cublasStatus_t s) {
    if (pref) cublasLtMatmulPreferenceDestroy(pref);
    if (p.a) cublasLtMatrixLayoutDestroy(p.a);
    if (p.b) cublasLtMatrixLayoutDestroy(p.b);
    if (p.c) cublasLtMatrixLayoutDestroy(p.c);
    if (p.op) cublasLtMatmulDescDestroy(p.op);
    return s;
  };
  if ((st = cublasLtMatmulDescCreate(&p.op, CUBLAS_COMPUTE_32F, CUDA_R_32F)) != CUBLAS_STATUS_SUCCESS) return fail(st);
  const cublasOperation_t ta = CUBLAS_OP_T, tb = CUBLAS_OP_N;
  if ((st = cublasLtMatmulDescSetAttribute(p.op, CUBLASLT_MATMUL_DESC_TRANSA, &ta, sizeof ta)) != CUBLAS_STATUS_SUCCESS ||
      (st = cublasLtMatmulDescSetAttribute(p.op, CUBLASLT_MATMUL_DESC_TRANSB, &tb, sizeof tb)) != CUBLAS_STATUS_SUCCESS)
    return fail(st);
  if ((st = cublasLtMatrixLayoutCreate(&p.a, CUDA_R_16BF, K, N, K)) != CUBLAS_STATUS_SUCCESS ||
      (st = cublasLtMatrixLayoutCreate(&p.b, CUDA_R_16BF, K, T, K)) != CUBLAS_STATUS_SUCCESS ||
      (st = cublasLtMatrixLayoutCreate(&p.c, cd_type, N, T, N)) != CUBLAS_STATUS_SUCCESS)
    return fail(st);
  if ((st = cublasLtMatmulPreferenceCreate(&pref)) != CUBLAS_STATUS_SUCCESS) return fail(st);
  if ((st = cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES, &ws_bytes,
                                                 sizeof ws_bytes)) != CUBLAS_STATUS_SUCCESS)
    return fail(st);
  cublasLtMatmulHeuristicResult_t res{};
  int found = 0;
  st = cublasLtMatmulAlgoGetHeuristic(*h_out, p.op, p.a, p.b, p.c, p.c, pref, 1, &res, &found);
  if (st != CUBLAS_STATUS_SUCCESS) return fail(st);
  if (found < 1) return fail(CUBLAS_STATUS_NOT_SUPPORTED);
  cublasLtMatmulPreferenceDestroy(pref);
  p.algo = res.algo;
  lc.plans.emplace(key, p);
  *out = p;
  return CUBLAS_STATUS_SUCCESS;
}

}  // namespace

cudaError_t launch_linear(const uint16_t* x, const uint16_t* w, const void* residual, void* out, bool out_f32, int T,
                          int K, int N, void* workspace, size_t ws_bytes, cudaStream_t stream, bool* unsupported) {
  *unsupported = false;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  cublasLtHandle_t h = nullptr;
  Plan p;
  cublasStatus_t st = get_plan(dev, T, K, N, ws_bytes, out_f32 ? CUDA_R_32F : CUDA_R_16BF, &h, &p);
  if (st == CUBLAS_STATUS_NOT_SUPPORTED) {
    *unsupported = true;
    return cudaErrorNotSupported;
  }
  if (st != CUBLAS_STATUS_SUCCESS) return cudaErrorUnknown;
  const float alpha = 1.f, beta = residual ? 1.f : 0.f;
  st = cublasLtMatmul(h, p.op, &alpha, w, p.a, x, p.b, &beta, residual ? residual : out, p.c, out, p.c, &p.algo,
                      workspace, ws_bytes, stream);
  return st == CUBLAS_STATUS_SUCCESS ? cudaSuccess : cudaErrorUnknown;
}

}  // namespace gdn
