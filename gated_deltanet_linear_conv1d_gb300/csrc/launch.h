// launch.h - argument blocks and launchers shared between the C-ABI layer
// (api.cu) and the kernel files. Internal to libgdn.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace gdn {

struct StepArgs {
  const uint16_t* qkv0;       // [N*P][CH]
  const float* conv_w;        // [CH][4]
  uint16_t* conv_hist;        // [Rs][CH][3]
  float* state;               // [Rs][Hv][128][128]
  const int32_t* slot_idx;    // [N]
  const int32_t* spec_slot;   // [N][P] (verify) or nullptr (decode)
  const float* alpha;         // [N*P][Hv]
  const float* beta;          // [N*P][Hv]
  const uint16_t* z;          // [N*P][Hv][128]
  const float* gamma;         // [128]
  float eps;
  uint16_t* o;                // [N*P][Hv][128] or nullptr
  uint16_t* ogate;            // [N*P][Hv*128] or nullptr
  int32_t* dev_err;
  int Hk, Hv, G, CH, Rs, N, P;
};

struct CommitArgs {
  const int32_t* accepted;    // [N]
  const int32_t* spec_slot;   // [N][P]
  int32_t* slot_idx;          // [N]
  float* state;
  uint16_t* conv_hist;
  int32_t* dev_err;
  int Hv, CH, Rs, N, P, mode;
};

struct ConvArgs {
  const uint16_t* x;          // [T][CH]
  const float* conv_w;        // [CH][4]
  uint16_t* conv_hist;        // [Rs][CH][3]
  const int32_t* qsl;         // [N+1]
  const int32_t* slot_idx;    // [N]
  const uint8_t* has_init;    // [N] or nullptr
  uint16_t* y;                // [T][CH]
  int32_t* dev_err;
  int CH, Rs, N, T;
};

struct PrefillArgs {
  const uint16_t* qkv0;       // [T][CH]
  const float* conv_w;
  uint16_t* conv_hist;
  float* state;
  const int32_t* qsl;         // [N+1]
  const int32_t* slot_idx;    // [N]
  const uint8_t* has_init;    // [N] or nullptr
  const float* alpha;         // [T][Hv]
  const float* beta;
  const uint16_t* z;          // [T][Hv][128] or nullptr
  const float* gamma;
  float eps;
  uint16_t* o;                // or nullptr
  uint16_t* ogate;            // or nullptr
  int32_t* dev_err;
  int Hk, Hv, G, CH, Rs, N, T;
  int32_t* order;             // [N] scratch: requests, longest first (filled by launch_prefill), or nullptr
  // align mode (all nullptr / 0 otherwise): pos0[n] tokens already in request n's slot; chunks end on
  // absolute multiples of 64, and after every absolute multiple of snap_block the state and history go
  // to snap_slot[n][j] (j-th such boundary of this call; -1 skips)
  const int32_t* pos0;
  const int32_t* snap_slot;   // [N][max_snaps]
  int snap_block, max_snaps;
};

struct NormArgs {
  const uint16_t* o;
  const uint16_t* z;
  const float* gamma;
  uint16_t* out;
  float eps;
  int rows;  // T * H
  int D;
};

struct RmsArgs {
  const uint16_t* x;
  uint16_t* residual;  // NULL: no residual add
  const float* gamma;
  uint16_t* out;
  float eps;
  int rows;
  int D;
};

// Sets cudaFuncAttributeMaxDynamicSharedMemorySize once per (function, device).
cudaError_t ensure_dynamic_smem(const void* fn, size_t bytes);

size_t step_smem_bytes(int P);
cudaError_t launch_step(const StepArgs& a, bool spec, cudaStream_t stream);
// Persistent state-streaming kernel (decode: P = 1, spec_slot NULL; verify: P >= 1).
bool stream_supported(int G, int P);
cudaError_t launch_stream(const StepArgs& a, cudaStream_t stream);
cudaError_t launch_commit(const CommitArgs& a, cudaStream_t stream);
cudaError_t launch_conv(const ConvArgs& a, cudaStream_t stream);
cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream);

// Largest request count the allocation-free prefill accepts: the size of its
// file-scope schedule array (one int32 per request, 256 KiB).
constexpr int kStaticPrefillMaxSeqs = 65536;
// Device address of that array on the current device, looked up once per
// device with cudaGetSymbolAddress and cached.
cudaError_t static_prefill_order(int32_t** out);

// out[T][N] = x[T][K] w[N][K]^T (+ residual[T][N]) through cuBLASLt, bf16
// operands, fp32 accumulation, out (and residual) bf16 or fp32; sets
// *unsupported when the library offers no algorithm for the shape.
cudaError_t launch_linear(const uint16_t* x, const uint16_t* w, const void* residual, void* out, bool out_f32, int T,
                          int K, int N, void* workspace, size_t ws_bytes, cudaStream_t stream, bool* unsupported);
cudaError_t launch_gated_rmsnorm(const NormArgs& a, cudaStream_t stream);
cudaError_t launch_rmsnorm(const RmsArgs& a, cudaStream_t stream);

}  // namespace gdn
