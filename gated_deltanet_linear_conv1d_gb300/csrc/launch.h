// launch.h - argument blocks and launchers shared between the C-ABI layer
// (api.cu) and the kernel files. Internal to libgdn.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
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
  int32_t* order;             // [N] scratch: requests, longest first (filled by launch_prefill)
  int32_t* tickets;           // [N][Hk] scratch: CTAs of (request, key head) finished (zeroed by launch_prefill)
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

struct QuantActArgs {
  const uint16_t* x;  // [T][K] bf16
  uint8_t* x8;        // [T][K] e4m3
  float* scale;       // scale of (token t, group g) at t * scale_t + g * scale_g
  long long scale_t, scale_g;
  int T, K;
};

struct QuantWeightArgs {
  const uint16_t* w;  // [N][K] bf16
  uint8_t* w8;        // [N][K] e4m3
  float* scale;       // scale of block (nb, kb) at nb * scale_n + kb * scale_k
  long long scale_n, scale_k;
  int N, K;
};

// Block-scaled FP8 GEMM: out[T][N] = dequant(x8) dequant(w8)^T (+ residual).
struct Fp8Operands {
  const uint8_t* x8;         // [T][K] e4m3
  const float* xs;           // [T][K/128]
  const uint8_t* w8;         // [N][K] e4m3
  const float* ws;           // [ceil(N/128)][K/128]
  const uint16_t* residual;  // [T][N] bf16 or nullptr
  uint16_t* out;             // [T][N] bf16
  int T, K, N;
};

struct Fp8GemmArgs {
  const float* xs;
  const float* ws;
  const uint16_t* residual;
  uint16_t* out;
  float* partial;  // stream-K partial tiles [grid][2][128 x 128 fp32], the wide kernel's split
                   // parts [tiles][split][128 x 256 fp32], or nullptr
  int* tile_cnt;   // stream-K tickets [tiles] (zero on entry, left zero), or nullptr
  int32_t* dev_err;
  int T, N, KB;
  int mt, nt;
  int stream_k;          // 1: equal K-block ranges per CTA; 0: whole tiles, strided
  int split;             // wide kernel: 1 persistent over whole tiles; > 1 parts of K per tile (clusters)
  long long tiles, total;  // output tiles; tiles x K blocks
};

// The driver's tensor-map encoder (resolved once).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// Sets cudaFuncAttributeMaxDynamicSharedMemorySize once per (function, device).
cudaError_t ensure_dynamic_smem(const void* fn, size_t bytes);

// Clusters of `cluster_size` CTAs of kernel `fn` (blocks of `threads` threads,
// `smem` bytes of dynamic shared memory, set with ensure_dynamic_smem first)
// that the current device holds at once; queried once per (function, device,
// cluster size, threads, shared memory); 0 if the query fails.
int resident_clusters(const void* fn, int threads, size_t smem, int cluster_size);

// Persistent state-streaming kernel (decode: P = 1, spec_slot NULL; verify: P >= 1).
bool stream_supported(int G, int P);
cudaError_t launch_stream(const StepArgs& a, cudaStream_t stream);
cudaError_t launch_commit(const CommitArgs& a, cudaStream_t stream);
cudaError_t launch_conv(const ConvArgs& a, cudaStream_t stream);
cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream);

// Largest request count the allocation-free prefill accepts: the size of its
// file-scope schedule array (one int32 per request, just under 256 KiB). It is
// also the largest count any prefill launch takes (requests go on gridDim.y).
constexpr int kStaticPrefillMaxSeqs = 65535;
constexpr int kStaticPrefillMaxTickets = 1 << 20;  // requests x key heads
// Device address of that array on the current device, looked up once per
// device with cudaGetSymbolAddress and cached.
cudaError_t static_prefill_order(int32_t** order, int32_t** tickets);

// bf16 GEMM with up to three outputs sharing one input:
//   out_s[T][N_s] = x[T][K] w_s[N_s][K]^T (+ residual_s[T][N_s]), fp32 accumulation,
// out_s bf16 (with an optional bf16 residual, in place allowed) or fp32.
struct GemmSegOperands {
  const uint16_t* w;         // [N][K] bf16
  void* out;                 // [T][N] bf16 or fp32
  const uint16_t* residual;  // [T][N] bf16 or nullptr (bf16 out only)
  int N;
  bool out_f32;
};
struct GemmOperands {
  const uint16_t* x;  // [T][K] bf16
  int T, K;
  GemmSegOperands seg[3];
  int nseg;
};
struct GemmSeg {
  uint16_t* out_bf16;
  float* out_f32;
  const uint16_t* residual;
  int N;
  int tiles;  // n-tiles of this output per m-tile
};
struct GemmArgs {
  GemmSeg seg[3];
  int nseg;
  int T, K, KB;
  int swap;         // 1: A = 128 weight rows, B = all T <= 256 tokens
  int nt_tok;       // swapped: MMA N = T rounded up to 16
  int mt;           // m-tiles (1 when swapped)
  int tiles_per_m;  // sum of the outputs' n-tiles
  int pairs;        // pair tiles: two A tiles sharing one B tile
  int group_n;      // not swapped: weight tiles per band of the tile order
  int split;        // pairs per cluster, each one split-th of K; 1: clusters of one pair, persistent
  int32_t* dev_err;
};
// Launches the bf16 GEMM (no scratch memory: a split K meets in a cluster's shared memory).
cudaError_t launch_gemm(const GemmOperands& o, int32_t* dev_err, cudaStream_t stream);
cudaError_t launch_gated_rmsnorm(const NormArgs& a, cudaStream_t stream);
cudaError_t launch_rmsnorm(const RmsArgs& a, cudaStream_t stream);
cudaError_t launch_quant_act(const QuantActArgs& a, cudaStream_t stream);
cudaError_t launch_quant_weight(const QuantWeightArgs& a, cudaStream_t stream);
// Workspace bytes for the split-K partial tiles of a [T][N] output with K inputs
// (0 when the shape is not split on this device).
size_t fp8_gemm_workspace_bytes(int T, int N, int K);
// Launches the block-scaled FP8 GEMM; without enough workspace it runs one K split.
cudaError_t launch_fp8_gemm(const Fp8Operands& o, void* workspace, size_t ws_bytes, int32_t* dev_err,
                            cudaStream_t stream);

}  // namespace gdn
