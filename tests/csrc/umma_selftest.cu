// umma_selftest.cu - a single-CTA tcgen05 GEMM used by the tests to check the
// tensor-core operand layouts and descriptors of umma.cuh against numpy:
// D[M][N] = sum_k A[M][K] * B[N][K], operands converted to bf16 or tf32 and
// placed in shared memory K-major or MN-major, fp32 accumulation in tensor
// memory. Shared-memory buffers are padded well beyond the tiles so that every
// address a descriptor can reach stays inside the CTA's allocation.
#include <cuda_runtime.h>

#include "umma.cuh"

using namespace gdn;

namespace {

struct Args {
  const float* A;  // [M][K]
  const float* B;  // [N][K]
  float* D;        // [M][N]
  int* err;
  int M, N, K, kind, a_mn, b_mn;
  int b_cols;      // columns allocated per row of the B tile (>= its used extent): B may be a sub-block
};

constexpr int kBOffset = 64 * 1024;   // B tile offset; A tile at 0
constexpr int kSmemBytes = 224 * 1024; // every address either reading of LBO/SBO can reach fits in here

template <uint32_t kKind>
__device__ void issue(const Args& p, uint32_t tmem, uint32_t sa, uint32_t sb) {
  constexpr int es = kKind == umma::kTF32 ? 4 : 2;
  constexpr int kstep = kKind == umma::kTF32 ? 8 : 16;
  const int a_row_bytes = (p.a_mn ? p.M : p.K) * es;
  const int b_row_bytes = p.b_cols * es;
  const uint32_t b0 = p.b_mn ? (uint32_t)((p.b_cols - p.N) * es / 16) * 128 : 0;  // sub-block start
  const uint32_t id = umma::idesc(kKind, p.a_mn, p.b_mn, p.M, p.N);
  for (int kk = 0; kk < p.K / kstep; ++kk) {
    const uint32_t aoff = p.a_mn ? kk * (kstep / 8) * (a_row_bytes * 8) : kk * (kstep * es / 16) * 128;
    const uint32_t boff = p.b_mn ? kk * (kstep / 8) * (b_row_bytes * 8) : kk * (kstep * es / 16) * 128;
    umma::mma<kKind>(tmem, umma::smem_desc(sa + aoff, a_row_bytes, p.a_mn),
                     umma::smem_desc(sb + b0 + boff, b_row_bytes, p.b_mn), id, kk > 0);
  }
}

__global__ void __launch_bounds__(128) selftest_kernel(const Args p) {
  extern __shared__ __align__(1024) unsigned char smem[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tbase;
  unsigned char* sA = smem;
  unsigned char* sB = smem + kBOffset;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int es = p.kind == umma::kTF32 ? 4 : 2;
  const int a_row_bytes = (p.a_mn ? p.M : p.K) * es;
  const int b_row_bytes = p.b_cols * es;
  for (int i = tid; i < p.M * p.K; i += blockDim.x) {
    const int m = i / p.K, k = i % p.K;
    const uint32_t off = p.a_mn ? umma::tile_off(k, m * es, a_row_bytes) : umma::tile_off(m, k * es, a_row_bytes);
    if (es == 4) *reinterpret_cast<float*>(sA + off) = umma::to_tf32(p.A[i]);
    else *reinterpret_cast<uint16_t*>(sA + off) = f32_to_bf16(p.A[i]);
  }
  // A sub-block B sits in the last N of the tile's b_cols columns (MN-major only).
  const int b_col0 = p.b_mn ? p.b_cols - p.N : 0;
  for (int i = tid; i < p.N * p.K; i += blockDim.x) {
    const int n = i / p.K, k = i % p.K;
    const uint32_t off = p.b_mn ? umma::tile_off(k, (b_col0 + n) * es, b_row_bytes)
                                : umma::tile_off(n, k * es, b_row_bytes);
    if (es == 4) *reinterpret_cast<float*>(sB + off) = umma::to_tf32(p.B[i]);
    else *reinterpret_cast<uint16_t*>(sB + off) = f32_to_bf16(p.B[i]);
  }
  umma::fence_proxy_async_smem();
  if (warp == 0) umma::tmem_alloc(&tbase, 256);
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tmem = tbase;
  if (tid == 0) {
    if (p.kind == umma::kTF32) issue<umma::kTF32>(p, tmem, smem_u32(sA), smem_u32(sB));
    else issue<umma::kBF16>(p, tmem, smem_u32(sA), smem_u32(sB));
    umma::commit(&bar);
  }
  const int ok = __syncthreads_and(mbar_wait_bounded(&bar, 0) ? 1 : 0);
  umma::fence_after_sync();
  if (ok) {
    for (int c0 = 0; c0 < p.N; c0 += 32) {
      float v[32];
      umma::ld32(umma::taddr(tmem, 32 * warp, c0), v);
      for (int i = 0; i < 32; ++i) p.D[(size_t)(32 * warp + lane) * p.N + c0 + i] = v[i];
    }
  } else if (tid == 0) {
    atomicOr(p.err, GDN_DEVERR_TIMEOUT);
  }
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  if (warp == 0) umma::tmem_dealloc(tmem, 256);
}

// The same GEMM with A read from tensor memory (columns 128.. of the
// allocation): tf32 as one 32-bit column per element (a_raw: the unrounded
// fp32 value, to see how the tensor core reads it), bf16 as one column per
// pair of elements, the lower-indexed one in the low half. B is K-major in
// shared memory.
__global__ void __launch_bounds__(128) selftest_ts_kernel(const Args p, int a_raw) {
  extern __shared__ __align__(1024) unsigned char smem[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tbase;
  unsigned char* sB = smem + kBOffset;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool tf32 = p.kind == umma::kTF32;
  const int es = tf32 ? 4 : 2;
  const int b_row_bytes = p.K * es;
  for (int i = tid; i < p.N * p.K; i += blockDim.x) {
    const int n = i / p.K, k = i % p.K;
    const uint32_t off = umma::tile_off(n, k * es, b_row_bytes);
    if (tf32) *reinterpret_cast<float*>(sB + off) = umma::to_tf32(p.B[i]);
    else *reinterpret_cast<uint16_t*>(sB + off) = f32_to_bf16(p.B[i]);
  }
  umma::fence_proxy_async_smem();
  if (warp == 0) umma::tmem_alloc(&tbase, 256);
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tmem = tbase;
  // row m = 32 warp + lane of A into its lane, 8 columns at a time
  const int m = 32 * warp + lane;
  const int acols = tf32 ? p.K : p.K / 2;
  for (int c0 = 0; c0 < acols; c0 += 8) {
    float v[8];
    for (int e = 0; e < 8; ++e) {
      const int c = c0 + e;
      if (tf32) {
        const float x = p.A[(size_t)m * p.K + c];
        v[e] = a_raw ? x : umma::to_tf32(x);
      } else {
        const uint32_t lo = f32_to_bf16(p.A[(size_t)m * p.K + 2 * c]);
        const uint32_t hi = f32_to_bf16(p.A[(size_t)m * p.K + 2 * c + 1]);
        v[e] = __uint_as_float(lo | (hi << 16));
      }
    }
    umma::st8(umma::taddr(tmem, 32 * warp, 128 + c0), v);
  }
  umma::wait_st();
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  if (tid == 0) {
    const uint32_t id = umma::idesc(p.kind, false, false, p.M, p.N);
    const int kstep = tf32 ? 8 : 16;
    for (int kk = 0; kk < p.K / kstep; ++kk) {
      const uint32_t acol = 128 + kk * 8;  // 8 columns: 8 tf32 or 16 bf16 elements
      const uint64_t bdesc = umma::smem_desc(smem_u32(sB) + kk * (kstep * es / 16) * 128, b_row_bytes, false);
      if (tf32) umma::mma_ts<umma::kKindTF32>(tmem, tmem + acol, bdesc, id, kk > 0);
      else umma::mma_ts<umma::kKindF16>(tmem, tmem + acol, bdesc, id, kk > 0);
    }
    umma::commit(&bar);
  }
  const int ok = __syncthreads_and(mbar_wait_bounded(&bar, 0) ? 1 : 0);
  umma::fence_after_sync();
  if (ok) {
    for (int c0 = 0; c0 < p.N; c0 += 32) {
      float v[32];
      umma::ld32(umma::taddr(tmem, 32 * warp, c0), v);
      for (int i = 0; i < 32; ++i) p.D[(size_t)(32 * warp + lane) * p.N + c0 + i] = v[i];
    }
  } else if (tid == 0) {
    atomicOr(p.err, GDN_DEVERR_TIMEOUT);
  }
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  if (warp == 0) umma::tmem_dealloc(tmem, 256);
}

// A wait that can never succeed (nothing arrives on the barrier): the bounded
// wait gives up after its time limit and the kernel reports a timeout in the
// device error word, leaving the context usable.
__global__ void bounded_wait_kernel(int32_t* dev_err) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (!mbar_wait_bounded(&bar, 0) && threadIdx.x == 0) report(dev_err, GDN_DEVERR_TIMEOUT);
}

}  // namespace

extern "C" int bounded_wait_selftest(int32_t* dev_err, void* stream) {
  bounded_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(dev_err);
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

extern "C" int umma_selftest(const float* A, const float* B, float* D, int* err, int M, int N, int K, int kind,
                             int a_mn, int b_mn, int b_cols, void* stream) {
  // Shapes whose descriptor reach was checked against kSmemBytes: M = 128,
  // N in {64, 128}, K in {64, 128}; MN-major A only for bf16; B row length
  // b_cols = its own extent, or 128 for an MN-major bf16 B of N = 64.
  if (M != 128 || (N != 64 && N != 128) || (K != 64 && K != 128)) return 1;
  if (kind != umma::kBF16 && kind != umma::kTF32) return 1;
  if (kind == umma::kTF32 && (a_mn || (K == 128 && b_mn && N == 128))) return 1;
  const int b_extent = b_mn ? N : K;
  if (b_cols != b_extent && !(kind == umma::kBF16 && b_mn && N == 64 && b_cols == 128)) return 1;
  const size_t smem = kSmemBytes;
  if (cudaFuncSetAttribute(selftest_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return 3;
  Args a{A, B, D, err, M, N, K, kind, a_mn, b_mn, b_cols};
  selftest_kernel<<<1, 128, smem, static_cast<cudaStream_t>(stream)>>>(a);
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

// A from tensor memory: M = 128, N in {64, 128}, K in {64, 128}, B K-major.
extern "C" int umma_selftest_ts(const float* A, const float* B, float* D, int* err, int N, int K, int kind,
                                int a_raw, void* stream) {
  if ((N != 64 && N != 128) || (K != 64 && K != 128)) return 1;
  if (kind != umma::kBF16 && kind != umma::kTF32) return 1;
  if (a_raw && kind != umma::kTF32) return 1;
  const size_t smem = kSmemBytes;
  if (cudaFuncSetAttribute(selftest_ts_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return 3;
  Args a{A, B, D, err, 128, N, K, kind, 0, 0, K};
  selftest_ts_kernel<<<1, 128, smem, static_cast<cudaStream_t>(stream)>>>(a, a_raw);
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}
