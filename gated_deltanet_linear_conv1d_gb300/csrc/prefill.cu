// prefill.cu - gdn_chunk_prefill on the tensor cores: varlen prefill through
// the whole mixer core (page "Qwen3.8-27B: from model structure to vLLM
// inference data flow", section 01 GDN operator table), with the gated delta
// rule evaluated in chunks of 64 tokens in its WY / UT form.
//
// Chunked form (derived from the recurrence row S = a S + b (v - a S k) k^T;
// the page only says that the block recurrence uses the associative structure
// to run in parallel). For a chunk starting from state S0 with, per token r,
// g_r = sum_{i<=r} ln a_i and Gamma[r][i] = exp(g_r - g_i):
//   (I + A) E = diag(b) V - diag(b e^g) K S0^T,  A[r][i] = b_r Gamma[r][i] k_r.k_i (i < r)
//   E^T = (V^T - S0 Kg^T) Tb^T,   Kg = diag(e^g) K,  Tb = (I + A)^-1 diag(b)
//   O^T = diag_cols(e^g) S0 Q^T + E^T P^T,  P[r][i] = Gamma[r][i] q_r.k_i (i <= r)
//   S_C = e^{g_C} S0 + E^T diag(Gamma[C][.]) K
// with q, k unit-normalised; the per-token norms are folded into the
// products' readouts, so the tensor cores take the raw conv outputs.
//
// One CTA per (value head h, request n), 256 threads; the G CTAs of a key
// head form a cluster (only to order the in-place conv-history update). The
// fp32 state lives in tensor memory (128 lanes x 128 columns) for the whole
// request. Per chunk:
//   conv + SiLU (CUDA cores, thread = channel)  -> raw q, k (bf16, channel-major),
//       k e^g (bf16), k (tf32, channel-major), v (fp32), per-token |q|, |k|
//   [K;Q] K^T                 tcgen05 bf16  M=128 N=64  K=128  (operands MN-major)
//   S0 -> bf16 operand, S *= e^{g_C} in tensor memory
//   X = S0 Kg^T, Z = S0 Q^T   tcgen05 bf16  M=128 N=64  K=128
//   A, P from K K^T, Q K^T;  T = (I + A)^-1 on CUDA cores (blocked by 16)
//   Y = V^T - X  -> tf32;  E^T = Y Tb^T   tcgen05 tf32 M=128 N=64 K=64
//   S += (E^T diag(Gamma_C / |k|)) K     tcgen05 tf32 M=128 N=128 K=64 (accumulate)
//   O' = E^T P^T                tcgen05 bf16 M=128 N=64 K=64
//   o = e^g Z / |q| + O',  gated RMSNorm, bf16 out.
// The two products that feed the carried state (E and the state update) take
// tf32 operands; the others take bf16 (measured against the fp64 oracle:
// state error ~6e-4, output error ~3e-3 relative L2).
#include <cooperative_groups.h>
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>
#include <type_traits>

#include "device.cuh"
#include "launch.h"
#include "umma.cuh"

namespace cg = cooperative_groups;

namespace gdn {

namespace {

constexpr int kThreads = 256;
constexpr int kC = 64;  // chunk length
constexpr float kInvSqrtDk = 0.08838834764831845f;

// Shared-memory regions (byte offsets, 1024-aligned).
constexpr int kKQ = 0;                  // bf16 [128 dk][128 t]: k tokens 0-63, q tokens 64-127 (MN-major)
constexpr int kKG = kKQ + 32768;        // bf16 [128 dk][64 t]: k e^g (MN-major B)      | later E bf16 [128 dv][64 t]
constexpr int kKT = kKG + 16384;        // tf32 [128 dk][64 t]: raw k (K-major B)
constexpr int kS0 = kKT + 32768;        // bf16 [128 dv][128 dk]: S0 (K-major A)       | later Y, E' tf32 [128][64]
// Scratch: raw QKV0 rows of a chunk [3 parts][64 t][128] bf16 (bulk-copied, read by
// the conv), later the inverse's A [64][68], T [64][68] and block products [3][16][20];
// then the raw rows of the next chunk. Its tail holds the chunk's z rows [64][128]
// bf16, overwritten in place by Ogate before they are bulk-stored.
constexpr int kSCR = kS0 + 32768;
constexpr int kXS = kSCR;               // raw QKV0 rows, 49152 B
constexpr int kLd = 68;                 // row stride (floats) of A and T: 16-byte aligned rows
constexpr int kMsLd = 20, kMsBlk = 16 * kMsLd;  // M blocks [3][16][20]
constexpr int kAM = kSCR;               // fp32 [64][kLd]
constexpr int kTS = kAM + 64 * kLd * 4;  // fp32 [64][kLd]
constexpr int kMS = kTS + 64 * kLd * 4;  // fp32 [3][16][kMsLd]
static_assert(kMS + 3 * kMsBlk * 4 <= kSCR + 49152, "inverse scratch overlaps the z rows");
constexpr int kZS = kSCR + 49152;       // bf16 [64][128]: z rows, then Ogate rows
constexpr int kTB = kSCR + 65536;       // tf32 [64 r][64 i]: T diag(b) (K-major B)
constexpr int kPB = kTB + 16384;        // bf16 [64 r][64 i]: P (K-major B)
constexpr int kSmall = kPB + 8192;      // small per-chunk vectors
constexpr int kSmallFloats = 64 * 8 + 8 * 64 + 4 * 64 + 64;
constexpr int kBars = kSmall + kSmallFloats * 4;
constexpr int kSmemBytes = kBars + 128;

// Tensor-memory columns (v, fp32 channel-major, lives in the last 64).
constexpr uint32_t kTS_S = 0, kT_D1 = 128, kT_X = 192, kT_Z = 256, kT_E = 320, kT_O = 384, kT_V = 448,
                   kTmemCols = 512;

__device__ __forceinline__ float to_tf32(float x) { return umma::to_tf32(x); }

// Sums v[0..7] over the 32 lanes of a warp, 8 values at once (9 shuffles).
// Returns the total of value index tok8(lane) in every lane.
__device__ __forceinline__ float reduce8(float (&v)[8], int lane) {
  {
    const bool hi = lane & 16;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float send = hi ? v[i] : v[i + 4], keep = hi ? v[i + 4] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
  }
  {
    const bool hi = lane & 8;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const float send = hi ? v[i] : v[i + 2], keep = hi ? v[i + 2] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
  }
  {
    const bool hi = lane & 4;
    const float send = hi ? v[0] : v[1], keep = hi ? v[1] : v[0];
    v[0] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
  }
  v[0] += __shfl_xor_sync(0xffffffffu, v[0], 2);
  v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
  return v[0];
}
__device__ __forceinline__ int tok8(int lane) {
  return ((lane >> 2) & 1) | (((lane >> 3) & 1) << 1) | (((lane >> 4) & 1) << 2);
}

// 2^x via the hardware approximation (ex2.approx); its error is far below the
// bf16 / tf32 rounding that every use of it is followed by.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two floats to a bf16 pair (round to nearest even), a in the low half.
__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(b), "f"(a));
  return d;
}

// SiLU(x) = x / (1 + e^-x) with e^-x = 2^(-x log2 e), on the flush-to-zero
// ex2 and reciprocal approximations. Large negative x gives -0.
__device__ __forceinline__ float silu_ftz(float x) {
  float e, r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(x * -1.4426950408889634f));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.f + e));
  return x * r;
}

// Waits for an MMA-completion phase; the verdict is uniform over the CTA.
__device__ __forceinline__ bool wait_mma(uint64_t* bar, uint32_t parity) {
  const int ok = __syncthreads_and(mbar_wait_bounded(bar, parity) ? 1 : 0);
  umma::fence_after_sync();
  return ok != 0;
}

// Syncs the CTA after shared-memory operand writes and tensor-memory stores,
// so that the MMAs issued next see them.
__device__ __forceinline__ void sync_for_mma() {
  umma::fence_proxy_async_smem();
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
}

// Tensor maps: tmx over QKV0 [T][CH] (box 64 tokens x 128 channels); tmz, tmo over
// z and Ogate [T][Hv][128] (box 64 tokens x 1 head x 128).
__global__ void __launch_bounds__(kThreads, 1) prefill_tc_kernel(const PrefillArgs p,
                                                                  const __grid_constant__ CUtensorMap tmx,
                                                                  const __grid_constant__ CUtensorMap tmz,
                                                                  const __grid_constant__ CUtensorMap tmo) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const int h = blockIdx.x, n = blockIdx.y;
  const int g = h % p.G, j = h / p.G;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3, half = warp >> 2;
  const int row = 32 * quarter + lane;  // tensor-memory lane read by this thread

  // ---- request checks (uniform over the cluster: same request)
  const int slot = p.slot_idx[n];
  if (slot < 0) return;
  const int t0 = p.qsl[n], t1 = p.qsl[n + 1];
  if (t0 < 0 || t1 < t0 || t1 > p.T || (n == 0 && t0 != 0) || (n == p.N - 1 && t1 != p.T)) {
    if (tid == 0 && g == 0) report(p.dev_err, GDN_DEVERR_OFFSETS);
    return;
  }
  if (slot >= p.Rs) {
    if (tid == 0 && g == 0) report(p.dev_err, GDN_DEVERR_SLOT);
    return;
  }
  if (t1 == t0) return;  // no tokens: the slot is left untouched
  const bool init = p.has_init ? p.has_init[n] != 0 : true;

  uint16_t* KQ = reinterpret_cast<uint16_t*>(smem + kKQ);
  unsigned char* KGb = smem + kKG;
  unsigned char* KTb = smem + kKT;
  const uint16_t* XS = reinterpret_cast<const uint16_t*>(smem + kXS);
  uint16_t* ZS = reinterpret_cast<uint16_t*>(smem + kZS);
  unsigned char* S0b = smem + kS0;
  float* AM = reinterpret_cast<float*>(smem + kAM);
  float* TS = reinterpret_cast<float*>(smem + kTS);
  unsigned char* TBb = smem + kTB;
  unsigned char* PBb = smem + kPB;
  float* small = reinterpret_cast<float*>(smem + kSmall);
  float* gv = small;             // [64] g / ln 2 (cumulative log2 of alpha)
  float* egv = gv + 64;          // [64] e^g
  float* glv = egv + 64;         // [64] e^{g_C - g_t} (0 past the chunk end)
  float* bv = glv + 64;          // [64] beta
  float* iqv = bv + 64;          // [64] 1/|q|
  float* ikv = iqv + 64;         // [64] 1/|k|
  float* rinv = ikv + 64;        // [64] gate 1/rms
  float* scan = rinv + 64;       // [64] scan scratch
  float* npart = scan + 64;      // [8][64] norm partials (warps 0-3: q, 4-7: k)
  float* rpart = npart + 8 * 64; // [4][64] gate partials
  float* MS = reinterpret_cast<float*>(smem + kMS);
  // MMA completions 0: [K;Q]K^T  1: X,Z  2: E  3: S, O';  copies 4: raw QKV0 rows  5: z rows
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 6);
  const bool want_gate = p.ogate != nullptr;
  // Thread 0: TMA the raw QKV0 rows (q_j, k_j, v_h segments, 64 tokens each, from
  // token tcs) into the scratch area. Rows past the request are masked by the
  // conv; rows past T arrive as zeros.
  auto issue_x = [&](int tcs) {
    mbar_arrive_expect_tx(&bars[4], (uint32_t)(3 * kC * kHeadDim * 2));
    tma_load_2d(smem + kXS + 0 * kC * 256, &tmx, j * kHeadDim, tcs, &bars[4]);
    tma_load_2d(smem + kXS + 1 * kC * 256, &tmx, (p.Hk + j) * kHeadDim, tcs, &bars[4]);
    tma_load_2d(smem + kXS + 2 * kC * 256, &tmx, (2 * p.Hk + h) * kHeadDim, tcs, &bars[4]);
  };

  // ---- conv channels of this thread: q (tid < 128) and v (tid < 128), or k
  const bool qv = tid < 128;
  const int d = qv ? tid : tid - 128;
  const int gc_a = qv ? j * kHeadDim + d : (p.Hk + j) * kHeadDim + d;  // q or k channel
  const int gc_v = (2 * p.Hk + h) * kHeadDim + d;                       // v channel (qv threads)
  const float4 wa = *reinterpret_cast<const float4*>(p.conv_w + (size_t)gc_a * kTaps);
  const float4 wv = *reinterpret_cast<const float4*>(p.conv_w + (size_t)gc_v * kTaps);
  uint16_t ha[3] = {0, 0, 0}, hv[3] = {0, 0, 0};  // conv windows, oldest first
  if (init) {
    const uint16_t* hp = p.conv_hist + ((size_t)slot * p.CH + gc_a) * 3;
    ha[0] = hp[0]; ha[1] = hp[1]; ha[2] = hp[2];
    if (qv) {
      const uint16_t* hq = p.conv_hist + ((size_t)slot * p.CH + gc_v) * 3;
      hv[0] = hq[0]; hv[1] = hq[1]; hv[2] = hq[2];
    }
  }

  if (warp == 0) umma::tmem_alloc(tmem_slot, kTmemCols);
  if (tid == 0) {
    for (int b = 0; b < 6; ++b) mbar_init(&bars[b], 1);
    fence_mbar_init();
    issue_x(t0);  // raw rows of the first chunk
  }
  umma::fence_before_sync();
  // All CTAs of the key-head group have read the old history from here on.
  cg::this_cluster().sync();
  umma::fence_after_sync();
  const uint32_t tm = *tmem_slot;
  const uint32_t lane_base = (uint32_t)(32 * quarter) << 16;

  // ---- initial state into tensor memory: thread (row, half) owns 64 columns
  {
    const float* src = p.state + (((size_t)slot * p.Hv + h) * kHeadDim + row) * kHeadDim + half * 64;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      float v[32];
#pragma unroll
      for (int i = 0; i < 32; i += 4) {
        const float4 f = init ? *reinterpret_cast<const float4*>(src + c * 32 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
        v[i] = f.x; v[i + 1] = f.y; v[i + 2] = f.z; v[i + 3] = f.w;
      }
      umma::st32(tm + lane_base + kTS_S + half * 64 + c * 32, v);
    }
  }
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();

  const uint32_t id_kk = umma::idesc(umma::kBF16, true, true, 128, 64);
  const uint32_t id_xz = umma::idesc(umma::kBF16, false, true, 128, 64);
  const uint32_t id_e = umma::idesc(umma::kTF32, false, false, 128, 64);
  const uint32_t id_s = umma::idesc(umma::kTF32, false, false, 128, 128);
  const uint32_t id_o = umma::idesc(umma::kBF16, false, false, 128, 64);
  const uint32_t sKQ = smem_u32(KQ), sKG = smem_u32(KGb), sKT = smem_u32(KTb), sS0 = smem_u32(S0b);
  const uint32_t sTB = smem_u32(TBb), sPB = smem_u32(PBb);

  const int nchunks = (t1 - t0 + kC - 1) / kC;
  bool ok = true;
  for (int c = 0; c < nchunks && ok; ++c) {
    const int tc = t0 + c * kC;
    const int L = min(kC, t1 - tc);
    const uint32_t par = c & 1;

    // ---- z rows of the chunk (the previous chunk's Ogate store must have read ZS)
    if (tid == 0 && want_gate) {
      bulk_wait_read_all();
      mbar_arrive_expect_tx(&bars[5], (uint32_t)(kC * kHeadDim * 2));
      tma_load_3d(ZS, &tmz, 0, h, tc, &bars[5]);
    }

    // ---- gates: g = inclusive cumsum of ln(alpha), e^g, beta
    if (tid < kC) {
      float la = 0.f, b = 0.f;
      if (tid < L) {
        const size_t ai = (size_t)(tc + tid) * p.Hv + h;
        la = fmaxf(log2f(p.alpha[ai]), -115.f);  // log2(alpha), alpha in (0, 1]
        b = p.beta[ai];
      }
      float s = la;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float u = __shfl_up_sync(0xffffffffu, s, o);
        if (lane >= o) s += u;
      }
      scan[tid] = s;
      bv[tid] = b;
    }
    __syncthreads();
    if (tid < kC) {
      const float gt = scan[tid] + (tid >= 32 ? scan[31] : 0.f);
      gv[tid] = gt;
      egv[tid] = ex2(gt);
    }
    __syncthreads();
    if (tid < kC) glv[tid] = tid < L ? ex2(gv[L - 1] - gv[tid]) : 0.f;

    // ---- conv + SiLU from the bulk-copied raw rows, 8 tokens at a time;
    // q, k written channel-major to shared memory, v to tensor memory. The v
    // channel of lane d is split by tokens: warps 0-3 (which also carry q) take
    // tokens 0-31, warps 4-7 (k) take 32-63. Every token row of the staging
    // area is valid to read (rows past T arrive as zeros), so the loop runs
    // branch-free over all 64 rows and masks outputs past the chunk end.
    if (!wait_mma(&bars[4], par)) { ok = false; break; }
    const uint16_t* xa_s = XS + (qv ? 0 : kC) * kHeadDim + d;  // q or k part, channel d
    const uint16_t* xv_s = XS + 2 * kC * kHeadDim + d;          // v part
    auto conv_half = [&](auto qv_c, auto hf_c) {
      constexpr bool kQV = decltype(qv_c)::value;
      constexpr int kHF = decltype(hf_c)::value;
      constexpr bool kV = kQV == (kHF == 0);  // v computed here for these 32 tokens
      // windows (oldest first): a runs on from the previous half; v starts from
      // the slot history (q/v warps, tokens 0..) or from rows 29-31 (k warps, 32..)
      uint16_t wv3[3];
      if constexpr (kQV) {
        wv3[0] = hv[0]; wv3[1] = hv[1]; wv3[2] = hv[2];
      } else {
        wv3[0] = xv_s[29 * kHeadDim]; wv3[1] = xv_s[30 * kHeadDim]; wv3[2] = xv_s[31 * kHeadDim];
      }
      float yv32[32];
#pragma unroll
      for (int gi = 0; gi < 4; ++gi) {
        const int grp = kHF * 4 + gi;
        float ya[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int t = grp * 8 + e;
          const uint16_t xa = xa_s[t * kHeadDim];
          float pre = wa.x * bf16_to_f32(xa);
          pre = fmaf(wa.y, bf16_to_f32(ha[2]), pre);
          pre = fmaf(wa.z, bf16_to_f32(ha[1]), pre);
          pre = fmaf(wa.w, bf16_to_f32(ha[0]), pre);
          ya[e] = t < L ? silu_ftz(pre) : 0.f;
          ha[0] = ha[1]; ha[1] = ha[2]; ha[2] = xa;
          if constexpr (kV) {
            const uint16_t xv = xv_s[t * kHeadDim];
            float pv = wv.x * bf16_to_f32(xv);
            pv = fmaf(wv.y, bf16_to_f32(wv3[2]), pv);
            pv = fmaf(wv.z, bf16_to_f32(wv3[1]), pv);
            pv = fmaf(wv.w, bf16_to_f32(wv3[0]), pv);
            yv32[gi * 8 + e] = t < L ? silu_ftz(pv) : 0.f;
            wv3[0] = wv3[1]; wv3[1] = wv3[2]; wv3[2] = xv;
          }
        }
        // raw q or k, bf16: row d of KQ, tokens (q ? 64 : 0) + 8 grp ...
        {
          uint4 pk;
          pk.x = pack_bf16(ya[0], ya[1]);
          pk.y = pack_bf16(ya[2], ya[3]);
          pk.z = pack_bf16(ya[4], ya[5]);
          pk.w = pack_bf16(ya[6], ya[7]);
          const int col = (kQV ? 64 : 0) + grp * 8;
          *reinterpret_cast<uint4*>(reinterpret_cast<unsigned char*>(KQ) + umma::tile_off(d, col * 2, 256)) = pk;
        }
        if constexpr (!kQV) {
          uint4 pk;
          const int t = grp * 8;
          pk.x = pack_bf16(ya[0] * egv[t + 0], ya[1] * egv[t + 1]);
          pk.y = pack_bf16(ya[2] * egv[t + 2], ya[3] * egv[t + 3]);
          pk.z = pack_bf16(ya[4] * egv[t + 4], ya[5] * egv[t + 5]);
          pk.w = pack_bf16(ya[6] * egv[t + 6], ya[7] * egv[t + 7]);
          *reinterpret_cast<uint4*>(KGb + umma::tile_off(d, t * 2, 128)) = pk;
          *reinterpret_cast<float4*>(KTb + umma::tile_off(d, t * 4, 256)) =
              make_float4(to_tf32(ya[0]), to_tf32(ya[1]), to_tf32(ya[2]), to_tf32(ya[3]));
          *reinterpret_cast<float4*>(KTb + umma::tile_off(d, t * 4 + 16, 256)) =
              make_float4(to_tf32(ya[4]), to_tf32(ya[5]), to_tf32(ya[6]), to_tf32(ya[7]));
        }
        // per-token sum of squares of the raw q (warps 0-3) or k (warps 4-7)
        float sq[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) sq[e] = ya[e] * ya[e];
        const float tot = reduce8(sq, lane);
        if ((lane & 3) == 0) npart[warp * 64 + grp * 8 + tok8(lane)] = tot;
      }
      // v rows d = this thread's lane, columns 32 hf ..
      if constexpr (kV) umma::st32_nowait(tm + lane_base + kT_V + kHF * 32, yv32);
    };
    {
      // the windows carried to the next chunk: raw rows L-3 .. L-1, reaching
      // back into the previous window when the chunk is shorter than 3
      const uint16_t na[3] = {L >= 3 ? xa_s[(L - 3) * kHeadDim] : (L == 2 ? ha[2] : ha[1]),
                              L >= 2 ? xa_s[(L - 2) * kHeadDim] : ha[2], xa_s[(L - 1) * kHeadDim]};
      const uint16_t nv[3] = {L >= 3 ? xv_s[(L - 3) * kHeadDim] : (L == 2 ? hv[2] : hv[1]),
                              L >= 2 ? xv_s[(L - 2) * kHeadDim] : hv[2], xv_s[(L - 1) * kHeadDim]};
      if (qv) {
        conv_half(std::true_type{}, std::integral_constant<int, 0>{});
        conv_half(std::true_type{}, std::integral_constant<int, 1>{});
      } else {
        conv_half(std::false_type{}, std::integral_constant<int, 0>{});
        conv_half(std::false_type{}, std::integral_constant<int, 1>{});
      }
#pragma unroll
      for (int i = 0; i < 3; ++i) {
        ha[i] = na[i];
        hv[i] = nv[i];
      }
    }
    umma::wait_st();
    sync_for_mma();

    // ---- [K;Q] K^T (bf16): D1 lanes 0-63 = K K^T rows, lanes 64-127 = Q K^T rows
    if (tid == 0) {
#pragma unroll
      for (int kk = 0; kk < kHeadDim / 16; ++kk) {
        const uint64_t a = umma::smem_desc(sKQ + kk * 4096, 256, true);
        umma::mma<umma::kBF16>(tm + kT_D1, a, a, id_kk, kk > 0);
      }
      umma::commit(&bars[0]);
    }
    if (tid < kC) {
      const float sq = (npart[0 * 64 + tid] + npart[1 * 64 + tid]) + (npart[2 * 64 + tid] + npart[3 * 64 + tid]);
      const float sk = (npart[4 * 64 + tid] + npart[5 * 64 + tid]) + (npart[6 * 64 + tid] + npart[7 * 64 + tid]);
      iqv[tid] = rsqrtf(sq + 1e-12f);
      ikv[tid] = rsqrtf(sk + 1e-12f);
    }
    // ---- S0 as a bf16 operand; S *= e^{g_C} in tensor memory for the update below
    {
      const float decay = egv[L - 1];
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        float v[32];
        const uint32_t col = kTS_S + half * 64 + cc * 32;
        umma::ld32(tm + lane_base + col, v);
#pragma unroll
        for (int q8 = 0; q8 < 4; ++q8) {
          uint4 pk;
          pk.x = pack_bf16(v[q8 * 8 + 0], v[q8 * 8 + 1]);
          pk.y = pack_bf16(v[q8 * 8 + 2], v[q8 * 8 + 3]);
          pk.z = pack_bf16(v[q8 * 8 + 4], v[q8 * 8 + 5]);
          pk.w = pack_bf16(v[q8 * 8 + 6], v[q8 * 8 + 7]);
          const int dk = half * 64 + cc * 32 + q8 * 8;
          *reinterpret_cast<uint4*>(S0b + umma::tile_off(row, dk * 2, 256)) = pk;
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] *= decay;
        umma::st32(tm + lane_base + col, v);
      }
    }
    sync_for_mma();
    // ---- X = S0 Kg^T and Z = S0 Q^T (bf16)
    if (tid == 0) {
#pragma unroll
      for (int kk = 0; kk < kHeadDim / 16; ++kk) {
        const uint64_t a = umma::smem_desc(sS0 + kk * 256, 256, false);
        umma::mma<umma::kBF16>(tm + kT_X, a, umma::smem_desc(sKG + kk * 2048, 128, true), id_xz, kk > 0);
        umma::mma<umma::kBF16>(tm + kT_Z, a, umma::smem_desc(sKQ + 1024 + kk * 4096, 256, true), id_xz, kk > 0);
      }
      umma::commit(&bars[1]);
    }

    // ---- A (for the inverse) and P from K K^T and Q K^T
    if (!wait_mma(&bars[0], par)) { ok = false; break; }
    {
      float v[32];
      umma::ld32(tm + lane_base + kT_D1 + half * 32, v);
      if (row < 64) {
        const int r = row;
        const float br = bv[r], gr = gv[r], ikr = ikv[r];
#pragma unroll
        for (int e4 = 0; e4 < 8; ++e4) {
          float a4[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int i = half * 32 + e4 * 4 + e;
            a4[e] = i < r ? br * ex2(gr - gv[i]) * v[e4 * 4 + e] * ikr * ikv[i] : 0.f;
          }
          *reinterpret_cast<float4*>(AM + r * kLd + half * 32 + e4 * 4) = make_float4(a4[0], a4[1], a4[2], a4[3]);
        }
      } else {
        const int r = row - 64;
        const float gr = gv[r], iqr = iqv[r];
#pragma unroll
        for (int q8 = 0; q8 < 4; ++q8) {
          float pe[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int i = half * 32 + q8 * 8 + e;
            pe[e] = i <= r ? ex2(gr - gv[i]) * v[q8 * 8 + e] * iqr * ikv[i] : 0.f;
          }
          uint4 pk;
          pk.x = pack_bf16(pe[0], pe[1]);
          pk.y = pack_bf16(pe[2], pe[3]);
          pk.z = pack_bf16(pe[4], pe[5]);
          pk.w = pack_bf16(pe[6], pe[7]);
          *reinterpret_cast<uint4*>(PBb + umma::tile_off(r, (half * 32 + q8 * 8) * 2, 128)) = pk;
        }
      }
    }
    __syncthreads();
    // ---- T = (I + A)^-1, blocked by 16 (T row-major in TS, rows of kLd floats).
    // Diagonal blocks by forward substitution (one column per thread); then the
    // off-diagonal blocks one block diagonal at a time, T_ab = -T_aa M with
    // M = sum_{b<=c<a} A_ac T_cb, each thread producing 4 adjacent columns from
    // 16-byte shared-memory loads. The strictly upper blocks are never written:
    // the Tb pass below masks them.
    if (tid < kC) {
      const int a = tid >> 4, cc = tid & 15;
      const float* Ab = AM + (16 * a) * kLd + 16 * a;
      float x[16];
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < r; ++i) s = fmaf(Ab[r * kLd + i], x[i], s);
        x[r] = r < cc ? 0.f : (r == cc ? 1.f : -s);
      }
#pragma unroll
      for (int r = 0; r < 16; ++r) TS[(16 * a + r) * kLd + 16 * a + cc] = x[r];
    }
    __syncthreads();
#pragma unroll 1
    for (int dist = 1; dist < 4; ++dist) {
      const int nblk = 4 - dist;  // blocks (a, a - dist) for a = dist .. 3
      const bool act = tid < nblk * 64;
      const int blk = tid >> 6, r = (tid >> 2) & 15, c4 = tid & 3;
      const int a = dist + blk, b = a - dist;
      if (act) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        const float* ar = AM + (16 * a + r) * kLd;
        const float* tc0 = TS + 16 * b + 4 * c4;
#pragma unroll 2
        for (int i0 = 16 * b; i0 < 16 * a; i0 += 4) {
          const float4 av = *reinterpret_cast<const float4*>(ar + i0);
          const float ae[4] = {av.x, av.y, av.z, av.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float4 tv = *reinterpret_cast<const float4*>(tc0 + (i0 + e) * kLd);
            acc.x = fmaf(ae[e], tv.x, acc.x);
            acc.y = fmaf(ae[e], tv.y, acc.y);
            acc.z = fmaf(ae[e], tv.z, acc.z);
            acc.w = fmaf(ae[e], tv.w, acc.w);
          }
        }
        *reinterpret_cast<float4*>(MS + blk * kMsBlk + r * kMsLd + 4 * c4) = acc;
      }
      __syncthreads();
      if (act) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        const float* tr = TS + (16 * a + r) * kLd + 16 * a;
        const float* mc = MS + blk * kMsBlk + 4 * c4;
#pragma unroll
        for (int i0 = 0; i0 < 16; i0 += 4) {
          const float4 tv4 = *reinterpret_cast<const float4*>(tr + i0);
          const float te[4] = {tv4.x, tv4.y, tv4.z, tv4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float4 mv = *reinterpret_cast<const float4*>(mc + (i0 + e) * kMsLd);
            acc.x = fmaf(te[e], mv.x, acc.x);
            acc.y = fmaf(te[e], mv.y, acc.y);
            acc.z = fmaf(te[e], mv.z, acc.z);
            acc.w = fmaf(te[e], mv.w, acc.w);
          }
        }
        *reinterpret_cast<float4*>(TS + (16 * a + r) * kLd + 16 * b + 4 * c4) =
            make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
      }
      __syncthreads();
    }
    // ---- Tb = T diag(beta) as a tf32 K-major operand: rows r, 16-byte chunks of 4 columns
    for (int it = tid; it < kC * 16; it += kThreads) {
      const int r = it >> 4, ck = it & 15;
      float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
      if ((ck >> 2) <= (r >> 4)) {  // on or below the block diagonal
        const float4 t4 = *reinterpret_cast<const float4*>(TS + r * kLd + 4 * ck);
        f.x = to_tf32(t4.x * bv[4 * ck + 0]);
        f.y = to_tf32(t4.y * bv[4 * ck + 1]);
        f.z = to_tf32(t4.z * bv[4 * ck + 2]);
        f.w = to_tf32(t4.w * bv[4 * ck + 3]);
      }
      *reinterpret_cast<float4*>(TBb + umma::tile_off(r, ck * 16, 256)) = f;
    }
    // ---- Y = V^T - X (tf32, rows dv), over S0's now-free space
    if (!wait_mma(&bars[1], par)) { ok = false; break; }
    // the scratch area is free again (A and T consumed): raw rows of the next chunk
    if (tid == 0 && c + 1 < nchunks) issue_x(tc + kC);
    {
      float v[32], vv[32];
      umma::ld32(tm + lane_base + kT_X + half * 32, v);
      umma::ld32(tm + lane_base + kT_V + half * 32, vv);
#pragma unroll
      for (int q4 = 0; q4 < 8; ++q4) {
        float y4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int t = half * 32 + q4 * 4 + e;
          y4[e] = to_tf32(vv[q4 * 4 + e] - v[q4 * 4 + e] * ikv[t]);
        }
        *reinterpret_cast<float4*>(S0b + umma::tile_off(row, (half * 32 + q4 * 4) * 4, 256)) =
            make_float4(y4[0], y4[1], y4[2], y4[3]);
      }
    }
    sync_for_mma();
    // ---- E^T = Y Tb^T (tf32)
    if (tid == 0) {
#pragma unroll
      for (int kk = 0; kk < kC / 8; ++kk)
        umma::mma<umma::kTF32>(tm + kT_E, umma::smem_desc(sS0 + kk * 256, 256, false),
                               umma::smem_desc(sTB + kk * 256, 256, false), id_e, kk > 0);
      umma::commit(&bars[2]);
    }
    if (!wait_mma(&bars[2], par)) { ok = false; break; }
    // ---- E as bf16 (A of O' = E^T P^T) and E' = E diag(Gamma_C / |k|) as tf32 (A of the update)
    {
      float v[32];
      umma::ld32(tm + lane_base + kT_E + half * 32, v);
#pragma unroll
      for (int q8 = 0; q8 < 4; ++q8) {
        uint4 pk;
        pk.x = pack_bf16(v[q8 * 8 + 0], v[q8 * 8 + 1]);
        pk.y = pack_bf16(v[q8 * 8 + 2], v[q8 * 8 + 3]);
        pk.z = pack_bf16(v[q8 * 8 + 4], v[q8 * 8 + 5]);
        pk.w = pack_bf16(v[q8 * 8 + 6], v[q8 * 8 + 7]);
        *reinterpret_cast<uint4*>(KGb + umma::tile_off(row, (half * 32 + q8 * 8) * 2, 128)) = pk;
      }
#pragma unroll
      for (int q4 = 0; q4 < 8; ++q4) {
        float e4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int t = half * 32 + q4 * 4 + e;
          e4[e] = to_tf32(v[q4 * 4 + e] * glv[t] * ikv[t]);
        }
        *reinterpret_cast<float4*>(S0b + umma::tile_off(row, (half * 32 + q4 * 4) * 4, 256)) =
            make_float4(e4[0], e4[1], e4[2], e4[3]);
      }
    }
    sync_for_mma();
    // ---- S += E' K (tf32, accumulate) and O' = E^T P^T (bf16)
    if (tid == 0) {
#pragma unroll
      for (int kk = 0; kk < kC / 8; ++kk)
        umma::mma<umma::kTF32>(tm + kTS_S, umma::smem_desc(sS0 + kk * 256, 256, false),
                               umma::smem_desc(sKT + kk * 256, 256, false), id_s, 1);
#pragma unroll
      for (int kk = 0; kk < kC / 16; ++kk)
        umma::mma<umma::kBF16>(tm + kT_O, umma::smem_desc(sKG + kk * 256, 128, false),
                               umma::smem_desc(sPB + kk * 256, 128, false), id_o, kk > 0);
      umma::commit(&bars[3]);
    }
    if (!wait_mma(&bars[3], par)) { ok = false; break; }
    // ---- o = (e^g Z / |q| + O') / sqrt(dk), then the gated RMSNorm over dv
    float ov[32];
    {
      float z[32];
      umma::ld32(tm + lane_base + kT_Z + half * 32, z);
      umma::ld32(tm + lane_base + kT_O + half * 32, ov);
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const int t = half * 32 + e;
        ov[e] = fmaf(egv[t] * iqv[t], z[e], ov[e]) * kInvSqrtDk;
      }
#pragma unroll
      for (int q8 = 0; q8 < 4; ++q8) {
        float sq[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) sq[e] = ov[q8 * 8 + e] * ov[q8 * 8 + e];
        const float tot = reduce8(sq, lane);
        if ((lane & 3) == 0) rpart[quarter * 64 + half * 32 + q8 * 8 + tok8(lane)] = tot;
      }
    }
    __syncthreads();
    if (tid < kC)
      rinv[tid] = rsqrtf(((rpart[tid] + rpart[64 + tid]) + (rpart[128 + tid] + rpart[192 + tid])) *
                             (1.0f / kHeadDim) + p.eps);
    if (want_gate && !wait_mma(&bars[5], par)) { ok = false; break; }  // z rows landed (also syncs)
    if (!want_gate) __syncthreads();
    {
      if (p.o) {
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int t = half * 32 + e;
          if (t < L) p.o[((size_t)(tc + t) * p.Hv + h) * kHeadDim + row] = f32_to_bf16(ov[e]);
        }
      }
      if (want_gate) {
        // Ogate over the z rows in place (thread: column `row` of 32 token rows) ...
        const float gm = p.gamma[row];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int t = half * 32 + e;
          uint16_t* zp = ZS + t * kHeadDim + row;
          *zp = f32_to_bf16(ov[e] * rinv[t] * gm * silu_ftz(bf16_to_f32(*zp)));
        }
      }
    }
    umma::fence_proxy_async_smem();
    __syncthreads();
    // ... then stored with one tensor copy (a partial last chunk row by row, so
    // that the next request's rows are not touched); the next chunk's z rows
    // wait until these stores have read ZS
    if (tid == 0 && want_gate) {
      if (L == kC) {
        tma_store_3d(&tmo, 0, h, tc, ZS);
      } else {
        for (int t = 0; t < L; ++t)
          bulk_s2g(p.ogate + ((size_t)(tc + t) * p.Hv + h) * kHeadDim, ZS + t * kHeadDim, 256);
      }
      bulk_commit();
    }
  }

  if (ok) {
    // ---- final state back to the slot, history to the owners' channels
    float* dst = p.state + (((size_t)slot * p.Hv + h) * kHeadDim + row) * kHeadDim + half * 64;
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      float v[32];
      umma::ld32(tm + lane_base + kTS_S + half * 64 + cc * 32, v);
#pragma unroll
      for (int i = 0; i < 32; i += 4)
        *reinterpret_cast<float4*>(dst + cc * 32 + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
    }
    if (g == 0) {  // q and k history: the group's first CTA
      uint16_t* hp = p.conv_hist + ((size_t)slot * p.CH + gc_a) * 3;
      hp[0] = ha[0]; hp[1] = ha[1]; hp[2] = ha[2];
    }
    if (qv) {  // v history: the head's own CTA
      uint16_t* hp = p.conv_hist + ((size_t)slot * p.CH + gc_v) * 3;
      hp[0] = hv[0]; hp[1] = hv[1]; hp[2] = hv[2];
    }
  } else {
    if (tid == 0) report(p.dev_err, GDN_DEVERR_TIMEOUT);
    // give MMAs still in flight a second bounded chance before the memory is freed
    for (int b = 0; b < 6; ++b) mbar_wait_bounded(&bars[b], 0);
  }
  if (tid == 0) bulk_wait_all();  // Ogate rows stored
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  if (warp == 0) umma::tmem_dealloc(tm, kTmemCols);
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// bf16 tensor map of `rank` dims (innermost first) with a box of `box` elements.
bool encode_bf16(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
                 const cuuint32_t* box) {
  const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint32_t elem[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides, box, elem,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream) {
  CUtensorMap tmx{}, tmz{}, tmo{};
  {
    const cuuint64_t dims[2] = {(cuuint64_t)a.CH, (cuuint64_t)a.T};
    const cuuint64_t strides[1] = {(cuuint64_t)a.CH * 2};
    const cuuint32_t box[2] = {kHeadDim, kC};
    if (!encode_bf16(&tmx, a.qkv0, 2, dims, strides, box)) return cudaErrorInvalidValue;
  }
  if (a.ogate) {
    const cuuint64_t dims[3] = {kHeadDim, (cuuint64_t)a.Hv, (cuuint64_t)a.T};
    const cuuint64_t strides[2] = {kHeadDim * 2, (cuuint64_t)a.Hv * kHeadDim * 2};
    const cuuint32_t box[3] = {kHeadDim, 1, kC};
    if (!encode_bf16(&tmz, a.z, 3, dims, strides, box) || !encode_bf16(&tmo, a.ogate, 3, dims, strides, box))
      return cudaErrorInvalidValue;
  }
  cudaError_t err = ensure_dynamic_smem(reinterpret_cast<const void*>(&prefill_tc_kernel), kSmemBytes);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.Hv, a.N, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = a.G;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, prefill_tc_kernel, a, tmx, tmz, tmo);
}

}  // namespace gdn
