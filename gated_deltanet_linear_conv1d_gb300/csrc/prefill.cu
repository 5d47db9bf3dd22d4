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
// One CTA per (value head h, request n), 512 threads (16 warps, four per
// tensor-memory lane quarter, splitting the columns of every readout). The G
// CTAs of a key head all read the key head's old q/k conv history; the last of
// them to start (an atomic ticket per (request, key head)) writes the new one,
// so the in-place update needs no co-scheduling (a cluster of 3 would leave 14
// of the 152 SMs idle at this kernel's footprint). The fp32 state lives in tensor memory (128 lanes x 128 columns) for
// the whole request. The raw QKV0 rows and the z rows of the next chunk are
// fetched by TMA while the current chunk runs. Per chunk:
//   S0 -> packed bf16 pairs in tensor memory, S *= e^{g_C} in tensor memory
//   conv + SiLU (CUDA cores, thread = channel x token range) -> raw q, k (bf16,
//       channel-major), k (fp32, channel-major), |q|, |k|
//   [K;Q] K^T                 tcgen05 bf16  M=128 N=128 K=128 (operands MN-major)
//   [X' | Z] = S0 [K;Q]^T      tcgen05 bf16  M=128 N=128 K=128 (A = S0 from tensor
//       memory; X = X' diag(e^g) at read-out)
//   A, P from K K^T, Q K^T;  T = (I + A)^-1 on CUDA cores (recursive doubling
//       over 16-row blocks), written as Tb = T diag(b) in tf32
//   Y = V^T - X -> tf32 in tensor memory;  E^T = Y Tb^T   tcgen05 tf32 M=128 N=64 K=64
//   K' = diag(Gamma_C / |k|) K in tf32 (shared memory, in place)
//   S += E^T K'                 tcgen05 tf32 M=128 N=128 K=64 (accumulate; A = E^T
//       straight from tensor memory)
//   O' = E^T P^T                tcgen05 tf32 M=128 N=64 K=64 (A = E^T from tensor memory)
//   o = e^g Z / |q| + O' -> token-major in shared memory, then the gated
//       RMSNorm with eight threads per token, bf16 out.
// The two products that feed the carried state (E and the state update) take
// tf32 operands, and so does O'; the Gram product and [X' | Z] take bf16
// (measured against the fp64 oracle: state error ~6e-4, output error ~3e-3
// relative L2).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>
#include <type_traits>

#include "device.cuh"
#include "launch.h"
#include "umma.cuh"


namespace gdn {

namespace {

constexpr int kThreads = 512;  // 16 warps: 4 per tensor-memory lane quarter
constexpr int kTmaThread = kThreads - 32;  // issues the in-loop TMA copies (thread 0 issues the MMAs)
constexpr int kC = 64;  // chunk length
constexpr float kInvSqrtDk = 0.08838834764831845f;

// Shared-memory regions (byte offsets, 1024-aligned).
// The two conv-written tiles have rows of 256 bytes, their row octets 16 bytes
// further apart than dense (2064 instead of 2048): the conv's 16-byte stores to
// rows 2j and 2j + 1 of eight threads then hit distinct banks.
constexpr int kOct = 2048 + 16;
constexpr int kKQ = 0;                  // bf16 [128 dk][128 t]: k tokens 0-63, q tokens 64-127 (MN-major)
constexpr int kKT = kKQ + 33792;        // fp32 [128 dk][64 t]: raw k, then k diag(Gamma_C / |k|) as tf32 (K-major B)
constexpr int kOT = kKT + 33792;        // fp32 [64 t][128 dv]: o of the chunk, token-major (the gate's input)
static_assert(16 * kOct <= 33792, "padded tile overruns its region");
// Scratch: raw q and k rows of a chunk [2 parts][64 t][128] bf16 (TMA, read by
// the conv), later the inverse's A [64][68], T [64][68] and block products
// [32][36]; then the q and k rows of the next chunk.
constexpr int kSCR = kOT + 32768;
constexpr int kScrBytes = 40960;
constexpr int kXS = kSCR;               // raw q, k rows, 32768 B
constexpr int kLd = 68;                 // row stride (floats) of A and T: 16-byte aligned rows
constexpr int kMsLd = 36;               // row stride (floats) of the inverse's block products
constexpr int kAM = kSCR;               // fp32 [64][kLd]
constexpr int kTS = kAM + 64 * kLd * 4;  // fp32 [64][kLd]
constexpr int kMS = kTS + 64 * kLd * 4;  // fp32 [32][kMsLd]
static_assert(kMS + 32 * kMsLd * 4 <= kSCR + kScrBytes, "inverse scratch overruns its region");
static_assert(2 * kC * kHeadDim * 2 <= kScrBytes, "q, k rows overrun the scratch region");
constexpr int kXV = kSCR + kScrBytes;   // bf16 [64 t][128]: raw v rows of the next chunk (TMA)
constexpr int kZS = kXV + 16384;        // bf16 [64][128]: z rows, then Ogate rows
constexpr int kTB = kZS + 16384;        // tf32 [64 r][64 i]: T diag(b) (K-major B)
constexpr int kPB = kTB + 16384;        // tf32 [64 r][64 i]: P (K-major B)
constexpr int kSmall = kPB + 16384;     // small per-chunk vectors
constexpr int kSmallFloats = 2 * 4 * 64 + 64 * 2 + kHeadDim;
constexpr int kBars = kSmall + kSmallFloats * 4;
constexpr int kSmemBytes = kBars + 128;

// Tensor-memory columns. D1 = [K;Q][K;Q]^T takes 128 columns; E reuses its
// first 64 once A, P and the norms have been read out of it. X' (then Y in
// place) and Z share 128. S0 as packed bf16 pairs (the A operand of [X' | Z])
// sits in O''s 64 columns until O' is written. v (fp32, channel-major) lives
// in the last 64.
constexpr uint32_t kTS_S = 0, kT_D1 = 128, kT_E = 128, kT_X = 256, kT_Z = 320, kT_O = 384, kT_S0 = 384,
                   kT_V = 448, kTmemCols = 512;

__device__ __forceinline__ float to_tf32(float x) { return umma::to_tf32(x); }

// 2^x via the hardware approximation (ex2.approx); its error is far below the
// bf16 / tf32 rounding that every use of it is followed by.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// log2(x) via the hardware approximation (lg2.approx); its absolute error is
// far below the rounding of the products the gates scale.
__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two floats to a bf16 pair (round to nearest even), a in the low half.
__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(b), "f"(a));
  return d;
}

// Barrier 1 over warps 0-7 only (the triangular inverse runs there while the
// other warps form Y).
__device__ __forceinline__ void inv_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// Waits for an MMA-completion phase; the outcome is uniform over the CTA.
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
  const int h = blockIdx.x, n = p.order ? p.order[blockIdx.y] : blockIdx.y;
  const int g = h % p.G, j = h / p.G;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // warp w reads tensor-memory lanes 32 (w % 4) ..; the four warps of a lane
  // quarter split the columns of every readout (part = w / 4)
  const int quarter = warp & 3, part = warp >> 2;
  const int row = 32 * quarter + lane;  // tensor-memory lane read by this thread

  // ---- request checks (uniform over the request's CTAs); the request's scalars
  // are loaded together, before the first check, so their latencies overlap
  const int slot = p.slot_idx[n];
  const int t0 = p.qsl[n], t1 = p.qsl[n + 1];
  const int p0 = p.pos0 ? p.pos0[n] : 0;  // tokens of the request before this call
  const bool init = p.has_init ? p.has_init[n] != 0 : true;
  if (slot < 0) return;
  if (t0 < 0 || t1 < t0 || t1 > p.T || (n == 0 && t0 != 0) || (n == p.N - 1 && t1 != p.T)) {
    if (tid == 0 && g == 0) report(p.dev_err, GDN_DEVERR_OFFSETS);
    return;
  }
  if (slot >= p.Rs) {
    if (tid == 0 && g == 0) report(p.dev_err, GDN_DEVERR_SLOT);
    return;
  }
  if (t1 == t0) return;  // no tokens: the slot is left untouched
  if (p0 < 0) {
    if (tid == 0 && g == 0) report(p.dev_err, GDN_DEVERR_OFFSETS);
    return;
  }

  // chunks end on absolute multiples of 64 (p0 tokens precede this call), so
  // the first one may be short
  const int first = min(kC - p0 % kC, t1 - t0);
  const int nchunks = 1 + (t1 - t0 - first + kC - 1) / kC;
  // the gate warp's first alpha, beta loads are issued here, ahead of the setup
  constexpr int kGateWarp = kThreads / 32 - 1;
  float alpha_n0 = 1.f, beta_n0 = 0.f, alpha_n1 = 1.f, beta_n1 = 0.f;
  auto load_ab = [&](int ts, int len) {  // alpha, beta of tokens ts .. ts + len - 1
    if (lane < len) {
      alpha_n0 = p.alpha[(size_t)(ts + lane) * p.Hv + h];
      beta_n0 = p.beta[(size_t)(ts + lane) * p.Hv + h];
    }
    if (lane + 32 < len) {
      alpha_n1 = p.alpha[(size_t)(ts + lane + 32) * p.Hv + h];
      beta_n1 = p.beta[(size_t)(ts + lane + 32) * p.Hv + h];
    }
  };
  if (warp == kGateWarp) load_ab(t0, first);

  uint16_t* KQ = reinterpret_cast<uint16_t*>(smem + kKQ);
  unsigned char* KTb = smem + kKT;
  const uint16_t* XS = reinterpret_cast<const uint16_t*>(smem + kXS);
  uint16_t* const ZS = reinterpret_cast<uint16_t*>(smem + kZS);
  const uint16_t* XV = reinterpret_cast<const uint16_t*>(smem + kXV);
  float* OT = reinterpret_cast<float*>(smem + kOT);
  float* AM = reinterpret_cast<float*>(smem + kAM);
  float* TS = reinterpret_cast<float*>(smem + kTS);
  // the four 16 x 16 diagonal blocks of A, transposed (block a: [16 i][16 r]),
  // for the forward substitution; in OT, which is free until the chunk's o
  float* ATD = OT;
  unsigned char* TBb = smem + kTB;
  unsigned char* PBb = smem + kPB;
  float* small = reinterpret_cast<float*>(smem + kSmall);
  // per-chunk gate vectors, double-buffered by chunk parity (chunk c + 1's are
  // computed while chunk c runs): [64] g / ln 2 (cumulative log2 of alpha), [64]
  // e^g, [64] e^{g_C - g_t} (0 past the chunk end), [64] beta
  float* gates = small;          // [2][4][64]
  float* iqv = gates + 2 * 4 * 64;  // [64] 1/|q|
  float* ikv = iqv + 64;         // [64] 1/|k|
  float* gam = ikv + 64;         // [128] the RMSNorm gain
  float* MS = reinterpret_cast<float*>(smem + kMS);
  // MMA completions 0: [K;Q][K;Q]^T  1: X,Z  2: E  3: S, O';  copies 4: raw q, k rows
  // 5: z rows  6: raw v rows
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 7);
  const bool want_gate = p.ogate != nullptr;
  // Thread 0: TMA the raw QKV0 rows (q_j, k_j, v_h segments, 64 tokens each, from
  // token tcs) into the scratch area. Rows past the request are masked by the
  // conv; rows past T arrive as zeros.
  auto issue_x = [&](int tcs) {
    mbar_arrive_expect_tx(&bars[4], (uint32_t)(2 * kC * kHeadDim * 2));
    tma_load_2d(smem + kXS + 0 * kC * 256, &tmx, j * kHeadDim, tcs, &bars[4]);
    tma_load_2d(smem + kXS + 1 * kC * 256, &tmx, (p.Hk + j) * kHeadDim, tcs, &bars[4]);
  };
  // The v rows of the chunk starting at token tcs into XV (their conv runs one chunk early).
  auto issue_v = [&](int tcs) {
    mbar_arrive_expect_tx(&bars[6], (uint32_t)(kC * kHeadDim * 2));
    tma_load_2d(smem + kXV, &tmx, (2 * p.Hk + h) * kHeadDim, tcs, &bars[6]);
  };
  // Thread 0: TMA the z rows of the chunk starting at token tcs into buffer zb.
  auto issue_z = [&](int tcs) {
    mbar_arrive_expect_tx(&bars[5], (uint32_t)(kC * kHeadDim * 2));
    tma_load_3d(ZS, &tmz, 0, h, tcs, &bars[5]);
  };

  // ---- conv work of this thread. q and k at the start of every chunk: thread t
  // takes the adjacent channels 2 (t % 128), + 1 of the key head's 256 q and k
  // channels (q below 128, k above) for tokens 16 (t / 128) .. + 15, the pair
  // computed together in packed fp32x2 arithmetic. v one chunk early, during the
  // previous chunk's triangular inverse: warps 8-15, channel d = row (its
  // tensor-memory lane), tokens 32 (part - 2) .. + 31.
  const int d = row;
  const int qp = tid & 127, qq = tid >> 7;
  const bool isq = qp < 64;
  const int dq = (2 * qp) & 127;  // the pair's first channel within its q or k head
  const int gqk = isq ? j * kHeadDim + dq : (p.Hk + j) * kHeadDim + dq;
  float2 wqk[kTaps];  // tap i of the pair's two channels
  {
    const float4 wa = *reinterpret_cast<const float4*>(p.conv_w + (size_t)gqk * kTaps);
    const float4 wb = *reinterpret_cast<const float4*>(p.conv_w + (size_t)(gqk + 1) * kTaps);
    wqk[0] = make_float2(wa.x, wb.x); wqk[1] = make_float2(wa.y, wb.y);
    wqk[2] = make_float2(wa.z, wb.z); wqk[3] = make_float2(wa.w, wb.w);
  }
  const int gvc = (2 * p.Hk + h) * kHeadDim + d;
  const float4 wv = *reinterpret_cast<const float4*>(p.conv_w + (size_t)gvc * kTaps);
  const bool own_qk = qq == 0;    // carries the pair's running q/k window
  const bool own_v = part == 2;    // carries channel d's running v window
  // running windows (raw inputs, oldest first; the q/k window as bf16 pairs, the
  // pair's first channel in the low half); hv_end is the v window at the end of
  // the current chunk once hv has moved on to the next one
  uint32_t hqk[3] = {0, 0, 0};
  uint16_t hv[3] = {0, 0, 0}, hv_end[3] = {0, 0, 0};
  if (init) {
    if (own_qk) {
      const uint16_t* hp = p.conv_hist + ((size_t)slot * p.CH + gqk) * 3;
      hqk[0] = hp[0] | ((uint32_t)hp[3] << 16);
      hqk[1] = hp[1] | ((uint32_t)hp[4] << 16);
      hqk[2] = hp[2] | ((uint32_t)hp[5] << 16);
    }
    if (own_v) {
      const uint16_t* hp = p.conv_hist + ((size_t)slot * p.CH + gvc) * 3;
      hv[0] = hp[0]; hv[1] = hp[1]; hv[2] = hp[2];
    }
  }

  if (warp == 0) umma::tmem_alloc(tmem_slot, kTmemCols);
  if (tid == 0) {
    for (int b = 0; b < 7; ++b) mbar_init(&bars[b], 1);
    fence_mbar_init();
    issue_x(t0);  // raw rows of the first chunk
    issue_v(t0);
    if (want_gate) issue_z(t0);
  }
  if (tid < kHeadDim) gam[tid] = p.gamma[tid];
  // the initial state (thread (row, part) owns 32 columns) is loaded now and
  // stored into tensor memory after the barrier, so its latency overlaps the setup
  float s0v[32];
  {
    const float* src = p.state + (((size_t)slot * p.Hv + h) * kHeadDim + row) * kHeadDim + part * 32;
#pragma unroll
    for (int i = 0; i < 32; i += 4) {
      const float4 f = init ? *reinterpret_cast<const float4*>(src + i) : make_float4(0.f, 0.f, 0.f, 0.f);
      s0v[i] = f.x; s0v[i + 1] = f.y; s0v[i + 2] = f.z; s0v[i + 3] = f.w;
    }
  }
  // T diag(beta) above the block diagonal stays zero; the rest is rewritten per chunk
  for (int it = tid; it < kC * kC / 4; it += kThreads)
    reinterpret_cast<float4*>(TBb)[it] = make_float4(0.f, 0.f, 0.f, 0.f);
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tm = *tmem_slot;
  const uint32_t lane_base = (uint32_t)(32 * quarter) << 16;
  // This CTA has read the key head's old q/k history (before the barrier above):
  // take its ticket. The group's last CTA to get here writes the new history
  // at its end, when every CTA of the group has read the old one.
  volatile int* last_of_group = reinterpret_cast<volatile int*>(tmem_slot + 1);
  if (tid == 0) {
    __threadfence();
    *last_of_group = atomicAdd(p.tickets + (size_t)n * p.Hk + j, 1) == p.G - 1;
  }

  // ---- initial state into tensor memory
  umma::st32(tm + lane_base + kTS_S + part * 32, s0v);
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();

  const uint32_t id_kk = umma::idesc(umma::kBF16, true, true, 128, 128);
  const uint32_t id_xz = umma::idesc(umma::kBF16, false, true, 128, 128);  // [X' | Z] = S0 [K; Q]^T
  const uint32_t id_e = umma::idesc(umma::kTF32, false, false, 128, 64);
  const uint32_t id_s = umma::idesc(umma::kTF32, false, false, 128, 128);
  const uint32_t id_o = umma::idesc(umma::kTF32, false, false, 128, 64);
  const uint32_t sKQ = smem_u32(KQ), sKT = smem_u32(KTb);
  const uint32_t sTB = smem_u32(TBb), sPB = smem_u32(PBb);

  bool ok = true;
  // ---- gates of a chunk (warp 15, two tokens per lane, no CTA barrier): g =
  // inclusive cumsum of log2(alpha) (so e^{g ln 2} = prod alpha), e^g,
  // e^{g_C - g_t}, beta. The chunk's alpha and beta sit in the lanes' registers,
  // loaded one chunk before they are needed.
  auto make_gates = [&](float* gb, int len) {
    float* g_ = gb;
    float* eg = gb + 64;
    float* gl_ = gb + 128;
    float* b_ = gb + 192;
    const float la0 = lane < len ? fmaxf(lg2(alpha_n0), -115.f) : 0.f;  // alpha in (0, 1]
    const float la1 = lane + 32 < len ? fmaxf(lg2(alpha_n1), -115.f) : 0.f;
    b_[lane] = lane < len ? beta_n0 : 0.f;
    b_[lane + 32] = lane + 32 < len ? beta_n1 : 0.f;
    float s0 = la0, s1 = la1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float u0 = __shfl_up_sync(0xffffffffu, s0, o), u1 = __shfl_up_sync(0xffffffffu, s1, o);
      if (lane >= o) {
        s0 += u0;
        s1 += u1;
      }
    }
    s1 += __shfl_sync(0xffffffffu, s0, 31);
    const float gl = __shfl_sync(0xffffffffu, len - 1 < 32 ? s0 : s1, (len - 1) & 31);  // g at the chunk end
    g_[lane] = s0;
    g_[lane + 32] = s1;
    eg[lane] = ex2(s0);
    eg[lane + 32] = ex2(s1);
    gl_[lane] = lane < len ? ex2(gl - s0) : 0.f;
    gl_[lane + 32] = lane + 32 < len ? ex2(gl - s1) : 0.f;
  };
  if (warp == kGateWarp) {  // chunk 0's gates now (its alpha, beta loaded at entry), chunk 1's into the registers
    make_gates(gates, first);
    if (nchunks > 1) load_ab(t0 + first, min(kC, t1 - t0 - first));
  }
  // Ogate rows of a chunk waiting to be stored (TMA thread): a full chunk with one
  // tensor copy, a partial one row by row so that the next request's rows are
  // not touched. Issued after the CTA barrier that follows the rows' writes.
  int st_tc = -1, st_len = 0;
  auto store_pending = [&]() {
    if (st_tc < 0) return;
    const uint16_t* zsb = ZS;
    if (st_len == kC) {
      tma_store_3d(&tmo, 0, h, st_tc, zsb);
    } else {
      for (int t = 0; t < st_len; ++t)
        bulk_s2g(p.ogate + ((size_t)(st_tc + t) * p.Hv + h) * kHeadDim, zsb + t * kHeadDim, 256);
    }
    bulk_commit();
    st_tc = -1;
  };
  // the window carried past a chunk of len tokens: raw rows len-3 .. len-1,
  // reaching back into the previous window when the chunk is shorter than 3
  auto next_window = [&](const uint16_t* x, const uint16_t (&w)[3], uint16_t (&nw)[3], int len) {
    nw[0] = len >= 3 ? x[(len - 3) * kHeadDim] : (len == 2 ? w[2] : w[1]);
    nw[1] = len >= 2 ? x[(len - 2) * kHeadDim] : w[2];
    nw[2] = x[(len - 1) * kHeadDim];
  };
  // ---- v conv + SiLU of the chunk whose raw v rows are in XV (len tokens), into
  // tensor memory (warps 8-15; the caller has waited for XV)
  auto v_conv = [&](int len) {
    const uint16_t* xv = XV + d;
    const int tb = 32 * (part - 2);
    float w3[3];
    if (own_v) {
      w3[0] = bf16_to_f32(hv[0]); w3[1] = bf16_to_f32(hv[1]); w3[2] = bf16_to_f32(hv[2]);
    } else {
      w3[0] = bf16_to_f32(xv[(tb - 3) * kHeadDim]); w3[1] = bf16_to_f32(xv[(tb - 2) * kHeadDim]);
      w3[2] = bf16_to_f32(xv[(tb - 1) * kHeadDim]);
    }
    float yv[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      const int t = tb + e;
      const float x = bf16_to_f32(xv[t * kHeadDim]);
      float pre = wv.x * x;
      pre = fmaf(wv.y, w3[2], pre);
      pre = fmaf(wv.z, w3[1], pre);
      pre = fmaf(wv.w, w3[0], pre);
      const float y = silu_tanh(pre);
      yv[e] = t < len ? y : 0.f;
      w3[0] = w3[1]; w3[1] = w3[2]; w3[2] = x;
    }
    umma::st32_nowait(tm + lane_base + kT_V + tb, yv);  // v row d = this thread's lane
    umma::wait_st();
    if (own_v) {
      uint16_t nw[3];
      next_window(xv, hv, nw, len);
      hv_end[0] = hv[0]; hv_end[1] = hv[1]; hv_end[2] = hv[2];
      hv[0] = nw[0]; hv[1] = nw[1]; hv[2] = nw[2];
    }
  };
  if (warp >= 8) {  // chunk 0's v
    if (!mbar_wait_bounded(&bars[6], 0)) ok = false;
    if (ok) v_conv(first);
  }
  if (!__syncthreads_and(ok ? 1 : 0)) ok = false;
  int tc = t0, L = first;  // this chunk: tokens tc .. tc + L - 1
  for (int c = 0; c < nchunks && ok; ++c, tc += L, L = min(kC, t1 - tc)) {
    const uint32_t par = c & 1;


    // this chunk's gate vectors (written before the loop or during the previous chunk)
    const float* gv = gates + (c & 1) * 256;
    const float* egv = gv + 64;
    const float* glv = gv + 128;
    const float* bv = gv + 192;

    // ---- S0 as packed bf16 pairs in tensor memory (the A operand of the
    // [X' | Z] MMA), and S *= e^{g_C} in place for this chunk's update; first
    // thing in the chunk, so it overlaps the wait for the raw q, k rows (the
    // previous chunk's MMAs on S have completed and its o has been read)
    {
      const float decay = egv[L - 1];
      float v[32], pk[16];
      const uint32_t col = kTS_S + part * 32;
      umma::ld32(tm + lane_base + col, v);
#pragma unroll
      for (int i = 0; i < 16; ++i) pk[i] = __uint_as_float(pack_bf16(v[2 * i], v[2 * i + 1]));
      umma::st16_nowait(tm + lane_base + kT_S0 + part * 16, pk);
#pragma unroll
      for (int i = 0; i < 32; i += 2) {
        const float2 d2 = __fmul2_rn(make_float2(v[i], v[i + 1]), make_float2(decay, decay));
        v[i] = d2.x;
        v[i + 1] = d2.y;
      }
      umma::st32(tm + lane_base + col, v);
    }
    // ---- conv + SiLU of q and k from the TMA-staged raw rows, written
    // channel-major to shared memory (v was done during the previous chunk).
    // Every token row of the staging area is valid to read (rows past T arrive
    // as zeros), so the loop runs branch-free and masks outputs past the chunk end.
    if (!wait_mma(&bars[4], par)) { ok = false; break; }
    if (tid == kTmaThread) {
      store_pending();  // the previous chunk's Ogate rows
      if (want_gate && c > 0) {
        bulk_wait_read_all();  // ... have been read out of ZS: this chunk's z rows may land
        issue_z(tc);
      }
      if (c + 1 < nchunks) issue_v(tc + L);  // XV is free: the v rows of the next chunk
    }
    {
      // raw rows as bf16 pairs: word t * 64 holds the pair's two channels of token t
      const uint32_t* xs = reinterpret_cast<const uint32_t*>(XS + (isq ? 0 : kC) * kHeadDim + dq);
      auto unpack = [](uint32_t u) { return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u)); };
      uint32_t nw[3];
      if (own_qk) {
        nw[0] = L >= 3 ? xs[(L - 3) * 64] : (L == 2 ? hqk[2] : hqk[1]);
        nw[1] = L >= 2 ? xs[(L - 2) * 64] : hqk[2];
        nw[2] = xs[(L - 1) * 64];
      }
      float2 w3[3];
      if (own_qk) {
        w3[0] = unpack(hqk[0]); w3[1] = unpack(hqk[1]); w3[2] = unpack(hqk[2]);
      } else {
        const int t3 = 16 * qq - 3;
        w3[0] = unpack(xs[t3 * 64]); w3[1] = unpack(xs[(t3 + 1) * 64]); w3[2] = unpack(xs[(t3 + 2) * 64]);
      }
      const float2 half2 = make_float2(0.5f, 0.5f);
#pragma unroll
      for (int gi = 0; gi < 2; ++gi) {
        const int tb = 16 * qq + 8 * gi;
        float2 ya[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int t = tb + e;
          const float2 x = unpack(xs[t * 64]);
          float2 pre = __fmul2_rn(wqk[0], x);
          pre = __ffma2_rn(wqk[1], w3[2], pre);
          pre = __ffma2_rn(wqk[2], w3[1], pre);
          pre = __ffma2_rn(wqk[3], w3[0], pre);
          // SiLU(x) = h + h tanh(h), h = x / 2
          const float2 hh = __fmul2_rn(pre, half2);
          float2 th;
          asm("tanh.approx.f32 %0, %1;" : "=f"(th.x) : "f"(hh.x));
          asm("tanh.approx.f32 %0, %1;" : "=f"(th.y) : "f"(hh.y));
          const float2 y = __ffma2_rn(hh, th, hh);
          ya[e] = t < L ? y : make_float2(0.f, 0.f);
          w3[0] = w3[1]; w3[1] = w3[2]; w3[2] = x;
        }
        // raw q or k, bf16: rows dq, dq + 1 of KQ, tokens (q ? 64 : 0) + tb ..
        unsigned char* kq = reinterpret_cast<unsigned char*>(KQ);
        const int cb = ((isq ? kC : 0) + tb) * 2;
        *reinterpret_cast<uint4*>(kq + umma::tile_off_oct(dq, cb, kOct)) =
            make_uint4(pack_bf16(ya[0].x, ya[1].x), pack_bf16(ya[2].x, ya[3].x), pack_bf16(ya[4].x, ya[5].x),
                       pack_bf16(ya[6].x, ya[7].x));
        *reinterpret_cast<uint4*>(kq + umma::tile_off_oct(dq + 1, cb, kOct)) =
            make_uint4(pack_bf16(ya[0].y, ya[1].y), pack_bf16(ya[2].y, ya[3].y), pack_bf16(ya[4].y, ya[5].y),
                       pack_bf16(ya[6].y, ya[7].y));
        if (!isq) {
          // raw k in fp32 (scaled and rounded to tf32 once the norms are known)
          *reinterpret_cast<float4*>(KTb + umma::tile_off_oct(dq, tb * 4, kOct)) =
              make_float4(ya[0].x, ya[1].x, ya[2].x, ya[3].x);
          *reinterpret_cast<float4*>(KTb + umma::tile_off_oct(dq, tb * 4 + 16, kOct)) =
              make_float4(ya[4].x, ya[5].x, ya[6].x, ya[7].x);
          *reinterpret_cast<float4*>(KTb + umma::tile_off_oct(dq + 1, tb * 4, kOct)) =
              make_float4(ya[0].y, ya[1].y, ya[2].y, ya[3].y);
          *reinterpret_cast<float4*>(KTb + umma::tile_off_oct(dq + 1, tb * 4 + 16, kOct)) =
              make_float4(ya[4].y, ya[5].y, ya[6].y, ya[7].y);
        }
      }
      if (own_qk) {
        hqk[0] = nw[0]; hqk[1] = nw[1]; hqk[2] = nw[2];
      }
    }
    sync_for_mma();

    // ---- [K;Q][K;Q]^T (bf16): D1 lanes 0-63 = K rows, 64-127 = Q rows; columns
    // 0-63 against K, 64-127 against Q. A and P use columns 0-63, the per-token
    // norms |k|^2 and |q|^2 are its diagonal.
    if (tid == 0) {
#pragma unroll
      for (int kk = 0; kk < kHeadDim / 16; ++kk) {
        const uint64_t a = umma::smem_desc_oct(sKQ + kk * 2 * kOct, kOct, true);
        umma::mma<umma::kBF16>(tm + kT_D1, a, a, id_kk, kk > 0);
      }
      umma::commit(&bars[0]);
    } else if (tid == 32) {
      // ---- X' = S0 K^T and Z = S0 Q^T in one MMA over [K; Q] (bf16; S0 was
      // packed into tensor memory at the start of the chunk), issued from another
      // warp so that the Gram product's issue does not wait behind it
#pragma unroll
      for (int kk = 0; kk < kHeadDim / 16; ++kk)
        umma::mma_ts<umma::kKindF16>(tm + kT_X, tm + kT_S0 + kk * 8, umma::smem_desc_oct(sKQ + kk * 2 * kOct, kOct, true),
                                     id_xz, kk > 0);
      umma::commit(&bars[1]);
    }

    // ---- 1/|k|, 1/|q| (L2 norm, eps 1e-12 under the root) from the diagonal of
    // D1: warp (quarter, part 0) reads the 32 columns of its own rows
    if (!wait_mma(&bars[0], par)) { ok = false; break; }
    if (part == 0) {
      float v[32];
      umma::ld32(tm + lane_base + kT_D1 + 32 * quarter, v);
      float dg = v[0];
#pragma unroll
      for (int e = 1; e < 32; ++e) dg = e == lane ? v[e] : dg;
      const float inv = rsqrtf(dg + 1e-12f);
      if (row < 64) ikv[row] = inv;
      else iqv[row - 64] = inv;
    }
    __syncthreads();
    // ---- A (for the inverse) and P from K K^T and Q K^T; the warps whose 32
    // rows lie wholly above their 16 columns (strictly lower A, lower P) only
    // write zeros
    if ((quarter & 1) == 0 && part >= 2) {
      const int r = row & 63;
      if (row < 64) {
#pragma unroll
        for (int e4 = 0; e4 < 4; ++e4)
          *reinterpret_cast<float4*>(AM + r * kLd + part * 16 + e4 * 4) = make_float4(0.f, 0.f, 0.f, 0.f);
      } else {
#pragma unroll
        for (int e4 = 0; e4 < 4; ++e4)
          *reinterpret_cast<float4*>(PBb + umma::tile_off(r, (part * 16 + e4 * 4) * 4, 256)) =
              make_float4(0.f, 0.f, 0.f, 0.f);
      }
    } else {
      float v[16];
      umma::ld16(tm + lane_base + kT_D1 + part * 16, v);
      if (row < 64) {
        const int r = row;
        const float gr = gv[r], bkr = bv[r] * ikv[r];
        float a16[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int i = part * 16 + e;
          // masked entries take ex2(-inf) = 0: no select around the exponential
          a16[e] = (bkr * ex2(i < r ? gr - gv[i] : -INFINITY)) * (v[e] * ikv[i]);
        }
#pragma unroll
        for (int e4 = 0; e4 < 4; ++e4)
          *reinterpret_cast<float4*>(AM + r * kLd + part * 16 + e4 * 4) =
              make_float4(a16[4 * e4], a16[4 * e4 + 1], a16[4 * e4 + 2], a16[4 * e4 + 3]);
        if (part == (r >> 4)) {  // a diagonal block: also transposed (after the branch-free part)
#pragma unroll
          for (int e = 0; e < 16; ++e) ATD[part * 256 + e * 16 + (r & 15)] = a16[e];
        }
      } else {
        const int r = row - 64;
        const float gr = gv[r], iqr = iqv[r];
#pragma unroll
        for (int q8 = 0; q8 < 2; ++q8) {
          float pe[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int i = part * 16 + q8 * 8 + e;
            pe[e] = to_tf32((iqr * ex2(i <= r ? gr - gv[i] : -INFINITY)) * (v[q8 * 8 + e] * ikv[i]));
          }
          // P as tf32 (the B operand of O' = E^T P^T, K-major over i)
          const int i0 = part * 16 + q8 * 8;
          *reinterpret_cast<float4*>(PBb + umma::tile_off(r, i0 * 4, 256)) = make_float4(pe[0], pe[1], pe[2], pe[3]);
          *reinterpret_cast<float4*>(PBb + umma::tile_off(r, i0 * 4 + 16, 256)) =
              make_float4(pe[4], pe[5], pe[6], pe[7]);
        }
      }
    }
    __syncthreads();
    // ---- warps 0-7 invert (I + A) while warps 8-15 form Y (the two are
    // independent; the inverse synchronises on named barrier 1 only)
    bool part_ok = true;
    if (warp < 8) {
      // ---- T = (I + A)^-1 by recursive doubling over 16-row blocks (T row-major
      // in TS, rows of kLd floats), with T diag(beta) written as the tf32 K-major
      // operand as each block is finished:
      //   diagonal blocks T_aa by forward substitution (one column per thread,
      //   the rows of A in 16-byte loads, two partial sums per row);
      //   T_10 = -T_11 A_10 T_00 and T_32 = -T_33 A_32 T_22;
      //   then the lower-left 32x32 block = -T_hi (A_lo-left T_lo), T_hi and T_lo
      //   being the two 32x32 diagonal blocks.
      // A product thread owns a 2x2 (16 -> 32) or 4x2 (32 -> 64) tile over half of
      // the inner index (the partner lane's half is added with shuffles); rows of
      // the left operand come in 16-byte loads.
      if (tid < kC) {
        // 8 x 8 diagonal blocks of T by right-looking forward substitution: thread
        // (block b8, column cc) solves for column cc of (I + A_b8)^-1; once x[i]
        // is final, s[r] += A[r][i] x[i] for every r > i (one dependent FMA per
        // step), column i of A_b8 read from the transposed 16-block in two
        // 16-byte broadcast loads
        const int b8 = tid >> 3, cc = tid & 7, o = 8 * (b8 & 1);
        const float* ATc = ATD + (b8 >> 1) * 256 + o * 16 + o;  // ATc[i * 16 + r] = A[8 b8 + r][8 b8 + i]
        float s8[8], x[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) s8[r] = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          x[i] = i < cc ? 0.f : (i == cc ? 1.f : -s8[i]);
          if (i < 7) {
            const float4 lo = *reinterpret_cast<const float4*>(ATc + i * 16);
            const float4 hi = *reinterpret_cast<const float4*>(ATc + i * 16 + 4);
            const float ac[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
            for (int r = i + 1; r < 8; ++r) s8[r] = fmaf(ac[r], x[i], s8[r]);
          }
        }
        const int col = 8 * b8 + cc;
        const float bc = bv[col];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          TS[(8 * b8 + r) * kLd + col] = x[r];
          *reinterpret_cast<float*>(TBb + umma::tile_off(8 * b8 + r, col * 4, 256)) = to_tf32(x[r] * bc);
        }
      }
      inv_sync();
      {  // 8 -> 16 in each 16-block a: T_10 = -T_11 (A_10 T_00); 256 threads = 4 blocks x 8 x 8
        const int a = tid >> 6, r = (tid >> 3) & 7, c = tid & 7, R0 = 16 * a;
        float* Mb = MS + a * 64;  // [8][8] A_10 T_00 of block a
        {
          // A_10 T_00: T_00 is zero above its diagonal, so all eight terms are taken
          const float4 a0 = *reinterpret_cast<const float4*>(AM + (R0 + 8 + r) * kLd + R0);
          const float4 a1 = *reinterpret_cast<const float4*>(AM + (R0 + 8 + r) * kLd + R0 + 4);
          const float ar[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
          float m = 0.f;
#pragma unroll
          for (int i = 0; i < 8; ++i) m = fmaf(ar[i], TS[(R0 + i) * kLd + R0 + c], m);
          Mb[r * 8 + c] = m;
        }
        inv_sync();
        {
          const float4 t0 = *reinterpret_cast<const float4*>(TS + (R0 + 8 + r) * kLd + R0 + 8);
          const float4 t1 = *reinterpret_cast<const float4*>(TS + (R0 + 8 + r) * kLd + R0 + 12);
          const float tr[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
          float t = 0.f;
#pragma unroll
          for (int i = 0; i < 8; ++i) t = fmaf(tr[i], Mb[i * 8 + c], t);
          TS[(R0 + 8 + r) * kLd + R0 + c] = -t;
          *reinterpret_cast<float*>(TBb + umma::tile_off(R0 + 8 + r, (R0 + c) * 4, 256)) = to_tf32(-t * bv[R0 + c]);
          TS[(R0 + r) * kLd + R0 + 8 + c] = 0.f;  // the 16-block's upper-right 8 x 8 is zero
        }
      }
      inv_sync();
      {  // 16 -> 32: blocks (1,0) and (3,2); 256 threads = block x 64 tiles of 2x2 x 2 shares
        const int kq = tid & 1, c0 = 2 * ((tid >> 1) & 7), r0 = 2 * ((tid >> 4) & 7), blk = tid >> 7;
        const int a = 1 + 2 * blk, b = a - 1;
        // acc[rr][cc] += X[rr][i] Y[i][cc] for i = i0, i0 + 8 below i1 (4 at a time)
        auto mm22 = [](float (&acc)[2][2], const float* X, int ldx, const float* Y, int ldy, int i0, int i1) {
#pragma unroll
          for (int i = i0; i < i1; i += 8) {
            float xs[2][4];
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
              const float4 xv = *reinterpret_cast<const float4*>(X + rr * ldx + i);
              xs[rr][0] = xv.x; xs[rr][1] = xv.y; xs[rr][2] = xv.z; xs[rr][3] = xv.w;
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 yv = *reinterpret_cast<const float2*>(Y + (i + e) * ldy);
#pragma unroll
              for (int rr = 0; rr < 2; ++rr) {
                acc[rr][0] = fmaf(xs[rr][e], yv.x, acc[rr][0]);
                acc[rr][1] = fmaf(xs[rr][e], yv.y, acc[rr][1]);
              }
            }
          }
        };
        {
          float acc[2][2] = {};
          mm22(acc, AM + (16 * a + r0) * kLd, kLd, TS + 16 * b + c0, kLd, 16 * b + 4 * kq, 16 * a);
#pragma unroll
          for (int rr = 0; rr < 2; ++rr)
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) acc[rr][cc] += __shfl_xor_sync(0xffffffffu, acc[rr][cc], 1);
          *reinterpret_cast<float2*>(MS + (16 * blk + r0 + kq) * kMsLd + c0) =
              kq ? make_float2(acc[1][0], acc[1][1]) : make_float2(acc[0][0], acc[0][1]);
        }
        inv_sync();
        {
          float acc[2][2] = {};
          mm22(acc, TS + (16 * a + r0) * kLd + 16 * a, kLd, MS + 16 * blk * kMsLd + c0, kMsLd, 4 * kq, 16);
#pragma unroll
          for (int rr = 0; rr < 2; ++rr)
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) acc[rr][cc] += __shfl_xor_sync(0xffffffffu, acc[rr][cc], 1);
          const float t0v = -(kq ? acc[1][0] : acc[0][0]), t1v = -(kq ? acc[1][1] : acc[0][1]);
          const int r = 16 * a + r0 + kq, cb = 16 * b + c0;
          *reinterpret_cast<float2*>(TS + r * kLd + cb) = make_float2(t0v, t1v);
          *reinterpret_cast<float2*>(TBb + umma::tile_off(r, cb * 4, 256)) =
              make_float2(to_tf32(t0v * bv[cb]), to_tf32(t1v * bv[cb + 1]));
        }
        inv_sync();
      }
      {  // 32 -> 64: rows 32-63, columns 0-31; 256 threads = 128 tiles of 4x2 x 2 shares
        const int kq = tid & 1, c0 = 2 * ((tid >> 1) & 15), r0 = 4 * (tid >> 5);
        // acc[rr][cc] += X[rr][i] Y[i][cc] for i = i0, i0 + 8, ... below i1 (4 at a time)
        auto mm42 = [](float (&acc)[4][2], const float* X, int ldx, const float* Y, int ldy, int i0, int i1) {
#pragma unroll 2
          for (int i = i0; i < i1; i += 8) {
            float xs[4][4];
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) {
              const float4 xv = *reinterpret_cast<const float4*>(X + rr * ldx + i);
              xs[rr][0] = xv.x; xs[rr][1] = xv.y; xs[rr][2] = xv.z; xs[rr][3] = xv.w;
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 yv = *reinterpret_cast<const float2*>(Y + (i + e) * ldy);
#pragma unroll
              for (int rr = 0; rr < 4; ++rr) {
                acc[rr][0] = fmaf(xs[rr][e], yv.x, acc[rr][0]);
                acc[rr][1] = fmaf(xs[rr][e], yv.y, acc[rr][1]);
              }
            }
          }
        };
        auto share2 = [](float (&acc)[4][2]) {  // sum with the partner lane (the other half of i)
#pragma unroll
          for (int rr = 0; rr < 4; ++rr)
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) acc[rr][cc] += __shfl_xor_sync(0xffffffffu, acc[rr][cc], 1);
        };
        {
          // M = A[32 + r][0..32) T[0..32)[c..]: T_lo is zero above its block diagonal
          float acc[4][2] = {};
          mm42(acc, AM + (32 + r0) * kLd, kLd, TS + c0, kLd, (c0 < 16 ? 0 : 16) + 4 * kq, 32);
          share2(acc);
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            const int rr = 2 * kq + h2;  // lane kq writes rows 2kq, 2kq + 1 of the tile
            *reinterpret_cast<float2*>(MS + (r0 + rr) * kMsLd + c0) =
                make_float2(kq ? acc[2 + h2][0] : acc[h2][0], kq ? acc[2 + h2][1] : acc[h2][1]);
          }
        }
        inv_sync();
        {
          // -T_hi[r][0..32) M[0..32)[c..]: T_hi is zero above its block diagonal
          float acc[4][2] = {};
          mm42(acc, TS + (32 + r0) * kLd + 32, kLd, MS + c0, kMsLd, 4 * kq, r0 < 16 ? 16 : 32);
          share2(acc);
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            const int rr = 2 * kq + h2;
            const float t0v = -(kq ? acc[2 + h2][0] : acc[h2][0]), t1v = -(kq ? acc[2 + h2][1] : acc[h2][1]);
            *reinterpret_cast<float2*>(TBb + umma::tile_off(32 + r0 + rr, c0 * 4, 256)) =
                make_float2(to_tf32(t0v * bv[c0]), to_tf32(t1v * bv[c0 + 1]));
          }
        }
      }
    } else {
      // ---- Y = V^T - X (tf32, rows dv), X = (S0 K^T) diag(e^g / |k|), over S0's space once X, Z are done;
      // warps 8-11 take columns 0-31, warps 12-15 columns 32-63
      part_ok = mbar_wait_bounded(&bars[1], par);
      umma::fence_after_sync();
#pragma unroll
      for (int hq = 0; hq < 2; ++hq) {
        const int c0 = (part - 2) * 32 + hq * 16;
        float v[16], vv[16];
        umma::ld16(tm + lane_base + kT_X + c0, v);
        umma::ld16(tm + lane_base + kT_V + c0, vv);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int t = c0 + e;
          v[e] = to_tf32(vv[e] - v[e] * (egv[t] * ikv[t]));  // X = (S0 K^T) e^g / |k|
        }
        // Y in place of X' (the A operand of E^T = Y Tb^T, read from tensor memory)
        umma::st16_nowait(tm + lane_base + kT_X + c0, v);
      }
      umma::wait_st();
      // the next chunk's gates while the inverse runs (published by the barrier below),
      // and the alpha, beta of the one after into the registers
      if (warp == kGateWarp && c + 1 < nchunks) {
        const int tn = tc + L, ln = min(kC, t1 - tn);
        make_gates(gates + ((c + 1) & 1) * 256, ln);
        if (c + 2 < nchunks) load_ab(tn + ln, min(kC, t1 - tn - ln));
      }
      // K' = diag(Gamma_C / |k|) K as tf32, in place (the B operand of the state
      // update): thread (dk row, 32-token half), rows of 16-byte groups
      {
        const int u = tid - 256, r = u & 127, th = u >> 7;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int t = 32 * th + 4 * q;
          float4* kp = reinterpret_cast<float4*>(KTb + umma::tile_off_oct(r, t * 4, kOct));
          const float4 k4 = *kp;
          const float4 g4 = *reinterpret_cast<const float4*>(glv + t);
          const float4 n4 = *reinterpret_cast<const float4*>(ikv + t);
          *kp = make_float4(to_tf32(k4.x * (g4.x * n4.x)), to_tf32(k4.y * (g4.y * n4.y)),
                            to_tf32(k4.z * (g4.z * n4.z)), to_tf32(k4.w * (g4.w * n4.w)));
        }
      }
      // the next chunk's v into tensor memory (this chunk's was read by Y above)
      if (c + 1 < nchunks) {
        if (!mbar_wait_bounded(&bars[6], (c + 1) & 1)) part_ok = false;
        if (part_ok) v_conv(min(kC, t1 - tc - L));
      }
    }
    umma::fence_proxy_async_smem();
    umma::fence_before_sync();
    if (__syncthreads_or(part_ok ? 0 : 1)) { ok = false; break; }
    umma::fence_after_sync();
    // the scratch area is free again (A and T consumed): raw rows of the next chunk
    if (tid == kTmaThread && c + 1 < nchunks) issue_x(tc + L);
    // ---- E^T = Y Tb^T (tf32, Y from tensor memory); once E is in tensor memory,
    // S += E^T K' and O' = E^T P^T (tf32) with E^T read from there in turn (the
    // tensor core reads the fp32 accumulator at tf32 precision, low bits dropped)
    if (tid == 0) {
#pragma unroll
      for (int kk = 0; kk < kC / 8; ++kk)
        umma::mma_ts<umma::kKindTF32>(tm + kT_E, tm + kT_X + kk * 8, umma::smem_desc(sTB + kk * 256, 256, false),
                                      id_e, kk > 0);
      umma::commit(&bars[2]);
      if (mbar_wait_bounded(&bars[2], par)) {
        umma::fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < kC / 8; ++kk)
          umma::mma_ts<umma::kKindTF32>(tm + kTS_S, tm + kT_E + kk * 8, umma::smem_desc_oct(sKT + kk * 256, kOct, false),
                                        id_s, 1);
#pragma unroll
        for (int kk = 0; kk < kC / 8; ++kk)
          umma::mma_ts<umma::kKindTF32>(tm + kT_O, tm + kT_E + kk * 8, umma::smem_desc(sPB + kk * 256, 256, false),
                                        id_o, kk > 0);
        umma::commit(&bars[3]);
      }
    }
    if (!wait_mma(&bars[3], par)) { ok = false; break; }
    // ---- o = (e^g Z / |q| + O') / sqrt(dk), written token-major to OT (thread:
    // dv row `row`, tokens 16 part ..; a warp writes 32 consecutive floats)
    {
      uint32_t zr[16], orr[16];
      umma::ld16_nowait(tm + lane_base + kT_Z + part * 16, zr);
      umma::ld16_nowait(tm + lane_base + kT_O + part * 16, orr);
      umma::wait_ld();
      float z[16], ov[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        z[e] = __uint_as_float(zr[e]);
        ov[e] = __uint_as_float(orr[e]);
      }
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int t = part * 16 + e;
        OT[t * kHeadDim + row] = fmaf(egv[t] * iqv[t], z[e], ov[e]) * kInvSqrtDk;
      }
    }
    // one barrier: o is in OT and (when gating) the z rows have landed
    if (want_gate) {
      if (!wait_mma(&bars[5], par)) { ok = false; break; }
    } else {
      __syncthreads();
    }
    // ---- the gated RMSNorm over dv, token-major: eight threads per token, each
    // with four groups of 4 dv (group q at 4 (s8 + 8 q)), the sum of squares
    // over the eight by shuffles
    {
      const int t = tid >> 3, s8 = tid & 7;
      const float* orow = OT + t * kHeadDim;
      float4 o4[4];
      float ss = 0.f;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        o4[q] = *reinterpret_cast<const float4*>(orow + 4 * (s8 + 8 * q));
        ss = fmaf(o4[q].x, o4[q].x, ss);
        ss = fmaf(o4[q].y, o4[q].y, ss);
        ss = fmaf(o4[q].z, o4[q].z, ss);
        ss = fmaf(o4[q].w, o4[q].w, ss);
      }
      ss += __shfl_xor_sync(0xffffffffu, ss, 1);
      ss += __shfl_xor_sync(0xffffffffu, ss, 2);
      ss += __shfl_xor_sync(0xffffffffu, ss, 4);
      const float rinv = rsqrtf(ss * (1.0f / kHeadDim) + p.eps);
      if (p.o && t < L) {
        uint16_t* op = p.o + ((size_t)(tc + t) * p.Hv + h) * kHeadDim;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          *reinterpret_cast<uint2*>(op + 4 * (s8 + 8 * q)) =
              make_uint2(pack_bf16(o4[q].x, o4[q].y), pack_bf16(o4[q].z, o4[q].w));
      }
      if (want_gate) {
        // Ogate over the z rows in place ...
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int dv0 = 4 * (s8 + 8 * q);
          uint2* zp = reinterpret_cast<uint2*>(ZS + t * kHeadDim + dv0);
          const uint2 z2 = *zp;
          const float4 g4 = *reinterpret_cast<const float4*>(gam + dv0);
          const float z0 = __uint_as_float(z2.x << 16), z1 = __uint_as_float(z2.x & 0xffff0000u);
          const float z2f = __uint_as_float(z2.y << 16), z3 = __uint_as_float(z2.y & 0xffff0000u);
          *zp = make_uint2(pack_bf16(o4[q].x * rinv * g4.x * silu_tanh(z0), o4[q].y * rinv * g4.y * silu_tanh(z1)),
                           pack_bf16(o4[q].z * rinv * g4.z * silu_tanh(z2f), o4[q].w * rinv * g4.w * silu_tanh(z3)));
        }
      }
    }
    // ... then stored with one tensor copy after the next CTA barrier (the next
    // chunk's first, or the one after the loop), which the rows' writes precede
    umma::fence_proxy_async_smem();
    if (tid == kTmaThread && want_gate) {
      st_tc = tc;
      st_len = L;
    }
    // ---- align mode: after an absolute multiple of the block, the state (tensor
    // memory, updated by this chunk's MMAs) and the conv windows go to a snapshot slot
    if (p.snap_slot) {
      const int done = p0 + (tc + L - t0);
      if (done % p.snap_block == 0) {
        const int js = done / p.snap_block - p0 / p.snap_block - 1;
        const int ss = js < p.max_snaps ? p.snap_slot[(size_t)n * p.max_snaps + js] : -1;
        if (ss >= p.Rs) {
          if (tid == 0 && g == 0) report(p.dev_err, GDN_DEVERR_SLOT);
        } else if (ss >= 0) {
          float* sd = p.state + (((size_t)ss * p.Hv + h) * kHeadDim + row) * kHeadDim + part * 32;
          float v[32];
          umma::ld32(tm + lane_base + kTS_S + part * 32, v);
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4*>(sd + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
          if (own_v) {  // hv has already moved past the next chunk when there is one
            const uint16_t* w = c + 1 < nchunks ? hv_end : hv;
            uint16_t* hp = p.conv_hist + ((size_t)ss * p.CH + gvc) * 3;
            hp[0] = w[0]; hp[1] = w[1]; hp[2] = w[2];
          }
          if (own_qk && g == 0) {
            uint16_t* hp = p.conv_hist + ((size_t)ss * p.CH + gqk) * 3;
            hp[0] = (uint16_t)hqk[0]; hp[1] = (uint16_t)hqk[1]; hp[2] = (uint16_t)hqk[2];
            hp[3] = (uint16_t)(hqk[0] >> 16); hp[4] = (uint16_t)(hqk[1] >> 16); hp[5] = (uint16_t)(hqk[2] >> 16);
          }
        }
      }
    }
  }

  __syncthreads();  // the last chunk's Ogate rows are written
  if (ok && tid == kTmaThread) store_pending();
  if (ok) {
    // ---- final state back to the slot, history to the owners' channels
    float* dst = p.state + (((size_t)slot * p.Hv + h) * kHeadDim + row) * kHeadDim + part * 32;
    {
      float v[32];
      umma::ld32(tm + lane_base + kTS_S + part * 32, v);
#pragma unroll
      for (int i = 0; i < 32; i += 4)
        *reinterpret_cast<float4*>(dst + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
    }
    // history: q and k channels by the group's first CTA, v channels by the head's own
    if (own_v) {  // v history: the head's own CTA
      uint16_t* hp = p.conv_hist + ((size_t)slot * p.CH + gvc) * 3;
      hp[0] = hv[0]; hp[1] = hv[1]; hp[2] = hv[2];
    }
    // q and k history (the same in every CTA of the group): by the group's last
    // CTA to start (its ticket, taken after the old history was read)
    if (*last_of_group && own_qk) {
      uint16_t* hp = p.conv_hist + ((size_t)slot * p.CH + gqk) * 3;
      hp[0] = (uint16_t)hqk[0]; hp[1] = (uint16_t)hqk[1]; hp[2] = (uint16_t)hqk[2];
      hp[3] = (uint16_t)(hqk[0] >> 16); hp[4] = (uint16_t)(hqk[1] >> 16); hp[5] = (uint16_t)(hqk[2] >> 16);
    }
  } else {
    if (tid == 0) report(p.dev_err, GDN_DEVERR_TIMEOUT);
    // give MMAs still in flight a second bounded chance before the memory is freed
    for (int b = 0; b < 7; ++b) mbar_wait_bounded(&bars[b], 0);  // (bounded; phases may not match)
  }
  if (tid == kTmaThread) bulk_wait_all();  // Ogate rows stored
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  if (warp == 0) umma::tmem_dealloc(tm, kTmemCols);
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

// Writes the request indices into order[] longest first (by 64-token chunk
// count, capped at kOrderBuckets - 1; ties in any order), so that the prefill's
// CTAs, dispatched in blockIdx order, start the longest (request, head) chains
// first and the short ones fill in behind them. One CTA: a counting sort.
constexpr int kOrderThreads = 1024, kOrderBuckets = 2 * kOrderThreads;

__global__ void __launch_bounds__(kOrderThreads) prefill_order_kernel(const int32_t* qsl, int N, int32_t* order,
                                                                      int32_t* tickets, int n_tickets) {
  __shared__ int cnt[kOrderBuckets];
  __shared__ int wsum[kOrderThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  auto key = [&](int n) {
    const int len = qsl[n + 1] - qsl[n];
    return len <= 0 ? 0 : min((len + kC - 1) / kC, kOrderBuckets - 1);
  };
  for (int b = tid; b < kOrderBuckets; b += kOrderThreads) cnt[b] = 0;
  for (int i = tid; i < n_tickets; i += kOrderThreads) tickets[i] = 0;  // the prefill's group tickets
  __syncthreads();
  for (int n = tid; n < N; n += kOrderThreads) atomicAdd(&cnt[key(n)], 1);
  __syncthreads();
  // first position of each bucket in descending key order: thread t owns the
  // buckets at descending positions 2t and 2t + 1
  const int b0 = kOrderBuckets - 1 - 2 * tid, b1 = b0 - 1;
  const int c0 = cnt[b0], c1 = cnt[b1];
  int incl = c0 + c1;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = wsum[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += u;
    }
    wsum[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  const int excl = incl - (c0 + c1) + (warp > 0 ? wsum[warp - 1] : 0);
  cnt[b0] = excl;
  cnt[b1] = excl + c0;
  __syncthreads();
  for (int n = tid; n < N; n += kOrderThreads) order[atomicAdd(&cnt[key(n)], 1)] = n;
}

}  // namespace

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

// Schedule scratch of gdn_chunk_prefill_noalloc, for callers that cannot hand
// the library a workspace because they cannot allocate device memory at the
// call site (a host whose device memory is all reserved up front by its own
// pool, with no allocation hook). Fixed size, one per device; it needs no
// clearing (the order kernel writes all N entries and zeroes the N x Hk
// tickets before the prefill reads them), and two such calls in flight at once
// on one device race on it.
static __device__ __align__(256) int32_t g_static_prefill_order[kStaticPrefillMaxSeqs];
static __device__ __align__(256) int32_t g_static_prefill_tickets[kStaticPrefillMaxTickets];

namespace {

// Id of the calling thread's current CUDA context (0 when there is none yet).
// The arrays above get new addresses when the device's context is torn down and
// made again (cudaDeviceReset), so the cached addresses are keyed by it.
unsigned long long current_context_id() {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

}  // namespace

cudaError_t static_prefill_order(int32_t** order, int32_t** tickets) {
  constexpr int kMaxDevices = 64;
  struct Entry {
    unsigned long long ctx;
    int32_t* order;
    int32_t* tickets;
  };
  static std::mutex mu;
  static Entry cache[kMaxDevices] = {};
  int dev = -1;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  Entry& e = cache[dev];
  const unsigned long long ctx = current_context_id();
  if (!e.order || ctx == 0 || ctx != e.ctx) {
    void* po = nullptr;
    void* pt = nullptr;
    if ((err = cudaGetSymbolAddress(&po, g_static_prefill_order)) != cudaSuccess) return err;
    if ((err = cudaGetSymbolAddress(&pt, g_static_prefill_tickets)) != cudaSuccess) return err;
    e.order = static_cast<int32_t*>(po);
    e.tickets = static_cast<int32_t*>(pt);
    e.ctx = current_context_id();  // the lookup above has made the context current
  }
  *order = e.order;
  *tickets = e.tickets;
  return cudaSuccess;
}

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream) {
  if (a.T == 0) return cudaSuccess;  // every request is empty: nothing is read or written
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
  if (!a.order || !a.tickets) return cudaErrorInvalidValue;
  prefill_order_kernel<<<1, kOrderThreads, 0, stream>>>(a.qsl, a.N, a.order, a.tickets, a.N * a.Hk);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  prefill_tc_kernel<<<dim3(a.Hv, a.N, 1), kThreads, kSmemBytes, stream>>>(a, tmx, tmz, tmo);
  return cudaGetLastError();
}

}  // namespace gdn
