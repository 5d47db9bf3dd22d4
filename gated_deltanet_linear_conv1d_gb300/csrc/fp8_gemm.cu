// fp8_gemm.cu - gdn_fp8_linear: out[T][N] = dequant(X8) dequant(W8)^T (+ residual)
// with DeepSeek-style block scales (page "Qwen3.8-27B: from model structure to
// vLLM inference data flow", section 04, precision and cache: FP8 E4M3 linear
// weights with one scale per 128 x 128 weight block, activations quantised
// dynamically; here one scale per token and 128-wide group of K).
//
//   out[t][n] = sum_kb xs[t][kb] * ws[n/128][kb] * sum_{k in block kb} X8[t][k] W8[n][k]
//
// Because the scales change every 128 elements of K, the tensor cores compute
// one 128 x 128 x 128 block product at a time into tensor memory (four
// kind::f8f6f4 MMAs of K = 32, exact E4M3 products, fp32 sums) and eight
// "promotion" warps fold each block product into fp32 registers with its scale
// product. Four tensor-memory buffers let the MMAs run up to three blocks ahead
// of the folding.
//
// Schedules, by the number of 128 x 256 output tiles. With at least two waves of
// them (prefill token counts) fp8_gemm_wide_kernel below runs on persistent CTA
// pairs: a pair takes 256 tokens x 256 outputs with M = 256 pair MMAs
// (cta_group::2), each CTA loading its own 128 token rows and half of the W
// tile, and folding and storing its own 128 x 256 outputs (two 256-column
// buffers). With at most one wave (decode batches) the same kernel, unpaired,
// splits each tile's K blocks over a cluster of CTAs, which add their parts
// through the workspace (see the kernel). In between, fp8_gemm_kernel takes
// 128 x 128 tiles: whole tiles blockIdx.x, blockIdx.x + gridDim.x, ... on
// persistent CTAs, stored as bf16 rows directly, unless the last wave of whole
// tiles would leave SMs idle for longer than the exchange below costs. Then the
// K blocks of all tiles, laid end to end, are cut into gridDim.x equal
// contiguous ranges (stream-K), so every SM does the same work; a CTA stores the
// fp32 partial of a tile it covers only in part into its own workspace slice
// (plain coalesced stores), and the CTA that finishes a tile's last piece (an
// atomic ticket, no waiting) adds the pieces in CTA order, stores the bf16 tile
// and resets the ticket.
//
// Warp roles (320 threads): warp 0 lane 0 issues the TMA copies into a 4-stage
// ring (X8 and W8 tiles, 128 B x 128 rows each, 128-byte swizzle), warp 1
// allocates tensor memory and its lane 0 issues the MMAs, warps 2-9 promote and
// store: warp w reads tensor-memory lanes 32 (w % 4) .. +31 (its 32 tokens) and
// columns 64 ((w - 2) / 4) .. +63 (its half of the 128 outputs).
#include <cuda.h>

#include "device.cuh"
#include "launch.h"
#include "pair.cuh"
#include "umma.cuh"

namespace gdn {

namespace {

constexpr int kBM = 128, kBN = 128, kBK = 128;  // kBK: one scale block of K (bytes = elements)
constexpr int kStages = 4;
constexpr int kPromoWarps = 8;
constexpr int kThreads = 32 * (2 + kPromoWarps);
constexpr int kTileBytes = kBM * kBK;            // 16 KB per operand tile
constexpr int kStageBytes = 2 * kTileBytes;      // X tile, then W tile
constexpr int kBarOff = kStages * kStageBytes;   // barriers after the ring
constexpr int kSmemBytes = kBarOff + 256 + 1024; // + barriers + alignment slack
constexpr int kTmemBufs = 4;
constexpr int kTmemCols = kTmemBufs * kBN;       // four partial-product buffers (all 512 columns)
constexpr int kCols = kBN / 2;                   // output columns per promotion thread
constexpr int kScaleAhead = 4;                   // block scales are loaded this many K blocks ahead
constexpr int kPromo = 32 * kPromoWarps;         // promotion threads

// f8f6f4, E4M3 x E4M3, fp32 accumulator, both K-major, M = 128, N = 128
constexpr uint32_t kIdesc = umma::idesc(umma::kE4M3, false, false, kBM, kBN);

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void promo_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// Columns n .. n+7 of one output row: v (+ residual) rounded to bf16, one 16-byte store.
__device__ __forceinline__ void store_row8(uint16_t* out_row, const uint16_t* res_row, int n, int N, const float (&v)[8]) {
  if (n >= N) return;
  float f[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) f[e] = v[e];
  if (res_row) {
    const uint4 r = *reinterpret_cast<const uint4*>(res_row + n);
    const uint32_t rw[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      f[2 * e] += bf16_to_f32(rw[e] & 0xffff);
      f[2 * e + 1] += bf16_to_f32(rw[e] >> 16);
    }
  }
  uint32_t w4[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) w4[e] = (uint32_t)f32_to_bf16(f[2 * e]) | ((uint32_t)f32_to_bf16(f[2 * e + 1]) << 16);
  *reinterpret_cast<uint4*>(out_row + n) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
}

// 64 consecutive outputs n0 .. n0+63 of one row (+ residual) as eight 16-byte stores, the
// residual's eight pieces loaded before the first store (out may be the residual, so a
// load after a store to it could not start before that store).
__device__ __forceinline__ void store_row64(uint16_t* out_row, const uint16_t* res_row, int n0, int N,
                                            const float (&acc)[64]) {
  uint4 r[8];
#pragma unroll
  for (int j = 0; j < 8; ++j)
    r[j] = (res_row && n0 + 8 * j < N) ? *reinterpret_cast<const uint4*>(res_row + n0 + 8 * j)
                                       : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (n0 + 8 * j >= N) continue;
    const uint32_t rw[4] = {r[j].x, r[j].y, r[j].z, r[j].w};
    uint32_t w4[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float lo = acc[8 * j + 2 * e] + bf16_to_f32(rw[e] & 0xffff);
      const float hi = acc[8 * j + 2 * e + 1] + bf16_to_f32(rw[e] >> 16);
      w4[e] = (uint32_t)f32_to_bf16(lo) | ((uint32_t)f32_to_bf16(hi) << 16);
    }
    *reinterpret_cast<uint4*>(out_row + n0 + 8 * j) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
  }
}

__device__ __forceinline__ void arrive_one(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__global__ void __launch_bounds__(kThreads, 1) fp8_gemm_kernel(const Fp8GemmArgs p,
                                                                const __grid_constant__ CUtensorMap tmx,
                                                                const __grid_constant__ CUtensorMap tmw) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kBarOff);  // [kStages] TMA -> MMA
  uint64_t* empty = full + kStages;                                // [kStages] MMA -> TMA
  uint64_t* tfull = empty + kStages;                               // [kTmemBufs] MMA -> promotion
  uint64_t* tempty = tfull + kTmemBufs;                            // [kTmemBufs] promotion -> MMA
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + kTmemBufs);
  int* flags = reinterpret_cast<int*>(tmem_slot + 1);              // [0] abort, [1] last-split ticket

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < kTmemBufs; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], kPromoWarps);  // one arrival per promotion warp
    }
    flags[0] = 0;
    fence_mbar_init();
  }
  if (warp == 1) umma::tmem_alloc(tmem_slot, kTmemCols);
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tm = *tmem_slot;
  volatile int* abort_flag = flags;

  // ---- the pieces this CTA computes: (tile t, K blocks kb0 .. kb1-1)
  const long long G = gridDim.x;
  const long long r0 = p.stream_k ? (long long)blockIdx.x * p.total / G : blockIdx.x;
  const long long r1 = p.stream_k ? (long long)(blockIdx.x + 1) * p.total / G : p.tiles;
  auto next_piece = [&](long long& cur, int& t, int& kb0, int& kb1) -> bool {
    if (p.stream_k) {
      if (cur >= r1) return false;
      t = (int)(cur / p.KB);
      kb0 = (int)(cur - (long long)t * p.KB);
      kb1 = (int)min((long long)p.KB, kb0 + (r1 - cur));
      cur += kb1 - kb0;
    } else {
      if (cur >= r1) return false;
      t = (int)cur;
      kb0 = 0;
      kb1 = p.KB;
      cur += G;
    }
    return true;
  };

  if (warp == 0) {
    // ---- TMA producer
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmx)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmw)) : "memory");
      uint32_t gk = 0;
      bool ok = true;
      long long cur = r0;
      int t, kb0, kb1;
      while (ok && next_piece(cur, t, kb0, kb1)) {
        const int m_t = t / p.nt, n_t = t % p.nt;
        for (int kb = kb0; kb < kb1; ++kb, ++gk) {
          const int s = gk % kStages;
          if (gk >= (uint32_t)kStages && !mbar_wait_bounded(&empty[s], ((gk / kStages) - 1) & 1)) {
            ok = false;
            break;
          }
          if (*abort_flag) { ok = false; break; }
          unsigned char* st = smem + s * kStageBytes;
          mbar_arrive_expect_tx(&full[s], kStageBytes);
          tma_load_2d(st, &tmx, kb * kBK, m_t * kBM, &full[s]);
          tma_load_2d(st + kTileBytes, &tmw, kb * kBK, n_t * kBN, &full[s]);
        }
      }
      if (!ok) {
        report(p.dev_err, GDN_DEVERR_TIMEOUT);
        *abort_flag = 1;
        // copies still in flight land before the CTA leaves: wait (bounded) for the last ones issued
        for (uint32_t j = (gk > (uint32_t)kStages ? gk - kStages : 0); j < gk; ++j)
          mbar_wait_bounded(&full[j % kStages], (j / kStages) & 1);
      }
    }
  } else if (warp == 1) {
    // ---- MMA issuer
    if (lane == 0) {
      uint32_t gk = 0;
      bool ok = true;
      long long cur = r0;
      int t, kb0, kb1;
      while (ok && next_piece(cur, t, kb0, kb1)) {
        for (int kb = kb0; kb < kb1; ++kb, ++gk) {
          const int s = gk % kStages;
          const uint32_t b = gk % kTmemBufs, use = gk / kTmemBufs;
          if (!mbar_wait_bounded(&full[s], (gk / kStages) & 1) ||
              (gk >= (uint32_t)kTmemBufs && !mbar_wait_bounded(&tempty[b], (use - 1) & 1)) || *abort_flag) {
            ok = false;
            break;
          }
          umma::fence_after_sync();
          const uint32_t sx = smem_u32(smem + s * kStageBytes), sw = sx + kTileBytes;
#pragma unroll
          for (int kk = 0; kk < kBK / 32; ++kk)
            umma::mma<umma::kKindF8>(tm + b * kBN, umma::smem_desc_sw128(sx + kk * 32),
                                     umma::smem_desc_sw128(sw + kk * 32), kIdesc, kk > 0);
          umma::commit(&empty[s]);
          umma::commit(&tfull[b]);
        }
      }
      if (!ok) {
        report(p.dev_err, GDN_DEVERR_TIMEOUT);
        *abort_flag = 1;
      }
      // the MMAs issued last have finished before tensor memory is released
      if (gk > 0) mbar_wait_bounded(&tfull[(gk - 1) % kTmemBufs], ((gk - 1) / kTmemBufs) & 1);
    }
  } else {
    // ---- promotion and store (warps 2-9). These warps never leave the item loop
    // early, so the named barriers of the split-K store stay matched; once a wait
    // has timed out (abort flag) they only skip the work.
    const int q = warp & 3;                 // tensor-memory lane quarter
    const int half = (warp - 2) >> 2;       // which 64 of the tile's 128 columns
    const uint32_t lane_base = ((uint32_t)(32 * q) << 16) + half * kCols;
    uint32_t gk = 0;
    long long cur = r0;
    int t, kb0, kb1;
    const int my_first_tile = p.stream_k ? (int)(r0 / p.KB) : -1;
    while (next_piece(cur, t, kb0, kb1)) {
      const int m_t = t / p.nt, n_t = t % p.nt;
      const int row = m_t * kBM + 32 * q + lane;  // this thread's token
      const bool live = row < p.T;
      const float* xs_row = p.xs + (size_t)(live ? row : 0) * p.KB;
      const float* ws_row = p.ws + (size_t)n_t * p.KB;
      float acc[kCols];
#pragma unroll
      for (int i = 0; i < kCols; ++i) acc[i] = 0.f;
      // the block scales, loaded kScaleAhead blocks before they are used so that
      // their latency stays off the folding loop
      float sx[kScaleAhead], sw[kScaleAhead];
#pragma unroll
      for (int i = 0; i < kScaleAhead; ++i) {
        const int kb = min(kb0 + i, kb1 - 1);
        sx[i] = live ? __ldg(xs_row + kb) : 0.f;
        sw[i] = __ldg(ws_row + kb);
      }
      for (int kb = kb0; kb < kb1; ++kb, ++gk) {
        const uint32_t b = gk % kTmemBufs, use = gk / kTmemBufs;
        const float scale = sx[0] * sw[0];
#pragma unroll
        for (int i = 0; i + 1 < kScaleAhead; ++i) {
          sx[i] = sx[i + 1];
          sw[i] = sw[i + 1];
        }
        {
          const int kn = min(kb + kScaleAhead, kb1 - 1);
          sx[kScaleAhead - 1] = live ? __ldg(xs_row + kn) : 0.f;
          sw[kScaleAhead - 1] = __ldg(ws_row + kn);
        }
        if (*abort_flag) continue;
        if (!mbar_wait_bounded(&tfull[b], use & 1)) {
          report(p.dev_err, GDN_DEVERR_TIMEOUT);
          *abort_flag = 1;
          continue;
        }
        umma::fence_after_sync();
        {
          uint32_t v0[32], v1[32];
          umma::ld32_nowait(tm + lane_base + b * kBN, v0);
          umma::ld32_nowait(tm + lane_base + b * kBN + 32, v1);
          umma::wait_ld();
          const float2 sc2 = make_float2(scale, scale);  // packed fp32x2 FMAs
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const float2 a0 = __ffma2_rn(sc2, make_float2(__uint_as_float(v0[i]), __uint_as_float(v0[i + 1])),
                                         make_float2(acc[i], acc[i + 1]));
            acc[i] = a0.x;
            acc[i + 1] = a0.y;
            const float2 a1 = __ffma2_rn(sc2, make_float2(__uint_as_float(v1[i]), __uint_as_float(v1[i + 1])),
                                         make_float2(acc[32 + i], acc[32 + i + 1]));
            acc[32 + i] = a1.x;
            acc[32 + i + 1] = a1.y;
          }
        }
        umma::fence_before_sync();
        __syncwarp();
        if (lane == 0) arrive_one(&tempty[b]);
      }
      const bool aborted = *abort_flag != 0;

      // ---- store: bf16 rows directly, or through the split-K workspace
      const int n0 = n_t * kBN + half * kCols;
      uint16_t* out_row = p.out + (size_t)row * p.N;
      const uint16_t* res_row = p.residual ? p.residual + (size_t)row * p.N : nullptr;
      if (kb0 == 0 && kb1 == p.KB) {  // the whole tile
        if (live && !aborted) store_row64(out_row, res_row, n0, p.N, acc);
      } else {
        // a piece of the tile: partial slice (CTA, 0 for its first tile / 1 for its
        // last), float4 j of promotion thread i at [j][i], so that a warp's 32
        // lanes store 512 contiguous bytes
        const int pid = tid - 64;  // promotion thread index 0 .. kPromo-1
        auto slice = [&](long long cta, int slot) {
          return reinterpret_cast<float4*>(p.partial) + ((size_t)cta * 2 + slot) * (kCols / 4) * kPromo + pid;
        };
        auto owner = [&](long long L) { return ((L + 1) * G - 1) / p.total; };  // the CTA whose range holds L
        const long long tl = (long long)t * p.KB;
        const long long c_first = owner(tl), c_last = owner(tl + p.KB - 1);
        // The tile's first piece (K from 0) ends this CTA's range, so this CTA usually finishes the
        // tile last. If every other piece is already in the workspace (their tickets all taken), it
        // adds them to its own running sum in registers and stores neither its piece nor a ticket.
        if (tid == 2 * 32)
          flags[1] = (!aborted && blockIdx.x == c_first &&
                      ld_acquire(p.tile_cnt + t) == (int)(c_last - c_first)) ? 2 : 0;
        promo_sync();
        if (flags[1] == 0) {
          if (!aborted) {
            float4* dst = slice(blockIdx.x, t == my_first_tile ? 0 : 1);
#pragma unroll
            for (int j = 0; j < kCols / 4; ++j)
              dst[(size_t)j * kPromo] = make_float4(acc[4 * j], acc[4 * j + 1], acc[4 * j + 2], acc[4 * j + 3]);
          }
          __threadfence();
          promo_sync();
          if (tid == 2 * 32)
            flags[1] = aborted ? 0 : (atomicAdd(p.tile_cnt + t, 1) == (int)(c_last - c_first));
          promo_sync();
        }
        if (flags[1] != 0) {  // this CTA finished the tile's last piece: add up the pieces
          __threadfence();
          // every piece in CTA order, the first one taken as it is: the sum does not depend on
          // which CTA finished last or on which of the two ways it got here, so results repeat
          // bit for bit (the first piece is this CTA's own running sum when flags[1] is 2)
          auto piece = [&](long long c2) {
            return slice(c2, t == (int)((c2 * p.total / G) / p.KB) ? 0 : 1);
          };
          if (flags[1] == 1) {
            const float4* src = piece(c_first);
#pragma unroll
            for (int j = 0; j < kCols / 4; ++j) {
              const float4 v = __ldcg(src + (size_t)j * kPromo);
              acc[4 * j] = v.x; acc[4 * j + 1] = v.y; acc[4 * j + 2] = v.z; acc[4 * j + 3] = v.w;
            }
          }
          for (long long c2 = c_first + 1; c2 <= c_last; ++c2) {
            const float4* src = piece(c2);
#pragma unroll
            for (int j = 0; j < kCols / 4; ++j) {
              const float4 v = __ldcg(src + (size_t)j * kPromo);
              acc[4 * j] += v.x; acc[4 * j + 1] += v.y; acc[4 * j + 2] += v.z; acc[4 * j + 3] += v.w;
            }
          }
          if (live) store_row64(out_row, res_row, n0, p.N, acc);
          if (tid == 2 * 32) p.tile_cnt[t] = 0;
        }
        promo_sync();  // flags[1] is rewritten by the next piece
      }
    }
  }

  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  if (warp == 1) umma::tmem_dealloc(tm, kTmemCols);
}

// ---- many tiles: 128 x 256 output tiles, one N = 256 MMA per K step --------
//
// With at least two waves of tiles the kernel below takes 256 outputs per tile
// (two weight-scale blocks): each K step is one N = 256 MMA (its cost is about
// 1.6 times an N = 128 one for twice the work) and each K block's product lands
// in one of two 256-column tensor-memory buffers, so the folding of block kb
// overlaps the MMAs of block kb + 1. The fp32 running sum of the tile stays in
// registers: promotion warp w holds the 128 columns of half (w - 2) / 4 for the
// 32 rows of its tensor-memory lane quarter.
//
// With at most one wave of such tiles (a decode batch: 40 tiles for Wo at 256
// tokens) the same kernel splits K instead (p.split > 1): the grid is tiles x
// split CTAs in clusters of `split`, CTA b takes K blocks [r KB / split,
// (r + 1) KB / split) of tile b / split (r = b % split), and the parts meet
// through the caller's workspace in L2: each part stores its running sums of
// the whole tile with coalesced 16-byte stores, a cluster barrier orders those
// stores before the loads, and part k adds up the parts of row band [k 128 /
// split, (k + 1) 128 / split) in part order (the bits do not depend on timing)
// and stores it.
constexpr int kWN = 256;
constexpr int kWStages = 4;
constexpr int kWStageBytes = kTileBytes + kWN * kBK;   // 16 KB of X rows + 32 KB of W rows
constexpr int kWBarOff = kWStages * kWStageBytes;
// CTA pairs (kPair): a cluster of 2 takes 256 tokens x 256 outputs, the even CTA
// issuing M = 256 pair MMAs; each CTA's stage holds its own 128 X rows and one
// half (128 rows) of the W tile, 32 KB instead of 48, in a 6-deep ring.
constexpr int kPStages = 6;
constexpr int kPStageBytes = 2 * kTileBytes;
static_assert(kPStages * kPStageBytes == kWBarOff, "both rings end where the barriers start");
// Epilogue stage of whole tiles: each promotion warp turns its 32 token rows x
// 128 outputs around 32 outputs at a time through [32 rows][33 floats] (the odd
// stride keeps both the row-wise writes and the piece-wise reads free of bank
// conflicts), so the output leaves in 16-byte pieces, 64 contiguous bytes per
// token, with the pieces' residual loaded ahead, instead of one 16-byte store
// per row per instruction with a dependent residual load before each.
constexpr int kWStgLd = 33;
constexpr int kWStgOff = kWBarOff + 256;
constexpr int kWStgBytes = kPromoWarps * 32 * kWStgLd * 4;
constexpr int kWSmemBytes = kWStgOff + kWStgBytes + 1024;
static_assert(kWSmemBytes <= 227 * 1024, "wide kernel shared memory");
// Launches that split K never store a whole tile: they take the ring (which also
// holds their own band of partial sums) and the barriers only, and leave the rest
// of the SM's storage to L1.
constexpr int kWSplitSmemBytes = kWStgOff + 1024;
constexpr int kWScaleAhead = 2;  // fewer registers than the narrow kernel: the sum takes 128
constexpr uint32_t kWIdesc = umma::idesc(umma::kE4M3, false, false, kBM, kWN);
constexpr uint32_t kPIdesc = umma::idesc(umma::kE4M3, false, false, 2 * kBM, kWN);
constexpr int kMaxSplitW = 4;  // parts of K per tile at most

// kPair = false: one CTA per 128 x 256 tile (persistent, or K split over a
// cluster); kPair = true: persistent CTA pairs (clusters of 2) over 256 x 256
// pair tiles, p.split = 1. Either way each CTA folds and stores its own 128
// token rows x 256 outputs; the pair only shares the W tile's loads: every
// stage both CTAs' copies complete on the even CTA's `full` barrier, the even
// CTA's MMA completion is multicast to both CTAs' `empty` and `tfull`
// barriers, and both CTAs' promotion warps arrive on the even CTA's `tempty`.
template <bool kPair>
__global__ void __launch_bounds__(kThreads, 1) fp8_gemm_wide_kernel(const Fp8GemmArgs p,
                                                                     const __grid_constant__ CUtensorMap tmx,
                                                                     const __grid_constant__ CUtensorMap tmw) {
  constexpr int kStg = kPair ? kPStages : kWStages;
  constexpr int kStgBytes = kPair ? kPStageBytes : kWStageBytes;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kWBarOff);  // [kStg] TMA -> MMA
  uint64_t* empty = full + kStg;                                    // [kStg] MMA -> TMA
  uint64_t* tfull = empty + kStg;                                   // [2] K block's product ready
  uint64_t* tempty = tfull + 2;                                     // [2] K block's product folded
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  int* flags = reinterpret_cast<int*>(tmem_slot + 1);               // [0] abort
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < kStg; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], (kPair ? 2 : 1) * kPromoWarps);
    }
    flags[0] = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    if constexpr (kPair) tmem_alloc_pair(tmem_slot, 512);
    else umma::tmem_alloc(tmem_slot, 512);
  }
  umma::fence_before_sync();
  __syncthreads();
  if constexpr (kPair) cluster_sync_all();  // both CTAs' barriers exist before either copies or arrives on them
  umma::fence_after_sync();
  const uint32_t tm = *tmem_slot;
  volatile int* abort_flag = flags;
  const int nt = (p.N + kWN - 1) / kWN;
  // pair member (0: the even CTA, which issues the MMAs) and the pair's barrier addresses
  const int pr = kPair ? (int)(cluster_ctarank() & 1u) : 0;
  // tiles: 128 x 256 (kPair false) or pair tiles of 256 x 256 (the launcher keeps the count below 2^31)
  const int tiles = kPair ? ((p.mt + 1) / 2) * nt : p.mt * nt;
  // split == 1: persistent CTAs (pairs) take whole tiles first, first + step, ...;
  // split > 1: this CTA takes part `part` of tile blockIdx.x / split, K blocks kb_lo .. kb_hi-1
  const int split = kPair ? 1 : p.split;
  const int part = split > 1 ? (int)(blockIdx.x % (unsigned)split) : 0;
  const int t_first = kPair ? (int)(blockIdx.x >> 1) : (split > 1 ? (int)(blockIdx.x / (unsigned)split) : (int)blockIdx.x);
  const int t_step = kPair ? (int)(gridDim.x >> 1) : (split > 1 ? tiles : (int)gridDim.x);
  const int kb_lo = part * p.KB / split, kb_hi = (part + 1) * p.KB / split;
  // this CTA's 128-row token tile of tile t
  auto m_tile = [&](int t) { return kPair ? 2 * (t / nt) + pr : t / nt; };

  if (warp == 0) {
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmx)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmw)) : "memory");
      uint64_t keep = 0, normal = 0;
      if constexpr (kPair) {
        keep = l2_policy_evict_last();  // W: every token tile of the wave reads it
        normal = l2_policy_evict_normal();
      }
      uint32_t gk = 0;
      bool ok = true;
      for (int t = t_first; t < tiles && ok; t += t_step) {
        const int m_t = m_tile(t), n_t = t % nt;
        for (int kb = kb_lo; kb < kb_hi; ++kb, ++gk) {
          const int s = gk % kStg;
          if ((gk >= (uint32_t)kStg && !mbar_wait_bounded(&empty[s], ((gk / kStg) - 1) & 1)) || *abort_flag) {
            ok = false;
            break;
          }
          unsigned char* st = smem + s * kStgBytes;
          if constexpr (kPair) {
            // both CTAs' copies count on the even CTA's barrier, which expects the bytes of both
            const uint32_t fb = cluster_addr(&full[s], 0);
            if (pr == 0) mbar_arrive_expect_tx(&full[s], 2 * kPStageBytes);
            tma_load_2d_pair(st, &tmx, kb * kBK, m_t * kBM, fb, normal);
            tma_load_2d_pair(st + kTileBytes, &tmw, kb * kBK, n_t * kWN + pr * (kWN / 2), fb, keep);
          } else {
            mbar_arrive_expect_tx(&full[s], kWStageBytes);
            tma_load_2d(st, &tmx, kb * kBK, m_t * kBM, &full[s]);
            tma_load_2d(st + kTileBytes, &tmw, kb * kBK, n_t * kWN, &full[s]);
          }
        }
      }
      if (!ok) {
        report(p.dev_err, GDN_DEVERR_TIMEOUT);
        *abort_flag = 1;
        // copies still in flight land before the CTA goes on (bounded waits; with
        // pairs the even CTA holds the barriers that count them)
        if (!kPair || pr == 0)
          for (uint32_t j = (gk > (uint32_t)kStg ? gk - kStg : 0); j < gk; ++j)
            mbar_wait_bounded(&full[j % kStg], (j / kStg) & 1);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && pr == 0) {
      uint32_t gk = 0;
      bool ok = true;
      for (int t = t_first; t < tiles && ok; t += t_step) {
        for (int kb = kb_lo; kb < kb_hi; ++kb, ++gk) {
          const int s = gk % kStg;
          const uint32_t b = gk & 1, use = gk >> 1;
          if (!mbar_wait_bounded(&full[s], (gk / kStg) & 1) ||
              (gk >= 2 && !mbar_wait_bounded(&tempty[b], (use - 1) & 1)) || *abort_flag) {
            ok = false;
            break;
          }
          umma::fence_after_sync();
          const uint32_t sx = smem_u32(smem + s * kStgBytes), sw = sx + kTileBytes;
          if constexpr (kPair) {
#pragma unroll
            for (int kk = 0; kk < kBK / 32; ++kk)
              mma_pair<true>(tm + b * kWN, umma::smem_desc_sw128(sx + kk * 32), umma::smem_desc_sw128(sw + kk * 32),
                             kPIdesc, kk > 0);
            commit_pair(&empty[s], 3);  // the stage may be refilled in both CTAs
            commit_pair(&tfull[b], 3);  // both CTAs may fold their rows of the block product
          } else {
#pragma unroll
            for (int kk = 0; kk < kBK / 32; ++kk)
              umma::mma<umma::kKindF8>(tm + b * kWN, umma::smem_desc_sw128(sx + kk * 32),
                                       umma::smem_desc_sw128(sw + kk * 32), kWIdesc, kk > 0);
            umma::commit(&empty[s]);
            umma::commit(&tfull[b]);
          }
        }
      }
      if (!ok) {
        report(p.dev_err, GDN_DEVERR_TIMEOUT);
        *abort_flag = 1;
      }
      if (gk > 0) mbar_wait_bounded(&tfull[(gk - 1) & 1], ((gk - 1) >> 1) & 1);
    }
  } else {
    const int q = warp & 3, h = (warp - 2) >> 2;
    const uint32_t lane_off = (uint32_t)(32 * q) << 16;
    const int NB = (p.N + 127) / 128;
    uint32_t gk = 0;
    for (int t = t_first; t < tiles; t += t_step) {
      const int m_t = m_tile(t), n_t = t % nt;
      const int row = m_t * kBM + 32 * q + lane;
      const bool live = row < p.T;
      const int nb = min(2 * n_t + h, NB - 1);  // weight-scale block of this half
      const float* xs_row = p.xs + (size_t)(live ? row : 0) * p.KB;
      const float* ws_row = p.ws + (size_t)nb * p.KB;
      float sx[kWScaleAhead], sw[kWScaleAhead];
#pragma unroll
      for (int i = 0; i < kWScaleAhead; ++i) {
        const int kb = min(kb_lo + i, kb_hi - 1);
        sx[i] = live ? __ldg(xs_row + kb) : 0.f;
        sw[i] = __ldg(ws_row + kb);
      }
      float acc[128];
#pragma unroll
      for (int i = 0; i < 128; ++i) acc[i] = 0.f;
      for (int kb = kb_lo; kb < kb_hi; ++kb, ++gk) {
        const uint32_t b = gk & 1, use = gk >> 1;
        const float scale = sx[0] * sw[0];
#pragma unroll
        for (int i = 0; i + 1 < kWScaleAhead; ++i) {
          sx[i] = sx[i + 1];
          sw[i] = sw[i + 1];
        }
        {
          const int kn = min(kb + kWScaleAhead, kb_hi - 1);
          sx[kWScaleAhead - 1] = live ? __ldg(xs_row + kn) : 0.f;
          sw[kWScaleAhead - 1] = __ldg(ws_row + kn);
        }
        if (__shfl_sync(0xffffffffu, *abort_flag, 0) != 0) continue;
        const bool got = mbar_wait_bounded(&tfull[b], use & 1);
        if (!__all_sync(0xffffffffu, got)) {  // the warp leaves together
          if (lane == 0) report(p.dev_err, GDN_DEVERR_TIMEOUT);
          *abort_flag = 1;
          continue;
        }
        umma::fence_after_sync();
        const uint32_t tp = tm + lane_off + b * kWN + 128 * h;
        // 32 columns per tensor-memory round trip (two loads under one wait), folded
        // with packed fp32x2 FMAs
        const float2 sc2 = make_float2(scale, scale);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t v0[16], v1[16];
          umma::ld16_nowait(tp + 32 * c, v0);
          umma::ld16_nowait(tp + 32 * c + 16, v1);
          umma::wait_ld();
#pragma unroll
          for (int i = 0; i < 16; i += 2) {
            const float2 a0 = __ffma2_rn(sc2, make_float2(__uint_as_float(v0[i]), __uint_as_float(v0[i + 1])),
                                         make_float2(acc[32 * c + i], acc[32 * c + i + 1]));
            acc[32 * c + i] = a0.x;
            acc[32 * c + i + 1] = a0.y;
            const float2 a1 = __ffma2_rn(sc2, make_float2(__uint_as_float(v1[i]), __uint_as_float(v1[i + 1])),
                                         make_float2(acc[32 * c + 16 + i], acc[32 * c + 16 + i + 1]));
            acc[32 * c + 16 + i] = a1.x;
            acc[32 * c + 16 + i + 1] = a1.y;
          }
        }
        umma::fence_before_sync();
        __syncwarp();
        if (lane == 0) {
          if constexpr (kPair) arrive_cluster(cluster_addr(&tempty[b], 0));  // the even CTA may refill the buffer
          else arrive_one(&tempty[b]);
        }
      }
      if (split == 1) {
        // ---- whole tile: out (+ residual) through the warp's stage (see kWStgLd)
        if (__any_sync(0xffffffffu, *abort_flag != 0)) continue;
        float* stg = reinterpret_cast<float*>(smem + kWStgOff) + (warp - 2) * (32 * kWStgLd);
        const int tok0 = m_t * kBM + 32 * q, col_base = n_t * kWN + 128 * h;
#pragma unroll
        for (int st = 0; st < 4; ++st) {
#pragma unroll
          for (int j = 0; j < 32; ++j) stg[lane * kWStgLd + j] = acc[32 * st + j];
          __syncwarp();
          // piece k = lane + 32 m: token tok0 + k / 4, outputs col_base + 32 st + 8 (k % 4) ..
          uint4 res[4];
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const int k = lane + 32 * m, trow = tok0 + (k >> 2), col = col_base + 32 * st + 8 * (k & 3);
            res[m] = (p.residual && trow < p.T && col < p.N)
                         ? *reinterpret_cast<const uint4*>(p.residual + (size_t)trow * p.N + col)
                         : make_uint4(0u, 0u, 0u, 0u);
          }
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const int k = lane + 32 * m, t = k >> 2, cc = 8 * (k & 3);
            const int trow = tok0 + t, col = col_base + 32 * st + cc;
            if (trow < p.T && col < p.N) {
              const uint32_t rw[4] = {res[m].x, res[m].y, res[m].z, res[m].w};
              uint32_t w4[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float lo = stg[t * kWStgLd + cc + 2 * e] + bf16_to_f32(rw[e] & 0xffff);
                const float hi = stg[t * kWStgLd + cc + 2 * e + 1] + bf16_to_f32(rw[e] >> 16);
                w4[e] = (uint32_t)f32_to_bf16(lo) | ((uint32_t)f32_to_bf16(hi) << 16);
              }
              *reinterpret_cast<uint4*>(p.out + (size_t)trow * p.N + col) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
            }
          }
          __syncwarp();  // the stage is rewritten in the next step
        }
        continue;
      }
      if (*abort_flag != 0 || !live) continue;
      if (split > 1) {
        // this part's running sums of the tile: the rows of its own band into
        // shared memory (the operand ring is idle now), [64 column quads][band
        // rows] float4s; the other rows to its slot of the workspace, [64 column
        // quads][128 rows] float4s (a warp's 32 rows are 512 contiguous bytes).
        // Rows past T are never read back.
        const int r = 32 * q + lane;
        const int r0 = part * kBM / split, nrows = (part + 1) * kBM / split - r0;
        if (r >= r0 && r < r0 + nrows) {
          float4* dst = reinterpret_cast<float4*>(smem) + (size_t)32 * h * nrows + (r - r0);
#pragma unroll
          for (int j = 0; j < 32; ++j)
            dst[(size_t)j * nrows] = make_float4(acc[4 * j], acc[4 * j + 1], acc[4 * j + 2], acc[4 * j + 3]);
        } else {
          float4* dst = reinterpret_cast<float4*>(p.partial) + ((size_t)t * split + part) * (kBM * kWN / 4) +
                        (size_t)32 * h * kBM + r;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            __stcg(dst + (size_t)j * kBM, make_float4(acc[4 * j], acc[4 * j + 1], acc[4 * j + 2], acc[4 * j + 3]));
        }
        continue;
      }
    }
    if (split > 1) {
      // ---- once every part of the cluster has stored its sums (the barrier), the
      // promotion threads add up the parts of this part's band of rows, [r0, r1),
      // in part order (its own part from shared memory): item (row r, 8-column
      // group g), consecutive threads on consecutive rows; the loads of three
      // items are issued before any sum
      __threadfence();
      __syncwarp();
      cluster_sync_all();
      const int t = t_first, m_t = m_tile(t), n_t = t % nt;
      const int r0 = part * kBM / split, nrows = (part + 1) * kBM / split - r0;
      const int items = nrows * (kWN / 8);
      const float4* base = reinterpret_cast<const float4*>(p.partial) + (size_t)t * split * (kBM * kWN / 4);
      const int tp = tid - 64;
      const float4* own = reinterpret_cast<const float4*>(smem);
      constexpr int kItems = 3;
      for (int i0 = tp; i0 < items && *abort_flag == 0; i0 += kItems * kPromo) {
        float4 lo[kItems][kMaxSplitW], hi[kItems][kMaxSplitW];
        uint4 res[kItems];
        int rr[kItems], gg[kItems];
#pragma unroll
        for (int u = 0; u < kItems; ++u) {
          const int i = min(i0 + u * kPromo, items - 1);
          gg[u] = i / nrows;
          rr[u] = r0 + i % nrows;
          // the residual is loaded with the parts, before any store (out may be the residual)
          const int row = m_t * kBM + rr[u], col = n_t * kWN + 8 * gg[u];
          res[u] = (p.residual && row < p.T && col < p.N)
                       ? *reinterpret_cast<const uint4*>(p.residual + (size_t)row * p.N + col)
                       : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
          for (int k = 0; k < kMaxSplitW; ++k) {
            if (k == part) {
              const float4* src = own + (size_t)(2 * gg[u]) * nrows + (rr[u] - r0);
              lo[u][k] = src[0];
              hi[u][k] = src[nrows];
            } else if (k < split) {
              const float4* src = base + (size_t)k * (kBM * kWN / 4) + (size_t)(2 * gg[u]) * kBM + rr[u];
              lo[u][k] = __ldcg(src);
              hi[u][k] = __ldcg(src + kBM);
            }
          }
        }
#pragma unroll
        for (int u = 0; u < kItems; ++u) {
          const int row = m_t * kBM + rr[u];
          if (i0 + u * kPromo >= items || row >= p.T) continue;
          float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int k = 0; k < kMaxSplitW; ++k) {
            if (k < split) {
              v[0] += lo[u][k].x; v[1] += lo[u][k].y; v[2] += lo[u][k].z; v[3] += lo[u][k].w;
              v[4] += hi[u][k].x; v[5] += hi[u][k].y; v[6] += hi[u][k].z; v[7] += hi[u][k].w;
            }
          }
          const uint32_t rw[4] = {res[u].x, res[u].y, res[u].z, res[u].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            v[2 * e] += bf16_to_f32(rw[e] & 0xffff);
            v[2 * e + 1] += bf16_to_f32(rw[e] >> 16);
          }
          store_row8(p.out + (size_t)row * p.N, nullptr, n_t * kWN + 8 * gg[u], p.N, v);
        }
      }
    }
  }
  if (split > 1 && warp < 2) {
    __syncwarp();
    cluster_sync_all();  // the producer and MMA warps take part in the cluster barrier too
  }

  umma::fence_before_sync();
  __syncthreads();
  if constexpr (kPair) {
    // neither CTA leaves while its partner may still copy into it, read its
    // shared memory in an MMA, or arrive on its barriers
    cluster_sync_all();
    umma::fence_after_sync();
    if (warp == 1) tmem_dealloc_pair(tm, 512);
  } else {
    umma::fence_after_sync();
    if (warp == 1) umma::tmem_dealloc(tm, 512);
  }
}

bool encode_u8(CUtensorMap* m, const void* base, int rows, int cols, int box_rows = 128) {
  const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols};
  const cuuint32_t box[2] = {kBK, (cuuint32_t)box_rows};
  const cuuint32_t elem[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, elem,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 1;
  return n > 0 ? n : 1;
}

// Clusters of `csize` CTAs of the wide kernel, launched with K split, that fit on
// the GPU at once.
int wide_resident_clusters(int csize) {
  const void* fn = reinterpret_cast<const void*>(fp8_gemm_wide_kernel<false>);
  if (ensure_dynamic_smem(fn, kWSmemBytes) != cudaSuccess) return 0;  // the largest launch of this kernel
  return resident_clusters(fn, kThreads, kWSplitSmemBytes, csize);
}

// CTA pairs of the pair kernel that fit on the GPU at once.
int pair_resident_clusters() {
  const void* fn = reinterpret_cast<const void*>(fp8_gemm_wide_kernel<true>);
  if (ensure_dynamic_smem(fn, kWSmemBytes) != cudaSuccess) return 0;
  return resident_clusters(fn, kThreads, kWSmemBytes, 2);
}

}  // namespace

// Schedules, by the number of 128 x 256 tiles:
//  - at least two waves: the wide kernel, persistent CTA pairs over whole 256 x
//    256 pair tiles (persistent single CTAs if no pair fits);
//  - at most one wave: the wide kernel with K split over clusters of `split`
//    CTAs (split 1: one CTA per tile), as many parts as leave every part at
//    least four K blocks and let all the clusters run at once;
//  - in between: the 128 x 128 kernel, stream-K (equal K-block ranges) when the
//    last wave of whole tiles would leave SMs idle for longer than the exchange
//    of partial tiles costs (320 tiles on 152 SMs: 3 waves of 48 blocks, or
//    102 blocks each and the exchange).
struct Plan8 {
  int kind;  // 0: 128 x 128 kernel, 1: wide persistent, 2: wide, one wave, split K
  int split;
  bool pair;  // kind 1: CTA pairs (grid = 2 x pairs)
  bool stream_k;
  long long tiles, total;
  int grid;
};

// The partial-tile exchange of a stream-K CTA (its partial sums to L2, the last CTA of a tile
// adding them up) costs about as much as this many K blocks of MMAs and folding.
constexpr int kStreamKFixupBlocks = 16;

Plan8 plan_fp8(int T, int N, int K, int sms) {
  Plan8 pl{};
  const int KB = K / kBK;
  const long long wide_tiles = (long long)((T + kBM - 1) / kBM) * ((N + kWN - 1) / kWN);
  if (wide_tiles >= 2LL * sms && wide_tiles < (1LL << 31)) {
    pl.kind = 1;
    pl.split = 1;
    pl.tiles = wide_tiles;
    pl.grid = sms;
    const long long pair_tiles = (long long)((T + 2 * kBM - 1) / (2 * kBM)) * ((N + kWN - 1) / kWN);
    const int pairs = pair_resident_clusters();
    if (pairs > 0) {
      pl.pair = true;
      pl.grid = 2 * (int)(pair_tiles < pairs ? pair_tiles : pairs);
    }
    return pl;
  }
  if (wide_tiles <= sms) {
    int split = (int)(sms / wide_tiles);
    if (split > kMaxSplitW) split = kMaxSplitW;
    if (split > KB / 4) split = KB / 4;
    while (split >= 2 && wide_tiles > wide_resident_clusters(split)) --split;
    if (split < 2) split = 1;
    pl.kind = 2;
    pl.split = split;
    pl.tiles = wide_tiles;
    pl.grid = (int)(wide_tiles * split);
    return pl;
  }
  pl.kind = 0;
  pl.split = 1;
  pl.tiles = (long long)((T + kBM - 1) / kBM) * ((N + kBN - 1) / kBN);
  pl.total = pl.tiles * KB;
  // whole tiles take ceil(tiles / sms) waves of KB blocks each; stream-K takes an equal share of all
  // K blocks per CTA plus the partial-tile exchange (counted as kStreamKFixupBlocks K blocks)
  const long long whole_blocks = (pl.tiles + sms - 1) / sms * KB;
  const long long sk_blocks = (pl.total + sms - 1) / sms + kStreamKFixupBlocks;
  pl.stream_k = pl.total > pl.tiles && sk_blocks < whole_blocks;
  const long long work = pl.stream_k ? pl.total : pl.tiles;
  pl.grid = (int)(work < sms ? work : sms);
  return pl;
}

size_t plan_workspace_bytes(const Plan8& pl) {
  if (pl.kind == 2 && pl.split > 1) return (size_t)pl.tiles * pl.split * kBM * kWN * 4;
  if (pl.kind == 0 && pl.stream_k) return (size_t)pl.grid * 2 * kBM * kBN * 4 + ((size_t)pl.tiles * 4 + 255) / 256 * 256;
  return 0;
}

size_t fp8_gemm_workspace_bytes(int T, int N, int K) { return plan_workspace_bytes(plan_fp8(T, N, K, num_sms())); }

cudaError_t launch_fp8_gemm(const Fp8Operands& o, void* workspace, size_t ws_bytes, int32_t* dev_err,
                            cudaStream_t stream) {
  if (o.T == 0) return cudaSuccess;
  const int sms = num_sms();
  Plan8 pl = plan_fp8(o.T, o.N, o.K, sms);
  const bool room = workspace && ws_bytes >= plan_workspace_bytes(pl);
  Fp8GemmArgs a{};
  a.xs = o.xs;
  a.ws = o.ws;
  a.residual = o.residual;
  a.out = o.out;
  a.dev_err = dev_err;
  a.T = o.T;
  a.N = o.N;
  a.KB = o.K / kBK;
  a.mt = (o.T + kBM - 1) / kBM;
  a.split = 1;
  if (pl.pair) {  // persistent CTA pairs: each CTA loads half (128 rows) of the W tile
    CUtensorMap tmx{}, tmw{};
    if (!encode_u8(&tmx, o.x8, o.T, o.K) || !encode_u8(&tmw, o.w8, o.N, o.K, kWN / 2)) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)pl.grid, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kWSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fp8_gemm_wide_kernel<true>, a, tmx, tmw);
  }
  if (pl.kind != 0) {  // 128 x 256 tiles
    CUtensorMap tmx{}, tmw{};
    if (!encode_u8(&tmx, o.x8, o.T, o.K) || !encode_u8(&tmw, o.w8, o.N, o.K, kWN)) return cudaErrorInvalidValue;
    cudaError_t err = ensure_dynamic_smem(reinterpret_cast<const void*>(fp8_gemm_wide_kernel<false>), kWSmemBytes);
    if (err != cudaSuccess) return err;
    if (pl.kind == 2 && pl.split > 1 && !room) {  // no room for the parts: one CTA per tile
      pl.split = 1;
      pl.grid = (int)pl.tiles;
    }
    if (pl.split == 1) {
      fp8_gemm_wide_kernel<false><<<pl.grid, kThreads, kWSmemBytes, stream>>>(a, tmx, tmw);
      return cudaGetLastError();
    }
    a.split = pl.split;
    a.partial = static_cast<float*>(workspace);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)pl.grid, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kWSplitSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)pl.split;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fp8_gemm_wide_kernel<false>, a, tmx, tmw);
  }
  CUtensorMap tmx{}, tmw{};
  if (!encode_u8(&tmx, o.x8, o.T, o.K) || !encode_u8(&tmw, o.w8, o.N, o.K)) return cudaErrorInvalidValue;
  a.nt = (o.N + kBN - 1) / kBN;
  if (pl.stream_k && !room) {
    pl.stream_k = false;  // no room for the partial tiles: whole tiles only
    pl.grid = (int)(pl.tiles < sms ? pl.tiles : sms);
  }
  a.stream_k = pl.stream_k ? 1 : 0;
  a.tiles = pl.tiles;
  a.total = pl.total;
  if (pl.stream_k) {
    a.partial = static_cast<float*>(workspace);
    a.tile_cnt = reinterpret_cast<int*>(static_cast<unsigned char*>(workspace) + (size_t)pl.grid * 2 * kBM * kBN * 4);
  }
  cudaError_t err = ensure_dynamic_smem(reinterpret_cast<const void*>(fp8_gemm_kernel), kSmemBytes);
  if (err != cudaSuccess) return err;
  fp8_gemm_kernel<<<pl.grid, kThreads, kSmemBytes, stream>>>(a, tmx, tmw);
  return cudaGetLastError();
}

}  // namespace gdn
