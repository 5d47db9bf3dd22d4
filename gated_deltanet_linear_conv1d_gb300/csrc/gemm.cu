// gemm.cu - the bf16 projections around the mixer core (page "Qwen3.8-27B:
// from model structure to vLLM inference data flow", section 01 GDN operator
// table): gdn_in_proj, the rows in front of the conv ([T,5120] -> QKV0
// [T,10240], Z [T,6144] and the raw a, b projections), and gdn_out_proj, the Wo
// row ([T,6144] -> [T,5120]) with the residual add. The conv is fused into the
// mixer kernels that read QKV0 and the gated RMSNorm into the ones that write
// Ogate, so what is left on either side is a plain GEMM:
//
//   out_s[t][n] = sum_k X[t][k] W_s[n][k]  (+ residual_s[t][n]),   s = 1 .. 3 outputs
//
// bf16 operands, fp32 accumulation in tensor memory, bf16 (or fp32) out.
//
// One kernel, warp-specialised (320 threads): warp 0 lane 0 issues TMA copies
// of 64-wide K slices (128-byte rows, 128-byte swizzle) into a 4-stage ring;
// warp 1 owns 512 tensor-memory columns (two 128 x 256 fp32 accumulators) and
// its lane 0 issues four tcgen05.mma kind::f16 (K = 16) per stage; warps 2-9
// drain an accumulator (warp w: lanes 32 (w % 4) .., columns 128 ((w - 2) / 4)
// ..) while the MMAs fill the other one.
//
// Tile shapes:
//  - many tokens: 128 tokens x 256 outputs per tile (A = X, B = W; N = 256
//    MMAs, the widest and the cheapest per flop on this GPU);
//  - at most 256 tokens (a decode batch): the operands swap, A = 128 weight
//    rows, B = all T tokens (N = T rounded up to 16), so that one MMA covers the
//    whole batch and every weight byte is read once.
// CTA pairs: the two CTAs of a pair (a cluster of 2, or the pairs of a larger
// cluster) compute two tiles with the same B operand (two token tiles of one
// weight tile; when swapped, two weight tiles of the one token tile). Each
// loads its own A tile and one half of B into its own shared memory (the pair
// MMA reads B from both), so a CTA pulls 32 KB from L2 per K slice instead of 48 KB (at
// the MMA rate the unpaired kernel would need about 22 TB/s from L2 over the
// GPU). A stage is refilled only when both CTAs' MMAs are done with it: the
// MMA completion arrives on the stage's barrier in both CTAs.
// Schedules:
//  - pair tiles >= SMs / 4: persistent pairs take whole pair tiles in turn;
//  - fewer (the decode batch: 20 pairs of weight tiles for Wo): s =
//    floor(SMs / (2 x pairs)) <= 4 pairs per cluster split the K range. Each CTA
//    writes its fp32 partial tile into its own shared memory (the operand ring
//    is free by then); after a cluster barrier each CTA adds up, over
//    distributed shared memory and in a fixed order (reproducible bits), the
//    partials of its share of its tile's rows, and stores them. No workspace.
// Every wait on a copy or an MMA is bounded: a stalled one sets
// GDN_DEVERR_TIMEOUT and the CTA skips its remaining work.
#include <cuda.h>

#include "device.cuh"
#include "launch.h"
#include "pair.cuh"
#include "umma.cuh"

namespace gdn {

namespace {

constexpr int kBM = 128;  // MMA M: tokens, or weight rows when swapped
constexpr int kBN = 256;  // MMA N at most: weight rows, or tokens when swapped
constexpr int kBK = 64;   // K elements per stage: one 128-byte swizzled row of bf16
constexpr int kStages = 6;
constexpr int kTileA = kBM * 128;        // 16 KB: this CTA's 128 A rows
constexpr int kTileB = (kBN / 2) * 128;  // 16 KB: this CTA's half of the B rows
constexpr int kStageBytes = kTileA + kTileB;
constexpr int kBarOff = kStages * kStageBytes;
// Swapped bf16 epilogue: each half of the epilogue warps stages 16 tokens x 128
// outputs of fp32 here, so that rows of the token-major output leave in 16-byte
// pieces, 256 contiguous bytes per token, instead of one 2-byte store per token
// per thread.
constexpr int kStgTokens = 16;
constexpr int kStgOff = kBarOff + 256;
constexpr int kStgBytes = 2 * kStgTokens * kBM * 4;
constexpr int kSmemBytes = kStgOff + kStgBytes + 1024;  // + alignment slack
// Tiles that are not swapped stage nothing: their launches take less shared memory.
constexpr int kSmemBytesNoStage = kStgOff + 1024;
constexpr int kEpiWarps = 8;
constexpr int kThreads = 32 * (2 + kEpiWarps);
constexpr int kCols = kBN / 2;  // accumulator columns per epilogue thread
constexpr int kMaxSplit = 4;
// Partial tile in shared memory, [output row][output column] fp32 with 4 floats
// of padding per row (16-byte accesses of 8 consecutive rows hit distinct banks):
// not swapped 128 tokens x 256 outputs, swapped up to 256 tokens x 128 outputs.
constexpr int kPadNormal = kBN + 4, kPadSwap = kBM + 4;
static_assert(kBM * kPadNormal * 4 <= kBarOff && kBN * kPadSwap * 4 <= kBarOff, "partial tile overruns the ring");

// The 16 bytes at the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ float4 ld_cluster_v4(const float* local, uint32_t rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(local)), "r"(rank));
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(a)
               : "memory");
  return v;
}

// Output segment and tile of a tile index: tiles run m-tile major, then over
// the segments' n-tiles in order.
struct TileRef {
  int m_t, s, n_t;
};
__device__ __forceinline__ TileRef tile_ref(const GemmArgs& p, int t) {
  TileRef r;
  r.m_t = t / p.tiles_per_m;
  int rest = t - r.m_t * p.tiles_per_m;
  r.s = 0;
  while (r.s + 1 < p.nseg && rest >= p.seg[r.s].tiles) {
    rest -= p.seg[r.s].tiles;
    ++r.s;
  }
  r.n_t = rest;
  return r;
}

// Streaming accesses of the epilogue (the residual and the output pass through
// once): 16-byte load and store with an L2 evict-first policy, so they do not
// push the weights out of L2.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p, uint64_t pol) {
  uint4 v;
  asm volatile("ld.global.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(pol));
  return v;
}
__device__ __forceinline__ void st_stream_v4(void* p, uint4 v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w), "l"(pol)
               : "memory");
}

// 32 accumulator columns of one thread, stored. Not swapped: row `arow` (a
// token), outputs n0 .. n0+31 (8 at a time, 16-byte accesses). Swapped: output
// `arow` (a weight row) for tokens n0 .. n0 + ncols - 1 (one element each; a
// warp's lanes hold consecutive outputs, so each access of a warp is 64
// contiguous bytes). The residual (which may be the output itself) is loaded for
// all 32 columns before the first store, so the loads are in flight together
// rather than each waiting for the previous store.
__device__ __forceinline__ void store32(const GemmSeg& g, bool swap, int arow, int n0, int ncols, const float (&v)[32]) {
  if (!swap) {
    if (g.out_f32) {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (n0 + 4 * j < g.N)
          *reinterpret_cast<float4*>(g.out_f32 + (size_t)arow * g.N + n0 + 4 * j) =
              make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
      return;
    }
    const uint64_t pol = l2_policy_evict_first();
    uint4 r[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      r[j] = (g.residual && n0 + 8 * j < g.N) ? ld_stream_v4(g.residual + (size_t)arow * g.N + n0 + 8 * j, pol)
                                              : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (n0 + 8 * j >= g.N) continue;
      const uint32_t rw[4] = {r[j].x, r[j].y, r[j].z, r[j].w};
      uint32_t w4[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float lo = v[8 * j + 2 * e] + bf16_to_f32(rw[e] & 0xffff);
        const float hi = v[8 * j + 2 * e + 1] + bf16_to_f32(rw[e] >> 16);
        w4[e] = (uint32_t)f32_to_bf16(lo) | ((uint32_t)f32_to_bf16(hi) << 16);
      }
      st_stream_v4(g.out_bf16 + (size_t)arow * g.N + n0 + 8 * j, make_uint4(w4[0], w4[1], w4[2], w4[3]), pol);
    }
    return;
  }
  if (g.out_f32) {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (i < ncols) g.out_f32[(size_t)(n0 + i) * g.N + arow] = v[i];
    return;
  }
  float r[32];
#pragma unroll
  for (int i = 0; i < 32; ++i)
    r[i] = (g.residual && i < ncols) ? bf16_to_f32(g.residual[(size_t)(n0 + i) * g.N + arow]) : 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i)
    if (i < ncols) g.out_bf16[(size_t)(n0 + i) * g.N + arow] = f32_to_bf16(v[i] + r[i]);
}

// The residual of four consecutive outputs (token `row`, outputs n .. n+3), or zeros.
__device__ __forceinline__ uint2 residual4(const GemmSeg& g, int row, int n) {
  return (!g.out_f32 && g.residual) ? *reinterpret_cast<const uint2*>(g.residual + (size_t)row * g.N + n)
                                    : make_uint2(0u, 0u);
}

// Four consecutive outputs (token `row`, outputs n .. n+3, n a multiple of 4) + their
// residual r, loaded by residual4 before any store that might overwrite it.
__device__ __forceinline__ void store4(const GemmSeg& g, int row, int n, float4 v, uint2 r) {
  if (g.out_f32) {
    *reinterpret_cast<float4*>(g.out_f32 + (size_t)row * g.N + n) = v;
    return;
  }
  if (g.residual) {
    v.x += bf16_to_f32(r.x & 0xffff);
    v.y += bf16_to_f32(r.x >> 16);
    v.z += bf16_to_f32(r.y & 0xffff);
    v.w += bf16_to_f32(r.y >> 16);
  }
  *reinterpret_cast<uint2*>(g.out_bf16 + (size_t)row * g.N + n) =
      make_uint2((uint32_t)f32_to_bf16(v.x) | ((uint32_t)f32_to_bf16(v.y) << 16),
                 (uint32_t)f32_to_bf16(v.z) | ((uint32_t)f32_to_bf16(v.w) << 16));
}

// tmx: X [T][K] (box 64 x 128 tokens, or 64 x NT when swapped); tmw0..2: W_s [N_s][K]
// (box 64 x 256 rows, or 64 x 128 when swapped); all 128-byte swizzled.
// grid: split 1: min(tiles, SMs) persistent CTAs; split s > 1: tiles x s CTAs in
// clusters of s along x.
__global__ void __launch_bounds__(kThreads, 1) gemm_bf16_kernel(const __grid_constant__ GemmArgs p,
                                                                  const __grid_constant__ CUtensorMap tmx,
                                                                  const __grid_constant__ CUtensorMap tmw0,
                                                                  const __grid_constant__ CUtensorMap tmw1,
                                                                  const __grid_constant__ CUtensorMap tmw2) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kBarOff);  // [kStages] TMA -> MMA
  uint64_t* empty = full + kStages;                                // [kStages] MMA -> TMA
  uint64_t* tfull = empty + kStages;                               // [2] accumulator complete
  uint64_t* tempty = tfull + 2;                                    // [2] accumulator drained
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  int* flags = reinterpret_cast<int*>(tmem_slot + 1);              // [0] abort

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);   // even CTA: its producer's arrival + both CTAs' bytes
      mbar_init(&empty[s], 1);  // the pair's MMA completion (multicast to both CTAs)
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 2 * kEpiWarps);  // even CTA: both CTAs' epilogue warps
    }
    flags[0] = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc_pair(tmem_slot, 2 * kBN);  // one allocation for the pair: a warp of each CTA takes part
  umma::fence_before_sync();
  __syncthreads();
  cluster_sync_all();  // every CTA's barriers are initialised before the partner copies or arrives on them
  umma::fence_after_sync();
  const uint32_t tm = *tmem_slot;
  volatile int* abort_flag = flags;
  const uint32_t b_rows = p.swap ? (uint32_t)p.nt_tok : (uint32_t)kBN;
  const uint32_t stage_tx = 2u * ((uint32_t)kTileA + (b_rows / 2) * 128u);  // both CTAs' A tile and B half

  // ---- cluster layout: rank = pair member pr + 2 x K part rs. The cluster
  // takes pair tiles first, first + stride, ...; of each, this CTA loads the A
  // tile of its pair member and half pr of the shared B tile over K slices
  // kb_lo .. kb_hi-1, and the pair's even CTA issues M = 256 MMAs over both.
  const int split = p.split;
  const int crank = (int)cluster_ctarank();
  const int pr = crank & 1, rs = crank >> 1;
  const uint16_t pair_mask = (uint16_t)(3u << (2 * rs));
  const uint32_t lead = (uint32_t)(2 * rs);  // the pair's even CTA: it issues the MMAs
  const int csize = 2 * split;
  const int first = (int)blockIdx.x / csize;
  const int stride = split > 1 ? p.pairs : (int)gridDim.x / 2;  // split: one pair tile per cluster
  const int kb_lo = rs * p.KB / split, kb_hi = (rs + 1) * p.KB / split;
  const uint32_t b_half_rows = b_rows / 2;
  // this CTA's tile of pair tile u; valid = false for the missing partner of an odd count
  auto own_tile = [&](int u, bool& valid) -> TileRef {
    if (p.swap) {
      const int w = 2 * u + pr;  // weight tile (over the outputs' tiles in order)
      valid = w < p.tiles_per_m;
      return tile_ref(p, valid ? w : p.tiles_per_m - 1);
    }
    // bands of group_n weight tiles, each walked down all token-tile pairs, so a
    // band's weights stay in L2 while every token tile passes them
    const int mpairs = (p.mt + 1) / 2;
    const int band = u / (mpairs * p.group_n), in_band = u - band * (mpairs * p.group_n);
    const int width = min(p.group_n, p.tiles_per_m - band * p.group_n);
    const int mp = in_band / width, n_idx = band * p.group_n + in_band % width;
    TileRef r = tile_ref(p, n_idx);
    r.m_t = 2 * mp + pr;
    valid = r.m_t < p.mt;
    return r;
  };

  if (warp == 0) {
    // ---- TMA producer
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmx)) : "memory");
      // the B tile is shared by every A tile of its column (all token tiles of a
      // weight tile; when swapped, every weight tile of the tokens): kept in L2.
      // Swapped, the A tiles (weights) are read once: evicted first. Not swapped,
      // the A tiles (tokens) serve the n-tiles of a wave: default priority.
      const uint64_t keep = l2_policy_evict_last(), stream_pol = l2_policy_evict_first();
      const uint64_t a_pol = p.swap ? stream_pol : l2_policy_evict_normal();
      uint32_t gk = 0;
      bool ok = true;
      for (int u = first; ok && u < p.pairs; u += stride) {
        bool valid;
        const TileRef tr = own_tile(u, valid);
        const CUtensorMap* mw = tr.s == 0 ? &tmw0 : (tr.s == 1 ? &tmw1 : &tmw2);
        for (int kb = kb_lo; kb < kb_hi; ++kb, ++gk) {
          const int s = gk % kStages;
          if (gk >= (uint32_t)kStages && !mbar_wait_bounded(&empty[s], ((gk / kStages) - 1) & 1)) {
            ok = false;
            break;
          }
          if (*abort_flag) { ok = false; break; }
          unsigned char* st = smem + s * kStageBytes;
          const uint32_t fb = cluster_addr(&full[s], lead);  // both CTAs' copies count on the even CTA's barrier
          if (pr == 0) mbar_arrive_expect_tx(&full[s], stage_tx);
          if (p.swap) {
            tma_load_2d_pair(st, mw, kb * kBK, tr.n_t * kBM, fb, stream_pol);
            tma_load_2d_pair(st + kTileA, &tmx, kb * kBK, pr * (int)b_half_rows, fb, keep);
          } else {
            tma_load_2d_pair(st, &tmx, kb * kBK, tr.m_t * kBM, fb, a_pol);
            tma_load_2d_pair(st + kTileA, mw, kb * kBK, tr.n_t * kBN + pr * (int)b_half_rows, fb, keep);
          }
        }
      }
      if (!ok) {
        report(p.dev_err, GDN_DEVERR_TIMEOUT);
        *abort_flag = 1;
        // copies still in flight land before the CTA goes on (bounded waits; the
        // even CTA holds the barriers that count them)
        if (pr == 0)
          for (uint32_t j = (gk > (uint32_t)kStages ? gk - kStages : 0); j < gk; ++j)
            mbar_wait_bounded(&full[j % kStages], (j / kStages) & 1);
      }
    }
  } else if (warp == 1) {
    // ---- MMA issuer (the pair's even CTA): one accumulator per tile,
    // alternating between the two; M = 256 over the pair
    if (lane == 0 && pr == 0) {
      const uint32_t idesc = umma::idesc(umma::kBF16, false, false, 2 * kBM, p.swap ? p.nt_tok : kBN);
      uint32_t gk = 0, piece = 0;
      bool ok = true;
      for (int u = first; ok && u < p.pairs; u += stride) {
        const uint32_t b = piece & 1, use = piece >> 1;
        if (piece >= 2 && !mbar_wait_bounded(&tempty[b], (use - 1) & 1)) {
          ok = false;
          break;
        }
        umma::fence_after_sync();
        for (int kb = kb_lo; kb < kb_hi; ++kb, ++gk) {
          const int s = gk % kStages;
          if (!mbar_wait_bounded(&full[s], (gk / kStages) & 1) || *abort_flag) {
            ok = false;
            break;
          }
          umma::fence_after_sync();
          const uint32_t sa = smem_u32(smem + s * kStageBytes), sb = sa + kTileA;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            mma_pair<false>(tm + b * kBN, umma::smem_desc_sw128(sa + kk * 32), umma::smem_desc_sw128(sb + kk * 32), idesc,
                     (kb > kb_lo || kk > 0) ? 1u : 0u);
          commit_pair(&empty[s], pair_mask);  // the stage may be refilled in both CTAs
        }
        if (!ok) break;
        commit_pair(&tfull[b], pair_mask);  // both CTAs' epilogues may read their halves
        ++piece;
      }
      if (!ok) {
        report(p.dev_err, GDN_DEVERR_TIMEOUT);
        *abort_flag = 1;
      }
      // the MMAs issued last have finished before tensor memory is released
      if (piece > 0) mbar_wait_bounded(&tfull[(piece - 1) & 1], ((piece - 1) >> 1) & 1);
    }
  } else if (split == 1) {
    // ---- epilogue (warps 2-9): whole tiles, stored from registers. Once a wait
    // has timed out (abort flag) these warps only skip the work.
    const int q = warp & 3;            // tensor-memory lane quarter
    const int half = (warp - 2) >> 2;  // which 128 of the accumulator's 256 columns
    uint32_t piece = 0;
    for (int u = first; u < p.pairs; u += stride) {
      bool valid;
      const TileRef tr = own_tile(u, valid);
      const GemmSeg& g = p.seg[tr.s];
      const uint32_t b = piece & 1, use = piece >> 1;
      ++piece;
      const uint32_t col0 = b * kBN + half * kCols;
      const uint32_t lane_base = (uint32_t)(32 * q) << 16;
      // not swapped: row = token, columns = outputs c0 ..; swapped: row = output, columns = tokens c0 ..
      const int arow = (p.swap ? tr.n_t : tr.m_t) * kBM + 32 * q + lane;
      const int c0 = p.swap ? half * kCols : tr.n_t * kBN + half * kCols;
      const int ncols = p.swap ? min(kCols, p.T - half * kCols) : kCols;
      const bool rows_ok = valid && (p.swap ? arow < g.N : arow < p.T);
      bool aborted = *abort_flag != 0;
      if (!aborted && !mbar_wait_bounded(&tfull[b], use & 1)) {
        report(p.dev_err, GDN_DEVERR_TIMEOUT);
        *abort_flag = 1;
        aborted = true;
      }
      aborted = __any_sync(0xffffffffu, aborted);  // warp-uniform: the tensor-memory loads are .aligned
      umma::fence_after_sync();
      if (p.swap && g.out_bf16 && valid) {
        // swapped, bf16 out: the four warps of this half (the same loop count, so
        // they pass the same named barriers) stage 16 tokens x 128 outputs at a
        // time; thread i of the half then stores 8 consecutive outputs of a token
        // (with their residual) as one 16-byte piece, two pieces per round
        float* stg = reinterpret_cast<float*>(smem + kStgOff) + half * (kStgTokens * kBM);
        const int hi = tid - 64 - 128 * half;  // 0 .. 127 within the half
        const int row_base = tr.n_t * kBM;
        for (int c = 0; c * kStgTokens < ncols; ++c) {
          if (!aborted) {
            float v[16];
            umma::ld16(tm + lane_base + col0 + kStgTokens * c, v);
#pragma unroll
            for (int i = 0; i < kStgTokens; ++i) stg[i * kBM + 32 * q + lane] = v[i];
          }
          asm volatile("bar.sync %0, 128;" ::"r"(2 + half) : "memory");
#pragma unroll
          for (int m = 0; m < 2; ++m) {
            const int k = hi + 128 * m, t = k >> 4, rc = (k & 15) * 8;
            const int token = c0 + kStgTokens * c + t, n = row_base + rc;
            if (!aborted && t < ncols - kStgTokens * c && n < g.N) {
              const float4 a = *reinterpret_cast<const float4*>(stg + t * kBM + rc);
              const float4 bq = *reinterpret_cast<const float4*>(stg + t * kBM + rc + 4);
              float f[8] = {a.x, a.y, a.z, a.w, bq.x, bq.y, bq.z, bq.w};
              uint16_t* dst = g.out_bf16 + (size_t)token * g.N + n;
              if (g.residual) {
                const uint4 r = *reinterpret_cast<const uint4*>(g.residual + (size_t)token * g.N + n);
                const uint32_t rw[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  f[2 * e] += bf16_to_f32(rw[e] & 0xffff);
                  f[2 * e + 1] += bf16_to_f32(rw[e] >> 16);
                }
              }
              uint32_t w4[4];
#pragma unroll
              for (int e = 0; e < 4; ++e)
                w4[e] = (uint32_t)f32_to_bf16(f[2 * e]) | ((uint32_t)f32_to_bf16(f[2 * e + 1]) << 16);
              *reinterpret_cast<uint4*>(dst) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
            }
          }
          asm volatile("bar.sync %0, 128;" ::"r"(2 + half) : "memory");  // the stage may be refilled
        }
      } else if (!aborted && valid && ncols > 0) {
#pragma unroll 1
        for (int c = 0; c < kCols / 32 && 32 * c < ncols; ++c) {
          float v[32];
          umma::ld32(tm + lane_base + col0 + 32 * c, v);
          if (rows_ok) store32(g, p.swap, arow, c0 + 32 * c, ncols - 32 * c, v);
        }
      }
      umma::fence_before_sync();
      __syncwarp();
      if (lane == 0) arrive_cluster(cluster_addr(&tempty[b], lead));  // the even CTA may refill the accumulator
    }
  }

  if (split > 1) {
    // ---- split K: partial tile -> own shared memory; cluster barrier; each CTA
    // adds up, over the K parts of its pair member, its share of the tile's rows
    // in a fixed order, and stores them. Every thread of every CTA passes both
    // cluster barriers.
    __syncthreads();  // the producer and MMA loops are done with the ring
    bool valid;
    const TileRef tr = own_tile(first, valid);
    const GemmSeg& g = p.seg[tr.s];
    float* part = reinterpret_cast<float*>(smem);
    const int ld = p.swap ? kPadSwap : kPadNormal;
    if (warp >= 2) {
      const int q = warp & 3, half = (warp - 2) >> 2;
      bool aborted = *abort_flag != 0;
      if (!aborted && !mbar_wait_bounded(&tfull[0], 0)) {
        report(p.dev_err, GDN_DEVERR_TIMEOUT);
        *abort_flag = 1;
        aborted = true;
      }
      aborted = __any_sync(0xffffffffu, aborted);
      umma::fence_after_sync();
      const int r = 32 * q + lane;  // accumulator lane: a token (not swapped) or an output (swapped)
      const int ncols = p.swap ? min(kCols, p.T - half * kCols) : kCols;
      if (!aborted && ncols > 0) {
#pragma unroll 1
        for (int c = 0; c < kCols / 32 && 32 * c < ncols; ++c) {
          float v[32];
          umma::ld32(tm + ((uint32_t)(32 * q) << 16) + half * kCols + 32 * c, v);
          const int col = half * kCols + 32 * c;  // accumulator column
          if (!p.swap) {
#pragma unroll
            for (int j = 0; j < 8; ++j)
              *reinterpret_cast<float4*>(part + r * ld + col + 4 * j) =
                  make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) part[(col + i) * ld + r] = v[i];  // [token][output]
          }
        }
      }
    }
    umma::fence_before_sync();
    cluster_sync_all();  // every CTA's partial is in its shared memory
    if (!*abort_flag && valid) {
      const int R = p.swap ? p.T : kBM;        // tile rows (tokens)
      const int C4 = (p.swap ? kBM : kBN) / 4;  // tile columns (outputs) in groups of 4
      const int row_lo = rs * R / split, row_hi = (rs + 1) * R / split;
      const int items = (row_hi - row_lo) * C4;
      // a thread's kItems items (4 outputs each) at a time: the K parts of all of them
      // (distributed shared memory) and their residual are loaded before any sum or
      // store, so the round trips overlap instead of following one another
      constexpr int kItems = 4;
      for (int i0 = tid; i0 < items; i0 += kItems * kThreads) {
        float4 pv[kItems][kMaxSplit];
        uint2 res[kItems];
        int tok[kItems], nn[kItems];
        bool live[kItems];
#pragma unroll
        for (int u = 0; u < kItems; ++u) {
          const int i = i0 + u * kThreads;
          const int ii = i < items ? i : i0;  // an item in range for the loads
          const int rr = row_lo + ii / C4, cc = 4 * (ii % C4);
          tok[u] = p.swap ? rr : tr.m_t * kBM + rr;
          nn[u] = (p.swap ? tr.n_t * kBM : tr.n_t * kBN) + cc;
          live[u] = i < items && tok[u] < p.T && nn[u] < g.N;
          const float* src = part + rr * ld + cc;
#pragma unroll
          for (int q2 = 0; q2 < kMaxSplit; ++q2)
            if (q2 < split) pv[u][q2] = ld_cluster_v4(src, (uint32_t)(pr + 2 * q2));
          res[u] = live[u] ? residual4(g, tok[u], nn[u]) : make_uint2(0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < kItems; ++u) {
          if (!live[u]) continue;
          float4 acc = pv[u][0];  // the parts in rank order: the same bits whichever CTA ran first
#pragma unroll
          for (int q2 = 1; q2 < kMaxSplit; ++q2)
            if (q2 < split) {
              acc.x += pv[u][q2].x; acc.y += pv[u][q2].y; acc.z += pv[u][q2].z; acc.w += pv[u][q2].w;
            }
          store4(g, tok[u], nn[u], acc, res[u]);
        }
      }
    }
  }

  umma::fence_before_sync();
  __syncthreads();
  // no CTA leaves while its partner may still copy into it or arrive on its
  // barriers, or a peer may still read its partial tile
  cluster_sync_all();
  umma::fence_after_sync();
  if (warp == 1) tmem_dealloc_pair(tm, 2 * kBN);
}

// bf16 [rows][cols] tensor map, box 64 columns x box_rows rows, 128-byte swizzle.
bool encode_bf16_sw128(CUtensorMap* m, const void* base, int rows, int cols, int box_rows) {
  const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {kBK, (cuuint32_t)box_rows};
  const cuuint32_t elem[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, elem,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 1;
  return n > 0 ? n : 1;
}

// Clusters of `csize` CTAs of this kernel that fit on the GPU at once.
int gemm_resident_clusters(int csize) {
  return resident_clusters(reinterpret_cast<const void*>(gemm_bf16_kernel), kThreads, kSmemBytes, csize);
}

}  // namespace

cudaError_t launch_gemm(const GemmOperands& o, int32_t* dev_err, cudaStream_t stream) {
  if (o.T == 0) return cudaSuccess;
  if (o.nseg < 1 || o.nseg > 3) return cudaErrorInvalidValue;
  const int sms = num_sms();
  GemmArgs a{};
  a.nseg = o.nseg;
  a.T = o.T;
  a.K = o.K;
  a.KB = (o.K + kBK - 1) / kBK;
  a.swap = o.T <= kBN ? 1 : 0;
  a.nt_tok = (o.T + 15) / 16 * 16;
  a.mt = a.swap ? 1 : (o.T + kBM - 1) / kBM;
  a.tiles_per_m = 0;
  // boxes: the own A tile (128 rows) and one half of the B tile (128 weight rows, or NT / 2 tokens)
  CUtensorMap tmx{}, tmw[3]{};
  if (!encode_bf16_sw128(&tmx, o.x, o.T, o.K, a.swap ? a.nt_tok / 2 : kBM)) return cudaErrorInvalidValue;
  for (int s = 0; s < 3; ++s) {
    const int si = s < o.nseg ? s : 0;  // unused maps repeat the first
    const GemmSegOperands& so = o.seg[si];
    if (!encode_bf16_sw128(&tmw[s], so.w, so.N, o.K, kBM)) return cudaErrorInvalidValue;
    if (s < o.nseg) {
      a.seg[s].out_bf16 = so.out_f32 ? nullptr : static_cast<uint16_t*>(so.out);
      a.seg[s].out_f32 = so.out_f32 ? static_cast<float*>(so.out) : nullptr;
      a.seg[s].residual = so.residual;
      a.seg[s].N = so.N;
      a.seg[s].tiles = (so.N + (a.swap ? kBM : kBN) - 1) / (a.swap ? kBM : kBN);
      a.tiles_per_m += a.seg[s].tiles;
    }
  }
  a.dev_err = dev_err;
  // band width: about 24 MB of weights (256 rows x K bf16 per weight tile)
  a.group_n = (int)((24ll << 20) / ((long long)kBN * o.K * 2));
  if (a.group_n < 1) a.group_n = 1;
  if (a.group_n > a.tiles_per_m) a.group_n = a.tiles_per_m;
  const long long pairs = a.swap ? (a.tiles_per_m + 1) / 2 : (long long)((a.mt + 1) / 2) * a.tiles_per_m;
  if (pairs >= (1LL << 30)) return cudaErrorInvalidValue;
  a.pairs = (int)pairs;
  cudaError_t err = ensure_dynamic_smem(reinterpret_cast<const void*>(gemm_bf16_kernel), kSmemBytes);
  if (err != cudaSuccess) return err;
  // K split over the pairs of a cluster when the pairs alone leave at least half
  // the SMs idle, as far as all the clusters fit on the GPU at once
  int split = (int)(sms / (2 * pairs));
  if (split > kMaxSplit) split = kMaxSplit;
  if (split > a.KB) split = a.KB;
  while (split >= 2 && pairs > gemm_resident_clusters(2 * split)) --split;
  if (split < 2) split = 1;
  a.split = split;
  long long clusters = pairs;
  if (split == 1) {  // persistent pairs: as many as fit at once
    const int fit = gemm_resident_clusters(2);
    const long long cap = fit > 0 ? fit : sms / 2;
    if (clusters > cap) clusters = cap;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(clusters * 2 * split), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = a.swap ? kSmemBytes : kSmemBytesNoStage;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)(2 * split);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemm_bf16_kernel, a, tmx, tmw[0], tmw[1], tmw[2]);
}

}  // namespace gdn
