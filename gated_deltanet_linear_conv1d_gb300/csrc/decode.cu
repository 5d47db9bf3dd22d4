// decode.cu - the persistent, warp-specialised state-streaming kernel behind
// gdn_decode_step (one token per request, the state updated in place) and
// gdn_spec_verify (P positions per request, the state after every position kept
// in its checkpoint slot).
//
// Math (page "Qwen3.8-27B: from model structure to vLLM inference data flow",
// section 01 GDN operator table; section 08: decay first, then predict from the
// decayed state), per value head h with key head j = h / G and position p:
//   y = SiLU(sum_i w_i x_{t-i});  q = y_q/|y_q|,  k = y_k/|y_k|,  v = y_v
//   e = v - a (S k);  S' = a S + b e k^T;  o = (a (S q) + b e (k . q)) / sqrt(dk)
//   Ogate = o / sqrt(mean(o^2) + eps) * gamma * SiLU(z)
// so each state element is read once and written once per position.
//
// Design. The path is bound by HBM bandwidth: nearly all of its bytes are the
// fp32 state read and written back. The kernel keeps the state stream
// continuous:
//  - one CTA per SM, claiming work units from a device-wide counter (one unit
//    ahead, so the claim's latency stays off the stream) until none is left,
//    so SMs that stream faster take more units and all finish together; a unit
//    is (request n, key head j) with its G = Hv/Hk value heads, so the unit owns
//    the conv channels of q_j, k_j and its value heads outright (the in-place
//    history update needs no cross-CTA ordering). The counter is one of a small
//    static array, chosen per stream, and the last CTA to finish resets it;
//  - a producer warp streams the unit's 2G half-tiles of state (64 rows x 128
//    fp32 = 32 KiB each) through a ring of shared-memory stages with bulk (TMA)
//    copies completing on mbarriers, running ahead of the consumers; it also
//    stages the unit's QKV0, conv history and z segments (double-buffered);
//  - sixteen consumer warps compute the conv of the unit for all P positions
//    and |q|^2, |k|^2, k . q in one reduction pass (q and k are normalised as
//    they are loaded into registers), then each warp takes 4 rows of a
//    half-tile (8 lanes per row): four 16-byte shared loads per lane, then per
//    position the two dot products (S k, S q) reduced over the 8 lanes, the
//    update kept in registers, and four coalesced 16-byte stores per lane
//    straight to HBM; then the gated RMSNorm of all the unit's heads and
//    positions at once. Four consumer barriers per unit; the next unit's slot,
//    alpha and beta are loaded while the current one runs, so the consumers
//    keep pace with the copies and the producer, not the consumers, sets the
//    rate.
// Every wait is bounded: a stalled copy sets GDN_DEVERR_TIMEOUT and the CTA
// leaves instead of hanging.
#include <mutex>
#include <unordered_map>

#include "device.cuh"
#include "launch.h"

namespace gdn {

namespace {

constexpr int kConsumerWarps = 16;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;  // + one producer warp
constexpr int kMaxStages = 6;
constexpr int kMaxPos = 8;
constexpr int kHalfRows = 64;
constexpr int kHalfFloats = kHalfRows * kHeadDim;
constexpr uint32_t kHalfBytes = kHalfFloats * 4;           // 32 KiB
constexpr int kRowsPerWarp = kHalfRows / kConsumerWarps;   // 4: lanes 8r..8r+7 share row r
constexpr float kInvSqrtDk = 0.08838834764831845f;         // 1/sqrt(128)
constexpr int kSmemLimit = 227 * 1024;
constexpr int kSchedSlots = 64;  // unit counters, one per stream in use
constexpr int kIdRing = 4;       // claimed unit ids in flight (two iterations ahead)

// Dynamic shared-memory layout for group size G and P positions (byte offsets,
// 16-byte aligned). The stage ring takes what the rest leaves, up to 6 stages.
struct Layout {
  int stages, stage, x, hist, z, q, k, v, o, red, ab, bars, total;
  __host__ __device__ Layout(int G, int P) {
    const int nseg = 2 + G;  // q, k, G value heads
    int rest = 0;
    x = rest;        rest += 2 * P * nseg * kHeadDim * 2;   // [2][P][nseg*128] bf16
    hist = rest;     rest += 2 * nseg * kHeadDim * 3 * 2;   // [2][nseg*128*3] bf16
    z = rest;        rest += 2 * P * G * kHeadDim * 2;      // [2][P][G*128] bf16
    q = rest;        rest += P * kHeadDim * 4;              // [P][128] fp32
    k = rest;        rest += P * kHeadDim * 4;              // [P][128] fp32
    v = rest;        rest += G * P * kHeadDim * 4;          // [G][P][128] fp32
    o = rest;        rest += G * P * kHeadDim * 4;          // [G][P][128] fp32
    red = rest;      rest += (P * 16 + G * P * 4) * 4;      // [P][16] norm and [G*P][4] RMS partial sums
    ab = rest;       rest += kMaxGroup * kMaxPos * 4 * 4 + kMaxPos * 4;  // [G][P][4] alpha, beta; [P] output slots
    bars = rest;     rest += (2 * kMaxStages + 8) * 8 + 32; // mbarriers + abort flag + claimed unit ids
    stages = (kSmemLimit - rest) / (int)kHalfBytes;
    if (stages > kMaxStages) stages = kMaxStages;
    const int off = stages * (int)kHalfBytes;
    stage = 0;
    x += off; hist += off; z += off; q += off; k += off; v += off; o += off; red += off; ab += off; bars += off;
    total = off + rest;
  }
};

__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void bulk_g2s_nohint(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Slot that receives the state after position p: the live slot (decode) or the
// position's checkpoint slot (speculative verify). -1 when out of range.
__device__ __forceinline__ bool unit_slots_ok(const StepArgs& p, int n) {
  const int slot = p.slot_idx[n];
  if (slot < 0 || slot >= p.Rs) return false;
  if (p.spec_slot)
    for (int q = 0; q < p.P; ++q) {
      const int s = p.spec_slot[n * p.P + q];
      if (s < 0 || s >= p.Rs) return false;
    }
  return true;
}

// Unit counters: [slot][0] = next unit to claim, [slot][1] = CTAs finished.
// Both are zero between launches (the last CTA of a launch resets them).
__device__ int g_unit_counter[kSchedSlots * 2];

// kOne: exactly one position (decode), so the per-position vectors are loaded once per unit.
template <bool kOne>
__global__ void __launch_bounds__(kThreads, 1) stream_kernel(const StepArgs p, const int units, const int sched) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const int G = p.G, P = kOne ? 1 : p.P;
  const Layout L(G, P);
  const int S_N = L.stages;
  float* stage = reinterpret_cast<float*>(smem + L.stage);
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem + L.x);
  uint16_t* hs = reinterpret_cast<uint16_t*>(smem + L.hist);
  uint16_t* zs = reinterpret_cast<uint16_t*>(smem + L.z);
  float* qs = reinterpret_cast<float*>(smem + L.q);
  float* ks = reinterpret_cast<float*>(smem + L.k);
  float* vs = reinterpret_cast<float*>(smem + L.v);
  float* os = reinterpret_cast<float*>(smem + L.o);
  float* red = reinterpret_cast<float*>(smem + L.red);
  float* ab = reinterpret_cast<float*>(smem + L.ab);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + kMaxStages;
  uint64_t* in_full = empty + kMaxStages;
  uint64_t* in_empty = in_full + 2;
  uint64_t* id_full = in_empty + 2;  // [kIdRing] a claimed unit id is in uid[i % kIdRing]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(id_full + kIdRing);
  volatile int* uid = reinterpret_cast<volatile int*>(id_full + kIdRing) + 1;  // [kIdRing], -1: none left
  int* counter = g_unit_counter + 2 * sched;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nseg = 2 + G;
  const int xrow_len = nseg * kHeadDim;  // bf16 per position in the x buffer
  const bool want_z = p.ogate != nullptr;  // z may be NULL when only o is written

  if (tid == 0) {
    for (int s = 0; s < S_N; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&in_full[b], 1);
      mbar_init(&in_empty[b], 1);
    }
    for (int r = 0; r < kIdRing; ++r) mbar_init(&id_full[r], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane != 0) return;
    const uint64_t pol = l2_policy_evict_first();
    int t = 0, kin = 0;
    for (int i = 0; !*abort_flag; ++i) {
      // the unit the consumers claimed for their i-th iteration
      if (!mbar_wait_bounded(&id_full[i % kIdRing], (i / kIdRing) & 1)) { *abort_flag = 1; break; }
      const int u = uid[i % kIdRing];
      if (u < 0) break;
      const int n = u / p.Hk, j = u % p.Hk;
      if (!unit_slots_ok(p, n)) {  // the consumers skip the same unit: an empty hand-over
        const int b = kin & 1;
        if (!mbar_wait_bounded(&in_empty[b], ((kin >> 1) & 1) ^ 1)) { *abort_flag = 1; break; }
        mbar_arrive(&in_full[b]);
        ++kin;
        continue;
      }
      const int slot = p.slot_idx[n];
      const int b = kin & 1;
      if (!mbar_wait_bounded(&in_empty[b], ((kin >> 1) & 1) ^ 1)) { *abort_flag = 1; break; }
      const uint32_t in_bytes = P * (nseg * kHeadDim * 2 + (want_z ? G * kHeadDim * 2 : 0)) + nseg * kHeadDim * 6;
      mbar_arrive_expect_tx(&in_full[b], in_bytes);
      for (int q = 0; q < P; ++q) {
        const uint16_t* xrow = p.qkv0 + (size_t)(n * P + q) * p.CH;
        uint16_t* xb = xs + (b * P + q) * xrow_len;
        bulk_g2s_nohint(xb, xrow + j * kHeadDim, kHeadDim * 2, &in_full[b]);
        bulk_g2s_nohint(xb + kHeadDim, xrow + (p.Hk + j) * kHeadDim, kHeadDim * 2, &in_full[b]);
        bulk_g2s_nohint(xb + 2 * kHeadDim, xrow + (2 * p.Hk + G * j) * kHeadDim, G * kHeadDim * 2, &in_full[b]);
        if (want_z)
          bulk_g2s_nohint(zs + (b * P + q) * G * kHeadDim, p.z + ((size_t)(n * P + q) * p.Hv + G * j) * kHeadDim,
                          G * kHeadDim * 2, &in_full[b]);
      }
      const uint16_t* hrow = p.conv_hist + (size_t)slot * p.CH * 3;
      uint16_t* hb = hs + b * nseg * kHeadDim * 3;
      bulk_g2s(hb, hrow + (size_t)j * kHeadDim * 3, kHeadDim * 6, &in_full[b], pol);
      bulk_g2s(hb + kHeadDim * 3, hrow + (size_t)(p.Hk + j) * kHeadDim * 3, kHeadDim * 6, &in_full[b], pol);
      bulk_g2s(hb + 2 * kHeadDim * 3, hrow + (size_t)(2 * p.Hk + G * j) * kHeadDim * 3, G * kHeadDim * 6,
               &in_full[b], pol);
      ++kin;
      const float* sbase = p.state + ((size_t)slot * p.Hv + G * j) * (kHeadDim * kHeadDim);
      for (int h2 = 0; h2 < 2 * G; ++h2, ++t) {
        const int s = t % S_N;
        if (!mbar_wait_bounded(&empty[s], ((t / S_N) & 1) ^ 1)) { *abort_flag = 1; break; }
        mbar_arrive_expect_tx(&full[s], kHalfBytes);
        const float* src = sbase + (size_t)h2 * kHalfFloats;
        float* dst = stage + s * kHalfFloats;
        bulk_g2s(dst, src, kHalfBytes / 2, &full[s], pol);
        bulk_g2s(dst + kHalfFloats / 2, src + kHalfFloats / 2, kHalfBytes / 2, &full[s], pol);
      }
    }
    if (*abort_flag) {
      report(p.dev_err, GDN_DEVERR_TIMEOUT);
      // let copies already in flight land before the CTA may exit (bounded)
      for (int back = 1; back <= S_N && t - back >= 0; ++back) {
        const int tt = t - back;
        mbar_wait_bounded(&full[tt % S_N], (tt / S_N) & 1);
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  // A consumer whose bounded wait fails marks itself dead: it skips all data
  // work but still passes every barrier, so no thread is left waiting at one.
  const int ctid = tid;  // 0 .. kConsumers-1
  const uint64_t wpol = l2_policy_evict_first();
  float* rms_part = red + P * 16;  // [G*P][4]
  int* out_slot = reinterpret_cast<int*>(ab + kMaxGroup * kMaxPos * 4);  // [P] slot written after position q
  bool dead = false;
  int t = 0, kin = 0;
  // Units are claimed two iterations ahead by consumer thread 0 (uid[i %
  // kIdRing] for iteration i, announced to the producer on id_full), so both
  // the producer and the consumers find the next unit's id already there; the
  // next unit's slot and (threads < G*P) its alpha, beta are loaded one unit
  // ahead.
  auto claim = [&](int i) {
    if (ctid == 0) {
      const int u = atomicAdd(counter, 1);
      uid[i % kIdRing] = u < units ? u : -1;
      mbar_arrive(&id_full[i % kIdRing]);
    }
  };
  int slot_nx = -1, oslot_nx = -1;
  float a_nx = 0.f, b_nx = 0.f;
  auto prefetch = [&](int u) {
    const int n = u / p.Hk, j = u % p.Hk;
    slot_nx = p.slot_idx[n];
    if (p.spec_slot && ctid < P) oslot_nx = p.spec_slot[n * P + ctid];
    if (ctid < G * P) {
      const size_t ai = (size_t)(n * P + ctid % P) * p.Hv + G * j + ctid / P;
      a_nx = p.alpha[ai];
      b_nx = p.beta[ai];
    }
  };
  claim(0);
  claim(1);
  consumer_sync();
  int u_nx = uid[0];
  if (u_nx >= 0) prefetch(u_nx);
  for (int i = 0; u_nx >= 0; ++i) {
    const int u = u_nx, n = u / p.Hk, j = u % p.Hk;
    const int slot = slot_nx, oslot_cur = oslot_nx;
    const float a_cur = a_nx, b_cur = b_nx;
    u_nx = uid[(i + 1) % kIdRing];  // claimed in the previous iteration, visible since its barriers
    if (u_nx >= 0) prefetch(u_nx);
    claim(i + 2);
    const int b = kin & 1;
    const bool skip = slot < 0 || slot >= p.Rs || (p.spec_slot && !unit_slots_ok(p, n));
    if (!skip) {
      if (ctid < G * P) {
        ab[ctid * 4 + 0] = a_cur;  // [g][q] with g = ctid / P, q = ctid % P
        ab[ctid * 4 + 1] = b_cur;
      }
      if (ctid < P) out_slot[ctid] = p.spec_slot ? oslot_cur : slot;
    }
    dead = dead || *abort_flag;
    if (!dead && !mbar_wait_bounded(&in_full[b], (kin >> 1) & 1)) {
      dead = true;
      *abort_flag = 1;
      report(p.dev_err, GDN_DEVERR_TIMEOUT);
    }
    if (skip) {  // a bad or padding slot: the producer handed over nothing
      if (ctid == 0 && slot >= 0) report(p.dev_err, GDN_DEVERR_SLOT);
      consumer_sync();
      if (ctid == 0) mbar_arrive(&in_empty[b]);
      ++kin;
      continue;
    }
    // ---- conv + SiLU of the unit's channels for every position; the history
    // after each position goes to its checkpoint slot (verify), or the final
    // one back to the live slot (decode)
    const uint16_t* hb = hs + b * nseg * kHeadDim * 3;
    for (int cc = ctid; cc < nseg * kHeadDim && !dead; cc += kConsumers) {
      const int seg = cc >> 7, d = cc & 127;
      const int gc = seg == 0 ? j * kHeadDim + d
                   : seg == 1 ? (p.Hk + j) * kHeadDim + d
                              : (2 * p.Hk + G * j + (seg - 2)) * kHeadDim + d;
      const float4 w = __ldg(reinterpret_cast<const float4*>(p.conv_w) + gc);
      uint16_t h0 = hb[cc * 3], h1 = hb[cc * 3 + 1], h2 = hb[cc * 3 + 2];
      for (int q = 0; q < P; ++q) {
        const uint16_t x0 = xs[(b * P + q) * xrow_len + cc];
        float pre = w.x * bf16_to_f32(x0);
        pre = fmaf(w.y, bf16_to_f32(h2), pre);
        pre = fmaf(w.z, bf16_to_f32(h1), pre);
        pre = fmaf(w.w, bf16_to_f32(h0), pre);
        const float y = silu(pre);
        if (seg == 0) qs[q * kHeadDim + d] = y;
        else if (seg == 1) ks[q * kHeadDim + d] = y;
        else vs[((seg - 2) * P + q) * kHeadDim + d] = y;
        h0 = h1;
        h1 = h2;
        h2 = x0;
        if (p.spec_slot) {
          uint16_t* hp = p.conv_hist + ((size_t)p.spec_slot[n * P + q] * p.CH + gc) * 3;
          hp[0] = h0;
          hp[1] = h1;
          hp[2] = h2;
        }
      }
      if (!p.spec_slot) {
        uint16_t* hp = p.conv_hist + ((size_t)slot * p.CH + gc) * 3;
        hp[0] = h0;
        hp[1] = h1;
        hp[2] = h2;
      }
    }
    consumer_sync();
    // ---- |q|^2, |k|^2 and k . q of the raw conv outputs per position in one
    // pass (warps 0-3, a quarter of the channels each); q and k are normalised
    // where they are loaded into registers below
    for (int q = 0; q < P; ++q)
      if (warp < 4) {
        const float xq = qs[q * kHeadDim + warp * 32 + lane], xk = ks[q * kHeadDim + warp * 32 + lane];
        const float sq = warp_sum(xq * xq), sk = warp_sum(xk * xk), skq = warp_sum(xk * xq);
        if (lane == 0) {
          red[q * 16 + warp] = sq;
          red[q * 16 + 4 + warp] = sk;
          red[q * 16 + 8 + warp] = skq;
        }
      }
    consumer_sync();
    // per position: 1/|q|, 1/|k| (L2 norm, eps 1e-12 under the root) and the normalised k . q
    auto norms = [&](int q, float& iq, float& ik, float& kqn) {
      const float* r = red + q * 16;
      iq = rsqrtf(((r[0] + r[1]) + (r[2] + r[3])) + 1e-12f);
      ik = rsqrtf(((r[4] + r[5]) + (r[6] + r[7])) + 1e-12f);
      kqn = ((r[8] + r[9]) + (r[10] + r[11])) * iq * ik;
    };

    // Row layout: the 8 lanes 8r..8r+7 of a warp share one state row; lane
    // c = lane & 7 holds columns 4c + 32m .. 4c + 32m + 3 for m = 0..3, so each
    // 16-byte access of a quarter-warp covers 128 contiguous bytes of one row
    // (conflict-free in shared memory, full sectors in HBM) and the row's dot
    // products need three shuffle levels.
    const int sub = lane >> 3, cl = lane & 7;
    float4 kk1[4], qq1[4];
    float kq1 = 0.f;
    if constexpr (kOne) {
      float iq, ik;
      norms(0, iq, ik, kq1);
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const float4 kr = reinterpret_cast<const float4*>(ks)[cl + 8 * m];
        const float4 qr = reinterpret_cast<const float4*>(qs)[cl + 8 * m];
        kk1[m] = make_float4(kr.x * ik, kr.y * ik, kr.z * ik, kr.w * ik);
        qq1[m] = make_float4(qr.x * iq, qr.y * iq, qr.z * iq, qr.w * iq);
      }
    }
    for (int g = 0; g < G; ++g) {
      const int h = G * j + g;
      for (int hh = 0; hh < 2; ++hh, ++t) {
        const int s = t % S_N;
        dead = dead || *abort_flag;
        if (!dead && !mbar_wait_bounded(&full[s], (t / S_N) & 1)) {
          dead = true;
          *abort_flag = 1;
          report(p.dev_err, GDN_DEVERR_TIMEOUT);
        }
        if (!dead) {
          const int lr = warp * kRowsPerWarp + sub;
          const int ri = hh * kHalfRows + lr;  // row of the head's state
          const float* srow = stage + s * kHalfFloats + lr * kHeadDim;
          float4 sv[4];
#pragma unroll
          for (int m = 0; m < 4; ++m) sv[m] = reinterpret_cast<const float4*>(srow)[cl + 8 * m];
          for (int q = 0; q < P; ++q) {
            const float a = ab[(g * P + q) * 4 + 0], bb = ab[(g * P + q) * 4 + 1];
            float kq;
            float4 kk[4], qq[4];
            if constexpr (kOne) {
              kq = kq1;
#pragma unroll
              for (int m = 0; m < 4; ++m) {
                kk[m] = kk1[m];
                qq[m] = qq1[m];
              }
            } else {
              float iq, ik;
              norms(q, iq, ik, kq);
#pragma unroll
              for (int m = 0; m < 4; ++m) {
                const float4 kr = reinterpret_cast<const float4*>(ks + q * kHeadDim)[cl + 8 * m];
                const float4 qr = reinterpret_cast<const float4*>(qs + q * kHeadDim)[cl + 8 * m];
                kk[m] = make_float4(kr.x * ik, kr.y * ik, kr.z * ik, kr.w * ik);
                qq[m] = make_float4(qr.x * iq, qr.y * iq, qr.z * iq, qr.w * iq);
              }
            }
            float pk = 0.f, pq = 0.f;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              pk = fmaf(sv[m].x, kk[m].x, pk);
              pk = fmaf(sv[m].y, kk[m].y, pk);
              pk = fmaf(sv[m].z, kk[m].z, pk);
              pk = fmaf(sv[m].w, kk[m].w, pk);
              pq = fmaf(sv[m].x, qq[m].x, pq);
              pq = fmaf(sv[m].y, qq[m].y, pq);
              pq = fmaf(sv[m].z, qq[m].z, pq);
              pq = fmaf(sv[m].w, qq[m].w, pq);
            }
#pragma unroll
            for (int x = 1; x < 8; x <<= 1) {
              pk += __shfl_xor_sync(0xffffffffu, pk, x);  // (S k)_i over the row's 8 lanes
              pq += __shfl_xor_sync(0xffffffffu, pq, x);  // (S q)_i
            }
            const float e = vs[(g * P + q) * kHeadDim + ri] - a * pk;  // v - Sbar k
            const float be = bb * e;
            const int oslot = out_slot[q];
            float* grow = p.state + (((size_t)oslot * p.Hv + h) * kHeadDim + ri) * kHeadDim;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              sv[m].x = fmaf(be, kk[m].x, a * sv[m].x);
              sv[m].y = fmaf(be, kk[m].y, a * sv[m].y);
              sv[m].z = fmaf(be, kk[m].z, a * sv[m].z);
              sv[m].w = fmaf(be, kk[m].w, a * sv[m].w);
              st_global_v4_hint(grow + 4 * (cl + 8 * m), sv[m], wpol);
            }
            if (cl == 0) os[(g * P + q) * kHeadDim + ri] = fmaf(be, kq, a * pq) * kInvSqrtDk;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
      }
    }
    consumer_sync();
    // ---- gated RMSNorm of every (head, position) of the unit: thread (gq, i)
    const int GP = G * P;
    for (int r = ctid; r < GP * kHeadDim; r += kConsumers) {  // whole warps: 128 | r's step
      const float oi = os[r];
      const float ss = warp_sum(oi * oi);
      if (lane == 0) rms_part[(r >> 7) * 4 + ((r >> 5) & 3)] = ss;
    }
    consumer_sync();
    for (int r = ctid; r < GP * kHeadDim && !dead; r += kConsumers) {
      const int gq = r >> 7, i = r & 127, g = gq / P, q = gq % P;
      const float* rp = rms_part + gq * 4;
      const float rinv = rsqrtf(((rp[0] + rp[1]) + (rp[2] + rp[3])) * (1.0f / kHeadDim) + p.eps);
      const float oi = os[r];
      const size_t orow = ((size_t)(n * P + q) * p.Hv + G * j + g) * kHeadDim + i;
      if (p.o) p.o[orow] = f32_to_bf16(oi);
      if (p.ogate) {
        const float zz = bf16_to_f32(zs[((b * P + q) * G + g) * kHeadDim + i]);
        p.ogate[orow] = f32_to_bf16(oi * rinv * p.gamma[i] * silu(zz));
      }
    }
    consumer_sync();  // the unit's staged inputs (z above) are no longer read
    if (ctid == 0) mbar_arrive(&in_empty[b]);
    ++kin;
  }
  // the last CTA to finish leaves the counter at zero for the next launch
  consumer_sync();
  if (ctid == 0) {
    __threadfence();
    if (atomicAdd(counter + 1, 1) == (int)gridDim.x - 1) {
      counter[0] = 0;
      counter[1] = 0;
      __threadfence();
    }
  }
}

// ---------------------------------------------------------------------------
// Small decode batches (fewer (request, key head) units than SMs): one
// thread-block cluster per unit, its nsplit CTAs splitting the rows of the
// unit's G value-head states (rows of S are independent given k, q, alpha and
// beta), so the grid covers the SMs even for a single request. Every CTA runs
// the conv of the unit's q and k channels and of the value channels of its own
// rows, takes its state rows straight into registers (8 lanes per row, 16-byte
// loads issued before the conv), updates and stores them, and adds up the
// squares of its rows' outputs per head; the RMSNorm's sums meet over
// distributed shared memory after a cluster barrier. The q/k history is shared
// by the cluster: its rank-0 CTA writes it after that barrier, when every CTA
// has read the old one; the value-channel history belongs to the row owner.
// A second cluster barrier keeps every CTA's partial sums alive until all have
// read them.
constexpr int kMaxSplit = 8;

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The float at the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ float ld_cluster_f32(const float* local, uint32_t rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(local)), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
  return v;
}

__device__ __forceinline__ float4 ld_global_stream(const float* p) {
  return __ldcs(reinterpret_cast<const float4*>(p));
}

// grid: units x nsplit CTAs, clusters of nsplit along x; blockDim >= 256 and >= 8 x G x (128 / nsplit)
__global__ void __launch_bounds__(1024) split_kernel(const StepArgs p, const int nsplit) {
  __shared__ float qs[kHeadDim], ks[kHeadDim];
  __shared__ float vs[kMaxGroup * kHeadDim / 2];  // [row of this CTA], G x rph <= 8 x 64
  __shared__ float os[kMaxGroup * kHeadDim / 2];
  __shared__ float red[12];                        // |q|^2, |k|^2, k.q: partials of 4 warps
  __shared__ float rms[kMaxGroup];                 // this CTA's sum of o^2 per head
  const int G = p.G;
  const int unit = blockIdx.x / nsplit;
  const int part = (int)cluster_ctarank();
  const int n = unit / p.Hk, j = unit % p.Hk;
  const int rph = kHeadDim / nsplit, r0 = part * rph, nrows = G * rph;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // the same slot for every CTA of the cluster: all of them leave here, or none
  const int slot = p.slot_idx[n];
  if (slot < 0) return;  // padding
  if (slot >= p.Rs) {
    if (part == 0 && tid == 0) report(p.dev_err, GDN_DEVERR_SLOT);
    return;
  }
  const uint64_t wpol = l2_policy_evict_first();
  // ---- this thread's state row (8 lanes per row), loaded first so the loads fly during the conv
  const bool has_row = tid < nrows * 8;
  const int rl = tid >> 3, c8 = tid & 7;
  const int g_row = rl / rph, ri = r0 + rl % rph, h_row = G * j + g_row;
  float* grow = p.state + (((size_t)slot * p.Hv + h_row) * kHeadDim + ri) * kHeadDim;
  float4 sv[4];
  if (has_row) {
#pragma unroll
    for (int m = 0; m < 4; ++m) sv[m] = ld_global_stream(grow + 4 * (c8 + 8 * m));
  }
  // ---- conv + SiLU: q/k channels (threads 0-255), the value channels of this CTA's rows
  const uint16_t* xrow = p.qkv0 + (size_t)n * p.CH;
  uint16_t* hrow = p.conv_hist + (size_t)slot * p.CH * 3;
  uint16_t nh[3] = {0, 0, 0};
  int qk_ch = 0;
  if (tid < 2 * kHeadDim) {
    qk_ch = (tid < kHeadDim ? j : p.Hk + j) * kHeadDim + (tid & (kHeadDim - 1));
    const float4 w = __ldg(reinterpret_cast<const float4*>(p.conv_w) + qk_ch);
    const uint16_t h0 = hrow[qk_ch * 3], h1 = hrow[qk_ch * 3 + 1], h2 = hrow[qk_ch * 3 + 2], x0 = xrow[qk_ch];
    float pre = w.x * bf16_to_f32(x0);
    pre = fmaf(w.y, bf16_to_f32(h2), pre);
    pre = fmaf(w.z, bf16_to_f32(h1), pre);
    pre = fmaf(w.w, bf16_to_f32(h0), pre);
    (tid < kHeadDim ? qs : ks)[tid & (kHeadDim - 1)] = silu(pre);
    nh[0] = h1; nh[1] = h2; nh[2] = x0;
  }
  if (tid < nrows) {
    const int vc = (2 * p.Hk + G * j + tid / rph) * kHeadDim + r0 + tid % rph;
    const float4 w = __ldg(reinterpret_cast<const float4*>(p.conv_w) + vc);
    uint16_t* hp = hrow + (size_t)vc * 3;
    const uint16_t h0 = hp[0], h1 = hp[1], h2 = hp[2], x0 = xrow[vc];
    float pre = w.x * bf16_to_f32(x0);
    pre = fmaf(w.y, bf16_to_f32(h2), pre);
    pre = fmaf(w.z, bf16_to_f32(h1), pre);
    pre = fmaf(w.w, bf16_to_f32(h0), pre);
    vs[tid] = silu(pre);
    hp[0] = h1;  // the value channel's history: read and written by this thread only
    hp[1] = h2;
    hp[2] = x0;
  }
  __syncthreads();
  if (warp < 4) {
    const float xq = qs[warp * 32 + lane], xk = ks[warp * 32 + lane];
    const float sq = warp_sum(xq * xq), sk = warp_sum(xk * xk), skq = warp_sum(xk * xq);
    if (lane == 0) {
      red[warp] = sq;
      red[4 + warp] = sk;
      red[8 + warp] = skq;
    }
  }
  __syncthreads();
  const float iq = rsqrtf(((red[0] + red[1]) + (red[2] + red[3])) + 1e-12f);
  const float ik = rsqrtf(((red[4] + red[5]) + (red[6] + red[7])) + 1e-12f);
  const float kq = ((red[8] + red[9]) + (red[10] + red[11])) * iq * ik;
  // ---- the row update (the same arithmetic as the streaming kernel)
  if (has_row) {
    const float a = p.alpha[(size_t)n * p.Hv + h_row], bb = p.beta[(size_t)n * p.Hv + h_row];
    float pk = 0.f, pq = 0.f;
    float4 kk[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const float4 kr = reinterpret_cast<const float4*>(ks)[c8 + 8 * m];
      const float4 qr = reinterpret_cast<const float4*>(qs)[c8 + 8 * m];
      kk[m] = make_float4(kr.x * ik, kr.y * ik, kr.z * ik, kr.w * ik);
      const float4 qq = make_float4(qr.x * iq, qr.y * iq, qr.z * iq, qr.w * iq);
      pk = fmaf(sv[m].x, kk[m].x, pk);
      pk = fmaf(sv[m].y, kk[m].y, pk);
      pk = fmaf(sv[m].z, kk[m].z, pk);
      pk = fmaf(sv[m].w, kk[m].w, pk);
      pq = fmaf(sv[m].x, qq.x, pq);
      pq = fmaf(sv[m].y, qq.y, pq);
      pq = fmaf(sv[m].z, qq.z, pq);
      pq = fmaf(sv[m].w, qq.w, pq);
    }
#pragma unroll
    for (int x = 1; x < 8; x <<= 1) {
      pk += __shfl_xor_sync(0xffffffffu, pk, x);
      pq += __shfl_xor_sync(0xffffffffu, pq, x);
    }
    const float e = vs[rl] - a * pk;
    const float be = bb * e;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      sv[m].x = fmaf(be, kk[m].x, a * sv[m].x);
      sv[m].y = fmaf(be, kk[m].y, a * sv[m].y);
      sv[m].z = fmaf(be, kk[m].z, a * sv[m].z);
      sv[m].w = fmaf(be, kk[m].w, a * sv[m].w);
      st_global_v4_hint(grow + 4 * (c8 + 8 * m), sv[m], wpol);
    }
    if (c8 == 0) os[rl] = fmaf(be, kq, a * pq) * kInvSqrtDk;
  }
  __syncthreads();
  if (tid < G) {  // this CTA's part of each head's sum of squares
    float ss = 0.f;
    for (int r = 0; r < rph; ++r) ss = fmaf(os[tid * rph + r], os[tid * rph + r], ss);
    rms[tid] = ss;
  }
  cluster_sync_all();  // partial sums published; every CTA of the cluster has read the old history
  if (part == 0 && tid < 2 * kHeadDim) {
    uint16_t* hp = hrow + (size_t)qk_ch * 3;
    hp[0] = nh[0];
    hp[1] = nh[1];
    hp[2] = nh[2];
  }
  if (tid < nrows) {
    const int g = tid / rph, i = r0 + tid % rph, h = G * j + g;
    float ss = 0.f;
    for (int c = 0; c < nsplit; ++c) ss += ld_cluster_f32(&rms[g], (uint32_t)c);
    const float rinv = rsqrtf(ss * (1.0f / kHeadDim) + p.eps);
    const float oi = os[tid];
    const size_t orow = ((size_t)n * p.Hv + h) * kHeadDim + i;
    if (p.o) p.o[orow] = f32_to_bf16(oi);
    if (p.ogate) p.ogate[orow] = f32_to_bf16(oi * rinv * p.gamma[i] * silu(bf16_to_f32(p.z[orow])));
  }
  cluster_sync_all();  // no CTA leaves while a peer may still read its partial sums
}

// Counter slot of a stream: streams get slots in order of first use (wrapping
// after kSchedSlots streams), so launches on one stream share a slot (they run
// one after the other) and launches on different streams use different slots.
// The per-thread default stream is one handle for every thread but a different
// stream in each, so each calling thread gets its own slot for it.
int sched_slot(cudaStream_t stream) {
  static std::mutex mu;
  static std::unordered_map<cudaStream_t, int> slots;
  static int next = 0;
  thread_local int per_thread_slot = -1;
  std::lock_guard<std::mutex> lock(mu);
  if (stream == cudaStreamPerThread) {
    if (per_thread_slot < 0) {
      per_thread_slot = next;
      next = (next + 1) % kSchedSlots;
    }
    return per_thread_slot;
  }
  auto it = slots.find(stream);
  if (it != slots.end()) return it->second;
  const int s = next;
  next = (next + 1) % kSchedSlots;
  slots.emplace(stream, s);
  return s;
}

int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev < 64 && cached[dev]) return cached[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev < 64) cached[dev] = n;
  return n;
}

}  // namespace

bool stream_supported(int G, int P) { return P >= 1 && P <= kMaxPos && Layout(G, P).stages >= 2; }

// Launch shape of the row-split kernel for nsplit CTAs per unit.
void split_config(const StepArgs& a, int nsplit, cudaLaunchConfig_t* cfg, cudaLaunchAttribute* attr) {
  const int rows = a.G * (kHeadDim / nsplit);
  const int threads = rows * 8 > 256 ? rows * 8 : 256;
  *cfg = {};
  cfg->gridDim = dim3((unsigned)(a.N * a.Hk * nsplit), 1, 1);
  cfg->blockDim = dim3((unsigned)threads, 1, 1);
  cfg->dynamicSmemBytes = 0;
  attr->id = cudaLaunchAttributeClusterDimension;
  attr->val.clusterDim.x = (unsigned)nsplit;
  attr->val.clusterDim.y = 1;
  attr->val.clusterDim.z = 1;
  cfg->attrs = attr;
  cfg->numAttrs = 1;
}

// Clusters of the row-split kernel that fit on the GPU at once.
int split_clusters_resident(const StepArgs& a, int nsplit) {
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr;
  split_config(a, nsplit, &cfg, &attr);
  return resident_clusters(reinterpret_cast<const void*>(split_kernel), (int)cfg.blockDim.x, cfg.dynamicSmemBytes,
                           nsplit);
}

// Rows of a unit split over nsplit CTAs when the units alone would leave SMs
// idle (decode only): the smallest power of two that covers the SMs, at least
// G (so a CTA holds at most 128 state rows, 8 lanes each), at most 8. The split
// is taken only when all the clusters fit on the GPU at once (one wave); with
// more than that, the persistent kernel streams the units faster (measured: 8
// requests at 16/48 heads, 512 CTAs of 768 threads, 25.8 us split against 13.8
// us persistent). 1: no split.
int split_factor(const StepArgs& a, int sms) {
  const int units = a.N * a.Hk;
  if (a.P != 1 || a.spec_slot != nullptr || units >= sms) return 1;
  int s = 2;
  while (s < kMaxSplit && (s < a.G || units * s < sms)) s *= 2;
  return units <= split_clusters_resident(a, s) ? s : 1;
}

cudaError_t launch_split(const StepArgs& a, int nsplit, cudaStream_t stream) {
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr;
  split_config(a, nsplit, &cfg, &attr);
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, split_kernel, a, nsplit);
}

cudaError_t launch_stream(const StepArgs& a, cudaStream_t stream) {
  const Layout L(a.G, a.P);
  if (L.stages < 2 || a.P > kMaxPos) return cudaErrorInvalidValue;
  {
    const int sms = sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    const int nsplit = split_factor(a, sms);
    if (nsplit > 1) return launch_split(a, nsplit, stream);
  }
  const bool one = a.P == 1 && a.spec_slot == nullptr;
  const void* fn = one ? reinterpret_cast<const void*>(&stream_kernel<true>)
                       : reinterpret_cast<const void*>(&stream_kernel<false>);
  cudaError_t err = ensure_dynamic_smem(fn, L.total);
  if (err != cudaSuccess) return err;
  const int units = a.N * a.Hk;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const int grid = units < sms ? units : sms;
  const int sched = sched_slot(stream);
  if (one) stream_kernel<true><<<grid, kThreads, L.total, stream>>>(a, units, sched);
  else stream_kernel<false><<<grid, kThreads, L.total, stream>>>(a, units, sched);
  return cudaGetLastError();
}

}  // namespace gdn
