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

// Counter slot of a stream: streams get slots in order of first use (wrapping
// after kSchedSlots streams), so launches on one stream share a slot (they run
// one after the other) and launches on different streams use different slots.
int sched_slot(cudaStream_t stream) {
  static std::mutex mu;
  static std::unordered_map<cudaStream_t, int> slots;
  static int next = 0;
  std::lock_guard<std::mutex> lock(mu);
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

cudaError_t launch_stream(const StepArgs& a, cudaStream_t stream) {
  const Layout L(a.G, a.P);
  if (L.stages < 2 || a.P > kMaxPos) return cudaErrorInvalidValue;
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
