// conv.cu - gdn_conv_update: varlen causal depthwise conv (4 taps) + SiLU
// with the per-slot history updated in place (page "Qwen3.8-27B: from model
// structure to vLLM inference data flow", section 01, conv row and the L00
// table's conv-history row).
//
// The packed token axis is cut into segments of S tokens (S a power of two
// from 4 to 64, about the mean request length) and a thread walks one segment
// for four adjacent channels, so every token row is read and written as
// coalesced 8-byte words and long requests spread over many threads.
//
// A segment may hold the end of one request, whole requests and the start of
// another. The thread whose segment holds a request's first token is that
// request's owner: it reads the old history, computes the request's first
// max(3, rest of its segment) tokens and writes the new history (the last three
// raw inputs, read back from x when the request is longer than what it
// computed). Every other thread starts a request at token t0 + 3 or later,
// where the window is made of raw inputs only, so the history of a slot is read
// and written by one thread and the in-place update needs no ordering.
//
// Written plainly the kernel is bound by instruction issue, not by HBM (ncu:
// 77 % issue-active at 56 % of DRAM bandwidth), so the window is kept as floats
// (one unpack per new input), SiLU takes one tanh.approx instead of an
// exponential and a division, and pairs are packed with one bf16x2 conversion.
// Then it waited on its loads: each thread now issues the next batch of rows
// before computing the current one, and the register budget is set for six
// 128-thread blocks per SM (five or seven moved fewer bytes per second).
#include "device.cuh"
#include "launch.h"

namespace gdn {

namespace {

constexpr int kThreads = 128;  // 512 channels per block
constexpr int kBatch = 8;      // token rows loaded together by a thread

__device__ __forceinline__ float lo_f(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float hi_f(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// Two floats to a bf16 pair (round to nearest even), a in the low half.
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
  return r;
}

// Largest n in [0, N) with qsl[n] <= t (offsets assumed non-decreasing; stays in
// range whatever they hold).
__device__ __forceinline__ int find_request(const int32_t* qsl, int N, int t) {
  int lo = 0, hi = N - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (qsl[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Four channels c .. c+3 as two packed pairs: word .x = (c, c+1), .y = (c+2, c+3).
struct Quad {
  uint32_t a, b;
};

// One channel: window f0 (oldest) .. f2 (newest) plus the new input x.
__device__ __forceinline__ float conv1(float x, float f2, float f1, float f0, const float4& w) {
  float pre = w.x * x;
  pre = fmaf(w.y, f2, pre);
  pre = fmaf(w.z, f1, pre);
  pre = fmaf(w.w, f0, pre);
  return silu_tanh(pre);
}

// History of two channels (lo, hi) as three words [l0 l1] [l2 h0] [h1 h2] <->
// window words (oldest first) w0 = (l0, h0), w1 = (l1, h1), w2 = (l2, h2).
__device__ __forceinline__ void hist_to_window(const uint32_t* hp, bool init, uint32_t& w0, uint32_t& w1,
                                               uint32_t& w2) {
  const uint32_t h0 = init ? hp[0] : 0u, h1 = init ? hp[1] : 0u, h2 = init ? hp[2] : 0u;
  w0 = (h0 & 0xffffu) | (h1 & 0xffff0000u);
  w1 = (h0 >> 16) | (h2 << 16);
  w2 = (h1 & 0xffffu) | (h2 & 0xffff0000u);
}
__device__ __forceinline__ void window_to_hist(uint32_t* hp, uint32_t w0, uint32_t w1, uint32_t w2) {
  hp[0] = (w0 & 0xffffu) | (w1 << 16);
  hp[1] = (w2 & 0xffffu) | (w0 & 0xffff0000u);
  hp[2] = (w1 >> 16) | (w2 & 0xffff0000u);
}

__global__ void __launch_bounds__(kThreads, 6) conv_kernel(const ConvArgs p, int seg) {
  const int c = 4 * (blockIdx.y * kThreads + threadIdx.x);  // channels c .. c + 3
  const int s0 = blockIdx.x * seg, s1 = min(s0 + seg, p.T);

  // offsets check (one block): monotone, starting at 0 and ending at T
  if (blockIdx.x == 0 && blockIdx.y == 0) {
    for (int n = threadIdx.x; n < p.N; n += kThreads) {
      const int a = p.qsl[n], b = p.qsl[n + 1];
      if (a < 0 || b < a || b > p.T || (n == 0 && a != 0) || (n == p.N - 1 && b != p.T))
        report(p.dev_err, GDN_DEVERR_OFFSETS);
    }
  }
  if (c >= p.CH || s0 >= p.T) return;

  float4 w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) w[i] = *reinterpret_cast<const float4*>(p.conv_w + (size_t)(c + i) * kTaps);
  const uint2* x = reinterpret_cast<const uint2*>(p.x) + (c >> 2);
  uint2* y = reinterpret_cast<uint2*>(p.y) + (c >> 2);
  const size_t ld = (size_t)p.CH >> 2;  // row stride in channel quads

  int n = find_request(p.qsl, p.N, s0);
  int t = s0;
  while (t < s1 && n < p.N) {
    const int t0 = p.qsl[n], t1 = p.qsl[n + 1];
    if (t0 < 0 || t1 < t0 || t1 > p.T || t0 > t) break;  // bad offsets: flagged above
    const int slot = p.slot_idx[n];
    const bool owner = t == t0;
    const int start = owner ? t0 : max(t, t0 + 3);
    const int end = owner ? min(t1, max(s1, t0 + 3)) : min(t1, s1);
    if (slot >= p.Rs) {
      if (owner && c == 0) report(p.dev_err, GDN_DEVERR_SLOT);
    } else if (slot >= 0 && start < end) {
      // windows of raw inputs (oldest first) for the pairs (c, c+1) and (c+2, c+3)
      uint32_t a0, a1, a2, b0, b1, b2;
      uint32_t* hp = nullptr;
      if (owner) {
        hp = reinterpret_cast<uint32_t*>(p.conv_hist + ((size_t)slot * p.CH + c) * (kTaps - 1));
        const bool init = p.has_init ? p.has_init[n] != 0 : true;
        hist_to_window(hp, init, a0, a1, a2);
        hist_to_window(hp + 3, init, b0, b1, b2);
      } else {
        const uint2 v0 = x[(size_t)(start - 3) * ld], v1 = x[(size_t)(start - 2) * ld],
                    v2 = x[(size_t)(start - 1) * ld];
        a0 = v0.x; a1 = v1.x; a2 = v2.x;
        b0 = v0.y; b1 = v1.y; b2 = v2.y;
      }
      // the windows as floats, channel e of the four at f[e][0 (oldest) .. 2]
      float f[4][3];
      {
        const uint32_t wa[3] = {a0, a1, a2}, wb[3] = {b0, b1, b2};
#pragma unroll
        for (int k = 0; k < 3; ++k) {
          f[0][k] = lo_f(wa[k]); f[1][k] = hi_f(wa[k]);
          f[2][k] = lo_f(wb[k]); f[3][k] = hi_f(wb[k]);
        }
      }
      // kBatch tokens at a time, the next batch's loads issued before this batch is
      // computed, so rows stay in flight while the thread computes
      uint2 xv[kBatch];
      {
        const int nt = min(kBatch, end - start);
#pragma unroll
        for (int i = 0; i < kBatch; ++i) xv[i] = i < nt ? x[(size_t)(start + i) * ld] : make_uint2(0u, 0u);
      }
      for (int tb = start; tb < end; tb += kBatch) {
        const int nt = min(kBatch, end - tb);
        const int nt2 = min(kBatch, end - tb - kBatch);  // <= 0 after the last batch
        uint2 xq[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i)
          xq[i] = i < nt2 ? x[(size_t)(tb + kBatch + i) * ld] : make_uint2(0u, 0u);
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
          if (i < nt) {
            const float xn[4] = {lo_f(xv[i].x), hi_f(xv[i].x), lo_f(xv[i].y), hi_f(xv[i].y)};
            float r[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              r[e] = conv1(xn[e], f[e][2], f[e][1], f[e][0], w[e]);
              f[e][0] = f[e][1]; f[e][1] = f[e][2]; f[e][2] = xn[e];
            }
            y[(size_t)(tb + i) * ld] = make_uint2(pack2(r[0], r[1]), pack2(r[2], r[3]));
          }
        }
#pragma unroll
        for (int i = 0; i < kBatch; ++i) xv[i] = xq[i];
      }
      // packed windows back from the floats (exact: they hold bf16 values)
      if (owner) {
        auto bits = [](float v) { return __float_as_uint(v) >> 16; };
        a0 = bits(f[0][0]) | (bits(f[1][0]) << 16); a1 = bits(f[0][1]) | (bits(f[1][1]) << 16);
        a2 = bits(f[0][2]) | (bits(f[1][2]) << 16);
        b0 = bits(f[2][0]) | (bits(f[3][0]) << 16); b1 = bits(f[2][1]) | (bits(f[3][1]) << 16);
        b2 = bits(f[2][2]) | (bits(f[3][2]) << 16);
      }
      if (owner) {
        if (end < t1) {  // longer than computed here (so at least 4 tokens)
          const uint2 v0 = x[(size_t)(t1 - 3) * ld], v1 = x[(size_t)(t1 - 2) * ld], v2 = x[(size_t)(t1 - 1) * ld];
          a0 = v0.x; a1 = v1.x; a2 = v2.x;
          b0 = v0.y; b1 = v1.y; b2 = v2.y;
        }
        window_to_hist(hp, a0, a1, a2);
        window_to_hist(hp + 3, b0, b1, b2);
      }
    }
    if (t1 > s1) break;  // the request runs on past this segment
    t = t1;
    ++n;
  }
}

}  // namespace

cudaError_t launch_conv(const ConvArgs& a, cudaStream_t stream) {
  if (a.T == 0) {  // nothing to compute; still check the offsets
    conv_kernel<<<dim3(1, 1, 1), kThreads, 0, stream>>>(a, 1);
    return cudaGetLastError();
  }
  const int mean = (a.T + a.N - 1) / a.N;
  int seg = 4;
  while (seg < 64 && seg < mean) seg <<= 1;
  const int quads = a.CH / 4;
  dim3 grid((a.T + seg - 1) / seg, (quads + kThreads - 1) / kThreads, 1);
  conv_kernel<<<grid, kThreads, 0, stream>>>(a, seg);
  return cudaGetLastError();
}

}  // namespace gdn
