/*
 * gdn_oracle.c - plain fp64 CPU oracle of the Gated DeltaNet (GDN) mixer core.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg load this library. The GPU product path never links, loads
 * or calls it, and it shares no code, header, table or constant with the GPU
 * path.
 *
 * Sources, cited by page and section:
 *  [P1] "Qwen3.8-27B: from model structure to vLLM inference data flow"
 *       (ai-learning.gods8.com). Section 01 LAYER-BY-LAYER, operator table of a
 *       GDN layer (L00): the conv row c_t = SiLU(sum_{i=0..3} w_i * QKV0_{t-i}),
 *       q = normalize(q), k = normalize(k); the recurrence row
 *       Sbar = alpha*S_prev, e = v - Sbar*k, S = Sbar + beta*e*k^T, o = S*q/sqrt(dk);
 *       the gate row Ogate = RMSNorm(o) (.) SiLU(Z). Same section
 *       data-structure table: Q/K [T,16,128], V/Z [T,48,128],
 *       S [R,48,128,128] fp32 (3 MiB per sequence per layer), conv history
 *       [R,10240,3] holding 3 past inputs (4 taps with the current one).
 *       Section 03 MEMORY LABS, GDN state lab: the same update written as
 *       S_t = alpha_t S_{t-1} + beta_t (v_t - Sbar_t k_t) k_t^T.
 *       Section 06 TP4: rank r holds GDN QK heads 4r..4r+3 and V heads
 *       12r..12r+11, so value head h reads key head floor(h / 3).
 *       Section 08 EVIDENCE MATRIX: the state is decayed first and the error is
 *       predicted from the decayed state; the GDN output gate is SiLU after
 *       RMSNorm.
 *  [P2] "How Qwen3.8-27B's 64 layers are dispatched in vLLM" (iqilian.com),
 *       step 4: the GDN layer is built with gqa_interleaved_layout=False, read
 *       here as the channel layout [Q heads | K heads | V heads].
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - tap w[c][i] multiplies the input i steps back, x_{t-i} (the index in the
 *    conv row); the history [c][0..K-2] is time-ascending, entry K-2 newest;
 *  - no conv bias; a request without initial state starts from S = 0 and a
 *    zero history (left zero padding);
 *  - normalize(x) = x / sqrt(sum x^2 + 1e-12);
 *  - RMSNorm is taken per head over dv with a gain gamma[dv] shared by heads:
 *    o / sqrt(mean(o^2) + eps) * gamma;
 *  - state index order [slot][h][i][j], i over dv (rows), j over dk, so
 *    (S k)_i = sum_j S[i][j] k_j.
 *
 * All arithmetic is fp64. bf16 inputs arrive as uint16 bit patterns and are
 * widened exactly; states are stored back to the fp32 pool by one rounding.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* SiLU(x) = x * sigmoid(x) [P1 §01, conv row and gate row]. */
static double silu(double x) { return x / (1.0 + exp(-x)); }

/* normalize(x) = x / ||x|| [P1 §01, conv row: q = normalize(q), k = normalize(k)]. */
static void l2_normalize(double *x, int n)
{
    double ss = 0.0;
    for (int i = 0; i < n; ++i) ss += x[i] * x[i];
    double r = 1.0 / sqrt(ss + 1e-12);
    for (int i = 0; i < n; ++i) x[i] *= r;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Causal depthwise conv + SiLU for one channel of one request [P1 §01, conv row]:
 *   y_t = SiLU( sum_{i=0..K-1} w[i] * x_{t-i} ),
 * where inputs before the request's first token come from the K-1 history
 * entries (oldest first), or are zero without a history. x points at the
 * channel's first token, consecutive tokens are `stride` elements apart.
 * hist_new receives the last K-1 inputs of [history, x_0 .. x_{L-1}].
 */
static void conv_channel(int K, int L, const uint16_t *x, int64_t stride, const float *w,
                         const uint16_t *hist_old /* [K-1] or NULL */,
                         double *y, int64_t ystride, uint16_t *hist_new /* [K-1] */)
{
    uint16_t h[16];
    for (int m = 0; m < K - 1; ++m) h[m] = hist_old ? hist_old[m] : 0;
    for (int t = 0; t < L; ++t) {
        double pre = 0.0;
        for (int i = 0; i < K; ++i) {
            int s = t - i; /* time of the input that tap i multiplies */
            uint16_t xi = s >= 0 ? x[(int64_t)s * stride] : h[K - 1 + s];
            pre += (double)w[i] * bf16_to_double(xi);
        }
        y[(int64_t)t * ystride] = silu(pre);
    }
    for (int m = 0; m < K - 1; ++m) {
        int s = L - (K - 1) + m; /* time of history entry m after the request */
        hist_new[m] = s >= 0 ? x[(int64_t)s * stride] : h[K - 1 + s];
    }
}

/*
 * One token of the gated delta rule on one value head [P1 §01 recurrence row;
 * §03 state lab; §08: decay first, then predict from the decayed state]:
 *   Sbar = alpha * S;  e = v - Sbar k;  S = Sbar + beta * e k^T;  o = S q / sqrt(dk).
 * S is [dv][dk] row-major. q and k are used as given (already normalized).
 */
void oracle_delta_rule_step(int dk, int dv, double *S, const double *q, const double *k,
                            const double *v, double alpha, double beta, double *o)
{
    double e[512];
    for (int i = 0; i < dv; ++i)
        for (int j = 0; j < dk; ++j) S[i * dk + j] *= alpha;
    for (int i = 0; i < dv; ++i) {
        double pred = 0.0;
        for (int j = 0; j < dk; ++j) pred += S[i * dk + j] * k[j];
        e[i] = v[i] - pred;
    }
    for (int i = 0; i < dv; ++i)
        for (int j = 0; j < dk; ++j) S[i * dk + j] += beta * e[i] * k[j];
    double scale = 1.0 / sqrt((double)dk);
    for (int i = 0; i < dv; ++i) {
        double r = 0.0;
        for (int j = 0; j < dk; ++j) r += S[i * dk + j] * q[j];
        o[i] = r * scale;
    }
}

/*
 * The recurrence over T tokens of one head, optionally with the q/k L2
 * normalization first (normalize != 0). q, k: [T][dk]; v, o: [T][dv];
 * S: [dv][dk] in/out. Used directly by the closed-form checks, which feed
 * keys straight to the core.
 */
void oracle_delta_rule_seq(int dk, int dv, int T, const double *q, const double *k,
                           const double *v, const double *alpha, const double *beta,
                           double *S, double *o, int normalize)
{
    double qn[512], kn[512];
    for (int t = 0; t < T; ++t) {
        memcpy(qn, q + (int64_t)t * dk, sizeof(double) * dk);
        memcpy(kn, k + (int64_t)t * dk, sizeof(double) * dk);
        if (normalize) {
            l2_normalize(qn, dk);
            l2_normalize(kn, dk);
        }
        oracle_delta_rule_step(dk, dv, S, qn, kn, v + (int64_t)t * dv, alpha[t], beta[t],
                               o + (int64_t)t * dv);
    }
}

/* Gated RMSNorm of one head row [P1 §01 gate row]: out = o / sqrt(mean(o^2)+eps) * gamma * SiLU(z). */
static void gated_rmsnorm_row(int D, const double *o, const double *z, const float *gamma,
                              double eps, double *out)
{
    double ms = 0.0;
    for (int d = 0; d < D; ++d) ms += o[d] * o[d];
    ms /= D;
    double r = 1.0 / sqrt(ms + eps);
    for (int d = 0; d < D; ++d) out[d] = o[d] * r * (double)gamma[d] * silu(z[d]);
}

/* Standalone gated RMSNorm over [T][H][D] bf16 o and z; out is [T][H*D]. */
void oracle_gated_rmsnorm(int T, int H, int D, const uint16_t *o, const uint16_t *z,
                          const float *gamma, double eps, double *out)
{
    double ob[1024], zb[1024];
    for (int64_t r = 0; r < (int64_t)T * H; ++r) {
        for (int d = 0; d < D; ++d) {
            ob[d] = bf16_to_double(o[r * D + d]);
            zb[d] = bf16_to_double(z[r * D + d]);
        }
        gated_rmsnorm_row(D, ob, zb, gamma, eps, out + r * D);
    }
}

/*
 * Standalone varlen conv update [P1 §01 conv row; L00 table, conv history row].
 * x [T][CH] bf16; w [CH][K]; hist_pool [Rs][CH][K-1] bf16, updated in place for
 * every request's slot; y [T][CH] receives SiLU(conv) in fp64. A request with
 * has_init[n] == 0 starts from a zero history; slot_idx[n] < 0 marks padding.
 */
void oracle_conv_update(int CH, int K, const uint16_t *x, const float *w, uint16_t *hist_pool,
                        const int32_t *qsl, const int32_t *slot_idx, const uint8_t *has_init,
                        int N, double *y)
{
    for (int n = 0; n < N; ++n) {
        int slot = slot_idx[n];
        if (slot < 0) continue;
        int t0 = qsl[n], L = qsl[n + 1] - qsl[n];
        int init = has_init ? has_init[n] : 1;
        if (L <= 0) continue; /* no tokens: the slot is left untouched */
        for (int c = 0; c < CH; ++c) {
            uint16_t *h = hist_pool + ((int64_t)slot * CH + c) * (K - 1);
            uint16_t hn[16];
            conv_channel(K, L, x + (int64_t)t0 * CH + c, CH, w + (int64_t)c * K, init ? h : NULL,
                         y + (int64_t)t0 * CH + c, CH, hn);
            memcpy(h, hn, sizeof(uint16_t) * (K - 1));
        }
    }
}

/*
 * The whole mixer core for packed varlen requests, slot gather -> conv+SiLU ->
 * q/k L2 norm -> gated delta rule -> gated RMSNorm -> slot scatter.
 *
 *  qkv0      [T][CH] bf16, channels [Q heads | K heads | V heads], head-major
 *  conv_w    [CH][K] fp32
 *  hist_pool [Rs][CH][K-1] bf16        (in/out)
 *  state     [Rs][Hv][dv][dk] fp32     (in/out)
 *  qsl       [N+1] token offsets; slot_idx [N]; has_init [N] or NULL (all 1)
 *  alpha, beta [T][Hv] fp32;  z [T][Hv][dv] bf16;  gamma [dv] fp32
 *  ckpt_slot [T] or NULL. When given, the state and history after token t are
 *            written to slot ckpt_slot[t] and the live slot is left unchanged
 *            (speculative verify keeps one checkpoint per position).
 *  o [T][Hv][dv], ogate [T][Hv*dv]: fp64 outputs. y [T][CH] or NULL: the fp64
 *            conv outputs (before the L2 norm), for tests.
 *
 * Work is split into independent (request, key head) units: each owns the
 * conv channels of its q head, its k head and its Hv/Hk value heads, so the
 * units touch disjoint data and may run in any order.
 */
void oracle_gdn_forward(int Hk, int Hv, int dk, int dv, int K, const uint16_t *qkv0,
                        const float *conv_w, uint16_t *hist_pool, float *state, int Rs,
                        const int32_t *qsl, const int32_t *slot_idx, const uint8_t *has_init,
                        int N, const float *alpha, const float *beta, const uint16_t *z,
                        const float *gamma, double eps, const int32_t *ckpt_slot,
                        double *o, double *ogate, double *y)
{
    (void)Rs;
    const int G = Hv / Hk;
    const int CH = 2 * Hk * dk + Hv * dv;
    const int64_t head_elems = (int64_t)dv * dk;

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t unit = 0; unit < (int64_t)N * Hk; ++unit) {
        const int n = (int)(unit / Hk), j = (int)(unit % Hk);
        const int slot = slot_idx[n];
        if (slot < 0) continue; /* padding entry */
        const int t0 = qsl[n], L = qsl[n + 1] - qsl[n];
        const int init = has_init ? has_init[n] : 1;
        if (L <= 0) continue;

        /* The unit's channels: q head j, k head j, value heads G*j .. G*j+G-1. */
        const int nch = 2 * dk + G * dv;
        int *chan = (int *)malloc(sizeof(int) * nch);
        for (int c = 0; c < dk; ++c) chan[c] = j * dk + c;
        for (int c = 0; c < dk; ++c) chan[dk + c] = Hk * dk + j * dk + c;
        for (int g = 0; g < G; ++g)
            for (int c = 0; c < dv; ++c) chan[2 * dk + g * dv + c] = 2 * Hk * dk + (G * j + g) * dv + c;

        /* a1 slot gather + a2 conv + SiLU over the request's tokens. The
         * per-token histories are kept so that checkpoints can be written. */
        double *yu = (double *)malloc(sizeof(double) * (size_t)L * nch);
        uint16_t *hist_after = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)nch * (K - 1) *
                                                  (ckpt_slot ? L : 1));
        for (int c = 0; c < nch; ++c) {
            const int gc = chan[c];
            const uint16_t *hold = init ? hist_pool + ((int64_t)slot * CH + gc) * (K - 1) : NULL;
            const uint16_t *xc = qkv0 + (int64_t)t0 * CH + gc;
            conv_channel(K, L, xc, CH, conv_w + (int64_t)gc * K, hold, yu + c, nch,
                         hist_after + (int64_t)c * (K - 1));
            if (ckpt_slot) {
                /* history after each prefix t+1 of the request */
                for (int t = 0; t < L; ++t) {
                    double ydummy;
                    conv_channel(K, t + 1, xc, CH, conv_w + (int64_t)gc * K, hold, &ydummy, 0,
                                 hist_after + ((int64_t)t * nch + c) * (K - 1));
                }
            }
            if (y)
                for (int t = 0; t < L; ++t) y[(int64_t)(t0 + t) * CH + gc] = yu[(int64_t)t * nch + c];
        }

        /* a3 L2 norm of q and k for every token. */
        for (int t = 0; t < L; ++t) {
            l2_normalize(yu + (int64_t)t * nch, dk);
            l2_normalize(yu + (int64_t)t * nch + dk, dk);
        }

        /* a4 gated delta rule per value head, then a5 gated RMSNorm, then a6 scatter. */
        double *S = (double *)malloc(sizeof(double) * head_elems);
        double zb[512];
        for (int g = 0; g < G; ++g) {
            const int h = G * j + g;
            float *Sslot = state + ((int64_t)slot * Hv + h) * head_elems;
            for (int64_t e = 0; e < head_elems; ++e) S[e] = init ? (double)Sslot[e] : 0.0;
            for (int t = 0; t < L; ++t) {
                const int64_t tt = t0 + t;
                const double *yt = yu + (int64_t)t * nch;
                double *ot = o + (tt * Hv + h) * dv;
                oracle_delta_rule_step(dk, dv, S, yt, yt + dk, yt + 2 * dk + g * dv,
                                       (double)alpha[tt * Hv + h], (double)beta[tt * Hv + h], ot);
                for (int d = 0; d < dv; ++d) zb[d] = bf16_to_double(z[(tt * Hv + h) * dv + d]);
                gated_rmsnorm_row(dv, ot, zb, gamma, eps, ogate + (tt * Hv + h) * dv);
                if (ckpt_slot) {
                    float *Sck = state + ((int64_t)ckpt_slot[tt] * Hv + h) * head_elems;
                    for (int64_t e = 0; e < head_elems; ++e) Sck[e] = (float)S[e];
                }
            }
            if (!ckpt_slot)
                for (int64_t e = 0; e < head_elems; ++e) Sslot[e] = (float)S[e];
        }

        /* a6 history scatter: to the live slot, or one checkpoint per token. */
        for (int c = 0; c < nch; ++c) {
            const int gc = chan[c];
            if (ckpt_slot) {
                for (int t = 0; t < L; ++t)
                    memcpy(hist_pool + ((int64_t)ckpt_slot[t0 + t] * CH + gc) * (K - 1),
                           hist_after + ((int64_t)t * nch + c) * (K - 1), sizeof(uint16_t) * (K - 1));
            } else {
                memcpy(hist_pool + ((int64_t)slot * CH + gc) * (K - 1),
                       hist_after + (int64_t)c * (K - 1), sizeof(uint16_t) * (K - 1));
            }
        }
        free(S);
        free(hist_after);
        free(yu);
        free(chan);
    }
}
