/*
 * gdn.h - C ABI of libgdn, the Gated DeltaNet (GDN) mixer core for one GB300
 * (sm_103a).
 *
 * The mixer core is the chain of the GDN operator table on the page
 * "Qwen3.8-27B: from model structure to vLLM inference data flow"
 * (ai-learning.gods8.com), section 01 LAYER-BY-LAYER, GDN layer L00:
 *
 *   c_t  = SiLU( sum_{i=0..3} w_i (.) QKV0_{t-i} )      causal depthwise conv, 4 taps
 *   q    = normalize(q),  k = normalize(k)              per key head (dk = 128)
 *   Sbar = alpha S_prev;  e = v - Sbar k;  S = Sbar + beta e k^T;  o = S q / sqrt(dk)
 *   Ogate = RMSNorm(o) (.) SiLU(Z)                      per value head (dv = 128)
 *
 * with the shapes of that section's L00 data-structure table: packed QKV0
 * [T, 10240] = [Q 16x128 | K 16x128 | V 48x128], Z [T, 48, 128], the recurrent
 * state S [R, 48, 128, 128] fp32 (3 MiB per sequence per layer) and the conv
 * history [R, 10240, 3] (3 past inputs; 4 taps with the current one). Value
 * head h reads key head floor(h / (Hv / Hk)) (section 06, TP4 head split).
 * Requests are packed along the token axis and split by query_start_loc
 * (section 01, "vLLM can pack several requests into [T, 5120];
 * query_start_loc / seq_lens separate them"), and each request owns one slot
 * of the state and conv-history caches.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every pointer argument is DEVICE memory owned by the caller, unless its
 *   comment says otherwise. libgdn allocates nothing and keeps no state
 *   besides per-device function attributes set on first use.
 * - bf16 tensors are passed as uint16_t bit patterns (IEEE bfloat16).
 * - Layouts are dense and row-major in the order of the bracketed shapes:
 *     qkv0 / x   [T][CH]          CH = 2*Hk*dk + Hv*dv, channels [Q | K | V],
 *                                 head-major inside each part
 *     conv_w     [CH][K]          conv_w[c][i] multiplies the input i steps back
 *     conv_hist  [Rs][CH][K-1]    time-ascending: entry K-2 is the newest input
 *     state      [Rs][Hv][dv][dk] fp32; row i (over dv) gives (S k)_i = sum_j S[i][j] k_j
 *     alpha,beta [T][Hv]          fp32 (the per-token gates, given directly)
 *     z, o       [T][Hv][dv]      bf16
 *     ogate      [T][Hv*dv]       bf16
 *     gamma      [dv]             fp32, shared by all heads
 * - Every call is asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *   default stream), performs no host synchronisation and no allocation, and
 *   may be captured in a CUDA graph.
 * - Host-side argument errors return GDN_ERR_INVALID_ARG or GDN_ERR_UNSUPPORTED
 *   before anything is launched. Launch failures return GDN_ERR_CUDA.
 * - Errors that only the device can see (a slot index outside [0, num_slots),
 *   non-monotone query_start_loc, an accepted length outside [0, num_pos), a
 *   bounded wait that ran out) set bits of *dev_err (GDN_DEVERR_*), when
 *   dev_err is non-NULL, and the affected request writes nothing. Nothing
 *   traps. Read the word with gdn_read_device_error().
 * - A negative slot index marks a padding request: it is skipped and its
 *   output rows are left untouched. A request with no tokens leaves its slot
 *   untouched, whatever its has_init flag.
 * - Two requests of one call must not name the same slot (undefined result).
 * - Supported geometry: dk = dv = 128, K = 4, Hv a multiple of Hk with
 *   Hv / Hk <= 8. Anything else returns GDN_ERR_UNSUPPORTED.
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Geometry of one GDN layer and its cache pools (the linear_* config fields
 * that size the recurrent state, "How Qwen3.8-27B's 64 layers are dispatched
 * in vLLM", step 5: key heads, value heads, key/value head dims, conv kernel). */
typedef struct gdn_dims {
    int32_t num_k_heads; /* Hk: q and k heads (16, or 4 per TP4 rank)          */
    int32_t num_v_heads; /* Hv: v and z heads (48, or 12 per TP4 rank)         */
    int32_t head_k_dim;  /* dk = 128                                           */
    int32_t head_v_dim;  /* dv = 128                                           */
    int32_t conv_kernel; /* K = 4 conv taps (the current input + 3 history)    */
    int32_t num_slots;   /* Rs: slots in the state and conv-history pools      */
} gdn_dims;

typedef enum gdn_status {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = 1,  /* NULL pointer, negative size, bad mode, misaligned buffer */
    GDN_ERR_UNSUPPORTED = 2,  /* geometry outside the supported set                      */
    GDN_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed                    */
    GDN_ERR_DEVICE_CHECK = 4, /* returned by gdn_read_device_error when *dev_err != 0    */
    GDN_ERR_TIMEOUT = 5       /* returned by gdn_read_device_error for a timed-out wait  */
} gdn_status;

/* Bits of the device error word. */
#define GDN_DEVERR_SLOT 1      /* slot index >= num_slots                       */
#define GDN_DEVERR_OFFSETS 2   /* query_start_loc not monotone or out of range  */
#define GDN_DEVERR_TIMEOUT 4   /* a bounded wait on an async copy ran out       */
#define GDN_DEVERR_ACCEPTED 8  /* accepted length outside [0, num_pos)          */

/* Commit modes of gdn_spec_commit. */
#define GDN_COMMIT_COPY 0    /* copy the accepted checkpoint into the live slot */
#define GDN_COMMIT_REPOINT 1 /* make the checkpoint's slot the live slot        */

/*
 * gdn_conv_update - varlen causal depthwise conv + SiLU with history update.
 * Page: section 01, conv row c_t = SiLU(sum_i w_i QKV0_{t-i}); L00 table,
 * conv history row (3 past inputs, 4 taps with the current one).
 *
 *   x               [T][CH] bf16 packed tokens (T = num_tokens)
 *   conv_w          [CH][K] fp32
 *   conv_hist       [Rs][CH][K-1] bf16, in/out: after the call, the slot of
 *                   request n holds the last K-1 inputs of [history, its tokens]
 *   query_start_loc [num_seqs+1] int32, 0 = q[0] <= q[1] <= ... <= q[N] = T
 *   slot_idx        [num_seqs] int32
 *   has_init        [num_seqs] uint8 or NULL (= all 1); 0 starts from a zero
 *                   history without reading the slot
 *   y               [T][CH] bf16 out: SiLU(conv)
 * x and y must be 8-byte aligned, conv_hist 4-byte and conv_w 16-byte aligned
 * (GDN_ERR_INVALID_ARG otherwise).
 */
gdn_status gdn_conv_update(const gdn_dims *dims, const uint16_t *x, const float *conv_w,
                           uint16_t *conv_hist, const int32_t *query_start_loc,
                           const int32_t *slot_idx, const uint8_t *has_init, int32_t num_seqs,
                           int32_t num_tokens, uint16_t *y, int32_t *dev_err, void *stream);

/*
 * gdn_decode_step - one token per request through the whole mixer core:
 * slot gather, conv + SiLU with in-place history update, q/k L2 norm, one
 * gated-delta-rule step on the fp32 state (in place), gated RMSNorm.
 * Page: section 01 GDN operator table (conv, recurrence and gate rows);
 * section 08, decay first, then predict from the decayed state.
 *
 *   qkv0      [N][CH] bf16 (N = num_seqs, one token each)
 *   conv_w    [CH][K] fp32;  conv_hist [Rs][CH][K-1] bf16 in/out
 *   state     [Rs][Hv][dv][dk] fp32 in/out, 16-byte aligned
 *   slot_idx  [N] int32
 *   alpha, beta [N][Hv] fp32;  z [N][Hv][dv] bf16;  gamma [dv] fp32;  eps >= 0
 *   o         [N][Hv][dv] bf16 out, or NULL
 *   ogate     [N][Hv*dv] bf16 out, or NULL (at least one of o, ogate)
 *
 * Scheduling: the kernel's CTAs claim (request, key head) units from a device
 * counter that the library keeps per stream (a static array of 64, given to
 * streams in order of first use and reused round-robin after that). Calls on
 * one stream run one after another; calls that run at the same time must be
 * on streams holding different counters, i.e. at most 64 streams in use. The
 * per-thread default stream (cudaStreamPerThread) is a different stream in
 * every thread, and each calling thread gets its own counter for it. A
 * captured graph keeps the counter of the stream it was captured on. The same
 * holds for gdn_spec_verify.
 */
gdn_status gdn_decode_step(const gdn_dims *dims, const uint16_t *qkv0, const float *conv_w,
                           uint16_t *conv_hist, float *state, const int32_t *slot_idx,
                           const float *alpha, const float *beta, const uint16_t *z,
                           const float *gamma, float eps, uint16_t *o, uint16_t *ogate,
                           int32_t num_seqs, int32_t *dev_err, void *stream);

/*
 * gdn_chunk_prefill - varlen prefill of packed requests through the whole
 * mixer core, the conv fused in, the state carried from chunk to chunk of 64
 * tokens (a chunk never crosses a request boundary). Page: section 01 GDN
 * operator table, and "GDN's block recurrence uses the associative structure
 * to run in parallel" (prefill paragraph after the 64-layer list).
 *
 *   qkv0      [T][CH] bf16 packed tokens (T = num_tokens)
 *   conv_w, conv_hist, state: as gdn_decode_step (in/out)
 *   query_start_loc [N+1] int32 (as gdn_conv_update); slot_idx [N]
 *   has_init  [N] uint8 or NULL (= all 1); 0 starts from S = 0 and a zero
 *             history without reading the slot
 *   alpha, beta [T][Hv] fp32;  z [T][Hv][dv] bf16 or NULL (then ogate must be
 *             NULL);  gamma [dv];  eps
 *   o [T][Hv][dv] bf16 or NULL;  ogate [T][Hv*dv] bf16 or NULL (not both NULL)
 *   num_tokens 0: every request is empty; nothing is read or written.
 *   workspace, workspace_bytes: device scratch of at least
 *             gdn_prefill_workspace_bytes(dims, N, T) bytes, 256-byte aligned.
 *             Contents need not be zeroed and are clobbered: the call writes
 *             there the order in which the (request, head) chains are started,
 *             longest request first, and one ticket per (request, key head)
 *             counting its value-head chains that have started (the last to
 *             start writes the key head's new q/k conv history at its end).
 *             Two calls in flight
 *             at once need two workspaces.
 */
gdn_status gdn_chunk_prefill(const gdn_dims *dims, const uint16_t *qkv0, const float *conv_w,
                             uint16_t *conv_hist, float *state, const int32_t *query_start_loc,
                             const int32_t *slot_idx, const uint8_t *has_init, const float *alpha,
                             const float *beta, const uint16_t *z, const float *gamma, float eps,
                             uint16_t *o, uint16_t *ogate, int32_t num_seqs, int32_t num_tokens,
                             void *workspace, size_t workspace_bytes, int32_t *dev_err,
                             void *stream);

/*
 * gdn_chunk_prefill_align - gdn_chunk_prefill in "align" prefix-cache mode:
 * snapshots of the recurrent state at block-aligned positions, so that a later
 * request sharing a block-aligned prefix can start from a snapshot instead of
 * recomputing the prefix. Pages: "Qwen3.8-27B: from model structure to vLLM
 * inference data flow", section 05 (a prefix hit reuses whole computed blocks
 * and skips their prefill); "how the 64 layers are dispatched in vLLM"
 * (Qwen3.5 refuses the "all" prefix-cache mode for its GDN layers and asks for
 * --mamba-cache-mode=align). The pages do not spell out the snapshot rule; the
 * reading implemented: after every absolute position that is a multiple of
 * block_tokens, the state of every value head and the conv history are copied
 * to a snapshot slot of the same pools.
 *
 *   arguments as gdn_chunk_prefill, plus
 *   prefix_len   [N] int32 >= 0 or NULL (= 0): tokens of request n already
 *                folded into its slot before this call (its absolute start).
 *                Chunks end on absolute multiples of 64 (the first chunk of a
 *                request may be short); the results do not depend on it.
 *   block_tokens snapshot period, a positive multiple of 64
 *   snap_slot    [N][max_snaps] int32: slot receiving the j-th block boundary
 *                crossed by request n in this call (state after the token at
 *                absolute position b*block_tokens - 1); -1 skips; boundaries
 *                past max_snaps are skipped; >= num_slots sets
 *                GDN_DEVERR_SLOT. Snapshot slots must differ from every live
 *                slot of the call.
 *   max_snaps    >= 0 (0: no snapshots, snap_slot may be NULL)
 */
gdn_status gdn_chunk_prefill_align(const gdn_dims *dims, const uint16_t *qkv0, const float *conv_w,
                                   uint16_t *conv_hist, float *state, const int32_t *query_start_loc,
                                   const int32_t *slot_idx, const uint8_t *has_init, const float *alpha,
                                   const float *beta, const uint16_t *z, const float *gamma, float eps,
                                   uint16_t *o, uint16_t *ogate, int32_t num_seqs, int32_t num_tokens,
                                   const int32_t *prefix_len, int32_t block_tokens,
                                   const int32_t *snap_slot, int32_t max_snaps, void *workspace,
                                   size_t workspace_bytes, int32_t *dev_err, void *stream);

/*
 * gdn_chunk_prefill_noalloc - gdn_chunk_prefill without a workspace argument,
 * for callers that cannot allocate device memory at the call site (a host
 * whose device memory is all reserved up front by its own pool, with no
 * allocation hook). It has no counterpart in the pages: it is an interface
 * convenience of this library, and computes exactly what gdn_chunk_prefill
 * computes.
 *
 * Its scratch is two fixed file-scope device arrays per device: the schedule,
 * 65535 int32 (just under 256 KiB), and the (request, key head) tickets, 2^20
 * int32 (4 MiB): num_seqs above 65535, or num_seqs x num_k_heads above 2^20,
 * is rejected with GDN_ERR_INVALID_ARG before anything is launched. Every GPU
 * that loads the library holds the two arrays until the process exits. The
 * library allocates nothing; the first call on each device looks up the
 * arrays' addresses (cudaGetSymbolAddress) and caches them per device and
 * context (looked up again after cudaDeviceReset), so make that first call
 * before any stream capture. The scratch needs no clearing. Calls that
 * overlap in time on one device (two streams, or two threads) race on the
 * arrays: serialise them.
 *
 * Arguments, layouts, errors: as gdn_chunk_prefill, without workspace and
 * workspace_bytes.
 */
gdn_status gdn_chunk_prefill_noalloc(const gdn_dims *dims, const uint16_t *qkv0, const float *conv_w,
                                     uint16_t *conv_hist, float *state, const int32_t *query_start_loc,
                                     const int32_t *slot_idx, const uint8_t *has_init, const float *alpha,
                                     const float *beta, const uint16_t *z, const float *gamma, float eps,
                                     uint16_t *o, uint16_t *ogate, int32_t num_seqs, int32_t num_tokens,
                                     int32_t *dev_err, void *stream);

/*
 * gdn_spec_verify - speculative verify: P = num_pos positions per request (the
 * last sampled token and P-1 drafts, verified in one forward) through the
 * whole mixer core, keeping the state and conv history after EVERY position p
 * in checkpoint slot spec_slot_idx[n][p] of the same pools. The live slot
 * slot_idx[n] is only read. Pages: "Qwen3.8 MTP" (huashanblogllm.xyz),
 * section 4 (verify: context + drafts in one pass) and section 5 (accept /
 * reject); the DeepSeek-V3 pipeline page, section 7.3 (the input
 * [..., t_{T+1}, d1 .. dk] is verified in parallel); first page, L00 table
 * ("extra speculative slots counted separately").
 *
 *   qkv0 [N*P][CH] bf16, request-major (row n*P + p);  alpha, beta [N*P][Hv];
 *   z [N*P][Hv][dv];  o [N*P][Hv][dv] or NULL;  ogate [N*P][Hv*dv] or NULL
 *   conv_hist, state: the pools (live slots read, checkpoint slots written)
 *   slot_idx [N];  spec_slot_idx [N][P] int32, distinct from every live slot
 *   num_pos: 1 <= P <= 8
 * qkv0, conv_w, conv_hist, state and (with ogate) z must be 16-byte aligned
 * (GDN_ERR_INVALID_ARG otherwise): the kernel stages them with bulk copies.
 */
gdn_status gdn_spec_verify(const gdn_dims *dims, const uint16_t *qkv0, const float *conv_w,
                           uint16_t *conv_hist, float *state, const int32_t *slot_idx,
                           const int32_t *spec_slot_idx, const float *alpha, const float *beta,
                           const uint16_t *z, const float *gamma, float eps, uint16_t *o,
                           uint16_t *ogate, int32_t num_seqs, int32_t num_pos, int32_t *dev_err,
                           void *stream);

/*
 * gdn_spec_commit - make the state after the accepted position a = accepted[n]
 * (0 <= a < num_pos; position 0 is the last sampled token) the request's
 * state ("Qwen3.8 MTP" page, section 5: the longest matching prefix is kept).
 *
 *   mode GDN_COMMIT_COPY:    state and conv history of slot spec_slot_idx[n][a]
 *                            are copied into slot slot_idx[n] (slot_idx read)
 *   mode GDN_COMMIT_REPOINT: slot_idx[n] = spec_slot_idx[n][a] (nothing copied)
 *   accepted [N] int32; spec_slot_idx [N][P]; slot_idx [N] (in/out for REPOINT)
 */
gdn_status gdn_spec_commit(const gdn_dims *dims, const int32_t *accepted,
                           const int32_t *spec_slot_idx, int32_t *slot_idx, float *state,
                           uint16_t *conv_hist, int32_t num_seqs, int32_t num_pos, int32_t mode,
                           int32_t *dev_err, void *stream);

/*
 * gdn_gated_rmsnorm - Ogate = RMSNorm(o) (.) SiLU(z) per head row of D values:
 * out = o / sqrt(mean(o^2) + eps) * gamma * SiLU(z). Page: section 01, gate row
 * ([T,48,128] -> [T,6144]); section 08 (the GDN output gate is SiLU after
 * RMSNorm).
 *
 *   o, z [T][H][D] bf16;  gamma [D] fp32;  out [T][H*D] bf16
 *   D a multiple of 4, 4 <= D <= 1024
 */
gdn_status gdn_gated_rmsnorm(const uint16_t *o, const uint16_t *z, const float *gamma, float eps,
                             uint16_t *out, int32_t num_tokens, int32_t num_heads,
                             int32_t head_dim, void *stream);

/*
 * gdn_rmsnorm - the layer's input RMSNorm U = X / sqrt(mean(X^2) + eps) (.) gamma
 * over the hidden size, optionally fused with the residual add in front of it.
 * Page "Qwen3.8-27B: from model structure to vLLM inference data flow", section
 * 01 operator table, the U row (and the N = RMSNorm(Y) row, same form); page
 * "DeepSeek-V3 inference pipeline walk-through" section 4.2 for the fused
 * add-and-norm.
 *
 *   x         [T][D] bf16, D = hidden_size (a multiple of 8, at most 8192)
 *   residual  [T][D] bf16 or NULL. When given, residual <- bf16(x + residual)
 *             (rounded once, in place) and the norm is taken of that sum.
 *   gamma     [D] fp32;  eps > 0 and finite
 *   out       [T][D] bf16; may be x itself (in place)
 * Pointers 16-byte aligned. num_tokens 0 is a no-op.
 */
gdn_status gdn_rmsnorm(const uint16_t *x, uint16_t *residual, const float *gamma, float eps, uint16_t *out,
                       int32_t num_tokens, int32_t hidden_size, void *stream);

/*
 * gdn_in_proj - the input projections in front of the mixer core: QKV0 = U
 * W_qkv^T, Z = U W_z^T and (optionally) the raw a, b projections [a | b] = U
 * W_ab^T, bf16 operands, fp32 accumulation, in one launch of the library's
 * tcgen05 GEMM (the three outputs share the input tiles). Page: section 01 GDN
 * operator table, the in_proj rows ([T,5120] -> QKV0 [T,10240], Z [T,6144], a
 * and b [T,48]). The 4-tap conv that the table puts right after is fused into
 * the mixer entry points that read QKV0; the map from a, b to alpha, beta is
 * not on the pages, so a, b come out raw (fp32).
 *
 *   hidden  [T][D] bf16, D = hidden_size (a multiple of 8)
 *   w_qkv   [CH][D] bf16;  qkv0 [T][CH] bf16 out      (the nn.Linear weight layout)
 *   w_z     [Hv*dv][D] bf16;  z [T][Hv*dv] bf16 out
 *   w_ab    [2*Hv][D] bf16 or NULL;  ab [T][2*Hv] fp32 out or NULL (both or neither;
 *           a in columns 0 .. Hv-1, b in Hv .. 2Hv-1)
 *   dev_err GDN_DEVERR_TIMEOUT if a bounded wait inside the kernel ran out, or NULL
 * Pointers 16-byte aligned.
 */
gdn_status gdn_in_proj(const gdn_dims *dims, const uint16_t *hidden, int32_t hidden_size,
                       const uint16_t *w_qkv, const uint16_t *w_z, const uint16_t *w_ab, uint16_t *qkv0,
                       uint16_t *z, float *ab, int32_t num_tokens, int32_t *dev_err, void *stream);

/*
 * FP8 block-scaled projections. Page "Qwen3.8-27B: from model structure to vLLM
 * inference data flow", section 04 (precision and cache): the checkpoint's
 * linear weights are FP8 E4M3 with one scale per 128 x 128 weight block and the
 * activations are quantised to FP8 dynamically. A scale s dequantises its
 * block: value = E4M3(code) * s. Both quantisers set s = max(amax, 1e-12) / 448
 * (amax = the block's largest |x|, 448 = the largest finite E4M3 value) and
 * code = E4M3(x / s) rounded to nearest even with saturation; the divisions
 * are IEEE-rounded fp32, so the codes are reproducible bit for bit.
 *
 * gdn_fp8_quant_act - x [T][K] bf16 -> x8 [T][K] e4m3 and x_scale, one scale per
 *   token and 128-wide group of K, stored [T][K/128] (group fastest). K a
 *   multiple of 128; pointers 16-byte aligned.
 * gdn_fp8_quant_weight - w [N][K] bf16 -> w8 [N][K] e4m3 and w_scale, one scale
 *   per 128 x 128 block, stored [ceil(N/128)][K/128] (K block fastest); a last
 *   partial row block takes the largest |w| of its rows. K a multiple of 128;
 *   pointers 16-byte aligned.
 * gdn_fp8_linear - out [T][N] = dequant(x8) dequant(w8)^T (+ residual [T][N]),
 *   bf16 out; in place on the residual is allowed. x_scale [T][K/128] and
 *   w_scale [ceil(N/128)][K/128] as the two quantisers write them. The tensor
 *   cores form each 128-wide block product of K exactly (E4M3 products, fp32
 *   sums) and fp32 registers take the scaled sum over blocks. K a multiple of
 *   128, N a multiple of 16.
 *   workspace: when K is split across CTAs, the fp32 partial sums of the
 *   parts (one 128 x 256 tile per K part at decode-sized token counts, where a
 *   cluster of CTAs shares each output tile; one 128 x 128 tile per CTA and a
 *   ticket per output tile for the stream-K schedule of mid-sized counts),
 *   gdn_fp8_linear_workspace_bytes(T, K, N) bytes (0: this shape is not split
 *   on the current GPU), 256-byte aligned and ZERO-FILLED before its first use:
 *   the tickets must start at zero, and every call that completes resets them,
 *   so the workspace is reusable without clearing (after a call that reports a
 *   device error, clear it again). NULL or too small: K is not split. Calls
 *   sharing one workspace must not overlap.
 *   dev_err: GDN_DEVERR_TIMEOUT if a bounded wait inside the kernel ran out.
 */
gdn_status gdn_fp8_quant_act(const uint16_t *x, uint8_t *x8, float *x_scale, int32_t num_tokens, int32_t k,
                             void *stream);
gdn_status gdn_fp8_quant_weight(const uint16_t *w, uint8_t *w8, float *w_scale, int32_t n, int32_t k,
                                void *stream);
size_t gdn_fp8_linear_workspace_bytes(int32_t num_tokens, int32_t k, int32_t n);
gdn_status gdn_fp8_linear(const uint8_t *x8, const float *x_scale, const uint8_t *w8, const float *w_scale,
                          const uint16_t *residual, uint16_t *out, int32_t num_tokens, int32_t k, int32_t n,
                          void *workspace, size_t workspace_bytes, int32_t *dev_err, void *stream);

/*
 * gdn_out_proj - the output projection after the mixer core and the residual
 * add: out = ogate W^T (+ residual), bf16 operands, fp32 accumulation in tensor
 * memory, bf16 out (round to nearest even). Page: section 01 GDN operator
 * table, the Wo row ([T,6144] -> [T,5120]) and the residual stream around the
 * mixer. The gated RMSNorm that the page puts before Wo is fused into the mixer
 * entry points' ogate output, so this is a plain GEMM, run by the library's own
 * tcgen05 kernel: 128-token x 256-output tiles for large T; for T <= 256 the
 * operands swap (128 weight rows x all tokens per tile, every weight byte read
 * once); when the tiles leave at least half the SMs idle, a cluster of up to 4
 * CTAs splits each tile's K range and adds the partial tiles up in shared
 * memory, in a fixed order (the bits do not depend on timing). It allocates
 * nothing and takes no workspace.
 *
 *   ogate     [T][K] bf16 (T = num_tokens, K = in_features)
 *   w         [N][K] bf16, the nn.Linear weight layout (N = out_features)
 *   residual  [T][N] bf16 or NULL; may equal out (in-place residual add)
 *   out       [T][N] bf16
 *   dev_err   GDN_DEVERR_TIMEOUT if a bounded wait inside the kernel ran out, or NULL.
 * Pointers 16-byte aligned; K and N multiples of 8 (GDN_ERR_UNSUPPORTED
 * otherwise).
 */
gdn_status gdn_out_proj(const uint16_t *ogate, const uint16_t *w, const uint16_t *residual, uint16_t *out,
                        int32_t num_tokens, int32_t in_features, int32_t out_features, int32_t *dev_err,
                        void *stream);

/* Bytes of one slot of the fp32 state pool: Hv*dv*dk*4 (3 MiB at 48x128x128,
 * the L00 table's "3 MiB per sequence per layer"). 0 for invalid dims. */
size_t gdn_state_bytes(const gdn_dims *dims);

/* Bytes of one slot of the bf16 conv-history pool: CH*(K-1)*2. 0 for invalid dims. */
size_t gdn_conv_hist_bytes(const gdn_dims *dims);

/* Device scratch gdn_chunk_prefill needs for N requests and T packed tokens:
 * N int32 rounded up to 256 bytes, then N x num_k_heads int32 rounded up to 256
 * bytes (0 for invalid dims or N <= 0). */
size_t gdn_prefill_workspace_bytes(const gdn_dims *dims, int32_t num_seqs, int32_t num_tokens);

/* Static, human-readable name of a status code. */
const char *gdn_status_string(gdn_status status);

/*
 * Synchronises `stream`, copies the device error word to *host_err (host
 * memory) and, if reset != 0, zeroes it. Returns GDN_OK when the word is 0,
 * GDN_ERR_TIMEOUT when the timeout bit is set, else GDN_ERR_DEVICE_CHECK.
 * This is the only entry point that synchronises.
 */
gdn_status gdn_read_device_error(int32_t *dev_err, int32_t *host_err, int32_t reset, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */
