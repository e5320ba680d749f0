/*
 * kvr.h -- C ABI of libkvr: selective KV-cache refresh on one GB300 GPU.
 *
 * After a context edit (a deleted span, a changed block seam, or an updated
 * adapter), a chosen set of retained-suffix positions is recomputed layer by
 * layer against a mixed cache of fresh and stale K/V.  Per layer, the rows of
 * all selected positions are packed together, normalised, projected, rotated
 * at their global positions, and their K/V rows are written back into the
 * cache before any of them attends ("Budgeted KV-Cache Repair for Evolving
 * Contexts", Sec. 13.2, Eq. 21).  Each packed query then attends causally
 * over the whole cache, every key j <= g_i, fresh or stale (ibid. Eq. 22),
 * with the per-key logit bias of operator F,
 *     s_ij = <q_i, k_j>/sqrt(d_h) + alpha*1[type_j = local] + beta*1[j in S']
 * ("kv-cross-attention-reuse", Sec. 6.4, Logit form), and finishes with the
 * output projection, residual, RMSNorm and SwiGLU MLP.  After the last layer
 * the refreshed positions become type global (ibid., physical repair mode).
 *
 * Conventions for every entry point:
 *   - Plain C; every call returns a kvr_status; a thread-local message for
 *     the last failure is available from kvr_last_error().
 *   - "device" pointers are CUDA global-memory addresses on the current
 *     device; "host" pointers are CPU memory.  The caller owns every buffer
 *     passed in; the library owns only the kvr_cache object and the small
 *     device buffers it allocates in kvr_create_cache (selection lists,
 *     metadata bit masks, the execution plan, the rotary table, counters)
 *     and frees them in kvr_destroy_cache.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls only enqueue work unless documented as synchronous;
 *     kvr_sync_status() synchronises and reports device-side failures.
 *   - Arguments are validated on the host before anything is enqueued; a
 *     failed validation enqueues nothing and leaves the cache unchanged.
 *   - After any error the cache can still be destroyed.
 *   - KVR_PDL=0 in the environment (read once per process) turns off
 *     programmatic dependent launch between the kernels of a call; it
 *     changes how work is launched, never what it computes.
 *   - KVR_ATTN_MERGE=cta|kernel and KVR_ATTN_CHUNK=C in the environment
 *     (read by every kvr_select) narrow the attention's split choice, for
 *     tests and tuning: the merge of split K/V ranges by the last CTA of each
 *     query tile or by a merge kernel, and the K/V tiles per CTA.  At the same
 *     chunk both merges give the same output bits.
 *   - KVR_FAULT in the environment (read at the start of every call) makes
 *     one host-side step fail, for tests of the error paths; no GPU fault is
 *     made.  "alloc" or "alloc:N": the device allocations of
 *     kvr_create_cache (the N-th one; 1-based) return out-of-memory, so the
 *     call returns ENOMEM after freeing what it had allocated.  "upload": the
 *     position upload of a selection fails (ECUDA); the cache then has no
 *     valid selection (ESTATE until the next successful select).  "launch":
 *     every kernel launch of the call fails before it is issued (ECUDA).
 *     "timeout": each refresh layer marks the device error word as a bounded
 *     device wait does when it gives up, so kvr_sync_status reports ETIMEOUT.
 */
#ifndef KVR_H
#define KVR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KVR_OK = 0,
    KVR_EINVAL = 1,       /* malformed argument: NULL, duplicate position, budget mismatch, bad shape */
    KVR_ERANGE = 2,       /* index out of range: position outside the suffix, layer >= n_layers */
    KVR_ENOMEM = 3,       /* a library-owned allocation failed */
    KVR_ECUDA = 4,        /* a CUDA runtime call or launch failed */
    KVR_ETIMEOUT = 5,     /* a device-side wait gave up (reported by kvr_sync_status) */
    KVR_EDEVICE = 6,      /* a device-side check failed (reported by kvr_sync_status) */
    KVR_ESTATE = 7,       /* call out of order, e.g. a refresh before any kvr_select */
    KVR_EUNSUPPORTED = 8  /* shape or dtype this build does not implement */
} kvr_status;

typedef enum { KVR_F32 = 0, KVR_BF16 = 1 } kvr_dtype;

/* kvr_create_cache flags */
#define KVR_SINK_STATIC 0x1u   /* S' keeps its beta penalty after refresh */

/* kvr_refresh_layer / kvr_refresh flags */
#define KVR_COMMIT_META 0x1u   /* after this layer: type_t <- global (and t leaves S') for the selection */

/* Model shape, copied by kvr_create_cache.  Dense pre-norm decoder with
 * rotate-half RoPE (no scaling) and grouped-query attention; the shapes of
 * Llama-3 and Qwen2.5 ("Budgeted KV-Cache Repair", Sec. 13.2: native dense
 * Llama/Qwen with default fixed RoPE).
 * Constraints: head_dim == 128 (bf16) or 64/128 (f32); n_q_heads a multiple
 * of n_kv_heads; d_model, n_q_heads*head_dim and ffn_dim multiples of 64. */
typedef struct {
    int32_t n_layers;
    int32_t d_model;
    int32_t n_q_heads;
    int32_t n_kv_heads;
    int32_t head_dim;
    int32_t ffn_dim;
    double  rope_theta;     /* inv_freq_i = theta^(-2i/head_dim) */
    float   rms_eps;
    int32_t dtype;          /* kvr_dtype of weights, cache and hidden rows */
    int32_t has_qkv_bias;   /* Qwen2.5 shapes carry q/k/v biases */
    int32_t has_qk_norm;    /* Qwen3 shapes: RMSNorm of every Q and K head (over head_dim,
                               eps = rms_eps) before RoPE; the recompute of "Budgeted
                               KV-Cache Repair", Sec. 13.2, runs the model's own block */
} kvr_model_desc;

/* One layer's weights: caller-owned device pointers in the model dtype,
 * nn.Linear layout (row = output feature, contiguous over input features).
 * All pointers 16-byte aligned. */
typedef struct {
    const void* w_qkv;      /* [(Hq + 2*Hkv)*dh, d]: Q heads, then K heads, then V heads */
    const void* b_qkv;      /* [(Hq + 2*Hkv)*dh] or NULL */
    const void* w_o;        /* [d, Hq*dh] */
    const void* w_gate_up;  /* [2*F, d]: rows 0..F-1 gate, rows F..2F-1 up */
    const void* w_down;     /* [d, F] */
    const void* norm1;      /* [d] RMSNorm weight before attention */
    const void* norm2;      /* [d] RMSNorm weight before the MLP */
    const void* q_norm;     /* [head_dim] per-head RMSNorm weight of Q, or NULL without has_qk_norm */
    const void* k_norm;     /* [head_dim] per-head RMSNorm weight of K, or NULL without has_qk_norm */
} kvr_layer_weights;

typedef struct kvr_cache kvr_cache;   /* opaque */

/* ---------------------------------------------------------------------------
 * kvr_create_cache -- bind a mixed cache L[t, l] = (K_t,l, V_t,l, m_t)
 * ("kv-cross-attention-reuse", Sec. 6.2).
 *
 *   m           model shape (copied).
 *   batch       independent sequences sharing the weights (>= 1).
 *   capacity    cache rows per sequence (>= n_tokens).
 *   k_base, v_base  device, caller-owned, model dtype, layout
 *               [batch][n_layers][n_kv_heads][capacity][head_dim], 16-byte
 *               aligned.  Rows outside a selection are never written.
 *   n_tokens    valid cache length per sequence; keys >= n_tokens are never
 *               read.
 *   suffix_start  retained prefix [0, suffix_start) is valid; only
 *               positions in [suffix_start, n_tokens) are selectable
 *               ("Budgeted KV-Cache Repair", Sec. 7.1).
 *   local_bits, sink_bits  host, nullable (= all zero), uint32 words
 *               [batch][ceil(capacity/32)], bit b of word w = position 32w+b:
 *               type_t = local, and t in S' (spurious sinks).
 *   alpha, beta  logit bias of local keys and of S' keys (operator F).
 *   flags       KVR_SINK_STATIC.
 *   out         receives the handle.
 * Synchronous with respect to `stream` for the metadata upload.
 * Errors: EINVAL (NULL, bad shape), EUNSUPPORTED, ENOMEM, ECUDA.
 * ------------------------------------------------------------------------- */
kvr_status kvr_create_cache(const kvr_model_desc* m, int32_t batch, int32_t capacity,
                            void* k_base, void* v_base, int32_t n_tokens, int32_t suffix_start,
                            const uint32_t* local_bits, const uint32_t* sink_bits,
                            float alpha, float beta, uint32_t flags, void* stream,
                            kvr_cache** out);

/* Free the library-owned buffers of `c` (never the caller's). NULL is a no-op.
 * Synchronises the device first so no enqueued work still uses them. */
kvr_status kvr_destroy_cache(kvr_cache* c);

/* ---------------------------------------------------------------------------
 * kvr_select -- fix the support of one refresh and pack its rows.
 * ("Budgeted KV-Cache Repair", Sec. 7.1 Eq. 3 exact budget; Sec. 3.2 and
 * Algorithm 1: sort the selected positions and coalesce adjacent ones into
 * execution intervals; Sec. 13.2: gather the selected rows once into a
 * compact B-row hidden buffer; Eqs. 23-24 reusable per-query-tile plan.)
 *
 *   positions   host int32, zero-based positions in any order, sequence-major:
 *               counts[0] positions of sequence 0, then sequence 1, ...
 *   counts      host int32 [batch]; 0 is allowed.
 *   budget_percent  -1 skips the check; otherwise each count must equal
 *               min(S, ceil(S*b/100)), S = n_tokens - suffix_start.
 *   Row source (exactly one):
 *     token_ids + embed_table: device int32 [batch][capacity] token ids and
 *               device [vocab][d] embedding table (model dtype); row r gets
 *               embed_table[token_ids[seq][u_r]]; vocab = rows of embed_table (a
               token id outside [0, vocab) is reported as EDEVICE by
               kvr_sync_status and its row is left unwritten).
 *     hidden_src: device [batch][capacity][d] per-position layer-0 inputs.
 *   hidden_out  device [sum(counts)][d] (model dtype), rows in sorted
 *               position order, sequence-major.
 *   n_rows_out, n_intervals_out  host, nullable: total rows and intervals.
 * Host validation (before any launch): every position in
 * [suffix_start, n_tokens) else ERANGE; no duplicates within a sequence
 * else EINVAL; budget else EINVAL.  The device then builds the sorted list
 * U, intervals, the selected / effective-local / effective-sink bit masks
 * and the plan, and gathers the rows.  Replaces any previous selection.
 * ------------------------------------------------------------------------- */
kvr_status kvr_select(kvr_cache* c, const int32_t* positions, const int32_t* counts,
                      int32_t budget_percent, const int32_t* token_ids, const void* embed_table,
                      int32_t vocab, const void* hidden_src, void* hidden_out, int32_t* n_rows_out,
                      int32_t* n_intervals_out, void* stream);

/* Bytes of workspace kvr_refresh_layer / kvr_refresh / kvr_attend need for up
 * to `max_rows` packed rows (0 = the current selection). */
size_t kvr_workspace_bytes(const kvr_cache* c, int32_t max_rows);

/* ---------------------------------------------------------------------------
 * kvr_refresh_layer -- one layer of the packed refresh over the current
 * selection ("Budgeted KV-Cache Repair", Sec. 13.2, Eqs. 21-22):
 *   xn = RMSNorm(x); [q|k|v] = xn W_qkv^T (+ b); RoPE(q, k) at u_r;
 *   K_l[u_r] <- k, V_l[u_r] <- v for every row r (before any attention);
 *   o_r = softmax_j<=u_r(q_r k_j/sqrt(d_h) + alpha*loc_j + beta*snk_j) V_j,
 *     loc_j = local_j & !selected_j, snk_j = sink_j & !selected_j (or sink_j
 *     under KVR_SINK_STATIC): a selected key is fresh whenever it is read;
 *   h = x + o W_o^T; x' = h + (silu(hn W_g^T) * (hn W_u^T)) W_d^T,
 *     hn = RMSNorm(h).
 *   layer       [0, n_layers) else ERANGE.
 *   w           this layer's weights (host struct of device pointers).
 *   hidden_inout  device [rows][d] model dtype, from kvr_select; updated.
 *   workspace   device, >= kvr_workspace_bytes(c, 0) bytes, 256-byte aligned.
 *   flags       KVR_COMMIT_META: after the layer, clear local (and sink unless
 *               static) for the selected positions.
 * Errors: ESTATE (no selection), ERANGE, EINVAL (NULL / small workspace),
 * ECUDA.
 * ------------------------------------------------------------------------- */
kvr_status kvr_refresh_layer(kvr_cache* c, int32_t layer, const kvr_layer_weights* w,
                             void* hidden_inout, void* workspace, size_t ws_bytes,
                             uint32_t flags, void* stream);

/* Layers [layer_begin, layer_end) in order, then the metadata commit when
 * flags has KVR_COMMIT_META.  `w` is a host array indexed by layer
 * (w[layer_begin] .. w[layer_end-1] are read).  Same errors as above. */
kvr_status kvr_refresh(kvr_cache* c, const kvr_layer_weights* w, int32_t layer_begin,
                       int32_t layer_end, void* hidden_inout, void* workspace, size_t ws_bytes,
                       uint32_t flags, void* stream);

/* ---------------------------------------------------------------------------
 * kvr_refresh_interval_wise -- the interval-major schedule ("Budgeted KV-Cache
 * Repair", Sec. 7.1, sequential maximal-interval replay): each maximal
 * interval of selected positions, sequence by sequence in position order, is
 * forwarded through layers [layer_begin, layer_end) against the cache as the
 * earlier intervals left it, then committed (KVR_COMMIT_META in flags) before
 * the next interval starts.  In real arithmetic this equals the packed
 * refresh ([BKR] Sec. 13.2); it is the comparator for the packed executor.
 *   Selection arguments as kvr_select (validated as a whole first); `w` as
 *   kvr_refresh.  hidden_out: device [sum(counts)][d], rows in sorted position
 *   order.  workspace >= kvr_workspace_bytes(c, longest interval).
 *   n_intervals_out: host, nullable.  Leaves the last interval selected.
 * ------------------------------------------------------------------------- */
kvr_status kvr_refresh_interval_wise(kvr_cache* c, const int32_t* positions, const int32_t* counts,
                                     int32_t budget_percent, const int32_t* token_ids, const void* embed_table,
                                     int32_t vocab, const void* hidden_src, const kvr_layer_weights* w,
                                     int32_t layer_begin, int32_t layer_end, void* hidden_out, void* workspace,
                                     size_t ws_bytes, uint32_t flags, int32_t* n_intervals_out, void* stream);

/* ---------------------------------------------------------------------------
 * kvr_reselect -- switch the selection mid-refresh, carrying rows over
 * ("CacheReforge", Bounded Recovery, "Executable restart": a layer range is
 * recomputed over the whole affected suffix from the hidden states stored at
 * the range's first layer, while the positions refreshed so far keep their
 * current state).  New positions/counts as kvr_select (no budget check).
 *   carry_rows  device [current rows][d]: the current selection's rows (as the
 *               last refresh left them); a new row whose position was
 *               selected takes its row from here.
 *   fill_rows   device [batch][capacity][d]: per-position rows for every other
 *               new position (e.g. the stored boundary states).
 *   hidden_out  device [sum(counts)][d]; must not be carry_rows.
 * Metadata bits are untouched until a commit.
 * ------------------------------------------------------------------------- */
kvr_status kvr_reselect(kvr_cache* c, const int32_t* positions, const int32_t* counts, const void* carry_rows,
                        const void* fill_rows, void* hidden_out, int32_t* n_rows_out, int32_t* n_intervals_out,
                        void* stream);

/* ---------------------------------------------------------------------------
 * kvr_refresh_range -- the adapter-drift repair of one edit in one call
 * ("CacheReforge", Bounded Recovery, "Executable restart"): layers
 * [range_begin, range_end) are recomputed over every position of the
 * affected suffix [suffix_start, n_tokens) of every sequence, all other
 * layers only over the selected positions.  In order, on one stream:
 *   1. select `positions` (as kvr_select, no budget check; rows from
 *      token_ids + embed_table, or from hidden_src) into hidden_sel;
 *   2. layers [0, range_begin) over the selected rows;
 *   3. switch to the whole suffix (kvr_reselect): a selected position keeps
 *      its refreshed row, every other suffix position enters from
 *      `boundary`, the stored hidden states at layer range_begin; rows go to
 *      hidden_full;
 *   4. layers [range_begin, range_end) over the whole suffix;
 *   5. switch back to the selected positions, carrying their rows;
 *   6. layers [range_end, n_layers) over the selected rows, then `flags`
 *      (KVR_COMMIT_META clears local/sink of the selected positions only).
 * With range_begin == range_end steps 3-5 are skipped (a plain refresh).
 *   boundary    device [batch][capacity][d_model], model dtype.
 *   hidden_sel  device [sum(counts)][d_model]: the selected rows' output.
 *   hidden_full device [batch * (n_tokens - suffix_start)][d_model]
 *               (scratch for the range; may be NULL when the range is empty).
 *   workspace   at least kvr_workspace_bytes(c, batch * (n_tokens -
 *               suffix_start)) bytes when the range is not empty, else
 *               kvr_workspace_bytes(c, sum(counts)); 256-byte aligned.
 * Errors as the calls it makes; ERANGE for a range outside [0, n_layers].
 * On an error the selection may be either one; select again before reuse.
 * ------------------------------------------------------------------------- */
kvr_status kvr_refresh_range(kvr_cache* c, const kvr_layer_weights* w, int32_t range_begin, int32_t range_end,
                             const int32_t* positions, const int32_t* counts, const int32_t* token_ids,
                             const void* embed_table, int32_t vocab, const void* hidden_src, const void* boundary,
                             void* hidden_sel, void* hidden_full, void* workspace, size_t ws_bytes, uint32_t flags,
                             void* stream);

/* ---------------------------------------------------------------------------
 * kvr_lora_merge -- fold a low-rank adapter into a projection
 * ("CacheReforge", Implementation: a LoRA on the cache-producing projections):
 *   w_out[i][k] = w[i][k] + scale * sum_j b[i - row_begin][j] * a[j][k]
 * for rows [row_begin, row_begin + row_count) of the [n_out, K] matrix
 * (nn.Linear layout); other rows are copied.  w_out may equal w.
 *   a: device [rank][K], b: device [row_count][rank], model dtype; fp32
 *   accumulation, one rounding to the dtype.
 * ------------------------------------------------------------------------- */
kvr_status kvr_lora_merge(const void* w, void* w_out, int32_t n_out, int32_t K, int32_t row_begin,
                          int32_t row_count, const void* a, const void* b, int32_t rank, float scale, int32_t dtype,
                          void* stream);

/* ---------------------------------------------------------------------------
 * kvr_refresh_layer_noalloc -- kvr_refresh_layer without a caller workspace
 * and without any allocation.  The paper has no counterpart: this entry point
 * exists for callers that cannot hand the library scratch memory when they
 * refresh (a host framework whose allocator owns all device memory, a
 * serving loop that must not allocate after start-up).
 *   The layer's scratch lives in one fixed 64 MiB array in device global
 *   memory inside the library image; every GPU that loads the image holds it
 *   until the process exits.  A selection whose scratch is larger
 *   (kvr_workspace_bytes(c, 0) > 64 MiB) is rejected with EINVAL before
 *   anything is enqueued.
 *   The first call on a device looks up the array's address; make that call
 *   before any stream capture on the device.  The cache's device must be the
 *   current device (else EINVAL).  Calls share the array: calls
 *   whose GPU work overlaps race on it and must be serialised by the caller.
 *   The array keeps the last call's contents; a layer never reads scratch it
 *   has not written in the same call.
 *   Arguments, results and errors otherwise as kvr_refresh_layer.
 * ------------------------------------------------------------------------- */
kvr_status kvr_refresh_layer_noalloc(kvr_cache* c, int32_t layer, const kvr_layer_weights* w,
                                     void* hidden_inout, uint32_t flags, void* stream);

/* ---------------------------------------------------------------------------
 * kvr_attend -- inference mode of operator F ("kv-cross-attention-reuse",
 * Sec. 6.4): attention only, no write-back, with the stored correction masks
 * (type_j = local, j in S') as they are now.
 *   q    device [rows][n_q_heads][head_dim], rotated, model dtype; row r is
 *        the query at position u_r of the current selection.
 *   out  device [rows][n_q_heads*head_dim], model dtype.
 *   workspace as for kvr_refresh_layer.
 * ------------------------------------------------------------------------- */
kvr_status kvr_attend(kvr_cache* c, int32_t layer, const void* q, void* out,
                      void* workspace, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * kvr_shift -- Shift after a deletion ("Budgeted KV-Cache Repair for Evolving
 * Contexts", Sec. 7.1, Eq. 2): positions [start, start + d) are removed from
 * every sequence.  In every (sequence, layer, K/V head) the rows
 * [start + d, n_tokens) move down to [start, n_tokens - d).  Keys are stored
 * after the rotary map, so a key that moves from i to i - d becomes
 * R_{i-d} R_i^{-1} k = R_{-d} k: one rotation by -d positions, the same for
 * every row.  Values carry no position and move unchanged.  The local and
 * sink bits move with their positions; the bits of [n_tokens - d, n_tokens)
 * are cleared.  Cache rows [n_tokens - d, n_tokens) keep their old contents
 * (they are now past the end and no attention reads them).
 *   In place, on the cache's own K/V buffers, with one read and one write of
 *   each moved row.  Afterwards n_tokens -= d and
 *   suffix_start = min(suffix_start, start): every row from the deletion on
 *   was computed with the deleted span visible.  The current selection is
 *   dropped (kvr_select again before a refresh or kvr_attend).
 *   EINVAL: start < 0, d < 0, start + d > n_tokens, or d == n_tokens.
 *   d == 0 enqueues nothing.
 * ------------------------------------------------------------------------- */
kvr_status kvr_shift(kvr_cache* c, int32_t start, int32_t d, void* stream);

/* kvr_splice flags */
#define KVR_SPLICE_LOCAL 0x1u   /* mark the spliced positions type local */
#define KVR_SPLICE_SINK 0x2u    /* mark the block's first min(4, n) positions as members of S' */

/* ---------------------------------------------------------------------------
 * kvr_splice -- place a block whose K/V were computed on their own at new
 * global positions ("Models Take Notes at Prefill: KV Cache Can Be Editable
 * and Composable", Sec. 5: the chunk's keys are re-rotated from their source
 * positions to the target positions; values carry no position).  This builds
 * a mixed cache out of independently prefilled blocks ("kv-cross-attention-
 * reuse", Sec. 6: blocks B_1..B_m).
 *   k_src, v_src  device [n_layers][n_kv_heads][n][head_dim], model dtype;
 *                 row i holds the block's token i, its key rotated at
 *                 position src_pos + i.  Must not overlap the cache.
 *   Row i lands in cache row dst_pos + i of sequence `seq` in every layer and
 *   head, its key rotated by dst_pos - src_pos.  Other rows are untouched.
 *   flags: KVR_SPLICE_LOCAL sets the local bit of [dst_pos, dst_pos + n);
 *   KVR_SPLICE_SINK sets the sink bit of the block's first min(4, n)
 *   positions (the block's own attention sinks, "kv-cross-attention-reuse",
 *   Sec. 6.4).  Bits are only ever set, never cleared, by this call.
 *   EINVAL: NULL or non-16-byte-aligned sources, seq outside [0, batch),
 *   n < 0, dst_pos < 0, src_pos < 0, or dst_pos + n > n_tokens.
 *   n == 0 enqueues nothing.  The selection, if any, stays as it is.
 * ------------------------------------------------------------------------- */
kvr_status kvr_splice(kvr_cache* c, int32_t seq, int32_t dst_pos, int32_t n, const void* k_src,
                      const void* v_src, int32_t src_pos, uint32_t flags, void* stream);

/* ---------------------------------------------------------------------------
 * kvr_sur_select -- Semantic-Unit Refresh selection ("Budgeted KV-Cache
 * Repair for Evolving Contexts", Sec. 3.2 and Sec. 7.3, Eqs. 1/7 and 8).
 *   Token scores: r_i = max_j cos(E[s_i], E[q_j]) + 0.25 * 1[s_i in q], in
 *   fp32 (a zero-norm embedding row scores cosine 0; a token that occurs in
 *   the query meets its own embedding, cosine exactly 1, and scores exactly
 *   1.25, so the tie rule below is not decided by rounding).
 *   Unit score: the mean of the unit's four largest token scores (all of
 *   them when it has fewer than four).  Units are ranked by score, earlier
 *   start first on ties, and admitted whole in that order while they fit the
 *   allowance B = min(S, ceil(S * b / 100)) (Eq. 3).  The first unit that
 *   does not fit the remaining w positions contributes the width-w window
 *   that maximises the sum of the forward envelope
 *   u_t = max(exp(r_t - r_max), exp(-1/16) u_{t-1}), u_0 = 0 (t runs over the
 *   unit's tokens in order, r_max is the unit's largest score; the earliest
 *   window wins ties), and selection stops.  The envelope and the window
 *   sums are formed in double.
 *   embed       device [vocab][d] (dtype KVR_F32 or KVR_BF16).
 *   suffix_ids  device int32 [S]: token ids of the retained suffix, whose
 *               first token sits at global position suffix_start.
 *   query_ids   device int32 [Q], Q >= 1.
 *   unit_bounds device int32 [n_units + 1]: 0 = b_0 < b_1 < ... < b_n = S;
 *               unit k is suffix tokens [b_k, b_{k+1}).  Segmenting text into
 *               units happens before this call.
 *   workspace   device, >= kvr_sur_workspace_bytes(S, Q, d, n_units),
 *               256-byte aligned.
 *   positions_out device int32 [B]: the selected global positions,
 *               ascending (ready for kvr_select).  n_out (host) receives B.
 *   scores_out  device float [S] or NULL: the token scores r_i.
 * EINVAL on NULL arguments, budget_percent outside [0, 100] or a small
 * workspace; ERANGE when n_units > min(S, 65536).  Ids outside the
 * vocabulary and empty units are caught on the device and reported by
 * kvr_sur_status.  Enqueues only; synchronise the stream before reading.
 * ------------------------------------------------------------------------- */
size_t kvr_sur_workspace_bytes(int32_t S, int32_t Q, int32_t d, int32_t n_units);
kvr_status kvr_sur_select(const void* embed, int32_t vocab, int32_t d, int32_t dtype, const int32_t* suffix_ids,
                          int32_t S, int32_t suffix_start, const int32_t* query_ids, int32_t Q,
                          const int32_t* unit_bounds, int32_t n_units, int32_t budget_percent, void* workspace,
                          size_t ws_bytes, int32_t* positions_out, int32_t* n_out, float* scores_out,
                          void* stream);
/* Synchronise `stream` and report a device-side failure of the last
 * kvr_sur_select that used `workspace` (an id outside the vocabulary or a
 * malformed partition: EDEVICE), clearing it. */
kvr_status kvr_sur_status(void* workspace, void* stream);

/* ---------------------------------------------------------------------------
 * Layer-range policy of "CacheReforge: Bounded Recovery for Stale KV Caches
 * under Evolving Adapters" (Methodology: Layerwise Risk; Runtime risk and
 * range selection; Cache and anchor updates).  The adapter is one flat
 * parameter vector theta (n_params elements in device memory, the caller
 * packs its LoRA matrices into it).  Every cached layer keeps its own anchor,
 * the theta that produced its K/V, and a version number.
 * ------------------------------------------------------------------------- */
typedef struct kvr_policy kvr_policy;

/* updated module, for the restart layer r_KV(m, s) */
enum { KVR_MOD_Q = 0, KVR_MOD_K, KVR_MOD_V, KVR_MOD_O, KVR_MOD_MLP };

/* r_KV(m, s) (CacheReforge, supplementary Eq. S4): the first cache layer an
 * update of module m at layer s can change: s for K or V, min(s + 1, N) for
 * Q, O or the MLP; N (= n_layers) means no cached layer changes.
 * Returns -1 for an unknown module or s outside [0, n_layers). */
int32_t kvr_restart_layer(int32_t module, int32_t s, int32_t n_layers);

/* Layer sensitivities from a calibration split (CacheReforge, Eqs. 6-7), on
 * the host.  Condition i has restart layer restart[i], first safe window
 * window[i] (layers recomputed from restart[i]; 0 = direct reuse) and adapter
 * distance drift[i].  Layer l is labelled for i when
 * restart[i] <= l < restart[i] + window[i]; with D_l the labelled distances
 * (n_l of them, ascending), delta_l = max(D_l[floor(0.05 n_l)], 1e-12) and
 * s_l = 1 / delta_l, or 0 when D_l is empty.  s_out: host [n_layers].
 * EINVAL on NULL arrays, n_layers < 1, n_cond < 0, a negative window or
 * drift, or a restart outside [0, n_layers). */
kvr_status kvr_policy_sensitivity(int32_t n_layers, int32_t n_cond, const int32_t* restart,
                                  const int32_t* window, const double* drift, double* s_out);

/* Create a policy for n_layers cached layers.  theta0: device [n_params] in
 * `dtype` (KVR_F32 or KVR_BF16), the adapter that produced every layer's
 * cache (version 0); it is copied into each layer's anchor, which the policy
 * owns (n_layers * n_params elements of device memory).  sensitivity: host
 * [n_layers], s_l >= 0, copied.  Synchronous on `stream`. */
kvr_status kvr_policy_create(int32_t n_layers, int64_t n_params, int32_t dtype, const void* theta0,
                             const double* sensitivity, void* stream, kvr_policy** out);
kvr_status kvr_policy_destroy(kvr_policy* p);

/* Runtime risk and range (CacheReforge, Eqs. 8-9), synchronous:
 *   d_l = ||theta_t - anchor_l||_2 on the GPU (differences and squares in
 *   double, a fixed reduction order, so the result is deterministic);
 *   q_l = s_l * d_l; layer l triggers when q_l >= 1;
 *   b_t = 1 + max{l : q_l >= 1}.
 * The update is to module `module` at layer `update_layer` (the executable
 * restart r = update_layer).  The recovery range is [r, b_t).  It is empty
 * (range_out = {r, r}) when no layer triggers or when b_t <= r_KV(module,
 * update_layer): such a range replaces no affected K/V, which is reuse.
 *   theta_t: device [n_params], the policy's dtype.  drift_out, risk_out:
 *   host [n_layers], nullable.  range_out: host int32[2].
 * EINVAL on NULL theta_t/range_out or a bad module/layer. */
kvr_status kvr_policy_plan(kvr_policy* p, const void* theta_t, int32_t module, int32_t update_layer,
                           double* drift_out, double* risk_out, int32_t* range_out, void* stream);

/* Cache and anchor updates (CacheReforge): after layers [begin, end) were
 * recomputed under theta_t, their anchors become theta_t and their version
 * `version`; other layers keep their older anchors.  Enqueued on `stream`
 * (device copies); an empty range does nothing. */
kvr_status kvr_policy_commit(kvr_policy* p, const void* theta_t, int32_t begin, int32_t end, int64_t version,
                             void* stream);

/* Per-layer versions (host [n_layers]); synchronous. */
kvr_status kvr_policy_versions(kvr_policy* p, int64_t* versions);

/* Synchronise `stream` and report device-side failures recorded since the
 * last call (ETIMEOUT / EDEVICE), clearing them. */
kvr_status kvr_sync_status(kvr_cache* c, void* stream);

/* Message for the last failing call on this thread ("" if none). */
const char* kvr_last_error(void);

/* ---------------------------------------------------------------------------
 * kvr_wait_check -- a health check of the bounded device waits.  The pages
 * have no counterpart: every pipeline wait in the library's kernels (TMA
 * copies, tensor-core products, stage hand-offs) gives up after a cycle
 * budget and records a timeout instead of hanging the GPU.  This call runs
 * one thread block whose wait, with a budget of `cycles` SM clock cycles,
 * is on an mbarrier phase that nothing completes; when the budget runs out
 * it records the timeout in the cache's error word and returns, touching
 * nothing else (no copy or product is in flight).  kvr_sync_status then
 * reports ETIMEOUT.  cycles in [1, 2^31); EINVAL otherwise.
 * ------------------------------------------------------------------------- */
kvr_status kvr_wait_check(kvr_cache* c, int64_t cycles, void* stream);

/* ---------------------------------------------------------------------------
 * Inspection (synchronous; copies device state to host buffers).
 * kvr_read_selection: for sequence `seq` of the current selection:
 *   U        int32 [count]           sorted positions
 *   iv       int32 [n_intervals][2]  half-open intervals [a, b)
 *   sel, eloc, esnk  uint32 [ceil(capacity/32)]: selected, effective local,
 *            effective sink bit masks
 *   plan     int32 [n_tiles][6] (row0, nrows, u_min, u_max, n_full, n_total)
 *            over the attention kernel's query tiles of rows_per_tile rows and
 *            keys_per_tile keys; n_tiles/rows_per_tile/keys_per_tile returned.
 * Any output pointer may be NULL; caps bound what is written.
 * kvr_read_meta: local and sink masks [batch][ceil(capacity/32)].
 * ------------------------------------------------------------------------- */
kvr_status kvr_read_selection(kvr_cache* c, int32_t seq, int32_t* U, int32_t u_cap, int32_t* iv,
                              int32_t iv_cap, uint32_t* sel, uint32_t* eloc, uint32_t* esnk,
                              int32_t* plan, int32_t plan_cap, int32_t* n_tiles,
                              int32_t* rows_per_tile, int32_t* keys_per_tile);
kvr_status kvr_read_meta(kvr_cache* c, uint32_t* local_bits, uint32_t* sink_bits);
/* kvr_cache_info: the cache's current n_tokens and suffix_start (host state,
 * no device work).  Either pointer may be NULL. */
kvr_status kvr_cache_info(kvr_cache* c, int32_t* n_tokens, int32_t* suffix_start);

/* ---------------------------------------------------------------------------
 * Per-kernel timing.  When enabled, every launch of a library kernel on the
 * call's stream is bracketed by CUDA events; kvr_profile_read returns, per
 * kernel class (KVR_K_* below), the number of kernel launches (the attention
 * class counts its split merge too) and the summed device
 * time in milliseconds since the last read (synchronous), and resets them.
 * ------------------------------------------------------------------------- */
enum {
    KVR_K_SELECT = 0, KVR_K_GATHER, KVR_K_RMSNORM, KVR_K_GEMM_QKV, KVR_K_EPI_QKV,
    KVR_K_ATTN, KVR_K_GEMM_O, KVR_K_EPI_O, KVR_K_GEMM_GATEUP, KVR_K_EPI_GATEUP,
    KVR_K_GEMM_DOWN, KVR_K_EPI_DOWN, KVR_K_COMMIT, KVR_K_COUNT
};
kvr_status kvr_profile_enable(kvr_cache* c, int32_t enable);
kvr_status kvr_profile_read(kvr_cache* c, double* ms, int64_t* launches, int32_t n);

#ifdef __cplusplus
}
#endif
#endif /* KVR_H */
