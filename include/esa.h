/*
 * esa.h — C ABI of the gated fine-grained sparse attention library (libesa.so).
 *
 * The method (sources named per call below):
 *   1. an Indexer scores each query against every causal-prefix key, without
 *      RoPE ("超大规模MoE架构中稀疏注意力机制的演进与实践", sections 二.1 and 二.2);
 *   2. a per-query Top-K keeps the K best positions (same page, section 二.1;
 *      "混合注意力架构演进…", section 三);
 *   3. K/V are gathered at those positions and exact softmax attention runs
 *      over them (the pseudo-code of section 四.1 of the first page; section
 *      三 of the second, softmax(Q K_sel^T / sqrt(d)) V_sel);
 *   4. a per-head gate mixes that output with a linear-attention branch,
 *      final = g*attn + (1-g)*linear_output (first page, sections 二.3, 四.1);
 *   5. optionally a per-head route sends each head to full causal attention or
 *      to the sparse path inside one launch ("Elastic Attention…", 2.2, 3.1);
 *      the route itself comes from a small MLP router (esa_route_heads);
 *   6. the linear branch that step 4 mixes in: KDA (esa_kda).
 *
 * Conventions shared by every call
 *   - Pointers named as tensors are DEVICE pointers owned by the caller; all
 *     tensors are dense, row-major, with the layouts stated below. bf16 data
 *     is passed as its 16-bit patterns (uint16_t).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream). Every call is asynchronous on it.
 *   - Host-detectable errors (null pointers, bad sizes, unsupported shapes,
 *     workspace too small) are returned before anything is launched.
 *   - Device-side errors never trap: kernels record the first error code in
 *     the workspace status word and return; read it with esa_read_status().
 *   - The library allocates no device memory at run time and keeps no
 *     state between calls beyond what this header names: the fixed scratch
 *     array of esa_topk_select_noalloc, and the side stream and events of
 *     esa_kda's chunked form (one set per host thread and device, created
 *     on first use and kept). It is thread-safe as long as concurrent calls
 *     use distinct workspaces.
 *   - Workspace: a caller-allocated device buffer of at least
 *     esa_workspace_size() bytes, 256-byte aligned, zero-filled once before
 *     its first use (esa_workspace_init). Calls leave it ready for the next
 *     call (they clear what they use), except after a device error, after
 *     which it must be re-initialised. Calls that share a workspace must not
 *     overlap in time (use one stream per workspace).
 *   - Decode-like calls (esa_topk_select, esa_sparse_attn,
 *     esa_gated_sparse_attn and esa_topk_select_noalloc on few rows with
 *     long prefixes) keep a small state between calls (a call counter,
 *     barrier counters, histograms; the attention's per-block ready
 *     records), each call clearing what the next one needs. Such calls may
 *     share one workspace (sized for the largest) across shapes. A
 *     workspace that any other call used since (another op, or a
 *     prefill-like shape) must be re-initialised with esa_workspace_init
 *     before the next decode-like call: their scratch may overlap that
 *     state. Stale state makes results wrong (or sets a status), never an
 *     out-of-bounds access.
 *
 * Shapes (esa_shape):
 *   B sequences; Tq query rows per sequence; Tk key positions per sequence;
 *   query row t sits at absolute position p = q_offset + t and its causal
 *   prefix is keys 0..p inclusive (n = p+1 keys). Prefill: Tq = Tk,
 *   q_offset = 0. Decode: Tq = 1, q_offset = Tk-1 (the cache already holds
 *   the new token). Chunked prefill: q_offset + Tq <= Tk.
 *   Hq query heads, Hkv key/value heads (Hq % Hkv == 0; query head h reads
 *   key/value head h / (Hq/Hkv)), head dim D in {64, 128};
 *   H_I indexer heads (1..16) of dim D_I in {16, 32, 64, 128}.
 *   flags: indexer options, 0 for the Gated DSA indexer (one index set per
 *   query row, scored by sum_h wI[h] * (qI[h] . kI), shared by every query
 *   head), or an OR of
 *     ESA_INDEXER_RELU   score by sum_h wI[h] * max(0, qI[h] . kI): a ReLU on
 *                        each indexer head's dot product (with one set per
 *                        head: max(0, qI[h] . kI));
 *     ESA_PER_HEAD_SETS  one index set per indexer head, scored by that head
 *                        alone and without its weight (the per-head
 *                        [batch, heads, top_k] index shape of the Gated DSA
 *                        page's pseudo-code, section 四.1); query head h
 *                        attends to the set of indexer head h / (Hq/H_I),
 *                        which needs Hq % H_I == 0 and, for attention, one of
 *                        Hq/H_I and Hq/Hkv to divide the other. The routed
 *                        call masks each sparse head with its own set (on its
 *                        warp-specialised kernel; shapes it does not fit
 *                        return ESA_ERR_UNSUPPORTED).
 *
 * Tensor layouts:
 *   qI  int8  [B, Tq, H_I, D_I]     indexer queries
 *   kI  int8  [B, Tk, D_I]          indexer keys, one per position, shared by
 *                                    all indexer heads
 *   wI  int32 [H_I]                 indexer head weights
 *   q   bf16  [B, Tq, Hq, D]
 *   k,v bf16  [B, Tk, Hkv, D]
 *   idx int32 [B, Tq, top_k]        selected positions, ascending, -1 padded
 *                                    ([B, Tq, H_I, top_k] with per-head sets)
 *   cnt int32 [B, Tq]               min(top_k, p+1) ([B, Tq, H_I] with per-head sets)
 *   g   fp32  [Hq]                  gate, already in (0,1)
 *   lin bf16  [B, Tq, Hq, D]        linear-attention branch output
 *   out fp32  [B, Tq, Hq, D]
 *   lse fp32  [B, Tq, Hq]           natural-log sum-exp of the scaled logits
 *   route uint8 [B, Hq]             1 = sparse head, 0 = full head
 */
#ifndef ESA_H
#define ESA_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define ESA_API __attribute__((visibility("default")))
#else
#define ESA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t esa_status;

#define ESA_OK 0
#define ESA_ERR_INVALID 1     /* bad argument (null pointer, size, shape, top_k) */
#define ESA_ERR_UNSUPPORTED 2 /* well-formed but outside what this build handles */
#define ESA_ERR_CUDA 3        /* a CUDA runtime call failed (launch, copy, sync) */
#define ESA_ERR_TIMEOUT 4     /* device: a bounded inter-block wait gave up */
#define ESA_ERR_BAD_INDEX 5   /* device: an index outside the causal prefix, or cnt
                                 outside 0..min(top_k, p+1); the row is skipped */
#define ESA_ERR_WORKSPACE 6   /* workspace null, misaligned or too small */
#define ESA_ERR_INTERNAL 7    /* device: a kernel's own consistency check failed; the
                                 outputs of that call are not valid */

typedef struct esa_shape {
    int64_t B;
    int64_t Tq;
    int64_t Tk;
    int64_t q_offset;
    int32_t Hq;
    int32_t Hkv;
    int32_t D;
    int32_t H_I;
    int32_t D_I;
    int32_t flags; /* ESA_INDEXER_RELU | ESA_PER_HEAD_SETS, or 0 */
} esa_shape;

#define ESA_INDEXER_RELU 1
#define ESA_PER_HEAD_SETS 2

/* Operation ids for esa_workspace_size. */
#define ESA_OP_INDEXER_SCORE 0
#define ESA_OP_TOPK_SELECT 1
#define ESA_OP_SPARSE_ATTN 2
#define ESA_OP_GATED_MIX 3
#define ESA_OP_ROUTED_ATTN 4
#define ESA_OP_ROUTE_HEADS 5
#define ESA_OP_TOPK_THRESHOLD 6
#define ESA_OP_GATED_SPARSE_ATTN 7

/* Bytes of workspace that `op` needs for shape `s` and `top_k` (0 when the
 * op needs none beyond the status word, which every op may write; the
 * minimum returned is 256). Returns 0 for an invalid op or shape. */
ESA_API size_t esa_workspace_size(int op, const esa_shape *s, int top_k);

/* Zero-fill a workspace (cudaMemsetAsync on `stream`). Needed once before
 * first use and after any device error. */
ESA_API esa_status esa_workspace_init(void *ws, size_t ws_bytes, void *stream);

/* Indexer scores (Gated DSA page, section 二.1: the query's relevance to every
 * history position; section 二.2: no RoPE):
 *   scores[b,t,j] = sum_h wI[h] * sum_c qI[b,t,h,c] * kI[b,j,c]   for j <= p,
 *   scores[b,t,j] = INT32_MIN                                      for j > p.
 * With ESA_INDEXER_RELU each head's dot product is max(0, .) before the
 * weighted sum; with ESA_PER_HEAD_SETS the scores are per indexer head,
 * scores[b,t,h,j] = (max(0, .) of) sum_c qI[b,t,h,c] * kI[b,j,c], int32
 * [B, Tq, H_I, Tk].
 * scores int32 [B, Tq, Tk] (a diagnostic: the selection never materialises
 * this). Every score must fit in int32, which holds when
 * sum_h |wI[h]| * D_I * 16384 < 2^31. */
ESA_API esa_status esa_indexer_score(const int8_t *qI, const int8_t *kI, const int32_t *wI, const esa_shape *s,
                             int32_t *scores, void *ws, size_t ws_bytes, void *stream);

/* Top-K selection (Gated DSA page, section 二.1, K = 2048 in its setting;
 * the hybrid-architecture page, section 三: idx = topk(indexer_score(Q,K))).
 * For each query row: the min(top_k, p+1) positions j <= p with the largest
 * indexer score, ties going to the lower position, written ascending to
 * idx[b,t,:], -1 padded; cnt[b,t] = min(top_k, p+1). Exact (integer) and
 * deterministic. top_k in 1..65536. The full score row is never written to
 * device memory. */
ESA_API esa_status esa_topk_select(const int8_t *qI, const int8_t *kI, const int32_t *wI, const esa_shape *s, int top_k,
                           int32_t *idx, int32_t *cnt, void *ws, size_t ws_bytes, void *stream);

/* Attention over the selected keys (Gated DSA pseudo-code, section 四.1:
 * gather then scaled_dot_product_attention; hybrid page, section 三). For
 * each row and query head h (key/value head kh = h / (Hq/Hkv)):
 *   l_j = scale * q[b,t,h,:] . k[b,j,kh,:]  over j in idx[b,t,0..cnt-1],
 *   o   = sum_j softmax(l)_j v[b,j,kh,:],   lse = log sum_j exp(l_j),
 *   out = g[h]*o + (1-g[h])*lin[b,t,h,:]    when g and lin are both given
 *         (the gate mix of sections 二.3/四.1, fused), else out = o.
 * fp32 accumulation, fp32 output. scale is normally 1/sqrt(D). g, lin and
 * lse may be NULL (g and lin together). A row with cnt = 0 gets out = 0 (or
 * the linear branch share when gated) and lse = -inf. Indices outside
 * 0..p, or cnt outside 0..min(top_k, p+1), set ESA_ERR_BAD_INDEX in the
 * status word; the offending row is left unwritten. Rows whose index list
 * is split over several blocks (few rows: decode) exchange partial results
 * through the workspace and wait for one another with a bounded wait
 * (ESA_ERR_TIMEOUT when it runs out, the rows left unwritten). */
ESA_API esa_status esa_sparse_attn(const uint16_t *q, const uint16_t *k, const uint16_t *v, const int32_t *idx,
                           const int32_t *cnt, const esa_shape *s, int top_k, float scale, const float *g,
                           const uint16_t *lin, float *out, float *lse, void *ws, size_t ws_bytes, void *stream);

/* The whole gated sparse path in one call: the Gated DSA pseudo-code's
 * gated_sparse_attention(query, history_keys, history_values, top_k) (first
 * page, section 四.1; sections 二.1-二.3): indexer scores, per-row top-K,
 * attention over the gathered keys, gate mix. Computes exactly what
 * esa_topk_select followed by esa_sparse_attn computes (same index sets,
 * outputs within the same tolerance of the exact result), and writes the
 * index sets to idx/cnt when they are given (both or neither; layouts as
 * esa_topk_select's).
 * It runs the selection kernel and the gathered-attention kernel back to
 * back on `stream` (the attention launched early on the programmatic
 * edge). Prefill-like shapes whose causal prefixes hold at most 12 times
 * the selected keys (summed over the rows) and whose buffers fit the routed
 * kernel, called without lse, run esa_routed_attn's path instead with every
 * head sparse: the selection also writes its bitmask of selected keys and
 * the attention masks dense tiles on the tensor cores (same index sets,
 * outputs within the same tolerance). With the environment variable
 * ESA_DECODE_PATH=fused, decode-like
 * shapes (few rows, long prefixes: B*Tq up to half the SMs, one index set
 * per row, D in {64, 128}, (Hq/Hkv rounded up to 16) * Hkv up to 128
 * query-head rows) take ONE cooperative launch instead: each block scores
 * its span of the cache, the row's blocks agree on the threshold, each
 * block attends over its own selected keys, and their partial softmax
 * results are merged inside the same launch. Both give the same index sets
 * and outputs within the same tolerance; the two launches are the default
 * because they measured faster on B300. Workspace:
 * esa_workspace_size(ESA_OP_GATED_SPARSE_ATTN, s, top_k) bytes. g, lin, lse
 * nullable as in esa_sparse_attn; idx, cnt nullable. */
ESA_API esa_status esa_gated_sparse_attn(const uint16_t *q, const uint16_t *k, const uint16_t *v, const int8_t *qI,
                                         const int8_t *kI, const int32_t *wI, const esa_shape *s, int top_k,
                                         float scale, const float *g, const uint16_t *lin, float *out, float *lse,
                                         int32_t *idx, int32_t *cnt, void *ws, size_t ws_bytes, void *stream);

/* Gate mix on its own (Gated DSA page, sections 二.3 and 四.1 step 5):
 *   out[b,t,h,:] = g[h]*attn[b,t,h,:] + (1-g[h])*lin[b,t,h,:]
 * for heads with head_mask[b,h] != 0 (all heads when head_mask is NULL);
 * other heads copy attn. attn/out fp32 [B,Tq,Hq,D] (out may alias attn),
 * lin bf16 [B,Tq,Hq,D], g fp32 [Hq], head_mask uint8 [B,Hq]. */
ESA_API esa_status esa_gated_mix(const float *attn, const uint16_t *lin, const float *g, const uint8_t *head_mask,
                         const esa_shape *s, float *out, void *stream);

/* Per-head routed attention (Elastic Attention page, sections 2.2 and 3.1:
 * each head runs either full or sparse attention, decided per head, inside
 * one fused kernel). route[b,h] = 0: exact causal attention over all keys
 * 0..p, output without the gate. route[b,h] = 1: the sparse path — the
 * index set of esa_topk_select (one set per (b,t), shared by all sparse
 * heads; with ESA_PER_HEAD_SETS the set of indexer head h / (Hq/H_I)),
 * attention over it, then the gate mix with lin when g and lin are
 * given. Every head of the layer runs in one attention launch (on the
 * tensor cores, accumulators in tensor memory); the selection before it
 * leaves every row's selected keys as a bitmask in the workspace (about
 * B*Tq*Tk/8 bytes, times H_I with per-head sets), which the sparse heads
 * mask with. scale is normally 1/sqrt(D). */
ESA_API esa_status esa_routed_attn(const uint16_t *q, const uint16_t *k, const uint16_t *v, const int8_t *qI,
                           const int8_t *kI, const int32_t *wI, const uint8_t *route, const esa_shape *s, int top_k,
                           float scale, const float *g, const uint16_t *lin, float *out, void *ws, size_t ws_bytes,
                           void *stream);

/* The threshold form of every query row's Top-K set: the selection step of
 * esa_routed_attn, whose sparse heads rebuild their index set from it inside
 * the fused attention launch (Elastic Attention page, section 3.1; the set
 * itself is the Gated DSA page's top-K, section 二.1). For each row, with s_j
 * the indexer score of esa_indexer_score and n = p+1:
 *   n <= top_k:  thr[b,t,0] = INT32_MIN, thr[b,t,1] = p   (the whole prefix);
 *   otherwise:   order the positions 0..p by (score descending, position
 *                ascending); thr[b,t,0] = T, the score of the top_k-th of
 *                that order, and thr[b,t,1] = P, its position.
 * Key j <= p is in the row's set iff s_j > T, or s_j == T and j <= P: the
 * same set as esa_topk_select's idx row. thr int32 [B, Tq, 2], or
 * [B, Tq, H_I, 2] with ESA_PER_HEAD_SETS (each set scored by its own
 * indexer head, as esa_topk_select's per-head rows).
 * Workspace esa_workspace_size(ESA_OP_TOPK_THRESHOLD, s, top_k) bytes;
 * the same kernels and workspace layout as the routed call's selection. */
ESA_API esa_status esa_topk_threshold(const int8_t *qI, const int8_t *kI, const int32_t *wI, const esa_shape *s,
                                      int top_k, int32_t *thr, void *ws, size_t ws_bytes, void *stream);

/* Attention router (Elastic Attention page, section 2.2: a lightweight
 * 2-layer MLP on the current key hidden states decides, per attention head,
 * full or sparse attention; its decisions are the routing metadata of
 * esa_routed_attn). Per sequence b, with C = Hkv*D:
 *   x[c]   = (1/Tk) * sum_{j<Tk} k[b, j, c/D, c%D]         (mean key state)
 *   hid[f] = max(0, b1[f] + sum_c W1[f, c] * x[c])          f < hidden
 *   z_o    = b2[2h+o] + sum_f W2[2h+o, f] * hid[f]           o = 0 full, 1 sparse
 *   route[b, h] = 1 (sparse) iff z_1 >= z_0, else 0 (full); margin[b, h] = z_1 - z_0.
 * k bf16 [B, Tk, Hkv, D]; W1 fp32 [hidden, C]; b1 fp32 [hidden]; W2 fp32
 * [2*Hq, hidden]; b2 fp32 [2*Hq]; route uint8 [B, Hq]; margin fp32 [B, Hq]
 * or NULL. hidden in 1..4096. Sums in fp32 in a fixed order: the same inputs give the same bits
 * on every call. Device memory owned by the caller; workspace
 * esa_workspace_size(ESA_OP_ROUTE_HEADS, s, hidden) bytes. */
ESA_API esa_status esa_route_heads(const uint16_t *k, const float *W1, const float *b1, const float *W2,
                                   const float *b2, const esa_shape *s, int hidden, uint8_t *route, float *margin,
                                   void *ws, size_t ws_bytes, void *stream);

/* The linear-attention branch (KDA) whose output is the gate mix's `lin`.
 * The Gated DSA page (sections 一, 二.3 and 三) keeps KDA, a gated linear
 * attention that folds the history into a recurrent state, beside the sparse
 * attention and mixes the two outputs; it prints no formula, and this call
 * computes the published Kimi Delta Attention recurrence. Per sequence b and
 * head h, a state S of Dk x Dv values (row i: key channel i) starts from
 * state_in (or zero when state_in is NULL) and for t = 0 .. T-1:
 *   S[i][c] *= alpha[b,t,h,i]                         (forgetting, per key channel)
 *   u[c]     = sum_i k[b,t,h,i] S[i][c]
 *   S[i][c] += beta[b,t,h] k[b,t,h,i] (v[b,t,h,c] - u[c])   (delta rule)
 *   o[b,t,h,c] = scale * sum_i q[b,t,h,i] S[i][c]
 * The final S goes to state_out (NULL: dropped). Chunked prefill and decode
 * carry the state across calls (state_out may be the same buffer as
 * state_in); T = 0 copies state_in to state_out.
 *   q, k   bf16 [B, T, H, Dk]      (the model normally gives unit-norm keys)
 *   v      bf16 [B, T, H, Dv]
 *   alpha  fp32 [B, T, H, Dk]      forgetting factors, normally in (0, 1]
 *   beta   fp32 [B, T, H]          write strengths, normally in [0, 1]
 *   state_in, state_out  fp32 [B, H, Dk, Dv]
 *   o      fp32 [B, T, H, Dv] or NULL
 *   lin    bf16 [B, T, H, Dv] or NULL: o rounded to bf16, the input of
 *          esa_gated_mix / esa_sparse_attn when H = Hq and Dv = D
 * Dk in {64, 128}; Dv a multiple of 16 in 16..512 (else ESA_ERR_UNSUPPORTED);
 * B, H <= 65535. q, k, v, alpha, state_in, state_out and o 16-byte aligned,
 * lin 8-byte, beta 4-byte (else ESA_ERR_INVALID). o and lin must not overlap
 * any input. fp32 arithmetic in a fixed order (deterministic).
 * Workspace (optional): with ws == NULL the steps run one after another on
 * the state, and no device-side error is possible. With ws != NULL and
 * T > 4, the call takes the chunked form: the steps in chunks of 16, each
 * chunk's couplings computed for all chunks at once, then the state carried
 * from chunk to chunk by a few small matrix products (the same results up to
 * fp32 rounding order). A chunk whose cumulative forgetting factor leaves
 * [2^-60, 2^60] for some key channel runs its steps one by one. ws must then
 * hold esa_kda_workspace_size() bytes and be 256-byte aligned (else
 * ESA_ERR_WORKSPACE); it needs no initialisation. Its first word is a status
 * word that the call clears first: a bounded device wait for a chunk's data
 * that runs out sets ESA_ERR_TIMEOUT there (read it with esa_read_status)
 * and leaves that block's outputs unwritten. T <= 4 never uses ws.
 * Streams: a call of more than 256 chunks (4096 steps) carries the state
 * through each 256 chunks on a second stream of this library's own (one per
 * host thread and device, at the device's greatest priority, created on
 * first use and kept) while `stream` computes the next 256 chunks'
 * couplings; event edges join the two, and `stream` waits for the last
 * carry, so the call is ordered on `stream` as any other and may be captured
 * in a CUDA graph. */
ESA_API esa_status esa_kda(const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *alpha,
                           const float *beta, const float *state_in, int64_t B, int64_t T, int32_t H, int32_t Dk,
                           int32_t Dv, float scale, float *o, uint16_t *lin, float *state_out, void *ws,
                           size_t ws_bytes, void *stream);

/* Bytes of workspace esa_kda() needs for its chunked form at this shape: a
 * status word, one record of fp32 matrices per (sequence, head, chunk of 16
 * steps) for at most 256 chunks at a time, and when there are more chunks a
 * carried state and a second set of records (one set filled while the other
 * is read); 0 when T <= 4 or the shape is not supported. */
ESA_API size_t esa_kda_workspace_size(int64_t B, int64_t T, int32_t H, int32_t Dk, int32_t Dv);

/* Top-K selection without a caller workspace. The pages have no counterpart
 * to this call: it is a convenience of this library.
 *
 * For callers that cannot allocate device memory themselves — code running
 * inside a runtime that owns every device allocation (a framework's caching
 * allocator, a serving engine with a reserved memory pool) and may not call
 * cudaMalloc. Same inputs, outputs and results as esa_topk_select(), but the
 * scratch state (status word, barrier counters, histograms) lives in one
 * fixed device array inside this library, ESA_NOALLOC_SCRATCH_BYTES large,
 * which every GPU that loads the library holds until the process exits. The
 * call itself allocates nothing (no cudaMalloc or cudaFree).
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture on the device.
 *   - Shapes whose scratch would exceed ESA_NOALLOC_SCRATCH_BYTES return
 *     ESA_ERR_UNSUPPORTED. The limit counts selection rows: B*Tq, times H_I
 *     with ESA_PER_HEAD_SETS. A decode batch whose selection spreads over
 *     the SMs (at most half as many rows as SMs) fits with up to about 26
 *     selection rows on a 148-SM GPU (per-block published counts, ~4.9 MB,
 *     plus ~128 KB of control state per row); shapes that take the
 *     row-tiled selection (prefill, long batches) need only the status word
 *     and fit at any size.
 *   - Every call shares the one array: it clears the parts that must start
 *     at zero on `stream` before launching, and calls whose GPU work overlaps
 *     in time (different streams, or several host threads) race on it.
 *   - dev_status (nullable): a caller-owned device int32 that receives this
 *     call's device status code (ESA_OK, ESA_ERR_TIMEOUT, ...), copied on
 *     `stream` after the kernel. */
#define ESA_NOALLOC_SCRATCH_BYTES (8u << 20)
ESA_API esa_status esa_topk_select_noalloc(const int8_t *qI, const int8_t *kI, const int32_t *wI, const esa_shape *s,
                                           int top_k, int32_t *idx, int32_t *cnt, int32_t *dev_status, void *stream);

/* Synchronise `stream`, read the workspace status word into *dev_status
 * (ESA_OK when no kernel recorded an error) and clear it. Returns ESA_OK, or
 * ESA_ERR_CUDA when the synchronisation or the copy failed. */
ESA_API esa_status esa_read_status(void *ws, void *stream, int32_t *dev_status);

/* Write a step's new key rows into the caches: for b < B and t < Tq,
 *   k[b, q_offset + t, :, :] = k_new[b, t, :, :]   (k_new, v_new bf16 [B, Tq, Hkv, D])
 *   v[b, q_offset + t, :, :] = v_new[b, t, :, :]
 *   kI[b, q_offset + t, :]   = kI_new[b, t, :]     (kI_new int8 [B, Tq, D_I])
 * with the caches in the layouts above: a decode step appends Tq = 1
 * position at q_offset = Tk - 1 before its selection reads the cache (the
 * key cache is the "history_keys" the Gated DSA pseudo-code indexes,
 * section 四.1). One launch writes all three; a cache whose pointer and new
 * rows are both NULL is skipped (one without the other is an error). All
 * pointers 16-byte aligned; new rows must not overlap the caches. Device
 * memory owned by the caller; no workspace. */
ESA_API esa_status esa_cache_append(const uint16_t *k_new, const uint16_t *v_new, const int8_t *kI_new, uint16_t *k,
                                    uint16_t *v, int8_t *kI, const esa_shape *s, void *stream);

/* A static, human-readable name for a status code. */
ESA_API const char *esa_status_string(esa_status st);

/* The compute capability the library's kernels were compiled for, as the
 * CUDA runtime reports it for the current device (cudaFuncAttributes
 * binaryVersion of one of its kernels: 103 for sm_103a), or -1 when the
 * runtime cannot load them (no device, or a device they were not built
 * for). */
ESA_API int esa_binary_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ESA_H */
