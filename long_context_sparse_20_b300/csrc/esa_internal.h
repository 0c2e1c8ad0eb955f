// Internal launchers of libesa.so. Not part of the C ABI.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/esa.h"

namespace esa {

struct Shape {
    long long B, Tq, Tk, q_offset;
    int Hq, Hkv, D, H_I, D_I;
    int flags = 0;    // ESA_INDEXER_RELU | ESA_PER_HEAD_SETS
    int pos_div = 1;  // selection rows per query position (per-head sets: H_I)
};

inline bool relu_of(const Shape &s) { return (s.flags & ESA_INDEXER_RELU) != 0; }
inline bool per_head_of(const Shape &s) { return (s.flags & ESA_PER_HEAD_SETS) != 0; }

// The selection problem of a shape. With per-head sets every (query row,
// indexer head) pair is a row of its own: B x (Tq * H_I) rows of ONE indexer
// head (weight 1, see unit_weight), H_I consecutive rows per query position,
// whose idx/cnt rows are exactly the [B, Tq, H_I, K] / [B, Tq, H_I] layout.
inline Shape selection_rows(const Shape &s) {
    Shape r = s;
    if (per_head_of(s)) {
        r.Tq = s.Tq * s.H_I;
        r.pos_div = s.H_I;
        r.H_I = 1;
    }
    return r;
}
// Device address of an int32 holding 1 (the weight of a per-head row).
const int32_t *unit_weight();

struct DevInfo {
    int sms;
    size_t smem_optin;
};

// Immutable attributes of the current device (cached per device ordinal).
DevInfo device_info();

// Raise a kernel's dynamic shared-memory limit to at least `smem` on the
// current device (the attribute is set once per kernel, device and size).
bool ensure_smem(const void *fn, size_t smem);
// Resident blocks per SM for (kernel, threads, smem) on the current device,
// cached; 0 on failure.
int occupancy(const void *fn, int threads, size_t smem);

// Workspace carving: [0,256) status word area, then 256-aligned regions.
constexpr size_t kStatusBytes = 256;
inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// binaryVersion of the library's kernels on the current device (-1: not loadable)
int mix_binary_version();

// ---- cache append (k, v, kI rows of new positions; null pairs skipped) ---
cudaError_t launch_cache_append(const uint16_t *k_new, const uint16_t *v_new, const int8_t *kI_new, uint16_t *k,
                                uint16_t *v, int8_t *kI, const Shape &s, cudaStream_t st);

// ---- gate mix -----------------------------------------------------------
cudaError_t launch_gated_mix(const float *attn, const uint16_t *lin, const float *g, const uint8_t *head_mask,
                             const Shape &s, float *out, cudaStream_t st);

// ---- indexer scores (diagnostic) ----------------------------------------
cudaError_t launch_indexer_score(const int8_t *qI, const int8_t *kI, const int32_t *wI, const Shape &s,
                                 int32_t *scores, cudaStream_t st);

// ---- top-K selection ----------------------------------------------------
// Split plan: rows whose keys are spread over several co-resident blocks that
// meet at bounded inter-block barriers (few rows, long prefixes).
struct SplitPlan {
    bool ok;
    int chunks;         // blocks per row
    int grid;           // rows * chunks
    size_t smem;        // dynamic shared memory per block
    int stages;         // depth of the kI stage ring
    size_t hdr_off;     // workspace: call-counter header (zero before first use)
    size_t pub_off;     // per-block publications (written before read; no zeroing)
    size_t ctrl_off;    // per-row control state, two parities (zero before first use)
    size_t ctrl_bytes;
    int ctrl_rows_max;  // the most rows any split plan on this device uses
    size_t ws_bytes;
};
SplitPlan plan_split_select(const Shape &s, int K);
// ws_bytes: the workspace's size (bounds the control state a call may clear)
esa_status launch_split_select(const int8_t *qI, const int8_t *kI, const int32_t *wI, const Shape &s, int K,
                               int32_t *idx, int32_t *cnt, void *ws, size_t ws_bytes, const SplitPlan &plan,
                               cudaStream_t st);
// Bytes of persistent selection state (status, header, publications, the
// control rows of the most rows any split plan uses): scratch that other
// calls write fresh lies past this, so workspaces can be shared.
size_t split_state_max_bytes();

// The fused decode step: the split selection, then attention over each
// block's own selected keys, the row's partials merged after a second
// barrier, and the gate mix — one cooperative launch (few rows, long
// prefixes, one index set per row). idx/cnt may be null.
struct DecodePlan {
    bool ok;
    SplitPlan sel;     // the selection's plan (its stages and smem are the fused kernel's)
    int MPK, MTT, KG;  // m-tiles per key/value head, m-tiles, key groups of 8 per stage
    int sel_cap;       // entries of the block's selected-key list
    size_t off_q, off_sel, off_aux;  // dynamic shared memory offsets
    size_t part_off, ml_off;         // workspace: per-block partial outputs, (max, sum)
    size_t ws_bytes;
};
DecodePlan plan_decode_step(const Shape &s, int K);
esa_status launch_decode_step(const uint16_t *q, const uint16_t *k, const uint16_t *v, const int8_t *qI,
                              const int8_t *kI, const int32_t *wI, const Shape &s, int K, float scale, const float *g,
                              const uint16_t *lin, float *out, float *lse, int32_t *idx, int32_t *cnt, void *ws,
                              const DecodePlan &plan, cudaStream_t st);

// Row-tiled selection of many query rows. Writes idx/cnt when idx !=
// nullptr and the threshold form (T, P) of every row to thr (int32 pairs
// [rows][2]) when thr != nullptr. Workspace: [status word][tensor-core
// scratch]; ws_row_select() is the size that enables the tensor-core kernel
// (fp16 indexer keys and per-tile flags), and any smaller workspace of at
// least kStatusBytes runs the dp4a kernel alone.
size_t ws_row_select(const Shape &s, int K);
// With mask != nullptr the final pass also writes each row's selected keys
// as a bitmask, word-major: uint32 [sel_mask_words(s)][rows], bit j of
// word w of a row = key 32 w + j selected (keys past the row's prefix: 0;
// words past its last key tile: not written). Rows hold whole 128-key
// tiles: both selection kernels write a tile's words at once.
inline long long sel_mask_words(const Shape &s) { return 4 * ((s.Tk + 127) / 128); }
esa_status launch_row_select(const int8_t *qI, const int8_t *kI, const int32_t *wI, const Shape &s, int K,
                             int32_t *idx, int32_t *cnt, int32_t *thr, void *ws, size_t ws_bytes, cudaStream_t st,
                             uint32_t *mask = nullptr);
// The dp4a kernel (32 query rows per block); with only_flagged != nullptr
// it does only the 128-row query tiles whose flag is 1.
esa_status launch_rows_dp4a(const int8_t *qI, const int8_t *kI, const int32_t *wI, const Shape &s, int K,
                            int32_t *idx, int32_t *cnt, int32_t *thr, const int32_t *only_flagged, int32_t *status,
                            cudaStream_t st, uint32_t *mask = nullptr);

// ---- attention over gathered keys ---------------------------------------
struct AttnPlan {
    int gt;      // query heads per block (16, 32 or 64)
    int hg;      // head groups per key/value head
    int nsets;   // index sets per query row (1, or H_I with per-head sets)
    int hs;      // query heads per index set
    int seg;     // heads of one key/value head sharing one index set
    int gps;     // head groups per segment
    int var;     // kernel variant: 0 column split, 1 key split (16-head tiles), 2 keys as rows (<= 8 heads),
                 // 3 split index lists (the decode kernel, 8 warps over key slices)
    int splits;  // key splits per (row, kv head, head group)
    int keys_per_split;
    long long grid;
    size_t smem;
    size_t rec_bytes;  // the decode kernel's (max, sum) records (dec_rec_bytes; zero between calls)
    size_t x_bytes;    // the decode kernel's partial outputs
    size_t ws_bytes;   // status word + records + partials
};
AttnPlan plan_sparse_attn(const Shape &s, int K);
// Bytes of the decode kernel's records region on this device (the same for
// every shape, so that one region serves alternating shapes).
size_t dec_rec_bytes();
// The status word is at ws; the decode kernel's records at xrec and partials
// at xpart (defaults: ws + kStatusBytes, then + rec_bytes).
esa_status launch_sparse_attn(const uint16_t *q, const uint16_t *k, const uint16_t *v, const int32_t *idx,
                              const int32_t *cnt, const Shape &s, int K, float scale, const float *g,
                              const uint16_t *lin, float *out, float *lse, void *ws, const AttnPlan &plan,
                              cudaStream_t st, void *xrec = nullptr, void *xpart = nullptr);

// ---- routed (full | sparse per head) attention ---------------------------
size_t ws_routed(const Shape &s, int K);
// route == nullptr: every head sparse (the warp-specialised kernel only).
// idx/cnt (optional) receive the selection's index sets as well.
esa_status launch_routed_attn(const uint16_t *q, const uint16_t *k, const uint16_t *v, const int8_t *qI,
                              const int8_t *kI, const int32_t *wI, const uint8_t *route, const Shape &s, int K,
                              float scale, const float *g, const uint16_t *lin, float *out, void *ws,
                              cudaStream_t st, int32_t *idx = nullptr, int32_t *cnt = nullptr);

// tcgen05 routed attention (tensor-memory accumulators), given the threshold
// form (T, P) of every row's Top-K set in thr (int32 pairs [rows][2]).
esa_status launch_routed_tc(const uint16_t *q, const uint16_t *k, const uint16_t *v, const int8_t *qI,
                            const int8_t *kI, const int32_t *wI, const uint8_t *route, const int32_t *thr,
                            const Shape &s, float scale, const float *g, const uint16_t *lin, float *out,
                            int32_t *status, cudaStream_t st);

// Warp-specialised variant (two query tiles per CTA; TMA producer warp, MMA
// warp, two softmax warpgroups); routed_pp_supported() tells whether its
// buffers fit for this shape. Sparse heads mask with `mask`, the
// selection's bitmask of every row's selected keys (launch_row_select's
// mask output, word-major: [sel_mask_words][selection rows]).
// Its workspace (ws_routed_pp bytes): a flag word area and an fp16 copy of V.
bool routed_pp_supported(const Shape &s);
size_t ws_routed_pp(const Shape &s);
esa_status launch_routed_pp(const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint8_t *route,
                            const int32_t *thr, const uint32_t *mask, const Shape &s, float scale, const float *g,
                            const uint16_t *lin, float *out, void *pp_ws, int32_t *status, cudaStream_t st);

// ---- attention router (full or sparse per head) --------------------------
size_t ws_route_heads(const Shape &s);
esa_status launch_route_heads(const uint16_t *k, const float *W1, const float *b1, const float *W2, const float *b2,
                              const Shape &s, int hidden, uint8_t *route, float *margin, void *ws, cudaStream_t st);

// ---- KDA linear-attention branch ----------------------------------------
// ws == nullptr: the step-by-step kernels; otherwise (more than a few steps)
// the chunked form, whose chunk records take kda_chunked_ws_bytes() of ws
esa_status launch_kda(const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *alpha, const float *beta,
                      const float *state_in, long long B, long long T, int H, int Dk, int Dv, float scale, float *o,
                      uint16_t *lin, float *state_out, void *ws, cudaStream_t st);
bool kda_uses_chunks(long long T);
size_t kda_chunked_ws_bytes(long long B, long long T, int H, int Dk, int Dv);
esa_status launch_kda_chunked(const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *alpha,
                              const float *beta, const float *state_in, long long B, long long T, int H, int Dk,
                              int Dv, float scale, float *o, uint16_t *lin, float *state_out, void *ws,
                              cudaStream_t st);

// Wait limit for inter-block waits, in ns (ESA_WAIT_LIMIT_NS overrides) and
// the count of extra arrivals a barrier waits for (ESA_DEBUG_EXTRA_ARRIVALS;
// 0 normally — a positive value makes every barrier wait run out, which the
// timeout test uses).
long long wait_limit_ns();
int debug_extra_arrivals();

}  // namespace esa
