// Per-head routed attention: the launcher.
//
// Method ("Elastic Attention：动态路由优化大模型长文本处理", sections 2.2 and
// 3.1): each head runs either full or sparse attention, decided per head, in
// one fused launch whose blocks branch on the routing metadata. Sparse heads
// follow the Gated DSA path (indexer, top-K, attention over the selected
// keys, gate mix with the linear branch: "超大规模MoE架构中稀疏注意力机制的演进与实践",
// sections 二.1-二.3, 四.1).
//
// Two launches: the row-tiled selection reduces every query row's index set
// to its threshold form (T, P) — key j <= p is selected iff s_j > T, or
// s_j == T and j <= P, which is exactly the top-K set with ties to the lower
// position — and a tensor-core kernel runs every head (k_routed_pp.cu, warp-
// specialised over two query tiles, where its buffers fit; else k_routed_tc.cu),
// full and sparse, rebuilding the sparse heads' masks from exact indexer
// scores. For multi-head prefill at 64K tokens this moves 64 bytes of indexer
// key per key tile instead of gathering 512 bytes per selected key per head
// from a cache that L2 cannot hold.
#include "esa_device.cuh"
#include "esa_internal.h"

namespace esa {

// workspace: [row selection: status word, tensor-core scratch][thr][routed_pp: flag, fp16 values].
// With per-head index sets the selection runs on the per-head rows (one
// (T, P) per row and indexer head, [B, Tq, H_I, 2]).
// The selection's bitmask of every row's selected keys (the warp-specialised
// kernel masks sparse heads with it instead of recomputing indexer scores).
size_t routed_mask_bytes(const Shape &s) {
    const Shape r = selection_rows(s);
    return align256((size_t)(r.B * r.Tq) * (size_t)sel_mask_words(r) * 4);
}

size_t ws_routed(const Shape &s, int K) {
    const Shape r = selection_rows(s);
    return align256(ws_row_select(r, K)) + align256((size_t)r.B * r.Tq * 2 * 4) +
           (routed_pp_supported(s) ? align256(ws_routed_pp(s)) + routed_mask_bytes(s) : 0);
}

esa_status launch_routed_attn(const uint16_t *q, const uint16_t *k, const uint16_t *v, const int8_t *qI,
                              const int8_t *kI, const int32_t *wI, const uint8_t *route, const Shape &s, int K,
                              float scale, const float *g, const uint16_t *lin, float *out, void *ws,
                              cudaStream_t st, int32_t *idx, int32_t *cnt) {
    char *base = static_cast<char *>(ws);
    const Shape r = selection_rows(s);
    const size_t sel_bytes = align256(ws_row_select(r, K));
    int32_t *thr = reinterpret_cast<int32_t *>(base + sel_bytes);
    const int32_t *w = per_head_of(s) ? unit_weight() : wI;
    if (!w) return ESA_ERR_CUDA;
    const bool pp = routed_pp_supported(s);
    char *pp_ws = base + sel_bytes + align256((size_t)r.B * r.Tq * 2 * 4);
    uint32_t *mask = pp ? reinterpret_cast<uint32_t *>(pp_ws + align256(ws_routed_pp(s))) : nullptr;
    if (!pp && !route) return ESA_ERR_UNSUPPORTED;
    esa_status e = launch_row_select(qI, kI, w, r, K, idx, cnt, thr, ws, sel_bytes, st, mask);
    if (e != ESA_OK) return e;
    int32_t *status = reinterpret_cast<int32_t *>(ws);
    if (pp) return launch_routed_pp(q, k, v, route, thr, mask, s, scale, g, lin, out, pp_ws, status, st);
    if (per_head_of(s)) return ESA_ERR_UNSUPPORTED;  // the fallback kernel masks with one set per row
    return launch_routed_tc(q, k, v, qI, kI, wI, route, thr, s, scale, g, lin, out, status, st);
}

}  // namespace esa
