// extern "C" entry points of libesa.so: argument checks, workspace planning
// and dispatch to the kernels. See include/esa.h for the contract.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <tuple>

#include "esa_internal.h"

namespace esa {

DevInfo device_info() {
    static std::mutex mu;
    static DevInfo cache[64];
    static bool have[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lk(mu);
    if (dev >= 0 && dev < 64 && have[dev]) return cache[dev];
    DevInfo di{};
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    di.sms = v > 0 ? v : 1;
    cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    di.smem_optin = (size_t)v;
    if (dev >= 0 && dev < 64) {
        cache[dev] = di;
        have[dev] = true;
    }
    return di;
}

bool ensure_smem(const void *fn, size_t smem) {
    static std::mutex mu;
    static std::map<std::pair<int, const void *>, size_t> set_to;
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lk(mu);
    auto key = std::make_pair(dev, fn);
    auto it = set_to.find(key);
    if (it != set_to.end() && it->second >= smem) return true;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    set_to[key] = smem;
    return true;
}

int occupancy(const void *fn, int threads, size_t smem) {
    static std::mutex mu;
    static std::map<std::tuple<int, const void *, int, size_t>, int> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    auto key = std::make_tuple(dev, fn, threads, smem);
    {
        std::lock_guard<std::mutex> lk(mu);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    if (!ensure_smem(fn, smem)) return 0;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, threads, smem) != cudaSuccess) {
        cudaGetLastError();
        per_sm = 0;
    }
    std::lock_guard<std::mutex> lk(mu);
    cache[key] = per_sm;
    return per_sm;
}

long long wait_limit_ns() {
    const char *e = getenv("ESA_WAIT_LIMIT_NS");
    long long v = e ? atoll(e) : 0;
    return v > 0 ? v : 1000000000ll;  // 1 s
}

int debug_extra_arrivals() {
    const char *e = getenv("ESA_DEBUG_EXTRA_ARRIVALS");
    int v = e ? atoi(e) : 0;
    return v > 0 ? v : 0;
}

namespace {
__device__ int32_t g_unit_weight = 1;
}  // namespace

const int32_t *unit_weight() {
    static std::mutex mu;
    static const int32_t *cache[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lk(mu);
    if (dev >= 0 && dev < 64 && cache[dev]) return cache[dev];
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_unit_weight) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (dev >= 0 && dev < 64) cache[dev] = static_cast<const int32_t *>(p);
    return static_cast<const int32_t *>(p);
}

}  // namespace esa

using namespace esa;

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shape checks common to every call; `need_attn` adds the attention fields,
// `need_index` the indexer fields.
esa_status check_shape(const esa_shape *s, bool need_attn, bool need_index) {
    if (!s) return ESA_ERR_INVALID;
    if (s->B < 0 || s->Tq < 0 || s->Tk < 0 || s->q_offset < 0) return ESA_ERR_INVALID;
    if (s->q_offset + s->Tq > s->Tk) return ESA_ERR_INVALID;
    if (s->Tk > (int64_t)INT32_MAX) return ESA_ERR_UNSUPPORTED;
    if (need_attn) {
        if (s->Hq <= 0 || s->Hkv <= 0 || s->Hq % s->Hkv) return ESA_ERR_INVALID;
        if (s->D != 64 && s->D != 128) return ESA_ERR_UNSUPPORTED;
    }
    if (need_index) {
        if (s->H_I <= 0 || s->H_I > 16) return ESA_ERR_UNSUPPORTED;
        if (s->D_I != 16 && s->D_I != 32 && s->D_I != 64 && s->D_I != 128) return ESA_ERR_UNSUPPORTED;
    }
    if (s->flags & ~(ESA_INDEXER_RELU | ESA_PER_HEAD_SETS)) return ESA_ERR_INVALID;
    if ((s->flags & ESA_PER_HEAD_SETS) && (s->H_I <= 0 || s->H_I > 16)) return ESA_ERR_UNSUPPORTED;
    if ((s->flags & ESA_PER_HEAD_SETS) && need_attn) {
        // query head h attends to set h / (Hq/H_I); a block of heads that
        // shares one gather must lie in one set and one key/value head
        if (s->Hq % s->H_I) return ESA_ERR_INVALID;
        const int hs = s->Hq / s->H_I, G = s->Hq / s->Hkv;
        if (hs % G && G % hs) return ESA_ERR_UNSUPPORTED;
    }
    return ESA_OK;
}

Shape to_shape(const esa_shape *s) {
    Shape x;
    x.B = s->B;
    x.Tq = s->Tq;
    x.Tk = s->Tk;
    x.q_offset = s->q_offset;
    x.Hq = s->Hq;
    x.Hkv = s->Hkv;
    x.D = s->D;
    x.H_I = s->H_I;
    x.D_I = s->D_I;
    x.flags = s->flags;
    x.pos_div = 1;
    return x;
}

esa_status check_ws(void *ws, size_t ws_bytes, size_t need) {
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return ESA_ERR_WORKSPACE;
    if (ws_bytes < need) return ESA_ERR_WORKSPACE;
    return ESA_OK;
}

size_t topk_ws(const Shape &s, int K) {
    const Shape r = selection_rows(s);
    SplitPlan sp = plan_split_select(r, K);
    size_t w = sp.ok ? sp.ws_bytes : ws_row_select(r, K);
    return w < kStatusBytes ? kStatusBytes : w;
}

// The single-launch decode step (selection, attention and merge in one
// cooperative kernel) is taken only when ESA_DECODE_PATH=fused: measured on
// B300 it is slower than the selection kernel followed by the gathered
// attention kernel (launched early on the programmatic edge), so the two
// launches are the default. Both give the same index sets and outputs
// within the same tolerance.
bool decode_single_launch() {
    const char *e = getenv("ESA_DECODE_PATH");
    return e && strcmp(e, "fused") == 0;
}

// The two-launch path's layout: the selection's own workspace and any
// shape's persistent selection state, the attention's records region (the
// same offset for every decode-like shape), then idx/cnt room and the
// attention's partials.
size_t gated_rec_off(const Shape &x, int K) { return align256(std::max(topk_ws(x, K), split_state_max_bytes())); }
size_t gated_scratch_off(const Shape &x, int K) { return gated_rec_off(x, K) + dec_rec_bytes(); }

// Workspace of esa_gated_sparse_attn: the fused step's, or for the two
// launches the selection's workspace plus room for idx/cnt when the caller
// passes none.
// The attention's exchange area follows.
size_t gated_xoff(const Shape &x, int K) {
    const Shape r = selection_rows(x);
    const size_t sets = (size_t)(r.B * r.Tq);
    return gated_scratch_off(x, K) + align256(sets * K * 4) + align256(sets * 4);
}
// Prefill-like shapes (not the split selection's) whose dense masked
// attention visits at most kRoutedPairRatio times the selected pairs run
// the selection with its bitmask output and the routed kernel with every
// head sparse: on the tensor cores that beats gathering the selected keys
// (long prefill, S = 32768, K = 2048: 8.1x the pairs, 7.96 against 9.76 ms;
// a 16K chunk over a 131072-key cache: 60x, 27.1 against 8.35 ms).
constexpr double kRoutedPairRatio = 12.0;
bool gated_routed_path(const Shape &x, int K) {
    if (plan_split_select(selection_rows(x), K).ok || !routed_pp_supported(x)) return false;
    // per sequence: sum over rows of (p + 1) and of min(K, p + 1), p = q_offset + t
    const double Tq = (double)x.Tq, qo = (double)x.q_offset;
    const double dense = Tq * qo + Tq * (Tq + 1) / 2;
    const double ts = std::min(Tq, std::max(0.0, (double)K - qo));  // rows whose whole prefix is kept
    const double sel = ts * qo + ts * (ts + 1) / 2 + (Tq - ts) * K;
    return sel > 0 && dense <= kRoutedPairRatio * sel;
}

size_t gated_ws(const Shape &x, int K) {
    DecodePlan dp = decode_single_launch() ? plan_decode_step(x, K) : DecodePlan{};
    if (dp.ok) return dp.ws_bytes;
    const size_t two = gated_xoff(x, K) + align256(plan_sparse_attn(x, K).x_bytes);
    return gated_routed_path(x, K) ? std::max(two, ws_routed(x, K)) : two;
}

}  // namespace

extern "C" {

size_t esa_workspace_size(int op, const esa_shape *s, int top_k) {
    bool attn = op == ESA_OP_SPARSE_ATTN || op == ESA_OP_ROUTED_ATTN || op == ESA_OP_GATED_MIX;
    bool index = op == ESA_OP_INDEXER_SCORE || op == ESA_OP_TOPK_SELECT || op == ESA_OP_ROUTED_ATTN;
    if (op == ESA_OP_TOPK_THRESHOLD) {
        if (check_shape(s, false, true) != ESA_OK || top_k <= 0) return 0;
        const size_t w = ws_row_select(selection_rows(to_shape(s)), top_k);
        return w < kStatusBytes ? kStatusBytes : w;
    }
    if (op == ESA_OP_GATED_SPARSE_ATTN) {
        if (check_shape(s, true, true) != ESA_OK || top_k <= 0) return 0;
        return gated_ws(to_shape(s), top_k);
    }
    if (op == ESA_OP_ROUTE_HEADS) {
        if (check_shape(s, true, false) != ESA_OK) return 0;
        return ws_route_heads(to_shape(s));
    }
    if (op < 0 || op > 4 || check_shape(s, attn, index) != ESA_OK) return 0;
    if ((op == ESA_OP_TOPK_SELECT || op == ESA_OP_SPARSE_ATTN || op == ESA_OP_ROUTED_ATTN) && top_k <= 0) return 0;
    Shape x = to_shape(s);
    switch (op) {
        case ESA_OP_TOPK_SELECT: return topk_ws(x, top_k);
        case ESA_OP_SPARSE_ATTN: return plan_sparse_attn(x, top_k).ws_bytes;
        case ESA_OP_ROUTED_ATTN: return ws_routed(x, top_k);
        default: return kStatusBytes;
    }
}

esa_status esa_workspace_init(void *ws, size_t ws_bytes, void *stream) {
    if (!ws || ws_bytes == 0) return ESA_ERR_WORKSPACE;
    return cudaMemsetAsync(ws, 0, ws_bytes, (cudaStream_t)stream) == cudaSuccess ? ESA_OK : ESA_ERR_CUDA;
}

esa_status esa_indexer_score(const int8_t *qI, const int8_t *kI, const int32_t *wI, const esa_shape *s,
                             int32_t *scores, void *ws, size_t ws_bytes, void *stream) {
    esa_status e = check_shape(s, false, true);
    if (e) return e;
    if (!qI || !kI || !wI || !scores) return ESA_ERR_INVALID;
    if (!aligned16(qI) || !aligned16(kI) || !aligned16(scores)) return ESA_ERR_INVALID;
    if ((e = check_ws(ws, ws_bytes, kStatusBytes))) return e;
    // per-head scores are the scores of the per-head selection rows
    const Shape r = selection_rows(to_shape(s));
    const int32_t *w = per_head_of(r) ? unit_weight() : wI;
    if (!w) return ESA_ERR_CUDA;
    return launch_indexer_score(qI, kI, w, r, scores, (cudaStream_t)stream) == cudaSuccess ? ESA_OK : ESA_ERR_CUDA;
}

esa_status esa_topk_select(const int8_t *qI, const int8_t *kI, const int32_t *wI, const esa_shape *s, int top_k,
                           int32_t *idx, int32_t *cnt, void *ws, size_t ws_bytes, void *stream) {
    esa_status e = check_shape(s, false, true);
    if (e) return e;
    if (!qI || !kI || !wI || !idx || !cnt) return ESA_ERR_INVALID;
    if (top_k <= 0 || top_k > 65536) return ESA_ERR_INVALID;
    if (!aligned16(qI) || !aligned16(kI)) return ESA_ERR_INVALID;
    const Shape x = selection_rows(to_shape(s));  // per-head sets: one row per (query, indexer head)
    if (x.B * x.Tq == 0) return ESA_OK;
    const int32_t *w = per_head_of(x) ? unit_weight() : wI;
    if (!w) return ESA_ERR_CUDA;
    SplitPlan sp = plan_split_select(x, top_k);
    if ((e = check_ws(ws, ws_bytes, sp.ok ? sp.ws_bytes : ws_row_select(x, top_k)))) return e;
    if (sp.ok) return launch_split_select(qI, kI, w, x, top_k, idx, cnt, ws, ws_bytes, sp, (cudaStream_t)stream);
    return launch_row_select(qI, kI, w, x, top_k, idx, cnt, nullptr, ws, ws_bytes, (cudaStream_t)stream);
}

esa_status esa_topk_threshold(const int8_t *qI, const int8_t *kI, const int32_t *wI, const esa_shape *s, int top_k,
                              int32_t *thr, void *ws, size_t ws_bytes, void *stream) {
    esa_status e = check_shape(s, false, true);
    if (e) return e;
    if (!qI || !kI || !wI || !thr) return ESA_ERR_INVALID;
    if (top_k <= 0 || top_k > 65536) return ESA_ERR_INVALID;
    if (!aligned16(qI) || !aligned16(kI)) return ESA_ERR_INVALID;
    const Shape x = selection_rows(to_shape(s));  // per-head sets: one row per (query, indexer head)
    if (x.B * x.Tq == 0) return ESA_OK;
    if ((e = check_ws(ws, ws_bytes, ws_row_select(x, top_k)))) return e;
    const int32_t *w = per_head_of(x) ? unit_weight() : wI;
    if (!w) return ESA_ERR_CUDA;
    // the routed call's own selection step: no index list, the threshold form only
    return launch_row_select(qI, kI, w, x, top_k, nullptr, nullptr, thr, ws, ws_bytes, (cudaStream_t)stream);
}

esa_status esa_sparse_attn(const uint16_t *q, const uint16_t *k, const uint16_t *v, const int32_t *idx,
                           const int32_t *cnt, const esa_shape *s, int top_k, float scale, const float *g,
                           const uint16_t *lin, float *out, float *lse, void *ws, size_t ws_bytes, void *stream) {
    esa_status e = check_shape(s, true, false);
    if (e) return e;
    if (!q || !k || !v || !idx || !cnt || !out) return ESA_ERR_INVALID;
    if ((g == nullptr) != (lin == nullptr)) return ESA_ERR_INVALID;
    if (top_k <= 0 || top_k > 65536) return ESA_ERR_INVALID;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || (lin && !aligned16(lin)))
        return ESA_ERR_INVALID;
    if (!(scale > 0.f) || scale != scale) return ESA_ERR_INVALID;
    Shape x = to_shape(s);
    if (x.B * x.Tq == 0) return ESA_OK;
    AttnPlan p = plan_sparse_attn(x, top_k);
    if ((e = check_ws(ws, ws_bytes, p.ws_bytes))) return e;
    return launch_sparse_attn(q, k, v, idx, cnt, x, top_k, scale, g, lin, out, lse, ws, p, (cudaStream_t)stream);
}

esa_status esa_gated_sparse_attn(const uint16_t *q, const uint16_t *k, const uint16_t *v, const int8_t *qI,
                                 const int8_t *kI, const int32_t *wI, const esa_shape *s, int top_k, float scale,
                                 const float *g, const uint16_t *lin, float *out, float *lse, int32_t *idx,
                                 int32_t *cnt, void *ws, size_t ws_bytes, void *stream) {
    esa_status e = check_shape(s, true, true);
    if (e) return e;
    if (!q || !k || !v || !qI || !kI || !wI || !out) return ESA_ERR_INVALID;
    if ((g == nullptr) != (lin == nullptr) || (idx == nullptr) != (cnt == nullptr)) return ESA_ERR_INVALID;
    if (top_k <= 0 || top_k > 65536) return ESA_ERR_INVALID;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(qI) || !aligned16(kI) || !aligned16(out) ||
        (lin && !aligned16(lin)))
        return ESA_ERR_INVALID;
    if (!(scale > 0.f) || scale != scale) return ESA_ERR_INVALID;
    const Shape x = to_shape(s);
    if (x.B * x.Tq == 0) return ESA_OK;
    cudaStream_t st = (cudaStream_t)stream;
    DecodePlan dp = decode_single_launch() ? plan_decode_step(x, top_k) : DecodePlan{};
    if (dp.ok) {
        if ((e = check_ws(ws, ws_bytes, dp.ws_bytes))) return e;
        return launch_decode_step(q, k, v, qI, kI, wI, x, top_k, scale, g, lin, out, lse, idx, cnt, ws, dp, st);
    }
    if ((e = check_ws(ws, ws_bytes, gated_ws(x, top_k)))) return e;
    // prefill where dense masked tiles on the tensor cores beat gathers: the
    // selection (index sets, threshold forms, bitmask), then the routed
    // kernel with every head sparse (it has no log-sum-exp output)
    if (!lse && gated_routed_path(x, top_k))
        return launch_routed_attn(q, k, v, qI, kI, wI, nullptr, x, top_k, scale, g, lin, out, ws, st, idx, cnt);
    // two launches: the selection into idx/cnt (or workspace room), then the
    // attention over the gathered keys
    const Shape r = selection_rows(x);
    const size_t sel_bytes = align256(topk_ws(x, top_k));
    const size_t scr = gated_scratch_off(x, top_k);
    char *base = static_cast<char *>(ws);
    int32_t *ii = idx ? idx : reinterpret_cast<int32_t *>(base + scr);
    int32_t *cc = cnt ? cnt : reinterpret_cast<int32_t *>(base + scr + align256((size_t)(r.B * r.Tq) * top_k * 4));
    const int32_t *w = per_head_of(r) ? unit_weight() : wI;
    if (!w) return ESA_ERR_CUDA;
    SplitPlan sp = plan_split_select(r, top_k);
    e = sp.ok ? launch_split_select(qI, kI, w, r, top_k, ii, cc, ws, gated_rec_off(x, top_k), sp, st)
              : launch_row_select(qI, kI, w, r, top_k, ii, cc, nullptr, ws, sel_bytes, st);
    if (e != ESA_OK) return e;
    AttnPlan ap = plan_sparse_attn(x, top_k);
    return launch_sparse_attn(q, k, v, ii, cc, x, top_k, scale, g, lin, out, lse, ws, ap, st,
                              base + gated_rec_off(x, top_k), base + gated_xoff(x, top_k));
}

esa_status esa_gated_mix(const float *attn, const uint16_t *lin, const float *g, const uint8_t *head_mask,
                         const esa_shape *s, float *out, void *stream) {
    esa_status e = check_shape(s, true, false);
    if (e) return e;
    if (!attn || !lin || !g || !out) return ESA_ERR_INVALID;
    if (!aligned16(attn) || !aligned16(out) || (reinterpret_cast<uintptr_t>(lin) & 7u)) return ESA_ERR_INVALID;
    return launch_gated_mix(attn, lin, g, head_mask, to_shape(s), out, (cudaStream_t)stream) == cudaSuccess
               ? ESA_OK
               : ESA_ERR_CUDA;
}

esa_status esa_routed_attn(const uint16_t *q, const uint16_t *k, const uint16_t *v, const int8_t *qI,
                           const int8_t *kI, const int32_t *wI, const uint8_t *route, const esa_shape *s, int top_k,
                           float scale, const float *g, const uint16_t *lin, float *out, void *ws, size_t ws_bytes,
                           void *stream) {
    esa_status e = check_shape(s, true, true);
    if (e) return e;
    if (!q || !k || !v || !qI || !kI || !wI || !route || !out) return ESA_ERR_INVALID;
    if ((g == nullptr) != (lin == nullptr)) return ESA_ERR_INVALID;
    if (top_k <= 0 || top_k > 65536) return ESA_ERR_INVALID;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(qI) || !aligned16(kI) || !aligned16(out) ||
        (lin && !aligned16(lin)))
        return ESA_ERR_INVALID;
    if (!(scale > 0.f) || scale != scale) return ESA_ERR_INVALID;
    Shape x = to_shape(s);
    // per-head index sets: on the warp-specialised kernel only
    if (per_head_of(x) && !routed_pp_supported(x)) return ESA_ERR_UNSUPPORTED;
    if (x.B * x.Tq == 0) return ESA_OK;
    if ((e = check_ws(ws, ws_bytes, ws_routed(x, top_k)))) return e;
    return launch_routed_attn(q, k, v, qI, kI, wI, route, x, top_k, scale, g, lin, out, ws, (cudaStream_t)stream);
}

esa_status esa_route_heads(const uint16_t *k, const float *W1, const float *b1, const float *W2, const float *b2,
                           const esa_shape *s, int hidden, uint8_t *route, float *margin, void *ws, size_t ws_bytes,
                           void *stream) {
    esa_status e = check_shape(s, true, false);
    if (e) return e;
    if (!k || !W1 || !b1 || !W2 || !b2 || !route) return ESA_ERR_INVALID;
    if (hidden <= 0 || hidden > 4096) return ESA_ERR_INVALID;
    if (!aligned16(k)) return ESA_ERR_INVALID;
    if (s->B > 65535) return ESA_ERR_UNSUPPORTED;
    const Shape x = to_shape(s);
    if (x.B == 0) return ESA_OK;
    if ((e = check_ws(ws, ws_bytes, ws_route_heads(x)))) return e;
    return launch_route_heads(k, W1, b1, W2, b2, x, hidden, route, margin, ws, (cudaStream_t)stream);
}

static esa_status kda_shape_ok(int64_t B, int64_t T, int32_t H, int32_t Dk, int32_t Dv) {
    if (B < 0 || T < 0 || H < 1) return ESA_ERR_INVALID;
    if (Dk != 64 && Dk != 128) return ESA_ERR_UNSUPPORTED;
    if (Dv < 16 || Dv > 512 || Dv % 16 != 0) return ESA_ERR_UNSUPPORTED;
    if (B > 65535 || H > 65535) return ESA_ERR_UNSUPPORTED;
    return ESA_OK;
}

size_t esa_kda_workspace_size(int64_t B, int64_t T, int32_t H, int32_t Dk, int32_t Dv) {
    if (kda_shape_ok(B, T, H, Dk, Dv) != ESA_OK || !kda_uses_chunks(T)) return 0;
    return kda_chunked_ws_bytes(B, T, H, Dk, Dv);
}

esa_status esa_kda(const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *alpha, const float *beta,
                   const float *state_in, int64_t B, int64_t T, int32_t H, int32_t Dk, int32_t Dv, float scale, float *o,
                   uint16_t *lin, float *state_out, void *ws, size_t ws_bytes, void *stream) {
    esa_status e = kda_shape_ok(B, T, H, Dk, Dv);
    if (e) return e;
    if (T > 0 && (!q || !k || !v || !alpha || !beta)) return ESA_ERR_INVALID;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(alpha) || !aligned16(state_in) ||
        !aligned16(state_out) || !aligned16(o) || (reinterpret_cast<uintptr_t>(lin) & 7u) ||
        (reinterpret_cast<uintptr_t>(beta) & 3u))
        return ESA_ERR_INVALID;
    if (B == 0 || (T == 0 && !state_out)) return ESA_OK;
    if (ws && kda_uses_chunks(T) && (e = check_ws(ws, ws_bytes, kda_chunked_ws_bytes(B, T, H, Dk, Dv)))) return e;
    return launch_kda(q, k, v, alpha, beta, state_in, B, T, H, Dk, Dv, scale, o, lin, state_out, ws,
                      (cudaStream_t)stream);
}

esa_status esa_read_status(void *ws, void *stream, int32_t *dev_status) {
    if (!ws || !dev_status) return ESA_ERR_INVALID;
    cudaStream_t st = (cudaStream_t)stream;
    if (cudaStreamSynchronize(st) != cudaSuccess) return ESA_ERR_CUDA;
    int32_t v = 0;
    if (cudaMemcpy(&v, ws, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return ESA_ERR_CUDA;
    *dev_status = v;
    if (v != 0 && cudaMemset(ws, 0, sizeof v) != cudaSuccess) return ESA_ERR_CUDA;
    return ESA_OK;
}

int esa_binary_version(void) { return mix_binary_version(); }

esa_status esa_cache_append(const uint16_t *k_new, const uint16_t *v_new, const int8_t *kI_new, uint16_t *k,
                            uint16_t *v, int8_t *kI, const esa_shape *s, void *stream) {
    if ((k_new == nullptr) != (k == nullptr) || (v_new == nullptr) != (v == nullptr) ||
        (kI_new == nullptr) != (kI == nullptr))
        return ESA_ERR_INVALID;
    const bool kv = k || v;
    if (!kv && !kI) return ESA_ERR_INVALID;
    esa_status e = check_shape(s, kv, kI != nullptr);
    if (e) return e;
    for (const void *p : {(const void *)k_new, (const void *)v_new, (const void *)kI_new, (const void *)k,
                          (const void *)v, (const void *)kI})
        if (p && !aligned16(p)) return ESA_ERR_INVALID;
    const Shape x = to_shape(s);
    if (x.B * x.Tq == 0) return ESA_OK;
    return launch_cache_append(k_new, v_new, kI_new, k, v, kI, x, (cudaStream_t)stream) == cudaSuccess ? ESA_OK
                                                                                                        : ESA_ERR_CUDA;
}

const char *esa_status_string(esa_status st) {
    switch (st) {
        case ESA_OK: return "ok";
        case ESA_ERR_INVALID: return "invalid argument";
        case ESA_ERR_UNSUPPORTED: return "unsupported shape or size";
        case ESA_ERR_CUDA: return "CUDA runtime error";
        case ESA_ERR_TIMEOUT: return "device wait timed out";
        case ESA_ERR_BAD_INDEX: return "index outside the causal prefix";
        case ESA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case ESA_ERR_INTERNAL: return "kernel consistency check failed";
        default: return "unknown status";
    }
}

}  // extern "C"
