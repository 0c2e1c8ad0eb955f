// Per-head routed attention on the tensor cores, warp-specialised: two
// query tiles per CTA so that one tile's softmax overlaps the other tile's
// matrix products.
//
// Method ("Elastic Attention：动态路由优化大模型长文本处理", sections 2.2 and
// 3.1): every head runs either full causal attention or the sparse path,
// decided per head, inside one launch; sparse heads attend to exactly the
// Top-K positions of the Indexer ("超大规模MoE架构中稀疏注意力机制的演进与实践",
// sections 二.1-二.3) and are mixed with the linear branch by the gate.
//
// The selection (k_select_rows_tc.cu, before this launch) leaves every row's
// selected keys as a bitmask; a sparse head masks its scores with the row's
// word of each key tile, so it costs what a full head costs.
//
// Roles in one CTA (one sequence, one head, query tiles A and B of 128 rows):
//   warps 0-3  softmax of tile A, one thread per query row (TMEM lane)
//   warps 4-7  softmax of tile B
//   warp 8     TMA producer: Q once, then K and V per 64-key tile into a
//              ring of shared-memory slots
//   warp 9     one thread issues every tcgen05.mma:
//                S  = Q K^T            (bf16, fp32 in TMEM)
//                O += P V              (P from TMEM: fp16 against an fp16
//                                       copy of V, or a bf16 hi + lo pair)
//              event-driven: it polls both query tiles' barriers and issues
//              whichever tile's next work is ready; a tile's scores of key
//              tile t+1 go out as soon as its softmax holds S(t) in
//              registers, so they are ready when that softmax finishes.
// All hand-offs are mbarriers (scores ready, scores read, P ready, P V done,
// slot free); no CTA-wide barrier runs inside the key loop. Per query tile
// the tensor memory holds S (64 columns), P (the next 64) and O (D columns).
// The softmax keeps a running max raised only past 2^8 growth, so O is
// rescaled rarely; the gate epilogue is as in k_routed_tc.cu, which serves
// the shapes whose buffers do not fit here.
#include <algorithm>

#include "esa_device.cuh"
#include "esa_internal.h"
#include "tc_util.cuh"

namespace esa {

namespace {

constexpr int kRowsT = 128;  // rows per query tile (TMEM lanes)
constexpr int kBN = 64;      // keys per key tile
constexpr int kProducerWarp = 8, kMmaWarp = 9;
constexpr int kThreads = 320;
constexpr int kMaxSlots = 8;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColsPerTile = 256;  // per query tile: S 64 | SI, P 64 | O D
constexpr float kRescaleLog2 = 8.f;

template <int D>
struct PLay {
    static constexpr int NP = D / 64;                 // 64-element swizzled panels per row
    static constexpr int QT = kRowsT * D * 2;         // one query tile
    static constexpr int Q = 0;                       // 2 query tiles
    static constexpr int RING = Q + 2 * QT;
    static constexpr int SK = 0, SV = kBN * D * 2;
    static constexpr int SLOT = 2 * kBN * D * 2;      // K and V of one key tile
    static constexpr int BUDGET = 227 * 1024 - 1024;  // less the alignment slack
    static constexpr int SLOTS = (BUDGET - RING) / SLOT < kMaxSlots ? (BUDGET - RING) / SLOT : kMaxSlots;
    static constexpr int TOTAL = RING + SLOTS * SLOT + 1024;
    static constexpr bool FITS = SLOTS >= 3;
};

struct PpArgs {
    const int32_t *v_wide;  // set when some |V| is beyond fp16: the fp16-P variant stands down
    const uint16_t *lin;
    const uint8_t *route;
    const int32_t *thr;
    const float *g;
    float *out;
    int32_t *status;
    long long B, Tq, Tk, q_offset, wait_ns;
    int Hq, Hkv, H_I;
    int pset;  // one index set per indexer head: query head h masks with set h / (Hq / H_I)
    // the selection's bitmask of every row's selected keys: uint32 words,
    // word-major ([word][selection row]: a warp's 32 rows read 128 bytes),
    // bit c of word w = key 32 w + c
    const uint32_t *mask;
    long long mask_rows;
    float scale_log2;
};

struct PpBars {
    unsigned long long full[kMaxSlots], slot_free[kMaxSlots];
    unsigned long long s_ready[2], s_free[2], p_ready[2], pv_done[2];
    unsigned long long bar_q, mma_end;
};

// Bounded wait that also gives up when another role has aborted the CTA.
// F16P: P is one fp16 operand and V (tm_v) an fp16 copy of the values: one
// P V product per key tile. Otherwise P is a bf16 hi + lo pair against the
// bf16 values: two products. fp16 holds every bf16 value below 65504
// exactly (smaller ones lose only bits below 2^-24), and rounding p in
// [0, 256] to fp16 changes the output by < 1e-3 where one bf16 P changes it
// by up to 5e-3; the variant used follows the values' range.
template <int D, bool F16P>
__global__ void __launch_bounds__(kThreads, 1)
    routed_pp_kernel(const __grid_constant__ PpArgs a, const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v) {
    using L = PLay<D>;
    constexpr int NP = L::NP, NS = L::SLOTS;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ __align__(8) PpBars bars;
    __shared__ uint32_t tmem_base;
    __shared__ volatile int abort_flag;

    // one of the two variants runs each call (uniform over the grid)
    if ((*a.v_wide != 0) == F16P) return;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const long long nqt = (a.Tq + kRowsT - 1) / kRowsT;
    const long long npair = (nqt + 1) / 2;
    // pairs of query tiles of one (sequence, head) are consecutive, longest
    // prefixes first: the CTAs running together share that head's K/V in L2
    long long bid = blockIdx.x;
    const long long qp = npair - 1 - bid % npair;
    bid /= npair;
    const int h = (int)(bid % a.Hq);
    const long long b = bid / a.Hq;
    const int kvh = h / (a.Hq / a.Hkv);
    const bool sparse = a.route ? a.route[b * a.Hq + h] != 0 : true;  // no routes: every head sparse
    // the index set this head masks with: its own indexer head's (per-head
    // sets) or the row's one set
    const int iset = a.pset ? h / (a.Hq / a.H_I) : 0;
    const int nsets = a.pset ? a.H_I : 1;
    long long t0x[2];
    int rowsx[2], ntx[2];
    for (int x = 0; x < 2; x++) {
        t0x[x] = (2 * qp + x) * kRowsT;
        rowsx[x] = (int)max(0ll, min((long long)kRowsT, a.Tq - t0x[x]));
        ntx[x] = rowsx[x] > 0 ? (int)((a.q_offset + t0x[x] + rowsx[x] + kBN - 1) / kBN) : 0;
    }
    const int nt = max(ntx[0], ntx[1]);
    const uint32_t sbase = smem_u32(smem);
    // param-space addresses of the tensor maps (never copies of them)
    const CUtensorMap *mq = &tm_q, *mk = &tm_k, *mv = &tm_v;
    auto bar = [](unsigned long long &x) { return smem_u32(&x); };

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (tid == kProducerWarp * 32) {
        for (int i = 0; i < NS; i++) {
            mbar_init(bar(bars.full[i]), 1);
            mbar_init(bar(bars.slot_free[i]), 1);
        }
        for (int i = 0; i < 2; i++) {
            mbar_init(bar(bars.s_ready[i]), 1);
            mbar_init(bar(bars.s_free[i]), kRowsT);
            mbar_init(bar(bars.p_ready[i]), kRowsT);
            mbar_init(bar(bars.pv_done[i]), 1);
        }
        mbar_init(bar(bars.bar_q), 1);
        mbar_init(bar(bars.mma_end), 1);
        mbar_fence_init();
        abort_flag = 0;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;

    if (warp < 8) {
        // ================================================= softmax warps
        const int x = warp >> 2, q4 = warp & 3;
        const int r = 32 * q4 + lane;  // row within tile x, and its TMEM lane
        const int rows = rowsx[x], ntt = ntx[x];
        const long long row0 = b * a.Tq + t0x[x];
        const long long pos = r < rows ? a.q_offset + t0x[x] + r : -1;
        const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
        const uint32_t colS = x * kColsPerTile, colP = colS + 64, colO = colS + 128;
        // a sparse row keeps the keys its mask words select (a row whose
        // whole prefix is kept, T = INT32_MIN, keeps every key); the next
        // key tile's two words are loaded one tile ahead
        const bool use_mask = sparse && r < rows && a.thr[2 * ((row0 + r) * nsets + iset)] != INT32_MIN;
        const uint32_t *mrow = a.mask + (row0 + (r < rows ? r : 0)) * nsets + iset;
        auto mask_word = [&](int t) -> uint64_t {
            if (!use_mask) return ~0ull;
            const uint32_t lo = __ldg(mrow + (size_t)(2 * t) * a.mask_rows);
            const uint32_t hi = __ldg(mrow + (size_t)(2 * t + 1) * a.mask_rows);
            return (uint64_t)lo | ((uint64_t)hi << 32);
        };
        uint64_t mnext = ntt > 0 ? mask_word(0) : ~0ull;

        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        for (int t = 0; t < ntt && ok; t++) {
            if (!wait_or_abort(bar(bars.s_ready[x]), (uint32_t)t & 1u, a.wait_ns, &abort_flag, a.status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sr[64];
            tmem_ld32(tmem + lane_base + colS, sr);
            tmem_ld32(tmem + lane_base + colS + 32, sr + 32);
            const long long j0 = (long long)t * kBN;
            const uint64_t keep = mnext;  // bit c: key j0+c is selected
            mnext = t + 1 < ntt ? mask_word(t + 1) : ~0ull;
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(bar(bars.s_free[x]));  // S is in registers
            // causal: key j0+c is visible to this row iff c <= pos - j0; the
            // maximum is taken over the raw scores (scale > 0 keeps the order)
            const int lim = (int)max(-1ll, min(64ll, pos - j0));
            float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
            if (use_mask) {
                const uint64_t vis = lim >= 63 ? keep : keep & ((2ull << (lim < 0 ? 0 : lim)) - 1ull) & (lim < 0 ? 0ull : ~0ull);
                const uint32_t v0 = (uint32_t)vis, v1 = (uint32_t)(vis >> 32);
#pragma unroll
                for (int c = 0; c < 64; c++) {
                    const bool valid = ((c < 32 ? v0 : v1) >> (c & 31)) & 1u;
                    const float xv = valid ? __uint_as_float(sr[c]) : -INFINITY;
                    sr[c] = __float_as_uint(xv);
                    mx4[c & 3] = fmaxf(mx4[c & 3], xv);
                }
            } else if (lim >= 63) {  // no key past the row
#pragma unroll
                for (int c = 0; c < 64; c++) mx4[c & 3] = fmaxf(mx4[c & 3], __uint_as_float(sr[c]));
            } else {
#pragma unroll
                for (int c = 0; c < 64; c++) {
                    const float xv = c <= lim ? __uint_as_float(sr[c]) : -INFINITY;
                    sr[c] = __float_as_uint(xv);
                    mx4[c & 3] = fmaxf(mx4[c & 3], xv);
                }
            }
            const float mt = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * a.scale_log2;
            float corr = 1.f;
            bool rescale = false;
            if (mt > m_used + kRescaleLog2 || (m_used == -INFINITY && mt > -INFINITY)) {
                rescale = m_used != -INFINITY;  // O is still zero before the first kept key
                corr = rescale ? ex2_approx(m_used - mt) : 1.f;
                l *= corr;
                m_used = mt;
            }
            const float mu = m_used == -INFINITY ? 0.f : m_used;
            // the previous tile's P V is done: P's columns are free, O is stable
            if (t > 0 && !wait_or_abort(bar(bars.pv_done[x]), (uint32_t)(t - 1) & 1u, a.wait_ns, &abort_flag, a.status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t o_raw[32];
                    tmem_ld32(tmem + lane_base + colO + c0, o_raw);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; e++) o_raw[e] = __float_as_uint(__uint_as_float(o_raw[e]) * corr);
                    tmem_st32(tmem + lane_base + colO + c0, o_raw);
                }
            }
            // p = 2^(s*scale - mu) (0 for masked keys), fp16 or bf16 hi + lo,
            // written in two 32-key halves
            float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
            for (int half = 0; half < 2; half++) {
                uint32_t phi[16], plo[16];
#pragma unroll
                for (int c = 0; c < 32; c += 2) {
                    const int cc = half * 32 + c;
                    const float p0 = ex2_approx(fmaf(__uint_as_float(sr[cc]), a.scale_log2, -mu)),
                                p1 = ex2_approx(fmaf(__uint_as_float(sr[cc + 1]), a.scale_log2, -mu));
                    ls0 += p0;
                    ls1 += p1;
                    if constexpr (F16P) {
                        phi[c / 2] = pack_f16(p0, p1);
                    } else {
                        const uint32_t hw = pack_bf16(p0, p1);
                        phi[c / 2] = hw;
                        plo[c / 2] = pack_bf16(p0 - bf16lo(hw), p1 - bf16hi(hw));
                    }
                }
                tmem_st16(tmem + lane_base + colP + half * 16, phi);
                if constexpr (!F16P) tmem_st16(tmem + lane_base + colP + 32 + half * 16, plo);
            }
            l += ls0 + ls1;
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar(bars.p_ready[x]));
        }
        // ---- epilogue: O / l, gate mix for sparse heads
        if (ok && ntt > 0 &&
            wait_or_abort(bar(bars.pv_done[x]), (uint32_t)(ntt - 1) & 1u, a.wait_ns, &abort_flag, a.status)) {
            tc_fence_after();
            const bool gated = sparse && a.g != nullptr && a.lin != nullptr;
            const float gh = gated ? a.g[h] : 1.f, gl = 1.f - gh;
            const long long obase = ((row0 + r) * a.Hq + h) * (long long)D;
            const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t o_raw[32];
                tmem_ld32(tmem + lane_base + colO + c0, o_raw);
                tmem_wait_ld();
                if (r < rows) {
#pragma unroll
                    for (int e = 0; e < 32; e += 4) {
                        float4 v4 = make_float4(__uint_as_float(o_raw[e]) * inv, __uint_as_float(o_raw[e + 1]) * inv,
                                                __uint_as_float(o_raw[e + 2]) * inv, __uint_as_float(o_raw[e + 3]) * inv);
                        if (gated) {
                            const uint2 lw = *reinterpret_cast<const uint2 *>(a.lin + obase + c0 + e);
                            v4.x = fmaf(gh, v4.x, gl * bf16lo(lw.x));
                            v4.y = fmaf(gh, v4.y, gl * bf16hi(lw.x));
                            v4.z = fmaf(gh, v4.z, gl * bf16lo(lw.y));
                            v4.w = fmaf(gh, v4.w, gl * bf16hi(lw.y));
                        }
                        *reinterpret_cast<float4 *>(a.out + obase + c0 + e) = v4;
                    }
                }
            }
        }
    } else if (warp == kProducerWarp) {
        // ================================================= TMA producer
        int issued = -1;
        auto issue = [&](int t) {  // lane 0 issues; the whole warp waits for the slot
            const int slot = t % NS;
            if (t >= NS &&
                !wait_or_abort(bar(bars.slot_free[slot]), (uint32_t)(t / NS - 1) & 1u, a.wait_ns, &abort_flag, a.status))
                return false;
            if (lane == 0) {
                const uint32_t sl = sbase + L::RING + slot * L::SLOT;
                const uint32_t fb = bar(bars.full[slot]);
                const int krow = (int)(b * a.Tk + (long long)t * kBN);
                mbar_expect_tx(fb, (unsigned)(2 * kBN * D * 2));
#pragma unroll
                for (int p = 0; p < NP; p++) {
                    tma3(sl + L::SK + p * (kBN * 128), mk, p * 64, kvh, krow, fb);
                    tma3(sl + L::SV + p * (kBN * 128), mv, p * 64, kvh, krow, fb);
                }
            }
            issued = t;
            return true;
        };
        bool ok = true;
        if (lane == 0) {
            unsigned bytes = 0;
            for (int x = 0; x < 2; x++) bytes += rowsx[x] > 0 ? (unsigned)L::QT : 0u;
            mbar_expect_tx(bar(bars.bar_q), bytes);
            for (int x = 0; x < 2; x++)
                if (rowsx[x] > 0)
#pragma unroll
                    for (int p = 0; p < NP; p++)
                        tma3(sbase + L::Q + x * L::QT + p * (kRowsT * 128), mq, p * 64, h, (int)(b * a.Tq + t0x[x]),
                             bar(bars.bar_q));
        }
        for (int t = 0; t < nt && ok; t++) ok = issue(t);
        // copies still in flight after an abort: wait for them (bounded)
        if (!ok && lane == 0)
            for (int t = 0; t <= issued; t++) mbar_wait_bounded(bar(bars.full[t % NS]), (uint32_t)(t / NS) & 1u, a.wait_ns);
    } else if (warp == kMmaWarp) {
        // ================================================= MMA issuer
        if (lane == 0) {
            bool ok = wait_or_abort(bar(bars.bar_q), 0u, a.wait_ns, &abort_flag, a.status);
            constexpr uint32_t id_s = idesc(kBN, 1u, 0u), id_o = idesc(D, F16P ? 0u : 1u, 1u);
            constexpr int nparts = F16P ? 1 : 2;
            // S of key tile u for query tile x (its K in ring slot u % NS)
            auto issue_s = [&](int x, int u) {
                const uint32_t su = sbase + L::RING + (u % NS) * L::SLOT;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < D / 16; kk++)
                    mma_ss(tmem + x * kColsPerTile,
                           sdesc(sbase + L::Q + x * L::QT + (kk / 4) * (kRowsT * 128) + (kk % 4) * 32, 16, 1024, 2),
                           sdesc(su + L::SK + (kk / 4) * (kBN * 128) + (kk % 4) * 32, 16, 1024, 2), id_s, kk > 0);
            };
            auto done = [&](unsigned long long &x, uint32_t parity) { return mbar_try_wait(bar(x), parity); };
            // Event-driven issue: per query tile x, ns[x] is the next key tile
            // whose scores go out, np[x] the next whose P V does. S(u) needs
            // K(u) and the softmax to hold S(u-1) in registers (S's columns
            // are free), so it is computed while that softmax works on tile
            // u-1; P V(u) needs the softmax's P(u). Whichever query tile is
            // ready goes first. Ring slot t is released once both tiles' P V(t)
            // are issued.
            int ns[2] = {0, 0}, np[2] = {0, 0}, fr = 0;
            unsigned long long t_idle = 0;
            bool idle = false;
            while (ok && (np[0] < ntx[0] || np[1] < ntx[1])) {
                bool progress = false;
                for (int x = 0; x < 2; x++) {
                    const int u = ns[x];
                    if (u < ntx[x] && done(bars.full[u % NS], (uint32_t)(u / NS) & 1u) &&
                        (u == 0 || done(bars.s_free[x], (uint32_t)(u - 1) & 1u))) {
                        issue_s(x, u);
                        mma_commit(bar(bars.s_ready[x]));
                        ns[x] = u + 1;
                        progress = true;
                    }
                    const int v = np[x];
                    if (v < ns[x] && done(bars.p_ready[x], (uint32_t)v & 1u)) {
                        tc_fence_after();
                        const uint32_t colS = x * kColsPerTile;
                        const uint32_t sl = sbase + L::RING + (v % NS) * L::SLOT;
#pragma unroll
                        for (int part = 0; part < nparts; part++)
#pragma unroll
                            for (int kk = 0; kk < kBN / 16; kk++)
                                mma_ts(tmem + colS + 128, tmem + colS + 64 + part * 32 + kk * 8,
                                       sdesc(sl + L::SV + kk * 2048, kBN * 128, 1024, 2), id_o,
                                       (v > 0 || part > 0 || kk > 0));
                        mma_commit(bar(bars.pv_done[x]));
                        np[x] = v + 1;
                        progress = true;
                        while (fr < nt && (np[0] > fr || fr >= ntx[0]) && (np[1] > fr || fr >= ntx[1])) {
                            mma_commit(bar(bars.slot_free[fr % NS]));
                            fr++;
                        }
                    }
                }
                // a bounded wait for the next event: on time-out the call
                // aborts with the status set (every waiter then gives up)
                if (progress) {
                    idle = false;
                } else {
                    unsigned long long now;
                    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(now));
                    if (!idle) {
                        idle = true;
                        t_idle = now;
                    } else if ((long long)(now - t_idle) > a.wait_ns || abort_flag) {
                        set_status(a.status, ESA_ERR_TIMEOUT);
                        abort_flag = 1;
                        ok = false;
                    }
                }
            }
            // every MMA issued has completed before the CTA frees tensor memory
            mma_commit(bar(bars.mma_end));
            mbar_wait_bounded(bar(bars.mma_end), 0u, a.wait_ns);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
    }
}

template <int D, bool F16P>
void *pp_kernel(size_t *smem) {
    if constexpr (!PLay<D>::FITS) {
        return nullptr;
    } else {
        *smem = PLay<D>::TOTAL;
        return (void *)routed_pp_kernel<D, F16P>;
    }
}

template <bool F16P>
void *pp_kernel_for(const Shape &s, size_t *smem) {
    return s.D == 64 ? pp_kernel<64, F16P>(smem) : pp_kernel<128, F16P>(smem);
}

// values (bf16) -> fp16 copy; *wide = 1 when some |v| > 65504 (fp16 cannot hold it)
__global__ void __launch_bounds__(256) v_to_f16_kernel(const uint4 *__restrict__ v, uint4 *__restrict__ vh,
                                                       long long n8, int32_t *__restrict__ wide) {
    bool big = false;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n8; i += (long long)gridDim.x * blockDim.x) {
        const uint4 w = ldg_stream16(v + i);
        uint32_t in[4] = {w.x, w.y, w.z, w.w}, o[4];
#pragma unroll
        for (int e = 0; e < 4; e++) {
            const float lo = bf16lo(in[e]), hi = bf16hi(in[e]);
            big = big || fabsf(lo) > 65504.f || fabsf(hi) > 65504.f;
            o[e] = pack_f16(lo, hi);
        }
        vh[i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
    if (__syncthreads_or(big) && threadIdx.x == 0) atomicOr(wide, 1);
}

}  // namespace

size_t ws_routed_pp(const Shape &s) {
    return align256((size_t)s.B * s.Tk * s.Hkv * s.D * 2) + kStatusBytes;  // fp16 values, range flag
}

bool routed_pp_supported(const Shape &s) {
    size_t smem = 0;
    void *fn = pp_kernel_for<true>(s, &smem);
    return fn != nullptr && s.B * s.Tq < (1ll << 31) && s.B * s.Tk < (1ll << 31);
}

esa_status launch_routed_pp(const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint8_t *route,
                            const int32_t *thr, const uint32_t *mask, const Shape &s, float scale, const float *g,
                            const uint16_t *lin, float *out, void *pp_ws, int32_t *status, cudaStream_t st) {
    if (!mask) return ESA_ERR_INTERNAL;
    const Shape r = selection_rows(s);
    PpArgs a{};
    a.mask = mask;
    a.mask_rows = r.B * r.Tq;
    a.lin = lin;
    a.route = route;
    a.thr = thr;
    a.g = g;
    a.out = out;
    a.status = status;
    a.B = s.B;
    a.Tq = s.Tq;
    a.Tk = s.Tk;
    a.q_offset = s.q_offset;
    a.wait_ns = wait_limit_ns();
    a.Hq = s.Hq;
    a.Hkv = s.Hkv;
    a.H_I = s.H_I;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.pset = per_head_of(s) ? 1 : 0;
    const long long nqt = (s.Tq + kRowsT - 1) / kRowsT;
    const long long blocks = s.B * s.Hq * ((nqt + 1) / 2);
    if (blocks == 0) return ESA_OK;
    size_t smem16 = 0, smem2 = 0;
    void *fn16 = pp_kernel_for<true>(s, &smem16), *fn2 = pp_kernel_for<false>(s, &smem2);
    if (!fn16 || !fn2) return ESA_ERR_UNSUPPORTED;
    // fp16 copy of the values and the flag that picks the variant
    int32_t *wide = static_cast<int32_t *>(pp_ws);
    uint16_t *vh = reinterpret_cast<uint16_t *>(static_cast<char *>(pp_ws) + kStatusBytes);
    a.v_wide = wide;
    if (cudaMemsetAsync(wide, 0, sizeof(int32_t), st) != cudaSuccess) return ESA_ERR_CUDA;
    {
        const long long n8 = s.B * s.Tk * s.Hkv * s.D / 8;
        const long long want = (n8 + 255) / 256, cap = (long long)device_info().sms * 8;
        if (n8 > 0)
            v_to_f16_kernel<<<(unsigned)(want < cap ? want : cap), 256, 0, st>>>(
                reinterpret_cast<const uint4 *>(v), reinterpret_cast<uint4 *>(vh), n8, wide);
        if (cudaGetLastError() != cudaSuccess) return ESA_ERR_CUDA;
    }
    CUtensorMap tq, tk, tv, tvh;
    if (!map_rows_heads_d(&tq, q, s.B * s.Tq, s.Hq, s.D, kRowsT) || !map_rows_heads_d(&tk, k, s.B * s.Tk, s.Hkv, s.D, kBN) ||
        !map_rows_heads_d(&tv, v, s.B * s.Tk, s.Hkv, s.D, kBN) || !map_rows_heads_d(&tvh, vh, s.B * s.Tk, s.Hkv, s.D, kBN))
        return ESA_ERR_CUDA;
    if (!ensure_smem(fn16, smem16) || !ensure_smem(fn2, smem2)) return ESA_ERR_CUDA;
    // the fp16-P variant; then the bf16 hi + lo variant, whose blocks return at
    // once unless some value is beyond fp16 (tensor maps copy bits: the fp16
    // copy uses the same 2-byte map shape)
    void *args16[] = {(void *)&a, (void *)&tq, (void *)&tk, (void *)&tvh};
    if (cudaLaunchKernel(fn16, dim3((unsigned)blocks), dim3(kThreads), args16, smem16, st) != cudaSuccess)
        return ESA_ERR_CUDA;
    void *args2[] = {(void *)&a, (void *)&tq, (void *)&tk, (void *)&tv};
    cudaError_t ce = cudaLaunchKernel(fn2, dim3((unsigned)blocks), dim3(kThreads), args2, smem2, st);
    return ce == cudaSuccess ? ESA_OK : ESA_ERR_CUDA;
}

}  // namespace esa
