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
// Roles in one CTA (one sequence, one head, query tiles A and B of 128 rows):
//   warps 0-3  softmax of tile A, one thread per query row (TMEM lane)
//   warps 4-7  softmax of tile B
//   warp 8     TMA producer: Q once, then K, V (and raw int8 indexer keys)
//              per 64-key tile into a ring of shared-memory slots; converts
//              the indexer keys to fp16 for the tensor cores
//   warp 9     one thread issues every tcgen05.mma:
//                S  = Q K^T            (bf16, fp32 in TMEM)
//                SI = q_eff kI^T       (fp16 holding exact small integers; the
//                                       Top-K mask of sparse heads)
//                O += P_hi V + P_lo V  (P from TMEM)
// All hand-offs are mbarriers (scores ready, scores read, P ready, P V done,
// slot free, indexer keys converted / consumed); no CTA-wide barrier runs
// inside the key loop. Per query tile the tensor memory holds S (64
// columns), SI and then P over the same 64 columns, and O (D columns).
// The mask, the softmax (running max raised only past 2^8 growth, so O is
// rescaled rarely), the bf16 hi + lo split of P and the gate epilogue are as
// in k_routed_tc.cu, which serves the shapes whose buffers do not fit here.
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
constexpr int kSlots = 3;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColsPerTile = 256;  // per query tile: S 64 | SI, P 64 | O D
constexpr float kRescaleLog2 = 8.f;

template <int D, int DI>
struct PLay {
    static constexpr int NP = D / 64;                 // 64-element swizzled panels per row
    static constexpr int QT = kRowsT * D * 2;         // one query tile
    static constexpr int Q = 0;                       // 2 query tiles
    static constexpr int QET = kRowsT * DI * 2;       // one collapsed indexer query tile (fp16)
    static constexpr int QE = Q + 2 * QT;
    static constexpr int KHB = kBN * DI * 2;          // fp16 indexer keys of one key tile
    static constexpr int KH = QE + 2 * QET;           // 2 buffers
    static constexpr int RING = KH + 2 * KHB;
    static constexpr int SK = 0, SV = kBN * D * 2, SKI = 2 * kBN * D * 2;
    static constexpr int SLOT = (SKI + kBN * DI + 1023) / 1024 * 1024;
    static constexpr int TOTAL = RING + kSlots * SLOT + 1024;  // + alignment slack
    static constexpr bool FITS = TOTAL <= 227 * 1024;
};

struct PpArgs {
    const int32_t *v_wide;  // set when some |V| is beyond fp16: the fp16-P variant stands down
    const uint16_t *lin;
    const int8_t *qI;
    const int32_t *wI;
    const uint8_t *route;
    const int32_t *thr;
    const float *g;
    float *out;
    int32_t *status;
    long long B, Tq, Tk, q_offset, wait_ns;
    int Hq, Hkv, H_I;
    int relu;  // ReLU on each indexer head's dot product
    int pset;  // one index set per indexer head: query head h masks with set h / (Hq / H_I), weight 1
    // the selection's bitmask of every row's selected keys ([rows][mask_w64]
    // 64-bit words, bit c of word t = key 64 t + c), or null: then sparse
    // heads rebuild the mask from indexer scores on the tensor cores
    const uint64_t *mask;
    long long mask_w64;
    float scale_log2;
};

struct PpBars {
    unsigned long long full[kSlots], slot_free[kSlots], kh_ready[2], kh_free[2];
    unsigned long long s_ready[2], s_free[2], p_ready[2], pv_done[2];
    unsigned long long bar_q, qe_ready, mma_end;
};

// Bounded wait that also gives up when another role has aborted the CTA.
// F16P: P is one fp16 operand and V (tm_v) an fp16 copy of the values: one
// P V product per key tile. Otherwise P is a bf16 hi + lo pair against the
// bf16 values: two products. fp16 holds every bf16 value below 65504
// exactly (smaller ones lose only bits below 2^-24), and rounding p in
// [0, 256] to fp16 changes the output by < 1e-3 where one bf16 P changes it
// by up to 5e-3; the variant used follows the values' range.
template <int D, int DI, bool F16P>
__global__ void __launch_bounds__(kThreads, 1)
    routed_pp_kernel(const __grid_constant__ PpArgs a, const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                     const __grid_constant__ CUtensorMap tm_ki) {
    using L = PLay<D, DI>;
    constexpr int NP = L::NP;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ __align__(8) PpBars bars;
    __shared__ uint32_t tmem_base;
    __shared__ int exact_all;
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
    const bool sparse = a.route[b * a.Hq + h] != 0;
    // the index set this head masks with: its own indexer head's (per-head
    // sets, weight 1) or the row's one weighted set
    const int iset = a.pset ? h / (a.Hq / a.H_I) : 0;
    const int nsets = a.pset ? a.H_I : 1, nih = a.pset ? 1 : a.H_I;
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
    const CUtensorMap *mq = &tm_q, *mk = &tm_k, *mv = &tm_v, *mki = &tm_ki;
    auto bar = [](unsigned long long &x) { return smem_u32(&x); };

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (tid == kProducerWarp * 32) {
        for (int i = 0; i < kSlots; i++) {
            mbar_init(bar(bars.full[i]), 1);
            mbar_init(bar(bars.slot_free[i]), 1);
        }
        for (int i = 0; i < 2; i++) {
            mbar_init(bar(bars.kh_ready[i]), 1);
            mbar_init(bar(bars.kh_free[i]), 1);
            mbar_init(bar(bars.s_ready[i]), 1);
            mbar_init(bar(bars.s_free[i]), kRowsT);
            mbar_init(bar(bars.p_ready[i]), kRowsT);
            mbar_init(bar(bars.pv_done[i]), 1);
        }
        mbar_init(bar(bars.bar_q), 1);
        mbar_init(bar(bars.qe_ready), 2 * kRowsT);
        mbar_init(bar(bars.mma_end), 1);
        mbar_fence_init();
        // a ReLU stays exact on the tensor cores for one indexer head of
        // non-negative weight (max(0, w d) = w max(0, d)); several heads do
        // not collapse, so their mask scores come from dp4a
        exact_all = (a.relu && !(nih == 1 && (a.pset || a.wI[0] >= 0))) ? 0 : 1;
        if (a.mask) exact_all = 0;  // the mask replaces the indexer scores
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
        const uint32_t colS = x * kColsPerTile, colSI = colS + 64, colO = colS + 128;
        float Tf = 0.f;
        int Tint = 0, Pp = -1;
        if (sparse) {
            if (r < rows) {
                Tint = a.thr[2 * ((row0 + r) * nsets + iset)];
                Pp = a.thr[2 * ((row0 + r) * nsets + iset) + 1];
            }
            Tf = (float)Tint;
        }
        if (sparse && !a.mask) {
            // collapsed indexer query q_eff = sum_h w_h qI_h (fp16, exact while
            // |q_eff| <= 2048 and every partial sum of q_eff . kI stays below 2^24)
            long long absum = 0;
            bool fits = true;
            const int8_t *qrow = a.qI + ((row0 + (r < rows ? r : 0)) * (long long)a.H_I + iset) * DI;
            for (int c0 = 0; c0 < DI; c0 += 8) {
                long long acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};  // 64-bit: any int32 weight
                for (int hh = 0; hh < nih; hh++) {
                    const long long wv = a.pset ? 1 : a.wI[hh];
                    const uint2 raw = *reinterpret_cast<const uint2 *>(qrow + hh * DI + c0);
#pragma unroll
                    for (int e = 0; e < 8; e++) {
                        const int8_t qv = (int8_t)(((e < 4 ? raw.x : raw.y) >> (8 * (e & 3))) & 0xFF);
                        acc[e] += wv * qv;
                    }
                }
                uint32_t pk[4];
#pragma unroll
                for (int e = 0; e < 8; e++) {
                    fits = fits && acc[e] >= -2048 && acc[e] <= 2048;
                    absum += acc[e] < 0 ? -(long long)acc[e] : acc[e];
                }
#pragma unroll
                for (int e = 0; e < 4; e++) pk[e] = pack_f16((float)acc[2 * e], (float)acc[2 * e + 1]);
                if (r >= rows) pk[0] = pk[1] = pk[2] = pk[3] = 0u;
                *reinterpret_cast<uint4 *>(smem + L::QE + x * L::QET + (r / 8) * (DI / 8 * 128) + (c0 / 8) * 128 +
                                           (r % 8) * 16) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
            fits = fits && absum * 128 < (1ll << 24);
            if (!fits && r < rows) atomicAnd(&exact_all, 0);
            fence_async_smem();
        }
        asm volatile("bar.sync 1, 256;" ::: "memory");  // every softmax thread has voted
        const bool exact = exact_all != 0;
        mbar_arrive(bar(bars.qe_ready));

        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        // with the selection's bitmask: this row's word of the next key tile,
        // loaded one tile ahead (whole-prefix rows, T = INT32_MIN, keep every key)
        const bool use_mask = sparse && a.mask != nullptr && r < rows && Tint != INT32_MIN;
        const uint64_t *mrow = use_mask ? a.mask + ((row0 + r) * nsets + iset) * a.mask_w64 : nullptr;
        uint64_t mnext = use_mask && ntt > 0 ? __ldg(mrow) : ~0ull;
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
            uint64_t keep = ~0ull;  // bit c: key j0+c passes the Top-K test
            if (sparse && exact) {
#pragma unroll
                for (int half = 0; half < 2; half++) {
                    uint32_t ir[32];
                    tmem_ld32(tmem + lane_base + colSI + half * 32, ir);
                    tmem_wait_ld();
                    if (a.relu) {  // one head of non-negative weight: exact
#pragma unroll
                        for (int c = 0; c < 32; c++) ir[c] = __float_as_uint(fmaxf(__uint_as_float(ir[c]), 0.f));
                    }
                    const int pl = (int)max(-1ll, min(64ll, (long long)Pp - j0));  // ties kept for c <= pl
                    if (pl < 0 || pl >= 63) {
                        // the tie position is outside this tile: kept iff s >= cut,
                        // with cut = T (ties kept) or T + 1 (exact: integer scores)
                        const float cut = pl < 0 ? Tf + 1.f : Tf;
#pragma unroll
                        for (int c = 0; c < 32; c++)
                            if (!(__uint_as_float(ir[c]) >= cut)) sr[half * 32 + c] = 0xff800000u;  // -inf
                    } else {
#pragma unroll
                        for (int c = 0; c < 32; c++) {
                            const float si = __uint_as_float(ir[c]);
                            if (!(si > Tf || (si == Tf && half * 32 + c <= pl))) sr[half * 32 + c] = 0xff800000u;
                        }
                    }
                }
            } else if (sparse && a.mask) {
                keep = mnext;
                mnext = use_mask && t + 1 < ntt ? __ldg(mrow + t + 1) : ~0ull;
            } else if (sparse) {
                // exact integer mask scores with dp4a from the raw keys of the slot
                const int slot = t % kSlots;
                if (!wait_or_abort(bar(bars.full[slot]), (uint32_t)(t / kSlots) & 1u, a.wait_ns, &abort_flag, a.status)) {
                    ok = false;
                    break;
                }
                const unsigned char *raw = smem + L::RING + slot * L::SLOT + L::SKI;
                const int8_t *qrow = a.qI + ((row0 + (r < rows ? r : 0)) * (long long)a.H_I + iset) * DI;
                for (int c = 0; c < 64; c++) {
                    unsigned acc = 0;
                    for (int hh = 0; hh < nih; hh++) {
                        int d = 0;
#pragma unroll
                        for (int w4 = 0; w4 < DI / 4; w4++)
                            d = __dp4a(reinterpret_cast<const int *>(qrow + hh * DI)[w4],
                                       reinterpret_cast<const int *>(raw + c * DI)[w4], d);
                        acc += (unsigned)(a.pset ? 1 : a.wI[hh]) * (unsigned)(a.relu ? max(d, 0) : d);
                    }
                    const int si = (int)acc;
                    if (!(si > Tint || (si == Tint && j0 + c <= Pp))) keep &= ~(1ull << c);
                }
            }
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(bar(bars.s_free[x]));  // S (and SI) are in registers
            // causal: key j0+c is visible to this row iff c <= pos - j0; the
            // maximum is taken over the raw scores (scale > 0 keeps the order)
            const int lim = (int)max(-1ll, min(64ll, pos - j0));
            float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
            if (sparse && !exact) {
#pragma unroll
                for (int c = 0; c < 64; c++) {
                    const bool valid = c <= lim && ((keep >> c) & 1ull);
                    const float xv = valid ? __uint_as_float(sr[c]) : -INFINITY;
                    sr[c] = __float_as_uint(xv);
                    mx4[c & 3] = fmaxf(mx4[c & 3], xv);
                }
            } else if (lim >= 63) {  // the Top-K mask (if any) is already in sr; no key past the row
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
            // written over the indexer-score columns in two 32-key halves
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
                tmem_st16(tmem + lane_base + colSI + half * 16, phi);
                if constexpr (!F16P) tmem_st16(tmem + lane_base + colSI + 32 + half * 16, plo);
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
            const int slot = t % kSlots;
            if (t >= kSlots &&
                !wait_or_abort(bar(bars.slot_free[slot]), (uint32_t)(t / kSlots - 1) & 1u, a.wait_ns, &abort_flag, a.status))
                return false;
            if (lane == 0) {
                const uint32_t sl = sbase + L::RING + slot * L::SLOT;
                const uint32_t fb = bar(bars.full[slot]);
                const int krow = (int)(b * a.Tk + (long long)t * kBN);
                const bool raw_ki = sparse && !a.mask;  // the indexer keys, unless the mask replaces them
                mbar_expect_tx(fb, (unsigned)(2 * kBN * D * 2 + (raw_ki ? kBN * DI : 0)));
#pragma unroll
                for (int p = 0; p < NP; p++) {
                    tma3(sl + L::SK + p * (kBN * 128), mk, p * 64, kvh, krow, fb);
                    tma3(sl + L::SV + p * (kBN * 128), mv, p * 64, kvh, krow, fb);
                }
                if (raw_ki) tma2(sl + L::SKI, mki, 0, krow, fb);
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
        for (int t = 0; t < kSlots - 1 && t < nt && ok; t++) ok = issue(t);
        bool exact = true;
        if (sparse) {
            ok = ok && wait_or_abort(bar(bars.qe_ready), 0u, a.wait_ns, &abort_flag, a.status);
            exact = exact_all != 0;
        }
        for (int t = 0; t < nt && ok; t++) {
            if (sparse && exact) {
                // tile t's raw indexer keys -> fp16 KH buffer t % 2 (its previous
                // user, tile t-2, has had its indexer products read)
                const int slot = t % kSlots;
                if (!wait_or_abort(bar(bars.full[slot]), (uint32_t)(t / kSlots) & 1u, a.wait_ns, &abort_flag, a.status) ||
                    (t >= 2 &&
                     !wait_or_abort(bar(bars.kh_free[t % 2]), (uint32_t)((t - 2) / 2) & 1u, a.wait_ns, &abort_flag, a.status))) {
                    ok = false;
                    break;
                }
                const unsigned char *raw = smem + L::RING + slot * L::SLOT + L::SKI;
                unsigned char *dst = smem + L::KH + (t % 2) * L::KHB;
                for (int i = lane; i < kBN * DI / 8; i += 32) {
                    const int c8 = (i / 8) % (DI / 8), kk = (i % 8) + 8 * ((i / 8) / (DI / 8));
                    const uint2 rv = *reinterpret_cast<const uint2 *>(raw + kk * DI + c8 * 8);
                    uint32_t pk[4];
#pragma unroll
                    for (int e = 0; e < 4; e++) {
                        const uint32_t w = e < 2 ? rv.x : rv.y;
                        const int sh = (e & 1) * 16;
                        pk[e] = pack_f16((float)(int8_t)((w >> sh) & 0xFF), (float)(int8_t)((w >> (sh + 8)) & 0xFF));
                    }
                    *reinterpret_cast<uint4 *>(dst + (kk / 8) * (DI / 8 * 128) + c8 * 128 + (kk % 8) * 16) =
                        make_uint4(pk[0], pk[1], pk[2], pk[3]);
                }
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(bars.kh_ready[t % 2]));
            }
            if (t + kSlots - 1 < nt) ok = issue(t + kSlots - 1);
        }
        // copies still in flight after an abort: wait for them (bounded)
        if (!ok && lane == 0)
            for (int t = 0; t <= issued; t++) mbar_wait_bounded(bar(bars.full[t % kSlots]), (uint32_t)(t / kSlots) & 1u, a.wait_ns);
    } else if (warp == kMmaWarp) {
        // ================================================= MMA issuer
        if (lane == 0) {
            bool ok = wait_or_abort(bar(bars.bar_q), 0u, a.wait_ns, &abort_flag, a.status) &&
                      wait_or_abort(bar(bars.qe_ready), 0u, a.wait_ns, &abort_flag, a.status);
            const bool exact = exact_all != 0;
            const bool use_si = sparse && exact;
            constexpr uint32_t id_s = idesc(kBN, 1u, 0u), id_i = idesc(kBN, 0u, 0u),
                               id_o = idesc(D, F16P ? 0u : 1u, 1u);
            constexpr int nparts = F16P ? 1 : 2;
            // S of key tile u for query tile x (its K in ring slot u % kSlots)
            auto issue_s = [&](int x, int u) {
                const uint32_t su = sbase + L::RING + (u % kSlots) * L::SLOT;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < D / 16; kk++)
                    mma_ss(tmem + x * kColsPerTile,
                           sdesc(sbase + L::Q + x * L::QT + (kk / 4) * (kRowsT * 128) + (kk % 4) * 32, 16, 1024, 2),
                           sdesc(su + L::SK + (kk / 4) * (kBN * 128) + (kk % 4) * 32, 16, 1024, 2), id_s, kk > 0);
            };
            auto done = [&](unsigned long long &x, uint32_t parity) { return mbar_try_wait(bar(x), parity); };
            // Full heads, event-driven issue: per query tile x, ns[x] is the
            // next key tile whose scores go out, np[x] the next whose P V does.
            // S(u) needs K(u) and the softmax to hold S(u-1) in registers (S's
            // columns are free), so it is computed while that softmax works on
            // tile u-1; P V(u) needs the softmax's P(u). Whichever query tile
            // is ready goes first. Ring slot t is released once both tiles'
            // P V(t) are issued. (Sparse heads keep a fixed order below: their
            // indexer scores overwrite P's columns, and there the event-driven
            // order measured slower.)
            if (!use_si) {
                int ns[2] = {0, 0}, np[2] = {0, 0}, fr = 0;
                unsigned long long t_idle = 0;
                bool idle = false;
                while (ok && (np[0] < ntx[0] || np[1] < ntx[1])) {
                    bool progress = false;
                    for (int x = 0; x < 2; x++) {
                        const int u = ns[x];
                        if (u < ntx[x] && done(bars.full[u % kSlots], (uint32_t)(u / kSlots) & 1u) &&
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
                            const uint32_t sl = sbase + L::RING + (v % kSlots) * L::SLOT;
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
                                mma_commit(bar(bars.slot_free[fr % kSlots]));
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
            } else {
                for (int t = 0; t < nt && ok; t++) {
                    const int slot = t % kSlots;
                    const uint32_t sl = sbase + L::RING + slot * L::SLOT;
                    ok = wait_or_abort(bar(bars.full[slot]), (uint32_t)(t / kSlots) & 1u, a.wait_ns, &abort_flag, a.status) &&
                         (!use_si || wait_or_abort(bar(bars.kh_ready[t % 2]), (uint32_t)(t / 2) & 1u, a.wait_ns, &abort_flag,
                                             a.status));
                    if (!ok) break;
                    for (int x = 0; x < 2 && ok; x++) {
                        if (t >= ntx[x]) continue;
                        if (t > 0)
                            ok = wait_or_abort(bar(bars.s_free[x]), (uint32_t)(t - 1) & 1u, a.wait_ns, &abort_flag, a.status);
                        if (!ok) break;
                        tc_fence_after();
                        const uint32_t colS = x * kColsPerTile;
#pragma unroll
                        for (int kk = 0; kk < D / 16; kk++)
                            mma_ss(tmem + colS,
                                   sdesc(sbase + L::Q + x * L::QT + (kk / 4) * (kRowsT * 128) + (kk % 4) * 32, 16, 1024, 2),
                                   sdesc(sl + L::SK + (kk / 4) * (kBN * 128) + (kk % 4) * 32, 16, 1024, 2), id_s, kk > 0);
                        if (use_si) {
                            // SI overwrites the columns that held P of tile t-1
                            if (t > 0)
                                ok = wait_or_abort(bar(bars.pv_done[x]), (uint32_t)(t - 1) & 1u, a.wait_ns, &abort_flag,
                                             a.status);
                            if (!ok) break;
                            tc_fence_after();
                            const uint32_t kh = sbase + L::KH + (t % 2) * L::KHB;
#pragma unroll
                            for (int kk = 0; kk < DI / 16; kk++)
                                mma_ss(tmem + colS + 64, sdesc(sbase + L::QE + x * L::QET + kk * 256, 128, DI / 8 * 128),
                                       sdesc(kh + kk * 256, 128, DI / 8 * 128), id_i, kk > 0);
                        }
                        mma_commit(bar(bars.s_ready[x]));
                    }
                    if (!ok) break;
                    if (use_si) mma_commit(bar(bars.kh_free[t % 2]));
                    for (int x = 0; x < 2 && ok; x++) {
                        if (t >= ntx[x]) continue;
                        ok = wait_or_abort(bar(bars.p_ready[x]), (uint32_t)t & 1u, a.wait_ns, &abort_flag, a.status);
                        if (!ok) break;
                        tc_fence_after();
                        const uint32_t colS = x * kColsPerTile;
#pragma unroll
                        for (int part = 0; part < nparts; part++)
#pragma unroll
                            for (int kk = 0; kk < kBN / 16; kk++)
                                mma_ts(tmem + colS + 128, tmem + colS + 64 + part * 32 + kk * 8,
                                       sdesc(sl + L::SV + kk * 2048, kBN * 128, 1024, 2), id_o,
                                       (t > 0 || part > 0 || kk > 0));
                        mma_commit(bar(bars.pv_done[x]));
                    }
                    if (ok) mma_commit(bar(bars.slot_free[slot]));
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

template <int D, int DI, bool F16P>
void *pp_kernel(size_t *smem) {
    if constexpr (!PLay<D, DI>::FITS) {
        return nullptr;
    } else {
        *smem = PLay<D, DI>::TOTAL;
        return (void *)routed_pp_kernel<D, DI, F16P>;
    }
}

template <int D, bool F16P>
void *pp_kernel_d(int DI, size_t *smem) {
    switch (DI) {
        case 16: return pp_kernel<D, 16, F16P>(smem);
        case 32: return pp_kernel<D, 32, F16P>(smem);
        case 64: return pp_kernel<D, 64, F16P>(smem);
        default: return pp_kernel<D, 128, F16P>(smem);
    }
}

template <bool F16P>
void *pp_kernel_for(const Shape &s, size_t *smem) {
    return s.D == 64 ? pp_kernel_d<64, F16P>(s.D_I, smem) : pp_kernel_d<128, F16P>(s.D_I, smem);
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

esa_status launch_routed_pp(const uint16_t *q, const uint16_t *k, const uint16_t *v, const int8_t *qI,
                            const int8_t *kI, const int32_t *wI, const uint8_t *route, const int32_t *thr,
                            const Shape &s, float scale, const float *g, const uint16_t *lin, float *out,
                            void *pp_ws, int32_t *status, cudaStream_t st, const uint64_t *mask) {
    PpArgs a{};
    a.mask = mask;
    a.mask_w64 = sel_mask_words(s) / 2;
    a.lin = lin;
    a.qI = qI;
    a.wI = wI;
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
    a.relu = relu_of(s) ? 1 : 0;
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
    CUtensorMap tq, tk, tv, tvh, tki;
    if (!map_rows_heads_d(&tq, q, s.B * s.Tq, s.Hq, s.D, kRowsT) || !map_rows_heads_d(&tk, k, s.B * s.Tk, s.Hkv, s.D, kBN) ||
        !map_rows_heads_d(&tv, v, s.B * s.Tk, s.Hkv, s.D, kBN) || !map_rows_heads_d(&tvh, vh, s.B * s.Tk, s.Hkv, s.D, kBN) ||
        !map_rows_bytes(&tki, kI, s.B * s.Tk, s.D_I, kBN))
        return ESA_ERR_CUDA;
    if (!ensure_smem(fn16, smem16) || !ensure_smem(fn2, smem2)) return ESA_ERR_CUDA;
    // the fp16-P variant; then the bf16 hi + lo variant, whose blocks return at
    // once unless some value is beyond fp16 (tensor maps copy bits: the fp16
    // copy uses the same 2-byte map shape)
    void *args16[] = {(void *)&a, (void *)&tq, (void *)&tk, (void *)&tvh, (void *)&tki};
    if (cudaLaunchKernel(fn16, dim3((unsigned)blocks), dim3(kThreads), args16, smem16, st) != cudaSuccess)
        return ESA_ERR_CUDA;
    void *args2[] = {(void *)&a, (void *)&tq, (void *)&tk, (void *)&tv, (void *)&tki};
    cudaError_t ce = cudaLaunchKernel(fn2, dim3((unsigned)blocks), dim3(kThreads), args2, smem2, st);
    return ce == cudaSuccess ? ESA_OK : ESA_ERR_CUDA;
}

}  // namespace esa
