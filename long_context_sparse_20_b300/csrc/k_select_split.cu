// Top-K selection for few query rows with long prefixes (decode).
//
// Method: the Indexer scores the query against every causal-prefix position
// and the K best positions are kept ("超大规模MoE架构中稀疏注意力机制的演进与实践",
// section 二.1, K = 2048; no RoPE, section 二.2). Ties go to the lower position.
//
// Design (one launch, one co-resident block per SM):
//   * each query row's prefix 0..p is cut into `chunks` contiguous spans,
//     one block per span; the block streams its span of kI once from HBM
//     through a ring of shared-memory stages, one bulk copy per stage
//     issued by one thread and landing on the slot's mbarrier (128 KB in
//     flight per SM, which a one-block-per-SM stream needs to approach HBM
//     bandwidth; ~94% of the measured copy rate, against ~80% with
//     per-thread 16-byte cp.async), scores each key with dp4a and keeps the int32
//     scores in shared memory — the score row never reaches HBM;
//   * level 1: a histogram exact for |s| < 2048 (one bin per value) with 64
//     log bins per octave above. Every block adds its bins to the row's
//     global histogram (L2 atomics) and publishes, for the exact window, how
//     many of its own scores lie at or above each value. After ONE bounded
//     barrier among the row's blocks every block finds the bin of the K-th
//     largest score; when that bin is a single value T (always, for scores
//     below 2048 in magnitude) each block reads from the earlier blocks'
//     publications how many scores above T and ties at T precede its span and
//     writes its part of the ascending index list — no further exchange;
//   * wider scores fall back to exact refinement levels (4096 bins of the
//     crossing bucket per level, a barrier each) before the same final write.
// Control state lives in the caller's workspace in two copies selected by
// the parity of a call counter (the epoch): a call works on one copy and
// zeroes the other (which the previous call used), so no call has to wait
// at its end to return its state to zero. The last block to arrive advances
// the epoch.
//
// The fused decode step (the D > 0 instantiations) continues in the same
// launch with the rest of the Gated DSA path (the pseudo-code of section
// 四.1: gather the selected K/V, scaled dot-product attention, then the gate
// mix final = g*attn + (1-g)*linear_output, sections 二.3 and 四.1):
//   * the ordered write also lists the block's own selected positions in
//     shared memory; each block gathers those keys' K and V rows (16-byte
//     cp.async, two stages in flight) and runs warp MMAs for every query
//     head: warp (m-tile, key group) scores 8 keys of each stage against 16
//     heads (bf16 m16n8k16, fp32 accumulation) and keeps its own online
//     softmax (max, sum, unnormalised output) over its keys; P enters P V
//     as a bf16 hi + lo pair (m16n8k8), ~16 significant bits;
//   * the warps of a block merge in shared memory in a fixed order, and the
//     block publishes one partial (max, sum, output) per head;
//   * after a second barrier of the row each block merges all of the row's
//     partials for its slice of the Hq x D outputs (online rescaling, fixed
//     order), applies the gate mix and writes out and lse.
// The score row, the index list and the attention partials never leave
// the chip except the partials' one round trip through L2.
#include <algorithm>

#include "esa_device.cuh"
#include "esa_internal.h"

namespace esa {

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kRingBytes = 128 * 1024;  // kI bytes in flight per SM (stages of kThreads keys)
constexpr int kMinStages = 2;
constexpr size_t kSmemBudget = 227 * 1024;
constexpr int kExact = 2048;        // level 1 holds one bin per value for |s| < kExact
constexpr int kHalf1 = kExact + 21 * 64;  // bin of score 0; octaves 2^11..2^31, 64 bins each
constexpr int kNB1 = 2 * kHalf1 + 1;
constexpr int kNB2 = 4096;
constexpr int kMaxChunk = 16384;
// exact publication window: bins kHalf1-(kExact-1) .. kHalf1+kExact
constexpr int kWinLo = kHalf1 - (kExact - 1);
constexpr int kWin = 2 * kExact;
// level-1 histogram padded so that every thread reads 16 bins with 16-byte loads
constexpr int kNB1P = 16 * kThreads;
static_assert(kNB1P >= kNB1, "padded level-1 histogram");
// per (row, parity) control words: [0] barrier counter, then the level
// histograms (level 1 padded, level 2, level 3); rounded to 256 bytes
constexpr size_t kRowCtrl = ((4 + kNB1P + 2 * (size_t)kNB2) + 63) / 64 * 64;
// per-block publication: [0] lowest bin, [1] highest bin, [2] count,
// [4 .. 4+kWin) level-1 suffix counts over the exact window, then the deeper
// exact level: [0] count above the bucket, [1+v] suffix counts, [1+nb] = 0
constexpr size_t kPubDeep = 4 + kWin;
constexpr size_t kPubWords = kPubDeep + kNB2 + 4;
// workspace header words: [0] epoch, [1], [2] rows used by the last call of
// each parity, [3] arrivals of the current call
constexpr size_t kHdrBytes = 256;

__device__ __forceinline__ int bin1(int s) {
    unsigned a = s < 0 ? 0u - (unsigned)s : (unsigned)s;
    int m;
    if (a < (unsigned)kExact) {
        m = (int)a;
    } else {
        int e = 31 - __clz(a);
        m = kExact + (e - 11) * 64 + (int)((a >> (e - 6)) & 63u);
    }
    return s >= 0 ? kHalf1 + m : kHalf1 - m;
}

__device__ __forceinline__ void bin1_range(int bin, long long &lo, long long &hi) {
    int m = bin >= kHalf1 ? bin - kHalf1 : kHalf1 - bin;
    long long alo, ahi;
    if (m < kExact) {
        alo = ahi = m;
    } else {
        int e = 11 + (m - kExact) / 64, mant = (m - kExact) % 64;
        alo = (long long)(64 + mant) << (e - 6);
        ahi = ((long long)(65 + mant) << (e - 6)) - 1;
    }
    if (bin >= kHalf1) {
        lo = alo;
        hi = ahi;
    } else {
        lo = -ahi;
        hi = -alo;
    }
    if (lo < INT32_MIN) lo = INT32_MIN;
    if (hi > INT32_MAX) hi = INT32_MAX;
}

struct SelArgs {
    const int8_t *qI, *kI;
    const int32_t *wI;
    int32_t *idx, *cnt;
    unsigned *hdr, *ctrl, *pub;
    int32_t *status;
    long long Tq, Tk, q_offset, wait_ns;
    int pos_div;  // rows per query position (one per indexer head with per-head sets)
    int relu;     // ReLU on the (single) indexer head's dot product
    int H_I, K, chunks, rows, extra, stages;
    int ctrl_cap;  // rows of control state (both parities) the workspace holds
    // the fused decode step's attention stage (the D > 0 instantiations)
    const uint16_t *q, *k, *v, *lin;
    const float *g;
    float *out, *lse;
    float *part;  // [rows * chunks][Hq][D] unnormalised block outputs
    float2 *ml;   // [rows * chunks][Hq] (max, sum) of the block's logits, log2 domain
    int Hq, Hkv, MPK, MTT, KG, sel_cap;
    float scale_log2;
    int off_q, off_sel, off_aux;  // dynamic shared memory offsets (bytes)
};

constexpr int kMaxStages = 32;  // ring slots, at most (D_I >= 16: stages of >= 8 KB)

struct Smem {
    unsigned long long full[kMaxStages];  // per ring slot: the stage's bulk copy has landed
    unsigned h1[kNB1];
    int32_t q[16 * 32];  // indexer query words [H_I][D_I/4]
    int32_t w[16];
    unsigned red[64];
    unsigned wsum[2][kWarps];
    int mn[kWarps], mx[kWarps];
    int flag, bin, epoch, ru_other;
    unsigned above;
    // followed by the scores of the block's span (int32)
};

// Bytes of the Smem header in dynamic shared memory (the scores that follow
// start on a 128-byte boundary: 16-byte vector reads).
constexpr size_t kSmemHdr = (sizeof(Smem) + 127) & ~size_t(127);

// Block-wide: among bins [0,nb) of the global histogram h, find v with
// sum_{u>v} h[u] < need <= sum_{u>=v} h[u]. Result in sm.bin / sm.above
// (sm.bin = -1 if there is none). Every thread reads its own contiguous 16
// bins with four independent 16-byte loads (h is 16-byte aligned and padded
// with zeros to 16 * kThreads words): one L2 round trip, no staging.
__device__ void find_crossing(const unsigned *h, unsigned need, Smem &sm) {
    int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) sm.bin = -1;
    unsigned v[16];
    const uint4 *h4 = reinterpret_cast<const uint4 *>(h) + tid * 4;
#pragma unroll
    for (int c = 0; c < 4; c++) {
        uint4 x = __ldcg(h4 + c);
        v[4 * c] = x.x;
        v[4 * c + 1] = x.y;
        v[4 * c + 2] = x.z;
        v[4 * c + 3] = x.w;
    }
    unsigned seg = 0;
#pragma unroll
    for (int i = 0; i < 16; i++) seg += v[i];
    unsigned x = seg;  // inclusive suffix sum within the warp (higher lanes = higher bins)
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        unsigned y = __shfl_down_sync(0xffffffffu, x, d);
        if (lane + d < 32) x += y;
    }
    if (lane == 0) sm.red[warp] = x;
    __syncthreads();
    unsigned higher = 0;
    for (int w = warp + 1; w < kWarps; w++) higher += sm.red[w];
    unsigned incl = x + higher, excl = incl - seg;
    if (excl < need && need <= incl) {
        unsigned a = excl;
        int found = -1;
        unsigned ab = 0;
#pragma unroll
        for (int i = 15; i >= 0; i--) {
            if (found < 0 && a + v[i] >= need) {
                found = i;
                ab = a;
            }
            a += v[i];
        }
        sm.bin = tid * 16 + found;
        sm.above = ab;
    }
    __syncthreads();
}

// The same search over nb <= kNB2 bins of a deeper level, staged in shared
// memory first (`stage`, >= nb words).
__device__ void find_crossing_staged(const unsigned *h, int nb, unsigned need, unsigned *stage, Smem &sm) {
    int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) sm.bin = -1;
#pragma unroll 8
    for (int i = tid; i < nb; i += kThreads) stage[i] = __ldcg(h + i);
    __syncthreads();
    int per = (nb + kThreads - 1) / kThreads;
    int b0 = tid * per, b1 = min(nb, b0 + per);
    unsigned seg = 0;
    for (int v = b0; v < b1; v++) seg += stage[v];
    unsigned x = seg;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        unsigned y = __shfl_down_sync(0xffffffffu, x, d);
        if (lane + d < 32) x += y;
    }
    if (lane == 0) sm.red[warp] = x;
    __syncthreads();
    unsigned higher = 0;
    for (int w = warp + 1; w < kWarps; w++) higher += sm.red[w];
    unsigned incl = x + higher, excl = incl - seg;
    if (excl < need && need <= incl) {
        unsigned a = excl;
        for (int v = b1 - 1; v >= b0; v--) {
            unsigned c = stage[v];
            if (a + c >= need) {
                sm.bin = v;
                sm.above = a;
                break;
            }
            a += c;
        }
    }
    __syncthreads();
}

// Block-wide suffix counts of the shared histogram h over bins [lo, hi]:
// dst[v - wlo] = sum_{lo <= u <= hi, u >= v} h[u] for v in [lo, hi] ∩ [wlo, whi].
__device__ void publish_suffix(const unsigned *h, int lo, int hi, unsigned *dst, int wlo, int whi, Smem &sm) {
    int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int nb = hi - lo + 1;
    int per = (nb + kThreads - 1) / kThreads;
    int b0 = lo + tid * per, b1 = min(hi + 1, b0 + per);
    unsigned seg = 0;
    for (int v = b0; v < b1; v++) seg += h[v];
    unsigned x = seg;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        unsigned y = __shfl_down_sync(0xffffffffu, x, d);
        if (lane + d < 32) x += y;
    }
    __syncthreads();
    if (lane == 0) sm.red[32 + warp] = x;
    __syncthreads();
    unsigned a = x - seg;  // bins above b1-1 within the warp
    for (int w = warp + 1; w < kWarps; w++) a += sm.red[32 + w];
    for (int v = b1 - 1; v >= b0; v--) {
        a += h[v];
        if (v >= wlo && v <= whi) dst[v - wlo] = a;
    }
}

// Thread 0 only, once the block has read the header: count this block's
// arrival in the call (issued early; the result is needed only later).
__device__ __forceinline__ unsigned epoch_arrive(unsigned *hdr) { return atomicAdd(hdr + 3, 1u); }
// Thread 0 only: the last block to arrive records the rows this parity used
// and advances the epoch (every block has read the header by then).
__device__ __forceinline__ void epoch_finish(unsigned *hdr, unsigned old, int epoch, int rows) {
    if (old == gridDim.x - 1) {
        volatile unsigned *vh = hdr;
        vh[1 + (epoch & 1)] = (unsigned)rows;
        vh[3] = 0u;
        vh[0] = (unsigned)(epoch + 1);
    }
}

// One step of the online softmax merge: fold (mx, lx, ox) into (m, l, o).
// Empty parts (max -inf) contribute nothing.
__device__ __forceinline__ void merge_part(float &m, float &l, float4 &o, float mx, float lx, float4 ox) {
    const float mn = fmaxf(m, mx);
    if (mn == -INFINITY) return;
    const float s1 = m == -INFINITY ? 0.f : exp2f(m - mn), s2 = mx == -INFINITY ? 0.f : exp2f(mx - mn);
    l = l * s1 + lx * s2;
    o.x = o.x * s1 + ox.x * s2;
    o.y = o.y * s1 + ox.y * s2;
    o.z = o.z * s1 + ox.z * s2;
    o.w = o.w * s1 + ox.w * s2;
    m = mn;
}

// Earlier blocks' counts above T and at T, published before the row's
// barrier; the fused step issues their loads early and reads them late.
struct PendingPub {
    bool have;
    int vstar, clo, chi;
    unsigned tot, s0, s1;
};

// The fused decode step after the threshold T is known: this block's
// selected keys (those above T, then the ties it takes) listed in shared
// memory with the first stage's gathers issued as soon as the keys above T
// are listed; attention over the list (warp MMAs, per-warp online
// softmax); the warps of each m-tile merged in a fixed-order tree; the
// block's partial published; the row's second barrier; this block's slice
// of the merged, gated outputs. A whole prefix (n <= K) attends to every
// key of its span, positions lo .. lo+n_span-1.
template <int D>
__device__ __noinline__ void fused_tail(const SelArgs &a, unsigned char *smem_raw, unsigned char *ring,
                                           const int32_t *sc, Smem &sm, long long row, long long b, int ci,
                                           long long lo, int span, bool whole, int n_span, int T, unsigned above,
                                           unsigned gt_b, unsigned eq_b, const PendingPub &pp, unsigned *bar,
                                           int nbar) {
    constexpr int RS = D + 8;   // padded row stride of the Q and K/V tiles (bf16 elements)
    constexpr int RSO = D + 8;  // padded row stride of the merge buffer (fp32): conflict-free float2 per half-warp
    constexpr int DK = D / 16;  // k-steps of Q K^T
    constexpr int DN = D / 8;   // output n-tiles
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g8 = lane >> 2, c4 = lane & 3;
    const int Hkv = a.Hkv, KG = a.KG, SK = 8 * KG, SR = SK * Hkv, K = a.K;
    const int mt = warp / KG, kg = warp % KG;
    const bool active = mt < a.MTT;
    const int kvh = active ? mt / a.MPK : 0;
    const uint16_t *Qs = reinterpret_cast<const uint16_t *>(smem_raw + a.off_q);
    int32_t *sel = reinterpret_cast<int32_t *>(smem_raw + a.off_sel);
    float *Mw = reinterpret_cast<float *>(smem_raw + a.off_aux);  // [warps][16] per-warp max
    float *Lw = Mw + kWarps * 16;                                   // [warps][16] per-warp sum
    uint16_t *KV = reinterpret_cast<uint16_t *>(ring);  // [2 stages][K rows, V rows][RS]
    const long long kvrow0 = b * a.Tk * Hkv;             // K/V row of (b, position 0, head 0)
    const unsigned lt = lanemask_lt();
    int n_sel = 0;

    // tile rows [r0, r1) of stage s (row r: key s*SK + r/Hkv of the list,
    // key/value head r%Hkv); keys at or past n_valid are zero-filled
    auto gather_rows = [&](int s, int r0, int r1, int n_valid) {
        uint16_t *Kt = KV + (size_t)(s & 1) * 2 * SR * RS;
        uint16_t *Vt = Kt + (size_t)SR * RS;
        constexpr int CH = D / 8;
        for (int i = tid; i < (r1 - r0) * CH; i += kThreads) {
            const int r = r0 + i / CH, ch = i % CH;
            const int key = s * SK + r / Hkv, hh = r % Hkv;
            bool valid = key < n_valid;
            long long pos = valid ? (whole ? lo + key : (long long)sel[key]) : 0;
            if (pos < 0 || pos >= a.Tk) {  // consistency check; never reached
                set_status(a.status, ESA_ERR_INTERNAL);
                pos = 0;
                valid = false;
            }
            const long long off = ((kvrow0 + pos * Hkv + hh) * D) + ch * 8;
            cp_async16_zfill(smem_u32(Kt + r * RS + ch * 8), a.k + off, valid);
            cp_async16_zfill(smem_u32(Vt + r * RS + ch * 8), a.v + off, valid);
        }
    };

    cp_async_wait<0>();  // the Q tile (nothing else is in flight)
    __syncthreads();     // the ring is idle
    if (whole) {
        n_sel = n_span;
        gather_rows(0, 0, SR, n_sel);
        cp_async_commit();
    } else {
        // ---- keys above T and at T, per warp over its contiguous segment
        const int seg = ((span + kWarps * 32 - 1) / (kWarps * 32)) * 32;
        const int s0 = warp * seg, s1 = min(span, s0 + seg);
        unsigned wgt = 0, weq = 0;
        for (int j0 = s0; j0 < s1; j0 += 32) {
            const int j = j0 + lane;
            const int sv = j < s1 ? sc[j] : INT32_MIN;
            const unsigned gem = __ballot_sync(0xffffffffu, sv >= T);
            if (gem) {
                const unsigned eqm = __ballot_sync(0xffffffffu, sv == T);
                wgt += __popc(gem & ~eqm);
                weq += __popc(eqm);
            }
        }
        if (lane == 0) {
            sm.wsum[0][warp] = wgt;
            sm.wsum[1][warp] = weq;
        }
        __syncthreads();
        // exclusive prefix of both counts over the warps (every warp alike)
        const unsigned vg = lane < kWarps ? sm.wsum[0][lane] : 0u, ve = lane < kWarps ? sm.wsum[1][lane] : 0u;
        unsigned ig = vg, ie = ve;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const unsigned ug = __shfl_up_sync(0xffffffffu, ig, d), ue = __shfl_up_sync(0xffffffffu, ie, d);
            if (lane >= d) {
                ig += ug;
                ie += ue;
            }
        }
        const unsigned tot_gt = __shfl_sync(0xffffffffu, ig, 31), tot_eq = __shfl_sync(0xffffffffu, ie, 31);
        const unsigned base_gt = __shfl_sync(0xffffffffu, ig - vg, warp);
        const unsigned base_eq = __shfl_sync(0xffffffffu, ie - ve, warp);
        const int n_gt = (int)min(tot_gt, (unsigned)a.sel_cap);
        if (tot_gt > (unsigned)a.sel_cap && tid == 0) set_status(a.status, ESA_ERR_INTERNAL);  // never reached
        // ---- the keys above T, in position order
        if (wgt) {
            unsigned o = base_gt;
            for (int j0 = s0; j0 < s1; j0 += 32) {
                const int j = j0 + lane;
                const int sv = j < s1 ? sc[j] : INT32_MIN;
                const unsigned gtm = __ballot_sync(0xffffffffu, sv > T);
                if (gtm) {
                    const unsigned li = o + __popc(gtm & lt);
                    if (((gtm >> lane) & 1u) && li < (unsigned)a.sel_cap) sel[li] = (int32_t)(lo + j);
                    o += __popc(gtm);
                }
            }
        }
        __syncthreads();
        // ---- the first stage's keys above T go out now (group A)
        const int kA = min(n_gt, SK);
        gather_rows(0, 0, kA * Hkv, n_gt);
        cp_async_commit();
        // ---- earlier blocks' counts (their loads were issued before the passes)
        unsigned gtp = gt_b, eqp = eq_b;
        if (pp.have) {
            const unsigned S0 = pp.vstar <= pp.clo ? pp.tot : (pp.vstar > pp.chi ? 0u : pp.s0);
            const unsigned S1 = pp.vstar + 1 <= pp.clo ? pp.tot : (pp.vstar + 1 > pp.chi ? 0u : pp.s1);
            gtp += S1;
            eqp += S0 - S1;
        }
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) {
            gtp += __shfl_xor_sync(0xffffffffu, gtp, d);
            eqp += __shfl_xor_sync(0xffffffffu, eqp, d);
        }
        if (lane == 0) {
            sm.red[warp] = gtp;
            sm.red[32 + warp] = eqp;
        }
        __syncthreads();
        unsigned gt_before = lane < kWarps ? sm.red[lane] : 0u, eq_before = lane < kWarps ? sm.red[32 + lane] : 0u;
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) {
            gt_before += __shfl_xor_sync(0xffffffffu, gt_before, d);
            eq_before += __shfl_xor_sync(0xffffffffu, eq_before, d);
        }
        const unsigned need_ties = (unsigned)K - above;  // ties at T the row takes, >= 1
        const unsigned take = eq_before >= need_ties ? 0u : min(tot_eq, need_ties - eq_before);
        // ---- the ties this block takes: its first `take` ties, after the keys above T
        if (weq && base_eq < take) {
            unsigned o = base_eq;
            for (int j0 = s0; j0 < s1 && o < take; j0 += 32) {
                const int j = j0 + lane;
                const int sv = j < s1 ? sc[j] : INT32_MIN;
                const unsigned eqm = __ballot_sync(0xffffffffu, sv == T);
                if (eqm) {
                    const unsigned ti = o + __popc(eqm & lt);
                    const unsigned li = (unsigned)n_gt + ti;
                    if (((eqm >> lane) & 1u) && ti < take && li < (unsigned)a.sel_cap) sel[li] = (int32_t)(lo + j);
                    o += __popc(eqm);
                }
            }
        }
        n_sel = (int)min((unsigned)n_gt + take, (unsigned)a.sel_cap);
        __syncthreads();
        // ---- the rest of the first stage (group B: ties, zero fill)
        gather_rows(0, kA * Hkv, SR, n_sel);
        cp_async_commit();
        // ---- the ordered index list, when the caller wants it (overlaps the gathers)
        if (a.idx) {
            int32_t *idx_row = a.idx + row * (long long)K;
            const unsigned blk_base = gt_before + min(eq_before, need_ties);
            unsigned out = blk_base + base_gt + min(base_eq, take);
            unsigned tie_seen = base_eq;
            for (int j0 = s0; j0 < s1; j0 += 32) {
                const int j = j0 + lane;
                const int sv = j < s1 ? sc[j] : INT32_MIN;
                const unsigned gem = __ballot_sync(0xffffffffu, sv >= T);
                if (gem == 0u) continue;
                const unsigned eqm = __ballot_sync(0xffffffffu, sv == T);
                const unsigned gtm = gem & ~eqm;
                const unsigned ne = __popc(eqm);
                const unsigned tk = tie_seen >= take ? 0u : min(ne, take - tie_seen);
                unsigned tmask = 0u;
                if (tk == ne) {
                    tmask = eqm;
                } else if (tk > 0u) {  // the lowest `tk` ties (warp-uniform branch)
                    tmask = __ballot_sync(0xffffffffu, ((eqm >> lane) & 1u) && __popc(eqm & lt) < tk);
                }
                const unsigned selm = gtm | tmask;
                if ((selm >> lane) & 1u) {
                    const unsigned pos = out + __popc(selm & lt);
                    if (pos < (unsigned)K) idx_row[pos] = (int32_t)(lo + j);
                    else set_status(a.status, ESA_ERR_INTERNAL);
                }
                out += __popc(selm);
                tie_seen += ne;
            }
            if (ci == 0 && tid == 0 && a.cnt) a.cnt[row] = K;
        }
    }

    // ---- attention over the list: stage s holds keys s*SK .. s*SK+SK-1
    const int nst = (n_sel + SK - 1) / SK;
    float o[DN][4];
#pragma unroll
    for (int i = 0; i < DN; i++) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float mr[2] = {-INFINITY, -INFINITY}, lr[2] = {0.f, 0.f};  // rows g8, g8+8 of the m-tile
    const int qrow = mt * 16 + (lane & 15);
    const int krow = (kg * 8 + (lane & 7)) * Hkv + kvh;  // this lane's K/V tile row for ldmatrix
    for (int s = 0; s < nst; s++) {
        if (s + 1 < nst) {
            gather_rows(s + 1, 0, SR, n_sel);
            cp_async_commit();
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        if (active) {
            const uint16_t *Kt = KV + (size_t)(s & 1) * 2 * SR * RS;
            const uint16_t *Vt = Kt + (size_t)SR * RS;
            // S (16 heads x 8 keys) = Q K^T
            float sc4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int kk = 0; kk < DK; kk += 2) {
                uint32_t qa[4], qb[4], b0, b1, b2, b3;
                ldmatrix_x4(smem_u32(Qs + qrow * RS + kk * 16 + (lane >> 4) * 8), qa[0], qa[1], qa[2], qa[3]);
                ldmatrix_x4(smem_u32(Qs + qrow * RS + (kk + 1) * 16 + (lane >> 4) * 8), qb[0], qb[1], qb[2], qb[3]);
                ldmatrix_x4(smem_u32(Kt + krow * RS + kk * 16 + (lane >> 3) * 8), b0, b1, b2, b3);
                mma_bf16_16816(sc4, qa, b0, b1);
                mma_bf16_16816(sc4, qb, b2, b3);
            }
            // online softmax in the log2 domain over this warp's keys
            const int key0 = s * SK + kg * 8 + 2 * c4;
            const bool v0 = key0 < n_sel, v1 = key0 + 1 < n_sel;
            const float x0 = v0 ? sc4[0] * a.scale_log2 : -INFINITY, x1 = v1 ? sc4[1] * a.scale_log2 : -INFINITY;
            const float x2 = v0 ? sc4[2] * a.scale_log2 : -INFINITY, x3 = v1 ? sc4[3] * a.scale_log2 : -INFINITY;
            float mx[2] = {fmaxf(x0, x1), fmaxf(x2, x3)}, corr[2];
#pragma unroll
            for (int r = 0; r < 2; r++) {
                mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
                mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
                const float mnew = fmaxf(mr[r], mx[r]);
                const float muse = mnew == -INFINITY ? 0.f : mnew;
                corr[r] = exp2f(mr[r] - muse);
                mr[r] = mnew;
                mx[r] = muse;
            }
            const float p0 = exp2f(x0 - mx[0]), p1 = exp2f(x1 - mx[0]);
            const float p2 = exp2f(x2 - mx[1]), p3 = exp2f(x3 - mx[1]);
            float rs[2] = {p0 + p1, p2 + p3};
#pragma unroll
            for (int r = 0; r < 2; r++) {
                rs[r] += __shfl_xor_sync(0xffffffffu, rs[r], 1);
                rs[r] += __shfl_xor_sync(0xffffffffu, rs[r], 2);
                lr[r] = lr[r] * corr[r] + rs[r];
            }
#pragma unroll
            for (int dn = 0; dn < DN; dn++) {
                o[dn][0] *= corr[0];
                o[dn][1] *= corr[0];
                o[dn][2] *= corr[1];
                o[dn][3] *= corr[1];
            }
            // P (16 heads x 8 keys) as bf16 hi + lo A fragments, straight from
            // the score layout; O += P V over every output column
            const uint32_t ah0 = pack_bf16(p0, p1), ah1 = pack_bf16(p2, p3);
            const uint32_t al0 = pack_bf16(p0 - bf16lo(ah0), p1 - bf16hi(ah0));
            const uint32_t al1 = pack_bf16(p2 - bf16lo(ah1), p3 - bf16hi(ah1));
#pragma unroll
            for (int dq = 0; dq < D / 32; dq++) {
                uint32_t vb[4];
                ldmatrix_x4_trans(smem_u32(Vt + krow * RS + dq * 32 + (lane >> 3) * 8), vb[0], vb[1], vb[2], vb[3]);
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    mma_bf16_1688(o[4 * dq + i], ah0, ah1, vb[i]);
                    mma_bf16_1688(o[4 * dq + i], al0, al1, vb[i]);
                }
            }
        }
        __syncthreads();  // the stage's buffer is free for the gather two stages on
    }
    cp_async_wait<0>();  // nothing in flight before the ring is reused

    // ---- merge the key groups of each m-tile: scale to the m-tile's
    // per-row maximum, then a fixed-order pairwise tree in shared memory
    if (active && c4 == 0) {
        Mw[warp * 16 + g8] = mr[0];
        Mw[warp * 16 + g8 + 8] = mr[1];
        Lw[warp * 16 + g8] = lr[0];
        Lw[warp * 16 + g8 + 8] = lr[1];
    }
    __syncthreads();
    float Mrow[2] = {-INFINITY, -INFINITY};
    if (active) {
#pragma unroll
        for (int r = 0; r < 2; r++) {
            for (int k2 = 0; k2 < KG; k2++) Mrow[r] = fmaxf(Mrow[r], Mw[(mt * KG + k2) * 16 + g8 + 8 * r]);
            const float scl = mr[r] == -INFINITY ? 0.f : exp2f(mr[r] - Mrow[r]);
#pragma unroll
            for (int dn = 0; dn < DN; dn++) {
                o[dn][2 * r] *= scl;
                o[dn][2 * r + 1] *= scl;
            }
        }
    }
    float *Ob = reinterpret_cast<float *>(ring);  // [pairs][MTT * 16][RSO]
    for (int step = 1; step < KG; step <<= 1) {
        const int pair = kg / (2 * step);
        float *slot = Ob + ((size_t)pair * a.MTT + mt) * 16 * RSO;
        if (active && kg % (2 * step) == step) {
#pragma unroll
            for (int r = 0; r < 2; r++)
#pragma unroll
                for (int dn = 0; dn < DN; dn++)
                    *reinterpret_cast<float2 *>(slot + (g8 + 8 * r) * RSO + dn * 8 + 2 * c4) =
                        make_float2(o[dn][2 * r], o[dn][2 * r + 1]);
        }
        __syncthreads();
        if (active && kg % (2 * step) == 0 && kg + step < KG) {
#pragma unroll
            for (int r = 0; r < 2; r++)
#pragma unroll
                for (int dn = 0; dn < DN; dn++) {
                    const float2 w = *reinterpret_cast<const float2 *>(slot + (g8 + 8 * r) * RSO + dn * 8 + 2 * c4);
                    o[dn][2 * r] += w.x;
                    o[dn][2 * r + 1] += w.y;
                }
        }
        __syncthreads();
    }
    // ---- publish the block's partial of every query head, from registers
    const int G = a.Hq / Hkv;
    const long long prow = row * a.chunks + ci;  // this block's partial slot
    if (active && kg == 0) {
#pragma unroll
        for (int r = 0; r < 2; r++) {
            const int hl = (mt % a.MPK) * 16 + g8 + 8 * r;
            if (hl >= G) continue;
            const int head = (mt / a.MPK) * G + hl;
            float *dst = a.part + (prow * a.Hq + head) * D + 2 * c4;
#pragma unroll
            for (int dn = 0; dn < DN; dn++)
                *reinterpret_cast<float2 *>(dst + dn * 8) = make_float2(o[dn][2 * r], o[dn][2 * r + 1]);
            if (c4 == 0) {
                float L = 0.f;
                for (int k2 = 0; k2 < KG; k2++) {
                    const float mw = Mw[(mt * KG + k2) * 16 + g8 + 8 * r];
                    if (mw != -INFINITY) L += Lw[(mt * KG + k2) * 16 + g8 + 8 * r] * exp2f(mw - Mrow[r]);
                }
                a.ml[prow * a.Hq + head] = make_float2(Mrow[r], L);
            }
        }
    }

    // ---- the row's second barrier: every block's partial is published
    if (!group_barrier(bar, (unsigned)((nbar + 1) * a.chunks + a.extra), a.wait_ns, a.status, &sm.flag)) return;

    // ---- this block's slice of the row's Hq x D outputs: groups of LP
    // lanes merge all blocks' partials of one float4 (lane l takes blocks
    // l, l+LP, ...; then a butterfly over the group), normalise, gate, write
    const int HD = a.Hq * D;
    const int per = ((HD + a.chunks - 1) / a.chunks + 3) / 4 * 4;
    const int e0 = ci * per, e1 = min(HD, e0 + per);
    const int nE4 = max(0, (e1 - e0) / 4);
    int LP = 32;
    while (LP > 1 && nE4 * LP > kThreads) LP >>= 1;
    const int units = kThreads / LP;
    const int gl = tid % LP, u = tid / LP;
    const bool gated = a.g != nullptr && a.lin != nullptr;
    const long long base = row * a.chunks;
    for (int f0 = 0; f0 < nE4; f0 += units) {
        const int f = f0 + u;
        const bool have = f < nE4;
        const int e = e0 + 4 * (have ? f : 0), h = e / D, c = e % D;
        float m = -INFINITY, l = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (have) {
            int cc = gl;
            for (; cc + 3 * LP < a.chunks; cc += 4 * LP) {  // four blocks' loads in flight
                float2 x[4];
                float4 y[4];
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    const long long pr = base + cc + q * LP;
                    x[q] = __ldcg(a.ml + pr * a.Hq + h);
                    y[q] = __ldcg(reinterpret_cast<const float4 *>(a.part + (pr * a.Hq + h) * D + c));
                }
#pragma unroll
                for (int q = 0; q < 4; q++) merge_part(m, l, acc, x[q].x, x[q].y, y[q]);
            }
            for (; cc < a.chunks; cc += LP) {
                const long long pr = base + cc;
                const float2 x = __ldcg(a.ml + pr * a.Hq + h);
                const float4 y = __ldcg(reinterpret_cast<const float4 *>(a.part + (pr * a.Hq + h) * D + c));
                merge_part(m, l, acc, x.x, x.y, y);
            }
        }
        for (int d = LP / 2; d > 0; d >>= 1) {  // the group's lanes, in a fixed butterfly
            const float mo = __shfl_xor_sync(0xffffffffu, m, d), lo2 = __shfl_xor_sync(0xffffffffu, l, d);
            float4 ao;
            ao.x = __shfl_xor_sync(0xffffffffu, acc.x, d);
            ao.y = __shfl_xor_sync(0xffffffffu, acc.y, d);
            ao.z = __shfl_xor_sync(0xffffffffu, acc.z, d);
            ao.w = __shfl_xor_sync(0xffffffffu, acc.w, d);
            merge_part(m, l, acc, mo, lo2, ao);
        }
        if (have && gl == 0) {
            const float inv = l > 0.f ? 1.f / l : 0.f;
            float4 res = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
            const long long off = (row * a.Hq + h) * (long long)D + c;
            if (gated) {
                const float gh = a.g[h], gq = 1.0f - gh;
                const uint2 lw = *reinterpret_cast<const uint2 *>(a.lin + off);
                res.x = fmaf(gh, res.x, gq * bf16lo(lw.x));
                res.y = fmaf(gh, res.y, gq * bf16hi(lw.x));
                res.z = fmaf(gh, res.z, gq * bf16lo(lw.y));
                res.w = fmaf(gh, res.w, gq * bf16hi(lw.y));
            }
            *reinterpret_cast<float4 *>(a.out + off) = res;
            if (a.lse && c == 0) a.lse[row * a.Hq + h] = l > 0.f ? (m + log2f(l)) * 0.69314718055994531f : -INFINITY;
        }
    }
}

template <int DI, int D>
__global__ void __launch_bounds__(kThreads, 1) split_select_kernel(SelArgs a) {
    constexpr int W = DI / 4;               // int32 words per indexer vector
    constexpr int TPK = DI / 16;            // lanes per key group, 16 bytes of a key each
    constexpr int NG = kThreads / TPK;      // key groups
    constexpr int SK = kThreads;            // keys per stage: every lane finishes one
    constexpr int SB = SK * DI;             // bytes per stage
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int NS = a.stages;
    unsigned char *ring = smem_raw;
    Smem &sm = *reinterpret_cast<Smem *>(smem_raw + NS * SB);
    int32_t *sc = reinterpret_cast<int32_t *>(smem_raw + NS * SB + kSmemHdr);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const long long row = blockIdx.x / a.chunks;
    const int ci = blockIdx.x % a.chunks;
    const long long b = row / a.Tq, t = (row % a.Tq) / a.pos_div;
    const long long n = a.q_offset + t + 1;
    const int K = a.K;
    const bool whole = n <= K;  // the whole prefix is kept
    const long long len = (n + a.chunks - 1) / a.chunks;
    const long long lo = ci * len;
    const long long hi = min(n, lo + len);
    const int span = whole ? 0 : (int)max(0ll, hi - lo);
    const int nst = (span + SK - 1) / SK;
    const int8_t *ksrc = a.kI + (b * a.Tk + lo) * DI;
    const long long span_bytes = (long long)span * DI;

    // stage s -> ring slot s % NS: one bulk copy (thread 0) of the stage's
    // bytes (the last stage is short; the slot's stale tail is never
    // scored), completing on the slot's barrier; kI is read once
    const uint64_t pol = l2_evict_first_policy();
    auto issue = [&](int s) {
        const int slot = s % NS;
        const long long off0 = (long long)s * SB;
        const unsigned bytes = (unsigned)min((long long)SB, span_bytes - off0);
        const uint32_t fb = smem_u32(&sm.full[slot]);
        mbar_expect_tx(fb, bytes);
        bulk_g2s(smem_u32(ring + slot * SB), ksrc + off0, bytes, fb, pol);
    };

    pdl_wait();
    // small loads first, so that they do not queue behind the stream
    unsigned hd0 = 0, hd1 = 0, hd2 = 0;
    if (tid == 0) {
        hd0 = __ldcg(a.hdr);
        hd1 = __ldcg(a.hdr + 1);
        hd2 = __ldcg(a.hdr + 2);
    }
    const int32_t qword = tid < a.H_I * W ? reinterpret_cast<const int32_t *>(a.qI + row * (long long)a.H_I * DI)[tid] : 0;
    const int32_t wword = tid < a.H_I ? a.wI[tid] : 0;
    if constexpr (D > 0) {
        // the row's query heads, as 16-row m-tiles per key/value head (rows
        // past the G heads of a key/value head are zero); the oldest copy group
        uint16_t *Qs = reinterpret_cast<uint16_t *>(smem_raw + a.off_q);
        const int G = a.Hq / a.Hkv;
        constexpr int CH = D / 8;
        for (int i = tid; i < a.MTT * 16 * CH; i += kThreads) {
            const int rr = i / CH, ch = i % CH, mt = rr >> 4;
            const int hl = (mt % a.MPK) * 16 + (rr & 15);
            const bool valid = hl < G;
            const int head = (mt / a.MPK) * G + (valid ? hl : 0);
            cp_async16_zfill(smem_u32(Qs + rr * (D + 8) + ch * 8), a.q + (row * a.Hq + head) * (long long)D + ch * 8,
                             valid);
        }
        cp_async_commit();
    }
    if (tid == 0) {  // prologue: NS-1 stages in flight
        for (int i = 0; i < NS; i++) mbar_init(smem_u32(&sm.full[i]), 1);
        mbar_fence_init();
        for (int s = 0; s < NS - 1 && s < nst; s++) issue(s);
    }
    for (int i = tid; i < kNB1; i += kThreads) sm.h1[i] = 0u;
    if (tid < a.H_I * W) sm.q[tid] = qword;
    if (tid < a.H_I) sm.w[tid] = wword;
    if (tid == 0) {
        sm.epoch = (int)hd0;
        // rows the previous call of the other parity used; never more than the
        // workspace holds, whatever an earlier use of the buffer left there
        sm.ru_other = (int)min(((hd0 + 1) & 1) ? hd2 : hd1, (unsigned)a.ctrl_cap);
    }
    __syncthreads();
    const int epoch = sm.epoch, par = epoch & 1;
    const unsigned arrived = tid == 0 ? epoch_arrive(a.hdr) : 0u;

    // zero the other parity's control state (the previous call's), spread
    // over the whole grid
    {
        const long long per_row = kRowCtrl / 4;  // 16-byte words
        const long long total = (long long)sm.ru_other * per_row;
        for (long long c = (long long)blockIdx.x * kThreads + tid; c < total; c += (long long)gridDim.x * kThreads) {
            long long r = c / per_row, o = c % per_row;
            reinterpret_cast<uint4 *>(a.ctrl + (2 * r + (par ^ 1)) * kRowCtrl)[o] = make_uint4(0u, 0u, 0u, 0u);
        }
    }

    int32_t *idx_row = a.idx ? a.idx + row * (long long)K : nullptr;
    unsigned *rc = a.ctrl + (2 * row + par) * kRowCtrl;
    unsigned *bar = rc;
    int n_span = 0;  // fused step, whole prefix: the keys of this block's span
    int nbar = 0;    // row barriers passed so far
    bool ok = true;
    if (whole) {
        if (ci == 0 && idx_row) {
            for (long long i = tid; i < K; i += kThreads) idx_row[i] = i < n ? (int32_t)i : -1;
            if (tid == 0) a.cnt[row] = (int32_t)n;
        }
        if (tid == 0) epoch_finish(a.hdr, arrived, epoch, a.rows);
        if constexpr (D == 0) {
            pdl_launch_dependents();
            return;
        }
        n_span = (int)max(0ll, hi - lo);  // every key of the span: positions lo, lo+1, ...
    } else {
    unsigned *g1 = rc + 4;
    unsigned *gl[2] = {g1 + kNB1P, g1 + kNB1P + kNB2};
    unsigned *mypub = a.pub + ((size_t)row * a.chunks + ci) * kPubWords;

    // ---- phase A: stream the span through the stage ring, score, level-1 histogram.
    // Lane j of key group g holds the 16-byte piece j of keys r*NG + g
    // (r = 0..TPK-1: consecutive groups read consecutive keys, conflict-free);
    // a reduce-scatter over the group's lanes leaves lane j with the whole
    // score of key j*NG + g, so every lane finishes one key per stage.
    int mn = INT32_MAX, mx = INT32_MIN;
    {
        const int j = tid % TPK, g = tid / TPK;
        int32_t q0[4];
#pragma unroll
        for (int c = 0; c < 4; c++) q0[c] = sm.q[j * 4 + c];
        const int w0 = sm.w[0];
        const int mykey = j * NG + g;  // this lane's finished key within a stage
        for (int s = 0; s < nst; s++) {
            // stage s has landed (a bounded wait: on time-out the status says
            // so and the stream runs on, every later wait bounded too)
            if (!mbar_wait_bounded(smem_u32(&sm.full[s % NS]), (uint32_t)(s / NS) & 1u, a.wait_ns))
                set_status(a.status, ESA_ERR_TIMEOUT);
            __syncthreads();  // everyone is done with slot (s-1) % NS
            if (tid == 0 && s + NS - 1 < nst) issue(s + NS - 1);
            const unsigned char *buf = ring + (s % NS) * SB;
            unsigned part[TPK];
#pragma unroll
            for (int r = 0; r < TPK; r++) {
                const uint4 v = *reinterpret_cast<const uint4 *>(buf + (r * NG + g) * DI + j * 16);
                int d = __dp4a(q0[0], (int)v.x, 0);
                d = __dp4a(q0[1], (int)v.y, d);
                d = __dp4a(q0[2], (int)v.z, d);
                d = __dp4a(q0[3], (int)v.w, d);
                // with the ReLU (one indexer head) the weight waits for the whole dot product
                unsigned acc = a.relu ? (unsigned)d : (unsigned)w0 * (unsigned)d;
                for (int h = 1; h < a.H_I; h++) {
                    const int32_t *qh = sm.q + h * W + j * 4;
                    int e = __dp4a(qh[0], (int)v.x, 0);
                    e = __dp4a(qh[1], (int)v.y, e);
                    e = __dp4a(qh[2], (int)v.z, e);
                    e = __dp4a(qh[3], (int)v.w, e);
                    acc += (unsigned)sm.w[h] * (unsigned)e;
                }
                part[r] = acc;
            }
            // reduce-scatter: halve the vector each step, keeping the half
            // whose index bit matches this lane's
#pragma unroll
            for (int m = TPK / 2; m >= 1; m >>= 1) {
                const bool up = (j & m) != 0;
#pragma unroll
                for (int i = 0; i < m; i++) {
                    unsigned send = up ? part[i] : part[i + m];
                    unsigned keep = up ? part[i + m] : part[i];
                    part[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
                }
            }
            const int kk = s * SK + mykey;
            if (kk < span) {
                const int sv = a.relu ? (int)((unsigned)w0 * (unsigned)max((int)part[0], 0)) : (int)part[0];
                sc[kk] = sv;
                atomicAdd(&sm.h1[bin1(sv)], 1u);
                mn = min(mn, sv);
                mx = max(mx, sv);
            }
        }
        cp_async_wait<0>();
    }
    // block range of scores -> range of level-1 bins
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
        mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, d));
        mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, d));
    }
    if (lane == 0) {
        sm.mn[warp] = mn;
        sm.mx[warp] = mx;
    }
    __syncthreads();
    for (int w2 = 0; w2 < kWarps; w2++) {
        mn = min(mn, sm.mn[w2]);
        mx = max(mx, sm.mx[w2]);
    }
    const int blo = span > 0 ? bin1(mn) : 1, bhi = span > 0 ? bin1(mx) : 0;
    for (int i = blo + tid; i <= bhi; i += kThreads)
        if (sm.h1[i]) atomicAdd(g1 + i, sm.h1[i]);
    if (span > 0) publish_suffix(sm.h1, blo, bhi, mypub + 4, kWinLo, kWinLo + kWin - 1, sm);
    if (tid == 0) {
        mypub[0] = (unsigned)blo;
        mypub[1] = (unsigned)bhi;
        mypub[2] = (unsigned)span;
    }
    // ---- the row's barrier (and this block's arrival in the call)
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        red_release_add_u32(bar, 1u);
        bool ok1 = bounded_wait_geq(bar, (unsigned)a.chunks + a.extra, a.wait_ns);
        if (!ok1) set_status(a.status, ESA_ERR_TIMEOUT);
        sm.flag = ok1 ? 0 : 1;
        epoch_finish(a.hdr, arrived, epoch, a.rows);
    }
    __syncthreads();
    ok = sm.flag == 0;
    nbar = 1;
    pdl_launch_dependents();

    // ---- the threshold: exact from level 1, else refined
    // the ring is idle now: it stages deeper-level histograms and holds their bins
    unsigned *stage = reinterpret_cast<unsigned *>(ring);
    unsigned *h2 = stage + kNB2;
    int T = 0;
    unsigned above = 0, gt_b = 0, eq_b = 0;
    PendingPub pend{false, 0, 0, -1, 0u, 0u, 0u};
    if (ok) {
        find_crossing(g1, (unsigned)K, sm);
        if (sm.bin < 0) {
            if (tid == 0) set_status(a.status, ESA_ERR_INTERNAL);
            ok = false;
        }
    }
    if (ok) {
        const int vstar = sm.bin;
        above = sm.above;
        long long vlo, vhi;
        bin1_range(vstar, vlo, vhi);
        if (vlo == vhi) {
            // exact at level 1: earlier spans' counts above T and at T from
            // their published suffix counts (S(v) = #{bin >= v})
            T = (int)vlo;
            const int x = vstar - kWinLo;  // in [0, kWin-1)
            {
                // issued now, read only after this block's own counts (phase
                // C) or its keys above T and their gathers (the fused step)
                if (tid < ci) {
                    const unsigned *pq = a.pub + ((size_t)row * a.chunks + tid) * kPubWords;
                    pend.have = true;
                    pend.vstar = vstar;
                    pend.clo = (int)__ldcg(pq);
                    pend.chi = (int)__ldcg(pq + 1);
                    pend.tot = __ldcg(pq + 2);
                    pend.s0 = __ldcg(pq + 4 + x);
                    pend.s1 = __ldcg(pq + 5 + x);
                }
            }
        } else {
            // refine inside the crossing bucket: 4096 bins per level, a
            // barrier each, until the bucket is one value
            int shift = 1;
            for (int level = 2; level <= 3 && ok; level++) {
                long long Wd = vhi - vlo + 1;
                shift = 0;
                while (((Wd - 1) >> shift) >= kNB2) shift++;
                const int nb = (int)(((Wd - 1) >> shift) + 1);
                for (int i = tid; i < nb; i += kThreads) h2[i] = 0u;
                __syncthreads();
                unsigned mine_above = 0;
                for (int j = tid; j < span; j += kThreads) {
                    long long s = sc[j];
                    if (s >= vlo && s <= vhi) atomicAdd(&h2[(int)((s - vlo) >> shift)], 1u);
                    mine_above += (s > vhi);
                }
                __syncthreads();
                unsigned *gdst = gl[level - 2];
                for (int i = tid; i < nb; i += kThreads)
                    if (h2[i]) atomicAdd(gdst + i, h2[i]);
                if (shift == 0) {
                    // publish: [0] count above the bucket, [1+v] = #scores >=
                    // vlo+v within the bucket, [1+nb] = 0
                    unsigned *dp = mypub + kPubDeep;
#pragma unroll
                    for (int d = 16; d > 0; d >>= 1) mine_above += __shfl_xor_sync(0xffffffffu, mine_above, d);
                    if (lane == 0) sm.red[warp] = mine_above;
                    publish_suffix(h2, 0, nb - 1, dp + 1, 0, nb - 1, sm);
                    __syncthreads();
                    if (tid == 0) {
                        unsigned tot = 0;
                        for (int w2 = 0; w2 < kWarps; w2++) tot += sm.red[w2];
                        dp[0] = tot;
                        dp[1 + nb] = 0u;
                    }
                }
                ok = group_barrier(bar, (unsigned)(level * a.chunks + a.extra), a.wait_ns, a.status, &sm.flag);
                nbar = level;
                if (!ok) break;
                find_crossing_staged(gdst, nb, (unsigned)K - above, stage, sm);
                if (sm.bin < 0) {
                    if (tid == 0) set_status(a.status, ESA_ERR_INTERNAL);
                    ok = false;
                    break;
                }
                above += sm.above;
                if (shift == 0) {
                    T = (int)(vlo + sm.bin);
                    const int vb = sm.bin;
                    for (int c = tid; c < ci; c += kThreads) {
                        const unsigned *pp = a.pub + ((size_t)row * a.chunks + c) * kPubWords + kPubDeep;
                        unsigned ge = __ldcg(pp + 1 + vb), gt = __ldcg(pp + 2 + vb);
                        gt_b += __ldcg(pp) + gt;
                        eq_b += ge - gt;
                    }
                    break;
                }
                vlo = vlo + ((long long)sm.bin << shift);
                vhi = min(vhi, vlo + (1ll << shift) - 1);
            }
            if (ok && shift != 0) {  // cannot happen: three levels always resolve an int32 score
                if (tid == 0) set_status(a.status, ESA_ERR_INTERNAL);
                ok = false;
            }
        }
    }

    // ---- phase C: ordered write of this span's selected positions (the
    // fused step lists its keys and writes idx in its own tail instead).
    // Each thread holds 16 consecutive scores in registers; one block-wide
    // scan of (keys above T, keys at T) gives every thread its output slot:
    // above T always, at T while the row's first K - #(above T) ties (in
    // position order) are not all taken.
    if (D == 0 && ok) {
        const unsigned need_ties = (unsigned)K - above;  // ties at T to take, >= 1
        // earlier spans' counts above T and at T (loads issued before)
        unsigned gtp = gt_b, eqp = eq_b;
        unsigned carry_gt = 0, carry_eq = 0;  // keys of earlier rounds of this span
        unsigned gt_before = 0, eq_before = 0;
        const int nchunk = (span + 15) / 16;
        for (int c0 = 0; c0 < nchunk; c0 += kThreads) {
            const int c = c0 + tid, j0 = c * 16;
            int v[16];
            if (c < nchunk) {
                const int4 *p4 = reinterpret_cast<const int4 *>(sc + j0);
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    const int4 w4 = p4[q];
                    v[4 * q] = w4.x;
                    v[4 * q + 1] = w4.y;
                    v[4 * q + 2] = w4.z;
                    v[4 * q + 3] = w4.w;
                }
            }
            unsigned ng = 0, ne = 0;
#pragma unroll
            for (int i = 0; i < 16; i++) {
                if (c >= nchunk || j0 + i >= span) v[i] = INT32_MIN;  // past the span: never taken
                ng += v[i] > T;
                ne += v[i] == T;
            }
            // inclusive scan of (ng, ne) over the warp, then over the warps
            unsigned ig = ng, ie = ne;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const unsigned ug = __shfl_up_sync(0xffffffffu, ig, d), ue = __shfl_up_sync(0xffffffffu, ie, d);
                if (lane >= d) {
                    ig += ug;
                    ie += ue;
                }
            }
            if (c0 == 0 && pend.have) {  // the earlier spans' counts, now that their loads have landed
                const unsigned S0 = pend.vstar <= pend.clo ? pend.tot : (pend.vstar > pend.chi ? 0u : pend.s0);
                const unsigned S1 =
                    pend.vstar + 1 <= pend.clo ? pend.tot : (pend.vstar + 1 > pend.chi ? 0u : pend.s1);
                gtp += S1;
                eqp += S0 - S1;
            }
            if (c0 == 0) {
#pragma unroll
                for (int d = 16; d > 0; d >>= 1) {
                    gtp += __shfl_xor_sync(0xffffffffu, gtp, d);
                    eqp += __shfl_xor_sync(0xffffffffu, eqp, d);
                }
            }
            __syncthreads();  // sm.red / sm.wsum free (the previous round's readers are done)
            if (lane == 31) {
                sm.wsum[0][warp] = ig;
                sm.wsum[1][warp] = ie;
            }
            if (c0 == 0 && lane == 0) {
                sm.red[warp] = gtp;
                sm.red[32 + warp] = eqp;
            }
            __syncthreads();
            // every warp scans the warp totals (lanes < kWarps) alike
            const unsigned wg = lane < kWarps ? sm.wsum[0][lane] : 0u, we = lane < kWarps ? sm.wsum[1][lane] : 0u;
            unsigned sg = wg, se = we;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const unsigned ug = __shfl_up_sync(0xffffffffu, sg, d), ue = __shfl_up_sync(0xffffffffu, se, d);
                if (lane >= d) {
                    sg += ug;
                    se += ue;
                }
            }
            if (c0 == 0) {
                unsigned rg = lane < kWarps ? sm.red[lane] : 0u, re = lane < kWarps ? sm.red[32 + lane] : 0u;
#pragma unroll
                for (int d = 16; d > 0; d >>= 1) {
                    rg += __shfl_xor_sync(0xffffffffu, rg, d);
                    re += __shfl_xor_sync(0xffffffffu, re, d);
                }
                gt_before = rg;
                eq_before = re;
            }
            const unsigned tot_g = __shfl_sync(0xffffffffu, sg, 31), tot_e = __shfl_sync(0xffffffffu, se, 31);
            const unsigned pre_g = carry_gt + __shfl_sync(0xffffffffu, sg - wg, warp) + (ig - ng);
            const unsigned pre_e = carry_eq + __shfl_sync(0xffffffffu, se - we, warp) + (ie - ne);
            // ties at T taken before this thread's keys, and by them
            const unsigned tie0 = eq_before + pre_e;
            const unsigned take_before = min(tie0, need_ties) - min(eq_before, need_ties);
            unsigned tk = tie0 >= need_ties ? 0u : min(ne, need_ties - tie0);
            unsigned out = gt_before + min(eq_before, need_ties) + pre_g + take_before;
            if (ng + tk > 0) {
#pragma unroll
                for (int i = 0; i < 16; i++) {
                    const bool take = v[i] > T || (v[i] == T && tk > 0);
                    if (v[i] == T && tk > 0) tk--;
                    if (take) {
                        if (out < (unsigned)K) idx_row[out] = (int32_t)(lo + j0 + i);
                        else set_status(a.status, ESA_ERR_INTERNAL);
                        out++;
                    }
                }
            }
            carry_gt += tot_g;
            carry_eq += tot_e;
        }
        if (ci == 0 && tid == 0) a.cnt[row] = K;
    }
    if constexpr (D > 0) {
        if (ok)
            fused_tail<D>(a, smem_raw, ring, sc, sm, row, b, ci, lo, span, false, 0, T, above, gt_b, eq_b, pend,
                          bar, nbar);
    }
    }  // !whole
    if constexpr (D > 0) {
        if (whole) {
            const PendingPub none{false, 0, 0, -1, 0u, 0u, 0u};
            fused_tail<D>(a, smem_raw, ring, sc, sm, row, b, ci, lo, 0, true, n_span, 0, 0u, 0u, 0u, none, bar, 0);
        }
    }
}

void *kernel_ptr(int DI) {
    switch (DI) {
        case 16: return (void *)split_select_kernel<16, 0>;
        case 32: return (void *)split_select_kernel<32, 0>;
        case 64: return (void *)split_select_kernel<64, 0>;
        default: return (void *)split_select_kernel<128, 0>;
    }
}

// The fused decode step: selection, attention and gate mix in one launch.
void *fused_kernel_ptr(int DI, int D) {
    if (D == 64) {
        switch (DI) {
            case 16: return (void *)split_select_kernel<16, 64>;
            case 32: return (void *)split_select_kernel<32, 64>;
            case 64: return (void *)split_select_kernel<64, 64>;
            default: return (void *)split_select_kernel<128, 64>;
        }
    }
    switch (DI) {
        case 16: return (void *)split_select_kernel<16, 128>;
        case 32: return (void *)split_select_kernel<32, 128>;
        case 64: return (void *)split_select_kernel<64, 128>;
        default: return (void *)split_select_kernel<128, 128>;
    }
}

size_t scores_bytes(long long len) { return (size_t)((len + 31) / 32 * 32) * sizeof(int32_t); }

size_t stage_bytes(int DI) { return (size_t)kThreads * DI; }

// Ring depth for a span of `len` keys: kRingBytes in flight when the shared
// memory budget allows, at least kMinStages and enough room for the deeper
// levels' bins and for `min_ring` bytes of later use (0 if that does not
// fit); `extra` bytes of shared memory follow the scores.
int stages_for(long long len, int DI, size_t extra = 0, size_t min_ring = 0) {
    size_t fixed = kSmemHdr + scores_bytes(len) + extra;
    if (fixed >= kSmemBudget) return 0;
    size_t sb = stage_bytes(DI);
    size_t want = std::max<size_t>(std::max<size_t>(kRingBytes / sb, kMinStages), (min_ring + sb - 1) / sb);
    int st = (int)std::min<size_t>(std::min<size_t>(want, (kSmemBudget - fixed) / sb), kMaxStages);
    if (st < kMinStages || (size_t)st * sb < 2 * (size_t)kNB2 * 4 || (size_t)st * sb < min_ring) return 0;
    return st;
}

size_t smem_for(long long len, int DI, int stages, size_t extra = 0) {
    return (size_t)stages * stage_bytes(DI) + kSmemHdr + scores_bytes(len) + extra;
}

}  // namespace

SplitPlan plan_split_select(const Shape &s, int K) {
    SplitPlan p{};
    p.ok = false;
    long long rows = s.B * s.Tq;
    if (rows <= 0) return p;
    long long nmax = s.q_offset + (s.Tq + s.pos_div - 1) / s.pos_div;  // longest prefix
    // the lane groups sum partial dot products after weighting: a ReLU on
    // each of several heads' whole dot products is left to the row kernels
    if (relu_of(s) && s.H_I > 1) return p;
    DevInfo di = device_info();
    void *fn = kernel_ptr(s.D_I);
    // one block per SM (the launch reserves more than half an SM's shared memory)
    int per_sm = occupancy(fn, kThreads, smem_for(kMaxChunk, s.D_I, stages_for(kMaxChunk, s.D_I)));
    if (per_sm < 1) return p;
    long long resident = (long long)di.sms * per_sm;
    if (rows > resident / 2) return p;  // each row should get >= 2 blocks
    int chunks = (int)(resident / rows);
    long long len = (nmax + chunks - 1) / chunks;
    if (len > kMaxChunk) return p;
    p.ok = true;
    p.chunks = chunks;
    p.grid = (int)(rows * chunks);
    p.stages = stages_for(len, s.D_I);
    if (p.stages == 0) {
        p.ok = false;
        return p;
    }
    p.smem = std::max(smem_for(len, s.D_I, p.stages), (size_t)117 * 1024);
    // workspace: [status][header][publications: one slot per resident block]
    // [control: two parities per row]
    p.hdr_off = kStatusBytes;
    p.pub_off = p.hdr_off + kHdrBytes;
    p.ctrl_off = p.pub_off + align256((size_t)resident * kPubWords * 4);
    p.ctrl_bytes = (size_t)rows * 2 * kRowCtrl * 4;
    p.ctrl_rows_max = (int)(resident / 2);
    p.ws_bytes = p.ctrl_off + p.ctrl_bytes;
    return p;
}

size_t split_state_max_bytes() {
    DevInfo di = device_info();
    const int per_sm = occupancy(kernel_ptr(64), kThreads, smem_for(kMaxChunk, 64, stages_for(kMaxChunk, 64)));
    const size_t resident = (size_t)di.sms * (per_sm > 0 ? per_sm : 1);
    return kStatusBytes + kHdrBytes + align256(resident * kPubWords * 4) + resident / 2 * 2 * kRowCtrl * 4;
}

esa_status launch_split_select(const int8_t *qI, const int8_t *kI, const int32_t *wI, const Shape &s, int K,
                               int32_t *idx, int32_t *cnt, void *ws, size_t ws_bytes, const SplitPlan &plan,
                               cudaStream_t st) {
    char *base = static_cast<char *>(ws);
    SelArgs a{};
    a.qI = qI;
    a.kI = kI;
    a.wI = wI;
    a.idx = idx;
    a.cnt = cnt;
    a.status = reinterpret_cast<int32_t *>(base);
    a.hdr = reinterpret_cast<unsigned *>(base + plan.hdr_off);
    a.pub = reinterpret_cast<unsigned *>(base + plan.pub_off);
    a.ctrl = reinterpret_cast<unsigned *>(base + plan.ctrl_off);
    a.Tq = s.Tq;
    a.Tk = s.Tk;
    a.q_offset = s.q_offset;
    a.wait_ns = wait_limit_ns();
    a.pos_div = s.pos_div;
    a.relu = relu_of(s) ? 1 : 0;
    a.H_I = s.H_I;
    a.K = K;
    a.chunks = plan.chunks;
    a.rows = (int)(s.B * s.Tq);
    a.extra = debug_extra_arrivals();
    a.stages = plan.stages;
    a.ctrl_cap = (int)std::min<size_t>((size_t)plan.ctrl_rows_max,
                                       ws_bytes > plan.ctrl_off ? (ws_bytes - plan.ctrl_off) / (2 * kRowCtrl * 4) : 0);
    void *fn = kernel_ptr(s.D_I);
    if (!ensure_smem(fn, plan.smem)) return ESA_ERR_CUDA;
    void *args[] = {(void *)&a};
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(plan.grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = plan.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
    return e == cudaSuccess ? ESA_OK : ESA_ERR_CUDA;
}

DecodePlan plan_decode_step(const Shape &s, int K) {
    DecodePlan p{};
    p.ok = false;
    if (per_head_of(s) || s.pos_div != 1) return p;  // one index set per row
    if (s.D != 64 && s.D != 128) return p;
    const int G = s.Hq / s.Hkv, MPK = (G + 15) / 16, MTT = s.Hkv * MPK;
    if (MTT > 8) return p;  // at most 8 m-tiles of 16 query heads
    int KG = std::min(8, 16 / MTT);
    while (KG > 1 && 8 * KG * s.Hkv > 64) KG /= 2;  // at most 64 K (and V) rows per stage
    SplitPlan sp = plan_split_select(s, K);
    if (!sp.ok) return p;
    const long long nmax = s.q_offset + s.Tq;
    const long long len = (nmax + sp.chunks - 1) / sp.chunks;
    const int sel_cap = (int)std::min<long long>(K, len);
    const size_t RS = (size_t)s.D + 8;
    const size_t q_bytes = align_up((size_t)MTT * 16 * RS * 2);
    const size_t sel_bytes = align_up((size_t)sel_cap * 4);
    const size_t aux_bytes = align_up((size_t)2 * kWarps * 16 * 4);
    const size_t extra = q_bytes + sel_bytes + aux_bytes + 128;  // + the Q tile's alignment
    const size_t stage2 = (size_t)2 * 2 * (8 * KG) * s.Hkv * RS * 2;  // two stages of K and V rows
    const size_t tree = (size_t)std::max(1, KG / 2) * MTT * 16 * (s.D + 8) * 4;  // pairwise merge buffer
    const size_t min_ring = std::max(stage2, tree);
    const int stages = stages_for(len, s.D_I, extra, min_ring);
    if (stages == 0) return p;
    // the Q tile (cp.async and ldmatrix rows) starts on a 128-byte boundary
    const size_t base = ((size_t)stages * stage_bytes(s.D_I) + kSmemHdr + scores_bytes(len) + 127) & ~size_t(127);
    void *fn = fused_kernel_ptr(s.D_I, s.D);
    const size_t smem = base + q_bytes + sel_bytes + aux_bytes;
    if (occupancy(fn, kThreads, smem) < 1) return p;
    p.sel = sp;
    p.sel.stages = stages;
    p.sel.smem = smem;
    p.MPK = MPK;
    p.MTT = MTT;
    p.KG = KG;
    p.sel_cap = sel_cap;
    p.off_q = base;
    p.off_sel = base + q_bytes;
    p.off_aux = base + q_bytes + sel_bytes;
    const size_t slots = (size_t)s.B * s.Tq * sp.chunks * s.Hq;
    // the partials lie past the control state of the most rows any shape's
    // selection uses, so calls of other shapes sharing the workspace keep
    // their control state
    p.part_off = align256(std::max(sp.ws_bytes, split_state_max_bytes()));
    p.ml_off = p.part_off + align256(slots * s.D * 4);
    p.ws_bytes = p.ml_off + align256(slots * 8);
    p.ok = true;
    return p;
}

esa_status launch_decode_step(const uint16_t *q, const uint16_t *k, const uint16_t *v, const int8_t *qI,
                              const int8_t *kI, const int32_t *wI, const Shape &s, int K, float scale, const float *g,
                              const uint16_t *lin, float *out, float *lse, int32_t *idx, int32_t *cnt, void *ws,
                              const DecodePlan &plan, cudaStream_t st) {
    const SplitPlan &sp = plan.sel;
    char *base = static_cast<char *>(ws);
    SelArgs a{};
    a.qI = qI;
    a.kI = kI;
    a.wI = wI;
    a.idx = idx;
    a.cnt = cnt;
    a.status = reinterpret_cast<int32_t *>(base);
    a.hdr = reinterpret_cast<unsigned *>(base + sp.hdr_off);
    a.pub = reinterpret_cast<unsigned *>(base + sp.pub_off);
    a.ctrl = reinterpret_cast<unsigned *>(base + sp.ctrl_off);
    a.Tq = s.Tq;
    a.Tk = s.Tk;
    a.q_offset = s.q_offset;
    a.wait_ns = wait_limit_ns();
    a.pos_div = 1;
    a.relu = relu_of(s) ? 1 : 0;
    a.H_I = s.H_I;
    a.K = K;
    a.chunks = sp.chunks;
    a.rows = (int)(s.B * s.Tq);
    a.extra = debug_extra_arrivals();
    a.stages = sp.stages;
    a.ctrl_cap = sp.ctrl_rows_max;
    a.q = q;
    a.k = k;
    a.v = v;
    a.lin = lin;
    a.g = g;
    a.out = out;
    a.lse = lse;
    a.part = reinterpret_cast<float *>(base + plan.part_off);
    a.ml = reinterpret_cast<float2 *>(base + plan.ml_off);
    a.Hq = s.Hq;
    a.Hkv = s.Hkv;
    a.MPK = plan.MPK;
    a.MTT = plan.MTT;
    a.KG = plan.KG;
    a.sel_cap = plan.sel_cap;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.off_q = (int)plan.off_q;
    a.off_sel = (int)plan.off_sel;
    a.off_aux = (int)plan.off_aux;
    void *fn = fused_kernel_ptr(s.D_I, s.D);
    if (!ensure_smem(fn, sp.smem)) return ESA_ERR_CUDA;
    void *args[] = {(void *)&a};
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(sp.grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = sp.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
    return e == cudaSuccess ? ESA_OK : ESA_ERR_CUDA;
}

}  // namespace esa
