// Top-K selection for few query rows with long prefixes (decode).
//
// Method: the Indexer scores the query against every causal-prefix position
// and the K best positions are kept ("超大规模MoE架构中稀疏注意力机制的演进与实践",
// section 二.1, K = 2048; no RoPE, section 二.2). Ties go to the lower position.
//
// Design (one launch, one co-resident block per SM):
//   * each query row's prefix 0..p is cut into `chunks` contiguous spans,
//     one block per span; the block streams its span of kI once from HBM
//     through a ring of shared-memory stages filled by per-thread 16-byte
//     cp.async copies (128 KB in flight per SM, which a one-block-per-SM
//     stream needs to approach HBM bandwidth; one-dimensional bulk copies
//     measured well below it), scores each key with dp4a and keeps the int32
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
};

struct Smem {
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

template <int DI>
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
    int32_t *sc = reinterpret_cast<int32_t *>(smem_raw + NS * SB + sizeof(Smem));

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

    // stage s -> ring slot s % NS; each thread copies 16-byte pieces
    // tid, tid + kThreads, ... of the stage (zero-filled past the span)
    auto issue = [&](int s) {
        const uint32_t dst = smem_u32(ring + (s % NS) * SB);
        const long long off0 = (long long)s * SB;
#pragma unroll
        for (int c = tid * 16; c < SB; c += kThreads * 16) {
            const bool ok = off0 + c < span_bytes;
            cp_async16_zfill(dst + c, ksrc + (ok ? off0 + c : 0), ok);
        }
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
    for (int s = 0; s < NS - 1; s++) {  // prologue: NS-1 stages in flight
        if (s < nst) issue(s);
        cp_async_commit();
    }
    for (int i = tid; i < kNB1; i += kThreads) sm.h1[i] = 0u;
    if (tid < a.H_I * W) sm.q[tid] = qword;
    if (tid < a.H_I) sm.w[tid] = wword;
    if (tid == 0) {
        sm.epoch = (int)hd0;
        sm.ru_other = (int)(((hd0 + 1) & 1) ? hd2 : hd1);
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

    int32_t *idx_row = a.idx + row * (long long)K;
    if (whole) {
        if (ci == 0) {
            for (long long i = tid; i < K; i += kThreads) idx_row[i] = i < n ? (int32_t)i : -1;
            if (tid == 0) a.cnt[row] = (int32_t)n;
        }
        if (tid == 0) epoch_finish(a.hdr, arrived, epoch, a.rows);
        pdl_launch_dependents();
        return;
    }

    unsigned *rc = a.ctrl + (2 * row + par) * kRowCtrl;
    unsigned *bar = rc;
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
            cp_async_wait_dyn(NS - 2);  // this thread's copies of stage s have landed
            __syncthreads();            // ... and everyone's; slot (s-1) % NS is free
            if (s + NS - 1 < nst) issue(s + NS - 1);
            cp_async_commit();
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
    bool ok = sm.flag == 0;
    pdl_launch_dependents();

    // ---- the threshold: exact from level 1, else refined
    // the ring is idle now: it stages deeper-level histograms and holds their bins
    unsigned *stage = reinterpret_cast<unsigned *>(ring);
    unsigned *h2 = stage + kNB2;
    int T = 0;
    unsigned above = 0, gt_b = 0, eq_b = 0;
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
            for (int c = tid; c < ci; c += kThreads) {
                const unsigned *pp = a.pub + ((size_t)row * a.chunks + c) * kPubWords;
                const int clo = (int)__ldcg(pp), chi = (int)__ldcg(pp + 1);
                const unsigned ctot = __ldcg(pp + 2);
                const unsigned s0 = __ldcg(pp + 4 + x), s1 = __ldcg(pp + 5 + x);
                const unsigned S0 = vstar <= clo ? ctot : (vstar > chi ? 0u : s0);
                const unsigned S1 = vstar + 1 <= clo ? ctot : (vstar + 1 > chi ? 0u : s1);
                gt_b += S1;
                eq_b += S0 - S1;
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

    // ---- phase C: ordered write of this span's selected positions
    if (ok) {
        const unsigned need_ties = (unsigned)K - above;  // ties at T to take, >= 1
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) {
            gt_b += __shfl_xor_sync(0xffffffffu, gt_b, d);
            eq_b += __shfl_xor_sync(0xffffffffu, eq_b, d);
        }
        __syncthreads();
        if (lane == 0) {
            sm.red[warp] = gt_b;
            sm.red[32 + warp] = eq_b;
        }
        // per-warp counts over contiguous segments of the span. Almost every
        // 32-key chunk lies wholly below T: one ballot on s >= T skips it.
        const int seg = ((span + kWarps * 32 - 1) / (kWarps * 32)) * 32;
        const int s0 = warp * seg, s1 = min(span, s0 + seg);
        unsigned wgt = 0, weq = 0;
#pragma unroll 4
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
        unsigned gt_before = 0, eq_before = 0;
        for (int w2 = 0; w2 < kWarps; w2++) {
            gt_before += sm.red[w2];
            eq_before += sm.red[32 + w2];
        }
        // output base of this span and of this warp's segment
        unsigned out = gt_before + min(eq_before, need_ties);
        unsigned tie = eq_before;
        for (int w2 = 0; w2 < warp; w2++) {
            unsigned e = sm.wsum[1][w2];
            unsigned take = tie >= need_ties ? 0u : min(e, need_ties - tie);
            out += sm.wsum[0][w2] + take;
            tie += e;
        }
        // ordered write: same chunks, same skip
        const unsigned lt = lanemask_lt();
        if (wgt + weq > 0u) {
#pragma unroll 4
            for (int j0 = s0; j0 < s1; j0 += 32) {
                const int j = j0 + lane;
                const int sv = j < s1 ? sc[j] : INT32_MIN;
                const unsigned gem = __ballot_sync(0xffffffffu, sv >= T);
                if (gem == 0u) continue;
                const unsigned eqm = __ballot_sync(0xffffffffu, sv == T);
                const unsigned gtm = gem & ~eqm;
                // ties taken in this chunk: its first min(#ties, need - taken so far)
                const unsigned ne = __popc(eqm);
                const unsigned take = tie >= need_ties ? 0u : min(ne, need_ties - tie);
                unsigned tmask = 0u;
                if (take == ne) {
                    tmask = eqm;
                } else if (take > 0u) {  // the lowest `take` ties (warp-uniform branch)
                    tmask = __ballot_sync(0xffffffffu, ((eqm >> lane) & 1u) && __popc(eqm & lt) < take);
                }
                const unsigned selm = gtm | tmask;
                if ((selm >> lane) & 1u) {
                    const unsigned pos = out + __popc(selm & lt);
                    if (pos < (unsigned)K) idx_row[pos] = (int32_t)(lo + j);
                    else set_status(a.status, ESA_ERR_INTERNAL);
                }
                out += __popc(selm);
                tie += ne;
            }
        }
        if (ci == 0 && tid == 0) a.cnt[row] = K;
    }
}

void *kernel_ptr(int DI) {
    switch (DI) {
        case 16: return (void *)split_select_kernel<16>;
        case 32: return (void *)split_select_kernel<32>;
        case 64: return (void *)split_select_kernel<64>;
        default: return (void *)split_select_kernel<128>;
    }
}

size_t scores_bytes(long long len) { return (size_t)((len + 31) / 32 * 32) * sizeof(int32_t); }

size_t stage_bytes(int DI) { return (size_t)kThreads * DI; }

// Ring depth for a span of `len` keys: kRingBytes in flight when the shared
// memory budget allows, at least kMinStages and enough room for the deeper
// levels' bins (0 if that does not fit).
int stages_for(long long len, int DI) {
    size_t fixed = sizeof(Smem) + scores_bytes(len);
    if (fixed >= kSmemBudget) return 0;
    size_t sb = stage_bytes(DI);
    int st = (int)std::min<size_t>(std::max<size_t>(kRingBytes / sb, kMinStages), (kSmemBudget - fixed) / sb);
    if (st < kMinStages || (size_t)st * sb < 2 * (size_t)kNB2 * 4) return 0;
    return st;
}

size_t smem_for(long long len, int DI, int stages) {
    return (size_t)stages * stage_bytes(DI) + sizeof(Smem) + scores_bytes(len);
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
    p.ws_bytes = p.ctrl_off + p.ctrl_bytes;
    return p;
}

esa_status launch_split_select(const int8_t *qI, const int8_t *kI, const int32_t *wI, const Shape &s, int K,
                               int32_t *idx, int32_t *cnt, void *ws, const SplitPlan &plan, cudaStream_t st) {
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

}  // namespace esa
