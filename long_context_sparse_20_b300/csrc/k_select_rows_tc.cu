// Top-K selection for many query rows on the tensor cores (prefill, chunked
// prefill, and the thresholds that the routed kernel rebuilds its masks from).
//
// Method: per query row, the Indexer score against every causal-prefix key
// (no RoPE) and the K best positions, ties to the lower position
// ("超大规模MoE架构中稀疏注意力机制的演进与实践", sections 二.1-二.2), computed
// blockwise over the queries without materialising the score matrix
// ("大模型推理架构演进：从稀疏注意力到隐式专家路由", section 2.3).
//
// Design. The scores of 128 query rows against a tile of 128 keys are one
// M=128 N=128 K=D_I matrix product. The indexer heads collapse into
// q_eff = sum_h w_h qI_h (integer algebra, since every indexer head scores
// the same key vector); q_eff and kI are held as fp16, which represents them
// exactly while |q_eff| <= 2048, and the fp32 accumulator of tcgen05.mma then
// holds every partial sum exactly while sum_c |q_eff[c]| * 128 < 2^24: the
// scores leave tensor memory as exact integers. A query tile that fails that
// test is flagged and left to the dp4a kernel (k_select_rows.cu), which a
// second launch runs on the flagged tiles only.
//
// Roles in one CTA (576 threads; one sequence, 128 query rows):
//   warps 0-15 read scores from tensor memory, four warps per 32-row quarter
//              (warp w takes key columns 32*(w/4) .. +31 of every tile)
//   warp 16    bulk-copies fp16 key tiles (converted once per call by
//              kh_convert_kernel into the tensor cores' core-matrix layout,
//              so that a tile is one contiguous 16-KiB block) into a ring
//   warp 17    one thread issues the MMAs into four 128-column buffers
// Passes over the keys; the scores are recomputed by every pass:
//   sample (query tiles whose prefixes span 48 key tiles or more) a log
//          histogram (4 classes per octave) of every 4th, 8th or 16th key
//          tile (prefixes of 48, 128, 256 key tiles and more);
//          it brackets each row's K-th largest score: the scores between
//          the sample's (r - d)-th and (r + d)-th largest, r = K m / n the
//          K-th score's expected rank among the m sampled of n keys and
//          d = 4 sqrt(r) + 8; a second pass over the same tiles bins the
//          sample inside that log-bin bracket (512 bins) and narrows its
//          edges to those two ranks;
//   bracket every key: counted above the bracket, counted below it, or
//          binned inside it (512 16-bit bins); the counts verify the bracket
//          (fewer than K keys above it, at least K above its floor, the
//          bins summing to the keys inside) and a row whose bracket misses
//          falls back to the passes below;
//   1      (without a sample, or on fallback) a log histogram per row;
//          keys below a running lower bound on the row's K-th largest score
//          are not counted, so most keys cost one comparison;
//   2 ..   256 bins over the bucket that holds the K-th score, until the
//          threshold T is exact (one pass while that bucket spans at most
//          256 integers);
//   final  selected = s > T, or s == T among the first K - #{s > T} ties in
//          position order, written in ascending order; also the threshold
//          form (T, P), P the position of the last tie taken, and on request
//          the selected keys as a bitmask (one word per 32 keys and row,
//          word-major), which the routed kernel masks sparse heads with.
#include <stdlib.h>
#include <string.h>

#include "esa_device.cuh"
#include "esa_internal.h"
#include "tc_util.cuh"

namespace esa {

namespace {

constexpr int kRowsT = 128;   // query rows per CTA (TMEM lanes)
constexpr int kKT = 128;      // keys per tile (MMA N)
constexpr int kTBufs = 4;     // TMEM score buffers of kKT columns
constexpr int kParts = 4;               // threads per query row (each reads 32 key columns)
constexpr int kCols = kKT / kParts;     // key columns per thread and tile
constexpr int kCons = kRowsT * kParts;  // score-reading threads (16 warps)
constexpr int kConsWarps = kCons / 32;
constexpr int kProdWarp = kConsWarps, kMmaWarp = kConsWarps + 1;
constexpr int kThreadsTc = kCons + 64;
constexpr int kNB = 256;      // histogram bins per row
constexpr int kHS = kNB + 1;  // row stride of the histograms (words)
constexpr int kLog0 = 100;    // level-1 bin of the score 0
constexpr int kRing = 65536;  // bytes of key-tile ring
constexpr int kMaxStages = 8;
constexpr int kMaxLevels = 8;
constexpr int kSampleMinTiles = 48;  // sample only prefixes of at least this many key tiles

enum { kModeStart = -1, kModeHist = 0, kModeFinal = 1, kModeDone = 2, kModeSample = 3 };
// what a row's histogram pass does
enum { kKindLog = 0, kKindBucket = 1, kKindBracket = 2 };

template <int DI>
struct TcLay {
    static constexpr int KT_BYTES = kKT * DI * 2;
    static constexpr int STAGES = kRing / KT_BYTES < kMaxStages ? kRing / KT_BYTES : kMaxStages;
    static constexpr int RING = 0;
    static constexpr int QE = RING + STAGES * KT_BYTES;
    static constexpr int HIST = QE + kRowsT * DI * 2;
    static constexpr int TOTAL = HIST + kRowsT * kHS * 4;
};

struct TcShared {
    unsigned long long full[kMaxStages], sfree[kMaxStages], tfull[kTBufs], tfree[kTBufs], mma_end;
    int n[kRowsT];      // prefix length of the row (0 past the last row)
    int lo[kRowsT], hi[kRowsT], sh[kRowsT];  // level >= 2: bucket [lo, hi], bin width 2^sh
    int T[kRowsT], P[kRowsT];
    unsigned need[kRowsT];   // ties at T to take
    unsigned above[kRowsT];  // keys above the current bucket
    int open[kRowsT];        // threshold not exact yet
    int w16[kRowsT];         // level >= 2: 512 16-bit bins
    int kind[kRowsT];        // kKindLog, kKindBucket or kKindBracket
    unsigned cab[kRowsT], cbe[kRowsT];  // bracket pass: keys above / below the bracket
    uint32_t tmem_base;
    int mode, level, exact_all;
    int stride, toff;  // sample pass: key tiles toff, toff + stride, ...
    int sround;        // sample passes done (the log histogram, then the bracket refinement)
    unsigned rhi[kRowsT], rlo[kRowsT];  // sample ranks that bound the K-th score
};

struct TcSelArgs {
    const int8_t *qI;
    const uint16_t *kh;
    const int32_t *wI;
    int32_t *idx, *cnt, *thr, *flags, *status;
    uint32_t *mask;  // optional: selected keys as bits, word-major [words][mask_rows]
    long long mask_rows;
    long long B, Tq, Tk, Tkp, q_offset, wait_ns;
    int H_I, K;
    int pos_div;  // rows per query position (one per indexer head with per-head sets)
    int relu;     // one indexer head: score = w * max(0, q . k)
};

// ---- level-1 (log) classes of an exact integer score held in fp32:
// class m = 0 for 0, else 4 * floor(log2|s|) + (two bits below the leading
// one) + 1; bin = kLog0 +- m. |s| < 2^24 keeps m <= 97.
__device__ __forceinline__ int log_bin(float f) {
    const unsigned u = __float_as_uint(f);
    const int m = max(0, (int)((u & 0x7fffffffu) >> 21) - 507);
    return (int)u < 0 ? kLog0 - m : kLog0 + m;
}
// integers of magnitude class m: [lo, hi] (empty when lo > hi)
__device__ __forceinline__ void mag_range(int m, int &lo, int &hi) {
    if (m == 0) {
        lo = hi = 0;
        return;
    }
    const int E = (m - 1) >> 2, m2 = (m - 1) & 3;
    lo = (int)((((long long)(4 + m2) << E) + 3) >> 2);
    hi = (int)((((long long)(5 + m2) << E) + 3) >> 2) - 1;
}
__device__ __forceinline__ void bin_range1(int bin, int &lo, int &hi) {
    int l, h;
    mag_range(bin >= kLog0 ? bin - kLog0 : kLog0 - bin, l, h);
    if (bin >= kLog0) {
        lo = l;
        hi = h;
    } else {
        lo = -h;
        hi = -l;
    }
}
// lowest score of level-1 bin `bin` or above: every key in a bin >= bin
// scores at least this
__device__ __forceinline__ float bin_floor1(int bin) {
    int lo, hi;
    bin_range1(bin, lo, hi);
    return (float)lo;  // also for an empty bin: every higher bin starts above it
}
// walk a row's level-1 histogram down from its top bin: the floor of the
// bin where the count reaches `need` bounds the row's need-th largest score
// from below (the counts only ever grow, so a racing read is conservative)
__device__ __forceinline__ float rescan1(const volatile unsigned *h, int top, unsigned need) {
    unsigned cum = 0;
    for (int bn = top; bn >= 0; bn--) {
        cum += h[bn];
        if (cum >= need) return bin_floor1(bn);
    }
    return -INFINITY;
}

// Shared-memory counter update under a predicate, without a branch: the
// per-element histogram updates of the passes below stay in straight-line
// code whatever the other rows of the warp do (the address is formed for
// every element and used only where the predicate holds).
__device__ __forceinline__ void red_smem_if(const unsigned *p, unsigned v, bool pred) {
    asm volatile(
        "{\n .reg .pred q;\n setp.ne.u32 q, %2, 0;\n @q red.shared.add.u32 [%0], %1;\n}\n" ::"r"(smem_u32(p)),
        "r"(v), "r"((unsigned)pred)
        : "memory");
}

// bins of a level >= 2 histogram: 256 x 32-bit counters, or 512 x 16-bit
// counters (two per word) when the bucket holds fewer than 2^16 keys
__device__ __forceinline__ unsigned bin_count(const unsigned *h, int b, bool w16) {
    return w16 ? (h[b >> 1] >> ((b & 1) * 16)) & 0xFFFFu : h[b];
}

// One warp, one row's histogram hh (bpl bins per lane; wide: 512 16-bit
// bins): the bin v where the count of keys in bins above v stays below
// `need` and reaches it with bin v. Returns -1 in `found` when the
// histogram holds fewer than `need` keys; `total` = all keys counted.
__device__ __forceinline__ void warp_crossing(const unsigned *hh, bool wide, unsigned need, int lane, int &found,
                                              unsigned &above_in, unsigned &in_bin, unsigned &total) {
    const int bpl = wide ? 16 : 8;  // bins per lane
    const int b0 = lane * bpl;
    unsigned seg = 0;
    for (int v = 0; v < bpl; v++) seg += bin_count(hh, b0 + v, wide);
    unsigned xs = seg;  // keys in the bins of lanes >= lane
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const unsigned y = __shfl_down_sync(0xffffffffu, xs, d);
        if (lane + d < 32) xs += y;
    }
    total = __shfl_sync(0xffffffffu, xs, 0);
    const unsigned excl = xs - seg;
    int f = -1;
    unsigned ab = 0, ib = 0;
    if (excl < need && need <= xs) {
        unsigned acc = excl;
        for (int v = b0 + bpl - 1; v >= b0; v--) {
            const unsigned hv = bin_count(hh, v, wide);
            if (acc + hv >= need) {
                f = v;
                ab = acc;
                ib = hv;
                break;
            }
            acc += hv;
        }
    }
    const unsigned fl = __ballot_sync(0xffffffffu, f >= 0);
    found = -1;
    above_in = in_bin = 0;
    if (fl != 0u) {
        const int src = __ffs(fl) - 1;
        found = __shfl_sync(0xffffffffu, f, src);
        above_in = __shfl_sync(0xffffffffu, ab, src);
        in_bin = __shfl_sync(0xffffffffu, ib, src);
    }
}

template <int DI>
__global__ void __launch_bounds__(kThreadsTc, 1) rows_tc_kernel(const __grid_constant__ TcSelArgs a) {
    using L = TcLay<DI>;
    constexpr int S = L::STAGES;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ TcShared st;
    __shared__ volatile int abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int K = a.K;
    const long long ntile = (a.Tq + kRowsT - 1) / kRowsT;
    const long long b = (long long)blockIdx.x % a.B;
    const long long tile = ntile - 1 - (long long)blockIdx.x / a.B;  // longest prefixes first
    const long long t0 = tile * kRowsT;
    const long long row0 = b * a.Tq + t0;
    const int nrows = (int)min((long long)kRowsT, a.Tq - t0);
    const long long nmax = a.q_offset + (t0 + nrows - 1) / a.pos_div + 1;
    const int ntk = (int)((nmax + kKT - 1) / kKT);  // key tiles per pass
    const uint32_t sbase = smem_u32(smem);
    unsigned *hist = reinterpret_cast<unsigned *>(smem + L::HIST);
    auto bar = [](unsigned long long &x) { return smem_u32(&x); };

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&st.tmem_base)),
                     "r"(kTBufs * kKT));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (tid == kProdWarp * 32) {
        for (int i = 0; i < S; i++) {
            mbar_init(bar(st.full[i]), 1);
            mbar_init(bar(st.sfree[i]), 1);
        }
        for (int i = 0; i < kTBufs; i++) {
            mbar_init(bar(st.tfull[i]), 1);
            mbar_init(bar(st.tfree[i]), kCons / 32);
        }
        mbar_init(bar(st.mma_end), 1);
        mbar_fence_init();
        abort_flag = 0;
        st.exact_all = 1;
        st.mode = kModeStart;
        st.level = 0;
    }
    __syncthreads();
    if (warp < kConsWarps) {
        // collapsed indexer query of row r, fp16 in the core-matrix layout
        // (8 rows x 16 B per core matrix; K-adjacent core matrices 128 B
        // apart, 8-row groups DI*16 B apart); thread part pt writes the
        // 8-column groups g with g % 4 == pt and checks the whole row
        const int r = tid & (kRowsT - 1), pt = tid >> 7;
        const int8_t *qrow = a.qI + (row0 + (r < nrows ? r : 0)) * (long long)a.H_I * DI;
        long long absum = 0;
        bool fits = true;
        for (int c0 = 0; c0 < DI; c0 += 8) {
            long long acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            for (int hh = 0; hh < a.H_I; hh++) {
                // with the ReLU the (single) head's weight is applied to the clamped score
                const long long wv = a.relu ? 1 : a.wI[hh];
                const uint2 raw = *reinterpret_cast<const uint2 *>(qrow + hh * DI + c0);
#pragma unroll
                for (int e = 0; e < 8; e++)
                    acc[e] += wv * (int8_t)(((e < 4 ? raw.x : raw.y) >> (8 * (e & 3))) & 0xFF);
            }
#pragma unroll
            for (int e = 0; e < 8; e++) {
                fits = fits && acc[e] >= -2048 && acc[e] <= 2048;
                absum += acc[e] < 0 ? -acc[e] : acc[e];
            }
            if (((c0 >> 3) & (kParts - 1)) == pt) {
                uint32_t pk[4];
#pragma unroll
                for (int e = 0; e < 4; e++) pk[e] = pack_f16((float)acc[2 * e], (float)acc[2 * e + 1]);
                if (r >= nrows || !fits) pk[0] = pk[1] = pk[2] = pk[3] = 0u;
                *reinterpret_cast<uint4 *>(smem + L::QE + (r >> 3) * (DI * 16) + (c0 >> 3) * 128 + (r & 7) * 16) =
                    make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
        }
        const long long wmul = a.relu ? (a.wI[0] < 0 ? -(long long)a.wI[0] : (long long)a.wI[0]) : 1;
        fits = fits && absum * 128 * wmul < (1ll << 24);
        if (r < nrows && !fits) atomicAnd(&st.exact_all, 0);
        if (pt == 0) {
            const int n = r < nrows ? (int)(a.q_offset + (t0 + r) / a.pos_div + 1) : 0;
            st.n[r] = n;
            st.open[r] = n > K;  // a prefix of at most K keys is taken whole
            st.T[r] = INT32_MIN;
            st.P[r] = n - 1;
            st.need[r] = (unsigned)K;
            st.above[r] = 0u;
            st.w16[r] = 0;
            st.lo[r] = st.hi[r] = st.sh[r] = 0;
            st.kind[r] = kKindLog;
        }
        fence_async_smem();  // q_eff is read by the tensor cores
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = st.tmem_base;
    const bool exact = st.exact_all != 0;
    if (tid == 0) a.flags[b * ntile + tile] = exact ? 0 : 1;

    if (exact) {
        int g0 = 0;  // key tiles issued by earlier passes (barrier phases run on across passes)
        // per-thread state of the consumer threads
        const int q4 = warp & 3, pt = (warp >> 2) & (kParts - 1), r = 32 * q4 + lane;
        const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
        for (;;) {
            if (tid == 0) {
                int any = 0;
                for (int i = 0; i < kRowsT; i++) any |= st.open[i];
                const int m = st.mode;
                int next = m == kModeFinal ? kModeDone : (any ? kModeHist : kModeFinal);
                if (m == kModeStart && any && ntk >= kSampleMinTiles) next = kModeSample;
                if (m == kModeSample && any && st.sround < 2) next = kModeSample;
                if (abort_flag) next = kModeDone;
                if (next == kModeSample) {
                    if (m == kModeStart) {
                        st.stride = ntk >= 256 ? 16 : (ntk >= 128 ? 8 : 4);
                        st.toff = st.stride / 2;
                        st.level = 0;
                        st.sround = 0;
                    }
                    st.sround++;
                } else if (next == kModeHist) {
                    st.level = st.level + 1;
                    if (st.level > kMaxLevels) {  // consistency check; never reached
                        set_status(a.status, ESA_ERR_INTERNAL);
                        next = kModeDone;
                    }
                }
                st.mode = next;
            }
            __syncthreads();
            const int mode = st.mode;
            if (mode == kModeDone) break;
            // key tiles of this pass: all of the prefix's, or the sample's
            const int tstep = mode == kModeSample ? st.stride : 1, toff = mode == kModeSample ? st.toff : 0;
            const int ntp = mode == kModeSample ? (ntk - toff + tstep - 1) / tstep : ntk;

            if (warp == kProdWarp) {
                // ---------------------------------------------- key tiles
                if (lane == 0) {
                    const uint64_t pol = l2_evict_last_policy();
                    const char *src = reinterpret_cast<const char *>(a.kh) + (size_t)(b * a.Tkp) * DI * 2;
                    for (int it = 0; it < ntp; it++) {
                        const int t = toff + it * tstep;
                        const int g = g0 + it, slot = g % S;
                        if (g >= S && !wait_or_abort(bar(st.sfree[slot]), (uint32_t)(g / S - 1) & 1u, a.wait_ns,
                                                     &abort_flag, a.status))
                            break;
                        mbar_expect_tx(bar(st.full[slot]), (unsigned)L::KT_BYTES);
                        bulk_g2s(sbase + L::RING + slot * L::KT_BYTES, src + (size_t)t * L::KT_BYTES,
                                 (unsigned)L::KT_BYTES, bar(st.full[slot]), pol);
                    }
                }
                __syncwarp();
            } else if (warp == kMmaWarp) {
                // ---------------------------------------------- MMA issue
                if (lane == 0) {
                    constexpr uint32_t id = idesc(kKT, 0u, 0u);  // fp16 x fp16 -> fp32, N = 128
                    for (int it = 0; it < ntp; it++) {
                        const int g = g0 + it, slot = g % S, buf = g % kTBufs;
                        if (!wait_or_abort(bar(st.full[slot]), (uint32_t)(g / S) & 1u, a.wait_ns, &abort_flag,
                                           a.status))
                            break;
                        if (g >= kTBufs && !wait_or_abort(bar(st.tfree[buf]), (uint32_t)(g / kTBufs - 1) & 1u,
                                                          a.wait_ns, &abort_flag, a.status))
                            break;
                        tc_fence_after();
                        const uint32_t ks = sbase + L::RING + slot * L::KT_BYTES;
#pragma unroll
                        for (int kk = 0; kk < DI / 16; kk++)
                            mma_ss(tmem + buf * kKT, sdesc(sbase + L::QE + kk * 256, 128, DI * 16),
                                   sdesc(ks + kk * 256, 128, DI * 16), id, kk > 0);
                        mma_commit(bar(st.sfree[slot]));
                        mma_commit(bar(st.tfull[buf]));
                    }
                }
                __syncwarp();
            } else {
                // ---------------------------------------------- scores
                const int n_r = st.n[r];
                const bool open_r = st.open[r] != 0;
                unsigned *h = hist + r * kHS;
                if (mode == kModeHist || mode == kModeSample) {
                    for (int i = tid; i < kRowsT * kHS; i += kCons) hist[i] = 0u;
                    if (tid < kRowsT) st.cab[tid] = st.cbe[tid] = 0u;
                    __syncwarp();
                    asm volatile("bar.sync 5, %0;" ::"n"(kCons) : "memory");  // histograms cleared
                }
                const int kind_r = st.kind[r];
                unsigned ca = 0, cb = 0;  // bracket pass: this part's keys above / below the bracket
                const int lo = st.lo[r], hi = st.hi[r], sh = st.sh[r];
                const float flo = (float)lo, fhi = (float)hi;
                const float Tf = (float)st.T[r];
                const unsigned need = st.need[r];
                const bool w16 = st.w16[r] != 0;
                const float wf = a.relu ? (float)a.wI[0] : 1.f;
                // level 1: running lower bound on the K-th largest score; it starts
                // below every score (|s| < 2^24) and above the -inf that marks
                // keys past the prefix, which therefore never count
                float fb = -33554432.f;
                int since_scan = 0;
                unsigned tie_run = 0, out_run = 0;  // final pass: ties seen, positions written
                int32_t *orow = (a.idx && r < nrows) ? a.idx + (row0 + r) * (long long)K : nullptr;
                uint2 *xch = reinterpret_cast<uint2 *>(hist);  // final pass: [2][kRowsT][kParts] (g, e)
                for (int it = 0; it < ntp; it++) {
                    const int t = toff + it * tstep;
                    const int g = g0 + it, buf = g % kTBufs;
                    wait_or_abort(bar(st.tfull[buf]), (uint32_t)(g / kTBufs) & 1u, a.wait_ns, &abort_flag, a.status);
                    __syncwarp();  // tcgen05.ld is warp-collective
                    tc_fence_after();
                    uint32_t x[kCols];
                    tmem_ld32(tmem + lane_base + buf * kKT + pt * kCols, x);
                    tmem_wait_ld();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(st.tfree[buf]));  // the warp's scores are in registers
                    if (a.relu) {  // w * max(0, q . k): exact, |w| * sum|q| * 128 < 2^24
#pragma unroll
                        for (int c = 0; c < kCols; c++) x[c] = __float_as_uint(wf * fmaxf(__uint_as_float(x[c]), 0.f));
                    }
                    const int j0 = t * kKT + pt * kCols;
                    const int lim = max(0, min(kCols, n_r - j0));  // columns c < lim are in the prefix
                    if (mode == kModeSample && kind_r == kKindLog) {
                        // every sampled key of the prefix, log histogram
                        if (!open_r || lim == 0) continue;
#pragma unroll
                        for (int c = 0; c < kCols; c++) red_smem_if(h + log_bin(__uint_as_float(x[c])), 1u, c < lim);
                    } else if (mode == kModeHist || mode == kModeSample) {
                        if (!open_r || lim == 0) continue;
                        if (kind_r == kKindBracket) {
                            // above, below or inside the bracket [lo, hi]
#pragma unroll
                            for (int c = 0; c < kCols; c++) {
                                const float f = __uint_as_float(x[c]);
                                const bool in = c < lim, up = f > fhi, dn = f < flo;
                                ca += in && up;
                                cb += in && dn;
                                const int bn = (int)((unsigned)(__float2int_rz(f) - lo) >> sh) & (2 * kNB - 1);
                                red_smem_if(h + (bn >> 1), 1u << ((bn & 1) * 16), in && !up && !dn);
                            }
                            continue;
                        }
                        if (lim < kCols) {  // keys past the row's prefix never count
#pragma unroll
                            for (int c = 0; c < kCols; c++)
                                if (c >= lim) x[c] = 0xff800000u;  // -inf
                        }
                        if (kind_r == kKindLog) {
#pragma unroll
                            for (int c = 0; c < kCols; c++) {
                                const float f = __uint_as_float(x[c]);
                                red_smem_if(h + log_bin(f), 1u, f >= fb);
                            }
                            // raise the bound: every tile until it is positive, then every 8th
                            if (fb <= 0.f || ++since_scan == 8) {
                                since_scan = 0;
                                fb = fmaxf(fb, rescan1(h, 2 * kLog0, (unsigned)K));
                            }
                        } else {
#pragma unroll
                            for (int c = 0; c < kCols; c++) {
                                const float f = __uint_as_float(x[c]);
                                const int bn = (int)((unsigned)(__float2int_rz(f) - lo) >> sh) & (2 * kNB - 1);
                                red_smem_if(w16 ? h + (bn >> 1) : h + (bn & (kNB - 1)), w16 ? 1u << ((bn & 1) * 16) : 1u,
                                            f >= flo && f <= fhi);
                            }
                        }
                    } else {
                        // final pass: ordered write of the selected positions
                        unsigned gt = 0u, eq = 0u;
                        if (lim > 0) {
#pragma unroll
                            for (int c = 0; c < kCols; c++) {
                                const float f = __uint_as_float(x[c]);
                                gt |= (unsigned)(f > Tf) << c;
                                eq |= (unsigned)(f == Tf) << c;
                            }
                            const unsigned in = lim == kCols ? ~0u : (1u << lim) - 1u;  // keys in the prefix
                            gt &= in;
                            eq &= in;
                        }
                        const int slot = ((t & 1) * kRowsT + r) * kParts;
                        xch[slot + pt] = make_uint2((unsigned)__popc(gt), (unsigned)__popc(eq));
                        __syncwarp();
                        asm volatile("bar.sync %0, %1;" ::"r"(1 + q4), "n"(32 * kParts) : "memory");
                        // the row's parts in key order: ties taken while fewer than
                        // `need` have been, and this part's first output slot
                        unsigned tie = tie_run, ob = out_run, my_tb = 0u, my_take = 0u, my_ob = 0u;
#pragma unroll
                        for (int i = 0; i < kParts; i++) {
                            const uint2 ci = xch[slot + i];
                            const unsigned take_i = tie >= need ? 0u : min(ci.y, need - tie);
                            if (i == pt) {
                                my_tb = tie;
                                my_take = take_i;
                                my_ob = ob;
                            }
                            ob += ci.x + take_i;
                            tie += ci.y;
                        }
                        out_run = ob;
                        tie_run = tie;
                        unsigned sel = gt, ee = eq;
                        int last = -1;
                        for (unsigned i = 0; i < my_take; i++) {
                            const unsigned lb = ee & (0u - ee);
                            sel |= lb;
                            ee ^= lb;
                            last = __ffs(lb) - 1;
                        }
                        if (my_take > 0 && my_tb + my_take == need) st.P[r] = j0 + last;
                        if (a.mask && r < nrows) a.mask[(long long)(j0 >> 5) * a.mask_rows + row0 + r] = sel;
                        if (orow) {
                            while (sel) {
                                const int bit = __ffs(sel) - 1;
                                sel &= sel - 1;
                                if (my_ob < (unsigned)K) orow[my_ob] = j0 + bit;
                                else set_status(a.status, ESA_ERR_INTERNAL);
                                my_ob++;
                            }
                        }
                    }
                }
                if (mode == kModeFinal && r < nrows && pt == 0 && !abort_flag &&
                    out_run != (unsigned)min(K, n_r))  // consistency check; never reached
                    set_status(a.status, ESA_ERR_INTERNAL);
                if ((mode == kModeHist || mode == kModeSample) && open_r && kind_r == kKindBracket) {
                    atomicAdd(&st.cab[r], ca);
                    atomicAdd(&st.cbe[r], cb);
                }
            }
            g0 += ntp;
            __syncthreads();  // pass drained: every MMA read, every histogram count in
            if ((mode == kModeHist || mode == kModeSample) && warp < kConsWarps && !abort_flag) {
                // ---------------------------------------------- next bucket
                // warp w resolves rows w, w+16, ...
                for (int rr = warp; rr < kRowsT; rr += kConsWarps) {
                    if (!st.open[rr]) continue;
                    const unsigned *hh = hist + rr * kHS;
                    int found;
                    unsigned above_in, in_bin, total;
                    if (mode == kModeSample && st.kind[rr] == kKindBracket) {
                        // second sample pass: the sample's keys above, below and in
                        // 512 bins of the log-bin bracket; narrow the bracket to
                        // the bins that hold the sample ranks rhi and rlo
                        const unsigned up = st.cab[rr], r_hi = st.rhi[rr], r_lo = st.rlo[rr];
                        int lo2 = st.lo[rr], hi2 = st.hi[rr];
                        const int sh2 = st.sh[rr];
                        if (up < r_hi) {
                            int bh;
                            warp_crossing(hh, true, r_hi - up, lane, bh, above_in, in_bin, total);
                            if (bh >= 0) hi2 = (int)min((long long)hi2, (long long)lo2 + ((long long)(bh + 1) << sh2) - 1);
                        }
                        if (r_lo > up) {
                            int bl;
                            warp_crossing(hh, true, r_lo - up, lane, bl, above_in, in_bin, total);
                            if (bl >= 0) lo2 = lo2 + (bl << sh2);
                        }
                        if (lane == 0) {
                            int s2 = 0;
                            while ((((long long)hi2 - lo2) >> s2) >= 2 * kNB) s2++;
                            st.lo[rr] = lo2;
                            st.hi[rr] = hi2;
                            st.sh[rr] = s2;
                        }
                        continue;
                    }
                    if (mode == kModeSample) {
                        // bracket the K-th score from the sample: the sample ranks
                        // r -+ d, r = K m / n the expected rank, d = 4 sqrt(r) + 8
                        warp_crossing(hh, false, 0xffffffffu, lane, found, above_in, in_bin, total);
                        const unsigned m = total, n = (unsigned)st.n[rr];
                        const unsigned rx = max(1u, (unsigned)(((unsigned long long)K * m + n / 2) / n));
                        const unsigned dd = (unsigned)(4.f * sqrtf((float)rx)) + 8u;
                        const unsigned r_hi = rx > dd ? rx - dd : 1u, r_lo = rx + dd;
                        int bhi, blo;
                        warp_crossing(hh, false, r_hi, lane, bhi, above_in, in_bin, total);
                        int vlo = -(1 << 24), vhi = 1 << 24;  // |s| < 2^24 (the exactness bound)
                        if (bhi >= 0) {
                            int l2, h2;
                            bin_range1(bhi, l2, h2);
                            vhi = h2;
                        }
                        if (r_lo <= m) {
                            warp_crossing(hh, false, r_lo, lane, blo, above_in, in_bin, total);
                            if (blo >= 0) {
                                int l2, h2;
                                bin_range1(blo, l2, h2);
                                vlo = l2;
                            }
                        }
                        if (lane == 0) {
                            int s2 = 0;
                            while ((((long long)vhi - vlo) >> s2) >= 2 * kNB) s2++;
                            st.kind[rr] = kKindBracket;
                            st.lo[rr] = vlo;
                            st.hi[rr] = vhi;
                            st.sh[rr] = s2;
                            st.w16[rr] = 1;
                            st.above[rr] = 0u;
                            st.rhi[rr] = r_hi;
                            st.rlo[rr] = r_lo;
                        }
                        continue;
                    }
                    const int kind = st.kind[rr];
                    if (kind == kKindBracket) {
                        // the bracket holds the K-th score iff fewer than K keys lie
                        // above it and at least K at or above its floor; 16-bit bins
                        // must sum to the keys inside it (no carry between bins)
                        const unsigned up = st.cab[rr], dn = st.cbe[rr], n = (unsigned)st.n[rr];
                        const unsigned inb = n - up - dn;
                        warp_crossing(hh, true, 0xffffffffu, lane, found, above_in, in_bin, total);
                        const bool valid = total == inb && up < (unsigned)K && up + inb >= (unsigned)K;
                        if (!valid) {  // fall back to the full log histogram
                            if (lane == 0) {
                                st.kind[rr] = kKindLog;
                                st.above[rr] = 0u;
                                st.w16[rr] = 0;
                            }
                            continue;
                        }
                        if (lane == 0) st.above[rr] = up;
                        __syncwarp();
                    }
                    const unsigned need = (unsigned)K - st.above[rr];
                    const bool wide = kind != kKindLog && st.w16[rr] != 0;  // 512 16-bit bins
                    warp_crossing(hh, wide, need, lane, found, above_in, in_bin, total);
                    if (found < 0) {  // consistency check; never reached
                        if (lane == 0) {
                            set_status(a.status, ESA_ERR_INTERNAL);
                            st.open[rr] = 0;
                        }
                        continue;
                    }
                    if (lane == 0) {
                        int nlo, nhi;
                        if (kind == kKindLog) {
                            bin_range1(found, nlo, nhi);
                        } else {
                            nlo = st.lo[rr] + (found << st.sh[rr]);
                            nhi = (int)min((long long)st.hi[rr], (long long)nlo + (1ll << st.sh[rr]) - 1);
                        }
                        st.above[rr] += above_in;
                        if (nlo == nhi) {
                            st.open[rr] = 0;
                            st.T[rr] = nlo;
                            st.need[rr] = (unsigned)K - st.above[rr];
                        } else {
                            // the next level counts only this bucket's keys: 16-bit
                            // counters suffice below 2^16 of them
                            const bool w = in_bin < 65536u;
                            const int nb = w ? 2 * kNB : kNB;
                            int s2 = 0;
                            while ((((long long)nhi - nlo) >> s2) >= nb) s2++;
                            st.kind[rr] = kKindBucket;
                            st.lo[rr] = nlo;
                            st.hi[rr] = nhi;
                            st.sh[rr] = s2;
                            st.w16[rr] = w ? 1 : 0;
                        }
                    }
                }
            }
            __syncthreads();
        }

        // ---- counts, padding and threshold form (one warp per row)
        if (warp < kConsWarps) {
            for (int rr = warp; rr < nrows; rr += kConsWarps) {
                const int n = st.n[rr];
                const int c = min(K, n);
                if (a.idx) {
                    int32_t *orr = a.idx + (row0 + rr) * (long long)K;
                    for (int i = c + lane; i < K; i += 32) orr[i] = -1;
                    if (lane == 0) a.cnt[row0 + rr] = c;
                }
                if (a.thr && lane == 0) {
                    a.thr[2 * (row0 + rr)] = st.T[rr];
                    a.thr[2 * (row0 + rr) + 1] = st.P[rr];
                }
            }
        }
        if (warp == kMmaWarp && lane == 0) {
            // every MMA issued has completed before tensor memory is freed
            mma_commit(bar(st.mma_end));
            mbar_wait_bounded(bar(st.mma_end), 0u, a.wait_ns);
        }
        if (warp == kProdWarp && lane == 0 && abort_flag) {
            // after an abort: let bulk copies still in flight land
            for (int g = max(0, g0 - S); g < g0; g++)
                mbar_wait_bounded(bar(st.full[g % S]), (uint32_t)(g / S) & 1u, a.wait_ns);
        }
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTBufs * kKT));
    }
}

// int8 indexer keys [B, Tk, DI] -> fp16 [B, Tkp, DI] in the core-matrix
// layout: the 16-byte unit U holds keys 8*grp + (U & 7), columns 8*c8 .. +7,
// with U = (grp * DI/8 + c8) * 8 + (U & 7); keys Tk .. Tkp-1 are zero.
__global__ void __launch_bounds__(256) kh_convert_kernel(const int8_t *__restrict__ kI, uint4 *__restrict__ kh,
                                                         long long B, long long Tk, long long Tkp, int DI) {
    const int G = DI / 8;
    const long long units = B * Tkp * G;
    for (long long U = blockIdx.x * (long long)blockDim.x + threadIdx.x; U < units;
         U += (long long)gridDim.x * blockDim.x) {
        const long long rest = U >> 3;
        const int c8 = (int)(rest % G);
        const long long row = (rest / G) * 8 + (U & 7);
        const long long bb = row / Tkp, j = row - bb * Tkp;
        uint4 o = make_uint4(0u, 0u, 0u, 0u);
        if (j < Tk) {
            const uint2 raw = *reinterpret_cast<const uint2 *>(kI + (bb * Tk + j) * DI + c8 * 8);
            auto cv = [](uint32_t w, int e) { return (float)(int8_t)((w >> (8 * e)) & 0xFFu); };
            o.x = pack_f16(cv(raw.x, 0), cv(raw.x, 1));
            o.y = pack_f16(cv(raw.x, 2), cv(raw.x, 3));
            o.z = pack_f16(cv(raw.y, 0), cv(raw.y, 1));
            o.w = pack_f16(cv(raw.y, 2), cv(raw.y, 3));
        }
        kh[U] = o;
    }
}

template <int DI>
constexpr size_t tc_smem() {
    return (size_t)TcLay<DI>::TOTAL;
}

void *tc_kernel(int DI, size_t *smem) {
    switch (DI) {
        case 16: *smem = tc_smem<16>(); return (void *)rows_tc_kernel<16>;
        case 32: *smem = tc_smem<32>(); return (void *)rows_tc_kernel<32>;
        case 64: *smem = tc_smem<64>(); return (void *)rows_tc_kernel<64>;
        default: return nullptr;  // D_I = 128: its buffers do not fit; the dp4a kernel runs it
    }
}

struct TcPlan {
    bool ok;
    long long Tkp, ntile;
    size_t kh_off, flag_off, bytes;
};

// ESA_ROW_SELECT=dp4a keeps the row-tiled selection on the dp4a kernel,
// ESA_ROW_SELECT=tc on the tensor cores wherever they apply (switches for
// comparing the two kernels; both give identical results)
bool tc_disabled() {
    const char *e = getenv("ESA_ROW_SELECT");
    return e && strcmp(e, "dp4a") == 0;
}
bool tc_forced() {
    const char *e = getenv("ESA_ROW_SELECT");
    return e && strcmp(e, "tc") == 0;
}

TcPlan plan_tc(const Shape &s, int) {
    TcPlan p{};
    size_t smem = 0;
    if (!tc_kernel(s.D_I, &smem) || tc_disabled()) return p;
    if (relu_of(s) && s.H_I > 1) return p;  // the ReLU of several heads does not collapse: dp4a
    if (smem + sizeof(TcShared) + 1024 > device_info().smem_optin) return p;
    p.Tkp = (s.Tk + kKT - 1) / kKT * kKT;
    p.ntile = (s.Tq + kRowsT - 1) / kRowsT;
    // a small problem on few 128-row query tiles (fewer than an eighth of the
    // SMs, at most 4M query-key pairs): the dp4a kernel's 32-row tiles give
    // four times the blocks and finish sooner (1024 queries over 1024 keys:
    // 82 against 125 us). ESA_ROW_SELECT=tc keeps the tensor cores.
    if (!tc_forced() && s.B * p.ntile * 8 < device_info().sms && s.B * s.Tq * s.Tk <= (1LL << 22)) return TcPlan{};
    p.kh_off = kStatusBytes;
    p.flag_off = p.kh_off + align256((size_t)s.B * p.Tkp * s.D_I * 2);
    p.bytes = p.flag_off + align256((size_t)s.B * p.ntile * 4);
    p.ok = true;
    return p;
}

}  // namespace

size_t ws_row_select(const Shape &s, int K) {
    TcPlan p = plan_tc(s, K);
    return p.ok ? p.bytes : kStatusBytes;
}

esa_status launch_row_select(const int8_t *qI, const int8_t *kI, const int32_t *wI, const Shape &s, int K,
                             int32_t *idx, int32_t *cnt, int32_t *thr, void *ws, size_t ws_bytes, cudaStream_t st,
                             uint32_t *mask) {
    int32_t *status = reinterpret_cast<int32_t *>(ws);
    if (s.B * s.Tq == 0) return ESA_OK;
    TcPlan p = plan_tc(s, K);
    if (!p.ok || ws_bytes < p.bytes)
        return launch_rows_dp4a(qI, kI, wI, s, K, idx, cnt, thr, nullptr, status, st, mask);
    char *base = static_cast<char *>(ws);
    uint16_t *kh = reinterpret_cast<uint16_t *>(base + p.kh_off);
    int32_t *flags = reinterpret_cast<int32_t *>(base + p.flag_off);
    {
        const long long units = s.B * p.Tkp * (s.D_I / 8);
        const long long want = (units + 255) / 256, cap = (long long)device_info().sms * 16;
        kh_convert_kernel<<<(unsigned)(want < cap ? want : cap), 256, 0, st>>>(kI, reinterpret_cast<uint4 *>(kh), s.B,
                                                                            s.Tk, p.Tkp, s.D_I);
        if (cudaGetLastError() != cudaSuccess) return ESA_ERR_CUDA;
    }
    size_t smem = 0;
    void *fn = tc_kernel(s.D_I, &smem);
    if (!ensure_smem(fn, smem)) return ESA_ERR_CUDA;
    TcSelArgs a{};
    a.qI = qI;
    a.kh = kh;
    a.wI = wI;
    a.idx = idx;
    a.cnt = cnt;
    a.thr = thr;
    a.mask = mask;
    a.mask_rows = s.B * s.Tq;
    a.flags = flags;
    a.status = status;
    a.B = s.B;
    a.Tq = s.Tq;
    a.Tk = s.Tk;
    a.Tkp = p.Tkp;
    a.q_offset = s.q_offset;
    a.wait_ns = wait_limit_ns();
    a.H_I = s.H_I;
    a.K = K;
    a.pos_div = s.pos_div;
    a.relu = relu_of(s) ? 1 : 0;
    void *args[] = {(void *)&a};
    if (cudaLaunchKernel(fn, dim3((unsigned)(s.B * p.ntile)), dim3(kThreadsTc), args, smem, st) != cudaSuccess)
        return ESA_ERR_CUDA;
    // query tiles whose collapsed indexer query is not exact in fp16
    return launch_rows_dp4a(qI, kI, wI, s, K, idx, cnt, thr, flags, status, st, mask);
}

}  // namespace esa
