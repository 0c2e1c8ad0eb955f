// Top-K selection for few query rows with long prefixes (decode).
//
// Method: the Indexer scores the query against every causal-prefix position
// and the K best positions are kept ("超大规模MoE架构中稀疏注意力机制的演进与实践",
// section 二.1, K = 2048; no RoPE, section 二.2). Ties go to the lower position.
//
// Design (one launch, co-resident blocks):
//   * each query row's prefix 0..p is cut into `chunks` contiguous spans,
//     one block per span; the block streams its span of kI once from HBM
//     (16-byte non-allocating loads, 4 threads per key, dp4a) and keeps the
//     int32 scores in shared memory — the score row never reaches HBM;
//   * level 1: a 3330-bin log-scale histogram of the scores (exact below
//     |s| = 128, 6 mantissa bits above), summed across the row's blocks with
//     global atomics, then a bounded barrier among the row's blocks;
//   * every block finds the bucket holding the K-th largest score; level 2
//     histograms that bucket exactly (a level 3 follows only when the bucket
//     is wider than 4096 values, i.e. |s| >= 2^18);
//   * at the exact level each block also publishes its own suffix counts, so
//     after the last barrier every block knows the threshold T, how many
//     scores above T and ties at T lie in earlier spans, and writes its part
//     of the ascending index list with warp ballots — no further exchange.
// Control state (barrier counters, global histograms) lives in the caller's
// workspace and is returned to zero by every launch: each block clears its
// slice of a level's histogram once the next barrier shows that every block
// of the row has read it, and the last block of a row to finish clears the
// final level and the counters.
#include <cooperative_groups.h>

#include "esa_device.cuh"
#include "esa_internal.h"

namespace esa {

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kNB1 = 3330;
constexpr int kHalf1 = 1665;
constexpr int kNB2 = 4096;
constexpr int kMaxChunk = 16384;
constexpr int kUnroll = 8;
// per-row control words: [0] barrier counter, [1] exit counter, then the
// level histograms
constexpr size_t kRowCtrl = 4 + kNB1 + 2 * (size_t)kNB2;
constexpr size_t kPubWords = kNB2 + 2;

__device__ __forceinline__ int log_bin(int s) {
    unsigned a = s < 0 ? 0u - (unsigned)s : (unsigned)s;
    int m;
    if (a < 128u) {
        m = (int)a;
    } else {
        int e = 31 - __clz(a);
        m = 128 + (e - 7) * 64 + (int)((a >> (e - 6)) & 63u);
    }
    return s >= 0 ? kHalf1 + m : kHalf1 - m;
}

__device__ __forceinline__ void log_bin_range(int bin, long long &lo, long long &hi) {
    int m = bin >= kHalf1 ? bin - kHalf1 : kHalf1 - bin;
    long long alo, ahi;
    if (m < 128) {
        alo = ahi = m;
    } else {
        int e = 7 + (m - 128) / 64, mant = (m - 128) % 64;
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

struct Smem {
    unsigned h1[kNB1];
    unsigned h2[kNB2];
    int32_t q[16 * 32];  // indexer query words [H_I][D_I/4]
    int32_t w[16];
    unsigned red[64];
    unsigned wsum[2][kWarps];
    int flag;
    int bin;
    unsigned above;
    int pad[5];
    // followed by the scores of the block's span (int32)
};

// Block-wide: among bins [0,nb) of the global histogram h, find v with
// sum_{u>v} h[u] < need <= sum_{u>=v} h[u]. Result in sm.bin / sm.above
// (sm.bin = -1 if there is none). The bins are first staged into `stage`
// (shared, >= nb words) with independent loads, so the search costs one L2
// round trip.
__device__ void find_crossing(const unsigned *h, int nb, unsigned need, unsigned *stage, Smem &sm) {
    int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) sm.bin = -1;
#pragma unroll 8
    for (int i = tid; i < nb; i += kThreads) stage[i] = __ldcg(h + i);
    __syncthreads();
    int per = (nb + kThreads - 1) / kThreads;
    int b0 = tid * per, b1 = min(nb, b0 + per);
    unsigned seg = 0;
    for (int v = b0; v < b1; v++) seg += stage[v];
    // inclusive suffix sum within the warp (lanes with higher index = higher bins)
    unsigned x = seg;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        unsigned y = __shfl_down_sync(0xffffffffu, x, d);
        if (lane + d < 32) x += y;
    }
    if (lane == 0) sm.red[warp] = x;  // warp total
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

template <int DI>
__global__ void __launch_bounds__(kThreads) split_select_kernel(
    const int8_t *__restrict__ qI, const int8_t *__restrict__ kI, const int32_t *__restrict__ wI,
    int32_t *__restrict__ idx, int32_t *__restrict__ cnt, long long Tq, long long Tk, long long q_offset, int H_I,
    int K, int chunks, unsigned *ctrl, unsigned *pub, int32_t *status, long long wait_ns, int extra) {
    constexpr int W = DI / 4;       // int32 words per indexer vector
    constexpr int TPK = 4;          // threads per key
    constexpr int WPT = W / TPK;    // words per thread (1, 2, 4 or 8)
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Smem &sm = *reinterpret_cast<Smem *>(smem_raw);
    int32_t *sc = reinterpret_cast<int32_t *>(smem_raw + sizeof(Smem));

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const long long row = blockIdx.x / chunks;
    const int ci = blockIdx.x % chunks;
    const long long b = row / Tq, t = row % Tq;
    const long long n = q_offset + t + 1;

    pdl_wait();

    int32_t *idx_row = idx + row * (long long)K;
    if (n <= K) {  // the whole prefix is kept
        if (ci == 0) {
            for (long long i = tid; i < K; i += kThreads) idx_row[i] = i < n ? (int32_t)i : -1;
            if (tid == 0) cnt[row] = (int32_t)n;
        }
    } else {
        unsigned *rc = ctrl + row * kRowCtrl;
        unsigned *bar = rc;
        unsigned *row_exit = rc + 1;
        unsigned *g1 = rc + 4;
        unsigned *gl[2] = {g1 + kNB1, g1 + kNB1 + kNB2};
        unsigned *mypub = pub + ((size_t)row * chunks + ci) * kPubWords;
        const long long len = (n + chunks - 1) / chunks;
        const long long lo = ci * len;
        const long long hi = min(n, lo + len);
        const int span = (int)max(0ll, hi - lo);

        for (int i = tid; i < kNB1; i += kThreads) sm.h1[i] = 0u;
        for (int i = tid; i < H_I * W; i += kThreads)
            sm.q[i] = reinterpret_cast<const int32_t *>(qI + row * (long long)H_I * DI)[i];
        if (tid < H_I) sm.w[tid] = wI[tid];
        __syncthreads();

        // ---- phase A: stream this span of kI, score, level-1 histogram
        {
            const int quad = tid / TPK, part = tid % TPK;
            const int8_t *kbase = kI + (b * Tk + lo) * DI + part * (DI / TPK);
            constexpr int kQuads = kThreads / TPK;
            for (int base = 0; base < span; base += kQuads * kUnroll) {
                uint32_t kw[kUnroll][WPT];
#pragma unroll
                for (int u = 0; u < kUnroll; u++) {
                    int j = base + u * kQuads + quad;
                    if (j < span) {
                        const int8_t *p = kbase + (long long)j * DI;
                        if constexpr (WPT == 1) {
                            kw[u][0] = __ldg(reinterpret_cast<const uint32_t *>(p));
                        } else if constexpr (WPT == 2) {
                            uint2 v = __ldg(reinterpret_cast<const uint2 *>(p));
                            kw[u][0] = v.x;
                            kw[u][1] = v.y;
                        } else {
#pragma unroll
                            for (int c = 0; c < WPT / 4; c++) {
                                uint4 v = ldg_stream16(p + 16 * c);
                                kw[u][4 * c] = v.x;
                                kw[u][4 * c + 1] = v.y;
                                kw[u][4 * c + 2] = v.z;
                                kw[u][4 * c + 3] = v.w;
                            }
                        }
                    }
                }
#pragma unroll
                for (int u = 0; u < kUnroll; u++) {
                    int j = base + u * kQuads + quad;
                    unsigned acc = 0;
                    for (int h = 0; h < H_I; h++) {
                        int d = 0;
#pragma unroll
                        for (int c = 0; c < WPT; c++) d = __dp4a(sm.q[h * W + part * WPT + c], (int)kw[u][c], d);
                        acc += (unsigned)sm.w[h] * (unsigned)d;
                    }
                    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
                    acc += __shfl_xor_sync(0xffffffffu, acc, 2);
                    if (part == 0 && j < span) {
                        int s = (int)acc;
                        sc[j] = s;
                        atomicAdd(&sm.h1[log_bin(s)], 1u);
                    }
                }
            }
        }
        __syncthreads();
        for (int i = tid; i < kNB1; i += kThreads)
            if (sm.h1[i]) atomicAdd(g1 + i, sm.h1[i]);
        bool ok = group_barrier(bar, (unsigned)chunks + extra, wait_ns, status, &sm.flag);

        // ---- levels 2 (and 3): exact threshold
        long long vlo = 0, vhi = 0;
        unsigned above = 0;
        int T = 0;
        int shift = 0, nb = 1, levels_used = 1;
        if (ok) {
            find_crossing(g1, kNB1, (unsigned)K, sm.h1, sm);
            if (sm.bin < 0) {
                if (tid == 0) set_status(status, ESA_ERR_INTERNAL);
                ok = false;
            } else {
                above = sm.above;
                log_bin_range(sm.bin, vlo, vhi);
            }
        }
        for (int level = 2; level <= 3 && ok; level++) {
            levels_used = level;
            long long Wd = vhi - vlo + 1;
            shift = 0;
            while (((Wd - 1) >> shift) >= kNB2) shift++;
            nb = (int)(((Wd - 1) >> shift) + 1);
            for (int i = tid; i < nb; i += kThreads) sm.h2[i] = 0u;
            __syncthreads();
            unsigned mine_above = 0;
            for (int j = tid; j < span; j += kThreads) {
                long long s = sc[j];
                if (s >= vlo && s <= vhi) atomicAdd(&sm.h2[(int)((s - vlo) >> shift)], 1u);
                mine_above += (s > vhi);
            }
            __syncthreads();
            unsigned *gdst = gl[level - 2];
            for (int i = tid; i < nb; i += kThreads)
                if (sm.h2[i]) atomicAdd(gdst + i, sm.h2[i]);
            if (shift == 0) {
                // publish: [0] count above the bucket, [1+v] = #scores >= vlo+v
                // within the bucket (suffix counts), [1+nb] = 0
#pragma unroll
                for (int d = 16; d > 0; d >>= 1) mine_above += __shfl_xor_sync(0xffffffffu, mine_above, d);
                if (lane == 0) sm.red[warp] = mine_above;
                // suffix scan of h2 over nb bins, in place into mypub
                int per = (nb + kThreads - 1) / kThreads;
                int b0 = tid * per, b1 = min(nb, b0 + per);
                unsigned seg = 0;
                for (int v = b0; v < b1; v++) seg += sm.h2[v];
                unsigned x = seg;
#pragma unroll
                for (int d = 1; d < 32; d <<= 1) {
                    unsigned y = __shfl_down_sync(0xffffffffu, x, d);
                    if (lane + d < 32) x += y;
                }
                if (lane == 0) sm.red[32 + warp] = x;
                __syncthreads();
                unsigned higher = 0;
                for (int w2 = warp + 1; w2 < kWarps; w2++) higher += sm.red[32 + w2];
                unsigned a = x + higher - seg;  // count in bins above b1-1
                for (int v = b1 - 1; v >= b0; v--) {
                    a += sm.h2[v];
                    mypub[1 + v] = a;
                }
                if (tid == 0) {
                    unsigned tot = 0;
                    for (int w2 = 0; w2 < kWarps; w2++) tot += sm.red[w2];
                    mypub[0] = tot;
                    mypub[1 + nb] = 0u;
                }
            }
            ok = group_barrier(bar, (unsigned)(level * chunks + extra), wait_ns, status, &sm.flag);
            if (!ok) break;
            {  // every block of the row has read the previous level: clear my slice of it
                unsigned *prev = level == 2 ? g1 : gl[0];
                int pn = level == 2 ? kNB1 : kNB2;
                int per = (pn + chunks - 1) / chunks;
                for (int i = ci * per + tid; i < min(pn, (ci + 1) * per); i += kThreads) prev[i] = 0u;
            }
            find_crossing(gdst, nb, (unsigned)K - above, sm.h2, sm);
            if (sm.bin < 0) {
                if (tid == 0) set_status(status, ESA_ERR_INTERNAL);
                ok = false;
                break;
            }
            above += sm.above;
            if (shift == 0) {
                T = (int)(vlo + sm.bin);
                break;
            }
            vlo = vlo + ((long long)sm.bin << shift);
            vhi = min(vhi, vlo + (1ll << shift) - 1);
        }

        if (ok && shift != 0) {  // cannot happen: three levels always resolve an int32 score
            if (tid == 0) set_status(status, ESA_ERR_INTERNAL);
            ok = false;
        }
        // ---- phase C: ordered write of this span's selected positions
        if (ok) {
            const int vstar = sm.bin;
            const unsigned need_ties = (unsigned)K - above;  // ties at T to take, >= 1
            // earlier spans: scores above T and ties at T
            unsigned gt_b = 0, eq_b = 0;
            for (int c = tid; c < ci; c += kThreads) {
                const unsigned *pp = pub + ((size_t)row * chunks + c) * kPubWords;
                unsigned ge = __ldcg(pp + 1 + vstar), gt = __ldcg(pp + 2 + vstar);
                gt_b += __ldcg(pp) + gt;
                eq_b += ge - gt;
            }
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
            // per-warp counts over contiguous segments of the span
            const int seg = ((span + kWarps * 32 - 1) / (kWarps * 32)) * 32;
            const int s0 = warp * seg, s1 = min(span, s0 + seg);
            unsigned wgt = 0, weq = 0;
            for (int j = s0 + lane; j < s1; j += 32) {
                int s = sc[j];
                wgt += (s > T);
                weq += (s == T);
            }
#pragma unroll
            for (int d = 16; d > 0; d >>= 1) {
                wgt += __shfl_xor_sync(0xffffffffu, wgt, d);
                weq += __shfl_xor_sync(0xffffffffu, weq, d);
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
            for (int j0 = s0; j0 < s1; j0 += 32) {
                int j = j0 + lane;
                int s = j < s1 ? sc[j] : INT32_MIN;
                bool in = j < s1;
                bool gt = in && s > T, eq = in && s == T;
                unsigned eqm = __ballot_sync(0xffffffffu, eq);
                unsigned rank = tie + __popc(eqm & lanemask_lt());
                bool sel = gt || (eq && rank < need_ties);
                unsigned selm = __ballot_sync(0xffffffffu, sel);
                if (sel) {
                    unsigned pos = out + __popc(selm & lanemask_lt());
                    if (pos < (unsigned)K) idx_row[pos] = (int32_t)(lo + j);
                    else set_status(status, ESA_ERR_INTERNAL);
                }
                out += __popc(selm);
                tie += __popc(eqm);
            }
            if (ci == 0 && tid == 0) cnt[row] = K;

            // ---- exit: the last block of the row clears the final level and
            // the counters (every block of the row has read them by now)
            __syncthreads();
            if (tid == 0) {
                __threadfence();
                sm.flag = (atomicAdd(row_exit, 1u) == (unsigned)chunks - 1) ? 1 : 0;
            }
            __syncthreads();
            if (sm.flag) {
                unsigned *fin = shift == 0 && levels_used == 3 ? gl[1] : gl[0];
                for (int i = tid; i < nb; i += kThreads) fin[i] = 0u;
                if (tid == 0) {
                    *bar = 0u;
                    *row_exit = 0u;
                }
            }
        }
    }
    pdl_launch_dependents();
}

template <int DI>
size_t smem_bytes(int chunk) {
    return sizeof(Smem) + (size_t)chunk * sizeof(int32_t);
}

void *kernel_ptr(int DI) {
    switch (DI) {
        case 16: return (void *)split_select_kernel<16>;
        case 32: return (void *)split_select_kernel<32>;
        case 64: return (void *)split_select_kernel<64>;
        default: return (void *)split_select_kernel<128>;
    }
}

}  // namespace

SplitPlan plan_split_select(const Shape &s, int K) {
    SplitPlan p{};
    p.ok = false;
    long long rows = s.B * s.Tq;
    if (rows <= 0) return p;
    long long nmax = s.q_offset + s.Tq;  // longest prefix
    DevInfo di = device_info();
    size_t smem = sizeof(Smem) + (size_t)kMaxChunk * sizeof(int32_t);
    void *fn = kernel_ptr(s.D_I);
    int per_sm = occupancy(fn, kThreads, smem);
    if (per_sm < 1) return p;
    long long resident = (long long)di.sms * per_sm;
    if (rows > resident / 2) return p;  // each row should get >= 2 blocks
    int chunks = (int)(resident / rows);
    long long len = (nmax + chunks - 1) / chunks;
    if (len > kMaxChunk) return p;
    // shrink shared memory to the span actually needed
    size_t need = sizeof(Smem) + (size_t)((len + 31) / 32 * 32) * sizeof(int32_t);
    p.ok = true;
    p.chunks = chunks;
    p.grid = (int)(rows * chunks);
    p.smem = need;
    p.ctrl_words = (size_t)rows * kRowCtrl;
    size_t ctrl_bytes = align256(p.ctrl_words * 4);
    size_t pub_bytes = align256((size_t)rows * chunks * kPubWords * 4);
    p.ws_bytes = kStatusBytes + ctrl_bytes + pub_bytes;
    return p;
}

esa_status launch_split_select(const int8_t *qI, const int8_t *kI, const int32_t *wI, const Shape &s, int K,
                               int32_t *idx, int32_t *cnt, void *ws, const SplitPlan &plan, cudaStream_t st) {
    char *base = static_cast<char *>(ws);
    int32_t *status = reinterpret_cast<int32_t *>(base);
    unsigned *ctrl = reinterpret_cast<unsigned *>(base + kStatusBytes);
    unsigned *pub = ctrl + align256(plan.ctrl_words * 4) / 4;
    void *fn = kernel_ptr(s.D_I);
    if (!ensure_smem(fn, plan.smem)) return ESA_ERR_CUDA;
    long long Tq = s.Tq, Tk = s.Tk, qo = s.q_offset;
    int H_I = s.H_I, chunks = plan.chunks;
    long long wns = wait_limit_ns();
    int extra = debug_extra_arrivals();
    void *args[] = {(void *)&qI, (void *)&kI, (void *)&wI, (void *)&idx, (void *)&cnt, (void *)&Tq,
                    (void *)&Tk, (void *)&qo, (void *)&H_I, (void *)&K, (void *)&chunks, (void *)&ctrl,
                    (void *)&pub, (void *)&status, (void *)&wns, (void *)&extra};
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
