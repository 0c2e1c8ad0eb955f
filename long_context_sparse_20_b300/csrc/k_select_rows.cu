// Top-K selection for many query rows (prefill, chunked prefill).
//
// Method: per query row, the Indexer score against every causal-prefix key
// (no RoPE) and the K best positions, ties to the lower position
// ("超大规模MoE架构中稀疏注意力机制的演进与实践", sections 二.1-二.2; the blockwise
// query loop of "大模型推理架构演进：从稀疏注意力到隐式专家路由", section 2.3,
// without materialising the full score matrix).
//
// Design: one block owns 32 consecutive query rows of one sequence; lane l of
// every warp works for row l, so a row's histogram is only ever touched by
// that row's lanes. kI tiles of 128 keys are staged in shared memory with
// cp.async and broadcast to the 32 lanes; each lane scores its row with dp4a
// (the indexer heads collapse into one int8 vector sum_h w_h qI_h whenever
// that fits int8, which is exact integer algebra). Scores are recomputed on
// every pass instead of being stored:
//   pass 1      a 466-bin log histogram per row (exact below |s| = 16);
//   pass 2..    the bucket holding the K-th score, 512 bins at a time, until
//               the threshold T is exact (one pass for |s| < 2^12);
//   final pass  selected = s > T, or s == T among the first (K - #{s > T})
//               ties in position order; written ascending.
// The threshold form (T, P) — P the position of the last tie taken — is
// also returned so that a later kernel can rebuild the set from scores.
#include "esa_device.cuh"
#include "esa_internal.h"

namespace esa {

namespace {

constexpr int kThreads = 256;
constexpr int kRows = 32;
constexpr int kTK = 128;   // keys per tile
constexpr int kNBR = 512;  // histogram bins per row per level
constexpr int kHStride = kNBR + 1;
constexpr int kHalfR = 233;  // log bins: 16 exact + 27 exponents x 8, +1

__device__ __forceinline__ int rlog_bin(int s) {
    unsigned a = s < 0 ? 0u - (unsigned)s : (unsigned)s;
    int m;
    if (a < 16u) {
        m = (int)a;
    } else {
        int e = 31 - __clz(a);
        m = 16 + (e - 4) * 8 + (int)((a >> (e - 3)) & 7u);
    }
    return s >= 0 ? kHalfR + m : kHalfR - m;
}

__device__ __forceinline__ void rlog_range(int bin, long long &lo, long long &hi) {
    int m = bin >= kHalfR ? bin - kHalfR : kHalfR - bin;
    long long alo, ahi;
    if (m < 16) {
        alo = ahi = m;
    } else {
        int e = 4 + (m - 16) / 8, mant = (m - 16) % 8;
        alo = (long long)(8 + mant) << (e - 3);
        ahi = ((long long)(9 + mant) << (e - 3)) - 1;
    }
    if (bin >= kHalfR) {
        lo = alo;
        hi = ahi;
    } else {
        lo = -ahi;
        hi = -alo;
    }
    if (lo < INT32_MIN) lo = INT32_MIN;
    if (hi > INT32_MAX) hi = INT32_MAX;
}

struct RowState {
    long long vlo[kRows], vhi[kRows];
    long long n[kRows];
    int T[kRows];
    int P[kRows];
    unsigned need[kRows];   // ties at T to take
    unsigned above[kRows];  // scores above the current bucket
    int shift[kRows];
    int exact[kRows];
    unsigned out[kRows];
    unsigned tie[kRows];
    unsigned mk[8][kRows];
    int any_open;
    int collapsed;
};

template <int DI>
__global__ void __launch_bounds__(kThreads) row_select_kernel(const int8_t *__restrict__ qI,
                                                              const int8_t *__restrict__ kI,
                                                              const int32_t *__restrict__ wI, int32_t *__restrict__ idx,
                                                              int32_t *__restrict__ cnt, int32_t *__restrict__ thr,
                                                              long long B, long long Tq, long long Tk,
                                                              long long q_offset, int H_I, int K, int pos_div,
                                                              int relu, const int32_t *__restrict__ only_flagged,
                                                              int32_t *__restrict__ status, uint32_t *__restrict__ mask,
                                                              long long mask_rows) {
    constexpr int W = DI / 4;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    RowState &rs = *reinterpret_cast<RowState *>(smem_raw);
    unsigned *hist = reinterpret_cast<unsigned *>(smem_raw + align_up(sizeof(RowState)));
    int8_t *ktile = reinterpret_cast<int8_t *>(hist + kRows * kHStride);  // 2 x kTK x DI
    int32_t *qs = reinterpret_cast<int32_t *>(ktile + 2 * kTK * DI);      // [kRows][H_I][W] (+w)

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const long long tiles_per_seq = (Tq + kRows - 1) / kRows;
    const long long L = blockIdx.x;
    const long long b = L % B;
    const long long tile = tiles_per_seq - 1 - L / B;  // heaviest tiles first
    const long long t0 = tile * kRows;
    const long long row0 = b * Tq + t0;
    const int nrows = (int)min((long long)kRows, Tq - t0);
    // rows per query position: pos_div (per-head sets: one row per indexer head)
    const long long nmax = q_offset + (t0 + nrows - 1) / pos_div + 1;  // keys to visit
    // second launch after the tensor-core selection: only the 128-row query
    // tiles that it left (flag 1) are done here
    if (only_flagged && only_flagged[b * ((Tq + 127) / 128) + t0 / 128] == 0) return;

    // ---- prologue: row state and indexer queries
    if (tid < kRows) {
        long long n = tid < nrows ? q_offset + (t0 + tid) / pos_div + 1 : 0;
        rs.n[tid] = n;
        rs.out[tid] = 0;
        rs.tie[tid] = 0;
        rs.above[tid] = 0;
        rs.shift[tid] = 0;
        bool all = n <= K;  // whole prefix kept (also the empty tail rows)
        rs.exact[tid] = all ? 1 : 0;
        rs.T[tid] = INT32_MIN;
        rs.need[tid] = (unsigned)K;
        rs.P[tid] = (int)(n - 1);
    }
    int32_t *wsm = qs + kRows * H_I * W;
    if (tid < H_I) wsm[tid] = wI[tid];
    for (int i = tid; i < kRows * H_I * W; i += kThreads) {
        int r = i / (H_I * W);
        qs[i] = r < nrows ? reinterpret_cast<const int32_t *>(qI + (row0 + r) * (long long)H_I * DI)[i % (H_I * W)]
                          : 0;
    }
    __syncthreads();
    // collapse the indexer heads into q_eff = sum_h w_h qI_h when every
    // component of every row fits int8 (exact: integer algebra); never with
    // the ReLU, which acts on each head's own dot product
    if (tid == 0) rs.collapsed = relu ? 0 : 1;
    __syncthreads();
    {
        bool fits = true;
        for (int i = tid; i < kRows * DI; i += kThreads) {
            int r = i / DI, c = i % DI;
            long long acc = 0;  // 64-bit: any int32 weight
            for (int h = 0; h < H_I; h++)
                acc += (long long)wsm[h] * reinterpret_cast<const int8_t *>(qs + (r * H_I + h) * W)[c];
            fits = fits && acc >= -128 && acc <= 127;
        }
        if (!__syncthreads_and(fits)) {
            if (tid == 0) rs.collapsed = 0;
        }
    }
    __syncthreads();
    uint32_t qr[W];
    const bool collapsed = rs.collapsed != 0;
    if (collapsed) {
#pragma unroll
        for (int c = 0; c < W; c++) {
            int v[4];
#pragma unroll
            for (int e = 0; e < 4; e++) {
                unsigned acc = 0;  // exact modulo 2^32; the value fits int8 here
                for (int h = 0; h < H_I; h++)
                    acc += (unsigned)wsm[h] *
                           (unsigned)(int)reinterpret_cast<const int8_t *>(qs + (lane * H_I + h) * W)[4 * c + e];
                v[e] = (int)acc;
            }
            qr[c] = (uint32_t)(v[0] & 255) | ((uint32_t)(v[1] & 255) << 8) | ((uint32_t)(v[2] & 255) << 16) |
                    ((uint32_t)(v[3] & 255) << 24);
        }
    }

    auto score = [&](const int8_t *krow) -> int {
        const uint4 *kp = reinterpret_cast<const uint4 *>(krow);
        uint32_t kw[W];
#pragma unroll
        for (int c = 0; c < W / 4; c++) {
            uint4 v = kp[c];
            kw[4 * c] = v.x;
            kw[4 * c + 1] = v.y;
            kw[4 * c + 2] = v.z;
            kw[4 * c + 3] = v.w;
        }
        if (collapsed) {
            int d = 0;
#pragma unroll
            for (int c = 0; c < W; c++) d = __dp4a((int)qr[c], (int)kw[c], d);
            return d;
        }
        unsigned acc = 0;
        for (int h = 0; h < H_I; h++) {
            const int32_t *qh = qs + (lane * H_I + h) * W;
            int d = 0;
#pragma unroll
            for (int c = 0; c < W; c++) d = __dp4a(qh[c], (int)kw[c], d);
            acc += (unsigned)wsm[h] * (unsigned)(relu ? max(d, 0) : d);
        }
        return (int)acc;
    };

    const int8_t *kseq = kI + b * Tk * DI;
    const int ntiles = (int)((nmax + kTK - 1) / kTK);
    auto load_tile = [&](int ti, int buf) {
        const long long j0 = (long long)ti * kTK;
        constexpr int chunks = kTK * DI / 16;
        uint32_t dst = smem_u32(ktile + buf * kTK * DI);
        for (int c = tid; c < chunks; c += kThreads) {
            long long j = j0 + (c * 16) / DI;
            bool valid = j < nmax;
            cp_async16_zfill(dst + c * 16, kseq + (valid ? j0 * DI + c * 16 : 0), valid);
        }
        cp_async_commit();
    };

    // one sweep over all key tiles; `op` consumes (key j, score s, row lane)
    auto sweep = [&](auto &&op, auto &&after_tile) {
        load_tile(0, 0);
        for (int ti = 0; ti < ntiles; ti++) {
            if (ti + 1 < ntiles) {
                load_tile(ti + 1, (ti + 1) & 1);
                cp_async_wait<1>();
            } else {
                cp_async_wait<0>();
            }
            __syncthreads();
            const int8_t *kt = ktile + (ti & 1) * kTK * DI;
            const long long j0 = (long long)ti * kTK + warp * 16;
            op(kt + warp * 16 * DI, j0);
            __syncthreads();
            after_tile(ti);
        }
    };

    // ---- histogram levels until every row has an exact threshold (a log
    // level and at most three 512-bin levels resolve any int32 score)
    for (int level = 1;; level++) {
        if (tid == 0) {
            int open = 0;
            for (int r = 0; r < kRows; r++) open |= !rs.exact[r];
            rs.any_open = open;
        }
        __syncthreads();
        if (!rs.any_open) break;
        if (level > 6) {  // consistency check; never reached
            if (tid == 0) set_status(status, ESA_ERR_INTERNAL);
            return;
        }
        for (int i = tid; i < kRows * kHStride; i += kThreads) hist[i] = 0u;
        __syncthreads();
        const bool mine_open = !rs.exact[lane];
        const long long my_n = rs.n[lane];
        const long long vlo = rs.vlo[lane], vhi = rs.vhi[lane];
        const int sh = rs.shift[lane];
        unsigned *hrow = hist + lane * kHStride;
        sweep(
            [&](const int8_t *kt, long long j0) {
                if (!mine_open) return;
#pragma unroll 4
                for (int k = 0; k < 16; k++) {
                    long long j = j0 + k;
                    if (j >= my_n) break;
                    int s = score(kt + k * DI);
                    if (level == 1) {
                        atomicAdd(hrow + rlog_bin(s), 1u);
                    } else if (s >= vlo && s <= vhi) {
                        atomicAdd(hrow + (int)(((long long)s - vlo) >> sh), 1u);
                    }
                }
            },
            [](int) {});
        // per-row crossing: warp w serves rows w, w+8, w+16, w+24
        for (int r = warp; r < kRows; r += 8) {
            if (rs.exact[r]) continue;
            const unsigned need = (unsigned)K - rs.above[r];
            const unsigned *h = hist + r * kHStride;
            int b0 = lane * (kNBR / 32), b1 = b0 + kNBR / 32;
            unsigned seg = 0;
            for (int v = b0; v < b1; v++) seg += h[v];
            unsigned x = seg;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                unsigned y = __shfl_down_sync(0xffffffffu, x, d);
                if (lane + d < 32) x += y;
            }
            unsigned excl = x - seg;
            int found = -1;
            unsigned above_in = 0;
            if (excl < need && need <= x) {
                unsigned a = excl;
                for (int v = b1 - 1; v >= b0; v--) {
                    if (a + h[v] >= need) {
                        found = v;
                        above_in = a;
                        break;
                    }
                    a += h[v];
                }
            }
            unsigned fl = __ballot_sync(0xffffffffu, found >= 0);
            if (fl == 0u) {  // consistency check; never reached
                if (lane == 0) {
                    set_status(status, ESA_ERR_INTERNAL);
                    rs.exact[r] = 1;
                }
                continue;
            }
            int src = __ffs(fl) - 1;
            found = __shfl_sync(0xffffffffu, found, src);
            above_in = __shfl_sync(0xffffffffu, above_in, src);
            if (lane == 0) {
                long long lo, hi;
                if (level == 1) {
                    rlog_range(found, lo, hi);
                } else {
                    lo = rs.vlo[r] + ((long long)found << rs.shift[r]);
                    hi = min(rs.vhi[r], lo + (1ll << rs.shift[r]) - 1);
                }
                rs.above[r] += above_in;
                if (lo == hi) {
                    rs.exact[r] = 1;
                    rs.T[r] = (int)lo;
                    rs.need[r] = (unsigned)K - rs.above[r];
                } else {
                    int s2 = 0;
                    while (((hi - lo) >> s2) >= kNBR) s2++;
                    rs.vlo[r] = lo;
                    rs.vhi[r] = hi;
                    rs.shift[r] = s2;
                }
            }
        }
        __syncthreads();
    }

    // ---- final pass: ordered write of the selected positions
    const bool write_idx = idx != nullptr;
    {
        const long long my_n = rs.n[lane];
        const int T = rs.T[lane];
        sweep(
            [&](const int8_t *kt, long long j0) {
                unsigned gtm = 0, eqm = 0;
#pragma unroll 4
                for (int k = 0; k < 16; k++) {
                    long long j = j0 + k;
                    if (j >= my_n) break;
                    int s = score(kt + k * DI);
                    gtm |= (unsigned)(s > T) << k;
                    eqm |= (unsigned)(s == T) << k;
                }
                rs.mk[warp][lane] = gtm | (eqm << 16);
            },
            [&](int ti) {
                // thread (warp w, lane r): row r's 16-key word w of this tile
                const int r = lane, w = warp;
                const unsigned need = rs.need[r];
                unsigned tie = rs.tie[r], out = rs.out[r];
                unsigned sel = 0, take_bits_hi = 0;
                for (int w2 = 0; w2 <= w; w2++) {
                    unsigned m = rs.mk[w2][r];
                    unsigned g = m & 0xffffu, e = m >> 16;
                    unsigned ne = __popc(e);
                    unsigned take = tie >= need ? 0u : min(ne, need - tie);
                    unsigned tb = 0, ee = e;
                    for (unsigned i = 0; i < take; i++) {
                        unsigned lowbit = ee & (0u - ee);
                        tb |= lowbit;
                        ee ^= lowbit;
                    }
                    if (w2 < w) {
                        out += __popc(g) + take;
                    } else {
                        sel = g | tb;
                        if (take > 0 && tie + take == need) take_bits_hi = 31 - __clz(tb);
                        else take_bits_hi = 0xffffffffu;
                    }
                    tie += ne;
                }
                const long long tkey = (long long)ti * kTK + w * 16;
                if (take_bits_hi != 0xffffffffu) rs.P[r] = (int)(tkey + take_bits_hi);
                if (mask && r < nrows)  // the row's bitmask (word-major), 16 keys at a time
                    reinterpret_cast<uint16_t *>(mask)[((tkey >> 5) * mask_rows + row0 + r) * 2 + ((tkey >> 4) & 1)] =
                        (uint16_t)sel;
                if (write_idx && r < nrows) {
                    int32_t *orow = idx + (row0 + r) * (long long)K;
                    unsigned sb = sel;
                    while (sb) {
                        int bit = __ffs(sb) - 1;
                        sb &= sb - 1;
                        if (out < (unsigned)K) orow[out] = (int32_t)(tkey + bit);
                        else set_status(status, ESA_ERR_INTERNAL);
                        out++;
                    }
                }
                __syncthreads();
                if (w == 7) {  // advance the row's running counts by the whole tile
                    unsigned o = rs.out[r], te = rs.tie[r];
                    for (int w2 = 0; w2 < 8; w2++) {
                        unsigned m = rs.mk[w2][r];
                        unsigned ne = __popc(m >> 16);
                        unsigned take = te >= need ? 0u : min(ne, need - te);
                        o += __popc(m & 0xffffu) + take;
                        te += ne;
                    }
                    rs.out[r] = o;
                    rs.tie[r] = te;
                }
                __syncthreads();
            });
    }

    // ---- counts, padding and threshold form
    for (int r = warp; r < nrows; r += 8) {
        const long long n = rs.n[r];
        const int c = (int)min((long long)K, n);
        if (write_idx) {
            int32_t *orow = idx + (row0 + r) * (long long)K;
            for (int i = c + lane; i < K; i += 32) orow[i] = -1;
            if (lane == 0) cnt[row0 + r] = c;
        }
        if (thr && lane == 0) {
            thr[2 * (row0 + r)] = rs.T[r];
            thr[2 * (row0 + r) + 1] = rs.P[r];
        }
    }
}

size_t row_smem(int DI, int H_I) {
    return align_up(sizeof(RowState)) + (size_t)kRows * kHStride * 4 + 2 * (size_t)kTK * DI +
           (size_t)kRows * H_I * (DI / 4) * 4 + 64;
}

void *row_kernel(int DI) {
    switch (DI) {
        case 16: return (void *)row_select_kernel<16>;
        case 32: return (void *)row_select_kernel<32>;
        case 64: return (void *)row_select_kernel<64>;
        default: return (void *)row_select_kernel<128>;
    }
}

}  // namespace

esa_status launch_rows_dp4a(const int8_t *qI, const int8_t *kI, const int32_t *wI, const Shape &s, int K,
                            int32_t *idx, int32_t *cnt, int32_t *thr, const int32_t *only_flagged, int32_t *status,
                            cudaStream_t st, uint32_t *mask) {
    long long tiles = s.B * ((s.Tq + kRows - 1) / kRows);
    if (tiles == 0) return ESA_OK;
    size_t smem = row_smem(s.D_I, s.H_I);
    void *fn = row_kernel(s.D_I);
    if (!ensure_smem(fn, smem)) return ESA_ERR_CUDA;
    long long B = s.B, Tq = s.Tq, Tk = s.Tk, qo = s.q_offset;
    int H_I = s.H_I, pos_div = s.pos_div, relu = relu_of(s) ? 1 : 0;
    long long mask_rows = s.B * s.Tq;
    void *args[] = {(void *)&qI,  (void *)&kI,      (void *)&wI,   (void *)&idx, (void *)&cnt,
                    (void *)&thr, (void *)&B,       (void *)&Tq,   (void *)&Tk,  (void *)&qo,
                    (void *)&H_I, (void *)&K,       (void *)&pos_div, (void *)&relu,
                    (void *)&only_flagged, (void *)&status, (void *)&mask, (void *)&mask_rows};
    cudaError_t e = cudaLaunchKernel(fn, dim3((unsigned)tiles), dim3(kThreads), args, smem, st);
    return e == cudaSuccess ? ESA_OK : ESA_ERR_CUDA;
}

}  // namespace esa
