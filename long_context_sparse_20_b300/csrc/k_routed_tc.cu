// Per-head routed attention on the fifth-generation tensor cores (tcgen05,
// accumulators in tensor memory).
//
// Method ("Elastic Attention：动态路由优化大模型长文本处理", sections 2.2 and
// 3.1): every head runs either full causal attention or the sparse path,
// decided per head, inside one launch. Sparse heads attend to exactly the
// Top-K positions of the Indexer ("超大规模MoE架构中稀疏注意力机制的演进与实践",
// sections 二.1-二.3) and are mixed with the linear branch by the gate.
//
// Design: one CTA per (sequence, head, 128-row query tile); thread r owns
// query row r, which is also tensor-memory lane r. Keys are visited in
// 64-key tiles, K/V (and, for sparse heads, the int8 indexer keys) staged by
// cp.async in a ring of shared-memory slots in the tensor cores' no-swizzle
// core-matrix layout. One thread issues the MMAs:
//   S  = Q K^T                       bf16 x bf16 -> fp32 (TMEM, 3 buffers)
//   SI = q_eff kI^T                  fp16 x fp16 -> fp32 (TMEM, 2 buffers):
//        the indexer scores, exact — q_eff = sum_h w_h qI_h and kI are small
//        integers, exact in fp16, and every partial sum stays below 2^24;
//   O += P_hi V + P_lo V             P read from tensor memory
// The softmax threads read S (and SI) from tensor memory, mask — causal for
// full heads; for sparse heads the threshold form of the Top-K set
// (s > T, or s == T and j <= P, which is exactly the K best positions with
// ties to the lower position) — and write P as a bf16 hi + lo pair over the
// consumed S columns. The running max is only raised when it grows by more
// than 2^8, so O (in tensor memory) is rescaled rarely. A CTA whose
// collapsed indexer query is not exact in fp16 computes its mask scores
// with dp4a instead.
#include <cuda_fp16.h>

#include <algorithm>

#include "esa_device.cuh"
#include "esa_internal.h"

namespace esa {

namespace {

constexpr int kThreads = 128;
constexpr int kBM = 128;  // query rows per CTA (tensor-memory lanes)
constexpr int kBN = 64;   // keys per tile
constexpr uint32_t kColS = 0;     // 3 x 64 columns: scores, then P (hi 32 + lo 32)
constexpr uint32_t kColSI = 192;  // 2 x 64 columns: indexer scores
constexpr uint32_t kColO = 320;   // D columns: output accumulator
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleLog2 = 8.f;  // raise the running max only past 2^8 growth

template <int D, int DI>
struct Lay {
    static constexpr int Q = 0;                          // kBM x D bf16
    static constexpr int QE = Q + kBM * D * 2;           // kBM x DI fp16 (collapsed indexer query)
    static constexpr int KH = QE + kBM * DI * 2;         // 2 x kBN x DI fp16 (indexer keys)
    static constexpr int RING = KH + 2 * kBN * DI * 2;
    static constexpr int SK = 0, SV = kBN * D * 2, SKI = 2 * kBN * D * 2;  // within a slot
    static constexpr int SLOT = SKI + kBN * DI;
    static constexpr int SLOTS = RING + 4 * SLOT <= 220 * 1024 ? 4 : 3;
    static constexpr int TOTAL = RING + SLOTS * SLOT;
};

struct TcArgs {
    const uint16_t *q, *k, *v, *lin;
    const int8_t *qI, *kI;
    const int32_t *wI;
    const uint8_t *route;
    const int32_t *thr;
    const float *g;
    float *out;
    int32_t *status;
    long long B, Tq, Tk, q_offset, wait_ns;
    int Hq, Hkv, H_I;
    float scale_log2;
};

__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}
// instruction descriptor: fp32 accumulate, M = 128; ab = 1 for bf16, 0 for fp16
__host__ __device__ constexpr uint32_t idesc(int N, uint32_t ab, uint32_t b_mn_major) {
    return (1u << 4) | (ab << 7) | (ab << 10) | (b_mn_major << 16) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(kBM >> 4) << 24);
}
__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
        "l"(a), "l"(b), "r"(id), "r"(acc)
        : "memory");
}
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t id, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(
            d),
        "r"(a_tmem), "l"(b), "r"(id), "r"(acc)
        : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// 32 consecutive columns of this warp's 32 lanes
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t *r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
        "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
          "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t *r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
        "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
        "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
        "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

template <int D, int DI>
__global__ void __launch_bounds__(kThreads, 1) routed_tc_kernel(TcArgs a) {
    using L = Lay<D, DI>;
    constexpr int NS = L::SLOTS;
    extern __shared__ __align__(1024) unsigned char smem[];
    __shared__ __align__(8) unsigned long long bar_s[3], bar_pv;
    __shared__ uint32_t tmem_base;
    __shared__ int flag_bad;

    const int tid = threadIdx.x, warp = tid >> 5;
    const long long nqt = (a.Tq + kBM - 1) / kBM;
    // query tiles of one (sequence, head) are consecutive, longest prefixes
    // first: the CTAs running together share that head's K/V through L2
    long long bid = blockIdx.x;
    const long long qt = nqt - 1 - bid % nqt;
    bid /= nqt;
    const int h = (int)(bid % a.Hq);
    const long long b = bid / a.Hq;
    const long long t0 = qt * kBM;
    const int rows = (int)min((long long)kBM, a.Tq - t0);
    const int kvh = h / (a.Hq / a.Hkv);
    const bool sparse = a.route[b * a.Hq + h] != 0;
    const long long row0 = b * a.Tq + t0;
    const long long kend = a.q_offset + t0 + rows;  // keys 0..kend-1 are visible to some row
    const int nt = (int)((kend + kBN - 1) / kBN);
    const long long pos = tid < rows ? a.q_offset + t0 + tid : -1;  // this thread's query position

    const uint32_t sbase = smem_u32(smem);
    const uint16_t *kb = a.k + (b * a.Tk * a.Hkv + kvh) * (long long)D;
    const uint16_t *vb = a.v + (b * a.Tk * a.Hkv + kvh) * (long long)D;
    const long long kst = (long long)a.Hkv * D;
    const int8_t *kib = a.kI + b * a.Tk * (long long)DI;

    // ---- tensor memory and barriers
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (tid == 0) {
        for (int i = 0; i < 3; i++) mbar_init(smem_u32(&bar_s[i]), 1);
        mbar_init(smem_u32(&bar_pv), 1);
        mbar_fence_init();
        flag_bad = 0;
    }

    // ---- Q tile (zero rows past the sequence), one cp.async group
    for (int i = tid; i < kBM * (D / 8); i += kThreads) {
        const int r = i / (D / 8), c = i % (D / 8);
        const bool ok = r < rows;
        cp_async16_zfill(sbase + L::Q + (r / 8) * (D / 8 * 128) + c * 128 + (r % 8) * 16,
                         a.q + ((row0 + (ok ? r : 0)) * a.Hq + h) * (long long)D + c * 8, ok);
    }
    cp_async_commit();
    // key tile t -> ring slot t % NS (zero-filled past kend); one group per tile
    auto load_tile = [&](int t) {
        const uint32_t sl = sbase + L::RING + (t % NS) * L::SLOT;
        const long long j0 = (long long)t * kBN;
        for (int i = tid; i < kBN * (D / 8); i += kThreads) {
            const int kk = i / (D / 8), c = i % (D / 8);
            const long long j = j0 + kk;
            const bool ok = j < kend;
            const long long js = ok ? j : 0;
            cp_async16_zfill(sl + L::SK + (kk / 8) * (D / 8 * 128) + c * 128 + (kk % 8) * 16, kb + js * kst + c * 8, ok);
            cp_async16_zfill(sl + L::SV + c * (kBN / 8 * 128) + (kk / 8) * 128 + (kk % 8) * 16, vb + js * kst + c * 8, ok);
        }
        if (sparse) {
            for (int i = tid; i < kBN * DI / 16; i += kThreads) {
                const long long j = j0 + (i * 16) / DI;
                const bool ok = j < kend;
                cp_async16_zfill(sl + L::SKI + i * 16, kib + (ok ? j0 * DI + i * 16 : 0), ok);
            }
        }
    };
    for (int t = 0; t < NS - 1; t++) {
        if (t < nt) load_tile(t);
        cp_async_commit();
    }

    // ---- sparse heads: threshold form and the collapsed indexer query
    float Tf = 0.f;
    int Tint = 0, Pp = -1;
    bool exact = true;
    if (sparse) {
        if (tid < rows) {
            Tint = a.thr[2 * (row0 + tid)];
            Pp = a.thr[2 * (row0 + tid) + 1];
        }
        Tf = (float)Tint;
        long long absum = 0;
        bool fits = true;
        const int8_t *qrow = a.qI + (row0 + (tid < rows ? tid : 0)) * (long long)a.H_I * DI;
        for (int c0 = 0; c0 < DI; c0 += 8) {
            int acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            for (int hh = 0; hh < a.H_I; hh++) {
                const int wv = a.wI[hh];
                const uint2 raw = *reinterpret_cast<const uint2 *>(qrow + hh * DI + c0);
#pragma unroll
                for (int e = 0; e < 8; e++) {
                    const int8_t qv = (int8_t)(((e < 4 ? raw.x : raw.y) >> (8 * (e & 3))) & 0xFF);
                    acc[e] += wv * (int)qv;
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
            if (tid >= rows) pk[0] = pk[1] = pk[2] = pk[3] = 0u;
            *reinterpret_cast<uint4 *>(smem + L::QE + (tid / 8) * (DI / 8 * 128) + (c0 / 8) * 128 + (tid % 8) * 16) =
                make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
        // every partial sum of q_eff . kI (|kI| <= 128) must stay below 2^24
        fits = fits && absum * 128 < (1ll << 24);
        exact = __syncthreads_and(fits || tid >= rows) != 0;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;
    const uint32_t lane_base = (uint32_t)(32 * warp) << 16;

    // convert tile t's raw indexer keys to fp16 into KH buffer t % 2
    auto convert_ki = [&](int t) {
        const unsigned char *raw = smem + L::RING + (t % NS) * L::SLOT + L::SKI;
        unsigned char *dst = smem + L::KH + (t % 2) * (kBN * DI * 2);
        for (int i = tid; i < kBN * DI / 8; i += kThreads) {
            const int kk = i / (DI / 8), c8 = i % (DI / 8);
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
    };
    // one thread issues S (and SI) for tile t, then commits to bar_s[t % 3]
    auto issue_scores = [&](int t) {
        const uint32_t sl = sbase + L::RING + (t % NS) * L::SLOT;
        constexpr uint32_t id_s = idesc(kBN, 1u, 0u);
#pragma unroll
        for (int kk = 0; kk < D / 16; kk++)
            mma_ss(tmem + kColS + (t % 3) * 64, sdesc(sbase + L::Q + kk * 256, 128, D / 8 * 128),
                   sdesc(sl + L::SK + kk * 256, 128, D / 8 * 128), id_s, kk > 0);
        if (sparse && exact) {
            constexpr uint32_t id_i = idesc(kBN, 0u, 0u);
            const uint32_t kh = sbase + L::KH + (t % 2) * (kBN * DI * 2);
#pragma unroll
            for (int kk = 0; kk < DI / 16; kk++)
                mma_ss(tmem + kColSI + (t % 2) * 64, sdesc(sbase + L::QE + kk * 256, 128, DI / 8 * 128),
                       sdesc(kh + kk * 256, 128, DI / 8 * 128), id_i, kk > 0);
        }
        mma_commit(smem_u32(&bar_s[t % 3]));
    };

    // ---- prologue: Q, tile 0 -> scores of tile 0
    bool bad = false;
    cp_async_wait_dyn(NS - 2);  // Q and tile 0 have landed (this thread's copies)
    if (sparse && exact && nt > 0) {
        __syncthreads();  // ... and everyone's, before converting them
        convert_ki(0);
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && nt > 0) {
        tc_fence_after();
        issue_scores(0);
    }

    float m_used = -INFINITY, l = 0.f;
    for (int j = 0; j < nt; j++) {
        // A. tile j+1 landed: its scores go to the tensor cores while this
        //    tile's softmax runs
        if (j + 1 < nt) {
            cp_async_wait_dyn(NS - 3);  // tile t is cp.async group t + 1
            if (sparse && exact) {
                __syncthreads();  // every thread's copies of tile j+1 have landed
                convert_ki(j + 1);
            }
            fence_async_smem();
            tc_fence_before();
            __syncthreads();
            if (tid == 0) {
                tc_fence_after();
                issue_scores(j + 1);
            }
        }
        // B. scores of tile j
        if (!mbar_wait_bounded(smem_u32(&bar_s[j % 3]), (unsigned)(j / 3) & 1u, a.wait_ns)) bad = true;
        tc_fence_after();
        // C. softmax of tile j -> P (hi, lo) over the consumed S columns
        uint32_t sr[64];
        tmem_ld32(tmem + lane_base + kColS + (j % 3) * 64, sr);
        tmem_ld32(tmem + lane_base + kColS + (j % 3) * 64 + 32, sr + 32);
        const long long j0 = (long long)j * kBN;
        // keep bit c: key j0+c passes the Top-K test (sparse heads)
        uint64_t keep = ~0ull;
        if (sparse && exact) {
#pragma unroll
            for (int half = 0; half < 2; half++) {
                uint32_t ir[32];
                tmem_ld32(tmem + lane_base + kColSI + (j % 2) * 64 + half * 32, ir);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < 32; c++) {
                    const float si = __uint_as_float(ir[c]);
                    const bool sel = si > Tf || (si == Tf && j0 + half * 32 + c <= Pp);
                    if (!sel) keep &= ~(1ull << (half * 32 + c));
                }
            }
        } else if (sparse) {
            // exact integer mask scores with dp4a (collapsed query not exact in fp16)
            const unsigned char *raw = smem + L::RING + (j % NS) * L::SLOT + L::SKI;
            const int8_t *qrow = a.qI + (row0 + (tid < rows ? tid : 0)) * (long long)a.H_I * DI;
            for (int c = 0; c < 64; c++) {
                unsigned acc = 0;
                for (int hh = 0; hh < a.H_I; hh++) {
                    int d = 0;
#pragma unroll
                    for (int w4 = 0; w4 < DI / 4; w4++)
                        d = __dp4a(reinterpret_cast<const int *>(qrow + hh * DI)[w4],
                                   reinterpret_cast<const int *>(raw + c * DI)[w4], d);
                    acc += (unsigned)a.wI[hh] * (unsigned)d;
                }
                const int si = (int)acc;
                if (!(si > Tint || (si == Tint && j0 + c <= Pp))) keep &= ~(1ull << c);
            }
        }
        tmem_wait_ld();
        // causal: key j0+c is visible to this row iff c <= pos - j0
        const int lim = (int)max(-1ll, min(64ll, pos - j0));
        float mt = -INFINITY;
#pragma unroll
        for (int c = 0; c < 64; c++) {
            const bool valid = c <= lim && ((keep >> c) & 1ull);
            const float xv = valid ? __uint_as_float(sr[c]) * a.scale_log2 : -INFINITY;
            sr[c] = __float_as_uint(xv);
            mt = fmaxf(mt, xv);
        }
        float corr = 1.f;
        bool rescale = false;
        if (mt > m_used + kRescaleLog2 || (m_used == -INFINITY && mt > -INFINITY)) {
            rescale = m_used != -INFINITY;  // O is still zero before the first kept key
            corr = rescale ? exp2f(m_used - mt) : 1.f;
            l *= corr;
            m_used = mt;
        }
        const float mu = m_used == -INFINITY ? 0.f : m_used;
        uint32_t phi[32], plo[32];
        float ls = 0.f;
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
            const float p0 = exp2f(__uint_as_float(sr[c]) - mu), p1 = exp2f(__uint_as_float(sr[c + 1]) - mu);
            ls += p0 + p1;
            const uint32_t hw = pack_bf16(p0, p1);
            phi[c / 2] = hw;
            plo[c / 2] = pack_bf16(p0 - bf16lo(hw), p1 - bf16hi(hw));
        }
        l += ls;
        tmem_st32(tmem + lane_base + kColS + (j % 3) * 64, phi);
        tmem_st32(tmem + lane_base + kColS + (j % 3) * 64 + 32, plo);
        tmem_wait_st();
        // D. the previous tile's P V has finished: O is stable, its slot is free
        if (j > 0 && !mbar_wait_bounded(smem_u32(&bar_pv), (unsigned)(j - 1) & 1u, a.wait_ns)) bad = true;
        tc_fence_after();
        // E. rescale O rows whose running max was raised (warp-wide: tensor
        //    memory access is collective)
        if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t o_raw[32];
                tmem_ld32(tmem + lane_base + kColO + c0, o_raw);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; e++) o_raw[e] = __float_as_uint(__uint_as_float(o_raw[e]) * corr);
                tmem_st32(tmem + lane_base + kColO + c0, o_raw);
            }
            tmem_wait_st();
        }
        // F. the slot of tile j-1 is free (its S and P V are done): load tile j-1+NS
        if (j - 1 + NS < nt) load_tile(j - 1 + NS);
        cp_async_commit();
        // G. P V of tile j
        tc_fence_before();
        if (__syncthreads_or(bad)) {
            // give up: wait (bounded) for the tensor cores, free tensor memory
            if (tid == 0) {
                set_status(a.status, ESA_ERR_TIMEOUT);
                if (j > 0) mbar_wait_bounded(smem_u32(&bar_pv), (unsigned)(j - 1) & 1u, a.wait_ns);
                if (j + 1 < nt) mbar_wait_bounded(smem_u32(&bar_s[(j + 1) % 3]), (unsigned)((j + 1) / 3) & 1u, a.wait_ns);
            }
            cp_async_wait<0>();
            tc_fence_before();
            __syncthreads();
            if (warp == 0) {
                tc_fence_after();
                asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
            }
            return;
        }
        if (tid == 0) {
            tc_fence_after();
            const uint32_t sl = sbase + L::RING + (j % NS) * L::SLOT;
            constexpr uint32_t id_o = idesc(D, 1u, 1u);
#pragma unroll
            for (int part = 0; part < 2; part++)
#pragma unroll
                for (int kk = 0; kk < kBN / 16; kk++)
                    mma_ts(tmem + kColO, tmem + kColS + (j % 3) * 64 + part * 32 + kk * 8,
                           sdesc(sl + L::SV + kk * 256, 128, kBN / 8 * 128), id_o, (j > 0 || part > 0 || kk > 0));
            mma_commit(smem_u32(&bar_pv));
        }
    }

    // ---- epilogue: O / l, gate mix for sparse heads
    if (nt > 0 && !mbar_wait_bounded(smem_u32(&bar_pv), (unsigned)(nt - 1) & 1u, a.wait_ns)) {
        set_status(a.status, ESA_ERR_TIMEOUT);
        bad = true;
    }
    tc_fence_after();
    const bool gated = sparse && a.g != nullptr && a.lin != nullptr;
    const float gh = gated ? a.g[h] : 1.f, gl = 1.f - gh;
    const long long obase = ((row0 + tid) * a.Hq + h) * (long long)D;
#pragma unroll
    for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t o_raw[32];
        if (nt > 0) {
            tmem_ld32(tmem + lane_base + kColO + c0, o_raw);
            tmem_wait_ld();
        }
        if (tid < rows && !bad) {
            const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
                float4 r = nt > 0 ? make_float4(__uint_as_float(o_raw[e]) * inv, __uint_as_float(o_raw[e + 1]) * inv,
                                                __uint_as_float(o_raw[e + 2]) * inv, __uint_as_float(o_raw[e + 3]) * inv)
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
                if (gated) {
                    const uint2 lw = *reinterpret_cast<const uint2 *>(a.lin + obase + c0 + e);
                    r.x = fmaf(gh, r.x, gl * bf16lo(lw.x));
                    r.y = fmaf(gh, r.y, gl * bf16hi(lw.x));
                    r.z = fmaf(gh, r.z, gl * bf16lo(lw.y));
                    r.w = fmaf(gh, r.w, gl * bf16hi(lw.y));
                }
                *reinterpret_cast<float4 *>(a.out + obase + c0 + e) = r;
            }
        }
    }
    cp_async_wait<0>();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
    }
}

template <int D, int DI>
void *tc_kernel(size_t *smem) {
    *smem = std::max<size_t>(Lay<D, DI>::TOTAL, 117 * 1024);  // one CTA per SM: it holds all of tensor memory
    return (void *)routed_tc_kernel<D, DI>;
}

template <int D>
void *tc_kernel_d(int DI, size_t *smem) {
    switch (DI) {
        case 16: return tc_kernel<D, 16>(smem);
        case 32: return tc_kernel<D, 32>(smem);
        case 64: return tc_kernel<D, 64>(smem);
        default: return tc_kernel<D, 128>(smem);
    }
}

}  // namespace

esa_status launch_routed_tc(const uint16_t *q, const uint16_t *k, const uint16_t *v, const int8_t *qI,
                            const int8_t *kI, const int32_t *wI, const uint8_t *route, const int32_t *thr,
                            const Shape &s, float scale, const float *g, const uint16_t *lin, float *out,
                            int32_t *status, cudaStream_t st) {
    TcArgs a{};
    a.q = q;
    a.k = k;
    a.v = v;
    a.lin = lin;
    a.qI = qI;
    a.kI = kI;
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
    long long blocks = s.B * s.Hq * ((s.Tq + kBM - 1) / kBM);
    if (blocks == 0) return ESA_OK;
    size_t smem = 0;
    void *fn = s.D == 64 ? tc_kernel_d<64>(s.D_I, &smem) : tc_kernel_d<128>(s.D_I, &smem);
    if (!ensure_smem(fn, smem)) return ESA_ERR_CUDA;
    void *args[] = {(void *)&a};
    cudaError_t ce = cudaLaunchKernel(fn, dim3((unsigned)blocks), dim3(kThreads), args, smem, st);
    return ce == cudaSuccess ? ESA_OK : ESA_ERR_CUDA;
}

}  // namespace esa
