// Per-head routed attention on the fifth-generation tensor cores (tcgen05,
// accumulators in tensor memory).
//
// Method ("Elastic Attention：动态路由优化大模型长文本处理", sections 2.2 and
// 3.1): every head runs either full causal attention or the sparse path,
// decided per head, inside one launch. Sparse heads attend to exactly the
// Top-K positions of the Indexer ("超大规模MoE架构中稀疏注意力机制的演进与实践",
// sections 二.1-二.3) and are mixed with the linear branch by the gate.
//
// Design: one CTA per (sequence, head, 128-row query tile); query row r is
// tensor-memory lane r, owned by two threads that split each tile's columns
// (and O's columns) and exchange row maxima and sums. Keys are visited in
// 64-key tiles, K/V (and, for sparse heads, the int8 indexer keys) staged by
// the tensor memory accelerator (TMA: 3-D tensor maps over [tokens, heads,
// D], 128-byte swizzled 64-element panels that are the tensor cores' operand
// layout as loaded) in a ring of shared-memory slots completed on mbarriers.
// One thread issues the TMA copies and the MMAs:
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
#include <algorithm>

#include "esa_device.cuh"
#include "esa_internal.h"
#include "tc_util.cuh"

namespace esa {

namespace {

constexpr int kThreads = 256;  // two threads per query row
constexpr int kBM = 128;       // query rows per CTA (tensor-memory lanes)
constexpr int kBN = 64;   // keys per tile
constexpr uint32_t kColS = 0;     // 3 x 64 columns: scores, then P (hi 32 + lo 32)
constexpr uint32_t kColSI = 192;  // 2 x 64 columns: indexer scores
constexpr uint32_t kColO = 320;   // D columns: output accumulator
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleLog2 = 8.f;  // raise the running max only past 2^8 growth

template <int D, int DI>
struct Lay {
    // 128-byte swizzled operands come in 64-element panels, 1024-byte aligned
    static constexpr int NP = D / 64;                    // panels per row of D elements
    static constexpr int Q = 0;                          // NP x (kBM rows x 128 B) bf16
    static constexpr int QE = Q + kBM * D * 2;           // kBM x DI fp16 (collapsed indexer query)
    static constexpr int KH = QE + kBM * DI * 2;         // 2 x kBN x DI fp16 (indexer keys)
    static constexpr int RING = KH + 2 * kBN * DI * 2;
    static constexpr int SK = 0, SV = kBN * D * 2, SKI = 2 * kBN * D * 2;  // within a slot: K, V panels, raw kI
    static constexpr int SLOT = (SKI + kBN * DI + 1023) / 1024 * 1024;
    static constexpr int SLOTS = RING + 4 * SLOT <= 219 * 1024 ? 4 : 3;
    static constexpr int TOTAL = RING + SLOTS * SLOT + 1024;  // + alignment slack
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
    int relu;  // ReLU on each indexer head's dot product (mask scores on dp4a)
    float scale_log2;
};

template <int D, int DI>
__global__ void __launch_bounds__(kThreads, 1)
    routed_tc_kernel(const __grid_constant__ TcArgs a, const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                     const __grid_constant__ CUtensorMap tm_ki) {
    using L = Lay<D, DI>;
    constexpr int NS = L::SLOTS;
    constexpr int NP = L::NP;
    constexpr int HD = D / 2;    // output columns per thread
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // swizzled panels need 1024-byte alignment
    unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ __align__(8) unsigned long long bar_s[3], bar_pv, bar_full[4], bar_q;
    __shared__ uint32_t tmem_base;
    __shared__ float xmax[2][kThreads];  // per-thread partial row max, by tile parity
    __shared__ float xsum[kThreads];

    // thread = (row quarter, column half, lane): warps w and w+4 share rows
    // 32*(w%4) .. +31 (their tensor-memory lanes) and split the columns
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q4 = warp & 3, hf = warp >> 2;
    const int r = 32 * q4 + lane;  // query row within the tile
    const int partner = tid ^ 128;

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
    const long long pos = r < rows ? a.q_offset + t0 + r : -1;  // this row's query position

    const uint32_t sbase = smem_u32(smem);
    // param-space addresses of the tensor maps (never copies of them)
    const CUtensorMap *mq = &tm_q, *mk = &tm_k, *mv = &tm_v, *mki = &tm_ki;

    // ---- tensor memory and barriers
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    // key tile t -> ring slot t % NS, completed on bar_full[slot] (thread 0
    // issues; rows past the tensor read as zeros, rows past kend are masked)
    auto issue_tile = [&](int t) {
        const int slot = t % NS;
        const uint32_t sl = sbase + L::RING + slot * L::SLOT;
        const uint32_t bar = smem_u32(&bar_full[slot]);
        const int krow = (int)(b * a.Tk + (long long)t * kBN);
        mbar_expect_tx(bar, (unsigned)(2 * kBN * D * 2 + (sparse ? kBN * DI : 0)));
#pragma unroll
        for (int p = 0; p < NP; p++) {
            tma3(sl + L::SK + p * (kBN * 128), mk, p * 64, kvh, krow, bar);
            tma3(sl + L::SV + p * (kBN * 128), mv, p * 64, kvh, krow, bar);
        }
        if (sparse) tma2(sl + L::SKI, mki, 0, krow, bar);
    };
    int issued = -1;  // last tile issued (thread 0)
    if (tid == 0) {
        for (int i = 0; i < 3; i++) mbar_init(smem_u32(&bar_s[i]), 1);
        for (int i = 0; i < NS; i++) mbar_init(smem_u32(&bar_full[i]), 1);
        mbar_init(smem_u32(&bar_pv), 1);
        mbar_init(smem_u32(&bar_q), 1);
        mbar_fence_init();
        // Q tile (rows past the sequence are never written out)
        mbar_expect_tx(smem_u32(&bar_q), (unsigned)(kBM * D * 2));
#pragma unroll
        for (int p = 0; p < NP; p++) tma3(sbase + L::Q + p * (kBM * 128), mq, p * 64, h, (int)row0, smem_u32(&bar_q));
        for (int t = 0; t < NS - 1 && t < nt; t++) {
            issue_tile(t);
            issued = t;
        }
    }

    // ---- sparse heads: threshold form and the collapsed indexer query
    // (each of a row's two threads collapses half of its components)
    float Tf = 0.f;
    int Tint = 0, Pp = -1;
    bool exact = true;
    if (sparse) {
        if (r < rows) {
            Tint = a.thr[2 * (row0 + r)];
            Pp = a.thr[2 * (row0 + r) + 1];
        }
        Tf = (float)Tint;
        long long absum = 0;
        bool fits = true;
        const int8_t *qrow = a.qI + (row0 + (r < rows ? r : 0)) * (long long)a.H_I * DI;
        for (int c0 = hf * (DI / 2); c0 < (hf + 1) * (DI / 2); c0 += 8) {
            long long acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};  // 64-bit: any int32 weight
            for (int hh = 0; hh < a.H_I; hh++) {
                const int wv = a.wI[hh];
                const uint2 raw = *reinterpret_cast<const uint2 *>(qrow + hh * DI + c0);
#pragma unroll
                for (int e = 0; e < 8; e++) {
                    const int8_t qv = (int8_t)(((e < 4 ? raw.x : raw.y) >> (8 * (e & 3))) & 0xFF);
                    acc[e] += (long long)wv * qv;
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
            *reinterpret_cast<uint4 *>(smem + L::QE + (r / 8) * (DI / 8 * 128) + (c0 / 8) * 128 + (r % 8) * 16) =
                make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
        // every partial sum of q_eff . kI (|kI| <= 128) must stay below 2^24:
        // each half of the components below 2^23
        fits = fits && absum * 128 < (1ll << 23);
        exact = __syncthreads_and((fits || r >= rows) && !a.relu) != 0;  // no collapse under the ReLU
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;
    const uint32_t lane_base = (uint32_t)(32 * q4) << 16;

    // convert tile t's raw indexer keys to fp16 into KH buffer t % 2 (eight
    // consecutive lanes write one 128-byte core-matrix row)
    auto convert_ki = [&](int t) {
        const unsigned char *raw = smem + L::RING + (t % NS) * L::SLOT + L::SKI;
        unsigned char *dst = smem + L::KH + (t % 2) * (kBN * DI * 2);
        for (int i = tid; i < kBN * DI / 8; i += kThreads) {
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
    };
    // one thread issues S (and SI) for tile t, then commits to bar_s[t % 3]
    auto issue_scores = [&](int t) {
        const uint32_t sl = sbase + L::RING + (t % NS) * L::SLOT;
        constexpr uint32_t id_s = idesc(kBN, 1u, 0u);
#pragma unroll
        for (int kk = 0; kk < D / 16; kk++)
            mma_ss(tmem + kColS + (t % 3) * 64,
                   sdesc(sbase + L::Q + (kk / 4) * (kBM * 128) + (kk % 4) * 32, 16, 1024, 2),
                   sdesc(sl + L::SK + (kk / 4) * (kBN * 128) + (kk % 4) * 32, 16, 1024, 2), id_s, kk > 0);
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
    if (!mbar_wait_bounded(smem_u32(&bar_q), 0u, a.wait_ns)) bad = true;
    if (nt > 0 && !mbar_wait_bounded(smem_u32(&bar_full[0]), 0u, a.wait_ns)) bad = true;
    if (sparse && exact && nt > 0) convert_ki(0);
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && nt > 0) {
        tc_fence_after();
        issue_scores(0);
    }

    float m_used = -INFINITY, l = 0.f;  // l: this thread's half of the row sum
    for (int j = 0; j < nt; j++) {
        // A. tile j+1 landed: its scores go to the tensor cores while this
        //    tile's softmax runs
        if (j + 1 < nt) {
            if (!mbar_wait_bounded(smem_u32(&bar_full[(j + 1) % NS]), (unsigned)((j + 1) / NS) & 1u, a.wait_ns))
                bad = true;
            if (sparse && exact) convert_ki(j + 1);
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
        // C. softmax of tile j (this thread: keys 32*hf .. +31 of the tile) ->
        //    P (hi, lo) over the consumed S columns
        uint32_t sr[32];
        tmem_ld32(tmem + lane_base + kColS + (j % 3) * 64 + hf * 32, sr);
        const long long j0 = (long long)j * kBN + hf * 32;
        uint32_t keep = 0xffffffffu;  // bit c: key j0+c passes the Top-K test
        if (sparse && exact) {
            uint32_t ir[32];
            tmem_ld32(tmem + lane_base + kColSI + (j % 2) * 64 + hf * 32, ir);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 32; c++) {
                const float si = __uint_as_float(ir[c]);
                if (!(si > Tf || (si == Tf && j0 + c <= Pp))) keep &= ~(1u << c);
            }
        } else if (sparse) {
            // exact integer mask scores with dp4a (collapsed query not exact in fp16)
            const unsigned char *raw = smem + L::RING + (j % NS) * L::SLOT + L::SKI + hf * 32 * DI;
            const int8_t *qrow = a.qI + (row0 + (r < rows ? r : 0)) * (long long)a.H_I * DI;
            for (int c = 0; c < 32; c++) {
                unsigned acc = 0;
                for (int hh = 0; hh < a.H_I; hh++) {
                    int d = 0;
#pragma unroll
                    for (int w4 = 0; w4 < DI / 4; w4++)
                        d = __dp4a(reinterpret_cast<const int *>(qrow + hh * DI)[w4],
                                   reinterpret_cast<const int *>(raw + c * DI)[w4], d);
                    acc += (unsigned)a.wI[hh] * (unsigned)(a.relu ? max(d, 0) : d);
                }
                const int si = (int)acc;
                if (!(si > Tint || (si == Tint && j0 + c <= Pp))) keep &= ~(1u << c);
            }
        }
        tmem_wait_ld();
        // causal: key j0+c is visible to this row iff c <= pos - j0
        const int lim = (int)max(-1ll, min(32ll, pos - j0));
        float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int c = 0; c < 32; c++) {
            const bool valid = c <= lim && ((keep >> c) & 1u);
            const float xv = valid ? __uint_as_float(sr[c]) * a.scale_log2 : -INFINITY;
            sr[c] = __float_as_uint(xv);
            mx4[c & 3] = fmaxf(mx4[c & 3], xv);
        }
        // row max: this half and the partner thread's half
        xmax[j & 1][tid] = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
        pair_sync(q4);
        const float mt = fmaxf(xmax[j & 1][tid], xmax[j & 1][partner]);
        float corr = 1.f;
        bool rescale = false;
        if (mt > m_used + kRescaleLog2 || (m_used == -INFINITY && mt > -INFINITY)) {
            rescale = m_used != -INFINITY;  // O is still zero before the first kept key
            corr = rescale ? ex2_approx(m_used - mt) : 1.f;
            l *= corr;
            m_used = mt;
        }
        const float mu = m_used == -INFINITY ? 0.f : m_used;
        uint32_t phi[16], plo[16];
        float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
            const float p0 = ex2_approx(__uint_as_float(sr[c]) - mu), p1 = ex2_approx(__uint_as_float(sr[c + 1]) - mu);
            ls0 += p0;
            ls1 += p1;
            const uint32_t hw = pack_bf16(p0, p1);
            phi[c / 2] = hw;
            plo[c / 2] = pack_bf16(p0 - bf16lo(hw), p1 - bf16hi(hw));
        }
        l += ls0 + ls1;
        tmem_st16(tmem + lane_base + kColS + (j % 3) * 64 + hf * 16, phi);
        tmem_st16(tmem + lane_base + kColS + (j % 3) * 64 + 32 + hf * 16, plo);
        tmem_wait_st();
        // D. the previous tile's P V has finished: O is stable, its slot is free
        if (j > 0 && !mbar_wait_bounded(smem_u32(&bar_pv), (unsigned)(j - 1) & 1u, a.wait_ns)) bad = true;
        tc_fence_after();
        // E. rescale this thread's half of the O row when the running max was
        //    raised (warp-wide: tensor memory access is collective)
        if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
            for (int c0 = 0; c0 < HD; c0 += 32) {
                uint32_t o_raw[32];
                tmem_ld32(tmem + lane_base + kColO + hf * HD + c0, o_raw);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; e++) o_raw[e] = __float_as_uint(__uint_as_float(o_raw[e]) * corr);
                tmem_st32(tmem + lane_base + kColO + hf * HD + c0, o_raw);
            }
            tmem_wait_st();
        }
        // F. the slot of tile j-1 is free (its S and P V are done): load tile j-1+NS
        if (tid == 0 && j - 1 + NS < nt && !bad) {
            issue_tile(j - 1 + NS);
            issued = j - 1 + NS;
        }
        // G. P V of tile j
        tc_fence_before();
        if (__syncthreads_or(bad)) {
            // give up: wait (bounded) for the tensor cores, free tensor memory
            if (tid == 0) {
                set_status(a.status, ESA_ERR_TIMEOUT);
                if (j > 0) mbar_wait_bounded(smem_u32(&bar_pv), (unsigned)(j - 1) & 1u, a.wait_ns);
                if (j + 1 < nt) mbar_wait_bounded(smem_u32(&bar_s[(j + 1) % 3]), (unsigned)((j + 1) / 3) & 1u, a.wait_ns);
                for (int t = j + 2; t <= issued; t++)  // copies still in flight
                    mbar_wait_bounded(smem_u32(&bar_full[t % NS]), (unsigned)(t / NS) & 1u, a.wait_ns);
            }
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
                           sdesc(sl + L::SV + kk * 2048, kBN * 128, 1024, 2), id_o, (j > 0 || part > 0 || kk > 0));
            mma_commit(smem_u32(&bar_pv));
        }
    }

    // ---- epilogue: O / l (both halves of the row sum), gate mix for sparse heads
    if (nt > 0 && !mbar_wait_bounded(smem_u32(&bar_pv), (unsigned)(nt - 1) & 1u, a.wait_ns)) {
        set_status(a.status, ESA_ERR_TIMEOUT);
        bad = true;
    }
    tc_fence_after();
    xsum[tid] = l;
    pair_sync(q4);
    const float lt = l + xsum[partner];
    const bool gated = sparse && a.g != nullptr && a.lin != nullptr;
    const float gh = gated ? a.g[h] : 1.f, gl = 1.f - gh;
    const long long obase = ((row0 + r) * a.Hq + h) * (long long)D + hf * HD;
#pragma unroll
    for (int c0 = 0; c0 < HD; c0 += 32) {
        uint32_t o_raw[32];
        if (nt > 0) {
            tmem_ld32(tmem + lane_base + kColO + hf * HD + c0, o_raw);
            tmem_wait_ld();
        }
        if (r < rows && !bad) {
            const float inv = lt > 0.f ? 1.f / lt : 0.f;
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
                float4 v4 = nt > 0 ? make_float4(__uint_as_float(o_raw[e]) * inv, __uint_as_float(o_raw[e + 1]) * inv,
                                                 __uint_as_float(o_raw[e + 2]) * inv, __uint_as_float(o_raw[e + 3]) * inv)
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
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
    a.relu = relu_of(s) ? 1 : 0;
    long long blocks = s.B * s.Hq * ((s.Tq + kBM - 1) / kBM);
    if (blocks == 0) return ESA_OK;
    if (s.B * s.Tq >= (1ll << 31) || s.B * s.Tk >= (1ll << 31)) return ESA_ERR_UNSUPPORTED;  // TMA coordinates
    CUtensorMap tq, tk, tv, tki;
    if (!map_rows_heads_d(&tq, q, s.B * s.Tq, s.Hq, s.D, kBM) || !map_rows_heads_d(&tk, k, s.B * s.Tk, s.Hkv, s.D, kBN) ||
        !map_rows_heads_d(&tv, v, s.B * s.Tk, s.Hkv, s.D, kBN) || !map_rows_bytes(&tki, kI, s.B * s.Tk, s.D_I, kBN))
        return ESA_ERR_CUDA;
    size_t smem = 0;
    void *fn = s.D == 64 ? tc_kernel_d<64>(s.D_I, &smem) : tc_kernel_d<128>(s.D_I, &smem);
    if (!ensure_smem(fn, smem)) return ESA_ERR_CUDA;
    void *args[] = {(void *)&a, (void *)&tq, (void *)&tk, (void *)&tv, (void *)&tki};
    cudaError_t ce = cudaLaunchKernel(fn, dim3((unsigned)blocks), dim3(kThreads), args, smem, st);
    return ce == cudaSuccess ? ESA_OK : ESA_ERR_CUDA;
}

}  // namespace esa
