// Attention over gathered keys, with the gate mix fused in the epilogue.
//
// Method: K_sel, V_sel = gather(K, idx), gather(V, idx);
// out = softmax(Q K_sel^T / sqrt(d)) V_sel ("混合注意力架构演进…", section 三;
// the Gated DSA pseudo-code, section 四.1), then final = g*attn + (1-g)*lin
// (Gated DSA page, sections 二.3 and 四.1). The softmax is the streaming
// (online) form, so the full score row never exists anywhere.
//
// Design: one block serves one (query row, key/value head, group of GT query
// heads that share it, split of the index list). The index set of a row is
// shared by all its query heads, so each gathered 256-byte K/V row feeds GT
// heads at once. Rows are gathered with 16-byte cp.async into padded shared
// tiles (bank-conflict-free ldmatrix), two 64-key stages in flight. Q K^T
// and P V run on bf16 warp MMAs (m16n8k16, fp32 accumulation), 16 heads per
// MMA row tile; the warps that share a head tile each score the whole stage
// and split the output columns of P V between them, so a block's partial
// needs no merge across its warps. P stays in registers and enters P V as a
// bf16 hi + lo pair (two MMAs), so the probabilities keep ~16 significant bits.
// Decode rows split the index list over the blocks of one thread-block
// cluster: each block pushes every head's (max, sum, unnormalised output)
// into the shared memory of the block that finalises that head (distributed
// shared memory stores, no round trip), and after one cluster barrier each
// block merges its heads from its own shared memory — no partials in global
// memory. Rows that are not split finish straight from registers.
#include <cooperative_groups.h>

#include <algorithm>
#include <cstdlib>
#include <mutex>
#include <set>
#include <string>
#include <utility>

#include "esa_device.cuh"
#include "esa_internal.h"

namespace cg = cooperative_groups;

namespace esa {

namespace {

constexpr int kThreads = 128;
constexpr int kKeys = 64;  // keys per stage
constexpr int kMaxSplits = 16;  // at most 32: the decode kernel's merge gives each block one lane
constexpr int kIdxWin = 512;  // staged indices (a multiple of kKeys; small enough for 3 blocks per SM)

template <int D>
struct Cfg {
    static constexpr int RS = D + 8;  // padded row stride (bf16 elements)
    static constexpr int TILE = kKeys * RS;
};

struct AttnArgs {
    const uint16_t *q, *k, *v;
    const int32_t *idx, *cnt;
    const float *g;
    const uint16_t *lin;
    float *out, *lse;
    int32_t *status;
    long long Tq, Tk, q_offset;
    int Hq, Hkv, K, hg, splits, kps;
    int nsets;  // index sets per query row (1, or H_I with per-head sets)
    int hs;     // query heads per index set
    int seg;    // heads of one key/value head that share one index set
    int gps;    // head groups per segment
    float scale_log2;
    // split index lists (the decode kernel): the blocks' merged partials and
    // their (max, sum) records in the workspace
    float *xpart;
    unsigned long long *xrec;
    long long wait_ns;
    int extra;  // extra arrivals the barrier waits for (0; > 0 only to test the timeout path)
};

// Variants (one split per index list for the key-split ones):
//  kColSplit  the warps that share a head tile score the whole stage and
//             split P V's output columns (the cluster-split decode path);
//  kKeySplit  (16-head tiles) warp w takes keys 16w..16w+15 of every 64-key
//             stage for all 16 heads with its own online softmax over every
//             output column; the four warps merge (m, l, O) through shared
//             memory at the end: no warp recomputes another's scores;
//  kKeyRows   (at most 8 heads) the same split with the keys as the MMA
//             rows: S^T = K Q^T (16 keys x 8 heads) and O^T = V^T P^T (D x 8
//             heads), P^T's fragments by movmatrix transposes — no padded
//             head rows when a key/value head serves 8 query heads or fewer.
enum { kColSplit = 0, kKeySplit = 1, kKeyRows = 2, kDecode = 3 };
template <int D, int GT, int VAR>
__global__ void __launch_bounds__(kThreads) sparse_attn_kernel(AttnArgs a) {
    constexpr bool KS = VAR == kKeySplit;
    constexpr int RS = Cfg<D>::RS;
    constexpr int HT = GT >= 16 ? GT / 16 : 1;  // head tiles of 16 heads
    constexpr int WPH = 4 / HT;       // warps per head tile: they split the output columns
    constexpr int NT = kKeys / 8;     // n-tiles of 8 keys (every warp scores the whole stage)
    constexpr int DK = D / 16;        // k-steps over the head dim
    constexpr int DW = D / WPH;       // output columns per warp
    constexpr int DNW = DW / 8;       // output n-tiles per warp
    static_assert(DNW % 2 == 0, "pairs of output n-tiles");
    extern __shared__ __align__(16) unsigned char smem_raw[];
    uint16_t *Qs = reinterpret_cast<uint16_t *>(smem_raw);
    uint16_t *KVs = Qs + GT * RS;  // [2 stages][K tile, V tile]
    __shared__ int bad_row;
    __shared__ int kidx[kIdxWin];  // a window of this split's key positions (-1: invalid)

    cg::cluster_group cluster = cg::this_cluster();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int ht = warp % HT, dsl = warp / HT;
    const int g8 = lane >> 2, c4 = lane & 3;

    long long bid = blockIdx.x;
    const int split = (int)(bid % a.splits);  // == rank in the cluster
    bid /= a.splits;
    const int hgi = (int)(bid % a.hg);
    bid /= a.hg;
    const int kvh = (int)(bid % a.Hkv);
    const long long row = bid / a.Hkv;  // b*Tq + t
    const long long b = row / a.Tq, t = row % a.Tq;
    const long long p = a.q_offset + t;
    const int G = a.Hq / a.Hkv;
    // the block's heads lie in one segment: heads of key/value head kvh that
    // share one index set (all G of them with one set per row)
    const int sg = hgi / a.gps, sub = hgi % a.gps;
    const int h0 = kvh * G + sg * a.seg + sub * GT;  // first query head of this block
    const int nh = min(GT, a.seg - sub * GT);
    const long long set = a.nsets > 1 ? row * a.nsets + h0 / a.hs : row;  // idx/cnt row of the block's set

    if (tid == 0) bad_row = 0;
    // ---- Q tile (GT heads x D), zero rows past the group
    {
        const uint16_t *qrow = a.q + (row * a.Hq + h0) * (long long)D;
        constexpr int CH = D / 8;  // 16-byte chunks per head row
        for (int i = tid; i < GT * CH; i += kThreads) {
            int hr = i / CH, ch = i % CH;
            cp_async16_zfill(smem_u32(Qs + hr * RS + ch * 8), qrow + (hr < nh ? hr * D + ch * 8 : 0), hr < nh);
        }
        cp_async_commit();
    }
    pdl_wait();
    int c = a.cnt[set];
    const int cmax = (int)min((long long)a.K, p + 1);
    __syncthreads();
    if (c < 0 || c > cmax) {
        if (tid == 0) bad_row = 1;
        c = 0;
    }
    const int k_begin = split * a.kps;
    const int k_end = min(c, k_begin + a.kps);
    const int nkeys = max(0, k_end - k_begin);

    // this split's indices, staged in windows of kIdxWin (validated here,
    // then read by the gathers of the following stages)
    const int32_t *idx_row = a.idx + set * (long long)a.K + k_begin;
    int win0 = 0;
    auto fill_idx = [&](int base) {
#pragma unroll 8
        for (int i = tid; i < kIdxWin && base + i < nkeys; i += kThreads) {
            int j = __ldg(idx_row + base + i);
            if (j < 0 || j > p) {
                bad_row = 1;
                j = -1;
            }
            kidx[i] = j;
        }
        win0 = base;
        __syncthreads();
    };
    fill_idx(0);
    const uint16_t *kbase = a.k + (b * a.Tk * a.Hkv + kvh) * (long long)D;
    const uint16_t *vbase = a.v + (b * a.Tk * a.Hkv + kvh) * (long long)D;
    const long long kstride = (long long)a.Hkv * D;
    auto load_stage = [&](int st, int kb) {
        uint16_t *Kt = KVs + st * 2 * Cfg<D>::TILE;
        uint16_t *Vt = Kt + Cfg<D>::TILE;
        constexpr int CH = D / 8;
        for (int i = tid; i < kKeys * CH; i += kThreads) {
            int key = i / CH, ch = i % CH;
            int pos = kb + key;  // position within this split
            long long j = pos < nkeys ? kidx[pos - win0] : -1;
            bool valid = j >= 0;
            if (!valid) j = 0;
            cp_async16_zfill(smem_u32(Kt + key * RS + ch * 8), kbase + j * kstride + ch * 8, valid);
            cp_async16_zfill(smem_u32(Vt + key * RS + ch * 8), vbase + j * kstride + ch * 8, valid);
        }
        cp_async_commit();
    };

    const int nstages = (nkeys + kKeys - 1) / kKeys;
    if (nstages > 0) load_stage(0, 0);
    cp_async_wait<0>();  // Q tile (and maybe stage 0)
    __syncthreads();

    if constexpr (VAR == kKeyRows) {
        static_assert(GT == 8, "keys as rows: 8 heads per block");
        constexpr int MT = D / 16;  // O^T m-tiles (16 output columns each)
        // Q^T as the B operand (k = head dim, n = head): lane holds
        // Q[g8][16kk + 2c4 ..] (qb[kk][0]) and Q[g8][16kk + 8 + 2c4 ..] (qb[kk][1])
        uint32_t qb[DK][2];
#pragma unroll
        for (int k2 = 0; k2 < DK / 2; k2++)
            ldmatrix_x4(smem_u32(Qs + (lane & 7) * RS + k2 * 32 + (lane >> 3) * 8), qb[2 * k2][0], qb[2 * k2][1],
                        qb[2 * k2 + 1][0], qb[2 * k2 + 1][1]);
        float ot[MT][4];  // O^T: (column 16mt + g8 (+8), heads 2c4, 2c4+1)
#pragma unroll
        for (int i = 0; i < MT; i++) ot[i][0] = ot[i][1] = ot[i][2] = ot[i][3] = 0.f;
        float km[2] = {-INFINITY, -INFINITY}, kl[2] = {0.f, 0.f};  // heads 2c4, 2c4+1
        const int kb = warp * 16;  // this warp's keys within a stage
        for (int s = 0; s < nstages; s++) {
            if (s + 1 < nstages) {
                if ((s + 1) * kKeys - win0 >= kIdxWin) fill_idx((s + 1) * kKeys);
                load_stage((s + 1) & 1, (s + 1) * kKeys);
                cp_async_wait<1>();
            } else {
                cp_async_wait<0>();
            }
            __syncthreads();
            const uint16_t *Kt = KVs + (s & 1) * 2 * Cfg<D>::TILE;
            const uint16_t *Vt = Kt + Cfg<D>::TILE;
            const int kvalid = min(kKeys, nkeys - s * kKeys);
            // S^T (keys kb+g8, kb+g8+8) x (heads 2c4, 2c4+1)
            float st[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int kk = 0; kk < DK; kk++) {
                uint32_t a0, a1, a2, a3;
                ldmatrix_x4(smem_u32(Kt + (kb + (lane & 15)) * RS + kk * 16 + (lane >> 4) * 8), a0, a1, a2, a3);
                const uint32_t af[4] = {a0, a1, a2, a3};
                mma_bf16_16816(st, af, qb[kk][0], qb[kk][1]);
            }
            const bool in0 = kb + g8 < kvalid, in1 = kb + g8 + 8 < kvalid;
            st[0] = in0 ? st[0] * a.scale_log2 : -INFINITY;
            st[1] = in0 ? st[1] * a.scale_log2 : -INFINITY;
            st[2] = in1 ? st[2] * a.scale_log2 : -INFINITY;
            st[3] = in1 ? st[3] * a.scale_log2 : -INFINITY;
            float mx[2] = {fmaxf(st[0], st[2]), fmaxf(st[1], st[3])};
            float corr[2];
#pragma unroll
            for (int e = 0; e < 2; e++) {
#pragma unroll
                for (int d = 4; d < 32; d <<= 1) mx[e] = fmaxf(mx[e], __shfl_xor_sync(0xffffffffu, mx[e], d));
                const float mnew = fmaxf(km[e], mx[e]);
                const float muse = mnew == -INFINITY ? 0.f : mnew;
                corr[e] = exp2f(km[e] - muse);
                km[e] = mnew;
                mx[e] = muse;
            }
            const float p0 = exp2f(st[0] - mx[0]), p1 = exp2f(st[1] - mx[1]);
            const float p2 = exp2f(st[2] - mx[0]), p3 = exp2f(st[3] - mx[1]);
            float rs[2] = {p0 + p2, p1 + p3};
#pragma unroll
            for (int e = 0; e < 2; e++) {
#pragma unroll
                for (int d = 4; d < 32; d <<= 1) rs[e] += __shfl_xor_sync(0xffffffffu, rs[e], d);
                kl[e] = kl[e] * corr[e] + rs[e];
            }
#pragma unroll
            for (int mt = 0; mt < MT; mt++) {
                ot[mt][0] *= corr[0];
                ot[mt][1] *= corr[1];
                ot[mt][2] *= corr[0];
                ot[mt][3] *= corr[1];
            }
            // P^T as the B operand (k = key, n = head), bf16 hi + lo: the two
            // 8x8 (key, head) blocks of P transposed in registers
            const uint32_t ph0 = pack_bf16(p0, p1), ph1 = pack_bf16(p2, p3);
            const uint32_t pl0 = pack_bf16(p0 - bf16lo(ph0), p1 - bf16hi(ph0));
            const uint32_t pl1 = pack_bf16(p2 - bf16lo(ph1), p3 - bf16hi(ph1));
            const uint32_t bh0 = movmatrix_trans(ph0), bh1 = movmatrix_trans(ph1);
            const uint32_t bl0 = movmatrix_trans(pl0), bl1 = movmatrix_trans(pl1);
#pragma unroll
            for (int mt = 0; mt < MT; mt++) {
                uint32_t a0, a1, a2, a3;  // V^T: (columns 16mt.., keys kb..)
                ldmatrix_x4_trans(smem_u32(Vt + (kb + (lane & 7) + ((lane >> 4) & 1) * 8) * RS + mt * 16 +
                                           ((lane >> 3) & 1) * 8),
                                  a0, a1, a2, a3);
                const uint32_t af[4] = {a0, a1, a2, a3};
                mma_bf16_16816(ot[mt], af, bh0, bh1);
                mma_bf16_16816(ot[mt], af, bl0, bl1);
            }
            __syncthreads();
        }
        if (bad_row) {
            if (tid == 0) set_status(a.status, ESA_ERR_BAD_INDEX);
            return;
        }
        // merge the four warps' (m, l, O) through the idle stage buffers
        float *Om = reinterpret_cast<float *>(KVs);  // [4 warps][8 heads][D]
        float *Mw = Om + 4 * 8 * D, *Lw = Mw + 4 * 8;  // [4][8] each
#pragma unroll
        for (int mt = 0; mt < MT; mt++) {
            Om[(warp * 8 + 2 * c4) * D + mt * 16 + g8] = ot[mt][0];
            Om[(warp * 8 + 2 * c4 + 1) * D + mt * 16 + g8] = ot[mt][1];
            Om[(warp * 8 + 2 * c4) * D + mt * 16 + g8 + 8] = ot[mt][2];
            Om[(warp * 8 + 2 * c4 + 1) * D + mt * 16 + g8 + 8] = ot[mt][3];
        }
        if (g8 == 0) {
            Mw[warp * 8 + 2 * c4] = km[0];
            Mw[warp * 8 + 2 * c4 + 1] = km[1];
            Lw[warp * 8 + 2 * c4] = kl[0];
            Lw[warp * 8 + 2 * c4 + 1] = kl[1];
        }
        __syncthreads();
        const bool gated = a.g != nullptr && a.lin != nullptr;
        constexpr int TPR = kThreads / 8;  // threads per head
        constexpr int CPT = D / TPR;       // columns per thread
        const int hr = tid / TPR, c0 = (tid % TPR) * CPT;
        if (hr < nh) {
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < 4; w++) M = fmaxf(M, Mw[w * 8 + hr]);
            float sw[4], L = 0.f;
#pragma unroll
            for (int w = 0; w < 4; w++) {
                sw[w] = Mw[w * 8 + hr] == -INFINITY ? 0.f : exp2f(Mw[w * 8 + hr] - M);
                L += sw[w] * Lw[w * 8 + hr];
            }
            const int h = h0 + hr;
            const float gh = gated ? a.g[h] : 1.f, inv = L > 0.f ? 1.f / L : 0.f;
            const long long base = (row * a.Hq + h) * (long long)D;
#pragma unroll
            for (int c = 0; c < CPT; c += 2) {
                float v0 = 0.f, v1 = 0.f;
#pragma unroll
                for (int w = 0; w < 4; w++) {
                    const float2 t = *reinterpret_cast<const float2 *>(Om + (w * 8 + hr) * D + c0 + c);
                    v0 = fmaf(sw[w], t.x, v0);
                    v1 = fmaf(sw[w], t.y, v1);
                }
                v0 = L > 0.f ? v0 * inv : 0.f;
                v1 = L > 0.f ? v1 * inv : 0.f;
                if (gated) {
                    const uint32_t lw = *reinterpret_cast<const uint32_t *>(a.lin + base + c0 + c);
                    v0 = fmaf(gh, v0, (1.0f - gh) * bf16lo(lw));
                    v1 = fmaf(gh, v1, (1.0f - gh) * bf16hi(lw));
                }
                *reinterpret_cast<float2 *>(a.out + base + c0 + c) = make_float2(v0, v1);
            }
            if (a.lse && c0 == 0)
                a.lse[row * a.Hq + h] = L > 0.f ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
        }
        return;
    } else {
    uint32_t qf[DK][4];
#pragma unroll
    for (int kk = 0; kk < DK; kk++) {
        int r = ht * 16 + (lane & 15), col = kk * 16 + (lane >> 4) * 8;
        ldmatrix_x4(smem_u32(Qs + r * RS + col), qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
    }

    if constexpr (KS) {
        static_assert(GT == 16, "key split: one 16-head tile per block");
        constexpr int DN = D / 8;  // output n-tiles: every column
        float ok[DN][4];
#pragma unroll
        for (int i = 0; i < DN; i++) ok[i][0] = ok[i][1] = ok[i][2] = ok[i][3] = 0.f;
        float km[2] = {-INFINITY, -INFINITY}, kl[2] = {0.f, 0.f};
        const int kb = warp * 16;  // this warp's keys within a stage
        for (int s = 0; s < nstages; s++) {
            if (s + 1 < nstages) {
                if ((s + 1) * kKeys - win0 >= kIdxWin) fill_idx((s + 1) * kKeys);
                load_stage((s + 1) & 1, (s + 1) * kKeys);
                cp_async_wait<1>();
            } else {
                cp_async_wait<0>();
            }
            __syncthreads();
            const uint16_t *Kt = KVs + (s & 1) * 2 * Cfg<D>::TILE;
            const uint16_t *Vt = Kt + Cfg<D>::TILE;
            const int kvalid = min(kKeys, nkeys - s * kKeys);
            float sc[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; nt++) {
                sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
                for (int kk = 0; kk < DK; kk += 2) {
                    uint32_t b0, b1, b2, b3;
                    const int key = kb + nt * 8 + (lane & 7), col = kk * 16 + (lane >> 3) * 8;
                    ldmatrix_x4(smem_u32(Kt + key * RS + col), b0, b1, b2, b3);
                    mma_bf16_16816(sc[nt], qf[kk], b0, b1);
                    mma_bf16_16816(sc[nt], qf[kk + 1], b2, b3);
                }
            }
            float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
            for (int nt = 0; nt < 2; nt++) {
#pragma unroll
                for (int e = 0; e < 4; e++) {
                    const int key = kb + nt * 8 + 2 * c4 + (e & 1);
                    const float x = key < kvalid ? sc[nt][e] * a.scale_log2 : -INFINITY;
                    sc[nt][e] = x;
                    mx[e >> 1] = fmaxf(mx[e >> 1], x);
                }
            }
            float corr[2];
#pragma unroll
            for (int r = 0; r < 2; r++) {
                mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
                mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
                const float mnew = fmaxf(km[r], mx[r]);
                const float muse = mnew == -INFINITY ? 0.f : mnew;
                corr[r] = exp2f(km[r] - muse);
                km[r] = mnew;
                mx[r] = muse;
            }
            float rs[2] = {0.f, 0.f};
            uint32_t ah[4], al[4];  // P (16 heads x 16 keys) as bf16 hi + lo, A-fragment order
#pragma unroll
            for (int nt = 0; nt < 2; nt++) {
                const float p0 = exp2f(sc[nt][0] - mx[0]), p1 = exp2f(sc[nt][1] - mx[0]);
                const float p2 = exp2f(sc[nt][2] - mx[1]), p3 = exp2f(sc[nt][3] - mx[1]);
                rs[0] += p0 + p1;
                rs[1] += p2 + p3;
                ah[2 * nt] = pack_bf16(p0, p1);
                ah[2 * nt + 1] = pack_bf16(p2, p3);
                al[2 * nt] = pack_bf16(p0 - bf16lo(ah[2 * nt]), p1 - bf16hi(ah[2 * nt]));
                al[2 * nt + 1] = pack_bf16(p2 - bf16lo(ah[2 * nt + 1]), p3 - bf16hi(ah[2 * nt + 1]));
            }
#pragma unroll
            for (int r = 0; r < 2; r++) {
                rs[r] += __shfl_xor_sync(0xffffffffu, rs[r], 1);
                rs[r] += __shfl_xor_sync(0xffffffffu, rs[r], 2);
                kl[r] = kl[r] * corr[r] + rs[r];
            }
#pragma unroll
            for (int dn = 0; dn < DN; dn++) {
                ok[dn][0] *= corr[0];
                ok[dn][1] *= corr[0];
                ok[dn][2] *= corr[1];
                ok[dn][3] *= corr[1];
            }
#pragma unroll
            for (int dn = 0; dn < DN / 2; dn++) {
                uint32_t b0, b1, b2, b3;
                const int key = kb + (lane & 7) + ((lane >> 3) & 1) * 8;
                const int col = dn * 16 + (lane >> 4) * 8;
                ldmatrix_x4_trans(smem_u32(Vt + key * RS + col), b0, b1, b2, b3);
                mma_bf16_16816(ok[2 * dn], ah, b0, b1);
                mma_bf16_16816(ok[2 * dn + 1], ah, b2, b3);
                mma_bf16_16816(ok[2 * dn], al, b0, b1);
                mma_bf16_16816(ok[2 * dn + 1], al, b2, b3);
            }
            __syncthreads();
        }
        // merge the four warps' (m, l, O) through the (now idle) stage buffers
        if (bad_row) {
            if (tid == 0) set_status(a.status, ESA_ERR_BAD_INDEX);
            return;
        }
        float *Om = reinterpret_cast<float *>(KVs);  // [4 warps][16 heads][D]
        float *Mw = Om + 4 * 16 * D, *Lw = Mw + 4 * 16;  // [4][16] each
#pragma unroll
        for (int rr = 0; rr < 2; rr++) {
            const int hr = g8 + rr * 8;
#pragma unroll
            for (int dn = 0; dn < DN; dn++)
                *reinterpret_cast<float2 *>(Om + (warp * 16 + hr) * D + dn * 8 + 2 * c4) =
                    make_float2(ok[dn][2 * rr], ok[dn][2 * rr + 1]);
            if (c4 == 0) {
                Mw[warp * 16 + hr] = km[rr];
                Lw[warp * 16 + hr] = kl[rr];
            }
        }
        __syncthreads();
        const bool gated = a.g != nullptr && a.lin != nullptr;
        constexpr int TPR = kThreads / 16;  // threads per head row
        constexpr int CPT = D / TPR;        // columns per thread
        const int hr = tid / TPR, c0 = (tid % TPR) * CPT;
        if (hr < nh) {
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < 4; w++) M = fmaxf(M, Mw[w * 16 + hr]);
            float sw[4], L = 0.f;
#pragma unroll
            for (int w = 0; w < 4; w++) {
                sw[w] = Mw[w * 16 + hr] == -INFINITY ? 0.f : exp2f(Mw[w * 16 + hr] - M);
                L += sw[w] * Lw[w * 16 + hr];
            }
            const int h = h0 + hr;
            const float gh = gated ? a.g[h] : 1.f, inv = L > 0.f ? 1.f / L : 0.f;
            const long long base = (row * a.Hq + h) * (long long)D;
#pragma unroll
            for (int c = 0; c < CPT; c += 2) {
                float v0 = 0.f, v1 = 0.f;
#pragma unroll
                for (int w = 0; w < 4; w++) {
                    const float2 t = *reinterpret_cast<const float2 *>(Om + (w * 16 + hr) * D + c0 + c);
                    v0 = fmaf(sw[w], t.x, v0);
                    v1 = fmaf(sw[w], t.y, v1);
                }
                v0 = L > 0.f ? v0 * inv : 0.f;
                v1 = L > 0.f ? v1 * inv : 0.f;
                if (gated) {
                    const uint32_t lw = *reinterpret_cast<const uint32_t *>(a.lin + base + c0 + c);
                    v0 = fmaf(gh, v0, (1.0f - gh) * bf16lo(lw));
                    v1 = fmaf(gh, v1, (1.0f - gh) * bf16hi(lw));
                }
                *reinterpret_cast<float2 *>(a.out + base + c0 + c) = make_float2(v0, v1);
            }
            if (a.lse && c0 == 0)
                a.lse[row * a.Hq + h] = L > 0.f ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
        }
        return;
    } else {

    float o[DNW][4];
#pragma unroll
    for (int i = 0; i < DNW; i++) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};
    const int col0 = dsl * DW;  // this warp's first output column

    for (int s = 0; s < nstages; s++) {
        if (s + 1 < nstages) {
            if ((s + 1) * kKeys - win0 >= kIdxWin) fill_idx((s + 1) * kKeys);
            load_stage((s + 1) & 1, (s + 1) * kKeys);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const uint16_t *Kt = KVs + (s & 1) * 2 * Cfg<D>::TILE;
        const uint16_t *Vt = Kt + Cfg<D>::TILE;
        const int kvalid = min(kKeys, nkeys - s * kKeys);

        float sc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; nt++) {
            sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < DK; kk += 2) {
                uint32_t b0, b1, b2, b3;
                int key = nt * 8 + (lane & 7), col = kk * 16 + (lane >> 3) * 8;
                ldmatrix_x4(smem_u32(Kt + key * RS + col), b0, b1, b2, b3);
                mma_bf16_16816(sc[nt], qf[kk], b0, b1);
                mma_bf16_16816(sc[nt], qf[kk + 1], b2, b3);
            }
        }
        // online softmax (log2 domain); rows g8 and g8+8 of the head tile
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int nt = 0; nt < NT; nt++) {
#pragma unroll
            for (int e = 0; e < 4; e++) {
                int key = nt * 8 + 2 * c4 + (e & 1);
                float x = key < kvalid ? sc[nt][e] * a.scale_log2 : -INFINITY;
                sc[nt][e] = x;
                mx[e >> 1] = fmaxf(mx[e >> 1], x);
            }
        }
        float corr[2];
#pragma unroll
        for (int r = 0; r < 2; r++) {
            mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
            mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
            float mnew = fmaxf(m_r[r], mx[r]);
            float muse = mnew == -INFINITY ? 0.f : mnew;
            corr[r] = exp2f(m_r[r] - muse);
            m_r[r] = mnew;
            mx[r] = muse;
        }
        float rs[2] = {0.f, 0.f};
        uint32_t ph[NT][2], pl[NT][2];  // P as bf16 hi + lo
#pragma unroll
        for (int nt = 0; nt < NT; nt++) {
            float p0 = exp2f(sc[nt][0] - mx[0]), p1 = exp2f(sc[nt][1] - mx[0]);
            float p2 = exp2f(sc[nt][2] - mx[1]), p3 = exp2f(sc[nt][3] - mx[1]);
            rs[0] += p0 + p1;
            rs[1] += p2 + p3;
            ph[nt][0] = pack_bf16(p0, p1);
            ph[nt][1] = pack_bf16(p2, p3);
            pl[nt][0] = pack_bf16(p0 - bf16lo(ph[nt][0]), p1 - bf16hi(ph[nt][0]));
            pl[nt][1] = pack_bf16(p2 - bf16lo(ph[nt][1]), p3 - bf16hi(ph[nt][1]));
        }
#pragma unroll
        for (int r = 0; r < 2; r++) {
            rs[r] += __shfl_xor_sync(0xffffffffu, rs[r], 1);
            rs[r] += __shfl_xor_sync(0xffffffffu, rs[r], 2);
            l_r[r] = l_r[r] * corr[r] + rs[r];
        }
#pragma unroll
        for (int dn = 0; dn < DNW; dn++) {
            o[dn][0] *= corr[0];
            o[dn][1] *= corr[0];
            o[dn][2] *= corr[1];
            o[dn][3] *= corr[1];
        }
        // P V over this warp's output columns: A = P (16 heads x 16 keys)
        // straight from the score registers
#pragma unroll
        for (int kk2 = 0; kk2 < NT / 2; kk2++) {
            uint32_t ah[4] = {ph[2 * kk2][0], ph[2 * kk2][1], ph[2 * kk2 + 1][0], ph[2 * kk2 + 1][1]};
            uint32_t al[4] = {pl[2 * kk2][0], pl[2 * kk2][1], pl[2 * kk2 + 1][0], pl[2 * kk2 + 1][1]};
#pragma unroll
            for (int dn = 0; dn < DNW / 2; dn++) {
                uint32_t b0, b1, b2, b3;
                int key = kk2 * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                int col = col0 + dn * 16 + (lane >> 4) * 8;
                ldmatrix_x4_trans(smem_u32(Vt + key * RS + col), b0, b1, b2, b3);
                mma_bf16_16816(o[2 * dn], ah, b0, b1);
                mma_bf16_16816(o[2 * dn + 1], ah, b2, b3);
                mma_bf16_16816(o[2 * dn], al, b0, b1);
                mma_bf16_16816(o[2 * dn + 1], al, b2, b3);
            }
        }
        __syncthreads();
    }

    // ---- epilogue
    const bool gated = a.g != nullptr && a.lin != nullptr;
    const int S = a.splits;
    __syncthreads();  // bad_row is final
    if (S == 1) {
        // the whole index list was this block's: every warp finishes its own
        // rows and columns straight from registers
        if (bad_row) {
            if (tid == 0) set_status(a.status, ESA_ERR_BAD_INDEX);
            return;
        }
#pragma unroll
        for (int rr = 0; rr < 2; rr++) {
            const int hr = ht * 16 + g8 + rr * 8;
            if (hr >= nh) continue;
            const int h = h0 + hr;
            const float L = l_r[rr];
            const float gh = gated ? a.g[h] : 1.f;
            const long long base = (row * a.Hq + h) * (long long)D;
#pragma unroll
            for (int dn = 0; dn < DNW; dn++) {
                const int col = col0 + dn * 8 + 2 * c4;
                float v0 = L > 0.f ? o[dn][2 * rr] / L : 0.f, v1 = L > 0.f ? o[dn][2 * rr + 1] / L : 0.f;
                if (gated) {
                    const uint32_t lw = *reinterpret_cast<const uint32_t *>(a.lin + base + col);
                    v0 = fmaf(gh, v0, (1.0f - gh) * bf16lo(lw));
                    v1 = fmaf(gh, v1, (1.0f - gh) * bf16hi(lw));
                }
                *reinterpret_cast<float2 *>(a.out + base + col) = make_float2(v0, v1);
            }
            if (a.lse && dsl == 0 && c4 == 0)
                a.lse[row * a.Hq + h] = L > 0.f ? (m_r[rr] + log2f(L)) * 0.69314718055994531f : -INFINITY;
        }
        return;
    }
    // several splits (one cluster): push each head's partial (unnormalised
    // output, max, sum) into the shared memory of the block that finalises
    // it (head hr -> block hr % S, slot hr / S), then one cluster barrier;
    // every block then reduces only from its own shared memory
    const int MM = (GT + S - 1) / S;  // heads per finalising block, at most
    float *RB = reinterpret_cast<float *>(KVs + 2 * 2 * Cfg<D>::TILE);  // [MM][S][D]
    float *RM = RB + (size_t)MM * S * D;                               // [MM][S]
    float *RL = RM + MM * S;                                           // [MM][S]
    int *RBad = reinterpret_cast<int *>(RL + MM * S);                  // [S]
    float *Wt = reinterpret_cast<float *>(RBad + S);                   // [MM][S] merge weights
    float *Mf = Wt + MM * S, *Lf = Mf + MM;                            // [MM]
#pragma unroll
    for (int rr = 0; rr < 2; rr++) {
        const int hr = ht * 16 + g8 + rr * 8;
        if (hr < nh) {
            const int dst = hr % S, i = hr / S;
            float *rb = cluster.map_shared_rank(RB + ((size_t)i * S + split) * D, dst);
#pragma unroll
            for (int dn = 0; dn < DNW; dn++) {
                const int col = col0 + dn * 8 + 2 * c4;
                *reinterpret_cast<float2 *>(rb + col) = make_float2(o[dn][2 * rr], o[dn][2 * rr + 1]);
            }
            if (dsl == 0 && c4 == 0) {
                *cluster.map_shared_rank(RM + i * S + split, dst) = m_r[rr];
                *cluster.map_shared_rank(RL + i * S + split, dst) = l_r[rr];
            }
        }
    }
    if (tid < S) *cluster.map_shared_rank(RBad + split, tid) = bad_row;
    cluster.sync();  // every push has landed; nobody touches another block's memory after this
    int any_bad = 0;
    for (int s2 = 0; s2 < S; s2++) any_bad |= RBad[s2];
    if (any_bad) {
        if (split == 0 && tid == 0) set_status(a.status, ESA_ERR_BAD_INDEX);
        return;
    }
    const int mine = nh > split ? (nh - split + S - 1) / S : 0;  // heads this block finalises
    if (tid < mine) {
        float M = -INFINITY;
        for (int s2 = 0; s2 < S; s2++) M = fmaxf(M, RM[tid * S + s2]);
        const float Mu = M == -INFINITY ? 0.f : M;
        float L = 0.f;
        for (int s2 = 0; s2 < S; s2++) {
            const float w = exp2f(RM[tid * S + s2] - Mu);
            Wt[tid * S + s2] = w;
            L += RL[tid * S + s2] * w;
        }
        Mf[tid] = M;
        Lf[tid] = L;
    }
    __syncthreads();
    for (int e = tid; e < mine * (D / 4); e += kThreads) {
        const int i = e / (D / 4), d4 = (e % (D / 4)) * 4;
        const int h = h0 + split + i * S;
        float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int s2 = 0; s2 < S; s2++) {
            const float w = Wt[i * S + s2];
            const float4 v = *reinterpret_cast<const float4 *>(RB + ((size_t)i * S + s2) * D + d4);
            O.x = fmaf(v.x, w, O.x);
            O.y = fmaf(v.y, w, O.y);
            O.z = fmaf(v.z, w, O.z);
            O.w = fmaf(v.w, w, O.w);
        }
        const float L = Lf[i];
        float4 res = L > 0.f ? make_float4(O.x / L, O.y / L, O.z / L, O.w / L) : make_float4(0.f, 0.f, 0.f, 0.f);
        const long long off = (row * a.Hq + h) * (long long)D + d4;
        if (gated) {
            const float gh = a.g[h], gl = 1.0f - gh;
            const uint2 lw = *reinterpret_cast<const uint2 *>(a.lin + off);
            res.x = fmaf(gh, res.x, gl * bf16lo(lw.x));
            res.y = fmaf(gh, res.y, gl * bf16hi(lw.x));
            res.z = fmaf(gh, res.z, gl * bf16lo(lw.y));
            res.w = fmaf(gh, res.w, gl * bf16hi(lw.y));
        }
        *reinterpret_cast<float4 *>(a.out + off) = res;
        if (a.lse && d4 == 0)
            a.lse[row * a.Hq + h] = L > 0.f ? (Mf[i] + log2f(L)) * 0.69314718055994531f : -INFINITY;
    }
    }  // !KS
    }  // !kKeyRows
}

// Floats of one (row, head group)'s partial outputs: [S blocks][GT heads][D].
// Its (max, sum) records, [S][GT] 64-bit words, live in a separate region
// (zero between calls), followed by one word nothing writes (the timeout
// test waits on it).
__host__ __device__ inline size_t dec_group_floats(int GT, int D, int S) { return (size_t)S * GT * D; }

// A block's (max, sum) record: max's bits low, sum's high. Zero means "not
// yet written" (a written record never is: sum >= 1 whenever max is finite,
// and max = -inf when sum = 0); an all-ones sum marks a block that found an
// invalid index.
constexpr unsigned kBadSum = 0xffffffffu;
__device__ __forceinline__ unsigned long long ml_record(float M, float L) {
    return (unsigned long long)__float_as_uint(M) | ((unsigned long long)__float_as_uint(L) << 32);
}

// Decode rows (the index list split over S blocks): 8 warps, and each warp
// owns a slice of every stage's keys for one 16-head tile, so no score is
// computed twice. A stage holds 128 keys; with GT = 16 * HT heads, warp w
// takes head tile w % HT and keys (w / HT) * SL .. + SL of the stage (SL =
// 16 * HT). A warp keeps its own online softmax over every output column;
// at the end the warps of a head tile merge through shared memory and each
// block publishes its merged (max, sum, unnormalised output) per head to the
// workspace (L2), then a (max, sum) record per head with a release store.
// Block `split` finalises heads split, split + S, ...: it polls the S
// records of each (acquire loads, bounded), clears them, and merges the S
// partials. The launch is cooperative (every block resident; one block per
// SM by registers), so no thread-block cluster has to fit in one GPC:
// 16-block clusters at one block per SM fit only 7 at a time here.
constexpr int kDecThreads = 256;
constexpr int kDecKeys = 128;  // keys per stage

template <int D>
struct DecCfg {
    static constexpr int RS = D + 8;             // padded K/V row stride (bf16 elements)
    static constexpr int TILE = kDecKeys * RS;   // one K or V stage tile (elements)
    static constexpr int OS = D + 8;             // padded row stride of a warp's fp32 partial
    static constexpr size_t STAGE_BYTES = (size_t)2 * TILE * 2;
    static constexpr size_t MERGE_BYTES = (size_t)8 * 16 * OS * 4 + 2 * 8 * 16 * 4;
};

template <int D, int GT>
__global__ void __launch_bounds__(kDecThreads) decode_attn_kernel(AttnArgs a) {
    constexpr int RS = DecCfg<D>::RS, TILE = DecCfg<D>::TILE, OS = DecCfg<D>::OS;
    constexpr int HT = GT / 16;         // head tiles
    constexpr int KQ = 8 / HT;          // key slices per stage
    constexpr int SL = kDecKeys / KQ;   // keys per warp and stage
    constexpr int NT = SL / 8;          // score n-tiles of 8 keys
    constexpr int DK = D / 16;          // k-steps over the head dim
    constexpr int DN = D / 8;           // output n-tiles (every column)
    constexpr int CH = D / 8;           // 16-byte chunks per K/V row
    constexpr int KPR = kDecThreads / CH;  // keys per gather round
    constexpr int GR = kDecKeys / KPR;     // gather rounds per stage
    static_assert(HT * KQ == 8 && NT % 2 == 0 && DN % 2 == 0, "tile split");
    extern __shared__ __align__(16) unsigned char smem_raw[];
    uint16_t *Qs = reinterpret_cast<uint16_t *>(smem_raw);
    unsigned char *work = smem_raw + (size_t)GT * RS * 2;  // stage buffers, then the warps' partials
    uint16_t *KVs = reinterpret_cast<uint16_t *>(work);

    __shared__ int fin_state;  // finalising: 0 ok, 1 an invalid index, 2 a wait ran out
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int ht = warp % HT, kq = warp / HT;
    const int g8 = lane >> 2, c4 = lane & 3;

    long long bid = blockIdx.x;
    const int split = (int)(bid % a.splits);
    const long long grp = bid / a.splits;  // (row, key/value head, head group)
    bid = grp;
    const int hgi = (int)(bid % a.hg);
    bid /= a.hg;
    const int kvh = (int)(bid % a.Hkv);
    const long long row = bid / a.Hkv;  // b*Tq + t
    const long long b = row / a.Tq, t = row % a.Tq;
    const long long p = a.q_offset + t;
    const int G = a.Hq / a.Hkv;
    const int sg = hgi / a.gps, sub = hgi % a.gps;
    const int h0 = kvh * G + sg * a.seg + sub * GT;  // first query head of this block
    const int nh = min(GT, a.seg - sub * GT);
    const long long set = a.nsets > 1 ? row * a.nsets + h0 / a.hs : row;

    // ---- Q tile (GT heads x D), zero rows past the group (independent of the selection)
    {
        const uint16_t *qrow = a.q + (row * a.Hq + h0) * (long long)D;
        for (int i = tid; i < GT * CH; i += kDecThreads) {
            const int hr = i / CH, ch = i % CH;
            cp_async16_zfill(smem_u32(Qs + hr * RS + ch * 8), qrow + (hr < nh ? hr * D + ch * 8 : 0), hr < nh);
        }
        cp_async_commit();
    }
    pdl_wait();
    const int k_begin = split * a.kps;
    const int lim = max(0, min(a.kps, a.K - k_begin));  // list positions of this split
    const int32_t *idx_row = a.idx + set * (long long)a.K + k_begin;
    const uint16_t *kbase = a.k + (b * a.Tk * a.Hkv + kvh) * (long long)D;
    const uint16_t *vbase = a.v + (b * a.Tk * a.Hkv + kvh) * (long long)D;
    const long long kstride = (long long)a.Hkv * D;
    // gathers: thread tid fetches chunk tid % CH of keys tid / CH + r * KPR;
    // the indices are read first (for stage 0 together with the count)
    const int ch = tid % CH, k0 = tid / CH;
    auto load_idx = [&](int kb, int *j) {
#pragma unroll
        for (int r = 0; r < GR; r++) {
            const int pos = kb + k0 + r * KPR;
            j[r] = pos < lim ? __ldg(idx_row + pos) : -1;
        }
    };
    int j0[GR];
    load_idx(0, j0);
    int bad = 0;
    int c = a.cnt[set];
    // this block's first output element of the finalising merge: its gate
    // and linear-branch values are fetched now, off the critical path
    const bool gated = a.g != nullptr && a.lin != nullptr;
    const int S = a.splits;
    const int mine = nh > split ? (nh - split + S - 1) / S : 0;  // heads this block finalises
    uint2 lw0 = make_uint2(0u, 0u);
    float gh0 = 1.f;
    if (gated && tid < mine * (D / 4)) {
        const int h = h0 + split + (tid / (D / 4)) * S;
        lw0 = *reinterpret_cast<const uint2 *>(a.lin + (row * a.Hq + h) * (long long)D + (tid % (D / 4)) * 4);
        gh0 = a.g[h];
    }
    const int cmax = (int)min((long long)a.K, p + 1);
    if (c < 0 || c > cmax) {
        bad = 1;
        c = 0;
    }
    const int k_end = min(c, k_begin + a.kps);
    const int nkeys = max(0, k_end - k_begin);
    auto load_stage = [&](int buf, int kb, int *j) {
        uint16_t *Kt = KVs + buf * 2 * TILE;
        uint16_t *Vt = Kt + TILE;
#pragma unroll
        for (int r = 0; r < GR; r++) {
            const int pos = kb + k0 + r * KPR;
            int jr = pos < nkeys ? j[r] : -1;
            if (pos < nkeys && (jr < 0 || jr > p)) {
                bad = 1;
                jr = -1;
            }
            const bool valid = jr >= 0;
            const long long off = (valid ? jr : 0) * kstride + ch * 8;
            const int key = k0 + r * KPR;
            cp_async16_zfill(smem_u32(Kt + key * RS + ch * 8), kbase + off, valid);
            cp_async16_zfill(smem_u32(Vt + key * RS + ch * 8), vbase + off, valid);
        }
        cp_async_commit();
    };

    const int nst = (nkeys + kDecKeys - 1) / kDecKeys;
    if (nst > 0) load_stage(0, 0, j0);
    if (nst > 0) cp_async_wait<1>(); else cp_async_wait<0>();  // the Q tile
    __syncthreads();
    // Q fragments are re-read from shared memory at every k-step (registers
    // for two blocks per SM: a 16-block cluster then needs only 8 SMs of a GPC)
    const uint32_t qaddr = smem_u32(Qs + (ht * 16 + (lane & 15)) * RS + (lane >> 4) * 8);

    float o[DN][4];
#pragma unroll
    for (int i = 0; i < DN; i++) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};  // head rows g8, g8 + 8
    const int kb = kq * SL;  // this warp's first key within a stage

    for (int s = 0; s < nst; s++) {
        if (s + 1 < nst) {
            int jn[GR];
            load_idx((s + 1) * kDecKeys, jn);
            load_stage((s + 1) & 1, (s + 1) * kDecKeys, jn);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const uint16_t *Kt = KVs + (s & 1) * 2 * TILE;
        const uint16_t *Vt = Kt + TILE;
        const int kvalid = min(kDecKeys, nkeys - s * kDecKeys);
        if (kb < kvalid) {
            float sc[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; nt++) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < DK; kk += 2) {
                uint32_t qa[4], qb[4];
                ldmatrix_x4(qaddr + kk * 32, qa[0], qa[1], qa[2], qa[3]);
                ldmatrix_x4(qaddr + kk * 32 + 32, qb[0], qb[1], qb[2], qb[3]);
#pragma unroll
                for (int nt = 0; nt < NT; nt++) {
                    uint32_t b0, b1, b2, b3;
                    const int key = kb + nt * 8 + (lane & 7), col = kk * 16 + (lane >> 3) * 8;
                    ldmatrix_x4(smem_u32(Kt + key * RS + col), b0, b1, b2, b3);
                    mma_bf16_16816(sc[nt], qa, b0, b1);
                    mma_bf16_16816(sc[nt], qb, b2, b3);
                }
            }
            float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
            for (int nt = 0; nt < NT; nt++) {
#pragma unroll
                for (int e = 0; e < 4; e++) {
                    const int key = kb + nt * 8 + 2 * c4 + (e & 1);
                    const float x = key < kvalid ? sc[nt][e] * a.scale_log2 : -INFINITY;
                    sc[nt][e] = x;
                    mx[e >> 1] = fmaxf(mx[e >> 1], x);
                }
            }
            float corr[2];
#pragma unroll
            for (int r = 0; r < 2; r++) {
                mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
                mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
                const float mnew = fmaxf(m_r[r], mx[r]);
                const float muse = mnew == -INFINITY ? 0.f : mnew;
                corr[r] = exp2f(m_r[r] - muse);
                m_r[r] = mnew;
                mx[r] = muse;
            }
            float rs[2] = {0.f, 0.f};
            uint32_t ph[NT][2], pl[NT][2];  // P as bf16 hi + lo (~16 significant bits)
#pragma unroll
            for (int nt = 0; nt < NT; nt++) {
                const float p0 = exp2f(sc[nt][0] - mx[0]), p1 = exp2f(sc[nt][1] - mx[0]);
                const float p2 = exp2f(sc[nt][2] - mx[1]), p3 = exp2f(sc[nt][3] - mx[1]);
                rs[0] += p0 + p1;
                rs[1] += p2 + p3;
                ph[nt][0] = pack_bf16(p0, p1);
                ph[nt][1] = pack_bf16(p2, p3);
                pl[nt][0] = pack_bf16(p0 - bf16lo(ph[nt][0]), p1 - bf16hi(ph[nt][0]));
                pl[nt][1] = pack_bf16(p2 - bf16lo(ph[nt][1]), p3 - bf16hi(ph[nt][1]));
            }
#pragma unroll
            for (int r = 0; r < 2; r++) {
                rs[r] += __shfl_xor_sync(0xffffffffu, rs[r], 1);
                rs[r] += __shfl_xor_sync(0xffffffffu, rs[r], 2);
                l_r[r] = l_r[r] * corr[r] + rs[r];
            }
#pragma unroll
            for (int dn = 0; dn < DN; dn++) {
                o[dn][0] *= corr[0];
                o[dn][1] *= corr[0];
                o[dn][2] *= corr[1];
                o[dn][3] *= corr[1];
            }
#pragma unroll
            for (int kk2 = 0; kk2 < NT / 2; kk2++) {
                const uint32_t ah[4] = {ph[2 * kk2][0], ph[2 * kk2][1], ph[2 * kk2 + 1][0], ph[2 * kk2 + 1][1]};
                const uint32_t al[4] = {pl[2 * kk2][0], pl[2 * kk2][1], pl[2 * kk2 + 1][0], pl[2 * kk2 + 1][1]};
#pragma unroll
                for (int dn = 0; dn < DN / 2; dn++) {
                    uint32_t b0, b1, b2, b3;
                    const int key = kb + kk2 * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                    const int col = dn * 16 + (lane >> 4) * 8;
                    ldmatrix_x4_trans(smem_u32(Vt + key * RS + col), b0, b1, b2, b3);
                    mma_bf16_16816(o[2 * dn], ah, b0, b1);
                    mma_bf16_16816(o[2 * dn + 1], ah, b2, b3);
                    mma_bf16_16816(o[2 * dn], al, b0, b1);
                    mma_bf16_16816(o[2 * dn + 1], al, b2, b3);
                }
            }
        }
        __syncthreads();  // the buffer is free for the stage after next
    }
    bad = __syncthreads_or(bad);  // also: every warp is done with the stage buffers

    // ---- the warps' partials -> shared memory
    float *Wo = reinterpret_cast<float *>(work);  // [8 warps][16 heads][OS]
    float *Wm = Wo + 8 * 16 * OS, *Wl = Wm + 8 * 16;
#pragma unroll
    for (int rr = 0; rr < 2; rr++) {
        const int hr = g8 + rr * 8;
#pragma unroll
        for (int dn = 0; dn < DN; dn++)
            *reinterpret_cast<float2 *>(Wo + (warp * 16 + hr) * OS + dn * 8 + 2 * c4) =
                make_float2(o[dn][2 * rr], o[dn][2 * rr + 1]);
        if (c4 == 0) {
            Wm[warp * 16 + hr] = m_r[rr];
            Wl[warp * 16 + hr] = l_r[rr];
        }
    }
    // the group's exchange area (dec_group_floats)
    float *XP = a.xpart + (size_t)grp * dec_group_floats(GT, D, S);
    unsigned long long *XR = a.xrec + (size_t)grp * S * GT;
    const unsigned long long *never = a.xrec + (size_t)gridDim.x * GT;
    const int MM = (GT + S - 1) / S;  // heads per finalising block, at most
    const size_t stage_bytes = DecCfg<D>::STAGE_BYTES * (a.kps > kDecKeys ? 2 : 1);
    float *Wt = reinterpret_cast<float *>(
        work + (stage_bytes > DecCfg<D>::MERGE_BYTES ? stage_bytes : DecCfg<D>::MERGE_BYTES));  // [MM][S]
    float *Mf = Wt + MM * S, *Lf = Mf + MM;                                                   // [MM]
    __syncthreads();
    // merge each head's key slices (TPH threads per head), store the block's
    // partial, then (after a barrier: every thread's stores come first) its
    // record
    {
        constexpr int TPH = kDecThreads / GT;  // threads per head
        constexpr int FPT = D / 4 / TPH;       // float4 columns per thread
        static_assert(FPT * TPH * 4 == D, "column split");
        const int hr = tid / TPH, w0 = hr / 16, r16 = hr % 16;  // warps w0 + HT * q hold this head
        float M = -INFINITY, L = 0.f;
        if (hr < nh) {
#pragma unroll
            for (int q = 0; q < KQ; q++) M = fmaxf(M, Wm[(w0 + HT * q) * 16 + r16]);
            float sw[KQ];
#pragma unroll
            for (int q = 0; q < KQ; q++) {
                const int w = w0 + HT * q;
                const float mw = Wm[w * 16 + r16];
                sw[q] = mw == -INFINITY ? 0.f : exp2f(mw - M);
                L = fmaf(sw[q], Wl[w * 16 + r16], L);
            }
            float *xp = XP + ((size_t)split * GT + hr) * D;
#pragma unroll
            for (int f = 0; f < FPT; f++) {
                const int d4 = (tid % TPH + f * TPH) * 4;
                float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int q = 0; q < KQ; q++) {
                    const float4 v = *reinterpret_cast<const float4 *>(Wo + ((w0 + HT * q) * 16 + r16) * OS + d4);
                    O.x = fmaf(sw[q], v.x, O.x);
                    O.y = fmaf(sw[q], v.y, O.y);
                    O.z = fmaf(sw[q], v.z, O.z);
                    O.w = fmaf(sw[q], v.w, O.w);
                }
                __stcg(reinterpret_cast<float4 *>(xp + d4), O);
            }
        }
        __syncthreads();
        if (hr < nh && tid % TPH == 0)
            st_release_u64(XR + (size_t)split * GT + hr,
                           bad ? ((unsigned long long)kBadSum << 32) : ml_record(M, L));
    }
    // finalise: one warp per head, one lane per block's record (S < 32);
    // with test-only extra arrivals, lane S also waits on a word nothing writes
    if (tid == 0) fin_state = 0;
    __syncthreads();
    for (int i = warp; i < mine; i += kDecThreads / 32) {
        const int hr = split + i * S;
        unsigned long long rec = ml_record(-INFINITY, 0.f);
        bool timed_out = false;
        if (lane < S || (lane == S && a.extra > 0)) {
            const unsigned long long *src = lane < S ? XR + (size_t)lane * GT + hr : never;
            rec = ld_acquire_u64(src);
            if (rec == 0) {
                unsigned long long t0, t;
                asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
                unsigned ns = 32;
                while ((rec = ld_acquire_u64(src)) == 0) {
                    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
                    if ((long long)(t - t0) > a.wait_ns) {
                        timed_out = true;
                        break;
                    }
                    __nanosleep(ns);
                    if (ns < 256) ns <<= 1;
                }
            }
            if (lane < S) XR[(size_t)lane * GT + hr] = 0ull;  // cleared for the next call
            if (lane == S) rec = ml_record(-INFINITY, 0.f);
        }
        const bool badrec = (unsigned)(rec >> 32) == kBadSum;
        if (__any_sync(0xffffffffu, timed_out)) {
            if (lane == 0) atomicMax(&fin_state, 2);
        } else if (__any_sync(0xffffffffu, badrec)) {
            if (lane == 0) atomicMax(&fin_state, 1);
        }
        const float mb = __uint_as_float((unsigned)rec), lb = __uint_as_float((unsigned)(rec >> 32));
        float Mx = mb;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) Mx = fmaxf(Mx, __shfl_xor_sync(0xffffffffu, Mx, o));
        const float Mu = Mx == -INFINITY ? 0.f : Mx;
        const float w = lane < S ? exp2f(mb - Mu) : 0.f;
        float Ls = lane < S ? lb * w : 0.f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, o);
        if (lane < S) Wt[i * S + lane] = w;
        if (lane == 0) {
            Mf[i] = Mx;
            Lf[i] = Ls;
        }
    }
    __syncthreads();
    if (fin_state != 0) {
        if (tid == 0) set_status(a.status, fin_state == 2 ? ESA_ERR_TIMEOUT : ESA_ERR_BAD_INDEX);
        return;
    }
    for (int e = tid; e < mine * (D / 4); e += kDecThreads) {
        const int i = e / (D / 4), d4 = (e % (D / 4)) * 4;
        const int hr = split + i * S, h = h0 + hr;
        float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
        const float *xp = XP + (size_t)hr * D + d4;
        // eight blocks' partials in flight at a time
        for (int s0 = 0; s0 < S; s0 += 8) {
            float4 v[8];
#pragma unroll
            for (int u = 0; u < 8; u++)
                if (s0 + u < S) v[u] = __ldcg(reinterpret_cast<const float4 *>(xp + (size_t)(s0 + u) * GT * D));
#pragma unroll
            for (int u = 0; u < 8; u++) {
                if (s0 + u < S) {
                    const float w = Wt[i * S + s0 + u];
                    O.x = fmaf(v[u].x, w, O.x);
                    O.y = fmaf(v[u].y, w, O.y);
                    O.z = fmaf(v[u].z, w, O.z);
                    O.w = fmaf(v[u].w, w, O.w);
                }
            }
        }
        const float L = Lf[i];
        float4 res = L > 0.f ? make_float4(O.x / L, O.y / L, O.z / L, O.w / L) : make_float4(0.f, 0.f, 0.f, 0.f);
        const long long off = (row * a.Hq + h) * (long long)D + d4;
        if (gated) {
            const bool first = e == tid;
            const float gh = first ? gh0 : a.g[h], gl = 1.0f - gh;
            const uint2 lw = first ? lw0 : *reinterpret_cast<const uint2 *>(a.lin + off);
            res.x = fmaf(gh, res.x, gl * bf16lo(lw.x));
            res.y = fmaf(gh, res.y, gl * bf16hi(lw.x));
            res.z = fmaf(gh, res.z, gl * bf16lo(lw.y));
            res.w = fmaf(gh, res.w, gl * bf16hi(lw.y));
        }
        *reinterpret_cast<float4 *>(a.out + off) = res;
        if (a.lse && d4 == 0)
            a.lse[row * a.Hq + h] = L > 0.f ? (Mf[i] + log2f(L)) * 0.69314718055994531f : -INFINITY;
    }
}

template <int D>
size_t dec_smem(int GT, int S, int kps) {
    const size_t work = std::max(DecCfg<D>::STAGE_BYTES * (kps > kDecKeys ? 2 : 1), DecCfg<D>::MERGE_BYTES);
    const size_t MM = (size_t)(GT + S - 1) / S;
    return (size_t)GT * DecCfg<D>::RS * 2 + work + (MM * S + 2 * MM) * 4;
}
size_t dec_part_bytes(long long groups, int GT, int D, int S) {
    return align256((size_t)groups * dec_group_floats(GT, D, S) * 4);
}
// Records region: every decode-kernel shape on this device indexes it from
// its start, so one region (zero between calls: each call clears the
// records it read) serves any sequence of shapes.
constexpr int kMaxRecBlocksPerSm = 2, kMaxRecHeads = 64;
size_t dec_rec_entries() { return (size_t)device_info().sms * kMaxRecBlocksPerSm * kMaxRecHeads; }

template <int D, int GT>
size_t attn_smem() {
    return (size_t)GT * Cfg<D>::RS * 2 + (size_t)2 * 2 * Cfg<D>::TILE * 2;  // Q tile + 2 stages x (K, V)
}

// Shared memory that the cluster merge adds when the index list is split S ways.
size_t recv_smem(int D, int GT, int S) {
    if (S <= 1) return 0;
    size_t MM = (size_t)(GT + S - 1) / S;
    return (MM * S * D + 3 * MM * S + S + 2 * MM) * 4;
}

void *attn_kernel(int D, int GT, size_t *smem, int var = kColSplit) {
    if (var == kKeyRows) {  // keys as MMA rows: 8-head blocks, one split per index list
        if (D == 64) { *smem = attn_smem<64, 8>(); return (void *)sparse_attn_kernel<64, 8, kKeyRows>; }
        *smem = attn_smem<128, 8>();
        return (void *)sparse_attn_kernel<128, 8, kKeyRows>;
    }
    if (var == kKeySplit) {  // key split: 16-head tiles, one split per index list
        if (D == 64) { *smem = attn_smem<64, 16>(); return (void *)sparse_attn_kernel<64, 16, kKeySplit>; }
        *smem = attn_smem<128, 16>();
        return (void *)sparse_attn_kernel<128, 16, kKeySplit>;
    }
    if (D == 64) {
        if (GT == 16) { *smem = attn_smem<64, 16>(); return (void *)sparse_attn_kernel<64, 16, kColSplit>; }
        if (GT == 32) { *smem = attn_smem<64, 32>(); return (void *)sparse_attn_kernel<64, 32, kColSplit>; }
        *smem = attn_smem<64, 64>();
        return (void *)sparse_attn_kernel<64, 64, kColSplit>;
    }
    if (GT == 16) { *smem = attn_smem<128, 16>(); return (void *)sparse_attn_kernel<128, 16, kColSplit>; }
    if (GT == 32) { *smem = attn_smem<128, 32>(); return (void *)sparse_attn_kernel<128, 32, kColSplit>; }
    *smem = attn_smem<128, 64>();
    return (void *)sparse_attn_kernel<128, 64, kColSplit>;
}

// Shared-memory opt-in and non-portable cluster sizes, once per kernel and device.
bool prepare_attn(void *fn, size_t smem) {
    static std::mutex mu;
    static std::set<std::pair<int, void *>> done;
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lk(mu);
    if (done.count({dev, fn})) return ensure_smem(fn, smem);
    // the largest shared-memory carveout: several blocks of ~77 KB per SM
    if (!ensure_smem(fn, smem) ||
        cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess ||
        cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    done.insert({dev, fn});
    return true;
}

void *dec_kernel(int D, int GT) {
    if (D == 64) {
        if (GT == 16) return (void *)decode_attn_kernel<64, 16>;
        if (GT == 32) return (void *)decode_attn_kernel<64, 32>;
        return (void *)decode_attn_kernel<64, 64>;
    }
    if (GT == 16) return (void *)decode_attn_kernel<128, 16>;
    if (GT == 32) return (void *)decode_attn_kernel<128, 32>;
    return (void *)decode_attn_kernel<128, 64>;
}
size_t dec_smem_of(int D, int GT, int S, int kps) {
    return D == 64 ? dec_smem<64>(GT, S, kps) : dec_smem<128>(GT, S, kps);
}
// The column-split kernel for split index lists instead of the decode
// kernel (ESA_DECODE_ATTN=colsplit; read once).
bool decode_colsplit() {
    static const bool v = [] {
        const char *e = getenv("ESA_DECODE_ATTN");
        return e && std::string(e) == "colsplit";
    }();
    return v;
}

// Whether a cluster of `n` blocks of this kernel can be resident (cached).
bool cluster_fits(void *fn, size_t smem, int n, int threads = kThreads) {
    static std::mutex mu;
    static std::set<std::pair<std::pair<int, void *>, int>> ok, bad;
    int dev = 0;
    cudaGetDevice(&dev);
    auto key = std::make_pair(std::make_pair(dev, fn), n);
    {
        std::lock_guard<std::mutex> lk(mu);
        if (ok.count(key)) return true;
        if (bad.count(key)) return false;
    }
    if (!prepare_attn(fn, smem)) return false;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)n);
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)n;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    bool fits = cudaOccupancyMaxActiveClusters(&clusters, fn, &cfg) == cudaSuccess && clusters > 0;
    cudaGetLastError();
    std::lock_guard<std::mutex> lk(mu);
    (fits ? ok : bad).insert(key);
    return fits;
}

}  // namespace

size_t dec_rec_bytes() { return align256((dec_rec_entries() + 1) * 8); }

AttnPlan plan_sparse_attn(const Shape &s, int K) {
    AttnPlan p{};
    const int G = s.Hq / s.Hkv;
    const long long units = s.B * s.Tq * s.Hkv;
    DevInfo di = device_info();
    const int max_splits = std::min(kMaxSplits, (K + kKeys - 1) / kKeys);
    // decode-like (few units): split the index list over a cluster, and use
    // smaller head groups until about half the SMs have a block
    int splits = units >= di.sms ? 1 : max_splits;
    // segments: the heads of one key/value head that share one index set
    const bool ph = per_head_of(s);
    const int hs = ph ? s.Hq / s.H_I : s.Hq;
    const int seg = ph ? std::min(hs, G) : G;
    int gt = seg <= 16 ? 16 : (seg <= 32 ? 32 : 64);
    while (gt > 16 && units * (G / seg) * ((seg + gt - 1) / gt) * splits < di.sms / 2) gt /= 2;
    p.gt = gt;
    p.nsets = ph ? s.H_I : 1;
    p.hs = hs;
    p.seg = seg;
    p.gps = (seg + gt - 1) / gt;
    p.hg = (G / seg) * p.gps;
    int kps = (K + splits - 1) / splits;
    kps = (kps + kKeys - 1) / kKeys * kKeys;
    splits = (K + kps - 1) / kps;
    size_t base = 0;
    void *fn = attn_kernel(s.D, gt, &base);
    auto fewer = [&]() {
        splits = (splits + 1) / 2;
        kps = (K + splits - 1) / splits;
        kps = (kps + kKeys - 1) / kKeys * kKeys;
        splits = (K + kps - 1) / kps;
    };
    if (splits > 1 && !decode_colsplit()) {
        // the decode kernel: every block resident (a cooperative launch), so
        // fewer splits until the grid fits the device
        auto cap = [&]() {
            return (long long)occupancy(dec_kernel(s.D, gt), kDecThreads, dec_smem_of(s.D, gt, splits, kps)) * di.sms;
        };
        while (splits > 1 && (units * p.hg * splits > cap() ||
                              (size_t)(units * p.hg * splits) * gt >= dec_rec_entries()))
            fewer();
        if (splits > 1) {
            p.var = kDecode;
            p.splits = splits;
            p.smem = dec_smem_of(s.D, gt, splits, kps);
            p.keys_per_split = kps;
            p.grid = units * p.hg * splits;
            p.x_bytes = dec_part_bytes(units * p.hg, gt, s.D, splits);
            p.rec_bytes = dec_rec_bytes();
            p.ws_bytes = kStatusBytes + p.rec_bytes + p.x_bytes;
            return p;
        }
    }
    // the column-split kernel over a cluster: shrink it until the device can hold one
    while (splits > 1 && !cluster_fits(fn, base + recv_smem(s.D, gt, splits), splits)) fewer();
    p.smem = base + recv_smem(s.D, gt, splits);
    p.splits = splits;
    // each block owns its whole index list: split the keys over the warps,
    // with the keys as the MMA rows when a segment has at most 8 heads
    p.var = kColSplit;
    if (splits == 1 && seg <= 8) {
        p.var = kKeyRows;
        p.gt = 8;
        p.gps = 1;
        p.hg = G / seg;
        attn_kernel(s.D, 8, &base, kKeyRows);
        p.smem = base;
    } else if (splits == 1 && gt == 16) {
        p.var = kKeySplit;
    }
    p.keys_per_split = kps;
    p.grid = units * p.hg * splits;
    p.ws_bytes = kStatusBytes;
    return p;
}

esa_status launch_sparse_attn(const uint16_t *q, const uint16_t *k, const uint16_t *v, const int32_t *idx,
                              const int32_t *cnt, const Shape &s, int K, float scale, const float *g,
                              const uint16_t *lin, float *out, float *lse, void *ws, const AttnPlan &plan,
                              cudaStream_t st, void *xrec, void *xpart) {
    if (plan.grid == 0) return ESA_OK;
    AttnArgs a{};
    a.q = q;
    a.k = k;
    a.v = v;
    a.idx = idx;
    a.cnt = cnt;
    a.g = g;
    a.lin = lin;
    a.out = out;
    a.lse = lse;
    a.status = reinterpret_cast<int32_t *>(ws);
    a.Tq = s.Tq;
    a.Tk = s.Tk;
    a.q_offset = s.q_offset;
    a.Hq = s.Hq;
    a.Hkv = s.Hkv;
    a.K = K;
    a.hg = plan.hg;
    a.nsets = plan.nsets;
    a.hs = plan.hs;
    a.seg = plan.seg;
    a.gps = plan.gps;
    a.splits = plan.splits;
    a.kps = plan.keys_per_split;
    a.scale_log2 = scale * 1.4426950408889634f;
    if (plan.var == kDecode) {
        char *w = static_cast<char *>(ws);
        a.xrec = reinterpret_cast<unsigned long long *>(xrec ? xrec : w + kStatusBytes);
        a.xpart = reinterpret_cast<float *>(xpart ? xpart : w + kStatusBytes + plan.rec_bytes);
        a.wait_ns = wait_limit_ns();
        a.extra = debug_extra_arrivals();
    }
    size_t base = 0;
    void *fn = plan.var == kDecode ? dec_kernel(s.D, plan.gt) : attn_kernel(s.D, plan.gt, &base, plan.var);
    const size_t smem = plan.smem;
    if (!prepare_attn(fn, smem)) return ESA_ERR_CUDA;
    void *args[] = {(void *)&a};
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)plan.grid);
    cfg.blockDim = dim3(plan.var == kDecode ? kDecThreads : kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    if (plan.var == kDecode) {
        attr[1].id = cudaLaunchAttributeCooperative;
        attr[1].val.cooperative = 1;
    } else {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = (unsigned)plan.splits;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
    }
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
    if (e != cudaSuccess && plan.var == kDecode) {
        // a cooperative launch without the programmatic edge
        cudaGetLastError();
        cfg.attrs = attr + 1;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelExC(&cfg, fn, args);
    }
    return e == cudaSuccess ? ESA_OK : ESA_ERR_CUDA;
}

}  // namespace esa
