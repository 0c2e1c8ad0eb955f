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
// MMA row tile; P stays in registers and enters P V as a bf16 hi + lo pair
// (two MMAs), so the probabilities keep ~16 significant bits.
// Decode rows split the index list over the blocks of one thread-block
// cluster: each block leaves its (max, sum, unnormalised output) in its own
// shared memory and, after a cluster barrier, merges a share of the heads by
// reading every block's partial through distributed shared memory — no
// partials in global memory and no serial merge.
#include <cooperative_groups.h>

#include <algorithm>
#include <mutex>
#include <set>
#include <utility>

#include "esa_device.cuh"
#include "esa_internal.h"

namespace cg = cooperative_groups;

namespace esa {

namespace {

constexpr int kThreads = 128;
constexpr int kKeys = 64;  // keys per stage
constexpr int kMaxSplits = 16;
constexpr int kIdxWin = 1024;  // staged indices (a multiple of kKeys)

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
    float scale_log2;
};

template <int D, int GT>
__global__ void __launch_bounds__(kThreads) sparse_attn_kernel(AttnArgs a) {
    constexpr int RS = Cfg<D>::RS;
    constexpr int HT = GT / 16;       // head tiles
    constexpr int KS = 4 / HT;        // key subsets (warps per head tile)
    constexpr int KW = kKeys / KS;    // keys per warp per stage
    constexpr int NT = KW / 8;        // n-tiles of 8 keys per warp
    constexpr int DK = D / 16;        // k-steps over the head dim
    constexpr int DN = D / 8;         // n-tiles over the head dim
    extern __shared__ __align__(16) unsigned char smem_raw[];
    uint16_t *Qs = reinterpret_cast<uint16_t *>(smem_raw);
    uint16_t *KVs = Qs + GT * RS;  // [2 stages][K tile, V tile]
    __shared__ int bad_row;
    __shared__ float Pm[GT], Pl[GT];  // this block's partial: max and sum per head
    __shared__ int Pbad;
    __shared__ int kidx[kIdxWin];  // a window of this split's key positions (-1: invalid)

    cg::cluster_group cluster = cg::this_cluster();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int ht = warp % HT, ks = warp / HT;
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
    const int h0 = kvh * G + hgi * GT;  // first query head of this block
    const int nh = min(GT, G - hgi * GT);

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
    int c = a.cnt[row];
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
    const int32_t *idx_row = a.idx + row * (long long)a.K + k_begin;
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

    uint32_t qf[DK][4];
#pragma unroll
    for (int kk = 0; kk < DK; kk++) {
        int r = ht * 16 + (lane & 15), col = kk * 16 + (lane >> 4) * 8;
        ldmatrix_x4(smem_u32(Qs + r * RS + col), qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
    }

    float o[DN][4];
#pragma unroll
    for (int i = 0; i < DN; i++) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};

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
        const int kw0 = ks * KW;  // this warp's first key in the stage
        const int kvalid = min(kKeys, nkeys - s * kKeys);

        float sc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; nt++) {
            sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < DK; kk += 2) {
                uint32_t b0, b1, b2, b3;
                int key = kw0 + nt * 8 + (lane & 7), col = kk * 16 + (lane >> 3) * 8;
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
                int key = kw0 + nt * 8 + 2 * c4 + (e & 1);
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
        for (int dn = 0; dn < DN; dn++) {
            o[dn][0] *= corr[0];
            o[dn][1] *= corr[0];
            o[dn][2] *= corr[1];
            o[dn][3] *= corr[1];
        }
        // P V: A = P (16 heads x 16 keys) straight from the score registers
#pragma unroll
        for (int kk2 = 0; kk2 < NT / 2; kk2++) {
            uint32_t ah[4] = {ph[2 * kk2][0], ph[2 * kk2][1], ph[2 * kk2 + 1][0], ph[2 * kk2 + 1][1]};
            uint32_t al[4] = {pl[2 * kk2][0], pl[2 * kk2][1], pl[2 * kk2 + 1][0], pl[2 * kk2 + 1][1]};
#pragma unroll
            for (int dn = 0; dn < DN / 2; dn++) {
                uint32_t b0, b1, b2, b3;
                int key = kw0 + kk2 * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                int col = dn * 16 + (lane >> 4) * 8;
                ldmatrix_x4_trans(smem_u32(Vt + key * RS + col), b0, b1, b2, b3);
                mma_bf16_16816(o[2 * dn], ah, b0, b1);
                mma_bf16_16816(o[2 * dn + 1], ah, b2, b3);
                mma_bf16_16816(o[2 * dn], al, b0, b1);
                mma_bf16_16816(o[2 * dn + 1], al, b2, b3);
            }
        }
        __syncthreads();
    }

    // ---- merge the KS warps of each head tile into this block's partial
    float *mo = reinterpret_cast<float *>(KVs);  // [KS][HT][16][D] per-warp outputs
    float *mm = mo + KS * HT * 16 * D;           // [KS][HT][16]
    float *ml = mm + KS * HT * 16;
    float *PO = ml + KS * HT * 16;               // [GT][D] this block's partial output
    {
        float *myo = mo + ((ks * HT + ht) * 16) * D;
#pragma unroll
        for (int dn = 0; dn < DN; dn++) {
            int col = dn * 8 + 2 * c4;
            *reinterpret_cast<float2 *>(myo + g8 * D + col) = make_float2(o[dn][0], o[dn][1]);
            *reinterpret_cast<float2 *>(myo + (g8 + 8) * D + col) = make_float2(o[dn][2], o[dn][3]);
        }
        if (c4 == 0) {
            mm[(ks * HT + ht) * 16 + g8] = m_r[0];
            mm[(ks * HT + ht) * 16 + g8 + 8] = m_r[1];
            ml[(ks * HT + ht) * 16 + g8] = l_r[0];
            ml[(ks * HT + ht) * 16 + g8 + 8] = l_r[1];
        }
    }
    __syncthreads();
    for (int e = tid; e < GT * D; e += kThreads) {
        int hr = e / D, d = e % D, htt = hr / 16, r = hr % 16;
        float M = -INFINITY;
#pragma unroll
        for (int q = 0; q < KS; q++) M = fmaxf(M, mm[(q * HT + htt) * 16 + r]);
        float Mu = M == -INFINITY ? 0.f : M, L = 0.f, O = 0.f;
#pragma unroll
        for (int q = 0; q < KS; q++) {
            float w = exp2f(mm[(q * HT + htt) * 16 + r] - Mu);
            L += ml[(q * HT + htt) * 16 + r] * w;
            O += mo[((q * HT + htt) * 16 + r) * D + d] * w;
        }
        PO[hr * D + d] = O;
        if (d == 0) {
            Pm[hr] = M;
            Pl[hr] = L;
        }
    }
    if (tid == 0) Pbad = bad_row;
    // ---- merge the splits of the cluster: every partial stays in its block's
    // shared memory; block `split` finalises heads split, split+S, ...
    cluster.sync();
    const bool gated = a.g != nullptr && a.lin != nullptr;
    int any_bad = 0;
    for (int s2 = 0; s2 < a.splits; s2++) any_bad |= *cluster.map_shared_rank(&Pbad, s2);
    if (any_bad) {
        if (split == 0 && tid == 0) set_status(a.status, ESA_ERR_BAD_INDEX);
    } else {
        __shared__ float wts[kMaxSplits];
        __shared__ float Msh, Lsh;
        for (int hr = split; hr < nh; hr += a.splits) {
            if (warp == 0) {  // the head's merge weights 2^(m_s - M) and total sum
                float mloc = lane < a.splits ? *cluster.map_shared_rank(&Pm[hr], lane) : -INFINITY;
                float lloc = lane < a.splits ? *cluster.map_shared_rank(&Pl[hr], lane) : 0.f;
                float M = mloc;
#pragma unroll
                for (int d = 16; d > 0; d >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, d));
                const float Mu = M == -INFINITY ? 0.f : M;
                float w = lane < a.splits ? exp2f(mloc - Mu) : 0.f;
                float L = lloc * w;
#pragma unroll
                for (int d = 16; d > 0; d >>= 1) L += __shfl_xor_sync(0xffffffffu, L, d);
                if (lane < a.splits) wts[lane] = w;
                if (lane == 0) {
                    Msh = M;
                    Lsh = L;
                }
            }
            __syncthreads();
            const float L = Lsh, M = Msh;
            const int h = h0 + hr;
            for (int d = tid; d < D; d += kThreads) {
                float O = 0.f;
                float part[kMaxSplits];
#pragma unroll
                for (int s2 = 0; s2 < kMaxSplits; s2++)  // independent remote loads, issued together
                    part[s2] = s2 < a.splits ? *cluster.map_shared_rank(&PO[hr * D + d], s2) : 0.f;
#pragma unroll
                for (int s2 = 0; s2 < kMaxSplits; s2++) O += s2 < a.splits ? part[s2] * wts[s2] : 0.f;
                float res = L > 0.f ? O / L : 0.f;
                const long long off = (row * a.Hq + h) * (long long)D + d;
                if (gated) {
                    float gh = a.g[h];
                    res = fmaf(gh, res, (1.0f - gh) * __uint_as_float((uint32_t)a.lin[off] << 16));
                }
                a.out[off] = res;
            }
            if (a.lse && tid == 0)
                a.lse[row * a.Hq + h] = L > 0.f ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
            __syncthreads();
        }
    }
    cluster.sync();  // keep every partial alive until all blocks have read it
}

template <int D, int GT>
size_t attn_smem() {
    size_t stage = (size_t)2 * 2 * Cfg<D>::TILE * 2;  // 2 stages x (K,V) x bf16
    size_t merge = ((size_t)4 * 16 * D + 2 * 4 * 16 + (size_t)GT * D) * 4;
    return (size_t)GT * Cfg<D>::RS * 2 + (stage > merge ? stage : merge);
}

void *attn_kernel(int D, int GT, size_t *smem) {
    if (D == 64) {
        if (GT == 16) { *smem = attn_smem<64, 16>(); return (void *)sparse_attn_kernel<64, 16>; }
        if (GT == 32) { *smem = attn_smem<64, 32>(); return (void *)sparse_attn_kernel<64, 32>; }
        *smem = attn_smem<64, 64>();
        return (void *)sparse_attn_kernel<64, 64>;
    }
    if (GT == 16) { *smem = attn_smem<128, 16>(); return (void *)sparse_attn_kernel<128, 16>; }
    if (GT == 32) { *smem = attn_smem<128, 32>(); return (void *)sparse_attn_kernel<128, 32>; }
    *smem = attn_smem<128, 64>();
    return (void *)sparse_attn_kernel<128, 64>;
}

// Shared-memory opt-in and non-portable cluster sizes, once per kernel and device.
bool prepare_attn(void *fn, size_t smem) {
    static std::mutex mu;
    static std::set<std::pair<int, void *>> done;
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lk(mu);
    if (done.count({dev, fn})) return ensure_smem(fn, smem);
    if (!ensure_smem(fn, smem) ||
        cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    done.insert({dev, fn});
    return true;
}

// Whether a cluster of `n` blocks of this kernel can be resident (cached).
bool cluster_fits(void *fn, size_t smem, int n) {
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
    cfg.blockDim = dim3(kThreads);
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

AttnPlan plan_sparse_attn(const Shape &s, int K) {
    AttnPlan p{};
    const int G = s.Hq / s.Hkv;
    const long long units = s.B * s.Tq * s.Hkv;
    DevInfo di = device_info();
    const int max_splits = std::min(kMaxSplits, (K + kKeys - 1) / kKeys);
    // decode-like (few units): split the index list over a cluster, and use
    // smaller head groups until about half the SMs have a block
    int splits = units >= di.sms ? 1 : max_splits;
    int gt = G <= 16 ? 16 : (G <= 32 ? 32 : 64);
    while (gt > 16 && units * ((G + gt - 1) / gt) * splits < di.sms / 2) gt /= 2;
    p.gt = gt;
    p.hg = (G + gt - 1) / gt;
    int kps = (K + splits - 1) / splits;
    kps = (kps + kKeys - 1) / kKeys * kKeys;
    splits = (K + kps - 1) / kps;
    void *fn = attn_kernel(s.D, gt, &p.smem);
    // shrink the cluster until the device can hold one
    while (splits > 1 && !cluster_fits(fn, p.smem, splits)) {
        splits = (splits + 1) / 2;
        kps = (K + splits - 1) / splits;
        kps = (kps + kKeys - 1) / kKeys * kKeys;
        splits = (K + kps - 1) / kps;
    }
    p.splits = splits;
    p.keys_per_split = kps;
    p.grid = units * p.hg * splits;
    p.ws_bytes = kStatusBytes;
    return p;
}

esa_status launch_sparse_attn(const uint16_t *q, const uint16_t *k, const uint16_t *v, const int32_t *idx,
                              const int32_t *cnt, const Shape &s, int K, float scale, const float *g,
                              const uint16_t *lin, float *out, float *lse, void *ws, const AttnPlan &plan,
                              cudaStream_t st) {
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
    a.splits = plan.splits;
    a.kps = plan.keys_per_split;
    a.scale_log2 = scale * 1.4426950408889634f;
    size_t smem = 0;
    void *fn = attn_kernel(s.D, plan.gt, &smem);
    if (!prepare_attn(fn, smem)) return ESA_ERR_CUDA;
    void *args[] = {(void *)&a};
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)plan.grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)plan.splits;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
    return e == cudaSuccess ? ESA_OK : ESA_ERR_CUDA;
}

}  // namespace esa
