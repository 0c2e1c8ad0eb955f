// Per-head routed attention: full causal heads and sparse heads in one launch.
//
// Method ("Elastic Attention：动态路由优化大模型长文本处理", sections 2.2 and
// 3.1): each head runs either full attention or sparse attention, decided per
// head, in one fused kernel whose blocks branch on routing metadata. Sparse
// heads follow the Gated DSA path (indexer, top-K, attention over the
// selected keys, gate mix with the linear branch: "超大规模MoE架构中稀疏注意力机制
// 的演进与实践", sections 二.1-二.3, 四.1).
//
// Design: a row-tiled selection pass first reduces every query row's index
// set to its threshold form (T, P): key j <= p is selected iff
// s_j > T, or s_j == T and j <= P — exactly the top-K set with ties to the
// lower position. The attention launch then walks, for every (sequence,
// head, 64-row query tile), the causal key tiles of 64 keys with bf16 warp
// MMAs and online softmax (flash-attention order). A sparse head recomputes
// the indexer scores of the tile on int8 warp MMAs (m16n8k32, exact int32)
// and masks every unselected key; a full head masks only the future.
// Rebuilding the mask from scores costs 64/256 of the tile's MMA work and
// moves 64 bytes per key, where gathering the selected rows of a long
// multi-head prefix would fetch 512 bytes per selected key per head.
#include "esa_device.cuh"
#include "esa_internal.h"

namespace esa {

namespace {

constexpr int kThreads = 128;
constexpr int kBM = 64;  // query rows per block
constexpr int kBN = 64;  // keys per tile

struct RoutedArgs {
    const uint16_t *q, *k, *v, *lin;
    const int8_t *qI, *kI;
    const int32_t *wI;
    const uint8_t *route;
    const int32_t *thr;
    const float *g;
    float *out;
    long long B, Tq, Tk, q_offset;
    int Hq, Hkv, H_I;
    float scale_log2;
};

template <int D, int DI>
__global__ void __launch_bounds__(kThreads) routed_attn_kernel(RoutedArgs a) {
    constexpr int RS = D + 8;      // bf16 row stride in shared memory
    constexpr int IS = DI + 16;    // int8 row stride (bytes)
    constexpr int DK = D / 16, DN = D / 8, NT = kBN / 8, IK = DI / 32;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    uint16_t *Qs = reinterpret_cast<uint16_t *>(smem_raw);              // kBM x RS
    uint16_t *KV = Qs + kBM * RS;                                       // 2 x (K, V) x kBN x RS
    int8_t *KIs = reinterpret_cast<int8_t *>(KV + 2 * 2 * kBN * RS);    // 2 x kBN x IS
    int8_t *QIs = KIs + 2 * kBN * IS;                                   // H_I x kBM x IS

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g8 = lane >> 2, c4 = lane & 3;
    const long long qtiles = (a.Tq + kBM - 1) / kBM;
    long long bid = blockIdx.x;
    const int h = (int)(bid % a.Hq);
    bid /= a.Hq;
    const long long b = bid % a.B;
    const long long qt = qtiles - 1 - bid / a.B;  // longest prefixes first
    const long long t0 = qt * kBM;
    const int rows = (int)min((long long)kBM, a.Tq - t0);
    const int kvh = h / (a.Hq / a.Hkv);
    const bool sparse = a.route[b * a.Hq + h] != 0;
    const long long row0 = b * a.Tq + t0;
    const long long kend = a.q_offset + t0 + rows;  // keys 0..kend-1 are visible to some row

    // ---- Q tile (and the indexer queries of sparse heads)
    for (int i = tid; i < kBM * (D / 8); i += kThreads) {
        int r = i / (D / 8), ch = i % (D / 8);
        bool ok = r < rows;
        cp_async16_zfill(smem_u32(Qs + r * RS + ch * 8),
                         a.q + ((row0 + (ok ? r : 0)) * a.Hq + h) * (long long)D + ch * 8, ok);
    }
    if (sparse) {
        for (int i = tid; i < a.H_I * kBM * (DI / 16); i += kThreads) {
            int hh = i / (kBM * (DI / 16)), rem = i % (kBM * (DI / 16));
            int r = rem / (DI / 16), ch = rem % (DI / 16);
            bool ok = r < rows;
            cp_async16_zfill(smem_u32(QIs + (hh * kBM + r) * IS + ch * 16),
                             a.qI + ((row0 + (ok ? r : 0)) * a.H_I + hh) * (long long)DI + ch * 16, ok);
        }
    }
    cp_async_commit();

    const uint16_t *kb = a.k + (b * a.Tk * a.Hkv + kvh) * (long long)D;
    const uint16_t *vb = a.v + (b * a.Tk * a.Hkv + kvh) * (long long)D;
    const int8_t *kib = a.kI + b * a.Tk * (long long)DI;
    const long long kst = (long long)a.Hkv * D;
    auto load_tile = [&](int st, long long j0) {
        uint16_t *Kt = KV + st * 2 * kBN * RS, *Vt = Kt + kBN * RS;
        for (int i = tid; i < kBN * (D / 8); i += kThreads) {
            int key = i / (D / 8), ch = i % (D / 8);
            long long j = j0 + key;
            bool ok = j < kend;
            long long js = ok ? j : 0;
            cp_async16_zfill(smem_u32(Kt + key * RS + ch * 8), kb + js * kst + ch * 8, ok);
            cp_async16_zfill(smem_u32(Vt + key * RS + ch * 8), vb + js * kst + ch * 8, ok);
        }
        if (sparse) {
            int8_t *KIt = KIs + st * kBN * IS;
            for (int i = tid; i < kBN * (DI / 16); i += kThreads) {
                int key = i / (DI / 16), ch = i % (DI / 16);
                long long j = j0 + key;
                bool ok = j < kend;
                cp_async16_zfill(smem_u32(KIt + key * IS + ch * 16), kib + (ok ? j : 0) * DI + ch * 16, ok);
            }
        }
        cp_async_commit();
    };

    // per-thread rows g8 and g8+8 of this warp's 16
    const int r0 = warp * 16 + g8;
    long long pos[2];
    int T[2] = {INT32_MIN, INT32_MIN}, P[2] = {-1, -1};
#pragma unroll
    for (int rr = 0; rr < 2; rr++) {
        int r = r0 + rr * 8;
        pos[rr] = a.q_offset + t0 + r;
        if (r >= rows) pos[rr] = -1;  // padding row: sees nothing
        if (sparse && r < rows) {
            T[rr] = a.thr[2 * (row0 + r)];
            P[rr] = a.thr[2 * (row0 + r) + 1];
        }
    }
    int32_t wv[16];
    if (sparse) {
        for (int hh = 0; hh < a.H_I; hh++) wv[hh] = a.wI[hh];
    }

    const int ntiles = (int)((kend + kBN - 1) / kBN);
    load_tile(0, 0);
    cp_async_wait<1>();  // Q (+ qI) landed
    __syncthreads();
    uint32_t qf[DK][4];
#pragma unroll
    for (int kk = 0; kk < DK; kk++) {
        int r = warp * 16 + (lane & 15), col = kk * 16 + (lane >> 4) * 8;
        ldmatrix_x4(smem_u32(Qs + r * RS + col), qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
    }
    float o[DN][4];
#pragma unroll
    for (int i = 0; i < DN; i++) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};

    for (int ti = 0; ti < ntiles; ti++) {
        if (ti + 1 < ntiles) {
            load_tile((ti + 1) & 1, (long long)(ti + 1) * kBN);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const uint16_t *Kt = KV + (ti & 1) * 2 * kBN * RS, *Vt = Kt + kBN * RS;
        const long long j0 = (long long)ti * kBN;
        // selection mask: causal for full heads; the threshold form for sparse heads
        unsigned keep[NT];
        if (sparse) {
            const int8_t *KIt = KIs + (ti & 1) * kBN * IS;
            int si[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; nt++) si[nt][0] = si[nt][1] = si[nt][2] = si[nt][3] = 0;
            for (int hh = 0; hh < a.H_I; hh++) {
                int acc[NT][4];
#pragma unroll
                for (int nt = 0; nt < NT; nt++) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0;
#pragma unroll
                for (int ik = 0; ik < IK; ik++) {
                    uint32_t af[4];
                    int r = warp * 16 + (lane & 15), col = ik * 32 + (lane >> 4) * 16;
                    ldmatrix_x4(smem_u32(QIs + (hh * kBM + r) * IS + col), af[0], af[1], af[2], af[3]);
#pragma unroll
                    for (int nt = 0; nt < NT; nt++) {
                        uint32_t b0, b1;
                        const int8_t *kr = KIt + (nt * 8 + g8) * IS + ik * 32 + 4 * c4;
                        b0 = *reinterpret_cast<const uint32_t *>(kr);
                        b1 = *reinterpret_cast<const uint32_t *>(kr + 16);
                        mma_s8_16832(acc[nt], af, b0, b1);
                    }
                }
#pragma unroll
                for (int nt = 0; nt < NT; nt++)
#pragma unroll
                    for (int e = 0; e < 4; e++) si[nt][e] = (int)((unsigned)si[nt][e] + (unsigned)wv[hh] * (unsigned)acc[nt][e]);
            }
#pragma unroll
            for (int nt = 0; nt < NT; nt++) {
                unsigned kbits = 0;
#pragma unroll
                for (int e = 0; e < 4; e++) {
                    int rr = e >> 1;
                    long long j = j0 + nt * 8 + 2 * c4 + (e & 1);
                    bool sel = j <= pos[rr] && (si[nt][e] > T[rr] || (si[nt][e] == T[rr] && j <= P[rr]));
                    kbits |= (unsigned)sel << e;
                }
                keep[nt] = kbits;
            }
        } else {
#pragma unroll
            for (int nt = 0; nt < NT; nt++) {
                unsigned kbits = 0;
#pragma unroll
                for (int e = 0; e < 4; e++) {
                    long long j = j0 + nt * 8 + 2 * c4 + (e & 1);
                    kbits |= (unsigned)(j <= pos[e >> 1]) << e;
                }
                keep[nt] = kbits;
            }
        }
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
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int nt = 0; nt < NT; nt++)
#pragma unroll
            for (int e = 0; e < 4; e++) {
                float x = ((keep[nt] >> e) & 1u) ? sc[nt][e] * a.scale_log2 : -INFINITY;
                sc[nt][e] = x;
                mx[e >> 1] = fmaxf(mx[e >> 1], x);
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
        float rsum[2] = {0.f, 0.f};
        uint32_t ph[NT][2], pl[NT][2];  // P as bf16 hi + lo (~16 significant bits)
#pragma unroll
        for (int nt = 0; nt < NT; nt++) {
            float p0 = exp2f(sc[nt][0] - mx[0]), p1 = exp2f(sc[nt][1] - mx[0]);
            float p2 = exp2f(sc[nt][2] - mx[1]), p3 = exp2f(sc[nt][3] - mx[1]);
            rsum[0] += p0 + p1;
            rsum[1] += p2 + p3;
            ph[nt][0] = pack_bf16(p0, p1);
            ph[nt][1] = pack_bf16(p2, p3);
            pl[nt][0] = pack_bf16(p0 - bf16lo(ph[nt][0]), p1 - bf16hi(ph[nt][0]));
            pl[nt][1] = pack_bf16(p2 - bf16lo(ph[nt][1]), p3 - bf16hi(ph[nt][1]));
        }
#pragma unroll
        for (int r = 0; r < 2; r++) {
            rsum[r] += __shfl_xor_sync(0xffffffffu, rsum[r], 1);
            rsum[r] += __shfl_xor_sync(0xffffffffu, rsum[r], 2);
            l_r[r] = l_r[r] * corr[r] + rsum[r];
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
            uint32_t ah[4] = {ph[2 * kk2][0], ph[2 * kk2][1], ph[2 * kk2 + 1][0], ph[2 * kk2 + 1][1]};
            uint32_t al[4] = {pl[2 * kk2][0], pl[2 * kk2][1], pl[2 * kk2 + 1][0], pl[2 * kk2 + 1][1]};
#pragma unroll
            for (int dn = 0; dn < DN / 2; dn++) {
                uint32_t b0, b1, b2, b3;
                int key = kk2 * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
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

    // ---- epilogue: normalise, gate sparse heads, write fp32
    const bool gated = sparse && a.g != nullptr && a.lin != nullptr;
    const float gh = gated ? a.g[h] : 1.f;
#pragma unroll
    for (int rr = 0; rr < 2; rr++) {
        int r = r0 + rr * 8;
        if (r >= rows) continue;
        float inv = l_r[rr] > 0.f ? 1.f / l_r[rr] : 0.f;
        const long long off = ((row0 + r) * a.Hq + h) * (long long)D;
#pragma unroll
        for (int dn = 0; dn < DN; dn++) {
            int col = dn * 8 + 2 * c4;
            float x0 = o[dn][2 * rr] * inv, x1 = o[dn][2 * rr + 1] * inv;
            if (gated) {
                uint32_t lw = *reinterpret_cast<const uint32_t *>(a.lin + off + col);
                x0 = fmaf(gh, x0, (1.f - gh) * bf16lo(lw));
                x1 = fmaf(gh, x1, (1.f - gh) * bf16hi(lw));
            }
            *reinterpret_cast<float2 *>(a.out + off + col) = make_float2(x0, x1);
        }
    }
}

template <int D, int DI>
size_t routed_smem(int H_I) {
    return (size_t)kBM * (D + 8) * 2 + (size_t)2 * 2 * kBN * (D + 8) * 2 + (size_t)2 * kBN * (DI + 16) +
           (size_t)H_I * kBM * (DI + 16);
}

template <int D>
void *routed_kernel_d(int DI, int H_I, size_t *smem) {
    switch (DI) {
        case 32: *smem = routed_smem<D, 32>(H_I); return (void *)routed_attn_kernel<D, 32>;
        case 64: *smem = routed_smem<D, 64>(H_I); return (void *)routed_attn_kernel<D, 64>;
        default: *smem = routed_smem<D, 128>(H_I); return (void *)routed_attn_kernel<D, 128>;
    }
}

}  // namespace

size_t ws_routed(const Shape &s, int) { return kStatusBytes + align256((size_t)s.B * s.Tq * 2 * 4); }

esa_status launch_routed_attn(const uint16_t *q, const uint16_t *k, const uint16_t *v, const int8_t *qI,
                              const int8_t *kI, const int32_t *wI, const uint8_t *route, const Shape &s, int K,
                              float scale, const float *g, const uint16_t *lin, float *out, void *ws,
                              cudaStream_t st) {
    char *base = static_cast<char *>(ws);
    int32_t *thr = reinterpret_cast<int32_t *>(base + kStatusBytes);
    esa_status e = launch_row_select(qI, kI, wI, s, K, nullptr, nullptr, thr, ws, st);
    if (e != ESA_OK) return e;
    RoutedArgs a{};
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
    a.B = s.B;
    a.Tq = s.Tq;
    a.Tk = s.Tk;
    a.q_offset = s.q_offset;
    a.Hq = s.Hq;
    a.Hkv = s.Hkv;
    a.H_I = s.H_I;
    a.scale_log2 = scale * 1.4426950408889634f;
    long long blocks = s.B * s.Hq * ((s.Tq + kBM - 1) / kBM);
    if (blocks == 0) return ESA_OK;
    size_t smem = 0;
    void *fn = s.D == 64 ? routed_kernel_d<64>(s.D_I, s.H_I, &smem) : routed_kernel_d<128>(s.D_I, s.H_I, &smem);
    if (!ensure_smem(fn, smem)) return ESA_ERR_CUDA;
    void *args[] = {(void *)&a};
    cudaError_t ce = cudaLaunchKernel(fn, dim3((unsigned)blocks), dim3(kThreads), args, smem, st);
    return ce == cudaSuccess ? ESA_OK : ESA_ERR_CUDA;
}

}  // namespace esa
