// KDA: the gated linear-attention branch whose output is the linear_output of
// the gate mix.
//
// Method: the Gated DSA page ("超大规模MoE架构中稀疏注意力机制的演进与实践",
// sections 一, 二.3 and 三) keeps KDA — a gated linear attention that folds the
// history into a recurrent state — in most layers, and gates its output
// against the sparse attention output. The page prints no formula; this is
// the published Kimi Delta Attention recurrence. Per (sequence, head) a state
// S of Dk x Dv values, per step t:
//   S = diag(alpha_t) S;  u = S^T k_t;  S += beta_t k_t (v_t - u)^T;
//   o_t = scale S^T q_t.
//
// The recurrence is sequential in t but independent per value column c:
// column c of S is a Dk-vector s with s = alpha_t * s, then
// s += beta_t (v_t[c] - k_t . s) k_t. So the kernel spreads the columns over
// the chip and holds each column in registers for the whole sequence:
//   - 8 lanes per column, each holding Dk/8 key channels; a step is Dk/8
//     multiplies and 3 Dk/8 FMAs per lane, plus two 3-level shuffle sums
//     (k . s, on the step-to-step chain, and q . s, off it);
//   - block = 4 warps = 16 columns of one (sequence, head); grid (Dv/16, H, B);
//   - the inputs of CT steps (the head's q, k and alpha rows, the block's 16
//     v values, beta) are staged in shared memory with cp.async, double
//     buffered, laid out so that the 8 lanes of a column read 8 consecutive
//     16-byte pieces (no bank conflicts; the 4 columns of a warp read the
//     same pieces);
//   - a chunk's outputs are staged in shared memory and stored as 64-byte rows
//     (fp32 o and/or its bf16 rounding, the gate mix's lin input);
//   - the state tile is read and written once, through shared memory, in
//     64-byte rows (state_out may alias state_in: each block owns its tile).
// Every sum is fp32 in a fixed order, so results are deterministic.
#include <algorithm>

#include "esa_device.cuh"
#include "esa_internal.h"

namespace esa {

namespace {

constexpr int kNS = 8;  // lanes per value column
constexpr int kKdaWarps = 4;
constexpr int kKdaThreads = kKdaWarps * 32;
constexpr int kColsB = kKdaThreads / kNS;  // value columns per block (16)

template <int DK, int CT>
struct KdaLayout {
    static constexpr int R = DK / kNS;  // key channels per lane
    static constexpr int Q = 0;         // bf16 [CT][DK], pieces permuted (below)
    static constexpr int K = Q + CT * DK * 2;
    static constexpr int A = K + CT * DK * 2;         // fp32 [CT][DK], pieces permuted
    static constexpr int V = A + CT * DK * 4;         // bf16 [CT][kColsB]
    static constexpr int BETA = V + CT * kColsB * 2;  // fp32 [CT]
    static constexpr int IN = (BETA + CT * 4 + 15) / 16 * 16;
    static constexpr int TILE = DK * kColsB * 4;  // the state tile, staged in one buffer
    static constexpr int BUF = IN > TILE ? IN : TILE;
    static constexpr int OUT = 2 * BUF;  // fp32 [2][CT][kColsB]
    static constexpr int TOTAL = OUT + 2 * CT * kColsB * 4;
};

// A row of DK elements of `es` bytes is split into 16-byte pieces; lane slice s
// owns key channels s*R .. s*R+R-1, i.e. pieces s*PPL .. s*PPL+PPL-1. Piece p
// is stored at (p % PPL) * 128 + (p / PPL) * 16, so that for each of its PPL
// pieces the 8 slices read 128 consecutive bytes.
__device__ __forceinline__ uint32_t piece_off(int p, int ppl) { return (p % ppl) * (kNS * 16) + (p / ppl) * 16; }

__device__ __forceinline__ void cp_async4(uint32_t dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

struct KdaArgs {
    const uint16_t *q, *k, *v;
    const float *alpha, *beta, *state_in;
    float *o, *state_out;
    uint16_t *lin;
    long long T;
    int H, Dv;
    float scale;
};

template <int DK, int CT>
__device__ __forceinline__ void kda_issue(uint32_t sb, const KdaArgs &a, long long b, int h, int c0, long long t0,
                                          int n, int tid) {
    using L = KdaLayout<DK, CT>;
    constexpr int PQ = DK * 2 / 16, PA = DK * 4 / 16;  // 16-byte pieces per q/k row, per alpha row
    const long long row0 = (b * a.T + t0) * a.H + h;
    for (int i = tid; i < n * PQ; i += kKdaThreads) {
        const int tt = i / PQ, p = i % PQ;
        const long long row = row0 + (long long)tt * a.H;
        const uint32_t off = tt * DK * 2 + piece_off(p, PQ / kNS);
        cp_async16(sb + L::Q + off, a.q + row * DK + p * 8);
        cp_async16(sb + L::K + off, a.k + row * DK + p * 8);
    }
    for (int i = tid; i < n * PA; i += kKdaThreads) {
        const int tt = i / PA, p = i % PA;
        const long long row = row0 + (long long)tt * a.H;
        cp_async16(sb + L::A + tt * DK * 4 + piece_off(p, PA / kNS), a.alpha + row * DK + p * 4);
    }
    for (int i = tid; i < n * 2; i += kKdaThreads) {  // the block's 16 v values: two pieces
        const int tt = i / 2, p = i % 2;
        const long long row = row0 + (long long)tt * a.H;
        cp_async16(sb + L::V + tt * kColsB * 2 + p * 16, a.v + row * a.Dv + c0 + p * 8);
    }
    for (int i = tid; i < n; i += kKdaThreads) cp_async4(sb + L::BETA + i * 4, a.beta + row0 + (long long)i * a.H);
}

template <int DK, int CT>
__device__ __forceinline__ void kda_store(const float *ob, const KdaArgs &a, long long b, int h, int c0, long long t0,
                                          int n, int tid) {
    for (int i = tid; i < n * (kColsB / 4); i += kKdaThreads) {
        const int tt = i / (kColsB / 4), q4 = i % (kColsB / 4);
        const float4 x = *reinterpret_cast<const float4 *>(ob + tt * kColsB + q4 * 4);
        const long long e = ((b * a.T + t0 + tt) * a.H + h) * (long long)a.Dv + c0 + q4 * 4;
        if (a.o) *reinterpret_cast<float4 *>(a.o + e) = x;
        if (a.lin) *reinterpret_cast<uint2 *>(a.lin + e) = make_uint2(pack_bf16(x.x, x.y), pack_bf16(x.z, x.w));
    }
}

__device__ __forceinline__ float sum8(float x) {  // over the 8 lanes of a column; every lane gets the same bits
    x += __shfl_xor_sync(0xffffffffu, x, 1);
    x += __shfl_xor_sync(0xffffffffu, x, 2);
    x += __shfl_xor_sync(0xffffffffu, x, 4);
    return x;
}

template <int DK, int CT>
__global__ void __launch_bounds__(kKdaThreads) kda_kernel(const KdaArgs a) {
    using L = KdaLayout<DK, CT>;
    constexpr int R = L::R;
    extern __shared__ __align__(128) unsigned char smem[];
    const int tid = threadIdx.x, lane = tid & 31;
    const int cl = (tid >> 5) * (32 / kNS) + lane / kNS;  // block column 0..15
    const int s = lane % kNS;                             // key channels s*R .. s*R+R-1
    const int c0 = blockIdx.x * kColsB, h = blockIdx.y;
    const long long b = blockIdx.z;
    const uint32_t sb = smem_u32(smem);
    const int nch = (int)((a.T + CT - 1) / CT);

    if (nch > 0) kda_issue<DK, CT>(sb, a, b, h, c0, 0, (int)min((long long)CT, a.T), tid);
    cp_async_commit();

    // the state tile [DK][16] through buffer 1 (no copy targets it yet)
    float *tile = reinterpret_cast<float *>(smem + L::BUF);
    const long long sbase = (b * a.H + h) * (long long)DK * a.Dv + c0;
    for (int i = tid; i < DK * (kColsB / 4); i += kKdaThreads) {
        const int r = i / (kColsB / 4), q4 = i % (kColsB / 4);
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (a.state_in) x = *reinterpret_cast<const float4 *>(a.state_in + sbase + (long long)r * a.Dv + q4 * 4);
        *reinterpret_cast<float4 *>(tile + r * kColsB + q4 * 4) = x;
    }
    __syncthreads();
    float st[R];
#pragma unroll
    for (int m = 0; m < R; m++) st[m] = tile[(s * R + m) * kColsB + cl];
    __syncthreads();

    for (int c = 0; c < nch; c++) {
        const long long t0 = (long long)c * CT;
        const int n = (int)min((long long)CT, a.T - t0);
        if (c + 1 < nch)
            kda_issue<DK, CT>(sb + ((c + 1) & 1) * L::BUF, a, b, h, c0, t0 + CT,
                              (int)min((long long)CT, a.T - t0 - CT), tid);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        if (c > 0)
            kda_store<DK, CT>(reinterpret_cast<const float *>(smem + L::OUT) + ((c - 1) & 1) * CT * kColsB, a, b, h,
                              c0, t0 - CT, CT, tid);
        const unsigned char *in = smem + (c & 1) * L::BUF;
        float *ob = reinterpret_cast<float *>(smem + L::OUT) + (c & 1) * CT * kColsB;
        for (int tt = 0; tt < n; tt++) {
            float kf[R], qf[R], af[R];
            const unsigned char *rq = in + L::Q + tt * DK * 2 + s * 16, *rk = in + L::K + tt * DK * 2 + s * 16;
            const unsigned char *ra = in + L::A + tt * DK * 4 + s * 16;
#pragma unroll
            for (int j = 0; j < R / 8; j++) {
                const uint4 wk = *reinterpret_cast<const uint4 *>(rk + j * kNS * 16);
                const uint4 wq = *reinterpret_cast<const uint4 *>(rq + j * kNS * 16);
                const uint32_t ks[4] = {wk.x, wk.y, wk.z, wk.w}, qs[4] = {wq.x, wq.y, wq.z, wq.w};
#pragma unroll
                for (int e = 0; e < 4; e++) {
                    kf[j * 8 + 2 * e] = bf16lo(ks[e]);
                    kf[j * 8 + 2 * e + 1] = bf16hi(ks[e]);
                    qf[j * 8 + 2 * e] = bf16lo(qs[e]);
                    qf[j * 8 + 2 * e + 1] = bf16hi(qs[e]);
                }
            }
#pragma unroll
            for (int j = 0; j < R / 4; j++) {
                const float4 av = *reinterpret_cast<const float4 *>(ra + j * kNS * 16);
                af[j * 4] = av.x;
                af[j * 4 + 1] = av.y;
                af[j * 4 + 2] = av.z;
                af[j * 4 + 3] = av.w;
            }
            const float vc = __uint_as_float((uint32_t)reinterpret_cast<const uint16_t *>(in + L::V)[tt * kColsB + cl]
                                             << 16);
            const float bt = reinterpret_cast<const float *>(in + L::BETA)[tt];
            // forget, then read what the column returns for k_t
            float p[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int m = 0; m < R; m++) {
                st[m] *= af[m];
                p[m & 3] = fmaf(kf[m], st[m], p[m & 3]);
            }
            const float u = sum8((p[0] + p[1]) + (p[2] + p[3]));
            // write beta_t (v_t - u) along k_t, then read out with q_t
            const float d = bt * (vc - u);
            float ov[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int m = 0; m < R; m++) {
                st[m] = fmaf(kf[m], d, st[m]);
                ov[m & 3] = fmaf(qf[m], st[m], ov[m & 3]);
            }
            const float o = sum8((ov[0] + ov[1]) + (ov[2] + ov[3]));
            if (s == 0) ob[tt * kColsB + cl] = o * a.scale;
        }
        __syncthreads();  // buffer c&1 is read; the next chunk may refill it
    }
    if (nch > 0) {
        const long long t0 = (long long)(nch - 1) * CT;
        kda_store<DK, CT>(reinterpret_cast<const float *>(smem + L::OUT) + ((nch - 1) & 1) * CT * kColsB, a, b, h, c0,
                          t0, (int)(a.T - t0), tid);
    }
    if (a.state_out) {
        cp_async_wait<0>();
        __syncthreads();
        float *t2 = reinterpret_cast<float *>(smem);
#pragma unroll
        for (int m = 0; m < R; m++) t2[(s * R + m) * kColsB + cl] = st[m];
        __syncthreads();
        for (int i = tid; i < DK * (kColsB / 4); i += kKdaThreads) {
            const int r = i / (kColsB / 4), q4 = i % (kColsB / 4);
            *reinterpret_cast<float4 *>(a.state_out + sbase + (long long)r * a.Dv + q4 * 4) =
                *reinterpret_cast<const float4 *>(t2 + r * kColsB + q4 * 4);
        }
    }
}

template <int DK, int CT>
esa_status launch_kda_t(const KdaArgs &a, long long B, cudaStream_t st) {
    using L = KdaLayout<DK, CT>;
    const void *fn = reinterpret_cast<const void *>(&kda_kernel<DK, CT>);
    if (!ensure_smem(fn, L::TOTAL)) return ESA_ERR_CUDA;
    dim3 grid((unsigned)(a.Dv / kColsB), (unsigned)a.H, (unsigned)B);
    kda_kernel<DK, CT><<<grid, kKdaThreads, L::TOTAL, st>>>(a);
    return cudaGetLastError() == cudaSuccess ? ESA_OK : ESA_ERR_CUDA;
}

}  // namespace

esa_status launch_kda(const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *alpha, const float *beta,
                      const float *state_in, long long B, long long T, int H, int Dk, int Dv, float scale, float *o,
                      uint16_t *lin, float *state_out, cudaStream_t st) {
    const KdaArgs a{q, k, v, alpha, beta, state_in, o, state_out, lin, T, H, Dv, scale};
    // decode-sized calls stage few steps: a smaller block footprint, more blocks per SM
    const bool small = T <= 4;
    if (Dk == 128) return small ? launch_kda_t<128, 4>(a, B, st) : launch_kda_t<128, 32>(a, B, st);
    if (Dk == 64) return small ? launch_kda_t<64, 4>(a, B, st) : launch_kda_t<64, 32>(a, B, st);
    return ESA_ERR_UNSUPPORTED;
}

}  // namespace esa
