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
// s += beta_t (v_t[c] - k_t . s) k_t. Two kernels:
//   kda_kernel (many steps) holds the state in registers for the whole
//   sequence: NS lanes share CC columns, each lane R = Dk/NS key channels of
//   them (Dk = 128: 16 lanes x 8 channels x 2 columns, or x 1 column when
//   that grid fits on the SMs at one block each; Dk = 64: 8 x 8 x 1); a
//   block of 4 warps holds 16 (or 8) columns of one (sequence, head), grid
//   (Dv/16 or Dv/8, H, B).
//   - The inputs of 32 steps (the head's q, k and alpha rows, the block's v
//     values, beta) are staged in shared memory with cp.async, double
//     buffered, laid out so that the NS lanes of a column group read
//     consecutive 16-byte pieces (no bank conflicts).
//   - Steps go in pairs: both steps' reads are written against the state
//     before the pair (kda_step2), so one shuffle tree over the NS lanes
//     serves two steps; the lanes' shares of q . s go to shared memory and a
//     chunk's outputs are summed in lane order and stored once (fp32 o and/or
//     its bf16 rounding, the gate mix's lin input).
//   - The state tile is read and written once, through shared memory, in
//     whole rows (state_out may alias state_in: each block owns its tile).
//   kda_decode_kernel (at most 4 steps) streams the state through registers
//   once per step in float4 rows (below).
// Every sum is fp32 in a fixed order, so results are deterministic.
#include <algorithm>
#include <mutex>
#include <set>

#include "esa_device.cuh"
#include "esa_internal.h"

namespace esa {

namespace {

constexpr int kKdaWarps = 4;
constexpr int kKdaThreads = kKdaWarps * 32;
constexpr int kCT = 32;          // steps staged per chunk
constexpr int kDecCols = 16;     // value columns per decode block
constexpr int kDecodeSteps = 4;  // calls with at most this many steps stream the state once per step

// NS lanes share CC value columns, R = DK / NS key channels each; a block
// holds COLS = 128 / NS * CC columns of one head.
template <int DK, int NS, int CC>
struct KdaLayout {
    static constexpr int R = DK / NS;
    static constexpr int COLS = kKdaThreads / NS * CC;
    static constexpr int Q = 0;  // bf16 [kCT][DK], pieces permuted (below)
    static constexpr int K = Q + kCT * DK * 2;
    static constexpr int A = K + kCT * DK * 2;       // fp32 [kCT][DK], pieces permuted
    static constexpr int V = A + kCT * DK * 4;       // bf16 [kCT][COLS]
    static constexpr int BETA = V + kCT * COLS * 2;  // fp32 [kCT]
    static constexpr int IN = (BETA + kCT * 4 + 15) / 16 * 16;
    static constexpr int TILE = DK * COLS * 4;  // the state tile, staged in one buffer
    static constexpr int BUF = IN > TILE ? IN : TILE;
    static constexpr int PART = 2 * BUF;  // fp32 [kCT][COLS][NS]: per-lane shares of q . s
    static constexpr int TOTAL = PART + kCT * COLS * NS * 4;
    static_assert(R % 8 == 0 && COLS % 8 == 0, "whole 16-byte pieces per lane and per v row");
};

// A row of DK elements of `es` bytes is split into 16-byte pieces; lane slice s
// owns key channels s*R .. s*R+R-1, i.e. pieces s*PPL .. s*PPL+PPL-1. Piece p
// is stored at (p % PPL) * NS * 16 + (p / PPL) * 16, so that for each of its
// PPL pieces the NS slices read NS * 16 consecutive bytes.
template <int NS>
__device__ __forceinline__ uint32_t piece_off(int p, int ppl) {
    return (p % ppl) * (NS * 16) + (p / ppl) * 16;
}

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

template <int DK, int NS, int CC>
__device__ __forceinline__ void kda_issue(uint32_t sb, const KdaArgs &a, long long b, int h, int c0, long long t0,
                                          int n, int tid) {
    using L = KdaLayout<DK, NS, CC>;
    constexpr int PQ = DK * 2 / 16, PA = DK * 4 / 16;  // 16-byte pieces per q/k row, per alpha row
    constexpr int PV = L::COLS * 2 / 16;                // per row of the block's v values
    const long long row0 = (b * a.T + t0) * a.H + h;
    for (int i = tid; i < n * PQ; i += kKdaThreads) {
        const int tt = i / PQ, p = i % PQ;
        const long long row = row0 + (long long)tt * a.H;
        const uint32_t off = tt * DK * 2 + piece_off<NS>(p, PQ / NS);
        cp_async16(sb + L::Q + off, a.q + row * DK + p * 8);
        cp_async16(sb + L::K + off, a.k + row * DK + p * 8);
    }
    for (int i = tid; i < n * PA; i += kKdaThreads) {
        const int tt = i / PA, p = i % PA;
        const long long row = row0 + (long long)tt * a.H;
        cp_async16(sb + L::A + tt * DK * 4 + piece_off<NS>(p, PA / NS), a.alpha + row * DK + p * 4);
    }
    for (int i = tid; i < n * PV; i += kKdaThreads) {
        const int tt = i / PV, p = i % PV;
        const long long row = row0 + (long long)tt * a.H;
        cp_async16(sb + L::V + tt * L::COLS * 2 + p * 16, a.v + row * a.Dv + c0 + p * 8);
    }
    for (int i = tid; i < n; i += kKdaThreads) cp_async4(sb + L::BETA + i * 4, a.beta + row0 + (long long)i * a.H);
}

// One step's operands for a lane: its R key channels of k_t, q_t and alpha_t,
// v_t of its CC columns, beta_t.
template <int R, int CC>
struct StepIn {
    float k[R], q[R], a[R], v[CC], b;
};

template <int DK, int NS, int CC>
__device__ __forceinline__ void load_step(const unsigned char *in, int tt, int s, int cl,
                                          StepIn<DK / NS, CC> &x) {
    using L = KdaLayout<DK, NS, CC>;
    constexpr int R = L::R;
    const unsigned char *rq = in + L::Q + tt * DK * 2 + s * 16, *rk = in + L::K + tt * DK * 2 + s * 16;
    const unsigned char *ra = in + L::A + tt * DK * 4 + s * 16;
#pragma unroll
    for (int j = 0; j < R / 8; j++) {
        const uint4 wk = *reinterpret_cast<const uint4 *>(rk + j * NS * 16);
        const uint4 wq = *reinterpret_cast<const uint4 *>(rq + j * NS * 16);
        const uint32_t ks[4] = {wk.x, wk.y, wk.z, wk.w}, qs[4] = {wq.x, wq.y, wq.z, wq.w};
#pragma unroll
        for (int e = 0; e < 4; e++) {
            x.k[j * 8 + 2 * e] = bf16lo(ks[e]);
            x.k[j * 8 + 2 * e + 1] = bf16hi(ks[e]);
            x.q[j * 8 + 2 * e] = bf16lo(qs[e]);
            x.q[j * 8 + 2 * e + 1] = bf16hi(qs[e]);
        }
    }
#pragma unroll
    for (int j = 0; j < R / 4; j++) {
        const float4 av = *reinterpret_cast<const float4 *>(ra + j * NS * 16);
        x.a[j * 4] = av.x;
        x.a[j * 4 + 1] = av.y;
        x.a[j * 4 + 2] = av.z;
        x.a[j * 4 + 3] = av.w;
    }
#pragma unroll
    for (int cc = 0; cc < CC; cc++)
        x.v[cc] = __uint_as_float((uint32_t)reinterpret_cast<const uint16_t *>(in + L::V)[tt * L::COLS + cl * CC + cc]
                                  << 16);
    x.b = reinterpret_cast<const float *>(in + L::BETA)[tt];
}

// One step for this lane's R key channels of its CC columns: forget, read
// u = k_t . s (summed over the columns' NS lanes; the CC sums interleave),
// write beta_t (v_t - u) along k_t, and store this lane's share of q_t . s for
// each column (share[cc * NS]). The products k*alpha and alpha*s do not wait
// for the previous step's sums.
template <int R, int NS, int CC>
__device__ __forceinline__ void kda_step(const StepIn<R, CC> &x, float (&st)[CC][R], float *share) {
    float ka[R], u[CC], sa[CC][R];
#pragma unroll
    for (int m = 0; m < R; m++) ka[m] = x.k[m] * x.a[m];
#pragma unroll
    for (int cc = 0; cc < CC; cc++) {
        float p[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int m = 0; m < R; m++) {
            p[m & 3] = fmaf(ka[m], st[cc][m], p[m & 3]);
            sa[cc][m] = st[cc][m] * x.a[m];
        }
        u[cc] = (p[0] + p[1]) + (p[2] + p[3]);
    }
#pragma unroll
    for (int off = 1; off < NS; off <<= 1)
#pragma unroll
        for (int cc = 0; cc < CC; cc++) u[cc] += __shfl_xor_sync(0xffffffffu, u[cc], off);
#pragma unroll
    for (int cc = 0; cc < CC; cc++) {
        const float d = x.b * (x.v[cc] - u[cc]);
        float ov[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int m = 0; m < R; m++) {
            st[cc][m] = fmaf(x.k[m], d, sa[cc][m]);
            ov[m & 3] = fmaf(x.q[m], st[cc][m], ov[m & 3]);
        }
        share[cc * NS] = (ov[0] + ov[1]) + (ov[2] + ov[3]);
    }
}

// Two steps t, t+1 with one lane-sum tree. From the state s before step t,
//   u_t     = (k_t a_t) . s
//   u_{t+1} = k_{t+1} . (a_{t+1} * (a_t * s + k_t d_t))
//           = (k_{t+1} a_{t+1} a_t) . s + d_t ((k_{t+1} a_{t+1}) . k_t),
// so the lane shares of (k_t a_t).s and (k_{t+1} a_{t+1} a_t).s for each
// column and of the column-free (k_{t+1} a_{t+1}).k_t are summed over the NS
// lanes together: one shuffle chain per two steps instead of two.
template <int R, int NS, int CC>
__device__ __forceinline__ void kda_step2(const StepIn<R, CC> &x0, const StepIn<R, CC> &x1, float (&st)[CC][R],
                                          float *share0, float *share1) {
    float kk1[R], red[2 * CC + 1];
#pragma unroll
    for (int m = 0; m < R; m++) kk1[m] = x1.k[m] * x1.a[m];
    {
        float pa[2] = {0.f, 0.f};
#pragma unroll
        for (int m = 0; m < R; m++) pa[m & 1] = fmaf(kk1[m], x0.k[m], pa[m & 1]);
        red[2 * CC] = pa[0] + pa[1];
    }
#pragma unroll
    for (int cc = 0; cc < CC; cc++) {
        float p0[2] = {0.f, 0.f}, p1[2] = {0.f, 0.f};
#pragma unroll
        for (int m = 0; m < R; m++) {
            p0[m & 1] = fmaf(x0.k[m] * x0.a[m], st[cc][m], p0[m & 1]);
            p1[m & 1] = fmaf(kk1[m] * x0.a[m], st[cc][m], p1[m & 1]);
        }
        red[cc] = p0[0] + p0[1];
        red[CC + cc] = p1[0] + p1[1];
    }
#pragma unroll
    for (int off = 1; off < NS; off <<= 1)
#pragma unroll
        for (int i = 0; i < 2 * CC + 1; i++) red[i] += __shfl_xor_sync(0xffffffffu, red[i], off);
#pragma unroll
    for (int cc = 0; cc < CC; cc++) {
        const float d0 = x0.b * (x0.v[cc] - red[cc]);
        const float d1 = x1.b * (x1.v[cc] - fmaf(red[2 * CC], d0, red[CC + cc]));
        float o0[2] = {0.f, 0.f}, o1[2] = {0.f, 0.f};
#pragma unroll
        for (int m = 0; m < R; m++) {
            float v = fmaf(x0.k[m], d0, st[cc][m] * x0.a[m]);
            o0[m & 1] = fmaf(x0.q[m], v, o0[m & 1]);
            v = fmaf(x1.k[m], d1, v * x1.a[m]);
            o1[m & 1] = fmaf(x1.q[m], v, o1[m & 1]);
            st[cc][m] = v;
        }
        share0[cc * NS] = o0[0] + o0[1];
        share1[cc * NS] = o1[0] + o1[1];
    }
}

template <int DK, int NS, int CC>
__global__ void __launch_bounds__(kKdaThreads) kda_kernel(const KdaArgs a) {
    using L = KdaLayout<DK, NS, CC>;
    constexpr int R = L::R, COLS = L::COLS;
    extern __shared__ __align__(128) unsigned char smem[];
    const int tid = threadIdx.x, lane = tid & 31;
    const int cl = (tid >> 5) * (32 / NS) + lane / NS;  // block columns cl*CC .. cl*CC+CC-1
    const int s = lane % NS;                            // key channels s*R .. s*R+R-1
    const int c0 = blockIdx.x * COLS, h = blockIdx.y;
    const long long b = blockIdx.z;
    const uint32_t sb = smem_u32(smem);
    const int nch = (int)((a.T + kCT - 1) / kCT);

    if (nch > 0) kda_issue<DK, NS, CC>(sb, a, b, h, c0, 0, (int)min((long long)kCT, a.T), tid);
    cp_async_commit();

    // the state tile [DK][COLS] through buffer 1 (no copy targets it yet)
    float *tile = reinterpret_cast<float *>(smem + L::BUF);
    const long long sbase = (b * a.H + h) * (long long)DK * a.Dv + c0;
    for (int i = tid; i < DK * (COLS / 4); i += kKdaThreads) {
        const int r = i / (COLS / 4), q4 = i % (COLS / 4);
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (a.state_in) x = *reinterpret_cast<const float4 *>(a.state_in + sbase + (long long)r * a.Dv + q4 * 4);
        *reinterpret_cast<float4 *>(tile + r * COLS + q4 * 4) = x;
    }
    __syncthreads();
    float st[CC][R];
#pragma unroll
    for (int cc = 0; cc < CC; cc++)
#pragma unroll
        for (int m = 0; m < R; m++) st[cc][m] = tile[(s * R + m) * COLS + cl * CC + cc];
    __syncthreads();

    float *part = reinterpret_cast<float *>(smem + L::PART);
    for (int c = 0; c < nch; c++) {
        const long long t0 = (long long)c * kCT;
        const int n = (int)min((long long)kCT, a.T - t0);
        if (c + 1 < nch)
            kda_issue<DK, NS, CC>(sb + ((c + 1) & 1) * L::BUF, a, b, h, c0, t0 + kCT,
                              (int)min((long long)kCT, a.T - t0 - kCT), tid);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        const unsigned char *in = smem + (c & 1) * L::BUF;
        // shares [kCT][COLS][NS]: this lane's column cl*CC+cc at (cl*CC+cc)*NS + s
        float *my = part + cl * CC * NS + s;
        // steps in pairs; two operand-set pairs alternate so that the next
        // pair's operands are read while this pair's chain runs; an odd last
        // step runs alone
        StepIn<R, CC> xa0, xa1, xb0, xb1;
        load_step<DK, NS, CC>(in, 0, s, cl, xa0);
        load_step<DK, NS, CC>(in, min(1, n - 1), s, cl, xa1);
        int tt = 0;
        while (tt + 1 < n) {
            load_step<DK, NS, CC>(in, min(tt + 2, n - 1), s, cl, xb0);
            load_step<DK, NS, CC>(in, min(tt + 3, n - 1), s, cl, xb1);
            kda_step2<R, NS, CC>(xa0, xa1, st, my + tt * COLS * NS, my + (tt + 1) * COLS * NS);
            tt += 2;
            if (tt + 1 >= n) {
                if (tt < n) kda_step<R, NS, CC>(xb0, st, my + tt * COLS * NS);
                tt = n;
                break;
            }
            load_step<DK, NS, CC>(in, min(tt + 2, n - 1), s, cl, xa0);
            load_step<DK, NS, CC>(in, min(tt + 3, n - 1), s, cl, xa1);
            kda_step2<R, NS, CC>(xb0, xb1, st, my + tt * COLS * NS, my + (tt + 1) * COLS * NS);
            tt += 2;
        }
        if (tt < n) kda_step<R, NS, CC>(xa0, st, my + tt * COLS * NS);
        __syncthreads();  // the shares are complete; buffer c&1 is read and may be refilled
        // o_t[c] = scale * (the NS shares, in lane order); COLS consecutive
        // threads write one step's columns
        for (int i = tid; i < n * COLS; i += kKdaThreads) {
            const int tt = i / COLS, col = i % COLS;
            const float *pp = part + (tt * COLS + col) * NS;
            float o = pp[0];
#pragma unroll
            for (int j = 1; j < NS; j++) o += pp[j];
            o *= a.scale;
            const long long e = ((b * a.T + t0 + tt) * a.H + h) * (long long)a.Dv + c0 + col;
            if (a.o) a.o[e] = o;
            if (a.lin) a.lin[e] = (uint16_t)(pack_bf16(o, 0.f) & 0xffffu);
        }
    }
    if (a.state_out) {
        cp_async_wait<0>();
        __syncthreads();
        float *t2 = reinterpret_cast<float *>(smem);
#pragma unroll
        for (int cc = 0; cc < CC; cc++)
#pragma unroll
            for (int m = 0; m < R; m++) t2[(s * R + m) * COLS + cl * CC + cc] = st[cc][m];
        __syncthreads();
        for (int i = tid; i < DK * (COLS / 4); i += kKdaThreads) {
            const int r = i / (COLS / 4), q4 = i % (COLS / 4);
            *reinterpret_cast<float4 *>(a.state_out + sbase + (long long)r * a.Dv + q4 * 4) =
                *reinterpret_cast<const float4 *>(t2 + r * COLS + q4 * 4);
        }
    }
}

// A few steps (decode): the state streams through registers once. Block =
// 128 threads = 16 columns of one (sequence, head); thread (rg = tid / 4,
// cg = tid % 4) holds rows rg + 32 j and columns 4 cg .. 4 cg + 3 as float4,
// so each warp load reads 8 rows x 64 contiguous bytes. Per step, with
// S' = alpha * S (per row):
//   u[c] = sum_i (alpha_i k_i) S[i][c],  z[c] = sum_i (alpha_i q_i) S[i][c],
// summed over the thread's rows, then over the warp's 8 row groups (shuffles)
// and the 4 warps (shared memory, in warp order); then
//   d[c] = beta (v[c] - u[c]),  o[c] = scale (z[c] + (q . k) d[c]),
//   S[i][c] = alpha_i S[i][c] + k_i d[c].
constexpr int kDecRowGroups = kKdaThreads / 4;

template <int DK>
__global__ void __launch_bounds__(kKdaThreads) kda_decode_kernel(const KdaArgs a) {
    constexpr int RJ = DK / kDecRowGroups;  // rows per thread
    __shared__ float red[kKdaWarps][2 * kDecCols + 1];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rg = tid >> 2, cg = tid & 3;
    const int c0 = blockIdx.x * kDecCols, h = blockIdx.y;
    const long long b = blockIdx.z;
    const long long sbase = (b * a.H + h) * (long long)DK * a.Dv + c0 + cg * 4;
    // launched as a programmatic dependent: the next launch in the stream may
    // be scheduled now, and this one reads nothing before the previous work
    // in the stream has completed
    pdl_launch_dependents();
    pdl_wait();
    float4 S[RJ];
#pragma unroll
    for (int j = 0; j < RJ; j++)
        S[j] = a.state_in ? *reinterpret_cast<const float4 *>(a.state_in + sbase + (long long)(rg + kDecRowGroups * j) * a.Dv)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
    for (long long t = 0; t < a.T; t++) {
        const long long row = (b * a.T + t) * a.H + h;
        float al[RJ], kk[RJ];
        float u[4] = {0.f, 0.f, 0.f, 0.f}, z[4] = {0.f, 0.f, 0.f, 0.f}, qk = 0.f;
#pragma unroll
        for (int j = 0; j < RJ; j++) {
            const int i = rg + kDecRowGroups * j;
            al[j] = a.alpha[row * DK + i];
            kk[j] = __uint_as_float((uint32_t)a.k[row * DK + i] << 16);
            const float qq = __uint_as_float((uint32_t)a.q[row * DK + i] << 16);
            const float ak = al[j] * kk[j], aq = al[j] * qq;
            if (cg == 0) qk = fmaf(qq, kk[j], qk);
            u[0] = fmaf(ak, S[j].x, u[0]);
            u[1] = fmaf(ak, S[j].y, u[1]);
            u[2] = fmaf(ak, S[j].z, u[2]);
            u[3] = fmaf(ak, S[j].w, u[3]);
            z[0] = fmaf(aq, S[j].x, z[0]);
            z[1] = fmaf(aq, S[j].y, z[1]);
            z[2] = fmaf(aq, S[j].z, z[2]);
            z[3] = fmaf(aq, S[j].w, z[3]);
        }
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
#pragma unroll
            for (int e = 0; e < 4; e++) {
                u[e] += __shfl_xor_sync(0xffffffffu, u[e], off);
                z[e] += __shfl_xor_sync(0xffffffffu, z[e], off);
            }
            qk += __shfl_xor_sync(0xffffffffu, qk, off);
        }
        if (lane < 4) {
#pragma unroll
            for (int e = 0; e < 4; e++) {
                red[warp][cg * 4 + e] = u[e];
                red[warp][kDecCols + cg * 4 + e] = z[e];
            }
            if (lane == 0) red[warp][2 * kDecCols] = qk;
        }
        __syncthreads();
        float U[4], Z[4];
        qk = red[0][2 * kDecCols];
#pragma unroll
        for (int e = 0; e < 4; e++) {
            U[e] = red[0][cg * 4 + e];
            Z[e] = red[0][kDecCols + cg * 4 + e];
        }
#pragma unroll
        for (int w = 1; w < kKdaWarps; w++) {
            qk += red[w][2 * kDecCols];
#pragma unroll
            for (int e = 0; e < 4; e++) {
                U[e] += red[w][cg * 4 + e];
                Z[e] += red[w][kDecCols + cg * 4 + e];
            }
        }
        __syncthreads();  // red is rewritten by the next step
        const float bt = a.beta[row];
        const uint2 vw = *reinterpret_cast<const uint2 *>(a.v + row * a.Dv + c0 + cg * 4);
        const float vv[4] = {bf16lo(vw.x), bf16hi(vw.x), bf16lo(vw.y), bf16hi(vw.y)};
        float d[4];
#pragma unroll
        for (int e = 0; e < 4; e++) d[e] = bt * (vv[e] - U[e]);
        if (rg == 0) {
            float o[4];
#pragma unroll
            for (int e = 0; e < 4; e++) o[e] = a.scale * fmaf(qk, d[e], Z[e]);
            const long long oe = row * a.Dv + c0 + cg * 4;
            if (a.o) *reinterpret_cast<float4 *>(a.o + oe) = make_float4(o[0], o[1], o[2], o[3]);
            if (a.lin) *reinterpret_cast<uint2 *>(a.lin + oe) = make_uint2(pack_bf16(o[0], o[1]), pack_bf16(o[2], o[3]));
        }
#pragma unroll
        for (int j = 0; j < RJ; j++) {
            S[j].x = fmaf(kk[j], d[0], al[j] * S[j].x);
            S[j].y = fmaf(kk[j], d[1], al[j] * S[j].y);
            S[j].z = fmaf(kk[j], d[2], al[j] * S[j].z);
            S[j].w = fmaf(kk[j], d[3], al[j] * S[j].w);
        }
    }
    if (a.state_out) {
#pragma unroll
        for (int j = 0; j < RJ; j++)
            *reinterpret_cast<float4 *>(a.state_out + sbase + (long long)(rg + kDecRowGroups * j) * a.Dv) = S[j];
    }
}

// the largest shared-memory carveout
bool kda_configure(const void *fn, size_t smem) {
    static std::mutex mu;
    static std::set<std::pair<int, const void *>> done;
    int dev = 0;
    cudaGetDevice(&dev);
    {
        std::lock_guard<std::mutex> lk(mu);
        if (done.count({dev, fn})) return true;
    }
    if (!ensure_smem(fn, smem) ||
        cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    std::lock_guard<std::mutex> lk(mu);
    done.insert({dev, fn});
    return true;
}

template <int DK, int NS, int CC>
esa_status launch_kda_t(const KdaArgs &a, long long B, cudaStream_t st) {
    using L = KdaLayout<DK, NS, CC>;
    const void *fn = reinterpret_cast<const void *>(&kda_kernel<DK, NS, CC>);
    if (!kda_configure(fn, L::TOTAL)) return ESA_ERR_CUDA;
    dim3 grid((unsigned)(a.Dv / L::COLS), (unsigned)a.H, (unsigned)B);
    kda_kernel<DK, NS, CC><<<grid, kKdaThreads, L::TOTAL, st>>>(a);
    return cudaGetLastError() == cudaSuccess ? ESA_OK : ESA_ERR_CUDA;
}

}  // namespace

bool kda_uses_chunks(long long T) { return T > kDecodeSteps; }

esa_status launch_kda(const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *alpha, const float *beta,
                      const float *state_in, long long B, long long T, int H, int Dk, int Dv, float scale, float *o,
                      uint16_t *lin, float *state_out, void *ws, cudaStream_t st) {
    const KdaArgs a{q, k, v, alpha, beta, state_in, o, state_out, lin, T, H, Dv, scale};
    if (ws && kda_uses_chunks(T))
        return launch_kda_chunked(q, k, v, alpha, beta, state_in, B, T, H, Dk, Dv, scale, o, lin, state_out, ws, st);
    if (T <= kDecodeSteps) {  // a few steps: one streaming pass over the state
        const void *fn = Dk == 128 ? reinterpret_cast<const void *>(&kda_decode_kernel<128>)
                                   : reinterpret_cast<const void *>(&kda_decode_kernel<64>);
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3((unsigned)(Dv / kDecCols), (unsigned)H, (unsigned)B);
        cfg.blockDim = dim3(kKdaThreads);
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        void *args[] = {(void *)&a};
        cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
        if (e != cudaSuccess) {  // a plain launch
            cudaGetLastError();
            cfg.numAttrs = 0;
            e = cudaLaunchKernelExC(&cfg, fn, args);
        }
        return e == cudaSuccess ? ESA_OK : ESA_ERR_CUDA;
    }
    // 8 key channels per lane: at Dk = 128, 16 lanes hold two columns each
    // (the operands a lane loads serve both), or one column each when that
    // grid of twice the blocks still gives every block an SM of its own: a
    // block's steps are one dependent chain per warp, so half the columns
    // finish sooner (B1 x 32768 steps, 8 heads: 4.35 ms against 5.52 ms).
    // Two such blocks on one SM issue more instructions for the same columns
    // than one two-column block (16 heads: 6.46 ms against 5.52 ms). At
    // Dk = 64, 8 lanes one column.
    if (Dk == 128) {
        if ((long long)(Dv / 8) * H * B <= device_info().sms) return launch_kda_t<128, 16, 1>(a, B, st);
        return launch_kda_t<128, 16, 2>(a, B, st);
    }
    if (Dk == 64) return launch_kda_t<64, 8, 1>(a, B, st);
    return ESA_ERR_UNSUPPORTED;
}

}  // namespace esa
