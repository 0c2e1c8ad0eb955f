// KDA, chunked form: the same recurrence as k_kda.cu, computed chunk by chunk
// of kC steps so that the work of a chunk is a few small matrix products
// instead of kC dependent steps.
//
// Method: the Gated DSA page ("超大规模MoE架构中稀疏注意力机制的演进与实践",
// sections 一, 二.3 and 三) keeps KDA, a gated linear attention, beside the
// sparse attention; the recurrence is the published Kimi Delta Attention one:
//   S = diag(alpha_t) S;  u = S^T k_t;  S += beta_t k_t (v_t - u)^T;
//   o_t = scale S^T q_t.
// Within a chunk whose steps are t = 0 .. C-1 (rows of K, Q, V, alpha), with
// g_t = alpha_0 * ... * alpha_t per key channel (G its rows) and S the state
// before the chunk, unrolling the steps gives
//   Kt = K * G, Qt = Q * G, Ki = K / G                       (per channel)
//   A  = strictly-lower(Kt Ki^T),  Bm = lower(Qt Ki^T)        (C x C)
//   D  = (I + diag(beta) A)^-1 diag(beta) (V - Kt S)          (the writes)
//   O  = scale (Qt S + Bm D)
//   S' = g_last * S + (Ki * g_last)^T D.
// With M = (I + diag(beta) A)^-1 diag(beta) (lower triangular, solved by
// forward substitution), Wk = M Kt, U = M V, Qp = Qt - Bm Wk, Up = Bm U:
//   D = U - Wk S,   O = scale (Qp S + Up),   S' = g_last * S + Kl^T D
// where Kl = Ki * g_last. Everything but S is known before the chunk starts.
// Two kernels per segment of up to kSegChunks chunks:
//   kda_prep_kernel: one block per (sequence, head, chunk), all chunks in
//   parallel; computes Wk, Qp, Kl, g_last, U, Up and writes them to the
//   workspace (a chunk record). A chunk in which some g leaves
//   [2^-60, 2^60] (a forgetting factor near 0, or not finite) would make
//   K / G overflow: its record is flagged and the scan runs its steps one by
//   one instead.
//   kda_scan_kernel: one block per (sequence, head, 16 value columns); the
//   state slice (Dk x 16) stays on chip for the whole segment, in warp-MMA
//   accumulators; per chunk X = [Wk; Qp] S (2C x 16, the one product over
//   Dk), then D and O, then S' = g_last * S + Kl^T D. Both products run on
//   the tensor cores (mma.sync, tf32): each fp32 operand is split into two
//   tf32 parts and three products are summed, which keeps near-fp32
//   accuracy (within 2^-19 relative per product).
//   A block's part of a chunk record is two contiguous pieces, brought in by
//   bulk copies up to kStages chunks ahead: a copy warp posts them, eight
//   compute warps consume them.
// Padded steps of a ragged last chunk have k = q = 0, alpha = 1, beta = 0:
// they write nothing and forget nothing. Every sum is fp32 in a fixed order.
#include <climits>

#include "esa_device.cuh"
#include "esa_internal.h"

namespace esa {

namespace {

constexpr int kC = 16;             // steps per chunk
constexpr int kNC = 16;            // value columns per scan block
constexpr int kPrepThreads = 128;
constexpr int kScanThreads = 256;  // the scan's compute threads (a copy warp besides)
constexpr int kSegChunks = 256;    // chunks per prep + scan pair
constexpr int kStages = 3;         // chunk records in flight per scan block
constexpr float kGLo = 0x1p-60f, kGHi = 0x1p60f;

// Chunk record, fp32 words. The part every column block reads, rows padded
// as the scan keeps them in shared memory (so that the warp-MMA operand
// reads hit 32 different banks):
//   Wk [kC][Dk+4], Qp [kC][Dk+4], Kl [kC][Dk+8], g_last [Dk], flag (one
//   word, padded to four)
// then, per block of 16 value columns, U [kC][16] and Up [kC][16].
__host__ __device__ constexpr int rec_a_floats(int Dk) { return 2 * kC * (Dk + 4) + kC * (Dk + 8) + Dk + 4; }
__host__ __device__ inline long long rec_floats(int Dk, int Dv) { return rec_a_floats(Dk) + 2LL * kC * Dv; }

struct ChunkArgs {
    const uint16_t *q, *k, *v;
    const float *alpha, *beta;
    const float *src;  // state before the segment (NULL: zero)
    float *dst;        // state after the segment (NULL: dropped)
    float *o;
    uint16_t *lin;
    float *rec;         // records of this segment: [B][H][seg_cap]
    int32_t *status;    // the workspace status word
    long long wait_ns;  // limit of a wait for a chunk record
    int hold_from;      // the copy warp posts no chunk from this one on (a
                        // test's way to make the wait run out; else never)
    long long T;        // steps per sequence
    long long c_begin;  // first chunk of the segment
    int nch;            // chunks in the segment
    int seg_cap;        // records per (sequence, head)
    int H, Dv;
    float scale;
};

__device__ __forceinline__ float bf(uint16_t x) { return __uint_as_float((uint32_t)x << 16); }

// acc[i] = sum_{l <= i} L[i][l] x(l) for a lower-triangular kC x kC matrix
// L held transposed in shared memory (LT[l][i] = L[i][l], rows of MS words,
// 16-byte aligned): column l of L is read four entries at a time (the same
// address in every lane: one broadcast), and every acc[i] adds its terms in
// order of l.
template <int MS, typename X>
__device__ __forceinline__ void tri_cols(const float *LT, X x, float (&acc)[kC]) {
#pragma unroll
    for (int i = 0; i < kC; i++) acc[i] = 0.f;
#pragma unroll
    for (int l = 0; l < kC; l++) {
        const float xl = x(l);
#pragma unroll
        for (int i4 = l / 4 * 4; i4 < kC; i4 += 4) {
            const float4 m = *reinterpret_cast<const float4 *>(LT + l * MS + i4);
            if (i4 >= l) acc[i4] = fmaf(m.x, xl, acc[i4]);
            if (i4 + 1 >= l) acc[i4 + 1] = fmaf(m.y, xl, acc[i4 + 1]);
            if (i4 + 2 >= l) acc[i4 + 2] = fmaf(m.z, xl, acc[i4 + 2]);
            acc[i4 + 3] = fmaf(m.w, xl, acc[i4 + 3]);
        }
    }
}

// Prep block shared memory, in floats: Kt, Qt, Ki (rows padded), A, Bm^T,
// M^T (rows of kC + 4), beta, then the chunk's raw inputs staged by cp.async:
// k, q (bf16 [kC][Dk]), alpha (fp32 [kC][Dk]), v (bf16 [kC][Dv], last: its
// size depends on Dv).
template <int DK>
struct PrepLayout {
    static constexpr int P = DK + 4, MS = kC + 4;
    static constexpr int KT = 0, QT = KT + kC * P, KI = QT + kC * P, AM = KI + kC * P, BM = AM + kC * MS;
    static constexpr int MM = BM + kC * MS, SB = MM + kC * MS, RK = SB + kC, RQ = RK + kC * DK / 2;
    static constexpr int RA = RQ + kC * DK / 2, RV = RA + kC * DK;
    static size_t bytes(int Dv) { return (size_t)(RV + kC * Dv / 2) * 4; }
    static_assert(RK % 4 == 0 && RQ % 4 == 0 && RA % 4 == 0 && RV % 4 == 0, "16-byte aligned staging");
};

template <int DK>
__global__ void __launch_bounds__(kPrepThreads, 4) kda_prep_kernel(const ChunkArgs a) {
    using L = PrepLayout<DK>;
    constexpr int P = L::P, MS = L::MS;
    extern __shared__ __align__(128) float sm[];
    float *Kt = sm + L::KT, *Qt = sm + L::QT, *Ki = sm + L::KI, *Am = sm + L::AM, *BmT = sm + L::BM, *MT = sm + L::MM;
    float *sb = sm + L::SB;
    const uint16_t *RKs = reinterpret_cast<const uint16_t *>(sm + L::RK);
    const uint16_t *RQs = reinterpret_cast<const uint16_t *>(sm + L::RQ);
    const uint16_t *RVs = reinterpret_cast<const uint16_t *>(sm + L::RV);
    const float *RAs = sm + L::RA;
    const int tid = threadIdx.x, h = blockIdx.y;
    const long long b = blockIdx.z;
    const long long t0 = (a.c_begin + blockIdx.x) * kC;
    const int n = (int)min((long long)kC, a.T - t0);
    const int Dv = a.Dv;
    float *rec = a.rec + ((b * a.H + h) * a.seg_cap + blockIdx.x) * rec_floats(DK, Dv);
    constexpr int PK = DK + 8;
    float *Wk = rec, *Qp = rec + kC * P, *Kl = rec + 2 * kC * P, *gl = Kl + kC * PK;
    float *Ucol = rec + rec_a_floats(DK);  // [Dv/16][U, Up][kC][16]
    if (a.status && a.c_begin == 0 && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && threadIdx.x == 0)
        *a.status = 0;  // this call's status starts clear (the scans run after this kernel)

    // stage the chunk's k, q, alpha and v rows (steps past the end: zeros)
    {
        const long long row0 = (b * a.T + t0) * a.H + h;
        constexpr int PK = DK / 8, PA = DK / 4;  // 16-byte pieces per k (q) row, per alpha row
        const int PV = Dv / 8;
        for (int p = tid; p < kC * (2 * PK + PA); p += kPrepThreads) {
            const int t = p / (2 * PK + PA), r = p % (2 * PK + PA);
            const bool ok = t < n;
            const long long row = row0 + (long long)(ok ? t : 0) * a.H;
            if (r < PK)
                cp_async16_zfill(smem_u32(sm + L::RK + t * DK / 2 + 4 * r), a.k + row * DK + 8 * r, ok);
            else if (r < 2 * PK)
                cp_async16_zfill(smem_u32(sm + L::RQ + t * DK / 2 + 4 * (r - PK)), a.q + row * DK + 8 * (r - PK), ok);
            else
                cp_async16_zfill(smem_u32(sm + L::RA + t * DK + 4 * (r - 2 * PK)), a.alpha + row * DK + 4 * (r - 2 * PK),
                                 ok);
        }
        for (int p = tid; p < kC * PV; p += kPrepThreads) {
            const int t = p / PV, r = p % PV;
            const bool ok = t < n;
            const long long row = row0 + (long long)(ok ? t : 0) * a.H;
            cp_async16_zfill(smem_u32(sm + L::RV + t * Dv / 2 + 4 * r), a.v + row * Dv + 8 * r, ok);
        }
        cp_async_commit();
        if (tid < kC) sb[tid] = tid < n ? a.beta[row0 + (long long)tid * a.H] : 0.f;
        cp_async_wait<0>();
        __syncthreads();
    }

    // g, Kt, Qt, Ki, Kl per key channel
    bool bad = false;
    if (tid < DK) {
        const int d = tid;
        float g = 1.f;
#pragma unroll
        for (int t = 0; t < kC; t++) {
            const float al = t < n ? RAs[t * DK + d] : 1.f;
            const float kv = bf(RKs[t * DK + d]), qv = bf(RQs[t * DK + d]);
            g *= al;
            bad |= !(g >= kGLo && g <= kGHi);
            Kt[t * P + d] = kv * g;
            Qt[t * P + d] = qv * g;
            Ki[t * P + d] = __fdividef(kv, g);  // g in [2^-60, 2^60] unless flagged
        }
        gl[d] = g;
#pragma unroll
        for (int t = 0; t < kC; t++) Kl[t * PK + d] = Ki[t * P + d] * g;
    }
    const int flagged = __syncthreads_or(bad);

    // A = strictly-lower(Kt Ki^T), Bm = lower(Qt Ki^T): only the 2 x 2 tiles
    // on or below the diagonal (36 of each), one per thread; the entries
    // above the diagonal are never read
    if (tid < 72) {
        const int which = tid / 36;
        int tq = tid % 36, I = 0;
        while (tq > I) tq -= ++I;  // tile (I, J = tq), J <= I
        const int J = tq;
        const float *x0 = (which ? Qt : Kt) + 2 * I * P, *x1 = x0 + P;
        const float *y0 = Ki + 2 * J * P, *y1 = y0 + P;
        float s00 = 0.f, s01 = 0.f, s10 = 0.f, s11 = 0.f;
#pragma unroll 4
        for (int d = 0; d < DK; d += 4) {
            const float4 a0 = *reinterpret_cast<const float4 *>(x0 + d), a1 = *reinterpret_cast<const float4 *>(x1 + d);
            const float4 b0 = *reinterpret_cast<const float4 *>(y0 + d), b1 = *reinterpret_cast<const float4 *>(y1 + d);
            s00 = fmaf(a0.x, b0.x, s00); s00 = fmaf(a0.y, b0.y, s00); s00 = fmaf(a0.z, b0.z, s00); s00 = fmaf(a0.w, b0.w, s00);
            s01 = fmaf(a0.x, b1.x, s01); s01 = fmaf(a0.y, b1.y, s01); s01 = fmaf(a0.z, b1.z, s01); s01 = fmaf(a0.w, b1.w, s01);
            s10 = fmaf(a1.x, b0.x, s10); s10 = fmaf(a1.y, b0.y, s10); s10 = fmaf(a1.z, b0.z, s10); s10 = fmaf(a1.w, b0.w, s10);
            s11 = fmaf(a1.x, b1.x, s11); s11 = fmaf(a1.y, b1.y, s11); s11 = fmaf(a1.z, b1.z, s11); s11 = fmaf(a1.w, b1.w, s11);
        }
        // A as is, Bm transposed; A keeps j < i, Bm j <= i
        const int lo = which ? 0 : 1, si = which ? 1 : MS, sj = which ? MS : 1;
        float *R = (which ? BmT : Am) + 2 * I * si + 2 * J * sj;
        R[0] = 2 * J <= 2 * I - lo ? s00 : 0.f;
        R[sj] = 2 * J + 1 <= 2 * I - lo ? s01 : 0.f;
        R[si] = 2 * J <= 2 * I + 1 - lo ? s10 : 0.f;
        R[si + sj] = 2 * J + 1 <= 2 * I + 1 - lo ? s11 : 0.f;
    }
    __syncthreads();

    // M = (I + diag(beta) A)^-1 diag(beta): column j by thread j, forward
    // substitution M[i][j] = beta_i (delta_ij - sum_{l<i} A[i][l] M[l][j]),
    // each new M[i][j] added at once into the sums of the rows below
    if (tid < kC) {
        const int j = tid;
        float acc[kC];
#pragma unroll
        for (int i = 0; i < kC; i++) acc[i] = 0.f;
#pragma unroll
        for (int i = 0; i < kC; i++) {
            const float m = sb[i] * ((i == j ? 1.f : 0.f) - acc[i]);
            MT[j * MS + i] = m;
#pragma unroll
            for (int l = i + 1; l < kC; l++) acc[l] = fmaf(Am[l * MS + i], m, acc[l]);
        }
    }
    __syncthreads();

    // Wk = M Kt, Qp = Qt - Bm Wk, per key channel
    if (tid < DK) {
        const int d = tid;
        float wk[kC], bw[kC];
        tri_cols<MS>(MT, [&](int l) { return Kt[l * P + d]; }, wk);
#pragma unroll
        for (int i = 0; i < kC; i++) Wk[i * P + d] = wk[i];
        tri_cols<MS>(BmT, [&](int l) { return wk[l]; }, bw);
#pragma unroll
        for (int i = 0; i < kC; i++) Qp[i * P + d] = Qt[i * P + d] - bw[i];
    }
    // U = M V, Up = Bm U, per value column
    for (int c = tid; c < Dv; c += kPrepThreads) {
        // keep the compiler from holding M^T and Bm^T in registers across
        // columns (it would need several hundred)
        asm volatile("" ::: "memory");
        float *U = Ucol + (c / kNC) * 2 * kC * kNC + c % kNC, *Up = U + kC * kNC;
        float u[kC], up[kC];
        tri_cols<MS>(MT, [&](int l) { return bf(RVs[l * Dv + c]); }, u);
#pragma unroll
        for (int i = 0; i < kC; i++) U[i * kNC] = u[i];
        tri_cols<MS>(BmT, [&](int l) { return u[l]; }, up);
#pragma unroll
        for (int i = 0; i < kC; i++) Up[i * kNC] = up[i];
    }
    if (tid == 0) reinterpret_cast<int *>(gl + DK)[0] = flagged;
}

// fp32 x as the sum of two tf32 values, each its leading 11 significant
// bits (the low 13 of the fp32 pattern cleared): hi, then lo from the exact
// remainder x - hi (at most 13 significant bits). |x - hi - lo| < 2^-21 |x|,
// and three tf32 products (hi*hi, hi*lo, lo*hi) give a product to within
// 2^-19 relative, the dropped lo*lo the largest part.
__device__ __forceinline__ void tf32_split(float x, uint32_t &hi, uint32_t &lo) {
    hi = __float_as_uint(x) & 0xffffe000u;
    lo = __float_as_uint(x - __uint_as_float(hi)) & 0xffffe000u;
}
// D(16x8 f32) += A(16x8 tf32, row) * B(8x8 tf32, col)
__device__ __forceinline__ void mma_tf32_1688(float *d, const uint32_t *a, const uint32_t *b) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
// Scan block shared memory, in floats: the state slice transposed (ST, 16
// rows of Dk, padded), kStages chunk stages (a record's shared part, then
// this block's U and Up), D, the split-sum partials, the stage barriers.
template <int DK>
struct ScanLayout {
    static constexpr int P = DK + 4, PK = DK + 8, PD = 24, PR = 24;  // padded rows (banks)
    static constexpr int RA = rec_a_floats(DK);
    static constexpr int WK = 0, QP = WK + kC * P, KL = QP + kC * P, GL = KL + kC * PK, FLAG = GL + DK;
    static constexpr int UU = RA, UP = UU + kC * kNC, STAGE = UP + kC * kNC;
    static constexpr int ST = 0, S0 = ST + kNC * P, DD = S0 + kStages * STAGE, RED = DD + kC * PD;
    static constexpr int BARS = RED + 4 * 2 * kC * PR;  // four K quarters of the 2C x 16 product
    static constexpr size_t BYTES = (size_t)BARS * 4 + 2 * kStages * 8;  // full, then free barriers
    static constexpr int TPD = kScanThreads / DK;  // threads per key channel in the step-by-step path
    static constexpr int CPT = kNC / TPD;          // columns per such thread
    static constexpr int MT = DK / 16;             // 16-row tiles of the state slice
    static constexpr int TPW = MT * 2 / 8;         // state tiles (16 x 8) per warp
    static_assert(FLAG + 4 == RA, "record part A layout");
    static_assert(RA % 4 == 0 && STAGE % 4 == 0 && S0 % 4 == 0 && DD % 4 == 0 && RED % 4 == 0 && BARS % 2 == 0,
                  "16-byte aligned pieces, 8-byte aligned barriers");
    static_assert(CPT % 4 == 0 && TPW >= 1, "thread shapes");
};

// Post chunk j's two pieces on the stage's barrier (one thread).
template <int DK>
__device__ __forceinline__ void scan_issue(float *stage, uint32_t bar, const ChunkArgs &a, long long b, int h, int cb,
                                           int j, uint64_t pol) {
    using L = ScanLayout<DK>;
    const float *rec = a.rec + ((b * a.H + h) * a.seg_cap + j) * rec_floats(DK, a.Dv);
    mbar_expect_tx(bar, (L::RA + 2 * kC * kNC) * 4);
    bulk_g2s(smem_u32(stage), rec, L::RA * 4, bar, pol);
    bulk_g2s(smem_u32(stage + L::UU), rec + L::RA + (long long)cb * 2 * kC * kNC, 2 * kC * kNC * 4, bar, pol);
}

// Barrier 1 over the scan's compute threads only (the copy warp never
// joins): a plain one, and one that also ANDs a flag over them.
__device__ __forceinline__ void cbar() { asm volatile("bar.sync 1, %0;" ::"n"(kScanThreads) : "memory"); }
__device__ __forceinline__ bool cbar_and(bool v) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, 1, %2, p;\n selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)v), "n"(kScanThreads)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Warp MMA fragment coordinates (m16n8k8, tf32): lane = 4 g + t.
//   A (16 x 8): a0 (g, t), a1 (g + 8, t), a2 (g, t + 4), a3 (g + 8, t + 4)
//   B (8 x 8):  b0 (k = t, n = g), b1 (k = t + 4, n = g)
//   C (16 x 8): c0 (g, 2t), c1 (g, 2t + 1), c2 (g + 8, 2t), c3 (g + 8, 2t + 1)
template <int DK>
__global__ void __launch_bounds__(kScanThreads + 32) kda_scan_kernel(const ChunkArgs a) {
    using L = ScanLayout<DK>;
    constexpr int P = L::P, PK = L::PK, PD = L::PD, PR = L::PR, CPT = L::CPT, WPC = DK / 32, TPW = L::TPW;
    extern __shared__ __align__(128) float sm[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g = lane >> 2, t4 = lane & 3;
    const int cb = blockIdx.x, c0 = cb * kNC, h = blockIdx.y;
    const long long b = blockIdx.z;
    float *ST = sm + L::ST, *DD = sm + L::DD, *RED = sm + L::RED;
    // stage s: barrier full(s) completes when chunk data has landed in it,
    // free(s) when every compute warp is done with it
    const uint32_t bar0 = smem_u32(sm + L::BARS), fbar0 = bar0 + 8 * kStages;

    if (tid == 0) {
        for (int i = 0; i < kStages; i++) {
            mbar_init(bar0 + 8 * i, 1);
            mbar_init(fbar0 + 8 * i, kScanThreads / 32);
        }
        mbar_fence_init();
    }
    __syncthreads();  // the last barrier over all threads: the copy warp leaves below
    if (warp == kScanThreads / 32) {
        // the copy warp: chunk j into stage j % kStages once that stage is free
        if (lane == 0) {
            const uint64_t pol = l2_evict_last_policy();  // a record's shared part is read by every column block
            int issued = 0;
            for (int j = 0; j < a.nch && j < a.hold_from; j++) {
                const int sj = j % kStages;
                if (j >= kStages && !mbar_wait_bounded(fbar0 + 8 * sj, (uint32_t)(j / kStages - 1) & 1u, a.wait_ns)) {
                    atomicCAS(reinterpret_cast<int *>(a.status), 0, (int)ESA_ERR_TIMEOUT);
                    break;
                }
                scan_issue<DK>(sm + L::S0 + sj * L::STAGE, bar0 + 8 * sj, a, b, h, cb, j, pol);
                issued = j + 1;
            }
            // no copy may still be landing when the block ends
            for (int i = issued > kStages ? issued - kStages : 0; i < issued; i++)
                mbar_wait_bounded(bar0 + 8 * (i % kStages), (uint32_t)(i / kStages) & 1u, a.wait_ns);
        }
        return;
    }

    // The state slice S (Dk x 16) in warp-MMA accumulator form: warp w holds
    // tiles (m-tile, n-tile) = (w % MT, w / MT + i) for i < TPW, i.e. rows
    // 16 mt + g (+8), columns 8 nt + 2 t (+1); a copy transposed in ST.
    const int mt2 = warp % L::MT, nt2 = warp / L::MT * TPW;
    const long long sbase = (b * a.H + h) * (long long)DK * a.Dv + c0;
    float acc[TPW][4];
    auto st_row = [&](int i, int e) { return 16 * mt2 + g + ((e & 2) ? 8 : 0); };
    auto st_col = [&](int i, int e) { return 8 * (nt2 + i) + 2 * t4 + (e & 1); };
#pragma unroll
    for (int i = 0; i < TPW; i++)
#pragma unroll
        for (int e = 0; e < 4; e++) {
            const int r = st_row(i, e), c = st_col(i, e);
            acc[i][e] = a.src ? a.src[sbase + (long long)r * a.Dv + c] : 0.f;
            ST[c * P + r] = acc[i][e];
        }

    // X = [Wk; Qp] S by warp (m-tile mt: Wk or Qp rows; K quarter kq; both n-tiles)
    const int mt = warp & 1, kq = warp >> 1;

    int j = 0;
    for (; j < a.nch; j++) {
        const long long t0 = (a.c_begin + j) * kC;
        const int n = (int)min((long long)kC, a.T - t0);
        const int sj = j % kStages;
        const uint32_t bar = bar0 + 8 * sj;
        const bool got = mbar_wait_bounded(bar, (uint32_t)(j / kStages) & 1u, a.wait_ns);
        if (!cbar_and(got)) break;  // chunk j's record and the state slice are in place
        const float *buf = sm + L::S0 + sj * L::STAGE;

        if (reinterpret_cast<const int *>(buf + L::FLAG)[0] == 0) {
            {
                const float *X = buf + (mt ? L::QP : L::WK);
                float xa[2][3][4];
#pragma unroll
                for (int u = 0; u < 2; u++)
#pragma unroll
                    for (int p3 = 0; p3 < 3; p3++)
#pragma unroll
                        for (int e = 0; e < 4; e++) xa[u][p3][e] = 0.f;
#pragma unroll
                for (int ks = 0; ks < DK / 32; ks++) {
                    const int k0 = kq * (DK / 4) + 8 * ks;
                    const float af[4] = {X[g * P + k0 + t4], X[(g + 8) * P + k0 + t4], X[g * P + k0 + t4 + 4],
                                         X[(g + 8) * P + k0 + t4 + 4]};
                    uint32_t ah[4], al[4];
#pragma unroll
                    for (int i = 0; i < 4; i++) tf32_split(af[i], ah[i], al[i]);
#pragma unroll
                    for (int u = 0; u < 2; u++) {
                        const float *Y = ST + (8 * u + g) * P + k0 + t4;
                        uint32_t bh[2], bl[2];
                        tf32_split(Y[0], bh[0], bl[0]);
                        tf32_split(Y[4], bh[1], bl[1]);
                        mma_tf32_1688(xa[u][0], al, bh);
                        mma_tf32_1688(xa[u][1], ah, bl);
                        mma_tf32_1688(xa[u][2], ah, bh);
                    }
                }
#pragma unroll
                for (int u = 0; u < 2; u++) {
                    float x[4];
#pragma unroll
                    for (int e = 0; e < 4; e++) x[e] = (xa[u][0][e] + xa[u][1][e]) + xa[u][2][e];
                    float *R = RED + kq * 2 * kC * PR + (16 * mt + g) * PR + 8 * u + 2 * t4;
                    *reinterpret_cast<float2 *>(R) = make_float2(x[0], x[1]);
                    *reinterpret_cast<float2 *>(R + 8 * PR) = make_float2(x[2], x[3]);
                }
            }
            cbar();
            {
                // thread tid: D at (row, col) = (tid / 16, tid % 16); O at the same place
                const int row = tid >> 4, col = tid & 15;
                constexpr int Q = 2 * kC * PR;  // one K quarter's partial sums
                const float *Rw = RED + row * PR + col, *Rz = Rw + 16 * PR;
                const float w = ((Rw[0] + Rw[Q]) + Rw[2 * Q]) + Rw[3 * Q];
                const float z = ((Rz[0] + Rz[Q]) + Rz[2 * Q]) + Rz[3 * Q];
                DD[row * PD + col] = buf[L::UU + row * kNC + col] - w;
                if (row < n) {
                    const float o = a.scale * (z + buf[L::UP + row * kNC + col]);
                    const long long e = ((b * a.T + t0 + row) * a.H + h) * (long long)a.Dv + c0 + col;
                    if (a.o) a.o[e] = o;
                    if (a.lin) a.lin[e] = (uint16_t)(pack_bf16(o, 0.f) & 0xffffu);
                }
            }
            cbar();
            // S' = g_last * S + Kl^T D: A = Kl^T (rows d, columns i), B = D
            const float *KL = buf + L::KL, *GL = buf + L::GL;
            const float g0 = GL[16 * mt2 + g], g8 = GL[16 * mt2 + g + 8];
            float pa[TPW][3][4];
#pragma unroll
            for (int i = 0; i < TPW; i++)
#pragma unroll
                for (int p3 = 0; p3 < 3; p3++)
#pragma unroll
                    for (int e = 0; e < 4; e++) pa[i][p3][e] = 0.f;
#pragma unroll
            for (int ks = 0; ks < kC / 8; ks++) {
                const float *K0 = KL + (8 * ks + t4) * PK + 16 * mt2 + g, *K4 = K0 + 4 * PK;
                const float af[4] = {K0[0], K0[8], K4[0], K4[8]};
                uint32_t ah[4], al[4];
#pragma unroll
                for (int i = 0; i < 4; i++) tf32_split(af[i], ah[i], al[i]);
#pragma unroll
                for (int i = 0; i < TPW; i++) {
                    const float *D0 = DD + (8 * ks + t4) * PD + 8 * (nt2 + i) + g;
                    uint32_t bh[2], bl[2];
                    tf32_split(D0[0], bh[0], bl[0]);
                    tf32_split(D0[4 * PD], bh[1], bl[1]);
                    mma_tf32_1688(pa[i][0], al, bh);
                    mma_tf32_1688(pa[i][1], ah, bl);
                    mma_tf32_1688(pa[i][2], ah, bh);
                }
            }
#pragma unroll
            for (int i = 0; i < TPW; i++)
#pragma unroll
                for (int e = 0; e < 4; e++)
                    acc[i][e] = fmaf(e < 2 ? g0 : g8, acc[i][e], (pa[i][0][e] + pa[i][1][e]) + pa[i][2][e]);
#pragma unroll
            for (int i = 0; i < TPW; i++)
#pragma unroll
                for (int e = 0; e < 4; e++) ST[st_col(i, e) * P + st_row(i, e)] = acc[i][e];
        } else {
            // a flagged chunk: its steps one by one on the state slice, thread
            // (d, ch) holding row d, columns ch*CPT .. +CPT-1 (from ST).
            // RED[0 ..) holds the per-warp sums of k . S, RED[256 ..) of q . S.
            const int d = tid % DK, ch = tid / DK, wd = d >> 5;
            float s[CPT];
#pragma unroll
            for (int c = 0; c < CPT; c++) s[c] = ST[(ch * CPT + c) * P + d];
            for (int t = 0; t < n; t++) {
                const long long row = (b * a.T + t0 + t) * a.H + h;
                const float al = a.alpha[row * DK + d], kv = bf(a.k[row * DK + d]), qv = bf(a.q[row * DK + d]);
                float p[CPT];
#pragma unroll
                for (int c = 0; c < CPT; c++) {
                    s[c] *= al;
                    p[c] = kv * s[c];
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1)
#pragma unroll
                    for (int c = 0; c < CPT; c++) p[c] += __shfl_xor_sync(0xffffffffu, p[c], off);
                if (lane == 0)
#pragma unroll
                    for (int c = 0; c < CPT; c++) RED[(ch * WPC + wd) * CPT + c] = p[c];
                cbar();
                const float bt = a.beta[row];
#pragma unroll
                for (int c = 0; c < CPT; c++) {
                    float u = RED[ch * WPC * CPT + c];
#pragma unroll
                    for (int w = 1; w < WPC; w++) u += RED[(ch * WPC + w) * CPT + c];
                    const float dl = bt * (bf(a.v[row * a.Dv + c0 + ch * CPT + c]) - u);
                    s[c] = fmaf(kv, dl, s[c]);
                    p[c] = qv * s[c];
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1)
#pragma unroll
                    for (int c = 0; c < CPT; c++) p[c] += __shfl_xor_sync(0xffffffffu, p[c], off);
                if (lane == 0)
#pragma unroll
                    for (int c = 0; c < CPT; c++) RED[256 + (ch * WPC + wd) * CPT + c] = p[c];
                cbar();
                if (d == 0) {
#pragma unroll
                    for (int c = 0; c < CPT; c++) {
                        float z = RED[256 + ch * WPC * CPT + c];
#pragma unroll
                        for (int w = 1; w < WPC; w++) z += RED[256 + (ch * WPC + w) * CPT + c];
                        const float o = a.scale * z;
                        const long long e = row * a.Dv + c0 + ch * CPT + c;
                        if (a.o) a.o[e] = o;
                        if (a.lin) a.lin[e] = (uint16_t)(pack_bf16(o, 0.f) & 0xffffu);
                    }
                }
            }
#pragma unroll
            for (int c = 0; c < CPT; c++) ST[(ch * CPT + c) * P + d] = s[c];
            cbar();
#pragma unroll
            for (int i = 0; i < TPW; i++)
#pragma unroll
                for (int e = 0; e < 4; e++) acc[i][e] = ST[st_col(i, e) * P + st_row(i, e)];
        }
        // this warp is done with stage sj (the next chunk's top barrier
        // orders the state slice, D and the partial sums)
        __syncwarp();
        if (lane == 0) mbar_arrive(fbar0 + 8 * sj);
    }
    if (j < a.nch) {
        // a record never arrived: report it and leave the state as is (the
        // copy warp waits, bounded, for its copies in flight)
        if (tid == 0) atomicCAS(reinterpret_cast<int *>(a.status), 0, (int)ESA_ERR_TIMEOUT);
        return;
    }
    if (a.dst) {
#pragma unroll
        for (int i = 0; i < TPW; i++)
#pragma unroll
            for (int e = 0; e < 4; e++) a.dst[sbase + (long long)st_row(i, e) * a.Dv + st_col(i, e)] = acc[i][e];
    }
}

// A side stream (at the device's greatest priority) and five events per
// host thread and device, for running the scans beside the next segments'
// preps (created once, kept).
struct SideStream {
    cudaStream_t s = nullptr;
    cudaEvent_t fork = nullptr, prep[2] = {}, scan[2] = {};
    bool ok = false, tried = false;
};
SideStream &side_stream() {
    thread_local SideStream r[64];
    int dev = 0;
    cudaGetDevice(&dev);
    SideStream &x = r[dev & 63];
    if (!x.tried) {
        x.tried = true;
        int least = 0, greatest = 0;
        bool ok = cudaDeviceGetStreamPriorityRange(&least, &greatest) == cudaSuccess &&
                  cudaStreamCreateWithPriority(&x.s, cudaStreamNonBlocking, greatest) == cudaSuccess;
        for (cudaEvent_t *e : {&x.fork, &x.prep[0], &x.prep[1], &x.scan[0], &x.scan[1]})
            ok = ok && cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess;
        if (!ok) cudaGetLastError();
        x.ok = ok;
    }
    return x;
}

// Segments of up to kSegChunks chunks. With more than one, segment s's
// records go to buffer s & 1; the preps run on `st` and the scans on the
// side stream, so that prep(s + 1) runs beside scan(s) (the scan block
// leaves room on its SM for two prep blocks, and the side stream's priority
// places scan blocks first as SMs free up). Event edges order scan(s) after
// prep(s), prep(s) after scan(s - 2) (its buffer is free), and `st` after
// the last scan. Nothing waits on a flag: only stream events.
template <int DK>
esa_status launch_chunked_t(ChunkArgs a, long long B, long long nchunks, const float *state_in, float *state_out,
                            float *carry, float *rec1, cudaStream_t st) {
    using L = ScanLayout<DK>;
    const void *fn = reinterpret_cast<const void *>(&kda_scan_kernel<DK>);
    const size_t smem = L::BYTES, psmem = PrepLayout<DK>::bytes(a.Dv);
    if (!ensure_smem(fn, smem) ||
        !ensure_smem(reinterpret_cast<const void *>(&kda_prep_kernel<DK>), PrepLayout<DK>::bytes(512)))
        return ESA_ERR_CUDA;
    float *rec0 = a.rec;
    const long long nseg = (nchunks + kSegChunks - 1) / kSegChunks;
    SideStream *side = nseg > 1 ? &side_stream() : nullptr;
    const bool overlap = side && side->ok && rec1;
    if (overlap && (cudaEventRecord(side->fork, st) != cudaSuccess || cudaStreamWaitEvent(side->s, side->fork) != cudaSuccess))
        return ESA_ERR_CUDA;
    for (long long sg = 0; sg < nseg; sg++) {
        const long long c = sg * kSegChunks;
        const bool last = sg == nseg - 1;
        ChunkArgs x = a;
        x.c_begin = c;
        x.nch = (int)(last ? nchunks - c : kSegChunks);
        x.src = sg == 0 ? state_in : carry;
        x.dst = last ? state_out : carry;
        x.rec = overlap && (sg & 1) ? rec1 : rec0;
        const dim3 pgrid((unsigned)x.nch, (unsigned)x.H, (unsigned)B), sgrid((unsigned)(x.Dv / kNC), (unsigned)x.H,
                                                                           (unsigned)B);
        if (!overlap) {
            kda_prep_kernel<DK><<<pgrid, kPrepThreads, psmem, st>>>(x);
            kda_scan_kernel<DK><<<sgrid, kScanThreads + 32, smem, st>>>(x);
            continue;
        }
        const int ib = (int)(sg & 1);
        if (sg >= 2 && cudaStreamWaitEvent(st, side->scan[ib]) != cudaSuccess) return ESA_ERR_CUDA;
        kda_prep_kernel<DK><<<pgrid, kPrepThreads, psmem, st>>>(x);
        if (cudaEventRecord(side->prep[ib], st) != cudaSuccess ||
            cudaStreamWaitEvent(side->s, side->prep[ib]) != cudaSuccess)
            return ESA_ERR_CUDA;
        kda_scan_kernel<DK><<<sgrid, kScanThreads + 32, smem, side->s>>>(x);
        if (cudaEventRecord(side->scan[ib], side->s) != cudaSuccess) return ESA_ERR_CUDA;
        if (last && cudaStreamWaitEvent(st, side->scan[ib]) != cudaSuccess) return ESA_ERR_CUDA;
    }
    return cudaGetLastError() == cudaSuccess ? ESA_OK : ESA_ERR_CUDA;
}

}  // namespace

// Workspace: the status word (kStatusBytes); with more than one segment the
// carried state and two record buffers, else one.
size_t kda_chunked_ws_bytes(long long B, long long T, int H, int Dk, int Dv) {
    if (T <= 0) return 0;
    const long long nchunks = (T + kC - 1) / kC;
    const bool multi = nchunks > kSegChunks;
    const long long cap = multi ? kSegChunks : nchunks;
    const size_t carry = multi ? align256((size_t)B * H * Dk * Dv * 4) : 0;
    const size_t recs = align256((size_t)B * H * cap * rec_floats(Dk, Dv) * 4);
    return kStatusBytes + carry + (multi ? 2 : 1) * recs;
}

esa_status launch_kda_chunked(const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *alpha,
                              const float *beta, const float *state_in, long long B, long long T, int H, int Dk,
                              int Dv, float scale, float *o, uint16_t *lin, float *state_out, void *ws,
                              cudaStream_t st) {
    const long long nchunks = (T + kC - 1) / kC;
    const bool multi = nchunks > kSegChunks;
    const long long cap = multi ? kSegChunks : nchunks;
    char *p = static_cast<char *>(ws) + kStatusBytes;
    float *carry = nullptr, *rec1 = nullptr;
    if (multi) {
        carry = reinterpret_cast<float *>(p);
        p += align256((size_t)B * H * Dk * Dv * 4);
        rec1 = reinterpret_cast<float *>(p + align256((size_t)B * H * cap * rec_floats(Dk, Dv) * 4));
    }
    ChunkArgs a{q, k, v, alpha, beta, nullptr, nullptr, o, lin, reinterpret_cast<float *>(p),
                static_cast<int32_t *>(ws), wait_limit_ns(), debug_extra_arrivals() > 0 ? 1 : INT_MAX, T, 0, 0,
                (int)cap, H, Dv, scale};
    if (Dk == 128) return launch_chunked_t<128>(a, B, nchunks, state_in, state_out, carry, rec1, st);
    if (Dk == 64) return launch_chunked_t<64>(a, B, nchunks, state_in, state_out, carry, rec1, st);
    return ESA_ERR_UNSUPPORTED;
}

}  // namespace esa
