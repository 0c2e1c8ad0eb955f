// Gate mix and the diagnostic indexer-score kernel.
//
// Gate mix: final = g*attn + (1-g)*linear_output ("超大规模MoE架构中稀疏注意力机制的
// 演进与实践", sections 二.3 and 四.1). HBM-bound elementwise work: 16-byte
// loads of attn (fp32) and 8-byte loads of lin (bf16) per 4 outputs.
//
// Indexer score: relevance of a query to every history position without
// RoPE (same page, sections 二.1-二.2), int8 dot products with exact int32
// accumulation (dp4a), weighted over indexer heads.
#include "esa_device.cuh"
#include "esa_internal.h"

namespace esa {

__global__ void __launch_bounds__(256) gated_mix_kernel(const float4 *__restrict__ attn, const uint2 *__restrict__ lin,
                                                        const float *__restrict__ g,
                                                        const uint8_t *__restrict__ head_mask, float4 *__restrict__ out,
                                                        long long n4, int Hq, int D4, long long Tq) {
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n4; i += (long long)gridDim.x * blockDim.x) {
        long long row_h = i / D4;  // (b, t, h) flat
        int h = (int)(row_h % Hq);
        long long b = row_h / Hq / Tq;
        float4 a = attn[i];
        bool mix = head_mask ? head_mask[b * Hq + h] != 0 : true;
        if (mix) {
            float gh = g[h], gl = 1.0f - gh;
            uint2 l = lin[i];
            a.x = fmaf(gh, a.x, gl * bf16lo(l.x));
            a.y = fmaf(gh, a.y, gl * bf16hi(l.x));
            a.z = fmaf(gh, a.z, gl * bf16lo(l.y));
            a.w = fmaf(gh, a.w, gl * bf16hi(l.y));
        }
        out[i] = a;
    }
}

// The step's new K, V and indexer-key rows into the caches: one block per
// (sequence, new position), 16-byte copies.
__global__ void __launch_bounds__(128) cache_append_kernel(const uint4 *__restrict__ kn, const uint4 *__restrict__ vn,
                                                           const uint4 *__restrict__ kin, uint4 *k, uint4 *v,
                                                           uint4 *ki, long long Tq, long long Tk, long long q_offset,
                                                           int kv16, int ki16) {
    const long long r = blockIdx.x, b = r / Tq, t = r % Tq;
    const long long dst = b * Tk + q_offset + t;
    for (int i = threadIdx.x; i < kv16; i += blockDim.x) {
        if (kn) k[dst * kv16 + i] = kn[r * kv16 + i];
        if (vn) v[dst * kv16 + i] = vn[r * kv16 + i];
    }
    if (kin)
        for (int i = threadIdx.x; i < ki16; i += blockDim.x) ki[dst * ki16 + i] = kin[r * ki16 + i];
}

cudaError_t launch_cache_append(const uint16_t *k_new, const uint16_t *v_new, const int8_t *kI_new, uint16_t *k,
                                uint16_t *v, int8_t *kI, const Shape &s, cudaStream_t st) {
    const long long rows = s.B * s.Tq;
    if (rows == 0) return cudaSuccess;
    const int kv16 = (k || v) ? s.Hkv * s.D * 2 / 16 : 0, ki16 = kI ? s.D_I / 16 : 0;
    cache_append_kernel<<<(unsigned)rows, 128, 0, st>>>(
        reinterpret_cast<const uint4 *>(k_new), reinterpret_cast<const uint4 *>(v_new),
        reinterpret_cast<const uint4 *>(kI_new), reinterpret_cast<uint4 *>(k), reinterpret_cast<uint4 *>(v),
        reinterpret_cast<uint4 *>(kI), s.Tq, s.Tk, s.q_offset, kv16, ki16);
    return cudaGetLastError();
}

int mix_binary_version() {
    cudaFuncAttributes fa{};
    if (cudaFuncGetAttributes(&fa, gated_mix_kernel) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    return fa.binaryVersion;
}

cudaError_t launch_gated_mix(const float *attn, const uint16_t *lin, const float *g, const uint8_t *head_mask,
                             const Shape &s, float *out, cudaStream_t st) {
    long long n4 = s.B * s.Tq * s.Hq * (long long)s.D / 4;
    if (n4 == 0) return cudaSuccess;
    DevInfo di = device_info();
    long long blocks = (n4 + 255) / 256;
    long long cap = (long long)di.sms * 8;
    int grid = (int)(blocks < cap ? blocks : cap);
    gated_mix_kernel<<<grid, 256, 0, st>>>(reinterpret_cast<const float4 *>(attn), reinterpret_cast<const uint2 *>(lin),
                                           g, head_mask, reinterpret_cast<float4 *>(out), n4, s.Hq, s.D / 4, s.Tq);
    return cudaGetLastError();
}

// One block per (query row, 1024-key span). The row's indexer query sits in
// shared memory; each thread scores keys with 16-byte loads of kI.
template <int DI>
__global__ void __launch_bounds__(256) indexer_score_kernel(const int8_t *__restrict__ qI, const int8_t *__restrict__ kI,
                                                            const int32_t *__restrict__ wI, int32_t *__restrict__ scores,
                                                            long long Tq, long long Tk, long long q_offset, int H_I,
                                                            int pos_div, int relu) {
    constexpr int W = DI / 4;  // 32-bit words per vector
    __shared__ int32_t qs[16 * W];
    __shared__ int32_t ws_[16];
    long long row = blockIdx.x;  // b*Tq + t (pos_div rows per query position)
    long long b = row / Tq, t = (row % Tq) / pos_div;
    long long p = q_offset + t;
    const int32_t *qrow = reinterpret_cast<const int32_t *>(qI + row * (long long)H_I * DI);
    for (int i = threadIdx.x; i < H_I * W; i += blockDim.x) qs[i] = qrow[i];
    if (threadIdx.x < H_I) ws_[threadIdx.x] = wI[threadIdx.x];
    __syncthreads();
    long long j = blockIdx.y * 1024ll + threadIdx.x;
    for (int it = 0; it < 4; it++, j += 256) {
        if (j >= Tk) break;
        int32_t outv = INT32_MIN;
        if (j <= p) {
            const int4 *kp = reinterpret_cast<const int4 *>(kI + (b * Tk + j) * DI);
            int kw[W];
#pragma unroll
            for (int c = 0; c < W / 4; c++) {
                int4 v = kp[c];
                kw[4 * c] = v.x;
                kw[4 * c + 1] = v.y;
                kw[4 * c + 2] = v.z;
                kw[4 * c + 3] = v.w;
            }
            unsigned acc = 0;
            for (int h = 0; h < H_I; h++) {
                int d = 0;
#pragma unroll
                for (int c = 0; c < W; c++) d = __dp4a(qs[h * W + c], kw[c], d);
                acc += (unsigned)ws_[h] * (unsigned)(relu ? max(d, 0) : d);
            }
            outv = (int32_t)acc;
        }
        scores[row * Tk + j] = outv;
    }
}

cudaError_t launch_indexer_score(const int8_t *qI, const int8_t *kI, const int32_t *wI, const Shape &s,
                                 int32_t *scores, cudaStream_t st) {
    long long rows = s.B * s.Tq;
    if (rows == 0 || s.Tk == 0) return cudaSuccess;
    if ((s.Tk + 1023) / 1024 > 65535 || rows > 0x7fffffffll) return cudaErrorInvalidValue;
    dim3 grid((unsigned)rows, (unsigned)((s.Tk + 1023) / 1024));
    const int pd = s.pos_div, relu = relu_of(s) ? 1 : 0;
    switch (s.D_I) {
        case 16: indexer_score_kernel<16><<<grid, 256, 0, st>>>(qI, kI, wI, scores, s.Tq, s.Tk, s.q_offset, s.H_I, pd, relu); break;
        case 32: indexer_score_kernel<32><<<grid, 256, 0, st>>>(qI, kI, wI, scores, s.Tq, s.Tk, s.q_offset, s.H_I, pd, relu); break;
        case 64: indexer_score_kernel<64><<<grid, 256, 0, st>>>(qI, kI, wI, scores, s.Tq, s.Tk, s.q_offset, s.H_I, pd, relu); break;
        default: indexer_score_kernel<128><<<grid, 256, 0, st>>>(qI, kI, wI, scores, s.Tq, s.Tk, s.q_offset, s.H_I, pd, relu); break;
    }
    return cudaGetLastError();
}

}  // namespace esa
