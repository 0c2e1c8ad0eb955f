// Attention router: full or sparse attention per (sequence, query head).
//
// Method ("Elastic Attention：动态路由优化大模型长文本处理", section 2.2): a
// lightweight router, a 2-layer MLP that takes the current key hidden states,
// decides per attention head between full and sparse attention; its decisions
// are the metadata that the fused routed launch branches on (section 3.1).
// The pages give no trained weights: the weights are inputs.
//
// Computed: x = mean over the Tk cached positions of k[b, j, :, :] (Hkv*D
// values), hid = max(0, b1 + W1 x), z_o = b2[2h+o] + W2[2h+o] . hid
// (o = 0 full, o = 1 sparse), route[b, h] = 1 iff z_1 >= z_0.
//
// Four launches, every sum in fp32 in a fixed order (deterministic):
//   route_pool_kernel  streams k once (16-byte loads, a warp reads 512
//                      contiguous bytes per position); block (column block,
//                      position chunk, sequence) writes its chunk's partial
//                      column sums to the workspace;
//   route_mean_kernel, route_hidden_kernel, route_out_kernel
//                      the chunks summed in order per column (divided by
//                      Tk), then the two layers with one warp per output
//                      and a fixed shuffle tree.
#include <algorithm>

#include "esa_device.cuh"
#include "esa_internal.h"

namespace esa {

namespace {

constexpr int kPoolThreads = 256;
constexpr int kColsPerThread = 8;  // one 16-byte load of bf16
constexpr int kColsPerBlock = kPoolThreads * kColsPerThread;

__global__ void __launch_bounds__(kPoolThreads) route_pool_kernel(const uint16_t *__restrict__ k,
                                                                  float *__restrict__ partial, long long Tk, int C,
                                                                  int chunks, long long chunk_len) {
    const int col = (blockIdx.x * kPoolThreads + threadIdx.x) * kColsPerThread;
    const int ch = blockIdx.y;
    const long long b = blockIdx.z;
    if (col >= C) return;
    const long long j0 = ch * chunk_len, j1 = min(Tk, j0 + chunk_len);
    float acc[kColsPerThread] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    const uint16_t *base = k + (b * Tk) * (long long)C + col;
    auto add = [&](const uint4 &w) {
        const uint32_t v[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; e++) {
            acc[2 * e] += bf16lo(v[e]);
            acc[2 * e + 1] += bf16hi(v[e]);
        }
    };
    long long j = j0;
    for (; j + 4 <= j1; j += 4) {  // four loads in flight, then the adds in position order
        const uint4 w0 = ldg_stream16(base + j * C), w1 = ldg_stream16(base + (j + 1) * C),
                    w2 = ldg_stream16(base + (j + 2) * C), w3 = ldg_stream16(base + (j + 3) * C);
        add(w0);
        add(w1);
        add(w2);
        add(w3);
    }
    for (; j < j1; j++) add(ldg_stream16(base + j * C));
    float *dst = partial + ((b * chunks + ch) * (long long)C + col);
    *reinterpret_cast<float4 *>(dst) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    *reinterpret_cast<float4 *>(dst + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
}

__device__ __forceinline__ float warp_sum_fixed(float v) {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
    return v;
}

// x[b, c] = (sum of the position chunks' partial sums, in chunk order) / Tk
__global__ void __launch_bounds__(256) route_mean_kernel(const float *__restrict__ partial, float *__restrict__ x,
                                                         long long Tk, int C, int chunks) {
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    const long long b = blockIdx.y;
    if (c >= C) return;
    float s = 0.f;
    for (int ch = 0; ch < chunks; ch++) s += partial[(b * chunks + ch) * (long long)C + c];
    x[b * C + c] = Tk > 0 ? s * (1.f / (float)Tk) : 0.f;
}

// hid[b, f] = max(0, b1[f] + W1[f] . x[b]): one warp per hidden unit, lanes
// striding over the inputs, a fixed shuffle tree
__global__ void __launch_bounds__(256) route_hidden_kernel(const float *__restrict__ x, const float *__restrict__ W1,
                                                           const float *__restrict__ b1, float *__restrict__ hid, int C,
                                                           int F) {
    const int lane = threadIdx.x & 31, f = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    const long long b = blockIdx.y;
    if (f >= F) return;
    const float *w = W1 + (long long)f * C, *xb = x + b * C;
    float s = 0.f;
    for (int c = lane; c < C; c += 32) s = fmaf(w[c], xb[c], s);
    s = warp_sum_fixed(s) + b1[f];
    if (lane == 0) hid[b * F + f] = fmaxf(s, 0.f);
}

// z_o = b2[2h+o] + W2[2h+o] . hid[b]; route = z_1 >= z_0 (one warp per head)
__global__ void __launch_bounds__(256) route_out_kernel(const float *__restrict__ hid, const float *__restrict__ W2,
                                                        const float *__restrict__ b2, int F, int Hq,
                                                        uint8_t *__restrict__ route, float *__restrict__ margin) {
    const int lane = threadIdx.x & 31, h = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    const long long b = blockIdx.y;
    if (h >= Hq) return;
    const float *hb = hid + b * F;
    float z[2];
#pragma unroll
    for (int o = 0; o < 2; o++) {
        const float *w = W2 + (long long)(2 * h + o) * F;
        float s = 0.f;
        for (int f = lane; f < F; f += 32) s = fmaf(w[f], hb[f], s);
        z[o] = warp_sum_fixed(s) + b2[2 * h + o];
    }
    if (lane == 0) {
        route[b * Hq + h] = z[1] >= z[0] ? 1 : 0;
        if (margin) margin[b * Hq + h] = z[1] - z[0];
    }
}

struct RoutePlan {
    int chunks;
    long long chunk_len;
    size_t x_off;  // workspace: [status][partial sums][x: B x C][hid: B x 4096]
    size_t ws_bytes;
};

RoutePlan plan_route(const Shape &s) {
    RoutePlan p{};
    const int C = s.Hkv * s.D;
    const long long colblocks = (C + kColsPerBlock - 1) / kColsPerBlock;
    // enough blocks for every SM a few times over, chunks of >= 64 positions
    const long long want = 4ll * device_info().sms;
    long long chunks = (want + s.B * colblocks - 1) / (s.B * colblocks);
    chunks = std::max(1ll, std::min(chunks, (s.Tk + 63) / 64));
    p.chunks = (int)chunks;
    p.chunk_len = (s.Tk + chunks - 1) / chunks;
    p.x_off = kStatusBytes + align256((size_t)s.B * chunks * C * sizeof(float));
    p.ws_bytes = p.x_off + align256((size_t)s.B * C * sizeof(float)) + align256((size_t)s.B * 4096 * sizeof(float));
    return p;
}

}  // namespace

size_t ws_route_heads(const Shape &s) { return plan_route(s).ws_bytes; }

esa_status launch_route_heads(const uint16_t *k, const float *W1, const float *b1, const float *W2, const float *b2,
                              const Shape &s, int hidden, uint8_t *route, float *margin, void *ws, cudaStream_t st) {
    const int C = s.Hkv * s.D;
    const RoutePlan p = plan_route(s);
    float *partial = reinterpret_cast<float *>(static_cast<char *>(ws) + kStatusBytes);
    dim3 g1((unsigned)((C + kColsPerBlock - 1) / kColsPerBlock), (unsigned)p.chunks, (unsigned)s.B);
    route_pool_kernel<<<g1, kPoolThreads, 0, st>>>(k, partial, s.Tk, C, p.chunks, p.chunk_len);
    if (cudaGetLastError() != cudaSuccess) return ESA_ERR_CUDA;
    float *x = reinterpret_cast<float *>(static_cast<char *>(ws) + p.x_off);
    float *hid = x + align256((size_t)s.B * C * sizeof(float)) / sizeof(float);
    route_mean_kernel<<<dim3((unsigned)((C + 255) / 256), (unsigned)s.B), 256, 0, st>>>(partial, x, s.Tk, C, p.chunks);
    route_hidden_kernel<<<dim3((unsigned)((hidden + 7) / 8), (unsigned)s.B), 256, 0, st>>>(x, W1, b1, hid, C, hidden);
    route_out_kernel<<<dim3((unsigned)((s.Hq + 7) / 8), (unsigned)s.B), 256, 0, st>>>(hid, W2, b2, hidden, s.Hq, route,
                                                                                    margin);
    return cudaGetLastError() == cudaSuccess ? ESA_OK : ESA_ERR_CUDA;
}

}  // namespace esa
