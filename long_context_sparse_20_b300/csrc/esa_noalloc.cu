// Top-K selection for callers that cannot allocate device memory.
//
// Some callers of this library run inside a runtime that owns every device
// allocation (a framework's caching allocator, or a serving engine that
// reserves its whole memory pool up front) and are not allowed to call
// cudaMalloc themselves, so they cannot hand esa_topk_select() a workspace.
// esa_topk_select_noalloc() runs the same selection kernels with their
// scratch state in one fixed device array that belongs to this library.
#include <cuda_runtime.h>

#include <mutex>

#include "esa_internal.h"

namespace {

// The scratch array. Every GPU that loads the library holds it until exit.
// Host code must never pass `g_noalloc_scratch` itself to a kernel: on the
// host the name is only a stand-in for the device symbol. The device address
// comes from cudaGetSymbolAddress (noalloc_scratch_ptr below).
static __device__ __align__(256) unsigned char g_noalloc_scratch[ESA_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch, looked up once per device with that
// device current (the first call of the entry point on each device).
void *noalloc_scratch_ptr(esa_status *err) {
    static std::mutex mu;
    static void *ptr[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        *err = ESA_ERR_CUDA;
        return nullptr;
    }
    std::lock_guard<std::mutex> lk(mu);
    if (!ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            *err = ESA_ERR_CUDA;
            return nullptr;
        }
        ptr[dev] = p;
    }
    return ptr[dev];
}

}  // namespace

using namespace esa;

extern "C" ESA_API esa_status esa_topk_select_noalloc(const int8_t *qI, const int8_t *kI, const int32_t *wI,
                                                      const esa_shape *s, int top_k, int32_t *idx, int32_t *cnt,
                                                      int32_t *dev_status, void *stream) {
    if (!s || !qI || !kI || !wI || !idx || !cnt) return ESA_ERR_INVALID;
    if (s->B < 0 || s->Tq < 0 || s->Tk < 0 || s->q_offset < 0 || s->q_offset + s->Tq > s->Tk) return ESA_ERR_INVALID;
    if (s->Tk > (int64_t)INT32_MAX) return ESA_ERR_UNSUPPORTED;
    if (s->H_I <= 0 || s->H_I > 16) return ESA_ERR_UNSUPPORTED;
    if (s->D_I != 16 && s->D_I != 32 && s->D_I != 64 && s->D_I != 128) return ESA_ERR_UNSUPPORTED;
    if (top_k <= 0 || top_k > 65536) return ESA_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(qI) & 15u) || (reinterpret_cast<uintptr_t>(kI) & 15u)) return ESA_ERR_INVALID;
    if (s->flags & ~(ESA_INDEXER_RELU | ESA_PER_HEAD_SETS)) return ESA_ERR_INVALID;
    Shape x0{s->B, s->Tq, s->Tk, s->q_offset, s->Hq, s->Hkv, s->D, s->H_I, s->D_I};
    x0.flags = s->flags;
    const Shape x = selection_rows(x0);  // per-head sets: one row per (query, indexer head)
    if (per_head_of(x) && !(wI = unit_weight())) return ESA_ERR_CUDA;
    if (x.B * x.Tq == 0) return ESA_OK;

    SplitPlan sp = plan_split_select(x, top_k);
    // the row-tiled path needs only the status word; it takes the tensor-core
    // kernel when that kernel's scratch fits too
    const size_t need = sp.ok ? sp.ws_bytes : kStatusBytes;
    if (need > (size_t)ESA_NOALLOC_SCRATCH_BYTES) return ESA_ERR_UNSUPPORTED;  // beyond the fixed scratch size

    esa_status err = ESA_OK;
    void *scratch = noalloc_scratch_ptr(&err);
    if (!scratch) return err;
    cudaStream_t st = (cudaStream_t)stream;
    // The array keeps the previous call's contents: clear the status word and
    // the control state (call counter, barrier counters, histograms) that must
    // start at zero.
    const size_t clear = sp.ok ? sp.pub_off : kStatusBytes;
    if (cudaMemsetAsync(scratch, 0, clear, st) != cudaSuccess) return ESA_ERR_CUDA;
    if (sp.ok && cudaMemsetAsync(static_cast<char *>(scratch) + sp.ctrl_off, 0, sp.ctrl_bytes, st) != cudaSuccess)
        return ESA_ERR_CUDA;
    esa_status e = sp.ok ? launch_split_select(qI, kI, wI, x, top_k, idx, cnt, scratch,
                                               (size_t)ESA_NOALLOC_SCRATCH_BYTES, sp, st)
                         : launch_row_select(qI, kI, wI, x, top_k, idx, cnt, nullptr, scratch,
                                             (size_t)ESA_NOALLOC_SCRATCH_BYTES, st);
    if (e != ESA_OK) return e;
    if (dev_status && cudaMemcpyAsync(dev_status, scratch, sizeof(int32_t), cudaMemcpyDeviceToDevice, st) != cudaSuccess)
        return ESA_ERR_CUDA;
    return ESA_OK;
}
