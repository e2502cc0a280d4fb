// lmhead_noalloc.cu -- w8_lmhead_argmax for callers that cannot allocate.
//
// Some callers cannot hand the library a workspace: a plugin inside another
// inference engine whose execute step may not allocate device memory, or a
// serving loop whose device memory is already fully partitioned by its own
// allocator (and cudaMalloc would also synchronize the device in the middle
// of a latency-critical decode step).  For them this entry point keeps the
// lm_head's only scratch -- the per-row best keys and the arrival counter of
// the cross-CTA argmax -- in a file-scope device array that every GPU which
// loads the library holds until the process exits.  The kernel is the same
// one w8_lmhead_argmax launches; only where its scratch lives differs.
#include <mutex>

#include "runtime.h"

namespace w4v {
namespace {

constexpr size_t kNoAllocScratchBytes = 4096;   // keys for 128 rows + counter need 1280
static __device__ __align__(256) unsigned char g_lmhead_scratch[kNoAllocScratchBytes];

constexpr int kMaxDev = 64;
std::mutex g_scratch_mutex;
void *g_scratch_ptr[kMaxDev] = {};

// Device address of the scratch array for the current device.  In host code
// the array's name is only a host-side stand-in, so the address must come
// from cudaGetSymbolAddress, once per device, with that device current.
w4v_status scratch_for_current_device(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) {
        cudaGetLastError();
        return W4V_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_lmhead_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return W4V_ERR_CUDA;
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return W4V_OK;
}

}  // namespace
}  // namespace w4v

extern "C" w4v_status w8_lmhead_argmax_noalloc(const uint16_t *X, const int8_t *W, const uint16_t *scale, int M,
                                              int K, int V, int32_t *argmax_out, float *maxlogit,
                                              float *logits_debug, w4v_stream_t stream) {
    if (M < 0 || M > 128 || K <= 0 || V <= 0 || K % 128 != 0 || V % 8 != 0) return W4V_ERR_SHAPE;
    if (M == 0) return W4V_OK;
    if (X == nullptr || W == nullptr || scale == nullptr || argmax_out == nullptr) return W4V_ERR_ARG;
    if (!w4v::aligned16(X) || !w4v::aligned16(W) || !w4v::aligned16(scale)) return W4V_ERR_ALIGN;
    if ((reinterpret_cast<uintptr_t>(argmax_out) & 3u) || (reinterpret_cast<uintptr_t>(maxlogit) & 3u) ||
        (reinterpret_cast<uintptr_t>(logits_debug) & 3u))
        return W4V_ERR_ALIGN;
    const size_t need = w4v::w8_lmhead_ws_bytes(M, V);
    if (need > w4v::kNoAllocScratchBytes) return W4V_ERR_SHAPE;
    const w4v::DeviceInfo *info = nullptr;
    w4v_status st = w4v::device_info(&info);
    if (st != W4V_OK) return st;
    void *scratch = nullptr;
    st = w4v::scratch_for_current_device(&scratch);
    if (st != W4V_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // The array keeps whatever the previous call left; the kernel needs its
    // keys and counter at zero.
    if (cudaMemsetAsync(scratch, 0, need, s) != cudaSuccess) {
        cudaGetLastError();
        return W4V_ERR_CUDA;
    }
    return w4v::launch_w8_lmhead_argmax(X, W, scale, M, K, V, argmax_out, maxlogit, logits_debug, scratch, s);
}
