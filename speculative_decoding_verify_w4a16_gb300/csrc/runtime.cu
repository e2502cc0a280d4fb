// runtime.cu -- per-device set-up: architecture check with a smoke launch,
// SM count, the device status word, and TMA tensor-map encoding through the
// driver entry point (no link-time dependency on libcuda).
#include <mutex>

#include "runtime.h"

namespace w4v {

// Bit (1 << code) is set by a kernel that abandons a bounded wait.
__device__ uint32_t g_status_word;

namespace {

constexpr int kMaxDevices = 64;

struct Slot {
    bool ready = false;
    DeviceInfo info;
};

Slot g_slots[kMaxDevices];
std::mutex g_mutex;

__global__ void smoke_kernel(uint32_t *out) { *out = 0x5eedu; }

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

}  // namespace

w4v_status device_info(const DeviceInfo **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return W4V_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_mutex);
    Slot &s = g_slots[dev];
    if (!s.ready) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return W4V_ERR_CUDA;
        }
        if (major != 10 || minor != 3) return W4V_ERR_ARCH;
        uint32_t *status = nullptr;
        if (cudaGetSymbolAddress(reinterpret_cast<void **>(&status), g_status_word) != cudaSuccess) {
            cudaError_t e = cudaGetLastError();
            return e == cudaErrorNoKernelImageForDevice || e == cudaErrorInvalidDeviceFunction
                       ? W4V_ERR_ARCH : W4V_ERR_CUDA;
        }
        // Smoke launch: a library built for another architecture fails here.
        cudaStream_t st = nullptr;
        if (cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) != cudaSuccess) {
            cudaGetLastError();
            return W4V_ERR_CUDA;
        }
        smoke_kernel<<<1, 1, 0, st>>>(status);
        cudaError_t e = cudaGetLastError();
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
        uint32_t v = 0;
        if (e == cudaSuccess) e = cudaMemcpyAsync(&v, status, 4, cudaMemcpyDeviceToHost, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
        const uint32_t zero = 0;
        if (e == cudaSuccess) e = cudaMemcpyAsync(status, &zero, 4, cudaMemcpyHostToDevice, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
        cudaStreamDestroy(st);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return (e == cudaErrorNoKernelImageForDevice || e == cudaErrorInvalidDeviceFunction)
                       ? W4V_ERR_ARCH : W4V_ERR_CUDA;
        }
        if (v != 0x5eedu) return W4V_ERR_ARCH;
        if (g_encode == nullptr) {
            void *fn = nullptr;
            cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                 cudaEnableDefault, &q) != cudaSuccess ||
                q != cudaDriverEntryPointSuccess || fn == nullptr) {
                cudaGetLastError();
                return W4V_ERR_CUDA;
            }
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
        }
        s.info.sm_count = sms;
        s.info.status = status;
        s.ready = true;
    }
    *out = &s.info;
    return W4V_OK;
}

w4v_status encode_tmap_2d(CUtensorMap *map, CUtensorMapDataType dtype, const void *base,
                          uint64_t inner, uint64_t outer, uint64_t row_bytes,
                          uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle) {
    if (g_encode == nullptr) return W4V_ERR_CUDA;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, dtype, 2, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? W4V_OK : W4V_ERR_ARG;
}

w4v_status encode_tmap_kblocks(CUtensorMap *map, CUtensorMapDataType dtype, uint32_t elem_bytes, const void *base,
                               uint64_t inner, uint64_t rows, uint32_t inner_box, uint32_t box_rows,
                               uint32_t box_blocks, CUtensorMapSwizzle swizzle) {
    if (g_encode == nullptr || inner % inner_box != 0) return W4V_ERR_CUDA;
    cuuint64_t dims[3] = {inner_box, rows, inner / inner_box};
    cuuint64_t strides[2] = {inner * elem_bytes, uint64_t(inner_box) * elem_bytes};
    cuuint32_t box[3] = {inner_box, box_rows, box_blocks};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(map, dtype, 3, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? W4V_OK : W4V_ERR_ARG;
}

}  // namespace w4v

extern "C" w4v_status w4v_init(void) {
    const w4v::DeviceInfo *info = nullptr;
    return w4v::device_info(&info);
}

extern "C" w4v_status w4v_get_status(w4v_stream_t stream) {
    const w4v::DeviceInfo *info = nullptr;
    w4v_status st = w4v::device_info(&info);
    if (st != W4V_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint32_t v = 0;
    const uint32_t zero = 0;
    if (cudaMemcpyAsync(&v, info->status, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemcpyAsync(info->status, &zero, 4, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return W4V_ERR_CUDA;
    }
    if (v & (1u << W4V_ERR_TIMEOUT)) return W4V_ERR_TIMEOUT;
    return v ? W4V_ERR_CUDA : W4V_OK;
}
