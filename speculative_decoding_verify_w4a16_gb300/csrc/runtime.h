// runtime.h -- internal host-side helpers shared by the launchers (not part
// of the public ABI).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/w4v.h"

namespace w4v {

// Upper bound on the CTAs of one persistent launch; it sizes workspaces
// without querying a device.
constexpr int kMaxCtas = 256;

struct DeviceInfo {
    int sm_count = 0;
    uint32_t *status = nullptr;   // device status word (bit per w4v_status code)
};

// Arch check, smoke launch and per-device facts for the current device
// (cached after the first successful call on that device).
w4v_status device_info(const DeviceInfo **out);

// Row-major 2-D tensor map: `outer` rows of `inner` elements, rows
// `row_bytes` apart, boxes of box_inner x box_outer elements, zero fill out
// of bounds.
w4v_status encode_tmap_2d(CUtensorMap *map, CUtensorMapDataType dtype, const void *base,
                          uint64_t inner, uint64_t outer, uint64_t row_bytes,
                          uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle);

// 3-D map over a row-major [outer][inner] matrix viewed as
// (inner_box elements, rows, inner / inner_box blocks): the block dimension
// steps inner_box elements along a row, so one box of {inner_box, box_rows,
// box_blocks} lands in shared memory as box_blocks consecutive
// [box_rows][inner_box] tiles -- the K-major layout the MMA descriptors use.
w4v_status encode_tmap_kblocks(CUtensorMap *map, CUtensorMapDataType dtype, uint32_t elem_bytes, const void *base,
                               uint64_t inner, uint64_t rows, uint32_t inner_box, uint32_t box_rows,
                               uint32_t box_blocks, CUtensorMapSwizzle swizzle);

// Launches `kernel` with programmatic stream serialization, so its grid can
// be scheduled while the previous kernel of the stream drains; the kernel
// itself orders its memory accesses after that kernel (grid_dep_wait).
// Same, optionally as thread-block clusters of `cluster` CTAs along x
// (0: no cluster launch).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                               int cluster, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    int n = 1;
    if (cluster > 0) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = cluster;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        n = 2;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args &&...args) {
    return launch_pdl_cluster(kernel, grid, block, smem, stream, 0, static_cast<Args &&>(args)...);
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Stream-K style even split of `units` over `ctas`: CTA c owns
// [c*units/ctas, (c+1)*units/ctas).
__host__ __device__ inline long long split_begin(long long c, long long units, long long ctas) {
    return c * units / ctas;
}
// The CTA whose range holds unit u.
__host__ __device__ inline int split_owner(long long u, long long units, long long ctas) {
    return static_cast<int>(((u + 1) * ctas - 1) / units);
}

// Launchers (one per kernel family), called after argument validation.
// group: 128 or 32 (scales and zero points [K/group][N]).
w4v_status launch_w4a16_decode(const uint16_t *A, const void *Bq, const uint16_t *scales,
                               const uint8_t *zeros, int group, uint16_t *C, int M, int N, int K,
                               void *ws, bool static_weights, cudaStream_t stream);
size_t w4a16_decode_ws_bytes(int M, int N, int K);
// Grouped launch of the verify-sized kernel (arguments validated by the caller).
size_t w4a16_grouped_table_bytes(int n_problems);
w4v_status build_w4a16_grouped(const w4a16_problem *probs, int n, int M, int group, void *plan,
                               w4a16_grouped_t *handle, cudaStream_t stream);
bool w4a16_grouped_handle_ok(const w4a16_grouped_t &handle);
size_t w4a16_grouped_ws_bytes(const w4a16_grouped_t &handle);
w4v_status launch_w4a16_grouped(const w4a16_grouped_t &handle, void *ws, bool static_weights, cudaStream_t stream);
constexpr int kGroupedMaxProblems = 4096;
size_t w4a16_prefill_ws_bytes(int M, int N, int K);
w4v_status launch_w4a16_prefill(const uint16_t *A, const void *Bq, const uint16_t *scales, const uint8_t *zeros,
                                int group, uint16_t *C, int M, int N, int K, void *ws, cudaStream_t stream);
// Rows up to which the verify-sized (HBM-bound) kernel is used.
constexpr int kDecodeMaxRows = 32;

// Prompt-lookup drafting: longest suffix n-gram searched, n <= kNgramMax.
constexpr int kNgramMax = 64;
size_t ngram_ws_bytes(int B);
w4v_status launch_ngram_draft(const int32_t *context, const int32_t *lengths, int B, long long ld, int n_min,
                              int n_max, int K, int32_t *draft, int32_t *match, void *ws, cudaStream_t stream);

// Gated DeltaNet state over a verify block: key width and longest block.
constexpr int kGdnDk = 128;
constexpr int kGdnMaxT = 64;
w4v_status launch_gdn(bool commit, float *state, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                      const float *alpha, const float *beta, const int32_t *n_accepted, uint16_t *o, int B, int T,
                      int H, int dv, cudaStream_t stream);
// Commit of the previous block (T_prev positions, n_prev accepted; T_prev = 0:
// none), then verify of the current one, in one launch.
w4v_status launch_gdn_step(float *state, const uint16_t *k_prev, const uint16_t *v_prev, const float *alpha_prev,
                           const float *beta_prev, const int32_t *n_prev, int T_prev, const uint16_t *q,
                           const uint16_t *k, const uint16_t *v, const float *alpha, const float *beta, uint16_t *o,
                           int B, int T, int H, int dv, cudaStream_t stream);

// Greedy acceptance fused into the lm_head's last CTA: the M = B*(n_draft+1)
// rows are B verify blocks of n_draft+1 positions each.
struct LmAccept {
    const int32_t *draft;      // [B][n_draft]
    int B, n_draft;
    int32_t *n_accepted;       // [B]
    int32_t *out_tokens;       // [B][n_draft+1] or null
};
w4v_status launch_w8_lmhead_argmax(const uint16_t *X, const int8_t *W, const uint16_t *scale,
                                   int M, int K, int V, int32_t *argmax_out, float *maxlogit,
                                   float *logits, void *ws, cudaStream_t stream,
                                   const LmAccept *accept = nullptr);
size_t w8_lmhead_ws_bytes(int M, int V);

w4v_status launch_spec_accept(const int32_t *target, const int32_t *draft, int B, int K,
                              int32_t *n_accepted, int32_t *out_tokens, cudaStream_t stream);

}  // namespace w4v
