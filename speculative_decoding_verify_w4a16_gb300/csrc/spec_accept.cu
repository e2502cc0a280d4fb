// spec_accept.cu -- longest-prefix greedy acceptance, one warp per sequence.
//
// "Efficient LLM Challenge Results", section 3: the target keeps the longest
// draft prefix equal to its own greedy tokens; a -1 padding sentinel is
// accepted only if it equals the verifier's greedy token, i.e. never.  Each
// lane compares one position, a warp ballot marks the mismatches and the
// first set bit is the accepted length.
#include "runtime.h"
#include "sm103_ptx.cuh"

namespace w4v {
namespace {

constexpr int kWarps = 8;

__global__ void __launch_bounds__(32 * kWarps)
spec_accept_kernel(const int32_t *__restrict__ target, const int32_t *__restrict__ draft, int B, int K,
                   int32_t *__restrict__ n_out, int32_t *__restrict__ tok_out) {
    grid_dep_wait();       // target tokens come from the previous kernel
    grid_dep_launch();
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (b >= B) return;
    const int32_t *t = target + size_t(b) * (K + 1);
    const int32_t *d = draft + size_t(b) * K;
    int n = K;
    for (int base = 0; base < K; base += 32) {
        const int j = base + lane;
        bool miss = false;
        if (j < K) {
            const int32_t dj = d[j];
            miss = !(dj >= 0 && dj == t[j]);
        }
        const unsigned m = __ballot_sync(0xFFFFFFFFu, miss);
        if (m != 0u) {
            n = base + __ffs(m) - 1;
            break;
        }
    }
    if (lane == 0) n_out[b] = n;
    if (tok_out != nullptr) {
        int32_t *o = tok_out + size_t(b) * (K + 1);
        for (int j = lane; j <= K; j += 32) o[j] = j <= n ? t[j] : -1;
    }
}

}  // namespace

w4v_status launch_spec_accept(const int32_t *target, const int32_t *draft, int B, int K,
                              int32_t *n_accepted, int32_t *out_tokens, cudaStream_t stream) {
    const DeviceInfo *info = nullptr;
    w4v_status st = device_info(&info);
    if (st != W4V_OK) return st;
    const int grid = (B + kWarps - 1) / kWarps;
    if (launch_pdl(spec_accept_kernel, dim3(grid), dim3(32 * kWarps), 0, stream, target, draft, B, K, n_accepted,
                   out_tokens) != cudaSuccess) {
        cudaGetLastError();
        return W4V_ERR_CUDA;
    }
    return W4V_OK;
}

}  // namespace w4v
