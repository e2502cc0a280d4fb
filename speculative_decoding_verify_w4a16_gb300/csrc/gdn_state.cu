// gdn_state.cu -- the Gated DeltaNet recurrent state across a verify block.
//
// Most of the target's layers are Gated DeltaNet, and a rejected draft must
// not leave its update in their recurrent state ("Efficient LLM Challenge
// Results", section 3, runner-up paragraph; "DFlash K=15 for Qwen3.5-4B on a
// single A10G", "What transfers").  The recurrence is the one of the first
// page's reference [12] (Yang et al., "Gated Delta Networks"), per head with
// state S [dv][dk]:
//     S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,  o_t = S_t q_t.
// Rolling back is done by never writing a speculative state: the verify
// kernel reads the committed state, runs the K+1 positions in registers and
// writes only the outputs; once the acceptance is known (on the device), the
// commit kernel replays positions 0..n of the block from the committed state
// and writes the result in place.  State traffic per step is one read for
// verify plus one read and one write for the commit -- no per-position
// snapshots (K+1 states per head) ever reach HBM.
//
// Each row of S evolves on its own: with u = S_{t-1} k_t,
//     S_t[i][:] = alpha_t S_{t-1}[i][:] + beta_t (v_t[i] - alpha_t u[i]) k_t^T,
// which is the same product expanded.  So a warp owns 8 rows (each lane 4
// columns of dk = 128, held in registers for the whole block), a CTA 32 rows,
// and a head's rows are spread over dv/32 CTAs.  k, q (fp16) and the CTA's
// v, alpha, beta for the whole block are staged in shared memory first.
#include "runtime.h"
#include "sm103_ptx.cuh"

namespace w4v {
namespace {

constexpr int kDk = kGdnDk;                 // 128 columns: 4 per lane
constexpr int kRowsPerWarp = 8;
constexpr int kWarps = 4;
constexpr int kRows = kRowsPerWarp * kWarps;   // rows of S per CTA
constexpr int kMaxT = kGdnMaxT;

struct Args {
    float *state;                 // [B][H][dv][dk]
    const __half *q, *k, *v;      // [B][T][H][dk|dk|dv]
    const float *alpha, *beta;    // [B][T][H]
    const int32_t *n_accepted;    // commit: [B]
    __half *o;                    // verify: [B][T][H][dv]
    int B, T, H, dv;
};

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, m);
    return x;
}

// kCommit = false: outputs o_t for t < T, state untouched.
// kCommit = true:  state <- state after positions 0..n[b], no outputs.
template <bool kCommit>
__global__ void __launch_bounds__(32 * kWarps)
gdn_state_kernel(const Args p) {
    __shared__ __half ks[kMaxT][kDk];
    __shared__ __half qs[kCommit ? 1 : kMaxT][kDk];
    __shared__ float vs[kMaxT][kRows];
    __shared__ float as[kMaxT], bs[kMaxT];
    grid_dep_wait();                         // inputs come from the previous kernels
    grid_dep_launch();
    const int b = blockIdx.z, h = blockIdx.y;
    const int row0 = blockIdx.x * kRows;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int T = p.T;
    if (kCommit) {
        const int n = p.n_accepted[b];
        T = n < 0 ? 1 : (n + 1 > p.T ? p.T : n + 1);
    }
    // stage the block's keys, queries, this CTA's values and the gates
    for (int i = threadIdx.x; i < T * kDk; i += 32 * kWarps) {
        const int t = i / kDk, c = i % kDk;
        const size_t base = ((size_t(b) * p.T + t) * p.H + h) * kDk + c;
        ks[t][c] = p.k[base];
        if (!kCommit) qs[t][c] = p.q[base];
    }
    for (int i = threadIdx.x; i < T * kRows; i += 32 * kWarps) {
        const int t = i / kRows, r = i % kRows;
        vs[t][r] = __half2float(p.v[((size_t(b) * p.T + t) * p.H + h) * p.dv + row0 + r]);
    }
    for (int t = threadIdx.x; t < T; t += 32 * kWarps) {
        as[t] = p.alpha[(size_t(b) * p.T + t) * p.H + h];
        bs[t] = p.beta[(size_t(b) * p.T + t) * p.H + h];
    }
    // this warp's rows of the committed state, 4 columns per lane
    float *S = p.state + ((size_t(b) * p.H + h) * p.dv + row0 + warp * kRowsPerWarp) * kDk;
    float s[kRowsPerWarp][4];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) s[r][c] = S[r * kDk + lane + 32 * c];
    __syncthreads();

    for (int t = 0; t < T; ++t) {
        float kk[4], qq[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            kk[c] = __half2float(ks[t][lane + 32 * c]);
            qq[c] = kCommit ? 0.f : __half2float(qs[t][lane + 32 * c]);
        }
        const float a = as[t], be = bs[t];
        float o_mine = 0.f;                  // lane r < 8 keeps row r's output
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) {
            float u = 0.f;
#pragma unroll
            for (int c = 0; c < 4; ++c) u = fmaf(s[r][c], kk[c], u);
            u = warp_sum(u);                 // (S_{t-1} k_t)[row]
            const float coef = be * (vs[t][warp * kRowsPerWarp + r] - a * u);
#pragma unroll
            for (int c = 0; c < 4; ++c) s[r][c] = fmaf(a, s[r][c], coef * kk[c]);
            if (!kCommit) {
                float y = 0.f;
#pragma unroll
                for (int c = 0; c < 4; ++c) y = fmaf(s[r][c], qq[c], y);
                y = warp_sum(y);             // (S_t q_t)[row]
                if (lane == r) o_mine = y;
            }
        }
        if (!kCommit && lane < kRowsPerWarp)
            p.o[((size_t(b) * p.T + t) * p.H + h) * p.dv + row0 + warp * kRowsPerWarp + lane] = __float2half_rn(o_mine);
    }
    if (kCommit) {
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
            for (int c = 0; c < 4; ++c) S[r * kDk + lane + 32 * c] = s[r][c];
    }
}

template <bool kCommit>
w4v_status launch(const Args &a, cudaStream_t stream) {
    const dim3 grid(a.dv / kRows, a.H, a.B);
    if (launch_pdl(gdn_state_kernel<kCommit>, grid, dim3(32 * kWarps), 0, stream, a) != cudaSuccess) {
        cudaGetLastError();
        return W4V_ERR_CUDA;
    }
    return W4V_OK;
}

}  // namespace

w4v_status launch_gdn(bool commit, float *state, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                      const float *alpha, const float *beta, const int32_t *n_accepted, uint16_t *o, int B, int T,
                      int H, int dv, cudaStream_t stream) {
    const DeviceInfo *info = nullptr;
    w4v_status st = device_info(&info);
    if (st != W4V_OK) return st;
    Args a;
    a.state = state;
    a.q = reinterpret_cast<const __half *>(q);
    a.k = reinterpret_cast<const __half *>(k);
    a.v = reinterpret_cast<const __half *>(v);
    a.alpha = alpha;
    a.beta = beta;
    a.n_accepted = n_accepted;
    a.o = reinterpret_cast<__half *>(o);
    a.B = B;
    a.T = T;
    a.H = H;
    a.dv = dv;
    return commit ? launch<true>(a, stream) : launch<false>(a, stream);
}

}  // namespace w4v
