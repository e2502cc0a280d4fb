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
//     S_t[i][:] = alpha_t S_{t-1}[i][:] + c_t[i] k_t^T,  c_t = beta_t (v_t - alpha_t u),
// which is the same product expanded, and the output follows from the same
// old state: o_t = S_t q_t = alpha_t (S_{t-1} q_t) + c_t (k_t . q_t).  So both
// dot products of a position read S_{t-1} side by side, and k_t . q_t is one
// number per position and head, formed once while staging.
//
// A warp owns 8 rows of S, lane l their columns 4l..4l+3 (32 values in
// registers for the whole block), a CTA 32 rows, and a head's rows are
// spread over dv/32 CTAs.  Each position reads k_t and q_t from shared memory
// once per warp (one 16-byte piece per lane, no lane reading what another
// does), forms the 8 rows' partial dot products in registers and reduces them
// across the warp by halving: at each of the first three butterfly steps a
// lane keeps half of its rows and sends the other half, so the 8 sums take 9
// shuffles and land in lane group l >> 2 (row l >> 2); 8 more shuffles hand
// every lane the 8 rows' update coefficients.  k, q (as fp32), k.q and the
// CTA's v, alpha, beta for the whole block are staged in shared memory first.
// Verify and commit run the same update, so the committed state is bit for
// bit the state verify ran through.
// gdn_step runs the commit of one block and the verify of the next in one
// launch (the state read once and written once); the same update code.
#include <algorithm>

#include "runtime.h"
#include "sm103_ptx.cuh"

namespace w4v {
namespace {

constexpr int kDk = kGdnDk;                 // 128 columns: 4 per lane
constexpr int kRowsPerWarp = 8;
constexpr int kWarps = 4;
constexpr int kRows = kRowsPerWarp * kWarps;   // rows of S per CTA
constexpr int kMaxT = kGdnMaxT;
static_assert(kDk == 4 * 32 && kRowsPerWarp == 8, "lane l owns columns 4l..4l+3 of 8 rows");

struct Args {
    float *state;                 // [B][H][dv][dk]
    const __half *q, *k, *v;      // [B][T][H][dk|dk|dv]
    const float *alpha, *beta;    // [B][T][H]
    const int32_t *n_accepted;    // commit: [B]
    __half *o;                    // verify: [B][T][H][dv]
    int B, T, H, dv;
};

// Dynamic shared memory: fp32 ks[T][dk], qs[T][dk] (verify), vs[T][kRows],
// as[T], bs[T], kq[T] (verify), then the raw fp16 copies kr[T][dk],
// qr[T][dk] (verify), vr[T][kRows] the fp32 arrays are made from.
__host__ __device__ constexpr size_t smem_f32(bool commit, int T) {
    return size_t(T) * (commit ? kDk + kRows + 2 : 2 * kDk + kRows + 3) * sizeof(float);
}
__host__ __device__ constexpr size_t smem_bytes(bool commit, int T) {
    return ((smem_f32(commit, T) + 15) & ~size_t(15)) + size_t(T) * (commit ? kDk + kRows : 2 * kDk + kRows) * 2;
}

// Two-wide fp32 arithmetic (each half rounds exactly like fmaf / a product):
// (s.x k.x + s.z k.z) + (s.y k.y + s.w k.w), each pair one fused step.
__device__ __forceinline__ float dot4(const float4 &s, const float4 &k) {
    const float2 m = __fmul2_rn(make_float2(s.z, s.w), make_float2(k.z, k.w));
    const float2 f = __ffma2_rn(make_float2(s.x, s.y), make_float2(k.x, k.y), m);
    return f.x + f.y;
}
// s <- fmaf(a, s, c k) per element.
__device__ __forceinline__ void update4(float4 &s, float a, float c, const float4 &k) {
    const float2 aa = make_float2(a, a), cc = make_float2(c, c);
    const float2 lo = __ffma2_rn(aa, make_float2(s.x, s.y), __fmul2_rn(cc, make_float2(k.x, k.y)));
    const float2 hi = __ffma2_rn(aa, make_float2(s.z, s.w), __fmul2_rn(cc, make_float2(k.z, k.w)));
    s = make_float4(lo.x, lo.y, hi.x, hi.y);
}

// The 8 rows' partial sums v[0..7] of every lane, summed over the warp;
// returns row (lane >> 2)'s total, the same bits in its four lanes.
__device__ __forceinline__ float warp_rows_sum(const float (&v)[kRowsPerWarp], int lane) {
    const bool b4 = (lane >> 4) & 1, b3 = (lane >> 3) & 1, b2 = (lane >> 2) & 1;
    float a[4], b[2];
#pragma unroll
    for (int i = 0; i < 4; ++i) {   // keep rows 4 b4 + i, send the others to lane ^ 16
        const float keep = b4 ? v[4 + i] : v[i], send = b4 ? v[i] : v[4 + i];
        a[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 16);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {   // rows 4 b4 + 2 b3 + i
        const float keep = b3 ? a[2 + i] : a[i], send = b3 ? a[i] : a[2 + i];
        b[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 8);
    }
    float c = (b2 ? b[1] : b[0]) + __shfl_xor_sync(0xFFFFFFFFu, b2 ? b[0] : b[1], 4);   // row lane >> 2
    c += __shfl_xor_sync(0xFFFFFFFFu, c, 2);
    c += __shfl_xor_sync(0xFFFFFFFFu, c, 1);
    return c;
}

// kCommit = false: outputs o_t for t < T, state untouched.
// kCommit = true:  state <- state after positions 0..n[b], no outputs.
template <bool kCommit>
__global__ void __launch_bounds__(32 * kWarps)
gdn_state_kernel(const Args p) {
    extern __shared__ __align__(16) float smem[];
    grid_dep_wait();                         // inputs come from the previous kernels
    grid_dep_launch();
    const int b = blockIdx.z, h = blockIdx.y;
    const int row0 = blockIdx.x * kRows;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rw = warp * kRowsPerWarp + (lane >> 2);   // the row whose sums this lane ends with
    int T = p.T;
    if (kCommit) {
        const int n = p.n_accepted[b];
        T = n < 0 ? 1 : (n + 1 > p.T ? p.T : n + 1);
    }
    float *ks = smem;
    float *qs = ks + size_t(p.T) * kDk;
    float *vs = qs + (kCommit ? 0 : size_t(p.T) * kDk);
    float *as = vs + size_t(p.T) * kRows;
    float *bs = as + p.T;
    float *kq = bs + p.T;
    __half *kr = reinterpret_cast<__half *>(reinterpret_cast<uint8_t *>(smem) +
                                            ((smem_f32(kCommit, p.T) + 15) & ~size_t(15)));
    __half *qr = kr + size_t(p.T) * kDk;
    __half *vr = qr + (kCommit ? 0 : size_t(p.T) * kDk);
    // this warp's 8 rows of the committed state, columns 4 lane..4 lane+3:
    // in flight while the block's inputs are copied
    float *S = p.state + ((size_t(b) * p.H + h) * p.dv + row0 + warp * kRowsPerWarp) * kDk + 4 * lane;
    float4 s[kRowsPerWarp];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) s[r] = *reinterpret_cast<const float4 *>(S + r * kDk);
    // every copy of the block's keys, queries, this CTA's values and the
    // gates issued at once (16-byte pieces; 4 bytes for the gates)
    for (int i = threadIdx.x; i < T * (kDk / 8); i += 32 * kWarps) {
        const int t = i / (kDk / 8), c = 8 * (i % (kDk / 8));
        const size_t base = ((size_t(b) * p.T + t) * p.H + h) * kDk + c;
        cp_async<16>(smem_u32(kr + t * kDk + c), p.k + base, 16u);
        if (!kCommit) cp_async<16>(smem_u32(qr + t * kDk + c), p.q + base, 16u);
    }
    for (int i = threadIdx.x; i < T * (kRows / 8); i += 32 * kWarps) {
        const int t = i / (kRows / 8), c = 8 * (i % (kRows / 8));
        cp_async<16>(smem_u32(vr + t * kRows + c), p.v + ((size_t(b) * p.T + t) * p.H + h) * p.dv + row0 + c, 16u);
    }
    for (int t = threadIdx.x; t < T; t += 32 * kWarps) {
        cp_async<4>(smem_u32(as + t), p.alpha + (size_t(b) * p.T + t) * p.H + h, 4u);
        cp_async<4>(smem_u32(bs + t), p.beta + (size_t(b) * p.T + t) * p.H + h, 4u);
    }
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();
    // to fp32: one warp per position for k and q (and k_t . q_t: lane l adds
    // columns 4l..4l+3, then a fixed tree), all threads for v
    for (int t = warp; t < T; t += kWarps) {
        const uint2 kw = *reinterpret_cast<const uint2 *>(kr + t * kDk + 4 * lane);
        const float2 k01 = __half22float2(u32_as_h2(kw.x)), k23 = __half22float2(u32_as_h2(kw.y));
        *reinterpret_cast<float4 *>(ks + t * kDk + 4 * lane) = make_float4(k01.x, k01.y, k23.x, k23.y);
        if (!kCommit) {
            const uint2 qw = *reinterpret_cast<const uint2 *>(qr + t * kDk + 4 * lane);
            const float2 q01 = __half22float2(u32_as_h2(qw.x)), q23 = __half22float2(u32_as_h2(qw.y));
            *reinterpret_cast<float4 *>(qs + t * kDk + 4 * lane) = make_float4(q01.x, q01.y, q23.x, q23.y);
            float d = (k01.x * q01.x + k01.y * q01.y) + (k23.x * q23.x + k23.y * q23.y);
#pragma unroll
            for (int m = 16; m > 0; m >>= 1) d += __shfl_xor_sync(0xFFFFFFFFu, d, m);
            if (lane == 0) kq[t] = d;
        }
    }
    for (int i = threadIdx.x; i < T * kRows; i += 32 * kWarps) vs[i] = __half2float(vr[i]);
    __syncthreads();

    for (int t = 0; t < T; ++t) {
        const float4 kv = *reinterpret_cast<const float4 *>(ks + t * kDk + 4 * lane);
        const float a = as[t], be = bs[t];
        // the 8 rows' parts of u = S_{t-1} k_t and w = S_{t-1} q_t
        float pu[kRowsPerWarp], pw[kRowsPerWarp];
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) pu[r] = dot4(s[r], kv);
        if (!kCommit) {
            const float4 qv = *reinterpret_cast<const float4 *>(qs + t * kDk + 4 * lane);
#pragma unroll
            for (int r = 0; r < kRowsPerWarp; ++r) pw[r] = dot4(s[r], qv);
        }
        const float u = warp_rows_sum(pu, lane);                          // row rw
        const float coef = be * (vs[t * kRows + rw] - a * u);
        if (!kCommit) {
            const float w = warp_rows_sum(pw, lane);
            const float y = fmaf(a, w, coef * kq[t]);                     // (S_t q_t)[rw]
            if ((lane & 3) == 0) p.o[((size_t(b) * p.T + t) * p.H + h) * p.dv + row0 + rw] = __float2half_rn(y);
        }
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) {
            const float cr = __shfl_sync(0xFFFFFFFFu, coef, 4 * r);       // row r's coefficient
            update4(s[r], a, cr, kv);
        }
    }
    if (kCommit) {
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) *reinterpret_cast<float4 *>(S + r * kDk) = s[r];
    }
}

template <bool kCommit>
w4v_status launch(const Args &a, cudaStream_t stream) {
    static int configured_for = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_for != dev) {
        if (cudaFuncSetAttribute(gdn_state_kernel<kCommit>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(smem_bytes(kCommit, kMaxT))) != cudaSuccess) {
            cudaGetLastError();
            return W4V_ERR_CUDA;
        }
        configured_for = dev;
    }
    const dim3 grid(a.dv / kRows, a.H, a.B);
    if (launch_pdl(gdn_state_kernel<kCommit>, grid, dim3(32 * kWarps), smem_bytes(kCommit, a.T), stream, a) !=
        cudaSuccess) {
        cudaGetLastError();
        return W4V_ERR_CUDA;
    }
    return W4V_OK;
}


// One verify block's inputs (and outputs).
struct Block {
    const __half *q, *k, *v;      // [B][T][H][dk|dk|dv] (q: verify only)
    const float *alpha, *beta;    // [B][T][H]
    __half *o;                    // verify: [B][T][H][dv]
    int T;                        // positions in the block (its arrays' T)
};

struct StepArgs {
    float *state;                 // [B][H][dv][dk]
    Block cur;                    // the block verified
    Block prev;                   // the previous block, committed first (T = 0: none)
    const int32_t *n_accepted;    // accepted drafts of the previous block [B]
    int B, H, dv;
};

// Runs positions 0..T-1 of block `blk` on the lane's rows s (8 rows, columns
// 4 lane..4 lane+3).  kCommit = false: writes o_t; kCommit = true: only
// advances s.  Every thread of the CTA calls it (it stages through shared
// memory and synchronises).  The same arithmetic as gdn_state_kernel, which
// keeps its own copy: written through this function the single-block
// kernels were compiled to fewer registers (64 / 56 against 72 / 64) and ran
// 10-17 % slower.
template <bool kCommit>
__device__ __forceinline__ void run_block(const Block &blk, int T, float4 (&s)[kRowsPerWarp], float *smem, int b,
                                          int h, int H, int dv, int row0) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rw = warp * kRowsPerWarp + (lane >> 2);   // the row whose sums this lane ends with
    const int BT = blk.T;
    float *ks = smem;
    float *qs = ks + size_t(BT) * kDk;
    float *vs = qs + (kCommit ? 0 : size_t(BT) * kDk);
    float *as = vs + size_t(BT) * kRows;
    float *bs = as + BT;
    float *kq = bs + BT;
    __half *kr = reinterpret_cast<__half *>(reinterpret_cast<uint8_t *>(smem) +
                                            ((smem_f32(kCommit, BT) + 15) & ~size_t(15)));
    __half *qr = kr + size_t(BT) * kDk;
    __half *vr = qr + (kCommit ? 0 : size_t(BT) * kDk);
    // every copy of the block's keys, queries, this CTA's values and the
    // gates issued at once (16-byte pieces; 4 bytes for the gates)
    for (int i = threadIdx.x; i < T * (kDk / 8); i += 32 * kWarps) {
        const int t = i / (kDk / 8), c = 8 * (i % (kDk / 8));
        const size_t base = ((size_t(b) * BT + t) * H + h) * kDk + c;
        cp_async<16>(smem_u32(kr + t * kDk + c), blk.k + base, 16u);
        if (!kCommit) cp_async<16>(smem_u32(qr + t * kDk + c), blk.q + base, 16u);
    }
    for (int i = threadIdx.x; i < T * (kRows / 8); i += 32 * kWarps) {
        const int t = i / (kRows / 8), c = 8 * (i % (kRows / 8));
        cp_async<16>(smem_u32(vr + t * kRows + c), blk.v + ((size_t(b) * BT + t) * H + h) * dv + row0 + c, 16u);
    }
    for (int t = threadIdx.x; t < T; t += 32 * kWarps) {
        cp_async<4>(smem_u32(as + t), blk.alpha + (size_t(b) * BT + t) * H + h, 4u);
        cp_async<4>(smem_u32(bs + t), blk.beta + (size_t(b) * BT + t) * H + h, 4u);
    }
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();
    // to fp32: one warp per position for k and q (and k_t . q_t: lane l adds
    // columns 4l..4l+3, then a fixed tree), all threads for v
    for (int t = warp; t < T; t += kWarps) {
        const uint2 kw = *reinterpret_cast<const uint2 *>(kr + t * kDk + 4 * lane);
        const float2 k01 = __half22float2(u32_as_h2(kw.x)), k23 = __half22float2(u32_as_h2(kw.y));
        *reinterpret_cast<float4 *>(ks + t * kDk + 4 * lane) = make_float4(k01.x, k01.y, k23.x, k23.y);
        if (!kCommit) {
            const uint2 qw = *reinterpret_cast<const uint2 *>(qr + t * kDk + 4 * lane);
            const float2 q01 = __half22float2(u32_as_h2(qw.x)), q23 = __half22float2(u32_as_h2(qw.y));
            *reinterpret_cast<float4 *>(qs + t * kDk + 4 * lane) = make_float4(q01.x, q01.y, q23.x, q23.y);
            float d = (k01.x * q01.x + k01.y * q01.y) + (k23.x * q23.x + k23.y * q23.y);
#pragma unroll
            for (int m = 16; m > 0; m >>= 1) d += __shfl_xor_sync(0xFFFFFFFFu, d, m);
            if (lane == 0) kq[t] = d;
        }
    }
    for (int i = threadIdx.x; i < T * kRows; i += 32 * kWarps) vs[i] = __half2float(vr[i]);
    __syncthreads();

    for (int t = 0; t < T; ++t) {
        const float4 kv = *reinterpret_cast<const float4 *>(ks + t * kDk + 4 * lane);
        const float a = as[t], be = bs[t];
        // the 8 rows' parts of u = S_{t-1} k_t and w = S_{t-1} q_t
        float pu[kRowsPerWarp], pw[kRowsPerWarp];
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) pu[r] = dot4(s[r], kv);
        if (!kCommit) {
            const float4 qv = *reinterpret_cast<const float4 *>(qs + t * kDk + 4 * lane);
#pragma unroll
            for (int r = 0; r < kRowsPerWarp; ++r) pw[r] = dot4(s[r], qv);
        }
        const float u = warp_rows_sum(pu, lane);                          // row rw
        const float coef = be * (vs[t * kRows + rw] - a * u);
        if (!kCommit) {
            const float w = warp_rows_sum(pw, lane);
            const float y = fmaf(a, w, coef * kq[t]);                     // (S_t q_t)[rw]
            if ((lane & 3) == 0) blk.o[((size_t(b) * BT + t) * H + h) * dv + row0 + rw] = __float2half_rn(y);
        }
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) {
            const float cr = __shfl_sync(0xFFFFFFFFu, coef, 4 * r);       // row r's coefficient
            update4(s[r], a, cr, kv);
        }
    }
}

__device__ __forceinline__ int accepted_positions(const int32_t *n_accepted, int b, int T) {
    const int n = n_accepted[b];
    return n < 0 ? 1 : (n + 1 > T ? T : n + 1);     // positions 0..n, n clamped to [0, T-1]
}

// Commit of the previous block, then verify of the current one from the
// state just committed: one read and one write of the state for both.
__global__ void __launch_bounds__(32 * kWarps)
gdn_step_kernel(const StepArgs p) {
    extern __shared__ __align__(16) float smem[];
    grid_dep_wait();                         // inputs come from the previous kernels
    grid_dep_launch();
    const int b = blockIdx.z, h = blockIdx.y;
    const int row0 = blockIdx.x * kRows;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float *S = p.state + ((size_t(b) * p.H + h) * p.dv + row0 + warp * kRowsPerWarp) * kDk + 4 * lane;
    float4 s[kRowsPerWarp];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) s[r] = *reinterpret_cast<const float4 *>(S + r * kDk);
    if (p.prev.T > 0) {
        run_block<true>(p.prev, accepted_positions(p.n_accepted, b, p.prev.T), s, smem, b, h, p.H, p.dv, row0);
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) *reinterpret_cast<float4 *>(S + r * kDk) = s[r];
        __syncthreads();                     // shared memory is staged again for the next block
    }
    run_block<false>(p.cur, p.cur.T, s, smem, b, h, p.H, p.dv, row0);
}

size_t step_smem(int T, int T_prev) { return std::max(smem_bytes(false, T), smem_bytes(true, T_prev)); }

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

w4v_status launch_gdn_step(float *state, const uint16_t *k_prev, const uint16_t *v_prev, const float *alpha_prev,
                           const float *beta_prev, const int32_t *n_prev, int T_prev, const uint16_t *q,
                           const uint16_t *k, const uint16_t *v, const float *alpha, const float *beta, uint16_t *o,
                           int B, int T, int H, int dv, cudaStream_t stream) {
    const DeviceInfo *info = nullptr;
    w4v_status st = device_info(&info);
    if (st != W4V_OK) return st;
    static int configured_for = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_for != dev) {
        if (cudaFuncSetAttribute(gdn_step_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(step_smem(kMaxT, kMaxT))) != cudaSuccess) {
            cudaGetLastError();
            return W4V_ERR_CUDA;
        }
        configured_for = dev;
    }
    StepArgs a = {};
    a.state = state;
    a.cur = Block{reinterpret_cast<const __half *>(q), reinterpret_cast<const __half *>(k),
                  reinterpret_cast<const __half *>(v), alpha, beta, reinterpret_cast<__half *>(o), T};
    a.prev = Block{nullptr, reinterpret_cast<const __half *>(k_prev), reinterpret_cast<const __half *>(v_prev),
                   alpha_prev, beta_prev, nullptr, T_prev};
    a.n_accepted = n_prev;
    a.B = B;
    a.H = H;
    a.dv = dv;
    if (launch_pdl(gdn_step_kernel, dim3(dv / kRows, H, B), dim3(32 * kWarps), step_smem(T, T_prev), stream, a) !=
        cudaSuccess) {
        cudaGetLastError();
        return W4V_ERR_CUDA;
    }
    return W4V_OK;
}

}  // namespace w4v
