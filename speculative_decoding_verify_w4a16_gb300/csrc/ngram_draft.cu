// ngram_draft.cu -- model-free drafting by prompt lookup, on the device.
//
// "Efficient LLM Challenge Results", section 3 (table of drafting methods):
// n-gram / prompt-lookup drafting copies spans from the prompt and needs no
// auxiliary model; the runner-up pads drafts to a constant K with -1.  For a
// context c[0..L-1] the drafts follow the latest earlier occurrence of the
// longest suffix n-gram (n_min <= n <= n_max) that has one, padded with -1
// where the context ends.
//
// Instead of one search per n, every candidate end position e (0 <= e <= L-2)
// gets its backward match length against the context's end,
//     l(e) = max m <= n_max with c[e-i] == c[L-1-i] for all i < m,
// so the n-gram of length n occurs ending at e exactly when l(e) >= n.  The
// longest n with an occurrence is the largest l(e), and its latest
// occurrence the largest e with that l: one maximum of the 64-bit key
// (l << 32 | e) over all e, where e + 1 is where the drafts start.
//
// Design: a row's end positions are split over CTAs of 2048 (one read of the
// context, coalesced, each thread's eight first compares issued together;
// almost every position stops at its first compare).
// Each CTA reduces its best key in registers and shared memory and folds it
// into the row's key in the workspace with one 64-bit atomicMax; the last
// CTA of the row to arrive (acquire-release counter, no waiting) reads and
// clears it and writes the drafts.
#include "runtime.h"
#include "sm103_ptx.cuh"

namespace w4v {
namespace {

constexpr int kThreads = 256;
constexpr int kPerThread = 8;
constexpr int kChunk = kThreads * kPerThread;     // end positions per CTA

struct Args {
    const int32_t *ctx;
    const int32_t *len;
    int32_t *draft;
    int32_t *match;
    unsigned long long *key;     // [B], zero between calls
    uint32_t *counter;           // [B], zero between calls
    long long ld;
    int B, n_min, n_max, K, chunks;
};

__global__ void __launch_bounds__(kThreads)
ngram_draft_kernel(const Args p) {
    __shared__ int32_t suf[kNgramMax];
    __shared__ unsigned long long best;
    __shared__ uint32_t last;
    grid_dep_wait();       // the context may come from the previous kernel
    grid_dep_launch();
    const int b = blockIdx.y;
    const int tid = threadIdx.x;
    const int32_t *c = p.ctx + size_t(b) * size_t(p.ld);
    long long L = p.len[b];
    L = L < 0 ? 0 : (L > p.ld ? p.ld : L);
    const int nmax = static_cast<int>(L - 1 < p.n_max ? (L - 1 < 0 ? 0 : L - 1) : p.n_max);
    // suf[nmax-1-i] = c[L-1-i]: the context's last nmax tokens, right-aligned
    if (tid < nmax) suf[tid] = c[L - nmax + tid];
    if (tid == 0) best = 0ull;
    __syncthreads();

    unsigned long long mine = 0ull;
    if (nmax >= p.n_min) {
        const long long e0 = (long long)blockIdx.x * kChunk + tid;
        const long long e1 = L - 1;                             // ends e <= L - 2
        // all of this thread's first compares in flight at once; almost every
        // position stops there, the rest walk back from the second token
        int32_t v[kPerThread];
#pragma unroll
        for (int j = 0; j < kPerThread; ++j) {
            const long long e = e0 + j * kThreads;
            v[j] = e < e1 ? c[e] : 0;
        }
        const int32_t last_tok = suf[nmax - 1];
#pragma unroll
        for (int j = 0; j < kPerThread; ++j) {
            const long long e = e0 + j * kThreads;
            if (e < e1 && v[j] == last_tok) {
                int l = 1;
                while (l < nmax && l <= e && c[e - l] == suf[nmax - 1 - l]) ++l;
                if (l >= p.n_min) {
                    const unsigned long long k = (static_cast<unsigned long long>(l) << 32) | static_cast<uint32_t>(e);
                    mine = k > mine ? k : mine;
                }
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long other = __shfl_xor_sync(0xFFFFFFFFu, mine, o);
        mine = other > mine ? other : mine;
    }
    if ((tid & 31) == 0 && mine != 0ull) atomicMax(&best, mine);
    __syncthreads();
    if (tid == 0) {
        if (best != 0ull) atomicMax(p.key + b, best);
        const uint32_t prev = atom_add_acq_rel_gpu(p.counter + b, 1u);
        last = prev == uint32_t(p.chunks - 1) ? 1u : 0u;
        if (last) {
            best = atomicExch(p.key + b, 0ull);
            p.counter[b] = 0u;
        }
    }
    __syncthreads();
    if (!last) return;
    const int n = static_cast<int>(best >> 32);
    const long long start = n > 0 ? static_cast<long long>(best & 0xFFFFFFFFull) + 1 : L;
    if (tid == 0 && p.match != nullptr) p.match[b] = n;
    int32_t *d = p.draft + size_t(b) * p.K;
    for (int i = tid; i < p.K; i += kThreads) d[i] = start + i < L ? c[start + i] : -1;
}

}  // namespace

size_t ngram_ws_bytes(int B) { return size_t(B > 0 ? B : 0) * 16 + 256; }

w4v_status launch_ngram_draft(const int32_t *context, const int32_t *lengths, int B, long long ld, int n_min,
                              int n_max, int K, int32_t *draft, int32_t *match, void *ws, cudaStream_t stream) {
    const DeviceInfo *info = nullptr;
    w4v_status st = device_info(&info);
    if (st != W4V_OK) return st;
    Args a;
    a.ctx = context;
    a.len = lengths;
    a.draft = draft;
    a.match = match;
    a.key = static_cast<unsigned long long *>(ws);
    a.counter = reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(ws) + size_t(B) * 8);
    a.ld = ld;
    a.B = B;
    a.n_min = n_min;
    a.n_max = n_max;
    a.K = K;
    a.chunks = static_cast<int>(ld <= 1 ? 1 : (ld - 1 + kChunk - 1) / kChunk);
    if (launch_pdl(ngram_draft_kernel, dim3(a.chunks, B), dim3(kThreads), 0, stream, a) != cudaSuccess) {
        cudaGetLastError();
        return W4V_ERR_CUDA;
    }
    return W4V_OK;
}

}  // namespace w4v
