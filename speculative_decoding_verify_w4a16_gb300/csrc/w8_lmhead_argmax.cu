// w8_lmhead_argmax.cu -- int8 lm_head fused with the greedy argmax.
//
// What it computes ("Efficient LLM Challenge Results", sections 3 and 5: an
// untied lm_head quantized to 8 bits; greedy, temperature-0 decoding):
//     tok[m] = argmax_v  s[v] * sum_k X[m][k] * W[v][k]
// fp32 accumulation, the per-row scale applied to the finished sum, ties to
// the lowest v, NaN counted as -inf.  The [M][V] logits never reach HBM.
//
// Design (the lm_head is one full read of V x K int8 weights per verify step,
// so it is bound by HBM bandwidth for the verify sizes):
//   * 128-row vocabulary tiles are the MMA's M side, activation rows its N
//     side in blocks of 16 (M <= 128).  Each CTA owns a contiguous run of
//     whole tiles.
//   * The int8 tile (128 x 128 bytes per k-chunk) arrives by 2-D TMA with
//     128-byte swizzle straight from the row-major [V][K] matrix; the
//     activation slice arrives the same way (reused from L2 by every CTA).
//   * Math warps widen int8 to exact fp16 (XOR 0x80, PRMT into the mantissa
//     of 1024, subtract 1152) and store the tile into tensor memory; one
//     thread issues tcgen05.mma with A from TMEM, accumulating the whole K in
//     TMEM.
//   * At the end of a tile each thread owns one vocabulary row: it scales its
//     logits, turns each into an order-preserving 32-bit key, and a warp
//     max-reduction plus a min-reduction over the winning lanes gives the
//     lowest-index maximum of the warp; a shared-memory 64-bit atomicMax of
//     (key, ~index) keeps the CTA's best per row.
//   * CTAs publish their best keys; the last CTA to arrive (atomic counter,
//     no waiting) takes the maximum over CTAs and writes the token ids.
#include "runtime.h"
#include "sm103_ptx.cuh"

namespace w4v {
namespace {

constexpr int kTileV = 128;
constexpr int kChunk = 128;                 // k per unit (bytes of int8)
constexpr int kWBytes = kTileV * kChunk;    // 16 KB per unit
constexpr int kMathWarps = 8;
constexpr int kThreads = 32 * (4 + kMathWarps);
constexpr int kMaxRows = 128;

template <int NBLK>
struct Layout {
    static constexpr int kRows = 16 * NBLK;
    static constexpr int kActBox = kRows * 128;
    static constexpr int kAct = 2 * kActBox;
    static constexpr int kW = kAct;                     // 1024-aligned
    static constexpr int kS = kW + kWBytes;
    static constexpr int kStage = ((kS + 256 + 1023) / 1024) * 1024;
    static constexpr int kStages = (200 * 1024) / kStage > 8 ? 8 : (200 * 1024) / kStage;
    static constexpr int kASlots = NBLK <= 2 ? 3 : 4;
    static constexpr uint32_t kTmemCols = NBLK <= 2 ? 256 : 512;
    static constexpr uint32_t kAcol0 = 0;
    static constexpr uint32_t kDcol0 = kASlots * 64;
    static constexpr int kBar = kStages * kStage;
    static constexpr int kNumBars = 2 * kStages + 2 * kASlots + 4 + 2;
    static constexpr int kBest = ((kBar + 8 * kNumBars + 7) / 8) * 8;   // u64 [128]
    static constexpr int kMisc = kBest + 8 * kMaxRows;
    static constexpr int kBytes = kMisc + 64 + 1024;
    static_assert(kDcol0 + 2 * 16 * NBLK <= kTmemCols, "tensor memory plan");
};

struct Args {
    const int8_t *W;
    const __half *scale;
    int32_t *argmax_out;
    float *maxlogit;
    float *logits;
    unsigned long long *keys;   // [kMaxCtas][128]
    uint32_t *counter;
    uint32_t *status;
    int M, K, V;
    int n_tiles, n_chunks;
    int P;
};

// Order-preserving map of an fp32 logit to uint32 (NaN -> -inf, -0 -> +0).
__device__ __forceinline__ uint32_t logit_key(float x) {
    uint32_t b = __float_as_uint(x);
    if ((b & 0x7F800000u) == 0x7F800000u && (b & 0x007FFFFFu)) b = 0xFF800000u;   // NaN
    if ((b & 0x7FFFFFFFu) == 0u) b = 0u;                                            // -0
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float key_logit(uint32_t k) {
    const uint32_t b = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
    return __uint_as_float(b);
}

template <int NBLK>
__global__ void __launch_bounds__(kThreads, 1)
w8_lmhead_argmax_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap wmap,
                        const Args p) {
    using L = Layout<NBLK>;
    constexpr int kStages = L::kStages;
    constexpr int kASlots = L::kASlots;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    uint8_t *base = smem_raw + (base_s - raw_s);

    const uint32_t bar0 = base_s + L::kBar;
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (kStages + s); };
    auto afull = [&](int a) { return bar0 + 8u * (2 * kStages + a); };
    auto aempty = [&](int a) { return bar0 + 8u * (2 * kStages + kASlots + a); };
    auto dfull = [&](int b) { return bar0 + 8u * (2 * kStages + 2 * kASlots + b); };
    auto dempty = [&](int b) { return bar0 + 8u * (2 * kStages + 2 * kASlots + 2 + b); };
    const uint32_t done_bar = bar0 + 8u * (2 * kStages + 2 * kASlots + 4);
    const uint32_t math_bar = bar0 + 8u * (2 * kStages + 2 * kASlots + 5);
    unsigned long long *best = reinterpret_cast<unsigned long long *>(base + L::kBest);
    uint32_t *misc = reinterpret_cast<uint32_t *>(base + L::kMisc);   // [0] tmem, [1] abort, [2] last

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int cta = blockIdx.x;
    const int tb = static_cast<int>(split_begin(cta, p.n_tiles, p.P));
    const int te = static_cast<int>(split_begin(cta + 1, p.n_tiles, p.P));
    const int nunits = (te - tb) * p.n_chunks;
    AbortState ab{reinterpret_cast<volatile uint32_t *>(&misc[1]), p.status};

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), kMathWarps + 1);
        }
        for (int a = 0; a < kASlots; ++a) {
            mbar_init(afull(a), kMathWarps);
            mbar_init(aempty(a), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(dfull(b), 1);
            mbar_init(dempty(b), kMathWarps);
        }
        mbar_init(done_bar, 1);
        mbar_init(math_bar, kMathWarps);
        misc[1] = 0;
        misc[2] = 0;
        fence_barrier_init();
    }
    if (threadIdx.x < kMaxRows) best[threadIdx.x] = 0ull;
    if (warp == 2) {
        tmem_alloc(smem_u32(&misc[0]), L::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];

    if (warp == 0) {
        if (lane == 0) {
            prefetch_tensormap(&xmap);
            prefetch_tensormap(&wmap);
            const uint64_t pol_w = l2_policy_evict_first();
            const uint64_t pol_x = l2_policy_evict_last();
            int issued = 0;
            for (int i = 0; i < nunits; ++i) {
                const int s = i % kStages;
                if (i >= kStages && !mbar_wait(empty(s), ((i / kStages) - 1) & 1, ab)) break;
                const int t = tb + i / p.n_chunks;
                const int c = i % p.n_chunks;
                const uint32_t st = base_s + s * L::kStage;
                const uint32_t sbytes = c == 0 ? 2u * uint32_t(min(kTileV, p.V - t * kTileV)) : 0u;
                mbar_arrive_expect_tx(full(s), kWBytes + L::kAct + sbytes);
                tma_load_2d(st + L::kW, &wmap, c * kChunk, t * kTileV, full(s), pol_w);
                tma_load_2d(st, &xmap, c * kChunk, 0, full(s), pol_x);
                tma_load_2d(st + L::kActBox, &xmap, c * kChunk + 64, 0, full(s), pol_x);
                if (sbytes) bulk_load(st + L::kS, p.scale + size_t(t) * kTileV, sbytes, full(s), pol_w);
                ++issued;
            }
            if (*ab.flag) {
                for (int i = max(0, issued - kStages); i < issued; ++i)
                    mbar_wait_bounded(full(i % kStages), (i / kStages) & 1);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16_f32(128, 16);
            for (int i = 0; i < nunits; ++i) {
                const int s = i % kStages;
                const int slot = i % kASlots;
                const int j = i / p.n_chunks;
                const int c = i % p.n_chunks;
                const int buf = j & 1;
                if (!mbar_wait(full(s), (i / kStages) & 1, ab)) break;
                if (!mbar_wait(afull(slot), (i / kASlots) & 1, ab)) break;
                if (c == 0 && j >= 2 && !mbar_wait(dempty(buf), ((j >> 1) - 1) & 1, ab)) break;
                tc_fence_after();
                const uint32_t act = base_s + s * L::kStage;
#pragma unroll
                for (int kk = 0; kk < kChunk / 16; ++kk) {
#pragma unroll
                    for (int b = 0; b < NBLK; ++b) {
                        const uint32_t baddr = act + (kk >> 2) * L::kActBox + b * 2048 + (kk & 3) * 32;
                        mma_f16_ts(tmem + L::kDcol0 + buf * 16 * NBLK + 16 * b,
                                   tmem + L::kAcol0 + slot * 64 + 8 * kk, sdesc_sw128(baddr), idesc,
                                   (c > 0 || kk > 0) ? 1u : 0u);
                    }
                }
                mma_commit(empty(s));
                mma_commit(aempty(slot));
                if (c == p.n_chunks - 1) mma_commit(dfull(buf));
            }
            mma_commit(done_bar);
            mbar_wait_bounded(done_bar, 0);
        }
    } else if (warp >= 4) {
        const int mw = warp - 4;
        const int q = warp & 3;
        const int h = mw >> 2;
        const int r = 32 * q + lane;
        const uint32_t lane_base = uint32_t(32 * q) << 16;
        float scale_q[2] = {0.f, 0.f};
        const __half2 bias = u32_as_h2(0x64806480u);    // 1152 = 1024 + 128 in both halves
        uint32_t math_syncs = 0;
        auto math_sync = [&]() -> bool {
            __syncwarp();
            if (lane == 0) mbar_arrive(math_bar);
            return warp_wait(math_bar, (math_syncs++) & 1, ab);
        };

        auto dequant = [&](int i) -> bool {
            const int s = i % kStages;
            if (!warp_wait(full(s), (i / kStages) & 1, ab)) return false;
            const uint8_t *st = base + s * L::kStage;
            const int j = i / p.n_chunks;
            const int c = i % p.n_chunks;
            uint4 w[4];
#pragma unroll
            for (int ci = 0; ci < 4; ++ci) {
                const int chunk = 4 * h + ci;
                const int phys = chunk ^ (r & 7);            // 128-byte swizzle of the TMA box
                w[ci] = *reinterpret_cast<const uint4 *>(st + L::kW + r * 128 + phys * 16);
            }
            if (c == 0) {
                const int v = (tb + j) * kTileV + r;
                scale_q[j & 1] = v < p.V ? __half2float(reinterpret_cast<const __half *>(st + L::kS)[r]) : 0.f;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty(s));
            uint32_t regs[32];
#pragma unroll
            for (int ci = 0; ci < 4; ++ci) {
                const uint32_t words[4] = {w[ci].x, w[ci].y, w[ci].z, w[ci].w};
#pragma unroll
                for (int wd = 0; wd < 4; ++wd) {
                    const uint32_t u = words[wd] ^ 0x80808080u;        // int8 b -> b + 128
                    const uint32_t p01 = prmt(u, 0x64646464u, 0x4140u); // (1024+u0, 1024+u1)
                    const uint32_t p23 = prmt(u, 0x64646464u, 0x4342u); // (1024+u2, 1024+u3)
                    regs[8 * ci + 2 * wd + 0] = h2_as_u32(__hsub2(u32_as_h2(p01), bias));
                    regs[8 * ci + 2 * wd + 1] = h2_as_u32(__hsub2(u32_as_h2(p23), bias));
                }
            }
            const int slot = i % kASlots;
            if (i >= kASlots && !warp_wait(aempty(slot), ((i / kASlots) - 1) & 1, ab)) return false;
            tc_fence_after();
            tmem_st_32x32b_x32(tmem + lane_base + L::kAcol0 + slot * 64 + 32 * h, regs);
            tc_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(afull(slot));
            return true;
        };

        auto drain_tile = [&](int j) -> bool {
            const int buf = j & 1;
            if (!warp_wait(dfull(buf), (j >> 1) & 1, ab)) return false;
            tc_fence_after();
            uint32_t d[NBLK][8];
#pragma unroll
            for (int b = 0; b < NBLK; ++b)
                tmem_ld_32x32b_x8(tmem + lane_base + L::kDcol0 + buf * 16 * NBLK + 16 * b + 8 * h, d[b]);
            tc_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(dempty(buf));
            const int t = tb + j;
            const int v = t * kTileV + r;
            const bool valid = v < p.V;
            const float sc = scale_q[j & 1];
#pragma unroll
            for (int b = 0; b < NBLK; ++b) {
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) {
                    const int m = 16 * b + 8 * h + jj;
                    const float x = sc * __uint_as_float(d[b][jj]);
                    if (p.logits != nullptr && valid && m < p.M) p.logits[size_t(m) * p.V + v] = x;
                    const uint32_t key = valid ? logit_key(x) : 0u;
                    const uint32_t wmax = __reduce_max_sync(0xFFFFFFFFu, key);
                    const uint32_t wlane = __reduce_min_sync(0xFFFFFFFFu, key == wmax ? uint32_t(lane) : 32u);
                    if (lane == 0 && m < p.M && wmax != 0u) {
                        const uint32_t vbest = uint32_t(t * kTileV + 32 * q) + wlane;
                        atomicMax(&best[m], (static_cast<unsigned long long>(wmax) << 32) |
                                                (0xFFFFFFFFull - vbest));
                    }
                }
            }
            return true;
        };

        bool ok = true;
        for (int i = 0; i < nunits && ok; ++i) {
            ok = dequant(i);
            if (ok && i > 0 && (i % p.n_chunks) == 0) ok = drain_tile(i / p.n_chunks - 1);
        }
        if (ok && nunits > 0) ok = drain_tile(nunits / p.n_chunks - 1);

        // Publish this CTA's best per row; the last CTA reduces over all CTAs.
        if (ok) ok = math_sync();
        if (ok) {
            const int tid = mw * 32 + lane;
            if (tid < p.M) __stcg(p.keys + size_t(cta) * kMaxRows + tid, best[tid]);
            __threadfence();
            ok = math_sync();
        }
        if (ok) {
            if (mw == 0 && lane == 0) {
                const uint32_t prev = atomicAdd(p.counter, 1u);
                const bool last = prev == uint32_t(p.P - 1);
                if (last) atomicExch(p.counter, 0u);
                misc[2] = last ? 1u : 0u;
            }
            ok = math_sync();
        }
        if (ok && misc[2]) {
            __threadfence();
            const int tid = mw * 32 + lane;
            if (tid < p.M) {
                unsigned long long k = 0ull;
                for (int cc = 0; cc < p.P; ++cc) {
                    const unsigned long long o = __ldcg(p.keys + size_t(cc) * kMaxRows + tid);
                    k = o > k ? o : k;
                }
                p.argmax_out[tid] = static_cast<int32_t>(0xFFFFFFFFu - uint32_t(k & 0xFFFFFFFFull));
                if (p.maxlogit != nullptr) p.maxlogit[tid] = key_logit(uint32_t(k >> 32));
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, L::kTmemCols);
    }
}

template <int NBLK>
w4v_status launch(const CUtensorMap &xmap, const CUtensorMap &wmap, const Args &a, cudaStream_t stream) {
    using L = Layout<NBLK>;
    static int configured_for = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_for != dev) {
        if (cudaFuncSetAttribute(w8_lmhead_argmax_kernel<NBLK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 L::kBytes) != cudaSuccess) {
            cudaGetLastError();
            return W4V_ERR_CUDA;
        }
        configured_for = dev;
    }
    w8_lmhead_argmax_kernel<NBLK><<<a.P, kThreads, L::kBytes, stream>>>(xmap, wmap, a);
    return cudaGetLastError() == cudaSuccess ? W4V_OK : W4V_ERR_CUDA;
}

}  // namespace

size_t w8_lmhead_ws_bytes(int M, int V) {
    (void)M;
    (void)V;
    return size_t(kMaxCtas) * kMaxRows * sizeof(unsigned long long) + 256;
}

w4v_status launch_w8_lmhead_argmax(const uint16_t *X, const int8_t *W, const uint16_t *scale,
                                   int M, int K, int V, int32_t *argmax_out, float *maxlogit,
                                   float *logits, void *ws, cudaStream_t stream) {
    const DeviceInfo *info = nullptr;
    w4v_status st = device_info(&info);
    if (st != W4V_OK) return st;
    int nblk = (M + 15) / 16;
    nblk = nblk <= 1 ? 1 : nblk <= 2 ? 2 : nblk <= 4 ? 4 : 8;
    Args a;
    a.W = W;
    a.scale = reinterpret_cast<const __half *>(scale);
    a.argmax_out = argmax_out;
    a.maxlogit = maxlogit;
    a.logits = logits;
    a.keys = static_cast<unsigned long long *>(ws);
    a.counter = reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(ws) +
                                             size_t(kMaxCtas) * kMaxRows * sizeof(unsigned long long));
    a.status = info->status;
    a.M = M;
    a.K = K;
    a.V = V;
    a.n_tiles = (V + kTileV - 1) / kTileV;
    a.n_chunks = K / kChunk;
    a.P = std::min(std::min(info->sm_count, kMaxCtas), a.n_tiles);
    CUtensorMap xmap, wmap;
    st = encode_tmap_2d(&xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, X, uint64_t(K), uint64_t(M),
                        uint64_t(K) * 2, 64, 16 * nblk, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != W4V_OK) return st;
    st = encode_tmap_2d(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, W, uint64_t(K), uint64_t(V), uint64_t(K),
                        kChunk, kTileV, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != W4V_OK) return st;
    switch (nblk) {
        case 1: return launch<1>(xmap, wmap, a, stream);
        case 2: return launch<2>(xmap, wmap, a, stream);
        case 4: return launch<4>(xmap, wmap, a, stream);
        default: return launch<8>(xmap, wmap, a, stream);
    }
}

}  // namespace w4v
