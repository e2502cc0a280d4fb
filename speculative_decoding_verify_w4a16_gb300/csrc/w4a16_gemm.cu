// w4a16_gemm.cu -- W4A16 projection GEMM for verify-sized M (<= 32 rows).
//
// What it computes ("Efficient LLM Challenge Results", sections 3 and 5: a
// 4-bit W4A16 GPTQ target with group size 128 and fp16 activations):
//     C[m][n] = sum_g s[g][n] * sum_{k in g} A[m][k] * (q[n][k] - z[g][n])
// with fp32 accumulation per group and fp32 scaling, C rounded to fp16.
//
// Why it looks like this (section 2 of the same page: decode reads the whole
// weight set from HBM per step, so the K+1 verify rows must share one weight
// read):
//   * The weights are the wide operand.  A 128-row weight tile is the MMA's
//     M side; the (<= 32) activation rows are its N side in blocks of 16, so
//     every output element comes from the same instruction shape whatever M
//     is (batch invariance for M <= 32).
//   * Packed int4 blocks stream from HBM with 1-D bulk copies (8 KB per
//     128x128 block, evict-first), the group scales / zeros ride along, and
//     the activation slice arrives by 2-D TMA with 128-byte swizzle.
//   * Eight math warps turn nibbles into exact fp16 integers (q - z) with a
//     LOP3 + HFMA2 bit trick and store them straight into tensor memory with
//     tcgen05.st: the dequantized operand never touches shared memory, which
//     keeps shared-memory bandwidth for the copies.
//   * One thread issues tcgen05.mma (A from TMEM, B from shared memory, D in
//     TMEM) per group; the math warps drain each group's fp32 result with
//     tcgen05.ld and apply the group scale in fp32 (0.125 FMA per weight).
//   * Work is the flat list of (tile, group) units split evenly over one CTA
//     per SM; a tile shared by several CTAs is finished by the last one to
//     arrive, which sums the fp32 partial tiles in CTA order (deterministic,
//     no waiting between CTAs).
#include "runtime.h"
#include "sm103_ptx.cuh"

namespace w4v {
namespace {

constexpr int kTileN = 128;                     // weight rows per tile (MMA M)
constexpr int kGroup = 128;                     // k per unit = one quant group
constexpr int kBlockBytes = kTileN * kGroup / 2; // packed bytes per unit
constexpr int kMathWarps = 8;
constexpr int kThreads = 32 * (4 + kMathWarps);
constexpr int kStages = 8;
constexpr int kASlots = 3;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kAcol0 = 0;
constexpr uint32_t kDcol0 = kASlots * 64;

template <int NBLK>
struct Layout {
    static constexpr int kRows = 16 * NBLK;             // activation rows per box
    static constexpr int kActBox = kRows * 128;         // one 64-k box, swizzled
    static constexpr int kAct = 2 * kActBox;
    static constexpr int kW = kAct;
    static constexpr int kS = kW + kBlockBytes;
    static constexpr int kZ = kS + 256;
    static constexpr int kStage = ((kZ + 128 + 1023) / 1024) * 1024;
    static constexpr int kBar = kStages * kStage;
    static constexpr int kNumBars = 2 * kStages + 2 * kASlots + 4 + 2;
    static constexpr int kMisc = kBar + 8 * kNumBars;
    static constexpr int kBytes = kMisc + 64 + 1024;     // + alignment slack
};

struct Args {
    const uint8_t *wq;
    const __half *scales;
    const uint8_t *zeros;
    __half *C;
    float *partial;        // [P][2][16*NBLK][128]
    uint32_t *tile_cnt;    // [n_tiles]
    uint32_t *status;
    int M, N, K;
    int n_tiles, n_groups;
    int P;
    long long U;
};

template <int NBLK>
__global__ void __launch_bounds__(kThreads, 1)
w4a16_decode_kernel(const __grid_constant__ CUtensorMap xmap, const Args p) {
    using L = Layout<NBLK>;
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
    uint32_t *misc = reinterpret_cast<uint32_t *>(base + L::kMisc);  // [0] tmem, [1] abort, [2] fixer

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int cta = blockIdx.x;
    const long long ub = split_begin(cta, p.U, p.P);
    const long long ue = split_begin(cta + 1, p.U, p.P);
    const int nunits = static_cast<int>(ue - ub);
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
    if (warp == 2) {
        tmem_alloc(smem_u32(&misc[0]), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];

    if (warp == 0) {
        // ------------------------------------------------------- producer
        if (lane == 0) {
            prefetch_tensormap(&xmap);
            const uint64_t pol_w = l2_policy_evict_first();
            const uint64_t pol_x = l2_policy_evict_last();
            int issued = 0;
            for (int i = 0; i < nunits; ++i) {
                const int s = i % kStages;
                if (i >= kStages && !mbar_wait(empty(s), ((i / kStages) - 1) & 1, ab)) break;
                const long long u = ub + i;
                const int t = static_cast<int>(u / p.n_groups);
                const int g = static_cast<int>(u % p.n_groups);
                const int rows = min(kTileN, p.N - t * kTileN);
                const uint32_t sbytes = 2u * rows;
                const uint32_t zbytes = p.zeros ? uint32_t(rows) : 0u;
                const uint32_t st = base_s + s * L::kStage;
                mbar_arrive_expect_tx(full(s), kBlockBytes + sbytes + zbytes + L::kAct);
                bulk_load(st + L::kW, p.wq + (size_t(t) * p.n_groups + g) * kBlockBytes, kBlockBytes,
                          full(s), pol_w);
                bulk_load(st + L::kS, p.scales + size_t(g) * p.N + size_t(t) * kTileN, sbytes, full(s),
                          pol_w);
                if (p.zeros)
                    bulk_load(st + L::kZ, p.zeros + size_t(g) * p.N + size_t(t) * kTileN, zbytes,
                              full(s), pol_w);
                tma_load_2d(st, &xmap, g * kGroup, 0, full(s), pol_x);
                tma_load_2d(st + L::kActBox, &xmap, g * kGroup + 64, 0, full(s), pol_x);
                ++issued;
            }
            if (*ab.flag) {
                // Let every copy still in flight land before the CTA exits.
                for (int i = max(0, issued - kStages); i < issued; ++i)
                    mbar_wait_bounded(full(i % kStages), (i / kStages) & 1);
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16_f32(128, 16);
            for (int i = 0; i < nunits; ++i) {
                const int s = i % kStages;
                const int slot = i % kASlots;
                const int buf = i & 1;
                if (!mbar_wait(full(s), (i / kStages) & 1, ab)) break;
                if (!mbar_wait(afull(slot), (i / kASlots) & 1, ab)) break;
                if (i >= 2 && !mbar_wait(dempty(buf), ((i >> 1) - 1) & 1, ab)) break;
                tc_fence_after();
                const uint32_t act = base_s + s * L::kStage;
#pragma unroll
                for (int j = 0; j < kGroup / 16; ++j) {
#pragma unroll
                    for (int b = 0; b < NBLK; ++b) {
                        const uint32_t baddr = act + (j >> 2) * L::kActBox + b * 2048 + (j & 3) * 32;
                        mma_f16_ts(tmem + kDcol0 + buf * 16 * NBLK + 16 * b,
                                   tmem + kAcol0 + slot * 64 + 8 * j, sdesc_sw128(baddr), idesc,
                                   j > 0 ? 1u : 0u);
                    }
                }
                mma_commit(empty(s));
                mma_commit(aempty(slot));
                mma_commit(dfull(buf));
            }
            // Every MMA this thread issued has finished once this arrives.
            mma_commit(done_bar);
            mbar_wait_bounded(done_bar, 0);
        }
    } else if (warp >= 4) {
        // ------------------------------------------- dequant + epilogue
        const int mw = warp - 4;
        const int q = warp & 3;                 // TMEM lane quarter
        const int h = mw >> 2;                  // k half (dequant), column half (drain)
        const int r = 32 * q + lane;            // row inside the tile
        const uint32_t lane_base = uint32_t(32 * q) << 16;
        float acc[NBLK][8];
#pragma unroll
        for (int b = 0; b < NBLK; ++b)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[b][j] = 0.f;
        float scale_q[2] = {0.f, 0.f};
        const __half2 sixteenth = __float2half2_rn(0.0625f);
        uint32_t math_syncs = 0;
        // Barrier over the math warps only, bounded like every other wait.
        auto math_sync = [&]() -> bool {
            __syncwarp();
            if (lane == 0) mbar_arrive(math_bar);
            return warp_wait(math_bar, (math_syncs++) & 1, ab);
        };

        auto dequant = [&](int i) -> bool {
            const int s = i % kStages;
            if (!warp_wait(full(s), (i / kStages) & 1, ab)) return false;
            const uint8_t *st = base + s * L::kStage;
            const uint4 w0 = *reinterpret_cast<const uint4 *>(st + L::kW + ((2 * h) * 128 + r) * 16);
            const uint4 w1 = *reinterpret_cast<const uint4 *>(st + L::kW + ((2 * h + 1) * 128 + r) * 16);
            const long long u = ub + i;
            const int t = static_cast<int>(u / p.n_groups);
            const int n = t * kTileN + r;
            float sc = 0.f;
            uint32_t z = 8;
            if (n < p.N) {
                sc = __half2float(reinterpret_cast<const __half *>(st + L::kS)[r]);
                if (p.zeros) z = st[L::kZ + r];
            }
            scale_q[i & 1] = sc;
            __syncwarp();
            if (lane == 0) mbar_arrive(empty(s));

            const __half2 zlo = u32_as_h2((0x6400u + z) * 0x10001u);          // 1024 + z
            const __half2 zhi = __float2half2_rn(-(64.f + float(z)));
            const uint32_t words[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
            uint32_t regs[32];
#pragma unroll
            for (int wi = 0; wi < 8; ++wi) {
                const uint32_t v = words[wi];
                const uint32_t v8 = v >> 8;
                // low nibbles give 1024 + q, high nibbles 1024 + 16 q (exact)
                const uint32_t lo0 = lop_and_or(v, 0x000F000Fu, 0x64006400u);
                const uint32_t hi0 = lop_and_or(v, 0x00F000F0u, 0x64006400u);
                const uint32_t lo1 = lop_and_or(v8, 0x000F000Fu, 0x64006400u);
                const uint32_t hi1 = lop_and_or(v8, 0x00F000F0u, 0x64006400u);
                regs[4 * wi + 0] = h2_as_u32(__hsub2(u32_as_h2(lo0), zlo));
                regs[4 * wi + 1] = h2_as_u32(__hfma2(u32_as_h2(hi0), sixteenth, zhi));
                regs[4 * wi + 2] = h2_as_u32(__hsub2(u32_as_h2(lo1), zlo));
                regs[4 * wi + 3] = h2_as_u32(__hfma2(u32_as_h2(hi1), sixteenth, zhi));
            }
            const int slot = i % kASlots;
            if (i >= kASlots && !warp_wait(aempty(slot), ((i / kASlots) - 1) & 1, ab)) return false;
            tc_fence_after();
            tmem_st_32x32b_x32(tmem + lane_base + kAcol0 + slot * 64 + 32 * h, regs);
            tc_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(afull(slot));
            return true;
        };

        auto flush = [&](int t) -> bool {
            const long long t0u = (long long)t * p.n_groups;
            const long long t1u = t0u + p.n_groups;
            const int n = t * kTileN + r;
            if (ub <= t0u && t1u <= ue) {
                if (n < p.N) {
#pragma unroll
                    for (int b = 0; b < NBLK; ++b)
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const int m = 16 * b + 8 * h + j;
                            if (m < p.M) p.C[size_t(m) * p.N + n] = __float2half_rn(acc[b][j]);
                        }
                }
                return true;
            }
            constexpr int kPart = 16 * NBLK * kTileN;
            const int slot = (ub >= t0u) ? 0 : 1;
            float *part = p.partial + (size_t(cta) * 2 + slot) * kPart;
#pragma unroll
            for (int b = 0; b < NBLK; ++b)
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int m = 16 * b + 8 * h + j;
                    if (m < p.M) __stcg(part + m * kTileN + r, acc[b][j]);
                }
            __threadfence();
            if (!math_sync()) return false;
            const int cf = split_owner(t0u, p.U, p.P);
            const int cl = split_owner(t1u - 1, p.U, p.P);
            if (mw == 0 && lane == 0) {
                const uint32_t prev = atomicAdd(&p.tile_cnt[t], 1u);
                const bool last = prev == uint32_t(cl - cf);
                if (last) atomicExch(&p.tile_cnt[t], 0u);
                misc[2] = last ? 1u : 0u;
            }
            if (!math_sync()) return false;
            if (misc[2]) {
                __threadfence();
                float sum[NBLK][8];
#pragma unroll
                for (int b = 0; b < NBLK; ++b)
#pragma unroll
                    for (int j = 0; j < 8; ++j) sum[b][j] = 0.f;
                for (int cc = cf; cc <= cl; ++cc) {
                    const int sl = (split_begin(cc, p.U, p.P) >= t0u) ? 0 : 1;
                    const float *src = p.partial + (size_t(cc) * 2 + sl) * kPart;
#pragma unroll
                    for (int b = 0; b < NBLK; ++b)
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const int m = 16 * b + 8 * h + j;
                            if (m < p.M) sum[b][j] += __ldcg(src + m * kTileN + r);
                        }
                }
                if (n < p.N) {
#pragma unroll
                    for (int b = 0; b < NBLK; ++b)
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const int m = 16 * b + 8 * h + j;
                            if (m < p.M) p.C[size_t(m) * p.N + n] = __float2half_rn(sum[b][j]);
                        }
                }
            }
            return true;
        };

        auto drain = [&](int i) -> bool {
            const int buf = i & 1;
            if (!warp_wait(dfull(buf), (i >> 1) & 1, ab)) return false;
            tc_fence_after();
            uint32_t d[NBLK][8];
#pragma unroll
            for (int b = 0; b < NBLK; ++b)
                tmem_ld_32x32b_x8(tmem + lane_base + kDcol0 + buf * 16 * NBLK + 16 * b + 8 * h, d[b]);
            tc_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(dempty(buf));
            const float sc = scale_q[i & 1];
#pragma unroll
            for (int b = 0; b < NBLK; ++b)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[b][j] = fmaf(sc, __uint_as_float(d[b][j]), acc[b][j]);
            const long long u = ub + i;
            const int t = static_cast<int>(u / p.n_groups);
            if (u + 1 == (long long)(t + 1) * p.n_groups || u + 1 == ue) {
                if (!flush(t)) return false;
#pragma unroll
                for (int b = 0; b < NBLK; ++b)
#pragma unroll
                    for (int j = 0; j < 8; ++j) acc[b][j] = 0.f;
            }
            return true;
        };

        bool ok = true;
        for (int i = 0; i < nunits && ok; ++i) {
            ok = dequant(i);
            if (ok && i > 0) ok = drain(i - 1);
        }
        if (ok && nunits > 0) drain(nunits - 1);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int NBLK>
w4v_status launch(const DeviceInfo *info, const CUtensorMap &xmap, const Args &a, cudaStream_t stream) {
    using L = Layout<NBLK>;
    static int configured_for = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_for != dev) {
        if (cudaFuncSetAttribute(w4a16_decode_kernel<NBLK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 L::kBytes) != cudaSuccess) {
            cudaGetLastError();
            return W4V_ERR_CUDA;
        }
        configured_for = dev;
    }
    w4a16_decode_kernel<NBLK><<<a.P, kThreads, L::kBytes, stream>>>(xmap, a);
    return cudaGetLastError() == cudaSuccess ? W4V_OK : W4V_ERR_CUDA;
}

}  // namespace

size_t w4a16_decode_ws_bytes(int M, int N, int K) {
    (void)K;
    const int nblk = (M + 15) / 16 < 1 ? 1 : (M + 15) / 16;
    const size_t n_tiles = (size_t(N) + kTileN - 1) / kTileN;
    const size_t part = size_t(kMaxCtas) * 2 * 16 * nblk * kTileN * sizeof(float);
    return part + ((n_tiles * sizeof(uint32_t) + 255) & ~size_t(255));
}

w4v_status launch_w4a16_decode(const uint16_t *A, const void *Bq, const uint16_t *scales,
                               const uint8_t *zeros, uint16_t *C, int M, int N, int K,
                               void *ws, cudaStream_t stream) {
    const DeviceInfo *info = nullptr;
    w4v_status st = device_info(&info);
    if (st != W4V_OK) return st;
    const int nblk = (M + 15) / 16;
    Args a;
    a.wq = static_cast<const uint8_t *>(Bq);
    a.scales = reinterpret_cast<const __half *>(scales);
    a.zeros = zeros;
    a.C = reinterpret_cast<__half *>(C);
    a.M = M;
    a.N = N;
    a.K = K;
    a.n_tiles = (N + kTileN - 1) / kTileN;
    a.n_groups = K / kGroup;
    a.U = (long long)a.n_tiles * a.n_groups;
    a.P = static_cast<int>(std::min<long long>(std::min(info->sm_count, kMaxCtas), a.U));
    a.partial = static_cast<float *>(ws);
    a.tile_cnt = reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(ws) +
                                              size_t(kMaxCtas) * 2 * 16 * nblk * kTileN * sizeof(float));
    a.status = info->status;
    CUtensorMap xmap;
    st = encode_tmap_2d(&xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, A, uint64_t(K), uint64_t(M),
                        uint64_t(K) * 2, 64, 16 * nblk, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != W4V_OK) return st;
    if (nblk == 1) return launch<1>(info, xmap, a, stream);
    return launch<2>(info, xmap, a, stream);
}

}  // namespace w4v
