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
//     whole tiles; units are (tile, 128-k chunk).
//   * An SM completes about one TMA copy per ~650 cycles whatever its size,
//     so a stage is two k-chunks of a tile: one 3-D TMA of 32 KB of int8
//     weights (128-byte swizzle, straight from the row-major [V][K] matrix)
//     and one 3-D TMA of the matching activation slices, both issued by one
//     producer thread.  A unit is one stage: 128 rows x 256 k.  Every
//     hand-off between roles costs a few hundred cycles of latency whatever
//     it carries, so units are as large as tensor memory allows (A slots of
//     128 columns).
//   * Eight dequant warps widen int8 to exact fp16 (XOR 0x80, PRMT into the
//     mantissa of 1024, subtract 1152) and store it into tensor memory with
//     32-column stores.  Warp (quarter, parity) owns its 32 rows of every
//     other unit and does the unit's whole k in four 64-k steps, alternating
//     two register sets so each store overlaps the next step's arithmetic;
//     the two warps sharing a scheduler work on different units.
//   * Three issuer threads (one MMA per ~55 cycles each) run tcgen05.mma with
//     A from TMEM, accumulating the whole K of a tile in TMEM; the k-steps go
//     round-robin into independent accumulators, each (accumulator, column
//     block) slice owned by one issuer, so the order of every sum is fixed.
//   * Four drain warps finish a tile: add the accumulators in a fixed order,
//     scale, turn each logit into an order-preserving 32-bit key, and a warp
//     max-reduction plus a min-reduction over the winning lanes gives the
//     lowest-index maximum; a shared-memory 64-bit atomicMax of (key, ~index)
//     keeps the CTA's best per row.
//   * Each CTA folds its best keys into one global 64-bit atomicMax per row;
//     the last CTA to arrive (acquire-release counter, no waiting) reads and
//     clears them and writes the token ids.  When the rows are verify blocks
//     with drafts attached, that CTA also runs the greedy acceptance on the
//     tokens it just wrote (one warp per block, from shared memory), so the
//     verify step's last two operations are one launch.
//   * Launched with programmatic stream serialization: set-up and an L2
//     prefetch of the first weight stages overlap the previous kernel's end.
#include "runtime.h"
#include "sm103_ptx.cuh"

namespace w4v {
namespace {

constexpr int kTileV = 128;
constexpr int kChunk = 128;                 // k per unit (bytes of int8)
constexpr int kWBytes = kTileV * kChunk;    // 16 KB per unit
constexpr int kMaxRows = 128;
constexpr int kIssuers = 3;
constexpr int kDqWarps = 8;
constexpr int kDrWarps = 4;
constexpr int kWarpProd = 0;
constexpr int kWarpIss0 = 1;                // 1..3 (1 also owns TMEM)
constexpr int kWarpDr0 = 4;                 // 4..7
constexpr int kWarpDq0 = 8;                 // 8..15
constexpr int kWarps = kWarpDq0 + kDqWarps;
constexpr int kThreads = 32 * kWarps;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAcol0 = 0;
// k-chunks per stage = per unit: two up to 32 rows; one beyond, where each
// chunk's activations (64 rows or more x 128 k) are as large as its weights,
// so that four shorter stages fit instead of two long ones (a stage is
// held until its MMAs complete, and with two the ring stalled on reloads).
__host__ __device__ constexpr int stage_chunks(int nblk) { return nblk >= 4 ? 1 : 2; }

template <int NBLK>
struct Layout {
    static constexpr int kStageChunks = stage_chunks(NBLK);
    static constexpr uint32_t kASlotCols = kStageChunks * 64;
    static constexpr int kRows = 16 * NBLK;
    static constexpr int kActBox = kRows * 128;         // one 64-k block, swizzled
    static constexpr int kAct = 2 * kStageChunks * kActBox;
    static constexpr int kW = kAct;                     // 1024-aligned
    static constexpr int kStage = kW + kStageChunks * kWBytes;
    static constexpr int kStages = (196 * 1024) / kStage > 6 ? 6 : (196 * 1024) / kStage;
    // Independent accumulators per tile: the same count for every M <= 32,
    // so the per-logit arithmetic does not depend on M there.
    // (M = 128 keeps one accumulator and two D sets: two accumulators in a
    // single set ran 19% slower, the tile's drain then stalling the MMAs.)
    static constexpr int kAcc = NBLK <= 2 ? 3 : 8 / NBLK;
    static constexpr int kDSets = 2;
    // M <= 16: one M128 N16 MMA per k-step.  M > 16: one MMA of N = 16 NBLK
    // per k-step (an MMA costs about the same to issue up to N = 128), D laid
    // out [acc][block][16].
    static constexpr bool kWide = NBLK >= 2;
    static constexpr uint32_t kDSet = kAcc * 16 * NBLK;
    // A slots: as many units as fit beside two accumulator sets
    static constexpr int kASlots = (kTmemCols - kDSets * kDSet) / kASlotCols > 4
                                       ? 4 : int((kTmemCols - kDSets * kDSet) / kASlotCols);
    static constexpr uint32_t kDcol0 = kASlots * kASlotCols;
    static constexpr int kBar = kStages * kStage;
    static constexpr int kNumBars = 2 * kStages + 2 * kASlots + 4 + 2;
    static constexpr int kBest = ((kBar + 8 * kNumBars + 7) / 8) * 8;   // u64 [128]
    static constexpr int kMisc = kBest + 8 * kMaxRows;
    static constexpr int kBytes = kMisc + 64 + 1024;
    static_assert(kStage % 1024 == 0, "stage alignment");
    static_assert(kDcol0 + kDSets * kDSet <= kTmemCols, "tensor memory plan");
    static_assert(kBytes <= 227 * 1024, "shared memory plan");
};

// Stages: runs of at most SC consecutive k-chunks of one tile.
template <int SC>
struct ChunkWalk {
    int j, c, nch, ntiles;
    __device__ ChunkWalk(int n_chunks, int tiles) : j(0), c(0), nch(n_chunks), ntiles(tiles) {}
    __device__ bool more() const { return j < ntiles; }
    __device__ int size() const { return min(SC, nch - c); }
    __device__ void next(int ng) {
        c += ng;
        if (c == nch) {
            c = 0;
            ++j;
        }
    }
};

struct Args {
    const int8_t *W;
    const __half *scale;
    int32_t *argmax_out;
    float *maxlogit;
    float *logits;
    unsigned long long *keys;   // [128], zero between calls
    uint32_t *counter;
    uint32_t *status;
    const int32_t *draft;       // acceptance epilogue (B > 0): drafts [B][n_draft]
    int32_t *n_accepted;
    int32_t *out_tokens;
    int B, n_draft;
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
    constexpr int S = L::kStages;
    constexpr int kASlots = L::kASlots;
    constexpr uint32_t kDcol0 = L::kDcol0;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    uint8_t *base = smem_raw + (base_s - raw_s);

    const uint32_t bar0 = base_s + L::kBar;
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (S + s); };
    auto afull = [&](int a) { return bar0 + 8u * (2 * S + a); };
    auto aempty = [&](int a) { return bar0 + 8u * (2 * S + kASlots + a); };
    auto dfull = [&](int b) { return bar0 + 8u * (2 * S + 2 * kASlots + b); };
    auto dempty = [&](int b) { return bar0 + 8u * (2 * S + 2 * kASlots + 2 + b); };
    const uint32_t done_bar = bar0 + 8u * (2 * S + 2 * kASlots + 4);
    const uint32_t drain_bar = done_bar + 8u;
    unsigned long long *best = reinterpret_cast<unsigned long long *>(base + L::kBest);
    uint32_t *misc = reinterpret_cast<uint32_t *>(base + L::kMisc);   // [0] tmem, [1] abort, [2] last

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int cta = blockIdx.x;
    const int tb = static_cast<int>(split_begin(cta, p.n_tiles, p.P));
    const int te = static_cast<int>(split_begin(cta + 1, p.n_tiles, p.P));
    const int ntiles = te - tb;
    AbortState ab{reinterpret_cast<volatile uint32_t *>(&misc[1]), p.status};

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), kDqWarps / 2 + kIssuers);   // the unit's four dequant warps + issuers
        }
        for (int a = 0; a < kASlots; ++a) {
            mbar_init(afull(a), kDqWarps / 2);
            mbar_init(aempty(a), kIssuers);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(dfull(b), kIssuers);
            mbar_init(dempty(b), kDrWarps);
        }
        mbar_init(done_bar, kIssuers);
        mbar_init(drain_bar, kDrWarps);
        misc[1] = 0;
        misc[2] = 0;
        fence_barrier_init();
    }
    if (threadIdx.x < kMaxRows) best[threadIdx.x] = 0ull;
    if (warp == kWarpIss0) {
        tmem_alloc(smem_u32(&misc[0]), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    grid_dep_launch();

    if (warp == kWarpProd) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            prefetch_tensormap(&wmap);
            prefetch_tensormap(&xmap);
            // Only L2 is warmed before the dependency wait (L2 is the point
            // of coherence, so this is safe whatever the previous kernel writes).
            ChunkWalk<L::kStageChunks> pw(p.n_chunks, ntiles);
            for (int st = 0; st < S && pw.more(); ++st) {
                prefetch_l2_3d(&wmap, 0, (tb + pw.j) * kTileV, pw.c);
                pw.next(pw.size());
            }
        }
        grid_dep_wait();
        if (lane == 0) {
            const uint64_t pol_w = l2_policy_evict_first();
            const uint64_t pol_x = l2_policy_evict_last();
            int issued = 0;
            ChunkWalk<L::kStageChunks> cw(p.n_chunks, ntiles);
            for (int st = 0; cw.more(); ++st) {
                const int ng = cw.size();
                const int s = st % S;
                if (st >= S && !mbar_wait(empty(s), ((st / S) - 1) & 1, ab)) break;
                const uint32_t sa = base_s + s * L::kStage;
                mbar_arrive_expect_tx(full(s), L::kStageChunks * kWBytes + L::kAct);
                tma_load_3d(sa + L::kW, &wmap, 0, (tb + cw.j) * kTileV, cw.c, full(s), pol_w);
                tma_load_3d(sa, &xmap, 0, 0, 2 * cw.c, full(s), pol_x);
                ++issued;
                cw.next(ng);
            }
            if (*ab.flag) {
                for (int i = max(0, issued - S); i < issued; ++i)
                    mbar_wait_bounded(full(i % S), (i / S) & 1);
            }
        }
    } else if (warp >= kWarpIss0 && warp < kWarpIss0 + kIssuers) {
        // ------------------------------------------------------ MMA issuers
        // The whole warp runs the loop and lane 0 alone issues, so the
        // operands stay warp-uniform.
        grid_dep_wait();
        {
            const int me = warp - kWarpIss0;
            constexpr uint32_t idesc = idesc_f16_f32(128, 16);
            constexpr uint32_t idesc_wide = idesc_f16_f32(128, 16 * NBLK);
            ChunkWalk<L::kStageChunks> cw(p.n_chunks, ntiles);
            bool ok = true;
            for (int st = 0; cw.more() && ok; ++st) {      // unit st = stage st
                const int ng = cw.size();
                const int s = st % S;
                const int j = cw.j;
                const int slot = st % kASlots;
                const int buf = j % L::kDSets, use = j / L::kDSets;   // D set and its use count
                if (!warp_wait(full(s), (st / S) & 1, ab) || !warp_wait(afull(slot), (st / kASlots) & 1, ab) ||
                    (cw.c == 0 && use >= 1 && !warp_wait(dempty(buf), (use - 1) & 1, ab))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t dset = tmem + kDcol0 + buf * L::kDSet;
                for (int jj = 0; jj < ng; ++jj) {
                    const int c = cw.c + jj;
                    const uint32_t act = base_s + s * L::kStage + 2 * jj * L::kActBox;
#pragma unroll
                    for (int kk = 0; kk < kChunk / 16; ++kk) {
                        const int a = kk % L::kAcc;
                        if constexpr (L::kWide) {
                            // accumulator a belongs to issuer a: all NBLK blocks in one MMA
                            if (a % kIssuers != me) continue;
                            const uint32_t baddr = act + (kk >> 2) * L::kActBox + (kk & 3) * 32;
                            mma_f16_ts_lane0(dset + a * (16 * NBLK), tmem + kAcol0 + slot * L::kASlotCols + jj * 64 + 8 * kk,
                                       sdesc_sw128(baddr), idesc_wide, (c > 0 || kk >= L::kAcc) ? 1u : 0u);
                        } else {
#pragma unroll
                            for (int b = 0; b < NBLK; ++b) {
                                if ((a * NBLK + b) % kIssuers != me) continue;
                                const uint32_t baddr = act + (kk >> 2) * L::kActBox + b * 2048 + (kk & 3) * 32;
                                mma_f16_ts_lane0(dset + (b * L::kAcc + a) * 16,
                                           tmem + kAcol0 + slot * L::kASlotCols + jj * 64 + 8 * kk, sdesc_sw128(baddr),
                                           idesc, (c > 0 || kk >= L::kAcc) ? 1u : 0u);
                            }
                        }
                    }
                }
                mma_commit_lane0(aempty(slot));
                if (cw.c + ng == p.n_chunks) mma_commit_lane0(dfull(buf));
                mma_commit_lane0(empty(s));
                cw.next(ng);
            }
            mma_commit_lane0(done_bar);
            mbar_wait_bounded(done_bar, 0);
            __syncwarp();
        }
    } else if (warp >= kWarpDq0) {
        grid_dep_wait();
        // --------------------------------------------------------- dequant
        const int dq = warp - kWarpDq0;
        const int q = warp & 3;
        const int par = dq >> 2;                // units (stages) st with st % 2 == par
        const int r = 32 * q + lane;
        const uint32_t lane_base = uint32_t(32 * q) << 16;
        const __half2 bias = u32_as_h2(0x64806480u);    // 1152 = 1024 + 128 in both halves

        // 64 bytes (half kh of chunk row r) of the chunk at shared address `ch`, widened to
        // 32 half2 registers.
        auto dequant = [&](uint32_t ch, int kh, uint32_t (&regs)[32]) {
            uint4 w[4];
#pragma unroll
            for (int ci = 0; ci < 4; ++ci) {
                const int chunk = 4 * kh + ci;
                const int phys = chunk ^ (r & 7);            // 128-byte swizzle of the TMA box
                w[ci] = lds128(ch + r * 128 + phys * 16);
            }
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
        };
        auto release = [&](int s) {
            __syncwarp();
            if (lane == 0) mbar_arrive(empty(s));
        };

        ChunkWalk<L::kStageChunks> cw(p.n_chunks, ntiles);
        uint32_t ra[32], rb[32];
        for (int st = 0; cw.more(); ++st) {
            const int ng = cw.size();
            cw.next(ng);
            if ((st & 1) != par) continue;
            const int s = st % S;
            const int slot = st % kASlots;
            if (!warp_wait(full(s), (st / S) & 1, ab)) break;
            const uint32_t c0p = base_s + s * L::kStage + L::kW;
            const uint32_t c1p = c0p + kWBytes;
            const uint32_t col = tmem + lane_base + kAcol0 + slot * L::kASlotCols;
            dequant(c0p, 0, ra);
            if (st >= kASlots && !warp_wait(aempty(slot), ((st / kASlots) - 1) & 1, ab)) {
                release(s);
                break;
            }
            tc_fence_after();
            tmem_st_32x32b_x32(col + 0, ra);
            dequant(c0p, 1, rb);
            if (ng == 1) release(s);             // last shared-memory read of the stage
            tc_wait_st();
            tc_keep_alive<32>(ra);
            tmem_st_32x32b_x32(col + 32, rb);
            if (ng > 1) {
                dequant(c1p, 0, ra);
                tc_wait_st();
                tc_keep_alive<32>(rb);
                tmem_st_32x32b_x32(col + 64, ra);
                dequant(c1p, 1, rb);
                release(s);
                tc_wait_st();
                tc_keep_alive<32>(ra);
                tmem_st_32x32b_x32(col + 96, rb);
            }
            tc_wait_st();
            tc_keep_alive<32>(rb);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(afull(slot));
        }
    } else if (warp >= kWarpDr0 && warp < kWarpDr0 + kDrWarps) {
        // ----------------------------------------------------------- drain
        grid_dep_wait();
        const int dr = warp - kWarpDr0;
        const int q = warp & 3;
        const int r = 32 * q + lane;
        const uint32_t lane_base = uint32_t(32 * q) << 16;
        uint32_t drain_syncs = 0;
        auto drain_sync = [&]() -> bool {
            __syncwarp();
            if (lane == 0) mbar_arrive(drain_bar);
            return warp_wait(drain_bar, (drain_syncs++) & 1, ab);
        };

        bool ok = true;
        for (int j = 0; j < ntiles && ok; ++j) {
            const int buf = j % L::kDSets, use = j / L::kDSets;
            const int t = tb + j;
            const int v = t * kTileV + r;
            const bool valid = v < p.V;
            const float sc = valid ? __half2float(__ldg(p.scale + v)) : 0.f;
            if (!warp_wait(dfull(buf), use & 1, ab)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t dset = tmem + lane_base + kDcol0 + buf * L::kDSet;
#pragma unroll 1
            for (int b = 0; b < NBLK; ++b) {
                // the block's accumulators, added in a fixed order
                float g[16];
                if constexpr (L::kAcc == 3 && NBLK == 1) {
                    uint32_t d01[32], d2[16];
                    tmem_ld_32x32b_x32(dset + (b * 3) * 16, d01);
                    tmem_ld_32x32b_x16(dset + (b * 3 + 2) * 16, d2);
                    tc_wait_ld_keep<32>(d01);
                    tc_wait_ld_keep<16>(d2);
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj)
                        g[jj] = (__uint_as_float(d01[jj]) + __uint_as_float(d01[16 + jj])) + __uint_as_float(d2[jj]);
                } else if constexpr (L::kAcc == 3) {
                    // wide layout [acc][block][16], accumulators added in order
                    uint32_t d0[16], d1[16], d2[16];
                    tmem_ld_32x32b_x16(dset + b * 16, d0);
                    tmem_ld_32x32b_x16(dset + 16 * NBLK + b * 16, d1);
                    tmem_ld_32x32b_x16(dset + 32 * NBLK + b * 16, d2);
                    tc_wait_ld_keep<16>(d0);
                    tc_wait_ld_keep<16>(d1);
                    tc_wait_ld_keep<16>(d2);
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj)
                        g[jj] = (__uint_as_float(d0[jj]) + __uint_as_float(d1[jj])) + __uint_as_float(d2[jj]);
                } else if constexpr (L::kAcc == 2) {
                    // wide layout [acc][block][16]
                    uint32_t d0[16], d1[16];
                    tmem_ld_32x32b_x16(dset + b * 16, d0);
                    tmem_ld_32x32b_x16(dset + 16 * NBLK + b * 16, d1);
                    tc_wait_ld_keep<16>(d0);
                    tc_wait_ld_keep<16>(d1);
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) g[jj] = __uint_as_float(d0[jj]) + __uint_as_float(d1[jj]);
                } else {
                    uint32_t d[16];
                    tmem_ld_32x32b_x16(dset + b * 16, d);
                    tc_wait_ld_keep<16>(d);
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) g[jj] = __uint_as_float(d[jj]);
                }
                if (b == NBLK - 1) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(dempty(buf));
                }
                // the warp's best key and lowest winning lane for each of the
                // block's 16 rows land in lane jj; lanes 0..15 then fold them
                // into the CTA's row keys with one atomic instruction
                uint32_t mykey = 0u, mylane = 0u;
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) {
                    const int m = 16 * b + jj;
                    const float x = sc * g[jj];
                    if (p.logits != nullptr && valid && m < p.M) p.logits[size_t(m) * p.V + v] = x;
                    const uint32_t key = valid ? logit_key(x) : 0u;
                    const uint32_t wmax = __reduce_max_sync(0xFFFFFFFFu, key);
                    const uint32_t wlane = __reduce_min_sync(0xFFFFFFFFu, key == wmax ? uint32_t(lane) : 32u);
                    if (lane == jj) {
                        mykey = wmax;
                        mylane = wlane;
                    }
                }
                const int mrow = 16 * b + lane;
                if (lane < 16 && mrow < p.M && mykey != 0u) {
                    const uint32_t vbest = uint32_t(t * kTileV + 32 * q) + mylane;
                    atomicMax(&best[mrow], (static_cast<unsigned long long>(mykey) << 32) | (0xFFFFFFFFull - vbest));
                }
            }
        }

        // Fold this CTA's best per row into the global keys; the last CTA to
        // arrive reads and clears them.
        const int tid = dr * 32 + lane;
        if (ok) ok = drain_sync();
        if (ok) {
            if (tid < p.M) atomicMax(p.keys + tid, best[tid]);
            ok = drain_sync();
        }
        if (ok) {
            if (tid == 0) {
                const uint32_t prev = atom_add_acq_rel_gpu(p.counter, 1u);
                const bool last = prev == uint32_t(p.P - 1);
                if (last) *p.counter = 0u;
                misc[2] = last ? 1u : 0u;
            }
            ok = drain_sync();
        }
        if (ok && misc[2]) {
            // The CTA's own best keys are folded already: their shared array
            // now holds the finished tokens for the acceptance epilogue.
            int32_t *tok_s = reinterpret_cast<int32_t *>(best);
            if (tid < p.M) {
                const unsigned long long k = atomicExch(p.keys + tid, 0ull);
                const int32_t t = static_cast<int32_t>(0xFFFFFFFFu - uint32_t(k & 0xFFFFFFFFull));
                p.argmax_out[tid] = t;
                tok_s[tid] = t;
                if (p.maxlogit != nullptr) p.maxlogit[tid] = key_logit(uint32_t(k >> 32));
            }
            // Greedy acceptance ("Efficient LLM Challenge Results", section 3):
            // rows b*(n+1) .. b*(n+1)+n are verify block b; keep the longest
            // draft prefix equal to the target's tokens, a negative draft (the
            // -1 sentinel) never matching.  One drain warp per block.
            if (p.B > 0 && drain_sync()) {
                const int nd = p.n_draft;
                for (int b = dr; b < p.B; b += kDrWarps) {
                    const int32_t *t = tok_s + b * (nd + 1);
                    const int32_t *d = p.draft + size_t(b) * nd;
                    int n = nd;
                    for (int j0 = 0; j0 < nd; j0 += 32) {
                        const int j = j0 + lane;
                        bool miss = false;
                        if (j < nd) {
                            const int32_t dj = d[j];
                            miss = !(dj >= 0 && dj == t[j]);
                        }
                        const unsigned m = __ballot_sync(0xFFFFFFFFu, miss);
                        if (m != 0u) {
                            n = j0 + __ffs(m) - 1;
                            break;
                        }
                    }
                    if (lane == 0) p.n_accepted[b] = n;
                    if (p.out_tokens != nullptr)
                        for (int j = lane; j <= nd; j += 32) p.out_tokens[size_t(b) * (nd + 1) + j] = j <= n ? t[j] : -1;
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWarpIss0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
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
    if (launch_pdl(w8_lmhead_argmax_kernel<NBLK>, dim3(a.P), dim3(kThreads), L::kBytes, stream, xmap, wmap, a) !=
        cudaSuccess) {
        cudaGetLastError();
        return W4V_ERR_CUDA;
    }
    return W4V_OK;
}

}  // namespace

size_t w8_lmhead_ws_bytes(int M, int V) {
    (void)M;
    (void)V;
    return size_t(kMaxRows) * sizeof(unsigned long long) + 256;
}

w4v_status launch_w8_lmhead_argmax(const uint16_t *X, const int8_t *W, const uint16_t *scale,
                                   int M, int K, int V, int32_t *argmax_out, float *maxlogit,
                                   float *logits, void *ws, cudaStream_t stream, const LmAccept *accept) {
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
    a.counter = reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(ws) + size_t(kMaxRows) * sizeof(unsigned long long));
    a.status = info->status;
    a.draft = accept != nullptr ? accept->draft : nullptr;
    a.n_accepted = accept != nullptr ? accept->n_accepted : nullptr;
    a.out_tokens = accept != nullptr ? accept->out_tokens : nullptr;
    a.B = accept != nullptr ? accept->B : 0;
    a.n_draft = accept != nullptr ? accept->n_draft : 0;
    a.M = M;
    a.K = K;
    a.V = V;
    a.n_tiles = (V + kTileV - 1) / kTileV;
    a.n_chunks = K / kChunk;
    a.P = std::min(std::min(info->sm_count, kMaxCtas), a.n_tiles);
    CUtensorMap xmap, wmap;
    st = encode_tmap_kblocks(&xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, X, uint64_t(K), uint64_t(M), 64, 16 * nblk,
                             2 * stage_chunks(nblk), CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != W4V_OK) return st;
    st = encode_tmap_kblocks(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, W, uint64_t(K), uint64_t(V), kChunk, kTileV,
                             stage_chunks(nblk), CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != W4V_OK) return st;
    switch (nblk) {
        case 1: return launch<1>(xmap, wmap, a, stream);
        case 2: return launch<2>(xmap, wmap, a, stream);
        case 4: return launch<4>(xmap, wmap, a, stream);
        default: return launch<8>(xmap, wmap, a, stream);
    }
}

}  // namespace w4v
