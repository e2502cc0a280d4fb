// w4a16_gemm.cu -- W4A16 projection GEMM for verify-sized M (<= 32 rows).
//
// What it computes ("Efficient LLM Challenge Results", sections 3 and 5: a
// 4-bit W4A16 GPTQ target with group size 128 and fp16 activations):
//     C[m][n] = sum_g s[g][n] * sum_{k in g} A[m][k] * (q[n][k] - z[g][n])
// with fp32 accumulation per group and fp32 scaling, C rounded to fp16.
//
// Why it looks like this (section 2 of the same page: decode reads the whole
// weight set from HBM per step, so the K+1 verify rows must share one weight
// read; at M = 16 the kernel must move ~45 int4 weights per SM cycle):
//   * The weights are the wide operand: a 128-row weight tile is the MMA's
//     M side, the (<= 32) activation rows its N side in blocks of 16, so
//     every output element comes from the same instruction shape whatever M
//     is (batch invariance for M <= 32).
//   * Units are (128-row tile, 128-k group).  An SM completes about one TMA
//     or bulk copy per ~650 cycles whatever its size, so copies are large:
//     a stage is up to 4 consecutive groups of one tile, fetched as one 32 KB
//     bulk copy of packed int4 (the library's tile layout, evict-first) and
//     one 3-D TMA of the 4 groups' activation slices (128-byte swizzle),
//     both issued by one producer thread.
//   * Eight dequant warps (one per TMEM lane quarter and k half) turn
//     nibbles into exact fp16 (q - z) with LOP3 + HFMA2 and store them into
//     tensor memory with 32-column tcgen05.st; two register sets alternate so
//     the store of one unit overlaps the dequant of the next.  The
//     dequantized operand never touches shared memory.
//   * tcgen05.mma (A from TMEM, B = activations from shared memory, D in
//     TMEM) is issued by three threads in three warps, unit u by issuer
//     u % 3: one thread alone issues at most one MMA per ~55 cycles.  A unit
//     accumulates its 8 k-steps into its own accumulator set, so every
//     output element is the same chain of MMAs whatever the timing or M.
//   * Four drain warps read each unit's accumulators (16-column tcgen05.ld)
//     and apply the group scale in fp32, with the scales prefetched from
//     global memory four units ahead.
//   * Work is the flat list of units split evenly over one CTA per SM; a
//     tile shared by several CTAs is finished by the last one to arrive
//     (release/acquire counter, no waiting between CTAs), which sums the fp32
//     partial tiles in CTA order, so the result is deterministic.
#include "runtime.h"
#include "sm103_ptx.cuh"

namespace w4v {
namespace {

constexpr int kTileN = 128;                       // weight rows per tile (MMA M)
constexpr int kGroup = 128;                       // k per unit = one quant group
constexpr int kBlockBytes = kTileN * kGroup / 2;  // packed bytes per unit
constexpr int kIssuers = 3;
constexpr int kDqWarps = 8;
constexpr int kDrWarps = 4;
constexpr int kWarpProd = 0;                      // producer
constexpr int kWarpIss0 = 1;                      // 1..3 MMA issuers (1 also owns TMEM)
constexpr int kWarpDr0 = 4;                       // 4..7 drain
constexpr int kWarpDq0 = 8;                       // 8..15 dequant
constexpr int kWarps = kWarpDq0 + kDqWarps;
constexpr int kThreads = 32 * kWarps;
constexpr int kASlots = 4;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAcol0 = 0;
constexpr uint32_t kDcol0 = kASlots * 64;
constexpr int kScaleAhead = 4;                    // drain-side scale prefetch distance
constexpr int kStageGroups = 4;                   // groups fetched per stage

template <int NBLK>
struct Layout {
    static constexpr int kRows = 16 * NBLK;             // activation rows per box
    static constexpr int kActBox = kRows * 128;         // one 64-k block, swizzled
    static constexpr int kAct = 2 * kStageGroups * kActBox;
    static constexpr int kW = kAct;
    static constexpr int kStage = kW + kStageGroups * kBlockBytes;
    static constexpr int kStages = (192 * 1024) / kStage;
    static constexpr int kDSets = 8;                    // ring of per-unit accumulator sets
    static constexpr uint32_t kDSet = 16 * NBLK;        // columns per set
    static constexpr int kBar = kStages * kStage;
    // full, empty per stage; afull, aempty per A slot; dfull, dempty per set; done; drain sync
    static constexpr int kNumBars = 2 * kStages + 2 * kASlots + 2 * kDSets + 2;
    static constexpr int kMisc = kBar + 8 * kNumBars;
    static constexpr int kBytes = kMisc + 64 + 1024;     // + alignment slack
    static_assert(kStage % 1024 == 0, "stage alignment");
    static_assert(kDcol0 + kDSets * kDSet <= kTmemCols, "tensor memory plan");
    static_assert(kBytes <= 227 * 1024, "shared memory plan");
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

// Stages: runs of at most kStageGroups consecutive groups of one tile.
struct StageWalk {
    int t, g, G, left;
    __device__ StageWalk(long long u, int n_groups, int units)
        : t(static_cast<int>(u / n_groups)), g(static_cast<int>(u % n_groups)), G(n_groups), left(units) {}
    __device__ int size() const { return min(min(kStageGroups, G - g), left); }
    __device__ void next(int ng) {
        g += ng;
        left -= ng;
        if (g == G) {
            g = 0;
            ++t;
        }
    }
};

// Walks (tile, group) in unit order without dividing per unit.
struct UnitWalk {
    int t, g, G;
    __device__ UnitWalk(long long u, int n_groups)
        : t(static_cast<int>(u / n_groups)), g(static_cast<int>(u % n_groups)), G(n_groups) {}
    __device__ void next() {
        if (++g == G) {
            g = 0;
            ++t;
        }
    }
};

template <int NBLK>
__global__ void __launch_bounds__(kThreads, 1)
w4a16_decode_kernel(const __grid_constant__ CUtensorMap xmap, const Args p) {
    using L = Layout<NBLK>;
    constexpr int S = L::kStages;
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
    auto dempty = [&](int b) { return bar0 + 8u * (2 * S + 2 * kASlots + L::kDSets + b); };
    const uint32_t done_bar = bar0 + 8u * (2 * S + 2 * kASlots + 2 * L::kDSets);
    const uint32_t drain_bar = done_bar + 8u;
    // [0] tmem base, [1] abort flag, [2..3] pending tile + 1 per slot, [4..5] last-arriver flags
    uint32_t *misc = reinterpret_cast<uint32_t *>(base + L::kMisc);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int cta = blockIdx.x;
    const long long ub = split_begin(cta, p.U, p.P);
    const long long ue = split_begin(cta + 1, p.U, p.P);
    const int nunits = static_cast<int>(ue - ub);
    AbortState ab{reinterpret_cast<volatile uint32_t *>(&misc[1]), p.status};

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), kDqWarps + kIssuers);
        }
        for (int a = 0; a < kASlots; ++a) {
            mbar_init(afull(a), kDqWarps);
            mbar_init(aempty(a), 1);
        }
        for (int b = 0; b < L::kDSets; ++b) {
            mbar_init(dfull(b), 1);
            mbar_init(dempty(b), kDrWarps);
        }
        mbar_init(done_bar, kIssuers);
        mbar_init(drain_bar, kDrWarps);
        for (int k = 1; k < 16; ++k) misc[k] = 0;
        fence_barrier_init();
    }
    if (warp == kWarpIss0) {
        tmem_alloc(smem_u32(&misc[0]), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];

    if (warp == kWarpProd) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            prefetch_tensormap(&xmap);
            const uint64_t pol_w = l2_policy_evict_first();
            const uint64_t pol_x = l2_policy_evict_last();
            StageWalk sw(ub, p.n_groups, nunits);
            int issued = 0;
            for (int st = 0; sw.left > 0; ++st) {
                const int ng = sw.size();
                const int s = st % S;
                if (st >= S && !mbar_wait(empty(s), ((st / S) - 1) & 1, ab)) break;
                const uint32_t sa = base_s + s * L::kStage;
                mbar_arrive_expect_tx(full(s), ng * kBlockBytes + L::kAct);
                bulk_load(sa + L::kW, p.wq + (size_t(sw.t) * p.n_groups + sw.g) * kBlockBytes, ng * kBlockBytes,
                          full(s), pol_w);
                tma_load_3d(sa, &xmap, 0, 0, 2 * sw.g, full(s), pol_x);
                ++issued;
                sw.next(ng);
            }
            if (*ab.flag) {
                // Let every copy still in flight land before the CTA exits.
                for (int i = max(0, issued - S); i < issued; ++i)
                    mbar_wait_bounded(full(i % S), (i / S) & 1);
            }
        }
    } else if (warp >= kWarpIss0 && warp < kWarpIss0 + kIssuers) {
        // ------------------------------------------------------ MMA issuers
        if (lane == 0) {
            const int me = warp - kWarpIss0;
            constexpr uint32_t idesc = idesc_f16_f32(128, 16);
            StageWalk sw(ub, p.n_groups, nunits);
            bool ok = true;
            int i = 0;                          // first unit of the stage
            for (int st = 0; sw.left > 0 && ok; ++st) {
                const int ng = sw.size();
                const int s = st % S;
                // Every issuer waits for every stage, so its once-per-stage
                // release below always lands in the phase of this stage.
                if (!mbar_wait(full(s), (st / S) & 1, ab)) break;
                for (int jj = 0; jj < ng; ++jj) {
                    const int u = i + jj;
                    if (u % kIssuers != me) continue;
                    const int slot = u % kASlots;
                    const int set = u % L::kDSets;
                    if (!mbar_wait(afull(slot), (u / kASlots) & 1, ab) ||
                        (u >= L::kDSets && !mbar_wait(dempty(set), ((u / L::kDSets) - 1) & 1, ab))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t act = base_s + s * L::kStage + 2 * jj * L::kActBox;
                    const uint32_t dset = tmem + kDcol0 + set * L::kDSet;
#pragma unroll
                    for (int j = 0; j < kGroup / 16; ++j) {
#pragma unroll
                        for (int b = 0; b < NBLK; ++b) {
                            const uint32_t baddr = act + (j >> 2) * L::kActBox + b * 2048 + (j & 3) * 32;
                            mma_f16_ts(dset + 16 * b, tmem + kAcol0 + slot * 64 + 8 * j, sdesc_sw128(baddr), idesc,
                                       j > 0 ? 1u : 0u);
                        }
                    }
                    mma_commit(aempty(slot));
                    mma_commit(dfull(set));
                }
                mma_commit(empty(s));
                i += ng;
                sw.next(ng);
            }
            // Every MMA of this issuer has finished once this arrives.
            mma_commit(done_bar);
            mbar_wait_bounded(done_bar, 0);
        }
    } else if (warp >= kWarpDq0) {
        // --------------------------------------------------------- dequant
        const int dq = warp - kWarpDq0;
        const int q = warp & 3;                 // TMEM lane quarter
        const int kh = dq >> 2;                 // k half: chunks 2kh, 2kh+1 of the packed row
        const int r = 32 * q + lane;            // row inside the tile
        const uint32_t lane_base = uint32_t(32 * q) << 16;
        const __half2 sixteenth = __float2half2_rn(0.0625f);
        StageWalk sw(ub, p.n_groups, nunits);
        int d_st = 0, d_jj = 0, d_ng = sw.size();

        // Loads the next unit's 64 codes of this row and k half (units are
        // taken in order), releases its stage after the stage's last unit and
        // dequantizes into 32 half2 registers.
        auto load_dequant = [&](uint32_t (&regs)[32]) -> bool {
            const int s = d_st % S;
            if (d_jj == 0 && !warp_wait(full(s), (d_st / S) & 1, ab)) return false;
            const uint8_t *st = base + s * L::kStage + L::kW + d_jj * kBlockBytes;
            const uint4 va = *reinterpret_cast<const uint4 *>(st + ((2 * kh) * 128 + r) * 16);
            const uint4 vb = *reinterpret_cast<const uint4 *>(st + ((2 * kh + 1) * 128 + r) * 16);
            uint32_t z = 8;
            const int n = sw.t * kTileN + r;
            if (p.zeros != nullptr && n < p.N) z = __ldg(p.zeros + size_t(sw.g + d_jj) * p.N + n);
            if (++d_jj == d_ng) {
                __syncwarp();
                if (lane == 0) mbar_arrive(empty(s));
                sw.next(d_ng);
                ++d_st;
                d_jj = 0;
                d_ng = sw.size();
            }
            const __half2 zlo = u32_as_h2((0x6400u + z) * 0x10001u);          // 1024 + z
            const __half2 zhi = __float2half2_rn(-(64.f + float(z)));
            const uint32_t words[8] = {va.x, va.y, va.z, va.w, vb.x, vb.y, vb.z, vb.w};
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
            return true;
        };

        // Store unit i's registers into its A slot, dequantize the next unit
        // into the other register set while the store runs, then publish.
        auto store = [&](int i, const uint32_t (&regs)[32]) -> bool {
            const int slot = i % kASlots;
            if (i >= kASlots && !warp_wait(aempty(slot), ((i / kASlots) - 1) & 1, ab)) return false;
            tc_fence_after();
            tmem_st_32x32b_x32(tmem + lane_base + kAcol0 + slot * 64 + 32 * kh, regs);
            return true;
        };
        auto publish = [&](int i, const uint32_t (&regs)[32]) {
            tc_wait_st();
            tc_keep_alive<32>(regs);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(afull(i % kASlots));
        };
        uint32_t ra[32], rb[32];
        bool ok = nunits > 0 && load_dequant(ra);
        for (int i = 0; i < nunits && ok; i += 2) {
            if (!store(i, ra)) break;
            if (i + 1 < nunits) ok = load_dequant(rb);
            publish(i, ra);
            if (!ok || i + 1 >= nunits) break;
            if (!store(i + 1, rb)) break;
            if (i + 2 < nunits) ok = load_dequant(ra);
            publish(i + 1, rb);
        }
    } else if (warp >= kWarpDr0 && warp < kWarpDr0 + kDrWarps) {
        // ----------------------------------------------------------- drain
        const int dr = warp - kWarpDr0;
        const int q = warp & 3;
        const int r = 32 * q + lane;
        const uint32_t lane_base = uint32_t(32 * q) << 16;
        float acc[NBLK][16];
#pragma unroll
        for (int b = 0; b < NBLK; ++b)
#pragma unroll
            for (int j = 0; j < 16; ++j) acc[b][j] = 0.f;
        uint32_t pend_prev[2] = {0u, 0u};
        uint32_t drain_syncs = 0;
        auto drain_sync = [&]() -> bool {
            __syncwarp();
            if (lane == 0) mbar_arrive(drain_bar);
            return warp_wait(drain_bar, (drain_syncs++) & 1, ab);
        };

        // Group scales, prefetched kScaleAhead units ahead.
        UnitWalk ws(ub, p.n_groups);
        float sp[kScaleAhead];
        auto load_scale = [&](int i) -> float {
            float v = 0.f;
            if (i < nunits) {
                const int n = ws.t * kTileN + r;
                if (n < p.N) v = __half2float(__ldg(p.scales + size_t(ws.g) * p.N + n));
                ws.next();
            }
            return v;
        };
#pragma unroll
        for (int k = 0; k < kScaleAhead; ++k) sp[k] = load_scale(k);

        // Tile finished by this CTA alone: write C.  Otherwise publish the fp32
        // partial tile and count this CTA in; whether it arrived last is read
        // back after the CTA's last group (see fixup).
        auto flush = [&](int t) -> bool {
            const long long t0u = (long long)t * p.n_groups;
            const long long t1u = t0u + p.n_groups;
            const int n = t * kTileN + r;
            if (ub <= t0u && t1u <= ue) {
                if (n < p.N) {
#pragma unroll
                    for (int b = 0; b < NBLK; ++b)
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const int m = 16 * b + j;
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
                for (int j = 0; j < 16; ++j) {
                    const int m = 16 * b + j;
                    if (m < p.M) __stcg(part + m * kTileN + r, acc[b][j]);
                }
            if (!drain_sync()) return false;
            if (dr == 0 && lane == 0) {
                misc[2 + slot] = uint32_t(t) + 1u;
                pend_prev[slot] = atom_add_release_gpu(&p.tile_cnt[t], 1u);
            }
            return true;
        };

        // After the CTA's last group: for each published partial tile, if this
        // CTA arrived last, sum every contributor's partial in CTA order.
        auto fixup = [&]() -> bool {
            if (dr == 0 && lane == 0) {
                for (int sl = 0; sl < 2; ++sl) {
                    const uint32_t tp = misc[2 + sl];
                    uint32_t last = 0u;
                    if (tp != 0u) {
                        const long long t0u = (long long)(tp - 1u) * p.n_groups;
                        const int cf = split_owner(t0u, p.U, p.P);
                        const int cl = split_owner(t0u + p.n_groups - 1, p.U, p.P);
                        last = pend_prev[sl] == uint32_t(cl - cf) ? 1u : 0u;
                        if (last) {
                            fence_acq_rel_gpu();
                            p.tile_cnt[tp - 1u] = 0u;
                        }
                    }
                    misc[4 + sl] = last;
                }
            }
            if (!drain_sync()) return false;
            constexpr int kPart = 16 * NBLK * kTileN;
            for (int sl = 0; sl < 2; ++sl) {
                if (!misc[4 + sl]) continue;
                const int t = int(misc[2 + sl]) - 1;
                const long long t0u = (long long)t * p.n_groups;
                const int cf = split_owner(t0u, p.U, p.P);
                const int cl = split_owner(t0u + p.n_groups - 1, p.U, p.P);
                const int n = t * kTileN + r;
                float sum[NBLK][16];
#pragma unroll
                for (int b = 0; b < NBLK; ++b)
#pragma unroll
                    for (int j = 0; j < 16; ++j) sum[b][j] = 0.f;
                constexpr int kBatch = NBLK == 1 ? 4 : 2;     // independent loads in flight
                for (int c0 = cf; c0 <= cl; c0 += kBatch) {
                    float v[kBatch][NBLK][16];
#pragma unroll
                    for (int u = 0; u < kBatch; ++u) {
                        const int cc = c0 + u;
                        const int sl2 = (cc <= cl && split_begin(cc, p.U, p.P) >= t0u) ? 0 : 1;
                        const float *src = p.partial + (size_t(cc <= cl ? cc : cl) * 2 + sl2) * kPart;
#pragma unroll
                        for (int b = 0; b < NBLK; ++b)
#pragma unroll
                            for (int j = 0; j < 16; ++j) {
                                const int m = 16 * b + j;
                                v[u][b][j] = (cc <= cl && m < p.M) ? __ldcg(src + m * kTileN + r) : 0.f;
                            }
                    }
#pragma unroll
                    for (int u = 0; u < kBatch; ++u)
                        if (c0 + u <= cl) {
#pragma unroll
                            for (int b = 0; b < NBLK; ++b)
#pragma unroll
                                for (int j = 0; j < 16; ++j) sum[b][j] += v[u][b][j];
                        }
                }
                if (n < p.N) {
#pragma unroll
                    for (int b = 0; b < NBLK; ++b)
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const int m = 16 * b + j;
                            if (m < p.M) p.C[size_t(m) * p.N + n] = __float2half_rn(sum[b][j]);
                        }
                }
            }
            return true;
        };

        UnitWalk wd(ub, p.n_groups);
        bool ok = true;
        for (int i = 0; i < nunits && ok; ++i) {
            const int set = i % L::kDSets;
            if (!warp_wait(dfull(set), (i / L::kDSets) & 1, ab)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const float sc = sp[0];
#pragma unroll
            for (int k = 0; k + 1 < kScaleAhead; ++k) sp[k] = sp[k + 1];
            sp[kScaleAhead - 1] = load_scale(i + kScaleAhead);
            const uint32_t dset = tmem + lane_base + kDcol0 + set * L::kDSet;
            uint32_t d[NBLK][16];
#pragma unroll
            for (int b = 0; b < NBLK; ++b) tmem_ld_32x32b_x16(dset + 16 * b, d[b]);
#pragma unroll
            for (int b = 0; b < NBLK; ++b) tc_wait_ld_keep<16>(d[b]);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(dempty(set));
#pragma unroll
            for (int b = 0; b < NBLK; ++b)
#pragma unroll
                for (int j = 0; j < 16; ++j) acc[b][j] = fmaf(sc, __uint_as_float(d[b][j]), acc[b][j]);
            const int t = wd.t;
            const bool tile_end = wd.g == p.n_groups - 1;
            wd.next();
            if (tile_end || i == nunits - 1) {
                if (!flush(t)) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int b = 0; b < NBLK; ++b)
#pragma unroll
                    for (int j = 0; j < 16; ++j) acc[b][j] = 0.f;
            }
        }
        if (ok) fixup();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWarpIss0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int NBLK>
w4v_status launch(const CUtensorMap &xmap, const Args &a, cudaStream_t stream) {
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
    st = encode_tmap_kblocks(&xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, A, uint64_t(K), uint64_t(M), 64, 16 * nblk,
                             2 * kStageGroups, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != W4V_OK) return st;
    if (nblk == 1) return launch<1>(xmap, a, stream);
    return launch<2>(xmap, a, stream);
}

}  // namespace w4v
