// w4a16_prefill.cu -- W4A16 projection GEMM for prefill-sized M (> 32 rows).
//
// Same operation as the verify-sized kernel ("Efficient LLM Challenge
// Results", sections 3 and 5: 4-bit W4A16 GPTQ weights, group size 128, fp16
// activations), in the regime section 2 and 4 of that page call prefill
// compute: every weight is reused by M rows, so the kernel is bound by the
// tensor cores, not by HBM.
//
//     C[m][n] = sum_k A[m][k] * w[n][k],  w[n][k] = fp16(fp16(q - z) * s[k/128][n])
//
// The dequantized weight is rounded to fp16 once (scale applied in fp16) and
// the whole K is accumulated in fp32 in tensor memory.  (The verify-sized
// kernel instead applies each group's scale in fp32 to that group's fp32 sum;
// here the per-group fold would need 128 accumulators per thread.)  With
// s in [0.005, 0.02] and |q - z| <= 15 the rounding of w is at most 2^-11
// relative, which keeps the output within the 2e-3 relative bound.
//
// Design:
//   * One CTA per SM computes 128 weight rows x 256 activation rows over the
//     whole K, tile after tile (two CTAs per SM with 128 x 128 tiles kept
//     the tensor pipe ~50% busy, this ~70%).
//   * Per 128-k group: one 8 KB bulk copy of packed int4 and one 64 KB 3-D
//     TMA of the activation slice (128-byte swizzle), three stages.
//   * Two sets of four dequant warps, taking alternate groups (set s always
//     fills A slot s), turn a group into fp16 s * (q - z) and write it into
//     tensor memory (64-column tcgen05.st).  Two issuing threads each issue
//     eight tcgen05.mma.kind::f16 per group for one 128-column half of the
//     tile: A = weights from TMEM (M = 128), B = half the activation rows
//     from shared memory (N = 128), D in TMEM.
//   * Four epilogue warps read the finished tile (32-column tcgen05.ld),
//     round to fp16 and store C.  The two accumulator halves rotate over
//     three 128-column regions of tensor memory, so a tile's epilogue
//     overlaps the next tile's MMAs (with one 256-column accumulator the
//     epilogue stalled them: ~10 % of the layer set's time).
//   * When the last wave of tiles would leave most SMs idle, the tiles of
//     that wave are cut by activation rows into 2 or 4 slices of 128 or 64
//     rows, each an output tile of its own over the whole k range (N = 128
//     or 64 MMAs, the activation box as narrow as the slice): a slice costs
//     about half a tile or less, since the weights' dequantization, not the
//     MMAs, then paces it, and nothing is added across CTAs.  (o and down at
//     2048 rows: 160 tiles for 152 SMs, the last 8 as 32 slices.)
//   * Alternatively each tile's k range is split in two halves done by two
//     CTAs at the same time: each writes its fp32 partial tile to the
//     workspace, and the second to arrive (acquire-release counter, no
//     waiting) adds half 0 and half 1 in that order and writes C, so the
//     result does not depend on timing.  The host takes whichever of whole
//     tiles, slices and halves its cost model finds shortest.
#include "runtime.h"
#include "sm103_ptx.cuh"

namespace w4v {
namespace {

constexpr int kTileN = 128;                       // weight rows per tile (MMA M)
constexpr int kTileM = 256;                       // activation rows per tile (MMA N)
constexpr int kGroup = 128;
constexpr int kBlockBytes = kTileN * kGroup / 2;  // 8 KB packed per (tile, group)
constexpr int kActBox = kTileM * 128;             // one 64-k block of activations, 32 KB
constexpr int kAct = 2 * kActBox;                 // one group, 64 KB
constexpr int kStage = kAct + kBlockBytes;        // 72 KB, 1024-aligned
constexpr int kStages = 3;
constexpr int kASlots = 2;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAcol0 = 0;
constexpr uint32_t kDcol0 = kASlots * 64;
constexpr int kWarpProd = 0;
constexpr int kWarpMma = 1;                       // also owns TMEM
constexpr int kWarpDq0 = 2;                       // 2..9: two sets of four, alternate groups
constexpr int kWarpEp0 = 10;                      // 10..13
constexpr int kWarpMma2 = 14;                     // second issuer: the upper column half of every tile
constexpr int kWarps = 15;
constexpr int kThreads = 32 * kWarps;
// Accumulators: three 128-column regions after the A slots.  Tile nt's lower
// and upper column halves go to regions (2 nt) % 3 and (2 nt + 1) % 3, so the
// next tile's lower half always finds a free region and its upper half waits
// only for the epilogue to have read this tile's lower half.
constexpr int kRegions = 3;
constexpr uint32_t kRegionCols = 128;
constexpr int kBar = kStages * kStage;
constexpr int kNumBars = 2 * kStages + 2 * kASlots + 2 * kRegions + 2;
constexpr int kPart = kTileM * kTileN;             // floats of one output tile
// Tiles are split in two k halves only for launches of at most this many
// tiles (the workspace holds both halves' fp32 partials of every tile).
constexpr int kSplitMaxTiles = 1024;
constexpr int kMisc = kBar + 8 * kNumBars;
constexpr int kBytes = kMisc + 64 + 1024;
static_assert(kStage % 1024 == 0, "stage alignment");
static_assert(kBytes <= 227 * 1024, "shared memory plan");
static_assert(kDcol0 + kRegions * kRegionCols <= kTmemCols && 2 * kRegionCols >= kTileM, "tensor memory plan");
static_assert(kASlots == 2, "dequant set s fills A slot s (groups alternate between the two)");

struct Args {
    const uint8_t *wq;
    const __half *scales;
    const uint8_t *zeros;
    __half *C;
    float *partial;          // [tiles][2][kTileM][kTileN] fp32 (halves == 2)
    uint32_t *tile_cnt;      // [tiles] arrivals, zero between calls (halves == 2)
    uint32_t *status;
    int M, N, K;
    int n_tiles_n, n_tiles_m, n_groups;
    int halves;              // 1, or 2: each tile's k range done by two CTAs
    int n_whole;             // halves == 1: items before this are whole tiles,
    int slices;              // the rest `slices` slices of each later tile
    int items;
};

// Work item i.  With halves == 2: tile i / 2, k groups of half i % 2.
// Otherwise the first n_whole items are whole tiles and each later tile is
// `slices` items of kTileM / slices activation rows, each over the whole k.
struct Item {
    int tile, half, g0, g1, col0, width;
    __device__ Item(int i, const Args &p) {
        const int G = p.n_groups;
        half = 0;
        g0 = 0;
        g1 = G;
        col0 = 0;
        width = kTileM;
        if (p.halves == 2) {
            tile = i >> 1;
            half = i & 1;
            g0 = half ? G / 2 : 0;
            g1 = half ? G : G / 2;
        } else if (i < p.n_whole) {
            tile = i;
        } else {
            const int k = i - p.n_whole;
            width = kTileM / p.slices;
            tile = p.n_whole + k / p.slices;
            col0 = (k % p.slices) * width;
        }
    }
};

// kG32: group size 32, so each 32-k chunk of a 128-k block has its own
// scale and zero point (four per block instead of one).
template <bool kG32>
__global__ void __launch_bounds__(kThreads, 1)
w4a16_prefill_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap xmap128,
                     const __grid_constant__ CUtensorMap xmap64, const Args p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    uint8_t *base = smem_raw + (base_s - raw_s);
    const uint32_t bar0 = base_s + kBar;
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (kStages + s); };
    auto afull = [&](int a) { return bar0 + 8u * (2 * kStages + a); };
    auto aempty = [&](int a) { return bar0 + 8u * (2 * kStages + kASlots + a); };
    auto rfull = [&](int R) { return bar0 + 8u * (2 * kStages + 2 * kASlots + R); };
    auto rempty = [&](int R) { return bar0 + 8u * (2 * kStages + 2 * kASlots + kRegions + R); };
    const uint32_t done_bar = bar0 + 8u * (2 * kStages + 2 * kASlots + 2 * kRegions);
    const uint32_t ep_bar = done_bar + 8u;                            // epilogue warps' sync
    uint32_t *misc = reinterpret_cast<uint32_t *>(base + kMisc);     // [0] tmem, [1] abort, [2] last

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int items = p.items;
    AbortState ab{reinterpret_cast<volatile uint32_t *>(&misc[1]), p.status};

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 4 + 2);          // the group's dequant set + both issuers' commits
        }
        for (int a = 0; a < kASlots; ++a) {
            mbar_init(afull(a), 4);              // dequant set a
            mbar_init(aempty(a), 2);
        }
        for (int R = 0; R < kRegions; ++R) {
            mbar_init(rfull(R), 1);              // the issuer of the half using it
            mbar_init(rempty(R), 4);             // epilogue warps
        }
        mbar_init(done_bar, 2);
        mbar_init(ep_bar, 4);
        misc[1] = 0;
        misc[2] = 0;
        fence_barrier_init();
    }
    if (warp == kWarpMma) {
        tmem_alloc(smem_u32(&misc[0]), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    grid_dep_launch();
    grid_dep_wait();

    // Tiles are taken round-robin; consecutive CTAs share an activation tile
    // (weights tile index varies fastest), so activations are reused in L2.
    if (warp == kWarpProd) {
        if (lane == 0) {
            prefetch_tensormap(&xmap);
            if (p.slices > 1) prefetch_tensormap(p.slices == 2 ? &xmap128 : &xmap64);
            const uint64_t pol_w = l2_policy_evict_last();
            const uint64_t pol_x = l2_policy_evict_last();
            int it = 0;
            for (int i = blockIdx.x; i < items; i += gridDim.x) {
                const Item w(i, p);
                const int tn = w.tile % p.n_tiles_n, tm = w.tile / p.n_tiles_n;
                // the activation box is the item's rows only (blocks of width x 128 bytes)
                const CUtensorMap *xm = w.width == kTileM ? &xmap : (w.width == 128 ? &xmap128 : &xmap64);
                const uint32_t xbytes = 2u * uint32_t(w.width) * 128u;
                bool ok = true;
                for (int g = w.g0; g < w.g1; ++g, ++it) {
                    const int s = it % kStages;
                    if (it >= kStages && !mbar_wait(empty(s), ((it / kStages) - 1) & 1, ab)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = base_s + s * kStage;
                    mbar_arrive_expect_tx(full(s), xbytes + kBlockBytes);
                    tma_load_3d(sa, xm, 0, tm * kTileM + w.col0, 2 * g, full(s), pol_x);
                    bulk_load(sa + kAct, p.wq + (size_t(tn) * p.n_groups + g) * kBlockBytes, kBlockBytes, full(s),
                              pol_w);
                }
                if (!ok) break;
            }
            if (*ab.flag) {
                for (int i = max(0, it - kStages); i < it; ++i) mbar_wait_bounded(full(i % kStages), (i / kStages) & 1);
            }
        }
    } else if (warp == kWarpMma || warp == kWarpMma2) {
        // Issuer h owns column half h of every whole-width tile (N = 128; each
        // column's k order is the same as with one N = 256 MMA).  A slice
        // (64 or 128 rows) is issued whole by issuer 0 -- it has no epilogue
        // stall to hide, and N = 32 halves ran slower -- while issuer 1 keeps
        // the same waits and commits with no MMAs.  The whole warp runs the
        // loop and lane 0 alone issues, so the operands stay warp-uniform.
        {
            const int h = warp == kWarpMma ? 0 : 1;
            int it = 0, nt = 0;
            bool ok = true;
            for (int i = blockIdx.x; i < items && ok; i += gridDim.x, ++nt) {
                const Item w(i, p);
                const bool split = w.width == kTileM;
                const int hw = split ? w.width / 2 : w.width;
                const bool issue = split || h == 0;
                const uint32_t idesc = idesc_f16_f32(128, hw);
                const uint32_t xblk = uint32_t(w.width) * 128u;     // one 64-k block of the item's rows
                const int x = 2 * nt + h, R = x % kRegions, u = x / kRegions;   // region R's use u
                if (u > 0 && !warp_wait(rempty(R), (u - 1) & 1, ab)) break;
                const uint32_t dcol = tmem + kDcol0 + uint32_t(R) * kRegionCols;
                for (int g = w.g0; g < w.g1; ++g, ++it) {
                    const int s = it % kStages;
                    const int slot = it % kASlots;
                    if (!warp_wait(full(s), (it / kStages) & 1, ab) ||
                        !warp_wait(afull(slot), (it / kASlots) & 1, ab)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t act = base_s + s * kStage;
                    if (issue) {
#pragma unroll
                        for (int j = 0; j < kGroup / 16; ++j) {
                            const uint32_t baddr = act + (j >> 2) * xblk + uint32_t(h * hw) * 128u + (j & 3) * 32;
                            mma_f16_ts_lane0(dcol, tmem + kAcol0 + slot * 64 + 8 * j, sdesc_sw128(baddr), idesc,
                                       (g > w.g0 || j > 0) ? 1u : 0u);
                        }
                    }
                    mma_commit_lane0(empty(s));
                    mma_commit_lane0(aempty(slot));
                }
                if (ok) mma_commit_lane0(rfull(R));
            }
            mma_commit_lane0(done_bar);
            mbar_wait_bounded(done_bar, 0);
            __syncwarp();
        }
    } else if (warp >= kWarpDq0 && warp < kWarpDq0 + 8) {
        const int q = warp & 3;
        const int set = (warp - kWarpDq0) >> 2;           // groups it with it % 2 == set
        const int r = 32 * q + lane;
        const uint32_t lane_base = uint32_t(32 * q) << 16;
        const __half2 sixteenth = __float2half2_rn(0.0625f);
        int it = 0;
        bool ok = true;
        for (int i = blockIdx.x; i < items && ok; i += gridDim.x) {
            const Item w(i, p);
            const int tn = w.tile % p.n_tiles_n;
            const int n = tn * kTileN + r;
            const bool valid = n < p.N;
            // scale rows per 128-k block: 1, or 4 with group size 32
            constexpr int kSub = kG32 ? 4 : 1;
            // The item's scale (and zero-point) rows are fetched into L2 up
            // front, one row of the tile's 128 columns per lane of set 0, so
            // the per-group loads below hit L2.
            if (set == 0 && tn * kTileN + kTileN <= p.N) {
                for (int row = 32 * q + lane; row < kSub * (w.g1 - w.g0); row += 128) {
                    const size_t off = size_t(kSub * w.g0 + row) * p.N + size_t(tn) * kTileN;
                    const __half *sp = p.scales + off;
                    if ((reinterpret_cast<uintptr_t>(sp) & 15u) == 0u) prefetch_l2(sp, kTileN * 2);
                    if (p.zeros != nullptr && (reinterpret_cast<uintptr_t>(p.zeros + off) & 15u) == 0u)
                        prefetch_l2(p.zeros + off, kTileN);
                }
            }
            for (int g = w.g0; g < w.g1; ++g, ++it) {
                if ((it & 1) != set) continue;
                const int s = it % kStages;
                const int slot = it % kASlots;
                float sc[kSub];
                uint32_t z[kSub];
#pragma unroll
                for (int c = 0; c < kSub; ++c) {
                    sc[c] = valid ? __half2float(__ldg(p.scales + size_t(kSub * g + c) * p.N + n)) : 0.f;
                    z[c] = 8;
                    if (p.zeros != nullptr && valid) z[c] = __ldg(p.zeros + size_t(kSub * g + c) * p.N + n);
                }
                if (!warp_wait(full(s), (it / kStages) & 1, ab)) {
                    ok = false;
                    break;
                }
                const uint8_t *wsm = base + s * kStage + kAct;
                uint4 v[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) v[j] = *reinterpret_cast<const uint4 *>(wsm + (j * 128 + r) * 16);
                __syncwarp();
                if (lane == 0) mbar_arrive(empty(s));
                uint32_t regs[64];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int c = kG32 ? j : 0;          // chunk j holds k = 32j .. 32j+31 of the block
                    const __half2 zlo = u32_as_h2((0x6400u + z[c]) * 0x10001u);
                    const __half2 zhi = __float2half2_rn(-(64.f + float(z[c])));
                    const __half2 scl = __float2half2_rn(sc[c]);
                    const uint32_t words[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
                    for (int wi = 0; wi < 4; ++wi) {
                        const uint32_t w = words[wi];
                        const uint32_t w8 = w >> 8;
                        const int o = 16 * j + 4 * wi;
                        regs[o + 0] = h2_as_u32(__hmul2(__hsub2(u32_as_h2(lop_and_or(w, 0x000F000Fu, 0x64006400u)), zlo), scl));
                        regs[o + 1] = h2_as_u32(__hmul2(__hfma2(u32_as_h2(lop_and_or(w, 0x00F000F0u, 0x64006400u)), sixteenth, zhi), scl));
                        regs[o + 2] = h2_as_u32(__hmul2(__hsub2(u32_as_h2(lop_and_or(w8, 0x000F000Fu, 0x64006400u)), zlo), scl));
                        regs[o + 3] = h2_as_u32(__hmul2(__hfma2(u32_as_h2(lop_and_or(w8, 0x00F000F0u, 0x64006400u)), sixteenth, zhi), scl));
                    }
                }
                if (it >= kASlots && !warp_wait(aempty(slot), ((it / kASlots) - 1) & 1, ab)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                tmem_st_32x32b_x32(tmem + lane_base + kAcol0 + slot * 64, *reinterpret_cast<uint32_t(*)[32]>(&regs[0]));
                tmem_st_32x32b_x32(tmem + lane_base + kAcol0 + slot * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&regs[32]));
                tc_wait_st();
                tc_keep_alive<64>(regs);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(afull(slot));
            }
        }
    } else if (warp >= kWarpEp0 && warp < kWarpEp0 + 4) {
        const int q = warp & 3;
        const int r = 32 * q + lane;
        const int ep = warp - kWarpEp0;
        const uint32_t lane_base = uint32_t(32 * q) << 16;
        uint32_t syncs = 0;
        auto ep_sync = [&]() -> bool {
            __syncwarp();
            if (lane == 0) mbar_arrive(ep_bar);
            return warp_wait(ep_bar, (syncs++) & 1, ab);
        };
        int nt = 0;
        for (int i = blockIdx.x; i < items; i += gridDim.x, ++nt) {
            const Item w(i, p);
            const int tn = w.tile % p.n_tiles_n, tm = w.tile / p.n_tiles_n;
            const int n = tn * kTileN + r;
            float *part = p.partial + (size_t(w.tile) * 2 + w.half) * kPart;
            // the tile's two column halves (a slice: all of it in the first),
            // each region released once read
            const bool split = w.width == kTileM;
            const int hw = split ? w.width / 2 : w.width;
            bool got = true;
            for (int h = 0; h < 2 && got; ++h) {
                const int x = 2 * nt + h, R = x % kRegions, u = x / kRegions;
                if (!warp_wait(rfull(R), u & 1, ab)) {
                    got = false;
                    break;
                }
                tc_fence_after();
                if (!split && h == 1) {                  // nothing was issued into it
                    __syncwarp();
                    if (lane == 0) mbar_arrive(rempty(R));
                    continue;
                }
                const uint32_t dcol = tmem + lane_base + kDcol0 + uint32_t(R) * kRegionCols;
#pragma unroll 1
                for (int c = 0; c < hw; c += 32) {
                    uint32_t d[32];
                    tmem_ld_32x32b_x32(dcol + c, d);
                    tc_wait_ld_keep<32>(d);
                    if (c + 32 == hw) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(rempty(R));
                    }
                    const int cc = h * hw + c;           // the item's column
                    if (p.halves == 1) {
                        if (n < p.N) {
#pragma unroll
                            for (int j = 0; j < 32; ++j) {
                                const int m = tm * kTileM + w.col0 + cc + j;
                                if (m < p.M) p.C[size_t(m) * p.N + n] = __float2half_rn(__uint_as_float(d[j]));
                            }
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j) __stcg(part + (cc + j) * kTileN + r, __uint_as_float(d[j]));
                    }
                }
            }
            if (!got) break;
            if (p.halves == 1) continue;
            // Split tile: the second half to arrive adds the two fp32 partials,
            // half 0 first (a fixed order, so the result is deterministic).
            if (!ep_sync()) break;
            if (ep == 0 && lane == 0) {
                const uint32_t prev = atom_add_acq_rel_gpu(p.tile_cnt + w.tile, 1u);
                const bool last = prev == 1u;
                if (last) p.tile_cnt[w.tile] = 0u;
                misc[2] = last ? 1u : 0u;
            }
            if (!ep_sync()) break;
            if (!misc[2]) continue;
            const float4 *p0 = reinterpret_cast<const float4 *>(p.partial + size_t(w.tile) * 2 * kPart);
            const float4 *p1 = p0 + kPart / 4;
            constexpr int kB = 8;                     // float4s per thread in flight
            for (int e0 = ep * 32 + lane; e0 < kPart / 4; e0 += 128 * kB) {
                float4 a[kB], b[kB];
#pragma unroll
                for (int k = 0; k < kB; ++k) {
                    a[k] = __ldcg(p0 + e0 + k * 128);
                    b[k] = __ldcg(p1 + e0 + k * 128);
                }
#pragma unroll
                for (int k = 0; k < kB; ++k) {
                    const int e = 4 * (e0 + k * 128);      // [m][n] element, consecutive threads: consecutive n
                    const int gm = tm * kTileM + e / kTileN, gn = tn * kTileN + e % kTileN;
                    if (gm < p.M && gn < p.N) {             // N % 8 == 0: four n are all in or all out
                        uint2 h;
                        h.x = h2_as_u32(__floats2half2_rn(a[k].x + b[k].x, a[k].y + b[k].y));
                        h.y = h2_as_u32(__floats2half2_rn(a[k].z + b[k].z, a[k].w + b[k].w));
                        *reinterpret_cast<uint2 *>(p.C + size_t(gm) * p.N + gn) = h;
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <bool kG32>
w4v_status launch(const CUtensorMap &xmap, const CUtensorMap &xmap128, const CUtensorMap &xmap64, const Args &a,
                  int grid, cudaStream_t stream) {
    static int configured_for = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_for != dev) {
        if (cudaFuncSetAttribute(w4a16_prefill_kernel<kG32>, cudaFuncAttributeMaxDynamicSharedMemorySize, kBytes) !=
            cudaSuccess) {
            cudaGetLastError();
            return W4V_ERR_CUDA;
        }
        configured_for = dev;
    }
    if (launch_pdl(w4a16_prefill_kernel<kG32>, dim3(grid), dim3(kThreads), kBytes, stream, xmap, xmap128, xmap64,
                   a) != cudaSuccess) {
        cudaGetLastError();
        return W4V_ERR_CUDA;
    }
    return W4V_OK;
}

}  // namespace

size_t w4a16_prefill_ws_bytes(int M, int N, int K) {
    (void)K;
    const size_t tiles = ((size_t(N) + kTileN - 1) / kTileN) * ((size_t(M) + kTileM - 1) / kTileM);
    const size_t partials = tiles <= size_t(kSplitMaxTiles) ? tiles * 2 * kPart * sizeof(float) : 0;
    return partials + ((tiles * sizeof(uint32_t) + 255) & ~size_t(255));
}

w4v_status launch_w4a16_prefill(const uint16_t *A, const void *Bq, const uint16_t *scales, const uint8_t *zeros,
                                int group, uint16_t *C, int M, int N, int K, void *ws, cudaStream_t stream) {
    const DeviceInfo *info = nullptr;
    w4v_status st = device_info(&info);
    if (st != W4V_OK) return st;
    Args a;
    a.wq = static_cast<const uint8_t *>(Bq);
    a.scales = reinterpret_cast<const __half *>(scales);
    a.zeros = zeros;
    a.C = reinterpret_cast<__half *>(C);
    a.status = info->status;
    a.M = M;
    a.N = N;
    a.K = K;
    a.n_tiles_n = (N + kTileN - 1) / kTileN;
    a.n_tiles_m = (M + kTileM - 1) / kTileM;
    a.n_groups = K / kGroup;
    // activation boxes of a whole tile's rows and of 128- and 64-row slices
    CUtensorMap xmap, xmap128, xmap64;
    st = encode_tmap_kblocks(&xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, A, uint64_t(K), uint64_t(M), 64, kTileM, 2,
                             CU_TENSOR_MAP_SWIZZLE_128B);
    if (st == W4V_OK)
        st = encode_tmap_kblocks(&xmap128, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, A, uint64_t(K), uint64_t(M), 64, 128, 2,
                                 CU_TENSOR_MAP_SWIZZLE_128B);
    if (st == W4V_OK)
        st = encode_tmap_kblocks(&xmap64, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, A, uint64_t(K), uint64_t(M), 64, 64, 2,
                                 CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != W4V_OK) return st;
    const long long tiles = (long long)a.n_tiles_n * a.n_tiles_m;
    // Split each tile's k range in two when that shortens the launch: a
    // whole tile costs G groups plus about 2 groups' time of epilogue, a half
    // G/2 plus about 4 (its fp32 partial out, and for the second half the
    // sum of both in).  E.g. down (G = 76) at 2048 rows: 160 tiles on 152
    // SMs are two waves of whole tiles, or three of halves.
    //
    // Or keep the full waves of whole tiles and cut each tile of a short last
    // wave into f slices (f * remaining tiles <= SMs, so they are one wave):
    // a slice of 64 rows costs about 0.45 of a whole tile's time (measured on
    // down and o at 2048 rows: 0.44-0.59, the dequantization pacing it), one
    // of 128 rows is taken as 0.6.
    const long long sms = info->sm_count;
    const long long G = a.n_groups;
    const long long waves1 = (tiles + sms - 1) / sms, waves2 = (2 * tiles + sms - 1) / sms;
    const long long rem = tiles % sms, whole = tiles - rem;
    const int f = rem == 0 ? 1 : (rem * 4 <= sms ? 4 : (rem * 2 <= sms ? 2 : 1));
    const double cost_whole = double(waves1) * double(G + 2);
    const double cost_halves = (G >= 2 && tiles <= kSplitMaxTiles) ? double(waves2) * double(G / 2 + 4) : 1e30;
    const double cost_slices =
        f > 1 ? double(whole / sms) * double(G + 2) + double(G) * (f == 4 ? 0.45 : 0.6) + 2.0 : 1e30;
    a.halves = 1;
    a.n_whole = static_cast<int>(tiles);
    a.slices = 1;
    if (cost_halves < cost_whole && cost_halves <= cost_slices) {
        a.halves = 2;
    } else if (cost_slices < cost_whole) {
        a.n_whole = static_cast<int>(whole);
        a.slices = f;
    }
    a.items = static_cast<int>(a.halves == 2 ? 2 * tiles : a.n_whole + (tiles - a.n_whole) * a.slices);
    const size_t part_bytes = tiles <= kSplitMaxTiles ? size_t(tiles) * 2 * kPart * sizeof(float) : 0;
    a.partial = static_cast<float *>(ws);
    a.tile_cnt = reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(ws) + part_bytes);
    const int grid = static_cast<int>(std::min<long long>(sms, a.items));
    return group == 32 ? launch<true>(xmap, xmap128, xmap64, a, grid, stream)
                       : launch<false>(xmap, xmap128, xmap64, a, grid, stream);
}

}  // namespace w4v
