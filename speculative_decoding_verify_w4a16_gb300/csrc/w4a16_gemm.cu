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
//   * A unit is a 128-row tile times two quantization groups (256 k).  Every
//     hand-off between roles costs a few hundred cycles of latency whatever
//     it carries, so units are made as large as tensor memory allows: three
//     A slots of 128 columns plus the accumulators fill the 512 columns.
//   * An SM completes about one TMA or bulk copy per ~650 cycles whatever its
//     size, so a stage is two units (four groups) of one tile: one 32 KB bulk
//     copy of packed int4 (the library's tile layout, evict-first) and one
//     3-D TMA of the four groups' activation slices (128-byte swizzle), both
//     issued by one producer thread.
//   * Eight dequant warps turn nibbles into exact fp16 (q - z) with LOP3 +
//     HFMA2 and store them into tensor memory with 32-column tcgen05.st.
//     Warp (quarter, parity) owns its 32 tile rows of every other unit and
//     does that unit's whole k in four 64-k steps, alternating two register
//     sets so each store overlaps the next step's arithmetic; the two warps
//     sharing a scheduler work on different units and so fall naturally out
//     of phase.  The dequantized operand never touches shared memory.
//   * tcgen05.mma (A from TMEM, B = activations from shared memory, D in
//     TMEM) is issued by three warps, unit f wholly by warp f % 3 (which so
//     owns A slot f % 3), the loop run by the whole warp with lane 0 issuing
//     so the operands stay warp-uniform.  Each wait on a completed barrier
//     and each commit costs a couple of hundred cycles, so a unit takes one
//     of each per barrier, and three units are in flight.  Each group
//     accumulates its 8 k-steps into its own accumulator block, so every
//     output element is the same chain of MMAs whatever the timing or M.
//   * Every wait is on an mbarrier phase parity, which names the phase only
//     if the barrier is neither a phase behind nor two ahead.  A waiter that
//     sees only some uses of a resource therefore gets a barrier of its own:
//     the A slot a unit frees is released to the dequant warps of the next
//     user's parity, the accumulator set to the issuer of its next user.
//   * Four drain warps read a unit's accumulators (one tcgen05.ld for both
//     groups) and apply the group scales in fp32, groups in ascending order.
//     The drain warps pace the pipeline (the accumulator sets they free gate
//     the issuers), so they issue no global loads: the producer copies each
//     stage's scales (four groups of one tile) with one 2-D TMA into a ring
//     of eight slots, which the drain frees stage by stage.  A load issued
//     by a drain warp stalls behind the weight stream's queued requests.
//     Zero points (and the group-32 scales) come the same way: the
//     producer's 2-D TMA of the stage's rows lands on the stage's weight
//     barrier, in per-stage slots that the dequant warps read.
//   * Work split.  With few 128-row tiles, each tile belongs to a
//     thread-block cluster of C CTAs (C about the square root of the units
//     per tile, at most 8, all clusters in one wave)
//     that split its k range; each CTA leaves its fp32 partial tile in its
//     own shared memory, and after one cluster barrier every CTA finishes
//     1/C of the tile's rows, reading the others' partials through
//     distributed shared memory and adding them in rank order: no global
//     round trip (well over a microsecond each on this two-die part), and
//     the remote reads are spread over the whole cluster.  With at least
//     as many tiles as SMs, the flat list of units is split evenly over one
//     CTA per SM (stream-K); a tile shared by several CTAs is finished by the
//     last one to arrive (acquire-release counter, no waiting between CTAs),
//     whose threads all load every contributor's float4 at once and add them
//     in CTA order.  Both orders are fixed, so the result is deterministic.
//   * The kernel is launched with programmatic stream serialization: barrier
//     set-up, tensor-memory allocation and an L2 prefetch of the first
//     weight stages overlap the end of the previous kernel in the stream.
//     When the caller declares the weights static (nothing still running
//     writes them), the first stages' weights are loaded, and their units
//     dequantized into tensor memory, before the dependency wait; only the
//     activation copies and the output wait for the previous kernel.  Each
//     stage therefore has separate weight and activation barriers.
#include <cstring>
#include <mutex>
#include <vector>

#include "runtime.h"
#define W4V_COMPACT_WAITS 1
#include "sm103_ptx.cuh"

namespace w4v {
namespace {

constexpr int kTileN = 128;                        // weight rows per tile (MMA M)
constexpr int kGroup = 128;                        // k per quantization group
constexpr int kGroupBytes = kTileN * kGroup / 2;   // packed bytes per (tile, group)
constexpr int kUnitGroups = 2;                     // groups per unit
constexpr int kStageUnits = 2;                     // units per stage
constexpr int kStageGroups = kUnitGroups * kStageUnits;
constexpr int kIssuers = 3;
constexpr int kDqWarps = 8;
constexpr int kDrWarps = 4;
constexpr int kWarpProd = 0;                       // producer
constexpr int kWarpIss0 = 1;                       // 1..3 MMA issuers (1 also owns TMEM)
constexpr int kWarpDr0 = 4;                        // 4..7 drain
constexpr int kWarpDq0 = 8;                        // 8..15 dequant
constexpr int kWarps = kWarpDq0 + kDqWarps;
constexpr int kThreads = 32 * kWarps;
constexpr int kASlots = 3;                         // unit f uses A slot f % 3
static_assert(kASlots == kIssuers && kStageUnits <= kIssuers,
              "issuer f % 3 owns A slot f % 3 and at most one unit of a stage");
constexpr uint32_t kASlotCols = kUnitGroups * 64;  // fp16 pairs of 128 rows x 256 k
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kDcol0 = kASlots * kASlotCols;
constexpr int kRing = 32;                          // sizes the metadata region below
// Group size 32 (scales folded into the weights): each stage's sub-group
// scales (16 rows of one tile, 4 KB) and zero points (2 KB) arrive with the
// stage's weights, into per-stage slots of the metadata region.
constexpr int kFSclSlotBytes = 4 * kStageGroups * kTileN * 2;
constexpr int kFZroSlotBytes = 4 * kStageGroups * kTileN;
// Group size 128 with zero points: each stage's rows of the zero table (four
// groups x one tile) arrive with its weights into a per-stage slot.
constexpr int kZroSlotBytes = kStageGroups * kTileN;

// Group size 128: the producer copies each stage's scales (its four groups'
// rows of one tile) into a ring of kSclSlots slots with one 2-D TMA, and the
// drain warps read them from there.
constexpr int kSclSlots = 8;
constexpr int kSclSlotBytes = kStageGroups * kTileN * 2;

constexpr int kMaxStages = 4;
constexpr int kMaxSmem = 227 * 1024;
// Largest cluster (portable size).  Measured on the 4B shapes at M = 16, each
// extra member costs about as much as one more unit per CTA, so the cluster
// size chosen is about the square root of the units per tile.
constexpr int kMaxCluster = 8;

// Shared memory: S stages, then a fixed block of barriers, metadata slots and flags.
// In cluster mode each CTA's partial tile ([row][16 NBLK] fp32) is left in
// its first stage once all its MMAs have completed.
template <int NBLK>
struct Layout {
    static constexpr int kRows = 16 * NBLK;                    // activation rows per box
    static constexpr int kActBox = kRows * 128;                // one 64-k block, swizzled
    static constexpr int kAct = 2 * kStageGroups * kActBox;
    static constexpr int kW = kAct;
    static constexpr int kStage = kW + kStageGroups * kGroupBytes;
    static constexpr uint32_t kDUnit = kUnitGroups * 16 * NBLK;   // accumulator columns per unit
    static constexpr int kDSets = int((kTmemCols - kDcol0) / kDUnit);
    // wfull, xfull, empty per stage (room for kMaxStages); afull per A slot
    // and group, aempty per A slot and dequant parity;
    // dfull, dempty per set; done; drain sync; sfull, sempty per scale slot
    static constexpr int kNumBars = 3 * kMaxStages + 4 * kASlots + (1 + kIssuers) * kDSets + 2 + 2 * kSclSlots;
    static constexpr int kBarBytes = (8 * kNumBars + 127) & ~127;
    static constexpr int kScl = kBarBytes;                         // offsets inside the fixed block
    static constexpr int kZro = kScl + kDrWarps * kRing * 64;      // group-32 scale slots from kScl
    static constexpr int kMisc = kZro + kDqWarps * kRing * 32;     // group-128 zero slots from kZro
    static_assert(kMaxStages * kFSclSlotBytes <= kMisc - kScl, "group-32 stage scales fit the metadata region");
    static constexpr int kSst = kMisc + 128;                        // stage scale ring (128-byte aligned)
    static_assert(kMisc % 16 == 0, "misc words hold 8-byte fields");
    static constexpr int kFixed = kSst + kSclSlots * kSclSlotBytes;
    static_assert(kMaxStages * kFZroSlotBytes <= kSclSlots * kSclSlotBytes, "group-32 stage zeros fit");
    static_assert(kMaxStages * kZroSlotBytes <= kMisc - kZro, "group-128 stage zeros fit");
    static constexpr int kPart = 16 * NBLK * kTileN;               // floats of one partial tile
    __host__ __device__ static constexpr int bytes(int stages) { return stages * kStage + kFixed + 1024; }
    static_assert(kStage % 1024 == 0, "stage alignment");
    static_assert(kDSets >= 2, "tensor memory plan");
    static constexpr int kStagesMax = (kMaxSmem - kFixed - 1024) / kStage < kMaxStages
                                          ? (kMaxSmem - kFixed - 1024) / kStage
                                          : kMaxStages;
    static_assert(kStagesMax >= 2 && bytes(kStagesMax) <= kMaxSmem, "shared memory plan");
    static_assert(kPart * 4 <= kStage, "partial tile fits a stage");
};

// One problem of a grouped launch (w4a16_gemm_grouped): the tensor maps and
// sizes every role needs, read from a device table written by the host.
// Problem i owns the global units [u0, u0 + n_tiles * n_pairs) and the
// global output tiles [tile0, tile0 + n_tiles).
struct GroupProb {   // 64-byte aligned, as its first member
    CUtensorMap xmap, smap, zmap;   // activations, scales, zero points (as for one problem)
    const uint8_t *wq;
    __half *C;
    long long u0;
    int N, n_groups, n_pairs, n_tiles, tile0, sbox_w, sbox_h, pad;
};
static_assert(sizeof(GroupProb) % 64 == 0, "tensor maps in the table stay 64-byte aligned");

struct Args {
    const GroupProb *probs;   // grouped launch: the problem table (else null)
    int n_probs;
    const uint8_t *wq;
    const __half *scales;
    const uint8_t *zeros;
    __half *C;
    float *partial;        // [P][2][16*NBLK][128] (stream-K only)
    uint32_t *tile_cnt;    // [n_tiles] (stream-K only)
    uint32_t *status;
    int M, N, K;
    int n_tiles, n_groups, n_pairs;   // n_pairs = units per tile
    int P;                            // CTAs
    long long U;                      // units
    int stages;                       // pipeline stages in shared memory
    int cluster;                      // CTAs per tile (cluster size); 0 = stream-K
    int static_w;                     // weights, scales, zeros not written by earlier work in flight
    int sbox_w, sbox_h;               // scale box of one stage: min(128, N) x min(4 or 16, K / group)
};

// The sizes of the problem a walker is in: units per tile, groups, tiles.
struct ProbDims {
    int nP, G, nT;
};

// The problem whose unit range holds global unit u (the table is ordered by
// u0 and starts at 0).
__device__ __forceinline__ int find_prob(const GroupProb *probs, int n, long long u) {
    int lo = 0, hi = n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(&probs[mid].u0) <= u) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ ProbDims prob_dims(const GroupProb *g) {
    return ProbDims{__ldg(&g->n_pairs), __ldg(&g->n_groups), __ldg(&g->n_tiles)};
}

// A unit: problem pi (grouped launches only, else 0), tile t of that
// problem, pair p (groups 2p and, if it exists, 2p + 1).
template <bool kG>
struct UnitPos {
    const GroupProb *probs;
    int n_probs, pi, t, p, nP, G, nT;
    __device__ UnitPos(long long u, const Args &a)
        : probs(a.probs), n_probs(a.n_probs), pi(0), nP(a.n_pairs), G(a.n_groups), nT(a.n_tiles) {
        if constexpr (kG) {
            pi = find_prob(probs, n_probs, u);
            u -= __ldg(&probs[pi].u0);
            const ProbDims d = prob_dims(probs + pi);
            nP = d.nP;
            G = d.G;
            nT = d.nT;
        }
        t = static_cast<int>(u / nP);
        p = static_cast<int>(u % nP);
    }
    __device__ int g0() const { return 2 * p; }
    __device__ int ng() const { return min(kUnitGroups, G - 2 * p); }
    __device__ bool tile_last() const { return p == nP - 1; }
    __device__ void next() {
        if (++p == nP) {
            p = 0;
            ++t;
            if (kG && t == nT && pi + 1 < n_probs) {
                t = 0;
                const ProbDims d = prob_dims(probs + ++pi);
                nP = d.nP;
                G = d.G;
                nT = d.nT;
            }
        }
    }
};

// Stages: runs of at most kStageUnits consecutive units of one tile.
template <bool kG>
struct StageWalk {
    const GroupProb *probs;
    int n_probs, pi, t, p, nP, G, nT, left;
    __device__ StageWalk(long long u, const Args &a, int units)
        : probs(a.probs), n_probs(a.n_probs), pi(0), nP(a.n_pairs), G(a.n_groups), nT(a.n_tiles), left(units) {
        if constexpr (kG) {
            pi = find_prob(probs, n_probs, u);
            u -= __ldg(&probs[pi].u0);
            const ProbDims d = prob_dims(probs + pi);
            nP = d.nP;
            G = d.G;
            nT = d.nT;
        }
        t = static_cast<int>(u / nP);
        p = static_cast<int>(u % nP);
    }
    __device__ int size() const { return min(min(kStageUnits, nP - p), left); }
    __device__ int gbeg() const { return 2 * p; }
    __device__ int gend(int n) const { return min(2 * (p + n), G); }
    __device__ void next(int n) {
        p += n;
        left -= n;
        if (p == nP) {
            p = 0;
            ++t;
            if (kG && t == nT && left > 0 && pi + 1 < n_probs) {
                t = 0;
                const ProbDims d = prob_dims(probs + ++pi);
                nP = d.nP;
                G = d.G;
                nT = d.nT;
            }
        }
    }
};

// Position in the ring of S stages: slot and phase parity of the current use
// (kept incrementally; S is a launch parameter).
struct StageRing {
    int S, s = 0;
    uint32_t ph = 0;
    bool wrapped = false;
    __device__ explicit StageRing(int stages) : S(stages) {}
    __device__ void next() {
        if (++s == S) {
            s = 0;
            ph ^= 1u;
            wrapped = true;
        }
    }
};

// kFold: group size 32.  The dequant warps multiply each weight by its
// sub-group's scale (fp16, one rounding) and the accumulators of a 128-k
// group are added unscaled; with group size 128 the scale is applied to each
// group's fp32 sum instead.
// kG: grouped launch.  The units of every problem of the table are numbered
// one after the other and split over the CTAs as one stream-K list; each
// role follows the problem of the unit it is on (its weights, tensor maps,
// output), so one pipeline and one ramp serve the whole list.
// kZ (group size 128 only): a zero-point table is given; without one the
// zero point 8 is a compile-time constant of the dequantization (its
// offsets become immediates: ~5 % of the unit period).
template <int NBLK, bool kFold, bool kG, bool kZ = false>
__global__ void __launch_bounds__(kThreads, 1)
w4a16_decode_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap smap,
                    const __grid_constant__ CUtensorMap zmap, const Args p) {
    using L = Layout<NBLK>;
    constexpr int DS = L::kDSets;
    constexpr int MS = kMaxStages;
    const int S = p.stages;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    uint8_t *base = smem_raw + (base_s - raw_s);
    const uint32_t fixed_off = uint32_t(S) * L::kStage;

    const uint32_t bar0 = base_s + fixed_off;
    auto wfull = [&](int s) { return bar0 + 8u * s; };          // stage's weights landed
    auto xfull = [&](int s) { return bar0 + 8u * (MS + s); };   // stage's activations landed
    auto empty = [&](int s) { return bar0 + 8u * (2 * MS + s); };
    // group g of the unit in A slot a dequantized (the slot's issuer starts
    // on group 0 while group 1 is still being dequantized)
    auto afull = [&](int a, int g) { return bar0 + 8u * (3 * MS + 2 * a + g); };
    // A slot a freed for the dequant warps of parity par: unit u's MMAs release
    // slot u % 3 to its next user u + 3, of parity (u + 1) % 2.  Each waiter
    // so sees every phase of its barrier in turn (one barrier per slot would
    // let a parity skip a phase).
    auto aempty = [&](int a, int par) { return bar0 + 8u * (3 * MS + 2 * kASlots + 2 * a + par); };
    auto dfull = [&](int b) { return bar0 + 8u * (3 * MS + 4 * kASlots + b); };
    // accumulator set b freed for issuer i: the drain of unit u releases set
    // u % DS to its next user u + DS, issued by (u + DS) % 3, so each issuer
    // sees every phase of its own barriers
    auto dempty = [&](int b, int i) { return bar0 + 8u * (3 * MS + 4 * kASlots + DS + b * kIssuers + i); };
    const uint32_t done_bar = bar0 + 8u * (3 * MS + 4 * kASlots + (1 + kIssuers) * DS);
    const uint32_t drain_bar = done_bar + 8u;
    auto sfull = [&](int b) { return drain_bar + 8u * (1 + b); };               // a stage's scales landed
    auto sempty = [&](int b) { return drain_bar + 8u * (1 + kSclSlots + b); };  // the drain has read them
    const uint32_t sst = base_s + fixed_off + L::kSst;
    // [0] tmem base, [1] abort flag, [2..3] pending tile + 1 per slot, [4..5] last-arriver flags,
    // [8..27] the pending tiles themselves (PendTile, one per slot)
    uint32_t *misc = reinterpret_cast<uint32_t *>(base + fixed_off + L::kMisc);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int cta = blockIdx.x;
    // 0: stream-K (a grouped launch is always stream-K); the divisions below
    // see CL only where it is positive
    const int CL = kG ? 0 : p.cluster;
    const int CLd = kG ? 1 : max(p.cluster, 1);
    const int crank = CL > 0 ? static_cast<int>(cluster_ctarank()) : 0;
    long long ub, ue;
    if (CL > 0) {
        // one tile per cluster; member `crank` takes its share of the tile's units
        const int nP = p.n_pairs;
        const long long t0u = (long long)(cta / CLd) * nP;
        ub = t0u + (long long)crank * nP / CLd;
        ue = t0u + (long long)(crank + 1) * nP / CLd;
    } else {
        ub = split_begin(cta, p.U, p.P);
        ue = split_begin(cta + 1, p.U, p.P);
    }
    const int nunits = static_cast<int>(ue - ub);
    AbortState ab{reinterpret_cast<volatile uint32_t *>(&misc[1]), p.status};

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(wfull(s), 1);
            mbar_init(xfull(s), 1);
            mbar_init(empty(s), kDqWarps + kStageUnits);   // dequant warps + one per unit's issuer
        }
        for (int a = 0; a < kASlots; ++a) {
            mbar_init(afull(a, 0), kDqWarps / 2);  // the four quarter warps of the unit's parity
            mbar_init(afull(a, 1), kDqWarps / 2);
            mbar_init(aempty(a, 0), 1);            // the unit's issuer
            mbar_init(aempty(a, 1), 1);
        }
        for (int b = 0; b < DS; ++b) {
            mbar_init(dfull(b), 1);
            for (int i = 0; i < kIssuers; ++i) mbar_init(dempty(b, i), kDrWarps);
        }
        mbar_init(done_bar, kIssuers);
        mbar_init(drain_bar, kDrWarps);
        for (int b = 0; b < kSclSlots; ++b) {
            mbar_init(sfull(b), 1);
            mbar_init(sempty(b), kDrWarps);
        }
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
    grid_dep_launch();

    // What each role needs of the problem it is on (a grouped launch reads
    // the table; one problem reads the launch arguments).
    auto pr_wq = [&](int pi) -> const uint8_t * {
        if constexpr (kG) return p.probs[pi].wq;
        return p.wq;
    };
    auto pr_xmap = [&](int pi) -> const CUtensorMap * {
        if constexpr (kG) return &p.probs[pi].xmap;
        return &xmap;
    };
    auto pr_smap = [&](int pi) -> const CUtensorMap * {
        if constexpr (kG) return &p.probs[pi].smap;
        return &smap;
    };
    auto pr_zmap = [&](int pi) -> const CUtensorMap * {
        if constexpr (kG) return &p.probs[pi].zmap;
        return &zmap;
    };
    auto pr_sbox_w = [&](int pi) -> int {
        if constexpr (kG) return p.probs[pi].sbox_w;
        return p.sbox_w;
    };
    auto pr_sbox_h = [&](int pi) -> int {
        if constexpr (kG) return p.probs[pi].sbox_h;
        return p.sbox_h;
    };
    using Walk = StageWalk<kG>;
    // Tile t of problem pi: its first unit (global numbering), units, rows,
    // output and index among all tiles of the launch (arrival counters).
    struct TileRef {
        long long t0u;
        int nP, N, T;
        __half *C;
    };
    // A split tile this CTA published a partial of, as the drain saw it when
    // it flushed (the fix-up then needs no second look at the problem table),
    // with the CTAs contributing to it.
    struct PendTile {
        TileRef tr;
        int cf, cl;
    };
    static_assert(2 * sizeof(PendTile) <= 20 * sizeof(uint32_t), "pending tiles fit the misc words");
    PendTile *pend = reinterpret_cast<PendTile *>(misc + 8);
    auto tile_ref = [&](int pi, int t) -> TileRef {
        if constexpr (kG) {
            const GroupProb &g = p.probs[pi];
            const int nPp = g.n_pairs;
            return TileRef{g.u0 + (long long)t * nPp, nPp, g.N, g.tile0 + t, g.C};
        }
        return TileRef{(long long)t * p.n_pairs, p.n_pairs, p.N, t, p.C};
    };

    if (warp == kWarpProd) {
        // ---------------------------------------------------------- producer
        const uint64_t pol_w = l2_policy_evict_first();
        const uint64_t pol_x = l2_policy_evict_last();
        const bool stage_zeros = p.zeros != nullptr;
        // bytes riding on the weight barrier: group 32 scales (and zeros), group 128 zeros
        auto meta_bytes = [&](int pi) -> uint32_t {
            return uint32_t(pr_sbox_w(pi) * pr_sbox_h(pi)) *
                   (kFold ? (stage_zeros ? 3u : 2u) : (stage_zeros ? 1u : 0u));
        };
        auto load_weights = [&](const Walk &w, int n, int s) {
            const int g0 = w.gbeg();
            const uint32_t wbytes = (w.gend(n) - g0) * kGroupBytes;
            mbar_arrive_expect_tx(wfull(s), wbytes + meta_bytes(w.pi));
            bulk_load(base_s + s * L::kStage + L::kW, pr_wq(w.pi) + (size_t(w.t) * w.G + g0) * kGroupBytes, wbytes,
                      wfull(s), pol_w);
            if (kFold) {
                // the stage's sub-group scales and zero points ride with its weights
                // (rows past N or K land as zero)
                tma_load_2d(base_s + fixed_off + L::kScl + uint32_t(s * kFSclSlotBytes), pr_smap(w.pi), w.t * kTileN,
                            4 * g0, wfull(s), pol_w);
                if (stage_zeros)
                    tma_load_2d(base_s + fixed_off + L::kSst + uint32_t(s * kFZroSlotBytes), pr_zmap(w.pi),
                                w.t * kTileN, 4 * g0, wfull(s), pol_w);
            } else if (stage_zeros) {
                tma_load_2d(base_s + fixed_off + L::kZro + uint32_t(s * kZroSlotBytes), pr_zmap(w.pi), w.t * kTileN,
                            g0, wfull(s), pol_w);
            }
        };
        // stage use u's scales into slot u % kSclSlots (rows past N or K land as zero)
        auto load_scales = [&](const Walk &w, int u) {
            if (kFold) return;
            const int b = u % kSclSlots;
            mbar_arrive_expect_tx(sfull(b), uint32_t(pr_sbox_w(w.pi) * pr_sbox_h(w.pi) * 2));
            tma_load_2d(sst + uint32_t(b * kSclSlotBytes), pr_smap(w.pi), w.t * kTileN, w.gbeg(), sfull(b), pol_w);
        };
        int w_early = 0;                         // stages whose weights went out before the wait
        if (lane == 0) {
            if constexpr (!kG) {
                prefetch_tensormap(&xmap);
                prefetch_tensormap(&smap);
                if (p.zeros != nullptr) prefetch_tensormap(&zmap);
            }
            Walk pw(ub, p, nunits);
            for (int st = 0; st < S && pw.left > 0; ++st) {
                const int n = pw.size();
                if (p.static_w) {
                    load_weights(pw, n, st);
                    load_scales(pw, st);         // st < S <= kSclSlots: the slot is fresh
                    ++w_early;
                } else {
                    // Only L2 is warmed before the dependency wait: L2 is the
                    // point of coherence, so this stays correct even if the
                    // previous kernel writes the weights.
                    prefetch_l2(pr_wq(pw.pi) + (size_t(pw.t) * pw.G + pw.gbeg()) * kGroupBytes,
                                (pw.gend(n) - pw.gbeg()) * kGroupBytes);
                }
                pw.next(n);
            }
        }
        Walk sw(ub, p, nunits);
        int issued = 0;
        grid_dep_wait();
        if (lane == 0) {
            StageRing rg(S);
            for (; sw.left > 0; rg.next()) {
                const int n = sw.size();
                const int s = rg.s;
                if (rg.wrapped && !mbar_wait(empty(s), rg.ph ^ 1u, ab)) break;
                if (issued >= w_early) {
                    // the slot's previous stage must have been read by the drain
                    if (!kFold && issued >= kSclSlots &&
                        !mbar_wait(sempty(issued % kSclSlots), uint32_t(issued / kSclSlots - 1) & 1u, ab))
                        break;
                    load_weights(sw, n, s);
                    load_scales(sw, issued);
                }
                mbar_arrive_expect_tx(xfull(s), L::kAct);
                tma_load_3d(base_s + s * L::kStage, pr_xmap(sw.pi), 0, 0, 2 * sw.gbeg(), xfull(s), pol_x);
                ++issued;
                sw.next(n);
            }
            if (*ab.flag) {
                // Let every copy still in flight land before the CTA exits.
                const int w_issued = max(issued, w_early);
                for (int i = max(0, w_issued - S); i < w_issued; ++i)
                    mbar_wait_bounded(wfull(i % S), uint32_t(i / S) & 1u);
                for (int i = max(0, issued - S); i < issued; ++i)
                    mbar_wait_bounded(xfull(i % S), uint32_t(i / S) & 1u);
                if (!kFold)
                    for (int i = max(0, w_issued - kSclSlots); i < w_issued; ++i)
                        mbar_wait_bounded(sfull(i % kSclSlots), uint32_t(i / kSclSlots) & 1u);
            }
        }
    } else if (warp >= kWarpIss0 && warp < kWarpIss0 + kIssuers) {
        // ------------------------------------------------------ MMA issuers
        // (shared and tensor memory only: ordered by the stage barriers).
        // Issuer me owns every unit f with f % 3 == me -- both of its groups,
        // so one wait per barrier and one commit per consumer a unit -- and
        // with it A slot me.  The whole warp runs the loop and lane 0 alone
        // issues, so the operands stay warp-uniform.
        {
            const int me = warp - kWarpIss0;
            constexpr uint32_t idesc = idesc_f16_f32(128, 16 * NBLK);
            constexpr int kSetPeriod = DS * kIssuers;       // units between uses of one dempty barrier
            const int slot = me;                            // unit f uses A slot f % 3
            // The issuer visits its own units f = me, me + 3, ... only (never two
            // in one stage): the stage walker is advanced to the unit's stage.
            Walk sw(ub, p, nunits);
            int f0 = 0, n = sw.size();
            StageRing rg(S);
            int set = me % DS;
            for (int f = me; f < nunits; f += kIssuers) {
                while (f >= f0 + n) {
                    f0 += n;
                    sw.next(n);
                    rg.next();
                    n = sw.size();
                }
                const int jj = f - f0;
                const int s = rg.s;
                const int ng = min(kUnitGroups, sw.G - 2 * (sw.p + jj));
                const uint32_t apar = uint32_t(f / kASlots) & 1u;
                const uint32_t dpar = uint32_t((f - DS) / kSetPeriod) & 1u;
                // afull before xfull: the unit's weights were dequantized, so
                // this stage's previous use is complete and the parity of xfull
                // names this use (an issuer skips the stages it has no unit
                // in).  The free accumulator set is waited for first with four
                // sets (M <= 16), last with two (measured).  Every unit arrives
                // on both group barriers of its slot (a unit with one group
                // without data on the second).
                const bool set_ok = f < DS || NBLK != 1 || warp_wait(dempty(set, me), dpar, ab);
                if (!set_ok || !warp_wait(afull(slot, 0), apar, ab) || !warp_wait(xfull(s), rg.ph, ab) ||
                    (NBLK != 1 && f >= DS && !warp_wait(dempty(set, me), dpar, ab)))
                    break;
                tc_fence_after();
                const uint32_t dset = tmem + kDcol0 + set * L::kDUnit;
                const uint32_t act = base_s + s * L::kStage + 2 * (kUnitGroups * jj) * L::kActBox;
                bool gok = true;
                for (int gg = 0; gg < ng; ++gg) {
                    if (gg > 0) {
                        if (!warp_wait(afull(slot, gg), apar, ab)) {
                            gok = false;
                            break;
                        }
                        tc_fence_after();
                    }
                    const uint64_t desc0 = sdesc_sw128(act + 2 * gg * L::kActBox);
#pragma unroll
                    for (int j = 0; j < kGroup / 16; ++j) {
                        // all 16 NBLK activation rows in one MMA (N = 16 NBLK); the
                        // descriptor's start address field is in 16-byte units
                        const uint64_t desc = desc0 + uint64_t(((j >> 2) * L::kActBox + (j & 3) * 32) >> 4);
                        mma_f16_ts_lane0(dset + gg * NBLK * 16, tmem + slot * kASlotCols + gg * 64 + 8 * j, desc,
                                         idesc, j > 0 ? 1u : 0u);
                    }
                }
                if (!gok) break;
                if (ng == 1 && !warp_wait(afull(slot, 1), apar, ab)) break;
                mma_commit_lane0(aempty(slot, (f + 1) & 1));
                mma_commit_lane0(dfull(set));
                // one release of the stage per unit (a one-unit stage counts twice)
                mma_commit_lane0(empty(s));
                if (n == 1) mma_commit_lane0(empty(s));
                set = (set + kIssuers) % DS;     // DS may be smaller than the stride
            }
            // Every MMA of this issuer has finished once this arrives.
            mma_commit_lane0(done_bar);
            mbar_wait_bounded(done_bar, 0);
            __syncwarp();
        }
    } else if (warp >= kWarpDq0) {
        // --------------------------------------------------------- dequant
        const int dq = warp - kWarpDq0;
        const int q = warp & 3;                 // TMEM lane quarter
        const int par = dq >> 2;                // units f with f % 2 == par
        const int r = 32 * q + lane;            // row inside the tile
        const uint32_t lane_base = uint32_t(32 * q) << 16;
        const __half2 sixteenth = __float2half2_rn(0.0625f);
        // reads only weights, zero points and shared memory
        if (!p.static_w) grid_dep_wait();

        // Zero points (group 128): row g of the stage's slot, for this lane's
        // row of the tile (rows past N read as 0 and are never stored).
        const bool has_zeros = p.zeros != nullptr;
        // (sbw: the stage's scale and zero box width, min(128, N))
        auto zero_read = [&](int s, int gs, int sbw) -> uint32_t {
            return lds_u8(base_s + fixed_off + L::kZro + uint32_t(s * kZroSlotBytes) + uint32_t(gs * sbw + r));
        };

        // Group size 32: the four sub-groups' zero points (bytes of zz) and
        // scales (halves of ss0, ss1) of 128-k group gs of the stage in slot s,
        // for this lane's row.
        auto fold_read = [&](int s, int gs, int sbw, uint32_t &zz, uint32_t &ss0, uint32_t &ss1) {
            const uint32_t sp = uint32_t(sbw * 2), zp = uint32_t(sbw);
            const uint32_t e = base_s + fixed_off + L::kScl + uint32_t(s * kFSclSlotBytes) + uint32_t(4 * gs) * sp +
                               uint32_t(2 * r);
            ss0 = uint32_t(lds_u16(e)) | (uint32_t(lds_u16(e + sp)) << 16);
            ss1 = uint32_t(lds_u16(e + 2 * sp)) | (uint32_t(lds_u16(e + 3 * sp)) << 16);
            zz = 0x08080808u;
            if (has_zeros) {
                const uint32_t z = base_s + fixed_off + L::kSst + uint32_t(s * kFZroSlotBytes) + uint32_t(4 * gs) * zp +
                                   uint32_t(r);
                zz = lds_u8(z) | (lds_u8(z + zp) << 8) | (lds_u8(z + 2 * zp) << 16) | (lds_u8(z + 3 * zp) << 24);
            }
        };

        // One 64-k step: chunks 2kh, 2kh+1 of the packed group at shared address `grp`,
        // dequantized with zero point z into 32 half2 registers.
        auto load_half = [&](uint32_t grp, int kh, uint4 &va, uint4 &vb) {
            va = lds128(grp + ((2 * kh) * 128 + r) * 16);
            vb = lds128(grp + ((2 * kh + 1) * 128 + r) * 16);
        };
        auto convert = [&](const uint4 &va, const uint4 &vb, uint32_t z, uint32_t (&regs)[32]) {
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
        };
        // Group size 32: the same, each 32-k chunk c (c = 2kh, 2kh+1) with its
        // own zero point (byte c of zz) and scale (half c of ss0:ss1), and the
        // exact q - z multiplied by the scale in fp16.
        auto dequant_fold = [&](uint32_t grp, int kh, uint32_t zz, uint32_t ss0, uint32_t ss1, uint32_t (&regs)[32]) {
            const uint4 va = lds128(grp + ((2 * kh) * 128 + r) * 16);
            const uint4 vb = lds128(grp + ((2 * kh + 1) * 128 + r) * 16);
            const uint32_t ss = kh == 0 ? ss0 : ss1;
            const uint32_t words[8] = {va.x, va.y, va.z, va.w, vb.x, vb.y, vb.z, vb.w};
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const uint32_t z = (zz >> (8 * (2 * kh + half))) & 0xFFu;
                const uint32_t sh = half == 0 ? (ss & 0xFFFFu) : (ss >> 16);
                const __half2 sc = u32_as_h2(sh * 0x10001u);
                const __half2 zlo = u32_as_h2((0x6400u + z) * 0x10001u);
                const __half2 zhi = __float2half2_rn(-(64.f + float(z)));
#pragma unroll
                for (int wj = 0; wj < 4; ++wj) {
                    const int wi = 4 * half + wj;
                    const uint32_t v = words[wi];
                    const uint32_t v8 = v >> 8;
                    const uint32_t lo0 = lop_and_or(v, 0x000F000Fu, 0x64006400u);
                    const uint32_t hi0 = lop_and_or(v, 0x00F000F0u, 0x64006400u);
                    const uint32_t lo1 = lop_and_or(v8, 0x000F000Fu, 0x64006400u);
                    const uint32_t hi1 = lop_and_or(v8, 0x00F000F0u, 0x64006400u);
                    regs[4 * wi + 0] = h2_as_u32(__hmul2(__hsub2(u32_as_h2(lo0), zlo), sc));
                    regs[4 * wi + 1] = h2_as_u32(__hmul2(__hfma2(u32_as_h2(hi0), sixteenth, zhi), sc));
                    regs[4 * wi + 2] = h2_as_u32(__hmul2(__hsub2(u32_as_h2(lo1), zlo), sc));
                    regs[4 * wi + 3] = h2_as_u32(__hmul2(__hfma2(u32_as_h2(hi1), sixteenth, zhi), sc));
                }
            }
        };
        auto release = [&](int s) {
            __syncwarp();
            if (lane == 0) mbar_arrive(empty(s));
        };

        Walk sw(ub, p, nunits);
        int f0 = 0;
        uint32_t ra[32], rb[32];
        StageRing rg(S);
        for (; sw.left > 0; rg.next()) {
            const int n = sw.size();
            const int s = rg.s;
            // Every dequant warp waits for every stage and releases it once.
            if (!warp_wait(wfull(s), rg.ph, ab)) break;
            const int jj = (par - f0) & 1;       // this warp's unit in the stage, if any
            if (jj >= n) {
                release(s);
            } else {
                const int f = f0 + jj;
                const int ng = min(kUnitGroups, sw.G - 2 * (sw.p + jj));
                const int slot = f % kASlots;
                const int sbw = (kZ || kFold) ? pr_sbox_w(sw.pi) : 0;
                const uint32_t g0p = base_s + s * L::kStage + L::kW + (kUnitGroups * jj) * kGroupBytes;
                const uint32_t g1p = g0p + kGroupBytes;
                const uint32_t col = tmem + lane_base + slot * kASlotCols;
                // group gg: half 0 into ra, half 1 into rb; each store
                // overlaps the next half's arithmetic.  Both groups are
                // unrolled, so the second group's loads and arithmetic
                // schedule against the first's tail (~14 % of the unit
                // period against a loop of one group per trip).
                bool aborted = false, released = false;
#pragma unroll
                for (int gg = 0; gg < kUnitGroups; ++gg) {
                    if (gg >= ng) break;
                    const uint32_t gp = gg == 0 ? g0p : g1p;
                    const uint32_t z = (!kFold && kZ) ? zero_read(s, kUnitGroups * jj + gg, sbw) : 8u;
                    uint32_t zz = 0u, ss0 = 0u, ss1 = 0u;
                    // group size 128: both halves' packed words are loaded up
                    // front, so the shared-memory latency is paid once a group
                    uint4 h0a, h0b, h1a, h1b;
                    if constexpr (kFold) {
                        fold_read(s, kUnitGroups * jj + gg, sbw, zz, ss0, ss1);
                        dequant_fold(gp, 0, zz, ss0, ss1, ra);
                    } else {
                        load_half(gp, 0, h0a, h0b);
                        load_half(gp, 1, h1a, h1b);
                        if (gg == ng - 1) {               // last shared-memory read of the stage
                            release(s);
                            released = true;
                        }
                        convert(h0a, h0b, z, ra);
                    }
                    if (gg == 0) {
                        // the release by unit f - 3: this parity's ((f - 3) / 6)-th on the barrier
                        if (f >= kASlots && !warp_wait(aempty(slot, f & 1), uint32_t((f - kASlots) / 6) & 1u, ab)) {
                            aborted = true;
                            break;
                        }
                        tc_fence_after();
                    }
                    tmem_st_32x32b_x32(col + 64 * gg, ra);
                    if constexpr (kFold) {
                        dequant_fold(gp, 1, zz, ss0, ss1, rb);
                        if (gg == ng - 1) {               // last shared-memory read of the stage
                            release(s);
                            released = true;
                        }
                    } else {
                        convert(h1a, h1b, z, rb);
                    }
                    tmem_st_32x32b_x32(col + 64 * gg + 32, rb);
                    // the group is in tensor memory: the slot's issuer may start on
                    // it while the next group is being dequantized
                    tc_wait_st();
                    tc_keep_alive<32>(ra);
                    tc_keep_alive<32>(rb);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(afull(slot, gg));
                }
                if (aborted) {
                    if (!released) release(s);
                    break;
                }
                // a unit with one group still completes its group-1 barrier
                if (ng == 1 && lane == 0) mbar_arrive(afull(slot, 1));
            }
            f0 += n;
            sw.next(n);
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
        if (!p.static_w) grid_dep_wait();

        // The unit's group scales come from the stage scale ring (rows past
        // N read as 0 and are never stored): dw walks the stages as the
        // producer does, du is the stage use, dj the unit within the stage.
        Walk dw(ub, p, nunits);
        int du = 0, dj = 0;
        const uint32_t srow = uint32_t(2 * r);
        if (p.static_w) grid_dep_wait();     // before any write of C or the workspace

        // Tile finished by this CTA alone: write C.  Otherwise publish the fp32
        // partial tile and count this CTA in; whether it arrived last is read
        // back after the CTA's last unit (see fixup).
        auto flush = [&](int pi, int t) -> bool {
            const TileRef tr = tile_ref(pi, t);
            const long long t0u = tr.t0u;
            const long long t1u = t0u + tr.nP;
            const int n = t * kTileN + r;
            if (CL > 1) {
                // cluster: partial tile [row][16 NBLK] into this CTA's first
                // stage (every MMA of this CTA has completed); the cluster
                // adds the partials after the role loops
                const uint32_t dst = base_s + uint32_t(r) * (16 * NBLK * 4);
#pragma unroll
                for (int b = 0; b < NBLK; ++b)
#pragma unroll
                    for (int j = 0; j < 16; j += 4)
                        sts_f32x4(dst + (16 * b + j) * 4, acc[b][j], acc[b][j + 1], acc[b][j + 2], acc[b][j + 3]);
                return true;
            }
            if (ub <= t0u && t1u <= ue) {
                if (n < tr.N) {
#pragma unroll
                    for (int b = 0; b < NBLK; ++b)
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const int m = 16 * b + j;
                            if (m < p.M) tr.C[size_t(m) * tr.N + n] = __float2half_rn(acc[b][j]);
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
                pend_prev[slot] = atom_add_acq_rel_gpu(&p.tile_cnt[tr.T], 1u);
                misc[2 + slot] = uint32_t(t) + 1u;
                pend[slot] = PendTile{tr, split_owner(t0u, p.U, p.P), split_owner(t1u - 1, p.U, p.P)};
            }
            return true;
        };

        // After the CTA's last unit: decide, for each published partial tile,
        // whether this CTA arrived last (the sum itself is shared by all
        // threads after the role loops).
        auto mark_last = [&]() {
            if (dr == 0 && lane == 0) {
                for (int sl = 0; sl < 2; ++sl) {
                    uint32_t last = 0u;
                    if (misc[2 + sl] != 0u) {
                        const PendTile &pt = pend[sl];
                        last = pend_prev[sl] == uint32_t(pt.cl - pt.cf) ? 1u : 0u;
                        if (last) p.tile_cnt[pt.tr.T] = 0u;
                    }
                    misc[4 + sl] = last;
                }
            }
        };

        UnitPos<kG> wd(ub, p);
        bool ok = true;
        for (int f = 0; f < nunits && ok; ++f) {
            const int set = f % DS;
            if (!warp_wait(dfull(set), (f / DS) & 1, ab)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int ng = wd.ng();
            const uint32_t dset = tmem + lane_base + kDcol0 + set * L::kDUnit;
            // accumulators [group][block][16]; group 1 only if the unit has it
            if constexpr (NBLK == 1) {
                uint32_t d[kUnitGroups][16];
                uint32_t d2[32];
                tmem_ld_32x32b_x32(dset, d2);
                tc_wait_ld_keep<32>(d2);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    d[0][j] = d2[j];
                    d[1][j] = d2[16 + j];
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(dempty(set, (f + DS) % kIssuers));
                // groups in ascending order, each scaled in fp32 (group size 32:
                // the weights carry their scales, the sums are added as they are)
                float s0 = 1.f, s1 = 1.f;
                if (!kFold) {
                    const int b = du % kSclSlots;
                    // once per stage (on an abort the values are never stored)
                    if (dj == 0) warp_wait(sfull(b), uint32_t(du / kSclSlots) & 1u, ab);
                    const uint32_t row0 = sst + uint32_t(b * kSclSlotBytes) + srow;
                    const uint32_t pitch = uint32_t(pr_sbox_w(wd.pi) * 2);
                    s0 = __half2float(__ushort_as_half(lds_u16(row0 + uint32_t(2 * dj) * pitch)));
                    if (ng > 1) s1 = __half2float(__ushort_as_half(lds_u16(row0 + uint32_t(2 * dj + 1) * pitch)));
                }
                // two lanes of fp32 per instruction (each lane rounds like fmaf)
#pragma unroll
                for (int j = 0; j < 16; j += 2) fma_f32x2(acc[0][j], acc[0][j + 1], s0, d[0][j], d[0][j + 1]);
                if (ng > 1) {
#pragma unroll
                    for (int j = 0; j < 16; j += 2) fma_f32x2(acc[0][j], acc[0][j + 1], s1, d[1][j], d[1][j + 1]);
                }
            } else {
                // 17..32 rows: one group (both 16-row blocks, 32 words) in
                // registers at a time beside the 32 sums; the second group is
                // read after the first is added in (same order per sum)
                float s0 = 1.f, s1 = 1.f;
                uint32_t dg[32];
                tmem_ld_32x32b_x32(dset, dg);
                if (!kFold) {
                    const int b = du % kSclSlots;
                    // once per stage (on an abort the values are never stored)
                    if (dj == 0) warp_wait(sfull(b), uint32_t(du / kSclSlots) & 1u, ab);
                    const uint32_t row0 = sst + uint32_t(b * kSclSlotBytes) + srow;
                    const uint32_t pitch = uint32_t(pr_sbox_w(wd.pi) * 2);
                    s0 = __half2float(__ushort_as_half(lds_u16(row0 + uint32_t(2 * dj) * pitch)));
                    if (ng > 1) s1 = __half2float(__ushort_as_half(lds_u16(row0 + uint32_t(2 * dj + 1) * pitch)));
                }
                tc_wait_ld_keep<32>(dg);
#pragma unroll
                for (int b = 0; b < NBLK; ++b)
#pragma unroll
                    for (int j = 0; j < 16; j += 2)
                        fma_f32x2(acc[b][j], acc[b][j + 1], s0, dg[16 * b + j], dg[16 * b + j + 1]);
                if (ng > 1) {
                    tmem_ld_32x32b_x32(dset + 32, dg);
                    tc_wait_ld_keep<32>(dg);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(dempty(set, (f + DS) % kIssuers));
                if (ng > 1) {
#pragma unroll
                    for (int b = 0; b < NBLK; ++b)
#pragma unroll
                        for (int j = 0; j < 16; j += 2)
                            fma_f32x2(acc[b][j], acc[b][j + 1], s1, dg[16 * b + j], dg[16 * b + j + 1]);
                }
            }
            if (++dj == dw.size()) {             // the stage's last unit: its scales are read
                if (!kFold) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(sempty(du % kSclSlots));
                }
                dw.next(dj);
                ++du;
                dj = 0;
            }
            const int t = wd.t, tpi = wd.pi;
            const bool tile_end = wd.tile_last();
            wd.next();
            if (tile_end || f == nunits - 1) {
                if (!flush(tpi, t)) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int b = 0; b < NBLK; ++b)
#pragma unroll
                    for (int j = 0; j < 16; ++j) acc[b][j] = 0.f;
            }
        }
        if (ok) mark_last();
    }

    __syncthreads();
    if (!kG && CL > 1) {
        // -------------------- cluster reduction: each CTA finishes 1/CL of the rows
        cluster_sync_all();                       // every CTA's partial is in its shared memory
        if (*ab.flag == 0u) {
            grid_dep_wait();                      // every thread that writes C waits itself
            const int t = cta / CLd;
            const int r0 = crank * kTileN / CLd, r1 = (crank + 1) * kTileN / CLd;
            const int nrows = r1 - r0;
            for (int item = threadIdx.x; item < nrows * 4 * NBLK; item += kThreads) {
                const int m4 = item / nrows, row = r0 + item % nrows;   // consecutive threads: consecutive rows
                const uint32_t off = base_s + uint32_t(row) * (16 * NBLK * 4) + uint32_t(m4) * 16;
                float4 v[kMaxCluster];
#pragma unroll
                for (int k = 0; k < kMaxCluster; ++k)
                    if (k < CL) v[k] = k == crank ? ld_shared_f32x4(off) : ld_cluster_f32x4(mapa_shared(off, uint32_t(k)));
                float4 sum = v[0];                 // ranks in order: the k range in order
#pragma unroll
                for (int k = 1; k < kMaxCluster; ++k)
                    if (k < CL) {
                        sum.x += v[k].x;
                        sum.y += v[k].y;
                        sum.z += v[k].z;
                        sum.w += v[k].w;
                    }
                const int n = t * kTileN + row;
                if (n < p.N) {
                    const float sv[4] = {sum.x, sum.y, sum.z, sum.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int m = 4 * m4 + i;
                        if (m < p.M) p.C[size_t(m) * p.N + n] = __float2half_rn(sv[i]);
                    }
                }
            }
        }
        // nobody leaves while another CTA reads its partial (nothing to
        // publish: a relaxed arrive, no memory barrier)
        asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\tbarrier.cluster.wait.aligned;" ::: "memory");
    }

    // ----------------------------- stream-K split-tile fix-up (all threads)
    if (CL == 0 && *ab.flag == 0u) {
        grid_dep_wait();                      // every thread that writes C waits itself
        constexpr int kPart = 16 * NBLK * kTileN;
        constexpr int kBatch = 8;                           // contributors loaded at once
        for (int sl = 0; sl < 2; ++sl) {
            if (!misc[4 + sl]) continue;
            const int t = int(misc[2 + sl]) - 1;
            const TileRef tr = pend[sl].tr;
            const long long t0u = tr.t0u;
            const int cf = pend[sl].cf;
            const int cl = pend[sl].cl;
            for (int e4 = threadIdx.x; e4 < kPart / 4; e4 += kThreads) {   // float4 of the [m][128] tile
                const int m = e4 / (kTileN / 4);
                const int n0 = t * kTileN + 4 * (e4 % (kTileN / 4));
                if (m >= p.M) continue;
                float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int c0 = cf; c0 <= cl; c0 += kBatch) {
                    float4 v[kBatch];
#pragma unroll
                    for (int u = 0; u < kBatch; ++u) {
                        const int cc = c0 + u;
                        v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                        if (cc <= cl) {
                            const int sl2 = split_begin(cc, p.U, p.P) >= t0u ? 0 : 1;
                            const float4 *src = reinterpret_cast<const float4 *>(
                                p.partial + (size_t(cc) * 2 + sl2) * kPart + size_t(m) * kTileN + (n0 - t * kTileN));
                            v[u] = __ldcg(src);
                        }
                    }
#pragma unroll
                    for (int u = 0; u < kBatch; ++u)
                        if (c0 + u <= cl) {
                            sum.x += v[u].x;
                            sum.y += v[u].y;
                            sum.z += v[u].z;
                            sum.w += v[u].w;
                        }
                }
                if (n0 < tr.N) {
                    const __half2 lo = __floats2half2_rn(sum.x, sum.y);
                    const __half2 hi = __floats2half2_rn(sum.z, sum.w);
                    uint2 packed;
                    packed.x = h2_as_u32(lo);
                    packed.y = h2_as_u32(hi);
                    *reinterpret_cast<uint2 *>(tr.C + size_t(m) * tr.N + n0) = packed;
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

// A stream-K fix-up (counter round trip plus one round of partial loads)
// costs about as much as this many units of work.
constexpr int kFixupUnits = 2;

// Cluster size for a shape: the largest c <= kMaxCluster, <= units per tile and
// <= SMs per tile whose clusters all fit one wave, or 0 for stream-K when
// that leaves each CTA more than kFixupUnits units beyond stream-K's share.
// It depends on the shape only (never on M), so every M <= 32 splits k the
// same way and sums the same partials in the same order (batch invariance).
int pick_cluster(int n_tiles, int n_pairs, int sm_count) {
    if (n_tiles * 2 > sm_count) return 0;
    const long long units = (long long)n_tiles * n_pairs;
    const long long streamk_share = (units + sm_count - 1) / sm_count;
    int root = 1;
    while ((root + 1) * (root + 1) <= n_pairs) ++root;
    if (root * (root + 1) < n_pairs) ++root;          // nearest integer to sqrt(n_pairs)
    int c = std::min(std::min(kMaxCluster, std::max(2, root)), std::min(n_pairs, sm_count / n_tiles));
    if ((n_pairs + c - 1) / c > streamk_share + kFixupUnits) return 0;
    for (; c >= 2; --c) {
        // one CTA per SM for either variant; the larger one's query bounds both
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(n_tiles * c);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = Layout<2>::bytes(Layout<2>::kStagesMax);
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = c;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int fit = 0;
        if (cudaOccupancyMaxActiveClusters(&fit, w4a16_decode_kernel<2, false, false>, &cfg) != cudaSuccess) {
            cudaGetLastError();
            continue;
        }
        if (fit >= n_tiles) return c;
    }
    return 0;
}

template <int NBLK, bool kFold, bool kG = false, bool kZ = false>
w4v_status configure() {
    static int configured_for = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_for != dev) {
        if (cudaFuncSetAttribute(w4a16_decode_kernel<NBLK, kFold, kG, kZ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kMaxSmem) != cudaSuccess) {
            cudaGetLastError();
            return W4V_ERR_CUDA;
        }
        configured_for = dev;
    }
    return W4V_OK;
}

template <int NBLK, bool kFold, bool kG = false, bool kZ = false>
w4v_status launch(const CUtensorMap &xmap, const CUtensorMap &smap, const CUtensorMap &zmap, Args &a, int cluster,
                  cudaStream_t stream) {
    using L = Layout<NBLK>;
    w4v_status st = configure<NBLK, kFold, kG, kZ>();
    if (st != W4V_OK) return st;
    a.cluster = cluster;
    a.stages = L::kStagesMax;
    if (cluster > 0) a.P = a.n_tiles * cluster;
    const size_t smem = size_t(L::bytes(a.stages));
    if (launch_pdl_cluster(w4a16_decode_kernel<NBLK, kFold, kG, kZ>, dim3(a.P), dim3(kThreads), smem, stream, cluster,
                           xmap, smap, zmap, a) !=
        cudaSuccess) {
        cudaGetLastError();
        return W4V_ERR_CUDA;
    }
    return W4V_OK;
}

// Cluster size per (device, tiles, units per tile), cached (the occupancy
// query needs both kernel variants configured).
int cluster_for(int n_tiles, int n_pairs, int sm_count) {
    struct Entry { int dev, n_tiles, n_pairs, cluster; };
    static Entry cache[64];
    static int n_cache = 0;
    static std::mutex mu;
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n_cache; ++i)
        if (cache[i].dev == dev && cache[i].n_tiles == n_tiles && cache[i].n_pairs == n_pairs) return cache[i].cluster;
    if (configure<1, false>() != W4V_OK || configure<2, false>() != W4V_OK) return 0;
    const int c = pick_cluster(n_tiles, n_pairs, sm_count);
    if (n_cache < 64) cache[n_cache++] = Entry{dev, n_tiles, n_pairs, c};
    return c;
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
                               const uint8_t *zeros, int group, uint16_t *C, int M, int N, int K,
                               void *ws, bool static_weights, cudaStream_t stream) {
    const DeviceInfo *info = nullptr;
    w4v_status st = device_info(&info);
    if (st != W4V_OK) return st;
    const int nblk = (M + 15) / 16;
    Args a;
    a.probs = nullptr;
    a.n_probs = 0;
    a.wq = static_cast<const uint8_t *>(Bq);
    a.scales = reinterpret_cast<const __half *>(scales);
    a.zeros = zeros;
    a.C = reinterpret_cast<__half *>(C);
    a.M = M;
    a.N = N;
    a.K = K;
    a.n_tiles = (N + kTileN - 1) / kTileN;
    a.n_groups = K / kGroup;
    a.n_pairs = (a.n_groups + kUnitGroups - 1) / kUnitGroups;
    a.U = (long long)a.n_tiles * a.n_pairs;
    a.P = static_cast<int>(std::min<long long>(std::min(info->sm_count, kMaxCtas), a.U));
    a.partial = static_cast<float *>(ws);
    a.tile_cnt = reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(ws) +
                                              size_t(kMaxCtas) * 2 * 16 * nblk * kTileN * sizeof(float));
    a.status = info->status;
    a.static_w = static_weights ? 1 : 0;
    CUtensorMap xmap;
    st = encode_tmap_kblocks(&xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, A, uint64_t(K), uint64_t(M), 64, 16 * nblk,
                             2 * kStageGroups, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != W4V_OK) return st;
    // scales [K/group][N]: one stage's rows (up to 4 groups) of one tile (up to 128 columns)
    a.sbox_w = std::min(kTileN, N);
    a.sbox_h = std::min(kStageGroups * (kGroup / group), K / group);
    CUtensorMap smap;
    st = encode_tmap_2d(&smap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, scales, uint64_t(N), uint64_t(K / group),
                        uint64_t(N) * 2, uint32_t(a.sbox_w), uint32_t(a.sbox_h), CU_TENSOR_MAP_SWIZZLE_NONE);
    if (st != W4V_OK) return st;
    // zero points [K/group][N] uint8, the same box (N is a multiple of 16)
    CUtensorMap zmap = {};
    if (zeros != nullptr) {
        st = encode_tmap_2d(&zmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, zeros, uint64_t(N), uint64_t(K / group), uint64_t(N),
                            uint32_t(a.sbox_w), uint32_t(a.sbox_h), CU_TENSOR_MAP_SWIZZLE_NONE);
        if (st != W4V_OK) return st;
    }
    const int cluster = cluster_for(a.n_tiles, a.n_pairs, info->sm_count);
    if (group == 32)
        return nblk == 1 ? launch<1, true>(xmap, smap, zmap, a, cluster, stream)
                         : launch<2, true>(xmap, smap, zmap, a, cluster, stream);
    if (zeros != nullptr)
        return nblk == 1 ? launch<1, false, false, true>(xmap, smap, zmap, a, cluster, stream)
                         : launch<2, false, false, true>(xmap, smap, zmap, a, cluster, stream);
    return nblk == 1 ? launch<1, false>(xmap, smap, zmap, a, cluster, stream)
                     : launch<2, false>(xmap, smap, zmap, a, cluster, stream);
}

// ---------------------------------------------------------------- grouped launch
namespace {

// FNV-1a over the handle fields a launch relies on, so that a handle not
// written by w4a16_grouped_plan (or changed since) is refused.
uint32_t handle_tag(const w4a16_grouped_t &h) {
    uint32_t x = 2166136261u;
    auto mix = [&](uint64_t v) {
        for (int i = 0; i < 8; ++i) {
            x ^= uint32_t(v >> (8 * i)) & 0xFFu;
            x *= 16777619u;
        }
    };
    mix(reinterpret_cast<uintptr_t>(h.plan));
    mix(uint64_t(h.units));
    mix(uint64_t(uint32_t(h.n_problems)));
    mix(uint64_t(uint32_t(h.M)));
    mix(uint64_t(uint32_t(h.group)));
    mix(uint64_t(uint32_t(h.has_zeros)));
    mix(uint64_t(uint32_t(h.tiles)));
    return x ^ 0x57344750u;
}

}  // namespace

size_t w4a16_grouped_table_bytes(int n_problems) { return size_t(n_problems) * sizeof(GroupProb); }

w4v_status build_w4a16_grouped(const w4a16_problem *probs, int n, int M, int group, void *plan,
                               w4a16_grouped_t *h, cudaStream_t stream) {
    const int nblk = (M + 15) / 16;
    std::vector<GroupProb> table(static_cast<size_t>(n));
    long long u0 = 0;
    int tile0 = 0;
    for (int i = 0; i < n; ++i) {
        const w4a16_problem &q = probs[i];
        GroupProb &g = table[size_t(i)];
        std::memset(&g, 0, sizeof(g));
        w4v_status st = encode_tmap_kblocks(&g.xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, q.A, uint64_t(q.K),
                                            uint64_t(M), 64, 16 * nblk, 2 * kStageGroups, CU_TENSOR_MAP_SWIZZLE_128B);
        if (st != W4V_OK) return st;
        g.sbox_w = std::min(kTileN, q.N);
        g.sbox_h = std::min(kStageGroups * (kGroup / group), q.K / group);
        st = encode_tmap_2d(&g.smap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, q.scales, uint64_t(q.N), uint64_t(q.K / group),
                            uint64_t(q.N) * 2, uint32_t(g.sbox_w), uint32_t(g.sbox_h), CU_TENSOR_MAP_SWIZZLE_NONE);
        if (st != W4V_OK) return st;
        if (q.zeros != nullptr) {
            st = encode_tmap_2d(&g.zmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, q.zeros, uint64_t(q.N), uint64_t(q.K / group),
                                uint64_t(q.N), uint32_t(g.sbox_w), uint32_t(g.sbox_h), CU_TENSOR_MAP_SWIZZLE_NONE);
            if (st != W4V_OK) return st;
        }
        g.wq = static_cast<const uint8_t *>(q.Bq);
        g.C = reinterpret_cast<__half *>(q.C);
        g.N = q.N;
        g.n_groups = q.K / kGroup;
        g.n_pairs = (g.n_groups + kUnitGroups - 1) / kUnitGroups;
        g.n_tiles = (q.N + kTileN - 1) / kTileN;
        g.u0 = u0;
        g.tile0 = tile0;
        u0 += (long long)g.n_tiles * g.n_pairs;
        tile0 += g.n_tiles;
    }
    // The table goes to the device once, synchronously: the handle then
    // describes device memory that no later host change can affect.
    if (cudaMemcpyAsync(plan, table.data(), table.size() * sizeof(GroupProb), cudaMemcpyHostToDevice, stream) !=
            cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess) {
        cudaGetLastError();
        return W4V_ERR_CUDA;
    }
    h->plan = plan;
    h->units = u0;
    h->n_problems = n;
    h->M = M;
    h->group = group;
    h->has_zeros = probs[0].zeros != nullptr ? 1 : 0;
    h->tiles = tile0;
    h->check = handle_tag(*h);
    return W4V_OK;
}

bool w4a16_grouped_handle_ok(const w4a16_grouped_t &h) {
    return h.plan != nullptr && h.check == handle_tag(h) && h.n_problems >= 1 && h.M >= 1 &&
           h.M <= kDecodeMaxRows && (h.group == 128 || h.group == 32) && h.units >= 1 && h.tiles >= 1;
}

size_t w4a16_grouped_ws_bytes(const w4a16_grouped_t &h) {
    const int nblk = (h.M + 15) / 16;
    const size_t part = size_t(kMaxCtas) * 2 * 16 * nblk * kTileN * sizeof(float);
    return part + ((size_t(h.tiles) * sizeof(uint32_t) + 255) & ~size_t(255));
}

w4v_status launch_w4a16_grouped(const w4a16_grouped_t &h, void *ws, bool static_weights, cudaStream_t stream) {
    const DeviceInfo *info = nullptr;
    w4v_status st = device_info(&info);
    if (st != W4V_OK) return st;
    const int nblk = (h.M + 15) / 16;
    Args a;
    std::memset(&a, 0, sizeof(a));
    a.probs = static_cast<const GroupProb *>(h.plan);
    a.n_probs = h.n_problems;
    // only tested against null inside the kernel: whether the problems carry zero points
    a.zeros = h.has_zeros ? static_cast<const uint8_t *>(h.plan) : nullptr;
    a.M = h.M;
    a.U = h.units;
    a.P = static_cast<int>(std::min<long long>(std::min(info->sm_count, kMaxCtas), a.U));
    a.partial = static_cast<float *>(ws);
    a.tile_cnt = reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(ws) +
                                              size_t(kMaxCtas) * 2 * 16 * nblk * kTileN * sizeof(float));
    a.status = info->status;
    a.static_w = static_weights ? 1 : 0;
    CUtensorMap unused;
    std::memset(&unused, 0, sizeof(unused));
    if (h.group == 32)
        return nblk == 1 ? launch<1, true, true>(unused, unused, unused, a, 0, stream)
                         : launch<2, true, true>(unused, unused, unused, a, 0, stream);
    if (h.has_zeros)
        return nblk == 1 ? launch<1, false, true, true>(unused, unused, unused, a, 0, stream)
                         : launch<2, false, true, true>(unused, unused, unused, a, 0, stream);
    return nblk == 1 ? launch<1, false, true>(unused, unused, unused, a, 0, stream)
                     : launch<2, false, true>(unused, unused, unused, a, 0, stream);
}

}  // namespace w4v
