/*
 * w4v.h -- C ABI of libw4v, the GB300 (sm_103a) speculative-decoding verify
 * step for a W4A16 target with an int8 lm_head.
 *
 * The operations follow the statement of the problem in "Efficient LLM
 * Challenge Results" (AdaptFM @ ICML 2026):
 *   - section 3 "Speculative decoding did the heavy lifting": a drafter
 *     proposes K tokens, the target runs all K+1 positions in one forward
 *     pass, and greedy verification keeps the longest draft prefix equal to
 *     the target's own tokens; drafts may be padded to a constant K with -1
 *     sentinels, which are never accepted (runner-up paragraph);
 *   - sections 3 and 5 "Quantization was common, but not the deciding lever":
 *     the target's projections are 4-bit W4A16 GPTQ with group size 128 and
 *     fp16 activations, and its untied lm_head is quantized to 8 bits;
 *   - section 2 "Where the time goes": decode is bound by reading the weights
 *     from HBM, so the K+1 positions share one weight read.
 * The pages give no interface; this one is the plainest that carries those
 * operations.
 *
 * Conventions (all entry points):
 *   - fp16 data is passed as uint16_t holding IEEE-754 binary16 bit patterns.
 *   - Matrices are dense row-major with the leading dimension equal to the
 *     row length given.  Device pointers must be 16-byte aligned.
 *   - The caller owns every buffer, including the workspace; no entry point
 *     allocates device memory.  A workspace must be zero-filled once before
 *     its first use; every call that returns W4V_OK leaves the parts that
 *     must start at zero (arrival counters, best-key slots) at zero again,
 *     so it can be reused by the next call on the same stream (scratch
 *     parts such as fp32 partial tiles keep whatever the last call wrote and
 *     are always written before they are read).
 *   - Calls are asynchronous on `stream` (NULL = legacy default stream).
 *     Argument, shape and alignment errors are returned before anything is
 *     launched.  A launch failure returns W4V_ERR_CUDA.  A kernel that gives
 *     up on an internal wait (bounded at about two seconds) records
 *     W4V_ERR_TIMEOUT in a device status word read by w4v_get_status(); after
 *     that the workspace must be zero-filled again.
 *   - Nothing here is thread-safe against concurrent use of the same
 *     workspace; distinct workspaces may be used concurrently.
 */
#ifndef W4V_H
#define W4V_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
/* A cudaStream_t. */
typedef struct CUstream_st *w4v_stream_t;

typedef enum {
    W4V_OK = 0,
    W4V_ERR_ARG = 1,        /* null pointer or invalid enum/flag            */
    W4V_ERR_SHAPE = 2,      /* unsupported sizes (see each entry point)     */
    W4V_ERR_ALIGN = 3,      /* pointer not 16-byte aligned                  */
    W4V_ERR_WORKSPACE = 4,  /* workspace missing or smaller than required   */
    W4V_ERR_ARCH = 5,       /* current device is not sm_103 (GB300)         */
    W4V_ERR_CUDA = 6,       /* CUDA runtime / launch error                  */
    W4V_ERR_TIMEOUT = 7     /* a kernel abandoned a bounded wait            */
} w4v_status;

/* Short English text for a status code (static storage, never NULL). */
const char *w4v_status_string(w4v_status status);

/* Checks that the current device is compute capability 10.3 and runs one
 * tiny kernel, so that a library built for another architecture fails here
 * rather than at the first real launch ("DFlash K=15 for Qwen3.5-4B on a
 * single A10G", section "What transfers": build for the card you run on).
 * Idempotent per device; every entry point calls it implicitly.  What it
 * finds (the SM count, the device status word's address) is kept per device
 * for the life of the process, so a process that resets a device
 * (cudaDeviceReset) must be restarted before it calls the library again. */
w4v_status w4v_init(void);

/* Synchronizes `stream`, then returns and clears the device status word of
 * the current device: W4V_OK, or W4V_ERR_TIMEOUT if a kernel gave up a wait
 * since the last call. */
w4v_status w4v_get_status(w4v_stream_t stream);

/* ------------------------------------------------------- int4 weight packing
 * The logical W4A16 weight is q[N][K], one 4-bit code (0..15) per byte, with
 * w[n][k] = s[k/G][n] * (q[n][k] - z) (z = 8, or a per-group zero table).
 * The device format is this library's own tile layout: N is split into tiles
 * of 128 rows (the last one zero-padded), K into groups of 128; every
 * (tile, group) block is 8192 contiguous bytes, blocks ordered tile-major.
 * Inside a block, 16-byte chunk j (j = 0..3, k = 32j..32j+31 of the group)
 * of row r sits at byte (j*128 + r)*16 and holds four little-endian 32-bit
 * words; word w covers k = 32j+8w .. +7 with nibble i holding the code of
 * k offset {0,2,4,6,1,3,5,7}[i].
 * Sizes: K % 128 == 0, N % 8 == 0, N, K > 0.  Host memory only. */
size_t w4v_packed_bytes(int N, int K);
w4v_status w4v_pack_int4(const uint8_t *q_host, int N, int K, void *packed_host_out);
/* Inverse of w4v_pack_int4 (rows >= N of the padded tile are dropped). */
w4v_status w4v_unpack_int4(const void *packed_host, int N, int K, uint8_t *q_host_out);

/* ------------------------------------------------------------- w4a16_gemm
 * C[M][N] = A[M][K] * W^T, W[n][k] = scales[k/G][n] * (q[n][k] - z[k/G][n]),
 * z = 8 when zeros == NULL (symmetric GPTQ) else the uint8 table
 * zeros[K/G][N] (values 0..15, AWQ style).  A, scales, C are fp16; products
 * are accumulated in fp32.  For M <= 32 (verify sizes, HBM-bound) with
 * G = 128 each group's fp32 sum is multiplied by its scale in fp32; for
 * M > 32 (prefill, tensor-bound), and for G = 32 at any M, the dequantized
 * weight s*(q-z) is rounded to fp16 once.  The whole K is accumulated in
 * fp32, and for M <= 32 the per-element arithmetic does not depend on M.
 * C is rounded to fp16 (round to nearest even).  G = 128 is the GPTQ
 * target of "Efficient LLM Challenge Results" sections 3 and 5; G = 32 is
 * the group size of the compressed-tensors W4A16 target listed there.
 *   A        device, fp16 [M][K]
 *   Bq       device, packed int4 from w4v_pack_int4 (w4v_packed_bytes(N,K);
 *            the packed layout does not depend on G)
 *   scales   device, fp16 [K/G][N]
 *   zeros    device, uint8 [K/G][N] or NULL (requires N % 16 == 0)
 *   group    G: 128 or 32
 *   C        device, fp16 [M][N] (written, never read)
 * Sizes: M >= 0 (M == 0 is a no-op), N % 8 == 0, K % 128 == 0.
 * Workspace: w4a16_workspace_bytes(M, N, K) bytes, zero-filled before first
 * use: fp32 partial sums of output tiles whose k range is split between
 * CTAs, and one arrival counter per tile.  About 1 MB for M <= 16 and 2 MB
 * for M <= 32; for M > 32, the larger of the 32-row size and 256 KB per
 * 128 x 256 output tile when there are at most 1024 tiles (the prefill
 * kernel may then split tiles in two k halves), plus 4 bytes per tile. */
size_t w4a16_workspace_bytes(int M, int N, int K);
w4v_status w4a16_gemm(const uint16_t *A, const void *Bq, const uint16_t *scales,
                      const uint8_t *zeros, int group, uint16_t *C, int M, int N, int K,
                      void *workspace, size_t workspace_bytes, w4v_stream_t stream);

/* w4a16_gemm with flags (w4a16_gemm is w4a16_gemm_ex with flags == 0).
 *   W4V_STATIC_WEIGHTS: Bq, scales and zeros are not written by any GPU
 *     work that may still be running when this call's kernel starts (the
 *     weights of a model during inference).  The verify-sized kernel then
 *     loads and dequantizes its first weight stages while the previous
 *     kernel of the stream is still finishing; A is still read, and C and
 *     the workspace still written, only after that kernel has completed.
 *     Without the flag the weights are only prefetched into L2 early.  The
 *     pages have no counterpart: it is a scheduling promise of the caller,
 *     the result is the same either way.
 *   W4V_BATCH_INVARIANT: for M > 32, run the rows in blocks of 32 through
 *     the verify-sized kernel (one launch per block, the weights read once
 *     per block) instead of the prefill kernel, so that every row of C is
 *     bit for bit the row a call with that row alone would give.  Greedy
 *     speculative decoding then emits exactly the tokens of plain greedy
 *     decoding also when several sequences' verify blocks share one call
 *     ("Efficient LLM Challenge Results", section 3: verification leaves the
 *     output unchanged whatever the drafts).  No effect for M <= 32, which
 *     is batch-invariant anyway.
 * Unknown flag bits: W4V_ERR_ARG. */
#define W4V_STATIC_WEIGHTS 1u
#define W4V_BATCH_INVARIANT 2u
w4v_status w4a16_gemm_ex(const uint16_t *A, const void *Bq, const uint16_t *scales,
                         const uint8_t *zeros, int group, uint16_t *C, int M, int N, int K,
                         void *workspace, size_t workspace_bytes, unsigned flags, w4v_stream_t stream);

/* ----------------------------------------------------- w4a16_gemm_grouped
 * Several independent W4A16 products C_i = A_i * W_i^T (each exactly as
 * w4a16_gemm defines it) in one launch.  Decode and verify read every weight
 * from HBM once per step ("Efficient LLM Challenge Results", section 2
 * "Where the time goes"), and a decoder layer's projections are a few MB
 * each: one launch per projection pays a start-up and a drain of the weight
 * stream that are comparable to its transfer time.  A grouped launch streams
 * the weights of every problem through one pipeline, with one start-up.
 * All problems share M (1..32, the verify-sized kernel), the group size and
 * whether they carry zero points.  Each output element is computed by the
 * same arithmetic for every M in 1..32 (batch invariance), but a grouped
 * launch splits the k ranges differently from a one-problem launch, so its
 * results may differ from w4a16_gemm in the last fp32 bits before the fp16
 * rounding; both are within the same error bound of the exact product.
 *
 * Use: w4a16_grouped_plan once for a fixed set of buffers (it encodes the
 * problems into `plan`, device memory of w4a16_grouped_plan_bytes(n) bytes,
 * 64-byte aligned, and fills the host handle), then w4a16_gemm_grouped per
 * step.  The plan holds the buffers' addresses: it stays valid while they
 * do, and must be rebuilt if any of them moves.
 *   problems[i].A       device, fp16 [M][K_i]
 *   problems[i].Bq      device, packed int4 of q_i [N_i][K_i] (w4v_pack_int4)
 *   problems[i].scales  device, fp16 [K_i/G][N_i]
 *   problems[i].zeros   device, uint8 [K_i/G][N_i] or NULL (all NULL or none;
 *                       with zero points N_i % 16 == 0)
 *   problems[i].C       device, fp16 [M][N_i] (written, never read)
 * Sizes: 1 <= n_problems <= 4096, 1 <= M <= 32, G = 128 or 32,
 * N_i % 8 == 0, K_i % 128 == 0, N_i, K_i > 0.
 * w4a16_grouped_plan copies the table to the device and waits for the copy
 * (it synchronizes `stream`), so it must not be called while `stream` is
 * being captured into a graph (W4V_ERR_ARG); w4a16_gemm_grouped only
 * launches and may be captured.  A handle not written by w4a16_grouped_plan,
 * or changed since, is refused with W4V_ERR_ARG.
 * Workspace: w4a16_grouped_workspace_bytes(handle) bytes, zero-filled before
 * first use (fp32 partial tiles and one arrival counter per output tile).
 * Flags: W4V_STATIC_WEIGHTS as for w4a16_gemm_ex. */
typedef struct {
    const uint16_t *A;
    const void *Bq;
    const uint16_t *scales;
    const uint8_t *zeros;
    uint16_t *C;
    int N, K;
} w4a16_problem;

/* Filled by w4a16_grouped_plan; read-only for the caller. */
typedef struct {
    const void *plan;       /* the device table this handle describes */
    long long units;        /* work units of one launch */
    int n_problems, M, group, has_zeros, tiles;
    unsigned check;         /* consistency tag */
} w4a16_grouped_t;

size_t w4a16_grouped_plan_bytes(int n_problems);
w4v_status w4a16_grouped_plan(const w4a16_problem *problems, int n_problems, int M, int group, void *plan,
                              size_t plan_bytes, w4a16_grouped_t *handle, w4v_stream_t stream);
size_t w4a16_grouped_workspace_bytes(const w4a16_grouped_t *handle);
w4v_status w4a16_gemm_grouped(const w4a16_grouped_t *handle, void *workspace, size_t workspace_bytes,
                              unsigned flags, w4v_stream_t stream);

/* ------------------------------------------------------- w8_lmhead_argmax
 * Greedy token per row: argmax_out[r] = argmax_v scale[v] * sum_k X[r][k]*W[v][k],
 * int8 weights, one fp16 scale per vocabulary row, fp32 accumulation with
 * the scale applied to the finished sum.  Ties go to the lowest v; a NaN
 * logit counts as -inf; -0 equals +0.  Full logits are never written unless
 * logits_debug is given.
 *   X              device, fp16 [M][K]
 *   W              device, int8 [V][K]
 *   scale          device, fp16 [V]
 *   argmax_out     device, int32 [M]
 *   maxlogit       device, float [M] or NULL: the winning logit
 *   logits_debug   device, float [M][V] or NULL: every logit (testing aid)
 * Sizes: 0 <= M <= 128, K % 128 == 0, V % 8 == 0, V > 0.
 * Workspace: w8_lmhead_argmax_workspace_bytes(M, V) bytes, zero-filled
 * before first use (one best key per row and an arrival counter). */
size_t w8_lmhead_argmax_workspace_bytes(int M, int V);
w4v_status w8_lmhead_argmax(const uint16_t *X, const int8_t *W, const uint16_t *scale,
                            int M, int K, int V, int32_t *argmax_out, float *maxlogit,
                            float *logits_debug, void *workspace, size_t workspace_bytes,
                            w4v_stream_t stream);

/* w8_lmhead_argmax with flags (w8_lmhead_argmax is this with flags == 0).
 *   W4V_BATCH_INVARIANT: for M > 32, run the rows in blocks of 32 (one launch
 *     each, the weights read once per block), so that every row's logits and
 *     token are bit for bit those of a call with that row alone.  Up to 32
 *     rows every logit comes from the same arithmetic whatever M is; a
 *     single launch over more rows sums each logit in another order (within
 *     the same fp32 error bound), which may flip a token between two logits
 *     that close.  Several sequences' verify blocks in one call then accept
 *     exactly the tokens each would accept alone ("Efficient LLM Challenge
 *     Results", section 3: greedy verification leaves the output unchanged).
 * Unknown flag bits: W4V_ERR_ARG.  Other arguments as w8_lmhead_argmax. */
w4v_status w8_lmhead_argmax_ex(const uint16_t *X, const int8_t *W, const uint16_t *scale,
                               int M, int K, int V, int32_t *argmax_out, float *maxlogit,
                               float *logits_debug, void *workspace, size_t workspace_bytes,
                               unsigned flags, w4v_stream_t stream);

/* ---------------------------------------------- w8_lmhead_argmax_noalloc
 * The paper has no counterpart to this entry point; it exists for callers
 * that cannot allocate device memory for a workspace -- for example a plugin
 * running inside another inference engine whose execute step may not
 * allocate, or a serving loop whose device memory is already handed out by
 * its own allocator (cudaMalloc would also synchronize the device in the
 * middle of a decode step).  It computes exactly what w8_lmhead_argmax
 * computes, with the same arguments minus the workspace: the scratch lives
 * in a 4 KB device array inside this library, which every GPU that loads the
 * library keeps until the process exits.
 *   - Allocates nothing: no cudaMalloc, no cudaFree, no allocating library
 *     call.  It clears the scratch with an asynchronous memset on `stream`
 *     before each launch.  That memset sits between the previous kernel on
 *     the stream and the lm_head, so the lm_head's programmatic launch no
 *     longer overlaps its set-up with the previous kernel's end (the
 *     workspace entry keeps that overlap; the kernel itself leaves the
 *     scratch cleared on success, and the memset covers a call that gave
 *     up a bounded wait).
 *   - The first call on a device looks up that device's address of the
 *     array (cudaGetSymbolAddress with the device current) and keeps it for
 *     the life of the process; make that first call outside any stream
 *     capture.  After cudaDeviceReset (or anything else that unloads the
 *     library's module from a device) the kept address is stale: restart
 *     the process before calling this entry point again, as for the
 *     library's other per-device state (w4v_init).
 *   - Every call on a device shares the one array: calls that overlap on the
 *     GPU (different streams without ordering between them) race and give
 *     wrong tokens.  Serialize them, or use w8_lmhead_argmax with a
 *     workspace per stream.
 *   - Sizes: 0 <= M <= 128 (the array holds the keys of at most 128 rows);
 *     larger M returns W4V_ERR_SHAPE.  Other sizes as w8_lmhead_argmax. */
w4v_status w8_lmhead_argmax_noalloc(const uint16_t *X, const int8_t *W, const uint16_t *scale,
                                    int M, int K, int V, int32_t *argmax_out, float *maxlogit,
                                    float *logits_debug, w4v_stream_t stream);

/* ----------------------------------------------------------- spec_accept
 * Longest-prefix greedy acceptance for B sequences:
 *   n[b] = the largest j <= K with draft[b][i] == target[b][i] for all i < j,
 * where a negative draft (the -1 padding sentinel) never matches.  The
 * emitted tokens are target[b][0..n[b]] (= drafts 0..n-1 then the target's
 * own next token); out_tokens[b][j] = target[b][j] for j <= n[b], else -1.
 *   target      device, int32 [B][K+1]: the target's greedy token after
 *               each verify position (row b*(K+1)+j of the verify block)
 *   draft       device, int32 [B][K] (may be NULL when K == 0)
 *   n_accepted  device, int32 [B]
 *   out_tokens  device, int32 [B][K+1] or NULL
 * Sizes: B >= 0 (0 is a no-op), 0 <= K <= 1024. */
w4v_status spec_accept(const int32_t *target, const int32_t *draft, int B, int K,
                       int32_t *n_accepted, int32_t *out_tokens, w4v_stream_t stream);

/* ----------------------------------------------- w8_lmhead_argmax_accept
 * The last two operations of a verify step in one launch: the int8 lm_head
 * argmax of w8_lmhead_argmax over M = B*(n_draft+1) rows, then the greedy
 * acceptance of spec_accept with target = those tokens viewed as
 * [B][n_draft+1] (row b*(n_draft+1)+j is position j of verify block b).
 * Results are identical to w8_lmhead_argmax followed by spec_accept; the
 * acceptance runs in the lm_head's last CTA, on the tokens it has just
 * written, so no second launch or dependency is needed.
 *   X, W, scale, argmax_out, maxlogit, workspace: as w8_lmhead_argmax
 *   draft       device, int32 [B][n_draft] (may be NULL when n_draft == 0)
 *   n_accepted  device, int32 [B]
 *   out_tokens  device, int32 [B][n_draft+1] or NULL (as spec_accept)
 * Sizes: B >= 0 (0 is a no-op), n_draft >= 0, B*(n_draft+1) <= 128,
 * K % 128 == 0, V % 8 == 0, V > 0.  Workspace: w8_lmhead_argmax_workspace_bytes
 * for M = B*(n_draft+1). */
w4v_status w8_lmhead_argmax_accept(const uint16_t *X, const int8_t *W, const uint16_t *scale,
                                   int B, int n_draft, int K, int V, const int32_t *draft,
                                   int32_t *argmax_out, int32_t *n_accepted, int32_t *out_tokens,
                                   float *maxlogit, void *workspace, size_t workspace_bytes,
                                   w4v_stream_t stream);

/* w8_lmhead_argmax_accept with flags (the plain entry point is this with
 * flags == 0).  W4V_BATCH_INVARIANT: for M = B*(n_draft+1) > 32, the argmax
 * runs as in w8_lmhead_argmax_ex with that flag (blocks of 32 rows) and the
 * acceptance follows in one more launch; the results are those of
 * w8_lmhead_argmax_ex followed by spec_accept.  Unknown flag bits:
 * W4V_ERR_ARG. */
w4v_status w8_lmhead_argmax_accept_ex(const uint16_t *X, const int8_t *W, const uint16_t *scale,
                                      int B, int n_draft, int K, int V, const int32_t *draft,
                                      int32_t *argmax_out, int32_t *n_accepted, int32_t *out_tokens,
                                      float *maxlogit, void *workspace, size_t workspace_bytes,
                                      unsigned flags, w4v_stream_t stream);

/* ------------------------------------------------------------ ngram_draft
 * Model-free drafts by prompt lookup ("Efficient LLM Challenge Results",
 * section 3, table of drafting methods: n-gram / prompt-lookup drafting
 * copies spans from the prompt; the runner-up pads drafts to a constant K
 * with -1).  For row b of `context`, c[0..L-1] with L = lengths[b] (values
 * outside [0, ld] are clamped to it): for n from n_max down to n_min, the
 * n-gram is c[L-n..L-1]; its latest earlier occurrence is the largest p with
 * p + n <= L - 1 and c[p+i] == c[L-n+i] for i < n.  The first n with an
 * occurrence gives drafts[b][i] = c[p+n+i] while p+n+i < L, else -1, and
 * match_len[b] = n; with none, every draft is -1 and match_len[b] = 0.
 *   context    device, int32 [B][ld] (tokens past a row's length are ignored)
 *   lengths    device, int32 [B]
 *   drafts     device, int32 [B][K] (may be NULL when K == 0)
 *   match_len  device, int32 [B] or NULL
 * Sizes: 0 <= B <= 65535 (0 is a no-op), ld >= 1, 1 <= n_min <= n_max <= 64,
 * 0 <= K <= 1024.  Workspace: ngram_draft_workspace_bytes(B) bytes,
 * zero-filled before first use (one best key and one arrival counter per
 * row). */
size_t ngram_draft_workspace_bytes(int B);
w4v_status ngram_draft(const int32_t *context, const int32_t *lengths, int B, int ld, int n_min,
                       int n_max, int K, int32_t *drafts, int32_t *match_len,
                       void *workspace, size_t workspace_bytes, w4v_stream_t stream);

/* --------------------------------------------------- gdn_verify / gdn_commit
 * The Gated DeltaNet recurrent state across a verify block, rolled back
 * under rejection.  Most of the target's layers are Gated DeltaNet, and a
 * rejected draft must not leave its update in their state ("Efficient LLM
 * Challenge Results", section 3, runner-up paragraph; "DFlash K=15 for
 * Qwen3.5-4B on a single A10G", "What transfers").  Per sequence b and head
 * h, with the recurrence of the first page's reference [12]:
 *     S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
 *     o_t = S_t q_t,
 * S the state [dv][dk] (row i = value index, column j = key index).
 * gdn_verify runs the T positions of a verify block from the committed state
 * and writes o_t for every t; it never writes the state.  gdn_commit then
 * advances the committed state in place by positions 0..n_accepted[b] of the
 * block (the last context token and the accepted drafts; n is clamped to
 * [0, T-1]), so the rejected positions leave no trace.  Keys and queries are
 * used as given (Gated DeltaNet normalises them to unit length upstream).
 *   state       device, fp32 [B][H][dv][dk] (read by gdn_verify, read and
 *               written by gdn_commit)
 *   q, k        device, fp16 [B][T][H][dk]  (gdn_commit takes no q)
 *   v           device, fp16 [B][T][H][dv]
 *   alpha, beta device, fp32 [B][T][H]
 *   o           device, fp16 [B][T][H][dv] (written; fp32 arithmetic inside)
 *   n_accepted  device, int32 [B] (as written by spec_accept or
 *               w8_lmhead_argmax_accept)
 * Sizes: 0 <= B <= 65535 (0 is a no-op), 1 <= T <= 64, 1 <= H <= 65535,
 * dk == 128, dv a multiple of 32 up to 4096.  No workspace. */
w4v_status gdn_verify(const float *state, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                      const float *alpha, const float *beta, int B, int T, int H, int dk, int dv,
                      uint16_t *o, w4v_stream_t stream);
w4v_status gdn_commit(float *state, const uint16_t *k, const uint16_t *v, const float *alpha,
                      const float *beta, const int32_t *n_accepted, int B, int T, int H, int dk,
                      int dv, w4v_stream_t stream);

/* gdn_step: the commit of the previous block and the verify of the next one
 * in one launch, reading and writing the state once: the state is advanced
 * by positions 0..n_prev[b] of the previous block (k_prev, v_prev,
 * alpha_prev, beta_prev over T_prev positions; n clamped as in gdn_commit)
 * and written back, then o_t of the current block is produced from it, with
 * the same arithmetic as gdn_commit followed by gdn_verify (bit for bit).
 * T_prev = 0 means no previous block (the *_prev pointers and n_prev are
 * then ignored and the state is not written).  Arrays, layouts and limits as
 * above, 0 <= T_prev <= 64. */
w4v_status gdn_step(float *state, const uint16_t *k_prev, const uint16_t *v_prev,
                    const float *alpha_prev, const float *beta_prev, const int32_t *n_prev, int T_prev,
                    const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *alpha,
                    const float *beta, int B, int T, int H, int dk, int dv, uint16_t *o,
                    w4v_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* W4V_H */
