// api.cpp -- the C ABI: argument validation (before anything touches the
// GPU), workspace sizing, the host int4 packer, and dispatch to launchers.
#include <algorithm>
#include <cstring>

#include "runtime.h"

namespace {

constexpr int kGroup = 128;
constexpr int kTile = 128;
constexpr int kBlockBytes = kTile * kGroup / 2;
// Nibble i of a packed word holds the code of k offset kNibbleK[i].
constexpr int kNibbleK[8] = {0, 2, 4, 6, 1, 3, 5, 7};

inline size_t packed_offset(int t, int g, int n_groups, int r, int j) {
    return (size_t(t) * n_groups + g) * kBlockBytes + (size_t(j) * kTile + r) * 16;
}

bool pack_shape_ok(int N, int K) { return N > 0 && K > 0 && K % kGroup == 0 && N % 8 == 0; }

}  // namespace

extern "C" {

const char *w4v_status_string(w4v_status s) {
    switch (s) {
        case W4V_OK: return "ok";
        case W4V_ERR_ARG: return "invalid argument (null pointer or bad flag)";
        case W4V_ERR_SHAPE: return "unsupported shape";
        case W4V_ERR_ALIGN: return "pointer not 16-byte aligned";
        case W4V_ERR_WORKSPACE: return "workspace missing or too small";
        case W4V_ERR_ARCH: return "current device is not sm_103 (GB300) or the library was built for another GPU";
        case W4V_ERR_CUDA: return "CUDA runtime or launch error";
        case W4V_ERR_TIMEOUT: return "a kernel abandoned a bounded wait";
    }
    return "unknown status";
}

size_t w4v_packed_bytes(int N, int K) {
    if (!pack_shape_ok(N, K)) return 0;
    const size_t tiles = (size_t(N) + kTile - 1) / kTile;
    return tiles * size_t(K / kGroup) * kBlockBytes;
}

w4v_status w4v_pack_int4(const uint8_t *q, int N, int K, void *out) {
    if (q == nullptr || out == nullptr) return W4V_ERR_ARG;
    if (!pack_shape_ok(N, K)) return W4V_ERR_SHAPE;
    const int n_groups = K / kGroup;
    const int n_tiles = (N + kTile - 1) / kTile;
    uint8_t *o = static_cast<uint8_t *>(out);
    for (int t = 0; t < n_tiles; ++t)
        for (int g = 0; g < n_groups; ++g)
            for (int r = 0; r < kTile; ++r) {
                const int n = t * kTile + r;
                for (int j = 0; j < 4; ++j) {
                    uint8_t *chunk = o + packed_offset(t, g, n_groups, r, j);
                    for (int w = 0; w < 4; ++w) {
                        const int k0 = g * kGroup + 32 * j + 8 * w;
                        uint32_t word = 0;
                        for (int i = 0; i < 8; ++i) {
                            const uint32_t code = n < N ? (q[size_t(n) * K + k0 + kNibbleK[i]] & 15u) : 8u;
                            word |= code << (4 * i);
                        }
                        for (int b = 0; b < 4; ++b) chunk[4 * w + b] = uint8_t(word >> (8 * b));
                    }
                }
            }
    return W4V_OK;
}

w4v_status w4v_unpack_int4(const void *packed, int N, int K, uint8_t *q) {
    if (q == nullptr || packed == nullptr) return W4V_ERR_ARG;
    if (!pack_shape_ok(N, K)) return W4V_ERR_SHAPE;
    const int n_groups = K / kGroup;
    const uint8_t *p = static_cast<const uint8_t *>(packed);
    for (int n = 0; n < N; ++n) {
        const int t = n / kTile, r = n % kTile;
        for (int g = 0; g < n_groups; ++g)
            for (int j = 0; j < 4; ++j) {
                const uint8_t *chunk = p + packed_offset(t, g, n_groups, r, j);
                for (int w = 0; w < 4; ++w) {
                    uint32_t word = 0;
                    for (int b = 0; b < 4; ++b) word |= uint32_t(chunk[4 * w + b]) << (8 * b);
                    const int k0 = g * kGroup + 32 * j + 8 * w;
                    for (int i = 0; i < 8; ++i) q[size_t(n) * K + k0 + kNibbleK[i]] = uint8_t((word >> (4 * i)) & 15u);
                }
            }
    }
    return W4V_OK;
}

size_t w4a16_workspace_bytes(int M, int N, int K) {
    if (M < 0 || !pack_shape_ok(N, K)) return 0;
    // M > 32: enough for the prefill kernel and for the 32-row blocks of
    // the batch-invariant path, whichever the call takes
    if (M > w4v::kDecodeMaxRows)
        return std::max(w4v::w4a16_prefill_ws_bytes(M, N, K), w4v::w4a16_decode_ws_bytes(w4v::kDecodeMaxRows, N, K));
    return w4v::w4a16_decode_ws_bytes(M, N, K);
}

w4v_status w4a16_gemm(const uint16_t *A, const void *Bq, const uint16_t *scales, const uint8_t *zeros, int group,
                      uint16_t *C, int M, int N, int K, void *ws, size_t ws_bytes, w4v_stream_t stream) {
    return w4a16_gemm_ex(A, Bq, scales, zeros, group, C, M, N, K, ws, ws_bytes, 0u, stream);
}

w4v_status w4a16_gemm_ex(const uint16_t *A, const void *Bq, const uint16_t *scales, const uint8_t *zeros,
                         int group, uint16_t *C, int M, int N, int K, void *ws, size_t ws_bytes, unsigned flags,
                         w4v_stream_t stream) {
    if ((flags & ~unsigned(W4V_STATIC_WEIGHTS | W4V_BATCH_INVARIANT)) != 0u) return W4V_ERR_ARG;
    if (M < 0 || N <= 0 || K <= 0) return W4V_ERR_SHAPE;
    if (group != kGroup && group != 32) return W4V_ERR_SHAPE;
    if (K % kGroup != 0 || N % 8 != 0) return W4V_ERR_SHAPE;
    if (zeros != nullptr && N % 16 != 0) return W4V_ERR_SHAPE;
    if (M == 0) return W4V_OK;
    if (A == nullptr || Bq == nullptr || scales == nullptr || C == nullptr) return W4V_ERR_ARG;
    if (!w4v::aligned16(A) || !w4v::aligned16(Bq) || !w4v::aligned16(scales) ||
        (zeros != nullptr && !w4v::aligned16(zeros)))
        return W4V_ERR_ALIGN;
    if (ws == nullptr || ws_bytes < w4a16_workspace_bytes(M, N, K)) return W4V_ERR_WORKSPACE;
    if (!w4v::aligned16(ws)) return W4V_ERR_ALIGN;
    const bool static_w = (flags & W4V_STATIC_WEIGHTS) != 0u;
    if (M > w4v::kDecodeMaxRows && (flags & W4V_BATCH_INVARIANT) != 0u) {
        // Blocks of 32 rows through the verify-sized kernel, in order on the
        // stream (each leaves the workspace zeroed for the next): every row
        // gets the arithmetic it gets in a call of 1..32 rows.
        for (int m0 = 0; m0 < M; m0 += w4v::kDecodeMaxRows) {
            const int mb = std::min(w4v::kDecodeMaxRows, M - m0);
            const w4v_status st = w4v::launch_w4a16_decode(A + size_t(m0) * K, Bq, scales, zeros, group,
                                                           C + size_t(m0) * N, mb, N, K, ws, static_w,
                                                           reinterpret_cast<cudaStream_t>(stream));
            if (st != W4V_OK) return st;
        }
        return W4V_OK;
    }
    if (M > w4v::kDecodeMaxRows)
        return w4v::launch_w4a16_prefill(A, Bq, scales, zeros, group, C, M, N, K, ws,
                                         reinterpret_cast<cudaStream_t>(stream));
    return w4v::launch_w4a16_decode(A, Bq, scales, zeros, group, C, M, N, K, ws, static_w,
                                    reinterpret_cast<cudaStream_t>(stream));
}

size_t w4a16_grouped_plan_bytes(int n_problems) {
    if (n_problems < 1 || n_problems > w4v::kGroupedMaxProblems) return 0;
    return w4v::w4a16_grouped_table_bytes(n_problems);
}

w4v_status w4a16_grouped_plan(const w4a16_problem *problems, int n, int M, int group, void *plan,
                              size_t plan_bytes, w4a16_grouped_t *handle, w4v_stream_t stream) {
    if (n < 1 || n > w4v::kGroupedMaxProblems || M < 1 || M > w4v::kDecodeMaxRows) return W4V_ERR_SHAPE;
    if (group != kGroup && group != 32) return W4V_ERR_SHAPE;
    if (problems == nullptr || plan == nullptr || handle == nullptr) return W4V_ERR_ARG;
    const bool zeros = problems[0].zeros != nullptr;
    for (int i = 0; i < n; ++i) {
        const w4a16_problem &q = problems[i];
        if (q.N <= 0 || q.K <= 0 || q.K % kGroup != 0 || q.N % 8 != 0) return W4V_ERR_SHAPE;
        if (zeros && q.N % 16 != 0) return W4V_ERR_SHAPE;
        if ((q.zeros != nullptr) != zeros) return W4V_ERR_ARG;
        if (q.A == nullptr || q.Bq == nullptr || q.scales == nullptr || q.C == nullptr) return W4V_ERR_ARG;
        if (!w4v::aligned16(q.A) || !w4v::aligned16(q.Bq) || !w4v::aligned16(q.scales) ||
            (q.zeros != nullptr && !w4v::aligned16(q.zeros)) || !w4v::aligned16(q.C))
            return W4V_ERR_ALIGN;
    }
    if (plan_bytes < w4v::w4a16_grouped_table_bytes(n)) return W4V_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(plan) & 63u) return W4V_ERR_ALIGN;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(reinterpret_cast<cudaStream_t>(stream), &cap) != cudaSuccess) {
        cudaGetLastError();
        return W4V_ERR_CUDA;
    }
    if (cap != cudaStreamCaptureStatusNone) return W4V_ERR_ARG;
    const w4v::DeviceInfo *info = nullptr;
    w4v_status st = w4v::device_info(&info);
    if (st != W4V_OK) return st;
    return w4v::build_w4a16_grouped(problems, n, M, group, plan, handle, reinterpret_cast<cudaStream_t>(stream));
}

size_t w4a16_grouped_workspace_bytes(const w4a16_grouped_t *handle) {
    if (handle == nullptr || !w4v::w4a16_grouped_handle_ok(*handle)) return 0;
    return w4v::w4a16_grouped_ws_bytes(*handle);
}

w4v_status w4a16_gemm_grouped(const w4a16_grouped_t *handle, void *ws, size_t ws_bytes, unsigned flags,
                              w4v_stream_t stream) {
    if ((flags & ~unsigned(W4V_STATIC_WEIGHTS)) != 0u) return W4V_ERR_ARG;
    if (handle == nullptr || !w4v::w4a16_grouped_handle_ok(*handle)) return W4V_ERR_ARG;
    if (ws == nullptr || ws_bytes < w4v::w4a16_grouped_ws_bytes(*handle)) return W4V_ERR_WORKSPACE;
    if (!w4v::aligned16(ws)) return W4V_ERR_ALIGN;
    return w4v::launch_w4a16_grouped(*handle, ws, (flags & W4V_STATIC_WEIGHTS) != 0u,
                                     reinterpret_cast<cudaStream_t>(stream));
}

size_t w8_lmhead_argmax_workspace_bytes(int M, int V) {
    if (M < 0 || M > 128 || V <= 0) return 0;
    return w4v::w8_lmhead_ws_bytes(M, V);
}

w4v_status w8_lmhead_argmax(const uint16_t *X, const int8_t *W, const uint16_t *scale, int M, int K,
                            int V, int32_t *argmax_out, float *maxlogit, float *logits_debug,
                            void *ws, size_t ws_bytes, w4v_stream_t stream) {
    return w8_lmhead_argmax_ex(X, W, scale, M, K, V, argmax_out, maxlogit, logits_debug, ws, ws_bytes, 0u, stream);
}

namespace {
// The rows in blocks of at most 32, one launch each, in order on the stream
// (each leaves the workspace cleared for the next): every row gets the
// arithmetic of a call with 1..32 rows.
w4v_status lmhead_row_blocks(const uint16_t *X, const int8_t *W, const uint16_t *scale, int M, int K, int V,
                             int32_t *argmax_out, float *maxlogit, float *logits, void *ws, cudaStream_t stream) {
    for (int m0 = 0; m0 < M; m0 += w4v::kDecodeMaxRows) {
        const int mb = std::min(w4v::kDecodeMaxRows, M - m0);
        const w4v_status st = w4v::launch_w8_lmhead_argmax(
            X + size_t(m0) * K, W, scale, mb, K, V, argmax_out + m0, maxlogit != nullptr ? maxlogit + m0 : nullptr,
            logits != nullptr ? logits + size_t(m0) * V : nullptr, ws, stream);
        if (st != W4V_OK) return st;
    }
    return W4V_OK;
}
}  // namespace

w4v_status w8_lmhead_argmax_ex(const uint16_t *X, const int8_t *W, const uint16_t *scale, int M, int K,
                               int V, int32_t *argmax_out, float *maxlogit, float *logits_debug,
                               void *ws, size_t ws_bytes, unsigned flags, w4v_stream_t stream) {
    if ((flags & ~unsigned(W4V_BATCH_INVARIANT)) != 0u) return W4V_ERR_ARG;
    if (M < 0 || M > 128 || K <= 0 || V <= 0 || K % 128 != 0 || V % 8 != 0) return W4V_ERR_SHAPE;
    if (M == 0) return W4V_OK;
    if (X == nullptr || W == nullptr || scale == nullptr || argmax_out == nullptr) return W4V_ERR_ARG;
    if (!w4v::aligned16(X) || !w4v::aligned16(W) || !w4v::aligned16(scale)) return W4V_ERR_ALIGN;
    if ((reinterpret_cast<uintptr_t>(argmax_out) & 3u) || (reinterpret_cast<uintptr_t>(maxlogit) & 3u) ||
        (reinterpret_cast<uintptr_t>(logits_debug) & 3u))
        return W4V_ERR_ALIGN;
    if (ws == nullptr || ws_bytes < w4v::w8_lmhead_ws_bytes(M, V)) return W4V_ERR_WORKSPACE;
    if (!w4v::aligned16(ws)) return W4V_ERR_ALIGN;
    if (M > w4v::kDecodeMaxRows && (flags & W4V_BATCH_INVARIANT) != 0u)
        return lmhead_row_blocks(X, W, scale, M, K, V, argmax_out, maxlogit, logits_debug, ws,
                                 reinterpret_cast<cudaStream_t>(stream));
    return w4v::launch_w8_lmhead_argmax(X, W, scale, M, K, V, argmax_out, maxlogit, logits_debug, ws,
                                        reinterpret_cast<cudaStream_t>(stream));
}

w4v_status w8_lmhead_argmax_accept(const uint16_t *X, const int8_t *W, const uint16_t *scale, int B, int n_draft,
                                   int K, int V, const int32_t *draft, int32_t *argmax_out, int32_t *n_accepted,
                                   int32_t *out_tokens, float *maxlogit, void *ws, size_t ws_bytes,
                                   w4v_stream_t stream) {
    return w8_lmhead_argmax_accept_ex(X, W, scale, B, n_draft, K, V, draft, argmax_out, n_accepted, out_tokens,
                                      maxlogit, ws, ws_bytes, 0u, stream);
}

w4v_status w8_lmhead_argmax_accept_ex(const uint16_t *X, const int8_t *W, const uint16_t *scale, int B,
                                      int n_draft, int K, int V, const int32_t *draft, int32_t *argmax_out,
                                      int32_t *n_accepted, int32_t *out_tokens, float *maxlogit, void *ws,
                                      size_t ws_bytes, unsigned flags, w4v_stream_t stream) {
    if ((flags & ~unsigned(W4V_BATCH_INVARIANT)) != 0u) return W4V_ERR_ARG;
    if (B < 0 || n_draft < 0 || K <= 0 || V <= 0 || K % 128 != 0 || V % 8 != 0) return W4V_ERR_SHAPE;
    if (B > 128 || long(B) * (n_draft + 1) > 128) return W4V_ERR_SHAPE;
    if (B == 0) return W4V_OK;
    const int M = B * (n_draft + 1);
    if (X == nullptr || W == nullptr || scale == nullptr || argmax_out == nullptr || n_accepted == nullptr ||
        (n_draft > 0 && draft == nullptr))
        return W4V_ERR_ARG;
    if (!w4v::aligned16(X) || !w4v::aligned16(W) || !w4v::aligned16(scale)) return W4V_ERR_ALIGN;
    if ((reinterpret_cast<uintptr_t>(argmax_out) & 3u) || (reinterpret_cast<uintptr_t>(maxlogit) & 3u) ||
        (reinterpret_cast<uintptr_t>(draft) & 3u) || (reinterpret_cast<uintptr_t>(n_accepted) & 3u) ||
        (reinterpret_cast<uintptr_t>(out_tokens) & 3u))
        return W4V_ERR_ALIGN;
    if (ws == nullptr || ws_bytes < w4v::w8_lmhead_ws_bytes(M, V)) return W4V_ERR_WORKSPACE;
    if (!w4v::aligned16(ws)) return W4V_ERR_ALIGN;
    if (M > w4v::kDecodeMaxRows && (flags & W4V_BATCH_INVARIANT) != 0u) {
        // the row blocks' tokens, then the acceptance of every sequence over them
        const w4v_status st = lmhead_row_blocks(X, W, scale, M, K, V, argmax_out, maxlogit, nullptr, ws,
                                                reinterpret_cast<cudaStream_t>(stream));
        if (st != W4V_OK) return st;
        return w4v::launch_spec_accept(argmax_out, draft, B, n_draft, n_accepted, out_tokens,
                                       reinterpret_cast<cudaStream_t>(stream));
    }
    const w4v::LmAccept acc{draft, B, n_draft, n_accepted, out_tokens};
    return w4v::launch_w8_lmhead_argmax(X, W, scale, M, K, V, argmax_out, maxlogit, nullptr, ws,
                                        reinterpret_cast<cudaStream_t>(stream), &acc);
}

size_t ngram_draft_workspace_bytes(int B) {
    if (B < 0 || B > 65535) return 0;
    return w4v::ngram_ws_bytes(B);
}

w4v_status ngram_draft(const int32_t *context, const int32_t *lengths, int B, int ld, int n_min, int n_max, int K,
                       int32_t *drafts, int32_t *match_len, void *ws, size_t ws_bytes, w4v_stream_t stream) {
    if (B < 0 || B > 65535 || ld < 1 || n_min < 1 || n_max < n_min || n_max > w4v::kNgramMax || K < 0 || K > 1024)
        return W4V_ERR_SHAPE;
    if (B == 0) return W4V_OK;
    if (context == nullptr || lengths == nullptr || (K > 0 && drafts == nullptr)) return W4V_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(context) & 3u) || (reinterpret_cast<uintptr_t>(lengths) & 3u) ||
        (reinterpret_cast<uintptr_t>(drafts) & 3u) || (reinterpret_cast<uintptr_t>(match_len) & 3u))
        return W4V_ERR_ALIGN;
    if (ws == nullptr || ws_bytes < w4v::ngram_ws_bytes(B)) return W4V_ERR_WORKSPACE;
    if (!w4v::aligned16(ws)) return W4V_ERR_ALIGN;
    return w4v::launch_ngram_draft(context, lengths, B, ld, n_min, n_max, K, drafts, match_len, ws,
                                   reinterpret_cast<cudaStream_t>(stream));
}

namespace {
w4v_status gdn_check(const float *state, const uint16_t *k, const uint16_t *v, const float *alpha,
                     const float *beta, int B, int T, int H, int dk, int dv) {
    if (B < 0 || B > 65535 || T < 1 || T > w4v::kGdnMaxT || H < 1 || H > 65535 || dk != w4v::kGdnDk || dv < 32 ||
        dv % 32 != 0 || dv > 4096)
        return W4V_ERR_SHAPE;
    if (B == 0) return W4V_OK;
    if (state == nullptr || k == nullptr || v == nullptr || alpha == nullptr || beta == nullptr) return W4V_ERR_ARG;
    if (!w4v::aligned16(state) || !w4v::aligned16(k) || !w4v::aligned16(v) ||
        (reinterpret_cast<uintptr_t>(alpha) & 3u) || (reinterpret_cast<uintptr_t>(beta) & 3u))
        return W4V_ERR_ALIGN;
    return W4V_OK;
}
}  // namespace

w4v_status gdn_verify(const float *state, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                      const float *alpha, const float *beta, int B, int T, int H, int dk, int dv, uint16_t *o,
                      w4v_stream_t stream) {
    w4v_status st = gdn_check(state, k, v, alpha, beta, B, T, H, dk, dv);
    if (st != W4V_OK || B == 0) return st;
    if (q == nullptr || o == nullptr) return W4V_ERR_ARG;
    if (!w4v::aligned16(q) || !w4v::aligned16(o)) return W4V_ERR_ALIGN;
    return w4v::launch_gdn(false, const_cast<float *>(state), q, k, v, alpha, beta, nullptr, o, B, T, H, dv,
                           reinterpret_cast<cudaStream_t>(stream));
}

w4v_status gdn_commit(float *state, const uint16_t *k, const uint16_t *v, const float *alpha, const float *beta,
                      const int32_t *n_accepted, int B, int T, int H, int dk, int dv, w4v_stream_t stream) {
    w4v_status st = gdn_check(state, k, v, alpha, beta, B, T, H, dk, dv);
    if (st != W4V_OK || B == 0) return st;
    if (n_accepted == nullptr) return W4V_ERR_ARG;
    if (reinterpret_cast<uintptr_t>(n_accepted) & 3u) return W4V_ERR_ALIGN;
    return w4v::launch_gdn(true, state, nullptr, k, v, alpha, beta, n_accepted, nullptr, B, T, H, dv,
                           reinterpret_cast<cudaStream_t>(stream));
}

w4v_status gdn_step(float *state, const uint16_t *k_prev, const uint16_t *v_prev, const float *alpha_prev,
                    const float *beta_prev, const int32_t *n_prev, int T_prev, const uint16_t *q, const uint16_t *k,
                    const uint16_t *v, const float *alpha, const float *beta, int B, int T, int H, int dk, int dv,
                    uint16_t *o, w4v_stream_t stream) {
    w4v_status st = gdn_check(state, k, v, alpha, beta, B, T, H, dk, dv);
    if (st != W4V_OK) return st;
    if (T_prev < 0 || T_prev > w4v::kGdnMaxT) return W4V_ERR_SHAPE;
    if (B == 0) return W4V_OK;
    if (q == nullptr || o == nullptr) return W4V_ERR_ARG;
    if (!w4v::aligned16(q) || !w4v::aligned16(o)) return W4V_ERR_ALIGN;
    if (T_prev > 0) {
        st = gdn_check(state, k_prev, v_prev, alpha_prev, beta_prev, B, T_prev, H, dk, dv);
        if (st != W4V_OK) return st;
        if (n_prev == nullptr) return W4V_ERR_ARG;
        if (reinterpret_cast<uintptr_t>(n_prev) & 3u) return W4V_ERR_ALIGN;
    }
    return w4v::launch_gdn_step(state, k_prev, v_prev, alpha_prev, beta_prev, n_prev, T_prev, q, k, v, alpha, beta,
                                o, B, T, H, dv, reinterpret_cast<cudaStream_t>(stream));
}

w4v_status spec_accept(const int32_t *target, const int32_t *draft, int B, int K, int32_t *n_accepted,
                       int32_t *out_tokens, w4v_stream_t stream) {
    if (B < 0 || K < 0 || K > 1024) return W4V_ERR_SHAPE;
    if (B == 0) return W4V_OK;
    if (target == nullptr || n_accepted == nullptr || (K > 0 && draft == nullptr)) return W4V_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(target) & 3u) || (reinterpret_cast<uintptr_t>(draft) & 3u) ||
        (reinterpret_cast<uintptr_t>(n_accepted) & 3u) || (reinterpret_cast<uintptr_t>(out_tokens) & 3u))
        return W4V_ERR_ALIGN;
    return w4v::launch_spec_accept(target, draft, B, K, n_accepted, out_tokens,
                                   reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
