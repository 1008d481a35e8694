// C ABI of libkda: argument validation, workspace layout and kernel dispatch.
// Every entry point is declared and documented in include/kda.h.
#include "attnres.h"
#include "kda_internal.h"

#include <mutex>

namespace kda {

int sm_count() {
    static std::mutex mu;
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
    if (dev >= 64) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        return n;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
            cached[dev] = n;
    }
    return cached[dev];
}

}  // namespace kda

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void* a, size_t an, const void* b, size_t bn) {
    if (!a || !b || an == 0 || bn == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + bn && b0 < a0 + an;
}

}  // namespace

namespace kda {

kda_status prefill_impl(const void* q, const void* k, const void* v, const void* alpha,
                        const float* beta, const float* S0, const int32_t* cu_seqlens,
                        int32_t num_seqs, int64_t total_tokens, int32_t H, int32_t d_k,
                        int32_t d_v, kda_dtype dtype, int32_t chunk, void* o, float* S_T,
                        void* workspace, size_t workspace_bytes, kda_prefill_kernel kernel,
                        kda_stream_t stream_, kda_gate_format gate, bool additive) {
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    if (num_seqs < 0 || total_tokens < 0 || H < 1 || d_k < 1 || d_v < 1)
        return KDA_ERR_INVALID_ARG;
    if (dtype != KDA_BF16 && dtype != KDA_FP32) return KDA_ERR_INVALID_ARG;
    if (kernel != KDA_KERNEL_AUTO && kernel != KDA_KERNEL_CHUNK_SIMT &&
        kernel != KDA_KERNEL_CHUNK_TC && kernel != KDA_KERNEL_CHUNK_TC_SPLIT)
        return KDA_ERR_INVALID_ARG;
    if (gate != KDA_GATE_CHANNEL_F32 && gate != KDA_GATE_HEAD_F32 &&
        gate != KDA_GATE_CHANNEL_LOG_BF16)
        return KDA_ERR_INVALID_ARG;
    if (chunk != 16 && chunk != 32 && chunk != 64) return KDA_ERR_UNSUPPORTED;
    if (d_k % 16 != 0 || d_k > 128 || d_v % 16 != 0 || d_v > 1024) return KDA_ERR_UNSUPPORTED;
    if (total_tokens > (int64_t)INT32_MAX) return KDA_ERR_UNSUPPORTED;
    if (gate != KDA_GATE_CHANNEL_F32 && kernel == KDA_KERNEL_CHUNK_TC_SPLIT)
        return KDA_ERR_UNSUPPORTED;
    // the additive update has no sequence-axis split
    if (additive && kernel == KDA_KERNEL_CHUNK_TC_SPLIT) return KDA_ERR_UNSUPPORTED;
    if ((int64_t)num_seqs * H > (int64_t)INT32_MAX / 64) return KDA_ERR_UNSUPPORTED;
    if (!cu_seqlens || !workspace || (num_seqs > 0 && !S_T)) return KDA_ERR_INVALID_ARG;
    if (total_tokens > 0 && (!q || !k || !v || !alpha || !beta || !o)) return KDA_ERR_INVALID_ARG;
    if (workspace_bytes < kda::WorkspaceLayout::bytes(num_seqs)) return KDA_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, alpha, beta, S0, o, S_T, workspace, cu_seqlens};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return KDA_ERR_INVALID_ARG;
    const size_t esz = dtype == KDA_BF16 ? 2 : 4;
    const size_t n_o = (size_t)total_tokens * H * d_v * esz;
    const size_t n_s = (size_t)num_seqs * H * d_v * d_k * sizeof(float);
    // outputs may not overlap inputs, except S_T == S0 exactly
    if (S0 && S_T != S0 && overlaps(S_T, n_s, S0, n_s)) return KDA_ERR_INVALID_ARG;
    const size_t n_qk = (size_t)total_tokens * H * d_k * esz;
    const size_t n_v = (size_t)total_tokens * H * d_v * esz;
    const size_t n_a = gate == KDA_GATE_HEAD_F32 ? (size_t)total_tokens * H * sizeof(float)
                       : gate == KDA_GATE_CHANNEL_LOG_BF16 ? (size_t)total_tokens * H * d_v * 2
                                                           : (size_t)total_tokens * H * d_v * sizeof(float);
    const void* ins[] = {q, k, v, alpha, beta};
    const size_t in_n[] = {n_qk, n_qk, n_v, n_a, (size_t)total_tokens * H * sizeof(float)};
    for (int i = 0; i < 5; ++i)
        if (overlaps(o, n_o, ins[i], in_n[i]) || overlaps(S_T, n_s, ins[i], in_n[i]))
            return KDA_ERR_INVALID_ARG;
    if (overlaps(o, n_o, S_T, n_s) || overlaps(o, n_o, S0, n_s)) return KDA_ERR_INVALID_ARG;

    kda::PrefillArgs a;
    a.q = q; a.k = k; a.v = v; a.alpha = alpha; a.beta = beta; a.S0 = S0;
    a.cu_seqlens = cu_seqlens; a.num_seqs = num_seqs; a.total_tokens = total_tokens;
    a.gate = gate;
    a.additive = additive ? 1 : 0;
    a.H = H; a.d_k = d_k; a.d_v = d_v; a.dtype = dtype; a.chunk = chunk; a.o = o; a.S_T = S_T;
    char* ws = static_cast<char*>(workspace);
    a.status = reinterpret_cast<int32_t*>(ws + kda::WorkspaceLayout::kStatus);
    a.counter = reinterpret_cast<int32_t*>(ws + kda::WorkspaceLayout::kCounter);
    a.order = reinterpret_cast<int32_t*>(ws + kda::WorkspaceLayout::kOrder);

    const bool tc_ok = kda::prefill_tc_supports(a);
    const bool want_tc = kernel == KDA_KERNEL_CHUNK_TC || kernel == KDA_KERNEL_CHUNK_TC_SPLIT;
    if (want_tc && !tc_ok) return KDA_ERR_UNSUPPORTED;
    const bool use_tc = want_tc || (kernel == KDA_KERNEL_AUTO && tc_ok);
    // sequence-axis split: few chains, long sequences, room in the workspace
    kda::SplitLayout split;
    if (use_tc && kernel != KDA_KERNEL_CHUNK_TC && num_seqs > 0 && gate == KDA_GATE_CHANNEL_F32 &&
        !additive) {
        const int M = kda::split_segments(num_seqs, H, d_k, d_v, chunk);
        const bool forced = kernel == KDA_KERNEL_CHUNK_TC_SPLIT;
        if (forced && M < 2) return KDA_ERR_UNSUPPORTED;
        const bool long_enough = total_tokens >= (int64_t)num_seqs * M * 2048;
        if (M >= 2 && (long_enough || forced)) {
            split = kda::split_layout(num_seqs, total_tokens, H, d_k, d_v, M);
            if (workspace_bytes < split.end) {
                if (forced) return KDA_ERR_INVALID_ARG;
                split.M = 1;
            }
        }
    }

    // room for the channels the tensor-core kernel may hand back to the portable one
    const size_t redo_at = kda::WorkspaceLayout::bytes(num_seqs);
    const size_t redo_n = kda::WorkspaceLayout::redo_bytes(num_seqs, H, d_v);
    if (use_tc && split.M < 2 && redo_n > 0 && workspace_bytes >= redo_at + redo_n && d_v % 128 == 0)
        a.redo = reinterpret_cast<uint32_t*>(ws + redo_at);

    if (kda::launch_planner(a, stream, redo_n) != cudaSuccess) return KDA_ERR_CUDA;
    if (num_seqs == 0) return KDA_OK;
    cudaError_t err;
    if (use_tc && split.M >= 2) {
        err = kda::launch_prefill_tc_split(a, split, ws, stream);
    } else if (use_tc) {
        err = kda::launch_prefill_tc(a, stream);
        if (err == cudaSuccess && a.redo && total_tokens > 0)
            err = kda::launch_prefill_simt_redo(a, stream);
    } else {
        err = kda::launch_prefill_simt(a, stream);
    }
    return err == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // namespace kda

extern "C" {

size_t kda_prefill_workspace_size(int32_t num_seqs, int32_t H, int32_t d_k, int32_t d_v,
                                  int32_t chunk) {
    (void)chunk;
    if (num_seqs < 0) return 0;
    const size_t base = kda::WorkspaceLayout::bytes(num_seqs);
    if (H < 1 || d_k < 1 || d_v < 1) return base;
    // the channels handed back by the tensor-core kernel
    return base + kda::WorkspaceLayout::redo_bytes(num_seqs, H, d_v);
}

size_t kda_prefill_workspace_size_tokens(int32_t num_seqs, int64_t total_tokens, int32_t H,
                                         int32_t d_k, int32_t d_v, int32_t chunk) {
    if (num_seqs < 0 || total_tokens < 0) return 0;
    const size_t plain = kda_prefill_workspace_size(num_seqs, H, d_k, d_v, chunk);
    if (H < 1 || d_k < 1 || d_v < 1) return plain;
    // the sequence-axis split's buffers, in the bitmap's place, when it splits
    const int M = kda::split_segments(num_seqs, H, d_k, d_v, chunk);
    if (M < 2) return plain;
    const size_t split = kda::split_layout(num_seqs, total_tokens, H, d_k, d_v, M).end;
    return split > plain ? split : plain;
}

kda_status kda_prefill(const void* q, const void* k, const void* v, const float* alpha,
                       const float* beta, const float* S0, const int32_t* cu_seqlens,
                       int32_t num_seqs, int64_t total_tokens, int32_t H, int32_t d_k,
                       int32_t d_v, kda_dtype dtype, int32_t chunk, void* o, float* S_T,
                       void* workspace, size_t workspace_bytes, kda_stream_t stream) {
    return kda::prefill_impl(q, k, v, alpha, beta, S0, cu_seqlens, num_seqs, total_tokens, H,
                             d_k, d_v, dtype, chunk, o, S_T, workspace, workspace_bytes,
                             KDA_KERNEL_AUTO, stream);
}

kda_status kda_prefill_ex(const void* q, const void* k, const void* v, const float* alpha,
                          const float* beta, const float* S0, const int32_t* cu_seqlens,
                          int32_t num_seqs, int64_t total_tokens, int32_t H, int32_t d_k,
                          int32_t d_v, kda_dtype dtype, int32_t chunk, void* o, float* S_T,
                          void* workspace, size_t workspace_bytes, kda_prefill_kernel kernel,
                          kda_stream_t stream) {
    return kda::prefill_impl(q, k, v, alpha, beta, S0, cu_seqlens, num_seqs, total_tokens, H,
                             d_k, d_v, dtype, chunk, o, S_T, workspace, workspace_bytes, kernel,
                             stream);
}

kda_status kda_prefill_gates(const void* q, const void* k, const void* v, const void* alpha,
                             kda_gate_format gate_format, const float* beta, const float* S0,
                             const int32_t* cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                             int32_t H, int32_t d_k, int32_t d_v, kda_dtype dtype,
                             int32_t chunk, void* o, float* S_T, void* workspace,
                             size_t workspace_bytes, kda_prefill_kernel kernel,
                             kda_stream_t stream) {
    return kda::prefill_impl(q, k, v, alpha, beta, S0, cu_seqlens, num_seqs, total_tokens, H,
                             d_k, d_v, dtype, chunk, o, S_T, workspace, workspace_bytes, kernel,
                             stream, gate_format);
}

kda_status kda_prefill_supported(kda_prefill_kernel kernel, int32_t H, int32_t d_k, int32_t d_v,
                                 kda_dtype dtype, int32_t chunk) {
    if (kernel != KDA_KERNEL_AUTO && kernel != KDA_KERNEL_CHUNK_SIMT &&
        kernel != KDA_KERNEL_CHUNK_TC && kernel != KDA_KERNEL_CHUNK_TC_SPLIT)
        return KDA_ERR_INVALID_ARG;
    if (dtype != KDA_BF16 && dtype != KDA_FP32) return KDA_ERR_INVALID_ARG;
    if (H < 1 || d_k < 1 || d_v < 1) return KDA_ERR_INVALID_ARG;
    if (chunk != 16 && chunk != 32 && chunk != 64) return KDA_ERR_UNSUPPORTED;
    if (d_k % 16 != 0 || d_k > 128 || d_v % 16 != 0 || d_v > 1024) return KDA_ERR_UNSUPPORTED;
    if (kernel != KDA_KERNEL_CHUNK_TC && kernel != KDA_KERNEL_CHUNK_TC_SPLIT) return KDA_OK;
    kda::PrefillArgs a = {};
    a.H = H; a.d_k = d_k; a.d_v = d_v; a.dtype = dtype; a.chunk = chunk;
    return kda::prefill_tc_supports(a) ? KDA_OK : KDA_ERR_UNSUPPORTED;
}

kda_status kda_prefill_device_status(const void* workspace, kda_stream_t stream) {
    if (!workspace) return KDA_ERR_INVALID_ARG;
    int32_t st = 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(&st, static_cast<const char*>(workspace) + kda::WorkspaceLayout::kStatus,
                        sizeof st, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return KDA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return KDA_ERR_CUDA;
    if (st == 0) return KDA_OK;
    if (st == KDA_ERR_DEVICE_TIMEOUT || st == KDA_ERR_DEVICE_RANGE) return (kda_status)st;
    return KDA_ERR_DEVICE_INPUT;
}

kda_status kda_segment_combine(const float* S_in, const float* g, const float* P, const float* R,
                               int32_t num_seqs, int32_t H, int32_t d_k, int32_t d_v,
                               float* S_out, kda_stream_t stream) {
    if (num_seqs < 0 || H < 1 || d_k < 1 || d_v < 1) return KDA_ERR_INVALID_ARG;
    if (d_k > 128) return KDA_ERR_UNSUPPORTED;
    if (num_seqs == 0) return KDA_OK;
    if (!S_in || !g || !P || !R || !S_out) return KDA_ERR_INVALID_ARG;
    const void* ptrs[] = {S_in, g, P, R, S_out};
    for (const void* p : ptrs)
        if (!aligned16(p)) return KDA_ERR_INVALID_ARG;
    const size_t ns = (size_t)num_seqs * H * d_v * d_k * sizeof(float);
    const void* ins[] = {g, P, R};
    const size_t in_n[] = {(size_t)num_seqs * H * d_v * sizeof(float),
                           (size_t)num_seqs * H * d_k * d_k * sizeof(float), ns};
    for (int i = 0; i < 3; ++i)
        if (overlaps(S_out, ns, ins[i], in_n[i])) return KDA_ERR_INVALID_ARG;
    if (S_out != S_in && overlaps(S_out, ns, S_in, ns)) return KDA_ERR_INVALID_ARG;
    return kda::launch_segment_combine(S_in, g, P, R, num_seqs, H, d_k, d_v, S_out,
                                       static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? KDA_OK
               : KDA_ERR_CUDA;
}

kda_status kda_check_wait_timeout(void* workspace, size_t workspace_bytes, uint64_t timeout_ns,
                                  kda_stream_t stream) {
    if (!workspace || !aligned16(workspace) || workspace_bytes < kda::WorkspaceLayout::bytes(0))
        return KDA_ERR_INVALID_ARG;
    if (timeout_ns < 1000 || timeout_ns > 1000000000ull) return KDA_ERR_INVALID_ARG;
    int32_t* status =
        reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + kda::WorkspaceLayout::kStatus);
    return kda::launch_wait_probe(status, timeout_ns, static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? KDA_OK
               : KDA_ERR_CUDA;
}

// Validation and launch behind kda_decode_step / kda_decode_step_gates.
static kda_status decode_impl(const void* q, const void* k, const void* v, const void* alpha,
                              kda_gate_format gate, const float* beta, float* S, int32_t B,
                              int32_t H, int32_t d_k, int32_t d_v, kda_dtype dtype, void* o,
                              kda_stream_t stream, bool additive = false) {
    if (B < 0 || H < 1 || d_v < 1) return KDA_ERR_INVALID_ARG;
    if (gate != KDA_GATE_CHANNEL_F32 && gate != KDA_GATE_HEAD_F32 &&
        gate != KDA_GATE_CHANNEL_LOG_BF16)
        return KDA_ERR_INVALID_ARG;
    if (dtype != KDA_BF16 && dtype != KDA_FP32) return KDA_ERR_INVALID_ARG;
    if (d_k != 16 && d_k != 32 && d_k != 64 && d_k != 128 && d_k != 256)
        return KDA_ERR_UNSUPPORTED;
    if (d_v > 4096) return KDA_ERR_UNSUPPORTED;
    if ((int64_t)B * H > (int64_t)INT32_MAX) return KDA_ERR_UNSUPPORTED;
    if (B == 0) return KDA_OK;
    if (!q || !k || !v || !alpha || !beta || !S || !o) return KDA_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, alpha, beta, S, o};
    for (const void* p : ptrs)
        if (!aligned16(p)) return KDA_ERR_INVALID_ARG;
    const size_t esz = dtype == KDA_BF16 ? 2 : 4;
    const size_t n_s = (size_t)B * H * d_v * d_k * sizeof(float);
    const size_t n_o = (size_t)B * H * d_v * esz;
    const void* ins[] = {q, k, v, alpha, beta};
    const size_t n_a = gate == KDA_GATE_HEAD_F32 ? (size_t)B * H * sizeof(float)
                       : gate == KDA_GATE_CHANNEL_LOG_BF16 ? (size_t)B * H * d_v * 2
                                                           : (size_t)B * H * d_v * sizeof(float);
    const size_t in_n[] = {(size_t)B * H * d_k * esz, (size_t)B * H * d_k * esz,
                           (size_t)B * H * d_v * esz, n_a, (size_t)B * H * sizeof(float)};
    for (int i = 0; i < 5; ++i)
        if (overlaps(S, n_s, ins[i], in_n[i]) || overlaps(o, n_o, ins[i], in_n[i]))
            return KDA_ERR_INVALID_ARG;
    if (overlaps(o, n_o, S, n_s)) return KDA_ERR_INVALID_ARG;

    kda::DecodeArgs a;
    a.q = q; a.k = k; a.v = v; a.alpha = alpha; a.beta = beta; a.S = S;
    a.B = B; a.H = H; a.d_k = d_k; a.d_v = d_v; a.dtype = dtype; a.o = o; a.gate = gate;
    a.additive = additive ? 1 : 0;
    return kda::launch_decode(a, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? KDA_OK
               : KDA_ERR_CUDA;
}

kda_status kda_decode_step(const void* q, const void* k, const void* v, const float* alpha,
                           const float* beta, float* S, int32_t B, int32_t H, int32_t d_k,
                           int32_t d_v, kda_dtype dtype, void* o, kda_stream_t stream) {
    return decode_impl(q, k, v, alpha, KDA_GATE_CHANNEL_F32, beta, S, B, H, d_k, d_v, dtype,
                            o, stream);
}

kda_status kda_decode_step_gates(const void* q, const void* k, const void* v, const void* alpha,
                                 kda_gate_format gate_format, const float* beta, float* S,
                                 int32_t B, int32_t H, int32_t d_k, int32_t d_v, kda_dtype dtype,
                                 void* o, kda_stream_t stream) {
    return decode_impl(q, k, v, alpha, gate_format, beta, S, B, H, d_k, d_v, dtype, o,
                            stream);
}

// Bytes kda_backward_gates needs: the backward layout, plus for the gate
// layouts other than per-channel fp32 the gate expanded per channel and the
// gradient with respect to it (fp32 [T][H][d_v] each).
static size_t backward_bytes(int32_t num_seqs, int64_t total_tokens, int32_t H, int32_t d_k,
                             int32_t d_v, int32_t chunk, kda_gate_format gate) {
    if (num_seqs < 0 || total_tokens < 0 || H < 1 || d_k != 128 || d_v < 64 || d_v % 64 != 0 ||
        chunk != 64)
        return 0;
    if (gate != KDA_GATE_CHANNEL_F32 && gate != KDA_GATE_HEAD_F32 &&
        gate != KDA_GATE_CHANNEL_LOG_BF16)
        return 0;
    size_t bytes = kda::backward_layout(num_seqs, total_tokens, H, d_v).end;
    if (gate != KDA_GATE_CHANNEL_F32)
        bytes += 2 * (((size_t)total_tokens * H * d_v * sizeof(float) + 255) & ~(size_t)255);
    return bytes;
}

// Validation and launches behind kda_backward / kda_backward_gates.
static kda_status backward_impl(const void* q, const void* k, const void* v, const void* alpha,
                                kda_gate_format gate, const float* beta, const float* S0,
                                const int32_t* cu_seqlens, int32_t num_seqs,
                                int64_t total_tokens, int32_t H, int32_t d_k, int32_t d_v,
                                kda_dtype dtype, int32_t chunk, const void* d_o,
                                const float* dS_T, float* dq, float* dk, float* dv,
                                float* dalpha, float* dbeta, float* dS0, void* workspace,
                                size_t workspace_bytes, kda_stream_t stream_) {
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    if (num_seqs < 0 || total_tokens < 0 || H < 1 || d_k < 1 || d_v < 1)
        return KDA_ERR_INVALID_ARG;
    if (dtype != KDA_BF16 && dtype != KDA_FP32) return KDA_ERR_INVALID_ARG;
    if (gate != KDA_GATE_CHANNEL_F32 && gate != KDA_GATE_HEAD_F32 &&
        gate != KDA_GATE_CHANNEL_LOG_BF16)
        return KDA_ERR_INVALID_ARG;
    if (dtype != KDA_BF16 || d_k != 128 || d_v % 64 != 0 || d_v > 1024 || chunk != 64)
        return KDA_ERR_UNSUPPORTED;
    if (total_tokens > (int64_t)INT32_MAX) return KDA_ERR_UNSUPPORTED;
    if ((int64_t)num_seqs * H * (d_v / 64) > (int64_t)INT32_MAX) return KDA_ERR_UNSUPPORTED;
    if (!cu_seqlens || !workspace) return KDA_ERR_INVALID_ARG;
    if (total_tokens > 0 && (!q || !k || !v || !alpha || !beta || !d_o || !dq || !dk || !dv ||
                             !dalpha || !dbeta))
        return KDA_ERR_INVALID_ARG;
    const kda::BackwardLayout L = kda::backward_layout(num_seqs, total_tokens, H, d_v);
    if (workspace_bytes < backward_bytes(num_seqs, total_tokens, H, d_k, d_v, chunk, gate))
        return KDA_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, alpha, beta, S0, cu_seqlens, d_o, dS_T, dq, dk, dv,
                          dalpha, dbeta, dS0, workspace};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return KDA_ERR_INVALID_ARG;
    // no output may overlap an input or another output
    const size_t tq = (size_t)total_tokens * H * d_k, tv = (size_t)total_tokens * H * d_v;
    const size_t ts = (size_t)total_tokens * H, ns = (size_t)num_seqs * H * d_v * d_k;
    const size_t n_gate = gate == KDA_GATE_HEAD_F32 ? 4 * ts
                          : gate == KDA_GATE_CHANNEL_LOG_BF16 ? 2 * tv : 4 * tv;
    const size_t n_dgate = gate == KDA_GATE_HEAD_F32 ? 4 * ts : 4 * tv;
    const void* ins[] = {q, k, v, alpha, beta, S0, d_o, dS_T, workspace};
    const size_t in_n[] = {2 * tq, 2 * tq, 2 * tv, n_gate, 4 * ts, 4 * ns, 2 * tv, 4 * ns,
                           workspace_bytes};
    const void* outs[] = {dq, dk, dv, dalpha, dbeta, dS0};
    const size_t out_n[] = {4 * tq, 4 * tq, 4 * tv, n_dgate, 4 * ts, 4 * ns};
    for (int o = 0; o < 6; ++o) {
        for (int i = 0; i < 9; ++i)
            if (overlaps(outs[o], out_n[o], ins[i], in_n[i])) return KDA_ERR_INVALID_ARG;
        for (int o2 = o + 1; o2 < 6; ++o2)
            if (overlaps(outs[o], out_n[o], outs[o2], out_n[o2])) return KDA_ERR_INVALID_ARG;
    }

    char* ws = static_cast<char*>(workspace);
    kda::PrefillArgs pa = {};
    pa.cu_seqlens = cu_seqlens; pa.num_seqs = num_seqs; pa.total_tokens = total_tokens;
    pa.H = H; pa.d_k = d_k; pa.d_v = d_v; pa.dtype = dtype; pa.chunk = chunk;
    pa.status = reinterpret_cast<int32_t*>(ws + kda::WorkspaceLayout::kStatus);
    pa.counter = reinterpret_cast<int32_t*>(ws + kda::WorkspaceLayout::kCounter);
    pa.order = reinterpret_cast<int32_t*>(ws + kda::WorkspaceLayout::kOrder);
    if (kda::launch_planner(pa, stream) != cudaSuccess) return KDA_ERR_CUDA;
    if (num_seqs == 0) return KDA_OK;
    kda::BackwardArgs a;
    a.q = q; a.k = k; a.v = v; a.dO = d_o; a.beta = beta; a.S0 = S0;
    a.dS_T = dS_T; a.cu_seqlens = cu_seqlens; a.num_seqs = num_seqs;
    a.total_tokens = total_tokens; a.H = H; a.d_v = d_v;
    a.dq = dq; a.dk = dk; a.dv = dv; a.dbeta = dbeta; a.dS0 = dS0;
    if (gate == KDA_GATE_CHANNEL_F32) {
        a.alpha = static_cast<const float*>(alpha);
        a.dalpha = dalpha;
        return kda::launch_backward(a, L, ws, stream) == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
    }
    // the gate per channel and its gradient, in the workspace after the layout
    const size_t plane = ((size_t)total_tokens * H * d_v * sizeof(float) + 255) & ~(size_t)255;
    float* ax = reinterpret_cast<float*>(ws + L.end);
    float* dax = reinterpret_cast<float*>(ws + L.end + plane);
    a.alpha = ax;
    a.dalpha = dax;
    if (kda::launch_gate_expand(alpha, gate, a, ax, pa.status, stream) != cudaSuccess)
        return KDA_ERR_CUDA;
    if (kda::launch_backward(a, L, ws, stream) != cudaSuccess) return KDA_ERR_CUDA;
    return kda::launch_gate_grad(gate, a, ax, dax, dalpha, pa.status, stream) == cudaSuccess
               ? KDA_OK
               : KDA_ERR_CUDA;
}

kda_status kda_prefill_additive(const void* q, const void* k, const void* v, const float* alpha,
                                const float* beta, const float* S0, const int32_t* cu_seqlens,
                                int32_t num_seqs, int64_t total_tokens, int32_t H, int32_t d_k,
                                int32_t d_v, kda_dtype dtype, int32_t chunk, void* o, float* S_T,
                                void* workspace, size_t workspace_bytes,
                                kda_prefill_kernel kernel, kda_stream_t stream) {
    return kda::prefill_impl(q, k, v, alpha, beta, S0, cu_seqlens, num_seqs, total_tokens, H,
                             d_k, d_v, dtype, chunk, o, S_T, workspace, workspace_bytes, kernel,
                             stream, KDA_GATE_CHANNEL_F32, true);
}

kda_status kda_decode_step_additive(const void* q, const void* k, const void* v,
                                    const float* alpha, const float* beta, float* S, int32_t B,
                                    int32_t H, int32_t d_k, int32_t d_v, kda_dtype dtype,
                                    void* o, kda_stream_t stream) {
    return decode_impl(q, k, v, alpha, KDA_GATE_CHANNEL_F32, beta, S, B, H, d_k, d_v, dtype, o,
                       stream, true);
}

size_t kda_backward_workspace_size(int32_t num_seqs, int64_t total_tokens, int32_t H,
                                   int32_t d_k, int32_t d_v, int32_t chunk) {
    return backward_bytes(num_seqs, total_tokens, H, d_k, d_v, chunk, KDA_GATE_CHANNEL_F32);
}

size_t kda_backward_gates_workspace_size(int32_t num_seqs, int64_t total_tokens, int32_t H,
                                         int32_t d_k, int32_t d_v, int32_t chunk,
                                         kda_gate_format gate_format) {
    return backward_bytes(num_seqs, total_tokens, H, d_k, d_v, chunk, gate_format);
}

kda_status kda_backward(const void* q, const void* k, const void* v, const float* alpha,
                        const float* beta, const float* S0, const int32_t* cu_seqlens,
                        int32_t num_seqs, int64_t total_tokens, int32_t H, int32_t d_k,
                        int32_t d_v, kda_dtype dtype, int32_t chunk, const void* d_o,
                        const float* dS_T, float* dq, float* dk, float* dv, float* dalpha,
                        float* dbeta, float* dS0, void* workspace, size_t workspace_bytes,
                        kda_stream_t stream) {
    return backward_impl(q, k, v, alpha, KDA_GATE_CHANNEL_F32, beta, S0, cu_seqlens, num_seqs,
                         total_tokens, H, d_k, d_v, dtype, chunk, d_o, dS_T, dq, dk, dv, dalpha,
                         dbeta, dS0, workspace, workspace_bytes, stream);
}

kda_status kda_backward_gates(const void* q, const void* k, const void* v, const void* alpha,
                              kda_gate_format gate_format, const float* beta, const float* S0,
                              const int32_t* cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                              int32_t H, int32_t d_k, int32_t d_v, kda_dtype dtype,
                              int32_t chunk, const void* d_o, const float* dS_T, float* dq,
                              float* dk, float* dv, float* dgate, float* dbeta, float* dS0,
                              void* workspace, size_t workspace_bytes, kda_stream_t stream) {
    return backward_impl(q, k, v, alpha, gate_format, beta, S0, cu_seqlens, num_seqs,
                         total_tokens, H, d_k, d_v, dtype, chunk, d_o, dS_T, dq, dk, dv, dgate,
                         dbeta, dS0, workspace, workspace_bytes, stream);
}

kda_status attnres_layer(const void* blocks, int32_t num_blocks, const float* partial,
                         const void* h_last, float* partial_out, void* block_out,
                         const float* q, float scale, int64_t T, int32_t d, kda_dtype dtype,
                         void* h, kda_stream_t stream) {
    if (num_blocks < 0 || T < 0 || d < 1) return KDA_ERR_INVALID_ARG;
    if (dtype != KDA_BF16 && dtype != KDA_FP32) return KDA_ERR_INVALID_ARG;
    const bool has_p = partial || h_last;
    const int64_t m = (int64_t)num_blocks + (has_p ? 1 : 0);
    if (m < 1) return KDA_ERR_INVALID_ARG;
    if ((partial_out || block_out) && !has_p) return KDA_ERR_INVALID_ARG;
    if (d % 8 != 0 || m > 64) return KDA_ERR_UNSUPPORTED;
    if (T == 0) return KDA_OK;
    if (!q || !h || (num_blocks > 0 && !blocks)) return KDA_ERR_INVALID_ARG;
    const void* ptrs[] = {blocks, partial, h_last, partial_out, block_out, q, h};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return KDA_ERR_INVALID_ARG;
    const size_t esz = dtype == KDA_BF16 ? 2 : 4;
    const size_t row = (size_t)T * d;
    const void* ins[] = {blocks, partial, h_last, q};
    const size_t in_n[] = {(size_t)num_blocks * row * esz, row * 4, row * esz, (size_t)d * 4};
    const void* outs[] = {h, partial_out, block_out};
    const size_t out_n[] = {row * esz, row * 4, row * esz};
    for (int o = 0; o < 3; ++o) {
        for (int i = 0; i < 4; ++i) {
            if (o == 1 && i == 1 && partial_out == partial) continue;   // in place
            if (overlaps(outs[o], out_n[o], ins[i], in_n[i])) return KDA_ERR_INVALID_ARG;
        }
        for (int o2 = o + 1; o2 < 3; ++o2)
            if (overlaps(outs[o], out_n[o], outs[o2], out_n[o2])) return KDA_ERR_INVALID_ARG;
    }
    return kda::launch_attnres(blocks, num_blocks, partial, h_last, partial_out, block_out, q,
                               scale, T, d, dtype, h, static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? KDA_OK
               : KDA_ERR_CUDA;
}

const char* kda_status_string(kda_status s) {
    switch (s) {
        case KDA_OK: return "ok";
        case KDA_ERR_INVALID_ARG: return "invalid argument";
        case KDA_ERR_UNSUPPORTED: return "unsupported size or option";
        case KDA_ERR_CUDA: return "CUDA error";
        case KDA_ERR_DEVICE_INPUT: return "invalid device input (cu_seqlens)";
        case KDA_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
        case KDA_ERR_DEVICE_RANGE: return "alpha decays too fast for the chunk form (device input)";
        default: return "unknown status";
    }
}

int32_t kda_version(void) { return (1 << 16) | 0; }

}  // extern "C"
