// Internal declarations shared by the libkda translation units (CUDA path only).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "kda.h"

namespace kda {

// Smallest product of alpha over the tokens of one pass of the chunk form,
// per channel: the form divides by it, so it must stay far from the float
// range's end.  A chunk below it on some channel is taken again in passes of
// 16 tokens; a pass of 16 below it is reported as KDA_ERR_DEVICE_RANGE.
constexpr float kDecayFloor = 1e-30f;
// Sequence-axis split: a later segment's zero-start output is kept in fp32
// for the chunks whose decay from the segment start is at least this.
constexpr float kOresFloor = 0x1p-10f;

// Layout of the prefill workspace (all offsets in bytes from its start).
//   [0, 4)    int32 device status (0 = ok, or a KDA_ERR_DEVICE_* code)
//   [4, 8)    int32 work counter of the persistent tensor-core kernel
//   [16, ...) int32 order[num_seqs]: sequence indices, longest first, then
//             int32 [num_seqs]: the planner's sorted runs (batches of more
//             than 1024 sequences)
//   then, for the tensor-core kernel without the sequence-axis split (whose
//   buffers take the same place), when the workspace has room: uint32
//   [num_seqs][H][d_v / 128][4], for each 128-channel block the channels whose
//   chunks decayed too fast for the one-pass chunk form (one bit each); the
//   portable kernel redoes those channels
struct WorkspaceLayout {
    static constexpr size_t kStatus = 0;
    static constexpr size_t kCounter = 4;
    static constexpr size_t kOrder = 16;
    // order[num_seqs], then the planner's sorted runs (num_seqs more)
    static size_t bytes(int32_t num_seqs) {
        size_t b = kOrder + 2 * sizeof(int32_t) * (size_t)(num_seqs > 0 ? num_seqs : 0);
        return (b + 255) & ~(size_t)255;
    }
    static size_t redo_bytes(int32_t num_seqs, int32_t H, int32_t d_v) {
        if (num_seqs <= 0 || H <= 0 || d_v < 128) return 0;
        const size_t b = (size_t)num_seqs * H * (d_v / 128) * 4 * sizeof(uint32_t);
        return (b + 255) & ~(size_t)255;
    }
};

// Sequence-axis split of the tensor-core prefill (few long chains): each
// sequence is cut into M segments of whole chunks.  Virtual sequence
// v = j * N + n is segment j of sequence n.  Buffers appended to the workspace:
//   vt0    int64 [M N]                  first token of each segment
//   vlen   int32 [M N]                  its length
//   sfin   fp32 [M N][H][d_v][d_k]      final state of each segment (segment 0
//                                       from the true S0, the others from zero)
//   pbuf   fp32 [(M-1) N][H][d_k][d_k]  transition P of segments 1..M-1
//   gbuf   fp32 [M N][H][d_v]           prod alpha over each segment
//   sst    fp32 [(M-1) N][H][d_v][d_k]  true initial state of segments 1..M-1
//   rnorm  fp32 [(M-1) N][H][d_v]       norms of the rows of sst
//   gstart fp32 [T / 64 + N + 1][H][d_v] per chunk of segments 1..M-1: prod
//                                       alpha from the segment start to the
//                                       chunk start (slot cu[n] / 64 + n + c)
//   qtil   fp32 [T][H][d_k]             P_{<=t} q_t for the tokens of
//                                       segments 1..M-1 (P_{<=t}: the product
//                                       of (I - beta k k^T) from the segment
//                                       start through token t)
//   qfro   fp32 [T / 64 + N + 1][H]     per chunk of segments 1..M-1: the sum of
//                                       squares of P_{<=t} q_t over its tokens
//   ores   fp32 [T][H][d_v]             o of segments 1..M-1 from a zero start,
//                                       for the chunks (and channels) whose
//                                       gstart is at least kOresFloor
//   clist  int32 count (16 bytes), then int32 [slots H d_v/128][4]: the
//          (chunk slot, head x 128-channel block, sequence, segment) of the
//          chunks whose output the initial state can still change
struct SplitLayout {
    int M = 1;
    size_t vt0 = 0, vlen = 0, sfin = 0, pbuf = 0, gbuf = 0, sst = 0, rnorm = 0, gstart = 0,
           qtil = 0, qfro = 0, qfro_bytes = 0, ores = 0, clist = 0, end = 0;
};
// Segments for this shape on the current device (1: no split).
int split_segments(int32_t num_seqs, int32_t H, int32_t d_k, int32_t d_v, int32_t chunk);
SplitLayout split_layout(int32_t num_seqs, int64_t total_tokens, int32_t H, int32_t d_k,
                         int32_t d_v, int M);

struct PrefillArgs {
    const void* q;
    const void* k;
    const void* v;
    const void* alpha;   // layout by gate (kda_gate_format)
    const float* beta;
    const float* S0;
    const int32_t* cu_seqlens;
    int32_t num_seqs;
    int64_t total_tokens;
    int32_t H, d_k, d_v;
    kda_dtype dtype;
    int32_t chunk;
    void* o;
    float* S_T;
    int32_t* status;    // device
    int32_t* counter;   // device
    int32_t* order;     // device, [num_seqs]
    int32_t gate = 0;   // kda_gate_format
    int32_t additive = 0;   // additive update of linear attention instead of the delta rule
    // channels the tensor-core kernel hands back (WorkspaceLayout), or null
    uint32_t* redo = nullptr;
};

struct DecodeArgs {
    const void* q;
    const void* k;
    const void* v;
    const void* alpha;   // layout by gate (kda_gate_format)
    const float* beta;
    float* S;
    int32_t B, H, d_k, d_v;
    kda_dtype dtype;
    void* o;
    int32_t gate = 0;    // kda_gate_format
    int32_t additive = 0;   // additive update of linear attention instead of the delta rule
};

// Backward pass (kda_backward.cu).  Buffers appended to the base workspace:
//   ckpt     fp32 [T / 64 + N][H][d_v][d_k]   chunk-start states; chunk c of
//            sequence n (first token t0) in slot t0 / 64 + n + c
//   tbuf     [T / 64 + N][H][d_v / 64] x 16 KB  each chunk's T as bf16 hi/lo
//   dq_part  fp32 [d_v / 64][T][H][d_k]       dq of each 64-row block
//   dk_part  fp32 [d_v / 64][T][H][d_k]
//   db_part  fp32 [d_v / 64][T][H]
//   o_tc     bf16 [T][H][d_v], st_tc fp32 [N][H][d_v][d_k]: scratch outputs of
//            the tensor-core forward that writes ckpt (d_v a multiple of 128);
//            other widths run their own forward sweep and keep T in tbuf
struct BackwardLayout {
    bool tc = false;
    size_t ckpt = 0, tbuf = 0, o_tc = 0, st_tc = 0, dq_part = 0, dk_part = 0, db_part = 0,
           end = 0;
};
BackwardLayout backward_layout(int32_t num_seqs, int64_t total_tokens, int32_t H, int32_t d_v);

struct BackwardArgs {
    const void *q, *k, *v, *dO;   // bf16
    const float *alpha, *beta, *S0, *dS_T;
    const int32_t* cu_seqlens;
    int32_t num_seqs;
    int64_t total_tokens;
    int32_t H, d_v;
    float *dq, *dk, *dv, *dalpha, *dbeta, *dS0;
};

// Launchers; each returns the CUDA error of its launch.
cudaError_t launch_planner(const PrefillArgs& a, cudaStream_t stream, size_t redo_bytes = 0);
cudaError_t launch_prefill_simt(const PrefillArgs& a, cudaStream_t stream);
cudaError_t launch_prefill_tc(const PrefillArgs& a, cudaStream_t stream);
// The portable kernel over the channels the tensor-core kernel handed back in
// a.redo: every (sequence, head, 128-channel block) with a bit set is run again
// from S0, and only the marked channels' o and S_T are written.
cudaError_t launch_prefill_simt_redo(const PrefillArgs& a, cudaStream_t stream);
// The tensor-core prefill that also writes every chunk's start state (fp32
// [slots][H][d_v][d_k], slot t0 / 64 + n + chunk) for the backward pass.
cudaError_t launch_prefill_tc_ckpt(const PrefillArgs& a, float* ckpt, cudaStream_t stream);
// The split form: segment planner, three chunk-kernel launches and the scan of
// the segment maps in between (ws: the workspace base).
cudaError_t launch_prefill_tc_split(const PrefillArgs& a, const SplitLayout& L, char* ws,
                                    cudaStream_t stream);
cudaError_t launch_split_plan(const PrefillArgs& a, const SplitLayout& L, char* ws,
                              cudaStream_t stream);
cudaError_t launch_split_combine(const PrefillArgs& a, const SplitLayout& L, char* ws,
                                 cudaStream_t stream);
// o of segments 1..M-1 += diag(decay from the segment start) S_start P_{<=t} q_t.
cudaError_t launch_split_correct(const PrefillArgs& a, const SplitLayout& L, char* ws,
                                 cudaStream_t stream);
// S_out = diag(g) S_in P + R per (sequence, head) (kda_segment_combine).
cudaError_t launch_segment_combine(const float* S_in, const float* g, const float* P,
                                   const float* R, int32_t N, int32_t H, int32_t d_k,
                                   int32_t d_v, float* S_out, cudaStream_t stream);
bool prefill_tc_supports(const PrefillArgs& a);
// One CTA that runs the prefill kernel's wait-timeout path with nothing to
// wait for (status: the workspace's status word, cleared first).
cudaError_t launch_wait_probe(int32_t* status, uint64_t timeout_ns, cudaStream_t stream);
// The chain kernel and the row-block reduction of the backward pass (ws: the
// workspace base, planner already enqueued).
cudaError_t launch_backward(const BackwardArgs& a, const BackwardLayout& L, char* ws,
                            cudaStream_t stream);
// Gate layouts of the backward pass: the gate expanded per channel (ax) before
// the chain kernel, and the gradient (dax, per channel) reduced to the gate's
// layout after it (a: the sizes and cu_seqlens; status: the planner's word).
cudaError_t launch_gate_expand(const void* gate_in, kda_gate_format gate, const BackwardArgs& a,
                               float* ax, const int32_t* status, cudaStream_t stream);
cudaError_t launch_gate_grad(kda_gate_format gate, const BackwardArgs& a, const float* ax,
                             const float* dax, float* dgate, const int32_t* status,
                             cudaStream_t stream);
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream);
// Blocked Attention Residuals, one layer (attnres.cu; arguments as attnres_layer).
cudaError_t launch_attnres(const void* blocks, int32_t nb, const float* partial,
                           const void* h_last, float* partial_out, void* block_out,
                           const float* q, float scale, int64_t T, int32_t d, kda_dtype dtype,
                           void* h, cudaStream_t stream);

int sm_count();   // of the current device, cached per device

// Validation and dispatch behind kda_prefill / kda_prefill_ex (kda_api.cu).
kda_status prefill_impl(const void* q, const void* k, const void* v, const void* alpha,
                        const float* beta, const float* S0, const int32_t* cu_seqlens,
                        int32_t num_seqs, int64_t total_tokens, int32_t H, int32_t d_k,
                        int32_t d_v, kda_dtype dtype, int32_t chunk, void* o, float* S_T,
                        void* workspace, size_t workspace_bytes, kda_prefill_kernel kernel,
                        kda_stream_t stream, kda_gate_format gate = KDA_GATE_CHANNEL_F32,
                        bool additive = false);

// ---- small device helpers ------------------------------------------------

template <typename T>
struct Elem;

template <>
struct Elem<float> {
    static __device__ __forceinline__ float load(const float* p) { return *p; }
    static __device__ __forceinline__ void store(float* p, float x) { *p = x; }
};

template <>
struct Elem<__nv_bfloat16> {
    static __device__ __forceinline__ float load(const __nv_bfloat16* p) {
        return __bfloat162float(*p);
    }
    static __device__ __forceinline__ void store(__nv_bfloat16* p, float x) {
        *p = __float2bfloat16_rn(x);
    }
};

}  // namespace kda
