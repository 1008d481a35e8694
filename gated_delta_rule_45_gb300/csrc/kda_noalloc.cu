// kda_prefill_noalloc: kda_prefill with a built-in scratch area instead of a
// caller-provided workspace, for callers that cannot allocate device memory.
//
// The scratch is a file-scope __device__ array, so every GPU that loads this
// library holds it (about 768 KB) until
// the process exits.  Host code must not pass the array's name to a kernel:
// on the host that name is only a stand-in for the symbol.  Its device
// address is looked up on every call, with the caller's device and context
// current, through cudaGetSymbolAddress (which allocates nothing).  A symbol's
// address belongs to one CUDA context, so no address is cached: a caller that
// switches between driver contexts, or resets the device, gets the address of
// the module loaded in the context that is current at the call.  The first
// call in a context loads the module there; make it before any stream
// capture.
//
// All calls share the one array.  The planner clears the status word and the
// work counter at the start of every call and rewrites the sequence order, so
// nothing left by the previous call is read; but two calls whose work
// overlaps on the GPU (different streams, no ordering between them) race on
// the array and must not be issued.  The array holds no room for the buffers
// of the sequence-axis split, so this call never splits the sequence axis.
#include "kda_internal.h"

namespace {

// the schedule of KDA_NOALLOC_MAX_SEQS sequences, then room for the channels
// the tensor-core kernel may hand back to the portable one (16 bytes per
// (sequence, head, 128-channel block): up to 16384 such blocks)
constexpr size_t kScheduleBytes =
    (kda::WorkspaceLayout::kOrder + 2 * sizeof(int32_t) * (size_t)KDA_NOALLOC_MAX_SEQS + 255) &
    ~(size_t)255;
constexpr size_t kScratchBytes = kScheduleBytes + 16 * 16384;

static __device__ __align__(256) unsigned char kda_noalloc_scratch[kScratchBytes];

// Device address of the scratch array in the current context.
kda_status scratch_in_current_context(void** out) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, kda_noalloc_scratch) != cudaSuccess || p == nullptr)
        return KDA_ERR_CUDA;
    *out = p;
    return KDA_OK;
}

}  // namespace

extern "C" kda_status kda_prefill_noalloc(const void* q, const void* k, const void* v,
                                          const float* alpha, const float* beta,
                                          const float* S0, const int32_t* cu_seqlens,
                                          int32_t num_seqs, int64_t total_tokens, int32_t H,
                                          int32_t d_k, int32_t d_v, kda_dtype dtype,
                                          int32_t chunk, void* o, float* S_T,
                                          kda_stream_t stream) {
    if (num_seqs > KDA_NOALLOC_MAX_SEQS) return KDA_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    const kda_status st = scratch_in_current_context(&scratch);
    if (st != KDA_OK) return st;
    // kScratchBytes has no room for the buffers of the sequence-axis split, so
    // that is never chosen (prefill_impl splits only when the workspace has room)
    return kda::prefill_impl(q, k, v, alpha, beta, S0, cu_seqlens, num_seqs, total_tokens, H,
                             d_k, d_v, dtype, chunk, o, S_T, scratch, kScratchBytes,
                             KDA_KERNEL_AUTO, stream);
}
