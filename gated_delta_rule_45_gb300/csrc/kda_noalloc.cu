// kda_prefill_noalloc: kda_prefill with a built-in scratch area instead of a
// caller-provided workspace, for callers that cannot allocate device memory.
//
// The scratch is a file-scope __device__ array, so every GPU that loads this
// library holds it (KDA_NOALLOC_MAX_SEQS sequences' worth, about 256 KB) until
// the process exits.  Host code must not pass the array's name to a kernel:
// on the host that name is only a stand-in for the symbol.  Its device
// address is looked up once per device, with that device current, through
// cudaGetSymbolAddress, on the first call made on that device.
//
// All calls share the one array.  The planner clears the status word and the
// work counter at the start of every call and rewrites the sequence order, so
// nothing left by the previous call is read; but two calls whose work
// overlaps on the GPU (different streams, no ordering between them) race on
// the array and must not be issued.
#include "kda_internal.h"

#include <mutex>

namespace {

constexpr int kMaxDevices = 64;
constexpr size_t kScratchBytes =
    (kda::WorkspaceLayout::kOrder + sizeof(int32_t) * (size_t)KDA_NOALLOC_MAX_SEQS + 255) &
    ~(size_t)255;

static __device__ __align__(256) unsigned char kda_noalloc_scratch[kScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device.
kda_status scratch_on_current_device(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return KDA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, kda_noalloc_scratch) != cudaSuccess || p == nullptr)
            return KDA_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
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
    const kda_status st = scratch_on_current_device(&scratch);
    if (st != KDA_OK) return st;
    return kda::prefill_impl(q, k, v, alpha, beta, S0, cu_seqlens, num_seqs, total_tokens, H,
                             d_k, d_v, dtype, chunk, o, S_T, scratch, kScratchBytes,
                             KDA_KERNEL_AUTO, stream);
}
