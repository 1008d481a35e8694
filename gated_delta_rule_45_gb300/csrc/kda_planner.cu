// Varlen planner: validates cu_seqlens on the device and orders sequences
// longest first (ties by index), so that the prefill kernels start the long
// sequential chains first and finish with short ones (longest-processing-time
// scheduling of independent (sequence, head) chains).
//
// One thread per sequence computes the sequence's rank in the order
// (-length, index) by scanning all lengths in shared-memory tiles, then
// writes order[rank] = its index.  The comparison is a strict total order for
// any integers, so the ranks always form a permutation, even for invalid input.
//
// The same launch clears the tensor-core kernel's fast-decay bitmap (grid
// stride, extra blocks when it is large) and, when it is a single block, the
// status word and work counter (before any check can write the status), so a
// call makes no separate memset launches.
#include "kda_internal.h"

#include <climits>

namespace kda {
namespace {

constexpr int kPlannerThreads = 256;

__global__ void __launch_bounds__(kPlannerThreads)
kda_planner_kernel(const int32_t* __restrict__ cu, int32_t num_seqs, int64_t total_tokens,
                   int32_t* __restrict__ status, int32_t* __restrict__ order,
                   uint4* __restrict__ zero, size_t zero_n16, int seq_blocks, bool clear_status) {
    __shared__ int32_t lens[kPlannerThreads];
    if (clear_status) {   // single block: status and work counter
        if (threadIdx.x < 2) status[threadIdx.x] = 0;
        __syncthreads();
    }
    for (size_t z = (size_t)blockIdx.x * kPlannerThreads + threadIdx.x; z < zero_n16;
         z += (size_t)gridDim.x * kPlannerThreads)
        zero[z] = make_uint4(0u, 0u, 0u, 0u);
    if ((int)blockIdx.x >= seq_blocks) return;   // a block that only clears
    const int i = blockIdx.x * kPlannerThreads + threadIdx.x;
    int32_t my_len = 0;
    if (i < num_seqs) {
        const int32_t lo = cu[i], hi = cu[i + 1];
        my_len = hi - lo;
        if (hi < lo) atomicExch(status, (int32_t)KDA_ERR_DEVICE_INPUT);
    }
    if (i == 0 && (cu[0] != 0 || (int64_t)cu[num_seqs] > total_tokens))
        atomicExch(status, (int32_t)KDA_ERR_DEVICE_INPUT);

    int32_t rank = 0;
    for (int j0 = 0; j0 < num_seqs; j0 += kPlannerThreads) {
        const int j = j0 + threadIdx.x;
        lens[threadIdx.x] = j < num_seqs ? cu[j + 1] - cu[j] : INT_MIN;
        __syncthreads();
        const int cnt = min(kPlannerThreads, num_seqs - j0);
        for (int jj = 0; jj < cnt; ++jj) {
            const int32_t L = lens[jj];
            rank += (L > my_len) || (L == my_len && j0 + jj < i);
        }
        __syncthreads();
    }
    if (i < num_seqs) order[rank] = i;
}

}  // namespace

cudaError_t launch_planner(const PrefillArgs& a, cudaStream_t stream, size_t redo_bytes) {
    // status and work counter start at zero on every call, and so does the
    // fast-decay bitmap (a.redo, redo_bytes: a multiple of 16)
    const int seq_blocks = a.num_seqs > 0 ? (a.num_seqs + kPlannerThreads - 1) / kPlannerThreads : 0;
    const size_t zero_n16 = a.redo ? redo_bytes / 16 : 0;
    const size_t zero_blocks = (zero_n16 + 4 * kPlannerThreads - 1) / (4 * kPlannerThreads);
    int blocks = seq_blocks;
    if ((size_t)blocks < zero_blocks) blocks = zero_blocks < 1024 ? (int)zero_blocks : 1024;
    const bool clear_status = blocks == 1;
    if (!clear_status) {
        const cudaError_t err = cudaMemsetAsync(a.status, 0, 2 * sizeof(int32_t), stream);
        if (err != cudaSuccess || blocks == 0) return err;
    }
    kda_planner_kernel<<<blocks, kPlannerThreads, 0, stream>>>(
        a.cu_seqlens, a.num_seqs, a.total_tokens, a.status, a.order,
        reinterpret_cast<uint4*>(a.redo), zero_n16, seq_blocks, clear_status);
    return cudaGetLastError();
}

}  // namespace kda
