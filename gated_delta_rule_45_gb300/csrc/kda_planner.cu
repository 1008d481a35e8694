// Varlen planner: validates cu_seqlens on the device and orders sequences
// longest first (ties by index), so that the prefill kernels start the long
// sequential chains first and finish with short ones (longest-processing-time
// scheduling of independent (sequence, head) chains).
//
// The order (-length, index) is a strict total order for any integers, so
// the result is a permutation even for invalid input.  A batch of at most
// kCountMax sequences is ranked by counting, each sequence against all the
// others in shared memory (cheapest at that size).  Otherwise blocks of kRun
// threads each sort kRun sequences with a bitonic network in shared memory; a single
// block writes the order directly.  With more sequences, the blocks write
// sorted runs and a second kernel gives each sequence its rank: its place in
// its own run plus, for every other run, how many of that run's sequences
// come before it (a binary search), O(N log kRun) work per run count.
//
// The same launch clears the tensor-core kernel's fast-decay bitmap (grid
// stride, extra blocks when it is large) and, when it is a single block, the
// status word and work counter (before any check can write the status), so a
// call makes no separate memset launches.
#include "kda_internal.h"

#include <climits>

namespace kda {
namespace {

constexpr int kRun = 1024;          // sequences per sorted run (one block)
constexpr int kRankThreads = 256;
constexpr int kCountMax = 256;      // batches ranked by counting

// a before b in the order: longer first, then lower index
__device__ __forceinline__ bool precedes(int32_t la, int32_t ia, int32_t lb, int32_t ib) {
    return la > lb || (la == lb && ia < ib);
}

__global__ void __launch_bounds__(kRun)
kda_planner_kernel(const int32_t* __restrict__ cu, int32_t num_seqs, int64_t total_tokens,
                   int32_t* __restrict__ status, int32_t* __restrict__ out,
                   uint4* __restrict__ zero, size_t zero_n16, int seq_blocks, bool clear_status) {
    __shared__ int32_t slen[kRun];
    __shared__ int32_t sidx[kRun];
    if (clear_status) {   // single block: status and work counter
        if (threadIdx.x < 2) status[threadIdx.x] = 0;
        __syncthreads();
    }
    for (size_t z = (size_t)blockIdx.x * kRun + threadIdx.x; z < zero_n16;
         z += (size_t)gridDim.x * kRun)
        zero[z] = make_uint4(0u, 0u, 0u, 0u);
    if ((int)blockIdx.x >= seq_blocks) return;   // a block that only clears
    const int tid = threadIdx.x;
    const int i = blockIdx.x * kRun + tid;
    int32_t len = INT_MIN, idx = INT_MAX;   // padding sorts after every sequence
    if (i < num_seqs) {
        const int32_t lo = cu[i], hi = cu[i + 1];
        len = hi - lo;
        idx = i;
        if (hi < lo) atomicExch(status, (int32_t)KDA_ERR_DEVICE_INPUT);
    }
    if (i == 0 && (cu[0] != 0 || (int64_t)cu[num_seqs] > total_tokens))
        atomicExch(status, (int32_t)KDA_ERR_DEVICE_INPUT);
    slen[tid] = len;
    sidx[tid] = idx;
    __syncthreads();
    if (num_seqs <= kCountMax) {   // one block: rank by counting
        if (i < num_seqs) {
            int rank = 0;
            for (int j = 0; j < num_seqs; ++j) rank += precedes(slen[j], sidx[j], len, idx);
            out[rank] = idx;
        }
        return;
    }
    // bitonic sort of the block's kRun keys into the order
    for (int size = 2; size <= kRun; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const int partner = tid ^ stride;
            if (partner > tid) {
                const bool up = (tid & size) == 0;   // this pair's half sorts ascending
                const int32_t la = slen[tid], ia = sidx[tid];
                const int32_t lb = slen[partner], ib = sidx[partner];
                // ascending halves put the earlier key first
                if (up ? precedes(lb, ib, la, ia) : precedes(la, ia, lb, ib)) {
                    slen[tid] = lb; sidx[tid] = ib;
                    slen[partner] = la; sidx[partner] = ia;
                }
            }
            __syncthreads();
        }
    }
    const int base = blockIdx.x * kRun;
    if (base + tid < num_seqs) out[base + tid] = sidx[tid];
}

// Ranks across runs: sequence at place p of run r goes to
// p + sum over runs r' != r of |{keys of r' before it}|.
__global__ void __launch_bounds__(kRankThreads)
kda_planner_rank_kernel(const int32_t* __restrict__ cu, int32_t num_seqs,
                        const int32_t* __restrict__ runs, int32_t* __restrict__ order) {
    const int i = blockIdx.x * kRankThreads + threadIdx.x;
    if (i >= num_seqs) return;
    const int r = i / kRun, p = i % kRun;
    const int32_t idx = runs[i];
    const int32_t len = cu[idx + 1] - cu[idx];
    const int nruns = (num_seqs + kRun - 1) / kRun;
    int64_t rank = p;
    for (int q = 0; q < nruns; ++q) {
        if (q == r) continue;
        const int b = q * kRun, n = min(kRun, num_seqs - b);
        int lo = 0, hi = n;   // first place in run q whose key does not come before ours
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            const int32_t j = runs[b + mid];
            if (precedes(cu[j + 1] - cu[j], j, len, idx)) lo = mid + 1;
            else hi = mid;
        }
        rank += lo;
    }
    order[rank] = idx;
}

}  // namespace

cudaError_t launch_planner(const PrefillArgs& a, cudaStream_t stream, size_t redo_bytes) {
    // status and work counter start at zero on every call, and so does the
    // fast-decay bitmap (a.redo, redo_bytes: a multiple of 16)
    const int seq_blocks = a.num_seqs > 0 ? (a.num_seqs + kRun - 1) / kRun : 0;
    const size_t zero_n16 = a.redo ? redo_bytes / 16 : 0;
    const size_t zero_blocks = (zero_n16 + 4 * kRun - 1) / (4 * kRun);
    int blocks = seq_blocks;
    if ((size_t)blocks < zero_blocks) blocks = zero_blocks < 1024 ? (int)zero_blocks : 1024;
    const bool clear_status = blocks == 1;
    if (!clear_status) {
        const cudaError_t err = cudaMemsetAsync(a.status, 0, 2 * sizeof(int32_t), stream);
        if (err != cudaSuccess || blocks == 0) return err;
    }
    // one run: straight into the order; several: runs after the order, then ranks
    int32_t* runs = seq_blocks > 1 ? a.order + a.num_seqs : a.order;
    kda_planner_kernel<<<blocks, kRun, 0, stream>>>(a.cu_seqlens, a.num_seqs, a.total_tokens,
                                                   a.status, runs, reinterpret_cast<uint4*>(a.redo),
                                                   zero_n16, seq_blocks, clear_status);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess || seq_blocks <= 1) return err;
    kda_planner_rank_kernel<<<(a.num_seqs + kRankThreads - 1) / kRankThreads, kRankThreads, 0,
                              stream>>>(a.cu_seqlens, a.num_seqs, runs, a.order);
    return cudaGetLastError();
}

}  // namespace kda
