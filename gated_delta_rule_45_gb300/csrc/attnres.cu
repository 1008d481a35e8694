// Blocked Attention Residuals: one layer's input as softmax attention over
// depth ("Kimi (AI)", section "Attention Residuals").  For every token t,
//
//   h[t] = sum_j softmax_j(scale * q . s_j[t]) s_j[t]
//
// over the sources s_0..s_{m-1}: the stored sums of the finished blocks
// (block 0 is the network input), then the running sum P = partial + h_last
// of the current block's earlier outputs (or, at a block's first layer, of the
// block just finished), formed on the fly in fp32 and optionally written back
// in fp32 and in the storage type.
//
// HBM-bound: each source is read once per token (the second read, for the
// weighted sum, is served by L1/L2).  One CTA per token at a time, every
// thread a 16-byte piece of the hidden vector, the pieces of up to four
// stored blocks in flight together; per-source dot products are reduced with
// warp shuffles, then across warps in shared memory; the softmax is fp32.
#include "attnres.h"
#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kMaxSources = 64;
constexpr int kThreads = 256;

// One 16-byte piece of a row: loaded raw through the read-only path, then
// unpacked to floats; stored from floats.
template <typename T>
struct Vec;
template <>
struct Vec<__nv_bfloat16> {
    static constexpr int N = 8;
    static __device__ __forceinline__ void unpack(const uint4 u, float (&x)[8]) {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[2 * i] = __uint_as_float(w[i] << 16);
            x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
    static __device__ __forceinline__ void store(__nv_bfloat16* p, const float (&x)[8]) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 b = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
            w[i] = *reinterpret_cast<const uint32_t*>(&b);
        }
        *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
    }
};
template <>
struct Vec<float> {
    static constexpr int N = 4;
    static __device__ __forceinline__ void unpack(const uint4 u, float (&x)[4]) {
        x[0] = __uint_as_float(u.x); x[1] = __uint_as_float(u.y);
        x[2] = __uint_as_float(u.z); x[3] = __uint_as_float(u.w);
    }
    static __device__ __forceinline__ void store(float* p, const float (&x)[4]) {
        *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]);
    }
};

template <typename T>
__device__ __forceinline__ uint4 ld_raw(const T* p) {
    return __ldg(reinterpret_cast<const uint4*>(p));
}

// V fp32 values of the running sum: plain accesses, since the kernel may write
// where it reads (partial_out == partial).
template <int V>
__device__ __forceinline__ void ld_f32(const float* p, float (&x)[V]) {
#pragma unroll
    for (int e = 0; e < V; e += 4) {
        const float4 u = *reinterpret_cast<const float4*>(p + e);
        x[e] = u.x; x[e + 1] = u.y; x[e + 2] = u.z; x[e + 3] = u.w;
    }
}
template <int V>
__device__ __forceinline__ void st_f32(float* p, const float (&x)[V]) {
#pragma unroll
    for (int e = 0; e < V; e += 4)
        *reinterpret_cast<float4*>(p + e) = make_float4(x[e], x[e + 1], x[e + 2], x[e + 3]);
}

// A contiguous row brought into L2 by the bulk-copy unit (no registers, no
// completion to wait for).  The address and the size are multiples of 16 bytes.
__device__ __forceinline__ void l2_prefetch_row(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

struct AttnResParams {
    const void* blocks;
    const float* partial;
    const void* h_last;
    float* partial_out;
    void* block_out;
    const float* q;
    void* h;
    int64_t T;
    int32_t d, nb;
    float scale;
};

constexpr int kBatch = 4;   // stored blocks whose pieces are in flight together
static_assert(kBatch == 4, "the warp reduce-scatter of pass 1 is written for four sources");
constexpr int kCtasPerSm = 4;   // resident CTAs: 64 registers a thread

template <typename T>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) attnres_kernel(const AttnResParams p) {
    constexpr int V = Vec<T>::N;
    __shared__ float red[kThreads / 32][kMaxSources];
    __shared__ float wgt[kMaxSources];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nwarps = blockDim.x >> 5;
    const bool has_p = p.partial || p.h_last;
    const int nb = p.nb;
    const int m = nb + (has_p ? 1 : 0);
    const int pieces = p.d / V;
    const T* blocks = static_cast<const T*>(p.blocks);
    const float* partial = p.partial;
    const T* h_last = static_cast<const T*>(p.h_last);
    float* partial_out = p.partial_out;
    T* block_out = static_cast<T*>(p.block_out);
    T* hout = static_cast<T*>(p.h);
    const size_t plane = (size_t)p.T * p.d;

    for (int64_t t = blockIdx.x; t < p.T; t += gridDim.x) {
        const size_t row = (size_t)t * p.d;
        {   // the next token's source rows: one bulk L2 prefetch per source, so that
            // they stream in from HBM while this token's dependent rounds run
            const int64_t tn = t + gridDim.x;
            const size_t nrow = (size_t)tn * p.d;
            for (int j = tid; tn < p.T && j < nb + 2; j += blockDim.x) {
                const void* src = nullptr;
                uint32_t bytes = (uint32_t)(p.d * sizeof(T));
                if (j < nb) src = blocks + (size_t)j * plane + nrow;
                else if (j == nb) { src = partial ? partial + nrow : nullptr; bytes = (uint32_t)(p.d * 4); }
                else src = h_last ? h_last + nrow : nullptr;
                if (src) l2_prefetch_row(src, bytes);
            }
        }
        // the running sum partial + h_last (partial may be the output buffer itself)
        auto running = [&](int c, float (&x)[V]) {
            float y[V];
#pragma unroll
            for (int e = 0; e < V; ++e) x[e] = 0.f;
            if (partial) {
                ld_f32<V>(partial + row + (size_t)c * V, y);
#pragma unroll
                for (int e = 0; e < V; ++e) x[e] += y[e];
            }
            if (h_last) {
                Vec<T>::unpack(ld_raw(h_last + row + (size_t)c * V), y);
#pragma unroll
                for (int e = 0; e < V; ++e) x[e] += y[e];
            }
        };
        auto qpiece = [&](int c, float (&qv)[V]) {
#pragma unroll
            for (int e = 0; e < V; e += 4) {
                const float4 qq = __ldg(reinterpret_cast<const float4*>(p.q + (size_t)c * V + e));
                qv[e] = qq.x; qv[e + 1] = qq.y; qv[e + 2] = qq.z; qv[e + 3] = qq.w;
            }
        };
        // pass 1: q . s_j, kBatch stored blocks at a time with their loads in flight together
        for (int j0 = 0; j0 < nb; j0 += kBatch) {
            float acc[kBatch];
#pragma unroll
            for (int jj = 0; jj < kBatch; ++jj) acc[jj] = 0.f;
            for (int c = tid; c < pieces; c += blockDim.x) {
                uint4 raw[kBatch];
#pragma unroll
                for (int jj = 0; jj < kBatch; ++jj)
                    if (j0 + jj < nb) raw[jj] = ld_raw(blocks + (size_t)(j0 + jj) * plane + row + (size_t)c * V);
                float qv[V];
                qpiece(c, qv);
#pragma unroll
                for (int jj = 0; jj < kBatch; ++jj) {
                    if (j0 + jj < nb) {
                        float x[V];
                        Vec<T>::unpack(raw[jj], x);
#pragma unroll
                        for (int e = 0; e < V; ++e) acc[jj] = fmaf(x[e], qv[e], acc[jj]);
                    }
                }
            }
            // reduce-scatter of the four sums over the warp: after the exchanges
            // across 16 and 8 lanes each lane carries one source's partial sum,
            // and lane 8 v ends with source v's total
            const bool hi16 = lane & 16, hi8 = lane & 8;
            const float b0 = (hi16 ? acc[2] : acc[0]) +
                             __shfl_xor_sync(0xffffffffu, hi16 ? acc[0] : acc[2], 16);
            const float b1 = (hi16 ? acc[3] : acc[1]) +
                             __shfl_xor_sync(0xffffffffu, hi16 ? acc[1] : acc[3], 16);
            float a = (hi8 ? b1 : b0) + __shfl_xor_sync(0xffffffffu, hi8 ? b0 : b1, 8);
#pragma unroll
            for (int o = 4; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
            if ((lane & 7) == 0 && j0 + (lane >> 3) < nb) red[warp][j0 + (lane >> 3)] = a;
        }
        if (has_p) {   // the running sum, stored on the way
            float acc = 0.f;
            for (int c = tid; c < pieces; c += blockDim.x) {
                float x[V], qv[V];
                running(c, x);
                if (partial_out) st_f32<V>(partial_out + row + (size_t)c * V, x);
                if (block_out) Vec<T>::store(block_out + row + (size_t)c * V, x);
                qpiece(c, qv);
#pragma unroll
                for (int e = 0; e < V; ++e) acc = fmaf(x[e], qv[e], acc);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
            if (lane == 0) red[warp][nb] = acc;
        }
        __syncthreads();
        if (warp == 0) {   // softmax over the m logits, two per lane
            float l0 = -INFINITY, l1 = -INFINITY;
            if (lane < m) {
                float s = 0.f;
                for (int w = 0; w < nwarps; ++w) s += red[w][lane];
                l0 = p.scale * s;
            }
            if (lane + 32 < m) {
                float s = 0.f;
                for (int w = 0; w < nwarps; ++w) s += red[w][lane + 32];
                l1 = p.scale * s;
            }
            float mx = fmaxf(l0, l1);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            const float e0 = lane < m ? __expf(l0 - mx) : 0.f;
            const float e1 = lane + 32 < m ? __expf(l1 - mx) : 0.f;
            float sum = e0 + e1;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
            const float inv = 1.f / sum;
            if (lane < m) wgt[lane] = e0 * inv;
            if (lane + 32 < m) wgt[lane + 32] = e1 * inv;
        }
        __syncthreads();
        // pass 2: the weighted sum, kBatch stored blocks at a time, then the running sum
        for (int c = tid; c < pieces; c += blockDim.x) {
            float o[V];
#pragma unroll
            for (int e = 0; e < V; ++e) o[e] = 0.f;
            for (int j0 = 0; j0 < nb; j0 += kBatch) {
                uint4 raw[kBatch];
#pragma unroll
                for (int jj = 0; jj < kBatch; ++jj)
                    if (j0 + jj < nb) raw[jj] = ld_raw(blocks + (size_t)(j0 + jj) * plane + row + (size_t)c * V);
#pragma unroll
                for (int jj = 0; jj < kBatch; ++jj) {
                    if (j0 + jj < nb) {
                        float x[V];
                        Vec<T>::unpack(raw[jj], x);
                        const float w = wgt[j0 + jj];
#pragma unroll
                        for (int e = 0; e < V; ++e) o[e] = fmaf(w, x[e], o[e]);
                    }
                }
            }
            if (has_p) {
                float x[V];
                if (partial_out) ld_f32<V>(partial_out + row + (size_t)c * V, x);
                else running(c, x);
                const float w = wgt[nb];
#pragma unroll
                for (int e = 0; e < V; ++e) o[e] = fmaf(w, x[e], o[e]);
            }
            Vec<T>::store(hout + row + (size_t)c * V, o);
        }
        // No barrier here: the next token writes red only after passing this
        // token's second barrier (warp 0 has read red by then), and rewrites wgt
        // only after its own first barrier (every thread has read wgt by then).
    }
}

}  // namespace

cudaError_t launch_attnres(const void* blocks, int32_t nb, const float* partial,
                           const void* h_last, float* partial_out, void* block_out,
                           const float* q, float scale, int64_t T, int32_t d, kda_dtype dtype,
                           void* h, cudaStream_t stream) {
    AttnResParams p{blocks, partial, h_last, partial_out, block_out, q, h, T, d, nb, scale};
    const int vec = dtype == KDA_BF16 ? 8 : 4;
    int threads = (d / vec + 31) / 32 * 32;
    if (threads > kThreads) threads = kThreads;
    const int sms = sm_count();
    const int64_t grid64 = T < (int64_t)sms * kCtasPerSm ? T : (int64_t)sms * kCtasPerSm;
    const int grid = grid64 > 0 ? (int)grid64 : 1;
    if (dtype == KDA_BF16)
        attnres_kernel<__nv_bfloat16><<<grid, threads, 0, stream>>>(p);
    else
        attnres_kernel<float><<<grid, threads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace kda
