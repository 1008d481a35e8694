// Sequence-axis split of the tensor-core prefill, for batches with fewer
// (sequence, head, block) chains than SMs: the segment planner and the scan
// of the segment maps.
//
// Over a segment of tokens the recurrence is affine in its initial state
// ("Kimi (AI)", section "Kimi Delta Attention (KDA)": S_t = diag(alpha_t)
// S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T, with the decay on the
// rows and the projector on the columns):
//   S_end = diag(g) S_start P + R,
// g = prod alpha (per value channel), P = prod (I - beta k k^T) (d_k x d_k),
// R = the state reached from S_start = 0.  The first pass runs segment 0 from
// the true S0 and, for segments 1..M-2, R (from zero) and P (alpha = 1, v = 0,
// S_start = I); this scan then chains the maps; the second pass reruns
// segments 1..M-1 from their true initial states.
#include "kda_internal.h"

namespace kda {

int split_segments(int32_t num_seqs, int32_t H, int32_t d_k, int32_t d_v, int32_t chunk) {
    if (num_seqs <= 0 || H <= 0 || d_k != 128 || d_v % 128 != 0 || chunk != 64) return 1;
    const int64_t chains = (int64_t)num_seqs * H * (d_v / 128);
    const int64_t sms = sm_count();
    if (sms <= 0 || 2 * chains + (int64_t)num_seqs * H > sms) return 1;
    // a pass takes (waves of its items) x (chunks per segment) chunk times: the
    // first pass has (M-1) items per chain plus (M-2) transition items per
    // (sequence, head), the second (M-1) per chain; pick the M in [3, 8] with
    // the fewest waves per segment of the sequence (ties: the smaller M)
    int M = 1;
    double best = 0.0;
    for (int m = 3; m <= 8; ++m) {
        const int64_t p1 = (m - 1) * chains + (int64_t)(m - 2) * num_seqs * H;
        const int64_t p2 = (m - 1) * chains;
        const double cost = (double)((p1 + sms - 1) / sms + (p2 + sms - 1) / sms) / m;
        if (M == 1 || cost < best - 1e-9) {
            M = m;
            best = cost;
        }
    }
    return M;
}

SplitLayout split_layout(int32_t num_seqs, int32_t H, int32_t d_k, int32_t d_v, int M) {
    SplitLayout L;
    L.M = M;
    if (M <= 1 || num_seqs <= 0) return L;
    size_t off = WorkspaceLayout::bytes(num_seqs);
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = (off + bytes + 255) & ~(size_t)255;
        return at;
    };
    const size_t N = (size_t)num_seqs, st = (size_t)H * d_v * d_k * sizeof(float);
    L.vt0 = take(sizeof(int64_t) * M * N);
    L.vlen = take(sizeof(int32_t) * M * N);
    L.sfin = take((M - 1) * N * st);
    L.pbuf = take((M - 2) * N * (size_t)H * d_k * d_k * sizeof(float));
    L.gbuf = take((M - 1) * N * (size_t)H * d_v * sizeof(float));
    L.sst = take((M - 1) * N * st);
    L.end = off;
    return L;
}

namespace {

// Segment j of sequence n = whole chunks [j nc / M, (j + 1) nc / M) of its nc.
__global__ void split_plan_kernel(const int32_t* __restrict__ cu, int N, int M,
                                  int64_t* __restrict__ vt0, int32_t* __restrict__ vlen,
                                  const int32_t* __restrict__ status) {
    if (*status == KDA_ERR_DEVICE_INPUT) return;
    for (int n = blockIdx.x * blockDim.x + threadIdx.x; n < N; n += gridDim.x * blockDim.x) {
        const int64_t t0 = cu[n];
        const int len = cu[n + 1] - cu[n];
        const int nc = (len + 63) / 64;
        for (int j = 0; j < M; ++j) {
            const int c0 = (int)((int64_t)j * nc / M), c1 = (int)((int64_t)(j + 1) * nc / M);
            const int a = 64 * c0, b = min(len, 64 * c1);
            vt0[(size_t)j * N + n] = t0 + a;
            vlen[(size_t)j * N + n] = b - a;
        }
    }
}

constexpr int kB = 128;        // rows and columns of a state block
constexpr int kLd = kB + 4;    // padded row stride in shared memory

// One CTA per (sequence, head, 128-row block): S_1 = S_fin(0);
// S_{j+1} = diag(g_j) S_j P_j + R_j for j = 1..M-2, R_j = S_fin(j).  fp32,
// S and P in shared memory, each thread an 8 x 8 tile of the product.
__global__ void __launch_bounds__(256) split_combine_kernel(
    int N, int H, int d_v, int M, const float* __restrict__ sfin, const float* __restrict__ pbuf,
    const float* __restrict__ gbuf, float* __restrict__ sst, const int32_t* __restrict__ status) {
    if (*status == KDA_ERR_DEVICE_INPUT) return;
    extern __shared__ float sh[];
    float* sS = sh;              // [128][kLd]
    float* sP = sh + kB * kLd;   // [128][kLd]
    const int nvb = d_v / kB;
    const int n = blockIdx.x / (H * nvb), rem = blockIdx.x % (H * nvb);
    const int h = rem / nvb, vb = rem % nvb;
    const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
    // offset of rows vb*128.. of the [v][H][d_v][128] state of virtual sequence v
    auto state = [&](size_t v) { return ((v * H + h) * (size_t)d_v + (size_t)vb * kB) * kB; };
    {
        const float* src = sfin + state((size_t)n);
        float* dst = sst + state((size_t)n);
        for (int e = tid * 4; e < kB * kB; e += 256 * 4) {
            const float4 x = *reinterpret_cast<const float4*>(src + e);
            *reinterpret_cast<float4*>(dst + e) = x;
            float* d = sS + (e / kB) * kLd + e % kB;
            d[0] = x.x; d[1] = x.y; d[2] = x.z; d[3] = x.w;
        }
    }
    for (int j = 1; j <= M - 2; ++j) {
        const size_t v = (size_t)j * N + n;
        const float* P = pbuf + (((v - N) * H + h) * (size_t)kB) * kB;
        for (int e = tid * 4; e < kB * kB; e += 256 * 4) {
            const float4 x = *reinterpret_cast<const float4*>(P + e);
            float* d = sP + (e / kB) * kLd + e % kB;
            d[0] = x.x; d[1] = x.y; d[2] = x.z; d[3] = x.w;
        }
        __syncthreads();
        float acc[8][8] = {};
        for (int k = 0; k < kB; ++k) {
            float a[8], b[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) a[i] = sS[(8 * ty + i) * kLd + k];
#pragma unroll
            for (int c = 0; c < 8; ++c) b[c] = sP[k * kLd + 8 * tx + c];
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int c = 0; c < 8; ++c) acc[i][c] = fmaf(a[i], b[c], acc[i][c]);
        }
        __syncthreads();   // every thread is done reading S_j
        const float* R = sfin + state(v);
        const float* gv = gbuf + (v * H + h) * (size_t)d_v + (size_t)vb * kB;
        float* dst = sst + state(v);   // S_{j+1}: row (j + 1) N + n - N of sst
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int r = 8 * ty + i;
            const float gr = gv[r];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const int col = 8 * tx + c;
                const float x = fmaf(gr, acc[i][c], R[r * kB + col]);
                sS[r * kLd + col] = x;
                dst[r * kB + col] = x;
            }
        }
        __syncthreads();
    }
}

// S_out = diag(g) S_in P + R for every (sequence, head): one CTA per
// (sequence, head, 32-row block); P (d_k x d_k) and the block's rows of S_in
// in shared memory, fp32, each thread 4 rows x up to 4 columns of the product.
// The rows of a block are read before any is written, so S_out may be S_in.
constexpr int kCombRows = 32;
__global__ void __launch_bounds__(256) segment_combine_kernel(
    const float* __restrict__ S_in, const float* __restrict__ g, const float* __restrict__ P,
    const float* __restrict__ R, int H, int d_k, int d_v, float* S_out) {
    extern __shared__ float sh[];
    const int ld = d_k + 1;
    float* sP = sh;                    // [d_k][ld]
    float* sS = sh + (size_t)d_k * ld;   // [kCombRows][ld]
    const int nrb = (d_v + kCombRows - 1) / kCombRows;
    const int nh = blockIdx.x / nrb, rb = blockIdx.x % nrb;
    const int r0 = rb * kCombRows, rows = min(kCombRows, d_v - r0);
    const size_t soff = ((size_t)nh * d_v + r0) * d_k;
    const float* Pm = P + (size_t)nh * d_k * d_k;
    for (int e = threadIdx.x; e < d_k * d_k; e += blockDim.x) sP[(e / d_k) * ld + e % d_k] = Pm[e];
    for (int e = threadIdx.x; e < rows * d_k; e += blockDim.x)
        sS[(e / d_k) * ld + e % d_k] = S_in[soff + e];
    __syncthreads();
    // thread (ty, tx): rows ty, ty + 8, ty + 16, ty + 24; columns tx + 32 c
    const int ty = threadIdx.x >> 5, tx = threadIdx.x & 31;
    for (int c0 = tx; c0 < d_k; c0 += 32) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        for (int k = 0; k < d_k; ++k) {
            const float pk = sP[k * ld + c0];
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[i] = fmaf(sS[(ty + 8 * i) * ld + k], pk, acc[i]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = ty + 8 * i;
            if (r < rows) {
                const size_t e = soff + (size_t)r * d_k + c0;
                S_out[e] = fmaf(g[(size_t)nh * d_v + r0 + r], acc[i], R[e]);
            }
        }
    }
}

}  // namespace

cudaError_t launch_segment_combine(const float* S_in, const float* g, const float* P,
                                   const float* R, int32_t N, int32_t H, int32_t d_k,
                                   int32_t d_v, float* S_out, cudaStream_t stream) {
    const int smem = (d_k + kCombRows) * (d_k + 1) * (int)sizeof(float);
    cudaError_t err = cudaFuncSetAttribute(segment_combine_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    const int64_t blocks = (int64_t)N * H * ((d_v + kCombRows - 1) / kCombRows);
    if (blocks == 0) return cudaSuccess;
    segment_combine_kernel<<<(unsigned)blocks, 256, smem, stream>>>(S_in, g, P, R, H, d_k, d_v,
                                                                    S_out);
    return cudaGetLastError();
}

cudaError_t launch_split_plan(const PrefillArgs& a, const SplitLayout& L, char* ws,
                              cudaStream_t stream) {
    const int threads = 256, blocks = (a.num_seqs + threads - 1) / threads;
    split_plan_kernel<<<blocks, threads, 0, stream>>>(
        a.cu_seqlens, a.num_seqs, L.M, reinterpret_cast<int64_t*>(ws + L.vt0),
        reinterpret_cast<int32_t*>(ws + L.vlen), a.status);
    return cudaGetLastError();
}

cudaError_t launch_split_combine(const PrefillArgs& a, const SplitLayout& L, char* ws,
                                 cudaStream_t stream) {
    const int smem = 2 * kB * kLd * (int)sizeof(float);
    cudaError_t err = cudaFuncSetAttribute(split_combine_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    const int blocks = a.num_seqs * a.H * (a.d_v / kB);
    split_combine_kernel<<<blocks, 256, smem, stream>>>(
        a.num_seqs, a.H, a.d_v, L.M, reinterpret_cast<const float*>(ws + L.sfin),
        reinterpret_cast<const float*>(ws + L.pbuf), reinterpret_cast<const float*>(ws + L.gbuf),
        reinterpret_cast<float*>(ws + L.sst), a.status);
    return cudaGetLastError();
}

}  // namespace kda
