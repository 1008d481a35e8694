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
// R = the state reached from S_start = 0.  The same holds for every token t
// of the segment: the output is affine in S_start,
//   o_t = o_t(from zero) + G_t * (S_start P_{<=t} q_t),
// with G_t = prod alpha from the segment start through t (per channel) and
// P_{<=t} the product of the segment's (I - beta k k^T) through t.
//
// One pass of the chunk kernel runs segment 0 from the true S0 (its o is
// final) and, for segments 1..M-1, the segment from zero (o from zero, R,
// g, G at each chunk start) and the transition from S_start = I with
// alpha = 1 and v = 0 (P, and its outputs P_{<=t} q_t).  The scan below
// chains the maps into each segment's true initial state and S_T; the
// correction kernels then add each segment's G_t * S_start P_{<=t} q_t to o,
// only where it can change the stored value.
#include "kda_internal.h"

#include <cfloat>

namespace kda {

int split_segments(int32_t num_seqs, int32_t H, int32_t d_k, int32_t d_v, int32_t chunk) {
    if (num_seqs <= 0 || H <= 0 || d_k != 128 || d_v % 128 != 0 || chunk != 64) return 1;
    const int64_t chains = (int64_t)num_seqs * H * (d_v / 128);
    const int64_t trans = (int64_t)num_seqs * H;
    const int64_t sms = sm_count();
    if (sms <= 0 || 2 * chains + trans > sms) return 1;
    // the pass has M items per chain and M - 1 transition items per (sequence,
    // head); it takes (waves of its items) x (chunks per segment) chunk
    // times: pick the M in [2, 16] with the fewest waves per segment of the
    // sequence (ties: the smaller M)
    int M = 1;
    double best = 0.0;
    for (int m = 2; m <= 16; ++m) {
        const int64_t items = m * chains + (m - 1) * trans;
        const double cost = (double)((items + sms - 1) / sms) / m;
        if (M == 1 || cost < best - 1e-9) {
            M = m;
            best = cost;
        }
    }
    return M;
}

SplitLayout split_layout(int32_t num_seqs, int64_t total_tokens, int32_t H, int32_t d_k,
                         int32_t d_v, int M) {
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
    const size_t T = total_tokens > 0 ? (size_t)total_tokens : 0;
    const size_t slots = T / 64 + N + 1;
    L.vt0 = take(sizeof(int64_t) * M * N);
    L.vlen = take(sizeof(int32_t) * M * N);
    L.sfin = take(M * N * st);
    L.pbuf = take((M - 1) * N * (size_t)H * d_k * d_k * sizeof(float));
    L.gbuf = take(M * N * (size_t)H * d_v * sizeof(float));
    L.sst = take((M - 1) * N * st);
    L.rnorm = take((M - 1) * N * (size_t)H * d_v * sizeof(float));
    L.gstart = take(slots * (size_t)H * d_v * sizeof(float));
    L.qtil = take(T * (size_t)H * d_k * sizeof(float));
    L.qfro_bytes = slots * (size_t)H * sizeof(float);
    L.qfro = take(L.qfro_bytes);
    L.ores = take(T * (size_t)H * d_v * sizeof(float));
    // the correction's work list: a count, then (slot, head-block) pairs
    L.clist = take(16 + sizeof(int32_t) * 4 * slots * (size_t)H * (d_v / 128));
    L.end = off;
    return L;
}

namespace {

// Segment j of sequence n = whole chunks [j nc / M, (j + 1) nc / M) of its nc.
__global__ void split_plan_kernel(const int32_t* __restrict__ cu, int N, int M,
                                  int64_t* __restrict__ vt0, int32_t* __restrict__ vlen,
                                  int32_t* __restrict__ ccount,
                                  const int32_t* __restrict__ status) {
    if (blockIdx.x == 0 && threadIdx.x == 0) *ccount = 0;   // the correction list
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
// S_{j+1} = diag(g_j) S_j P_j + R_j for j = 1..M-1, R_j = S_fin(j); S_M is the
// sequence's S_T.  fp32, S and P in shared memory, each thread an 8 x 8 tile
// of the product.  S_1..S_{M-1} go to sst with the norms of their rows.
__global__ void __launch_bounds__(256) split_combine_kernel(
    int N, int H, int d_v, int M, const float* __restrict__ sfin, const float* __restrict__ pbuf,
    const float* __restrict__ gbuf, float* __restrict__ sst, float* __restrict__ rnorm,
    float* __restrict__ S_T, const int32_t* __restrict__ status) {
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
    for (int j = 1; j <= M - 1; ++j) {
        const size_t v = (size_t)j * N + n;
        const float* P = pbuf + (((v - N) * H + h) * (size_t)kB) * kB;
        for (int e = tid * 4; e < kB * kB; e += 256 * 4) {
            const float4 x = *reinterpret_cast<const float4*>(P + e);
            float* d = sP + (e / kB) * kLd + e % kB;
            d[0] = x.x; d[1] = x.y; d[2] = x.z; d[3] = x.w;
        }
        __syncthreads();
        if (tid < kB) {   // norms of the rows of S_j, the initial state of segment j
            float acc = 0.f;
            for (int k = 0; k < kB; ++k) acc = fmaf(sS[tid * kLd + k], sS[tid * kLd + k], acc);
            rnorm[((v - N) * H + h) * (size_t)d_v + (size_t)vb * kB + tid] = sqrtf(acc);
        }
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
        // S_{j+1}: row j N + n of sst, or S_T after the last segment
        float* dst = j < M - 1 ? sst + state(v) : S_T + state((size_t)n);
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

// Chunk slot s (as laid out in SplitLayout::gstart) -> sequence n, chunk c
// within it and its segment j; false if s holds no chunk of a segment j >= 1.
__device__ bool slot_chunk(const int32_t* __restrict__ cu, int N, int M,
                           const int64_t* __restrict__ vt0, const int32_t* __restrict__ vlen,
                           int64_t s, int& n, int& c, int& j) {
    int lo = 0, hi = N - 1;   // the largest n with cu[n] / 64 + n <= s (increasing in n)
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((int64_t)cu[mid] / 64 + mid <= s) lo = mid;
        else hi = mid - 1;
    }
    n = lo;
    const int64_t cc = s - ((int64_t)cu[n] / 64 + n);
    const int len = cu[n + 1] - cu[n];
    if (cc < 0 || cc >= (len + 63) / 64) return false;
    c = (int)cc;
    const int64_t t0 = cu[n] + 64 * cc;
    for (j = 1; j < M; ++j) {
        const int64_t a = vt0[(size_t)j * N + n];
        if (t0 >= a && t0 < a + vlen[(size_t)j * N + n]) return true;
    }
    return false;   // segment 0: its o is exact
}

// One warp per (chunk slot, head, 128-channel block): the chunk is listed for
// the correction unless, in every row, the decay from the segment start is
// below the smallest normal float or the state's row is zero.  (A product of
// alphas that reached the denormals can stay at the smallest one for good.)
__global__ void __launch_bounds__(256) split_select_kernel(
    const int32_t* __restrict__ cu, int N, int M, int H, int d_v, int64_t slots,
    const int64_t* __restrict__ vt0, const int32_t* __restrict__ vlen,
    const float* __restrict__ gstart, const float* __restrict__ rnorm,
    int32_t* __restrict__ ccount, int4* __restrict__ clist, const int32_t* __restrict__ status) {
    if (*status == KDA_ERR_DEVICE_INPUT) return;
    const int lane = threadIdx.x & 31;
    const int nvb = d_v / kB;
    const int64_t items = slots * H * nvb;
    for (int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; w < items;
         w += ((int64_t)gridDim.x * blockDim.x) >> 5) {
        const int64_t s = w / (H * nvb);
        const int hv = (int)(w % (H * nvb)), h = hv / nvb, vb = hv % nvb;
        int n, c, j;
        if (!slot_chunk(cu, N, M, vt0, vlen, s, n, c, j)) continue;   // uniform over the warp
        const float* gs = gstart + ((size_t)s * H + h) * d_v + (size_t)vb * kB;
        const float* rn = rnorm + ((((size_t)(j - 1) * N + n) * H + h) * d_v) + (size_t)vb * kB;
        bool live = false;
#pragma unroll
        for (int i = 0; i < 4; ++i)
            live |= !(gs[lane + 32 * i] < FLT_MIN) && !(rn[lane + 32 * i] == 0.f);
        if (__any_sync(0xffffffffu, live) && lane == 0) {
            const int at = atomicAdd(ccount, 1);
            clist[at] = make_int4((int)s, hv, n, j);
        }
    }
}

constexpr int kQld = kB + 4;   // row stride of the q~ tile (16-byte rows)
constexpr int kCorrThreads = 512;

// Persistent: each CTA takes listed chunks in turn.  Thread (r, quarter):
// value channel r of the block, tokens 16 quarter .. 16 quarter + 15.
//   G_t,r   = gstart_r * prod_{i <= t} alpha_i,r  <= gstart_r  (alpha <= 1)
//   bound   = gstart_r * |S_start row r| * |Q~|_F >= |G_t,r (S_start q~_t)_r|,
// |Q~|_F the Frobenius norm of the chunk's q~ (accumulated by the transition
// items), so this first test reads only o; a chunk it keeps is tested again
// with each token's own |q~_t| (reading q~) before anything is computed.
// o holds bf16(o from zero) already.  If bound <= 2^-20 |o_t,r| for every
// element, the share is below 2^-12 of half a bf16 ulp of the value, so the
// stored value is the rounding of the exact one except in the rare case of
// a value within that distance of a rounding boundary; the chunk is left as
// it is.  Otherwise alpha is read and
// o_t,r = bf16(o from zero + G_t,r (S_start q~_t)_r), with o from zero in
// fp32 (ores) where the chunk kernel kept it (gstart_r >= kOresFloor), else
// the bf16 value (where the decay is below kOresFloor the share is small
// beside it, so the second rounding is rare and one ulp).
__global__ void __launch_bounds__(kCorrThreads, 2) split_correct_kernel(
    int N, int H, int d_v, const float* __restrict__ alpha, const float* __restrict__ qtil,
    const float* __restrict__ gstart, const float* __restrict__ sst,
    const float* __restrict__ rnorm, const float* __restrict__ qfro,
    const int32_t* __restrict__ cu, const int32_t* __restrict__ ccount,
    const int4* __restrict__ clist,
    const float* __restrict__ ores, __nv_bfloat16* __restrict__ o,
    const int32_t* __restrict__ status) {
    if (*status == KDA_ERR_DEVICE_INPUT) return;
    extern __shared__ float sh[];
    float* sQ = sh;                  // [64][kQld]
    float* sN = sQ + 64 * kQld;      // [64] norms of the q~ rows
    float* sTot = sN + 64;           // [4][128] products of alpha over each token quarter
    float* sS = sTot + 4 * kB;       // [128][kB + 1] rows of the initial state
    const int tid = threadIdx.x, r = tid & (kB - 1), qt = tid >> 7;
    const int nvb = d_v / kB;
    const int count = *ccount;
    const int64_t ostride = (int64_t)H * d_v, qstride = (int64_t)H * kB;
    for (int it = blockIdx.x; it < count; it += gridDim.x) {
        const int4 e = clist[it];
        const int h = e.y / nvb, vb = e.y % nvb, n = e.z, j = e.w;
        const int64_t base = cu[n];
        const int c = e.x - (int)(base / 64) - n;
        const int64_t t0 = base + 64 * (int64_t)c;
        const int nvalid = min(64, cu[n + 1] - (int)base - 64 * c);
        const int ch = vb * kB + r;
        const size_t srow = (((size_t)(j - 1) * N + n) * H + h) * d_v + ch;   // row of sst / rnorm
        __syncthreads();   // the previous item's tiles are no longer read
        const float* arow = alpha + t0 * ostride + (int64_t)h * d_v + ch;
        __nv_bfloat16* orow = o + t0 * ostride + (int64_t)h * d_v + ch;
        const float g0 = gstart[((size_t)e.x * H + h) * d_v + ch];
        // |q~_t| <= the chunk's Frobenius norm of q~; alpha <= 1, so the decay
        // at every token of the chunk is at most g0
        const float b0 = g0 * rnorm[srow] * sqrtf(qfro[(size_t)e.x * H + h]);
        bool need = false;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int t = 16 * qt + i;
            if (t < nvalid)
                need |= !(b0 <= 0x1p-20f * fabsf(__bfloat162float(orow[t * ostride])));
        }
        if (!__syncthreads_or(need)) continue;
        {   // the q~ tile: all four loads of a thread in flight together
            float4 q[64 * (kB / 4) / kCorrThreads];
#pragma unroll
            for (int u = 0; u < 64 * (kB / 4) / kCorrThreads; ++u) {
                const int x = tid + u * kCorrThreads, t = x / (kB / 4), k4 = x % (kB / 4);
                q[u] = t < nvalid ? *reinterpret_cast<const float4*>(qtil + (t0 + t) * qstride +
                                                                     (int64_t)h * kB + 4 * k4)
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < 64 * (kB / 4) / kCorrThreads; ++u) {
                const int x = tid + u * kCorrThreads, t = x / (kB / 4), k4 = x % (kB / 4);
                *reinterpret_cast<float4*>(sQ + t * kQld + 4 * k4) = q[u];
            }
        }
        __syncthreads();
        {   // norms of the q~ rows: 8 threads per token
            const int t = tid >> 3, part = tid & 7;
            float acc = 0.f;
#pragma unroll
            for (int k = 0; k < 16; ++k) acc = fmaf(sQ[t * kQld + 16 * part + k], sQ[t * kQld + 16 * part + k], acc);
            acc += __shfl_xor_sync(0xffffffffu, acc, 1);
            acc += __shfl_xor_sync(0xffffffffu, acc, 2);
            acc += __shfl_xor_sync(0xffffffffu, acc, 4);
            if (part == 0) sN[t] = sqrtf(acc);
        }
        __syncthreads();
        {   // the same test with each token's own |q~_t|
            const float b1 = g0 * rnorm[srow];
            need = false;
#pragma unroll 4
            for (int i = 0; i < 16; ++i) {
                const int t = 16 * qt + i;
                if (t < nvalid)
                    need |= !(b1 * sN[t] <= 0x1p-20f * fabsf(__bfloat162float(orow[t * ostride])));
            }
        }
        if (!__syncthreads_or(need)) continue;
        {   // the block's rows of S_start, coalesced, all loads in flight together
            const float4* Sg = reinterpret_cast<const float4*>(sst + (srow - r) * kB);
#pragma unroll 1
            for (int h2 = 0; h2 < 2; ++h2) {   // two rounds of four loads
                float4 v[kB * kB / 8 / kCorrThreads];
#pragma unroll
                for (int u = 0; u < kB * kB / 8 / kCorrThreads; ++u)
                    v[u] = Sg[tid + (u + h2 * (kB * kB / 8 / kCorrThreads)) * kCorrThreads];
#pragma unroll
                for (int u = 0; u < kB * kB / 8 / kCorrThreads; ++u) {
                    const int x = tid + (u + h2 * (kB * kB / 8 / kCorrThreads)) * kCorrThreads;
                    float* d = sS + (x / (kB / 4)) * (kB + 1) + 4 * (x % (kB / 4));
                    d[0] = v[u].x; d[1] = v[u].y; d[2] = v[u].z; d[3] = v[u].w;
                }
            }
        }
        __syncthreads();
        float y[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) y[i] = 0.f;
#pragma unroll 2
        for (int k4 = 0; k4 < kB / 4; ++k4) {
            const float* sr = sS + r * (kB + 1) + 4 * k4;
            const float s0 = sr[0], s1 = sr[1], s2 = sr[2], s3 = sr[3];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float4 q = *reinterpret_cast<const float4*>(sQ + (16 * qt + i) * kQld + 4 * k4);
                y[i] = fmaf(q.x, s0, fmaf(q.y, s1, fmaf(q.z, s2, fmaf(q.w, s3, y[i]))));
            }
        }
        // the decay: this quarter's running product of alpha after the earlier quarters'
        float a16[16], run = 1.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int t = 16 * qt + i;
            a16[i] = t < nvalid ? arow[t * ostride] : 1.f;
            run *= a16[i];
        }
        __syncthreads();   // every thread is done with the state tile
        sTot[qt * kB + r] = run;
        __syncthreads();
        float pre = g0;
        for (int q = 0; q < qt; ++q) pre *= sTot[q * kB + r];
        const float* orr = ores + t0 * ostride + (int64_t)h * d_v + ch;
        const bool exact = g0 >= kOresFloor;   // the zero-start o was kept in fp32
        float G = pre;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int t = 16 * qt + i;
            if (t < nvalid) {
                G *= a16[i];
                const float base = exact ? orr[t * ostride] : __bfloat162float(orow[t * ostride]);
                orow[t * ostride] = __float2bfloat16_rn(fmaf(G, y[i], base));
            }
        }
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
        reinterpret_cast<int32_t*>(ws + L.vlen), reinterpret_cast<int32_t*>(ws + L.clist),
        a.status);
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
        reinterpret_cast<float*>(ws + L.sst), reinterpret_cast<float*>(ws + L.rnorm), a.S_T,
        a.status);
    return cudaGetLastError();
}

cudaError_t launch_split_correct(const PrefillArgs& a, const SplitLayout& L, char* ws,
                                 cudaStream_t stream) {
    const int64_t slots = a.total_tokens / 64 + a.num_seqs + 1;
    const int sms = sm_count();
    if (sms <= 0) return cudaErrorInvalidValue;
    int32_t* ccount = reinterpret_cast<int32_t*>(ws + L.clist);
    int4* clist = reinterpret_cast<int4*>(ws + L.clist + 16);
    const int64_t warps = slots * a.H * (a.d_v / kB);
    const int64_t want = (warps + 7) / 8;
    const int sel_blocks = (int)(want < 16 * sms ? want : 16 * sms);
    split_select_kernel<<<sel_blocks, 256, 0, stream>>>(
        a.cu_seqlens, a.num_seqs, L.M, a.H, a.d_v, slots,
        reinterpret_cast<const int64_t*>(ws + L.vt0), reinterpret_cast<const int32_t*>(ws + L.vlen),
        reinterpret_cast<const float*>(ws + L.gstart), reinterpret_cast<const float*>(ws + L.rnorm),
        ccount, clist, a.status);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    const int smem = (64 * kQld + 64 + 4 * kB + kB * (kB + 1)) * (int)sizeof(float);
    err = cudaFuncSetAttribute(split_correct_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               smem);
    if (err != cudaSuccess) return err;
    split_correct_kernel<<<2 * sms, kCorrThreads, smem, stream>>>(
        a.num_seqs, a.H, a.d_v, static_cast<const float*>(a.alpha),
        reinterpret_cast<const float*>(ws + L.qtil), reinterpret_cast<const float*>(ws + L.gstart),
        reinterpret_cast<const float*>(ws + L.sst), reinterpret_cast<const float*>(ws + L.rnorm),
        reinterpret_cast<const float*>(ws + L.qfro), a.cu_seqlens, ccount, clist,
        reinterpret_cast<const float*>(ws + L.ores),
        static_cast<__nv_bfloat16*>(a.o), a.status);
    return cudaGetLastError();
}

}  // namespace kda
