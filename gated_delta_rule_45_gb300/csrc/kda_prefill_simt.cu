// Portable chunkwise KDA prefill on CUDA cores, all arithmetic in fp32.
//
// Chunk form of the recurrence ("Kimi (AI)", section "Kimi Delta Attention
// (KDA)"; chunking: "grouping multiple steps" in the Kimi K3 architecture
// walkthrough).  With D_t = diag(alpha_t) the update is
// S_t = D_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T; D_t acts on rows
// and the projector on columns, so each row of S is a scalar-gated delta rule.
// For a chunk of C tokens, gamma_t = prod_{j<=t} alpha_j (per value channel):
//
//   A = I + diag(beta) strict_lower(K K^T),  T = A^{-1}     (C x C, shared by all rows)
//   X = diag(beta) (V / Gamma - K S^T)                       (C x d_v)
//   U = T X
//   O = Gamma * (Q S^T + tril_incl(Q K^T) U)
//   S <- diag(gamma_C) (S + U^T K)
//
// Rows past the end of a sequence are padded with k = q = v = 0, alpha = 1,
// beta = 0; they leave S unchanged and their o is not stored.
//
// The additive update of linear attention (no prediction: S_t = D_t S_{t-1} +
// beta_t v_t k_t^T) is the same chunk form with the K S^T term dropped from X
// and T = I.
//
// One CTA per (sequence, head, block of 64 value channels); CTAs are issued
// in the planner's longest-first order.  This kernel covers every supported
// shape (d_k <= 128, chunk 16/32/64, bf16 or fp32 storage) and is the path for
// shapes the tensor-core kernel does not take.
#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kThreads = 256;
constexpr int kDVB = 64;           // value channels per CTA
constexpr int kDVP = kDVB + 1;     // padded row stride of [C][d_v-block] tiles
constexpr int kMaxDK = 128;

struct SimtSmem {
    int KP, CP;
    float *Ks, *Qs, *Ss, *Xs, *Us, *Gs, *Ls, *Ts, *Ps, *bs;
};

__host__ __device__ inline size_t simt_smem_floats(int C, int d_k) {
    const int KP = d_k + 1, CP = C + 1;
    return (size_t)2 * C * KP + (size_t)kDVB * KP + (size_t)3 * C * kDVP + (size_t)3 * C * CP + C;
}

__device__ inline SimtSmem carve(float* base, int C, int d_k) {
    SimtSmem s;
    s.KP = d_k + 1;
    s.CP = C + 1;
    float* p = base;
    s.Ks = p; p += C * s.KP;
    s.Qs = p; p += C * s.KP;
    s.Ss = p; p += kDVB * s.KP;
    s.Xs = p; p += C * kDVP;
    s.Us = p; p += C * kDVP;
    s.Gs = p; p += C * kDVP;
    s.Ls = p; p += C * s.CP;
    s.Ts = p; p += C * s.CP;
    s.Ps = p; p += C * s.CP;
    s.bs = p;
    return s;
}

// acc[i][j] += sum_k A(m_i, k) B(n_j, k) for m_i = ty + 16 i < M, n_j = n0 + tx + 16 j < N,
// with A(m, k) = A[m * sam + k * sak] and B(n, k) = B[n * sbn + k * sbk].
__device__ __forceinline__ void mm_acc(float (&acc)[4][4], const float* A, int sam, int sak,
                                       const float* B, int sbn, int sbk, int M, int N, int K,
                                       int n0, int ty, int tx) {
    for (int k = 0; k < K; ++k) {
        float a[4], b[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int m = ty + 16 * i;
            a[i] = m < M ? A[m * sam + k * sak] : 0.f;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = n0 + tx + 16 * j;
            b[j] = n < N ? B[n * sbn + k * sbk] : 0.f;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
}

__device__ __forceinline__ void zero(float (&acc)[4][4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
}

// One (sequence n, head h, block vb of 64 value channels) from S0 to S_T.
// rowmask: null (every channel written) or two words marking the channels of
// the block whose o and S_T are written.
template <typename T, int C>
__device__ void simt_item(const PrefillArgs& a, float* smem, int n, int h, int vb,
                          const uint32_t* rowmask = nullptr) {
    const uint32_t wm0 = rowmask ? rowmask[0] : 0xffffffffu;
    const uint32_t wm1 = rowmask ? rowmask[1] : 0xffffffffu;
    auto marked = [&](int r) { return ((r < 32 ? wm0 >> r : wm1 >> (r - 32)) & 1u) != 0u; };
    const int d_k = a.d_k, d_v = a.d_v, H = a.H;
    SimtSmem s = carve(smem, C, d_k);
    const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
    const int64_t t_begin = a.cu_seqlens[n], t_end = a.cu_seqlens[n + 1];
    const int r0 = vb * kDVB;
    const int rows = min(kDVB, d_v - r0);

    const T* q = static_cast<const T*>(a.q);
    const T* k = static_cast<const T*>(a.k);
    const T* v = static_cast<const T*>(a.v);
    T* o = static_cast<T*>(a.o);
    const size_t state_off = ((size_t)n * H + h) * (size_t)d_v * d_k + (size_t)r0 * d_k;

    for (int idx = tid; idx < kDVB * d_k; idx += kThreads) {
        const int r = idx / d_k, c = idx % d_k;
        float x = 0.f;
        if (r < rows && a.S0) x = a.S0[state_off + (size_t)r * d_k + c];
        s.Ss[r * s.KP + c] = x;
    }
    __syncthreads();

    // A chunk whose product of alpha falls below kDecayFloor on some channel of
    // this block is taken again as a chunk of 16 tokens (1 / gamma must stay
    // finite); the loop then advances by the tokens actually processed.
    int step = C;
    for (int64_t c0 = t_begin; c0 < t_end; c0 += step) {
      int nvalid = (int)min((int64_t)C, t_end - c0);
      for (;;) {
        // load the chunk; padded tokens: k = q = v = 0, alpha = 1, beta = 0
        for (int idx = tid; idx < C * d_k; idx += kThreads) {
            const int t = idx / d_k, c = idx % d_k;
            float kx = 0.f, qx = 0.f;
            if (t < nvalid) {
                const size_t gi = ((size_t)(c0 + t) * H + h) * d_k + c;
                kx = Elem<T>::load(k + gi);
                qx = Elem<T>::load(q + gi);
            }
            s.Ks[t * s.KP + c] = kx;
            s.Qs[t * s.KP + c] = qx;
        }
        for (int idx = tid; idx < C * kDVB; idx += kThreads) {
            const int t = idx / kDVB, r = idx % kDVB;
            float vx = 0.f, ax = 1.f;
            if (t < nvalid && r < rows) {
                const size_t gi = ((size_t)(c0 + t) * H + h) * d_v + r0 + r;
                vx = Elem<T>::load(v + gi);
                if (a.gate == KDA_GATE_HEAD_F32)   // one gate per (token, head)
                    ax = static_cast<const float*>(a.alpha)[(size_t)(c0 + t) * H + h];
                else if (a.gate == KDA_GATE_CHANNEL_LOG_BF16)
                    ax = __expf(__bfloat162float(static_cast<const __nv_bfloat16*>(a.alpha)[gi]));
                else
                    ax = static_cast<const float*>(a.alpha)[gi];
            }
            s.Xs[t * kDVP + r] = vx;
            s.Gs[t * kDVP + r] = ax;
        }
        if (tid < C) s.bs[tid] = tid < nvalid ? a.beta[(size_t)(c0 + tid) * H + h] : 0.f;
        __syncthreads();

        // Gamma: running product of alpha over the chunk, per value channel
        bool fast = false;
        if (tid < kDVB) {
            float g = 1.f;
            for (int t = 0; t < C; ++t) {
                g *= s.Gs[t * kDVP + tid];
                s.Gs[t * kDVP + tid] = g;
            }
            fast = !(g >= kDecayFloor);
        }
        if (__syncthreads_or(fast)) {
            if (nvalid > 16) {   // once more, over the first 16 tokens only
                nvalid = 16;
                continue;
            }
            // even 16 tokens decay too fast for the chunk form: reported
            if (tid == 0) atomicCAS(a.status, 0, (int32_t)KDA_ERR_DEVICE_RANGE);
        }
        step = nvalid;
        break;
      }
        // L = diag(beta) strict_lower(K K^T);  P = tril_incl(Q K^T)
        {
            float acc[4][4], accp[4][4];
            zero(acc);
            zero(accp);
            mm_acc(acc, s.Ks, s.KP, 1, s.Ks, s.KP, 1, C, C, d_k, 0, ty, tx);
            mm_acc(accp, s.Qs, s.KP, 1, s.Ks, s.KP, 1, C, C, d_k, 0, ty, tx);
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int m = ty + 16 * i, nn = tx + 16 * j;
                    if (m < C && nn < C) {
                        s.Ls[m * s.CP + nn] = nn < m ? s.bs[m] * acc[i][j] : 0.f;
                        s.Ps[m * s.CP + nn] = nn <= m ? accp[i][j] : 0.f;
                    }
                }
        }
        __syncthreads();

        // T = (I + L)^{-1}, unit lower triangular; one thread per column,
        // forward substitution T[i][c] = delta_ic - sum_{j<i} L[i][j] T[j][c]
        // (the additive update has no prediction: T = I)
        if (tid < C) {
            const int c = tid;
            for (int i = 0; i < C; ++i) {
                float x = (i == c) ? 1.f : 0.f;
                if (i > c && !a.additive) {
                    for (int j = c; j < i; ++j) x = fmaf(-s.Ls[i * s.CP + j], s.Ts[j * s.CP + c], x);
                }
                s.Ts[i * s.CP + c] = x;
            }
        }
        // X = diag(beta) (V / Gamma - K S^T), written over V (no K S^T term in the
        // additive update)
        {
            float acc[4][4];
            zero(acc);
            if (!a.additive) mm_acc(acc, s.Ks, s.KP, 1, s.Ss, s.KP, 1, C, kDVB, d_k, 0, ty, tx);
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int t = ty + 16 * i, r = tx + 16 * j;
                    if (t < C) {
                        const float vg = s.Xs[t * kDVP + r] / s.Gs[t * kDVP + r];
                        s.Xs[t * kDVP + r] = s.bs[t] * (vg - acc[i][j]);
                    }
                }
        }
        __syncthreads();

        // U = T X
        {
            float acc[4][4];
            zero(acc);
            mm_acc(acc, s.Ts, s.CP, 1, s.Xs, 1, kDVP, C, kDVB, C, 0, ty, tx);
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int t = ty + 16 * i, r = tx + 16 * j;
                    if (t < C) s.Us[t * kDVP + r] = acc[i][j];
                }
        }
        __syncthreads();

        // O = Gamma * (Q S^T + P U)
        {
            float acc[4][4];
            zero(acc);
            mm_acc(acc, s.Qs, s.KP, 1, s.Ss, s.KP, 1, C, kDVB, d_k, 0, ty, tx);
            mm_acc(acc, s.Ps, s.CP, 1, s.Us, 1, kDVP, C, kDVB, C, 0, ty, tx);
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int t = ty + 16 * i, r = tx + 16 * j;
                    if (t < nvalid && r < rows && marked(r)) {
                        const float y = s.Gs[t * kDVP + r] * acc[i][j];
                        Elem<T>::store(o + ((size_t)(c0 + t) * H + h) * d_v + r0 + r, y);
                    }
                }
        }
        __syncthreads();

        // S <- diag(gamma_C) (S + U^T K)
        for (int n0 = 0; n0 < d_k; n0 += 64) {
            float acc[4][4];
            zero(acc);
            mm_acc(acc, s.Us, 1, kDVP, s.Ks, 1, s.KP, kDVB, d_k, C, n0, ty, tx);
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int r = ty + 16 * i, c = n0 + tx + 16 * j;
                    if (c < d_k) {
                        const float gC = s.Gs[(C - 1) * kDVP + r];
                        s.Ss[r * s.KP + c] = gC * (s.Ss[r * s.KP + c] + acc[i][j]);
                    }
                }
        }
        __syncthreads();
    }

    for (int idx = tid; idx < rows * d_k; idx += kThreads) {
        const int r = idx / d_k, c = idx % d_k;
        if (marked(r)) a.S_T[state_off + (size_t)r * d_k + c] = s.Ss[r * s.KP + c];
    }
}

template <typename T, int C>
__global__ void __launch_bounds__(kThreads)
kda_prefill_simt_kernel(PrefillArgs a) {
    if (*a.status == KDA_ERR_DEVICE_INPUT) return;   // planner rejected cu_seqlens
    extern __shared__ float smem[];
    const int nvb = (a.d_v + kDVB - 1) / kDVB;
    const int item = blockIdx.x;
    const int rank = item / (a.H * nvb);
    simt_item<T, C>(a, smem, a.order[rank], (item / nvb) % a.H, item % nvb);
}

// The channels the tensor-core kernel handed back (their decay too fast for
// its one-pass chunks): a persistent grid walks every (sequence, head,
// 64-channel block) and runs those with a marked channel again from S0,
// writing o and S_T of the marked channels only (the others are right, and
// their S0 may already be overwritten by S_T).
template <typename T, int C>
__global__ void __launch_bounds__(kThreads)
kda_prefill_simt_redo_kernel(PrefillArgs a) {
    if (*a.status == KDA_ERR_DEVICE_INPUT) return;
    extern __shared__ float smem[];
    const int nb64 = a.d_v / 64;
    const int total = a.num_seqs * a.H * nb64;
    for (int i = blockIdx.x; i < total; i += gridDim.x) {
        const uint32_t* m = a.redo + 2 * (size_t)i;   // 64 channels: two mask words
        if ((m[0] | m[1]) == 0u) continue;             // uniform across the CTA
        const int n = i / (a.H * nb64), h = (i / nb64) % a.H, vb = i % nb64;
        simt_item<T, C>(a, smem, n, h, vb, m);
        __syncthreads();   // the next item reuses the shared memory
    }
}

template <typename T, int C>
cudaError_t launch_simt_t(const PrefillArgs& a, cudaStream_t stream) {
    const size_t smem = simt_smem_floats(C, kMaxDK) * sizeof(float);
    cudaError_t err = cudaFuncSetAttribute(kda_prefill_simt_kernel<T, C>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    const int nvb = (a.d_v + kDVB - 1) / kDVB;
    const int64_t blocks = (int64_t)a.num_seqs * a.H * nvb;
    if (blocks == 0) return cudaSuccess;
    kda_prefill_simt_kernel<T, C><<<(unsigned)blocks, kThreads,
                                    simt_smem_floats(C, a.d_k) * sizeof(float), stream>>>(a);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_simt_c(const PrefillArgs& a, cudaStream_t stream) {
    switch (a.chunk) {
        case 16: return launch_simt_t<T, 16>(a, stream);
        case 32: return launch_simt_t<T, 32>(a, stream);
        case 64: return launch_simt_t<T, 64>(a, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_prefill_simt_redo(const PrefillArgs& a, cudaStream_t stream) {
    if (!a.redo || a.dtype != KDA_BF16 || a.chunk != 64 || a.d_k > kMaxDK || a.d_v % 128 != 0)
        return cudaErrorInvalidValue;
    if (a.num_seqs == 0) return cudaSuccess;
    const size_t smem = simt_smem_floats(64, kMaxDK) * sizeof(float);
    cudaError_t err = cudaFuncSetAttribute(kda_prefill_simt_redo_kernel<__nv_bfloat16, 64>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    kda_prefill_simt_redo_kernel<__nv_bfloat16, 64><<<sm_count(), kThreads,
                                                      simt_smem_floats(64, a.d_k) * sizeof(float),
                                                      stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_prefill_simt(const PrefillArgs& a, cudaStream_t stream) {
    if (a.d_k > kMaxDK) return cudaErrorInvalidValue;
    if (a.dtype == KDA_BF16) return launch_simt_c<__nv_bfloat16>(a, stream);
    return launch_simt_c<float>(a, stream);
}

}  // namespace kda
