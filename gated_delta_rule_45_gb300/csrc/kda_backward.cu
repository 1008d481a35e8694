// Backward pass of the KDA prefill: gradients of a loss with respect to q, k,
// v, alpha, beta and S0, given its gradients with respect to o and S_T.
//
// The recurrence ("Kimi (AI)", section "Kimi Delta Attention (KDA)"),
// S_t = diag(alpha_t) S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T and
// o_t = S_t q_t, is differentiated in its chunkwise form (chunks of C = 64
// tokens, per value channel gamma = cumulative product of alpha):
//
//   forward   T = (I + diag(beta) strict_lower(K K^T))^-1,  M = tril_incl(Q K^T)
//             Y = V / Gamma - K S^T,  U = T diag(beta) Y,  P = Q S^T + M U
//             O = Gamma * P,  S_next = diag(gamma_C) (S + U^T K)
//   backward  with D = dL/dS_next:
//             dS^ = diag(gamma_C) D,  dP = Gamma * dO
//             dU = M^T dP + K dS^^T,  dX = T^T dU,  dY = diag(beta) dX
//             dT = dU (diag(beta) Y)^T,  sdA = strict_lower(-T^T dT T^T)
//             dM = tril_incl(dP U^T)
//             dq = dP S + dM K
//             dk = dM^T Q + U dS^ - dY S + diag(beta) sdA K + sdA^T diag(beta) K
//             dv = dY / Gamma
//             dbeta_r = sum_i dX_ri Y_ri + k_r . (sdA K)_r
//             E = dP * P - dY * V / Gamma,  E[C-1] += rowsum(dS^ * (S + U^T K))
//             dalpha = reverse_cumsum_over_tokens(E) / alpha
//             D <- dS^ + dP^T Q - dY^T K
//
// Value channels (rows of S) only interact through sums that end in dq, dk
// and dbeta, so one CTA owns one (sequence, head, 64-row block) chain: a
// forward sweep over its chunks writes the chunk-start states to the
// workspace, a backward sweep walks the chunks in reverse carrying D in shared
// memory.  dq, dk and dbeta are written per row block and summed by a second
// kernel in a fixed order, so results are deterministic.  Arithmetic is fp32
// on the CUDA cores: every product above is a shared-memory tile product of
// at most 64 x 128 x 128.
#include "kda_internal.h"

namespace kda {
namespace {

constexpr int C = 64;      // tokens per chunk
constexpr int DK = 128;    // key channels
constexpr int R = 64;      // value rows per CTA
constexpr int NTH = 256;   // threads: a 16 x 16 grid of 4 x 4 (or 4 x 8) output tiles
constexpr int LDH = 130;   // bf16 row stride of K and Q (65 words: conflict-free columns)
constexpr int LDS = 129;   // fp32 row stride of S and D
constexpr int LDC = 65;    // fp32 row stride of the 64 x 64 tiles

// shared memory (bytes)
constexpr int OFF_K = 0;
constexpr int OFF_Q = OFF_K + C * LDH * 2;
constexpr int OFF_S = OFF_Q + C * LDH * 2;
constexpr int OFF_D = OFF_S + R * LDS * 4;
constexpr int OFF_T64 = OFF_D + R * LDS * 4;
constexpr int T64_BYTES = 64 * LDC * 4;
enum { T_G = 0, T_T, T_M, T_Y, T_U, T_P, T_W, N_T64 };
constexpr int OFF_RED = OFF_T64 + N_T64 * T64_BYTES;        // fp32 [16][64]
constexpr int OFF_MISC = OFF_RED + 16 * 64 * 4;             // beta, dbeta, e, gamma_C
constexpr int SMEM_BYTES = OFF_MISC + 4 * 64 * 4;

struct BwdParams {
    const __nv_bfloat16 *q, *k, *v, *dO;
    const float *alpha, *beta, *S0, *dS_T;
    const int32_t *cu, *order, *status;
    int32_t N, H, d_v, nrb;
    int64_t T;
    float* ckpt;              // [slots][H][d_v][DK], slot = t0 / C + n + chunk
    float *dq_part, *dk_part; // [nrb][T][H][DK]
    float* db_part;           // [nrb][T][H]
    float *dv, *dalpha;       // [T][H][d_v]
    float* dS0;               // [N][H][d_v][DK] or null
};

// acc[m][n] += sum_k A(ty + 16 m, k) B(k, tx + 16 n)
template <int MT, int NT, int KD, class FA, class FB>
__device__ __forceinline__ void mm(float (&acc)[MT][NT], FA A, FB B) {
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
#pragma unroll 4
    for (int k = 0; k < KD; ++k) {
        float a[MT], b[NT];
#pragma unroll
        for (int m = 0; m < MT; ++m) a[m] = A(ty + 16 * m, k);
#pragma unroll
        for (int n = 0; n < NT; ++n) b[n] = B(k, tx + 16 * n);
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int n = 0; n < NT; ++n) acc[m][n] = fmaf(a[m], b[n], acc[m][n]);
    }
}

template <int MT, int NT>
__device__ __forceinline__ void zero(float (&acc)[MT][NT]) {
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int n = 0; n < NT; ++n) acc[m][n] = 0.f;
}

__device__ __forceinline__ float bf(const __nv_bfloat16* p) { return __bfloat162float(*p); }

// Rows tok0 .. tok0 + 63 of a [T][H][DK] bf16 tensor into a [64][LDH] tile
// (rows at or past nvalid are zero).
__device__ void load_rows_bf16(__nv_bfloat16* dst, const __nv_bfloat16* src, int64_t tok0,
                               int nvalid, int H, int h) {
    const int r = threadIdx.x >> 2, part = threadIdx.x & 3;
    uint32_t* d = reinterpret_cast<uint32_t*>(dst + r * LDH + 32 * part);
    if (r < nvalid) {
        const uint4* s = reinterpret_cast<const uint4*>(src + ((tok0 + r) * H + h) * DK + 32 * part);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint4 x = s[j];
            d[4 * j] = x.x; d[4 * j + 1] = x.y; d[4 * j + 2] = x.z; d[4 * j + 3] = x.w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) d[j] = 0u;
    }
}

// A 64 x 128 fp32 block, rows contiguous in global memory, into a [64][LDS] tile.
__device__ void load_state(float* dst, const float* src) {
    for (int e = 4 * threadIdx.x; e < R * DK; e += 4 * NTH) {
        float4 x = src ? *reinterpret_cast<const float4*>(src + e) : make_float4(0.f, 0.f, 0.f, 0.f);
        float* d = dst + (e / DK) * LDS + e % DK;
        d[0] = x.x; d[1] = x.y; d[2] = x.z; d[3] = x.w;
    }
}

__device__ void store_state(float* dst, const float* src) {
    for (int e = 4 * threadIdx.x; e < R * DK; e += 4 * NTH) {
        const float* s = src + (e / DK) * LDS + e % DK;
        *reinterpret_cast<float4*>(dst + e) = make_float4(s[0], s[1], s[2], s[3]);
    }
}

// Per-chunk inputs shared by both sweeps: K (and Q), beta, Gamma and gamma_C,
// then T = (I + diag(beta) strict_lower(K K^T))^-1 by forward substitution.
__device__ void chunk_setup(const BwdParams& p, char* sm, int64_t tok0, int nvalid, int h,
                            int row0, bool with_q) {
    __nv_bfloat16* Ks = reinterpret_cast<__nv_bfloat16*>(sm + OFF_K);
    __nv_bfloat16* Qs = reinterpret_cast<__nv_bfloat16*>(sm + OFF_Q);
    float* tG = reinterpret_cast<float*>(sm + OFF_T64 + T_G * T64_BYTES);
    float* tT = reinterpret_cast<float*>(sm + OFF_T64 + T_T * T64_BYTES);
    float* tW = reinterpret_cast<float*>(sm + OFF_T64 + T_W * T64_BYTES);
    float* bet = reinterpret_cast<float*>(sm + OFF_MISC);
    float* gC = bet + 192;
    const int tid = threadIdx.x;
    load_rows_bf16(Ks, p.k, tok0, nvalid, p.H, h);
    if (with_q) load_rows_bf16(Qs, p.q, tok0, nvalid, p.H, h);
    if (tid < C) bet[tid] = tid < nvalid ? p.beta[(tok0 + tid) * p.H + h] : 0.f;
    if (tid >= 64 && tid < 128) {   // Gamma, one value channel per thread
        const int i = tid - 64;
        const float* al = p.alpha + (tok0 * p.H + h) * (int64_t)p.d_v + row0 + i;
        const int64_t stride = (int64_t)p.H * p.d_v;
        float run = 1.f;
        for (int r = 0; r < C; ++r) {
            if (r < nvalid) run *= al[r * stride];
            tG[r * LDC + i] = run;
        }
        gC[i] = run;
    }
    // T starts as the identity
    for (int e = tid; e < C * C; e += NTH) tT[(e >> 6) * LDC + (e & 63)] = (e >> 6) == (e & 63) ? 1.f : 0.f;
    __syncthreads();
    {   // L' = diag(beta) strict_lower(K K^T)
        float acc[4][4];
        zero(acc);
        mm<4, 4, DK>(acc, [&](int r, int c) { return bf(Ks + r * LDH + c); },
                     [&](int c, int s) { return bf(Ks + s * LDH + c); });
        const int tx = tid & 15, ty = tid >> 4;
#pragma unroll
        for (int m = 0; m < 4; ++m)
#pragma unroll
            for (int n = 0; n < 4; ++n) {
                const int r = ty + 16 * m, s = tx + 16 * n;
                tW[r * LDC + s] = s < r ? bet[r] * acc[m][n] : 0.f;
            }
    }
    __syncthreads();
    {   // row r of T: T[r][j] = -sum_{s<r} L'[r][s] T[s][j] for j < r; four lanes per column
        const int j = tid >> 2, part = tid & 3;
        for (int r = 1; r < C; ++r) {
            float acc = 0.f;
            for (int s = part; s < r; s += 4) acc = fmaf(tW[r * LDC + s], tT[s * LDC + j], acc);
            acc += __shfl_xor_sync(0xffffffffu, acc, 1);
            acc += __shfl_xor_sync(0xffffffffu, acc, 2);
            if (part == 0 && j < r) tT[r * LDC + j] = -acc;
            __syncwarp();
        }
    }
    __syncthreads();
}

__global__ void __launch_bounds__(NTH, 1) kda_backward_kernel(const BwdParams p) {
    if (*p.status != 0) return;
    extern __shared__ __align__(16) char sm[];
    const __nv_bfloat16* Ks = reinterpret_cast<const __nv_bfloat16*>(sm + OFF_K);
    const __nv_bfloat16* Qs = reinterpret_cast<const __nv_bfloat16*>(sm + OFF_Q);
    float* Ss = reinterpret_cast<float*>(sm + OFF_S);
    float* Ds = reinterpret_cast<float*>(sm + OFF_D);
    float* tG = reinterpret_cast<float*>(sm + OFF_T64 + T_G * T64_BYTES);
    float* tT = reinterpret_cast<float*>(sm + OFF_T64 + T_T * T64_BYTES);
    float* tM = reinterpret_cast<float*>(sm + OFF_T64 + T_M * T64_BYTES);
    float* tY = reinterpret_cast<float*>(sm + OFF_T64 + T_Y * T64_BYTES);
    float* tU = reinterpret_cast<float*>(sm + OFF_T64 + T_U * T64_BYTES);
    float* tP = reinterpret_cast<float*>(sm + OFF_T64 + T_P * T64_BYTES);
    float* tW = reinterpret_cast<float*>(sm + OFF_T64 + T_W * T64_BYTES);
    float* red = reinterpret_cast<float*>(sm + OFF_RED);
    float* bet = reinterpret_cast<float*>(sm + OFF_MISC);
    float* dbr = bet + 64;
    float* ecol = bet + 128;
    float* gC = bet + 192;

    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int rb = blockIdx.x % p.nrb;
    const int h = (blockIdx.x / p.nrb) % p.H;
    const int n = p.order[blockIdx.x / (p.nrb * p.H)];
    const int64_t t0 = p.cu[n];
    const int len = p.cu[n + 1] - p.cu[n];
    const int nc = (len + C - 1) / C;
    const int row0 = rb * R;
    const int64_t slot0 = t0 / C + n;
    const size_t st_rows = (size_t)p.d_v * DK;   // one head's state
    auto ckpt_at = [&](int c) {
        return p.ckpt + ((size_t)(slot0 + c) * p.H + h) * st_rows + (size_t)row0 * DK;
    };
    const int64_t vstride = (int64_t)p.H * p.d_v;
    auto vidx = [&](int64_t tok, int i) { return tok * vstride + (int64_t)h * p.d_v + row0 + i; };

    // ---- forward sweep: chunk-start states into the workspace ----
    load_state(Ss, p.S0 ? p.S0 + ((size_t)n * p.H + h) * st_rows + (size_t)row0 * DK : nullptr);
    __syncthreads();
    for (int c = 0; c < nc; ++c) {
        const int64_t tok0 = t0 + (int64_t)c * C;
        const int nvalid = min(C, len - c * C);
        store_state(ckpt_at(c), Ss);
        chunk_setup(p, sm, tok0, nvalid, h, row0, false);
        {   // Y = V / Gamma - K S^T
            float acc[4][4];
            zero(acc);
            mm<4, 4, DK>(acc, [&](int r, int c2) { return bf(Ks + r * LDH + c2); },
                         [&](int c2, int i) { return Ss[i * LDS + c2]; });
#pragma unroll
            for (int m = 0; m < 4; ++m)
#pragma unroll
                for (int n2 = 0; n2 < 4; ++n2) {
                    const int r = ty + 16 * m, i = tx + 16 * n2;
                    const float v = r < nvalid ? bf(p.v + vidx(tok0 + r, i)) : 0.f;
                    tY[r * LDC + i] = v / tG[r * LDC + i] - acc[m][n2];
                }
        }
        __syncthreads();
        {   // U = T diag(beta) Y
            float acc[4][4];
            zero(acc);
            mm<4, 4, C>(acc, [&](int r, int s) { return tT[r * LDC + s]; },
                        [&](int s, int i) { return bet[s] * tY[s * LDC + i]; });
#pragma unroll
            for (int m = 0; m < 4; ++m)
#pragma unroll
                for (int n2 = 0; n2 < 4; ++n2) tU[(ty + 16 * m) * LDC + tx + 16 * n2] = acc[m][n2];
        }
        __syncthreads();
        {   // S <- diag(gamma_C) (S + U^T K)
            float acc[4][8];
            zero(acc);
            mm<4, 8, C>(acc, [&](int i, int s) { return tU[s * LDC + i]; },
                        [&](int s, int c2) { return bf(Ks + s * LDH + c2); });
#pragma unroll
            for (int m = 0; m < 4; ++m)
#pragma unroll
                for (int n2 = 0; n2 < 8; ++n2) {
                    const int i = ty + 16 * m, c2 = tx + 16 * n2;
                    Ss[i * LDS + c2] = gC[i] * (Ss[i * LDS + c2] + acc[m][n2]);
                }
        }
        __syncthreads();
    }

    // ---- backward sweep ----
    load_state(Ds, p.dS_T ? p.dS_T + ((size_t)n * p.H + h) * st_rows + (size_t)row0 * DK : nullptr);
    __syncthreads();
    for (int c = nc - 1; c >= 0; --c) {
        const int64_t tok0 = t0 + (int64_t)c * C;
        const int nvalid = min(C, len - c * C);
        load_state(Ss, ckpt_at(c));
        chunk_setup(p, sm, tok0, nvalid, h, row0, true);
        {   // M = tril_incl(Q K^T)
            float acc[4][4];
            zero(acc);
            mm<4, 4, DK>(acc, [&](int r, int c2) { return bf(Qs + r * LDH + c2); },
                         [&](int c2, int s) { return bf(Ks + s * LDH + c2); });
#pragma unroll
            for (int m = 0; m < 4; ++m)
#pragma unroll
                for (int n2 = 0; n2 < 4; ++n2) {
                    const int r = ty + 16 * m, s = tx + 16 * n2;
                    tM[r * LDC + s] = s <= r ? acc[m][n2] : 0.f;
                }
        }
        {   // Y = V / Gamma - K S^T and dP = Gamma * dO
            float acc[4][4];
            zero(acc);
            mm<4, 4, DK>(acc, [&](int r, int c2) { return bf(Ks + r * LDH + c2); },
                         [&](int c2, int i) { return Ss[i * LDS + c2]; });
#pragma unroll
            for (int m = 0; m < 4; ++m)
#pragma unroll
                for (int n2 = 0; n2 < 4; ++n2) {
                    const int r = ty + 16 * m, i = tx + 16 * n2;
                    const bool ok = r < nvalid;
                    const float v = ok ? bf(p.v + vidx(tok0 + r, i)) : 0.f;
                    const float d = ok ? bf(p.dO + vidx(tok0 + r, i)) : 0.f;
                    const float g = tG[r * LDC + i];
                    tY[r * LDC + i] = v / g - acc[m][n2];
                    tP[r * LDC + i] = g * d;
                }
        }
        __syncthreads();
        {   // U = T diag(beta) Y; dS^ = diag(gamma_C) D
            float acc[4][4];
            zero(acc);
            mm<4, 4, C>(acc, [&](int r, int s) { return tT[r * LDC + s]; },
                        [&](int s, int i) { return bet[s] * tY[s * LDC + i]; });
#pragma unroll
            for (int m = 0; m < 4; ++m)
#pragma unroll
                for (int n2 = 0; n2 < 4; ++n2) tU[(ty + 16 * m) * LDC + tx + 16 * n2] = acc[m][n2];
            for (int e = tid; e < R * DK; e += NTH) {
                const int i = e >> 7;
                Ds[i * LDS + (e & 127)] *= gC[i];
            }
        }
        __syncthreads();
        // E = dP * P with P = Q S^T + M U, kept in registers (same tiles as dX below)
        float E[4][4];
        zero(E);
        mm<4, 4, DK>(E, [&](int r, int c2) { return bf(Qs + r * LDH + c2); },
                     [&](int c2, int i) { return Ss[i * LDS + c2]; });
        mm<4, 4, C>(E, [&](int r, int s) { return tM[r * LDC + s]; },
                    [&](int s, int i) { return tU[s * LDC + i]; });
#pragma unroll
        for (int m = 0; m < 4; ++m)
#pragma unroll
            for (int n2 = 0; n2 < 4; ++n2) E[m][n2] *= tP[(ty + 16 * m) * LDC + tx + 16 * n2];
        {   // dU = K dS^^T + M^T dP; the first term also gives sum_r U_ri (K dS^^T)_ri
            float acc[4][4];
            zero(acc);
            mm<4, 4, DK>(acc, [&](int r, int c2) { return bf(Ks + r * LDH + c2); },
                         [&](int c2, int i) { return Ds[i * LDS + c2]; });
#pragma unroll
            for (int n2 = 0; n2 < 4; ++n2) {
                float s = 0.f;
#pragma unroll
                for (int m = 0; m < 4; ++m) s = fmaf(tU[(ty + 16 * m) * LDC + tx + 16 * n2], acc[m][n2], s);
                red[ty * 64 + tx + 16 * n2] = s;
            }
            mm<4, 4, C>(acc, [&](int r, int s) { return tM[s * LDC + r]; },
                        [&](int s, int i) { return tP[s * LDC + i]; });
#pragma unroll
            for (int m = 0; m < 4; ++m)
#pragma unroll
                for (int n2 = 0; n2 < 4; ++n2) tW[(ty + 16 * m) * LDC + tx + 16 * n2] = acc[m][n2];
        }
        __syncthreads();
        {   // dT = dU (diag(beta) Y)^T into M's tile; finish the column sums
            float acc[4][4];
            zero(acc);
            mm<4, 4, R>(acc, [&](int r, int i) { return tW[r * LDC + i]; },
                        [&](int i, int s) { return bet[s] * tY[s * LDC + i]; });
#pragma unroll
            for (int m = 0; m < 4; ++m)
#pragma unroll
                for (int n2 = 0; n2 < 4; ++n2) tM[(ty + 16 * m) * LDC + tx + 16 * n2] = acc[m][n2];
            if (tid < 64) {
                float s = 0.f;
                for (int j = 0; j < 16; ++j) s += red[j * 64 + tid];
                ecol[tid] = s;
            }
        }
        __syncthreads();
        {   // dX = T^T dU: dbeta (first part), dY (over Y), dv, E -= dY V / Gamma
            float acc[4][4];
            zero(acc);
            mm<4, 4, C>(acc, [&](int r, int s) { return tT[s * LDC + r]; },
                        [&](int s, int i) { return tW[s * LDC + i]; });
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int r = ty + 16 * m;
                const bool ok = r < nvalid;
                float part = 0.f;
#pragma unroll
                for (int n2 = 0; n2 < 4; ++n2) {
                    const int i = tx + 16 * n2;
                    const float dx = acc[m][n2];
                    part = fmaf(dx, tY[r * LDC + i], part);
                    const float dy = bet[r] * dx;
                    tY[r * LDC + i] = dy;
                    const float g = tG[r * LDC + i];
                    const float v = ok ? bf(p.v + vidx(tok0 + r, i)) : 0.f;
                    E[m][n2] -= dy * v / g;
                    if (ok) p.dv[vidx(tok0 + r, i)] = dy / g;
                }
                red[tx * 64 + r] = part;
            }
        }
        __syncthreads();
        {   // tmp = dT T^T over dU's tile; finish the dbeta row sums
            float acc[4][4];
            zero(acc);
            mm<4, 4, C>(acc, [&](int r, int s) { return tM[r * LDC + s]; },
                        [&](int s, int j) { return tT[j * LDC + s]; });
#pragma unroll
            for (int m = 0; m < 4; ++m)
#pragma unroll
                for (int n2 = 0; n2 < 4; ++n2) tW[(ty + 16 * m) * LDC + tx + 16 * n2] = acc[m][n2];
            if (tid < 64) {
                float s = 0.f;
                for (int j = 0; j < 16; ++j) s += red[j * 64 + tid];
                dbr[tid] = s;
            }
        }
        __syncthreads();
        {   // sdA = strict_lower(-T^T tmp) over M's tile
            float acc[4][4];
            zero(acc);
            mm<4, 4, C>(acc, [&](int r, int s) { return tT[s * LDC + r]; },
                        [&](int s, int j) { return tW[s * LDC + j]; });
#pragma unroll
            for (int m = 0; m < 4; ++m)
#pragma unroll
                for (int n2 = 0; n2 < 4; ++n2) {
                    const int r = ty + 16 * m, j = tx + 16 * n2;
                    tM[r * LDC + j] = j < r ? -acc[m][n2] : 0.f;
                }
        }
        __syncthreads();
        {   // dM = tril_incl(dP U^T) over the tmp tile
            float acc[4][4];
            zero(acc);
            mm<4, 4, R>(acc, [&](int r, int i) { return tP[r * LDC + i]; },
                        [&](int i, int s) { return tU[s * LDC + i]; });
#pragma unroll
            for (int m = 0; m < 4; ++m)
#pragma unroll
                for (int n2 = 0; n2 < 4; ++n2) {
                    const int r = ty + 16 * m, s = tx + 16 * n2;
                    tW[r * LDC + s] = s <= r ? acc[m][n2] : 0.f;
                }
        }
        __syncthreads();
        const size_t part_base = (size_t)rb * p.T;
        auto qk_idx = [&](int r, int c2) {
            return ((part_base + tok0 + r) * p.H + h) * DK + c2;
        };
        {   // dq = dP S + dM K
            float acc[4][8];
            zero(acc);
            mm<4, 8, R>(acc, [&](int r, int i) { return tP[r * LDC + i]; },
                        [&](int i, int c2) { return Ss[i * LDS + c2]; });
            mm<4, 8, C>(acc, [&](int r, int s) { return tW[r * LDC + s]; },
                        [&](int s, int c2) { return bf(Ks + s * LDH + c2); });
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int r = ty + 16 * m;
                if (r < nvalid)
#pragma unroll
                    for (int n2 = 0; n2 < 8; ++n2) p.dq_part[qk_idx(r, tx + 16 * n2)] = acc[m][n2];
            }
        }
        {   // dk = beta sdA K + dM^T Q + U dS^ - dY S + sdA^T beta K; dbeta += k . (sdA K)
            float acc[4][8];
            zero(acc);
            mm<4, 8, C>(acc, [&](int r, int s) { return tM[r * LDC + s]; },
                        [&](int s, int c2) { return bf(Ks + s * LDH + c2); });
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int r = ty + 16 * m;
                float part = 0.f;
#pragma unroll
                for (int n2 = 0; n2 < 8; ++n2) {
                    part = fmaf(bf(Ks + r * LDH + tx + 16 * n2), acc[m][n2], part);
                    acc[m][n2] *= bet[r];
                }
                red[tx * 64 + r] = part;
            }
            mm<4, 8, C>(acc, [&](int r, int s) { return tW[s * LDC + r]; },
                        [&](int s, int c2) { return bf(Qs + s * LDH + c2); });
            mm<4, 8, R>(acc, [&](int r, int i) { return tU[r * LDC + i]; },
                        [&](int i, int c2) { return Ds[i * LDS + c2]; });
            mm<4, 8, R>(acc, [&](int r, int i) { return -tY[r * LDC + i]; },
                        [&](int i, int c2) { return Ss[i * LDS + c2]; });
            mm<4, 8, C>(acc, [&](int r, int s) { return tM[s * LDC + r]; },
                        [&](int s, int c2) { return bet[s] * bf(Ks + s * LDH + c2); });
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int r = ty + 16 * m;
                if (r < nvalid)
#pragma unroll
                    for (int n2 = 0; n2 < 8; ++n2) p.dk_part[qk_idx(r, tx + 16 * n2)] = acc[m][n2];
            }
        }
        {   // ecol += rowsum(dS^ * S), four lanes per row
            const int i = tid >> 2, part = tid & 3;
            float s = 0.f;
            for (int c2 = part; c2 < DK; c2 += 4) s = fmaf(Ds[i * LDS + c2], Ss[i * LDS + c2], s);
            s += __shfl_xor_sync(0xffffffffu, s, 1);
            s += __shfl_xor_sync(0xffffffffu, s, 2);
            if (part == 0) ecol[i] += s;
        }
        __syncthreads();
        // E (with the state term on the last token) over Gamma's tile; dbeta out
#pragma unroll
        for (int m = 0; m < 4; ++m)
#pragma unroll
            for (int n2 = 0; n2 < 4; ++n2) {
                const int r = ty + 16 * m, i = tx + 16 * n2;
                tG[r * LDC + i] = E[m][n2] + (r == C - 1 ? ecol[i] : 0.f);
            }
        if (tid < 64 && tid < nvalid) {
            float s = dbr[tid];
            for (int j = 0; j < 16; ++j) s += red[j * 64 + tid];
            p.db_part[(part_base + tok0 + tid) * p.H + h] = s;
        }
        {   // D <- dS^ + dP^T Q - dY^T K
            float acc[4][8];
            zero(acc);
            mm<4, 8, C>(acc, [&](int i, int r) { return tP[r * LDC + i]; },
                        [&](int r, int c2) { return bf(Qs + r * LDH + c2); });
            mm<4, 8, C>(acc, [&](int i, int r) { return -tY[r * LDC + i]; },
                        [&](int r, int c2) { return bf(Ks + r * LDH + c2); });
#pragma unroll
            for (int m = 0; m < 4; ++m)
#pragma unroll
                for (int n2 = 0; n2 < 8; ++n2) Ds[(ty + 16 * m) * LDS + tx + 16 * n2] += acc[m][n2];
        }
        __syncthreads();
        if (tid < 64) {   // dalpha = reverse cumulative sum of E over tokens / alpha
            float run = 0.f;
            for (int r = C - 1; r >= 0; --r) {
                run += tG[r * LDC + tid];
                if (r < nvalid) {
                    const int64_t at = vidx(tok0 + r, tid);
                    p.dalpha[at] = run / p.alpha[at];
                }
            }
        }
        __syncthreads();
    }
    if (p.dS0) store_state(p.dS0 + ((size_t)n * p.H + h) * st_rows + (size_t)row0 * DK, Ds);
}

// dq, dk and dbeta: sums over the row blocks, in block order.
__global__ void kda_backward_reduce(const BwdParams p, float* __restrict__ dq,
                                    float* __restrict__ dk, float* __restrict__ dbeta) {
    if (*p.status != 0) return;
    const int64_t used = p.cu[p.N];
    const int64_t n4 = used * p.H * (DK / 4);
    const size_t part = (size_t)p.T * p.H * DK;
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < n4;
         e += (int64_t)gridDim.x * blockDim.x) {
        float4 sq = reinterpret_cast<const float4*>(p.dq_part)[e];
        float4 sk = reinterpret_cast<const float4*>(p.dk_part)[e];
        for (int b = 1; b < p.nrb; ++b) {
            const float4 xq = reinterpret_cast<const float4*>(p.dq_part + b * part)[e];
            const float4 xk = reinterpret_cast<const float4*>(p.dk_part + b * part)[e];
            sq.x += xq.x; sq.y += xq.y; sq.z += xq.z; sq.w += xq.w;
            sk.x += xk.x; sk.y += xk.y; sk.z += xk.z; sk.w += xk.w;
        }
        reinterpret_cast<float4*>(dq)[e] = sq;
        reinterpret_cast<float4*>(dk)[e] = sk;
        if (e < used * p.H) {
            float s = p.db_part[e];
            for (int b = 1; b < p.nrb; ++b) s += p.db_part[b * (size_t)p.T * p.H + e];
            dbeta[e] = s;
        }
    }
}

}  // namespace

BackwardLayout backward_layout(int32_t num_seqs, int64_t total_tokens, int32_t H, int32_t d_v) {
    BackwardLayout L;
    size_t off = WorkspaceLayout::bytes(num_seqs);
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = (off + bytes + 255) & ~(size_t)255;
        return at;
    };
    const size_t N = num_seqs > 0 ? (size_t)num_seqs : 0, T = total_tokens > 0 ? (size_t)total_tokens : 0;
    const size_t nrb = (size_t)(d_v > 0 ? d_v : 0) / R;
    const size_t slots = (T + C - 1) / C + N;
    L.ckpt = take(slots * H * (size_t)d_v * DK * sizeof(float));
    L.dq_part = take(nrb * T * H * DK * sizeof(float));
    L.dk_part = take(nrb * T * H * DK * sizeof(float));
    L.db_part = take(nrb * T * H * sizeof(float));
    L.end = off;
    return L;
}

cudaError_t launch_backward(const BackwardArgs& a, const BackwardLayout& L, char* ws,
                            cudaStream_t stream) {
    BwdParams p;
    p.q = static_cast<const __nv_bfloat16*>(a.q);
    p.k = static_cast<const __nv_bfloat16*>(a.k);
    p.v = static_cast<const __nv_bfloat16*>(a.v);
    p.dO = static_cast<const __nv_bfloat16*>(a.dO);
    p.alpha = a.alpha; p.beta = a.beta; p.S0 = a.S0; p.dS_T = a.dS_T;
    p.cu = a.cu_seqlens;
    p.order = reinterpret_cast<const int32_t*>(ws + WorkspaceLayout::kOrder);
    p.status = reinterpret_cast<const int32_t*>(ws + WorkspaceLayout::kStatus);
    p.N = a.num_seqs; p.H = a.H; p.d_v = a.d_v; p.nrb = a.d_v / R;
    p.T = a.total_tokens;
    p.ckpt = reinterpret_cast<float*>(ws + L.ckpt);
    p.dq_part = reinterpret_cast<float*>(ws + L.dq_part);
    p.dk_part = reinterpret_cast<float*>(ws + L.dk_part);
    p.db_part = reinterpret_cast<float*>(ws + L.db_part);
    p.dv = a.dv; p.dalpha = a.dalpha; p.dS0 = a.dS0;
    cudaError_t err = cudaFuncSetAttribute(kda_backward_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (err != cudaSuccess) return err;
    const int blocks = a.num_seqs * a.H * p.nrb;
    kda_backward_kernel<<<blocks, NTH, SMEM_BYTES, stream>>>(p);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    if (a.total_tokens == 0) return cudaSuccess;
    const int rblocks = 4 * sm_count();
    kda_backward_reduce<<<rblocks > 0 ? rblocks : 1, 256, 0, stream>>>(p, a.dq, a.dk, a.dbeta);
    return cudaGetLastError();
}

}  // namespace kda
