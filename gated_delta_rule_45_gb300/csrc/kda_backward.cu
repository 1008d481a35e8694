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
//             dk = dM^T Q + U dS^ - dY S + diag(beta) sdA K + (diag(beta) sdA)^T K
//             dv = dY / Gamma
//             dbeta_r = sum_i dX_ri Y_ri + k_r . (sdA K)_r
//             E = dP * P - dY * V / Gamma,  E[C-1] += rowsum(dS^ * (S + U^T K))
//             dalpha = reverse_cumsum_over_tokens(E) / alpha
//             D <- dS^ + dP^T Q - dY^T K
//
// Value channels (rows of S) only interact through sums that end in dq, dk
// and dbeta, so one CTA owns one (sequence, head, 64-row block) chain and
// walks its chunks in reverse.  The chunk-start states it needs come from the
// tensor-core prefill (launched first, writing them to the workspace) when
// d_v is a multiple of 128; for other widths the CTA first runs a forward
// sweep of its own, keeping the states and each chunk's T.  dq, dk and dbeta
// are written per row block and summed by a second kernel in a fixed order,
// so results are deterministic.
//
// Every product is a warp-level bf16 tensor-core MMA (m16n8k16, fp32
// accumulate) on shared-memory tiles loaded with ldmatrix.  Values that are
// not bf16 already are carried as hi + lo bf16 pairs (hi = bf16(x),
// lo = bf16(x - hi)) and multiplied as hi*hi + hi*lo + lo*hi, which keeps
// about 16 bits of each operand: q, k, v and dO are bf16 inputs and need no
// lo part.  The state S (forward sweep) and the state gradient D (backward
// sweep) stay in fp32 accumulator registers across chunks; only their bf16
// hi/lo copies go to shared memory as operands.
#include "kda_internal.h"

namespace kda {
namespace {

constexpr int C = 64;      // tokens per chunk
constexpr int DK = 128;    // key channels
constexpr int R = 64;      // value rows per CTA
constexpr int NTH = 256;   // 8 warps

// Shared memory.  bf16 tiles are row-major with their 16-byte chunks
// XOR-swizzled by (row & 7), so ldmatrix rows and fragment stores hit
// distinct banks.  64 x 128 tiles: K, Q, S hi/lo, D hi/lo.  64 x 64 tiles
// come in hi/lo pairs; a pair's 16 KB also holds a 64 x 64 fp32 matrix while
// T is being built.  G: fp32 64 x 64 (Gamma, later E).
constexpr int BIG = 64 * 128 * 2;
constexpr int SMALL = 64 * 64 * 2;
constexpr int PAIR = 2 * SMALL;
constexpr int OFF_K = 0;
constexpr int OFF_Q = OFF_K + BIG;
constexpr int OFF_SH = OFF_Q + BIG;
constexpr int OFF_SL = OFF_SH + BIG;
constexpr int OFF_DH = OFF_SL + BIG;
constexpr int OFF_DL = OFF_DH + BIG;
constexpr int OFF_PAIR = OFF_DL + BIG;
enum { P_A = 0, P_T, P_X, P_U, P_P, P_W, N_PAIR };
constexpr int OFF_G = OFF_PAIR + N_PAIR * PAIR;
constexpr int OFF_RED = OFF_G + 64 * 64 * 4;     // fp32 [8][64]
constexpr int OFF_MISC = OFF_RED + 8 * 64 * 4;   // beta, gamma_C, ecol, dbeta (64 each)
constexpr int OFF_V = OFF_MISC + 4 * 64 * 4;     // the chunk's V and dO, swizzled 64 x 64 bf16
constexpr int OFF_DO = OFF_V + SMALL;
constexpr int SMEM_BYTES = OFF_DO + SMALL;
static_assert(SMEM_BYTES <= 232448, "shared memory");

__host__ __device__ constexpr int pair_hi(int p) { return OFF_PAIR + p * PAIR; }
__host__ __device__ constexpr int pair_lo(int p) { return OFF_PAIR + p * PAIR + SMALL; }

struct BwdParams {
    const __nv_bfloat16 *q, *k, *v, *dO;
    const float *alpha, *beta, *S0, *dS_T;
    const int32_t *cu, *order, *status;
    int32_t N, H, d_v, nrb;
    int64_t T;
    float* ckpt;              // [slots][H][d_v][DK], slot = t0 / C + n + chunk
    uint4* tbuf;              // [slots][H][nrb] the chunk's T pair (PAIR bytes)
    int32_t tc_ckpt;          // ckpt already written by the tensor-core forward
    float *dq_part, *dk_part; // [nrb][T][H][DK]
    float* db_part;           // [nrb][T][H]
    float *dv, *dalpha;       // [T][H][d_v]
    float* dS0;               // [N][H][d_v][DK] or null
};

// Byte offset of element (row, col) of a swizzled bf16 tile with `wb` bytes per row.
__device__ __forceinline__ uint32_t swz(int row, int col, int wb) {
    return (uint32_t)(row * wb + ((((col >> 3) ^ row) & 7) << 4) + (((col >> 3) & ~7) << 4) +
                      ((col & 7) << 1));
}

// Index of (row, col) in a 64 x 64 fp32 matrix, 4-word groups XOR-swizzled by row.
__device__ __forceinline__ int gidx(int r, int c) { return r * 64 + (c ^ ((r & 7) << 2)); }

__device__ __forceinline__ void ldsm4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr) : "memory");
}
__device__ __forceinline__ void ldsm4t(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr) : "memory");
}
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// A tile operand: shared-memory addresses of its hi and lo parts, bytes per row.
struct Op {
    uint32_t hi, lo;
    int wb;
};

// c[nt] += sum over k < 16 KS of A(m, k) B(k, n) for the warp's 16 x 8 NT
// tile at (m0, n0).  TA: A(m, k) is stored at [k][m] (else [m][k]); TB: B(k, n)
// is stored at [k][n] (else [n][k]).  ALO / BLO: the operand has a lo part.
template <int NT, int KS, bool TA, bool TB, bool ALO, bool BLO>
__device__ __forceinline__ void mma_tile(float (&c)[NT][4], const Op& A, const Op& B, int m0,
                                         int n0) {
    const int l = threadIdx.x & 31;
    const int r8 = l & 7, j1 = (l >> 3) & 1, j2 = l >> 4;
#pragma unroll 2
    for (int ks = 0; ks < KS; ++ks) {
        const int k = 16 * ks;
        uint32_t ah[4], al[4], bh[NT / 2][4], bl[NT / 2][4];
        const uint32_t aoff = TA ? swz(k + r8 + 8 * j2, m0 + 8 * j1, A.wb)
                                 : swz(m0 + r8 + 8 * j1, k + 8 * j2, A.wb);
        if (TA) ldsm4t(A.hi + aoff, ah); else ldsm4(A.hi + aoff, ah);
        if (ALO) { if (TA) ldsm4t(A.lo + aoff, al); else ldsm4(A.lo + aoff, al); }
#pragma unroll
        for (int np = 0; np < NT / 2; ++np) {
            const int n = n0 + 16 * np;
            const uint32_t boff = TB ? swz(k + r8 + 8 * j1, n + 8 * j2, B.wb)
                                     : swz(n + r8 + 8 * j2, k + 8 * j1, B.wb);
            if (TB) ldsm4t(B.hi + boff, bh[np]); else ldsm4(B.hi + boff, bh[np]);
            if (BLO) { if (TB) ldsm4t(B.lo + boff, bl[np]); else ldsm4(B.lo + boff, bl[np]); }
        }
        // pass by pass over all n-tiles, so that dependent MMAs are NT apart
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma16816(c[nt], ah, bh[nt >> 1][2 * (nt & 1)], bh[nt >> 1][2 * (nt & 1) + 1]);
        if (BLO) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma16816(c[nt], ah, bl[nt >> 1][2 * (nt & 1)], bl[nt >> 1][2 * (nt & 1) + 1]);
        }
        if (ALO) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma16816(c[nt], al, bh[nt >> 1][2 * (nt & 1)], bh[nt >> 1][2 * (nt & 1) + 1]);
        }
    }
}

template <int NT>
__device__ __forceinline__ void zero(float (&c)[NT][4]) {
#pragma unroll
    for (int i = 0; i < NT; ++i) c[i][0] = c[i][1] = c[i][2] = c[i][3] = 0.f;
}

// (x0, x1) at (row, col), col even, as hi and lo bf16 pairs into a swizzled tile.
__device__ __forceinline__ void st_pair(char* sm, int off_hi, int off_lo, int wb, int row,
                                        int col, float x0, float x1) {
    const uint32_t o = swz(row, col, wb);
    const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
    const float2 hf = __bfloat1622float2(h);
    *reinterpret_cast<__nv_bfloat162*>(sm + off_hi + o) = h;
    *reinterpret_cast<__nv_bfloat162*>(sm + off_lo + o) =
        __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
}

__device__ __forceinline__ float2 ld_pair(const char* sm, int off_hi, int off_lo, int wb, int row,
                                          int col) {
    const uint32_t o = swz(row, col, wb);
    const float2 h = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(sm + off_hi + o));
    const float2 l = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(sm + off_lo + o));
    return make_float2(h.x + l.x, h.y + l.y);
}

// (row, col) and (row, col + 1) of a swizzled 64 x 64 bf16 tile, as floats.
__device__ __forceinline__ float2 ld_tile2(const char* sm, int off, int row, int col) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(sm + off + swz(row, col, 128)));
}

__device__ __forceinline__ void cp16(char* dst, const void* src, bool ok) {
    const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n"
                 :: "r"(d), "l"(src), "r"(ok ? 16 : 0) : "memory");
}

// Asynchronous copies of one chunk's inputs into shared memory: K and this
// block's 64 channels of V and alpha (alpha into G), plus Q and dO in the
// backward sweep and the chunk's stored T when `tglob` is given.  Rows at or
// past nvalid are zero-filled.
__device__ void prefetch_chunk(const BwdParams& p, char* sm, int64_t tok0, int nvalid, int h,
                               int row0, bool backward, const uint4* tglob) {
    const int tid = threadIdx.x;
    const int64_t vstride = (int64_t)p.H * p.d_v;
#pragma unroll
    for (int e = tid; e < 64 * 16; e += NTH) {   // K, Q: 64 rows of 16 pieces
        const int row = e >> 4, c = e & 15;
        const bool ok = row < nvalid;
        const int64_t off = ok ? ((tok0 + row) * p.H + h) * DK + 8 * c : 0;
        cp16(sm + OFF_K + swz(row, 8 * c, 256), p.k + off, ok);
        if (backward) cp16(sm + OFF_Q + swz(row, 8 * c, 256), p.q + off, ok);
    }
#pragma unroll
    for (int e = tid; e < 64 * 8; e += NTH) {    // V, dO: 64 rows of 8 pieces
        const int row = e >> 3, c = e & 7;
        const bool ok = row < nvalid;
        const int64_t off = ok ? (tok0 + row) * vstride + (int64_t)h * p.d_v + row0 + 8 * c : 0;
        cp16(sm + OFF_V + swz(row, 8 * c, 128), p.v + off, ok);
        if (backward) cp16(sm + OFF_DO + swz(row, 8 * c, 128), p.dO + off, ok);
    }
#pragma unroll
    for (int e = tid; e < 64 * 16; e += NTH) {   // alpha: 64 rows of 16 groups of 4 channels
        const int row = e >> 4, c = 4 * (e & 15);
        const bool ok = row < nvalid;
        const int64_t off = ok ? (tok0 + row) * vstride + (int64_t)h * p.d_v + row0 + c : 0;
        cp16(sm + OFF_G + 4 * gidx(row, c), p.alpha + off, ok);
    }
    if (tglob) {
#pragma unroll
        for (int e = tid; e < PAIR / 16; e += NTH) cp16(sm + pair_hi(P_T) + 16 * e, tglob + e, true);
    }
    asm volatile("cp.async.commit_group;\n" ::: "memory");
}

// Fragment coordinates of the calling thread: a 64 x 64 output is tiled by the
// 8 warps as 4 (rows) x 2 (32 columns), a 64 x 128 output as 4 x 2 (64 columns).
struct Frag {
    int m0, n64, n128, g, t;
    __device__ Frag() {
        const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
        m0 = 16 * (w & 3);
        n64 = 32 * (w >> 2);
        n128 = 64 * (w >> 2);
        g = l >> 2;
        t = l & 3;
    }
    __device__ int row(int e) const { return m0 + g + 8 * (e >> 1); }
    __device__ int col64(int nt) const { return n64 + 8 * nt + 2 * t; }
    __device__ int col128(int nt) const { return n128 + 8 * nt + 2 * t; }
};

// Per-chunk inputs shared by both sweeps, after prefetch_chunk: beta, Gamma,
// gamma_C and T = (I + diag(beta) strict_lower(K K^T))^-1 as a hi/lo pair,
// built here when `build_t` (a copy kept at `tstore` when given), else already
// prefetched from the forward sweep's copy.
__device__ void chunk_setup(const BwdParams& p, char* sm, int64_t tok0, int nvalid, int h,
                            int row0, bool build_t, uint4* tstore, const Frag& f) {
    float* G = reinterpret_cast<float*>(sm + OFF_G);
    float* Lf = reinterpret_cast<float*>(sm + pair_hi(P_A));
    float* Tf = reinterpret_cast<float*>(sm + pair_hi(P_T));
    float* bet = reinterpret_cast<float*>(sm + OFF_MISC);
    float* gC = bet + 64;
    const int tid = threadIdx.x;
    if (tid < C) bet[tid] = tid < nvalid ? p.beta[(tok0 + tid) * p.H + h] : 0.f;
    asm volatile("cp.async.wait_all;\n" ::: "memory");
    __syncthreads();
    {   // Gamma over alpha in G: four threads per value channel, 16 tokens each,
        // products scanned across them
        const int i = tid >> 2, part = tid & 3;
        float a[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int r = 16 * part + j;
            a[j] = r < nvalid ? G[gidx(r, i)] : 1.f;
        }
#pragma unroll
        for (int j = 1; j < 16; ++j) a[j] *= a[j - 1];
        float s = a[15], y;
        y = __shfl_up_sync(0xffffffffu, s, 1);
        if (part >= 1) s *= y;
        y = __shfl_up_sync(0xffffffffu, s, 2);
        if (part >= 2) s *= y;
        float before = __shfl_up_sync(0xffffffffu, s, 1);
        if (part == 0) before = 1.f;
#pragma unroll
        for (int j = 0; j < 16; ++j) G[gidx(16 * part + j, i)] = before * a[j];
        if (part == 3) gC[i] = s;
    }
    if (!build_t) {
        __syncthreads();
        return;
    }
    for (int e = tid; e < C * C; e += NTH) Tf[gidx(e >> 6, e & 63)] = (e >> 6) == (e & 63) ? 1.f : 0.f;
    __syncthreads();
    {   // L' = diag(beta) strict_lower(K K^T), fp32
        float c[4][4];
        zero(c);
        const Op K{(uint32_t)__cvta_generic_to_shared(sm + OFF_K), 0u, 256};
        mma_tile<4, 8, false, false, false, false>(c, K, K, f.m0, f.n64);
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int e = 0; e < 4; e += 2) {
                const int r = f.row(e), s = f.col64(nt);
                Lf[gidx(r, s)] = s < r ? bet[r] * c[nt][e] : 0.f;
                Lf[gidx(r, s + 1)] = s + 1 < r ? bet[r] * c[nt][e + 1] : 0.f;
            }
    }
    __syncthreads();
    {   // row r of T: T[r][j] = -sum_{s<r} L'[r][s] T[s][j] for j < r; four lanes per column
        const int j = tid >> 2, part = tid & 3;
        for (int r = 1; r < C; ++r) {
            float acc = 0.f;
            for (int s = part; s < r; s += 4) acc = fmaf(Lf[gidx(r, s)], Tf[gidx(s, j)], acc);
            acc += __shfl_xor_sync(0xffffffffu, acc, 1);
            acc += __shfl_xor_sync(0xffffffffu, acc, 2);
            if (part == 0 && j < r) Tf[gidx(r, j)] = -acc;
            __syncwarp();
        }
    }
    __syncthreads();
    {   // T as a hi/lo pair over its own fp32 storage
        float2 v[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int e = tid + NTH * q;
            v[q] = *reinterpret_cast<const float2*>(Tf + gidx(e >> 5, 2 * (e & 31)));
        }
        __syncthreads();
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int e = tid + NTH * q;
            st_pair(sm, pair_hi(P_T), pair_lo(P_T), 128, e >> 5, 2 * (e & 31), v[q].x, v[q].y);
        }
    }
    __syncthreads();
    if (tstore) {
        const uint4* tsm = reinterpret_cast<const uint4*>(sm + pair_hi(P_T));
#pragma unroll
        for (int e = tid; e < PAIR / 16; e += NTH) tstore[e] = tsm[e];
    }
}

__global__ void __launch_bounds__(NTH, 1) kda_backward_kernel(const BwdParams p) {
    if (*p.status == KDA_ERR_DEVICE_INPUT) return;
    extern __shared__ __align__(128) char sm[];
    const uint32_t sb = (uint32_t)__cvta_generic_to_shared(sm);
    float* G = reinterpret_cast<float*>(sm + OFF_G);
    // red rows: 0-3 column sums of U * K dS^^T (one per row group of warps), later
    // 0-1 the rowsums of dS^ * S; 4-5 and 6-7 the two parts of dbeta (one per column half)
    float* red = reinterpret_cast<float*>(sm + OFF_RED);
    float* bet = reinterpret_cast<float*>(sm + OFF_MISC);
    float* gC = bet + 64;
    float* ecol = bet + 128;
    float* dbr = bet + 192;
    const Frag f;
    const int tid = threadIdx.x, w = tid >> 5;

    const int rb = blockIdx.x % p.nrb;
    const int h = (blockIdx.x / p.nrb) % p.H;
    const int n = p.order[blockIdx.x / (p.nrb * p.H)];
    const int64_t t0 = p.cu[n];
    const int len = p.cu[n + 1] - p.cu[n];
    const int nc = (len + C - 1) / C;
    const int row0 = rb * R;
    const int64_t slot0 = t0 / C + n;
    const size_t st_rows = (size_t)p.d_v * DK;   // one head's state
    const size_t head_state = ((size_t)n * p.H + h) * st_rows + (size_t)row0 * DK;
    auto ckpt_at = [&](int c) {
        return p.ckpt + ((size_t)(slot0 + c) * p.H + h) * st_rows + (size_t)row0 * DK;
    };
    auto tbuf_at = [&](int c) {
        return p.tbuf + (((size_t)(slot0 + c) * p.H + h) * p.nrb + rb) * (PAIR / 16);
    };
    const int64_t vstride = (int64_t)p.H * p.d_v;
    auto vidx = [&](int64_t tok, int i) { return tok * vstride + (int64_t)h * p.d_v + row0 + i; };

    const Op opK{sb + OFF_K, 0u, 256}, opQ{sb + OFF_Q, 0u, 256};
    const Op opS{sb + OFF_SH, sb + OFF_SL, 256}, opD{sb + OFF_DH, sb + OFF_DL, 256};
    auto pop = [&](int pi) { return Op{sb + pair_hi(pi), sb + pair_lo(pi), 128}; };
    const Op opA = pop(P_A), opT = pop(P_T), opX = pop(P_X), opU = pop(P_U), opP = pop(P_P),
             opW = pop(P_W);

    // ---- forward sweep: chunk-start states into the workspace (unless the
    // tensor-core forward has written them) ----
    if (!p.tc_ckpt) {
        float Sm[8][4];   // this block's rows of S, fp32, in accumulator layout
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; e += 2) {
                const int r = f.row(e), col = f.col128(nt);
                float2 x = make_float2(0.f, 0.f);
                if (p.S0) x = *reinterpret_cast<const float2*>(p.S0 + head_state + r * DK + col);
                Sm[nt][e] = x.x;
                Sm[nt][e + 1] = x.y;
                st_pair(sm, OFF_SH, OFF_SL, 256, r, col, x.x, x.y);
            }
        __syncthreads();
        for (int c = 0; c < nc; ++c) {
            const int64_t tok0 = t0 + (int64_t)c * C;
            const int nvalid = min(C, len - c * C);
            float* ck = ckpt_at(c);
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                for (int e = 0; e < 4; e += 2)
                    *reinterpret_cast<float2*>(ck + f.row(e) * DK + f.col128(nt)) =
                        make_float2(Sm[nt][e], Sm[nt][e + 1]);
            prefetch_chunk(p, sm, tok0, nvalid, h, row0, false, nullptr);
            chunk_setup(p, sm, tok0, nvalid, h, row0, true, tbuf_at(c), f);
            {   // X = diag(beta) (V / Gamma - K S^T)
                float cY[4][4];
                zero(cY);
                mma_tile<4, 8, false, false, false, true>(cY, opK, opS, f.m0, f.n64);
#pragma unroll
                for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; e += 2) {
                        const int r = f.row(e), i = f.col64(nt);
                        const float2 vv = ld_tile2(sm, OFF_V, r, i);
                        const float y0 = vv.x / G[gidx(r, i)] - cY[nt][e];
                        const float y1 = vv.y / G[gidx(r, i + 1)] - cY[nt][e + 1];
                        st_pair(sm, pair_hi(P_X), pair_lo(P_X), 128, r, i, bet[r] * y0, bet[r] * y1);
                    }
            }
            __syncthreads();
            {   // U = T X
                float cU[4][4];
                zero(cU);
                mma_tile<4, 4, false, true, true, true>(cU, opT, opX, f.m0, f.n64);
#pragma unroll
                for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; e += 2)
                        st_pair(sm, pair_hi(P_U), pair_lo(P_U), 128, f.row(e), f.col64(nt),
                                cU[nt][e], cU[nt][e + 1]);
            }
            __syncthreads();
            // S <- diag(gamma_C) (S + U^T K)
            mma_tile<8, 4, true, true, true, false>(Sm, opU, opK, f.m0, f.n128);
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                for (int e = 0; e < 4; e += 2) {
                    const int r = f.row(e), col = f.col128(nt);
                    Sm[nt][e] *= gC[r];
                    Sm[nt][e + 1] *= gC[r];
                    st_pair(sm, OFF_SH, OFF_SL, 256, r, col, Sm[nt][e], Sm[nt][e + 1]);
                }
            __syncthreads();
        }
    }

    // ---- backward sweep ----
    float Dm[8][4];   // this block's rows of D (dL/d state at the chunk's end), fp32
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; e += 2) {
            float2 x = make_float2(0.f, 0.f);
            if (p.dS_T)
                x = *reinterpret_cast<const float2*>(p.dS_T + head_state + f.row(e) * DK + f.col128(nt));
            Dm[nt][e] = x.x;
            Dm[nt][e + 1] = x.y;
        }
    for (int c = nc - 1; c >= 0; --c) {
        const int64_t tok0 = t0 + (int64_t)c * C;
        const int nvalid = min(C, len - c * C);
        prefetch_chunk(p, sm, tok0, nvalid, h, row0, true, p.tc_ckpt ? nullptr : tbuf_at(c));
        {   // the chunk-start state as hi/lo tiles
            const float* ck = ckpt_at(c);
#pragma unroll
            for (int e = tid; e < 64 * 32; e += NTH) {
                const int r = e >> 5, col = 4 * (e & 31);
                const float4 x = *reinterpret_cast<const float4*>(ck + r * DK + col);
                st_pair(sm, OFF_SH, OFF_SL, 256, r, col, x.x, x.y);
                st_pair(sm, OFF_SH, OFF_SL, 256, r, col + 2, x.z, x.w);
            }
        }
        chunk_setup(p, sm, tok0, nvalid, h, row0, p.tc_ckpt != 0, nullptr, f);
        {   // M = tril_incl(Q K^T) into pair A
            float cM[4][4];
            zero(cM);
            mma_tile<4, 8, false, false, false, false>(cM, opQ, opK, f.m0, f.n64);
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int e = 0; e < 4; e += 2) {
                    const int r = f.row(e), s = f.col64(nt);
                    st_pair(sm, pair_hi(P_A), pair_lo(P_A), 128, r, s, s <= r ? cM[nt][e] : 0.f,
                            s + 1 <= r ? cM[nt][e + 1] : 0.f);
                }
        }
        float Y[4][4], dP[4][4];
        {   // Y = V / Gamma - K S^T, X = diag(beta) Y into pair X, dP = Gamma * dO into pair P
            zero(Y);
            mma_tile<4, 8, false, false, false, true>(Y, opK, opS, f.m0, f.n64);
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int e = 0; e < 4; e += 2) {
                    const int r = f.row(e), i = f.col64(nt);
                    const float2 vv = ld_tile2(sm, OFF_V, r, i);
                    const float2 dd = ld_tile2(sm, OFF_DO, r, i);
                    const float g0 = G[gidx(r, i)], g1 = G[gidx(r, i + 1)];
                    Y[nt][e] = vv.x / g0 - Y[nt][e];
                    Y[nt][e + 1] = vv.y / g1 - Y[nt][e + 1];
                    st_pair(sm, pair_hi(P_X), pair_lo(P_X), 128, r, i, bet[r] * Y[nt][e],
                            bet[r] * Y[nt][e + 1]);
                    dP[nt][e] = g0 * dd.x;
                    dP[nt][e + 1] = g1 * dd.y;
                    st_pair(sm, pair_hi(P_P), pair_lo(P_P), 128, r, i, dP[nt][e], dP[nt][e + 1]);
                }
        }
        __syncthreads();
        float U[4][4];
        {   // U = T X into pair U; dS^ = diag(gamma_C) D as hi/lo tiles
            zero(U);
            mma_tile<4, 4, false, true, true, true>(U, opT, opX, f.m0, f.n64);
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int e = 0; e < 4; e += 2)
                    st_pair(sm, pair_hi(P_U), pair_lo(P_U), 128, f.row(e), f.col64(nt), U[nt][e],
                            U[nt][e + 1]);
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                for (int e = 0; e < 4; e += 2) {
                    const int r = f.row(e);
                    Dm[nt][e] *= gC[r];
                    Dm[nt][e + 1] *= gC[r];
                    st_pair(sm, OFF_DH, OFF_DL, 256, r, f.col128(nt), Dm[nt][e], Dm[nt][e + 1]);
                }
        }
        __syncthreads();
        float E[4][4];
        {   // E = dP * (Q S^T + M U)
            zero(E);
            mma_tile<4, 8, false, false, false, true>(E, opQ, opS, f.m0, f.n64);
            mma_tile<4, 4, false, true, true, true>(E, opA, opU, f.m0, f.n64);
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) E[nt][e] *= dP[nt][e];
        }
        {   // Z = K dS^^T; column sums of U * Z; dU = Z + M^T dP into pair W
            float Z[4][4];
            zero(Z);
            mma_tile<4, 8, false, false, false, true>(Z, opK, opD, f.m0, f.n64);
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    float s = fmaf(U[nt][q], Z[nt][q], U[nt][q + 2] * Z[nt][q + 2]);
                    s += __shfl_xor_sync(0xffffffffu, s, 4);
                    s += __shfl_xor_sync(0xffffffffu, s, 8);
                    s += __shfl_xor_sync(0xffffffffu, s, 16);
                    if (f.g == 0) red[(w & 3) * 64 + f.col64(nt) + q] = s;
                }
            mma_tile<4, 4, true, true, true, true>(Z, opA, opP, f.m0, f.n64);
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int e = 0; e < 4; e += 2)
                    st_pair(sm, pair_hi(P_W), pair_lo(P_W), 128, f.row(e), f.col64(nt), Z[nt][e],
                            Z[nt][e + 1]);
        }
        __syncthreads();
        {   // dT = dU X^T into pair A; finish the column sums
            float c2[4][4];
            zero(c2);
            mma_tile<4, 4, false, false, true, true>(c2, opW, opX, f.m0, f.n64);
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int e = 0; e < 4; e += 2)
                    st_pair(sm, pair_hi(P_A), pair_lo(P_A), 128, f.row(e), f.col64(nt), c2[nt][e],
                            c2[nt][e + 1]);
            if (tid < 64) ecol[tid] = red[tid] + red[64 + tid] + red[128 + tid] + red[192 + tid];
        }
        __syncthreads();
        {   // dX = T^T dU: dbeta (first part), -dY into pair X, dv, E -= dY V / Gamma
            float c2[4][4];
            zero(c2);
            mma_tile<4, 4, true, true, true, true>(c2, opT, opW, f.m0, f.n64);
            float part[2] = {0.f, 0.f};
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int e = 0; e < 4; e += 2) {
                    const int r = f.row(e), i = f.col64(nt);
                    const bool ok = r < nvalid;
                    part[e >> 1] = fmaf(c2[nt][e], Y[nt][e], fmaf(c2[nt][e + 1], Y[nt][e + 1], part[e >> 1]));
                    const float dy0 = bet[r] * c2[nt][e], dy1 = bet[r] * c2[nt][e + 1];
                    st_pair(sm, pair_hi(P_X), pair_lo(P_X), 128, r, i, -dy0, -dy1);
                    const float g0 = G[gidx(r, i)], g1 = G[gidx(r, i + 1)];
                    const float2 vv = ld_tile2(sm, OFF_V, r, i);
                    E[nt][e] -= dy0 * vv.x / g0;
                    E[nt][e + 1] -= dy1 * vv.y / g1;
                    if (ok)
                        *reinterpret_cast<float2*>(p.dv + vidx(tok0 + r, i)) = make_float2(dy0 / g0, dy1 / g1);
                }
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                float s = part[q];
                s += __shfl_xor_sync(0xffffffffu, s, 1);
                s += __shfl_xor_sync(0xffffffffu, s, 2);
                if (f.t == 0) red[(4 + (w >> 2)) * 64 + f.m0 + f.g + 8 * q] = s;
            }
        }
        __syncthreads();
        {   // dT T^T into pair W; finish the first dbeta part
            float c2[4][4];
            zero(c2);
            mma_tile<4, 4, false, false, true, true>(c2, opA, opT, f.m0, f.n64);
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int e = 0; e < 4; e += 2)
                    st_pair(sm, pair_hi(P_W), pair_lo(P_W), 128, f.row(e), f.col64(nt), c2[nt][e],
                            c2[nt][e + 1]);
            if (tid < 64) dbr[tid] = red[256 + tid] + red[320 + tid];
        }
        __syncthreads();
        {   // sdA = strict_lower(-T^T (dT T^T)) into pair A
            float c2[4][4];
            zero(c2);
            mma_tile<4, 4, true, true, true, true>(c2, opT, opW, f.m0, f.n64);
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int e = 0; e < 4; e += 2) {
                    const int r = f.row(e), j = f.col64(nt);
                    st_pair(sm, pair_hi(P_A), pair_lo(P_A), 128, r, j, j < r ? -c2[nt][e] : 0.f,
                            j + 1 < r ? -c2[nt][e + 1] : 0.f);
                }
        }
        __syncthreads();
        {   // dM = tril_incl(dP U^T) into pair W; diag(beta) sdA into pair T
            float c2[4][4];
            zero(c2);
            mma_tile<4, 4, false, false, true, true>(c2, opP, opU, f.m0, f.n64);
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int e = 0; e < 4; e += 2) {
                    const int r = f.row(e), s = f.col64(nt);
                    st_pair(sm, pair_hi(P_W), pair_lo(P_W), 128, r, s, s <= r ? c2[nt][e] : 0.f,
                            s + 1 <= r ? c2[nt][e + 1] : 0.f);
                }
            for (int e2 = tid; e2 < 64 * 32; e2 += NTH) {
                const int r = e2 >> 5, s = 2 * (e2 & 31);
                const float2 a = ld_pair(sm, pair_hi(P_A), pair_lo(P_A), 128, r, s);
                st_pair(sm, pair_hi(P_T), pair_lo(P_T), 128, r, s, bet[r] * a.x, bet[r] * a.y);
            }
        }
        __syncthreads();
        const size_t part_base = (size_t)rb * p.T;
        auto qk_idx = [&](int r, int col) { return ((part_base + tok0 + r) * p.H + h) * DK + col; };
        {   // dq = dP S + dM K
            float c8[8][4];
            zero(c8);
            mma_tile<8, 4, false, true, true, true>(c8, opP, opS, f.m0, f.n128);
            mma_tile<8, 4, false, true, true, false>(c8, opW, opK, f.m0, f.n128);
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                for (int e = 0; e < 4; e += 2) {
                    const int r = f.row(e);
                    if (r < nvalid)
                        *reinterpret_cast<float2*>(p.dq_part + qk_idx(r, f.col128(nt))) =
                            make_float2(c8[nt][e], c8[nt][e + 1]);
                }
        }
        {   // dk = diag(beta) sdA K + dM^T Q + U dS^ - dY S + (diag(beta) sdA)^T K;
            // dbeta second part k_r . (sdA K)_r
            float c8[8][4];
            zero(c8);
            mma_tile<8, 4, false, true, true, false>(c8, opA, opK, f.m0, f.n128);
            float part[2] = {0.f, 0.f};
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                for (int e = 0; e < 4; e += 2) {
                    const int r = f.row(e), col = f.col128(nt);
                    const float2 kk = __bfloat1622float2(
                        *reinterpret_cast<const __nv_bfloat162*>(sm + OFF_K + swz(r, col, 256)));
                    part[e >> 1] = fmaf(kk.x, c8[nt][e], fmaf(kk.y, c8[nt][e + 1], part[e >> 1]));
                    c8[nt][e] *= bet[r];
                    c8[nt][e + 1] *= bet[r];
                }
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                float s = part[q];
                s += __shfl_xor_sync(0xffffffffu, s, 1);
                s += __shfl_xor_sync(0xffffffffu, s, 2);
                if (f.t == 0) red[(6 + (w >> 2)) * 64 + f.m0 + f.g + 8 * q] = s;
            }
            mma_tile<8, 4, true, true, true, false>(c8, opW, opQ, f.m0, f.n128);
            mma_tile<8, 4, false, true, true, true>(c8, opU, opD, f.m0, f.n128);
            mma_tile<8, 4, false, true, true, true>(c8, opX, opS, f.m0, f.n128);
            mma_tile<8, 4, true, true, true, false>(c8, opT, opK, f.m0, f.n128);
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                for (int e = 0; e < 4; e += 2) {
                    const int r = f.row(e);
                    if (r < nvalid)
                        *reinterpret_cast<float2*>(p.dk_part + qk_idx(r, f.col128(nt))) =
                            make_float2(c8[nt][e], c8[nt][e + 1]);
                }
        }
        {   // rowsum(dS^ * S) per value channel, into red rows 0-1
            float part[2] = {0.f, 0.f};
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                for (int e = 0; e < 4; e += 2) {
                    const float2 s2 = ld_pair(sm, OFF_SH, OFF_SL, 256, f.row(e), f.col128(nt));
                    part[e >> 1] = fmaf(Dm[nt][e], s2.x, fmaf(Dm[nt][e + 1], s2.y, part[e >> 1]));
                }
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                float s = part[q];
                s += __shfl_xor_sync(0xffffffffu, s, 1);
                s += __shfl_xor_sync(0xffffffffu, s, 2);
                if (f.t == 0) red[(w >> 2) * 64 + f.m0 + f.g + 8 * q] = s;
            }
        }
        __syncthreads();
        // E with the state term on the chunk's last token, into G; dbeta out
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int e = 0; e < 4; e += 2) {
                const int r = f.row(e), i = f.col64(nt);
                float a0 = E[nt][e], a1 = E[nt][e + 1];
                if (r == C - 1) {
                    a0 += ecol[i] + red[i] + red[64 + i];
                    a1 += ecol[i + 1] + red[i + 1] + red[64 + i + 1];
                }
                *reinterpret_cast<float2*>(G + gidx(r, i)) = make_float2(a0, a1);
            }
        if (tid < nvalid)
            p.db_part[(part_base + tok0 + tid) * p.H + h] = dbr[tid] + red[384 + tid] + red[448 + tid];
        // D <- dS^ + dP^T Q - dY^T K
        mma_tile<8, 4, true, true, true, false>(Dm, opP, opQ, f.m0, f.n128);
        mma_tile<8, 4, true, true, true, false>(Dm, opX, opK, f.m0, f.n128);
        __syncthreads();
        {   // dalpha = reverse cumulative sum of E over tokens / alpha; four threads per
            // value channel, 16 tokens each, sums scanned across them
            const int i = tid >> 2, part = tid & 3;
            float e[16], a[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int r = 16 * part + j;
                e[j] = G[gidx(r, i)];
                a[j] = r < nvalid ? p.alpha[vidx(tok0 + r, i)] : 1.f;
            }
#pragma unroll
            for (int j = 14; j >= 0; --j) e[j] += e[j + 1];
            float s = e[0], y;
            y = __shfl_down_sync(0xffffffffu, s, 1);
            if (part <= 2) s += y;
            y = __shfl_down_sync(0xffffffffu, s, 2);
            if (part <= 1) s += y;
            float after = __shfl_down_sync(0xffffffffu, s, 1);
            if (part == 3) after = 0.f;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int r = 16 * part + j;
                if (r < nvalid) p.dalpha[vidx(tok0 + r, i)] = (e[j] + after) / a[j];
            }
        }
        __syncthreads();
    }
    if (p.dS0) {
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; e += 2)
                *reinterpret_cast<float2*>(p.dS0 + head_state + f.row(e) * DK + f.col128(nt)) =
                    make_float2(Dm[nt][e], Dm[nt][e + 1]);
    }
}

__global__ void kda_backward_reduce(const BwdParams p, float* __restrict__ dq,
                                    float* __restrict__ dk, float* __restrict__ dbeta) {
    if (*p.status == KDA_ERR_DEVICE_INPUT) return;
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

// The gate of one (token, head) per value channel: the head's scalar gate, or
// exp of the bf16 log gate.  Tokens past cu_seqlens[N] are left alone.
__global__ void gate_expand_kernel(const void* gate_in, int gate, const int32_t* __restrict__ cu,
                                   int N, int H, int d_v, float* __restrict__ ax,
                                   const int32_t* __restrict__ status) {
    if (*status == KDA_ERR_DEVICE_INPUT) return;
    const int64_t n = (int64_t)cu[N] * H * d_v;
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < n;
         e += (int64_t)gridDim.x * blockDim.x) {
        if (gate == KDA_GATE_HEAD_F32)
            ax[e] = static_cast<const float*>(gate_in)[e / d_v];
        else
            ax[e] = __expf(__bfloat162float(static_cast<const __nv_bfloat16*>(gate_in)[e]));
    }
}

// The gradient with respect to the gate in its own layout (chain rule through
// the expansion): the sum over the head's channels for a scalar gate (one warp
// per token and head, fixed reduction order), alpha * dL/dalpha for log alpha.
__global__ void gate_grad_kernel(int gate, const int32_t* __restrict__ cu, int N, int H, int d_v,
                                 const float* __restrict__ ax, const float* __restrict__ dax,
                                 float* __restrict__ dgate, const int32_t* __restrict__ status) {
    if (*status == KDA_ERR_DEVICE_INPUT) return;
    const int64_t th_n = (int64_t)cu[N] * H;
    if (gate == KDA_GATE_HEAD_F32) {
        const int lane = threadIdx.x & 31;
        const int64_t w0 = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
        const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
        for (int64_t th = w0; th < th_n; th += nw) {
            float s = 0.f;
            for (int i = lane; i < d_v; i += 32) s += dax[th * d_v + i];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
            if (lane == 0) dgate[th] = s;
        }
    } else {
        const int64_t n = th_n * d_v;
        for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < n;
             e += (int64_t)gridDim.x * blockDim.x)
            dgate[e] = ax[e] * dax[e];
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
    L.tc = d_v > 0 && d_v % 128 == 0 && d_v <= 1024;
    L.ckpt = take(slots * H * (size_t)d_v * DK * sizeof(float));
    if (L.tc) {
        L.o_tc = take(T * H * (size_t)d_v * 2);
        L.st_tc = take(N * H * (size_t)d_v * DK * sizeof(float));
    } else {
        L.tbuf = take(slots * H * nrb * (size_t)PAIR);
    }
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
    p.tbuf = reinterpret_cast<uint4*>(ws + L.tbuf);
    p.tc_ckpt = 0;
    cudaError_t err;
    if (L.tc) {   // the tensor-core forward writes the chunk-start states
        PrefillArgs f = {};
        f.q = a.q; f.k = a.k; f.v = a.v; f.alpha = a.alpha; f.beta = a.beta; f.S0 = a.S0;
        f.cu_seqlens = a.cu_seqlens; f.num_seqs = a.num_seqs; f.total_tokens = a.total_tokens;
        f.H = a.H; f.d_k = DK; f.d_v = a.d_v; f.dtype = KDA_BF16; f.chunk = C;
        f.o = ws + L.o_tc;
        f.S_T = reinterpret_cast<float*>(ws + L.st_tc);
        f.status = reinterpret_cast<int32_t*>(ws + WorkspaceLayout::kStatus);
        f.counter = reinterpret_cast<int32_t*>(ws + WorkspaceLayout::kCounter);
        f.order = reinterpret_cast<int32_t*>(ws + WorkspaceLayout::kOrder);
        f.gate = KDA_GATE_CHANNEL_F32;
        if ((err = launch_prefill_tc_ckpt(f, p.ckpt, stream)) != cudaSuccess) return err;
        p.tc_ckpt = 1;
    }
    p.dq_part = reinterpret_cast<float*>(ws + L.dq_part);
    p.dk_part = reinterpret_cast<float*>(ws + L.dk_part);
    p.db_part = reinterpret_cast<float*>(ws + L.db_part);
    p.dv = a.dv; p.dalpha = a.dalpha; p.dS0 = a.dS0;
    err = cudaFuncSetAttribute(kda_backward_kernel,
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

namespace kda {

cudaError_t launch_gate_expand(const void* gate_in, kda_gate_format gate, const BackwardArgs& a,
                               float* ax, const int32_t* status, cudaStream_t stream) {
    const int blocks = 4 * (sm_count() > 0 ? sm_count() : 1);
    gate_expand_kernel<<<blocks, 256, 0, stream>>>(gate_in, (int)gate, a.cu_seqlens, a.num_seqs,
                                                   a.H, a.d_v, ax, status);
    return cudaGetLastError();
}

cudaError_t launch_gate_grad(kda_gate_format gate, const BackwardArgs& a, const float* ax,
                             const float* dax, float* dgate, const int32_t* status,
                             cudaStream_t stream) {
    const int blocks = 4 * (sm_count() > 0 ? sm_count() : 1);
    gate_grad_kernel<<<blocks, 256, 0, stream>>>((int)gate, a.cu_seqlens, a.num_seqs, a.H, a.d_v,
                                                 ax, dax, dgate, status);
    return cudaGetLastError();
}

}  // namespace kda
