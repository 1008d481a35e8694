// Tensor-core chunkwise KDA prefill for GB300: tcgen05 MMAs with fp32
// accumulators in TMEM, operands staged by TMA, persistent CTAs.
//
// Chunk form of the recurrence ("Kimi (AI)", section "Kimi Delta Attention
// (KDA)"; chunk-wise parallelism as in the Kimi K3 architecture walkthrough):
// per chunk of C = 64 tokens, gamma_t = prod_{j<=t} alpha_j per value channel,
//
//   T  = (I + diag(beta) strict_lower(K K^T))^{-1}          (64 x 64, shared by all rows)
//   X  = diag(beta) (V / Gamma - K S^T)
//   U  = T X
//   O  = Gamma * (Q S^T + tril_incl(Q K^T) U)
//   S <- diag(gamma_C) (S + U^T K)
//
// Everything is computed value-channel-major (the M = 128 dimension of every
// MMA is a block of 128 rows of S), so each MMA result lands with one value
// channel per TMEM lane:
//   SK   = S K^T            M128 N64  K128   (A = S from TMEM, B = K tile); then S Q^T
//   KQK  = [K;Q] K^T        M128 N64  K128   (rows 0-63: K K^T, rows 64-127: Q K^T)
//   U^T  = X^T T^T          M128 N64  K64    (A = X^T from TMEM, B = T)
//   O^T += U^T P^T          M128 N64  K64    (accumulates onto the Q S^T half of SKQ)
//   S   += U^T K            M128 N128 K64    (B = the K tile read MN-major)
// Operands that are not exact bf16 inputs (S, X, U, T, P) are split into
// bf16 hi + lo parts, giving ~16 significant bits: products with exact bf16
// data take two MMAs, products of two split operands three (hi*hi, hi*lo,
// lo*hi).  Plain bf16 rounding of these intermediates would cost ~1e-3
// relative error on its own.
//
// Roles (448 threads, one CTA per SM, items (sequence, head, 128-channel
// block) assigned round-robin in the planner's longest-first order):
//   warp 0      TMA producer: K, Q (128B-swizzled) and alpha, V tiles, beta
//   warp 1      MMA issuer (one thread)
//   warps 2-5   token group: T by blocked (16 x 16) inversion, P = tril_incl(Q K^T)
//   warps 6-13  row group: two threads per value channel (one per half of the
//               chunk's tokens / of the key channels): Gamma, X, U staging,
//               state decay and hi/lo staging of S, then the output
// Every wait is bounded; on a timeout the CTA records KDA_ERR_DEVICE_TIMEOUT,
// stops issuing work, drains what it issued, frees TMEM and exits.
#include "kda_internal.h"
#include "kda_tc.cuh"

#include <cudaTypedefs.h>

#include <mutex>

namespace kda {
namespace {

using namespace tc;

constexpr int C = 64;        // tokens per chunk
constexpr int DK = 128;      // key channels
constexpr int DVB = 128;     // value channels per work item
constexpr int kThreads = 448;
// Limit of every device-side wait of a prefill launch (wall time)
constexpr uint64_t kTimeoutNs = 2000000000ull;

// TMEM columns (512 allocated)
constexpr uint32_t TM_S = 0;       // S, fp32, 128 columns
constexpr uint32_t TM_SKQ = 128;   // S K^T | S Q^T (+ U P^T), then U^T in the first half
constexpr uint32_t TM_KQK = 256;   // [K;Q] K^T, 64 columns
constexpr uint32_t TM_SHI = 320;   // S hi, bf16 pairs, 64 columns
constexpr uint32_t TM_SLO = 384;   // S lo
constexpr uint32_t TM_XHI = 448;   // X^T then U^T hi, 32 columns
constexpr uint32_t TM_XLO = 480;   // X^T then U^T lo
constexpr uint32_t TM_COLS = 512;

// Shared memory (offsets from a 1024-byte aligned base)
constexpr uint32_t SM_KQ = 0;            // 2 stages: [k-block 2][128 rows: 64 K, 64 Q][128 B]
constexpr uint32_t KQ_STAGE = 32768;
constexpr uint32_t KQ_KBLOCK = 16384;
constexpr uint32_t SM_ALPHA = 65536;     // [64 tokens][128 channels] fp32
constexpr uint32_t SM_V = 98304;         // [64][128] bf16, V buffer 0 (buffer 1 at SM_V1)
constexpr uint32_t SM_T = 114688;        // 2 buffers x (hi, lo) x [64][64] bf16, swizzled
constexpr uint32_t SM_P = 147456;        // same for P
constexpr uint32_t TP_BUF = 16384;
constexpr uint32_t TP_LO = 8192;
constexpr uint32_t SM_BETA = 180224;     // 2 stages x 64 fp32
constexpr uint32_t SM_L = 180736;        // [64][LSTR] fp32: diag(beta) strict_lower(K K^T), then T in place
constexpr uint32_t LSTR = 68;
constexpr uint32_t SM_V1 = 198144;       // V buffer 1
constexpr uint32_t SM_Y = 214528;        // [4 warps][16][YSTR] fp32 scratch of the blocked inverse
constexpr uint32_t YSTR = 24;
constexpr uint32_t SM_BAR = 220672;
constexpr uint32_t SM_MISC = SM_BAR + 256;
constexpr uint32_t SM_HALF = SM_MISC + 64;   // [2][128] fp32: per-half products of alpha
constexpr uint32_t SM_OST = SM_HALF + 1024;   // [8 row warps][16 tokens][32 channels] bf16
constexpr uint32_t SMEM_BYTES = SM_OST + 8 * 1024 + 1024;

// mbarrier indices
enum {
    B_KQ_FULL = 0,     // [2] producer -> K/Q/beta stage loaded
    B_KQ_EMPTY = 2,    // [2] MMA commit -> stage free
    B_A_FULL = 4,      // producer -> alpha loaded
    B_A_EMPTY = 5,     // row group (8 warps) -> alpha read
    B_KQK_DONE = 6,    // MMA commit -> [K;Q]K^T ready
    B_KQK_FREE = 7,    // token group (4 warps) -> KQK read
    B_TP_READY = 8,    // [2] token group (4 warps) -> T, P written
    B_TP_FREE = 10,    // [2] MMA commit -> T, P buffer consumed
    B_S_READY = 12,    // row group (8 warps) -> S and S hi/lo staged
    B_SKQ_DONE = 13,   // MMA commit
    B_X_READY = 14,    // row group (8 warps)
    B_U_DONE = 15,     // MMA commit
    B_U_READY = 16,    // row group (8 warps)
    B_S_DONE = 17,     // MMA commit: S += U^T K complete
    B_O_DONE = 18,     // MMA commit: O^T += U^T P^T complete
    B_O_READ = 19,     // row group (8 warps) -> O read out of TMEM (its columns are free)
    B_PAIR = 20,       // [4] the two row warps of a TMEM lane quarter swap half-chunk products
    B_V_FULL = 24,     // [2] producer -> V buffer loaded
    B_V_EMPTY = 26,    // [2] row group (8 warps) -> V buffer read
    B_COUNT = 28
};

struct TcParams {
    CUtensorMap tm_q, tm_k, tm_v, tm_a;
    const float* beta;
    const float* S0;
    float* S_T;
    __nv_bfloat16* o;
    const int32_t* cu;
    const int32_t* order;
    int32_t* status;
    int32_t H, d_v, nvb, num_items;
    // Sequence-axis split (null vt0: plain launch).  Items then run over virtual
    // sequences v = n_base + rank with token ranges [vt0[v], vt0[v] + vlen[v]);
    // S0 is read for v in [s0_lo, s0_hi) (row v - s0_lo, zero elsewhere) and the
    // final state written for v in [st_lo, st_hi) (row v - st_lo); g_out[v]
    // receives prod alpha over the item per channel.  CTAs from a_ctas on run
    // transition items instead: v = n_base_p + rank, alpha = 1, v = 0, S0 = I,
    // one 128-row block, final state to P_out[v - n_base_p], no output.
    const int64_t* vt0;
    const int32_t* vlen;
    int32_t n_base, n_base_p, s0_lo, s0_hi, st_lo, st_hi, a_ctas, num_items_p;
    float* g_out;
    float* P_out;
    // channels whose chunks decayed too fast for the one-pass chunk form, one
    // bit per channel of [N][H][d_v / 128] blocks (null: reported instead)
    uint32_t* redo;
    // Split launches: plain items of virtual sequences v >= gstart_lo write,
    // for each chunk, prod alpha from the segment's start to the chunk's start
    // per channel, to gstart [slot][H][d_v] with slot = cu[n] / C + n + (the
    // chunk's index within sequence n = v % gstart_lo); transition items write
    // their outputs P_{<=t} q_t in fp32 to qtil [T][H][DK] (null: none).
    // Plain items of v >= gstart_lo also keep their o in fp32 in ores
    // [T][H][d_v] for the chunks whose decay from the segment start is at
    // least kOresFloor, for the correction that adds the initial state's
    // share (elsewhere that share is small beside the bf16 rounding).
    float* gstart;
    float* qtil;
    float* ores;
    // transition items also add each chunk's sum of squares of P_{<=t} q_t
    // (over its tokens and rows) to qfro [slot][H], zeroed beforehand
    float* qfro;
    int32_t gstart_lo;
    const float* alpha_s;   // GATE_SCALAR: alpha [T][H]
    // GATE_F32_CKPT: fp32 [slots][H][d_v][DK]; chunk c of sequence n starting
    // at token t0 in slot t0 / C + n + c
    float* ckpt;
};

struct ItemInfo {
    int n, h, vb, len, nc;
    int64_t t0;
};

// Gate formats (the GATE template parameter): per value channel fp32 alpha
// [T][H][d_v]; one fp32 gate per (token, head) [T][H] (Gated DeltaNet's
// scalar gate, broadcast over the value channels); per value channel log alpha
// in bf16 [T][H][d_v] (half the bytes of the largest prefill input).
// GATE_F32_CKPT: the fp32 gate, and every chunk's start state is written to
// TcParams::ckpt for the backward pass.  GATE_F32_ADD: the fp32 gate with the
// additive update of linear attention (no prediction): beta is taken as zero
// in L, so T = I, and X = beta V / Gamma without the S K^T term; the MMA
// schedule is unchanged.
enum { GATE_F32 = 0, GATE_SCALAR = 1, GATE_LOG_BF16 = 2, GATE_F32_CKPT = 3, GATE_F32_ADD = 4 };

// SPLIT: the kernel serves the split launches (virtual sequences, transition
// items); the plain instantiation compiles none of that.
template <bool SPLIT>
__device__ __forceinline__ ItemInfo item_info(const TcParams& p, int item, bool pk) {
    ItemInfo it;
    const int nvb = pk ? 1 : p.nvb;
    const int per_rank = p.H * nvb;
    const int rank = item / per_rank, rem = item % per_rank;
    it.h = rem / nvb;
    it.vb = rem % nvb;
    if (SPLIT) {
        it.n = (pk ? p.n_base_p : p.n_base) + rank;
        it.t0 = p.vt0[it.n];
        it.len = p.vlen[it.n];
    } else {
        it.n = p.order[rank];
        it.t0 = p.cu[it.n];
        it.len = p.cu[it.n + 1] - p.cu[it.n];
    }
    it.nc = (it.len + C - 1) / C;
    return it;
}

// This CTA's share of the items: its kind (plain / transition), first item,
// stride and item count.
template <bool SPLIT>
struct ItemRange {
    bool pk;
    int first, stride, count;
    __device__ explicit ItemRange(const TcParams& p) {
        pk = SPLIT && (int)blockIdx.x >= p.a_ctas;
        first = pk ? (int)blockIdx.x - p.a_ctas : (int)blockIdx.x;
        stride = pk ? (int)gridDim.x - p.a_ctas : p.a_ctas;
        count = pk ? p.num_items_p : p.num_items;
    }
};

// Walks the chunks of this CTA's items in order, skipping empty items.
template <bool SPLIT>
struct ChunkCursor {
    int item, c;
    bool valid;
    ItemInfo info;
    ItemRange<SPLIT> rg;
    __device__ explicit ChunkCursor(const TcParams& p) : rg(p) {}
    __device__ void init(const TcParams& p) {
        item = rg.first;
        c = 0;
        seek(p);
    }
    __device__ void seek(const TcParams& p) {
        valid = false;
        while (item < rg.count) {
            info = item_info<SPLIT>(p, item, rg.pk);
            if (info.nc > 0) {
                valid = true;
                return;
            }
            item += rg.stride;
        }
    }
    __device__ void next(const TcParams& p) {
        if (++c >= info.nc) {
            c = 0;
            item += rg.stride;
            seek(p);
        }
    }
};

struct Ctx {
    uint8_t* smem;
    uint64_t* bars;
    volatile int* abort;
    volatile int* slots;   // [2] broadcast slots of the token group
    volatile int* never;   // always 0: lets drain waits ignore the abort flag
    uint32_t tmem;
    int32_t* status;
    uint64_t timeout_ns;   // limit of every wait
};

__device__ __forceinline__ void fail(const Ctx& cx) {
    *cx.abort = 1;
    atomicExch(cx.status, (int32_t)KDA_ERR_DEVICE_TIMEOUT);
}

__device__ __forceinline__ bool wait1(const Ctx& cx, int b, uint32_t parity) {
    if (mbar_wait(&cx.bars[b], parity, cx.abort, cx.timeout_ns)) return true;
    fail(cx);
    return false;
}

// Every lane of the calling warp waits; the warp goes on only if all lanes
// saw the phase complete, so its control flow stays uniform.
__device__ __forceinline__ bool warp_wait(const Ctx& cx, int b, uint32_t parity) {
    const bool ok = mbar_wait(&cx.bars[b], parity, cx.abort, cx.timeout_ns);
    if (__all_sync(0xffffffffu, ok)) return true;
    fail(cx);
    return false;
}

// One thread of a thread group waits; the outcome is shared through a
// named barrier, so the whole group continues or stops together.  Each
// thread then takes its own acquire on the (already completed) phase.
struct Group {
    int tid, bar_id, nthreads, flip;
    volatile int* slot;
    __device__ bool wait(const Ctx& cx, int b, uint32_t parity) {
        volatile int* s = slot + flip;
        flip ^= 1;
        if (tid == 0) *s = wait1(cx, b, parity) ? 1 : 0;
        __syncwarp();   // bar.sync is warp-aligned: reconverge after the elected wait
        named_bar_sync(bar_id, nthreads);
        if (*s == 0) return false;
        if (!mbar_wait(&cx.bars[b], parity, cx.abort, cx.timeout_ns)) {
            fail(cx);
            return false;
        }
        return true;
    }
};

__device__ __forceinline__ float bf2f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

__device__ __forceinline__ uint32_t kq_addr(const Ctx& cx, int s) {
    return smem_u32(cx.smem + SM_KQ + s * KQ_STAGE);
}

// ------------------------------------------------------------------ producer
template <bool SPLIT, int GATE>
__device__ void run_producer(const TcParams& p, const Ctx& cx, int lane) {
    ChunkCursor<SPLIT> cur(p);
    cur.init(p);
    const bool pk = cur.rg.pk;
    uint32_t g = 0;
    uint32_t kq_issued[2] = {0, 0}, a_issued = 0, v_issued[2] = {0, 0};
    const float* beta_st = reinterpret_cast<const float*>(cx.smem + SM_BETA);
    while (cur.valid) {
        const int s = g & 1;
        const int64_t tok0 = cur.info.t0 + (int64_t)cur.c * C;
        const int nvalid = min(C, cur.info.len - cur.c * C);
        const int h = cur.info.h;
        if (g >= 2) {
            int r = 1;
            if (lane == 0) r = wait1(cx, B_KQ_EMPTY + s, ((g >> 1) + 1) & 1);
            __syncwarp();
            if (!__shfl_sync(0xffffffffu, r, 0)) break;
        }
        float* bst = const_cast<float*>(beta_st) + s * C;
        for (int j = lane; j < C; j += 32)
            bst[j] = j < nvalid ? p.beta[(tok0 + j) * p.H + h] : 0.f;
        if (GATE == GATE_SCALAR) {   // one gate per token rides with beta
            float* ast = reinterpret_cast<float*>(cx.smem + SM_ALPHA) + s * C;
            for (int j = lane; j < C; j += 32)
                ast[j] = j < nvalid ? p.alpha_s[(tok0 + j) * p.H + h] : 1.f;
        }
        __syncwarp();
        if (lane == 0) {
            uint64_t* bar = &cx.bars[B_KQ_FULL + s];
            uint8_t* st = cx.smem + SM_KQ + s * KQ_STAGE;
            mbar_arrive_expect_tx(bar, KQ_STAGE);
            tma_load_3d(st, &p.tm_k, bar, 0, h, (int32_t)tok0);
            tma_load_3d(st + KQ_KBLOCK, &p.tm_k, bar, 64, h, (int32_t)tok0);
            tma_load_3d(st + 8192, &p.tm_q, bar, 0, h, (int32_t)tok0);
            tma_load_3d(st + KQ_KBLOCK + 8192, &p.tm_q, bar, 64, h, (int32_t)tok0);
        }
        ++kq_issued[s];
        if (pk) {   // transition items: alpha = 1 and v = 0, nothing to load
            ++g;
            cur.next(p);
            continue;
        }
        // alpha: one buffer, free once the row group has read it into registers
        if (GATE != GATE_SCALAR) {
            if (g >= 1) {
                int r = 1;
                if (lane == 0) r = wait1(cx, B_A_EMPTY, (g - 1) & 1);
                __syncwarp();
                if (!__shfl_sync(0xffffffffu, r, 0)) break;
            }
            if (lane == 0) {
                uint64_t* bar = &cx.bars[B_A_FULL];
                mbar_arrive_expect_tx(bar, 64 * DVB * (GATE == GATE_LOG_BF16 ? 2 : 4));
                tma_load_3d(cx.smem + SM_ALPHA, &p.tm_a, bar, cur.info.vb * DVB, h, (int32_t)tok0);
            }
            ++a_issued;
        }
        // V: two buffers
        if (g >= 2) {
            int r = 1;
            if (lane == 0) r = wait1(cx, B_V_EMPTY + s, ((g >> 1) + 1) & 1);
            __syncwarp();
            if (!__shfl_sync(0xffffffffu, r, 0)) break;
        }
        if (lane == 0) {
            uint64_t* bar = &cx.bars[B_V_FULL + s];
            mbar_arrive_expect_tx(bar, 64 * DVB * 2);
            tma_load_3d(cx.smem + (s ? SM_V1 : SM_V), &p.tm_v, bar, cur.info.vb * DVB, h,
                        (int32_t)tok0);
        }
        ++v_issued[s];
        ++g;
        cur.next(p);
    }
    // drain: every issued copy must have landed before the CTA may exit
    if (lane == 0) {
        for (int s = 0; s < 2; ++s)
            if (kq_issued[s]) mbar_wait(&cx.bars[B_KQ_FULL + s], (kq_issued[s] - 1) & 1, cx.never, cx.timeout_ns);
        if (a_issued) mbar_wait(&cx.bars[B_A_FULL], (a_issued - 1) & 1, cx.never, cx.timeout_ns);
        for (int s = 0; s < 2; ++s)
            if (v_issued[s]) mbar_wait(&cx.bars[B_V_FULL + s], (v_issued[s] - 1) & 1, cx.never, cx.timeout_ns);
    }
    __syncwarp();
}

// ------------------------------------------------------------------ MMA issuer
__device__ bool issue_kqk(const TcParams& p, const Ctx& cx, uint32_t g) {
    const int s = g & 1;
    if (!warp_wait(cx, B_KQ_FULL + s, (g >> 1) & 1)) return false;
    if (g >= 1 && !warp_wait(cx, B_KQK_FREE, (g - 1) & 1)) return false;
    tc_fence_after();
    if (elect_one()) {
        const uint32_t base = kq_addr(cx, s);
        // A = 128 rows [K;Q], B = its first 64 rows; one 128-byte k-block per group
#pragma unroll 1
        for (int kb = 0; kb < 2; ++kb)
            mma_ss4_same(cx.tmem + TM_KQK, smem_desc_sw128(base + kb * KQ_KBLOCK, 0, 1024), 2,
                         idesc_bf16_f32(128, 64, 0, 0), kb != 0);
        mma_commit(&cx.bars[B_KQK_DONE]);
    }
    __syncwarp();
    return true;
}

// True when [K;Q]K^T of chunk g could be issued without waiting (warp-uniform).
__device__ __forceinline__ bool kqk_ready(const Ctx& cx, uint32_t g) {
    bool r = mbar_test_wait(&cx.bars[B_KQ_FULL + (g & 1)], (g >> 1) & 1);
    if (g >= 1) r = r && mbar_test_wait(&cx.bars[B_KQK_FREE], (g - 1) & 1);
    return __all_sync(0xffffffffu, r);
}

// The whole warp runs the schedule and waits; one elected lane issues each
// group of MMAs together with the commit that tracks it.
template <bool SPLIT>
__device__ void run_mma(const TcParams& p, const Ctx& cx) {
    ChunkCursor<SPLIT> cur(p), ahead(p);
    cur.init(p);
    ahead = cur;
    uint32_t g = 0;
    int last_commit_bar = -1;
    uint32_t last_commit_parity = 0;
    const uint32_t tm = cx.tmem;
    const uint32_t id_n64 = idesc_bf16_f32(128, 64, 0, 0);
    const uint32_t id_n128_bmn = idesc_bf16_f32(128, 128, 0, 1);
    bool ok = true;
    if (cur.valid) {
        ok = issue_kqk(p, cx, 0);
        last_commit_bar = B_KQK_DONE;
        last_commit_parity = 0;
        ahead.next(p);
    }
    while (cur.valid && ok) {
        const int s = g & 1;
        const uint32_t kq = kq_addr(cx, s);
        // S K^T = S_hi K^T + S_lo K^T first (it feeds the next step of the chain),
        // then S Q^T (needed only for the output)
        if (!(ok = warp_wait(cx, B_S_READY, g & 1))) break;
        tc_fence_after();
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            if (elect_one()) {
                // groups: (S_hi, k-block 0), (S_hi, 1), (S_lo, 0), (S_lo, 1)
#pragma unroll 1
                for (int i = 0; i < 4; ++i) {
                    const uint32_t a0 = tm + ((i >> 1) == 0 ? TM_SHI : TM_SLO) + 32 * (i & 1);
                    const uint64_t b =
                        smem_desc_sw128(kq + (i & 1) * KQ_KBLOCK + half * 8192, 0, 1024);
                    mma_ts4(tm + TM_SKQ + 64 * half, a0, 8, b, 2, id_n64, i != 0);
                }
                if (half == 0) mma_commit(&cx.bars[B_SKQ_DONE]);
            }
            __syncwarp();
            if (half == 0) {
                last_commit_bar = B_SKQ_DONE;
                last_commit_parity = g & 1;
                // S Q^T reuses the columns the previous chunk's O was read from
                if (g >= 1 && !(ok = warp_wait(cx, B_O_READ, (g - 1) & 1))) break;
            }
        }
        if (!ok) break;
        // next chunk's [K;Q]K^T, so the token group can build its T and P early;
        // issued here only if its tiles are in, else after the U or the S MMAs,
        // so that it never holds up this chunk's chain
        bool kqk_due = ahead.valid;
        if (kqk_due && kqk_ready(cx, g + 1)) {
            if (!(ok = issue_kqk(p, cx, g + 1))) break;
            last_commit_bar = B_KQK_DONE;
            last_commit_parity = (g + 1) & 1;
            ahead.next(p);
            kqk_due = false;
        }
        // U^T = X^T T^T   (hi*hi + hi*lo + lo*hi)
        if (!(ok = warp_wait(cx, B_X_READY, g & 1))) break;
        if (!(ok = warp_wait(cx, B_TP_READY + s, (g >> 1) & 1))) break;
        tc_fence_after();
        if (elect_one()) {
            const uint32_t t_hi = smem_u32(cx.smem + SM_T + s * TP_BUF);
#pragma unroll 1
            for (int part = 0; part < 3; ++part)
                mma_ts4(tm + TM_SKQ, tm + (part == 2 ? TM_XLO : TM_XHI), 8,
                        smem_desc_sw128(t_hi + (part == 1 ? TP_LO : 0), 0, 1024), 2, id_n64,
                        part != 0);
            mma_commit(&cx.bars[B_U_DONE]);
        }
        __syncwarp();
        last_commit_bar = B_U_DONE;
        last_commit_parity = g & 1;
        if (kqk_due && kqk_ready(cx, g + 1)) {
            if (!(ok = issue_kqk(p, cx, g + 1))) break;
            last_commit_bar = B_KQK_DONE;
            last_commit_parity = (g + 1) & 1;
            ahead.next(p);
            kqk_due = false;
        }
        // S += U^T K first (the chain), then O^T += U^T P^T
        if (!(ok = warp_wait(cx, B_U_READY, g & 1))) break;
        tc_fence_after();
        if (elect_one()) {
            // B = the K tile read MN-major: 16 tokens (2048 bytes) per k-step
#pragma unroll 1
            for (int part = 0; part < 2; ++part)
                mma_ts4(tm + TM_S, tm + (part == 0 ? TM_XHI : TM_XLO), 8,
                        smem_desc_sw128(kq, KQ_KBLOCK, 1024), 2048 >> 4, id_n128_bmn, 1);
            mma_commit(&cx.bars[B_S_DONE]);
            mma_commit(&cx.bars[B_KQ_EMPTY + s]);   // the O MMAs do not read K or Q
            const uint32_t p_hi = smem_u32(cx.smem + SM_P + s * TP_BUF);
#pragma unroll 1
            for (int part = 0; part < 3; ++part)
                mma_ts4(tm + TM_SKQ + 64, tm + (part == 2 ? TM_XLO : TM_XHI), 8,
                        smem_desc_sw128(p_hi + (part == 1 ? TP_LO : 0), 0, 1024), 2, id_n64, 1);
            mma_commit(&cx.bars[B_O_DONE]);
            mma_commit(&cx.bars[B_TP_FREE + s]);
        }
        __syncwarp();
        last_commit_bar = B_O_DONE;
        last_commit_parity = g & 1;
        if (kqk_due) {
            if (!(ok = issue_kqk(p, cx, g + 1))) break;
            last_commit_bar = B_KQK_DONE;
            last_commit_parity = (g + 1) & 1;
            ahead.next(p);
        }
        ++g;
        cur.next(p);
    }
    // drain: the MMAs issued last must finish before TMEM is released
    if (last_commit_bar >= 0)
        mbar_wait(&cx.bars[last_commit_bar], last_commit_parity, cx.never, cx.timeout_ns);
    __syncwarp();
}

// ------------------------------------------------------------------ token group
// acc (16 x 16 as two 16 x 8 tiles) += A (16 x 16) * B (16 x 16), both fp32 in
// shared memory with row strides lda / ldb, on one warp (tf32 mma.sync).
__device__ __forceinline__ void warp_mm16(float (&acc)[2][4], const float* A, int lda,
                                          const float* B, int ldb, int lane) {
    const int g = lane >> 2, tq = lane & 3;
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
        uint32_t a[4];
        a[0] = f32_to_tf32(A[g * lda + 8 * ks + tq]);
        a[1] = f32_to_tf32(A[(g + 8) * lda + 8 * ks + tq]);
        a[2] = f32_to_tf32(A[g * lda + 8 * ks + tq + 4]);
        a[3] = f32_to_tf32(A[(g + 8) * lda + 8 * ks + tq + 4]);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            uint32_t b[2];
            b[0] = f32_to_tf32(B[(8 * ks + tq) * ldb + 8 * nt + g]);
            b[1] = f32_to_tf32(B[(8 * ks + tq + 4) * ldb + 8 * nt + g]);
            mma_sync_tf32(acc[nt], a, b);
        }
    }
}

__device__ __forceinline__ void warp_store16(float* Y, int ldy, const float (&acc)[2][4],
                                             float scale, int lane) {
    const int g = lane >> 2, tq = lane & 3;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        Y[g * ldy + 8 * nt + 2 * tq] = scale * acc[nt][0];
        Y[g * ldy + 8 * nt + 2 * tq + 1] = scale * acc[nt][1];
        Y[(g + 8) * ldy + 8 * nt + 2 * tq] = scale * acc[nt][2];
        Y[(g + 8) * ldy + 8 * nt + 2 * tq + 1] = scale * acc[nt][3];
    }
}

// Per chunk: L = diag(beta) strict_lower(K K^T) and P = tril_incl(Q K^T) from
// the KQK accumulator, then T = (I + L)^{-1} by blocks of 16: the four
// diagonal blocks D_b by forward substitution, the rest by recursive doubling
// of the block-triangular inverse, and finally T and P as bf16 hi/lo tiles.
template <bool SPLIT, int GATE>
__device__ void run_token_group(const TcParams& p, const Ctx& cx, int t, int warp, int lane) {
    Group grp{t, 1, 128, 0, cx.slots};
    const int quarter = warp & 3;
    const int kr = 32 * quarter + lane;   // accumulator row: 0-63 K K^T, 64-127 Q K^T
    const uint32_t lane_base = (uint32_t)(32 * quarter) << 16;
    float* Ls = reinterpret_cast<float*>(cx.smem + SM_L);
    float* Ys = reinterpret_cast<float*>(cx.smem + SM_Y);
    ChunkCursor<SPLIT> cur(p);
    cur.init(p);
    uint32_t g = 0;
    while (cur.valid) {
        const int s = g & 1;
        if (!grp.wait(cx, B_KQK_DONE, g & 1)) break;
        if (!grp.wait(cx, B_KQ_FULL + s, (g >> 1) & 1)) break;   // acquire for beta
        if (g >= 2 && !grp.wait(cx, B_TP_FREE + s, ((g >> 1) + 1) & 1)) break;
        tc_fence_after();
        const float* bst = reinterpret_cast<const float*>(cx.smem + SM_BETA) + s * C;
        uint8_t* t_hi = cx.smem + SM_T + s * TP_BUF;
        uint8_t* p_hi = cx.smem + SM_P + s * TP_BUF;
        const bool krow = kr < 64;           // warp-uniform
        const float bt = krow && GATE != GATE_F32_ADD ? bst[kr] : 0.f;
        const int tq = kr - 64;
#pragma unroll 1
        for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t v[16];
            tmem_ld16(cx.tmem + lane_base + TM_KQK + 16 * q4, v);
            tmem_ld_wait();
            if (krow) {
#pragma unroll
                for (int j = 0; j < 16; j += 4) {
                    const int col = 16 * q4 + j;
                    float4 l;
                    l.x = col + 0 < kr ? bt * __uint_as_float(v[j + 0]) : 0.f;
                    l.y = col + 1 < kr ? bt * __uint_as_float(v[j + 1]) : 0.f;
                    l.z = col + 2 < kr ? bt * __uint_as_float(v[j + 2]) : 0.f;
                    l.w = col + 3 < kr ? bt * __uint_as_float(v[j + 3]) : 0.f;
                    *reinterpret_cast<float4*>(Ls + kr * LSTR + col) = l;
                }
            } else {
#pragma unroll
                for (int h8 = 0; h8 < 2; ++h8) {
                    uint32_t hi[4], lo[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int col = 16 * q4 + 8 * h8 + 2 * e;
                        const float x0 = col <= tq ? __uint_as_float(v[8 * h8 + 2 * e]) : 0.f;
                        const float x1 = col + 1 <= tq ? __uint_as_float(v[8 * h8 + 2 * e + 1]) : 0.f;
                        split2_bf16(x0, x1, hi[e], lo[e]);
                    }
                    const uint32_t off = sw128_offset(tq, 16 * q4 + 8 * h8);
                    *reinterpret_cast<uint4*>(p_hi + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                    *reinterpret_cast<uint4*>(p_hi + TP_LO + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                }
            }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&cx.bars[B_KQK_FREE]);
        named_bar_sync(1, 128);   // L complete

        // T is built in place over L: the blocks of L above the diagonal are
        // already zero, and each block below it is read for the last time before
        // its block of T is written.
        // Diagonal blocks D_b = (I + L_bb)^{-1}: one thread per column, the column
        // held in registers until every column of the block is solved.
        {
            const int b = (t >> 4) & 3, cc = t & 15;
            float col[16];
            if (t < 64) {
                const float* Lb = Ls + (16 * b) * LSTR + 16 * b;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float x0 = i == cc ? 1.f : 0.f, x1 = 0.f;
#pragma unroll
                    for (int j = 0; j < i; ++j) {
                        if (j & 1) x1 = fmaf(-Lb[i * LSTR + j], col[j], x1);
                        else x0 = fmaf(-Lb[i * LSTR + j], col[j], x0);
                    }
                    col[i] = x0 + x1;
                }
            }
            named_bar_sync(1, 128);
            if (t < 64) {
#pragma unroll
                for (int i = 0; i < 16; ++i) Ls[(16 * b + i) * LSTR + 16 * b + cc] = col[i];
            }
            named_bar_sync(1, 128);
        }
        // blocks below the diagonal by recursive doubling, 16 x 16 products on
        // tf32 mma.sync (T(i,j) is block (i,j) of T, N(i,j) the same block of L
        // before it is overwritten):
        //   T(1,0) = -D_1 N(1,0) D_0,   T(3,2) = -D_3 N(3,2) D_2
        //   Y = N(2:4, 0:2) T(0:2, 0:2),  T(2:4, 0:2) = -T(2:4, 2:4) Y
        {
            const int w = t >> 5;
            auto Bk = [&](int i, int j) { return Ls + (16 * i) * LSTR + 16 * j; };
            auto Yb = [&](int k) { return Ys + k * (16 * YSTR); };
            if (w < 2) {
                const int i = 1 + 2 * w, j = i - 1;
                float acc[2][4] = {};
                warp_mm16(acc, Bk(i, j), LSTR, Bk(j, j), LSTR, lane);
                warp_store16(Yb(w), YSTR, acc, 1.f, lane);
                __syncwarp();
                float acc2[2][4] = {};
                warp_mm16(acc2, Bk(i, i), LSTR, Yb(w), YSTR, lane);
                warp_store16(Bk(i, j), LSTR, acc2, -1.f, lane);
            }
            named_bar_sync(1, 128);
            const int i = 2 + (w >> 1), j = w & 1;
            {
                float acc[2][4] = {};
                warp_mm16(acc, Bk(i, j), LSTR, Bk(j, j), LSTR, lane);
                if (j == 0) warp_mm16(acc, Bk(i, 1), LSTR, Bk(1, 0), LSTR, lane);
                warp_store16(Yb(w), YSTR, acc, 1.f, lane);
            }
            named_bar_sync(1, 128);
            {
                float acc[2][4] = {};
                if (i == 3) warp_mm16(acc, Bk(3, 2), LSTR, Yb(j), YSTR, lane);
                warp_mm16(acc, Bk(i, i), LSTR, Yb(w), YSTR, lane);
                warp_store16(Bk(i, j), LSTR, acc, -1.f, lane);
            }
            named_bar_sync(1, 128);
        }
        // T as bf16 hi/lo, 128B-swizzled B operand: thread t writes half of row t / 2
        {
            const int i = t >> 1, c0 = (t & 1) * 32;
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
                const float4 x0 = *reinterpret_cast<const float4*>(Ls + i * LSTR + c0 + 8 * ch);
                const float4 x1 = *reinterpret_cast<const float4*>(Ls + i * LSTR + c0 + 8 * ch + 4);
                uint32_t hi[4], lo[4];
                split2_bf16(x0.x, x0.y, hi[0], lo[0]);
                split2_bf16(x0.z, x0.w, hi[1], lo[1]);
                split2_bf16(x1.x, x1.y, hi[2], lo[2]);
                split2_bf16(x1.z, x1.w, hi[3], lo[3]);
                const uint32_t off = sw128_offset(i, c0 + 8 * ch);
                *reinterpret_cast<uint4*>(t_hi + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                *reinterpret_cast<uint4*>(t_hi + TP_LO + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&cx.bars[B_TP_READY + s]);
        ++g;
        cur.next(p);
    }
}

// ------------------------------------------------------------------ row group
// A chunk whose product of alpha over some channel falls below kDecayFloor is
// beyond the one-pass chunk form (it divides by the running product): that
// channel is handed back, in the workspace's bitmap, to the portable kernel,
// which runs it again from S0 (so its S_T is not written here).  Without a
// bitmap (the sequence-axis split), it is reported as KDA_ERR_DEVICE_RANGE.
// No register carries this across the chunk loop: the bit is set after the
// chunk's state is handed back, and read back (a global load of the bit this
// same thread set) before the item's final state is written.
// Split outputs, out of line so that the chunk loop's code stays small:
// 32 token rows of one channel in fp32, from TMEM (the transition items'
// P_{<=t} q_t) or from registers (a later segment's o from a zero start).
// The TMEM version also adds the warp's sum of squares of the stored values
// to *fro (one atomic per warp) when fro is not null.
__device__ __noinline__ void store_tmem_column_f32(uint32_t taddr, float* dst, int64_t stride,
                                                   int lim, float* fro) {
    float acc = 0.f;
#pragma unroll 1
    for (int q2 = 0; q2 < 2; ++q2) {
        uint32_t v[16];
        tmem_ld16(taddr + 16 * q2, v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j)
            if (16 * q2 + j < lim) {
                const float x = __uint_as_float(v[j]);
                dst[(16 * q2 + j) * stride] = x;
                acc = fmaf(x, x, acc);
            }
    }
    if (fro) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if ((threadIdx.x & 31) == 0) atomicAdd(fro, acc);
    }
}
struct Column32 {
    uint32_t v[32];
};
__device__ __noinline__ void store_column_f32(Column32 x, float* dst, int64_t stride, int lim) {
#pragma unroll 4
    for (int j = 0; j < 32; ++j)
        if (j < lim) dst[j * stride] = __uint_as_float(x.v[j]);
}

template <bool SPLIT>
__device__ __noinline__ void report_fast_decay(const TcParams& p, const ItemInfo& it, int r) {
    if (!SPLIT && p.redo)
        atomicOr(p.redo + (((size_t)it.n * p.H + it.h) * p.nvb + it.vb) * 4 + (r >> 5), 1u << (r & 31));
    else
        atomicCAS(p.status, 0, (int32_t)KDA_ERR_DEVICE_RANGE);
}
template <bool SPLIT>
__device__ __forceinline__ bool handed_back(const TcParams& p, const ItemInfo& it, int r) {
    if (SPLIT || !p.redo) return false;
    const volatile uint32_t* w = p.redo + (((size_t)it.n * p.H + it.h) * p.nvb + it.vb) * 4 + (r >> 5);
    return (*w >> (r & 31)) & 1u;
}

// Thread (r, h): value channel r of the item's block; h selects tokens
// 32h..32h+31 for X, U and O, and key channels 64h..64h+63 for S.
// 32 key channels (piece q of this thread's half): fp32 S and its bf16 hi/lo pairs
__device__ __forceinline__ void stage_state_piece(uint32_t lane_addr, int h, int q,
                                                  const float (&x)[32]) {
    uint32_t raw[32], hi[16], lo[16];
#pragma unroll
    for (int j = 0; j < 32; ++j) raw[j] = __float_as_uint(x[j]);
    tmem_st32(lane_addr + TM_S + 64 * h + 32 * q, raw);
#pragma unroll
    for (int j = 0; j < 16; ++j) split2_bf16(x[2 * j], x[2 * j + 1], hi[j], lo[j]);
    tmem_st16(lane_addr + TM_SHI + 32 * h + 16 * q, hi);
    tmem_st16(lane_addr + TM_SLO + 32 * h + 16 * q, lo);
}

template <bool SPLIT, int GATE>
__device__ void run_row_group(const TcParams& p, const Ctx& cx, int rt, int warp, int lane) {
    const int quarter = warp & 3;
    const int h = rt >> 7;                 // token half / key-channel half
    const int r = 32 * quarter + lane;     // value channel within the block = TMEM lane
    const uint32_t lane_addr = cx.tmem + ((uint32_t)(32 * quarter) << 16);
    uint32_t g = 0;
    bool ok = true;
    const float* al = reinterpret_cast<const float*>(cx.smem + SM_ALPHA);
    const ItemRange<SPLIT> rg(p);
    float* const st_base = rg.pk ? p.P_out : p.S_T;
    const int dvs = rg.pk ? DK : p.d_v;   // rows per head of the state layout
    for (int item = rg.first; item < rg.count && ok; item += rg.stride) {
        const ItemInfo it = item_info<SPLIT>(p, item, rg.pk);
        const int ch = it.vb * DVB + r;   // value channel
        // rows of the initial and final state of this item (-1: zero / not written)
        int s0_row = p.S0 ? it.n : -1, st_row = it.n;
        if (SPLIT) {
            s0_row = -1;
            st_row = it.n - p.n_base_p;
            if (!rg.pk) {
                if (p.S0 && it.n >= p.s0_lo && it.n < p.s0_hi) s0_row = it.n - p.s0_lo;
                st_row = it.n >= p.st_lo && it.n < p.st_hi ? it.n - p.st_lo : -1;
            }
        }
        const size_t s0off = (((size_t)s0_row * p.H + it.h) * dvs + ch) * DK + 64 * h;
        const size_t stoff = (((size_t)st_row * p.H + it.h) * dvs + ch) * DK + 64 * h;
        // initial state, 4 key channels from 64 h + j: S0, zero, or the identity
        auto init4 = [&](int j) {
            if (rg.pk) {
                const int c0 = 64 * h + j;
                return make_float4(c0 == ch ? 1.f : 0.f, c0 + 1 == ch ? 1.f : 0.f,
                                   c0 + 2 == ch ? 1.f : 0.f, c0 + 3 == ch ? 1.f : 0.f);
            }
            return s0_row >= 0 ? *reinterpret_cast<const float4*>(p.S0 + s0off + j)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
        };
        if (it.nc == 0) {
            if (st_row >= 0)
                for (int j = 0; j < 64; j += 4)
                    *reinterpret_cast<float4*>(st_base + stoff + j) = init4(j);
            if (SPLIT && p.g_out && !rg.pk && h == 0)
                p.g_out[((size_t)it.n * p.H + it.h) * p.d_v + ch] = 1.f;
            continue;
        }
        // GATE_F32_CKPT: this thread's 64 key channels of chunk c's start state
        auto ckpt_row = [&](int c) {
            return p.ckpt + (((size_t)(it.t0 / C + it.n + c) * p.H + it.h) * p.d_v + ch) * DK + 64 * h;
        };
#pragma unroll 1
        for (int q = 0; q < 2; ++q) {
            float x[32];
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
                const float4 v4 = init4(32 * q + j);
                x[j] = v4.x; x[j + 1] = v4.y; x[j + 2] = v4.z; x[j + 3] = v4.w;
            }
            if (GATE == GATE_F32_CKPT) {
#pragma unroll
                for (int j = 0; j < 32; j += 4)
                    *reinterpret_cast<float4*>(ckpt_row(0) + 32 * q + j) =
                        make_float4(x[j], x[j + 1], x[j + 2], x[j + 3]);
            }
            stage_state_piece(lane_addr, h, q, x);
        }
        float gtot = 1.f;   // prod alpha over the item, for g_out
        // where this item's per-chunk decay from the segment start goes (split only)
        float* gs_row = nullptr;
        float* qf_row = nullptr;   // transition items: the chunk sums of squares of their outputs
        if (SPLIT && p.gstart && (rg.pk || h == 0) && it.n >= p.gstart_lo) {
            const int n0 = it.n % p.gstart_lo;
            const int64_t c0 = p.cu[n0];
            const int64_t slot = c0 / C + n0 + (it.t0 - c0) / C;
            if (rg.pk)
                qf_row = p.qfro ? p.qfro + (size_t)slot * p.H + it.h : nullptr;
            else
                gs_row = p.gstart + ((size_t)slot * p.H + it.h) * p.d_v + ch;
        }

        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&cx.bars[B_S_READY]);

        for (int c = 0; c < it.nc; ++c, ++g) {
            const int64_t tok0 = it.t0 + (int64_t)c * C;
            const int nvalid = min(C, it.len - c * C);
            const bool last = c + 1 == it.nc;
            if (!(ok = warp_wait(cx, B_KQ_FULL + (g & 1), (g >> 1) & 1))) break;
            const float* bst = reinterpret_cast<const float*>(cx.smem + SM_BETA) + (g & 1) * C;
            // Gamma (padded tokens: alpha = 1): each thread takes the running
            // product over its half of the tokens, the halves swap their totals
            // through shared memory; then vg = beta V / Gamma for its tokens.
            // Transition items have alpha = 1 and v = 0.
            float gam[32], vg[32], gC = 1.f;
            if (rg.pk) {
#pragma unroll
                for (int j = 0; j < 32; ++j) vg[j] = 0.f;
            } else {
                float* half_tot = reinterpret_cast<float*>(cx.smem + SM_HALF);
                // The tiles always hold finite values (TMA fills rows past the tensor
                // with zeros; rows past the sequence belong to the next one), so the
                // loads are unconditional and padded tokens are masked afterwards.
                float a[32], inv[32];
                if (GATE == GATE_SCALAR) {
                    // one gate per token (padded tokens: 1), from the beta stage
                    const float* ast = reinterpret_cast<const float*>(cx.smem + SM_ALPHA) + (g & 1) * C;
#pragma unroll
                    for (int j = 0; j < 32; ++j) a[j] = ast[32 * h + j];
                } else {
                    if (!(ok = warp_wait(cx, B_A_FULL, g & 1))) break;
                    if (GATE == GATE_LOG_BF16) {   // alpha = exp(log alpha)
                        const uint16_t* la = reinterpret_cast<const uint16_t*>(al);
#pragma unroll
                        for (int j = 0; j < 32; ++j) a[j] = __expf(bf2f(la[(32 * h + j) * DVB + r]));
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j) a[j] = al[(32 * h + j) * DVB + r];
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&cx.bars[B_A_EMPTY]);   // alpha is in registers
                }
                {
                    float run = 1.f;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        a[j] = 32 * h + j < nvalid ? a[j] : 1.f;
                        run *= a[j];
                        gam[j] = run;
                    }
                    half_tot[h * DVB + r] = run;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&cx.bars[B_PAIR + quarter]);
                    if (!(ok = warp_wait(cx, B_PAIR + quarter, g & 1))) break;
                    const float other = half_tot[(1 - h) * DVB + r];
                    if (h == 1) {
#pragma unroll
                        for (int j = 0; j < 32; j += 2) {
                            const float2 gg = __fmul2_rn(make_float2(gam[j], gam[j + 1]),
                                                         make_float2(other, other));
                            gam[j] = gg.x;
                            gam[j + 1] = gg.y;
                        }
                    }
                    gC = h == 0 ? run * other : gam[31];
                    // the chunk form divides by the running product: a chunk whose
                    // product falls below kDecayFloor leaves this channel's result
                    // to the portable kernel (both threads of a channel agree)
                    // 1 / gamma_t from one reciprocal and the products of the later alphas
                    inv[31] = __frcp_rn(gam[31]);
#pragma unroll
                    for (int j = 30; j >= 0; --j) inv[j] = inv[j + 1] * a[j + 1];
                }
                if (!(ok = warp_wait(cx, B_V_FULL + (g & 1), (g >> 1) & 1))) break;
                const uint16_t* vs =
                    reinterpret_cast<const uint16_t*>(cx.smem + ((g & 1) ? SM_V1 : SM_V));
                const float4* b4 = reinterpret_cast<const float4*>(bst + 32 * h);
#pragma unroll
                for (int j4 = 0; j4 < 8; ++j4) {
                    const float4 bq = b4[j4];
                    const int j = 4 * j4, t = 32 * h + j;
                    float vq[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float q = bf2f(vs[(t + e) * DVB + r]) * inv[j + e];
                        vq[e] = t + e < nvalid ? q : 0.f;
                    }
                    const float2 v01 = __fmul2_rn(make_float2(vq[0], vq[1]), make_float2(bq.x, bq.y));
                    const float2 v23 = __fmul2_rn(make_float2(vq[2], vq[3]), make_float2(bq.z, bq.w));
                    vg[j] = v01.x; vg[j + 1] = v01.y; vg[j + 2] = v23.x; vg[j + 3] = v23.y;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&cx.bars[B_V_EMPTY + (g & 1)]);   // V consumed
            }
            if (SPLIT && gs_row) gs_row[(size_t)c * p.H * p.d_v] = gtot;
            const bool keep_fp32 = SPLIT && gtot >= kOresFloor;   // see TcParams::ores
            gtot *= gC;

            // X = vg - beta (S K^T), split and staged as the A operand of U^T = X^T T^T
            if (!(ok = warp_wait(cx, B_SKQ_DONE, g & 1))) break;
            tc_fence_after();
            {
                uint32_t sk[2][16];
                tmem_ld16(lane_addr + TM_SKQ + 32 * h, sk[0]);
                tmem_ld16(lane_addr + TM_SKQ + 32 * h + 16, sk[1]);
                tmem_ld_wait();
                const float4* b4 = reinterpret_cast<const float4*>(bst + 32 * h);
#pragma unroll
                for (int q2 = 0; q2 < 2; ++q2) {
                    uint32_t hi[8], lo[8];
#pragma unroll
                    for (int j2 = 0; j2 < 4; ++j2) {
                        const float4 bq = GATE == GATE_F32_ADD ? make_float4(0.f, 0.f, 0.f, 0.f)
                                                               : b4[4 * q2 + j2];
                        const int jj = 16 * q2 + 4 * j2;
                        const float2 x01 = __ffma2_rn(
                            make_float2(-bq.x, -bq.y),
                            make_float2(__uint_as_float(sk[q2][4 * j2]), __uint_as_float(sk[q2][4 * j2 + 1])),
                            make_float2(vg[jj], vg[jj + 1]));
                        const float2 x23 = __ffma2_rn(
                            make_float2(-bq.z, -bq.w),
                            make_float2(__uint_as_float(sk[q2][4 * j2 + 2]), __uint_as_float(sk[q2][4 * j2 + 3])),
                            make_float2(vg[jj + 2], vg[jj + 3]));
                        split2_bf16(x01.x, x01.y, hi[2 * j2], lo[2 * j2]);
                        split2_bf16(x23.x, x23.y, hi[2 * j2 + 1], lo[2 * j2 + 1]);
                    }
                    tmem_st8(lane_addr + TM_XHI + 16 * h + 8 * q2, hi);
                    tmem_st8(lane_addr + TM_XLO + 16 * h + 8 * q2, lo);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&cx.bars[B_X_READY]);

            // U^T back from TMEM, split and staged as the A operand of U^T P^T and U^T K
            if (!(ok = warp_wait(cx, B_U_DONE, g & 1))) break;
            tc_fence_after();
            {
                uint32_t u[2][16];
                tmem_ld16(lane_addr + TM_SKQ + 32 * h, u[0]);
                tmem_ld16(lane_addr + TM_SKQ + 32 * h + 16, u[1]);
                tmem_ld_wait();
#pragma unroll
                for (int q2 = 0; q2 < 2; ++q2) {
                    uint32_t hi[8], lo[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        split2_bf16(__uint_as_float(u[q2][2 * j]), __uint_as_float(u[q2][2 * j + 1]),
                                    hi[j], lo[j]);
                    tmem_st8(lane_addr + TM_XHI + 16 * h + 8 * q2, hi);
                    tmem_st8(lane_addr + TM_XLO + 16 * h + 8 * q2, lo);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&cx.bars[B_U_READY]);

            // S <- gamma_C (S + U^T K), handed back to the MMA warp
            if (!(ok = warp_wait(cx, B_S_DONE, g & 1))) break;
            tc_fence_after();
#pragma unroll 1
            for (int q = 0; q < 2; ++q) {
                uint32_t sv[32];
                tmem_ld32(lane_addr + TM_S + 64 * h + 32 * q, sv);
                tmem_ld_wait();
                float x[32];
#pragma unroll
                for (int j = 0; j < 32; j += 2) {
                    const float2 xx = __fmul2_rn(
                        make_float2(__uint_as_float(sv[j]), __uint_as_float(sv[j + 1])),
                        make_float2(gC, gC));
                    x[j] = xx.x;
                    x[j + 1] = xx.y;
                }
                if (last) {
                    if (st_row >= 0 && gC >= kDecayFloor && !handed_back<SPLIT>(p, it, r)) {
#pragma unroll
                        for (int j = 0; j < 32; j += 4)
                            *reinterpret_cast<float4*>(st_base + stoff + 32 * q + j) =
                                make_float4(x[j], x[j + 1], x[j + 2], x[j + 3]);
                    }
                } else {
                    if (GATE == GATE_F32_CKPT) {
#pragma unroll
                        for (int j = 0; j < 32; j += 4)
                            *reinterpret_cast<float4*>(ckpt_row(c + 1) + 32 * q + j) =
                                make_float4(x[j], x[j + 1], x[j + 2], x[j + 3]);
                    }
                    stage_state_piece(lane_addr, h, q, x);
                }
            }
            if (!last) {
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&cx.bars[B_S_READY]);
            }
            if (!(gC >= kDecayFloor)) report_fast_decay<SPLIT>(p, it, r);
            if (SPLIT && last && p.g_out && !rg.pk && h == 0)
                p.g_out[((size_t)it.n * p.H + it.h) * p.d_v + ch] = gtot;
            // O = Gamma * (Q S^T + P U); leaves after the state has been handed back
            if (!(ok = warp_wait(cx, B_O_DONE, g & 1))) break;
            if (rg.pk) {   // transition items: o_t = P_{<=t} q_t, kept in fp32 if asked
                if (SPLIT && p.qtil) {
                    tc_fence_after();
                    const int64_t qstride = (int64_t)p.H * DK;
                    store_tmem_column_f32(lane_addr + TM_SKQ + 64 + 32 * h,
                                          p.qtil + (tok0 + 32 * h) * qstride + (int64_t)it.h * DK + ch,
                                          qstride, nvalid - 32 * h,
                                          qf_row ? qf_row + (size_t)c * p.H : nullptr);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&cx.bars[B_O_READ]);
                } else {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&cx.bars[B_O_READ]);
                }
                continue;
            }
            tc_fence_after();
            uint32_t opk[16];
            {
                uint32_t ov[32];
                tmem_ld32(lane_addr + TM_SKQ + 64 + 32 * h, ov);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float2 oo = __fmul2_rn(make_float2(gam[2 * j], gam[2 * j + 1]),
                                                 make_float2(__uint_as_float(ov[2 * j]),
                                                             __uint_as_float(ov[2 * j + 1])));
                    if (SPLIT) {   // a later segment's o, kept in fp32 (ov no longer needed)
                        ov[2 * j] = __float_as_uint(oo.x);
                        ov[2 * j + 1] = __float_as_uint(oo.y);
                    }
                    opk[j] = pack_bf16x2(oo.x, oo.y);
                }
                if (SPLIT && keep_fp32 && p.ores && it.n >= p.gstart_lo) {
                    const int64_t rs = (int64_t)p.H * p.d_v;
                    Column32 col;
#pragma unroll
                    for (int j = 0; j < 32; ++j) col.v[j] = ov[j];
                    store_column_f32(col, p.ores + (tok0 + 32 * h) * rs + (int64_t)it.h * p.d_v + ch,
                                     rs, nvalid - 32 * h);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&cx.bars[B_O_READ]);
            // Out through a transpose in this warp's shared-memory slot: its 32
            // channels x 16 tokens at a time leave as 16-byte pieces of token rows.
            uint16_t* ost = reinterpret_cast<uint16_t*>(cx.smem + SM_OST + (warp - 6) * 1024);
            const int64_t ostride = (int64_t)p.H * p.d_v;
            __nv_bfloat16* obase = p.o + (tok0 + 32 * h) * ostride + (int64_t)it.h * p.d_v +
                                   it.vb * DVB + 32 * quarter;
            const int lim = nvalid - 32 * h;   // tokens of this half inside the sequence
            const int prow = lane >> 2, pcol = (lane & 3) * 8;
#pragma unroll
            for (int k = 0; k < 2; ++k) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    ost[(2 * j) * 32 + lane] = (uint16_t)(opk[8 * k + j] & 0xffffu);
                    ost[(2 * j + 1) * 32 + lane] = (uint16_t)(opk[8 * k + j] >> 16);
                }
                __syncwarp();
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int row = prow + 8 * e;
                    const uint4 v = *reinterpret_cast<const uint4*>(ost + row * 32 + pcol);
                    if (16 * k + row < lim)
                        *reinterpret_cast<uint4*>(obase + (int64_t)(16 * k + row) * ostride + pcol) = v;
                }
                __syncwarp();
            }
        }
    }
}

// ------------------------------------------------------------------ kernel
template <bool SPLIT, int GATE>
__global__ void __launch_bounds__(kThreads, 1) kda_prefill_tc_kernel(const __grid_constant__ TcParams p) {
    if (*p.status == KDA_ERR_DEVICE_INPUT) return;   // planner rejected cu_seqlens
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    Ctx cx;
    cx.smem = smem;
    cx.bars = reinterpret_cast<uint64_t*>(smem + SM_BAR);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + SM_MISC);
    cx.abort = reinterpret_cast<volatile int*>(smem + SM_MISC + 4);
    cx.never = reinterpret_cast<volatile int*>(smem + SM_MISC + 8);
    cx.slots = reinterpret_cast<volatile int*>(smem + SM_MISC + 16);
    cx.status = p.status;
    cx.timeout_ns = kTimeoutNs;   // a constant here: it costs the roles no register

    if (tid == 0) {
        *cx.abort = 0;
        *cx.never = 0;
        // arrivals per phase: 1 for TMA / MMA commits, one per warp of a group
        const uint32_t counts[B_COUNT] = {1, 1, 1, 1, 1, 8, 1, 4, 4, 4, 1, 1, 8, 1,
                                          8, 1, 8, 1, 1, 8, 2, 2, 2, 2, 1, 1, 8, 8};
        for (int b = 0; b < B_COUNT; ++b) mbar_init(&cx.bars[b], counts[b]);
        fence_mbar_init();
        tma_prefetch_desc(&p.tm_q);
        tma_prefetch_desc(&p.tm_k);
        tma_prefetch_desc(&p.tm_v);
        tma_prefetch_desc(&p.tm_a);
    }
    if (warp == 0) {
        tmem_alloc(tslot, TM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    cx.tmem = *tslot;

    if (warp == 0) {
        run_producer<SPLIT, GATE>(p, cx, lane);
    } else if (warp == 1) {
        run_mma<SPLIT>(p, cx);
    } else if (warp >= 2 && warp < 6) {
        run_token_group<SPLIT, GATE>(p, cx, tid - 64, warp, lane);
    } else {
        run_row_group<SPLIT, GATE>(p, cx, tid - 192, warp, lane);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(cx.tmem, TM_COLS);
}

// ------------------------------------------------------------------ wait probe
// The timeout path of the kernel above, run on purpose: a CTA that allocates
// its TMEM like the prefill kernel, one warp waiting with a short limit on an
// mbarrier nothing arrives on (it records KDA_ERR_DEVICE_TIMEOUT and raises
// the abort flag), a second warp waiting with the prefill's full limit on
// another such mbarrier (it must end early, through the abort flag), then the
// same join and TMEM release as the prefill kernel.
__global__ void __launch_bounds__(64, 1) kda_wait_probe_kernel(int32_t* status, uint64_t timeout_ns) {
    __shared__ __align__(8) uint64_t bars[2];
    __shared__ int flags[4];
    __shared__ uint32_t tslot;
    const int warp = threadIdx.x >> 5;
    Ctx cx;
    cx.smem = nullptr;
    cx.bars = bars;
    cx.abort = &flags[0];
    cx.never = &flags[1];
    cx.slots = &flags[2];
    cx.status = status;
    cx.timeout_ns = timeout_ns;
    if (threadIdx.x == 0) {
        flags[0] = flags[1] = flags[2] = flags[3] = 0;
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&tslot, TM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    cx.tmem = tslot;
    if (warp == 0) {
        warp_wait(cx, 0, 0);
    } else {
        Ctx full = cx;
        full.timeout_ns = kTimeoutNs;
        warp_wait(full, 1, 0);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(cx.tmem, TM_COLS);
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// 3-D map over a [T][H][D] tensor with a (box_d, 1, 64) box.
bool make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, size_t esz, int64_t T,
              int H, int D, uint32_t box_d, CUtensorMapSwizzle sw) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T};
    cuuint64_t strides[2] = {(cuuint64_t)D * esz, (cuuint64_t)H * D * esz};
    cuuint32_t box[3] = {box_d, 1, (cuuint32_t)C};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, dt, 3, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor maps and the fields every launch shares; a plain launch over the
// real sequences unless the caller changes the split fields.
bool init_params(const PrefillArgs& a, TcParams& p) {
    if (!make_map(&p.tm_q, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.total_tokens, a.H, DK, 64,
                  CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&p.tm_k, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.total_tokens, a.H, DK, 64,
                  CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&p.tm_v, a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.total_tokens, a.H, a.d_v,
                  DVB, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        (a.gate == GATE_F32 &&
         !make_map(&p.tm_a, a.alpha, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.total_tokens, a.H,
                   a.d_v, DVB, CU_TENSOR_MAP_SWIZZLE_NONE)) ||
        (a.gate == GATE_LOG_BF16 &&
         !make_map(&p.tm_a, a.alpha, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.total_tokens, a.H,
                   a.d_v, DVB, CU_TENSOR_MAP_SWIZZLE_NONE)))
        return false;
    if (a.gate == GATE_SCALAR) p.tm_a = p.tm_v;   // not read; a valid map to prefetch
    p.alpha_s = static_cast<const float*>(a.alpha);
    p.beta = a.beta;
    p.S0 = a.S0;
    p.S_T = a.S_T;
    p.o = static_cast<__nv_bfloat16*>(a.o);
    p.cu = a.cu_seqlens;
    p.order = a.order;
    p.status = a.status;
    p.H = a.H;
    p.d_v = a.d_v;
    p.nvb = a.d_v / DVB;
    p.num_items = a.num_seqs * a.H * p.nvb;
    p.vt0 = nullptr;
    p.vlen = nullptr;
    p.n_base = 0;
    p.n_base_p = 0;
    p.s0_lo = 0;
    p.s0_hi = a.num_seqs;
    p.st_lo = 0;
    p.st_hi = a.num_seqs;
    p.num_items_p = 0;
    p.g_out = nullptr;
    p.P_out = nullptr;
    p.ckpt = nullptr;
    p.redo = a.redo;
    p.gstart = nullptr;
    p.qtil = nullptr;
    p.ores = nullptr;
    p.qfro = nullptr;
    p.gstart_lo = 0;
    return true;
}

template <bool SPLIT, int GATE>
cudaError_t launch_g(TcParams& p, int grid, cudaStream_t stream) {
    cudaError_t err = cudaFuncSetAttribute(kda_prefill_tc_kernel<SPLIT, GATE>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)SMEM_BYTES);
    if (err != cudaSuccess) return err;
    kda_prefill_tc_kernel<SPLIT, GATE><<<grid, kThreads, SMEM_BYTES, stream>>>(p);
    return cudaGetLastError();
}

template <bool SPLIT>
cudaError_t launch(TcParams& p, int grid, cudaStream_t stream) {
    return launch_g<SPLIT, GATE_F32>(p, grid, stream);
}

}  // namespace

cudaError_t launch_wait_probe(int32_t* status, uint64_t timeout_ns, cudaStream_t stream) {
    cudaError_t err = cudaMemsetAsync(status, 0, sizeof(int32_t), stream);
    if (err != cudaSuccess) return err;
    kda_wait_probe_kernel<<<1, 64, 0, stream>>>(status, timeout_ns);
    return cudaGetLastError();
}

bool prefill_tc_supports(const PrefillArgs& a) {
    // o is written in 16-byte pieces
    return a.dtype == KDA_BF16 && a.d_k == DK && a.d_v % DVB == 0 && a.d_v <= 1024 &&
           a.chunk == C && (reinterpret_cast<uintptr_t>(a.o) & 15u) == 0;
}

cudaError_t launch_prefill_tc(const PrefillArgs& a, cudaStream_t stream) {
    if (!prefill_tc_supports(a)) return cudaErrorInvalidValue;
    // nothing to load: the portable kernel copies S0 to S_T
    if (a.total_tokens == 0) return launch_prefill_simt(a, stream);
    TcParams p;
    if (!init_params(a, p)) return cudaErrorInvalidValue;
    if (p.num_items == 0) return cudaSuccess;
    const int sms = sm_count();
    const int grid = p.num_items < sms ? p.num_items : sms;
    p.a_ctas = grid;
    if (a.additive) {
        if (a.gate != GATE_F32) return cudaErrorInvalidValue;
        return launch_g<false, GATE_F32_ADD>(p, grid, stream);
    }
    switch (a.gate) {
        case GATE_F32: return launch_g<false, GATE_F32>(p, grid, stream);
        case GATE_SCALAR: return launch_g<false, GATE_SCALAR>(p, grid, stream);
        case GATE_LOG_BF16: return launch_g<false, GATE_LOG_BF16>(p, grid, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_prefill_tc_ckpt(const PrefillArgs& a, float* ckpt, cudaStream_t stream) {
    if (!prefill_tc_supports(a) || a.gate != GATE_F32 || !ckpt) return cudaErrorInvalidValue;
    if (a.total_tokens == 0) return launch_prefill_simt(a, stream);   // no chunk to record
    TcParams p;
    if (!init_params(a, p)) return cudaErrorInvalidValue;
    if (p.num_items == 0) return cudaSuccess;
    p.ckpt = ckpt;
    p.redo = nullptr;
    const int sms = sm_count();
    const int grid = p.num_items < sms ? p.num_items : sms;
    p.a_ctas = grid;
    return launch_g<false, GATE_F32_CKPT>(p, grid, stream);
}

cudaError_t launch_prefill_tc_split(const PrefillArgs& a, const SplitLayout& L, char* ws,
                                    cudaStream_t stream) {
    if (!prefill_tc_supports(a) || L.M < 2 || a.gate != GATE_F32) return cudaErrorInvalidValue;
    if (a.total_tokens == 0 || a.num_seqs == 0) return launch_prefill_tc(a, stream);
    TcParams p;
    if (!init_params(a, p)) return cudaErrorInvalidValue;
    const int M = L.M, N = a.num_seqs;
    p.redo = nullptr;   // the segments' results feed the scan: a fast decay is reported
    cudaError_t err = launch_split_plan(a, L, ws, stream);
    if (err != cudaSuccess) return err;
    p.vt0 = reinterpret_cast<const int64_t*>(ws + L.vt0);
    p.vlen = reinterpret_cast<const int32_t*>(ws + L.vlen);
    const int sms = sm_count();
    // One pass over every segment: segment 0 from S0 (its o is final),
    // segments 1..M-1 from zero (o from a zero start, final state R, prod
    // alpha, and the decay from the segment start at each chunk), and the
    // transitions P of segments 1..M-1 with their outputs P_{<=t} q_t.
    p.num_items = M * N * a.H * p.nvb;
    p.S_T = reinterpret_cast<float*>(ws + L.sfin);
    p.s0_lo = 0;
    p.s0_hi = N;
    p.st_lo = 0;
    p.st_hi = M * N;
    p.g_out = reinterpret_cast<float*>(ws + L.gbuf);
    p.gstart = reinterpret_cast<float*>(ws + L.gstart);
    p.gstart_lo = N;
    p.n_base_p = N;
    p.num_items_p = (M - 1) * N * a.H;
    p.P_out = reinterpret_cast<float*>(ws + L.pbuf);
    p.qtil = reinterpret_cast<float*>(ws + L.qtil);
    p.ores = reinterpret_cast<float*>(ws + L.ores);
    p.qfro = reinterpret_cast<float*>(ws + L.qfro);
    if ((err = cudaMemsetAsync(p.qfro, 0, L.qfro_bytes, stream)) != cudaSuccess) return err;
    // one CTA per item when they all fit; otherwise the SMs are divided in
    // proportion to the two kinds of items, so that both take the same number
    // of waves
    int a_ctas, p_ctas;
    const int64_t all = (int64_t)p.num_items + p.num_items_p;
    if (all <= sms) {
        a_ctas = p.num_items;
        p_ctas = p.num_items_p;
    } else {
        a_ctas = (int)(((int64_t)sms * p.num_items + all / 2) / all);
        if (a_ctas < 1) a_ctas = 1;
        if (a_ctas > sms - 1) a_ctas = sms - 1;
        p_ctas = sms - a_ctas;
    }
    p.a_ctas = a_ctas;
    if ((err = launch<true>(p, a_ctas + p_ctas, stream)) != cudaSuccess) return err;
    // the scan of the segment maps: true initial states of segments 1..M-1
    // (and their row norms), the last map's image is S_T
    if ((err = launch_split_combine(a, L, ws, stream)) != cudaSuccess) return err;
    // each later segment's output gets its initial state's share
    return launch_split_correct(a, L, ws, stream);
}

}  // namespace kda
