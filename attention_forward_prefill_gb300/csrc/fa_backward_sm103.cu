// fa_backward_sm103.cu -- backward pass of the fused attention (the training
// step that the flash-attention-cuda README lists under "Future work"), for
// sm_103a.  Given Q, K, V, the forward output O, its gradient dO and the row
// log-sum-exp L saved by the forward, it recomputes the weights tile by tile
// and never stores them:
//   P_ij  = exp(s_ij - L_i),  s_ij = scale q_i.k_j     (2^(c s - L2) with c = scale log2 e)
//   D_i   = dO_i . O_i
//   dV_j  = sum_i P_ij dO_i
//   dS_ij = P_ij (dO_i . v_j - D_i)
//   dK_j  = scale sum_i dS_ij q_i,    dQ_i = scale sum_j dS_ij k_j
// (the chain rule through softmax: sum_j P_ij dP_ij = dO_i . O_i).
//
// Kernels, no atomics, so every gradient is bit-identical run to run:
//   bwd_prep     -D_i and -L2_i = -L_i log2 e for every row (fp32), per head padded
//                to whole 128-row tiles;
//   bwd_dkdv     per unit, a 128-key tile of a key/value head: S^T = K Q_i^T and
//                dP^T = V dO_i^T in TMEM, then P^T and dS^T as 16-bit (over them
//                at d = 128, in columns of their own at d = 64), then
//                dV += P^T dO_i and dK += dS^T Q_i accumulate in TMEM over the
//                query tiles that see the keys, of every query head that reads
//                this key/value head.  It also writes each dS block to a table in
//                HBM (the tensor core's layout for the dQ product);
//   bwd_dq_gemm  per unit, a 128-query tile: dQ = scale sum_j dS_ij K_j from the
//                table, one product per key tile;
//   bwd_dq       (without a table) per unit, a 128-query tile: S = Q K_j^T,
//                dP = dO V_j^T, dS in columns of its own, dQ += dS K_j over the
//                key tiles the queries see.
// The main kernels are persistent (one CTA per SM, units dealt in snake order);
// bwd_dkdv and bwd_dq issue the next tile's score products while the elementwise
// warps still work on the current one, as far as TMEM and the rings allow.
// Warp roles of bwd_dkdv and bwd_dq (320 threads): warps 0-7 elementwise work,
// thread = TMEM lane = tile row, two warps per row quadrant taking half of the
// tile's columns each; warp 8 TMA producer; warp 9 tcgen05 issuer and TMEM
// owner.  bwd_dq_gemm: warps 0-3 epilogue, 4 copies, 5 tcgen05 issuer.
#include <cfloat>

#include "fa_internal.h"
#include "fa_tiles.cuh"
#include "sm103_ptx.cuh"

namespace fa {

namespace {

// warps 0-7: elementwise, two per sub-partition: warp w serves TMEM lanes
// 32 (w % 4) .. +31 and half w / 4 of a tile's 128 columns; 8: TMA; 9: MMA
constexpr int kBwdThreads = 320;
constexpr int kBwdEltWarps = 8;
constexpr int kBwdTmaWarp = 8;
constexpr int kBwdMmaWarp = 9;
constexpr int kRows = 128;

__device__ int g_backward_status = 0;

template <int D>
struct BwdLayout {
    static constexpr int kChunks = D / 64;
    static constexpr int kTileBytes = kChunks * kSlabBytes;  // 128 rows x D 16-bit
    static constexpr int kStages = (D == 128) ? 2 : 3;
    static constexpr int kFixOff = 0;                       // K_j, V_j: loaded once per unit
    static constexpr int kRingOff = 2 * kTileBytes;         // stages of Q_i, dO_i and the vectors
    // L2 and D of the stage's 128 queries (two 512-byte bulk copies) after its tiles
    static constexpr int kVecInStage = 2 * kTileBytes;
    static constexpr int kStageBytes = 2 * kTileBytes + 2 * kRows * 4;
    static constexpr int kBarOff = kRingOff + kStages * kStageBytes;
    // fix_full, s_full, p_ready, acc_done, drain, s_loaded, ring_full[S], ring_empty[S], pd_done,
    // dp_full, dp_loaded, ds_ready, fix_empty
    static constexpr int kNumBars = 11 + 2 * kStages;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    static constexpr int kSmemBytes = kMiscOff + 16 + 1024;
    // TMEM: X (S^T) | Y (dP^T) | accumulator A (dV) | accumulator B (dK).  At
    // d = 64 that leaves columns 384-511, where P^T and dS^T get 64 columns each;
    // at d = 128 they are written over S^T and dP^T.
    static constexpr uint32_t kXCol = 0, kYCol = 128, kACol = 256, kBCol = 256 + D;
    static constexpr bool kOwnPds = D == 64;
    static constexpr uint32_t kPCol = kOwnPds ? 384 : kXCol, kDsCol = kOwnPds ? 448 : kYCol;
};

// The dQ kernel's shared memory: Q_i and dO_i loaded once, then K_j and V_j
// through rings of their own.  V_j is free once dP is computed, K_j only after
// dQ += dS K_j, so K gets one stage more; with it the tiles the next score
// products read are in place while the current elementwise work runs.
template <int D>
struct DqLayout {
    static constexpr int kChunks = D / 64;
    static constexpr int kTileBytes = kChunks * kSlabBytes;  // 128 rows x D 16-bit
    static constexpr int kKStages = D == 128 ? 3 : 4, kVStages = D == 128 ? 2 : 3;
    static constexpr int kFixOff = 0;                        // Q_i, dO_i
    static constexpr int kKOff = 2 * kTileBytes;
    static constexpr int kVOff = kKOff + kKStages * kTileBytes;
    static constexpr int kBarOff = kVOff + kVStages * kTileBytes;
    // fix_full, s_full, p_ready, acc_done, drain, s_loaded, dq_done, fix_empty,
    // k_full[KS], k_empty[KS], v_full[VS], v_empty[VS]
    static constexpr int kNumBars = 8 + 2 * kKStages + 2 * kVStages;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    static constexpr int kSmemBytes = kMiscOff + 16 + 1024;
    // TMEM: S | dP | dQ accumulator | dS (16-bit, 64 columns)
    static constexpr uint32_t kXCol = 0, kYCol = 128, kACol = 256, kDsCol = 384;
};

struct BwdParams {
    const float *lse2;  // [B Hq][npad] minus the row log-sum-exp in log2 units, -L_i log2 e
    const float *dsum;  // [B Hq][npad] minus D_i = dO_i . O_i
    void *g0;           // dkdv: dK [B Hkv][N][d]; dq: dQ [B Hq][N][d]
    void *g1;           // dkdv: dV [B Hkv][N][d]
    int group;          // flat over (batch, head): query head x reads key/value head x / group
    int N;
    int n_t;            // 128-row tiles per head
    int npad;           // n_t * 128: row stride of lse2 and dsum per head (zero past N)
    int causal;
    int grad_dtype;
    float scale;
    float c;            // scale * log2(e)
    int n_units;        // units dealt to the persistent CTAs: dkdv (key/value head, key
                        // tile), dq (query head, query tile)
    // dkdv: when set, dS of every (key tile j, query tile i) item of query head h is
    // also written here, one 32 KB block per (h, j, i), for the dQ product pass that
    // reads it instead of recomputing S and dP.
    uint16_t *ds_t;
};

// Untiled bulk copy (as bulk_load) with an L2 cache policy (createpolicy) for the
// source lines.
__device__ __forceinline__ void bulk_load_hint(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                               uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
            "r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Shared-memory matrix descriptor of an unswizzled (interleaved) operand: 8 x 16-byte
// core matrices of 128 bytes.  For an MN-major operand, lbo is the byte stride between
// core matrices along K and sbo the one along M/N.
__device__ __forceinline__ uint64_t sdesc_plain(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;  // descriptor version (tcgen05); layout 0: no swizzle
    return d;
}

// The dS table.  A block holds the 128 x 128 16-bit dS values of (query head h,
// key tile j, query tile i) in the tensor core's unswizzled layout for an MN-major
// operand, so that the dQ pass copies it to shared memory as it is: 8 x 8 core
// matrices of 128 bytes (8 keys, each with 8 consecutive queries), the 16 key
// groups of a query group adjacent (128 bytes apart), query groups 2 KB apart.
// Key row r of a warp's 32 writes its 8 queries of query group g at
// g * 2048 + (r / 8) * 128 + (r % 8) * 16 bytes: the warp's 32 16-byte stores
// fill 512 contiguous bytes.
constexpr int kDsCoreBytes = 128;                    // 8 keys x 8 queries
constexpr int kDsGroupBytes = 16 * kDsCoreBytes;     // a query group: 128 keys
constexpr int kDsBlockBytes = kRows * kRows * 2;     // 32 KB

__device__ __forceinline__ uint16_t *ds_block(const BwdParams &p, int h, int j, int i) {
    return p.ds_t + ((static_cast<size_t>(h) * p.n_t + j) * p.n_t + i) * (kRows * kRows);
}

// Key row r's slot in query group 0 of its block.
__device__ __forceinline__ uint16_t *ds_key_row(uint16_t *block, int r) {
    return block + ((r >> 3) * kDsCoreBytes + (r & 7) * 16) / 2;
}

// Key row r's 32 dS values of queries 32 q .. 32 q + 31 (16 packed words), four
// query groups, as streaming (evict-first) stores: the table passes through L2
// once and should not push out the Q and dO tiles that the other key tiles read
// there again.
__device__ __forceinline__ void store_ds_quarter(uint16_t *row, int q, const uint32_t (&w)[16]) {
#pragma unroll
    for (int v = 0; v < 4; ++v)
        __stcs(reinterpret_cast<uint4 *>(row + (4 * q + v) * (kDsGroupBytes / 2)),
               make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]));
}

// ---------------------------------------------------------------- D and L2
// Rows of the padded [B Hq][npad] layout; rows past N get zeros, so that every
// 128-row tile of it can be copied whole.  Both are stored negated, the sign the
// elementwise work adds them with.  A row is read as 16-byte words, one per lane
// (d / 8 lanes a row), and every thread keeps kPrepRows such words of O and of
// dO in flight; each lane sums its eight products in order, then the row's lanes
// combine by a fixed butterfly, so D is the same on every run.
constexpr int kPrepThreads = 256;
constexpr int kPrepRows = 2;

template <int D, bool BF16>
__device__ __forceinline__ float dot8(const uint4 &a, const uint4 &b) {
    const uint32_t ua[4] = {a.x, a.y, a.z, a.w}, ub[4] = {b.x, b.y, b.z, b.w};
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float a0, a1, b0, b1;
        if constexpr (BF16) {
            a0 = __uint_as_float(ua[i] << 16); a1 = __uint_as_float(ua[i] & 0xffff0000u);
            b0 = __uint_as_float(ub[i] << 16); b1 = __uint_as_float(ub[i] & 0xffff0000u);
        } else {
            const float2 fa = __half22float2(*reinterpret_cast<const __half2 *>(&ua[i]));
            const float2 fb = __half22float2(*reinterpret_cast<const __half2 *>(&ub[i]));
            a0 = fa.x; a1 = fa.y; b0 = fb.x; b1 = fb.y;
        }
        acc = fmaf(a0, b0, acc);
        acc = fmaf(a1, b1, acc);
    }
    return acc;
}

template <int D, bool BF16>
__global__ void __launch_bounds__(kPrepThreads) bwd_prep_kernel(const uint16_t *o, const uint16_t *dout,
                                                                const float *lse, float *lse2, float *dsum,
                                                                long long rows_pad, int N, int npad) {
    constexpr int LPR = D / 8;       // lanes per row
    constexpr int RPW = 32 / LPR;    // rows per warp and word
    // The dK/dV pass (launched with programmatic dependent launch) may start its
    // set-up now; it waits for this grid before it reads D and L2.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int lane = threadIdx.x & 31, sub = lane % LPR;
    const long long warp_g = (static_cast<long long>(blockIdx.x) * kPrepThreads + threadIdx.x) >> 5;
    const long long first = warp_g * RPW * kPrepRows + lane / LPR;
    uint4 a[kPrepRows], b[kPrepRows];
    long long row[kPrepRows];
#pragma unroll
    for (int u = 0; u < kPrepRows; ++u) {
        const long long prow = first + u * RPW;
        const long long i = prow % npad;
        const bool live = prow < rows_pad && i < N;
        row[u] = live ? (prow / npad) * N + i : -1;
        a[u] = live ? __ldg(reinterpret_cast<const uint4 *>(o + row[u] * D) + sub) : make_uint4(0, 0, 0, 0);
        b[u] = live ? __ldg(reinterpret_cast<const uint4 *>(dout + row[u] * D) + sub) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kPrepRows; ++u) {
        float acc = dot8<D, BF16>(a[u], b[u]);
#pragma unroll
        for (int off = 1; off < LPR; off <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        const long long prow = first + u * RPW;
        if (sub == 0 && prow < rows_pad) {
            dsum[prow] = row[u] >= 0 ? -acc : 0.f;
            lse2[prow] = row[u] >= 0 ? -(lse[row[u]] * 1.4426950408889634f) : 0.f;
        }
    }
}

// Elementwise work on one 32-column quarter of a score tile held in TMEM:
// returns, for the thread's row, the packed 16-bit weights and dS values.  The
// L2 and D values come negated (nl2 = -L2, nd = -D), per column from shared
// memory or per row, and the arithmetic runs on fp32 pairs:
//   p = 2^(c s + nl2),  dS = p (dP + nd).
template <bool BF16, bool WANT_P, bool MASKED>
__device__ __forceinline__ void weights_quarter_impl(const uint32_t (&sr)[32], const uint32_t (&dr)[32],
                                                     uint32_t (&pk)[16], uint32_t (&dk)[16], float c,
                                                     const float *nl2_col, const float *nd_col,
                                                     float nl2_row, float nd_row, uint32_t vis_mask) {
    const uint64_t c2 = f2_pack(c, c);
#pragma unroll
    for (int e2 = 0; e2 < 16; ++e2) {
        const int col = 2 * e2;
        const uint64_t nl2 = nl2_col ? *reinterpret_cast<const uint64_t *>(nl2_col + col) : f2_pack(nl2_row, nl2_row);
        const uint64_t nd = nd_col ? *reinterpret_cast<const uint64_t *>(nd_col + col) : f2_pack(nd_row, nd_row);
        const uint64_t x = ffma2(f2_pack(__uint_as_float(sr[col]), __uint_as_float(sr[col + 1])), c2, nl2);
        float p0 = ex2_approx(f2_lo(x)), p1 = ex2_approx(f2_hi(x));
        if (MASKED) {
            p0 = ((vis_mask >> col) & 1u) ? p0 : 0.f;
            p1 = ((vis_mask >> (col + 1)) & 1u) ? p1 : 0.f;
        }
        const uint64_t dd =
            fmul2(f2_pack(p0, p1), fadd2(f2_pack(__uint_as_float(dr[col]), __uint_as_float(dr[col + 1])), nd));
        if (WANT_P) pk[e2] = pack2t<BF16>(p0, p1);
        dk[e2] = pack2t<BF16>(f2_lo(dd), f2_hi(dd));
    }
}

// The weights of a 32-column quarter; the select is only paid where some
// column of the thread's row is masked.
template <bool BF16, bool WANT_P>
__device__ __forceinline__ void weights_quarter(const uint32_t (&sr)[32], const uint32_t (&dr)[32],
                                                uint32_t (&pk)[16], uint32_t (&dk)[16], float c,
                                                const float *nl2_col, const float *nd_col,
                                                float nl2_row, float nd_row, uint32_t vis_mask) {
    if (vis_mask == 0xffffffffu)
        weights_quarter_impl<BF16, WANT_P, false>(sr, dr, pk, dk, c, nl2_col, nd_col, nl2_row, nd_row,
                                                  vis_mask);
    else
        weights_quarter_impl<BF16, WANT_P, true>(sr, dr, pk, dk, c, nl2_col, nd_col, nl2_row, nd_row,
                                                 vis_mask);
}

// The same work in two steps, for a pipeline that multiplies P^T before dS^T is
// known.  First the weights of a quarter: sr holds the scores on entry and the
// fp32 weights on return, pk the packed 16-bit weights.
template <bool BF16, bool MASKED>
__device__ __forceinline__ void p_quarter_impl(uint32_t (&sr)[32], uint32_t (&pk)[16], float c,
                                               const float *nl2_col, uint32_t vis_mask) {
    const uint64_t c2 = f2_pack(c, c);
#pragma unroll
    for (int e2 = 0; e2 < 16; ++e2) {
        const int col = 2 * e2;
        const uint64_t x = ffma2(f2_pack(__uint_as_float(sr[col]), __uint_as_float(sr[col + 1])), c2,
                                 *reinterpret_cast<const uint64_t *>(nl2_col + col));
        float p0 = ex2_approx(f2_lo(x)), p1 = ex2_approx(f2_hi(x));
        if (MASKED) {
            p0 = ((vis_mask >> col) & 1u) ? p0 : 0.f;
            p1 = ((vis_mask >> (col + 1)) & 1u) ? p1 : 0.f;
        }
        sr[col] = __float_as_uint(p0);
        sr[col + 1] = __float_as_uint(p1);
        pk[e2] = pack2t<BF16>(p0, p1);
    }
}

template <bool BF16>
__device__ __forceinline__ void p_quarter(uint32_t (&sr)[32], uint32_t (&pk)[16], float c, const float *nl2_col,
                                          uint32_t vis_mask) {
    if (vis_mask == 0xffffffffu)
        p_quarter_impl<BF16, false>(sr, pk, c, nl2_col, vis_mask);
    else
        p_quarter_impl<BF16, true>(sr, pk, c, nl2_col, vis_mask);
}

// Then dS = P (dP - D) of the quarter from the kept weights (the arithmetic of
// weights_quarter, so the two pipelines give the same bits).
template <bool BF16>
__device__ __forceinline__ void ds_quarter(const uint32_t (&pr)[32], const uint32_t (&dr)[32], uint32_t (&dk)[16],
                                           const float *nd_col) {
#pragma unroll
    for (int e2 = 0; e2 < 16; ++e2) {
        const int col = 2 * e2;
        const uint64_t dd = fmul2(f2_pack(__uint_as_float(pr[col]), __uint_as_float(pr[col + 1])),
                                  fadd2(f2_pack(__uint_as_float(dr[col]), __uint_as_float(dr[col + 1])),
                                        *reinterpret_cast<const uint64_t *>(nd_col + col)));
        dk[e2] = pack2t<BF16>(f2_lo(dd), f2_hi(dd));
    }
}

// ---------------------------------------------------------------- dK, dV
// One unit of the dK/dV pass: key tile `jt` of (batch, key/value head) `bhk`,
// against every query tile that sees it of every query head of its group.  A
// persistent CTA takes units k = 0, 1, ... in snake order over rounds of
// G = gridDim.x, as in the dQ pass; causal units come heaviest first (the first
// key tiles of every head see the most query tiles).
struct DkdvUnit {
    int bhk, jt, i_first, n_qt, n_iter, bhq0;
};

__device__ __forceinline__ bool dkdv_unit(const BwdParams &p, int k, DkdvUnit &u) {
    const long long G = gridDim.x, c = blockIdx.x;
    const long long idx = static_cast<long long>(k) * G + ((k & 1) ? G - 1 - c : c);
    if (idx >= p.n_units) return false;
    const int n_heads = p.n_units / p.n_t;
    if (p.causal) {
        u.bhk = static_cast<int>(idx % n_heads);
        u.jt = static_cast<int>(idx / n_heads);
    } else {
        u.bhk = static_cast<int>(idx / p.n_t);
        u.jt = static_cast<int>(idx % p.n_t);
    }
    u.i_first = p.causal ? u.jt : 0;  // query tiles that see key tile jt
    u.n_qt = p.n_t - u.i_first;
    u.n_iter = p.group * u.n_qt;      // every query head of the group, every tile
    u.bhq0 = u.bhk * p.group;         // first query head
    return true;
}

template <int D, bool BF16>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                    const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_do,
                    const BwdParams p) {
    using L = BwdLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBarOff);
    uint64_t *fix_full = bars + 0, *s_full = bars + 1, *p_ready = bars + 2, *acc_done = bars + 3;
    uint64_t *drain = bars + 4, *s_loaded = bars + 5;
    uint64_t *ring_full = bars + 6, *ring_empty = bars + 6 + L::kStages;
    uint64_t *pd_done = bars + 6 + 2 * L::kStages;
    // d = 128: dP^T ready, every warp's dP^T loaded, dS^T ready
    uint64_t *dp_full = pd_done + 1, *dp_loaded = pd_done + 2, *ds_ready = pd_done + 3;
    uint64_t *fix_empty = pd_done + 4;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kMiscOff);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kMiscOff + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Barriers that complete once per unit (fix_full, fix_empty, acc_done) wait on
    // the parity of the unit counter k; those that complete once per item on the
    // parity of the CTA's item counter g, which runs on across units, and so does
    // the ring of (Q, dO) stages.
    // The dQ pass (programmatic dependent launch) may start its set-up once this
    // grid runs; it waits for this grid to finish before it reads D and L2.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (threadIdx.x == 0) {
        mbar_init(fix_full, 1);
        mbar_init(s_full, 1);
        mbar_init(p_ready, kBwdEltWarps);
        mbar_init(acc_done, 1);
        mbar_init(drain, 1);
        mbar_init(s_loaded, kBwdEltWarps);
        mbar_init(pd_done, 1);
        mbar_init(dp_full, 1);
        mbar_init(dp_loaded, kBwdEltWarps);
        mbar_init(ds_ready, kBwdEltWarps);
        mbar_init(fix_empty, 1);
        for (int s = 0; s < L::kStages; ++s) {
            mbar_init(ring_full + s, 1);
            mbar_init(ring_empty + s, 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kBwdMmaWarp) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    if (warp == kBwdTmaWarp && lane == 0) {
        prefetch_tensormap(&map_q);
        prefetch_tensormap(&map_k);
        prefetch_tensormap(&map_v);
        prefetch_tensormap(&map_do);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kBwdTmaWarp) {
        if (lane == 0) {
            uint8_t *fix = smem + L::kFixOff, *ring = smem + L::kRingOff;
            const uint64_t pol = l2_policy_evict_last();
            bool ok = true;
            int nfix = 0, ni = 0;  // K/V pairs and ring items issued
            bool prep_done = false;  // D and L2 come from the grid before (prep)
            DkdvUnit u;
            for (int k = 0; ok && dkdv_unit(p, k, u); ++k) {
                // K and V of the unit before must have been read by its last products
                if (k > 0 && !mbar_wait(fix_empty, (k - 1) & 1, abort_flag, kWatchdogNs)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(fix_full, 2 * L::kTileBytes);
                for (int c = 0; c < L::kChunks; ++c) {
                    tma_load_3d(fix + c * kSlabBytes, &map_k, fix_full, c * 64, u.jt * kRows, u.bhk, pol);
                    tma_load_3d(fix + L::kTileBytes + c * kSlabBytes, &map_v, fix_full, c * 64, u.jt * kRows,
                                u.bhk, pol);
                }
                ++nfix;
                for (int n = 0; n < u.n_iter; ++n) {
                    const int slot = ni % L::kStages;
                    if (ni >= L::kStages &&
                        !mbar_wait(ring_empty + slot, ((ni / L::kStages) - 1) & 1, abort_flag, kWatchdogNs)) {
                        ok = false;
                        break;
                    }
                    const int row = (u.i_first + n % u.n_qt) * kRows;
                    const int bhq = u.bhq0 + n / u.n_qt;
                    uint8_t *st = ring + slot * L::kStageBytes;
                    mbar_arrive_expect_tx(ring_full + slot, 2 * L::kTileBytes + 2 * kRows * 4);
                    for (int c = 0; c < L::kChunks; ++c) {
                        tma_load_3d(st + c * kSlabBytes, &map_q, ring_full + slot, c * 64, row, bhq, pol);
                        tma_load_3d(st + L::kTileBytes + c * kSlabBytes, &map_do, ring_full + slot, c * 64, row,
                                    bhq, pol);
                    }
                    // the 128 queries' L2 and D (the padded layout keeps both copies whole),
                    // written by the prep grid this one may have started beside
                    if (!prep_done) {
                        asm volatile("griddepcontrol.wait;" ::: "memory");
                        prep_done = true;
                    }
                    const size_t vrow = static_cast<size_t>(bhq) * p.npad + row;
                    bulk_load(st + L::kVecInStage, p.lse2 + vrow, kRows * 4, ring_full + slot);
                    bulk_load(st + L::kVecInStage + kRows * 4, p.dsum + vrow, kRows * 4, ring_full + slot);
                    ++ni;
                }
            }
            if (!ok) {  // let every copy already issued land (only the last K/V can be in flight)
                constexpr uint64_t kDrainNs = 200ull * 1000ull * 1000ull;
                int dummy = 0;
                if (nfix > 0) mbar_wait(fix_full, (nfix - 1) & 1, &dummy, kDrainNs);
                for (int m = (ni > L::kStages ? ni - L::kStages : 0); m < ni; ++m)
                    mbar_wait(ring_full + (m % L::kStages), (m / L::kStages) & 1, &dummy, kDrainNs);
            }
        }
        __syncwarp();
    } else if (warp == kBwdMmaWarp) {
        if (lane == 0) {
            const uint32_t idesc_s = idesc_f16(BF16, kRows, kRows, false, false);
            const uint32_t idesc_acc = idesc_f16(BF16, kRows, D, false, true);
            const uint32_t fix = smem_u32(smem + L::kFixOff), ring = smem_u32(smem + L::kRingOff);
            const uint64_t k_desc = sdesc_sw128(fix, 16, 1024);
            const uint64_t v_desc = sdesc_sw128(fix + L::kTileBytes, 16, 1024);
            bool ok = true;
            int g = 0;
            DkdvUnit u;
            auto stage_ready = [&](int j) {
                if (!mbar_wait(ring_full + j % L::kStages, (j / L::kStages) & 1, abort_flag, kWatchdogNs))
                    return false;
                tc_fence_after();
                return true;
            };
            for (int k = 0; ok && dkdv_unit(p, k, u); ++k) {
                if (!mbar_wait(fix_full, k & 1, abort_flag, kWatchdogNs)) { ok = false; break; }
                tc_fence_after();
                if constexpr (!L::kOwnPds) {
                    // d = 128: P^T and dS^T are written over S^T and dP^T, in two steps.
                    // dP^T runs while the weights are computed, dV += P^T dO_i while dS^T is.
                    // S^T of item j (Q_j from its stage) and dP^T (dO_j).  At a unit's
                    // start they overwrite the last unit's P^T and dS^T, which the dV and
                    // dK products issued before them (and run in order) read.
                    auto issue_s = [&](int j) {
                        const uint32_t st = ring + (j % L::kStages) * L::kStageBytes;
                        issue_qk<D>(tmem + L::kXCol, k_desc, sdesc_sw128(st, 16, 1024), idesc_s);
                        umma_commit(s_full);
                    };
                    auto issue_dp = [&](int j) {
                        const uint32_t st = ring + (j % L::kStages) * L::kStageBytes;
                        issue_qk<D>(tmem + L::kYCol, v_desc, sdesc_sw128(st + L::kTileBytes, 16, 1024), idesc_s);
                        umma_commit(dp_full);
                    };
                    if (!stage_ready(g)) { ok = false; break; }
                    issue_s(g);
                    issue_dp(g);
                    if (u.n_iter == 1) umma_commit(fix_empty);
                    for (int n = 0; n < u.n_iter && ok; ++n) {
                        const int gi = g + n;
                        const int slot = gi % L::kStages;
                        const uint32_t st = ring + slot * L::kStageBytes;
                        if (!mbar_wait(p_ready, gi & 1, abort_flag, kWatchdogNs)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        issue_pv<D>(tmem + L::kACol, tmem + L::kPCol,
                                    sdesc_sw128(st + L::kTileBytes, kSlabBytes, 1024), idesc_acc, n > 0);
                        // S^T of the next item may overwrite P^T once dV has been issued (the
                        // products run in order); take it now if its Q tile has landed, so it
                        // runs under the dS^T step, else after dK.
                        const bool more = n + 1 < u.n_iter;
                        bool s_issued = false;
                        if (more && mbar_test_wait(ring_full + (gi + 1) % L::kStages, ((gi + 1) / L::kStages) & 1)) {
                            tc_fence_after();
                            issue_s(gi + 1);
                            s_issued = true;
                        }
                        if (!mbar_wait(ds_ready, gi & 1, abort_flag, kWatchdogNs)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        issue_pv<D>(tmem + L::kBCol, tmem + L::kDsCol, sdesc_sw128(st, kSlabBytes, 1024), idesc_acc,
                                    n > 0);
                        umma_commit(ring_empty + slot);
                        if (more) {
                            if (!s_issued) {
                                if (!stage_ready(gi + 1)) {
                                    ok = false;
                                    break;
                                }
                                issue_s(gi + 1);
                            }
                            issue_dp(gi + 1);  // over dS^T, after the dK product that reads it
                            // the unit's last reads of K and V are issued: free them once done
                            if (n + 2 == u.n_iter) umma_commit(fix_empty);
                        }
                    }
                } else {
                    // S^T = K Q_i^T and dP^T = V dO_i^T (keys on TMEM lanes) for ring item j
                    auto issue_scores = [&](int j) {
                        if (!stage_ready(j)) return false;
                        const uint32_t st = ring + (j % L::kStages) * L::kStageBytes;
                        issue_qk<D>(tmem + L::kXCol, k_desc, sdesc_sw128(st, 16, 1024), idesc_s);
                        issue_qk<D>(tmem + L::kYCol, v_desc, sdesc_sw128(st + L::kTileBytes, 16, 1024), idesc_s);
                        umma_commit(s_full);
                        return true;
                    };
                    // The unit's first scores overwrite the last unit's S^T and dP^T:
                    // every warp holds those (implied by its P-ready arrival, awaited).
                    if (g > 0) {
                        if (!mbar_wait(s_loaded, (g - 1) & 1, abort_flag, kWatchdogNs)) { ok = false; break; }
                        tc_fence_after();
                    }
                    if (!issue_scores(g)) { ok = false; break; }
                    if (u.n_iter == 1) umma_commit(fix_empty);
                    for (int n = 0; n < u.n_iter && ok; ++n) {
                        const int gi = g + n;
                        // P^T and dS^T have columns of their own: once every elementwise warp
                        // holds this item's scores, the next item's products may start.
                        if (n + 1 < u.n_iter) {
                            if (!mbar_wait(s_loaded, gi & 1, abort_flag, kWatchdogNs)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            if (!issue_scores(gi + 1)) {
                                ok = false;
                                break;
                            }
                            if (n + 2 == u.n_iter) umma_commit(fix_empty);
                        }
                        if (!mbar_wait(p_ready, gi & 1, abort_flag, kWatchdogNs)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        // dV += P^T dO_i and dK += dS^T Q_i (P^T, dS^T from TMEM; dO_i, Q_i MN-major)
                        const int slot = gi % L::kStages;
                        const uint32_t st = ring + slot * L::kStageBytes;
                        issue_pv<D>(tmem + L::kACol, tmem + L::kPCol,
                                    sdesc_sw128(st + L::kTileBytes, kSlabBytes, 1024), idesc_acc, n > 0);
                        issue_pv<D>(tmem + L::kBCol, tmem + L::kDsCol, sdesc_sw128(st, kSlabBytes, 1024), idesc_acc,
                                    n > 0);
                        umma_commit(ring_empty + slot);
                        umma_commit(pd_done);
                    }
                }
                if (!ok) break;
                umma_commit(acc_done);
                g += u.n_iter;
            }
            umma_commit(drain);
            int dummy = 0;
            mbar_wait(drain, 0, &dummy, kWatchdogNs);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------------- elementwise
        const int wq = warp & 3, hf = warp >> 2;  // TMEM lane quadrant; column half
        const int r = wq * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
        bool ok = true;
        int g = 0;
        DkdvUnit u;
        for (int k = 0; ok && dkdv_unit(p, k, u); ++k) {
            const int key = u.jt * kRows + r;
            const int g_end = g + u.n_iter;
            int qt = u.i_first;  // the item's query tile: i_first .. n_t - 1, once per query head
            int hq = u.bhq0;     // the item's query head
            for (int gi = g; gi < g_end && ok; ++gi) {
                const int q0 = qt * kRows;
                uint16_t *const ds_row = p.ds_t ? ds_key_row(ds_block(p, hq, u.jt, qt), r) : nullptr;
                if (++qt == p.n_t) {
                    qt = u.i_first;
                    ++hq;
                }
                // this half's 64 query columns: L2 and D, brought into the ring stage with
                // Q_i and dO_i (the MMA thread waited for the same barrier; so do we)
                const int slot = gi % L::kStages;
                if (!warp_wait(ring_full + slot, (gi / L::kStages) & 1, abort_flag)) { ok = false; break; }
                const float *vstage = reinterpret_cast<const float *>(smem + L::kRingOff + slot * L::kStageBytes +
                                                                      L::kVecInStage);
                const float *nl2_v = vstage + hf * 64, *nd_v = vstage + kRows + hf * 64;
                if (!warp_wait(s_full, gi & 1, abort_flag)) { ok = false; break; }
                tc_fence_after();
                if constexpr (L::kOwnPds) {
                    // d = 64: P^T and dS^T have columns of their own
                    uint32_t sr[2][32], dr[2][32];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        tmem_ld32(tmem + lane_off + L::kXCol + (2 * hf + h) * 32, sr[h]);
                        tmem_ld32(tmem + lane_off + L::kYCol + (2 * hf + h) * 32, dr[h]);
                    }
                    tmem_ld_wait();
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        reg_fence32(sr[h]);
                        reg_fence32(dr[h]);
                    }
                    // The arrival tells the MMA thread the score columns are free.
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(s_loaded);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int q = 2 * hf + h;
                        // column col is query q0 + 32 q + col; it sees the key when it exists
                        // and, causally, when key <= query
                        const int qb = q0 + q * 32;
                        uint32_t vis = 0xffffffffu;
                        if (qb + 32 > p.N) vis = p.N > qb ? (0xffffffffu >> (32 - (p.N - qb))) : 0u;
                        if (key >= p.N) vis = 0u;  // a padding key row: P and dS stay 0
                        if (p.causal) {
                            const int lo = key - qb;  // first visible column
                            vis &= lo <= 0 ? 0xffffffffu : (lo >= 32 ? 0u : (0xffffffffu << lo));
                        }
                        uint32_t pk[16], dk[16];
                        weights_quarter<BF16, true>(sr[h], dr[h], pk, dk, p.c, nl2_v + h * 32, nd_v + h * 32, 0.f, 0.f,
                                                    vis);
                        if (h == 0 && gi > 0) {
                            // the previous item's P^T and dS^T must have been read.  This
                            // also keeps p_ready from completing twice before the MMA
                            // thread, which committed pd_done after seeing it, looks.
                            if (!warp_wait(pd_done, (gi - 1) & 1, abort_flag)) { ok = false; break; }
                            tc_fence_after();
                        }
                        tmem_st16(tmem + lane_off + L::kPCol + q * 16, pk);
                        tmem_st16(tmem + lane_off + L::kDsCol + q * 16, dk);
                        if (ds_row) store_ds_quarter(ds_row, q, dk);
                    }
                    if (!ok) break;
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(p_ready);
                } else {
                    // d = 128 in two steps.  First P^T from S^T, over S^T: the upper
                    // half's P^T lands on columns the lower half reads, so every warp's
                    // loads complete before any warp stores.
                    uint32_t sr[2][32], dr[2][32];
#pragma unroll
                    for (int h = 0; h < 2; ++h) tmem_ld32(tmem + lane_off + L::kXCol + (2 * hf + h) * 32, sr[h]);
                    tmem_ld_wait();
#pragma unroll
                    for (int h = 0; h < 2; ++h) reg_fence32(sr[h]);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(s_loaded);
                    if (!warp_wait(s_loaded, gi & 1, abort_flag)) { ok = false; break; }
                    tc_fence_after();
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int q = 2 * hf + h;
                        // column col is query q0 + 32 q + col; it sees the key when it
                        // exists and, causally, when key <= query
                        const int qb = q0 + q * 32;
                        uint32_t vis = 0xffffffffu;
                        if (qb + 32 > p.N) vis = p.N > qb ? (0xffffffffu >> (32 - (p.N - qb))) : 0u;
                        if (key >= p.N) vis = 0u;  // a padding key row: P and dS stay 0
                        if (p.causal) {
                            const int lo = key - qb;  // first visible column
                            vis &= lo <= 0 ? 0xffffffffu : (lo >= 32 ? 0u : (0xffffffffu << lo));
                        }
                        uint32_t pk[16];
                        p_quarter<BF16>(sr[h], pk, p.c, nl2_v + h * 32, vis);
                        tmem_st16(tmem + lane_off + L::kPCol + q * 16, pk);
                    }
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(p_ready);
                    // Then dS^T = P^T (dP^T - D) over dP^T, the same way.
                    if (!warp_wait(dp_full, gi & 1, abort_flag)) { ok = false; break; }
                    tc_fence_after();
#pragma unroll
                    for (int h = 0; h < 2; ++h) tmem_ld32(tmem + lane_off + L::kYCol + (2 * hf + h) * 32, dr[h]);
                    tmem_ld_wait();
#pragma unroll
                    for (int h = 0; h < 2; ++h) reg_fence32(dr[h]);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(dp_loaded);
                    if (!warp_wait(dp_loaded, gi & 1, abort_flag)) { ok = false; break; }
                    tc_fence_after();
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint32_t dk[16];
                        ds_quarter<BF16>(sr[h], dr[h], dk, nd_v + h * 32);
                        tmem_st16(tmem + lane_off + L::kDsCol + (2 * hf + h) * 16, dk);
                        if (ds_row) store_ds_quarter(ds_row, 2 * hf + h, dk);
                    }
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(ds_ready);
                }
            }
            if (!ok || !warp_wait(acc_done, k & 1, abort_flag)) {
                ok = false;
                break;
            }
            // the lower half stores dV, the upper half dK; the next unit's first dV and
            // dK products (which overwrite the accumulators) wait for this warp's next
            // P-ready (and, at d = 128, dS-ready) arrival, after these loads
            tc_fence_after();
            const int osize = p.grad_dtype == FA_F32 ? 4 : 2;
            const size_t row_off = (static_cast<size_t>(u.bhk) * p.N + key) * D * osize;
            uint8_t *dst = static_cast<uint8_t *>(hf ? p.g0 : p.g1) + row_off;
            const uint32_t acc_col = hf ? L::kBCol : L::kACol;
            const float mul = hf ? p.scale : 1.f;
#pragma unroll
            for (int q = 0; q < D / 32; ++q) {
                uint32_t o[32];
                tmem_ld32(tmem + lane_off + acc_col + q * 32, o);
                tmem_ld_wait();
                reg_fence32(o);
                if (key < p.N) store_out32(dst + q * 32 * osize, o, mul, p.grad_dtype);
            }
            tc_fence_before();
            g = g_end;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kBwdMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    if (threadIdx.x == 0 && *abort_flag) atomicCAS(&g_backward_status, 0, (int)FA_ERR_WATCHDOG);
}

// ---------------------------------------------------------------- dQ
// One unit of the dQ pass: query tile `it` of (batch, query head) `bh`, and the
// key tiles it sees.  A persistent CTA takes units k = 0, 1, ... of its own:
// unit k * G + c, or k * G + G - 1 - c in odd rounds (snake order over rounds of
// G = gridDim.x).  Causal units come heaviest first (the last query tiles of
// every head), so the light ones fill the last round.
struct DqUnit {
    int bh, bhk, it, n_iter;
};

__device__ __forceinline__ bool dq_unit(const BwdParams &p, int k, DqUnit &u) {
    const long long G = gridDim.x, c = blockIdx.x;
    const long long idx = static_cast<long long>(k) * G + ((k & 1) ? G - 1 - c : c);
    if (idx >= p.n_units) return false;
    const int n_heads = p.n_units / p.n_t;
    if (p.causal) {
        u.bh = static_cast<int>(idx % n_heads);
        u.it = p.n_t - 1 - static_cast<int>(idx / n_heads);
    } else {
        u.bh = static_cast<int>(idx / p.n_t);
        u.it = static_cast<int>(idx % p.n_t);
    }
    u.bhk = u.bh / p.group;                                    // its key/value head
    u.n_iter = p.causal ? u.it + 1 : p.n_t;                    // key tiles the queries see
    return true;
}

template <int D, bool BF16>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                  const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_do,
                  const BwdParams p) {
    using L = DqLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBarOff);
    uint64_t *fix_full = bars + 0, *s_full = bars + 1, *p_ready = bars + 2, *acc_done = bars + 3;
    uint64_t *drain = bars + 4, *s_loaded = bars + 5;
    uint64_t *dq_done = bars + 6, *fix_empty = bars + 7;
    uint64_t *k_full = bars + 8, *k_empty = k_full + L::kKStages;
    uint64_t *v_full = k_empty + L::kKStages, *v_empty = v_full + L::kVStages;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kMiscOff);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kMiscOff + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Barriers that complete once per unit (fix_full, fix_empty, acc_done) wait on
    // the parity of the unit counter k; those that complete once per key tile on
    // the parity of the CTA's key-tile counter g, which runs on across units, and
    // so do the K and V rings.

    if (threadIdx.x == 0) {
        mbar_init(fix_full, 1);
        mbar_init(s_full, 1);
        mbar_init(p_ready, kBwdEltWarps);
        mbar_init(acc_done, 1);
        mbar_init(drain, 1);
        mbar_init(s_loaded, kBwdEltWarps);
        mbar_init(dq_done, 1);
        mbar_init(fix_empty, 1);
        for (int s = 0; s < L::kKStages; ++s) {
            mbar_init(k_full + s, 1);
            mbar_init(k_empty + s, 1);
        }
        for (int s = 0; s < L::kVStages; ++s) {
            mbar_init(v_full + s, 1);
            mbar_init(v_empty + s, 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kBwdMmaWarp) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    if (warp == kBwdTmaWarp && lane == 0) {
        prefetch_tensormap(&map_q);
        prefetch_tensormap(&map_k);
        prefetch_tensormap(&map_v);
        prefetch_tensormap(&map_do);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kBwdTmaWarp) {
        if (lane == 0) {
            uint8_t *fix = smem + L::kFixOff, *kring = smem + L::kKOff, *vring = smem + L::kVOff;
            const uint64_t pol = l2_policy_evict_last();
            bool ok = true;
            int nfix = 0, nk = 0, nv = 0;  // Q/dO, K and V tiles issued
            DqUnit u;
            for (int k = 0; ok && dq_unit(p, k, u); ++k) {
                // Q and dO of the unit before must have been read by its last products
                if (k > 0 && !mbar_wait(fix_empty, (k - 1) & 1, abort_flag, kWatchdogNs)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(fix_full, 2 * L::kTileBytes);
                for (int c = 0; c < L::kChunks; ++c) {
                    tma_load_3d(fix + c * kSlabBytes, &map_q, fix_full, c * 64, u.it * kRows, u.bh, pol);
                    tma_load_3d(fix + L::kTileBytes + c * kSlabBytes, &map_do, fix_full, c * 64, u.it * kRows,
                                u.bh, pol);
                }
                ++nfix;
                for (int n = 0; n < u.n_iter; ++n) {
                    const int ks = nk % L::kKStages;
                    if (nk >= L::kKStages &&
                        !mbar_wait(k_empty + ks, ((nk / L::kKStages) - 1) & 1, abort_flag, kWatchdogNs)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(k_full + ks, L::kTileBytes);
                    for (int c = 0; c < L::kChunks; ++c)
                        tma_load_3d(kring + ks * L::kTileBytes + c * kSlabBytes, &map_k, k_full + ks, c * 64,
                                    n * kRows, u.bhk, pol);
                    ++nk;
                    const int vs = nv % L::kVStages;
                    if (nv >= L::kVStages &&
                        !mbar_wait(v_empty + vs, ((nv / L::kVStages) - 1) & 1, abort_flag, kWatchdogNs)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(v_full + vs, L::kTileBytes);
                    for (int c = 0; c < L::kChunks; ++c)
                        tma_load_3d(vring + vs * L::kTileBytes + c * kSlabBytes, &map_v, v_full + vs, c * 64,
                                    n * kRows, u.bhk, pol);
                    ++nv;
                }
            }
            if (!ok) {  // let every copy already issued land (only the last Q/dO can be in flight)
                constexpr uint64_t kDrainNs = 200ull * 1000ull * 1000ull;
                int dummy = 0;
                if (nfix > 0) mbar_wait(fix_full, (nfix - 1) & 1, &dummy, kDrainNs);
                for (int m = (nk > L::kKStages ? nk - L::kKStages : 0); m < nk; ++m)
                    mbar_wait(k_full + (m % L::kKStages), (m / L::kKStages) & 1, &dummy, kDrainNs);
                for (int m = (nv > L::kVStages ? nv - L::kVStages : 0); m < nv; ++m)
                    mbar_wait(v_full + (m % L::kVStages), (m / L::kVStages) & 1, &dummy, kDrainNs);
            }
        }
        __syncwarp();
    } else if (warp == kBwdMmaWarp) {
        if (lane == 0) {
            const uint32_t idesc_s = idesc_f16(BF16, kRows, kRows, false, false);
            const uint32_t idesc_acc = idesc_f16(BF16, kRows, D, false, true);
            const uint32_t fix = smem_u32(smem + L::kFixOff);
            const uint32_t kring = smem_u32(smem + L::kKOff), vring = smem_u32(smem + L::kVOff);
            const uint64_t q_desc = sdesc_sw128(fix, 16, 1024);
            const uint64_t do_desc = sdesc_sw128(fix + L::kTileBytes, 16, 1024);
            // S = Q K_j^T and dP = dO V_j^T (queries on TMEM lanes) for the CTA's key tile j
            auto issue_scores = [&](int j) {
                const int ks = j % L::kKStages, vs = j % L::kVStages;
                if (!mbar_wait(k_full + ks, (j / L::kKStages) & 1, abort_flag, kWatchdogNs)) return false;
                if (!mbar_wait(v_full + vs, (j / L::kVStages) & 1, abort_flag, kWatchdogNs)) return false;
                tc_fence_after();
                issue_qk<D>(tmem + L::kXCol, q_desc, sdesc_sw128(kring + ks * L::kTileBytes, 16, 1024), idesc_s);
                issue_qk<D>(tmem + L::kYCol, do_desc, sdesc_sw128(vring + vs * L::kTileBytes, 16, 1024), idesc_s);
                umma_commit(s_full);
                umma_commit(v_empty + vs);  // V_j is read by dP alone
                return true;
            };
            bool ok = true;
            int g = 0;
            DqUnit u;
            for (int k = 0; ok && dq_unit(p, k, u); ++k) {
                if (!mbar_wait(fix_full, k & 1, abort_flag, kWatchdogNs)) { ok = false; break; }
                tc_fence_after();
                // The unit's first scores overwrite the last unit's S and dP: every
                // warp holds those (implied by its P-ready arrival, awaited below).
                if (g > 0) {
                    if (!mbar_wait(s_loaded, (g - 1) & 1, abort_flag, kWatchdogNs)) { ok = false; break; }
                    tc_fence_after();
                }
                if (!issue_scores(g)) { ok = false; break; }
                if (u.n_iter == 1) umma_commit(fix_empty);
                for (int n = 0; n < u.n_iter && ok; ++n) {
                    const int gi = g + n;
                    // Once every elementwise warp holds S and dP of tile gi in
                    // registers, the next tile's products run under their work.
                    if (n + 1 < u.n_iter) {
                        if (!mbar_wait(s_loaded, gi & 1, abort_flag, kWatchdogNs)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        if (!issue_scores(gi + 1)) {
                            ok = false;
                            break;
                        }
                        // the unit's last reads of Q and dO are issued: free them once done
                        if (n + 2 == u.n_iter) umma_commit(fix_empty);
                    }
                    if (!mbar_wait(p_ready, gi & 1, abort_flag, kWatchdogNs)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // dQ += dS K_n (dS from its TMEM columns; K_n MN-major)
                    const int ks = gi % L::kKStages;
                    issue_pv<D>(tmem + L::kACol, tmem + L::kDsCol, sdesc_sw128(kring + ks * L::kTileBytes, kSlabBytes, 1024),
                                idesc_acc, n > 0);
                    umma_commit(k_empty + ks);
                    umma_commit(dq_done);
                }
                if (!ok) break;
                umma_commit(acc_done);
                g += u.n_iter;
            }
            umma_commit(drain);
            int dummy = 0;
            mbar_wait(drain, 0, &dummy, kWatchdogNs);
        }
        __syncwarp();
    } else {
        const int wq = warp & 3, hf = warp >> 2;  // TMEM lane quadrant; column half
        const int r = wq * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
        // D and L2 are written by prep, two grids back: wait for the grids before
        // this one (launched early beside the dK/dV pass) to finish.
        asm volatile("griddepcontrol.wait;" ::: "memory");
        bool ok = true;
        int g = 0;
        DqUnit u;
        for (int k = 0; ok && dq_unit(p, k, u); ++k) {
            const int qrow = u.it * kRows + r;
            // the vectors are padded to whole tiles per head; dQ rows are not
            const size_t vi = static_cast<size_t>(u.bh) * p.npad + qrow;
            const size_t li = static_cast<size_t>(u.bh) * p.N + qrow;
            const float nl2_r = qrow < p.N ? p.lse2[vi] : 0.f;
            const float nd_r = qrow < p.N ? p.dsum[vi] : 0.f;
            for (int n = 0; n < u.n_iter && ok; ++n) {
                const int gi = g + n;
                if (!warp_wait(s_full, gi & 1, abort_flag)) { ok = false; break; }
                tc_fence_after();
                uint32_t sr[2][32], dr[2][32];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    tmem_ld32(tmem + lane_off + L::kXCol + (2 * hf + h) * 32, sr[h]);
                    tmem_ld32(tmem + lane_off + L::kYCol + (2 * hf + h) * 32, dr[h]);
                }
                tmem_ld_wait();
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    reg_fence32(sr[h]);
                    reg_fence32(dr[h]);
                }
                // S and dP are in registers: the MMA thread may overwrite them
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(s_loaded);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int q = 2 * hf + h;
                    // column col is key n * 128 + 32 q + col: visible when it exists, the
                    // row exists and, causally, key <= query
                    const int kb = n * kRows + q * 32;
                    uint32_t vis = 0xffffffffu;
                    if (kb + 32 > p.N) vis = p.N > kb ? (0xffffffffu >> (32 - (p.N - kb))) : 0u;
                    if (qrow >= p.N) vis = 0u;
                    if (p.causal) {
                        const int hi = qrow - kb;  // last visible column
                        vis &= hi < 0 ? 0u : (hi >= 31 ? 0xffffffffu : (0xffffffffu >> (31 - hi)));
                    }
                    uint32_t pk[16], dk[16];
                    weights_quarter<BF16, false>(sr[h], dr[h], pk, dk, p.c, nullptr, nullptr, nl2_r, nd_r, vis);
                    if (h == 0 && gi > 0) {
                        // dS of the CTA's previous key tile must have been read by its
                        // product.  This also keeps p_ready from completing twice before
                        // the MMA thread, which committed dq_done after seeing the
                        // previous p_ready, looks.
                        if (!warp_wait(dq_done, (gi - 1) & 1, abort_flag)) { ok = false; break; }
                        tc_fence_after();
                    }
                    tmem_st16(tmem + lane_off + L::kDsCol + q * 16, dk);
                }
                if (!ok) break;
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(p_ready);
            }
            if (!ok || !warp_wait(acc_done, k & 1, abort_flag)) {
                ok = false;
                break;
            }
            // each half stores half of the dQ columns; the next unit's first
            // product (which overwrites the accumulator) waits for this warp's next
            // P-ready arrival, after these loads
            tc_fence_after();
            const int osize = p.grad_dtype == FA_F32 ? 4 : 2;
            const size_t row_off = li * D * osize;
#pragma unroll
            for (int q = 0; q < D / 64; ++q) {
                const int cq = hf * (D / 64) + q;
                uint32_t o[32];
                tmem_ld32(tmem + lane_off + L::kACol + cq * 32, o);
                tmem_ld_wait();
                reg_fence32(o);
                if (qrow < p.N)
                    store_out32(static_cast<uint8_t *>(p.g0) + row_off + cq * 32 * osize, o, p.scale,
                                p.grad_dtype);
            }
            tc_fence_before();
            g += u.n_iter;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kBwdMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    if (threadIdx.x == 0 && *abort_flag) atomicCAS(&g_backward_status, 0, (int)FA_ERR_WATCHDOG);
}

// ---------------------------------------------------------------- dQ from stored dS
// dQ_i = scale sum_j dS_ij K_j, with the dS blocks the dK/dV pass wrote: a
// pipelined product, no recomputation of S and dP.  Warps 0-3 epilogue (thread =
// TMEM lane = query row), warp 4 copy producer, warp 5 MMA issuer.  Each ring
// stage holds the dS block (j, i), copied whole by one bulk copy, and K_j
// [128 keys][d] by TMA.  Both are MN-major operands: A = dS (queries along M) in
// the unswizzled core-matrix layout, 256 bytes per 16 keys; B = K_j with d
// contiguous, 128-byte swizzled, 2 KB per 16 keys.  Two TMEM accumulators let the
// epilogue of one unit run under the next unit's products.  Units are the dQ
// pass's (query head, query tile), dealt in the same snake order.
template <int D>
struct DqgLayout {
    static constexpr int kChunks = D / 64;
    static constexpr int kDsBytes = kDsBlockBytes;             // 128 keys x 128 queries
    static constexpr int kKBytes = kChunks * kSlabBytes;       // 128 keys x D
    static constexpr int kStageBytes = kDsBytes + kKBytes;
    static constexpr int kStages = D == 128 ? 3 : 4;
    static constexpr int kBarOff = kStages * kStageBytes;
    // full[S], empty[S], acc_full[2], acc_free[2], drain
    static constexpr int kNumBars = 2 * kStages + 5;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    static constexpr int kSmemBytes = kMiscOff + 16 + 1024;
    static constexpr uint32_t kTmemCols = 256;                 // two accumulators of D columns
};
constexpr int kDqgThreads = 192;
constexpr int kDqgTmaWarp = 4;
constexpr int kDqgMmaWarp = 5;

// O (+)= A B over 128 keys with both operands MN-major in shared memory: eight
// products of 16 keys, each 256 bytes further on in A (16 in the descriptor's
// address field) and 2 KB in B (128).
#define FA_MMA_SS_MN(OA, OB)                                                  \
    "add.u32 xa, %1, " #OA ";\n\t"                                          \
    "add.u32 xb, %3, " #OB ";\n\t"                                          \
    "mov.b64 a, {xa, %2};\n\t"                                              \
    "mov.b64 b, {xb, %4};\n\t"                                              \
    "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %5, pt;\n\t"

__device__ __forceinline__ void issue_ss_mn(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            bool accumulate) {
    const uint32_t alo = static_cast<uint32_t>(a_desc), ahi = static_cast<uint32_t>(a_desc >> 32);
    const uint32_t blo = static_cast<uint32_t>(b_desc), bhi = static_cast<uint32_t>(b_desc >> 32);
    asm volatile(
        "{\n\t.reg .pred pf, pt;\n\t.reg .b64 a, b;\n\t.reg .b32 xa, xb;\n\t"
        "setp.ne.b32 pf, %6, 0;\n\t"
        "setp.eq.b32 pt, %6, %6;\n\t"
        "mov.b64 a, {%1, %2};\n\t"
        "mov.b64 b, {%3, %4};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %5, pf;\n\t"
        FA_MMA_SS_MN(16, 128) FA_MMA_SS_MN(32, 256) FA_MMA_SS_MN(48, 384) FA_MMA_SS_MN(64, 512)
        FA_MMA_SS_MN(80, 640) FA_MMA_SS_MN(96, 768) FA_MMA_SS_MN(112, 896)
        "}" ::"r"(d_tmem), "r"(alo), "r"(ahi), "r"(blo), "r"(bhi), "r"(idesc), "r"(accumulate ? 1u : 0u)
        : "memory");
}
#undef FA_MMA_SS_MN

template <int D, bool BF16>
__global__ void __launch_bounds__(kDqgThreads, 1)
    bwd_dq_gemm_kernel(const __grid_constant__ CUtensorMap map_k, const BwdParams p) {
    using L = DqgLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBarOff);
    uint64_t *full = bars, *empty = bars + L::kStages;
    uint64_t *acc_full = bars + 2 * L::kStages, *acc_free = acc_full + 2, *drain = acc_full + 4;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kMiscOff);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kMiscOff + 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < L::kStages; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(acc_full + b, 1);
            mbar_init(acc_free + b, 4);  // one arrival per epilogue warp
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kDqgMmaWarp) {
        tmem_alloc(tmem_slot, L::kTmemCols);
        tmem_relinquish();
    }
    if (warp == kDqgTmaWarp && lane == 0) prefetch_tensormap(&map_k);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kDqgTmaWarp) {
        if (lane == 0) {
            // dS is read once; K_j by every query tile of the head
            const uint64_t pol = l2_policy_evict_last(), pol_ds = l2_policy_evict_first();
            bool ok = true;
            int ni = 0;  // stages issued
            // dS comes from the dK/dV grid this one may have started beside
            asm volatile("griddepcontrol.wait;" ::: "memory");
            DqUnit u;
            for (int k = 0; ok && dq_unit(p, k, u); ++k) {
                for (int j = 0; j < u.n_iter; ++j) {
                    const int slot = ni % L::kStages;
                    if (ni >= L::kStages &&
                        !mbar_wait(empty + slot, ((ni / L::kStages) - 1) & 1, abort_flag, kWatchdogNs)) {
                        ok = false;
                        break;
                    }
                    uint8_t *st = smem + slot * L::kStageBytes;
                    mbar_arrive_expect_tx(full + slot, L::kStageBytes);
                    bulk_load_hint(st, ds_block(p, u.bh, j, u.it), kDsBlockBytes, full + slot, pol_ds);
                    for (int c = 0; c < L::kChunks; ++c)
                        tma_load_3d(st + L::kDsBytes + c * kSlabBytes, &map_k, full + slot, c * 64, j * kRows,
                                    u.bhk, pol);
                    ++ni;
                }
            }
            if (!ok) {  // let every copy already issued land
                constexpr uint64_t kDrainNs = 200ull * 1000ull * 1000ull;
                int dummy = 0;
                for (int m = (ni > L::kStages ? ni - L::kStages : 0); m < ni; ++m)
                    mbar_wait(full + (m % L::kStages), (m / L::kStages) & 1, &dummy, kDrainNs);
            }
        }
        __syncwarp();
    } else if (warp == kDqgMmaWarp) {
        if (lane == 0) {
            const uint32_t idesc = idesc_f16(BF16, kRows, D, true, true);
            const uint32_t ring = smem_u32(smem);
            bool ok = true;
            int ni = 0;
            DqUnit u;
            for (int k = 0; ok && dq_unit(p, k, u); ++k) {
                const int b = k & 1;
                // this accumulator's last reader: the epilogue of unit k - 2
                if (k >= 2 && !mbar_wait(acc_free + b, ((k - 2) >> 1) & 1, abort_flag, kWatchdogNs)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int j = 0; j < u.n_iter; ++j) {
                    const int slot = ni % L::kStages;
                    if (!mbar_wait(full + slot, (ni / L::kStages) & 1, abort_flag, kWatchdogNs)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t st = ring + slot * L::kStageBytes;
                    issue_ss_mn(tmem + b * D, sdesc_plain(st, kDsCoreBytes, kDsGroupBytes),
                                sdesc_sw128(st + L::kDsBytes, kSlabBytes, 1024), idesc, j > 0);
                    umma_commit(empty + slot);
                    ++ni;
                }
                if (!ok) break;
                umma_commit(acc_full + b);
            }
            umma_commit(drain);
            int dummy = 0;
            mbar_wait(drain, 0, &dummy, kWatchdogNs);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------------- epilogue
        const int r = warp * 32 + lane;  // warps 0-3: TMEM lane quadrant = warp
        const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
        const int osize = p.grad_dtype == FA_F32 ? 4 : 2;
        DqUnit u;
        for (int k = 0; dq_unit(p, k, u); ++k) {
            const int b = k & 1;
            if (!warp_wait(acc_full + b, (k >> 1) & 1, abort_flag)) break;
            tc_fence_after();
            const int qrow = u.it * kRows + r;
            uint8_t *dst = static_cast<uint8_t *>(p.g0) + (static_cast<size_t>(u.bh) * p.N + qrow) * D * osize;
#pragma unroll
            for (int q = 0; q < D / 32; ++q) {
                uint32_t o[32];
                tmem_ld32(tmem + lane_off + b * D + q * 32, o);
                tmem_ld_wait();
                reg_fence32(o);
                if (qrow < p.N) store_out32(dst + q * 32 * osize, o, p.scale, p.grad_dtype);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_free + b);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kDqgMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, L::kTmemCols);
    }
    if (threadIdx.x == 0 && *abort_flag) atomicCAS(&g_backward_status, 0, (int)FA_ERR_WATCHDOG);
}

// A backward main kernel, launched so that it may start while the grid before it
// still runs (programmatic dependent launch); it waits for that grid itself where
// it reads what the grid wrote.
template <typename K, typename... Args>
cudaError_t launch_pdl(K kernel, int grid, int threads, size_t smem, cudaStream_t stream, const Args &...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(static_cast<unsigned>(threads));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
    return e == cudaSuccess ? cudaGetLastError() : e;
}

// The dS table takes at most this much memory; larger problems run in chunks of
// key/value heads that fit.
constexpr size_t kDsWorkspaceMax = 4ull << 30;

template <int D, bool BF16>
int launch_bwd_d(const BackwardLaunch &a, cudaStream_t stream) {
    using L = BwdLayout<D>;
    static_assert(L::kSmemBytes <= 227 * 1024 && DqLayout<D>::kSmemBytes <= 227 * 1024,
                  "shared memory budget");
    const long long BH = static_cast<long long>(a.B) * a.H;      // query heads
    const long long BHk = static_cast<long long>(a.B) * a.Hkv;   // key/value heads
    const int n_t = (a.N + kRows - 1) / kRows;
    const long long rows_pad = BH * n_t * kRows;  // lse2 and dsum, padded to whole tiles
    const int group = a.H / a.Hkv;
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(bwd_dkdv_kernel<D, BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  L::kSmemBytes)) != cudaSuccess ||
        (e = cudaFuncSetAttribute(bwd_dq_kernel<D, BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  DqLayout<D>::kSmemBytes)) != cudaSuccess ||
        (e = cudaFuncSetAttribute(bwd_dq_gemm_kernel<D, BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  DqgLayout<D>::kSmemBytes)) != cudaSuccess)
        return cuda_fail(e);
    void *ws = nullptr;
    if ((e = scratch_alloc(&ws, static_cast<size_t>(rows_pad) * 2 * sizeof(float), stream)) != cudaSuccess) {
        cuda_fail(e);
        return FA_ERR_WORKSPACE;
    }
    float *lse2 = static_cast<float *>(ws), *dsum = lse2 + rows_pad;
    // The dS table for the dQ product pass.  It holds the blocks of `chunk` key/value
    // heads (their chunk x group query heads); a problem whose table would pass the
    // limit runs both passes chunk by chunk over the same table.  Without a table
    // (a flag, no key/value head fits, or no memory) the dQ pass recomputes S and dP.
    long long chunk = BHk;
    void *ds = nullptr;
    const size_t head_bytes = static_cast<size_t>(n_t) * n_t * kDsBlockBytes * group;  // per key/value head
    if (!a.recompute_dq && head_bytes <= kDsWorkspaceMax) {
        const long long fit = static_cast<long long>(kDsWorkspaceMax / head_bytes);
        const long long n_chunks = (BHk + fit - 1) / fit;
        chunk = (BHk + n_chunks - 1) / n_chunks;  // even chunks
        if (scratch_alloc(&ds, static_cast<size_t>(chunk) * head_bytes, stream) != cudaSuccess) {
            cudaGetLastError();  // an allocation failure only selects the recomputing pass
            ds = nullptr;
            chunk = BHk;
        }
    }
    constexpr long long kPrepRowsPerBlock = (kPrepThreads / 32) * (32 / (D / 8)) * kPrepRows;
    bwd_prep_kernel<D, BF16><<<static_cast<unsigned>((rows_pad + kPrepRowsPerBlock - 1) / kPrepRowsPerBlock),
                               kPrepThreads, 0, stream>>>(
        static_cast<const uint16_t *>(a.out), static_cast<const uint16_t *>(a.dout), a.lse, lse2, dsum, rows_pad,
        a.N, n_t * kRows);
    e = cudaGetLastError();
    // The kernels see the (batch, head) pairs as one flat list: query head x of a chunk
    // reads key/value head x / group.
    BwdParams p;
    p.group = group;
    p.N = a.N;
    p.n_t = n_t;
    p.npad = n_t * kRows;
    p.causal = a.causal ? 1 : 0;
    p.grad_dtype = a.grad_dtype;
    p.scale = a.scale;
    p.c = a.scale * 1.4426950408889634f;
    p.ds_t = static_cast<uint16_t *>(ds);
    const size_t in_head = static_cast<size_t>(a.N) * D * 2;                              // bytes of a 16-bit head
    const size_t g_head = static_cast<size_t>(a.N) * D * (a.grad_dtype == FA_F32 ? 4 : 2);  // of a gradient head
    for (long long c0 = 0; c0 < BHk && e == cudaSuccess; c0 += chunk) {
        const long long ck = chunk < BHk - c0 ? chunk : BHk - c0;  // key/value heads of this chunk
        const long long h0 = c0 * group;                             // its first query head
        CUtensorMap mq, mk, mv, mdo;
        int rc;
        if ((rc = make_map(&mq, static_cast<const char *>(a.q) + h0 * in_head, D, false, a.N, ck * group,
                           a.in_bf16)) != FA_OK ||
            (rc = make_map(&mk, static_cast<const char *>(a.k) + c0 * in_head, D, false, a.N, ck, a.in_bf16)) !=
                FA_OK ||
            (rc = make_map(&mv, static_cast<const char *>(a.v) + c0 * in_head, D, false, a.N, ck, a.in_bf16)) !=
                FA_OK ||
            (rc = make_map(&mdo, static_cast<const char *>(a.dout) + h0 * in_head, D, false, a.N, ck * group,
                           a.in_bf16)) != FA_OK) {
            scratch_free(ws, stream);
            if (ds) scratch_free(ds, stream);
            return rc;
        }
        p.lse2 = lse2 + h0 * p.npad;
        p.dsum = dsum + h0 * p.npad;
        // one persistent CTA per SM (or per unit, when there are fewer units)
        p.g0 = static_cast<char *>(a.dk) + c0 * g_head;
        p.g1 = static_cast<char *>(a.dv) + c0 * g_head;
        p.n_units = static_cast<int>(ck * p.n_t);
        int grid = p.n_units < a.num_sms ? p.n_units : a.num_sms;
        e = launch_pdl(bwd_dkdv_kernel<D, BF16>, grid, kBwdThreads, L::kSmemBytes, stream, mq, mk, mv, mdo, p);
        if (e != cudaSuccess) break;
        p.g0 = static_cast<char *>(a.dq) + h0 * g_head;
        p.g1 = nullptr;
        p.n_units = static_cast<int>(ck * group * p.n_t);
        grid = p.n_units < a.num_sms ? p.n_units : a.num_sms;
        if (ds) {
            e = launch_pdl(bwd_dq_gemm_kernel<D, BF16>, grid, kDqgThreads, DqgLayout<D>::kSmemBytes, stream, mk, p);
        } else {
            e = launch_pdl(bwd_dq_kernel<D, BF16>, grid, kBwdThreads, DqLayout<D>::kSmemBytes, stream, mq, mk,
                           mv, mdo, p);
        }
    }
    cudaError_t e2 = scratch_free(ws, stream);
    if (e == cudaSuccess) e = e2;
    if (ds) {
        e2 = scratch_free(ds, stream);
        if (e == cudaSuccess) e = e2;
    }
    if (e != cudaSuccess) return cuda_fail(e);
    return FA_OK;
}

}  // namespace

int launch_backward(const BackwardLaunch &a, cudaStream_t stream) {
    if (a.d == 64) return a.in_bf16 ? launch_bwd_d<64, true>(a, stream) : launch_bwd_d<64, false>(a, stream);
    if (a.d == 128) return a.in_bf16 ? launch_bwd_d<128, true>(a, stream) : launch_bwd_d<128, false>(a, stream);
    return FA_ERR_HEAD_DIM;
}

int read_backward_status(int reset) {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_backward_status, sizeof(int)) != cudaSuccess) return -1;
    if (reset && v) {
        int z = 0;
        if (cudaMemcpyToSymbol(g_backward_status, &z, sizeof(int)) != cudaSuccess) return -1;
    }
    return v;
}

}  // namespace fa
