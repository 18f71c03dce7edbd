// fa_prefill_sm103.cu -- fused attention forward, prefill, for sm_103a.
//
// Method (flash-attention-cuda README, "What is Flash Attention?" and the
// "Kernel design" table; "B200 attention kernel from scratch to near-SOTA in
// 60 diagrams" for the Blackwell setting): the keys and values are streamed
// through on-chip memory one 128-row tile at a time, each query row keeps a
// running maximum m and a running denominator l in fp32, the fp32 output
// accumulator is rescaled when m moves, and the N x N score table never
// reaches HBM.  Tiles wholly above the causal diagonal are never visited.
//
// GB300 mapping (one persistent CTA per SM, 12 warps = 3 warpgroups):
//   warps 0-3  softmax for query tile 0 (thread = row; TMEM lanes 0..127)
//   warps 4-7  softmax for query tile 1
//   warp  8    TMA producer: Q tiles, then K_j / V_j into a shared-memory ring
//   warp  9    tcgen05 MMA issuer (one thread) and TMEM owner
//   warps 10-11 idle
// The softmax warpgroups hold a whole 128-key score row per thread, so they
// take registers from the producer/MMA warpgroup with setmaxnreg.
// TMEM (512 columns): S0 | S1 (128 fp32 columns each) | O0 | O1 (d columns
// each).  P (16-bit) overwrites the first 64 columns of its S tile and feeds
// the PV product straight from TMEM.  The two query tiles ping-pong: while
// the softmax warps of one tile work on exponentials, the tensor core runs
// the other tile's products.
//
// Softmax in the exp2 domain: with c = scale * log2(e), p = 2^(s*c - m_ref).
// Rescaling is lazy: m_ref only moves when the tile maximum exceeds it by more
// than TAU (log2 units), so p <= 2^TAU; O and l share m_ref, so the final O/l
// is unchanged.
#include <algorithm>
#include <type_traits>
#include <cfloat>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fa_internal.h"
#include "fa_tiles.cuh"
#include "sm103_ptx.cuh"

namespace fa {

namespace {

constexpr int kThreads = 384;
// setmaxnreg split: 2 x 128 threads x kRegsSoftmax + 128 x kRegsOther must not
// exceed kThreads x (registers at launch); the host checks the launch count.
constexpr int kRegsSoftmax = 176;
constexpr int kRegsOther = 152;
constexpr int kMinLaunchRegs = (2 * 128 * kRegsSoftmax + 128 * kRegsOther + kThreads - 1) / kThreads;
constexpr int kTmaWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kBlockM = 128;   // query rows per tile
constexpr int kBlockN = 128;   // keys per tile
constexpr int kRowsPerUnit = 2 * kBlockM;
constexpr float kTau = 8.0f;   // lazy-rescale threshold, log2 units
constexpr uint32_t kTmemCols = 512;

__device__ int g_prefill_status = 0;

template <int D>
struct Layout {
    static constexpr int kChunkBytes = kBlockM * 128;  // 128 rows x 64 16-bit columns
    static constexpr int kChunks = D / 64;
    static constexpr int kTileBytes = kChunks * kChunkBytes;
    static constexpr int kStages = 4;  // two key/value groups of two tiles
    static constexpr int kQOff = 0;
    static constexpr int kRingOff = 2 * kTileBytes;
    static constexpr int kBarOff = kRingOff + kStages * kTileBytes;
    // q_full, q_empty, s_full[2], p_full[2], o_done[2], drain, s_free[2], pv_done[2],
    // kv_full[S], kv_empty[S]
    static constexpr int kNumBars = 13 + 2 * kStages;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    static constexpr int kSmemBytes = kMiscOff + 16 + 1024;  // + alignment slack
    static constexpr uint32_t kSCol0 = 0, kSCol1 = 128;
    static constexpr uint32_t kOCol0 = 256, kOCol1 = 256 + D;
    // d = 64 leaves room for P beside S (columns 384..511): the softmax then
    // frees S as soon as it has loaded it, and the next Q K^T overlaps the
    // exponentials.  At d = 128, P overwrites the first 64 columns of S.
    static constexpr bool kSepP = (D == 64);
    static constexpr uint32_t kPCol0 = kSepP ? 256 + 2 * D : kSCol0;
    static constexpr uint32_t kPCol1 = kSepP ? 256 + 2 * D + 64 : kSCol1;
    static_assert(!kSepP || kPCol1 + 64 <= 512, "TMEM columns");
};

constexpr int kMaxPre = 1024;  // stream-K: query blocks per head with a step table

struct Params {
    void *out;
    float *lse;            // optional: natural-log log-sum-exp of every row (dense [B][Hq][Nq],
                           // packed [tokens][Hq]); -inf for a row that sees no key
    // A packed batch (variable lengths) keeps tokens [cu_q[b], cu_q[b+1]) of
    // sequence b in a [tokens][H][d] tensor; a dense batch is [B][H][N][d].
    const int *cu_q;       // packed: [B+1] query-token offsets (device); null when dense
    const int *cu_k;       // packed: [B+1] key-token offsets
    int B, Hq, Hkv, group; // query head h reads key/value head h / group
    int Nq, Nk;            // dense: every sequence's lengths; packed: the maxima
    int total_q, total_k;  // packed: tokens in q and in k/v
    int BH;                // B * Hq
    int n_qb;              // 256-row query blocks per (sequence, query head)
    int n_units;           // BH * n_qb
    int causal;            // bottom-right aligned: query i sees keys j <= i + Nk - Nq
    int no_skip;
    int in_bf16;
    int out_dtype;
    int scale_neg;
    float scale_log2;      // c = scale * log2(e)
    float scale_log2_abs;  // |c|
    // Stream-K (dense batches): the W = BH * HT (unit, key tile) steps are cut
    // into gridDim.x equal contiguous ranges; a unit cut between two CTAs is
    // finished by the fixup kernel from the partials in ws_o / ws_ml.
    int stream_k;
    // Causal unit schedule in one round (the paired instantiation): unit i
    // of a head pairs query tile i with tile T - 1 - i (T = 128-row tiles per
    // sequence), so that no unit holds more than T - i key tiles and its two
    // tiles overlap for the first i + 1.
    int n_tt;              // T
    int HT;                // key-tile steps per (sequence, head) = pre[n_qb]
    long long W;           // BH * HT
    // Non-causal stream-K first deals dp_full whole units to every CTA (unit
    // blockIdx.x + k * gridDim.x); only the steps [sk_s0, W) after them are cut
    // into equal ranges, so fewer units are split.  Causal: dp_full = sk_s0 = 0.
    int dp_full;
    long long sk_s0;
    float *ws_o;           // [gridDim.x][2 slots][256 rows][D]  unnormalised O
    float *ws_ml;          // [gridDim.x][2 slots][256 rows][2]  (m_ref, l)
    // The ordered schedule (packed batches over more than one round of units):
    // the (sequence, query block) classes, most key-tile products first (written
    // by packed_order_kernel just before); unit u is head u % Hq of class
    // order[u / Hq].
    const int *order;
};

// Unit schedules, each its own kernel instantiation so that one's code does not
// touch the others': plain (round robin, causal heaviest query blocks first),
// paired (causal tiles i and T - 1 - i in one unit) and ordered (packed batches,
// heaviest (sequence, block) classes first).
constexpr int kSchedPlain = 0, kSchedPaired = 1, kSchedOrdered = 2;

// Stream-K: key-tile steps of a head before query block qb.  A kernel argument
// of its own, so that only this table is indexed at run time and every field
// of Params stays a plain constant operand.
struct StepTable {
    int pre[kMaxPre + 1];
};

// One piece of work: unit u = (sequence b, query head h, query block) and its
// key tiles [j0, j1).  n0 / n1: key tiles the two 128-row query tiles need
// (0 = none: no rows, or rows that see no key).
struct Work {
    int u, b, h, hk;
    int r0, r1;            // first query rows of the unit's two tiles, within the sequence
    int nq, nk, off;       // the sequence's lengths; off = nk - nq (causal alignment)
    long long qt0, kt0;    // packed: first query / key token of the sequence
    int j0, j1, n0, n1;
};

struct SegCursor {
    long long s, s_end;  // stream-K step range
    int u;               // units taken so far (unit schedule: rounds of gridDim.x units)
};

__device__ __forceinline__ void seg_begin(const Params &p, SegCursor &c) {
    const long long span = p.W - p.sk_s0;
    c.s = p.sk_s0 + static_cast<long long>(blockIdx.x) * span / gridDim.x;
    c.s_end = p.sk_s0 + static_cast<long long>(blockIdx.x + 1) * span / gridDim.x;
    c.u = 0;
}

// Key tiles a 128-row query tile starting at row0 must visit.
__device__ __forceinline__ int kv_tiles(int causal, int no_skip, int nq, int nk, int off, int row0) {
    if (row0 >= nq) return 0;
    const int tk = (nk + kBlockN - 1) / kBlockN;
    if (!causal || no_skip) return tk;
    const int last = min(row0 + kBlockM - 1, nq - 1) + off;
    if (last < 0) return 0;
    return min(tk, last / kBlockN + 1);
}

// Fill sequence fields of w from (b, h).  Packed offsets are clamped into the
// tensors (check_seq reports values that needed it).
__device__ __forceinline__ void load_seq(const Params &p, Work &w) {
    w.hk = w.h / p.group;
    if (p.cu_q) {
        const int q_lo = min(max(__ldg(p.cu_q + w.b), 0), p.total_q);
        const int q_hi = min(max(__ldg(p.cu_q + w.b + 1), q_lo), p.total_q);
        const int k_lo = min(max(__ldg(p.cu_k + w.b), 0), p.total_k);
        const int k_hi = min(max(__ldg(p.cu_k + w.b + 1), k_lo), p.total_k);
        w.qt0 = q_lo;
        w.kt0 = k_lo;
        w.nq = min(q_hi - q_lo, p.Nq);
        w.nk = min(k_hi - k_lo, p.Nk);
    } else {
        w.qt0 = 0;
        w.kt0 = 0;
        w.nq = p.Nq;
        w.nk = p.Nk;
    }
    w.off = w.nk - w.nq;
}

// Packed batch: record FA_ERR_SEQ_LEN when sequence w.b's offsets had to be
// clamped (outside [0, total] or decreasing) or a length exceeds the stated
// maximum.  Run by the producer thread only, for every unit it visits.
__device__ __forceinline__ void check_seq(const Params &p, const Work &w) {
    const int q0 = __ldg(p.cu_q + w.b), q1 = __ldg(p.cu_q + w.b + 1);
    const int k0 = __ldg(p.cu_k + w.b), k1 = __ldg(p.cu_k + w.b + 1);
    const bool bad = q0 < 0 || q1 < q0 || q1 > p.total_q || q1 - q0 > p.Nq || k0 < 0 || k1 < k0 ||
                     k1 > p.total_k || k1 - k0 > p.Nk;
    if (bad) atomicCAS(&g_prefill_status, 0, static_cast<int>(FA_ERR_SEQ_LEN));
}

template <int SCHED>
__device__ __forceinline__ bool seg_next(const Params &p, const StepTable &tab, SegCursor &c,
                                         Work &w) {
    int bh, qb;
    if (p.stream_k && c.u < p.dp_full) {  // a whole unit dealt before the cut ranges
        w.u = blockIdx.x + c.u * gridDim.x;
        ++c.u;
        bh = w.u / p.n_qb;
        qb = w.u % p.n_qb;
        w.j0 = 0;
        w.j1 = -1;
    } else if (p.stream_k) {
        if (c.s >= c.s_end) return false;
        bh = static_cast<int>(c.s / p.HT);
        const int rem = static_cast<int>(c.s - static_cast<long long>(bh) * p.HT);
        int lo = 0, hi = p.n_qb - 1;  // last qb with pre[qb] <= rem
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (tab.pre[mid] <= rem) lo = mid; else hi = mid - 1;
        }
        qb = lo;
        w.j0 = rem - tab.pre[qb];
        const int cost = tab.pre[qb + 1] - tab.pre[qb];
        const long long left = c.s_end - c.s;
        w.j1 = static_cast<int>(left < cost - w.j0 ? w.j0 + left : cost);
        c.s += w.j1 - w.j0;
        w.u = bh * p.n_qb + qb;
    } else {
        // Round k deals units [k G, (k + 1) G); odd rounds in reverse CTA order
        // ("snake"), so a CTA that drew a heavy causal block draws a light one next.
        const int k = c.u++;
        const int r = (k & 1) ? static_cast<int>(gridDim.x) - 1 - static_cast<int>(blockIdx.x)
                              : static_cast<int>(blockIdx.x);
        w.u = k * static_cast<int>(gridDim.x) + r;
        if (w.u >= p.n_units) return false;
        if constexpr (SCHED == kSchedPaired) {  // pair i (tiles i and T - 1 - i); pair 0 holds the most keys
            qb = w.u / p.BH;
            bh = w.u % p.BH;
        } else if constexpr (SCHED == kSchedOrdered) {  // heaviest (sequence, block) classes first
            const int cls = __ldg(p.order + w.u / p.Hq);
            qb = cls % p.n_qb;
            bh = (cls / p.n_qb) * p.Hq + w.u % p.Hq;
        } else if (p.causal) {  // heaviest query blocks first
            qb = p.n_qb - 1 - w.u / p.BH;
            bh = w.u % p.BH;
        } else {         // neighbouring CTAs share a head's K/V in L2
            bh = w.u / p.n_qb;
            qb = w.u % p.n_qb;
        }
        w.j0 = 0;
        w.j1 = -1;
    }
    w.b = bh / p.Hq;
    w.h = bh % p.Hq;
    load_seq(p, w);
    if constexpr (SCHED == kSchedPaired) {  // (dense: every sequence has T tiles)
        const int partner = p.n_tt - 1 - qb;
        w.r0 = qb * kBlockM;
        w.r1 = partner > qb ? partner * kBlockM : w.nq;  // an odd T leaves a middle tile alone
    } else {
        w.r0 = qb * kRowsPerUnit;
        w.r1 = w.r0 + kBlockM;
    }
    w.n0 = kv_tiles(p.causal, p.no_skip, w.nq, w.nk, w.off, w.r0);
    w.n1 = kv_tiles(p.causal, p.no_skip, w.nq, w.nk, w.off, w.r1);
    if (w.j1 < 0) w.j1 = max(w.n0, w.n1);
    return true;
}

// LSE: also write the row log-sum-exp (a separate instantiation, so that the
// plain forward keeps its registers).  SCHED: the unit schedule (kSched*).
template <int D, bool BF16, bool LSE, int SCHED>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap map_q,
                   const __grid_constant__ CUtensorMap map_k,
                   const __grid_constant__ CUtensorMap map_v, const Params p,
                   const __grid_constant__ StepTable tab) {
    using L = Layout<D>;
    constexpr uint32_t kGroups = L::kStages / 2;  // key/value groups of two ring slots
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBarOff);
    uint64_t *q_full = bars + 0;
    uint64_t *q_empty = bars + 1;
    uint64_t *s_full = bars + 2;   // [2]
    uint64_t *p_full = bars + 4;   // [2]
    uint64_t *o_done = bars + 6;   // [2]
    uint64_t *drain = bars + 8;
    uint64_t *s_free = bars + 9;    // [2] (separate-P mode)
    uint64_t *pv_done = bars + 11;  // [2] (separate-P mode)
    uint64_t *kv_full = bars + 13;
    uint64_t *kv_empty = bars + 13 + L::kStages;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kMiscOff);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kMiscOff + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        for (int t = 0; t < 2; ++t) {
            mbar_init(s_full + t, 1);
            mbar_init(p_full + t, 4);  // one arrival per softmax warp
            mbar_init(o_done + t, 1);
            mbar_init(s_free + t, 4);  // one arrival per softmax warp
            mbar_init(pv_done + t, 1);
        }
        mbar_init(drain, 1);
        for (int s = 0; s < L::kStages; ++s) {
            mbar_init(kv_full + s, 1);
            mbar_init(kv_empty + s, 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    if (warp == kTmaWarp && lane == 0) {
        prefetch_tensormap(&map_q);
        prefetch_tensormap(&map_k);
        prefetch_tensormap(&map_v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kTmaWarp) {
        // ------------------------------------------------------------ producer
        regs_shrink<kRegsOther>();
        if (lane == 0) {
            const uint64_t pol_kv = l2_policy_evict_last();
            const uint64_t pol_q = l2_policy_evict_first();
            uint8_t *q_smem = smem + L::kQOff;
            uint8_t *ring = smem + L::kRingOff;
            uint32_t qc = 0, gc = 0;
            bool ok = true;
            SegCursor cur;
            seg_begin(p, cur);
            Work w;
            const bool packed = p.cu_q != nullptr;
            // Key/value tiles travel in groups, one per MMA step: {K_j0}, then
            // {V_j, K_j+1} for every step j, the last {V_j1-1}.  A group takes one
            // two-slot stage of the ring and one full/empty barrier pair.
            auto open_group = [&](uint32_t bytes) {
                const uint32_t st = gc % kGroups;
                if (gc >= kGroups &&
                    !mbar_wait(kv_empty + st, ((gc / kGroups) - 1) & 1, abort_flag, kWatchdogNs))
                    return -1;
                mbar_arrive_expect_tx(kv_full + st, bytes);
                return static_cast<int>(st);
            };
            auto load_tile = [&](int st, int half, bool is_v, int j) {
                uint8_t *dst = ring + (2 * st + half) * L::kTileBytes;
                const CUtensorMap *m = is_v ? &map_v : &map_k;
                for (int c = 0; c < L::kChunks; ++c) {
                    if (packed)
                        tma_load_3d(dst + c * L::kChunkBytes, m, kv_full + st, c * 64, w.hk,
                                    static_cast<int>(w.kt0 + j * kBlockN), pol_kv);
                    else
                        tma_load_3d(dst + c * L::kChunkBytes, m, kv_full + st, c * 64, j * kBlockN,
                                    w.b * p.Hkv + w.hk, pol_kv);
                }
            };
            while (ok && seg_next<SCHED>(p, tab, cur, w)) {
                if (packed) check_seq(p, w);
                if (w.j1 <= w.j0) continue;  // no key tiles: the softmax warps write zeros
                // query tile t is loaded when it has key tiles in [j0, j1)
                const bool need0 = min(w.n0, w.j1) > w.j0, need1 = min(w.n1, w.j1) > w.j0;
                if (qc > 0 && !mbar_wait(q_empty, (qc - 1) & 1, abort_flag, kWatchdogNs)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(q_full, ((need0 ? 1 : 0) + (need1 ? 1 : 0)) * L::kTileBytes);
                for (int t = 0; t < 2; ++t) {
                    if (!(t ? need1 : need0)) continue;
                    const int row = t ? w.r1 : w.r0;
                    for (int c = 0; c < L::kChunks; ++c) {
                        if (packed)
                            tma_load_3d(q_smem + t * L::kTileBytes + c * L::kChunkBytes, &map_q, q_full,
                                        c * 64, w.h, static_cast<int>(w.qt0 + row), pol_q);
                        else
                            tma_load_3d(q_smem + t * L::kTileBytes + c * L::kChunkBytes, &map_q, q_full,
                                        c * 64, row, w.b * p.Hq + w.h, pol_q);
                    }
                }
                ++qc;
                int st = open_group(L::kTileBytes);
                if (st < 0) { ok = false; break; }
                load_tile(st, 0, false, w.j0);
                ++gc;
                for (int j = w.j0; j < w.j1; ++j) {
                    const bool next_k = j + 1 < w.j1;
                    st = open_group((next_k ? 2 : 1) * L::kTileBytes);
                    if (st < 0) { ok = false; break; }
                    load_tile(st, 0, true, j);
                    if (next_k) load_tile(st, 1, false, j + 1);
                    ++gc;
                }
            }
            if (!ok) {
                // Let every copy already issued land before the CTA goes away.
                constexpr uint64_t kDrainNs = 200ull * 1000ull * 1000ull;
                int dummy = 0;
                if (qc > 0) mbar_wait(q_full, (qc - 1) & 1, &dummy, kDrainNs);
                for (uint32_t i = (gc > (uint32_t)kGroups ? gc - kGroups : 0); i < gc; ++i)
                    mbar_wait(kv_full + (i % kGroups), (i / kGroups) & 1, &dummy, kDrainNs);
            }
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        regs_shrink<kRegsOther>();
        if (lane == 0) {
            const uint32_t idesc_qk = idesc_f16(BF16, kBlockM, kBlockN, false, false);
            const uint32_t idesc_pv = idesc_f16(BF16, kBlockM, D, false, true);
            const uint32_t q_addr = smem_u32(smem + L::kQOff);
            const uint64_t q_desc0 = sdesc_sw128(q_addr, 16, 1024);
            const uint64_t q_desc1 = sdesc_sw128(q_addr + L::kTileBytes, 16, 1024);
            const uint32_t ring_addr = smem_u32(smem + L::kRingOff);
            // Descriptors of every ring stage, built once: a step picks its stage
            // at compile time (below), so no descriptor is computed in the loop.
            // stage st: slot 2 st holds V_j (or K_j0 of a unit's first group), slot
            // 2 st + 1 holds K_j+1.
            uint64_t vdesc[kGroups], kdesc[kGroups], k0desc[kGroups];
#pragma unroll
            for (int g = 0; g < (int)kGroups; ++g) {
                const uint32_t a = ring_addr + 2 * g * L::kTileBytes;
                vdesc[g] = sdesc_sw128(a, L::kChunkBytes, 1024);
                kdesc[g] = sdesc_sw128(a + L::kTileBytes, 16, 1024);
                k0desc[g] = sdesc_sw128(a, 16, 1024);
            }
            const uint32_t s_tmem0 = tmem + L::kSCol0, s_tmem1 = tmem + L::kSCol1;
            const uint32_t o_tmem0 = tmem + L::kOCol0, o_tmem1 = tmem + L::kOCol1;
            const uint32_t p_tmem0 = tmem + L::kPCol0, p_tmem1 = tmem + L::kPCol1;
            uint32_t qc = 0, gc = 0, pc0 = 0, pc1 = 0;
            uint32_t qk0 = 0, qk1 = 0;  // Q K^T products issued per tile (separate-P mode)
            bool ok = true;
            SegCursor cur;
            seg_begin(p, cur);
            Work w;
            // the next key/value group in shared memory: its ring stage.  Within a
            // step the tcgen05 fence after the first P (or S-free) wait also covers it.
            auto take_group = [&](bool fence) {
                const uint32_t st = gc % kGroups;
                if (!mbar_wait(kv_full + st, (gc / kGroups) & 1, abort_flag, kWatchdogNs)) return -1;
                if (fence) tc_fence_after();
                return static_cast<int>(st);
            };
            while (ok && seg_next<SCHED>(p, tab, cur, w)) {
                const int j0 = w.j0, j1 = w.j1;
                if (j1 <= j0) continue;  // no key tiles: nothing to multiply
                // key tiles [j0, e_t) for query tile t (empty when e_t <= j0)
                const int n0 = min(w.n0, j1), n1 = min(w.n1, j1);
                if (!mbar_wait(q_full, qc & 1, abort_flag, kWatchdogNs)) { ok = false; break; }
                ++qc;
                tc_fence_after();
                {   // S_t = Q_t K_j0^T from the group {K_j0}
                    const int st = take_group(true);
                    if (st < 0) { ok = false; break; }
                    uint64_t k_desc = k0desc[0];
#pragma unroll
                    for (int g = 1; g < (int)kGroups; ++g)
                        if (st == g) k_desc = k0desc[g];
                    if constexpr (L::kSepP) {
                        // S_t is free once the softmax has loaded the previous one
                        if (n0 > j0) {
                            if (qk0 > 0 && !mbar_wait(s_free + 0, (qk0 - 1) & 1, abort_flag, kWatchdogNs)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            issue_qk<D>(s_tmem0, q_desc0, k_desc, idesc_qk);
                            umma_commit(s_full + 0);
                            ++qk0;
                        }
                        if (n1 > j0) {
                            if (qk1 > 0 && !mbar_wait(s_free + 1, (qk1 - 1) & 1, abort_flag, kWatchdogNs)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            issue_qk<D>(s_tmem1, q_desc1, k_desc, idesc_qk);
                            umma_commit(s_full + 1);
                            ++qk1;
                        }
                    } else {
                        if (n0 > j0) {
                            issue_qk<D>(s_tmem0, q_desc0, k_desc, idesc_qk);
                            umma_commit(s_full + 0);
                        }
                        if (n1 > j0) {
                            issue_qk<D>(s_tmem1, q_desc1, k_desc, idesc_qk);
                            umma_commit(s_full + 1);
                        }
                    }
                    umma_commit(kv_empty + st);
                    ++gc;
                    if (j1 - j0 == 1) umma_commit(q_empty);
                }
                for (int j = j0; j < j1 && ok; ++j) {
                    // the group {V_j, K_j+1} (the last step's group holds V_j alone)
                    const int st = take_group(false);
                    if (st < 0) { ok = false; break; }
                    // the step's body, instantiated per ring stage (a compile-time constant)
                    auto step = [&](auto stage) {
                    constexpr int ST = decltype(stage)::value;
                    const uint64_t v_desc = vdesc[ST];
                    const uint64_t k_desc = kdesc[ST];
                    // One query tile's step: wait for P_t, O_t (+)= P_t V_j, then
                    // S_t = Q_t K_{j+1}^T (issued after the PV product that reads P_t).
                    auto tile_step = [&](int nt, uint64_t *pf, uint32_t &pc, uint32_t s_t,
                                         uint32_t o_t, uint64_t q_desc, uint64_t *sf, uint64_t *od) {
                        if (j >= nt) return true;
                        // polled, not suspended: the product should start the moment P is in
                        if (!mbar_spin(pf, pc & 1, abort_flag, kWatchdogNs)) return false;
                        ++pc;
                        tc_fence_after();
                        issue_pv<D>(o_t, s_t, v_desc, idesc_pv, j > j0);
                        if (j == nt - 1) umma_commit(od);
                        if (j + 1 < nt) {
                            issue_qk<D>(s_t, q_desc, k_desc, idesc_qk);
                            umma_commit(sf);
                        }
                        return true;
                    };
                    // Separate-P step: S_t = Q_t K_{j+1}^T as soon as the softmax has
                    // loaded S_t(j), then O_t (+)= P_t V_j once P_t(j) is written.  Both
                    // tiles' Q K^T products go first, so neither tile's next scores wait
                    // behind the other tile's P.
                    auto sep_qk = [&](int nt, uint64_t *sfree, uint32_t &qk, uint32_t s_t, uint64_t q_desc,
                                      uint64_t *sf) {
                        if (j + 1 >= nt) return true;
                        if (!mbar_spin(sfree, (qk - 1) & 1, abort_flag, kWatchdogNs)) return false;
                        tc_fence_after();
                        issue_qk<D>(s_t, q_desc, k_desc, idesc_qk);
                        umma_commit(sf);
                        ++qk;
                        return true;
                    };
                    auto sep_pv = [&](int nt, uint64_t *pf, uint32_t &pc, uint32_t p_t, uint32_t o_t,
                                      uint64_t *pvd) {
                        if (j >= nt) return true;
                        if (!mbar_spin(pf, pc & 1, abort_flag, kWatchdogNs)) return false;
                        ++pc;
                        tc_fence_after();
                        issue_pv<D>(o_t, p_t, v_desc, idesc_pv, j > j0);
                        umma_commit(pvd);
                        return true;
                    };
                    if constexpr (L::kSepP) {
                        ok = sep_qk(n0, s_free + 0, qk0, s_tmem0, q_desc0, s_full + 0) &&
                             sep_qk(n1, s_free + 1, qk1, s_tmem1, q_desc1, s_full + 1) &&
                             sep_pv(n0, p_full + 0, pc0, p_tmem0, o_tmem0, pv_done + 0) &&
                             sep_pv(n1, p_full + 1, pc1, p_tmem1, o_tmem1, pv_done + 1);
                    } else {
                        ok = tile_step(n0, p_full + 0, pc0, s_tmem0, o_tmem0, q_desc0, s_full + 0,
                                       o_done + 0) &&
                             tile_step(n1, p_full + 1, pc1, s_tmem1, o_tmem1, q_desc1, s_full + 1,
                                       o_done + 1);
                    }
                    if (ok) umma_commit(kv_empty + ST);
                    };
                    static_assert(kGroups == 2, "two ring stages");
                    if (st == 0) step(std::integral_constant<int, 0>{});
                    else if (st == 1) step(std::integral_constant<int, 1>{});
                    if (!ok) break;
                    ++gc;
                    if (j + 1 == j1 - 1) umma_commit(q_empty);
                }
            }
            // Nothing may still be running on the tensor core at teardown.
            umma_commit(drain);
            int dummy = 0;
            mbar_wait(drain, 0, &dummy, kWatchdogNs);
        }
        __syncwarp();
    } else if (warp < 8) {
        // ------------------------------------------------------------ softmax
        regs_grow<kRegsSoftmax>();
        const int t = warp >> 2;
        const int wq = warp & 3;
        const int r = wq * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
        const uint32_t s_addr = tmem + lane_off + (t ? L::kSCol1 : L::kSCol0);
        const uint32_t o_addr = tmem + lane_off + (t ? L::kOCol1 : L::kOCol0);
        const uint32_t p_addr = tmem + lane_off + (t ? L::kPCol1 : L::kPCol0);
        const float cexp = p.scale_log2;
        const int osize = p.out_dtype == FA_F32 ? 4 : 2;
        uint32_t sc = 0, oc = 0, pvc = 0;
        bool ok = true;
        SegCursor cur;
        seg_begin(p, cur);
        Work w;
        for (int seg = 0; ok && seg_next<SCHED>(p, tab, cur, w); ++seg) {
            const int j0 = w.j0, j1 = w.j1;
            const int tile_row0 = t ? w.r1 : w.r0;
            const int row = tile_row0 + r;  // query index within the sequence
            // Output row: dense [B][Hq][Nq][d], packed [tokens][Hq][d].
            uint8_t *const orow = reinterpret_cast<uint8_t *>(p.out) +
                                  (p.cu_q ? ((w.qt0 + row) * p.Hq + w.h) * D
                                          : ((static_cast<long long>(w.b) * p.Hq + w.h) * p.Nq + row) * D) *
                                      osize;
            const bool row_ok = row < w.nq;
            // A stream-K piece of a unit keeps its partial state for the fixup.
            const bool partial = p.stream_k && !(j0 == 0 && j1 == max(w.n0, w.n1));
            const int ntile = min(t ? w.n1 : w.n0, j1);  // this tile's key tiles: [j0, ntile)
            if (ntile <= j0) {
                // Rows that see no key at all are zero rows.  (A stream-K piece
                // that only lacks this tile's keys leaves it to the other pieces.)
                if (!p.stream_k && row_ok) {
                    const uint32_t zero[32] = {};
#pragma unroll
                    for (int q = 0; q < D / 32; ++q) store_out32(orow + q * 32 * osize, zero, 0.f, p.out_dtype);
                }
                continue;
            }
            // last visible key of this row (< 0: none)
            const int lim = p.causal ? min(row + w.off, w.nk - 1) : w.nk - 1;
            float m_ref = -INFINITY;
            // -m_ref once a key has been seen; 0 before, so that the masked
            // scores of a row with nothing visible yet still map to exactly 0
            float neg_m = 0.f;
            float l = 0.f;
            for (int j = j0; j < ntile; ++j) {
                if (!warp_wait(s_full + t, sc & 1, abort_flag)) { ok = false; break; }
                ++sc;
                tc_fence_after();
                uint32_t sr[4][32];
#pragma unroll
                for (int q = 0; q < 4; ++q) tmem_ld32(s_addr + q * 32, sr[q]);
                tmem_ld_wait();
#pragma unroll
                for (int q = 0; q < 4; ++q) reg_fence32(sr[q]);
                if constexpr (L::kSepP) {
                    // S_t is in registers: the next Q K^T may overwrite it now.
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(s_free + t);
                }

                const int cmax = lim - j * kBlockN;  // columns > cmax are masked
                if (cmax < kBlockN - 1) {
                    // Masked columns get the score that the exponent maps to 0.
                    const uint32_t fill = __float_as_uint(p.scale_neg ? INFINITY : -INFINITY);
#pragma unroll
                    for (int c = 0; c < 128; ++c)
                        sr[c >> 5][c & 31] = c > cmax ? fill : sr[c >> 5][c & 31];
                }
                // m_tile = max_c (s_c * cexp), via max(+-s) * |cexp|
                const float mx = p.scale_neg ? row_max128<true>(sr) : row_max128<false>(sr);
                const float m_tile = (mx == -INFINITY) ? -INFINITY : mx * p.scale_log2_abs;
                __syncwarp();  // the masked branch above may diverge per lane
                const bool need = m_tile > m_ref + kTau;
                float alpha = 1.f;
                if (need) {  // (m_tile is finite here)
                    alpha = ex2_approx(m_ref - m_tile);  // 0 on the first tile
                    l *= alpha;
                    m_ref = m_tile;
                    neg_m = -m_tile;
                }
                const uint64_t c2 = f2_pack(cexp, cexp);
                const uint64_t nm2 = f2_pack(neg_m, neg_m);
                // eight fp32 partial sums: (lo, hi) halves of four pair slots
                float sum_lo[4] = {0.f, 0.f, 0.f, 0.f}, sum_hi[4] = {0.f, 0.f, 0.f, 0.f};
                // P in 32-key quarters: 16 packed registers per TMEM store.  With P
                // over S (d = 128) each quarter is stored as soon as it is made.  With
                // a separate P buffer (d = 64) the whole row is made first and the
                // store alone waits for the previous P V product (the last reader of
                // the buffer), so the exponentials overlap that product.
                uint32_t pk[4][16];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
#pragma unroll
                    for (int c2i = 0; c2i < 16; ++c2i) {
                        const uint64_t x = ffma2(f2_pack(__uint_as_float(sr[q][2 * c2i]),
                                                         __uint_as_float(sr[q][2 * c2i + 1])),
                                                 c2, nm2);
                        pk[q][c2i] = pack2t<BF16>(ex2_approx(f2_lo(x)), ex2_approx(f2_hi(x)));
                        // l sums the same rounded weights the PV product uses,
                        // so a row dominated by one key returns that value row.
                        // Each 16-bit weight is added straight into fp32.
                        add_pair16<BF16>(sum_lo[c2i & 3], sum_hi[c2i & 3], pk[q][c2i]);
                    }
                    if constexpr (!L::kSepP) tmem_st16(p_addr + q * 16, pk[q]);
                }
                if constexpr (L::kSepP) {
                    // P_t(j-1) and O_t must be done with before P_t(j) and a rescale
                    if (j > j0) {
                        if (!warp_wait(pv_done + t, pvc & 1, abort_flag)) { ok = false; break; }
                        ++pvc;
                        tc_fence_after();
                    }
#pragma unroll
                    for (int q = 0; q < 4; ++q) tmem_st16(p_addr + q * 16, pk[q]);
                }
                const uint64_t s01 = fadd2(f2_pack(sum_lo[0], sum_hi[0]), f2_pack(sum_lo[1], sum_hi[1]));
                const uint64_t s23 = fadd2(f2_pack(sum_lo[2], sum_hi[2]), f2_pack(sum_lo[3], sum_hi[3]));
                const uint64_t st = fadd2(s01, s23);
                l += f2_lo(st) + f2_hi(st);
                if (j > j0 && __any_sync(0xffffffffu, need)) {
                    // O rows are complete up to tile j-1: the commit that
                    // signalled S_t(j) also covers the earlier PV product.
                    // Done after P is written so the score registers are free.
#pragma unroll
                    for (int q = 0; q < D / 32; ++q) {
                        uint32_t o[32];
                        tmem_ld32(o_addr + q * 32, o);
                        tmem_ld_wait();
                        reg_fence32(o);
#pragma unroll
                        for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
                        tmem_st32(o_addr + q * 32, o);
                    }
                    tmem_st_wait();
                }
                tmem_st_wait();
                tc_fence_before();
                // Every lane's TMEM stores are ordered before the warp sync;
                // one arrival per warp keeps traffic on the barrier low.
                __syncwarp();
                if (lane == 0) mbar_arrive(p_full + t);
            }
            if (!ok) break;
            // ---- epilogue: O / l -> out
            if constexpr (L::kSepP) {
                if (!warp_wait(pv_done + t, pvc & 1, abort_flag)) { ok = false; break; }
                ++pvc;
            } else {
                if (!warp_wait(o_done + t, oc & 1, abort_flag)) { ok = false; break; }
                ++oc;
            }
            tc_fence_after();
            if (partial) {
                // Part of a unit: keep O unnormalised with its (m_ref, l) for the
                // fixup kernel.  Slot 0 = the CTA's first piece, 1 = its last.
                const size_t rec = (static_cast<size_t>(blockIdx.x) * 2 + (seg == p.dp_full ? 0 : 1)) * kRowsPerUnit +
                                   t * kBlockM + r;
                float *wo = p.ws_o + rec * D;
#pragma unroll
                for (int q = 0; q < D / 32; ++q) {
                    uint32_t o[32];
                    tmem_ld32(o_addr + q * 32, o);
                    tmem_ld_wait();
                    reg_fence32(o);
                    uint4 *d4 = reinterpret_cast<uint4 *>(wo + q * 32);
#pragma unroll
                    for (int v = 0; v < 8; ++v)
                        d4[v] = make_uint4(o[4 * v], o[4 * v + 1], o[4 * v + 2], o[4 * v + 3]);
                }
                p.ws_ml[rec * 2 + 0] = m_ref;
                p.ws_ml[rec * 2 + 1] = l;
                tc_fence_before();
                continue;
            }
            const float inv = l > 0.f ? 1.0f / l : 0.f;  // l = 0: no visible key
#pragma unroll
            for (int q = 0; q < D / 32; ++q) {
                uint32_t o[32];
                tmem_ld32(o_addr + q * 32, o);
                tmem_ld_wait();
                reg_fence32(o);
                if (row_ok) store_out32(orow + q * 32 * osize, o, inv, p.out_dtype);
            }
            tc_fence_before();
            if (LSE && row_ok) {
                // the row's index in [B][Hq][Nq] (dense) or [tokens][Hq] (packed) is its
                // output offset in elements divided by d
                const long long li = ((orow - reinterpret_cast<uint8_t *>(p.out)) >> (osize == 4 ? 2 : 1)) / D;
                p.lse[li] = l > 0.f ? (m_ref + __log2f(l)) * 0.6931471805599453f : -INFINITY;
            }
        }
    } else {
        regs_shrink<kRegsOther>();  // idle warps 10-11
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    if (threadIdx.x == 0 && *abort_flag) atomicCAS(&g_prefill_status, 0, (int)FA_ERR_WATCHDOG);
}

// ---------------------------------------------------------------- stream-K fixup
// Units cut between CTAs: merge the partial (O, m_ref, l) of every piece in CTA
// order, O = sum_k 2^(m_k - M) O_k / sum_k 2^(m_k - M) l_k, and write the rows.
// A piece holds a partial for a query tile only if its key range starts before
// the tile's last key tile (a causal unit's first tile ends one key tile early).
constexpr int kMaxSplit = 192;

struct FixupParams {
    void *out;
    float *lse;
    const float *ws_o;
    const float *ws_ml;
    int Hq, Nq, Nk;
    int n_qb;
    int causal, no_skip;
    int G;
    long long W;
    long long sk_s0;                 // first step of the cut ranges
    int out_dtype;
    int n_split;
    int4 item[kMaxSplit];            // (unit, first CTA, last CTA, unit's key-tile steps)
    long long ustart[kMaxSplit];     // first step of the unit
};

template <int D>
__global__ void __launch_bounds__(256) prefill_fixup(const __grid_constant__ FixupParams f) {
    // CTA (item, g): rows [32 g, 32 g + 32) of the cut unit, in query tile g / 4;
    // warp w merges four of them.  A warp reads one 512-byte record row per load
    // (lane = 4 or 2 columns) and keeps every piece of its rows in flight.
    constexpr int CPL = D / 32;
    constexpr int kRows = 4;     // rows per warp
    constexpr int kChunk = 4;    // pieces in flight per pass
    using Vec = typename std::conditional<CPL == 4, float4, float2>::type;
    __shared__ int s_rec[kMaxSplit];  // record index of row 0 of the unit, per piece
    __shared__ int s_np;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int4 it = f.item[blockIdx.x];
    const int u = it.x;
    const int bh = u / f.n_qb, qb = u % f.n_qb;
    const int t = blockIdx.y >> 2;
    const int tile_row0 = qb * kRowsPerUnit + t * kBlockM;
    const int n_t = kv_tiles(f.causal, f.no_skip, f.Nq, f.Nk, f.Nk - f.Nq, tile_row0);
    const long long ustart = f.ustart[blockIdx.x];
    // The pieces holding keys of this tile, in CTA order: CTA c's range starts at
    // sk_s0 + floor(c (W - sk_s0) / G); slot 0 when the piece opened it, 1 when it
    // closed it.  Worked out before the main kernel has finished.
    if (warp == 0) {
        const long long span = f.W - f.sk_s0;
        int np = 0;
        for (int c0 = it.y; c0 <= it.z; c0 += 32) {
            const int c = c0 + lane;
            bool has = false;
            int rec = 0;
            if (c <= it.z) {
                const long long first = f.sk_s0 + static_cast<long long>(c) * span / f.G;
                const long long next = f.sk_s0 + static_cast<long long>(c + 1) * span / f.G;
                const long long jf = first > ustart ? first - ustart : 0;
                has = next > first && jf < n_t;
                rec = (c * 2 + (first >= ustart ? 0 : 1)) * kRowsPerUnit;
            }
            const unsigned m = __ballot_sync(0xffffffffu, has);
            if (has) s_rec[np + __popc(m & ((1u << lane) - 1))] = rec;
            np += __popc(m);
        }
        if (lane == 0) s_np = np;
    }
    __syncthreads();
    // Launched with programmatic dependent launch: wait until the main kernel
    // has completed and its partials are visible.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int np = s_np;
    const int rr0 = blockIdx.y * 32 + warp * kRows;  // first row of the warp within the unit
    // the max and the weighted sum of l, per row (every lane computes all four)
    float M[kRows], L[kRows];
#pragma unroll
    for (int r = 0; r < kRows; ++r) M[r] = -INFINITY, L[r] = 0.f;
    for (int k = 0; k < np; ++k)
#pragma unroll
        for (int r = 0; r < kRows; ++r) M[r] = fmaxf(M[r], __ldg(f.ws_ml + (static_cast<size_t>(s_rec[k]) + rr0 + r) * 2));
    for (int k = 0; k < np; ++k)
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            const float2 ml = __ldg(reinterpret_cast<const float2 *>(f.ws_ml) + s_rec[k] + rr0 + r);
            if (ml.x != -INFINITY) L[r] = fmaf(ex2_approx(ml.x - M[r]), ml.y, L[r]);
        }
    float acc[kRows][CPL];
#pragma unroll
    for (int r = 0; r < kRows; ++r)
#pragma unroll
        for (int e = 0; e < CPL; ++e) acc[r][e] = 0.f;
    for (int k0 = 0; k0 < np; k0 += kChunk) {
        Vec x[kChunk][kRows];
        float wgt[kChunk][kRows];
#pragma unroll
        for (int j = 0; j < kChunk; ++j) {
            const int k = k0 + j < np ? k0 + j : k0;
            const size_t rec = static_cast<size_t>(s_rec[k]) + rr0;
#pragma unroll
            for (int r = 0; r < kRows; ++r) {
                x[j][r] = __ldg(reinterpret_cast<const Vec *>(f.ws_o + (rec + r) * D) + lane);
                const float m = __ldg(f.ws_ml + (rec + r) * 2);
                wgt[j][r] = (k0 + j < np && m != -INFINITY) ? ex2_approx(m - M[r]) : 0.f;
            }
        }
        // pieces in CTA order, one fma each: the same sum whatever the chunking
#pragma unroll
        for (int j = 0; j < kChunk; ++j) {
            if (k0 + j >= np) break;
#pragma unroll
            for (int r = 0; r < kRows; ++r) {
                const float *xv = reinterpret_cast<const float *>(&x[j][r]);
#pragma unroll
                for (int e = 0; e < CPL; ++e) acc[r][e] = fmaf(wgt[j][r], xv[e], acc[r][e]);
            }
        }
    }
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
        const int row = qb * kRowsPerUnit + rr0 + r;
        if (row >= f.Nq) break;
        const float inv = L[r] > 0.f ? 1.0f / L[r] : 0.f;
        if (f.lse != nullptr && lane == 0)
            f.lse[static_cast<size_t>(bh) * f.Nq + row] =
                L[r] > 0.f ? (M[r] + __log2f(L[r])) * 0.6931471805599453f : -INFINITY;
        const size_t off = (static_cast<size_t>(bh) * f.Nq + row) * D + lane * CPL;
        if (f.out_dtype == FA_F32) {
            float *dst = reinterpret_cast<float *>(f.out) + off;
#pragma unroll
            for (int e = 0; e < CPL; ++e) dst[e] = acc[r][e] * inv;
        } else {
            const int bf = f.out_dtype == FA_BF16;
            uint32_t *dst = reinterpret_cast<uint32_t *>(reinterpret_cast<uint16_t *>(f.out) + off);
#pragma unroll
            for (int e = 0; e < CPL; e += 2) dst[e / 2] = pack2(acc[r][e] * inv, acc[r][e + 1] * inv, bf);
        }
    }
}

// ---------------------------------------------------------------- watchdog self-test
// Two warps wait on barriers that nothing completes: warp 0 with a short
// limit (suspending between polls, as mbar_wait does everywhere), warp 1
// polling (as mbar_spin does for the MMA issuer) with the kernels' own limit,
// which it must abandon once warp 0 raises the abort flag.  The exit path is
// the attention kernel's: a raised flag becomes FA_ERR_WATCHDOG.
__global__ void __launch_bounds__(64, 1) watchdog_selftest_kernel(long long limit_ns, long long *result) {
    __shared__ __align__(8) uint64_t bars[2];
    __shared__ int abort_word;
    volatile int *abort_flag = &abort_word;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(bars + 0, 1);
        mbar_init(bars + 1, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (lane == 0) {
        const uint64_t t0 = globaltimer_ns();
        // phase 0 of a fresh barrier completes only after an arrival: never here
        const bool done = warp == 0 ? mbar_wait(bars + 0, 0, abort_flag, static_cast<uint64_t>(limit_ns))
                                    : mbar_spin(bars + 1, 0, abort_flag, kWatchdogNs);
        const uint64_t t1 = globaltimer_ns();
        result[warp] = done ? 0 : 1;
        result[2 + warp] = static_cast<long long>(t1 - t0);
    }
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag) atomicCAS(&g_prefill_status, 0, (int)FA_ERR_WATCHDOG);
}

// ---------------------------------------------------------------- host side
int host_kv_tiles(int causal, int no_skip, int nq, int nk, int row0) {
    if (row0 >= nq) return 0;
    const int tk = (nk + kBlockN - 1) / kBlockN;
    if (!causal || no_skip) return tk;
    const int last = std::min(row0 + kBlockM - 1, nq - 1) + (nk - nq);
    if (last < 0) return 0;
    return std::min(tk, last / kBlockN + 1);
}

// Stream-K costs, in key-tile steps, fitted to measured launch times on GB300
// (d = 64 and 128, dense and causal): cutting units between CTAs costs about
// 10 steps (partial writes, extra pipeline fills, the fixup pass of 7-10 us)
// when the units are non-causal and 20 when they are causal, and a causal
// stream-K step runs about 8% slower than a step of the unit schedule.
constexpr long long kMergeCostSteps = 10;
constexpr long long kCausalMergeCostSteps = 20;
constexpr long long kCausalStepPct = 108;

struct Plan {
    int stream_k;
    int paired;
    int grid;
    int n_qb;
    int HT;
    long long W;
    int dp_full;
    long long sk_s0;
    int n_split;
    int4 item[kMaxSplit];         // (unit, first CTA, last CTA, unit's steps)
    long long ustart[kMaxSplit];  // first step of the unit
    StepTable tab;
};

// The schedule of a problem, from the shapes and the SM count only.  Unit by
// unit (rounds of G units dealt in snake order, heaviest causal blocks first) the busiest CTA does
// `busiest` key-tile steps; cut into equal step ranges (stream-K) it does W / G
// (8% dearer when causal) plus the merge cost.  Take the cheaper, unless
// `schedule` forces one (1 units, 2 stream-K).  Stream-K needs every unit's
// cost on the host (dense batches) and every query row to see a key.
void make_plan(bool packed, int B, int Hq, int Nq, int Nk, int causal, int no_skip, int schedule,
               int num_sms, Plan &pl) {
    const int BH = B * Hq;
    const int n_qb = (Nq + kRowsPerUnit - 1) / kRowsPerUnit;
    const int n_units = BH * n_qb;
    const int sms = num_sms < kMaxSplit ? num_sms : kMaxSplit;
    pl.stream_k = 0;
    pl.paired = 0;
    pl.n_qb = n_qb;
    pl.HT = 0;
    pl.W = 0;
    pl.dp_full = 0;
    pl.sk_s0 = 0;
    pl.n_split = 0;
    pl.grid = n_units < num_sms ? n_units : num_sms;
    pl.tab.pre[0] = 0;
    // A causal dense problem whose units fit in one round runs unit by unit with
    // paired query tiles (i, T - 1 - i) unless stream-K is taken below.
    const bool pair_tiles = !packed && causal && !no_skip && n_units <= num_sms && schedule != 2;
    pl.paired = pair_tiles ? 1 : 0;
    const bool sk_ok = !packed && n_qb <= kMaxPre && n_units >= 2 && (!causal || no_skip || Nk >= Nq) &&
                       schedule != 1;
    if (!sk_ok) return;
    int *pre = pl.tab.pre;
    for (int qb = 0; qb < n_qb; ++qb) {
        const int c0 = host_kv_tiles(causal, no_skip, Nq, Nk, qb * kRowsPerUnit);
        const int c1 = host_kv_tiles(causal, no_skip, Nq, Nk, qb * kRowsPerUnit + kBlockM);
        pre[qb + 1] = pre[qb] + std::max(c0, c1);
    }
    const int HT = pre[n_qb];
    const long long W = static_cast<long long>(BH) * HT;
    bool take = schedule == 2;
    if (!take && n_units <= 65536) {
        const int gu = std::min(std::min(n_units, num_sms), 1024);
        long long busiest = 0;
        if (causal) {
            static thread_local long long load[1024];
            for (int c = 0; c < gu; ++c) load[c] = 0;
            for (int u = 0; u < n_units; ++u) {  // the kernel's snake order
                const int qb = n_qb - 1 - u / BH;
                const int k = u / gu, r = u % gu;
                load[(k & 1) ? gu - 1 - r : r] += pre[qb + 1] - pre[qb];
            }
            for (int c = 0; c < gu; ++c) busiest = std::max(busiest, load[c]);
        } else {
            busiest = static_cast<long long>((n_units + gu - 1) / gu) * pre[1];
        }
        const long long pct = causal ? kCausalStepPct : 100;
        take = (W * pct + 100LL * sms - 1) / (100LL * sms) +
                   (causal ? kCausalMergeCostSteps : kMergeCostSteps) < busiest;
    }
    if (!take) return;
    pl.stream_k = 1;
    pl.paired = 0;
    pl.HT = HT;
    pl.W = W;
    const int grid = sms;
    pl.grid = grid;
    // Non-causal units all cost the same: deal whole units round robin first
    // and cut only the remainder (every CTA still does about W / G steps).
    if (!causal) {
        pl.dp_full = n_units / grid;
        pl.sk_s0 = static_cast<long long>(pl.dp_full) * grid * pre[1];
    }
    const long long s0 = pl.sk_s0, span = W - s0;
    if (span == 0) return;  // whole units only: nothing is cut
    auto first_step = [&](long long c) { return s0 + c * span / grid; };
    auto cta_of = [&](long long step) {  // c with first_step(c) <= step < first_step(c + 1)
        long long c = (step - s0 + 1) * grid / span;
        if (c >= grid) c = grid - 1;
        while (c > 0 && first_step(c) > step) --c;
        while (c + 1 < grid && first_step(c + 1) <= step) ++c;
        return static_cast<int>(c);
    };
    auto unit_of = [&](long long step, long long &ustart, int &cost) {
        const long long bh = step / HT;
        const int rem = static_cast<int>(step - bh * HT);
        const int qb = static_cast<int>(std::upper_bound(pre, pre + n_qb + 1, rem) - pre) - 1;
        ustart = bh * HT + pre[qb];
        cost = pre[qb + 1] - pre[qb];
        return static_cast<int>(bh * n_qb + qb);
    };
    int last_u = -1;
    for (int c = 1; c < grid; ++c) {
        const long long b = first_step(c);
        if (b >= W) break;
        long long us;
        int cost;
        const int u = unit_of(b, us, cost);
        if (b == us || u == last_u) continue;  // a boundary between units, or done
        last_u = u;
        pl.item[pl.n_split] = make_int4(u, cta_of(us), cta_of(us + cost - 1), cost);
        pl.ustart[pl.n_split] = us;
        ++pl.n_split;
    }
}

// The (sequence, 256-row query block) classes of a packed batch, most 128 x 128
// tile products first (ties by class index), for the unit schedule: its rounds
// then deal heavy units before light ones across sequences of any length, where
// the plain order ranks blocks by their index alone.  One CTA sorts the at most
// kOrderMax classes in shared memory (bitonic, on 64-bit keys: inverted product
// count above, class index below, so the order is total and the same on every
// run).  The lengths are clamped as the prefill kernel clamps them.
constexpr int kOrderMax = 4096;
constexpr int kOrderThreads = 1024;

__global__ void __launch_bounds__(kOrderThreads)
    packed_order_kernel(const int *cu_q, const int *cu_k, int B, int n_qb, int Nq, int Nk, int total_q,
                        int total_k, int causal, int no_skip, int *order) {
    __shared__ unsigned long long key[kOrderMax];
    const int n = B * n_qb;
    int m = 1;
    while (m < n) m <<= 1;
    for (int i = threadIdx.x; i < m; i += kOrderThreads) {
        unsigned long long k = ~0ull;  // padding sorts last
        if (i < n) {
            const int b = i / n_qb, qb = i % n_qb;
            const int q_lo = min(max(cu_q[b], 0), total_q), q_hi = min(max(cu_q[b + 1], q_lo), total_q);
            const int k_lo = min(max(cu_k[b], 0), total_k), k_hi = min(max(cu_k[b + 1], k_lo), total_k);
            const int nq = min(q_hi - q_lo, Nq), nk = min(k_hi - k_lo, Nk);
            const int r0 = qb * kRowsPerUnit;
            const int c = kv_tiles(causal, no_skip, nq, nk, nk - nq, r0) +
                          kv_tiles(causal, no_skip, nq, nk, nk - nq, r0 + kBlockM);
            k = (static_cast<unsigned long long>(0x7fffffff - c) << 32) | static_cast<unsigned>(i);
        }
        key[i] = k;
    }
    __syncthreads();
    for (int size = 2; size <= m; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = threadIdx.x; i < m; i += kOrderThreads) {
                const int j = i ^ stride;
                if (j > i) {
                    const bool up = (i & size) == 0;
                    const unsigned long long a = key[i], c = key[j];
                    if ((a > c) == up) {
                        key[i] = c;
                        key[j] = a;
                    }
                }
            }
            __syncthreads();
        }
    }
    for (int i = threadIdx.x; i < n; i += kOrderThreads) order[i] = static_cast<int>(key[i] & 0xffffffffu);
}

template <int D, bool BF16, bool LSE>
int launch_d_lse(const PrefillLaunch &a, const DeviceInfo &dev, cudaStream_t stream) {
    using L = Layout<D>;
    static_assert(L::kSmemBytes <= 227 * 1024, "shared memory budget");
    const bool packed = a.cu_q != nullptr;
    CUtensorMap mq, mk, mv;
    int rc;
    if (packed) {
        if ((rc = make_map(&mq, a.q, D, true, a.total_q, a.Hq, a.in_bf16)) != FA_OK) return rc;
        if ((rc = make_map(&mk, a.k, D, true, a.total_k, a.Hkv, a.in_bf16)) != FA_OK) return rc;
        if ((rc = make_map(&mv, a.v, D, true, a.total_k, a.Hkv, a.in_bf16)) != FA_OK) return rc;
    } else {
        if ((rc = make_map(&mq, a.q, D, false, a.Nq, (long long)a.B * a.Hq, a.in_bf16)) != FA_OK) return rc;
        if ((rc = make_map(&mk, a.k, D, false, a.Nk, (long long)a.B * a.Hkv, a.in_bf16)) != FA_OK) return rc;
        if ((rc = make_map(&mv, a.v, D, false, a.Nk, (long long)a.B * a.Hkv, a.in_bf16)) != FA_OK) return rc;
    }
    Params p;
    p.out = a.out;
    p.lse = a.lse;
    p.cu_q = a.cu_q;
    p.cu_k = a.cu_k;
    p.order = nullptr;
    p.B = a.B;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.group = a.Hq / a.Hkv;
    p.Nq = a.Nq;
    p.Nk = a.Nk;
    p.total_q = a.total_q;
    p.total_k = a.total_k;
    p.BH = a.B * a.Hq;
    p.n_qb = (a.Nq + kRowsPerUnit - 1) / kRowsPerUnit;
    p.n_units = p.BH * p.n_qb;
    p.causal = a.causal ? 1 : 0;
    p.no_skip = a.no_skip ? 1 : 0;
    p.in_bf16 = a.in_bf16;
    p.out_dtype = a.out_dtype;
    // scale == 0 runs as 2^-100: every weight is then exactly 1 as well, and
    // masked scores (+-inf) never meet a zero multiplier.
    const float scale = a.scale == 0.f ? 0x1p-100f : a.scale;
    p.scale_neg = scale < 0.f ? 1 : 0;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.scale_log2_abs = fabsf(p.scale_log2);
    p.stream_k = 0;
    p.n_tt = 0;
    p.HT = 0;
    p.W = 0;
    p.ws_o = nullptr;
    p.ws_ml = nullptr;

    static thread_local Plan pl;  // ~8 KB: keep it off the stack
    make_plan(packed, a.B, a.Hq, a.Nq, a.Nk, p.causal, p.no_skip, a.schedule, dev.num_sms, pl);
    p.stream_k = pl.stream_k;
    p.n_tt = (a.Nq + kBlockM - 1) / kBlockM;
    // the ordered schedule for a packed batch over more than one round of units
    const long long n_cls = static_cast<long long>(a.B) * p.n_qb;
    const bool ordered = packed && !pl.stream_k && p.n_units > pl.grid && n_cls <= kOrderMax;
    const auto kernel = pl.paired ? prefill_kernel<D, BF16, LSE, kSchedPaired>
                                  : (ordered ? prefill_kernel<D, BF16, LSE, kSchedOrdered>
                                             : prefill_kernel<D, BF16, LSE, kSchedPlain>);
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemBytes);
    if (e != cudaSuccess) return cuda_fail(e);
    // The setmaxnreg split inside the kernel draws on the launch allocation:
    // refuse to launch a build whose register count would make it wait forever.
    cudaFuncAttributes fattr;
    e = cudaFuncGetAttributes(&fattr, kernel);
    if (e != cudaSuccess) return cuda_fail(e);
    if (fattr.numRegs < kMinLaunchRegs) return cuda_fail(cudaErrorInvalidConfiguration);
    p.HT = pl.HT;
    p.W = pl.W;
    p.dp_full = pl.dp_full;
    p.sk_s0 = pl.sk_s0;
    const int grid = pl.grid;
    static thread_local FixupParams f;
    f.n_split = 0;
    void *ws = nullptr;
    if (p.stream_k) {
        f.out = a.out;
        f.lse = a.lse;
        f.Hq = a.Hq;
        f.Nq = a.Nq;
        f.Nk = a.Nk;
        f.n_qb = p.n_qb;
        f.causal = p.causal;
        f.no_skip = p.no_skip;
        f.G = grid;
        f.W = p.W;
        f.sk_s0 = pl.sk_s0;
        f.out_dtype = a.out_dtype;
        f.n_split = pl.n_split;
        for (int i = 0; i < pl.n_split; ++i) {
            f.item[i] = pl.item[i];
            f.ustart[i] = pl.ustart[i];
        }
        if (f.n_split > 0) {
            const size_t o_bytes = static_cast<size_t>(grid) * 2 * kRowsPerUnit * D * sizeof(float);
            const size_t ml_bytes = static_cast<size_t>(grid) * 2 * kRowsPerUnit * 2 * sizeof(float);
            e = scratch_alloc(&ws, o_bytes + ml_bytes, stream);
            if (e != cudaSuccess) {
                cuda_fail(e);
                return FA_ERR_WORKSPACE;
            }
            p.ws_o = static_cast<float *>(ws);
            p.ws_ml = reinterpret_cast<float *>(static_cast<char *>(ws) + o_bytes);
            f.ws_o = p.ws_o;
            f.ws_ml = p.ws_ml;
        }
    }
    // A packed batch over more than one round of units takes its classes heaviest
    // first (the order comes from the device-resident offsets, so a small kernel
    // computes it on the stream just before).
    void *ord = nullptr;
    if (ordered) {
        if ((e = scratch_alloc(&ord, static_cast<size_t>(n_cls) * sizeof(int), stream)) != cudaSuccess) {
            cuda_fail(e);
            if (ws) scratch_free(ws, stream);
            return FA_ERR_WORKSPACE;
        }
        packed_order_kernel<<<1, kOrderThreads, 0, stream>>>(a.cu_q, a.cu_k, a.B, p.n_qb, a.Nq, a.Nk, a.total_q,
                                                             a.total_k, p.causal, p.no_skip,
                                                             static_cast<int *>(ord));
        e = cudaGetLastError();
        if (e != cudaSuccess) {
            scratch_free(ord, stream);
            if (ws) scratch_free(ws, stream);
            return cuda_fail(e);
        }
        p.order = static_cast<const int *>(ord);
    }
    const StepTable &tab = pl.tab;
    kernel<<<grid, kThreads, L::kSmemBytes, stream>>>(mq, mk, mv, p, tab);
    e = cudaGetLastError();
    if (e == cudaSuccess && f.n_split > 0) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(f.n_split, kRowsPerUnit / 32);
        cfg.blockDim = dim3(256);
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, prefill_fixup<D>, f);
        if (e == cudaSuccess) e = cudaGetLastError();
    }
    if (ws) {
        const cudaError_t e2 = scratch_free(ws, stream);
        if (e == cudaSuccess) e = e2;
    }
    if (ord) {
        const cudaError_t e2 = scratch_free(ord, stream);
        if (e == cudaSuccess) e = e2;
    }
    if (e != cudaSuccess) return cuda_fail(e);
    return FA_OK;
}

}  // namespace

int plan_prefill(int B, int Hq, int Nq, int Nk, int causal, int no_skip, int schedule, int num_sms,
                 long long *info, long long *items, int max_items) {
    static thread_local Plan pl;
    make_plan(false, B, Hq, Nq, Nk, causal ? 1 : 0, no_skip, schedule, num_sms, pl);
    info[0] = pl.stream_k;
    info[1] = pl.grid;
    info[2] = pl.W;
    info[3] = pl.HT;
    info[4] = pl.n_qb;
    info[5] = pl.n_split;
    info[6] = pl.dp_full;
    info[7] = pl.sk_s0;
    info[8] = pl.paired;
    if (items)
        for (int i = 0; i < pl.n_split && i < max_items; ++i) {
            items[i * 5 + 0] = pl.item[i].x;
            items[i * 5 + 1] = pl.item[i].y;
            items[i * 5 + 2] = pl.item[i].z;
            items[i * 5 + 3] = pl.item[i].w;
            items[i * 5 + 4] = pl.ustart[i];
        }
    return FA_OK;
}

template <int D, bool BF16>
int launch_d(const PrefillLaunch &a, const DeviceInfo &dev, cudaStream_t stream) {
    return a.lse ? launch_d_lse<D, BF16, true>(a, dev, stream) : launch_d_lse<D, BF16, false>(a, dev, stream);
}

int launch_prefill(const PrefillLaunch &a, const DeviceInfo &dev, cudaStream_t stream) {
    if (a.d == 64) return a.in_bf16 ? launch_d<64, true>(a, dev, stream) : launch_d<64, false>(a, dev, stream);
    if (a.d == 128) return a.in_bf16 ? launch_d<128, true>(a, dev, stream) : launch_d<128, false>(a, dev, stream);
    return FA_ERR_HEAD_DIM;
}

int read_prefill_status(int reset) {
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_prefill_status, sizeof(int));
    if (e != cudaSuccess) return -1;
    if (reset && v) {
        int z = 0;
        if (cudaMemcpyToSymbol(g_prefill_status, &z, sizeof(int)) != cudaSuccess) return -1;
    }
    return v;
}

}  // namespace fa

extern "C" int fa_watchdog_selftest(long long limit_ns, long long *result, void *stream) {
    if (!result) return FA_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(result) & 7u) return FA_ERR_ALIGN;
    if (limit_ns < 1000 || limit_ns > 1000000000LL) return FA_ERR_SHAPE;
    fa::DeviceInfo dev;
    const int rc = fa::current_device_info(&dev);
    if (rc != FA_OK) return rc;
    fa::watchdog_selftest_kernel<<<1, 64, 0, static_cast<cudaStream_t>(stream)>>>(limit_ns, result);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fa::cuda_fail(e);
    return FA_OK;
}
