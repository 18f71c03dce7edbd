// fa_decode_sm103.cu -- split-K decode: one query row per (b, h) over a ragged
// KV cache (flash-attention-cuda README, "What did I implement?" generation
// phase, and the "Kernel design" rows "Split-K decode + adaptive chunk" and
// "Two-pass merge, no atomics").
//
// Kernel 1 (split): CTA (s, h, b) covers cache rows
//   [s * chunk, min((s + 1) * chunk, len_b))
// and writes the partial (m_s, l_s, acc_s) with scores kept in the exp2 domain
// (c = scale * log2 e):  x_j = c * q.k_j,  m_s = max_j x_j,
//   l_s = sum_j 2^(x_j - m_s),  acc_s = sum_j 2^(x_j - m_s) v_j.
// A CTA whose chunk starts at or past len_b does nothing.
// Kernel 2 (merge): one warp per (b, h), splits combined in index order:
//   M = max_s m_s,  w_s = 2^(m_s - M),  O = sum_s w_s acc_s / sum_s w_s l_s.
// Every reduction runs in a fixed order, so a given split count gives the
// same bits on every run; there are no atomics.
//
// The split kernel is HBM-bound (about one FLOP per byte): it streams each K
// row and each V row once with 16-byte loads, eight in flight per thread,
// lanes of a warp covering whole rows so that every load is coalesced.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {

namespace {

constexpr int kSplitThreads = 128;
constexpr int kSplitWarps = kSplitThreads / 32;
constexpr int kUnroll = 8;
constexpr int kMergeWarps = 4;

// Device status word of the decode kernels: FA_ERR_SEQ_LEN once a length
// outside [0, max_len] has been clamped (the decode kernels have no waits).
__device__ int g_decode_status = 0;

struct DParams {
    const uint16_t *q;
    const uint16_t *k;
    const uint16_t *v;
    const int32_t *seq_lens;
    void *out;
    float *ml;
    float *acc;
    int H;         // query heads
    int BH;        // B * H
    int Hkv;       // cache heads (H for plain multi-head decode)
    int group;     // H / Hkv: query head h reads cache head h / group
    int gper;      // grouped decode: query heads per CTA (a slice of one group)
    int ngb;       // slices per group
    int max_len;
    int chunk;
    int splits;
    int in_bf16;
    int out_dtype;
    float scale_log2;
};

__device__ __forceinline__ int clamp_len(int len, int max_len) {
    return len < 0 ? 0 : (len > max_len ? max_len : len);
}

__device__ __forceinline__ void unpack8(const uint4 &w, int bf16, float (&f)[8]) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 t;
        if (bf16) {
            t = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u[i]));
        } else {
            t = __half22float2(*reinterpret_cast<const __half2 *>(&u[i]));
        }
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}

__device__ __forceinline__ uint4 ldg_stream(const uint16_t *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

template <int D>
__global__ void __launch_bounds__(kSplitThreads)
    decode_split_kernel(const DParams p) {
    constexpr int LPK = D * 2 / 16;          // lanes per cache row (16 bytes each)
    constexpr int KPW = 32 / LPK;            // rows per warp per step
    constexpr int KPC = KPW * kSplitWarps;   // rows per CTA per step
    extern __shared__ float sh[];            // [chunk] scores, then reduction scratch
    __shared__ float red[kSplitWarps][D];
    __shared__ float red1[kSplitWarps];

    // Let the merge kernel (launched with programmatic dependent launch) get
    // scheduled early; it still waits for this whole grid before reading.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int s = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int len = clamp_len(p.seq_lens[b], p.max_len);
    const int start = s * p.chunk;
    if (start >= len) return;
    const int n = min(start + p.chunk, len) - start;
    const size_t bh = static_cast<size_t>(b) * p.H + h;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sub = lane % LPK, kw = lane / LPK;

    float qf[8];
    unpack8(*reinterpret_cast<const uint4 *>(p.q + bh * D + sub * 8), p.in_bf16, qf);
    const uint16_t *kbase = p.k + (bh * p.max_len + start) * D + sub * 8;
    const uint16_t *vbase = p.v + (bh * p.max_len + start) * D + sub * 8;
    float *sc = sh;

    // ---- scores x_j = c * q.k_j
    // The loop bound is warp-uniform (base0); each lane's row is base0 + kw.
    for (int base0 = warp * KPW; base0 < n; base0 += KPC * kUnroll) {
        const int base = base0 + kw;
        uint4 kr[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int key = base + u * KPC;
            kr[u] = key < n ? ldg_stream(kbase + static_cast<size_t>(key) * D) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            float kf[8];
            unpack8(kr[u], p.in_bf16, kf);
            float dot = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) dot = fmaf(qf[e], kf[e], dot);
#pragma unroll
            for (int off = 1; off < LPK; off <<= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
            const int key = base + u * KPC;
            if (sub == 0 && key < n) sc[key] = dot * p.scale_log2;
        }
    }
    __syncthreads();

    // ---- chunk maximum
    float mx = -INFINITY;
    for (int i = threadIdx.x; i < n; i += kSplitThreads) mx = fmaxf(mx, sc[i]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if (lane == 0) red1[warp] = mx;
    __syncthreads();
    float m = red1[0];
#pragma unroll
    for (int w = 1; w < kSplitWarps; ++w) m = fmaxf(m, red1[w]);
    __syncthreads();

    // ---- weights 2^(x_j - m) and their sum
    float sum = 0.f;
    for (int i = threadIdx.x; i < n; i += kSplitThreads) {
        const float e = ex2_approx(sc[i] - m);
        sc[i] = e;
        sum += e;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    if (lane == 0) red1[warp] = sum;
    __syncthreads();
    float l = red1[0];
#pragma unroll
    for (int w = 1; w < kSplitWarps; ++w) l += red1[w];

    // ---- acc = sum_j w_j v_j
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    for (int base0 = warp * KPW; base0 < n; base0 += KPC * kUnroll) {
        const int base = base0 + kw;
        uint4 vr[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int key = base + u * KPC;
            vr[u] = key < n ? ldg_stream(vbase + static_cast<size_t>(key) * D) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int key = base + u * KPC;
            const float w = key < n ? sc[key] : 0.f;
            float vf[8];
            unpack8(vr[u], p.in_bf16, vf);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = fmaf(w, vf[e], acc[e]);
        }
    }
#pragma unroll
    for (int off = LPK; off < 32; off <<= 1)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], off);
    if (kw == 0)
#pragma unroll
        for (int e = 0; e < 8; ++e) red[warp][sub * 8 + e] = acc[e];
    __syncthreads();

    const size_t part = bh * p.splits + s;
    for (int c = threadIdx.x; c < D; c += kSplitThreads) {
        float a = red[0][c];
#pragma unroll
        for (int w = 1; w < kSplitWarps; ++w) a += red[w][c];
        p.acc[part * D + c] = a;
    }
    if (threadIdx.x == 0) {
        p.ml[part * 2 + 0] = m;
        p.ml[part * 2 + 1] = l;
    }
}

// Grouped decode: the query heads of one cache head (flash-attention-cuda
// README, "Future work": kernel-side GQA instead of a host-side repeat) share
// each K and V row the CTA streams.  CTA (s, hk * ngb + slice, b) covers up to
// GP query heads h0 .. h0 + gcnt - 1 of cache head hk over the same chunk as
// the plain kernel, and writes one partial per query head in the same layout,
// so the merge kernel is shared.
template <int D, int GP>
__global__ void __launch_bounds__(kSplitThreads)
    decode_split_gqa_kernel(const DParams p) {
    constexpr int LPK = D * 2 / 16;          // lanes per cache row (16 bytes each)
    constexpr int KPW = 32 / LPK;            // rows per warp per step
    constexpr int KPC = KPW * kSplitWarps;   // rows per CTA per step
    extern __shared__ float sh[];            // [GP][chunk] scores, then weights
    __shared__ float red[kSplitWarps][GP][D];
    __shared__ float red1[kSplitWarps][GP];

    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int s = blockIdx.x, b = blockIdx.z;
    const int hk = blockIdx.y / p.ngb, slice = blockIdx.y % p.ngb;
    const int h0 = hk * p.group + slice * p.gper;
    const int gcnt = min(p.gper, p.group - slice * p.gper);
    const int len = clamp_len(p.seq_lens[b], p.max_len);
    const int start = s * p.chunk;
    if (start >= len || gcnt <= 0) return;
    const int n = min(start + p.chunk, len) - start;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sub = lane % LPK, kw = lane / LPK;
    const int ch = p.chunk;

    float qf[GP][8];
#pragma unroll
    for (int g = 0; g < GP; ++g) {
        if (g < gcnt) {
            const size_t bhq = static_cast<size_t>(b) * p.H + h0 + g;
            unpack8(*reinterpret_cast<const uint4 *>(p.q + bhq * D + sub * 8), p.in_bf16, qf[g]);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) qf[g][e] = 0.f;
        }
    }
    const size_t bhk = static_cast<size_t>(b) * p.Hkv + hk;
    const uint16_t *kbase = p.k + (bhk * p.max_len + start) * D + sub * 8;
    const uint16_t *vbase = p.v + (bhk * p.max_len + start) * D + sub * 8;

    // ---- scores x_gj = c * q_g.k_j, each K row read once for all GP heads
    for (int base0 = warp * KPW; base0 < n; base0 += KPC * kUnroll) {
        const int base = base0 + kw;
        uint4 kr[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int key = base + u * KPC;
            kr[u] = key < n ? ldg_stream(kbase + static_cast<size_t>(key) * D) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            float kf[8];
            unpack8(kr[u], p.in_bf16, kf);
            const int key = base + u * KPC;
#pragma unroll
            for (int g = 0; g < GP; ++g) {
                float dot = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) dot = fmaf(qf[g][e], kf[e], dot);
#pragma unroll
                for (int off = 1; off < LPK; off <<= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
                if (sub == 0 && key < n) sh[g * ch + key] = dot * p.scale_log2;
            }
        }
    }
    __syncthreads();

    // ---- per head: chunk maximum, then weights 2^(x - m) and their sum
    float m[GP], l[GP];
#pragma unroll
    for (int g = 0; g < GP; ++g) {
        float mx = -INFINITY;
        for (int i = threadIdx.x; i < n; i += kSplitThreads) mx = fmaxf(mx, sh[g * ch + i]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        if (lane == 0) red1[warp][g] = mx;
    }
    __syncthreads();
#pragma unroll
    for (int g = 0; g < GP; ++g) {
        m[g] = red1[0][g];
#pragma unroll
        for (int w = 1; w < kSplitWarps; ++w) m[g] = fmaxf(m[g], red1[w][g]);
    }
    __syncthreads();
#pragma unroll
    for (int g = 0; g < GP; ++g) {
        float sum = 0.f;
        for (int i = threadIdx.x; i < n; i += kSplitThreads) {
            const float e = ex2_approx(sh[g * ch + i] - m[g]);
            sh[g * ch + i] = e;
            sum += e;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
        if (lane == 0) red1[warp][g] = sum;
    }
    __syncthreads();
#pragma unroll
    for (int g = 0; g < GP; ++g) {
        l[g] = red1[0][g];
#pragma unroll
        for (int w = 1; w < kSplitWarps; ++w) l[g] += red1[w][g];
    }

    // ---- acc_g = sum_j w_gj v_j, each V row read once for all GP heads
    float acc[GP][8];
#pragma unroll
    for (int g = 0; g < GP; ++g)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[g][e] = 0.f;
    for (int base0 = warp * KPW; base0 < n; base0 += KPC * kUnroll) {
        const int base = base0 + kw;
        uint4 vr[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int key = base + u * KPC;
            vr[u] = key < n ? ldg_stream(vbase + static_cast<size_t>(key) * D) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int key = base + u * KPC;
            float vf[8];
            unpack8(vr[u], p.in_bf16, vf);
#pragma unroll
            for (int g = 0; g < GP; ++g) {
                const float w = key < n ? sh[g * ch + key] : 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[g][e] = fmaf(w, vf[e], acc[g][e]);
            }
        }
    }
#pragma unroll
    for (int g = 0; g < GP; ++g)
#pragma unroll
        for (int off = LPK; off < 32; off <<= 1)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[g][e] += __shfl_xor_sync(0xffffffffu, acc[g][e], off);
    if (kw == 0)
#pragma unroll
        for (int g = 0; g < GP; ++g)
#pragma unroll
            for (int e = 0; e < 8; ++e) red[warp][g][sub * 8 + e] = acc[g][e];
    __syncthreads();

    for (int i = threadIdx.x; i < gcnt * D; i += kSplitThreads) {
        const int g = i / D, c = i % D;
        float a = red[0][g][c];
#pragma unroll
        for (int w = 1; w < kSplitWarps; ++w) a += red[w][g][c];
        const size_t part = (static_cast<size_t>(b) * p.H + h0 + g) * p.splits + s;
        p.acc[part * D + c] = a;
    }
    if (threadIdx.x < gcnt) {
        const int g = threadIdx.x;
        float mg = m[0], lg = l[0];
#pragma unroll
        for (int k = 1; k < GP; ++k)
            if (k == g) { mg = m[k]; lg = l[k]; }
        const size_t part = (static_cast<size_t>(b) * p.H + h0 + g) * p.splits + s;
        p.ml[part * 2 + 0] = mg;
        p.ml[part * 2 + 1] = lg;
    }
}

template <int N> struct VecF;
template <> struct VecF<2> { using T = float2; };
template <> struct VecF<4> { using T = float4; };

__device__ __forceinline__ void vadd_scaled(float (&o)[2], float w, const float2 &a) {
    o[0] = fmaf(w, a.x, o[0]);
    o[1] = fmaf(w, a.y, o[1]);
}
__device__ __forceinline__ void vadd_scaled(float (&o)[4], float w, const float4 &a) {
    o[0] = fmaf(w, a.x, o[0]);
    o[1] = fmaf(w, a.y, o[1]);
    o[2] = fmaf(w, a.z, o[2]);
    o[3] = fmaf(w, a.w, o[3]);
}

template <int D>
__global__ void __launch_bounds__(kMergeWarps * 32)
    decode_merge_kernel(const DParams p) {
    constexpr int EPL = D / 32;  // output elements per lane
    constexpr int G = 8;         // partial vectors in flight per lane
    using Vec = typename VecF<EPL>::T;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gw = blockIdx.x * kMergeWarps + warp;
    const bool live = gw < p.BH;
    // The lengths are the caller's input, not the split kernel's output, so
    // they are read before the wait.
    int n_act = 0;
    if (live) {
        const int raw = p.seq_lens[gw / p.H];
        // one report per sequence (its first head); the length is clamped either way
        if (lane == 0 && gw % p.H == 0 && (raw < 0 || raw > p.max_len))
            atomicCAS(&g_decode_status, 0, static_cast<int>(FA_ERR_SEQ_LEN));
        const int len = clamp_len(raw, p.max_len);
        n_act = (len + p.chunk - 1) / p.chunk;
    }
    // Wait until the split kernel has completed and its partials are visible.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (!live) return;
    float o[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) o[e] = 0.f;
    if (n_act > 0) {
        const float2 *ml = reinterpret_cast<const float2 *>(p.ml) + static_cast<size_t>(gw) * p.splits;
        const Vec *acc = reinterpret_cast<const Vec *>(p.acc + static_cast<size_t>(gw) * p.splits * D) + lane;
        constexpr int VPS = D / EPL;  // Vec per split
        // Split s's (m_s, l_s) lives in lane s % 32; the first G partial
        // vectors are requested together with them.
        Vec a[G];
#pragma unroll
        for (int u = 0; u < G; ++u) a[u] = u < n_act ? acc[u * VPS] : Vec{};
        float2 mv = lane < n_act ? ml[lane] : make_float2(-INFINITY, 0.f);
        float M = mv.x;
        for (int s = 32 + lane; s < n_act; s += 32) M = fmaxf(M, ml[s].x);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        float lsum = 0.f, w = 0.f;
        for (int g0 = 0; g0 < n_act; g0 += G) {
            if ((g0 & 31) == 0) {  // the next 32 splits' weights w_s = 2^(m_s - M)
                if (g0 > 0) mv = g0 + lane < n_act ? ml[g0 + lane] : make_float2(-INFINITY, 0.f);
                w = g0 + lane < n_act ? ex2_approx(mv.x - M) : 0.f;
                lsum = fmaf(w, mv.y, lsum);
            }
            if (g0 > 0) {
#pragma unroll
                for (int u = 0; u < G; ++u) a[u] = g0 + u < n_act ? acc[(g0 + u) * VPS] : Vec{};
            }
            // splits in index order; past n_act both w and a are 0
#pragma unroll
            for (int u = 0; u < G; ++u)
                vadd_scaled(o, __shfl_sync(0xffffffffu, w, (g0 & 31) + u), a[u]);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, off);
        const float inv = 1.0f / lsum;
#pragma unroll
        for (int e = 0; e < EPL; ++e) o[e] *= inv;
    }
    const size_t off = static_cast<size_t>(gw) * D + lane * EPL;
    if (p.out_dtype == FA_F32) {
        float *out = reinterpret_cast<float *>(p.out) + off;
#pragma unroll
        for (int e = 0; e < EPL; ++e) out[e] = o[e];
    } else if (p.out_dtype == FA_BF16) {
        __nv_bfloat16 *out = reinterpret_cast<__nv_bfloat16 *>(p.out) + off;
#pragma unroll
        for (int e = 0; e < EPL; ++e) out[e] = __float2bfloat16_rn(o[e]);
    } else {
        __half *out = reinterpret_cast<__half *>(p.out) + off;
#pragma unroll
        for (int e = 0; e < EPL; ++e) out[e] = __float2half_rn(o[e]);
    }
}

// Read-bandwidth probe: every thread streams 16-byte words with the split
// kernel's non-caching load, four in flight, over a grid-stride loop; the XOR
// of all words is the result, so no load can be dropped.
constexpr int kProbeThreads = 512;
constexpr int kProbeUnroll = 4;

__global__ void __launch_bounds__(kProbeThreads) read_probe_kernel(const uint4 *src, size_t n16,
                                                                   uint32_t *xor_out) {
    __shared__ uint32_t red[kProbeThreads / 32];
    const size_t stride = static_cast<size_t>(gridDim.x) * kProbeThreads;
    size_t i = static_cast<size_t>(blockIdx.x) * kProbeThreads + threadIdx.x;
    uint32_t x = 0;
    for (; i + (kProbeUnroll - 1) * stride < n16; i += kProbeUnroll * stride) {
        uint4 r[kProbeUnroll];
#pragma unroll
        for (int u = 0; u < kProbeUnroll; ++u)
            r[u] = ldg_stream(reinterpret_cast<const uint16_t *>(src + i + u * stride));
#pragma unroll
        for (int u = 0; u < kProbeUnroll; ++u) x ^= r[u].x ^ r[u].y ^ r[u].z ^ r[u].w;
    }
    for (; i < n16; i += stride) {
        const uint4 r = ldg_stream(reinterpret_cast<const uint16_t *>(src + i));
        x ^= r.x ^ r.y ^ r.z ^ r.w;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x ^= __shfl_xor_sync(0xffffffffu, x, off);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = x;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t t = 0;
#pragma unroll
        for (int w = 0; w < kProbeThreads / 32; ++w) t ^= red[w];
        atomicXor(xor_out, t);
    }
}

template <int D, int GP>
cudaError_t launch_gqa_split(const DParams &p, const DecodeLaunch &a, cudaStream_t stream) {
    const size_t smem = static_cast<size_t>(GP) * a.chunk * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(decode_split_gqa_kernel<D, GP>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(a.num_splits, a.Hkv * p.ngb, a.B);
    decode_split_gqa_kernel<D, GP><<<grid, kSplitThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

template <int D>
int launch_decode_d(const DecodeLaunch &a, cudaStream_t stream) {
    DParams p;
    p.q = static_cast<const uint16_t *>(a.q);
    p.k = static_cast<const uint16_t *>(a.k_cache);
    p.v = static_cast<const uint16_t *>(a.v_cache);
    p.seq_lens = a.seq_lens;
    p.out = a.out;
    p.ml = a.partial_ml;
    p.acc = a.partial_acc;
    p.H = a.H;
    p.BH = a.B * a.H;
    p.Hkv = a.Hkv;
    p.group = a.H / a.Hkv;
    p.ngb = decode_group_slices(p.group);
    p.gper = (p.group + p.ngb - 1) / p.ngb;
    p.max_len = a.max_len;
    p.chunk = a.chunk;
    p.splits = a.num_splits;
    p.in_bf16 = a.in_bf16;
    p.out_dtype = a.out_dtype;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    cudaError_t e;
    if (p.group == 1) {
        const size_t smem = static_cast<size_t>(a.chunk) * sizeof(float);
        e = cudaFuncSetAttribute(decode_split_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e != cudaSuccess) return cuda_fail(e);
        dim3 grid(a.num_splits, a.H, a.B);
        decode_split_kernel<D><<<grid, kSplitThreads, smem, stream>>>(p);
        e = cudaGetLastError();
    } else if (p.gper <= 2) {
        e = launch_gqa_split<D, 2>(p, a, stream);
    } else {  // decode_group_slices keeps gper <= 4
        e = launch_gqa_split<D, 4>(p, a, stream);
    }
    if (e != cudaSuccess) return cuda_fail(e);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((p.BH + kMergeWarps - 1) / kMergeWarps);
    cfg.blockDim = dim3(kMergeWarps * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, decode_merge_kernel<D>, p);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e);
    return FA_OK;
}

}  // namespace

int read_decode_status(int reset) {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_decode_status, sizeof(int)) != cudaSuccess) return -1;
    if (reset && v) {
        int z = 0;
        if (cudaMemcpyToSymbol(g_decode_status, &z, sizeof(int)) != cudaSuccess) return -1;
    }
    return v;
}

int launch_decode(const DecodeLaunch &a, const DeviceInfo &dev, cudaStream_t stream) {
    (void)dev;
    if (a.d == 64) return launch_decode_d<64>(a, stream);
    if (a.d == 128) return launch_decode_d<128>(a, stream);
    return FA_ERR_HEAD_DIM;
}

int launch_read_probe(const void *src, size_t bytes, uint32_t *xor_out, const DeviceInfo &dev,
                      cudaStream_t stream) {
    cudaError_t e = cudaMemsetAsync(xor_out, 0, sizeof(uint32_t), stream);
    if (e != cudaSuccess) return cuda_fail(e);
    // four CTAs of 512 threads per SM: 2048 resident threads, 128 KB of loads in flight
    read_probe_kernel<<<dev.num_sms * 4, kProbeThreads, 0, stream>>>(static_cast<const uint4 *>(src),
                                                                      bytes / 16, xor_out);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e);
    return FA_OK;
}

}  // namespace fa

// ---------------------------------------------------------------------------
// Decode without any allocation.  The split partials live in a fixed
// file-scope device array instead of a cudaMallocAsync'd or caller-provided
// buffer.  Every GPU that loads this library reserves the array until the
// process exits.  Host code may not pass the array's name to a kernel (on the
// host it is only a stand-in for the device symbol): its device address is
// looked up once per device with cudaGetSymbolAddress.
// ---------------------------------------------------------------------------
#include <mutex>

namespace fa {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;  // 4 MiB
static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of the static scratch on the current device (set up on the
// first call per device, with that device current).  The device and its
// architecture are checked first, so that a wrong device reports FA_ERR_ARCH
// as the allocating entry point does, not a failed symbol lookup.
int noalloc_scratch(void **out) {
    DeviceInfo info;
    const int rc = current_device_info(&info);
    if (rc != FA_OK) return rc;
    const int dev = info.device;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (e != cudaSuccess) return cuda_fail(e);
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return FA_OK;
}

}  // namespace
}  // namespace fa

extern "C" size_t fa_decode_noalloc_max_bytes(void) { return fa::kNoAllocScratchBytes; }

extern "C" int fa_decode_noalloc(const void *q, const void *k_cache, const void *v_cache,
                                 const int32_t *seq_lens, void *out, int B, int H, int max_len,
                                 int d, float scale, fa_dtype in_dtype, fa_dtype out_dtype,
                                 int num_splits, void *stream) {
    // Pointer and size checks first (host arithmetic once the split count is
    // known); every other argument error is left to fa_decode_ex.
    if (!q || !k_cache || !v_cache || !seq_lens || !out) return FA_ERR_NULL;
    if (B >= 1 && H >= 1 && max_len >= 1 && (d == 64 || d == 128) && num_splits >= 0) {
        int splits = num_splits;
        if (splits == 0) {
            splits = fa_decode_choose_splits(B, H, max_len, -1);
            if (splits < 0) return -splits;
        }
        if (fa_decode_workspace_bytes(B, H, max_len, d, splits) > fa::kNoAllocScratchBytes)
            return FA_ERR_WORKSPACE;
    }
    void *scratch = nullptr;
    int rc = fa::noalloc_scratch(&scratch);
    if (rc != FA_OK) return rc;
    // With a workspace supplied, fa_decode_ex allocates nothing.
    return fa_decode_ex(q, k_cache, v_cache, seq_lens, out, B, H, max_len, d, scale, in_dtype,
                        out_dtype, num_splits, scratch, fa::kNoAllocScratchBytes, stream);
}

extern "C" int fa_read_probe(const void *src, size_t bytes, uint32_t *xor_out, void *stream) {
    if (!src || !xor_out) return FA_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(src) & 15u) || (reinterpret_cast<uintptr_t>(xor_out) & 3u))
        return FA_ERR_ALIGN;
    if (bytes == 0 || bytes % 16 != 0) return FA_ERR_SHAPE;
    fa::DeviceInfo dev;
    const int rc = fa::current_device_info(&dev);
    if (rc != FA_OK) return rc;
    return fa::launch_read_probe(src, bytes, xor_out, dev, static_cast<cudaStream_t>(stream));
}
