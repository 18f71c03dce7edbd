// fa_tiles.cuh -- device helpers shared by the forward and backward attention
// kernels: bounded warp waits, the tcgen05 products of 128-row tiles (a score
// tile Q K^T with both operands K-major in shared memory, and an accumulation
// O += P V with P in TMEM and V MN-major in shared memory), and the packing of
// fp32 rows into 16-bit pairs and output rows.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>
#include <cuda.h>

#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {

constexpr uint64_t kWatchdogNs = 1500ull * 1000ull * 1000ull;  // every wait gives up after 1.5 s
constexpr int kTileKeys = 128;           // keys (K dimension of P V) per tile
constexpr int kSlabBytes = 128 * 128;    // 128 rows x 64 16-bit columns, 128-byte swizzled

// Warp-uniform bounded wait: lane 0 polls, the verdict is broadcast.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag) {
    int ok = 1;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, abort_flag, kWatchdogNs) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    return ok != 0;
}

// The MMA chains below are issued from one asm block each: the descriptors'
// start-address fields are advanced by 32-bit adds on their low words
// (shared addresses stay below 256 KB, so a field can never carry into the
// next), and only the first product of a chain reads its accumulate flag.
#define FA_MMA_SS(OFFA, OFFB)                                                 \
    "add.u32 xa, %1, " #OFFA ";\n\t"                                        \
    "add.u32 xb, %3, " #OFFB ";\n\t"                                        \
    "mov.b64 a, {xa, %2};\n\t"                                              \
    "mov.b64 b, {xb, %4};\n\t"                                              \
    "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %5, pt;\n\t"

// S = Q K^T over d: a_desc / b_desc describe the Q and K tiles at K-step 0;
// step kk moves (kk / 4) 64-column slabs and (kk % 4) 32-byte atoms along d,
// i.e. ((kk / 4) * 16384 + (kk % 4) * 32) / 16 in the descriptors' address field.
template <int D>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc) {
    const uint32_t alo = static_cast<uint32_t>(a_desc), ahi = static_cast<uint32_t>(a_desc >> 32);
    const uint32_t blo = static_cast<uint32_t>(b_desc), bhi = static_cast<uint32_t>(b_desc >> 32);
    if constexpr (D == 128) {
        asm volatile(
            "{\n\t.reg .pred pf, pt;\n\t.reg .b64 a, b;\n\t.reg .b32 xa, xb;\n\t"
            "setp.ne.b32 pf, %6, %6;\n\t"
            "setp.eq.b32 pt, %6, %6;\n\t"
            "mov.b64 a, {%1, %2};\n\t"
            "mov.b64 b, {%3, %4};\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %5, pf;\n\t"
            FA_MMA_SS(2, 2) FA_MMA_SS(4, 4) FA_MMA_SS(6, 6)
            FA_MMA_SS(1024, 1024) FA_MMA_SS(1026, 1026) FA_MMA_SS(1028, 1028) FA_MMA_SS(1030, 1030)
            "}" ::"r"(d_tmem), "r"(alo), "r"(ahi), "r"(blo), "r"(bhi), "r"(idesc), "r"(0)
            : "memory");
    } else {
        static_assert(D == 64, "head sizes 64 and 128");
        asm volatile(
            "{\n\t.reg .pred pf, pt;\n\t.reg .b64 a, b;\n\t.reg .b32 xa, xb;\n\t"
            "setp.ne.b32 pf, %6, %6;\n\t"
            "setp.eq.b32 pt, %6, %6;\n\t"
            "mov.b64 a, {%1, %2};\n\t"
            "mov.b64 b, {%3, %4};\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %5, pf;\n\t"
            FA_MMA_SS(2, 2) FA_MMA_SS(4, 4) FA_MMA_SS(6, 6)
            "}" ::"r"(d_tmem), "r"(alo), "r"(ahi), "r"(blo), "r"(bhi), "r"(idesc), "r"(0)
            : "memory");
    }
}
#undef FA_MMA_SS

// O (+)= P V: P from TMEM (16 keys = 8 columns per step), V tile [key][d] with d
// contiguous is an MN-major B operand: 16 keys per step = two 8-key groups
// (SBO apart), i.e. 16 * 128 / 16 = 128 in the descriptor's address field;
// 64-column slabs of d are LBO apart.  The first product accumulates only if
// `accumulate` is set.
#define FA_MMA_TS(OFFA, OFFB)                                                 \
    "add.u32 ta, %1, " #OFFA ";\n\t"                                        \
    "add.u32 xb, %2, " #OFFB ";\n\t"                                        \
    "mov.b64 b, {xb, %3};\n\t"                                              \
    "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], b, %4, pt;\n\t"

template <int D>
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint64_t v_desc,
                                         uint32_t idesc, bool accumulate) {
    static_assert(kTileKeys == 128, "eight 16-key products per tile");
    const uint32_t blo = static_cast<uint32_t>(v_desc), bhi = static_cast<uint32_t>(v_desc >> 32);
    asm volatile(
        "{\n\t.reg .pred pf, pt;\n\t.reg .b64 b;\n\t.reg .b32 ta, xb;\n\t"
        "setp.ne.b32 pf, %5, 0;\n\t"
        "setp.eq.b32 pt, %5, %5;\n\t"
        "mov.b64 b, {%2, %3};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], b, %4, pf;\n\t"
        FA_MMA_TS(8, 128) FA_MMA_TS(16, 256) FA_MMA_TS(24, 384) FA_MMA_TS(32, 512)
        FA_MMA_TS(40, 640) FA_MMA_TS(48, 768) FA_MMA_TS(56, 896)
        "}" ::"r"(d_tmem), "r"(p_tmem), "r"(blo), "r"(bhi), "r"(idesc), "r"(accumulate ? 1u : 0u)
        : "memory");
}
#undef FA_MMA_TS

// The two 16-bit values of a packed pair, back in fp32 (exact), as an f32x2.
template <bool BF16>
__device__ __forceinline__ uint64_t unpack2(uint32_t w) {
    if constexpr (BF16) {
        return f2_pack(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    } else {
        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w));
        return f2_pack(f.x, f.y);
    }
}

// lo += w.lo, hi += w.hi for the two 16-bit values of a packed pair, each
// widened exactly inside a mixed-precision add (sm_100+), round to nearest.
template <bool BF16>
__device__ __forceinline__ void add_pair16(float &lo, float &hi, uint32_t w) {
    if constexpr (BF16) {
        asm("{\n\t.reg .b16 a, b;\n\t"
            "mov.b32 {a, b}, %2;\n\t"
            "add.rn.f32.bf16 %0, a, %0;\n\t"
            "add.rn.f32.bf16 %1, b, %1;\n\t}"
            : "+f"(lo), "+f"(hi)
            : "r"(w));
    } else {
        asm("{\n\t.reg .b16 a, b;\n\t"
            "mov.b32 {a, b}, %2;\n\t"
            "add.rn.f32.f16 %0, a, %0;\n\t"
            "add.rn.f32.f16 %1, b, %1;\n\t}"
            : "+f"(lo), "+f"(hi)
            : "r"(w));
    }
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2t(float lo, float hi) {
    if constexpr (BF16) {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&h);
    } else {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&h);
    }
}

// Row maximum of 128 scores: eight independent chains of 3-input maxima.
template <bool NEG>
__device__ __forceinline__ float row_max128(const uint32_t (&sr)[4][32]) {
    float m[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float a = __uint_as_float(sr[i >> 1][(i & 1) * 16 + 0]);
        m[i] = NEG ? -a : a;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        // chain i covers columns [16 i, 16 i + 16)
#pragma unroll
        for (int c = 1; c < 16; c += 2) {
            const int col = 16 * i + c;
            const float a = __uint_as_float(sr[col >> 5][col & 31]);
            const float b = (c + 1 < 16) ? __uint_as_float(sr[(col + 1) >> 5][(col + 1) & 31]) : a;
            m[i] = NEG ? fmax3(m[i], -a, -b) : fmax3(m[i], a, b);
        }
    }
    return fmaxf(fmax3(m[0], m[1], m[2]), fmax3(fmax3(m[3], m[4], m[5]), m[6], m[7]));
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi, int bf16) {
    if (bf16) {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&h);
    }
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

// One 32-column slice of a finished output row: O * inv_l -> out dtype.
__device__ __forceinline__ void store_out32(void *dst, const uint32_t (&r)[32], float inv,
                                            int out_dtype) {
    if (out_dtype == FA_F32) {
        uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
        for (int v = 0; v < 8; ++v) {
            uint4 w;
            w.x = __float_as_uint(__uint_as_float(r[4 * v + 0]) * inv);
            w.y = __float_as_uint(__uint_as_float(r[4 * v + 1]) * inv);
            w.z = __float_as_uint(__uint_as_float(r[4 * v + 2]) * inv);
            w.w = __float_as_uint(__uint_as_float(r[4 * v + 3]) * inv);
            d4[v] = w;
        }
    } else {
        const int bf = out_dtype == FA_BF16;
        uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            uint4 w;
            w.x = pack2(__uint_as_float(r[8 * v + 0]) * inv, __uint_as_float(r[8 * v + 1]) * inv, bf);
            w.y = pack2(__uint_as_float(r[8 * v + 2]) * inv, __uint_as_float(r[8 * v + 3]) * inv, bf);
            w.z = pack2(__uint_as_float(r[8 * v + 4]) * inv, __uint_as_float(r[8 * v + 5]) * inv, bf);
            w.w = pack2(__uint_as_float(r[8 * v + 6]) * inv, __uint_as_float(r[8 * v + 7]) * inv, bf);
            d4[v] = w;
        }
    }
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult qres;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                             &qres) != cudaSuccess ||
            qres != cudaDriverEntryPointSuccess)
            ptr = nullptr;
        return reinterpret_cast<EncodeTiledFn>(ptr);
    }();
    return fn;
}

// A dense [BH][N][d] tensor is viewed as (d, N, BH) with 64 x 128 x 1 boxes; a
// packed [tokens][H][d] tensor as (d, H, tokens) with 64 x 1 x 128 boxes.  Both
// land in shared memory as 128 rows of 128 bytes, 128-byte swizzled.  Rows past
// the end of the tensor read as zero.
inline int make_map(CUtensorMap *map, const void *base, int d, bool packed, long long rows, long long outer,
             int bf16) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cuda_fail(cudaErrorNotSupported);
    cuuint64_t dims[3], strides[2];
    cuuint32_t box[3];
    if (packed) {  // rows = tokens, outer = heads
        dims[0] = d; dims[1] = (cuuint64_t)outer; dims[2] = (cuuint64_t)(rows > 0 ? rows : 1);
        strides[0] = (cuuint64_t)d * 2;
        strides[1] = (cuuint64_t)d * 2 * (cuuint64_t)outer;
        box[0] = 64; box[1] = 1; box[2] = 128;
    } else {       // rows = sequence length, outer = batch x heads
        dims[0] = d; dims[1] = (cuuint64_t)rows; dims[2] = (cuuint64_t)outer;
        strides[0] = (cuuint64_t)d * 2;
        strides[1] = (cuuint64_t)d * 2 * (cuuint64_t)rows;
        box[0] = 64; box[1] = 128; box[2] = 1;
    }
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                     const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue);
    return FA_OK;
}

}  // namespace fa
