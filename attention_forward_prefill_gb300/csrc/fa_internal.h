// fa_internal.h -- declarations shared between the C-ABI layer (fa_api.cu)
// and the kernel translation units.  Not part of the public interface.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/fa.h"

namespace fa {

// Per-device state (attribute cache, scratch pool, copy streams, the static
// decode scratch address) is kept for device ordinals below this bound.
constexpr int kMaxDevices = 64;

struct DeviceInfo {
    int device = -1;
    int num_sms = 0;
    int cc_major = 0;
    int cc_minor = 0;
    int l2_bytes = 0;
    size_t max_smem_optin = 0;
};

// Cached attributes of the current device; returns FA_OK / FA_ERR_CUDA / FA_ERR_ARCH.
int current_device_info(DeviceInfo *out);

// Record a CUDA error for fa_last_cuda_error() and return FA_ERR_CUDA.
int cuda_fail(cudaError_t e);

// Stream-ordered scratch memory from a pool the library owns on the current
// device.  The pool keeps freed memory mapped (up to a threshold), so a call
// made after a stream synchronisation does not pay to map its workspace again.
cudaError_t scratch_alloc(void **ptr, size_t bytes, cudaStream_t stream);
cudaError_t scratch_free(void *ptr, cudaStream_t stream);

struct PrefillLaunch {
    const void *q, *k, *v;
    void *out;
    float *lse;                  // optional row log-sum-exp output (natural log)
    const int32_t *cu_q, *cu_k;  // packed batch: [B+1] token offsets (device); null when dense
    int B, Hq, Hkv;
    int Nq, Nk;                  // dense: lengths; packed: max_seqlen_q / max_seqlen_k
    int total_q, total_k;        // packed: token counts
    int d;
    int causal;
    int no_skip;
    float scale;
    int in_bf16;    // 1: bf16 inputs, 0: fp16
    int out_dtype;  // fa_dtype
    int schedule;   // 0: choose, 1: unit by unit, 2: stream-K where possible
};

// Host-only: the schedule the launch would use (see fa_prefill_plan).
int plan_prefill(int B, int Hq, int Nq, int Nk, int causal, int no_skip, int schedule, int num_sms,
                 long long *info, long long *items, int max_items);

// Validated arguments -> encode tensor maps, launch the persistent kernel.
int launch_prefill(const PrefillLaunch &a, const DeviceInfo &dev, cudaStream_t stream);

// Grouped decode: a group of G query heads is cut into ceil(G / 4) slices,
// one CTA row each, so that a CTA holds at most 4 query heads.  (With 8 at
// d = 64, a thread's queries and accumulators took 168 registers and 3 CTAs fit
// an SM; with 4, 112 registers and 4 CTAs: 14 query heads over 2 cache heads
// decode 7-13% faster although each K/V row is read by two CTAs.)
inline int decode_group_slices(int group) { return (group + 3) / 4; }

struct DecodeLaunch {
    const void *q, *k_cache, *v_cache;
    const int32_t *seq_lens;
    void *out;
    int B, H, max_len, d;
    int Hkv;              // cache heads; H / Hkv query heads share each
    float scale;
    int in_bf16;
    int out_dtype;
    int num_splits;
    int chunk;
    float *partial_ml;   // [B][H][splits][2]  (m, l)
    float *partial_acc;  // [B][H][splits][d]
};

int launch_decode(const DecodeLaunch &a, const DeviceInfo &dev, cudaStream_t stream);

// Streaming-read probe over `bytes` (a multiple of 16) with the decode loads.
int launch_read_probe(const void *src, size_t bytes, uint32_t *xor_out, const DeviceInfo &dev,
                      cudaStream_t stream);

struct BackwardLaunch {
    const void *q, *k, *v, *out, *dout;  // q, out, dout [B][H][N][d]; k, v [B][Hkv][N][d] 16-bit
    const float *lse;                    // [B][H][N] natural-log row log-sum-exp of the forward
    void *dq, *dk, *dv;                  // dq [B][H][N][d], dk, dv [B][Hkv][N][d] in grad_dtype
    int B, H, Hkv, N, d;
    int causal;
    float scale;
    int in_bf16;
    int grad_dtype;
    int num_sms;                         // persistent grids: at most one CTA per SM
    int recompute_dq;                    // 1: the dQ pass recomputes S and dP instead of reading dS
};

int launch_backward(const BackwardLaunch &a, cudaStream_t stream);

// Device-side watchdog words (one per kernel translation unit).
int read_prefill_status(int reset);
int read_decode_status(int reset);
int read_backward_status(int reset);

}  // namespace fa
