// fa_api.cu -- the extern "C" boundary of libfa_gb300.so (declared in
// include/fa.h).  Argument validation happens before any CUDA call, so every
// argument error is reported without touching a device.  The interface
// follows the two calls of the flash-attention-cuda README ("Installation"
// usage: prefill(q, k, v, causal, scale) and decode(q, k_cache, v_cache,
// seq_lens, scale)) with the validation its bindings layer performs
// ("Project structure": bindings.cpp, "input validation").
#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "fa_internal.h"

namespace fa {

namespace {
thread_local int t_last_cuda_error = 0;

std::mutex g_dev_mu;
DeviceInfo g_dev_cache[kMaxDevices];
bool g_dev_have[kMaxDevices] = {};

cudaMemPool_t g_pool[kMaxDevices] = {};
constexpr uint64_t kPoolKeepBytes = 5ull << 30;  // freed scratch kept mapped (a backward dS table: up to 4 GiB)

constexpr int kDecodeRowAlign = 64;      // chunk lengths are multiples of this
constexpr int kDecodeAutoMaxChunk = 512;  // automatic choice: at most 512 rows per CTA
constexpr int kDecodeMaxChunk = 48 * 1024; // any choice: scores of a chunk <= 192 KB smem

bool misaligned(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + nb && b0 < a0 + na;
}

size_t dtype_size(int dt) { return dt == FA_F32 ? 4 : 2; }

long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }

int decode_effective_splits(int max_len, int splits, int *chunk_out) {
    const long long chunk =
        ceil_div(ceil_div(max_len, splits), kDecodeRowAlign) * kDecodeRowAlign;
    if (chunk_out) *chunk_out = static_cast<int>(chunk);
    return static_cast<int>(ceil_div(max_len, chunk));
}

size_t ws_ml_bytes(long long bh, int splits) {
    return static_cast<size_t>((bh * splits * 2 * 4 + 255) / 256 * 256);
}
}  // namespace

int cuda_fail(cudaError_t e) {
    t_last_cuda_error = static_cast<int>(e);
    return FA_ERR_CUDA;
}

int current_device_info(DeviceInfo *out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return cuda_fail(cudaErrorInvalidDevice);
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (!g_dev_have[dev]) {
        DeviceInfo d;
        d.device = dev;
        int v = 0;
        if ((e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev)) ||
            (e = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) ||
            (e = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) ||
            (e = cudaDeviceGetAttribute(&d.l2_bytes, cudaDevAttrL2CacheSize, dev)) ||
            (e = cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)))
            return cuda_fail(e);
        d.max_smem_optin = static_cast<size_t>(v);
        g_dev_cache[dev] = d;
        g_dev_have[dev] = true;
    }
    *out = g_dev_cache[dev];
    if (!(out->cc_major == 10 && out->cc_minor == 3)) return FA_ERR_ARCH;
    return FA_OK;
}

cudaError_t scratch_alloc(void **ptr, size_t bytes, cudaStream_t stream) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    cudaMemPool_t pool;
    {
        std::lock_guard<std::mutex> lk(g_dev_mu);
        if (!g_pool[dev]) {
            cudaMemPoolProps props = {};
            props.allocType = cudaMemAllocationTypePinned;
            props.location.type = cudaMemLocationTypeDevice;
            props.location.id = dev;
            cudaMemPool_t created;
            if ((e = cudaMemPoolCreate(&created, &props)) != cudaSuccess) return e;
            uint64_t keep = kPoolKeepBytes;
            if ((e = cudaMemPoolSetAttribute(created, cudaMemPoolAttrReleaseThreshold, &keep)) !=
                cudaSuccess) {
                cudaMemPoolDestroy(created);
                return e;
            }
            g_pool[dev] = created;
        }
        pool = g_pool[dev];
    }
    return cudaMallocFromPoolAsync(ptr, bytes, pool, stream);
}

cudaError_t scratch_free(void *ptr, cudaStream_t stream) { return cudaFreeAsync(ptr, stream); }

}  // namespace fa

using namespace fa;

extern "C" {

int fa_version(void) { return 2 * 10000 + 1 * 100 + 0; }

const char *fa_status_string(int status) {
    switch (status) {
        case FA_OK: return "ok";
        case FA_ERR_NULL: return "a required pointer is NULL";
        case FA_ERR_SHAPE: return "bad shape: sizes must be >= 1 and fit in int32";
        case FA_ERR_HEAD_DIM: return "unsupported head dimension (64 or 128)";
        case FA_ERR_DTYPE: return "unsupported dtype combination";
        case FA_ERR_ALIGN: return "a pointer is not 16-byte aligned";
        case FA_ERR_SCALE: return "scale is not finite";
        case FA_ERR_ARCH: return "device is not compute capability 10.3 (sm_103a)";
        case FA_ERR_WORKSPACE: return "workspace too small or allocation failed";
        case FA_ERR_CUDA: return "CUDA runtime error (see fa_last_cuda_error)";
        case FA_ERR_WATCHDOG: return "a device-side wait ran out of time";
        case FA_ERR_SEQ_LEN: return "a device-resident sequence length was out of range (clamped)";
        case FA_ERR_ALIAS: return "output overlaps an input";
        case FA_ERR_SPLITS: return "num_splits out of range";
        default: return "unknown status";
    }
}

int fa_last_cuda_error(void) { return t_last_cuda_error; }

int fa_device_status(int reset) {
    if (cudaDeviceSynchronize() != cudaSuccess) return -1;
    const int a = read_prefill_status(reset), b = read_decode_status(reset),
              c = read_backward_status(reset);
    if (a < 0 || b < 0 || c < 0) return -1;
    // a watchdog report wins over a clamped length
    for (int v : {a, b, c})
        if (v == FA_ERR_WATCHDOG) return v;
    return a ? a : (b ? b : c);
}

int fa_pool_stats(long long *out, int reset_high) {
    if (!out) return FA_ERR_NULL;
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return cuda_fail(cudaErrorInvalidDevice);
    cudaMemPool_t pool;
    {
        std::lock_guard<std::mutex> lk(g_dev_mu);
        pool = g_pool[dev];
    }
    for (int i = 0; i < 4; ++i) out[i] = 0;
    if (!pool) return FA_OK;  // nothing was ever allocated on this device
    const cudaMemPoolAttr attrs[4] = {cudaMemPoolAttrReservedMemCurrent, cudaMemPoolAttrReservedMemHigh,
                                      cudaMemPoolAttrUsedMemCurrent, cudaMemPoolAttrUsedMemHigh};
    for (int i = 0; i < 4; ++i) {
        uint64_t v = 0;
        if ((e = cudaMemPoolGetAttribute(pool, attrs[i], &v)) != cudaSuccess) return cuda_fail(e);
        out[i] = static_cast<long long>(v);
    }
    if (reset_high) {
        uint64_t zero = 0;
        if ((e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReservedMemHigh, &zero)) != cudaSuccess ||
            (e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrUsedMemHigh, &zero)) != cudaSuccess)
            return cuda_fail(e);
    }
    return FA_OK;
}

namespace {
int prefill_common_checks(const void *q, const void *k, const void *v, void *out, int d,
                          fa_dtype in_dtype, fa_dtype out_dtype, float scale) {
    if (!q || !k || !v || !out) return FA_ERR_NULL;
    if (d != 64 && d != 128) return FA_ERR_HEAD_DIM;
    if (in_dtype != FA_F16 && in_dtype != FA_BF16) return FA_ERR_DTYPE;
    if (out_dtype != FA_F16 && out_dtype != FA_BF16 && out_dtype != FA_F32) return FA_ERR_DTYPE;
    if (misaligned(q) || misaligned(k) || misaligned(v) || misaligned(out)) return FA_ERR_ALIGN;
    if (!std::isfinite(scale)) return FA_ERR_SCALE;
    return FA_OK;
}

int schedule_of(unsigned flags) {
    if (flags & FA_FLAG_SCHEDULE_UNITS) return 1;
    if (flags & FA_FLAG_SCHEDULE_STREAM_K) return 2;
    return 0;
}
}  // namespace

int fa_prefill_lse(const void *q, const void *k, const void *v, void *out, float *lse, int B,
                   int Hq, int Hkv, int Nq, int Nk, int d, int causal, float scale,
                   fa_dtype in_dtype, fa_dtype out_dtype, unsigned flags, void *stream) {
    int rc = prefill_common_checks(q, k, v, out, d, in_dtype, out_dtype, scale);
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return FA_ERR_ALIGN;
    if (rc != FA_OK) return rc;
    if (B < 1 || Hq < 1 || Hkv < 1 || Nq < 1 || Nk < 1) return FA_ERR_SHAPE;
    if (Hq % Hkv != 0) return FA_ERR_SHAPE;
    if (static_cast<long long>(B) * Hq * Nq > INT_MAX || static_cast<long long>(B) * Hkv * Nk > INT_MAX)
        return FA_ERR_SHAPE;
    const size_t q_bytes = static_cast<size_t>(B) * Hq * Nq * d * 2;
    const size_t kv_bytes = static_cast<size_t>(B) * Hkv * Nk * d * 2;
    const size_t out_bytes = static_cast<size_t>(B) * Hq * Nq * d * dtype_size(out_dtype);
    if (overlaps(out, out_bytes, q, q_bytes) || overlaps(out, out_bytes, k, kv_bytes) ||
        overlaps(out, out_bytes, v, kv_bytes))
        return FA_ERR_ALIAS;
    if (lse) {
        const size_t lse_bytes = static_cast<size_t>(B) * Hq * Nq * 4;
        if (overlaps(lse, lse_bytes, out, out_bytes) || overlaps(lse, lse_bytes, q, q_bytes) ||
            overlaps(lse, lse_bytes, k, kv_bytes) || overlaps(lse, lse_bytes, v, kv_bytes))
            return FA_ERR_ALIAS;
    }
    DeviceInfo dev;
    rc = current_device_info(&dev);
    if (rc != FA_OK) return rc;
    PrefillLaunch a;
    a.q = q;
    a.k = k;
    a.v = v;
    a.out = out;
    a.lse = lse;
    a.cu_q = nullptr;
    a.cu_k = nullptr;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.Nq = Nq;
    a.Nk = Nk;
    a.total_q = 0;
    a.total_k = 0;
    a.d = d;
    a.causal = causal ? 1 : 0;
    a.no_skip = (flags & FA_FLAG_NO_CAUSAL_SKIP) ? 1 : 0;
    a.scale = scale;
    a.in_bf16 = in_dtype == FA_BF16 ? 1 : 0;
    a.out_dtype = out_dtype;
    a.schedule = schedule_of(flags);
    return launch_prefill(a, dev, static_cast<cudaStream_t>(stream));
}

int fa_prefill_gqa(const void *q, const void *k, const void *v, void *out, int B, int Hq, int Hkv,
                   int Nq, int Nk, int d, int causal, float scale, fa_dtype in_dtype,
                   fa_dtype out_dtype, unsigned flags, void *stream) {
    return fa_prefill_lse(q, k, v, out, nullptr, B, Hq, Hkv, Nq, Nk, d, causal, scale, in_dtype,
                          out_dtype, flags, stream);
}

}  // extern "C"

namespace {
// Copy streams and events of the host-buffer pipeline, one set per device,
// created on first use and kept for the life of the process.  The input copies
// of every call share one stream (the host link carries one direction's copies
// at full rate, so the calls' inputs go in call order); the output copies take
// one of kOutStreams streams in turn, so that one call's outputs never queue
// behind another call's kernels.
constexpr int kHostChunks = 8;
constexpr int kOutStreams = 4;
struct HostPipe {
    bool ready = false;
    cudaStream_t s_in = nullptr, s_out[kOutStreams] = {};
    int next_out = 0;
    cudaEvent_t start = nullptr, done = nullptr;
    cudaEvent_t in[kHostChunks] = {}, comp[kHostChunks] = {};
};
std::mutex g_pipe_mu;
HostPipe g_pipe[kMaxDevices];

cudaError_t host_pipe(int dev, HostPipe **out) {
    HostPipe &hp = g_pipe[dev];
    if (!hp.ready) {
        cudaError_t e;
        if ((e = cudaStreamCreateWithFlags(&hp.s_in, cudaStreamNonBlocking)) ||
            (e = cudaEventCreateWithFlags(&hp.start, cudaEventDisableTiming)) ||
            (e = cudaEventCreateWithFlags(&hp.done, cudaEventDisableTiming)))
            return e;
        for (int i = 0; i < kOutStreams; ++i)
            if ((e = cudaStreamCreateWithFlags(&hp.s_out[i], cudaStreamNonBlocking))) return e;
        for (int c = 0; c < kHostChunks; ++c)
            if ((e = cudaEventCreateWithFlags(&hp.in[c], cudaEventDisableTiming)) ||
                (e = cudaEventCreateWithFlags(&hp.comp[c], cudaEventDisableTiming)))
                return e;
        hp.ready = true;
    }
    *out = &hp;
    return cudaSuccess;
}

size_t round_up256(size_t x) { return (x + 255) / 256 * 256; }

// Chunks of the host-buffer pipeline, as key/value-head boundaries
// bound[0] = 0 < bound[1] < ... < bound[n] = n_kv; returns n.  Only the first
// chunk's copy in and the last chunk's copy out run under no kernel, so the
// chunk sizes ramp up from a small first chunk and back down to a small last
// one (weights min(i + 1, n - i)).  Every chunk still holds at least
// kHostMinSteps key-tile steps per SM, so that its kernel keeps the GPU busy:
// long sequences can go a head at a time, short ones take fewer, larger chunks.
constexpr long long kHostMinSteps = 24;
int host_chunk_plan(long long n_kv, int group, int Nq, int Nk, bool causal, int num_sms,
                    long long bound[kHostChunks + 1]) {
    const long long q_tiles = (Nq + 127) / 128, k_tiles = (Nk + 127) / 128;
    long long steps = group * q_tiles * k_tiles;  // 128 x 128 tile products per key/value head
    if (causal) steps = (steps + 1) / 2;
    const long long min_heads = std::max(1LL, (kHostMinSteps * num_sms + steps - 1) / steps);
    int n = static_cast<int>(std::min<long long>(kHostChunks, n_kv));
    for (; n > 1; --n) {
        long long w = 0;
        for (int i = 0; i < n; ++i) w += std::min(i + 1, n - i);
        if (n_kv >= min_heads * w) break;  // the first and last chunks hold min_heads or more
    }
    long long w_total = 0;
    for (int i = 0; i < n; ++i) w_total += std::min(i + 1, n - i);
    bound[0] = 0;
    long long w_cum = 0;
    for (int i = 0; i < n; ++i) {
        w_cum += std::min(i + 1, n - i);
        const long long b = (n_kv * w_cum + w_total / 2) / w_total;
        bound[i + 1] = std::min(n_kv - (n - 1 - i), std::max(bound[i] + 1, b));
    }
    return n;
}
}  // namespace

extern "C" {

int fa_prefill_host(const void *q_host, const void *k_host, const void *v_host, void *out_host,
                    int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal, float scale,
                    fa_dtype in_dtype, fa_dtype out_dtype, unsigned flags, void *stream) {
    int rc = prefill_common_checks(q_host, k_host, v_host, out_host, d, in_dtype, out_dtype, scale);
    if (rc != FA_OK) return rc;
    if (B < 1 || Hq < 1 || Hkv < 1 || Nq < 1 || Nk < 1) return FA_ERR_SHAPE;
    if (Hq % Hkv != 0) return FA_ERR_SHAPE;
    if (static_cast<long long>(B) * Hq * Nq > INT_MAX || static_cast<long long>(B) * Hkv * Nk > INT_MAX)
        return FA_ERR_SHAPE;
    const int group = Hq / Hkv;
    const size_t q_head = static_cast<size_t>(Nq) * d * 2, kv_head = static_cast<size_t>(Nk) * d * 2;
    const size_t o_head = static_cast<size_t>(Nq) * d * dtype_size(out_dtype);
    const long long n_kv = static_cast<long long>(B) * Hkv;  // flattened key/value heads
    const size_t q_bytes = q_head * group * n_kv, kv_bytes = kv_head * n_kv, o_bytes = o_head * group * n_kv;
    if (overlaps(out_host, o_bytes, q_host, q_bytes) || overlaps(out_host, o_bytes, k_host, kv_bytes) ||
        overlaps(out_host, o_bytes, v_host, kv_bytes))
        return FA_ERR_ALIAS;
    DeviceInfo dev;
    rc = current_device_info(&dev);
    if (rc != FA_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    std::lock_guard<std::mutex> lk(g_pipe_mu);
    HostPipe *hp = nullptr;
    cudaError_t e = host_pipe(dev.device, &hp);
    if (e != cudaSuccess) return cuda_fail(e);
    void *buf = nullptr;
    const size_t off_k = round_up256(q_bytes), off_v = off_k + round_up256(kv_bytes),
                 off_o = off_v + round_up256(kv_bytes);
    e = scratch_alloc(&buf, off_o + o_bytes, st);
    if (e != cudaSuccess) {
        cuda_fail(e);
        return FA_ERR_WORKSPACE;
    }
    char *qd = static_cast<char *>(buf), *kd = qd + off_k, *vd = qd + off_v, *od = qd + off_o;
    const char *qh = static_cast<const char *>(q_host), *kh = static_cast<const char *>(k_host),
               *vh = static_cast<const char *>(v_host);
    char *oh = static_cast<char *>(out_host);
    // Small problems gain nothing from overlap: one chunk under 8 MB of traffic.
    const size_t total = q_bytes + 2 * kv_bytes + o_bytes;
    long long bound[kHostChunks + 1];
    int n_ch = 1;
    bound[0] = 0;
    bound[1] = n_kv;
    if (total >= (8u << 20)) n_ch = host_chunk_plan(n_kv, group, Nq, Nk, causal != 0, dev.num_sms, bound);
    // this call's output stream (the next of the pool)
    cudaStream_t s_out = hp->s_out[hp->next_out];
    hp->next_out = (hp->next_out + 1) % kOutStreams;
    // the copy streams start after the work already on `stream` (which also
    // orders the pool allocation before them)
    if ((e = cudaEventRecord(hp->start, st)) || (e = cudaStreamWaitEvent(hp->s_in, hp->start, 0)) ||
        (e = cudaStreamWaitEvent(s_out, hp->start, 0))) {
        scratch_free(buf, st);
        return cuda_fail(e);
    }
    rc = FA_OK;
    for (int c = 0; c < n_ch && rc == FA_OK; ++c) {
        const long long h0 = bound[c], h1 = bound[c + 1];  // key/value heads [h0, h1)
        const size_t qo = q_head * group * h0, qn = q_head * group * (h1 - h0);
        const size_t ko = kv_head * h0, kn = kv_head * (h1 - h0);
        const size_t oo = o_head * group * h0, on = o_head * group * (h1 - h0);
        if ((e = cudaMemcpyAsync(qd + qo, qh + qo, qn, cudaMemcpyHostToDevice, hp->s_in)) ||
            (e = cudaMemcpyAsync(kd + ko, kh + ko, kn, cudaMemcpyHostToDevice, hp->s_in)) ||
            (e = cudaMemcpyAsync(vd + ko, vh + ko, kn, cudaMemcpyHostToDevice, hp->s_in)) ||
            (e = cudaEventRecord(hp->in[c], hp->s_in)) || (e = cudaStreamWaitEvent(st, hp->in[c], 0))) {
            rc = cuda_fail(e);
            break;
        }
        // the chunk as one sequence batch of (h1 - h0) * group query heads
        PrefillLaunch a;
        a.q = qd + qo;
        a.k = kd + ko;
        a.v = vd + ko;
        a.out = od + oo;
        a.lse = nullptr;
        a.cu_q = nullptr;
        a.cu_k = nullptr;
        a.B = 1;
        a.Hq = static_cast<int>(h1 - h0) * group;
        a.Hkv = static_cast<int>(h1 - h0);
        a.Nq = Nq;
        a.Nk = Nk;
        a.total_q = 0;
        a.total_k = 0;
        a.d = d;
        a.causal = causal ? 1 : 0;
        a.no_skip = (flags & FA_FLAG_NO_CAUSAL_SKIP) ? 1 : 0;
        a.scale = scale;
        a.in_bf16 = in_dtype == FA_BF16 ? 1 : 0;
        a.out_dtype = out_dtype;
        a.schedule = schedule_of(flags);
        rc = launch_prefill(a, dev, st);
        if (rc != FA_OK) break;
        if ((e = cudaEventRecord(hp->comp[c], st)) || (e = cudaStreamWaitEvent(s_out, hp->comp[c], 0)) ||
            (e = cudaMemcpyAsync(oh + oo, od + oo, on, cudaMemcpyDeviceToHost, s_out)))
            rc = cuda_fail(e);
    }
    // `stream` continues after both copy streams (the last output copy, and on
    // an error any input copy already issued); the buffers then go back to the
    // pool, stream-ordered.
    for (cudaStream_t s : {hp->s_in, s_out}) {
        if ((e = cudaEventRecord(hp->done, s)) == cudaSuccess) e = cudaStreamWaitEvent(st, hp->done, 0);
        if (e != cudaSuccess && rc == FA_OK) rc = cuda_fail(e);
    }
    e = scratch_free(buf, st);
    if (e != cudaSuccess && rc == FA_OK) rc = cuda_fail(e);
    return rc;
}

int fa_prefill_varlen(const void *q, const void *k, const void *v, void *out,
                      const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k, int B, int Hq,
                      int Hkv, int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int d,
                      int causal, float scale, fa_dtype in_dtype, fa_dtype out_dtype,
                      unsigned flags, void *stream) {
    int rc = prefill_common_checks(q, k, v, out, d, in_dtype, out_dtype, scale);
    if (rc != FA_OK) return rc;
    if (!cu_seqlens_q || !cu_seqlens_k) return FA_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(cu_seqlens_q) & 3u) || (reinterpret_cast<uintptr_t>(cu_seqlens_k) & 3u))
        return FA_ERR_ALIGN;
    if (B < 1 || Hq < 1 || Hkv < 1 || total_q < 0 || total_k < 0 || max_seqlen_q < 0 ||
        max_seqlen_k < 0)
        return FA_ERR_SHAPE;
    if (Hq % Hkv != 0) return FA_ERR_SHAPE;
    if (static_cast<long long>(B) * Hq * ((static_cast<long long>(max_seqlen_q) + 255) / 256) > INT_MAX)
        return FA_ERR_SHAPE;
    if (total_q == 0 || max_seqlen_q == 0) return FA_OK;  // no query rows
    const size_t q_bytes = static_cast<size_t>(total_q) * Hq * d * 2;
    const size_t kv_bytes = static_cast<size_t>(total_k) * Hkv * d * 2;
    const size_t out_bytes = static_cast<size_t>(total_q) * Hq * d * dtype_size(out_dtype);
    if (overlaps(out, out_bytes, q, q_bytes) || overlaps(out, out_bytes, k, kv_bytes) ||
        overlaps(out, out_bytes, v, kv_bytes))
        return FA_ERR_ALIAS;
    DeviceInfo dev;
    rc = current_device_info(&dev);
    if (rc != FA_OK) return rc;
    PrefillLaunch a;
    a.q = q;
    a.k = k;
    a.v = v;
    a.out = out;
    a.lse = nullptr;
    a.cu_q = cu_seqlens_q;
    a.cu_k = cu_seqlens_k;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.Nq = max_seqlen_q;
    a.Nk = max_seqlen_k;
    a.total_q = total_q;
    a.total_k = total_k;
    a.d = d;
    a.causal = causal ? 1 : 0;
    a.no_skip = (flags & FA_FLAG_NO_CAUSAL_SKIP) ? 1 : 0;
    a.scale = scale;
    a.in_bf16 = in_dtype == FA_BF16 ? 1 : 0;
    a.out_dtype = out_dtype;
    a.schedule = 1;
    return launch_prefill(a, dev, static_cast<cudaStream_t>(stream));
}

int fa_prefill_plan(int B, int Hq, int Nq, int Nk, int causal, unsigned flags, int num_sms,
                    long long *info, long long *items, int max_items) {
    if (!info) return FA_ERR_NULL;
    if (B < 1 || Hq < 1 || Nq < 1 || Nk < 1 || max_items < 0) return FA_ERR_SHAPE;
    if (static_cast<long long>(B) * Hq * ((static_cast<long long>(Nq) + 255) / 256) > INT_MAX)
        return FA_ERR_SHAPE;
    if (num_sms <= 0) {
        DeviceInfo dev;
        const int rc = current_device_info(&dev);
        if (rc != FA_OK) return rc;
        num_sms = dev.num_sms;
    }
    return plan_prefill(B, Hq, Nq, Nk, causal, (flags & FA_FLAG_NO_CAUSAL_SKIP) ? 1 : 0,
                        schedule_of(flags), num_sms, info, items, max_items);
}

int fa_prefill_backward_ex(const void *q, const void *k, const void *v, const void *out,
                           const void *dout, const float *lse, void *dq, void *dk, void *dv, int B,
                           int H, int Hkv, int N, int d, int causal, float scale, fa_dtype in_dtype,
                           fa_dtype grad_dtype, unsigned flags, void *stream) {
    if (!q || !k || !v || !out || !dout || !lse || !dq || !dk || !dv) return FA_ERR_NULL;
    if (B < 1 || H < 1 || Hkv < 1 || N < 1 || H % Hkv != 0 ||
        static_cast<long long>(B) * H * N > INT_MAX)
        return FA_ERR_SHAPE;
    if (d != 64 && d != 128) return FA_ERR_HEAD_DIM;
    if (in_dtype != FA_F16 && in_dtype != FA_BF16) return FA_ERR_DTYPE;
    if (grad_dtype != FA_F16 && grad_dtype != FA_BF16 && grad_dtype != FA_F32) return FA_ERR_DTYPE;
    if (misaligned(q) || misaligned(k) || misaligned(v) || misaligned(out) || misaligned(dout) ||
        misaligned(dq) || misaligned(dk) || misaligned(dv) || (reinterpret_cast<uintptr_t>(lse) & 3u))
        return FA_ERR_ALIGN;
    if (!std::isfinite(scale)) return FA_ERR_SCALE;
    const size_t in_bytes = static_cast<size_t>(B) * H * N * d * 2;
    const size_t kv_bytes = static_cast<size_t>(B) * Hkv * N * d * 2;
    const size_t gq_bytes = static_cast<size_t>(B) * H * N * d * dtype_size(grad_dtype);
    const size_t gkv_bytes = static_cast<size_t>(B) * Hkv * N * d * dtype_size(grad_dtype);
    const size_t lse_bytes = static_cast<size_t>(B) * H * N * 4;
    const void *ins[6] = {q, k, v, out, dout, lse};
    const size_t in_sz[6] = {in_bytes, kv_bytes, kv_bytes, in_bytes, in_bytes, lse_bytes};
    void *gs[3] = {dq, dk, dv};
    const size_t g_sz[3] = {gq_bytes, gkv_bytes, gkv_bytes};
    for (int g = 0; g < 3; ++g) {
        for (int i = 0; i < 6; ++i)
            if (overlaps(gs[g], g_sz[g], ins[i], in_sz[i])) return FA_ERR_ALIAS;
        for (int h = g + 1; h < 3; ++h)
            if (overlaps(gs[g], g_sz[g], gs[h], g_sz[h])) return FA_ERR_ALIAS;
    }
    DeviceInfo dev;
    int rc = current_device_info(&dev);
    if (rc != FA_OK) return rc;
    BackwardLaunch a;
    a.q = q;
    a.k = k;
    a.v = v;
    a.out = out;
    a.dout = dout;
    a.lse = lse;
    a.dq = dq;
    a.dk = dk;
    a.dv = dv;
    a.B = B;
    a.H = H;
    a.Hkv = Hkv;
    a.N = N;
    a.d = d;
    a.causal = causal ? 1 : 0;
    a.scale = scale;
    a.in_bf16 = in_dtype == FA_BF16 ? 1 : 0;
    a.grad_dtype = grad_dtype;
    a.num_sms = dev.num_sms;
    a.recompute_dq = (flags & FA_BWD_RECOMPUTE_DQ) ? 1 : 0;
    return launch_backward(a, static_cast<cudaStream_t>(stream));
}

int fa_prefill_backward(const void *q, const void *k, const void *v, const void *out,
                        const void *dout, const float *lse, void *dq, void *dk, void *dv, int B,
                        int H, int Hkv, int N, int d, int causal, float scale, fa_dtype in_dtype,
                        fa_dtype grad_dtype, void *stream) {
    return fa_prefill_backward_ex(q, k, v, out, dout, lse, dq, dk, dv, B, H, Hkv, N, d, causal, scale,
                                  in_dtype, grad_dtype, FA_BWD_FLAG_NONE, stream);
}

int fa_prefill_ex(const void *q, const void *k, const void *v, void *out, int B, int H, int N,
                  int d, int causal, float scale, fa_dtype in_dtype, fa_dtype out_dtype,
                  void *stream) {
    return fa_prefill_gqa(q, k, v, out, B, H, H, N, N, d, causal, scale, in_dtype, out_dtype,
                          FA_FLAG_NONE, stream);
}

int fa_prefill(const void *q, const void *k, const void *v, void *out, int B, int H, int N, int d,
               int causal, float scale, void *stream) {
    return fa_prefill_ex(q, k, v, out, B, H, N, d, causal, scale, FA_F16, FA_F16, stream);
}

int fa_decode_chunk_len(int max_len, int num_splits) {
    if (max_len < 1 || num_splits < 1) return -FA_ERR_SHAPE;
    int chunk = 0;
    decode_effective_splits(max_len, num_splits, &chunk);
    return chunk;
}

namespace {
// About `per_sm` CTAs per SM over the whole (b, row, chunk) grid, and no CTA
// longer than 512 rows, so that ragged lengths do not leave a few long CTAs
// running alone at the end.
int choose_splits(int B, long long rows, int max_len, int num_sms, int per_sm) {
    long long splits = ceil_div(static_cast<long long>(per_sm) * num_sms, B * rows);
    const long long max_splits = ceil_div(max_len, kDecodeRowAlign);
    const long long min_splits = ceil_div(max_len, kDecodeAutoMaxChunk);
    if (splits > max_splits) splits = max_splits;
    if (splits < min_splits) splits = min_splits;
    if (splits < 1) splits = 1;
    return decode_effective_splits(max_len, static_cast<int>(splits), nullptr);
}
}  // namespace

int fa_decode_splits_for_sms(int B, int Hq, int Hkv, int max_len, int num_sms) {
    if (B < 1 || Hq < 1 || Hkv < 1 || max_len < 1 || Hq % Hkv != 0 || num_sms < 1)
        return -FA_ERR_SHAPE;
    // Plain decode: about three CTAs per SM (the pages' rule has two; three measured
    // 11 us against 13 at B = 1 and the same at B = 8 and 32).
    if (Hq == Hkv) return choose_splits(B, Hq, max_len, num_sms, 3);
    // A grouped CTA does up to 8 heads' arithmetic per row it loads, so it is
    // latency- rather than bandwidth-bound: aim for about 5 CTAs per SM
    // (measured best at B = 8 and 32 with 14 query over 2 cache heads).
    const long long rows = static_cast<long long>(Hkv) * decode_group_slices(Hq / Hkv);
    return choose_splits(B, rows, max_len, num_sms, 5);
}

namespace {
// SM count of a device ordinal (< 0: the current device), or a negative status.
int device_sms(int device) {
    cudaError_t e;
    if (device < 0 && (e = cudaGetDevice(&device)) != cudaSuccess) return -cuda_fail(e);
    int sms = 0;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device)) != cudaSuccess)
        return -cuda_fail(e);
    return sms;
}
}  // namespace

int fa_decode_gqa_choose_splits(int B, int Hq, int Hkv, int max_len, int device) {
    if (B < 1 || Hq < 1 || Hkv < 1 || max_len < 1 || Hq % Hkv != 0) return -FA_ERR_SHAPE;
    const int sms = device_sms(device);
    if (sms < 0) return sms;
    return fa_decode_splits_for_sms(B, Hq, Hkv, max_len, sms);
}

int fa_decode_choose_splits(int B, int H, int max_len, int device) {
    return fa_decode_gqa_choose_splits(B, H, H, max_len, device);
}

size_t fa_decode_workspace_bytes(int B, int H, int max_len, int d, int num_splits) {
    if (B < 1 || H < 1 || max_len < 1 || num_splits < 1) return 0;
    if (d != 64 && d != 128) return 0;
    const int splits = decode_effective_splits(max_len, num_splits, nullptr);
    const long long bh = static_cast<long long>(B) * H;
    return ws_ml_bytes(bh, splits) + static_cast<size_t>(bh) * splits * d * 4;
}

int fa_decode_gqa(const void *q, const void *k_cache, const void *v_cache, const int32_t *seq_lens,
                  void *out, int B, int Hq, int Hkv, int max_len, int d, float scale,
                  fa_dtype in_dtype, fa_dtype out_dtype, int num_splits, void *workspace,
                  size_t workspace_bytes, void *stream) {
    if (!q || !k_cache || !v_cache || !seq_lens || !out) return FA_ERR_NULL;
    if (B < 1 || Hq < 1 || Hkv < 1 || max_len < 1 || Hq % Hkv != 0) return FA_ERR_SHAPE;
    if (static_cast<long long>(B) * Hkv * max_len > INT_MAX || static_cast<long long>(B) * Hq > INT_MAX)
        return FA_ERR_SHAPE;
    if (d != 64 && d != 128) return FA_ERR_HEAD_DIM;
    if (in_dtype != FA_F16 && in_dtype != FA_BF16) return FA_ERR_DTYPE;
    if (out_dtype != FA_F16 && out_dtype != FA_BF16 && out_dtype != FA_F32) return FA_ERR_DTYPE;
    if (misaligned(q) || misaligned(k_cache) || misaligned(v_cache) || misaligned(out) ||
        (reinterpret_cast<uintptr_t>(seq_lens) & 3u) != 0 || (workspace && misaligned(workspace)))
        return FA_ERR_ALIGN;
    if (!std::isfinite(scale)) return FA_ERR_SCALE;
    const long long max_splits = ceil_div(max_len, kDecodeRowAlign);
    if (num_splits < 0 || num_splits > max_splits) return FA_ERR_SPLITS;
    const size_t bhq = static_cast<size_t>(B) * Hq;
    const size_t out_bytes = bhq * d * dtype_size(out_dtype);
    const size_t cache_bytes = static_cast<size_t>(B) * Hkv * static_cast<size_t>(max_len) * d * 2;
    if (overlaps(out, out_bytes, q, bhq * d * 2) || overlaps(out, out_bytes, k_cache, cache_bytes) ||
        overlaps(out, out_bytes, v_cache, cache_bytes) ||
        overlaps(out, out_bytes, seq_lens, static_cast<size_t>(B) * 4))
        return FA_ERR_ALIAS;

    int splits = num_splits;
    if (splits == 0) {
        splits = fa_decode_gqa_choose_splits(B, Hq, Hkv, max_len, -1);
        if (splits < 0) return -splits;
    }
    int chunk = 0;
    splits = decode_effective_splits(max_len, splits, &chunk);
    // A CTA keeps the scores of its chunk for up to 4 query heads (2 or 4
    // rows of shared memory) within 192 KB.
    const int group = Hq / Hkv;
    const int slices = decode_group_slices(group);
    const int gper = (group + slices - 1) / slices;
    const int rows = group == 1 ? 1 : (gper <= 2 ? 2 : 4);
    if (static_cast<long long>(chunk) * rows > kDecodeMaxChunk) return FA_ERR_SPLITS;
    const size_t need = fa_decode_workspace_bytes(B, Hq, max_len, d, splits);
    if (workspace && workspace_bytes < need) return FA_ERR_WORKSPACE;

    DeviceInfo dev;
    int rc = current_device_info(&dev);
    if (rc != FA_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    void *ws = workspace;
    if (!ws) {
        cudaError_t e = scratch_alloc(&ws, need, st);
        if (e != cudaSuccess) {
            cuda_fail(e);
            return FA_ERR_WORKSPACE;
        }
    }
    DecodeLaunch a;
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.seq_lens = seq_lens;
    a.out = out;
    a.B = B;
    a.H = Hq;
    a.Hkv = Hkv;
    a.max_len = max_len;
    a.d = d;
    a.scale = scale;
    a.in_bf16 = in_dtype == FA_BF16 ? 1 : 0;
    a.out_dtype = out_dtype;
    a.num_splits = splits;
    a.chunk = chunk;
    a.partial_ml = static_cast<float *>(ws);
    a.partial_acc = reinterpret_cast<float *>(static_cast<char *>(ws) +
                                              ws_ml_bytes(static_cast<long long>(bhq), splits));
    rc = launch_decode(a, dev, st);
    if (!workspace) {
        cudaError_t e = scratch_free(ws, st);
        if (rc == FA_OK && e != cudaSuccess) rc = cuda_fail(e);
    }
    return rc;
}

int fa_decode_ex(const void *q, const void *k_cache, const void *v_cache, const int32_t *seq_lens,
                 void *out, int B, int H, int max_len, int d, float scale, fa_dtype in_dtype,
                 fa_dtype out_dtype, int num_splits, void *workspace, size_t workspace_bytes,
                 void *stream) {
    return fa_decode_gqa(q, k_cache, v_cache, seq_lens, out, B, H, H, max_len, d, scale, in_dtype,
                         out_dtype, num_splits, workspace, workspace_bytes, stream);
}

int fa_decode(const void *q, const void *k_cache, const void *v_cache, const int32_t *seq_lens,
              void *out, int B, int H, int max_len, int d, float scale, void *stream) {
    return fa_decode_ex(q, k_cache, v_cache, seq_lens, out, B, H, max_len, d, scale, FA_F16,
                        FA_F16, 0, nullptr, 0, stream);
}

}  // extern "C"
