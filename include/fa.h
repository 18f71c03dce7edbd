/*
 * fa.h -- C ABI of libfa_gb300.so: fused scaled-dot-product attention forward
 * (prefill and split-K decode) for one NVIDIA GB300 (sm_103a).
 *
 * What is computed (flash-attention-cuda README, "What is Attention?", "What is
 * Flash Attention?" and the "Kernel design" table):
 *     O = softmax(scale * Q K^T [+ causal mask]) V
 * row by row, tile by tile, with the online-softmax recurrence (a running row
 * maximum m, a running denominator l and a rescaled fp32 accumulator), so the
 * N x N score table is never written to memory.  Inputs are fp16 or bf16, all
 * sums are fp32 ("fp16 in, fp32 accumulate" row of the "Kernel design" table).
 *
 * Conventions shared by every entry point
 *   - Tensors are dense, row-major, head dimension innermost:
 *       prefill q, k, v, out : [B][H][N][d]
 *       decode  q, out       : [B][H][1][d]
 *       decode  caches       : [B][H][max_len][d]
 *   - Every pointer is a device pointer owned by the caller, 16-byte aligned.
 *     The library keeps no pointer after the call returns.  Work is enqueued on
 *     `stream` (a cudaStream_t passed as void*; NULL = the legacy default
 *     stream) and runs asynchronously: inputs must stay alive and unmodified,
 *     and `out` untouched, until that stream work has completed.
 *   - `out` must not overlap any input.
 *   - Status: FA_OK (0) or an fa_status code, returned synchronously for bad
 *     arguments and for launch failures.  A fault during execution surfaces at
 *     the caller's next synchronisation, as for any CUDA call.  Nothing throws
 *     across this ABI.  On any non-zero status no work was enqueued.
 *   - The library runs only on compute capability 10.3 (sm_103a); any other
 *     device returns FA_ERR_ARCH.  There is no fallback path.
 *   - All entry points are thread-safe; the only global state is a per-device
 *     attribute cache and a device-side watchdog status word.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { FA_F16 = 0, FA_BF16 = 1, FA_F32 = 2 } fa_dtype;

typedef enum {
    FA_OK = 0,
    FA_ERR_NULL = 1,       /* a required pointer is NULL                          */
    FA_ERR_SHAPE = 2,      /* B, H, N or max_len < 1, or a size overflows int32   */
    FA_ERR_HEAD_DIM = 3,   /* d is not a supported head dimension                 */
    FA_ERR_DTYPE = 4,      /* unsupported input/output dtype combination          */
    FA_ERR_ALIGN = 5,      /* a pointer is not 16-byte aligned                    */
    FA_ERR_SCALE = 6,      /* scale is NaN or infinite                            */
    FA_ERR_ARCH = 7,       /* current device is not compute capability 10.3       */
    FA_ERR_WORKSPACE = 8,  /* caller workspace too small, or allocation failed    */
    FA_ERR_CUDA = 9,       /* a CUDA runtime call failed: see fa_last_cuda_error  */
    FA_ERR_WATCHDOG = 10,  /* a device-side wait ran out (see fa_device_status)   */
    FA_ERR_SEQ_LEN = 11,   /* a device-resident length was out of range and was
                              clamped (reported by fa_device_status only)         */
    FA_ERR_ALIAS = 12,     /* out overlaps an input                               */
    FA_ERR_SPLITS = 13     /* num_splits outside [0, ceil(max_len / 64)]          */
} fa_status;

/* Flags for fa_prefill_gqa and the other prefill forms that take `flags`. */
#define FA_FLAG_NONE 0u
/* Causal only: run the key-tile loop over every tile instead of stopping at
 * the diagonal (tiles above it are then fully masked).  The result must be
 * bit-identical to the default ("Kernel design" table, causal tile skipping,
 * "verified bit-identical"); the flag exists so that tests can check that. */
#define FA_FLAG_NO_CAUSAL_SKIP 1u
/* Work schedule of the prefill kernel (performance tuning and tests; the
 * result stays within the tolerance either way and is bit-identical run to run
 * for a given choice).  By default the library picks, from the shapes and the
 * SM count only: one CTA per SM walks whole 256-row query blocks, or, for a
 * dense batch, the key-tile steps of all blocks are cut into equal ranges per
 * CTA ("stream-K") and the blocks cut between CTAs are merged by a second
 * kernel.  UNITS forces the first; STREAM_K asks for the second where it
 * applies (dense batches in which every query row sees at least one key).
 * If both are set, UNITS wins.  Other bits are reserved and ignored. */
#define FA_FLAG_SCHEDULE_UNITS 2u
#define FA_FLAG_SCHEDULE_STREAM_K 4u

/*
 * Prefill (flash-attention-cuda README, "What did I implement?" prompt phase,
 * and "Installation" usage `prefill(q, k, v, causal, scale)`): batched,
 * multi-head attention of N queries over the same N keys.
 *   q, k, v : fp16 inputs [B][H][N][d]
 *   out     : fp16 output [B][H][N][d]
 *   d       : 64 or 128
 *   causal  : nonzero -> key j is visible to query i iff j <= i; tiles wholly
 *             above the diagonal are skipped by loop bounds.
 *   scale   : finite float multiplying Q K^T (0 gives the mean of the visible
 *             value rows; negative values are allowed).
 */
int fa_prefill(const void *q, const void *k, const void *v, void *out,
               int B, int H, int N, int d, int causal, float scale,
               void *stream);

/*
 * Prefill with explicit dtypes (the configurations need bf16 in / bf16 out
 * and fp16 in / fp32 out besides the plain fp16 form).
 *   in_dtype  : FA_F16 or FA_BF16 (q, k and v share it)
 *   out_dtype : FA_F16, FA_BF16 or FA_F32 (rounded to nearest even)
 * Other arguments as fa_prefill.  The library picks the work schedule; the
 * schedule flags are taken by fa_prefill_gqa.  Large problems may take a
 * stream-ordered scratch buffer (at most SMs x 2 x 256 x d x 4 bytes plus 8
 * bytes per row of it) from the library's device memory pool;
 * FA_ERR_WORKSPACE if that allocation fails.
 */
int fa_prefill_ex(const void *q, const void *k, const void *v, void *out,
                  int B, int H, int N, int d, int causal, float scale,
                  fa_dtype in_dtype, fa_dtype out_dtype, void *stream);

/*
 * Prefill with grouped key/value heads and separate query / key lengths
 * (flash-attention-cuda README, "Future work": kernel-side GQA instead of a
 * host-side repeat of the key/value heads; a prompt processed in chunks
 * attends from its newest Nq positions over all Nk keys, as the generation
 * phase of "What did I implement?" does with Nq = 1).
 *   q, out : [B][Hq][Nq][d]      k, v : [B][Hkv][Nk][d]
 *   Hq     : a multiple of Hkv; query head h reads key/value head h / (Hq / Hkv)
 *   causal : the queries are the last Nq positions: query i sees keys
 *            j <= i + (Nk - Nq).  When Nq > Nk the first Nq - Nk rows see no
 *            key and are written as zeros.
 *   flags  : FA_FLAG_* bits (schedule choice and the causal-skip check)
 * Other arguments as fa_prefill_ex.  Errors: FA_ERR_SHAPE when a size is < 1,
 * Hq % Hkv != 0 or an element count exceeds INT_MAX; the others as above.
 */
int fa_prefill_gqa(const void *q, const void *k, const void *v, void *out,
                   int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal,
                   float scale, fa_dtype in_dtype, fa_dtype out_dtype,
                   unsigned flags, void *stream);

/*
 * Prefill on host buffers (the end-to-end form of fa_prefill_gqa): copies q,
 * k and v to the device, computes, and copies the output back, all ordered on
 * `stream`.  The call returns once the work is enqueued; out_host holds the
 * result when the stream reaches that point, and the four host buffers must
 * stay valid until then.  Page-locked (pinned) host memory lets the copies run
 * asynchronously; other host memory works but its copies serialise.
 * The flattened key/value heads (B * Hkv) are cut into up to eight chunks:
 * chunk c's input copies (on a library-owned copy stream shared by all
 * calls), its kernel (on `stream`) and its output copy (on one of four
 * library-owned output streams, taken in turn by successive calls) overlap
 * the neighbouring chunks'.  Only the first chunk's input copies and the last
 * chunk's output copy overlap no kernel, so the chunk sizes ramp up from a
 * small first chunk and back down to a small last one, each chunk holding at
 * least 24 128 x 128 tile products per SM (fewer, larger chunks for short
 * sequences).  Device buffers for q, k, v and out come from the
 * library's stream-ordered pool and go back to it after the last copy.
 *   q_host, out_host : [B][Hq][Nq][d]    k_host, v_host : [B][Hkv][Nk][d]
 * Other arguments as fa_prefill_gqa.  Errors as fa_prefill_gqa, plus
 * FA_ERR_WORKSPACE when the device buffers cannot be allocated.  Calls from
 * several host threads are serialised while they enqueue.
 */
int fa_prefill_host(const void *q_host, const void *k_host, const void *v_host,
                    void *out_host, int B, int Hq, int Hkv, int Nq, int Nk, int d,
                    int causal, float scale, fa_dtype in_dtype,
                    fa_dtype out_dtype, unsigned flags, void *stream);

/*
 * Prefill that also returns, for every query row, the log-sum-exp of its
 * visible scores, lse_i = log sum_j exp(scale q_i.k_j) (natural log; -inf for
 * a row that sees no key).  It is what fa_prefill_backward needs to recompute
 * the weights.  Arguments as fa_prefill_gqa plus
 *   lse : fp32 device array [B][Hq][Nq] (4-byte aligned), or NULL (then this
 *         is fa_prefill_gqa)
 */
int fa_prefill_lse(const void *q, const void *k, const void *v, void *out,
                   float *lse, int B, int Hq, int Hkv, int Nq, int Nk, int d,
                   int causal, float scale, fa_dtype in_dtype,
                   fa_dtype out_dtype, unsigned flags, void *stream);

/*
 * Backward pass of prefill (flash-attention-cuda README, "Future work":
 * training), for square problems (Nq = Nk = N) with H query heads over Hkv
 * key/value heads: given the inputs, the forward output `out`, its gradient
 * `dout` and the forward's `lse`, writes
 *   dq = dL/dq, dk = dL/dk, dv = dL/dv
 * of L = sum(dout * out), with the weights recomputed tile by tile from lse
 * (the N x N weights never reach memory; the score gradients dS do, as the
 * 16-bit table described below).  The gradient of a shared key/value head is the
 * sum over the query heads that read it.  No atomics: the result is
 * bit-identical run to run.
 *   q, out, dout       : 16-bit [B][H][N][d] in in_dtype (out as written by
 *                        fa_prefill_lse with out_dtype == in_dtype)
 *   k, v               : 16-bit [B][Hkv][N][d]; H a multiple of Hkv
 *   lse                : fp32 [B][H][N] from fa_prefill_lse
 *   dq                 : [B][H][N][d], dk, dv : [B][Hkv][N][d], in grad_dtype
 *                        (FA_F16, FA_BF16, FA_F32), accumulated in fp32; none
 *                        may overlap another argument
 *   causal, scale      : as in the forward call
 * Scratch of 8 bytes per query row, with each head's rows rounded up to a
 * multiple of 128, comes from the library's pool.  So does a table of the
 * score gradients dS that the dK/dV pass writes in 16-bit and the dQ pass
 * multiplies by K: ceil(N / 128)^2 x 32 KB per query head, at most 4 GiB.  A
 * larger problem runs both passes in chunks of key/value heads over a table of
 * that size; when one key/value head's blocks alone pass 4 GiB, or the table
 * cannot be allocated, the dQ pass recomputes S and dP instead (as
 * FA_BWD_RECOMPUTE_DQ).  Errors as for
 * prefill: FA_ERR_NULL, FA_ERR_SHAPE, FA_ERR_HEAD_DIM, FA_ERR_DTYPE,
 * FA_ERR_ALIGN, FA_ERR_SCALE, FA_ERR_ALIAS, FA_ERR_WORKSPACE, FA_ERR_ARCH,
 * FA_ERR_CUDA.
 */
int fa_prefill_backward(const void *q, const void *k, const void *v,
                        const void *out, const void *dout, const float *lse,
                        void *dq, void *dk, void *dv, int B, int H, int Hkv, int N,
                        int d, int causal, float scale, fa_dtype in_dtype,
                        fa_dtype grad_dtype, void *stream);

/* Flags for fa_prefill_backward_ex. */
#define FA_BWD_FLAG_NONE 0u
/* The dQ pass recomputes the scores and their gradient tile by tile instead of
 * reading the dS table, and takes no table from the pool.  The result stays
 * within the tolerance either way and is bit-identical run to run for a given
 * choice.  Other bits are reserved and ignored. */
#define FA_BWD_RECOMPUTE_DQ 1u

/* fa_prefill_backward with `flags` (FA_BWD_* bits); same arguments, errors and
 * results otherwise.  fa_prefill_backward is this call with FA_BWD_FLAG_NONE. */
int fa_prefill_backward_ex(const void *q, const void *k, const void *v,
                           const void *out, const void *dout, const float *lse,
                           void *dq, void *dk, void *dv, int B, int H, int Hkv,
                           int N, int d, int causal, float scale,
                           fa_dtype in_dtype, fa_dtype grad_dtype,
                           unsigned flags, void *stream);

/*
 * The schedule fa_prefill_gqa would use for a dense problem on num_sms SMs
 * (num_sms <= 0: the current device's count).  Host arithmetic only, for
 * tuning and tests; nothing runs on a device.
 *   flags : FA_FLAG_NO_CAUSAL_SKIP and the FA_FLAG_SCHEDULE_* bits, as for
 *           the prefill call
 *   info  : 9 values: stream-K (1) or unit by unit (0), CTAs launched, key-tile
 *           steps W of all units, steps per (sequence, head), 256-row query
 *           blocks per head, units cut between CTAs, whole units dealt to
 *           every CTA before the cut ranges (CTA c takes units c + k * CTAs),
 *           the first step S0 of the cut ranges, and 1 when a causal unit
 *           schedule pairs 128-row query tiles i and T - 1 - i (T tiles per
 *           sequence) instead of taking adjacent ones
 *   items : NULL or room for max_items rows of 5 values, one per cut unit:
 *           unit, first CTA, last CTA, the unit's steps, the unit's first step.
 *           Units number (b * Hq + h) * blocks + block; CTA c owns the steps
 *           [S0 + c * (W - S0) / CTAs, S0 + (c + 1) * (W - S0) / CTAs).
 * Returns FA_OK, FA_ERR_NULL (info), FA_ERR_SHAPE (a size < 1).
 */
int fa_prefill_plan(int B, int Hq, int Nq, int Nk, int causal, unsigned flags,
                    int num_sms, long long *info, long long *items, int max_items);

/*
 * Prefill of a packed batch of variable-length sequences.  Sequence b owns
 * query tokens [cu_seqlens_q[b], cu_seqlens_q[b+1]) and key/value tokens
 * [cu_seqlens_k[b], cu_seqlens_k[b+1]); sequences never see each other.
 *   q, out      : [total_q][Hq][d]     k, v : [total_k][Hkv][d]
 *   cu_seqlens_q, cu_seqlens_k : int32 device arrays of B + 1 non-decreasing
 *                 offsets from 0 to total_q / total_k (4-byte aligned).  The
 *                 kernel clamps them to [0, total], so a bad array cannot make
 *                 it write outside `out`; an offset outside [0, total], a
 *                 decreasing pair or a length above max_seqlen_* is recorded as
 *                 FA_ERR_SEQ_LEN in the device status word (fa_device_status).
 *   max_seqlen_q, max_seqlen_k : host upper bounds of the per-sequence
 *                 lengths; rows past max_seqlen_q of a longer sequence are
 *                 left unwritten and keys past max_seqlen_k are ignored.
 *   causal      : per sequence, as fa_prefill_gqa (queries are the last
 *                 positions of their sequence).
 * A sequence with no keys gives zero rows; total_q == 0 returns FA_OK at once.
 * Always scheduled unit by unit.  When the units take more than one round of
 * the SMs (and the batch has at most 4096 (sequence, 256-query block) pairs), a
 * one-CTA kernel on `stream` first sorts those pairs by their work, from the
 * device-resident offsets, into 4 bytes per pair of scratch from the library's
 * pool (FA_ERR_WORKSPACE if that allocation fails), and the units are dealt
 * heaviest first; otherwise no scratch is used.  Either way every unit is
 * computed whole by one CTA, so the output does not depend on the order.  The
 * lengths stay on the device: nothing is copied back to the host.
 */
int fa_prefill_varlen(const void *q, const void *k, const void *v, void *out,
                      const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                      int B, int Hq, int Hkv, int total_q, int total_k,
                      int max_seqlen_q, int max_seqlen_k, int d, int causal,
                      float scale, fa_dtype in_dtype, fa_dtype out_dtype,
                      unsigned flags, void *stream);

/*
 * Split-K decode (flash-attention-cuda README, "What did I implement?"
 * generation phase; "Kernel design" rows "Split-K decode + adaptive chunk"
 * and "Two-pass merge, no atomics"): one query row per (b, h) attends over
 * the first seq_lens[b] rows of its KV cache.  The cache is split into
 * chunks, each chunk yields a partial (m, l, acc), and a second kernel merges
 * the partials in a fixed order, without atomics.
 *   q        : fp16 [B][H][1][d]
 *   k_cache, v_cache : fp16 [B][H][max_len][d]
 *   seq_lens : int32 device array [B]; precondition 1 <= seq_lens[b] <= max_len.
 *              Values are clamped to [0, max_len]; a length of 0 yields a zero
 *              output row.  A value outside [0, max_len] is recorded as
 *              FA_ERR_SEQ_LEN in the device status word, read (and cleared) by
 *              fa_device_status; the call itself has already returned FA_OK,
 *              since the lengths stay on the device.  The check runs in every
 *              build: it is one compare per (b, h) in the merge kernel.
 *   out      : fp16 [B][H][1][d]
 *   d        : 64 or 128
 * The split count is chosen from (B, H, max_len, SM count) only, never from
 * the device-resident lengths, so it needs no device-to-host copy and gives
 * bit-identical results run to run.  The partials workspace is allocated
 * stream-ordered on `stream` from a memory pool the library creates once per
 * device; the pool keeps up to 5 GiB of freed scratch mapped for reuse (the
 * largest backward dS table is 4 GiB).
 */
int fa_decode(const void *q, const void *k_cache, const void *v_cache,
              const int32_t *seq_lens, void *out,
              int B, int H, int max_len, int d, float scale, void *stream);

/*
 * Decode with explicit dtypes, split count and workspace.
 *   in_dtype / out_dtype : as for fa_prefill_ex
 *   num_splits : 0 = automatic (fa_decode_choose_splits), else the number of
 *                key chunks per (b, h), 1 <= num_splits <= ceil(max_len / 64)
 *   workspace  : NULL -> allocated stream-ordered; else a device buffer of at
 *                least fa_decode_workspace_bytes(B, H, max_len, d, splits)
 *                bytes, 16-byte aligned, owned by the caller, not used by any
 *                other work running at the same time.
 */
int fa_decode_ex(const void *q, const void *k_cache, const void *v_cache,
                 const int32_t *seq_lens, void *out,
                 int B, int H, int max_len, int d, float scale,
                 fa_dtype in_dtype, fa_dtype out_dtype, int num_splits,
                 void *workspace, size_t workspace_bytes, void *stream);

/*
 * The automatic split count ("Kernel design" table: choose_decode_split
 * targets about two resident blocks per SM; here three, measured faster on
 * GB300): enough (b, h, chunk) CTAs for three per SM, and chunks of at most
 * 512 rows so that ragged lengths do not
 * leave a few long CTAs running alone.  Host arithmetic on the arguments and
 * the SM count of `device` (a CUDA device ordinal; < 0 = the current device).
 * Returns the split count (>= 1), or a negative fa_status: -FA_ERR_SHAPE on
 * bad sizes, -FA_ERR_CUDA if the device cannot be queried.
 */
int fa_decode_choose_splits(int B, int H, int max_len, int device);

/*
 * The split count that fa_decode_gqa would choose on a GPU with num_sms SMs
 * (Hq == Hkv: plain multi-head decode, the rule of fa_decode_choose_splits).
 * Pure host arithmetic, for tuning and tests; nothing touches a device.
 * Returns the split count, or -FA_ERR_SHAPE on bad arguments (num_sms < 1
 * included).
 */
int fa_decode_splits_for_sms(int B, int Hq, int Hkv, int max_len, int num_sms);

/* Keys per chunk for a given split count: round_up(ceil(max_len/splits), 64). */
int fa_decode_chunk_len(int max_len, int num_splits);

/* Workspace bytes needed by fa_decode_ex for this problem (0 on bad args). */
size_t fa_decode_workspace_bytes(int B, int H, int max_len, int d,
                                 int num_splits);

/*
 * Grouped decode (flash-attention-cuda README, "Future work": kernel-side GQA,
 * instead of repeating the cache heads on the host).  Hq query heads share Hkv
 * cache heads; query head h reads cache head h / (Hq / Hkv).  Each K and V row
 * is read from HBM once for all query heads of its group.
 *   q, out  : [B][Hq][1][d]          k_cache, v_cache : [B][Hkv][max_len][d]
 *   Hq      : a multiple of Hkv (Hq == Hkv is plain multi-head decode and runs
 *             the same kernels as fa_decode_ex)
 *   workspace : NULL or at least fa_decode_workspace_bytes(B, Hq, max_len, d,
 *             splits) bytes, splits being num_splits or, for 0, the value of
 *             fa_decode_gqa_choose_splits(B, Hq, Hkv, max_len, -1)
 * Other arguments, results and errors as fa_decode_ex; in addition
 * FA_ERR_SHAPE when Hq % Hkv != 0, and FA_ERR_SPLITS when a chunk would need
 * more than 192 KB of shared memory for the scores of its query heads
 * (chunk x 4 > 48K rows when a CTA serves 3 or 4 query heads: a group of G
 * query heads is served by ceil(G / 4) CTAs per chunk).
 */
int fa_decode_gqa(const void *q, const void *k_cache, const void *v_cache,
                  const int32_t *seq_lens, void *out,
                  int B, int Hq, int Hkv, int max_len, int d, float scale,
                  fa_dtype in_dtype, fa_dtype out_dtype, int num_splits,
                  void *workspace, size_t workspace_bytes, void *stream);

/* Split count fa_decode_gqa uses for num_splits == 0 on `device` (< 0 = the
 * current device); a negative fa_status as for fa_decode_choose_splits. */
int fa_decode_gqa_choose_splits(int B, int Hq, int Hkv, int max_len, int device);

/*
 * Decode that allocates nothing.  The pages have no counterpart: this entry
 * point exists for callers that cannot allocate device memory while they run
 * -- for example a host that reserves the whole device up front for its own
 * memory pool, a latency-critical serving loop where an allocation may block
 * or synchronise, or a deployment that forbids allocation after start-up.
 * It computes exactly what fa_decode_ex computes (same kernels, same split
 * choice), with the split partials kept in a fixed 4 MiB device array built
 * into the library (fa_decode_noalloc_max_bytes()); every GPU that loads the
 * library holds that array until the process exits.
 *   - Arguments are those of fa_decode_ex, without the workspace.
 *   - A problem whose partials need more than the array holds
 *     (fa_decode_workspace_bytes(...) > fa_decode_noalloc_max_bytes())
 *     returns FA_ERR_WORKSPACE and enqueues nothing.
 *   - The first call on each device looks up the array's device address with
 *     that device current; make that first call before any stream capture.
 *   - All calls share the one array and it keeps the last call's contents.
 *     Nothing in it needs to start at zero (each call writes every partial it
 *     reads), but two calls whose work overlaps on the GPU -- different
 *     streams, or different host threads -- race on it and give wrong results.
 *     Serialise them, e.g. on one stream.
 */
int fa_decode_noalloc(const void *q, const void *k_cache, const void *v_cache,
                      const int32_t *seq_lens, void *out,
                      int B, int H, int max_len, int d, float scale,
                      fa_dtype in_dtype, fa_dtype out_dtype, int num_splits,
                      void *stream);

/* Bytes of the static scratch array behind fa_decode_noalloc. */
size_t fa_decode_noalloc_max_bytes(void);

/* Static text for a status code ("unknown status" for other values). */
const char *fa_status_string(int status);

/* The cudaError_t behind the calling thread's last FA_ERR_CUDA (0 if none). */
int fa_last_cuda_error(void);

/* Device-side status word of the current device: 0, FA_ERR_WATCHDOG after a
 * kernel's bounded wait ran out (this wins when both were recorded), or
 * FA_ERR_SEQ_LEN after a kernel clamped a device-resident length.
 * Synchronises the device.  If reset is nonzero the word is cleared.  Returns
 * a negative value if it cannot be read. */
int fa_device_status(int reset);

/* ---------------------------------------------------------------- diagnostics
 * The calls below have no counterpart in the pages: they exist to test the
 * library's failure detection and its memory use, and to measure the GPU. */

/*
 * Self-test of the bounded waits behind FA_ERR_WATCHDOG.  Launches one CTA of
 * two warps on `stream`.  Warp 0 waits, suspending between polls, on a
 * shared-memory barrier that nothing ever completes, for at most `limit_ns`;
 * warp 1 polls another such barrier with the kernels' own limit (1.5 s) and
 * must give up as soon as warp 0's timeout raises the CTA's abort flag.  The
 * CTA then records FA_ERR_WATCHDOG in the device status word exactly as the
 * attention kernels do at exit.  Nothing else is in flight, so the context
 * stays usable.
 *   limit_ns : 1e3 .. 1e9
 *   result   : device array of 4 int64 (8-byte aligned), written as
 *              [0] 1 if warp 0's wait reported a timeout, [1] 1 if warp 1's
 *              wait returned early on the abort flag, [2] and [3] the
 *              nanoseconds warps 0 and 1 waited (%globaltimer).
 * Errors: FA_ERR_NULL, FA_ERR_ALIGN, FA_ERR_SHAPE (limit out of range),
 * FA_ERR_ARCH, FA_ERR_CUDA.
 */
int fa_watchdog_selftest(long long limit_ns, long long *result, void *stream);

/*
 * Bytes of the library's stream-ordered scratch pool on the current device:
 * out[0] reserved now, out[1] reserved high-water mark, out[2] in use now,
 * out[3] in-use high-water mark; all 0 when the pool has never been used on
 * this device (nothing is created by this call).  With reset_high nonzero
 * both high-water marks are reset after they are read.  Does not
 * synchronise: sizes of stream-ordered work not yet run are not counted.
 */
int fa_pool_stats(long long *out, int reset_high);

/*
 * Read-bandwidth probe: streams `bytes` (a positive multiple of 16) from the
 * device buffer `src` (16-byte aligned) with the decode kernels' 16-byte
 * non-caching loads, over a grid sized to the SM count, and stores the XOR of
 * all its 32-bit words in *xor_out (device, 4-byte aligned; it is first set
 * to 0 on `stream`).  The XOR lets a caller check that every byte was read.
 * Errors: FA_ERR_NULL, FA_ERR_ALIGN, FA_ERR_SHAPE, FA_ERR_ARCH, FA_ERR_CUDA.
 */
int fa_read_probe(const void *src, size_t bytes, uint32_t *xor_out, void *stream);

/* ABI version: major * 10000 + minor * 100 + patch. */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
