/*
 * gqa.h — C ABI of the B300 (sm_103a) grouped-query attention decode library
 * (libgqa_b300.so).
 *
 * The operation.  One decode step of grouped-query attention: Hq query heads
 * share Hkv key/value heads; query head h reads KV head floor(h / G) with
 * G = Hq / Hkv, so heads 0..G-1 share KV head 0, heads G..2G-1 share KV head 1,
 * and so on ("Llama-2 70B uses 64 query heads, how many KV heads does it
 * actually keep?", What the choice does to attention; "GQA, decode the
 * acronym and describe its KV sharing pattern").  For every sequence b and
 * query head h the new token's query attends over the L_b = seq_lens[b] cached
 * tokens of its KV head with ordinary scaled dot-product attention:
 *
 *     s_t   = scale * dot(q[b,h,:], K[b,kvh,t,:])        t < L_b
 *     w     = softmax(s)
 *     out[b,h,:] = sum_t w_t * V[b,kvh,t,:]
 *
 * ("Grouped Query Attention (GQA): Efficient Multi-Head Attention", Worked
 * example 2: score = q.k / sqrt(head_dim), softmax, weighted sum of values; the
 * decode step attends over the cached K/V of all prior tokens, The
 * bottleneck).  G = 1 is multi-head attention and Hkv = 1 is multi-query
 * attention (same page, Two extremes).  The cache is read once per KV head and
 * serves all G query heads of its group; it is never expanded to Hq heads
 * ("Grouped Query Attention: Why 8 KV Heads Decide Your Batch Size", Why does
 * GQA speed up decode, and the repeat_kv trap).
 *
 * Layout (all row-major, contiguous, in DEVICE memory owned by the caller):
 *     q, out      [B, Hq, D]
 *     k/v cache   [B, Hkv, Smax, D]   valid prefix t < seq_lens[b]
 *     seq_lens    [B] int32
 *     k/v scales  [B, Hkv] fp32        (FP8 cache only)
 * Positions t >= seq_lens[b] are never used (they may hold anything, NaN
 * included).  seq_lens values are read on the device and never copied to the
 * host; a value below 0 counts as 0 and a value above Smax as Smax.  A
 * sequence with no valid token produces an all-zero output row.  The caller
 * appends the current token to the cache before the call.
 *
 * Numerics.  Products and sums are accumulated in fp32; the output is rounded
 * to nearest-even into the q/out dtype.  Results do not depend on run order
 * (no floating-point atomics): the same inputs on the same device give
 * bit-identical outputs.
 *
 * Execution.  Every compute call is asynchronous on `stream` (a cudaStream_t;
 * NULL means the legacy default stream) and never synchronises with the host.
 * The library keeps a small scratch buffer per (device, stream) for the
 * split-sequence partial results; it is allocated on the first call that needs
 * it (stream-ordered, from the device's default memory pool) and kept for
 * later calls (gqa_release_stream frees it).  Calls on one stream may follow
 * each other freely; calls that share a stream must not run concurrently
 * from several host threads.
 *
 * Errors.  Argument checks run on the host before anything is launched and
 * return GQA_ERR_INVALID_ARG or GQA_ERR_UNSUPPORTED without touching the GPU.
 * A CUDA error from a launch or an allocation returns GQA_ERR_CUDA.  No C++
 * exception crosses this interface.  The library keeps no pointer to caller
 * memory after a call returns.
 */
#ifndef GQA_B300_GQA_H_
#define GQA_B300_GQA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GQA_OK = 0,
  GQA_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size, bad scale  */
  GQA_ERR_UNSUPPORTED = 2, /* valid request this build does not implement   */
  GQA_ERR_CUDA = 3,        /* a CUDA call failed (launch, allocation, ...)  */
  GQA_ERR_DEVICE = 4       /* a kernel reported a fault: see gqa_device_errors */
} gqa_status;

typedef enum {
  GQA_F16 = 0,  /* IEEE binary16                                  */
  GQA_BF16 = 1, /* bfloat16                                       */
  GQA_E4M3 = 2, /* OCP FP8 E4M3 ("e4m3fn"), cache elements only   */
  GQA_E5M2 = 3  /* OCP FP8 E5M2, cache elements only             */
} gqa_dtype;

/*
 * gqa_decode — one GQA decode step with a 16-bit cache.
 *
 *   q        [B, Hq, D]        dtype, device, 16-byte aligned
 *   k_cache  [B, Hkv, Smax, D] dtype, device, 16-byte aligned
 *   v_cache  [B, Hkv, Smax, D] dtype, device, 16-byte aligned
 *   seq_lens [B] int32, device, 4-byte aligned
 *   scale    softmax scale, finite and > 0 (1/sqrt(D) by convention)
 *   out      [B, Hq, D]        dtype, device, 16-byte aligned; fully written
 *   B >= 1, Hkv >= 1, Hq % Hkv == 0, Smax >= 1, D in {64, 128}
 *   dtype    GQA_F16 or GQA_BF16 (q, caches and out share it)
 *
 * Returns GQA_OK once the work is enqueued on `stream`.
 */
gqa_status gqa_decode(const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* seq_lens, float scale, void* out, int B,
                      int Hq, int Hkv, int Smax, int D, gqa_dtype dtype,
                      void* stream);

/*
 * gqa_decode_fp8 — the same step with an 8-bit floating-point cache and one
 * fp32 scale per (sequence, KV head) for K and one for V ("Grouped-Query
 * Attention: How Sharing KV Heads Shrinks Inference Memory", FP8 KV cache: an
 * 8-bit cache with scaling factors, e4m3 or e5m2, halving the bytes read per
 * step).  The cached value of element x of K[b, j] is
 * decode(x) * k_scale[b*Hkv + j] (likewise for V).
 *
 *   k_cache, v_cache [B, Hkv, Smax, D] 8-bit codes, device, 16-byte aligned
 *   k_scale, v_scale [B, Hkv] fp32, device, 4-byte aligned, finite
 *   kv_dtype         GQA_E4M3 (OCP E4M3, max 448) or GQA_E5M2 (OCP E5M2,
 *                    max 57344): the code format of both caches
 *   qo_dtype         GQA_F16 or GQA_BF16: the dtype of q and out
 * Other arguments as for gqa_decode.
 */
gqa_status gqa_decode_fp8(const void* q, const void* k_cache,
                          const void* v_cache, const float* k_scale,
                          const float* v_scale, const int32_t* seq_lens,
                          float scale, void* out, int B, int Hq, int Hkv,
                          int Smax, int D, gqa_dtype kv_dtype,
                          gqa_dtype qo_dtype, void* stream);

/*
 * gqa_decode_chunk — T new tokens per sequence at once (chunked prefill,
 * speculative decoding): the T tokens are the last T of the L_b =
 * seq_lens[b] cached tokens (appended before the call), and new token i
 * (0-based) attends causally to cached tokens t <= L_b - T + i (scaled
 * dot-product attention with is_causal=True and GQA, "Grouped Query
 * Attention: Why 8 KV Heads Decide Your Batch Size", The repeat_kv trap).
 * T = 1 is gqa_decode.  A token that can see no cached token (L_b - T + i <
 * 0) gets an all-zero output row.
 *
 *   q, out  [B, Hq, T, D] dtype, device, 16-byte aligned
 *   T >= 1; other arguments as for gqa_decode (16-bit caches)
 */
gqa_status gqa_decode_chunk(const void* q, const void* k_cache,
                            const void* v_cache, const int32_t* seq_lens,
                            float scale, void* out, int B, int Hq, int Hkv,
                            int T, int Smax, int D, gqa_dtype dtype,
                            void* stream);

/*
 * gqa_append_kv — the step before the decode: writes the new token's K and V
 * rows of every KV head into the cache at position L_b = seq_lens[b] and sets
 * seq_lens[b] = L_b + 1 ("Grouped Query Attention (GQA): Efficient Multi-Head
 * Attention", The bottleneck: the cache grows by one token per step).
 *
 *   k_new, v_new     [B, Hkv, D] in_dtype (GQA_F16 / GQA_BF16), device,
 *                    16-byte aligned
 *   k_cache, v_cache [B, Hkv, Smax, D] cache_dtype, device, 16-byte aligned:
 *                    in_dtype (rows copied as they are), or GQA_E4M3 /
 *                    GQA_E5M2 (rows quantised)
 *   k_scale, v_scale [B, Hkv] fp32, device, read and updated (8-bit caches
 *                    only; may be NULL otherwise)
 *   seq_lens         [B] int32, device, read and incremented
 *   D in {64, 128}
 *
 * 8-bit caches ("Grouped-Query Attention: How Sharing KV Heads Shrinks
 * Inference Memory", FP8 KV cache: scaling factors) decide every code in fp32
 * (IEEE division, round to nearest even, clamped to the format's largest
 * value), per (sequence, KV head) and tensor: with a = max |x| of the new
 * row, an unset scale (<= 0) becomes a / MAX (1 if a == 0; earlier codes are
 * left as they are); otherwise the scale doubles until a / scale <= MAX and,
 * if it grew, the earlier codes are re-encoded with the power-of-two ratio
 * old / new (exact except below the format's normal range); the new codes
 * are x / scale.  MAX is 448 (E4M3) or 57344 (E5M2).
 *
 * A sequence with seq_lens[b] >= Smax is left unchanged and sets bit 2 of
 * gqa_device_errors; a negative length counts as 0.  Asynchronous on
 * `stream`; one kernel.
 */
gqa_status gqa_append_kv(const void* k_new, const void* v_new, void* k_cache,
                         void* v_cache, float* k_scale, float* v_scale,
                         int32_t* seq_lens, int B, int Hkv, int Smax, int D,
                         gqa_dtype in_dtype, gqa_dtype cache_dtype,
                         void* stream);

/*
 * gqa_decode_paged — gqa_decode over a paged KV cache: the cache lives in a
 * pool of fixed-size pages and a block table maps each sequence's token
 * ranges to pages ("Grouped-Query Attention: How Sharing KV Heads Shrinks
 * Inference Memory", Serving knobs: KV blocks; the paged kernels of serving
 * engines that "Grouped Query Attention: Why 8 KV Heads Decide Your Batch
 * Size" names in the repeat_kv trap).  Same arithmetic and output as
 * gqa_decode on the cache the pages describe.
 *
 *   k_pages, v_pages [num_pages, Hkv, page_size, D] dtype, device, 16-byte
 *                    aligned: page p holds page_size consecutive tokens of
 *                    every KV head of one sequence
 *   block_table      [B, max_pages] int32, device, 4-byte aligned: entry
 *                    (b, i) is the page holding tokens [i*page_size,
 *                    (i+1)*page_size) of sequence b; only entries
 *                    i < ceil(seq_lens[b] / page_size) are read, and each
 *                    must be in [0, num_pages)
 *   seq_lens         [B] int32, device: valid tokens, clamped to
 *                    [0, max_pages * page_size]
 *   page_size        a multiple of 64 (GQA_ERR_UNSUPPORTED otherwise)
 *   dtype            GQA_F16 or GQA_BF16
 * Other arguments as for gqa_decode.  A block-table entry outside
 * [0, num_pages) is not dereferenced: page 0 is read instead and bit 1 of
 * gqa_device_errors is set.
 */
gqa_status gqa_decode_paged(const void* q, const void* k_pages,
                            const void* v_pages, const int32_t* block_table,
                            const int32_t* seq_lens, float scale, void* out,
                            int B, int Hq, int Hkv, int num_pages,
                            int page_size, int max_pages, int D,
                            gqa_dtype dtype, void* stream);

/*
 * gqa_decode_static — gqa_decode without any device allocation.
 *
 * The pages have no counterpart to this call.  It is for callers that cannot
 * let a library allocate GPU memory while it runs: serving engines that
 * reserve the device's memory for their own pool at start-up and allow no
 * allocation behind their back afterwards, and latency-critical decode loops
 * in which an allocation could stall or fail at the wrong moment.  gqa_decode
 * keeps a growable scratch buffer per stream that it allocates on first use;
 * this entry point instead takes its scratch (the split partial results and
 * their arrival counters) from one fixed 16 MiB array that the library keeps
 * in static device memory on every GPU that loads it, until the process
 * exits.  It calls no cudaMalloc, cudaFree or other allocating routine.
 *
 * Arguments, layout, numerics and errors: as gqa_decode; the caller provides
 * every input and the output.  In addition:
 *  - Size limit.  A request whose scratch does not fit in the 16 MiB array
 *    returns GQA_ERR_UNSUPPORTED before anything is enqueued.  The scratch
 *    is about (blocks + B*Hkv*ceil(G/64)) x rows x D x 4 bytes, rows = 16, 32
 *    or 64 by G: e.g. B=8, Hq=64, Hkv=8, D=128 needs about 1.8 MB on a
 *    148-SM GPU, while B=32, Hq=Hkv=64, D=128 needs 18 MB and is refused.
 *  - Set-up.  The first call on each device looks up the device address of
 *    the array (once per device, with that device current).  Make that first
 *    call before any stream capture.
 *  - Sharing.  Every call on a device uses the same array, which keeps what
 *    the previous call left in it; each call first clears the part that must
 *    start at zero (an asynchronous memset on `stream`, then the kernel).
 *    Calls whose execution overlaps on the GPU (e.g. on two streams with no
 *    ordering between them) race on the array and give wrong results.
 *  - Fault flags raised by its kernel are not reported by gqa_device_errors.
 */
gqa_status gqa_decode_static(const void* q, const void* k_cache,
                             const void* v_cache, const int32_t* seq_lens,
                             float scale, void* out, int B, int Hq, int Hkv,
                             int Smax, int D, gqa_dtype dtype, void* stream);

/*
 * gqa_kv_bytes_per_token — KV-cache bytes one token occupies across a model:
 * 2 (K and V) x layers x kv_heads x head_dim x bytes_per_elem ("Grouped Query
 * Attention: Why 8 KV Heads Decide Your Batch Size", TL;DR; e.g. 327,680 B =
 * 320 KiB for 80 layers, 8 KV heads, head_dim 128, fp16).  Returns 0 if an
 * argument is not positive.  Host only.
 */
size_t gqa_kv_bytes_per_token(int layers, int kv_heads, int head_dim,
                              int bytes_per_elem);

/* gqa_status_string — static, NUL-terminated description of a status. */
const char* gqa_status_string(gqa_status status);

/*
 * gqa_device_errors — synchronises `stream`, then returns (and clears) the
 * fault flags the kernels raised on it since the last query: 0 when none.
 * Bit 0: a pipeline wait gave up after its time limit (the outputs of that
 * call are unspecified; the kernel still finished and left the GPU usable).
 * Bit 1: a paged call met a block-table entry outside [0, num_pages).
 * Bit 2: an append found a sequence's cache full.
 * Returns GQA_ERR_CUDA if the synchronisation fails.
 *
 * Recovery after bit 0.  A call whose wait gave up may leave some of the
 * stream's split-combine arrival counters non-zero.  Later calls are not
 * affected: every call tags its counts with a generation of its own and
 * ignores counts another call left.  The one exception is a call captured in
 * a CUDA graph, whose replays share one generation; when this function finds
 * bit 0 set it therefore also clears the stream's counters, after which
 * replays are correct again.
 */
gqa_status gqa_device_errors(void* stream, uint32_t* flags);

/*
 * gqa_set_kernel_path — test and tuning hook: which kernel the decode calls
 * launch (process-wide; host only).  0 (the default): the tensor-core kernel
 * (fifth-generation tensor core, accumulators in tensor memory) for units of
 * more than 32 query rows per KV head with a 16-bit cache and head_dim 128
 * (multi-query attention, wide groups, multi-token chunks of wide groups;
 * contiguous or paged), the warp-level mma kernel otherwise.  1: the
 * warp-level kernel everywhere.  2: the tensor-core kernel wherever it
 * applies, units of up to 32 rows included.  The result is the same within the stated tolerance
 * (fp32 accumulation both ways); other values count as 0.
 */
void gqa_set_kernel_path(int path);

/*
 * gqa_set_tuning — test and tuning hook (process-wide; host only): turns
 * single design choices of the decode calls off, for A/B measurements.  An
 * OR of GQA_TUNE_* bits; 0 (the default) keeps every choice.
 *   GQA_TUNE_NO_L2_WARMUP    no L2 prefetch of a block's first tiles and
 *                            first query rows before its wait for the
 *                            previous kernel in the stream
 *   GQA_TUNE_NO_CLUSTER      the tensor-core kernel never launches thread-
 *                            block clusters (units split between blocks
 *                            always merge through global memory)
 *   GQA_TUNE_NO_NARROW_ROWS  8-bit caches with at most 8 query rows per unit
 *                            take the 16-row operand path
 * The result is the same within the stated tolerance; unknown bits are
 * ignored.
 */
enum {
  GQA_TUNE_NO_L2_WARMUP = 1,
  GQA_TUNE_NO_CLUSTER = 2,
  GQA_TUNE_NO_NARROW_ROWS = 4
};
void gqa_set_tuning(int flags);

/*
 * gqa_set_wait_limit_ns — test hook: the time limit of every pipeline wait in
 * the decode kernels launched afterwards (process-wide; host only).  A wait
 * that runs out sets bit 0 of gqa_device_errors, and the kernel stops waiting
 * and finishes.  ns = 0 gives up at the first wait that is not already
 * complete (so a test can make a wait run out without withholding any work);
 * ns < 0 restores the default of 2 seconds.
 */
void gqa_set_wait_limit_ns(long long ns);

/*
 * gqa_set_num_ctas — test and tuning hook: fixes the number of persistent
 * thread blocks the decode kernels launch and makes all of them take part
 * (0 restores the default: one full wave of the device, of which a batch
 * whose sequences all have the same number of 64-token tiles may use a
 * smaller, unit-aligned count).  It changes how the sequence axis is split
 * between blocks, never the result beyond fp32 rounding.  Process-wide; host
 * only.
 */
void gqa_set_num_ctas(int num_ctas);

/*
 * gqa_release_stream — frees the scratch the library keeps for (the current
 * device, `stream`): stream-ordered frees enqueued on `stream`, after the
 * work already on it.  Call it before destroying a stream the library used
 * (the scratch is keyed by the stream handle, which a later stream may
 * reuse), or to return the memory; a later call on the stream allocates it
 * again.  The stream's pending fault flags (gqa_device_errors) are dropped
 * with it.  Returns GQA_OK also when the library holds nothing for the
 * stream, GQA_ERR_CUDA if a free cannot be enqueued.  Host only; must not
 * run concurrently with a compute call on the same stream.
 */
gqa_status gqa_release_stream(void* stream);

/*
 * gqa_last_launch_count — number of kernels the most recent compute call made
 * from this host thread enqueued (0 if it returned before launching).
 */
int gqa_last_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* GQA_B300_GQA_H_ */
