/*
 * dms.h -- C ABI of the DMS decode-attention library (libdms.so).
 *
 * Dynamic Memory Sparsification (DMS) keeps, for every (sequence, KV head), a
 * compacted KV cache: each appended token carries a binary eviction decision,
 * and a token marked for eviction leaves the cache w steps after it was
 * appended ("Inference-Time Hyper-Scaling with KV Cache Compression", AI
 * research-map summary, section "Approach": a learned per-head binary eviction
 * decision whose eviction is executed after a delay window; the window is 16
 * tokens in that summary's "Measured effects reported in the paper" table).
 * Decoding is bound by reading the KV cache from memory (same paper, notes
 * page, section "研究背景与动机": every autoregressive step reads the whole
 * cache), so the library streams only the retained K/V bytes.
 *
 * Conventions for every call:
 *  - Tensor arguments are DEVICE pointers on the cache's device, caller-owned,
 *    contiguous, row-major, 16-byte aligned.  They are read or written in
 *    stream order and are not retained after the enqueued work completes.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  All work of a
 *    cache must be enqueued on one stream; a cache is not thread-safe.
 *  - Return value: DMS_OK (0) or a negative DMS_ERR_* code.  Argument errors
 *    are detected on the host and enqueue nothing.  Errors raised on the
 *    device (capacity overflow, a timed-out wait) are sticky and surface at
 *    dms_cache_status().
 *  - bf16 means IEEE-754 binary16-brain (__nv_bfloat16), passed as void*.
 */
#ifndef DMS_H
#define DMS_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DMS_OK 0
#define DMS_ERR_INVALID_ARG (-1) /* bad size, null or misaligned pointer, wrong device */
#define DMS_ERR_CUDA (-2)        /* a CUDA allocation, copy or launch failed */
#define DMS_ERR_CAPACITY (-3)    /* sticky: an append found no free slot */
#define DMS_ERR_BAD_HANDLE (-4)  /* NULL, destroyed or foreign cache handle */
#define DMS_ERR_TIMEOUT (-5)     /* sticky: a device-side wait passed its time limit */
#define DMS_ERR_EMPTY (-6)       /* decode before any token was appended */
#define DMS_ERR_SCRATCH_LIMIT (-7) /* problem too large for the fixed scratch of dms_decode_attention_noalloc */

/* Largest query-head group per KV head (Hq / Hkv) the decode kernel supports. */
#define DMS_MAX_GROUP 8

/* Storage formats of the K and V pools (dms_cache_create_ex). */
#define DMS_KV_BF16 0     /* bf16 rows, as given */
#define DMS_KV_FP8_E4M3 1 /* FP8 E4M3 codes with a float32 scale per row */

typedef struct dms_cache dms_cache_t;

/*
 * Create a cache for `batch` sequences x `kv_heads` KV heads, each with
 * `capacity` slots of `head_dim` bf16 elements for K and for V, and delay
 * window `window` (>= 1; 16 in the method).  head_dim must be 64 or 128.
 * Allocates on the current CUDA device: K and V pools bf16
 * [batch][kv_heads][capacity][head_dim], the slot -> position map int32
 * [batch][kv_heads][capacity], the ring of the last `window` appends
 * (slot, decision), the lengths int32 [batch][kv_heads], a sticky error word
 * and the split-K scratch of the decode kernel; all zeroed.  The host keeps the
 * position counter t (all sequences advance in lock step).
 * Returns NULL on failure; dms_last_error() then gives the code.
 */
dms_cache_t* dms_cache_create(int batch, int kv_heads, int capacity, int head_dim, int window);

/*
 * As dms_cache_create, with the storage format of the K and V pools:
 * DMS_KV_BF16 (what dms_cache_create makes) or DMS_KV_FP8_E4M3.
 *
 * FP8 storage combines the method's eviction with quantization, which the
 * method's authors call orthogonal to it and combinable ("Inference-Time
 * Hyper-Scaling with KV Cache Compression", paper-notes page, "Related work":
 * KVQuant / KIVI).  Each retained K row and V row (one token, one KV head) is
 * stored as head_dim E4M3 codes and a float32 scale:
 *   scale = amax / 448 in float32 (amax = largest |x| of the row; 1 if amax = 0)
 *   code  = E4M3(x / scale): float32 quotient, rounded to nearest (ties to
 *           even) and saturated to +-448
 * and stands for code * scale.  Inputs and outputs of every call stay bf16 /
 * fp32 as documented; appends quantize, the decode attention dequantizes
 * (scores and probabilities are computed in fp32 as for bf16 storage).  Pools:
 * K rows of head_dim + 16 bytes (codes, then {K scale, V scale} and 8 bytes of
 * padding), V rows of head_dim bytes, i.e. 2 * head_dim + 16 bytes per slot
 * against 4 * head_dim for bf16.  On an FP8 cache dms_prefill runs its
 * definition, `chunk` rounds of append + decode (one fused step launch per
 * token, exact, far slower than the tensor-core path of bf16 caches); dms_step
 * is one launch as on bf16 caches.  An FP8 cache also holds a buffer for one
 * token's rows of those rounds.  dms_decode_attention_noalloc reads bf16 pools
 * only.
 */
dms_cache_t* dms_cache_create_ex(int batch, int kv_heads, int capacity, int head_dim, int window, int kv_format);

/* Storage format of a cache (DMS_KV_BF16 or DMS_KV_FP8_E4M3), or DMS_ERR_BAD_HANDLE. */
int dms_cache_kv_format(dms_cache_t* cache);

/* Code of the last failed dms_cache_create() on this thread (DMS_OK if none). */
int dms_last_error(void);

/* Free the cache's device memory.  Synchronizes the device first.  NULL or an
 * unknown handle is ignored. */
void dms_cache_destroy(dms_cache_t* cache);

/*
 * Append token t (= the number of tokens appended so far) to every
 * (sequence, KV head) -- the method's decision, delayed eviction and slot reuse
 * in one kernel, with no host round trip:
 *   k, v         bf16  [batch][kv_heads][head_dim]   the new token's K and V
 *   evict_logit  fp32  [batch][kv_heads]             decision = (logit > 0)
 * Per (b, h): if t >= window and token t - window was marked, that token leaves
 * and token t takes its slot; otherwise token t takes slot len and len grows.
 * With no free slot the token is dropped and DMS_ERR_CAPACITY is latched.
 * The host counter t advances by one.
 */
int dms_append(dms_cache_t* cache, const void* k, const void* v, const float* evict_logit,
               void* stream);

/*
 * Append `chunk` tokens (positions t .. t+chunk-1) in one launch; the result
 * is bit-identical to `chunk` calls of dms_append:
 *   k, v    bf16 [batch][kv_heads][chunk][head_dim]
 *   logits  fp32 [batch][kv_heads][chunk]
 * Used to fill the cache before decoding (the bookkeeping half of a chunked
 * prefill).
 */
int dms_append_chunk(dms_cache_t* cache, const void* k, const void* v, const float* logits,
                     int chunk, void* stream);

/*
 * Chunked prefill: attention for `chunk` new tokens (positions t .. t+chunk-1,
 * t = tokens appended so far), then their append.  The result equals `chunk`
 * rounds of dms_append followed by dms_decode_attention, one per token:
 *   q       bf16 [batch][q_heads][chunk][head_dim]
 *   k, v    bf16 [batch][kv_heads][chunk][head_dim]
 *   logits  fp32 [batch][kv_heads][chunk]        decision = (logit > 0)
 *   out     fp32 [batch][q_heads][chunk][head_dim]
 * The query of token c sees the retained cache and the chunk's tokens up to c
 * under the delayed eviction of the method ("Inference-Time Hyper-Scaling with
 * KV Cache Compression", AI research-map summary, "Approach"): a token marked
 * for eviction stays visible for the w - 1 positions after its own.  The
 * attention runs on the tensor cores (bf16 Q K^T, fp32 softmax, P V with p
 * carried as two bf16 terms, fp32 accumulation); then the chunk is appended
 * as by dms_append_chunk.  q_heads as for dms_decode_attention.  On an FP8
 * cache (dms_cache_create_ex) it runs the `chunk` rounds of dms_append +
 * dms_decode_attention themselves, token by token: per token a few pitched
 * device-to-device copies gather its rows, then one launch of the fused step
 * kernel (append + decode), then a copy scatters its output row (six stream
 * operations per token).  If one of them fails to enqueue, the call returns the error
 * and the cache stays at the position of the last round that was enqueued in
 * full (the tokens before it are appended, the rest are not).
 */
int dms_prefill(dms_cache_t* cache, const void* q, const void* k, const void* v, const float* logits, int chunk,
                float* out, float scale, int q_heads, void* stream);

/*
 * Decode attention for the query of the last appended token, over every
 * retained slot of each (sequence, KV head).  This is the step the method is
 * built to make cheaper: autoregressive decoding reads the whole KV cache at
 * every step, so its cost is the KV-cache token reads ("Inference-Time
 * Hyper-Scaling with KV Cache Compression", notes page, section "研究背景与动机";
 * AI research-map summary, "Experimental setup": KV-cache token reads), and
 * DMS cuts them by evicting tokens after the delay window (same summary,
 * "Approach").  The attention itself is plain softmax attention over the
 * retained keys:
 *   q    bf16 [batch][q_heads][head_dim]
 *   out  fp32 [batch][q_heads][head_dim]
 *   out[b][g] = softmax(scale * K_h q_g) V_h over the retained keys of KV head
 *   h = g / (q_heads / kv_heads), in fp32 (bf16 inputs widened exactly).
 * q_heads must be a multiple of kv_heads with q_heads / kv_heads <= 8.
 * The retained slots of all heads are split evenly across the warps of a
 * persistent grid (flash-decoding split-K balanced by retained length); the
 * partial results of a head split across warps are merged in the same kernel
 * by the last warp to finish that head.  Uses the split-K scratch that
 * dms_cache_create allocated; allocates nothing.  Returns DMS_ERR_EMPTY if
 * nothing was appended.
 */
int dms_decode_attention(dms_cache_t* cache, const void* q, float* out, float scale, int q_heads,
                         void* stream);

/*
 * One decode step in one call: the result of dms_append(k, v, evict_logit)
 * followed by dms_decode_attention(q, out, scale, q_heads), bit for bit, with
 * the arguments checked once (the method's decode step: append with delayed
 * eviction, then attention over the retained cache; AI research-map summary,
 * "Approach").
 *  - ONE kernel launch (bf16 or FP8 storage).  The decode kernel appends the
 *    token to every head (into generations of the cache state that the launch
 *    does not read; an FP8 cache quantizes it as dms_append does) and attends
 *    over the cache after the append.  When the previous
 *    call that advanced the cache added one token (dms_append, dms_step, or a
 *    step-graph launch) and window >= 2, the launch computes its lengths and
 *    work split and starts its first tile copies before the previous kernel
 *    on the stream has finished (programmatic dependent launch); it reads its
 *    inputs and writes anything only after that kernel has completed, so it
 *    may follow any kernel that produces q, k, v or evict_logit.
 */
int dms_step(dms_cache_t* cache, const void* k, const void* v, const float* evict_logit, const void* q, float* out,
             float scale, int q_heads, void* stream);

/*
 * dms_step with its inputs read from, and its output written to, HOST memory:
 * the call a serving loop makes when the token's rows arrive from, and the
 * attention output goes back to, the host.  Same result as dms_step on the
 * same rows, bit for bit (the same kernel runs on device copies of them).
 *   k, v         bf16 [batch][kv_heads][head_dim]   host memory
 *   evict_logit  fp32 [batch][kv_heads]             host memory
 *   q            bf16 [batch][q_heads][head_dim]    host memory
 *   out          fp32 [batch][q_heads][head_dim]    host memory, written
 * The cache keeps two sets of device rows and two copy streams of its own,
 * made (with cudaMalloc) on the first call.  Call i uses set i % 2: its
 * host->device copies wait only for the step of call i - 2, so they overlap
 * the step of call i - 1, and its device->host copy overlaps the step of
 * call i + 1.  The step itself runs on `stream`.  The copy streams wait for
 * the step kernels through events; the step kernel waits for its rows (and
 * for the copy-out of the call that last used its output rows) by polling
 * sequence numbers that the copy streams write to device memory when they
 * finish, so that `stream` holds only the step kernels and each step keeps
 * the early start of dms_step.  That wait is bounded (1.5 s); on expiry the
 * kernel latches DMS_ERR_TIMEOUT (dms_cache_status) and computes on stale
 * rows of its own buffers.
 * Everything is asynchronous:
 *  - the host input buffers must stay unchanged, and `out` unread, until the
 *    call's copies are done: dms_step_host_join(cache, s) makes stream s wait
 *    for every copy out enqueued so far, after which a synchronize of s (or
 *    an event recorded on it) says that all outputs are in host memory;
 *  - pinned (page-locked) host memory lets the copies overlap the steps;
 *    with pageable memory the copies are correct but serialize with the host.
 * Not allowed while `stream` is being captured into a CUDA graph
 * (DMS_ERR_INVALID_ARG).  Device pointers are refused (DMS_ERR_INVALID_ARG):
 * use dms_step for rows already on the device.
 */
int dms_step_host(dms_cache_t* cache, const void* k, const void* v, const float* evict_logit, const void* q,
                  float* out, float scale, int q_heads, void* stream);

/* Make `stream` wait for every device->host copy that dms_step_host has
 * enqueued on this cache so far.  Enqueues only waits; DMS_OK if no host step
 * was made. */
int dms_step_host_join(dms_cache_t* cache, void* stream);

/* Copy the retained length of every (sequence, KV head) into out_dev
 * (int32 [batch][kv_heads], device memory), stream-ordered. */
int dms_cache_lengths(dms_cache_t* cache, int32_t* out_dev, void* stream);

/* Copy the slot -> position map into out_dev (int32 [batch][kv_heads][capacity];
 * -1 = slot never written).  Slots [0, len) hold exactly the retained tokens. */
int dms_cache_slot_positions(dms_cache_t* cache, int32_t* out_dev, void* stream);

/* Copy the K and V pools, in logical element order, into k_out / v_out
 * (device memory, 16-byte aligned): bf16 [batch][kv_heads][capacity][head_dim]
 * each; on an FP8 cache the E4M3 codes, uint8 [batch][kv_heads][capacity][head_dim]
 * each (the scales: dms_cache_export_scales). */
int dms_cache_export_kv(dms_cache_t* cache, void* k_out, void* v_out, void* stream);

/* FP8 caches: copy the float32 scales of every slot's K row and V row into
 * k_scale / v_scale (float32 [batch][kv_heads][capacity] each, device memory).
 * DMS_ERR_INVALID_ARG on a bf16 cache. */
int dms_cache_export_scales(dms_cache_t* cache, float* k_scale, float* v_scale, void* stream);

/* Synchronize `stream`, then return the sticky device error (DMS_OK,
 * DMS_ERR_CAPACITY or DMS_ERR_TIMEOUT) or DMS_ERR_CUDA if the stream failed. */
int dms_cache_status(dms_cache_t* cache, void* stream);

/* Failure-path self-test: enqueue one device-side wait, the same bounded wait
 * the kernels use, on a barrier that nothing completes.  It gives up after the
 * library's time limit (1.5 s) and latches DMS_ERR_TIMEOUT in the cache's
 * error word, as a wait that ran out inside a kernel would; the next
 * dms_cache_status() returns DMS_ERR_TIMEOUT and the cache should be destroyed.
 * No fault or trap is involved; the GPU context stays usable.  (The method has
 * no counterpart; this exists to test error reporting.) */
int dms_cache_selftest_wait(dms_cache_t* cache, void* stream);

/*
 * A decode step over several caches (the layers of a model, say) captured
 * once into a CUDA graph and replayed per token, so that a step costs one
 * graph launch instead of one library call per layer.
 *
 * dms_step_graph_create captures, for i = 0 .. n-1, the fused step of
 * dms_step on caches[i] with the caller's buffers k[i], v[i], evict_logit[i],
 * q[i], out[i] (layouts as for dms_step; device memory, 16-byte aligned), the
 * given scale and q_heads; then one node that advances every cache's
 * position.  The buffers are bound by address: before each launch the caller
 * writes that step's inputs into them, and after it reads out[i].  The caches
 * must be distinct caches (bf16 or FP8 storage) on one device; the graph does
 * not own them and must be destroyed before they are.  Returns NULL on failure (dms_last_error()
 * gives the code; stream capture must not be active on the calling thread).
 *
 * dms_step_graph_launch enqueues one step on `stream`: the result equals
 * dms_step on every cache in order, bit for bit.  Each cache's position is
 * also kept in device memory, which the replayed kernels read; if a cache
 * advanced outside the graph since the last launch (dms_append, dms_step, ...)
 * a one-thread kernel first re-sends its position.  The host counters advance
 * by one.  No allocation.
 *
 * Method reference: the step is the method's decode (append with delayed
 * eviction, then attention over the retained cache), "Inference-Time
 * Hyper-Scaling with KV Cache Compression", AI research-map summary,
 * "Approach"; the graph only changes how it is launched.
 */
typedef struct dms_step_graph dms_step_graph_t;
dms_step_graph_t* dms_step_graph_create(dms_cache_t* const* caches, int n, const void* const* k,
                                        const void* const* v, const float* const* evict_logit,
                                        const void* const* q, float* const* out, float scale, int q_heads);
int dms_step_graph_launch(dms_step_graph_t* graph, void* stream);
/* Synchronizes the device, then frees the graph.  NULL is ignored. */
void dms_step_graph_destroy(dms_step_graph_t* graph);

/* Number of tokens appended so far (the host position counter t), or -1. */
int64_t dms_cache_position(dms_cache_t* cache);

/* Static description of a code. */
const char* dms_error_string(int code);

/*
 * Decode attention without any device allocation.  (The paper has no
 * counterpart: this entry point exists for callers, not for the method.)
 *
 * Some callers cannot call cudaMalloc when they decode: an inference engine
 * that reserved all device memory for its own pool at start-up, code running
 * where the caching allocator must not grow, or a component that is only
 * handed pointers to buffers another component owns.  This call computes the
 * same result as dms_decode_attention, but reads the cache from caller-owned
 * buffers and keeps the decode kernels' split-K scratch in a fixed array of
 * DMS_NOALLOC_SCRATCH_BYTES that the library holds in device memory on every
 * GPU that loads it, until the process exits.  It calls no allocating routine.
 *
 *   k_pool, v_pool  bf16 [batch][kv_heads][capacity][head_dim], the retained
 *                   tokens of (b, h) in slots [0, len[b][h]).  V rows are in
 *                   plain element order.  K rows use the library's layout:
 *                   16-byte chunk c of slot s is stored at chunk c ^ (s & 7).
 *   len             int32 [batch][kv_heads] (device memory): the retained
 *                   length of each head, normally 1 .. capacity.  The kernel
 *                   clamps every value to [0, capacity] before using it (a
 *                   value outside that range can never send a read past a
 *                   head's pool) and latches a length error in the scratch's
 *                   error word; a head whose length is 0 after clamping has no
 *                   keys, and its output rows are left unwritten.
 *   q, out, scale, q_heads: as for dms_decode_attention.
 * All pointers are device memory of the current device, 16-byte aligned
 * (len 4-byte aligned).
 *
 * Limits: batch * kv_heads <= DMS_NOALLOC_MAX_HEADS, and the scratch a call
 * needs, about (12 * SM count + batch * kv_heads) * G * (head_dim + 2) * 4
 * bytes plus 4 bytes per head (G = q_heads / kv_heads), must fit in
 * DMS_NOALLOC_SCRATCH_BYTES; otherwise DMS_ERR_SCRATCH_LIMIT is returned and
 * nothing is enqueued.  (On a 148-SM B300 with head_dim 128 that allows the
 * full 2048 heads at G = 4 and about 800 at G = 8.)
 *
 * The first call on a device looks up the scratch array's device address and
 * zeroes its error word (a synchronous step), so make that first call before
 * any stream capture.  Every call shares the one array: calls whose kernels
 * overlap on the GPU (other streams, other host threads) race on it and must
 * be ordered by the caller.  Each call first clears the per-head counters it
 * uses (a stream-ordered memset, which allocates nothing) and writes every
 * other scratch value before reading it.  A device
 * wait that times out is latched in the array's error word; this call does not
 * report it.
 */
#define DMS_NOALLOC_SCRATCH_BYTES (8u << 20)
#define DMS_NOALLOC_MAX_HEADS 2048
int dms_decode_attention_noalloc(const void* k_pool, const void* v_pool, const int32_t* len, int batch,
                                 int kv_heads, int capacity, int head_dim, const void* q, float* out,
                                 float scale, int q_heads, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DMS_H */
