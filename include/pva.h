/*
 * pva.h -- packed variable-length attention (scaled dot-product attention
 * over padding-free, variable-length sequences with MHA/GQA/MQA head
 * sharing) for NVIDIA GB300 (sm_103a).  C ABI of libpva.so.
 *
 * The operation is the one defined on the "onnx-runtime-ep-cuda" source page
 * packed_varlen_attention.rs (op `PackedVarlenAttention` v1):
 *
 *   - module doc "Packed layout & cumulative offsets": B sequences are
 *     concatenated on one token axis; sequence b owns query rows
 *     [cu_seqlens_q[b], cu_seqlens_q[b+1]) and key/value rows
 *     [cu_seqlens_kv[b], cu_seqlens_kv[b+1]); attention is block diagonal.
 *   - "Schema (v1)": Q [total_q, num_heads, head_size], K [total_kv,
 *     kv_num_heads, head_size], V [total_kv, kv_num_heads, v_head_size],
 *     output [total_q, num_heads, v_head_size]; a rank-2 [tokens, heads*dim]
 *     tensor has the same bytes.  kv_num_heads divides num_heads; query head h
 *     reads key/value head h / (num_heads / kv_num_heads).
 *   - "Causal alignment": with is_causal, local query i sees local key j iff
 *     j <= i + (L_kv - L_q) (tail aligned).
 *   - kernel stages 1-5: score = scale * q.k; with softcap != 0 the score is
 *     replaced by softcap * tanh(score / softcap) before masking; softmax over
 *     the visible keys; a row with no visible key is written as zeros;
 *     out = sum_j p_j V[j].  Storage is f32, f16 or bf16 (codes 0, 1, 2, as on
 *     the page); arithmetic is fp32; f16/bf16 outputs are rounded to nearest
 *     even.
 *
 * All calls are asynchronous and stream ordered unless stated otherwise.
 */
#ifndef PVA_H
#define PVA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes (negative = error; nothing was enqueued). */
typedef enum {
  PVA_OK = 0,
  PVA_ERR_INVALID_ARG = -1, /* null pointer, bad count, bad dtype, non-finite scalar */
  PVA_ERR_UNSUPPORTED = -2, /* valid request this build does not implement */
  PVA_ERR_CUDA = -3,        /* a CUDA runtime call failed (see pva_last_error) */
  PVA_ERR_OOM = -4          /* workspace allocation failed */
} pva_status;

/* Storage types of Q, K, V and the output (one type for all four). */
typedef enum { PVA_F32 = 0, PVA_F16 = 1, PVA_BF16 = 2 } pva_dtype;

/* Device-side status bits, latched by the on-device scheduler and read with
 * pva_get_status.  When any bit is set the call wrote nothing to `out`. */
#define PVA_DEV_CU_Q_START 0x1u   /* cu_seqlens_q[0] != 0 */
#define PVA_DEV_CU_KV_START 0x2u  /* cu_seqlens_kv[0] != 0 */
#define PVA_DEV_CU_Q_ORDER 0x4u   /* cu_seqlens_q decreases somewhere */
#define PVA_DEV_CU_KV_ORDER 0x8u  /* cu_seqlens_kv decreases somewhere */
#define PVA_DEV_TOO_MANY 0x10u    /* work count does not fit the 32-bit work index */
#define PVA_DEV_NULL_TENSOR 0x20u /* a NULL q/k/v/out with a nonzero token extent */
#define PVA_DEV_KV_LEN 0x40u      /* pva_forward_padded: a nonpad length outside [0, kv_seq] */
#define PVA_DEV_KV_CACHE 0x80u    /* pva_gqa_kvcache: a step outside the cache's bounds, or one
                                     after such a step (see there) */
#define PVA_DEV_WAIT_TIMEOUT 0x100u /* a pipeline wait in a kernel gave up (never expected) */

/*
 * pva_forward -- out = attention(q, k, v) over packed sequences.
 *
 * q, k, v, out : device pointers, row-major and contiguous, layouts as in
 *                the schema above, all of storage type `dtype`.  For f16 and
 *                bf16 each of q, k, v, out must be 16-byte aligned (tensor
 *                copies require it).  q, k, v are only read; out is only
 *                written; out must not overlap q, k or v.  q and out may be
 *                NULL when total_q is 0, k and v when total_kv is 0 (an empty
 *                tensor); a NULL pointer with a nonzero extent is caught on the
 *                device (PVA_DEV_NULL_TENSOR, nothing computed).
 * cu_seqlens_q, cu_seqlens_kv : device pointers to int32 [B+1] cumulative
 *                offsets, starting at 0 and non-decreasing.  cu_seqlens_q[B]
 *                must equal total_q and cu_seqlens_kv[B] must equal total_kv
 *                (the caller's contract: this signature carries no totals, and
 *                the library never copies the offsets back to the host).
 *                Violations of the start/order rules are detected on the
 *                device: a status bit is latched, nothing is computed and
 *                `out` is left untouched (see pva_get_status).
 * B            : number of sequences, >= 1.  Empty sequences are allowed.
 * num_heads, kv_num_heads : H >= 1 and Hkv >= 1 with H % Hkv == 0.
 * head_size, v_head_size  : d and dv.  f16/bf16: (d, dv) in {(64, 64),
 *                (96, 96), (128, 128), (192, 192), (256, 256), (192, 128)} and
 *                H / Hkv <= 128.  f32: 1 <= d, dv <= 256.
 * scale        : finite; 0 selects the default 1/sqrt(head_size) (computed in
 *                fp32).  Any other value is used as given.
 * is_causal    : nonzero selects the tail-aligned causal mask.
 * softcap      : finite; 0 disables the cap; c and -c give the same result.
 * dtype        : a pva_dtype code.
 * stream       : cudaStream_t to enqueue on (0 = legacy default stream).
 *
 * Returns PVA_OK once the work is enqueued; it does not wait for it.  Memory:
 * the library keeps one workspace per (device, stream), grown on demand
 * inside this call (the growth synchronises `stream`); after the first call
 * with the largest B, calls allocate nothing and never synchronise, so they
 * can be captured into a CUDA graph.  Growth during stream capture returns
 * PVA_ERR_INVALID_ARG.  Calls on one stream are ordered; calls on different
 * streams use different workspaces.  Not re-entrant across host threads for
 * the same stream.
 */
int pva_forward(const void* q, const void* k, const void* v,
                const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv,
                void* out, int B, int num_heads, int kv_num_heads,
                int head_size, int v_head_size, float scale, int is_causal,
                float softcap, int dtype, void* stream);

/*
 * pva_forward_from_host -- pva_forward for a batch held in host memory: the
 * same attention (packed_varlen_attention.rs, stages 1-5), with the copies in
 * and out of the device done by the call and overlapped with the attention.
 *
 * q_host, k_host, v_host, out_host : host buffers in the packed layouts of
 *                pva_forward (pinned memory lets the copies overlap the
 *                attention; pageable memory works but copies synchronously).
 * cu_seqlens_q_host, cu_seqlens_kv_host : HOST int32 [B+1] offsets, read by
 *                the call (starting at 0, non-decreasing; else
 *                PVA_ERR_INVALID_ARG with nothing enqueued).
 * q_dev, k_dev, v_dev, out_dev : device buffers of the same sizes as the host
 *                ones, owned by the caller; the call overwrites them.
 * cu_dev       : device int32 scratch of at least 4 * B + 34 words.
 * chunks       : runs of whole sequences moved and computed in turn (0: 8;
 *                at most 16 and at most B), cut to move about equal bytes:
 *                chunk c+1 is copied in while chunk c is computed and chunk
 *                c-1 copied out, on two library streams synchronised with
 *                `stream` by events.  Each chunk is one pva_forward call on
 *                `stream` (with offsets rebased on the device), so every row
 *                offset must keep pva_forward's 16-byte alignment.
 * Other arguments: as pva_forward.
 *
 * Returns PVA_OK once all work is enqueued; `stream` completes after the last
 * output copy.  The copies start after the work already on `stream`.  An
 * error from a chunk's pva_forward is returned as it is (earlier chunks'
 * work stays enqueued).  Calls on one device are serialised by a lock.
 */
int pva_forward_from_host(const void* q_host, const void* k_host, const void* v_host,
                          const int32_t* cu_seqlens_q_host, const int32_t* cu_seqlens_kv_host,
                          void* out_host, void* q_dev, void* k_dev, void* v_dev, void* out_dev,
                          int32_t* cu_dev, int B, int num_heads, int kv_num_heads, int head_size,
                          int v_head_size, float scale, int is_causal, float softcap, int dtype,
                          int chunks, void* stream);

/*
 * pva_forward_local -- pva_forward with a local (sliding) attention window,
 * the `local_window` of the softmax and grouped-query reference kernels on the
 * attention.rs and group_query_attention.rs pages.  With local_window = W > 0,
 * query row i of a sequence (causal limit c = i + L_kv - L_q) also ignores the
 * keys j < c + 1 - W, so it sees at most the W keys ending at c (causal) or the
 * keys [max(0, c + 1 - W), L_kv) (non-causal).  local_window <= 0 is exactly
 * pva_forward.  Key tiles wholly before a work item's window are never loaded,
 * and decode rows split only their last W keys.  Other arguments, errors and
 * asynchrony: as pva_forward.
 */
int pva_forward_local(const void* q, const void* k, const void* v,
                      const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv,
                      void* out, int B, int num_heads, int kv_num_heads,
                      int head_size, int v_head_size, float scale, int is_causal,
                      float softcap, int local_window, int dtype, void* stream);

/*
 * pva_forward_padded -- the padded form of the same attention: the opset-24
 * Attention input `nonpad_kv_seqlen` of the packed_varlen_attention.rs module
 * doc ("Relationship to ONNX Attention-24 nonpad_kv_seqlen") and of the
 * attention.rs page (the per-batch causal offset and padding frontier built
 * before the launch).  Batch entry b has q_seq query rows and a key/value slot
 * of kv_seq rows, of which the first nonpad_kv_seqlen[b] are its keys; query
 * row i sees key j iff j < nonpad_kv_seqlen[b] and, when is_causal,
 * j <= i + nonpad_kv_seqlen[b] - q_seq.  That is exactly pva_forward on the
 * same rows with the padding removed (cu_seqlens_kv the exclusive prefix sum
 * of nonpad_kv_seqlen); here nothing is copied or repacked.
 *
 * q    : [B, q_seq, num_heads, head_size]      (every query row is real)
 * k    : [B, kv_seq, kv_num_heads, head_size]
 * v    : [B, kv_seq, kv_num_heads, v_head_size]
 * out  : [B, q_seq, num_heads, v_head_size]    (every row written)
 * nonpad_kv_seqlen : device pointer to int64 [B].  A value outside
 *        [0, kv_seq] latches PVA_DEV_KV_LEN on the device; nothing is computed
 *        and `out` is left untouched.
 * B >= 1, q_seq >= 0, kv_seq >= 0, and B * q_seq and B * kv_seq must fit in
 * int32 (else PVA_ERR_INVALID_ARG, nothing enqueued).  The padding rows of k
 * and v are never read: K and V are loaded through per-slot tensor maps and
 * each slot's last key tile ends at its last key, so padding may hold
 * anything, NaN and Inf included.  The offsets are built on the device by a
 * small kernel in the stream, inside the library's workspace.  Other
 * arguments, errors, memory and asynchrony: as pva_forward.
 */
int pva_forward_padded(const void* q, const void* k, const void* v,
                       const int64_t* nonpad_kv_seqlen, void* out, int B, int q_seq,
                       int kv_seq, int num_heads, int kv_num_heads, int head_size,
                       int v_head_size, float scale, int is_causal, float softcap,
                       int dtype, void* stream);

/*
 * pva_gqa_kvcache -- one GroupQueryAttention step against a fixed-capacity
 * KV cache, as on the group_query_attention.rs page: the per-sequence
 * metadata of `gqa_prepare_metadata`, the in-place append of
 * `gqa_append_cache`, the rotary embedding of `gqa_rope_bnsh` (on the queries
 * and on the appended keys), then causal attention of every query row over
 * the sequence's valid cache rows, read straight from the BNSH cache.
 *
 * q       : [B, q_seq, num_heads, head_size]              (read)
 * k_new, v_new : [B, k_seq, kv_num_heads, head_size]      (read; NULL if k_seq 0)
 * k_cache, v_cache : [B, kv_num_heads, capacity, head_size] BNSH (appended)
 * seqlens_k : device int32 [B]; sequence b holds total_b = seqlens_k[b] + 1
 *           keys after this step.  The new rows go to cache rows
 *           [past_b, past_b + k_seq) with past_b = total_b - k_seq; query row
 *           s sits at position first_b + s with first_b = total_b - q_seq and
 *           sees cache rows j <= first_b + s (the tail-aligned causal rule) and,
 *           with local_window W > 0, only j >= first_b + s + 1 - W.
 * rotary_dim : 0 = no rotary embedding; else even, 2 <= rotary_dim <=
 *           head_size, and k_seq is 0 or q_seq.  cos_cache and sin_cache are
 *           [cache_rows, rotary_dim / 2] of type rotary_dtype (PVA_F32, or
 *           PVA_F16 when dtype is f16 or bf16).  Pair k < rotary_dim / 2 of a
 *           head row is (2k, 2k+1) if rotary_interleaved, else (k, k +
 *           rotary_dim/2); it is rotated by (c, s) = the tables' entry
 *           [position][k] as (c x0 - s x1, s x0 + c x1) in f32, each product
 *           and difference rounded on its own, then rounded to dtype; dims at
 *           or past rotary_dim are copied.  position_ids (device int64
 *           [B, q_seq], or NULL) gives the positions of the query rows and of
 *           the appended rows; NULL means first_b + s and past_b + s.
 *           Rotated queries go to library scratch; q itself is not written.
 * out     : [B, q_seq, num_heads, head_size] (every row written).
 * scale, softcap, dtype, stream : as pva_forward (v_head_size = head_size).
 *
 * Host errors (nothing enqueued): null pointers, B < 1, q_seq < 1, k_seq < 0,
 * capacity < 1, (B + 1) * capacity or B * q_seq beyond int32, odd head_size,
 * a bad rotary_dim / table / rotary_dtype, rotary with k_seq not in {0,
 * q_seq}, plus pva_forward's checks (head sizes, alignment, dtype).
 * Device errors: the step is all or nothing.  It is rejected if, for some b,
 * total_b exceeds int32, past_b < 0, first_b < 0, past_b > capacity or
 * total_b > capacity, or (rotary) a position lies outside [0, cache_rows) --
 * the bounds the page's metadata kernel checks -- and also if
 * PVA_DEV_KV_CACHE is already latched on the stream (a later step must not
 * append after rows a rejected step skipped: read and clear the bit with
 * pva_get_status, repair the cache, then go on).  A rejected step latches
 * PVA_DEV_KV_CACHE and writes neither the cache nor `out`.
 * Cache rows at or past total_b are never read (a sequence's last key tile
 * is shifted back to end at its last key), so they may hold anything, NaN
 * included.
 * k_new/v_new must not overlap the cache rows being written.
 */
int pva_gqa_kvcache(const void* q, const void* k_new, const void* v_new, void* k_cache,
                    void* v_cache, const int32_t* seqlens_k, const void* cos_cache,
                    const void* sin_cache, const int64_t* position_ids, void* out, int B,
                    int q_seq, int k_seq, int capacity, int num_heads, int kv_num_heads,
                    int head_size, int rotary_dim, int cache_rows, int rotary_interleaved,
                    int rotary_dtype, float scale, float softcap, int local_window, int dtype,
                    void* stream);

/*
 * pva_forward_noalloc -- the same attention as pva_forward, for callers that
 * cannot allocate device memory when they call (a runtime whose device memory
 * is planned ahead and owned by an arena or governor, code that runs while
 * another component holds the allocator, a process with a fixed device
 * footprint).  The pages have no counterpart of this entry point.
 *
 * It calls no cudaMalloc, cudaFree or allocating library routine: its scratch
 * (work lists, decode split partials and counters, a status word) is one
 * file-scope device array of 4 MiB.  A device holds it from the moment the
 * library's device code is loaded there (with CUDA's lazy module loading: the
 * first call that needs that code) until the process exits.  Arguments are
 * those of pva_forward, plus:
 *   device_status : optional device pointer to a uint32 the call ORs its
 *                   PVA_DEV_* bits into (the caller clears it).  NULL uses a
 *                   word inside the scratch, which each call clears first and
 *                   nothing reads back: device-side errors (malformed offsets,
 *                   NULL tensors with a nonzero extent, a wait that gave up)
 *                   then leave `out` unwritten without telling the caller.
 * Limits: B * (4 + kv_num_heads) int32 words of work lists must fit in 1 MiB
 * (else PVA_ERR_UNSUPPORTED with nothing enqueued); decode splits are limited
 * to the partials that fit in the rest of the array.  All calls on a device
 * share the array: calls whose kernels overlap on the GPU race and give wrong
 * results, so keep them ordered (one stream, or events between streams).  The
 * array keeps the last call's contents; what must start at zero is cleared
 * by each call.  The first call on each device looks up the array's device
 * address (cudaGetSymbolAddress with that device current) and caches it; make
 * it before any stream capture.  The cached address belongs to the context of
 * that call: after a device reset, call pva_release (which drops it) first.
 */
int pva_forward_noalloc(const void* q, const void* k, const void* v,
                        const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv,
                        void* out, int B, int num_heads, int kv_num_heads,
                        int head_size, int v_head_size, float scale, int is_causal,
                        float softcap, int dtype, uint32_t* device_status, void* stream);

/*
 * pva_get_status -- synchronises `stream`, then reads and clears the device
 * status bits (PVA_DEV_*) latched by the calls made on it since the last read.
 * *device_flags receives 0 when every call was well formed.  Returns PVA_OK or
 * PVA_ERR_CUDA (e.g. when no call has been made on this stream yet the flags
 * are simply 0).
 */
int pva_get_status(void* stream, uint32_t* device_flags);

/*
 * pva_schedule -- runs only the on-device scheduler for the given offsets and
 * copies its work description to host memory (synchronous; an inspection and
 * test entry point).  `dtype` and the head/size arguments select the kernel
 * family whose tiles are counted, exactly as pva_forward would.
 *
 * host_out receives int32 words:
 *   [0] status bits, [1] n_prefill (sequences with prefill work),
 *   [2] n_prefill_items, [3] n_decode (sequences routed to split-KV decode),
 *   [4] n_decode_units, [5] q-tile rows in tokens, [6] units per q-tile,
 *   [7] decode chunk in keys,
 *   then B words: prefill sequence order (longest first; -1 padded),
 *   then B+1 words: prefill item prefix sums in that order,
 *   then B words: decode sequence order, then B+1 words: decode unit prefix.
 * capacity is the number of int32 words host_out can hold (>= 8 + 4B + 2).
 */
int pva_schedule(const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv,
                 int B, int num_heads, int kv_num_heads, int head_size,
                 int v_head_size, int is_causal, int dtype, int32_t* host_out,
                 size_t capacity, void* stream);

/*
 * Per-kernel timing for benchmarks.  pva_profile(1) makes every later
 * pva_forward on this host thread bracket each kernel it launches with CUDA
 * events recorded on the caller's stream (do not enable it while capturing a
 * graph); pva_profile(0) turns it off.  pva_kernel_times synchronises the
 * stream of the last profiled call and writes the device durations, in
 * milliseconds, of its launches into ms[0..2]: [0] scheduler, [1] prefill
 * kernel (tensor-core or fp32), [2] split-KV decode kernel (-1 when it was not
 * launched).  Returns PVA_OK, or PVA_ERR_INVALID_ARG when no profiled call has
 * been made.
 */
int pva_profile(int enable);
int pva_kernel_times(float* ms, int capacity);

/*
 * pva_selftest_wait -- exercises the bounded waits that every kernel of this
 * library uses on its pipeline barriers: one CTA waits on an mbarrier that
 * nothing ever completes, with a limit of `limit_us` microseconds
 * (1 .. 1000000).  The wait gives up, latches PVA_DEV_WAIT_TIMEOUT and the
 * kernel returns; *device_flags receives the bits it latched.  Synchronous on
 * `stream`; allocates and frees a few bytes of device memory.  Returns PVA_OK,
 * PVA_ERR_INVALID_ARG (limit out of range) or PVA_ERR_CUDA.
 */
int pva_selftest_wait(uint32_t limit_us, void* stream, uint32_t* device_flags);

/* Human-readable text for a pva_status code (static storage). */
const char* pva_status_string(int code);

/* Text of the last error recorded by this host thread (static per thread). */
const char* pva_last_error(void);

/* Frees every workspace the library holds on the current device (waits for
 * the streams that used them first), destroys the copy streams and events of
 * pva_forward_from_host there, and drops pva_forward_noalloc's cached
 * address of its static scratch on that device. */
void pva_release(void);

/* Library version as (major << 16) | (minor << 8) | patch. */
int pva_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PVA_H */
