/*
 * engram.h -- C ABI of the GB300 (sm_103a) Engram layer forward.
 *
 * One Engram layer, as documented on the vLLM API page
 * "vllm.models.deepseek_v4_1.common.engram" (class Engram): hash ids fetch
 * one row per hash column from prime-sized hashed n-gram tables; the wkv
 * projection maps the concatenated rows to a key for each hc copy and a
 * value common to all copies; a gate -- sigmoid of the signed square root
 * of a normalised dot product of the residual stream against the key --
 * scales the value that is added to the stream; a False token mask leaves
 * a position untouched.
 *
 * Notation: T tokens, D = dim (hidden_size), H = hc_mult, C = n_hash_cols =
 * (max_ngram_size - 1) * n_heads, E = head_dim, K = C * E, N = D * (H + 1).
 *
 * Conventions for every entry point:
 *   - Pointers named "device" are CUDA device pointers (or, for the table of
 *     a host-offloaded handle, pinned host memory the GPU can address).
 *     The caller owns every buffer it passes; weights are borrowed by the
 *     handle and must outlive it.  The handle owns its workspace.
 *   - Work is enqueued on the given cudaStream_t (0 = legacy default stream)
 *     and the call returns without synchronising.  Ordering against work on
 *     other streams is the caller's, with CUDA events.
 *   - Return value: ENGRAM_OK (0) or a negative ENGRAM_ERR_* code.  No entry
 *     point aborts, traps or prints.  Errors found on the device (a hash id
 *     outside its table, a pipeline wait that gave up) set a sticky flag that
 *     engram_last_error() reports.
 *   - T == 0 is valid everywhere and launches nothing.
 */
#ifndef ENGRAM_GB300_H
#define ENGRAM_GB300_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ENGRAM_OK 0
#define ENGRAM_ERR_INVALID_ARG (-1)   /* null pointer, bad shape or stride */
#define ENGRAM_ERR_UNSUPPORTED (-2)   /* valid but not built: misalignment, H > 4, ... */
#define ENGRAM_ERR_T_EXCEEDS_MAX (-3) /* T larger than the handle's max_tokens */
#define ENGRAM_ERR_OOM (-4)           /* workspace allocation failed */
#define ENGRAM_ERR_NO_UVA (-5)        /* host-offloaded table needs unified addressing */
#define ENGRAM_ERR_DEVICE (-6)        /* the device reported an error (see below) */
#define ENGRAM_ERR_CUDA (-7)          /* a CUDA runtime call or launch failed */
#define ENGRAM_ERR_SCRATCH_LIMIT (-8) /* engram_gate_noalloc: the call needs more than
                                         ENGRAM_NOALLOC_MAX_PARTIALS scratch slots */

/* Bits of the sticky device error word returned by engram_device_error(). */
#define ENGRAM_DEVERR_BAD_HASH_ID 1u  /* an id outside [0, rows[c]): its row was zeroed */
#define ENGRAM_DEVERR_TIMEOUT 2u      /* a bounded pipeline wait gave up; outputs invalid */

#define ENGRAM_WKV_BF16 0   /* wkv bf16 [N, K] */
#define ENGRAM_WKV_MXFP8 1  /* wkv e4m3 [N, K] with E8M0 scales [N/32, K/32] */

/* Storage of the hash table's rows (class ParallelEngramEmbedding). */
#define ENGRAM_TABLE_FORMAT_BF16 0  /* bf16 [sum(rows), E] */
#define ENGRAM_TABLE_FORMAT_E4M3 1  /* e4m3 codes [sum(rows), E] with one ue8m0 scale per 32
                                       elements [sum(rows), E/32]; dequantized to bf16 on
                                       lookup: e4m3(code) * 2^(scale - 127), rounded to
                                       nearest even (E a multiple of 32) */

#define ENGRAM_TABLE_DEVICE 0       /* table rows in HBM */
#define ENGRAM_TABLE_HOST_PINNED 1  /* table rows in pinned host memory, read over the
                                       host link by the GPU (zero copy) */

/* Layer configuration (the HF config fields hidden_size, hc_mult,
 * rms_norm_eps, engram_max_ngram_size, engram_n_heads, engram_head_dim, and
 * the scheduler's max_num_batched_tokens, per class Engram.__init__). */
typedef struct engram_config {
    int64_t dim;            /* D; multiple of 256 */
    int64_t hc_mult;        /* H; 1..4 */
    int64_t max_ngram_size; /* >= 2 */
    int64_t n_heads;        /* >= 1 */
    int64_t head_dim;       /* E; multiple of 8, and C*E a multiple of 128 */
    double eps;             /* rms_norm_eps (1e-6 for DeepSeek-V4.1) */
    double clamp;           /* lower clamp of |dot| before the square root (1e-6) */
    int64_t max_tokens;     /* largest T any call will pass; sizes the workspace */
    int32_t wkv_format;     /* ENGRAM_WKV_* */
    int32_t table_location; /* ENGRAM_TABLE_* */
    int32_t device;         /* CUDA device ordinal the handle lives on */
    int32_t table_format;   /* ENGRAM_TABLE_FORMAT_* (0: bf16) */
} engram_config;

/* Weights, all borrowed.  Device pointers unless stated. */
typedef struct engram_weights {
    const void* table;          /* bf16 [sum(rows), E] row-major (or e4m3 codes for
                                   ENGRAM_TABLE_FORMAT_E4M3): every hash column's
                                   bucket concatenated (class ParallelEngramEmbedding);
                                   pinned host memory when table_location is HOST_PINNED;
                                   16-byte aligned */
    const int64_t* row_offset;  /* HOST array [C]: first table row of column c */
    const int64_t* rows;        /* HOST array [C]: rows in column c (a prime per
                                   class EngramLayout) */
    const void* wkv;            /* [N, K] row-major, K contiguous (the Linear layout);
                                   bf16, or e4m3 codes for MXFP8; 16-byte aligned */
    const uint8_t* wkv_scale;   /* MXFP8 only: E8M0 [N/32, K/32] row-major, one scale
                                   per 32x32 weight block; NULL for bf16 */
    const void* q_weight;       /* bf16 [H, D] */
    const void* k_weight;       /* bf16 [H, D] */
    const uint8_t* table_scale; /* ENGRAM_TABLE_FORMAT_E4M3 only: ue8m0 [sum(rows), E/32]
                                   row-major, in the same memory as the table; NULL for
                                   bf16 */
} engram_weights;

typedef struct engram_handle engram_t;

/* Create a handle on cfg->device: checks the configuration, copies the
 * row layout, precomputes q*k in fp32, allocates the workspace for
 * max_tokens (the counterpart of Engram.staged_rows) and builds the TMA
 * descriptors.  Synchronous.  Errors: INVALID_ARG, UNSUPPORTED, NO_UVA
 * (host-offloaded table without unified addressing, mirroring the
 * RuntimeError of ParallelEngramEmbedding.__init__), OOM, CUDA.  On error
 * *out is set to NULL. */
int engram_create(const engram_config* cfg, const engram_weights* w, engram_t** out);

/* Free the workspace (synchronises the device first).  NULL is accepted. */
int engram_destroy(engram_t* h);

/* Gather the rows of T tokens into the handle's staged-rows buffer
 * (Engram.prepare_embeddings / ParallelEngramEmbedding.lookup):
 *   staged[t, c*E + j] = table[row_offset[c] + hash_ids[t*ids_row_stride + c], j].
 * hash_ids: device int32, per-column local ids in [0, rows[c]); row stride
 * ids_row_stride >= C elements (column stride 1).  An id outside its range
 * gives a zero row and sets ENGRAM_DEVERR_BAD_HASH_ID.  background != 0
 * limits the grid to half of the SMs, leaving the rest to concurrent work.
 * A later engram_forward with hash_ids == NULL consumes these rows. */
int engram_lookup(engram_t* h, const int32_t* hash_ids, int64_t ids_row_stride, int64_t T,
                  int background, cudaStream_t stream);

/* Engram.forward: out = hidden + gate * value per (t, h), where
 *   key_h = kv[t, h*D:(h+1)*D], value = kv[t, H*D:(H+1)*D], kv = rows . wkv^T
 *   hr = rsqrt(mean_d hidden^2 + eps), kr = rsqrt(mean_d key_h^2 + eps)
 *   dot = sum_d(hidden * q[h] * k[h] * key_h) * hr * kr / sqrt(D)
 *   gate = sigmoid(sign(dot) * sqrt(max(|dot|, clamp)))
 * (the finish kernel of "vllm.models.deepseek_v41.amd.engram" with one rank).
 * Positions whose token_mask byte is 0 copy hidden's bits unchanged.
 *   hidden, out: device bf16 [T, H, D]; strides in ELEMENTS {t, h, d}; the d
 *       stride must be 1 and the t and h strides multiples of 8 (16-byte rows).
 *       out may be the same buffer as hidden with the same strides (in place);
 *       any other overlap with hidden, and any overlap of out with hash_ids
 *       or token_mask, is INVALID_ARG; so is an out whose T*H rows overlap
 *       each other (rows must nest copy-inside-token or token-inside-copy).
 *   hash_ids: as for engram_lookup, or NULL to use the rows staged by the
 *       last engram_lookup (which must have had the same T).
 *   token_mask: device bytes [T] (0 = False), or NULL for no mask.
 * The gate is computed in fp32 from an fp32 projection; out is rounded to
 * bf16 with round-to-nearest-even. */
int engram_forward(engram_t* h, const void* hidden, const int64_t hidden_strides[3],
                   const int32_t* hash_ids, int64_t ids_row_stride,
                   const uint8_t* token_mask, void* out, const int64_t out_strides[3],
                   int64_t T, cudaStream_t stream);

/* Validation hook, host only (no device is touched): the fused decode
 * kernel's plan for a configuration, T tokens and num_sms SMs, as
 * engram_forward would launch it.  out[0..ENGRAM_FUSED_PLAN_FIELDS) =
 *   used (1 if the fused kernel serves T), grid, widest column slice,
 *   token tiles, k-blocks, weight stages, token stages, weight stage bytes,
 *   token stage bytes, token ring offset, token ring bytes, q*k offset,
 *   barrier offset, dynamic shared memory bytes, two MMA issuers (0/1), Tn.
 * Offsets count from the 1024-byte aligned base of the shared memory. */
#define ENGRAM_FUSED_PLAN_FIELDS 16
int engram_debug_fused_plan(const engram_config* cfg, int64_t T, int32_t num_sms,
                            int64_t* out, int32_t n_out);

/* The same forward over HOST buffers: copies hidden, hash_ids and token_mask
 * (pinned host memory for asynchronous copies) into handle-owned device
 * buffers, runs engram_forward, and copies out back to the host buffer, all
 * on `stream`.  Contiguous [T, H, D] hidden/out.  The first call allocates
 * the host-path buffers for max_tokens. */
int engram_forward_host(engram_t* h, const void* hidden_host, const int32_t* hash_ids_host,
                        const uint8_t* token_mask_host, void* out_host, int64_t T,
                        cudaStream_t stream);

/* engram_forward_host for back-to-back calls (a serving loop): the input
 * copies of a call are NOT ordered after earlier work on `stream`; they
 * start on a handle-owned copy stream as soon as the call is made, so they
 * run during the previous call's forward and output copy.  The host buffers
 * must therefore already hold the inputs when the call is made (written by
 * the CPU, not by work still pending on a stream).  The forward runs on
 * `stream` after both its inputs and earlier work on `stream`; the output
 * copy runs on a second handle-owned stream, and `stream` waits for it, so
 * later work on `stream` (and a synchronisation of it) sees out_host
 * written.  Calls alternate between two handle-owned device slots, so a
 * call's input copy never overwrites what the previous call is still
 * reading or copying out.  The handle's copy streams are shared by every
 * caller stream: calls on one handle from several streams are serialised
 * on them.  While `stream` is being captured into a CUDA graph the call
 * behaves as engram_forward_host (all on `stream`) and flags are ignored.
 * The first call allocates the slots and creates the streams.
 *
 * flags = ENGRAM_HOST_DEFER_OUTPUT: `stream` waits for the PREVIOUS
 * pipelined call's output copy instead of this one's, so this call's output
 * copy overlaps the next call's forward.  After the call returns, later
 * work on `stream` sees the previous call's out_host written; this call's
 * out_host is written once engram_forward_host_flush has been called on
 * the handle and `stream` has reached that point.  Invalid flags:
 * ENGRAM_ERR_INVALID_ARG. */
#define ENGRAM_HOST_DEFER_OUTPUT 1u
int engram_forward_host_pipelined(engram_t* h, const void* hidden_host,
                                  const int32_t* hash_ids_host, const uint8_t* token_mask_host,
                                  void* out_host, int64_t T, uint32_t flags, cudaStream_t stream);

/* Make `stream` wait for the output copy of the handle's last
 * engram_forward_host_pipelined call (nothing to wait for: no-op; also a
 * no-op while `stream` is being captured, where the calls are ordered on
 * the stream anyway). */
int engram_forward_host_flush(engram_t* h, cudaStream_t stream);

/* Host-side error of the last call on this handle.  With sync != 0 the
 * device is synchronised and the sticky device error word is read and
 * cleared: a non-zero word returns ENGRAM_ERR_DEVICE. */
int engram_last_error(engram_t* h, int sync);

/* Read (and clear, if clear != 0) the sticky device error word into *bits
 * (ENGRAM_DEVERR_* bits).  Synchronises the device. */
int engram_device_error(engram_t* h, uint32_t* bits, int clear);

/* class EngramLayout: bucket sizes for n_layers layers.  For every layer
 * and n-gram order 2..max_ngram_size the counter restarts at vocab_size - 1
 * and each of n_heads heads takes the next prime above it not used before.
 * primes, offsets: HOST [n_layers, (max_ngram_size-1)*n_heads]; offsets are
 * the exclusive cumulative sums within a layer.  Pure host function. */
int engram_layout(int64_t vocab_size, int32_t max_ngram_size, int32_t n_heads,
                  int32_t n_layers, int64_t* primes, int64_t* offsets);

/* Validation hook (not part of the layer's semantics): after a forward on
 * this handle's stream, writes the fp32 gate [T, H] and value [T, D] of the
 * last call into device buffers, on `stream`.  A gate of 0 marks masked
 * tokens. */
int engram_debug_intermediates(engram_t* h, float* gate, float* value, int64_t T,
                               cudaStream_t stream);

/* Validation hook: with enable != 0, later forwards on the fused decode
 * path also store the fp32 value [T, D] (an extra T*D*4 bytes written per
 * call) so that engram_debug_intermediates can return it; otherwise that
 * call returns ENGRAM_ERR_INVALID_ARG for the value of a fused forward.
 * Off by default.  The prefill path always keeps its bf16 value. */
int engram_debug_keep_value(engram_t* h, int enable);

/* Validation hook: copy the staged rows [T, K] bf16 (the gather output) of
 * the last lookup into `rows` (device), on `stream`. */
int engram_debug_staged_rows(engram_t* h, void* rows, int64_t T, cudaStream_t stream);

/* Gate and masked residual only, over a projection computed by the caller,
 * with NO handle and NO device memory allocation on any call.
 *
 * The documented Engram layer has no such entry point: it is here for
 * callers that cannot allocate device memory while they serve -- engines
 * that run the wkv projection with their own GEMM and have already given
 * nearly all of HBM to their own pools (a cudaMalloc there can fail, and
 * cudaMalloc/cudaFree synchronise the device).
 *
 * Arithmetic: as engram_forward, split into partial sums per 256-dim slice
 * that are added in slice order (the partials/finish split of the gate in
 * "vllm.models.deepseek_v41.amd.engram", slices in place of ranks).
 *   hidden, out: device bf16 [T, H, D], strides as for engram_forward;
 *       out's rows must not overlap each other, out may be hidden itself
 *       (same pointer and strides), and any other overlap of out with
 *       hidden, kv, q_weight, k_weight or token_mask is INVALID_ARG.
 *   kv: device bf16 [T, (H+1)*D] with row stride kv_row_stride >= (H+1)*D
 *       elements (a multiple of 8): keys of copy h in columns [h*D, (h+1)*D),
 *       the shared value in [H*D, (H+1)*D).
 *   q_weight, k_weight: device bf16 [H, D] contiguous.
 *   token_mask: device bytes [T] (0 = False) or NULL.
 *   1 <= H <= 4; D a multiple of 256, at most 8192.
 * Scratch: one fixed array of ENGRAM_NOALLOC_MAX_PARTIALS 16-byte slots per
 * device, inside the library's device image; a call uses T * H * (D / 256)
 * slots and returns ENGRAM_ERR_SCRATCH_LIMIT, launching nothing, if that is
 * more.  No slot needs to start at zero (a call writes every slot it reads).
 * Calls on one device share the array: two calls that can run at the same
 * time (unordered streams, concurrent host threads) corrupt each other's
 * results, so order them.  The first call on each device (T = 0 does only
 * this) looks up the array's address and may load the library's device code
 * there; make it before capturing a stream.  The address is kept per device
 * together with the id of the context that was current, and looked up again
 * when another context is current there (after cudaDeviceReset, or a
 * caller's own driver-API context): make a T = 0 call after such a change,
 * before any capture.  Uses the current device. */
#define ENGRAM_NOALLOC_MAX_PARTIALS 131072
int engram_gate_noalloc(const void* hidden, const int64_t hidden_strides[3], const void* kv,
                        int64_t kv_row_stride, const void* q_weight, const void* k_weight,
                        const uint8_t* token_mask, void* out, const int64_t out_strides[3],
                        int64_t T, int64_t H, int64_t D, double eps, double clamp,
                        cudaStream_t stream);

/* Validation hook, MXFP8 handles only: copy the e4m3 codes [T, K] and the
 * E8M0 scales [T, K/32] (one per 32 consecutive k, row-major) of the rows
 * the last lookup or forward staged into device buffers, on `stream`.
 * Either pointer may be NULL. */
int engram_debug_staged_mx(engram_t* h, uint8_t* codes, uint8_t* scales, int64_t T,
                           cudaStream_t stream);

/* Measurement hook: with enable != 0, later engram_forward calls record a
 * CUDA event before and after each of their kernels on the call's stream
 * (this serialises the kernels, so programmatic launch overlap is lost).
 * engram_profile_read waits for the last recorded forward and writes the
 * durations in milliseconds of its gather, wkv and gate kernels into
 * ms[0..2] (0 for a kernel that did not run). */
int engram_profile_enable(engram_t* h, int enable);
int engram_profile_read(engram_t* h, float ms[3]);

/* Test hook for failure detection: adds delta (>= 0) to the fused decode
 * kernel's launch counter.  With delta > 0 the next fused launch waits at
 * its grid barriers for arrivals that never come.  Each bounded wait runs out
 * (1 s); the launch sets ENGRAM_DEVERR_TIMEOUT, lets its copies and MMAs
 * land, frees TMEM and returns without writing out.  engram_device_error
 * then reports the bit and resets the counters, and the next launch runs
 * normally.  Synchronous.  Nothing faults, traps or hangs. */
int engram_debug_barrier_skew(engram_t* h, int64_t delta);

/* The wkv projection alone: kv = rows . wkv^T rounded to bf16, the output of
 * Engram.forward's wkv (class Engram on the page
 * "vllm.models.deepseek_v4_1.common.engram"): keys of copies h = 0..H-1 in
 * columns [h*D, (h+1)*D), then the value in [H*D, N).  rows are gathered
 * from hash_ids (device int32 [T, C], row stride >= C), or with hash_ids
 * NULL taken from the last engram_lookup of the same T.  kv: device bf16
 * [T, kv_row_stride], 16-byte aligned, kv_row_stride >= N and a multiple of
 * 8.  Decode-sized T only (the configurations engram_forward runs in one
 * fused launch: T <= 256, MXFP8 T <= 128); others return
 * ENGRAM_ERR_UNSUPPORTED.  engram_gate_noalloc finishes the layer from kv. */
int engram_wkv(engram_t* h, const int32_t* hash_ids, int64_t ids_row_stride, void* kv,
               int64_t kv_row_stride, int64_t T, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Lookups of several layers run ahead on a side stream.  This follows the
 * prefetch page ("vllm.models.deepseek_v41.nvidia.specialized_decode.
 * engram.prefetch": class EngramPrefetch with start, forward and join, and
 * the module note on looking up rows on a prefetch stream ahead of the
 * decoder layers) and Engram.prepare_embeddings.  The engine learns a step's
 * hash ids before its decoder layers run.  engram_prefetch_start stages
 * every layer's rows at that point; each layer's forward then waits only
 * for its own rows.  The pages' side-stream wkv chain is not part of this.
 *
 * Host-side orchestration only: no kernel of its own.
 * engram_prefetch_create
 *   flags: 0, or ENGRAM_PREFETCH_WKV: where a layer's fused decode launch
 *   serves the start's T, start runs engram_wkv instead of the lookup into
 *   a kv buffer the prefetcher owns (allocated here), and the layer's
 *   forward is engram_gate_noalloc over it -- the pages' side-stream wkv
 *   chain; other T fall back to the lookup.
 *   layers: n_layers >= 1 handles on one device.  They are borrowed and must
 *   outlive the prefetcher; while it lives, only it may call engram_lookup
 *   on them.  It owns a non-blocking side stream and one event per layer.
 * engram_prefetch_start
 *   Orders the side stream after all work issued on `stream` so far.  That
 *   covers the hash ids, and the previous step's forwards if they ran on
 *   `stream`: their staged rows are about to be overwritten.  Then, on the
 *   side stream, it runs engram_lookup(layers[l], hash_ids[l],
 *   ids_row_stride[l], T, background) for every layer and records the
 *   layer's event.  hash_ids[l]: device int32 [T, C_l] with row stride
 *   ids_row_stride[l] >= C_l.  Each layer is then "pending".  Returns the
 *   first failing lookup's code; the layers before it stay pending.
 * engram_prefetch_forward
 *   Layer `layer`'s engram_forward on `stream`.  If the layer is pending,
 *   `stream` first waits on the layer's event, and the forward consumes the
 *   staged rows: T must equal the start's T, and hash_ids is ignored.  If
 *   not, it is the plain forward and needs hash_ids.  Either way the layer
 *   is no longer pending afterwards.
 * engram_prefetch_join
 *   Makes `stream` wait for every pending layer's lookup and clears the
 *   pending flags.  Call it before ending a stream capture that started the
 *   prefetch and did not forward every layer.
 * engram_prefetch_pending
 *   1 if the layer is pending, 0 if not, ENGRAM_ERR_INVALID_ARG for a bad
 *   argument.
 * A stream capture of start / forward / join on one stream records the side
 * stream's work into the graph. */
typedef struct engram_prefetch engram_prefetch_t;
#define ENGRAM_PREFETCH_WKV 1  /* flags: also run each layer's wkv on the side stream */
int engram_prefetch_create(engram_t* const* layers, int32_t n_layers, int32_t flags,
                           engram_prefetch_t** out);
int engram_prefetch_destroy(engram_prefetch_t* p);
int engram_prefetch_start(engram_prefetch_t* p, const int32_t* const* hash_ids,
                          const int64_t* ids_row_stride, int64_t T, int background,
                          cudaStream_t stream);
int engram_prefetch_forward(engram_prefetch_t* p, int32_t layer, const void* hidden,
                            const int64_t hidden_strides[3], const int32_t* hash_ids,
                            int64_t ids_row_stride, const uint8_t* token_mask, void* out,
                            const int64_t out_strides[3], int64_t T, cudaStream_t stream);
int engram_prefetch_join(engram_prefetch_t* p, cudaStream_t stream);
int engram_prefetch_pending(const engram_prefetch_t* p, int32_t layer);

#ifdef __cplusplus
}
#endif

#endif /* ENGRAM_GB300_H */
