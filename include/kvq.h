/*
 * kvq.h - quantised KV-cache append and decode attention on one GB300 GPU.
 *
 * The calls follow the problem statement of four pages:
 *   [P1] posttrainllm, "StreamingLLM + KIVI - long-context decode without
 *        growing the KV cache" (sections "StreamingLLM - Implementation",
 *        "RoPE caveat", "KIVI", "Affine quantisation formula", "Caveats").
 *   [P2] Foundry, "TurboQuant KV Cache Compression - Spec" (sections
 *        "Algorithm Detail", "API", "Codebook Generation",
 *        "Optimization: Fused dequant-dot").
 *   [P3] PR #2318, "KV cache: FP16 sliding window + attention sinks, and an
 *        optional 2-bit K / 4-bit V cache scheme" (section "Summary").
 *   [P4] VeloxQuant-MLX, "KVSink-Adapted Sink Protection" (sections
 *        "Usage", "How it works", "Known v1 limitation").
 *
 * Conventions for every call:
 *   - Device pointers are CUDA global-memory addresses on the device that
 *     was current when the cache was created; host pointers are ordinary
 *     process memory. The library never allocates device memory: the caller
 *     passes one device arena to kv_cache_create and owns it.
 *   - `cuda_stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream). Work is enqueued on it and the call returns without waiting,
 *     except where a call says it synchronises.
 *   - The library keeps the host-side counters of each layer (tokens
 *     appended L, eviction end E) and advances them when work is enqueued,
 *     so the decode loop needs no device-to-host read.
 *   - Every call returns a kv_status. Arguments are checked before anything
 *     is enqueued; a call that fails leaves the cache unchanged. The text of
 *     the last error of the calling thread is in kv_last_error().
 *   - One cache may be used by one host thread at a time; calls on one
 *     cache must be enqueued on streams that are ordered with each other.
 *   - Tensor layouts are dense, row-major, in the order written ([B,H,T,D]
 *     means D fastest).
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KV_OK = 0,
  KV_ERR_INVALID_ARG = 1, /* bad pointer, size, layer or configuration      */
  KV_ERR_CAPACITY = 2,    /* the append would exceed the cache's capacity   */
  KV_ERR_UNSUPPORTED = 3, /* a valid request this build does not implement  */
  KV_ERR_CUDA = 4,        /* a CUDA runtime call failed (text in last error) */
  KV_ERR_TIMEOUT = 5,     /* a bounded device wait gave up (device flag)     */
  KV_ERR_STATE = 6        /* the call does not fit the cache's state         */
} kv_status;

typedef enum { KV_MODE_KIVI = 0, KV_MODE_TURBOQUANT = 1 } kv_mode;
typedef enum { KV_DT_F16 = 0, KV_DT_BF16 = 1 } kv_dtype;

/*
 * Cache configuration (P4 "Usage": method, bit width, group size, residual
 * length, number of sink tokens; P1 flags --streaming-llm-sink/-window and
 * --kv-quantize; P3 --kv-window; P2 fa_tq_config and the seed of fa_tq_init).
 */
typedef struct {
  int n_layers;
  int batch;          /* B: sequences                                       */
  int n_kv_heads;     /* Hkv                                                */
  int n_q_heads;      /* Hq, a multiple of Hkv with Hq / Hkv <= 4           */
  int head_dim;       /* D: 64 or 128                                       */
  int64_t max_tokens; /* retained-token capacity per sequence per layer: the
                         span from the first stored quantised group to the
                         newest token may not exceed it                      */
  kv_mode mode;
  int k_bits, v_bits; /* KIVI: 2, 3, 4 or 8 each. TurboQuant: 2, 3 or 4.
                         Codes are packed tight: 3-bit codes eight to three
                         bytes ([P2] "Step 3: Packing", the no-waste form)  */
  int group_size;     /* KIVI token/channel group: must be 32               */
  int residual;       /* fp16 residual tail before a group is quantised:
                         32 (one group) in KIVI mode, 0 in TurboQuant mode  */
  int n_sink;         /* StreamingLLM first-N positions read exact (<= 32)  */
  int window;         /* most recent positions read exact (0 = none)        */
  int evict_window;   /* StreamingLLM retention window W_keep: 0 = never
                         evict, else >= max(window, 32)                     */
  int n_dyn_sinks;    /* KVSink top-k sinks (0 = off, <= 32; KIVI only, and
                         only with n_sink = window = evict_window = 0)      */
  kv_dtype act_dtype; /* dtype of K, V, q given to the cache; the exact
                         pools (sinks, window, residual) keep this dtype    */
  uint64_t seed;      /* TurboQuant sign seed (SplitMix64)                  */
  double rope_base;   /* > 0: the cache rotates keys at their absolute
                         position on append and the query at position L-1
                         on decode (vanilla RoPE, half-split pairs);
                         0: the caller applies RoPE                         */
  int64_t rope_max_pos; /* positions the RoPE table covers (rope_base > 0) */
  int max_splits;     /* upper bound on split-KV partitions per (b, h);
                         0 = library default (64)                           */
  int rope_reposition; /* 1 (with rope_base > 0): StreamingLLM position
                         re-encoding at read ([P1] "RoPE caveat"): every kept
                         key is read as if rotated at its slot in the cache
                         (sinks at 0 .. n_sink-1, the kept tokens after them
                         without the evicted gap) and the query at its own
                         slot. Relative rotations change only between the
                         query and the sinks, so the library reads the sink
                         rows against the query rotated at
                         L - 1 - (E - n_sink) and everything else as in the
                         vanilla scheme. 0: vanilla (absolute positions)    */
  int v_q4_0;         /* 1 (KIVI, v_bits = 4): V in the symmetric q4_0 form
                         ([P3] "Summary": V at 4 bits per token, q4_0): per
                         32 values d = m / -8 with m the value of largest
                         magnitude (the first on ties), code
                         min(15, floor(x / d + 8.5)), value (code - 8) d;
                         stored as scale d and zero -8 d (fp16). The codes
                         divide x by the STORED fp16 d with a correctly
                         rounded division (as the KIVI codes use the stored
                         scale); the widely used q4_0 quantiser instead
                         multiplies x by 1 / d of the fp32 d, so a code at
                         a rounding boundary can differ by one step and the
                         blocks are not interchangeable with such data.
                         0: the KIVI min/max affine form                    */
  int k_pre_rope;     /* 1 (KIVI, rope_base > 0, n_dyn_sinks = 0): keys are
                         stored (quantised, and in the exact pools) before
                         RoPE and rotated when read, at their absolute
                         position or, with rope_reposition, at their slot in
                         the cache (the query at its own slot) ([P1] "RoPE
                         caveat": the "true" re-positioning; "Caveats": the
                         per-channel K groups then see a basis that does not
                         turn with the position). 0: keys rotated before
                         they are stored                                    */
} kv_cache_config;

typedef struct kv_cache kv_cache; /* opaque host-side handle */

/* Token counts per read pool summed over the batch, and the bytes each pool
 * holds (all KV heads and the batch included). The pools partition the
 * tokens: n_quant + n_sink + n_tail + n_evicted == batch * length
 * (P4 "How it works" 4: sink and residual bytes counted apart). */
typedef struct {
  int64_t length;     /* L: tokens appended so far (absolute positions)     */
  int64_t evict_end;  /* E: positions [n_sink, E) are evicted               */
  int64_t quant_end;  /* Q_end: positions below it have codes               */
  int64_t fp16_begin; /* F: positions [F, L) are read from the exact tail   */
  int64_t n_quant, n_sink, n_tail, n_evicted;
  int64_t code_bytes;  /* packed K and V codes of the quantised pool         */
  int64_t kmeta_bytes; /* KIVI: fp16 K scale+zero of the groups read;
                          TurboQuant: fp32 K norms                           */
  int64_t vmeta_bytes; /* KIVI: fp16 V scale+zero per token and 32 channels;
                          TurboQuant: fp32 V norms                           */
  int64_t sink_bytes;  /* exact K and V rows read from the sink buffer       */
  int64_t tail_bytes;  /* exact K and V rows read from the tail              */
} kv_cache_stats_t;

/* Bytes of device memory kv_cache_create needs for `cfg` (256-byte aligned
 * arena). Host-only. */
kv_status kv_cache_required_bytes(const kv_cache_config* cfg, size_t* device_bytes);

/* Create a cache in the caller's device arena (at least
 * kv_cache_required_bytes, 256-byte aligned). Builds the tables the mode
 * needs (TurboQuant codebooks for Beta(D/2, D/2) by Lloyd-Max, P2 "Codebook
 * Generation"; the sign diagonal from `seed`; the RoPE table) on the host and
 * uploads them; synchronises the device. The arena must stay allocated until
 * kv_cache_destroy. *out receives the handle. */
kv_status kv_cache_create(const kv_cache_config* cfg, void* device_arena, size_t arena_bytes,
                          kv_cache** out);
kv_status kv_cache_destroy(kv_cache* cache);

/* Empty every layer (L = 0, no sinks) without touching the arena's data. */
kv_status kv_cache_reset(kv_cache* cache);

/*
 * Append n_new tokens to one layer (P1 "KIVI": per-layer cache.append;
 * P1 "RoPE caveat": keys keep the rotation of their absolute position).
 * k, v: device [B, Hkv, n_new, D] in act_dtype; the tokens take absolute
 * positions L .. L+n_new-1. Each 32-token group that completes is quantised
 * (KIVI: K per channel over the group, V per token over 32-channel groups,
 * min/max affine codes, P1 "Affine quantisation formula"; TurboQuant: every
 * token at once, P2 "Algorithm Detail"); the rest waits in the exact tail.
 * Positions below n_sink are also copied to the sink buffer. When
 * n_dyn_sinks > 0 (KVSink, P4 "How it works" 1-3), the call first folds its
 * tokens into each sequence's running top-k of key norms (the L2 norm of
 * each head's key averaged over the KV heads; norm descending, ties to the
 * lower position): the candidates are the call's tokens and the sinks whose
 * group was still unquantised when the call began; sinks in quantised
 * groups are locked (P4 "Known v1 limitation": a token quantised in an
 * earlier call is never restored), and the set holds min(n_dyn_sinks, L)
 * positions. Sink K/V rows are stored exact, and in every group quantised
 * afterwards each sink row is replaced by its nearest non-sink row of the
 * group before min/max calibration. Errors: KV_ERR_CAPACITY when the
 * retained span would exceed max_tokens (or the RoPE table), nothing
 * enqueued.
 */
kv_status kv_append(kv_cache* cache, int layer, const void* k, const void* v, int n_new,
                    void* cuda_stream);

/*
 * Prefill: the same state change as kv_append of the same n_tokens tokens
 * (KVSink selection included: on an empty layer it is the top n_dyn_sinks
 * positions of the call), run by a bulk quantiser sized for long inputs.
 */
kv_status kv_prefill_quantize(kv_cache* cache, int layer, const void* k, const void* v,
                              int n_tokens, void* cuda_stream);

/*
 * StreamingLLM eviction for one layer (P1 "StreamingLLM - Implementation":
 * after each per-layer append drop [sink, len - window)). When
 * L - evict_window > E, positions [E, L - evict_window) are dropped and E
 * moves to L - evict_window. Host-only (no data moves: quantised groups keep
 * their frozen scales; a group's slot is reused once every token in it is
 * evicted). *evicted_begin / *evicted_end receive the absolute range
 * (equal when nothing was dropped).
 */
kv_status kv_evict(kv_cache* cache, int layer, int64_t* evicted_begin, int64_t* evicted_end);

/*
 * Decode attention for one layer (P2 "Optimization: Fused dequant-dot";
 * P3 "Summary": sinks and the recent window read exact, the rest quantised).
 * q: device [B, Hq, D] act_dtype, 4-byte aligned (un-rotated when the cache
 * applies RoPE; it is rotated at position L-1). out: device [B, Hq, D] fp32
 * (4-byte aligned) =
 * softmax(q K^T / sqrt(D)) V over every retained position; query head j
 * reads KV head j / (Hq / Hkv). lse_or_null: device [B, Hq] fp32 natural-log
 * softmax denominator, or NULL. Split-KV: the quantised segment is cut into
 * partitions whose partial (max, sum, output) are merged by log-sum-exp.
 * Errors: KV_ERR_STATE on an empty layer.
 */
kv_status kv_decode_attn(kv_cache* cache, int layer, const void* q, float* out,
                         float* lse_or_null, void* cuda_stream);

/* Size in bytes of the library's own decode scratch block (32 MiB). */
#define KV_NOALLOC_SCRATCH_BYTES (32u << 20)

/*
 * kv_decode_attn with no allocation: the same computation, arguments and
 * errors, but the split partials go to a fixed block of device memory that
 * the library declares itself (KV_NOALLOC_SCRATCH_BYTES, reserved on every
 * GPU that loads the library until the process exits) instead of the
 * arena's partial region, which this call leaves untouched. The papers have
 * no counterpart of this entry point: it is for callers that may not
 * allocate device memory at decode time, such as a serving loop whose pool
 * has already reserved the whole GPU, a plug-in or custom operator that its
 * host framework gives no allocator, or a latency-bound loop that cannot
 * afford the device-wide synchronisation a cudaMalloc or cudaFree brings.
 * It calls no cudaMalloc, cudaFree or other allocating routine.
 * Limit: the partials take
 *   align256(batch * n_q_heads * (max_splits + 1) * head_dim * 4)
 *   + align256(batch * n_q_heads * (max_splits + 1) * 2 * 4)
 * bytes; a cache that needs more than KV_NOALLOC_SCRATCH_BYTES gets
 * KV_ERR_CAPACITY before anything is launched.
 * The cache's device must be current (KV_ERR_INVALID_ARG otherwise). The
 * first call on a device looks up the block's device address once
 * (cudaGetSymbolAddress); make that first call before any stream capture.
 * The address is kept for the life of the process: after cudaDeviceReset
 * (or anything else that creates a new primary context on the device) the
 * block may load elsewhere, so make no further call of this entry point in
 * that process.
 * Every call shares the one block and it keeps the last call's contents
 * (nothing in it needs clearing: each call writes every partial it reads).
 * Calls whose kernels overlap on the GPU (unordered streams, several host
 * threads) race on the block: order them on one stream or with events.
 */
kv_status kv_decode_attn_noalloc(kv_cache* cache, int layer, const void* q, float* out,
                                 float* lse_or_null, void* cuda_stream);

/* Host-only counters and byte accounting of one layer. In KVSink mode this
 * call reads the sink positions back (it synchronises the device). */
kv_status kv_cache_stats(kv_cache* cache, int layer, kv_cache_stats_t* out);

/* What kv_cache_export copies, in canonical (page-defined) layout. Ranges:
 * quantised tokens [T0, T1) = [32 * floor(E / 32), Q_end), n = T1 - T0;
 * G = n / 32 groups (KIVI); S = sinks stored per sequence; R = L - F. */
enum {
  KV_EXPORT_K_CODES = 0,  /* u8  [B][Hkv][n][D*k_bits/8]: each row one
                             little-endian bit string along D, code c at
                             bits c*k_bits .. (c+1)*k_bits-1                */
  KV_EXPORT_K_SCALE = 1,  /* f16 [B][Hkv][G][D]     (KIVI)                   */
  KV_EXPORT_K_ZERO = 2,   /* f16 [B][Hkv][G][D]     (KIVI)                   */
  KV_EXPORT_V_CODES = 3,  /* u8  [B][Hkv][n][D*v_bits/8], as K_CODES        */
  KV_EXPORT_V_SCALE = 4,  /* f16 [B][Hkv][n][D/32]  (KIVI)                   */
  KV_EXPORT_V_ZERO = 5,   /* f16 [B][Hkv][n][D/32]  (KIVI)                   */
  KV_EXPORT_K_NORM = 6,   /* f32 [B][Hkv][n]        (TurboQuant)             */
  KV_EXPORT_V_NORM = 7,   /* f32 [B][Hkv][n]        (TurboQuant)             */
  KV_EXPORT_SINK_POS = 8, /* i64 [B][S] ascending (the library keeps KVSink
                             slots in admission order; the export sorts)    */
  KV_EXPORT_SINK_K = 9,   /* act [B][Hkv][S][D], rows in SINK_POS order       */
  KV_EXPORT_SINK_V = 10,  /* act [B][Hkv][S][D], rows in SINK_POS order       */
  KV_EXPORT_TAIL_K = 11,  /* act [B][Hkv][R][D]                              */
  KV_EXPORT_TAIL_V = 12,  /* act [B][Hkv][R][D]                              */
  KV_EXPORT_SINK_MASK = 13, /* u32 [B][G] bit r: token 32g+r is a sink (KIVI) */
  KV_EXPORT_CODEBOOK_K = 14, /* f32 [2^k_bits - 1 boundaries, 2^k_bits centroids] (TQ) */
  KV_EXPORT_CODEBOOK_V = 15, /* f32, as above for v_bits                     */
  KV_EXPORT_TQ_SIGNS = 16,   /* f32 [D] of +-1                                */
  KV_EXPORT_ROPE = 17        /* f32 [rope_max_pos][D/2][2] (cos, sin)         */
};

/* Bytes kv_cache_export would copy for (layer, what) now. Host-only. */
kv_status kv_cache_export_bytes(kv_cache* cache, int layer, int what, size_t* bytes);

/* Copy one array of one layer to host memory in canonical layout; `bytes`
 * must equal kv_cache_export_bytes. Synchronises `cuda_stream`. A test and
 * inspection path (P2 keeps fa_tq_dequantize for the same purpose). */
kv_status kv_cache_export(kv_cache* cache, int layer, int what, void* host_dst, size_t bytes,
                          void* cuda_stream);

/* Read and clear the device error flag that bounded waits set when they give
 * up. Synchronises `cuda_stream`. KV_ERR_TIMEOUT when it was set. */
kv_status kv_cache_check_device_error(kv_cache* cache, void* cuda_stream);

/* Test hook of the failure path: one launch whose bounded device waits run
 * out on purpose (no fault, no hang). Two mbarriers that nothing arrives at
 * and no copy completes on are waited for by the same wait routines the
 * decode kernels use: one warp with `budget_cycles` SM clock cycles (in
 * [1000, 2^31]), a second warp with the default budget of about one second,
 * which must give up early through the abort flag the first warp raises,
 * then one thread through the two single-thread forms. Each give-up sets the
 * cache's device error flag, so a following kv_cache_check_device_error
 * returns KV_ERR_TIMEOUT (and clears it); the cache's data is untouched.
 * host_result receives 5 int64: per wait 1 if it returned "completed" (must
 * all be 0), then the SM cycles the second warp waited. Synchronises
 * `cuda_stream`. */
kv_status kv_cache_test_bounded_wait(kv_cache* cache, int64_t budget_cycles, int64_t* host_result,
                                     void* cuda_stream);

/* Optional timing hook: when both are non-NULL, kv_decode_attn records
 * ev_begin (a cudaEvent_t) right before its split kernel and ev_end right
 * after its merge kernel (the whole decode), on the call's stream. Pass
 * NULLs to turn it off. */
kv_status kv_cache_set_timing_events(kv_cache* cache, void* ev_begin, void* ev_end);

/* Number of kernels this library has launched in this process. */
int64_t kv_launch_count(void);

/* Device-to-device copy of `bytes` (a multiple of 16, both pointers 16-byte
 * aligned) with 16-byte vector loads and stores: the bandwidth reference the
 * decode kernel's effective bandwidth is compared with. */
kv_status kv_copy_bandwidth_kernel(const void* src, void* dst, size_t bytes, void* cuda_stream);

/* Thread-local text of the last failing call on this thread. */
const char* kv_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
