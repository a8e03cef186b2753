/*
 * libkvq -- quantized KV cache with fused decode attention, for GB300 (sm_103a).
 *
 * C ABI.  Plain pointers and sizes only; no CUDA or framework types in the
 * signatures (a stream is passed as `void *`, meaning a cudaStream_t; NULL is
 * the legacy default stream).  Every device buffer is allocated and owned by
 * the caller; the library never allocates device or host memory.  Calls are
 * asynchronous on the given stream unless stated otherwise.
 *
 * Method (page title, section):
 *   [KIVI]   "大模型量化技术原理：KIVI、IntactKV、KVQuant" (juejin.cn), KIVI /
 *            背景 and 工作原理: keys quantized per channel in groups of G
 *            tokens, values per token; the newest tokens stay fp16 in a
 *            residual that is quantized and appended every R tokens.
 *   [HF]     pgsm.cn KV-cache quantization how-to, §2.1 (asymmetric form
 *            X_Q = round(X/S) - Z) and §3.1 (fp16 residual buffer, quantized
 *            as a batch when full).
 *   [INNERQ] "【论文】InnerQ：硬件感知免调优KV缓存量化用于大语言模型"
 *            (euno.news), 方法论 1-5: groups along the inner (head) dimension,
 *            per-group symmetric/asymmetric choice, fp16 sink and recent
 *            windows, dequantization fused into the GEMV.
 *   [KVQ5]   the juejin page, KVQuant / 技术原理 五: first token kept fp16.
 *   [IKV]    the juejin page, IntactKV / KV Cache量化: fp16 tokens joined
 *            with the dequantized cache at attention time.
 *
 * Quantization formula (asymmetric, fp32, IEEE round-to-nearest-even):
 *   scale = (max - min) / (2^b - 1), zero = min,
 *   code  = clamp(rint((x - min) / scale), 0, 2^b - 1); x_hat = code*scale + zero.
 *   A constant group stores scale 0 and code 0.
 * Symmetric (InnerQ groups whose midpoint |max + min| <= (max - min)/(2^b - 1)):
 *   scale = max(|min|, |max|) / (2^(b-1) - 1), q = clamp(rint(x / scale)),
 *   code = q + 2^(b-1), zero = -2^(b-1) * scale (same dequantization formula).
 *
 * Packed layout.  cap = max_ctx rounded up to a multiple of 128 is the
 * per-head token capacity.  Every per-token quantity of the quantized region
 * lives in 32-token blocks, so one contiguous read fetches everything a
 * 32-token tile needs except the KIVI key statistics for G >= 64.  M below is
 * f32, or fp16 under KVQ_META_F16 (m = its size in bytes, 4 or 2):
 *   blocks  u8 [B][H][cap/32][block_bytes]; block j of a head holds tokens
 *           32j .. 32j+31 (token t at row i = t mod 32) as
 *             K codes  [32][d*bits/8]    channel c of a row at bits
 *             V codes  [32][d*bits/8]    (c mod (8/bits))*bits of byte c/(8/bits)
 *             V scale  M [32][d/v_group]   (per token, channel group)
 *             V zero   M [32][d/v_group]
 *             InnerQ only:
 *             K scale  M [32][d/k_group]   (per token, channel group)
 *             K zero   M [32][d/k_group]
 *             KIVI with G <= 32 only:
 *             K stats  M [32/G][2][d]  per key group of the block: scale
 *                      row, then zero (= min) row, one value per channel
 *             KIVI with o = cfg.outliers > 0 only:
 *             K outliers u32 [32][o]  per token: (channel << 16) | fp16 bits
 *             V outliers u32 [32][o]  of its o outliers, channels ascending
 *           block_bytes = 64*d*bits/8 + 64*m*(d/v_group + (InnerQ ? d/k_group : 0))
 *                         + (KIVI, G <= 32 ? (32/G)*2*m*d : 0) + 256*o,
 *           a multiple of 128.
 *           KVQ_INNERQ_KNORM: the blocks buffer ends with the key factors
 *             f32 [B][H][d] (n_c above), after the last head's blocks.
 *   KIVI with G >= 64:
 *           k_meta  M [B][H][cap/G][2][d]  the same two rows per key group
 *           (the buffer carries 64 bytes of slack after the last head)
 *   KIVI:   k_res, v_res   fp16 [B][H][R][d]  residual, oldest first; with
 *                           KVQ_VALUE_QUEUE, v_res is a ring: the fp16 value
 *                           of token t sits in slot t mod R
 *   InnerQ: k_mode, v_mode  u32 [B][H][cap*(d/group)/32]  bit i = group
 *                           i % (d/group) of token i / (d/group); 1 = symmetric
 *           k_res, v_res   fp16 [B][H][W][d]   recent window, a ring (see ring_head)
 *           k_sink, v_sink fp16 [B][H][S][d]   first S tokens
 *   KVQ_RAGGED: seq_prompt int32 [B]  each sequence's prompt length
 *   Quantized tokens occupy slots [0, n_quant) in arrival order.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes.  Validation happens before any launch; on a negative return
 * no cache state (host counters or device buffers) has changed. */
#define KVQ_OK 0
#define KVQ_EINVAL (-1)       /* null pointer, negative size, inconsistent config */
#define KVQ_EUNSUPPORTED (-2) /* valid but not built: head_dim, bits, group sizes */
#define KVQ_ECAPACITY (-3)    /* the call would exceed max_ctx or the workspace */
#define KVQ_EALIGN (-4)       /* a device buffer is not 16-byte aligned */
#define KVQ_ECUDA (-5)        /* a CUDA launch or copy failed */
#define KVQ_ETIMEOUT (-6)     /* a bounded device-side wait gave up (status word) */

#define KVQ_KIVI 0
#define KVQ_INNERQ 1
#define KVQ_INNERQ_KNORM 2 /* InnerQ with the one-shot per-channel key normalization */

/* Cache-format options (kvq_config.flags). */
#define KVQ_META_F16 1u    /* scales and zero points stored in fp16 */
#define KVQ_VALUE_QUEUE 2u /* KIVI: values leave the fp16 residual one at a time */
#define KVQ_RAGGED 4u      /* every sequence of the batch has its own length */

/*
 * Cache configuration.
 *   batch, n_q_heads, n_kv_heads: n_q_heads % n_kv_heads == 0; query head hq
 *     reads KV head hq / (n_q_heads / n_kv_heads) (GQA; MHA when equal).
 *   head_dim d: 64 or 128.   bits: 2 or 4.
 *   scheme KVQ_KIVI: k_group = G tokens per key group (16, 32, 64 or 128),
 *     v_group = channels per value group (multiple of 16 dividing d),
 *     residual = R (multiple of G, <= 1024), n_sink must be 0.
 *   scheme KVQ_INNERQ: k_group and v_group = channels per group (multiples of
 *     16 dividing d), residual = W recent fp16 tokens (0..1024), n_sink = S
 *     fp16 sink tokens (0..1024).
 *   scheme KVQ_INNERQ_KNORM: KVQ_INNERQ plus the one-shot per-channel key
 *     normalization ("InnerQ" paper summary, key contributions and
 *     methodology 4: keys scaled once per channel at prefill, the factor
 *     folded into the query).  kvq_quantize_prefill sets the factor n_c of
 *     channel c of every head to the largest |K[t][c]| over the T prompt
 *     tokens (1 if that is 0 or T = 0); every key that is quantized (now or
 *     when it later leaves the window) is first multiplied, in fp32, by
 *     r_c = 1 / n_c (fp32 division); decode multiplies q by n_c for the
 *     quantized tokens.  Sinks and window stay the raw fp16 keys.
 *   max_ctx: most tokens one sequence will hold (prompt + appended), at most
 *     2^30 (KVQ_EUNSUPPORTED above).
 *   flags: any of
 *     KVQ_META_F16 (pgsm.cn how-to §3.1 stores the residual design without
 *       fixing the statistics' precision): the fp32 scale and zero of the
 *       formula are each rounded once to fp16 (IEEE nearest-even) and the
 *       codes are taken with the stored values, code = clamp(rint((x -
 *       zero16) / scale16)) (symmetric: q = clamp(rint(x / scale16)), zero =
 *       -2^(b-1) * scale16), so dequantization uses exactly what is stored; a
 *       scale that rounds to 0 is a constant group.  Needs |x| small enough
 *       that every stored value is finite (|x| <= 8192 covers every case).
 *     KVQ_VALUE_QUEUE (KIVI only; [KIVI] 工作原理, value paragraph: the
 *       newest values wait in a queue, and once it reaches R the oldest is
 *       quantized): after n tokens the last min(n, R - 1) values are fp16 and
 *       the first max(0, n - R + 1) are quantized per token; keys still flush
 *       every R tokens.
 *     KVQ_RAGGED: sequences have their own prompt lengths
 *       (kvq_quantize_prefill_ragged); every append adds one token to every
 *       sequence.
 *   outliers (KIVI only; "大模型量化技术原理", KVQuant / 技术原理 四: per
 *     vector, the outliers are kept apart in fp16 and the rest quantized over
 *     the narrower range): o in 0..8.  Each token's o largest-magnitude key
 *     elements and o largest value elements (equal magnitudes: the lower
 *     channel) are kept as (channel, fp16) lists; the statistics of every key
 *     group (each channel over its G tokens) and value group come from the
 *     other elements only (none left: scale 0, zero 0), outlier positions
 *     store code 0, and decode uses the fp16 value there.
 */
typedef struct kvq_config {
  int32_t batch;
  int32_t n_q_heads;
  int32_t n_kv_heads;
  int32_t head_dim;
  int32_t bits;
  int32_t scheme;
  int32_t k_group;
  int32_t v_group;
  int32_t residual;
  int32_t n_sink;
  int64_t max_ctx;
  uint32_t flags;
  int32_t outliers;
} kvq_config;

/* Byte sizes of the cache buffers for a configuration (0 = unused). */
typedef struct kvq_sizes {
  size_t blocks;  /* 32-token blocks of codes and per-token statistics */
  size_t k_meta;  /* KIVI key statistics for G >= 64 (0 otherwise) */
  size_t k_mode, v_mode;
  size_t k_res, v_res;
  size_t k_sink, v_sink;
  size_t status;     /* one int32 status word */
  size_t seq_prompt; /* KVQ_RAGGED: int32 per sequence (0 otherwise) */
} kvq_sizes;

/*
 * Cache view.  The caller allocates every buffer (sizes from kvq_cache_sizes,
 * 16-byte aligned), zero-fills `dev_status` once, and keeps this struct; the
 * library updates the host counters below.  Copying the struct together with
 * the buffers checkpoints the cache.
 *   n_quant   tokens in the quantized region (slots [0, n_quant))
 *   n_resid   KIVI: fp16 residual tokens (< R); InnerQ: window tokens (<= W)
 *   n_sink    InnerQ: sink tokens held (<= S)
 *   ring_head InnerQ: window slot of the oldest token once the window is full
 *   n_appended  tokens appended to every sequence since the prefill
 * Without KVQ_RAGGED lengths are uniform across the batch and the counters
 * describe every sequence.  With KVQ_RAGGED they describe the longest
 * sequence (capacity checks and launch sizes use them); sequence b holds
 * seq_prompt[b] + n_appended tokens, and its own counters follow from that
 * length exactly as a uniform cache's would (the device reads seq_prompt).
 * Every call except the prefills (which reset them) first checks that the
 * counters describe a reachable state (n_sink <= S, n_resid <= R or W, KIVI
 * n_resid < R and n_quant a multiple of R, ring_head < W, n_quant <=
 * capacity, all tokens <= max_ctx, n_appended <= all tokens) and returns
 * KVQ_EINVAL otherwise.
 */
typedef struct kvq_cache {
  void *blocks;
  void *k_meta;
  uint32_t *k_mode, *v_mode;
  uint16_t *k_res, *v_res, *k_sink, *v_sink;
  int64_t n_quant, n_resid, n_sink, ring_head;
  int32_t *dev_status;
  int32_t *seq_prompt; /* KVQ_RAGGED: device int32 [B], written by the prefill */
  int64_t n_appended;
} kvq_cache;

/* Fills *out with the byte size of each cache buffer.  Returns KVQ_OK,
 * KVQ_EINVAL or KVQ_EUNSUPPORTED.  Host only, no CUDA call. */
int kvq_cache_sizes(const kvq_config *cfg, kvq_sizes *out);

/* Bytes of scratch (device) that kvq_decode_attention needs for any cache
 * state of this configuration.  The scratch must be zero-filled before its
 * first use; every decode call that succeeds leaves it zero again.  It must
 * not be shared by decode calls that can run at the same time. */
int kvq_workspace_bytes(const kvq_config *cfg, size_t *bytes);

/*
 * Prefill: quantize a prompt of T tokens into an empty cache.
 * K, V: device fp16 [B][H][T][d], contiguous.  Resets the cache counters.
 * KIVI ([KIVI] 工作原理): tokens [0, T - T mod R) are quantized (keys per
 *   channel in groups of G tokens, values per token in groups of v_group
 *   channels); the last T mod R tokens go to the fp16 residual.
 * InnerQ ([INNERQ] 方法论 1-4): the first min(S, T) tokens go to the sink,
 *   the last min(W, T - S) to the window, the rest are quantized per token in
 *   groups of k_group / v_group channels with a per-group mode.
 *   KVQ_INNERQ_KNORM: the per-channel key factors are computed first over all
 *   T tokens and the quantized keys are normalized by them (see the scheme).
 * Errors: KVQ_EINVAL (null, T < 0), KVQ_ECAPACITY (T > max_ctx), KVQ_EALIGN,
 *   KVQ_EUNSUPPORTED, KVQ_ECUDA.
 */
int kvq_quantize_prefill(const kvq_config *cfg, kvq_cache *cache, const uint16_t *K,
                         const uint16_t *V, int64_t T, void *stream);

/*
 * Prefill of sequences with their own prompt lengths (KVQ_RAGGED; pgsm.cn
 * how-to §3.1 keeps a residual per sequence).  K, V: device fp16
 * [B][H][T_max][d], sequence b's prompt in rows [0, lens[b]) (later rows are
 * not read).  lens: HOST int32 [B], 0 <= lens[b] <= T_max <= max_ctx, copied
 * to cache->seq_prompt on `stream` (a pageable host copy: the call returns
 * once lens is no longer needed).  Each sequence is quantized exactly as
 * kvq_quantize_prefill quantizes a prompt of its length; the host counters
 * then describe the longest one.  kvq_quantize_prefill on a KVQ_RAGGED cache
 * gives every sequence the length T.
 * Errors: as kvq_quantize_prefill; KVQ_EINVAL without KVQ_RAGGED.
 */
int kvq_quantize_prefill_ragged(const kvq_config *cfg, kvq_cache *cache, const uint16_t *K,
                                const uint16_t *V, int64_t T_max, const int32_t *lens,
                                void *stream);

/*
 * Append one decode token per (batch, kv head).  k, v: device fp16 [B][H][d].
 * KIVI ([KIVI] 工作原理; [HF] §3.1): the token enters residual slot n_resid;
 *   when the residual reaches R tokens the same launch quantizes all R of them
 *   to slots [n_quant, n_quant + R) and empties the residual.
 * InnerQ: the sink fills first, then the window; once the window holds W
 *   tokens its oldest token is quantized to slot n_quant (normalized by the
 *   prompt's key factors under KVQ_INNERQ_KNORM) and the new token takes its
 *   ring slot.
 * Errors: KVQ_EINVAL, KVQ_ECAPACITY (total tokens would exceed max_ctx),
 *   KVQ_EALIGN, KVQ_ECUDA.
 */
int kvq_append(const kvq_config *cfg, kvq_cache *cache, const uint16_t *k,
               const uint16_t *v, void *stream);

/*
 * Fused decode attention over the packed cache ([KIVI] 背景: each decode
 * step reads the whole cache; [INNERQ] 方法论 3: dequantization folded into
 * the q.K^T and P.V GEMVs; [IKV]: fp16 sink / residual tokens joined with
 * the quantized ones by an online-softmax merge).
 *   q:   device fp16 [B][n_q_heads][d]
 *   out: device fp32 [B][n_q_heads][d] = softmax(softmax_scale * q.K^T) V over
 *        every token held (sink, quantized, residual / window).  An empty
 *        cache yields zeros.
 *   ws:  device scratch of ws_bytes >= kvq_workspace_bytes (see there).
 * A decode step is kvq_append followed by kvq_decode_attention.
 * Errors: KVQ_EINVAL, KVQ_ECAPACITY (ws too small), KVQ_EALIGN, KVQ_ECUDA.
 */
int kvq_decode_attention(const kvq_config *cfg, const kvq_cache *cache, const uint16_t *q,
                         float *out, float softmax_scale, void *ws, size_t ws_bytes,
                         void *stream);

/*
 * Decode attention over keys cached BEFORE the rotary position embedding
 * ("大模型量化技术原理：KIVI、IntactKV、KVQuant", KVQuant / 技术原理 二: keys
 * are quantized pre-RoPE, and the embedding is applied after dequantization
 * inside the q.K^T kernel).  The cache holds the keys exactly as they were
 * given to kvq_quantize_prefill / kvq_append (un-rotated); q is un-rotated
 * too.  RoPE (RoFormer's rotation; the pages do not spell it out): channels
 * 2i and 2i+1 of a vector at position p are turned counter-clockwise by the
 * angle p * theta_i, theta_i = rope_base^(-2i/d).  Positions: the tokens held
 * are numbered 0, 1, ... in arrival order (sinks, quantized tokens,
 * residual / window oldest first), and q belongs to the newest token.
 *   out = softmax(softmax_scale * RoPE(q) . RoPE(K)^T) V, fp32, as
 *   kvq_decode_attention (values are not rotated; an empty cache gives zeros).
 *   ws: the decode scratch (kvq_workspace_bytes; zero-filled, left zero).
 * Errors: as kvq_decode_attention; KVQ_EINVAL for rope_base <= 0 or not
 *   finite; KVQ_EUNSUPPORTED for n_q_heads / n_kv_heads = 8, max_ctx > 2^24
 *   (positions are exact in fp32), or any kvq_config.flags / outliers option.
 */
int kvq_decode_attention_rope(const kvq_config *cfg, const kvq_cache *cache, const uint16_t *q,
                              float *out, float softmax_scale, double rope_base, void *ws,
                              size_t ws_bytes, void *stream);

/*
 * One decode step on device buffers: kvq_append(k, v) then
 * kvq_decode_attention(q) with the same arguments, results and errors.  When
 * the append only stores the new token (KIVI without a flush) and the decode
 * runs on the tensor-core path (head_dim 128, MHA), both happen in ONE kernel
 * launch: the decode reads the new token's rows from k, v directly and stores
 * them into the residual; otherwise it is the two launches.
 */
int kvq_append_decode(const kvq_config *cfg, kvq_cache *cache, const uint16_t *k,
                      const uint16_t *v, const uint16_t *q, float *out, float softmax_scale,
                      void *ws, size_t ws_bytes, void *stream);

/*
 * One decode step from HOST buffers, with one copy in and one copy out.
 *   h_in:  host fp16, the step's inputs back to back: k [B][H][d], then
 *          v [B][H][d], then q [B][n_q_heads][d] (2*B*H*d + B*n_q_heads*d
 *          halves).
 *   d_in:  device staging buffer of the same layout and size (16-byte aligned).
 *   h_out: host fp32 [B][n_q_heads][d]; d_out: its device staging buffer.
 * Enqueued on `stream`, no synchronization: one host-to-device copy of h_in,
 * kvq_append_decode on the staged rows, one device-to-host copy of the output.
 * Host buffers should be pinned for the copies to be asynchronous.  Errors:
 * as kvq_append_decode; KVQ_ECUDA when a copy fails to enqueue.
 */
int kvq_decode_step_host(const kvq_config *cfg, kvq_cache *cache, const uint16_t *h_in,
                         float *h_out, uint16_t *d_in, float *d_out, float softmax_scale,
                         void *ws, size_t ws_bytes, void *stream);

/*
 * Decode attention that allocates nothing, not even its scratch.  The pages
 * have no counterpart: this is a deployment convenience of the library.
 *
 * For callers that cannot hand the library a device buffer for scratch: code
 * that runs where no device allocator may be called (a plugin or callback
 * handed only its input and output tensors, a real-time or certified path
 * that forbids run-time device allocation, a process whose device memory is
 * entirely owned by another pool).  Same arguments, result and errors as
 * kvq_decode_attention minus ws / ws_bytes.
 *
 * The scratch is one file-scope device array of KVQ_NOALLOC_SCRATCH_BYTES
 * (16 MiB) that every GPU which loads the library holds until the process
 * exits.  Configurations whose kvq_workspace_bytes exceeds it are rejected
 * with KVQ_ECAPACITY; every other check of kvq_decode_attention runs too, and
 * a rejected call enqueues nothing and leaves the array alone.  The first call
 * on a device (with that device current) looks up the array's device address
 * with cudaGetSymbolAddress and keeps it; make that first call before any
 * stream capture.  Only the device's primary context (the CUDA runtime's) is
 * supported: the kept address is not valid in another context, nor after
 * cudaDeviceReset.  Each call clears the part of the scratch its
 * configuration uses (an asynchronous memset of kvq_workspace_bytes on
 * `stream`), then launches the decode, so a call that stopped early (a
 * timeout) leaves nothing behind for the next one.  All calls share the one
 * array: calls whose work can overlap on the GPU (different streams,
 * different caches) race and give wrong results; serialize them.
 */
#define KVQ_NOALLOC_SCRATCH_BYTES (16u << 20)
int kvq_decode_attention_noalloc(const kvq_config *cfg, const kvq_cache *cache,
                                 const uint16_t *q, float *out, float softmax_scale,
                                 void *stream);

/* Synchronizes `stream`, reads and clears the cache's device status word.
 * Returns KVQ_OK, or the error a kernel recorded (KVQ_ETIMEOUT), or KVQ_ECUDA. */
int kvq_get_device_status(kvq_cache *cache, void *stream);

/* Debug switch for the failure path of the decode kernel's bounded waits.
 * Every wait of the shared-memory pipeline gives up after a fixed poll cap
 * (2^24 polls, about a second or more), records KVQ_ETIMEOUT in the status
 * word, waits (bounded) for the block's own copies in flight and returns.
 * With iterations > 0, each block of later tensor-core decode launches first
 * waits, with that cap, on a barrier that nothing completes, so the timeout
 * path runs for certain; 0 switches it off.  After a timeout the output and
 * the workspace are undefined: zero-fill the workspace again.
 * Process-wide; not for production use. */
void kvq_debug_stall_waits(int64_t iterations);

/* Name of the decode kernel, with its template arguments, that
 * kvq_decode_attention launches for this configuration when n_quant tokens
 * are quantized (e.g. "tc_decode_kernel<bits=2,scheme=kivi,ngv=4,ngk=1,km=1>"),
 * written NUL-terminated into buf[len].  Host only, no CUDA call.  Returns
 * KVQ_OK, KVQ_EINVAL (null, n_quant < 0, buf too small) or a config error. */
int kvq_decode_kernel_name(const kvq_config *cfg, int64_t n_quant, char *buf, size_t len);

/* The same for kvq_decode_attention_rope (e.g.
 * "tc_decode_kernel<bits=2,scheme=kivi,ngv=4,km=1,rope=1>": the tensor-core
 * form, taken for head_dim 128, one query head per KV head, KIVI with key
 * groups of 32 or more and no cache options; other shapes name
 * "rope_decode_kernel<...>").  Host only, no CUDA call; same returns. */
int kvq_rope_kernel_name(const kvq_config *cfg, int64_t n_quant, char *buf, size_t len);

/* Number of kernel launches the last successful call of this thread enqueued. */
int kvq_last_launch_count(void);

/* Static description of a return code. */
const char *kvq_strerror(int code);

#ifdef __cplusplus
}
#endif
#endif /* KVQ_H */
