/*
 * mla.h -- C ABI of libmla: the forward pass of one Kimi-K2 multi-head latent attention
 * (MLA) layer on one NVIDIA GB300 (sm_103a), in prefill over an empty cache and in decode
 * against a latent KV cache.
 *
 * What the layer computes (Kimi K2 model-atlas pages):
 *   q      = q_b_proj(RMSNorm_q(q_a_proj(x)))                 per head [nope 128 | rope 64]
 *   c, k_r = split(kv_a_proj_with_mqa(x), [512, 64]);  c_hat = RMSNorm_kv(c)
 *   k_h    = [W_UK,h c_hat | RoPE(k_r)],  v_h = W_UV,h c_hat   (kv_b_proj rows per head)
 *   o_h    = softmax_fp32(q_h . k_h / sqrt(192) + causal mask) . v_h
 *   y      = o_proj(concat_h o_h)
 * ("Key-value latent" page: mla-init, mla-kv and rmsnorm excerpts; "Key content
 *  up-projection" page: the k^C = c^KV W_UK equation and the mla-prefill excerpt;
 *  "Latent attention (dense block, prefill)" page: the in/out signature and mla-output.)
 *
 * Conventions for every call:
 *   - Device pointers are CUDA global-memory addresses on the current device; host pointers
 *     are ordinary process memory.  The caller allocates and owns every buffer it passes and
 *     must keep weights, gains and caches alive for as long as the context uses them.
 *   - bf16 means IEEE bfloat16; e4m3 means OCP FP8 E4M3 ("fn": no infinities).
 *   - All layouts are row-major and densely packed unless a stride argument says otherwise.
 *   - `stream` is a cudaStream_t passed as void*; NULL is the legacy default stream.  Work is
 *     enqueued asynchronously; the call returns once the work is enqueued.
 *   - Every call checks its arguments on the host before enqueuing anything.  On any error
 *     nothing is enqueued and no caller buffer is written.  Calls never throw.
 *   - The context is not thread-safe; one host thread drives one context at a time.
 */
#ifndef MLA_H
#define MLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad enum, negative size            */
  MLA_ERR_SHAPE = 2,       /* a size disagrees with the layer (the pages raise ValueError) */
  MLA_ERR_UNSUPPORTED = 3, /* dimensions other than Kimi-K2's, or a mode not provided      */
  MLA_ERR_CAPACITY = 4,    /* cache length + new tokens exceeds the cache or RoPE table    */
  MLA_ERR_CUDA = 5,        /* a CUDA runtime call failed                                    */
  MLA_ERR_TIMEOUT = 6,     /* a device-side bounded wait gave up (read via device status)   */
  MLA_ERR_STATE = 7        /* weights or gains missing, or a device-side check failed       */
} mla_status;

typedef struct mla_ctx mla_ctx; /* opaque, host-side */

/* Projection ids for mla_upload_weights (names of the pages' nn.Linear modules). */
enum { MLA_W_Q_A = 0, MLA_W_Q_B = 1, MLA_W_KV_A = 2, MLA_W_KV_B = 3, MLA_W_O = 4 };
/* RMSNorm gain ids for mla_upload_norm: q_a_layernorm, kv_a_layernorm, and (with
 * mla_config.block = 1) the decoder block's input_layernorm. */
enum { MLA_NORM_Q = 0, MLA_NORM_KV = 1, MLA_NORM_INPUT = 2 };
/* RoPE pairing of the 64-wide rotary slice: pair j = (2j, 2j+1) or (j, j+32). */
enum { MLA_ROPE_ADJACENT = 0, MLA_ROPE_HALF = 1 };
/* RoPE frequencies: plain theta^(-2j/64), or YaRN (config.json rope_scaling, "KV cache" page). */
enum { MLA_ROPE_PLAIN = 0, MLA_ROPE_YARN = 1 };

typedef struct {
  int hidden, q_lora, kv_lora, heads, nope, rope, vdim; /* must be 7168,1536,512,64,128,64,128 */
  float eps;           /* RMSNorm epsilon (rms_norm_eps, 1e-6)                          */
  float rope_theta;    /* RoPE base (rope_theta, 50000)                                 */
  float softmax_scale; /* score scale; 1/sqrt(nope+rope) by default                     */
  int max_positions;   /* RoPE table rows: positions 0 .. max_positions-1 are allowed   */
  int rope_pairing;    /* MLA_ROPE_ADJACENT (default) or MLA_ROPE_HALF                  */
  int rope_scaling;    /* MLA_ROPE_PLAIN (default) or MLA_ROPE_YARN                     */
  float yarn_factor;              /* rope_scaling.factor (32)                           */
  int yarn_original_max_positions; /* rope_scaling.original_max_position_embeddings (4096) */
  float yarn_beta_fast, yarn_beta_slow;     /* rope_scaling.beta_fast / beta_slow (1, 1) */
  float yarn_mscale, yarn_mscale_all_dim;   /* rope_scaling.mscale / mscale_all_dim (1, 1) */
  int block;           /* 0: the layer alone (default); 1: the attention half of a decoder
                          block around it (see below)                                   */
  int fp8_activations; /* 0 (default) or 1: FP8 activations in the large projections      */
} mla_config;

/* Fills *cfg with Kimi-K2's dimensions (config.json on the "KV cache" page), eps 1e-6,
 * theta 50000, scale 1/sqrt(192), max_positions 131073 (max_position_embeddings 131072 is
 * not enforced by the pages' code, so position 131072 itself is allowed), adjacent pairs,
 * plain RoPE, and Kimi-K2's YaRN parameters ready for rope_scaling = MLA_ROPE_YARN.
 *
 * YaRN (published method, Peng et al. 2023; the pages give only the parameters): pair j
 * keeps its frequency while its wavelength turns more than beta_fast times over
 * original_max_positions, runs factor times slower below beta_slow turns, with a linear ramp
 * in j between the two boundary pairs; cos/sin are scaled by m(factor, mscale) /
 * m(factor, mscale_all_dim) and the score scale by m(factor, mscale_all_dim)^2, where
 * m(s, mu) = 0.1 mu ln s + 1 for s > 1, else 1. */
void mla_default_config(mla_config* cfg);

/* FP8 activations (fp8_activations = 1; the "linear" excerpt's quantization_config:
 * activation_scheme dynamic).  Projections of more than 64 token rows in mla_prefill,
 * mla_cache_append and their paged forms quantise their input to one e4m3 term per value
 * with one scale per (token, 128-wide group), s = amax / 448, and run one FP8 tensor-core
 * product per 128-wide k block instead of the two of the default, which multiplies the
 * bf16 input as an exact-to-2^-8 pair of e4m3 terms.  This is lossy: e4m3 keeps 3 mantissa
 * bits, and the layer output then misses the default bar of relative Frobenius error 1e-2
 * against the exact layer (measured values are in the design notes).  Decode and
 * projections of at most 64 rows are unchanged. */

/* The attention half of a decoder block (block = 1).  The "Attention input" page's `block`
 * excerpt keeps the block's input as the residual, normalises it with input_layernorm (the
 * `rmsnorm` excerpt over the hidden size, gain uploaded as MLA_NORM_INPUT, 7168 bf16 values),
 * runs the attention layer on the normalised input and adds the layer's output back to the
 * residual.  With block = 1 every token call (mla_cache_append, mla_prefill, mla_decode and
 * their paged forms) takes the block's input x: the cache rows are those of the normalised
 * input, and the output is out = bf16(x + bf16(layer(bf16(RMSNorm_in(x))))), the rounding of
 * the module's bf16 arithmetic.  The post-attention norm and the FFN that complete the block
 * are not part of this library.  mla_decode_noalloc does not take block = 1
 * (MLA_ERR_UNSUPPORTED). */

/* Creates a context on the current CUDA device.  Checks the dimensions (anything but
 * Kimi-K2's gives MLA_ERR_UNSUPPORTED), builds the RoPE cos/sin table on the host in double
 * precision (angle = pos * theta^(-2j/64), j = 0..31) and uploads it as float32.  That table,
 * a 4-byte device error word and the transposed W_UK copy described at mla_upload_weights are
 * the only device memory the context allocates; mla_destroy frees them.  *out is set only on
 * success. */
mla_status mla_create(const mla_config* cfg, mla_ctx** out);
void mla_destroy(mla_ctx* ctx); /* NULL is ignored; synchronises the device before freeing */

/* Registers one projection's FP8 weight ("linear" excerpt of the "Key-value latent" page:
 * fmt e4m3, weight_block_size [128, 128]).  e4m3_dev: device, [rows, cols] = [out, in],
 * 16-byte aligned; scale_dev: device float32 [ceil(rows/128), ceil(cols/128)], one scale per
 * 128x128 block, W[o,i] = e4m3(q[o,i]) * s[o/128][i/128].  rows/cols must equal the layer's
 * shape for `which` (q_a 1536x7168, q_b 12288x1536, kv_a 576x7168, kv_b 16384x512,
 * o 7168x8192), else MLA_ERR_SHAPE.  Only the pointers are recorded: the weights are not
 * copied and must stay valid while registered.  Registering kv_b also allocates (once per
 * context) a 4.2 MB device buffer for its W_UK rows transposed, filled by the next decode of 9
 * or more sequences, whose absorptions read it: after changing kv_b's contents in place,
 * register it again. */
mla_status mla_upload_weights(mla_ctx* ctx, int which, const void* e4m3_dev,
                              const float* scale_dev, int rows, int cols);

/* Registers an RMSNorm gain ("rmsnorm" excerpt): bf16 device vector of n = 1536 (MLA_NORM_Q),
 * 512 (MLA_NORM_KV) or 7168 (MLA_NORM_INPUT, needed when block = 1) values, 16-byte aligned.
 * Only the pointer is recorded. */
mla_status mla_upload_norm(mla_ctx* ctx, int which, const void* bf16_gain_dev, int n);

/* Bytes of caller-provided device workspace that mla_prefill / mla_decode /
 * mla_cache_append need for B sequences of T new tokens each over an empty cache.  The same
 * workspace may be reused by consecutive calls on one stream; calls that overlap on the GPU
 * need their own. */
size_t mla_workspace_bytes(const mla_ctx* ctx, int B, int T);

/* The same for a prefill over a non-empty cache: max_len >= seq_lens_host[b] + T for every b
 * (the largest total length a sequence reaches in the call).  Returns 0 for max_len < T or a
 * null ctx.  mla_workspace_bytes(ctx, B, T) == mla_workspace_bytes_len(ctx, B, T, T). */
size_t mla_workspace_bytes_len(const mla_ctx* ctx, int B, int T, int max_len);

/* Appends T tokens per sequence to the latent cache without computing attention: for each
 * token, the normalised latent (512) and the rotated shared rotary key (64) ("mla-kv"
 * excerpt, RoPE as for keys) are stored as one bf16 row of 576 values at position
 * seq_lens[b] + t, then seq_lens[b] += T on the device.
 *   x_bf16       device [B, T, 7168] hidden states
 *   cache_bf16   device [B, cap, 576]; row r of sequence b is at (b*cap + r)*576
 *   seq_lens_dev device int32 [B], current lengths, advanced by T
 *   seq_lens_host host int32 [B], the same lengths, used only to check capacity
 *   ws/ws_bytes  device workspace of at least mla_workspace_bytes(ctx, B, T) bytes
 * Errors: MLA_ERR_CAPACITY if seq_lens_host[b] + T > cap or > max_positions. */
mla_status mla_cache_append(mla_ctx* ctx, const void* x_bf16, int B, int T, void* cache_bf16,
                            int cap, int* seq_lens_dev, const int* seq_lens_host, void* ws,
                            size_t ws_bytes, void* stream);

/* Prefill of T new tokens per sequence ("Latent attention (dense block, prefill)" page: in
 * [B, T, 7168], out [B, T, 7168]).  Sequence b holds L_b = seq_lens[b] cached positions before
 * the call (0: prefill over an empty cache; more: a chunk of a longer prompt, "KV cache" page:
 * kv_seq_len = T + cached length).  Token t sits at position L_b + t and attends to positions
 * 0..L_b+t (the causal mask with the cache offset), all 64 heads, scores scaled by
 * softmax_scale, softmax in float32; the keys and values of the cached positions are rebuilt
 * from their latent rows (kv_b_proj), as for the new ones.  Writes out_bf16 [B, T, 7168],
 * appends cache rows L_b..L_b+T-1 and advances seq_lens_dev[b] by T.  seq_lens_host (host,
 * [B]) must equal the device lengths (a mismatch is flagged in the device status, not a
 * fault); with any L_b > 0 the workspace must hold mla_workspace_bytes_len(ctx, B, T,
 * max_b(L_b + T)) bytes.  out must not alias x. */
mla_status mla_prefill(mla_ctx* ctx, const void* x_bf16, int B, int T, void* cache_bf16,
                       int cap, int* seq_lens_dev, const int* seq_lens_host, void* out_bf16,
                       void* ws, size_t ws_bytes, void* stream);

/* One decode step for B sequences ("KV cache" page at p = seq_lens[b]): the new token of
 * sequence b, x_bf16[b] (device [B, 7168]), is placed at position seq_lens[b], its cache
 * row is appended, and it attends to all seq_lens[b] + 1 positions of its own cache.  The
 * attention runs in the absorbed form over the latent cache (W_UK folded into the query,
 * W_UV applied to the latent output), which equals the pages' explicit form in exact
 * arithmetic.  Writes out_bf16 [B, 7168] and advances seq_lens_dev by 1.  seq_lens_host
 * (host, [B]) must equal the device lengths; it sizes the split-KV schedule and is checked
 * against cap and max_positions (MLA_ERR_CAPACITY). */
mla_status mla_decode(mla_ctx* ctx, const void* x_bf16, int B, void* cache_bf16, int cap,
                      int* seq_lens_dev, const int* seq_lens_host, void* out_bf16, void* ws,
                      size_t ws_bytes, void* stream);

/* mla_decode with the hidden states and the output in host memory: one call enqueues the copy
 * of x_host [B, 7168] bf16 to the device, the decode step of mla_decode, and the copy of the
 * step's output to out_host [B, 7168] bf16, all on `stream`; it returns before they finish
 * (synchronise the stream before reading out_host or reusing x_host).  When a buffer is
 * page-locked host memory that the device addresses directly (cudaHostAlloc /
 * cudaMallocHost under unified addressing), its copy is a kernel of the decode chain; any other
 * host or device buffer is copied by cudaMemcpyAsync.  The input and output are staged in the
 * workspace, which must hold mla_decode_host_workspace_bytes(ctx, B) bytes.  The other
 * arguments, the step and the errors are those of mla_decode; x_host and out_host must differ
 * (MLA_ERR_INVALID_ARG otherwise). */
size_t mla_decode_host_workspace_bytes(const mla_ctx* ctx, int B);
mla_status mla_decode_host(mla_ctx* ctx, const void* x_host, int B, void* cache_bf16, int cap,
                           int* seq_lens_dev, const int* seq_lens_host, void* out_host, void* ws,
                           size_t ws_bytes, void* stream);

/* A paged latent cache.  The "KV cache" page describes a cache with no fixed size that grows
 * call by call (the cache's get_usable_length / update in the excerpt); here it is a pool of
 * fixed-size pages and a block table per sequence, so sequences can grow without reserving
 * their maximum length up front.  Position pos of sequence b is row
 * block_table[b * max_pages + pos / page_size] * page_size + pos % page_size of the pool, a
 * row holding the same 576 bf16 values as a dense cache row [c_hat (512) | RoPE(k_pe) (64)].
 * The caller allocates and owns the pool and the table and assigns the pages (any pool page,
 * in any order); the library only reads the table.  A table entry outside [0, num_pages)
 * for a position a call writes or reads is never followed: the row is skipped (writes) or
 * read as zeros (reads), and the device status reports MLA_ERR_STATE. */
typedef struct {
  void* pool;              /* device bf16 [num_pages, page_size, 576], 16-byte aligned        */
  int num_pages;           /* pages in the pool (num_pages * page_size < 2^31 - 256)          */
  int page_size;           /* positions per page: a positive multiple of 64                   */
  const int* block_table;  /* device int32 [B, max_pages]: pool page of logical page i of b   */
  int max_pages;           /* logical pages per sequence; capacity = max_pages * page_size    */
} mla_paged_cache;

/* mla_cache_append, mla_prefill and mla_decode over a paged latent cache: the same steps,
 * arguments and errors, with `cache` (host pointer to the descriptor, read during the call)
 * in place of the dense cache and its capacity; capacity errors (MLA_ERR_CAPACITY) are
 * judged against max_pages * page_size.  A malformed descriptor (null pointers, a page size
 * that is not a positive multiple of 64, an oversized pool) gives MLA_ERR_INVALID_ARG.  The
 * workspace sizes are those of the dense calls (mla_workspace_bytes_len covers the gathered
 * latents a chunk over a paged cache needs). */
mla_status mla_cache_append_paged(mla_ctx* ctx, const void* x_bf16, int B, int T,
                                  const mla_paged_cache* cache, int* seq_lens_dev,
                                  const int* seq_lens_host, void* ws, size_t ws_bytes,
                                  void* stream);
mla_status mla_prefill_paged(mla_ctx* ctx, const void* x_bf16, int B, int T,
                             const mla_paged_cache* cache, int* seq_lens_dev,
                             const int* seq_lens_host, void* out_bf16, void* ws, size_t ws_bytes,
                             void* stream);
mla_status mla_decode_paged(mla_ctx* ctx, const void* x_bf16, int B, const mla_paged_cache* cache,
                            int* seq_lens_dev, const int* seq_lens_host, void* out_bf16, void* ws,
                            size_t ws_bytes, void* stream);

/* mla_decode for callers that cannot allocate device memory when they decode (an arena that
 * owns all GPU memory, a runtime that forbids allocation after start-up): the same step and
 * the same arguments as mla_decode without the workspace.  The paper has no counterpart; this
 * is a deployment convenience.  Its scratch is one static 12 MiB device array inside the
 * library, held by every GPU that loads it until the process exits.
 *   - B must be at most 8 (else MLA_ERR_CAPACITY), on any GPU of up to 1024 SMs; the split-KV
 *     attention uses at most 48 work items, so long contexts run with fewer, longer splits
 *     than mla_decode's.
 *   - Every call shares the array: calls that overlap on the GPU race and must be serialised
 *     by the caller (one stream, one host thread).  The array keeps the last call's
 *     contents; nothing in it needs clearing, since every byte read is written first.
 *   - mla_create looks up the array's address on the context's device (then current) and
 *     keeps it in the context; calling with another device current gives
 *     MLA_ERR_INVALID_ARG.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library routine. */
mla_status mla_decode_noalloc(mla_ctx* ctx, const void* x_bf16, int B, void* cache_bf16, int cap,
                              int* seq_lens_dev, const int* seq_lens_host, void* out_bf16,
                              void* stream);

/* Verification helper: writes the float32 dequantisation of a registered weight,
 * out[o][i] = float(e4m3(q[o][i])) * s[o/128][i/128] (one rounded multiply), to the
 * caller's device buffer of rows*cols floats. */
mla_status mla_dequant_weight(mla_ctx* ctx, int which, float* out_dev, void* stream);

/* Synchronises `stream` and reads the context's device error word, which device-side checks
 * set instead of trapping (a bounded wait that gave up, a cache row out of range).  Returns
 * MLA_OK, MLA_ERR_TIMEOUT or MLA_ERR_STATE and clears the word. */
mla_status mla_get_device_status(mla_ctx* ctx, void* stream);

/* Observability.  With profiling on, every kernel a later token call launches is bracketed
 * by CUDA events recorded on the call's stream (also inside a CUDA-graph capture, where they
 * become event nodes).  Creates the context's event pool on first use. */
mla_status mla_set_profiling(mla_ctx* ctx, int on);

/* Kernels launched by the most recent mla_cache_append / mla_prefill / mla_decode call:
 * returns their count (or -1 for a NULL ctx) and fills up to `max` entries of names (static
 * strings, may be NULL) and ms (device milliseconds of each launch when that call ran with
 * profiling on, else -1; waits for the launch to finish; may be NULL). */
int mla_last_launches(mla_ctx* ctx, int max, const char** names, float* ms);

/* Self-test of the device-side bounded waits.  Every wait inside this library's kernels (on
 * an mbarrier completed by a TMA copy, an MMA or another warp) gives up after a limit (2 s),
 * records a timeout in the context's device error word and lets the kernel unwind, so a lost
 * completion never hangs the GPU.  This call enqueues one small kernel that waits, with the
 * same code and the given limit (at most 2e9 ns), on an mbarrier that nothing arrives at: the
 * wait runs out and a following mla_get_device_status returns MLA_ERR_TIMEOUT (and clears the
 * word), after which the context works as before.  MLA_ERR_INVALID_ARG for a NULL ctx or a
 * larger limit.
 *
 * Host-side failure injection (testing aid): a context created while the environment
 * variable MLA_TEST_FAIL_AFTER holds a number n >= 0 fails every later mla_cache_append,
 * mla_prefill and mla_decode call at the call's launch number n (0-based) with MLA_ERR_CUDA,
 * exactly as a failed CUDA launch returns: launches 0..n-1 are enqueued and run, launch n and
 * the rest are not.  Every token call advances seq_lens only in its last launch, so a call
 * that failed this way never advances them; it may have written the cache row at position
 * seq_lens[b], which lies past the sequence and is written again by the next call. */
mla_status mla_selftest_wait_timeout(mla_ctx* ctx, unsigned long long limit_ns, void* stream);

/* Static, human-readable name of a status code. */
const char* mla_status_string(mla_status s);

#ifdef __cplusplus
}
#endif

#endif /* MLA_H */
