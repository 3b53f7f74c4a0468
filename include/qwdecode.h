/*
 * qwdecode — forward pass of a Qwen3-0.6B-shaped decoder (prefill and KV-cached
 * decode) with its sampler, as hand-written CUDA for GB300 (sm_103a).
 *
 * The operations are those of "Inside an LLM: Pure Python Inference for
 * Qwen3-0.6B on MLX":
 *   Step 2  embedding lookup              x = E[ids]
 *   Step 3  RMSNorm                       x / sqrt(mean(x^2) + eps) * w
 *   Step 4  RoPE (half-split pairs)       angle = pos * theta^(-i/64)
 *   Step 5  attention with grouped query heads, QK-Norm, the KV cache and the
 *           causal mask
 *   Step 6  SwiGLU feed-forward           (silu(x Wg^T) * x Wu^T) Wd^T
 *   Step 7  pre-norm block with residuals
 *   Step 8  final norm, LM head (tied to E here) and sample()
 *   Step 9  the generation loop: one prefill, then one decode step per token
 *
 * Conventions for every call
 *   - Array arguments marked DEVICE are device pointers owned by the caller;
 *     HOST marks host pointers.  Work is enqueued on `stream` (a cudaStream_t
 *     passed as void*, NULL = legacy default stream); calls return once the work
 *     is enqueued, except where noted.
 *   - bf16 values cross the boundary as uint16_t bit patterns.
 *   - Return value: QW_OK (0) or a negative QW_E* code; the reason is available
 *     from qw_last_error_message() on the calling thread.  Nothing throws and no
 *     kernel traps: bad device-side inputs (token id out of range, position past
 *     the block table, page id outside the pool) are skipped by the kernels and
 *     recorded in a device error word that qw_check() reports.
 *   - A context is not thread-safe: serialise calls on one qw_ctx.
 */
#ifndef QWDECODE_H
#define QWDECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define QW_OK 0
#define QW_EINVAL (-1)    /* bad argument (null pointer, size out of range, unsupported shape) */
#define QW_ERANGE (-2)    /* token id, position or page id out of range (reported by qw_check) */
#define QW_ENOMEM (-3)    /* device allocation failed */
#define QW_EKVFULL (-4)   /* a KV pool request larger than the device can hold */
#define QW_ECUDA (-5)     /* a CUDA runtime or driver call failed */
#define QW_ETIMEOUT (-6)  /* a bounded device-side wait gave up (reported by qw_check) */

#define QW_PAGE_SIZE 16   /* tokens per KV page */
#define QW_HEAD_DIM 128   /* the only head size the kernels implement */
#define QW_NOALLOC_SCRATCH_FLOATS (1 << 20) /* fixed scratch of qw_attn_decode_noalloc: 4 MiB */
#define QW_TRACE_SLOTS 24  /* timestamps per CTA and layer in qw_debug_trace */

/* Kernel classes of qw_debug_profile. */
#define QW_PROF_GEMM 0     /* tensor-core projections (q|k|v, o_proj, gate/up, down) */
#define QW_PROF_ATTN 1     /* attention (prefill flash kernel, split-KV decode + merge) */
#define QW_PROF_OTHER 2    /* embedding, RMSNorm, QK-Norm/RoPE/cache write, RoPE table */
#define QW_PROF_LMHEAD 3   /* final norm + LM head */
#define QW_PROF_SAMPLE 4   /* sampler */
#define QW_PROF_FUSED 5    /* the fused batch-1 decode kernel */
#define QW_PROF_CLASSES 6

typedef struct qw_ctx qw_ctx;
typedef struct qw_kv qw_kv;

/* Model sizes and workspace limits.  qw_config_default() fills Qwen3-0.6B:
 * 28 layers, hidden 1024, 16 query / 8 KV heads of 128, SwiGLU 3072,
 * vocab 151936, eps 1e-6 (Step 3), RoPE base theta 1e6 (Step 4 gives one million
 * as the Qwen3 value). */
typedef struct qw_config {
    int32_t n_layers;
    int32_t hidden;        /* multiple of 256, at most 4096 */
    int32_t n_heads;       /* query heads; n_heads * head_dim is a multiple of 256 */
    int32_t n_kv_heads;    /* n_heads / G with G = 1 (MHA), 2, 4, 8 or 16 query heads per KV head (GQA; MQA
                            * when n_kv_heads = 1): Qwen3-0.6B and 1.7B have G = 2, 4B and 8B have G = 4 */
    int32_t head_dim;      /* must be QW_HEAD_DIM */
    int32_t intermediate;  /* multiple of 128 */
    int32_t vocab;         /* multiple of 32 */
    int32_t max_batch;     /* most rows in one qw_decode_step or qw_sample call (<= 256) */
    int32_t max_tokens;    /* most tokens in one qw_prefill call (sizes the workspaces) */
    int32_t debug_hidden;  /* nonzero: keep the residual after every layer for qw_debug_hidden */
    float rms_eps;
    double rope_theta;
    /* 16: bf16 weights as given.  8: weight-only int8, one scale per output channel (per row
     * of each projection and of the tied embedding): scale = the smallest power of two >=
     * max|w| / 127 (that quotient in IEEE fp32), code = w / scale rounded half to even, within
     * +-127.  The model then computes with the dequantised weights code * scale on every path
     * (exactly representable in bf16); the fused batch-1 decode streams the int8 codes (half
     * the bytes).  Not in the article, whose "What the script leaves out" section names
     * quantisation without defining one. */
    int32_t weight_bits;
} qw_config;

/* Weights as the checkpoint names them (Step 5-8 code): bf16 bit patterns,
 * row-major [out_features][in_features].  Per-layer members point to arrays of
 * n_layers pointers.  `on_device` = 1: every tensor pointer is a device pointer;
 * 0: host pointers.  qw_init copies everything; the caller may free its copies
 * afterwards.  The LM head is tied to embed_tokens (no lm_head tensor). */
typedef struct qw_weights {
    const uint16_t* embed_tokens;              /* model.embed_tokens.weight   [vocab][hidden] */
    const uint16_t* norm;                      /* model.norm.weight           [hidden] */
    const uint16_t* const* input_layernorm;    /* .input_layernorm.weight     [hidden] */
    const uint16_t* const* q_proj;             /* .self_attn.q_proj.weight    [n_heads*head_dim][hidden] */
    const uint16_t* const* k_proj;             /* .self_attn.k_proj.weight    [n_kv_heads*head_dim][hidden] */
    const uint16_t* const* v_proj;             /* .self_attn.v_proj.weight    [n_kv_heads*head_dim][hidden] */
    const uint16_t* const* q_norm;             /* .self_attn.q_norm.weight    [head_dim] */
    const uint16_t* const* k_norm;             /* .self_attn.k_norm.weight    [head_dim] */
    const uint16_t* const* o_proj;             /* .self_attn.o_proj.weight    [hidden][n_heads*head_dim] */
    const uint16_t* const* post_attention_layernorm; /* [hidden] */
    const uint16_t* const* gate_proj;          /* .mlp.gate_proj.weight       [intermediate][hidden] */
    const uint16_t* const* up_proj;            /* .mlp.up_proj.weight         [intermediate][hidden] */
    const uint16_t* const* down_proj;          /* .mlp.down_proj.weight       [hidden][intermediate] */
    int32_t on_device;
} qw_weights;

/* Per-row sampling parameters (Step 8 sample(), plus a top-k cap). */
typedef struct qw_sample_params {
    float temperature;  /* 0: greedy argmax (lowest id wins a tie); > 0: sample */
    int32_t top_k;      /* >= 0: at most this many candidates; 0 (or >= vocab): no cap (used when temperature > 0) */
    float top_p;        /* (0, 1]: keep the smallest prefix of the sorted distribution whose mass reaches top_p */
    uint32_t reserved;  /* set to 0 */
    uint64_t seed;      /* Philox4x32-10 key of this row (e.g. the sequence id) */
} qw_sample_params;

/* Fill `cfg` with the Qwen3-0.6B sizes, max_batch 64, max_tokens 16384. */
void qw_config_default(qw_config* cfg);

/* Validate `cfg`, upload and repack the weights, allocate workspaces.
 * On success *out owns all device memory it allocated; free with qw_destroy.
 * Synchronous.  Errors: QW_EINVAL (sizes), QW_ENOMEM, QW_ECUDA. */
int qw_init(const qw_config* cfg, const qw_weights* weights, qw_ctx** out);
int qw_destroy(qw_ctx* ctx);

/* Allocate a paged KV pool of `n_pages` pages for every layer.
 * Layout (bf16): [n_layers][n_pages][2 (K, V)][n_kv_heads][QW_PAGE_SIZE][head_dim];
 * one page holds QW_PAGE_SIZE consecutive positions of one sequence.  Keys are
 * stored after QK-Norm and RoPE (Step 5: the cache holds the rotated keys).
 * Errors: QW_EINVAL, QW_EKVFULL (more than the free device memory). */
int qw_kv_create(qw_ctx* ctx, int32_t n_pages, qw_kv** out);
int qw_kv_destroy(qw_kv* kv);
/* Base device address and byte strides of the pool (for injecting or reading caches). */
int qw_kv_layout(const qw_kv* kv, void** base, int64_t* layer_stride, int64_t* page_stride, int32_t* n_pages);

/* Prefill (Step 9): all prompt tokens of every sequence in one pass.
 *   ids, positions   DEVICE int32[n_tok], n_tok = cu_seqlens[n_seqs]: the tokens of
 *                    sequence s are rows cu_seqlens[s] .. cu_seqlens[s+1]-1, with
 *                    consecutive positions.  Every position below a sequence's first
 *                    position must already be in the cache (chunked prefill), so a
 *                    fresh sequence starts at position 0.
 *   cu_seqlens       HOST int32[n_seqs+1], cu_seqlens[0] = 0, nondecreasing, n_tok <= max_tokens.
 *   block_tables     DEVICE int32[n_seqs][bt_stride]: page ids; position p of sequence s
 *                    lives in page block_tables[s][p / QW_PAGE_SIZE], slot p % QW_PAGE_SIZE.
 *   last_logits      DEVICE float[n_seqs][vocab] or NULL: logits of each sequence's last token.
 * Writes K/V of every token into the pool.  Attention of a token at position p sees
 * the cached positions 0 .. p of its sequence (the causal mask of Step 5).
 * Sequences are independent, so one call may mix fresh prompts, prompt chunks appended
 * to cached prefixes and decode tokens (a sequence of one token at the position after its
 * cache): each gets the logits of its last token.
 * Errors: QW_EINVAL (null pointer, kv of another context, n_seqs or bt_stride < 1,
 * cu_seqlens[0] != 0, an empty sequence, n_tok > max_tokens, more than max_batch sequences
 * with last_logits NULL), QW_ECUDA (launch failure); bad ids, positions or page ids on the
 * device: QW_ERANGE from qw_check. */
int qw_prefill(qw_ctx* ctx, const int32_t* ids, const int32_t* positions, const int32_t* cu_seqlens,
               int32_t n_seqs, qw_kv* kv, const int32_t* block_tables, int32_t bt_stride,
               float* last_logits, void* stream);

/* One decode step for `batch` sequences, one token each (Step 9 loop body).
 *   tokens, positions  DEVICE int32[batch]; row b is at position positions[b] and sees
 *                      positions 0 .. positions[b] of its cache (its own K/V included).
 *   block_tables       DEVICE int32[batch][bt_stride].
 *   logits             DEVICE float[batch][vocab], or NULL to keep them in the context
 *                      (qw_sample with logits == NULL then reads them).
 * 1 <= batch <= max_batch.
 * Errors: QW_EINVAL (null pointer, kv of another context, batch outside [1, max_batch],
 * bt_stride < 1, or the fused path forced for a call it cannot take), QW_ECUDA (launch
 * failure); bad ids, positions or page ids on the device: QW_ERANGE from qw_check, a
 * bounded wait that gave up: QW_ETIMEOUT from qw_check. */
int qw_decode_step(qw_ctx* ctx, const int32_t* tokens, const int32_t* positions, int32_t batch,
                   qw_kv* kv, const int32_t* block_tables, int32_t bt_stride, float* logits,
                   void* stream);

/* Sample one id per row (Step 8 sample()).
 *   logits   DEVICE float[batch][vocab], or NULL for the context's logits from the last
 *            qw_decode_step / qw_prefill call that returned them in the context (those
 *            come with per-tile maxima from the LM head, so greedy rows read no logits).
 *   params   DEVICE qw_sample_params[batch].
 *   rng_counter  Philox counter of this step: row b draws u from Philox4x32-10 with
 *            key = params[b].seed and counter = (rng_counter, 0, 0) as four 32-bit
 *            words (low word first); u = (word0 >> 8) * 2^-24.
 *   out_ids  DEVICE int32[batch].
 * Greedy rows take the argmax (lowest id on ties).  Sampling rows take softmax(logits /
 * temperature) over the whole vocabulary, in the order probability descending, id
 * ascending; keep cutoff = 1 + #(cumsum < top_p) entries, capped at top_k when top_k > 0;
 * and return the first kept entry whose cumulative kept mass exceeds u * (kept mass).  Any
 * nucleus size is supported (top_k = 0 with top_p < 1 is the article's sample()).  The
 * cuts are found without sorting (radix searches over the logits by count and by mass), so
 * a draw whose cumulative sum lies within fp32 rounding of a cut may differ from an exact
 * sorted evaluation.  Invalid parameters (top_k < 0, top_p outside (0, 1]) record QW_EINVAL
 * for qw_check and are clamped.
 * Errors: QW_EINVAL (null params or out_ids, batch outside [1, max_batch], logits NULL while
 * the context holds fewer than batch rows), QW_ECUDA (launch failure). */
int qw_sample(qw_ctx* ctx, const float* logits, int32_t batch, const qw_sample_params* params,
              uint64_t rng_counter, int32_t* out_ids, void* stream);

/* Generate n_steps tokens of one sequence with the article's Step 9 loop run entirely on
 * the device: step i runs qw_decode_step on the token fed back by step i - 1 at position
 * start_pos + i, then qw_sample with rng_counter + i, and writes the id to out_ids[i]; the
 * host never waits on the device.  The same kernels as a host loop of qw_decode_step +
 * qw_sample, so the ids are identical.
 *   block_tables  DEVICE int32[1][bt_stride]: pages for positions up to start_pos + n_steps - 1.
 *   first_token   DEVICE int32[1]: the token at start_pos (e.g. sampled from the prefill).
 *   params        DEVICE qw_sample_params[1].
 *   out_ids       DEVICE int32[n_steps]: out_ids[i] is the token for position start_pos + i + 1.
 * Errors: QW_EINVAL for bad arguments (n_steps < 1, start_pos < 0, or positions beyond
 * bt_stride * QW_PAGE_SIZE); device-side range errors as for qw_decode_step. */
int qw_generate(qw_ctx* ctx, qw_kv* kv, const int32_t* block_tables, int32_t bt_stride,
                const int32_t* first_token, int32_t start_pos, int32_t n_steps,
                const qw_sample_params* params, uint64_t rng_counter, int32_t* out_ids, void* stream);

/* Decode attention of one layer over the paged cache (Step 5 for one new token per
 * sequence): out[b][h] = softmax(q[b][h] . K^T / sqrt(128)) V over the cached positions
 * 0 .. positions[b] of sequence b, with query head h reading KV head
 * h / (n_heads / n_kv_heads).
 *   q            DEVICE float[batch][n_heads][128], after QK-Norm and RoPE.
 *   positions    DEVICE int32[batch]; block_tables DEVICE int32[batch][bt_stride].
 *   layer        which layer's pages of `kv` to read.
 *   out          DEVICE bf16[batch][n_heads * 128].
 * The cache is split into chunks whose partial results (running max, sum, weighted
 * values) go to the context's workspace and are merged by a second kernel.
 * 1 <= batch <= max_batch. */
int qw_attn_decode(qw_ctx* ctx, const float* q, const int32_t* positions, int32_t batch, qw_kv* kv,
                   int32_t layer, const int32_t* block_tables, int32_t bt_stride, uint16_t* out, void* stream);

/* qw_attn_decode for callers that cannot allocate device memory.  The article has no
 * counterpart: this is a memory-management variant of the call above, not a step of
 * the method.
 *
 * Who needs it: code that must not call cudaMalloc/cudaFree on its path, such as a
 * latency-critical decode loop (cudaMalloc and cudaFree can synchronise the whole
 * device and stall other streams), a process whose device memory is entirely handed to
 * another allocator (a framework's caching allocator or a fixed-size pool, where an extra
 * allocation fails or fragments it), or a library that must own no device memory.  It
 * takes no context and allocates nothing: the caller passes the query, the pages of one
 * layer, the block tables and the output, and the split partials go to a fixed array
 * of QW_NOALLOC_SCRATCH_FLOATS floats (4 MiB) compiled into this library, which every
 * GPU that loads the library holds until the process exits.
 *   kv_layer   DEVICE bf16 pages of one layer, [n_pages][2][n_kv_heads][16][128]
 *              (qw_kv_layout's base plus layer * layer_stride for a qw_kv pool).
 *   q, positions, block_tables, bt_stride, out: as in qw_attn_decode; n_heads must be
 *              n_kv_heads times 1, 2, 4, 8 or 16.
 * Limits: batch * n_heads * 130 <= QW_NOALLOC_SCRATCH_FLOATS (batch * n_heads <= 8065),
 * else QW_EINVAL with nothing launched.  Page ids outside [0, n_pages) are skipped but,
 * with no context, not reported.
 * Every call looks up the array's address in the current device's current context (a
 * lookup, no allocation), so a cudaDeviceReset or a change of context in between is safe;
 * the first call on a device may also load the library's device code, so make that first
 * call before any stream capture.  All calls
 * share the one array and nothing in it needs to start at zero: calls whose GPU work can
 * overlap (different streams, several host threads) race on it, so serialise them. */
int qw_attn_decode_noalloc(const float* q, const int32_t* positions, int32_t batch, int32_t n_heads,
                           int32_t n_kv_heads, const uint16_t* kv_layer, int32_t n_pages,
                           const int32_t* block_tables, int32_t bt_stride, uint16_t* out, void* stream);

/* Wait for `stream`, then return and clear the first error the kernels recorded
 * since the last check (QW_OK if none). */
int qw_check(qw_ctx* ctx, void* stream);

/* Reason for the last non-zero return on this thread ("" if none). */
const char* qw_last_error_message(void);

/* Copy the residual stream after layer `layer` (0 .. n_layers-1) of the last
 * qw_prefill or qw_decode_step into DEVICE float[n_rows][hidden] (n_rows = tokens of
 * that call).  Needs debug_hidden; for checking, not for speed. */
int qw_debug_hidden(qw_ctx* ctx, int32_t layer, float* out, int32_t n_rows, void* stream);

/* Test hook for the tensor-core projection kernel alone: C = A . B^T with
 *   A DEVICE bf16[M][K], B DEVICE bf16[N][K] (the layout of every weight), K % 64 == 0,
 *   N % 32 == 0, bn = 128 or 256 (output tile width; 32 or 64 too with split = 1) and the epilogue
 *   epi = 0: C is float[M][N], C = A B^T;  1: C += A B^T (residual add);
 *   epi = 2: C is bf16[M][N/2], C[m][j] = silu(Y[m][2j]) * Y[m][2j+1] with Y = A B^T
 *   (the SwiGLU of Step 6 on gate/up rows interleaved);
 *   epi = 3: C += A B^T with K split across SMs and fp32 atomic adds (small-M path).
 * split = 1: A holds ceil(M/64) blocks of 128 rows, rows 0..63 of a block the bf16 "hi"
 *   parts of 64 activation rows and rows 64..127 their "lo" remainders; the product uses
 *   hi + lo (the layout decode batches use), and with epi = 2 the output is written in the
 *   same hi/lo layout.  split = 0: plain A[M][K].  split = 2: plain A, and with bn = 256,
 *   M > 128 and epi != 3 the product runs in clusters of two CTAs that share (multicast)
 *   each weight tile (the prefill configuration). */
int qw_debug_gemm(const uint16_t* A, const uint16_t* B, void* C, int32_t M, int32_t N, int32_t K, int32_t epi,
                  int32_t bn, int32_t split, void* stream);

/* Tracing hook of the fused batch-1 decode kernel.  enable = 1: the following fused
 * steps record %globaltimer stamps (ns) at every phase boundary; enable = 0: stop.
 * host_out (nullable, HOST uint64[n]): receives the stamps of the last traced step,
 * [CTA][layer 0..n_layers][QW_TRACE_SLOTS]: slot 0/1: before/after the wait for the layer
 * input; attention CTAs: 2 q|k|v rows done, 3 q|k|v exchange complete, 4 keys done,
 * 5 attention partials exchanged, 6 o_proj rows done, 7 o_proj reduced in the cluster,
 * 8 group slot published; every CTA: 9/10 before/after the wait for the attention output,
 * 11 gate/up rows and SwiGLU done, 12 down_proj rows done, 13 reduced in the cluster, 14 cluster
 * slot published, 17 feed-forward input normalised,
 * 18 (attention CTAs) queries and the new key/value ready; layer n_layers: LM head wait
 * begin/end (0/1) and rows done (2); unused slots hold 0.  *n_needed receives the buffer
 * length.  Synchronous. */
int qw_debug_trace(qw_ctx* ctx, int32_t enable, uint64_t* host_out, int64_t n, int64_t* n_needed);

/* Device time per kernel class, for measurement.  enable = 1: from now on record a CUDA
 * event pair on the launching stream around every launch (forgetting earlier records);
 * enable = 0: stop recording.  ms_out (nullable, HOST double[QW_PROF_CLASSES]) and
 * count_out (nullable, HOST int64[QW_PROF_CLASSES]) receive, after a device
 * synchronisation, the summed milliseconds and the number of launches of each class
 * (QW_PROF_*) recorded since the last enable.  Not for use inside stream capture. */
int qw_debug_profile(qw_ctx* ctx, int32_t enable, double* ms_out, int64_t* count_out);

/* Failure-detection test hook: the next fused batch-1 decode step waits at one grid-wide
 * exchange for one arrival more than will ever come, with a 2 ms limit instead of the usual
 * 2 s.  That step gives up everywhere without a device fault; qw_check then returns
 * QW_ETIMEOUT, clears the kernel's counters, and the context keeps working.  Errors:
 * QW_EINVAL without a fused kernel. */
int qw_debug_inject_timeout(qw_ctx* ctx);

/* Select the prefill attention kernel: 0 = tcgen05/TMEM flash kernel (default),
 * 1 = mma.sync flash kernel.  For comparisons in tests. */
int qw_set_prefill_attention(qw_ctx* ctx, int32_t variant);

/* Number of kernels this library has launched in the process so far (all contexts). */
uint64_t qw_kernel_launches(void);

/* Select the decode implementation: 0 = automatic, 1 = per-op kernels,
 * 2 = the fused persistent small-batch kernel (batch <= 8).  For tests. */
int qw_set_decode_path(qw_ctx* ctx, int32_t path);

#ifdef __cplusplus
}
#endif
#endif /* QWDECODE_H */
