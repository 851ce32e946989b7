/* tinfer.h -- C ABI of the GB300 batch-1 decode engine.
 *
 * One call runs one decode step of a Llama-family dense transformer for a single sequence:
 * embedding, every decoder layer (RMSNorm, fused QKV GEMV, NEOX RoPE plus K/V append, grouped-query
 * split-K attention with a log-sum-exp merge, O GEMV plus residual, RMSNorm, gate/up GEMV with
 * SwiGLU, down GEMV plus residual), final RMSNorm, LM head and greedy argmax. The problem statement
 * follows "Decoding in tiles" (TileInfer), sections 4-5 (create once, launch per token, greedy
 * choice on the device) and "One launch per token", section "Slow, because the launches are still
 * there" (token and position handed to a fixed-shape step).
 *
 * Conventions for every entry point:
 *   - Pointers named *_dev are device pointers (cudaMalloc or equivalent); *_host are host
 *     pointers. `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *   - Every call returns a tinfer_status and never aborts the process. Host-side validation
 *     failures return TINFER_ERR_INVALID_ARG / TINFER_ERR_UNSUPPORTED before anything is launched.
 *   - Work is asynchronous on `stream` unless stated otherwise. Device-side failures (a non-finite
 *     logit, a synchronisation wait that ran out) are recorded in the context's error word; the
 *     next tinfer_decode_step* call returns them without launching, and tinfer_get_error reports
 *     and clears them.
 *   - Matrices are row-major [rows = outputs][cols = inputs]. bf16 values are IEEE bfloat16 bit
 *     patterns. int4 matrices are [rows][cols/2] bytes, input element 2j in the low nibble of byte
 *     j and 2j+1 in the high nibble, value (q - 8) * scale, one fp16 or bf16 scale per `group_size`
 *     consecutive inputs of a row ([rows][cols/group] scales). This is the canonical layout; the
 *     engine streams its own packed layout, made by tinfer_pack_layer.
 *   - The KV cache is two caller-owned bf16 buffers, K and V, each [n_layers][n_kv_heads][max_ctx]
 *     [head_dim]. Position `pos` is 0-based; a step at `pos` writes slot `pos` of every layer and
 *     attends over slots [0, pos], so slots [0, pos) must hold earlier keys/values.
 */
#ifndef TINFER_H
#define TINFER_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TINFER_OK = 0,
  TINFER_ERR_INVALID_ARG = 1,   /* a pointer, size, token or position outside its contract */
  TINFER_ERR_UNSUPPORTED = 2,   /* a shape or format this build does not handle */
  TINFER_ERR_CUDA = 3,          /* a CUDA runtime call failed (launch, capture, copy) */
  TINFER_ERR_OOM = 4,           /* a device or pinned-host allocation failed */
  TINFER_ERR_NONFINITE = 5,     /* a logit was NaN or infinite (the argmax output is -1) */
  TINFER_ERR_TIMEOUT = 6        /* a device-side wait gave up (a phase's stamped results or a
                                   pipeline stage that never arrived) */
} tinfer_status;

enum { TINFER_BF16 = 0, TINFER_INT4 = 1 };              /* weight_format */
enum { TINFER_SCALE_FP16 = 0, TINFER_SCALE_BF16 = 1 };  /* scale_dtype (int4 only) */
enum { TINFER_MEGAKERNEL = 0, TINFER_GRAPH = 1 };       /* exec_mode */

typedef struct {
  int n_layers, hidden, n_heads, n_kv_heads, head_dim, ffn, vocab, max_ctx;
  double rope_theta;   /* RoPE base; angle of pair i at position p is p * theta^(-2i/head_dim) */
  double rms_eps;      /* RMSNorm epsilon inside the square root */
  int weight_format;   /* TINFER_BF16 or TINFER_INT4 (int4 covers q,k,v,o,gate,up,down) */
  int group_size;      /* int4: inputs per scale; a multiple of 32 dividing hidden, n_heads*head_dim, ffn */
  int scale_dtype;     /* int4: TINFER_SCALE_FP16 or TINFER_SCALE_BF16 */
  int tied_embeddings; /* informational: lm_head may equal embed */
  int qkv_bias;        /* 1: bf16 biases are added to q, k, v before RoPE */
  int exec_mode;       /* TINFER_MEGAKERNEL (one persistent launch per step) or TINFER_GRAPH */
  int ffn_split;       /* 1: the MLP's down projection split by columns ("Decoding in tiles", section
                          4, "FFN" and "FFN reduce"): each CTA multiplies its own SwiGLU rows by the
                          matching columns of Wd and the partial sums are reduced in a fixed order.
                          The packed layer then stores Wd transposed. bf16 weights and
                          TINFER_MEGAKERNEL only (else TINFER_ERR_UNSUPPORTED); 0: row-split down. */
} tinfer_config;

/* Canonical per-layer weights (device pointers), the input of tinfer_pack_layer.
 * w*: bf16 [rows][cols] or int4 bytes [rows][cols/2]; s*: int4 scales (NULL for bf16);
 * b*: bf16 biases of length rows (NULL unless qkv_bias); g1, g2: bf16 RMSNorm gains [hidden]. */
typedef struct {
  const void *wq, *wk, *wv, *wo, *wg, *wu, *wd;
  const void *sq, *sk, *sv, *so, *sg, *su, *sd;
  const void *bq, *bk, *bv;
  const void *g1, *g2;
} tinfer_layer_src;

/* Model weights for tinfer_create (device pointers, borrowed: they must outlive the context).
 * embed, lm_head: bf16 [vocab][hidden] (lm_head may equal embed); final_norm: bf16 [hidden];
 * layer_blobs: HOST array of n_layers device pointers, each a packed layer made by
 * tinfer_pack_layer (16-byte aligned, tinfer_packed_layer_bytes long). */
typedef struct {
  const void* embed;
  const void* lm_head;
  const void* final_norm;
  const void* const* layer_blobs;
} tinfer_weights;

typedef struct tinfer_ctx tinfer_ctx;

const char* tinfer_status_string(tinfer_status s);

/* Validates a configuration without allocating anything. */
tinfer_status tinfer_check_config(const tinfer_config* cfg);

/* Offline weight packer (the "concatenate QKV and gate/up at load" step of tinyinfer, "Round 3:
 * fusion", and "One launch per token", "The oracle, then the kernels"). The packed layer holds, in
 * order and 256-byte aligned: [Wq;Wk;Wv] rows, Wo rows, gate/up rows interleaved (row 2i = gate i,
 * row 2i+1 = up i), Wd rows, g1 and g2 as fp32, and the QKV bias as fp32. Every row is padded to a
 * multiple of 16 bytes; an int4 row stores its cols/2 nibble bytes followed by its cols/group scales.
 * tinfer_packed_layer_bytes returns 0 for an invalid config. pack writes packed_dev (caller-owned,
 * 16-byte aligned) on `stream`; unpack inverts it into the canonical buffers of dst (the bytes of
 * every weight, scale, bias and gain reproduced exactly; gains and biases round-trip through fp32
 * exactly). */
size_t tinfer_packed_layer_bytes(const tinfer_config* cfg);
tinfer_status tinfer_pack_layer(const tinfer_config* cfg, const tinfer_layer_src* src,
                                void* packed_dev, void* stream);
tinfer_status tinfer_unpack_layer(const tinfer_config* cfg, const void* packed_dev,
                                  const tinfer_layer_src* dst, void* stream);

/* Creates an engine over borrowed weights and a borrowed KV cache (k_cache_dev, v_cache_dev: bf16
 * [n_layers][n_kv_heads][max_ctx][head_dim]). Set-up happens once per model and GPU, and every
 * launch after it follows the same fixed schedule ("Decoding in tiles", section 4: the plan is made
 * and validated once, and the launch makes no scheduling decision). The context owns its scratch
 * (stamped hand-off buffers, split-K partials, ticket words, argmax slots, the fp32 RoPE cos/sin
 * table, the CUDA graph in graph mode) and frees it in tinfer_destroy. Uses the current CUDA device.
 * Weights, scales and the KV cache must be 16-byte aligned; a NULL or misaligned pointer returns
 * TINFER_ERR_INVALID_ARG, an unsupported shape TINFER_ERR_UNSUPPORTED, a failed allocation
 * TINFER_ERR_OOM, all before anything is launched. */
tinfer_status tinfer_create(const tinfer_config* cfg, const tinfer_weights* w, void* k_cache_dev,
                            void* v_cache_dev, tinfer_ctx** out);

/* One decode step for token_id at position pos on `stream` ("Decoding in tiles", section 5 "One
 * token, end to end": every layer, the final norm, lm_head and a greedy choice on the device, the
 * largest logit with the lowest token id among ties, an error word on a non-finite logit).
 * logits_dev (fp32 [vocab]) may be NULL to skip writing the logits; argmax_dev (int32 [1]) receives
 * the greedy token, or -1 when a logit is non-finite. Returns at once (asynchronous).
 * token_id outside [0, vocab) or pos outside [0, max_ctx) returns TINFER_ERR_INVALID_ARG without
 * launching; so does an error a previous step left in the error word (its own status). */
tinfer_status tinfer_decode_step(tinfer_ctx* ctx, int32_t token_id, int32_t pos, void* stream,
                                 float* logits_dev, int32_t* argmax_dev);

/* Same step, but the token id is read on the device from token_dev (int32 [1]) when the step runs,
 * so that greedy decoding can chain steps without a host round trip (token_dev may be the previous
 * step's argmax_dev). An out-of-range device token sets TINFER_ERR_INVALID_ARG in the error word. */
tinfer_status tinfer_decode_step_dev(tinfer_ctx* ctx, const int32_t* token_dev, int32_t pos,
                                     void* stream, float* logits_dev, int32_t* argmax_dev);

/* Greedy generation with the host in the loop: for k in [0, n_steps) the step at pos0 + k is fed
 * (from pinned host memory) token first_token for k = 0 and the previous step's choice after that;
 * each step's choice is copied back to the host and written to tokens_host[k]. Synchronous: returns
 * when all steps are done. */
tinfer_status tinfer_generate(tinfer_ctx* ctx, int32_t first_token, int32_t pos0, int32_t n_steps,
                              void* stream, int32_t* tokens_host);

/* Greedy generation in one launch ("Decoding in tiles", section 5, Figure 10: one cooperative
 * launch decodes consecutive tokens with greedy selection inside the kernel). Step k (k in
 * [0, n_steps)) runs at position pos0 + k with token first_token for k = 0 and step k - 1's choice
 * after that; tokens_dev (device int32 [n_steps]) receives every step's choice (-1 for a step with a
 * non-finite logit, which also sets TINFER_ERR_NONFINITE and ends the run). When eos_token >= 0 the
 * run ends after the step that chose it. count_dev (device int32 [1], may be NULL) receives the
 * number of steps completed. Asynchronous on `stream`; slots [pos0, pos0 + count) of the KV cache are
 * written. Host checks: n_steps >= 1, pos0 + n_steps <= max_ctx, first_token and eos_token in range
 * (eos_token may be -1), 4-byte aligned outputs; else TINFER_ERR_INVALID_ARG. In graph mode the
 * steps are separate graph launches chained on the device (eos_token must be -1 and count_dev NULL,
 * else TINFER_ERR_UNSUPPORTED). */
tinfer_status tinfer_generate_dev(tinfer_ctx* ctx, int32_t first_token, int32_t pos0, int32_t n_steps,
                                  int32_t eos_token, void* stream, int32_t* tokens_dev,
                                  int32_t* count_dev);

/* Waits for all work of the context, then returns and clears the device error word (TINFER_OK if
 * none): TINFER_ERR_NONFINITE for a non-finite logit, TINFER_ERR_TIMEOUT for a device wait that ran
 * out, TINFER_ERR_INVALID_ARG for an out-of-range device token ("Decoding in tiles", section 5:
 * worker 0 records the token, the count, the end flag and an error code for the host). Clearing
 * also resets the context's ticket words. Synchronises the device. */
tinfer_status tinfer_get_error(tinfer_ctx* ctx);

/* Introspection: TINFER_Q_GRID (CTAs of the persistent launch = SM count), TINFER_Q_SMEM (dynamic
 * shared memory per CTA of the persistent kernel), TINFER_Q_RING_STAGES, TINFER_Q_SLOT_BYTES,
 * TINFER_Q_KERNELS_PER_STEP (kernel launches one step makes), TINFER_Q_BLOCK_THREADS (threads per
 * CTA of the step kernels of the context's mode). Returns -1 for an unknown query. */
enum { TINFER_Q_GRID = 0, TINFER_Q_SMEM = 1, TINFER_Q_RING_STAGES = 2, TINFER_Q_SLOT_BYTES = 3,
       TINFER_Q_KERNELS_PER_STEP = 4, TINFER_Q_TRACE_BYTES = 5, TINFER_Q_BLOCK_THREADS = 6 };
long long tinfer_query(const tinfer_ctx* ctx, int what);

/* Per-worker timeline of the persistent kernel ("Decoding in tiles", section 5, Figure 9: each
 * worker's time split into streaming, waiting and small work). When trace_dev is not NULL (device
 * memory of TINFER_Q_TRACE_BYTES bytes, caller-owned), every following megakernel step writes, for
 * every CTA c and phase k (k = 5*layer + {0 QKV, 1 attention, 2 O, 3 gate/up, 4 down}, the LM head
 * last), ten uint64 %globaltimer nanosecond stamps at [(c * phases + k) * 10 + f] (0 where nothing
 * was recorded): f = 0 phase start (the CTA is done with the previous phase), 2 phase end, 3 producer starts
 * issuing the phase's copies, 4 producer has issued them; GEMV phases: 1 activations normalised and
 * ready, 5 input activations in registers, 6 GEMV code entered, 7 input vector in shared memory,
 * 8 first weight stage available, 9 last weight stage consumed;
 * attention phases (first unit of the CTA): 1 keys arrived, 5 queries rotated, 6 scores done,
 * 7 partials written, 8 values arrived, 9 the merge has seen every sibling's partials (first unit
 * of the CTA). NULL turns tracing off. */
tinfer_status tinfer_set_trace(tinfer_ctx* ctx, void* trace_dev);

/* Test hooks: timeout of every device-side wait in nanoseconds (default 200 ms), and a fault
 * injected on the host side of the contract: in the next persistent step, CTA `cta` withholds its
 * results of GEMV phase number `phase` (k = 5*layer + {0 QKV, 2 O, 3 gate/up, 4 down}; the LM head
 * 5*n_layers), so that the CTAs waiting for them run out of time and the step reports
 * TINFER_ERR_TIMEOUT (cta = -1 disables; a CTA without rows in that phase withholds nothing).
 * TINFER_ERR_UNSUPPORTED in graph mode. */
tinfer_status tinfer_set_timeout_ns(tinfer_ctx* ctx, long long ns);
tinfer_status tinfer_debug_withhold_results(tinfer_ctx* ctx, int cta, int phase);

/* The producer's schedule ("Decoding in tiles", section 1: Hazy Research's kernel overlaps the next
 * instruction's loads with the current one; section 4: TileInfer does not): how far the weight
 * stream runs ahead of the consumers. TINFER_S_INFLIGHT: bulk copies outstanding per CTA (default
 * 2; clamped to the ring's stages, 0 = the whole ring); TINFER_S_INFLIGHT_LM: the same during the LM
 * head (default 4); TINFER_S_L2_LOOKAHEAD: bytes per CTA prefetched into L2 ahead of the ring while
 * the ring is full (default 512 KiB for bf16 models, 0 for int4); TINFER_S_L2_PACE: nanoseconds per
 * KiB between those prefetches (default 24, about one SM's share of HBM bandwidth). Values outside
 * [0, 64 MiB] (lookahead), [0, 100000] (pace) or [0, 8] (copies) return TINFER_ERR_INVALID_ARG.
 * Takes effect from the next step; results do not depend on it. tinfer_get_schedule returns the
 * current value, or -1 for an unknown knob. */
enum { TINFER_S_INFLIGHT = 0, TINFER_S_INFLIGHT_LM = 1, TINFER_S_L2_LOOKAHEAD = 2, TINFER_S_L2_PACE = 3,
       TINFER_S_SYNC = 4, TINFER_S_ATTN_CHUNKS = 5 };
/* TINFER_S_ATTN_CHUNKS: chunks per KV head of the split-K attention ("One launch per token", "The
 * attention trap": split the context across the SMs, then combine). 0 (default): the automatic
 * split, enough chunks that the (KV head, chunk) units cover the grid; n > 0: n chunks of
 * ceil((pos + 1) / n) positions at every position (chunks past the context are empty and weigh 0).
 * n must be at least the number of chunks that keeps every chunk within one ring slot at max_ctx
 * and at most the automatic split's count at max_ctx (the partial buffers' capacity), else
 * TINFER_ERR_INVALID_ARG. Results change only by the order of the combine's additions. */
/* TINFER_S_SYNC: how a phase waits for the one before it. TINFER_SYNC_STAMPS (default): each CTA
 * waits only for the stamped results it reads. TINFER_SYNC_GRID_BARRIER: every CTA also passes a
 * grid barrier before every phase ("Decoding in tiles", section 4: every wave ends at a grid
 * barrier), for comparison. Persistent kernel only (TINFER_ERR_UNSUPPORTED in graph mode); switching
 * to it synchronises the device. */
enum { TINFER_SYNC_STAMPS = 0, TINFER_SYNC_GRID_BARRIER = 1 };
tinfer_status tinfer_set_schedule(tinfer_ctx* ctx, int knob, long long value);
long long tinfer_get_schedule(const tinfer_ctx* ctx, int knob);

void tinfer_destroy(tinfer_ctx* ctx);

/* ---------------------------------------------------------------------------------------------
 * Single-operation entry points. They run the same device code as the step, one operation at a
 * time, for the per-kernel parity tests. All pointers are device pointers owned by the caller.
 * --------------------------------------------------------------------------------------------- */

/* Bytes of one packed row of `cols` inputs (0 if the format cannot hold that width). */
size_t tinfer_packed_row_bytes(int weight_format, int cols, int group_size);

/* Packs a canonical matrix (bf16, or int4 bytes plus scales) into packed rows. */
tinfer_status tinfer_pack_matrix(int weight_format, int group_size, int scale_dtype, int rows,
                                 int cols, const void* w_dev, const void* scales_dev,
                                 void* packed_dev, void* stream);

enum { TINFER_EPI_STORE = 0, TINFER_EPI_RESIDUAL = 1, TINFER_EPI_SWIGLU = 2, TINFER_EPI_ARGMAX = 3 };

/* y = W a through the streaming GEMV (TMA bulk copies into a shared-memory ring, fp32 accumulate).
 * a = x, or a = rmsnorm(x) * gain when gain_dev (fp32 [cols]) is not NULL (eps = rms_eps).
 * Epilogue: STORE y[r] = v (+ bias_dev[r] if not NULL); RESIDUAL y[r] += v; SWIGLU: rows come in
 * (gate, up) pairs, y[i] = silu(v[2i]) * v[2i+1] (rows must be even); ARGMAX: y[r] = v (y may be
 * NULL) and argmax_dev[0] = the lowest row among the maxima, or -1 and TINFER_ERR_NONFINITE if any v
 * is non-finite. x_dev: fp32 [cols]. Synchronises `stream` for ARGMAX so that the status is exact. */
tinfer_status tinfer_op_gemv(int weight_format, int group_size, int scale_dtype, int rows, int cols,
                             const void* packed_dev, const float* x_dev, const float* gain_dev,
                             double rms_eps, const float* bias_dev, int epilogue, float* y_dev,
                             int32_t* argmax_dev, void* stream);

/* The same streaming GEMV over a batch of m activation vectors (m in {1, 2, 4, 8}), the verify
 * shape of speculative decoding (flint, "speculative decode": K + 1 positions verified in one launch,
 * the weights read once): y[j][r] = sum_c W[r][c] x[j][c] for j < m, fp32 accumulation, each int4
 * weight decoded once for all m vectors. x_dev: fp32 [m][cols], y_dev: fp32 [m][rows] (both
 * row-major), bias_dev: fp32 [rows] or NULL. epilogue: TINFER_EPI_STORE (y = W x + bias) or
 * TINFER_EPI_RESIDUAL (y += W x). A row is cut into at most 8 segments of at most 2048 / m inputs
 * (int4: whole runs of 8 / m words), so m * cols <= 16384; other shapes return
 * TINFER_ERR_UNSUPPORTED. Asynchronous on `stream`. */
tinfer_status tinfer_op_gemv_batch(int weight_format, int group_size, int scale_dtype, int rows, int cols,
                                   int m, const void* packed_dev, const float* x_dev,
                                   const float* bias_dev, int epilogue, float* y_dev, void* stream);

/* Attention for one layer at position pos: qkv_dev holds the raw projections [q (n_heads*head_dim) |
 * k (n_kv_heads*head_dim) | v (n_kv_heads*head_dim)] in fp32 (bias already added). The op applies
 * RoPE (fp32 cos/sin table built on the host in double from rope_theta) to q and k, writes
 * bf16(k_rot) and bf16(v) to slot pos of k_layer_dev / v_layer_dev ([n_kv_heads][max_ctx][head_dim]),
 * runs split-K attention over [0, pos] in n_chunks chunks of ceil((pos+1)/n_chunks) slots (n_chunks
 * = 0: the engine's own choice) and merges the partials into out_dev (fp32 [n_heads*head_dim]).
 * part_m_dev, part_l_dev ([n_heads][n_chunks]) and part_o_dev ([n_heads][n_chunks][head_dim]) may be
 * NULL; when given (with explicit n_chunks) they receive the unnormalised partials. */
tinfer_status tinfer_op_attention(int n_heads, int n_kv_heads, int head_dim, int max_ctx,
                                  double rope_theta, int pos, int n_chunks, const float* qkv_dev,
                                  void* k_layer_dev, void* v_layer_dev, float* out_dev,
                                  float* part_m_dev, float* part_l_dev, float* part_o_dev,
                                  void* stream);

/* Gathered-expert SwiGLU MLP of a mixture-of-experts layer ("One launch per token", section "The
 * same trick, sparser: a 64-expert MoE": the router writes the chosen expert ids into a device
 * tensor and two fixed-shape kernels read the weights through that index, one for the gated/up
 * SwiGLU of the chosen experts, one for the down projection and the weighted sum):
 *   y = sum_{i < top_k} weights[i] * Wd[ids[i]] (silu(Wg[ids[i]] x) * (Wu[ids[i]] x))   (accumulate 0)
 *   y += the same                                                                       (accumulate 1)
 * Canonical expert weights (device, stacked expert after expert): wg, wu [n_experts][ffn_e][hidden],
 * wd [n_experts][hidden][ffn_e], bf16 or int4 with scales as in tinfer_layer_src. tinfer_pack_moe
 * packs them into gu_packed (tinfer_moe_packed_bytes(..., 0) bytes: each expert's gate/up rows
 * interleaved) and down_packed (..., 1); both 16-byte aligned, caller-owned. tinfer_op_moe: ids_dev
 * (int32 [top_k]) and weights_dev (fp32 [top_k]) are read on the device when the kernels run, so the
 * call has a fixed shape; x_dev (fp32 [hidden]), h_dev (fp32 [top_k][ffn_e], scratch that receives
 * the SwiGLU outputs) and y_dev (fp32 [hidden]) are 16-byte aligned. An id outside [0, n_experts)
 * reads expert 0 instead and sets *status_dev (int32, may be NULL; cleared first) to 1.
 * Asynchronous on `stream`. Supported: top_k in {1, 2, 4, 8}, hidden a width the step supports,
 * ffn_e a multiple of 8 (bf16) or 32 (int4) up to 2048; else TINFER_ERR_UNSUPPORTED. */
size_t tinfer_moe_packed_bytes(int weight_format, int group_size, int n_experts, int hidden, int ffn_e,
                               int which);
tinfer_status tinfer_pack_moe(int weight_format, int group_size, int scale_dtype, int n_experts,
                              int hidden, int ffn_e, const void* wg_dev, const void* sg_dev,
                              const void* wu_dev, const void* su_dev, const void* wd_dev,
                              const void* sd_dev, void* gu_packed_dev, void* down_packed_dev,
                              void* stream);
tinfer_status tinfer_op_moe(int weight_format, int group_size, int scale_dtype, int n_experts,
                            int top_k, int hidden, int ffn_e, const void* gu_packed_dev,
                            const void* down_packed_dev, const int32_t* ids_dev,
                            const float* weights_dev, const float* x_dev, float* h_dev, float* y_dev,
                            int accumulate, int32_t* status_dev, void* stream);

/* Dense bf16 matrix product of a batched prefill on the tensor cores ("How I built an LLM inference
 * engine from scratch in CUDA", "What I'd tell someone starting, and what's next": the prompt's
 * tokens processed as one batch turn each linear layer's matrix-vector products into one
 * matrix-matrix product, where tensor cores apply; "Llama-1B: optimizing kernels": GEMM for prefill,
 * GEMV for decode): y[i][r] = sum_c x[i][c] w[r][c] for i < m, r < n, products of bf16 values
 * accumulated in fp32 (tcgen05.mma, accumulator in tensor memory).
 * x_dev: bf16 [m][k] row-major (the prompt's normalised activations), w_dev: bf16 [n][k] row-major
 * (a canonical weight matrix, or the bf16 rows of a packed layer, which have the same layout),
 * y_dev: fp32 [m][n] row-major; all caller-owned device memory. k must be a multiple of 8 and x_dev,
 * w_dev 16-byte aligned (TMA tensor maps), else TINFER_ERR_INVALID_ARG; m and n are free (edges are
 * zero-filled and masked). Synchronises `stream` before returning; a device wait that ran out
 * returns TINFER_ERR_TIMEOUT. */
tinfer_status tinfer_op_gemm_bf16(int m, int n, int k, const void* x_dev, const void* w_dev, float* y_dev,
                                  void* stream);

/* ---------------------------------------------------------------------------------------------
 * Attention that allocates nothing. The pages have no counterpart of this call: it is an
 * engineering addition for embedders.
 *
 * Same operation, arguments, layouts and results as tinfer_op_attention with the optional partial
 * outputs left out. The difference: the call allocates no device memory. Its working set (the
 * RoPE row of pos, the per-KV-head merge tickets, the error word and the chunk partials) lives in
 * one scratch array of TINFER_NOALLOC_SCRATCH_BYTES compiled into the library, one per device.
 * It exists for callers that cannot allocate while they run: a serving process that has handed
 * the rest of device memory to its KV pool (a cudaMalloc would fail there), or one that must not
 * let a cudaMalloc / cudaFree synchronise the device under its other streams.
 *
 * - Size limit: n_kv_heads <= 256 and n_heads * n_chunks * (head_dim + 2) * 4 bytes <=
 *   TINFER_NOALLOC_SCRATCH_BYTES - 2048 (n_chunks as chosen when 0 is passed). A call beyond it
 *   returns TINFER_ERR_UNSUPPORTED before touching the device.
 * - Set-up: the first call on a device, made with that device current, looks up the scratch
 *   array's address (cudaGetSymbolAddress) and keeps it; make that first call before any stream
 *   capture begins.
 * - Each call clears the error word and the tickets on `stream` before its launch.
 * - The scratch is shared by every call on a device: calls that overlap in time (other streams,
 *   other host threads) race on it and must be serialised by the caller.
 * - Synchronises `stream` before returning; device-side failures come back as the status
 *   (TINFER_ERR_TIMEOUT, TINFER_ERR_NONFINITE) exactly as for tinfer_op_attention.
 * --------------------------------------------------------------------------------------------- */
#define TINFER_NOALLOC_SCRATCH_BYTES (1u << 20)
tinfer_status tinfer_op_attention_noalloc(int n_heads, int n_kv_heads, int head_dim, int max_ctx,
                                          double rope_theta, int pos, int n_chunks,
                                          const float* qkv_dev, void* k_layer_dev,
                                          void* v_layer_dev, float* out_dev, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* TINFER_H */
