/* oracle.h -- reference CPU decoder for the batch-1 decode step (test infrastructure).
 *
 * This header belongs to the oracle alone. It is used by the oracle's own C source and, through
 * ctypes, by the tests, the smoke check and the benchmark's CPU-baseline leg. The CUDA library
 * shares nothing with it: no header, no helper, no table.
 *
 * Precision: every floating-point value is `orc_real`, which is double in the default build
 * (liboracle_f64.so) and float in the fp32 build (liboracle_f32.so). Weights stay in their stored
 * format (bf16 bits, or int4 nibbles plus fp16/bf16 scale bits) and are decoded exactly.
 *
 * Canonical layouts (the oracle's input contract; the GPU packer starts from the same bytes):
 *   bf16 matrix     : uint16 bits, row-major [rows][cols]  (rows = outputs, cols = inputs)
 *   int4 matrix     : uint8, row-major [rows][cols/2]; input element 2j is the low nibble of byte j,
 *                     element 2j+1 the high nibble; value w = (q - 8) * s
 *   int4 scales     : uint16 bits (fp16 or bf16), row-major [rows][cols/group]; group = consecutive
 *                     `group` inputs of one row
 *   KV cache        : bf16 bits [n_layers][n_kv_heads][max_ctx][head_dim], K and V separate
 */
#ifndef ORACLE_H
#define ORACLE_H
#include <stdint.h>

#ifndef ORACLE_REAL
#define ORACLE_REAL double
#endif
typedef ORACLE_REAL orc_real;

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_OK = 0, ORC_ERR_NONFINITE = -1, ORC_ERR_INVALID = -2 };
enum { ORC_BF16 = 0, ORC_INT4 = 1 };

typedef struct {
  const void* wq; const void* wk; const void* wv; const void* wo;   /* bf16 bits or int4 bytes */
  const void* wg; const void* wu; const void* wd;
  const uint16_t* sq; const uint16_t* sk; const uint16_t* sv; const uint16_t* so;  /* int4 scales */
  const uint16_t* sg; const uint16_t* su; const uint16_t* sd;
  const uint16_t* bq; const uint16_t* bk; const uint16_t* bv;  /* bf16 bias, or NULL */
  const uint16_t* g1; const uint16_t* g2;                      /* bf16 RMSNorm gains [hidden] */
} orc_layer;

typedef struct {
  int n_layers, hidden, n_heads, n_kv_heads, head_dim, ffn, vocab, max_ctx;
  double rope_theta, rms_eps;
  int weight_format;   /* ORC_BF16 or ORC_INT4 (int4 covers q,k,v,o,gate,up,down only) */
  int group_size;      /* int4 group length along the input dimension */
  int scale_is_bf16;   /* int4 scale format: 0 = fp16, 1 = bf16 */
  int qkv_bias;        /* 1: add bq/bk/bv before RoPE */
  const uint16_t* embed;       /* [vocab][hidden] bf16 */
  const uint16_t* lm_head;     /* [vocab][hidden] bf16 (same pointer as embed when tied) */
  const uint16_t* final_norm;  /* [hidden] bf16 */
  const orc_layer* layers;     /* [n_layers] */
} orc_model;

int  orc_real_bytes(void);
void orc_set_threads(int n);
int  orc_get_threads(void);

/* scalar formats */
double   orc_bf16_value(uint16_t bits);
double   orc_fp16_value(uint16_t bits);
uint16_t orc_round_bf16(double v);

/* building blocks */
void orc_rmsnorm(const orc_real* x, const uint16_t* gain, int n, double eps, orc_real* y);
void orc_gemv_bf16(const uint16_t* w, int rows, int cols, const orc_real* x, orc_real* y);
void orc_dequant_int4(const uint8_t* wq, const uint16_t* scales, int scale_is_bf16, int rows,
                      int cols, int group, orc_real* w_out);
void orc_gemv_int4(const uint8_t* wq, const uint16_t* scales, int scale_is_bf16, int rows, int cols,
                   int group, const orc_real* x, orc_real* y);
void orc_rope(orc_real* v, int head_dim, int pos, double theta);
void orc_softmax(const orc_real* s, int n, orc_real* p);
void orc_attention(const orc_real* q, const uint16_t* k, const uint16_t* v, int n_heads,
                   int n_kv_heads, int head_dim, int n_ctx, int ctx_stride, orc_real* out);
void orc_attention_partials(const orc_real* q, const uint16_t* k, const uint16_t* v, int n_heads,
                            int n_kv_heads, int head_dim, int n_ctx, int ctx_stride,
                            int chunk_len, int n_chunks, orc_real* m, orc_real* l, orc_real* o);
void orc_attention_combine(const orc_real* m, const orc_real* l, const orc_real* o, int n_heads,
                           int head_dim, int n_chunks, orc_real* out);
void orc_swiglu(const orc_real* gate, const orc_real* up, int n, orc_real* a);
int  orc_argmax(const orc_real* logits, int n, int* idx);

/* Gathered-expert SwiGLU MLP ("One launch per token", section "The same trick, sparser: a 64-expert
 * MoE": the router's chosen expert ids sit in a tensor, one kernel computes the gated/up SwiGLU of
 * the chosen experts gathered by id, another the down projection and the weighted sum):
 *   y = sum_{i < top_k} weight[i] * Wd[id_i] (silu(Wg[id_i] x) * (Wu[id_i] x)).
 * Expert e's matrices: gate, up [ffn_e][hidden] and down [hidden][ffn_e], stored expert after expert
 * (bf16 bits, or int4 bytes with scales as in the dense linears); x [hidden], y [hidden]. */
void orc_moe_mlp(int weight_format, int group, int scale_is_bf16, int hidden, int ffn_e,
                 const void* wg, const uint16_t* sg, const void* wu, const uint16_t* su,
                 const void* wd, const uint16_t* sd, int top_k, const int32_t* ids,
                 const orc_real* weights, const orc_real* x, orc_real* y);

/* the whole step: embed, n_layers decoder layers, final norm, LM head, argmax. Writes K/V of
 * every layer at slot `pos` and attends over [0, pos]. trace_x (optional, [n_layers][hidden])
 * receives the residual stream after each layer. */
int orc_decode_step(const orc_model* m, int token, int pos, uint16_t* kcache, uint16_t* vcache,
                    orc_real* logits, int* argmax, orc_real* trace_x);

#ifdef __cplusplus
}
#endif
#endif
