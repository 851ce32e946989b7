// api.cu -- host side of the C ABI declared in include/tinfer.h.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdlib>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "engine.h"
#include "kernels.h"
#include "tinfer.h"

using namespace tinfer;

namespace {

constexpr int SLOT_MIN = 32 * 1024;
constexpr long long DEFAULT_TIMEOUT_NS = 200LL * 1000 * 1000;

tinfer_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return TINFER_OK;
  if (e == cudaErrorMemoryAllocation) return TINFER_ERR_OOM;
  return TINFER_ERR_CUDA;
}

#define TRY_CUDA(expr)                                    \
  do {                                                    \
    cudaError_t e_ = (expr);                              \
    if (e_ != cudaSuccess) return from_cuda(e_);          \
  } while (0)

tinfer_status status_of_word(int w) {
  if (w & EW_TIMEOUT) return TINFER_ERR_TIMEOUT;
  if (w & EW_NONFINITE) return TINFER_ERR_NONFINITE;
  if (w & EW_BADTOKEN) return TINFER_ERR_INVALID_ARG;
  return w ? TINFER_ERR_CUDA : TINFER_OK;
}

int max_row_bytes(const tinfer_config* c) {
  const int g = c->group_size;
  size_t m = packed_row_bytes(c->weight_format, c->hidden, g) * 2;  // one gate/up pair
  m = std::max(m, packed_row_bytes(c->weight_format, c->n_heads * c->head_dim, g));
  m = std::max(m, packed_row_bytes(c->weight_format, c->ffn, g));
  m = std::max(m, (size_t)c->hidden * 2);
  return (int)m;
}

// bytes of the shared-memory copy of the widest GEMV input vector (fp32 hidden, attention output or
// SwiGLU output)


int slot_bytes_for(const tinfer_config* c) {
  const int m = max_row_bytes(c);
  return m <= SLOT_MIN ? SLOT_MIN : (int)align_up((size_t)m, 1024);
}

// Chunks per KV head the attention uses at any position up to max_ctx (the partial buffers'
// capacity), by the device split's rule: enough chunks to cover the grid, each fitting one slot.
int nch_capacity(int max_ctx, int nkv, int d, int grid, int slot) {
  int tmax = slot / (2 * d);
  if (tmax > T_MAX) tmax = T_MAX;
  const int nmin = (max_ctx + tmax - 1) / tmax;
  int want = grid / nkv;
  if (want < 1) want = 1;
  if (want > T_MAX) want = T_MAX;
  return nmin > want ? nmin : want;
}

// The input-vector buffer: the longest GEMV input in fp32.
int xs_bytes_for(const tinfer_config* c) {
  int n = c->hidden;
  if (c->n_heads * c->head_dim > n) n = c->n_heads * c->head_dim;
  if (c->ffn > n) n = c->ffn;
  return (int)align_up((size_t)n * 4, 128);
}

void rope_table(std::vector<float2>& t, int max_ctx, int d, double theta) {
  const int half = d / 2;
  t.resize((size_t)max_ctx * half);
  for (int p = 0; p < max_ctx; ++p)
    for (int i = 0; i < half; ++i) {
      const double ang = (double)p * std::pow(theta, -2.0 * (double)i / (double)d);
      t[(size_t)p * half + i] = make_float2((float)std::cos(ang), (float)std::sin(ang));
    }
}

}  // namespace

struct tinfer_ctx {
  tinfer_config cfg{};
  int device = 0;
  int num_sms = 0;
  StepParams p{};
  int slot = 0;
  int stages_mega = 0, stages_phase = 0, xs_bytes = 0;
  size_t smem_mega = 0, smem_phase = 0;
  void* scratch = nullptr;
  float2* rope_dev = nullptr;
  int* err_host = nullptr;     // mapped pinned
  int* err_host_dev = nullptr;
  int* pinned = nullptr;       // [2] host staging for tinfer_generate
  int* gen_dev = nullptr;      // [2] token in, argmax out for tinfer_generate
  int* argmax_fallback = nullptr;
  size_t tickets_off = 0, err_off = 0;
  // graph mode
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t gexec = nullptr;
  cudaGraphNode_t begin_node = nullptr;
  cudaKernelNodeParams begin_kp{};
  struct BeginArgs {
    int* step_dev; int token; const int* token_dev; int pos; int V; int* err; int* err_host;
  } bargs{};
  void* bptrs[7]{};
  float* graph_logits = nullptr;
  int* graph_argmax = nullptr;
  cudaStream_t cap_stream = nullptr;
};

extern "C" {

const char* tinfer_status_string(tinfer_status s) {
  switch (s) {
    case TINFER_OK: return "ok";
    case TINFER_ERR_INVALID_ARG: return "invalid argument";
    case TINFER_ERR_UNSUPPORTED: return "unsupported shape or format";
    case TINFER_ERR_CUDA: return "CUDA runtime error";
    case TINFER_ERR_OOM: return "out of memory";
    case TINFER_ERR_NONFINITE: return "non-finite logit";
    case TINFER_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

// The bf16 GEMV instance of the step kernels for a model: bf16 models stream every matrix in bf16,
// int4 models only the LM head.
static int model_nchl(const tinfer_config* c) {
  const int cols[4] = {c->hidden, c->n_heads * c->head_dim, c->ffn, c->hidden};
  return c->weight_format == TINFER_BF16 ? nchl_instance(cols, 4) : nchl_instance(cols + 3, 1);
}

tinfer_status tinfer_check_config(const tinfer_config* c) {
  if (!c) return TINFER_ERR_INVALID_ARG;
  if (c->n_layers <= 0 || c->hidden <= 0 || c->n_heads <= 0 || c->n_kv_heads <= 0 ||
      c->head_dim <= 0 || c->ffn <= 0 || c->vocab <= 0 || c->max_ctx <= 0)
    return TINFER_ERR_INVALID_ARG;
  if (!(c->rope_theta > 0.0) || !(c->rms_eps >= 0.0)) return TINFER_ERR_INVALID_ARG;
  if (c->n_heads % c->n_kv_heads != 0 || c->head_dim % 2 != 0) return TINFER_ERR_INVALID_ARG;
  if (c->exec_mode != TINFER_MEGAKERNEL && c->exec_mode != TINFER_GRAPH) return TINFER_ERR_INVALID_ARG;
  if (c->ffn_split != 0 && c->ffn_split != 1) return TINFER_ERR_INVALID_ARG;
  // the column-split down projection: bf16 rows of hidden outputs, at most two 8-output chunks per
  // consumer thread; its in-kernel reduce needs the co-resident CTAs of the persistent launch
  if (c->ffn_split && (c->weight_format != TINFER_BF16 || c->exec_mode != TINFER_MEGAKERNEL ||
                       c->hidden % 8 != 0 || c->hidden / 8 > 2 * NCT))
    return TINFER_ERR_UNSUPPORTED;
  if (c->n_layers > MAX_LAYERS) return TINFER_ERR_UNSUPPORTED;
  if (c->weight_format != TINFER_BF16 && c->weight_format != TINFER_INT4) return TINFER_ERR_INVALID_ARG;
  if (c->n_heads / c->n_kv_heads > G_MAX || c->head_dim % 8 != 0 || c->head_dim > D_MAX)
    return TINFER_ERR_UNSUPPORTED;
  const int qd = c->n_heads * c->head_dim;
  const int widths[3] = {c->hidden, qd, c->ffn};
  for (int w : widths) {
    if (packed_row_bytes(c->weight_format, w, c->group_size) == 0) return TINFER_ERR_UNSUPPORTED;
    if (!seg_ok(c->weight_format, w)) return TINFER_ERR_UNSUPPORTED;
  }
  if (c->weight_format == TINFER_INT4 && c->scale_dtype != TINFER_SCALE_FP16 &&
      c->scale_dtype != TINFER_SCALE_BF16)
    return TINFER_ERR_INVALID_ARG;
  if (c->hidden % 8 != 0 || !seg_ok(TINFER_BF16, c->hidden)) return TINFER_ERR_UNSUPPORTED;  // LM head
  if (model_nchl(c) == 0) return TINFER_ERR_UNSUPPORTED;
  const int slot = slot_bytes_for(c);
  int tmax = slot / (2 * c->head_dim);
  if (tmax > T_MAX) tmax = T_MAX;
  if ((c->max_ctx + tmax - 1) / tmax > T_MAX) return TINFER_ERR_UNSUPPORTED;
  return TINFER_OK;
}

size_t tinfer_packed_row_bytes(int weight_format, int cols, int group_size) {
  return packed_row_bytes(weight_format, cols, group_size);
}

size_t tinfer_packed_layer_bytes(const tinfer_config* c) {
  if (tinfer_check_config(c) != TINFER_OK) return 0;
  return layer_layout(c->hidden, c->n_heads, c->n_kv_heads, c->head_dim, c->ffn, c->weight_format,
                      c->group_size, c->qkv_bias)
      .total;
}

static tinfer_status pack_one(int fmt, int group, const void* w, const void* s, int rows, int cols,
                              uint8_t* dst, int step, int first, cudaStream_t st) {
  const int rb = (int)packed_row_bytes(fmt, cols, group);
  const int wb = fmt == TINFER_INT4 ? cols / 2 : cols * 2;
  const int sb = fmt == TINFER_INT4 ? 2 * (cols / group) : 0;
  if (!w || (fmt == TINFER_INT4 && !s)) return TINFER_ERR_INVALID_ARG;
  TRY_CUDA(launch_pack_rows(dst, rb, step, first, rows, (const uint8_t*)w, wb,
                            fmt == TINFER_INT4 ? (const uint8_t*)s : nullptr, sb, st));
  return TINFER_OK;
}

static tinfer_status unpack_one(int fmt, int group, const void* w, const void* s, int rows, int cols,
                                const uint8_t* src, int step, int first, cudaStream_t st) {
  const int rb = (int)packed_row_bytes(fmt, cols, group);
  const int wb = fmt == TINFER_INT4 ? cols / 2 : cols * 2;
  const int sb = fmt == TINFER_INT4 ? 2 * (cols / group) : 0;
  if (!w || (fmt == TINFER_INT4 && !s)) return TINFER_ERR_INVALID_ARG;
  TRY_CUDA(launch_unpack_rows(src, rb, step, first, rows, (uint8_t*)w, wb,
                              fmt == TINFER_INT4 ? (uint8_t*)s : nullptr, sb, st));
  return TINFER_OK;
}

tinfer_status tinfer_pack_matrix(int fmt, int group, int scale_dtype, int rows, int cols,
                                 const void* w_dev, const void* scales_dev, void* packed_dev,
                                 void* stream) {
  (void)scale_dtype;
  if (rows <= 0 || !packed_dev || packed_row_bytes(fmt, cols, group) == 0) return TINFER_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(packed_dev) & 15) != 0) return TINFER_ERR_INVALID_ARG;
  return pack_one(fmt, group, w_dev, scales_dev, rows, cols, (uint8_t*)packed_dev, 1, 0,
                  (cudaStream_t)stream);
}

#define TRY(x)                                  \
  do {                                          \
    tinfer_status s_ = (x);                     \
    if (s_ != TINFER_OK) return s_;             \
  } while (0)

tinfer_status tinfer_pack_layer(const tinfer_config* c, const tinfer_layer_src* src,
                                void* packed_dev, void* stream) {
  TRY(tinfer_check_config(c));
  if (!src || !packed_dev || (reinterpret_cast<uintptr_t>(packed_dev) & 15) != 0)
    return TINFER_ERR_INVALID_ARG;
  const int H = c->hidden, nq = c->n_heads, nkv = c->n_kv_heads, d = c->head_dim, F = c->ffn;
  const int f = c->weight_format, g = c->group_size;
  const LayerLayout L = layer_layout(H, nq, nkv, d, F, f, g, c->qkv_bias);
  uint8_t* b = (uint8_t*)packed_dev;
  cudaStream_t st = (cudaStream_t)stream;
  TRY(pack_one(f, g, src->wq, src->sq, nq * d, H, b + L.off_qkv, 1, 0, st));
  TRY(pack_one(f, g, src->wk, src->sk, nkv * d, H, b + L.off_qkv, 1, nq * d, st));
  TRY(pack_one(f, g, src->wv, src->sv, nkv * d, H, b + L.off_qkv, 1, (nq + nkv) * d, st));
  TRY(pack_one(f, g, src->wo, src->so, H, nq * d, b + L.off_o, 1, 0, st));
  TRY(pack_one(f, g, src->wg, src->sg, F, H, b + L.off_gu, 2, 0, st));
  TRY(pack_one(f, g, src->wu, src->su, F, H, b + L.off_gu, 2, 1, st));
  if (c->ffn_split) {  // Wd^T: row f holds the weights of ffn input f for every hidden output
    if (!src->wd) return TINFER_ERR_INVALID_ARG;
    TRY_CUDA(launch_transpose_u16((const uint16_t*)src->wd, H, F, (uint16_t*)(b + L.off_down), st));
  } else {
    TRY(pack_one(f, g, src->wd, src->sd, H, F, b + L.off_down, 1, 0, st));
  }
  if (!src->g1 || !src->g2) return TINFER_ERR_INVALID_ARG;
  TRY_CUDA(launch_bf16_to_f32((const uint16_t*)src->g1, (float*)(b + L.off_g1), H, st));
  TRY_CUDA(launch_bf16_to_f32((const uint16_t*)src->g2, (float*)(b + L.off_g2), H, st));
  if (c->qkv_bias) {
    if (!src->bq || !src->bk || !src->bv) return TINFER_ERR_INVALID_ARG;
    float* bias = (float*)(b + L.off_bias);
    TRY_CUDA(launch_bf16_to_f32((const uint16_t*)src->bq, bias, nq * d, st));
    TRY_CUDA(launch_bf16_to_f32((const uint16_t*)src->bk, bias + nq * d, nkv * d, st));
    TRY_CUDA(launch_bf16_to_f32((const uint16_t*)src->bv, bias + (nq + nkv) * d, nkv * d, st));
  }
  return TINFER_OK;
}

tinfer_status tinfer_unpack_layer(const tinfer_config* c, const void* packed_dev,
                                  const tinfer_layer_src* dst, void* stream) {
  TRY(tinfer_check_config(c));
  if (!dst || !packed_dev) return TINFER_ERR_INVALID_ARG;
  const int H = c->hidden, nq = c->n_heads, nkv = c->n_kv_heads, d = c->head_dim, F = c->ffn;
  const int f = c->weight_format, g = c->group_size;
  const LayerLayout L = layer_layout(H, nq, nkv, d, F, f, g, c->qkv_bias);
  const uint8_t* b = (const uint8_t*)packed_dev;
  cudaStream_t st = (cudaStream_t)stream;
  TRY(unpack_one(f, g, dst->wq, dst->sq, nq * d, H, b + L.off_qkv, 1, 0, st));
  TRY(unpack_one(f, g, dst->wk, dst->sk, nkv * d, H, b + L.off_qkv, 1, nq * d, st));
  TRY(unpack_one(f, g, dst->wv, dst->sv, nkv * d, H, b + L.off_qkv, 1, (nq + nkv) * d, st));
  TRY(unpack_one(f, g, dst->wo, dst->so, H, nq * d, b + L.off_o, 1, 0, st));
  TRY(unpack_one(f, g, dst->wg, dst->sg, F, H, b + L.off_gu, 2, 0, st));
  TRY(unpack_one(f, g, dst->wu, dst->su, F, H, b + L.off_gu, 2, 1, st));
  if (c->ffn_split) {
    if (!dst->wd) return TINFER_ERR_INVALID_ARG;
    TRY_CUDA(launch_transpose_u16((const uint16_t*)(b + L.off_down), F, H, (uint16_t*)dst->wd, st));
  } else {
    TRY(unpack_one(f, g, dst->wd, dst->sd, H, F, b + L.off_down, 1, 0, st));
  }
  if (!dst->g1 || !dst->g2) return TINFER_ERR_INVALID_ARG;
  TRY_CUDA(launch_f32_to_bf16((const float*)(b + L.off_g1), (uint16_t*)dst->g1, H, st));
  TRY_CUDA(launch_f32_to_bf16((const float*)(b + L.off_g2), (uint16_t*)dst->g2, H, st));
  if (c->qkv_bias) {
    if (!dst->bq || !dst->bk || !dst->bv) return TINFER_ERR_INVALID_ARG;
    const float* bias = (const float*)(b + L.off_bias);
    TRY_CUDA(launch_f32_to_bf16(bias, (uint16_t*)dst->bq, nq * d, st));
    TRY_CUDA(launch_f32_to_bf16(bias + nq * d, (uint16_t*)dst->bk, nkv * d, st));
    TRY_CUDA(launch_f32_to_bf16(bias + (nq + nkv) * d, (uint16_t*)dst->bv, nkv * d, st));
  }
  return TINFER_OK;
}

static void free_ctx(tinfer_ctx* x) {
  if (!x) return;
  if (x->gexec) cudaGraphExecDestroy(x->gexec);
  if (x->graph) cudaGraphDestroy(x->graph);
  if (x->cap_stream) cudaStreamDestroy(x->cap_stream);
  if (x->scratch) cudaFree(x->scratch);
  if (x->rope_dev) cudaFree(x->rope_dev);
  if (x->err_host) cudaFreeHost(x->err_host);
  if (x->pinned) cudaFreeHost(x->pinned);
  delete x;
}

tinfer_status tinfer_create(const tinfer_config* c, const tinfer_weights* w, void* k_cache_dev,
                            void* v_cache_dev, tinfer_ctx** out) {
  if (!out) return TINFER_ERR_INVALID_ARG;
  *out = nullptr;
  TRY(tinfer_check_config(c));
  if (!w || !w->embed || !w->lm_head || !w->final_norm || !w->layer_blobs || !k_cache_dev || !v_cache_dev)
    return TINFER_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(w->embed) & 15) != 0 || (reinterpret_cast<uintptr_t>(w->final_norm) & 7) != 0)
    return TINFER_ERR_INVALID_ARG;
  for (int l = 0; l < c->n_layers; ++l)
    if (!w->layer_blobs[l] || (reinterpret_cast<uintptr_t>(w->layer_blobs[l]) & 15) != 0)
      return TINFER_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(w->lm_head) & 15) != 0 ||
      (reinterpret_cast<uintptr_t>(k_cache_dev) & 15) != 0 ||
      (reinterpret_cast<uintptr_t>(v_cache_dev) & 15) != 0)
    return TINFER_ERR_INVALID_ARG;

  tinfer_ctx* x = new (std::nothrow) tinfer_ctx();
  if (!x) return TINFER_ERR_OOM;
  x->cfg = *c;
  tinfer_status st = TINFER_OK;
  auto fail = [&](tinfer_status s) { free_ctx(x); return s; };
  auto cu = [&](cudaError_t e) { return e == cudaSuccess ? TINFER_OK : from_cuda(e); };

  if ((st = cu(cudaGetDevice(&x->device))) != TINFER_OK) return fail(st);
  int smem_optin = 0;
  if ((st = cu(cudaDeviceGetAttribute(&x->num_sms, cudaDevAttrMultiProcessorCount, x->device))) != TINFER_OK) return fail(st);
  if ((st = cu(cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, x->device))) != TINFER_OK) return fail(st);
  int smem_per_sm = 0;
  if ((st = cu(cudaDeviceGetAttribute(&smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, x->device))) != TINFER_OK) return fail(st);

  x->slot = slot_bytes_for(c);
  x->xs_bytes = xs_bytes_for(c);
  const size_t misc = smem_for(0, 0, x->xs_bytes);
  smem_optin -= (int)static_smem_mega();  // the persistent kernel's static shared memory
  x->stages_mega = (int)((smem_optin - misc) / x->slot);
  if (x->stages_mega > 8) x->stages_mega = 8;
  while (x->stages_mega > 2 && smem_for(x->stages_mega, x->slot, x->xs_bytes) > (size_t)smem_optin) --x->stages_mega;
  // two CTAs of the per-phase kernel per SM, so that the next kernel's prefetch overlaps
  x->stages_phase = (int)((smem_per_sm / 2 - 1024 - misc) / x->slot);
  if (x->stages_phase > 4) x->stages_phase = 4;
  if (x->stages_phase < 2) x->stages_phase = x->stages_mega < 4 ? x->stages_mega : 4;
  while (x->stages_phase > 2 && smem_for(x->stages_phase, x->slot, x->xs_bytes) > (size_t)smem_optin) --x->stages_phase;
  if (x->stages_mega < 2 || x->stages_phase < 2) return fail(TINFER_ERR_UNSUPPORTED);
  x->smem_mega = smem_for(x->stages_mega, x->slot, x->xs_bytes);
  x->smem_phase = smem_for(x->stages_phase, x->slot, x->xs_bytes);
  const int nchl = model_nchl(c);
  if ((st = cu(set_smem_mega(x->smem_mega, c->weight_format, nchl))) != TINFER_OK) return fail(st);
  if ((st = cu(set_smem_phase(x->smem_phase, c->weight_format, nchl))) != TINFER_OK) return fail(st);
  int occ = 0;
  if ((st = cu(megakernel_occupancy(&occ, x->smem_mega, c->weight_format, nchl))) != TINFER_OK) return fail(st);
  if (occ < 1) return fail(TINFER_ERR_UNSUPPORTED);
  const int grid = x->num_sms;  // one persistent CTA per SM (co-residency: cooperative launch)
  if (c->ffn_split && grid > 256) return fail(TINFER_ERR_UNSUPPORTED);  // partials per reduce lane
  {
    // row results of one GEMV phase must fit the per-CTA shared-memory buffer
    const int f = c->weight_format;
    const int qd = c->n_heads * c->head_dim;
    const int rows[4] = {(c->n_heads + 2 * c->n_kv_heads) * c->head_dim, c->hidden, 2 * c->ffn, c->hidden};
    const int cols[4] = {c->hidden, qd, c->hidden, c->ffn};
    for (int i = 0; i < 4; ++i)
      if ((long long)((rows[i] + grid - 1) / grid + 1) * seg_info(f, cols[i]).nseg > ROWV_MAX)
        return fail(TINFER_ERR_UNSUPPORTED);
    const int lm_seg = seg_info(TINFER_BF16, c->hidden).nseg;  // LM rows wider than one segment
    if (lm_seg > 1 && (long long)((c->vocab + grid - 1) / grid) * lm_seg > ROWV_MAX)
      return fail(TINFER_ERR_UNSUPPORTED);
  }

  const int H = c->hidden, nq = c->n_heads, nkv = c->n_kv_heads, d = c->head_dim, F = c->ffn;
  const int qkv_rows = (nq + 2 * nkv) * d;
  const int nch_cap = nch_capacity(c->max_ctx, nkv, d, grid, x->slot);

  // scratch: one allocation
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t o = off; off = align_up(off + bytes, 256); return o; };
  // activations handed between phases: stamped 8-byte words
  const size_t o_xa = take((size_t)H * 8), o_xb = take((size_t)H * 8), o_qkv = take((size_t)qkv_rows * 8);
  const size_t o_attn = take((size_t)nq * d * 8), o_act = take((size_t)F * 8);
  const size_t o_pm = take((size_t)nq * nch_cap * 4), o_pl = take((size_t)nq * nch_cap * 4);
  const size_t o_po = take((size_t)nq * nch_cap * d * 4);
  const size_t o_pmw = take((size_t)nq * nch_cap * 8), o_plw = take((size_t)nq * nch_cap * 8);
  const size_t o_pow = take((size_t)nq * nch_cap * d * 8);
  const size_t o_tk = take((size_t)(nkv + 1) * 4);
  const size_t o_bv = take((size_t)grid * 4), o_bi = take((size_t)grid * 4), o_bb = take((size_t)grid * 4);
  const size_t o_err = take(4), o_step = take(2 * 4), o_gen = take(2 * 4), o_am = take(4);
  const size_t o_bw = take((size_t)grid * 16), o_kvf = take((size_t)c->n_layers * nkv * 4);
  const size_t o_pf = take(c->ffn_split ? (size_t)grid * H * 8 : 8);
  const size_t o_bar = take(8);
  if ((st = cu(cudaMalloc(&x->scratch, off))) != TINFER_OK) return fail(st);
  if ((st = cu(cudaMemset(x->scratch, 0, off))) != TINFER_OK) return fail(st);
  uint8_t* s = (uint8_t*)x->scratch;
  x->tickets_off = o_tk; x->err_off = o_err;

  // layers
  const LayerLayout LL = layer_layout(H, nq, nkv, d, F, c->weight_format, c->group_size, c->qkv_bias);
  std::vector<LayerDev> ld(c->n_layers);
  if (c->n_layers > MAX_LAYERS) return fail(TINFER_ERR_UNSUPPORTED);
  for (int l = 0; l < c->n_layers; ++l) {
    const uint8_t* b = (const uint8_t*)w->layer_blobs[l];
    ld[l].qkv = b + LL.off_qkv; ld[l].o = b + LL.off_o; ld[l].gu = b + LL.off_gu;
    ld[l].down = b + LL.off_down; ld[l].g1 = (const float*)(b + LL.off_g1);
    ld[l].g2 = (const float*)(b + LL.off_g2);
    ld[l].bias = c->qkv_bias ? (const float*)(b + LL.off_bias) : nullptr;
  }

  std::vector<float2> rt;
  rope_table(rt, c->max_ctx, d, c->rope_theta);
  if ((st = cu(cudaMalloc(&x->rope_dev, sizeof(float2) * rt.size()))) != TINFER_OK) return fail(st);
  if ((st = cu(cudaMemcpy(x->rope_dev, rt.data(), sizeof(float2) * rt.size(), cudaMemcpyHostToDevice))) != TINFER_OK) return fail(st);

  if ((st = cu(cudaHostAlloc(&x->err_host, 4, cudaHostAllocMapped))) != TINFER_OK) return fail(st);
  *x->err_host = 0;
  if ((st = cu(cudaHostGetDevicePointer((void**)&x->err_host_dev, x->err_host, 0))) != TINFER_OK) return fail(st);
  if ((st = cu(cudaHostAlloc(&x->pinned, 8, cudaHostAllocDefault))) != TINFER_OK) return fail(st);

  StepParams& p = x->p;
  Dims& m = p.m;
  m.L = c->n_layers; m.H = H; m.nq = nq; m.nkv = nkv; m.d = d; m.F = F; m.V = c->vocab;
  m.max_ctx = c->max_ctx; m.fmt = c->weight_format; m.group = c->group_size;
  m.scale_bf16 = c->scale_dtype == TINFER_SCALE_BF16; m.eps = (float)c->rms_eps;
  m.rb_h = (int)packed_row_bytes(m.fmt, H, m.group);
  m.rb_qd = (int)packed_row_bytes(m.fmt, nq * d, m.group);
  m.rb_f = (int)packed_row_bytes(m.fmt, F, m.group);
  m.rb_lm = H * 2;
  m.qkv_rows = qkv_rows;
  m.nchl = nchl;
  m.ffn_split = c->ffn_split;
  for (int l = 0; l < c->n_layers; ++l) p.layers[l] = ld[l];
  p.embed = (const uint16_t*)w->embed;
  p.lm_head = (const uint16_t*)w->lm_head;
  p.final_norm = (const uint16_t*)w->final_norm;
  p.kcache = (uint16_t*)k_cache_dev;
  p.vcache = (uint16_t*)v_cache_dev;
  p.rope = x->rope_dev;
  p.xa = (uint64_t*)(s + o_xa); p.xb = (uint64_t*)(s + o_xb); p.qkv = (uint64_t*)(s + o_qkv);
  p.attn = (uint64_t*)(s + o_attn); p.act = (uint64_t*)(s + o_act);
  p.part_ffn = (uint64_t*)(s + o_pf);
  p.sync_barrier = 0;
  p.bar_count = (unsigned long long*)(s + o_bar);
  p.bar_base = 0;
  p.epoch = 1;  // the buffers start zeroed: stamp 0 is never expected
  p.stamp_check = c->exec_mode == TINFER_MEGAKERNEL;
  p.part_m = (float*)(s + o_pm); p.part_l = (float*)(s + o_pl); p.part_o = (float*)(s + o_po);
  p.part_mw = (uint64_t*)(s + o_pmw); p.part_lw = (uint64_t*)(s + o_plw); p.part_ow = (uint64_t*)(s + o_pow);
  p.tickets = (unsigned*)(s + o_tk);
  p.best_val = (float*)(s + o_bv); p.best_idx = (int*)(s + o_bi); p.best_bad = (int*)(s + o_bb);
  p.err = (int*)(s + o_err);
  p.err_host = x->err_host_dev;
  p.nch_cap = nch_cap;
  p.grid = grid;
  p.slot_bytes = x->slot;
  // producer schedule (tinfer_set_schedule changes it): two bulk copies in flight, four during the
  // LM head; bf16 models prefetch up to 512 KB per CTA into L2 ahead of the ring at about one SM's
  // share of HBM bandwidth. int4 models do not: their consumers are bound by the dequantisation
  // arithmetic, not by the stream, and the extra traffic only lengthens their L2 round trips
  // (TinyLlama-shaped step 0.755 ms with the lookahead, 0.730 ms without, on one GB300).
  p.inflight = 2;
  p.inflight_lm = 4;
  p.l2_lookahead = c->weight_format == TINFER_BF16 ? 512 * 1024 : 0;
  p.l2_pace_ns_per_kb = 24;
  p.timeout_ns = DEFAULT_TIMEOUT_NS;
  p.step_dev = (int*)(s + o_step);
  x->gen_dev = (int*)(s + o_gen);
  x->argmax_fallback = (int*)(s + o_am);
  p.n_chunks_override = 0;
  p.n_steps = 1;
  p.tokens_out = nullptr;
  p.count_out = nullptr;
  p.eos = -1;
  p.best_w = (uint64_t*)(s + o_bw);
  p.kvflag = (unsigned*)(s + o_kvf);
  p.dbg_skip_cta = -1;
  p.dbg_skip_phase = -1;
  p.trace = nullptr;
  *out = x;
  return TINFER_OK;
}

void tinfer_destroy(tinfer_ctx* x) { free_ctx(x); }

static tinfer_status build_graph(tinfer_ctx* x, float* logits, int* argmax) {
  if (x->gexec || x->graph) TRY_CUDA(cudaDeviceSynchronize());  // no launch of the old graph in flight
  if (x->gexec) { cudaGraphExecDestroy(x->gexec); x->gexec = nullptr; }
  if (x->graph) { cudaGraphDestroy(x->graph); x->graph = nullptr; }
  if (!x->cap_stream) TRY_CUDA(cudaStreamCreateWithFlags(&x->cap_stream, cudaStreamNonBlocking));
  StepParams p = x->p;
  p.ring_stages = x->stages_phase;
  p.token = 0; p.token_dev = nullptr; p.pos = 0;
  p.logits = logits; p.argmax = argmax;
  p.dbg_skip_cta = -1;
  p.trace = nullptr;
  cudaStream_t cs = x->cap_stream;
  TRY_CUDA(cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal));
  cudaError_t e = launch_begin(const_cast<int*>(p.step_dev), 0, nullptr, 0, x->cfg.vocab, p.err, p.err_host, cs);
  const int nph = x->cfg.n_layers * PHASES_PER_LAYER + 1;
  for (int k = 0; k < nph && e == cudaSuccess; ++k) e = launch_phase(p, k, x->smem_phase, cs, k > 0);
  cudaGraph_t g = nullptr;
  cudaError_t e2 = cudaStreamEndCapture(cs, &g);
  if (e != cudaSuccess || e2 != cudaSuccess) {
    if (g) cudaGraphDestroy(g);
    return from_cuda(e != cudaSuccess ? e : e2);
  }
  x->graph = g;
  size_t n = 0;
  TRY_CUDA(cudaGraphGetNodes(g, nullptr, &n));
  std::vector<cudaGraphNode_t> nodes(n);
  TRY_CUDA(cudaGraphGetNodes(g, nodes.data(), &n));
  x->begin_node = nullptr;
  for (auto nd : nodes) {
    cudaGraphNodeType t;
    TRY_CUDA(cudaGraphNodeGetType(nd, &t));
    if (t != cudaGraphNodeTypeKernel) continue;
    cudaKernelNodeParams kp;
    TRY_CUDA(cudaGraphKernelNodeGetParams(nd, &kp));
    if (kp.func == begin_kernel_fn()) { x->begin_node = nd; x->begin_kp = kp; }
  }
  if (!x->begin_node) return TINFER_ERR_CUDA;
  TRY_CUDA(cudaGraphInstantiate(&x->gexec, g, 0));
  x->bargs = tinfer_ctx::BeginArgs{const_cast<int*>(p.step_dev), 0, nullptr, 0, x->cfg.vocab, p.err, p.err_host};
  x->bptrs[0] = &x->bargs.step_dev; x->bptrs[1] = &x->bargs.token; x->bptrs[2] = &x->bargs.token_dev;
  x->bptrs[3] = &x->bargs.pos; x->bptrs[4] = &x->bargs.V; x->bptrs[5] = &x->bargs.err;
  x->bptrs[6] = &x->bargs.err_host;
  x->begin_kp.kernelParams = x->bptrs;
  x->begin_kp.extra = nullptr;
  x->graph_logits = logits;
  x->graph_argmax = argmax;
  return TINFER_OK;
}

static tinfer_status step_impl(tinfer_ctx* x, int token, const int* token_dev, int pos,
                               cudaStream_t st, float* logits, int* argmax) {
  if (!x) return TINFER_ERR_INVALID_ARG;
  if (pos < 0 || pos >= x->cfg.max_ctx) return TINFER_ERR_INVALID_ARG;
  if (!token_dev && (token < 0 || token >= x->cfg.vocab)) return TINFER_ERR_INVALID_ARG;
  const int pending = *reinterpret_cast<volatile int*>(x->err_host);
  if (pending) return status_of_word(pending);
  if (!argmax) argmax = x->argmax_fallback;
  if (x->cfg.exec_mode == TINFER_MEGAKERNEL) {
    StepParams p = x->p;
    p.ring_stages = x->stages_mega;
    p.token = token; p.token_dev = token_dev; p.pos = pos;
    p.logits = logits; p.argmax = argmax;
    TRY_CUDA(launch_megakernel(p, x->smem_mega, st));
    x->p.dbg_skip_cta = -1;  // an injected fault applies to one step only
    x->p.epoch += (unsigned)(x->cfg.n_layers * PHASES_PER_LAYER + 2);  // fresh stamps for the next step
    if (x->p.sync_barrier) x->p.bar_base += (unsigned long long)(x->cfg.n_layers * PHASES_PER_LAYER);
    return TINFER_OK;
  }
  if (!x->gexec || x->graph_logits != logits || x->graph_argmax != argmax)
    TRY(build_graph(x, logits, argmax));
  x->bargs.token = token; x->bargs.token_dev = token_dev; x->bargs.pos = pos;
  TRY_CUDA(cudaGraphExecKernelNodeSetParams(x->gexec, x->begin_node, &x->begin_kp));
  TRY_CUDA(cudaGraphLaunch(x->gexec, st));
  return TINFER_OK;
}

tinfer_status tinfer_decode_step(tinfer_ctx* x, int32_t token_id, int32_t pos, void* stream,
                                 float* logits_dev, int32_t* argmax_dev) {
  return step_impl(x, token_id, nullptr, pos, (cudaStream_t)stream, logits_dev, argmax_dev);
}

tinfer_status tinfer_decode_step_dev(tinfer_ctx* x, const int32_t* token_dev, int32_t pos,
                                     void* stream, float* logits_dev, int32_t* argmax_dev) {
  if (!token_dev) return TINFER_ERR_INVALID_ARG;
  return step_impl(x, 0, token_dev, pos, (cudaStream_t)stream, logits_dev, argmax_dev);
}

tinfer_status tinfer_generate_dev(tinfer_ctx* x, int32_t first_token, int32_t pos0, int32_t n_steps,
                                  int32_t eos_token, void* stream, int32_t* tokens_dev,
                                  int32_t* count_dev) {
  if (!x || n_steps <= 0 || !tokens_dev) return TINFER_ERR_INVALID_ARG;
  if (pos0 < 0 || (long long)pos0 + n_steps > x->cfg.max_ctx) return TINFER_ERR_INVALID_ARG;
  if (first_token < 0 || first_token >= x->cfg.vocab) return TINFER_ERR_INVALID_ARG;
  if (eos_token < -1 || eos_token >= x->cfg.vocab) return TINFER_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(tokens_dev) & 3) || (reinterpret_cast<uintptr_t>(count_dev) & 3))
    return TINFER_ERR_INVALID_ARG;
  const int pending = *reinterpret_cast<volatile int*>(x->err_host);
  if (pending) return status_of_word(pending);
  cudaStream_t st = (cudaStream_t)stream;
  if (x->cfg.exec_mode != TINFER_MEGAKERNEL) {
    // the baseline: one graph launch per token, chained on the device
    if (eos_token >= 0 || count_dev) return TINFER_ERR_UNSUPPORTED;
    for (int k = 0; k < n_steps; ++k)
      TRY(step_impl(x, first_token, k ? tokens_dev + k - 1 : nullptr, pos0 + k, st, nullptr, tokens_dev + k));
    return TINFER_OK;
  }
  StepParams p = x->p;
  p.ring_stages = x->stages_mega;
  p.token = first_token; p.token_dev = nullptr; p.pos = pos0;
  p.logits = nullptr; p.argmax = x->argmax_fallback;
  p.n_steps = n_steps;
  p.tokens_out = tokens_dev;
  p.count_out = count_dev;
  p.eos = eos_token;
  TRY_CUDA(launch_megakernel(p, x->smem_mega, st));
  x->p.dbg_skip_cta = -1;
  x->p.epoch += (unsigned)n_steps * (unsigned)(x->cfg.n_layers * PHASES_PER_LAYER + 2);
  if (x->p.sync_barrier) x->p.bar_base += (unsigned long long)n_steps * (unsigned long long)(x->cfg.n_layers * PHASES_PER_LAYER);
  return TINFER_OK;
}

tinfer_status tinfer_get_error(tinfer_ctx* x) {
  if (!x) return TINFER_ERR_INVALID_ARG;
  TRY_CUDA(cudaDeviceSynchronize());
  int w = 0;
  TRY_CUDA(cudaMemcpy(&w, x->p.err, 4, cudaMemcpyDeviceToHost));
  if (w || *reinterpret_cast<volatile int*>(x->err_host)) {
    uint8_t* s = (uint8_t*)x->scratch;
    TRY_CUDA(cudaMemset(s + x->err_off, 0, 4));
    TRY_CUDA(cudaMemset(s + x->tickets_off, 0, (size_t)(x->cfg.n_kv_heads + 1) * 4));
    TRY_CUDA(cudaMemset(x->p.bar_count, 0, 8));
    x->p.bar_base = 0;
    TRY_CUDA(cudaDeviceSynchronize());
    *reinterpret_cast<volatile int*>(x->err_host) = 0;
  }
  return status_of_word(w);
}

tinfer_status tinfer_generate(tinfer_ctx* x, int32_t first_token, int32_t pos0, int32_t n_steps,
                              void* stream, int32_t* tokens_host) {
  if (!x || n_steps < 0 || !tokens_host) return TINFER_ERR_INVALID_ARG;
  if (pos0 < 0 || (long long)pos0 + n_steps > x->cfg.max_ctx) return TINFER_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  int tok = first_token;
  for (int k = 0; k < n_steps; ++k) {
    x->pinned[0] = tok;
    TRY_CUDA(cudaMemcpyAsync(x->gen_dev, x->pinned, 4, cudaMemcpyHostToDevice, st));
    TRY(step_impl(x, 0, x->gen_dev, pos0 + k, st, nullptr, x->gen_dev + 1));
    TRY_CUDA(cudaMemcpyAsync(x->pinned + 1, x->gen_dev + 1, 4, cudaMemcpyDeviceToHost, st));
    TRY_CUDA(cudaStreamSynchronize(st));
    const int w = *reinterpret_cast<volatile int*>(x->err_host);
    if (w) return tinfer_get_error(x);
    tok = x->pinned[1];
    tokens_host[k] = tok;
  }
  return TINFER_OK;
}

long long tinfer_query(const tinfer_ctx* x, int what) {
  if (!x) return -1;
  switch (what) {
    case TINFER_Q_GRID: return x->p.grid;
    case TINFER_Q_BLOCK_THREADS: return x->cfg.exec_mode == TINFER_MEGAKERNEL ? NTHREADS_MEGA : NTHREADS;
    case TINFER_Q_SMEM: return (long long)x->smem_mega;
    case TINFER_Q_RING_STAGES: return x->stages_mega;
    case TINFER_Q_SLOT_BYTES: return x->slot;
    case TINFER_Q_KERNELS_PER_STEP:
      return x->cfg.exec_mode == TINFER_MEGAKERNEL ? 1 : x->cfg.n_layers * PHASES_PER_LAYER + 2;
    case TINFER_Q_TRACE_BYTES:
      return (long long)x->p.grid * (x->cfg.n_layers * PHASES_PER_LAYER + 1) * TRACE_FIELDS * 8;
  }
  return -1;
}

tinfer_status tinfer_set_trace(tinfer_ctx* x, void* trace_dev) {
  if (!x) return TINFER_ERR_INVALID_ARG;
  if (trace_dev && (reinterpret_cast<uintptr_t>(trace_dev) & 7) != 0) return TINFER_ERR_INVALID_ARG;
  x->p.trace = (unsigned long long*)trace_dev;
  return TINFER_OK;
}

tinfer_status tinfer_set_schedule(tinfer_ctx* x, int knob, long long value) {
  if (!x) return TINFER_ERR_INVALID_ARG;
  StepParams& p = x->p;
  switch (knob) {
    case TINFER_S_L2_LOOKAHEAD:
      if (value < 0 || value > (64LL << 20)) return TINFER_ERR_INVALID_ARG;
      p.l2_lookahead = (int)value;
      break;
    case TINFER_S_L2_PACE:
      if (value < 0 || value > 100000) return TINFER_ERR_INVALID_ARG;
      p.l2_pace_ns_per_kb = (int)value;
      break;
    case TINFER_S_INFLIGHT:
      if (value < 0 || value > MAX_STAGES) return TINFER_ERR_INVALID_ARG;
      p.inflight = (int)value;
      break;
    case TINFER_S_INFLIGHT_LM:
      if (value < 0 || value > MAX_STAGES) return TINFER_ERR_INVALID_ARG;
      p.inflight_lm = (int)value;
      break;
    case TINFER_S_ATTN_CHUNKS: {
      // 0: the automatic split; n: every chunk must still fit one ring slot at max_ctx (n at least
      // the automatic split's minimum) and the partial buffers hold at most nch_cap chunks
      if (value == 0) { p.n_chunks_override = 0; break; }
      int tmax = p.slot_bytes / (2 * p.m.d);
      if (tmax > T_MAX) tmax = T_MAX;
      const long long nmin = (p.m.max_ctx + tmax - 1) / tmax;
      if (value < nmin || value > p.nch_cap) return TINFER_ERR_INVALID_ARG;
      p.n_chunks_override = (int)value;
      break;
    }
    case TINFER_S_SYNC:
      if (value != TINFER_SYNC_STAMPS && value != TINFER_SYNC_GRID_BARRIER) return TINFER_ERR_INVALID_ARG;
      if (x->cfg.exec_mode != TINFER_MEGAKERNEL) return TINFER_ERR_UNSUPPORTED;
      if (value == TINFER_SYNC_GRID_BARRIER && !p.sync_barrier) {
        // a fresh count: nothing of the context is running (the caller's stream order)
        TRY_CUDA(cudaDeviceSynchronize());
        TRY_CUDA(cudaMemset(p.bar_count, 0, 8));
        p.bar_base = 0;
      }
      p.sync_barrier = (int)value;
      break;
    default:
      return TINFER_ERR_INVALID_ARG;
  }
  if (x->gexec) { cudaGraphExecDestroy(x->gexec); x->gexec = nullptr; }  // rebuilt with the new values
  return TINFER_OK;
}

long long tinfer_get_schedule(const tinfer_ctx* x, int knob) {
  if (!x) return -1;
  switch (knob) {
    case TINFER_S_L2_LOOKAHEAD: return x->p.l2_lookahead;
    case TINFER_S_L2_PACE: return x->p.l2_pace_ns_per_kb;
    case TINFER_S_SYNC: return x->p.sync_barrier;
    case TINFER_S_INFLIGHT: return x->p.inflight;
    case TINFER_S_INFLIGHT_LM: return x->p.inflight_lm;
    case TINFER_S_ATTN_CHUNKS: return x->p.n_chunks_override;
  }
  return -1;
}

tinfer_status tinfer_set_timeout_ns(tinfer_ctx* x, long long ns) {
  if (!x || ns <= 0) return TINFER_ERR_INVALID_ARG;
  x->p.timeout_ns = ns;
  if (x->gexec) { cudaGraphExecDestroy(x->gexec); x->gexec = nullptr; }
  return TINFER_OK;
}

tinfer_status tinfer_debug_withhold_results(tinfer_ctx* x, int cta, int phase) {
  if (!x || cta >= x->p.grid) return TINFER_ERR_INVALID_ARG;
  if (x->cfg.exec_mode != TINFER_MEGAKERNEL) return TINFER_ERR_UNSUPPORTED;
  x->p.dbg_skip_cta = cta;
  x->p.dbg_skip_phase = phase;
  return TINFER_OK;
}

// ---------------------------------------------------------------- single operations

namespace {
struct OpScratch {
  int device = -1;
  uint8_t* mem = nullptr;
  float* slot_v = nullptr;
  int* slot_i = nullptr;
  int* slot_bad = nullptr;
  unsigned* ticket = nullptr;
  int* err = nullptr;
};
OpScratch g_op;

tinfer_status op_scratch() {
  int dev = 0;
  TRY_CUDA(cudaGetDevice(&dev));
  if (g_op.mem && g_op.device == dev) return TINFER_OK;
  const size_t bytes = 3 * 4096 + 256;
  TRY_CUDA(cudaMalloc(&g_op.mem, bytes));
  TRY_CUDA(cudaMemset(g_op.mem, 0, bytes));
  g_op.device = dev;
  g_op.slot_v = (float*)g_op.mem;
  g_op.slot_i = (int*)(g_op.mem + 4096);
  g_op.slot_bad = (int*)(g_op.mem + 8192);
  g_op.ticket = (unsigned*)(g_op.mem + 12288);
  g_op.err = (int*)(g_op.mem + 12288 + 64);
  return TINFER_OK;
}

int op_grid(int units) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return units < sms ? (units > 0 ? units : 1) : sms;
}
}  // namespace

tinfer_status tinfer_op_gemv(int fmt, int group, int scale_dtype, int rows, int cols,
                             const void* packed_dev, const float* x_dev, const float* gain_dev,
                             double rms_eps, const float* bias_dev, int epilogue, float* y_dev,
                             int32_t* argmax_dev, void* stream) {
  const size_t rb = packed_row_bytes(fmt, cols, group);
  if (rows <= 0 || rb == 0 || !packed_dev || !x_dev) return TINFER_ERR_INVALID_ARG;
  if (epilogue < TINFER_EPI_STORE || epilogue > TINFER_EPI_ARGMAX) return TINFER_ERR_INVALID_ARG;
  if (epilogue != TINFER_EPI_ARGMAX && !y_dev) return TINFER_ERR_INVALID_ARG;
  if (epilogue == TINFER_EPI_ARGMAX && !argmax_dev) return TINFER_ERR_INVALID_ARG;
  if (epilogue == TINFER_EPI_SWIGLU && rows % 2) return TINFER_ERR_INVALID_ARG;
  if (!seg_ok(fmt, cols)) return TINFER_ERR_UNSUPPORTED;
  if (gain_dev && (reinterpret_cast<uintptr_t>(gain_dev) & 15) != 0) return TINFER_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(packed_dev) & 15) != 0) return TINFER_ERR_INVALID_ARG;
  TRY(op_scratch());
  size_t need_slot = rb * 2;
  const int slot = need_slot <= SLOT_MIN ? SLOT_MIN : (int)align_up(need_slot, 1024);
  const int stages = 4;
  const int xs = (int)align_up((size_t)cols * 4, 128);
  const size_t smem = smem_for(stages, slot, xs);
  if (smem > 227 * 1024) return TINFER_ERR_UNSUPPORTED;
  TRY_CUDA(set_smem_op_gemv(smem));
  OpGemvParams q{};
  q.w = (const uint8_t*)packed_dev; q.rows = rows; q.cols = cols; q.rb = (int)rb;
  q.fmt = fmt; q.group = group; q.scale_bf16 = scale_dtype == TINFER_SCALE_BF16;
  q.x = x_dev; q.gain = gain_dev; q.eps = (float)rms_eps; q.bias = bias_dev; q.epi = epilogue;
  q.y = y_dev; q.argmax = argmax_dev;
  q.slot_v = g_op.slot_v; q.slot_i = g_op.slot_i; q.slot_bad = g_op.slot_bad; q.ticket = g_op.ticket;
  q.err = g_op.err; q.stages = stages; q.slot = slot; q.timeout_ns = DEFAULT_TIMEOUT_NS;
  const int quantum = epilogue == TINFER_EPI_SWIGLU ? 2 : 1;
  int grid = op_grid(rows / quantum);
  if (epilogue != TINFER_EPI_ARGMAX || seg_info(fmt, cols).nseg > 1) {
    // enough CTAs that each one's row results fit its shared-memory buffer
    const int nseg = seg_info(fmt, cols).nseg;
    const int per = ROWV_MAX / nseg - quantum;
    const int need = (rows + per - 1) / per;
    if (need > grid) grid = need;
  }
  if (epilogue == TINFER_EPI_ARGMAX && grid > 1024) return TINFER_ERR_UNSUPPORTED;  // argmax slots
  cudaStream_t st = (cudaStream_t)stream;
  TRY_CUDA(launch_op_gemv(q, grid, smem, st));
  if (epilogue == TINFER_EPI_ARGMAX) {
    TRY_CUDA(cudaStreamSynchronize(st));
    int w = 0;
    TRY_CUDA(cudaMemcpy(&w, g_op.err, 4, cudaMemcpyDeviceToHost));
    if (w) {
      TRY_CUDA(cudaMemset(g_op.err, 0, 4));
      TRY_CUDA(cudaMemset(g_op.ticket, 0, 4));
      return status_of_word(w);
    }
  }
  return TINFER_OK;
}

tinfer_status tinfer_op_attention(int nq, int nkv, int d, int max_ctx, double theta, int pos,
                                  int n_chunks, const float* qkv_dev, void* k_layer_dev,
                                  void* v_layer_dev, float* out_dev, float* part_m_dev,
                                  float* part_l_dev, float* part_o_dev, void* stream) {
  if (nq <= 0 || nkv <= 0 || nq % nkv || nq / nkv > G_MAX || d % 8 || d > D_MAX || max_ctx <= 0)
    return TINFER_ERR_INVALID_ARG;
  if (pos < 0 || pos >= max_ctx || !qkv_dev || !k_layer_dev || !v_layer_dev || !out_dev)
    return TINFER_ERR_INVALID_ARG;
  const bool user_parts = part_m_dev || part_l_dev || part_o_dev;
  if (user_parts && (!part_m_dev || !part_l_dev || !part_o_dev || n_chunks <= 0))
    return TINFER_ERR_INVALID_ARG;
  TRY(op_scratch());
  const int slot = SLOT_MIN;
  int tmax = slot / (2 * d);
  if (tmax > T_MAX) tmax = T_MAX;
  const int grid = op_grid(1 << 30);
  int nch = n_chunks;
  if (nch <= 0) nch = nch_capacity(pos + 1, nkv, d, grid, slot);
  if (nch > T_MAX || (pos + nch) / nch > tmax) return TINFER_ERR_UNSUPPORTED;  // ceil((pos+1)/nch)
  cudaStream_t st = (cudaStream_t)stream;
  std::vector<float2> rt;
  rope_table(rt, pos + 1, d, theta);
  float2* rope = nullptr;
  float* parts = nullptr;
  unsigned* tickets = nullptr;
  tinfer_status rc = TINFER_OK;
  do {
    if ((rc = from_cuda(cudaMalloc(&rope, sizeof(float2) * rt.size()))) != TINFER_OK) break;
    if ((rc = from_cuda(cudaMemcpy(rope, rt.data(), sizeof(float2) * rt.size(), cudaMemcpyHostToDevice))) != TINFER_OK) break;
    if ((rc = from_cuda(cudaMalloc(&tickets, 4 * nkv))) != TINFER_OK) break;
    if ((rc = from_cuda(cudaMemset(tickets, 0, 4 * nkv))) != TINFER_OK) break;
    OpAttnParams q{};
    if (!user_parts) {
      if ((rc = from_cuda(cudaMalloc(&parts, (size_t)nq * nch * (d + 2) * 4))) != TINFER_OK) break;
      q.part_m = parts; q.part_l = parts + (size_t)nq * nch; q.part_o = parts + (size_t)2 * nq * nch;
    } else {
      q.part_m = part_m_dev; q.part_l = part_l_dev; q.part_o = part_o_dev;
    }
    q.qkv = qkv_dev; q.kc = (uint16_t*)k_layer_dev; q.vc = (uint16_t*)v_layer_dev; q.rope = rope;
    q.nch_cap = nch; q.tickets = tickets; q.out = out_dev;
    q.nq = nq; q.nkv = nkv; q.d = d; q.max_ctx = max_ctx; q.pos = pos; q.n_chunks = nch;
    q.err = g_op.err; q.stages = 4; q.slot = slot; q.timeout_ns = DEFAULT_TIMEOUT_NS;
    const size_t smem = smem_for(4, slot, 0);
    if ((rc = from_cuda(set_smem_op_attention(smem))) != TINFER_OK) break;
    if ((rc = from_cuda(launch_op_attention(q, grid, smem, st))) != TINFER_OK) break;
    if ((rc = from_cuda(cudaStreamSynchronize(st))) != TINFER_OK) break;
    int w = 0;
    if ((rc = from_cuda(cudaMemcpy(&w, g_op.err, 4, cudaMemcpyDeviceToHost))) != TINFER_OK) break;
    if (w) { cudaMemset(g_op.err, 0, 4); rc = status_of_word(w); }
  } while (0);
  if (rope) cudaFree(rope);
  if (parts) cudaFree(parts);
  if (tickets) cudaFree(tickets);
  return rc;
}

tinfer_status tinfer_op_gemv_batch(int fmt, int group, int scale_dtype, int rows, int cols, int m,
                                   const void* packed_dev, const float* x_dev, const float* bias_dev,
                                   int epilogue, float* y_dev, void* stream) {
  const size_t rb = packed_row_bytes(fmt, cols, group);
  if (rows <= 0 || rb == 0 || !packed_dev || !x_dev || !y_dev) return TINFER_ERR_INVALID_ARG;
  if (epilogue != TINFER_EPI_STORE && epilogue != TINFER_EPI_RESIDUAL) return TINFER_ERR_INVALID_ARG;
  if (m != 1 && m != 2 && m != 4 && m != 8) return TINFER_ERR_UNSUPPORTED;
  for (const void* ptr : {packed_dev, (const void*)x_dev})
    if (reinterpret_cast<uintptr_t>(ptr) & 15) return TINFER_ERR_INVALID_ARG;
  // segments: a lane holds 8 / m units of 8 inputs of every vector, so a segment spans at most
  // 2048 / m inputs; int4 segments hold whole groups of a lane's 8 / m consecutive words
  int nseg = 1;
  while (nseg < NCW && cols / nseg > 2048 / m) nseg *= 2;
  const int ks = cols / nseg, unit = fmt == TINFER_INT4 ? 8 * (8 / m) : 8;
  if (cols % nseg || ks > 2048 / m || ks % unit) return TINFER_ERR_UNSUPPORTED;
  int dev = 0, sms = 0;
  TRY_CUDA(cudaGetDevice(&dev));
  TRY_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  TRY(op_scratch());
  OpGemvMParams q{};
  q.w = (const uint8_t*)packed_dev; q.rows = rows; q.cols = cols; q.rb = (int)rb;
  q.fmt = fmt; q.group = group; q.scale_bf16 = scale_dtype == TINFER_SCALE_BF16;
  q.m = m; q.nseg = nseg; q.x = x_dev; q.bias = bias_dev; q.y = y_dev;
  q.residual = epilogue == TINFER_EPI_RESIDUAL; q.err = g_op.err; q.timeout_ns = DEFAULT_TIMEOUT_NS;
  q.stages = 4;
  q.slot = (int)std::max<size_t>(SLOT_MIN, align_up(rb * (size_t)(NCW / nseg), 1024));
  size_t smem = smem_for(q.stages, q.slot, (int)align_up((size_t)m * cols * 4, 128));
  while (smem > 227 * 1024 && q.stages > 2) smem = smem_for(--q.stages, q.slot, (int)align_up((size_t)m * cols * 4, 128));
  if (smem > 227 * 1024) return TINFER_ERR_UNSUPPORTED;
  // enough CTAs that one CTA's row results fit its shared row buffer
  int grid = rows < sms ? rows : sms;
  const int per = std::max(ROWV_MAX, m * cols) / (nseg * m) - 1;  // row results: the larger buffer
  if (per < 1) return TINFER_ERR_UNSUPPORTED;
  if ((rows + per - 1) / per > grid) grid = (rows + per - 1) / per;
  TRY_CUDA(set_smem_op_gemv_m(fmt, m, smem));
  TRY_CUDA(launch_op_gemv_m(q, grid, smem, (cudaStream_t)stream));
  return TINFER_OK;
}

size_t tinfer_moe_packed_bytes(int fmt, int group, int n_experts, int hidden, int ffn_e, int which) {
  if (n_experts <= 0) return 0;
  const size_t rbh = packed_row_bytes(fmt, hidden, group), rbf = packed_row_bytes(fmt, ffn_e, group);
  if (!rbh || !rbf) return 0;
  return which == 0 ? (size_t)n_experts * 2 * ffn_e * rbh : (size_t)n_experts * hidden * rbf;
}

tinfer_status tinfer_pack_moe(int fmt, int group, int scale_dtype, int n_experts, int hidden, int ffn_e,
                              const void* wg, const void* sg, const void* wu, const void* su,
                              const void* wd, const void* sd, void* gu_packed_dev, void* down_packed_dev,
                              void* stream) {
  (void)scale_dtype;
  if (!tinfer_moe_packed_bytes(fmt, group, n_experts, hidden, ffn_e, 0) || !gu_packed_dev || !down_packed_dev)
    return TINFER_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(gu_packed_dev) & 15) || (reinterpret_cast<uintptr_t>(down_packed_dev) & 15))
    return TINFER_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  // every expert's gate rows land on even packed rows and its up rows on odd ones: expert e's row j
  // is stacked row e * ffn_e + j, packed row 2 (e * ffn_e + j) (+ 1)
  TRY(pack_one(fmt, group, wg, sg, n_experts * ffn_e, hidden, (uint8_t*)gu_packed_dev, 2, 0, st));
  TRY(pack_one(fmt, group, wu, su, n_experts * ffn_e, hidden, (uint8_t*)gu_packed_dev, 2, 1, st));
  TRY(pack_one(fmt, group, wd, sd, n_experts * hidden, ffn_e, (uint8_t*)down_packed_dev, 1, 0, st));
  return TINFER_OK;
}

tinfer_status tinfer_op_moe(int fmt, int group, int scale_dtype, int n_experts, int top_k, int hidden,
                            int ffn_e, const void* gu_packed_dev, const void* down_packed_dev,
                            const int32_t* ids_dev, const float* weights_dev, const float* x_dev,
                            float* h_dev, float* y_dev, int accumulate, int32_t* status_dev,
                            void* stream) {
  if (!tinfer_moe_packed_bytes(fmt, group, n_experts, hidden, ffn_e, 0)) return TINFER_ERR_INVALID_ARG;
  if (top_k < 1 || top_k > n_experts || NCW % top_k != 0) return TINFER_ERR_UNSUPPORTED;
  if (!gu_packed_dev || !down_packed_dev || !ids_dev || !weights_dev || !x_dev || !h_dev || !y_dev)
    return TINFER_ERR_INVALID_ARG;
  for (const void* ptr : {gu_packed_dev, down_packed_dev, (const void*)x_dev, (const void*)h_dev, (const void*)y_dev})
    if (reinterpret_cast<uintptr_t>(ptr) & 15) return TINFER_ERR_INVALID_ARG;
  if (accumulate != 0 && accumulate != 1) return TINFER_ERR_INVALID_ARG;
  // the gate/up GEMV reads rows of `hidden` inputs; the down projection gives each expert one warp
  // group and a segment of ffn_e inputs, whose activations a lane keeps in registers
  const int E = fmt == TINFER_INT4 ? 32 : 8;
  if (!seg_ok(fmt, hidden) || ffn_e % E || ffn_e / E > 32 * (fmt == TINFER_INT4 ? 2 : 8))
    return TINFER_ERR_UNSUPPORTED;
  int nchl = 4;
  if (fmt == TINFER_BF16) {
    const int need = std::max((seg_info(0, hidden).chs + 31) / 32, (ffn_e / 8 + 31) / 32);
    nchl = need <= 4 ? 4 : 8;
  }
  int dev = 0, sms = 0;
  TRY_CUDA(cudaGetDevice(&dev));
  TRY_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  TRY(op_scratch());
  OpMoeParams q{};
  q.gu = (const uint8_t*)gu_packed_dev; q.down = (const uint8_t*)down_packed_dev;
  q.ids = ids_dev; q.weights = weights_dev; q.x = x_dev; q.h = h_dev; q.y = y_dev; q.status = status_dev;
  q.n_experts = n_experts; q.k = top_k; q.hidden = hidden; q.ffn_e = ffn_e;
  q.rb_h = (int)packed_row_bytes(fmt, hidden, group); q.rb_f = (int)packed_row_bytes(fmt, ffn_e, group);
  q.fmt = fmt; q.group = group; q.scale_bf16 = scale_dtype == TINFER_SCALE_BF16; q.nchl = nchl;
  q.accumulate = accumulate; q.err = g_op.err; q.timeout_ns = DEFAULT_TIMEOUT_NS;
  cudaStream_t st = (cudaStream_t)stream;
  if (status_dev) TRY_CUDA(cudaMemsetAsync(status_dev, 0, 4, st));
  // rows of one CTA's share must fit the shared row-result buffer
  const long long rows_a = ((long long)top_k * 2 * ffn_e + sms - 1) / sms + 2, rows_b = (hidden + sms - 1) / sms + 1;
  if (rows_a * seg_info(fmt, hidden).nseg > ROWV_MAX || rows_b * top_k > ROWV_MAX) return TINFER_ERR_UNSUPPORTED;
  // gate/up: 4 stages of 32 KB (several rows of `hidden` inputs each)
  q.stages = 4;
  q.slot = (int)std::max<size_t>(SLOT_MIN, align_up((size_t)q.rb_h * 2, 1024));
  size_t smem = smem_for(q.stages, q.slot, (int)align_up((size_t)hidden * 4, 128));
  if (smem > 227 * 1024) return TINFER_ERR_UNSUPPORTED;
  TRY_CUDA(set_smem_op_moe(fmt, nchl, 0, smem));
  TRY_CUDA(launch_op_moe(q, 0, sms, smem, st));
  // down: 3 stages, each holding a few rows of every chosen expert
  q.stages = 3;
  q.slot = (int)std::max<size_t>(48 * 1024, align_up((size_t)top_k * q.rb_f * (NCW / top_k), 1024));
  smem = smem_for(q.stages, q.slot, (int)align_up((size_t)top_k * ffn_e * 4, 128));
  if (smem > 227 * 1024) return TINFER_ERR_UNSUPPORTED;
  TRY_CUDA(set_smem_op_moe(fmt, nchl, 1, smem));
  TRY_CUDA(launch_op_moe(q, 1, sms, smem, st));
  return TINFER_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------- attention without allocation
// The scratch of tinfer_op_attention_noalloc: a fixed array in the library's device image, so that
// the call never allocates. Layout: [0, 256) error word; [256, 1280) merge tickets (one word per KV
// head); [1280, 2048) the cos/sin row of pos; [2048, end) chunk partials m, l, o.
static __device__ __align__(256) unsigned char g_noalloc_scratch[TINFER_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr size_t NA_ERR = 0, NA_TICKETS = 256, NA_ROPE = 1280, NA_PARTS = 2048;

// Device address of the scratch array, looked up once per device (with that device current) and
// kept; later calls on the device only read the table.
tinfer_status noalloc_scratch(unsigned char** base) {
  static unsigned char* addr[64] = {};
  static std::mutex mu;
  int dev = 0;
  TRY_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return TINFER_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return from_cuda(e);
    addr[dev] = static_cast<unsigned char*>(p);
  }
  *base = addr[dev];
  return TINFER_OK;
}
}  // namespace

extern "C" tinfer_status tinfer_op_attention_noalloc(int nq, int nkv, int d, int max_ctx,
                                                     double theta, int pos, int n_chunks,
                                                     const float* qkv_dev, void* k_layer_dev,
                                                     void* v_layer_dev, float* out_dev,
                                                     void* stream) {
  if (nq <= 0 || nkv <= 0 || nq % nkv || nq / nkv > G_MAX || d % 8 || d > D_MAX || max_ctx <= 0)
    return TINFER_ERR_INVALID_ARG;
  if (pos < 0 || pos >= max_ctx || !qkv_dev || !k_layer_dev || !v_layer_dev || !out_dev)
    return TINFER_ERR_INVALID_ARG;
  const int slot = SLOT_MIN;
  int tmax = slot / (2 * d);
  if (tmax > T_MAX) tmax = T_MAX;
  const int grid = op_grid(1 << 30);
  int nch = n_chunks;
  if (nch <= 0) nch = nch_capacity(pos + 1, nkv, d, grid, slot);
  if (nch > T_MAX || (pos + nch) / nch > tmax) return TINFER_ERR_UNSUPPORTED;  // ceil((pos+1)/nch)
  // the fixed scratch bounds the problem: tickets and partials must fit their regions
  const size_t part_floats = (size_t)nq * nch * (d + 2);
  if ((size_t)nkv * 4 > NA_ROPE - NA_TICKETS || part_floats * 4 > TINFER_NOALLOC_SCRATCH_BYTES - NA_PARTS)
    return TINFER_ERR_UNSUPPORTED;
  unsigned char* base = nullptr;
  TRY(noalloc_scratch(&base));
  cudaStream_t st = (cudaStream_t)stream;

  // cos/sin of position pos only (same formula and rounding as the engine's table): a one-row
  // table whose first row is position pos
  const int half = d / 2;
  float2 row[D_MAX / 2];
  for (int i = 0; i < half; ++i) {
    const double ang = (double)pos * std::pow(theta, -2.0 * (double)i / (double)d);
    row[i] = make_float2((float)std::cos(ang), (float)std::sin(ang));
  }
  TRY_CUDA(cudaMemsetAsync(base, 0, NA_ROPE, st));  // error word and tickets start at zero
  TRY_CUDA(cudaMemcpyAsync(base + NA_ROPE, row, sizeof(float2) * half, cudaMemcpyHostToDevice, st));

  float* parts = reinterpret_cast<float*>(base + NA_PARTS);
  OpAttnParams q{};
  q.qkv = qkv_dev; q.kc = (uint16_t*)k_layer_dev; q.vc = (uint16_t*)v_layer_dev;
  q.rope = reinterpret_cast<const float2*>(base + NA_ROPE);
  q.rope_pos0 = pos;
  q.part_m = parts; q.part_l = parts + (size_t)nq * nch; q.part_o = parts + (size_t)2 * nq * nch;
  q.nch_cap = nch; q.tickets = reinterpret_cast<unsigned*>(base + NA_TICKETS); q.out = out_dev;
  q.nq = nq; q.nkv = nkv; q.d = d; q.max_ctx = max_ctx; q.pos = pos; q.n_chunks = nch;
  q.err = reinterpret_cast<int*>(base + NA_ERR); q.stages = 4; q.slot = slot;
  q.timeout_ns = DEFAULT_TIMEOUT_NS;
  const size_t smem = smem_for(4, slot, 0);
  TRY_CUDA(set_smem_op_attention(smem));
  TRY_CUDA(launch_op_attention(q, grid, smem, st));
  TRY_CUDA(cudaStreamSynchronize(st));
  int w = 0;
  TRY_CUDA(cudaMemcpy(&w, base + NA_ERR, 4, cudaMemcpyDeviceToHost));
  return w ? status_of_word(w) : TINFER_OK;
}
