// kernels.h -- launch wrappers of kernels.cu, used by the host side of the engine (api.cu).
#pragma once
#include <cuda_runtime.h>

#include "engine.h"

namespace tinfer {

struct OpGemvParams {
  const uint8_t* w;
  int rows, cols, rb;
  int fmt, group, scale_bf16;
  const float* x;
  const float* gain;
  float eps;
  const float* bias;
  int epi;
  float* y;
  int* argmax;
  float* slot_v;
  int* slot_i;
  int* slot_bad;
  unsigned* ticket;
  int* err;
  int stages, slot;
  long long timeout_ns;
};

struct OpAttnParams {
  const float* qkv;
  uint16_t* kc;
  uint16_t* vc;
  const float2* rope;
  int rope_pos0;  // position of the table's first row (0: the full table)
  float* part_m;
  float* part_l;
  float* part_o;
  int nch_cap;
  unsigned* tickets;
  float* out;
  int nq, nkv, d, max_ctx, pos, n_chunks;
  int* err;
  int stages, slot;
  long long timeout_ns;
};

// The gathered-expert MLP (two kernels: gate/up with SwiGLU over the chosen experts' rows, then the
// down projections with the weighted sum).
struct OpMoeParams {
  const uint8_t* gu;      // packed gate/up rows of every expert, [n_experts][2 ffn_e] rows of rb_h bytes
  const uint8_t* down;    // packed down rows of every expert, [n_experts][hidden] rows of rb_f bytes
  const int* ids;         // [k] chosen experts
  const float* weights;   // [k] their routing weights
  const float* x;         // [hidden]
  float* h;               // [k][ffn_e] SwiGLU outputs of the chosen experts
  float* y;               // [hidden]
  int* status;            // may be null: set to 1 when an id was outside [0, n_experts)
  int n_experts, k, hidden, ffn_e, rb_h, rb_f;
  int fmt, group, scale_bf16, nchl;
  int accumulate;         // 0: y = MLP(x); 1: y += MLP(x)
  int* err;
  int stages, slot;
  long long timeout_ns;
};
cudaError_t launch_op_moe(const OpMoeParams& q, int phase, int grid, size_t smem, cudaStream_t st);

// GEMV over a batch of m activation vectors (op_gemv_m_kernel).
struct OpGemvMParams {
  const uint8_t* w;
  int rows, cols, rb;
  int fmt, group, scale_bf16;
  int m, nseg;
  const float* x;      // [m][cols]
  const float* bias;   // [rows] or null
  float* y;            // [m][rows]
  int residual;
  int* err;
  int stages, slot;
  long long timeout_ns;
};
cudaError_t launch_op_gemv_m(const OpGemvMParams& q, int grid, size_t smem, cudaStream_t st);
cudaError_t set_smem_op_gemv_m(int fmt, int m, size_t bytes);
cudaError_t set_smem_op_moe(int fmt, int nchl, int phase, size_t bytes);

cudaError_t launch_megakernel(const StepParams& p, size_t smem, cudaStream_t st);
cudaError_t launch_phase(const StepParams& p, int k, size_t smem, cudaStream_t st, bool pdl);
cudaError_t launch_begin(int* step_dev, int token, const int* token_dev, int pos, int V, int* err,
                         int* err_host, cudaStream_t st);
const void* begin_kernel_fn();
cudaError_t launch_op_gemv(const OpGemvParams& q, int grid, size_t smem, cudaStream_t st);
cudaError_t launch_op_attention(const OpAttnParams& q, int grid, size_t smem, cudaStream_t st);
cudaError_t set_smem_mega(size_t bytes, int fmt, int nchl);
cudaError_t set_smem_phase(size_t bytes, int fmt, int nchl);
cudaError_t set_smem_op_gemv(size_t bytes);
cudaError_t set_smem_op_attention(size_t bytes);
cudaError_t megakernel_occupancy(int* blocks_per_sm, size_t smem, int fmt, int nchl);
cudaError_t phase_occupancy(int* blocks_per_sm, size_t smem, int fmt, int nchl);
size_t smem_for(int stages, int slot, int xs_bytes);
size_t static_smem_mega();  // static shared memory of the persistent kernel, with a margin

cudaError_t launch_pack_rows(uint8_t* dst, int dst_rb, int dst_step, int dst_first, int rows,
                             const uint8_t* w, int w_bytes, const uint8_t* s, int s_bytes,
                             cudaStream_t st);
cudaError_t launch_unpack_rows(const uint8_t* src, int src_rb, int src_step, int src_first, int rows,
                               uint8_t* w, int w_bytes, uint8_t* s, int s_bytes, cudaStream_t st);
cudaError_t launch_bf16_to_f32(const uint16_t* in, float* out, int n, cudaStream_t st);
cudaError_t launch_transpose_u16(const uint16_t* in, int rows, int cols, uint16_t* out, cudaStream_t st);
cudaError_t launch_f32_to_bf16(const float* in, uint16_t* out, int n, cudaStream_t st);

}  // namespace tinfer
