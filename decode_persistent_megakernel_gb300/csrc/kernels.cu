// kernels.cu -- the kernels of the engine and their launch wrappers.
//
// The step kernels themselves are in megakernel.cuh (instantiated by mega_bf16.cu, mega_int4.cu):
//   decode_megakernel    one cooperative launch per step: every phase of every layer; each phase
//                        waits for the stamped results of the one before it (no grid barrier), the
//                        weight stream running ahead of them
//   decode_phase_kernel  one phase of one layer; the CUDA-graph path chains 5 L + 1 of them with
//                        programmatic dependent launch so that the next kernel's weight prefetch
//                        starts while the current one finishes
//   op_gemv_kernel, op_attention_kernel   single operations for the per-kernel parity tests
//   pack / unpack kernels                 canonical <-> streaming layout
#include <cuda_runtime.h>

#include <mutex>

#include "engine.h"
#include "kernels.h"
// Diagnostic 549 ("used before its value is set") is a false positive in the batched GEMV
// (gemv_rows_m): its reduction window reads rl[rr] only for rr < filled, the slots written since the
// last flush. This is the only unit that instantiates it.
#pragma nv_diag_suppress 549
#include "step.cuh"
#pragma nv_diag_default 549

namespace tinfer {

__global__ void decode_begin_kernel(int* step_dev, int token, const int* token_dev, int pos, int V,
                                    int* err, int* err_host) {
  const int tok = token_dev ? *token_dev : token;
  if ((tok < 0 || tok >= V) && ld_volatile_int(err) == 0) raise_error(err, err_host, EW_BADTOKEN);
  step_dev[0] = tok;
  step_dev[1] = pos;
}

// ------------------------------------------------------------------------------ single operations

__global__ void __launch_bounds__(NTHREADS, 1) op_gemv_kernel(const __grid_constant__ OpGemvParams q) {
  extern __shared__ __align__(128) unsigned char smem[];
  Pipe pp;
  pipe_init(pp, smem, q.stages, q.slot, q.timeout_ns, q.err, nullptr);
  pipe_setup(pp);
  __syncthreads();
  const GemvDesc g{q.w, q.rows, q.cols, q.rb, q.fmt, q.group, q.scale_bf16, q.epi == EK_SWIGLU ? 2 : 1};
  const RowSplit rs = row_split(g, blockIdx.x, gridDim.x, q.slot);
  const int tid = threadIdx.x;
  if (tid >= NCT) {
    if (tid == NCT) {
      bool dead = false;
      produce_rows(pp, g, rs, policy_evict_first(), dead);
      prod_drain(pp);
    }
  } else {
    GemvPlan pl;
    pl.g = g;
    pl.rs = rs;
    pl.src = ActSrc{};
    pl.src.xf = q.x; pl.src.gf = q.gain; pl.src.eps = q.eps; pl.src.n = q.cols;
    pl.epi = Epi{q.epi, q.y, q.bias, nullptr, 0u, 0};
    Best best{-CUDART_INF_F, 0x7FFFFFFF, 0};
    gemv_consume_any(pp, pl, best, tid, nullptr);
    if (q.epi == EK_ARGMAX) {
      const Best cb = best_block_reduce(best, pp.ms, tid);
      argmax_publish(cb, q.slot_v, q.slot_i, q.slot_bad, q.ticket, gridDim.x, blockIdx.x, q.argmax,
                     q.err, nullptr, pp.ms, tid);
    }
    if (tid == 0) *reinterpret_cast<volatile int*>(&pp.ms->cons_done) = 1;
  }
  __syncthreads();
}

__global__ void __launch_bounds__(NTHREADS, 1) op_attention_kernel(const __grid_constant__ OpAttnParams q) {
  extern __shared__ __align__(128) unsigned char smem[];
  Pipe pp;
  pipe_init(pp, smem, q.stages, q.slot, q.timeout_ns, q.err, nullptr);
  pipe_setup(pp);
  __syncthreads();
  AttnArgs A;
  A.qkv = q.qkv; A.kc = q.kc; A.vc = q.vc; A.rope = q.rope; A.rope_pos0 = q.rope_pos0;
  A.part_m = q.part_m; A.part_l = q.part_l; A.part_o = q.part_o; A.nch_cap = q.nch_cap;
  A.tickets = q.tickets; A.out = q.out;
  A.nq = q.nq; A.nkv = q.nkv; A.d = q.d; A.max_ctx = q.max_ctx; A.pos = q.pos;
  const AttnSplit sp = attn_split(q.pos, q.nkv, q.d, gridDim.x, q.slot, q.n_chunks);
  const int units = q.nkv * sp.nch;
  const int tid = threadIdx.x;
  if (tid >= NCT) {
    if (tid == NCT) {
      bool dead = false;
      const uint64_t pol = policy_evict_normal();
      for (int u = blockIdx.x; u < units; u += gridDim.x) produce_attn_unit(pp, A, u / sp.nch, u % sp.nch, sp, pol, dead);
      prod_drain(pp);
    }
  } else {
    for (int u = blockIdx.x; u < units; u += gridDim.x)
      if (!attn_unit(pp, A, sp, u / sp.nch, u % sp.nch, tid)) break;
    if (tid == 0) *reinterpret_cast<volatile int*>(&pp.ms->cons_done) = 1;
  }
  __syncthreads();
}

// GEMV over a batch of MV vectors (the verify shape): the same ring and producer as the one-vector
// GEMV, the batched consumer gemv_rows_m.
template <int FMT, int MV>
__global__ void __launch_bounds__(NTHREADS, 1) op_gemv_m_kernel(const __grid_constant__ OpGemvMParams q) {
  extern __shared__ __align__(128) unsigned char smem[];
  Pipe pp;
  pipe_init(pp, smem, q.stages, q.slot, q.timeout_ns, q.err, nullptr);
  pipe_setup(pp);
  __syncthreads();
  const GemvDesc g{q.w, q.rows, q.cols, q.rb, q.fmt, q.group, q.scale_bf16, 1};
  RowSplit rs = row_split(g, blockIdx.x, gridDim.x, q.slot);
  const int wg = NCW / q.nseg;
  int fit = q.slot / q.rb;
  if (fit > NR_MAX) fit = NR_MAX;
  rs.nr = fit - fit % wg;
  const int tid = threadIdx.x;
  if (tid >= NCT) {
    if (tid == NCT) {
      bool dead = false;
      produce_rows(pp, g, rs, policy_evict_first(), dead);
      prod_drain(pp);
    }
  } else {
    gemv_rows_m<FMT, MV>(pp, g, rs, GemvMArgs{q.x, q.y, q.bias, q.residual, q.nseg}, tid);
    if (tid == 0) *reinterpret_cast<volatile int*>(&pp.ms->cons_done) = 1;
  }
  __syncthreads();
}

static const void* gemv_m_fn(int fmt, int m) {
  switch (fmt * 16 + m) {
    case 1: return (const void*)op_gemv_m_kernel<0, 1>;
    case 2: return (const void*)op_gemv_m_kernel<0, 2>;
    case 4: return (const void*)op_gemv_m_kernel<0, 4>;
    case 8: return (const void*)op_gemv_m_kernel<0, 8>;
    case 17: return (const void*)op_gemv_m_kernel<1, 1>;
    case 18: return (const void*)op_gemv_m_kernel<1, 2>;
    case 20: return (const void*)op_gemv_m_kernel<1, 4>;
    case 24: return (const void*)op_gemv_m_kernel<1, 8>;
  }
  return nullptr;
}

// ------------------------------------------------------------------------------ gathered experts

// The chosen expert ids in shared memory; an id outside [0, n_experts) reads expert 0 and is
// reported through q.status (the kernels never address outside the packed experts).
__device__ __forceinline__ void moe_load_ids(const OpMoeParams& q, int* s_ids) {
  if (threadIdx.x < (unsigned)q.k) {
    int e = q.ids[threadIdx.x];
    if (e < 0 || e >= q.n_experts) {
      if (q.status) atomicExch(q.status, 1);
      e = 0;
    }
    s_ids[threadIdx.x] = e;
  }
}

// Gate/up of the chosen experts ("One launch per token", "The same trick, sparser: a 64-expert MoE":
// one kernel does the gated/up SwiGLU for the selected experts gathered by id). The matrix is the k
// experts' interleaved gate/up rows one after another, k * 2 ffn_e "virtual" rows; the producer
// gathers each stage from the experts its rows belong to (two bulk copies when a stage straddles
// two experts), and the consumers run the ordinary GEMV with the SwiGLU epilogue into h [k][ffn_e].
template <int FMT, int NCHL>
__global__ void __launch_bounds__(NTHREADS, 1) op_moe_gu_kernel(const __grid_constant__ OpMoeParams q) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ int s_ids[G_MAX];
  Pipe pp;
  pipe_init(pp, smem, q.stages, q.slot, q.timeout_ns, q.err, nullptr);
  pipe_setup(pp);
  moe_load_ids(q, s_ids);
  __syncthreads();
  const int per = 2 * q.ffn_e;  // virtual rows per expert
  const GemvDesc g{nullptr, q.k * per, q.hidden, q.rb_h, q.fmt, q.group, q.scale_bf16, 2};
  const RowSplit rs = row_split(g, blockIdx.x, gridDim.x, q.slot);
  const int tid = threadIdx.x;
  if (tid >= NCT) {
    if (tid == NCT) {
      bool dead = false;
      const uint64_t pol = policy_evict_first();
      for (int s0 = rs.r0; s0 < rs.r1 && !dead; s0 += rs.nr) {
        const int nrs = min(rs.nr, rs.r1 - s0);
        uint32_t dst, bar;
        if (!prod_open(pp, (uint32_t)(nrs * q.rb_h), dst, bar, dead)) break;
        for (int v = s0; v < s0 + nrs;) {
          const int i = v / per, r = v - i * per, n = min(s0 + nrs - v, per - r);
          const uint8_t* src = q.gu + ((size_t)s_ids[i] * per + r) * q.rb_h;
          bulk_g2s(dst + (uint32_t)(v - s0) * q.rb_h, src, (uint32_t)(n * q.rb_h), bar, pol);
          v += n;
        }
        pipe_advance(pp);
      }
      prod_drain(pp);
    }
  } else {
    GemvPlan pl;
    pl.g = g;
    pl.rs = rs;
    pl.src = ActSrc{};
    pl.src.xf = q.x;
    pl.src.n = q.hidden;
    pl.epi = Epi{EK_SWIGLU, q.h, nullptr, nullptr, 0u, 0};
    Best best{-CUDART_INF_F, 0x7FFFFFFF, 0};
    if (FMT == 1) gemv_rows<1, 2>(pp, pl, best, tid, nullptr);
    else gemv_rows<0, NCHL>(pp, pl, best, tid, nullptr);
    if (tid == 0) *reinterpret_cast<volatile int*>(&pp.ms->cons_done) = 1;
  }
  __syncthreads();
}

// Down projections of the chosen experts and their weighted sum (the page's second kernel). Row o
// of the gathered matrix is the concatenation of the k experts' row o; a stage holds its rows
// expert after expert (segment-major: one bulk copy per expert), warp w takes expert w's segment
// with its SwiGLU outputs h[w] in registers, and the epilogue adds the k segment sums weighted by
// the routing weights, in order.
template <int FMT, int NCHL>
__global__ void __launch_bounds__(NTHREADS, 1) op_moe_down_kernel(const __grid_constant__ OpMoeParams q) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ int s_ids[G_MAX];
  Pipe pp;
  pipe_init(pp, smem, q.stages, q.slot, q.timeout_ns, q.err, nullptr);
  pipe_setup(pp);
  moe_load_ids(q, s_ids);
  __syncthreads();
  GemvDesc g{nullptr, q.hidden, q.k * q.ffn_e, q.k * q.rb_f, q.fmt, q.group, q.scale_bf16, 1};
  g.nsegs = q.k;
  g.rbs = q.rb_f;
  RowSplit rs = row_split(g, blockIdx.x, gridDim.x, q.slot);
  const int wg = NCW / q.k;
  int fit = q.slot / (q.k * q.rb_f);
  if (fit > NR_MAX) fit = NR_MAX;
  rs.nr = fit - fit % wg;
  const int tid = threadIdx.x;
  if (tid >= NCT) {
    if (tid == NCT) {
      bool dead = false;
      const uint64_t pol = policy_evict_first();
      for (int s0 = rs.r0; s0 < rs.r1 && !dead; s0 += rs.nr) {
        const int nrs = min(rs.nr, rs.r1 - s0);
        const uint32_t seg_bytes = (uint32_t)(nrs * q.rb_f);
        uint32_t dst, bar;
        if (!prod_open(pp, seg_bytes * (uint32_t)q.k, dst, bar, dead)) break;
        for (int i = 0; i < q.k; ++i)
          bulk_g2s(dst + (uint32_t)i * seg_bytes, q.down + ((size_t)s_ids[i] * q.hidden + s0) * q.rb_f,
                   seg_bytes, bar, pol);
        pipe_advance(pp);
      }
      prod_drain(pp);
    }
  } else {
    GemvPlan pl;
    pl.g = g;
    pl.rs = rs;
    pl.src = ActSrc{};
    pl.src.xf = q.h;
    pl.src.n = q.k * q.ffn_e;
    pl.epi = Epi{q.accumulate ? EK_RESIDUAL : EK_STORE, q.y, q.weights, nullptr, 0u, 0};
    Best best{-CUDART_INF_F, 0x7FFFFFFF, 0};
    if (FMT == 1) gemv_rows<1, 2, 4, true>(pp, pl, best, tid, nullptr);
    else gemv_rows<0, NCHL, 4, true>(pp, pl, best, tid, nullptr);
    if (tid == 0) *reinterpret_cast<volatile int*>(&pp.ms->cons_done) = 1;
  }
  __syncthreads();
}

static const void* moe_fn(int fmt, int nchl, int phase) {
  if (fmt == 1) return phase ? (const void*)op_moe_down_kernel<1, 2> : (const void*)op_moe_gu_kernel<1, 2>;
  switch (nchl) {
    case 4: return phase ? (const void*)op_moe_down_kernel<0, 4> : (const void*)op_moe_gu_kernel<0, 4>;
    case 8: return phase ? (const void*)op_moe_down_kernel<0, 8> : (const void*)op_moe_gu_kernel<0, 8>;
  }
  return nullptr;
}

// ------------------------------------------------------------------------------ packing

// dst row (r * dst_step + dst_first) of width dst_rb <- src row r: src_bytes bytes of w, then
// s_bytes bytes of scales, then zero padding.
__global__ void pack_rows_kernel(uint8_t* dst, int dst_rb, int dst_step, int dst_first, int rows,
                                 const uint8_t* w, int w_bytes, const uint8_t* s, int s_bytes) {
  for (int r = blockIdx.x; r < rows; r += gridDim.x) {
    uint8_t* o = dst + ((size_t)r * dst_step + dst_first) * dst_rb;
    const uint8_t* wr = w + (size_t)r * w_bytes;
    const uint8_t* sr = s ? s + (size_t)r * s_bytes : nullptr;
    for (int i = threadIdx.x; i < dst_rb; i += blockDim.x) {
      uint8_t v = 0;
      if (i < w_bytes) v = wr[i];
      else if (sr && i < w_bytes + s_bytes) v = sr[i - w_bytes];
      o[i] = v;
    }
  }
}

__global__ void unpack_rows_kernel(const uint8_t* src, int src_rb, int src_step, int src_first,
                                   int rows, uint8_t* w, int w_bytes, uint8_t* s, int s_bytes) {
  for (int r = blockIdx.x; r < rows; r += gridDim.x) {
    const uint8_t* in = src + ((size_t)r * src_step + src_first) * src_rb;
    for (int i = threadIdx.x; i < w_bytes + (s ? s_bytes : 0); i += blockDim.x) {
      if (i < w_bytes) w[(size_t)r * w_bytes + i] = in[i];
      else s[(size_t)r * s_bytes + i - w_bytes] = in[i];
    }
  }
}

// out[c][r] = in[r][c] for 16-bit elements (the packer's transposed down projection), 32 x 32
// tiles through shared memory.
__global__ void transpose_u16_kernel(const uint16_t* in, int rows, int cols, uint16_t* out) {
  __shared__ uint16_t t[32][33];
  const int r0 = blockIdx.y * 32, c0 = blockIdx.x * 32;
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int r = r0 + i, c = c0 + threadIdx.x;
    if (r < rows && c < cols) t[i][threadIdx.x] = in[(size_t)r * cols + c];
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int c = c0 + i, r = r0 + threadIdx.x;
    if (r < rows && c < cols) out[(size_t)c * rows + r] = t[threadIdx.x][i];
  }
}

__global__ void bf16_to_f32_kernel(const uint16_t* in, float* out, int n) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
    out[i] = __uint_as_float((uint32_t)in[i] << 16);
}

// exact inverse for values that came from bf16
__global__ void f32_to_bf16_kernel(const float* in, uint16_t* out, int n) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
    out[i] = (uint16_t)(__float_as_uint(in[i]) >> 16);
}

// ------------------------------------------------------------------------------ launch wrappers

// kernel instances of mega_bf16.cu / mega_int4.cu; kind 0: persistent kernel, 1: persistent kernel
// recording a timeline, 2: per-phase kernel, 3: persistent kernel with the token loop, 4: persistent
// kernel with the column-split down projection (bf16)
const void* step_kernel_bf16(int nchl, int kind);
const void* step_kernel_int4(int nchl, int kind);
static const void* step_fn(int fmt, int nchl, int kind) {
  return fmt == 1 ? step_kernel_int4(nchl, kind) : step_kernel_bf16(nchl, kind);
}

cudaError_t launch_megakernel(const StepParams& p, size_t smem, cudaStream_t st) {
  const void* fn = step_fn(p.m.fmt, p.m.nchl, p.m.ffn_split ? 4 : p.n_steps > 1 ? 3 : p.trace ? 1 : 0);
  if (!fn) return cudaErrorInvalidDeviceFunction;
  void* args[] = {const_cast<StepParams*>(&p)};
  return cudaLaunchCooperativeKernel(fn, dim3(p.grid), dim3(NTHREADS_MEGA), args, smem, st);
}

cudaError_t launch_phase(const StepParams& p, int k, size_t smem, cudaStream_t st, bool pdl) {
  const void* fn = step_fn(p.m.fmt, p.m.nchl, 2);
  if (!fn) return cudaErrorInvalidDeviceFunction;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(p.grid);
  cfg.blockDim = dim3(NTHREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  void* args[] = {const_cast<StepParams*>(&p), &k};
  return cudaLaunchKernelExC(&cfg, fn, args);
}

cudaError_t launch_begin(int* step_dev, int token, const int* token_dev, int pos, int V, int* err,
                         int* err_host, cudaStream_t st) {
  decode_begin_kernel<<<1, 1, 0, st>>>(step_dev, token, token_dev, pos, V, err, err_host);
  return cudaGetLastError();
}

const void* begin_kernel_fn() { return reinterpret_cast<const void*>(&decode_begin_kernel); }

cudaError_t launch_op_gemv(const OpGemvParams& q, int grid, size_t smem, cudaStream_t st) {
  op_gemv_kernel<<<grid, NTHREADS, smem, st>>>(q);
  return cudaGetLastError();
}

cudaError_t launch_op_attention(const OpAttnParams& q, int grid, size_t smem, cudaStream_t st) {
  op_attention_kernel<<<grid, NTHREADS, smem, st>>>(q);
  return cudaGetLastError();
}

// Raises (never lowers) a kernel's dynamic shared-memory limit; one limit per kernel and device.
static cudaError_t raise_limit(const void* fn, size_t bytes) {
  struct Entry {
    const void* fn;
    int dev;
    size_t bytes;
  };
  static Entry table[256];
  static int used = 0;
  static std::mutex mu;
  if (!fn) return cudaErrorInvalidDeviceFunction;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  Entry* hit = nullptr;
  for (int i = 0; i < used; ++i)
    if (table[i].fn == fn && table[i].dev == dev) hit = &table[i];
  if (hit && bytes <= hit->bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  if (hit) hit->bytes = bytes;
  else if (used < 256) table[used++] = Entry{fn, dev, bytes};
  return cudaSuccess;
}
cudaError_t set_smem_mega(size_t b, int fmt, int nchl) {
  for (int kind : {0, 1, 3, 4}) {
    const void* fn = step_fn(fmt, nchl, kind);
    if (!fn && kind == 4) continue;  // no column-split instance for int4
    const cudaError_t e = raise_limit(fn, b);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}
cudaError_t set_smem_phase(size_t b, int fmt, int nchl) { return raise_limit(step_fn(fmt, nchl, 2), b); }
cudaError_t set_smem_op_gemv(size_t b) { return raise_limit((const void*)op_gemv_kernel, b); }
cudaError_t set_smem_op_moe(int fmt, int nchl, int phase, size_t b) { return raise_limit(moe_fn(fmt, nchl, phase), b); }
cudaError_t set_smem_op_gemv_m(int fmt, int m, size_t b) { return raise_limit(gemv_m_fn(fmt, m), b); }
cudaError_t launch_op_gemv_m(const OpGemvMParams& q, int grid, size_t smem, cudaStream_t st) {
  const void* fn = gemv_m_fn(q.fmt, q.m);
  if (!fn) return cudaErrorInvalidDeviceFunction;
  void* args[] = {const_cast<OpGemvMParams*>(&q)};
  return cudaLaunchKernel(fn, dim3(grid), dim3(NTHREADS), args, smem, st);
}
cudaError_t launch_op_moe(const OpMoeParams& q, int phase, int grid, size_t smem, cudaStream_t st) {
  const void* fn = moe_fn(q.fmt, q.nchl, phase);
  if (!fn) return cudaErrorInvalidDeviceFunction;
  void* args[] = {const_cast<OpMoeParams*>(&q)};
  return cudaLaunchKernel(fn, dim3(grid), dim3(NTHREADS), args, smem, st);
}
cudaError_t set_smem_op_attention(size_t b) { return raise_limit((const void*)op_attention_kernel, b); }

cudaError_t megakernel_occupancy(int* blocks_per_sm, size_t smem, int fmt, int nchl) {
  const void* fn = step_fn(fmt, nchl, 0);
  if (!fn) return cudaErrorInvalidDeviceFunction;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, fn, NTHREADS_MEGA, smem);
}
cudaError_t phase_occupancy(int* blocks_per_sm, size_t smem, int fmt, int nchl) {
  const void* fn = step_fn(fmt, nchl, 2);
  if (!fn) return cudaErrorInvalidDeviceFunction;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, fn, NTHREADS, smem);
}

size_t smem_for(int stages, int slot, int xs_bytes) { return step_smem_bytes(stages, slot, xs_bytes); }

cudaError_t launch_pack_rows(uint8_t* dst, int dst_rb, int dst_step, int dst_first, int rows,
                             const uint8_t* w, int w_bytes, const uint8_t* s, int s_bytes,
                             cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  pack_rows_kernel<<<rows < 4096 ? rows : 4096, 128, 0, st>>>(dst, dst_rb, dst_step, dst_first, rows, w,
                                                            w_bytes, s, s_bytes);
  return cudaGetLastError();
}
cudaError_t launch_unpack_rows(const uint8_t* src, int src_rb, int src_step, int src_first, int rows,
                               uint8_t* w, int w_bytes, uint8_t* s, int s_bytes, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  unpack_rows_kernel<<<rows < 4096 ? rows : 4096, 128, 0, st>>>(src, src_rb, src_step, src_first, rows,
                                                              w, w_bytes, s, s_bytes);
  return cudaGetLastError();
}
cudaError_t launch_transpose_u16(const uint16_t* in, int rows, int cols, uint16_t* out, cudaStream_t st) {
  if (rows <= 0 || cols <= 0) return cudaSuccess;
  transpose_u16_kernel<<<dim3((cols + 31) / 32, (rows + 31) / 32), dim3(32, 8), 0, st>>>(in, rows, cols, out);
  return cudaGetLastError();
}
cudaError_t launch_bf16_to_f32(const uint16_t* in, float* out, int n, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  bf16_to_f32_kernel<<<(n + 255) / 256, 256, 0, st>>>(in, out, n);
  return cudaGetLastError();
}
cudaError_t launch_f32_to_bf16(const float* in, uint16_t* out, int n, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  f32_to_bf16_kernel<<<(n + 255) / 256, 256, 0, st>>>(in, out, n);
  return cudaGetLastError();
}

}  // namespace tinfer
