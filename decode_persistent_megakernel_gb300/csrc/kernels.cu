// kernels.cu -- the kernels of the engine and their launch wrappers.
//
//   decode_megakernel    one cooperative launch per step: every phase of every layer, grid
//                        barriers between dependent phases, the weight stream running ahead of them
//   decode_phase_kernel  one phase of one layer; the CUDA-graph path chains 5 L + 1 of them with
//                        programmatic dependent launch so that the next kernel's weight prefetch
//                        starts while the current one finishes
//   op_gemv_kernel, op_attention_kernel   single operations for the per-kernel parity tests
//   pack / unpack kernels                 canonical <-> streaming layout
#include <cuda_runtime.h>

#include "engine.h"
#include "kernels.h"
#include "step.cuh"

namespace tinfer {

// ------------------------------------------------------------------------------ step schedule

__device__ __forceinline__ void phase_of(int k, int L, int& phase, int& layer) {
  if (k >= L * PHASES_PER_LAYER) { phase = PH_LM; layer = 0; return; }
  layer = k / PHASES_PER_LAYER;
  const int r = k - layer * PHASES_PER_LAYER;
  phase = r == 0 ? PH_QKV : r == 1 ? PH_ATTN : r == 2 ? PH_O : r == 3 ? PH_GU : PH_DOWN;
}

__device__ __forceinline__ GemvDesc phase_gemv(const StepParams& p, int phase, int layer) {
  const Dims& m = p.m;
  GemvDesc g;
  g.fmt = m.fmt;
  g.group = m.group;
  g.scale_bf16 = m.scale_bf16;
  g.quantum = 1;
  const LayerDev& L = p.layers[layer];
  switch (phase) {
    case PH_QKV: g.w = L.qkv; g.rows = m.qkv_rows; g.cols = m.H; g.rb = m.rb_h; break;
    case PH_O: g.w = L.o; g.rows = m.H; g.cols = m.nq * m.d; g.rb = m.rb_qd; break;
    case PH_GU: g.w = L.gu; g.rows = 2 * m.F; g.cols = m.H; g.rb = m.rb_h; g.quantum = 2; break;
    case PH_DOWN: g.w = L.down; g.rows = m.H; g.cols = m.F; g.rb = m.rb_f; break;
    default:
      g.w = reinterpret_cast<const uint8_t*>(p.lm_head);
      g.rows = m.V; g.cols = m.H; g.rb = m.rb_lm; g.fmt = 0;
      break;
  }
  return g;
}

__device__ __forceinline__ AttnArgs step_attn_args(const StepParams& p, int layer, int pos) {
  const Dims& m = p.m;
  AttnArgs A;
  A.qkv = p.qkv;
  const size_t lay = (size_t)layer * m.nkv * m.max_ctx * m.d;
  A.kc = p.kcache + lay;
  A.vc = p.vcache + lay;
  A.rope = p.rope;
  A.part_m = p.part_m;
  A.part_l = p.part_l;
  A.part_o = p.part_o;
  A.nch_cap = p.nch_cap;
  A.tickets = p.tickets;
  A.out = p.attn;
  A.nq = m.nq; A.nkv = m.nkv; A.d = m.d; A.max_ctx = m.max_ctx; A.pos = pos;
  return A;
}

__device__ void produce_phase(const StepParams& p, Pipe& pp, int phase, int layer, int pos,
                              uint64_t pol_w, uint64_t pol_kv, bool& dead) {
  if (phase == PH_ATTN) {
    const AttnArgs A = step_attn_args(p, layer, pos);
    const AttnSplit sp = attn_split(pos, A.nkv, A.d, p.grid, p.slot_bytes, p.n_chunks_override);
    const int units = A.nkv * sp.nch;
    for (int u = blockIdx.x; u < units; u += p.grid)
      produce_attn_unit(pp, A, u / sp.nch, u % sp.nch, sp, pol_kv, dead);
    return;
  }
  const GemvDesc g = phase_gemv(p, phase, layer);
  const void* gain = nullptr;
  uint32_t gain_bytes = 0;
  if (phase == PH_QKV) { gain = p.layers[layer].g1; gain_bytes = p.m.H * 4; }
  else if (phase == PH_GU) { gain = p.layers[layer].g2; gain_bytes = p.m.H * 4; }
  else if (phase == PH_LM) { gain = p.final_norm; gain_bytes = p.m.H * 2; }
  produce_rows(pp, g, row_split(g, blockIdx.x, p.grid, p.slot_bytes), pol_w, dead, gain, gain_bytes);
}

__device__ __forceinline__ unsigned long long* trace_at(const StepParams& p, int k, int field) {
  if (!p.trace) return nullptr;
  const int nph = p.m.L * PHASES_PER_LAYER + 1;
  return p.trace + ((size_t)blockIdx.x * nph + k) * TRACE_FIELDS + field;
}

// Consumer side of one attention phase (every unit this CTA owns). Separate from the GEMV phase so
// that each gets its own register allocation; the pipe state goes in and comes back by value.
__device__ __forceinline__ Pipe consume_attn_phase(const StepParams& p, Pipe pp, int layer, int pos,
                                                int tid, int k) {
  unsigned long long* tr_ready = trace_at(p, k, TR_READY);
  if (tr_ready && tid == 0) *tr_ready = globaltimer();
  const AttnArgs A = step_attn_args(p, layer, pos);
  const AttnSplit sp = attn_split(pos, A.nkv, A.d, p.grid, p.slot_bytes, p.n_chunks_override);
  const int units = A.nkv * sp.nch;
  for (int u = blockIdx.x; u < units; u += p.grid) attn_unit(pp, A, sp, u / sp.nch, u % sp.nch, tid);
  return pp;
}

// Consumer side of one GEMV phase: QKV (RMSNorm prologue, bias), O (+ residual), gate/up (RMSNorm,
// SwiGLU), down (+ residual) or the LM head (final RMSNorm, logits, argmax).
template <int FMT>
__device__ __forceinline__ Pipe consume_gemv_phase(const StepParams& p, Pipe pp, int phase, int layer,
                                                int token, int tid, int k) {
  const Dims& m = p.m;
  unsigned long long* tr_ready = trace_at(p, k, TR_READY);
  const GemvDesc g = phase_gemv(p, phase, layer);
  const RowSplit rs = row_split(g, blockIdx.x, p.grid, p.slot_bytes);
  const LayerDev& L = p.layers[layer];
  ActSrc src{};
  Epi epi{};
  src.eps = m.eps;
  switch (phase) {
    case PH_QKV:
      if (layer == 0) src.xb = p.embed + (size_t)token * m.H; else src.xf = p.x;
      src.gf = L.g1; src.n = m.H;
      epi = Epi{EK_STORE, p.qkv, L.bias};
      break;
    case PH_O:
      src.xf = p.attn; src.n = m.nq * m.d;
      epi = Epi{EK_RESIDUAL, p.x, nullptr};
      break;
    case PH_GU:
      src.xf = p.x; src.gf = L.g2; src.n = m.H;
      epi = Epi{EK_SWIGLU, p.act, nullptr};
      break;
    case PH_DOWN:
      src.xf = p.act; src.n = m.F;
      epi = Epi{EK_RESIDUAL, p.x, nullptr};
      break;
    default:
      src.xf = p.x; src.gb = p.final_norm; src.n = m.H;
      epi = Epi{EK_ARGMAX, p.logits, nullptr};
      break;
  }
  Best best{-CUDART_INF_F, 0x7FFFFFFF, 0};
  // int4 models stream their linears as int4 and the LM head as bf16; bf16 models need one instance
  if (FMT == 1 && g.fmt == 1) gemv_rows<1, 2>(pp, g, rs, src, epi, best, tid, tr_ready);
  else gemv_rows<0, 8>(pp, g, rs, src, epi, best, tid, tr_ready);
  if (phase == PH_QKV && layer == 0 && blockIdx.x == 0)
    for (int i = tid; i < m.H; i += NCT) p.x[i] = bf16_to_f(p.embed[(size_t)token * m.H + i]);
  if (phase == PH_LM) {
    const Best cb = best_block_reduce(best, pp.ms, tid);
    argmax_publish(cb, p.best_val, p.best_idx, p.best_bad, p.tickets + m.nkv, p.grid, blockIdx.x,
                   p.argmax, p.err, p.err_host, pp.ms, tid);
  }
  return pp;
}

template <int FMT>
__device__ __forceinline__ void consume_phase(const StepParams& p, Pipe& pp, int phase, int layer,
                                              int token, int pos, int tid, int k) {
  if (phase == PH_ATTN) pp = consume_attn_phase(p, pp, layer, pos, tid, k);
  else pp = consume_gemv_phase<FMT>(p, pp, phase, layer, token, tid, k);
}

// Barrier over the CTAs of the cooperative launch, run by the consumer warps: one monotonic
// arrival counter (it never resets; barrier k of a launch waits for bar_base + (k+1) * grid).
// Thread 0 arrives with a release reduction that publishes the CTA's writes and polls with acquire
// loads under a time limit; the poll also ends when another CTA has raised an error. Returns false,
// the same in every consumer thread, when the step must stop.
__device__ bool grid_sync(const StepParams& p, Misc* ms, int tid, int index) {
  named_sync(BAR_CONS, NCT);
  if (tid == 0) {
    int stop = *reinterpret_cast<volatile int*>(&ms->abort);
    const bool skip = (p.dbg_skip_cta == (int)blockIdx.x && p.dbg_skip_barrier == index);
    if (!stop && !skip) {
      // barrier `index` of this launch completes when the counter reaches its target
      const unsigned target = p.bar_base + (unsigned)(index + 1) * (unsigned)p.grid;
      red_add_release(p.gbar, 1u);
      const uint64_t t0 = globaltimer();
      unsigned spins = 0;
      while ((int)(ld_acquire(p.gbar) - target) < 0) {
        if ((++spins & 63u) == 0) {
          if (ld_volatile_int(p.err) != 0) { stop = 1; break; }
          if ((long long)(globaltimer() - t0) > p.timeout_ns) {
            raise_error(p.err, p.err_host, EW_TIMEOUT);
            stop = 1;
            break;
          }
        }
      }
    }
    ms->exit_now = stop;
  }
  named_sync(BAR_CONS, NCT);
  return !*reinterpret_cast<volatile int*>(&ms->exit_now);
}

// Start-of-step decision, identical in every CTA: skip when an earlier step left an error, or when
// the token id is out of range (CTA 0 records that).
__device__ __forceinline__ bool step_prologue(const StepParams& p, int& token, int pos, int* s_tok) {
  if (threadIdx.x == 0) {
    int e = ld_volatile_int(p.err);
    const int tok = p.token_dev ? *p.token_dev : p.token;
    if (e == 0 && (tok < 0 || tok >= p.m.V)) {
      if (blockIdx.x == 0) raise_error(p.err, p.err_host, EW_BADTOKEN);
      e = 1;
    }
    s_tok[0] = tok;
    s_tok[1] = e;
  }
  __syncthreads();
  token = s_tok[0];
  (void)pos;
  return s_tok[1] == 0;
}

template <int FMT>
__global__ void __launch_bounds__(NTHREADS_MEGA, 1) decode_megakernel(const __grid_constant__ StepParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ int s_tok[2];
  Pipe pp;
  pipe_init(pp, smem, p.ring_stages, p.slot_bytes, p.timeout_ns, p.err, p.err_host);
  pp.inflight = p.inflight;
  pipe_setup(pp);
  int token = 0;
  const int pos = p.pos;
  if (!step_prologue(p, token, pos, s_tok)) return;
  const int nph = p.m.L * PHASES_PER_LAYER + 1;
  const int tid = threadIdx.x;
  if (tid >= NCT) {
    reg_dealloc<REG_PRODUCER>();
    if (tid == NCT) {
      const uint64_t pw = policy_evict_first(), pkv = policy_evict_normal();
      bool dead = false;
      for (int k = 0; k < nph && !dead; ++k) {
        int phase, layer;
        phase_of(k, p.m.L, phase, layer);
        if (unsigned long long* t = trace_at(p, k, TR_PROD_BEGIN)) *t = globaltimer();
        produce_phase(p, pp, phase, layer, pos, pw, pkv, dead);
        if (unsigned long long* t = trace_at(p, k, TR_PROD_END)) *t = globaltimer();
      }
      prod_drain(pp);
    }
  } else {
    reg_alloc<REG_CONSUMER>();
    for (int k = 0; k < nph; ++k) {
      int phase, layer;
      phase_of(k, p.m.L, phase, layer);
      if (unsigned long long* t = trace_at(p, k, TR_START)) if (tid == 0) *t = globaltimer();
      consume_phase<FMT>(p, pp, phase, layer, token, pos, tid, k);
      if (unsigned long long* t = trace_at(p, k, TR_END)) if (tid == 0) *t = globaltimer();
      if (k + 1 < nph && !grid_sync(p, pp.ms, tid, k)) break;
    }
    if (tid == 0) *reinterpret_cast<volatile int*>(&pp.ms->cons_done) = 1;
  }
  __syncthreads();
}

template <int FMT>
__global__ void __launch_bounds__(NTHREADS, 2) decode_phase_kernel(const __grid_constant__ StepParams p, int k) {
  extern __shared__ __align__(128) unsigned char smem[];
  Pipe pp;
  pipe_init(pp, smem, p.ring_stages, p.slot_bytes, p.timeout_ns, p.err, p.err_host);
  pp.inflight = p.inflight;
  pipe_setup(pp);
  __syncthreads();
  pdl_launch_dependents();
  int phase, layer;
  phase_of(k, p.m.L, phase, layer);
  const int tid = threadIdx.x;
  if (tid >= NCT) {
    if (tid == NCT) {
      // the step block was written by the step's first node, which completed before this grid
      // could start; only the attention producer needs pos
      const int pos = phase == PH_ATTN ? p.step_dev[1] : 0;
      bool dead = false;
      produce_phase(p, pp, phase, layer, pos, policy_evict_first(), policy_evict_normal(), dead);
      prod_drain(pp);
    }
  } else {
    pdl_wait();
    if (tid == 0) pp.ms->exit_now = ld_volatile_int(p.err) != 0;
    named_sync(BAR_CONS, NCT);
    if (!*reinterpret_cast<volatile int*>(&pp.ms->exit_now)) {
      const int token = p.step_dev[0], pos = p.step_dev[1];
      consume_phase<FMT>(p, pp, phase, layer, token, pos, tid, k);
    }
    named_sync(BAR_CONS, NCT);
    if (tid == 0) *reinterpret_cast<volatile int*>(&pp.ms->cons_done) = 1;
  }
  __syncthreads();
}

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
      produce_rows(pp, g, rs, policy_evict_first(), dead, q.gain, q.gain ? (uint32_t)q.cols * 4u : 0u);
      prod_drain(pp);
    }
  } else {
    ActSrc src{};
    src.xf = q.x; src.gf = q.gain; src.eps = q.eps; src.n = q.cols;
    const Epi epi{q.epi, q.y, q.bias};
    Best best{-CUDART_INF_F, 0x7FFFFFFF, 0};
    gemv_consume_any(pp, g, rs, src, epi, best, tid, nullptr);
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
  A.qkv = q.qkv; A.kc = q.kc; A.vc = q.vc; A.rope = q.rope;
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
    for (int u = blockIdx.x; u < units; u += gridDim.x) attn_unit(pp, A, sp, u / sp.nch, u % sp.nch, tid);
    if (tid == 0) *reinterpret_cast<volatile int*>(&pp.ms->cons_done) = 1;
  }
  __syncthreads();
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

static const void* mega_fn(int fmt) {
  return fmt == 1 ? reinterpret_cast<const void*>(&decode_megakernel<1>)
                  : reinterpret_cast<const void*>(&decode_megakernel<0>);
}

cudaError_t launch_megakernel(const StepParams& p, size_t smem, cudaStream_t st) {
  void* args[] = {const_cast<StepParams*>(&p)};
  return cudaLaunchCooperativeKernel(mega_fn(p.m.fmt), dim3(p.grid), dim3(NTHREADS_MEGA), args, smem, st);
}

cudaError_t launch_phase(const StepParams& p, int k, size_t smem, cudaStream_t st, bool pdl) {
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
  if (p.m.fmt == 1) return cudaLaunchKernelEx(&cfg, decode_phase_kernel<1>, p, k);
  return cudaLaunchKernelEx(&cfg, decode_phase_kernel<0>, p, k);
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
static cudaError_t raise_limit(const void* fn, int which, size_t bytes) {
  static size_t cur[6][64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (bytes <= cur[which][dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) cur[which][dev] = bytes;
  return e;
}
cudaError_t set_smem_mega(size_t b) {
  cudaError_t e = raise_limit((const void*)&decode_megakernel<0>, 0, b);
  return e != cudaSuccess ? e : raise_limit((const void*)&decode_megakernel<1>, 4, b);
}
cudaError_t set_smem_phase(size_t b) {
  cudaError_t e = raise_limit((const void*)&decode_phase_kernel<0>, 1, b);
  return e != cudaSuccess ? e : raise_limit((const void*)&decode_phase_kernel<1>, 5, b);
}
cudaError_t set_smem_op_gemv(size_t b) { return raise_limit((const void*)op_gemv_kernel, 2, b); }
cudaError_t set_smem_op_attention(size_t b) { return raise_limit((const void*)op_attention_kernel, 3, b); }

cudaError_t megakernel_occupancy(int* blocks_per_sm, size_t smem, int fmt) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, mega_fn(fmt), NTHREADS_MEGA, smem);
}
cudaError_t phase_occupancy(int* blocks_per_sm, size_t smem, int fmt) {
  if (fmt == 1) return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, decode_phase_kernel<1>, NTHREADS, smem);
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, decode_phase_kernel<0>, NTHREADS, smem);
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
