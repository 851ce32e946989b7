// step.cuh -- device code of one decode step, shared by the persistent kernel, the per-phase
// kernels of the CUDA-graph path and the single-operation kernels.
//
// Execution model. A CTA is NCW consumer warps plus one producer warp. The producer's elected lane
// walks the CTA's static schedule (which rows of which matrix, which K/V chunks) and streams those
// bytes from HBM into a ring of shared-memory slots with bulk asynchronous copies that complete on
// per-slot mbarriers. Weights and cached K/V never depend on the current token ("Decoding in tiles",
// section 1: the next kernel cannot start loading its weights although the weights never depend on
// the token), so the producer runs ahead across phase boundaries, bounded only by the ring; the
// consumers wait for the data dependency (the stamped results of the previous phase, or stream
// order between the per-phase kernels) and then drain the slots.
// This is the cross-phase weight prefetch of Hazy Research's megakernel as summarised in "Decoding
// in tiles" (section 1 and section 4), built on Blackwell's bulk-copy engine instead of per-thread
// loads.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math_constants.h>

#include "engine.h"
#include "ptx.cuh"

namespace tinfer {

struct __align__(16) Misc {
  unsigned long long full[MAX_STAGES];
  unsigned long long empty[MAX_STAGES];
  // GEMV phases and attention phases use the same scratch: a CTA's consumer warps pass a named
  // barrier between the last read of one and the first write of the other
  union {
    float rowv[ROWV_MAX];      // row results (per segment) of the current GEMV phase
    struct {
      float qs[G_MAX * D_MAX]; // rotated, pre-scaled queries of the current attention unit
      float sc[G_MAX * T_MAX]; // scores, then probabilities; merge weights in the merge
      float kn[D_MAX];         // new key of this position (bf16-rounded, as float)
      float vn[D_MAX];         // new value of this position (bf16-rounded, as float)
    } at;
  };
  float wred[NCW];             // block-reduction scratch
  float hm[G_MAX];
  float hl[G_MAX];
  float bv[NCW];
  int bi[NCW];
  int bbad[NCW];
  int flag;
  int abort;      // a consumer wait gave up: results of this step are void
  int cons_done;  // consumers have left their loop: the producer stops issuing
  int exit_now;   // uniform stop decision, written by consumer thread 0 between two named barriers
};

// Dynamic shared memory: [ring: stages x slot][Misc][input vector: xs_bytes], every part starting
// on a 128-byte boundary (bulk copies and 16-byte shared loads need 16).
__host__ __device__ inline size_t misc_offset(int stages, int slot_bytes) {
  return ((size_t)stages * slot_bytes + 127) / 128 * 128;
}
__host__ __device__ inline size_t xs_offset(int stages, int slot_bytes) {
  return (misc_offset(stages, slot_bytes) + sizeof(Misc) + 127) / 128 * 128;
}
__host__ __device__ inline size_t step_smem_bytes(int stages, int slot_bytes, int xs_bytes) {
  return xs_offset(stages, slot_bytes) + (size_t)xs_bytes;
}

constexpr int BAR_CONS = 1;  // named barrier id used by the consumer warps

struct Pipe {
  int inflight;     // producer: copies kept outstanding at most (0 = the whole ring)
  uint32_t ring;    // shared address of slot 0
  uint32_t full0;   // shared address of full[0]
  uint32_t empty0;  // shared address of empty[0]
  int stages;
  int slot;
  uint32_t it;      // stages issued (producer) or consumed (consumers)
  int s;            // current slot
  uint32_t ph;      // parity of the current slot's phase
  uint32_t xs;      // shared address of the input-vector buffer
  Misc* ms;
  long long timeout;
  int* err;
  int* err_host;
};

__device__ __forceinline__ void raise_error(int* err, int* err_host, int bits) {
  atomicOr(err, bits);
  if (err_host) *reinterpret_cast<volatile int*>(err_host) = bits;
}

// Waits until the phase of `parity` of mbarrier `bar` completes. Gives up after `timeout` ns, or as
// soon as *stop is non-zero. Returns true on completion.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, long long timeout,
                                      const volatile int* stop) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*stop) return false;
    if ((long long)(globaltimer() - t0) > timeout) return false;
  }
}

__device__ __forceinline__ void pipe_advance(Pipe& pp) {
  ++pp.it;
  if (++pp.s == pp.stages) { pp.s = 0; pp.ph ^= 1u; }
}

__device__ __forceinline__ uint32_t cons_acquire(Pipe& pp) {
  const int s = pp.s;
  if (mbar_try_wait(pp.full0 + 8u * s, pp.ph)) return pp.ring + (uint32_t)s * pp.slot;
  volatile int* ab = &pp.ms->abort;
  if (!*ab) {
    if (!wait_bar(pp.full0 + 8u * s, pp.ph, pp.timeout, ab)) {
      if (!*ab) {
        *ab = 1;
        raise_error(pp.err, pp.err_host, EW_TIMEOUT);
      }
    }
  }
  return pp.ring + (uint32_t)s * pp.slot;
}

__device__ __forceinline__ void cons_release(Pipe& pp, int lane) {
  __syncwarp();
  if (lane == 0) mbar_arrive(pp.empty0 + 8u * pp.s);
  pipe_advance(pp);
}

// Producer: one stage of `bytes` contiguous bytes (multiple of 16, <= slot) from src.
__device__ __forceinline__ void prod_push(Pipe& pp, const void* src, uint32_t bytes, uint64_t pol,
                                          bool& dead) {
  if (dead) return;
  const int s = pp.s;
  if (!wait_bar(pp.empty0 + 8u * s, pp.ph ^ 1u, pp.timeout, &pp.ms->cons_done)) {
    dead = true;
    if (!*reinterpret_cast<volatile int*>(&pp.ms->cons_done))
      raise_error(pp.err, pp.err_host, EW_TIMEOUT);
    return;
  }
  const int k = pp.inflight < pp.stages ? pp.inflight : pp.stages;  // never beyond the ring
  if (k > 0 && pp.it >= (uint32_t)k) {
    // bound the bytes in flight: the copy issued `k` stages ago must have landed
    const int s2 = s >= k ? s - k : s - k + pp.stages;
    const uint32_t p2 = s >= k ? pp.ph : pp.ph ^ 1u;
    if (!mbar_try_wait(pp.full0 + 8u * s2, p2) &&
        !wait_bar(pp.full0 + 8u * s2, p2, pp.timeout, &pp.ms->cons_done)) {
      dead = true;
      return;
    }
  }
  const uint32_t fb = pp.full0 + 8u * s;
  mbar_arrive_expect_tx(fb, bytes);
  if (bytes) bulk_g2s(pp.ring + (uint32_t)s * pp.slot, src, bytes, fb, pol);
  pipe_advance(pp);
}

// Producer: opens the next stage for `bytes` bytes, which the caller then fills with one or more
// bulk copies into the shared address *dst completing on *bar, and closes with pipe_advance. False
// (and dead set) when the consumers are gone or a wait ran out.
__device__ __forceinline__ bool prod_open(Pipe& pp, uint32_t bytes, uint32_t& dst, uint32_t& bar, bool& dead) {
  if (dead) return false;
  const int s = pp.s;
  if (!wait_bar(pp.empty0 + 8u * s, pp.ph ^ 1u, pp.timeout, &pp.ms->cons_done)) {
    dead = true;
    if (!*reinterpret_cast<volatile int*>(&pp.ms->cons_done)) raise_error(pp.err, pp.err_host, EW_TIMEOUT);
    return false;
  }
  const int k = pp.inflight < pp.stages ? pp.inflight : pp.stages;
  if (k > 0 && pp.it >= (uint32_t)k) {
    const int s2 = s >= k ? s - k : s - k + pp.stages;
    const uint32_t p2 = s >= k ? pp.ph : pp.ph ^ 1u;
    if (!mbar_try_wait(pp.full0 + 8u * s2, p2) &&
        !wait_bar(pp.full0 + 8u * s2, p2, pp.timeout, &pp.ms->cons_done)) {
      dead = true;
      return false;
    }
  }
  bar = pp.full0 + 8u * s;
  dst = pp.ring + (uint32_t)s * pp.slot;
  mbar_arrive_expect_tx(bar, bytes);
  return true;
}

// Before the CTA exits: every copy this producer issued has landed (bounded wait).
static __device__ void prod_drain(Pipe& pp) {
  const uint32_t n = pp.it < (uint32_t)pp.stages ? pp.it : (uint32_t)pp.stages;
  int never = 0;
  for (uint32_t k = pp.it - n; k < pp.it; ++k)
    wait_bar(pp.full0 + 8u * (k % pp.stages), (k / pp.stages) & 1u, pp.timeout, &never);
}

static_assert(sizeof(Misc) % 16 == 0, "Misc keeps 16-byte alignment");

__device__ __forceinline__ void pipe_init(Pipe& pp, unsigned char* smem, int stages, int slot,
                                          long long timeout, int* err, int* err_host) {
  pp.ring = smem_addr(smem);
  pp.ms = reinterpret_cast<Misc*>(smem + misc_offset(stages, slot));
  pp.full0 = smem_addr(&pp.ms->full[0]);
  pp.empty0 = smem_addr(&pp.ms->empty[0]);
  pp.xs = smem_addr(smem + xs_offset(stages, slot));
  pp.stages = stages;
  pp.slot = slot;
  pp.inflight = 0;
  pp.it = 0;
  pp.s = 0;
  pp.ph = 0;
  pp.timeout = timeout;
  pp.err = err;
  pp.err_host = err_host;
}

// Thread 0 initialises the barriers; call before __syncthreads.
__device__ __forceinline__ void pipe_setup(Pipe& pp) {
  if (threadIdx.x == 0) {
    for (int s = 0; s < pp.stages; ++s) {
      mbar_init(pp.full0 + 8u * s, 1);
      mbar_init(pp.empty0 + 8u * s, NCW);
    }
    pp.ms->flag = 0;
    pp.ms->abort = 0;
    pp.ms->cons_done = 0;
    pp.ms->exit_now = 0;
    mbar_fence_init();
  }
}

// ------------------------------------------------------------------------------ small helpers

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_to_f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }
// Typed pointer to the dynamic shared memory at shared address `addr`. Loads through it are plain
// C++ loads the compiler knows to be shared-memory loads, so it can batch and reorder them (the
// barrier and mbarrier waits carry memory clobbers, which keep the loads after the waits).
extern __shared__ __align__(128) unsigned char tinfer_dyn_smem[];
template <class T>
__device__ __forceinline__ const T* sptr(uint32_t addr) {
  return reinterpret_cast<const T*>(tinfer_dyn_smem + (addr - smem_addr(tinfer_dyn_smem)));
}
template <class T>
__device__ __forceinline__ T* sptr_w(uint32_t addr) {
  return reinterpret_cast<T*>(tinfer_dyn_smem + (addr - smem_addr(tinfer_dyn_smem)));
}

__device__ __forceinline__ uint16_t f_to_bf16_bits(float v) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

// ---- stamped words: fp32 value in the low half, the writing phase's stamp in the high half -------
__device__ __forceinline__ uint64_t stamp_word(float v, unsigned stamp) {
  return ((uint64_t)stamp << 32) | (uint64_t)__float_as_uint(v);
}
__device__ __forceinline__ float word_value(uint64_t w) { return __uint_as_float((uint32_t)w); }
__device__ __forceinline__ unsigned word_stamp(uint64_t w) { return (unsigned)(w >> 32); }

// Bounded polling of stamped words another CTA writes: again() is called after each stale read; it
// returns false once the time limit has passed (raising the time-out error) or another CTA has
// raised an error, and then sets the CTA's abort flag.
struct Poll {
  uint64_t t0 = 0;
  unsigned n = 0;
  __device__ __forceinline__ bool again(const Pipe& pp) {
    if (n++ == 0) t0 = globaltimer();
    if ((n & 15u) == 0) {
      volatile int* ab = &pp.ms->abort;
      if (*ab || ld_volatile_int(pp.err) != 0) { *ab = 1; return false; }
      if ((long long)(globaltimer() - t0) > pp.timeout) {
        raise_error(pp.err, pp.err_host, EW_TIMEOUT);
        *ab = 1;
        return false;
      }
    }
    return true;
  }
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

// Reduces 8 per-lane partials (8 rows) across the 32 lanes with 9 shuffles. Afterwards lanes with
// (lane & 3) == 0 hold the warp total of row transpose_row8(lane). Every row's total is the same
// summation tree, so identical rows give identical totals.
__device__ __forceinline__ float transpose_reduce8(const float (&v)[8], int lane) {
  float a[4];
  {
    const bool up = lane & 16;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float send = up ? v[k] : v[k + 4];
      const float keep = up ? v[k + 4] : v[k];
      a[k] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 16);
    }
  }
  float b[2];
  {
    const bool up = lane & 8;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const float send = up ? a[k] : a[k + 2];
      const float keep = up ? a[k + 2] : a[k];
      b[k] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 8);
    }
  }
  float c;
  {
    const bool up = lane & 4;
    const float send = up ? b[0] : b[1];
    const float keep = up ? b[1] : b[0];
    c = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 4);
  }
  c += __shfl_xor_sync(0xFFFFFFFFu, c, 2);
  c += __shfl_xor_sync(0xFFFFFFFFu, c, 1);
  return c;
}
__device__ __forceinline__ int transpose_row8(int lane) {
  return ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1);
}

// ------------------------------------------------------------------------------ GEMV

// 8 bf16 weights (one 16-byte chunk) times 8 activations, accumulated as (even, odd) pairs on the
// packed f32x2 FMA units.
__device__ __forceinline__ float2 dot8_bf16(const uint4 w, const float* a, float2 acc) {
  acc = fma2(make_float2(bf16_lo(w.x), bf16_hi(w.x)), make_float2(a[0], a[1]), acc);
  acc = fma2(make_float2(bf16_lo(w.y), bf16_hi(w.y)), make_float2(a[2], a[3]), acc);
  acc = fma2(make_float2(bf16_lo(w.z), bf16_hi(w.z)), make_float2(a[4], a[5]), acc);
  acc = fma2(make_float2(bf16_lo(w.w), bf16_hi(w.w)), make_float2(a[6], a[7]), acc);
  return acc;
}

// A 32-bit register holding `v` that the compiler cannot fold into an instruction's immediate.
__device__ __forceinline__ uint32_t opaque_u32(uint32_t v) {
  uint32_t r;
  asm volatile("mov.b32 %0, %1;" : "=r"(r) : "r"(v));
  return r;
}

// (x & MASK) | m in one logic instruction: the mask is the immediate, m a register. Written out
// because a mask and a magic number that are both literals need two instructions.
template <uint32_t MASK>
__device__ __forceinline__ uint32_t and_or(uint32_t x, uint32_t m) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(x), "n"(MASK), "r"(m));
  return d;
}

// 32 int4 weights (one 16-byte chunk) dotted with 32 activations, returning sum_k q_k * a_k with
// q_k in [0, 15] (the zero point is applied by the caller). Dequantisation uses the exponent trick
// of tinyinfer ("v0.1": OR the nibble into the mantissa of 2^23 and subtract), generalised so that
// no shift is needed per nibble: masking nibble i of a 16-bit half in place gives the float
// 2^23 + q * 16^i exactly, and the activation of that element is stored pre-multiplied by 16^-i
// (exact, a power of two). (f - 2^23) * a' then equals q * a exactly before rounding, so each
// product is rounded exactly as q * a would be. Pairs go through Blackwell's packed f32x2 units.
// mag holds 0x4B000000 (the bits of 2^23) in a register: one logic instruction per nibble.
__device__ __forceinline__ float dot32_int4(const uint4 w, const float* a, uint32_t mag) {
  const float2 B = make_float2(-8388608.f, -8388608.f);
  float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
  const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t lo = words[k], hi = words[k] >> 16;
    const float2 f01 = make_float2(__uint_as_float(and_or<0x000Fu>(lo, mag)), __uint_as_float(and_or<0x00F0u>(lo, mag)));
    const float2 f23 = make_float2(__uint_as_float(and_or<0x0F00u>(lo, mag)), __uint_as_float(and_or<0xF000u>(lo, mag)));
    const float2 f45 = make_float2(__uint_as_float(and_or<0x000Fu>(hi, mag)), __uint_as_float(and_or<0x00F0u>(hi, mag)));
    const float2 f67 = make_float2(__uint_as_float(and_or<0x0F00u>(hi, mag)), __uint_as_float(and_or<0xF000u>(hi, mag)));
    acc0 = fma2(add2(f01, B), make_float2(a[8 * k + 0], a[8 * k + 1]), acc0);
    acc1 = fma2(add2(f23, B), make_float2(a[8 * k + 2], a[8 * k + 3]), acc1);
    acc0 = fma2(add2(f45, B), make_float2(a[8 * k + 4], a[8 * k + 5]), acc0);
    acc1 = fma2(add2(f67, B), make_float2(a[8 * k + 6], a[8 * k + 7]), acc1);
  }
  return (acc0.x + acc0.y) + (acc1.x + acc1.y);
}

// Where the activation vector of a GEMV comes from.
struct ActSrc {
  const float* xf;     // fp32 source (single-operation path), or
  const uint64_t* xw;  // stamped words another phase wrote (read through L2), or
  const uint16_t* xb;  // bf16 source (the embedding row)
  unsigned stamp;      // stamp the words must carry (xw)
  int check;           // wait for the stamp (xw)
  const float* gf;     // fp32 RMSNorm gain, or
  const uint16_t* gb;  // bf16 RMSNorm gain, or neither (no norm)
  float eps;
  int n;
};


struct GemvDesc {
  const uint8_t* w;
  int rows, cols, rb;
  int fmt, group, scale_bf16;
  int quantum;  // 2: rows come in (gate, up) pairs that one stage never splits
  // segment-major stages (gemv_rows<..., SEGMAJOR>): a stage holds nsegs blocks, block s the stage's
  // rows of segment s (rbs bytes per row), as gathered from nsegs separate matrices
  // (both 0 for row-major stages; no default member initialisers, so that a __shared__ table of
  // descriptors needs no constructor)
  int nsegs, rbs;
};

// Rows of a matrix owned by one CTA: an even split of row quanta; nr rows per ring stage.
struct RowSplit {
  int r0, r1, nr;
};
__device__ __forceinline__ RowSplit row_split(const GemvDesc& g, int cta, int grid, int slot) {
  const unsigned units = (unsigned)(g.rows / g.quantum);  // units * grid < 2^32 for every model here
  const int u0 = (int)(units * (unsigned)cta / (unsigned)grid);
  const int u1 = (int)(units * (unsigned)(cta + 1) / (unsigned)grid);
  return RowSplit{u0 * g.quantum, u1 * g.quantum, stage_rows(g.fmt, g.cols, g.rb, slot, g.quantum)};
}

enum EpiKind : int { EK_STORE = 0, EK_RESIDUAL = 1, EK_SWIGLU = 2, EK_ARGMAX = 3, EK_COLSPLIT = 4 };
struct Epi {
  int kind;
  void* out;              // output: plain floats (single operations, logits) or stamped words
  const float* bias;
  const void* res;        // EK_RESIDUAL input: null (out itself), stamped words or bf16 (flags)
  unsigned stamp;         // stamp of stamped output words
  int flags;              // EF_* below
};
enum : int { EF_OUT_STAMPED = 1, EF_RES_STAMPED = 2, EF_RES_BF16 = 4, EF_WITHHOLD = 8 };

// Residual input of row r (EK_RESIDUAL): the rows are this thread's own, written by it in an
// earlier phase (or constant), so no stamp needs checking.
__device__ __forceinline__ float residual_at(const Epi& e, int r) {
  if (e.flags & EF_RES_STAMPED) return word_value(static_cast<const uint64_t*>(e.res)[r]);
  if (e.flags & EF_RES_BF16) return bf16_to_f(static_cast<const uint16_t*>(e.res)[r]);
  return __ldcg(static_cast<const float*>(e.out) + r);
}
__device__ __forceinline__ void epi_write(const Epi& e, int r, float v) {
  if (e.flags & EF_WITHHOLD) return;
  if (e.flags & EF_OUT_STAMPED) st_relaxed_u64(static_cast<uint64_t*>(e.out) + r, stamp_word(v, e.stamp));
  else static_cast<float*>(e.out)[r] = v;
}

struct Best {
  float v;
  int i;
  int bad;
};

__device__ __forceinline__ void best_update(Best& b, float v, int i) {
  if (!isfinite(v)) b.bad = 1;
  else if (v > b.v || (v == b.v && i < b.i)) { b.v = v; b.i = i; }
}


__device__ __forceinline__ float4 gain_block(const ActSrc& src, int j) {
  if (src.gf) return __ldg(reinterpret_cast<const float4*>(src.gf) + j);
  const uint2 w = __ldg(reinterpret_cast<const uint2*>(src.gb) + j);
  return make_float4(bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y));
}

// The phase's input vector, written by other CTAs in the previous phase, fetched once per CTA into
// shared memory by all consumer threads together (16-byte loads through L2, thread t taking blocks
// t, t + NCT, ...): every warp of every CTA reading the same few cache lines serialises on those
// lines, one read per CTA does not, and the load path does not queue behind the CTA's own bulk
// weight copies. Stamped sources are read again, all stale blocks of a thread together, until the
// writers' stamps show.
// With an RMSNorm gain the stored values are x * g and the sum of squares of x is reduced on the
// way; the return value is 1 / rms(x) (1 without a norm), the same in every consumer thread.
// Returns after the named barrier that publishes the copy; the CTA's abort flag is then set (the
// same in every thread) if a stamped source never showed up.
// Layout in shared memory, for the GEMV's 16-byte weight chunks of E inputs (E = 8 for bf16, 32 for
// int4): the inputs of chunk C are its E / 4 float4 blocks, block b stored at C * E / 4 +
// (b ^ chunk_swizzle(C)), so that the lanes of a quarter-warp, which read consecutive chunks, hit
// distinct banks while every lane reads its blocks in order (no register shuffling). For int4 the
// stored values are also pre-multiplied by 16^-(i mod 4) for input i of the chunk (exact: powers of
// two), the activation scaling of the in-place nibble decode (dot32_int4).
template <int E>
__device__ __forceinline__ int chunk_swizzle(int c) {
  return E == 8 ? (c >> 2) & 1 : c & (E / 4 - 1);
}
template <int IF>
__device__ __forceinline__ float fetch_vector_n(Pipe& pp, const ActSrc& src, int tid, int fmt) {
  const bool norm = src.gf || src.gb;
  const int nb = src.n / 4;
  float4* xs = sptr_w<float4>(pp.xs);
  // block j is block j % B of chunk j / B (B = E / 4 blocks per chunk)
  const int bsh = fmt == 1 ? 3 : 1;
  const float4 pre = fmt == 1 ? make_float4(1.f, 0.0625f, 0.00390625f, 0.000244140625f)
                              : make_float4(1.f, 1.f, 1.f, 1.f);
  float ss = 0.f;
  for (int j0 = tid; j0 < nb; j0 += IF * NCT) {
    float4 x[IF];
    // the gains do not depend on the previous phase: their loads issue first, so that their
    // latency hides under the wait for the stamped input instead of following it
    float4 gv[IF];
#pragma unroll
    for (int u = 0; u < IF; ++u) {
      const int j = j0 + u * NCT;
      gv[u] = norm && j < nb ? gain_block(src, j) : make_float4(1.f, 1.f, 1.f, 1.f);
    }
    if (src.xw) {
      // one 32-byte load per block of 4 stamped words; stale blocks are read again until their
      // writers' stamps show (bounded)
      const uint64_t* xw = src.xw;
      ulonglong2 w0[IF], w1[IF];
#pragma unroll
      for (int u = 0; u < IF; ++u) {
        const int j = j0 + u * NCT;
        if (j < nb) ld_relaxed_v4u64(xw + 4 * j, w0[u], w1[u]);
      }
      if (src.check) {
        // every block still stale is read again in the same turn, so that one more L2 round trip
        // settles all of them (reading them again one after another would take one per block)
        const unsigned sv = src.stamp;
        auto fresh = [&](int u) {
          return word_stamp(w0[u].x) == sv && word_stamp(w0[u].y) == sv && word_stamp(w1[u].x) == sv &&
                 word_stamp(w1[u].y) == sv;
        };
        unsigned stale = 0;
#pragma unroll
        for (int u = 0; u < IF; ++u)
          if (j0 + u * NCT < nb && !fresh(u)) stale |= 1u << u;
        Poll pl;
        while (stale && pl.again(pp)) {
#pragma unroll
          for (int u = 0; u < IF; ++u) {
            if (stale & (1u << u)) ld_relaxed_v4u64(xw + 4 * (j0 + u * NCT), w0[u], w1[u]);
          }
#pragma unroll
          for (int u = 0; u < IF; ++u)
            if ((stale & (1u << u)) && fresh(u)) stale &= ~(1u << u);
        }
      }
#pragma unroll
      for (int u = 0; u < IF; ++u) {
        const int j = j0 + u * NCT;
        if (j < nb) {
          x[u] = make_float4(word_value(w0[u].x), word_value(w0[u].y), word_value(w1[u].x), word_value(w1[u].y));
        } else {
          x[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
    } else if (src.xf) {
      const float4* xf = reinterpret_cast<const float4*>(src.xf);
#pragma unroll
      for (int u = 0; u < IF; ++u) {
        const int j = j0 + u * NCT;
        x[u] = j < nb ? __ldcg(xf + j) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    } else {
      const uint2* xb = reinterpret_cast<const uint2*>(src.xb);
#pragma unroll
      for (int u = 0; u < IF; ++u) {
        const int j = j0 + u * NCT;
        const uint2 w = j < nb ? __ldg(xb + j) : make_uint2(0u, 0u);
        x[u] = make_float4(bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y));
      }
    }
#pragma unroll
    for (int u = 0; u < IF; ++u) {
      const int j = j0 + u * NCT;
      if (j < nb) {
        ss = fmaf(x[u].x, x[u].x, ss);
        ss = fmaf(x[u].y, x[u].y, ss);
        ss = fmaf(x[u].z, x[u].z, ss);
        ss = fmaf(x[u].w, x[u].w, ss);
        const float4 g = gv[u];
        const int c = j >> bsh, b = j & ((1 << bsh) - 1);
        const int key = fmt == 1 ? chunk_swizzle<32>(c) : chunk_swizzle<8>(c);
        xs[(c << bsh) + (b ^ key)] = make_float4(x[u].x * g.x * pre.x, x[u].y * g.y * pre.y,
                                                 x[u].z * g.z * pre.z, x[u].w * g.w * pre.w);
      }
    }
  }
  if (norm) {
    ss = warp_sum(ss);
    if ((tid & 31) == 0) pp.ms->wred[tid >> 5] = ss;
  }
  named_sync(BAR_CONS, NCT);
  if (!norm) return 1.f;
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < NCW; ++w) tot += pp.ms->wred[w];
  return 1.f / sqrtf(tot / (float)src.n + src.eps);
}



// One lane's chunk C of the input vector from the shared-memory copy (fetch_vector_n's layout): its
// E / 4 float4 blocks in order, each read from its swizzled place.
template <int E>
__device__ __forceinline__ void load_chunk(const float4* xs, int c, float4 (&v)[E / 4]) {
  constexpr int B = E / 4;
  const int key = chunk_swizzle<E>(c);
#pragma unroll
  for (int b = 0; b < B; ++b) v[b] = xs[c * B + (b ^ key)];
}

// Everything a GEMV phase needs that does not depend on other CTAs' results of the previous phase:
// the matrix, this CTA's rows, where the input vector comes from and the epilogue.
struct GemvPlan {
  GemvDesc g;
  RowSplit rs;
  ActSrc src;
  Epi epi;
};

// Consumes one CTA's rows [rs.r0, rs.r1) of a matrix from the ring ("How I built an LLM inference
// engine from scratch in CUDA", v0.1 and "Round 1": a warp per row, 16-byte lane loads, several
// rows per warp; here the rows come from the shared-memory ring instead of global memory).
// A row is cut into nseg segments (seg_info); warp w owns segment w % nseg of rows
// w / nseg, w / nseg + NCW / nseg, ... of every stage, and keeps that segment's activations in
// registers for the whole matrix (lane owns chunks lane + 32 k). Per row: a warp dot product and a
// butterfly reduction. The LM head applies its epilogue in the warp; every other matrix leaves its
// per-segment row results in shared memory, and one pass at the end of the phase sums the
// segments in a fixed order and applies the epilogue (bias, residual add, SwiGLU on gate/up pairs).
// IF: input blocks in flight per thread while fetching the input vector (four: eight made the
// Llama-shaped bf16 step 8 % slower and the int4 instances spill).
// SEGMAJOR: segment-major stages (GemvDesc::nsegs blocks of GemvDesc::rbs-byte rows), one warp group
// per segment, and an epilogue that weighs the segment sums with epi.bias[s] before adding them in
// order (the gathered-expert down projection: segment s is expert s's row).
template <int FMT, int NCHL, int IF = 4, bool SEGMAJOR = false>
__device__ __forceinline__ bool gemv_rows(Pipe& pp, const GemvPlan& pl, Best& best, int tid,
                          unsigned long long* tr_ready) {
  constexpr int E = FMT == 0 ? 8 : 32;
  const GemvDesc& g = pl.g;
  const RowSplit& rs = pl.rs;
  const ActSrc& src = pl.src;
  const Epi& epi = pl.epi;
  Misc* ms = pp.ms;
  const int lane = tid & 31, warp = tid >> 5;
  const SegInfo si = SEGMAJOR ? SegInfo{g.nsegs, g.cols / g.nsegs, g.cols / g.nsegs / E} : seg_info(FMT, g.cols);
  const int seg = warp % si.nseg, grp = warp / si.nseg, WG = NCW / si.nseg;
  const int nrows = rs.r1 - rs.r0;
  const bool direct = epi.kind == EK_ARGMAX && si.nseg == 1;  // the warp holds whole rows
  const bool norm = src.gf || src.gb;
  // epilogue operand of row rs.r0 + tid, loaded now so that its latency hides under the fetch
  float pre = 0.f;
  if (!direct && tid < nrows && epi.kind != EK_ARGMAX) {
    if (epi.kind == EK_RESIDUAL) pre = residual_at(epi, rs.r0 + tid);
    else if (epi.kind == EK_STORE && epi.bias && !SEGMAJOR) pre = __ldg(epi.bias + rs.r0 + tid);
  }

  // the input vector (x * g for RMSNorm phases) into shared memory, then this warp's segment into
  // registers; 1 / rms(x) scales each row segment's sum instead (once per row, not per input).
  // Chunks past the segment read the segment's last chunk slot and are zeroed, so that the row loop
  // needs no per-lane branches
  if (tr_ready && tid == 0) tr_ready[TR_ENTRY - TR_READY] = globaltimer();
  const float inv = fetch_vector_n<IF>(pp, src, tid, FMT);
  if (tr_ready && tid == 0) tr_ready[TR_FETCHED - TR_READY] = globaltimer();
  if (*reinterpret_cast<volatile int*>(&pp.ms->abort)) return false;  // uniform after the fetch
  (void)norm;
  float a[NCHL][E];
  float S[NCHL];
  {
    const float4* xsv = sptr<float4>(pp.xs);
#pragma unroll
    for (int k = 0; k < NCHL; ++k) {
      const bool ok = lane + 32 * k < si.chs;
      const int c = min(lane + 32 * k, si.chs - 1);  // clamped chunk: always a valid address
      float4 v[E / 4];
      load_chunk<E>(xsv, (seg * si.ks) / E + c, v);
#pragma unroll
      for (int b = 0; b < E / 4; ++b) {
        a[k][4 * b + 0] = ok ? v[b].x : 0.f;
        a[k][4 * b + 1] = ok ? v[b].y : 0.f;
        a[k][4 * b + 2] = ok ? v[b].z : 0.f;
        a[k][4 * b + 3] = ok ? v[b].w : 0.f;
      }
    }
  }
  if (tr_ready && tid == 0) tr_ready[TR_ACT - TR_READY] = globaltimer() + (unsigned long long)(a[0][0] * 0.f);
  if (FMT == 1) {
    // the chunk's sum of (unscaled) inputs for the zero point, as a tree: the inputs arrive
    // pre-multiplied by 16^-(i mod 4), and scaling back by the same powers of two is exact
#pragma unroll
    for (int k = 0; k < NCHL; ++k) {
      float sb[E / 4];
#pragma unroll
      for (int b = 0; b < E / 4; ++b)
        sb[b] = fmaf(4096.f, a[k][4 * b + 3], fmaf(256.f, a[k][4 * b + 2], fmaf(16.f, a[k][4 * b + 1], a[k][4 * b])));
#pragma unroll
      for (int w = E / 8; w >= 1; w >>= 1)
#pragma unroll
        for (int b = 0; b < w; ++b) sb[b] += sb[b + w];
      S[k] = sb[0];
    }
  }
  if (tr_ready && tid == 0) *tr_ready = globaltimer();

  const uint32_t seg_off = SEGMAJOR ? 0u : FMT == 0 ? (uint32_t)(seg * si.ks * 2) : (uint32_t)(seg * si.ks / 2);
  const uint32_t mag = opaque_u32(0x4B000000u);  // int4 exponent-trick magic, kept in a register
  const uint32_t scale_off = (uint32_t)((SEGMAJOR ? si.ks : g.cols) / 2);
  // byte offsets inside a row of this lane's chunks (chunk k = lane + 32 k, clamped) and scales
  uint32_t coff[NCHL], soff[NCHL];
#pragma unroll
  for (int k = 0; k < NCHL; ++k) {
    const int c = min(lane + 32 * k, si.chs - 1);
    coff[k] = seg_off + (uint32_t)c * 16u;
    soff[k] = FMT == 1 ? scale_off + 2u * (uint32_t)(((SEGMAJOR ? 0 : seg * si.ks) + c * 32) / g.group) : 0u;
  }

  // The warp walks its rows stage by stage (rows grp, grp + WG, ... of each stage). Lane partials
  // of the last eight rows ride in a shift window; a full window is finished by one transposed
  // reduction (9 shuffles for 8 rows). Row ids follow from the warp's row counter: its n-th row is
  // row (n / m) * nr + grp + (n % m) * WG of the CTA's slice, m rows per full stage. A stage is
  // released as soon as the warp's last row in it has been read.
  const int m = rs.nr > grp ? (rs.nr - grp + WG - 1) / WG : 0;
  float w0 = 0.f, w1 = 0.f, w2 = 0.f, w3 = 0.f, w4 = 0.f, w5 = 0.f, w6 = 0.f, w7 = 0.f;
  int nrow = 0, filled = 0;
  auto flush = [&]() {
    const float part[8] = {w0, w1, w2, w3, w4, w5, w6, w7};
    const float v = transpose_reduce8(part, lane) * inv;  // the RMSNorm scale, once per row segment
    const int q8 = transpose_row8(lane);
    if ((lane & 3) == 0 && q8 < filled) {
      const int n = nrow - 1 - q8;  // slot q holds the warp's row nrow - 1 - q
      const int rl = (n / m) * rs.nr + grp + (n % m) * WG;
      if (direct) {
        const int r = rs.r0 + rl;
        if (epi.out) static_cast<float*>(epi.out)[r] = v;
        best_update(best, v, r);
      } else {
        ms->rowv[rl * si.nseg + seg] = v;
      }
    }
    w0 = w1 = w2 = w3 = w4 = w5 = w6 = w7 = 0.f;
    filled = 0;
  };
  for (int s0 = rs.r0; s0 < rs.r1; s0 += rs.nr) {
    const int nrs = min(rs.nr, rs.r1 - s0);
    const uint32_t st = cons_acquire(pp);
    if (tr_ready && tid == 0 && s0 == rs.r0) tr_ready[TR_AUX0 - TR_READY] = globaltimer();
    int i0 = grp;
#pragma unroll 1
    for (int i = i0; i < nrs; i += WG) {
      const uint32_t rowp = SEGMAJOR ? st + (uint32_t)(seg * nrs + i) * (uint32_t)g.rbs : st + (uint32_t)i * g.rb;
      float2 acc = make_float2(0.f, 0.f), acc2 = make_float2(0.f, 0.f);
      // every chunk is loaded unconditionally (clamped offsets, zero activations past the row), so
      // that all loads of the row issue back to back
      uint4 wv[NCHL];
#pragma unroll
      for (int k = 0; k < NCHL; ++k) wv[k] = lds128(rowp + coff[k]);
#pragma unroll
      for (int k = 0; k < NCHL; ++k) {
        if (FMT == 0) {
          if (k & 1) acc2 = dot8_bf16(wv[k], a[k], acc2);
          else acc = dot8_bf16(wv[k], a[k], acc);
        } else {
          const float dq = dot32_int4(wv[k], a[k], mag);
          const uint16_t sb = lds16(rowp + soff[k]);
          const float sc = g.scale_bf16 ? bf16_to_f(sb) : __half2float(__ushort_as_half(sb));
          acc.x = fmaf(sc, dq - 8.f * S[k], acc.x);
        }
      }
      // shift the window: the newest row enters at w0
      w7 = w6; w6 = w5; w5 = w4; w4 = w3; w3 = w2; w2 = w1; w1 = w0;
      w0 = (acc.x + acc.y) + (acc2.x + acc2.y);
      ++nrow;
      if (++filled == 8) flush();
    }
    cons_release(pp, lane);
  }
  if (tr_ready && tid == 0) tr_ready[TR_AUX1 - TR_READY] = globaltimer();
  if (filled) flush();
  if (direct) return true;
  named_sync(BAR_CONS, NCT);
  if (epi.kind == EK_SWIGLU) {
    for (int p = tid; p < nrows / 2; p += NCT) {
      float gt = 0.f, up = 0.f;
      for (int s2 = 0; s2 < si.nseg; ++s2) gt += ms->rowv[(2 * p) * si.nseg + s2];
      for (int s2 = 0; s2 < si.nseg; ++s2) up += ms->rowv[(2 * p + 1) * si.nseg + s2];
      epi_write(epi, rs.r0 / 2 + p, gt / (1.f + expf(-gt)) * up);
    }
  } else {
    for (int t = tid; t < nrows; t += NCT) {
      float v = 0.f;
      if (SEGMAJOR) {
        for (int s2 = 0; s2 < si.nseg; ++s2) v = fmaf(__ldg(epi.bias + s2), ms->rowv[t * si.nseg + s2], v);
      } else {
        for (int s2 = 0; s2 < si.nseg; ++s2) v += ms->rowv[t * si.nseg + s2];
      }
      const int r = rs.r0 + t;
      if (epi.kind == EK_ARGMAX) {
        if (epi.out) static_cast<float*>(epi.out)[r] = v;
        best_update(best, v, r);
        continue;
      }
      float base = pre;
      const bool row_bias = epi.bias && !SEGMAJOR;  // segment-major: bias holds the segment weights
      if (t >= NCT) base = epi.kind == EK_RESIDUAL ? residual_at(epi, r) : (row_bias ? epi.bias[r] : 0.f);
      epi_write(epi, r, (epi.kind == EK_RESIDUAL || row_bias) ? base + v : v);
    }
  }
  return true;
}

// The MLP's down projection split by columns ("Decoding in tiles", section 4: each worker
// multiplies its SwiGLU rows by the matching columns of the down projection, an fp32 partial sum of
// every output, and an FFN-reduce task sums the partials in a fixed order and adds the residual).
// pl.g is Wd^T with this CTA's ffn inputs [rs.r0, rs.r1) as rows; their SwiGLU values are this
// CTA's own results of the gate/up phase (the same split), read from pl.src.xw after a barrier.
// Thread t accumulates hidden outputs [8 c, 8 c + 8) for chunks c = t, t + NCT (row by row, in
// order), publishes them as stamped words (the gate/up phase's stamp, which nothing else uses in
// this mode), and the CTA then reduces its output rows ro over every CTA's partials: sixteen lanes
// per row, lane s summing the partials of CTAs s, s + 16, ... in order, a fixed xor tree over the
// sixteen, the residual added last. So the gate/up results never cross CTAs, and the reduce is
// the only hand-off between the gate/up and the next phase. False when a partial never showed up.
__device__ __forceinline__ bool colsplit_down(Pipe& pp, const GemvPlan& pl, const RowSplit& ro, uint64_t* part,
                                           int grid, int tid) {
  constexpr int CPT = 2;  // 8-output chunks per thread: hidden sizes up to 16 * NCT
  Misc* ms = pp.ms;
  const GemvDesc& g = pl.g;
  const RowSplit& rs = pl.rs;
  const Epi& epi = pl.epi;
  const int H = g.cols, nchunk = H / 8, nrows = rs.r1 - rs.r0;
  const unsigned ps = epi.stamp - 1u;
  float* act_s = sptr_w<float>(smem_addr(ms->rowv));
  named_sync(BAR_CONS, NCT);  // the gate/up epilogue has written every SwiGLU value of this CTA
  for (int t = tid; t < nrows; t += NCT) act_s[t] = word_value(ld_relaxed_u64(pl.src.xw + rs.r0 + t));
  named_sync(BAR_CONS, NCT);
  float2 acc[CPT][4];
#pragma unroll
  for (int c = 0; c < CPT; ++c)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[c][e] = make_float2(0.f, 0.f);
  const int lane = tid & 31;
  for (int s0 = rs.r0; s0 < rs.r1; s0 += rs.nr) {
    const int nrs = min(rs.nr, rs.r1 - s0);
    const uint32_t st = cons_acquire(pp);
#pragma unroll 1
    for (int i = 0; i < nrs; ++i) {
      const float a = act_s[s0 - rs.r0 + i];
      const float2 a2 = make_float2(a, a);
#pragma unroll
      for (int c = 0; c < CPT; ++c) {
        const int ch = tid + c * NCT;
        if (ch < nchunk) {
          const uint4 w = lds128(st + (uint32_t)i * g.rb + (uint32_t)ch * 16u);
          acc[c][0] = fma2(a2, make_float2(bf16_lo(w.x), bf16_hi(w.x)), acc[c][0]);
          acc[c][1] = fma2(a2, make_float2(bf16_lo(w.y), bf16_hi(w.y)), acc[c][1]);
          acc[c][2] = fma2(a2, make_float2(bf16_lo(w.z), bf16_hi(w.z)), acc[c][2]);
          acc[c][3] = fma2(a2, make_float2(bf16_lo(w.w), bf16_hi(w.w)), acc[c][3]);
        }
      }
    }
    cons_release(pp, lane);
  }
  uint64_t* mine = part + (size_t)blockIdx.x * H;
#pragma unroll
  for (int c = 0; c < CPT; ++c) {
    const int ch = tid + c * NCT;
    if (ch < nchunk) {
#pragma unroll
      for (int e = 0; e < 4; ++e)
        st_relaxed_v2u64(mine + ch * 8 + 2 * e, stamp_word(acc[c][e].x, ps), stamp_word(acc[c][e].y, ps));
    }
  }
  // the reduce: two rows per warp and turn (one per half-warp), every lane in every shuffle
  const int warp = tid >> 5, half = lane >> 4, sub = lane & 15;
  const int nout = ro.r1 - ro.r0;
  constexpr int PER = 16;  // partials per lane: grids up to 256 CTAs
  for (int rb = 2 * warp; rb < nout; rb += 2 * NCW) {
    const int rr = rb + half;
    const bool on = rr < nout;
    const int r = ro.r0 + rr;
    uint64_t w[PER];
    unsigned need = 0;
#pragma unroll
    for (int e = 0; e < PER; ++e) {
      const int cta = sub + 16 * e;
      if (on && cta < grid) {
        w[e] = ld_relaxed_u64(part + (size_t)cta * H + r);
        need |= 1u << e;
      } else {
        w[e] = 0;
      }
    }
    {
      unsigned stale = 0;
#pragma unroll
      for (int e = 0; e < PER; ++e)
        if ((need & (1u << e)) && word_stamp(w[e]) != ps) stale |= 1u << e;
      Poll pl2;
      while (stale && pl2.again(pp)) {
#pragma unroll
        for (int e = 0; e < PER; ++e)
          if (stale & (1u << e)) w[e] = ld_relaxed_u64(part + (size_t)(sub + 16 * e) * H + r);
#pragma unroll
        for (int e = 0; e < PER; ++e)
          if ((stale & (1u << e)) && word_stamp(w[e]) == ps) stale &= ~(1u << e);
      }
    }
    float v = 0.f;
#pragma unroll
    for (int e = 0; e < PER; ++e)
      if (need & (1u << e)) v += word_value(w[e]);
#pragma unroll
    for (int o = 8; o; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    if (on && sub == 0) epi_write(epi, r, residual_at(epi, r) + v);
  }
  named_sync(BAR_CONS, NCT);
  return !*reinterpret_cast<volatile int*>(&ms->abort);
}

// GEMV over MV activation vectors at once, the verify shape of speculative decoding (flint,
// "speculative decode": the megakernel verifies K + 1 tokens in one launch with the weights read
// once): y[j][r] = sum_c W[r][c] x[j][c] for j < MV, fp32 accumulation. A lane keeps the
// activations of all MV vectors for its part of a row segment in registers (NCH = 8 / MV units of
// 8 inputs: 16-byte bf16 chunks, or 4-byte int4 words), so a row segment holds at most 2048 / MV
// inputs and the weights of a row are decoded once for all MV vectors. int4 words are decoded in
// place as for one vector (2^23 + q 16^i, activations pre-multiplied by 16^-i), with the zero
// point subtracted exactly as 2^23 + 8 16^i and the scale applied to the decoded values, so each
// product is (q - 8) s x rounded once. Row partials of 8 / MV rows ride in one window and meet in
// one transposed reduction; the epilogue sums a row's segments in order (STORE with an optional
// row bias, or RESIDUAL: y += .).
struct GemvMArgs {
  const float* x;      // [MV][cols]
  float* y;            // [MV][rows]
  const float* bias;   // [rows] or null
  int residual;
  int nseg;            // segments per row (a power of two dividing NCW)
};
template <int FMT, int MV>
__device__ __forceinline__ bool gemv_rows_m(Pipe& pp, const GemvDesc& g, const RowSplit& rs, const GemvMArgs& q,
                                            int tid) {
  constexpr int NCH = 8 / MV;    // units per lane and segment
  Misc* ms = pp.ms;
  const int lane = tid & 31, warp = tid >> 5;
  const int nseg = q.nseg, ks = g.cols / nseg, us = ks / 8;  // inputs and units per segment
  const int seg = warp % nseg, grp = warp / nseg, WG = NCW / nseg;
  const int nrows = rs.r1 - rs.r0;
  // the MV input vectors into shared memory, then this lane's units into registers
  float* xs = sptr_w<float>(pp.xs);
  for (int i = tid; i < MV * g.cols / 4; i += NCT)
    reinterpret_cast<float4*>(xs)[i] = __ldcg(reinterpret_cast<const float4*>(q.x) + i);
  named_sync(BAR_CONS, NCT);
  // unit k of the lane: bf16 u = lane + 32 k (lanes read consecutive 16-byte chunks); int4
  // u = lane * NCH + k (a lane's words are consecutive: one vector load)
  float a[MV][NCH][8];
#pragma unroll
  for (int k = 0; k < NCH; ++k) {
    const int u = FMT == 0 ? lane + 32 * k : lane * NCH + k;
    const bool ok = u < us;
    const int uc = ok ? u : 0;
#pragma unroll
    for (int j = 0; j < MV; ++j) {
      const float* src = xs + j * g.cols + seg * ks + uc * 8;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float v = ok ? src[e] : 0.f;
        a[j][k][e] = FMT == 0 ? v : v * ((e & 3) == 0 ? 1.f : (e & 3) == 1 ? 0.0625f : (e & 3) == 2 ? 0.00390625f : 0.000244140625f);
      }
    }
  }
  // once every warp holds its activations, the input buffer (m * cols floats) takes the row results
  // when it is the larger of the two buffers
  named_sync(BAR_CONS, NCT);
  float* rowv = MV * g.cols > ROWV_MAX ? xs : ms->rowv;
  const uint32_t mag = opaque_u32(0x4B000000u);
  const float2 B01 = make_float2(-8388616.f, -8388736.f);    // -(2^23 + 8 * 16^i), i = 0, 1
  const float2 B23 = make_float2(-8390656.f, -8421376.f);    // i = 2, 3
  const uint32_t seg_off = FMT == 0 ? (uint32_t)(seg * ks * 2) : (uint32_t)(seg * ks / 2);
  const int m = rs.nr > grp ? (rs.nr - grp + WG - 1) / WG : 0;  // rows of the warp per full stage
  constexpr int R = 8 / MV;                                     // rows per reduction window
  float w[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) w[e] = 0.f;
  int rl[R];
  int filled = 0, nrow = 0;
  auto flush = [&]() {
    const float v = transpose_reduce8(w, lane);
    const int qv = transpose_row8(lane), rr = qv / MV, j = qv % MV;
    if ((lane & 3) == 0 && rr < filled) rowv[(rl[rr] * nseg + seg) * MV + j] = v;
#pragma unroll
    for (int e = 0; e < 8; ++e) w[e] = 0.f;
    filled = 0;
  };
  for (int s0 = rs.r0; s0 < rs.r1; s0 += rs.nr) {
    const int nrs = min(rs.nr, rs.r1 - s0);
    const uint32_t st = cons_acquire(pp);
#pragma unroll 1
    for (int i = grp; i < nrs; i += WG) {
      const uint32_t rowp = st + (uint32_t)i * g.rb + seg_off;
      float2 acc[MV];
#pragma unroll
      for (int j = 0; j < MV; ++j) acc[j] = make_float2(0.f, 0.f);
      if (FMT == 0) {
#pragma unroll
        for (int k = 0; k < NCH; ++k) {
          const int u = min(lane + 32 * k, us - 1);
          const uint4 wv = lds128(rowp + (uint32_t)u * 16u);
          const float2 p0 = make_float2(bf16_lo(wv.x), bf16_hi(wv.x)), p1 = make_float2(bf16_lo(wv.y), bf16_hi(wv.y));
          const float2 p2 = make_float2(bf16_lo(wv.z), bf16_hi(wv.z)), p3 = make_float2(bf16_lo(wv.w), bf16_hi(wv.w));
#pragma unroll
          for (int j = 0; j < MV; ++j) {
            acc[j] = fma2(p0, make_float2(a[j][k][0], a[j][k][1]), acc[j]);
            acc[j] = fma2(p1, make_float2(a[j][k][2], a[j][k][3]), acc[j]);
            acc[j] = fma2(p2, make_float2(a[j][k][4], a[j][k][5]), acc[j]);
            acc[j] = fma2(p3, make_float2(a[j][k][6], a[j][k][7]), acc[j]);
          }
        }
      } else {
        const int u0 = lane * NCH < us ? lane * NCH : 0;  // a lane past the segment reads word 0 (zero activations)
        uint32_t wd[NCH];
        if (NCH == 4) {
          const uint4 v = lds128(rowp + (uint32_t)u0 * 4u);
          wd[0] = v.x; wd[NCH > 1 ? 1 : 0] = v.y; wd[NCH > 2 ? 2 : 0] = v.z; wd[NCH > 3 ? 3 : 0] = v.w;
        } else {
#pragma unroll
          for (int k = 0; k < NCH; ++k) wd[k] = lds32(rowp + (uint32_t)(u0 + k) * 4u);
        }
#pragma unroll
        for (int k = 0; k < NCH; ++k) {
          const int col = seg * ks + (u0 + k) * 8;
          const uint16_t sb = lds16(st + (uint32_t)i * g.rb + (uint32_t)(g.cols / 2) + 2u * (uint32_t)(col / g.group));
          const float sc = g.scale_bf16 ? bf16_to_f(sb) : __half2float(__ushort_as_half(sb));
          const float2 s2 = make_float2(sc, sc);
          const uint32_t lo = wd[k], hi = wd[k] >> 16;
          const float2 d01 = __fmul2_rn(add2(make_float2(__uint_as_float(and_or<0x000Fu>(lo, mag)), __uint_as_float(and_or<0x00F0u>(lo, mag))), B01), s2);
          const float2 d23 = __fmul2_rn(add2(make_float2(__uint_as_float(and_or<0x0F00u>(lo, mag)), __uint_as_float(and_or<0xF000u>(lo, mag))), B23), s2);
          const float2 d45 = __fmul2_rn(add2(make_float2(__uint_as_float(and_or<0x000Fu>(hi, mag)), __uint_as_float(and_or<0x00F0u>(hi, mag))), B01), s2);
          const float2 d67 = __fmul2_rn(add2(make_float2(__uint_as_float(and_or<0x0F00u>(hi, mag)), __uint_as_float(and_or<0xF000u>(hi, mag))), B23), s2);
#pragma unroll
          for (int j = 0; j < MV; ++j) {
            acc[j] = fma2(d01, make_float2(a[j][k][0], a[j][k][1]), acc[j]);
            acc[j] = fma2(d23, make_float2(a[j][k][2], a[j][k][3]), acc[j]);
            acc[j] = fma2(d45, make_float2(a[j][k][4], a[j][k][5]), acc[j]);
            acc[j] = fma2(d67, make_float2(a[j][k][6], a[j][k][7]), acc[j]);
          }
        }
      }
      // the row's MV partials enter the window at slots filled * MV + j
      const int n = nrow++;
      const int rlocal = (n / m) * rs.nr + grp + (n % m) * WG;
#pragma unroll
      for (int rr = 0; rr < R; ++rr)
        if (rr == filled) {
          rl[rr] = rlocal;
#pragma unroll
          for (int j = 0; j < MV; ++j) w[rr * MV + j] = acc[j].x + acc[j].y;
        }
      if (++filled == R) flush();
    }
    cons_release(pp, lane);
  }
  if (filled) flush();
  named_sync(BAR_CONS, NCT);
  for (int t = tid; t < nrows * MV; t += NCT) {
    const int row = t / MV, j = t - row * MV, r = rs.r0 + row;
    float v = 0.f;
    for (int s2 = 0; s2 < nseg; ++s2) v += rowv[(row * nseg + s2) * MV + j];
    float* out = q.y + (size_t)j * g.rows + r;
    if (q.residual) *out = __ldcg(out) + v;
    else *out = q.bias ? q.bias[r] + v : v;
  }
  return !*reinterpret_cast<volatile int*>(&ms->abort);
}

// Dispatch to the instance of the weight format and chunk count per lane (rounded up to even).
__device__ __forceinline__ bool gemv_consume_any(Pipe& pp, const GemvPlan& pl, Best& best, int tid,
                                                 unsigned long long* tr_ready) {
  if (pl.g.fmt == 1) return gemv_rows<1, 2>(pp, pl, best, tid, tr_ready);
  const int nchl = (seg_info(0, pl.g.cols).chs + 31) / 32;
  if (nchl > 6) return gemv_rows<0, 8>(pp, pl, best, tid, tr_ready);
  if (nchl > 4) return gemv_rows<0, 6>(pp, pl, best, tid, tr_ready);
  if (nchl > 2) return gemv_rows<0, 4>(pp, pl, best, tid, tr_ready);
  return gemv_rows<0, 2>(pp, pl, best, tid, tr_ready);
}

__device__ __forceinline__ void produce_rows(Pipe& pp, const GemvDesc& g, const RowSplit& rs,
                                             uint64_t pol, bool& dead) {
  for (int s0 = rs.r0; s0 < rs.r1; s0 += rs.nr) {
    const int nrs = min(rs.nr, rs.r1 - s0);
    prod_push(pp, g.w + (size_t)s0 * g.rb, (uint32_t)(nrs * g.rb), pol, dead);
  }
}

// Per-CTA (max, lowest index, non-finite) over the consumer threads. Result valid in thread 0.
__device__ __forceinline__ Best best_block_reduce(Best b, Misc* ms, int tid) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float ov = __shfl_xor_sync(0xFFFFFFFFu, b.v, o);
    const int oi = __shfl_xor_sync(0xFFFFFFFFu, b.i, o);
    const int ob = __shfl_xor_sync(0xFFFFFFFFu, b.bad, o);
    if (ov > b.v || (ov == b.v && oi < b.i)) { b.v = ov; b.i = oi; }
    b.bad |= ob;
  }
  if ((tid & 31) == 0) { ms->bv[tid >> 5] = b.v; ms->bi[tid >> 5] = b.i; ms->bbad[tid >> 5] = b.bad; }
  named_sync(BAR_CONS, NCT);
  Best r{-CUDART_INF_F, 0x7FFFFFFF, 0};
  if (tid == 0) {
    for (int w = 0; w < NCW; ++w) {
      if (ms->bv[w] > r.v || (ms->bv[w] == r.v && ms->bi[w] < r.i)) { r.v = ms->bv[w]; r.i = ms->bi[w]; }
      r.bad |= ms->bbad[w];
    }
  }
  named_sync(BAR_CONS, NCT);
  return r;
}

// Argmax across CTAs: each CTA publishes its best in slot `cta`; the last CTA to take a ticket
// combines all slots (order-independent: max value, then lowest index) and writes the token, or -1
// and the non-finite error bit ("Decoding in tiles", section 5: per-task best candidates, lowest
// token id among ties, an error word on a non-finite logit).
static __device__ void argmax_publish(const Best& mine, float* slot_v, int* slot_i, int* slot_bad,
                               unsigned* ticket, int nslots, int cta, int* out, int* err,
                               int* err_host, Misc* ms, int tid) {
  if (tid == 0) {
    slot_v[cta] = mine.v;
    slot_i[cta] = mine.i;
    slot_bad[cta] = mine.bad;
    const unsigned old = atom_add_acq_rel(ticket, 1u);
    ms->flag = (old == (unsigned)nslots - 1);
  }
  named_sync(BAR_CONS, NCT);
  if (ms->flag && tid < 32) {
    Best b{-CUDART_INF_F, 0x7FFFFFFF, 0};
    for (int s = tid; s < nslots; s += 32) {
      const float v = __ldcg(slot_v + s);
      const int i = __ldcg(slot_i + s);
      if (v > b.v || (v == b.v && i < b.i)) { b.v = v; b.i = i; }
      b.bad |= __ldcg(slot_bad + s);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float ov = __shfl_xor_sync(0xFFFFFFFFu, b.v, o);
      const int oi = __shfl_xor_sync(0xFFFFFFFFu, b.i, o);
      const int ob = __shfl_xor_sync(0xFFFFFFFFu, b.bad, o);
      if (ov > b.v || (ov == b.v && oi < b.i)) { b.v = ov; b.i = oi; }
      b.bad |= ob;
    }
    if (tid == 0) {
      *out = b.bad ? -1 : b.i;
      if (b.bad) raise_error(err, err_host, EW_NONFINITE);
      atomicExch(ticket, 0u);
    }
  }
  named_sync(BAR_CONS, NCT);
}

// ------------------------------------------------------------------------------ attention

struct AttnSplit {
  int nch;  // chunks per KV head
  int cl;   // slots per chunk
};

// Split of [0, pos] into chunks: enough chunks that the units (KV head, chunk) cover the grid, each
// chunk no longer than min(slot / (2 d), T_MAX) positions (its keys fill at most one ring slot). The
// unit's work is latency-bound, so spreading it over every SM beats fewer, longer chunks even with
// the merge's extra partials. override_nch > 0 fixes the count (single-op tests).
__device__ __forceinline__ AttnSplit attn_split(int pos, int nkv, int d, int grid, int slot,
                                                int override_nch) {
  const int n_ctx = pos + 1;
  int tmax = slot / (2 * d);
  if (tmax > T_MAX) tmax = T_MAX;
  int nch;
  if (override_nch > 0) {
    nch = override_nch;
  } else {
    const int nmin = (n_ctx + tmax - 1) / tmax;
    int want = grid / nkv;
    if (want < 1) want = 1;
    if (want > n_ctx) want = n_ctx;
    if (want > T_MAX) want = T_MAX;
    nch = nmin > want ? nmin : want;
  }
  return AttnSplit{nch, (n_ctx + nch - 1) / nch};
}

struct AttnArgs {
  const float* qkv;        // [q | k | v] raw projections (single operation), or
  const uint64_t* qkvw = nullptr;  // the same as stamped words (the step): wait for stamp_in
  unsigned stamp_in = 0;
  int check = 0;
  uint64_t* outw = nullptr;        // stamped output (the step), written with stamp_out
  unsigned stamp_out = 0;
  // sliced merge (persistent kernel): partials as stamped words, no ticket; every unit then
  // merges a slice of its head's outputs (attn_merge_slice)
  uint64_t* pmw = nullptr;
  uint64_t* plw = nullptr;
  uint64_t* pow_ = nullptr;
  uint16_t* kc;            // this layer's K cache [nkv][max_ctx][d]
  uint16_t* vc;
  const float2* rope;      // RoPE table rows [rope_pos0, ...][d/2]
  int rope_pos0 = 0;       // position of the table's first row (0: the full table)
  float* part_m;
  float* part_l;
  float* part_o;
  int nch_cap;
  unsigned* tickets;       // [nkv]
  float* out;              // [nq * d]
  int nq, nkv, d, max_ctx, pos;
};

__device__ __forceinline__ void produce_attn_unit(Pipe& pp, const AttnArgs& A, int j, int c,
                                                  const AttnSplit& sp, uint64_t pol, bool& dead) {
  const int t0 = c * sp.cl;
  int tend = t0 + sp.cl;
  if (tend > A.pos) tend = A.pos;  // the slot at pos is written in this step: never streamed
  const int nk = tend > t0 ? tend - t0 : 0;
  const size_t base = ((size_t)j * A.max_ctx + t0) * A.d;
  prod_push(pp, A.kc + base, (uint32_t)(nk * A.d * 2), pol, dead);
  prod_push(pp, A.vc + base, (uint32_t)(nk * A.d * 2), pol, dead);
}

// One batch (32 chunks, lane = chunk) of the log-sum-exp combine: running maximum M, numerator and
// denominator, with explicit roundings so that every merge computes the same bits.
__device__ __forceinline__ void merge_step(float& M, float& num, float& den, float m, float l, float v) {
  const float Mn = fmaxf(M, warp_max(m));
  const float keep = M == -CUDART_INF_F ? 0.f : expf(M - Mn);
  const float w = m == -CUDART_INF_F ? 0.f : expf(m - Mn);  // an empty chunk weighs exactly 0
  num = __fmaf_rn(num, keep, warp_sum(__fmul_rn(w, v)));
  den = __fmaf_rn(den, keep, warp_sum(__fmul_rn(w, l)));
  M = Mn;
}

// One merged attention output (the log-sum-exp combine of a head's chunk partials for one
// dimension): lanes over chunks, 32 at a time, combined with a running maximum. part(cc, m, l, v)
// delivers chunk cc's max, sum and output value. Both merges (ticket and sliced) follow it, so that
// the persistent kernel and the per-phase kernels produce the same bits. Result in every lane.
template <class Part>
__device__ __forceinline__ float merge_one(int nch, int lane, Part part) {
  float M = -CUDART_INF_F, num = 0.f, den = 0.f;
  for (int cb = 0; cb < nch; cb += 32) {
    const int cc = cb + lane;
    float m = -CUDART_INF_F, l = 0.f, v = 0.f;
    if (cc < nch) part(cc, m, l, v);
    merge_step(M, num, den, m, l, v);
  }
  return num / den;
}

// The sum warp_sum leaves in every lane, computed by one thread from the 32 lane values: the same
// xor butterfly (partners 16, 8, 4, 2, 1), so the same additions in the same order, the same bits.
__device__ __forceinline__ float butterfly_sum32(float (&v)[32]) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
#pragma unroll
    for (int i = 0; i < o; ++i) v[i] = v[i] + v[i + o];
  }
  return v[0];
}

// Merge of one KV head's chunk partials for its query heads by the CTA that took the head's last
// ticket (per-phase kernels). Warp g computes head g's chunk weights and denominator exactly as
// merge_one does; then one thread per output repeats merge_one's numerator with butterfly_sum32,
// so that the result has merge_one's bits while the G * d outputs are computed in parallel.
static __device__ void attn_merge(const AttnArgs& A, Misc* ms, int tid, int j, int nch) {
  const int G = A.nq / A.nkv, d = A.d;
  const int warp = tid >> 5, lane = tid & 31;
  const int nb = (nch + 31) / 32;
  float* w = ms->at.sc;     // [g][c] chunk weights
  float* keep = ms->at.qs;  // [g][batch] rescale of the running sums
  if (warp < G) {
    const int h = j * G + warp;
    float M = -CUDART_INF_F, den = 0.f;
    for (int b = 0; b < nb; ++b) {
      const int cc = 32 * b + lane;
      float m = -CUDART_INF_F, l = 0.f;
      if (cc < nch) {
        m = __ldcg(A.part_m + (size_t)h * A.nch_cap + cc);
        l = __ldcg(A.part_l + (size_t)h * A.nch_cap + cc);
      }
      const float Mn = fmaxf(M, warp_max(m));
      const float kp = M == -CUDART_INF_F ? 0.f : expf(M - Mn);
      const float wc = m == -CUDART_INF_F ? 0.f : expf(m - Mn);
      if (cc < nch) w[warp * T_MAX + cc] = wc;
      if (lane == 0) keep[warp * (T_MAX / 32) + b] = kp;
      den = __fmaf_rn(den, kp, warp_sum(__fmul_rn(wc, l)));
      M = Mn;
    }
    if (lane == 0) ms->hl[warp] = den;
  }
  named_sync(BAR_CONS, NCT);
  for (int o = tid; o < G * d; o += NCT) {
    const int g = o / d, i = o - g * d, h = j * G + g;
    const float* po = A.part_o + (size_t)h * A.nch_cap * d + i;
    float num = 0.f;
    for (int b = 0; b < nb; ++b) {
      float t[32];
#pragma unroll
      for (int q = 0; q < 32; ++q) {
        const int cc = 32 * b + q;
        t[q] = cc < nch ? __fmul_rn(w[g * T_MAX + cc], __ldcg(po + (size_t)cc * d)) : 0.f;
      }
      num = __fmaf_rn(num, keep[g * (T_MAX / 32) + b], butterfly_sum32(t));
    }
    const float r = num / ms->hl[g];
    const size_t oi = (size_t)h * d + i;
    if (A.outw) st_relaxed_u64(A.outw + oi, stamp_word(r, A.stamp_out));
    else A.out[oi] = r;
  }
}

// Scores of the cached positions [0, nk) and, when T > nk, of the new position (from kn), for heads
// g < G into sc[g][t]. Lane groups of LG = d / 8 lanes take one position each: lane li holds dims
// [8 li, 8 li + 8) of GP >= G query heads in registers and loads one 16-byte key chunk (a warp reads
// 32 / LG consecutive rows: no bank conflicts). The GP partial sums then meet by a reduce-scatter
// over the group (each level halves the values a lane keeps), which leaves head li / (LG / GP) in
// lane li after log2(GP) + log2(LG / GP) shuffles per position instead of GP * log2(LG).
// A warp takes two positions per lane group and loop turn, with no branch between them, so that the
// two dependent chains (key load, dot products, shuffles) overlap: the step is latency-bound.
template <int GP, int LG>
__device__ __forceinline__ void attn_scores_groups(uint32_t kst, const float* qs, const float* kn,
                                                   float* sc, int nk, int T, int G, int tid) {
  static_assert(GP <= LG, "a lane keeps at least one head");
  constexpr int D = LG * 8, PW = 32 / LG, NW = NCT / 32, STEP = NW * PW;
  const int lane = tid & 31, warp = tid >> 5;
  const int li = lane % LG, pl = lane / LG;
  float qr[GP][8];
#pragma unroll
  for (int g = 0; g < GP; ++g) {
    const float4 a = *reinterpret_cast<const float4*>(qs + g * D + li * 8);
    const float4 b = *reinterpret_cast<const float4*>(qs + g * D + li * 8 + 4);
    const bool on = g < G;
    qr[g][0] = on ? a.x : 0.f; qr[g][1] = on ? a.y : 0.f; qr[g][2] = on ? a.z : 0.f; qr[g][3] = on ? a.w : 0.f;
    qr[g][4] = on ? b.x : 0.f; qr[g][5] = on ? b.y : 0.f; qr[g][6] = on ? b.z : 0.f; qr[g][7] = on ? b.w : 0.f;
  }
  // the new position's key chunk (read only where t == nk; stale but unused in a chunk without pos)
  float kn8[8];
  {
    const float4 a = *reinterpret_cast<const float4*>(kn + li * 8);
    const float4 b = *reinterpret_cast<const float4*>(kn + li * 8 + 4);
    kn8[0] = a.x; kn8[1] = a.y; kn8[2] = a.z; kn8[3] = a.w; kn8[4] = b.x; kn8[5] = b.y; kn8[6] = b.z; kn8[7] = b.w;
  }
  const uint4* Ks = sptr<uint4>(kst);
  const int kl = nk > 0 ? nk - 1 : 0;  // rows past the cached ones read row kl: always in the stage
  // key chunk of position t: cached row, the new key, or zeros past the chunk (result unused)
  auto key = [&](int t, float (&k8)[8]) {
    const uint4 kv = Ks[(size_t)min(t, kl) * LG + li];
    const float c[8] = {bf16_lo(kv.x), bf16_hi(kv.x), bf16_lo(kv.y), bf16_hi(kv.y),
                        bf16_lo(kv.z), bf16_hi(kv.z), bf16_lo(kv.w), bf16_hi(kv.w)};
    const bool cached = t < nk, fresh = t < T;
#pragma unroll
    for (int e = 0; e < 8; ++e) k8[e] = cached ? c[e] : fresh ? kn8[e] : 0.f;
  };
  auto dots = [&](const float (&k8)[8], float (&v)[GP]) {
#pragma unroll
    for (int g = 0; g < GP; ++g) {
      float a = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) a = fmaf(qr[g][e], k8[e], a);
      v[g] = a;
    }
  };
  // reduce-scatter over the LG lanes of the group
  auto reduce = [&](float (&v)[GP]) {
#pragma unroll
    for (int n = GP, off = LG / 2; off > 0; off >>= 1) {
      const bool up = (li & off) != 0;
      if (n > 1) {
#pragma unroll
        for (int i = 0; i < GP / 2; ++i) {
          if (i < n / 2) {
            const float send = up ? v[i] : v[i + n / 2];
            const float keep = up ? v[i + n / 2] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
          }
        }
        n /= 2;
      } else {
        v[0] += __shfl_xor_sync(0xffffffffu, v[0], off);
      }
    }
  };
  const int head = li / (LG / GP);
  const bool writer = li % (LG / GP) == 0 && head < G;
  for (int tb = warp * PW; tb < T; tb += 2 * STEP) {
    const int ta = tb + pl, tc = tb + STEP + pl;
    float ka[8], kc[8], va[GP], vc[GP];
    key(ta, ka);
    key(tc, kc);
    dots(ka, va);
    dots(kc, vc);
    reduce(va);
    reduce(vc);
    if (writer && ta < T) sc[head * T_MAX + ta] = va[0];
    if (writer && tc < T) sc[head * T_MAX + tc] = vc[0];
  }
}

// The same scores, one thread per (head, position) with a full dot product (any d multiple of 8);
// key chunks in a rotated order so that the lanes of a quarter-warp hit distinct banks.
__device__ __forceinline__ void attn_scores_threads(uint32_t kst, const float* qs, const float* kn,
                                                    float* sc, int nk, int T, int G, int d, int tid) {
  const uint4* Ks = sptr<uint4>(kst);
  const int nc = d / 8;
  for (int idx = tid; idx < G * T; idx += NCT) {
    const int g = idx / T, t = idx - g * T;
    const float* qg = qs + g * d;
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
    if (t < nk) {
      const uint4* krow = Ks + (size_t)t * nc;
      int ch = t % nc;
      for (int cc = 0; cc < nc; ++cc) {
        const uint4 kv = krow[ch];
        const float4 qa = *reinterpret_cast<const float4*>(qg + ch * 8);
        const float4 qb = *reinterpret_cast<const float4*>(qg + ch * 8 + 4);
        a0 = fmaf(qa.x, bf16_lo(kv.x), a0);
        a1 = fmaf(qa.y, bf16_hi(kv.x), a1);
        a2 = fmaf(qa.z, bf16_lo(kv.y), a2);
        a3 = fmaf(qa.w, bf16_hi(kv.y), a3);
        a0 = fmaf(qb.x, bf16_lo(kv.z), a0);
        a1 = fmaf(qb.y, bf16_hi(kv.z), a1);
        a2 = fmaf(qb.z, bf16_lo(kv.w), a2);
        a3 = fmaf(qb.w, bf16_hi(kv.w), a3);
        ch = ch + 1 == nc ? 0 : ch + 1;
      }
    } else {
      for (int i = 0; i < d; i += 4) {
        a0 = fmaf(qg[i], kn[i], a0);
        a1 = fmaf(qg[i + 1], kn[i + 1], a1);
        a2 = fmaf(qg[i + 2], kn[i + 2], a2);
        a3 = fmaf(qg[i + 3], kn[i + 3], a3);
      }
    }
    sc[g * T_MAX + t] = (a0 + a1) + (a2 + a3);
  }
}

// One attention unit: KV head j, chunk c. RoPE on the group's queries (and, in the chunk holding
// pos, on the new key, which is written to the cache with the new value), scores over the chunk,
// per-head max / exponentials / sum, the value sum, and the partial (m, l, o) of the chunk
// ("One launch per token", "The attention trap"; "How I built an LLM inference engine", "Round 2":
// one unit per KV head and chunk serving all grouped query heads, K/V read once). With plain
// partials (per-phase kernels) the last CTA done with head j merges; with stamped partials (the
// persistent kernel) every unit later merges a slice of its head (attn_merge_slice). The work is
// spread so that no step waits on a long dependent chain:
//   scores: d / 8 lanes per position holding the group's heads, two positions per turn
//           (attn_scores_groups); other head sizes one thread per (head, position);
//   softmax: one warp per head, its first 64 scores kept in registers;
//   values: one thread per (head, dimension pair), eight positions per turn into four accumulators.
// tr: optional timeline row of the phase (fields TR_READY, TR_ACT, TR_ENTRY, TR_AUX0, TR_FETCHED,
// TR_AUX1 receive the keys' arrival, the ends of the query set-up and the scores, the values'
// arrival, the end of the partials and the merge start).
static __device__ bool attn_unit(Pipe& pp, const AttnArgs& A, const AttnSplit& sp, int j, int c, int tid,
                                 unsigned long long* tr = nullptr) {
  Misc* ms = pp.ms;
  const int lane = tid & 31, warp = tid >> 5;
  const int d = A.d, half = d / 2, G = A.nq / A.nkv;
  const int pos = A.pos, n_ctx = pos + 1;
  const int t0 = c * sp.cl;
  const int t1 = min(t0 + sp.cl, n_ctx);
  const bool has_pos = t0 <= pos && pos < t1;
  const int nk = max(0, min(t1, pos) - t0);  // cached positions, streamed through the ring
  const int T = max(0, t1 - t0);             // positions of the chunk: nk, plus pos itself
  const float scale = 1.f / sqrtf((float)d);
  const float2* rt = A.rope + (size_t)(pos - A.rope_pos0) * half;
  const size_t qo = (size_t)j * G * d;                      // q of the group's heads
  const size_t ko = (size_t)A.nq * d + (size_t)j * d;       // k of KV head j
  const size_t vo = ko + (size_t)A.nkv * d;                 // v of KV head j
  // inputs: every load is issued first (stamped words, or plain floats as their bits); for stamped
  // words every stale one is then read again in the same turn until the QKV phase's stamps show
  auto raw = [&](size_t i) -> uint64_t {
    return A.qkvw ? ld_relaxed_u64(A.qkvw + i)
                  : (uint64_t)__float_as_uint(__ldcg(A.qkv + i));
  };
  float* qs = sptr_w<float>(smem_addr(ms->at.qs));
  float* sc = sptr_w<float>(smem_addr(ms->at.sc));
  float* kn = sptr_w<float>(smem_addr(ms->at.kn));
  float* vn = sptr_w<float>(smem_addr(ms->at.vn));

  constexpr int QR = (G_MAX * D_MAX / 2 + NCT - 1) / NCT;  // query pairs per thread, at most
  constexpr int NW = 2 * QR + 3;                            // words per thread: q pairs, k pair, v
  uint64_t wd[NW];
  size_t ix[NW];
  unsigned need = 0;  // the words this thread reads
#pragma unroll
  for (int r = 0; r < QR; ++r) {
    const int idx = tid + r * NCT;
    if (idx < G * half) {
      const int g = idx / half, i = idx - g * half;
      ix[2 * r] = qo + g * d + i;
      ix[2 * r + 1] = qo + g * d + i + half;
      need |= 3u << (2 * r);
    }
  }
  const bool hk = has_pos && tid < half, hv = has_pos && tid < d;
  if (hk) { ix[2 * QR] = ko + tid; ix[2 * QR + 1] = ko + tid + half; need |= 3u << (2 * QR); }
  if (hv) { ix[2 * QR + 2] = vo + tid; need |= 1u << (2 * QR + 2); }
#pragma unroll
  for (int e = 0; e < NW; ++e) wd[e] = (need & (1u << e)) ? raw(ix[e]) : 0;
  if (A.qkvw && A.check) {
    const unsigned sv = A.stamp_in;
    unsigned stale = 0;
#pragma unroll
    for (int e = 0; e < NW; ++e)
      if ((need & (1u << e)) && word_stamp(wd[e]) != sv) stale |= 1u << e;
    Poll pl;
    while (stale && pl.again(pp)) {
#pragma unroll
      for (int e = 0; e < NW; ++e)
        if (stale & (1u << e)) wd[e] = ld_relaxed_u64(A.qkvw + ix[e]);
#pragma unroll
      for (int e = 0; e < NW; ++e)
        if ((stale & (1u << e)) && word_stamp(wd[e]) == sv) stale &= ~(1u << e);
    }
  }
#pragma unroll
  for (int r = 0; r < QR; ++r) {
    const int idx = tid + r * NCT;
    if (idx < G * half) {
      const int g = idx / half, i = idx - g * half;
      const float x0 = word_value(wd[2 * r]), x1 = word_value(wd[2 * r + 1]);
      const float2 cs = rt[i];
      qs[g * d + i] = (x0 * cs.x - x1 * cs.y) * scale;
      qs[g * d + i + half] = (x1 * cs.x + x0 * cs.y) * scale;
    }
  }
  if (has_pos) {
    const size_t slot = ((size_t)j * A.max_ctx + pos) * d;
    if (hk) {
      const int i = tid;
      const float x0 = word_value(wd[2 * QR]), x1 = word_value(wd[2 * QR + 1]);
      const float2 cs = rt[i];
      const uint16_t b0 = f_to_bf16_bits(x0 * cs.x - x1 * cs.y);
      const uint16_t b1 = f_to_bf16_bits(x1 * cs.x + x0 * cs.y);
      A.kc[slot + i] = b0;
      A.kc[slot + i + half] = b1;
      kn[i] = bf16_to_f(b0);
      kn[i + half] = bf16_to_f(b1);
    }
    if (hv) {
      const uint16_t b = f_to_bf16_bits(word_value(wd[2 * QR + 2]));
      A.vc[slot + tid] = b;
      vn[tid] = bf16_to_f(b);
    }
  }
  named_sync(BAR_CONS, NCT);
  if (tr && tid == 0) tr[TR_ACT] = globaltimer();
  if (*reinterpret_cast<volatile int*>(&ms->abort)) return false;  // inputs never showed up

  // ---- scores
  const uint32_t kst = cons_acquire(pp);
  if (tr && tid == 0) tr[TR_READY] = globaltimer();  // the chunk's keys have arrived
  if (d == 64 && G <= 4) attn_scores_groups<4, 8>(kst, qs, kn, sc, nk, T, G, tid);
  else if (d == 64) attn_scores_groups<8, 8>(kst, qs, kn, sc, nk, T, G, tid);
  else if (d == 128 && G <= 4) attn_scores_groups<4, 16>(kst, qs, kn, sc, nk, T, G, tid);
  else if (d == 128) attn_scores_groups<8, 16>(kst, qs, kn, sc, nk, T, G, tid);
  else attn_scores_threads(kst, qs, kn, sc, nk, T, G, d, tid);
  cons_release(pp, lane);
  named_sync(BAR_CONS, NCT);
  if (tr && tid == 0) tr[TR_ENTRY] = globaltimer();

  // ---- softmax statistics per head (unnormalised probabilities stay in sc); a lane's first two
  // scores stay in registers between the maximum and the exponentials, the rest (T > 64) is re-read
  if (warp < G) {
    float* sg = sc + warp * T_MAX;
    const float s0 = lane < T ? sg[lane] : -CUDART_INF_F;
    const float s1 = lane + 32 < T ? sg[lane + 32] : -CUDART_INF_F;
    float m = fmaxf(s0, s1);
    for (int t = lane + 64; t < T; t += 32) m = fmaxf(m, sg[t]);
    m = warp_max(m);
    float l = 0.f;
    if (lane < T) {
      const float e = expf(s0 - m);
      sg[lane] = e;
      l += e;
    }
    if (lane + 32 < T) {
      const float e = expf(s1 - m);
      sg[lane + 32] = e;
      l += e;
    }
    for (int t = lane + 64; t < T; t += 32) {
      const float e = expf(sg[t] - m);
      sg[t] = e;
      l += e;
    }
    l = warp_sum(l);
    if (lane == 0) { ms->hm[warp] = m; ms->hl[warp] = l; }
  }
  named_sync(BAR_CONS, NCT);

  // ---- values
  const uint32_t vst = cons_acquire(pp);
  if (tr && tid == 0) tr[TR_AUX0] = globaltimer();  // the chunk's values have arrived
  {
    const uint32_t* Vw = sptr<uint32_t>(vst);  // bf16 pairs, half words per position
    for (int idx = tid; idx < G * half; idx += NCT) {
      const int g = idx / half, i2 = idx - g * half;
      const float* pg = sc + g * T_MAX;
      const uint32_t* vc = Vw + i2;
      float2 o0 = make_float2(0.f, 0.f), o1 = o0, o2 = o0, o3 = o0;
      int t = 0;
      // eight positions per turn, position t always into accumulator t mod 4 in order: the loads
      // of a turn issue together (the step is latency-bound), the sums are those of the 4-wide loop
      for (; t + 8 <= nk; t += 8) {
        const float4 pa = *reinterpret_cast<const float4*>(pg + t);
        const float4 pb = *reinterpret_cast<const float4*>(pg + t + 4);
        uint32_t w[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) w[u] = vc[(size_t)(t + u) * half];
        o0 = fma2(make_float2(pa.x, pa.x), make_float2(bf16_lo(w[0]), bf16_hi(w[0])), o0);
        o1 = fma2(make_float2(pa.y, pa.y), make_float2(bf16_lo(w[1]), bf16_hi(w[1])), o1);
        o2 = fma2(make_float2(pa.z, pa.z), make_float2(bf16_lo(w[2]), bf16_hi(w[2])), o2);
        o3 = fma2(make_float2(pa.w, pa.w), make_float2(bf16_lo(w[3]), bf16_hi(w[3])), o3);
        o0 = fma2(make_float2(pb.x, pb.x), make_float2(bf16_lo(w[4]), bf16_hi(w[4])), o0);
        o1 = fma2(make_float2(pb.y, pb.y), make_float2(bf16_lo(w[5]), bf16_hi(w[5])), o1);
        o2 = fma2(make_float2(pb.z, pb.z), make_float2(bf16_lo(w[6]), bf16_hi(w[6])), o2);
        o3 = fma2(make_float2(pb.w, pb.w), make_float2(bf16_lo(w[7]), bf16_hi(w[7])), o3);
      }
      for (; t + 4 <= nk; t += 4) {
        const float4 p4 = *reinterpret_cast<const float4*>(pg + t);
        const uint32_t w0 = vc[(size_t)t * half], w1 = vc[(size_t)(t + 1) * half];
        const uint32_t w2 = vc[(size_t)(t + 2) * half], w3 = vc[(size_t)(t + 3) * half];
        o0 = fma2(make_float2(p4.x, p4.x), make_float2(bf16_lo(w0), bf16_hi(w0)), o0);
        o1 = fma2(make_float2(p4.y, p4.y), make_float2(bf16_lo(w1), bf16_hi(w1)), o1);
        o2 = fma2(make_float2(p4.z, p4.z), make_float2(bf16_lo(w2), bf16_hi(w2)), o2);
        o3 = fma2(make_float2(p4.w, p4.w), make_float2(bf16_lo(w3), bf16_hi(w3)), o3);
      }
      for (; t < nk; ++t) {
        const uint32_t w = vc[(size_t)t * half];
        o0 = fma2(make_float2(pg[t], pg[t]), make_float2(bf16_lo(w), bf16_hi(w)), o0);
      }
      if (has_pos) o1 = fma2(make_float2(pg[nk], pg[nk]), make_float2(vn[2 * i2], vn[2 * i2 + 1]), o1);
      const float2 o = make_float2((o0.x + o1.x) + (o2.x + o3.x), (o0.y + o1.y) + (o2.y + o3.y));
      const int h = j * G + g;
      const size_t oi = ((size_t)h * A.nch_cap + c) * d + 2 * i2;
      if (A.pow_) {
        st_relaxed_v2u64(A.pow_ + oi, stamp_word(o.x, A.stamp_out), stamp_word(o.y, A.stamp_out));
      } else {
        *reinterpret_cast<float2*>(A.part_o + oi) = o;
      }
    }
  }
  cons_release(pp, lane);
  if (tid < G) {
    const int h = j * G + tid;
    const size_t mi = (size_t)h * A.nch_cap + c;
    if (A.pmw) {
      st_relaxed_u64(A.pmw + mi, stamp_word(ms->hm[tid], A.stamp_out));
      st_relaxed_u64(A.plw + mi, stamp_word(ms->hl[tid], A.stamp_out));
    } else {
      A.part_m[mi] = ms->hm[tid];
      A.part_l[mi] = ms->hl[tid];
    }
  }
  named_sync(BAR_CONS, NCT);
  if (tr && tid == 0) tr[TR_FETCHED] = globaltimer();
  if (A.pmw) return true;  // sliced merge: attn_merge_slice follows once every unit is done
  if (tid == 0) {
    // release publishes this CTA's partials (ordered before by the barrier); acquire makes the
    // other CTAs' partials visible to the merging CTA
    const unsigned old = atom_add_acq_rel(A.tickets + j, 1u);
    ms->flag = (old == (unsigned)sp.nch - 1);
  }
  named_sync(BAR_CONS, NCT);
  if (ms->flag) {
    if (tr && tid == 0) tr[TR_AUX1] = globaltimer();
    attn_merge(A, ms, tid, j, sp.nch);
    if (tid == 0) atomicExch(A.tickets + j, 0u);
  }
  named_sync(BAR_CONS, NCT);
  return true;
}

// Sliced merge of unit (KV head j, chunk c): once the partials of every chunk of head j carry this
// phase's stamp, the unit combines the outputs [c * per, (c + 1) * per) of the head's G * d outputs
// (per = ceil(G * d / nch)), one warp per output, lanes over chunks, and writes them as stamped
// words. No ticket: every unit waits only for its siblings' partials, and the whole merge is spread
// over the head's units. Returns false (the same in every consumer thread) if partials never came.
template <int MB>
__device__ __forceinline__ bool attn_merge_slice_mb(Pipe& pp, const AttnArgs& A, const AttnSplit& sp, int j,
                                                    int c, int tid, unsigned long long* tr) {
  const int G = A.nq / A.nkv, d = A.d, nch = sp.nch;
  const int lane = tid & 31, warp = tid >> 5;
  const int nout = G * d, per = (nout + nch - 1) / nch;
  const int o0 = c * per, o1 = min(o0 + per, nout);
  const unsigned sv = A.stamp_out;
  const bool check = A.check != 0;
  // two outputs per warp and pass: the six loads of up to MB chunk batches (32 chunks each) are all
  // issued before any is used, and every stale one is read again in the same turn until its
  // sibling's stamp shows; the batches are then merged in order (the same arithmetic as one batch
  // at a time, so the graph path's ticket merge still gives the same bits)
  for (int oa = o0 + warp; oa < o1; oa += 2 * NCW) {
    const int ob = oa + NCW;
    const bool hb = ob < o1;  // warp-uniform
    const int ga = oa / d, ia = oa - ga * d, ha = j * G + ga;
    const int gb = hb ? ob / d : ga, ib = hb ? ob - gb * d : ia, hb_ = j * G + gb;
    float Ma = -CUDART_INF_F, na = 0.f, da = 0.f, Mb = -CUDART_INF_F, nb = 0.f, db = 0.f;
    for (int cb0 = 0; cb0 < nch; cb0 += 32 * MB) {
      uint64_t w[MB][6];
      const uint64_t* src[MB][6];
      unsigned need = 0;  // bit 6 * q + e: word e of batch q
#pragma unroll
      for (int q = 0; q < MB; ++q) {
        const int cc = cb0 + 32 * q + lane;
        const bool on = cc < nch;
        const int ca = on ? cc : nch - 1;  // addresses stay inside the partial buffers
        const size_t mia = (size_t)ha * A.nch_cap + ca, mib = (size_t)hb_ * A.nch_cap + ca;
        src[q][0] = A.pmw + mia; src[q][1] = A.plw + mia; src[q][2] = A.pow_ + mia * d + ia;
        src[q][3] = A.pmw + mib; src[q][4] = A.plw + mib; src[q][5] = A.pow_ + mib * d + ib;
        if (on) need |= (hb ? 0x3Fu : 0x07u) << (6 * q);
#pragma unroll
        for (int e = 0; e < 6; ++e) w[q][e] = (need >> (6 * q + e)) & 1u ? ld_relaxed_u64(src[q][e]) : 0;
      }
      if (check) {
        unsigned stale = 0;
#pragma unroll
        for (int q = 0; q < MB; ++q)
#pragma unroll
          for (int e = 0; e < 6; ++e)
            if (((need >> (6 * q + e)) & 1u) && word_stamp(w[q][e]) != sv) stale |= 1u << (6 * q + e);
        Poll pl;
        while (stale && pl.again(pp)) {
#pragma unroll
          for (int q = 0; q < MB; ++q)
#pragma unroll
            for (int e = 0; e < 6; ++e)
              if ((stale >> (6 * q + e)) & 1u) w[q][e] = ld_relaxed_u64(src[q][e]);
#pragma unroll
          for (int q = 0; q < MB; ++q)
#pragma unroll
            for (int e = 0; e < 6; ++e)
              if (((stale >> (6 * q + e)) & 1u) && word_stamp(w[q][e]) == sv) stale &= ~(1u << (6 * q + e));
        }
      }
      if (tr && tid == 0 && cb0 == 0 && oa == o0) tr[TR_AUX1] = globaltimer();  // siblings' partials seen
#pragma unroll
      for (int q = 0; q < MB; ++q) {
        if (cb0 + 32 * q >= nch) break;  // warp-uniform: the batches the one-at-a-time merge would run
        const bool on = cb0 + 32 * q + lane < nch;
        float ma = -CUDART_INF_F, la = 0.f, va = 0.f, mb = -CUDART_INF_F, lb = 0.f, vb = 0.f;
        if (on) {
          ma = word_value(w[q][0]); la = word_value(w[q][1]); va = word_value(w[q][2]);
          if (hb) { mb = word_value(w[q][3]); lb = word_value(w[q][4]); vb = word_value(w[q][5]); }
        }
        merge_step(Ma, na, da, ma, la, va);
        if (hb) merge_step(Mb, nb, db, mb, lb, vb);
      }
    }
    if (lane == 0) {
      st_relaxed_u64(A.outw + (size_t)ha * d + ia, stamp_word(na / da, A.stamp_out));
      if (hb) st_relaxed_u64(A.outw + (size_t)hb_ * d + ib, stamp_word(nb / db, A.stamp_out));
    }
  }
  named_sync(BAR_CONS, NCT);
  return !*reinterpret_cast<volatile int*>(&pp.ms->abort);
}

// The merge with as many chunk batches in flight as the head has (up to four): one L2 round trip for
// the partials of up to 128 chunks (the Qwen-shaped step: 76 chunks, 9 % faster than one batch at a
// time), while heads of at most 32 chunks keep the one-batch code.
static __device__ bool attn_merge_slice(Pipe& pp, const AttnArgs& A, const AttnSplit& sp, int j, int c,
                                        int tid, unsigned long long* tr = nullptr) {
  if (sp.nch <= 32) return attn_merge_slice_mb<1>(pp, A, sp, j, c, tid, tr);
  if (sp.nch <= 64) return attn_merge_slice_mb<2>(pp, A, sp, j, c, tid, tr);
  return attn_merge_slice_mb<4>(pp, A, sp, j, c, tid, tr);
}

}  // namespace tinfer
