// megakernel.cuh -- device side of the decode step: the step schedule, the persistent producer,
// the consumer phases, the persistent kernel and the per-phase kernel. Included by the translation
// units that instantiate the kernels (one per weight format, so that they compile in parallel).
//
// The kernels are templates over the weight format, the number of 16-byte chunks a lane holds in
// the bf16 GEMV (NCHL) and, for the persistent kernel, whether it records a timeline. One bf16 GEMV
// width per kernel keeps the register allocation of the persistent kernel free of spills: the host
// picks the instance that covers every bf16 matrix of the model.
#pragma once
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
  g.nsegs = 0;
  g.rbs = 0;
  const LayerDev& L = p.layers[layer];
  switch (phase) {
    case PH_QKV: g.w = L.qkv; g.rows = m.qkv_rows; g.cols = m.H; g.rb = m.rb_h; break;
    case PH_O: g.w = L.o; g.rows = m.H; g.cols = m.nq * m.d; g.rb = m.rb_qd; break;
    case PH_GU: g.w = L.gu; g.rows = 2 * m.F; g.cols = m.H; g.rb = m.rb_h; g.quantum = 2; break;
    case PH_DOWN:
      g.w = L.down;
      if (m.ffn_split) { g.rows = m.F; g.cols = m.H; g.rb = m.rb_h; }  // Wd^T, this CTA's ffn inputs
      else { g.rows = m.H; g.cols = m.F; g.rb = m.rb_f; }
      break;
    default:
      g.w = reinterpret_cast<const uint8_t*>(p.lm_head);
      g.rows = m.V; g.cols = m.H; g.rb = m.rb_lm; g.fmt = 0;
      break;
  }
  return g;
}

// Stamps of the launch's step s: phase k of step s writes epoch + s * stride + k (stride: the
// phases of a step plus one), so that stamps keep increasing across the steps of one launch.
__device__ __forceinline__ int phases_per_step(const StepParams& p) { return p.m.L * PHASES_PER_LAYER + 1; }
__device__ __forceinline__ unsigned step_epoch(const StepParams& p, int s) {
  return p.epoch + (unsigned)s * (unsigned)(phases_per_step(p) + 1);
}

// Attention of phase k (layer `layer`) of the step whose stamps start at ep: q/k/v from the QKV phase
// k - 1, output for the O phase.
__device__ __forceinline__ AttnArgs step_attn_args(const StepParams& p, int layer, int pos, int k, unsigned ep,
                                                   bool loop = false) {
  (void)loop;
  const Dims& m = p.m;
  AttnArgs A;
  A.qkv = nullptr;
  A.qkvw = p.qkv;
  A.stamp_in = ep + (unsigned)(k - 1);
  A.check = p.stamp_check;
  A.outw = p.attn;
  A.stamp_out = ep + (unsigned)k;
  const size_t lay = (size_t)layer * m.nkv * m.max_ctx * m.d;
  A.kc = p.kcache + lay;
  A.vc = p.vcache + lay;
  A.rope = p.rope;
  A.part_m = p.part_m;
  A.part_l = p.part_l;
  A.part_o = p.part_o;
  if (p.stamp_check) {  // persistent kernel: sliced merge over stamped partials
    A.pmw = p.part_mw;
    A.plw = p.part_lw;
    A.pow_ = p.part_ow;
  }
  A.nch_cap = p.nch_cap;
  A.tickets = p.tickets;
  A.out = nullptr;
  A.nq = m.nq; A.nkv = m.nkv; A.d = m.d; A.max_ctx = m.max_ctx; A.pos = pos;
  return A;
}

__device__ __forceinline__ void produce_phase(const StepParams& p, Pipe& pp, int phase, int layer, int pos,
                              uint64_t pol_w, uint64_t pol_kv, bool& dead) {
  if (phase == PH_ATTN) {
    const AttnArgs A = step_attn_args(p, layer, pos, 0, p.epoch);  // the producer uses the cache pointers only
    const AttnSplit sp = attn_split(pos, A.nkv, A.d, p.grid, p.slot_bytes, p.n_chunks_override);
    const int units = A.nkv * sp.nch;
    for (int u = blockIdx.x; u < units; u += p.grid)
      produce_attn_unit(pp, A, u / sp.nch, u % sp.nch, sp, pol_kv, dead);
    return;
  }
  const GemvDesc g = phase_gemv(p, phase, layer);
  produce_rows(pp, g, row_split(g, blockIdx.x, p.grid, p.slot_bytes), pol_w, dead);
}

// Timeline slot of (this CTA, phase k, field); null when the launch records no timeline. The
// persistent kernel passes a compile-time null in its untraced instance, so that the stamps cost
// nothing there.
__device__ __forceinline__ unsigned long long* trace_at(unsigned long long* trace, const StepParams& p,
                                                        int k, int field) {
  if (!trace) return nullptr;
  const int nph = p.m.L * PHASES_PER_LAYER + 1;
  return trace + ((size_t)blockIdx.x * nph + k) * TRACE_FIELDS + field;
}

// The persistent producer's view of the launch: one pass over this CTA's copy schedule, stage by
// stage, in the order the consumers take them (per GEMV phase its rows; per attention unit the
// cached K chunk, then the V chunk). k counts the phases of the whole launch; only the instance
// with the token loop has more than one step, and only it tracks the step of a phase.
struct StageCursor {
  int k, j;                        // phase index, stage within the phase
  int attn;                        // the phase is attention
  const uint8_t* w;                // GEMV: matrix, row bytes, this CTA's rows, rows per stage
  int rb, r0, r1, nr;
  const uint16_t* kc;              // attention: this layer's K and V caches
  const uint16_t* vc;
  int u, units, nch, cl, sub;      // unit cursor, split, K/V half of the unit
  int klocal, pos;                 // token loop: phase index within its step, that step's position
  int kvl;                         // token loop: that step's index
};

template <bool LOOP>
__device__ __forceinline__ void cursor_enter(const StepParams& p, StageCursor& c, int& pos, int n_steps) {
  const int nph = phases_per_step(p);
  if (c.k >= nph * n_steps) return;
  int k = c.k, s = 0;
  if constexpr (LOOP) {
    s = c.k / nph;
    k = c.k - s * nph;
    c.klocal = k;
    c.pos = pos = p.pos + s;
  }
  int phase, layer;
  phase_of(k, p.m.L, phase, layer);
  if (phase == PH_ATTN) {
    const AttnSplit sp = attn_split(pos, p.m.nkv, p.m.d, p.grid, p.slot_bytes, p.n_chunks_override);
    const size_t lay = (size_t)layer * p.m.nkv * p.m.max_ctx * p.m.d;
    c.attn = 1; c.kc = p.kcache + lay; c.vc = p.vcache + lay;
    c.nch = sp.nch; c.cl = sp.cl; c.units = p.m.nkv * sp.nch; c.u = blockIdx.x; c.sub = 0;
    if constexpr (LOOP) c.kvl = s;
    return;
  }
  const GemvDesc g = phase_gemv(p, phase, layer);
  const RowSplit rs = row_split(g, blockIdx.x, p.grid, p.slot_bytes);
  c.attn = 0; c.w = g.w; c.rb = g.rb; c.r0 = rs.r0; c.r1 = rs.r1; c.nr = rs.nr;
  c.j = 0;
}

// The next stage's copy. In the token loop, *wait (when set) is the flag of a K/V slot another CTA
// wrote in the previous step of this launch: the copy may be issued once the flag carries `stamp`.
template <bool LOOP>
__device__ __forceinline__ bool cursor_next(const StepParams& p, StageCursor& c, int pos, const void*& src,
                                            uint32_t& bytes, const unsigned*& wait, unsigned& stamp,
                                            int n_steps) {
  const int nk_all = phases_per_step(p) * n_steps;
  if constexpr (LOOP) {
    wait = nullptr;
    pos = c.pos;
  }
  while (c.k < nk_all) {
    if (!c.attn) {
      const int s0 = c.r0 + c.j * c.nr;
      if (s0 < c.r1) {
        src = c.w + (size_t)s0 * c.rb;
        bytes = (uint32_t)(min(c.nr, c.r1 - s0) * c.rb);
        ++c.j;
        return true;
      }
    } else if (c.u < c.units) {
      const int j = c.u / c.nch, ch = c.u - j * c.nch;
      const int t0 = ch * c.cl;
      const int tend = min(t0 + c.cl, pos);  // the slot at pos is written in this step: never streamed
      const int nk = tend > t0 ? tend - t0 : 0;
      const size_t base = ((size_t)j * p.m.max_ctx + t0) * p.m.d;
      src = (c.sub == 0 ? c.kc : c.vc) + base;
      bytes = (uint32_t)(nk * p.m.d * 2);
      if constexpr (LOOP) {
        if (c.kvl > 0 && nk > 0 && tend == pos) {  // holds slot pos - 1, written by the previous step
          wait = p.kvflag + j;
          stamp = step_epoch(p, c.kvl - 1);
        }
      }
      if (c.sub) { c.sub = 0; c.u += p.grid; } else { c.sub = 1; }
      return true;
    }
    ++c.k;
    cursor_enter<LOOP>(p, c, pos, n_steps);
  }
  return false;
}

// The persistent kernel's producer: feeds the ring in schedule order with bulk copies (at most
// p.inflight outstanding, p.inflight_lm during the LM head). While the ring is full -- the consumers
// are in a latency-bound stretch (a hand-off, attention, a small matrix) -- it walks a second cursor
// ahead and prefetches upcoming stages into L2, paced at about this SM's share of HBM bandwidth and
// at most l2_lookahead bytes beyond the copies, so that HBM keeps streaming while the ring cannot
// take more. Later copies of those stages hit L2. In the token loop, the copy that reads the slot
// the previous step wrote first acquires that slot's flag, then orders the acquired view before the
// bulk copy (a generic-proxy write read by the async proxy).
template <bool LOOP>
__device__ __forceinline__ void produce_step(const StepParams& p, Pipe& pp, unsigned long long* trace,
                                             int n_steps) {
  const uint64_t pol_w = policy_evict_first(), pol_pf = policy_evict_normal();
  // both cursors start before phase 0 with no stage left, so that their first cursor_next enters
  // it (one inlined copy of the cursor code per cursor keeps the producer's code small)
  StageCursor cp{}, pf{};
  cp.k = -1;
  pf.k = -1;
  int pos_c = p.pos, pos_f = p.pos;
  long long cend = 0, pend = 0;  // stream offsets: end of the current copy, end of prefetched bytes
  uint64_t next_pf = 0;
  bool dead = false;
  const void* src;
  uint32_t bytes;
  const unsigned* wait = nullptr;
  unsigned wstamp = 0;
  const volatile int* done = &pp.ms->cons_done;
  int last_k = -1;
  const int nph = phases_per_step(p);
  while (!dead && cursor_next<LOOP>(p, cp, pos_c, src, bytes, wait, wstamp, n_steps)) {
    if (trace && cp.k != last_k && cp.k < nph) {  // timeline (first step): the producer moves on to phase cp.k
      const uint64_t t = globaltimer();
      if (last_k >= 0) *trace_at(trace, p, last_k, TR_PROD_END) = t;
      *trace_at(trace, p, cp.k, TR_PROD_BEGIN) = t;
    }
    if (cp.k < nph) last_k = cp.k;
    cend += bytes;
    const int s = pp.s;
    const uint32_t eb = pp.empty0 + 8u * s;
    if (!mbar_try_wait(eb, pp.ph ^ 1u)) {
      const uint64_t t0 = globaltimer();
      while (!mbar_try_wait(eb, pp.ph ^ 1u)) {
        if (*done) { dead = true; break; }
        const uint64_t now = globaltimer();
        if (p.l2_lookahead > 0 && now >= next_pf) {
          // prefetch the next stage the copies have not reached, within the lookahead window;
          // stages the copy cursor has already taken are skipped
          while (pend < (1LL << 62) && pend - cend < p.l2_lookahead) {
            const void* ps;
            uint32_t pb;
            const unsigned* pw;
            unsigned pst;
            if (!cursor_next<LOOP>(p, pf, pos_f, ps, pb, pw, pst, n_steps)) { pend = 1LL << 62; break; }
            const long long start = pend;
            pend += pb;
            if (start >= cend) {
              if (pb) bulk_prefetch_l2(ps, pb, pol_pf);
              next_pf = now + (uint64_t)pb * (uint64_t)p.l2_pace_ns_per_kb / 1024u;
              break;
            }
          }
        }
        if ((long long)(now - t0) > pp.timeout) {
          dead = true;
          if (!*done) raise_error(pp.err, pp.err_host, EW_TIMEOUT);
          break;
        }
      }
      if (dead) break;
    }
    if constexpr (LOOP) {
      if (wait) {
        // bounded: the writer published the flag a step ago, so this normally passes at once
        if (ld_acquire(wait) != wstamp) {
          const uint64_t t0 = globaltimer();
          while (ld_acquire(wait) != wstamp) {
            if (*done) { dead = true; break; }
            if ((long long)(globaltimer() - t0) > pp.timeout) {
              dead = true;
              raise_error(pp.err, pp.err_host, EW_TIMEOUT);
              break;
            }
          }
          if (dead) break;
        }
        fence_proxy_async_global();
      }
    }
    const int klocal = LOOP ? cp.klocal : cp.k;
    const int infl = min(klocal == nph - 1 ? p.inflight_lm : pp.inflight, pp.stages);  // <= ring
    if (infl > 0 && pp.it >= (uint32_t)infl) {
      const int k = infl;
      const int s2 = s >= k ? s - k : s - k + pp.stages;
      const uint32_t p2 = s >= k ? pp.ph : pp.ph ^ 1u;
      if (!mbar_try_wait(pp.full0 + 8u * s2, p2) &&
          !wait_bar(pp.full0 + 8u * s2, p2, pp.timeout, &pp.ms->cons_done))
        break;
    }
    const uint32_t fb = pp.full0 + 8u * s;
    mbar_arrive_expect_tx(fb, bytes);
    if (bytes) bulk_g2s(pp.ring + (uint32_t)s * pp.slot, src, bytes, fb, pol_w);
    pipe_advance(pp);
  }
  if (trace && last_k >= 0) *trace_at(trace, p, last_k, TR_PROD_END) = globaltimer();
  prod_drain(pp);
}


// Consumer side of one attention phase (every unit this CTA owns). Separate from the GEMV phase so
// that each gets its own register allocation; the pipe state goes in and comes back by value.
template <bool LOOP>
__device__ __forceinline__ bool consume_attn_phase(const StepParams& p, Pipe& pp, int layer, int pos,
                                                   int tid, int k, unsigned long long* trace, unsigned ep) {
  unsigned long long* tr_ready = trace_at(trace, p, k, TR_READY);
  if (tr_ready && tid == 0) *tr_ready = globaltimer();
  // the attention scratch shares shared memory with the row results the QKV epilogue still reads
  named_sync(BAR_CONS, NCT);
  const AttnArgs A = step_attn_args(p, layer, pos, k, ep, LOOP);
  const AttnSplit sp = attn_split(pos, A.nkv, A.d, p.grid, p.slot_bytes, p.n_chunks_override);
  const int units = A.nkv * sp.nch;
  unsigned long long* tr = trace_at(trace, p, k, 0);  // the first unit of the CTA records sub-steps
  for (int u = blockIdx.x; u < units; u += p.grid) {
    if (!attn_unit(pp, A, sp, u / sp.nch, u % sp.nch, tid, tr)) return false;
    tr = nullptr;
  }
  if (A.pmw) {  // every unit of the CTA has published its partials: now merge the slices
    unsigned long long* trm = trace_at(trace, p, k, 0);
    for (int u = blockIdx.x; u < units; u += p.grid) {
      if (!attn_merge_slice(pp, A, sp, u / sp.nch, u % sp.nch, tid, trm)) return false;
      trm = nullptr;
    }
  }
  return true;
}

// Per-launch shared-memory copy of what every GEMV phase's plan needs: the descriptor and this
// CTA's row split of each of the five matrix kinds (the same for every layer) and the layer table.
// Without it each phase start would recompute the split (integer divisions) and read the layer
// table through the constant cache, whose misses cost about a microsecond per phase.
struct PhaseTable {
  GemvDesc desc[6];   // indexed by Phase (PH_ATTN unused); w = nullptr
  RowSplit rs[6];
  LayerDev layers[MAX_LAYERS];
};
__device__ __forceinline__ void fill_phase_table(const StepParams& p, PhaseTable& t, int tid) {
  if (tid < 6 && tid != PH_ATTN) {
    GemvDesc g = phase_gemv(p, tid, 0);
    g.w = nullptr;
    t.desc[tid] = g;
    t.rs[tid] = row_split(g, blockIdx.x, p.grid, p.slot_bytes);
  }
  for (int l = tid; l < p.m.L; l += NCT) t.layers[l] = p.layers[l];
}

// The plan of a GEMV phase: QKV (RMSNorm prologue, bias), O (+ residual), gate/up (RMSNorm,
// SwiGLU), down (+ residual) or the LM head (final RMSNorm, logits, argmax).
//
// Hand-off buffers without barriers. Phase k of a step writes its results as stamped words with
// stamp ep + k (ep: the step's first stamp); phase k + 1 reads them once they carry that stamp. A buffer is rewritten only by a
// later phase of the same kind (qkv by the next layer's QKV, xa by the next O, act by the next
// gate/up, xb by the next down; the attention output and partials by the next attention). A CTA
// that rewrites buffer B in phase k' has, in its own phase k' - 1, read the complete results of
// phase k' - 1 (or, for attention, its heads' q/k/v, whose writers had read the complete results
// before them), and every CTA produced its part of those results only after it had read B in an
// earlier phase. So no reader of B is still reading when B is rewritten. The residual rows a
// GEMV adds to are this CTA's own (the same row split in O and down), written by the same thread,
// so they need no stamp check.
//
// In memory-model terms: every stamped word is stored with a relaxed gpu-scope 64-bit store and
// polled with relaxed gpu-scope loads (ptx.cuh). Those accesses are morally strong, so a poll that
// races with the store is not a data race, and a 64-bit access is single-copy atomic, so a reader
// that sees the stamp it waits for sees the value stored with it; the value needs no further
// ordering because it travels in the same word. Write-after-read safety of a rewritten buffer rests
// on the chain above: a CTA's results are computed from the values it loaded, so its loads of B
// complete before it stores anything derived from them, and every rewrite of B depends, through at
// least one complete phase of such results, on those stores. The PTX model alone does not order a
// relaxed load before a later relaxed store to another address (a fence per thread and phase would,
// at about the cost of the grid barrier this hand-off replaces); the data dependency through the
// stored values is what orders them.
__device__ __forceinline__ GemvPlan plan_gemv(const StepParams& p, Pipe& pp, int phase, int layer,
                                              int k, int token, int tid, const PhaseTable* tab,
                                              unsigned ep) {
  const Dims& m = p.m;
  GemvPlan pl;
  const LayerDev& L = tab ? tab->layers[layer] : p.layers[layer];
  if (tab) {
    pl.g = tab->desc[phase];
    pl.g.w = phase == PH_QKV ? L.qkv : phase == PH_O ? L.o : phase == PH_GU ? L.gu : phase == PH_DOWN
             ? L.down : reinterpret_cast<const uint8_t*>(p.lm_head);
    pl.rs = tab->rs[phase];
  } else {
    pl.g = phase_gemv(p, phase, layer);
    pl.rs = row_split(pl.g, blockIdx.x, p.grid, p.slot_bytes);
  }
  pl.src = ActSrc{};
  pl.src.eps = m.eps;
  // phase k reads the stamped results of phase k - 1 and writes its own with stamp ep + k
  pl.src.stamp = ep + (unsigned)(k - 1);
  pl.src.check = p.stamp_check;
  const unsigned own = ep + (unsigned)k;
  const uint16_t* erow = p.embed + (size_t)token * m.H;
  switch (phase) {
    case PH_QKV:
      if (layer == 0) pl.src.xb = erow; else pl.src.xw = p.xb;
      pl.src.gf = L.g1; pl.src.n = m.H;
      pl.epi = Epi{EK_STORE, p.qkv, L.bias, nullptr, own, EF_OUT_STAMPED};
      break;
    case PH_O:
      pl.src.xw = p.attn; pl.src.n = m.nq * m.d;
      if (layer == 0) pl.epi = Epi{EK_RESIDUAL, p.xa, nullptr, erow, own, EF_OUT_STAMPED | EF_RES_BF16};
      else pl.epi = Epi{EK_RESIDUAL, p.xa, nullptr, p.xb, own, EF_OUT_STAMPED | EF_RES_STAMPED};
      break;
    case PH_GU:
      pl.src.xw = p.xa; pl.src.gf = L.g2; pl.src.n = m.H;
      pl.epi = Epi{EK_SWIGLU, p.act, nullptr, nullptr, own, EF_OUT_STAMPED};
      break;
    case PH_DOWN:
      pl.src.xw = p.act; pl.src.n = m.F;
      pl.epi = Epi{m.ffn_split ? EK_COLSPLIT : EK_RESIDUAL, p.xb, nullptr, p.xa, own,
                   EF_OUT_STAMPED | EF_RES_STAMPED};
      break;
    default:
      pl.src.xw = p.xb; pl.src.gb = p.final_norm; pl.src.n = m.H;
      pl.epi = Epi{EK_ARGMAX, p.logits, nullptr, nullptr, own, 0};
      break;
  }
  if (p.dbg_skip_cta == (int)blockIdx.x && p.dbg_skip_phase == k) pl.epi.flags |= EF_WITHHOLD;
  return pl;
}

// Consumer side of one GEMV phase from its plan; false when its input never showed up.
template <int FMT, int NCHL, int IF, bool LOOP, bool SPLIT>
__device__ __forceinline__ bool run_gemv_phase(const StepParams& p, Pipe& pp, const GemvPlan& pl,
                                               int phase, int tid, int k, unsigned long long* trace) {
  const Dims& m = p.m;
  unsigned long long* tr_ready = trace_at(trace, p, k, TR_READY);
  Best best{-CUDART_INF_F, 0x7FFFFFFF, 0};
  if constexpr (FMT == 0 && SPLIT) {
    if (pl.epi.kind == EK_COLSPLIT) {
    // the output rows of the reduce are the O phase's split of the hidden rows (their residual
    // rows are this CTA's own)
      const RowSplit ro = row_split(GemvDesc{nullptr, m.H, m.F, 0, 0, 0, 0, 1}, blockIdx.x, p.grid, p.slot_bytes);
      return colsplit_down(pp, pl, ro, p.part_ffn, p.grid, tid);
    }
  }
  // int4 models stream their linears as int4 and the LM head as bf16; bf16 models need one format
  const bool ok = (FMT == 1 && pl.g.fmt == 1) ? gemv_rows<1, 2>(pp, pl, best, tid, tr_ready)
                                              : gemv_rows<0, NCHL, IF>(pp, pl, best, tid, tr_ready);
  if (!ok) return false;
  if (phase == PH_LM) {
    const Best cb = best_block_reduce(best, pp.ms, tid);
    if (LOOP) {
      // token loop: this CTA's best as two stamped words; every CTA combines all of them at the
      // start of the next step
      if (tid == 0)
        st_relaxed_v2u64(p.best_w + 2 * blockIdx.x, stamp_word(cb.v, pl.epi.stamp),
                         ((uint64_t)pl.epi.stamp << 32) | ((uint64_t)(cb.bad ? 1u : 0u) << 31) |
                             (uint64_t)(unsigned)(cb.i & 0x7FFFFFFF));
    } else {
      argmax_publish(cb, p.best_val, p.best_idx, p.best_bad, p.tickets + m.nkv, p.grid, blockIdx.x,
                     p.argmax, p.err, p.err_host, pp.ms, tid);
    }
  }
  return true;
}

// Token loop: the greedy choice of a step from every CTA's stamped best (the largest logit, the
// lowest token id among ties, and whether any logit was non-finite), combined by warp 0 and handed
// to the CTA's consumer threads. Every CTA reads the same slots and applies the same
// order-independent rule, so all of them reach the same token and the same stop decision with no
// barrier ("Decoding in tiles", section 5: each lm_head task writes its best candidate to its own
// slot, and every worker combines all slots at the start of the next step). False when a slot never
// showed up (the CTA's abort flag is then set).
__device__ __forceinline__ bool gather_best(const StepParams& p, Pipe& pp, unsigned stamp, int tid, Best& out) {
  Misc* ms = pp.ms;
  constexpr int PER = 5;  // slots per lane and batch: one batch covers 160 CTAs
  if (tid < 32) {
    Best b{-CUDART_INF_F, 0x7FFFFFFF, 0};
    for (int c0 = 0; c0 < p.grid; c0 += 32 * PER) {
      uint64_t w0[PER], w1[PER];
      unsigned need = 0;
#pragma unroll
      for (int e = 0; e < PER; ++e) {
        const int c = c0 + tid + 32 * e;
        if (c < p.grid) {
          const ulonglong2 v = ld_relaxed_v2u64(p.best_w + 2 * c);
          w0[e] = v.x;
          w1[e] = v.y;
          need |= 1u << e;
        }
      }
      unsigned stale = 0;
#pragma unroll
      for (int e = 0; e < PER; ++e)
        if ((need & (1u << e)) && (word_stamp(w0[e]) != stamp || word_stamp(w1[e]) != stamp)) stale |= 1u << e;
      Poll pl;
      while (stale && pl.again(pp)) {
#pragma unroll
        for (int e = 0; e < PER; ++e) {
          if (stale & (1u << e)) {
            const ulonglong2 v = ld_relaxed_v2u64(p.best_w + 2 * (c0 + tid + 32 * e));
            w0[e] = v.x;
            w1[e] = v.y;
          }
        }
#pragma unroll
        for (int e = 0; e < PER; ++e)
          if ((stale & (1u << e)) && word_stamp(w0[e]) == stamp && word_stamp(w1[e]) == stamp) stale &= ~(1u << e);
      }
#pragma unroll
      for (int e = 0; e < PER; ++e) {
        if (need & (1u << e)) {
          const float v = word_value(w0[e]);
          const int i = (int)((uint32_t)w1[e] & 0x7FFFFFFFu);
          if (v > b.v || (v == b.v && i < b.i)) { b.v = v; b.i = i; }
          b.bad |= (int)(((uint32_t)w1[e] >> 31) & 1u);
        }
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float ov = __shfl_xor_sync(0xFFFFFFFFu, b.v, o);
      const int oi = __shfl_xor_sync(0xFFFFFFFFu, b.i, o);
      const int ob = __shfl_xor_sync(0xFFFFFFFFu, b.bad, o);
      if (ov > b.v || (ov == b.v && oi < b.i)) { b.v = ov; b.i = oi; }
      b.bad |= ob;
    }
    if (tid == 0) { ms->bv[0] = b.v; ms->bi[0] = b.i; ms->bbad[0] = b.bad; }
  }
  named_sync(BAR_CONS, NCT);
  out = Best{ms->bv[0], ms->bi[0], ms->bbad[0]};
  const bool ok = !*reinterpret_cast<volatile int*>(&ms->abort);
  named_sync(BAR_CONS, NCT);  // the slots of ms are free again
  return ok;
}

// Phase k: its plan (GEMV phases) and its run.
__device__ __forceinline__ GemvPlan plan_phase(const StepParams& p, Pipe& pp, int k, int token,
                                               int tid, const PhaseTable* tab, unsigned ep) {
  int phase, layer;
  phase_of(k, p.m.L, phase, layer);
  if (phase == PH_ATTN) return GemvPlan{};
  return plan_gemv(p, pp, phase, layer, k, token, tid, tab, ep);
}

template <int FMT, int NCHL, int IF, bool LOOP, bool SPLIT>
__device__ __forceinline__ bool run_phase(const StepParams& p, Pipe& pp, const GemvPlan& pl, int k,
                                          int pos, int tid, unsigned long long* trace, unsigned ep) {
  int phase, layer;
  phase_of(k, p.m.L, phase, layer);
  if (phase == PH_ATTN) return consume_attn_phase<LOOP>(p, pp, layer, pos, tid, k, trace, ep);
  return run_gemv_phase<FMT, NCHL, IF, LOOP, SPLIT>(p, pp, pl, phase, tid, k, trace);
}

// The grid-barrier schedule ("Decoding in tiles", section 4: every wave ends at a grid barrier that
// all workers pass): barrier number n of the context completes when the monotonic counter reaches
// (n + 1) * grid. Thread 0 arrives with release semantics (ordering, through the consumer barrier
// before it, the CTA's results of the previous phase) and waits with acquire semantics, bounded.
__device__ __forceinline__ bool grid_barrier(const StepParams& p, Pipe& pp, unsigned long long n, int tid) {
  named_sync(BAR_CONS, NCT);
  if (tid == 0) {
    red_add_release_u64(p.bar_count, 1ull);
    const unsigned long long target = (n + 1ull) * (unsigned long long)p.grid;
    if (ld_acquire_u64(p.bar_count) < target) {
      const uint64_t t0 = globaltimer();
      while (ld_acquire_u64(p.bar_count) < target) {
        if (ld_volatile_int(p.err) != 0 || (long long)(globaltimer() - t0) > p.timeout_ns) {
          if (ld_volatile_int(p.err) == 0) raise_error(p.err, p.err_host, EW_TIMEOUT);
          pp.ms->abort = 1;
          break;
        }
      }
    }
  }
  named_sync(BAR_CONS, NCT);
  return !*reinterpret_cast<volatile int*>(&pp.ms->abort);
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

// LOOP: the instance that runs the token loop (n_steps decode steps per launch); the single-step
// instance carries none of its state, which keeps the int4 consumers' registers free of spills.
// SPLIT: the instance for the column-split down projection (Dims::ffn_split). Each variant is its
// own instance because the persistent kernel's speed depends on its code size and registers: the
// column-split code compiled into the other instances made the Llama-shaped step 13 % slower.
template <int FMT, int NCHL, bool TRACE, bool LOOP, bool SPLIT = false>
__global__ void __launch_bounds__(NTHREADS_MEGA, 1) decode_megakernel(const __grid_constant__ StepParams p) {
  unsigned long long* const trace = TRACE ? p.trace : nullptr;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ int s_tok[2];
  __shared__ PhaseTable s_tab;
  Pipe pp;
  pipe_init(pp, smem, p.ring_stages, p.slot_bytes, p.timeout_ns, p.err, p.err_host);
  pp.inflight = p.inflight;
  pipe_setup(pp);
  int token = 0;
  if (!step_prologue(p, token, p.pos, s_tok)) return;
  const int nph = phases_per_step(p);
  const int tid = threadIdx.x;
  if (tid >= NCT) {
    reg_dealloc<FMT ? REG_PRODUCER_INT4 : REG_PRODUCER>();
    if (tid == NCT) produce_step<LOOP>(p, pp, trace, LOOP ? p.n_steps : 1);
  } else {
    reg_alloc<FMT ? REG_CONSUMER_INT4 : REG_CONSUMER>();
    // no grid barrier: each phase waits, inside its input fetch, for the stamps of the results it
    // reads, so a CTA starts a phase as soon as its own inputs are complete. With n_steps > 1 the
    // steps follow one another in this launch ("Decoding in tiles", section 5, Figure 10: one
    // launch decodes consecutive tokens, greedy selection inside the kernel); stamps keep rising
    // across steps, so a step needs no barrier either.
    fill_phase_table(p, s_tab, tid);
    named_sync(BAR_CONS, NCT);
    int done_steps = 0;
    const int n_steps = LOOP ? p.n_steps : 1;
    for (int s = 0; s < n_steps; ++s) {
      const unsigned ep = step_epoch(p, s);
      const int pos = p.pos + s;
      if (LOOP && s > 0) {  // the previous step's choice is this step's token
        Best b;
        if (!gather_best(p, pp, step_epoch(p, s - 1) + (unsigned)(nph - 1), tid, b)) break;
        const int tk = b.bad ? -1 : b.i;
        if (blockIdx.x == 0 && tid == 0) {
          p.tokens_out[s - 1] = tk;
          if (b.bad) raise_error(p.err, p.err_host, EW_NONFINITE);
        }
        done_steps = s;
        if (b.bad || tk == p.eos) break;  // the same decision in every CTA
        token = tk;
      }
      unsigned long long* tr = s == 0 ? trace : nullptr;  // the timeline records the first step
      bool ok = true;
      for (int k = 0; k < nph && ok; ++k) {
        if (p.sync_barrier && k > 0 &&
            !grid_barrier(p, pp, p.bar_base + (unsigned long long)s * (unsigned long long)(nph - 1) + (unsigned long long)(k - 1), tid)) {
          ok = false;
          break;
        }
        if (unsigned long long* t = trace_at(tr, p, k, TR_START)) if (tid == 0) *t = globaltimer();
        const GemvPlan plan = plan_phase(p, pp, k, token, tid, &s_tab, ep);
        ok = run_phase<FMT, NCHL, 4, LOOP, SPLIT>(p, pp, plan, k, pos, tid, tr, ep);
        if (unsigned long long* t = trace_at(tr, p, k, TR_END)) if (tid == 0) *t = globaltimer();
      }
      if (!ok) break;
      if (LOOP && s + 1 < n_steps) {
        // the next step streams slot pos of every layer with bulk copies from other CTAs: the CTA
        // that wrote it for KV head j (the owner of the chunk holding pos) makes the step's K/V
        // writes visible at gpu scope and publishes the step's first stamp for j. Done here, after
        // the LM head's results, the fence delays neither a layer's hand-offs nor the choice.
        const AttnSplit sp = attn_split(pos, p.m.nkv, p.m.d, p.grid, p.slot_bytes, p.n_chunks_override);
        const int cpos = pos / sp.cl;
        bool owner = false;
        for (int j = 0; j < p.m.nkv; ++j) owner |= (j * sp.nch + cpos) % p.grid == (int)blockIdx.x;
        if (owner) {
          fence_acq_rel_gpu();
          named_sync(BAR_CONS, NCT);
          if (tid < p.m.nkv && (tid * sp.nch + cpos) % p.grid == (int)blockIdx.x) st_relaxed_u32(p.kvflag + tid, ep);
        }
      }
      if (s == n_steps - 1) {
        done_steps = s + 1;
        if (LOOP && blockIdx.x == 0) {  // the last step's choice, recorded by CTA 0
          Best b;
          if (gather_best(p, pp, ep + (unsigned)(nph - 1), tid, b) && tid == 0) {
            p.tokens_out[s] = b.bad ? -1 : b.i;
            if (b.bad) raise_error(p.err, p.err_host, EW_NONFINITE);
          }
        }
      }
    }
    if (LOOP && blockIdx.x == 0 && tid == 0 && p.count_out) *p.count_out = done_steps;
    if (tid == 0) *reinterpret_cast<volatile int*>(&pp.ms->cons_done) = 1;
  }
  __syncthreads();
}

template <int FMT, int NCHL>
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
      // after the wait: reads x of the previous kernel
      const GemvPlan plan = plan_phase(p, pp, k, token, tid, nullptr, p.epoch);
      (void)run_phase<FMT, NCHL, 4, false, false>(p, pp, plan, k, pos, tid, p.trace, p.epoch);
    }
    named_sync(BAR_CONS, NCT);
    if (tid == 0) *reinterpret_cast<volatile int*>(&pp.ms->cons_done) = 1;
  }
  __syncthreads();
}


// The instances one translation unit provides for its weight format (see mega_bf16.cu and
// mega_int4.cu): nchl is 4, 6 or 8; kind 0 the persistent kernel, 1 the same recording a timeline,
// 2 the per-phase kernel, 3 the persistent kernel with the token loop, 4 the persistent kernel with
// the column-split down projection (bf16 only).
#define TINFER_MEGA_CASES(FMT, N)                                                                \
  case N * 8 + 0: return reinterpret_cast<const void*>(&decode_megakernel<FMT, N, false, false>); \
  case N * 8 + 1: return reinterpret_cast<const void*>(&decode_megakernel<FMT, N, true, false>);  \
  case N * 8 + 2: return reinterpret_cast<const void*>(&decode_phase_kernel<FMT, N>);             \
  case N * 8 + 3: return reinterpret_cast<const void*>(&decode_megakernel<FMT, N, false, true>);  \
  case N * 8 + 4: return FMT == 0 ? reinterpret_cast<const void*>(                                \
                             &decode_megakernel<FMT, N, false, false, FMT == 0>) : nullptr;
#define TINFER_MEGA_INSTANCES(FMT, NAME)                                                          \
  const void* NAME(int nchl, int kind) {                                                          \
    switch (nchl * 8 + kind) {                                                                    \
      TINFER_MEGA_CASES(FMT, 4)                                                                   \
      TINFER_MEGA_CASES(FMT, 6)                                                                   \
      TINFER_MEGA_CASES(FMT, 8)                                                                   \
      default: return nullptr;                                                                    \
    }                                                                                             \
  }

}  // namespace tinfer
