// engine.h -- internal structures of the decode engine, shared by its host and device code.
#pragma once
#include <cstddef>
#include <cstdint>

#ifdef __CUDACC__
#define TINFER_HD __host__ __device__
#else
#define TINFER_HD
#endif

namespace tinfer {

// Thread block: NCW consumer warps that compute, plus one producer warp whose elected lane streams
// weight and K/V bytes into the shared-memory ring with bulk asynchronous copies.
constexpr int NCW = 8;
constexpr int NCT = NCW * 32;
constexpr int NTHREADS = NCT + 32;
// The persistent kernel runs a 4-warp producer group instead of one producer warp, so that the two
// groups can trade registers (setmaxnreg): the producer group keeps REG_PRODUCER registers per
// thread (its copy cursor and the L2 lookahead cursor), the consumer warps grow to REG_CONSUMER.
// Launch total: 12 warps x 32 x 168 = 64512 = 8 x 32 x REG_CONSUMER + 4 x 32 x REG_PRODUCER.
constexpr int NTHREADS_MEGA = NCT + 128;
// The int4 instances carry a second GEMV (int4 linears and the bf16 LM head) and the dequantisation
// temporaries, so their consumers take more and their producer group less.
constexpr int REG_CONSUMER = 200, REG_CONSUMER_INT4 = 216;
constexpr int REG_PRODUCER = 104, REG_PRODUCER_INT4 = 72;
static_assert(NCW * 32 * REG_CONSUMER + 4 * 32 * REG_PRODUCER <= (NTHREADS_MEGA / 32) * 32 * 168,
              "register split exceeds the launch allocation");
static_assert(NCW * 32 * REG_CONSUMER_INT4 + 4 * 32 * REG_PRODUCER_INT4 <= (NTHREADS_MEGA / 32) * 32 * 168,
              "register split exceeds the launch allocation");
constexpr int MAX_STAGES = 8;  // ring stages of the shared-memory weight ring, at most
constexpr int NR_MAX = 32;    // rows of one matrix held by one ring stage, at most
constexpr int G_MAX = 8;      // query heads sharing one KV head, at most
constexpr int D_MAX = 128;    // head_dim, at most
constexpr int T_MAX = 256;    // cache slots in one attention chunk, at most
constexpr int MAX_LAYERS = 64;   // layer descriptors travel in the kernel parameters

enum Phase : int { PH_QKV = 0, PH_ATTN = 1, PH_O = 2, PH_GU = 3, PH_DOWN = 4, PH_LM = 5 };
constexpr int PHASES_PER_LAYER = 5;

// bits of the device error word
enum : int {
  EW_NONFINITE = 1,
  EW_TIMEOUT = 2,
  EW_BADTOKEN = 4,
};

struct __align__(8) LayerDev {
  const uint8_t* qkv;   // [(nq + 2 nkv) d] packed rows of hidden inputs
  const uint8_t* o;     // [hidden] packed rows of nq*d inputs
  const uint8_t* gu;    // [2 ffn] packed rows (gate, up interleaved) of hidden inputs
  const uint8_t* down;  // [hidden] packed rows of ffn inputs
  const float* g1;      // [hidden]
  const float* g2;      // [hidden]
  const float* bias;    // [(nq + 2 nkv) d] or nullptr
};

struct Dims {
  int L, H, nq, nkv, d, F, V, max_ctx;
  int fmt;         // 0 bf16, 1 int4
  int group;       // int4 inputs per scale
  int scale_bf16;  // int4 scale format (0 fp16, 1 bf16)
  float eps;
  int rb_h, rb_qd, rb_f;  // packed row bytes for hidden, nq*d and ffn inputs
  int rb_lm;              // bf16 LM head row bytes (2 * hidden)
  int qkv_rows;           // (nq + 2 nkv) * d
  int nchl;               // bf16 GEMV instance of the step kernels: 16-byte chunks per lane (4, 6, 8)
  int ffn_split;          // down projection split by columns (Wd stored transposed: [F][H])
};

// Everything one step needs; passed by value to every kernel (16-byte multiple: copied to shared
// memory in 16-byte words).
struct __align__(16) StepParams {
  Dims m;
  LayerDev layers[MAX_LAYERS];  // read through the constant cache
  const uint16_t* embed;
  const uint16_t* lm_head;
  const uint16_t* final_norm;
  uint16_t* kcache;
  uint16_t* vcache;
  const float2* rope;      // [max_ctx][d/2] (cos, sin)
  // Activations handed from one phase to the next, as stamped words: the low 32 bits hold the fp32
  // value, the high 32 bits the stamp of the phase that wrote it (epoch + phase index). A reader
  // waits for the stamp it expects instead of for a grid barrier.
  uint64_t* xa;            // [H] residual stream after the attention block of a layer
  uint64_t* xb;            // [H] residual stream after the MLP block of a layer
  uint64_t* qkv;           // [qkv_rows]
  uint64_t* attn;          // [nq * d]
  uint64_t* act;           // [F]
  uint64_t* part_ffn;      // [grid][H] column-split down projection: per-CTA partial sums (stamped)
  unsigned epoch;          // stamps of this launch: phase k writes epoch + k
  int sync_barrier;        // 1: a grid barrier before every phase (the grid-barrier schedule)
  unsigned long long* bar_count;  // its monotonic arrival counter
  unsigned long long bar_base;    // barriers completed before this launch
  int stamp_check;         // readers wait for the stamp (persistent kernel); 0: stream order suffices
  float* part_m;           // [nq][nch_cap]      (per-phase kernels: ticket merge)
  float* part_l;           // [nq][nch_cap]
  float* part_o;           // [nq][nch_cap][d]
  uint64_t* part_mw;       // [nq][nch_cap]      stamped copies (persistent kernel: every unit
  uint64_t* part_lw;       // [nq][nch_cap]      merges a slice of its head's outputs)
  uint64_t* part_ow;       // [nq][nch_cap][d]
  unsigned* tickets;       // [nkv + 1]: attention merge per KV head, then the argmax ticket
  float* best_val;         // [grid]
  int* best_idx;           // [grid]
  int* best_bad;           // [grid]
  int* err;                // device error word
  int* err_host;           // mapped pinned host mirror of the error word (may be null)
  int nch_cap;             // capacity of the partial buffers in chunks per head
  int grid;                // CTAs
  int ring_stages;
  int slot_bytes;
  int inflight;            // bulk copies the producer keeps outstanding at most
  int inflight_lm;         // the same during the LM head, which streams from HBM with nothing to overlap
  int l2_lookahead;        // persistent kernel: bytes per CTA prefetched into L2 ahead of the ring
  int l2_pace_ns_per_kb;   // spacing of those prefetches (about the per-SM share of HBM bandwidth)
  long long timeout_ns;
  // per step
  int token;               // used when token_dev is null
  const int* token_dev;
  int pos;                 // used when step_dev is null
  const int* step_dev;     // graph mode: {token, pos} written by the step's first node
  int n_chunks_override;   // >0: fixed number of attention chunks (single-op test path)
  float* logits;           // [V] or null
  int* argmax;             // [1]
  // the in-kernel token loop (persistent kernel): n_steps decode steps in one launch, step s at
  // position pos + s, its token the greedy choice of step s - 1
  int n_steps;             // 1: one step (argmax through the ticketed last CTA)
  int* tokens_out;         // [n_steps] greedy token of every step (-1: a non-finite logit)
  int* count_out;          // steps completed, or null
  int eos;                 // stop after a step that chose this token (-1: never)
  uint64_t* best_w;        // [grid][2] per-CTA best of the LM head as stamped words (value; index)
  unsigned* kvflag;        // [nkv] token loop: the first stamp of the step whose K/V slot is visible
  int dbg_skip_cta;        // fault injection: CTA that withholds its results of one GEMV phase (-1 none)
  int dbg_skip_phase;      // ... the phase index
  unsigned long long* trace;  // optional timeline [grid][phases][TRACE_FIELDS] of %globaltimer ns
};

// Timeline fields recorded per CTA and phase when StepParams::trace is set.
enum TraceField : int {
  TR_START = 0,      // consumers begin the phase
  TR_READY = 1,      // activations loaded (norm done): the stage loop starts
  TR_END = 2,        // consumers done with the phase
  TR_PROD_BEGIN = 3, // producer starts issuing the phase's copies
  TR_PROD_END = 4,   // producer has issued the phase's last copy
  TR_ACT = 5,        // the phase's input activations are in registers (before the norm)
  TR_ENTRY = 6,      // the GEMV code of the phase starts (after the phase set-up)
  TR_FETCHED = 7,    // the input vector is in shared memory
  TR_AUX0 = 8,       // GEMV: the first weight stage is in; attention: the first unit's values are in
  TR_AUX1 = 9,       // GEMV: the last weight stage is consumed; attention: merge started
  TRACE_FIELDS = 10
};

// Op-level GEMV description (the single-operation entry point uses the same device code).
struct GemvOp {
  const uint8_t* w;
  int rows, cols, rb;
  int fmt, group, scale_bf16;
  const float* x;
  const float* gain;   // nullptr: no RMSNorm prologue
  float eps;
  const float* bias;
  int epi;             // TINFER_EPI_*
  float* y;
  int* argmax;
};

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }


constexpr int SEG_MAX_INPUTS = 2048;  // inputs of one row segment (activations held per lane: 64)
constexpr int ROWV_MAX = 4096;        // row results of one phase kept in shared memory per CTA

// GEMV row segmenting: a row of `cols` inputs is cut into nseg (a power of two, at most NCW)
// contiguous segments of ks inputs, chs 16-byte chunks each. A warp owns one segment of a row; the
// activations of that segment stay in its lanes' registers (chunk c = lane + 32 k). bf16 rows are
// halved while their segments hold 2048 inputs or more, so that a 2048-input row becomes two
// 1024-input segments: every warp then takes two segments of each 8-row ring stage instead of one
// whole row, which halves the stage hand-offs per byte and the activation registers, while rows of
// 1024-2047 inputs stay whole (each lane keeps at least four chunks). int4 rows keep up to 2048
// inputs, which is what fills their lanes' two chunks.
struct SegInfo {
  int nseg, ks, chs;
};
TINFER_HD inline SegInfo seg_info(int fmt, int cols) {
  const int E = fmt ? 32 : 8;
  int nseg = 1;
  while (nseg < NCW && (cols / nseg > SEG_MAX_INPUTS || (fmt == 0 && cols / nseg >= SEG_MAX_INPUTS)))
    nseg *= 2;
  return SegInfo{nseg, cols / nseg, cols / nseg / E};
}
// True when the segmenting covers the row exactly and fits the per-lane register budget.
TINFER_HD inline bool seg_ok(int fmt, int cols) {
  const int E = fmt ? 32 : 8;
  const SegInfo s = seg_info(fmt, cols);
  return cols % s.nseg == 0 && s.ks % E == 0 && s.ks <= SEG_MAX_INPUTS && (s.chs + 31) / 32 <= 8;
}
// Rows of one ring stage: as many as fit a slot, rounded down to a multiple of the warps that
// share a stage (NCW / nseg) and of the row quantum (2 for gate/up pairs), at least one quantum.
TINFER_HD inline int stage_rows(int fmt, int cols, int rb, int slot, int quantum) {
  const SegInfo s = seg_info(fmt, cols);
  int wg = NCW / s.nseg;
  int step = wg % quantum == 0 ? wg : wg * quantum;
  int fit = slot / rb;
  if (fit > NR_MAX) fit = NR_MAX;
  int nr = fit - fit % step;
  if (nr == 0) nr = fit - fit % quantum;
  return nr;
}

// The bf16 GEMV instance (chunks per lane, 4, 6 or 8) that covers rows of every given width; 0 when
// some width does not fit the register budget.
inline int nchl_instance(const int* cols, int n) {
  int need = 1;
  for (int i = 0; i < n; ++i) {
    if (!seg_ok(0, cols[i])) return 0;
    const int c = (seg_info(0, cols[i]).chs + 31) / 32;
    if (c > need) need = c;
  }
  return need <= 4 ? 4 : need <= 6 ? 6 : 8;
}

// Packed row bytes: bf16 rows are 2*cols (cols % 8 == 0); int4 rows are cols/2 nibble bytes plus
// 2*cols/group scale bytes, padded to 16 (cols % 32 == 0, group % 32 == 0, cols % group == 0).
inline size_t packed_row_bytes(int fmt, int cols, int group) {
  if (cols <= 0) return 0;
  if (fmt == 0) return (cols % 8 == 0) ? (size_t)cols * 2 : 0;
  if (group <= 0 || group % 32 != 0 || cols % 32 != 0 || cols % group != 0) return 0;
  return align_up((size_t)cols / 2 + (size_t)2 * (cols / group), 16);
}

struct LayerLayout {
  size_t off_qkv, off_o, off_gu, off_down, off_g1, off_g2, off_bias, total;
};

inline LayerLayout layer_layout(int H, int nq, int nkv, int d, int F, int fmt, int group, int bias) {
  LayerLayout L{};
  size_t rbh = packed_row_bytes(fmt, H, group), rbq = packed_row_bytes(fmt, nq * d, group);
  size_t rbf = packed_row_bytes(fmt, F, group);
  size_t qkv_rows = (size_t)(nq + 2 * nkv) * d;
  size_t o = 0;
  L.off_qkv = o;  o = align_up(o + qkv_rows * rbh, 256);
  L.off_o = o;    o = align_up(o + (size_t)H * rbq, 256);
  L.off_gu = o;   o = align_up(o + (size_t)2 * F * rbh, 256);
  L.off_down = o; o = align_up(o + (size_t)H * rbf, 256);
  L.off_g1 = o;   o = align_up(o + (size_t)H * 4, 256);
  L.off_g2 = o;   o = align_up(o + (size_t)H * 4, 256);
  L.off_bias = bias ? o : 0;
  if (bias) o = align_up(o + qkv_rows * 4, 256);
  L.total = o;
  return L;
}

}  // namespace tinfer
