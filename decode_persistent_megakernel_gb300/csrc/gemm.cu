// gemm.cu -- the dense contraction of a batched prefill on Blackwell's fifth-generation tensor cores:
// Y[M][N] = X[M][K] W[N][K]^T in bf16 with fp32 accumulation ("How I built an LLM inference engine
// from scratch in CUDA", "What I'd tell someone starting, and what's next": a prompt processed as
// one batch makes every linear layer a matrix-matrix product, the case tensor cores are for; and
// "Llama-1B: optimizing kernels": prefill runs GEMM kernels, decode GEMV kernels). Decode at batch 1
// stays on the CUDA cores (a matrix-vector stream); this is the path whose M is the prompt length.
//
// Persistent CTAs (one per SM) walk 128 x 256 tiles of Y (128 x 128 when the wider tiles would not
// cover the SMs: a short prompt), consecutive CTAs on the same W tile so that it is read from L2 by
// all of them. Warp 0's elected thread loads 128 x 64 tiles of X and 256 x 64
// tiles of W with the tensor memory accelerator (TMA), 128-byte swizzled, into a 4-stage
// shared-memory ring (full / empty mbarriers); warp 1's elected thread issues tcgen05.mma (M 128,
// N 256, K 16 per instruction, both operands K-major from shared memory) into one of two 256-column
// accumulators in tensor memory and tcgen05.commit frees each stage when its products are done;
// warps 4-7 drain the other accumulator (tcgen05.ld 32x32b, each warp its quarter of the lanes)
// while the next tile is computed. Every wait is bounded; tensor memory is always released.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <mutex>

#include "ptx.cuh"
#include "tinfer.h"

namespace tinfer {
namespace gemm {

constexpr int BM = 128, BK = 64;             // tile rows; BK bf16 = 128 bytes, one swizzle atom wide
constexpr int A_BYTES = BM * BK * 2;         // 16 KiB of X per stage
constexpr int NTHREADS = 256;
// Tile width BN (256, or 128 when 256-wide tiles would leave SMs idle): W bytes per stage, stages
// (the ring holds about 192 KiB), the dynamic shared memory with 1 KiB of alignment slack, and two
// fp32 accumulators of 128 lanes x BN columns in tensor memory.
template <int BN>
struct Tile {
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = BN == 256 ? 4 : 6;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024;
  static constexpr int TMEM_COLS = 2 * BN;
};
constexpr int EW_GEMM_TIMEOUT = 2;

// Shared-memory matrix descriptor of a K-major operand tile in the 128-byte swizzled layout that a
// TMA load with CU_TENSOR_MAP_SWIZZLE_128B writes: rows of 128 bytes, groups of 8 rows 1024 bytes
// apart (stride byte offset), the leading byte offset unused for this layout (1), descriptor
// version 1, layout type 2 (128-byte swizzle). The tile starts on a 1024-byte boundary.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, both K-major, N and M.
__host__ __device__ constexpr uint32_t instr_desc_bf16(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         int accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(tmem_d), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The mbarrier receives one arrival when every tcgen05.mma this thread issued before it is complete.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

// Bounded wait for the phase of `parity` of an mbarrier; false when it ran out.
__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t parity, long long timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity))
    if ((long long)(globaltimer() - t0) > timeout_ns) return false;
  return true;
}

struct GemmParams {
  int m, n, k;
  float* y;       // [m][n] fp32
  int* err;       // error word (bit EW_GEMM_TIMEOUT: a wait ran out)
  long long timeout_ns;
};

template <int BN>
__global__ void __launch_bounds__(NTHREADS, 1) gemm_bf16_tcgen05(const __grid_constant__ CUtensorMap map_x,
                                                                const __grid_constant__ CUtensorMap map_w,
                                                                const __grid_constant__ GemmParams q) {
  constexpr int STAGES = Tile<BN>::STAGES, STAGE_BYTES = Tile<BN>::STAGE_BYTES, TMEM_COLS = Tile<BN>::TMEM_COLS;
  extern __shared__ unsigned char smem_raw[];
  __shared__ __align__(8) unsigned long long full[STAGES], empty[STAGES], tfull[2], tempty[2];
  __shared__ uint32_t tmem_base_s;
  __shared__ int bad;
  __shared__ int go[2];  // epilogue: the poller's decision for tiles of even and odd parity
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t base = (smem_addr(smem_raw) + 1023u) & ~1023u;  // 1 KiB-aligned ring
  const int tiles_m = (q.m + BM - 1) / BM, tiles_n = (q.n + BN - 1) / BN;
  const int ntiles = tiles_m * tiles_n;
  const int nk = (q.k + BK - 1) / BK;
  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_addr(&full[s]), 1);
      mbar_init(smem_addr(&empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_addr(&tfull[b]), 1);   // the MMA thread's commit
      mbar_init(smem_addr(&tempty[b]), 4);  // one arrival per epilogue warp
    }
    bad = 0;
    mbar_fence_init();
  }
  if (warp == 2) {  // two 128 x BN fp32 accumulators
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&tmem_base_s)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  volatile int* failed = &bad;  // read again on every turn: a failed role stops the others promptly
  // tile t of this CTA: t = blockIdx.x + i * gridDim.x; consecutive t share the W tile (n)
  auto tile_mn = [&](int t, int& m0, int& n0) {
    m0 = (t % tiles_m) * BM;
    n0 = (t / tiles_m) * BN;
  };

  if (warp == 0 && lane == 0) {
    // producer: stage s of round r waits until the products of round r - 1 freed it
    uint32_t it = 0;
    for (int t = blockIdx.x; t < ntiles && !*failed; t += gridDim.x) {
      int m0, n0;
      tile_mn(t, m0, n0);
      for (int kb = 0; kb < nk; ++kb, ++it) {
        const int s = (int)(it % STAGES);
        const uint32_t r = it / STAGES;
        if (!bar_wait(smem_addr(&empty[s]), (r & 1u) ^ 1u, q.timeout_ns)) { *failed = 1; break; }
        const uint32_t st = base + (uint32_t)s * STAGE_BYTES;
        mbar_arrive_expect_tx(smem_addr(&full[s]), STAGE_BYTES);
        tma_load_2d(st, &map_x, kb * BK, m0, smem_addr(&full[s]));
        tma_load_2d(st + A_BYTES, &map_w, kb * BK, n0, smem_addr(&full[s]));
      }
    }
  } else if (warp == 1 && lane == 0) {
    // MMA issuer: accumulator b of its u-th use waits until the epilogue drained use u - 1
    const uint32_t idesc = instr_desc_bf16(BM, BN);
    uint32_t it = 0, tc = 0;
    for (int t = blockIdx.x; t < ntiles && !*failed; t += gridDim.x, ++tc) {
      const uint32_t b = tc & 1u, u = tc >> 1;
      if (!bar_wait(smem_addr(&tempty[b]), (u & 1u) ^ 1u, q.timeout_ns)) { *failed = 1; break; }
      tc_fence_after();
      const uint32_t acc = tmem + b * BN;
      for (int kb = 0; kb < nk; ++kb, ++it) {
        const int s = (int)(it % STAGES);
        const uint32_t r = it / STAGES;
        if (!bar_wait(smem_addr(&full[s]), r & 1u, q.timeout_ns)) { *failed = 1; break; }
        tc_fence_after();
        const uint32_t st = base + (uint32_t)s * STAGE_BYTES;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          mma_bf16(acc, smem_desc_sw128(st + 32u * kk), smem_desc_sw128(st + A_BYTES + 32u * kk), idesc,
                   (kb | kk) != 0);
        mma_commit(smem_addr(&empty[s]));  // the stage is free once these products are done
      }
      mma_commit(smem_addr(&tfull[b]));  // this tile's accumulator is complete
      if (*failed) break;
    }
  } else if (warp >= 4) {
    // epilogue: warp 4 + e drains accumulator lanes 32 e .. 32 e + 31 (rows m0 + 32 e + lane)
    const int e = warp - 4;
    const bool vec = (q.n & 3) == 0 && (reinterpret_cast<uintptr_t>(q.y) & 15) == 0;
    uint32_t tc = 0;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++tc) {
      const uint32_t b = tc & 1u, u = tc >> 1;
      // one thread polls for the accumulator; the other epilogue threads wait at a named barrier,
      // which takes no issue slots from the producer and MMA threads sharing their schedulers. The
      // poller's decision (in a slot of its own per tile parity) is what every epilogue thread
      // follows, so that all of them pass the same barriers.
      if (e == 0 && lane == 0) {
        const bool ok = !*failed && bar_wait(smem_addr(&tfull[b]), u & 1u, q.timeout_ns);
        if (!ok) *failed = 1;
        go[tc & 1u] = ok ? 1 : 0;
      }
      named_sync(1, 128);
      if (!reinterpret_cast<volatile int*>(go)[tc & 1u]) break;
      tc_fence_after();
      int m0, n0;
      tile_mn(t, m0, n0);
      const int row = m0 + 32 * e + lane;
      for (int c0 = 0; c0 < BN; c0 += 32) {
        uint32_t v[32];
        const uint32_t taddr = tmem + ((uint32_t)(32 * e) << 16) + b * BN + (uint32_t)c0;
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
            "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
            : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
              "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
              "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]),
              "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]),
              "=r"(v[30]), "=r"(v[31])
            : "r"(taddr));
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        if (row < q.m) {
          float* yr = q.y + (size_t)row * q.n + n0 + c0;
          const int lim = q.n - (n0 + c0);  // columns of this chunk inside Y
          if (vec && lim >= 32) {
#pragma unroll
            for (int i = 0; i < 32; i += 4)
              *reinterpret_cast<float4*>(yr + i) = make_float4(__uint_as_float(v[i]), __uint_as_float(v[i + 1]),
                                                              __uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]));
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (i < lim) yr[i] = __uint_as_float(v[i]);
          }
        }
      }
      // the accumulator may be overwritten once all four warps have read it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&tempty[b]));
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && *failed) atomicOr(q.err, EW_GEMM_TIMEOUT);
  if (warp == 2)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
}

// ---------------------------------------------------------------------------------------- host

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &qr) == cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// A [rows][k] bf16 row-major matrix as a 2-D tensor map with box_rows x 64 boxes, 128-byte swizzle
// and zero fill past its edges.
bool make_map(CUtensorMap* map, const void* ptr, int rows, int k, int box_rows) {
  const auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)k, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)k * 2};
  const cuuint32_t box[2] = {BK, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct ErrWord {
  int* p = nullptr;
  int device = -1;
};
ErrWord g_err;
std::mutex g_err_mu;

}  // namespace gemm
}  // namespace tinfer

using namespace tinfer;

extern "C" tinfer_status tinfer_op_gemm_bf16(int m, int n, int k, const void* x_dev, const void* w_dev,
                                             float* y_dev, void* stream) {
  if (m <= 0 || n <= 0 || k <= 0 || !x_dev || !w_dev || !y_dev) return TINFER_ERR_INVALID_ARG;
  // the tensor maps need 16-byte aligned bases and row strides (k a multiple of 8)
  if (k % 8 || (reinterpret_cast<uintptr_t>(x_dev) & 15) || (reinterpret_cast<uintptr_t>(w_dev) & 15) ||
      (reinterpret_cast<uintptr_t>(y_dev) & 3))
    return TINFER_ERR_INVALID_ARG;
  if ((long long)((m + gemm::BM - 1) / gemm::BM) * ((n + 127) / 128) > (1LL << 30)) return TINFER_ERR_UNSUPPORTED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return TINFER_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lk(gemm::g_err_mu);
    if (!gemm::g_err.p || gemm::g_err.device != dev) {
      if (cudaMalloc(&gemm::g_err.p, 16) != cudaSuccess) return TINFER_ERR_OOM;
      gemm::g_err.device = dev;
    }
  }
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return TINFER_ERR_CUDA;
  // 128 x 256 tiles, or 128 x 128 ones when the wider tiles would not cover the SMs (short prompts)
  const long long tiles_m = (m + gemm::BM - 1) / gemm::BM;
  const int bn = tiles_m * ((n + 255) / 256) < sms ? 128 : 256;
  const long long tiles = tiles_m * ((n + bn - 1) / bn);
  CUtensorMap mx, mw;
  if (!gemm::make_map(&mx, x_dev, m, k, gemm::BM) || !gemm::make_map(&mw, w_dev, n, k, bn))
    return TINFER_ERR_UNSUPPORTED;
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(gemm::gemm_bf16_tcgen05<256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    gemm::Tile<256>::SMEM_BYTES);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(gemm::gemm_bf16_tcgen05<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      gemm::Tile<128>::SMEM_BYTES);
  });
  if (attr_err != cudaSuccess) return TINFER_ERR_CUDA;
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemsetAsync(gemm::g_err.p, 0, 4, st) != cudaSuccess) return TINFER_ERR_CUDA;
  gemm::GemmParams q{m, n, k, y_dev, gemm::g_err.p, 200LL * 1000 * 1000};
  const int grid = (int)(tiles < sms ? tiles : sms);  // persistent: one CTA per SM at most
  if (bn == 256)
    gemm::gemm_bf16_tcgen05<256><<<grid, gemm::NTHREADS, gemm::Tile<256>::SMEM_BYTES, st>>>(mx, mw, q);
  else
    gemm::gemm_bf16_tcgen05<128><<<grid, gemm::NTHREADS, gemm::Tile<128>::SMEM_BYTES, st>>>(mx, mw, q);
  if (cudaGetLastError() != cudaSuccess) return TINFER_ERR_CUDA;
  int h = 0;
  if (cudaMemcpyAsync(&h, gemm::g_err.p, 4, cudaMemcpyDeviceToHost, st) != cudaSuccess) return TINFER_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return TINFER_ERR_CUDA;
  return h ? TINFER_ERR_TIMEOUT : TINFER_OK;
}
