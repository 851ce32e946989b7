// mega_bf16.cu -- instances of the persistent kernel and the per-phase kernel for bf16 weight
// matrices (one translation unit per format, compiled in parallel).
#include "megakernel.cuh"

namespace tinfer {

TINFER_MEGA_INSTANCES(0, step_kernel_bf16)

size_t static_smem_mega() { return sizeof(PhaseTable) + 256; }

}  // namespace tinfer
