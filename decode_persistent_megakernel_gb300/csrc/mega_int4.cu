// mega_int4.cu -- instances of the persistent kernel and the per-phase kernel for int4 weight
// matrices (one translation unit per format, compiled in parallel).
#include "megakernel.cuh"

namespace tinfer {

TINFER_MEGA_INSTANCES(1, step_kernel_int4)

}  // namespace tinfer
