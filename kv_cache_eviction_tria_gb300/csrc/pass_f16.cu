// Fused eviction pass, fp16 keys (instantiations of pass.cuh).
#include "pass.cuh"

namespace tria {

cudaError_t launch_pass_f16(FPass& P, cudaStream_t st) { return launch_pass_k<TRIA_F16>(P, st); }

}  // namespace tria
