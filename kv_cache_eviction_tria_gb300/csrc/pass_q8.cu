// Fused eviction pass, q8_0 keys (instantiations of pass.cuh).
#include "pass.cuh"

namespace tria {

cudaError_t launch_pass_q8(FPass& P, cudaStream_t st) { return launch_pass_k<TRIA_Q8_0>(P, st); }

}  // namespace tria
