// Shared-slot variant: one keep-set per token for all layers and KV heads.
//
// Sources cited by page title and section:
//   [Doc] "TriAttention KV-Cache Eviction (--triattention)": §5 Phase B (score
//         each cached token, keep the best, compact in place) and Phase C
//         (per-query-head z-normalisation, max across the GQA group), whose
//         Vulkan port lists a global z-normalisation shader for caches whose
//         token cells are shared by every layer.
//   [Worklog] "TriAttention Native C++ Worklog": the per-layer / aggregated
//         score comparison that names cross-layer aggregation.
// The pages do not state how the per-(layer, KV head) scores of a token
// combine; the reading taken here extends the GQA rule: a token's score is
// the maximum of its z-max scores over all layers and KV heads (NaN scores
// are ignored unless all are NaN).
#include <math.h>

#include "tria_internal.cuh"

namespace tria {

namespace {

// combined[row0_s + t] = max over layers l and KV heads g of
// scores[l * stride + row0_s + g * cap_s + t], t < n_live[s]
__global__ void __launch_bounds__(kThreads) k_shared_combine(const Pass P, const float* __restrict__ scores,
                                                            int64_t stride, int n_layers, float* combined) {
  const int s = blockIdx.y;
  const SeqInfo& q = P.seq[s];
  const int n = *((volatile const int32_t*)(P.n_live + s));
  if (n < 0 || n > q.cap) {
    if (blockIdx.x == 0 && threadIdx.x == 0) report(P.ctrl, TRIA_ERR_DEVICE_ARG, (uint32_t)s);
    return;
  }
  for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < n; t += gridDim.x * blockDim.x) {
    float m = NAN;
    for (int l = 0; l < n_layers; ++l) {
      const float* sl = scores + (size_t)l * stride + q.row0 + t;
      for (int g = 0; g < P.n_kv; ++g) m = fmaxf(m, __ldg(sl + (size_t)g * q.cap));
    }
    combined[q.row0 + t] = m;
  }
}

// keep lists of the KV-head-0 slot copied to the other KV heads of the
// sequence: entries i < min(n_live, B)
__global__ void __launch_bounds__(kThreads) k_shared_broadcast(const Pass P, int32_t* keep) {
  const int s = blockIdx.y;
  const SeqInfo& q = P.seq[s];
  const int n = *((volatile const int32_t*)(P.n_live + s));
  if (n < 0 || n > q.cap) return;   // reported by the select
  const int m = min(n, q.budget);
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < m; i += gridDim.x * blockDim.x) {
    const int32_t v = keep[q.row0 + i];
    for (int g = 1; g < P.n_kv; ++g) keep[q.row0 + (int64_t)g * q.cap + i] = v;
  }
}

int row_blocks(const Pass& P) {
  int cap_max = 1;
  for (int s = 0; s < P.n_seqs; ++s) cap_max = cap_max > P.seq[s].cap ? cap_max : P.seq[s].cap;
  const int b = (cap_max + kThreads - 1) / kThreads;
  return b < 64 ? b : 64;
}

}  // namespace

cudaError_t launch_shared_combine(const Pass& P, const float* scores, int64_t stride, int n_layers, float* combined,
                                  cudaStream_t st) {
  k_shared_combine<<<dim3(row_blocks(P), P.n_seqs), kThreads, 0, st>>>(P, scores, stride, n_layers, combined);
  return cudaGetLastError();
}

cudaError_t launch_shared_broadcast(const Pass& P, int32_t* keep, cudaStream_t st) {
  k_shared_broadcast<<<dim3(row_blocks(P), P.n_seqs), kThreads, 0, st>>>(P, keep);
  return cudaGetLastError();
}

}  // namespace tria
