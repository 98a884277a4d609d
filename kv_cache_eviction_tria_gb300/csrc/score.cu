// Score stage: raw per-query-head scores, per-segment moments, z-max score.
//
// [Worklog] "TriAttention Native C++ Worklog", Phase 9 (direct K_rot scorer:
// Q_mean * conj(K_rot), query-side trig term only, additive MLR term on
// |K_rot|) and 2026-04-18 (phases from the absolute decode position).
// [Doc] "TriAttention KV-Cache Eviction (--triattention)", §5 Phase C
// (z-normalise each query head, then max over the GQA group).
//
// Per row r and query head h of the segment's group:
//   raw_h(r) = sum_f  Wr_{h,f} K[r][f] + Wi_{h,f} K[r][f+fc] + M_{h,f} |k_f|
// with W = qbar E_f e^{i w_f p} (built once per CTA) and M = q_abs - |qbar|.
//
// Layout of the work: one CTA = one chunk of rows of one segment; each of its
// 8 warps owns a contiguous piece of the chunk, which one lane brings into
// shared memory with a single bulk async copy (TMA, non-tensor form) completed
// on the warp's own mbarrier. A row is handled by TPR lanes; lane q holds the
// PPT frequency pairs [q*PPT, q*PPT+PPT) of every head in registers, reads the
// matching 2*PPT elements (both NEOX halves) of the row from shared memory,
// and the TPR partial sums are combined with warp shuffles.
#include "tria_internal.cuh"

namespace tria {

template <int KT, int PPT>
struct Loader;

template <int PPT>
struct Loader<TRIA_F16, PPT> {
  static __device__ __forceinline__ void half(const uint8_t* row, int e0, float* x) {
    const __half2* p = reinterpret_cast<const __half2*>(row + 2 * e0);
    if constexpr (PPT == 8) {
      uint4 u = *reinterpret_cast<const uint4*>(p);
      const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float2 f = __half22float2(h[i]);
        x[2 * i] = f.x;
        x[2 * i + 1] = f.y;
      }
    } else {
      uint2 u = *reinterpret_cast<const uint2*>(p);
      const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        float2 f = __half22float2(h[i]);
        x[2 * i] = f.x;
        x[2 * i + 1] = f.y;
      }
    }
  }
};

template <int PPT>
struct Loader<TRIA_F32, PPT> {
  static __device__ __forceinline__ void half(const uint8_t* row, int e0, float* x) {
    const float4* p = reinterpret_cast<const float4*>(row + 4 * e0);
#pragma unroll
    for (int i = 0; i < PPT / 4; ++i) {
      float4 v = p[i];
      x[4 * i] = v.x;
      x[4 * i + 1] = v.y;
      x[4 * i + 2] = v.z;
      x[4 * i + 3] = v.w;
    }
  }
};

template <int PPT>
struct Loader<TRIA_Q8_0, PPT> {
  static __device__ __forceinline__ void half(const uint8_t* row, int e0, float* x) {
    if constexpr (PPT == 8) {
      uint2 u = *reinterpret_cast<const uint2*>(row + e0);
#pragma unroll
      for (int i = 0; i < 4; ++i) x[i] = (float)(int)(int8_t)(u.x >> (8 * i));
#pragma unroll
      for (int i = 0; i < 4; ++i) x[4 + i] = (float)(int)(int8_t)(u.y >> (8 * i));
    } else {
      uint32_t u = *reinterpret_cast<const uint32_t*>(row + e0);
#pragma unroll
      for (int i = 0; i < 4; ++i) x[i] = (float)(int)(int8_t)(u >> (8 * i));
    }
  }
};

struct ScoreSmem {
  // byte offsets inside dynamic shared memory
  int data, w, m, raw, bar, total;
};

__host__ __device__ inline ScoreSmem score_smem_layout(int cs_rows, int k_rb, int G, int fc) {
  ScoreSmem L;
  int off = 0;
  L.data = off;
  off += cs_rows * k_rb;
  off = (off + 15) & ~15;
  L.w = off;
  off += G * fc * 8;
  L.m = off;
  off += G * fc * 4;
  off = (off + 15) & ~15;
  L.raw = off;
  off += cs_rows * G * 4;
  off = (off + 15) & ~15;
  L.bar = off;
  off += 8 * 8;
  L.total = off;
  return L;
}

template <int KT, int G, int TPR, int PPT>
__global__ void __launch_bounds__(kThreads, 2) k_score(const __grid_constant__ Pass P) {
  const int seg = blockIdx.y;
  const SegView sv = seg_view(P, seg);
  if (!sv.valid) {
    if (blockIdx.x == 0 && threadIdx.x == 0) report(P.ctrl, TRIA_ERR_DEVICE_ARG, (uint32_t)sv.s);
    return;
  }
  if (P.only_active && !sv.active) return;
  const int n = sv.n;
  const int c0 = blockIdx.x * P.cs_rows;
  if (c0 >= n) return;
  const int rows = min(P.cs_rows, n - c0);
  const int nchunks = (n + P.cs_rows - 1) / P.cs_rows;
  const int fc = P.fc;
  const int k_rb = P.k_rb;

  extern __shared__ __align__(128) uint8_t smem[];
  const ScoreSmem L = score_smem_layout(P.cs_rows, k_rb, G, fc);
  uint8_t* sdata = smem + L.data;
  float2* sW = reinterpret_cast<float2*>(smem + L.w);
  float* sM = reinterpret_cast<float*>(smem + L.m);
  float* sraw = reinterpret_cast<float*>(smem + L.raw);
  uint64_t* sbar = reinterpret_cast<uint64_t*>(smem + L.bar);
  __shared__ int s_last;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int piece_rows = P.cs_rows >> 3;
  const int pr0 = warp * piece_rows;
  const int prows = max(0, min(piece_rows, rows - pr0));

  // 1. each warp starts the bulk copy of its piece
  if (lane == 0) {
    mbar_init(&sbar[warp], 1);
    fence_mbar_init();
  }
  __syncwarp();
  if (lane == 0 && prows > 0) {
    const uint32_t bytes = (uint32_t)(prows * k_rb);
    mbar_arrive_expect_tx(&sbar[warp], bytes);
    bulk_g2s(sdata + (size_t)pr0 * k_rb, P.k + (size_t)(sv.row0 + c0 + pr0) * k_rb, bytes, &sbar[warp]);
  }

  // 2. folded weights of this segment at the current position:
  //    W = qe * e^{i w_f p}, phase from the exact fixed-point turn count
  const unsigned long long p = (unsigned long long)P.seq[sv.s].cur_pos;
  const float2* qe = P.qe + (size_t)sv.g * G * fc;
  const float* mw = P.mw + (size_t)sv.g * G * fc;
  for (int i = threadIdx.x; i < G * fc; i += blockDim.x) {
    const int f = i % fc;
    const unsigned long long x = P.turns[f] * p;
    const float half_turns = (float)(int)(x >> 32) * 0x1p-31f;   // [-1, 1) half turns
    float sn, cs;
    sincospif(half_turns, &sn, &cs);
    const float2 q = qe[i];
    sW[i] = make_float2(q.x * cs - q.y * sn, q.x * sn + q.y * cs);
    sM[i] = mw[i];
  }
  __syncthreads();

  // 3. this lane's pairs of every head into registers
  const int q = lane % TPR;
  const int f0 = q * PPT;
  const bool lane_on = f0 < fc;
  float wr[G][PPT], wi[G][PPT], wm[G][PPT];
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int j = 0; j < PPT; ++j) {
      const int idx = h * fc + f0 + j;
      const bool on = lane_on;
      const float2 w2 = on ? sW[idx] : make_float2(0.f, 0.f);
      wr[h][j] = w2.x;
      wi[h][j] = w2.y;
      wm[h][j] = on ? sM[idx] : 0.f;
    }

  // 4. rows of my piece
  if (prows > 0) {
    if (!mbar_wait_bounded(&sbar[warp], 0, P.spin_limit)) {
      if (lane == 0) report(P.ctrl, TRIA_ERR_TIMEOUT, (uint32_t)seg);
    } else {
      constexpr int kRowsPerStep = 32 / TPR;
      const int steps = (prows + kRowsPerStep - 1) / kRowsPerStep;
      for (int stp = 0; stp < steps; ++stp) {
        const int rr = stp * kRowsPerStep + lane / TPR;
        const bool row_on = rr < prows;
        float kr[PPT], ki[PPT];
        if (row_on && lane_on) {
          const uint8_t* row = sdata + (size_t)(pr0 + rr) * k_rb;
          Loader<KT, PPT>::half(row, f0, kr);
          Loader<KT, PPT>::half(row, fc + f0, ki);
          if constexpr (KT == TRIA_Q8_0) {
            const __half* sc = reinterpret_cast<const __half*>(P.ks + (size_t)(sv.row0 + c0 + pr0 + rr) * P.ks_rb);
            const float d1 = __half2float(sc[f0 >> 5]);
            const float d2 = __half2float(sc[(fc + f0) >> 5]);
#pragma unroll
            for (int j = 0; j < PPT; ++j) {
              kr[j] *= d1;
              ki[j] *= d2;
            }
          }
        } else {
#pragma unroll
          for (int j = 0; j < PPT; ++j) kr[j] = ki[j] = 0.f;
        }
        float acc[G];
#pragma unroll
        for (int h = 0; h < G; ++h) acc[h] = 0.f;
#pragma unroll
        for (int j = 0; j < PPT; ++j) {
          const float mag = sqrtf(fmaf(kr[j], kr[j], ki[j] * ki[j]));
#pragma unroll
          for (int h = 0; h < G; ++h) {
            acc[h] = fmaf(wr[h][j], kr[j], acc[h]);
            acc[h] = fmaf(wi[h][j], ki[j], acc[h]);
            acc[h] = fmaf(wm[h][j], mag, acc[h]);
          }
        }
#pragma unroll
        for (int o = TPR / 2; o > 0; o >>= 1)
#pragma unroll
          for (int h = 0; h < G; ++h) acc[h] += __shfl_xor_sync(0xffffffffu, acc[h], o);
        // every lane holds all G sums; lane q writes the heads h with h % TPR == q
        if (row_on) {
#pragma unroll
          for (int h = 0; h < G; ++h)
            if ((h % TPR) == q) sraw[(pr0 + rr) * G + h] = acc[h];
        }
      }
    }
  }
  __syncthreads();

  // 5. raw scores out (coalesced) and the chunk's moments (two passes in fp32)
  float* graw = P.raw + (size_t)(sv.row0 + c0) * G;
  for (int i = threadIdx.x; i < rows * G; i += blockDim.x) graw[i] = sraw[i];
  if (warp < G) {
    float sum = 0.f;
    for (int r = lane; r < rows; r += 32) sum += sraw[r * G + warp];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    const float mean = sum / (float)rows;
    float m2 = 0.f;
    for (int r = lane; r < rows; r += 32) {
      const float dlt = sraw[r * G + warp] - mean;
      m2 = fmaf(dlt, dlt, m2);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m2 += __shfl_xor_sync(0xffffffffu, m2, o);
    if (lane == 0) {
      ScoreChunk* sc = P.schunk + (size_t)seg * P.cs_max + blockIdx.x;
      sc->mean[warp] = mean;
      sc->m2[warp] = m2;
      if (warp == 0) sc->n = rows;
    }
  }

  // 6. the last chunk of the segment merges the moments (Chan et al. pairwise
  //    update, fp64, fixed order) into mean and 1 / (std + 1e-6)
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(&P.seg[seg].cnt, 1) == nchunks - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (warp < G) {
    double cn = 0.0, cmean = 0.0, cm2 = 0.0;
    for (int ci = lane; ci < nchunks; ci += 32) {
      const ScoreChunk* sc = P.schunk + (size_t)seg * P.cs_max + ci;
      const double bn = (double)__ldcg(&sc->n);
      const double bmean = (double)__ldcg(&sc->mean[warp]);
      const double bm2 = (double)__ldcg(&sc->m2[warp]);
      const double tn = cn + bn;
      const double dlt = bmean - cmean;
      cmean += dlt * bn / tn;
      cm2 += bm2 + dlt * dlt * cn * bn / tn;
      cn = tn;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const double bn = __shfl_xor_sync(0xffffffffu, cn, o);
      const double bmean = __shfl_xor_sync(0xffffffffu, cmean, o);
      const double bm2 = __shfl_xor_sync(0xffffffffu, cm2, o);
      const double tn = cn + bn;
      if (tn > 0.0) {
        const double dlt = bmean - cmean;
        const double nmean = cmean + dlt * bn / tn;
        const double nm2 = cm2 + bm2 + dlt * dlt * cn * bn / tn;
        cmean = nmean;
        cm2 = nm2;
      }
      cn = tn;
    }
    if (lane == 0) {
      const double sd = sqrt(cm2 / cn);
      P.seg[seg].mu[warp] = (float)cmean;
      P.seg[seg].inv[warp] = (float)(1.0 / (sd + (double)kZEps));
    }
  }
  if (threadIdx.x == 0) P.seg[seg].cnt = 0;
}

// z-max score per live row: s = max_h (raw_h - mu_h) * inv_h
template <int G>
__global__ void __launch_bounds__(kThreads) k_zscore(const __grid_constant__ Pass P) {
  const int seg = blockIdx.y;
  const SegView sv = seg_view(P, seg);
  if (!sv.valid || (P.only_active && !sv.active)) return;
  float mu[G], inv[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    mu[h] = P.seg[seg].mu[h];
    inv[h] = P.seg[seg].inv[h];
  }
  const int r_end = min(sv.n, (int)(blockIdx.x + 1) * 1024);
  for (int r = blockIdx.x * 1024 + threadIdx.x; r < r_end; r += blockDim.x) {
    const float* rp = P.raw + (size_t)(sv.row0 + r) * G;
    float s = (rp[0] - mu[0]) * inv[0];
#pragma unroll
    for (int h = 1; h < G; ++h) s = fmaxf(s, (rp[h] - mu[h]) * inv[h]);
    P.score[sv.row0 + r] = s;
  }
}

size_t score_smem_bytes(const Pass& P) {
  return (size_t)score_smem_layout(P.cs_rows, P.k_rb, P.G, P.fc).total;
}

namespace {

template <int KT, int G, int TPR, int PPT>
cudaError_t launch_score_t(const Pass& P, cudaStream_t st) {
  const size_t smem = score_smem_bytes(P);
  auto kern = k_score<KT, G, TPR, PPT>;
  // the largest dynamic shared memory any layout of this instantiation needs;
  // set once per process (the attribute is per function, not per call)
  static const cudaError_t attr =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
  if (attr != cudaSuccess) return attr;
  if (smem > 200 * 1024) return cudaErrorInvalidValue;
  dim3 grid(P.cs_max, P.n_seg);
  kern<<<grid, kThreads, smem, st>>>(P);
  return cudaGetLastError();
}

template <int KT, int G>
cudaError_t launch_score_g(const Pass& P, cudaStream_t st) {
  constexpr int PPT = G >= 8 ? 4 : 8;
  int tpr = 1;
  while (tpr * PPT < P.fc) tpr <<= 1;
  if constexpr (PPT == 8) {
    switch (tpr) {
      case 2: return launch_score_t<KT, G, 2, PPT>(P, st);
      case 4: return launch_score_t<KT, G, 4, PPT>(P, st);
      case 8: return launch_score_t<KT, G, 8, PPT>(P, st);
      case 16: return launch_score_t<KT, G, 16, PPT>(P, st);
    }
  } else {
    switch (tpr) {
      case 4: return launch_score_t<KT, G, 4, PPT>(P, st);
      case 8: return launch_score_t<KT, G, 8, PPT>(P, st);
      case 16: return launch_score_t<KT, G, 16, PPT>(P, st);
      case 32: return launch_score_t<KT, G, 32, PPT>(P, st);
    }
  }
  return cudaErrorInvalidValue;
}

template <int KT>
cudaError_t launch_score_k(const Pass& P, cudaStream_t st) {
  switch (P.G) {
    case 1: return launch_score_g<KT, 1>(P, st);
    case 2: return launch_score_g<KT, 2>(P, st);
    case 4: return launch_score_g<KT, 4>(P, st);
    case 8: return launch_score_g<KT, 8>(P, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_score(const Pass& P, cudaStream_t st) {
  switch (P.k_type) {
    case TRIA_F32: return launch_score_k<TRIA_F32>(P, st);
    case TRIA_F16: return launch_score_k<TRIA_F16>(P, st);
    case TRIA_Q8_0: return launch_score_k<TRIA_Q8_0>(P, st);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_zscore(const Pass& P, cudaStream_t st) {
  const int cap_max_blocks = (P.c_max * kChunk + 1023) / 1024;
  dim3 grid(cap_max_blocks, P.n_seg);
  switch (P.G) {
    case 1: k_zscore<1><<<grid, kThreads, 0, st>>>(P); break;
    case 2: k_zscore<2><<<grid, kThreads, 0, st>>>(P); break;
    case 4: k_zscore<4><<<grid, kThreads, 0, st>>>(P); break;
    case 8: k_zscore<8><<<grid, kThreads, 0, st>>>(P); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace tria
