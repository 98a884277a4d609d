// Compaction stage: in-place, order-preserving repack of the kept rows.
//
// [Doc] "TriAttention KV-Cache Eviction (--triattention)", §5 Phase B step 4
// (compact the KV cache in place, no padding gaps); [Worklog] "TriAttention
// Native C++ Worklog", "K-cache repack correctness is also no longer the
// leading suspect" and "Later correction ..." (the post-compaction K and V are
// exact gathers of the pre-compaction rows at the kept indices) and "6. Keep
// GPU work on GPU" (one gather kernel instead of thousands of small copies).
//
// Kept row i of a segment moves to row i, and i <= keep[i], so data only moves
// towards lower rows. The CTA that owns source chunk c (64 rows) moves its kept
// rows to the contiguous destination range [prefix[c], prefix[c+1]). Those
// destination rows can belong only to chunks <= c. The CTA therefore
//   1. copies its moving rows (all planes) into shared memory,
//   2. publishes "chunk c read" (flag = epoch + 1, release),
//   3. waits (bounded) for the flags of the lower chunks whose rows it will
//      overwrite - at most two, since 64 destination rows span at most two
//      64-row source chunks - and
//   4. writes the rows out.
// CTAs take tickets in the order they start, and chunk c only waits on chunks
// with smaller tickets, which are already running or done: no deadlock. Each
// byte moved is read once and written once.
#include "tria_internal.cuh"

namespace tria {

struct MoveSmem {
  int k, ks, v, vs, pos, src, total;
};

__host__ __device__ inline MoveSmem move_smem_layout(int k_rb, int ks_rb, int v_rb, int vs_rb) {
  MoveSmem L;
  int off = 0;
  auto take = [&](int bytes) {
    int at = off;
    off = (off + bytes + 15) & ~15;
    return at;
  };
  L.k = take(kChunk * k_rb);
  L.ks = take(kChunk * ks_rb);
  L.v = take(kChunk * v_rb);
  L.vs = take(kChunk * vs_rb);
  L.pos = take(kChunk * 4);
  L.src = take(kChunk * 4);
  L.total = off;
  return L;
}

// Copy `rows` rows of `rb` bytes from scattered source rows into packed shared
// memory (gather) or from packed shared memory to consecutive rows (scatter),
// with the widest unit that divides the row size.
template <bool kGather>
__device__ __forceinline__ void copy_rows(uint8_t* plane, int64_t row0, int rb, uint8_t* stage,
                                          const int* src_rows, int dst_row, int rows) {
  if (rb == 0 || rows == 0) return;
  if ((rb & 15) == 0) {
    const int per = rb >> 4;
    const int units = rows * per;
    for (int u = threadIdx.x; u < units; u += blockDim.x) {
      const int j = u / per, w = u - j * per;
      uint4* sp = reinterpret_cast<uint4*>(stage + (size_t)j * rb) + w;
      if (kGather) {
        const uint4* gp = reinterpret_cast<const uint4*>(plane + (size_t)(row0 + src_rows[j]) * rb) + w;
        *sp = __ldcg(gp);
      } else {
        uint4* gp = reinterpret_cast<uint4*>(plane + (size_t)(row0 + dst_row + j) * rb) + w;
        *gp = *sp;
      }
    }
  } else if ((rb & 3) == 0) {
    const int per = rb >> 2;
    const int units = rows * per;
    for (int u = threadIdx.x; u < units; u += blockDim.x) {
      const int j = u / per, w = u - j * per;
      uint32_t* sp = reinterpret_cast<uint32_t*>(stage + (size_t)j * rb) + w;
      if (kGather) {
        const uint32_t* gp = reinterpret_cast<const uint32_t*>(plane + (size_t)(row0 + src_rows[j]) * rb) + w;
        *sp = __ldcg(gp);
      } else {
        uint32_t* gp = reinterpret_cast<uint32_t*>(plane + (size_t)(row0 + dst_row + j) * rb) + w;
        *gp = *sp;
      }
    }
  } else {
    const int per = rb >> 1;
    const int units = rows * per;
    for (int u = threadIdx.x; u < units; u += blockDim.x) {
      const int j = u / per, w = u - j * per;
      uint16_t* sp = reinterpret_cast<uint16_t*>(stage + (size_t)j * rb) + w;
      if (kGather) {
        const uint16_t* gp = reinterpret_cast<const uint16_t*>(plane + (size_t)(row0 + src_rows[j]) * rb) + w;
        *sp = __ldcg(gp);
      } else {
        uint16_t* gp = reinterpret_cast<uint16_t*>(plane + (size_t)(row0 + dst_row + j) * rb) + w;
        *gp = *sp;
      }
    }
  }
}

__global__ void __launch_bounds__(kThreads) k_move(const __grid_constant__ Pass P) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint32_t s_ticket, s_epoch, s_bad;
  __shared__ int s_first, s_timeout;
  if (threadIdx.x == 0) {
    s_ticket = atomicAdd(&P.ctrl->move_ticket, 1u);
    s_epoch = ld_acquire_u32(&P.ctrl->epoch);
    s_bad = ld_acquire_u32(&P.ctrl->bad_keep);
    s_first = kChunk;
    s_timeout = 0;
  }
  __syncthreads();
  const int seg = (int)(s_ticket / (uint32_t)P.c_max);
  const int c = (int)(s_ticket % (uint32_t)P.c_max);
  bool work = seg < P.n_seg && s_bad == 0;
  SegView sv;
  if (work) {
    sv = seg_view(P, seg);
    work = sv.active && c * kChunk < sv.n;
  }
  if (work) {
    const MoveSmem L = move_smem_layout(P.k_rb, P.ks_rb, P.v_rb, P.vs_rb);
    int* ssrc = reinterpret_cast<int*>(smem + L.src);
    const int* pre = P.prefix + (size_t)seg * (P.c_max + 1);
    const int i0 = __ldcg(&pre[c]), i1 = __ldcg(&pre[c + 1]);
    const int nk = i1 - i0;
    // a chunk keeps at most its 64 rows, inside [0, B)
    const bool sane = i0 >= 0 && nk >= 0 && nk <= kChunk && i1 <= min(sv.B, sv.n);
    if (!sane && threadIdx.x == 0) {
      s_timeout = 1;
      report(P.ctrl, TRIA_ERR_INVALID_ARG, 0x10000000u | (uint32_t)seg);
    }
    // kept rows of this chunk and the first one that changes row
    for (int j = threadIdx.x; sane && j < nk; j += blockDim.x) {
      const int src = __ldcg(&P.keep[sv.row0 + i0 + j]);
      ssrc[j] = src;
      if (src < c * kChunk || src >= min(sv.n, (c + 1) * kChunk)) {
        s_timeout = 1;
        report(P.ctrl, TRIA_ERR_INVALID_ARG, 0x08000000u | (uint32_t)seg);
      }
      if (src != i0 + j) atomicMin(&s_first, j);
    }
    __syncthreads();
    if (s_timeout) {
      // inconsistent kept-row list: move nothing for this chunk, but still
      // publish the flag so that no other chunk waits on it
      if (threadIdx.x == 0) st_release_u32(&P.flags[(size_t)seg * P.c_max + c], s_epoch + 1u);
      goto done;
    }
    {
    const int first = min(s_first, nk);
    const int nmove = nk - first;
    const int dst0 = i0 + first;
    const int* msrc = ssrc + first;
    copy_rows<true>(P.k, sv.row0, P.k_rb, smem + L.k, msrc, 0, nmove);
    copy_rows<true>(P.ks, sv.row0, P.ks_rb, smem + L.ks, msrc, 0, nmove);
    copy_rows<true>(P.v, sv.row0, P.v_rb, smem + L.v, msrc, 0, nmove);
    copy_rows<true>(P.vs, sv.row0, P.vs_rb, smem + L.vs, msrc, 0, nmove);
    copy_rows<true>(reinterpret_cast<uint8_t*>(P.pos), sv.row0, 4, smem + L.pos, msrc, 0, nmove);
    __syncthreads();
    uint32_t* flags = P.flags + (size_t)seg * P.c_max;
    if (threadIdx.x == 0) {
      __threadfence();
      st_release_u32(&flags[c], s_epoch + 1u);
      if (nmove > 0) {
        const int lo = dst0 / kChunk, hi = min((i1 - 1) / kChunk, c - 1);
        for (int cc = lo; cc <= hi; ++cc)
          if (!wait_flag_bounded(&flags[cc], s_epoch + 1u, P.spin_limit)) {
            s_timeout = 1;
            report(P.ctrl, TRIA_ERR_TIMEOUT, (uint32_t)seg);
            break;
          }
      }
    }
    __syncthreads();
    if (!s_timeout && nmove > 0) {
      copy_rows<false>(P.k, sv.row0, P.k_rb, smem + L.k, nullptr, dst0, nmove);
      copy_rows<false>(P.ks, sv.row0, P.ks_rb, smem + L.ks, nullptr, dst0, nmove);
      copy_rows<false>(P.v, sv.row0, P.v_rb, smem + L.v, nullptr, dst0, nmove);
      copy_rows<false>(P.vs, sv.row0, P.vs_rb, smem + L.vs, nullptr, dst0, nmove);
      copy_rows<false>(reinterpret_cast<uint8_t*>(P.pos), sv.row0, 4, smem + L.pos, nullptr, dst0, nmove);
    }
    }
  }
done:
  // the last CTA to finish sets n_live and resets the call's counters
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const uint32_t done = atomicAdd(&P.ctrl->move_done, 1u);
    if (done == gridDim.x - 1) {
      __threadfence();
      if (s_bad == 0) {
        for (int s = 0; s < P.n_seqs; ++s) {
          const int n = *((volatile int32_t*)(P.n_live + s));
          if (n >= 0 && n <= P.seq[s].cap && n > P.seq[s].budget) P.n_live[s] = P.seq[s].budget;
        }
      }
      P.ctrl->move_ticket = 0u;
      P.ctrl->move_done = 0u;
      P.ctrl->bad_keep = 0u;
      __threadfence();
      atomicAdd(&P.ctrl->epoch, 1u);
    }
  }
}

// Caller-given keep lists: check them and derive the kept-row prefix of every
// 64-row source chunk (the entries of chunk c are keep[prefix[c] .. prefix[c+1])).
__global__ void __launch_bounds__(kThreads) k_keep_prepass(const __grid_constant__ Pass P) {
  const int seg = blockIdx.y;
  const SegView sv = seg_view(P, seg);
  if (!sv.valid) {
    if (blockIdx.x == 0 && threadIdx.x == 0) report(P.ctrl, TRIA_ERR_DEVICE_ARG, (uint32_t)sv.s);
    return;
  }
  if (!sv.active) return;
  const int n = sv.n, B = sv.B;
  const int nch = (n + kChunk - 1) / kChunk;
  int* pre = P.prefix + (size_t)seg * (P.c_max + 1);
  const int32_t* keep = P.keep + sv.row0;
  if (B == 0) {
    if (blockIdx.x == 0)
      for (int cc = threadIdx.x; cc <= nch; cc += blockDim.x) pre[cc] = 0;
    return;
  }
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= B) return;
  const int v = keep[i];
  const int prev = i > 0 ? keep[i - 1] : -1;
  if (v < 0 || v >= n || v <= prev) {
    atomicAdd(&P.ctrl->bad_keep, 1u);
    report(P.ctrl, TRIA_ERR_KEEP_LIST, (uint32_t)seg);
    return;
  }
  const int cp = prev < 0 ? -1 : prev / kChunk;
  const int cv = v / kChunk;
  for (int cc = cp + 1; cc <= cv; ++cc) pre[cc] = i;
  if (i == B - 1)
    for (int cc = cv + 1; cc <= nch; ++cc) pre[cc] = B;
}

__global__ void k_wait_selftest(const __grid_constant__ Pass P) {
  if (threadIdx.x == 0 && blockIdx.x == 0) {
    if (!wait_flag_bounded(&P.ctrl->wait_flag, 1u, P.spin_limit)) report(P.ctrl, TRIA_ERR_TIMEOUT, 0u);
  }
}

cudaError_t launch_keep_prepass(const Pass& P, cudaStream_t st) {
  const int cap_rows = P.c_max * kChunk;
  dim3 grid((cap_rows + kThreads - 1) / kThreads, P.n_seg);
  k_keep_prepass<<<grid, kThreads, 0, st>>>(P);
  return cudaGetLastError();
}

cudaError_t launch_move(const Pass& P, cudaStream_t st) {
  const MoveSmem L = move_smem_layout(P.k_rb, P.ks_rb, P.v_rb, P.vs_rb);
  static const cudaError_t attr =
      cudaFuncSetAttribute(k_move, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
  if (attr != cudaSuccess) return attr;
  if (L.total > 200 * 1024) return cudaErrorInvalidValue;
  const int grid = P.n_seg * P.c_max;
  k_move<<<grid, kThreads, L.total, st>>>(P);
  return cudaGetLastError();
}

cudaError_t launch_wait_selftest(const Pass& P, cudaStream_t st) {
  k_wait_selftest<<<1, 32, 0, st>>>(P);
  return cudaGetLastError();
}

}  // namespace tria
