// Select stage: keep the budget's best rows of each segment.
//
// [Doc] "TriAttention KV-Cache Eviction (--triattention)", §1 CLI flags
// (--tri-budget, --tri-window, --tri-sink) and §5 Phase B steps 2-3 (protect
// the first sink and last window tokens, sort the rest by score, evict the
// lowest down to the budget).
//
// Exact top-k by radix select on an order-preserving 32-bit key of the score:
//   pass 0: histogram of key bits [31:21] over the candidates
//   pass 1: bits [20:10] of the candidates whose bits [31:21] match
//   pass 2: bits [9:0]  of those whose bits [31:10] match
// After each pass the last CTA of the segment to finish (an atomic counter,
// no spinning) locates the bin holding the k-th largest key, so that T = the
// k-th largest key and kr = how many rows with key == T are kept. The count
// pass then finds the row of the kr-th tie (lowest row indices win ties) and
// the number of kept rows before every 64-row chunk; the keep-list pass writes
// the kept row indices in ascending order.
#include "tria_internal.cuh"

namespace tria {

__device__ __forceinline__ SelChunk load_chunk(const SelChunk* p) {
  const int4 v = __ldcg(reinterpret_cast<const int4*>(p));
  SelChunk c;
  c.n_gt = v.x;
  c.n_tie = v.y;
  c.n_prot = v.z;
  c.pad = v.w;
  return c;
}

__device__ __forceinline__ const float* score_base(const Pass& P, const SegView& sv) {
  return P.score_in + sv.row0;
}

template <int PASS>
__global__ void __launch_bounds__(kThreads) k_hist(const __grid_constant__ Pass P) {
  constexpr int NB = PASS == 2 ? 1024 : 2048;
  constexpr int PER = NB / kThreads;
  const int seg = blockIdx.y;
  const SegView sv = seg_view(P, seg);
  if (!sv.active || sv.k <= 0) return;
  const int n = sv.n;
  const int nblk = (n + kHistRowsPerCta - 1) / kHistRowsPerCta;
  if ((int)blockIdx.x >= nblk) return;

  __shared__ uint32_t h[NB];
  __shared__ int sbuf[40];
  __shared__ int s_last;
  for (int i = threadIdx.x; i < NB; i += blockDim.x) h[i] = 0;
  __syncthreads();

  const uint32_t prefix = PASS > 0 ? __ldcg(&P.seg[seg].prefix) : 0u;
  const int lo = max(P.sink, (int)blockIdx.x * kHistRowsPerCta);
  const int hi = min(n - P.window, ((int)blockIdx.x + 1) * kHistRowsPerCta);
  const float* s = score_base(P, sv);
  for (int r = lo + threadIdx.x; r < hi; r += blockDim.x) {
    const uint32_t key = score_key(s[r]);
    if (PASS == 0) {
      atomicAdd(&h[key >> 21], 1u);
    } else if (PASS == 1) {
      if ((key >> 21) == prefix) atomicAdd(&h[(key >> 10) & 0x7FFu], 1u);
    } else {
      if ((key >> 10) == prefix) atomicAdd(&h[key & 0x3FFu], 1u);
    }
  }
  __syncthreads();
  uint32_t* gh = P.hist + (size_t)seg * kHistBins;
  for (int i = threadIdx.x; i < NB; i += blockDim.x)
    if (h[i]) atomicAdd(&gh[i], h[i]);
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(&P.seg[seg].cnt, 1) == nblk - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // bins scanned from the top: thread t owns bins NB-1-(PER*t) .. NB-PER*(t+1)
  const int kr = PASS == 0 ? sv.k : __ldcg(&P.seg[seg].kr);
  uint32_t cnt[PER];
  int local = 0;
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    cnt[j] = __ldcg(&gh[NB - 1 - (PER * threadIdx.x + j)]);
    local += (int)cnt[j];
  }
  int total;
  const int before = block_exclusive_scan(local, &total, sbuf);
  if (before < kr && kr <= before + local) {
    int cum = before;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const int b = NB - 1 - (PER * threadIdx.x + j);
      if (cum + (int)cnt[j] >= kr) {
        const uint32_t np = PASS == 0 ? (uint32_t)b : PASS == 1 ? ((prefix << 11) | (uint32_t)b)
                                                                : ((prefix << 10) | (uint32_t)b);
        P.seg[seg].prefix = np;
        P.seg[seg].kr = kr - cum;
        if (PASS == 2) P.seg[seg].T = np;
        break;
      }
      cum += (int)cnt[j];
    }
  }
  if (threadIdx.x == 0 && total < kr) report(P.ctrl, TRIA_ERR_INVALID_ARG, 0x80000000u | (uint32_t)seg);
  __syncthreads();
  for (int i = threadIdx.x; i < NB; i += blockDim.x) gh[i] = 0u;
  if (threadIdx.x == 0) P.seg[seg].cnt = 0;
}

// Per chunk: candidates above T, ties at T, protected rows. The last CTA
// of the segment places the tie cut and writes the kept-row prefix per chunk.
__global__ void __launch_bounds__(kThreads) k_count(const __grid_constant__ Pass P) {
  const int seg = blockIdx.y;
  const SegView sv = seg_view(P, seg);
  if (!sv.active) return;
  const int n = sv.n;
  const int nch = (n + kChunk - 1) / kChunk;
  const int nblk = (nch + kCountChunksPerCta - 1) / kCountChunksPerCta;
  if ((int)blockIdx.x >= nblk) return;
  const bool none = sv.k <= 0;
  const uint32_t T = none ? 0xFFFFFFFFu : __ldcg(&P.seg[seg].T);
  const float* s = score_base(P, sv);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  SelChunk* ch = P.chunk + (size_t)seg * P.c_max;

  __shared__ int sbuf[40];
  __shared__ int s_last, s_cstar, s_need, s_tie_row;

  for (int cc = 0; cc < kCountChunksPerCta / 8; ++cc) {
    const int c = blockIdx.x * kCountChunksPerCta + warp * (kCountChunksPerCta / 8) + cc;
    if (c >= nch) break;
    int gt = 0, tie = 0, prot = 0;
#pragma unroll
    for (int half = 0; half < kChunk / 32; ++half) {
      const int r = c * kChunk + half * 32 + lane;
      const bool in = r < n;
      const bool pr = in && is_protected(r, n, P.sink, P.window);
      const bool cand = in && !pr && !none;
      const uint32_t key = cand ? score_key(s[r]) : 0u;
      gt += __popc(__ballot_sync(0xffffffffu, cand && key > T));
      tie += __popc(__ballot_sync(0xffffffffu, cand && key == T));
      prot += __popc(__ballot_sync(0xffffffffu, pr));
    }
    if (lane == 0) {
      SelChunk v;
      v.n_gt = gt;
      v.n_tie = tie;
      v.n_prot = prot;
      v.pad = 0;
      ch[c] = v;
    }
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(&P.seg[seg].cnt, 1) == nblk - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // 1. the chunk holding the kr-th tie (kr ties at T are kept, lowest rows first)
  const int kr = none ? 0 : __ldcg(&P.seg[seg].kr);
  const int per = (nch + kThreads - 1) / kThreads;
  const int cbeg = min(nch, (int)threadIdx.x * per), cend = min(nch, cbeg + per);
  int local = 0;
  for (int c = cbeg; c < cend; ++c) local += __ldcg(&ch[c].n_tie);
  int total;
  int before = block_exclusive_scan(local, &total, sbuf);
  if (threadIdx.x == 0) {
    s_cstar = -1;
    s_need = 0;
    s_tie_row = -1;
  }
  __syncthreads();
  if (kr > 0 && before < kr && kr <= before + local) {
    int cum = before;
    for (int c = cbeg; c < cend; ++c) {
      const int t = __ldcg(&ch[c].n_tie);
      if (cum + t >= kr) {
        s_cstar = c;
        s_need = kr - cum;
        break;
      }
      cum += t;
    }
  }
  __syncthreads();
  const int cstar = s_cstar, need = s_need;
  // 2. the row of that tie
  if (cstar >= 0 && warp == 0) {
    int seen = 0;
    for (int half = 0; half < kChunk / 32; ++half) {
      const int r = cstar * kChunk + half * 32 + lane;
      const bool in = r < n;
      const bool cand = in && !is_protected(r, n, P.sink, P.window);
      const bool t = cand && score_key(s[r]) == T;
      const uint32_t b = __ballot_sync(0xffffffffu, t);
      const int cnt = __popc(b);
      if (seen + cnt >= need) {
        // the (need - seen)-th set bit of b
        int want = need - seen;
        const int rank = __popc(b & ((1u << lane) - 1u));
        if (t && rank == want - 1) s_tie_row = r;
        break;
      }
      seen += cnt;
    }
  }
  if (kr > 0 && threadIdx.x == 0 && total < kr)
    report(P.ctrl, TRIA_ERR_INVALID_ARG, 0x40000000u | (uint32_t)seg);
  __syncthreads();

  // 3. kept rows per chunk -> exclusive prefix
  int keep_local = 0;
  for (int c = cbeg; c < cend; ++c) {
    const SelChunk v = load_chunk(&ch[c]);
    keep_local += v.n_prot + v.n_gt + (c < cstar ? v.n_tie : (c == cstar ? need : 0));
  }
  int keep_total;
  const int kbefore = block_exclusive_scan(keep_local, &keep_total, sbuf);
  int* pre = P.prefix + (size_t)seg * (P.c_max + 1);
  int cum = kbefore;
  for (int c = cbeg; c < cend; ++c) {
    pre[c] = cum;
    const SelChunk v = load_chunk(&ch[c]);
    cum += v.n_prot + v.n_gt + (c < cstar ? v.n_tie : (c == cstar ? need : 0));
  }
  if (threadIdx.x == 0) {
    pre[nch] = keep_total;
    if (keep_total != sv.B) report(P.ctrl, TRIA_ERR_INVALID_ARG, 0x20000000u | (uint32_t)seg);
    P.seg[seg].tie_row = s_tie_row;
    P.seg[seg].cnt = 0;
  }
}

// Kept row indices of every segment, ascending, at keep[seg_row0 + i].
__global__ void __launch_bounds__(kThreads) k_keeplist(const __grid_constant__ Pass P) {
  const int seg = blockIdx.y;
  const SegView sv = seg_view(P, seg);
  if (!sv.valid) return;
  const int n = sv.n;
  int32_t* keep = P.keep + sv.row0;
  const int r_beg = blockIdx.x * kCountChunksPerCta * kChunk;
  if (!sv.active) {
    if (P.only_active) return;
    const int r_end = min(n, r_beg + kCountChunksPerCta * kChunk);
    for (int r = r_beg + threadIdx.x; r < r_end; r += blockDim.x) keep[r] = r;
    return;
  }
  const int nch = (n + kChunk - 1) / kChunk;
  const bool none = sv.k <= 0;
  const uint32_t T = none ? 0xFFFFFFFFu : __ldcg(&P.seg[seg].T);
  const int tie_row = none ? -1 : __ldcg(&P.seg[seg].tie_row);
  const float* s = score_base(P, sv);
  const int* pre = P.prefix + (size_t)seg * (P.c_max + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int cc = 0; cc < kCountChunksPerCta / 8; ++cc) {
    const int c = blockIdx.x * kCountChunksPerCta + warp * (kCountChunksPerCta / 8) + cc;
    if (c >= nch) break;
    int base = __ldcg(&pre[c]);
#pragma unroll
    for (int half = 0; half < kChunk / 32; ++half) {
      const int r = c * kChunk + half * 32 + lane;
      const bool in = r < n;
      const bool pr = in && is_protected(r, n, P.sink, P.window);
      bool kp = pr;
      if (in && !pr && !none) {
        const uint32_t key = score_key(s[r]);
        kp = key > T || (key == T && r <= tie_row);
      }
      const uint32_t b = __ballot_sync(0xffffffffu, kp);
      if (kp) keep[base + __popc(b & ((1u << lane) - 1u))] = r;
      base += __popc(b);
    }
  }
}

cudaError_t launch_select(const Pass& P, bool write_keep, cudaStream_t st) {
  const int cap_rows = P.c_max * kChunk;
  dim3 gh((cap_rows + kHistRowsPerCta - 1) / kHistRowsPerCta, P.n_seg);
  k_hist<0><<<gh, kThreads, 0, st>>>(P);
  k_hist<1><<<gh, kThreads, 0, st>>>(P);
  k_hist<2><<<gh, kThreads, 0, st>>>(P);
  dim3 gc((P.c_max + kCountChunksPerCta - 1) / kCountChunksPerCta, P.n_seg);
  k_count<<<gc, kThreads, 0, st>>>(P);
  if (write_keep) k_keeplist<<<gc, kThreads, 0, st>>>(P);
  return cudaGetLastError();
}

}  // namespace tria
