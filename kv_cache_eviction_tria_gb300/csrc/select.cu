// Select stage: keep the budget's best rows of each segment.
//
// [Doc] "TriAttention KV-Cache Eviction (--triattention)", §1 CLI flags
// (--tri-budget, --tri-window, --tri-sink) and §5 Phase B steps 2-3 (protect
// the first sink and last window tokens, sort the rest by score, evict the
// lowest down to the budget); §5 Phase C (z-normalise per query head, then max
// over the GQA group) for the score this stage starts from on the evict path.
//
// Exact top-k by radix select on an order-preserving 32-bit key of the score:
//   pass 0: histogram of key bits [31:21] over the candidates
//   pass 1: bits [20:10] of the candidates whose bits [31:21] match
//   pass 2: bits [9:0]  of those whose bits [31:10] match
// After each pass the last CTA of the segment to finish (an atomic counter,
// no spinning) locates the bin holding the k-th largest key, so that T = the
// k-th largest key and kr = how many rows with key == T are kept. The count
// pass then finds the row of the kr-th tie (lowest row indices win ties) and
// the number of kept rows before every chunk; the keep-list pass writes the
// kept row indices in ascending order.
//
// All passes run in one cooperative kernel (every CTA resident), separated by
// bounded grid barriers; work items of a pass are (segment, row block) pairs
// dealt round-robin to the CTAs.
#include <cooperative_groups.h>

#include "tria_internal.cuh"

namespace cg = cooperative_groups;

namespace tria {

namespace {

__device__ __forceinline__ SelChunk load_chunk(const SelChunk* p) {
  const int4 v = __ldcg(reinterpret_cast<const int4*>(p));
  SelChunk c;
  c.n_gt = v.x;
  c.n_tie = v.y;
  c.n_prot = v.z;
  c.pad = v.w;
  return c;
}

struct SelShared {
  uint32_t h[kHistBins];
  int sbuf[40];
  int last, cstar, need, tie_row;
};

// One row block of one radix pass. PASS 0 on the evict path (G > 0) first
// turns the raw scores into the z-max score and stores it.
template <int PASS, int G>
__device__ void hist_block(const Pass& P, int seg, int blk, const SegView& sv, SelShared& sh) {
  constexpr int NB = PASS == 2 ? 1024 : 2048;
  constexpr int PER = NB / kThreads;
  const int n = sv.n;
  const int nblk = (n + kHistRowsPerCta - 1) / kHistRowsPerCta;
  for (int i = threadIdx.x; i < NB; i += blockDim.x) sh.h[i] = 0;
  float mu[G > 0 ? G : 1], inv[G > 0 ? G : 1];
  if constexpr (PASS == 0 && G > 0) block_segment_moments<G>(P, seg, mu, inv);
  __syncthreads();

  const uint32_t prefix = PASS > 0 ? __ldcg(&P.seg[seg].prefix) : 0u;
  const int r_beg = blk * kHistRowsPerCta, r_end = min(n, r_beg + kHistRowsPerCta);
  const int lo = sv.sink, hi = n - P.window;
  const bool do_hist = sv.k > 0;
  for (int r = r_beg + threadIdx.x; r < r_end; r += blockDim.x) {
    float s;
    if constexpr (PASS == 0 && G > 0) {
      const float* rp = P.raw + (size_t)(sv.row0 + r) * G;
      s = (rp[0] - mu[0]) * inv[0];
#pragma unroll
      for (int h = 1; h < G; ++h) s = fmaxf(s, (rp[h] - mu[h]) * inv[h]);
      P.score[sv.row0 + r] = s;
    } else {
      if (!do_hist || r < lo || r >= hi) continue;
      s = __ldcg(&P.score_in[sv.row0 + r]);
    }
    if (!do_hist || r < lo || r >= hi) continue;
    const uint32_t key = score_key(s);
    if (PASS == 0) {
      atomicAdd(&sh.h[key >> 21], 1u);
    } else if (PASS == 1) {
      if ((key >> 21) == prefix) atomicAdd(&sh.h[(key >> 10) & 0x7FFu], 1u);
    } else {
      if ((key >> 10) == prefix) atomicAdd(&sh.h[key & 0x3FFu], 1u);
    }
  }
  __syncthreads();
  if (!do_hist) return;
  uint32_t* gh = P.hist + (size_t)seg * kHistBins;
  for (int i = threadIdx.x; i < NB; i += blockDim.x)
    if (sh.h[i]) atomicAdd(&gh[i], sh.h[i]);
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) sh.last = (atomicAdd(&P.seg[seg].cnt, 1) == nblk - 1);
  __syncthreads();
  if (!sh.last) return;
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
  const int before = block_exclusive_scan(local, &total, sh.sbuf);
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

// One block of kCountChunksPerCta chunks: candidates above T, ties at T,
// protected rows. The last block of the segment places the tie cut and writes
// the kept-row prefix of every chunk.
__device__ void count_block(const Pass& P, int seg, int blk, const SegView& sv, SelShared& sh) {
  const int n = sv.n;
  const int nch = (n + kChunk - 1) / kChunk;
  const int nblk = (nch + kCountChunksPerCta - 1) / kCountChunksPerCta;
  const bool none = sv.k <= 0;
  const uint32_t T = none ? 0xFFFFFFFFu : __ldcg(&P.seg[seg].T);
  const float* s = P.score_in + sv.row0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  SelChunk* ch = P.chunk + (size_t)seg * P.c_max;

  for (int cc = 0; cc < kCountChunksPerCta / 8; ++cc) {
    const int c = blk * kCountChunksPerCta + warp * (kCountChunksPerCta / 8) + cc;
    if (c >= nch) break;
    int gt = 0, tie = 0, prot = 0;
#pragma unroll
    for (int half = 0; half < kChunk / 32; ++half) {
      const int r = c * kChunk + half * 32 + lane;
      const bool in = r < n;
      const bool pr = in && is_protected(r, n, sv.sink, P.window);
      const bool cand = in && !pr && !none;
      const uint32_t key = cand ? score_key(__ldcg(&s[r])) : 0u;
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
  if (threadIdx.x == 0) sh.last = (atomicAdd(&P.seg[seg].cnt, 1) == nblk - 1);
  __syncthreads();
  if (!sh.last) return;
  __threadfence();

  // 1. the chunk holding the kr-th tie (kr ties at T are kept, lowest rows first)
  const int kr = none ? 0 : __ldcg(&P.seg[seg].kr);
  const int per = (nch + kThreads - 1) / kThreads;
  const int cbeg = min(nch, (int)threadIdx.x * per), cend = min(nch, cbeg + per);
  int local = 0;
  for (int c = cbeg; c < cend; ++c) local += __ldcg(&ch[c].n_tie);
  int total;
  const int before = block_exclusive_scan(local, &total, sh.sbuf);
  if (threadIdx.x == 0) {
    sh.cstar = -1;
    sh.need = 0;
    sh.tie_row = -1;
  }
  __syncthreads();
  if (kr > 0 && before < kr && kr <= before + local) {
    int cum = before;
    for (int c = cbeg; c < cend; ++c) {
      const int t = __ldcg(&ch[c].n_tie);
      if (cum + t >= kr) {
        sh.cstar = c;
        sh.need = kr - cum;
        break;
      }
      cum += t;
    }
  }
  __syncthreads();
  const int cstar = sh.cstar, need = sh.need;
  // 2. the row of that tie
  if (cstar >= 0 && warp == 0) {
    int seen = 0;
    for (int half = 0; half < kChunk / 32; ++half) {
      const int r = cstar * kChunk + half * 32 + lane;
      const bool in = r < n;
      const bool cand = in && !is_protected(r, n, sv.sink, P.window);
      const bool t = cand && score_key(__ldcg(&s[r])) == T;
      const uint32_t b = __ballot_sync(0xffffffffu, t);
      const int cnt = __popc(b);
      if (seen + cnt >= need) {
        const int want = need - seen;
        const int rank = __popc(b & ((1u << lane) - 1u));
        if (t && rank == want - 1) sh.tie_row = r;
        break;
      }
      seen += cnt;
    }
  }
  if (kr > 0 && threadIdx.x == 0 && total < kr) report(P.ctrl, TRIA_ERR_INVALID_ARG, 0x40000000u | (uint32_t)seg);
  __syncthreads();

  // 3. kept rows per chunk -> exclusive prefix
  int keep_local = 0;
  for (int c = cbeg; c < cend; ++c) {
    const SelChunk v = load_chunk(&ch[c]);
    keep_local += v.n_prot + v.n_gt + (c < cstar ? v.n_tie : (c == cstar ? need : 0));
  }
  int keep_total;
  const int kbefore = block_exclusive_scan(keep_local, &keep_total, sh.sbuf);
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
    P.seg[seg].tie_row = sh.tie_row;
    P.seg[seg].cnt = 0;
  }
}

// Kept row indices of one block of chunks, ascending, at keep[seg_row0 + i];
// segments at or below budget get the identity list.
__device__ void keeplist_block(const Pass& P, int seg, int blk, const SegView& sv) {
  const int n = sv.n;
  int32_t* keep = P.keep + sv.row0;
  const int r_beg = blk * kCountChunksPerCta * kChunk;
  if (!sv.active) {
    const int r_end = min(n, r_beg + kCountChunksPerCta * kChunk);
    for (int r = r_beg + threadIdx.x; r < r_end; r += blockDim.x) keep[r] = r;
    return;
  }
  const int nch = (n + kChunk - 1) / kChunk;
  const bool none = sv.k <= 0;
  const uint32_t T = none ? 0xFFFFFFFFu : __ldcg(&P.seg[seg].T);
  const int tie_row = none ? -1 : __ldcg(&P.seg[seg].tie_row);
  const float* s = P.score_in + sv.row0;
  const int* pre = P.prefix + (size_t)seg * (P.c_max + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int cc = 0; cc < kCountChunksPerCta / 8; ++cc) {
    const int c = blk * kCountChunksPerCta + warp * (kCountChunksPerCta / 8) + cc;
    if (c >= nch) break;
    int base = __ldcg(&pre[c]);
#pragma unroll
    for (int half = 0; half < kChunk / 32; ++half) {
      const int r = c * kChunk + half * 32 + lane;
      const bool in = r < n;
      const bool pr = in && is_protected(r, n, sv.sink, P.window);
      bool kp = pr;
      if (in && !pr && !none) {
        const uint32_t key = score_key(__ldcg(&s[r]));
        kp = key > T || (key == T && r <= tie_row);
      }
      const uint32_t b = __ballot_sync(0xffffffffu, kp);
      if (kp) keep[base + __popc(b & ((1u << lane) - 1u))] = r;
      base += __popc(b);
    }
  }
}

// The whole select stage (and, with G > 0, the z-max score) in one
// cooperative launch.
template <int G>
__global__ void __launch_bounds__(kThreads) k_select(const __grid_constant__ Pass P, int write_keep) {
  __shared__ SelShared sh;
  const int hist_blocks = (P.c_max * kChunk + kHistRowsPerCta - 1) / kHistRowsPerCta;
  const int hist_items = P.n_seg * hist_blocks;
  const int count_blocks = (P.c_max + kCountChunksPerCta - 1) / kCountChunksPerCta;
  const int count_items = P.n_seg * count_blocks;

  // pass 0 (+ z-max score): every active segment
  for (int it = blockIdx.x; it < hist_items; it += gridDim.x) {
    const int seg = it / hist_blocks, blk = it - seg * hist_blocks;
    const SegView sv = seg_view(P, seg);
    if (!sv.valid) {
      if (blk == 0 && threadIdx.x == 0) report(P.ctrl, TRIA_ERR_DEVICE_ARG, (uint32_t)sv.s);
      continue;
    }
    if (!sv.active || blk * kHistRowsPerCta >= sv.n) continue;
    hist_block<0, G>(P, seg, blk, sv, sh);
  }
  grid_barrier(P);
  for (int it = blockIdx.x; it < hist_items; it += gridDim.x) {
    const int seg = it / hist_blocks, blk = it - seg * hist_blocks;
    const SegView sv = seg_view(P, seg);
    if (!sv.active || sv.k <= 0 || blk * kHistRowsPerCta >= sv.n) continue;
    hist_block<1, 0>(P, seg, blk, sv, sh);
  }
  grid_barrier(P);
  for (int it = blockIdx.x; it < hist_items; it += gridDim.x) {
    const int seg = it / hist_blocks, blk = it - seg * hist_blocks;
    const SegView sv = seg_view(P, seg);
    if (!sv.active || sv.k <= 0 || blk * kHistRowsPerCta >= sv.n) continue;
    hist_block<2, 0>(P, seg, blk, sv, sh);
  }
  grid_barrier(P);
  for (int it = blockIdx.x; it < count_items; it += gridDim.x) {
    const int seg = it / count_blocks, blk = it - seg * count_blocks;
    const SegView sv = seg_view(P, seg);
    if (!sv.active || blk * kCountChunksPerCta * kChunk >= sv.n) continue;
    count_block(P, seg, blk, sv, sh);
  }
  if (!write_keep) return;
  grid_barrier(P);
  for (int it = blockIdx.x; it < count_items; it += gridDim.x) {
    const int seg = it / count_blocks, blk = it - seg * count_blocks;
    const SegView sv = seg_view(P, seg);
    if (!sv.valid || blk * kCountChunksPerCta * kChunk >= sv.n) continue;
    if (!sv.active && P.only_active) continue;
    keeplist_block(P, seg, blk, sv);
  }
}

// ---------------------------------------------------------------------------
// Cluster path: one thread-block cluster of kClusterCtas CTAs per segment. CTA
// `rank` owns the contiguous, chunk-aligned row range [rank*RPC, rank*RPC+RPC)
// and keeps the 32-bit keys of its rows in shared memory for all passes.
// Radix histograms: each CTA counts its keys locally, then adds each non-zero
// bin into the cluster total held by the bin's owner (rank = bin / (bins / 8),
// remote atomic adds through distributed shared memory; score keys fall in
// few bins, so the adds are few); after one cluster barrier every CTA reads
// the eight owners' slices (one vector per thread) and finds the cut's bin by
// itself. Tie counts and kept counts are read from the other ranks.
// ---------------------------------------------------------------------------

constexpr int kClusterCtas = 8;
constexpr int kClThreads = 512;
constexpr int kClMaxRowsPerCta = 32768;   // 128 KiB of keys

struct ClShared {
  alignas(16) uint32_t h[kHistBins];        // this CTA's histogram of the current pass
  // cluster totals of the bins this CTA owns, one buffer per pass (never reused)
  alignas(16) uint32_t own[3][kHistBins / kClusterCtas];
  int sbuf[40];
  int info[4];                  // prefix, kr, keys in the cut's bin after the current pass
  int cnt[2];                   // ties, strict keeps (gt + protected) of this CTA
  int warp_tie[kClThreads / 32], warp_keep[kClThreads / 32];
};

// the G raw scores of one row (vector loads; rows are G consecutive floats,
// so 16-byte aligned for G = 4 and 8)
template <int G>
__device__ __forceinline__ void load_raw_row(const float* rp, float* x) {
  if constexpr (G % 4 == 0) {
#pragma unroll
    for (int h = 0; h < G; h += 4) {
      const float4 v = __ldcg(reinterpret_cast<const float4*>(rp + h));
      x[h] = v.x;
      x[h + 1] = v.y;
      x[h + 2] = v.z;
      x[h + 3] = v.w;
    }
  } else if constexpr (G == 2) {
    const float2 v = __ldcg(reinterpret_cast<const float2*>(rp));
    x[0] = v.x;
    x[1] = v.y;
  } else {
#pragma unroll
    for (int h = 0; h < G; ++h) x[h] = __ldcg(rp + h);
  }
}

// Split cluster barrier (all threads of every CTA): arrive with release
// semantics, wait with acquire semantics.
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

template <int G>
__global__ void __launch_bounds__(kClThreads) k_select_cl(const __grid_constant__ Pass P, int write_keep) {
  extern __shared__ __align__(16) uint32_t keys[];
  __shared__ ClShared sh;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int seg = blockIdx.y;
  const SegView sv = seg_view(P, seg);
  if (!sv.valid) {
    if (rank == 0 && threadIdx.x == 0) report(P.ctrl, TRIA_ERR_DEVICE_ARG, (uint32_t)sv.s);
    return;   // the whole cluster leaves (same segment)
  }
  const int n = sv.n;
  const int rpc = (((n + kClusterCtas - 1) / kClusterCtas) + kChunk - 1) / kChunk * kChunk;
  const int r0 = min(n, rank * rpc), r1 = min(n, r0 + rpc);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int32_t* keep = P.keep + sv.row0;
  if (!sv.active) {
    if (write_keep && !P.only_active)
      for (int r = r0 + threadIdx.x; r < r1; r += blockDim.x) keep[r] = r;
    return;
  }
  const int lo = sv.sink, hi = n - P.window;
  const bool none = sv.k <= 0;
  // the owned totals start at zero; every rank must have cleared its own
  // before any rank adds into them (the barrier completes before the first
  // pass, its latency hidden behind the keys)
  for (int i = threadIdx.x; i < 3 * (kHistBins / kClusterCtas); i += blockDim.x) (&sh.own[0][0])[i] = 0u;
  __syncwarp();
  cluster_arrive_release();

  // keys of my rows (the evict path turns raw scores into the z-max score
  // here); loads are batched U rows per thread so that they are in flight
  // together, and the first batch is loaded before the segment's moments are
  // merged so that the two latencies overlap
  {
    constexpr int GG = G > 0 ? G : 1;
    constexpr int U = G > 4 ? 4 : 8;
    float x[U][GG];
    auto load_batch = [&](int base) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int r = base + u * kClThreads;
        if (r < r1) {
          if constexpr (G > 0) load_raw_row<G>(P.raw + (size_t)(sv.row0 + r) * G, x[u]);
          else x[u][0] = __ldcg(&P.score_in[sv.row0 + r]);
        }
      }
    };
    float mu[GG], inv[GG];
    load_batch(r0 + threadIdx.x);
    // segment moments: every CTA of the cluster sums all of the segment's
    // score runs itself (shifted sums, one coalesced load round), so no
    // cluster exchange is needed
    if constexpr (G > 0) block_segment_moments<G>(P, seg, mu, inv);
    for (int base = r0 + threadIdx.x; base < r1; base += U * kClThreads) {
      if (base != r0 + (int)threadIdx.x) load_batch(base);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int r = base + u * kClThreads;
        if (r < r1) {
          float s = x[u][0];
          if constexpr (G > 0) {
            s = (x[u][0] - mu[0]) * inv[0];
#pragma unroll
            for (int h = 1; h < G; ++h) s = fmaxf(s, (x[u][h] - mu[h]) * inv[h]);
            P.score[sv.row0 + r] = s;   // the evict path's z-max, kept in the workspace
          }
          keys[r - r0] = score_key(s);
        }
      }
    }
  }

  // up to three radix passes over the candidates [lo, hi). When the bin that
  // holds the cut contains exactly the keys still to take, every key with
  // that prefix is kept: the cut is "key >= prefix * 2^shift" and the later
  // passes are skipped (all CTAs of the cluster see the same totals).
  uint32_t prefix = 0, T = 0xFFFFFFFFu;
  int kr = sv.k;
  bool cut_at_prefix = false;
  __syncthreads();
  cluster_wait_acquire();
  if (!none) {
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
      const int NB = pass == 2 ? 1024 : 2048;
      const int SL = NB / kClusterCtas;   // bins per owner
      uint32_t* hb = sh.h;
      uint32_t* own = sh.own[pass];
      for (int i = threadIdx.x; i < NB; i += blockDim.x) hb[i] = 0;
      __syncthreads();
      for (int r = max(r0, lo) + threadIdx.x; r < min(r1, hi); r += blockDim.x) {
        const uint32_t key = keys[r - r0];
        if (pass == 0) atomicAdd(&hb[key >> 21], 1u);
        else if (pass == 1) { if ((key >> 21) == prefix) atomicAdd(&hb[(key >> 10) & 0x7FFu], 1u); }
        else if ((key >> 10) == prefix) atomicAdd(&hb[key & 0x3FFu], 1u);
      }
      __syncthreads();
      // my non-zero bins into their owners' totals
      for (int b = threadIdx.x; b < NB; b += blockDim.x) {
        const uint32_t c = hb[b];
        if (c != 0u) {
          const int q = b / SL;
          atomicAdd(cluster.map_shared_rank(own, q) + (b - q * SL), c);
        }
      }
      cluster.sync();
      // the bin of the kr-th largest key: thread t reads bins
      // NB-1-per*t-j, j = 0..per-1 (descending), one vector from their owner
      const int per = NB / kClThreads;   // 4 or 2 bins per thread, scanned from the top
      uint32_t tot[4] = {0u, 0u, 0u, 0u};
      int local = 0;
      {
        const int b0 = NB - per * ((int)threadIdx.x + 1);   // lowest of my bins
        const int q = b0 / SL;
        const uint32_t* src = cluster.map_shared_rank(own, q) + (b0 - q * SL);
        if (per == 4) {
          const uint4 v = *reinterpret_cast<const uint4*>(src);
          tot[0] = v.w;
          tot[1] = v.z;
          tot[2] = v.y;
          tot[3] = v.x;
        } else {
          const uint2 v = *reinterpret_cast<const uint2*>(src);
          tot[0] = v.y;
          tot[1] = v.x;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) local += (int)tot[j];
      }
      int total;
      const int before = block_exclusive_scan(local, &total, sh.sbuf);
      if (before < kr && kr <= before + local) {
        int cum = before;
        bool found = false;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (found || j >= per) continue;
          const int b = NB - 1 - (per * threadIdx.x + j);
          if (cum + (int)tot[j] >= kr) {
            sh.info[0] = (int)(pass == 0 ? (uint32_t)b : pass == 1 ? ((prefix << 11) | (uint32_t)b)
                                                                     : ((prefix << 10) | (uint32_t)b));
            sh.info[1] = kr - cum;
            sh.info[2] = (int)tot[j];   // keys of the cluster in that bin
            found = true;
            continue;
          }
          cum += (int)tot[j];
        }
      }
      if (threadIdx.x == 0 && total < kr && rank == 0)
        report(P.ctrl, TRIA_ERR_INVALID_ARG, 0x80000000u | (uint32_t)seg);
      __syncthreads();
      prefix = (uint32_t)sh.info[0];
      kr = sh.info[1];
      if (pass < 2 && kr == sh.info[2]) {
        const uint32_t lo_key = prefix << (pass == 0 ? 21 : 10);
        if (lo_key != 0u) {
          T = lo_key - 1u;   // keep key > T, no ties taken
          kr = 0;
          cut_at_prefix = true;
          break;
        }
      }
    }
    if (!cut_at_prefix) T = prefix;
  }

  // counts of my rows; ties at T are kept lowest rows first across the cluster
  const int nch_mine = (r1 - r0 + kChunk - 1) / kChunk;
  const int cpw = (nch_mine + (kClThreads / 32) - 1) / (kClThreads / 32);   // chunks per warp
  int w_tie = 0, w_keep = 0;
  for (int ci = warp * cpw; ci < min(nch_mine, (warp + 1) * cpw); ++ci) {
    const int r = r0 + ci * kChunk + lane;
    const bool in = r < r1;
    const bool pr = in && is_protected(r, n, lo, P.window);
    const bool cand = in && !pr && !none;
    const uint32_t key = in ? keys[r - r0] : 0u;
    w_tie += __popc(__ballot_sync(0xffffffffu, cand && key == T));
    w_keep += __popc(__ballot_sync(0xffffffffu, pr || (cand && key > T)));
  }
  if (lane == 0) {
    sh.warp_tie[warp] = w_tie;
    sh.warp_keep[warp] = w_keep;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int a = 0, b = 0;
    for (int w = 0; w < kClThreads / 32; ++w) {
      a += sh.warp_tie[w];
      b += sh.warp_keep[w];
    }
    sh.cnt[0] = a;
    sh.cnt[1] = b;
  }
  cluster.sync();
  // ties and kept rows of the lower ranks
  __shared__ int s_off[3];
  if (threadIdx.x == 0) {
    int tie_before = 0, keep_before = 0;
    for (int q = 0; q < rank; ++q) {
      const int* c = cluster.map_shared_rank(sh.cnt, q);
      const int tq = c[0];
      const int kept_ties = max(0, min(tq, kr - tie_before));
      keep_before += c[1] + kept_ties;
      tie_before += tq;
    }
    s_off[0] = keep_before;
    s_off[1] = max(0, min(sh.cnt[0], kr - tie_before));   // my ties that are kept
    s_off[2] = 0;
  }
  __syncthreads();
  const int keep_base = s_off[0], my_ties = s_off[1];
  // per-warp offsets (ties and kept rows of the lower warps of this CTA)
  int tie_off = 0, keep_off = 0;
  for (int w = 0; w < warp; ++w) {
    const int tw = sh.warp_tie[w];
    tie_off += tw;
  }
  {
    // kept rows of lower warps = strict keeps + their kept ties
    int t_run = 0;
    for (int w = 0; w < warp; ++w) {
      const int tw = sh.warp_tie[w];
      keep_off += sh.warp_keep[w] + max(0, min(tw, my_ties - t_run));
      t_run += tw;
    }
  }
  int* pre = P.prefix + (size_t)seg * (P.c_max + 1);
  const int chunk0 = r0 / kChunk;
  int tie_run = tie_off, keep_run = keep_base + keep_off;
  for (int ci = warp * cpw; ci < min(nch_mine, (warp + 1) * cpw); ++ci) {
    const int r = r0 + ci * kChunk + lane;
    const bool in = r < r1;
    const bool pr = in && is_protected(r, n, lo, P.window);
    const bool cand = in && !pr && !none;
    const uint32_t key = in ? keys[r - r0] : 0u;
    const bool is_tie = cand && key == T;
    const uint32_t bt = __ballot_sync(0xffffffffu, is_tie);
    const int trank = tie_run + __popc(bt & ((1u << lane) - 1u));
    const bool kp = pr || (cand && key > T) || (is_tie && trank < my_ties);
    const uint32_t bk = __ballot_sync(0xffffffffu, kp);
    if (lane == 0) pre[chunk0 + ci] = keep_run;
    if (write_keep && kp) keep[keep_run + __popc(bk & ((1u << lane) - 1u))] = r;
    tie_run += __popc(bt);
    keep_run += __popc(bk);
  }
  if (rank == 0 && threadIdx.x == 0) {
    pre[(n + kChunk - 1) / kChunk] = sv.B;
    if (sv.B > n) report(P.ctrl, TRIA_ERR_INVALID_ARG, 0x20000000u | (uint32_t)seg);
  }
  cluster.sync();   // no CTA leaves while another may still read its shared memory
}

template <int G>
cudaError_t launch_select_cl(const Pass& P, bool write_keep, cudaStream_t st, int cap_max) {
  const int rpc_max = (((cap_max + kClusterCtas - 1) / kClusterCtas) + kChunk - 1) / kChunk * kChunk;
  const size_t smem = (size_t)rpc_max * 4;
  static const cudaError_t attr =
      set_smem_attrs(k_select_cl<G>, kClMaxRowsPerCta * 4);
  if (attr != cudaSuccess) return attr;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kClusterCtas, P.n_seg, 1);
  cfg.blockDim = dim3(kClThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = kClusterCtas;
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_select_cl<G>, P, write_keep ? 1 : 0);
}

template <int G>
cudaError_t launch_select_g(const Pass& P, bool write_keep, cudaStream_t st) {
  static int per_sm = -1;
  if (per_sm < 0) {
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_select<G>, kThreads, 0);
    if (e != cudaSuccess) {
      per_sm = -1;
      return e;
    }
  }
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int hist_blocks = (P.c_max * kChunk + kHistRowsPerCta - 1) / kHistRowsPerCta;
  const int count_blocks = (P.c_max + kCountChunksPerCta - 1) / kCountChunksPerCta;
  const int items = P.n_seg * (hist_blocks > count_blocks ? hist_blocks : count_blocks);
  int grid = sms * (per_sm < 2 ? per_sm : 2);
  if (grid > items) grid = items;
  if (grid < 1) grid = 1;
  int wk = write_keep ? 1 : 0;
  void* args[] = {const_cast<Pass*>(&P), &wk};
  return cudaLaunchCooperativeKernel((const void*)k_select<G>, dim3(grid), dim3(kThreads), args, 0, st);
}

}  // namespace

cudaError_t launch_select(const Pass& P, bool write_keep, cudaStream_t st, int score_group) {
  // segments up to kClusterCtas * kClMaxRowsPerCta rows: one cluster per
  // segment; longer ones: the cooperative grid path
  const int cap_max = P.c_max * kChunk;
  if (cap_max <= kClusterCtas * kClMaxRowsPerCta) {
    switch (score_group) {
      case 0: return launch_select_cl<0>(P, write_keep, st, cap_max);
      case 1: return launch_select_cl<1>(P, write_keep, st, cap_max);
      case 2: return launch_select_cl<2>(P, write_keep, st, cap_max);
      case 4: return launch_select_cl<4>(P, write_keep, st, cap_max);
      case 8: return launch_select_cl<8>(P, write_keep, st, cap_max);
    }
    return cudaErrorInvalidValue;
  }
  switch (score_group) {
    case 0: return launch_select_g<0>(P, write_keep, st);
    case 1: return launch_select_g<1>(P, write_keep, st);
    case 2: return launch_select_g<2>(P, write_keep, st);
    case 4: return launch_select_g<4>(P, write_keep, st);
    case 8: return launch_select_g<8>(P, write_keep, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace tria
