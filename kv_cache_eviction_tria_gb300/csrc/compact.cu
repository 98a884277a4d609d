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
// towards lower rows. Work is split by 32-row DESTINATION block: block j
// gathers rows keep[32j .. 32j+32) and writes them to rows [32j, 32j+32), so
// every block but a segment's last moves a full stage. Block j overwrites
// source rows [32j, 32j+32), which are read by the blocks that own keep
// entries [prefix[j], prefix[j+1]) (prefix[c] = kept rows before source chunk
// c) - blocks <= j, at most two of them lower than j. So block j
//   1. copies its moving rows (all planes) into its own shared-memory stage,
//   2. publishes "block j read" (flag = the call's tag, see flag_tag),
//   3. waits (bounded) for the flags of those lower blocks, and
//   4. writes the stage out.
// Warps take blocks in increasing order and every warp of the cooperative
// grid is resident, so the lowest unpublished block can always proceed: no
// deadlock. Each byte moved is read once and written once.
#include "move.cuh"

namespace tria {

// One work item: destination block j of segment sg, with this lane's keep
// entry and the keep-index range [p0, p1) that reads the block's source rows.
struct MoveItem {
  int t, sg, j, a, p0, p1, n;
  bool valid;   // block j exists in segment sg (an active segment with j < its block count)
};

// Persistent compaction, one destination block per warp at a time. Item t is
// block t / n_seg of segment t % n_seg (block-major; items past a segment's
// block count are empty); warp w of the grid takes items w, w + W, w + 2W, ...
// in order and loads the next item's keep entries while it moves the current
// one. For its block a warp
//   1. gathers the moving rows of every plane into its own shared-memory
//      stage with cp.async and waits for them,
//   2. publishes "block read" (flag = the call's tag; the reads are complete, so
//      no fence is needed before the flag),
//   3. waits (bounded) for the lower blocks that read its destination rows,
//   4. writes the stage out to the contiguous destination rows (TMA bulk
//      stores for key and value rows).
__global__ void k_move(const __grid_constant__ Pass P) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint32_t s_epoch, s_bad;
  __shared__ int s_nbmax;
  // moving source rows of each warp's block; once gathered, their positions
  __shared__ int s_src[kMoveMaxWarps][kChunk];
  const MoveStage L = move_stage_layout(P.k_rb, P.ks_rb, P.v_rb, P.vs_rb);
  if (threadIdx.x == 0) {
    s_epoch = ld_acquire_u32(&P.ctrl->epoch);
    s_bad = ld_acquire_u32(&P.ctrl->bad_keep);
  }
  // destination blocks of the active segments; items are enumerated
  // block-major (block j of every segment before block j + 1 of any), so a
  // block's readers - blocks near j * B / n of the same segment - come in
  // earlier rounds of the grid, not beside it
  auto blocks_of = [&](int sg) {   // destination blocks of a segment (0: inactive)
    const SegView v = seg_view(P, sg);
    return v.active ? (v.B + kChunk - 1) / kChunk : 0;
  };
  if (threadIdx.x == 0) s_nbmax = 0;
  __syncthreads();
  for (int sg = threadIdx.x; sg < P.n_seg; sg += blockDim.x) atomicMax(&s_nbmax, blocks_of(sg));
  __syncthreads();
  const uint32_t tag = flag_tag(s_epoch);
  const int total = P.n_seg * s_nbmax;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps_cta = blockDim.x >> 5;
  const int W = gridDim.x * nwarps_cta;
  uint8_t* stg = smem + (size_t)warp * L.bytes;
  int* msrc = s_src[warp];
  const PlaneMap mk = plane_map(P.k_rb, lane), mks = plane_map(P.ks_rb, lane), mv = plane_map(P.v_rb, lane),
                 mvs = plane_map(P.vs_rb, lane);

  auto row0_of = [&](int sg) {
    const int sq = sg / P.n_kv;
    return P.seq[sq].row0 + (int64_t)(sg - sq * P.n_kv) * P.seq[sq].cap;
  };
  auto fetch = [&](int t, MoveItem& m) {
    m.t = t;
    m.valid = false;
    if (t >= total) return;
    m.sg = t % P.n_seg;
    m.j = t / P.n_seg;
    if (m.j >= blocks_of(m.sg)) return;
    m.valid = true;
    const int B = P.seq[m.sg / P.n_kv].budget;
    const int i = m.j * kChunk + lane;
    m.a = i < B ? __ldcg(&P.keep[row0_of(m.sg) + i]) : -1;
    const int* pre = P.prefix + (size_t)m.sg * (P.c_max + 1);
    m.p0 = __ldcg(&pre[m.j]);
    m.p1 = __ldcg(&pre[m.j + 1]);
    m.n = *((volatile const int32_t*)(P.n_live + m.sg / P.n_kv));
  };

  // the key / value rows and positions of a staged block to its contiguous
  // destination rows: one TMA bulk store per plane of the key and value rows
  // (off the L1 path the gathers use), the small planes with plain stores
  auto write_out = [&](int64_t row0, int dst0, int nmove) {
    if (lane == 0) {
      fence_proxy_async_smem();
      bulk_s2g(P.k + (size_t)(row0 + dst0) * P.k_rb, stg + L.k, (uint32_t)(nmove * P.k_rb));
      bulk_s2g(P.v + (size_t)(row0 + dst0) * P.v_rb, stg + L.v, (uint32_t)(nmove * P.v_rb));
      bulk_commit();
    }
    warp_scatter(P.ks, row0, P.ks_rb, stg + L.ks, dst0, nmove, lane);
    warp_scatter(P.vs, row0, P.vs_rb, stg + L.vs, dst0, nmove, lane);
    if (lane < nmove) P.pos[row0 + dst0 + lane] = msrc[lane];
  };
  // When every block has a warp of its own (one round), all blocks gather,
  // one grid barrier marks every read done, and all write: the per-block
  // read flags would be polled while the gathers still load the memory
  // system, which makes each poll slow. Otherwise blocks publish read flags
  // and wait only for their readers.
  const bool one_round = total <= W;
  bool pend = false;   // one round: a staged block waits for the barrier
  int64_t pend_row0 = 0;
  int pend_dst0 = 0, pend_n = 0;

  if (s_bad == 0) {
    MoveItem m;
    fetch(blockIdx.x * nwarps_cta + warp, m);
    while (m.t < total) {
      if (!m.valid) {   // no such block in this segment
        MoveItem nx;
        fetch(m.t + W, nx);
        m = nx;
        continue;
      }
      const int sg = m.sg, j = m.j;
      const int sq = sg / P.n_kv;
      const int64_t row0 = row0_of(sg);
      const int B = P.seq[sq].budget;
      const int n = m.n;
      const int i0 = j * kChunk, cnt = min(kChunk, B - i0);
      // every entry reads a row at or above its destination, inside the
      // segment; the readers of this block's rows are at most 32 entries
      // ending at or before the budget
      const bool bad_entry = lane < cnt && (m.a < i0 + lane || m.a >= n);
      const bool ok = !__any_sync(0xffffffffu, bad_entry) && m.p0 >= 0 && m.p0 <= m.p1 &&
                      m.p1 - m.p0 <= kChunk && m.p1 <= B;
      if (!ok && lane == 0) report(P.ctrl, TRIA_ERR_INVALID_ARG, 0x10000000u | (uint32_t)sg);
      // moving entries (keep[i] != i) are a suffix of the block
      const unsigned mvm = __ballot_sync(0xffffffffu, ok && lane < cnt && m.a != i0 + lane);
      const int first = mvm ? __ffs(mvm) - 1 : cnt;
      const int nmove = ok ? cnt - first : 0;
      if (lane >= first && lane < cnt) msrc[lane - first] = m.a;
      __syncwarp();
      MoveItem nx;
      fetch(m.t + W, nx);   // next item's keep entries load while this one moves
      // the previous item's bulk stores must have read the stage
      if (lane == 0) bulk_wait_read_all();
      __syncwarp();
      int my_pos = 0;
      if (nmove > 0) {
        warp_gather(P.k, row0, mk, stg + L.k, msrc, nmove);
        warp_gather(P.ks, row0, mks, stg + L.ks, msrc, nmove);
        warp_gather(P.v, row0, mv, stg + L.v, msrc, nmove);
        warp_gather(P.vs, row0, mvs, stg + L.vs, msrc, nmove);
        if (lane < nmove) my_pos = __ldcg(P.pos + row0 + msrc[lane]);
      }
      cp_async_commit();
      cp_async_wait<0>();
      __syncwarp();
      // the source table is no longer needed: it holds the positions from
      // here on (the shared store also completes the position load before
      // the block is published as read)
      if (lane < nmove) msrc[lane] = my_pos;
      __syncwarp();
      if (one_round) {   // the only item of this warp: write after the barrier
        pend = ok && nmove > 0;
        pend_row0 = row0;
        pend_dst0 = i0 + first;
        pend_n = nmove;
        break;
      }
      // publish "read"; then wait for the lower blocks that read my destination rows
      uint32_t* flags = P.flags + (size_t)sg * P.c_max;
      int go = 0;
      if (lane == 0) {
        st_relaxed_u32(&flags[j], tag);
        go = ok;
        if (go && nmove > 0 && m.p1 > m.p0) {
          const int lo = m.p0 / kChunk, hi = min((m.p1 - 1) / kChunk, j - 1);
          for (int cc = lo; cc <= hi; ++cc)
            if (!wait_flag_bounded(&flags[cc], tag, P.spin_limit)) {
              go = 0;
              report(P.ctrl, TRIA_ERR_TIMEOUT, (uint32_t)sg);
              break;
            }
        }
      }
      go = __shfl_sync(0xffffffffu, go, 0);
      if (go && nmove > 0) write_out(row0, i0 + first, nmove);
      __syncwarp();
      m = nx;
    }
  }
  if (one_round && s_bad == 0) {
    // every warp of the grid (with a block or not) reaches the barrier; after
    // it every staged block's sources have been read
    const bool in_time = grid_barrier(P);
    if (pend && in_time) write_out(pend_row0, pend_dst0, pend_n);
    __syncwarp();
  }

  if (lane == 0) bulk_wait_all();   // this warp's bulk stores are complete
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
// source chunk (the entries of chunk c are keep[prefix[c] .. prefix[c+1])).
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
  const MoveStage L = move_stage_layout(P.k_rb, P.ks_rb, P.v_rb, P.vs_rb);
  const int warps = move_warps(L);
  if (warps < 1) return cudaErrorInvalidValue;
  const int threads = warps * 32;
  const int smem = warps * L.bytes;
  static const cudaError_t attr =
      set_smem_attrs(k_move, kMoveSmemLimit);
  if (attr != cudaSuccess) return attr;
  int dev = 0, sms = 0, per_sm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_move, threads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  int grid = sms * per_sm;
  // at most ceil(min(budget, capacity) / 32) destination blocks per segment
  int64_t items = 0;
  for (int s = 0; s < P.n_seqs; ++s) {
    const int b = P.seq[s].budget < P.seq[s].cap ? P.seq[s].budget : P.seq[s].cap;
    items += (int64_t)P.n_kv * ((b + kChunk - 1) / kChunk);
  }
  const int64_t need = (items + warps - 1) / warps;
  if (grid > need) grid = (int)need;
  if (grid < 1) grid = 1;
  void* args[] = {const_cast<Pass*>(&P)};
  return cudaLaunchCooperativeKernel((const void*)k_move, dim3(grid), dim3(threads), args, (size_t)smem, st);
}

cudaError_t launch_wait_selftest(const Pass& P, cudaStream_t st) {
  k_wait_selftest<<<1, 32, 0, st>>>(P);
  return cudaGetLastError();
}

}  // namespace tria
