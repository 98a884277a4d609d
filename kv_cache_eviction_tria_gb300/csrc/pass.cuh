// Fused eviction pass: score, select and compact every segment of one or
// more layers in one persistent kernel.
//
// [Doc] "TriAttention KV-Cache Eviction (--triattention)", §5 Phase B (score
// every cached token, protect the first sink and last window tokens, keep the
// best down to the budget, compact the cache in place) and Phase C
// (z-normalise each query head over the segment, then max over the GQA
// group); [Worklog] "TriAttention Native C++ Worklog", Phase 9 (the score on
// the stored rotated keys) and the exact-gather checks of the compaction.
// The arithmetic of each step is that of the staged kernels (score_tc.cuh,
// the cluster select, k_move); what this kernel changes is the schedule.
//
// Schedule. A segment is (layer, sequence, KV head). One CTA per SM (a
// cooperative launch: every CTA is resident, so waits on other CTAs end).
//  * Score items: a segment's live rows are cut into items of 12 warps x ppw
//    pieces (a piece is at most 8 KB of keys; ppw from 1 to 8, larger for
//    larger passes). A CTA claims items two ahead (an atomic counter in
//    segment order); each warp streams its pieces
//    through a two-stage ring (bulk async copies completing on mbarriers) and
//    issues the first piece of the CTA's next item while it computes its last
//    piece of the current one, so the key stream does not stop between
//    items. At the end of an item the CTA merges its warps' moments into one
//    partial per item.
//  * Select: the CTA that completes a segment's last item (an atomic count,
//    read back one item later) selects that segment: segment moments from
//    the item partials,
//    z-max keys and the first radix histogram in one sweep, up to two more
//    radix passes over the keys, then the keep list and the kept-row prefix
//    of every 32-row chunk; it publishes the segment in the ready list. The
//    ring keeps loading the next item meanwhile (the select uses its own
//    shared memory).
//  * Moves: once the score items are all claimed, a CTA's warps claim 32-row
//    destination blocks of ready segments (in order, one counter per
//    segment) and move them as k_move does: gather the block's moving rows
//    into the warp's stage, publish "read", wait (bounded) for the lower
//    blocks that read its destination rows, store. The ready list and the
//    per-segment counters live at a fixed place of the workspace (PassCtl).
//  * The last CTA to finish sets n_live and resets the call's counters.
// Every wait is bounded (TRIA_ERR_TIMEOUT after the spin limit); a wait only
// ever waits for work that an earlier claim started, so the schedule cannot
// deadlock.
#pragma once

#include "move.cuh"
#include "score_tc.cuh"

namespace tria {

constexpr int kPassWarps = 12;
constexpr int kPassThreads = kPassWarps * 32;
constexpr int kPassPPWMax = 8;               // pieces per warp per score item (at most)
constexpr int kPassPieceBytes = 8192;
constexpr int kPassScaleStage = kPassPieceBytes / 16;   // q8_0 block scales of a piece
constexpr int kPassRing = kPassWarps * 2 * kPassPieceBytes;
constexpr int kPassMaxSegs = kPassCtlSegs;   // layers x sequences x KV heads per call
constexpr int kPassMaxLayers = 128;

// One layer of the call: its cache planes, live rows and statistics.
struct LayerRef {
  uint8_t* k;
  uint8_t* ks;
  uint8_t* v;
  uint8_t* vs;
  int32_t* pos;
  int32_t* n_live;      // [n_seqs], this layer's
  int64_t qe_off;       // this layer's statistics (elements from qe / mw)
  int64_t pad;
};

struct FPass {
  int32_t n_layers, n_seqs, n_kv, n_seg, G, hd, fc, window;
  int32_t k_rb, ks_rb, v_rb, vs_rb;
  int32_t spin_limit;
  int32_t item_rows;    // key rows per score item (kPassWarps x ppw x piece_rows)
  int32_t piece_rows;   // key rows per piece
  int32_t ppw;          // pieces per warp per score item
  int32_t cs_max;       // columns of a segment's item-partial table (>= items per segment)
  int32_t c_max;        // chunks per segment (max)
  int64_t rows_per_layer;   // workspace rows of one layer
  const float2* qe;
  const float* mw;
  const unsigned long long* turns;   // [fc] frac(w_f / 2pi) * 2^64 (shared by the call's layers)
  float* raw;                        // [layer rows][G]
  uint32_t* keys;                    // [layer rows] z-max keys
  float* score_out;                  // [layer rows] z-max scores, or null
  int32_t* keep;                     // [layer rows]
  Ctrl* ctrl;
  PassCtl* ctl;                      // ready list and per-segment counters
  float* parts;                      // [n_seg][kRunCols][cs_max] item moment partials
  int32_t* prefix;                   // [n_seg][c_max + 1]
  uint32_t* flags;                   // [n_seg][c_max]
  SeqInfo seq[kMaxSeqs];             // shared by the call's layers (qe_off unused)
  LayerRef lay[kPassMaxLayers];
};

struct PSeg {
  int li, s, g;
  int64_t row0;    // first row of the segment in the layer's planes
  int64_t wrow0;   // first row of the segment in the workspace row arrays
  int n, B, sink;
  bool valid, active;
};

__device__ __forceinline__ PSeg pass_seg(const FPass& P, int sg) {
  PSeg v;
  const int per_layer = P.n_seqs * P.n_kv;
  v.li = sg / per_layer;
  const int r = sg - v.li * per_layer;
  v.s = r / P.n_kv;
  v.g = r - v.s * P.n_kv;
  const SeqInfo& q = P.seq[v.s];
  v.row0 = q.row0 + (int64_t)v.g * q.cap;
  v.wrow0 = (int64_t)v.li * P.rows_per_layer + v.row0;
  v.n = *((volatile const int32_t*)(P.lay[v.li].n_live + v.s));
  v.B = q.budget;
  v.sink = q.sink;
  v.valid = v.n >= 0 && v.n <= q.cap;
  v.active = v.valid && v.n > v.B;
  return v;
}

// dynamic shared memory: ring (or move stages) | q8_0 scale ring | mbarriers |
// item table | turn factors | select histogram
struct PassSmem {
  static constexpr int kRing = 0;
  static constexpr int kScales = kRing + kPassRing;
  static constexpr int kBars = kScales + kPassWarps * 2 * kPassScaleStage;
  static constexpr int kItem0 = kBars + kPassWarps * 2 * 8;
  static constexpr int kTurns = kItem0 + ((kPassMaxSegs + 1) * 4 + 15) / 16 * 16;
  static constexpr int kHist = kTurns + 128 * 8;
  static constexpr int kBytes = kHist + kHistBins * 4;
};

template <int G>
__device__ __forceinline__ void load_raw_g(const float* rp, float* x) {
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
    x[0] = __ldcg(rp);
  }
}

// Selection of one segment by the whole CTA (see the file comment). Writes
// the keep list (B entries) and the kept-row prefix of every chunk.
template <int G>
__device__ __noinline__ void pass_select(const FPass& P, int sg, int n_items, uint32_t* hist) {
  __shared__ int s_info[4];
  __shared__ int s_sbuf[40];
  __shared__ int s_wt[kPassWarps], s_wk[kPassWarps];
  const PSeg v = pass_seg(P, sg);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = v.n, lo = v.sink, hi = n - P.window;
  const int k = v.B - v.sink - P.window;
  uint32_t* keys = P.keys + v.wrow0;

  float mu[G], inv[G];
  block_moments_of_runs<G>(P.parts + (size_t)sg * kRunCols * P.cs_max, P.cs_max, n_items, mu, inv);
  for (int i = tid; i < kHistBins; i += blockDim.x) hist[i] = 0u;
  __syncthreads();

  // z-max keys of every live row and the first radix histogram of the
  // candidates [lo, hi); loads of U rows per thread are in flight together
  {
    constexpr int U = G > 4 ? 4 : 8;
    const float* raw = P.raw + (size_t)v.wrow0 * G;
    float* so = P.score_out ? P.score_out + v.wrow0 : nullptr;
    for (int base = tid; base < n; base += U * kPassThreads) {
      float x[U][G];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int r = base + u * kPassThreads;
        if (r < n) load_raw_g<G>(raw + (size_t)r * G, x[u]);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int r = base + u * kPassThreads;
        if (r < n) {
          float s = (x[u][0] - mu[0]) * inv[0];
#pragma unroll
          for (int h = 1; h < G; ++h) s = fmaxf(s, (x[u][h] - mu[h]) * inv[h]);
          const uint32_t key = score_key(s);
          __stcg(keys + r, key);
          if (so) so[r] = s;
          if (k > 0 && r >= lo && r < hi) atomicAdd(&hist[key >> 21], 1u);
        }
      }
    }
  }
  __syncthreads();

  // radix select of the k-th largest key over the candidates: T = that key,
  // kr = how many candidates with key == T are kept (lowest rows first); a
  // bin holding exactly the keys still to take ends the search early
  uint32_t T = 0xFFFFFFFFu;
  int kr = 0;
  if (k > 0) {
    uint32_t prefix = 0;
    kr = k;
    bool cut = false;
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
      const int NB = pass == 2 ? 1024 : 2048;
      if (pass > 0) {
        for (int i = tid; i < NB; i += blockDim.x) hist[i] = 0u;
        __syncthreads();
        constexpr int UB = 8;   // key loads in flight per thread
        for (int base = lo + tid; base < hi; base += UB * kPassThreads) {
          uint32_t kk[UB];
#pragma unroll
          for (int u = 0; u < UB; ++u) {
            const int r = base + u * kPassThreads;
            kk[u] = r < hi ? __ldcg(keys + r) : 0u;
          }
#pragma unroll
          for (int u = 0; u < UB; ++u) {
            if (base + u * kPassThreads >= hi) break;
            const uint32_t key = kk[u];
            if (pass == 1) {
              if ((key >> 21) == prefix) atomicAdd(&hist[(key >> 10) & 0x7FFu], 1u);
            } else if ((key >> 10) == prefix) {
              atomicAdd(&hist[key & 0x3FFu], 1u);
            }
          }
        }
        __syncthreads();
      }
      // thread t scans bins NB-1-per*t .. NB-per*(t+1) (descending)
      const int per = (NB + kPassThreads - 1) / kPassThreads;
      uint32_t cnt[6];
      int local = 0;
#pragma unroll
      for (int j = 0; j < 6; ++j) {
        const int b = NB - 1 - (per * tid + j);
        cnt[j] = (j < per && b >= 0) ? hist[b] : 0u;
        local += (int)cnt[j];
      }
      int total;
      const int before = block_exclusive_scan(local, &total, s_sbuf);
      if (before < kr && kr <= before + local) {
        int cum = before;
#pragma unroll
        for (int j = 0; j < 6; ++j) {
          const int b = NB - 1 - (per * tid + j);
          if (j >= per || b < 0) break;
          if (cum + (int)cnt[j] >= kr) {
            s_info[0] = (int)(pass == 0 ? (uint32_t)b : pass == 1 ? ((prefix << 11) | (uint32_t)b)
                                                                   : ((prefix << 10) | (uint32_t)b));
            s_info[1] = kr - cum;
            s_info[2] = (int)cnt[j];
            break;
          }
          cum += (int)cnt[j];
        }
      }
      if (tid == 0 && total < kr) report(P.ctrl, TRIA_ERR_INVALID_ARG, 0x80000000u | (uint32_t)sg);
      __syncthreads();
      prefix = (uint32_t)s_info[0];
      kr = s_info[1];
      const int in_bin = s_info[2];
      __syncthreads();
      if (pass < 2 && kr == in_bin) {
        const uint32_t lo_key = prefix << (pass == 0 ? 21 : 10);
        if (lo_key != 0u) {
          T = lo_key - 1u;   // keep key > T, no ties taken
          kr = 0;
          cut = true;
          break;
        }
      }
    }
    if (!cut) T = prefix;
  }

  // keep list: warps take contiguous chunk ranges; sweep 1 counts each warp's
  // ties and strict keeps, sweep 2 writes the kept rows and chunk prefixes
  const int nch = (n + kChunk - 1) / kChunk;
  const int cpw = (nch + kPassWarps - 1) / kPassWarps;
  const int c0 = min(nch, warp * cpw), c1 = min(nch, c0 + cpw);
  constexpr int CB = 8;   // chunks whose keys load together
  {
    int wt = 0, wk = 0;
    for (int cb = c0; cb < c1; cb += CB) {
      uint32_t kk[CB];
#pragma unroll
      for (int u = 0; u < CB; ++u) {
        const int r = (cb + u) * kChunk + lane;
        kk[u] = (cb + u < c1 && r < n && r >= lo && r < hi && k > 0) ? __ldcg(keys + r) : 0u;
      }
#pragma unroll
      for (int u = 0; u < CB; ++u) {
        if (cb + u >= c1) break;
        const int r = (cb + u) * kChunk + lane;
        const bool in = r < n;
        const bool pr = in && (r < lo || r >= hi);
        const bool cand = in && !pr && k > 0;
        wt += __popc(__ballot_sync(0xffffffffu, cand && kk[u] == T));
        wk += __popc(__ballot_sync(0xffffffffu, pr || (cand && kk[u] > T)));
      }
    }
    if (lane == 0) {
      s_wt[warp] = wt;
      s_wk[warp] = wk;
    }
  }
  __syncthreads();
  int tie_run = 0, keep_run = 0;
  for (int w = 0; w < warp; ++w) {
    keep_run += s_wk[w] + max(0, min(s_wt[w], kr - tie_run));
    tie_run += s_wt[w];
  }
  int32_t* keep = P.keep + v.wrow0;
  int* pre = P.prefix + (size_t)sg * (P.c_max + 1);
  for (int cb = c0; cb < c1; cb += CB) {
    uint32_t kk[CB];
#pragma unroll
    for (int u = 0; u < CB; ++u) {
      const int r = (cb + u) * kChunk + lane;
      kk[u] = (cb + u < c1 && r < n && r >= lo && r < hi && k > 0) ? __ldcg(keys + r) : 0u;
    }
#pragma unroll
    for (int u = 0; u < CB; ++u) {
      const int ci = cb + u;
      if (ci >= c1) break;
      const int r = ci * kChunk + lane;
      const bool in = r < n;
      const bool pr = in && (r < lo || r >= hi);
      const bool cand = in && !pr && k > 0;
      const bool is_tie = cand && kk[u] == T;
      const uint32_t bt = __ballot_sync(0xffffffffu, is_tie);
      const int trank = tie_run + __popc(bt & ((1u << lane) - 1u));
      const bool kp = pr || (cand && kk[u] > T) || (is_tie && trank < kr);
      const uint32_t bk = __ballot_sync(0xffffffffu, kp);
      if (lane == 0) pre[ci] = keep_run;
      if (kp) keep[keep_run + __popc(bk & ((1u << lane) - 1u))] = r;
      tie_run += __popc(bt);
      keep_run += __popc(bk);
    }
  }
  if (warp == kPassWarps - 1 && lane == 0) {
    pre[nch] = v.B;
    if (keep_run != v.B) report(P.ctrl, TRIA_ERR_INVALID_ARG, 0x20000000u | (uint32_t)sg);
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    P.ctl->items_done[sg] = 0;
    const uint32_t slot = atomicAdd(&P.ctrl->ready_count, 1u);
    st_release_u32(reinterpret_cast<uint32_t*>(P.ctl->ready + slot), (uint32_t)(sg + 1));
  }
}

// One warp's share of the moves: claim 32-row destination blocks of ready
// segments (the next claim is issued while the current block's rows load)
// and move each as k_move does. Returns when every active segment's blocks
// are claimed (or a bounded wait gave up).
static __device__ __noinline__ void pass_moves(const FPass& P, uint8_t* stg, int* msrc, uint32_t tag, int n_active) {
  const int lane = threadIdx.x & 31;
  const MoveStage L = move_stage_layout(P.k_rb, P.ks_rb, P.v_rb, P.vs_rb);
  const PlaneMap mk = plane_map(P.k_rb, lane), mks = plane_map(P.ks_rb, lane), mv = plane_map(P.v_rb, lane),
                 mvs = plane_map(P.vs_rb, lane);
  // lane 0: 0 = block (sg, j), 1 = none ready yet, 2 = every block claimed
  auto claim = [&](int& sg, int& j) {
    int state = 1;
    sg = 0;
    j = 0;
    if (lane == 0) {
      while (true) {
        const uint32_t c = ld_acquire_u32(&P.ctrl->move_cursor);
        if ((int)c >= n_active) {
          state = 2;
          break;
        }
        const uint32_t e = ld_acquire_u32(reinterpret_cast<const uint32_t*>(P.ctl->ready + c));
        if (e == 0u) break;
        sg = (int)e - 1;
        if (sg >= P.n_seg) {   // cannot happen: the list holds this call's segments
          report(P.ctrl, TRIA_ERR_INVALID_ARG, 0x08000000u);
          state = 2;
          break;
        }
        const int nb = (P.seq[(sg % (P.n_seqs * P.n_kv)) / P.n_kv].budget + kChunk - 1) / kChunk;
        j = atomicAdd(&P.ctl->move_next[sg], 1);
        if (j >= 0 && j < nb) {
          state = 0;
          break;
        }
        atomicCAS(&P.ctrl->move_cursor, c, c + 1u);   // exhausted: move past it
      }
    }
    return state;
  };
  int nsg, nj;
  int nstate = claim(nsg, nj);
  int idle = 0;
  while (true) {
    const int state = __shfl_sync(0xffffffffu, nstate, 0);
    if (state == 2) break;
    if (state == 1) {
      if (++idle > P.spin_limit) {
        if (lane == 0) report(P.ctrl, TRIA_ERR_TIMEOUT, 0xA0000000u);
        break;
      }
      __nanosleep(idle < 64 ? 64 : 512);
      nstate = claim(nsg, nj);
      continue;
    }
    idle = 0;
    const int sg = __shfl_sync(0xffffffffu, nsg, 0);
    const int j = __shfl_sync(0xffffffffu, nj, 0);
    const PSeg v = pass_seg(P, sg);
    const LayerRef& lr = P.lay[v.li];
    const int B = v.B, n = v.n;
    const int i0 = j * kChunk, cnt = min(kChunk, B - i0);
    const int a = lane < cnt ? __ldcg(P.keep + v.wrow0 + i0 + lane) : -1;
    const int* pre = P.prefix + (size_t)sg * (P.c_max + 1);
    const int p0 = __ldcg(&pre[j]), p1 = __ldcg(&pre[j + 1]);
    const bool bad_entry = lane < cnt && (a < i0 + lane || a >= n);
    const bool ok = !__any_sync(0xffffffffu, bad_entry) && p0 >= 0 && p0 <= p1 && p1 - p0 <= kChunk && p1 <= B;
    if (!ok && lane == 0) report(P.ctrl, TRIA_ERR_INVALID_ARG, 0x10000000u | (uint32_t)sg);
    // moving entries (keep[i] != i) are a suffix of the block
    const unsigned mvm = __ballot_sync(0xffffffffu, ok && lane < cnt && a != i0 + lane);
    const int first = mvm ? __ffs(mvm) - 1 : cnt;
    const int nmove = ok ? cnt - first : 0;
    if (lane == 0) bulk_wait_read_all();   // the previous block's stores have read the stage
    __syncwarp();
    if (lane >= first && lane < cnt) msrc[lane - first] = a;
    __syncwarp();
    int my_pos = 0;
    if (nmove > 0) {
      warp_gather(lr.k, v.row0, mk, stg + L.k, msrc, nmove);
      warp_gather(lr.ks, v.row0, mks, stg + L.ks, msrc, nmove);
      warp_gather(lr.v, v.row0, mv, stg + L.v, msrc, nmove);
      warp_gather(lr.vs, v.row0, mvs, stg + L.vs, msrc, nmove);
      if (lane < nmove) my_pos = __ldcg(lr.pos + v.row0 + msrc[lane]);
    }
    cp_async_commit();
    nstate = claim(nsg, nj);   // the next block's claim travels while the rows load
    cp_async_wait<0>();
    __syncwarp();
    if (lane < nmove) msrc[lane] = my_pos;
    __syncwarp();
    // publish "read"; then wait for the lower blocks that read my destination rows
    uint32_t* flags = P.flags + (size_t)sg * P.c_max;
    int go = 0;
    if (lane == 0) {
      st_relaxed_u32(&flags[j], tag);
      go = ok;
      if (go && nmove > 0 && p1 > p0) {
        const int lo_b = p0 / kChunk, hi_b = min((p1 - 1) / kChunk, j - 1);
        for (int cc = lo_b; cc <= hi_b; ++cc)
          if (!wait_flag_bounded(&flags[cc], tag, P.spin_limit)) {
            go = 0;
            report(P.ctrl, TRIA_ERR_TIMEOUT, (uint32_t)sg);
            break;
          }
      }
    }
    go = __shfl_sync(0xffffffffu, go, 0);
    if (go && nmove > 0) {
      const int dst0 = i0 + first;
      if (lane == 0) {
        fence_proxy_async_smem();
        bulk_s2g(lr.k + (size_t)(v.row0 + dst0) * P.k_rb, stg + L.k, (uint32_t)(nmove * P.k_rb));
        bulk_s2g(lr.v + (size_t)(v.row0 + dst0) * P.v_rb, stg + L.v, (uint32_t)(nmove * P.v_rb));
        bulk_commit();
      }
      warp_scatter(lr.ks, v.row0, P.ks_rb, stg + L.ks, dst0, nmove, lane);
      warp_scatter(lr.vs, v.row0, P.vs_rb, stg + L.vs, dst0, nmove, lane);
      if (lane < nmove) lr.pos[v.row0 + dst0 + lane] = msrc[lane];
    }
    __syncwarp();
  }
  if (lane == 0) bulk_wait_all();
}

template <int KT, int G, int S>
__global__ void __launch_bounds__(kPassThreads, 1) k_pass(const __grid_constant__ FPass P) {
  using Body = TcBody<KT, G, S>;
  constexpr bool kQ8 = Body::kQ8;
  constexpr int FC = Body::FC;
  constexpr int kHeads = Body::kHeads;
  static_assert(FC <= 128, "turn table");

  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_item[2];      // current and next score item (-1: none)
  __shared__ int s_total, s_active, s_last;
  __shared__ uint32_t s_epoch;
  __shared__ Mom s_mom[kPassWarps][kMaxG];
  __shared__ int s_src[kPassWarps][kChunk];
  __shared__ int s_sbuf[40];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint8_t* ring = smem + PassSmem::kRing + (size_t)warp * 2 * kPassPieceBytes;
  uint8_t* sc_ring = smem + PassSmem::kScales + (size_t)warp * 2 * kPassScaleStage;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + PassSmem::kBars) + warp * 2;
  int* item0 = reinterpret_cast<int*>(smem + PassSmem::kItem0);
  unsigned long long* s_turns = reinterpret_cast<unsigned long long*>(smem + PassSmem::kTurns);
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem + PassSmem::kHist);

  // ---- prologue: item table (first score item of every segment), active
  // segments, turn factors, ring barriers
  if (tid < FC) s_turns[tid] = __ldg(P.turns + tid);
  {
    constexpr int kPer = (kPassMaxSegs + kPassThreads - 1) / kPassThreads;
    const int sb = min(P.n_seg, tid * kPer), se = min(P.n_seg, sb + kPer);
    int cnt[kPer];
    int local = 0, act = 0;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      cnt[i] = 0;
      const int sg = sb + i;
      if (sg < se) {
        const PSeg v = pass_seg(P, sg);
        if (!v.valid) {
          if (blockIdx.x == 0 && v.g == 0) report(P.ctrl, TRIA_ERR_DEVICE_ARG, (uint32_t)(v.li * P.n_seqs + v.s));
        } else if (v.active) {
          cnt[i] = (v.n + P.item_rows - 1) / P.item_rows;
          ++act;
        }
        local += cnt[i];
      }
    }
    int tot;
    int before = block_exclusive_scan(local, &tot, s_sbuf);
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int sg = sb + i;
      if (sg < se) {
        item0[sg] = before;
        before += cnt[i];
      }
    }
    if (tid == 0) {
      item0[P.n_seg] = tot;
      s_total = tot;
      s_active = 0;
    }
    __syncthreads();
    if (act) atomicAdd(&s_active, act);
  }
  if (lane == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_mbar_init();
  }
  __syncthreads();
  const int total = s_total, n_active = s_active;
  if (tid == 0) {
    s_epoch = ld_acquire_u32(&P.ctrl->epoch);
    int a = -1, b = -1;
    if (total > 0) {
      a = (int)atomicAdd(&P.ctrl->score_next, 1u);
      if (a >= total) a = -1;
      if (a >= 0) {
        b = (int)atomicAdd(&P.ctrl->score_next, 1u);
        if (b >= total) b = -1;
      }
    }
    s_item[0] = a;
    s_item[1] = b;
  }
  __syncthreads();

  auto seg_of_item = [&](int it) {   // largest sg with item0[sg] <= it
    int lo = 0, hi = P.n_seg - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (item0[mid] <= it) lo = mid;
      else hi = mid - 1;
    }
    return lo;
  };

  // ---- score items
  Body body;
  body.init(lane);
  int body_seg = -1;
  int n_issued = 0, n_done = 0;   // pieces of this warp through its ring
  int carried = 0;                // pieces of the current item issued during the previous one
  bool failed = false;
  // thread 0: the claim of the item after next (in flight during the current
  // item) and the completion count of the previous item, checked one item
  // later so that neither round trip sits between two items
  int pend_sg = -1, pend_items = 0, pend_old = 0;

  // item `it` as seen by this warp: its segment, the segment's geometry (live
  // rows are read only for a segment's last item: the others are full), and
  // this warp's pieces in it
  struct ItemView {
    int it, sg, n_pieces, rows_end;   // rows_end: first row past the item
  };
  auto view_of = [&](int it) {
    ItemView iv;
    iv.it = it;
    iv.sg = 0;
    iv.n_pieces = 0;
    iv.rows_end = 0;
    if (it < 0) return iv;
    iv.sg = seg_of_item(it);
    const int j = it - item0[iv.sg];
    if (it == item0[iv.sg + 1] - 1) {   // a segment's last item ends at its live rows
      const int li = iv.sg / (P.n_seqs * P.n_kv);
      const int s = (iv.sg - li * P.n_seqs * P.n_kv) / P.n_kv;
      iv.rows_end = *((volatile const int32_t*)(P.lay[li].n_live + s));
    } else {
      iv.rows_end = (j + 1) * P.item_rows;
    }
    const int r_beg = j * P.item_rows + warp * P.ppw * P.piece_rows;
    const int left = iv.rows_end - r_beg;
    iv.n_pieces = left <= 0 ? 0 : min(P.ppw, (left + P.piece_rows - 1) / P.piece_rows);
    return iv;
  };
  // first row of segment sg in its layer's planes
  auto seg_row0 = [&](int sg) {
    const int r = sg % (P.n_seqs * P.n_kv);
    const int s = r / P.n_kv;
    return P.seq[s].row0 + (int64_t)(r - s * P.n_kv) * P.seq[s].cap;
  };
  // rows [r0, r0 + rows) of piece i of this warp in item iv
  auto piece_r0 = [&](const ItemView& iv, int i) {
    return (iv.it - item0[iv.sg]) * P.item_rows + (warp * P.ppw + i) * P.piece_rows;
  };
  auto issue = [&](const ItemView& iv, int i) {   // warp-collective
    const int st = n_issued & 1;
    const int r0 = piece_r0(iv, i);
    const int rows = min(P.piece_rows, iv.rows_end - r0);
    const int64_t grow = seg_row0(iv.sg) + r0;
    const int li = iv.sg / (P.n_seqs * P.n_kv);
    if (lane == 0) {
      const uint32_t bytes = (uint32_t)(rows * P.k_rb);
      mbar_arrive_expect_tx(&bars[st], bytes);
      bulk_g2s(ring + st * kPassPieceBytes, P.lay[li].k + (size_t)grow * P.k_rb, bytes, &bars[st]);
    }
    if constexpr (kQ8) {
      const uint8_t* src = P.lay[li].ks + (size_t)grow * P.ks_rb;
      uint8_t* dst = sc_ring + st * kPassScaleStage;
      for (int u = lane; u < rows * P.ks_rb / 4; u += 32) cp_async4(dst + 4 * u, src + 4 * u);
      cp_async_commit();
    }
    ++n_issued;
  };

  ItemView nv = view_of(s_item[1]);
  while (s_item[0] >= 0) {
    const int cur = s_item[0], nxt = s_item[1];
    const ItemView cv = nv.it == cur ? nv : view_of(cur);
    nv = failed ? view_of(-1) : view_of(nxt);
    int claim = -1;
    if (tid == 0 && nxt >= 0) claim = (int)atomicAdd(&P.ctrl->score_next, 1u);   // used after this item
    const int nc = cv.n_pieces, nn = nv.n_pieces;
    if (cv.sg != body_seg) {
      const int li = cv.sg / (P.n_seqs * P.n_kv);
      const int r = cv.sg - li * P.n_seqs * P.n_kv;
      const int s = r / P.n_kv;
      const size_t qo = P.lay[li].qe_off + (size_t)(r - s * P.n_kv) * G * FC;
      body.load_consts(P.qe + qo, P.mw + qo, s_turns, (unsigned long long)P.seq[s].cur_pos);
      body_seg = cv.sg;
    }
    int iss = carried;   // pieces of [current item..., next item...] issued so far
    auto issue_seq = [&](int idx) {
      if (idx < nc) issue(cv, idx);
      else issue(nv, idx - nc);
    };
    for (int i = 0; i < nc && !failed; ++i) {
      while (iss <= i) issue_seq(iss++);
      if (iss == i + 1 && (i + 1 < nc || i + 1 - nc < nn)) issue_seq(iss++);   // one ahead, possibly the next item's
      const int st = n_done & 1;
      if (!mbar_wait_bounded(&bars[st], (uint32_t)((n_done >> 1) & 1), P.spin_limit)) {
        if (lane == 0) report(P.ctrl, TRIA_ERR_TIMEOUT, (uint32_t)cv.sg);
        // wait again (bounded) for every copy still in flight, then stop scoring
        for (int d = n_done; d < n_issued; ++d) mbar_wait_bounded(&bars[d & 1], (uint32_t)((d >> 1) & 1), P.spin_limit);
        if constexpr (kQ8) cp_async_wait<0>();
        n_done = n_issued;
        failed = true;
        break;
      }
      if constexpr (kQ8) {
        if (n_issued - n_done >= 2) cp_async_wait<1>();
        else cp_async_wait<0>();
        __syncwarp();
      }
      const int r0 = piece_r0(cv, i);
      const int64_t wrow = (int64_t)(cv.sg / (P.n_seqs * P.n_kv)) * P.rows_per_layer + seg_row0(cv.sg) + r0;
      body.piece(ring + st * kPassPieceBytes, sc_ring + st * kPassScaleStage, min(P.piece_rows, cv.rows_end - r0),
                 P.k_rb, P.ks_rb, P.raw + (size_t)wrow * G);
      __syncwarp();
      ++n_done;
    }
    if (nc == 0 && !failed)
      while (iss < min(2, nn)) issue_seq(iss++);   // an idle warp starts the next item's pieces
    carried = failed ? 0 : iss - nc;

    // the item's moments: per warp, then merged over the warps in order
    {
      Mom m[kHeads];
      body.flush(m);
      if (body.flush_writer()) {
#pragma unroll
        for (int kk = 0; kk < kHeads; ++kk) s_mom[warp][body.oh + kk] = m[kk];
      }
    }
    __syncthreads();
    if (tid < G) {
      Mom a{0.f, 0.f, 0.f};
      for (int w = 0; w < kPassWarps; ++w) a = mom_merge(a, s_mom[w][tid]);
      float* tab = P.parts + (size_t)cv.sg * kRunCols * P.cs_max;
      const int j = cur - item0[cv.sg];
      tab[(1 + tid) * P.cs_max + j] = a.mean;
      tab[(1 + kMaxG + tid) * P.cs_max + j] = a.m2;
      if (tid == 0) tab[j] = a.n;
    }
    __syncthreads();
    if (tid == 0) {
      // the previous item's completion count has arrived by now
      s_last = (pend_sg >= 0 && pend_old == pend_items - 1) ? pend_sg : -1;
      // this item's raw scores and moments (every thread's, ordered by the
      // barrier) before its completion count
      __threadfence();
      pend_sg = cv.sg;
      pend_items = item0[cv.sg + 1] - item0[cv.sg];
      pend_old = atomicAdd(&P.ctl->items_done[cv.sg], 1);
      s_item[0] = nxt;
      s_item[1] = claim < total ? claim : -1;
    }
    __syncthreads();
    // selections due: the segment the previous item completed (s_last), and
    // once no item is left, the one the last item completed
    while (true) {
      if (s_last >= 0) {
        __threadfence();
        pass_select<G>(P, s_last, item0[s_last + 1] - item0[s_last], hist);
      }
      if (s_item[0] >= 0) break;
      __syncthreads();
      if (tid == 0) {
        s_last = (pend_sg >= 0 && pend_old == pend_items - 1) ? pend_sg : -1;
        pend_sg = -1;
      }
      __syncthreads();
      if (s_last < 0) break;
    }
  }

  // ---- moves: warps claim destination blocks of ready segments
  {
    const MoveStage L = move_stage_layout(P.k_rb, P.ks_rb, P.v_rb, P.vs_rb);
    if (warp < min(kPassWarps, kPassRing / L.bytes) && n_active > 0)
      pass_moves(P, smem + PassSmem::kRing + (size_t)warp * L.bytes, s_src[warp], flag_tag(s_epoch), n_active);
  }

  // ---- the last CTA: n_live of the active sequences, counters reset
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    s_last = atomicAdd(&P.ctrl->pass_done, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int i = tid; i < P.n_layers * P.n_seqs; i += blockDim.x) {
    const int li = i / P.n_seqs, s = i - li * P.n_seqs;
    int32_t* nl = P.lay[li].n_live + s;
    const int n = *((volatile int32_t*)nl);
    if (n >= 0 && n <= P.seq[s].cap && n > P.seq[s].budget) *nl = P.seq[s].budget;
  }
  const int n_ready = (int)ld_acquire_u32(&P.ctrl->ready_count);
  for (int i = tid; i < min(n_ready, P.n_seg); i += blockDim.x) P.ctl->ready[i] = 0;
  for (int sg = tid; sg < P.n_seg; sg += blockDim.x) {
    P.ctl->items_done[sg] = 0;
    P.ctl->move_next[sg] = 0;
  }
  __syncthreads();
  if (tid == 0) {
    P.ctrl->score_next = 0u;
    P.ctrl->ready_count = 0u;
    P.ctrl->move_cursor = 0u;
    P.ctrl->pass_done = 0u;
    __threadfence();
    atomicAdd(&P.ctrl->epoch, 1u);
  }
}

}  // namespace tria

namespace tria {

// Host side of the fused pass.
// Rows of keys per scorer piece (whole 16-row tiles, at most 8 KB).
inline int pass_piece_rows(int k_rb) {
  int r = kPassPieceBytes / k_rb;
  if (r > 64) r = 64;
  if (r >= 16) r &= ~15;
  return r < 1 ? 1 : r;
}

// fp16 / q8_0 keys with head_dim 64, 128 or 256 (group <= 4 at 256): the
// tensor-core body's shapes that the fused kernel is built for
inline bool pass_supported(int k_type, int hd, int G) {
  if (k_type != TRIA_F16 && k_type != TRIA_Q8_0) return false;
  if (G != 1 && G != 2 && G != 4 && G != 8) return false;
  if (hd == 64 || hd == 128) return true;
  return hd == 256 && G <= 4;
}

cudaError_t launch_pass_f16(const FPass& P, cudaStream_t st);   // pass_f16.cu
cudaError_t launch_pass_q8(const FPass& P, cudaStream_t st);    // pass_q8.cu

template <int KT, int G, int S>
cudaError_t launch_pass_t(const FPass& P, cudaStream_t st) {
  auto kern = k_pass<KT, G, S>;
  static const cudaError_t attr = set_smem_attrs(kern, PassSmem::kBytes);
  if (attr != cudaSuccess) return attr;
  static int grid = 0;
  if (grid == 0) {
    int dev = 0, sms = 0, per_sm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kPassThreads, PassSmem::kBytes);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    grid = sms;   // one CTA per SM
  }
  void* args[] = {const_cast<FPass*>(&P)};
  return cudaLaunchCooperativeKernel((const void*)kern, dim3(grid), dim3(kPassThreads), args,
                                     (size_t)PassSmem::kBytes, st);
}

template <int KT>
cudaError_t launch_pass_k(const FPass& P, cudaStream_t st) {
  switch (P.hd) {
    case 64:
      switch (P.G) {
        case 1: return launch_pass_t<KT, 1, 2>(P, st);
        case 2: return launch_pass_t<KT, 2, 2>(P, st);
        case 4: return launch_pass_t<KT, 4, 2>(P, st);
        case 8: return launch_pass_t<KT, 8, 2>(P, st);
      }
      break;
    case 128:
      switch (P.G) {
        case 1: return launch_pass_t<KT, 1, 4>(P, st);
        case 2: return launch_pass_t<KT, 2, 4>(P, st);
        case 4: return launch_pass_t<KT, 4, 4>(P, st);
        case 8: return launch_pass_t<KT, 8, 4>(P, st);
      }
      break;
    case 256:
      switch (P.G) {
        case 1: return launch_pass_t<KT, 1, 8>(P, st);
        case 2: return launch_pass_t<KT, 2, 8>(P, st);
        case 4: return launch_pass_t<KT, 4, 8>(P, st);
      }
      break;
  }
  return cudaErrorInvalidValue;
}

}  // namespace tria
