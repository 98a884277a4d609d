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
//  * Scoring: the live rows of all segments, in segment order, are cut into
//    pieces of at most 8 KB of keys, and every warp of the grid takes one
//    contiguous run of them, streamed through a private two-stage ring (bulk
//    async copies completing on mbarriers), exactly as the staged scorer
//    does; no CTA-wide step interrupts the stream. A warp writes one moment
//    partial per (run, segment) and adds its pieces to the segment's scored
//    count; the warp that completes a segment appends it to the scored list.
//  * Service: a CTA whose warps have all finished scoring selects scored
//    segments (one CTA per segment: segment moments from the run partials,
//    z-max keys in shared memory where they fit, radix select, keep list and
//    the kept-row prefix of every 32-row chunk) and appends each to the ready
//    list; while no segment waits for selection its warps move one block
//    each; once every segment is selected they only move. A move claims a
//    32-row destination block of a ready segment (one counter per segment)
//    and moves it as k_move does: gather the block's moving rows into the
//    warp's stage, publish "read", wait (bounded) for the lower blocks that
//    read its destination rows, store. The next block's claim and keep
//    entries load while the current block's rows load.
//  * Final moves: once every segment is selected (a grid barrier), the
//    blocks left move in k_move's block-major order, with the whole dynamic
//    shared memory as move stages (224 KB).
//  * The last CTA to finish sets n_live and resets the call's counters.
// The scored / ready lists and the per-segment counters live at a fixed
// place of the workspace (PassCtl). Every wait is bounded
// (TRIA_ERR_TIMEOUT after the spin limit), and a wait only ever waits for
// work that a running warp has started, so the schedule cannot deadlock.
#pragma once

#include "move.cuh"
#include "score_tc.cuh"

namespace tria {

constexpr int kPassWarps = 12;
constexpr int kPassThreads = kPassWarps * 32;
constexpr int kPassPieceBytes = 8192;
constexpr int kPassScaleStage = kPassPieceBytes / 16;   // q8_0 block scales of a piece
constexpr int kPassRing = kPassWarps * 2 * kPassPieceBytes;
constexpr int kPassMaxSegs = kPassCtlSegs;   // layers x sequences x KV heads per call
constexpr int kPassMaxLayers = 128;
// A select keeps its radix histogram in the last 8 KB of the ring area and up
// to kPassSmemKeys z-max keys before it (the ring is free once scoring ends).
constexpr int kPassHistOff = kPassRing - kHistBins * 4;
constexpr int kPassSmemKeys = kPassHistOff / 4;

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
  int32_t piece_rows;   // key rows per piece
  int32_t cs_max;       // columns of a segment's run-partial table (>= its score runs)
  int32_t dyn_bytes;    // dynamic shared memory of the launch (set by the launcher)
  int32_t c_max;        // chunks per segment (max)
  int64_t rows_per_layer;   // workspace rows of one layer
  const float2* qe;
  const float* mw;
  const unsigned long long* turns;   // [fc] frac(w_f / 2pi) * 2^64 (shared by the call's layers)
  float* raw;                        // [layer rows][G]
  uint32_t* keys;                    // [layer rows] z-max keys of segments too long for shared memory
  float* score_out;                  // [layer rows] z-max scores, or null
  int32_t* keep;                     // [layer rows]
  Ctrl* ctrl;
  PassCtl* ctl;                      // scored / ready lists and per-segment counters
  float* parts;                      // [n_seg][kRunCols][cs_max] score-run moment partials
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

// dynamic shared memory: ring (score stream; then a select's z-max keys and
// histogram, or move stages) | q8_0 scale ring | mbarriers | piece table |
// turn factors
struct PassSmem {
  static constexpr int kRing = 0;
  static constexpr int kScales = kRing + kPassRing;
  static constexpr int kBars = kScales + kPassWarps * 2 * kPassScaleStage;
  static constexpr int kFirst = kBars + kPassWarps * 2 * 8;
  static constexpr int kTurns = kFirst + ((kPassMaxSegs + 1) * 4 + 15) / 16 * 16;
  static constexpr int kBytes = kTurns + 128 * 8;
};
// The final move phase reuses all of it (and a little more) as move stages:
// k_move's 224 KB, seven 32 KB stages of head_dim-256 fp16 key + value rows.
constexpr int kPassDynBytes = PassSmem::kBytes > kMoveSmemLimit ? PassSmem::kBytes : kMoveSmemLimit;

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

// z-max keys: in shared memory (kSmem) or in the workspace
template <bool kSmem>
struct KeyStore {
  uint32_t* p;
  __device__ __forceinline__ uint32_t get(int r) const {
    if constexpr (kSmem) return p[r];
    else return __ldcg(p + r);
  }
  __device__ __forceinline__ void put(int r, uint32_t k) const {
    if constexpr (kSmem) p[r] = k;
    else __stcg(p + r, k);
  }
};

// Selection of one segment by the whole CTA: segment moments from its nr
// score-run partials, z-max keys and the first radix histogram in one sweep,
// up to two more radix passes, then the keep list (B entries) and the
// kept-row prefix of every chunk; publishes the segment in the ready list.
// smem_keys: the keys (kSmem) or, with the keys in the workspace, scratch
// for the chunks' ballots (both in the ring area, below the histogram).
template <int G, bool kSmem>
__device__ __noinline__ void pass_select(const FPass& P, int sg, int nr, uint32_t* smem_keys, uint32_t* hist) {
  __shared__ int s_info[4];
  __shared__ int s_sbuf[40];
  __shared__ int s_wt[kPassWarps], s_wk[kPassWarps];
  const PSeg v = pass_seg(P, sg);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = v.n, lo = v.sink, hi = n - P.window;
  const int k = v.B - v.sink - P.window;
  const KeyStore<kSmem> keys{kSmem ? smem_keys : P.keys + v.wrow0};
  constexpr int UB = kSmem ? 1 : 32;   // key loads in flight per thread (global keys)

  float mu[G], inv[G];
  // the histogram's words serve as the merge's scratch first
  block_moments_of_runs<G>(P.parts + (size_t)sg * kRunCols * P.cs_max, P.cs_max, nr, mu, inv,
                           reinterpret_cast<float*>(hist));
  __syncthreads();
  for (int i = tid; i < kHistBins; i += blockDim.x) hist[i] = 0u;
  __syncthreads();

  // z-max keys of every live row and the first radix histogram of the
  // candidates [lo, hi); loads of U rows per thread are in flight together,
  // and the next batch's lines are asked for in L2 meanwhile (one prefetch
  // per 128-byte line, by the thread whose row starts it)
  {
    constexpr int U = G > 4 ? 4 : (G == 4 ? 8 : 16);   // raw rows in flight per thread
    constexpr int kRowsPerLine = 128 / (4 * G);
    const float* raw = P.raw + (size_t)v.wrow0 * G;
    float* so = P.score_out ? P.score_out + v.wrow0 : nullptr;
    const bool line_head = (v.wrow0 + tid) % kRowsPerLine == 0;   // rows of this thread start lines
    for (int base = tid; base < n; base += U * kPassThreads) {
      float x[U][G];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int r = base + u * kPassThreads;
        if (r < n) load_raw_g<G>(raw + (size_t)r * G, x[u]);
      }
      if (line_head) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int r = base + (U + u) * kPassThreads;
          if (r < n) asm volatile("prefetch.global.L2 [%0];" ::"l"(raw + (size_t)r * G));
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int r = base + u * kPassThreads;
        if (r < n) {
          float s = (x[u][0] - mu[0]) * inv[0];
#pragma unroll
          for (int h = 1; h < G; ++h) s = fmaxf(s, (x[u][h] - mu[h]) * inv[h]);
          const uint32_t key = score_key(s);
          keys.put(r, key);
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
        for (int base = lo + tid; base < hi; base += UB * kPassThreads) {
          uint32_t kk[UB];
#pragma unroll
          for (int u = 0; u < UB; ++u) {
            const int r = base + u * kPassThreads;
            kk[u] = r < hi ? keys.get(r) : 0u;
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
  // ties and strict keeps, sweep 2 writes the kept rows and chunk prefixes.
  // With the keys in the workspace, sweep 1 also leaves each chunk's tie and
  // strict-keep ballots in shared memory (the ring area is free then; 8 bytes
  // a chunk), so that sweep 2 reads no key again.
  const int nch = (n + kChunk - 1) / kChunk;
  const int cpw = (nch + kPassWarps - 1) / kPassWarps;
  const int c0 = min(nch, warp * cpw), c1 = min(nch, c0 + cpw);
  constexpr int CB = kSmem ? 1 : 16;   // chunks whose keys load together (global keys)
  uint2* masks = !kSmem && nch * 8 <= kPassHistOff ? reinterpret_cast<uint2*>(smem_keys) : nullptr;
  {
    int wt = 0, wk = 0;
    for (int cb = c0; cb < c1; cb += CB) {
      uint32_t kk[CB];
#pragma unroll
      for (int u = 0; u < CB; ++u) {
        const int r = (cb + u) * kChunk + lane;
        kk[u] = (cb + u < c1 && r < n && r >= lo && r < hi && k > 0) ? keys.get(r) : 0u;
      }
#pragma unroll
      for (int u = 0; u < CB; ++u) {
        if (cb + u >= c1) break;
        const int r = (cb + u) * kChunk + lane;
        const bool in = r < n;
        const bool pr = in && (r < lo || r >= hi);
        const bool cand = in && !pr && k > 0;
        const uint32_t bt = __ballot_sync(0xffffffffu, cand && kk[u] == T);
        const uint32_t bs = __ballot_sync(0xffffffffu, pr || (cand && kk[u] > T));
        if (masks && lane == 0) masks[cb + u] = make_uint2(bt, bs);
        wt += __popc(bt);
        wk += __popc(bs);
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
  const uint32_t lt = (1u << lane) - 1u;
  // one chunk: its tie and strict-keep ballots -> its kept rows (the ties by
  // rank), written at the run's position
  auto emit_chunk = [&](int ci, uint32_t bt, uint32_t bs) {
    const int r = ci * kChunk + lane;
    const bool is_tie = (bt >> lane) & 1u;
    const int trank = tie_run + __popc(bt & lt);
    const bool kp = ((bs >> lane) & 1u) || (is_tie && trank < kr);
    const uint32_t bk = __ballot_sync(0xffffffffu, kp);
    if (lane == 0) pre[ci] = keep_run;
    if (kp) keep[keep_run + __popc(bk & lt)] = r;
    tie_run += __popc(bt);
    keep_run += __popc(bk);
  };
  if (masks) {
    for (int ci = c0; ci < c1; ++ci) {
      const uint2 m = masks[ci];
      emit_chunk(ci, m.x, m.y);
    }
  } else {
    for (int cb = c0; cb < c1; cb += CB) {
      uint32_t kk[CB];
#pragma unroll
      for (int u = 0; u < CB; ++u) {
        const int r = (cb + u) * kChunk + lane;
        kk[u] = (cb + u < c1 && r < n && r >= lo && r < hi && k > 0) ? keys.get(r) : 0u;
      }
#pragma unroll
      for (int u = 0; u < CB; ++u) {
        const int ci = cb + u;
        if (ci >= c1) break;
        const int r = ci * kChunk + lane;
        const bool in = r < n;
        const bool pr = in && (r < lo || r >= hi);
        const bool cand = in && !pr && k > 0;
        emit_chunk(ci, __ballot_sync(0xffffffffu, cand && kk[u] == T),
                   __ballot_sync(0xffffffffu, pr || (cand && kk[u] > T)));
      }
    }
  }
  if (warp == kPassWarps - 1 && lane == 0) {
    pre[nch] = v.B;
    if (keep_run != v.B) report(P.ctrl, TRIA_ERR_INVALID_ARG, 0x20000000u | (uint32_t)sg);
  }
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const uint32_t slot = atomicAdd(&P.ctrl->ready_count, 1u);
    st_release_u32(reinterpret_cast<uint32_t*>(P.ctl->ready + slot), (uint32_t)(sg + 1));
  }
  __syncthreads();
}

// A claimed destination block: segment, block index, the lane's keep entry,
// the keep-index range that reads the block's source rows, and the
// segment's geometry.
struct MoveClaim {
  int state;   // 0 block, 1 none ready yet, 2 every block claimed
  int sg, j, a, p0, p1;
  int n, B, li;
  int64_t row0, wrow0;
};

// lane 0 claims the next block, first from the segment of its previous claim
// (one atomic), else from the oldest ready segment that has one; then every
// lane loads the block's keep entries (warp-collective)
__device__ __forceinline__ MoveClaim pass_claim(const FPass& P, int n_active, int& last_sg) {
  const int lane = threadIdx.x & 31;
  int state = 1, sg = 0, j = 0;
  auto blocks_of = [&](int g) {
    return (P.seq[(g % (P.n_seqs * P.n_kv)) / P.n_kv].budget + kChunk - 1) / kChunk;
  };
  if (lane == 0) {
    if (last_sg >= 0) {
      j = atomicAdd(&P.ctl->move_next[last_sg], 1);
      if (j < blocks_of(last_sg)) {
        state = 0;
        sg = last_sg;
      }
    }
    while (state != 0) {
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
      j = atomicAdd(&P.ctl->move_next[sg], 1);
      if (j >= 0 && j < blocks_of(sg)) {
        state = 0;
        break;
      }
      atomicCAS(&P.ctrl->move_cursor, c, c + 1u);   // exhausted: move past it
    }
    last_sg = state == 0 ? sg : -1;
  }
  MoveClaim m;
  m.state = __shfl_sync(0xffffffffu, state, 0);
  m.sg = __shfl_sync(0xffffffffu, sg, 0);
  m.j = __shfl_sync(0xffffffffu, j, 0);
  m.a = -1;
  m.p0 = m.p1 = 0;
  if (m.state == 0) {
    const PSeg v = pass_seg(P, m.sg);
    m.n = v.n;
    m.B = v.B;
    m.li = v.li;
    m.row0 = v.row0;
    m.wrow0 = v.wrow0;
    const int i = m.j * kChunk + lane;
    m.a = i < v.B ? __ldcg(P.keep + v.wrow0 + i) : -1;
    const int* pre = P.prefix + (size_t)m.sg * (P.c_max + 1);
    m.p0 = __ldcg(&pre[m.j]);
    m.p1 = __ldcg(&pre[m.j + 1]);
  }
  return m;
}

// k_move's steps for one claimed block, split at the gather: start_gather
// validates the block, records its moving source rows in msrc and starts
// the cp.async gathers into stg (one commit group); finish writes the rows
// out once they have landed (publish "read", wait for the lower blocks that
// read the destination rows, TMA bulk stores, one bulk group).
struct MoveWork {
  int first, nmove, my_pos;
  bool ok;
};

__device__ __forceinline__ MoveWork pass_gather(const FPass& P, const MoveClaim& m, uint8_t* stg, int* msrc) {
  const int lane = threadIdx.x & 31;
  const MoveStage L = move_stage_layout(P.k_rb, P.ks_rb, P.v_rb, P.vs_rb);
  const PlaneMap mk = plane_map(P.k_rb, lane), mks = plane_map(P.ks_rb, lane), mv = plane_map(P.v_rb, lane),
                 mvs = plane_map(P.vs_rb, lane);
  const LayerRef& lr = P.lay[m.li];
  const int i0 = m.j * kChunk, cnt = min(kChunk, m.B - i0);
  const bool bad_entry = lane < cnt && (m.a < i0 + lane || m.a >= m.n);
  MoveWork w;
  w.ok = !__any_sync(0xffffffffu, bad_entry) && m.p0 >= 0 && m.p0 <= m.p1 && m.p1 - m.p0 <= kChunk &&
         m.p1 <= m.B;
  if (!w.ok && lane == 0) report(P.ctrl, TRIA_ERR_INVALID_ARG, 0x10000000u | (uint32_t)m.sg);
  // moving entries (keep[i] != i) are a suffix of the block
  const unsigned mvm = __ballot_sync(0xffffffffu, w.ok && lane < cnt && m.a != i0 + lane);
  w.first = mvm ? __ffs(mvm) - 1 : cnt;
  w.nmove = w.ok ? cnt - w.first : 0;
  if (lane >= w.first && lane < cnt) msrc[lane - w.first] = m.a;
  __syncwarp();
  w.my_pos = 0;
  if (w.nmove > 0) {
    warp_gather(lr.k, m.row0, mk, stg + L.k, msrc, w.nmove);
    warp_gather(lr.ks, m.row0, mks, stg + L.ks, msrc, w.nmove);
    warp_gather(lr.v, m.row0, mv, stg + L.v, msrc, w.nmove);
    warp_gather(lr.vs, m.row0, mvs, stg + L.vs, msrc, w.nmove);
    if (lane < w.nmove) w.my_pos = __ldcg(lr.pos + m.row0 + msrc[lane]);
  }
  cp_async_commit();
  return w;
}

// call once the block's gather group has completed (cp.async wait + syncwarp)
__device__ __forceinline__ void pass_store(const FPass& P, const MoveClaim& m, const MoveWork& w, uint8_t* stg,
                                           int* msrc, uint32_t tag) {
  const int lane = threadIdx.x & 31;
  const MoveStage L = move_stage_layout(P.k_rb, P.ks_rb, P.v_rb, P.vs_rb);
  const LayerRef& lr = P.lay[m.li];
  if (lane < w.nmove) msrc[lane] = w.my_pos;
  __syncwarp();
  // publish "read"; then wait for the lower blocks that read my destination rows
  uint32_t* flags = P.flags + (size_t)m.sg * P.c_max;
  int go = 0;
  if (lane == 0) {
    st_relaxed_u32(&flags[m.j], tag);
    go = w.ok;
    if (go && w.nmove > 0 && m.p1 > m.p0) {
      const int lo_b = m.p0 / kChunk, hi_b = min((m.p1 - 1) / kChunk, m.j - 1);
      for (int cc = lo_b; cc <= hi_b; ++cc)
        if (!wait_flag_bounded(&flags[cc], tag, P.spin_limit)) {
          go = 0;
          report(P.ctrl, TRIA_ERR_TIMEOUT, (uint32_t)m.sg);
          break;
        }
    }
  }
  go = __shfl_sync(0xffffffffu, go, 0);
  if (go && w.nmove > 0) {
    const int dst0 = m.j * kChunk + w.first;
    if (lane == 0) {
      fence_proxy_async_smem();
      bulk_s2g(lr.k + (size_t)(m.row0 + dst0) * P.k_rb, stg + L.k, (uint32_t)(w.nmove * P.k_rb));
      bulk_s2g(lr.v + (size_t)(m.row0 + dst0) * P.v_rb, stg + L.v, (uint32_t)(w.nmove * P.v_rb));
    }
    warp_scatter(lr.ks, m.row0, P.ks_rb, stg + L.ks, dst0, w.nmove, lane);
    warp_scatter(lr.vs, m.row0, P.vs_rb, stg + L.vs, dst0, w.nmove, lane);
    if (lane < w.nmove) lr.pos[m.row0 + dst0 + lane] = msrc[lane];
  }
  if (lane == 0) bulk_commit();   // one bulk group per block (possibly empty)
  __syncwarp();
}

// Grid barrier of the pass (every CTA resident), bounded: after the spin
// limit it records TRIA_ERR_TIMEOUT and lets the CTA go on.
__device__ __forceinline__ bool pass_grid_barrier(const FPass& P) {
  __shared__ int s_to;
  __syncthreads();
  if (threadIdx.x == 0) {
    s_to = 0;
    const uint32_t gen = ld_acquire_u32(&P.ctrl->bar_gen);
    __threadfence();
    if (atomicAdd(&P.ctrl->bar_count, 1u) == gridDim.x - 1) {
      atomicExch(&P.ctrl->bar_count, 0u);
      __threadfence();
      atomicAdd(&P.ctrl->bar_gen, 1u);
    } else if (!wait_flag_bounded_ne(&P.ctrl->bar_gen, gen, P.spin_limit)) {
      s_to = 1;
      report(P.ctrl, TRIA_ERR_TIMEOUT, 0xB0000002u);
    }
    __threadfence();
  }
  __syncthreads();
  return s_to == 0;
}

// The moves left once every segment is selected, in k_move's order: item t
// is block base[sg] + t / n_act of the segment in ready slot t % n_act
// (block-major, so the lower blocks that read a block's rows come in earlier
// rounds), mover warp w of the grid takes items w, w + Wm, ... and loads the
// next item's keep entries while it moves the current one. When every item
// has a warp of its own, all gather, one grid barrier marks every read done,
// and all write (no read-done flags). Every CTA calls it (grid barriers).
static __device__ __noinline__ void pass_moves_final(const FPass& P, uint8_t* stg, int* msrc, uint32_t tag, int n_act,
                                              int mover_warps, int j_span) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const bool mover = warp < mover_warps;
  const int Wm = gridDim.x * mover_warps;
  const int total = n_act * j_span;
  const bool one_round = total <= Wm;
  auto fetch = [&](int t, MoveClaim& m) {
    m.state = 2;
    if (t >= total) return;
    const int slot = t % n_act;
    const int sg = __ldcg(P.ctl->ready + slot) - 1;
    const PSeg v = pass_seg(P, sg);
    const int nb = (v.B + kChunk - 1) / kChunk;
    const int j = __ldcg(P.ctl->move_next + sg) + t / n_act;   // blocks below were moved while selecting
    m.state = j < nb ? 0 : 1;   // 1: no such block in this segment
    m.sg = sg;
    m.j = j;
    m.n = v.n;
    m.B = v.B;
    m.li = v.li;
    m.row0 = v.row0;
    m.wrow0 = v.wrow0;
    m.a = -1;
    m.p0 = m.p1 = 0;
    if (m.state == 0) {
      const int i = j * kChunk + lane;
      m.a = i < v.B ? __ldcg(P.keep + v.wrow0 + i) : -1;
      const int* pre = P.prefix + (size_t)sg * (P.c_max + 1);
      m.p0 = __ldcg(&pre[j]);
      m.p1 = __ldcg(&pre[j + 1]);
    }
  };
  MoveClaim pend{};
  MoveWork pend_w{};
  bool pending = false;
  // this warp's items, in order
  if (mover) {
    int t = blockIdx.x * mover_warps + warp;
    MoveClaim m;
    fetch(t, m);
    while (m.state != 2) {
      MoveClaim nx;
      fetch(t + Wm, nx);   // the next item's keep entries load while this one moves
      if (m.state == 0) {
        if (lane == 0) bulk_wait_read_all();   // the previous item's stores have read the stage
        __syncwarp();
        const MoveWork w = pass_gather(P, m, stg, msrc);
        cp_async_wait<0>();
        __syncwarp();
        if (one_round) {   // the only item of this warp: write after the barrier
          pend = m;
          pend_w = w;
          pending = true;
          if (lane < w.nmove) msrc[lane] = w.my_pos;
          __syncwarp();
          break;
        }
        pass_store(P, m, w, stg, msrc, tag);
      }
      m = nx;
      t += Wm;
    }
  }
  if (one_round) {
    const bool in_time = pass_grid_barrier(P);
    if (pending && in_time && pend_w.nmove > 0) {
      const MoveStage L = move_stage_layout(P.k_rb, P.ks_rb, P.v_rb, P.vs_rb);
      const LayerRef& lr = P.lay[pend.li];
      const int dst0 = pend.j * kChunk + pend_w.first;
      if (lane == 0) {
        fence_proxy_async_smem();
        bulk_s2g(lr.k + (size_t)(pend.row0 + dst0) * P.k_rb, stg + L.k, (uint32_t)(pend_w.nmove * P.k_rb));
        bulk_s2g(lr.v + (size_t)(pend.row0 + dst0) * P.v_rb, stg + L.v, (uint32_t)(pend_w.nmove * P.v_rb));
        bulk_commit();
      }
      warp_scatter(lr.ks, pend.row0, P.ks_rb, stg + L.ks, dst0, pend_w.nmove, lane);
      warp_scatter(lr.vs, pend.row0, P.vs_rb, stg + L.vs, dst0, pend_w.nmove, lane);
      if (lane < pend_w.nmove) lr.pos[pend.row0 + dst0 + lane] = msrc[lane];
      __syncwarp();
    }
  }
  if (mover && lane == 0) bulk_wait_all();
}

template <int KT, int G, int S>
__global__ void __launch_bounds__(kPassThreads, 1) k_pass(const __grid_constant__ FPass P) {
  using Body = TcBody<KT, G, S>;
  constexpr bool kQ8 = Body::kQ8;
  constexpr int FC = Body::FC;
  constexpr int kHeads = Body::kHeads;
  static_assert(FC <= 128, "turn table");

  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_active, s_sel, s_last;
  __shared__ uint32_t s_epoch;
  __shared__ int s_src[kPassWarps][kChunk];   // per warp: a block's source rows, then positions
  __shared__ int s_sbuf[40];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint8_t* ring = smem + PassSmem::kRing + (size_t)warp * 2 * kPassPieceBytes;
  uint8_t* sc_ring = smem + PassSmem::kScales + (size_t)warp * 2 * kPassScaleStage;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + PassSmem::kBars) + warp * 2;
  int* seg_first = reinterpret_cast<int*>(smem + PassSmem::kFirst);   // first piece of every segment
  unsigned long long* s_turns = reinterpret_cast<unsigned long long*>(smem + PassSmem::kTurns);
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem + PassSmem::kRing + kPassHistOff);   // service phase only

  // ---- prologue: piece table (pieces of the active segments, in segment
  // order), active segments, turn factors, ring barriers
  if (tid < FC) s_turns[tid] = __ldg(P.turns + tid);
  if (tid == 0) {
    s_active = 0;
    s_epoch = ld_acquire_u32(&P.ctrl->epoch);
  }
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
          cnt[i] = (v.n + P.piece_rows - 1) / P.piece_rows;
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
        seg_first[sg] = before;
        before += cnt[i];
      }
    }
    if (tid == 0) seg_first[P.n_seg] = tot;
    if (act) atomicAdd(&s_active, act);
  }
  if (lane == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_mbar_init();
  }
  __syncthreads();
  const int total = seg_first[P.n_seg], n_active = s_active;
  const int nwarps = gridDim.x * kPassWarps;
  const int per = (total + nwarps - 1) / nwarps;   // pieces per warp run

  // ---- scoring: this warp's run of pieces [p_beg, p_end)
  {
    const int gw = blockIdx.x * kPassWarps + warp;
    const int p_beg = min(total, gw * per), p_end = min(total, p_beg + per);
    auto seg_of = [&](int p, int from) {
      int sg = from;
      while (seg_first[sg + 1] <= p) ++sg;
      return sg;
    };
    // bulk copy of piece p of segment sg (v: the segment, its live rows)
    auto issue = [&](int p, int sg, const PSeg& v, int stage_i) {   // warp-collective
      const int r = (p - seg_first[sg]) * P.piece_rows;
      const int rows = min(P.piece_rows, v.n - r);
      const int64_t grow = v.row0 + r;
      if (lane == 0) {
        const uint32_t bytes = (uint32_t)(rows * P.k_rb);
        mbar_arrive_expect_tx(&bars[stage_i], bytes);
        bulk_g2s(ring + stage_i * kPassPieceBytes, P.lay[v.li].k + (size_t)grow * P.k_rb, bytes, &bars[stage_i]);
      }
      if constexpr (kQ8) {
        const uint8_t* src = P.lay[v.li].ks + (size_t)grow * P.ks_rb;
        uint8_t* dst = sc_ring + stage_i * kPassScaleStage;
        for (int u = lane; u < rows * P.ks_rb / 4; u += 32) cp_async4(dst + 4 * u, src + 4 * u);
        cp_async_commit();
      }
    };
    if (p_beg < p_end) {
      Body body;
      body.init(lane, FC);
      int seg = seg_of(p_beg, 0);
      PSeg sv = pass_seg(P, seg);
      issue(p_beg, seg, sv, 0);
      auto load_consts = [&]() {
        const size_t qo = P.lay[sv.li].qe_off + (size_t)sv.g * G * FC;
        body.load_consts(P.qe + qo, P.mw + qo, s_turns, (unsigned long long)P.seq[sv.s].cur_pos);
      };
      load_consts();
      int run_first = p_beg;
      // the run's moment partial, then its pieces into the segment's scored
      // count; the warp that completes the segment lists it as scored
      auto finish_run = [&](int p_stop) {
        Mom m[kHeads];
        body.flush(m);
        if (body.flush_writer()) {
          float* tab = P.parts + (size_t)seg * kRunCols * P.cs_max;
          const int r = run_index(run_first, seg_first[seg], per);
#pragma unroll
          for (int kk = 0; kk < kHeads; ++kk) {
            tab[(1 + body.oh + kk) * P.cs_max + r] = m[kk].mean;
            tab[(1 + kMaxG + body.oh + kk) * P.cs_max + r] = m[kk].m2;
          }
          if (body.q == 0) tab[r] = m[0].n;
        }
        __syncwarp();
        if (lane == 0) {
          __threadfence();
          const int np = p_stop - run_first;
          const int want = seg_first[seg + 1] - seg_first[seg];
          if (atomicAdd(&P.ctl->pieces_done[seg], np) + np == want) {
            __threadfence();
            const uint32_t slot = atomicAdd(&P.ctrl->scored_count, 1u);
            st_release_u32(reinterpret_cast<uint32_t*>(P.ctl->scored + slot), (uint32_t)(seg + 1));
          }
        }
      };
      for (int p = p_beg; p < p_end; ++p) {
        const int kp = p - p_beg;
        const int st = kp & 1;
        // next piece into the other stage (its previous contents were consumed)
        if (p + 1 < p_end) {
          const int sn = seg_of(p + 1, seg);
          if (sn == seg) issue(p + 1, sn, sv, st ^ 1);
          else issue(p + 1, sn, pass_seg(P, sn), st ^ 1);   // the next segment's first piece
        } else if constexpr (kQ8) {
          cp_async_commit();   // keep one group per piece
        }
        if (seg_first[seg + 1] <= p) {
          finish_run(p);
          seg = seg_of(p, seg);
          sv = pass_seg(P, seg);
          load_consts();
          run_first = p;
        }
        const int r0 = (p - seg_first[seg]) * P.piece_rows;
        const int rows = min(P.piece_rows, sv.n - r0);
        if (!mbar_wait_bounded(&bars[st], (uint32_t)((kp >> 1) & 1), P.spin_limit)) {
          if (lane == 0) report(P.ctrl, TRIA_ERR_TIMEOUT, (uint32_t)seg);
          // wait again (bounded) for the copies still in flight before leaving
          mbar_wait_bounded(&bars[st], (uint32_t)((kp >> 1) & 1), P.spin_limit);
          if (p + 1 < p_end) mbar_wait_bounded(&bars[st ^ 1], (uint32_t)(((kp + 1) >> 1) & 1), P.spin_limit);
          if constexpr (kQ8) cp_async_wait<0>();
          break;
        }
        if constexpr (kQ8) {
          cp_async_wait<1>();   // this piece's scales (the next piece's may still be in flight)
          __syncwarp();
        }
        body.template piece_t<S / 2>(ring + st * kPassPieceBytes, sc_ring + st * kPassScaleStage, rows, P.k_rb, P.ks_rb,
                   P.raw + (size_t)(sv.wrow0 + r0) * G);
        __syncwarp();
        if (p + 1 == p_end) finish_run(p_end);
      }
    }
  }
  __syncthreads();   // the ring is free from here on

  // ---- service: select scored segments; while none is waiting, move
  const MoveStage L = move_stage_layout(P.k_rb, P.ks_rb, P.v_rb, P.vs_rb);
  const bool mover = warp < min(kPassWarps, kPassRing / L.bytes);
  uint8_t* stg = smem + PassSmem::kRing + (size_t)warp * L.bytes;
  const uint32_t tag = flag_tag(s_epoch);
  if (n_active > 0) {
    int idle = 0;
    while (true) {
      if (tid == 0) {
        // -2: every segment is selected or being selected; -1: none waits now
        int sel = -1;
        const uint32_t h = ld_acquire_u32(&P.ctrl->sel_next);
        if ((int)h >= n_active) {
          sel = -2;
        } else if (h < ld_acquire_u32(&P.ctrl->scored_count)) {
          // a ticket in the scored list; taken past the scored count only in
          // a race with other CTAs, when its segment is being scored now
          // (bounded wait for the slot)
          const uint32_t t = atomicAdd(&P.ctrl->sel_next, 1u);
          if ((int)t >= n_active) {
            sel = -2;
          } else {
            const uint32_t* q = reinterpret_cast<const uint32_t*>(P.ctl->scored + t);
            uint32_t e = 0;
            for (int it = 0; it < P.spin_limit && (e = ld_acquire_u32(q)) == 0u; ++it) __nanosleep(64);
            if (e == 0u) report(P.ctrl, TRIA_ERR_TIMEOUT, 0xC0000000u);
            sel = e == 0u ? -1 : (int)e - 1;
          }
        }
        s_sel = sel;
      }
      __syncthreads();
      const int sel = s_sel;
      if (sel >= 0) {
        idle = 0;
        __threadfence();
        const int nr = segment_runs(seg_first[sel], seg_first[sel + 1], per);
        if (pass_seg(P, sel).n <= kPassSmemKeys)
          pass_select<G, true>(P, sel, nr, reinterpret_cast<uint32_t*>(smem + PassSmem::kRing), hist);
        else
          pass_select<G, false>(P, sel, nr, reinterpret_cast<uint32_t*>(smem + PassSmem::kRing), hist);
        continue;
      }
      if (sel == -2) break;
      // no segment waits for selection: when a ready segment may still have
      // blocks (thread 0 checks, so idle CTAs poll with one thread), each
      // warp moves at most one block
      if (tid == 0) s_sel = ld_acquire_u32(&P.ctrl->move_cursor) < ld_acquire_u32(&P.ctrl->ready_count) ? 1 : 0;
      __syncthreads();
      int moved = 0;
      if (mover && s_sel) {
        int last_sg = -1;
        const MoveClaim m = pass_claim(P, n_active, last_sg);
        if (m.state == 0) {
          const MoveWork w = pass_gather(P, m, stg, s_src[warp]);
          cp_async_wait<0>();
          __syncwarp();
          pass_store(P, m, w, stg, s_src[warp], tag);
          moved = 1;
        }
        if (lane == 0) bulk_wait_read_all();   // the stage may hold keys next
      }
      if (__syncthreads_or(moved)) {
        idle = 0;
      } else {
        if (++idle > P.spin_limit) {
          if (tid == 0) report(P.ctrl, TRIA_ERR_TIMEOUT, 0xB0000001u);
          break;
        }
        __nanosleep(min(4096, 128 << min(idle, 5)));   // back off: idle CTAs poll rarely
      }
    }
    if (mover && lane == 0) bulk_wait_all();   // the stores of the service loop
    // the ring barriers are done with: their words become move stages
    if (lane == 0) {
      mbar_inval(&bars[0]);
      mbar_inval(&bars[1]);
    }
    // every segment is selected (each CTA finished its selects before here):
    // the moves left, in k_move's order
    __shared__ int s_span;
    if (tid == 0) s_span = 0;
    pass_grid_barrier(P);
    for (int slot = tid; slot < n_active; slot += blockDim.x) {
      const int sg = __ldcg(P.ctl->ready + slot) - 1;
      if (sg < 0 || sg >= P.n_seg) continue;
      const int nb = (P.seq[(sg % (P.n_seqs * P.n_kv)) / P.n_kv].budget + kChunk - 1) / kChunk;
      atomicMax(&s_span, nb - min(nb, __ldcg(P.ctl->move_next + sg)));
    }
    __syncthreads();
    pass_moves_final(P, stg, s_src[warp], tag, n_active, min(kPassWarps, P.dyn_bytes / L.bytes), s_span);
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
  for (int sg = tid; sg < P.n_seg; sg += blockDim.x) {
    P.ctl->ready[sg] = 0;
    P.ctl->scored[sg] = 0;
    P.ctl->pieces_done[sg] = 0;
    P.ctl->move_next[sg] = 0;
  }
  __syncthreads();
  if (tid == 0) {
    P.ctrl->scored_count = 0u;
    P.ctrl->sel_next = 0u;
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

cudaError_t launch_pass_f16(FPass& P, cudaStream_t st);   // pass_f16.cu
cudaError_t launch_pass_q8(FPass& P, cudaStream_t st);    // pass_q8.cu

// Sets P.dyn_bytes: the dynamic shared memory of the launch, kPassDynBytes
// or what the kernel's static shared memory leaves of the per-block limit
// (at least the scoring layout's).
template <int KT, int G, int S>
cudaError_t launch_pass_t(FPass& P, cudaStream_t st) {
  auto kern = k_pass<KT, G, S>;
  static int grid = 0, dyn = 0;
  if (grid == 0) {
    int dev = 0, sms = 0, per_sm = 0, optin = 0;
    cudaFuncAttributes fa{};
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    int d = optin - (int)fa.sharedSizeBytes;
    d = (d < kPassDynBytes ? d : kPassDynBytes) & ~127;
    if (d < PassSmem::kBytes) return cudaErrorInvalidConfiguration;
    e = set_smem_attrs(kern, d);
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kPassThreads, d);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    dyn = d;
    grid = sms;   // one CTA per SM
  }
  P.dyn_bytes = dyn;
  void* args[] = {&P};
  return cudaLaunchCooperativeKernel((const void*)kern, dim3(grid), dim3(kPassThreads), args, (size_t)dyn, st);
}

template <int KT>
cudaError_t launch_pass_k(FPass& P, cudaStream_t st) {
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
