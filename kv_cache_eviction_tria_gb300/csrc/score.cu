// Score stage: raw per-query-head scores, per-segment moments, z-max score.
//
// [Worklog] "TriAttention Native C++ Worklog", Phase 9 (the score is taken on
// the stored rotated keys: the calibrated mean query times the conjugate key,
// the rotation applied on the query side only, plus a norm term on the keys'
// magnitudes) and 2026-04-18 (phases from the absolute decode position).
// [Doc] "TriAttention KV-Cache Eviction (--triattention)", §5 Phase C
// (z-normalise each query head, then max over the GQA group).
//
// Per row r and query head h of the segment's group:
//   raw_h(r) = sum_f  Wr_{h,f} K[r][f] + Wi_{h,f} K[r][f+fc] + M_{h,f} |k_f|
// with W = qbar E_f e^{i w_f p} and M = q_abs - |qbar|.
//
// Work layout (persistent, one CTA per SM): the live rows of all segments are
// cut into pieces of at most 8 KB of keys; the pieces, in segment order, are
// split into equal contiguous runs, one per warp. Each warp streams its run
// through a private two-stage ring in shared memory: lane 0 starts the bulk
// async copy (TMA, non-tensor form, completion on an mbarrier) of piece i+1
// before the warp computes piece i. A row is handled by TPR lanes; lane q owns
// the PPT frequency pairs [q*PPT, q*PPT+PPT) of every head of the group, with
// its slice of W and M in registers, and works on pairs of consecutive
// frequencies with packed fp32x2 FMAs. The TPR partial sums are combined with a
// transposed shuffle reduction (each step halves the heads a lane carries).
//
// Moments: each lane keeps shifted sums of the heads it ends up owning; a warp
// merges them (Chan et al. pairwise update) into one partial per contiguous
// run of a segment, stored in the segment's run table (row = run index); the
// consumer merges the runs into mean and 1 / (std + 1e-6).
#include "tria_internal.cuh"

namespace tria {

constexpr int kScoreWarps = 12;
constexpr int kScoreThreads = kScoreWarps * 32;
constexpr int kPieceBytes = 8192;
constexpr int kMaxSegs = 1024;
constexpr int kMomTable = kScoreWarps * 32 * 2 * (12 + 4);   // per-warp [lane][slot] moments + head
// q8_0 block scales of a piece (rows x head_dim / 16 bytes <= piece bytes / 16)
constexpr int kScaleStage = kPieceBytes / 16;
constexpr int kScaleRing = kScoreWarps * 2 * kScaleStage;
constexpr int kScoreSmemMax =
    kScoreWarps * 2 * kPieceBytes + kScoreWarps * 2 * 8 + 2 * (kMaxSegs + 1) * 4 + kMomTable + kScaleRing + 16;

// After a wait that gave up: wait again, bounded, for the copies this warp
// still has in flight (piece k in stage st and, if issued, piece k + 1 in the
// other stage), so that the warp does not leave while a bulk copy may still
// write its shared memory.
__device__ __forceinline__ void drain_ring(uint64_t* bars, int st, int k, bool next_issued, int limit) {
  mbar_wait_bounded(&bars[st], (uint32_t)((k >> 1) & 1), limit);
  if (next_issued) mbar_wait_bounded(&bars[st ^ 1], (uint32_t)(((k + 1) >> 1) & 1), limit);
}

__device__ __forceinline__ float sqrt_approx(float x) {
  float y;
  asm("sqrt.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Loads PPT consecutive elements of one NEOX half as PPT/2 float2 (consecutive pairs).
template <int KT, int PPT>
struct Loader;

template <int PPT>
struct Loader<TRIA_F16, PPT> {
  static __device__ __forceinline__ void half(const uint8_t* row, int e0, float2* x) {
    if constexpr (PPT == 8) {
      const uint4 u = *reinterpret_cast<const uint4*>(row + 2 * e0);
      const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
      for (int i = 0; i < 4; ++i) x[i] = __half22float2(h[i]);
    } else {
      const uint2 u = *reinterpret_cast<const uint2*>(row + 2 * e0);
      const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
      for (int i = 0; i < 2; ++i) x[i] = __half22float2(h[i]);
    }
  }
};

template <int PPT>
struct Loader<TRIA_F32, PPT> {
  static __device__ __forceinline__ void half(const uint8_t* row, int e0, float2* x) {
    const float4* p = reinterpret_cast<const float4*>(row + 4 * e0);
#pragma unroll
    for (int i = 0; i < PPT / 4; ++i) {
      const float4 v = p[i];
      x[2 * i] = make_float2(v.x, v.y);
      x[2 * i + 1] = make_float2(v.z, v.w);
    }
  }
};

template <int PPT>
struct Loader<TRIA_Q8_0, PPT> {
  static __device__ __forceinline__ void half(const uint8_t* row, int e0, float2* x) {
    if constexpr (PPT == 8) {
      const uint2 u = *reinterpret_cast<const uint2*>(row + e0);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        x[i] = make_float2((float)(int8_t)(u.x >> (16 * i)), (float)(int8_t)(u.x >> (16 * i + 8)));
        x[2 + i] = make_float2((float)(int8_t)(u.y >> (16 * i)), (float)(int8_t)(u.y >> (16 * i + 8)));
      }
    } else {
      const uint32_t u = *reinterpret_cast<const uint32_t*>(row + e0);
#pragma unroll
      for (int i = 0; i < 2; ++i)
        x[i] = make_float2((float)(int8_t)(u >> (16 * i)), (float)(int8_t)(u >> (16 * i + 8)));
    }
  }
};

// Transposed reduction of NV partial sums over the TPR lanes of a row group:
// each step with more than one value left sends half of them to the partner
// lane and keeps the other half; once a lane carries one value the rest is a
// butterfly. Afterwards the lane holds the full sums of the flattened values
// [base, base + kOut) in v[0 .. kOut); `writer` is false on butterfly duplicates.
template <int NV, int TPR>
struct HeadReduce {
  static constexpr int kOut = NV >= TPR ? NV / TPR : 1;
  static __device__ __forceinline__ int run(float (&v)[NV], int q, bool& writer) {
    int base = 0;
    writer = true;
    int m = NV;
#pragma unroll
    for (int span = TPR / 2; span >= 1; span >>= 1) {
      if (m > 1) {
        const int half = m / 2;
        const bool upper = (q & span) != 0;
#pragma unroll
        for (int i = 0; i < (NV > 1 ? NV / 2 : 1); ++i) {
          if (i < half) {
            const float send = upper ? v[i] : v[i + half];
            const float keep = upper ? v[i + half] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, span);
          }
        }
        if (upper) base += half;
        m = half;
      } else {
        v[0] += __shfl_xor_sync(0xffffffffu, v[0], span);
        if (q & span) writer = false;
      }
    }
    return base;
  }
};

// Compile-time shape of the row batch a lane accumulates before one reduction.
template <int KT, int G, int TPR, int PPT>
struct Batch {
  static constexpr int kElem = KT == TRIA_F32 ? 4 : (KT == TRIA_F16 ? 2 : 1);
  static constexpr int kRowsPerStep = 32 / TPR;
  static constexpr int kRbMax = kElem * 2 * TPR * PPT;   // key bytes of the widest row
  static constexpr int kPieceRows = (kPieceBytes / kRbMax) > 64 ? 64 : (kPieceBytes / kRbMax);
  static constexpr int kSteps = (kPieceRows / kRowsPerStep) > 0 ? (kPieceRows / kRowsPerStep) : 1;
  static constexpr int kTarget = TPR / G > 0 ? TPR / G : 1;   // NV = TPR: no butterfly duplicates
  static constexpr int kRowsB = kTarget < kSteps ? kTarget : kSteps;   // rows per lane per batch
  static constexpr int kNV = kRowsB * G;
};

struct ScoreGeom {
  int R;       // rows per piece
  int stage;   // bytes per ring stage
};

__host__ __device__ inline ScoreGeom score_geom(int k_rb) {
  ScoreGeom g;
  g.R = kPieceBytes / k_rb;
  if (g.R > 64) g.R = 64;
  if (g.R >= 16) g.R &= ~15;   // whole 16-row tiles for the tensor-core body
  if (g.R < 1) g.R = 1;
  g.stage = (g.R * k_rb + 15) & ~15;
  return g;
}

__host__ __device__ inline int score_smem_bytes_for(int k_rb) {
  const ScoreGeom g = score_geom(k_rb);
  return kScoreWarps * 2 * g.stage + kScoreWarps * 2 * 8 + 2 * (kMaxSegs + 1) * 4 + kMomTable + kScaleRing + 16;
}

// Ask L2 for the weight inputs of the first sequence's layer (qbar E, M, turn
// factors: a few tens of KB) before the key stream starts, so that the warps' weight loads hit L2
// instead of queueing in DRAM behind the first pieces. Lines are dealt over
// all threads of the grid.
__device__ __forceinline__ void prefetch_layer_stats(const Pass& P) {
  const size_t n = (size_t)P.n_kv * P.G * P.fc;
  const size_t lines_qe = (n * sizeof(float2) + 127) / 128, lines_mw = (n * sizeof(float) + 127) / 128,
               lines_t = ((size_t)P.fc * 8 + 127) / 128;
  const size_t total = lines_qe + lines_mw + lines_t;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
    const char* a = i < lines_qe ? reinterpret_cast<const char*>(P.qe + P.seq[0].qe_off) + 128 * i
                    : i < lines_qe + lines_mw ? reinterpret_cast<const char*>(P.mw + P.seq[0].qe_off) + 128 * (i - lines_qe)
                                              : reinterpret_cast<const char*>(P.turns) + 128 * (i - lines_qe - lines_mw);
    asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
  }
}

// Segment tables (first piece and live rows of every scored segment, pieces
// in segment order, skipped segments have none), the piece layout that the
// consumer of the moment partials needs (CTA 0), and this warp's two ring
// barriers. Called by every thread of the CTA.
__device__ __forceinline__ void score_prologue(const Pass& P, const ScoreGeom& geo, int* seg_first, int* seg_rows,
                                               uint64_t* bars, int lane) {
  // thread t counts segments [t*per_t, t*per_t + per_t), then a block scan
  {
    __shared__ int sbuf[40];
    const int per_t = (P.n_seg + kScoreThreads - 1) / kScoreThreads;
    const int sb = min(P.n_seg, (int)threadIdx.x * per_t), se = min(P.n_seg, sb + per_t);
    int cnt[(kMaxSegs + kScoreThreads - 1) / kScoreThreads];
    int local = 0;
#pragma unroll
    for (int i = 0; i < (kMaxSegs + kScoreThreads - 1) / kScoreThreads; ++i) {
      cnt[i] = 0;
      const int s = sb + i;
      if (s < se) {
        const SegView v = seg_view(P, s);
        if (!v.valid) {
          if (blockIdx.x == 0 && v.g == 0) report(P.ctrl, TRIA_ERR_DEVICE_ARG, (uint32_t)v.s);
        } else if (!P.only_active || v.active) {
          cnt[i] = (v.n + geo.R - 1) / geo.R;
        }
        seg_rows[s] = cnt[i] ? v.n : 0;
        local += cnt[i];
      }
    }
    int tot;
    int before = block_exclusive_scan(local, &tot, sbuf);
#pragma unroll
    for (int i = 0; i < (kMaxSegs + kScoreThreads - 1) / kScoreThreads; ++i) {
      const int s = sb + i;
      if (s < se) {
        seg_first[s] = before;
        before += cnt[i];
      }
    }
    if (threadIdx.x == 0) seg_first[P.n_seg] = tot;
  }
  __syncthreads();
  // the consumer of the moment partials needs the piece layout
  if (blockIdx.x == 0) {
    const int nw = gridDim.x * kScoreWarps;
    for (int s = threadIdx.x; s < P.n_seg; s += blockDim.x) {
      P.seg[s].piece_first = seg_first[s];
      P.seg[s].piece_end = seg_first[s + 1];
      P.seg[s].piece_per = (seg_first[P.n_seg] + nw - 1) / nw;
    }
  }
  if (lane == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_mbar_init();
  }
  __syncthreads();
}

template <int KT, int G, int TPR, int PPT>
__global__ void __launch_bounds__(kScoreThreads, 1) k_score(const __grid_constant__ Pass P) {
  static_assert(PPT % 2 == 0, "pairs of frequencies");
  static_assert(HeadReduce<Batch<KT, G, TPR, PPT>::kNV, TPR>::kOut <= 2, "moment table holds 2 slots");
  using BT = Batch<KT, G, TPR, PPT>;
  constexpr int kRowsPerStep = BT::kRowsPerStep;
  constexpr int kRowsB = BT::kRowsB;
  constexpr int kNV = BT::kNV;
  using Red = HeadReduce<kNV, TPR>;
  constexpr int kOut = Red::kOut;

  extern __shared__ __align__(128) uint8_t smem[];
  const ScoreGeom geo = score_geom(P.k_rb);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* ring = smem + (size_t)warp * 2 * geo.stage;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)kScoreWarps * 2 * geo.stage) + warp * 2;
  int* seg_first = reinterpret_cast<int*>(smem + (size_t)kScoreWarps * 2 * geo.stage + kScoreWarps * 2 * 8);
  int* seg_rows = seg_first + (kMaxSegs + 1);   // live rows of each scored segment

  prefetch_layer_stats(P);
  score_prologue(P, geo, seg_first, seg_rows, bars, lane);

  const int total = seg_first[P.n_seg];
  const int nwarps = gridDim.x * kScoreWarps;
  const int per = (total + nwarps - 1) / nwarps;
  const int gw = blockIdx.x * kScoreWarps + warp;
  const int p_beg = min(total, gw * per), p_end = min(total, p_beg + per);
  if (p_beg >= p_end) return;

  auto seg_of = [&](int p, int from) {
    int s = from;
    while (seg_first[s + 1] <= p) ++s;
    return s;
  };
  // lane 0: start the bulk copy of piece p (segment sg) into ring stage `stage_i`
  auto seg_row0 = [&](int sg) {
    const int sq = sg / P.n_kv;
    return P.seq[sq].row0 + (int64_t)(sg - sq * P.n_kv) * P.seq[sq].cap;
  };
  auto issue = [&](int p, int sg, int stage_i) {
    const int r = (p - seg_first[sg]) * geo.R;
    const int rows = min(geo.R, seg_rows[sg] - r);
    const uint32_t bytes = (uint32_t)(rows * P.k_rb);
    mbar_arrive_expect_tx(&bars[stage_i], bytes);
    bulk_g2s(ring + stage_i * geo.stage, P.k + (size_t)(seg_row0(sg) + r) * P.k_rb, bytes, &bars[stage_i]);
  };

  const int q = lane % TPR;
  const int f0 = q * PPT;
  const int fc = P.fc;
  const bool lane_on = f0 < fc;

  // this lane's slice of W (real / imaginary) and M for the current segment,
  // on pairs of consecutive frequencies
  float2 wr[G][PPT / 2], wi[G][PPT / 2], wm[G][PPT / 2];
  auto load_consts = [&](const SegView& v) {
    const unsigned long long p = (unsigned long long)P.seq[v.s].cur_pos;
    float cs[PPT], sn[PPT];
#pragma unroll
    for (int j = 0; j < PPT; ++j) {
      if (lane_on) {
        const unsigned long long x = P.turns[f0 + j] * p;   // exact turn fraction of w_f * p
        sincospif((float)(int)(x >> 32) * 0x1p-31f, &sn[j], &cs[j]);
      } else {
        sn[j] = 0.f;
        cs[j] = 0.f;
      }
    }
    const float2* qe = P.qe + P.seq[v.s].qe_off + (size_t)v.g * G * fc;
    const float* mw = P.mw + P.seq[v.s].qe_off + (size_t)v.g * G * fc;
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int j = 0; j < PPT; j += 2) {
        float2 a = make_float2(0.f, 0.f), b = make_float2(0.f, 0.f), m = make_float2(0.f, 0.f);
        if (lane_on) {
          a = qe[h * fc + f0 + j];
          b = qe[h * fc + f0 + j + 1];
          m = make_float2(mw[h * fc + f0 + j], mw[h * fc + f0 + j + 1]);
        }
        wr[h][j / 2] = make_float2(a.x * cs[j] - a.y * sn[j], b.x * cs[j + 1] - b.y * sn[j + 1]);
        wi[h][j / 2] = make_float2(a.x * sn[j] + a.y * cs[j], b.x * sn[j + 1] + b.y * cs[j + 1]);
        wm[h][j / 2] = m;
      }
  };

  int seg = seg_of(p_beg, 0);
  if (lane == 0) issue(p_beg, seg, 0);
  SegView sv = seg_view(P, seg);
  load_consts(sv);

  // flattened (row, head) values this lane owns after the reduction: constant
  // per lane, so slot o always carries head (vbase + o) % G
  bool writer = true;
  int vbase = 0;
  {
    float dummy[kNV];
#pragma unroll
    for (int i = 0; i < kNV; ++i) dummy[i] = 0.f;
    vbase = Red::run(dummy, q, writer);
  }
  Mom* mtab = reinterpret_cast<Mom*>(seg_rows + (kMaxSegs + 1)) + warp * 32 * 2;
  int* mhead = reinterpret_cast<int*>(reinterpret_cast<Mom*>(seg_rows + (kMaxSegs + 1)) + kScoreWarps * 32 * 2) +
               warp * 32 * 2;

  Mom run_m[kOut];
#pragma unroll
  for (int o = 0; o < kOut; ++o) run_m[o] = Mom{0.f, 0.f, 0.f};
  int run_first = p_beg;   // global index of the run's first piece

  auto flush_run = [&]() {
    // every lane lists its slots (head, moments); lane h < G merges the
    // entries of head h in lane-major order
#pragma unroll
    for (int o = 0; o < kOut; ++o) {
      mtab[lane * kOut + o] = writer ? run_m[o] : Mom{0.f, 0.f, 0.f};
      mhead[lane * kOut + o] = (vbase + o) % G;
    }
    __syncwarp();
    if (lane < G) {
      Mom a{0.f, 0.f, 0.f};
      for (int e = 0; e < 32 * kOut; ++e)
        if (mhead[e] == lane) a = mom_merge(a, mtab[e]);
      float* tab = run_table(P, seg);
      const int r = run_index(run_first, seg_first[seg], per);
      tab[(1 + lane) * P.cs_max + r] = a.mean;
      tab[(1 + kMaxG + lane) * P.cs_max + r] = a.m2;
      if (lane == 0) tab[r] = a.n;
    }
#pragma unroll
    for (int o = 0; o < kOut; ++o) run_m[o] = Mom{0.f, 0.f, 0.f};
  };

  for (int p = p_beg; p < p_end; ++p) {
    const int k = p - p_beg;
    const int st = k & 1;
    // next piece into the other stage (its previous contents were consumed)
    if (p + 1 < p_end && lane == 0) issue(p + 1, seg_of(p + 1, seg), st ^ 1);
    if (seg_first[seg + 1] <= p) {
      flush_run();
      seg = seg_of(p, seg);
      sv = seg_view(P, seg);
      load_consts(sv);
      run_first = p;
    }
    const int r0 = (p - seg_first[seg]) * geo.R;
    const int rows = min(geo.R, seg_rows[seg] - r0);
    const int64_t grow = seg_row0(seg) + r0;
    if (!mbar_wait_bounded(&bars[st], (uint32_t)((k >> 1) & 1), P.spin_limit)) {
      if (lane == 0) report(P.ctrl, TRIA_ERR_TIMEOUT, (uint32_t)seg);
      drain_ring(bars, st, k, p + 1 < p_end, P.spin_limit);
      return;
    }
    const uint8_t* buf = ring + st * geo.stage;
    // lane-local shifted sums of this piece for my value slots
    float shift[kOut], s1[kOut], s2[kOut], cnt[kOut];
#pragma unroll
    for (int o = 0; o < kOut; ++o) shift[o] = s1[o] = s2[o] = cnt[o] = 0.f;
    const int steps = (rows + kRowsPerStep - 1) / kRowsPerStep;
    const int gi = lane / TPR;   // row group of this lane
    for (int b0 = 0; b0 < steps; b0 += kRowsB) {
      float v[kNV];
#pragma unroll
      for (int rb = 0; rb < kRowsB; ++rb) {
        const int rr = (b0 + rb) * kRowsPerStep + gi;
        float2 kr[PPT / 2], ki[PPT / 2];
        if (rr < rows && lane_on) {
          const uint8_t* row = buf + (size_t)rr * P.k_rb;
          Loader<KT, PPT>::half(row, f0, kr);
          Loader<KT, PPT>::half(row, fc + f0, ki);
          if constexpr (KT == TRIA_Q8_0) {
            const __half* sc = reinterpret_cast<const __half*>(P.ks + (size_t)(grow + rr) * P.ks_rb);
            const float d1 = __half2float(sc[f0 >> 5]);
            const float d2 = __half2float(sc[(fc + f0) >> 5]);
#pragma unroll
            for (int j = 0; j < PPT / 2; ++j) {
              kr[j] = __fmul2_rn(kr[j], make_float2(d1, d1));
              ki[j] = __fmul2_rn(ki[j], make_float2(d2, d2));
            }
          }
        } else {
#pragma unroll
          for (int j = 0; j < PPT / 2; ++j) kr[j] = ki[j] = make_float2(0.f, 0.f);
        }
        float2 mag[PPT / 2];
#pragma unroll
        for (int j = 0; j < PPT / 2; ++j) {
          const float2 sq = __ffma2_rn(ki[j], ki[j], __fmul2_rn(kr[j], kr[j]));
          mag[j] = make_float2(sqrt_approx(sq.x), sqrt_approx(sq.y));
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
          // two independent accumulation chains per head
          float2 a0 = __fmul2_rn(wr[h][0], kr[0]);
          float2 a1 = __fmul2_rn(wi[h][0], ki[0]);
          a0 = __ffma2_rn(wm[h][0], mag[0], a0);
#pragma unroll
          for (int j = 1; j < PPT / 2; ++j) {
            a0 = __ffma2_rn(wr[h][j], kr[j], a0);
            a1 = __ffma2_rn(wi[h][j], ki[j], a1);
            if (j & 1)
              a1 = __ffma2_rn(wm[h][j], mag[j], a1);
            else
              a0 = __ffma2_rn(wm[h][j], mag[j], a0);
          }
          v[rb * G + h] = (a0.x + a1.x) + (a0.y + a1.y);
        }
      }
      bool wr_lane;
      Red::run(v, q, wr_lane);
      if (wr_lane) {
#pragma unroll
        for (int o = 0; o < kOut; ++o) {
          const int idx = vbase + o;
          const int rr = (b0 + idx / G) * kRowsPerStep + gi;
          if (rr < rows) {
            P.raw[(size_t)(grow + rr) * G + (idx % G)] = v[o];
            if (cnt[o] == 0.f) shift[o] = v[o];
            const float d = v[o] - shift[o];
            s1[o] += d;
            s2[o] = fmaf(d, d, s2[o]);
            cnt[o] += 1.f;
          }
        }
      }
    }
    // this piece's moments (lane-local) -> the run's moments
#pragma unroll
    for (int o = 0; o < kOut; ++o) {
      Mom b;
      b.n = cnt[o];
      const float mean_d = cnt[o] > 0.f ? __fdividef(s1[o], cnt[o]) : 0.f;
      b.mean = shift[o] + mean_d;
      b.m2 = fmaxf(s2[o] - s1[o] * mean_d, 0.f);
      run_m[o] = mom_merge(run_m[o], b);
    }
    __syncwarp();
  }
  flush_run();
}

// z-max score per live row: s = max_h (raw_h - mu_h) * inv_h, with the
// segment's moments merged from the run partials by each block.
template <int G>
__global__ void __launch_bounds__(kThreads) k_zscore(const __grid_constant__ Pass P) {
  const int seg = blockIdx.y;
  const SegView sv = seg_view(P, seg);
  if (!sv.valid || (P.only_active && !sv.active)) return;
  if ((int)blockIdx.x * 1024 >= sv.n) return;
  float mu[G], inv[G];
  block_segment_moments<G>(P, seg, mu, inv);
  const int r_end = min(sv.n, (int)(blockIdx.x + 1) * 1024);
  for (int r = blockIdx.x * 1024 + threadIdx.x; r < r_end; r += blockDim.x) {
    const float* rp = P.raw + (size_t)(sv.row0 + r) * G;
    float s = (rp[0] - mu[0]) * inv[0];
#pragma unroll
    for (int h = 1; h < G; ++h) s = fmaxf(s, (rp[h] - mu[h]) * inv[h]);
    P.score[sv.row0 + r] = s;
  }
}

// ---------------------------------------------------------------------------
// Tensor-core body (fp16 keys, head_dim a multiple of 64).
//
// The phase term sum_f Wr K[f] + Wi K[f+fc] is a contraction of the key rows
// with a [head_dim x heads] weight matrix, and the keys are exact in fp16: it
// runs as m16n8k16 MMAs (fp32 accumulation) against W split into an fp16 high
// part and an fp16 remainder, scaled per head by a power of two so that both
// parts are normal. The magnitude term sum_f M |k_f| is formed in fp32 from
// the same key fragments and contracted with M by m16n8k8 tf32 MMAs, again on
// a high part and its remainder. The columns of one n-tile are [high parts of
// the G heads, remainders of the G heads], so a head's score is the sum of two
// accumulator columns: fp32-level accuracy from half-precision operands.
//
// A warp computes 16 rows (one m-tile) at a time. Lane (g, q) = (lane / 4,
// lane % 4) reads 16-byte granule q of the 64-byte step s of rows g and g + 8;
// the MMA k-slots are mapped to the granule's elements (the same map in A and
// B, which a contraction is free to permute), so no transposing load is
// needed. Real and imaginary parts of a frequency sit in steps s and
// s + S/2 at the same lane and register position.
// ---------------------------------------------------------------------------

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_tf32(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t to_tf32(float x) {
  uint32_t y;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Four signed 8-bit values (one 32-bit word) as two fp16 pairs, exactly: with
// u = x + 128 in a byte, the fp16 bit pattern 0x6400 | u is 1024 + u, and
// subtracting 1152 leaves x (both steps exact in fp16).
__device__ __forceinline__ void i8x4_to_h2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  const uint32_t a = __byte_perm(u, 0x64646464u, 0x4140u);
  const uint32_t b = __byte_perm(u, 0x64646464u, 0x4342u);
  const __half2 bias = __halves2half2(__ushort_as_half((unsigned short)0x6480u), __ushort_as_half((unsigned short)0x6480u));
  const __half2 ha = __hsub2(*reinterpret_cast<const __half2*>(&a), bias);
  const __half2 hb = __hsub2(*reinterpret_cast<const __half2*>(&b), bias);
  lo = *reinterpret_cast<const uint32_t*>(&ha);
  hi = *reinterpret_cast<const uint32_t*>(&hb);
}

// |k| of 8 frequencies from fp16 pairs of block values times their scales:
// real parts r * dr, imaginary parts i * di
__device__ __forceinline__ void q8_mag(const uint32_t* r, const uint32_t* i, float dr, float di, float* m) {
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const float2 a = __fmul2_rn(__half22float2(*reinterpret_cast<const __half2*>(&r[t])), make_float2(dr, dr));
    const float2 b = __fmul2_rn(__half22float2(*reinterpret_cast<const __half2*>(&i[t])), make_float2(di, di));
    const float2 sq = __ffma2_rn(b, b, __fmul2_rn(a, a));
    m[2 * t] = sqrt_approx(sq.x);
    m[2 * t + 1] = sqrt_approx(sq.y);
  }
}

// |k| of the 8 frequencies of one granule: real parts r, imaginary parts i
__device__ __forceinline__ void granule_mag(const uint4& r, const uint4& i, float* m) {
  const uint32_t rr[4] = {r.x, r.y, r.z, r.w}, ii[4] = {i.x, i.y, i.z, i.w};
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&rr[t]));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&ii[t]));
    const float2 sq = __ffma2_rn(b, b, __fmul2_rn(a, a));
    m[2 * t] = sqrt_approx(sq.x);
    m[2 * t + 1] = sqrt_approx(sq.y);
  }
}

template <int G, int S>
struct TcShape {
  static constexpr int NT = (2 * G + 7) / 8;   // n-tiles: G high-part columns, then G remainder columns
  static constexpr bool kOk = S % 2 == 0 && NT * S <= 8;
};

template <int KT, int G, int S>
__global__ void __launch_bounds__(kScoreThreads, 1) k_score_tc(const __grid_constant__ Pass P) {
  static_assert(KT == TRIA_F16 || KT == TRIA_Q8_0, "fp16 or q8_0 keys");
  constexpr bool kQ8 = KT == TRIA_Q8_0;
  using SH = TcShape<G, S>;
  constexpr int NT = SH::NT;
  constexpr int FC = 16 * S;   // frequency pairs (head_dim / 2)
  static_assert(SH::kOk, "tensor-core body shape");

  extern __shared__ __align__(128) uint8_t smem[];
  const ScoreGeom geo = score_geom(P.k_rb);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* ring = smem + (size_t)warp * 2 * geo.stage;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)kScoreWarps * 2 * geo.stage) + warp * 2;
  int* seg_first = reinterpret_cast<int*>(smem + (size_t)kScoreWarps * 2 * geo.stage + kScoreWarps * 2 * 8);
  int* seg_rows = seg_first + (kMaxSegs + 1);

  // q8_0: this warp's two stages of block scales, after the moment table
  uint8_t* sc_ring = smem + (size_t)kScoreWarps * 2 * geo.stage + kScoreWarps * 2 * 8 + 2 * (kMaxSegs + 1) * 4 +
                     kMomTable + (size_t)warp * 2 * kScaleStage;

  prefetch_layer_stats(P);
  // turn factors of the frequencies: loaded here so that their latency
  // overlaps the prologue's, kept in shared memory (the moment-table area,
  // which this body does not use)
  static_assert(FC <= kScoreThreads, "one frequency per thread");
  const unsigned long long my_turn = (int)threadIdx.x < FC ? __ldg(P.turns + threadIdx.x) : 0ull;
  score_prologue(P, geo, seg_first, seg_rows, bars, lane);
  unsigned long long* s_turns = reinterpret_cast<unsigned long long*>(seg_rows + (kMaxSegs + 1));
  if ((int)threadIdx.x < FC) s_turns[threadIdx.x] = my_turn;
  __syncthreads();

  const int total = seg_first[P.n_seg];
  const int nwarps = gridDim.x * kScoreWarps;
  const int per = (total + nwarps - 1) / nwarps;
  const int gw = blockIdx.x * kScoreWarps + warp;
  const int p_beg = min(total, gw * per), p_end = min(total, p_beg + per);
  if (p_beg >= p_end) return;

  auto seg_of = [&](int p, int from) {
    int sg = from;
    while (seg_first[sg + 1] <= p) ++sg;
    return sg;
  };
  auto seg_row0 = [&](int sg) {
    const int sq = sg / P.n_kv;
    return P.seq[sq].row0 + (int64_t)(sg - sq * P.n_kv) * P.seq[sq].cap;
  };
  auto issue = [&](int p, int sg, int stage_i) {
    const int r = (p - seg_first[sg]) * geo.R;
    const int rows = min(geo.R, seg_rows[sg] - r);
    const uint32_t bytes = (uint32_t)(rows * P.k_rb);
    mbar_arrive_expect_tx(&bars[stage_i], bytes);
    bulk_g2s(ring + stage_i * geo.stage, P.k + (size_t)(seg_row0(sg) + r) * P.k_rb, bytes, &bars[stage_i]);
  };
  // q8_0, all lanes: the block scales of piece p (rows x head_dim / 16 bytes,
  // 4-byte async copies), one commit group per piece
  auto issue_scales = [&](int p, int sg, int stage_i) {
    const int r = (p - seg_first[sg]) * geo.R;
    const int rows = min(geo.R, seg_rows[sg] - r);
    const uint8_t* src = P.ks + (size_t)(seg_row0(sg) + r) * P.ks_rb;
    uint8_t* dst = sc_ring + stage_i * kScaleStage;
    for (int u = lane; u < rows * P.ks_rb / 4; u += 32) cp_async4(dst + 4 * u, src + 4 * u);
    cp_async_commit();
  };

  const int g = lane >> 2, q = lane & 3;
  // this lane's output: heads (oh, oh + 1) (one head when G == 1) of one row
  // per m-tile (two rows when G == 8); with G <= 2 only lanes q < 2 write
  constexpr int kHeads = G >= 2 ? 2 : 1;
  const int oh = G == 8 ? 2 * q : (G == 4 ? 2 * (q & 1) : 0);
  const bool owriter = G >= 4 || q < 2;

  // B fragments of the current segment and the per-head unscaling factors.
  // Lane (g, q) builds column g of every n-tile, which belongs to head hl.
  const int hl = g < 2 * G ? g % G : 0;
  uint32_t bp[S][NT][4];            // phase weights, fp16 pairs
  uint32_t bm[S / 2][NT][4][2];     // magnitude weights, tf32
  float unscale[kHeads];
  auto load_consts = [&](const SegView& v) {
    const unsigned long long pos = (unsigned long long)P.seq[v.s].cur_pos;
    const float2* qe = P.qe + P.seq[v.s].qe_off + ((size_t)v.g * G + hl) * FC;
    const float* mw = P.mw + P.seq[v.s].qe_off + ((size_t)v.g * G + hl) * FC;
    // inputs of this lane's frequencies f = 32 s + 8 q + j (s < S / 2) of head
    // hl, all loaded up front
    float2 a[S / 2][8];
    float m[S / 2][8];
#pragma unroll
    for (int s2 = 0; s2 < S / 2; ++s2)
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int f = 32 * s2 + 8 * q + j;
        a[s2][j] = qe[f];
        m[s2][j] = mw[f];
      }
    // scale 2^e with max(|qbar E|, |M|) of the head (a bound of every weight,
    // since |Wr|, |Wi| <= |qbar E|) in [2^14, 2^15): both fp16 parts stay
    // normal; the four lanes of a column cover all frequencies
    float amax = 0.f;
#pragma unroll
    for (int s2 = 0; s2 < S / 2; ++s2)
#pragma unroll
      for (int j = 0; j < 8; ++j)
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(a[s2][j].x), fabsf(a[s2][j].y)), fabsf(m[s2][j])));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    int e = 0;
    if (amax > 0.f && amax < INFINITY) e = 14 - ilogbf(amax);
    e = max(-120, min(120, e));
    const float scale = __int_as_float((127 + e) << 23);
#pragma unroll
    for (int s2 = 0; s2 < S / 2; ++s2) {
      float wre_hi[8], wre_lo[8], wim_hi[8], wim_lo[8], wm_hi[8], wm_lo[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const unsigned long long x = s_turns[32 * s2 + 8 * q + j] * pos;   // exact turn fraction of w_f * p
        float sn, cs;
        sincospif((float)(int)(x >> 32) * 0x1p-31f, &sn, &cs);
        const float wr = (a[s2][j].x * cs - a[s2][j].y * sn) * scale;
        const float wi = (a[s2][j].x * sn + a[s2][j].y * cs) * scale;
        const float ms = m[s2][j] * scale;
        wre_hi[j] = __half2float(__float2half_rn(wr));
        wre_lo[j] = wr - wre_hi[j];
        wim_hi[j] = __half2float(__float2half_rn(wi));
        wim_lo[j] = wi - wim_hi[j];
        wm_hi[j] = __uint_as_float(to_tf32(ms));
        wm_lo[j] = ms - wm_hi[j];
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int c = 8 * nt + g;
        const bool live = c < 2 * G, rem = c >= G;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const float r0 = !live ? 0.f : (rem ? wre_lo[2 * t] : wre_hi[2 * t]);
          const float r1 = !live ? 0.f : (rem ? wre_lo[2 * t + 1] : wre_hi[2 * t + 1]);
          const float i0 = !live ? 0.f : (rem ? wim_lo[2 * t] : wim_hi[2 * t]);
          const float i1 = !live ? 0.f : (rem ? wim_lo[2 * t + 1] : wim_hi[2 * t + 1]);
          const float m0 = !live ? 0.f : (rem ? wm_lo[2 * t] : wm_hi[2 * t]);
          const float m1 = !live ? 0.f : (rem ? wm_lo[2 * t + 1] : wm_hi[2 * t + 1]);
          bp[s2][nt][t] = pack_f16x2(r0, r1);
          bp[s2 + S / 2][nt][t] = pack_f16x2(i0, i1);
          bm[s2][nt][t][0] = __float_as_uint(m0);
          bm[s2][nt][t][1] = __float_as_uint(m1);
        }
      }
    }
    // unscaling factors of the heads this lane writes: lane 4 h holds the
    // exponent of head h (column h of n-tile 0)
#pragma unroll
    for (int k = 0; k < kHeads; ++k) {
      const int eh = __shfl_sync(0xffffffffu, e, 4 * (oh + k));
      unscale[k] = __int_as_float((127 - eh) << 23);
    }
  };

  int seg = seg_of(p_beg, 0);
  if (lane == 0) issue(p_beg, seg, 0);
  if constexpr (kQ8) issue_scales(p_beg, seg, 0);
  SegView sv = seg_view(P, seg);
  load_consts(sv);

  Mom run_m[kHeads];
#pragma unroll
  for (int k = 0; k < kHeads; ++k) run_m[k] = Mom{0.f, 0.f, 0.f};
  int run_first = p_beg;

  auto flush_run = [&]() {
    // butterfly over the lanes that carry the same heads (lanes without
    // output carry zero counts), fixed order: deterministic. Afterwards the
    // lanes with g == 0 and q < kWriters hold the run's moments of heads
    // (oh, oh + 1).
#pragma unroll
    for (int k = 0; k < kHeads; ++k) {
      if (!owriter) run_m[k] = Mom{0.f, 0.f, 0.f};
#pragma unroll
      for (int mask = 1; mask < 32; mask <<= 1) {
        const bool same_heads = G == 8 ? mask >= 4 : (G == 4 ? mask >= 2 : true);
        if (same_heads) run_m[k] = mom_merge(run_m[k], mom_shfl(run_m[k], mask));
      }
    }
    constexpr int kWriters = G == 8 ? 4 : (G == 4 ? 2 : 1);
    if (g == 0 && q < kWriters) {
      float* tab = run_table(P, seg);
      const int r = run_index(run_first, seg_first[seg], per);
#pragma unroll
      for (int k = 0; k < kHeads; ++k) {
        tab[(1 + oh + k) * P.cs_max + r] = run_m[k].mean;
        tab[(1 + kMaxG + oh + k) * P.cs_max + r] = run_m[k].m2;
      }
      if (q == 0) tab[r] = run_m[0].n;
    }
#pragma unroll
    for (int k = 0; k < kHeads; ++k) run_m[k] = Mom{0.f, 0.f, 0.f};
  };

  for (int p = p_beg; p < p_end; ++p) {
    const int kp = p - p_beg;
    const int st = kp & 1;
    // next piece into the other stage (its previous contents were consumed)
    if (p + 1 < p_end && lane == 0) issue(p + 1, seg_of(p + 1, seg), st ^ 1);
    if constexpr (kQ8) {
      if (p + 1 < p_end) issue_scales(p + 1, seg_of(p + 1, seg), st ^ 1);
      else cp_async_commit();   // keep one group per piece
    }
    if (seg_first[seg + 1] <= p) {
      flush_run();
      seg = seg_of(p, seg);
      sv = seg_view(P, seg);
      load_consts(sv);
      run_first = p;
    }
    const int r0 = (p - seg_first[seg]) * geo.R;
    const int rows = min(geo.R, seg_rows[seg] - r0);
    const int64_t grow = seg_row0(seg) + r0;
    if (!mbar_wait_bounded(&bars[st], (uint32_t)((kp >> 1) & 1), P.spin_limit)) {
      if (lane == 0) report(P.ctrl, TRIA_ERR_TIMEOUT, (uint32_t)seg);
      drain_ring(bars, st, kp, p + 1 < p_end, P.spin_limit);
      if constexpr (kQ8) cp_async_wait<0>();
      return;
    }
    const uint8_t* buf = ring + st * geo.stage;
    const uint8_t* scb = sc_ring + st * kScaleStage;
    if constexpr (kQ8) {
      cp_async_wait<1>();   // this piece's scales (the next piece's may still be in flight)
      __syncwarp();
    }
    // shifted sums of this piece for my output heads
    float shift[kHeads], m1[kHeads], m2[kHeads], cnt[kHeads];
#pragma unroll
    for (int k = 0; k < kHeads; ++k) shift[k] = m1[k] = m2[k] = cnt[k] = 0.f;
    auto emit = [&](int rr, const float (&x)[kHeads]) {
      if (rr >= rows) return;
      float y[kHeads];
#pragma unroll
      for (int k = 0; k < kHeads; ++k) y[k] = x[k] * unscale[k];
      float* dst = P.raw + (size_t)(grow + rr) * G + oh;
      if constexpr (kHeads == 2) *reinterpret_cast<float2*>(dst) = make_float2(y[0], y[1]);
      else *dst = y[0];
#pragma unroll
      for (int k = 0; k < kHeads; ++k) {
        if (cnt[k] == 0.f) shift[k] = y[k];
        const float d = y[k] - shift[k];
        m1[k] += d;
        m2[k] = fmaf(d, d, m2[k]);
        cnt[k] += 1.f;
      }
    };
    for (int mt = 0; 16 * mt < rows; ++mt) {
      // independent accumulator chains, summed at the end: real, imaginary,
      // |k| high part, |k| remainder (two chains for head_dim > 128, where
      // registers are short and the chains are long enough anyway)
      constexpr bool kFour = S <= 4;
      float acc[NT][4], acc_i[NT][4], acc_mh[NT][4], acc_ml[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int t = 0; t < 4; ++t) acc[nt][t] = acc_i[nt][t] = acc_mh[nt][t] = acc_ml[nt][t] = 0.f;
      if constexpr (!kQ8) {
        const uint8_t* rg = buf + (size_t)(16 * mt + g) * P.k_rb + 16 * q;
        const uint8_t* rg8 = rg + (size_t)8 * P.k_rb;
  #pragma unroll
        for (int s2 = 0; s2 < S / 2; ++s2) {
          const uint4 kr0 = *reinterpret_cast<const uint4*>(rg + 64 * s2);
          const uint4 kr8 = *reinterpret_cast<const uint4*>(rg8 + 64 * s2);
          const uint4 ki0 = *reinterpret_cast<const uint4*>(rg + 64 * (s2 + S / 2));
          const uint4 ki8 = *reinterpret_cast<const uint4*>(rg8 + 64 * (s2 + S / 2));
  #pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            mma_f16(acc[nt], kr0.x, kr8.x, kr0.y, kr8.y, bp[s2][nt][0], bp[s2][nt][1]);
            float(&di)[4] = kFour ? acc_i[nt] : acc[nt];
            mma_f16(di, ki0.x, ki8.x, ki0.y, ki8.y, bp[s2 + S / 2][nt][0], bp[s2 + S / 2][nt][1]);
            mma_f16(acc[nt], kr0.z, kr8.z, kr0.w, kr8.w, bp[s2][nt][2], bp[s2][nt][3]);
            mma_f16(di, ki0.z, ki8.z, ki0.w, ki8.w, bp[s2 + S / 2][nt][2], bp[s2 + S / 2][nt][3]);
          }
          float mg0[8], mg8[8];
          granule_mag(kr0, ki0, mg0);
          granule_mag(kr8, ki8, mg8);
  #pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint32_t h0 = to_tf32(mg0[2 * u]), h1 = to_tf32(mg8[2 * u]);
            const uint32_t h2 = to_tf32(mg0[2 * u + 1]), h3 = to_tf32(mg8[2 * u + 1]);
            const uint32_t l0 = __float_as_uint(mg0[2 * u] - __uint_as_float(h0));
            const uint32_t l1 = __float_as_uint(mg8[2 * u] - __uint_as_float(h1));
            const uint32_t l2 = __float_as_uint(mg0[2 * u + 1] - __uint_as_float(h2));
            const uint32_t l3 = __float_as_uint(mg8[2 * u + 1] - __uint_as_float(h3));
  #pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              mma_tf32(acc_mh[nt], h0, h1, h2, h3, bm[s2][nt][u][0], bm[s2][nt][u][1]);
              float(&dl)[4] = kFour ? acc_ml[nt] : acc_mh[nt];
              mma_tf32(dl, l0, l1, l2, l3, bm[s2][nt][u][0], bm[s2][nt][u][1]);
            }
          }
        }
      } else {
        // q8_0: a 32-value block is one step s (bytes 32 s .. 32 s + 32 of the
        // row); its two MMAs go to a fresh accumulator scaled by the block's
        // scale of each row, and |k| uses the scaled values
        const uint8_t* rg = buf + (size_t)(16 * mt + g) * P.k_rb + 8 * q;
        const uint8_t* rg8 = rg + (size_t)8 * P.k_rb;
        const __half* sg0 = reinterpret_cast<const __half*>(scb + (size_t)(16 * mt + g) * P.ks_rb);
        const __half* sg8 = reinterpret_cast<const __half*>(scb + (size_t)(16 * mt + g + 8) * P.ks_rb);
#pragma unroll
        for (int s2 = 0; s2 < S / 2; ++s2) {
          const uint2 wr0 = *reinterpret_cast<const uint2*>(rg + 32 * s2);
          const uint2 wr8 = *reinterpret_cast<const uint2*>(rg8 + 32 * s2);
          const uint2 wi0 = *reinterpret_cast<const uint2*>(rg + 32 * (s2 + S / 2));
          const uint2 wi8 = *reinterpret_cast<const uint2*>(rg8 + 32 * (s2 + S / 2));
          const float dr0 = __half2float(sg0[s2]), dr8 = __half2float(sg8[s2]);
          const float di0 = __half2float(sg0[s2 + S / 2]), di8 = __half2float(sg8[s2 + S / 2]);
          uint32_t ar0[4], ar8[4], ai0[4], ai8[4];
          i8x4_to_h2x2(wr0.x, ar0[0], ar0[1]);
          i8x4_to_h2x2(wr0.y, ar0[2], ar0[3]);
          i8x4_to_h2x2(wr8.x, ar8[0], ar8[1]);
          i8x4_to_h2x2(wr8.y, ar8[2], ar8[3]);
          i8x4_to_h2x2(wi0.x, ai0[0], ai0[1]);
          i8x4_to_h2x2(wi0.y, ai0[2], ai0[3]);
          i8x4_to_h2x2(wi8.x, ai8[0], ai8[1]);
          i8x4_to_h2x2(wi8.y, ai8[2], ai8[3]);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            float tr[4] = {0.f, 0.f, 0.f, 0.f}, ti[4] = {0.f, 0.f, 0.f, 0.f};
            mma_f16(tr, ar0[0], ar8[0], ar0[1], ar8[1], bp[s2][nt][0], bp[s2][nt][1]);
            mma_f16(ti, ai0[0], ai8[0], ai0[1], ai8[1], bp[s2 + S / 2][nt][0], bp[s2 + S / 2][nt][1]);
            mma_f16(tr, ar0[2], ar8[2], ar0[3], ar8[3], bp[s2][nt][2], bp[s2][nt][3]);
            mma_f16(ti, ai0[2], ai8[2], ai0[3], ai8[3], bp[s2 + S / 2][nt][2], bp[s2 + S / 2][nt][3]);
            acc[nt][0] = fmaf(tr[0], dr0, fmaf(ti[0], di0, acc[nt][0]));
            acc[nt][1] = fmaf(tr[1], dr0, fmaf(ti[1], di0, acc[nt][1]));
            acc[nt][2] = fmaf(tr[2], dr8, fmaf(ti[2], di8, acc[nt][2]));
            acc[nt][3] = fmaf(tr[3], dr8, fmaf(ti[3], di8, acc[nt][3]));
          }
          float mg0[8], mg8[8];
          q8_mag(ar0, ai0, dr0, di0, mg0);
          q8_mag(ar8, ai8, dr8, di8, mg8);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint32_t h0 = to_tf32(mg0[2 * u]), h1 = to_tf32(mg8[2 * u]);
            const uint32_t h2 = to_tf32(mg0[2 * u + 1]), h3 = to_tf32(mg8[2 * u + 1]);
            const uint32_t l0 = __float_as_uint(mg0[2 * u] - __uint_as_float(h0));
            const uint32_t l1 = __float_as_uint(mg8[2 * u] - __uint_as_float(h1));
            const uint32_t l2 = __float_as_uint(mg0[2 * u + 1] - __uint_as_float(h2));
            const uint32_t l3 = __float_as_uint(mg8[2 * u + 1] - __uint_as_float(h3));
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              mma_tf32(acc_mh[nt], h0, h1, h2, h3, bm[s2][nt][u][0], bm[s2][nt][u][1]);
              float(&dl)[4] = kFour ? acc_ml[nt] : acc_mh[nt];
              mma_tf32(dl, l0, l1, l2, l3, bm[s2][nt][u][0], bm[s2][nt][u][1]);
            }
          }
        }
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int t = 0; t < 4; ++t)
          acc[nt][t] = kFour ? (acc[nt][t] + acc_i[nt][t]) + (acc_mh[nt][t] + acc_ml[nt][t]) : acc[nt][t] + acc_mh[nt][t];
      // column pairs (high part, remainder) -> head scores
      if constexpr (G == 8) {
        emit(16 * mt + g, {acc[0][0] + acc[1][0], acc[0][1] + acc[1][1]});
        emit(16 * mt + g + 8, {acc[0][2] + acc[1][2], acc[0][3] + acc[1][3]});
      } else if constexpr (G == 4) {
        float v[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) v[t] = acc[0][t] + __shfl_xor_sync(0xffffffffu, acc[0][t], 2);
        if (q & 2) emit(16 * mt + g + 8, {v[2], v[3]});
        else emit(16 * mt + g, {v[0], v[1]});
      } else if constexpr (G == 2) {
        float v[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) v[t] = acc[0][t] + __shfl_xor_sync(0xffffffffu, acc[0][t], 1);
        if (q == 0) emit(16 * mt + g, {v[0], v[1]});
        else if (q == 1) emit(16 * mt + g + 8, {v[2], v[3]});
      } else {
        const float a = acc[0][0] + acc[0][1], b = acc[0][2] + acc[0][3];
        const float b_from0 = __shfl_xor_sync(0xffffffffu, b, 1);
        if (q == 0) emit(16 * mt + g, {a});
        else if (q == 1) emit(16 * mt + g + 8, {b_from0});
      }
    }
    // this piece's moments -> the run's moments
#pragma unroll
    for (int k = 0; k < kHeads; ++k) {
      Mom b;
      b.n = cnt[k];
      const float mean_d = cnt[k] > 0.f ? __fdividef(m1[k], cnt[k]) : 0.f;
      b.mean = shift[k] + mean_d;
      b.m2 = fmaxf(m2[k] - m1[k] * mean_d, 0.f);
      run_m[k] = mom_merge(run_m[k], b);
    }
    __syncwarp();
  }
  flush_run();
}

size_t score_smem_bytes(const Pass& P) { return (size_t)score_smem_bytes_for(P.k_rb); }

int score_pieces_max(int k_rb, int cap) {
  const ScoreGeom g = score_geom(k_rb);
  return (cap + g.R - 1) / g.R;
}

namespace {

int sm_count() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

template <int KT, int G, int TPR, int PPT>
cudaError_t launch_score_t(const Pass& P, cudaStream_t st) {
  const size_t smem = score_smem_bytes(P);
  auto kern = k_score<KT, G, TPR, PPT>;
  // the attribute is per function: set the largest size any layout needs, once
  static const cudaError_t attr =
      set_smem_attrs(kern, kScoreSmemMax);
  if (attr != cudaSuccess) return attr;
  static const int sms = sm_count();
  kern<<<sms, kScoreThreads, smem, st>>>(P);
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

template <int KT, int G, int S>
cudaError_t launch_score_tc_t(const Pass& P, cudaStream_t st) {
  const size_t smem = score_smem_bytes(P);
  auto kern = k_score_tc<KT, G, S>;
  static const cudaError_t attr =
      set_smem_attrs(kern, kScoreSmemMax);
  if (attr != cudaSuccess) return attr;
  static const int sms = sm_count();
  kern<<<sms, kScoreThreads, smem, st>>>(P);
  return cudaGetLastError();
}

// fp16 or q8_0 keys with head_dim a multiple of 64 and the B fragments in
// registers (n-tiles x steps <= 8): the tensor-core body; false when it does
// not apply
template <int KT, int G>
bool launch_score_tc_g(const Pass& P, cudaStream_t st, cudaError_t* err) {
  switch (P.hd) {
    case 64: *err = launch_score_tc_t<KT, G, 2>(P, st); return true;
    case 128: *err = launch_score_tc_t<KT, G, 4>(P, st); return true;
    case 192:
      if constexpr (TcShape<G, 6>::kOk) {
        *err = launch_score_tc_t<KT, G, 6>(P, st);
        return true;
      }
      return false;
    case 256:
      if constexpr (TcShape<G, 8>::kOk) {
        *err = launch_score_tc_t<KT, G, 8>(P, st);
        return true;
      }
      return false;
  }
  return false;
}

template <int KT>
bool launch_score_tc_k(const Pass& P, cudaStream_t st, cudaError_t* err) {
  switch (P.G) {
    case 1: return launch_score_tc_g<KT, 1>(P, st, err);
    case 2: return launch_score_tc_g<KT, 2>(P, st, err);
    case 4: return launch_score_tc_g<KT, 4>(P, st, err);
    case 8: return launch_score_tc_g<KT, 8>(P, st, err);
  }
  return false;
}

bool launch_score_tc(const Pass& P, cudaStream_t st, cudaError_t* err) {
  if (P.k_type == TRIA_F16) return launch_score_tc_k<TRIA_F16>(P, st, err);
  if (P.k_type == TRIA_Q8_0) return launch_score_tc_k<TRIA_Q8_0>(P, st, err);
  return false;
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
  if (P.n_seg > kMaxSegs) return cudaErrorInvalidValue;
  cudaError_t e = cudaSuccess;
  if (launch_score_tc(P, st, &e)) return e;
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
