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
// with W = qbar E_f e^{i w_f p} and M = q_abs - |qbar|. Heads whose last
// nonrot dims are not rotary pair the fcr = (hd - nonrot) / 2 rotary pairs as
// (f, f + fcr) and add nonrot / 2 content pairs (f + fcr, f + fc) of
// frequency 0 and M = 0: their phase term is the mean non-rotary query's dot
// product with those dims ([Doc] §4 gate field nonrot=, §6 non-rotary models).
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
#include "score_tc.cuh"

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
  // pairs f < fcr are rotary, (f, f + fcr); the rest are the content pairs of
  // the non-rotary dims, (f + fcr, f + fc), with no norm term (fcr % PPT == 0)
  const bool lane_rot = f0 < P.fcr;
  const int e_re = lane_rot ? f0 : f0 + P.fcr, e_im = lane_rot ? f0 + P.fcr : f0 + fc;

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
          Loader<KT, PPT>::half(row, e_re, kr);
          Loader<KT, PPT>::half(row, e_im, ki);
          if constexpr (KT == TRIA_Q8_0) {
            const __half* sc = reinterpret_cast<const __half*>(P.ks + (size_t)(grow + rr) * P.ks_rb);
            const float d1 = __half2float(sc[e_re >> 5]);
            const float d2 = __half2float(sc[e_im >> 5]);
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
          mag[j] = lane_rot ? make_float2(sqrt_approx(sq.x), sqrt_approx(sq.y)) : make_float2(0.f, 0.f);
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
// Tensor-core scorer (fp16 / q8_0 keys, head_dim a multiple of 64): the same
// persistent layout as k_score, with the body of score_tc.cuh.
// ---------------------------------------------------------------------------

template <int KT, int G, int S>
__global__ void __launch_bounds__(kScoreThreads, 1) k_score_tc(const __grid_constant__ Pass P) {
  using Body = TcBody<KT, G, S>;
  constexpr bool kQ8 = Body::kQ8;
  constexpr int FC = Body::FC;
  constexpr int kHeads = Body::kHeads;

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

  Body body;
  body.init(lane, P.fcr);
  auto load_consts = [&](const SegView& v) {
    body.load_consts(P.qe + P.seq[v.s].qe_off + (size_t)v.g * G * FC, P.mw + P.seq[v.s].qe_off + (size_t)v.g * G * FC,
                     s_turns, (unsigned long long)P.seq[v.s].cur_pos);
  };

  int seg = seg_of(p_beg, 0);
  if (lane == 0) issue(p_beg, seg, 0);
  if constexpr (kQ8) issue_scales(p_beg, seg, 0);
  SegView sv = seg_view(P, seg);
  load_consts(sv);
  int run_first = p_beg;

  auto flush_run = [&]() {
    Mom m[kHeads];
    body.flush(m);
    if (body.flush_writer()) {
      float* tab = run_table(P, seg);
      const int r = run_index(run_first, seg_first[seg], per);
#pragma unroll
      for (int k = 0; k < kHeads; ++k) {
        tab[(1 + body.oh + k) * P.cs_max + r] = m[k].mean;
        tab[(1 + kMaxG + body.oh + k) * P.cs_max + r] = m[k].m2;
      }
      if (body.q == 0) tab[r] = m[0].n;
    }
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
    if constexpr (kQ8) {
      cp_async_wait<1>();   // this piece's scales (the next piece's may still be in flight)
      __syncwarp();
    }
    body.piece(ring + st * geo.stage, sc_ring + st * kScaleStage, rows, P.k_rb, P.ks_rb, P.raw + (size_t)grow * G);
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
  if (P.fcr % 32 != 0) return false;   // rotary pairs in whole 32-pair steps
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
