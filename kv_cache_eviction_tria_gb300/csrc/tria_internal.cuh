// Internal declarations shared by the kernels and the C ABI of the eviction pass.
//
// Sources cited by page title and section:
//   [Worklog] "TriAttention Native C++ Worklog"
//   [Doc]     "TriAttention KV-Cache Eviction (--triattention)"
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "tria.h"

namespace tria {

constexpr int kMaxSeqs = TRIA_MAX_SEQS;
constexpr int kMaxG = TRIA_MAX_GROUP;
constexpr int kChunk = 32;            // rows per select / compaction chunk (one warp lane per row)
constexpr int kHistRowsPerCta = 2048; // rows per CTA in the radix-histogram passes
constexpr int kCountChunksPerCta = 16;// chunks per CTA in the count / keep-list passes (2 per warp)
constexpr int kHistBins = 2048;       // 11-bit digits (last pass: 10 bits)
constexpr float kZEps = 1e-6f;        // z = (raw - mean) / (std + 1e-6)
constexpr int kThreads = 256;
constexpr int kDefaultSpinLimit = 1 << 22;
constexpr int kMaxSegments = 1024;    // sequences x KV heads per call

// ---------------------------------------------------------------------------
// workspace
// ---------------------------------------------------------------------------

// Call-wide control words. Counters are self-resetting: the last CTA that uses
// one puts it back to zero, so a zeroed workspace stays usable across calls.
struct Ctrl {
  uint32_t status;       // first device error of the calls since the last check
  uint32_t detail;       // sequence / segment of that error
  uint32_t move_ticket;  // compaction CTAs take tickets in start order
  uint32_t move_done;    // compaction CTAs that finished
  uint32_t epoch;        // compaction flags carry epoch + 1 of their call
  uint32_t bad_keep;     // keep-list entries rejected by the validation pass
  uint32_t wait_flag;    // never set: target of the bounded-wait self-test
  uint32_t bar_count;    // grid barrier: CTAs arrived (reset by the last one)
  uint32_t bar_gen;      // grid barrier: generation, bumped when all arrived
  uint32_t pad[55];
};

// Per-segment state (one segment = one sequence x KV head of the layer).
struct SegState {
  float mu[kMaxG];       // per query head mean of raw over the live rows
  float inv[kMaxG];      // 1 / (std + 1e-6)
  uint32_t prefix;       // radix digits fixed so far
  int32_t kr;            // rows still to take inside the current prefix
  uint32_t T;            // key of the last kept candidate (after three passes)
  int32_t tie_row;       // last kept row among those with key == T (-1: none)
  int32_t cnt;           // last-arriver counter of the current kernel
  int32_t piece_first;   // score pieces of the segment: [piece_first, piece_end)
  int32_t piece_end;
  int32_t piece_per;     // score pieces per warp (runs start at its multiples)
  int32_t pad[8];
};
static_assert(sizeof(SegState) == 128, "SegState layout");

struct ScoreChunk {      // moments of one contiguous run of score pieces
  float mean[kMaxG];
  float m2[kMaxG];
  int32_t n;
  int32_t pad[3];
};

struct SelChunk {        // counts of one chunk
  int32_t n_gt;          // candidates with key > T
  int32_t n_tie;         // candidates with key == T
  int32_t n_prot;        // protected rows (sink / window)
  int32_t pad;
};

struct SeqInfo {
  int64_t row0;          // first row of the sequence
  int64_t cur_pos;       // absolute decode position
  int32_t cap;           // rows per segment
  int32_t budget;        // B
  int32_t pad[2];
};

// Everything a kernel of the pass needs, passed by value.
struct Pass {
  int32_t n_seqs, n_kv, n_seg, G, hd, fc;
  int32_t sink, window;
  int32_t k_type, v_type;
  int32_t k_rb, ks_rb, v_rb, vs_rb;   // bytes per row of each plane (0: absent)
  int32_t only_active;                // skip segments with n_live <= B
  int32_t spin_limit;
  // cache (device)
  uint8_t* k;
  uint8_t* ks;
  uint8_t* v;
  uint8_t* vs;
  int32_t* pos;
  int32_t* n_live;
  // statistics of this layer (device)
  const float2* qe;                    // [n_kv][G][fc] qbar * offset average E_f
  const float* mw;                     // [n_kv][G][fc] q_abs - |qbar|
  const unsigned long long* turns;     // [fc] frac(w_f / 2pi) * 2^64
  // inputs / outputs indexed by global row
  float* raw;                          // [rows][G]
  float* score;                        // [rows] z-max score written by the score stage
  const float* score_in;               // [rows] score read by the select stage
  int32_t* keep;                       // [rows] keep lists
  // workspace
  Ctrl* ctrl;
  SegState* seg;
  ScoreChunk* schunk;                  // [n_seg * cs_max] indexed by global score piece
  SelChunk* chunk;                     // [n_seg][c_max]
  int32_t* prefix;                     // [n_seg][c_max + 1] kept rows before each chunk
  uint32_t* hist;                      // [n_seg][kHistBins]
  uint32_t* flags;                     // [n_seg][c_max] compaction read-done flags
  int32_t cs_rows;                     // unused (layout compatibility)
  int32_t cs_max;                      // score pieces per segment (max)
  int32_t c_max;                       // chunks per segment (max)
  int32_t pad0;
  SeqInfo seq[kMaxSeqs];
};

// ---------------------------------------------------------------------------
// per-segment view
// ---------------------------------------------------------------------------

struct SegView {
  int s, g;
  int64_t row0;
  int n, B, k;
  bool valid, active;
};

__device__ __forceinline__ SegView seg_view(const Pass& P, int seg) {
  SegView v;
  v.s = seg / P.n_kv;
  v.g = seg - v.s * P.n_kv;
  const SeqInfo& q = P.seq[v.s];
  v.row0 = q.row0 + (int64_t)v.g * q.cap;
  v.n = *((volatile const int32_t*)(P.n_live + v.s));
  v.B = q.budget;
  v.valid = v.n >= 0 && v.n <= q.cap;
  v.active = v.valid && v.n > v.B;
  v.k = v.B - P.sink - P.window;
  return v;
}

__device__ __forceinline__ void report(Ctrl* c, uint32_t code, uint32_t detail) {
  if (atomicCAS(&c->status, 0u, code) == 0u) atomicExch(&c->detail, detail);
}

// Order-preserving map float -> uint32: a > b  <=>  key(a) > key(b); -0 and +0
// share a key; NaN gets the lowest key (evicted first, like a stable sort that
// puts NaN last in descending order).
__device__ __forceinline__ uint32_t score_key(float s) {
  uint32_t u = __float_as_uint(s);
  if (s != s) return 0u;
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ bool is_protected(int r, int n, int sink, int window) {
  return r < sink || r >= n - window;
}

// ---------------------------------------------------------------------------
// PTX wrappers: mbarrier + bulk async copy (TMA, non-tensor form)
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

// Global -> shared bulk copy; dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait on an mbarrier phase; false when the limit ran out.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, int limit) {
  for (int it = 0; it < limit; ++it)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_u32(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void st_relaxed_u32(uint32_t* p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Bounded poll of a flag written by another CTA; false when the limit ran out.
__device__ __forceinline__ bool wait_flag_bounded(const uint32_t* flag, uint32_t target, int limit) {
  for (int it = 0; it < limit; ++it) {
    if (ld_acquire_u32(flag) == target) return true;
    __nanosleep(it < 64 ? 32 : 256);
  }
  return false;
}

// Bounded poll until a word differs from `old`; false when the limit ran out.
__device__ __forceinline__ bool wait_flag_bounded_ne(const uint32_t* flag, uint32_t old, int limit) {
  for (int it = 0; it < limit; ++it) {
    if (ld_acquire_u32(flag) != old) return true;
    __nanosleep(it < 64 ? 32 : 256);
  }
  return false;
}

// ---------------------------------------------------------------------------
// block-wide helpers
// ---------------------------------------------------------------------------

// Exclusive prefix sum over the block (kThreads threads); returns the thread's
// exclusive prefix and writes the total to *total.
__device__ __forceinline__ int block_exclusive_scan(int x, int* total, int* sbuf /* >= 33 ints */) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int v = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += y;
  }
  if (lane == 31) sbuf[warp] = v;
  __syncthreads();
  if (warp == 0) {
    int w = (lane < (int)(blockDim.x >> 5)) ? sbuf[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < 32) sbuf[lane] = w;  // inclusive per-warp totals
  }
  __syncthreads();
  int before = (warp > 0 ? sbuf[warp - 1] : 0) + v - x;
  *total = sbuf[(blockDim.x >> 5) - 1];
  __syncthreads();
  return before;
}

// ---------------------------------------------------------------------------
// moments (Chan et al. pairwise update) and the per-segment merge
// ---------------------------------------------------------------------------

// running (count, mean, M2) of one head
struct Mom {
  float n, mean, m2;
};

__device__ __forceinline__ Mom mom_merge(Mom a, Mom b) {
  const float n = a.n + b.n;
  if (n == 0.f) return a;
  const float d = b.mean - a.mean;
  const float fb = __fdividef(b.n, n);   // counts: n well inside the fast divide's range
  Mom r;
  r.n = n;
  r.mean = a.mean + d * fb;
  r.m2 = a.m2 + b.m2 + d * d * a.n * fb;
  return r;
}

__device__ __forceinline__ Mom mom_shfl(Mom a, int mask) {
  Mom b;
  b.n = __shfl_xor_sync(0xffffffffu, a.n, mask);
  b.mean = __shfl_xor_sync(0xffffffffu, a.mean, mask);
  b.m2 = __shfl_xor_sync(0xffffffffu, a.m2, mask);
  return b;
}

// Merge of a segment's run partials (written by k_score) into mean and
// 1 / (std + 1e-6), by one CTA: thread t merges runs t, t + blockDim, ...
// (Chan et al. pairwise update, fp32), then a butterfly over the lanes of each
// warp and a second butterfly over the warp results, which every warp
// computes identically (lane 0's result is broadcast), so no serial chain and
// one barrier. Runs start at the segment's first piece and at each multiple
// of the per-warp piece count after it. Deterministic for a given layout.
template <int G>
__device__ void merge_segment_moments(const Pass& P, int seg, float* mu, float* inv) {
  __shared__ Mom red[32][G];   // up to 32 warps
  const int s0 = __ldcg(&P.seg[seg].piece_first), s1 = __ldcg(&P.seg[seg].piece_end);
  const int per = max(1, __ldcg(&P.seg[seg].piece_per));
  const int first_mult = (s0 / per + 1) * per;
  const int nruns = s1 > s0 ? 1 + (s1 > first_mult ? (s1 - first_mult + per - 1) / per : 0) : 0;
  Mom acc[G];
#pragma unroll
  for (int h = 0; h < G; ++h) acc[h] = Mom{0.f, 0.f, 0.f};
  for (int i = threadIdx.x; i < nruns; i += blockDim.x) {
    const int j = i == 0 ? s0 : first_mult + (i - 1) * per;
    const ScoreChunk* pp = P.schunk + j;
    const float n = (float)__ldcg(&pp->n);
#pragma unroll
    for (int h = 0; h < G; ++h) acc[h] = mom_merge(acc[h], Mom{n, __ldcg(&pp->mean[h]), __ldcg(&pp->m2[h])});
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int mask = 1; mask < 32; mask <<= 1)
#pragma unroll
    for (int h = 0; h < G; ++h) acc[h] = mom_merge(acc[h], mom_shfl(acc[h], mask));
  if (lane == 0)
#pragma unroll
    for (int h = 0; h < G; ++h) red[warp][h] = acc[h];
  __syncthreads();
  const int nw = (int)(blockDim.x >> 5);
#pragma unroll
  for (int h = 0; h < G; ++h) acc[h] = lane < nw ? red[lane][h] : Mom{0.f, 0.f, 0.f};
#pragma unroll
  for (int mask = 1; mask < 32; mask <<= 1)
#pragma unroll
    for (int h = 0; h < G; ++h) acc[h] = mom_merge(acc[h], mom_shfl(acc[h], mask));
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const float n = __shfl_sync(0xffffffffu, acc[h].n, 0);
    const float m = __shfl_sync(0xffffffffu, acc[h].mean, 0);
    const float m2 = __shfl_sync(0xffffffffu, acc[h].m2, 0);
    mu[h] = m;
    inv[h] = 1.0f / (sqrtf(m2 / fmaxf(n, 1.f)) + kZEps);
  }
}

// Dynamic shared-memory limit and the largest shared-memory carveout of a
// kernel: the stages of a pass then keep one L1 / shared split, and the SMs
// need not switch it between them.
template <typename Kernel>
cudaError_t set_smem_attrs(Kernel* kern, int dyn_bytes) {
  const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn_bytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
}

// ---------------------------------------------------------------------------
// grid barrier of a cooperative launch (all CTAs resident), bounded: after the
// spin limit it records TRIA_ERR_TIMEOUT and lets the CTA go on (no hang)
// ---------------------------------------------------------------------------

__device__ __forceinline__ bool grid_barrier(const Pass& P) {
  __shared__ int s_timeout;
  __syncthreads();
  if (threadIdx.x == 0) {
    s_timeout = 0;
    const uint32_t gen = ld_acquire_u32(&P.ctrl->bar_gen);
    __threadfence();
    if (atomicAdd(&P.ctrl->bar_count, 1u) == gridDim.x - 1) {
      atomicExch(&P.ctrl->bar_count, 0u);
      __threadfence();
      atomicAdd(&P.ctrl->bar_gen, 1u);
    } else if (!wait_flag_bounded_ne(&P.ctrl->bar_gen, gen, P.spin_limit)) {
      s_timeout = 1;
      report(P.ctrl, TRIA_ERR_TIMEOUT, 0xB0000000u);
    }
    __threadfence();
  }
  __syncthreads();
  return s_timeout == 0;
}

// ---------------------------------------------------------------------------
// launchers (one per translation unit)
// ---------------------------------------------------------------------------

// score.cu
cudaError_t launch_score(const Pass& P, cudaStream_t st);
cudaError_t launch_zscore(const Pass& P, cudaStream_t st);
size_t score_smem_bytes(const Pass& P);
int score_pieces_max(int k_rb, int cap);   // score pieces of a segment of `cap` rows
// select.cu: score_group > 0 computes the z-max score from the raw scores of
// the score stage (evict path) and writes it to P.score; 0 reads P.score_in
cudaError_t launch_select(const Pass& P, bool write_keep, cudaStream_t st, int score_group = 0);
// compact.cu
cudaError_t launch_keep_prepass(const Pass& P, cudaStream_t st);
cudaError_t launch_move(const Pass& P, cudaStream_t st);
cudaError_t launch_wait_selftest(const Pass& P, cudaStream_t st);
// stats.cu
struct StatsDevice;

}  // namespace tria

// Opaque stats handle of the C ABI.
struct tria_stats {
  int32_t n_layers, n_q_heads, n_kv_heads, head_dim, group;
  float2* qe;                  // [L][n_kv][G][fc]
  float* mw;                   // [L][n_kv][G][fc]
  unsigned long long* turns;   // [fc]
};
