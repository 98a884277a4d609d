// Internal declarations shared by the kernels and the C ABI of the eviction pass.
//
// Sources cited by page title and section:
//   [Worklog] "TriAttention Native C++ Worklog"
//   [Doc]     "TriAttention KV-Cache Eviction (--triattention)"
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

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
  uint32_t append_ticket;  // append CTAs that finished (reset by the last one)
  // fused pass (k_pass): reset by its last CTA
  uint32_t scored_count; // segments completely scored (slots of the scored list)
  uint32_t sel_next;     // next scored segment to select
  uint32_t ready_count;  // segments whose selection is published (slots of the ready list)
  uint32_t move_cursor;  // first ready slot that may still have unclaimed move blocks
  uint32_t pass_done;    // CTAs of the pass that finished
  uint32_t pad[49];
};
static_assert(sizeof(Ctrl) == 256, "Ctrl layout");

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

// Moment partials of the score runs: per segment, columns of cs_max floats
// (count, then the mean of head 0 .. kMaxG-1, then the sum of squared
// deviations of head 0 .. kMaxG-1), run r of the segment in row r, so that a
// warp reads them with coalesced loads.
constexpr int kRunCols = 1 + 2 * kMaxG;

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
  int32_t sink;          // first rows always kept
  int32_t qe_off;        // this sequence's layer in the folded statistics (elements from P.qe / P.mw)
};

// Everything a kernel of the pass needs, passed by value.
struct Pass {
  int32_t n_seqs, n_kv, n_seg, G, hd, fc;
  int32_t fcr;                        // rotary pairs of fc (fc when every dim is rotary)
  int32_t window;
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
  float* runs;                         // [n_seg][kRunCols][cs_max] score-run moment partials
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
  int n, B, k, sink;
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
  v.sink = q.sink;
  v.k = v.B - v.sink - P.window;
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

// Tag of the compaction read-done flags of the call with control epoch e:
// (e + 1) times an odd constant (mod 2^32), so consecutive calls' tags differ
// and a tag is unlike the small counts or float bit patterns that other
// calls may have left in the same workspace bytes; never 0.
__host__ __device__ __forceinline__ uint32_t flag_tag(uint32_t epoch) {
  const uint32_t x = (epoch + 1u) * 0x9E3779B1u;
  return x ? x : 1u;
}

// Fixed-position state of the fused pass, right after the control words in
// every workspace layout (so calls with different layer counts on one
// workspace never read each other's data as counters): per segment of the
// call, the ready list, the completed score items and the next move block.
constexpr int kPassCtlSegs = 2048;
struct PassCtl {
  int32_t ready[kPassCtlSegs];        // selected segments + 1 in publication order (0: not yet)
  int32_t scored[kPassCtlSegs];       // segments + 1 whose last pieces are scored, in that order
  int32_t pieces_done[kPassCtlSegs];  // scored pieces per segment
  int32_t move_next[kPassCtlSegs];    // next destination block to claim per segment
};

__device__ __forceinline__ bool is_protected(int r, int n, int sink, int window) {
  return r < sink || r >= n - window;
}

// ---------------------------------------------------------------------------
// PTX wrappers: mbarrier + bulk async copy (TMA, non-tensor form)
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------------------
// async-copy helpers (cp.async: per-thread global -> shared copies that need
// no registers; completion per thread group, then a block barrier)
// ---------------------------------------------------------------------------

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async8(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_inval(uint64_t* bar) {
  asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
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

// Shared -> global bulk copy, completion by bulk group; dst, src and bytes must
// be multiples of 16.
__device__ __forceinline__ void bulk_s2g(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_u32(src)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// this thread's bulk groups have finished reading shared memory
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// this thread's bulk groups are complete
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// order generic-proxy shared-memory writes before later async-proxy reads
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
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

__device__ __forceinline__ float* run_table(const Pass& P, int seg) {
  return P.runs + (size_t)seg * kRunCols * P.cs_max;
}

// index, within its segment, of the score run that starts at piece p
__device__ __forceinline__ int run_index(int p, int s0, int per) {
  return p == s0 ? 0 : (p - (s0 / per + 1) * per) / per + 1;
}

// Number of score runs of a segment whose pieces are [s0, s1) when every warp
// takes `per` consecutive pieces: runs start at s0 and at each multiple of
// per after it.
__device__ __forceinline__ int segment_runs(int s0, int s1, int per) {
  if (s1 <= s0) return 0;
  const int first_mult = (s0 / per + 1) * per;
  return 1 + (s1 > first_mult ? (s1 - first_mult + per - 1) / per : 0);
}

// Segment moments from the score-run partials (count n_i, mean m_i, sum of
// squared deviations M2_i), by exact identities with a shift c (run 0's mean):
// with d_i = m_i - c,
//   N = sum n_i,  mean = c + (sum n_i d_i) / N,
//   N var = sum (M2_i + n_i d_i^2) - (sum n_i d_i)^2 / N,
// so partial sums over any split of the runs add up (no division per run),
// and the shifted sums stay small (fp32).
//
// mean and 1 / (std + 1e-6) of each head from the sums of all runs
template <int G>
__device__ __forceinline__ void moments_from_sums(const float* c, const float* sums, float* mu, float* inv) {
  const float n = fmaxf(sums[0], 1.f);
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const float md = sums[1 + h] / n;
    const float var = fmaxf(sums[1 + G + h] / n - md * md, 0.f);
    mu[h] = c[h] + md;
    inv[h] = 1.0f / (sqrtf(var) + kZEps);
  }
}

// Moments of one segment from its run partials (tab: kRunCols columns of cs
// floats, runs 0 .. nr-1), merged by one block; see block_segment_moments.
// scratch: shared memory for 33 x (1 + 2G) floats; the block may reuse it
// once it has passed a __syncthreads after the call.
template <int G>
__device__ void block_moments_of_runs(const float* tab, int cs, int nr, float* mu, float* inv, float* scratch) {
  float (*red)[1 + 2 * G] = reinterpret_cast<float (*)[1 + 2 * G]>(scratch);
  float* sums = scratch + 32 * (1 + 2 * G);
  float c[G];
#pragma unroll
  for (int h = 0; h < G; ++h) c[h] = __ldcg(&tab[(1 + h) * cs]);
  float n = 0.f, mean[G], m2[G];
  auto load_run = [&](int r) {
    n = __ldcg(&tab[r]);
#pragma unroll
    for (int h = 0; h < G; ++h) {
      mean[h] = __ldcg(&tab[(1 + h) * cs + r]);
      m2[h] = __ldcg(&tab[(1 + kMaxG + h) * cs + r]);
    }
  };
  float v[1 + 2 * G];
#pragma unroll
  for (int k = 0; k < 1 + 2 * G; ++k) v[k] = 0.f;
  auto add_run = [&]() {   // an empty run's mean is not used
    v[0] += n;
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float d = n > 0.f ? mean[h] - c[h] : 0.f;
      const float nd = n * d;
      v[1 + h] += nd;
      v[1 + G + h] += fmaf(nd, d, n > 0.f ? m2[h] : 0.f);
    }
  };
  int r = threadIdx.x;
  if (r < cs) load_run(r);
  if (r < nr) add_run();
  for (r += blockDim.x; r < nr; r += blockDim.x) {
    load_run(r);
    add_run();
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (int)(blockDim.x >> 5);
#pragma unroll
  for (int mask = 1; mask < 32; mask <<= 1)
#pragma unroll
    for (int k = 0; k < 1 + 2 * G; ++k) v[k] += __shfl_xor_sync(0xffffffffu, v[k], mask);
  if (lane == 0)
#pragma unroll
    for (int k = 0; k < 1 + 2 * G; ++k) red[warp][k] = v[k];
  __syncthreads();
  if (threadIdx.x < 1 + 2 * G) {
    float a = 0.f;
    for (int w = 0; w < nw; ++w) a += red[w][threadIdx.x];
    sums[threadIdx.x] = a;
  }
  __syncthreads();
  moments_from_sums<G>(c, sums, mu, inv);
}

template <int G>
__device__ void block_moments_of_runs(const float* tab, int cs, int nr, float* mu, float* inv) {
  __shared__ float scratch[33 * (1 + 2 * G)];
  block_moments_of_runs<G>(tab, cs, nr, mu, inv, scratch);
}

// Mean and 1 / (std + 1e-6) of the segment's heads, merged by one block
// (all threads call it) from the segment's score-run partials. Thread t adds
// runs t, t + blockDim, ... in order into {N, sum n d_h, sum (M2 + n d^2)_h},
// then fixed butterflies over lanes and warps (deterministic). The shift c
// (run 0's mean) and the first round of run partials are loaded together, so
// the merge waits for one load latency; first-round rows past the run count
// are loaded and ignored.
template <int G>
__device__ void block_segment_moments(const Pass& P, int seg, float* mu, float* inv) {
  const int s0 = __ldcg(&P.seg[seg].piece_first), s1 = __ldcg(&P.seg[seg].piece_end);
  const int per = max(1, __ldcg(&P.seg[seg].piece_per));
  block_moments_of_runs<G>(run_table(P, seg), P.cs_max, segment_runs(s0, s1, per), mu, inv);
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
// lifecycle.cu: rows [n_seqs][n_kv][n_tokens] appended after the live rows
struct AppendSrc {
  const uint8_t* k;
  const uint8_t* ks;
  const uint8_t* v;
  const uint8_t* vs;
  const int32_t* pos;                  // [n_seqs][n_tokens]
  int32_t n_tokens;
};
cudaError_t launch_append(const Pass& P, const AppendSrc& a, cudaStream_t st);
// shared.cu: shared-slot variant (one keep-set per token for all layers)
cudaError_t launch_shared_combine(const Pass& P, const float* scores, int64_t stride, int n_layers, float* combined,
                                  cudaStream_t st);
cudaError_t launch_shared_broadcast(const Pass& P, int32_t* keep, cudaStream_t st);
// stats.cu
struct StatsDevice;
// api.cu: the host-side argument checks every entry point on a layer cache
// shares (layout, pointers and alignment; budget, sink, window and position
// of every sequence). need_budget = false: scoring only, no budget checked.
tria_status check_cache(const tria_layer_cache* c);
tria_status check_policy(const tria_layer_cache* c, const tria_policy* p, bool need_pos, std::vector<int>& budget,
                         bool need_budget = true);

}  // namespace tria

// Opaque stats handle of the C ABI.
struct tria_stats {
  int32_t n_layers, n_q_heads, n_kv_heads, group;
  int32_t nonrot_dim;          // non-rotary dims of every head (the last ones)
  float2* qe;                  // per loaded layer l: [n_kv][G][fc_l] from qe_off[l]; fc_l = head_dim_l / 2
                               // pairs: the rotary ones, then the content pairs of the non-rotary dims
  float* mw;                   // same layout as qe
  unsigned long long* turns;   // per loaded layer l: [fc_l] from turns_off[l]
  std::vector<int32_t> head_dim;     // [L]
  std::vector<int64_t> qe_off;       // [L]; -1: layer not loaded (fails the gate)
  std::vector<int64_t> turns_off;    // [L]
  std::vector<double> freq;          // [L][head_dim_l / 2] host copy of the frequencies (theta or omega)
  std::vector<int64_t> freq_off;     // [L + 1] offsets into freq
};
