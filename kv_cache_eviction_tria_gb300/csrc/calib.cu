// Calibration statistics of one layer from a stream of pre-RoPE queries.
//
// [Doc] "TriAttention KV-Cache Eviction (--triattention)", §2 Calibration
// file (statistics per layer and head of the pre-RoPE queries seen on
// calibration text: the average query direction and a weight per frequency) and
// §5 Phase C (the q_mean / q_abs arrays, [layers][heads][frequency pairs]).
// With NEOX pairs z = q[f] + i q[f + hd/2]: q_mean = mean z, q_abs = mean |z|.
// Heads whose last nonrot dims are not rotary: the fcr = (hd - nonrot) / 2
// rotary pairs are (f, f + fcr) and the nonrot / 2 content pairs that follow
// are (f + fcr, f + hd/2), whose mean is the mean non-rotary query (the
// content term of [Doc] §6 "Non-rotary models"); the finish step splits them.
//
// One streaming read of the queries: a block takes a range of tokens and a
// block of 64 (head, 16-byte vector of pairs) slots, reads contiguous spans
// of every token row with 16-byte loads, accumulates in fp32 (sub-streams
// combined in shared memory) and adds its sums to the caller's fp64
// accumulator, one atomic per value and block. Rows whose halves are not
// whole 16-byte vectors take a scalar body (lane per pair).
#include "tria_internal.cuh"

namespace tria {
namespace {

constexpr int kCalibWarps = 8;
constexpr int kCalibTokens = 256;   // tokens per block
constexpr int kCalibMaxPairs = 256;  // head_dim <= 512
constexpr int kCalibPerLane = kCalibMaxPairs / 32;

template <typename T>
__device__ __forceinline__ float as_f32(T x);
template <>
__device__ __forceinline__ float as_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float as_f32<__half>(__half x) { return __half2float(x); }

// Vector body (every half-row a whole number of 16-byte vectors). Slot
// (head, v) = the P = 16 / sizeof(T) consecutive pairs of vector v of the
// head's half-rows. Block (c, b) takes slots [64 b, 64 b + 64) - whole
// adjacent half-rows, so every token read is one contiguous span - and token
// range c, split over kCalibStreams sub-streams of 64 threads; a thread reads
// two 16-byte vectors per token (real and imaginary half), four tokens in
// flight. The sub-streams add into shared memory, then one fp64 atomic per
// (head, pair, quantity) and block goes to the caller's accumulator.
constexpr int kCalibSlots = 64;
constexpr int kCalibStreams = 16;
constexpr int kCalibVecThreads = kCalibSlots * kCalibStreams;

template <typename T>
__global__ void __launch_bounds__(kCalibVecThreads) k_calib_acc(const T* __restrict__ q, int n_tokens, int n_heads,
                                                                 int hd, int fcr, int tok_per_block,
                                                                 double* __restrict__ acc) {
  constexpr int P = 16 / sizeof(T);
  __shared__ float red[kCalibSlots][3 * P];
  const int fc = hd / 2;
  const int vpr = fc / P;   // vectors per half-row
  const int slots = n_heads * vpr;
  const int sl = blockIdx.y * kCalibSlots + (threadIdx.x % kCalibSlots);
  const int stream = threadIdx.x / kCalibSlots;
  for (int i = threadIdx.x; i < kCalibSlots * 3 * P; i += blockDim.x) (&red[0][0])[i] = 0.f;
  __syncthreads();
  const int t0 = blockIdx.x * tok_per_block, t1 = min(n_tokens, t0 + tok_per_block);
  if (sl < slots) {
    const int h = sl / vpr, f0 = (sl - h * vpr) * P;
    // first dims of the pairs' two halves (fcr % P == 0: a vector is all
    // rotary or all content)
    const int d_re = f0 < fcr ? f0 : f0 + fcr, d_im = f0 < fcr ? f0 + fcr : f0 + fc;
    const T* base = q + (size_t)h * hd + d_re;
    const int im_off = d_im - d_re;
    const size_t stride = (size_t)n_heads * hd;
    float sr[P], si[P], sa[P];
#pragma unroll
    for (int k = 0; k < P; ++k) sr[k] = si[k] = sa[k] = 0.f;
    auto add = [&](const uint4& a, const uint4& b) {
      const T* re = reinterpret_cast<const T*>(&a);
      const T* im = reinterpret_cast<const T*>(&b);
#pragma unroll
      for (int k = 0; k < P; ++k) {
        const float x = as_f32(re[k]), y = as_f32(im[k]);
        sr[k] += x;
        si[k] += y;
        sa[k] += sqrtf(fmaf(x, x, y * y));
      }
    };
    constexpr int U = 4;   // tokens in flight per thread
    const size_t step = (size_t)kCalibStreams * stride;
    int t = t0 + stream;
    for (; t + (U - 1) * kCalibStreams < t1; t += U * kCalibStreams) {
      const T* r = base + (size_t)t * stride;
      uint4 a[U], b[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        a[u] = __ldcs(reinterpret_cast<const uint4*>(r + u * step));
        b[u] = __ldcs(reinterpret_cast<const uint4*>(r + u * step + im_off));
      }
#pragma unroll
      for (int u = 0; u < U; ++u) add(a[u], b[u]);
    }
    for (; t < t1; t += kCalibStreams) {
      const T* r0 = base + (size_t)t * stride;
      add(__ldcs(reinterpret_cast<const uint4*>(r0)), __ldcs(reinterpret_cast<const uint4*>(r0 + im_off)));
    }
    float* mine = red[threadIdx.x % kCalibSlots];
#pragma unroll
    for (int k = 0; k < P; ++k) {
      atomicAdd(&mine[3 * k], sr[k]);
      atomicAdd(&mine[3 * k + 1], si[k]);
      atomicAdd(&mine[3 * k + 2], sa[k]);
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < kCalibSlots * 3 * P; i += blockDim.x) {
    const int ls = i / (3 * P), r = i - ls * 3 * P;   // local slot, (pair, quantity)
    const int s2 = blockIdx.y * kCalibSlots + ls;
    if (s2 >= slots) continue;
    const int h = s2 / vpr, f0 = (s2 - h * vpr) * P;
    atomicAdd(&acc[((size_t)h * fc + f0) * 3 + r], (double)red[ls][r]);
  }
}

// Scalar body for head_dim not a multiple of 4: lane l owns pairs l, l + 32, ...
template <typename T>
__global__ void __launch_bounds__(kCalibWarps * 32) k_calib_acc_scalar(const T* __restrict__ q, int n_tokens,
                                                                        int n_heads, int hd, int fcr,
                                                                        double* __restrict__ acc) {
  __shared__ float part[kCalibWarps][3][kCalibMaxPairs];
  const int h = blockIdx.y;
  const int fc = hd / 2;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int t0 = blockIdx.x * kCalibTokens, t1 = min(n_tokens, t0 + kCalibTokens);
  float sr[kCalibPerLane], si[kCalibPerLane], sa[kCalibPerLane];
#pragma unroll
  for (int j = 0; j < kCalibPerLane; ++j) sr[j] = si[j] = sa[j] = 0.f;
  for (int t = t0 + warp; t < t1; t += kCalibWarps) {
    const T* row = q + ((size_t)t * n_heads + h) * hd;
#pragma unroll
    for (int j = 0; j < kCalibPerLane; ++j) {
      const int f = lane + 32 * j;
      if (f < fc) {
        const bool rot = f < fcr;
        const float re = as_f32(row[rot ? f : f + fcr]), im = as_f32(row[rot ? f + fcr : f + fc]);
        sr[j] += re;
        si[j] += im;
        sa[j] += sqrtf(fmaf(re, re, im * im));
      }
    }
  }
#pragma unroll
  for (int j = 0; j < kCalibPerLane; ++j) {
    const int f = lane + 32 * j;
    if (f < fc) {
      part[warp][0][f] = sr[j];
      part[warp][1][f] = si[j];
      part[warp][2][f] = sa[j];
    }
  }
  __syncthreads();
  for (int x = threadIdx.x; x < 3 * fc; x += blockDim.x) {
    const int k = x / fc, f = x - k * fc;
    float a = 0.f;
    for (int w = 0; w < kCalibWarps; ++w) a += part[w][k][f];
    atomicAdd(&acc[((size_t)h * fc + f) * 3 + k], (double)a);
  }
}

// acc [heads][fc][3] -> q_mean [heads][fcr][2], q_abs [heads][fcr] and
// q_nonrot [heads][2 (fc - fcr)] (content pair e: dims e and e + nonrot/2)
__global__ void k_calib_finish(const double* __restrict__ acc, double inv_n, int n_heads, int fc, int fcr,
                               float* __restrict__ q_mean, float* __restrict__ q_abs, float* __restrict__ q_nonrot) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;   // (head, pair)
  if (i >= n_heads * fc) return;
  const int h = i / fc, f = i - h * fc;
  if (f < fcr) {
    const int o = h * fcr + f;
    q_mean[2 * o] = (float)(acc[3 * i] * inv_n);
    q_mean[2 * o + 1] = (float)(acc[3 * i + 1] * inv_n);
    q_abs[o] = (float)(acc[3 * i + 2] * inv_n);
  } else {
    const int nr = 2 * (fc - fcr), e = f - fcr;
    q_nonrot[h * nr + e] = (float)(acc[3 * i] * inv_n);
    q_nonrot[h * nr + e + nr / 2] = (float)(acc[3 * i + 1] * inv_n);
  }
}

bool aligned4(const void* p) { return ((uintptr_t)p & 3u) == 0; }

}  // namespace
}  // namespace tria

using namespace tria;

extern "C" tria_status tria_calib_accumulate(const void* q, tria_dtype q_type, int32_t n_tokens, int32_t n_q_heads,
                                             int32_t head_dim, int32_t nonrot_dim, double* acc, void* stream) {
  if ((!q && n_tokens > 0) || !acc || n_tokens < 0 || n_q_heads < 1) return TRIA_ERR_INVALID_ARG;
  if (!aligned4(q) || ((uintptr_t)acc & 7u) != 0) return TRIA_ERR_INVALID_ARG;
  if (q_type != TRIA_F32 && q_type != TRIA_F16) return TRIA_ERR_UNSUPPORTED;
  if (head_dim < 2 || head_dim % 2 != 0 || head_dim > 2 * kCalibMaxPairs) return TRIA_ERR_UNSUPPORTED;
  if (nonrot_dim < 0 || nonrot_dim % 2 != 0 || nonrot_dim >= head_dim) return TRIA_ERR_INVALID_ARG;
  const int fcr = (head_dim - nonrot_dim) / 2;
  if (n_tokens == 0) return TRIA_OK;
  const dim3 grid((n_tokens + kCalibTokens - 1) / kCalibTokens, n_q_heads);
  if (grid.y > 65535) return TRIA_ERR_UNSUPPORTED;
  cudaStream_t st = (cudaStream_t)stream;
  // the vector body needs every half-row to be whole 16-byte vectors, and a
  // 16-byte aligned base
  const int esz = q_type == TRIA_F32 ? 4 : 2;
  const bool vec = ((head_dim / 2) * esz) % 16 == 0 && (fcr * esz) % 16 == 0 && ((uintptr_t)q % 16) == 0;
  if (vec) {
    // about one block per SM in all: slot blocks x token ranges
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int slot_blocks = (n_q_heads * ((head_dim / 2) / (16 / esz)) + kCalibSlots - 1) / kCalibSlots;
    if (slot_blocks > 65535) return TRIA_ERR_UNSUPPORTED;
    const int ranges = max(1, sms / slot_blocks);
    const int tpb = max(2 * kCalibStreams, (n_tokens + ranges - 1) / ranges);
    const dim3 vgrid((n_tokens + tpb - 1) / tpb, slot_blocks);
    if (q_type == TRIA_F32)
      k_calib_acc<float><<<vgrid, kCalibVecThreads, 0, st>>>((const float*)q, n_tokens, n_q_heads, head_dim, fcr,
                                                             tpb, acc);
    else
      k_calib_acc<__half><<<vgrid, kCalibVecThreads, 0, st>>>((const __half*)q, n_tokens, n_q_heads, head_dim, fcr,
                                                              tpb, acc);
  } else if (q_type == TRIA_F32) {
    k_calib_acc_scalar<float><<<grid, kCalibWarps * 32, 0, st>>>((const float*)q, n_tokens, n_q_heads, head_dim,
                                                                 fcr, acc);
  } else {
    k_calib_acc_scalar<__half><<<grid, kCalibWarps * 32, 0, st>>>((const __half*)q, n_tokens, n_q_heads, head_dim,
                                                                  fcr, acc);
  }
  return cudaGetLastError() == cudaSuccess ? TRIA_OK : TRIA_ERR_CUDA;
}

extern "C" tria_status tria_calib_finish(const double* acc, int64_t n_tokens, int32_t n_q_heads, int32_t head_dim,
                                         int32_t nonrot_dim, float* q_mean, float* q_abs, float* q_nonrot,
                                         void* stream) {
  if (!acc || !q_mean || !q_abs || n_tokens <= 0 || n_q_heads < 1) return TRIA_ERR_INVALID_ARG;
  if (((uintptr_t)acc & 7u) != 0 || !aligned4(q_mean) || !aligned4(q_abs)) return TRIA_ERR_INVALID_ARG;
  if (head_dim < 2 || head_dim % 2 != 0 || head_dim > 2 * kCalibMaxPairs) return TRIA_ERR_UNSUPPORTED;
  if (nonrot_dim < 0 || nonrot_dim % 2 != 0 || nonrot_dim >= head_dim) return TRIA_ERR_INVALID_ARG;
  if (nonrot_dim > 0 && (!q_nonrot || !aligned4(q_nonrot))) return TRIA_ERR_INVALID_ARG;
  const int n = n_q_heads * (head_dim / 2);
  k_calib_finish<<<(n + 255) / 256, 256, 0, (cudaStream_t)stream>>>(
      acc, 1.0 / (double)n_tokens, n_q_heads, head_dim / 2, (head_dim - nonrot_dim) / 2, q_mean, q_abs, q_nonrot);
  return cudaGetLastError() == cudaSuccess ? TRIA_OK : TRIA_ERR_CUDA;
}
