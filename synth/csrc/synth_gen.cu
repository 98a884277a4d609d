// Device form of the seeded cache generator (see synth/counter_rng.py).
//
// Bit-identical to the host form: SplitMix64 words, the sum of twelve 16-bit
// uniforms minus its mean scaled by 2^-16 (exact in float32), exact
// power-of-two outlier scaling, then the cache write: float16 round to nearest
// even, or q8_0 quantisation with IEEE float32 division and round half away
// from zero. No eviction arithmetic lives here.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

constexpr unsigned long long kGamma = 0x9E3779B97F4A7C15ull;
constexpr unsigned long long kM1 = 0xBF58476D1CE4E5B9ull;
constexpr unsigned long long kM2 = 0x94D049BB133111EBull;

__host__ __device__ inline unsigned long long mix64(unsigned long long z) {
  z = (z ^ (z >> 30)) * kM1;
  z = (z ^ (z >> 27)) * kM2;
  return z ^ (z >> 31);
}

__host__ __device__ inline unsigned long long stream_key(int seed, int tensor, int layer, int seq, int head) {
  unsigned long long k = mix64((unsigned long long)(seed + 1) * kGamma);
  k = mix64(k + (unsigned long long)(tensor + 1) * kGamma);
  k = mix64(k + (unsigned long long)(layer + 1) * kGamma);
  k = mix64(k + (unsigned long long)(seq + 1) * kGamma);
  k = mix64(k + (unsigned long long)(head + 1) * kGamma);
  return k;
}

__device__ inline float normal12(unsigned long long key, unsigned long long j) {
  int s = 0;
#pragma unroll
  for (int t = 0; t < 3; ++t) {
    const unsigned long long w = mix64(key + (3ull * j + (unsigned long long)t + 1ull) * kGamma);
    s += (int)(w & 0xFFFFull) + (int)((w >> 16) & 0xFFFFull) + (int)((w >> 32) & 0xFFFFull) + (int)(w >> 48);
  }
  return (float)(s - 393210) * (1.0f / 65536.0f);
}

struct SeqDesc {
  long long row0;
  int cap;
  int pad;
};

constexpr int kMaxSeqs = 128;

struct FillArgs {
  int n_seqs, n_kv, hd, k_type, v_type, seed, layer, pos_arange;
  const float* pair_scale;  // [n_kv][hd/2]
  uint8_t* k;
  uint8_t* ks;
  uint8_t* v;
  int* pos;
  SeqDesc seq[kMaxSeqs];
  long long units_prefix[kMaxSeqs + 1];  // 32-wide units before each sequence
};

// one thread = one 32-wide block of one row of one segment
__global__ void k_fill(const __grid_constant__ FillArgs A) {
  const long long total = A.units_prefix[A.n_seqs];
  const int blocks_per_row = A.hd / 32;
  for (long long u = blockIdx.x * (long long)blockDim.x + threadIdx.x; u < total;
       u += (long long)gridDim.x * blockDim.x) {
    int s = 0;
    while (u >= A.units_prefix[s + 1]) ++s;
    const long long local = u - A.units_prefix[s];
    const long long per_head = (long long)A.seq[s].cap * blocks_per_row;
    const int g = (int)(local / per_head);
    const long long rem = local - (long long)g * per_head;
    const int r = (int)(rem / blocks_per_row);
    const int b = (int)(rem - (long long)r * blocks_per_row);
    const long long row = A.seq[s].row0 + (long long)g * A.seq[s].cap + r;
    const unsigned long long kkey = stream_key(A.seed, 1, A.layer, s, g);
    const unsigned long long vkey = stream_key(A.seed, 2, A.layer, s, g);
    const int fc = A.hd / 2;
    float x[32];
#pragma unroll 4
    for (int i = 0; i < 32; ++i) {
      const int d = b * 32 + i;
      const float sc = A.pair_scale ? A.pair_scale[g * fc + (d % fc)] : 1.0f;
      x[i] = normal12(kkey, (unsigned long long)r * A.hd + d) * sc;
    }
    if (A.k_type == 1) {
      __half* kp = reinterpret_cast<__half*>(A.k) + row * A.hd + b * 32;
#pragma unroll
      for (int i = 0; i < 32; ++i) kp[i] = __float2half_rn(x[i]);
    } else if (A.k_type == 0) {
      float* kp = reinterpret_cast<float*>(A.k) + row * A.hd + b * 32;
#pragma unroll
      for (int i = 0; i < 32; ++i) kp[i] = x[i];
    } else {
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(x[i]));
      const float dd = __fdiv_rn(amax, 127.0f);
      int8_t* qp = reinterpret_cast<int8_t*>(A.k) + row * A.hd + b * 32;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        float q = 0.f;
        if (dd > 0.f) q = fminf(127.f, fmaxf(-127.f, roundf(__fdiv_rn(x[i], dd))));
        qp[i] = (int8_t)(int)q;
      }
      reinterpret_cast<__half*>(A.ks)[row * blocks_per_row + b] = __float2half_rn(dd);
    }
#pragma unroll 4
    for (int i = 0; i < 32; ++i) x[i] = normal12(vkey, (unsigned long long)r * A.hd + b * 32 + i);
    if (A.v_type == 1) {
      __half* vp = reinterpret_cast<__half*>(A.v) + row * A.hd + b * 32;
#pragma unroll
      for (int i = 0; i < 32; ++i) vp[i] = __float2half_rn(x[i]);
    } else {
      float* vp = reinterpret_cast<float*>(A.v) + row * A.hd + b * 32;
#pragma unroll
      for (int i = 0; i < 32; ++i) vp[i] = x[i];
    }
    if (A.pos && A.pos_arange && b == 0) A.pos[row] = r;
  }
}

}  // namespace

// Fill one layer's cache. Host arrays: seq_row0 [n_seqs], capacity [n_seqs].
// Device: pair_scale [n_kv][hd/2] (or NULL), k, k_scale (q8_0), v, pos (or NULL).
// Returns a cudaError_t value.
extern "C" int synth_fill_layer(int n_seqs, int n_kv, int hd, int k_type, int v_type, int seed, int layer,
                                const long long* seq_row0, const int* capacity, const float* pair_scale,
                                void* k, void* k_scale, void* v, int* pos, int pos_arange, void* stream) {
  if (n_seqs < 1 || n_seqs > kMaxSeqs || hd % 32 != 0) return (int)cudaErrorInvalidValue;
  FillArgs A{};
  A.n_seqs = n_seqs;
  A.n_kv = n_kv;
  A.hd = hd;
  A.k_type = k_type;
  A.v_type = v_type;
  A.seed = seed;
  A.layer = layer;
  A.pos_arange = pos_arange;
  A.pair_scale = pair_scale;
  A.k = (uint8_t*)k;
  A.ks = (uint8_t*)k_scale;
  A.v = (uint8_t*)v;
  A.pos = pos;
  A.units_prefix[0] = 0;
  for (int s = 0; s < n_seqs; ++s) {
    A.seq[s].row0 = seq_row0[s];
    A.seq[s].cap = capacity[s];
    A.units_prefix[s + 1] = A.units_prefix[s] + (long long)n_kv * capacity[s] * (hd / 32);
  }
  const long long total = A.units_prefix[n_seqs];
  long long blocks = (total + 255) / 256;
  if (blocks > 152 * 64) blocks = 152 * 64;
  if (blocks < 1) blocks = 1;
  k_fill<<<(int)blocks, 256, 0, (cudaStream_t)stream>>>(A);
  return (int)cudaGetLastError();
}
