// Calibration statistics: upload and load-time folding.
//
// [Doc] "TriAttention KV-Cache Eviction (--triattention)", §2 Calibration file
// (statistics per layer and head of the queries' RoPE directions: the average
// query direction and a weight for each frequency) and §5 Phase C (omega and per-head
// q_mean / q_abs arrays laid out [n_layers x n_heads x freq_count]).
//
// What is folded once at load, per (layer, KV head, group member j, pair f):
//   qe = qbar * E_f,  E_f = (1/|D|) sum_{d in D} e^{i w_f d}
//   mw = q_abs - |qbar|
// so that a pass needs only one phase e^{i w_f p} per pair:
//   mean_d Re(qbar e^{i w (p + d)} conj(k)) = Re(qe e^{i w p} conj(k)).
//
// Non-rotary dims ([Doc] §4 gate line field nonrot=, §6 "Non-rotary models";
// reading: the last nonrot dims of a head are never rotated and the first
// rot = hd - nonrot are NEOX pairs (f, f + rot/2) with w_f = theta^(-2f/rot)):
// the fcr = rot/2 rotary pairs are followed by nonrot/2 content pairs e of
// frequency 0, qe = (qn[e], qn[e + nonrot/2]) and mw = 0, so that every table
// still holds hd/2 pairs and the phase term of a content pair is the mean
// non-rotary query qn dotted with the key dims (rot + e, rot + nonrot/2 + e).
//
// Phase arithmetic: w_f / (2 pi) is stored as a 64-bit fixed-point fraction of
// a turn ("turns"). For an integer position x, turns * x mod 2^64 is the exact
// fractional turn of w_f * x (up to the rounding of w_f / 2pi itself), so no
// floating-point range reduction is needed at any context length.
#include <math.h>

#include <algorithm>
#include <vector>

#include "tria_internal.cuh"

namespace tria {

__global__ void k_stats_freq(int fc, int fcr, double theta, const double* __restrict__ omega_in,
                             const long long* __restrict__ offsets, int n_off,
                             unsigned long long* __restrict__ turns, double2* __restrict__ efold) {
  const int f = blockIdx.x * blockDim.x + threadIdx.x;
  if (f >= fc) return;
  if (f >= fcr) {   // content pair: frequency 0, every offset's phase is 1
    turns[f] = 0ull;
    efold[f] = make_double2(1.0, 0.0);
    return;
  }
  const double w = omega_in ? omega_in[f] : pow(theta, -2.0 * (double)f / (double)(2 * fcr));
  double t = w / (2.0 * 3.14159265358979323846);
  t -= floor(t);                                   // fraction of a turn in [0, 1)
  double scaled = ldexp(t, 64);
  unsigned long long tu = scaled >= 18446744073709551615.0 ? 0ull : (unsigned long long)scaled;
  turns[f] = tu;
  double re = 0.0, im = 0.0;
  for (int i = 0; i < n_off; ++i) {
    const unsigned long long x = tu * (unsigned long long)offsets[i];   // mod 2^64
    const double ang = ldexp((double)(long long)x, -64) * (2.0 * 3.14159265358979323846);
    double s, c;
    sincos(ang, &s, &c);
    re += c;
    im += s;
  }
  efold[f] = make_double2(re / n_off, im / n_off);
}

// q_mean / q_abs: [L][n_q][fcr]; q_nonrot: [L][n_q][2 (fc - fcr)] or NULL
__global__ void k_stats_heads(int L, int n_q, int n_kv, int G, int fc, int fcr, const float* __restrict__ q_mean,
                              const float* __restrict__ q_abs, const float* __restrict__ q_nonrot,
                              const int* __restrict__ head_order, const double2* __restrict__ efold,
                              float2* __restrict__ qe, float* __restrict__ mw) {
  const long long total = (long long)L * n_kv * G * fc;
  const int nr = 2 * (fc - fcr);
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int f = (int)(i % fc);
    const long long t = i / fc;
    const int slot = (int)(t % (n_kv * G));       // g * G + j
    const int l = (int)(t / (n_kv * G));
    const int h = head_order[slot];
    if (f >= fcr) {
      const int e = f - fcr;
      const long long src = ((long long)l * n_q + h) * nr + e;
      qe[i] = q_nonrot ? make_float2(q_nonrot[src], q_nonrot[src + nr / 2]) : make_float2(0.f, 0.f);
      mw[i] = 0.f;
      continue;
    }
    const long long src = ((long long)l * n_q + h) * fcr + f;
    const double a = q_mean[2 * src], b = q_mean[2 * src + 1];
    const double2 e = efold[f];
    qe[i] = make_float2((float)(a * e.x - b * e.y), (float)(a * e.y + b * e.x));
    const double mag = sqrt(a * a + b * b);
    mw[i] = q_abs ? (float)((double)q_abs[src] - mag) : 0.0f;
  }
}

}  // namespace tria

using namespace tria;

namespace {

template <typename T>
cudaError_t upload(T** dst, const T* src, size_t count) {
  *dst = nullptr;
  if (count == 0) return cudaSuccess;
  cudaError_t e = cudaMalloc((void**)dst, count * sizeof(T));
  if (e != cudaSuccess) return e;
  return cudaMemcpy(*dst, src, count * sizeof(T), cudaMemcpyHostToDevice);
}

}  // namespace

extern "C" tria_status tria_load_stats(const tria_stats_desc* d, tria_stats** out, void* stream) {
  if (!out) return TRIA_ERR_INVALID_ARG;
  *out = nullptr;
  if (!d || !d->q_mean || d->n_layers <= 0) return TRIA_ERR_INVALID_ARG;
  const int L = d->n_layers, nq = d->n_q_heads, nkv = d->n_kv_heads;
  if (nq <= 0 || nkv <= 0) return TRIA_ERR_INVALID_ARG;
  if (d->offsets && d->n_offsets <= 0) return TRIA_ERR_INVALID_ARG;
  const int nonrot = d->nonrot_dim;
  if (nonrot < 0 || nonrot % 2 != 0) return TRIA_ERR_INVALID_ARG;

  // per-layer head_dim and theta; a layer is loaded when its head_dim passes
  // the gate ([Doc] §4 GPU scoring requirements, §6 hybrid head_dim models)
  std::vector<int32_t> hd(L);
  std::vector<double> theta(L);
  std::vector<int64_t> src_pairs(L + 1, 0);   // rotary pairs before layer l in q_mean / q_abs (per head)
  int loaded = 0;
  tria_status first_gate = TRIA_OK;
  for (int l = 0; l < L; ++l) {
    hd[l] = d->layer_head_dim ? d->layer_head_dim[l] : d->head_dim;
    theta[l] = d->layer_rope_theta ? d->layer_rope_theta[l] : d->rope_theta;
    if (hd[l] <= nonrot || hd[l] % 2 != 0) return TRIA_ERR_INVALID_ARG;
    if (!d->omega && !(theta[l] > 1.0)) return TRIA_ERR_INVALID_ARG;
    src_pairs[l + 1] = src_pairs[l] + (hd[l] - nonrot) / 2;
    const tria_status g = tria_gate_check(nq, nkv, hd[l], nonrot);
    if (g == TRIA_OK) {
      ++loaded;
    } else if (g == TRIA_ERR_INVALID_ARG || !d->layer_head_dim) {
      return g;   // uniform models keep the whole-model gate
    } else if (first_gate == TRIA_OK) {
      first_gate = g;
    }
  }
  if (loaded == 0) return first_gate == TRIA_OK ? TRIA_ERR_UNSUPPORTED : first_gate;
  const int G = nq / nkv;

  // query heads of each KV head, ascending ([Worklog] "sampled-head mapping")
  std::vector<int> order;
  order.reserve(nq);
  for (int g = 0; g < nkv; ++g) {
    int cnt = 0;
    for (int h = 0; h < nq; ++h) {
      const int kv = d->kv_of_q ? d->kv_of_q[h] : h / G;
      if (kv < 0 || kv >= nkv) return TRIA_ERR_INVALID_ARG;
      if (kv == g) {
        order.push_back(h);
        ++cnt;
      }
    }
    if (cnt != G) return TRIA_ERR_INVALID_ARG;
  }
  std::vector<long long> offs;
  if (d->offsets) {
    offs.assign(d->offsets, d->offsets + d->n_offsets);
  } else {
    for (int j = 0; j <= 16; ++j) offs.push_back(1ll << j);
  }

  tria_stats* s = new tria_stats();
  s->n_layers = L;
  s->n_q_heads = nq;
  s->n_kv_heads = nkv;
  s->group = G;
  s->nonrot_dim = nonrot;
  s->head_dim = hd;
  s->qe_off.assign(L, -1);
  s->turns_off.assign(L, -1);
  // host copy of each layer's frequency definition (the base, or the given
  // frequencies), to check that layers scored in one call share their phases
  s->freq_off.assign(L + 1, 0);
  for (int l = 0; l < L; ++l) {
    if (d->omega) s->freq.insert(s->freq.end(), d->omega + src_pairs[l], d->omega + src_pairs[l + 1]);
    else s->freq.push_back(theta[l]);
    s->freq_off[l + 1] = (int64_t)s->freq.size();
  }
  int64_t n_fold = 0, n_turns = 0;
  int fc_max = 1;
  for (int l = 0; l < L; ++l) {
    if (tria_gate_check(nq, nkv, hd[l], nonrot) != TRIA_OK) continue;
    s->qe_off[l] = n_fold;
    s->turns_off[l] = n_turns;
    n_fold += (int64_t)nkv * G * (hd[l] / 2);
    n_turns += hd[l] / 2;
    fc_max = std::max(fc_max, hd[l] / 2);
  }

  cudaStream_t st = (cudaStream_t)stream;
  float* qm_d = nullptr;
  float* qa_d = nullptr;
  float* qn_d = nullptr;
  double* om_d = nullptr;
  long long* off_d = nullptr;
  int* order_d = nullptr;
  double2* ef_d = nullptr;
  const size_t nqm = (size_t)nq * src_pairs[L];
  auto fail = [&]() {
    cudaFree(qm_d); cudaFree(qa_d); cudaFree(qn_d); cudaFree(om_d); cudaFree(off_d); cudaFree(order_d); cudaFree(ef_d);
    cudaFree(s->qe); cudaFree(s->mw); cudaFree(s->turns);
    delete s;
    return TRIA_ERR_CUDA;
  };
  if ((upload(&qm_d, d->q_mean, 2 * nqm)) != cudaSuccess) return fail();
  if (d->q_abs && (upload(&qa_d, d->q_abs, nqm)) != cudaSuccess) return fail();
  if (nonrot > 0 && d->q_nonrot && (upload(&qn_d, d->q_nonrot, (size_t)L * nq * nonrot)) != cudaSuccess)
    return fail();
  if (d->omega && (upload(&om_d, d->omega, (size_t)src_pairs[L])) != cudaSuccess) return fail();
  if ((upload(&off_d, offs.data(), offs.size())) != cudaSuccess) return fail();
  if ((upload(&order_d, order.data(), order.size())) != cudaSuccess) return fail();
  if ((cudaMalloc((void**)&ef_d, fc_max * sizeof(double2))) != cudaSuccess) return fail();
  if ((cudaMalloc((void**)&s->turns, n_turns * sizeof(unsigned long long))) != cudaSuccess) return fail();
  if ((cudaMalloc((void**)&s->qe, n_fold * sizeof(float2))) != cudaSuccess) return fail();
  if ((cudaMalloc((void**)&s->mw, n_fold * sizeof(float))) != cudaSuccess) return fail();

  // one layer at a time (load time, not the pass): its frequencies, then its
  // folded head weights; the folding buffer is reused in stream order
  for (int l = 0; l < L; ++l) {
    if (s->qe_off[l] < 0) continue;
    const int fc = hd[l] / 2, fcr = (hd[l] - nonrot) / 2;
    const size_t src = (size_t)nq * src_pairs[l];
    k_stats_freq<<<(fc + 127) / 128, 128, 0, st>>>(fc, fcr, theta[l], om_d ? om_d + src_pairs[l] : nullptr,
                                                  off_d, (int)offs.size(), s->turns + s->turns_off[l], ef_d);
    const long long nf = (long long)nkv * G * fc;
    const int blocks = (int)std::min<long long>((nf + 255) / 256, 4096);
    k_stats_heads<<<blocks, 256, 0, st>>>(1, nq, nkv, G, fc, fcr, qm_d + 2 * src, qa_d ? qa_d + src : nullptr,
                                          qn_d ? qn_d + (size_t)l * nq * nonrot : nullptr, order_d, ef_d,
                                          s->qe + s->qe_off[l], s->mw + s->qe_off[l]);
  }
  if ((cudaGetLastError()) != cudaSuccess) return fail();
  if ((cudaStreamSynchronize(st)) != cudaSuccess) return fail();
  cudaFree(qm_d);
  cudaFree(qa_d);
  cudaFree(qn_d);
  cudaFree(om_d);
  cudaFree(off_d);
  cudaFree(order_d);
  cudaFree(ef_d);
  *out = s;
  return TRIA_OK;
}

extern "C" void tria_free_stats(tria_stats* s) {
  if (!s) return;
  cudaFree(s->qe);
  cudaFree(s->mw);
  cudaFree(s->turns);
  delete s;
}
