// Selection without a caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they select:
// code running inside a framework's allocator-free region (a captured or
// replayed decode step, a custom memory pool that hands out only the cache and
// its outputs, an embedding runtime that owns every allocation and forbids
// cudaMalloc after start-up). tria_select needs a workspace for its
// per-segment counters, histograms and chunk prefixes; this variant takes that
// scratch from a fixed array that lives in the library's device image instead.
//
// The array is a file-scope static device variable, so every GPU that loads
// the library keeps it for the life of the process. Host code cannot use the
// array's name as a device address (on the host it names a stand-in), so the
// address is obtained once per device with cudaGetSymbolAddress, on the first
// call made while that device is current.
#include <string.h>

#include <mutex>

#include "tria_internal.cuh"

using namespace tria;

namespace {

constexpr size_t kScratchBytes = (size_t)4 << 20;   // 4 MiB, the stated maximum
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_select_scratch[kScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up once).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_select_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

extern "C" tria_status tria_select_noalloc(const float* score, const tria_layer_cache* c, const tria_policy* p,
                                           int32_t* keep_out, void* stream) {
  if (!c || !p || !score || !keep_out) return TRIA_ERR_INVALID_ARG;
  if (c->n_seqs < 1 || c->n_seqs > kMaxSeqs || c->n_kv_heads < 1) return TRIA_ERR_INVALID_ARG;
  if (c->n_seqs * c->n_kv_heads > kMaxSegments) return TRIA_ERR_UNSUPPORTED;
  if (c->head_dim <= 0 || c->head_dim > TRIA_MAX_HEAD_DIM || c->head_dim % 32 != 0) return TRIA_ERR_UNSUPPORTED;
  if (!c->n_live || !c->seq_row0 || !c->capacity) return TRIA_ERR_INVALID_ARG;
  if (((uintptr_t)score % 4) != 0 || ((uintptr_t)keep_out % 4) != 0 || ((uintptr_t)c->n_live % 4) != 0)
    return TRIA_ERR_INVALID_ARG;
  if (p->window < 0 || p->sink < 0) return TRIA_ERR_INVALID_ARG;
  if (!p->budget_rows && (!p->n_ctx || !(p->budget_frac > 0.0) || p->budget_frac > 1.0))
    return TRIA_ERR_INVALID_ARG;

  Pass P;
  memset(&P, 0, sizeof(P));
  int cap_max = 1;
  for (int s = 0; s < c->n_seqs; ++s) {
    if (c->capacity[s] < 0 || c->seq_row0[s] < 0) return TRIA_ERR_INVALID_ARG;
    if (c->capacity[s] > cap_max) cap_max = c->capacity[s];
    int64_t b = p->budget_rows ? (int64_t)p->budget_rows[s] : tria_budget_rows(p->budget_frac, p->n_ctx[s]);
    if (b < 0 || b > INT32_MAX) return TRIA_ERR_INVALID_ARG;
    const int64_t sink = p->sink_rows ? (int64_t)p->sink_rows[s] : (int64_t)p->sink;
    if (sink < 0) return TRIA_ERR_INVALID_ARG;
    if (b < sink + p->window) return TRIA_ERR_BUDGET;
    P.seq[s].row0 = c->seq_row0[s];
    P.seq[s].sink = (int)sink;
    P.seq[s].cap = c->capacity[s];
    P.seq[s].budget = (int)b;
  }
  const int n_seg = c->n_seqs * c->n_kv_heads;
  const int c_max = (cap_max + kChunk - 1) / kChunk;

  // scratch layout: control words, segment states and histograms (must start
  // at zero), then chunk counts and chunk prefixes (fully rewritten each call)
  size_t off = 0;
  const size_t o_ctrl = off;
  off = up256(off + sizeof(Ctrl));
  const size_t o_seg = off;
  off = up256(off + (size_t)n_seg * sizeof(SegState));
  const size_t o_hist = off;
  off = up256(off + (size_t)n_seg * kHistBins * sizeof(uint32_t));
  const size_t zero_bytes = off;
  const size_t o_chunk = off;
  off = up256(off + (size_t)n_seg * c_max * sizeof(SelChunk));
  const size_t o_prefix = off;
  off = up256(off + (size_t)n_seg * (c_max + 1) * sizeof(int32_t));
  if (off > kScratchBytes) return TRIA_ERR_WORKSPACE;   // beyond the fixed scratch size

  void* base = nullptr;
  if (scratch_address(&base) != cudaSuccess) return TRIA_ERR_CUDA;
  cudaStream_t st = (cudaStream_t)stream;
  // the array keeps the previous call's contents: clear counters and histograms
  if (cudaMemsetAsync(base, 0, zero_bytes, st) != cudaSuccess) return TRIA_ERR_CUDA;

  uint8_t* w = (uint8_t*)base;
  P.n_seqs = c->n_seqs;
  P.n_kv = c->n_kv_heads;
  P.n_seg = n_seg;
  P.hd = c->head_dim;
  P.fc = c->head_dim / 2;
  P.window = p->window;
  P.spin_limit = kDefaultSpinLimit;
  P.n_live = c->n_live;
  P.score_in = score;
  P.keep = keep_out;
  P.ctrl = (Ctrl*)(w + o_ctrl);
  P.seg = (SegState*)(w + o_seg);
  P.hist = (uint32_t*)(w + o_hist);
  P.chunk = (SelChunk*)(w + o_chunk);
  P.prefix = (int32_t*)(w + o_prefix);
  P.c_max = c_max;
  P.only_active = 0;
  return launch_select(P, true, st) == cudaSuccess ? TRIA_OK : TRIA_ERR_CUDA;
}
