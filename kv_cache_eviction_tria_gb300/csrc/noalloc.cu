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
// address is looked up with cudaGetSymbolAddress, with the device current, on
// the first call in each CUDA context of that device. The lookup is repeated
// when the current context is a different one (after cudaDeviceReset the
// primary context is new and the old address is no longer valid); contexts
// are told apart by their driver-assigned id.
#include <cuda.h>
#include <string.h>

#include <mutex>

#include "tria_internal.cuh"

using namespace tria;

namespace {

constexpr size_t kScratchBytes = (size_t)4 << 20;   // 4 MiB, the stated maximum
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_select_scratch[kScratchBytes];

struct ScratchSlot {
  unsigned long long ctx_id;   // context the address belongs to (0: none yet)
  void* addr;
};

std::mutex g_setup_mutex;
ScratchSlot g_scratch[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Id of the calling thread's current context, 0 when there is none or the
// driver entry points are unavailable (then every call looks the address up).
unsigned long long current_ctx_id() {
  static CtxGetCurrentFn get_cur = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static bool looked_up = false;
  if (!looked_up) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_cur = reinterpret_cast<CtxGetCurrentFn>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(f);
    looked_up = true;
  }
  if (!get_cur || !get_id) return 0;
  CUcontext ctx = nullptr;
  if (get_cur(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  unsigned long long id = 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of the scratch array in the current context of the current
// device (looked up once per context).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  ScratchSlot& slot = g_scratch[dev];
  const unsigned long long id = current_ctx_id();
  if (id == 0 || slot.ctx_id != id || !slot.addr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_select_scratch);   // also makes the primary context current
    if (e != cudaSuccess) return e;
    slot.addr = p;
    slot.ctx_id = current_ctx_id();
  }
  *out = slot.addr;
  return cudaSuccess;
}

size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

extern "C" tria_status tria_select_noalloc(const float* score, const tria_layer_cache* c, const tria_policy* p,
                                           int32_t* keep_out, void* stream) {
  // the same host checks as tria_select (layout, overlap of sequences,
  // alignment, budget / sink / window of every sequence)
  tria_status r;
  if ((r = check_cache(c)) != TRIA_OK) return r;
  if (!score || !keep_out || ((uintptr_t)score % 4) != 0 || ((uintptr_t)keep_out % 4) != 0)
    return TRIA_ERR_INVALID_ARG;
  std::vector<int> budget;
  if ((r = check_policy(c, p, false, budget)) != TRIA_OK) return r;

  Pass P;
  memset(&P, 0, sizeof(P));
  int cap_max = 1;
  for (int s = 0; s < c->n_seqs; ++s) {
    if (c->capacity[s] > cap_max) cap_max = c->capacity[s];
    P.seq[s].row0 = c->seq_row0[s];
    P.seq[s].sink = p->sink_rows ? p->sink_rows[s] : p->sink;
    P.seq[s].cap = c->capacity[s];
    P.seq[s].budget = budget[s];
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
