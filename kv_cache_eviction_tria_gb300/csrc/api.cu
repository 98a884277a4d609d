// C ABI of the eviction pass: argument checks, workspace layout, launches.
//
// Sources cited by page title and section:
//   [Worklog] "TriAttention Native C++ Worklog"
//   [Doc]     "TriAttention KV-Cache Eviction (--triattention)"
#include <math.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <vector>

#include "pass.cuh"

using namespace tria;

namespace {

int row_bytes(tria_dtype t, int hd) {
  switch (t) {
    case TRIA_F32: return 4 * hd;
    case TRIA_F16: return 2 * hd;
    case TRIA_Q8_0: return hd;
  }
  return 0;
}

int scale_row_bytes(tria_dtype t, int hd) { return t == TRIA_Q8_0 ? hd / 16 : 0; }

bool dtype_ok(int t) { return t == TRIA_F32 || t == TRIA_F16 || t == TRIA_Q8_0; }

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

struct Layout {
  size_t ctrl, pass_ctl, seg, runs, chunk, prefix, hist, flags, score, keep, raw, total;
  int cs_rows, cs_max, c_max, n_seg;
  int64_t total_rows;       // rows of one layer
};

size_t up(size_t x) { return (x + 255) & ~(size_t)255; }

// Workspace layout of the single-layer calls on `cache`. Everything but `raw`
// is independent of the group size, and `raw` comes last, so one workspace
// serves every entry point on the same cache. The control words and the fused
// pass's fixed state come first.
Layout make_layout(const tria_layer_cache* c, int G) {
  Layout L{};
  const int hd = c->head_dim;
  const int k_rb = row_bytes(c->k_type, hd);
  L.cs_rows = 0;
  int cap_max = 0;
  int64_t total_rows = 0;
  for (int s = 0; s < c->n_seqs; ++s) {
    cap_max = std::max(cap_max, c->capacity[s]);
    total_rows = std::max(total_rows, c->seq_row0[s] + (int64_t)c->n_kv_heads * c->capacity[s]);
  }
  cap_max = std::max(cap_max, 1);
  L.total_rows = total_rows;
  L.n_seg = c->n_seqs * c->n_kv_heads;
  L.cs_max = score_pieces_max(k_rb, cap_max);
  L.c_max = (cap_max + kChunk - 1) / kChunk;
  size_t off = 0;
  L.ctrl = off;
  off = up(off + sizeof(Ctrl));
  L.pass_ctl = off;
  off = up(off + sizeof(PassCtl));
  L.seg = off;
  off = up(off + (size_t)L.n_seg * sizeof(SegState));
  L.runs = off;
  off = up(off + (size_t)L.n_seg * kRunCols * L.cs_max * sizeof(float));
  L.chunk = off;
  off = up(off + (size_t)L.n_seg * L.c_max * sizeof(SelChunk));
  L.prefix = off;
  off = up(off + (size_t)L.n_seg * (L.c_max + 1) * sizeof(int32_t));
  L.hist = off;
  off = up(off + (size_t)L.n_seg * kHistBins * sizeof(uint32_t));
  L.flags = off;
  off = up(off + (size_t)L.n_seg * L.c_max * sizeof(uint32_t));
  L.score = off;
  off = up(off + (size_t)total_rows * sizeof(float));
  L.keep = off;
  off = up(off + (size_t)total_rows * sizeof(int32_t));
  L.raw = off;
  off = up(off + (size_t)total_rows * std::max(G, 0) * sizeof(float));
  L.total = off;
  return L;
}

// Layout of a fused pass over n_layers > 1 layers: the single-layer layout
// (so that every single-layer call on one of the layers fits and finds its
// state where it left it), then the pass's own tables for all layers'
// segments and rows (item moment partials, chunk prefixes, read-done flags,
// keys, keep lists, raw scores).
Layout make_model_layout(const tria_layer_cache* c, int G, int n_layers) {
  const Layout L1 = make_layout(c, G);
  if (n_layers <= 1) return L1;
  Layout L = L1;
  const int k_rb = row_bytes(c->k_type, c->head_dim);
  const int cap_max = L1.c_max * kChunk;
  // score runs of a segment: at most one per warp of the grid, plus one
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms = 1024;
  const int piece_rows = pass_piece_rows(k_rb);
  L.n_seg = n_layers * L1.n_seg;
  L.cs_max = std::min((cap_max + piece_rows - 1) / piece_rows, kPassWarps * sms + 2);
  const int64_t rows = L1.total_rows * n_layers;
  size_t off = L1.total;
  L.runs = off;
  off = up(off + (size_t)L.n_seg * kRunCols * L.cs_max * sizeof(float));
  L.prefix = off;
  off = up(off + (size_t)L.n_seg * (L.c_max + 1) * sizeof(int32_t));
  L.flags = off;
  off = up(off + (size_t)L.n_seg * L.c_max * sizeof(uint32_t));
  L.score = off;
  off = up(off + (size_t)rows * sizeof(float));
  L.keep = off;
  off = up(off + (size_t)rows * sizeof(int32_t));
  L.raw = off;
  off = up(off + (size_t)rows * std::max(G, 0) * sizeof(float));
  L.total = off;
  L.seg = L.chunk = L.hist = 0;   // not used by the pass
  return L;
}

tria_status check_ws(void* ws, size_t ws_bytes, const Layout& L) {
  if (!ws || !aligned(ws, 256)) return TRIA_ERR_WORKSPACE;
  if (ws_bytes < L.total) return TRIA_ERR_WORKSPACE;
  return TRIA_OK;
}

void fill_pass(Pass& P, const tria_layer_cache* c, const tria_policy* p, const std::vector<int>& budget,
               const Layout& L, void* ws, int G) {
  memset(&P, 0, sizeof(P));
  P.n_seqs = c->n_seqs;
  P.n_kv = c->n_kv_heads;
  P.n_seg = L.n_seg;
  P.G = G;
  P.hd = c->head_dim;
  P.fc = c->head_dim / 2;
  P.fcr = P.fc;
  P.window = p ? p->window : 0;
  P.k_type = c->k_type;
  P.v_type = c->v_type;
  P.k_rb = row_bytes(c->k_type, c->head_dim);
  P.ks_rb = scale_row_bytes(c->k_type, c->head_dim);
  P.v_rb = row_bytes(c->v_type, c->head_dim);
  P.vs_rb = scale_row_bytes(c->v_type, c->head_dim);
  P.spin_limit = kDefaultSpinLimit;
  P.k = (uint8_t*)c->k;
  P.ks = (uint8_t*)c->k_scale;
  P.v = (uint8_t*)c->v;
  P.vs = (uint8_t*)c->v_scale;
  P.pos = c->pos;
  P.n_live = c->n_live;
  uint8_t* w = (uint8_t*)ws;
  P.ctrl = (Ctrl*)(w + L.ctrl);
  P.seg = (SegState*)(w + L.seg);
  P.runs = (float*)(w + L.runs);
  P.chunk = (SelChunk*)(w + L.chunk);
  P.prefix = (int32_t*)(w + L.prefix);
  P.hist = (uint32_t*)(w + L.hist);
  P.flags = (uint32_t*)(w + L.flags);
  P.cs_rows = L.cs_rows;
  P.cs_max = L.cs_max;
  P.c_max = L.c_max;
  for (int s = 0; s < c->n_seqs; ++s) {
    P.seq[s].row0 = c->seq_row0[s];
    P.seq[s].cap = c->capacity[s];
    P.seq[s].budget = budget.empty() ? 0 : budget[s];
    P.seq[s].cur_pos = (p && p->cur_pos) ? p->cur_pos[s] : 0;
    P.seq[s].sink = !p ? 0 : (p->sink_rows ? p->sink_rows[s] : p->sink);
  }
}

tria_status cuda_status(cudaError_t e) { return e == cudaSuccess ? TRIA_OK : TRIA_ERR_CUDA; }

tria_status check_stats(const tria_stats* st, int layer, const tria_layer_cache* c) {
  if (!st) return TRIA_ERR_INVALID_ARG;
  if (layer < 0 || layer >= st->n_layers) return TRIA_ERR_INVALID_ARG;
  if (st->n_kv_heads != c->n_kv_heads || st->head_dim[layer] != c->head_dim) return TRIA_ERR_INVALID_ARG;
  if (st->qe_off[layer] < 0) return TRIA_ERR_UNSUPPORTED;   // layer not loaded (fails the gate)
  return TRIA_OK;
}

void set_stats(Pass& P, const tria_stats* st, int layer) {
  P.qe = st->qe;
  P.mw = st->mw;
  P.turns = st->turns + st->turns_off[layer];
  P.fcr = (P.hd - st->nonrot_dim) / 2;
  for (int s = 0; s < P.n_seqs; ++s) P.seq[s].qe_off = (int32_t)st->qe_off[layer];
}

// The fused pass (k_pass) over layers[0 .. n_layers) of the statistics, one
// cache per layer (same sequences, shapes and types; checked by the caller).
tria_status launch_fused(const tria_stats* st, const int32_t* layers, int n_layers, const tria_layer_cache* caches,
                         const tria_policy* p, const std::vector<int>& budget, const Layout& L, void* ws,
                         float* score_out, cudaStream_t stream) {
  const tria_layer_cache* c = caches;
  FPass* F = new FPass;   // ~12 KB: off the stack
  memset(F, 0, sizeof(FPass));
  F->n_layers = n_layers;
  F->n_seqs = c->n_seqs;
  F->n_kv = c->n_kv_heads;
  F->n_seg = L.n_seg;
  F->G = st->group;
  F->hd = c->head_dim;
  F->fc = c->head_dim / 2;
  F->window = p->window;
  F->k_rb = row_bytes(c->k_type, c->head_dim);
  F->ks_rb = scale_row_bytes(c->k_type, c->head_dim);
  F->v_rb = row_bytes(c->v_type, c->head_dim);
  F->vs_rb = scale_row_bytes(c->v_type, c->head_dim);
  F->spin_limit = kDefaultSpinLimit;
  F->piece_rows = pass_piece_rows(F->k_rb);
  F->cs_max = L.cs_max;
  F->c_max = L.c_max;
  F->rows_per_layer = L.total_rows;
  F->qe = st->qe;
  F->mw = st->mw;
  F->turns = st->turns + st->turns_off[layers[0]];
  uint8_t* w = (uint8_t*)ws;
  F->raw = (float*)(w + L.raw);
  F->keys = (uint32_t*)(w + L.score);
  F->score_out = score_out;
  F->keep = (int32_t*)(w + L.keep);
  F->ctrl = (Ctrl*)(w + L.ctrl);
  F->ctl = (PassCtl*)(w + L.pass_ctl);
  F->parts = (float*)(w + L.runs);
  F->prefix = (int32_t*)(w + L.prefix);
  F->flags = (uint32_t*)(w + L.flags);
  for (int s = 0; s < c->n_seqs; ++s) {
    F->seq[s].row0 = c->seq_row0[s];
    F->seq[s].cap = c->capacity[s];
    F->seq[s].budget = budget[s];
    F->seq[s].cur_pos = p->cur_pos[s];
    F->seq[s].sink = p->sink_rows ? p->sink_rows[s] : p->sink;
  }
  for (int i = 0; i < n_layers; ++i) {
    F->lay[i].k = (uint8_t*)caches[i].k;
    F->lay[i].ks = (uint8_t*)caches[i].k_scale;
    F->lay[i].v = (uint8_t*)caches[i].v;
    F->lay[i].vs = (uint8_t*)caches[i].v_scale;
    F->lay[i].pos = caches[i].pos;
    F->lay[i].n_live = caches[i].n_live;
    F->lay[i].qe_off = st->qe_off[layers[i]];
  }
  const cudaError_t e = c->k_type == TRIA_F16 ? launch_pass_f16(*F, stream) : launch_pass_q8(*F, stream);
  delete F;
  return cuda_status(e);
}

// The fused kernel scores all-rotary heads only (heads with non-rotary dims
// take the staged kernels).
bool fused_ok(const tria_stats* st, const tria_layer_cache* c, int n_layers) {
  return st->nonrot_dim == 0 && pass_supported(c->k_type, c->head_dim, st->group) && n_layers >= 1 &&
         n_layers <= kPassMaxLayers &&
         (int64_t)n_layers * c->n_seqs * c->n_kv_heads <= kPassMaxSegs;
}

// The fused kernel pays the staged path's ramps and launch gaps once, but
// selects each segment on one CTA (the staged select uses an 8-CTA cluster)
// and moves the rows only once every segment is selected. Measured on GB300
// (whole-model steps): it is ahead from 128 segments on whatever their
// length (4 long-context layers of 32 segments of 35K-112K rows: 2.03 against
// 2.14 ms; 16 q8_0 layers: 1.15 against 1.55 ms), and from 32 segments on
// when no segment holds more than 65536 rows (4 Qwen3-8B steady-state layers:
// 0.10 against 0.16 ms; 4 q8_0 layers of 65536 rows: even); with a few long
// segments the staged kernels are faster (one Qwen3-8B layer of 8 x 32768
// rows: 61 against 111 us; one long-context layer: 0.53 against 0.68 ms).
constexpr int kFusedMinSegs = 128;
constexpr int kFusedMinShortSegs = 32;
constexpr int kFusedShortRows = 65536;
bool fused_preferred(const tria_stats* st, const tria_layer_cache* c, int n_layers) {
  if (!fused_ok(st, c, n_layers)) return false;
  const int64_t segs = (int64_t)n_layers * c->n_seqs * c->n_kv_heads;
  int cap_max = 0;
  for (int s = 0; s < c->n_seqs; ++s) cap_max = std::max(cap_max, c->capacity[s]);
  return segs >= kFusedMinSegs || (segs >= kFusedMinShortSegs && cap_max <= kFusedShortRows);
}

}  // namespace

namespace tria {

tria_status check_cache(const tria_layer_cache* c) {
  if (!c) return TRIA_ERR_INVALID_ARG;
  if (c->n_seqs < 1 || c->n_seqs > kMaxSeqs || c->n_kv_heads < 1) return TRIA_ERR_INVALID_ARG;
  if (c->n_seqs * c->n_kv_heads > kMaxSegments) return TRIA_ERR_UNSUPPORTED;
  const int hd = c->head_dim;
  if (hd <= 0 || hd > TRIA_MAX_HEAD_DIM || hd % 32 != 0) return TRIA_ERR_UNSUPPORTED;
  if (!dtype_ok(c->k_type) || !dtype_ok(c->v_type)) return TRIA_ERR_UNSUPPORTED;
  if (!c->k || !c->v || !c->pos || !c->n_live || !c->seq_row0 || !c->capacity) return TRIA_ERR_INVALID_ARG;
  if (!aligned(c->k, 16) || !aligned(c->v, 16) || !aligned(c->pos, 4) || !aligned(c->n_live, 4))
    return TRIA_ERR_INVALID_ARG;
  if ((c->k_type == TRIA_Q8_0) != (c->k_scale != nullptr)) return TRIA_ERR_INVALID_ARG;
  if ((c->v_type == TRIA_Q8_0) != (c->v_scale != nullptr)) return TRIA_ERR_INVALID_ARG;
  if (c->k_scale && !aligned(c->k_scale, 16)) return TRIA_ERR_INVALID_ARG;
  if (c->v_scale && !aligned(c->v_scale, 16)) return TRIA_ERR_INVALID_ARG;
  // segments of different sequences must not overlap
  std::vector<std::pair<int64_t, int64_t>> spans;
  for (int s = 0; s < c->n_seqs; ++s) {
    if (c->capacity[s] < 0 || c->seq_row0[s] < 0) return TRIA_ERR_INVALID_ARG;
    spans.push_back({c->seq_row0[s], c->seq_row0[s] + (int64_t)c->n_kv_heads * c->capacity[s]});
  }
  std::sort(spans.begin(), spans.end());
  for (size_t i = 1; i < spans.size(); ++i)
    if (spans[i].first < spans[i - 1].second) return TRIA_ERR_INVALID_ARG;
  return TRIA_OK;
}

// need_budget = false (scoring only): the budget is not used and not checked.
tria_status check_policy(const tria_layer_cache* c, const tria_policy* p, bool need_pos, std::vector<int>& budget,
                         bool need_budget) {
  if (!p) return TRIA_ERR_INVALID_ARG;
  if (p->window < 0 || p->sink < 0) return TRIA_ERR_INVALID_ARG;
  if (need_pos && !p->cur_pos) return TRIA_ERR_INVALID_ARG;
  if (!need_budget) {
    budget.assign(c->n_seqs, 0);
    for (int s = 0; s < c->n_seqs; ++s)
      if (need_pos && p->cur_pos[s] < 0) return TRIA_ERR_INVALID_ARG;
    return TRIA_OK;
  }
  if (!p->budget_rows && (!p->n_ctx || !(p->budget_frac > 0.0) || p->budget_frac > 1.0))
    return TRIA_ERR_INVALID_ARG;
  budget.assign(c->n_seqs, 0);
  for (int s = 0; s < c->n_seqs; ++s) {
    int64_t b;
    if (p->budget_rows) {
      b = p->budget_rows[s];
    } else {
      if (p->n_ctx[s] < 0) return TRIA_ERR_INVALID_ARG;
      b = tria_budget_rows(p->budget_frac, p->n_ctx[s]);
    }
    if (b < 0 || b > INT32_MAX) return TRIA_ERR_INVALID_ARG;
    const int64_t sink = p->sink_rows ? (int64_t)p->sink_rows[s] : (int64_t)p->sink;
    if (sink < 0) return TRIA_ERR_INVALID_ARG;
    if (b < sink + p->window) return TRIA_ERR_BUDGET;
    if (need_pos && p->cur_pos[s] < 0) return TRIA_ERR_INVALID_ARG;
    budget[s] = (int)b;
  }
  return TRIA_OK;
}

}  // namespace tria

// ---------------------------------------------------------------------------

extern "C" tria_status tria_gate_check(int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim,
                                       int32_t nonrot_dim) {
  if (n_q_heads <= 0 || n_kv_heads <= 0 || head_dim <= 0) return TRIA_ERR_INVALID_ARG;
  if (nonrot_dim < 0 || nonrot_dim >= head_dim) return TRIA_ERR_INVALID_ARG;
  if (n_q_heads % n_kv_heads != 0) return TRIA_ERR_UNSUPPORTED;          // [Doc] §4: nh % nkv == 0
  if (head_dim > TRIA_MAX_HEAD_DIM || head_dim % 32 != 0) return TRIA_ERR_UNSUPPORTED;  // hd <= 256, % 32
  const int G = n_q_heads / n_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8) return TRIA_ERR_UNSUPPORTED;
  // the scorers take a lane's rotary pairs in whole runs of 8
  if ((head_dim - nonrot_dim) % 16 != 0) return TRIA_ERR_UNSUPPORTED;
  return TRIA_OK;
}

extern "C" tria_status tria_gate_describe(int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim,
                                          int32_t nonrot_dim, tria_dtype k_type, char* buf, size_t buf_size) {
  const tria_status g = tria_gate_check(n_q_heads, n_kv_heads, head_dim, nonrot_dim);
  if (!buf || buf_size == 0) return g;
  const char* why = "";
  if (g == TRIA_ERR_INVALID_ARG) {
    why = n_q_heads <= 0 || n_kv_heads <= 0 || head_dim <= 0 ? " (heads / head_dim must be > 0)"
                                                            : " (nonrot must be in [0, head_dim))";
  } else if (g == TRIA_ERR_UNSUPPORTED) {
    if (n_q_heads % n_kv_heads != 0) why = " (nh % nkv != 0)";
    else if (head_dim > TRIA_MAX_HEAD_DIM) why = " (head_dim > 256)";
    else if (head_dim % 32 != 0) why = " (head_dim % 32 != 0)";
    else if ((head_dim - nonrot_dim) % 16 != 0) why = " (rotary dims % 16 != 0)";
    else why = " (group size not 1, 2, 4 or 8)";
  }
  snprintf(buf, buf_size, "tria: gpu gate - is_q8_0=%d nh=%d nkv=%d hd=%d nonrot=%d -> %s%s",
           k_type == TRIA_Q8_0 ? 1 : 0, (int)n_q_heads, (int)n_kv_heads, (int)head_dim, (int)nonrot_dim,
           g == TRIA_OK ? "eligible" : "ineligible", why);
  return g;
}

extern "C" int64_t tria_budget_rows(double budget_frac, int64_t n_ctx) {
  return (int64_t)floor(budget_frac * (double)n_ctx);
}

extern "C" int32_t tria_should_evict(int64_t n_live, int64_t budget, int64_t interval) {
  return n_live >= budget + interval ? 1 : 0;
}

extern "C" size_t tria_workspace_size(const tria_layer_cache* cache, int32_t group) {
  if (check_cache(cache) != TRIA_OK || group < 0 || group > kMaxG) return 0;
  return make_layout(cache, group).total;
}

extern "C" tria_status tria_workspace_init(void* ws, size_t ws_bytes, void* stream) {
  if (!ws || !aligned(ws, 256) || ws_bytes < sizeof(Ctrl)) return TRIA_ERR_WORKSPACE;
  return cuda_status(cudaMemsetAsync(ws, 0, ws_bytes, (cudaStream_t)stream));
}

extern "C" tria_status tria_score(const tria_stats* stats, int32_t layer, const tria_layer_cache* cache,
                                  const tria_policy* policy, float* score_out, float* raw_out, void* ws,
                                  size_t ws_bytes, void* stream) {
  tria_status r;
  if ((r = check_cache(cache)) != TRIA_OK) return r;
  if ((r = check_stats(stats, layer, cache)) != TRIA_OK) return r;
  if (!score_out || !aligned(score_out, 4) || (raw_out && !aligned(raw_out, 4))) return TRIA_ERR_INVALID_ARG;
  std::vector<int> budget;
  if ((r = check_policy(cache, policy, true, budget, false)) != TRIA_OK) return r;
  const Layout L = make_layout(cache, stats->group);
  if ((r = check_ws(ws, ws_bytes, L)) != TRIA_OK) return r;
  Pass P;
  fill_pass(P, cache, policy, budget, L, ws, stats->group);
  set_stats(P, stats, layer);
  P.only_active = 0;
  P.raw = raw_out ? raw_out : (float*)((uint8_t*)ws + L.raw);
  P.score = score_out;
  cudaStream_t st = (cudaStream_t)stream;
  if ((r = cuda_status(launch_score(P, st))) != TRIA_OK) return r;
  return cuda_status(launch_zscore(P, st));
}

extern "C" tria_status tria_select(const float* score, const tria_layer_cache* cache, const tria_policy* policy,
                                   int32_t* keep_out, void* ws, size_t ws_bytes, void* stream) {
  tria_status r;
  if ((r = check_cache(cache)) != TRIA_OK) return r;
  if (!score || !keep_out || !aligned(score, 4) || !aligned(keep_out, 4)) return TRIA_ERR_INVALID_ARG;
  std::vector<int> budget;
  if ((r = check_policy(cache, policy, false, budget)) != TRIA_OK) return r;
  const Layout L = make_layout(cache, 0);
  if ((r = check_ws(ws, ws_bytes, L)) != TRIA_OK) return r;
  Pass P;
  fill_pass(P, cache, policy, budget, L, ws, 0);
  P.only_active = 0;
  P.score_in = score;
  P.keep = keep_out;
  return cuda_status(launch_select(P, true, (cudaStream_t)stream));
}

extern "C" tria_status tria_shared_combine(const float* scores, int64_t layer_stride, int32_t n_layers,
                                           const tria_layer_cache* cache, float* combined, void* ws,
                                           size_t ws_bytes, void* stream) {
  tria_status r;
  if ((r = check_cache(cache)) != TRIA_OK) return r;
  if (!scores || !combined || !aligned(scores, 4) || !aligned(combined, 4) || n_layers < 1) return TRIA_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, 256) || ws_bytes < sizeof(Ctrl)) return TRIA_ERR_WORKSPACE;
  const Layout L = make_layout(cache, 0);
  if (layer_stride < L.total_rows) return TRIA_ERR_INVALID_ARG;   // layers must not overlap
  Pass P;
  fill_pass(P, cache, nullptr, {}, L, ws, 0);
  return cuda_status(launch_shared_combine(P, scores, layer_stride, n_layers, combined, (cudaStream_t)stream));
}

extern "C" tria_status tria_shared_select(const float* combined, const tria_layer_cache* cache,
                                          const tria_policy* policy, int32_t* keep_out, void* ws, size_t ws_bytes,
                                          void* stream) {
  tria_status r;
  if ((r = check_cache(cache)) != TRIA_OK) return r;
  if (!combined || !keep_out || !aligned(combined, 4) || !aligned(keep_out, 4)) return TRIA_ERR_INVALID_ARG;
  std::vector<int> budget;
  if ((r = check_policy(cache, policy, false, budget)) != TRIA_OK) return r;
  // the selection runs on the KV-head-0 slot of every sequence
  tria_layer_cache view = *cache;
  view.n_kv_heads = 1;
  const Layout L = make_layout(&view, 0);
  if ((r = check_ws(ws, ws_bytes, L)) != TRIA_OK) return r;
  Pass P;
  fill_pass(P, &view, policy, budget, L, ws, 0);
  P.only_active = 0;
  P.score_in = combined;
  P.keep = keep_out;
  cudaStream_t st = (cudaStream_t)stream;
  if ((r = cuda_status(launch_select(P, true, st))) != TRIA_OK) return r;
  if (cache->n_kv_heads == 1) return TRIA_OK;
  Pass B;
  fill_pass(B, cache, policy, budget, make_layout(cache, 0), ws, 0);
  return cuda_status(launch_shared_broadcast(B, keep_out, st));
}

extern "C" tria_status tria_append(const tria_layer_cache* cache, const void* k_new, const void* k_scale_new,
                                   const void* v_new, const void* v_scale_new, const int32_t* pos_new,
                                   int32_t n_tokens, void* ws, size_t ws_bytes, void* stream) {
  tria_status r;
  if ((r = check_cache(cache)) != TRIA_OK) return r;
  if (n_tokens < 0) return TRIA_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, 256) || ws_bytes < sizeof(Ctrl)) return TRIA_ERR_WORKSPACE;
  if (n_tokens == 0) return TRIA_OK;
  if (!k_new || !v_new || !pos_new) return TRIA_ERR_INVALID_ARG;
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(pos_new, 4)) return TRIA_ERR_INVALID_ARG;
  if ((cache->k_type == TRIA_Q8_0) != (k_scale_new != nullptr)) return TRIA_ERR_INVALID_ARG;
  if ((cache->v_type == TRIA_Q8_0) != (v_scale_new != nullptr)) return TRIA_ERR_INVALID_ARG;
  if ((k_scale_new && !aligned(k_scale_new, 2)) || (v_scale_new && !aligned(v_scale_new, 2)))
    return TRIA_ERR_INVALID_ARG;
  const Layout L = make_layout(cache, 0);
  Pass P;
  fill_pass(P, cache, nullptr, {}, L, ws, 0);
  AppendSrc a;
  a.k = (const uint8_t*)k_new;
  a.ks = (const uint8_t*)k_scale_new;
  a.v = (const uint8_t*)v_new;
  a.vs = (const uint8_t*)v_scale_new;
  a.pos = pos_new;
  a.n_tokens = n_tokens;
  return cuda_status(launch_append(P, a, (cudaStream_t)stream));
}

extern "C" tria_status tria_compact(const tria_layer_cache* cache, const tria_policy* policy, const int32_t* keep,
                                    void* ws, size_t ws_bytes, void* stream) {
  tria_status r;
  if ((r = check_cache(cache)) != TRIA_OK) return r;
  if (!keep || !aligned(keep, 4)) return TRIA_ERR_INVALID_ARG;
  std::vector<int> budget;
  if ((r = check_policy(cache, policy, false, budget)) != TRIA_OK) return r;
  const Layout L = make_layout(cache, 0);
  if ((r = check_ws(ws, ws_bytes, L)) != TRIA_OK) return r;
  Pass P;
  fill_pass(P, cache, policy, budget, L, ws, 0);
  P.only_active = 1;
  P.keep = const_cast<int32_t*>(keep);
  cudaStream_t st = (cudaStream_t)stream;
  if ((r = cuda_status(launch_keep_prepass(P, st))) != TRIA_OK) return r;
  return cuda_status(launch_move(P, st));
}

namespace {

// The staged pass: three kernels (score, select with the z-max score, move).
tria_status evict_staged(const tria_stats* stats, int32_t layer, const tria_layer_cache* cache,
                         const tria_policy* policy, const std::vector<int>& budget, const Layout& L, void* ws,
                         cudaStream_t st) {
  tria_status r;
  Pass P;
  fill_pass(P, cache, policy, budget, L, ws, stats->group);
  set_stats(P, stats, layer);
  P.only_active = 1;
  P.raw = (float*)((uint8_t*)ws + L.raw);
  P.score = (float*)((uint8_t*)ws + L.score);
  P.score_in = P.score;
  P.keep = (int32_t*)((uint8_t*)ws + L.keep);
  if ((r = cuda_status(launch_score(P, st))) != TRIA_OK) return r;
  if ((r = cuda_status(launch_select(P, true, st, stats->group))) != TRIA_OK) return r;
  return cuda_status(launch_move(P, st));
}

}  // namespace

extern "C" tria_status tria_evict(const tria_stats* stats, int32_t layer, const tria_layer_cache* cache,
                                  const tria_policy* policy, void* ws, size_t ws_bytes, void* stream) {
  tria_status r;
  if ((r = check_cache(cache)) != TRIA_OK) return r;
  if ((r = check_stats(stats, layer, cache)) != TRIA_OK) return r;
  std::vector<int> budget;
  if ((r = check_policy(cache, policy, true, budget)) != TRIA_OK) return r;
  const Layout L = make_layout(cache, stats->group);
  if ((r = check_ws(ws, ws_bytes, L)) != TRIA_OK) return r;
  cudaStream_t st = (cudaStream_t)stream;
  if (fused_preferred(stats, cache, 1))
    return launch_fused(stats, &layer, 1, cache, policy, budget, L, ws, nullptr, st);
  return evict_staged(stats, layer, cache, policy, budget, L, ws, st);
}

extern "C" tria_status tria_evict_staged(const tria_stats* stats, int32_t layer, const tria_layer_cache* cache,
                                         const tria_policy* policy, void* ws, size_t ws_bytes, void* stream) {
  tria_status r;
  if ((r = check_cache(cache)) != TRIA_OK) return r;
  if ((r = check_stats(stats, layer, cache)) != TRIA_OK) return r;
  std::vector<int> budget;
  if ((r = check_policy(cache, policy, true, budget)) != TRIA_OK) return r;
  const Layout L = make_layout(cache, stats->group);
  if ((r = check_ws(ws, ws_bytes, L)) != TRIA_OK) return r;
  return evict_staged(stats, layer, cache, policy, budget, L, ws, (cudaStream_t)stream);
}

namespace {

// The caches of a model pass describe the same sequences with the same shapes
// and types; each layer is loaded, has the cache's head_dim and the first
// layer's RoPE frequencies.
tria_status check_model(const tria_stats* stats, const int32_t* layers, int32_t n_layers,
                        const tria_layer_cache* caches) {
  tria_status r;
  if (!layers || !caches || n_layers < 1) return TRIA_ERR_INVALID_ARG;
  if (n_layers > kPassMaxLayers) return TRIA_ERR_UNSUPPORTED;
  const tria_layer_cache& c0 = caches[0];
  for (int i = 0; i < n_layers; ++i) {
    const tria_layer_cache& c = caches[i];
    if ((r = check_cache(&c)) != TRIA_OK) return r;
    if ((r = check_stats(stats, layers[i], &c)) != TRIA_OK) return r;
    if (c.n_seqs != c0.n_seqs || c.n_kv_heads != c0.n_kv_heads || c.head_dim != c0.head_dim ||
        c.k_type != c0.k_type || c.v_type != c0.v_type)
      return TRIA_ERR_INVALID_ARG;
    for (int s = 0; s < c0.n_seqs; ++s)
      if (c.seq_row0[s] != c0.seq_row0[s] || c.capacity[s] != c0.capacity[s]) return TRIA_ERR_INVALID_ARG;
    const int64_t f0 = stats->freq_off[layers[0]], f1 = stats->freq_off[layers[0] + 1];
    const int64_t g0 = stats->freq_off[layers[i]], g1 = stats->freq_off[layers[i] + 1];
    if (g1 - g0 != f1 - f0) return TRIA_ERR_UNSUPPORTED;
    for (int64_t k = 0; k < f1 - f0; ++k)
      if (stats->freq[g0 + k] != stats->freq[f0 + k]) return TRIA_ERR_UNSUPPORTED;
    for (int j = 0; j < i; ++j)   // one pass must not compact a layer twice
      if (caches[j].k == c.k || caches[j].n_live == c.n_live) return TRIA_ERR_INVALID_ARG;
  }
  return TRIA_OK;
}

}  // namespace

extern "C" size_t tria_model_workspace_size(const tria_layer_cache* cache, int32_t n_layers, int32_t group) {
  if (check_cache(cache) != TRIA_OK || group < 0 || group > kMaxG || n_layers < 1 || n_layers > kPassMaxLayers)
    return 0;
  return make_model_layout(cache, group, n_layers).total;
}

extern "C" int32_t tria_evict_model_fused(const tria_stats* stats, const int32_t* layers, int32_t n_layers,
                                          const tria_layer_cache* caches) {
  if (check_model(stats, layers, n_layers, caches) != TRIA_OK) return -1;
  return fused_preferred(stats, caches, n_layers) ? 1 : 0;
}

extern "C" tria_status tria_evict_model(const tria_stats* stats, const int32_t* layers, int32_t n_layers,
                                        const tria_layer_cache* caches, const tria_policy* policy,
                                        float* score_out, void* ws, size_t ws_bytes, void* stream) {
  tria_status r;
  if ((r = check_model(stats, layers, n_layers, caches)) != TRIA_OK) return r;
  std::vector<int> budget;
  if ((r = check_policy(caches, policy, true, budget)) != TRIA_OK) return r;
  if (score_out && ((uintptr_t)score_out % 4) != 0) return TRIA_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  if (fused_ok(stats, caches, n_layers) && (score_out || fused_preferred(stats, caches, n_layers))) {
    const Layout L = make_model_layout(caches, stats->group, n_layers);
    if ((r = check_ws(ws, ws_bytes, L)) != TRIA_OK) return r;
    return launch_fused(stats, layers, n_layers, caches, policy, budget, L, ws, score_out, st);
  }
  // shapes without the fused kernel: one staged pass per layer (no scores out)
  if (score_out) return TRIA_ERR_UNSUPPORTED;
  const Layout L = make_layout(caches, stats->group);
  if ((r = check_ws(ws, ws_bytes, L)) != TRIA_OK) return r;
  for (int i = 0; i < n_layers; ++i)
    if ((r = evict_staged(stats, layers[i], &caches[i], policy, budget, L, ws, st)) != TRIA_OK) return r;
  return TRIA_OK;
}

extern "C" tria_status tria_evict_layers(const tria_stats* stats, const int32_t* layer_of_seq,
                                         const tria_layer_cache* cache, const tria_policy* policy, void* ws,
                                         size_t ws_bytes, void* stream) {
  tria_status r;
  if ((r = check_cache(cache)) != TRIA_OK) return r;
  if (!layer_of_seq) return TRIA_ERR_INVALID_ARG;
  const int l0 = layer_of_seq[0];
  if ((r = check_stats(stats, l0, cache)) != TRIA_OK) return r;
  // every layer of the call: loaded, the cache's head_dim, the first layer's phases
  const int64_t f0 = stats->freq_off[l0], f1 = stats->freq_off[l0 + 1];
  for (int s = 1; s < cache->n_seqs; ++s) {
    const int l = layer_of_seq[s];
    if ((r = check_stats(stats, l, cache)) != TRIA_OK) return r;
    if (stats->freq_off[l + 1] - stats->freq_off[l] != f1 - f0) return TRIA_ERR_UNSUPPORTED;
    for (int64_t i = 0; i < f1 - f0; ++i)
      if (stats->freq[stats->freq_off[l] + i] != stats->freq[f0 + i]) return TRIA_ERR_UNSUPPORTED;
  }
  std::vector<int> budget;
  if ((r = check_policy(cache, policy, true, budget)) != TRIA_OK) return r;
  const Layout L = make_layout(cache, stats->group);
  if ((r = check_ws(ws, ws_bytes, L)) != TRIA_OK) return r;
  Pass P;
  fill_pass(P, cache, policy, budget, L, ws, stats->group);
  set_stats(P, stats, l0);
  for (int s = 0; s < cache->n_seqs; ++s) P.seq[s].qe_off = (int32_t)stats->qe_off[layer_of_seq[s]];
  P.only_active = 1;
  P.raw = (float*)((uint8_t*)ws + L.raw);
  P.score = (float*)((uint8_t*)ws + L.score);
  P.score_in = P.score;
  P.keep = (int32_t*)((uint8_t*)ws + L.keep);
  cudaStream_t st = (cudaStream_t)stream;
  if ((r = cuda_status(launch_score(P, st))) != TRIA_OK) return r;
  if ((r = cuda_status(launch_select(P, true, st, stats->group))) != TRIA_OK) return r;
  return cuda_status(launch_move(P, st));
}

extern "C" tria_status tria_evict_marked(const tria_stats* stats, int32_t layer, const tria_layer_cache* cache,
                                         const tria_policy* policy, void* ws, size_t ws_bytes, void* stream,
                                         void* const* events) {
  tria_status r;
  if (!events || !events[0] || !events[1] || !events[2] || !events[3]) return TRIA_ERR_INVALID_ARG;
  if ((r = check_cache(cache)) != TRIA_OK) return r;
  if ((r = check_stats(stats, layer, cache)) != TRIA_OK) return r;
  std::vector<int> budget;
  if ((r = check_policy(cache, policy, true, budget)) != TRIA_OK) return r;
  const Layout L = make_layout(cache, stats->group);
  if ((r = check_ws(ws, ws_bytes, L)) != TRIA_OK) return r;
  Pass P;
  fill_pass(P, cache, policy, budget, L, ws, stats->group);
  set_stats(P, stats, layer);
  P.only_active = 1;
  P.raw = (float*)((uint8_t*)ws + L.raw);
  P.score = (float*)((uint8_t*)ws + L.score);
  P.score_in = P.score;
  P.keep = (int32_t*)((uint8_t*)ws + L.keep);
  cudaStream_t st = (cudaStream_t)stream;
  cudaEvent_t const* ev = reinterpret_cast<cudaEvent_t const*>(events);
  // external records: inside a stream capture they become event-record nodes
  // that can be timed after the graph runs
  auto mark = [&](int i) { return cudaEventRecordWithFlags(ev[i], st, cudaEventRecordExternal); };
  cudaError_t e = mark(0);
  if (e == cudaSuccess) e = launch_score(P, st);
  if (e == cudaSuccess) e = mark(1);
  if (e == cudaSuccess) e = launch_select(P, true, st, stats->group);
  if (e == cudaSuccess) e = mark(2);
  if (e == cudaSuccess) e = launch_move(P, st);
  if (e == cudaSuccess) e = mark(3);
  return cuda_status(e);
}

extern "C" tria_status tria_evict_profiled(const tria_stats* stats, int32_t layer, const tria_layer_cache* cache,
                                           const tria_policy* policy, void* ws, size_t ws_bytes, void* stream,
                                           float* stage_ms, int32_t* launches) {
  tria_status r;
  if (!stage_ms || !launches) return TRIA_ERR_INVALID_ARG;
  if ((r = check_cache(cache)) != TRIA_OK) return r;
  if ((r = check_stats(stats, layer, cache)) != TRIA_OK) return r;
  std::vector<int> budget;
  if ((r = check_policy(cache, policy, true, budget)) != TRIA_OK) return r;
  const Layout L = make_layout(cache, stats->group);
  if ((r = check_ws(ws, ws_bytes, L)) != TRIA_OK) return r;
  Pass P;
  fill_pass(P, cache, policy, budget, L, ws, stats->group);
  set_stats(P, stats, layer);
  P.only_active = 1;
  P.raw = (float*)((uint8_t*)ws + L.raw);
  P.score = (float*)((uint8_t*)ws + L.score);
  P.score_in = P.score;
  P.keep = (int32_t*)((uint8_t*)ws + L.keep);
  cudaStream_t st = (cudaStream_t)stream;
  cudaEvent_t ev[5] = {};
  for (int i = 0; i < 5; ++i)
    if (cudaEventCreate(&ev[i]) != cudaSuccess) {
      for (int j = 0; j < i; ++j) cudaEventDestroy(ev[j]);
      return TRIA_ERR_CUDA;
    }
  // the z-max score is computed inside the select kernel: its stage time is 0
  cudaError_t e = cudaEventRecord(ev[0], st);
  if (e == cudaSuccess) e = launch_score(P, st);
  if (e == cudaSuccess) e = cudaEventRecord(ev[1], st);
  if (e == cudaSuccess) e = cudaEventRecord(ev[2], st);
  if (e == cudaSuccess) e = launch_select(P, true, st, stats->group);
  if (e == cudaSuccess) e = cudaEventRecord(ev[3], st);
  if (e == cudaSuccess) e = launch_move(P, st);
  if (e == cudaSuccess) e = cudaEventRecord(ev[4], st);
  if (e == cudaSuccess) e = cudaEventSynchronize(ev[4]);
  if (e == cudaSuccess) {
    for (int i = 0; i < 4; ++i) cudaEventElapsedTime(&stage_ms[i], ev[i], ev[i + 1]);
    cudaEventElapsedTime(&stage_ms[4], ev[0], ev[4]);
    *launches = 3;
  }
  for (int i = 0; i < 5; ++i) cudaEventDestroy(ev[i]);
  return cuda_status(e);
}

extern "C" tria_status tria_device_status(void* ws, void* stream) {
  if (!ws || !aligned(ws, 256)) return TRIA_ERR_WORKSPACE;
  cudaStream_t st = (cudaStream_t)stream;
  uint32_t words[2] = {0, 0};
  if (cudaMemcpyAsync(words, ws, sizeof(words), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return TRIA_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return TRIA_ERR_CUDA;
  if (words[0] != 0) {
    if (cudaMemsetAsync(ws, 0, sizeof(words), st) != cudaSuccess) return TRIA_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return TRIA_ERR_CUDA;
  }
  return (tria_status)words[0];
}

extern "C" tria_status tria_selftest_bounded_wait(int32_t spin_limit, void* ws, size_t ws_bytes, void* stream) {
  if (!ws || !aligned(ws, 256) || ws_bytes < sizeof(Ctrl) || spin_limit < 1) return TRIA_ERR_WORKSPACE;
  Pass P;
  memset(&P, 0, sizeof(P));
  P.ctrl = (Ctrl*)ws;
  P.spin_limit = spin_limit;
  cudaStream_t st = (cudaStream_t)stream;
  if (launch_wait_selftest(P, st) != cudaSuccess) return TRIA_ERR_CUDA;
  return tria_device_status(ws, stream);
}

extern "C" const char* tria_status_string(tria_status s) {
  switch (s) {
    case TRIA_OK: return "ok";
    case TRIA_ERR_INVALID_ARG: return "invalid argument";
    case TRIA_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case TRIA_ERR_BUDGET: return "budget smaller than sink + window";
    case TRIA_ERR_CUDA: return "CUDA error";
    case TRIA_ERR_WORKSPACE: return "workspace too small or misaligned";
    case TRIA_ERR_TIMEOUT: return "device wait timed out";
    case TRIA_ERR_DEVICE_ARG: return "n_live out of range";
    case TRIA_ERR_CAPACITY: return "rows do not fit the physical capacity";
    case TRIA_ERR_KEEP_LIST: return "invalid keep list";
  }
  return "unknown status";
}

extern "C" size_t tria_workspace_score_offset(const tria_layer_cache* cache) {
  if (check_cache(cache) != TRIA_OK) return 0;
  return make_layout(cache, 0).score;
}

extern "C" int32_t tria_version(void) { return TRIA_VERSION; }
