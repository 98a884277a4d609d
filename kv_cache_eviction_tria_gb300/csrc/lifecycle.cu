// Decode-loop lifecycle: the row append kernel and the host schedule that says
// when a pass runs and what it keeps.
//
// Sources cited by page title and section:
//   [Worklog] "TriAttention Native C++ Worklog": "Why this is still fair even
//             though the TriAttention bundle is tri12288" (trigger at
//             kv_budget + divide_length), "Sample9 compaction was then proven
//             live" (3200 -> 3072 at positions 3200, 3328, ...), "Same-prompt
//             boundary runs localized the divergence to the first compaction"
//             (158-token prompt, first pass at absolute position 7168),
//             "Sample9 boundary replay exposed a prompt-token accounting
//             mismatch" / "Aligned sample9 replay" (decode-only accounting),
//             "Phase 6: overflow bug during prompt prefill" and "4. Separate
//             physical cache limit from logical TriAttention budget".
//   [Doc]     "TriAttention KV-Cache Eviction (--triattention)": §1 CLI flags
//             (--tri-interval, --tri-budget, --tri-sink, --tri-window), §5
//             Phase B (the evictor fires only on single-token decode steps).
#include <math.h>
#include <string.h>

#include <algorithm>

#include "tria_internal.cuh"

namespace tria {

namespace {

constexpr int kAppendWarps = 8;

// One row of `bytes` (a multiple of 16) with 16-byte loads and stores.
__device__ __forceinline__ void copy_row16(uint8_t* dst, const uint8_t* src, int bytes, int lane) {
  const int4* s = reinterpret_cast<const int4*>(src);
  int4* d = reinterpret_cast<int4*>(dst);
  for (int i = lane; i < bytes / 16; i += 32) d[i] = __ldg(s + i);
}

// A q8_0 scale row (head_dim / 32 fp16 values) with 2-byte copies.
__device__ __forceinline__ void copy_row2(uint8_t* dst, const uint8_t* src, int bytes, int lane) {
  const uint16_t* s = reinterpret_cast<const uint16_t*>(src);
  uint16_t* d = reinterpret_cast<uint16_t*>(dst);
  for (int i = lane; i < bytes / 2; i += 32) d[i] = __ldg(s + i);
}

__device__ __forceinline__ uint32_t append_error(int n, int n_tokens, int cap) {
  if (n < 0 || n > cap) return TRIA_ERR_DEVICE_ARG;
  if ((int64_t)n + n_tokens > cap) return TRIA_ERR_CAPACITY;
  return 0u;
}

// A warp per appended row; the destination is read from n_live, which only the
// last CTA to finish changes (after every CTA has taken its ticket, so after
// every read of the old value).
__global__ void __launch_bounds__(kAppendWarps * 32) k_append(const Pass P, const AppendSrc a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t per_seq = (int64_t)P.n_kv * a.n_tokens;
  const int64_t total = per_seq * P.n_seqs;
  for (int64_t t = (int64_t)blockIdx.x * kAppendWarps + warp; t < total;
       t += (int64_t)gridDim.x * kAppendWarps) {
    const int s = (int)(t / per_seq);
    const int64_t rem = t - (int64_t)s * per_seq;
    const int g = (int)(rem / a.n_tokens);
    const int tok = (int)(rem - (int64_t)g * a.n_tokens);
    const SeqInfo& q = P.seq[s];
    const int n = *((volatile const int32_t*)(P.n_live + s));
    if (append_error(n, a.n_tokens, q.cap)) continue;
    const int64_t dst = q.row0 + (int64_t)g * q.cap + n + tok;
    copy_row16(P.k + dst * P.k_rb, a.k + t * P.k_rb, P.k_rb, lane);
    if (P.ks_rb) copy_row2(P.ks + dst * P.ks_rb, a.ks + t * P.ks_rb, P.ks_rb, lane);
    copy_row16(P.v + dst * P.v_rb, a.v + t * P.v_rb, P.v_rb, lane);
    if (P.vs_rb) copy_row2(P.vs + dst * P.vs_rb, a.vs + t * P.vs_rb, P.vs_rb, lane);
    if (lane == 0) P.pos[dst] = __ldg(a.pos + (int64_t)s * a.n_tokens + tok);
  }
  __syncthreads();
  if (threadIdx.x != 0) return;
  __threadfence();
  const uint32_t ticket = atomicAdd(&P.ctrl->append_ticket, 1u);
  if (ticket != gridDim.x - 1) return;
  __threadfence();
  for (int s = 0; s < P.n_seqs; ++s) {
    const int n = *((volatile const int32_t*)(P.n_live + s));
    const uint32_t e = append_error(n, a.n_tokens, P.seq[s].cap);
    if (e) {
      report(P.ctrl, e, (uint32_t)s);
      continue;
    }
    P.n_live[s] = n + a.n_tokens;
  }
  atomicExch(&P.ctrl->append_ticket, 0u);
}

}  // namespace

cudaError_t launch_append(const Pass& P, const AppendSrc& a, cudaStream_t st) {
  const int64_t total = (int64_t)P.n_seqs * P.n_kv * a.n_tokens;
  const int64_t want = (total + kAppendWarps - 1) / kAppendWarps;
  const int grid = (int)std::min<int64_t>(std::max<int64_t>(want, 1), 8 * 152);
  k_append<<<grid, kAppendWarps * 32, 0, st>>>(P, a);
  return cudaGetLastError();
}

}  // namespace tria

// ---------------------------------------------------------------------------
// host schedule (no GPU use)
// ---------------------------------------------------------------------------

namespace {

bool flag_ok(int32_t f) { return f == 0 || f == 1; }

// Counted rows a pass keeps.
int64_t counted_budget(const tria_schedule* sch) {
  if (sch->trigger == TRIA_TRIGGER_LENGTH) return sch->kv_budget;
  return (int64_t)floor(sch->budget_frac * (double)sch->n_ctx);
}

// Rows a pass keeps and the protected prefix: prompt rows outside the count
// are added to the budget when they are protected; protected prompt rows join
// the sink (they sit at the front: compaction keeps the order).
void pass_shape(const tria_schedule* sch, const tria_seq_state* st, int64_t* B, int64_t* sink) {
  const int64_t uncounted = st->rows - st->counted;
  *B = counted_budget(sch) + (sch->protect_prefill ? uncounted : 0);
  *sink = sch->protect_prefill ? std::max<int64_t>(sch->sink, st->prompt_rows) : sch->sink;
}

}  // namespace

extern "C" tria_status tria_schedule_check(const tria_schedule* sch) {
  if (!sch) return TRIA_ERR_INVALID_ARG;
  if (sch->trigger != TRIA_TRIGGER_LENGTH && sch->trigger != TRIA_TRIGGER_INTERVAL) return TRIA_ERR_INVALID_ARG;
  if (!flag_ok(sch->count_prompt_tokens) || !flag_ok(sch->protect_prefill)) return TRIA_ERR_INVALID_ARG;
  if (sch->sink < 0 || sch->window < 0 || sch->divide_length < 1) return TRIA_ERR_INVALID_ARG;
  if (sch->trigger == TRIA_TRIGGER_LENGTH) {
    if (sch->kv_budget < 1 || sch->kv_budget > INT32_MAX) return TRIA_ERR_INVALID_ARG;
  } else {
    if (!(sch->budget_frac > 0.0) || sch->budget_frac > 1.0 || sch->n_ctx < 0) return TRIA_ERR_INVALID_ARG;
  }
  return TRIA_OK;
}

extern "C" tria_status tria_seq_init(tria_seq_state* st, int64_t capacity) {
  if (!st || capacity < 0 || capacity > INT32_MAX) return TRIA_ERR_INVALID_ARG;
  memset(st, 0, sizeof(*st));
  st->capacity = capacity;
  return TRIA_OK;
}

extern "C" tria_status tria_seq_prefill(const tria_schedule* sch, tria_seq_state* st, int64_t n_tokens) {
  if (tria_schedule_check(sch) != TRIA_OK || !st || n_tokens < 0) return TRIA_ERR_INVALID_ARG;
  if (st->decode_steps != 0 || st->due) return TRIA_ERR_INVALID_ARG;
  if (st->rows + n_tokens > st->capacity) return TRIA_ERR_CAPACITY;
  st->rows += n_tokens;
  st->prompt_rows += n_tokens;
  st->next_pos += n_tokens;
  if (sch->count_prompt_tokens) st->counted += n_tokens;
  return TRIA_OK;
}

extern "C" tria_status tria_seq_decode(const tria_schedule* sch, tria_seq_state* st) {
  if (tria_schedule_check(sch) != TRIA_OK || !st || st->due) return TRIA_ERR_INVALID_ARG;
  if (st->rows + 1 > st->capacity) return TRIA_ERR_CAPACITY;
  st->rows += 1;
  st->counted += 1;
  st->next_pos += 1;
  st->decode_steps += 1;
  if (sch->trigger == TRIA_TRIGGER_LENGTH)
    st->due = st->counted >= sch->kv_budget + sch->divide_length ? 1 : 0;
  else
    st->due = st->decode_steps % sch->divide_length == 0 ? 1 : 0;
  return TRIA_OK;
}

extern "C" tria_status tria_schedule_plan(const tria_schedule* sch, const tria_seq_state* st, int32_t n_seqs,
                                          int32_t* budget_rows, int32_t* sink_rows, int64_t* cur_pos,
                                          int32_t* n_due) {
  if (tria_schedule_check(sch) != TRIA_OK || !st || n_seqs < 0 || !budget_rows || !sink_rows || !cur_pos || !n_due)
    return TRIA_ERR_INVALID_ARG;
  int32_t due = 0;
  for (int s = 0; s < n_seqs; ++s) {
    cur_pos[s] = st[s].next_pos;
    if (!st[s].due) {
      budget_rows[s] = TRIA_NO_PASS;
      sink_rows[s] = sch->sink;
      continue;
    }
    int64_t B, sink;
    pass_shape(sch, &st[s], &B, &sink);
    if (B > INT32_MAX || sink > INT32_MAX) return TRIA_ERR_INVALID_ARG;
    if (B < sink + sch->window) return TRIA_ERR_BUDGET;
    budget_rows[s] = (int32_t)B;
    sink_rows[s] = (int32_t)sink;
    ++due;
  }
  *n_due = due;
  return TRIA_OK;
}

extern "C" tria_status tria_schedule_passed(const tria_schedule* sch, tria_seq_state* st, int32_t n_seqs) {
  if (tria_schedule_check(sch) != TRIA_OK || !st || n_seqs < 0) return TRIA_ERR_INVALID_ARG;
  for (int s = 0; s < n_seqs; ++s) {
    if (!st[s].due) continue;
    int64_t B, sink;
    pass_shape(sch, &st[s], &B, &sink);
    const int64_t uncounted = st[s].rows - st[s].counted;
    if (st[s].rows > B) {
      st[s].rows = B;
      // protected prompt rows stay outside the count; otherwise every
      // surviving row counts from now on
      st[s].counted = sch->protect_prefill ? B - uncounted : B;
    }
    st[s].due = 0;
    st[s].passes += 1;
  }
  return TRIA_OK;
}
