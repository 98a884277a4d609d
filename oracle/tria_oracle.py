"""TriAttention eviction pass, restated step by step on the CPU (float64).

TEST INFRASTRUCTURE, NOT PRODUCT CODE (see :mod:`oracle`).

Sources - the two web pages this restates, cited by title and section:

  [Worklog] "TriAttention Native C++ Worklog" (TensorRT-Model-Connect).
            Sections used: "Phase 9: final root cause - native scorer used the
            wrong formulation" (direct K_rot scorer), "2026-04-18: later-
            compaction absolute-position bug isolated and fixed" (phases from
            the absolute decode position), "Hypothesis: sampled-head mapping
            ..." (query-to-KV head map), "K-cache repack correctness ..." and
            "Later correction ..." (compaction = exact gather of kept rows).
  [Doc]     "TriAttention KV-Cache Eviction (--triattention)" (llama.cpp fork
            docs). Sections used: "At a glance" (NEOX-RoPE GQA models),
            "§1 CLI flags" (budget %, window, sink, interval), "§2 Calibration
            file (.tria)" (per-head RoPE-direction statistics), "§4 Backend and
            model support" (GPU gate, q8_0 K), "§5 How it works - Phase B"
            (score, protect, sort, compact in place) and "Phase C" (per-query-
            head z-normalisation, max over the GQA group, omega / q_mean /
            q_abs arrays).

Readings where the pages are silent:

* NEOX pairing: frequency pair f of a head_dim-hd vector is the complex number
  x[f] + i x[f + hd/2]; omega_f = theta ** (-2 f / hd).
* Score of cached row r for query head h at decode position p
  ([Worklog] Phase 9: mean query times the conjugate of the stored rotated
  key, rotation on the query side only, plus a norm term on the rotated
  key's magnitudes)::

      raw_h(r) = (1/|D|) sum_{d in D} sum_f Re( qbar_{h,f} e^{i w_f (p+d)} conj(k_{r,f}) )
                 + sum_f M_{h,f} |k_{r,f}|

  with M = q_abs - |qbar|: "MLR" read as the mean resultant length
  R_f = |qbar_f| / q_abs_f, the norm term weighted by (1 - R_f) q_abs_f.
  D (future query offsets) is a load-time parameter; default {1, 2, 4, ..., 2^16}.
* Non-rotary (content) dims ([Doc] §4 gate line field ``nonrot=``, §6 "Non-
  rotary models": such models carry a content term besides the RoPE-direction
  term; the pages give no formula). Reading: the first rot = hd - nonrot_dim
  dims are rotary, NEOX-paired as (f, f + rot/2) with omega_f =
  theta ** (-2 f / rot); the last nonrot_dim dims are never rotated, so their
  share of a future query's logit does not depend on the position and its
  mean over the queries is the mean non-rotary query qn_h (calibrated like
  q_mean) dotted with the key's non-rotary dims:
      raw_h(r) += sum_e qn_{h,e} K[r][rot + e]
  with no offset average, no phase and no norm term.
* z-normalisation: population mean/std over all n live rows of the segment,
  z = (raw - mu) / (sigma + 1e-6); KV-head score s = max over its query heads.
* Budget B = floor(budget_frac * n_ctx) survivors in total, sink and window
  included; candidates are rows [sink, n - window); k = B - sink - window of
  them are kept by (s descending, row ascending). n <= B is a no-op;
  B < sink + window is an error.
* Compaction writes kept row i (ascending original order) to row i of K, V,
  the q8_0 scales and pos; rows at or past B keep their old contents.
* Shared-slot cells (one keep-set per token for all layers): the pages do
  not state the combine rule; a token's score is the maximum of its z-max
  scores over all layers and KV heads (NaN ignored unless all are NaN).
* Calibration ([Doc] §2: per-layer, per-head statistics of the pre-RoPE
  queries, giving the average query direction and a weight per frequency;
  §5 Phase C: q_mean / q_abs arrays [layers][heads][frequency pairs]):
  over the calibration tokens t of one layer, q_mean_{h,f} = mean_t of the
  complex pair Q_t[h][f] + i Q_t[h][f + hd/2], q_abs_{h,f} = mean_t of its
  modulus.
"""
from __future__ import annotations

import math

import numpy as np

Z_EPS = 1e-6


class BudgetError(ValueError):
    """Budget smaller than the protected sink + window rows."""


# ---------------------------------------------------------------------------
# RoPE frequencies, future offsets, calibration weights
# ---------------------------------------------------------------------------

def rope_omega(head_dim: int, theta: float, nonrot_dim: int = 0) -> np.ndarray:
    """omega_f = theta^(-2f/rot), f = 0 .. rot/2 - 1, rot = head_dim - nonrot_dim
    the rotary dims (NEOX pairs; [Doc] At a glance, Phase C "calibration omega";
    §4 gate line ``nonrot=``: dims past the rotary ones are never rotated)."""
    rot = head_dim - nonrot_dim
    return np.array([theta ** (-2.0 * f / rot) for f in range(rot // 2)], dtype=np.float64)


def default_future_offsets() -> np.ndarray:
    """Future query offsets D = {2^0, ..., 2^16} (reading; the pages give none)."""
    return np.array([2 ** j for j in range(17)], dtype=np.int64)


def as_complex(q_mean: np.ndarray) -> np.ndarray:
    """[..., fc, 2] (re, im) -> complex128 [..., fc]."""
    q = np.asarray(q_mean, dtype=np.float64)
    return q[..., 0] + 1j * q[..., 1]


def mlr_weight(q_mean: np.ndarray, q_abs: np.ndarray | None) -> np.ndarray:
    """M = q_abs - |qbar| per (head, pair) ([Worklog] Phase 9, its norm term;
    [Doc] §2, a weight per frequency; Phase C, the q_mean / q_abs arrays).
    ``q_abs`` None means M = 0."""
    qc = as_complex(q_mean)
    if q_abs is None:
        return np.zeros(qc.shape, dtype=np.float64)
    return np.asarray(q_abs, dtype=np.float64) - np.abs(qc)


def heads_of_kv(n_q_heads: int, n_kv_heads: int, kv_of_q=None) -> list:
    """Query heads of each KV head, ascending ([Worklog] "sampled-head mapping":
    follow the given map; default contiguous groups h // G)."""
    if kv_of_q is None:
        g = n_q_heads // n_kv_heads
        kv_of_q = [h // g for h in range(n_q_heads)]
    return [[h for h in range(n_q_heads) if kv_of_q[h] == kv] for kv in range(n_kv_heads)]


# ---------------------------------------------------------------------------
# keys
# ---------------------------------------------------------------------------

def dequant_q8_0(qs: np.ndarray, d: np.ndarray) -> np.ndarray:
    """Planar q8_0 rows -> float64: value = fp16 scale of the 32-wide block x code
    ([Doc] §4 "--cache-type-k q8_0"; ggml Q8_0 block = 32 int8 codes + fp16 scale)."""
    n, hd = qs.shape
    scale = np.repeat(np.asarray(d, dtype=np.float16).astype(np.float64), 32, axis=1)
    return qs.astype(np.float64) * scale[:, :hd]


def keys_f64(k: np.ndarray, k_scale: np.ndarray | None = None) -> np.ndarray:
    """Stored keys widened exactly to float64."""
    if k.dtype == np.int8:
        return dequant_q8_0(k, k_scale)
    return np.asarray(k, dtype=np.float64)


# ---------------------------------------------------------------------------
# scoring ([Worklog] Phase 9; [Doc] Phase C)
# ---------------------------------------------------------------------------

def raw_scores(k_rot: np.ndarray, q_mean_c: np.ndarray, m_weight: np.ndarray,
               omega: np.ndarray, p: int, offsets, q_nonrot: np.ndarray | None = None) -> np.ndarray:
    """raw[r, j] for rows r of one segment and the segment's query heads j.

    ``k_rot`` float64 [n, hd] stored keys (rotary dims already rotated);
    ``omega`` the rot/2 frequencies of the rotary dims [0, rot) (rot = hd when
    every dim is rotary); ``q_mean_c`` complex [G, rot/2]; ``m_weight``
    [G, rot/2]; ``q_nonrot`` [G, hd - rot] the mean non-rotary query, None for
    no content term; ``p`` absolute decode position ([Worklog] 2026-04-18:
    phases from the absolute position, not the row count).
    Loops over the offsets literally; each offset is one complex matmul.
    """
    k_rot = np.asarray(k_rot, dtype=np.float64)
    n, hd = k_rot.shape
    fc = len(omega)
    rot = 2 * fc
    kc = k_rot[:, :fc] + 1j * k_rot[:, fc:rot]
    g = q_mean_c.shape[0]
    trig = np.zeros((n, g), dtype=np.float64)
    offsets = list(offsets)
    for d in offsets:
        ang = np.fmod(omega * float(p + int(d)), 2.0 * math.pi)
        phase = np.cos(ang) + 1j * np.sin(ang)             # e^{i w_f (p + d)}
        q_rot = q_mean_c * phase[None, :]                    # mean query at position p + d
        trig += np.real(np.conj(kc) @ q_rot.T)              # sum_f Re(q_rot conj(k))
    trig /= len(offsets)
    norm = np.abs(kc) @ np.asarray(m_weight, dtype=np.float64).T   # sum_f M |k_f|
    if q_nonrot is None or rot == hd:
        return trig + norm
    # non-rotary dims: no rotation at any position, so every future query's
    # mean logit there is the mean query's plain dot product with the key
    content = k_rot[:, rot:] @ np.asarray(q_nonrot, dtype=np.float64).T
    return trig + norm + content


def znorm(raw: np.ndarray) -> np.ndarray:
    """Per-query-head z-score over all live rows ([Doc] Phase C). A segment
    without live rows has no rows to normalise (and no moments)."""
    if raw.shape[0] == 0:
        return np.array(raw, dtype=np.float64)
    mu = raw.mean(axis=0)
    sd = raw.std(axis=0)  # population
    return (raw - mu[None, :]) / (sd[None, :] + Z_EPS)


def gqa_max(z: np.ndarray) -> np.ndarray:
    """KV-head score = max over the group's query heads ([Doc] Phase C)."""
    return z.max(axis=1)


def segment_scores(k_rot, q_mean_c, m_weight, omega, p, offsets, q_nonrot=None):
    """(raw [n, G], s [n]) of one segment."""
    raw = raw_scores(k_rot, q_mean_c, m_weight, omega, p, offsets, q_nonrot)
    return raw, gqa_max(znorm(raw))


# ---------------------------------------------------------------------------
# selection ([Doc] §1, §5 Phase B)
# ---------------------------------------------------------------------------

def budget_rows(budget_frac: float, n_ctx: int) -> int:
    """B = floor(budget_frac * n_ctx) ([Doc] §1 --tri-budget: the kept share of n_ctx)."""
    return int(math.floor(float(budget_frac) * int(n_ctx)))


def select_keep(s: np.ndarray, n: int, budget: int, sink: int, window: int) -> np.ndarray:
    """Kept rows of one segment, ascending ([Doc] Phase B steps 2-3).

    Protect rows [0, sink) and [n - window, n); of the rest keep the
    k = B - sink - window best by (s descending, row ascending), via a stable
    sort of -s. NaN scores sort last.
    """
    if n <= budget:
        return np.arange(n, dtype=np.int64)
    if budget < sink + window:
        raise BudgetError(f"budget {budget} < sink {sink} + window {window}")
    cand = np.arange(sink, n - window, dtype=np.int64)
    k = budget - sink - window
    order = np.argsort(-np.asarray(s, dtype=np.float64)[cand], kind="stable")
    chosen = cand[order[:k]]
    keep = np.concatenate([np.arange(sink, dtype=np.int64), chosen,
                           np.arange(n - window, n, dtype=np.int64)])
    return np.sort(keep)


# ---------------------------------------------------------------------------
# compaction ([Doc] Phase B step 4; [Worklog] exact-gather checks)
# ---------------------------------------------------------------------------

def compact_rows(plane: np.ndarray, keep: np.ndarray) -> np.ndarray:
    """Kept rows gathered to the front in order; rows >= len(keep) unchanged."""
    out = plane.copy()
    out[:len(keep)] = plane[keep]
    return out


# ---------------------------------------------------------------------------
# one layer, global-row layout (the same layout the C ABI uses)
# ---------------------------------------------------------------------------

def evict_layer(layer_cache: dict, q_mean: np.ndarray, q_abs, *, layer: int, n_kv_heads: int,
                head_dim: int, rope_theta: float, cur_pos, n_ctx, budget_frac: float,
                window: int, sink: int, offsets=None, kv_of_q=None, omega=None,
                budget_rows_override=None, segments=None, nonrot_dim: int = 0, q_nonrot=None):
    """Run the pass on one layer's host cache.

    ``layer_cache`` holds ``k`` (float or int8 codes), ``k_scale`` (or None),
    ``v``, ``pos`` over global rows plus ``n_live``, ``seq_row0``,
    ``capacity`` per sequence. ``q_mean`` [L][Hq][fc][2], ``q_abs`` [L][Hq][fc]
    (arrays, or per-layer lists when head_dim differs across layers).
    ``segments`` optionally restricts the work to a list of (seq, head).
    ``nonrot_dim`` > 0: the last nonrot_dim dims of each head are not rotary
    (``q_mean`` / ``q_abs`` then cover (head_dim - nonrot_dim) / 2 pairs) and
    ``q_nonrot`` [L][Hq][nonrot_dim] (or None: no content term) is the mean
    non-rotary query.

    Returns ``(new_cache, info)``: ``info[(s, g)]`` = dict(raw, s, keep, B, n).
    """
    omega = (rope_omega(head_dim, rope_theta, nonrot_dim) if omega is None
             else np.asarray(omega, np.float64))
    if 2 * len(omega) + nonrot_dim != head_dim:
        raise ValueError("omega must hold (head_dim - nonrot_dim) / 2 frequencies")
    offsets = default_future_offsets() if offsets is None else np.asarray(offsets, np.int64)
    n_q = len(q_mean[layer])
    groups = heads_of_kv(n_q, n_kv_heads, kv_of_q)
    qc_all = as_complex(q_mean[layer])
    m_all = mlr_weight(q_mean[layer], None if q_abs is None else q_abs[layer])
    out = {key: (None if val is None else np.array(val, copy=True))
           for key, val in layer_cache.items()}
    info = {}
    n_seqs = len(layer_cache["n_live"])
    for s in range(n_seqs):
        n = int(layer_cache["n_live"][s])
        cap = int(layer_cache["capacity"][s])
        if budget_rows_override is not None:
            b = int(budget_rows_override[s])
        else:
            b = budget_rows(budget_frac, n_ctx[s])
        for g in range(n_kv_heads):
            if segments is not None and (s, g) not in segments:
                continue
            r0 = int(layer_cache["seq_row0"][s]) + g * cap
            ks = None if layer_cache.get("k_scale") is None else layer_cache["k_scale"][r0:r0 + n]
            kf = keys_f64(layer_cache["k"][r0:r0 + n], ks)
            hs = groups[g]
            qn = None if q_nonrot is None else np.asarray(q_nonrot[layer], np.float64)[hs]
            raw, sc = segment_scores(kf, qc_all[hs], m_all[hs], omega, int(cur_pos[s]), offsets, qn)
            keep = select_keep(sc, n, b, _per_seq(sink, s), window)
            info[(s, g)] = {"raw": raw, "s": sc, "keep": keep, "B": b, "n": n, "row0": r0}
            if n <= b:
                continue
            for name in ("k", "k_scale", "v", "v_scale", "pos"):
                if out.get(name) is None:
                    continue
                seg = out[name][r0:r0 + cap]
                out[name][r0:r0 + cap] = compact_rows(seg, keep)
    for s in range(n_seqs):
        n = int(layer_cache["n_live"][s])
        b = (int(budget_rows_override[s]) if budget_rows_override is not None
             else budget_rows(budget_frac, n_ctx[s]))
        if n > b:
            out["n_live"][s] = b
    return out, info


def shared_evict(layer_caches: list, q_mean, q_abs, *, n_kv_heads: int, head_dim: int, rope_theta: float,
                 cur_pos, n_ctx, budget_frac: float, window: int, sink: int, offsets=None, kv_of_q=None,
                 budget_rows_override=None):
    """Shared-slot pass: one keep-set per token for every layer and KV head
    (cells shared by all layers; [Doc] Phase B/C, the Vulkan port's global
    z-normalisation shader; [Worklog] cross-layer aggregation).

    The pages do not state how a token's per-(layer, KV head) scores combine.
    Reading: the combined score is the maximum of the token's z-max scores
    over all layers and KV heads, NaN ignored unless all are NaN (np.fmax),
    i.e. the GQA max rule of Phase C extended to every head of every layer.
    ``layer_caches[l]`` has the layout of :func:`evict_layer`; all layers
    share seq_row0, capacity and n_live.

    Returns ``(new_caches, info)``; ``info[s]`` = dict(combined, keep, B, n).
    """
    omega = rope_omega(head_dim, rope_theta)
    offsets = default_future_offsets() if offsets is None else np.asarray(offsets, np.int64)
    base = layer_caches[0]
    n_seqs = len(base["n_live"])
    out = [{key: (None if val is None else np.array(val, copy=True)) for key, val in c.items()}
           for c in layer_caches]
    info = {}
    for s in range(n_seqs):
        n = int(base["n_live"][s])
        cap = int(base["capacity"][s])
        row0 = int(base["seq_row0"][s])
        combined = np.full(n, np.nan)
        for layer, cache in enumerate(layer_caches):
            groups = heads_of_kv(len(q_mean[layer]), n_kv_heads, kv_of_q)
            qc = as_complex(q_mean[layer])
            mw = mlr_weight(q_mean[layer], None if q_abs is None else q_abs[layer])
            for g in range(n_kv_heads):
                r0 = row0 + g * cap
                ks = None if cache.get("k_scale") is None else cache["k_scale"][r0:r0 + n]
                kf = keys_f64(cache["k"][r0:r0 + n], ks)
                _, sc = segment_scores(kf, qc[groups[g]], mw[groups[g]], omega, int(cur_pos[s]), offsets)
                combined = np.fmax(combined, sc)
        b = (int(budget_rows_override[s]) if budget_rows_override is not None
             else budget_rows(budget_frac, n_ctx[s]))
        keep = select_keep(combined, n, b, _per_seq(sink, s), window)
        info[s] = {"combined": combined, "keep": keep, "B": b, "n": n}
        if n <= b:
            continue
        for o in out:
            for g in range(n_kv_heads):
                r0 = row0 + g * cap
                for name in ("k", "k_scale", "v", "v_scale", "pos"):
                    if o.get(name) is not None:
                        o[name][r0:r0 + cap] = compact_rows(o[name][r0:r0 + cap], keep)
            o["n_live"][s] = b
    return out, info


def _per_seq(value, s):
    """``value`` itself, or its s-th entry when it is a sequence."""
    return int(value[s]) if hasattr(value, "__len__") else int(value)


def should_evict(n_live: int, budget: int, interval: int) -> bool:
    """Lifecycle trigger: compact once the live rows reach budget + interval
    ([Worklog] "Final apples-to-apples check": trigger = kv_budget + divide_length;
    [Doc] §1 "--tri-interval")."""
    return n_live >= budget + interval


# ---------------------------------------------------------------------------
# decode-loop lifecycle ([Worklog] "Why this is still fair even though the
# TriAttention bundle is tri12288", "Sample9 compaction was then proven live",
# "Same-prompt boundary runs localized the divergence to the first
# compaction", "Sample9 boundary replay exposed a prompt-token accounting
# mismatch", "Aligned sample9 replay", "Phase 6: overflow bug during prompt
# prefill"; [Doc] §1 --tri-interval / --tri-budget, §5 Phase B)
# ---------------------------------------------------------------------------

class CapacityError(ValueError):
    """Rows appended beyond the physical capacity."""


def schedule_events(*, trigger: str, prompt: int, n_decode: int, capacity: int, kv_budget: int = 0,
                    divide_length: int = 128, count_prompt_tokens: bool = True, protect_prefill: bool = True,
                    sink: int = 0, window: int = 0, budget_frac: float = 0.0, n_ctx: int = 0):
    """Passes of one sequence that appends a prompt of ``prompt`` rows and then
    ``n_decode`` single-token decode steps.

    The cache is tracked as two groups of rows: the prompt rows and the rows
    the decode steps appended. The prompt is appended whole (no pass during
    prefill; it must fit the physical capacity). After each decode step:

    * trigger "length" ([Worklog]): a pass once the counted rows - the decode
      rows, plus the prompt rows when ``count_prompt_tokens`` - reach
      ``kv_budget + divide_length``; the pass keeps ``kv_budget`` counted rows.
    * trigger "interval" ([Doc] §1): a pass on every ``divide_length``-th
      decode step; it keeps ``floor(budget_frac * n_ctx)`` counted rows.

    With ``protect_prefill`` the prompt rows are all kept: they join the sink,
    and when they are not counted they come on top of the kept count. Without
    it the prompt rows compete with the rest, and after the first pass that
    evicts the survivors are plain rows. The pass position is the absolute
    position of the next token, i.e. the tokens appended so far.

    Returns a list of dicts: step (decode steps so far), pos, rows_before,
    counted_before, rows_after, budget (rows the pass keeps), sink.
    """
    if prompt > capacity:
        raise CapacityError(f"prompt of {prompt} rows > capacity {capacity}")
    p_rows, d_rows = prompt, 0
    keep_counted = kv_budget if trigger == "length" else budget_rows(budget_frac, n_ctx)
    events = []
    for step in range(1, n_decode + 1):
        if p_rows + d_rows + 1 > capacity:
            raise CapacityError(f"decode step {step}: capacity {capacity} full")
        d_rows += 1
        counted = d_rows + (p_rows if count_prompt_tokens else 0)
        if trigger == "length":
            due = counted >= kv_budget + divide_length
        else:
            due = step % divide_length == 0
        if not due:
            continue
        if protect_prefill:
            budget = keep_counted + (0 if count_prompt_tokens else p_rows)
            sink_s = max(sink, p_rows)
        else:
            budget, sink_s = keep_counted, sink
        if budget < sink_s + window:
            raise BudgetError(f"budget {budget} < sink {sink_s} + window {window}")
        before = p_rows + d_rows
        if before > budget:
            if protect_prefill:
                d_rows = budget - p_rows
            else:
                p_rows, d_rows = 0, budget
        events.append({"step": step, "pos": prompt + step, "rows_before": before, "counted_before": counted,
                       "rows_after": p_rows + d_rows, "budget": budget, "sink": sink_s})
    return events


# ---------------------------------------------------------------------------
# calibration ([Doc] §2 Calibration file; §5 Phase C q_mean / q_abs layout)
# ---------------------------------------------------------------------------

def calibrate(q: np.ndarray, nonrot_dim: int = 0) -> tuple:
    """Statistics of a stream of pre-RoPE queries q[tokens][heads][head_dim]:
    (q_mean [heads][fc][2] as (re, im), q_abs [heads][fc]), means over the
    tokens of the NEOX pairs q[.., f] + i q[.., f + rot/2] of the rotary dims
    rot = head_dim - nonrot_dim (fc = rot/2) and of their moduli."""
    q = np.asarray(q, dtype=np.float64)
    t, h, hd = q.shape
    if t == 0:
        raise ValueError("no calibration tokens")
    fc = (hd - nonrot_dim) // 2
    z = q[:, :, :fc] + 1j * q[:, :, fc:2 * fc]
    mean = z.mean(axis=0)
    q_mean = np.stack([mean.real, mean.imag], axis=-1)
    q_abs = np.abs(z).mean(axis=0)
    return q_mean, q_abs


def calibrate_nonrot(q: np.ndarray, nonrot_dim: int) -> np.ndarray:
    """Mean non-rotary query [heads][nonrot_dim]: the token mean of the last
    ``nonrot_dim`` dims of each head (the reading of the content term above)."""
    q = np.asarray(q, dtype=np.float64)
    if q.shape[0] == 0:
        raise ValueError("no calibration tokens")
    hd = q.shape[2]
    return q[:, :, hd - nonrot_dim:].mean(axis=0)
