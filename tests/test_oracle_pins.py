"""Pins of the CPU oracle against things other than itself.

Each test fixes one part of :mod:`oracle.tria_oracle` by an independent
computation (brute force with real rotation matrices, the relative-position
RoPE identity, textbook dot products, closed forms, a 40-digit reference, an
independent selection algorithm, exhaustive subsets) or by a value the pages
print. A dropped term, a wrong sign or index, a transposed operand or a wrong
tie-break fails at least one of them.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

from oracle import tria_oracle as O
from synth import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_stats(rng, g, fc, with_m=True):
    qm = rng.standard_normal((g, fc, 2))
    mag = np.hypot(qm[..., 0], qm[..., 1])
    q_abs = mag + (0.5 * np.abs(rng.standard_normal((g, fc))) if with_m else 0.0)
    return qm, q_abs


# ---------------------------------------------------------------- scoring ---

def _brute_raw(k_row, qm_head, q_abs_head, theta, hd, p, offsets):
    """One score by real arithmetic: rotate the real mean-query vector with 2x2
    rotation matrices at position p+d, dot it with the stored key row, average
    over d, add sum_f (q_abs - |qbar|) * sqrt(k_f^2 + k_{f+fc}^2)."""
    fc = hd // 2
    total = 0.0
    for d in offsets:
        qvec = [0.0] * hd
        for f in range(fc):
            w = math.pow(theta, -2.0 * f / hd)
            a, b = qm_head[f][0], qm_head[f][1]
            c, s = math.cos(w * (p + d)), math.sin(w * (p + d))
            qvec[f] = a * c - b * s
            qvec[f + fc] = a * s + b * c
        total += sum(qvec[i] * k_row[i] for i in range(hd))
    total /= len(offsets)
    for f in range(fc):
        m = q_abs_head[f] - math.hypot(qm_head[f][0], qm_head[f][1])
        total += m * math.sqrt(k_row[f] ** 2 + k_row[f + fc] ** 2)
    return total


@pytest.mark.parametrize("hd,g,theta,p,offsets", [
    (8, 2, 100.0, 13, [1, 3, 7]),
    (16, 4, 1e4, 4096, [1, 2, 4, 8, 16]),
    (4, 1, 10.0, 0, [0]),
])
def test_raw_score_matches_real_rotation_bruteforce(hd, g, theta, p, offsets):
    rng = np.random.default_rng(hd * 100 + g)
    n = 6
    k = rng.standard_normal((n, hd))
    qm, q_abs = _rand_stats(rng, g, hd // 2)
    got = O.raw_scores(k, O.as_complex(qm), O.mlr_weight(qm, q_abs),
                       O.rope_omega(hd, theta), p, offsets)
    for r in range(n):
        for j in range(g):
            want = _brute_raw(list(k[r]), qm[j].tolist(), list(q_abs[j]), theta, hd, p, offsets)
            assert abs(got[r, j] - want) <= 1e-12 * max(1.0, abs(want))


def _rope64(x, pos, theta):
    hd = x.shape[1]
    fc = hd // 2
    w = np.array([math.pow(theta, -2.0 * f / hd) for f in range(fc)])
    ang = pos[:, None].astype(np.float64) * w[None, :]
    c, s = np.cos(ang), np.sin(ang)
    a, b = x[:, :fc], x[:, fc:]
    return np.concatenate([a * c - b * s, a * s + b * c], axis=1)


def test_direct_krot_equals_unrotated_relative_position_form():
    """The direct K_rot score equals the older unrotate-then-rephase form
    (key rotated back by its own position, query phase at p + d - pos)
    ([Worklog] Phase 9, both formulations)."""
    w = W.get_workload("tiny")
    k_pre, _ = W.tiny_pre_rope(w)
    k_pre = k_pre[0, 0, 1, :64].astype(np.float64)
    pos = np.arange(64) * 7 + 3
    theta, hd = w.rope_theta, w.head_dim
    fc = hd // 2
    k_rot = _rope64(k_pre, pos, theta)
    rng = np.random.default_rng(3)
    qm, q_abs = _rand_stats(rng, 4, fc)
    offsets = [1, 2, 4, 1024, 65536]
    p = 9000
    got = O.raw_scores(k_rot, O.as_complex(qm), O.mlr_weight(qm, q_abs),
                       O.rope_omega(hd, theta), p, offsets)
    wv = np.array([math.pow(theta, -2.0 * f / hd) for f in range(fc)])
    kc_pre = k_pre[:, :fc] + 1j * k_pre[:, fc:]
    qc = qm[..., 0] + 1j * qm[..., 1]
    want = np.zeros((64, 4))
    for d in offsets:
        rel = np.exp(1j * wv[None, :] * (p + d - pos[:, None]))       # [n, fc]
        want += np.real((np.conj(kc_pre) * rel) @ qc.T)
    want /= len(offsets)
    want += np.abs(kc_pre) @ (q_abs - np.abs(qc)).T
    np.testing.assert_allclose(got, want, rtol=1e-10, atol=1e-10)


def test_zero_offset_zero_position_is_plain_dot_product():
    rng = np.random.default_rng(5)
    hd, g = 32, 3
    k = rng.standard_normal((10, hd))
    qm, _ = _rand_stats(rng, g, hd // 2)
    q_abs = np.hypot(qm[..., 0], qm[..., 1])       # M = 0
    got = O.raw_scores(k, O.as_complex(qm), O.mlr_weight(qm, q_abs),
                       O.rope_omega(hd, 1e4), 0, [0])
    qvec = np.concatenate([qm[..., 0], qm[..., 1]], axis=1)       # [g, hd]
    np.testing.assert_allclose(got, k @ qvec.T, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("p,nd,w", [(0, 8, 0.3), (1000, 128, 0.0123), (131072, 17, 1.0)])
def test_offset_average_dirichlet_closed_form(p, nd, w):
    """D = {0..N-1}: (1/N) sum cos(w(p+d)) = cos(w(p+(N-1)/2)) sin(Nw/2) / (N sin(w/2))."""
    k = np.array([[1.0, 0.0]])
    qm = np.array([[[1.0, 0.0]]])
    got = O.raw_scores(k, O.as_complex(qm), np.zeros((1, 1)), np.array([w]), p, range(nd))[0, 0]
    want = math.cos(w * (p + (nd - 1) / 2)) * math.sin(nd * w / 2) / (nd * math.sin(w / 2))
    assert abs(got - want) < 1e-11


def test_norm_term_closed_form_and_homogeneity():
    hd = 8
    fc = hd // 2
    q_abs = np.array([[0.5, 1.0, 2.0, 0.25]])
    qm = np.zeros((1, fc, 2))                        # qbar = 0 -> M = q_abs
    k = np.array([[3.0] * fc + [4.0] * fc])          # every |k_f| = 5
    got = O.raw_scores(k, O.as_complex(qm), O.mlr_weight(qm, q_abs),
                       O.rope_omega(hd, 1e4), 77, [1, 2])
    assert got[0, 0] == pytest.approx(5.0 * q_abs.sum(), rel=1e-15)
    rng = np.random.default_rng(9)
    qm2, qa2 = _rand_stats(rng, 2, fc)
    k2 = rng.standard_normal((4, hd))
    args = (O.as_complex(qm2), O.mlr_weight(qm2, qa2), O.rope_omega(hd, 1e4), 31, [1, 8])
    np.testing.assert_allclose(O.raw_scores(2.5 * k2, *args), 2.5 * O.raw_scores(k2, *args),
                               rtol=1e-12)


def test_mlr_weight_is_nonnegative_residual():
    qm = np.array([[[3.0, 4.0], [0.0, 0.0]]])
    q_abs = np.array([[6.0, 2.0]])
    np.testing.assert_allclose(O.mlr_weight(qm, q_abs), [[1.0, 2.0]])
    np.testing.assert_allclose(O.mlr_weight(qm, None), [[0.0, 0.0]])


def test_phase_precision_at_long_context_against_40_digits():
    """Phases at p + d up to 196608 match a 40-digit evaluation of the same
    float64 omega (the long-context precision the pass needs)."""
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 40
    hd, theta = 256, 1e7
    fc = hd // 2
    om = O.rope_omega(hd, theta)
    for f in (0, 1, 5, 60, 127):
        k = np.zeros((2, hd))
        k[0, f] = 1.0            # k_f = 1:  raw =  Re(e^{i w (p+d)}) = cos
        k[1, f + fc] = -1.0      # k_f = -i: raw = -Im(...)          = -sin
        qm = np.zeros((1, fc), dtype=complex)
        qm[0, f] = 1.0
        for p, d in ((131072, 65536), (98304, 1), (32768, 4096)):
            got = O.raw_scores(k, qm, np.zeros((1, fc)), om, p, [d])[:, 0]
            arg = mpmath.mpf(om[f]) * (p + d)
            # one float64 rounding of the product w*(p+d), then 1-ulp cos/sin
            tol = 2.0 * float(arg) * 2.0 ** -53 + 4e-16
            assert abs(got[0] - float(mpmath.cos(arg))) < tol
            assert abs(got[1] + float(mpmath.sin(arg))) < tol


def test_rope_omega_values():
    om = O.rope_omega(128, 1e6)
    assert om[0] == 1.0
    assert om[64 - 1] == pytest.approx(1e6 ** (-126 / 128), rel=1e-15)
    assert np.all(np.diff(om) < 0)
    assert list(O.default_future_offsets()) == [2 ** j for j in range(17)]


# ---------------------------------------------------------- normalisation ---

def test_znorm_closed_form():
    raw = np.array([[1.0], [2.0], [3.0], [4.0]])
    sd = math.sqrt(1.25)
    np.testing.assert_allclose(O.znorm(raw)[:, 0], (raw[:, 0] - 2.5) / (sd + 1e-6), rtol=1e-15)
    const = np.full((7, 2), 3.25)
    assert np.all(O.znorm(const) == 0.0)
    # a segment without live rows: nothing to normalise, and no moments are taken
    import warnings
    with warnings.catch_warnings():
        warnings.simplefilter("error")
        empty = O.znorm(np.zeros((0, 4)))
    assert empty.shape == (0, 4)
    assert O.gqa_max(empty).shape == (0,)


def test_znorm_moments_and_gqa_max():
    rng = np.random.default_rng(11)
    raw = rng.standard_normal((500, 4)) * [1.0, 10.0, 0.1, 3.0] + [5.0, -2.0, 100.0, 0.0]
    z = O.znorm(raw)
    np.testing.assert_allclose(z.mean(axis=0), 0.0, atol=1e-12)
    sd = raw.std(axis=0)
    np.testing.assert_allclose(z.std(axis=0), sd / (sd + 1e-6), rtol=1e-12)
    s = O.gqa_max(z)
    assert np.all(s >= z.max(axis=1)) and np.all(s <= z.max(axis=1))
    np.testing.assert_array_equal(O.gqa_max(z[:, :1]), z[:, 0])              # G = 1
    same = np.repeat(raw[:, :1], 4, axis=1)
    np.testing.assert_allclose(O.gqa_max(O.znorm(same)), O.znorm(raw[:, :1])[:, 0], rtol=1e-12)


def test_head_map_default_and_custom():
    assert O.heads_of_kv(8, 2) == [[0, 1, 2, 3], [4, 5, 6, 7]]
    assert O.heads_of_kv(4, 2, [1, 0, 1, 0]) == [[1, 3], [0, 2]]


# -------------------------------------------------------------- selection ---

def _select_by_repeated_best(s, n, b, sink, window):
    """Independent selection: pick the best remaining candidate k times
    (higher score first, lower row on equal scores, NaN never before a number)."""
    cand = list(range(sink, n - window))
    chosen = []
    for _ in range(b - sink - window):
        best = None
        for r in cand:
            if r in chosen:
                continue
            if best is None:
                best = r
                continue
            sr, sb = s[r], s[best]
            if math.isnan(sb) and not math.isnan(sr):
                best = r
            elif not math.isnan(sr) and not math.isnan(sb) and sr > sb:
                best = r
        chosen.append(best)
    return sorted(list(range(sink)) + chosen + list(range(n - window, n)))


@pytest.mark.parametrize("seed", range(40))
def test_select_matches_independent_selection_with_ties(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(6, 40))
    sink = int(rng.integers(0, 3))
    window = int(rng.integers(0, 4))
    b = int(rng.integers(sink + window, n))          # b < n: a real pass
    s = rng.choice([-1.5, 0.0, 0.25, 0.25, 2.0, np.nan if seed % 5 == 0 else 3.0], size=n)
    got = O.select_keep(s, n, b, sink, window)
    assert list(got) == _select_by_repeated_best(list(s), n, b, sink, window)


@pytest.mark.parametrize("seed", range(12))
def test_select_is_the_unique_ordered_top_k_exhaustive(seed):
    rng = np.random.default_rng(100 + seed)
    n, sink, window = 11, 1, 2
    b = int(rng.integers(sink + window, n))
    s = rng.choice([0.0, 1.0, 1.0, 2.0, -3.0], size=n).astype(np.float64)
    cand = list(range(sink, n - window))
    k = b - sink - window
    valid = []
    for subset in itertools.combinations(cand, k):
        inside = set(subset)
        ok = all((s[a] > s[c]) or (s[a] == s[c] and a < c)
                 for a in inside for c in cand if c not in inside)
        if ok:
            valid.append(sorted(list(range(sink)) + list(subset) + list(range(n - window, n))))
    assert len(valid) == 1
    assert list(O.select_keep(s, n, b, sink, window)) == valid[0]


def test_select_invariants_noop_and_budget_error():
    rng = np.random.default_rng(7)
    s = rng.standard_normal(100)
    keep = O.select_keep(s, 100, 40, 4, 16)
    assert len(keep) == 40
    assert np.all(np.diff(keep) > 0)
    assert set(range(4)) <= set(keep) and set(range(84, 100)) <= set(keep)
    np.testing.assert_array_equal(O.select_keep(s, 30, 40, 4, 16), np.arange(30))
    np.testing.assert_array_equal(O.select_keep(s, 40, 40, 4, 16), np.arange(40))
    with pytest.raises(O.BudgetError):
        O.select_keep(s, 100, 19, 4, 16)
    keep0 = O.select_keep(s, 100, 20, 4, 16)             # k = 0: only protected rows
    np.testing.assert_array_equal(keep0, list(range(4)) + list(range(84, 100)))


def test_select_signed_zero_is_a_tie():
    s = np.array([0.0, -0.0, 0.0, -0.0, 1.0])
    np.testing.assert_array_equal(O.select_keep(s, 5, 3, 0, 0), [0, 1, 4])


def test_budget_rows_floor():
    assert O.budget_rows(0.5, 512) == 256
    assert O.budget_rows(0.25, 32768) == 8192
    assert O.budget_rows(0.5, 12288) == 6144
    assert O.budget_rows(0.25, 98710) == 24677
    assert O.budget_rows(0.3, 10) == 3


# ------------------------------------------------------------- compaction ---

def test_compact_rows_exact_gather_and_untouched_tail():
    rng = np.random.default_rng(13)
    plane = rng.standard_normal((20, 3))
    keep = np.array([0, 2, 3, 7, 11, 19])
    out = O.compact_rows(plane, keep)
    np.testing.assert_array_equal(out[:6], plane[keep])
    np.testing.assert_array_equal(out[6:], plane[6:])


def test_q8_0_dequant_hand_block():
    qs = np.arange(-64, 64, dtype=np.int8).reshape(1, 128)
    d = np.array([[0.5, 0.25, 2.0, 0.0]], dtype=np.float16)
    got = O.dequant_q8_0(qs, d)
    want = np.concatenate([np.arange(-64, -32) * 0.5, np.arange(-32, 0) * 0.25,
                           np.arange(0, 32) * 2.0, np.zeros(32)])
    np.testing.assert_array_equal(got[0], want)


# ------------------------------------------------------------ whole layer ---

def test_evict_layer_tiny_invariants():
    w = W.get_workload("tiny")
    qm, qa = W.make_stats(w)
    cache = W.layer_host(w, 0)
    out, info = O.evict_layer(cache, qm, qa, layer=0, n_kv_heads=w.n_kv_heads,
                              head_dim=w.head_dim, rope_theta=w.rope_theta, cur_pos=w.cur_pos,
                              n_ctx=w.n_ctx, budget_frac=w.budget_frac, window=w.window,
                              sink=w.sink)
    assert list(out["n_live"]) == [256]
    for (s, g), it in info.items():
        r0, keep = it["row0"], it["keep"]
        assert len(keep) == 256
        np.testing.assert_array_equal(out["k"][r0:r0 + 256], cache["k"][r0 + keep])
        np.testing.assert_array_equal(out["v"][r0:r0 + 256], cache["v"][r0 + keep])
        pos = out["pos"][r0:r0 + 256]
        assert np.all(np.diff(pos) > 0)
        assert list(pos[:4]) == [0, 1, 2, 3] and list(pos[-64:]) == list(range(448, 512))
        np.testing.assert_array_equal(out["k"][r0 + 256:r0 + 512], cache["k"][r0 + 256:r0 + 512])


def test_evict_layer_noop_is_byte_identical():
    w = W.get_workload("tiny")
    qm, qa = W.make_stats(w)
    cache = W.layer_host(w, 0)
    out, _ = O.evict_layer(cache, qm, qa, layer=0, n_kv_heads=2, head_dim=64, rope_theta=1e4,
                           cur_pos=[512], n_ctx=[1024], budget_frac=0.5, window=64, sink=4)
    for key in ("k", "v", "pos", "n_live"):
        assert out[key].tobytes() == cache[key].tobytes()


def test_scores_follow_absolute_position_not_row_count():
    """Second pass: the phase position is the absolute decode position; using
    the compacted row count instead changes the scores ([Worklog] 2026-04-18)."""
    w = W.get_workload("tiny")
    qm, qa = W.make_stats(w)
    cache = W.layer_host(w, 0)
    kw = dict(layer=0, n_kv_heads=2, head_dim=64, rope_theta=1e4, n_ctx=[512],
              budget_frac=0.5, window=64, sink=4)
    out1, _ = O.evict_layer(cache, qm, qa, cur_pos=[512], **kw)
    out1["n_live"][:] = 300
    a, ia = O.evict_layer(out1, qm, qa, cur_pos=[640], **kw)
    b, ib = O.evict_layer(out1, qm, qa, cur_pos=[300], **kw)
    assert not np.allclose(ia[(0, 0)]["raw"], ib[(0, 0)]["raw"])
    kf = out1["k"][:300].astype(np.float64)
    ref = O.raw_scores(kf, O.as_complex(qm[0, :4]), O.mlr_weight(qm[0, :4], qa[0, :4]),
                       O.rope_omega(64, 1e4), 640, O.default_future_offsets())
    np.testing.assert_allclose(ia[(0, 0)]["raw"], ref, rtol=1e-14)


# ------------------------------------------------- values the pages print ---

def test_golden_worklog_compaction_schedule():
    """The worklog's profile log: trigger kv_budget + divide_length = 3200 and
    compactions #1-#4 at abs_pos 3200/3328/3456/3584, 3200 -> 3072 rows."""
    with open(os.path.join(GOLDEN, "worklog_compaction_schedule.json")) as fh:
        gold = json.load(fh)
    budget, interval = gold["kv_budget"], gold["divide_length"]
    assert budget + interval == gold["trigger"]
    rows, log = 0, []
    rng = np.random.default_rng(0)
    for abs_pos in range(1, gold["compactions"][-1]["abs_pos"] + 1):
        rows += 1          # one decoded token appended (decode-only accounting)
        if O.should_evict(rows, budget, interval):
            keep = O.select_keep(rng.standard_normal(rows), rows, budget, 0, 0)
            log.append({"abs_pos": abs_pos, "old_rows": rows, "kept_rows": len(keep)})
            rows = len(keep)
    assert log == gold["compactions"]


def test_golden_worklog_prompt_accounting():
    """6144/1024 policy: the native trigger row count is 7168 even though the
    dense cache (prompt included) is 155 rows longer."""
    with open(os.path.join(GOLDEN, "worklog_prompt_accounting.json")) as fh:
        gold = json.load(fh)
    assert gold["kv_budget"] + gold["divide_length"] == gold["native_rows_before"]
    assert O.should_evict(gold["native_rows_before"], gold["kv_budget"], gold["divide_length"])
    assert not O.should_evict(gold["native_rows_before"] - 1, gold["kv_budget"],
                              gold["divide_length"])
    assert gold["dense_cache_length"] - gold["native_rows_before"] == gold["gap"]


# ---------------------------------------------------------------------------
# calibration statistics ([Doc] §2; q_mean / q_abs layout of §5 Phase C)
# ---------------------------------------------------------------------------

def test_calibrate_constant_stream():
    # every token the same: the means are that token's pairs and moduli
    rng = np.random.default_rng(21)
    one = rng.standard_normal((1, 3, 8))
    q = np.repeat(one, 5, axis=0)
    q_mean, q_abs = O.calibrate(q)
    assert q_mean.shape == (3, 4, 2) and q_abs.shape == (3, 4)
    np.testing.assert_allclose(q_mean[..., 0], one[0, :, :4], rtol=0, atol=1e-15)
    np.testing.assert_allclose(q_mean[..., 1], one[0, :, 4:], rtol=0, atol=1e-15)
    np.testing.assert_allclose(q_abs, np.hypot(one[0, :, :4], one[0, :, 4:]), rtol=1e-15)


def test_calibrate_literal_loop():
    # brute force: a per-token, per-pair loop with math.hypot
    rng = np.random.default_rng(22)
    q = rng.standard_normal((7, 2, 6))
    q_mean, q_abs = O.calibrate(q)
    for h in range(2):
        for f in range(3):
            re = sum(q[t, h, f] for t in range(7)) / 7
            im = sum(q[t, h, f + 3] for t in range(7)) / 7
            ab = sum(math.hypot(q[t, h, f], q[t, h, f + 3]) for t in range(7)) / 7
            assert abs(q_mean[h, f, 0] - re) < 1e-14 and abs(q_mean[h, f, 1] - im) < 1e-14
            assert abs(q_abs[h, f] - ab) < 1e-14


def test_calibrate_concatenation_and_resultant_length():
    # the means over two batches weight the batch means by their token counts,
    # and |q_mean| <= q_abs (mean resultant length <= 1) with equality for a
    # stream whose pairs all point the same way
    rng = np.random.default_rng(23)
    a, b = rng.standard_normal((4, 2, 8)), rng.standard_normal((9, 2, 8))
    ma, aa = O.calibrate(a)
    mb, ab = O.calibrate(b)
    m, ab_all = O.calibrate(np.concatenate([a, b]))
    np.testing.assert_allclose(m, (4 * ma + 9 * mb) / 13, rtol=1e-13)
    np.testing.assert_allclose(ab_all, (4 * aa + 9 * ab) / 13, rtol=1e-13)
    assert np.all(np.hypot(m[..., 0], m[..., 1]) <= ab_all + 1e-15)
    scale = rng.uniform(0.5, 2.0, size=(6, 1, 1))
    aligned = scale * np.repeat(rng.standard_normal((1, 2, 8)), 6, axis=0)
    ma2, aa2 = O.calibrate(aligned)
    np.testing.assert_allclose(np.hypot(ma2[..., 0], ma2[..., 1]), aa2, rtol=1e-13)
    # M = q_abs - |q_mean| is then zero: no magnitude term
    np.testing.assert_allclose(O.mlr_weight(ma2.reshape(1, 2, 4, 2)[0], aa2), 0.0, atol=1e-13)


# ---------------------------------------------------------------------------
# non-rotary (content) dims ([Doc] §4 gate line ``nonrot=``, §6 "Non-rotary
# models"; reading: the first rot dims are NEOX-rotary, the rest never rotate)
# ---------------------------------------------------------------------------

def _brute_raw_partial(k_row, qm_head, q_abs_head, qn_head, theta, rot, p, offsets):
    """One score by real arithmetic on a head whose first ``rot`` dims are
    rotary: rotate the rotary half-pairs (f, f + rot/2) of the mean query by
    2x2 matrices at p + d, leave the other dims as the mean non-rotary query,
    dot the whole vector with the key, average over d, add the norm term on
    the rotary pairs only."""
    hd = len(k_row)
    fr = rot // 2
    total = 0.0
    for d in offsets:
        qvec = [0.0] * hd
        for f in range(fr):
            w = math.pow(theta, -2.0 * f / rot)
            a, b = qm_head[f][0], qm_head[f][1]
            c, s = math.cos(w * (p + d)), math.sin(w * (p + d))
            qvec[f] = a * c - b * s
            qvec[f + fr] = a * s + b * c
        for e in range(hd - rot):
            qvec[rot + e] = qn_head[e]
        total += sum(qvec[i] * k_row[i] for i in range(hd))
    total /= len(offsets)
    for f in range(fr):
        m = q_abs_head[f] - math.hypot(qm_head[f][0], qm_head[f][1])
        total += m * math.sqrt(k_row[f] ** 2 + k_row[f + fr] ** 2)
    return total


@pytest.mark.parametrize("hd,nonrot,g,theta,p,offsets", [
    (8, 4, 2, 100.0, 13, [1, 3, 7]),
    (16, 8, 4, 1e4, 4096, [1, 2, 4, 8, 16]),
    (12, 2, 1, 10.0, 5, [0, 2]),
    (16, 14, 2, 500.0, 70000, [1, 65536]),
])
def test_nonrot_raw_score_matches_real_vector_bruteforce(hd, nonrot, g, theta, p, offsets):
    rng = np.random.default_rng(hd * 31 + nonrot)
    rot = hd - nonrot
    k = rng.standard_normal((5, hd))
    qm, q_abs = _rand_stats(rng, g, rot // 2)
    qn = rng.standard_normal((g, nonrot))
    got = O.raw_scores(k, O.as_complex(qm), O.mlr_weight(qm, q_abs),
                       O.rope_omega(hd, theta, nonrot), p, offsets, qn)
    for r in range(5):
        for j in range(g):
            want = _brute_raw_partial(list(k[r]), qm[j].tolist(), list(q_abs[j]), list(qn[j]),
                                      theta, rot, p, offsets)
            # the brute force takes cos / sin of angles up to w (p + d) unreduced:
            # an absolute error of about 2^-53 (p + d) per unit of |q| |k|
            slack = 1e-15 * (p + max(offsets)) * float(np.abs(k[r]).sum() * (np.abs(qm[j]).sum() + 1.0))
            assert abs(got[r, j] - want) <= 1e-12 * max(1.0, abs(want)) + slack


def _rope_partial(x, pos, theta, rot):
    """Partial NEOX RoPE of rows x at positions pos: pairs (f, f + rot/2) of the
    first rot dims rotated by pos * theta^(-2f/rot), the other dims unchanged."""
    fr = rot // 2
    w = np.array([math.pow(theta, -2.0 * f / rot) for f in range(fr)])
    ang = np.asarray(pos, np.float64)[:, None] * w[None, :]
    c, s = np.cos(ang), np.sin(ang)
    a, b = x[:, :fr], x[:, fr:rot]
    return np.concatenate([a * c - b * s, a * s + b * c, x[:, rot:]], axis=1)


def test_nonrot_score_is_the_mean_logit_of_the_calibration_queries():
    """With M = 0 the score is the expected attention logit: the mean, over a
    stream of real pre-RoPE queries and over the offsets, of the partial-RoPE
    query at p + d dotted with the partial-RoPE key at its own position. The
    statistics come from calibrate / calibrate_nonrot of the same stream."""
    rng = np.random.default_rng(41)
    hd, nonrot, theta, n_tok = 16, 6, 1e4, 9
    rot = hd - nonrot
    q = rng.standard_normal((n_tok, 1, hd)) + 0.7
    qm, _ = O.calibrate(q, nonrot)
    qn = O.calibrate_nonrot(q, nonrot)
    k_pre = rng.standard_normal((6, hd))
    kpos = np.array([0, 3, 17, 100, 2048, 5000])
    k_rot = _rope_partial(k_pre, kpos, theta, rot)
    p, offsets = 6000, [1, 4, 64, 1024]
    got = O.raw_scores(k_rot, O.as_complex(qm), np.zeros((1, rot // 2)),
                       O.rope_omega(hd, theta, nonrot), p, offsets, qn)
    want = np.zeros(6)
    for d in offsets:
        for t in range(n_tok):
            q_at = _rope_partial(q[t], [p + d], theta, rot)[0]
            want += k_rot @ q_at
    want /= n_tok * len(offsets)
    np.testing.assert_allclose(got[:, 0], want, rtol=1e-11, atol=1e-11)


def test_nonrot_special_cases():
    rng = np.random.default_rng(43)
    hd, nonrot = 12, 4
    rot = hd - nonrot
    k = rng.standard_normal((7, hd))
    qn = rng.standard_normal((2, nonrot))
    zero = np.zeros((2, rot // 2, 2))
    om = O.rope_omega(hd, 1e4, nonrot)
    # no rotary statistics: the score is the textbook dot product on the content dims
    got = O.raw_scores(k, O.as_complex(zero), np.zeros((2, rot // 2)), om, 99, [1, 2], qn)
    np.testing.assert_allclose(got, k[:, rot:] @ qn.T, rtol=1e-14, atol=1e-14)
    # the content term does not depend on the position or the offsets
    qm, qa = _rand_stats(rng, 2, rot // 2)
    args = (O.as_complex(qm), O.mlr_weight(qm, qa), om)
    a = O.raw_scores(k, *args, 10, [1, 2], qn) - O.raw_scores(k, *args, 10, [1, 2], None)
    b = O.raw_scores(k, *args, 77777, [3], qn) - O.raw_scores(k, *args, 77777, [3], None)
    np.testing.assert_allclose(a, k[:, rot:] @ qn.T, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(b, a, rtol=1e-12, atol=1e-12)
    # the rotary part only sees the first rot dims: changing a content dim of
    # the key moves the score by exactly the matching query entry
    k2 = k.copy()
    k2[:, rot + 1] += 1.0
    d = O.raw_scores(k2, *args, 5, [1], qn) - O.raw_scores(k, *args, 5, [1], qn)
    np.testing.assert_allclose(d, np.broadcast_to(qn[:, 1], d.shape), rtol=1e-12, atol=1e-12)
    # frequencies over the rotary dims only
    np.testing.assert_allclose(om, [1e4 ** (-2.0 * f / rot) for f in range(rot // 2)], rtol=1e-15)
    # nonrot = 0 is the all-rotary score
    qm8, qa8 = _rand_stats(rng, 2, hd // 2)
    np.testing.assert_array_equal(
        O.raw_scores(k, O.as_complex(qm8), O.mlr_weight(qm8, qa8), O.rope_omega(hd, 1e4, 0), 8, [1, 2]),
        O.raw_scores(k, O.as_complex(qm8), O.mlr_weight(qm8, qa8), O.rope_omega(hd, 1e4), 8, [1, 2]))


def test_calibrate_nonrot_literal_loop():
    rng = np.random.default_rng(44)
    q = rng.standard_normal((5, 2, 10))
    qm, qa = O.calibrate(q, 4)
    qn = O.calibrate_nonrot(q, 4)
    assert qm.shape == (2, 3, 2) and qa.shape == (2, 3) and qn.shape == (2, 4)
    for h in range(2):
        for f in range(3):
            re = sum(q[t, h, f] for t in range(5)) / 5
            im = sum(q[t, h, f + 3] for t in range(5)) / 5
            assert abs(qm[h, f, 0] - re) < 1e-14 and abs(qm[h, f, 1] - im) < 1e-14
        for e in range(4):
            assert abs(qn[h, e] - sum(q[t, h, 6 + e] for t in range(5)) / 5) < 1e-14
