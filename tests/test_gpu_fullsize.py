"""Element-wise parity at full workload size, where the persistent scorer's
every warp streams several pieces through its two-stage ring (so the second
stage, the ring's phase flips and moment partials spanning several pieces are
all exercised), the z-max score the staged evict path selects with (kept in
the workspace), and the cooperative grid select that takes segments over
262144 rows.

Every row of each sampled segment is compared with the oracle at the stated
tolerance (scores: relative 1e-3, raw with tau = the head's RMS, z-max with
tau = 1); selections on given scores are bit-exact. The GPU reads caches from
the device generator, the oracle the bit-identical host twin.
"""
import numpy as np
import pytest

from oracle import tria_oracle as O
from synth import workloads as W

import _util as U

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

PIECE_BYTES = 8192          # bytes of keys per scorer piece (at most)
SCORE_WARPS_PER_SM = 12


def _oracle_scores(w, layer, s, g, qm, qa):
    seg = W.segment_host(w, layer, s, g, rows=w.n_live[s], values=False)
    kf = O.keys_f64(seg["k"], seg["k_scale"])
    hs = O.heads_of_kv(w.n_q_heads, w.n_kv_heads)[g]
    return O.segment_scores(kf, O.as_complex(qm[layer][hs]), O.mlr_weight(qm[layer][hs], qa[layer][hs]),
                            O.rope_omega(w.head_dim, w.rope_theta), w.cur_pos[s], O.default_future_offsets())


@pytest.mark.parametrize("name,layer,segs", [
    ("qwen3_8b_layer", 0, [(0, 0), (0, 3), (0, 7)]),
    ("q8_0", 5, [(0, 1), (0, 6)]),
    ("batched_long", 1, None),      # the longest sequence's head 2 and the shortest's head 0
])
def test_full_size_scores_every_row(lib, name, layer, segs):
    from synth import device as D
    D.build()
    w = W.get_workload(name)
    qm, qa = W.make_stats(w)
    st = lib.Stats(qm, qa, n_kv_heads=w.n_kv_heads, head_dim=w.head_dim, rope_theta=w.rope_theta)
    t = D.alloc_layer(w)
    D.fill_layer(w, layer, t)
    cache, pol = U.workload_cache(lib, w, t), U.workload_policy(lib, w)
    ws = U.new_workspace(lib, cache, w.group)
    rows = w.total_rows()
    s_out = torch.full((rows,), float("nan"), device="cuda")
    raw_out = torch.full((rows, w.group), float("nan"), device="cuda")
    lib.score(st, layer, cache, pol, s_out, raw_out, ws=ws)
    assert lib.device_status(ws) == lib.OK
    # the layer's pieces outnumber the scorer's warps: every warp takes several
    rows_per_piece = min(64, PIECE_BYTES // w.k_row_bytes()) // 16 * 16
    pieces = sum(w.n_kv_heads * -(-n // rows_per_piece) for n in w.n_live)
    warps = torch.cuda.get_device_properties(0).multi_processor_count * SCORE_WARPS_PER_SM
    assert pieces >= 4 * warps, (pieces, warps)
    if segs is None:
        lo, hi = int(np.argmin(w.n_live)), int(np.argmax(w.n_live))
        segs = [(hi, 2), (lo, 0)]
    r0s = w.seq_row0()
    for s, g in segs:
        n = w.n_live[s]
        r0 = int(r0s[s] + g * w.capacity[s])
        raw, sc = _oracle_scores(w, layer, s, g, qm, qa)
        e_raw, e_s = U.assert_scores_close(raw_out[r0:r0 + n].cpu().numpy(), raw, s_out[r0:r0 + n].cpu().numpy(),
                                           sc, f"{name} L{layer} s{s} g{g}")
        assert e_raw <= U.RTOL and e_s <= U.RTOL
    st.close()
    del t
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name,layer,segs", [
    ("qwen3_8b_layer", 0, [(0, 1), (0, 6)]),
    ("q8_0", 2, [(0, 4)]),
    ("batched_long", 0, None),      # the longest sequence's head 1
])
def test_staged_evict_zmax_every_row(lib, name, layer, segs):
    """The z-max score the staged evict path selects with (computed inside the
    cluster select and kept in the workspace) against the oracle, every live
    row of sampled full-size segments, then the keep-set rule on the same rows."""
    from synth import device as D
    D.build()
    w = W.get_workload(name)
    qm, qa = W.make_stats(w)
    st = lib.Stats(qm, qa, n_kv_heads=w.n_kv_heads, head_dim=w.head_dim, rope_theta=w.rope_theta)
    t = D.alloc_layer(w)
    D.fill_layer(w, layer, t)
    pos0 = t["pos"].clone()
    cache, pol = U.workload_cache(lib, w, t), U.workload_policy(lib, w)
    ws = U.new_workspace(lib, cache, w.group)
    lib.evict_staged(st, layer, cache, pol, ws=ws)
    assert lib.device_status(ws) == lib.OK
    zs = lib.workspace_scores(ws, cache)
    if segs is None:
        segs = [(int(np.argmax(w.n_live)), 1)]
    r0s = w.seq_row0()
    for s, g in segs:
        n = w.n_live[s]
        r0 = int(r0s[s] + g * w.capacity[s])
        raw, sc = _oracle_scores(w, layer, s, g, qm, qa)
        got = zs[r0:r0 + n].cpu().numpy()
        err = np.abs(got - sc) / np.maximum(np.abs(sc), 1.0)
        assert err.max() <= U.RTOL, f"{name} s{s} g{g}: z-max rel err {err.max():.3e}"
        b = lib.budget_rows(w.budget_frac, w.n_ctx[s])
        want = O.select_keep(sc, n, b, w.sink, w.window)
        kept_pos = t["pos"][r0:r0 + b].cpu().numpy()
        gk = np.searchsorted(pos0[r0:r0 + n].cpu().numpy(), kept_pos)
        U.assert_keep_sets_match(gk, want, sc, n, b, w.sink, w.window, f"{name} s{s} g{g}")
    st.close()
    del t
    torch.cuda.empty_cache()


def _dummy_cache(lib, case):
    """A layer cache for select-only calls: key / value / position planes are
    never read by the select, so small placeholder tensors stand in for them."""
    dummy = torch.zeros(64, dtype=torch.float16, device="cuda")
    n_live = torch.tensor(case.n_live, dtype=torch.int32, device="cuda")
    return lib.LayerCache(k=dummy, v=dummy, pos=dummy.view(torch.int32), n_live=n_live,
                          seq_row0=case.seq_row0(), capacity=case.capacity, head_dim=case.hd,
                          n_kv_heads=case.n_kv, k_type="f16", v_type="f16")


def test_cooperative_select_bit_exact_over_262144_rows(lib):
    """Segments over 8 x 32768 rows leave the cluster select for the cooperative
    grid path (bounded grid barriers, last-arriver bin search, tie cut): two
    sequences of 300000 and 270000 rows, two KV heads, forced ties, NaN, +-0."""
    case = U.Case(n_kv=2, group=1, hd=64, k_type="f16", v_type="f16", n_live=[300000, 269000],
                  capacity=[300000, 270000], cur_pos=[0, 0], budget_rows=[75000, 268000], sink=4, window=512)
    cache, pol = _dummy_cache(lib, case), U.lib_policy(lib, case)
    ws = U.new_workspace(lib, cache, 0)
    rows = case.total_rows()
    rng = np.random.default_rng(17)
    levels = np.array([-2.0, -0.0, 0.0, 0.5, 0.5, 1.25, np.inf, -np.inf, np.nan], np.float32)
    score = np.where(rng.random(rows) < 0.5, rng.choice(levels, rows), rng.standard_normal(rows)).astype(np.float32)
    keep = torch.full((rows,), -7, dtype=torch.int32, device="cuda")
    for _ in range(2):   # the second call reuses the workspace (self-resetting counters, barrier generation)
        keep.fill_(-7)
        lib.select(torch.from_numpy(score).cuda(), cache, pol, keep, ws=ws)
        assert lib.device_status(ws) == lib.OK
        got = keep.cpu().numpy()
        r0s = case.seq_row0()
        for s in range(case.n_seqs):
            for g in range(case.n_kv):
                r0 = int(r0s[s] + g * case.capacity[s])
                n, b = case.n_live[s], case.budget_rows[s]
                want = O.select_keep(score[r0:r0 + n], n, b, case.sink, case.window)
                np.testing.assert_array_equal(got[r0:r0 + len(want)], want, err_msg=f"seq {s} head {g}")
                assert np.all(got[r0 + len(want):r0 + case.capacity[s]] == -7)


def test_evict_end_to_end_over_262144_rows(lib):
    """A whole pass on a 300000-row segment: scores, the cooperative select and
    the compaction, against the oracle (keep-set rule at the cut, exact gathers)."""
    case = U.Case(n_kv=1, group=2, hd=64, k_type="f16", v_type="f16", n_live=[300000], capacity=[300000],
                  cur_pos=[300000], budget_frac=0.25, window=512, sink=4, seed=23)
    host = U.build_host(case)
    dev = U.to_device(host)
    cache, pol = U.lib_cache(lib, case, dev), U.lib_policy(lib, case)
    ws = U.new_workspace(lib, cache, case.group)
    st = lib.Stats(host["q_mean"], host["q_abs"], n_kv_heads=case.n_kv, head_dim=case.hd, rope_theta=case.theta)
    lib.evict(st, 0, cache, pol, ws=ws)
    assert lib.device_status(ws) == lib.OK
    n, b = case.n_live[0], case.budgets()[0]
    assert dev["n_live"].cpu().tolist() == [b]
    kf = O.keys_f64(host["k"][:n], None)
    hs = O.heads_of_kv(case.n_kv * case.group, case.n_kv)[0]
    raw, sc = O.segment_scores(kf, O.as_complex(host["q_mean"][0][hs]),
                               O.mlr_weight(host["q_mean"][0][hs], host["q_abs"][0][hs]),
                               O.rope_omega(case.hd, case.theta), case.cur_pos[0], O.default_future_offsets())
    # the cooperative path's z-max, every row
    got = lib.workspace_scores(ws, cache)[:n].cpu().numpy()
    err = np.abs(got - sc) / np.maximum(np.abs(sc), 1.0)
    assert err.max() <= U.RTOL, f"z-max rel err {err.max():.3e}"
    want = O.select_keep(sc, n, b, case.sink, case.window)
    pos_after = dev["pos"][:b].cpu().numpy()
    gk = np.searchsorted(host["pos"][:n], pos_after)
    U.assert_keep_sets_match(gk, want, sc, n, b, case.sink, case.window, "300000 rows")
    np.testing.assert_array_equal(dev["k"][:b].cpu().numpy(), host["k"][gk])
    np.testing.assert_array_equal(dev["v"][:b].cpu().numpy(), host["v"][gk])
    st.close()
