"""The fused pass (one persistent kernel: score items, last-finisher select,
moves) against the oracle, through tria_evict / tria_evict_model.

Checks: the z-max score of every live row of the evict path (score_out)
within the stated tolerance; keep-sets identical except rows within the
tolerance of the cut; compacted K / V / scales / positions exact gathers of the
kept rows; rows past the budget untouched; n_live set per layer; segments at
or below budget byte-identical; several layers in one call; a workspace shared
by fused, staged and model calls.
"""
import numpy as np
import pytest

from oracle import tria_oracle as O
from synth import workloads as W

import _util as U

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _layers(cfg, n_layers):
    """n_layers caches of one shape (different contents per layer) and the
    statistics of all layers."""
    cases, hosts = [], []
    for l in range(n_layers):
        case = U.Case(**dict(cfg, seed=cfg.get("seed", 11) + 100 * l))
        hosts.append(U.build_host(case))
        cases.append(case)
    qm = np.concatenate([h["q_mean"] for h in hosts], axis=0)
    qa = np.concatenate([h["q_abs"] for h in hosts], axis=0)
    return cases, hosts, qm, qa


def _oracle_segment(case, host, qm, qa, layer, s, g):
    r0 = int(host["seq_row0"][s] + g * case.capacity[s])
    n = case.n_live[s]
    kf = O.keys_f64(host["k"][r0:r0 + n], None if host["k_scale"] is None else host["k_scale"][r0:r0 + n])
    hs = O.heads_of_kv(case.n_kv * case.group, case.n_kv)[g]
    raw, sc = O.segment_scores(kf, O.as_complex(qm[layer][hs]), O.mlr_weight(qm[layer][hs], qa[layer][hs]),
                               O.rope_omega(case.hd, case.theta), case.cur_pos[s],
                               O.default_future_offsets() if case.offsets is None else case.offsets)
    return r0, n, raw, sc


def _check_layer(case, host, got, qm, qa, layer, scores=None, what=""):
    """One layer's compacted cache against the oracle (and its scores)."""
    budgets = case.budgets()
    n_live_got = got["n_live"]
    for s in range(case.n_seqs):
        n, b = case.n_live[s], budgets[s]
        assert n_live_got[s] == min(n, b), f"{what} seq {s} n_live"
        for g in range(case.n_kv):
            r0, _, raw, sc = _oracle_segment(case, host, qm, qa, layer, s, g)
            cap = case.capacity[s]
            if n <= b:
                for name in ("k", "k_scale", "v", "v_scale", "pos"):
                    if host[name] is not None:
                        assert got[name][r0:r0 + cap].tobytes() == host[name][r0:r0 + cap].tobytes(), what
                continue
            if scores is not None:
                err = np.abs(scores[r0:r0 + n] - sc) / np.maximum(np.abs(sc), 1.0)
                assert err.max() <= U.RTOL, f"{what} seq {s} head {g}: z-max rel err {err.max():.3e}"
            want = O.select_keep(sc, n, b, case.sink, case.window)
            gk = np.searchsorted(host["pos"][r0:r0 + n], got["pos"][r0:r0 + b])
            U.assert_keep_sets_match(gk, want, sc, n, b, case.sink, case.window, f"{what} seq {s} head {g}")
            for name in ("k", "k_scale", "v", "v_scale"):
                if host[name] is None:
                    continue
                np.testing.assert_array_equal(got[name][r0:r0 + b], host[name][r0 + gk], err_msg=f"{what} {name}")
                assert got[name][r0 + b:r0 + cap].tobytes() == host[name][r0 + b:r0 + cap].tobytes(), what


FUSED_CASES = [
    # fp16, hd 128, G 4, ragged sequences, a no-op sequence, window / sink
    dict(n_kv=2, group=4, hd=128, k_type="f16", v_type="f16", n_live=[3000, 1500, 100], capacity=[3072, 1600, 128],
         cur_pos=[100000, 1500, 3], budget_frac=0.25, n_ctx=[3000, 1500, 1000], window=128, sink=4),
    # q8_0 keys with fp16 values, several score items per segment
    dict(n_kv=2, group=4, hd=128, k_type="q8_0", v_type="f16", n_live=[5000, 3333], capacity=[5000, 3400],
         cur_pos=[65536, 777], budget_frac=0.5, window=512, sink=4),
    # hd 256, G 2, q8_0 values; hd 64 with G 8 and G 1; tiny segments (fewer rows than one item)
    dict(n_kv=1, group=2, hd=256, k_type="f16", v_type="q8_0", n_live=[4100, 50], capacity=[4100, 64],
         cur_pos=[9000, 50], budget_frac=0.5, window=16, sink=4),
    dict(n_kv=2, group=8, hd=64, k_type="f16", v_type="f16", n_live=[2500, 37], capacity=[2560, 40],
         cur_pos=[2500, 37], budget_frac=0.3, window=8, sink=2),
    dict(n_kv=3, group=1, hd=64, k_type="q8_0", v_type="q8_0", n_live=[1200], capacity=[1280], cur_pos=[1200],
         budget_frac=0.4, window=32, sink=0),
    # segments near the shared-memory key limit (47104 rows) on either side:
    # keys in shared memory or through the workspace (with the cut bin's keys
    # gathered for the last radix pass and the chunk ballots kept for the keep
    # list); odd capacities put every segment's rows (and keys) off the
    # 16-byte boundary; G 1, 2 and 4 make raw-score rows of 4, 8 and 16 bytes
    dict(n_kv=2, group=1, hd=128, k_type="f16", v_type="f16", n_live=[47105, 33000], capacity=[47107, 33001],
         cur_pos=[50000, 33000], budget_frac=0.3, window=100, sink=3),
    dict(n_kv=3, group=2, hd=64, k_type="q8_0", v_type="f16", n_live=[60001], capacity=[60003], cur_pos=[60001],
         budget_frac=0.45, window=64, sink=1),
    dict(n_kv=1, group=4, hd=64, k_type="f16", v_type="f16", n_live=[100003, 47104], capacity=[100005, 47104],
         cur_pos=[100003, 47104], budget_frac=0.25, window=1024, sink=4),
    # k = 0: the budget is exactly sink + window (only protected rows survive)
    dict(n_kv=2, group=4, hd=128, k_type="f16", v_type="f16", n_live=[900], capacity=[1024], cur_pos=[900],
         budget_rows=[132], window=128, sink=4),
]


@pytest.mark.parametrize("cfg", FUSED_CASES)
def test_fused_evict_matches_oracle_with_scores(lib, cfg):
    cases, hosts, qm, qa = _layers(cfg, 1)
    case, host = cases[0], hosts[0]
    dev = U.to_device(host)
    cache, pol = U.lib_cache(lib, case, dev), U.lib_policy(lib, case)
    ws = torch.empty(lib.model_workspace_size(cache, 1, case.group), dtype=torch.uint8, device="cuda")
    lib.workspace_init(ws)
    st = lib.Stats(qm, qa, n_kv_heads=case.n_kv, head_dim=case.hd, rope_theta=case.theta)
    scores = torch.full((case.total_rows(),), float("nan"), device="cuda")
    lib.evict_model(st, [0], [cache], pol, ws=ws, score_out=scores)
    assert lib.device_status(ws) == lib.OK
    got = {k: (None if v is None else v.cpu().numpy()) for k, v in dev.items()}
    _check_layer(case, host, got, qm, qa, 0, scores=scores.cpu().numpy(), what="fused")
    st.close()


def test_model_pass_several_layers(lib):
    """Four layers of ragged sequences in one call, each layer with its own
    live counts (one layer entirely at or below budget, one with a sequence
    below budget), scores out; then a second call on the same workspace after
    new rows."""
    cfg = dict(n_kv=2, group=4, hd=128, k_type="f16", v_type="f16", n_live=[2600, 1900], capacity=[2688, 2048],
               cur_pos=[30000, 1900], budget_frac=0.5, n_ctx=[2600, 1900], window=64, sink=4)
    L = 4
    cases, hosts, qm, qa = _layers(cfg, L)
    # per-layer live counts
    cases[1].n_live = [1300, 950]                   # both sequences at budget: no-op layer
    hosts[1]["n_live"] = np.asarray(cases[1].n_live, np.int32)
    cases[2].n_live = [2600, 900]                   # second sequence below budget
    hosts[2]["n_live"] = np.asarray(cases[2].n_live, np.int32)
    devs = [U.to_device(h) for h in hosts]
    caches = [U.lib_cache(lib, c, d) for c, d in zip(cases, devs)]
    pol = U.lib_policy(lib, cases[0])
    ws = torch.empty(lib.model_workspace_size(caches[0], L, 4), dtype=torch.uint8, device="cuda")
    lib.workspace_init(ws)
    st = lib.Stats(qm, qa, n_kv_heads=2, head_dim=128, rope_theta=cfg.get("theta", 1e4))
    rows = cases[0].total_rows()
    scores = torch.full((L, rows), float("nan"), device="cuda")
    lib.evict_model(st, list(range(L)), caches, pol, ws=ws, score_out=scores)
    assert lib.device_status(ws) == lib.OK
    sc = scores.cpu().numpy()
    for l in range(L):
        got = {k: (None if v is None else v.cpu().numpy()) for k, v in devs[l].items()}
        _check_layer(cases[l], hosts[l], got, qm, qa, l, scores=sc[l], what=f"layer {l}")
    # the same workspace again: a single-layer fused call and a staged call on
    # layer 0 after its rows were restored
    for name in ("k", "v", "pos", "n_live"):
        devs[0][name].copy_(torch.from_numpy(hosts[0][name]))
    lib.evict(st, 0, caches[0], pol, ws=ws)
    assert lib.device_status(ws) == lib.OK
    got = {k: (None if v is None else v.cpu().numpy()) for k, v in devs[0].items()}
    _check_layer(cases[0], hosts[0], got, qm, qa, 0, what="fused after model")
    for name in ("k", "v", "pos", "n_live"):
        devs[0][name].copy_(torch.from_numpy(hosts[0][name]))
    lib.evict_staged(st, 0, caches[0], pol, ws=ws)
    assert lib.device_status(ws) == lib.OK
    got = {k: (None if v is None else v.cpu().numpy()) for k, v in devs[0].items()}
    _check_layer(cases[0], hosts[0], got, qm, qa, 0, what="staged after model")
    # and the model pass once more, on restored layers, in a different layer order
    for l in range(L):
        for name in ("k", "v", "pos", "n_live"):
            devs[l][name].copy_(torch.from_numpy(hosts[l][name]))
    order = [2, 0, 3, 1]
    lib.evict_model(st, order, [caches[l] for l in order], pol, ws=ws)
    assert lib.device_status(ws) == lib.OK
    for l in range(L):
        got = {k: (None if v is None else v.cpu().numpy()) for k, v in devs[l].items()}
        _check_layer(cases[l], hosts[l], got, qm, qa, l, what=f"second call, layer {l}")
    st.close()


def test_model_pass_q8_and_bad_n_live(lib):
    """q8_0 keys over three layers; layer 1's first sequence has n_live above
    its capacity: reported, that sequence skipped, everything else compacted."""
    cfg = dict(n_kv=2, group=2, hd=128, k_type="q8_0", v_type="f16", n_live=[3000, 2000], capacity=[3072, 2048],
               cur_pos=[65536, 4000], budget_frac=0.5, n_ctx=[3000, 2000], window=256, sink=4)
    cases, hosts, qm, qa = _layers(cfg, 3)
    devs = [U.to_device(h) for h in hosts]
    devs[1]["n_live"][0] = 5000
    caches = [U.lib_cache(lib, c, d) for c, d in zip(cases, devs)]
    pol = U.lib_policy(lib, cases[0])
    ws = torch.empty(lib.model_workspace_size(caches[0], 3, 2), dtype=torch.uint8, device="cuda")
    lib.workspace_init(ws)
    st = lib.Stats(qm, qa, n_kv_heads=2, head_dim=128, rope_theta=1e4)
    lib.evict_model(st, [0, 1, 2], caches, pol, ws=ws)
    assert lib.device_status(ws) == lib.ERR_DEVICE_ARG
    for l in (0, 2):
        got = {k: (None if v is None else v.cpu().numpy()) for k, v in devs[l].items()}
        _check_layer(cases[l], hosts[l], got, qm, qa, l, what=f"layer {l}")
    got = {k: (None if v is None else v.cpu().numpy()) for k, v in devs[1].items()}
    assert got["n_live"].tolist() == [5000, cases[1].budgets()[1]]
    r0 = int(hosts[1]["seq_row0"][0])
    assert got["k"][r0:r0 + 2 * 3072].tobytes() == hosts[1]["k"][r0:r0 + 2 * 3072].tobytes()
    assert lib.device_status(ws) == lib.OK     # cleared by the read; the workspace stays usable
    st.close()


def test_model_dispatch_query_follows_the_documented_rule(lib):
    """tria_evict_model_fused: the fused kernel from 128 segments whatever
    their length, or from 32 with no capacity above 65536 rows; the staged
    kernels below that (the query reads host metadata only: the cache
    addresses are fake and never touched)."""
    w = W.get_workload("qwen3_8b_full")
    qm, qa = W.make_stats(w)
    st = lib.Stats(qm, qa, n_kv_heads=w.n_kv_heads, head_dim=w.head_dim, rope_theta=w.rope_theta)

    def caches(n, cap):
        return [lib.LayerCache(k=0x1000000 * (l + 1), v=0x1000000 * (l + 1) + 0x800000, pos=0x10000 * (l + 1),
                               n_live=0x100 * (l + 1), seq_row0=[0], capacity=[cap], head_dim=w.head_dim,
                               n_kv_heads=w.n_kv_heads) for l in range(n)]

    # 8 segments per layer
    for n_layers, cap, fused in [(36, 12288, True), (4, 12288, True), (3, 12288, False), (1, 32768, False),
                                 (4, 100000, False), (15, 100000, False), (16, 100000, True)]:
        got = lib.evict_model_fused(st, list(range(n_layers)), caches(n_layers, cap))
        assert got is fused, (n_layers, cap)
    one = caches(1, 12288)
    with pytest.raises(lib.TriaError):   # the same cache twice: the model call rejects it
        lib.evict_model_fused(st, [0, 1], one + one)
    st.close()


def test_whole_model_qwen3_steady_state(lib):
    """All 36 layers of the Qwen3-8B steady state (6272 live rows -> 6144 per
    segment) in one tria_evict_model call, in the launch configuration the
    benchmark times; the oracle checks sampled layers and segments, with their
    z-max scores row by row."""
    from synth import device as D
    D.build()
    w = W.get_workload("qwen3_8b_full")
    qm, qa = W.make_stats(w)
    st = lib.Stats(qm, qa, n_kv_heads=w.n_kv_heads, head_dim=w.head_dim, rope_theta=w.rope_theta)
    ts = [D.alloc_layer(w) for _ in range(w.n_layers)]
    for l, t in enumerate(ts):
        D.fill_layer(w, l, t)
    caches = [U.workload_cache(lib, w, t) for t in ts]
    pol = U.workload_policy(lib, w)
    ws = torch.empty(lib.model_workspace_size(caches[0], w.n_layers, w.group), dtype=torch.uint8, device="cuda")
    lib.workspace_init(ws)
    rows = w.total_rows()
    scores = torch.full((w.n_layers, rows), float("nan"), device="cuda")
    lib.evict_model(st, list(range(w.n_layers)), caches, pol, ws=ws, score_out=scores)
    assert lib.device_status(ws) == lib.OK
    budgets = [int(np.floor(w.budget_frac * c)) for c in w.n_ctx]
    r0s = w.seq_row0()
    for layer, (s, g) in [(0, (0, 0)), (17, (0, 5)), (35, (0, 7))]:
        assert ts[layer]["n_live"].cpu().tolist() == [min(n, b) for n, b in zip(w.n_live, budgets)]
        seg = W.segment_host(w, layer, s, g, rows=w.n_live[s])
        kf = O.keys_f64(seg["k"], seg["k_scale"])
        hs = O.heads_of_kv(w.n_q_heads, w.n_kv_heads)[g]
        _, sc = O.segment_scores(kf, O.as_complex(qm[layer][hs]), O.mlr_weight(qm[layer][hs], qa[layer][hs]),
                                 O.rope_omega(w.head_dim, w.rope_theta), w.cur_pos[s], O.default_future_offsets())
        n, b, cap = w.n_live[s], budgets[s], w.capacity[s]
        r0 = int(r0s[s] + g * cap)
        got_s = scores[layer, r0:r0 + n].cpu().numpy()
        err = np.abs(got_s - sc) / np.maximum(np.abs(sc), 1.0)
        assert err.max() <= U.RTOL, f"L{layer}: z-max rel err {err.max():.3e}"
        want = O.select_keep(sc, n, b, w.sink, w.window)
        gk = np.searchsorted(seg["pos"][:n], ts[layer]["pos"][r0:r0 + b].cpu().numpy())
        U.assert_keep_sets_match(gk, want, sc, n, b, w.sink, w.window, f"L{layer} s{s} g{g}")
        np.testing.assert_array_equal(ts[layer]["k"][r0:r0 + b].cpu().numpy(), seg["k"][gk])
        np.testing.assert_array_equal(ts[layer]["v"][r0:r0 + b].cpu().numpy(), seg["v"][gk])
    st.close()
    del ts
    torch.cuda.empty_cache()


def test_model_pass_host_checks(lib):
    """Rejected on the host: a layer twice, caches of different shapes, no layers."""
    cfg = dict(n_kv=2, group=4, hd=128, k_type="f16", v_type="f16", n_live=[300], capacity=[320], cur_pos=[300],
               budget_frac=0.5, window=16, sink=2)
    cases, hosts, qm, qa = _layers(cfg, 2)
    devs = [U.to_device(h) for h in hosts]
    caches = [U.lib_cache(lib, c, d) for c, d in zip(cases, devs)]
    pol = U.lib_policy(lib, cases[0])
    ws = torch.empty(lib.model_workspace_size(caches[0], 2, 4), dtype=torch.uint8, device="cuda")
    lib.workspace_init(ws)
    st = lib.Stats(qm, qa, n_kv_heads=2, head_dim=128, rope_theta=1e4)
    with pytest.raises(lib.TriaError) as e:
        lib.evict_model(st, [0, 1], [caches[0], caches[0]], pol, ws=ws)
    assert e.value.status == lib.ERR_INVALID_ARG
    other = U.Case(**dict(cfg, capacity=[400]))
    oh = U.build_host(other)
    oc = U.lib_cache(lib, other, U.to_device(oh))
    with pytest.raises(lib.TriaError) as e:
        lib.evict_model(st, [0, 1], [caches[0], oc], pol, ws=ws)
    assert e.value.status == lib.ERR_INVALID_ARG
    small = torch.empty(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(lib.TriaError) as e:
        lib.evict_model(st, [0, 1], caches, pol, ws=small)
    assert e.value.status == lib.ERR_WORKSPACE
    st.close()
