"""GPU parity of the eviction pass against the CPU oracle, through the C ABI.

Bars: scores within relative 1e-3 (raw: tau = the head's RMS; z-max: tau = 1);
select and compact bit-exact when both sides take the same score array / keep
list; end-to-end keep-sets identical except rows whose oracle score is within
the tolerance of the cut, and the compacted planes exact gathers of the input.
"""
import numpy as np
import pytest

from oracle import tria_oracle as O
from synth import workloads as W

import _util as U

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _oracle_segment(case, host, s, g, p=None):
    r0 = int(host["seq_row0"][s] + g * case.capacity[s])
    n = case.n_live[s]
    kf = O.keys_f64(host["k"][r0:r0 + n], None if host["k_scale"] is None else host["k_scale"][r0:r0 + n])
    hs = O.heads_of_kv(case.n_kv * case.group, case.n_kv)[g]
    qc = O.as_complex(host["q_mean"][0][hs])
    mw = O.mlr_weight(host["q_mean"][0][hs], host["q_abs"][0][hs])
    offs = O.default_future_offsets() if case.offsets is None else case.offsets
    raw, s_ = O.segment_scores(kf, qc, mw, O.rope_omega(case.hd, case.theta),
                               case.cur_pos[s] if p is None else p, offs)
    return r0, n, raw, s_


def _stats(lib, case, host):
    return lib.Stats(host["q_mean"], host["q_abs"], n_kv_heads=case.n_kv, head_dim=case.hd,
                     rope_theta=case.theta, offsets=case.offsets)


SCORE_CASES = [
    dict(n_kv=2, group=4, hd=64, k_type="f32", v_type="f32", n_live=[300], capacity=[320], cur_pos=[4000]),
    dict(n_kv=2, group=4, hd=128, k_type="f16", v_type="f16", n_live=[1000, 777], capacity=[1024, 800],
         cur_pos=[131072, 9]),
    dict(n_kv=1, group=8, hd=256, k_type="f16", v_type="f16", n_live=[513], capacity=[600], cur_pos=[70000]),
    dict(n_kv=4, group=1, hd=96, k_type="f32", v_type="f16", n_live=[257, 64, 0], capacity=[300, 64, 10],
         cur_pos=[5, 6, 7]),
    dict(n_kv=2, group=2, hd=128, k_type="q8_0", v_type="f16", n_live=[2000], capacity=[2048],
         cur_pos=[65536]),
    dict(n_kv=2, group=4, hd=32, k_type="q8_0", v_type="q8_0", n_live=[100], capacity=[128], cur_pos=[77]),
    dict(n_kv=2, group=8, hd=128, k_type="f16", v_type="f16", n_live=[700], capacity=[700], cur_pos=[1 << 20],
         offsets=[1, 2, 3, 1000, -5]),
    # fp16 shapes of the tensor-core body: one / two heads per group, head_dim
    # 64 / 192 / 256, ragged 16-row tiles; hd 96 takes the fp32 body
    dict(n_kv=3, group=1, hd=64, k_type="f16", v_type="f16", n_live=[37, 1, 16], capacity=[40, 8, 16],
         cur_pos=[100, 3, 1 << 30]),
    dict(n_kv=2, group=2, hd=192, k_type="f16", v_type="f32", n_live=[333], capacity=[350], cur_pos=[123457]),
    dict(n_kv=1, group=4, hd=256, k_type="f16", v_type="f16", n_live=[1000, 17], capacity=[1024, 32],
         cur_pos=[98765, 40]),
    dict(n_kv=2, group=2, hd=96, k_type="f16", v_type="f16", n_live=[150], capacity=[160], cur_pos=[50]),
    # q8_0 keys on the tensor-core body: block scales per 32 values, ragged tiles
    dict(n_kv=1, group=8, hd=64, k_type="q8_0", v_type="f16", n_live=[77, 300], capacity=[80, 320],
         cur_pos=[123, 99999]),
    dict(n_kv=2, group=1, hd=256, k_type="q8_0", v_type="q8_0", n_live=[333], capacity=[340], cur_pos=[7777]),
]


@pytest.mark.parametrize("cfg", SCORE_CASES)
def test_score_parity(lib, cfg):
    case = U.Case(**cfg)
    host = U.build_host(case)
    dev = U.to_device(host)
    cache, pol = U.lib_cache(lib, case, dev), U.lib_policy(lib, case)
    ws = U.new_workspace(lib, cache, case.group)
    st = _stats(lib, case, host)
    rows = case.total_rows()
    s_out = torch.full((rows,), float("nan"), device="cuda")
    raw_out = torch.full((rows, case.group), float("nan"), device="cuda")
    lib.score(st, 0, cache, pol, s_out, raw_out, ws=ws)
    assert lib.device_status(ws) == lib.OK
    s_gpu, raw_gpu = s_out.cpu().numpy(), raw_out.cpu().numpy()
    for s in range(case.n_seqs):
        for g in range(case.n_kv):
            r0, n, raw, sc = _oracle_segment(case, host, s, g)
            if n == 0:
                continue
            U.assert_scores_close(raw_gpu[r0:r0 + n], raw, s_gpu[r0:r0 + n], sc, f"seq {s} head {g}")
            cap = case.capacity[s]
            assert np.all(np.isnan(s_gpu[r0 + n:r0 + cap]))          # rows past n_live untouched


def _select_case(seed, n_live, cap, budget_rows, sink, window, n_kv=3):
    rng = np.random.default_rng(seed)
    case = U.Case(n_kv=n_kv, group=1, hd=64, k_type="f16", v_type="f16", n_live=n_live, capacity=cap,
                  cur_pos=[0] * len(n_live), budget_rows=budget_rows, sink=sink, window=window, seed=seed)
    rows = case.total_rows()
    levels = np.array([-2.0, -0.0, 0.0, 0.5, 0.5, 1.25, np.inf, -np.inf, np.nan], np.float32)
    score = np.where(rng.random(rows) < 0.5, rng.choice(levels, rows),
                     rng.standard_normal(rows)).astype(np.float32)
    return case, score


SELECT_CASES = [
    (1, [5000], [5000], [1250], 4, 512),
    (2, [4097, 130, 64, 0], [4100, 200, 64, 8], [2000, 100, 64, 20], 2, 16),   # ragged, no-op, empty
    (3, [3000], [3072], [520], 4, 512),                                        # one candidate kept
    (4, [3000], [3072], [516], 4, 512),                                        # k = 0
    (5, [777, 1000], [800, 1000], [700, 999], 0, 0),                           # no protection
    (6, [20000], [20000], [10000], 1, 3),
    # larger segments: ragged, no-op and near-budget cases
    (7, [17000, 9000, 40], [17408, 16384, 64], [4000, 9000, 80], 4, 64),
    (8, [40000], [40960], [10000], 4, 512),
    (9, [16384, 16000], [16384, 16384], [4096, 15999], 4, 512),
]


@pytest.mark.parametrize("seed,n_live,cap,budget,sink,window", SELECT_CASES)
def test_select_bit_exact_on_given_scores(lib, seed, n_live, cap, budget, sink, window):
    case, score = _select_case(seed, n_live, cap, budget, sink, window)
    host = U.build_host(case)
    dev = U.to_device(host)
    cache, pol = U.lib_cache(lib, case, dev), U.lib_policy(lib, case)
    ws = U.new_workspace(lib, cache, 0)
    keep_out = torch.full((case.total_rows(),), -7, dtype=torch.int32, device="cuda")
    lib.select(torch.from_numpy(score).cuda(), cache, pol, keep_out, ws=ws)
    assert lib.device_status(ws) == lib.OK
    keep_gpu = keep_out.cpu().numpy()
    r0s = case.seq_row0()
    for s in range(case.n_seqs):
        for g in range(case.n_kv):
            r0 = int(r0s[s] + g * case.capacity[s])
            n, b = case.n_live[s], budget[s]
            want = O.select_keep(score[r0:r0 + n], n, b, sink, window)
            got = keep_gpu[r0:r0 + len(want)]
            np.testing.assert_array_equal(got, want, err_msg=f"seq {s} head {g}")
            assert np.all(keep_gpu[r0 + len(want):r0 + case.capacity[s]] == -7)
    # a second call on the same workspace (self-resetting counters)
    lib.select(torch.from_numpy(score).cuda(), cache, pol, keep_out, ws=ws)
    np.testing.assert_array_equal(keep_out.cpu().numpy(), keep_gpu)


def _random_keep(rng, n, b, sink, window):
    if n <= b:
        return np.arange(n)
    cand = np.arange(sink, n - window)
    pick = np.sort(rng.choice(cand, b - sink - window, replace=False))
    return np.sort(np.concatenate([np.arange(sink), pick, np.arange(n - window, n)]))


COMPACT_CASES = [
    dict(n_kv=2, group=1, hd=128, k_type="f16", v_type="f16", n_live=[3000, 65, 0], capacity=[3072, 70, 4],
         cur_pos=[0, 0, 0], budget_rows=[1000, 64, 64], sink=4, window=60),
    dict(n_kv=1, group=1, hd=256, k_type="f16", v_type="f16", n_live=[9000], capacity=[9000], cur_pos=[0],
         budget_rows=[8999], sink=0, window=0),
    dict(n_kv=3, group=1, hd=64, k_type="q8_0", v_type="q8_0", n_live=[1500, 400], capacity=[1600, 512],
         cur_pos=[0, 0], budget_rows=[300, 399], sink=1, window=5),
    dict(n_kv=2, group=1, hd=32, k_type="f32", v_type="f32", n_live=[129], capacity=[200], cur_pos=[0],
         budget_rows=[2], sink=1, window=1),
    # more destination blocks than warps in the grid (fp32 rows: 7 warps per
    # CTA): several rounds, ordered by the per-block read flags; the cases
    # above take one round and a grid barrier
    dict(n_kv=4, group=1, hd=128, k_type="f32", v_type="f32", n_live=[40000], capacity=[40000], cur_pos=[0],
         budget_rows=[20000], sink=4, window=64),
    dict(n_kv=4, group=1, hd=128, k_type="f16", v_type="q8_0", n_live=[70000, 3000], capacity=[70016, 3008],
         cur_pos=[0, 0], budget_rows=[17500, 2999], sink=4, window=512),
]


@pytest.mark.parametrize("cfg", COMPACT_CASES)
def test_compact_bit_exact_on_given_keep_list(lib, cfg):
    case = U.Case(**cfg)
    host = U.build_host(case)
    dev = U.to_device(host)
    cache, pol = U.lib_cache(lib, case, dev), U.lib_policy(lib, case)
    ws = U.new_workspace(lib, cache, 0)
    rng = np.random.default_rng(3)
    keep_all = np.full(case.total_rows(), -1, np.int32)
    want = {k: (None if v is None else v.copy()) for k, v in host.items()
            if k in ("k", "k_scale", "v", "v_scale", "pos")}
    r0s = case.seq_row0()
    for s in range(case.n_seqs):
        for g in range(case.n_kv):
            r0 = int(r0s[s] + g * case.capacity[s])
            n, b = case.n_live[s], case.budget_rows[s]
            kp = _random_keep(rng, n, b, case.sink, case.window)
            keep_all[r0:r0 + len(kp)] = kp
            if n > b:
                for name, arr in want.items():
                    if arr is not None:
                        cap = case.capacity[s]
                        arr[r0:r0 + cap] = O.compact_rows(host[name][r0:r0 + cap], kp)
    lib.compact(cache, pol, torch.from_numpy(keep_all).cuda(), ws=ws)
    assert lib.device_status(ws) == lib.OK
    for name, arr in want.items():
        if arr is not None:
            got = dev[name].cpu().numpy()
            assert got.tobytes() == arr.tobytes(), name
    want_n = [min(n, b) for n, b in zip(case.n_live, case.budget_rows)]
    assert dev["n_live"].cpu().tolist() == want_n


def test_compact_rejects_bad_keep_list_and_moves_nothing(lib):
    case = U.Case(n_kv=1, group=1, hd=64, k_type="f16", v_type="f16", n_live=[500], capacity=[500],
                  cur_pos=[0], budget_rows=[100], sink=0, window=0)
    host = U.build_host(case)
    dev = U.to_device(host)
    cache, pol = U.lib_cache(lib, case, dev), U.lib_policy(lib, case)
    ws = U.new_workspace(lib, cache, 0)
    keep = np.arange(100, dtype=np.int32) * 3
    keep[50] = keep[49]                                   # not strictly ascending
    full = np.zeros(500, np.int32)
    full[:100] = keep
    lib.compact(cache, pol, torch.from_numpy(full).cuda(), ws=ws)
    assert lib.device_status(ws) == lib.ERR_KEEP_LIST
    assert dev["k"].cpu().numpy().tobytes() == host["k"].tobytes()
    assert dev["n_live"].cpu().tolist() == [500]
    # the workspace stays usable: a valid list now compacts
    full[:100] = np.arange(100) * 3
    lib.compact(cache, pol, torch.from_numpy(full).cuda(), ws=ws)
    assert lib.device_status(ws) == lib.OK
    np.testing.assert_array_equal(dev["pos"].cpu().numpy()[:100], host["pos"][np.arange(100) * 3])


EVICT_CASES = [
    dict(n_kv=2, group=4, hd=64, k_type="f32", v_type="f32", n_live=[512], capacity=[512], cur_pos=[512],
         budget_frac=0.5, window=64, sink=4),
    dict(n_kv=2, group=4, hd=128, k_type="f16", v_type="f16", n_live=[3000, 1500, 100], capacity=[3072, 1600, 128],
         cur_pos=[100000, 1500, 3], budget_frac=0.25, n_ctx=[3000, 1500, 1000], window=128, sink=4),
    dict(n_kv=1, group=8, hd=256, k_type="f16", v_type="f16", n_live=[4100], capacity=[4100], cur_pos=[9000],
         budget_frac=0.5, window=1024, sink=4),
    dict(n_kv=2, group=2, hd=128, k_type="q8_0", v_type="f16", n_live=[5000], capacity=[5000], cur_pos=[65536],
         budget_frac=0.5, window=512, sink=4),
    dict(n_kv=2, group=1, hd=96, k_type="f16", v_type="q8_0", n_live=[999], capacity=[1000], cur_pos=[12],
         budget_rows=[500], window=0, sink=0),
    # the most segments one call takes: 128 sequences x 8 KV heads, ragged short rows
    dict(n_kv=8, group=4, hd=64, k_type="f16", v_type="f16", n_live=[40 + (i * 37) % 200 for i in range(128)],
         capacity=[256] * 128, cur_pos=[300 + 7 * i for i in range(128)], budget_frac=0.5, window=8, sink=2),
]


@pytest.mark.parametrize("cfg", EVICT_CASES)
def test_evict_end_to_end(lib, cfg):
    case = U.Case(**cfg)
    host = U.build_host(case)
    dev = U.to_device(host)
    cache, pol = U.lib_cache(lib, case, dev), U.lib_policy(lib, case)
    ws = U.new_workspace(lib, cache, case.group)
    st = _stats(lib, case, host)
    lib.evict(st, 0, cache, pol, ws=ws)
    assert lib.device_status(ws) == lib.OK
    got = {k: (None if v is None else v.cpu().numpy()) for k, v in dev.items()}
    budgets = case.budgets()
    for s in range(case.n_seqs):
        n, b = case.n_live[s], budgets[s]
        assert got["n_live"][s] == min(n, b)
        for g in range(case.n_kv):
            r0, n_, raw, sc = _oracle_segment(case, host, s, g)
            cap = case.capacity[s]
            if n <= b:
                for name in ("k", "v", "pos"):
                    assert got[name][r0:r0 + cap].tobytes() == host[name][r0:r0 + cap].tobytes()
                continue
            want = O.select_keep(sc, n, b, case.sink, case.window)
            gk = np.searchsorted(host["pos"][r0:r0 + n], got["pos"][r0:r0 + b])
            U.assert_keep_sets_match(gk, want, sc, n, b, case.sink, case.window, f"seq {s} head {g}")
            for name in ("k", "k_scale", "v", "v_scale"):
                if host[name] is None:
                    continue
                np.testing.assert_array_equal(got[name][r0:r0 + b], host[name][r0 + gk])
                assert got[name][r0 + b:r0 + cap].tobytes() == host[name][r0 + b:r0 + cap].tobytes()


def test_evict_two_passes_use_absolute_position(lib):
    """Pass 2 runs at decode position 640 on 256 + 128 rows; the phases must come
    from the absolute position, not the row count."""
    case = U.Case(n_kv=2, group=4, hd=64, k_type="f32", v_type="f32", n_live=[512], capacity=[512],
                  cur_pos=[512], budget_frac=0.5, window=64, sink=4)
    host = U.build_host(case)
    dev = U.to_device(host)
    cache, pol = U.lib_cache(lib, case, dev), U.lib_policy(lib, case)
    ws = U.new_workspace(lib, cache, case.group)
    st = _stats(lib, case, host)
    lib.evict(st, 0, cache, pol, ws=ws)
    ora1, _ = O.evict_layer(host, host["q_mean"], host["q_abs"], layer=0, n_kv_heads=2, head_dim=64,
                            rope_theta=case.theta, cur_pos=[512], n_ctx=[512], budget_frac=0.5,
                            window=64, sink=4)
    for name in ("k", "v", "pos"):
        assert dev[name].cpu().numpy().tobytes() == ora1[name].tobytes(), name
    # decode 128 more tokens: rows 256..383 of each segment get fresh rows
    rng = np.random.default_rng(99)
    for g in range(2):
        a = g * 512 + 256
        ora1["k"][a:a + 128] = rng.standard_normal((128, 64)).astype(np.float32)
        ora1["v"][a:a + 128] = rng.standard_normal((128, 64)).astype(np.float32)
        ora1["pos"][a:a + 128] = np.arange(512, 640)
    ora1["n_live"][:] = 384
    for name in ("k", "v", "pos", "n_live"):
        dev[name].copy_(torch.from_numpy(ora1[name]))
    pol2 = lib.Policy(budget_frac=0.5, n_ctx=[512], window=64, sink=4, cur_pos=[640])
    lib.evict(st, 0, cache, pol2, ws=ws)
    assert lib.device_status(ws) == lib.OK
    ora2, info = O.evict_layer(ora1, host["q_mean"], host["q_abs"], layer=0, n_kv_heads=2, head_dim=64,
                               rope_theta=case.theta, cur_pos=[640], n_ctx=[512], budget_frac=0.5,
                               window=64, sink=4)
    for name in ("k", "v", "pos", "n_live"):
        assert dev[name].cpu().numpy().tobytes() == ora2[name].tobytes(), name
    # the same pass at the row-count position would have kept a different set
    _, wrong = O.evict_layer(ora1, host["q_mean"], host["q_abs"], layer=0, n_kv_heads=2, head_dim=64,
                             rope_theta=case.theta, cur_pos=[384], n_ctx=[512], budget_frac=0.5,
                             window=64, sink=4)
    assert any(not np.array_equal(info[k]["keep"], wrong[k]["keep"]) for k in info)


def test_n_live_out_of_range_is_reported_and_skipped(lib):
    case = U.Case(n_kv=1, group=4, hd=64, k_type="f16", v_type="f16", n_live=[300, 200], capacity=[256, 256],
                  cur_pos=[300, 200], budget_frac=0.5, window=8, sink=0)
    host = U.build_host(case)
    dev = U.to_device(host)
    cache, pol = U.lib_cache(lib, case, dev), U.lib_policy(lib, case)
    ws = U.new_workspace(lib, cache, case.group)
    st = _stats(lib, case, host)
    lib.evict(st, 0, cache, pol, ws=ws)
    assert lib.device_status(ws) == lib.ERR_DEVICE_ARG
    got_k = dev["k"].cpu().numpy()
    assert got_k[:256].tobytes() == host["k"][:256].tobytes()          # sequence 0 untouched
    assert dev["n_live"].cpu().tolist() == [300, 100]                  # sequence 1 compacted
    assert lib.device_status(ws) == lib.OK                             # status cleared by the read


def test_bounded_wait_gives_up_and_reports(lib):
    ws = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    assert lib.selftest_bounded_wait(1000, ws) == lib.ERR_TIMEOUT
    assert lib.device_status(ws) == lib.OK


def test_noop_when_at_or_below_budget_is_byte_identical(lib):
    case = U.Case(n_kv=2, group=4, hd=128, k_type="f16", v_type="f16", n_live=[1000, 999], capacity=[1024, 1024],
                  cur_pos=[1000, 999], budget_rows=[1000, 1000], window=16, sink=2)
    host = U.build_host(case)
    dev = U.to_device(host)
    cache, pol = U.lib_cache(lib, case, dev), U.lib_policy(lib, case)
    ws = U.new_workspace(lib, cache, case.group)
    st = _stats(lib, case, host)
    lib.evict(st, 0, cache, pol, ws=ws)
    assert lib.device_status(ws) == lib.OK
    for name in ("k", "v", "pos", "n_live"):
        assert dev[name].cpu().numpy().tobytes() == host[name].tobytes()


# --------------------------------------------------------------- full-size workloads

def _oracle_workload_segment(w, layer, s, g, qm, qa):
    seg = W.segment_host(w, layer, s, g, rows=w.n_live[s])
    kf = O.keys_f64(seg["k"], seg["k_scale"])
    hs = O.heads_of_kv(w.n_q_heads, w.n_kv_heads)[g]
    raw, sc = O.segment_scores(kf, O.as_complex(qm[layer][hs]), O.mlr_weight(qm[layer][hs], qa[layer][hs]),
                               O.rope_omega(w.head_dim, w.rope_theta), w.cur_pos[s], O.default_future_offsets())
    return seg, raw, sc


@pytest.mark.parametrize("name,layers,segs", [
    ("tiny", [0], None),
    ("qwen3_8b_layer", [0], None),
    ("qwen3_8b_full", [0, 35], [(0, 0), (0, 5)]),
    ("q8_0", [0, 35], [(0, 1), (0, 7)]),
    ("batched_long", [0, 47], [(2, 0), (1, 3), (5, 2)]),
])
def test_workload_parity_sampled(lib, name, layers, segs):
    """Each workload at full per-layer size, in the launch configuration the
    benchmark times; the oracle checks the listed segments (all when None)."""
    from synth import device as D
    D.build()
    w = W.get_workload(name)
    qm, qa = W.make_stats(w)
    st = lib.Stats(qm, qa, n_kv_heads=w.n_kv_heads, head_dim=w.head_dim, rope_theta=w.rope_theta)
    t = D.alloc_layer(w)
    cache = U.workload_cache(lib, w, t)
    pol = U.workload_policy(lib, w)
    ws = U.new_workspace(lib, cache, w.group)
    budgets = [int(np.floor(w.budget_frac * c)) for c in w.n_ctx]
    for layer in layers:
        D.fill_layer(w, layer, t)
        lib.evict(st, layer, cache, pol, ws=ws)
        assert lib.device_status(ws) == lib.OK
        assert t["n_live"].cpu().tolist() == [min(n, b) for n, b in zip(w.n_live, budgets)]
        chosen = segs if segs is not None else [(s, g) for s, g, *_ in w.segments()]
        r0s = w.seq_row0()
        for s, g in chosen:
            seg, raw, sc = _oracle_workload_segment(w, layer, s, g, qm, qa)
            n, b, cap = w.n_live[s], budgets[s], w.capacity[s]
            r0 = int(r0s[s] + g * cap)
            want = O.select_keep(sc, n, b, w.sink, w.window)
            pos_after = t["pos"][r0:r0 + b].cpu().numpy()
            gk = np.searchsorted(seg["pos"][:n], pos_after)
            U.assert_keep_sets_match(gk, want, sc, n, b, w.sink, w.window, f"{name} L{layer} s{s} g{g}")
            got_k = t["k"][r0:r0 + b].cpu().numpy()
            np.testing.assert_array_equal(got_k, seg["k"][gk])
            got_v = t["v"][r0:r0 + b].cpu().numpy()
            np.testing.assert_array_equal(got_v, seg["v"][gk])
            if seg["k_scale"] is not None:
                np.testing.assert_array_equal(t["k_scale"][r0:r0 + b].cpu().numpy(), seg["k_scale"][gk])
    st.close()


def test_device_generator_matches_host_twin(lib):
    from synth import device as D
    D.build()
    for name in ("qwen3_8b_layer", "q8_0", "batched_long"):
        w = W.get_workload(name)
        t = D.alloc_layer(w)
        D.fill_layer(w, 3 if w.n_layers > 3 else 0, t)
        s, g, r0, cap, n = list(w.segments())[-1]
        seg = W.segment_host(w, 3 if w.n_layers > 3 else 0, s, g, rows=min(cap, 700))
        rows = len(seg["pos"])
        assert t["k"][r0:r0 + rows].cpu().numpy().tobytes() == seg["k"].tobytes(), name
        assert t["v"][r0:r0 + rows].cpu().numpy().tobytes() == seg["v"].tobytes(), name
        if seg["k_scale"] is not None:
            assert t["k_scale"][r0:r0 + rows].cpu().numpy().tobytes() == seg["k_scale"].tobytes()
        del t
        torch.cuda.empty_cache()
