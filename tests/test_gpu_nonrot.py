"""GPU parity of heads with non-rotary dims against the oracle, through the C ABI.

Reading ([Doc] §4 gate line field ``nonrot=``, §6 "Non-rotary models": such
models carry a content term besides the RoPE-direction term): the first
rot = head_dim - nonrot dims are NEOX-rotary with frequencies over rot dims,
the last nonrot never rotate, and each row's score gains the mean non-rotary
query dotted with the key's non-rotary dims.

Cases cover the tensor-core body with rotary pair steps fewer than the head's
(rot a multiple of 64: fp16 and q8_0, head_dim 128 and 256) and the fp32 /
generic body (rot/2 not a multiple of 32: f32 with a group of 8, fp16 with 24
rotary pairs, q8_0 at head_dim 96), ragged tiles, zero statistics for the
content term, and the whole pass (a call of 128 segments, which takes the
staged kernels since the fused kernel scores all-rotary heads only). Bars as
in the other parity tests: scores within relative 1e-3 (raw: tau = the head's
RMS; z-max: tau = 1); keep-sets identical except rows whose oracle score is
within the tolerance of the cut; compacted planes exact gathers.
"""
import numpy as np
import pytest

from oracle import tria_oracle as O

import _util as U

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _nonrot_stats(case, nonrot, seed, content=True):
    """q_mean / q_abs over the rot/2 rotary pairs and the mean non-rotary query."""
    rng = np.random.default_rng(seed)
    nq, fcr = case.n_kv * case.group, (case.hd - nonrot) // 2
    qm = rng.standard_normal((1, nq, fcr, 2)).astype(np.float32)
    qa = (np.hypot(qm[..., 0], qm[..., 1]).astype(np.float64)
          + 0.5 * np.abs(rng.standard_normal((1, nq, fcr)))).astype(np.float32)
    qn = (1.5 * rng.standard_normal((1, nq, nonrot))).astype(np.float32) if content else None
    return qm, qa, qn


def _oracle_segment(case, host, s, g, nonrot, qm, qa, qn):
    r0 = int(host["seq_row0"][s] + g * case.capacity[s])
    n = case.n_live[s]
    kf = O.keys_f64(host["k"][r0:r0 + n], None if host["k_scale"] is None else host["k_scale"][r0:r0 + n])
    hs = O.heads_of_kv(case.n_kv * case.group, case.n_kv)[g]
    raw, sc = O.segment_scores(kf, O.as_complex(qm[0][hs]), O.mlr_weight(qm[0][hs], qa[0][hs]),
                               O.rope_omega(case.hd, case.theta, nonrot), case.cur_pos[s],
                               O.default_future_offsets(), None if qn is None else qn[0][hs])
    return r0, n, raw, sc


CASES = [
    # tensor-core body: rot 64 of 128 (one of two rotary pair steps)
    (dict(n_kv=2, group=4, hd=128, k_type="f16", v_type="f16", n_live=[1000, 333], capacity=[1024, 340],
          cur_pos=[131072, 50]), 64),
    (dict(n_kv=2, group=2, hd=128, k_type="q8_0", v_type="f16", n_live=[700], capacity=[704],
          cur_pos=[65536]), 64),
    # rot 64 of 256 (one of four) and 128 of 256 (two of four)
    (dict(n_kv=1, group=4, hd=256, k_type="f16", v_type="f16", n_live=[513, 17], capacity=[520, 32],
          cur_pos=[98765, 40]), 192),
    (dict(n_kv=2, group=8, hd=64, k_type="q8_0", v_type="q8_0", n_live=[77], capacity=[80],
          cur_pos=[999]), 0),
    (dict(n_kv=1, group=2, hd=256, k_type="q8_0", v_type="f16", n_live=[333], capacity=[340],
          cur_pos=[7777]), 128),
    (dict(n_kv=3, group=1, hd=128, k_type="f16", v_type="f16", n_live=[37, 1, 16], capacity=[40, 8, 16],
          cur_pos=[100, 3, 1 << 30]), 64),
    # generic body: 48 rotary pairs with a group of 8 (four pairs a lane), 24
    # pairs on fp16 keys, q8_0 at head_dim 96
    (dict(n_kv=2, group=8, hd=128, k_type="f32", v_type="f32", n_live=[300], capacity=[320],
          cur_pos=[4000]), 32),
    (dict(n_kv=2, group=2, hd=64, k_type="f16", v_type="f16", n_live=[150, 9], capacity=[160, 16],
          cur_pos=[50, 1 << 20]), 16),
    (dict(n_kv=1, group=4, hd=96, k_type="q8_0", v_type="f16", n_live=[200], capacity=[200],
          cur_pos=[12345]), 32),
]


@pytest.mark.parametrize("cfg,nonrot", CASES)
def test_nonrot_score_parity(lib, cfg, nonrot):
    case = U.Case(**cfg)
    host = U.build_host(case)
    dev = U.to_device(host)
    cache, pol = U.lib_cache(lib, case, dev), U.lib_policy(lib, case)
    ws = U.new_workspace(lib, cache, case.group)
    qm, qa, qn = _nonrot_stats(case, nonrot, seed=case.hd + nonrot)
    st = lib.Stats(qm, qa, n_kv_heads=case.n_kv, head_dim=case.hd, rope_theta=case.theta,
                   nonrot_dim=nonrot, q_nonrot=qn)
    rows = case.total_rows()
    s_out = torch.full((rows,), float("nan"), device="cuda")
    raw_out = torch.full((rows, case.group), float("nan"), device="cuda")
    lib.score(st, 0, cache, pol, s_out, raw_out, ws=ws)
    assert lib.device_status(ws) == lib.OK
    s_gpu, raw_gpu = s_out.cpu().numpy(), raw_out.cpu().numpy()
    for s in range(case.n_seqs):
        for g in range(case.n_kv):
            r0, n, raw, sc = _oracle_segment(case, host, s, g, nonrot, qm, qa, qn)
            if n == 0:
                continue
            U.assert_scores_close(raw_gpu[r0:r0 + n], raw, s_gpu[r0:r0 + n], sc, f"seq {s} head {g}")
            assert np.all(np.isnan(s_gpu[r0 + n:r0 + case.capacity[s]]))
    st.close()


def test_nonrot_without_content_statistics(lib):
    """q_nonrot NULL: no content term, but the rotary pairs are still (f, f + rot/2)."""
    case = U.Case(n_kv=2, group=4, hd=128, k_type="f16", v_type="f16", n_live=[500], capacity=[512],
                  cur_pos=[3000])
    host = U.build_host(case)
    dev = U.to_device(host)
    cache, pol = U.lib_cache(lib, case, dev), U.lib_policy(lib, case)
    ws = U.new_workspace(lib, cache, case.group)
    qm, qa, _ = _nonrot_stats(case, 64, seed=5, content=False)
    st = lib.Stats(qm, qa, n_kv_heads=2, head_dim=128, rope_theta=case.theta, nonrot_dim=64)
    s_out = torch.full((case.total_rows(),), float("nan"), device="cuda")
    raw_out = torch.full((case.total_rows(), 4), float("nan"), device="cuda")
    lib.score(st, 0, cache, pol, s_out, raw_out, ws=ws)
    assert lib.device_status(ws) == lib.OK
    for g in range(2):
        r0, n, raw, sc = _oracle_segment(case, host, 0, g, 64, qm, qa, None)
        U.assert_scores_close(raw_out[r0:r0 + n].cpu().numpy(), raw, s_out[r0:r0 + n].cpu().numpy(), sc)
    st.close()


def test_nonrot_evict_end_to_end_over_128_segments(lib):
    """A call of 16 sequences x 8 KV heads: tria_evict keeps the staged kernels
    for heads with non-rotary dims; keep-sets and gathers against the oracle."""
    n_live = [200 + 13 * i for i in range(16)]
    case = U.Case(n_kv=8, group=4, hd=128, k_type="f16", v_type="f16", n_live=n_live,
                  capacity=[n + 8 for n in n_live], cur_pos=[5000 + 7 * i for i in range(16)],
                  budget_frac=0.5, window=16, sink=2)
    host = U.build_host(case)
    dev = U.to_device(host)
    cache, pol = U.lib_cache(lib, case, dev), U.lib_policy(lib, case)
    ws = U.new_workspace(lib, cache, case.group)
    qm, qa, qn = _nonrot_stats(case, 64, seed=9)
    st = lib.Stats(qm, qa, n_kv_heads=8, head_dim=128, rope_theta=case.theta, nonrot_dim=64, q_nonrot=qn)
    lib.evict(st, 0, cache, pol, ws=ws)
    assert lib.device_status(ws) == lib.OK
    got = {k: (None if v is None else v.cpu().numpy()) for k, v in dev.items()}
    budgets = case.budgets()
    for s in range(case.n_seqs):
        n, b = case.n_live[s], budgets[s]
        assert got["n_live"][s] == min(n, b)
        for g in range(case.n_kv):
            r0, _, _, sc = _oracle_segment(case, host, s, g, 64, qm, qa, qn)
            want = O.select_keep(sc, n, b, case.sink, case.window)
            gk = np.searchsorted(host["pos"][r0:r0 + n], got["pos"][r0:r0 + b])
            U.assert_keep_sets_match(gk, want, sc, n, b, case.sink, case.window, f"seq {s} head {g}")
            np.testing.assert_array_equal(got["k"][r0:r0 + b], host["k"][r0 + gk])
            np.testing.assert_array_equal(got["v"][r0:r0 + b], host["v"][r0 + gk])
    st.close()


def test_nonrot_model_pass_runs_staged_and_scores_out_is_unsupported(lib):
    """tria_evict_model on heads with non-rotary dims: one staged pass per
    layer (results as the oracle's); score_out needs the fused kernel."""
    L = 2
    cases = [U.Case(n_kv=2, group=2, hd=128, k_type="q8_0", v_type="f16", n_live=[600, 250],
                    capacity=[640, 256], cur_pos=[9000, 300], seed=30 + l) for l in range(L)]
    hosts = [U.build_host(c) for c in cases]
    devs = [U.to_device(h) for h in hosts]
    caches = [U.lib_cache(lib, c, d) for c, d in zip(cases, devs)]
    pol = U.lib_policy(lib, cases[0])
    rng = np.random.default_rng(77)
    qm = rng.standard_normal((L, 4, 32, 2)).astype(np.float32)
    qa = (np.hypot(qm[..., 0], qm[..., 1]) + 0.3).astype(np.float32)
    qn = rng.standard_normal((L, 4, 64)).astype(np.float32)
    st = lib.Stats(qm, qa, n_kv_heads=2, head_dim=128, rope_theta=1e4, nonrot_dim=64, q_nonrot=qn)
    ws = torch.empty(lib.model_workspace_size(caches[0], L, 2), dtype=torch.uint8, device="cuda")
    lib.workspace_init(ws)
    scores = torch.zeros((L, cases[0].total_rows()), device="cuda")
    with pytest.raises(lib.TriaError) as err:
        lib.evict_model(st, [0, 1], caches, pol, ws=ws, score_out=scores)
    assert err.value.status == lib.ERR_UNSUPPORTED
    lib.evict_model(st, [0, 1], caches, pol, ws=ws)
    assert lib.device_status(ws) == lib.OK
    for l in range(L):
        case, host = cases[l], hosts[l]
        got = {k: (None if v is None else v.cpu().numpy()) for k, v in devs[l].items()}
        for s in range(case.n_seqs):
            n, b = case.n_live[s], case.budgets()[s]
            for g in range(case.n_kv):
                r0, _, _, sc = _oracle_segment(case, host, s, g, 64, qm[l:l + 1], qa[l:l + 1], qn[l:l + 1])
                want = O.select_keep(sc, n, b, case.sink, case.window)
                gk = np.searchsorted(host["pos"][r0:r0 + n], got["pos"][r0:r0 + b])
                U.assert_keep_sets_match(gk, want, sc, n, b, case.sink, case.window, f"L{l} seq {s} head {g}")
                np.testing.assert_array_equal(got["k"][r0:r0 + b], host["k"][r0 + gk])
                np.testing.assert_array_equal(got["k_scale"][r0:r0 + b], host["k_scale"][r0 + gk])
    st.close()


def test_nonrot_stats_host_checks(lib):
    qm = np.zeros((1, 8, 32, 2), np.float32)
    for bad in (-2, 3, 128):
        with pytest.raises(lib.TriaError) as err:
            lib.Stats(qm, None, n_kv_heads=2, head_dim=128, rope_theta=1e4, nonrot_dim=bad)
        assert err.value.status == lib.ERR_INVALID_ARG, bad
    with pytest.raises(lib.TriaError) as err:   # 120 rotary dims: not a multiple of 16
        lib.Stats(np.zeros((1, 8, 60, 2), np.float32), None, n_kv_heads=2, head_dim=128, rope_theta=1e4,
                  nonrot_dim=8)
    assert err.value.status == lib.ERR_UNSUPPORTED
