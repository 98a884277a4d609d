"""tria_evict_layers: sequences of several layers in one pass, each scored
with its own layer's statistics, against the oracle run per layer; with one
layer for every sequence it is tria_evict byte for byte."""
import numpy as np
import pytest

from oracle import tria_oracle as O

import _util as U

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

L, S = 3, 2


def _case(k_type):
    return U.Case(n_kv=2, group=4, hd=128, k_type=k_type, v_type="f16", n_live=[900, 400] * L,
                  capacity=[960, 416] * L, cur_pos=[5000, 400] * L, budget_frac=0.5, window=32, sink=2)


def _stats_arrays(seed=9, n_q=8, fc=64):
    rng = np.random.default_rng(seed)
    qm = rng.standard_normal((L, n_q, fc, 2)).astype(np.float32)
    qa = (np.hypot(qm[..., 0], qm[..., 1]) + 0.5 * np.abs(rng.standard_normal((L, n_q, fc)))).astype(np.float32)
    return qm, qa


@pytest.mark.parametrize("k_type", ["f16", "q8_0"])
def test_layers_in_one_pass_match_the_oracle(lib, k_type):
    case = _case(k_type)
    host = U.build_host(case)
    qm, qa = _stats_arrays()
    st = lib.Stats(qm, qa, n_kv_heads=2, head_dim=128, rope_theta=1e4)
    dev = U.to_device(host)
    cache, pol = U.lib_cache(lib, case, dev), U.lib_policy(lib, case)
    ws = U.new_workspace(lib, cache, 4)
    layer_of_seq = [l for l in range(L) for _ in range(S)]
    lib.evict_layers(st, layer_of_seq, cache, pol, ws=ws)
    assert lib.device_status(ws) == lib.OK
    got = {k: (None if v is None else v.cpu().numpy()) for k, v in dev.items()}
    for layer in range(L):
        segs = [(s, g) for s in range(len(layer_of_seq)) if layer_of_seq[s] == layer for g in range(2)]
        _, info = O.evict_layer(host, qm, qa, layer=layer, n_kv_heads=2, head_dim=128, rope_theta=1e4,
                                cur_pos=case.cur_pos, n_ctx=case.n_live, budget_frac=0.5, window=32, sink=2,
                                segments=segs)
        for (s, g), it in info.items():
            r0, n, b = it["row0"], it["n"], it["B"]
            assert got["n_live"][s] == min(n, b)
            gk = np.searchsorted(host["pos"][r0:r0 + n], got["pos"][r0:r0 + b])
            U.assert_keep_sets_match(gk, it["keep"], it["s"], n, b, 2, 32, f"layer {layer} seq {s} head {g}")
            for name in ("k", "k_scale", "v"):
                if host[name] is not None:
                    np.testing.assert_array_equal(got[name][r0:r0 + b], host[name][r0 + gk])


def test_one_layer_for_all_sequences_is_tria_evict(lib):
    case = _case("f16")
    host = U.build_host(case)
    qm, qa = _stats_arrays()
    st = lib.Stats(qm, qa, n_kv_heads=2, head_dim=128, rope_theta=1e4)
    outs = []
    for multi in (False, True):
        dev = U.to_device(host)
        cache, pol = U.lib_cache(lib, case, dev), U.lib_policy(lib, case)
        ws = U.new_workspace(lib, cache, 4)
        if multi:
            lib.evict_layers(st, [1] * case.n_seqs, cache, pol, ws=ws)
        else:
            lib.evict(st, 1, cache, pol, ws=ws)
        assert lib.device_status(ws) == lib.OK
        outs.append({k: dev[k].cpu().numpy().tobytes() for k in ("k", "v", "pos", "n_live")})
    assert outs[0] == outs[1]


def test_layers_with_different_phases_are_refused(lib):
    case = U.Case(n_kv=2, group=4, hd=128, k_type="f16", v_type="f16", n_live=[100, 100], capacity=[128, 128],
                  cur_pos=[100, 100], budget_frac=0.5, window=8, sink=0)
    host = U.build_host(case)
    qm, qa = _stats_arrays()
    st = lib.Stats(list(qm), list(qa), n_kv_heads=2, layer_head_dim=[128] * L, layer_rope_theta=[1e4, 1e6, 1e4])
    dev = U.to_device(host)
    cache, pol = U.lib_cache(lib, case, dev), U.lib_policy(lib, case)
    ws = U.new_workspace(lib, cache, 4)
    with pytest.raises(lib.TriaError) as e:
        lib.evict_layers(st, [0, 1], cache, pol, ws=ws)
    assert e.value.status == lib.ERR_UNSUPPORTED
    lib.evict_layers(st, [0, 2], cache, pol, ws=ws)      # equal bases: accepted
    assert lib.device_status(ws) == lib.OK
