"""Hybrid models ([Doc] §6 "Hybrid head_dim models": head_dim varies across
layers; the follow-on it names is a per-layer stats offset table so that the
eligible layers score on the GPU). One statistics handle holds layers of
head_dim 128, 256, 64, 512 and 96 with their own RoPE bases; passes on every
loaded layer match the oracle run with that layer's statistics, and the
hd = 512 layer is refused."""
import numpy as np
import pytest

from oracle import tria_oracle as O

import _util as U

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

HD = [128, 256, 64, 512, 96]
THETA = [1e6, 1e4, 1e4, 1e6, 5e5]
N_KV, G = 2, 4


def _stats_arrays(seed=7):
    rng = np.random.default_rng(seed)
    qm = [rng.standard_normal((N_KV * G, hd // 2, 2)).astype(np.float32) for hd in HD]
    qa = [(np.hypot(q[..., 0], q[..., 1]) + 0.5 * np.abs(rng.standard_normal(q.shape[:2]))).astype(np.float32)
          for q in qm]
    return qm, qa


@pytest.fixture(scope="module")
def hybrid(lib):
    qm, qa = _stats_arrays()
    return lib.Stats(qm, qa, n_kv_heads=N_KV, layer_head_dim=HD, layer_rope_theta=THETA), qm, qa


def _case(layer, k_type):
    return U.Case(n_kv=N_KV, group=G, hd=HD[layer], k_type=k_type, v_type="f16", n_live=[300, 77],
                  capacity=[320, 80], cur_pos=[5000, 123457], theta=THETA[layer], budget_frac=0.5, window=8, sink=2)


@pytest.mark.parametrize("layer,k_type", [(0, "f16"), (1, "f16"), (2, "f16"), (4, "f32"), (2, "q8_0"), (1, "q8_0")])
def test_hybrid_layer_scores_match_oracle(lib, hybrid, layer, k_type):
    st, qm, qa = hybrid
    case = _case(layer, k_type)
    host = U.build_host(case)
    dev = U.to_device(host)
    cache, pol = U.lib_cache(lib, case, dev), U.lib_policy(lib, case)
    ws = U.new_workspace(lib, cache, G)
    rows = case.total_rows()
    s_out = torch.full((rows,), float("nan"), device="cuda")
    raw_out = torch.full((rows, G), float("nan"), device="cuda")
    lib.score(st, layer, cache, pol, s_out, raw_out, ws=ws)
    assert lib.device_status(ws) == lib.OK
    s_gpu, raw_gpu = s_out.cpu().numpy(), raw_out.cpu().numpy()
    heads = O.heads_of_kv(N_KV * G, N_KV)
    for s in range(case.n_seqs):
        for g in range(N_KV):
            r0 = int(host["seq_row0"][s] + g * case.capacity[s])
            n = case.n_live[s]
            kf = O.keys_f64(host["k"][r0:r0 + n], None if host["k_scale"] is None else host["k_scale"][r0:r0 + n])
            hs = heads[g]
            raw, sc = O.segment_scores(kf, O.as_complex(qm[layer][hs]), O.mlr_weight(qm[layer][hs], qa[layer][hs]),
                                       O.rope_omega(HD[layer], THETA[layer]), case.cur_pos[s],
                                       O.default_future_offsets())
            U.assert_scores_close(raw_gpu[r0:r0 + n], raw, s_gpu[r0:r0 + n], sc, f"layer {layer} seq {s} head {g}")


@pytest.mark.parametrize("layer", [1, 4])
def test_hybrid_layer_evict_matches_oracle(lib, hybrid, layer):
    st, qm, qa = hybrid
    case = _case(layer, "f16" if layer != 4 else "f32")
    host = U.build_host(case)
    dev = U.to_device(host)
    cache, pol = U.lib_cache(lib, case, dev), U.lib_policy(lib, case)
    ws = U.new_workspace(lib, cache, G)
    lib.evict(st, layer, cache, pol, ws=ws)
    assert lib.device_status(ws) == lib.OK
    _, info = O.evict_layer(host, qm, qa, layer=layer, n_kv_heads=N_KV, head_dim=HD[layer],
                            rope_theta=THETA[layer], cur_pos=case.cur_pos, n_ctx=case.n_live,
                            budget_frac=case.budget_frac, window=case.window, sink=case.sink)
    got = {k: (None if v is None else v.cpu().numpy()) for k, v in dev.items()}
    for (s, g), it in info.items():
        r0, n, b = it["row0"], it["n"], it["B"]
        gk = np.searchsorted(host["pos"][r0:r0 + n], got["pos"][r0:r0 + b])
        U.assert_keep_sets_match(gk, it["keep"], it["s"], n, b, case.sink, case.window, f"seq {s} head {g}")
        np.testing.assert_array_equal(got["k"][r0:r0 + b], host["k"][r0 + gk])
        np.testing.assert_array_equal(got["v"][r0:r0 + b], host["v"][r0 + gk])


def test_hybrid_refuses_the_unloaded_layer_and_mismatched_caches(lib, hybrid):
    st, _, _ = hybrid
    case = _case(0, "f16")
    host = U.build_host(case)
    dev = U.to_device(host)
    cache, pol = U.lib_cache(lib, case, dev), U.lib_policy(lib, case)
    ws = U.new_workspace(lib, cache, G)
    for layer, want in ((1, lib.ERR_INVALID_ARG), (2, lib.ERR_INVALID_ARG), (5, lib.ERR_INVALID_ARG)):
        with pytest.raises(lib.TriaError) as e:      # layer 0's head_dim 128 on another layer
            lib.evict(st, layer, cache, pol, ws=ws)
        assert e.value.status == want
    # the hd = 512 layer was not loaded: a cache of that head_dim fails the gate
    big = lib.LayerCache(k=dev["k"], v=dev["v"], pos=dev["pos"], n_live=dev["n_live"], seq_row0=[0, 4000],
                         capacity=[10, 10], head_dim=512, n_kv_heads=N_KV)
    with pytest.raises(lib.TriaError) as e:
        lib.evict(st, 3, big, pol, ws=ws)
    assert e.value.status == lib.ERR_UNSUPPORTED
    assert torch.equal(dev["k"].cpu(), torch.from_numpy(host["k"]))


def test_uniform_table_equals_uniform_stats(lib):
    rng = np.random.default_rng(3)
    qm = rng.standard_normal((3, N_KV * G, 64, 2)).astype(np.float32)
    qa = (np.hypot(qm[..., 0], qm[..., 1]) + 0.3).astype(np.float32)
    a = lib.Stats(qm, qa, n_kv_heads=N_KV, head_dim=128, rope_theta=1e6)
    b = lib.Stats(list(qm), list(qa), n_kv_heads=N_KV, layer_head_dim=[128] * 3, layer_rope_theta=[1e6] * 3)
    case = U.Case(n_kv=N_KV, group=G, hd=128, k_type="f16", v_type="f16", n_live=[500], capacity=[512],
                  cur_pos=[70000])
    host = U.build_host(case)
    dev = U.to_device(host)
    cache, pol = U.lib_cache(lib, case, dev), U.lib_policy(lib, case)
    ws = U.new_workspace(lib, cache, G)
    rows = case.total_rows()
    for layer in range(3):
        outs = []
        for st in (a, b):
            s_out = torch.zeros(rows, device="cuda")
            raw_out = torch.zeros((rows, G), device="cuda")
            lib.score(st, layer, cache, pol, s_out, raw_out, ws=ws)
            outs.append((s_out.cpu(), raw_out.cpu()))
        assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
