"""Shared-slot pass on the GPU through the C ABI (tria_score per layer,
tria_shared_combine, tria_shared_select, tria_compact per layer) against the
oracle's shared_evict: combined scores within the score tolerance, one keep
list per sequence identical to the oracle's except rows within the tolerance
of the cut, the same list in every layer and KV head, exact gathers."""
import numpy as np
import pytest

from oracle import tria_oracle as O

import _util as U

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.mark.parametrize("k_type,n_layers", [("f16", 3), ("q8_0", 2), ("f32", 1)])
def test_shared_slot_pass_matches_oracle(lib, k_type, n_layers):
    base = dict(n_kv=2, group=4, hd=64, k_type=k_type, v_type="f16", n_live=[700, 333, 40],
                capacity=[720, 340, 48], cur_pos=[5000, 333, 40], budget_frac=0.5, window=16, sink=2)
    cases = [U.Case(seed=40 + l, **base) for l in range(n_layers)]
    hosts = [U.build_host(c) for c in cases]
    qm = np.concatenate([h["q_mean"] for h in hosts])
    qa = np.concatenate([h["q_abs"] for h in hosts])
    st = lib.Stats(qm, qa, n_kv_heads=2, head_dim=64, rope_theta=1e4)
    devs = [U.to_device(h) for h in hosts]
    caches = [U.lib_cache(lib, c, d) for c, d in zip(cases, devs)]
    pol = U.lib_policy(lib, cases[0])
    ws = U.new_workspace(lib, caches[0], 4)
    rows = cases[0].total_rows()
    scores = torch.full((n_layers, rows), float("nan"), device="cuda")
    for l in range(n_layers):
        lib.score(st, l, caches[l], pol, scores[l], ws=ws)
    combined = torch.full((rows,), float("nan"), device="cuda")
    lib.shared_combine(scores, caches[0], combined, ws=ws)
    keep = torch.full((rows,), -1, dtype=torch.int32, device="cuda")
    lib.shared_select(combined, caches[0], pol, keep, ws=ws)
    for l in range(n_layers):
        lib.compact(caches[l], pol, keep, ws=ws)
    assert lib.device_status(ws) == lib.OK

    layer_caches = [{k: h[k] for k in ("k", "k_scale", "v", "v_scale", "pos", "n_live", "seq_row0", "capacity")}
                    for h in hosts]
    _, info = O.shared_evict(layer_caches, qm, qa, n_kv_heads=2, head_dim=64, rope_theta=1e4,
                             cur_pos=base["cur_pos"], n_ctx=base["n_live"], budget_frac=0.5, window=16, sink=2)
    comb = combined.cpu().numpy()
    keep_h = keep.cpu().numpy()
    got = [{k: (None if v is None else v.cpu().numpy()) for k, v in d.items()} for d in devs]
    r0s = cases[0].seq_row0()
    for s, it in info.items():
        r0, cap, n, b = int(r0s[s]), base["capacity"][s], it["n"], it["B"]
        err = np.abs(comb[r0:r0 + n] - it["combined"]) / np.maximum(np.abs(it["combined"]), 1.0)
        assert err.max() <= U.RTOL, f"seq {s} combined rel err {err.max():.2e}"
        m = min(n, b)
        kp = keep_h[r0:r0 + m]
        U.assert_keep_sets_match(kp, it["keep"], it["combined"], n, b, 2, 16, f"seq {s}")
        for g in range(2):
            np.testing.assert_array_equal(keep_h[r0 + g * cap:r0 + g * cap + m], kp)
        for l in range(n_layers):
            assert got[l]["n_live"][s] == m
            for g in range(2):
                a = r0 + g * cap
                for name in ("k", "k_scale", "v", "pos"):
                    if hosts[l][name] is None:
                        continue
                    if n > b:
                        np.testing.assert_array_equal(got[l][name][a:a + m], hosts[l][name][a + kp])
                    else:
                        assert got[l][name][a:a + cap].tobytes() == hosts[l][name][a:a + cap].tobytes()
