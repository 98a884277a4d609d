"""Pins of the shared-slot oracle (one keep-set per token for all layers and
KV heads) against the per-segment pass it extends."""
import numpy as np

from oracle import tria_oracle as O


def _cache(seed, n_kv, cap, n, hd):
    r = np.random.default_rng(seed)
    rows = n_kv * cap
    return {"k": r.standard_normal((rows, hd)).astype(np.float32), "k_scale": None,
            "v": r.standard_normal((rows, hd)).astype(np.float32), "v_scale": None,
            "pos": np.tile(np.arange(cap, dtype=np.int32) * 2 + 1, n_kv), "n_live": np.array([n], np.int32),
            "seq_row0": np.array([0]), "capacity": np.array([cap], np.int32)}


def _stats(seed, n_q, fc):
    r = np.random.default_rng(seed)
    qm = r.standard_normal((1, n_q, fc, 2))
    return qm, np.hypot(qm[..., 0], qm[..., 1]) + 0.4


KW = dict(head_dim=32, rope_theta=1e4, cur_pos=[300], n_ctx=[90], budget_frac=0.5, window=5, sink=3)


def test_one_layer_one_head_is_the_per_segment_pass():
    c = _cache(1, 1, 96, 90, 32)
    qm, qa = _stats(2, 4, 16)
    out_s, info_s = O.shared_evict([c], qm, qa, n_kv_heads=1, **KW)
    out_e, info_e = O.evict_layer(c, qm, qa, layer=0, n_kv_heads=1, **KW)
    np.testing.assert_array_equal(info_s[0]["keep"], info_e[(0, 0)]["keep"])
    np.testing.assert_array_equal(info_s[0]["combined"], info_e[(0, 0)]["s"])
    for name in ("k", "v", "pos", "n_live"):
        assert out_s[0][name].tobytes() == out_e[name].tobytes(), name


def test_combined_is_the_max_over_layers_and_heads():
    caches = [_cache(10 + l, 2, 96, 90, 32) for l in range(3)]
    qm = np.concatenate([_stats(20 + l, 4, 16)[0] for l in range(3)])
    qa = np.hypot(qm[..., 0], qm[..., 1]) + 0.4
    _, info = O.shared_evict(caches, qm, qa, n_kv_heads=2, **KW)
    per = []
    for l in range(3):
        _, inf = O.evict_layer(caches[l], qm, qa, layer=l, n_kv_heads=2, **KW)
        per += [inf[(0, g)]["s"] for g in range(2)]
    np.testing.assert_array_equal(info[0]["combined"], np.max(np.stack(per), axis=0))


def test_identical_layers_and_heads_keep_the_per_segment_set():
    c = _cache(3, 1, 96, 90, 32)
    two = {k: (None if v is None else (np.concatenate([v, v]) if k in ("k", "v", "pos") else v.copy()))
           for k, v in c.items()}
    qm, qa = _stats(4, 2, 16)
    qm2 = np.concatenate([qm, qm], axis=1)      # both KV heads get the same query heads' stats
    qa2 = np.concatenate([qa, qa], axis=1)
    _, info1 = O.evict_layer(c, qm, qa, layer=0, n_kv_heads=1, **KW)
    out, info = O.shared_evict([two, two], np.concatenate([qm2, qm2]), np.concatenate([qa2, qa2]),
                               n_kv_heads=2, **KW)
    np.testing.assert_array_equal(info[0]["keep"], info1[(0, 0)]["keep"])
    # every layer and head compacted with the one keep list
    keep = info[0]["keep"]
    for o in out:
        for g in range(2):
            np.testing.assert_array_equal(o["pos"][g * 96:g * 96 + len(keep)], c["pos"][keep])


def test_nan_scores_are_ignored_by_the_combine():
    c = _cache(6, 2, 96, 90, 32)
    c["k"][5] = np.nan                            # a NaN key: every z of KV head 0 is NaN
    qm, qa = _stats(7, 4, 16)
    _, info = O.shared_evict([c], qm, qa, n_kv_heads=2, **KW)
    _, inf = O.evict_layer(c, qm, qa, layer=0, n_kv_heads=2, **KW)
    assert np.all(np.isnan(inf[(0, 0)]["s"]))
    np.testing.assert_array_equal(info[0]["combined"], inf[(0, 1)]["s"])
