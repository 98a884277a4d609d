"""Shared helpers of the GPU tests: seeded caches of arbitrary shape, the
library's structs for them, and the parity rules.

Inputs come from :mod:`synth` (host form); the oracle reads the host arrays,
the CUDA path gets a copy of the same bytes. Nothing here computes any part
of the eviction method.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

from synth import counter_rng as C
from synth import workloads as W

RTOL = 1e-3  # scores: |gpu - oracle| <= 1e-3 * max(|oracle|, tau)


@dataclass
class Case:
    n_kv: int
    group: int
    hd: int
    k_type: str
    v_type: str
    n_live: list
    capacity: list
    cur_pos: list
    budget_frac: float = 0.5
    window: int = 16
    sink: int = 2
    seed: int = 11
    n_ctx: list | None = None
    budget_rows: list | None = None
    offsets: list | None = None
    theta: float = 1e4
    host: dict = field(default_factory=dict)

    @property
    def n_seqs(self):
        return len(self.n_live)

    def seq_row0(self):
        out, acc = [], 0
        for c in self.capacity:
            out.append(acc)
            acc += self.n_kv * c
        return np.asarray(out, dtype=np.int64)

    def total_rows(self):
        return int(sum(self.n_kv * c for c in self.capacity))

    def budgets(self):
        if self.budget_rows is not None:
            return list(self.budget_rows)
        return [int(math.floor(self.budget_frac * c)) for c in (self.n_ctx or self.n_live)]


def build_host(case: Case):
    """Host cache + stats for ``case`` (keys/values from the counter generator)."""
    hd, fc, rows = case.hd, case.hd // 2, case.total_rows()
    kdt = {"f32": np.float32, "f16": np.float16, "q8_0": np.int8}[case.k_type]
    vdt = {"f32": np.float32, "f16": np.float16, "q8_0": np.int8}[case.v_type]
    k = np.zeros((rows, hd), kdt)
    ks = np.zeros((rows, hd // 32), np.float16) if case.k_type == "q8_0" else None
    v = np.zeros((rows, hd), vdt)
    vs = np.zeros((rows, hd // 32), np.float16) if case.v_type == "q8_0" else None
    pos = np.zeros(rows, np.int32)
    r0 = case.seq_row0()
    rng = np.random.default_rng(case.seed)
    for s in range(case.n_seqs):
        cap = case.capacity[s]
        for g in range(case.n_kv):
            a = int(r0[s] + g * cap)
            scale = np.where(rng.random(fc) < 0.1, 8.0, 1.0).astype(np.float32)
            kx = C.segment_values(C.stream_key(case.seed, C.TENSOR_K, 0, s, g), cap, hd, scale)
            vx = C.segment_values(C.stream_key(case.seed, C.TENSOR_V, 0, s, g), cap, hd, None)
            if case.k_type == "q8_0":
                k[a:a + cap], ks[a:a + cap] = C.quantize_q8_0(kx)
            else:
                k[a:a + cap] = kx.astype(kdt)
            if case.v_type == "q8_0":
                v[a:a + cap], vs[a:a + cap] = C.quantize_q8_0(vx)
            else:
                v[a:a + cap] = vx.astype(vdt)
            pos[a:a + cap] = np.arange(cap) * 3 + 7
    nq = case.n_kv * case.group
    qm = rng.standard_normal((1, nq, fc, 2)).astype(np.float32)
    qa = (np.hypot(qm[..., 0], qm[..., 1]).astype(np.float64)
          + 0.5 * np.abs(rng.standard_normal((1, nq, fc)))).astype(np.float32)
    case.host = {"k": k, "k_scale": ks, "v": v, "v_scale": vs, "pos": pos,
                 "n_live": np.asarray(case.n_live, np.int32), "seq_row0": r0,
                 "capacity": np.asarray(case.capacity, np.int32), "q_mean": qm, "q_abs": qa}
    return case.host


def to_device(host: dict):
    import torch
    out = {}
    for key in ("k", "k_scale", "v", "v_scale", "pos", "n_live"):
        val = host.get(key)
        out[key] = None if val is None else torch.from_numpy(np.ascontiguousarray(val)).cuda()
    return out


def lib_cache(tria, case: Case, dev: dict):
    return tria.LayerCache(k=dev["k"], v=dev["v"], pos=dev["pos"], n_live=dev["n_live"],
                           seq_row0=case.seq_row0(), capacity=case.capacity, head_dim=case.hd,
                           n_kv_heads=case.n_kv, k_type=case.k_type, v_type=case.v_type,
                           k_scale=dev.get("k_scale"), v_scale=dev.get("v_scale"))


def lib_policy(tria, case: Case):
    return tria.Policy(budget_frac=case.budget_frac, n_ctx=case.n_ctx or case.n_live,
                       budget_rows=case.budget_rows, window=case.window, sink=case.sink,
                       interval=128, cur_pos=case.cur_pos)


def workload_cache(tria, w: W.Workload, dev: dict):
    return tria.LayerCache(k=dev["k"], v=dev["v"], pos=dev["pos"], n_live=dev["n_live"],
                           seq_row0=w.seq_row0(), capacity=w.capacity, head_dim=w.head_dim,
                           n_kv_heads=w.n_kv_heads, k_type=w.k_type, v_type=w.v_type,
                           k_scale=dev.get("k_scale"))


def workload_policy(tria, w: W.Workload):
    return tria.Policy(budget_frac=w.budget_frac, n_ctx=w.n_ctx, window=w.window, sink=w.sink,
                       interval=w.interval, cur_pos=w.cur_pos)


def new_workspace(tria, cache, group):
    import torch
    nbytes = tria.workspace_size(cache, group)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    tria.workspace_init(ws)
    return ws


def assert_scores_close(gpu_raw, ora_raw, gpu_s, ora_s, what=""):
    """Raw: tau = RMS of that head's oracle raw scores; s (z-max): tau = 1."""
    tau = np.sqrt(np.mean(ora_raw ** 2, axis=0))[None, :]
    err_raw = np.abs(gpu_raw - ora_raw) / np.maximum(np.abs(ora_raw), tau)
    assert err_raw.max() <= RTOL, f"{what} raw rel err {err_raw.max():.3e}"
    err_s = np.abs(gpu_s - ora_s) / np.maximum(np.abs(ora_s), 1.0)
    assert err_s.max() <= RTOL, f"{what} s rel err {err_s.max():.3e}"
    return float(err_raw.max()), float(err_s.max())


def assert_keep_sets_match(gpu_keep, ora_keep, ora_s, n, budget, sink, window, what=""):
    """Identical except rows whose oracle score lies within the tolerance of the
    cut-off score (the k-th best candidate's)."""
    gpu_keep, ora_keep = np.asarray(gpu_keep), np.asarray(ora_keep)
    assert len(gpu_keep) == len(ora_keep) == min(n, budget), what
    assert np.all(np.diff(gpu_keep) > 0), what
    if n <= budget:
        assert np.array_equal(gpu_keep, np.arange(n)), what
        return 0
    cand = np.arange(sink, n - window)
    kk = budget - sink - window
    if kk <= 0:
        assert np.array_equal(gpu_keep, ora_keep), what
        return 0
    order = np.argsort(-ora_s[cand], kind="stable")
    s_cut = ora_s[cand[order[kk - 1]]]
    tol = RTOL * max(abs(s_cut), 1.0)
    diff = np.setxor1d(gpu_keep, ora_keep)
    bad = [r for r in diff if abs(ora_s[r] - s_cut) > tol]
    assert not bad, f"{what}: {len(bad)} keep-set differences away from the cut, e.g. {bad[:5]}"
    prot = np.concatenate([np.arange(sink), np.arange(n - window, n)])
    assert np.all(np.isin(prot, gpu_keep)), what
    return len(diff)
