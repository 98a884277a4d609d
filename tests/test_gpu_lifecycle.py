"""A decode loop on the GPU, through the C ABI: rows appended with
tria_append, passes run with tria_evict whenever the library's schedule says
so, and every pass checked against the oracle running the same loop on host
arrays (keep-sets identical except rows within the score tolerance of the
cut; the compacted planes exact gathers). A second, unchecked run of the same
loop - no host reads between steps - must end in the same bytes."""
import numpy as np
import pytest

from oracle import tria_oracle as O
from synth import counter_rng as C

import _util as U

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

NP = {"f32": np.float32, "f16": np.float16, "q8_0": np.int8}

LOOPS = [
    dict(n_kv=2, group=4, hd=64, k_type="f16", v_type="f16", capacity=[512, 384], prompts=[40, 100],
         n_decode=400, schedule=dict(trigger=0, kv_budget=200, divide_length=48, count_prompt_tokens=True,
                                     protect_prefill=True, window=16, sink=0)),
    dict(n_kv=1, group=8, hd=128, k_type="q8_0", v_type="f16", capacity=[300, 300, 304], prompts=[0, 17, 64],
         n_decode=300, schedule=dict(trigger=0, kv_budget=128, divide_length=32, count_prompt_tokens=False,
                                     protect_prefill=True, window=8, sink=2)),
    dict(n_kv=2, group=2, hd=96, k_type="f32", v_type="q8_0", capacity=[400], prompts=[150],
         n_decode=200, schedule=dict(trigger=1, divide_length=40, budget_frac=0.5, n_ctx=256,
                                     count_prompt_tokens=True, protect_prefill=False, window=16, sink=4)),
]


def _planes(cfg, seed=3):
    """Every token's rows per (sequence, KV head), in the cache's formats."""
    hd, out = cfg["hd"], {}
    rng = np.random.default_rng(seed)
    for s, p in enumerate(cfg["prompts"]):
        t = p + cfg["n_decode"]
        for g in range(cfg["n_kv"]):
            scale = np.where(rng.random(hd // 2) < 0.1, 8.0, 1.0).astype(np.float32)
            kx = C.segment_values(C.stream_key(seed, C.TENSOR_K, 0, s, g), t, hd, scale)
            vx = C.segment_values(C.stream_key(seed, C.TENSOR_V, 0, s, g), t, hd, None)
            rows = {}
            for name, x, dt in (("k", kx, cfg["k_type"]), ("v", vx, cfg["v_type"])):
                if dt == "q8_0":
                    rows[name], rows[name + "_scale"] = C.quantize_q8_0(x)
                else:
                    rows[name], rows[name + "_scale"] = x.astype(NP[dt]), None
            out[(s, g)] = rows
    nq = cfg["n_kv"] * cfg["group"]
    qm = rng.standard_normal((1, nq, hd // 2, 2)).astype(np.float32)
    qa = (np.hypot(qm[..., 0], qm[..., 1]) + 0.5 * np.abs(rng.standard_normal((1, nq, hd // 2)))).astype(np.float32)
    return out, qm, qa


class Loop:
    def __init__(self, lib, cfg, planes, qm, qa):
        self.lib, self.cfg, self.planes = lib, cfg, planes
        self.stats_q = (qm, qa)
        caps, n_kv, hd = cfg["capacity"], cfg["n_kv"], cfg["hd"]
        self.row0 = np.cumsum([0] + [n_kv * c for c in caps[:-1]]).astype(np.int64)
        rows = int(sum(n_kv * c for c in caps))
        self.host = {"k": np.zeros((rows, hd), NP[cfg["k_type"]]), "v": np.zeros((rows, hd), NP[cfg["v_type"]]),
                     "k_scale": np.zeros((rows, hd // 32), np.float16) if cfg["k_type"] == "q8_0" else None,
                     "v_scale": np.zeros((rows, hd // 32), np.float16) if cfg["v_type"] == "q8_0" else None,
                     "pos": np.zeros(rows, np.int32), "n_live": np.zeros(len(caps), np.int32),
                     "seq_row0": self.row0, "capacity": np.asarray(caps, np.int32)}
        self.dev = U.to_device(self.host)
        self.cache = self._cache(range(len(caps)))
        self.ws = U.new_workspace(lib, self.cache, cfg["group"])
        self.stats = lib.Stats(qm, qa, n_kv_heads=n_kv, head_dim=hd, rope_theta=1e4)
        self.sch = lib.Schedule(**cfg["schedule"])
        self.seqs = lib.Sequences(self.sch, caps)
        self.tok = [0] * len(caps)
        self.events = {s: [] for s in range(len(caps))}

    def _cache(self, seqs):
        seqs = list(seqs)
        n_live = self.dev["n_live"] if len(seqs) == len(self.cfg["capacity"]) else self.dev["n_live"][seqs[0]:seqs[0] + 1]
        return self.lib.LayerCache(k=self.dev["k"], v=self.dev["v"], pos=self.dev["pos"], n_live=n_live,
                                   seq_row0=self.row0[seqs], capacity=np.asarray(self.cfg["capacity"])[seqs],
                                   head_dim=self.cfg["hd"], n_kv_heads=self.cfg["n_kv"], k_type=self.cfg["k_type"],
                                   v_type=self.cfg["v_type"], k_scale=self.dev["k_scale"],
                                   v_scale=self.dev["v_scale"])

    def _append(self, seqs, n):
        """n tokens for every sequence in seqs: device via tria_append, host mirror by hand."""
        if n == 0:
            return
        new = {}
        for name in ("k", "k_scale", "v", "v_scale"):
            if self.host[name] is None:
                new[name] = None
                continue
            blk = np.stack([np.stack([self.planes[(s, g)][name][self.tok[s]:self.tok[s] + n]
                                      for g in range(self.cfg["n_kv"])]) for s in seqs])
            new[name] = torch.from_numpy(np.ascontiguousarray(blk)).cuda()
        pos = np.stack([np.arange(self.tok[s], self.tok[s] + n, dtype=np.int32) for s in seqs])
        cache = self.cache if len(seqs) == len(self.cfg["capacity"]) else self._cache(seqs)
        self.lib.append(cache, new["k"], new["v"], torch.from_numpy(pos).cuda(), ws=self.ws,
                        k_scale_new=new["k_scale"], v_scale_new=new["v_scale"])
        for i, s in enumerate(seqs):
            cap, nl = self.cfg["capacity"][s], int(self.host["n_live"][s])
            for g in range(self.cfg["n_kv"]):
                r = int(self.row0[s]) + g * cap + nl
                for name in ("k", "k_scale", "v", "v_scale"):
                    if self.host[name] is not None:
                        self.host[name][r:r + n] = self.planes[(s, g)][name][self.tok[s]:self.tok[s] + n]
                self.host["pos"][r:r + n] = pos[i]
            self.host["n_live"][s] += n
            self.tok[s] += n

    def run(self, check):
        lib, cfg = self.lib, self.cfg
        for s, p in enumerate(cfg["prompts"]):
            self.seqs.prefill(s, p)
            self._append([s], p)
        all_seqs = list(range(len(cfg["capacity"])))
        for step in range(1, cfg["n_decode"] + 1):
            self._append(all_seqs, 1)
            due = [self.seqs.decode(s) for s in all_seqs]
            if not any(due):
                continue
            pol, nd = self.seqs.policy()
            b, k, p = pol.budget_rows, pol.sink_rows, pol.cur_pos
            for s in all_seqs:
                if due[s]:
                    st = self.seqs.state(s)
                    self.events[s].append({"step": step, "pos": int(p[s]), "rows_before": st["rows"],
                                           "counted_before": st["counted"], "budget": int(b[s]), "sink": int(k[s])})
            lib.evict(self.stats, 0, self.cache, pol, ws=self.ws)
            if check:
                self._check_pass(due, b, k, p)
            self.seqs.passed()
            for s in all_seqs:
                if due[s]:
                    self.events[s][-1]["rows_after"] = self.seqs.state(s)["rows"]
        assert lib.device_status(self.ws) == lib.OK
        return {name: (None if t is None else t.cpu().numpy()) for name, t in self.dev.items()}

    def _check_pass(self, due, b, k, p):
        lib, cfg = self.lib, self.cfg
        assert lib.device_status(self.ws) == lib.OK
        got = {name: (None if t is None else t.cpu().numpy()) for name, t in self.dev.items()}
        window = cfg["schedule"]["window"]
        ora, info = O.evict_layer(self.host, self.stats_q[0], self.stats_q[1], layer=0, n_kv_heads=cfg["n_kv"],
                                  head_dim=cfg["hd"], rope_theta=1e4, cur_pos=p, n_ctx=None, budget_frac=0.0,
                                  window=window, sink=k, budget_rows_override=b)
        for s, d in enumerate(due):
            n, cap = int(self.host["n_live"][s]), cfg["capacity"][s]
            bs = min(n, int(b[s]))
            assert got["n_live"][s] == bs
            for g in range(cfg["n_kv"]):
                r0 = int(self.row0[s]) + g * cap
                if not d or n <= bs:
                    for name in ("k", "k_scale", "v", "v_scale", "pos"):
                        if got[name] is not None:
                            assert got[name][r0:r0 + cap].tobytes() == self.host[name][r0:r0 + cap].tobytes()
                    continue
                it = info[(s, g)]
                gk = np.searchsorted(self.host["pos"][r0:r0 + n], got["pos"][r0:r0 + bs])
                U.assert_keep_sets_match(gk, it["keep"], it["s"], n, bs, int(k[s]), window, f"seq {s} head {g}")
                for name in ("k", "k_scale", "v", "v_scale", "pos"):
                    if got[name] is None:
                        continue
                    np.testing.assert_array_equal(got[name][r0:r0 + bs], self.host[name][r0 + gk])
                    assert got[name][r0 + bs:r0 + cap].tobytes() == self.host[name][r0 + bs:r0 + cap].tobytes()
                # continue the oracle's loop from the (checked) device result
                for name in ("k", "k_scale", "v", "v_scale", "pos"):
                    if got[name] is not None:
                        self.host[name][r0:r0 + cap] = got[name][r0:r0 + cap]
            self.host["n_live"][s] = bs


@pytest.mark.parametrize("cfg", LOOPS)
def test_decode_loop_matches_oracle(lib, cfg):
    planes, qm, qa = _planes(cfg)
    loop = Loop(lib, cfg, planes, qm, qa)
    final = loop.run(check=True)
    # the schedule the library ran is the oracle's schedule
    trig = "length" if cfg["schedule"]["trigger"] == 0 else "interval"
    sch = {key: val for key, val in cfg["schedule"].items() if key != "trigger"}
    for s, prompt in enumerate(cfg["prompts"]):
        want = O.schedule_events(trigger=trig, prompt=prompt, n_decode=cfg["n_decode"],
                                 capacity=cfg["capacity"][s], **sch)
        assert loop.events[s] == want, f"seq {s}"
        assert len(want) >= 3
    for name in ("k", "k_scale", "v", "v_scale", "pos", "n_live"):
        if final[name] is not None:
            assert final[name].tobytes() == loop.host[name].tobytes(), name
    # the same loop with no host reads between steps ends in the same bytes
    again = Loop(lib, cfg, planes, qm, qa)
    final2 = again.run(check=False)
    for name in ("k", "k_scale", "v", "v_scale", "pos", "n_live"):
        if final[name] is not None:
            assert final2[name].tobytes() == final[name].tobytes(), name


def test_append_writes_rows_and_counts(lib):
    cfg = dict(n_kv=3, group=1, hd=32, k_type="q8_0", v_type="q8_0", capacity=[40, 24], prompts=[5, 0],
               n_decode=10, schedule=dict(trigger=0, kv_budget=30, divide_length=10, window=0, sink=0))
    planes, qm, qa = _planes(cfg)
    loop = Loop(lib, cfg, planes, qm, qa)
    loop._append([0], 5)
    loop._append([0, 1], 7)
    assert lib.device_status(loop.ws) == lib.OK
    for name in ("k", "k_scale", "v", "v_scale", "pos", "n_live"):
        assert loop.dev[name].cpu().numpy().tobytes() == loop.host[name].tobytes(), name


def test_append_beyond_capacity_is_reported_and_skipped(lib):
    cfg = dict(n_kv=2, group=2, hd=64, k_type="f16", v_type="f16", capacity=[16, 32], prompts=[0, 0],
               n_decode=20, schedule=dict(trigger=0, kv_budget=8, divide_length=4, window=0, sink=0))
    planes, qm, qa = _planes(cfg)
    loop = Loop(lib, cfg, planes, qm, qa)
    loop._append([0, 1], 10)
    assert lib.device_status(loop.ws) == lib.OK
    before = {name: loop.dev[name].cpu().numpy().copy() for name in ("k", "v", "pos", "n_live")}
    k_new = torch.ones((2, 2, 7, 64), dtype=torch.float16, device="cuda")
    pos = torch.full((2, 7), 99, dtype=torch.int32, device="cuda")
    lib.append(loop.cache, k_new, k_new, pos, ws=loop.ws)      # sequence 0: 10 + 7 > 16
    assert lib.device_status(loop.ws) == lib.ERR_CAPACITY
    got = {name: loop.dev[name].cpu().numpy() for name in ("k", "v", "pos", "n_live")}
    assert list(got["n_live"]) == [10, 17]
    r0 = 0
    for name in ("k", "v", "pos"):
        assert got[name][r0:r0 + 32].tobytes() == before[name][r0:r0 + 32].tobytes(), name
    r1 = 32
    for g in range(2):
        a = r1 + g * 32
        assert np.all(got["pos"][a + 10:a + 17] == 99) and np.all(got["k"][a + 10:a + 17] == 1.0)
        assert got["pos"][a:a + 10].tobytes() == before["pos"][a:a + 10].tobytes()
