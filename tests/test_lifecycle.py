"""Decode-loop lifecycle: the oracle's schedule pinned to the numbers the pages
print, and the library's host schedule (tria_seq_* / tria_schedule_*)
checked against the oracle. No GPU use."""
import json
import os

import numpy as np
import pytest

import kv_cache_eviction_tria_gb300 as tria
from oracle import tria_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLDEN, name)) as fh:
        return json.load(fh)


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(tria.LIB_PATH):
        from kv_cache_eviction_tria_gb300 import _build
        _build.build()
    return tria.load_library()


# ---------------------------------------------------------------- oracle pins

def test_oracle_reproduces_the_profile_log():
    """Worklog profile log: with 3072 / 128 the passes run at positions 3200,
    3328, 3456 and 3584, each taking 3200 rows to 3072 (sample9: 157-token
    prompt, prompt rows counted as the bundle's config says)."""
    gold = _gold("worklog_compaction_schedule.json")
    last = gold["compactions"][-1]["abs_pos"]
    ev = O.schedule_events(trigger="length", prompt=157, n_decode=last - 157 + 50, capacity=12288,
                           kv_budget=gold["kv_budget"], divide_length=gold["divide_length"])
    got = [{"abs_pos": e["pos"], "old_rows": e["rows_before"], "kept_rows": e["rows_after"]} for e in ev]
    assert got == gold["compactions"]


def test_oracle_first_compaction_after_a_158_token_prompt():
    gold = _gold("worklog_first_compaction.json")
    ev = O.schedule_events(trigger="length", prompt=gold["prompt_tokens"], n_decode=8000, capacity=32768,
                           kv_budget=gold["kv_budget"], divide_length=gold["divide_length"])
    assert ev[0]["pos"] == gold["first_compaction_abs_pos"]
    assert ev[0]["rows_after"] == gold["keep_count"]
    assert ev[0]["step"] == gold["generated_tokens"]


def test_oracle_decode_only_accounting():
    """Prompt rows outside the count: the trigger sees 7168 decode rows while
    the cache holds the prompt on top; the pass leaves 6144 decode rows
    ([Worklog] "Sample9 boundary replay ...", "Aligned sample9 replay":
    native rows 7168 -> 6144)."""
    gold = _gold("worklog_prompt_accounting.json")
    prompt = gold["prompt_tokens"]
    ev = O.schedule_events(trigger="length", prompt=prompt, n_decode=7300, capacity=32768,
                           kv_budget=gold["kv_budget"], divide_length=gold["divide_length"],
                           count_prompt_tokens=False, protect_prefill=True)
    e = ev[0]
    assert e["counted_before"] == gold["native_rows_before"]
    assert e["rows_before"] - e["counted_before"] == prompt
    assert e["rows_after"] - prompt == gold["kv_budget"]
    assert e["sink"] == prompt
    # with the prompt counted, the same pass comes `prompt` steps earlier
    ev2 = O.schedule_events(trigger="length", prompt=prompt, n_decode=7300, capacity=32768,
                            kv_budget=gold["kv_budget"], divide_length=gold["divide_length"])
    assert e["step"] - ev2[0]["step"] == prompt


def test_oracle_interval_trigger_fires_only_on_decode_steps():
    """[Doc]: a pass every --tri-interval decode steps, never during the
    prompt, keeping floor(budget % * n_ctx) rows (sink and window included)."""
    gold = _gold("doc_cli_flags.json")
    iv = gold["tri_interval"]
    ev = O.schedule_events(trigger="interval", prompt=5000, n_decode=5 * iv + 7, capacity=8192,
                           divide_length=iv, budget_frac=0.5, n_ctx=4096, count_prompt_tokens=True,
                           protect_prefill=False, sink=gold["tri_sink"], window=gold["tri_window"])
    assert [e["step"] for e in ev] == [iv * i for i in range(1, 6)]
    assert ev[0]["rows_before"] == 5000 + iv and ev[0]["rows_after"] == 2048
    assert all(e["rows_before"] == 2048 + iv and e["rows_after"] == 2048 for e in ev[1:])
    assert all(e["pos"] == 5000 + e["step"] for e in ev)


def test_oracle_interval_pass_below_budget_keeps_everything():
    ev = O.schedule_events(trigger="interval", prompt=10, n_decode=256, capacity=1024, divide_length=128,
                           budget_frac=1.0, n_ctx=1000, protect_prefill=False)
    assert [(e["rows_before"], e["rows_after"]) for e in ev] == [(138, 138), (266, 266)]


def test_oracle_prompt_must_fit_the_physical_capacity():
    """[Worklog] Phase 6: no compaction while the prompt is built; the physical
    capacity must hold it."""
    with pytest.raises(O.CapacityError):
        O.schedule_events(trigger="length", prompt=600, n_decode=0, capacity=512, kv_budget=128,
                          divide_length=32)
    with pytest.raises(O.CapacityError):   # decode rows beyond kv_budget + divide_length + prompt
        O.schedule_events(trigger="length", prompt=100, n_decode=300, capacity=259, kv_budget=128,
                          divide_length=32, count_prompt_tokens=False)


def test_oracle_length_invariants():
    """Counted rows never exceed kv_budget + divide_length, every pass leaves
    exactly kv_budget counted rows, and passes are divide_length steps apart."""
    for count, protect in [(True, True), (False, True), (True, False), (False, False)]:
        ev = O.schedule_events(trigger="length", prompt=37, n_decode=2000, capacity=4096, kv_budget=300,
                               divide_length=50, count_prompt_tokens=count, protect_prefill=protect)
        assert all(e["counted_before"] == 350 for e in ev)
        assert all(b["step"] - a["step"] == 50 for a, b in zip(ev, ev[1:]))
        if protect and not count:
            assert all(e["rows_after"] == 337 for e in ev)
        else:
            assert all(e["rows_after"] == 300 for e in ev)


# ------------------------------------------------- the library's host schedule

def _run_library(sch_kw, prompt, n_decode, capacity):
    sch = tria.Schedule(**sch_kw)
    q = tria.Sequences(sch, [capacity])
    q.prefill(0, prompt)
    events = []
    for step in range(1, n_decode + 1):
        before = q.state(0)
        if q.decode(0):
            st = q.state(0)
            b, k, p, nd = q.plan()
            assert nd == 1
            q.passed()
            events.append({"step": step, "pos": int(p[0]), "rows_before": st["rows"],
                           "counted_before": st["counted"], "rows_after": q.state(0)["rows"],
                           "budget": int(b[0]), "sink": int(k[0])})
        else:
            assert q.state(0)["rows"] == before["rows"] + 1
    return events


_CASES = []
_rng = np.random.default_rng(5)
for _ in range(40):
    trig = "length" if _rng.random() < 0.6 else "interval"
    kw = dict(count_prompt_tokens=bool(_rng.integers(2)), protect_prefill=bool(_rng.integers(2)),
              sink=int(_rng.integers(0, 5)), window=int(_rng.integers(0, 20)),
              divide_length=int(_rng.integers(1, 80)))
    prompt = int(_rng.integers(0, 60))
    if trig == "length":
        kw["kv_budget"] = int(_rng.integers(90, 400))
    else:
        kw["budget_frac"], kw["n_ctx"] = float(_rng.uniform(0.3, 1.0)), int(_rng.integers(200, 600))
    _CASES.append((trig, kw, prompt, int(_rng.integers(0, 1500))))


@pytest.mark.parametrize("trig,kw,prompt,n_decode", _CASES)
def test_library_schedule_matches_oracle(lib, trig, kw, prompt, n_decode):
    cap = 4096
    want = O.schedule_events(trigger=trig, prompt=prompt, n_decode=n_decode, capacity=cap, **kw)
    code = tria.TRIGGER_LENGTH if trig == "length" else tria.TRIGGER_INTERVAL
    got = _run_library(dict(trigger=code, **kw), prompt, n_decode, cap)
    assert got == want


def test_library_schedule_errors(lib):
    sch = tria.Schedule(kv_budget=100, divide_length=10, window=4)
    q = tria.Sequences(sch, [120])
    with pytest.raises(tria.TriaError) as e:
        q.prefill(0, 121)                      # the prompt does not fit: nothing appended
    assert e.value.status == tria.ERR_CAPACITY and q.state(0)["rows"] == 0
    q.prefill(0, 20)
    for _ in range(89):
        assert not q.decode(0)
    assert q.decode(0)                         # 110 counted rows
    with pytest.raises(tria.TriaError) as e:
        q.decode(0)                            # the due pass has not run
    assert e.value.status == tria.ERR_INVALID_ARG
    with pytest.raises(tria.TriaError):
        q.prefill(0, 1)                        # prompt after decode steps
    q.passed()
    assert q.state(0)["rows"] == 100 and q.state(0)["passes"] == 1
    # physical capacity smaller than kv_budget + divide_length
    q2 = tria.Sequences(sch, [105])
    q2.prefill(0, 100)
    for _ in range(5):
        q2.decode(0)
    with pytest.raises(tria.TriaError) as e:
        q2.decode(0)
    assert e.value.status == tria.ERR_CAPACITY and q2.state(0)["rows"] == 105
    # protected prompt larger than the budget allows
    sch3 = tria.Schedule(kv_budget=50, divide_length=10, window=8, count_prompt_tokens=True, protect_prefill=True)
    q3 = tria.Sequences(sch3, [200])
    q3.prefill(0, 45)
    while not q3.decode(0):
        pass
    with pytest.raises(tria.TriaError) as e:
        q3.plan()
    assert e.value.status == tria.ERR_BUDGET


def test_library_schedule_rejects_bad_schedules(lib):
    bad = [dict(trigger=2, kv_budget=10), dict(kv_budget=0), dict(kv_budget=10, divide_length=0),
           dict(kv_budget=10, sink=-1), dict(trigger=tria.TRIGGER_INTERVAL, budget_frac=0.0, n_ctx=10),
           dict(trigger=tria.TRIGGER_INTERVAL, budget_frac=1.5, n_ctx=10),
           dict(trigger=tria.TRIGGER_INTERVAL, budget_frac=0.5, n_ctx=-1)]
    for kw in bad:
        with pytest.raises(tria.TriaError):
            tria.Schedule(**kw)


def test_plan_of_several_sequences(lib):
    sch = tria.Schedule(kv_budget=64, divide_length=16, window=4, count_prompt_tokens=False, protect_prefill=True)
    q = tria.Sequences(sch, [256, 256, 256])
    for s, p in enumerate((3, 10, 0)):
        q.prefill(s, p)
    due = [False] * 3
    for _ in range(80):
        for s in range(3):
            due[s] = q.decode(s)
    assert due == [True, True, True]
    b, k, p, nd = q.plan()
    assert nd == 3 and list(b) == [67, 74, 64] and list(k) == [3, 10, 0] and list(p) == [83, 90, 80]
    q.passed()
    assert not q.decode(0)
    b, k, p, nd = q.plan()
    assert nd == 0 and list(b) == [tria.NO_PASS] * 3


def test_oracle_decode_loop_invariants():
    """A tiny decode loop on the CPU (oracle pass at every scheduled step):
    protected prompt rows survive every pass, positions stay strictly
    increasing, the live rows follow the schedule and the kept rows are
    always the last window rows plus the best of the rest."""
    rng = np.random.default_rng(3)
    hd, n_kv, g, cap, prompt, n_decode = 32, 2, 2, 200, 12, 260
    sch = dict(trigger="length", kv_budget=64, divide_length=16, count_prompt_tokens=False,
               protect_prefill=True, window=8, sink=0)
    events = O.schedule_events(prompt=prompt, n_decode=n_decode, capacity=cap, **sch)
    qm = rng.standard_normal((1, n_kv * g, hd // 2, 2))
    qa = np.hypot(qm[..., 0], qm[..., 1]) + 0.3
    tokens = rng.standard_normal((prompt + n_decode, n_kv, hd)).astype(np.float32)
    cache = {"k": np.zeros((n_kv * cap, hd), np.float32), "k_scale": None,
             "v": np.zeros((n_kv * cap, hd), np.float32), "v_scale": None,
             "pos": np.zeros(n_kv * cap, np.int32), "n_live": np.array([0], np.int32),
             "seq_row0": np.array([0]), "capacity": np.array([cap], np.int32)}

    def append(t):
        n = int(cache["n_live"][0])
        for h in range(n_kv):
            cache["k"][h * cap + n] = tokens[t, h]
            cache["v"][h * cap + n] = -tokens[t, h]
            cache["pos"][h * cap + n] = t
        cache["n_live"][0] = n + 1

    for t in range(prompt):
        append(t)
    ev = iter(events)
    nxt = next(ev, None)
    for step in range(1, n_decode + 1):
        append(prompt + step - 1)
        if nxt is not None and nxt["step"] == step:
            assert int(cache["n_live"][0]) == nxt["rows_before"]
            cache, _ = O.evict_layer(cache, qm, qa, layer=0, n_kv_heads=n_kv, head_dim=hd, rope_theta=1e4,
                                     cur_pos=[nxt["pos"]], n_ctx=None, budget_frac=0.0, window=8,
                                     sink=nxt["sink"], budget_rows_override=[nxt["budget"]])
            n = int(cache["n_live"][0])
            assert n == nxt["rows_after"]
            for h in range(n_kv):
                pos = cache["pos"][h * cap:h * cap + n]
                assert np.all(np.diff(pos) > 0)
                np.testing.assert_array_equal(pos[:prompt], np.arange(prompt))          # prompt kept
                np.testing.assert_array_equal(pos[-8:], np.arange(prompt + step - 8, prompt + step))
                np.testing.assert_array_equal(cache["v"][h * cap:h * cap + n], -cache["k"][h * cap:h * cap + n])
            nxt = next(ev, None)
    assert nxt is None and len(events) >= 10
