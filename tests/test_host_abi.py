"""Host-side checks of the C ABI: the library loads, exports what the header
declares, and rejects bad arguments before touching a GPU (no compute calls)."""
import ctypes
import json
import os
import re

import numpy as np
import pytest

import kv_cache_eviction_tria_gb300 as tria

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tria.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(tria.LIB_PATH):
        from kv_cache_eviction_tria_gb300 import _build
        _build.build()
    return tria.load_library()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\S[^;(]*?\b(tria_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_pass_entry_points():
    names = declared_functions()
    for n in ("tria_load_stats", "tria_score", "tria_select", "tria_compact", "tria_evict"):
        assert n in names


def test_header_is_plain_c99(tmp_path):
    """The boundary is a C ABI: the header compiles as strict C99 (no C++ in it)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "use.c"
    src.write_text('#include "tria.h"\n'
                   'int main(void) { tria_policy p = {0}; tria_schedule s = {0}; (void)p; (void)s;\n'
                   '  return tria_should_evict(10, 4, 2); }\n')
    res = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I",
                          os.path.dirname(HEADER), "-c", str(src), "-o", str(tmp_path / "use.o")],
                         capture_output=True, text=True)
    assert res.returncode == 0, res.stderr


def test_library_exports_every_declared_function(lib):
    names = declared_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(lib, n), f"{n} declared in tria.h but not exported"
    assert set(tria.EXPORTS) <= set(names)


def test_version_and_status_strings(lib):
    assert tria.version() == 2
    for code in range(9):
        assert tria.status_string(code) not in ("", "unknown status")
    assert tria.status_string(99) == "unknown status"


def test_gate_matches_the_documented_gate(lib):
    with open(os.path.join(ROOT, "tests", "golden", "doc_gpu_gate.json")) as fh:
        gold = json.load(fh)
    for row in gold["eligible"]:
        assert tria.gate_check(row["nh"], row["nkv"], row["hd"]) == tria.OK, row
    for row in gold["ineligible"]:
        assert tria.gate_check(row["nh"], row["nkv"], row["hd"]) == tria.ERR_UNSUPPORTED, row
    assert tria.gate_check(48, 3, 128) == tria.ERR_UNSUPPORTED   # group 16 > 8
    assert tria.gate_check(0, 8, 128) == tria.ERR_INVALID_ARG


def test_gate_log_line_matches_the_documented_line(lib):
    gold = json.load(open(os.path.join(ROOT, "tests", "golden", "doc_gpu_gate.json")))
    want = gold["source"].split("gate log line '")[1].split("'")[0]
    st, line = tria.gate_describe(32, 8, 128, "q8_0")
    assert st == tria.OK and line == want
    st, line = tria.gate_describe(32, 8, 512, "f16")
    assert st == tria.ERR_UNSUPPORTED and line.endswith("-> ineligible (head_dim > 256)") and "is_q8_0=0" in line
    st, line = tria.gate_describe(30, 8, 128, "q8_0")
    assert st == tria.ERR_UNSUPPORTED and "(nh % nkv != 0)" in line


def test_gate_non_rotary_dims(lib):
    """Heads with non-rotary dims: the gate line carries nonrot=; eligible
    when the rotary dims are a multiple of 16, invalid outside [0, head_dim)."""
    st, line = tria.gate_describe(32, 8, 128, "f16", nonrot_dim=64)
    assert st == tria.OK and "hd=128 nonrot=64 -> eligible" in line
    assert tria.gate_check(32, 8, 256, 192) == tria.OK
    assert tria.gate_check(32, 8, 128, 16) == tria.OK          # 112 rotary dims
    st, line = tria.gate_describe(32, 8, 128, "q8_0", nonrot_dim=8)
    assert st == tria.ERR_UNSUPPORTED and line.endswith("(rotary dims % 16 != 0)")
    assert tria.gate_check(32, 8, 128, 128) == tria.ERR_INVALID_ARG
    assert tria.gate_check(32, 8, 128, -2) == tria.ERR_INVALID_ARG


def test_budget_rows_and_trigger(lib):
    assert tria.budget_rows(0.5, 512) == 256
    assert tria.budget_rows(0.25, 98710) == 24677
    assert tria.budget_rows(0.3, 10) == 3
    gold = json.load(open(os.path.join(ROOT, "tests", "golden", "worklog_compaction_schedule.json")))
    assert tria.should_evict(gold["trigger"], gold["kv_budget"], gold["divide_length"])
    assert not tria.should_evict(gold["trigger"] - 1, gold["kv_budget"], gold["divide_length"])


def _fake_cache(n_seqs=2, cap=(1000, 900), k=0x10000, v=0x20000, k_type="f16", hd=128, n_kv=8,
                k_scale=None):
    """A cache struct with fake (never dereferenced) device addresses."""
    return tria.LayerCache(k=k, v=v, pos=0x30000, n_live=0x40000,
                           seq_row0=[0, n_kv * cap[0]][:n_seqs], capacity=list(cap)[:n_seqs],
                           head_dim=hd, n_kv_heads=n_kv, k_type=k_type, v_type="f16", k_scale=k_scale)


def test_workspace_size_layout_rules(lib):
    c = _fake_cache()
    n4 = tria.workspace_size(c, 4)
    n0 = tria.workspace_size(c, 0)
    rows = 8 * 1900
    assert n4 - n0 >= rows * 4 * 4          # raw scores for G = 4
    assert n0 >= rows * 8                   # score + keep per row
    with pytest.raises(tria.TriaError):
        tria.workspace_size(_fake_cache(k=0x10008), 4)            # k not 16-byte aligned
    with pytest.raises(tria.TriaError):
        tria.workspace_size(_fake_cache(hd=80), 4)                # head_dim % 32
    with pytest.raises(tria.TriaError):
        tria.workspace_size(_fake_cache(k_type="q8_0"), 4)        # q8_0 without scales
    overlap = tria.LayerCache(k=0x10000, v=0x20000, pos=0x30000, n_live=0x40000, seq_row0=[0, 100],
                              capacity=[64, 64], head_dim=64, n_kv_heads=2)
    with pytest.raises(tria.TriaError):
        tria.workspace_size(overlap, 4)                           # sequences overlap


def _call_select(c, pol, ws=0x100000, nbytes=1 << 30, score=0x50000, keep=0x60000):
    cs, ps = c.c_struct(), pol.c_struct()
    return tria.raw_call("tria_select", ctypes.c_void_p(score), ctypes.byref(cs), ctypes.byref(ps),
                         ctypes.c_void_p(keep), ctypes.c_void_p(ws), nbytes, None)


def test_host_validation_rejects_before_any_launch(lib):
    c = _fake_cache()
    good = tria.Policy(budget_frac=0.5, n_ctx=[1000, 900], window=64, sink=4, cur_pos=[1000, 900])
    assert _call_select(c, tria.Policy(budget_frac=0.05, n_ctx=[1000, 900], window=64, sink=4)) \
        == tria.ERR_BUDGET
    assert _call_select(c, good, ws=0x100010) == tria.ERR_WORKSPACE          # misaligned ws
    assert _call_select(c, good, nbytes=1024) == tria.ERR_WORKSPACE          # too small
    assert _call_select(c, good, score=0) == tria.ERR_INVALID_ARG
    assert _call_select(c, tria.Policy(budget_frac=1.5, n_ctx=[1, 1])) == tria.ERR_INVALID_ARG
    assert _call_select(c, tria.Policy(budget_rows=[100, -1], window=0, sink=0)) == tria.ERR_INVALID_ARG
    cs, ps = c.c_struct(), good.c_struct()
    # evict / score with no stats handle
    assert tria.raw_call("tria_evict", None, 0, ctypes.byref(cs), ctypes.byref(ps),
                         ctypes.c_void_p(0x100000), 1 << 30, None) == tria.ERR_INVALID_ARG
    assert tria.raw_call("tria_workspace_init", ctypes.c_void_p(0x100010), 4096, None) \
        == tria.ERR_WORKSPACE


def test_model_dispatch_query_host_checks(lib):
    # no stats handle, or no layers: the model call would reject them (-1)
    c = _fake_cache()
    structs = (tria._LayerCache * 1)(c.c_struct())
    layers = (ctypes.c_int32 * 1)(0)
    assert tria.raw_call("tria_evict_model_fused", None, layers, 1, structs) == -1
    assert tria.raw_call("tria_evict_model_fused", None, None, 0, structs) == -1


def test_shared_slot_and_append_argument_checks(lib):
    # rejected on the host before any launch (fake, aligned pointers are never touched)
    c = _fake_cache()
    cs = c.c_struct()
    good = tria.Policy(budget_frac=0.5, n_ctx=[1000, 900], window=64, sink=4, cur_pos=[1000, 900])
    ps = good.c_struct()
    rows = 8 * 1000 + 8 * 900
    comb = lambda scores, stride, nl, out, ws, nb: tria.raw_call(
        "tria_shared_combine", ctypes.c_void_p(scores), stride, nl, ctypes.byref(cs), ctypes.c_void_p(out),
        ctypes.c_void_p(ws), nb, None)
    assert comb(0x40000, rows - 1, 2, 0x50000, 0x100000, 4096) == tria.ERR_INVALID_ARG     # layers overlap
    assert comb(0x40000, rows, 0, 0x50000, 0x100000, 4096) == tria.ERR_INVALID_ARG         # no layer
    assert comb(0, rows, 1, 0x50000, 0x100000, 4096) == tria.ERR_INVALID_ARG
    assert comb(0x40002, rows, 1, 0x50000, 0x100000, 4096) == tria.ERR_INVALID_ARG         # misaligned
    assert comb(0x40000, rows, 1, 0x50000, 0x100010, 4096) == tria.ERR_WORKSPACE
    assert comb(0x40000, rows, 1, 0x50000, 0x100000, 16) == tria.ERR_WORKSPACE
    sel = lambda pol, keep, nb: tria.raw_call(
        "tria_shared_select", ctypes.c_void_p(0x50000), ctypes.byref(cs), ctypes.byref(pol.c_struct()),
        ctypes.c_void_p(keep), ctypes.c_void_p(0x100000), nb, None)
    assert sel(good, 0, 1 << 30) == tria.ERR_INVALID_ARG
    assert sel(good, 0x60000, 16) == tria.ERR_WORKSPACE
    assert sel(tria.Policy(budget_frac=0.05, n_ctx=[1000, 900], window=64, sink=4), 0x60000, 1 << 30) \
        == tria.ERR_BUDGET
    app = lambda k, ks, v, pos, n, ws: tria.raw_call(
        "tria_append", ctypes.byref(cs), ctypes.c_void_p(k), ctypes.c_void_p(ks), ctypes.c_void_p(v),
        None, ctypes.c_void_p(pos), n, ctypes.c_void_p(ws), 1 << 20, None)
    assert app(0x40000, 0, 0x48000, 0x50000, -1, 0x100000) == tria.ERR_INVALID_ARG
    assert app(0x40000, 0, 0x48000, 0x50000, 1, 0x100010) == tria.ERR_WORKSPACE
    assert app(0x40008, 0, 0x48000, 0x50000, 1, 0x100000) == tria.ERR_INVALID_ARG         # k not 16-aligned
    assert app(0x40000, 0x30000, 0x48000, 0x50000, 1, 0x100000) == tria.ERR_INVALID_ARG   # scale for fp16
    assert app(0, 0, 0, 0, 0, 0x100000) == tria.OK                                        # nothing to append


def test_load_stats_rejects_ineligible_shapes(lib):
    qm = np.zeros((1, 30, 64, 2), np.float32)
    with pytest.raises(tria.TriaError) as e:
        tria.Stats(qm, None, n_kv_heads=8, head_dim=128, rope_theta=1e6, stream=0)
    assert e.value.status == tria.ERR_UNSUPPORTED
    qm = np.zeros((1, 32, 40, 2), np.float32)
    with pytest.raises(tria.TriaError) as e:
        tria.Stats(qm, None, n_kv_heads=8, head_dim=80, rope_theta=1e6, stream=0)
    assert e.value.status == tria.ERR_UNSUPPORTED
    qm = np.zeros((1, 32, 64, 2), np.float32)
    with pytest.raises(tria.TriaError) as e:    # uneven head map
        tria.Stats(qm, None, n_kv_heads=8, head_dim=128, rope_theta=1e6, kv_of_q=[0] * 32, stream=0)
    assert e.value.status == tria.ERR_INVALID_ARG


def test_load_stats_hybrid_table_checks(lib):
    # per-layer head_dim table ([Doc] §6 hybrid models): rejected on the host
    # before any device allocation
    def stats(hds, thetas=None):
        qm = [np.zeros((8, hd // 2 if hd > 0 else 1, 2), np.float32) for hd in hds]
        return tria.Stats(qm, None, n_kv_heads=2, layer_head_dim=hds, rope_theta=1e4,
                          layer_rope_theta=thetas, stream=0)
    for hds in ([128, 0], [127], [64, -2]):
        with pytest.raises(tria.TriaError) as e:
            stats(hds)
        assert e.value.status == tria.ERR_INVALID_ARG, hds
    with pytest.raises(tria.TriaError) as e:       # no layer passes the gate
        stats([512, 80, 1024])
    assert e.value.status == tria.ERR_UNSUPPORTED
    with pytest.raises(tria.TriaError) as e:       # a theta of a layer <= 1
        stats([128, 64], thetas=[1e4, 1.0])
    assert e.value.status == tria.ERR_INVALID_ARG


def test_calibration_argument_checks(lib):
    # rejected on the host before any launch (fake, aligned pointers are never touched)
    q, acc = ctypes.c_void_p(0x100000), ctypes.c_void_p(0x200000)
    call = lambda *a: tria.raw_call("tria_calib_accumulate", *a)
    assert call(None, tria.F16, 8, 4, 128, 0, acc, None) == tria.ERR_INVALID_ARG
    assert call(q, tria.F16, 8, 4, 128, 0, None, None) == tria.ERR_INVALID_ARG
    assert call(q, tria.F16, -1, 4, 128, 0, acc, None) == tria.ERR_INVALID_ARG
    assert call(q, tria.F16, 8, 0, 128, 0, acc, None) == tria.ERR_INVALID_ARG
    assert call(ctypes.c_void_p(0x100002), tria.F16, 8, 4, 128, 0, acc, None) == tria.ERR_INVALID_ARG
    assert call(q, tria.F16, 8, 4, 128, 0, ctypes.c_void_p(0x200004), None) == tria.ERR_INVALID_ARG
    assert call(q, tria.Q8_0, 8, 4, 128, 0, acc, None) == tria.ERR_UNSUPPORTED
    assert call(q, tria.F32, 8, 4, 127, 0, acc, None) == tria.ERR_UNSUPPORTED
    assert call(q, tria.F32, 8, 4, 1024, 0, acc, None) == tria.ERR_UNSUPPORTED
    assert call(q, tria.F32, 0, 4, 128, 0, acc, None) == tria.OK   # nothing to add, no launch
    assert call(None, tria.F32, 0, 4, 128, 0, acc, None) == tria.OK
    fin = lambda *a: tria.raw_call("tria_calib_finish", *a)
    qm, qa = ctypes.c_void_p(0x300000), ctypes.c_void_p(0x400000)
    assert fin(acc, 0, 4, 128, 0, qm, qa, None, None) == tria.ERR_INVALID_ARG
    assert fin(acc, 10, 4, 128, 0, None, qa, None, None) == tria.ERR_INVALID_ARG
    assert fin(acc, 10, 4, 130000, 0, qm, qa, None, None) == tria.ERR_UNSUPPORTED
    # non-rotary dims: even, in [0, head_dim); the finish needs q_nonrot then
    assert call(q, tria.F16, 8, 4, 128, 3, acc, None) == tria.ERR_INVALID_ARG
    assert call(q, tria.F16, 8, 4, 128, 128, acc, None) == tria.ERR_INVALID_ARG
    assert fin(acc, 10, 4, 128, 64, qm, qa, None, None) == tria.ERR_INVALID_ARG
    assert fin(acc, 10, 4, 128, -2, qm, qa, ctypes.c_void_p(0x500000), None) == tria.ERR_INVALID_ARG


def test_workspace_score_offset(lib):
    """The staged evict path's z-max array sits inside the workspace, at the same
    place whatever the group; invalid caches give 0."""
    c = _fake_cache()
    off = tria.raw_call("tria_workspace_score_offset", ctypes.byref(c.c_struct()))
    assert 0 < off < tria.workspace_size(c, 0) <= tria.workspace_size(c, 4)
    assert off % 256 == 0
    bad = _fake_cache(n_kv=0)
    assert tria.raw_call("tria_workspace_score_offset", ctypes.byref(bad.c_struct())) == 0


def test_select_noalloc_host_checks_match_select(lib):
    """tria_select_noalloc rejects on the host exactly what tria_select rejects
    (checks that need no workspace): overlapping sequences, a negative n_ctx,
    misaligned pointers, a budget below sink + window."""
    def both(c, pol, score=0x50000, keep=0x60000):
        cs, ps = c.c_struct(), pol.c_struct()
        a = _call_select(c, pol, score=score, keep=keep)
        b = tria.raw_call("tria_select_noalloc", ctypes.c_void_p(score), ctypes.byref(cs), ctypes.byref(ps),
                          ctypes.c_void_p(keep), None)
        return a, b
    overlap = tria.LayerCache(k=0x10000, v=0x20000, pos=0x30000, n_live=0x40000, seq_row0=[0, 100],
                              capacity=[64, 64], head_dim=64, n_kv_heads=2)
    pol2 = tria.Policy(budget_rows=[32, 32], window=0, sink=0)
    assert both(overlap, pol2) == (tria.ERR_INVALID_ARG, tria.ERR_INVALID_ARG)
    c = _fake_cache()
    assert both(c, tria.Policy(budget_frac=0.5, n_ctx=[1000, -1], window=0, sink=0)) \
        == (tria.ERR_INVALID_ARG, tria.ERR_INVALID_ARG)
    good = tria.Policy(budget_frac=0.5, n_ctx=[1000, 900], window=64, sink=4)
    assert both(c, good, score=0x50002) == (tria.ERR_INVALID_ARG, tria.ERR_INVALID_ARG)
    assert both(c, good, keep=0x60001) == (tria.ERR_INVALID_ARG, tria.ERR_INVALID_ARG)
    assert both(_fake_cache(k=0x10008), good) == (tria.ERR_INVALID_ARG, tria.ERR_INVALID_ARG)
    assert both(c, tria.Policy(budget_frac=0.05, n_ctx=[1000, 900], window=64, sink=4)) \
        == (tria.ERR_BUDGET, tria.ERR_BUDGET)
