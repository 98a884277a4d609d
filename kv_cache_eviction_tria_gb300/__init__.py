"""Python binding of the TriAttention KV-cache eviction library (``libtria.so``).

Argument marshalling only: every step of the pass runs in the CUDA kernels of
``libtria.so``; the functions here turn tensors and Python values into the C
structs of ``include/tria.h`` and call the entry point of the same name. There
is no CPU fallback: if the library cannot be loaded, every call raises.

PyTorch supplies device memory and streams. Device arguments are CUDA
tensors; host arguments are sequences of ints / numpy arrays.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtria.so")

TRIA_MAX_SEQS = 128
F32, F16, Q8_0 = 0, 1, 2
DTYPES = {"f32": F32, "f16": F16, "q8_0": Q8_0}

STATUS = {
    0: "TRIA_OK", 1: "TRIA_ERR_INVALID_ARG", 2: "TRIA_ERR_UNSUPPORTED", 3: "TRIA_ERR_BUDGET",
    4: "TRIA_ERR_CUDA", 5: "TRIA_ERR_WORKSPACE", 6: "TRIA_ERR_TIMEOUT", 7: "TRIA_ERR_DEVICE_ARG",
    8: "TRIA_ERR_KEEP_LIST", 9: "TRIA_ERR_CAPACITY",
}
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_BUDGET, ERR_CUDA, ERR_WORKSPACE, ERR_TIMEOUT, \
    ERR_DEVICE_ARG, ERR_KEEP_LIST, ERR_CAPACITY = range(10)
TRIGGER_LENGTH, TRIGGER_INTERVAL = 0, 1
NO_PASS = 2 ** 31 - 1

EXPORTS = (
    "tria_gate_check", "tria_gate_describe", "tria_budget_rows", "tria_should_evict", "tria_load_stats", "tria_free_stats",
    "tria_workspace_size", "tria_workspace_init", "tria_score", "tria_select", "tria_compact",
    "tria_evict", "tria_evict_staged", "tria_evict_model", "tria_evict_model_fused", "tria_model_workspace_size",
    "tria_evict_layers",
    "tria_evict_profiled", "tria_evict_marked", "tria_select_noalloc", "tria_device_status", "tria_selftest_bounded_wait",
    "tria_calib_accumulate", "tria_calib_finish", "tria_append", "tria_schedule_check", "tria_seq_init",
    "tria_seq_prefill", "tria_seq_decode", "tria_schedule_plan", "tria_schedule_passed",
    "tria_shared_combine", "tria_shared_select",
    "tria_status_string", "tria_version", "tria_workspace_score_offset",
)


class TriaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}")


# --------------------------------------------------------------------------- C structs

class _StatsDesc(ctypes.Structure):
    _fields_ = [
        ("n_layers", ctypes.c_int32), ("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("rope_theta", ctypes.c_double),
        ("omega", ctypes.POINTER(ctypes.c_double)), ("q_mean", ctypes.POINTER(ctypes.c_float)),
        ("q_abs", ctypes.POINTER(ctypes.c_float)), ("kv_of_q", ctypes.POINTER(ctypes.c_int32)),
        ("offsets", ctypes.POINTER(ctypes.c_int64)), ("n_offsets", ctypes.c_int32),
        ("layer_head_dim", ctypes.POINTER(ctypes.c_int32)), ("layer_rope_theta", ctypes.POINTER(ctypes.c_double)),
        ("nonrot_dim", ctypes.c_int32), ("q_nonrot", ctypes.POINTER(ctypes.c_float)),
    ]


class _LayerCache(ctypes.Structure):
    _fields_ = [
        ("n_seqs", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("k_type", ctypes.c_int32), ("v_type", ctypes.c_int32),
        ("k", ctypes.c_void_p), ("k_scale", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("v_scale", ctypes.c_void_p), ("pos", ctypes.c_void_p), ("n_live", ctypes.c_void_p),
        ("seq_row0", ctypes.POINTER(ctypes.c_int64)), ("capacity", ctypes.POINTER(ctypes.c_int32)),
    ]


class _Policy(ctypes.Structure):
    _fields_ = [
        ("budget_frac", ctypes.c_double), ("n_ctx", ctypes.POINTER(ctypes.c_int32)),
        ("budget_rows", ctypes.POINTER(ctypes.c_int32)), ("window", ctypes.c_int32),
        ("sink", ctypes.c_int32), ("interval", ctypes.c_int32),
        ("cur_pos", ctypes.POINTER(ctypes.c_int64)), ("sink_rows", ctypes.POINTER(ctypes.c_int32)),
    ]


class _Schedule(ctypes.Structure):
    _fields_ = [
        ("trigger", ctypes.c_int32), ("count_prompt_tokens", ctypes.c_int32),
        ("protect_prefill", ctypes.c_int32), ("sink", ctypes.c_int32), ("window", ctypes.c_int32),
        ("pad", ctypes.c_int32), ("kv_budget", ctypes.c_int64), ("divide_length", ctypes.c_int64),
        ("budget_frac", ctypes.c_double), ("n_ctx", ctypes.c_int64),
    ]


class _SeqState(ctypes.Structure):
    _fields_ = [
        ("capacity", ctypes.c_int64), ("rows", ctypes.c_int64), ("counted", ctypes.c_int64),
        ("prompt_rows", ctypes.c_int64), ("next_pos", ctypes.c_int64), ("decode_steps", ctypes.c_int64),
        ("passes", ctypes.c_int64), ("due", ctypes.c_int32), ("pad", ctypes.c_int32),
    ]


_lib = None


def load_library(path: str | None = None):
    """Load ``libtria.so`` (raises if it is missing: there is no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"{path} not found: build it first (python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    lib.tria_gate_check.argtypes = [i32, i32, i32, i32]
    lib.tria_gate_check.restype = i32
    lib.tria_gate_describe.argtypes = [i32, i32, i32, i32, i32, ctypes.c_char_p, sz]
    lib.tria_gate_describe.restype = i32
    lib.tria_budget_rows.argtypes = [ctypes.c_double, i64]
    lib.tria_budget_rows.restype = i64
    lib.tria_should_evict.argtypes = [i64, i64, i64]
    lib.tria_should_evict.restype = i32
    lib.tria_load_stats.argtypes = [ctypes.POINTER(_StatsDesc), ctypes.POINTER(vp), vp]
    lib.tria_load_stats.restype = i32
    lib.tria_free_stats.argtypes = [vp]
    lib.tria_free_stats.restype = None
    lib.tria_workspace_size.argtypes = [ctypes.POINTER(_LayerCache), i32]
    lib.tria_workspace_size.restype = sz
    lib.tria_workspace_init.argtypes = [vp, sz, vp]
    lib.tria_workspace_init.restype = i32
    lib.tria_score.argtypes = [vp, i32, ctypes.POINTER(_LayerCache), ctypes.POINTER(_Policy), vp, vp, vp, sz, vp]
    lib.tria_score.restype = i32
    lib.tria_select.argtypes = [vp, ctypes.POINTER(_LayerCache), ctypes.POINTER(_Policy), vp, vp, sz, vp]
    lib.tria_select.restype = i32
    lib.tria_select_noalloc.argtypes = [vp, ctypes.POINTER(_LayerCache), ctypes.POINTER(_Policy), vp, vp]
    lib.tria_select_noalloc.restype = i32
    lib.tria_compact.argtypes = [ctypes.POINTER(_LayerCache), ctypes.POINTER(_Policy), vp, vp, sz, vp]
    lib.tria_compact.restype = i32
    lib.tria_evict.argtypes = [vp, i32, ctypes.POINTER(_LayerCache), ctypes.POINTER(_Policy), vp, sz, vp]
    lib.tria_evict.restype = i32
    lib.tria_evict_staged.argtypes = [vp, i32, ctypes.POINTER(_LayerCache), ctypes.POINTER(_Policy), vp, sz, vp]
    lib.tria_evict_staged.restype = i32
    lib.tria_model_workspace_size.argtypes = [ctypes.POINTER(_LayerCache), i32, i32]
    lib.tria_model_workspace_size.restype = sz
    lib.tria_evict_model.argtypes = [vp, ctypes.POINTER(i32), i32, ctypes.POINTER(_LayerCache),
                                     ctypes.POINTER(_Policy), vp, vp, sz, vp]
    lib.tria_evict_model.restype = i32
    lib.tria_evict_model_fused.argtypes = [vp, ctypes.POINTER(i32), i32, ctypes.POINTER(_LayerCache)]
    lib.tria_evict_model_fused.restype = i32
    lib.tria_evict_layers.argtypes = [vp, ctypes.POINTER(i32), ctypes.POINTER(_LayerCache), ctypes.POINTER(_Policy),
                                      vp, sz, vp]
    lib.tria_evict_layers.restype = i32
    lib.tria_evict_profiled.argtypes = [vp, i32, ctypes.POINTER(_LayerCache), ctypes.POINTER(_Policy), vp, sz,
                                        vp, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(i32)]
    lib.tria_evict_profiled.restype = i32
    lib.tria_evict_marked.argtypes = [vp, i32, ctypes.POINTER(_LayerCache), ctypes.POINTER(_Policy), vp, sz, vp,
                                      ctypes.POINTER(vp)]
    lib.tria_evict_marked.restype = i32
    lib.tria_device_status.argtypes = [vp, vp]
    lib.tria_device_status.restype = i32
    lib.tria_selftest_bounded_wait.argtypes = [i32, vp, sz, vp]
    lib.tria_selftest_bounded_wait.restype = i32
    lib.tria_calib_accumulate.argtypes = [vp, i32, i32, i32, i32, i32, vp, vp]
    lib.tria_calib_accumulate.restype = i32
    lib.tria_calib_finish.argtypes = [vp, i64, i32, i32, i32, vp, vp, vp, vp]
    lib.tria_calib_finish.restype = i32
    lib.tria_shared_combine.argtypes = [vp, i64, i32, ctypes.POINTER(_LayerCache), vp, vp, sz, vp]
    lib.tria_shared_combine.restype = i32
    lib.tria_shared_select.argtypes = [vp, ctypes.POINTER(_LayerCache), ctypes.POINTER(_Policy), vp, vp, sz, vp]
    lib.tria_shared_select.restype = i32
    lib.tria_append.argtypes = [ctypes.POINTER(_LayerCache), vp, vp, vp, vp, vp, i32, vp, sz, vp]
    lib.tria_append.restype = i32
    sch_p, st_p, i32_p = ctypes.POINTER(_Schedule), ctypes.POINTER(_SeqState), ctypes.POINTER(i32)
    lib.tria_schedule_check.argtypes = [sch_p]
    lib.tria_schedule_check.restype = i32
    lib.tria_seq_init.argtypes = [st_p, i64]
    lib.tria_seq_init.restype = i32
    lib.tria_seq_prefill.argtypes = [sch_p, st_p, i64]
    lib.tria_seq_prefill.restype = i32
    lib.tria_seq_decode.argtypes = [sch_p, st_p]
    lib.tria_seq_decode.restype = i32
    lib.tria_schedule_plan.argtypes = [sch_p, st_p, i32, i32_p, i32_p, ctypes.POINTER(i64), i32_p]
    lib.tria_schedule_plan.restype = i32
    lib.tria_schedule_passed.argtypes = [sch_p, st_p, i32]
    lib.tria_schedule_passed.restype = i32
    lib.tria_status_string.argtypes = [i32]
    lib.tria_status_string.restype = ctypes.c_char_p
    lib.tria_workspace_score_offset.argtypes = [ctypes.POINTER(_LayerCache)]
    lib.tria_workspace_score_offset.restype = sz
    lib.tria_version.argtypes = []
    lib.tria_version.restype = i32
    _lib = lib
    return lib


def _check(status: int, where: str):
    if status != OK:
        raise TriaError(status, where)


def _stream_handle(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return ctypes.c_void_p(t)
    if not t.is_cuda:
        raise ValueError("device argument must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("device argument must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _host_array(values, dtype, ctype):
    if values is None:
        return None, None
    arr = np.ascontiguousarray(np.asarray(values, dtype=dtype))
    return arr, arr.ctypes.data_as(ctypes.POINTER(ctype))


# --------------------------------------------------------------------------- host-only helpers

def gate_check(n_q_heads: int, n_kv_heads: int, head_dim: int, nonrot_dim: int = 0) -> int:
    return load_library().tria_gate_check(n_q_heads, n_kv_heads, head_dim, nonrot_dim)


def gate_describe(n_q_heads: int, n_kv_heads: int, head_dim: int, k_type: str = "q8_0",
                  nonrot_dim: int = 0) -> tuple:
    """tria_gate_describe: (status, the gate log line)."""
    buf = ctypes.create_string_buffer(256)
    st = load_library().tria_gate_describe(n_q_heads, n_kv_heads, head_dim, nonrot_dim, DTYPES[k_type], buf, 256)
    return st, buf.value.decode()


def budget_rows(budget_frac: float, n_ctx: int) -> int:
    return load_library().tria_budget_rows(budget_frac, n_ctx)


def should_evict(n_live: int, budget: int, interval: int) -> bool:
    return bool(load_library().tria_should_evict(n_live, budget, interval))


def status_string(status: int) -> str:
    return load_library().tria_status_string(status).decode()


def version() -> int:
    return load_library().tria_version()


# --------------------------------------------------------------------------- stats

class Stats:
    """Device-resident calibration statistics (``tria_load_stats``)."""

    def __init__(self, q_mean, q_abs, *, n_kv_heads: int, head_dim: int = 0, rope_theta: float = 0.0,
                 omega=None, kv_of_q=None, offsets=None, layer_head_dim=None, layer_rope_theta=None,
                 nonrot_dim: int = 0, q_nonrot=None, stream=None):
        """Uniform models: q_mean [L][n_q][rot/2][2], q_abs [L][n_q][rot/2] (or None),
        rot = hd - nonrot_dim the rotary dims; q_nonrot [L][n_q][nonrot_dim] the
        mean non-rotary query (or None: no content term).
        Hybrid models (layer_head_dim given): q_mean / q_abs / omega are lists with
        one array per layer, packed here layer after layer."""
        lib = load_library()
        if layer_head_dim is not None:
            n_layers, n_q = len(q_mean), len(q_mean[0])
            q_mean = np.concatenate([np.asarray(x, np.float32).ravel() for x in q_mean])
            if q_abs is not None:
                q_abs = np.concatenate([np.asarray(x, np.float32).ravel() for x in q_abs])
            if omega is not None:
                omega = np.concatenate([np.asarray(x, np.float64).ravel() for x in omega])
        else:
            q_mean = np.ascontiguousarray(np.asarray(q_mean, dtype=np.float32))
            n_layers, n_q = q_mean.shape[0], q_mean.shape[1]
        self._keep = []
        qm_arr, qm_p = _host_array(q_mean, np.float32, ctypes.c_float)
        qa_arr, qa_p = _host_array(q_abs, np.float32, ctypes.c_float)
        om_arr, om_p = _host_array(omega, np.float64, ctypes.c_double)
        kv_arr, kv_p = _host_array(kv_of_q, np.int32, ctypes.c_int32)
        of_arr, of_p = _host_array(offsets, np.int64, ctypes.c_int64)
        lh_arr, lh_p = _host_array(layer_head_dim, np.int32, ctypes.c_int32)
        lt_arr, lt_p = _host_array(layer_rope_theta, np.float64, ctypes.c_double)
        qn_arr, qn_p = _host_array(q_nonrot, np.float32, ctypes.c_float)
        self._keep += [qm_arr, qa_arr, om_arr, kv_arr, of_arr, lh_arr, lt_arr, qn_arr]
        desc = _StatsDesc(n_layers, n_q, n_kv_heads, head_dim, float(rope_theta), om_p, qm_p, qa_p,
                          kv_p, of_p, 0 if of_arr is None else len(of_arr), lh_p, lt_p, int(nonrot_dim), qn_p)
        handle = ctypes.c_void_p()
        _check(lib.tria_load_stats(ctypes.byref(desc), ctypes.byref(handle), _stream_handle(stream)),
               "tria_load_stats")
        self.handle = handle
        self.n_layers, self.n_q_heads, self.n_kv_heads, self.head_dim = n_layers, n_q, n_kv_heads, head_dim
        self.nonrot_dim = int(nonrot_dim)
        self.group = n_q // n_kv_heads

    def close(self):
        if self.handle:
            load_library().tria_free_stats(self.handle)
            self.handle = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def load_stats(q_mean, q_abs, **kw) -> Stats:
    return Stats(q_mean, q_abs, **kw)


# --------------------------------------------------------------------------- cache / policy

class LayerCache:
    """One layer's cache (``tria_layer_cache``): device tensors + host layout."""

    def __init__(self, *, k, v, pos, n_live, seq_row0, capacity, head_dim: int, n_kv_heads: int,
                 k_type: str = "f16", v_type: str = "f16", k_scale=None, v_scale=None):
        self.k, self.v, self.pos, self.n_live = k, v, pos, n_live
        self.k_scale, self.v_scale = k_scale, v_scale
        self.head_dim, self.n_kv_heads = head_dim, n_kv_heads
        self.k_type, self.v_type = DTYPES[k_type], DTYPES[v_type]
        self.seq_row0 = np.ascontiguousarray(np.asarray(seq_row0, dtype=np.int64))
        self.capacity = np.ascontiguousarray(np.asarray(capacity, dtype=np.int32))

    def c_struct(self) -> _LayerCache:
        return _LayerCache(
            len(self.seq_row0), self.n_kv_heads, self.head_dim, self.k_type, self.v_type,
            _ptr(self.k), _ptr(self.k_scale), _ptr(self.v), _ptr(self.v_scale), _ptr(self.pos),
            _ptr(self.n_live), self.seq_row0.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
            self.capacity.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)))


class Policy:
    """Eviction policy (``tria_policy``)."""

    def __init__(self, *, budget_frac: float = 0.0, n_ctx=None, budget_rows=None, window: int = 512,
                 sink: int = 0, interval: int = 128, cur_pos=None, sink_rows=None):
        self.budget_frac, self.window, self.sink, self.interval = budget_frac, window, sink, interval
        self.n_ctx, self._n_ctx_p = _host_array(n_ctx, np.int32, ctypes.c_int32)
        self.budget_rows, self._br_p = _host_array(budget_rows, np.int32, ctypes.c_int32)
        self.cur_pos, self._cp_p = _host_array(cur_pos, np.int64, ctypes.c_int64)
        self.sink_rows, self._sr_p = _host_array(sink_rows, np.int32, ctypes.c_int32)

    def c_struct(self) -> _Policy:
        return _Policy(float(self.budget_frac), self._n_ctx_p, self._br_p, self.window, self.sink,
                       self.interval, self._cp_p, self._sr_p)


# --------------------------------------------------------------------------- the pass

def workspace_size(cache: LayerCache, group: int) -> int:
    c = cache.c_struct()
    n = load_library().tria_workspace_size(ctypes.byref(c), group)
    if n == 0:
        raise TriaError(ERR_INVALID_ARG, "tria_workspace_size")
    return n


def workspace_scores(ws, cache: LayerCache):
    """tria_workspace_score_offset: the workspace's float view of the z-max
    scores the staged evict path selected with (valid after evict_staged for
    the live rows of segments above their budget)."""
    c = cache.c_struct()
    off = load_library().tria_workspace_score_offset(ctypes.byref(c))
    if off == 0:
        raise TriaError(ERR_INVALID_ARG, "tria_workspace_score_offset")
    rows = int(max(r0 + cache.n_kv_heads * cp for r0, cp in zip(cache.seq_row0, cache.capacity)))
    return ws[off:off + 4 * rows].view(__import__("torch").float32)


def workspace_init(ws, stream=None):
    _check(load_library().tria_workspace_init(_ptr(ws), ws.numel() * ws.element_size(),
                                              _stream_handle(stream)), "tria_workspace_init")


def _ws(ws):
    return _ptr(ws), ws.numel() * ws.element_size()


def score(stats: Stats, layer: int, cache: LayerCache, policy: Policy, score_out, raw_out=None,
          *, ws, stream=None):
    c, p = cache.c_struct(), policy.c_struct()
    wp, wb = _ws(ws)
    _check(load_library().tria_score(stats.handle, layer, ctypes.byref(c), ctypes.byref(p),
                                     _ptr(score_out), _ptr(raw_out), wp, wb, _stream_handle(stream)),
           "tria_score")


def select(score_in, cache: LayerCache, policy: Policy, keep_out, *, ws, stream=None):
    c, p = cache.c_struct(), policy.c_struct()
    wp, wb = _ws(ws)
    _check(load_library().tria_select(_ptr(score_in), ctypes.byref(c), ctypes.byref(p), _ptr(keep_out),
                                      wp, wb, _stream_handle(stream)), "tria_select")


def select_noalloc(score_in, cache: LayerCache, policy: Policy, keep_out, *, stream=None):
    """tria_select_noalloc: tria_select with the library's fixed scratch array
    instead of a workspace (for callers that cannot allocate)."""
    c, p = cache.c_struct(), policy.c_struct()
    _check(load_library().tria_select_noalloc(_ptr(score_in), ctypes.byref(c), ctypes.byref(p), _ptr(keep_out),
                                              _stream_handle(stream)), "tria_select_noalloc")


def compact(cache: LayerCache, policy: Policy, keep, *, ws, stream=None):
    c, p = cache.c_struct(), policy.c_struct()
    wp, wb = _ws(ws)
    _check(load_library().tria_compact(ctypes.byref(c), ctypes.byref(p), _ptr(keep), wp, wb,
                                       _stream_handle(stream)), "tria_compact")


def evict(stats: Stats, layer: int, cache: LayerCache, policy: Policy, *, ws, stream=None):
    c, p = cache.c_struct(), policy.c_struct()
    wp, wb = _ws(ws)
    _check(load_library().tria_evict(stats.handle, layer, ctypes.byref(c), ctypes.byref(p), wp, wb,
                                     _stream_handle(stream)), "tria_evict")


def evict_staged(stats: Stats, layer: int, cache: LayerCache, policy: Policy, *, ws, stream=None):
    """tria_evict_staged: the pass as three kernels (score, select, compact)."""
    c, p = cache.c_struct(), policy.c_struct()
    wp, wb = _ws(ws)
    _check(load_library().tria_evict_staged(stats.handle, layer, ctypes.byref(c), ctypes.byref(p), wp, wb,
                                            _stream_handle(stream)), "tria_evict_staged")


def model_workspace_size(cache: LayerCache, n_layers: int, group: int) -> int:
    c = cache.c_struct()
    n = load_library().tria_model_workspace_size(ctypes.byref(c), n_layers, group)
    if n == 0:
        raise TriaError(ERR_INVALID_ARG, "tria_model_workspace_size")
    return n


def evict_model(stats: Stats, layers, caches, policy: Policy, *, ws, score_out=None, stream=None):
    """tria_evict_model: one pass over several layers (caches[i] is the cache
    of layer layers[i]); score_out (optional device float tensor) receives the
    z-max scores of the compacted segments' live rows, [n_layers][layer rows]."""
    if len(caches) != len(layers) or not caches:
        raise ValueError("one cache per layer")
    structs = (_LayerCache * len(caches))(*[c.c_struct() for c in caches])
    arr, ptr = _host_array(layers, np.int32, ctypes.c_int32)
    p = policy.c_struct()
    wp, wb = _ws(ws)
    _check(load_library().tria_evict_model(stats.handle, ptr, len(layers), structs, ctypes.byref(p),
                                           _ptr(score_out) if score_out is not None else None, wp, wb,
                                           _stream_handle(stream)), "tria_evict_model")


def evict_model_fused(stats: Stats, layers, caches) -> bool:
    """tria_evict_model_fused: whether tria_evict_model (without score_out)
    runs these layers as one fused kernel (True) or as the staged kernels per
    layer (False). Host only."""
    if len(caches) != len(layers) or not caches:
        raise ValueError("one cache per layer")
    structs = (_LayerCache * len(caches))(*[c.c_struct() for c in caches])
    arr, ptr = _host_array(layers, np.int32, ctypes.c_int32)
    r = load_library().tria_evict_model_fused(stats.handle, ptr, len(layers), structs)
    if r < 0:
        raise TriaError(ERR_INVALID_ARG, "tria_evict_model_fused")
    return r == 1


def evict_layers(stats: Stats, layer_of_seq, cache: LayerCache, policy: Policy, *, ws, stream=None):
    """tria_evict_layers: one pass over sequences of several layers (sequence s
    scored with the statistics of layer layer_of_seq[s])."""
    c, p = cache.c_struct(), policy.c_struct()
    wp, wb = _ws(ws)
    arr, ptr = _host_array(layer_of_seq, np.int32, ctypes.c_int32)
    if arr is None or len(arr) != len(cache.seq_row0):
        raise ValueError("one layer per sequence")
    _check(load_library().tria_evict_layers(stats.handle, ptr, ctypes.byref(c), ctypes.byref(p), wp, wb,
                                            _stream_handle(stream)), "tria_evict_layers")


def evict_profiled(stats: Stats, layer: int, cache: LayerCache, policy: Policy, *, ws, stream=None):
    """tria_evict_profiled: returns ({stage: ms}, kernels launched); synchronises."""
    c, p = cache.c_struct(), policy.c_struct()
    wp, wb = _ws(ws)
    ms = (ctypes.c_float * 5)()
    nl = ctypes.c_int32()
    _check(load_library().tria_evict_profiled(stats.handle, layer, ctypes.byref(c), ctypes.byref(p), wp, wb,
                                              _stream_handle(stream), ms, ctypes.byref(nl)),
           "tria_evict_profiled")
    names = ("score", "zscore", "select", "compact", "total")
    return dict(zip(names, list(ms))), nl.value


def evict_marked(stats: Stats, layer: int, cache: LayerCache, policy: Policy, events, *, ws, stream=None):
    """tria_evict_marked: the pass with four torch.cuda.Event (timing) recorded
    before, between and after its kernels; no synchronisation (capturable)."""
    c, p = cache.c_struct(), policy.c_struct()
    wp, wb = _ws(ws)
    if len(events) != 4:
        raise ValueError("four events")
    handles = (ctypes.c_void_p * 4)(*[ctypes.c_void_p(int(e.cuda_event)) for e in events])
    _check(load_library().tria_evict_marked(stats.handle, layer, ctypes.byref(c), ctypes.byref(p), wp, wb,
                                            _stream_handle(stream), handles), "tria_evict_marked")


def device_status(ws, stream=None) -> int:
    return load_library().tria_device_status(_ptr(ws), _stream_handle(stream))


def selftest_bounded_wait(spin_limit: int, ws, stream=None) -> int:
    wp, wb = _ws(ws)
    return load_library().tria_selftest_bounded_wait(spin_limit, wp, wb, _stream_handle(stream))


def calib_accumulate(q, acc, *, nonrot_dim: int = 0, stream=None):
    """tria_calib_accumulate: add the sums of a batch of pre-RoPE queries
    q[tokens][heads][head_dim] (float32 or float16 CUDA tensor) to acc
    (float64 CUDA tensor [heads][head_dim/2][3], zeroed before the first batch);
    the last nonrot_dim dims of each head are the non-rotary ones."""
    import torch
    if q.dim() != 3:
        raise ValueError("q must be [tokens][heads][head_dim]")
    t, h, hd = q.shape
    qt = {torch.float32: F32, torch.float16: F16}.get(q.dtype)
    if qt is None:
        raise ValueError("q must be float32 or float16")
    if acc.dtype != torch.float64 or tuple(acc.shape) != (h, hd // 2, 3):
        raise ValueError("acc must be float64 [heads][head_dim/2][3]")
    qp = _ptr(q) if t > 0 else None
    _check(load_library().tria_calib_accumulate(qp, qt, t, h, hd, nonrot_dim, _ptr(acc), _stream_handle(stream)),
           "tria_calib_accumulate")


def calib_finish(acc, n_tokens: int, *, nonrot_dim: int = 0, stream=None):
    """tria_calib_finish: (q_mean [heads][rot/2][2], q_abs [heads][rot/2]) float32
    CUDA tensors, rot = head_dim - nonrot_dim; with nonrot_dim > 0 also the mean
    non-rotary query [heads][nonrot_dim] as a third element."""
    import torch
    h, fc, _ = acc.shape
    fcr = fc - nonrot_dim // 2
    q_mean = torch.empty((h, fcr, 2), dtype=torch.float32, device=acc.device)
    q_abs = torch.empty((h, fcr), dtype=torch.float32, device=acc.device)
    q_nonrot = torch.empty((h, nonrot_dim), dtype=torch.float32, device=acc.device) if nonrot_dim else None
    _check(load_library().tria_calib_finish(_ptr(acc), n_tokens, h, 2 * fc, nonrot_dim, _ptr(q_mean), _ptr(q_abs),
                                            _ptr(q_nonrot) if q_nonrot is not None else None,
                                            _stream_handle(stream)), "tria_calib_finish")
    return (q_mean, q_abs) if not nonrot_dim else (q_mean, q_abs, q_nonrot)


# --------------------------------------------------------------------------- shared-slot variant

def shared_combine(scores, cache: LayerCache, combined, *, ws, stream=None):
    """tria_shared_combine: scores float32 CUDA tensor [layers][rows] (tria_score output per layer)."""
    rows = int(max(r0 + cache.n_kv_heads * c for r0, c in zip(cache.seq_row0, cache.capacity)))
    if scores.dim() != 2 or scores.stride(1) != 1 or scores.shape[1] < rows:
        raise ValueError("scores must be [layers][rows] (rows contiguous, at least the cache layout's rows)")
    c = cache.c_struct()
    wp, wb = _ws(ws)
    _check(load_library().tria_shared_combine(_ptr(scores), scores.stride(0), scores.shape[0], ctypes.byref(c),
                                              _ptr(combined), wp, wb, _stream_handle(stream)),
           "tria_shared_combine")


def shared_select(combined, cache: LayerCache, policy: Policy, keep_out, *, ws, stream=None):
    """tria_shared_select: one keep list per sequence, written to every KV head's slot."""
    c, p = cache.c_struct(), policy.c_struct()
    wp, wb = _ws(ws)
    _check(load_library().tria_shared_select(_ptr(combined), ctypes.byref(c), ctypes.byref(p), _ptr(keep_out),
                                             wp, wb, _stream_handle(stream)), "tria_shared_select")


# --------------------------------------------------------------------------- decode-loop lifecycle

def append(cache: LayerCache, k_new, v_new, pos_new, *, ws, k_scale_new=None, v_scale_new=None, stream=None):
    """tria_append: rows k_new / v_new [n_seqs][n_kv_heads][n_tokens][...] (cache dtypes) and
    pos_new int32 [n_seqs][n_tokens] after the live rows of every segment; n_live += n_tokens."""
    n_seqs = len(cache.seq_row0)
    if pos_new.dim() != 2 or pos_new.shape[0] != n_seqs or pos_new.dtype.itemsize != 4:
        raise ValueError("pos_new must be int32 [n_seqs][n_tokens]")
    n_tokens = int(pos_new.shape[-1])
    row_bytes = {F32: 4, F16: 2, Q8_0: 1}
    for name, t, dt in (("k_new", k_new, cache.k_type), ("v_new", v_new, cache.v_type)):
        want = n_seqs * cache.n_kv_heads * n_tokens * cache.head_dim * row_bytes[dt]
        if t is None or not t.is_contiguous() or t.numel() * t.element_size() != want:
            raise ValueError(f"{name} must be contiguous [n_seqs][n_kv_heads][n_tokens][head_dim] rows of the cache type")
    c = cache.c_struct()
    wp, wb = _ws(ws)
    _check(load_library().tria_append(ctypes.byref(c), _ptr(k_new), _ptr(k_scale_new), _ptr(v_new),
                                      _ptr(v_scale_new), _ptr(pos_new), n_tokens, wp, wb,
                                      _stream_handle(stream)), "tria_append")


class Schedule:
    """Decode-loop schedule (``tria_schedule``)."""

    def __init__(self, *, trigger: int = TRIGGER_LENGTH, kv_budget: int = 0, divide_length: int = 128,
                 count_prompt_tokens: bool = True, protect_prefill: bool = True, sink: int = 0,
                 window: int = 0, budget_frac: float = 0.0, n_ctx: int = 0):
        self.c = _Schedule(int(trigger), int(bool(count_prompt_tokens)), int(bool(protect_prefill)), int(sink),
                           int(window), 0, int(kv_budget), int(divide_length), float(budget_frac), int(n_ctx))
        _check(load_library().tria_schedule_check(ctypes.byref(self.c)), "tria_schedule_check")

    @property
    def window(self) -> int:
        return self.c.window


class Sequences:
    """The ``tria_seq_state`` of every sequence of a loop (host memory)."""

    def __init__(self, schedule: Schedule, capacity):
        self.schedule = schedule
        self.n = len(capacity)
        self.st = (_SeqState * self.n)()
        for s, cap in enumerate(capacity):
            _check(load_library().tria_seq_init(ctypes.byref(self.st[s]), int(cap)), "tria_seq_init")

    def prefill(self, s: int, n_tokens: int):
        _check(load_library().tria_seq_prefill(ctypes.byref(self.schedule.c), ctypes.byref(self.st[s]),
                                               int(n_tokens)), "tria_seq_prefill")

    def decode(self, s: int) -> bool:
        _check(load_library().tria_seq_decode(ctypes.byref(self.schedule.c), ctypes.byref(self.st[s])),
               "tria_seq_decode")
        return bool(self.st[s].due)

    def plan(self):
        """tria_schedule_plan: (budget_rows, sink_rows, cur_pos, n_due)."""
        b = np.zeros(self.n, np.int32)
        k = np.zeros(self.n, np.int32)
        p = np.zeros(self.n, np.int64)
        nd = ctypes.c_int32()
        i32p = ctypes.POINTER(ctypes.c_int32)
        _check(load_library().tria_schedule_plan(ctypes.byref(self.schedule.c), self.st, self.n,
                                                 b.ctypes.data_as(i32p), k.ctypes.data_as(i32p),
                                                 p.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                                 ctypes.byref(nd)), "tria_schedule_plan")
        return b, k, p, nd.value

    def policy(self) -> tuple:
        """(Policy of the planned pass, sequences due)."""
        b, k, p, nd = self.plan()
        return Policy(budget_rows=b, sink_rows=k, cur_pos=p, window=self.schedule.window,
                      sink=self.schedule.c.sink), nd

    def passed(self):
        _check(load_library().tria_schedule_passed(ctypes.byref(self.schedule.c), self.st, self.n),
               "tria_schedule_passed")

    def state(self, s: int) -> dict:
        return {name: getattr(self.st[s], name) for name, _ in _SeqState._fields_ if name != "pad"}


def raw_call(name: str, *args):
    """Call an entry point by name with ctypes arguments (used by the host tests)."""
    return getattr(load_library(), name)(*args)
