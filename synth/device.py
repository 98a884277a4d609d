"""Device form of the seeded cache generator (``libtria_synth.so``).

Builds the library with nvcc (sm_103a), fills a layer's cache on the GPU with
the same bits :func:`synth.workloads.segment_host` produces on the host, and
allocates whole-layer tensors for a workload. Test / benchmark infrastructure.
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess

import numpy as np

from . import workloads as W

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_HERE, "csrc", "synth_gen.cu")
LIB = os.path.join(_HERE, "libtria_synth.so")
_lib = None


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
           "-Xcompiler", "-fPIC", "-shared", SRC, "-o", LIB + ".tmp"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed on {SRC}:\n{res.stdout}\n{res.stderr}")
    os.replace(LIB + ".tmp", LIB)
    return LIB


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise RuntimeError(f"{LIB} not built")
        lib = ctypes.CDLL(LIB)
        vp, i32 = ctypes.c_void_p, ctypes.c_int
        lib.synth_fill_layer.argtypes = [i32, i32, i32, i32, i32, i32, i32,
                                         ctypes.POINTER(ctypes.c_longlong), ctypes.POINTER(ctypes.c_int),
                                         vp, vp, vp, vp, vp, i32, vp]
        lib.synth_fill_layer.restype = i32
        _lib = lib
    return _lib


_KT = {"f32": 0, "f16": 1, "q8_0": 2}


def alloc_layer(w: W.Workload, device="cuda"):
    """Empty device tensors for one layer of workload ``w`` (16-byte aligned planes)."""
    import torch
    rows, hd = w.total_rows(), w.head_dim
    kdt = {"f32": torch.float32, "f16": torch.float16, "q8_0": torch.int8}[w.k_type]
    vdt = {"f32": torch.float32, "f16": torch.float16}[w.v_type]
    out = {
        "k": torch.empty((rows, hd), dtype=kdt, device=device),
        "k_scale": (torch.empty((rows, hd // 32), dtype=torch.float16, device=device)
                    if w.k_type == "q8_0" else None),
        "v": torch.empty((rows, hd), dtype=vdt, device=device),
        "pos": torch.empty(rows, dtype=torch.int32, device=device),
        "n_live": torch.tensor(w.n_live, dtype=torch.int32, device=device),
    }
    return out


def fill_layer(w: W.Workload, layer: int, t: dict, stream=None):
    """Fill tensors from :func:`alloc_layer` with layer ``layer`` of ``w``."""
    import torch
    if w.host_keys_pre_rope or w.pos_kind != "arange":
        # small / host-defined parts: copy what the host builds
        if w.host_keys_pre_rope:
            h = W.layer_host(w, layer)
            t["k"].copy_(torch.from_numpy(h["k"]))
            t["v"].copy_(torch.from_numpy(h["v"]))
            t["pos"].copy_(torch.from_numpy(h["pos"]))
            t["n_live"].copy_(torch.from_numpy(h["n_live"]))
            return
    lib = _load()
    scale = torch.from_numpy(W.pair_scales(w, layer)).to(t["k"].device)
    row0 = np.ascontiguousarray(w.seq_row0(), dtype=np.int64)
    cap = np.ascontiguousarray(np.asarray(w.capacity, dtype=np.int32))
    st = torch.cuda.current_stream() if stream is None else stream
    err = lib.synth_fill_layer(
        w.n_seqs, w.n_kv_heads, w.head_dim, _KT[w.k_type], _KT[w.v_type], w.layer_seed(layer), layer,
        row0.ctypes.data_as(ctypes.POINTER(ctypes.c_longlong)),
        cap.ctypes.data_as(ctypes.POINTER(ctypes.c_int)),
        ctypes.c_void_p(scale.data_ptr()), ctypes.c_void_p(t["k"].data_ptr()),
        ctypes.c_void_p(t["k_scale"].data_ptr() if t["k_scale"] is not None else 0),
        ctypes.c_void_p(t["v"].data_ptr()), ctypes.c_void_p(t["pos"].data_ptr()),
        1 if w.pos_kind == "arange" else 0, ctypes.c_void_p(st.cuda_stream))
    if err != 0:
        raise RuntimeError(f"synth_fill_layer failed with CUDA error {err}")
    if w.pos_kind != "arange":
        pos = np.concatenate([W.segment_positions(w, layer, s, g) for s, g, *_ in w.segments()])
        t["pos"].copy_(torch.from_numpy(pos))
    t["n_live"].copy_(torch.tensor(w.n_live, dtype=torch.int32))
    scale.record_stream(st) if hasattr(scale, "record_stream") else None
    torch.cuda.current_stream().synchronize()
