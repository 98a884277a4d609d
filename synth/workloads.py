"""The five synthetic workloads and their host-side builders.

The shapes follow the workloads the eviction pages run on (Qwen3-8B: 36 layers,
8 KV heads, 32 query heads, head_dim 128; a Qwen3.5-style hd-256 model with 4 KV
heads and 16 query heads) with synthetic contents: no weights or datasets are
involved.

Cache layout (shared with the C ABI): one layer's cache is a stack of rows.
Sequence ``s`` owns ``n_kv_heads * capacity[s]`` rows starting at
``seq_row0[s]``; KV head ``g`` of it (one *segment*) starts at row
``seq_row0[s] + g * capacity[s]``. Row ``r`` of a segment holds the RoPE-rotated
key (``[head_dim]``), value (``[head_dim]``) and absolute position (int32) of
one cached token; rows ascend in position.

Contents
--------
* Keys of workloads 2-5 come from :mod:`synth.counter_rng` directly in the
  rotated frame: each (dim f, dim f+hd/2) pair is an isotropic 2-D draw, and a
  rotation leaves an isotropic law unchanged, so the rotated keys have the same
  distribution as rotated pre-RoPE keys. Eight random frequency pairs per KV
  head are scaled by 8 (outliers) where the workload says so.
* Workload 1 keys are pre-RoPE float32 N(0,1) (numpy PCG64, seed 0) rotated on
  the host in float64 at positions 0..511 and rounded to float32, the way a
  model writes its cache; the pre-RoPE keys are kept for identity tests.
* Calibration statistics: complex mean query per (layer, query head, pair)
  ~ N(0,1) on each component, and the mean-resultant residual
  ``q_abs - |q_mean|`` = 0.5|N(0,1)|; workloads 2-5 scale both by 1/(1+f).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import counter_rng as crng

OUTLIER_SCALE = 8.0


@dataclass(frozen=True)
class Workload:
    name: str
    description: str
    n_layers: int
    n_kv_heads: int
    group: int
    head_dim: int
    rope_theta: float
    k_type: str            # 'f32' | 'f16' | 'q8_0'
    v_type: str            # 'f32' | 'f16'
    n_live: tuple          # live rows per sequence
    capacity: tuple        # physical rows per segment, per sequence
    cur_pos: tuple         # absolute decode position per sequence
    n_ctx: tuple           # context length the budget fraction refers to
    budget_frac: float
    window: int
    sink: int
    interval: int
    key_seed: int
    key_seed_stride: int   # layer l uses key_seed + l * key_seed_stride
    stats_seed: int
    n_outlier_pairs: int
    stats_decay: bool
    pos_kind: str          # 'arange' | 'steady'
    host_keys_pre_rope: bool = False

    @property
    def n_seqs(self) -> int:
        return len(self.n_live)

    @property
    def n_q_heads(self) -> int:
        return self.n_kv_heads * self.group

    @property
    def fc(self) -> int:
        return self.head_dim // 2

    def seq_row0(self) -> np.ndarray:
        out, acc = [], 0
        for cap in self.capacity:
            out.append(acc)
            acc += self.n_kv_heads * cap
        return np.asarray(out, dtype=np.int64)

    def total_rows(self) -> int:
        return int(sum(self.n_kv_heads * c for c in self.capacity))

    def layer_seed(self, layer: int) -> int:
        return self.key_seed + layer * self.key_seed_stride

    def k_row_bytes(self) -> int:
        return {"f32": 4 * self.head_dim, "f16": 2 * self.head_dim,
                "q8_0": self.head_dim + self.head_dim // 16}[self.k_type]

    def v_row_bytes(self) -> int:
        return {"f32": 4, "f16": 2}[self.v_type] * self.head_dim

    def segments(self):
        """(seq, head, first_row, capacity, n_live) for every segment."""
        r0 = self.seq_row0()
        for s in range(self.n_seqs):
            for g in range(self.n_kv_heads):
                yield s, g, int(r0[s] + g * self.capacity[s]), self.capacity[s], self.n_live[s]

    def total_live(self) -> int:
        return int(sum(self.n_kv_heads * n for n in self.n_live)) * self.n_layers


def _ragged_lengths(seed: int, n: int, lo: int, hi: int) -> tuple:
    rng = np.random.default_rng(seed)
    return tuple(int(x) for x in rng.integers(lo, hi, size=n, endpoint=True))


_W5_LEN = _ragged_lengths(5, 8, 32768, 131072)

WORKLOADS = {
    "tiny": Workload(
        name="tiny",
        description="1 layer, 2 KV heads, G=4, hd 64, theta 1e4, 512 fp32 rows, pos 512, 50% budget",
        n_layers=1, n_kv_heads=2, group=4, head_dim=64, rope_theta=1e4,
        k_type="f32", v_type="f32", n_live=(512,), capacity=(512,), cur_pos=(512,), n_ctx=(512,),
        budget_frac=0.5, window=64, sink=4, interval=128,
        key_seed=0, key_seed_stride=0, stats_seed=1, n_outlier_pairs=0, stats_decay=False,
        pos_kind="arange", host_keys_pre_rope=True),
    "qwen3_8b_layer": Workload(
        name="qwen3_8b_layer",
        description="Qwen3-8B single layer: 8 KV heads, 32 q heads, hd 128, 32768 fp16 rows, 25% budget",
        n_layers=1, n_kv_heads=8, group=4, head_dim=128, rope_theta=1e6,
        k_type="f16", v_type="f16", n_live=(32768,), capacity=(32768,), cur_pos=(32768,),
        n_ctx=(32768,), budget_frac=0.25, window=512, sink=4, interval=128,
        key_seed=2, key_seed_stride=0, stats_seed=2, n_outlier_pairs=8, stats_decay=True,
        pos_kind="arange"),
    "qwen3_8b_full": Workload(
        name="qwen3_8b_full",
        description="Qwen3-8B 36 layers steady state: capacity 12288, 6144+128 live rows -> 6144",
        n_layers=36, n_kv_heads=8, group=4, head_dim=128, rope_theta=1e6,
        k_type="f16", v_type="f16", n_live=(6272,), capacity=(12288,), cur_pos=(32768,),
        n_ctx=(12288,), budget_frac=0.5, window=512, sink=0, interval=128,
        key_seed=300, key_seed_stride=1, stats_seed=3, n_outlier_pairs=8, stats_decay=True,
        pos_kind="steady"),
    "q8_0": Workload(
        name="q8_0",
        description="Qwen3-8B shapes, 36 layers, 65536 rows, q8_0 keys, fp16 values, 50% budget",
        n_layers=36, n_kv_heads=8, group=4, head_dim=128, rope_theta=1e6,
        k_type="q8_0", v_type="f16", n_live=(65536,), capacity=(65536,), cur_pos=(65536,),
        n_ctx=(65536,), budget_frac=0.5, window=512, sink=4, interval=128,
        key_seed=4, key_seed_stride=0, stats_seed=4, n_outlier_pairs=0, stats_decay=True,
        pos_kind="arange"),
    "batched_long": Workload(
        name="batched_long",
        description="8 ragged sequences 32K-128K, 48 layers, 4 KV heads, 16 q heads, hd 256, theta 1e7",
        n_layers=48, n_kv_heads=4, group=4, head_dim=256, rope_theta=1e7,
        k_type="f16", v_type="f16", n_live=_W5_LEN, capacity=_W5_LEN, cur_pos=_W5_LEN,
        n_ctx=_W5_LEN, budget_frac=0.25, window=1024, sink=4, interval=128,
        key_seed=500, key_seed_stride=1, stats_seed=5, n_outlier_pairs=8, stats_decay=True,
        pos_kind="arange"),
}


def get_workload(name: str) -> Workload:
    return WORKLOADS[name]


# ---------------------------------------------------------------------------
# calibration statistics (host only; copied to the device by the caller)
# ---------------------------------------------------------------------------

def make_stats(w: Workload):
    """``(q_mean float32 [L][Hq][fc][2], q_abs float32 [L][Hq][fc])``."""
    rng = np.random.default_rng(w.stats_seed)
    L, hq, fc = w.n_layers, w.n_q_heads, w.fc
    decay = (1.0 / (1.0 + np.arange(fc))) if w.stats_decay else np.ones(fc)
    qm = rng.standard_normal((L, hq, fc, 2)) * decay[None, None, :, None]
    resid = 0.5 * np.abs(rng.standard_normal((L, hq, fc))) * decay[None, None, :]
    qm32 = qm.astype(np.float32)
    mag = np.hypot(qm32[..., 0].astype(np.float64), qm32[..., 1].astype(np.float64))
    q_abs = (mag + resid).astype(np.float32)
    return qm32, q_abs


# ---------------------------------------------------------------------------
# per-segment contents
# ---------------------------------------------------------------------------

def pair_scales(w: Workload, layer: int) -> np.ndarray:
    """float32 ``[n_kv_heads][fc]``: 8 on the outlier pairs of each KV head, else 1."""
    out = np.ones((w.n_kv_heads, w.fc), dtype=np.float32)
    if w.n_outlier_pairs:
        rng = np.random.default_rng((w.layer_seed(layer), 0xA5))
        for g in range(w.n_kv_heads):
            out[g, rng.choice(w.fc, w.n_outlier_pairs, replace=False)] = OUTLIER_SCALE
    return out


def segment_positions(w: Workload, layer: int, seq: int, head: int) -> np.ndarray:
    """int32 ``[capacity]`` positions; rows at or past n_live hold -1 (steady) or r."""
    cap, n, p = w.capacity[seq], w.n_live[seq], w.cur_pos[seq]
    if w.pos_kind == "arange":
        return np.arange(cap, dtype=np.int32)
    # steady state after earlier passes: n-128 surviving positions below p-128,
    # then the 128 tokens decoded since the last pass.
    rng = np.random.default_rng((w.layer_seed(layer), 0x5EED, seq, head))
    older = np.sort(rng.choice(p - 128, n - 128, replace=False))
    out = np.full(cap, -1, dtype=np.int32)
    out[:n - 128] = older
    out[n - 128:n] = np.arange(p - 128, p)
    return out


def _rope_host(x_pre: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """Model-side NEOX RoPE of float32 rows at integer positions, in float64."""
    hd = x_pre.shape[-1]
    fc = hd // 2
    inv = theta ** (-2.0 * np.arange(fc) / hd)
    ang = pos.astype(np.float64)[:, None] * inv[None, :]
    c, s = np.cos(ang), np.sin(ang)
    a = x_pre[:, :fc].astype(np.float64)
    b = x_pre[:, fc:].astype(np.float64)
    return np.concatenate([a * c - b * s, a * s + b * c], axis=1)


def tiny_pre_rope(w: Workload):
    """Workload-1 pre-RoPE float32 keys and values, ``[L][S][G][cap][hd]``."""
    shape = (w.n_layers, w.n_seqs, w.n_kv_heads, w.capacity[0], w.head_dim)
    k_pre = np.random.default_rng(w.key_seed).standard_normal(shape).astype(np.float32)
    v = np.random.default_rng(w.key_seed + 1000).standard_normal(shape).astype(np.float32)
    return k_pre, v


def segment_host(w: Workload, layer: int, seq: int, head: int, rows: int | None = None, values: bool = True):
    """Host twin of one segment's contents.

    Returns a dict with ``k`` (float32/float16 ``[rows, hd]``, or int8 codes for
    q8_0), ``k_scale`` (float16 ``[rows, hd/32]``, q8_0 only), ``v`` (None when
    ``values`` is false: keys only) and ``pos`` - bit-identical to what the
    device generator writes.
    """
    cap = w.capacity[seq]
    rows = cap if rows is None else rows
    pos = segment_positions(w, layer, seq, head)[:rows]
    if w.host_keys_pre_rope:
        k_pre, v = tiny_pre_rope(w)
        k = _rope_host(k_pre[layer, seq, head, :rows], pos, w.rope_theta).astype(np.float32)
        return {"k": k, "k_scale": None, "v": v[layer, seq, head, :rows].copy(), "pos": pos}
    seed = w.layer_seed(layer)
    kkey = crng.stream_key(seed, crng.TENSOR_K, layer, seq, head)
    vkey = crng.stream_key(seed, crng.TENSOR_V, layer, seq, head)
    scale = pair_scales(w, layer)[head]
    kx = crng.segment_values(kkey, rows, w.head_dim, scale)
    vx = crng.segment_values(vkey, rows, w.head_dim, None) if values else None
    out = {"pos": pos, "k_scale": None}
    if w.k_type == "f16":
        out["k"] = crng.to_f16(kx)
    elif w.k_type == "f32":
        out["k"] = kx
    else:
        out["k"], out["k_scale"] = crng.quantize_q8_0(kx)
    if vx is None:
        out["v"] = None
    else:
        out["v"] = crng.to_f16(vx) if w.v_type == "f16" else vx
    return out


def layer_host(w: Workload, layer: int):
    """Whole-layer cache on the host in the global-row layout (small workloads)."""
    total = w.total_rows()
    hd = w.head_dim
    kdt = {"f32": np.float32, "f16": np.float16, "q8_0": np.int8}[w.k_type]
    vdt = {"f32": np.float32, "f16": np.float16}[w.v_type]
    k = np.zeros((total, hd), dtype=kdt)
    ks = np.zeros((total, hd // 32), dtype=np.float16) if w.k_type == "q8_0" else None
    v = np.zeros((total, hd), dtype=vdt)
    pos = np.zeros(total, dtype=np.int32)
    for s, g, r0, cap, _n in w.segments():
        seg = segment_host(w, layer, s, g)
        k[r0:r0 + cap] = seg["k"]
        if ks is not None:
            ks[r0:r0 + cap] = seg["k_scale"]
        v[r0:r0 + cap] = seg["v"]
        pos[r0:r0 + cap] = seg["pos"]
    return {"k": k, "k_scale": ks, "v": v, "pos": pos,
            "n_live": np.asarray(w.n_live, dtype=np.int32),
            "seq_row0": w.seq_row0(), "capacity": np.asarray(w.capacity, dtype=np.int32)}

