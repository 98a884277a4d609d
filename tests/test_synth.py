"""Host-side checks of the seeded input generator (no eviction arithmetic here)."""
import numpy as np

from synth import counter_rng as C
from synth import workloads as W


def test_splitmix64_reference_values():
    # SplitMix64 seeded with 0: the first outputs are published reference values.
    assert C.words(0, np.arange(3, dtype=np.uint64)).tolist() == [
        0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_normal12_moments_and_exactness():
    x = C.normal12(C.stream_key(7, C.TENSOR_K, 0, 0, 0), 0, 1 << 18)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    assert x.min() >= -6.0 and x.max() <= 6.0
    # every value is an integer multiple of 2^-16 (exactly representable)
    assert np.all((x * 65536.0) == np.round(x * 65536.0))
    # counter-based: any sub-range regenerates identically
    y = C.normal12(C.stream_key(7, C.TENSOR_K, 0, 0, 0), 1000, 24)
    np.testing.assert_array_equal(y, x[1000:1024])


def test_stream_keys_differ_per_segment():
    keys = {C.stream_key(2, t, l, s, g) for t in (1, 2) for l in range(3)
            for s in range(2) for g in range(8)}
    assert len(keys) == 2 * 3 * 2 * 8


def test_q8_0_quantiser_error_bound():
    x = C.segment_values(C.stream_key(4, C.TENSOR_K, 0, 0, 0), 64, 128, None)
    qs, d = C.quantize_q8_0(x)
    d32 = (np.abs(x.reshape(64, 4, 32)).max(axis=2) / np.float32(127)).astype(np.float32)
    back = qs.reshape(64, 4, 32).astype(np.float64) * d32[:, :, None]
    assert np.all(np.abs(back - x.reshape(64, 4, 32)) <= d32[:, :, None] * 0.5 + 1e-12)
    assert np.abs(qs).max() == 127
    assert d.dtype == np.float16


def test_workload_layout_and_budgets():
    w = W.get_workload("qwen3_8b_full")
    assert w.total_rows() == 8 * 12288
    segs = list(w.segments())
    assert segs[3][2] == 3 * 12288 and segs[3][4] == 6272
    pos = W.segment_positions(w, 0, 0, 0)
    assert np.all(np.diff(pos[:6272]) > 0) and pos[6271] == 32767 and pos[6272] == -1
    w5 = W.get_workload("batched_long")
    assert len(w5.n_live) == 8 and all(32768 <= n <= 131072 for n in w5.n_live)
    assert w5.k_row_bytes() == 512 and W.get_workload("q8_0").k_row_bytes() == 136


def test_outlier_pairs_scale_both_dims():
    w = W.get_workload("qwen3_8b_layer")
    sc = W.pair_scales(w, 0)
    assert sc.shape == (8, 64) and (sc == 8.0).sum(axis=1).tolist() == [8] * 8


def test_normal12_equals_the_scalar_definition():
    """The vectorised draws equal the definition written out with Python ints:
    element j sums the twelve 16-bit fields of words 3j, 3j+1, 3j+2."""
    key = C.stream_key(3, C.TENSOR_V, 2, 1, 0)
    first = 12345
    got = C.normal12(key, first, 40)
    for i, j in enumerate(range(first, first + 40)):
        s = 0
        for t in range(3):
            w = C.mix64_int(key + (3 * j + t + 1) * C.GAMMA)
            s += sum((w >> sh) & 0xFFFF for sh in (0, 16, 32, 48))
        assert got[i] == np.float32((s - 393210) / 65536.0)
