"""Calibration statistics on the GPU (tria_calib_accumulate / tria_calib_finish)
against the oracle ([Doc] §2 Calibration file; §5 Phase C q_mean / q_abs layout)."""
import numpy as np
import pytest

from oracle import tria_oracle as O

pytestmark = pytest.mark.gpu

CASES = [
    # tokens, heads, head_dim, dtype
    (1, 1, 64, "f32"),
    (37, 3, 128, "f16"),
    (1000, 32, 128, "f16"),
    (513, 4, 256, "f32"),
    (300, 2, 96, "f16"),
    (4096, 8, 512, "f16"),
    (50, 2, 6, "f32"),      # head_dim not a multiple of 4: the scalar body
    (77, 3, 2, "f16"),      # one frequency pair
]


def _queries(t, h, hd, dtype, seed):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((t, h, hd)) * (1.0 + 3.0 * rng.random((1, h, hd)))   # per-channel scale
    q += rng.standard_normal((1, h, hd))                                           # non-zero means
    return q.astype(np.float16 if dtype == "f16" else np.float32)


@pytest.mark.parametrize("t,h,hd,dtype", CASES)
def test_calibration_matches_oracle(lib, t, h, hd, dtype):
    import torch
    q = _queries(t, h, hd, dtype, seed=t + 7 * h + hd)
    acc = torch.zeros((h, hd // 2, 3), dtype=torch.float64, device="cuda")
    lib.calib_accumulate(torch.from_numpy(q).cuda(), acc)
    q_mean, q_abs = lib.calib_finish(acc, t)
    torch.cuda.synchronize()
    ref_mean, ref_abs = O.calibrate(q.astype(np.float64))
    # fp32 sums of at most 256 tokens per block, fp64 across blocks
    scale = np.abs(q.astype(np.float64)).mean()
    np.testing.assert_allclose(q_mean.cpu().numpy(), ref_mean, rtol=1e-5, atol=1e-5 * scale)
    np.testing.assert_allclose(q_abs.cpu().numpy(), ref_abs, rtol=1e-5, atol=1e-5 * scale)


def test_calibration_accumulates_batches(lib):
    import torch
    q = _queries(2000, 4, 128, "f16", seed=99)
    acc = torch.zeros((4, 64, 3), dtype=torch.float64, device="cuda")
    qd = torch.from_numpy(q).cuda()
    for lo, hi in ((0, 1), (1, 700), (700, 700), (700, 2000)):   # ragged batches, an empty one
        lib.calib_accumulate(qd[lo:hi], acc)
    q_mean, q_abs = lib.calib_finish(acc, 2000)
    ref_mean, ref_abs = O.calibrate(q.astype(np.float64))
    np.testing.assert_allclose(q_mean.cpu().numpy(), ref_mean, rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(q_abs.cpu().numpy(), ref_abs, rtol=1e-5, atol=1e-6)


def test_calibrated_stats_load(lib):
    # the finished arrays are one layer's rows of tria_stats_desc: they load
    import torch
    q = _queries(500, 8, 64, "f32", seed=5)
    acc = torch.zeros((8, 32, 3), dtype=torch.float64, device="cuda")
    lib.calib_accumulate(torch.from_numpy(q).cuda(), acc)
    q_mean, q_abs = lib.calib_finish(acc, 500)
    qm = q_mean.cpu().numpy()[None].astype(np.float32)
    qa = q_abs.cpu().numpy()[None].astype(np.float32)
    st = lib.Stats(qm, qa, n_kv_heads=2, head_dim=64, rope_theta=1e4)
    assert st.handle
    ref_mean, ref_abs = O.calibrate(q.astype(np.float64))
    np.testing.assert_allclose(qm[0], ref_mean, rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(qa[0], ref_abs, rtol=1e-5, atol=1e-6)
    st.close()
