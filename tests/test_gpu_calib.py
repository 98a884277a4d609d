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


NONROT_CASES = [
    # tokens, heads, head_dim, nonrot, dtype
    (1000, 8, 128, 64, "f16"),    # vector body, content vectors after the rotary ones
    (513, 4, 256, 192, "f32"),
    (300, 2, 96, 32, "f16"),
    (77, 3, 128, 8, "f32"),       # 60 rotary pairs: not whole fp32 vectors -> scalar body
    (50, 2, 6, 2, "f32"),         # scalar body, one content pair
]


@pytest.mark.parametrize("t,h,hd,nonrot,dtype", NONROT_CASES)
def test_calibration_non_rotary_dims(lib, t, h, hd, nonrot, dtype):
    """Heads whose last nonrot dims are not rotary: rotary pairs (f, f + rot/2)
    and the mean non-rotary query, against calibrate / calibrate_nonrot."""
    import torch
    q = _queries(t, h, hd, dtype, seed=3 * t + hd + nonrot)
    acc = torch.zeros((h, hd // 2, 3), dtype=torch.float64, device="cuda")
    lib.calib_accumulate(torch.from_numpy(q).cuda(), acc, nonrot_dim=nonrot)
    q_mean, q_abs, q_nonrot = lib.calib_finish(acc, t, nonrot_dim=nonrot)
    torch.cuda.synchronize()
    q64 = q.astype(np.float64)
    ref_mean, ref_abs = O.calibrate(q64, nonrot)
    ref_nonrot = O.calibrate_nonrot(q64, nonrot)
    scale = np.abs(q64).mean()
    np.testing.assert_allclose(q_mean.cpu().numpy(), ref_mean, rtol=1e-5, atol=1e-5 * scale)
    np.testing.assert_allclose(q_abs.cpu().numpy(), ref_abs, rtol=1e-5, atol=1e-5 * scale)
    np.testing.assert_allclose(q_nonrot.cpu().numpy(), ref_nonrot, rtol=1e-5, atol=1e-5 * scale)


def test_calibration_non_rotary_host_checks(lib):
    import torch
    acc = torch.zeros((2, 32, 3), dtype=torch.float64, device="cuda")
    q = torch.zeros((4, 2, 64), dtype=torch.float32, device="cuda")
    for bad in (-2, 3, 64):
        with pytest.raises(lib.TriaError) as err:
            lib.calib_accumulate(q, acc, nonrot_dim=bad)
        assert err.value.status == lib.ERR_INVALID_ARG
