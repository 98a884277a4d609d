"""tria_select_noalloc, the selection entry point for callers that cannot
allocate device memory: its output must equal tria_select's (bit-exact keep
lists) on two calls in a row, which also shows that the shared fixed scratch
array is cleared between calls. Collected last on purpose."""
import numpy as np
import pytest

import _util as U
from oracle import tria_oracle as O

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _case(seed, n_live, cap, budget, sink, window):
    rng = np.random.default_rng(seed)
    case = U.Case(n_kv=4, group=1, hd=128, k_type="f16", v_type="f16", n_live=n_live, capacity=cap,
                  cur_pos=[0] * len(n_live), budget_rows=budget, sink=sink, window=window, seed=seed)
    rows = case.total_rows()
    levels = np.array([-1.0, 0.0, 0.5, 0.5, 2.0, np.nan], np.float32)
    score = np.where(rng.random(rows) < 0.4, rng.choice(levels, rows),
                     rng.standard_normal(rows)).astype(np.float32)
    return case, score


def test_select_noalloc_matches_select_twice(lib):
    case, score1 = _case(21, [6000, 1000, 300], [6144, 1024, 320], [1500, 600, 300], 4, 64)
    _, score2 = _case(22, [6000, 1000, 300], [6144, 1024, 320], [1500, 600, 300], 4, 64)
    host = U.build_host(case)
    dev = U.to_device(host)
    cache, pol = U.lib_cache(lib, case, dev), U.lib_policy(lib, case)
    ws = U.new_workspace(lib, cache, 0)
    rows = case.total_rows()
    for score in (score1, score2):
        s_dev = torch.from_numpy(score).cuda()
        want = torch.full((rows,), -3, dtype=torch.int32, device="cuda")
        got = torch.full((rows,), -3, dtype=torch.int32, device="cuda")
        lib.select(s_dev, cache, pol, want, ws=ws)
        lib.select_noalloc(s_dev, cache, pol, got)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(got.cpu().numpy(), want.cpu().numpy())
        # and both equal the oracle's selection on the same scores
        g = got.cpu().numpy()
        for s, g_ in [(0, 1), (1, 3), (2, 0)]:
            r0 = int(case.seq_row0()[s] + g_ * case.capacity[s])
            n, b = case.n_live[s], case.budget_rows[s]
            ref = O.select_keep(score[r0:r0 + n], n, b, case.sink, case.window)
            np.testing.assert_array_equal(g[r0:r0 + len(ref)], ref)


def test_select_noalloc_cooperative_path_matches_select_twice(lib):
    """Segments over 262144 rows take the cooperative grid select, whose grid
    barrier state lives in the fixed array too; one sequence of 300000 rows x 2
    KV heads fits the array. Bit-exact against tria_select and the oracle on two
    calls in a row."""
    n, b = 300000, 75000
    case = U.Case(n_kv=2, group=1, hd=64, k_type="f16", v_type="f16", n_live=[n], capacity=[n], cur_pos=[0],
                  budget_rows=[b], sink=4, window=512, seed=31)
    # the select reads scores and n_live only: small placeholder key / value /
    # position planes stand in for the cache's
    dummy = torch.zeros(64, dtype=torch.float16, device="cuda")
    cache = lib.LayerCache(k=dummy, v=dummy, pos=dummy.view(torch.int32),
                           n_live=torch.tensor([n], dtype=torch.int32, device="cuda"), seq_row0=case.seq_row0(),
                           capacity=case.capacity, head_dim=64, n_kv_heads=2)
    pol = U.lib_policy(lib, case)
    ws = U.new_workspace(lib, cache, 0)
    rows = case.total_rows()
    for seed in (41, 42):
        rng = np.random.default_rng(seed)
        levels = np.array([-1.0, 0.0, 0.5, 2.0, np.nan], np.float32)
        score = np.where(rng.random(rows) < 0.3, rng.choice(levels, rows),
                         rng.standard_normal(rows)).astype(np.float32)
        s_dev = torch.from_numpy(score).cuda()
        want = torch.full((rows,), -3, dtype=torch.int32, device="cuda")
        got = torch.full((rows,), -3, dtype=torch.int32, device="cuda")
        lib.select(s_dev, cache, pol, want, ws=ws)
        assert lib.device_status(ws) == lib.OK
        lib.select_noalloc(s_dev, cache, pol, got)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(got.cpu().numpy(), want.cpu().numpy())
        g = got.cpu().numpy()
        for h in range(2):
            ref = O.select_keep(score[h * n:h * n + n], n, b, case.sink, case.window)
            np.testing.assert_array_equal(g[h * n:h * n + b], ref)


def test_select_noalloc_rejects_oversized_calls(lib):
    case = U.Case(n_kv=8, group=1, hd=128, k_type="f16", v_type="f16", n_live=[100] * 64,
                  capacity=[1 << 20] * 64, cur_pos=[0] * 64, budget_rows=[50] * 64, sink=0, window=0)
    dummy = torch.zeros(16, dtype=torch.uint8, device="cuda")
    cache = lib.LayerCache(k=dummy, v=dummy, pos=dummy, n_live=torch.zeros(64, dtype=torch.int32, device="cuda"),
                           seq_row0=case.seq_row0(), capacity=case.capacity, head_dim=128, n_kv_heads=8)
    pol = U.lib_policy(lib, case)
    with pytest.raises(lib.TriaError) as e:
        lib.select_noalloc(dummy.view(torch.float32), cache, pol, dummy.view(torch.int32))
    assert e.value.status == lib.ERR_WORKSPACE
