"""The pass captured in a CUDA graph (stream capture through the C ABI) and
replayed gives the same bytes as a direct call, and replays again on fresh
input (n_live and the rows are read on the device at run time)."""
import numpy as np
import pytest

import _util as U

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.mark.parametrize("k_type", ["f16", "q8_0", "f32"])
def test_graph_replay_equals_direct_call(lib, k_type):
    case = U.Case(n_kv=2, group=4, hd=128, k_type=k_type, v_type="f16", n_live=[3000, 1700],
                  capacity=[3072, 2048], cur_pos=[40000, 1700], budget_frac=0.25, window=64, sink=4)
    host = U.build_host(case)
    dev = U.to_device(host)
    cache, pol = U.lib_cache(lib, case, dev), U.lib_policy(lib, case)
    ws = U.new_workspace(lib, cache, case.group)
    st = lib.Stats(host["q_mean"], host["q_abs"], n_kv_heads=case.n_kv, head_dim=case.hd, rope_theta=case.theta)
    planes = [k for k in ("k", "k_scale", "v", "pos", "n_live") if dev.get(k) is not None]

    def reset():
        for k in planes:
            dev[k].copy_(torch.from_numpy(np.ascontiguousarray(host[k])))
        torch.cuda.synchronize()

    reset()
    lib.evict(st, 0, cache, pol, ws=ws)          # direct (also the first-call set-up)
    torch.cuda.synchronize()
    assert lib.device_status(ws) == lib.OK
    want = {k: dev[k].cpu().clone() for k in planes}

    reset()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=s):
        lib.evict(st, 0, cache, pol, ws=ws)
    torch.cuda.synchronize()
    for k in planes:                              # capture runs nothing
        assert torch.equal(dev[k].cpu(), torch.from_numpy(np.ascontiguousarray(host[k]))), k
    for _ in range(2):
        reset()
        g.replay()
        torch.cuda.synchronize()
        assert lib.device_status(ws) == lib.OK
        for k in planes:
            assert torch.equal(dev[k].cpu(), want[k]), k


def test_marked_pass_in_a_graph_times_its_stages(lib):
    case = U.Case(n_kv=2, group=4, hd=128, k_type="f16", v_type="f16", n_live=[4096], capacity=[4096],
                  cur_pos=[9000], budget_frac=0.25, window=64, sink=4)
    host = U.build_host(case)
    dev = U.to_device(host)
    cache, pol = U.lib_cache(lib, case, dev), U.lib_policy(lib, case)
    ws = U.new_workspace(lib, cache, case.group)
    st = lib.Stats(host["q_mean"], host["q_abs"], n_kv_heads=case.n_kv, head_dim=case.hd, rope_theta=case.theta)
    lib.evict(st, 0, cache, pol, ws=ws)
    torch.cuda.synchronize()
    want = {k: dev[k].cpu().clone() for k in ("k", "v", "pos", "n_live")}
    for k in ("k", "v", "pos", "n_live"):
        dev[k].copy_(torch.from_numpy(np.ascontiguousarray(host[k])))
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    for e in evs:
        e.record()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=s):
        lib.evict_marked(st, 0, cache, pol, evs, ws=ws)
    g.replay()
    evs[3].synchronize()
    assert lib.device_status(ws) == lib.OK
    for k in want:
        assert torch.equal(dev[k].cpu(), want[k]), k
    stages = [evs[i].elapsed_time(evs[i + 1]) for i in range(3)]
    assert all(x > 0.0 for x in stages)
    assert abs(sum(stages) - evs[0].elapsed_time(evs[3])) < 1e-3
