"""The hot path captured in a CUDA graph and replayed: the plan's grid
barriers reset their counts at the end of every launch, so each replay of
the captured plan, dispatch and combine is as correct as a fresh launch."""
import numpy as np
import pytest
import torch

import combine_ep_plan_gb300 as ep
import oracle
from combine_ep_plan_gb300.inputs import WORKLOADS, bits_to_bf16_tensor, draw_hidden, draw_topk
from ep_testutil import assert_plan_equal, gpu_plan_arrays, u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from combine_ep_plan_gb300 import build
    build.build()
    ep.load_library()
    yield
    torch.cuda.synchronize()


@pytest.mark.parametrize("w", [WORKLOADS["bf16"].scaled(S=300, H=1024), WORKLOADS["tiny"]],
                         ids=["many_tiles", "one_tile"])
def test_captured_step_replays(w):
    idx0, wts0 = draw_topk(w, seed=0)
    idx_t = torch.from_numpy(idx0).cuda()
    wts_t = torch.from_numpy(wts0).cuda()
    x_t = bits_to_bf16_tensor(draw_hidden(w.T, w.H, 1)).cuda()
    cap = ep.worst_expanded_rows(w.T, w.K, w.E, w.A)
    recv = torch.empty((cap, w.H), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((w.T, w.H), dtype=torch.bfloat16, device="cuda")
    h = ep.plan(idx_t, w.P, w.E, w.A)

    def step():
        h.replan(idx_t)
        ep.dispatch(h, x_t, "bf16", True, recv_x=recv)
        ep.combine(h, recv, wts_t, out=out)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for seed in (3, 4, 5):
        idx, wts = draw_topk(w, seed=seed)
        x = draw_hidden(w.T, w.H, 10 + seed)
        idx_t.copy_(torch.from_numpy(idx))
        wts_t.copy_(torch.from_numpy(wts))
        x_t.copy_(bits_to_bf16_tensor(x))
        graph.replay()
        torch.cuda.synchronize()
        assert h.sync_status() == ep.EP_OK
        h.sizes(refresh=True)  # the replay planned without the Python object
        pl = oracle.plan(idx, w.S, w.P, w.E, w.A)
        assert_plan_equal(gpu_plan_arrays(h), pl)
        assert np.array_equal(u16(recv)[: pl.num_expanded], oracle.dispatch_bf16(x, pl))
        assert np.array_equal(u16(out), oracle.combine(oracle.dispatch_bf16(x, pl), pl, wts))
