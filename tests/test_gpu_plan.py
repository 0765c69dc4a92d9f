"""GPU parity of the routing plan: every plan array bit-exact with the oracle,
on cases that span several tiles with a ragged tail, the full-size
workloads, and the degenerate shapes; plus the device-side error paths."""
import numpy as np
import pytest
import torch

import combine_ep_plan_gb300 as ep
import oracle
from combine_ep_plan_gb300.inputs import WORKLOADS, draw_topk
from ep_testutil import assert_plan_equal, gpu_plan_arrays

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from combine_ep_plan_gb300 import build
    build.build()
    ep.load_library()
    yield
    torch.cuda.synchronize()


SMALL = [
    WORKLOADS["tiny"],
    WORKLOADS["bf16"].scaled(S=300),
    WORKLOADS["fp8"].scaled(S=100),
    WORKLOADS["zipf"].scaled(S=13),
    WORKLOADS["rt"].scaled(S=70),
]


def _run(w, idx, C=0):
    h = ep.plan(torch.from_numpy(idx).cuda(), w.P, w.E, w.A, C)
    gpu = gpu_plan_arrays(h)
    assert h.sync_status() == ep.EP_OK
    return h, gpu


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_plan_small(w):
    idx, _ = draw_topk(w)
    h, gpu = _run(w, idx)
    assert_plan_equal(gpu, oracle.plan(idx, w.S, w.P, w.E, w.A))
    h.destroy()


@pytest.mark.parametrize("name", ["tiny", "bf16", "fp8", "zipf", "rt"])
def test_plan_full_size(name):
    w = WORKLOADS[name]
    idx, _ = draw_topk(w)
    h, gpu = _run(w, idx)
    assert_plan_equal(gpu, oracle.plan(idx, w.S, w.P, w.E, w.A))
    h.destroy()


@pytest.mark.parametrize("S,C", [(1, 1), (10, 6), (37, 37), (300, 1), (513, 7)])
def test_plan_channels_and_small_sources(S, C):
    w = WORKLOADS["tiny"].scaled(P=8, E=16, S=S, K=3, A=4)
    idx, _ = draw_topk(w)
    h, gpu = _run(w, idx, C)
    assert_plan_equal(gpu, oracle.plan(idx, w.S, w.P, w.E, w.A, C))


def test_plan_single_rank_and_unused_slots():
    w = WORKLOADS["tiny"].scaled(P=1, E=8, S=700, K=3, A=16)
    idx, _ = draw_topk(w)
    idx[::5, 2] = -1
    idx[::11] = -1
    h, gpu = _run(w, idx)
    assert_plan_equal(gpu, oracle.plan(idx, w.S, w.P, w.E, w.A))


def test_plan_no_routing_at_all():
    w = WORKLOADS["tiny"].scaled(S=100)
    idx = -np.ones((w.T, w.K), np.int64)
    h, gpu = _run(w, idx)
    assert h.sizes() == (0, 0)
    assert_plan_equal(gpu, oracle.plan(idx, w.S, w.P, w.E, w.A))


def test_plan_one_expert_per_rank_many_tiles():
    w = WORKLOADS["tiny"].scaled(P=64, E=64, S=97, K=8, A=8)
    idx, _ = draw_topk(w)
    h, gpu = _run(w, idx)
    assert_plan_equal(gpu, oracle.plan(idx, w.S, w.P, w.E, w.A))


def test_plan_more_tiles_than_resident_ctas():
    """375 tiles: more than the co-resident grid, so CTAs loop over tiles in
    phase 1 and phase 2 takes every position from global memory."""
    w = WORKLOADS["tiny"].scaled(P=8, E=16, S=12000, K=2, A=4)
    idx, _ = draw_topk(w)
    idx[::7, 1] = -1
    h, gpu = _run(w, idx, 5)
    assert_plan_equal(gpu, oracle.plan(idx, w.S, w.P, w.E, w.A, 5))


def test_replan_reuses_handle():
    w = WORKLOADS["bf16"].scaled(S=257)
    idx0, _ = draw_topk(w, seed=3)
    idx1, _ = draw_topk(w, seed=4)
    h = ep.plan(torch.from_numpy(idx0).cuda(), w.P, w.E, w.A)
    h.replan(torch.from_numpy(idx1).cuda())
    assert_plan_equal(gpu_plan_arrays(h), oracle.plan(idx1, w.S, w.P, w.E, w.A))


def test_plan_is_deterministic():
    w = WORKLOADS["zipf"].scaled(S=40)
    idx, _ = draw_topk(w)
    a = gpu_plan_arrays(ep.plan(torch.from_numpy(idx).cuda(), w.P, w.E, w.A))
    b = gpu_plan_arrays(ep.plan(torch.from_numpy(idx).cuda(), w.P, w.E, w.A))
    for k in a:
        assert np.array_equal(a[k], b[k]), k


@pytest.mark.parametrize("mutate", ["range", "dup", "low"])
def test_device_reports_invalid_routing(mutate):
    w = WORKLOADS["tiny"]
    idx, _ = draw_topk(w)
    if mutate == "range":
        idx[5, 0] = w.E
    elif mutate == "dup":
        idx[7, 1] = idx[7, 0]
    else:
        idx[3, 1] = -2
    h = ep.plan(torch.from_numpy(idx).cuda(), w.P, w.E, w.A)
    assert h.sync_status() == ep.EP_ERR_INVALID
    assert h.sync_status() == ep.EP_OK  # cleared


def test_barrier_timeout_is_reported_and_recoverable():
    """A tile whose CTA never arrives at the first grid barrier makes the
    others' bounded wait run out: the plan reports EP_ERR_TIMEOUT and the
    next plan succeeds."""
    w = WORKLOADS["bf16"].scaled(S=200)  # 1600 tokens -> 7 tiles
    idx, _ = draw_topk(w)
    t = torch.from_numpy(idx).cuda()
    try:
        ep.set_plan_wait_debug(poll_limit=2000, suppress_tile=2)
        h = ep.plan(t, w.P, w.E, w.A)
        assert h.sync_status() == ep.EP_ERR_TIMEOUT
    finally:
        ep.set_plan_wait_debug(0, -1)
    h2 = ep.plan(t, w.P, w.E, w.A)
    assert h2.sync_status() == ep.EP_OK
    assert_plan_equal(gpu_plan_arrays(h2), oracle.plan(idx, w.S, w.P, w.E, w.A))
    # the handle that timed out recovers too
    h.replan(t)
    assert h.sync_status() == ep.EP_OK
    assert_plan_equal(gpu_plan_arrays(h), oracle.plan(idx, w.S, w.P, w.E, w.A))


def test_replan_right_after_a_timeout_does_no_barrier_work():
    """A plan whose grid-barrier wait ran out leaves its arrivals in the
    barrier count.  Plans enqueued right after it, with no status read in
    between, must not pass a barrier on those arrivals: they find the
    timed-out mark and arrive at no barrier, the status stays EP_ERR_TIMEOUT,
    and a dispatch on the unfinished plan writes nothing past its capacity.
    Reading the status clears the control words; the next plan is correct."""
    w = WORKLOADS["bf16"].scaled(S=200)  # 1600 tokens -> 7 tiles, a grid of more CTAs
    idx, _ = draw_topk(w)
    idx2, _ = draw_topk(w, seed=5)
    t, t2 = torch.from_numpy(idx).cuda(), torch.from_numpy(idx2).cuda()
    try:
        ep.set_plan_wait_debug(poll_limit=2000, suppress_tile=2)
        h = ep.plan(t, w.P, w.E, w.A)
    finally:
        ep.set_plan_wait_debug(0, -1)
    h.replan(t2)  # no status read in between
    h.replan(t2)
    H = 256
    cap = ep.worst_expanded_rows(w.T, w.K, w.E, w.A)
    x = torch.randn((w.T, H), device="cuda").to(torch.bfloat16)
    buf = torch.full((cap + 64, H), 5.0, dtype=torch.bfloat16, device="cuda")
    ep.dispatch(h, x, "bf16", True, recv_x=buf[:cap])
    assert h.sync_status() == ep.EP_ERR_TIMEOUT
    assert torch.all(buf[cap:] == 5.0)
    h.replan(t2)
    assert h.sync_status() == ep.EP_OK
    assert_plan_equal(gpu_plan_arrays(h), oracle.plan(idx2, w.S, w.P, w.E, w.A))


def test_worst_expanded_rows_bounds_exact_size():
    for name in ["tiny", "bf16", "fp8", "zipf", "rt"]:
        w = WORKLOADS[name]
        idx, _ = draw_topk(w)
        h = ep.plan(torch.from_numpy(idx).cuda(), w.P, w.E, w.A)
        assert h.sizes()[0] <= ep.worst_expanded_rows(w.T, w.K, w.E, w.A)


def test_new_handle_on_reused_pool_memory():
    """A handle made right after another one was destroyed gets the same pool
    memory back, stale barrier counts and scratch included: its plans must
    not depend on what that memory held."""
    w = WORKLOADS["bf16"].scaled(S=300)
    for seed in range(4):
        idx, _ = draw_topk(w, seed=100 + seed)
        h = ep.plan(torch.from_numpy(idx).cuda(), w.P, w.E, w.A)
        assert_plan_equal(gpu_plan_arrays(h), oracle.plan(idx, w.S, w.P, w.E, w.A))
        h.destroy()


def test_many_replans_with_changing_grids():
    """Hundreds of plans on one handle, the grid changing between them (SM
    budgets, profiling variants): every barrier must start from a zeroed
    count; spot checks against the oracle."""
    w = WORKLOADS["bf16"].scaled(S=300)  # 10 tiles
    h = None
    for i in range(240):
        idx, _ = draw_topk(w, seed=1000 + (i % 7))
        t = torch.from_numpy(idx).cuda()
        if h is None:
            h = ep.plan(t, w.P, w.E, w.A)
        h.set_num_sms([0, 3, 17, 152][i % 4])
        if i % 5 == 0:
            h.profile_begin(4096)
            h.replan(t)
            h.profile_end()
        else:
            h.replan(t)
        if i % 37 == 0 or i == 239:
            assert h.sync_status() == ep.EP_OK
            assert_plan_equal(gpu_plan_arrays(h), oracle.plan(idx, w.S, w.P, w.E, w.A))
    assert h.sync_status() == ep.EP_OK
