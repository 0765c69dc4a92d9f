"""GPU checks of the issue/wait calls with a deferred epilogue, the SM budget
and the per-CTA profile records.

Every result is compared bit for bit with the oracle or with the synchronous
calls on the same inputs: the budget, the communication stream and the
profiling variants of the kernels must not change a single output bit."""
import numpy as np
import pytest
import torch

import combine_ep_plan_gb300 as ep
import oracle
from combine_ep_plan_gb300.inputs import WORKLOADS, bits_to_bf16_tensor, draw_hidden, draw_topk, draw_y, hidden_seed
from ep_testutil import assert_plan_equal, gpu_plan_arrays, u8, u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from combine_ep_plan_gb300 import build
    build.build()
    ep.load_library()
    yield
    torch.cuda.synchronize()


CASES = [
    WORKLOADS["tiny"],
    WORKLOADS["bf16"].scaled(S=300, H=1024),
    WORKLOADS["rt"].scaled(S=40, H=512),
]


def _inputs(w, seed=None):
    idx, wts = draw_topk(w, seed)
    idx[::5, 0] = -1
    x = draw_hidden(w.T, w.H, hidden_seed(w))
    return idx, wts, x


def _all_outputs(h, w, x_t, wts_t, y_t, go_t):
    """Every kernel of the path on one handle, results as host arrays."""
    out = {}
    recv, _ = ep.dispatch(h, x_t, "bf16", True, capacity=ep.worst_expanded_rows(w.T, w.K, w.E, w.A))
    out["recv_bf16"] = u16(recv)
    if w.H % 128 == 0:
        q, sc = ep.dispatch(h, x_t, "fp8", True, capacity=recv.shape[0])
        out["recv_fp8"], out["scales"] = u8(q), sc.cpu().numpy()
        # pre-quantised input: arbitrary codes and scales, copied as they are
        g = torch.Generator(device="cuda").manual_seed(9)
        xq = torch.randint(0, 256, (w.T, w.H), dtype=torch.uint8, device="cuda", generator=g)
        xs = torch.rand((w.T, w.H // 128), device="cuda", generator=g)
        q2, sc2 = ep.dispatch(h, xq.view(torch.float8_e4m3fn), "fp8", True, x_scales=xs, capacity=recv.shape[0])
        out["recv_fp8_input"], out["scales_input"] = u8(q2), sc2.cpu().numpy()
    out["combine"] = u16(ep.combine(h, y_t, wts_t))
    out["dispatch_backward"] = u16(ep.dispatch_backward(h, y_t))
    gy, gw = ep.combine_backward(h, go_t, y_t, wts_t)
    out["combine_backward_y"], out["combine_backward_w"] = u16(gy), gw.cpu().numpy()
    return out


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_sm_budget_changes_no_result(w):
    idx, wts, x = _inputs(w)
    pl = oracle.plan(idx, w.S, w.P, w.E, w.A)
    idx_t = torch.from_numpy(idx).cuda()
    x_t = bits_to_bf16_tensor(x).cuda()
    wts_t = torch.from_numpy(wts).cuda()
    rows = ep.worst_expanded_rows(w.T, w.K, w.E, w.A)
    y_t = bits_to_bf16_tensor(draw_y(rows, w.H, 5)).cuda()
    go_t = bits_to_bf16_tensor(draw_y(w.T, w.H, 6)).cuda()
    ref = None
    for budget in [0, 1, 3, 17]:
        h = ep.plan(idx_t, w.P, w.E, w.A)
        h.set_num_sms(budget)
        h.replan(idx_t)  # the plan itself under the budget
        assert_plan_equal(gpu_plan_arrays(h), pl)
        got = _all_outputs(h, w, x_t, wts_t, y_t, go_t)
        assert h.sync_status() == ep.EP_OK
        if ref is None:
            ref = got
            continue
        for k in ref:
            if k in ("recv_bf16", "recv_fp8", "scales", "recv_fp8_input", "scales_input"):
                # rows beyond N_exp are not written
                n = pl.num_expanded
                assert np.array_equal(got[k][:n], ref[k][:n]), (budget, k)
            elif k == "combine_backward_y":
                n = pl.num_expanded
                assert np.array_equal(got[k][:n], ref[k][:n]), (budget, k)
            else:
                assert np.array_equal(got[k], ref[k]), (budget, k)
        h.destroy()


def test_plan_under_a_one_sm_budget_with_more_ranks_than_its_threads():
    """1024 ranks and a one-SM budget (two co-resident plan CTAs, 512
    threads): the dense [T,P] pass keeps one rank per thread, so the plan
    still takes enough CTAs for every rank."""
    w = WORKLOADS["tiny"].scaled(P=1024, E=1024, S=1, K=2, A=2, H=256)
    idx, _, _ = _inputs(w)
    h = ep.plan(torch.from_numpy(idx).cuda(), w.P, w.E, w.A)
    h.set_num_sms(1)
    h.replan(torch.from_numpy(idx).cuda())
    assert h.sync_status() == ep.EP_OK
    assert_plan_equal(gpu_plan_arrays(h), oracle.plan(idx, w.S, w.P, w.E, w.A))


def test_sm_budget_rejects_negative():
    w = WORKLOADS["tiny"]
    idx, _, _ = _inputs(w)
    h = ep.plan(torch.from_numpy(idx).cuda(), w.P, w.E, w.A)
    with pytest.raises(ep.EPError):
        h.set_num_sms(-1)
    h.set_num_sms(100000)  # more than the device has: no cap


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
@pytest.mark.parametrize("defer", [False, True])
@pytest.mark.parametrize("fresh", [False, True])
def test_dispatch_async_matches_oracle(w, defer, fresh):
    idx, wts, x = _inputs(w)
    idx2, _, _ = _inputs(w, seed=77)
    pl = oracle.plan(idx, w.S, w.P, w.E, w.A)
    x_t = bits_to_bf16_tensor(x).cuda()
    # the handle starts on other routing when the async call re-plans it
    h = ep.plan(torch.from_numpy(idx2 if fresh else idx).cuda(), w.P, w.E, w.A)
    pend = ep.dispatch_async(h, x_t, "bf16", True, topk_idx=torch.from_numpy(idx).cuda() if fresh else None,
                             defer_epilogue=defer)
    recv, scales, n_exp, n_recv = pend.wait()
    assert scales is None
    assert (n_exp, n_recv) == (pl.num_expanded, int(pl.num_recv.sum()))
    assert np.array_equal(u16(recv)[:n_exp], oracle.dispatch_bf16(x, pl))
    assert h.sync_status() == ep.EP_OK
    assert_plan_equal(gpu_plan_arrays(h), pl)
    h.destroy()


@pytest.mark.parametrize("col_major", [False, True])
def test_dispatch_async_fp8(col_major):
    w = CASES[1]
    idx, wts, x = _inputs(w)
    pl = oracle.plan(idx, w.S, w.P, w.E, w.A)
    h = ep.plan(torch.from_numpy(idx).cuda(), w.P, w.E, w.A)
    pend = ep.dispatch_async(h, bits_to_bf16_tensor(x).cuda(), "fp8", True, scales_col_major=col_major)
    q, sc, n_exp, _ = pend.wait()
    q_ref, sc_ref = oracle.dispatch_fp8(x, pl)
    assert np.array_equal(u8(q)[:n_exp], q_ref)
    assert np.array_equal(sc.cpu().numpy()[:n_exp], sc_ref)
    h.check()


def test_overlap_with_independent_compute_and_bias():
    """The pattern of an overlapped shared expert: dispatch issued, a matmul on
    the compute stream meanwhile, wait, expert work, combine issued with the
    shared output as bias, wait.  Results equal the oracle's."""
    w = CASES[1]
    idx, wts, x = _inputs(w)
    pl = oracle.plan(idx, w.S, w.P, w.E, w.A)
    idx_t = torch.from_numpy(idx).cuda()
    x_t = bits_to_bf16_tensor(x).cuda()
    wts_t = torch.from_numpy(wts).cuda()
    h = ep.plan(idx_t, w.P, w.E, w.A)
    h.set_num_sms(16)
    compute = torch.cuda.current_stream()
    pend = ep.dispatch_async(h, x_t, "bf16", True, topk_idx=idx_t, stream=compute)
    g = torch.Generator(device="cuda").manual_seed(3)
    wmat = (torch.randn((w.H, w.H), device="cuda", generator=g) / w.H ** 0.5).to(torch.bfloat16)
    shared = x_t @ wmat                                    # independent work on the compute stream
    recv, _, n_exp, _ = pend.wait()
    y = recv                                               # identity expert, in compute-stream order
    ready = torch.cuda.Event()
    ready.record(compute)
    pend_c = ep.combine_async(h, y, wts_t, bias=shared, previous=ready, stream=compute)
    out = pend_c.wait()
    ref = oracle.combine(oracle.dispatch_bf16(x, pl), pl, wts, u16(shared))
    assert np.array_equal(u16(out), ref)
    h.check()


def test_previous_event_orders_the_inputs():
    """x is rewritten on the compute stream after a delay; the dispatch is
    ordered after it by the event, so it must see the new rows."""
    w = CASES[1]
    idx, _, x = _inputs(w)
    pl = oracle.plan(idx, w.S, w.P, w.E, w.A)
    h = ep.plan(torch.from_numpy(idx).cuda(), w.P, w.E, w.A)
    x_new = bits_to_bf16_tensor(x).cuda()
    x_t = torch.zeros_like(x_new)
    compute = torch.cuda.current_stream()
    torch.cuda._sleep(20_000_000)                           # keep the compute stream busy
    x_t.copy_(x_new)
    ev = torch.cuda.Event()
    ev.record(compute)
    for previous in (ev, None):
        pend = ep.dispatch_async(h, x_t, "bf16", True, previous=previous, stream=compute)
        recv, _, n_exp, _ = pend.wait()
        assert np.array_equal(u16(recv)[:n_exp], oracle.dispatch_bf16(x, pl))


def test_pending_limit_and_destroy_order():
    w = WORKLOADS["tiny"]
    idx, _, x = _inputs(w)
    h = ep.plan(torch.from_numpy(idx).cuda(), w.P, w.E, w.A)
    x_t = bits_to_bf16_tensor(x).cuda()
    pend = [ep.dispatch_async(h, x_t) for _ in range(8)]
    with pytest.raises(ep.EPError) as e:
        ep.dispatch_async(h, x_t)
    assert e.value.code == ep.EP_ERR_CAPACITY
    with pytest.raises(ep.EPError) as e:
        h.destroy()                                        # pending calls first
    assert e.value.code == ep.EP_ERR_INVALID
    for p in pend:
        p.wait()
    with pytest.raises(RuntimeError):
        pend[0].wait()
    h.destroy()


@pytest.mark.parametrize("defer", [False, True])
def test_async_reports_invalid_routing(defer):
    w = WORKLOADS["tiny"]
    idx, _, x = _inputs(w)
    bad = idx.copy()
    bad[5, 1] = w.E
    h = ep.plan(torch.from_numpy(idx).cuda(), w.P, w.E, w.A)
    if defer:
        pend = ep.dispatch_async(h, bits_to_bf16_tensor(x).cuda(), topk_idx=torch.from_numpy(bad).cuda(),
                                 defer_epilogue=True)
        with pytest.raises(ep.EPError) as e:
            pend.wait()
    else:
        with pytest.raises(ep.EPError) as e:
            ep.dispatch_async(h, bits_to_bf16_tensor(x).cuda(), topk_idx=torch.from_numpy(bad).cuda(),
                              defer_epilogue=False).wait()
    assert e.value.code == ep.EP_ERR_INVALID
    assert h.sync_status() == ep.EP_ERR_INVALID           # still recorded on the device; cleared here
    assert h.sync_status() == ep.EP_OK


# ---------------------------------------------------------------- profiling

def _profiled_run(w, fp8=False):
    idx, wts, x = _inputs(w)
    pl = oracle.plan(idx, w.S, w.P, w.E, w.A)
    idx_t = torch.from_numpy(idx).cuda()
    x_t = bits_to_bf16_tensor(x).cuda()
    wts_t = torch.from_numpy(wts).cuda()
    cap = ep.worst_expanded_rows(w.T, w.K, w.E, w.A)
    h = ep.plan(idx_t, w.P, w.E, w.A)
    outs = {}
    for prof in (False, True):
        if prof:
            h.profile_begin(1 << 20)
        h.replan(idx_t)
        recv, sc = ep.dispatch(h, x_t, "fp8" if fp8 else "bf16", True, capacity=cap)
        y = bits_to_bf16_tensor(oracle.dispatch_bf16(x, pl)).cuda()
        comb = ep.combine(h, y, wts_t)
        dbwd = ep.dispatch_backward(h, y)
        outs[prof] = (u8(recv)[: pl.num_expanded] if fp8 else u16(recv)[: pl.num_expanded],
                      sc.cpu().numpy()[: pl.num_expanded] if fp8 else None, u16(comb), u16(dbwd))
        if prof:
            rec, dropped = h.profile_end()
    h.check()
    return pl, outs, rec, dropped


@pytest.mark.parametrize("fp8", [False, True], ids=["bf16", "fp8"])
def test_profile_records_count_the_payload_exactly(fp8):
    w = CASES[1]
    pl, outs, rec, dropped = _profiled_run(w, fp8)
    for a, b in zip(outs[False], outs[True]):   # the profiling kernels compute the same bits
        assert (a is None and b is None) or np.array_equal(a, b)
    assert dropped == 0
    s = ep.summarize_profile(rec)
    assert [r["kernel"] for r in s] == ["plan", "dispatch_fp8" if fp8 else "dispatch_bf16", "combine",
                                        "dispatch_backward"]
    plan, disp, comb, dbwd = s
    n_valid = int((pl.slot >= 0).sum())
    n_pad = pl.num_expanded - n_valid
    H, T = w.H, w.T
    assert plan["units"] == T and plan["bytes"] == 0
    if fp8:
        assert disp["bytes"] == T * H * 2 + (n_valid + n_pad) * (H + 4 * (H // 128))
    else:
        assert disp["bytes"] == T * H * 2 + (n_valid + n_pad) * H * 2
    # combine: every valid slot's row read, one output row per token
    assert comb["bytes"] == (n_valid + T) * H * 2
    assert dbwd["bytes"] == (n_valid + T) * H * 2
    r = rec.numpy().astype(np.uint64)
    kind = r[:, 0] >> np.uint64(56)
    for k in (1, 2, 3, 5, 6):
        m = kind == k
        if m.any():
            assert np.all(r[m, 5] >= r[m, 1])
            cta = (r[m, 0] & np.uint64(0xFFFFFFFF)).astype(np.int64)
            assert np.array_equal(np.sort(cta), np.arange(m.sum()))  # one record per CTA
    # plan stage marks in order on the CTAs that scanned a tile
    m = (kind == 1) & (r[:, 2] > 0)
    assert m.any()
    assert np.all(r[m, 1] <= r[m, 2]) and np.all(r[m, 2] <= r[m, 3]) and np.all(r[m, 3] <= r[m, 4])
    assert np.all(r[m, 4] <= r[m, 5])


def test_profile_drops_what_does_not_fit():
    w = CASES[1]
    idx, _, x = _inputs(w)
    h = ep.plan(torch.from_numpy(idx).cuda(), w.P, w.E, w.A)
    x_t = bits_to_bf16_tensor(x).cuda()
    h.profile_begin(8)
    ep.dispatch(h, x_t, "bf16", True, capacity=ep.worst_expanded_rows(w.T, w.K, w.E, w.A))
    rec, dropped = h.profile_end()
    assert rec.shape[0] == 8 and dropped > 0
    cta = (rec.numpy().astype(np.uint64)[:, 0] & np.uint64(0xFFFFFFFF)).astype(np.int64)
    assert np.array_equal(cta, np.arange(8))
    h.check()


def test_profile_records_of_async_calls():
    """Launches issued on the communication stream write their records too."""
    w = CASES[1]
    idx, wts, x = _inputs(w)
    pl = oracle.plan(idx, w.S, w.P, w.E, w.A)
    idx_t = torch.from_numpy(idx).cuda()
    h = ep.plan(idx_t, w.P, w.E, w.A)
    h.profile_begin(1 << 16)
    recv, _, n_exp, _ = ep.dispatch_async(h, bits_to_bf16_tensor(x).cuda(), topk_idx=idx_t).wait()
    out = ep.combine_async(h, recv, torch.from_numpy(wts).cuda()).wait()
    rec, dropped = h.profile_end()
    assert dropped == 0
    kinds = [r["kernel"] for r in ep.summarize_profile(rec)]
    assert kinds == ["plan", "dispatch_bf16", "combine"]
    assert np.array_equal(u16(recv)[:n_exp], oracle.dispatch_bf16(x, pl))
    assert np.array_equal(u16(out), oracle.combine(oracle.dispatch_bf16(x, pl), pl, wts))
    h.check()


@pytest.mark.parametrize("defer", [False, True])
def test_combine_async_matches_sync(defer):
    w = CASES[2]
    idx, wts, x = _inputs(w)
    pl = oracle.plan(idx, w.S, w.P, w.E, w.A)
    h = ep.plan(torch.from_numpy(idx).cuda(), w.P, w.E, w.A)
    y = bits_to_bf16_tensor(draw_y(pl.num_expanded, w.H, 12)).cuda()
    wts_t = torch.from_numpy(wts).cuda()
    ref = u16(ep.combine(h, y, wts_t))
    got = u16(ep.combine_async(h, y, wts_t, defer_epilogue=defer).wait())
    assert np.array_equal(got, ref)
    assert np.array_equal(got, oracle.combine(u16(y), pl, wts))


def test_wait_without_counts():
    """A dispatch waited on without counts joins the stream only (the counts
    come back as 0); the rows are there either way."""
    w = CASES[1]
    idx, _, x = _inputs(w)
    pl = oracle.plan(idx, w.S, w.P, w.E, w.A)
    h = ep.plan(torch.from_numpy(idx).cuda(), w.P, w.E, w.A)
    x_t = bits_to_bf16_tensor(x).cuda()
    recv, _, n_exp, n_recv = ep.dispatch_async(h, x_t, defer_epilogue=True).wait(counts=False)
    assert (n_exp, n_recv) == (0, 0)
    assert np.array_equal(u16(recv)[:pl.num_expanded], oracle.dispatch_bf16(x, pl))
    recv, _, n_exp, n_recv = ep.dispatch_async(h, x_t, defer_epilogue=False).wait(counts=False)
    assert (n_exp, n_recv) == (0, 0)
    assert np.array_equal(u16(recv)[:pl.num_expanded], oracle.dispatch_bf16(x, pl))
    h.check()


def test_one_tile_plan_profile_and_replan():
    """A plan of one tile runs as one CTA without grid barriers; its record,
    and plans before and after it on the same handle, stay right."""
    w = WORKLOADS["tiny"]  # 256 tokens: one tile
    idx, _, _ = _inputs(w)
    idx2, _, _ = _inputs(w, seed=5)
    t, t2 = torch.from_numpy(idx).cuda(), torch.from_numpy(idx2).cuda()
    h = ep.plan(t, w.P, w.E, w.A)
    h.profile_begin(64)
    h.replan(t2)
    rec, dropped = h.profile_end()
    s = ep.summarize_profile(rec)
    assert dropped == 0 and len(s) == 1 and s[0]["kernel"] == "plan"
    assert s[0]["ctas"] == 1 and s[0]["units"] == w.T
    assert_plan_equal(gpu_plan_arrays(h), oracle.plan(idx2, w.S, w.P, w.E, w.A))
    h.replan(t)
    assert_plan_equal(gpu_plan_arrays(h), oracle.plan(idx, w.S, w.P, w.E, w.A))
    h.check()
