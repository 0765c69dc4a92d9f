"""Seeded random shapes through the whole path on the GPU, every output
against the oracle.

Each case draws ranks, experts per rank, top-k, expert alignment, channels,
tokens per rank, hidden size, the routing (uniform or Zipf) and a share of
unused slots, then runs the plan, the BF16 and FP8 dispatches (zero
padding), the dispatch metadata, a combine of random expert outputs, and
both backward passes on one handle.  Plan arrays, dispatched rows, codes,
scales, metadata, combine and grad_x / grad_y are compared bit for bit;
grad_w within the error bound of an fp32 dot product.  The shapes cover one
tile and many, more tiles than channels and the reverse, P = 1, A = 1, one
token per rank and ragged tails.
"""
import numpy as np
import pytest
import torch

import combine_ep_plan_gb300 as ep
import oracle
from combine_ep_plan_gb300.inputs import Workload, bits_to_bf16_tensor, draw_hidden, draw_topk, draw_y
from ep_testutil import assert_bits_equal, assert_plan_equal, gpu_plan_arrays

pytestmark = pytest.mark.gpu

N_CASES = 100


@pytest.fixture(scope="module", autouse=True)
def _built():
    from combine_ep_plan_gb300 import build
    build.build()
    ep.load_library()
    yield
    torch.cuda.synchronize()


def _case(i: int):
    rng = np.random.default_rng(7000 + i)
    P = int(rng.choice([1, 2, 3, 4, 8, 16, 32, 64, 128]))
    El = int(rng.choice([1, 2, 3, 4, 8]))
    E = P * El
    K = int(rng.integers(1, min(E, 16) + 1))
    A = int(rng.choice([1, 2, 7, 16, 64, 128]))
    S = int(rng.choice([1, 3, 17, 64, 100, 255, 256, 257, 600, 1000]))
    while P * S > 20000:
        S = max(1, S // 2)
    C = int(rng.choice([0, 1, min(S, 5), S]))
    H = int(rng.choice([128, 256, 384, 1024]))
    routing = "zipf" if rng.random() < 0.3 else "uniform"
    w = Workload(f"fuzz{i}", P=P, E=E, S=S, H=H, K=K, A=A, routing=routing, seed=i)
    return w, C, float(rng.choice([0.0, 0.1, 0.5])), rng


def _grad_w_ok(got, ref, go_bits, y_bits, slot):
    """|got - ref| within H * 2^-23 * sum_h |grad_out * y| (+ 1e-6) per valid slot."""
    valid = slot >= 0
    if not valid.any():
        return True
    go = torch.from_numpy(np.ascontiguousarray(go_bits).view(np.int16)).view(torch.bfloat16).double().abs()
    y = torch.from_numpy(np.ascontiguousarray(y_bits).view(np.int16)).view(torch.bfloat16).double().abs()
    rows = torch.from_numpy(np.maximum(slot, 0)).long()
    mag = torch.stack([(go * y[rows[:, k]]).sum(dim=1) for k in range(slot.shape[1])], dim=1).numpy()
    tol = go.shape[1] * 2.0 ** -23 * mag + 1e-6
    return bool(np.all(np.abs(got - ref)[valid] <= tol[valid]))


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_shape_whole_path(i):
    w, C, p_unused, rng = _case(i)
    idx, wts = draw_topk(w)
    idx[rng.random(idx.shape) < p_unused] = -1
    idx[rng.random(w.T) < 0.02] = -1  # tokens with no slot at all
    Cq = C if C else min(16, w.S)
    pl = oracle.plan(idx, w.S, w.P, w.E, w.A, Cq)
    h = ep.plan(torch.from_numpy(idx).cuda(), w.P, w.E, w.A, C)
    assert h.sync_status() == ep.EP_OK
    assert_plan_equal(gpu_plan_arrays(h), pl)
    n = pl.num_expanded
    cap = ep.worst_expanded_rows(w.T, w.K, w.E, w.A)

    x = draw_hidden(w.T, w.H, 100 + i)
    xt = bits_to_bf16_tensor(x).cuda()
    recv, _ = ep.dispatch(h, xt, "bf16", True, capacity=cap)
    q, sc = ep.dispatch(h, xt, "fp8", True, capacity=cap)
    wts_t = torch.from_numpy(wts).cuda()
    rw, rm = ep.dispatch_metadata(h, wts_t, capacity=cap)
    y = draw_y(max(n, 1), w.H, 200 + i)
    yt = bits_to_bf16_tensor(y).cuda()
    out = ep.combine(h, yt, wts_t)
    gx = ep.dispatch_backward(h, yt)
    go = draw_y(w.T, w.H, 300 + i)
    gy, gw = ep.combine_backward(h, bits_to_bf16_tensor(go).cuda(), yt, wts_t, zero_pad=True)
    assert h.sync_status() == ep.EP_OK

    with oracle.parallel():
        assert_bits_equal(recv[:n], oracle.dispatch_bf16(x, pl, True), "bf16 rows")
        q_ref, s_ref = oracle.dispatch_fp8(x, pl, True)
        assert_bits_equal(q[:n].view(torch.uint8), q_ref, "fp8 codes")
        assert_bits_equal(sc[:n], s_ref, "fp8 scales")
        rw_ref, rm_ref = oracle.dispatch_metadata(pl, wts)
        assert_bits_equal(rw[:n], rw_ref, "recv weights")
        assert_bits_equal(rm[:n], rm_ref, "recv meta")
        assert_bits_equal(out, oracle.combine(y[:n], pl, wts), "combine")
        assert_bits_equal(gx, oracle.dispatch_backward(y[:n], pl), "grad_x")
        gy_ref, gw_ref = oracle.combine_backward(go, y[:n], pl, wts, zero_pad=True)
    assert_bits_equal(gy[:n], gy_ref, "grad_y")
    assert _grad_w_ok(gw.cpu().numpy().astype(np.float64), gw_ref, go, y[:n], pl.slot)
    assert np.all(gw.cpu().numpy()[pl.slot < 0] == 0)
    h.destroy()
