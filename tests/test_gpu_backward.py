"""GPU parity of the backward on the same handle (tutorial ch. 38 §2.3):
dispatch backward (unweighted combine) and combine backward (grad_y scatter
and grad_w dot products) against the oracle."""
import numpy as np
import pytest
import torch

import combine_ep_plan_gb300 as ep
import oracle
from combine_ep_plan_gb300.inputs import WORKLOADS, bits_to_bf16_tensor, draw_topk, draw_y
from ep_testutil import assert_bits_equal, u16

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
    WORKLOADS["bf16"].scaled(S=300, H=1024),
    WORKLOADS["zipf"].scaled(S=13, H=512),
    WORKLOADS["rt"].scaled(S=70, H=768),
]


def _f64(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).double().numpy()


def _grad_w_close(got, ref, go_bits, y_bits, pl):
    """fp32 dot products of H terms against float64: within H * 2^-23 of the
    sum of |terms| (plus a tiny absolute slack)."""
    H = go_bits.shape[1]
    go = _f64(go_bits)
    y = _f64(y_bits)
    rows = np.maximum(pl.slot, 0)
    mag = np.einsum("th,tkh->tk", np.abs(go), np.abs(y[rows]))
    tol = H * 2.0 ** -23 * mag + 1e-6
    assert np.all(np.abs(got - ref) <= tol)


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_backward_small(w):
    idx, wts = draw_topk(w)
    idx[::5, -1] = -1
    pl = oracle.plan(idx, w.S, w.P, w.E, w.A)
    gr = draw_y(pl.num_expanded, w.H, 21)
    y = draw_y(pl.num_expanded, w.H, 22)
    go = draw_y(w.T, w.H, 23)
    gx_ref = oracle.dispatch_backward(gr, pl)
    gy_ref, gw_ref = oracle.combine_backward(go, y, pl, wts, zero_pad=True)

    h = ep.plan(torch.from_numpy(idx).cuda(), w.P, w.E, w.A)
    gx = ep.dispatch_backward(h, bits_to_bf16_tensor(gr).cuda())
    gy_buf = torch.full((pl.num_expanded + 5, w.H), 9.0, dtype=torch.bfloat16, device="cuda")
    gy, gw = ep.combine_backward(h, bits_to_bf16_tensor(go).cuda(), bits_to_bf16_tensor(y).cuda(),
                                 torch.from_numpy(wts).cuda(), zero_pad=True, grad_y=gy_buf)
    assert h.sync_status() == ep.EP_OK
    assert np.array_equal(u16(gx), gx_ref)
    got_gy = u16(gy)
    assert np.array_equal(got_gy[: pl.num_expanded], gy_ref)
    nine = u16(torch.tensor([9.0], dtype=torch.bfloat16))[0]
    assert np.all(got_gy[pl.num_expanded:] == nine)  # rows past N_exp untouched
    _grad_w_close(gw.cpu().numpy().astype(np.float64), gw_ref, go, y, pl)
    assert np.all(gw.cpu().numpy()[pl.slot < 0] == 0)


def _grad_w_bound_gpu(go_t, y_t, slot, H):
    """H * 2^-23 * sum_h |grad_out[g,h] * y[slot,h]| + 1e-6 per (token, slot),
    in float64 on the device (the error bound of an fp32 dot product of H
    terms; a tolerance, not an expected value)."""
    go = go_t.double().abs()
    sl = torch.from_numpy(np.maximum(slot, 0)).cuda().long()
    mag = torch.zeros(slot.shape, dtype=torch.float64, device="cuda")
    for k in range(slot.shape[1]):
        mag[:, k] = (go * y_t[sl[:, k]].double().abs()).sum(dim=1)
    return H * 2.0 ** -23 * mag + 1e-6


@pytest.mark.parametrize("name", ["bf16", "rt"])
def test_backward_full_size_whole_arrays_and_deterministic(name):
    """Full-size backward on the forward plan: grad_x and grad_y whole arrays
    bit for bit against the oracle, grad_w within the fp32 dot-product bound of
    the oracle's float64 sums, rows past N_exp untouched, and two runs equal."""
    w = WORKLOADS[name]
    idx, wts = draw_topk(w)
    pl = oracle.plan(idx, w.S, w.P, w.E, w.A)
    h = ep.plan(torch.from_numpy(idx).cuda(), w.P, w.E, w.A)
    cap = ep.worst_expanded_rows(w.T, w.K, w.E, w.A)
    n = pl.num_expanded
    y = draw_y(cap, w.H, 31)
    go = draw_y(w.T, w.H, 32)
    y_t, go_t, w_t = bits_to_bf16_tensor(y).cuda(), bits_to_bf16_tensor(go).cuda(), torch.from_numpy(wts).cuda()
    gy_buf = torch.full((cap, w.H), 9.0, dtype=torch.bfloat16, device="cuda")
    gy1, gw1 = ep.combine_backward(h, go_t, y_t, w_t, zero_pad=True, grad_y=gy_buf)
    gy2, gw2 = ep.combine_backward(h, go_t, y_t, w_t, zero_pad=True)
    gx = ep.dispatch_backward(h, y_t)
    assert h.sync_status() == ep.EP_OK
    assert torch.equal(gw1, gw2) and torch.equal(gy1[:n], gy2[:n])
    with oracle.parallel():
        gx_ref = oracle.dispatch_backward(y[:n], pl)
        gy_ref, gw_ref = oracle.combine_backward(go, y[:n], pl, wts, zero_pad=True)
    assert_bits_equal(gx, gx_ref, "grad_x")
    assert_bits_equal(gy1[:n], gy_ref, "grad_y")
    assert torch.all(gy1[n:] == 9.0)
    bound = _grad_w_bound_gpu(go_t, y_t, pl.slot, w.H)
    err = (gw1.double() - torch.from_numpy(gw_ref).cuda()).abs()
    assert torch.all(err <= bound), float((err - bound).max())
    assert torch.all(gw1[torch.from_numpy(pl.slot < 0).cuda()] == 0)


def test_backward_capacity_errors():
    w = WORKLOADS["tiny"]
    idx, wts = draw_topk(w)
    h = ep.plan(torch.from_numpy(idx).cuda(), w.P, w.E, w.A)
    n_exp = h.sizes()[0]
    small = torch.zeros((n_exp // 2, w.H), dtype=torch.bfloat16, device="cuda")
    ep.dispatch_backward(h, small)
    assert h.sync_status() == ep.EP_ERR_CAPACITY
    go = torch.zeros((w.T, w.H), dtype=torch.bfloat16, device="cuda")
    ep.combine_backward(h, go, small, torch.from_numpy(wts).cuda())
    assert h.sync_status() == ep.EP_ERR_CAPACITY
