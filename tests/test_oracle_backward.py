"""Pins of the oracle's backward on the same handle (tutorial ch. 38 §2.3):
torch autograd through the forward written with index operations in
float64, and the adjoint identities of the linear maps."""
import numpy as np
import pytest
import torch

import oracle
from combine_ep_plan_gb300.inputs import WORKLOADS, draw_hidden, draw_topk, draw_y, hidden_seed

CASES = [WORKLOADS["tiny"], WORKLOADS["rt"].scaled(S=10, H=128), WORKLOADS["zipf"].scaled(S=3, H=256)]


def _f64(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).double()


def _setup(w, with_unused=True):
    idx, wts = draw_topk(w)
    if with_unused:
        idx[::5, -1] = -1
    pl = oracle.plan(idx, w.S, w.P, w.E, w.A)
    return idx, wts, pl


def _autograd(pl, idx, wts, x_bits, y_bits, grad_out_bits, grad_recv_bits):
    """Forward of dispatch and combine with gathers, differentiated by torch."""
    T, K = pl.slot.shape
    valid = torch.from_numpy(pl.slot >= 0)
    rows = torch.from_numpy(np.maximum(pl.slot, 0)).long()
    x = _f64(x_bits).requires_grad_(True)
    recv = torch.zeros(pl.num_expanded, x.shape[1], dtype=torch.float64)
    src = torch.from_numpy(pl.exp_src).long()
    recv = torch.where((src >= 0)[:, None], x[src.clamp(min=0)], recv)
    (recv * _f64(grad_recv_bits)).sum().backward()
    y = _f64(y_bits).requires_grad_(True)
    w = torch.from_numpy(wts).double().requires_grad_(True)
    out = (torch.where(valid[..., None], w[..., None] * y[rows], torch.zeros(1, dtype=torch.float64))).sum(1)
    (out * _f64(grad_out_bits)).sum().backward()
    return x.grad, y.grad, w.grad


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_backward_matches_autograd(w):
    idx, wts, pl = _setup(w)
    x = draw_hidden(w.T, w.H, hidden_seed(w))
    y = draw_y(pl.num_expanded, w.H, 5)
    go = draw_y(w.T, w.H, 6)
    gr = draw_y(pl.num_expanded, w.H, 7)
    gx_ref, gy_ref, gw_ref = _autograd(pl, idx, wts, x, y, go, gr)
    gx = _f64(oracle.dispatch_backward(gr, pl))
    gy, gw = oracle.combine_backward(go, y, pl, wts, zero_pad=True)
    # grad_x: fp32 sum of up to K bf16 values, rounded once to bf16
    assert torch.allclose(gx, gx_ref, rtol=8e-3, atol=1e-2)
    # grad_y: one fp32 product rounded to bf16 (half a bf16 ulp)
    real = torch.from_numpy(pl.exp_src >= 0)
    assert torch.allclose(_f64(gy)[real], gy_ref[real], rtol=2 ** -8, atol=0)
    assert not _f64(gy)[~real].any()
    # grad_w: the same dot product in float64
    assert np.allclose(gw, gw_ref.numpy(), rtol=1e-12, atol=1e-9)
    assert np.all(gw[pl.slot < 0] == 0)


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_adjoint_identities(w):
    """<dispatch(x), r> = <x, dispatch_backward(r)> and
    <combine(y), o> = <y, combine_backward_y(o)>, up to the bf16 roundings."""
    idx, wts, pl = _setup(w)
    x = draw_hidden(w.T, w.H, hidden_seed(w))
    r = draw_y(pl.num_expanded, w.H, 8)
    lhs = (_f64(oracle.dispatch_bf16(x, pl)) * _f64(r)).sum()
    rhs = (_f64(x) * _f64(oracle.dispatch_backward(r, pl))).sum()
    scale = (_f64(x).abs() * _f64(oracle.dispatch_backward(r, pl)).abs()).sum()
    assert abs(lhs - rhs) <= 1e-2 * scale
    y = draw_y(pl.num_expanded, w.H, 9)
    o = draw_y(w.T, w.H, 10)
    gy, _ = oracle.combine_backward(o, y, pl, wts)
    lhs = (_f64(oracle.combine(y, pl, wts)) * _f64(o)).sum()
    rhs = (_f64(y) * _f64(gy)).sum()
    scale = (_f64(y).abs() * _f64(gy).abs()).sum()
    assert abs(lhs - rhs) <= 1e-2 * scale


def test_dispatch_backward_single_slot_is_the_gradient_row():
    w = WORKLOADS["tiny"].scaled(K=1)
    idx, wts, pl = _setup(w, with_unused=False)
    gr = draw_y(pl.num_expanded, w.H, 11)
    # one slot per token: the token's gradient is its row, bit for bit
    assert np.array_equal(oracle.dispatch_backward(gr, pl), gr[pl.slot[:, 0]])
