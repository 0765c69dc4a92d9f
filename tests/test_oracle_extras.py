"""Pins of the oracle's metadata-carrying dispatch, pre-quantised FP8 input
and combine bias."""
import numpy as np
import pytest
import torch

import oracle
from combine_ep_plan_gb300.inputs import WORKLOADS, draw_hidden, draw_topk, draw_y, hidden_seed

CASES = [WORKLOADS["tiny"], WORKLOADS["bf16"].scaled(S=40, H=256), WORKLOADS["zipf"].scaled(S=3, H=256)]


def _setup(w):
    idx, wts = draw_topk(w)
    idx[::4, 0] = -1
    return idx, wts, oracle.plan(idx, w.S, w.P, w.E, w.A)


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_metadata_by_definition(w):
    idx, wts, pl = _setup(w)
    rw, rm = oracle.dispatch_metadata(pl, wts)
    real = pl.exp_src >= 0
    assert np.array_equal(rm[real, 0], pl.exp_src[real])  # the source token of each row
    g, k = rm[real, 0], rm[real, 1]
    assert np.array_equal(pl.slot[g, k], np.nonzero(real)[0])  # the (g,k) that owns the row
    assert np.array_equal(rw[real], wts[g, k])
    assert np.all(rm[~real] == -1) and np.all(rw[~real] == 0)


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_fp8_input_is_a_row_gather(w):
    idx, wts, pl = _setup(w)
    rng = np.random.default_rng(1)
    xq = rng.integers(0, 256, size=(w.T, w.H), dtype=np.uint8)
    xs = rng.standard_normal((w.T, w.H // 128)).astype(np.float32)
    oq, osc = oracle.dispatch_fp8_input(xq, xs, pl)
    real = pl.exp_src >= 0
    assert np.array_equal(oq[real], xq[pl.exp_src[real]])
    assert np.array_equal(osc[real], xs[pl.exp_src[real]])
    assert not oq[~real].any() and not osc[~real].any()


def test_fp8_input_round_trip_equals_fused_quantisation():
    # quantising first and dispatching the codes gives the same rows as the
    # dispatch that quantises inside
    w = CASES[1]
    idx, wts, pl = _setup(w)
    x = draw_hidden(w.T, w.H, hidden_seed(w))
    ident = oracle.Plan(**{**pl.__dict__, "exp_src": np.arange(w.T, dtype=np.int32),
                           "expert_offsets": np.array([0, w.T], np.int32)})
    xq, xs = oracle.dispatch_fp8(x, ident)  # per-token quantisation
    a = oracle.dispatch_fp8_input(xq, xs, pl)
    b = oracle.dispatch_fp8(x, pl)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_combine_bias(w):
    idx, wts, pl = _setup(w)
    y = draw_y(pl.num_expanded, w.H, 3)
    bias = draw_y(w.T, w.H, 4)
    # zero weights: the output is the bias itself
    assert np.array_equal(oracle.combine(y, pl, np.zeros_like(wts), bias), bias)
    # without bias argument, bias = 0 gives the plain combine bit for bit
    assert np.array_equal(oracle.combine(y, pl, wts, np.zeros_like(bias)), oracle.combine(y, pl, wts))
    # float64 closed form
    out = torch.from_numpy(oracle.combine(y, pl, wts, bias).view(np.int16)).view(torch.bfloat16).double().numpy()
    yf = torch.from_numpy(y.view(np.int16)).view(torch.bfloat16).double().numpy()
    bf = torch.from_numpy(bias.view(np.int16)).view(torch.bfloat16).double().numpy()
    ref = bf.copy()
    for k in range(w.K):
        r = pl.slot[:, k]
        ref += np.where(r[:, None] >= 0, wts[:, k:k + 1] * yf[np.maximum(r, 0)], 0)
    assert np.allclose(out, ref, rtol=8e-3, atol=1e-2)
