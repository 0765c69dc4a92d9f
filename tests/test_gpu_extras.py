"""GPU parity of the metadata-carrying dispatch, pre-quantised FP8 input,
column-major FP8 scales and the combine bias, against the oracle."""
import numpy as np
import pytest
import torch

import combine_ep_plan_gb300 as ep
import oracle
from combine_ep_plan_gb300.inputs import WORKLOADS, bits_to_bf16_tensor, draw_hidden, draw_topk, draw_y, hidden_seed
from ep_testutil import u8, u16

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
    WORKLOADS["zipf"].scaled(S=13, H=512),
]


def _setup(w):
    idx, wts = draw_topk(w)
    idx[::4, 0] = -1
    pl = oracle.plan(idx, w.S, w.P, w.E, w.A)
    h = ep.plan(torch.from_numpy(idx).cuda(), w.P, w.E, w.A)
    return idx, wts, pl, h


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_combine_bias(w):
    idx, wts, pl, h = _setup(w)
    y = draw_y(pl.num_expanded, w.H, 41)
    bias = draw_y(w.T, w.H, 42)
    ref = oracle.combine(y, pl, wts, bias)
    out = ep.combine(h, bits_to_bf16_tensor(y).cuda(), torch.from_numpy(wts).cuda(),
                     bias=bits_to_bf16_tensor(bias).cuda())
    assert h.sync_status() == ep.EP_OK
    assert np.array_equal(u16(out), ref)


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_dispatch_metadata(w):
    idx, wts, pl, h = _setup(w)
    rw_ref, rm_ref = oracle.dispatch_metadata(pl, wts)
    cap = pl.num_expanded + 3
    rw_buf = torch.full((cap,), 5.0, dtype=torch.float32, device="cuda")
    rm_buf = torch.full((cap, 2), 7, dtype=torch.int32, device="cuda")
    rw, rm = ep.dispatch_metadata(h, torch.from_numpy(wts).cuda(), recv_weights=rw_buf, recv_meta=rm_buf)
    assert h.sync_status() == ep.EP_OK
    n = pl.num_expanded
    assert np.array_equal(rw.cpu().numpy()[:n].view(np.uint32), rw_ref.view(np.uint32))
    assert np.array_equal(rm.cpu().numpy()[:n], rm_ref)
    assert np.all(rw.cpu().numpy()[n:] == 5.0) and np.all(rm.cpu().numpy()[n:] == 7)


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
@pytest.mark.parametrize("col_major", [False, True])
def test_fp8_input_passthrough(w, col_major):
    w = w.scaled(H=max(w.H, 128) // 128 * 128)
    idx, wts, pl, h = _setup(w)
    rng = np.random.default_rng(2)
    xq = rng.integers(0, 256, size=(w.T, w.H), dtype=np.uint8)
    xq[(xq & 0x7F) == 0x7F] = 0  # no NaN codes in the input
    xs = rng.standard_normal((w.T, w.H // 128)).astype(np.float32)
    q_ref, s_ref = oracle.dispatch_fp8_input(xq, xs, pl)
    xq_t = torch.from_numpy(xq).cuda().view(torch.float8_e4m3fn)
    recv, sc = ep.dispatch(h, xq_t, "fp8", True, x_scales=torch.from_numpy(xs).cuda(), scales_col_major=col_major)
    assert h.sync_status() == ep.EP_OK
    assert np.array_equal(u8(recv), q_ref)
    assert sc.shape == (pl.num_expanded, w.H // 128)
    if col_major:
        assert sc.stride() == (1, pl.num_expanded)
    assert np.array_equal(sc.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))


@pytest.mark.parametrize("w", CASES[1:], ids=lambda w: w.name)
def test_fp8_quantise_column_major_scales(w):
    w = w.scaled(H=max(w.H, 128) // 128 * 128)
    idx, wts, pl, h = _setup(w)
    x = draw_hidden(w.T, w.H, hidden_seed(w))
    q_ref, s_ref = oracle.dispatch_fp8(x, pl)
    cap = ep.worst_expanded_rows(w.T, w.K, w.E, w.A)
    recv, sc = ep.dispatch(h, bits_to_bf16_tensor(x).cuda(), "fp8", True, capacity=cap, scales_col_major=True)
    assert h.sync_status() == ep.EP_OK
    assert sc.stride() == (1, cap)
    n = pl.num_expanded
    assert np.array_equal(u8(recv)[:n], q_ref)
    assert np.array_equal(sc[:n].cpu().numpy().view(np.uint32), s_ref.view(np.uint32))


def test_quantise_then_dispatch_equals_fused_on_gpu():
    """Per-token quantisation (a dispatch with the identity plan) followed by
    the pre-quantised dispatch gives the same rows as the fused quantise."""
    w = CASES[1].scaled(H=1024)
    idx, wts, pl, h = _setup(w)
    x = bits_to_bf16_tensor(draw_hidden(w.T, w.H, hidden_seed(w))).cuda()
    ident_idx = torch.full((w.T, 1), 0, dtype=torch.int64, device="cuda")
    hi = ep.plan(ident_idx, 1, 1, 1)  # one expert on one rank: row r is token r
    xq, xs = ep.dispatch(hi, x, "fp8", True)
    a_q, a_s = ep.dispatch(h, xq, "fp8", True, x_scales=xs)
    b_q, b_s = ep.dispatch(h, x, "fp8", True)
    assert h.sync_status() == ep.EP_OK and hi.sync_status() == ep.EP_OK
    assert torch.equal(a_q.view(torch.uint8), b_q.view(torch.uint8)) and torch.equal(a_s, b_s)
