"""GPU parity at the implementation's limits: P = EP_MAX_RANKS (1024),
E = EP_MAX_EXPERTS (2048), K = EP_MAX_TOPK (16), and hidden sizes that leave
partial work chunks; against the oracle."""
import numpy as np
import pytest
import torch

import combine_ep_plan_gb300 as ep
import oracle
from combine_ep_plan_gb300.inputs import WORKLOADS, bits_to_bf16_tensor, draw_hidden, draw_topk, hidden_seed
from ep_testutil import assert_plan_equal, gpu_plan_arrays, u8, u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from combine_ep_plan_gb300 import build
    build.build()
    ep.load_library()
    yield
    torch.cuda.synchronize()


def _round_trip(w, out_dtype="bf16"):
    idx, wts = draw_topk(w)
    x = draw_hidden(w.T, w.H, hidden_seed(w))
    pl = oracle.plan(idx, w.S, w.P, w.E, w.A)
    h = ep.plan(torch.from_numpy(idx).cuda(), w.P, w.E, w.A)
    assert_plan_equal(gpu_plan_arrays(h), pl)
    xt = bits_to_bf16_tensor(x).cuda()
    if out_dtype == "fp8":
        q, sc = ep.dispatch(h, xt, "fp8")
        q_ref, s_ref = oracle.dispatch_fp8(x, pl)
        assert np.array_equal(u8(q), q_ref)
        assert np.array_equal(sc.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
    recv, _ = ep.dispatch(h, xt, "bf16")
    ref = oracle.dispatch_bf16(x, pl)
    assert np.array_equal(u16(recv), ref)
    out = ep.combine(h, recv, torch.from_numpy(wts).cuda())
    assert np.array_equal(u16(out), oracle.combine(ref, pl, wts))
    assert h.sync_status() == ep.EP_OK


def test_max_ranks_experts_topk():
    # 1024 ranks x 2 experts each, 16 distinct experts per token
    _round_trip(WORKLOADS["zipf"].scaled(P=1024, E=2048, S=4, K=16, H=256, A=8))


def test_max_topk_uniform_wide_hidden():
    _round_trip(WORKLOADS["bf16"].scaled(P=16, E=64, S=64, K=16, H=8192, A=16), out_dtype="fp8")


@pytest.mark.parametrize("H", [128, 384, 2176, 16384])
def test_fp8_partial_chunks(H):
    # the FP8 item covers 2048 elements: H = 2176 leaves a one-group tail
    _round_trip(WORKLOADS["fp8"].scaled(S=8, H=H), out_dtype="fp8")


@pytest.mark.parametrize("H", [8, 24, 1032])
def test_bf16_small_and_ragged_hidden(H):
    # rows of 1, 3 and 129 16-byte vectors
    _round_trip(WORKLOADS["tiny"].scaled(H=H))


def test_one_token_per_rank():
    _round_trip(WORKLOADS["rt"].scaled(S=1, H=256))


@pytest.mark.parametrize("H", [128, 4224, 16384, 16512])
def test_fp8_input_scale_group_counts(H):
    """Pre-quantised input with 1, 33, 128 and 129 scale groups per row: the
    scales of a row are held in registers up to 128 groups, beyond that the
    rest is read again per destination; row- and column-major scales."""
    w = WORKLOADS["fp8"].scaled(S=6, H=H)
    idx, _ = draw_topk(w)
    pl = oracle.plan(idx, w.S, w.P, w.E, w.A)
    h = ep.plan(torch.from_numpy(idx).cuda(), w.P, w.E, w.A)
    rng = np.random.default_rng(H)
    xq = rng.integers(0, 256, size=(w.T, H), dtype=np.uint8)
    xq[(xq & 0x7F) == 0x7F] = 0  # no NaN codes in the input
    xs = rng.standard_normal((w.T, H // 128)).astype(np.float32)
    q_ref, s_ref = oracle.dispatch_fp8_input(xq, xs, pl)
    xq_t = torch.from_numpy(xq).cuda().view(torch.float8_e4m3fn)
    for col_major in (False, True):
        recv, sc = ep.dispatch(h, xq_t, "fp8", True, x_scales=torch.from_numpy(xs).cuda(), scales_col_major=col_major)
        assert h.sync_status() == ep.EP_OK
        assert np.array_equal(u8(recv), q_ref)
        assert np.array_equal(sc.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))


def test_a_million_tokens():
    """2^20 tokens (8 ranks x 131072, 4096 tiles, about 6.3 M expanded rows):
    every plan array, the BF16 dispatch and the combine at H = 8, against the
    oracle, whole arrays."""
    w = WORKLOADS["bf16"].scaled(S=131072, H=8)
    idx, wts = draw_topk(w)
    idx[::9, 2] = -1
    with oracle.parallel():
        pl = oracle.plan(idx, w.S, w.P, w.E, w.A)
        h = ep.plan(torch.from_numpy(idx).cuda(), w.P, w.E, w.A)
        assert_plan_equal(gpu_plan_arrays(h), pl)
        x = draw_hidden(w.T, w.H, hidden_seed(w))
        recv, _ = ep.dispatch(h, bits_to_bf16_tensor(x).cuda(), "bf16", True)
        ref = oracle.dispatch_bf16(x, pl, True)
        assert np.array_equal(u16(recv), ref)
        out = ep.combine(h, recv, torch.from_numpy(wts).cuda())
        assert np.array_equal(u16(out), oracle.combine(ref, pl, wts))
    assert h.sync_status() == ep.EP_OK
