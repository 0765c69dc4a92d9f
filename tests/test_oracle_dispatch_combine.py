"""Pins of the oracle's dispatch (BF16, FP8) and combine.

Dispatch is checked by vectorised numpy gathers and torch's float8 cast,
combine by closed forms (identity and scaling experts) evaluated in float64.
"""
import numpy as np
import pytest
import torch

import oracle
from combine_ep_plan_gb300.inputs import WORKLOADS, draw_hidden, draw_topk, draw_y, hidden_seed

CASES = [
    WORKLOADS["tiny"],
    WORKLOADS["bf16"].scaled(S=48, H=384),
    WORKLOADS["fp8"].scaled(S=24, H=512),
    WORKLOADS["zipf"].scaled(S=4, H=256),
    WORKLOADS["rt"].scaled(S=12, H=256),
]


def _bf16_to_f32(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).float().numpy()


def _f32_to_bf16_bits(v):
    return torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _setup(w):
    idx, wts = draw_topk(w)
    x = draw_hidden(w.T, w.H, hidden_seed(w))
    pl = oracle.plan(idx, w.S, w.P, w.E, w.A)
    return idx, wts, x, pl


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
@pytest.mark.parametrize("zero_pad", [True, False])
def test_bf16_dispatch_is_a_row_gather(w, zero_pad):
    idx, wts, x, pl = _setup(w)
    out = oracle.dispatch_bf16(x, pl, zero_pad)
    real = pl.exp_src >= 0
    assert np.array_equal(out[real], x[pl.exp_src[real]])
    if zero_pad:
        assert not out[~real].any()
    # ledger: bytes of real rows = valid (token, slot) pairs * H * 2
    assert real.sum() * w.H * 2 == int(np.sum(idx >= 0)) * w.H * 2


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_fp8_dispatch_matches_numpy_and_torch_cast(w):
    idx, wts, x, pl = _setup(w)
    q, sc = oracle.dispatch_fp8(x, pl)
    real = pl.exp_src >= 0
    xf = _bf16_to_f32(x).reshape(w.T, w.H // 128, 128)
    amax = np.abs(xf).max(axis=2)
    scale = (amax / np.float32(448.0)).astype(np.float32)  # IEEE fp32 division
    assert np.array_equal(sc[real], scale[pl.exp_src[real]])
    ratio = np.where(amax[..., None] > 0, xf / np.where(scale > 0, scale, 1)[..., None], 0).astype(np.float32)
    ref = torch.from_numpy(ratio.reshape(w.T, w.H)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(q[real], ref[pl.exp_src[real]])
    assert not q[~real].any() and not sc[~real].any()
    # every non-zero group reaches the top code 448 at its amax element
    dec = torch.from_numpy(q[real]).view(torch.float8_e4m3fn).float().numpy().reshape(-1, w.H // 128, 128)
    assert np.all(np.abs(dec).max(axis=2)[sc[real] > 0] == 448.0)


def test_fp8_dequant_error_bound():
    w = CASES[2]
    idx, wts, x, pl = _setup(w)
    q, sc = oracle.dispatch_fp8(x, pl)
    real = pl.exp_src >= 0
    dec = torch.from_numpy(q[real]).view(torch.float8_e4m3fn).float().numpy().reshape(-1, w.H // 128, 128)
    xr = _bf16_to_f32(x[pl.exp_src[real]]).reshape(-1, w.H // 128, 128)
    s = sc[real][..., None].astype(np.float64)
    err = np.abs(dec * s - xr)
    # half a unit in the last place of E4M3 (3 fraction bits) relative to the
    # value, plus half the subnormal spacing 2^-9 in units of the scale
    bound = 2.0 ** -4 * np.abs(xr) * (1 + 1e-6) + 2.0 ** -10 * s * (1 + 1e-6)
    assert np.all(err <= bound)


def test_fp8_dequant_expert_matches_library_casts():
    """The dequantising identity expert, y = bf16_RNE(float(q) * scale of the
    element's group), against torch's E4M3 decode and bf16 cast on the FP8
    rows of a dispatch; it also stays within the E4M3 bound of the source
    rows plus one bf16 rounding."""
    w = CASES[2]
    idx, wts, x, pl = _setup(w)
    q, sc = oracle.dispatch_fp8(x, pl)
    y = oracle.expert_dequant(q, sc)
    G = w.H // 128
    dec = torch.from_numpy(q).view(torch.float8_e4m3fn).float().numpy().reshape(-1, G, 128)
    prod = (dec * sc[..., None]).astype(np.float32).reshape(-1, w.H)  # one fp32 product
    assert np.array_equal(y, _f32_to_bf16_bits(prod))
    real = pl.exp_src >= 0
    yr = _bf16_to_f32(y[real]).reshape(-1, G, 128).astype(np.float64)
    xr = _bf16_to_f32(x[pl.exp_src[real]]).reshape(-1, G, 128)
    s = sc[real][..., None].astype(np.float64)
    bound = (2.0 ** -4 * np.abs(xr) + 2.0 ** -10 * s) * (1 + 1e-6) + 2.0 ** -8 * np.abs(yr)
    assert np.all(np.abs(yr - xr) <= bound)
    assert not y[~real].any()


def test_fp8_zero_group_special_case():
    w = WORKLOADS["tiny"].scaled(H=256)
    idx, wts, x, pl = _setup(w)
    x = x.copy()
    x[3, :128] = 0          # an all-zero group: amax == 0
    x[5, 128:] = 0x8000     # negative zeros
    q, sc = oracle.dispatch_fp8(x, pl)
    for g, j in [(3, 0), (5, 1)]:
        rows = pl.slot[g][pl.slot[g] >= 0]
        assert len(rows) and np.all(sc[rows, j] == 0) and not q[rows, j * 128:(j + 1) * 128].any()


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_identity_round_trip(w):
    """Combine is the inverse of dispatch (tutorial ch. 38 §2.3): an identity
    expert and weights that sum to one give back x, within the bf16 bound."""
    idx, wts, x, pl = _setup(w)
    y = oracle.dispatch_bf16(x, pl)
    out = oracle.combine(y, pl, wts)
    xf = _bf16_to_f32(x).astype(np.float64)
    got = _bf16_to_f32(out).astype(np.float64)
    wsum = np.where(idx >= 0, wts, 0).sum(1, dtype=np.float64)[:, None]
    assert np.allclose(got, xf * wsum, rtol=8e-3, atol=1e-2)


def test_single_slot_unit_weight_is_exact():
    w = WORKLOADS["tiny"].scaled(K=1)
    idx, wts, x, pl = _setup(w)
    ones = np.ones_like(wts)
    out = oracle.combine(oracle.dispatch_bf16(x, pl), pl, ones)
    assert np.array_equal(out, x)


def test_unit_weights_sum_is_exact():
    """With all weights 1 the fp32 accumulation of k copies of a bf16 value is
    exact, so the result is bf16_RNE(k * x) in closed form."""
    w = WORKLOADS["rt"].scaled(S=8, H=128)
    idx, wts, x, pl = _setup(w)
    idx_k = (idx >= 0).sum(1)
    out = oracle.combine(oracle.dispatch_bf16(x, pl), pl, np.ones_like(wts))
    ref = _f32_to_bf16_bits(_bf16_to_f32(x) * idx_k[:, None].astype(np.float32))
    assert np.array_equal(out, ref)


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_scale_expert_round_trip(w):
    """y = bf16(x * (1 + e/E)) per expert, then weighted combine: compare with
    the same sum evaluated in float64."""
    idx, wts, x, pl = _setup(w)
    y = oracle.expert_scale(oracle.dispatch_bf16(x, pl), pl)
    out = _bf16_to_f32(oracle.combine(y, pl, wts)).astype(np.float64)
    xf = _bf16_to_f32(x)
    ref = np.zeros((w.T, w.H), np.float64)
    for k in range(w.K):
        e = idx[:, k]
        f = (np.float32(1.0) + e.astype(np.float32) / np.float32(w.E)).astype(np.float32)
        yk = _bf16_to_f32(_f32_to_bf16_bits(xf * f[:, None])).astype(np.float64)
        ref += np.where(e[:, None] >= 0, wts[:, k:k + 1].astype(np.float64) * yk, 0)
    assert np.allclose(out, ref, rtol=8e-3, atol=1e-2)


def test_combine_random_y_matches_float64():
    w = CASES[1]
    idx, wts, x, pl = _setup(w)
    y = draw_y(pl.num_expanded, w.H, 77)
    out = _bf16_to_f32(oracle.combine(y, pl, wts)).astype(np.float64)
    yf = _bf16_to_f32(y).astype(np.float64)
    ref = np.zeros((w.T, w.H))
    for k in range(w.K):
        r = pl.slot[:, k]
        ref += np.where(r[:, None] >= 0, wts[:, k:k + 1] * yf[np.maximum(r, 0)], 0)
    assert np.allclose(out, ref, rtol=8e-3, atol=1e-2)


def test_combine_token_without_slots_is_zero():
    w = WORKLOADS["tiny"]
    idx, wts, x, _ = _setup(w)
    idx[10, :] = -1
    pl = oracle.plan(idx, w.S, w.P, w.E, w.A)
    out = oracle.combine(oracle.dispatch_bf16(x, pl), pl, wts)
    assert not out[10].any()


def test_expert_scale_rows_matches_segment_form():
    w = CASES[4]
    idx, wts, x, pl = _setup(w)
    xe = oracle.dispatch_bf16(x, pl)
    seg = oracle.expert_scale(xe, pl)
    rows = np.arange(pl.num_expanded)
    e_of_row = (np.searchsorted(pl.expert_offsets, rows, side="right") - 1).astype(np.int32)
    e_of_row[pl.exp_src < 0] = -1
    assert np.array_equal(oracle.expert_scale_rows(xe, e_of_row, w.E), seg)
