"""Pins of the oracle on non-finite hidden values.

The pages (TileLang tutorial ch. 38 "DeepEP-Ascend", §3.6: one fp32 scale per
128 hidden elements, amax/448) define no behaviour for Inf or NaN in x.  The
reading taken, which the CUDA path shares:

  * amax of a group is the largest |x| over its non-NaN elements (0 if it has
    none), so a NaN element does not move the group's scale;
  * an infinite element makes amax and the scale +inf: the group's finite
    elements give signed zero codes (x/inf) and the infinite one NaN (inf/inf);
  * every NaN quotient encodes as 0x7F, S.1111.111 with the sign bit clear:
    IEEE arithmetic leaves the sign of a NaN result open, and x86 and Arm
    hosts give different ones for inf/inf, so the reading fixes it;
  * amax == 0 (a group of zeros and NaNs) keeps scale 0 and code 0 for every
    element;
  * BF16 dispatch is a bit copy (any bit pattern passes through), and the
    combine is IEEE fp32 arithmetic, whose NaN results may be any bf16 NaN.

The FP8 pins restate the reading with numpy fp32 division and torch's E4M3
cast (independent of the oracle's own encoder), and add invariants: a NaN
element changes no other code and not the scale.  CPU only.
"""
import ctypes
import struct

import numpy as np
import pytest
import torch

import oracle
from combine_ep_plan_gb300.inputs import WORKLOADS, draw_hidden, draw_topk, hidden_seed

NAN_BITS = [0x7FC00000, 0xFFC00000, 0x7F800001, 0xFF800001, 0x7FFFFFFF, 0xFFFFFFFF, 0x7FA00000, 0xFFA00000]


def _f32_from_bits(b: int) -> float:
    return struct.unpack("<f", struct.pack("<I", b))[0]


def _bf16_bits(vals) -> np.ndarray:
    return torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _bf16_f32(bits: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).float().numpy()


@pytest.mark.parametrize("bits", NAN_BITS, ids=hex)
def test_every_nan_encodes_as_0x7f(bits):
    assert oracle.f32_to_e4m3(_f32_from_bits(bits)) == 0x7F


def test_inf_over_inf_encodes_as_0x7f_on_this_host():
    # the host's inf/inf carries whatever sign its FPU gives a default NaN
    q = ctypes.c_float(float("inf")).value / ctypes.c_float(float("inf")).value
    assert np.isnan(q)
    assert oracle.f32_to_e4m3(q) == 0x7F


def _restated_fp8(x_bits: np.ndarray):
    """The reading, row by row: numpy amax and fp32 division, torch's E4M3 cast,
    NaN quotients forced to 0x7F."""
    x = _bf16_f32(x_bits).reshape(x_bits.shape[0], -1, 128)
    ax = np.abs(x)
    amax = np.where(np.isnan(ax), -np.inf, ax).max(axis=2)
    amax = np.where(amax == -np.inf, 0.0, amax).astype(np.float32)
    scale = (amax / np.float32(448.0)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        quot = (x / scale[:, :, None]).astype(np.float32)
    q = torch.from_numpy(np.ascontiguousarray(quot)).to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()
    q[np.isnan(quot)] = 0x7F
    q[np.broadcast_to(amax[:, :, None] == 0, q.shape)] = 0x00
    return q.reshape(x_bits.shape), scale


def _special_rows(H: int, rng) -> np.ndarray:
    """Rows of N(0,1) values with non-finite elements planted in chosen groups."""
    G = H // 128
    base = rng.standard_normal((12, H)).astype(np.float32)
    nan, inf = float("nan"), float("inf")
    rows = base.copy()
    rows[0, 5] = nan                                  # one NaN among finite values
    rows[1, 7] = -nan                                 # a negative NaN
    rows[2, 3] = inf                                  # +inf: scale inf, others signed zeros
    rows[3, 9] = -inf                                 # -inf: the same scale (amax of |x|)
    rows[4, :128] = nan                               # a group of NaNs only: amax 0
    rows[5, :128] = 0.0
    rows[5, 17] = nan                                 # zeros and one NaN: amax 0
    rows[6, 0], rows[6, 1], rows[6, 2] = inf, -inf, nan  # inf, -inf and NaN together
    rows[7, 4] = -0.0
    rows[7, 5] = inf                                  # -0 next to inf: code 0x80
    if G > 1:
        rows[8, 128 + 11] = nan                        # a NaN in the second group only
        rows[9, 128:256] = -inf                        # a group of -inf
    rows[10, :128] = 2.0 ** -130 * rows[10, :128]      # subnormal bf16 values ...
    rows[10, 1] = nan                                  # ... and a NaN
    rows[11, 0] = 3.3895314e38                         # the largest finite bf16 ...
    rows[11, 1] = nan                                  # ... and a NaN
    return _bf16_bits(rows)


def _plan_for(T_rows: int):
    w = WORKLOADS["tiny"].scaled(P=1, E=2, S=T_rows, K=1, A=1)
    idx = np.zeros((T_rows, 1), np.int64)
    return oracle.plan(idx, w.S, w.P, w.E, w.A)


@pytest.mark.parametrize("H", [128, 256])
def test_fp8_dispatch_non_finite_rows_follow_the_reading(H):
    rng = np.random.default_rng(17)
    x = _special_rows(H, rng)
    pl = _plan_for(x.shape[0])  # identity layout: expanded row r = token r
    q, sc = oracle.dispatch_fp8(x, pl, True)
    q_ref, sc_ref = _restated_fp8(x)
    assert np.array_equal(sc.view(np.uint32), sc_ref.view(np.uint32))
    assert np.array_equal(q, q_ref)
    # spot values the reading names
    assert q[0, 5] == 0x7F and q[1, 7] == 0x7F
    assert np.isinf(sc[2, 0]) and sc[2, 0] > 0 and np.isinf(sc[3, 0]) and sc[3, 0] > 0
    assert q[2, 3] == 0x7F and q[3, 9] == 0x7F
    assert set(np.unique(q[2, :128])) <= {0x00, 0x80, 0x7F}
    assert sc[4, 0] == 0 and not q[4, :128].any()
    assert sc[5, 0] == 0 and not q[5, :128].any()
    assert q[7, 4] == 0x80
    assert q[10, 1] == 0x7F and q[11, 1] == 0x7F


def test_a_nan_element_moves_nothing_else():
    rng = np.random.default_rng(23)
    H = 256
    x = _bf16_bits(rng.standard_normal((6, H)).astype(np.float32))
    y = x.copy()
    # in each row, the element of least magnitude of one group: never the group's amax
    xf = np.abs(_bf16_f32(x))
    spots = [(r, (r % 2) * 128 + int(np.argmin(xf[r, (r % 2) * 128:(r % 2) * 128 + 128]))) for r in range(6)]
    for r, c in spots:
        y[r, c] = 0xFFC0 if r % 2 else 0x7FC0  # NaN of either sign
    pl = _plan_for(6)
    qx, sx = oracle.dispatch_fp8(x, pl, True)
    qy, sy = oracle.dispatch_fp8(y, pl, True)
    # the NaN element was not the group's amax in x: scales are unchanged
    ax = np.abs(_bf16_f32(x)).reshape(6, -1, 128).max(axis=2)
    for r, c in spots:
        assert np.abs(_bf16_f32(x))[r, c] < ax[r, c // 128]
    assert np.array_equal(sx.view(np.uint32), sy.view(np.uint32))
    diff = np.argwhere(qx != qy)
    assert sorted(map(tuple, diff.tolist())) == sorted(spots)
    assert all(qy[r, c] == 0x7F for r, c in spots)


def test_bf16_dispatch_copies_non_finite_bits():
    rng = np.random.default_rng(5)
    x = _special_rows(256, rng)
    x[0, 9] = 0xFF81  # a negative signalling-NaN pattern: bits pass through untouched
    pl = _plan_for(x.shape[0])
    assert np.array_equal(oracle.dispatch_bf16(x, pl, True), x)


def test_combine_non_finite_follows_ieee():
    w = WORKLOADS["tiny"].scaled(S=16, H=256)
    idx, wts = draw_topk(w)
    x = draw_hidden(w.T, w.H, hidden_seed(w))
    pl = oracle.plan(idx, w.S, w.P, w.E, w.A)
    y = oracle.dispatch_bf16(x, pl, True)
    y[0, :8] = _bf16_bits([float("nan"), float("inf"), float("-inf"), float("inf"), 1.0, 2.0, 3.0, 4.0])
    # a token with two valid slots: +inf in one row and -inf in the other meet in its sum
    g = int(np.nonzero((pl.slot >= 0).sum(axis=1) >= 2)[0][0])
    r1, r2 = (int(r) for r in pl.slot[g][pl.slot[g] >= 0][:2])
    y[r1, 20] = _bf16_bits([float("inf")])[0]
    y[r2, 20] = _bf16_bits([float("-inf")])[0]
    out = _bf16_f32(oracle.combine(y, pl, wts))
    # float64 restatement of the sums: only the non-finite pattern is compared
    yf = _bf16_f32(y).astype(np.float64)
    ref = np.zeros((pl.T, w.H))
    with np.errstate(invalid="ignore"):
        for t in range(pl.T):
            for k in range(pl.K):
                if pl.slot[t, k] >= 0:
                    ref[t] += np.float64(wts[t, k]) * yf[pl.slot[t, k]]
    assert np.array_equal(np.isnan(out), np.isnan(ref))
    assert np.array_equal(np.isposinf(out), np.isposinf(ref))
    assert np.array_equal(np.isneginf(out), np.isneginf(ref))
    assert np.isnan(out).any() and np.isinf(out).any()
    assert np.isnan(out[g, 20])
