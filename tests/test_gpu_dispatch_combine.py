"""GPU parity of dispatch (BF16 bit copy, FP8 E4M3 quantised inside dispatch)
and combine, against the oracle: element by element on cases that span
several tiles with a ragged tail, and on sampled rows/tokens at the full
workload sizes in the launch configuration the benchmark uses."""
import numpy as np
import pytest
import torch

import combine_ep_plan_gb300 as ep
import oracle
from combine_ep_plan_gb300.inputs import (WORKLOADS, bits_to_bf16_tensor, draw_hidden, draw_topk, draw_y,
                                          hidden_seed)
from ep_testutil import draw, u8, u16

pytestmark = pytest.mark.gpu

RTOL, ATOL = 8e-3, 1e-2  # combine tolerance in bf16


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
    WORKLOADS["fp8"].scaled(S=100, H=1024),
    WORKLOADS["zipf"].scaled(S=13, H=512),
    WORKLOADS["rt"].scaled(S=70, H=768),
]


def _f32(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).float().numpy()


# ---------------------------------------------------------------------------
# dispatch
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
@pytest.mark.parametrize("zero_pad", [True, False])
def test_dispatch_bf16_small(w, zero_pad):
    idx, wts, x = draw(w)
    pl = oracle.plan(idx, w.S, w.P, w.E, w.A)
    ref = oracle.dispatch_bf16(x, pl, zero_pad)
    h = ep.plan(torch.from_numpy(idx).cuda(), w.P, w.E, w.A)
    n_exp = h.sizes()[0]
    cap = n_exp + 7
    sentinel = torch.full((cap, w.H), -7.0, dtype=torch.bfloat16, device="cuda")
    mark = u16(torch.tensor([-7.0], dtype=torch.bfloat16))[0]
    recv, _ = ep.dispatch(h, bits_to_bf16_tensor(x).cuda(), "bf16", zero_pad, recv_x=sentinel)
    assert h.sync_status() == ep.EP_OK
    got = u16(recv)
    real = pl.exp_src >= 0
    assert np.array_equal(got[:n_exp][real], ref[real])
    if zero_pad:
        assert np.array_equal(got[:n_exp], ref)
    else:
        assert np.all(got[:n_exp][~real] == mark)  # untouched
    assert np.all(got[n_exp:] == mark)  # capacity tail untouched


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_dispatch_fp8_small(w):
    w = w.scaled(H=max(w.H, 128) // 128 * 128)
    idx, wts, x = draw(w)
    x = x.copy()
    x[1, :128] = 0           # amax == 0 group
    x[2, 128:256] = 0x8000   # a group of negative zeros
    pl = oracle.plan(idx, w.S, w.P, w.E, w.A)
    q_ref, s_ref = oracle.dispatch_fp8(x, pl)
    h = ep.plan(torch.from_numpy(idx).cuda(), w.P, w.E, w.A)
    recv, scales = ep.dispatch(h, bits_to_bf16_tensor(x).cuda(), "fp8")
    assert h.sync_status() == ep.EP_OK
    q = u8(recv)
    s = scales.cpu().numpy()
    assert np.array_equal(q, q_ref)
    assert np.array_equal(s.view(np.uint32), s_ref.view(np.uint32))


@pytest.mark.parametrize("name", ["bf16", "zipf", "rt"])
def test_dispatch_bf16_full_size_sampled(name):
    w = WORKLOADS[name]
    idx, wts, x = draw(w)
    pl = oracle.plan(idx, w.S, w.P, w.E, w.A)
    h = ep.plan(torch.from_numpy(idx).cuda(), w.P, w.E, w.A)
    cap = ep.worst_expanded_rows(w.T, w.K, w.E, w.A)  # the benchmark's launch: worst-case capacity
    recv, _ = ep.dispatch(h, bits_to_bf16_tensor(x).cuda(), "bf16", True, capacity=cap)
    assert h.sync_status() == ep.EP_OK
    rng = np.random.default_rng(5)
    rows = rng.choice(pl.num_expanded, size=3000, replace=False)
    rows = np.concatenate([rows, np.nonzero(pl.exp_src < 0)[0][:500], [0, pl.num_expanded - 1]])
    sub = oracle.Plan(**{**pl.__dict__, "exp_src": pl.exp_src[rows].copy(),
                         "expert_offsets": np.array([0, len(rows)], np.int32)})
    ref = oracle.dispatch_bf16(x, sub)
    got = u16(recv[torch.from_numpy(rows).cuda()])
    assert np.array_equal(got, ref)
    # properties at any size: every real row equals its source row
    src = torch.from_numpy(pl.exp_src).cuda().long()
    real = src >= 0
    xt = bits_to_bf16_tensor(x).cuda()
    assert torch.equal(recv[: pl.num_expanded][real].view(torch.int16), xt[src[real]].view(torch.int16))
    assert not recv[: pl.num_expanded][~real].view(torch.int16).any()


def test_dispatch_fp8_full_size_sampled():
    w = WORKLOADS["fp8"]
    idx, wts, x = draw(w)
    pl = oracle.plan(idx, w.S, w.P, w.E, w.A)
    h = ep.plan(torch.from_numpy(idx).cuda(), w.P, w.E, w.A)
    cap = ep.worst_expanded_rows(w.T, w.K, w.E, w.A)
    recv, scales = ep.dispatch(h, bits_to_bf16_tensor(x).cuda(), "fp8", True, capacity=cap)
    assert h.sync_status() == ep.EP_OK
    rng = np.random.default_rng(6)
    rows = np.concatenate([rng.choice(pl.num_expanded, size=3000, replace=False),
                           np.nonzero(pl.exp_src < 0)[0][:300]])
    sub = oracle.Plan(**{**pl.__dict__, "exp_src": pl.exp_src[rows].copy(),
                         "expert_offsets": np.array([0, len(rows)], np.int32)})
    q_ref, s_ref = oracle.dispatch_fp8(x, sub)
    r = torch.from_numpy(rows).cuda()
    assert np.array_equal(u8(recv[r]), q_ref)
    assert np.array_equal(scales[r].cpu().numpy().view(np.uint32), s_ref.view(np.uint32))


def test_cached_dispatch_zipf_ten_steps():
    """Fresh plan, then 10 cached-handle dispatches with new x (seeds 1..10)."""
    w = WORKLOADS["zipf"].scaled(S=32, H=1024)
    idx, wts = draw_topk(w)
    pl = oracle.plan(idx, w.S, w.P, w.E, w.A)
    h, recv, _ = ep.dispatch_fresh(torch.from_numpy(idx).cuda(),
                                   bits_to_bf16_tensor(draw_hidden(w.T, w.H, hidden_seed(w, 0))).cuda(),
                                   w.P, w.E, w.A)
    for step in range(1, w.cached_steps + 1):
        x = draw_hidden(w.T, w.H, hidden_seed(w, step))
        recv, _ = ep.dispatch_cached(h, bits_to_bf16_tensor(x).cuda(), w.E, w.A, w.S, recv_x=recv)
        assert h.sync_status() == ep.EP_OK
        assert np.array_equal(u16(recv)[: pl.num_expanded], oracle.dispatch_bf16(x, pl))


def test_cached_dispatch_rejects_mismatch():
    w = WORKLOADS["tiny"]
    idx, wts, x = draw(w)
    h = ep.plan(torch.from_numpy(idx).cuda(), w.P, w.E, w.A)
    xt = bits_to_bf16_tensor(x).cuda()
    for E, A, S in [(w.E * 2, w.A, w.S), (w.E, w.A + 1, w.S), (w.E, w.A, w.S + 1)]:
        with pytest.raises(ep.EPError) as ei:
            ep.dispatch_cached(h, xt, E, A, S)
        assert ei.value.code == ep.EP_ERR_MISMATCH


def test_dispatch_capacity_error_writes_nothing_beyond():
    w = WORKLOADS["bf16"].scaled(S=64, H=256)
    idx, wts, x = draw(w)
    h = ep.plan(torch.from_numpy(idx).cuda(), w.P, w.E, w.A)
    n_exp = h.sizes()[0]
    cap = n_exp // 2
    buf = torch.full((n_exp, w.H), 3.0, dtype=torch.bfloat16, device="cuda")
    ep.dispatch(h, bits_to_bf16_tensor(x).cuda(), "bf16", True, recv_x=buf[:cap])
    assert h.sync_status() == ep.EP_ERR_CAPACITY
    assert torch.all(buf[cap:] == 3.0)


# ---------------------------------------------------------------------------
# combine
# ---------------------------------------------------------------------------

def _gpu_expert(kind, recv, scales, pl_gpu_exp_off, E):
    """The synthetic expert between dispatch and combine (test scaffolding)."""
    if kind == "identity":
        return recv
    if kind == "dequant":
        s = scales.repeat_interleave(128, dim=1)
        return (recv.float() * s).to(torch.bfloat16)
    if kind == "scale":
        rows = recv.shape[0]
        counts = torch.diff(pl_gpu_exp_off.long())
        e_of_row = torch.repeat_interleave(torch.arange(E, device=recv.device), counts)
        f = 1.0 + e_of_row.float() / float(E)
        out = torch.zeros_like(recv)
        out[: len(f)] = (recv[: len(f)].float() * f[:, None]).to(torch.bfloat16)
        return out
    raise ValueError(kind)


def _oracle_expert(kind, pl, x):
    if kind == "identity":
        return oracle.dispatch_bf16(x, pl)
    if kind == "dequant":
        q, s = oracle.dispatch_fp8(x, pl)
        return oracle.expert_dequant(q, s)
    if kind == "scale":
        return oracle.expert_scale(oracle.dispatch_bf16(x, pl), pl)
    raise ValueError(kind)


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
@pytest.mark.parametrize("kind", ["identity", "scale", "dequant"])
def test_round_trip_small(w, kind):
    if kind == "dequant":
        w = w.scaled(H=max(w.H, 128) // 128 * 128)
    idx, wts, x = draw(w)
    pl = oracle.plan(idx, w.S, w.P, w.E, w.A)
    ref = oracle.combine(_oracle_expert(kind, pl, x), pl, wts)
    h = ep.plan(torch.from_numpy(idx).cuda(), w.P, w.E, w.A)
    recv, scales = ep.dispatch(h, bits_to_bf16_tensor(x).cuda(), "fp8" if kind == "dequant" else "bf16")
    y = _gpu_expert(kind, recv, scales, h.field("expert_offsets"), w.E)
    out = ep.combine(h, y, torch.from_numpy(wts).cuda())
    assert h.sync_status() == ep.EP_OK
    got = _f32(u16(out))
    want = _f32(ref)
    np.testing.assert_allclose(got, want, rtol=RTOL, atol=ATOL)
    # fixed k order and fmaf: the result is in fact bit-identical
    assert np.array_equal(u16(out), ref)


@pytest.mark.parametrize("w", SMALL[1:3], ids=lambda w: w.name)
def test_combine_random_y(w):
    idx, wts, x = draw(w)
    pl = oracle.plan(idx, w.S, w.P, w.E, w.A)
    y = draw_y(pl.num_expanded, w.H, 91)
    ref = oracle.combine(y, pl, wts)
    h = ep.plan(torch.from_numpy(idx).cuda(), w.P, w.E, w.A)
    out = ep.combine(h, bits_to_bf16_tensor(y).cuda(), torch.from_numpy(wts).cuda())
    np.testing.assert_allclose(_f32(u16(out)), _f32(ref), rtol=RTOL, atol=ATOL)


def test_combine_unused_slots_and_empty_tokens():
    w = WORKLOADS["rt"].scaled(S=40, H=256)
    idx, wts, x = draw(w)
    idx[::3, 5] = -1
    idx[::17] = -1
    pl = oracle.plan(idx, w.S, w.P, w.E, w.A)
    ref = oracle.combine(oracle.dispatch_bf16(x, pl), pl, wts)
    h = ep.plan(torch.from_numpy(idx).cuda(), w.P, w.E, w.A)
    recv, _ = ep.dispatch(h, bits_to_bf16_tensor(x).cuda())
    out = ep.combine(h, recv, torch.from_numpy(wts).cuda())
    assert np.array_equal(u16(out), ref)
    assert not u16(out)[::17].any()


def test_combine_y_rows_capacity_error():
    w = WORKLOADS["tiny"]
    idx, wts, x = draw(w)
    h = ep.plan(torch.from_numpy(idx).cuda(), w.P, w.E, w.A)
    n_exp = h.sizes()[0]
    y = torch.zeros((n_exp // 2, w.H), dtype=torch.bfloat16, device="cuda")
    ep.combine(h, y, torch.from_numpy(wts).cuda())
    assert h.sync_status() == ep.EP_ERR_CAPACITY


@pytest.mark.parametrize("name,kind", [("bf16", "identity"), ("fp8", "dequant"), ("zipf", "identity"),
                                       ("rt", "scale")])
def test_round_trip_full_size_sampled(name, kind):
    """Full-size workloads in the benchmark's launch configuration (worst-case
    capacity, zero padding); the oracle computes a sample of tokens, each from
    its own dispatch of only the rows those tokens need."""
    w = WORKLOADS[name]
    idx, wts, x = draw(w)
    pl = oracle.plan(idx, w.S, w.P, w.E, w.A)
    h = ep.plan(torch.from_numpy(idx).cuda(), w.P, w.E, w.A)
    cap = ep.worst_expanded_rows(w.T, w.K, w.E, w.A)
    recv, scales = ep.dispatch(h, bits_to_bf16_tensor(x).cuda(), "fp8" if kind == "dequant" else "bf16",
                               True, capacity=cap)
    y = _gpu_expert(kind, recv, scales, h.field("expert_offsets"), w.E)
    out = ep.combine(h, y, torch.from_numpy(wts).cuda())
    assert h.sync_status() == ep.EP_OK
    rng = np.random.default_rng(7)
    toks = np.sort(rng.choice(w.T, size=600, replace=False))
    rows = np.unique(pl.slot[toks][pl.slot[toks] >= 0])
    # oracle y for just those rows: a one-segment plan over the needed rows
    remap = -np.ones(pl.num_expanded, np.int64)
    remap[rows] = np.arange(len(rows))
    sub = oracle.Plan(**{**pl.__dict__, "exp_src": pl.exp_src[rows].copy(),
                         "expert_offsets": np.array([0, len(rows)], np.int32)})
    if kind == "scale":
        e_of_row = (np.searchsorted(pl.expert_offsets, rows, side="right") - 1).astype(np.int32)
        y_rows = oracle.expert_scale_rows(oracle.dispatch_bf16(x, sub), e_of_row, w.E)
    else:
        y_rows = _oracle_expert(kind, sub, x)
    sl = pl.slot[toks]
    sub_slot = np.where(sl >= 0, remap[np.maximum(sl, 0)], -1).astype(np.int32)
    tp = oracle.Plan(**{**pl.__dict__, "slot": np.ascontiguousarray(sub_slot), "S": len(toks), "P": 1})
    ref = oracle.combine(y_rows, tp, np.ascontiguousarray(wts[toks]))
    got = u16(out[torch.from_numpy(toks).cuda()])
    np.testing.assert_allclose(_f32(got), _f32(ref), rtol=RTOL, atol=ATOL)
    assert np.array_equal(got, ref)


def _midpoint_stress_rows(T, H, seed):
    """bf16 rows whose 128-element groups put x/scale within a bf16 ulp of
    E4M3 rounding midpoints, plus signed zeros, subnormals, and groups below
    the kernel's fast-quotient threshold (amax < 2^-60)."""
    rng = np.random.default_rng(seed)
    codes = np.arange(0, 0x7F, dtype=np.uint8)  # finite non-negative E4M3 codes
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    mids = (vals[:-1] + vals[1:]) / 2
    amaxes = np.array([3.0, 0.7, 1.0e-3, 2.0 ** -60, 2.0 ** -61, 3.0e-25, 1.0e30, 448.0, 5.5, 2.0 ** -126])
    x = np.zeros((T, H), np.float32)
    for t in range(T):
        for j in range(H // 128):
            amax = amaxes[(t * 7 + j) % len(amaxes)] * (1 + 0.01 * rng.standard_normal())
            amax = float(torch.tensor(amax, dtype=torch.float32).to(torch.bfloat16).float())
            s = np.float32(amax) / np.float32(448.0)
            m = rng.choice(mids, size=127) * rng.choice([-1.0, 1.0], size=127)
            g = (m * float(s)).astype(np.float32)
            g = np.clip(g, -amax, amax)
            g[:3] = [0.0, -0.0, 2.0 ** -130]
            x[t, j * 128] = amax if t % 2 else -amax
            x[t, j * 128 + 1:(j + 1) * 128] = g
    bits = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()
    # nudge by -1/0/+1 bf16 ulp, keeping |x| <= amax of the group
    nudge = rng.integers(-1, 2, size=bits.shape).astype(np.int32)
    nudged = (bits.astype(np.int32) + nudge).astype(np.uint16)
    f0 = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    f1 = torch.from_numpy(nudged.view(np.int16)).view(torch.bfloat16).float().numpy()
    am = np.abs(f0).reshape(T, H // 128, 128).max(axis=2).repeat(128, axis=1)
    ok = np.isfinite(f1) & (np.abs(f1) <= am) & (np.sign(f1) == np.sign(f0))
    ok[:, ::128] = False  # keep the amax element itself
    bits[ok] = nudged[ok]
    return bits


def test_dispatch_fp8_rounding_midpoints_and_tiny_groups():
    w = WORKLOADS["tiny"].scaled(H=1280)
    idx, wts = draw_topk(w)
    x = _midpoint_stress_rows(w.T, w.H, seed=3)
    pl = oracle.plan(idx, w.S, w.P, w.E, w.A)
    q_ref, s_ref = oracle.dispatch_fp8(x, pl)
    h = ep.plan(torch.from_numpy(idx).cuda(), w.P, w.E, w.A)
    recv, scales = ep.dispatch(h, bits_to_bf16_tensor(x).cuda(), "fp8")
    assert h.sync_status() == ep.EP_OK
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
    q = u8(recv)
    bad = np.argwhere(q != q_ref)
    assert len(bad) == 0, f"{len(bad)} codes differ, first {bad[:3].tolist()}"
