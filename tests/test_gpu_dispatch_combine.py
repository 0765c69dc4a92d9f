"""GPU parity of dispatch (BF16 bit copy, FP8 E4M3 quantised inside dispatch)
and combine, against the oracle, element by element: on cases that span
several tiles with a ragged tail, and on whole arrays at the full workload
sizes in the launch configuration the benchmark uses."""
import numpy as np
import pytest
import torch

import combine_ep_plan_gb300 as ep
import oracle
from combine_ep_plan_gb300.inputs import (WORKLOADS, bits_to_bf16_tensor, draw_hidden, draw_topk, draw_y,
                                          hidden_seed)
from ep_testutil import assert_bits_equal, draw, u8, u16

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


FULL = ["tiny", "bf16", "fp8", "zipf", "rt"]
_SENTINEL_BF16 = -7.0  # rows past N_exp must keep it
_SENTINEL_CODE = 0x5A


@pytest.mark.parametrize("name", FULL)
def test_dispatch_bf16_full_size(name):
    """The whole expanded layout (token rows and zeroed padding rows) of each
    full-size workload, in the benchmark's launch configuration (worst-case
    capacity, zero padding), bit for bit against the oracle; rows past N_exp
    untouched."""
    w = WORKLOADS[name]
    idx, wts, x = draw(w)
    pl = oracle.plan(idx, w.S, w.P, w.E, w.A)
    h = ep.plan(torch.from_numpy(idx).cuda(), w.P, w.E, w.A)
    cap = ep.worst_expanded_rows(w.T, w.K, w.E, w.A)
    buf = torch.full((cap, w.H), _SENTINEL_BF16, dtype=torch.bfloat16, device="cuda")
    recv, _ = ep.dispatch(h, bits_to_bf16_tensor(x).cuda(), "bf16", True, recv_x=buf)
    assert h.sync_status() == ep.EP_OK
    with oracle.parallel():
        ref = oracle.dispatch_bf16(x, pl, True)
    assert_bits_equal(recv[: pl.num_expanded], ref, f"{name} recv_x")
    assert torch.all(recv[pl.num_expanded:] == _SENTINEL_BF16)


@pytest.mark.parametrize("name", FULL)
def test_dispatch_fp8_full_size(name):
    """FP8 dispatch (quantised inside) of each full-size workload's hidden
    states: every E4M3 code and every fp32 scale of the expanded layout bit
    for bit against the oracle; rows past N_exp untouched."""
    w = WORKLOADS[name]
    assert w.H % 128 == 0
    idx, wts, x = draw(w)
    pl = oracle.plan(idx, w.S, w.P, w.E, w.A)
    h = ep.plan(torch.from_numpy(idx).cuda(), w.P, w.E, w.A)
    cap = ep.worst_expanded_rows(w.T, w.K, w.E, w.A)
    codes = torch.full((cap, w.H), _SENTINEL_CODE, dtype=torch.uint8, device="cuda")
    scales = torch.full((cap, w.H // 128), -3.0, dtype=torch.float32, device="cuda")
    recv, sc = ep.dispatch(h, bits_to_bf16_tensor(x).cuda(), "fp8", True,
                           recv_x=codes.view(torch.float8_e4m3fn), recv_scales=scales)
    assert h.sync_status() == ep.EP_OK
    with oracle.parallel():
        q_ref, s_ref = oracle.dispatch_fp8(x, pl, True)
    n = pl.num_expanded
    assert_bits_equal(codes[:n], q_ref, f"{name} codes")
    assert_bits_equal(scales[:n], s_ref, f"{name} scales")
    assert torch.all(codes[n:] == _SENTINEL_CODE) and torch.all(scales[n:] == -3.0)


def test_cached_dispatch_zipf_ten_steps_full_size():
    """The skewed-routing workload at full size: a fresh plan and dispatch,
    then 10 cached-handle dispatches with new hidden states (the seeds of
    dispatches 1..10), each whole array against the oracle on the same plan."""
    w = WORKLOADS["zipf"]
    idx, wts = draw_topk(w)
    pl = oracle.plan(idx, w.S, w.P, w.E, w.A)
    cap = ep.worst_expanded_rows(w.T, w.K, w.E, w.A)
    x0 = draw_hidden(w.T, w.H, hidden_seed(w, 0))
    h, recv, _ = ep.dispatch_fresh(torch.from_numpy(idx).cuda(), bits_to_bf16_tensor(x0).cuda(),
                                   w.P, w.E, w.A)  # outputs sized for the worst case
    assert recv.shape[0] == cap
    assert h.sync_status() == ep.EP_OK
    with oracle.parallel():
        assert_bits_equal(recv[: pl.num_expanded], oracle.dispatch_bf16(x0, pl, True), "zipf fresh")
    for step in range(1, w.cached_steps + 1):
        x = draw_hidden(w.T, w.H, hidden_seed(w, step))
        recv, _ = ep.dispatch_cached(h, bits_to_bf16_tensor(x).cuda(), w.E, w.A, w.S, recv_x=recv)
        assert h.sync_status() == ep.EP_OK
        with oracle.parallel():
            assert_bits_equal(recv[: pl.num_expanded], oracle.dispatch_bf16(x, pl, True), f"zipf cached {step}")


def test_cached_dispatch_zipf_ten_steps():
    """Fresh plan, then 10 cached-handle dispatches with new x (seeds 1..10), at a reduced size."""
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


@pytest.mark.parametrize("name", FULL)
def test_round_trip_full_size(name):
    """Each full-size workload end to end in the benchmark's launch
    configuration (worst-case capacity, zero padding): dispatch (FP8 for the
    FP8 workload), the workload's synthetic expert, combine; the whole [T,H]
    output against the oracle's own dispatch -> expert -> combine, within the
    combine tolerance and in fact bit for bit."""
    w = WORKLOADS[name]
    kind = w.expert
    idx, wts, x = draw(w)
    pl = oracle.plan(idx, w.S, w.P, w.E, w.A)
    h = ep.plan(torch.from_numpy(idx).cuda(), w.P, w.E, w.A)
    cap = ep.worst_expanded_rows(w.T, w.K, w.E, w.A)
    recv, scales = ep.dispatch(h, bits_to_bf16_tensor(x).cuda(), "fp8" if w.fp8 else "bf16", True, capacity=cap)
    y = _gpu_expert(kind, recv, scales, h.field("expert_offsets"), w.E)
    out = ep.combine(h, y, torch.from_numpy(wts).cuda())
    assert h.sync_status() == ep.EP_OK
    with oracle.parallel():
        ref = oracle.combine(_oracle_expert(kind, pl, x), pl, wts)
    got = u16(out)
    np.testing.assert_allclose(_f32(got), _f32(ref), rtol=RTOL, atol=ATOL)
    assert_bits_equal(out, ref, f"{name} combine")


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


def _non_finite_rows(T, H, seed):
    """N(0,1) bf16 rows with non-finite elements planted group by group: one
    NaN of either sign, +inf or -inf, a group of NaNs, zeros with a NaN, and
    inf, -inf and NaN together."""
    rng = np.random.default_rng(seed)
    bits = draw_hidden(T, H, seed)
    G = H // 128
    kinds = rng.integers(0, 8, size=(T, G))
    pos = rng.integers(0, 128, size=(T, G, 3))
    PNAN, NNAN, PINF, NINF = 0x7FC0, 0xFFC0, 0x7F80, 0xFF80
    for t in range(T):
        for j in range(G):
            g = bits[t, j * 128:(j + 1) * 128]
            a, b, c = pos[t, j]
            k = kinds[t, j]
            if k == 1:
                g[a] = PNAN
            elif k == 2:
                g[a] = NNAN
            elif k == 3:
                g[a] = PINF
            elif k == 4:
                g[a] = NINF
            elif k == 5:
                g[:] = PNAN
            elif k == 6:
                g[:] = 0
                g[a] = NNAN
            elif k == 7:
                g[a], g[b], g[c] = PINF, NINF, NNAN
    return bits


@pytest.mark.parametrize("w", [WORKLOADS["tiny"].scaled(H=1024), WORKLOADS["fp8"].scaled(S=40, H=2048)],
                         ids=["tiny", "fp8"])
def test_non_finite_hidden_values(w):
    """Inf and NaN in x, under the reading the oracle pins (NaN elements left
    out of amax, an infinite element makes the scale +inf, every NaN quotient
    is code 0x7F): FP8 codes and scales and the BF16 bit copy bit for bit
    against the oracle; the combine equal wherever the oracle is not NaN, and
    NaN exactly where the oracle is."""
    idx, wts = draw_topk(w)
    x = _non_finite_rows(w.T, w.H, seed=29)
    pl = oracle.plan(idx, w.S, w.P, w.E, w.A)
    h = ep.plan(torch.from_numpy(idx).cuda(), w.P, w.E, w.A)
    xt = bits_to_bf16_tensor(x).cuda()
    q, sc = ep.dispatch(h, xt, "fp8")
    recv, _ = ep.dispatch(h, xt, "bf16")
    out = ep.combine(h, recv, torch.from_numpy(wts).cuda())
    assert h.sync_status() == ep.EP_OK
    q_ref, s_ref = oracle.dispatch_fp8(x, pl)
    assert_bits_equal(q.view(torch.uint8), q_ref, "codes")
    assert_bits_equal(sc, s_ref, "scales")
    assert (q_ref == 0x7F).any() and np.isinf(s_ref).any()
    assert_bits_equal(recv, oracle.dispatch_bf16(x, pl), "bf16 rows")
    ref = oracle.combine(oracle.dispatch_bf16(x, pl), pl, wts)
    got = u16(out)
    nan_ref, nan_got = np.isnan(_f32(ref)), np.isnan(_f32(got))
    assert nan_ref.any() and np.array_equal(nan_got, nan_ref)
    assert np.array_equal(got[~nan_ref], ref[~nan_ref])
