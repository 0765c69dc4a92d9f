"""Pins of the oracle's routing plan against what the pages and mathematics fix.

Each check takes a route independent of the oracle's nested-loop definition:
the pages' printed examples, closed forms, invariants, the V1 payload loop's
cursor walk, the deterministic layout's stable sort, brute force on tiny
inputs and the expected number of distinct destination ranks.
"""
import math

import numpy as np
import pytest

import oracle
from combine_ep_plan_gb300.inputs import WORKLOADS, draw_topk


def _plan(w, seed=None, C=0):
    idx, _ = draw_topk(w, seed)
    return idx, oracle.plan(idx, w.S, w.P, w.E, w.A, C)


SMALL = [
    WORKLOADS["tiny"],
    WORKLOADS["bf16"].scaled(S=96, H=256),
    WORKLOADS["fp8"].scaled(S=40, H=256),
    WORKLOADS["zipf"].scaled(S=6, H=256),
    WORKLOADS["rt"].scaled(S=24, H=128),
]


# ---------------------------------------------------------------------------
# the pages' printed examples (tests/golden)
# ---------------------------------------------------------------------------

def test_compact_plan_example(golden):
    g = golden("compact_plan_example.json")
    P, S, K = 32, 1, 3
    E = P  # one expert per rank: expert id == destination rank
    idx = -np.ones((P * S, K), np.int64)
    for tok, dests in g["token_destinations"].items():
        idx[int(tok), : len(dests)] = dests
    pl = oracle.plan(idx, S, P, E, A=1)
    for tok, dests in g["token_destinations"].items():
        assert list(np.nonzero(pl.is_token_in_rank[int(tok)])[0]) == dests
    for d in range(P):
        seg = pl.recv_src_idx[pl.recv_offsets[d]: pl.recv_offsets[d + 1]]
        # S == 1, so the source-local index is 0; the source rank is the token id
        srcs = [int(s) for s in np.nonzero(pl.send_head[:, d] >= 0)[0]]
        assert srcs == g["destination_segments"].get(str(d), [])
        assert len(seg) == len(srcs) and np.all(seg == 0)
        for pos, s in enumerate(srcs):
            assert pl.send_head[s, d] == pos


def test_local_expert_counts(golden):
    for case in golden("local_experts.json")["cases"]:
        E, P = case["num_experts"], case["num_ranks"]
        El = case["local_experts"]
        # one token per expert: each expert e lands on exactly one rank, and
        # the ranks each receive El tokens
        S = E // P
        idx = np.arange(E, dtype=np.int64).reshape(E, 1)
        pl = oracle.plan(idx, S, P, E, A=1)
        assert np.all(pl.num_recv == El)
        for e in range(E):
            assert np.nonzero(pl.is_token_in_rank[e])[0].tolist() == [e // El]


def test_byte_ledger(golden):
    g = golden("byte_ledger.json")
    H, K = g["hidden"], g["topk"]
    w = WORKLOADS["fp8"].scaled(S=8, H=H)  # every token has K valid slots
    idx, _ = draw_topk(w)
    pl = oracle.plan(idx, w.S, w.P, w.E, w.A)
    real_rows = int(np.sum(pl.exp_src >= 0))
    assert real_rows * H * 2 == w.T * g["bf16_dispatch_bytes"]
    assert real_rows * H * 1 == w.T * g["fp8_dispatch_bytes"]
    valid_slots = int(np.sum(pl.slot >= 0))
    assert valid_slots * H * 2 + valid_slots * 4 == w.T * g["bf16_combine_bytes_with_weights"]


def test_worst_tokens_padding(golden):
    # a fixed output length above the actual count leaves exactly the gap as
    # padding; the oracle's padded layout reproduces the page's 237/256/19
    g = golden("worst_tokens_example.json")
    P, E, K = 1, 1, 1
    S = g["actual_rows"]
    idx = np.zeros((S, K), np.int64)
    pl = oracle.plan(idx, S, P, E, A=g["worst_rows"])
    assert pl.num_expanded == g["worst_rows"]
    assert int(np.sum(pl.exp_src >= 0)) == g["actual_rows"]
    assert int(np.sum(pl.exp_src < 0)) == g["padding_rows"]


# ---------------------------------------------------------------------------
# closed forms and invariants
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_invariants(w):
    idx, pl = _plan(w)
    T, K, P, E, A, S = w.T, w.K, w.P, w.E, w.A, w.S
    El = E // P
    valid = idx >= 0
    # count conservation
    assert pl.expert_counts.sum() == valid.sum()
    assert np.array_equal(pl.expert_counts, np.bincount(idx[valid], minlength=E))
    ranks = np.where(valid, idx // El, -1)
    per_rank_pairs = sum(int(np.sum(ranks == d)) for d in range(P))
    assert per_rank_pairs == valid.sum()
    # per-token dedup: |dests(g)| equals the number of distinct ranks
    distinct = np.array([len(set(r[r >= 0].tolist())) for r in ranks])
    assert np.array_equal(pl.is_token_in_rank.sum(1), distinct)
    # padded segment sizes
    padded = (pl.expert_counts + A - 1) // A * A
    assert np.array_equal(np.diff(pl.expert_offsets), padded)
    assert pl.num_expanded == padded.sum()
    # prefix matrices
    assert np.array_equal(pl.rank_prefix[-1], pl.num_recv)
    assert np.array_equal(pl.rank_prefix, np.cumsum(pl.num_tokens_per_rank, axis=0))
    assert np.array_equal(pl.channel_prefix[:, :, -1], pl.num_tokens_per_rank)
    base = np.vstack([np.zeros((1, P), np.int32), pl.rank_prefix[:-1]])  # [s][d]
    cex = np.concatenate([np.zeros((P, P, 1), np.int32), pl.channel_prefix[:, :, :-1]], axis=2)
    assert np.array_equal(pl.recv_channel_prefix, (base[:, :, None] + cex).transpose(1, 0, 2))
    assert np.array_equal(pl.num_tokens_per_expert.sum(0), pl.expert_counts)
    assert np.array_equal(pl.num_tokens_per_rank.sum(0), pl.num_recv)


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_send_head_and_recv_src_idx_invert_each_other(w):
    idx, pl = _plan(w)
    S, P = w.S, w.P
    for d in range(P):
        win = pl.recv_src_idx[pl.recv_offsets[d]: pl.recv_offsets[d + 1]]
        assert len(win) == pl.num_recv[d] == int(np.sum(pl.send_head[:, d] >= 0))
        for s in range(P):
            lo = pl.rank_prefix[s - 1, d] if s else 0
            hi = pl.rank_prefix[s, d]
            for pos in range(lo, hi):
                assert pl.send_head[s * S + win[pos], d] == pos
    # and the other direction
    g, d = np.nonzero(pl.send_head >= 0)
    pos = pl.send_head[g, d]
    assert np.array_equal(pl.recv_src_idx[pl.recv_offsets[d] + pos], (g % S).astype(np.int32))


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_slot_and_exp_src_invert_each_other(w):
    idx, pl = _plan(w)
    g, k = np.nonzero(pl.slot >= 0)
    assert np.array_equal(pl.exp_src[pl.slot[g, k]], g.astype(np.int32))
    assert np.all((pl.slot >= 0) == (idx >= 0))
    # each real row is used by exactly one (g,k)
    assert len(np.unique(pl.slot[pl.slot >= 0])) == int(np.sum(pl.exp_src >= 0))
    # the row lies in its expert's segment
    e = idx[g, k]
    r = pl.slot[g, k]
    assert np.all((pl.expert_offsets[e] <= r) & (r < pl.expert_offsets[e] + pl.expert_counts[e]))


# ---------------------------------------------------------------------------
# independent routes through the same definitions
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
@pytest.mark.parametrize("C", [0, 1, 3])
def test_v1_cursor_walk(w, C):
    """Re-run the V1 payload loop of the pages (one cursor per destination,
    initialised from the rank and channel prefix bases, advanced through the
    channel's tokens in order, 'Device 侧如何把 channel 变成远端 Put') and check
    that it lands every (token, destination) where the plan says."""
    idx, pl = _plan(w, C=C)
    S, P, Cc = w.S, w.P, pl.C
    chunk = -(-S // Cc)
    for s in range(P):
        for c in range(Cc):
            cursor = [
                (pl.rank_prefix[(s - 1), d] if s > 0 else 0)
                + (pl.channel_prefix[s, d, c - 1] if c > 0 else 0)
                for d in range(P)
            ]
            for d in range(P):
                assert cursor[d] == pl.recv_channel_prefix[d, s, c]
            for t in range(min(S, c * chunk), min(S, (c + 1) * chunk)):
                g = s * S + t
                for d in range(P):
                    if not pl.is_token_in_rank[g, d]:
                        assert pl.send_head[g, d] == -1
                        continue
                    assert pl.send_head[g, d] == cursor[d]
                    assert pl.recv_src_idx[pl.recv_offsets[d] + cursor[d]] == t
                    cursor[d] += 1
            for d in range(P):
                assert cursor[d] == (pl.rank_prefix[s - 1, d] if s > 0 else 0) + pl.channel_prefix[s, d, c]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_deterministic_sort_layout(w):
    """The deterministic layout is a stable sort of the expanded (token, slot)
    pairs by expert * 1e10 + source global token (TileLang tutorial ch. 38,
    §3.5).  Rebuild the expanded layout that way and compare."""
    idx, pl = _plan(w)
    pairs = [(int(e) * 10 ** 10 + g, g, k) for g in range(w.T) for k, e in enumerate(idx[g]) if e >= 0]
    pairs.sort(key=lambda p: p[0])
    seen = {}
    for key, g, k in pairs:
        e = key // 10 ** 10
        j = seen.get(e, 0)
        seen[e] = j + 1
        row = int(pl.expert_offsets[e]) + j
        assert pl.slot[g, k] == row
        assert pl.exp_src[row] == g


def test_brute_force_tiny():
    """Enumerate the tiny workload with sets and dictionaries."""
    w = WORKLOADS["tiny"]
    idx, pl = _plan(w)
    S, P, E, A = w.S, w.P, w.E, w.A
    El = E // P
    dests = {g: sorted({int(e) // El for e in idx[g] if e >= 0}) for g in range(w.T)}
    windows = {d: [g for g in range(w.T) if d in dests[g]] for d in range(P)}
    for d in range(P):
        assert pl.num_recv[d] == len(windows[d])
        for pos, g in enumerate(windows[d]):
            assert pl.send_head[g, d] == pos
            assert pl.recv_src_idx[pl.recv_offsets[d] + pos] == g % S
    members = {e: [(g, k) for g in range(w.T) for k in range(w.K) if idx[g, k] == e] for e in range(E)}
    row = 0
    for e in range(E):
        assert pl.expert_offsets[e] == row
        for j, (g, k) in enumerate(members[e]):
            assert pl.slot[g, k] == row + j
        row += -(-len(members[e]) // A) * A
    assert pl.num_expanded == row


def _brute_plan(idx, S, P, E, A, C):
    """Every plan array from the definitions, with Python sets, lists and loops."""
    T, K = idx.shape
    El = E // P
    chunk = -(-S // C)
    dests = [sorted({int(e) // El for e in idx[g] if e >= 0}) for g in range(T)]
    in_rank = np.array([[1 if d in dests[g] else 0 for d in range(P)] for g in range(T)], np.uint8)
    ntpr = np.array([[sum(in_rank[s * S + t, d] for t in range(S)) for d in range(P)] for s in range(P)], np.int32)
    ntpe = np.array([[sum(int(idx[s * S + t, k] == e) for t in range(S) for k in range(K)) for e in range(E)]
                     for s in range(P)], np.int32)
    rpm = np.array([[sum(ntpr[s2, d] for s2 in range(s + 1)) for d in range(P)] for s in range(P)], np.int32)
    cpm = np.zeros((P, P, C), np.int32)
    for s in range(P):
        for d in range(P):
            for c in range(C):
                cpm[s, d, c] = sum(in_rank[s * S + t, d] for t in range(min(S, (c + 1) * chunk)))
    rcpm = np.zeros((P, P, C), np.int32)
    for d in range(P):
        for s in range(P):
            for c in range(C):
                rcpm[d, s, c] = (rpm[s - 1, d] if s > 0 else 0) + (cpm[s, d, c - 1] if c > 0 else 0)
    windows = [[g for g in range(T) if d in dests[g]] for d in range(P)]
    send_head = -np.ones((T, P), np.int32)
    recv_src = []
    for d in range(P):
        for pos, g in enumerate(windows[d]):
            send_head[g, d] = pos
            recv_src.append(g % S)
    slot = -np.ones((T, K), np.int32)
    exp_src, offsets = [], [0]
    for e in range(E):
        members = [(g, k) for g in range(T) for k in range(K) if idx[g, k] == e]
        for g, k in members:
            slot[g, k] = len(exp_src)
            exp_src.append(g)
        exp_src += [-1] * (-(-len(members) // A) * A - len(members))
        offsets.append(len(exp_src))
    return dict(is_token_in_rank=in_rank, num_tokens_per_rank=ntpr, num_tokens_per_expert=ntpe,
                expert_counts=ntpe.sum(axis=0).astype(np.int32), num_recv=in_rank.sum(axis=0).astype(np.int32),
                rank_prefix=rpm, channel_prefix=cpm, recv_channel_prefix=rcpm, send_head=send_head,
                recv_offsets=np.concatenate([[0], np.cumsum([len(wd) for wd in windows])]).astype(np.int32),
                recv_src_idx=np.array(recv_src, np.int32), expert_offsets=np.array(offsets, np.int32),
                slot=slot, exp_src=np.array(exp_src, np.int32))


@pytest.mark.parametrize("i", range(24))
def test_brute_force_random_shapes(i):
    """Every plan array of the oracle against the Python brute force, on
    random small shapes with unused slots, any channel count and padding."""
    rng = np.random.default_rng(500 + i)
    P = int(rng.integers(1, 7))
    E = P * int(rng.integers(1, 5))
    K = int(rng.integers(1, min(E, 5) + 1))
    S = int(rng.integers(1, 41))
    A = int(rng.choice([1, 2, 3, 8]))
    C = int(rng.integers(1, S + 1))
    w = WORKLOADS["tiny"].scaled(P=P, E=E, K=K, S=S, A=A, routing="zipf" if i % 3 == 0 else "uniform", seed=i)
    idx, _ = draw_topk(w)
    idx[rng.random(idx.shape) < 0.2] = -1
    pl = oracle.plan(idx, S, P, E, A, C)
    want = _brute_plan(idx, S, P, E, A, C)
    for name, arr in want.items():
        got = getattr(pl, name)
        assert got.shape == arr.shape and np.array_equal(got, arr), name


def test_single_rank_is_all_local():
    w = WORKLOADS["tiny"].scaled(P=1, S=128)
    idx, pl = _plan(w)
    assert np.all(pl.is_token_in_rank[:, 0] == 1)
    assert np.array_equal(pl.send_head[:, 0], np.arange(w.T))
    assert np.array_equal(pl.recv_src_idx, np.arange(w.T))


def test_unused_slots():
    w = WORKLOADS["tiny"]
    idx, _ = draw_topk(w)
    idx[::3, 1] = -1
    idx[::7, :] = -1  # tokens routed nowhere
    pl = oracle.plan(idx, w.S, w.P, w.E, w.A)
    assert np.all(pl.slot[idx < 0] == -1)
    assert np.all(pl.is_token_in_rank[::7].sum(1) == 0)
    assert np.all(pl.send_head[::7] == -1)
    assert pl.expert_counts.sum() == int(np.sum(idx >= 0))


def test_channels_equal_tokens():
    w = WORKLOADS["tiny"].scaled(S=16)
    idx, pl = _plan(w, C=16)
    # one token per channel: channel counts are the routing matrix itself
    for s in range(w.P):
        per_channel = np.diff(np.concatenate([np.zeros((w.P, 1), np.int32), pl.channel_prefix[s]], axis=1), axis=1)
        assert np.array_equal(per_channel.T, pl.is_token_in_rank[s * w.S:(s + 1) * w.S])


@pytest.mark.parametrize("mutate,kw", [
    ("range", {}), ("dup", {}), ("low", {}), (None, {"E": 9}), (None, {"A": 0}), (None, {"C": 100}),
    (None, {"C": 65}),  # one channel more than the 64 tokens per rank
])
def test_invalid_inputs(mutate, kw):
    w = WORKLOADS["tiny"]
    idx, _ = draw_topk(w)
    if mutate == "range":
        idx[5, 0] = w.E
    elif mutate == "dup":
        idx[7, 1] = idx[7, 0]
    elif mutate == "low":
        idx[3, 1] = -2
    E, A, C = kw.get("E", w.E), kw.get("A", w.A), kw.get("C", 0)
    assert oracle.validate(idx, w.S, w.P, E, A, C) == oracle.ERR_INVALID
    with pytest.raises(oracle.OracleError):
        oracle.plan(idx, w.S, w.P, E, A, C)


@pytest.mark.parametrize("P,E,K", [(2, 8, 4), (4, 8, 2)])
def test_receive_capacity_is_attained(P, E, K):
    """Every token reaching min(K, P) ranks fills the receive windows to the
    worst case T*min(K, P) the oracle sizes them for; random routing stays
    below it."""
    S, El = 8, E // P
    # each token's K experts spread round-robin over the ranks
    row = np.array([(k % P) * El + k // P for k in range(K)], np.int64)
    idx = np.tile(row, (P * S, 1))
    pl = oracle.plan(idx, S, P, E, A=1)
    assert len(set(row // El)) == min(K, P)
    assert pl.num_recv_total == oracle.max_recv_rows(S, P, K)
    rng = np.random.default_rng(3)
    idx = np.stack([rng.choice(E, K, replace=False) for _ in range(P * S)]).astype(np.int64)
    pl = oracle.plan(idx, S, P, E, A=1)
    assert pl.num_recv_total <= oracle.max_recv_rows(S, P, K)


# ---------------------------------------------------------------------------
# statistics: expected number of distinct destination ranks per token
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["bf16", "fp8", "rt"])
def test_expected_distinct_ranks(name):
    """Tutorial ch. 38 §1.3 gives R(1-(1-1/R)^k) for k independent draws with
    replacement.  The workloads draw K *distinct* experts uniformly, for which
    the exact expectation is P(1 - C(E-E_l, K)/C(E, K)); the sample mean must
    sit within 4 standard errors of it, and the page's form must be close."""
    w = WORKLOADS[name].scaled(S=min(WORKLOADS[name].S, 512))
    idx, pl = _plan(w)
    El = w.E // w.P
    exact = w.P * (1 - math.comb(w.E - El, w.K) / math.comb(w.E, w.K))
    page = w.P * (1 - (1 - 1 / w.P) ** w.K)
    per_token = pl.is_token_in_rank.sum(1).astype(np.float64)
    se = per_token.std(ddof=1) / math.sqrt(len(per_token))
    assert abs(per_token.mean() - exact) < 4 * se
    assert abs(page - exact) / exact < 0.06
