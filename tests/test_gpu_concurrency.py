"""Two handles at work at the same time on two CUDA streams (two micro-batches
in flight): each stream plans, replans with new routing, dispatches in BF16
and FP8 and combines, with no host synchronisation until the end; every
result of every round is compared with the oracle, whole arrays.  The
handles share nothing on the device, so the interleaving may not change a
bit."""
import numpy as np
import pytest
import torch

import combine_ep_plan_gb300 as ep
import oracle
from combine_ep_plan_gb300.inputs import WORKLOADS, bits_to_bf16_tensor, draw_hidden, draw_topk, hidden_seed
from ep_testutil import assert_bits_equal

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from combine_ep_plan_gb300 import build
    build.build()
    ep.load_library()
    yield
    torch.cuda.synchronize()


def test_two_handles_on_two_streams():
    cases = [WORKLOADS["bf16"].scaled(S=600, H=2048), WORKLOADS["fp8"].scaled(S=300, H=2048)]
    rounds = 3
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    inputs = []
    for w in cases:
        per_round = []
        for r in range(rounds):
            idx, wts = draw_topk(w, seed=100 + r)
            x = draw_hidden(w.T, w.H, hidden_seed(w) + r)
            per_round.append((idx, wts, x, torch.from_numpy(idx).cuda(), torch.from_numpy(wts).cuda(),
                              bits_to_bf16_tensor(x).cuda()))
        inputs.append(per_round)
    torch.cuda.synchronize()

    # enqueue everything, alternating between the streams round by round
    handles = [None, None]
    results = [[None] * rounds for _ in cases]
    for r in range(rounds):
        for i, w in enumerate(cases):
            s = streams[i]
            _, _, _, idx_t, wts_t, x_t = inputs[i][r]
            with torch.cuda.stream(s):
                if handles[i] is None:
                    handles[i] = ep.plan(idx_t, w.P, w.E, w.A, stream=s)
                else:
                    handles[i].replan(idx_t, stream=s)
                h = handles[i]
                cap = ep.worst_expanded_rows(w.T, w.K, w.E, w.A)
                recv, _ = ep.dispatch(h, x_t, "bf16", True, capacity=cap, stream=s)
                q, sc = ep.dispatch(h, x_t, "fp8", True, capacity=cap, stream=s)
                out = ep.combine(h, recv, wts_t, stream=s)
                slot = h.field("slot").clone()  # this round's plan, before the next replan
            results[i][r] = (recv, q, sc, out, slot)
    torch.cuda.synchronize()

    for i, w in enumerate(cases):
        assert handles[i].sync_status() == ep.EP_OK
        for r in range(rounds):
            idx, wts, x, *_ = inputs[i][r]
            recv, q, sc, out, slot = results[i][r]
            pl = oracle.plan(idx, w.S, w.P, w.E, w.A)
            n = pl.num_expanded
            assert np.array_equal(slot.cpu().numpy(), pl.slot)
            with oracle.parallel():
                ref = oracle.dispatch_bf16(x, pl, True)
                assert_bits_equal(recv[:n], ref, "bf16 rows")
                q_ref, s_ref = oracle.dispatch_fp8(x, pl, True)
                assert_bits_equal(q[:n].view(torch.uint8), q_ref, "fp8 codes")
                assert_bits_equal(sc[:n], s_ref, "fp8 scales")
                assert_bits_equal(out, oracle.combine(ref, pl, wts), "combine")
        handles[i].destroy()
