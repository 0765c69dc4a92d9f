"""The OpenMP build of the oracle gives the same bits as the single-threaded
build on every function whose row loop it splits over threads.

Both libraries come from the same ``ep_oracle.c``; the multi-core one only
distributes independent rows, each still computed by the same sequential code.
CPU only.
"""
import numpy as np
import pytest

import oracle
from combine_ep_plan_gb300.inputs import WORKLOADS, draw_hidden, draw_topk, draw_y, hidden_seed

pytestmark = pytest.mark.skipif(not oracle.omp_available(), reason="gcc without -fopenmp")


def _both(fn):
    a = fn()
    with oracle.parallel():
        b = fn()
    return a, b


def _same(a, b):
    if isinstance(a, tuple):
        return all(_same(x, y) for x, y in zip(a, b))
    return np.array_equal(np.asarray(a).view(np.uint8), np.asarray(b).view(np.uint8))


def test_parallel_build_uses_more_than_one_thread_when_the_host_has_them():
    import os
    with oracle.parallel():
        n = oracle.threads()
    assert n >= 1
    if (os.cpu_count() or 1) > 1 and "OMP_NUM_THREADS" not in os.environ:
        assert n > 1
    assert oracle.threads() == 1


@pytest.mark.parametrize("name", ["rt", "fp8"])
def test_parallel_build_is_bit_identical(name):
    w = WORKLOADS[name].scaled(S=24, H=512)
    idx, wts = draw_topk(w)
    idx[::5, -1] = -1
    x = draw_hidden(w.T, w.H, hidden_seed(w))
    pl = oracle.plan(idx, w.S, w.P, w.E, w.A)
    y = draw_y(pl.num_expanded, w.H, 3)
    bias = draw_y(pl.T, w.H, 4)
    cases = {
        "dispatch_bf16": lambda: oracle.dispatch_bf16(x, pl, True),
        "dispatch_bf16_nopad": lambda: oracle.dispatch_bf16(x, pl, False),
        "dispatch_fp8": lambda: oracle.dispatch_fp8(x, pl, True),
        "combine": lambda: oracle.combine(y, pl, wts),
        "combine_bias": lambda: oracle.combine(y, pl, wts, bias),
        "expert_scale": lambda: oracle.expert_scale(y, pl),
        "expert_dequant": lambda: oracle.expert_dequant(*oracle.dispatch_fp8(x, pl, True)),
        "dispatch_backward": lambda: oracle.dispatch_backward(y, pl),
        "combine_backward": lambda: oracle.combine_backward(bias, y, pl, wts, True),
    }
    q, s = oracle.dispatch_fp8(x, pl, True)
    cases["dispatch_fp8_input"] = lambda: oracle.dispatch_fp8_input(q[: pl.T], s[: pl.T], pl, True)
    e_of_row = (np.searchsorted(pl.expert_offsets, np.arange(pl.num_expanded), side="right") - 1).astype(np.int32)
    e_of_row[pl.exp_src < 0] = -1
    cases["expert_scale_rows"] = lambda: oracle.expert_scale_rows(y, e_of_row, w.E)
    for case, fn in cases.items():
        a, b = _both(fn)
        assert _same(a, b), case
