"""The allocation-free plan entry point, ep_plan_static_scratch, against ep_plan.

Some callers of this library cannot allocate device memory when they plan:
a serving runtime that gave all device memory to its own arena at start-up,
or a latency-critical loop where an allocation may block on the device or
fail under fragmentation.  ep_plan_static_scratch serves them: the caller
passes every output buffer, and the plan's scratch lives in a fixed array
inside the library.  This test calls it through the C ABI twice in a row
(different routing each time, so stale scratch from the first call would
show) and checks every plan array against the one ep_plan produces for the
same routing, and against the oracle directly (default and explicit channel
counts, expert alignment 1).  It is collected last, runs alone in a fresh
process as well as after the other tests, and allocates all its buffers
before the call.
"""
import ctypes

import numpy as np
import pytest
import torch

import combine_ep_plan_gb300 as ep
import oracle
from combine_ep_plan_gb300.inputs import WORKLOADS, draw_topk
from ep_testutil import PLAN_FIELDS, assert_plan_equal, gpu_plan_arrays

pytestmark = pytest.mark.gpu


class PlanBuffers(ctypes.Structure):
    _fields_ = [(name, ctypes.c_void_p) for name in [
        "is_token_in_rank", "send_head", "num_tokens_per_rank", "num_tokens_per_expert", "expert_counts",
        "num_recv", "rank_prefix", "channel_prefix", "recv_channel_prefix", "recv_offsets", "recv_src_idx",
        "expert_offsets", "slot", "exp_src", "pad_rows", "info"]]


@pytest.fixture(scope="module")
def lib():
    from combine_ep_plan_gb300 import build
    build.build()
    lib = ep.load_library()
    lib.ep_plan_static_scratch.restype = ctypes.c_int
    lib.ep_plan_static_scratch.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           ctypes.POINTER(PlanBuffers), ctypes.c_void_p]
    return lib


def _buffers(w, C):
    T, P, E, K, A = w.T, w.P, w.E, w.K, w.A
    i32 = dict(dtype=torch.int32, device="cuda")
    bufs = {
        "is_token_in_rank": torch.empty((T, P), dtype=torch.uint8, device="cuda"),
        "send_head": torch.empty((T, P), **i32),
        "num_tokens_per_rank": torch.empty((P, P), **i32),
        "num_tokens_per_expert": torch.empty((P, E), **i32),
        "expert_counts": torch.empty(E, **i32),
        "num_recv": torch.empty(P, **i32),
        "rank_prefix": torch.empty((P, P), **i32),
        "channel_prefix": torch.empty((P, P, C), **i32),
        "recv_channel_prefix": torch.empty((P, P, C), **i32),
        "recv_offsets": torch.empty(P + 1, **i32),
        "recv_src_idx": torch.empty(T * min(K, P), **i32),
        "expert_offsets": torch.empty(E + 1, **i32),
        "slot": torch.empty((T, K), **i32),
        "exp_src": torch.empty(T * K + E * (A - 1), **i32),
        "pad_rows": torch.empty(max(1, E * (A - 1)), **i32),
        "info": torch.empty(4, **i32),
    }
    for t in bufs.values():  # garbage that a missing write would expose
        t.fill_(0x5A if t.dtype == torch.uint8 else -12345)
    return bufs


@pytest.mark.parametrize("name", ["bf16", "zipf"])
def test_static_scratch_plan_matches_ep_plan_twice_in_a_row(lib, name):
    w = WORKLOADS[name]
    C = min(16, w.S)
    stream = torch.cuda.current_stream()
    for seed in (11, 12):
        idx, _ = draw_topk(w, seed=seed)
        idx_t = torch.from_numpy(idx).cuda()
        bufs = _buffers(w, C)
        st = PlanBuffers(**{k: v.data_ptr() for k, v in bufs.items()})
        torch.cuda.synchronize()
        rc = lib.ep_plan_static_scratch(idx_t.data_ptr(), w.S, w.P, w.K, w.E, w.A, 0, ctypes.byref(st),
                                        stream.cuda_stream)
        assert rc == ep.EP_OK
        torch.cuda.synchronize()
        n_recv, n_exp, n_pad, status = bufs["info"].tolist()
        assert status == 0
        # the existing entry point on the same routing
        h = ep.plan(idx_t, w.P, w.E, w.A)
        want = gpu_plan_arrays(h)
        assert (n_exp, n_recv) == h.sizes()
        got = {k: v.cpu().numpy() for k, v in bufs.items()}
        got["recv_src_idx"] = got["recv_src_idx"][:n_recv]
        got["exp_src"] = got["exp_src"][:n_exp]
        got["pad_rows"] = got["pad_rows"][:n_pad]
        for k in PLAN_FIELDS + ["pad_rows"]:
            assert np.array_equal(got[k], want[k]), k
        h.destroy()


@pytest.mark.parametrize("name,C,A", [("tiny", 0, 1), ("bf16", 5, 128), ("rt", 16, 1)])
def test_static_scratch_plan_matches_the_oracle(lib, name, C, A):
    """Every plan array of the allocation-free entry point against the oracle
    directly: the default channel count, an explicit one other than 16, and
    expert_alignment 1 (no padding rows: the one-entry pad_rows buffer)."""
    w = WORKLOADS[name].scaled(A=A)
    Cq = C if C else min(16, w.S)
    idx, _ = draw_topk(w, seed=13)
    idx_t = torch.from_numpy(idx).cuda()
    bufs = _buffers(w, Cq)
    st = PlanBuffers(**{k: v.data_ptr() for k, v in bufs.items()})
    torch.cuda.synchronize()
    rc = lib.ep_plan_static_scratch(idx_t.data_ptr(), w.S, w.P, w.K, w.E, w.A, C, ctypes.byref(st),
                                    torch.cuda.current_stream().cuda_stream)
    assert rc == ep.EP_OK
    torch.cuda.synchronize()
    n_recv, n_exp, n_pad, status = bufs["info"].tolist()
    assert status == 0
    got = {k: v.cpu().numpy() for k, v in bufs.items()}
    got["recv_src_idx"] = got["recv_src_idx"][:n_recv]
    got["exp_src"] = got["exp_src"][:n_exp]
    got["pad_rows"] = got["pad_rows"][:n_pad]
    assert_plan_equal(got, oracle.plan(idx, w.S, w.P, w.E, w.A, Cq))


def test_static_scratch_rejects_plans_beyond_its_limit(lib):
    # 2^20 tokens with P+E = 2048 would need over 500 MB of tile bit matrices and prefixes
    w = WORKLOADS["tiny"].scaled(P=64, E=1984, S=16384, K=2, A=1)
    st = PlanBuffers(**{f: 1 << 20 for f, _ in PlanBuffers._fields_})  # never dereferenced
    rc = lib.ep_plan_static_scratch(1 << 20, w.S, w.P, w.K, w.E, w.A, 0, ctypes.byref(st), None)
    assert rc == ep.EP_ERR_CAPACITY
