"""Helpers shared by the GPU parity tests: run the CUDA path, read its plan
arrays back, and compare with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from combine_ep_plan_gb300.inputs import bits_to_bf16_tensor, draw_hidden, draw_topk, hidden_seed

PLAN_FIELDS = [
    "is_token_in_rank", "send_head", "num_tokens_per_rank", "num_tokens_per_expert", "expert_counts",
    "num_recv", "rank_prefix", "channel_prefix", "recv_channel_prefix", "recv_offsets", "recv_src_idx",
    "expert_offsets", "slot", "exp_src",
]


def gpu_plan_arrays(h) -> dict:
    n_exp, n_recv = h.sizes()
    out = {name: h.field(name).cpu().numpy() for name in PLAN_FIELDS + ["pad_rows"]}
    out["recv_src_idx"] = out["recv_src_idx"][:n_recv]
    out["exp_src"] = out["exp_src"][:n_exp]
    n_pad = int(n_exp - out["expert_counts"].sum())
    out["pad_rows"] = out["pad_rows"][:n_pad]
    return out


def assert_plan_equal(gpu: dict, pl: oracle.Plan):
    for name in PLAN_FIELDS:
        a = gpu[name]
        b = getattr(pl, name)
        assert a.shape == b.shape, f"{name}: shape {a.shape} != oracle {b.shape}"
        if not np.array_equal(a, b):
            bad = np.argwhere(a != b)
            raise AssertionError(f"{name}: {len(bad)} mismatches, first at {bad[:5].tolist()}: "
                                 f"gpu {a[tuple(bad[0])]} oracle {b[tuple(bad[0])]}")
    assert np.array_equal(gpu["pad_rows"], np.nonzero(pl.exp_src < 0)[0].astype(np.int32))


def to_gpu_inputs(w, idx, weights, x_bits=None):
    idx_t = torch.from_numpy(idx).cuda()
    w_t = torch.from_numpy(weights).cuda()
    x_t = bits_to_bf16_tensor(x_bits).cuda() if x_bits is not None else None
    return idx_t, w_t, x_t


def draw(w, seed=None):
    idx, weights = draw_topk(w, seed)
    x = draw_hidden(w.T, w.H, hidden_seed(w))
    return idx, weights, x


def u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.uint8).numpy()


_BYTES = {1: torch.uint8, 2: torch.int16, 4: torch.int32, 8: torch.int64}


def assert_bits_equal(got: torch.Tensor, want: np.ndarray, name: str = "array"):
    """Bit-for-bit equality of a device tensor with an oracle array, compared
    on the device (whole arrays at full size); on a mismatch, the count and
    the first positions."""
    want = np.ascontiguousarray(want)
    assert tuple(got.shape) == want.shape, f"{name}: shape {tuple(got.shape)} != oracle {want.shape}"
    if got.numel() == 0:
        return
    dt = _BYTES[want.dtype.itemsize]
    assert got.element_size() == want.dtype.itemsize, f"{name}: element size differs"
    g = got.contiguous().view(dt)
    w = torch.from_numpy(want.view(np.dtype(str(dt).replace("torch.", "")))).to(got.device)
    if torch.equal(g, w):
        return
    bad = torch.nonzero(g != w)
    first = bad[:5].cpu().tolist()
    raise AssertionError(f"{name}: {bad.shape[0]} of {g.numel()} elements differ, first at {first}: "
                         f"gpu {[int(g[tuple(i)]) for i in first]} oracle {[int(w[tuple(i)]) for i in first]}")
