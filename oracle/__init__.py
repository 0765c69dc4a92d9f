"""CPU oracle for the MoE expert-parallel routing plan, dispatch and combine.

TEST INFRASTRUCTURE ONLY.  Only the test-suite, the smoke check and the CPU
baseline leg of the benchmark may import this package.  The product library
(``combine_ep_plan_gb300``) never imports it and shares no code with it.

The arithmetic lives in ``ep_oracle.c`` (plain C, compiled with gcc, no
fast-math, no FP contraction).  This module only compiles it on demand,
allocates numpy outputs and calls it through ctypes.

The source is built twice: ``libep_oracle.so`` (single-threaded, the default)
and ``libep_oracle_omp.so`` (the same source with ``-fopenmp``: the per-row
loops of the scatter, combine and synthetic experts run on all host cores;
every element is computed by the same code, so the bits are identical).
``with oracle.parallel():`` routes calls to the multi-core build.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
import tempfile
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
# EP_ORACLE_SOURCE: a modified copy of ep_oracle.c to build and load instead
# (the planted-mistake test runs the pins against such copies); its library
# is written next to it.
_SRC = os.environ.get("EP_ORACLE_SOURCE") or os.path.join(_HERE, "ep_oracle.c")
_LIB = (os.path.splitext(_SRC)[0] + ".so" if os.environ.get("EP_ORACLE_SOURCE")
        else os.path.join(_HERE, "libep_oracle.so"))
# the multi-core build of the same source (not made for a modified copy)
_LIB_OMP = None if os.environ.get("EP_ORACLE_SOURCE") else os.path.join(_HERE, "libep_oracle_omp.so")
_CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]

OK = 0
ERR_INVALID = 1
ERR_CAPACITY = 2


class OracleError(RuntimeError):
    def __init__(self, code: int):
        super().__init__({ERR_INVALID: "invalid routing input",
                          ERR_CAPACITY: "output capacity too small"}.get(code, f"error {code}"))
        self.code = code


def _compile(lib: str, extra) -> None:
    if os.path.exists(lib) and os.path.getmtime(lib) >= os.path.getmtime(_SRC):
        return
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=os.path.dirname(lib))
    os.close(fd)
    cmd = ["gcc", *_CFLAGS, *extra, "-o", tmp, _SRC, "-lm"]
    try:
        subprocess.run(cmd, check=True, capture_output=True, text=True)
        os.replace(tmp, lib)
    except subprocess.CalledProcessError as exc:  # pragma: no cover
        os.unlink(tmp)
        raise RuntimeError(f"oracle build failed:\n{exc.stderr}") from exc


def build(force: bool = False) -> str:
    """Compile the oracle source into its libraries next to it (atomic
    renames): the single-threaded one, and the OpenMP one when gcc supports
    -fopenmp.  Returns the single-threaded library's path."""
    if force:
        for lib in (_LIB, _LIB_OMP):
            if lib and os.path.exists(lib):
                os.unlink(lib)
    _compile(_LIB, [])
    if _LIB_OMP:
        try:
            _compile(_LIB_OMP, ["-fopenmp"])
        except RuntimeError:  # pragma: no cover - a gcc without OpenMP
            pass
    return _LIB


_libs = {}
_use_omp = False


def _load():
    """The active library: the OpenMP build inside ``parallel()``, else the
    single-threaded one."""
    omp = _use_omp and _LIB_OMP is not None
    if omp not in _libs:
        build()
        if omp:
            if not os.path.exists(_LIB_OMP):
                raise RuntimeError("the OpenMP build of the oracle is unavailable (gcc without -fopenmp)")
            # idle worker threads sleep instead of spinning between calls
            os.environ.setdefault("OMP_WAIT_POLICY", "PASSIVE")
        _libs[omp] = _setup(ctypes.CDLL(_LIB_OMP if omp else _LIB))
    return _libs[omp]


@contextlib.contextmanager
def parallel(enabled: bool = True):
    """Route oracle calls in this block to the OpenMP build (all host cores)."""
    global _use_omp
    old = _use_omp
    _use_omp = bool(enabled)
    try:
        yield
    finally:
        _use_omp = old


def threads() -> int:
    """Threads the active build's row loops use (1 for the plain build)."""
    return int(_load().ep_oracle_threads())


def omp_available() -> bool:
    build()
    return _LIB_OMP is not None and os.path.exists(_LIB_OMP)


def _setup(lib):
    P = ctypes.c_void_p
    i64 = ctypes.c_int64
    i32 = ctypes.c_int
    lib.ep_oracle_validate.argtypes = [P, i64, i32, i32, i32, i32, i32]
    lib.ep_oracle_validate.restype = i32
    lib.ep_oracle_plan.argtypes = [P, i64, i32, i32, i32, i32, i32] + [P] * 11 + [i64, P, P, P, i64, P]
    lib.ep_oracle_plan.restype = i32
    lib.ep_oracle_dispatch_bf16.argtypes = [P, i64, P, i64, i32, P]
    lib.ep_oracle_dispatch_bf16.restype = None
    lib.ep_oracle_dispatch_fp8.argtypes = [P, i64, P, i64, i32, P, P]
    lib.ep_oracle_dispatch_fp8.restype = None
    lib.ep_oracle_combine.argtypes = [P, i64, P, P, i64, i32, P]
    lib.ep_oracle_combine.restype = None
    lib.ep_oracle_expert_scale.argtypes = [P, i64, P, P, i32, P]
    lib.ep_oracle_expert_scale.restype = None
    lib.ep_oracle_expert_scale_rows.argtypes = [P, i64, P, i64, i32, P]
    lib.ep_oracle_expert_scale_rows.restype = None
    lib.ep_oracle_combine_bias.argtypes = [P, i64, P, P, P, i64, i32, P]
    lib.ep_oracle_combine_bias.restype = None
    lib.ep_oracle_dispatch_metadata.argtypes = [P, P, i64, i32, i64, P, P]
    lib.ep_oracle_dispatch_metadata.restype = None
    lib.ep_oracle_dispatch_fp8_input.argtypes = [P, P, i64, P, i64, i32, P, P]
    lib.ep_oracle_dispatch_fp8_input.restype = None
    lib.ep_oracle_dispatch_backward.argtypes = [P, i64, P, i64, i32, P]
    lib.ep_oracle_dispatch_backward.restype = None
    lib.ep_oracle_combine_backward.argtypes = [P, P, i64, P, P, i64, P, i64, i32, i32, P, P]
    lib.ep_oracle_combine_backward.restype = None
    lib.ep_oracle_expert_dequant.argtypes = [P, P, i64, i64, P]
    lib.ep_oracle_expert_dequant.restype = None
    lib.ep_oracle_f32_to_bf16.argtypes = [ctypes.c_float]
    lib.ep_oracle_f32_to_bf16.restype = ctypes.c_uint16
    lib.ep_oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
    lib.ep_oracle_bf16_to_f32.restype = ctypes.c_float
    lib.ep_oracle_f32_to_e4m3.argtypes = [ctypes.c_float]
    lib.ep_oracle_f32_to_e4m3.restype = ctypes.c_uint8
    lib.ep_oracle_e4m3_to_f32.argtypes = [ctypes.c_uint8]
    lib.ep_oracle_e4m3_to_f32.restype = ctypes.c_float
    lib.ep_oracle_max_recv_rows.argtypes = [i64, i32, i32]
    lib.ep_oracle_max_recv_rows.restype = i64
    lib.ep_oracle_max_expanded_rows.argtypes = [i64, i32, i32, i32, i32]
    lib.ep_oracle_max_expanded_rows.restype = i64
    lib.ep_oracle_threads.argtypes = []
    lib.ep_oracle_threads.restype = i32
    return lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


@dataclass
class Plan:
    """All plan outputs, named as in the dispatch handle of the pages."""
    S: int
    P: int
    K: int
    E: int
    A: int
    C: int
    is_token_in_rank: np.ndarray      # [T,P] u8
    num_tokens_per_rank: np.ndarray   # [P,P] i32  [s][d]
    num_tokens_per_expert: np.ndarray  # [P,E] i32  [s][e]
    expert_counts: np.ndarray         # [E]   i32
    num_recv: np.ndarray              # [P]   i32
    rank_prefix: np.ndarray           # [P,P] i32  inclusive over sources
    channel_prefix: np.ndarray        # [P,P,C] i32 [s][d][c] inclusive over channels
    recv_channel_prefix: np.ndarray   # [P,P,C] i32 [d][s][c] segment start
    send_head: np.ndarray             # [T,P] i32
    recv_offsets: np.ndarray          # [P+1] i32
    recv_src_idx: np.ndarray          # [N_recv] i32
    expert_offsets: np.ndarray        # [E+1] i32
    slot: np.ndarray                  # [T,K] i32
    exp_src: np.ndarray               # [N_exp] i32

    @property
    def T(self) -> int:
        return self.P * self.S

    @property
    def num_expanded(self) -> int:
        return int(self.expert_offsets[-1])

    @property
    def num_recv_total(self) -> int:
        return int(self.recv_offsets[-1])


def default_channels(S: int, C: int = 0) -> int:
    return C if C > 0 else max(1, min(16, S))


def validate(topk_idx: np.ndarray, S: int, P: int, E: int, A: int, C: int = 0) -> int:
    idx = np.ascontiguousarray(topk_idx, dtype=np.int64)
    K = idx.shape[1]
    return _load().ep_oracle_validate(_ptr(idx), S, P, K, E, A, default_channels(S, C))


def max_recv_rows(S: int, P: int, K: int) -> int:
    """Worst-case receive rows over all destinations (the recv_src_idx size)."""
    return int(_load().ep_oracle_max_recv_rows(S, P, K))


def max_expanded_rows(S: int, P: int, K: int, E: int, A: int) -> int:
    """Worst-case expanded rows, padding included (the exp_src size)."""
    return int(_load().ep_oracle_max_expanded_rows(S, P, K, E, A))


def plan(topk_idx: np.ndarray, S: int, P: int, E: int, A: int, C: int = 0) -> Plan:
    lib = _load()
    idx = np.ascontiguousarray(topk_idx, dtype=np.int64)
    T, K = idx.shape
    assert T == P * S, "topk_idx must have P*S rows"
    C = default_channels(S, C)
    rcap = max(1, lib.ep_oracle_max_recv_rows(S, P, K))
    xcap = max(1, lib.ep_oracle_max_expanded_rows(S, P, K, E, A))
    o = dict(
        is_token_in_rank=np.zeros((T, P), np.uint8),
        num_tokens_per_rank=np.zeros((P, P), np.int32),
        num_tokens_per_expert=np.zeros((P, E), np.int32),
        expert_counts=np.zeros(E, np.int32),
        num_recv=np.zeros(P, np.int32),
        rank_prefix=np.zeros((P, P), np.int32),
        channel_prefix=np.zeros((P, P, C), np.int32),
        recv_channel_prefix=np.zeros((P, P, C), np.int32),
        send_head=np.zeros((T, P), np.int32),
        recv_offsets=np.zeros(P + 1, np.int32),
        recv_src_idx=np.zeros(rcap, np.int32),
        expert_offsets=np.zeros(E + 1, np.int32),
        slot=np.zeros((T, K), np.int32),
        exp_src=np.zeros(xcap, np.int32),
    )
    sizes = np.zeros(2, np.int64)
    rc = lib.ep_oracle_plan(
        _ptr(idx), S, P, K, E, A, C,
        _ptr(o["is_token_in_rank"]), _ptr(o["num_tokens_per_rank"]),
        _ptr(o["num_tokens_per_expert"]), _ptr(o["expert_counts"]), _ptr(o["num_recv"]),
        _ptr(o["rank_prefix"]), _ptr(o["channel_prefix"]), _ptr(o["recv_channel_prefix"]),
        _ptr(o["send_head"]), _ptr(o["recv_offsets"]), _ptr(o["recv_src_idx"]), rcap,
        _ptr(o["expert_offsets"]), _ptr(o["slot"]), _ptr(o["exp_src"]), xcap, _ptr(sizes))
    if rc != OK:
        raise OracleError(rc)
    o["recv_src_idx"] = o["recv_src_idx"][: int(sizes[0])].copy()
    o["exp_src"] = o["exp_src"][: int(sizes[1])].copy()
    return Plan(S=S, P=P, K=K, E=E, A=A, C=C, **o)


def dispatch_bf16(x_bits: np.ndarray, pl: Plan, zero_pad: bool = True) -> np.ndarray:
    """x_bits: [T,H] uint16 bf16 bit patterns -> [N_exp,H] uint16."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    H = x.shape[1]
    n = pl.num_expanded
    out = np.zeros((n, H), np.uint16)
    _load().ep_oracle_dispatch_bf16(_ptr(x), H, _ptr(pl.exp_src), n, int(zero_pad), _ptr(out))
    return out


def dispatch_fp8(x_bits: np.ndarray, pl: Plan, zero_pad: bool = True):
    """-> (q [N_exp,H] uint8 E4M3 codes, scales [N_exp,H/128] float32)."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    H = x.shape[1]
    assert H % 128 == 0
    n = pl.num_expanded
    q = np.zeros((n, H), np.uint8)
    sc = np.zeros((n, H // 128), np.float32)
    _load().ep_oracle_dispatch_fp8(_ptr(x), H, _ptr(pl.exp_src), n, int(zero_pad), _ptr(q), _ptr(sc))
    return q, sc


def combine(y_bits: np.ndarray, pl: Plan, topk_weights: np.ndarray, bias_bits: np.ndarray = None) -> np.ndarray:
    """y_bits: [N_exp,H] uint16 bf16; topk_weights [T,K] f32; optional bias
    [T,H] bf16 bits -> [T,H] uint16 bf16."""
    y = np.ascontiguousarray(y_bits, dtype=np.uint16)
    w = np.ascontiguousarray(topk_weights, dtype=np.float32)
    H = y.shape[1]
    out = np.zeros((pl.T, H), np.uint16)
    if bias_bits is None:
        _load().ep_oracle_combine(_ptr(y), H, _ptr(pl.slot), _ptr(w), pl.T, pl.K, _ptr(out))
    else:
        b = np.ascontiguousarray(bias_bits, dtype=np.uint16)
        _load().ep_oracle_combine_bias(_ptr(y), H, _ptr(pl.slot), _ptr(w), _ptr(b), pl.T, pl.K, _ptr(out))
    return out


def dispatch_metadata(pl: Plan, topk_weights: np.ndarray):
    """-> (recv_weights [N_exp] f32, recv_meta [N_exp,2] i32 = {source token, slot k})."""
    w = np.ascontiguousarray(topk_weights, dtype=np.float32)
    n = pl.num_expanded
    rw = np.zeros(n, np.float32)
    rm = np.zeros((n, 2), np.int32)
    _load().ep_oracle_dispatch_metadata(_ptr(pl.slot), _ptr(w), pl.T, pl.K, n, _ptr(rw), _ptr(rm))
    return rw, rm


def dispatch_fp8_input(xq: np.ndarray, xs: np.ndarray, pl: Plan, zero_pad: bool = True):
    """Pre-quantised input: codes [T,H] u8 + scales [T,H/128] f32 -> expanded rows."""
    q = np.ascontiguousarray(xq, dtype=np.uint8)
    s = np.ascontiguousarray(xs, dtype=np.float32)
    H = q.shape[1]
    n = pl.num_expanded
    oq = np.zeros((n, H), np.uint8)
    osc = np.zeros((n, H // 128), np.float32)
    _load().ep_oracle_dispatch_fp8_input(_ptr(q), _ptr(s), H, _ptr(pl.exp_src), n, int(zero_pad), _ptr(oq), _ptr(osc))
    return oq, osc


def dispatch_backward(grad_recv_bits: np.ndarray, pl: Plan) -> np.ndarray:
    """grad_recv [N_exp,H] bf16 bits -> grad_x [T,H] bf16 bits."""
    g = np.ascontiguousarray(grad_recv_bits, dtype=np.uint16)
    H = g.shape[1]
    out = np.zeros((pl.T, H), np.uint16)
    _load().ep_oracle_dispatch_backward(_ptr(g), H, _ptr(pl.slot), pl.T, pl.K, _ptr(out))
    return out


def combine_backward(grad_out_bits: np.ndarray, y_bits: np.ndarray, pl: Plan, topk_weights: np.ndarray,
                     zero_pad: bool = True):
    """-> (grad_y [N_exp,H] bf16 bits, grad_w [T,K] float64)."""
    go = np.ascontiguousarray(grad_out_bits, dtype=np.uint16)
    y = np.ascontiguousarray(y_bits, dtype=np.uint16)
    w = np.ascontiguousarray(topk_weights, dtype=np.float32)
    H = go.shape[1]
    n = pl.num_expanded
    gy = np.zeros((n, H), np.uint16)
    gw = np.zeros((pl.T, pl.K), np.float64)
    _load().ep_oracle_combine_backward(_ptr(go), _ptr(y), H, _ptr(pl.slot), _ptr(pl.exp_src), n, _ptr(w),
                                       pl.T, pl.K, int(zero_pad), _ptr(gy), _ptr(gw))
    return gy, gw


def expert_scale(x_exp_bits: np.ndarray, pl: Plan) -> np.ndarray:
    x = np.ascontiguousarray(x_exp_bits, dtype=np.uint16)
    H = x.shape[1]
    y = np.zeros_like(x)
    _load().ep_oracle_expert_scale(_ptr(x), H, _ptr(pl.exp_src), _ptr(pl.expert_offsets), pl.E, _ptr(y))
    return y


def expert_scale_rows(x_rows_bits: np.ndarray, row_expert: np.ndarray, E: int) -> np.ndarray:
    x = np.ascontiguousarray(x_rows_bits, dtype=np.uint16)
    re = np.ascontiguousarray(row_expert, dtype=np.int32)
    n, H = x.shape
    y = np.zeros_like(x)
    _load().ep_oracle_expert_scale_rows(_ptr(x), H, _ptr(re), n, E, _ptr(y))
    return y


def expert_dequant(q: np.ndarray, scales: np.ndarray) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.uint8)
    sc = np.ascontiguousarray(scales, dtype=np.float32)
    n, H = q.shape
    y = np.zeros((n, H), np.uint16)
    _load().ep_oracle_expert_dequant(_ptr(q), _ptr(sc), H, n, _ptr(y))
    return y


def f32_to_bf16(v: float) -> int:
    return int(_load().ep_oracle_f32_to_bf16(v))


def bf16_to_f32(b: int) -> float:
    return float(_load().ep_oracle_bf16_to_f32(b))


def f32_to_e4m3(v: float) -> int:
    return int(_load().ep_oracle_f32_to_e4m3(v))


def e4m3_to_f32(b: int) -> float:
    return float(_load().ep_oracle_e4m3_to_f32(b))
