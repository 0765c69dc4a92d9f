"""The C ABI from a plain C program (tests/c_abi/ep_abi_client.c): compiled
with gcc against include/ep_plan.h and linked to libep_gb300.so, with no
Python or C++ in the caller.  On CPU it must compile and link; on the GPU
its plan arrays, BF16 and FP8 dispatches and combine are compared with the
oracle, whole arrays, bit for bit."""
import glob
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
from combine_ep_plan_gb300.inputs import WORKLOADS, draw_hidden, draw_topk

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_abi", "ep_abi_client.c")


def _cuda_home() -> str:
    nvcc = shutil.which("nvcc")
    return os.environ.get("CUDA_HOME") or (os.path.dirname(os.path.dirname(nvcc)) if nvcc else "/usr/local/cuda")


def _cudart_dir(cuda: str) -> str:
    for d in [os.path.join(cuda, "lib64")] + sorted(glob.glob(os.path.join(cuda, "targets", "*", "lib"))):
        if glob.glob(os.path.join(d, "libcudart.so*")):
            return d
    pytest.skip("libcudart not found")


def build_client(out_dir: str) -> str:
    """gcc, C11, the library's public header only; returns the executable."""
    from combine_ep_plan_gb300 import build
    lib = build.build()
    cuda = _cuda_home()
    exe = os.path.join(out_dir, "ep_abi_client")
    cmd = ["gcc", "-std=c11", "-O2", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(cuda, "include"), SRC, "-o", exe,
           "-L", os.path.dirname(lib), "-lep_gb300", "-L", _cudart_dir(cuda), "-lcudart",
           f"-Wl,-rpath,{os.path.dirname(lib)}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    return exe


def test_c_client_compiles_and_links(tmp_path):
    assert os.access(build_client(str(tmp_path)), os.X_OK)


@pytest.mark.gpu
@pytest.mark.parametrize("name,S,H", [("bf16", 300, 1024), ("fp8", 97, 2048)])
def test_c_client_matches_the_oracle(tmp_path, name, S, H):
    w = WORKLOADS[name].scaled(S=S, H=H)
    idx, wts = draw_topk(w)
    idx[::17, 1] = -1
    x = draw_hidden(w.T, w.H, 77)
    inp, outp = tmp_path / "in.bin", tmp_path / "out.bin"
    with open(inp, "wb") as f:
        f.write(np.array([w.S, w.P, w.K, w.E, w.A, w.H], np.int64).tobytes())
        f.write(np.ascontiguousarray(idx, np.int64).tobytes())
        f.write(np.ascontiguousarray(x).tobytes())
        f.write(np.ascontiguousarray(wts, np.float32).tobytes())
    exe = build_client(str(tmp_path))
    r = subprocess.run([exe, str(inp), str(outp)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr

    raw = open(outp, "rb").read()
    at = 0

    def take(dtype, n):
        nonlocal at
        a = np.frombuffer(raw, dtype, count=n, offset=at)
        at += a.nbytes
        return a

    n_exp, n_recv = (int(v) for v in take(np.int64, 2))
    T, K = w.T, w.K
    pl = oracle.plan(idx, w.S, w.P, w.E, w.A)
    assert (n_exp, n_recv) == (pl.num_expanded, pl.num_recv_total)
    assert np.array_equal(take(np.int32, T * K).reshape(T, K), pl.slot)
    assert np.array_equal(take(np.int32, n_exp), pl.exp_src)
    recv = take(np.uint16, n_exp * H).reshape(n_exp, H)
    q = take(np.uint8, n_exp * H).reshape(n_exp, H)
    sc = take(np.float32, n_exp * H // 128).reshape(n_exp, H // 128)
    out = take(np.uint16, T * H).reshape(T, H)
    assert at == len(raw)
    with oracle.parallel():
        assert np.array_equal(recv, oracle.dispatch_bf16(x, pl, True))
        q_ref, s_ref = oracle.dispatch_fp8(x, pl, True)
        assert np.array_equal(q, q_ref)
        assert np.array_equal(sc.view(np.uint32), np.ascontiguousarray(s_ref, np.float32).view(np.uint32))
        assert np.array_equal(out, oracle.combine(recv, pl, wts))
