"""Host logic of bench.py on CPU: the ledger, the max-over-ranks aggregation
of replicas (gloo, world size 2) and the profile-summary reader."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from combine_ep_plan_gb300.inputs import WORKLOADS  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    bench.dist_init(use_cuda=False)
    # each replica moves 1 GB per step; rank 1 is the slow one (4 ms per step)
    local_ms = [100.0, 200.0][rank]
    agg = bench.aggregate(1e9, 1000, local_ms, world, steps=50)
    bench.barrier()
    q.put((rank, agg))
    dist.destroy_process_group()


def test_replicas_aggregate_over_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in (0, 1):
        agg = res[r]
        assert agg["ms_per_step"] == pytest.approx(4.0)       # max over ranks: 200 ms / 50
        assert agg["gbs"] == pytest.approx(2 * 1e9 / 4e-3 / 1e9)  # both ranks' bytes / slowest time
        assert agg["tokens_per_s"] == pytest.approx(2 * 1000 / 4e-3)


def test_single_process_aggregate_is_identity():
    agg = bench.aggregate(2e9, 16384, 10.0, 1, steps=10)
    assert agg["ms_per_step"] == 1.0
    assert agg["gbs"] == pytest.approx(2000.0)


def test_ledger_matches_the_pages_per_token_bytes():
    # [TT] §1.2: k*d*b per token per direction; here per token with every
    # slot valid and no padding, dispatch writes K*H*2 and reads H*2
    w = WORKLOADS["bf16"]
    n_valid = w.T * w.K
    led = bench.ledger(w, n_exp=n_valid, n_valid=n_valid, n_recv=0)
    assert led["dispatch"] == w.T * (w.H * 2 + 86016 + w.K * 4)
    assert led["combine"] == w.T * (86016 + w.K * 8 + w.H * 2)
    assert led["total"] == led["plan"] + led["dispatch"] + led["combine"]


def test_profiled_traffic_requires_matching_source_hash(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    digest = bench.source_digest("ep_dispatch_kernels.cu")
    (prof / "k.bf16.md").write_text(f"# x\n- source_sha256: `{digest}` (sha256 prefix when captured)\n"
                                    "- dram_bytes_per_launch: 123.5\n")
    (prof / "k2.bf16.md").write_text("- source_sha256: `deadbeef`\n- dram_bytes_per_launch: 9\n")
    (prof / "k3.rt.md").write_text(f"- source_sha256: `{digest}`\n- dram_bytes_per_launch_captured: 7 (small)\n"
                                   "- dram_bytes_per_launch: 28 (scaled to a full launch)\n")
    real_root = bench.ROOT
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    os.makedirs(tmp_path / "combine_ep_plan_gb300" / "csrc")
    with open(os.path.join(real_root, "combine_ep_plan_gb300", "csrc", "ep_dispatch_kernels.cu"), "rb") as f:
        (tmp_path / "combine_ep_plan_gb300" / "csrc" / "ep_dispatch_kernels.cu").write_bytes(f.read())
    assert bench.profiled_traffic("k", "ep_dispatch_kernels.cu", "bf16") == 123.5
    assert bench.profiled_traffic("k2", "ep_dispatch_kernels.cu", "bf16") is None
    assert bench.profiled_traffic("missing", "ep_dispatch_kernels.cu", "bf16") is None
    assert bench.profiled_traffic("k3", "ep_dispatch_kernels.cu", "rt") == 28.0  # a scaled capture's note


def test_reference_arm_prints_one_line_on_cpu():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                        "--warmup", "3", "--workload", "tiny"], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"


def test_profile_summaries_name_their_command():
    """Every committed ncu summary states the command that made it, and that
    command runs committed files only (README.md is the index)."""
    prof = os.path.join(ROOT, "profiles")
    names = [n for n in os.listdir(prof) if n.endswith(".md") and n != "README.md"]
    assert names
    for n in names:
        text = open(os.path.join(prof, n)).read()
        cmds = [line for line in text.splitlines() if line.startswith("- command:")]
        assert cmds, n
        for line in cmds:
            assert "_work/" not in line and "python bench.py" in line, (n, line)


def test_reference_config_names_a_sample_only_when_it_is_smaller():
    """The reference arm's config equals the measured arm's when its sample
    is the whole workload, and names the sample size only when it is not."""
    w = WORKLOADS["bf16"]
    assert bench.workload_config(w, sample_S=w.S) == bench.workload_config(w)
    assert bench.workload_config(w, sample_S=w.S // 4)["sample_tokens_per_rank"] == w.S // 4
