"""The N > 1 path of bench.py on CPU: world-size-2 gloo ranks (replicas
only, so the only collectives are the timing barrier and the max over
ranks), and the reference arm under torchrun. No GPU."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, ws, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    got_ws, got_rank, local = bench.dist_init()
    assert (got_ws, got_rank, local) == (ws, rank, rank)
    import torch.distributed as dist
    assert dist.get_backend() == "gloo"
    bench.barrier(ws)
    # rank r took 1 + r seconds for 10 steps of batch 3: the job rate is every
    # rank's tokens over the slowest rank's time
    rate, el = bench.replica_rate(ws, 3, 10, 1.0 + rank)
    out[rank] = (rate, el)
    bench.barrier(ws)
    dist.destroy_process_group()


def test_replica_rate_two_gloo_ranks():
    ws = 2
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(_rank, args=(ws, _free_port(), out), nprocs=ws, join=True)
    for r in range(ws):
        rate, el = out[r]
        assert el == 2.0
        assert rate == pytest.approx(ws * 3 * 10 / 2.0)


def test_replica_rate_single_process():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.replica_rate(1, 16, 64, 2.0) == (16 * 64 / 2.0, 2.0)


WRAPPER = """
import sys
sys.path.insert(0, {root!r})
from transformer_decode_gb300 import synth
# the launch logic under test, on models the CPU makes fast
synth.QWEN2_0P5B = synth.TINY
synth.QWEN3_8B = synth.TINY_QKNORM
import bench
bench.main()
"""


@pytest.mark.parametrize("workload", [None, "qwen2_0p5b_b1_greedy64"])
def test_reference_arm_under_torchrun_prints_one_line(tmp_path, workload):
    """--impl reference at N = 2 under torchrun: rank 0 times the oracle and
    prints one JSON line; rank 1 exits 0 without work. The default workload
    (the 8B shape at 4096 past positions) and the 0.5B prompt run."""
    script = tmp_path / "bench_tiny.py"
    script.write_text(WRAPPER.format(root=ROOT))
    env = dict(os.environ, OMP_NUM_THREADS="2")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           str(script), "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3"]
    if workload:
        cmd += ["--workload", workload]
    r = subprocess.run(cmd, capture_output=True, text=True, cwd=ROOT, env=env, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["config"]["workload"] == (workload or "qwen3_8b_shape_b1_past4096")
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_step_bytes_against_the_page_counts():
    """The roofline's algorithmic bytes: every parameter read once per step
    (the tied embedding as the head) is 2 bytes x the nanoinfer page's
    494,032,768 parameters; the embedding row, the K/V of the cached
    positions (24 KiB per token in fp32 across the 24 layers, the page's
    figure), the new K/V, the logits and token/position words come on top."""
    sys.path.insert(0, ROOT)
    import bench
    from transformer_decode_gb300 import synth
    s = synth.QWEN2_0P5B
    total_params = 494032768
    H, V = s.hidden, s.vocab
    for p in (0, 31, 95):
        want = (2 * total_params + 2 * H          # weights once, plus the gathered row
                + (p + 1) * 24576 + 24576          # K/V read for slots 0..p, and written
                + 4 * V + 8)                       # logits out, token and position in
        assert bench.step_bytes(s, 1, [p]) == want
    # the bf16 cache halves only the K/V terms
    assert bench.step_bytes(s, 1, [95], kv_elem=2) == bench.step_bytes(s, 1, [95]) - 97 * 12288
    # W8A8: the seven projections at one byte per weight plus one fp32 scale per row
    proj = s.n_layers * ((s.q_dim + 2 * s.kv_dim) * H + s.q_dim * H + 3 * s.ffn * H)
    rows = s.n_layers * ((s.q_dim + 2 * s.kv_dim) + H + 2 * s.ffn + H)
    assert bench.step_bytes(s, 1, [95], w8a8=True) == \
        bench.step_bytes(s, 1, [95]) - 2 * proj + proj + 4 * rows


def test_step_bytes_int8_head():
    """With the tied head int8 (one fp32 scale a row), the head and the
    gathered row cost one byte a weight plus the scales instead of two."""
    sys.path.insert(0, ROOT)
    import bench
    from transformer_decode_gb300 import synth
    s = synth.QWEN2_0P5B
    a = bench.step_bytes(s, 1, [95], w8a8=True)
    b = bench.step_bytes(s, 1, [95], w8a8=True, int8_head=True)
    assert a - b == (s.vocab * s.hidden - 4 * s.vocab) + (s.hidden - 4)


def test_step_bytes_int4_matches_the_footprint_formula():
    """INT4 bytes per step: the projections' share equals the one the
    quantisation oracle's footprint (pinned to the page's table) implies:
    footprint(int4-gG) - footprint(fp32) + 4 x projection weights."""
    sys.path.insert(0, ROOT)
    import bench
    from oracle import quant
    from transformer_decode_gb300 import synth
    s = synth.QWEN2_0P5B
    proj = s.n_layers * ((s.q_dim + 2 * s.kv_dim) * s.hidden + s.q_dim * s.hidden
                         + 3 * s.ffn * s.hidden)
    for g in (32, 128):
        int4_proj = (quant.footprint_bytes(s, f"int4-g{g}") - quant.footprint_bytes(s, "fp32")
                     + 4 * proj)
        assert bench.step_bytes(s, 1, [95], int4_group=g) == \
            bench.step_bytes(s, 1, [95]) - 2 * proj + int4_proj
