"""Host-side logic of bench.py on the CPU: the algorithmic byte count against
the bandwidth figures the explainer prints, and the multi-rank aggregation
(gloo, world size 2)."""
import os
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_state_traffic_matches_the_explainer():
    """"ReplaySSM" explainer, section 1 and 5.1: the packed decode moves 8*dv*dk
    state bytes per head-step; ReplaySSM with one checkpoint read per step and a
    flush every L steps moves 4*dv*dk*(1 + 1/L) on average, 53.1% at L = 16."""
    K = V = 128
    for L in (1, 4, 8, 16, 32):
        cycle = [bench.head_step_parts(K, V, 2, p, p == L - 1, 2, 2, 2)["state"] for p in range(L)]
        assert sum(cycle) / L == pytest.approx(4 * V * K * (1 + 1 / L))
    packed = 8 * V * K
    ratio = sum(bench.head_step_parts(K, V, 2, p, p == 15, 2, 2, 2)["state"] for p in range(16)) / 16 / packed
    assert round(100 * ratio, 1) == 53.1
    # 64 KiB of fp32 state per 128 x 128 head, 128 KiB read + write (section 1)
    assert bench.head_step_parts(K, V, 2, 0, True, 2, 2, 0)["state"] == 128 * 1024


def test_amortised_bytes_per_head_step():
    """fp16 ring, bf16 in/out, GQA 2:1, L = 16, cursor uniform over the cycle:
    65536 (read) + 7.5 * 388 (replay) + 15/16 * 388 (append) + 4096 (flush)
    + 520 (inputs) + 256 (output) bytes."""
    L = 16
    mean = sum(bench.head_step_bytes(128, 128, 2, p, p == L - 1, 2, 2, 2) for p in range(L)) / L
    assert mean == pytest.approx(65536 + 7.5 * 388 + 15 / 16 * 388 + 4096 + 520 + 256)
    assert bench.packed_head_step_bytes(128, 128, 2, 2, 2) == 131072 + 520 + 256


def test_launch_bytes_counts_padding_rows():
    from linear_attention_decode_gb300 import inputs as I
    w = I.QWEN3NEXT_LAYER
    one = bench.launch_bytes(w, [3], [False], 2, 0)
    assert bench.launch_bytes(w, [3], [False], 2, 4) == one + 4 * w.HV * w.V * 2
    # the live row's cursor is read and written once by the fused advance
    assert one == w.HV * bench.head_step_bytes(128, 128, 2, 3, False, 2, 2, 2) + 8
    assert bench.launch_bytes(w, [3], [False], 2, 0, cursors=False) == one - 8


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    elapsed = [0.25, 0.5][rank]
    m = bench.max_over_ranks(elapsed, torch.device("cpu"))
    q.put((rank, m, bench.job_throughput(1000.0, world, m)))
    dist.destroy_process_group()


def test_two_rank_aggregation_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29000 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for _, m, v in res:
        assert m == 0.5 and v == pytest.approx(2 * 1000.0 / 0.5)


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "2", "--warmup", "3"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_spec_window_bytes():
    """A window of T tokens reads the checkpoint once (not T times): at the
    benchmark's head shape (K=V=128, G=2, fp16 ring, bf16 inputs and output)."""
    ring_entry = 128 * 2 + 128 * 2 / 2 + 4
    inputs = 2 * 128 * 2 / 2 + 128 * 2 + 4 + 4
    assert bench.spec_head_bytes(128, 128, 2, 5, 4, 2, 2, 2) == 65536 + 9 * ring_entry + 4 * inputs + 4 * 256
    assert bench.fold_head_bytes(128, 128, 2, 7, 2) == 131072 + 7 * ring_entry
    kda_entry = 128 * 2 + 128 * 2 + 512
    assert bench.fold_head_bytes(128, 128, 1, 3, 2, kda=True) == 131072 + 3 * kda_entry


def test_acceptance_pool_is_a_prefix_count():
    import numpy as np
    acc = bench.acceptance_pool(np.random.default_rng(0), 64, 32, 4, 0.7)
    assert acc.min() >= 0 and acc.max() <= 4
    assert 0 < (acc == 0).mean() < 1 and (acc == 4).any()
    assert abs(acc.mean() - sum(0.7 ** i for i in range(1, 5))) < 0.15


def test_lossless_bytes():
    """Lossless verify: the state once, T tokens of inputs and outputs, T fp32
    tuples (u per value head, k shared by the G heads of a key head, g); the
    commit: the state in and out plus the accepted tuples, nothing when none
    is accepted.  Against a snapshot verify (the state read, T states written)
    the verify moves about (T + 1) / (1 + small) times fewer bytes."""
    inputs = 2 * 128 * 2 / 2 + 128 * 2 + 4 + 4          # q, k (per key head, G = 2), v, g, beta
    tuples = 4 * 128 + 4 * 128 / 2 + 4                 # u, k (G = 2), g
    assert bench.lossless_verify_head_bytes(128, 128, 2, 4, 2, 2) == 65536 + 4 * (inputs + 256) + 4 * tuples
    assert bench.lossless_commit_head_bytes(128, 128, 2, 3) == 131072 + 3 * tuples
    assert bench.lossless_commit_head_bytes(128, 128, 2, 0) == 0.0
    kda_tuples = 4 * 128 + 4 * 128 + 4 * 128           # G = 1, g per channel
    assert bench.lossless_commit_head_bytes(128, 128, 1, 2, kda=True) == 131072 + 2 * kda_tuples
    snapshot = 65536 * (1 + 8)
    assert 7.0 < snapshot / bench.lossless_verify_head_bytes(128, 128, 2, 8, 2, 2) < 8.0


def test_lossless_tuple_ratio_matches_the_pages():
    """sglang #42388 (The idea): keeping (u, k, g) costs HV (V + K + 1) floats per
    draft step instead of an HV V K snapshot, 63.8x less at K = V = 128.  The
    tuple bytes of the verify's byte model give that ratio with one key head per
    value head (G = 1); sharing k across a GQA group (G = 2) makes it larger."""
    def tuple_bytes(G):  # the verify's bytes for T = 1 minus the state read, inputs and output
        inputs = 2 * 128 * 2 / G + 128 * 2 + 4 + 4
        return bench.lossless_verify_head_bytes(128, 128, G, 1, 2, 2) - 65536 - inputs - 128 * 2
    assert round(4 * 128 * 128 / tuple_bytes(1), 1) == 63.8
    assert 4 * 128 * 128 / tuple_bytes(2) > 80


def test_workload_names_parse():
    """The named workloads the bench and its profiles use resolve to the shapes
    their names state."""
    from linear_attention_decode_gb300.constants import F16, F32, GATE_PER_K
    w = bench.pick_workload("kda_layer:64:f32")
    assert (w.L, w.ring_dtype, w.gate, w.B, w.N, w.HV, w.HK) == (64, F32, GATE_PER_K, 128, 256, 32, 32)
    assert "L=64 fp32 ring" in w.name
    w = bench.pick_workload("stack30:64")
    assert (w.B, w.N, w.L, w.ring_dtype, w.layers) == (64, 320, 16, F16, 30)
    w = bench.pick_workload("sweep:128:32:f32")
    assert (w.B, w.L, w.ring_dtype) == (128, 32, F32)
    with pytest.raises(SystemExit):
        bench.pick_workload("no_such_workload")
