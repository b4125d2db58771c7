"""Host-side pieces of bench.py: byte accounting, the reference (oracle) arm
on the tiny workload, and the max-over-ranks timing across two gloo ranks."""
import json
import os
import subprocess
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from paged_kv_cache_xs_gb300 import workloads as wl  # noqa: E402


def test_step_bytes_tiny_config():
    cfg = wl.CONFIGS[0]
    lens = torch.tensor([8, 21], dtype=torch.int32)
    by = bench.step_bytes(cfg, lens)
    s = 4
    kv = (8 + 21) * 12 * 64 * 2 * s
    assert by["kv"] == kv
    tables = (1 + 2) * 4 + 4 * 2
    assert by["attn"] == kv + 2 * 12 * 64 * s + tables
    assert by["step"] == by["attn"] + 2 * 12 * 64 * s + 2 * 2 * 12 * 64 * s * 2


def test_reference_arm_tiny_config():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--config", "0", "--steps", "2", "--warmup", "3",
                        "--ref-step-seconds", "0.05"],
                       capture_output=True, text=True, timeout=300,
                       env={**os.environ, "CUDA_VISIBLE_DEVICES": ""})
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(dist)
    got = bench.max_over_ranks(1.5 + rank, dist)
    dist.destroy_process_group()
    q.put((rank, got))


def test_max_over_ranks_gloo_two_ranks():
    import multiprocessing as mp
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
    assert res == {0: 2.5, 1: 2.5}


def test_prefill_oracle_leg_on_host_tensors():
    # The prefill line's oracle leg on a small CPU case whose "GPU output" is
    # the oracle's own: the parity object reports zero error and the rate
    # bookkeeping is positive and consistent.
    import oracle
    g = torch.Generator().manual_seed(5)
    Hq, Hkv, D, bs, total = 4, 2, 64, 16, 48
    pages = total // bs
    ids = torch.randperm(2 * pages, generator=g)[:pages].to(torch.int32)
    kc = torch.randn(2 * pages, Hkv, bs, D, generator=g).to(torch.bfloat16)
    vc = torch.randn(2 * pages, Hkv, bs, D, generator=g).to(torch.bfloat16)
    q = torch.randn(total, Hq, D, generator=g).to(torch.bfloat16)
    out = oracle.paged_prefill(q, kc, vc, ids, 0, D ** -0.5)
    flop = 4 * D * Hq * total * (total + 1) / 2
    base, parity = bench.prefill_cpu_baseline(q, kc, vc, ids, out, total, flop, 0.01)
    assert parity["max_abs_err"] == 0.0 and parity["ok"] and 1 <= parity["rows"] <= total
    assert base["kind"] == "oracle" and base["value"] > 0 and base["tflops"] > 0


def test_swap_oracle_leg_on_host_tensors():
    g = torch.Generator().manual_seed(6)
    nb, n = 40, 12
    kd = torch.randn(nb, 2, 16, 64, generator=g).to(torch.bfloat16)
    vd = torch.randn(nb, 2, 16, 64, generator=g).to(torch.bfloat16)
    blocks = torch.randperm(nb, generator=g)[:n]
    kh, vh = kd[blocks].clone(), vd[blocks].clone()      # a correct swap-out
    base, parity = bench.swap_cpu_baseline(kd, vd, kh, vh, blocks, 0.02)
    assert parity["bit_exact"] and parity["blocks"] == n and base["value"] > 0
    vh[3, 1, 5, 7] += 1                                  # one element off
    _, parity = bench.swap_cpu_baseline(kd, vd, kh, vh, blocks, 0.02)
    assert not parity["bit_exact"]


def test_alloc_oracle_leg_on_host_tensors():
    import oracle
    g = torch.Generator().manual_seed(7)
    B, bs, width, nb, nsteps = 6, 16, 8, 64, 20
    lens = torch.randint(0, 60, (B,), generator=g, dtype=torch.int32)
    perm = torch.randperm(nb, generator=g).to(torch.int32)
    bt = torch.full((B, width), -1, dtype=torch.int32)
    pos = 0
    for b in range(B):
        p = (int(lens[b]) + bs - 1) // bs
        bt[b, :p] = perm[pos:pos + p]
        pos += p
    stack, top = perm[pos:].clone(), nb - pos
    obt, olens, otop = bt, lens, top
    for _ in range(nsteps):                       # stands in for the device's result
        obt, olens, otop, _ = oracle.block_alloc_decode(obt, olens, bs, stack, otop)
    base, parity = bench.alloc_cpu_baseline(bt, lens, stack, top, nsteps, bs, obt, olens, otop)
    assert parity["exact"] and base["value"] > 0
    bad = olens.clone()
    bad[2] += 1                                    # one length off
    _, parity = bench.alloc_cpu_baseline(bt, lens, stack, top, nsteps, bs, obt, bad, otop)
    assert not parity["exact"]


def test_reference_arm_under_torchrun_two_ranks():
    # The launch the driver uses for N > 1 (torchrun, one process per rank,
    # rendezvous on 127.0.0.1), here on gloo without a GPU: rank 0 alone runs
    # the oracle arm and prints one JSON line; the other rank exits 0.
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
                        "--nproc-per-node", "2", "--master-addr", "127.0.0.1",
                        "--master-port", str(port), os.path.join(ROOT, "bench.py"),
                        "--impl", "reference", "--config", "0", "--gpus", "2", "--steps", "2",
                        "--warmup", "3", "--ref-step-seconds", "0.05"],
                       capture_output=True, text=True, timeout=300,
                       env={**os.environ, "CUDA_VISIBLE_DEVICES": "", "OMP_NUM_THREADS": "1"})
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0


def test_decode_row_parity_covers_every_sequence_and_layer():
    # The rows' oracle leg: every sequence of every layer of the timed output
    # against the oracle.  Here the "GPU output" is the oracle's own, rounded
    # to bf16 (within tolerance); one element off in the last layer is caught.
    cfg = wl.custom_config(3, 8, 2, 64, torch.bfloat16, layers=2, history=("uniform", (1, 60)),
                           seed=9)
    w = wl.make_workload(cfg, device="cpu")
    out = torch.stack([bench.oracle_step(bench.oracle_sample(w, [0, 1, 2], layer), 1)
                       for layer in range(2)]).to(torch.bfloat16)
    par = bench.oracle_parity_all(w, out)
    assert par["ok"] and par["layers"] == 2 and par["sequences"] == 3
    assert par["max_abs_err"] <= 1e-2
    out[1, 2, 3, 4] += 0.5
    assert not bench.oracle_parity_all(w, out)["ok"]
