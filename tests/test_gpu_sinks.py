"""Sinks + sliding window (the gpt-oss variant) through the CUDA path, against
the oracle's paged_decode_sinks."""
import itertools

import pytest
import torch

import oracle
from paged_kv_cache_xs_gb300 import ops
from paged_kv_cache_xs_gb300 import workloads as wl
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu

CASES = list(itertools.product([torch.bfloat16, torch.float32], [1, 4], [0, 16, 37, 300]))


def _run(w, P, sinks, window, dynamic=True):
    cfg = w.cfg
    ws = ops.DecodeWorkspace(cfg.B, cfg.Hq, cfg.Hkv, cfg.D, w.max_blocks_per_seq, w.q.device,
                             partition_tokens=P)
    out = torch.full((cfg.B, cfg.Hq, cfg.D), float("nan"), dtype=cfg.dtype, device=w.q.device)
    err = torch.zeros(1, dtype=torch.int32, device=w.q.device)
    ops.xs_paged_decode_sinks(out, ws.part_o, ws.part_m, ws.part_l, w.q[0], w.k_cache[0],
                              w.v_cache[0], w.block_tables, w.context_lens, w.scale,
                              ws.partition_tokens, ws.max_partitions, sinks=sinks, window=window,
                              err_flag=err, work_counters=ws.work if dynamic else None)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return out


@pytest.mark.parametrize("dtype,G,window", CASES,
                         ids=[f"{'bf16' if d == torch.bfloat16 else 'f32'}-G{G}-W{W}"
                              for d, G, W in CASES])
def test_sinks_window_match_oracle(dtype, G, window):
    dev = gh.device()
    cfg = wl.custom_config(6, 8 * G, 8, 128, dtype, history=("uniform", (0, 1500)),
                           pool=("factor", 1.4), seed=150 + G + window)
    w = wl.make_workload(cfg, device=dev)
    g = torch.Generator(device=dev).manual_seed(window + G)
    sinks = (torch.randn(cfg.Hq, generator=g, device=dev) * 2).to(dtype)
    ref = oracle.paged_decode_sinks(w.q[0].cpu(), w.k_cache[0].cpu(), w.v_cache[0].cpu(),
                                    w.block_tables.cpu(), w.context_lens.cpu(), w.scale,
                                    sinks=sinks.cpu(), window=window)
    for P in (64, 256, 4096):   # many partitions, several, one
        out = _run(w, P, sinks, window)
        gh.assert_close(out, ref, dtype, what=f"P={P}")
    # Without sinks (window only), and the plain entry point when window == 0.
    ref_ns = oracle.paged_decode_sinks(w.q[0].cpu(), w.k_cache[0].cpu(), w.v_cache[0].cpu(),
                                       w.block_tables.cpu(), w.context_lens.cpu(), w.scale,
                                       window=window)
    gh.assert_close(_run(w, 128, None, window, dynamic=False), ref_ns, dtype, what="no sinks")


def test_window_one_is_the_last_v_row():
    # Window 1: only the newest token, whose weight is exactly 1 without a sink.
    dev = gh.device()
    cfg = wl.custom_config(5, 32, 8, 128, torch.bfloat16, history=("uniform", (3, 900)), seed=161)
    w = wl.make_workload(cfg, device=dev)
    out = _run(w, 64, None, 1)
    lens = w.context_lens.cpu()
    bs = cfg.block_size
    for b in range(cfg.B):
        p = int(lens[b]) - 1
        blk = int(w.block_tables[b, p // bs])
        want = w.v_cache[0][blk, :, p % bs].repeat_interleave(cfg.Hq // cfg.Hkv, dim=0)
        assert torch.equal(gh.int_view(out[b]), gh.int_view(want))
