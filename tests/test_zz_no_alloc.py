"""xs_paged_decode_noalloc: the decode entry point for callers that may not
allocate device memory (an engine that has handed all free memory to its own
pools, a plugin whose host owns every allocation, a loop that must not risk
the device-wide synchronisation or the failure of cudaMalloc/cudaFree).  Its
split-K partials live in the library's fixed device array instead of a
caller-provided workspace.

The GPU test calls it through the C ABI twice in a row, on different
batches, and checks each output against the allocating entry point
(xs_paged_decode with a PyTorch-allocated workspace) within the bf16
tolerance the other tests use.  This file is named so pytest collects it
last."""
import pytest
import torch

from paged_kv_cache_xs_gb300 import build as xsbuild
from paged_kv_cache_xs_gb300 import ops
from paged_kv_cache_xs_gb300 import workloads as wl


def _reference(w, P):
    cfg = w.cfg
    ws = ops.DecodeWorkspace(cfg.B, cfg.Hq, cfg.Hkv, cfg.D, w.max_blocks_per_seq,
                             w.q.device, partition_tokens=P)
    out = torch.empty(cfg.B, cfg.Hq, cfg.D, dtype=cfg.dtype, device=w.q.device)
    ops.xs_paged_decode(out, ws.part_o, ws.part_m, ws.part_l, w.q[0], w.k_cache[0],
                        w.v_cache[0], w.block_tables, w.context_lens, w.scale,
                        ws.partition_tokens, ws.max_partitions)
    return out


@pytest.mark.gpu
def test_noalloc_matches_allocating_entry_point_on_two_calls():
    xsbuild.build()
    ops.load()
    dev = torch.device("cuda:0")
    cases = [
        (wl.custom_config(6, 32, 8, 128, torch.bfloat16, history=("uniform", (100, 5000)),
                          pool=("factor", 1.5), seed=301), 256),
        (wl.custom_config(9, 32, 8, 128, torch.bfloat16, history=("uniform", (1, 2500)),
                          pool=("factor", 1.2), seed=302), 128),
    ]
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    for cfg, P in cases:
        w = wl.make_workload(cfg, device=dev)
        want = _reference(w, P)
        got = torch.full_like(want, float("nan"))
        ops.xs_paged_decode_noalloc(got, w.q[0], w.k_cache[0], w.v_cache[0], w.block_tables,
                                    w.context_lens, w.scale, partition_tokens=P, err_flag=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        diff = (got.float() - want.float()).abs().max().item()
        assert diff <= 1e-2, f"B={cfg.B} P={P}: max-abs {diff:.3e}"


def test_noalloc_rejects_a_split_larger_than_its_array():
    # 4096 sequences x 64 heads x 2049 partitions of 16 tokens needs far more
    # than 64 MiB of partials: refused on the host before any device work.
    xsbuild.build()
    lib = ops.load()
    A = 1 << 20
    code = lib.xs_paged_decode_noalloc(A, A, A, A, A, 2049, A, 4096, 64, 8, 128, 16, 10, 0.1,
                                       16, ops.XS_BF16, None, None)
    assert code == -9
    need = ops.xs_paged_decode_workspace_bytes(4096, 64, 128, 2049)
    assert need > ops.NOALLOC_SCRATCH_BYTES
