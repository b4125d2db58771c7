"""xs_paged_decode_noalloc: the decode entry point for callers that may not
allocate device memory (an engine that has handed all free memory to its own
pools, a plugin whose host owns every allocation, a loop that must not risk
the device-wide synchronisation or the failure of cudaMalloc/cudaFree).  Its
split-K partials live in the library's fixed device array instead of a
caller-provided workspace.

The GPU test calls it through the C ABI several times in a row, on different
batches (two with a given partition length, one where the library picks it),
and checks each output element by element against the fp64 CPU oracle within
the bf16 tolerance of the other decode tests, and against the allocating
entry point (xs_paged_decode with a PyTorch-allocated workspace).  This file
is named so pytest collects it last."""
import pytest
import torch

import oracle
from paged_kv_cache_xs_gb300 import build as xsbuild
from paged_kv_cache_xs_gb300 import ops
from paged_kv_cache_xs_gb300 import workloads as wl

TOL_BF16 = 1e-2


def _allocating(w, P):
    cfg = w.cfg
    ws = ops.DecodeWorkspace(cfg.B, cfg.Hq, cfg.Hkv, cfg.D, w.max_blocks_per_seq,
                             w.q.device, partition_tokens=P)
    out = torch.empty(cfg.B, cfg.Hq, cfg.D, dtype=cfg.dtype, device=w.q.device)
    ops.xs_paged_decode(out, ws.part_o, ws.part_m, ws.part_l, w.q[0], w.k_cache[0],
                        w.v_cache[0], w.block_tables, w.context_lens, w.scale,
                        ws.partition_tokens, ws.max_partitions)
    return out


def _oracle(w):
    return oracle.paged_decode(w.q[0].cpu(), w.k_cache[0].cpu(), w.v_cache[0].cpu(),
                               w.block_tables.cpu(), w.context_lens.cpu(), w.scale)


@pytest.mark.gpu
def test_noalloc_matches_oracle_and_allocating_entry_point_on_calls_in_a_row():
    xsbuild.build()
    lib = ops.load()
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    # (workload, partition_tokens); 0 lets the library pick the partition length.
    cases = [
        (wl.custom_config(6, 32, 8, 128, torch.bfloat16, history=("uniform", (100, 5000)),
                          pool=("factor", 1.5), seed=301), 256),
        (wl.custom_config(9, 32, 8, 128, torch.bfloat16, history=("uniform", (1, 2500)),
                          pool=("factor", 1.2), seed=302), 128),
        (wl.custom_config(5, 32, 8, 128, torch.bfloat16, history=("uniform", (1, 9000)),
                          pool=("factor", 1.3), seed=303), 0),
    ]
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    for cfg, P in cases:
        w = wl.make_workload(cfg, device=dev)
        got = torch.full((cfg.B, cfg.Hq, cfg.D), float("nan"), dtype=cfg.dtype, device=dev)
        # Straight through the C ABI, checking the status it returns.
        status = lib.xs_paged_decode_noalloc(
            got.data_ptr(), w.q[0].data_ptr(), w.k_cache[0].data_ptr(), w.v_cache[0].data_ptr(),
            w.block_tables.data_ptr(), w.max_blocks_per_seq, w.context_lens.data_ptr(), cfg.B,
            cfg.Hq, cfg.Hkv, cfg.D, cfg.block_size, w.num_blocks, w.scale, P, ops.XS_BF16,
            err.data_ptr(), stream)
        assert status == 0, f"xs_paged_decode_noalloc returned {ops.STATUS.get(status, status)}"
        torch.cuda.synchronize()
        assert int(err.item()) == 0, f"device error flag {int(err.item())}"
        ref = _oracle(w)
        d_oracle = (got.cpu().double() - ref).abs().max().item()
        assert d_oracle <= TOL_BF16, f"B={cfg.B} P={P}: max-abs {d_oracle:.3e} vs the oracle"
        if P:
            want = _allocating(w, P)
            torch.cuda.synchronize()
            d_alloc = (got.float() - want.float()).abs().max().item()
            assert d_alloc <= TOL_BF16, f"B={cfg.B} P={P}: max-abs {d_alloc:.3e} vs xs_paged_decode"


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
