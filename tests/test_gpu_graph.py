"""A captured decode step (append + attention + reduce for several layers)
replayed over new inputs written into the same device buffers."""
import pytest
import torch

import oracle
from paged_kv_cache_xs_gb300 import workloads as wl
from paged_kv_cache_xs_gb300.step import CapturedStep, PagedDecodeStep
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu


def test_captured_step_replays_new_inputs():
    dev = gh.device()
    cfg = wl.custom_config(6, 32, 8, 128, torch.bfloat16, layers=3,
                           history=("uniform", (50, 3000)), pool=("factor", 1.5), seed=131)
    w = wl.make_workload(cfg, device=dev)
    step = PagedDecodeStep(cfg.B, cfg.Hq, cfg.Hkv, cfg.D, w.max_blocks_per_seq, cfg.dtype, dev,
                           total_context_tokens=w.total_context_tokens,
                           max_context_len=w.max_context_len)
    out = torch.empty(cfg.layers, cfg.B, cfg.Hq, cfg.D, dtype=cfg.dtype, device=dev)
    q = w.q.clone()      # the captured graph reads these buffers
    kn = w.k_new.clone()
    vn = w.v_new.clone()

    def one_step():
        for layer in range(cfg.layers):
            step.run(out[layer], q[layer], kn[layer], vn[layer], w.k_cache[layer],
                     w.v_cache[layer], w.block_tables, w.context_lens, w.scale)

    graph = CapturedStep(one_step)
    g = torch.Generator(device=dev).manual_seed(5)
    for trial in range(2):
        # New query and new rows for every replay; the pools keep the last append.
        q.copy_(torch.randn(q.shape, generator=g, device=dev).to(cfg.dtype))
        kn.copy_(torch.randn(kn.shape, generator=g, device=dev).to(cfg.dtype))
        vn.copy_(torch.randn(vn.shape, generator=g, device=dev).to(cfg.dtype))
        before_k = [w.k_cache[l].cpu() for l in range(cfg.layers)]
        before_v = [w.v_cache[l].cpu() for l in range(cfg.layers)]
        graph.replay()
        torch.cuda.synchronize()
        assert step.error_flags() == 0
        bt, cl = w.block_tables.cpu(), w.context_lens.cpu()
        slots = oracle.slot_mapping(bt, cl, 16, w.num_blocks)
        for layer in range(cfg.layers):
            ek, ev = oracle.kv_append(kn[layer].cpu(), vn[layer].cpu(), before_k[layer],
                                      before_v[layer], slots)
            assert torch.equal(gh.int_view(w.k_cache[layer].cpu()), gh.int_view(ek))
            ref = oracle.paged_decode(q[layer].cpu(), ek, ev, bt, cl, w.scale)
            gh.assert_close(out[layer], ref, cfg.dtype, strict=True,
                            what=f"replay {trial} layer {layer}")
