"""The one-launch decode step (xs_paged_decode_step: append + attention +
split-K combine) against the oracle: ragged splits with more partitions than
a warp has lanes, sinks and windows, lengths beyond the table, bad block ids,
attention-only launches, and counters that stay zero across launches."""
import itertools

import pytest
import torch

import oracle
from paged_kv_cache_xs_gb300 import ops
from paged_kv_cache_xs_gb300 import workloads as wl
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu


def _ws(w, P):
    cfg = w.cfg
    return ops.DecodeWorkspace(cfg.B, cfg.Hq, cfg.Hkv, cfg.D, w.max_blocks_per_seq, w.q.device,
                               partition_tokens=P)


def _step(w, ws, sinks=None, window=0, append=True, out=None, err=None, early=False, layer=0,
          persistent=False):
    cfg = w.cfg
    dev = w.q.device
    out = torch.full((cfg.B, cfg.Hq, cfg.D), float("nan"), dtype=cfg.dtype, device=dev) \
        if out is None else out
    err = torch.zeros(1, dtype=torch.int32, device=dev) if err is None else err
    ops.xs_paged_decode_step(out, w.q[layer], w.k_new[layer] if append else None,
                             w.v_new[layer] if append else None, w.k_cache[layer],
                             w.v_cache[layer], w.block_tables, w.context_lens, w.scale,
                             ws.partition_tokens, ws.max_partitions, ws.part_o, ws.part_m,
                             ws.part_l, ws.work, sinks=sinks, window=window, err_flag=err,
                             early_reads=early, persistent=persistent)
    return out, err


def _appended(w, layer=0):
    """The oracle's append of this step's rows into copies of the pools."""
    slots = oracle.slot_mapping(w.block_tables.cpu(), w.context_lens.cpu(), gh.BS, w.num_blocks)
    return oracle.kv_append(w.k_new[layer].cpu(), w.v_new[layer].cpu(), w.k_cache[layer].cpu(),
                            w.v_cache[layer].cpu(), slots)


CASES = [(d, G, P, False) for d, G, P in
         itertools.product([torch.bfloat16, torch.float32], [1, 4, 8], [16, 64, 4096])]
CASES += [(torch.bfloat16, 4, 16, True), (torch.bfloat16, 8, 64, True), (torch.float32, 1, 64, True)]
# Partition lengths the step heuristic picks that are not powers of two.
CASES += [(torch.bfloat16, 4, 448, False), (torch.bfloat16, 4, 640, True),
          (torch.float32, 1, 192, False)]


# The bf16 cases again on the persistent grid (these small batches would run
# as clusters).
CASES = [c + (False,) for c in CASES] + [c + (True,) for c in CASES if c[0] == torch.bfloat16]


@pytest.mark.parametrize("dtype,G,P,early,persistent", CASES,
                         ids=[f"{'bf16' if d == torch.bfloat16 else 'f32'}-G{G}-P{P}"
                              f"{'-early' if e else ''}{'-persistent' if pe else ''}"
                              for d, G, P, e, pe in CASES])
def test_step_matches_oracle(dtype, G, P, early, persistent):
    # Lengths around page and partition edges, up to 63 partitions of 16
    # tokens (the combine walks its partials 32 at a time), and an empty slot.
    dev = gh.device()
    hist = torch.tensor([0, 14, 15, 16, 510, 511, 512, 1000, -1], dtype=torch.int32)
    cfg = wl.custom_config(len(hist), 2 * G, 2, 128, dtype, history=("uniform", (0, 1)),
                           pool=("factor", 1.5), seed=700 + G + P)
    w = wl.make_workload(cfg, device=dev, history=hist)
    ek, ev = _appended(w)
    ws = _ws(w, P)
    out, err = _step(w, ws, early=early, persistent=persistent)
    torch.cuda.synchronize()
    assert int(err.item()) == 0 and int(ws.work.count_nonzero()) == 0
    assert torch.equal(gh.int_view(w.k_cache[0].cpu()), gh.int_view(ek))
    assert torch.equal(gh.int_view(w.v_cache[0].cpu()), gh.int_view(ev))
    ref = oracle.paged_decode(w.q[0].cpu(), ek, ev, w.block_tables.cpu(), w.context_lens.cpu(),
                              w.scale)
    gh.assert_close(out, ref, dtype, what=f"P={P}")


@pytest.mark.parametrize("window", [0, 16, 37, 300])
def test_step_sinks_window(window):
    dev = gh.device()
    cfg = wl.custom_config(6, 32, 8, 128, torch.bfloat16, history=("uniform", (0, 1500)),
                           pool=("factor", 1.4), seed=750 + window)
    w = wl.make_workload(cfg, device=dev)
    g = torch.Generator(device=dev).manual_seed(window)
    sinks = (torch.randn(cfg.Hq, generator=g, device=dev) * 2).to(cfg.dtype)
    ek, ev = _appended(w)
    ref = oracle.paged_decode_sinks(w.q[0].cpu(), ek, ev, w.block_tables.cpu(),
                                    w.context_lens.cpu(), w.scale, sinks=sinks.cpu(),
                                    window=window)
    for P, persistent in itertools.product((64, 256, 4096), (False, True)):
        out, err = _step(w, _ws(w, P), sinks=sinks, window=window, persistent=persistent)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        gh.assert_close(out, ref, cfg.dtype, what=f"P={P} persistent={persistent}")


def test_attention_only_launch():
    # k_new = v_new = NULL: the pools are read, never written.
    dev = gh.device()
    cfg = wl.custom_config(9, 32, 8, 128, torch.bfloat16, history=("loguniform", (1, 3000)),
                           pool=("factor", 1.3), seed=761)
    w = wl.make_workload(cfg, device=dev)
    kc0, vc0 = w.k_cache[0].clone(), w.v_cache[0].clone()
    out, err = _step(w, _ws(w, 64), append=False)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(gh.int_view(kc0), gh.int_view(w.k_cache[0]))
    assert torch.equal(gh.int_view(vc0), gh.int_view(w.v_cache[0]))
    ref = oracle.paged_decode(w.q[0].cpu(), kc0.cpu(), vc0.cpu(), w.block_tables.cpu(),
                              w.context_lens.cpu(), w.scale)
    gh.assert_close(out, ref, torch.bfloat16)


def test_bad_length_and_bad_block_append_nothing():
    # Sequence 1's length runs past its table (XS_FLAG_BAD_LEN); sequence 3's
    # last page has an out-of-pool id (XS_FLAG_BAD_BLOCK).  Neither writes a
    # row; every other sequence appends as usual.  The attention of the
    # clamped sequence equals the three-launch path's.
    dev = gh.device()
    cfg = wl.custom_config(6, 32, 8, 128, torch.bfloat16, history=("uniform", (40, 600)),
                           pool=("factor", 1.3), seed=771)
    w = wl.make_workload(cfg, device=dev)
    cap = w.max_blocks_per_seq * gh.BS
    w.context_lens[1] = cap + 5
    n3 = int(w.context_lens[3])
    w.block_tables[3, (n3 - 1) // gh.BS] = w.num_blocks + 7
    lens_ok = w.context_lens.clone()
    lens_ok[1] = 0
    lens_ok[3] = 0
    want = gh.expected_rows(w.block_tables, lens_ok, w.num_blocks, cfg.Hkv)
    kc0, vc0 = w.k_cache[0].clone(), w.v_cache[0].clone()
    ws = _ws(w, 64)
    out, err = _step(w, ws, persistent=True)
    torch.cuda.synchronize()
    flags = int(err.item())
    assert flags & ops.FLAG_BAD_LEN and flags & ops.FLAG_BAD_BLOCK
    assert gh.changed_rows(kc0, w.k_cache[0]) == want
    assert gh.changed_rows(vc0, w.v_cache[0]) == want
    assert int(ws.work.count_nonzero()) == 0
    # The same launch through the separate calls, on the same (appended) pools.
    ref_out = torch.empty_like(out)
    ops.xs_paged_decode(ref_out, ws.part_o, ws.part_m, ws.part_l, w.q[0], w.k_cache[0],
                        w.v_cache[0], w.block_tables, w.context_lens, w.scale,
                        ws.partition_tokens, ws.max_partitions, err_flag=err)
    torch.cuda.synchronize()
    for b in (0, 1, 2, 4, 5):
        torch.testing.assert_close(out[b].float(), ref_out[b].float(), atol=1e-2, rtol=0)


def test_counters_zero_across_many_launches():
    # One workspace, eight launches in a row (as the layers of one step would
    # use it): each sees zeroed counters and produces the same output.
    dev = gh.device()
    cfg = wl.custom_config(31, 32, 8, 128, torch.bfloat16, history=("loguniform", (16, 9000)),
                           pool=("factor", 1.3), seed=781)
    w = wl.make_workload(cfg, device=dev)
    ek, ev = _appended(w)
    ref = oracle.paged_decode(w.q[0].cpu(), ek, ev, w.block_tables.cpu(), w.context_lens.cpu(),
                              w.scale)
    ws = _ws(w, 128)
    outs = [_step(w, ws)[0] for _ in range(8)]
    torch.cuda.synchronize()
    assert int(ws.work.count_nonzero()) == 0
    for out in outs:
        gh.assert_close(out, ref, torch.bfloat16)


@pytest.mark.parametrize("P", [16, 128])
def test_early_reads_layers_back_to_back(P):
    # Layers launched back to back with early reads: each launch reads its
    # lengths, tables and first pages while the previous layer's launch may
    # still run (it writes other pools), and sequences shorter than a ring
    # put the page that receives the new row in the first item.  Every layer
    # matches the oracle, and a second pass over the same pools (the previous
    # launch then appends the same rows) gives the same outputs.
    dev = gh.device()
    hist = torch.tensor([0, 3, 15, 16, 40, 127, 128, 129, 700, 2000, -1], dtype=torch.int32)
    L = 4
    cfg = wl.custom_config(len(hist), 32, 8, 128, torch.bfloat16, layers=L,
                           history=("uniform", (0, 1)), pool=("factor", 1.5), seed=790 + P)
    w = wl.make_workload(cfg, device=dev, history=hist)
    refs = []
    for layer in range(L):
        ek, ev = _appended(w, layer)
        refs.append(oracle.paged_decode(w.q[layer].cpu(), ek, ev, w.block_tables.cpu(),
                                        w.context_lens.cpu(), w.scale))
    ws = _ws(w, P)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    outs = [[_step(w, ws, err=err, early=True, layer=layer)[0] for layer in range(L)]
            for _ in range(2)]
    torch.cuda.synchronize()
    assert int(err.item()) == 0 and int(ws.work.count_nonzero()) == 0
    for rep in outs:
        for layer in range(L):
            gh.assert_close(rep[layer], refs[layer], torch.bfloat16, what=f"layer {layer}")



def test_early_reads_in_a_cuda_graph():
    # The same back-to-back layers captured in one CUDA graph (the launches
    # keep their programmatic dependencies), replayed three times.
    from paged_kv_cache_xs_gb300.step import CapturedStep
    dev = gh.device()
    L = 3
    cfg = wl.custom_config(7, 32, 8, 128, torch.bfloat16, layers=L,
                           history=("loguniform", (1, 3000)), pool=("factor", 1.4), seed=811)
    w = wl.make_workload(cfg, device=dev)
    refs = []
    for layer in range(L):
        ek, ev = _appended(w, layer)
        refs.append(oracle.paged_decode(w.q[layer].cpu(), ek, ev, w.block_tables.cpu(),
                                        w.context_lens.cpu(), w.scale))
    ws = _ws(w, 64)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    outs = [torch.full((cfg.B, cfg.Hq, cfg.D), float("nan"), dtype=cfg.dtype, device=dev)
            for _ in range(L)]
    g = CapturedStep(lambda: [_step(w, ws, err=err, early=True, layer=layer, out=outs[layer])
                              for layer in range(L)])
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert int(err.item()) == 0 and int(ws.work.count_nonzero()) == 0
    for layer in range(L):
        gh.assert_close(outs[layer], refs[layer], torch.bfloat16, what=f"layer {layer}")


@pytest.mark.parametrize("num_splits", [1, 3, 8])
def test_num_splits_form_matches_oracle(num_splits):
    # xs_paged_decode_attn_splits + xs_paged_decode_reduce_splits: the split
    # as a count for the whole batch, partials sized for num_splits.
    dev = gh.device()
    cfg = wl.custom_config(7, 32, 8, 128, torch.bfloat16, history=("loguniform", (1, 3000)),
                           pool=("factor", 1.3), seed=990 + num_splits)
    w = wl.make_workload(cfg, device=dev)
    B, Hq, D = cfg.B, cfg.Hq, cfg.D
    part_o = torch.empty(B, Hq, num_splits, D, dtype=torch.float32, device=dev)
    part_m = torch.empty(B, Hq, num_splits, dtype=torch.float32, device=dev)
    part_l = torch.empty(B, Hq, num_splits, dtype=torch.float32, device=dev)
    out = torch.full((B, Hq, D), float("nan"), dtype=cfg.dtype, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    ops.xs_paged_decode_splits(out, part_o, part_m, part_l, w.q[0], w.k_cache[0], w.v_cache[0],
                               w.block_tables, w.context_lens, w.scale, num_splits, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = oracle.paged_decode(w.q[0].cpu(), w.k_cache[0].cpu(), w.v_cache[0].cpu(),
                              w.block_tables.cpu(), w.context_lens.cpu(), w.scale)
    gh.assert_close(out, ref, cfg.dtype, what=f"num_splits={num_splits}")
