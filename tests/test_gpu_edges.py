"""Edge cases, variants and invariants of the CUDA path, against the oracle."""
import itertools

import pytest
import torch

import oracle
from paged_kv_cache_xs_gb300 import ops
from paged_kv_cache_xs_gb300 import workloads as wl
from paged_kv_cache_xs_gb300.step import PagedDecodeStep
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu


def _attend(w, layer, P, out=None, kc=None, vc=None, bt=None, err=None, dynamic=False,
            ws=None):
    cfg = w.cfg
    kc = w.k_cache[layer] if kc is None else kc
    vc = w.v_cache[layer] if vc is None else vc
    bt = w.block_tables if bt is None else bt
    ws = ws or ops.DecodeWorkspace(cfg.B, cfg.Hq, cfg.Hkv, cfg.D, bt.shape[1], kc.device,
                                   partition_tokens=P)
    out = torch.full((cfg.B, cfg.Hq, cfg.D), float("nan"), dtype=cfg.dtype, device=kc.device) \
        if out is None else out
    ops.xs_paged_decode(out, ws.part_o, ws.part_m, ws.part_l, w.q[layer], kc, vc, bt,
                        w.context_lens, w.scale, ws.partition_tokens, ws.max_partitions,
                        err_flag=err, work_counters=ws.work if dynamic else None)
    return out


def _oracle(w, layer, kc=None, vc=None):
    kc = w.k_cache[layer] if kc is None else kc
    vc = w.v_cache[layer] if vc is None else vc
    return oracle.paged_decode(w.q[layer].cpu(), kc.cpu(), vc.cpu(), w.block_tables.cpu(),
                               w.context_lens.cpu(), w.scale)


VARIANTS = list(itertools.product([torch.float32, torch.bfloat16], [64, 128], [1, 2, 4, 8]))


@pytest.mark.parametrize("dtype,D,G", VARIANTS,
                         ids=[f"{'f32' if d == torch.float32 else 'bf16'}-D{D}-G{G}"
                              for d, D, G in VARIANTS])
def test_variants_split_and_single(dtype, D, G):
    dev = gh.device()
    Hkv = 2
    cfg = wl.custom_config(5, Hkv * G, Hkv, D, dtype, history=("uniform", (0, 400)),
                           pool=("factor", 1.5), seed=100 + D + G)
    w = wl.make_workload(cfg, device=dev)
    ref = _oracle(w, 0)
    for P in (16, 48, 128, 512):
        for dynamic in (False, True):
            out = _attend(w, 0, P, dynamic=dynamic)
            torch.cuda.synchronize()
            gh.assert_close(out, ref, dtype, what=f"P={P} dynamic={dynamic}")


def test_dynamic_scheduler_counters_reset():
    # Several launches share one pair of work counters: each must see them at
    # zero (the previous launch's last CTA resets them) and produce the same,
    # correct output.
    dev = gh.device()
    cfg = wl.custom_config(23, 32, 8, 128, torch.bfloat16, history=("loguniform", (16, 6000)),
                           pool=("factor", 1.5), seed=121)
    w = wl.make_workload(cfg, device=dev)
    ref = _oracle(w, 0)
    ws = ops.DecodeWorkspace(cfg.B, cfg.Hq, cfg.Hkv, cfg.D, w.max_blocks_per_seq, dev,
                             partition_tokens=128)
    outs = []
    for _ in range(4):
        outs.append(_attend(w, 0, 128, dynamic=True, ws=ws))
    torch.cuda.synchronize()
    assert int(ws.work.count_nonzero()) == 0
    for out in outs:
        gh.assert_close(out, ref, torch.bfloat16)


def test_full_step_ragged_with_empty_sequences():
    dev = gh.device()
    cfg = wl.custom_config(7, 32, 8, 128, torch.bfloat16, history=("uniform", (0, 900)),
                           pool=("factor", 1.3), seed=31)
    hist = torch.tensor([0, 17, 255, 256, 257, 900, 31], dtype=torch.int32)
    w = wl.make_workload(cfg, device=dev, history=hist)
    step = PagedDecodeStep(cfg.B, cfg.Hq, cfg.Hkv, cfg.D, w.max_blocks_per_seq, cfg.dtype, dev,
                           partition_tokens=256)
    gh.check_step(w, 0, step, strict=False)
    # Sequences with nothing to attend to (context length 0) give zeros and write nothing.
    w.context_lens[2] = 0
    w.context_lens[5] = 0
    out = _attend(w, 0, 64)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out[2]).item() == 0 and torch.count_nonzero(out[5]).item() == 0
    gh.assert_close(out, _oracle(w, 0), torch.bfloat16)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_single_token_is_exact_v_row(dtype):
    # Context length 1: the one weight is exactly 1, so out = the new V row, bit for bit.
    dev = gh.device()
    cfg = wl.custom_config(6, 32, 8, 128, dtype, history=("fixed", (0,)), pool=("factor", 3.0),
                           seed=41)
    w = wl.make_workload(cfg, device=dev)
    step = PagedDecodeStep(cfg.B, cfg.Hq, cfg.Hkv, cfg.D, w.max_blocks_per_seq, dtype, dev,
                           partition_tokens=16)
    out = torch.empty(cfg.B, cfg.Hq, cfg.D, dtype=dtype, device=dev)
    step.run(out, w.q[0], w.k_new[0], w.v_new[0], w.k_cache[0], w.v_cache[0], w.block_tables,
             w.context_lens, w.scale)
    torch.cuda.synchronize()
    want = w.v_new[0].repeat_interleave(cfg.Hq // cfg.Hkv, dim=1)
    assert torch.equal(gh.int_view(out), gh.int_view(want))


def test_physical_permutation_is_bit_identical():
    dev = gh.device()
    cfg = wl.custom_config(6, 32, 8, 128, torch.bfloat16, history=("uniform", (1, 2000)),
                           pool=("factor", 2.0), seed=51)
    w = wl.make_workload(cfg, device=dev)
    a = _attend(w, 0, 128)
    g = torch.Generator().manual_seed(9)
    perm = torch.randperm(w.num_blocks, generator=g).to(dev)
    kc2 = torch.empty_like(w.k_cache[0])
    vc2 = torch.empty_like(w.v_cache[0])
    kc2[perm] = w.k_cache[0]
    vc2[perm] = w.v_cache[0]
    bt2 = w.block_tables.clone()
    used = bt2 >= 0
    bt2[used] = perm[bt2[used].long()].to(torch.int32)
    b = _attend(w, 0, 128, kc=kc2, vc=vc2, bt=bt2)
    torch.cuda.synchronize()
    assert torch.equal(gh.int_view(a), gh.int_view(b))
    gh.assert_close(a, _oracle(w, 0), torch.bfloat16)


def test_constant_v_gives_constant_output():
    dev = gh.device()
    cfg = wl.custom_config(4, 16, 4, 64, torch.bfloat16, history=("uniform", (1, 3000)),
                           pool=("factor", 1.2), seed=61)
    w = wl.make_workload(cfg, device=dev)
    c = torch.linspace(-2, 2, cfg.D, device=dev).to(torch.bfloat16)
    w.v_cache[0].copy_(c.expand_as(w.v_cache[0]))
    out = _attend(w, 0, 64)
    torch.cuda.synchronize()
    err = (out.float() - c.float()).abs().max().item()
    assert err <= 2 ** -8 * 2, err


def test_many_sequences_prefix_scan():
    # B well above the thread count exercises the chunked per-CTA prefix sum.
    dev = gh.device()
    cfg = wl.custom_config(3000, 32, 8, 128, torch.bfloat16, history=("uniform", (0, 60)),
                           pool=("factor", 1.1), seed=71)
    w = wl.make_workload(cfg, device=dev)
    step = PagedDecodeStep(cfg.B, cfg.Hq, cfg.Hkv, cfg.D, w.max_blocks_per_seq, cfg.dtype, dev,
                           partition_tokens=16)
    gh.check_step(w, 0, step, strict=False)


def test_one_long_sequence_many_partitions():
    dev = gh.device()
    cfg = wl.custom_config(1, 32, 8, 128, torch.bfloat16, history=("fixed", (32768,)),
                           pool=("needed", 1), seed=81)
    w = wl.make_workload(cfg, device=dev)
    for P in (16, 1024):
        step = PagedDecodeStep(1, 32, 8, 128, w.max_blocks_per_seq, cfg.dtype, dev,
                               partition_tokens=P)
        # re-draw the appended slot's pre-state each time: run append only once
        if P == 16:
            gh.check_step(w, 0, step, strict=False)
        else:
            out = _attend(w, 0, P)
            torch.cuda.synchronize()
            gh.assert_close(out, _oracle(w, 0), torch.bfloat16)


def test_side_stream():
    dev = gh.device()
    cfg = wl.custom_config(4, 32, 8, 128, torch.bfloat16, history=("uniform", (100, 1500)),
                           seed=91)
    w = wl.make_workload(cfg, device=dev)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        out = _attend(w, 0, 64)
    s.synchronize()
    gh.assert_close(out, _oracle(w, 0), torch.bfloat16)


def test_slot_mapping_matches_oracle():
    dev = gh.device()
    cfg = wl.custom_config(40, 8, 8, 64, torch.bfloat16, history=("uniform", (0, 100)),
                           pool=("factor", 2.0), seed=101)
    w = wl.make_workload(cfg, device=dev)
    lens = w.context_lens.clone()
    lens[3] = 0
    lens[7] = -5
    got = ops.xs_slot_mapping(w.block_tables, lens, 16, w.num_blocks)
    torch.cuda.synchronize()
    want = oracle.slot_mapping(w.block_tables.cpu(), lens.cpu(), 16, w.num_blocks)
    assert torch.equal(got.cpu(), want)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_append_slot_form_bit_exact(dtype):
    dev = gh.device()
    T, Hkv, D, nb = 37, 4, 128, 20
    g = torch.Generator().manual_seed(5)
    kc = torch.randn(nb, Hkv, 16, D, generator=g).to(dtype)
    vc = torch.randn(nb, Hkv, 16, D, generator=g).to(dtype)
    kn = torch.randn(T, Hkv, D, generator=g).to(dtype)
    vn = torch.randn(T, Hkv, D, generator=g).to(dtype)
    slots = torch.randperm(nb * 16, generator=g)[:T].to(torch.int64)
    slots[::5] = -1
    ek, ev = oracle.kv_append(kn, vn, kc, vc, slots)
    dkc, dvc = kc.to(dev), vc.to(dev)
    ops.xs_kv_append(kn.to(dev), vn.to(dev), dkc, dvc, slots.to(dev))
    torch.cuda.synchronize()
    assert torch.equal(gh.int_view(dkc.cpu()), gh.int_view(ek))
    assert torch.equal(gh.int_view(dvc.cpu()), gh.int_view(ev))


def test_device_errors_are_flagged_not_trapped():
    dev = gh.device()
    cfg = wl.custom_config(4, 32, 8, 128, torch.bfloat16, history=("uniform", (40, 300)),
                           pool=("factor", 1.5), seed=111)
    w = wl.make_workload(cfg, device=dev)
    ref = _oracle(w, 0)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    # (a) a block id past the pool in sequence 1: flagged, the other sequences unaffected.
    bt = w.block_tables.clone()
    bt[1, 0] = w.num_blocks + 5
    out = _attend(w, 0, 64, bt=bt, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & ops.FLAG_BAD_BLOCK
    keep = [0, 2, 3]
    gh.assert_close(out[keep], ref[keep], torch.bfloat16)
    # (b) a context length beyond the table: flagged and clamped.
    err.zero_()
    lens = w.context_lens.clone()
    w.context_lens[2] = w.max_blocks_per_seq * 16 + 40
    _attend(w, 0, 64, err=err)
    torch.cuda.synchronize()
    w.context_lens.copy_(lens)
    assert int(err.item()) & ops.FLAG_BAD_LEN
    # (c) an append slot past the pool: flagged, nothing written.
    err.zero_()
    before = w.k_cache[0].clone()
    slots = torch.tensor([w.num_blocks * 16 + 3, -1, -1, -1], dtype=torch.int64, device=dev)
    ops.xs_kv_append(w.k_new[0], w.v_new[0], w.k_cache[0], w.v_cache[0], slots, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & ops.FLAG_BAD_SLOT
    assert torch.equal(gh.int_view(before), gh.int_view(w.k_cache[0]))
