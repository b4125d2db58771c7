"""Shared helpers for the GPU parity tests (CUDA path vs the CPU oracle)."""
from __future__ import annotations

import torch

import oracle
from paged_kv_cache_xs_gb300 import build as xsbuild
from paged_kv_cache_xs_gb300 import ops

BS = 16
# Attention tolerances (max-abs against the fp64 oracle).
TOL = {torch.float32: 1e-5, torch.bfloat16: 1e-2}


def device() -> torch.device:
    xsbuild.build()
    ops.load()
    return torch.device("cuda:0")


def int_view(t: torch.Tensor) -> torch.Tensor:
    return t.view(torch.int16 if t.element_size() == 2 else torch.int32)


def compact_pages(block_tables, context_lens, seqs, k_pool, v_pool):
    """CPU copies of the pages the sequences `seqs` read, renumbered 0..n-1,
    with a matching block table.  (The oracle's output does not depend on
    where pages sit, which its permutation pin checks.)"""
    bt = block_tables[seqs].cpu()
    lens = context_lens[seqs].cpu()
    ids, rows = [], []
    for i in range(len(seqs)):
        n = max(int(lens[i]), 0)
        p = (n + BS - 1) // BS
        rows.append(list(range(len(ids), len(ids) + p)))
        ids.extend(bt[i, :p].tolist())
    width = max([1] + [len(r) for r in rows])
    new_bt = torch.full((len(seqs), width), -1, dtype=torch.int32)
    for i, r in enumerate(rows):
        if r:
            new_bt[i, :len(r)] = torch.tensor(r, dtype=torch.int32)
    idx = torch.tensor(ids, dtype=torch.long, device=k_pool.device)
    return k_pool.index_select(0, idx).cpu(), v_pool.index_select(0, idx).cpu(), new_bt, lens


def changed_rows(before: torch.Tensor, after: torch.Tensor) -> set:
    """(block, head, offset) of every pool row whose bytes differ."""
    diff = (int_view(before) != int_view(after)).any(dim=-1)
    return {tuple(x) for x in diff.nonzero().tolist()}


def expected_rows(block_tables, context_lens, num_blocks, Hkv) -> set:
    slots = oracle.slot_mapping(block_tables.cpu(), context_lens.cpu(), BS, num_blocks)
    return {(s // BS, h, s % BS) for s in slots.tolist() if s >= 0 for h in range(Hkv)}


def bf16_floor(ref: torch.Tensor) -> torch.Tensor:
    """Error a correct bf16 result can carry whatever the arithmetic's care:
    half an ulp of the bf16 output at |ref| (its own rounding) plus 2^-9 |ref|
    (the softmax weights enter P V on the tensor cores rounded to bf16, a
    relative error of at most 2^-9 each).  Below |ref| = 2 this is under
    1e-2."""
    _, e = torch.frexp(ref.abs())            # |ref| = m 2^e, m in [0.5, 1)
    half_ulp = torch.ldexp(torch.ones_like(ref), (e - 9).to(torch.int32))
    half_ulp = torch.where(ref == 0, torch.zeros_like(ref), half_ulp)
    return half_ulp + ref.abs() * 2.0 ** -9


def assert_close(out: torch.Tensor, ref: torch.Tensor, dtype, strict: bool = False,
                 what: str = "") -> float:
    """Attention parity.  The stated bounds are max-abs 1e-5 (fp32) and 1e-2
    (bf16).  A bf16 output of magnitude |o| >= 2 can carry more than 1e-2 of
    error that no arithmetic avoids (bf16_floor: its own rounding plus the
    bf16 softmax weights); edge tests whose outputs get that large (very short
    contexts) take the larger of 1e-2 and that floor (strict=False), which is
    exactly 1e-2 below |o| = 2.  The five workloads use the flat bound."""
    d = (out.detach().cpu().double() - ref).abs()
    bound = torch.full_like(ref, TOL[dtype])
    if dtype == torch.bfloat16 and not strict:
        bound = torch.maximum(bound, bf16_floor(ref))
    worst = (d - bound).max().item() if d.numel() else -1.0
    assert worst <= 0, f"{what}: max-abs {d.max().item():.3e} exceeds the bound by {worst:.3e}"
    return d.max().item() if d.numel() else 0.0


def max_abs(out: torch.Tensor, ref: torch.Tensor) -> float:
    if out.numel() == 0:
        return 0.0
    return (out.detach().cpu().double() - ref).abs().max().item()


def check_step(w, layer, step, seqs=None, check_unchanged=True, strict=True, fused=True,
               repeat=1, early_reads=False):
    """Run one decode step (append + attention) of layer `layer` through the
    CUDA path - as one fused launch, or as the three separate calls - and
    compare it with the oracle on the sequences `seqs`.  `repeat` launches
    the same step back to back (each appends the same rows again), with
    early reads if asked, as the benchmark loop does.  Returns the attention
    max-abs error of the last launch."""
    cfg = w.cfg
    seqs = list(range(cfg.B)) if seqs is None else list(seqs)
    kc, vc = w.k_cache[layer], w.v_cache[layer]
    kb, vb, bt_c, lens_c = compact_pages(w.block_tables, w.context_lens, seqs, kc, vc)
    before_k = kc.clone() if check_unchanged else None
    before_v = vc.clone() if check_unchanged else None
    out = torch.empty(cfg.B, cfg.Hq, cfg.D, dtype=cfg.dtype, device=kc.device)
    step.err_flag.zero_()
    for _ in range(repeat):
        if fused:
            step.run(out, w.q[layer], w.k_new[layer], w.v_new[layer], kc, vc, w.block_tables,
                     w.context_lens, w.scale, early_reads=early_reads)
        else:
            step.run_unfused(out, w.q[layer], w.k_new[layer], w.v_new[layer], kc, vc,
                             w.block_tables, w.context_lens, w.scale)
    torch.cuda.synchronize()
    assert step.error_flags() == 0, f"device error flag {step.error_flags()}"
    assert int(step.ws.work.count_nonzero()) == 0, "counters not left at zero"

    # Append: bit-exact against the oracle's append of the same pre-state.
    sel = torch.tensor(seqs, dtype=torch.long, device=kc.device)
    kn = w.k_new[layer].index_select(0, sel).cpu()
    vn = w.v_new[layer].index_select(0, sel).cpu()
    slots = oracle.slot_mapping(bt_c, lens_c, BS, kb.shape[0])
    ek, ev = oracle.kv_append(kn, vn, kb, vb, slots)
    ka, va, _, _ = compact_pages(w.block_tables, w.context_lens, seqs, kc, vc)
    assert torch.equal(int_view(ka), int_view(ek)), "K pages differ from the oracle append"
    assert torch.equal(int_view(va), int_view(ev)), "V pages differ from the oracle append"
    if check_unchanged:
        want = expected_rows(w.block_tables, w.context_lens, w.num_blocks, cfg.Hkv)
        assert changed_rows(before_k, kc) <= want, "append wrote outside the new slots"
        assert changed_rows(before_v, vc) <= want, "append wrote outside the new slots"
        del before_k, before_v

    # Attention over the appended cache.
    q = w.q[layer].index_select(0, sel).cpu()
    ref = oracle.paged_decode(q, ek, ev, bt_c, lens_c, w.scale)
    return assert_close(out.index_select(0, sel), ref, cfg.dtype, strict,
                        f"{cfg.name} layer {layer}")
