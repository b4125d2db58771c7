"""Pins that tie the CPU oracle to something other than itself.

Each ``pin_*`` takes a loaded oracle library (the real one, or a deliberately
broken copy built by test_oracle_mutants.py) and raises AssertionError if the
oracle disagrees with:

* hand-derived closed forms (tests/golden/hand_worked_cases.txt);
* an independent dense formulation: pages gathered to a contiguous copy with
  tensor indexing, K/V repeated over the GQA group (the repeat_kv equivalence
  of "xserv compare phase8...phase13", qwen3.rs), then torch.softmax and
  matmul in float64;
* brute force in pure Python on tiny inputs;
* invariants: physical-block permutation, constant V, zero query, one
  dominant key, linearity in V, exact bf16 widening, and the pages' own
  "cache == recompute" invariant ("xserv compare phase5...phase9",
  docs/benchmarks/phase9-kv-cache.md, Correctness table).
"""
from __future__ import annotations

import math
import random

import torch

import oracle
from paged_kv_cache_xs_gb300 import workloads as wl
from tests import golden_cases as gc

TOL = 1e-12


def _close(a: torch.Tensor, b: torch.Tensor, tol: float = TOL, what: str = "") -> None:
    a = a.to(torch.float64)
    b = b.to(torch.float64)
    assert a.shape == b.shape, f"{what}: shape {tuple(a.shape)} vs {tuple(b.shape)}"
    assert torch.isfinite(a).all(), f"{what}: non-finite oracle output"
    err = (a - b).abs().max().item() if a.numel() else 0.0
    assert err <= tol, f"{what}: max-abs error {err:.3e} > {tol:.1e}"


def _layer(w: wl.DecodeWorkload, layer: int = 0):
    return (w.q[layer], w.k_cache[layer], w.v_cache[layer], w.k_new[layer], w.v_new[layer])


def dense_reference(q, k_cache, v_cache, block_tables, context_lens, scale) -> torch.Tensor:
    """softmax(scale * q K^T) V per sequence on a contiguous float64 copy."""
    B, Hq, D = q.shape
    _, Hkv, bs, _ = k_cache.shape
    rep = Hq // Hkv
    out = torch.zeros(B, Hq, D, dtype=torch.float64)
    for b in range(B):
        n = int(context_lens[b])
        if n <= 0:
            continue
        pages = block_tables[b, : (n + bs - 1) // bs].long()
        K = k_cache[pages].to(torch.float64).permute(0, 2, 1, 3).reshape(-1, Hkv, D)[:n]
        V = v_cache[pages].to(torch.float64).permute(0, 2, 1, 3).reshape(-1, Hkv, D)[:n]
        K = K.transpose(0, 1).repeat_interleave(rep, dim=0)      # [Hq, n, D]
        V = V.transpose(0, 1).repeat_interleave(rep, dim=0)
        logits = torch.matmul(q[b].to(torch.float64).unsqueeze(1), K.transpose(1, 2)) * scale
        out[b] = torch.matmul(torch.softmax(logits, dim=-1), V).squeeze(1)
    return out


# ----------------------------------------------------------------- closed forms

def pin_slots_by_hand(lib):
    c = gc.load_cases()["slots_by_hand"]
    got = oracle.slot_mapping(torch.tensor(c["block_tables"]), torch.tensor(c["context_lens"]),
                              c["block_size"], c["num_blocks"], lib=lib)
    assert got.tolist() == c["expected_slots"], f"slots {got.tolist()}"


def _golden_attention(lib, name):
    c = gc.load_cases()[name]
    q = torch.tensor(c["q"], dtype=torch.float32)
    kc, vc = gc.pool_tensor(c, "k_cache"), gc.pool_tensor(c, "v_cache")
    out = oracle.paged_decode(q, kc, vc, torch.tensor(c["block_tables"]),
                              torch.tensor(c["context_lens"]), gc.scale_of(c), lib=lib)
    _close(out, gc.expected_of(c), 1e-14, name)


def pin_gqa_paged_by_hand(lib):
    _golden_attention(lib, "gqa_paged_by_hand")


def pin_single_token(lib):
    _golden_attention(lib, "single_token_is_v_row")


# ------------------------------------------------------- independent formulation

def _small_workloads():
    yield wl.make_workload(0)                                   # fp32 MHA, 8-block pool
    yield wl.make_workload(wl.custom_config(3, 8, 2, 16, torch.bfloat16, history=("uniform", (0, 70)),
                                            pool=("factor", 2.0), seed=11))
    yield wl.make_workload(wl.custom_config(4, 6, 3, 8, torch.float32, history=("uniform", (0, 40)),
                                            pool=("factor", 1.0), values="uniform", seed=12))


def pin_dense_equivalence(lib):
    for w in _small_workloads():
        q, kc, vc, _, _ = _layer(w)
        got = oracle.paged_decode(q, kc, vc, w.block_tables, w.context_lens, w.scale, lib=lib)
        ref = dense_reference(q, kc, vc, w.block_tables, w.context_lens, w.scale)
        _close(got, ref, TOL, f"dense {w.cfg.name}")


def pin_brute_force_python(lib):
    rng = random.Random(5)
    for trial in range(6):
        B = rng.randint(1, 3)
        Hkv = rng.choice([1, 2])
        Hq = Hkv * rng.choice([1, 2])
        D = rng.choice([4, 8])
        bs = rng.choice([2, 4, 16])
        lens = [rng.randint(1, 40) for _ in range(B)]
        pages = [(n + bs - 1) // bs for n in lens]
        nblk = sum(pages) + 2
        perm = list(range(nblk))
        rng.shuffle(perm)
        table, pos = [], 0
        for p in pages:
            table.append(perm[pos:pos + p] + [-1] * (max(pages) - p))
            pos += p
        # Store K/V as a dict keyed by (block, head, offset) in pure Python.
        kd = {(blk, h, o): [rng.uniform(-2, 2) for _ in range(D)]
              for blk in range(nblk) for h in range(Hkv) for o in range(bs)}
        vd = {key: [rng.uniform(-2, 2) for _ in range(D)] for key in kd}
        qv = [[[rng.uniform(-2, 2) for _ in range(D)] for _ in range(Hq)] for _ in range(B)]
        scale = 1.0 / math.sqrt(D)
        kc = torch.zeros(nblk, Hkv, bs, D, dtype=torch.float32)
        vc = torch.zeros_like(kc)
        for (blk, h, o), row in kd.items():
            kc[blk, h, o] = torch.tensor(row)
        for (blk, h, o), row in vd.items():
            vc[blk, h, o] = torch.tensor(row)
        # The Python side used the same fp32-rounded values the oracle sees.
        for key in kd:
            kd[key] = kc[key].double().tolist()
            vd[key] = vc[key].double().tolist()
        q = torch.tensor(qv, dtype=torch.float32)
        qv = q.double().tolist()
        expect = []
        for b in range(B):
            rows = []
            for h in range(Hq):
                g = h // (Hq // Hkv)
                keys = [(table[b][t // bs], g, t % bs) for t in range(lens[b])]
                logits = [scale * sum(a * c for a, c in zip(qv[b][h], kd[key])) for key in keys]
                top = max(logits)
                ws = [math.exp(x - top) for x in logits]
                tot = math.fsum(ws)
                rows.append([math.fsum(w * vd[key][d] for w, key in zip(ws, keys)) / tot
                             for d in range(D)])
            expect.append(rows)
        got = oracle.paged_decode(q, kc, vc, torch.tensor(table, dtype=torch.int32),
                                  torch.tensor(lens, dtype=torch.int32), scale, lib=lib)
        _close(got, torch.tensor(expect, dtype=torch.float64), TOL, f"brute force trial {trial}")


# ------------------------------------------------------------------- invariants

def pin_permutation_invariance(lib):
    w = wl.make_workload(wl.custom_config(3, 8, 4, 32, torch.bfloat16, history=("uniform", (5, 90)),
                                          pool=("factor", 2.0), seed=21))
    q, kc, vc, _, _ = _layer(w)
    base = oracle.paged_decode(q, kc, vc, w.block_tables, w.context_lens, w.scale, lib=lib)
    g = torch.Generator().manual_seed(3)
    perm = torch.randperm(w.num_blocks, generator=g)          # new position of each block
    kc2 = torch.empty_like(kc)
    vc2 = torch.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    bt2 = w.block_tables.clone()
    used = bt2 >= 0
    bt2[used] = perm[bt2[used].long()].to(torch.int32)
    moved = oracle.paged_decode(q, kc2, vc2, bt2, w.context_lens, w.scale, lib=lib)
    assert torch.equal(base, moved), "permuting physical blocks changed the output"


def pin_constant_v(lib):
    w = wl.make_workload(wl.custom_config(2, 4, 2, 16, torch.float32, history=("uniform", (0, 50)),
                                          seed=22))
    q, kc, vc, _, _ = _layer(w)
    c = torch.linspace(-3, 3, 16)
    vc = c.expand_as(vc).contiguous()
    out = oracle.paged_decode(q, kc, vc, w.block_tables, w.context_lens, w.scale, lib=lib)
    _close(out, c.double().expand_as(out), TOL, "constant V")


def _mean_v(vc, block_tables, context_lens, Hq):
    _, Hkv, bs, D = vc.shape
    B = context_lens.numel()
    out = torch.zeros(B, Hq, D, dtype=torch.float64)
    for b in range(B):
        n = int(context_lens[b])
        for h in range(Hq):
            g = h // (Hq // Hkv)
            rows = [vc[int(block_tables[b, t // bs]), g, t % bs].double() for t in range(n)]
            out[b, h] = torch.stack(rows).mean(0)
    return out


def pin_zero_query_mean(lib):
    w = wl.make_workload(wl.custom_config(3, 6, 2, 8, torch.float32, history=("uniform", (0, 45)),
                                          seed=23))
    _, kc, vc, _, _ = _layer(w)
    q = torch.zeros(w.cfg.B, w.cfg.Hq, w.cfg.D)
    out = oracle.paged_decode(q, kc, vc, w.block_tables, w.context_lens, w.scale, lib=lib)
    _close(out, _mean_v(vc, w.block_tables, w.context_lens, w.cfg.Hq), TOL, "q=0 mean")
    out0 = oracle.paged_decode(w.q[0], kc, vc, w.block_tables, w.context_lens, 0.0, lib=lib)
    _close(out0, _mean_v(vc, w.block_tables, w.context_lens, w.cfg.Hq), TOL, "scale=0 mean")


def pin_dominant_key(lib):
    # One key gets a logit near 1000 (exp would overflow without the max
    # subtraction); every other weight is below e^-900, so the output is that
    # token's V row to double precision.
    w = wl.make_workload(wl.custom_config(2, 4, 4, 8, torch.float32, history=("fixed", (30,)),
                                          seed=24))
    q, kc, vc, _, _ = _layer(w)
    q = torch.zeros_like(q)
    q[..., 0] = 1.0
    kc = kc.clone()
    kc[..., 0] = 0.0
    t_star = 17
    bs = w.cfg.block_size
    expect = torch.zeros(w.cfg.B, w.cfg.Hq, w.cfg.D, dtype=torch.float64)
    for b in range(w.cfg.B):
        blk = int(w.block_tables[b, t_star // bs])
        kc[blk, :, t_star % bs, 0] = 1000.0
        expect[b] = vc[blk, :, t_star % bs].double()
    out = oracle.paged_decode(q, kc, vc, w.block_tables, w.context_lens, 1.0, lib=lib)
    _close(out, expect, TOL, "dominant key")


def pin_linearity_in_v(lib):
    w = wl.make_workload(wl.custom_config(2, 4, 2, 8, torch.float32, history=("uniform", (3, 60)),
                                          seed=25))
    q, kc, vc, _, _ = _layer(w)
    # Values on a 2^-10 grid in [-2, 2]: every sum below is exact in fp32.
    vc = torch.round(vc * 1024) / 1024
    v2 = torch.round(torch.roll(vc, 1, dims=-1) * 512) / 1024
    a = oracle.paged_decode(q, kc, vc, w.block_tables, w.context_lens, w.scale, lib=lib)
    b = oracle.paged_decode(q, kc, v2, w.block_tables, w.context_lens, w.scale, lib=lib)
    s = oracle.paged_decode(q, kc, vc + v2, w.block_tables, w.context_lens, w.scale, lib=lib)
    _close(s, a + b, 1e-11, "linearity in V")


def pin_bf16_widening(lib):
    w = wl.make_workload(wl.custom_config(2, 4, 2, 16, torch.bfloat16, history=("uniform", (1, 40)),
                                          seed=26))
    q, kc, vc, _, _ = _layer(w)
    a = oracle.paged_decode(q, kc, vc, w.block_tables, w.context_lens, w.scale, lib=lib)
    b = oracle.paged_decode(q.float(), kc.float(), vc.float(), w.block_tables, w.context_lens,
                            w.scale, lib=lib)
    assert torch.equal(a, b), "bf16 widening is not exact"


def pin_append_bytes(lib):
    for dtype in (torch.float32, torch.bfloat16):
        w = wl.make_workload(wl.custom_config(5, 4, 2, 16, dtype, history=("uniform", (0, 40)),
                                              pool=("factor", 2.0), seed=27), pool_fill="canary")
        _, kc, vc, kn, vn = _layer(w)
        slots = oracle.slot_mapping(w.block_tables, w.context_lens, w.cfg.block_size, w.num_blocks,
                                    lib=lib)
        kc2, vc2 = oracle.kv_append(kn, vn, kc, vc, slots, lib=lib)
        itype = torch.int16 if dtype == torch.bfloat16 else torch.int32
        bs = w.cfg.block_size
        ek, ev = kc.clone(), vc.clone()
        for b in range(w.cfg.B):
            p = int(w.context_lens[b]) - 1
            blk = int(w.block_tables[b, p // bs])
            ek[blk, :, p % bs] = kn[b]
            ev[blk, :, p % bs] = vn[b]
        assert torch.equal(kc2.view(itype), ek.view(itype)), "K append bytes differ"
        assert torch.equal(vc2.view(itype), ev.view(itype)), "V append bytes differ"
    # Skipped tokens (slot < 0) write nothing.
    kc3, vc3 = oracle.kv_append(kn, vn, kc, vc, torch.full_like(slots, -1), lib=lib)
    assert torch.equal(kc3.view(itype), kc.view(itype)) and torch.equal(vc3.view(itype), vc.view(itype))


def pin_cache_equals_recompute(lib):
    w = wl.make_workload(wl.custom_config(4, 8, 2, 32, torch.bfloat16, history=("uniform", (0, 100)),
                                          pool=("factor", 1.5), seed=28))
    q, kc, vc, kn, vn = _layer(w)
    slots = oracle.slot_mapping(w.block_tables, w.context_lens, w.cfg.block_size, w.num_blocks, lib=lib)
    kc2, vc2 = oracle.kv_append(kn, vn, kc, vc, slots, lib=lib)
    cached = oracle.paged_decode(q, kc2, vc2, w.block_tables, w.context_lens, w.scale, lib=lib)
    # Recompute: history gathered from the untouched pool, the new row
    # appended from k_new/v_new, dense attention on the result.
    bs, Hkv, D = w.cfg.block_size, w.cfg.Hkv, w.cfg.D
    rep = w.cfg.Hq // Hkv
    for b in range(w.cfg.B):
        hist = int(w.history_lens[b])
        pages = w.block_tables[b, : (hist + bs - 1) // bs].long()
        K = kc[pages].double().permute(0, 2, 1, 3).reshape(-1, Hkv, D)[:hist]
        V = vc[pages].double().permute(0, 2, 1, 3).reshape(-1, Hkv, D)[:hist]
        K = torch.cat([K, kn[b].double().unsqueeze(0)]).transpose(0, 1).repeat_interleave(rep, 0)
        V = torch.cat([V, vn[b].double().unsqueeze(0)]).transpose(0, 1).repeat_interleave(rep, 0)
        att = torch.softmax(torch.matmul(q[b].double().unsqueeze(1), K.transpose(1, 2)) * w.scale, -1)
        _close(cached[b], torch.matmul(att, V).squeeze(1), TOL, f"cache==recompute seq {b}")


# ------------------------------------------------------- sinks + sliding window

def pin_sink_window_by_hand(lib):
    c = gc.load_cases()["sink_window_by_hand"]
    q = torch.tensor(c["q"], dtype=torch.float32)
    kc, vc = gc.pool_tensor(c, "k_cache"), gc.pool_tensor(c, "v_cache")
    out = oracle.paged_decode_sinks(q, kc, vc, torch.tensor(c["block_tables"]),
                                    torch.tensor(c["context_lens"]), gc.scale_of(c),
                                    sinks=torch.tensor(c["sinks"], dtype=torch.float32),
                                    window=c["window"], lib=lib)
    _close(out, gc.expected_of(c), 1e-14, "sink_window_by_hand")


def dense_sinks_window(q, k_cache, v_cache, block_tables, context_lens, scale, sinks, window):
    """Dense float64 formulation: the last `window` tokens gathered to a
    contiguous copy, the sink appended as one more key column whose value row
    is zero, then torch.softmax and matmul."""
    B, Hq, D = q.shape
    _, Hkv, bs, _ = k_cache.shape
    rep = Hq // Hkv
    out = torch.zeros(B, Hq, D, dtype=torch.float64)
    for b in range(B):
        n = int(context_lens[b])
        if n <= 0:
            continue
        pages = block_tables[b, : (n + bs - 1) // bs].long()
        K = k_cache[pages].double().permute(0, 2, 1, 3).reshape(-1, Hkv, D)[:n]
        V = v_cache[pages].double().permute(0, 2, 1, 3).reshape(-1, Hkv, D)[:n]
        if window > 0:
            K, V = K[-window:], V[-window:]
        K = K.transpose(0, 1).repeat_interleave(rep, dim=0)
        V = V.transpose(0, 1).repeat_interleave(rep, dim=0)
        logits = torch.matmul(q[b].double().unsqueeze(1), K.transpose(1, 2)).squeeze(1) * scale
        if sinks is not None:
            logits = torch.cat([logits, sinks.double().unsqueeze(1)], dim=1)
            V = torch.cat([V, torch.zeros(Hq, 1, D, dtype=torch.float64)], dim=1)
        out[b] = torch.matmul(torch.softmax(logits, dim=-1).unsqueeze(1), V).squeeze(1)
    return out


def pin_sinks_window_dense(lib):
    for dtype, G, window in ((torch.float32, 2, 5), (torch.bfloat16, 4, 33), (torch.float32, 1, 0)):
        w = wl.make_workload(wl.custom_config(4, 4 * G, 4, 16, dtype, history=("uniform", (0, 90)),
                                              pool=("factor", 1.5), seed=41 + G))
        q, kc, vc, _, _ = _layer(w)
        g = torch.Generator().manual_seed(G)
        sinks = (torch.randn(w.cfg.Hq, generator=g) * 2).to(dtype)
        got = oracle.paged_decode_sinks(q, kc, vc, w.block_tables, w.context_lens, w.scale,
                                        sinks=sinks, window=window, lib=lib)
        ref = dense_sinks_window(q, kc, vc, w.block_tables, w.context_lens, w.scale, sinks, window)
        _close(got, ref, TOL, f"sinks+window dense {dtype} G={G} W={window}")


def pin_sinks_window_reduce_to_plain(lib):
    w = wl.make_workload(wl.custom_config(3, 8, 2, 16, torch.bfloat16, history=("uniform", (1, 70)),
                                          pool=("factor", 2.0), seed=44))
    q, kc, vc, _, _ = _layer(w)
    plain = oracle.paged_decode(q, kc, vc, w.block_tables, w.context_lens, w.scale, lib=lib)
    # No sink and no window, or a window as long as every context: the plain oracle.
    a = oracle.paged_decode_sinks(q, kc, vc, w.block_tables, w.context_lens, w.scale, lib=lib)
    b = oracle.paged_decode_sinks(q, kc, vc, w.block_tables, w.context_lens, w.scale,
                                  window=int(w.context_lens.max()), lib=lib)
    _close(a, plain, TOL, "no sink, no window")
    _close(b, plain, TOL, "window >= context")
    # A sink far below every logit changes nothing; one far above sends the output to 0.
    low = oracle.paged_decode_sinks(q, kc, vc, w.block_tables, w.context_lens, w.scale,
                                    sinks=torch.full((w.cfg.Hq,), -1e4), lib=lib)
    high = oracle.paged_decode_sinks(q, kc, vc, w.block_tables, w.context_lens, w.scale,
                                     sinks=torch.full((w.cfg.Hq,), 1e4), lib=lib)
    _close(low, plain, TOL, "sink -> -inf")
    _close(high, torch.zeros_like(plain), TOL, "sink -> +inf")


# ------------------------------------------------------------------- KV swap

def pin_swap_by_indexing(lib):
    """Swap-out then swap-in against tensor indexing, bit for bit."""
    g = torch.Generator().manual_seed(51)
    for dtype in (torch.bfloat16, torch.float32):
        dev_k = torch.randn(12, 2, 16, 8, generator=g).to(dtype)
        dev_v = torch.randn(12, 2, 16, 8, generator=g).to(dtype)
        host_k = torch.randn(5, 2, 16, 8, generator=g).to(dtype)
        host_v = torch.randn(5, 2, 16, 8, generator=g).to(dtype)
        out_map = torch.tensor([[7, 0], [2, 3], [-1, 4], [11, 1]])
        hk, hv = oracle.kv_swap(dev_k, dev_v, host_k, host_v, out_map, lib=lib)
        ek, ev = host_k.clone(), host_v.clone()
        ek[[0, 3, 1]] = dev_k[[7, 2, 11]]
        ev[[0, 3, 1]] = dev_v[[7, 2, 11]]
        iv = lambda t: t.view(torch.int16 if t.element_size() == 2 else torch.int32)
        assert torch.equal(iv(hk), iv(ek)) and torch.equal(iv(hv), iv(ev)), "swap-out"
        # Swap the three blocks back in to other device blocks.
        in_map = torch.tensor([[0, 9], [3, 4], [1, 5]])
        dk, dv = oracle.kv_swap(hk, hv, dev_k, dev_v, in_map, lib=lib)
        fk, fv = dev_k.clone(), dev_v.clone()
        fk[[9, 4, 5]] = dev_k[[7, 2, 11]]
        fv[[9, 4, 5]] = dev_v[[7, 2, 11]]
        assert torch.equal(iv(dk), iv(fk)) and torch.equal(iv(dv), iv(fv)), "swap-in"
    # A block id past a pool is an error, never a silent copy.
    try:
        oracle.kv_swap(dev_k, dev_v, host_k, host_v, torch.tensor([[12, 0]]), lib=lib)
    except oracle.OracleError:
        pass
    else:
        raise AssertionError("out-of-range source block accepted")


# ---------------------------------------------------------------- allocator

def pin_alloc_by_hand(lib):
    c = gc.load_cases()["alloc_by_hand"]
    bt, cl, top, failed = oracle.block_alloc_decode(
        torch.tensor(c["block_tables"]), torch.tensor(c["context_lens"]), c["block_size"],
        torch.tensor(c["free_stack"]), c["free_top"], lib=lib)
    assert bt.tolist() == c["expected_tables"], bt.tolist()
    assert cl.tolist() == c["expected_lens"] and top == c["expected_top"]
    assert failed.tolist() == c["expected_failed"]


def pin_alloc_free_conserve_blocks(lib):
    """Blocks are neither lost nor duplicated: over many steps and releases,
    the blocks in use plus the free stack are always a permutation of the
    pool, and every sequence's table covers exactly its length."""
    g = torch.Generator().manual_seed(61)
    nb, B, bs, width = 40, 6, 4, 12
    stack = torch.randperm(nb, generator=g).to(torch.int32)
    top = nb
    bt = torch.full((B, width), -1, dtype=torch.int32)
    cl = torch.tensor([0, 3, -1, 7, 0, 1], dtype=torch.int32)
    # Give the non-empty sequences their pages by allocating token by token.
    lens0 = cl.clone()
    cl = torch.where(cl >= 0, torch.zeros_like(cl), cl)
    for step in range(int(lens0.max())):
        live = cl < lens0
        bt2, cl2, top, _ = oracle.block_alloc_decode(bt, torch.where(live, cl, -1), bs, stack, top,
                                                     lib=lib)
        bt, cl = bt2, torch.where(live, cl2, cl)
    for step in range(30):
        bt, cl, top, failed = oracle.block_alloc_decode(bt, cl, bs, stack, top, lib=lib)
        if step % 7 == 6:
            victim = int(torch.randint(0, B, (1,), generator=g))
            if cl[victim] >= 0:
                bt, cl, stack, top = oracle.block_free([victim], bt, cl, bs, stack, top, lib=lib)
                cl[victim] = 0          # register a new sequence in the freed slot
        used = [int(bt[b, p]) for b in range(B) if cl[b] > 0
                for p in range((int(cl[b]) + bs - 1) // bs)]
        pool = sorted(used + stack[:top].tolist())
        assert pool == list(range(nb)), f"step {step}: blocks lost or duplicated"
        for b in range(B):
            n = int(cl[b])
            if n >= 0:
                pages = (n + bs - 1) // bs
                assert (bt[b, :pages] >= 0).all() and (bt[b, pages:] == -1).all()


# ------------------------------------------------------------------ prefill

def pin_prefill_by_hand(lib):
    c = gc.load_cases()["prefill_by_hand"]
    kc, vc = gc.pool_tensor(c, "k_cache"), gc.pool_tensor(c, "v_cache")
    ids = torch.tensor(c["block_ids"], dtype=torch.int32)
    ks = torch.tensor(c["k_src"], dtype=torch.float32)
    vs = torch.tensor(c["v_src"], dtype=torch.float32)
    kc2, vc2 = oracle.prefill_append(ks, vs, kc, vc, ids, c["start_pos"], lib=lib)
    out = oracle.paged_prefill(torch.tensor(c["q"], dtype=torch.float32), kc2, vc2, ids,
                               c["start_pos"], gc.scale_of(c), lib=lib)
    _close(out, gc.expected_of(c), 1e-14, "prefill_by_hand")


def _prefill_case(seed, dtype, G, start, T, bs=16, Hkv=2, D=16):
    g = torch.Generator().manual_seed(seed)
    Hq = Hkv * G
    total = start + T
    pages = (total + bs - 1) // bs
    nb = pages + 3
    ids = torch.randperm(nb, generator=g)[:pages].to(torch.int32)
    kc = torch.randn(nb, Hkv, bs, D, generator=g).to(dtype)
    vc = torch.randn(nb, Hkv, bs, D, generator=g).to(dtype)
    ks = torch.randn(Hkv, T, D, generator=g).to(dtype)
    vs = torch.randn(Hkv, T, D, generator=g).to(dtype)
    q = torch.randn(T, Hq, D, generator=g).to(dtype)
    return q, kc, vc, ks, vs, ids


def pin_prefill_dense_and_decode_rows(lib):
    for seed, dtype, G, start, T in ((1, torch.float32, 1, 0, 37), (2, torch.bfloat16, 4, 21, 50),
                                     (3, torch.float32, 2, 48, 16)):
        q, kc, vc, ks, vs, ids = _prefill_case(seed, dtype, G, start, T)
        kc2, vc2 = oracle.prefill_append(ks, vs, kc, vc, ids, start, lib=lib)
        scale = 0.25
        out = oracle.paged_prefill(q, kc2, vc2, ids, start, scale, lib=lib)
        # Dense: contiguous copy of tokens 0 .. start+T-1, offset causal mask.
        _, Hkv, bs, D = kc.shape
        Hq = q.shape[1]
        total = start + T
        K = kc2[ids.long()].double().permute(0, 2, 1, 3).reshape(-1, Hkv, D)[:total]
        V = vc2[ids.long()].double().permute(0, 2, 1, 3).reshape(-1, Hkv, D)[:total]
        K = K.transpose(0, 1).repeat_interleave(Hq // Hkv, 0)           # [Hq, total, D]
        V = V.transpose(0, 1).repeat_interleave(Hq // Hkv, 0)
        s_ = torch.matmul(q.double().transpose(0, 1), K.transpose(1, 2)) * scale   # [Hq, T, total]
        mask = torch.arange(total)[None, :] > (start + torch.arange(T))[:, None]
        s_ = s_.masked_fill(mask, float("-inf"))
        dense = torch.matmul(torch.softmax(s_, -1), V).transpose(0, 1)           # [T, Hq, D]
        _close(out, dense, TOL, f"prefill dense seed {seed}")
        # Row i is the decode step of the token at position start + i.
        for i in (0, T // 2, T - 1):
            bt = ids.unsqueeze(0)
            dec = oracle.paged_decode(q[i:i + 1], kc2, vc2, bt,
                                      torch.tensor([start + i + 1], dtype=torch.int32), scale,
                                      lib=lib)
            assert torch.equal(dec[0], out[i]), f"prefill row {i} differs from decode"


def pin_prefill_chunking_and_append(lib):
    q, kc, vc, ks, vs, ids = _prefill_case(9, torch.bfloat16, 4, 5, 40)
    start, T, T1 = 5, 40, 17
    whole_k, whole_v = oracle.prefill_append(ks, vs, kc, vc, ids, start, lib=lib)
    a_k, a_v = oracle.prefill_append(ks[:, :T1].contiguous(), vs[:, :T1].contiguous(), kc, vc, ids,
                                     start, lib=lib)
    b_k, b_v = oracle.prefill_append(ks[:, T1:].contiguous(), vs[:, T1:].contiguous(), a_k, a_v,
                                     ids, start + T1, lib=lib)
    iv = lambda t: t.view(torch.int16)
    assert torch.equal(iv(whole_k), iv(b_k)) and torch.equal(iv(whole_v), iv(b_v))
    # The append against tensor indexing.
    ek, ev = kc.clone(), vc.clone()
    for i in range(T):
        pos = start + i
        ek[ids[pos // 16], :, pos % 16] = ks[:, i]
        ev[ids[pos // 16], :, pos % 16] = vs[:, i]
    assert torch.equal(iv(whole_k), iv(ek)) and torch.equal(iv(whole_v), iv(ev))
    # Chunked attention equals one-shot attention row for row.
    one = oracle.paged_prefill(q, whole_k, whole_v, ids, start, 0.3, lib=lib)
    first = oracle.paged_prefill(q[:T1].contiguous(), a_k, a_v, ids, start, 0.3, lib=lib)
    second = oracle.paged_prefill(q[T1:].contiguous(), b_k, b_v, ids, start + T1, 0.3, lib=lib)
    assert torch.equal(one, torch.cat([first, second]))


ALL_PINS = [
    pin_slots_by_hand, pin_gqa_paged_by_hand, pin_single_token, pin_dense_equivalence,
    pin_brute_force_python, pin_permutation_invariance, pin_constant_v, pin_zero_query_mean,
    pin_dominant_key, pin_linearity_in_v, pin_bf16_widening, pin_append_bytes,
    pin_cache_equals_recompute, pin_sink_window_by_hand, pin_sinks_window_dense,
    pin_sinks_window_reduce_to_plain, pin_swap_by_indexing, pin_alloc_by_hand,
    pin_alloc_free_conserve_blocks, pin_prefill_by_hand, pin_prefill_dense_and_decode_rows,
    pin_prefill_chunking_and_append,
]
