"""Chunked prefill attention on the tensor cores (xs_paged_prefill_tc) against
the oracle: ragged chunks at unaligned positions, every supported group size
and head dim, unwritten pool slots full of NaN bits, an out-of-pool block id,
and a long chunk that takes several waves of CTAs."""
import pytest
import torch

import oracle
from paged_kv_cache_xs_gb300 import ops
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu

CASES = [(4, 128), (1, 128), (2, 128), (8, 128), (1, 64), (2, 64), (4, 64), (8, 64)]


def _setup(g, Hkv, G, D, total, spare, fill_nan):
    bs = 16
    pages = (total + bs - 1) // bs
    nb = pages + spare
    ids = torch.randperm(nb, generator=g)[:pages].to(torch.int32)
    if fill_nan:
        kc = torch.full((nb, Hkv, bs, D), float("nan"), dtype=torch.bfloat16)
        vc = torch.full((nb, Hkv, bs, D), float("nan"), dtype=torch.bfloat16)
    else:
        kc = torch.randn(nb, Hkv, bs, D, generator=g).to(torch.bfloat16)
        vc = torch.randn(nb, Hkv, bs, D, generator=g).to(torch.bfloat16)
    return ids, kc, vc


@pytest.mark.parametrize("G,D", CASES, ids=[f"G{G}-D{D}" for G, D in CASES])
def test_chunks_match_oracle(G, D):
    # The pool starts as NaN: only appended rows hold numbers, so any read of
    # an unwritten slot (the tail of the last page) would show up as NaN.
    dev = gh.device()
    g = torch.Generator().manual_seed(500 + 10 * G + D)
    Hkv = 2
    Hq = Hkv * G
    chunks = [37, 256, 1, 129, 70]
    ids, kc, vc = _setup(g, Hkv, G, D, sum(chunks), 5, fill_nan=True)
    dkc, dvc, dids = kc.to(dev), vc.to(dev), ids.to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    start = 0
    for T in chunks:
        ks = torch.randn(Hkv, T, D, generator=g).to(torch.bfloat16)
        vs = torch.randn(Hkv, T, D, generator=g).to(torch.bfloat16)
        q = torch.randn(T, Hq, D, generator=g).to(torch.bfloat16)
        kc, vc = oracle.prefill_append(ks, vs, kc, vc, ids, start)
        ops.xs_prefill_append(ks.to(dev), vs.to(dev), dkc, dvc, dids, start, err_flag=err)
        ref = oracle.paged_prefill(q, kc, vc, ids, start, D ** -0.5)
        out = torch.full((T, Hq, D), float("nan"), dtype=torch.bfloat16, device=dev)
        ops.xs_paged_prefill_tc(out, q.to(dev), dkc, dvc, dids, start, D ** -0.5, err_flag=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert not torch.isnan(out).any(), f"NaN in the output of the chunk at {start}"
        gh.assert_close(out, ref, torch.bfloat16, what=f"chunk at {start} (T={T})")
        start += T


def test_long_chunk_several_waves():
    dev = gh.device()
    g = torch.Generator().manual_seed(77)
    Hkv, G, D = 8, 4, 128
    Hq = Hkv * G
    start, T = 1500, 1100
    ids, kc, vc = _setup(g, Hkv, G, D, start + T, 3, fill_nan=False)
    q = torch.randn(T, Hq, D, generator=g).to(torch.bfloat16)
    out = torch.empty(T, Hq, D, dtype=torch.bfloat16, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    ops.xs_paged_prefill_tc(out, q.to(dev), kc.to(dev), vc.to(dev), ids.to(dev), start,
                            D ** -0.5, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    # Sampled query rows (every CTA row position, first and last tokens).
    rows = sorted({0, 1, 15, 16, 17, 63, 64, 500, T - 2, T - 1} |
                  set(torch.randint(0, T, (20,), generator=g).tolist()))
    for r in rows:
        ref = oracle.paged_prefill(q[r:r + 1], kc, vc, ids, start + r, D ** -0.5)
        gh.assert_close(out[r:r + 1], ref, torch.bfloat16, what=f"row {r}")


def test_bad_block_is_flagged_and_read_as_zeros():
    dev = gh.device()
    g = torch.Generator().manual_seed(9)
    Hkv, G, D, T = 2, 4, 128, 40
    ids, kc, vc = _setup(g, Hkv, G, D, T, 2, fill_nan=False)
    ids_bad = ids.clone()
    ids_bad[1] = kc.shape[0] + 100                 # page 1 points outside the pool
    q = torch.randn(T, Hkv * G, D, generator=g).to(torch.bfloat16)
    out = torch.empty(T, Hkv * G, D, dtype=torch.bfloat16, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    ops.xs_paged_prefill_tc(out, q.to(dev), kc.to(dev), vc.to(dev), ids_bad.to(dev), 0,
                            D ** -0.5, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & ops.FLAG_BAD_BLOCK
    # Rows that only see page 0 are unaffected.
    ref = oracle.paged_prefill(q[:16], kc, vc, ids, 0, D ** -0.5)
    gh.assert_close(out[:16], ref, torch.bfloat16, what="rows before the bad page")


@pytest.mark.parametrize("G,D", [(4, 128), (1, 64), (8, 128)], ids=["G4-D128", "G1-D64", "G8-D128"])
def test_overlapped_chunks_match_oracle(G, D):
    # XS_PREFILL_OVERLAP: every chunk's append and attention launched back to
    # back with nothing between them on the stream (no host synchronisation,
    # no event), so chunk c + 1's append and the start of its attention run
    # beside chunk c's attention.  Ragged chunks at unaligned positions, the
    # pool starting as NaN; every chunk's output against the oracle's, and the
    # pages against the oracle's appends.
    dev = gh.device()
    g = torch.Generator().manual_seed(700 + 10 * G + D)
    Hkv = 2
    Hq = Hkv * G
    chunks = [300, 37, 512, 1, 129, 256, 70, 1024]
    ids, kc, vc = _setup(g, Hkv, G, D, sum(chunks), 5, fill_nan=True)
    dkc, dvc, dids = kc.to(dev), vc.to(dev), ids.to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    outs, refs = [], []
    start = 0
    inputs = []
    for T in chunks:
        ks = torch.randn(Hkv, T, D, generator=g).to(torch.bfloat16)
        vs = torch.randn(Hkv, T, D, generator=g).to(torch.bfloat16)
        q = torch.randn(T, Hq, D, generator=g).to(torch.bfloat16)
        inputs.append((ks.to(dev), vs.to(dev), q.to(dev)))
        kc, vc = oracle.prefill_append(ks, vs, kc, vc, ids, start)
        refs.append(oracle.paged_prefill(q, kc, vc, ids, start, D ** -0.5))
        outs.append(torch.full((T, Hq, D), float("nan"), dtype=torch.bfloat16, device=dev))
        start += T
    torch.cuda.synchronize()
    start = 0
    for (ks, vs, q), out, T in zip(inputs, outs, chunks):
        ops.xs_prefill_append(ks, vs, dkc, dvc, dids, start, err_flag=err, overlap=True)
        ops.xs_paged_prefill_tc(out, q, dkc, dvc, dids, start, D ** -0.5, err_flag=err,
                                overlap=True)
        start += T
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    start = 0
    for out, ref, T in zip(outs, refs, chunks):
        assert not torch.isnan(out).any(), f"NaN in the output of the chunk at {start}"
        gh.assert_close(out, ref, torch.bfloat16, what=f"chunk at {start} (T={T})")
        start += T
    assert torch.equal(gh.int_view(dkc.cpu()), gh.int_view(kc))
    assert torch.equal(gh.int_view(dvc.cpu()), gh.int_view(vc))
