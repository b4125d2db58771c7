"""Prefill append + chunked causal attention over the paged cache, against
the oracle; chunks of one sequence run back to back like a chunked prefill."""
import pytest
import torch

import oracle
from paged_kv_cache_xs_gb300 import ops
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,G,D", [(torch.bfloat16, 4, 128), (torch.float32, 1, 64),
                                       (torch.bfloat16, 8, 64), (torch.float32, 2, 128)])
def test_chunked_prefill_matches_oracle(dtype, G, D):
    dev = gh.device()
    g = torch.Generator().manual_seed(G * 1000 + D)
    Hkv, bs = 4, 16
    Hq = Hkv * G
    chunks = [37, 256, 1, 400]                     # ragged chunk sizes, one single token
    total = sum(chunks)
    pages = (total + bs - 1) // bs
    nb = pages + 11
    ids = torch.randperm(nb, generator=g)[:pages].to(torch.int32)
    kc = torch.randn(nb, Hkv, bs, D, generator=g).to(dtype)
    vc = torch.randn(nb, Hkv, bs, D, generator=g).to(dtype)
    dkc, dvc, dids = kc.to(dev), vc.to(dev), ids.to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    start = 0
    for T in chunks:
        ks = torch.randn(Hkv, T, D, generator=g).to(dtype)
        vs = torch.randn(Hkv, T, D, generator=g).to(dtype)
        q = torch.randn(T, Hq, D, generator=g).to(dtype)
        kc, vc = oracle.prefill_append(ks, vs, kc, vc, ids, start)
        ops.xs_prefill_append(ks.to(dev), vs.to(dev), dkc, dvc, dids, start, err_flag=err)
        ref = oracle.paged_prefill(q, kc, vc, ids, start, D ** -0.5)
        for P in (64, 4096):
            ws = ops.DecodeWorkspace(T, Hq, Hkv, D, pages, dev, partition_tokens=P)
            out = torch.full((T, Hq, D), float("nan"), dtype=dtype, device=dev)
            ops.xs_paged_prefill(out, ws.part_o, ws.part_m, ws.part_l, q.to(dev), dkc, dvc, dids,
                                 start, D ** -0.5, ws.partition_tokens, ws.max_partitions,
                                 err_flag=err, work_counters=ws.work)
            torch.cuda.synchronize()
            assert int(err.item()) == 0
            gh.assert_close(out, ref, dtype, what=f"chunk at {start} (T={T}) P={P}")
        assert torch.equal(gh.int_view(dkc.cpu()), gh.int_view(kc))
        assert torch.equal(gh.int_view(dvc.cpu()), gh.int_view(vc))
        start += T


def test_prefill_rejects_a_chunk_past_its_block_list():
    dev = gh.device()
    ids = torch.arange(2, dtype=torch.int32, device=dev)
    kc = torch.zeros(4, 2, 16, 64, dtype=torch.bfloat16, device=dev)
    q = torch.zeros(10, 2, 64, dtype=torch.bfloat16, device=dev)
    out = torch.empty_like(q)
    with pytest.raises(ops.XsError) as e:
        ops.xs_paged_prefill(out, None, None, None, q, kc, kc, ids, 25, 0.125, 64, 1)
    assert e.value.code == -2
