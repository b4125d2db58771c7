"""Device-side page allocator and a whole decode loop replayed as one CUDA
graph per step, against the oracle.

Which popped block lands in which sequence depends on the order of atomic
operations, so the tests compare what is unique (lengths, the stack top, the
set of blocks handed out) and check that the rest is valid.  Attention output
does not depend on where pages sit (a pinned oracle invariant), so the decode
loop is compared with the oracle running its own allocation on its own copy
of the state."""
import pytest
import torch

import oracle
from paged_kv_cache_xs_gb300 import ops
from paged_kv_cache_xs_gb300 import workloads as wl
from paged_kv_cache_xs_gb300.step import CapturedStep, PagedDecodeStep
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu


def _state(seed, B=24, width=6, nb=200, bs=16):
    g = torch.Generator().manual_seed(seed)
    lens = torch.randint(0, width * bs, (B,), generator=g, dtype=torch.int32)
    lens[::5] = (lens[::5] // bs) * bs          # some sit exactly on a page boundary
    lens[3] = -1                                # an empty slot
    lens[7] = width * bs                        # its next page is past the table
    perm = torch.randperm(nb, generator=g).to(torch.int32)
    bt = torch.full((B, width), -1, dtype=torch.int32)
    pos = 0
    for b in range(B):
        pages = (max(int(lens[b]), 0) + bs - 1) // bs
        bt[b, :pages] = perm[pos:pos + pages]
        pos += pages
    stack = perm[pos:].clone()
    return bt, lens, stack


@pytest.mark.parametrize("dry", [False, True])
def test_alloc_step_matches_oracle(dry):
    dev = gh.device()
    bt, lens, stack = _state(3)
    top = 2 if dry else stack.numel()          # dry: fewer free blocks than needed
    obt, olens, otop, ofailed = oracle.block_alloc_decode(bt, lens, 16, stack, top)
    dbt, dlens = bt.to(dev), lens.to(dev)
    dstack = stack.to(dev)
    dtop = torch.tensor([top], dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    ops.xs_block_alloc_decode(dbt, dlens, dstack, dtop, err_flag=err)
    torch.cuda.synchronize()
    gbt, glens, gtop = dbt.cpu(), dlens.cpu(), int(dtop.item())
    assert gtop == otop
    assert int(err.item()) & ops.FLAG_BAD_LEN                       # slot 7
    assert bool(int(err.item()) & ops.FLAG_POOL_EMPTY) == dry
    popped = sorted(stack[otop:top].tolist())
    new = sorted(int(gbt[b, p]) for b in range(bt.shape[0]) for p in range(bt.shape[1])
                 if gbt[b, p] != bt[b, p])
    assert new == popped, "the blocks handed out are not the popped ones"
    if not dry:
        assert torch.equal(glens, olens)
        changed = (gbt != bt)
        assert torch.equal(changed, obt != bt), "a page went to the wrong slot"
    else:
        # Exactly as many sequences advanced as the oracle's, each page-starting
        # one that advanced got a block, the others are untouched.
        assert int((glens != lens).sum()) == int((olens != lens).sum())
        for b in range(bt.shape[0]):
            if glens[b] != lens[b]:
                assert glens[b] == lens[b] + 1
                if lens[b] % 16 == 0:
                    assert gbt[b, lens[b] // 16] != bt[b, lens[b] // 16]


def test_free_matches_oracle():
    dev = gh.device()
    bt, lens, stack = _state(4)
    top = stack.numel() - 10
    cap = stack.numel() + 200
    full_stack = torch.cat([stack, torch.full((200,), -7, dtype=torch.int32)])
    ids = torch.tensor([0, 5, 11, 3], dtype=torch.int32)       # 3 is an empty slot
    obt, olens, ostack, otop = oracle.block_free(ids, bt, lens, 16, full_stack, top)
    dbt, dlens, dstack = bt.to(dev), lens.to(dev), full_stack.to(dev)
    dtop = torch.tensor([top], dtype=torch.int32, device=dev)
    ops.xs_block_free(ids.to(dev), dbt, dlens, dstack, dtop)
    torch.cuda.synchronize()
    assert int(dtop.item()) == otop
    assert torch.equal(dbt.cpu(), obt) and torch.equal(dlens.cpu(), olens)
    assert sorted(dstack.cpu()[top:otop].tolist()) == sorted(ostack[top:otop].tolist())
    assert dstack.numel() == cap


def test_decode_loop_as_one_graph_per_step():
    dev = gh.device()
    B, Hq, Hkv, D, bs, steps = 7, 32, 8, 128, 16, 40
    dtype = torch.bfloat16
    g = torch.Generator().manual_seed(11)
    hist = torch.randint(0, 300, (B,), dtype=torch.int32, generator=g)
    hist[2] = 15                               # the next token starts page 1
    hist[4] = -1                               # an empty slot
    width = (int(hist.max()) + steps + bs) // bs + 1
    nb = B * width + 8
    perm = torch.randperm(nb, generator=g).to(torch.int32)
    bt = torch.full((B, width), -1, dtype=torch.int32)
    pos = 0
    for b in range(B):
        pages = (max(int(hist[b]), 0) + bs - 1) // bs
        bt[b, :pages] = perm[pos:pos + pages]
        pos += pages
    stack = perm[pos:].clone()
    kc = torch.randn(nb, Hkv, bs, D, generator=g).to(dtype)
    vc = torch.randn(nb, Hkv, bs, D, generator=g).to(dtype)

    # Device state; the captured step reads q / k_new / v_new from fixed buffers.
    dbt, dlens, dstack = bt.to(dev), hist.to(dev), stack.to(dev)
    dtop = torch.tensor([stack.numel()], dtype=torch.int32, device=dev)
    dkc, dvc = kc.to(dev), vc.to(dev)
    q = torch.zeros(B, Hq, D, dtype=dtype, device=dev)
    kn = torch.zeros(B, Hkv, D, dtype=dtype, device=dev)
    vn = torch.zeros(B, Hkv, D, dtype=dtype, device=dev)
    out = torch.zeros(B, Hq, D, dtype=dtype, device=dev)
    step = PagedDecodeStep(B, Hq, Hkv, D, width, dtype, dev, partition_tokens=64)

    def one_step():
        ops.xs_block_alloc_decode(dbt, dlens, dstack, dtop, err_flag=step.err_flag)
        step.run(out, q, kn, vn, dkc, dvc, dbt, dlens, D ** -0.5)

    snap = [t.clone() for t in (dbt, dlens, dstack, dtop, dkc, dvc)]
    graph = CapturedStep(one_step)              # its warm-up advances the state once...
    for t, s0 in zip((dbt, dlens, dstack, dtop, dkc, dvc), snap):
        t.copy_(s0)                             # ...so put the state back before replaying
    obt, olens, otop, okc, ovc = bt.clone(), hist.clone(), stack.numel(), kc.clone(), vc.clone()
    for s in range(steps):
        q.copy_(torch.randn(B, Hq, D, generator=g).to(dtype))
        kn.copy_(torch.randn(B, Hkv, D, generator=g).to(dtype))
        vn.copy_(torch.randn(B, Hkv, D, generator=g).to(dtype))
        graph.replay()
        # The oracle's own step on its own state.
        obt, olens, otop, _ = oracle.block_alloc_decode(obt, olens, bs, stack, otop)
        slots = oracle.slot_mapping(obt, olens, bs, nb)
        okc, ovc = oracle.kv_append(kn.cpu(), vn.cpu(), okc, ovc, slots)
        ref = oracle.paged_decode(q.cpu(), okc, ovc, obt, olens, D ** -0.5)
        torch.cuda.synchronize()
        assert step.error_flags() == 0
        assert torch.equal(dlens.cpu(), olens) and int(dtop.item()) == otop
        live = [b for b in range(B) if olens[b] > 0]
        gh.assert_close(out[live], ref[live], dtype, what=f"step {s}")
