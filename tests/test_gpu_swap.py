"""KV swap between the device pool and a pinned host swap pool, bit-exact
against the oracle's kv_swap."""
import pytest
import torch

import oracle
from paged_kv_cache_xs_gb300 import ops
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_swap_out_and_in(dtype):
    dev = gh.device()
    g = torch.Generator().manual_seed(7)
    nb, nh, Hkv, D = 300, 64, 8, 128
    kd = torch.randn(nb, Hkv, 16, D, generator=g).to(dtype)
    vd = torch.randn(nb, Hkv, 16, D, generator=g).to(dtype)
    kh = torch.randn(nh, Hkv, 16, D, generator=g).to(dtype).pin_memory()
    vh = torch.randn(nh, Hkv, 16, D, generator=g).to(dtype).pin_memory()
    kdev, vdev = kd.to(dev), vd.to(dev)
    src = torch.randperm(nb, generator=g)[:50]
    dst = torch.randperm(nh, generator=g)[:50]
    out_map = torch.stack([src, dst], 1).to(torch.int64)
    out_map[7] = torch.tensor([-1, 3])            # skipped pair
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    # swap-out: device pool -> pinned host pool (mapping on the device)
    ek, ev = oracle.kv_swap(kd, vd, kh, vh, out_map)
    ops.xs_kv_swap(kdev, vdev, kh, vh, out_map.to(dev), err_flag=err)
    torch.cuda.synchronize()
    assert torch.equal(gh.int_view(kh), gh.int_view(ek)) and torch.equal(gh.int_view(vh), gh.int_view(ev))
    # swap-in: pinned host pool -> other device blocks (mapping in pinned host memory)
    in_map = torch.stack([dst, torch.randperm(nb, generator=g)[:50]], 1).to(torch.int64)
    in_map_h = in_map.pin_memory()
    fk, fv = oracle.kv_swap(kh, vh, kdev.cpu(), vdev.cpu(), in_map)
    ops.xs_kv_swap(kh, vh, kdev, vdev, in_map_h, err_flag=err)
    torch.cuda.synchronize()
    assert torch.equal(gh.int_view(kdev.cpu()), gh.int_view(fk))
    assert torch.equal(gh.int_view(vdev.cpu()), gh.int_view(fv))
    assert int(err.item()) == 0
    # Out-of-range ids are flagged and skipped.
    before = kh.clone()
    ops.xs_kv_swap(kdev, vdev, kh, vh, torch.tensor([[nb + 1, 0], [0, nh + 2]], device=dev),
                   err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & ops.FLAG_BAD_BLOCK
    assert torch.equal(gh.int_view(kh), gh.int_view(before))
