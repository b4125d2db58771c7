"""The GPU suite on the debug library.

libxs_paged_debug.so is built from the same sources with -DXS_DEBUG_BOUNDS:
before every global-memory access whose index a kernel computes (block-table
entries, q and new-row offsets, the pool slot an append writes, the partials
a combine reads, the rows an output write touches), the index is checked
against its buffer's extent; a failed check skips the access, raises
XS_FLAG_BOUNDS and is counted.  This stands in for a device memory checker,
which this pool does not offer.  A child pytest runs every other GPU test
with the debug library in place of the release one (XS_TEST_LIBRARY=debug,
see conftest.py), which also requires the count to be zero after each test.
"""
import os
import subprocess
import sys

import pytest
import torch

from paged_kv_cache_xs_gb300 import build as xsbuild
from paged_kv_cache_xs_gb300 import ops
from paged_kv_cache_xs_gb300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.gpu


def test_release_library_has_no_checks():
    xsbuild.build()
    release = ops.load(xsbuild.LIB_PATH)  # by path: whichever library is installed
    assert ops.xs_debug_bounds_failures(lib=release) == -5  # XS_EUNSUPPORTED


def test_debug_library_step_counts_no_failures():
    # In process: one one-launch step on the debug library, counter read back.
    xsbuild.build(debug_bounds=True)
    lib = ops.load_debug()
    assert ops.xs_debug_bounds_failures(reset=True, lib=lib) >= 0
    prev = ops.use_library(lib)
    try:
        dev = torch.device("cuda:0")
        cfg = wl.custom_config(7, 32, 8, 128, torch.bfloat16, history=("loguniform", (1, 3000)),
                               pool=("factor", 1.3), seed=881)
        w = wl.make_workload(cfg, device=dev)
        ws = ops.DecodeWorkspace(cfg.B, cfg.Hq, cfg.Hkv, cfg.D, w.max_blocks_per_seq, dev,
                                 partition_tokens=128)
        out = torch.empty(cfg.B, cfg.Hq, cfg.D, dtype=cfg.dtype, device=dev)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        ops.xs_paged_decode_step(out, w.q[0], w.k_new[0], w.v_new[0], w.k_cache[0],
                                 w.v_cache[0], w.block_tables, w.context_lens, w.scale,
                                 ws.partition_tokens, ws.max_partitions, ws.part_o, ws.part_m,
                                 ws.part_l, ws.work, err_flag=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert ops.xs_debug_bounds_failures(reset=True, lib=lib) == 0
    finally:
        ops.use_library(prev)


@pytest.mark.skipif(os.environ.get("XS_TEST_LIBRARY") == "debug",
                    reason="already running on the debug library")
def test_gpu_suite_on_debug_library():
    xsbuild.build(debug_bounds=True)
    torch.cuda.empty_cache()  # leave the device memory this process cached to the child
    env = dict(os.environ, XS_TEST_LIBRARY="debug")
    me = "tests/test_gpu_debug_bounds.py"
    r = subprocess.run([sys.executable, "-m", "pytest", "tests", "-m", "gpu", "-q", "-x",
                        "-p", "no:cacheprovider", "--deselect", f"{me}::test_gpu_suite_on_debug_library"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1500)
    tail = (r.stdout[-4000:] + "\n" + r.stderr[-2000:])
    print(tail)
    assert r.returncode == 0, tail
