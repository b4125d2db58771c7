"""The decode kernel's bounded waits, made to run out on purpose.

Every wait of the decode kernel (for a page, a q slot, a merge buffer, a
staged partial) gives up after a limit, raises XS_FLAG_TIMEOUT and lets the
launch drain its copies and return, so the context stays usable.  The debug
library can shorten that limit and make CTA 0's producer skip issuing one
page (xs_debug_wait_injection): nothing is in flight for that page, so the
consumer waiting for it runs out of time with no fault anywhere.  The tests
check the flag, that the launch returned within milliseconds, that no
in-kernel bounds check failed, and the recovery contract of
xs_paged_decode_step: after zeroing the counters, the next launch on the
same workspace is exact against the oracle - on the persistent grid and on
the cluster launch (where the skipped page is page 2 of the first
sequence's first KV head's first partition, and the CTA's other consumers,
its cluster's other CTAs and the cluster barriers all finish)."""
import time

import pytest
import torch

from paged_kv_cache_xs_gb300 import build as xsbuild
from paged_kv_cache_xs_gb300 import ops
from paged_kv_cache_xs_gb300 import workloads as wl
from paged_kv_cache_xs_gb300.step import PagedDecodeStep
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu

DEFAULT_LIMIT_NS = 4_000_000_000


def test_a_wait_that_runs_out_flags_timeout_and_the_next_launch_is_exact():
    dev = gh.device()
    xsbuild.build(debug_bounds=True)
    dbg = ops.load_debug()
    prev = ops.use_library(dbg)
    try:
        # Two split sequences: CTA 0's first item is partition 0 of sequence
        # 0, KV head 0 (16 pages of the 256-token partition), so its page 2
        # is one the kernel would otherwise stream.
        cfg = wl.custom_config(2, 32, 8, 128, torch.bfloat16, history=("fixed", (3000, 2500)),
                               pool=("factor", 1.5), seed=404, name="timeout_case")
        w = wl.make_workload(cfg, device=dev)
        step = PagedDecodeStep(cfg.B, cfg.Hq, cfg.Hkv, cfg.D, w.max_blocks_per_seq, cfg.dtype,
                               dev, partition_tokens=256)
        assert step.max_partitions > 1
        out = torch.empty(cfg.B, cfg.Hq, cfg.D, dtype=cfg.dtype, device=dev)
        torch.cuda.synchronize()
        ops.xs_debug_wait_injection(1_000_000, 2, lib=dbg)  # 1 ms waits; page 2 never issued
        try:
            t0 = time.perf_counter()
            step.run(out, w.q[0], w.k_new[0], w.v_new[0], w.k_cache[0], w.v_cache[0],
                     w.block_tables, w.context_lens, w.scale, persistent=True)
            torch.cuda.synchronize()
            elapsed = time.perf_counter() - t0
        finally:
            ops.xs_debug_wait_injection(DEFAULT_LIMIT_NS, -1, lib=dbg)
        flags = step.error_flags()
        assert flags == ops.FLAG_TIMEOUT, f"error flags {flags}, expected XS_FLAG_TIMEOUT only"
        assert elapsed < 1.0, f"the aborted launch took {elapsed:.3f} s with 1 ms waits"
        assert ops.xs_debug_bounds_failures(reset=True, lib=dbg) == 0
        # The aborted item never counted into its group, so some combine
        # count is left non-zero: the header tells the caller to zero them.
        assert int(step.ws.work.count_nonzero()) > 0
        step.ws.work.zero_()
        step.err_flag.zero_()
        # The same step again (it appends the same rows again): exact.
        gh.check_step(w, 0, step)
        assert ops.xs_debug_bounds_failures(reset=True, lib=dbg) == 0
    finally:
        ops.use_library(prev)



def test_a_wait_that_runs_out_in_a_cluster_launch():
    dev = gh.device()
    xsbuild.build(debug_bounds=True)
    dbg = ops.load_debug()
    prev = ops.use_library(dbg)
    try:
        # 8001 tokens split 12-16 ways: more pages a CTA than the ring has
        # stages, so after the consumer's wait for page 2 runs out, the
        # producer's wait for stage 2 to come free (for page 26) runs out too.
        cfg = wl.custom_config(1, 32, 8, 128, torch.bfloat16, history=("fixed", (8000,)),
                               pool=("factor", 1.2), seed=405, name="timeout_cluster_case")
        w = wl.make_workload(cfg, device=dev)
        cs = ops.xs_paged_decode_step_cluster_size(cfg.B, cfg.Hq, cfg.Hkv, cfg.D,
                                                   w.max_blocks_per_seq, 0, cfg.dtype)
        assert cs > 0 and -(-w.max_blocks_per_seq // cs) > 26
        step = PagedDecodeStep(cfg.B, cfg.Hq, cfg.Hkv, cfg.D, w.max_blocks_per_seq, cfg.dtype,
                               dev, partition_tokens=256)
        out = torch.empty(cfg.B, cfg.Hq, cfg.D, dtype=cfg.dtype, device=dev)
        torch.cuda.synchronize()
        ops.xs_debug_wait_injection(1_000_000, 2, lib=dbg)
        try:
            t0 = time.perf_counter()
            step.run(out, w.q[0], w.k_new[0], w.v_new[0], w.k_cache[0], w.v_cache[0],
                     w.block_tables, w.context_lens, w.scale)
            torch.cuda.synchronize()
            elapsed = time.perf_counter() - t0
        finally:
            ops.xs_debug_wait_injection(DEFAULT_LIMIT_NS, -1, lib=dbg)
        flags = step.error_flags()
        assert flags == ops.FLAG_TIMEOUT, f"error flags {flags}, expected XS_FLAG_TIMEOUT only"
        assert elapsed < 1.0, f"the aborted launch took {elapsed:.3f} s with 1 ms waits"
        assert ops.xs_debug_bounds_failures(reset=True, lib=dbg) == 0
        # The cluster launch keeps no counts: nothing to zero but the flag.
        assert int(step.ws.work.count_nonzero()) == 0
        step.err_flag.zero_()
        gh.check_step(w, 0, step)
        assert ops.xs_debug_bounds_failures(reset=True, lib=dbg) == 0
    finally:
        ops.use_library(prev)
