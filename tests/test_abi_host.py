"""libxs_paged without a GPU: it builds, loads, exports every entry point the
header declares, and its host-side logic (split heuristic, workspace sizes,
argument validation) behaves as documented.  Validation errors return before
any CUDA call, so these run on a machine with no GPU."""
import glob
import os
import re

import pytest

from paged_kv_cache_xs_gb300 import build as xsbuild
from paged_kv_cache_xs_gb300 import ops

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    xsbuild.build()
    return ops.load()


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        names.update(re.findall(r"^(?:int|int64_t|size_t|void)\s+(xs_\w+)\s*\(", text, flags=re.M))
    return sorted(names)


def test_header_declares_entry_points():
    names = declared_functions()
    for required in ("xs_kv_append", "xs_paged_decode_attn", "xs_paged_decode_reduce",
                     "xs_slot_mapping"):
        assert required in names


def test_every_defined_entry_point_is_declared():
    # The reverse direction: no extern "C" function of the sources ships
    # without its declaration (and documentation) in the header.
    defined = set()
    for src in glob.glob(os.path.join(ROOT, "paged_kv_cache_xs_gb300", "csrc", "*.cu")):
        text = open(src).read()
        defined.update(re.findall(r'extern "C"\s+(?:int|int64_t|size_t|void)\s+(xs_\w+)\s*\(',
                                  text))
    assert "xs_paged_decode_step" in defined
    undeclared = sorted(defined - set(declared_functions()))
    assert not undeclared, f"defined but not declared in include/: {undeclared}"


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, f"not exported: {missing}"


def test_binding_covers_every_declared_symbol():
    assert set(declared_functions()) <= set(ops.SIGNATURES), \
        set(declared_functions()) - set(ops.SIGNATURES)


def test_version(lib):
    assert lib.xs_version() >= 100


def test_partition_heuristic(lib):
    for B, Hkv, total, mx in [(128, 8, 128 * 18433, 32769), (1, 8, 4097, 4097),
                              (64, 8, 64 * 1300, 8193), (8, 12, 8 * 600, 1025), (2, 12, 29, 21)]:
        P = ops.xs_paged_decode_partition_tokens(B, Hkv, total, mx, 152)
        assert 64 <= P <= 2048 and (P & (P - 1)) == 0
    # Large batches get long partitions; a single stream gets short ones.
    assert ops.xs_paged_decode_partition_tokens(128, 8, 128 * 18433, 32769, 152) >= 1024
    assert ops.xs_paged_decode_partition_tokens(1, 8, 4097, 4097, 152) == 128
    # More SMs never asks for bigger partitions.
    a = ops.xs_paged_decode_partition_tokens(64, 8, 64 * 1300, 8193, 76)
    b = ops.xs_paged_decode_partition_tokens(64, 8, 64 * 1300, 8193, 152)
    assert b <= a
    assert ops.load().xs_paged_decode_partition_tokens(-1, 8, 0, 0, 152) == -2


def test_step_partition_heuristic(lib):
    # The one-launch step's choice on measured workloads (the persistent grid;
    # launches small enough for one wave of clusters take their own split).
    # Its constants were fitted to per-launch times swept over every
    # candidate P, launched back to back: the continuous-batching mix (64
    # sequences) ran 41.05 / 40.60 / 40.69 / 42.80 us at P = 448 / 512 / 576 /
    # 640; 48 log-uniform sequences 38.56 / 36.42 / 37.63 at 448 / 512 / 576;
    # the long batch is fastest at 2048.  Equal-length batches land on a
    # whole round of 304 CTAs: 4 x 4097 tokens at 512 (256 items), 8 x 2049
    # and 16 x 1025 at 576 (256 items, each shorter than at 640).
    pick = ops.xs_paged_decode_step_partition_tokens
    assert pick(64, 32, 8, 63638, 7598, 152) == 512
    assert pick(48, 32, 8, 55827, 7399, 152) == 512
    assert pick(1, 32, 8, 4097, 4097, 152) == 256
    assert pick(128, 32, 8, 2538762, 32769, 152) == 2048
    assert pick(4, 32, 8, 16388, 4097, 152) == 512
    assert pick(8, 32, 8, 8 * 2049, 2049, 152) == 576
    assert pick(16, 32, 8, 16 * 1025, 1025, 152) == 576
    assert pick(1, 32, 8, 1025, 1025, 152) in (128, 192)
    for B, Hq, Hkv, total, mx in [(8, 12, 12, 3439, 926), (2, 12, 12, 29, 21), (512, 32, 8, 10**6, 8193)]:
        P = pick(B, Hq, Hkv, total, mx, 152)
        assert 64 <= P <= 2048 and P % 64 == 0
    # More SMs never asks for bigger partitions.
    assert pick(64, 32, 8, 63638, 7598, 152) <= pick(64, 32, 8, 63638, 7598, 76)
    with pytest.raises(ops.XsError):
        pick(4, 12, 8, 100, 50, 152)   # Hq not a multiple of Hkv


def test_num_splits(lib):
    # The split-K factor of the longest sequence: the context cut into the
    # heuristic's partitions; a single stream is split, a large batch of
    # short contexts is not.
    for B, Hkv, mx in [(1, 8, 4097), (128, 8, 32769), (64, 8, 8193), (8, 12, 1025), (2, 12, 21)]:
        P = ops.xs_paged_decode_partition_tokens(B, Hkv, B * mx, mx, 152)
        assert ops.xs_paged_decode_num_splits(B, Hkv, mx, 152) == max(1, -(-mx // P))
    assert ops.xs_paged_decode_num_splits(1, 8, 4097, 152) > 1
    assert ops.xs_paged_decode_num_splits(512, 8, 64, 152) == 1
    assert ops.xs_paged_decode_num_splits(1, 8, 0, 152) == 1
    assert lib.xs_paged_decode_num_splits(1, 0, 100, 152) == -2   # XS_ESHAPE


def test_max_partitions_and_workspace(lib):
    assert ops.xs_paged_decode_max_partitions(2049, 16, 1024) == 33
    assert ops.xs_paged_decode_max_partitions(1, 16, 1024) == 1
    assert ops.xs_paged_decode_max_partitions(0, 16, 64) == 1
    n = 128 * 32 * 33
    up = lambda x: (x + 255) // 256 * 256
    assert ops.xs_paged_decode_workspace_bytes(128, 32, 128, 33) == up(n * 128 * 4) + 2 * up(n * 4)
    assert ops.xs_paged_decode_workspace_bytes(0, 32, 128, 33) == 0


# Fake, non-null, 16-byte-aligned "device" addresses: every call below is
# rejected by host-side validation before anything touches CUDA.
A = 1 << 20


def _attn(lib, **kw):
    args = dict(out=A, po=A, pm=A, pl=A, q=A, k=A, v=A, bt=A, maxb=4, lens=A, B=2, Hq=8, Hkv=2,
                D=128, bs=16, nb=10, scale=0.1, P=16, maxp=4, dtype=1, err=None, work=None,
                stream=None)
    args.update(kw)
    return lib.xs_paged_decode_attn(args["out"], args["po"], args["pm"], args["pl"], args["q"],
                                    args["k"], args["v"], args["bt"], args["maxb"], args["lens"],
                                    args["B"], args["Hq"], args["Hkv"], args["D"], args["bs"],
                                    args["nb"], args["scale"], args["P"], args["maxp"],
                                    args["dtype"], args["err"], args["work"], args["stream"])


def test_attn_argument_validation(lib):
    assert _attn(lib, B=0) == 0                     # nothing to do, nothing launched
    assert _attn(lib, q=None) == -1
    assert _attn(lib, bt=None) == -1
    assert _attn(lib, dtype=7) == -3
    assert _attn(lib, Hq=6, Hkv=4) == -2            # Hq % Hkv != 0
    assert _attn(lib, B=-1) == -2
    assert _attn(lib, D=96) == -5
    assert _attn(lib, bs=32) == -5
    assert _attn(lib, Hq=24, Hkv=2) == -5           # group of 12
    assert _attn(lib, P=24) == -2                   # not a multiple of 16
    assert _attn(lib, maxp=3) == -6                 # 4 blocks * 16 / 16 = 4 partitions needed
    assert _attn(lib, po=None) == -6
    assert _attn(lib, k=A + 8) == -4
    assert _attn(lib, out=A + 2) == -4
    assert _attn(lib, B=20000) == -5                # beyond the per-launch batch limit


def test_append_argument_validation(lib):
    f = lib.xs_kv_append
    assert f(A, A, A, A, A, 0, 8, 128, 16, 10, 1, None, None) == 0   # T == 0
    assert f(None, A, A, A, A, 3, 8, 128, 16, 10, 1, None, None) == -1
    assert f(A, A, A, A, None, 3, 8, 128, 16, 10, 1, None, None) == -1
    assert f(A, A, A, A, A, 3, 8, 128, 16, 10, 5, None, None) == -3
    assert f(A, A, A, A, A, 3, 0, 128, 16, 10, 1, None, None) == -2
    assert f(A, A, A, A, A, 3, 8, 4, 16, 10, 1, None, None) == -5     # 8-byte rows
    assert f(A, A, A + 4, A, A, 3, 8, 128, 16, 10, 1, None, None) == -4
    g = lib.xs_kv_append_paged
    assert g(A, A, A, A, None, 4, A, 3, 8, 128, 16, 10, 1, None, None) == -1
    assert g(A, A, A, A, A, 4, A, 0, 8, 128, 16, 10, 1, None, None) == 0
    assert lib.xs_slot_mapping(None, 4, A, 3, 16, 10, A, None, None) == -1
    assert lib.xs_slot_mapping(A, 4, A, 0, 16, 10, A, None, None) == 0
    assert lib.xs_paged_decode_reduce(A, A, A, A, A, 2, 8, 128, 16, 1, 1, None) == 0
    assert lib.xs_paged_decode_reduce(A, None, A, A, A, 2, 8, 128, 16, 4, 1, None) == -6
    assert lib.xs_paged_decode_reduce(A, A, A, A, A, 2, 8, 128, 16, 4, 9, None) == -3


def test_binding_raises_on_error_code(lib):
    with pytest.raises(ops.XsError) as e:
        ops._call("xs_slot_mapping", None, 4, A, 3, 16, 10, A, None, None)
    assert e.value.code == -1


def _fused(lib, **kw):
    a = dict(out=A, q=A, kn=A, vn=A, k=A, v=A, bt=A, maxb=4, lens=A, sinks=None, window=0, B=2,
             Hq=8, Hkv=2, D=128, bs=16, nb=10, scale=0.1, P=16, maxp=4, po=A, pm=A, pl=A,
             counters=A, dtype=1, err=None, stream=None)
    a.update(kw)
    return lib.xs_paged_decode_step(a["out"], a["q"], a["kn"], a["vn"], a["k"], a["v"], a["bt"],
                                    a["maxb"], a["lens"], a["sinks"], a["window"], a["B"],
                                    a["Hq"], a["Hkv"], a["D"], a["bs"], a["nb"], a["scale"],
                                    a["P"], a["maxp"], a["po"], a["pm"], a["pl"],
                                    a["counters"], a["dtype"], a["err"], a["stream"])


def test_fused_step_argument_validation(lib):
    assert _fused(lib, B=0) == 0                     # nothing to do, nothing launched
    assert _fused(lib, counters=None) == -6
    assert _fused(lib, kn=None) == -1                # k_new and v_new: both or neither
    assert _fused(lib, vn=None) == -1
    assert _fused(lib, kn=A + 4) == -4
    assert _fused(lib, window=-1) == -2
    assert _fused(lib, maxp=3) == -6
    assert _fused(lib, po=None) == -6
    assert _fused(lib, D=96) == -5
    assert _fused(lib, lens=None) == -1
    assert ops.xs_paged_decode_step_counters(128, 8) == 2 + 128 * 8
    assert lib.xs_paged_decode_step_counters(-1, 8) == -2


def test_prefill_tc_argument_validation(lib):
    f = lib.xs_paged_prefill_tc
    #        out q  k  v  ids n_ids T start Hq Hkv D  bs nb  scale dtype err stream
    assert f(A, A, A, A, A, 4, 0, 0, 8, 2, 128, 16, 10, 0.1, 1, None, None) == 0   # T == 0
    assert f(None, A, A, A, A, 4, 8, 0, 8, 2, 128, 16, 10, 0.1, 1, None, None) == -1
    assert f(A, A, A, A, A, 4, 8, 0, 8, 2, 128, 16, 10, 0.1, 0, None, None) == -5  # fp32
    assert f(A, A, A, A, A, 4, 8, 0, 8, 2, 128, 16, 10, 0.1, 7, None, None) == -3
    assert f(A, A, A, A, A, 4, 8, 0, 8, 3, 128, 16, 10, 0.1, 1, None, None) == -2  # Hq % Hkv
    assert f(A, A, A, A, A, 4, 8, 0, 8, 2, 96, 16, 10, 0.1, 1, None, None) == -5
    assert f(A, A, A, A, A, 4, 8, 0, 32, 2, 128, 16, 10, 0.1, 1, None, None) == -5  # G = 16
    assert f(A, A, A, A, A, 4, 60, 10, 8, 2, 128, 16, 10, 0.1, 1, None, None) == -2  # past ids
    assert f(A, A, A + 8, A, A, 4, 8, 0, 8, 2, 128, 16, 10, 0.1, 1, None, None) == -4


def test_step_ex_flags_validated(lib):
    # Unknown flag bits are refused before anything else is looked at.
    args = [None] * 7 + [0, None, None, 0, 1, 8, 8, 64, 16, 1, 0.125, 64, 1, None, None, None, None]
    assert lib.xs_paged_decode_step_ex(*args, 4, ops.XS_BF16, None, None) == -5
    assert lib.xs_paged_decode_step_ex(*args, 1 << 30, ops.XS_BF16, None, None) == -5
    # Known flags (XS_STEP_EARLY_READS, XS_STEP_PERSISTENT, both) pass through
    # to the usual checks (NULL counters here).
    for flags in (1, 2, 3):
        assert lib.xs_paged_decode_step_ex(*args, flags, ops.XS_BF16, None, None) == -6


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    # No CPU fallback: without the compiled library every wrapper raises
    # instead of computing anything another way.
    from paged_kv_cache_xs_gb300 import build as b
    with pytest.raises(ImportError):
        ops.load(str(tmp_path / "libxs_paged.so"))
    monkeypatch.setattr(b, "LIB_PATH", str(tmp_path / "libxs_paged.so"))
    prev = ops.use_library(None)
    try:
        with pytest.raises(ImportError):
            ops.xs_version()
        with pytest.raises(ImportError):
            ops.xs_paged_decode_num_splits(1, 8, 4097, 152)
    finally:
        ops.use_library(prev)


def test_workspace_holder_sizes(lib):
    # The binding's workspace holder (built on the host here: only sizes are
    # checked) agrees with the library's sizing calls: partition length from
    # the one-launch heuristic, partials for every partition a sequence of
    # the table's width can need, and the step's counters.
    import torch
    B, Hq, Hkv, D, maxb = 64, 32, 8, 128, 475
    ws = ops.DecodeWorkspace(B, Hq, Hkv, D, maxb, "cpu", total_context_tokens=63638,
                             max_context_len=7598, num_sms=152)
    assert ws.partition_tokens == ops.xs_paged_decode_step_partition_tokens(B, Hq, Hkv, 63638,
                                                                            7598, 152)
    mp = ops.xs_paged_decode_max_partitions(maxb, 16, ws.partition_tokens)
    assert ws.max_partitions == mp
    assert ws.part_o.numel() == B * Hq * mp * D and ws.part_m.numel() == B * Hq * mp
    assert ws.part_o.dtype == torch.float32
    assert ws.work.numel() == ops.xs_paged_decode_step_counters(B, Hkv) == 2 + B * Hkv
    assert not bool(ws.work.any())
    assert ws.partial_bytes <= ops.xs_paged_decode_workspace_bytes(B, Hq, D, mp)
    one = ops.DecodeWorkspace(4, 32, 8, 128, 2, "cpu", partition_tokens=64, num_sms=152)
    assert one.max_partitions == 1 and one.part_o is None and one.partial_bytes == 0


def test_wait_injection_is_debug_only(lib):
    # The release library refuses the debug-only wait injection without
    # touching the device; the debug library checks its arguments first.
    assert lib.xs_debug_wait_injection(1_000_000, 2) == -5       # XS_EUNSUPPORTED
    xsbuild.build(debug_bounds=True)
    dbg = ops.load_debug()
    assert dbg.xs_debug_wait_injection(0, -1) == -2              # XS_ESHAPE: no limit
    assert dbg.xs_debug_wait_injection(1_000_000, -2) == -2      # XS_ESHAPE: bad page


def test_num_splits_form_validation(lib):
    # The split as a count: num_splits <= 0 is refused before anything else;
    # B == 0 does nothing; num_splits == 1 needs no partials and no reduce.
    f, r = lib.xs_paged_decode_attn_splits, lib.xs_paged_decode_reduce_splits
    base = [A, A, A, A, A, A, A, A, 4, A, 2, 8, 2, 128, 16, 10, 0.1]
    assert f(*base, 0, 1, None, None) == -2
    assert f(*base, -3, 1, None, None) == -2
    assert r(A, A, A, A, A, 4, 2, 8, 128, 16, 0, 1, None) == -2
    assert f(A, A, A, A, A, A, A, A, 4, A, 0, 8, 2, 128, 16, 10, 0.1, 3, 1, None, None) == 0
    assert r(A, None, None, None, A, 4, 2, 8, 128, 16, 1, 1, None) == 0


def test_prefill_overlap_flags_validated(lib):
    # Unknown flag bits are refused first; XS_PREFILL_OVERLAP passes to the
    # usual checks (a NULL pointer here).
    app = lib.xs_prefill_append_ex
    assert app(A, A, A, A, A, 4, 8, 2, 128, 16, 10, 0, 2, 1, None, None) == -5
    assert app(None, A, A, A, A, 4, 8, 2, 128, 16, 10, 0, 1, 1, None, None) == -1
    tc = lib.xs_paged_prefill_tc_ex
    assert tc(A, A, A, A, A, 4, 8, 0, 8, 2, 128, 16, 10, 0.1, 2, 1, None, None) == -5
    assert tc(None, A, A, A, A, 4, 8, 0, 8, 2, 128, 16, 10, 0.1, 1, 1, None, None) == -1
