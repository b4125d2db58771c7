"""CPU fp64 oracle for the paged-KV decode step.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's ``cpu_baseline`` / ``--impl reference`` legs may import this
package.  The product path (``paged_kv_cache_xs_gb300``) never imports it and
shares no code with it.

The arithmetic lives in ``paged_oracle.c`` (plain C, fp64, OpenMP over
(sequence, query head)); this module only compiles it with gcc and marshals
arguments.  Each function follows the definition cited in the C source:

* ``slot_mapping``  - slot resolution of the token a decode step writes
  ("xserv compare phase10...cf1e9e4", attention.rs,
  ``reshape_and_cache_batched_bf16``: the per-sequence length passed to the
  append already counts the token being written).
* ``kv_append``     - byte copy of each new K/V row into its pool slot (same
  page, ``reshape_and_cache_bf16`` pool layout).
* ``prefill_append`` / ``paged_prefill`` - the prefill side: a chunk of T
  tokens written at start_pos (reshape_and_cache_bf16) and its causal
  attention over the paged cache (attention with an offset causal mask).
* ``block_alloc_decode`` / ``block_free`` - the page allocator of a decode
  step: a free stack of block ids, a new page whenever a token starts one.
* ``kv_swap``       - whole-block copies between a device pool and a host
  swap pool (the README's CPU swap-out/in of KV blocks).
* ``paged_decode_sinks`` - the gpt-oss variant: per-head sink logits in the
  softmax denominator and a sliding window (same page, paged_decode_attention_sinks).
* ``paged_decode``  - softmax(scale * q K^T) V over every cached token of the
  sequence, keys and values gathered through the block table, GQA head map
  h -> h / (Hq/Hkv) ("xserv compare phase8...phase13", qwen3.rs ``repeat_kv``;
  "xserv compare phase5...phase9", docs/09-kv-cache.md "After (with cache)").

Parity pins (tests/test_oracle_pins.py) tie these to closed forms,
hand-derived golden values, an independent dense formulation and
invariants.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "paged_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

F32 = 0
BF16 = 1

_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle C source with gcc (OpenMP, -O2, no -ffast-math)."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def load(path: str | None = None):
    """Load (building first if needed) the oracle shared library."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _bind(lib):
    P, I, L, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
    lib.oracle_slot_mapping.argtypes = [P, I, P, I, I, L, P]
    lib.oracle_kv_append.argtypes = [P, P, P, P, P, I, I, I, I, L, I]
    lib.oracle_paged_decode.argtypes = [P, P, P, P, I, P, I, I, I, I, I, L, D, I, P, I]
    lib.oracle_paged_decode_sinks.argtypes = [P, P, P, P, I, P, I, I, I, I, I, L, D, P, I, I, P, I]
    lib.oracle_kv_swap.argtypes = [P, P, P, P, P, I, L, L, L]
    lib.oracle_block_alloc_decode.argtypes = [P, I, P, I, I, P, P, P]
    lib.oracle_block_free.argtypes = [P, I, P, I, P, I, P, P, L]
    lib.oracle_prefill_append.argtypes = [P, P, P, P, P, I, I, I, I, I, L, I, I]
    lib.oracle_paged_prefill.argtypes = [P, P, P, P, I, I, I, I, I, I, I, L, D, I, P, I]
    lib.oracle_max_threads.argtypes = []
    for f in (lib.oracle_slot_mapping, lib.oracle_kv_append, lib.oracle_paged_decode,
              lib.oracle_paged_decode_sinks, lib.oracle_kv_swap, lib.oracle_block_alloc_decode,
              lib.oracle_block_free, lib.oracle_prefill_append, lib.oracle_paged_prefill,
              lib.oracle_max_threads):
        f.restype = ctypes.c_int
    return lib


class OracleError(RuntimeError):
    pass


def _check(status: int, what: str) -> None:
    if status != 0:
        raise OracleError(f"{what}: oracle status {status}")


def _cpu(t: torch.Tensor, dtype=None) -> torch.Tensor:
    if not isinstance(t, torch.Tensor):
        t = torch.as_tensor(np.asarray(t))
    if dtype is not None:
        t = t.to(dtype)
    return t.detach().to("cpu").contiguous()


def _code(dtype: torch.dtype) -> int:
    if dtype == torch.float32:
        return F32
    if dtype == torch.bfloat16:
        return BF16
    raise ValueError(f"oracle supports float32 and bfloat16, not {dtype}")


def default_threads() -> int:
    return len(os.sched_getaffinity(0))


def slot_mapping(block_tables, context_lens, block_size: int, num_blocks: int,
                 lib=None) -> torch.Tensor:
    """int64 [B] slots of the token each sequence writes this step (-1: none)."""
    lib = lib or load()
    bt = _cpu(block_tables, torch.int32)
    cl = _cpu(context_lens, torch.int32)
    B = cl.numel()
    out = torch.empty(B, dtype=torch.int64)
    st = lib.oracle_slot_mapping(bt.data_ptr(), bt.shape[1] if bt.dim() == 2 else 0,
                                 cl.data_ptr(), B, block_size, num_blocks, out.data_ptr())
    _check(st, "slot_mapping")
    return out


def kv_append(k_new, v_new, k_cache, v_cache, slot_mapping, lib=None):
    """Return copies of (k_cache, v_cache) with the new rows written in."""
    lib = lib or load()
    kn, vn = _cpu(k_new), _cpu(v_new)
    kc, vc = _cpu(k_cache).clone(), _cpu(v_cache).clone()
    sm = _cpu(slot_mapping, torch.int64)
    T, Hkv, D = kn.shape
    num_blocks, _, bs, _ = kc.shape
    st = lib.oracle_kv_append(kn.data_ptr(), vn.data_ptr(), kc.data_ptr(), vc.data_ptr(),
                              sm.data_ptr(), T, Hkv, D, bs, num_blocks, _code(kn.dtype))
    _check(st, "kv_append")
    return kc, vc


def paged_decode(q, k_cache, v_cache, block_tables, context_lens, scale: float,
                 nthreads: int | None = None, lib=None) -> torch.Tensor:
    """fp64 [B, Hq, D] attention output of one decode step."""
    lib = lib or load()
    qq, kc, vc = _cpu(q), _cpu(k_cache), _cpu(v_cache)
    bt = _cpu(block_tables, torch.int32)
    cl = _cpu(context_lens, torch.int32)
    B, Hq, D = qq.shape
    num_blocks, Hkv, bs, D2 = kc.shape
    if D2 != D or kc.dtype != qq.dtype or vc.dtype != qq.dtype:
        raise ValueError("q and pools must share head_dim and dtype")
    out = torch.empty(B, Hq, D, dtype=torch.float64)
    st = lib.oracle_paged_decode(qq.data_ptr(), kc.data_ptr(), vc.data_ptr(), bt.data_ptr(),
                                 bt.shape[1], cl.data_ptr(), B, Hq, Hkv, D, bs, num_blocks,
                                 float(scale), _code(qq.dtype), out.data_ptr(),
                                 nthreads or default_threads())
    _check(st, "paged_decode")
    return out


def paged_decode_sinks(q, k_cache, v_cache, block_tables, context_lens, scale: float,
                       sinks=None, window: int = 0, nthreads: int | None = None,
                       lib=None) -> torch.Tensor:
    """fp64 [B, Hq, D]: decode attention with per-head sinks ([Hq], q's dtype,
    or None) and a sliding window of the last ``window`` tokens (0 = all)."""
    lib = lib or load()
    qq, kc, vc = _cpu(q), _cpu(k_cache), _cpu(v_cache)
    bt = _cpu(block_tables, torch.int32)
    cl = _cpu(context_lens, torch.int32)
    B, Hq, D = qq.shape
    num_blocks, Hkv, bs, _ = kc.shape
    sk = None if sinks is None else _cpu(sinks, qq.dtype)
    out = torch.empty(B, Hq, D, dtype=torch.float64)
    st = lib.oracle_paged_decode_sinks(qq.data_ptr(), kc.data_ptr(), vc.data_ptr(), bt.data_ptr(),
                                       bt.shape[1], cl.data_ptr(), B, Hq, Hkv, D, bs, num_blocks,
                                       float(scale), None if sk is None else sk.data_ptr(),
                                       int(window), _code(qq.dtype), out.data_ptr(),
                                       nthreads or default_threads())
    _check(st, "paged_decode_sinks")
    return out


def kv_swap(src_k, src_v, dst_k, dst_v, mapping, lib=None):
    """Return copies of (dst_k, dst_v) with the mapped blocks of the source
    pools copied in; mapping is int64 [n, 2] of (source block, destination
    block), pools are [blocks, ...] tensors of one dtype."""
    lib = lib or load()
    sk, sv = _cpu(src_k), _cpu(src_v)
    dk, dv = _cpu(dst_k).clone(), _cpu(dst_v).clone()
    mp = _cpu(mapping, torch.int64).reshape(-1, 2).contiguous()
    block_bytes = sk[0].numel() * sk.element_size() if sk.shape[0] else \
        dk[0].numel() * dk.element_size()
    st = lib.oracle_kv_swap(sk.data_ptr(), sv.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                            mp.data_ptr(), mp.shape[0], block_bytes, sk.shape[0], dk.shape[0])
    _check(st, "kv_swap")
    return dk, dv


def block_alloc_decode(block_tables, context_lens, block_size, free_stack, free_top, lib=None):
    """One decode step's page allocation.  Returns new (block_tables,
    context_lens, free_top, failed) - inputs are not modified."""
    lib = lib or load()
    bt = _cpu(block_tables, torch.int32).clone()
    cl = _cpu(context_lens, torch.int32).clone()
    fs = _cpu(free_stack, torch.int32)
    top = torch.tensor([int(free_top)], dtype=torch.int32)
    failed = torch.zeros(cl.numel(), dtype=torch.int32)
    st = lib.oracle_block_alloc_decode(bt.data_ptr(), bt.shape[1], cl.data_ptr(), cl.numel(),
                                       block_size, fs.data_ptr(), top.data_ptr(), failed.data_ptr())
    _check(st, "block_alloc_decode")
    return bt, cl, int(top.item()), failed


def block_free(seq_ids, block_tables, context_lens, block_size, free_stack, free_top, lib=None):
    """Release sequences.  Returns new (block_tables, context_lens,
    free_stack, free_top)."""
    lib = lib or load()
    ids = _cpu(seq_ids, torch.int32)
    bt = _cpu(block_tables, torch.int32).clone()
    cl = _cpu(context_lens, torch.int32).clone()
    fs = _cpu(free_stack, torch.int32).clone()
    top = torch.tensor([int(free_top)], dtype=torch.int32)
    st = lib.oracle_block_free(ids.data_ptr(), ids.numel(), bt.data_ptr(), bt.shape[1],
                               cl.data_ptr(), block_size, fs.data_ptr(), top.data_ptr(),
                               fs.numel())
    _check(st, "block_free")
    return bt, cl, fs, int(top.item())


def prefill_append(k_src, v_src, k_cache, v_cache, block_ids, start_pos: int, lib=None):
    """Copies of (k_cache, v_cache) with the chunk k_src/v_src ([Hkv, T, D])
    written at positions start_pos .. start_pos + T - 1 of one sequence."""
    lib = lib or load()
    ks, vs = _cpu(k_src), _cpu(v_src)
    kc, vc = _cpu(k_cache).clone(), _cpu(v_cache).clone()
    ids = _cpu(block_ids, torch.int32).reshape(-1)
    Hkv, T, D = ks.shape
    num_blocks, _, bs, _ = kc.shape
    st = lib.oracle_prefill_append(ks.data_ptr(), vs.data_ptr(), kc.data_ptr(), vc.data_ptr(),
                                   ids.data_ptr(), ids.numel(), T, Hkv, D, bs, num_blocks,
                                   int(start_pos), _code(ks.dtype))
    _check(st, "prefill_append")
    return kc, vc


def paged_prefill(q, k_cache, v_cache, block_ids, start_pos: int, scale: float,
                  nthreads: int | None = None, lib=None) -> torch.Tensor:
    """fp64 [T, Hq, D]: causal attention of a T-token chunk (q [T, Hq, D],
    positions start_pos ..) over one sequence's paged cache."""
    lib = lib or load()
    qq, kc, vc = _cpu(q), _cpu(k_cache), _cpu(v_cache)
    ids = _cpu(block_ids, torch.int32).reshape(-1)
    T, Hq, D = qq.shape
    num_blocks, Hkv, bs, _ = kc.shape
    out = torch.empty(T, Hq, D, dtype=torch.float64)
    st = lib.oracle_paged_prefill(qq.data_ptr(), kc.data_ptr(), vc.data_ptr(), ids.data_ptr(),
                                  ids.numel(), T, int(start_pos), Hq, Hkv, D, bs, num_blocks,
                                  float(scale), _code(qq.dtype), out.data_ptr(),
                                  nthreads or default_threads())
    _check(st, "paged_prefill")
    return out
