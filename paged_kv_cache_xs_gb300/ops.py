"""Python binding of libxs_paged (argument marshalling only).

Each ``xs_*`` function here calls the C entry point of the same name in
``include/xs_paged.h`` with ``tensor.data_ptr()`` values and the current
PyTorch CUDA stream; every step of the decode path runs in the library's
kernels.  PyTorch supplies device memory and streams.  There is no fallback:
if the shared library is missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

XS_F32 = 0
XS_BF16 = 1
BLOCK_SIZE = 16

STATUS = {
    0: "XS_OK", -1: "XS_ENULL", -2: "XS_ESHAPE", -3: "XS_EDTYPE", -4: "XS_EALIGN",
    -5: "XS_EUNSUPPORTED", -6: "XS_EWORKSPACE", -7: "XS_ELAUNCH", -8: "XS_EDEVICE",
    -9: "XS_ESCRATCH",
}
NOALLOC_SCRATCH_BYTES = 64 << 20
FLAG_BAD_BLOCK, FLAG_BAD_LEN, FLAG_BAD_SLOT, FLAG_TIMEOUT, FLAG_CONFIG = 1, 2, 4, 8, 16
FLAG_POOL_EMPTY = 32

# name -> (restype, argtypes)
_P, _I, _L, _F, _S = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                      ctypes.c_size_t)
SIGNATURES = {
    "xs_slot_mapping": (_I, [_P, _I, _P, _I, _I, _L, _P, _P, _P]),
    "xs_kv_append": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _L, _I, _P, _P]),
    "xs_kv_append_paged": (_I, [_P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _L, _I, _P, _P]),
    "xs_paged_decode_partition_tokens": (_I, [_I, _I, _L, _I, _I]),
    "xs_paged_decode_max_partitions": (_I, [_I, _I, _I]),
    "xs_paged_decode_num_splits": (_I, [_I, _I, _I, _I]),
    "xs_paged_decode_workspace_bytes": (_S, [_I, _I, _I, _I]),
    "xs_paged_decode_attn": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I,
                                  _L, _F, _I, _I, _I, _P, _P, _P]),
    "xs_paged_decode_reduce": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P]),
    "xs_paged_decode": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _L, _F,
                             _I, _I, _I, _P, _P, _P]),
    "xs_paged_decode_noalloc": (_I, [_P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _L, _F,
                                     _I, _I, _P, _P]),
    "xs_paged_decode_attn_sinks": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _P, _P, _I, _I, _I,
                                        _I, _I, _I, _L, _F, _I, _I, _I, _P, _P, _P]),
    "xs_paged_decode_reduce_sinks": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I,
                                          _P]),
    "xs_paged_decode_sinks": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I,
                                   _I, _I, _L, _F, _I, _I, _I, _P, _P, _P]),
    "xs_kv_swap": (_I, [_P, _P, _P, _P, _P, _I, _L, _L, _L, _P, _P]),
    "xs_block_alloc_decode": (_I, [_P, _I, _P, _I, _I, _P, _P, _P, _P]),
    "xs_block_free": (_I, [_P, _I, _P, _I, _P, _I, _I, _P, _P, _L, _P, _P]),
    "xs_prefill_append": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _L, _I, _I, _P, _P]),
    "xs_prefill_append_ex": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _L, _I, _I, _I, _P,
                                  _P]),
    "xs_paged_prefill_attn": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I,
                                   _L, _F, _I, _I, _I, _P, _P, _P]),
    "xs_paged_prefill_reduce": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P]),
    "xs_paged_prefill": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _L, _F,
                              _I, _I, _I, _P, _P, _P]),
    "xs_paged_prefill_tc": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _L, _F, _I, _P,
                                 _P]),
    "xs_paged_prefill_tc_ex": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _L, _F, _I,
                                    _I, _P, _P]),
    "xs_paged_decode_step": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I,
                                  _I, _L, _F, _I, _I, _P, _P, _P, _P, _I, _P, _P]),
    "xs_paged_decode_step_ex": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I,
                                     _I, _L, _F, _I, _I, _P, _P, _P, _P, _I, _I, _P, _P]),
    "xs_paged_decode_step_counters": (_L, [_I, _I]),
    "xs_paged_decode_step_cluster_size": (_I, [_I, _I, _I, _I, _I, _I, _I]),
    "xs_paged_decode_attn_splits": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I,
                                         _I, _L, _F, _I, _I, _P, _P]),
    "xs_paged_decode_reduce_splits": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P]),
    "xs_paged_decode_step_partition_tokens": (_I, [_I, _I, _I, _L, _I, _I]),
    "xs_version": (_I, []),
    "xs_debug_bounds_failures": (_I, [_I]),
    "xs_debug_wait_injection": (_I, [_L, _I]),
}

_lock = threading.Lock()
_lib = None


class XsError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {STATUS.get(code, code)} ({code})")
        self.code = code


def lib_path() -> str:
    return _build.LIB_PATH


def load(path: str | None = None):
    """Load libxs_paged.so (built in-tree by ``build.build()``)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or _build.LIB_PATH
        if not os.path.exists(p):
            raise ImportError(f"{p} is missing: build it with paged_kv_cache_xs_gb300.build.build()")
        lib = ctypes.CDLL(p)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if path is None:
            _lib = lib
        return lib


def _call(name: str, *args) -> int:
    code = getattr(load(), name)(*args)
    if code != 0:
        raise XsError(name, code)
    return code


def dtype_code(dt: torch.dtype) -> int:
    if dt == torch.float32:
        return XS_F32
    if dt == torch.bfloat16:
        return XS_BF16
    raise ValueError(f"unsupported dtype {dt}")


def _ptr(t: torch.Tensor | None) -> int | None:
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to libxs_paged must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


# ---------------------------------------------------------------- entry points

def xs_slot_mapping(block_tables, context_lens, block_size, num_blocks, slot_mapping=None,
                    err_flag=None, stream=None) -> torch.Tensor:
    B = context_lens.numel()
    if slot_mapping is None:
        slot_mapping = torch.empty(B, dtype=torch.int64, device=context_lens.device)
    _call("xs_slot_mapping", _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), B,
          block_size, num_blocks, _ptr(slot_mapping), _ptr(err_flag), _stream(stream))
    return slot_mapping


def xs_kv_append(k_new, v_new, k_cache, v_cache, slot_mapping, err_flag=None, stream=None):
    T, Hkv, D = k_new.shape
    num_blocks, _, bs, _ = k_cache.shape
    _call("xs_kv_append", _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
          _ptr(slot_mapping), T, Hkv, D, bs, num_blocks, dtype_code(k_new.dtype), _ptr(err_flag),
          _stream(stream))


def xs_kv_append_paged(k_new, v_new, k_cache, v_cache, block_tables, context_lens, err_flag=None,
                       stream=None):
    B, Hkv, D = k_new.shape
    num_blocks, _, bs, _ = k_cache.shape
    _call("xs_kv_append_paged", _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
          _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), B, Hkv, D, bs,
          num_blocks, dtype_code(k_new.dtype), _ptr(err_flag), _stream(stream))


def xs_paged_decode_partition_tokens(B, Hkv, total_context_tokens, max_context_len, num_sms) -> int:
    r = load().xs_paged_decode_partition_tokens(B, Hkv, total_context_tokens, max_context_len,
                                                num_sms)
    if r < 0:
        raise XsError("xs_paged_decode_partition_tokens", r)
    return r


def xs_paged_decode_step_partition_tokens(B, Hq, Hkv, total_context_tokens, max_context_len,
                                          num_sms) -> int:
    r = load().xs_paged_decode_step_partition_tokens(B, Hq, Hkv, total_context_tokens,
                                                     max_context_len, num_sms)
    if r < 0:
        raise XsError("xs_paged_decode_step_partition_tokens", r)
    return r


def xs_paged_decode_max_partitions(max_blocks_per_seq, block_size, partition_tokens) -> int:
    r = load().xs_paged_decode_max_partitions(max_blocks_per_seq, block_size, partition_tokens)
    if r < 0:
        raise XsError("xs_paged_decode_max_partitions", r)
    return r


def xs_paged_decode_num_splits(B, Hkv, max_context_len, sm_count) -> int:
    """Partitions (split-K factor) of the longest sequence under the
    library's heuristic; 1 means no split."""
    r = load().xs_paged_decode_num_splits(B, Hkv, max_context_len, sm_count)
    if r < 0:
        raise XsError("xs_paged_decode_num_splits", r)
    return r


def xs_paged_decode_workspace_bytes(B, Hq, D, max_partitions) -> int:
    return int(load().xs_paged_decode_workspace_bytes(B, Hq, D, max_partitions))


def xs_paged_decode_attn(out, part_o, part_m, part_l, q, k_cache, v_cache, block_tables,
                         context_lens, scale, partition_tokens, max_partitions, err_flag=None,
                         work_counters=None, stream=None):
    B, Hq, D = q.shape
    num_blocks, Hkv, bs, _ = k_cache.shape
    _call("xs_paged_decode_attn", _ptr(out), _ptr(part_o), _ptr(part_m), _ptr(part_l), _ptr(q),
          _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.shape[1],
          _ptr(context_lens), B, Hq, Hkv, D, bs, num_blocks, float(scale), partition_tokens,
          max_partitions, dtype_code(q.dtype), _ptr(err_flag), _ptr(work_counters),
          _stream(stream))


def xs_paged_decode_reduce(out, part_o, part_m, part_l, context_lens, partition_tokens,
                           max_partitions, stream=None):
    B, Hq, D = out.shape
    _call("xs_paged_decode_reduce", _ptr(out), _ptr(part_o), _ptr(part_m), _ptr(part_l),
          _ptr(context_lens), B, Hq, D, partition_tokens, max_partitions, dtype_code(out.dtype),
          _stream(stream))


def xs_paged_decode(out, part_o, part_m, part_l, q, k_cache, v_cache, block_tables, context_lens,
                    scale, partition_tokens, max_partitions, err_flag=None, work_counters=None,
                    stream=None):
    B, Hq, D = q.shape
    num_blocks, Hkv, bs, _ = k_cache.shape
    _call("xs_paged_decode", _ptr(out), _ptr(part_o), _ptr(part_m), _ptr(part_l), _ptr(q),
          _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.shape[1],
          _ptr(context_lens), B, Hq, Hkv, D, bs, num_blocks, float(scale), partition_tokens,
          max_partitions, dtype_code(q.dtype), _ptr(err_flag), _ptr(work_counters),
          _stream(stream))


XS_STEP_EARLY_READS = 1
XS_STEP_PERSISTENT = 2
XS_PREFILL_OVERLAP = 1


def xs_paged_decode_step(out, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens,
                         scale, partition_tokens, max_partitions, part_o, part_m, part_l,
                         counters, sinks=None, window=0, err_flag=None, stream=None,
                         early_reads=False, persistent=False):
    """The whole decode step in one launch: append k_new/v_new ([B, Hkv, D],
    or both None), attend, combine the split-K partials.  ``counters`` holds
    xs_paged_decode_step_counters(B, Hkv) int32 zeros (left zero).
    ``early_reads`` (XS_STEP_EARLY_READS): lengths, tables and the first pages
    are read before the previous kernel on the stream completes; the caller
    promises that kernel writes none of them.  ``persistent``
    (XS_STEP_PERSISTENT): the persistent grid even for a launch that would
    run as clusters."""
    B, Hq, D = q.shape
    num_blocks, Hkv, bs, _ = k_cache.shape
    flags = (XS_STEP_EARLY_READS if early_reads else 0) | (XS_STEP_PERSISTENT if persistent else 0)
    if flags:
        _call("xs_paged_decode_step_ex", _ptr(out), _ptr(q), _ptr(k_new), _ptr(v_new),
              _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.shape[1],
              _ptr(context_lens), _ptr(sinks), int(window), B, Hq, Hkv, D, bs, num_blocks,
              float(scale), partition_tokens, max_partitions, _ptr(part_o), _ptr(part_m),
              _ptr(part_l), _ptr(counters), flags, dtype_code(q.dtype),
              _ptr(err_flag), _stream(stream))
        return
    _call("xs_paged_decode_step", _ptr(out), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache),
          _ptr(v_cache), _ptr(block_tables), block_tables.shape[1], _ptr(context_lens),
          _ptr(sinks), int(window), B, Hq, Hkv, D, bs, num_blocks, float(scale),
          partition_tokens, max_partitions, _ptr(part_o), _ptr(part_m), _ptr(part_l),
          _ptr(counters), dtype_code(q.dtype), _ptr(err_flag), _stream(stream))


def xs_paged_prefill_tc(out, q, k_cache, v_cache, block_ids, start_pos, scale, err_flag=None,
                        stream=None, overlap=False):
    """Causal attention of a prefill chunk (q [T, Hq, D]) over the paged
    cache on the tensor cores (bf16); one launch, no workspace.  ``overlap``
    (XS_PREFILL_OVERLAP): q, the block ids and the rows before start_pos are
    read before the previous kernel on the stream completes (it must write
    none of them: e.g. this chunk's append launched with overlap)."""
    T, Hq, D = q.shape
    num_blocks, Hkv, bs, _ = k_cache.shape
    _call("xs_paged_prefill_tc_ex", _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
          _ptr(block_ids), block_ids.numel(), T, int(start_pos), Hq, Hkv, D, bs, num_blocks,
          float(scale), XS_PREFILL_OVERLAP if overlap else 0, dtype_code(q.dtype),
          _ptr(err_flag), _stream(stream))


def xs_paged_decode_step_counters(B: int, Hkv: int) -> int:
    n = load().xs_paged_decode_step_counters(B, Hkv)
    if n < 0:
        raise XsError("xs_paged_decode_step_counters", n)
    return n


def xs_paged_decode_splits(out, part_o, part_m, part_l, q, k_cache, v_cache, block_tables,
                           context_lens, scale, num_splits, err_flag=None, stream=None):
    """The two passes with the split given as a count (xs_paged_decode_attn_splits,
    then xs_paged_decode_reduce_splits); partials sized for num_splits."""
    B, Hq, D = q.shape
    num_blocks, Hkv, bs, _ = k_cache.shape
    mb = block_tables.shape[1]
    _call("xs_paged_decode_attn_splits", _ptr(out), _ptr(part_o), _ptr(part_m), _ptr(part_l),
          _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), mb, _ptr(context_lens), B,
          Hq, Hkv, D, bs, num_blocks, float(scale), int(num_splits), dtype_code(q.dtype),
          _ptr(err_flag), _stream(stream))
    _call("xs_paged_decode_reduce_splits", _ptr(out), _ptr(part_o), _ptr(part_m), _ptr(part_l),
          _ptr(context_lens), mb, B, Hq, D, bs, int(num_splits), dtype_code(q.dtype),
          _stream(stream))


def xs_paged_decode_step_cluster_size(B, Hq, Hkv, D, max_blocks_per_seq, window, dtype) -> int:
    """Cluster size of a one-launch step of this shape on the current device
    (0: the persistent grid).  dtype: a torch dtype or an XS_* code."""
    code = dtype if isinstance(dtype, int) else dtype_code(dtype)
    r = load().xs_paged_decode_step_cluster_size(B, Hq, Hkv, D, max_blocks_per_seq, window, code)
    if r < 0:
        raise XsError("xs_paged_decode_step_cluster_size", r)
    return r


def xs_paged_decode_noalloc(out, q, k_cache, v_cache, block_tables, context_lens, scale,
                            partition_tokens=0, err_flag=None, stream=None):
    """xs_paged_decode without caller-provided partials: for callers that may
    not allocate device memory; the split-K partials live in the library's
    fixed 64 MiB device array (see include/xs_paged.h)."""
    B, Hq, D = q.shape
    num_blocks, Hkv, bs, _ = k_cache.shape
    _call("xs_paged_decode_noalloc", _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
          _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), B, Hq, Hkv, D, bs,
          num_blocks, float(scale), int(partition_tokens), dtype_code(q.dtype), _ptr(err_flag),
          _stream(stream))


def xs_paged_decode_sinks(out, part_o, part_m, part_l, q, k_cache, v_cache, block_tables,
                          context_lens, scale, partition_tokens, max_partitions, sinks=None,
                          window=0, err_flag=None, work_counters=None, stream=None):
    """Decode attention with per-head sinks ([Hq], q's dtype, or None) and a
    sliding window of the last ``window`` tokens (0 = all): attn + reduce."""
    B, Hq, D = q.shape
    num_blocks, Hkv, bs, _ = k_cache.shape
    _call("xs_paged_decode_sinks", _ptr(out), _ptr(part_o), _ptr(part_m), _ptr(part_l), _ptr(q),
          _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.shape[1],
          _ptr(context_lens), _ptr(sinks), int(window), B, Hq, Hkv, D, bs, num_blocks,
          float(scale), partition_tokens, max_partitions, dtype_code(q.dtype), _ptr(err_flag),
          _ptr(work_counters), _stream(stream))


def xs_paged_decode_attn_sinks(out, part_o, part_m, part_l, q, k_cache, v_cache, block_tables,
                               context_lens, scale, partition_tokens, max_partitions, sinks=None,
                               window=0, err_flag=None, work_counters=None, stream=None):
    B, Hq, D = q.shape
    num_blocks, Hkv, bs, _ = k_cache.shape
    _call("xs_paged_decode_attn_sinks", _ptr(out), _ptr(part_o), _ptr(part_m), _ptr(part_l),
          _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.shape[1],
          _ptr(context_lens), _ptr(sinks), int(window), B, Hq, Hkv, D, bs, num_blocks,
          float(scale), partition_tokens, max_partitions, dtype_code(q.dtype), _ptr(err_flag),
          _ptr(work_counters), _stream(stream))


def xs_paged_decode_reduce_sinks(out, part_o, part_m, part_l, context_lens, partition_tokens,
                                 max_partitions, sinks=None, window=0, stream=None):
    B, Hq, D = out.shape
    _call("xs_paged_decode_reduce_sinks", _ptr(out), _ptr(part_o), _ptr(part_m), _ptr(part_l),
          _ptr(context_lens), _ptr(sinks), int(window), B, Hq, D, partition_tokens,
          max_partitions, dtype_code(out.dtype), _stream(stream))


def xs_kv_swap(src_k, src_v, dst_k, dst_v, block_mapping, err_flag=None, stream=None):
    """Copy whole blocks src[s] -> dst[d] for every (s, d) row of the int64
    [n, 2] block_mapping (device or pinned host tensors; see xs_kv_swap)."""
    n = block_mapping.shape[0] if block_mapping.dim() == 2 else block_mapping.numel() // 2
    block_bytes = (src_k[0].numel() if src_k.shape[0] else dst_k[0].numel()) * src_k.element_size()
    _call("xs_kv_swap", src_k.data_ptr(), src_v.data_ptr(), dst_k.data_ptr(), dst_v.data_ptr(),
          _ptr(block_mapping), n, block_bytes, src_k.shape[0], dst_k.shape[0], _ptr(err_flag),
          _stream(stream))


def xs_block_alloc_decode(block_tables, context_lens, free_stack, free_top, block_size=BLOCK_SIZE,
                          err_flag=None, stream=None):
    """Advance every live sequence by one token, popping a block from the
    device free stack for each token that starts a page."""
    _call("xs_block_alloc_decode", _ptr(block_tables), block_tables.shape[1], _ptr(context_lens),
          context_lens.numel(), block_size, _ptr(free_stack), _ptr(free_top), _ptr(err_flag),
          _stream(stream))


def xs_block_free(seq_ids, block_tables, context_lens, free_stack, free_top,
                  block_size=BLOCK_SIZE, err_flag=None, stream=None):
    """Release the slots in seq_ids (device int32): their blocks go back on
    the free stack, their rows and lengths become -1."""
    _call("xs_block_free", _ptr(seq_ids), seq_ids.numel(), _ptr(block_tables),
          block_tables.shape[1], _ptr(context_lens), context_lens.numel(), block_size,
          _ptr(free_stack), _ptr(free_top), free_stack.numel(), _ptr(err_flag), _stream(stream))


def xs_prefill_append(k_src, v_src, k_cache, v_cache, block_ids, start_pos, err_flag=None,
                      stream=None, overlap=False):
    """Write a [Hkv, T, D] chunk at positions start_pos .. of one sequence.
    ``overlap`` (XS_PREFILL_OVERLAP): the launch does not wait for the
    previous kernel on the stream (which must write none of its inputs and
    touch none of these rows: e.g. the previous chunk's attention)."""
    Hkv, T, D = k_src.shape
    num_blocks, _, bs, _ = k_cache.shape
    _call("xs_prefill_append_ex", _ptr(k_src), _ptr(v_src), _ptr(k_cache), _ptr(v_cache),
          _ptr(block_ids), block_ids.numel(), T, Hkv, D, bs, num_blocks, int(start_pos),
          XS_PREFILL_OVERLAP if overlap else 0, dtype_code(k_src.dtype), _ptr(err_flag),
          _stream(stream))


def xs_paged_prefill(out, part_o, part_m, part_l, q, k_cache, v_cache, block_ids, start_pos,
                     scale, partition_tokens, max_partitions, err_flag=None, work_counters=None,
                     stream=None):
    """Causal attention of the chunk q [T, Hq, D] at start_pos over the pages."""
    T, Hq, D = q.shape
    num_blocks, Hkv, bs, _ = k_cache.shape
    _call("xs_paged_prefill", _ptr(out), _ptr(part_o), _ptr(part_m), _ptr(part_l), _ptr(q),
          _ptr(k_cache), _ptr(v_cache), _ptr(block_ids), block_ids.numel(), T, int(start_pos), Hq,
          Hkv, D, bs, num_blocks, float(scale), partition_tokens, max_partitions,
          dtype_code(q.dtype), _ptr(err_flag), _ptr(work_counters), _stream(stream))


def xs_version() -> int:
    return load().xs_version()


def xs_debug_bounds_failures(reset: bool = False, lib=None) -> int:
    """Failed in-kernel bounds checks on the current device (debug library
    only; the release library returns XS_EUNSUPPORTED)."""
    return (lib or load()).xs_debug_bounds_failures(int(bool(reset)))


def xs_debug_wait_injection(wait_limit_ns: int, skip_page: int = -1, lib=None) -> None:
    """Debug library only: set the decode kernel's wait limit and make CTA
    0's producer skip issuing one page (-1: none); see the header."""
    lib = lib or load()
    code = lib.xs_debug_wait_injection(int(wait_limit_ns), int(skip_page))
    if code != 0:
        raise XsError("xs_debug_wait_injection", code)


def load_debug():
    """The debug library (in-kernel bounds checks), as a separate handle: the
    release library stays the one the wrappers above use unless a caller
    installs this one with use_library()."""
    return load(_build.DEBUG_LIB_PATH)


def use_library(lib):
    """Make `lib` (e.g. load_debug()) the library every wrapper calls; returns
    the previous one (None if none was loaded yet)."""
    global _lib
    with _lock:
        prev, _lib = _lib, lib
    return prev


# ---------------------------------------------------------------- workspace holder

class DecodeWorkspace:
    """Split-K partials sized for a batch shape, allocated once through PyTorch.

    ``partition_tokens`` comes from the library's heuristic unless given: the
    one for the one-launch step (``fused``, the default) or the one for the
    separate attention + combine calls."""

    def __init__(self, B: int, Hq: int, Hkv: int, D: int, max_blocks_per_seq: int,
                 device, total_context_tokens: int = 0, max_context_len: int | None = None,
                 partition_tokens: int | None = None, num_sms: int | None = None,
                 fused: bool = True):
        device = torch.device(device)
        if num_sms is None:
            num_sms = torch.cuda.get_device_properties(device).multi_processor_count
        if max_context_len is None:
            max_context_len = max_blocks_per_seq * BLOCK_SIZE
        if partition_tokens:
            self.partition_tokens = partition_tokens
        elif fused:
            self.partition_tokens = xs_paged_decode_step_partition_tokens(
                B, Hq, Hkv, total_context_tokens, max_context_len, num_sms)
        else:
            self.partition_tokens = xs_paged_decode_partition_tokens(
                B, Hkv, total_context_tokens, max_context_len, num_sms)
        self.max_partitions = xs_paged_decode_max_partitions(max_blocks_per_seq, BLOCK_SIZE,
                                                             self.partition_tokens)
        n = B * Hq * self.max_partitions
        # Counters, zero between launches: the dynamic item scheduler's two,
        # then the fused step's per-(sequence, KV head) combine counts.  The
        # separate attention calls use the first two.
        self.work = torch.zeros(xs_paged_decode_step_counters(B, Hkv), dtype=torch.int32,
                                device=device)
        if self.max_partitions > 1:
            self.part_o = torch.empty(n * D, dtype=torch.float32, device=device)
            self.part_m = torch.empty(n, dtype=torch.float32, device=device)
            self.part_l = torch.empty(n, dtype=torch.float32, device=device)
        else:
            self.part_o = self.part_m = self.part_l = None

    @property
    def partial_bytes(self) -> int:
        if self.part_o is None:
            return 0
        return 4 * (self.part_o.numel() + self.part_m.numel() + self.part_l.numel())
