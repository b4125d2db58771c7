"""One continuous-batching decode step over a paged KV cache.

``PagedDecodeStep`` owns nothing but the split-K workspace; the KV pools,
block tables and lengths belong to the caller.  A step is

1. slot resolution + KV append (the pages' reshape_and_cache_batched_bf16,
   "xserv compare phase10...cf1e9e4", attention.rs);
2. paged decode attention over split-K partitions;
3. the split-K combine (only when a sequence can span several partitions).

``run`` enqueues all three as one launch (``xs_paged_decode_step``);
``run_unfused`` enqueues them as the separate calls ``xs_kv_append_paged``,
``xs_paged_decode_attn`` and ``xs_paged_decode_reduce`` (``append``,
``attend`` and ``reduce`` below).

``run_from_host`` is the same step fed from pinned host buffers: it copies
the step's inputs to the device, runs the step and copies the output back.
"""
from __future__ import annotations

import torch

from . import ops


class PagedDecodeStep:
    """sinks ([Hq] tensor of q's dtype, or None) and window (0 = all tokens)
    select the gpt-oss variant: per-head sink logits and a sliding window.
    ``fused`` picks the partition heuristic for ``run`` (True) or for
    ``run_unfused`` (False); both forms work with either."""

    def __init__(self, B: int, Hq: int, Hkv: int, D: int, max_blocks_per_seq: int, dtype,
                 device, total_context_tokens: int = 0, max_context_len: int | None = None,
                 partition_tokens: int | None = None, sinks=None, window: int = 0,
                 fused: bool = True):
        self.B, self.Hq, self.Hkv, self.D = B, Hq, Hkv, D
        self.sinks, self.window = sinks, int(window)
        self.dtype = dtype
        self.device = torch.device(device)
        self.max_blocks_per_seq = max_blocks_per_seq
        self.ws = ops.DecodeWorkspace(B, Hq, Hkv, D, max_blocks_per_seq, self.device,
                                      total_context_tokens=total_context_tokens,
                                      max_context_len=max_context_len,
                                      partition_tokens=partition_tokens, fused=fused)
        self.err_flag = torch.zeros(1, dtype=torch.int32, device=self.device)
        self._dev_inputs = None

    @property
    def partition_tokens(self) -> int:
        return self.ws.partition_tokens

    @property
    def max_partitions(self) -> int:
        return self.ws.max_partitions

    def cluster_size(self, fused: bool = True) -> int:
        """Cluster size the one-launch step runs with on the current device
        (0: the persistent grid, whose split is partition_tokens)."""
        if not fused:
            return 0
        return ops.xs_paged_decode_step_cluster_size(self.B, self.Hq, self.Hkv, self.D,
                                                     self.max_blocks_per_seq, self.window,
                                                     self.dtype)

    def launches_per_step(self, fused: bool = True) -> int:
        if fused:
            return 1
        return 3 if self.ws.max_partitions > 1 else 2

    def append(self, k_new, v_new, k_cache, v_cache, block_tables, context_lens):
        ops.xs_kv_append_paged(k_new, v_new, k_cache, v_cache, block_tables, context_lens,
                               err_flag=self.err_flag)

    def attend(self, out, q, k_cache, v_cache, block_tables, context_lens, scale):
        ws = self.ws
        if self.sinks is None and self.window == 0:
            ops.xs_paged_decode_attn(out, ws.part_o, ws.part_m, ws.part_l, q, k_cache, v_cache,
                                     block_tables, context_lens, scale, ws.partition_tokens,
                                     ws.max_partitions, err_flag=self.err_flag,
                                     work_counters=ws.work)
        else:
            ops.xs_paged_decode_attn_sinks(out, ws.part_o, ws.part_m, ws.part_l, q, k_cache,
                                           v_cache, block_tables, context_lens, scale,
                                           ws.partition_tokens, ws.max_partitions,
                                           sinks=self.sinks, window=self.window,
                                           err_flag=self.err_flag, work_counters=ws.work)

    def reduce(self, out, context_lens):
        ws = self.ws
        if ws.max_partitions <= 1:
            return
        if self.sinks is None and self.window == 0:
            ops.xs_paged_decode_reduce(out, ws.part_o, ws.part_m, ws.part_l, context_lens,
                                       ws.partition_tokens, ws.max_partitions)
        else:
            ops.xs_paged_decode_reduce_sinks(out, ws.part_o, ws.part_m, ws.part_l, context_lens,
                                             ws.partition_tokens, ws.max_partitions,
                                             sinks=self.sinks, window=self.window)

    def run(self, out, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, scale,
            early_reads: bool = False, persistent: bool = False):
        """Append this step's K/V, attend and combine in one launch; all
        tensors on the device.  ``early_reads``: the launch reads lengths,
        tables and its first pages before the previous kernel on the stream
        completes (that kernel must write none of them: e.g. another layer's
        step, or a projection).  ``persistent``: the persistent grid even
        where the launch would run as clusters."""
        ws = self.ws
        ops.xs_paged_decode_step(out, q, k_new, v_new, k_cache, v_cache, block_tables,
                                 context_lens, scale, ws.partition_tokens, ws.max_partitions,
                                 ws.part_o, ws.part_m, ws.part_l, ws.work, sinks=self.sinks,
                                 window=self.window, err_flag=self.err_flag,
                                 early_reads=early_reads, persistent=persistent)
        return out

    def run_unfused(self, out, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens,
                    scale):
        """The same step as three launches: append, attention, combine."""
        self.append(k_new, v_new, k_cache, v_cache, block_tables, context_lens)
        self.attend(out, q, k_cache, v_cache, block_tables, context_lens, scale)
        self.reduce(out, context_lens)
        return out

    def run_from_host(self, out_host, q, k_new, v_new, block_tables, context_lens, k_cache,
                      v_cache, scale):
        """Step fed from (pinned) host tensors q, k_new, v_new, block_tables and
        context_lens; the pools stay on the device.  Writes out_host and waits
        for it."""
        if self._dev_inputs is None or self._dev_inputs[0].shape != q.shape \
                or self._dev_inputs[3].shape != block_tables.shape:
            self._dev_inputs = tuple(torch.empty(t.shape, dtype=t.dtype, device=self.device)
                                     for t in (q, k_new, v_new, block_tables, context_lens))
            self._dev_out = torch.empty(q.shape, dtype=q.dtype, device=self.device)
        dq, dk, dv, dbt, dcl = self._dev_inputs
        for d, h in zip(self._dev_inputs, (q, k_new, v_new, block_tables, context_lens)):
            d.copy_(h, non_blocking=True)
        self.run(self._dev_out, dq, dk, dv, k_cache, v_cache, dbt, dcl, scale)
        out_host.copy_(self._dev_out, non_blocking=True)
        torch.cuda.current_stream().synchronize()
        return out_host

    def error_flags(self) -> int:
        return int(self.err_flag.item())


class CapturedStep:
    """A decode step (any sequence of library calls, e.g. every layer's
    append + attention + reduce) captured once into a CUDA graph and
    replayed.

    Every kernel of the path reads its per-step data (lengths, block tables,
    q, the new K/V rows) from device memory and takes only fixed sizes from
    the host, so a replay sees whatever the caller has written into the same
    buffers since the last one.  The split-K work counters reset themselves
    at the end of every launch, so replays need no host action."""

    def __init__(self, fn, warmup: int = 1):
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for _ in range(warmup):  # fills the library's per-kernel caches
                fn()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            fn()

    def replay(self):
        self.graph.replay()
