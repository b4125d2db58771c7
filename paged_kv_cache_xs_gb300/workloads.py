"""Seeded synthetic decode-step inputs.

This module only draws inputs: sequence lengths, a paged block allocation in a
shuffled physical order, pools, queries and the new K/V rows.  It holds none
of the decode step's arithmetic (slot resolution, append, attention, reduce),
so both the CUDA path and the CPU oracle can take their inputs from it.

Shapes follow the xserv pages ("xserv compare phase10...cf1e9e4",
crates/xserv-kernels/src/attention.rs, ``paged_decode_attention``):

* pools ``k_cache``/``v_cache``: ``[layers, num_blocks, Hkv, block_size, D]``
  (each layer's slice is one ``[num_blocks, Hkv, block_size, D]`` pool);
* ``block_tables``: int32 ``[B, max_blocks_per_seq]``, entries past a
  sequence's last page are ``-1`` (never read);
* ``context_lens``: int32 ``[B]`` = history length + 1 (the token this step
  writes is counted, as ``kv_lens`` in ``reshape_and_cache_batched_bf16``);
* ``q``: ``[layers, B, Hq, D]``; ``k_new``/``v_new``: ``[layers, B, Hkv, D]``.

Lengths and the block allocation come from a CPU generator seeded with
``seed``; values come from a generator on ``device`` seeded with ``seed + 1``,
so a workload is reproducible on a given device type.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

BLOCK_SIZE = 16


@dataclass(frozen=True)
class DecodeConfig:
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    dtype: torch.dtype
    layers: int
    history: str            # "fixed", "uniform", "loguniform"
    history_args: tuple
    pool: str                # "fixed", "needed", "factor", "at_least"
    pool_arg: float
    values: str              # "uniform", "normal", "normal_v_half"
    seed: int
    block_size: int = BLOCK_SIZE
    description: str = ""


# The five decode-step workloads.  History lengths are the cached tokens
# before the step; each step appends one token, so attention covers
# history + 1 tokens.
CONFIGS: list[DecodeConfig] = [
    DecodeConfig("tiny_fp32_mha", 2, 12, 12, 64, torch.float32, 1, "fixed", (7, 20),
                 "fixed", 8, "uniform", 1000,
                 description="2 seqs (history 7, 20), 12 heads x 64, fp32, 8-block pool"),
    DecodeConfig("gpt2_bf16_12layer", 8, 12, 12, 64, torch.bfloat16, 12, "uniform", (32, 1024),
                 "needed", 1, "normal", 1001,
                 description="8 seqs, history U[32,1024], 12 heads x 64, bf16, 12 layers"),
    DecodeConfig("qwen3_8b_single_stream", 1, 32, 8, 128, torch.bfloat16, 36, "fixed", (4096,),
                 "needed", 1, "normal_v_half", 1002,
                 description="1 seq, history 4096, 32q/8kv x 128, bf16, 36 layers"),
    DecodeConfig("qwen3_8b_cb_mix", 64, 32, 8, 128, torch.bfloat16, 1, "loguniform", (16, 8192),
                 "factor", 2, "normal", 1003,
                 description="64 seqs, history log-uniform [16,8192], 32q/8kv x 128, bf16, pool 2x"),
    DecodeConfig("qwen3_8b_long_batch", 128, 32, 8, 128, torch.bfloat16, 1, "uniform", (4096, 32768),
                 "at_least", 128 * 2048, "normal", 1004,
                 description="128 seqs, history U[4096,32768], 32q/8kv x 128, bf16, ~17 GB pool"),
]


@dataclass
class DecodeWorkload:
    cfg: DecodeConfig
    history_lens: torch.Tensor        # int32 [B], CPU
    context_lens: torch.Tensor        # int32 [B] on device
    block_tables: torch.Tensor        # int32 [B, max_blocks_per_seq] on device
    num_blocks: int
    k_cache: torch.Tensor             # [layers, num_blocks, Hkv, bs, D]
    v_cache: torch.Tensor
    q: torch.Tensor                   # [layers, B, Hq, D]
    k_new: torch.Tensor               # [layers, B, Hkv, D]
    v_new: torch.Tensor
    scale: float
    extra: dict = field(default_factory=dict)

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max().item()) if self.context_lens.numel() else 0

    @property
    def total_context_tokens(self) -> int:
        return int(self.history_lens.to(torch.int64).sum().item()) + self.cfg.B


def draw_history(cfg: DecodeConfig, gen: torch.Generator) -> torch.Tensor:
    """int32 [B] history lengths for a config (CPU generator)."""
    if cfg.history == "fixed":
        vals = list(cfg.history_args)
        if len(vals) == 1:
            vals = vals * cfg.B
        assert len(vals) == cfg.B
        return torch.tensor(vals, dtype=torch.int32)
    lo, hi = cfg.history_args
    if cfg.history == "uniform":
        return torch.randint(lo, hi + 1, (cfg.B,), generator=gen, dtype=torch.int64).to(torch.int32)
    if cfg.history == "loguniform":
        u = torch.rand(cfg.B, generator=gen, dtype=torch.float64)
        vals = torch.floor(torch.exp(math.log(lo) + u * (math.log(hi + 1) - math.log(lo))))
        return vals.clamp(lo, hi).to(torch.int32)
    raise ValueError(cfg.history)


def allocate_blocks(context_lens: torch.Tensor, block_size: int, pool: str, pool_arg: float,
                    gen: torch.Generator, max_blocks_per_seq: int | None = None):
    """Paged allocation: give each sequence the pages its tokens occupy, taken
    from a seeded permutation of the pool's physical blocks.

    Returns (block_tables int32 [B, width] with -1 padding, num_blocks)."""
    pages = [(int(n) + block_size - 1) // block_size for n in context_lens.tolist()]
    needed = sum(pages)
    if pool == "fixed":
        num_blocks = int(pool_arg)
    elif pool == "needed":
        num_blocks = needed
    elif pool == "factor":
        num_blocks = int(math.ceil(needed * pool_arg))
    elif pool == "at_least":
        num_blocks = max(int(pool_arg), needed)
    else:
        raise ValueError(pool)
    if needed > num_blocks:
        raise ValueError(f"pool of {num_blocks} blocks cannot hold {needed} pages")
    width = max(pages + [1]) if max_blocks_per_seq is None else max_blocks_per_seq
    perm = torch.randperm(num_blocks, generator=gen).to(torch.int32)
    bt = torch.full((len(pages), width), -1, dtype=torch.int32)
    pos = 0
    for b, p in enumerate(pages):
        bt[b, :p] = perm[pos:pos + p]
        pos += p
    return bt, num_blocks


def _values(shape, kind: str, role: str, dtype, gen, device):
    if kind == "uniform":
        x = torch.rand(shape, generator=gen, device=device, dtype=torch.float32) * 2 - 1
    elif kind in ("normal", "normal_v_half"):
        std = 0.5 if (kind == "normal_v_half" and role == "v") else 1.0
        x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
    else:
        raise ValueError(kind)
    return x.to(dtype)


def _fill_values(t: torch.Tensor, kind: str, role: str, gen, chunk_elems: int = 1 << 28):
    """Fill a (possibly huge) tensor in chunks so the fp32 temporary stays small."""
    flat = t.view(-1)
    for s in range(0, flat.numel(), chunk_elems):
        e = min(flat.numel(), s + chunk_elems)
        flat[s:e] = _values((e - s,), kind, role, t.dtype, gen, t.device)


def make_workload(cfg: DecodeConfig | int, device="cpu", seed: int | None = None,
                  layers: int | None = None, history: torch.Tensor | None = None,
                  pool_fill: str | None = None) -> DecodeWorkload:
    """Draw one decode-step workload.

    cfg: a DecodeConfig or an index into CONFIGS.  ``layers`` overrides the
    number of distinct per-layer pools; ``history`` overrides the drawn
    history lengths.  ``pool_fill='canary'`` fills every pool element with a
    fixed bit pattern before the used pages are drawn, so untouched slots are
    recognisable."""
    if isinstance(cfg, int):
        cfg = CONFIGS[cfg]
    device = torch.device(device)
    seed = cfg.seed if seed is None else seed
    L = cfg.layers if layers is None else layers
    cpu_gen = torch.Generator().manual_seed(seed)
    hist = draw_history(cfg, cpu_gen) if history is None else history.to(torch.int32).cpu()
    ctx = hist + 1
    bt, num_blocks = allocate_blocks(ctx, cfg.block_size, cfg.pool, cfg.pool_arg, cpu_gen)
    dev_gen = torch.Generator(device=device).manual_seed(seed + 1)
    pool_shape = (L, num_blocks, cfg.Hkv, cfg.block_size, cfg.D)
    k_cache = torch.empty(pool_shape, dtype=cfg.dtype, device=device)
    v_cache = torch.empty(pool_shape, dtype=cfg.dtype, device=device)
    if pool_fill == "canary":
        pattern = 0x5A5A if cfg.dtype == torch.bfloat16 else 0x5A5A5A5A
        itype = torch.int16 if cfg.dtype == torch.bfloat16 else torch.int32
        k_cache.view(itype).fill_(pattern)
        v_cache.view(itype).fill_(pattern)
        # Only the used pages get values.
        for b in range(cfg.B):
            pages = bt[b][bt[b] >= 0].to(torch.int64).to(device)
            for layer in range(L):
                shp = (pages.numel(), cfg.Hkv, cfg.block_size, cfg.D)
                k_cache[layer].index_copy_(0, pages, _values(shp, cfg.values, "k", cfg.dtype, dev_gen, device))
                v_cache[layer].index_copy_(0, pages, _values(shp, cfg.values, "v", cfg.dtype, dev_gen, device))
    else:
        _fill_values(k_cache, cfg.values, "k", dev_gen)
        _fill_values(v_cache, cfg.values, "v", dev_gen)
    q = _values((L, cfg.B, cfg.Hq, cfg.D), cfg.values, "q", cfg.dtype, dev_gen, device)
    k_new = _values((L, cfg.B, cfg.Hkv, cfg.D), cfg.values, "k", cfg.dtype, dev_gen, device)
    v_new = _values((L, cfg.B, cfg.Hkv, cfg.D), cfg.values, "v", cfg.dtype, dev_gen, device)
    return DecodeWorkload(cfg=cfg, history_lens=hist, context_lens=ctx.to(device),
                          block_tables=bt.to(device), num_blocks=num_blocks,
                          k_cache=k_cache, v_cache=v_cache, q=q, k_new=k_new, v_new=v_new,
                          scale=1.0 / math.sqrt(cfg.D))


def custom_config(B: int, Hq: int, Hkv: int, D: int, dtype=torch.bfloat16, layers: int = 1,
                  history=("uniform", (1, 300)), pool=("factor", 1.5), values="normal",
                  seed: int = 7, name: str = "custom") -> DecodeConfig:
    kind, args = history
    return DecodeConfig(name, B, Hq, Hkv, D, dtype, layers, kind, tuple(args), pool[0], pool[1],
                        values, seed)
