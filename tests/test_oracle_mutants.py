"""Plant plausible mistakes in a copy of the oracle source and check that the
pin suite catches every one.  The mutants are built in a temporary directory;
the committed oracle source is never modified."""
import os
import tempfile

import pytest

import oracle
from tests import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "paged_oracle.c")

# (name, text to replace, replacement): each is a single plausible bug.
MUTANTS = [
    ("gqa_map_modulo", "int g = h / group;", "int g = h % Hkv;"),
    ("scale_dropped", "logit[t] = scale * dot;", "logit[t] = dot;"),
    ("last_token_dropped_qk", "for (int32_t t = 0; t < n; ++t) {\n            int64_t blk",
     "for (int32_t t = 0; t < n - 1; ++t) {\n            int64_t blk"),
    ("page_index_swapped", "int64_t kbase = ((blk * Hkv + g) * block_size + t % block_size) * D;",
     "int64_t kbase = ((blk * Hkv + g) * block_size + t / block_size % block_size) * D;"),
    ("layout_head_block_swapped", "int64_t vbase = ((blk * Hkv + g) * block_size + t % block_size) * D;",
     "int64_t vbase = ((g * num_blocks + blk) * block_size + t % block_size) * D;"),
    ("no_max_subtraction", "double w = exp(logit[t] - mx);", "double w = exp(logit[t]);"),
    ("no_normalisation", "for (int d = 0; d < D; ++d) o[d] /= den;", ""),
    ("v_read_from_k", "o[d] += w * widen(v_cache, vbase + d, dtype);",
     "o[d] += w * widen(k_cache, vbase + d, dtype);"),
    ("bf16_widen_shift", "<< 16;", "<< 15;"),
    ("slot_position_off_by_one", "int64_t p = (int64_t)n - 1;", "int64_t p = (int64_t)n;"),
    ("append_rows_swapped", "memcpy((char *)v_cache + dst, (const char *)v_new + src, row);",
     "memcpy((char *)v_cache + dst, (const char *)k_new + src, row);"),
    ("append_offset_in_block", "int64_t blk = s / block_size, off = s % block_size;",
     "int64_t blk = s / block_size, off = 0;"),
    ("q_head_index", "const int64_t qbase = bh * D;", "const int64_t qbase = (int64_t)b * D;"),
    ("swap_k_into_v", "memcpy((char *)dst_v + d * block_bytes, (const char *)src_v + s * block_bytes,",
     "memcpy((char *)dst_v + d * block_bytes, (const char *)src_k + s * block_bytes,"),
    # (every mutant must keep its accesses in bounds: it runs inside the test process)
    ("swap_dst_stride", "memcpy((char *)dst_k + d * block_bytes, (const char *)src_k + s * block_bytes,",
     "memcpy((char *)dst_k + d * (block_bytes / 2), (const char *)src_k + s * block_bytes,"),
    ("alloc_every_token", "if (p % block_size == 0) {\n            if (*free_top == 0) {",
     "if (p % block_size >= 0) {\n            if (*free_top == 0) {"),
    ("alloc_wrong_page", "block_tables[(int64_t)b * max_blocks_per_seq + page] = free_stack[*free_top];",
     "block_tables[(int64_t)b * max_blocks_per_seq + (page > 0 ? page - 1 : 0)] = free_stack[*free_top];"),
    ("alloc_length_not_advanced", "context_lens[b] = p + 1;", "context_lens[b] = p;"),
    ("free_keeps_last_page", "for (int32_t pg = 0; pg < pages; ++pg) {\n            if (*free_top",
     "for (int32_t pg = 0; pg + 1 < pages; ++pg) {\n            if (*free_top"),
    ("prefill_causal_open", "for (int64_t t = 0; t <= last; ++t) {\n            int64_t blk = block_ids[t / block_size];\n            int64_t kr",
     "for (int64_t t = 0; t < last; ++t) {\n            int64_t blk = block_ids[t / block_size];\n            int64_t kr"),
    ("prefill_no_offset", "int64_t last = (int64_t)start_pos + i;", "int64_t last = i;"),
    ("prefill_src_token_major", "size_t src = (size_t)(((int64_t)h * T + i) * D) * eb;",
     "size_t src = (size_t)(((int64_t)i * Hkv + h) * D) * eb;"),
    ("sink_dropped", "double den = sinks ? exp(sink - top) : 0.0;", "double den = 0.0;"),
    ("sink_scaled", "sink = widen(sinks, h, dtype);", "sink = scale * widen(sinks, h, dtype);"),
    ("window_one_short", "(window > 0 && n > window) ? n - window : 0;",
     "(window > 0 && n > window) ? n - window + 1 : 0;"),
    ("window_one_long", "(window > 0 && n > window) ? n - window : 0;",
     "(window > 0 && n > window) ? n - window - 1 : 0;"),
]


def _build_mutant(name, old, new, workdir):
    text = open(SRC).read()
    assert text.count(old) >= 1, f"mutation anchor for {name} not found"
    path = os.path.join(workdir, f"{name}.c")
    with open(path, "w") as f:
        f.write(text.replace(old, new))
    return oracle.load(oracle.build(force=True, src=path, out=os.path.join(workdir, f"lib{name}.so")))


@pytest.mark.parametrize("mutant", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(mutant):
    name, old, new = mutant
    with tempfile.TemporaryDirectory() as d:
        lib = _build_mutant(name, old, new, d)
        caught = []
        for pin in oracle_pins.ALL_PINS:
            try:
                pin(lib)
            except Exception:          # an assertion, or an oracle error status
                caught.append(pin.__name__)
        assert caught, f"mutant {name} passed every pin"
