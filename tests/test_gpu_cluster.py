"""The one-launch decode step run as thread-block clusters: one cluster per
(sequence, KV head), CTA r attending over partition r of the group's tokens,
the split-K partials combined over distributed shared memory
(paged_decode_cluster_kernel).  Which launches take it, and parity with the
oracle - the appended rows bit-exact, the attention within the bf16 bound -
on the single-stream shape, ragged small batches with empty and unset
sequences, partitions that fill their 24 pages exactly, sinks and windows,
bad lengths and block ids, and back-to-back layers with early reads inside a
CUDA graph; on the same inputs the persistent grid agrees."""
import pytest
import torch

import oracle
from paged_kv_cache_xs_gb300 import ops
from paged_kv_cache_xs_gb300 import workloads as wl
from paged_kv_cache_xs_gb300.step import CapturedStep
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu


def _cluster_size(w, window=0):
    cfg = w.cfg
    return ops.xs_paged_decode_step_cluster_size(cfg.B, cfg.Hq, cfg.Hkv, cfg.D,
                                                 w.max_blocks_per_seq, window, cfg.dtype)


def _ws(w, P=256):
    cfg = w.cfg
    return ops.DecodeWorkspace(cfg.B, cfg.Hq, cfg.Hkv, cfg.D, w.max_blocks_per_seq, w.q.device,
                               partition_tokens=P)


def _step(w, ws, sinks=None, window=0, out=None, err=None, early=False, layer=0,
          persistent=False):
    cfg = w.cfg
    dev = w.q.device
    out = torch.full((cfg.B, cfg.Hq, cfg.D), float("nan"), dtype=cfg.dtype, device=dev) \
        if out is None else out
    err = torch.zeros(1, dtype=torch.int32, device=dev) if err is None else err
    ops.xs_paged_decode_step(out, w.q[layer], w.k_new[layer], w.v_new[layer], w.k_cache[layer],
                             w.v_cache[layer], w.block_tables, w.context_lens, w.scale,
                             ws.partition_tokens, ws.max_partitions, ws.part_o, ws.part_m,
                             ws.part_l, ws.work, sinks=sinks, window=window, err_flag=err,
                             early_reads=early, persistent=persistent)
    return out, err


def _appended(w, layer=0):
    slots = oracle.slot_mapping(w.block_tables.cpu(), w.context_lens.cpu(), gh.BS, w.num_blocks)
    return oracle.kv_append(w.k_new[layer].cpu(), w.v_new[layer].cpu(), w.k_cache[layer].cpu(),
                            w.v_cache[layer].cpu(), slots)


def _check(w, out, err, ek, ev, ws=None, sinks=None, window=0, layer=0, what=""):
    """Flags clear, counters untouched, pools equal to the oracle's append,
    attention within the bf16 bound of the oracle."""
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"{what}: device error flag {int(err.item())}"
    if ws is not None:
        assert int(ws.work.count_nonzero()) == 0
    assert torch.equal(gh.int_view(w.k_cache[layer].cpu()), gh.int_view(ek)), what
    assert torch.equal(gh.int_view(w.v_cache[layer].cpu()), gh.int_view(ev)), what
    ref = oracle.paged_decode_sinks(w.q[layer].cpu(), ek, ev, w.block_tables.cpu(),
                                    w.context_lens.cpu(), w.scale,
                                    sinks=None if sinks is None else sinks.cpu(), window=window)
    return gh.assert_close(out, ref, w.cfg.dtype, what=what)


def test_which_launches_run_as_clusters():
    gh.device()
    bf16, f32 = torch.bfloat16, torch.float32
    size = ops.xs_paged_decode_step_cluster_size
    # One group (one sequence, one KV head): a single cluster of up to 16.
    # 49152 tokens split 16 ways is 192 pages a CTA, the most it takes;
    # 49168 tokens would be 193.
    assert size(1, 4, 1, 128, 384, 0, bf16) == 16
    assert size(1, 4, 1, 128, 3072, 0, bf16) == 16
    assert size(1, 4, 1, 128, 3073, 0, bf16) == 0
    # A window bounds the tokens: 4096 of a 16000-token table (17 pages a CTA).
    assert size(1, 4, 1, 128, 1000, 4096, bf16) == 16
    # No more than one CTA per 64 tokens.
    assert size(1, 4, 1, 128, 8, 0, bf16) == 2
    assert size(1, 4, 1, 128, 4, 0, bf16) == 0
    assert size(1, 4, 1, 128, 1000, 64, bf16) == 0
    # Eight KV heads of one 4097-token sequence: eight clusters, a little
    # smaller than the largest eight of which fit at once, so that a slot is
    # left for the next launch; more groups, smaller clusters.
    single = size(1, 32, 8, 128, 257, 0, bf16)
    assert 8 <= single <= 16
    assert 2 <= size(4, 32, 8, 128, 63, 0, bf16) <= single
    # D = 64 runs two CTAs per SM: the GPT-2 shape (8 sequences, 12 heads)
    # fits where D = 128 would not.
    assert size(8, 12, 12, 64, 65, 0, bf16) >= 2
    assert size(8, 12, 12, 128, 65, 0, bf16) == 0
    # Not for fp32, no batch, or batches whose clusters do not fit at once.
    assert size(1, 32, 8, 128, 257, 0, f32) == 0
    assert size(64, 32, 8, 128, 257, 0, bf16) == 0
    assert size(0, 32, 8, 128, 257, 0, bf16) == 0


@pytest.mark.parametrize("early", [False, True])
def test_single_stream_matches_oracle(early):
    dev = gh.device()
    w = wl.make_workload(2, device=dev, layers=1)  # 1 sequence, 4096 + 1 tokens, 32q/8kv x 128
    assert _cluster_size(w) >= 8
    ek, ev = _appended(w)
    out, err = _step(w, _ws(w), early=early)
    err_oracle = _check(w, out, err, ek, ev, what=f"early={early}")
    assert err_oracle <= gh.TOL[torch.bfloat16]


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_ragged_small_batch(G, D):
    # Lengths around pages and partitions, an empty sequence and an unset
    # slot (length 0 after the append of nothing: history -1).
    dev = gh.device()
    hist = torch.tensor([0, 1, 14, 15, 16, 17, 255, 256, 257, 1000, -1], dtype=torch.int32)
    cfg = wl.custom_config(len(hist), 2 * G, 2, D, torch.bfloat16, history=("uniform", (0, 1)),
                           pool=("factor", 1.5), seed=900 + G + D)
    w = wl.make_workload(cfg, device=dev, history=hist)
    assert _cluster_size(w) > 0
    ek, ev = _appended(w)
    ws = _ws(w, 64)
    out, err = _step(w, ws)
    _check(w, out, err, ek, ev, ws, what=f"G={G} D={D}")


@pytest.mark.parametrize("early", [False, True])
def test_gpt2_shape(early):
    # The GPT-2 workload's layer (8 sequences, 12 heads x 64, MHA): clusters
    # of two CTAs per SM.
    dev = gh.device()
    w = wl.make_workload(1, device=dev, layers=1)
    assert _cluster_size(w) >= 2
    ek, ev = _appended(w)
    out, err = _step(w, _ws(w), early=early)
    _check(w, out, err, ek, ev, what=f"early={early}")


@pytest.mark.parametrize("G", [4, 8])
@pytest.mark.parametrize("hist", [6143, 6143 - 384, 5000, 0])
def test_full_and_empty_partitions(hist, G):
    # One KV head, a 384-block table split 16 ways: 24 pages a CTA, one lap
    # of the ring.  6144 tokens fill every page of every partition; 5760
    # leave the last partition empty; one token leaves fifteen of them empty.
    dev = gh.device()
    cfg = wl.custom_config(1, G, 1, 128, torch.bfloat16, history=("uniform", (0, 1)),
                           pool=("factor", 1.2), seed=910 + G)
    w = wl.make_workload(cfg, device=dev, history=torch.tensor([hist], dtype=torch.int32))
    if w.max_blocks_per_seq < 384:  # the same table width for every case
        bt = torch.full((1, 384), -1, dtype=torch.int32, device=dev)
        bt[:, :w.max_blocks_per_seq] = w.block_tables
        w.block_tables = bt
    assert _cluster_size(w) == 16
    ek, ev = _appended(w)
    out, err = _step(w, _ws(w))
    _check(w, out, err, ek, ev, what=f"history {hist} G={G}")


@pytest.mark.parametrize("hist,early", [((16383,), False), ((16383,), True),
                                        ((3000, 2500), False), ((3000, 2500), True),
                                        ((9000, 1, 0, 4000, 6000), False)])
def test_ring_laps(hist, early):
    # Partitions longer than the 24-stage ring: one sequence of 16384 tokens
    # (86 pages a CTA, four laps), two of 3001 and 2501 (the appended page
    # past the first lap), and a ragged batch; with and without early reads.
    dev = gh.device()
    cfg = wl.custom_config(len(hist), 32, 8, 128, torch.bfloat16, history=("uniform", (0, 1)),
                           pool=("factor", 1.2), seed=950 + len(hist))
    w = wl.make_workload(cfg, device=dev, history=torch.tensor(hist, dtype=torch.int32))
    cs = _cluster_size(w)
    assert cs > 0
    tokens = w.max_blocks_per_seq * gh.BS
    assert -(-tokens // cs) > 24 * gh.BS   # more than one lap of the ring
    ek, ev = _appended(w)
    out, err = _step(w, _ws(w), early=early)
    _check(w, out, err, ek, ev, what=f"{hist} early={early}")


@pytest.mark.parametrize("window", [0, 16, 37, 300, 1000])
def test_sinks_and_window(window):
    dev = gh.device()
    cfg = wl.custom_config(3, 32, 8, 128, torch.bfloat16, history=("uniform", (0, 1500)),
                           pool=("factor", 1.4), seed=920 + window)
    w = wl.make_workload(cfg, device=dev)
    # (A window under 128 tokens is too short to split: the persistent grid.)
    assert (_cluster_size(w, window) > 0) == (window == 0 or window >= 128)
    g = torch.Generator(device=dev).manual_seed(window)
    sinks = (torch.randn(cfg.Hq, generator=g, device=dev) * 2).to(cfg.dtype)
    ek, ev = _appended(w)
    out, err = _step(w, _ws(w), sinks=sinks, window=window)
    _check(w, out, err, ek, ev, sinks=sinks, window=window, what=f"window={window}")


def test_bad_length_and_bad_block_append_nothing():
    # As on the persistent grid: sequence 1's length runs past its table
    # (XS_FLAG_BAD_LEN, attention clamped to the table), sequence 3's last
    # page has an out-of-pool id (XS_FLAG_BAD_BLOCK, read as block 0); neither
    # appends.  The other sequences match the separate calls' attention.
    dev = gh.device()
    cfg = wl.custom_config(4, 32, 8, 128, torch.bfloat16, history=("uniform", (40, 600)),
                           pool=("factor", 1.3), seed=930)
    w = wl.make_workload(cfg, device=dev)
    assert _cluster_size(w) > 0
    w.context_lens[1] = w.max_blocks_per_seq * gh.BS + 5
    n3 = int(w.context_lens[3])
    w.block_tables[3, (n3 - 1) // gh.BS] = w.num_blocks + 7
    lens_ok = w.context_lens.clone()
    lens_ok[1] = 0
    lens_ok[3] = 0
    want = gh.expected_rows(w.block_tables, lens_ok, w.num_blocks, cfg.Hkv)
    kc0, vc0 = w.k_cache[0].clone(), w.v_cache[0].clone()
    ws = _ws(w, 64)
    out, err = _step(w, ws)
    torch.cuda.synchronize()
    flags = int(err.item())
    assert flags & ops.FLAG_BAD_LEN and flags & ops.FLAG_BAD_BLOCK
    assert flags & ~(ops.FLAG_BAD_LEN | ops.FLAG_BAD_BLOCK) == 0
    assert gh.changed_rows(kc0, w.k_cache[0]) == want
    assert gh.changed_rows(vc0, w.v_cache[0]) == want
    # The persistent grid on the same (already appended) pools, without
    # appending again.
    ref_out = torch.empty_like(out)
    ops.xs_paged_decode(ref_out, ws.part_o, ws.part_m, ws.part_l, w.q[0], w.k_cache[0],
                        w.v_cache[0], w.block_tables, w.context_lens, w.scale,
                        ws.partition_tokens, ws.max_partitions, err_flag=err)
    torch.cuda.synchronize()
    for b in (0, 2):
        torch.testing.assert_close(out[b].float(), ref_out[b].float(), atol=1e-2, rtol=0)


def test_layers_back_to_back_in_a_cuda_graph():
    # Three layers of a two-sequence batch with early reads, captured in one
    # CUDA graph and replayed three times (each replay appends the same rows
    # again); every layer matches the oracle, and the persistent grid run on
    # the same pools agrees.
    from paged_kv_cache_xs_gb300.step import PagedDecodeStep
    dev = gh.device()
    L = 3
    hist = torch.tensor([300, 1500], dtype=torch.int32)
    cfg = wl.custom_config(2, 32, 8, 128, torch.bfloat16, layers=L, history=("uniform", (0, 1)),
                           pool=("factor", 1.3), seed=940)
    w = wl.make_workload(cfg, device=dev, history=hist)
    assert _cluster_size(w) > 0
    refs = []
    for layer in range(L):
        ek, ev = _appended(w, layer)
        refs.append(oracle.paged_decode(w.q[layer].cpu(), ek, ev, w.block_tables.cpu(),
                                        w.context_lens.cpu(), w.scale))
    step = PagedDecodeStep(cfg.B, cfg.Hq, cfg.Hkv, cfg.D, w.max_blocks_per_seq, cfg.dtype, dev,
                           partition_tokens=256)
    outs = [torch.full((cfg.B, cfg.Hq, cfg.D), float("nan"), dtype=cfg.dtype, device=dev)
            for _ in range(L)]

    def one():
        for layer in range(L):
            step.run(outs[layer], w.q[layer], w.k_new[layer], w.v_new[layer], w.k_cache[layer],
                     w.v_cache[layer], w.block_tables, w.context_lens, w.scale, early_reads=True)
    g = CapturedStep(one)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert step.error_flags() == 0
    for layer in range(L):
        gh.assert_close(outs[layer], refs[layer], torch.bfloat16, what=f"layer {layer}")
        other = torch.empty_like(outs[layer])
        step.run(other, w.q[layer], w.k_new[layer], w.v_new[layer], w.k_cache[layer],
                 w.v_cache[layer], w.block_tables, w.context_lens, w.scale, persistent=True)
        torch.cuda.synchronize()
        torch.testing.assert_close(outs[layer].float(), other.float(), atol=1e-2, rtol=0)
    assert step.error_flags() == 0


def test_decode_loop_in_a_graph_with_a_growing_sequence():
    # One sequence, 8 KV heads: a step captured once and replayed 40 times
    # while the sequence grows from 1041 to 1080 tokens (a table of 70 pages,
    # so the launch's partitions stay fixed while the sequence crosses
    # page boundaries and a partition boundary).  Each replay reads the new
    # length, q and rows from the captured buffers; every step's append and
    # attention match the oracle's.
    from paged_kv_cache_xs_gb300.step import PagedDecodeStep
    dev = gh.device()
    cfg = wl.custom_config(1, 32, 8, 128, torch.bfloat16, history=("fixed", (1040,)),
                           pool=("factor", 3.0), seed=960)
    w = wl.make_workload(cfg, device=dev)
    width = 70
    used = w.block_tables[0, :w.max_blocks_per_seq].tolist()
    spare = [i for i in range(w.num_blocks) if i not in set(used)][:width - len(used)]
    bt = torch.tensor([used + spare], dtype=torch.int32, device=dev)
    assert bt.shape[1] == width
    w.block_tables = bt
    assert _cluster_size(w) > 0
    step = PagedDecodeStep(cfg.B, cfg.Hq, cfg.Hkv, cfg.D, width, cfg.dtype, dev,
                           partition_tokens=256)
    out = torch.empty(cfg.B, cfg.Hq, cfg.D, dtype=cfg.dtype, device=dev)
    q, kn, vn = w.q[0].clone(), w.k_new[0].clone(), w.v_new[0].clone()
    lens = w.context_lens.clone()
    graph = CapturedStep(lambda: step.run(out, q, kn, vn, w.k_cache[0], w.v_cache[0], bt, lens,
                                          w.scale, early_reads=True))
    g = torch.Generator(device=dev).manual_seed(961)
    lens.fill_(1041)
    graph.replay()  # (the capture's warm-up appended at 1041 too: replay it once more first)
    torch.cuda.synchronize()
    kc, vc = w.k_cache[0].cpu(), w.v_cache[0].cpu()
    for n in range(1041, 1081):
        lens.fill_(n)
        q.copy_(torch.randn(q.shape, generator=g, device=dev).to(cfg.dtype))
        kn.copy_(torch.randn(kn.shape, generator=g, device=dev).to(cfg.dtype))
        vn.copy_(torch.randn(vn.shape, generator=g, device=dev).to(cfg.dtype))
        graph.replay()
        torch.cuda.synchronize()
        assert step.error_flags() == 0
        slots = oracle.slot_mapping(bt.cpu(), lens.cpu(), gh.BS, w.num_blocks)
        kc, vc = oracle.kv_append(kn.cpu(), vn.cpu(), kc, vc, slots)
        assert torch.equal(gh.int_view(w.k_cache[0].cpu()), gh.int_view(kc)), f"n={n}"
        assert torch.equal(gh.int_view(w.v_cache[0].cpu()), gh.int_view(vc)), f"n={n}"
        ref = oracle.paged_decode(q.cpu(), kc, vc, bt.cpu(), lens.cpu(), w.scale)
        gh.assert_close(out, ref, torch.bfloat16, what=f"n={n}")


@pytest.mark.parametrize("window", [6000, 3001])
def test_window_over_a_long_sequence(window):
    # One 16,384-token sequence with sinks and a window whose first token
    # does not start a page: the window's partitions (one page more than
    # their length, for the unaligned start) run past the 24-stage ring at
    # window 6000.
    dev = gh.device()
    cfg = wl.custom_config(1, 32, 8, 128, torch.bfloat16, history=("fixed", (16383,)),
                           pool=("factor", 1.1), seed=970 + window)
    w = wl.make_workload(cfg, device=dev)
    assert _cluster_size(w, window) > 0
    g = torch.Generator(device=dev).manual_seed(window)
    sinks = (torch.randn(cfg.Hq, generator=g, device=dev) * 2).to(cfg.dtype)
    ek, ev = _appended(w)
    out, err = _step(w, _ws(w), sinks=sinks, window=window, early=True)
    _check(w, out, err, ek, ev, sinks=sinks, window=window, what=f"window={window}")
