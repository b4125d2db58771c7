"""The five decode-step workloads through the CUDA path, against the oracle.

Configs 0-3 are checked on every sequence and every layer.  Config 4 (128
sequences, contexts up to 32769 tokens, ~17 GB pool) runs in the launch
configuration the benchmark times and is checked on 8 sampled sequences
(including the longest and shortest) with all of their heads; its append is
checked on every sequence (bytes at the new slots, nothing else touched).
Each runs both as the one-launch fused step and as three separate launches."""
import pytest
import torch

from paged_kv_cache_xs_gb300 import workloads as wl
from paged_kv_cache_xs_gb300.step import PagedDecodeStep
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu


def _step_for(w, dev):
    cfg = w.cfg
    return PagedDecodeStep(cfg.B, cfg.Hq, cfg.Hkv, cfg.D, w.max_blocks_per_seq, cfg.dtype, dev,
                           total_context_tokens=w.total_context_tokens,
                           max_context_len=w.max_context_len)


@pytest.mark.parametrize("fused", [True, False], ids=["one-launch", "three-launch"])
@pytest.mark.parametrize("cfg_id", [0, 1, 2, 3])
def test_config_all_sequences(cfg_id, fused):
    dev = gh.device()
    w = wl.make_workload(cfg_id, device=dev)
    step = _step_for(w, dev)
    errs = [gh.check_step(w, layer, step, fused=fused) for layer in range(w.cfg.layers)]
    print(f"{w.cfg.name}: P={step.partition_tokens} fused={fused} max err {max(errs):.3e}")


def test_config4_sampled():
    # Both forms of the step, one after the other on the same workload: the
    # second appends the same rows again, so its pre-state is the first's result.
    dev = gh.device()
    w = wl.make_workload(4, device=dev)
    step = _step_for(w, dev)
    lens = w.context_lens.cpu()
    g = torch.Generator().manual_seed(4)
    pick = set(torch.randperm(w.cfg.B, generator=g)[:6].tolist())
    pick |= {int(lens.argmax()), int(lens.argmin())}
    for fused in (True, False):
        err = gh.check_step(w, 0, step, seqs=sorted(pick), check_unchanged=True, fused=fused)
        print(f"{w.cfg.name}: P={step.partition_tokens} parts<={step.max_partitions} "
              f"fused={fused} sampled max err {err:.3e}")


@pytest.mark.parametrize("cfg_id", [1, 3])
def test_config_early_reads_back_to_back(cfg_id):
    # The benchmark's loop: the one-launch step with early reads, several
    # launches back to back on the same pools and lengths (each appends the
    # same rows again and may start while the previous one finishes).
    dev = gh.device()
    w = wl.make_workload(cfg_id, device=dev)
    step = _step_for(w, dev)
    for layer in range(min(w.cfg.layers, 2)):
        gh.check_step(w, layer, step, repeat=4, early_reads=True)


def test_config4_sampled_early_reads():
    dev = gh.device()
    w = wl.make_workload(4, device=dev)
    step = _step_for(w, dev)
    lens = w.context_lens.cpu()
    g = torch.Generator().manual_seed(44)
    pick = set(torch.randperm(w.cfg.B, generator=g)[:6].tolist())
    pick |= {int(lens.argmax()), int(lens.argmin())}
    gh.check_step(w, 0, step, seqs=sorted(pick), check_unchanged=True, repeat=3,
                  early_reads=True)
