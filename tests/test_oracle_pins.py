"""The CPU oracle against closed forms, brute force, a dense formulation and
invariants (see tests/oracle_pins.py for what each pin checks)."""
import pytest

from tests import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin, oracle_lib):
    pin(oracle_lib)


def test_oracle_rejects_bad_inputs(oracle_lib):
    import torch
    import oracle

    # A block id outside the pool and a length beyond the table are errors,
    # never clamped.
    bt = torch.tensor([[0, 5]], dtype=torch.int32)
    with pytest.raises(oracle.OracleError):
        oracle.slot_mapping(bt, torch.tensor([20], dtype=torch.int32), 16, 4, lib=oracle_lib)
    with pytest.raises(oracle.OracleError):
        oracle.slot_mapping(bt, torch.tensor([40], dtype=torch.int32), 16, 8, lib=oracle_lib)
    q = torch.zeros(1, 2, 4)
    pool = torch.zeros(4, 2, 16, 4)
    with pytest.raises(oracle.OracleError):
        oracle.paged_decode(q, pool, pool, bt, torch.tensor([20], dtype=torch.int32), 1.0,
                            lib=oracle_lib)
    # Hq not a multiple of Hkv.
    with pytest.raises(oracle.OracleError):
        oracle.paged_decode(torch.zeros(1, 3, 4), pool, pool, bt,
                            torch.tensor([3], dtype=torch.int32), 1.0, lib=oracle_lib)


def test_oracle_empty_sequence_is_zero(oracle_lib):
    import torch
    import oracle

    bt = torch.tensor([[1], [-1]], dtype=torch.int32)
    pool = torch.randn(2, 1, 16, 4)
    out = oracle.paged_decode(torch.randn(2, 1, 4), pool, pool, bt,
                              torch.tensor([3, 0], dtype=torch.int32), 0.5, lib=oracle_lib)
    assert torch.equal(out[1], torch.zeros(1, 4, dtype=torch.float64))
    assert torch.isfinite(out).all()
