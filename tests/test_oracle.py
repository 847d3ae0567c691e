"""The CPU oracle against its pins (closed forms, library routines,
invariants, finite differences).  CPU only."""

import pytest

import oracle
import oracle_pins


@pytest.mark.parametrize("check", oracle_pins.ALL_CHECKS, ids=lambda f: f.__name__)
def test_oracle_pin(check):
    check(oracle)


def test_bf16_decode_matches_torch():
    """Every one of the 65536 bfloat16 patterns decodes to the value torch's
    own bfloat16 -> float64 conversion gives (NaNs as NaNs)."""
    import numpy as np
    import torch
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = oracle.decode_bf16_bits(bits)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(vals), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(vals[fin], ref[fin])
    assert oracle.decode_bf16_bits(np.array([0xFF80], dtype=np.uint16))[0] == -np.inf
    assert oracle.decode_bf16_bits(np.array([0x3F80], dtype=np.uint16))[0] == 1.0
