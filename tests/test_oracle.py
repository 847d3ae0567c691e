"""The CPU oracle against its pins (closed forms, library routines,
invariants, finite differences).  CPU only."""

import pytest

import oracle
import oracle_pins


@pytest.mark.parametrize("check", oracle_pins.ALL_CHECKS, ids=lambda f: f.__name__)
def test_oracle_pin(check):
    check(oracle)


def test_bf16_decode_roundtrip():
    import numpy as np
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = oracle.decode_bf16_bits(bits)
    finite = np.isfinite(vals)
    back = oracle.round_to_bf16_bits(vals[finite])
    assert np.array_equal(back, bits[finite])
    assert oracle.decode_bf16_bits(np.array([0xFF80], dtype=np.uint16))[0] == -np.inf
    assert oracle.decode_bf16_bits(np.array([0x3F80], dtype=np.uint16))[0] == 1.0
