"""The oracle against facts fixed outside it (CPU only)."""
import pytest

import oracle_pins as P


@pytest.mark.parametrize("pin", P.FAST_PINS, ids=lambda f: f.__name__)
def test_fast_pin(pin):
    pin(None)


def test_escape_fraction_k5120():
    frac, ana = P.pin_escape_fraction(None, N=2048, K=5120, seed=31)
    assert 5e-5 < frac < 1e-4


def test_escape_fraction_k17408():
    P.pin_escape_fraction(None, N=768, K=17408, seed=32)


def test_bits_per_weight():
    bpw = P.pin_bits_per_weight(None)
    assert bpw < 12.01


def test_converted_size_matches_printed():
    predicted = P.pin_converted_size()
    print(f"predicted converted size {predicted:.2f} GB (printed 33.58 GB)")
