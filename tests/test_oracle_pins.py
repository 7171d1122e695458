"""The CPU oracle against its pins (hand-derived fixtures, numpy, closed forms, brute force)."""
import pytest

import oracle
from oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin(oracle.bound(oracle.Oracle()))


def test_q8_0_bytes_per_weight():
    """34 bytes per 32 weights = 1.0625 B/w, the ratio fp8_ffi.rs (st_e4m3_enabled doc)
    reports as its measured resident byte ratio."""
    import numpy as np
    for k in (256, 1280, 4096):
        wb = oracle.quantize_q8_0(np.zeros((3, k), dtype=np.float32))
        assert wb.size / (3 * k) == 1.0625
        assert wb.shape[1] == k // 32 * (32 + 2)
