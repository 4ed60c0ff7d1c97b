"""The fp64 oracle against what the pages and the mathematics fix (CPU only)."""
import pytest

import oracle
from tests import pins


@pytest.mark.parametrize("pin", pins.ATTENTION_PINS, ids=lambda p: p.__name__)
def test_attention_pin(pin):
    pin(oracle.decode)


def test_f16_decoding_matches_numpy_on_all_patterns():
    pins.pin_f16_all_patterns(oracle.f16_to_f64)


def test_bf16_decoding_matches_torch_on_all_patterns():
    pins.pin_bf16_all_patterns(oracle.bf16_to_f64)


def test_rejects_out_of_range_table_entry():
    import numpy as np
    kp = np.zeros((2, 2, 1, 2), np.float32)
    with pytest.raises(ValueError):
        oracle.decode(np.zeros((1, 1, 2), np.float32), kp, kp, np.array([[5]], np.int32),
                      np.array([2], np.int32), 1.0, "f32", 1, 1, 2, 2)


def test_rejects_context_beyond_table():
    import numpy as np
    kp = np.zeros((2, 2, 1, 2), np.float32)
    with pytest.raises(ValueError):
        oracle.decode(np.zeros((1, 1, 2), np.float32), kp, kp, np.array([[0]], np.int32),
                      np.array([3], np.int32), 1.0, "f32", 1, 1, 2, 2)
