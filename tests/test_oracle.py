"""The fp64 oracle against its pins (CPU only), and planted mistakes caught."""
import os
import tempfile

import numpy as np
import pytest

import oracle
from oracle_pins import PINS


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin, oracle_lib):
    pin(oracle_lib)


# Each planted mistake (see PLANT in gqa_oracle.c) must fail at least one pin.
PLANTS = {1: "causal mask drops the diagonal", 2: "query head h mapped to kv head h % Hkv",
          3: "dK missing the softmax scale", 4: "Delta with the wrong sign", 5: "LSE in base 2"}


@pytest.mark.parametrize("plant", sorted(PLANTS), ids=[PLANTS[k] for k in sorted(PLANTS)])
def test_planted_mistake_is_caught(plant):
    with tempfile.TemporaryDirectory() as d:
        path = oracle.build_variant(os.path.join(d, f"plant{plant}.so"), [f"-DPLANT={plant}"])
        lib = oracle.load(path)
        failed = []
        for pin in PINS:
            try:
                with np.errstate(all="ignore"):
                    pin(lib)
            except (AssertionError, ValueError, FloatingPointError):
                failed.append(pin.__name__)
        assert failed, f"planted mistake {plant} ({PLANTS[plant]}) passed every pin"


def test_errors(oracle_lib):
    q = np.zeros((1, 3, 4, 2))
    k = np.zeros((1, 2, 4, 2))
    with pytest.raises(ValueError):
        oracle.fwd(q, k, k, lib=oracle_lib)      # Hq % Hkv != 0
    q = np.zeros((5, 2, 2))
    with pytest.raises(ValueError):
        oracle.varlen_fwd(q, q, q, [0, 3, 2, 5], lib=oracle_lib)   # decreasing cu_seqlens
    with pytest.raises(ValueError):
        oracle.varlen_fwd(q, q, q, [0, 3, 4], lib=oracle_lib)      # wrong total


def test_empty(oracle_lib):
    o, lse = oracle.fwd(np.zeros((1, 2, 0, 4)), np.zeros((1, 1, 0, 4)), np.zeros((1, 1, 0, 4)), lib=oracle_lib)
    assert o.shape == (1, 2, 0, 4) and lse.shape == (1, 2, 0)
    o, lse = oracle.varlen_fwd(np.zeros((0, 2, 4)), np.zeros((0, 1, 4)), np.zeros((0, 1, 4)), [0, 0, 0],
                               lib=oracle_lib)
    assert o.shape == (0, 2, 4)
