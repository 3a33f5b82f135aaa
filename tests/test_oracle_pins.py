"""The fp64 oracle against facts that do not come from the oracle itself."""
import numpy as np
import pytest
import torch

import oracle
import oracle_pins


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(lib, pin):
    pin(lib)


@pytest.mark.parametrize("pin", oracle_pins.FLOOR_PINS, ids=lambda f: f.__name__)
def test_floor_pin(lib, pin):
    pin(lib)


def test_thread_count_does_not_change_results(lib):
    rng = np.random.default_rng(3)
    q, k, v = (rng.standard_normal((2, 3, 33, 16)) for _ in range(3))
    a = oracle.attention(q, k, v, 0.25, True, nthreads=1, lib=lib)
    b = oracle.attention(q, k, v, 0.25, True, nthreads=7, lib=lib)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_bad_rows_rejected(lib):
    q = np.zeros((1, 1, 4, 2))
    with pytest.raises(RuntimeError):
        oracle.attention(q, q, q, 1.0, False, rows=[4], lib=lib)


# ---------------------------------------------------------------- rounding

@pytest.mark.parametrize("fmt,tdt", [(oracle.FMT_BF16, torch.bfloat16),
                                     (oracle.FMT_F16, torch.float16)])
def test_round_fmt_matches_torch_casts(lib, fmt, tdt):
    """The floor's 16-bit rounding equals torch's fp32 -> 16-bit cast (round
    to nearest even, gradual underflow), including ties and subnormals."""
    rng = np.random.default_rng(11)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.random(20000) * 2.0 ** -rng.integers(0, 30, 20000)).astype(np.float32),
        (rng.random(5000) * 1e-7).astype(np.float32),
        (rng.random(5000) * 1e-40).astype(np.float32),
        np.array([0.0, -0.0, 1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8,
                  1.0 + 2 ** -11, 1.0 + 3 * 2 ** -11, 2 ** -24, 3 * 2 ** -25,
                  2 ** -25, 65504.0], np.float32),
    ])
    got = oracle.round_fmt(x, fmt, lib=lib)
    ref = torch.from_numpy(x).to(tdt).float().numpy()
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
