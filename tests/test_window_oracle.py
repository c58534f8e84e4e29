"""The sliding-window oracle against the page's worked example, closed forms and
exact brute force (CPU only); planted mistakes must be caught."""
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load_window_fixture():
    vals = {}
    with open(os.path.join(GOLDEN, "dlsys_lecture12_s3_window5.txt")) as f:
        for raw in f:
            line = raw.split("#", 1)[0].split()
            if line:
                vals[line[0]] = [float(v) for v in line[1:]]
    return int(vals["W"][0]), np.array(vals["x"], np.float32), np.array(vals["y"])


def pin_worked_example(win):
    W, x, y = load_window_fixture()
    got = win(x, W)
    assert np.array_equal(got, y), got


def pin_constant_and_ramp(win):
    for W in (1, 3, 5, 9):
        assert np.all(win(np.full(40, 2.5, np.float32), W) == 2.5 * W)
        x = np.arange(50, dtype=np.float32)                  # x_i = i
        i = np.arange(50 - W + 1)
        assert np.array_equal(win(x, W), W * i + W * (W - 1) / 2)


def pin_bruteforce_exact(win):
    rng = np.random.default_rng(80)
    for W in (1, 2, 5, 7):
        for n in (1, 2, 9, 33):
            x = (rng.integers(-64, 65, n + W - 1) / 16).astype(np.float32)
            got = win(x, W)
            for i in range(n):
                want = sum((Fraction(float(v)) for v in x[i:i + W]), Fraction(0))
                assert Fraction(float(got[i])) == want, (W, n, i)


def pin_empty_and_single(win):
    assert win(np.zeros(4, np.float32), 5).shape == (0,)
    assert np.array_equal(win(np.array([3.0, -1.0], np.float32), 2), [2.0])


PINS = [pin_worked_example, pin_constant_and_ramp, pin_bruteforce_exact, pin_empty_and_single]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_window_f64_pin(pin):
    pin(lambda x, W: oracle.window_sum(x, W))


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_window_f32_ascending_pin(pin):
    # Every pin uses values whose sums are exact in float, so both forms agree with them.
    pin(lambda x, W: oracle.window_sum_f32_ascending(x, W).astype(np.float64))


def test_f32_ascending_is_left_to_right_float_sum():
    # 1 + 2^-24 + 2^-24: left to right each tiny addend is lost (ties to even);
    # the double sum keeps them.
    x = np.array([1.0, 2.0 ** -24, 2.0 ** -24], np.float32)
    assert oracle.window_sum_f32_ascending(x, 3)[0] == np.float32(1.0)
    assert oracle.window_sum(x, 3)[0] == 1.0 + 2.0 ** -23


MUTANTS = {
    "off_by_one_window": ("for (int d = 0; d < W; ++d) s += (double)x[i + d];",
                          "for (int d = 0; d < W - 1; ++d) s += (double)x[i + d];"),
    "centred_window": ("s += (double)x[i + d];", "s += (double)x[i + d - (d > 0)];"),
    "wrong_sign": ("s += (double)x[i + d];", "s -= (double)x[i + d];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    src_path = os.path.join(os.path.dirname(oracle.SOURCE), "window_oracle.c")
    old, new = MUTANTS[name]
    src = open(src_path).read()
    assert old in src
    c = os.path.join(tmp_path, "m.c")
    open(c, "w").write(src.replace(old, new, 1))
    lib = oracle.OracleLib.__new__(oracle.OracleLib)
    import ctypes
    so = oracle.compile_source([oracle.SOURCE, c], os.path.join(tmp_path, "m.so"))
    oracle.OracleLib.__init__(lib, so)
    failed = []
    for pin in PINS:
        try:
            pin(lambda x, W: lib.window_sum(x, W))
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, name
