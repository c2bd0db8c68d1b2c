"""The softcap's tanh is computed from its definition (the kernels' tanh_def): the odd Taylor series
x - x^3/3 + 2x^5/15 - 17x^7/315 below |x| = 1/8, and (1 - e) / (1 + e) with e = exp(-2|x|) above,
the sign restored.  This checks that choice of split and truncation in fp32 arithmetic against
fp64 tanh (the device code adds its approximate exp2 and division on top; the softcap parity tests
cover that end to end)."""
import numpy as np


def tanh_def_f32(x):
    x = np.asarray(x, dtype=np.float32)
    f = np.float32
    a = np.abs(x)
    with np.errstate(over="ignore", invalid="ignore"):  # (the unused branch may overflow, as on the GPU)
        x2 = x * x
        series = x * (f(1) + x2 * (f(-1 / 3) + x2 * (f(2 / 15) + x2 * f(-17 / 315))))
        e = np.exp(f(-2) * a).astype(np.float32)
        t = np.copysign((f(1) - e) / (f(1) + e), x)
    return np.where(a < f(0.125), series, t)


def test_relative_error_over_the_range():
    x = np.concatenate([np.linspace(-12, 12, 200001), np.geomspace(1e-30, 0.5, 20001),
                        -np.geomspace(1e-30, 0.5, 20001), [0.125, np.nextafter(0.125, 0), 0.1249999]])
    x = x.astype(np.float32)
    got = tanh_def_f32(x).astype(np.float64)
    ref = np.tanh(x.astype(np.float64))
    nz = ref != 0
    rel = np.abs(got[nz] - ref[nz]) / np.abs(ref[nz])
    assert rel.max() < 2e-6, rel.max()
    assert np.all(got[~nz] == 0)


def test_limits_and_nan():
    got = tanh_def_f32(np.array([np.inf, -np.inf, 1e30, -1e30, np.nan], dtype=np.float32))
    assert got[0] == 1 and got[1] == -1 and got[2] == 1 and got[3] == -1 and np.isnan(got[4])


def test_odd_and_bounded():
    x = np.linspace(0, 20, 40001, dtype=np.float32)
    assert np.array_equal(tanh_def_f32(-x), -tanh_def_f32(x))
    assert np.all(np.abs(tanh_def_f32(x)) <= 1)
