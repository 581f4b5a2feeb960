"""Host check of the float32 bound the one-mode builder uses before its exact
float64 test: a child of path sum zs, scaled logit zt, depth normaliser c and
bound theta passes exactly when fl64(fl64(zs + zt) - c) >= theta; the kernel
lists it only if ztf >= g, g = ((thf - m) + cf) - zsf, with every float32
operand the float64 value truncated toward zero and
m = 2^-18 (|thf| + |cf| + |zsf| + max|ztf|) + 1e-30.  Whatever passes
exactly must be listed.  numpy's float32 arithmetic rounds to nearest as
the device does; the cases put the exact score at theta or within 1e-12 of
it, over magnitudes from 1e-3 to 1e20 (the hardest cases for the margin).
"""
import numpy as np
import pytest

F32 = np.float32


def trunc32(x):
    """float64 -> float32 rounded toward zero, as the kernel's integer conversion."""
    x = np.asarray(x, dtype=np.float64)
    f = x.astype(F32)
    over = np.abs(f.astype(np.float64)) > np.abs(x)
    return np.where(over, np.nextafter(f, F32(0)), f).astype(F32)


def listed(zs, zt, c, theta, zmag):
    thf, cf, zsf, ztf = trunc32(theta), trunc32(c), trunc32(zs), trunc32(zt)
    m = F32(2.0 ** -18) * (np.abs(thf) + np.abs(cf) + np.abs(zsf) + zmag) + F32(1e-30)
    g = ((thf - m) + cf) - zsf
    return ztf >= g


@pytest.mark.parametrize("scale", [1e-3, 1.0, 30.0, 1e3, 1e6, 1e20])
def test_bound_never_drops_a_passing_child(scale):
    rng = np.random.default_rng(int(np.log10(scale) * 7) + 100)
    n = 100_000
    zs = rng.uniform(-50, 5, n) * scale
    zt = rng.uniform(-30, 10, n) * scale
    c = rng.uniform(0, 200, n) * scale
    s = (zs + zt) - c                              # the kernel's float64 evaluation
    theta = s - np.abs(s) * rng.choice([0.0, 1e-16, 1e-15, 1e-12], n)
    passes = s >= theta
    assert passes.all()
    zmag = np.abs(trunc32(zt))                     # the largest |ztf| of the row is at least this
    assert listed(zs, zt, c, theta, zmag).all()


def test_bound_is_not_vacuous():
    """Children well below the bound are not listed (the bound prunes)."""
    rng = np.random.default_rng(7)
    n = 10_000
    zs = rng.uniform(-20, 0, n)
    zt = rng.uniform(-10, 0, n)
    c = rng.uniform(0, 50, n)
    s = (zs + zt) - c
    theta = s + 1.0                                # one nat above every child
    assert not listed(zs, zt, c, theta, np.abs(trunc32(zt))).any()
