"""Derives the polynomials of the soft-cap tanh (lpd_xform.cuh).

tanh(y) = y * (1 + z * P(z)), z = y^2, on |y| < Y_MAX.  Two fits are used:
degree 4 on |y| < 0.6 (the general per-op chain) and degree 3 on |y| < 0.45
(the reduced single soft-cap pass, which evaluates the same series on x^2 with
the coefficients pre-multiplied by powers of 1/p^2; one fused multiply-add
less per value, and 0.67 ulp in float32 on its range).  Each P is a weighted
least-squares fit of (tanh(y)/y - 1) / z on Chebyshev nodes of z in
[0, Y_MAX^2].  The weight z * y / tanh(y) makes the
residual the relative error of tanh, and 30 reweighting passes push the fit
towards equal-ripple.  The coefficients are rounded to float32, and the script
reports the worst error of a float32 Horner evaluation (one rounding per fused
multiply-add) against 40-digit tanh, in units in the last place: 0.63 ulp
(degree 5 gives 0.70, degree 3 on the same range 2.6; the final rounding of
y (1 + z P) dominates once the fit is below it).

Run: python tanh_coeffs.py   (needs numpy and mpmath; not used at build time)
     python tanh_coeffs.py 0.45 3   (the reduced pass's fit)
"""
import numpy as np
from mpmath import mp, mpf, tanh as mtanh

mp.dps = 40
Y_MAX, DEGREE, NODES = 0.6, 4, 4000


def target(z):
    out = []
    for zz in z:
        y = mp.sqrt(mpf(float(zz)))
        out.append(float((mtanh(y) / y - 1) / mpf(float(zz))) if zz > 0 else -1.0 / 3.0)
    return np.array(out)


def fit():
    k = np.arange(NODES)
    z = (Y_MAX * Y_MAX) * (0.5 - 0.5 * np.cos(np.pi * (k + 0.5) / NODES))
    y = np.sqrt(z)
    w = z * y / np.array([float(mtanh(mpf(float(v)))) for v in y])
    V = np.vander(z, DEGREE + 1, increasing=True)
    tgt = target(z)
    c, *_ = np.linalg.lstsq(V * w[:, None], tgt * w, rcond=None)
    for _ in range(30):
        err = np.abs((V @ c - tgt) * w)
        ww = w * (1 + 30 * err / err.max())
        c, *_ = np.linalg.lstsq(V * ww[:, None], tgt * ww, rcond=None)
    return [np.float32(v) for v in c]


def fma32(a, b, c):
    return np.float32(np.float64(a) * np.float64(b) + np.float64(c))


def worst_ulp(cf, samples=20001):
    worst = 0.0
    for yv in np.float32(np.linspace(1e-6, Y_MAX, samples)):
        zz = np.float32(yv * yv)
        p = cf[-1]
        for cc in cf[-2::-1]:
            p = fma32(p, zz, cc)
        t = fma32(yv, np.float32(zz * p), yv)
        ex = float(mtanh(mpf(float(yv))))
        worst = max(worst, abs(float(t) - ex) / float(np.spacing(np.float32(ex))))
    return worst


if __name__ == "__main__":
    import sys

    if len(sys.argv) == 3:
        Y_MAX, DEGREE = float(sys.argv[1]), int(sys.argv[2])
    cf = fit()
    print("coefficients c0..c%d:" % DEGREE, ", ".join(f"{float(v):.9e}f" for v in cf))
    print("worst float32 error: %.3f ulp" % worst_ulp(cf))
