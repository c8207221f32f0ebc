"""Lloyd-Max quantizer for the standard normal N(0,1) (oracle side).

"spark_runtime/kv_cache.rs", ``KvCacheDtype::Turbo4/Turbo3/Turbo2``: 4-, 3-
and 2-bit "optimal Gaussian codebook" (Lloyd-Max) with 16, 8 and 4 levels.
The page prints no level values; they are recomputed here.

Lloyd's two optimality conditions for a density p:
  * boundaries are midpoints of adjacent levels: t_i = (c_i + c_{i+1}) / 2;
  * each level is the conditional mean of its cell:
        c_i = E[X | t_{i-1} < X <= t_i].
For N(0,1), with phi the density and Phi the CDF, the conditional mean has the
closed form  (phi(t_{i-1}) - phi(t_i)) / (Phi(t_i) - Phi(t_{i-1})).
The fixed-point iteration of the two conditions is run in fp64 until no level
moves by more than 1e-15 (well inside the 1e-9 the method asks for).

Codes are the level indices in ascending order (code 0 = most negative).  The
decision thresholds used to pick a code are the fp64 midpoints rounded once to
fp32; a value lying exactly on a threshold goes to the upper level (the code
is the number of thresholds <= v).

Pins (tests/test_oracle_codebook.py): the 1-bit closed form +-sqrt(2/pi);
Max's published N(0,1) tables for 2, 3 and 4 bits; the centroid condition
checked by numerical quadrature (scipy.integrate.quad, independent of the
closed form); the distortion closed form checked by quadrature and by Monte
Carlo on N(0,1) samples.
"""

import math

import numpy as np
from scipy.special import ndtr


def _pdf(x):
    return np.exp(-0.5 * x * x) / math.sqrt(2.0 * math.pi)


def lloyd_max_gaussian(bits, tol=1e-15, max_iter=1_000_000):
    """Levels (fp64, ascending) of the 2**bits-level Lloyd-Max N(0,1) quantizer."""
    n = 1 << bits
    c = np.linspace(-2.0, 2.0, n)
    for _ in range(max_iter):
        t = 0.5 * (c[:-1] + c[1:])
        lo = np.concatenate(([-np.inf], t))
        hi = np.concatenate((t, [np.inf]))
        c_new = (_pdf(lo) - _pdf(hi)) / (ndtr(hi) - ndtr(lo))
        moved = np.max(np.abs(c_new - c))
        c = c_new
        if moved < tol:
            break
    else:  # pragma: no cover - never reached for bits <= 4
        raise RuntimeError("Lloyd-Max iteration did not converge")
    # Exact symmetry of N(0,1): average the mirror pairs so c_i == -c_{n-1-i}.
    c = 0.5 * (c - c[::-1])
    return c


def codebook(bits):
    """(levels fp64, levels fp32, thresholds fp32) for a ``bits``-bit code."""
    lv = lloyd_max_gaussian(bits)
    thr = (0.5 * (lv[:-1] + lv[1:])).astype(np.float32)
    return lv, lv.astype(np.float32), thr


def distortion(levels):
    """Closed-form MSE E[(X - Q(X))^2] of the quantizer on N(0,1).

    Per cell (a, b] with level c:
      int (x - c)^2 phi = [Phi - x phi]_a^b - 2c [ -phi ]_a^b + c^2 [Phi]_a^b
    using int x^2 phi = Phi - x phi and int x phi = -phi.
    """
    c = np.asarray(levels, dtype=np.float64)
    t = 0.5 * (c[:-1] + c[1:])
    a = np.concatenate(([-np.inf], t))
    b = np.concatenate((t, [np.inf]))

    def xphi(x):
        out = np.zeros_like(x)
        fin = np.isfinite(x)
        out[fin] = x[fin] * _pdf(x[fin])
        return out

    mass = ndtr(b) - ndtr(a)
    second = mass - (xphi(b) - xphi(a))
    first = _pdf(a) - _pdf(b)
    return float(np.sum(second - 2.0 * c * first + c * c * mass))


def quantize_unit(v, thresholds):
    """Code of each fp32 value v: the number of thresholds <= v."""
    v = np.asarray(v, dtype=np.float32)
    return np.searchsorted(thresholds, v, side="right").astype(np.uint8)
