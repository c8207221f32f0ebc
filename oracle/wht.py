"""Normalised Walsh-Hadamard rotation over head_dim (oracle side).

"spark_runtime/kv_cache.rs", ``KvCacheDtype::Turbo4`` ("Walsh-Hadamard
rotation") and ``is_wht_rotated`` (the write path rotates before quantizing;
decode needs WHT(Q) before the scores and the inverse WHT on the output).

Reading adopted (the page gives no matrix): the Sylvester-ordered Hadamard
matrix H_n (H_1 = [1], H_2n = [[H_n, H_n], [H_n, -H_n]]) scaled by 1/sqrt(n),
no random sign diagonal.  That matrix is symmetric and orthonormal, so it is
its own inverse, which is what lets decode rotate Q forward and rotate the
output back with the same transform.

Two versions:
* ``fwht_f32``: the fast transform in fp32, in the fixed butterfly order the
  write path uses to decide stored bytes.  Stages h = 1, 2, 4, ..., n/2; in
  each stage, for every j whose bit h is clear, (x[j], x[j+h]) becomes
  (x[j] + x[j+h], x[j] - x[j+h]).  After the last stage every element is
  multiplied once by fp32(1/sqrt(n)).
* ``wht_f64``: the dense matrix product with scipy's Sylvester Hadamard
  matrix in fp64, used where attention is computed (a library primitive).

Pins (tests/test_oracle_wht.py): H H = I and norm preservation in fp64;
closed forms (e_0 -> all 1/sqrt(n); all-ones -> sqrt(n) e_0); fp32 fast
transform equal to the fp64 matrix product within a few fp32 ulp.
"""

import math

import numpy as np
from scipy.linalg import hadamard


def fwht_f32(x):
    """Rotate the last axis of fp32 ``x`` (length a power of two) in fp32."""
    x = np.array(x, dtype=np.float32, copy=True)
    n = x.shape[-1]
    assert n & (n - 1) == 0, "length must be a power of two"
    lead = x.shape[:-1]
    h = 1
    while h < n:
        blocks = x.reshape(lead + (n // (2 * h), 2, h))
        a = blocks[..., 0, :]
        b = blocks[..., 1, :]
        x = np.stack((a + b, a - b), axis=-2).reshape(lead + (n,))
        h *= 2
    return x * np.float32(1.0 / math.sqrt(n))


def wht_f64(x):
    """Normalised Sylvester WHT of the last axis, fp64 dense matrix product."""
    x = np.asarray(x, dtype=np.float64)
    n = x.shape[-1]
    h = hadamard(n).astype(np.float64) / math.sqrt(n)
    return x @ h  # h is symmetric, so x @ h == (h @ x^T)^T
