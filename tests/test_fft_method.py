"""The FFT frame kernels' Stockham schedule (one radix-2 stage when log2 n is
odd, then radix-4 stages), its index arithmetic mirrored on the CPU in
complex128 against numpy's FFT, both directions, every power-of-two size the
kernels take.  A wrong output index, twiddle index or butterfly sign fails it."""
from __future__ import annotations

import numpy as np
import pytest


def stockham(x, forward):
    n = x.size
    s = -1.0 if forward else 1.0
    tw = np.exp(2j * np.pi * np.arange(n) / n)           # the kernels' table, exp(+2 pi i j / n)
    a = x.astype(np.complex128).copy()
    log2n = n.bit_length() - 1
    Ls = 1
    if log2n % 2:                                        # radix 2: j = g Ls + k
        b = np.empty_like(a)
        for j in range(n // 2):
            k = j & (Ls - 1)
            w = tw[k * (n // (2 * Ls))]
            w = np.conj(w) if forward else w
            u, v = a[j], a[j + n // 2] * w
            d = 2 * (j - k) + k
            b[d], b[d + Ls] = u + v, u - v
        a, Ls = b, 2
    while Ls < n:                                        # radix 4
        b = np.empty_like(a)
        q = n // 4
        step = n // (4 * Ls)
        for j in range(q):
            k = j & (Ls - 1)
            x0 = a[j]
            xs = []
            for r in (1, 2, 3):
                w = tw[(r * k * step) % n]
                xs.append(a[j + r * q] * (np.conj(w) if forward else w))
            x1, x2, x3 = xs
            t0, t1 = x0 + x2, x0 - x2
            t2, t3 = x1 + x3, (x1 - x3) * (1j * s)
            d = 4 * (j - k) + k
            b[d] = t0 + t2
            b[d + Ls] = t1 + t3
            b[d + 2 * Ls] = t0 - t2
            b[d + 3 * Ls] = t1 - t3
        a, Ls = b, 4 * Ls
    return a


@pytest.mark.parametrize("n", [4, 8, 16, 32, 64, 256, 1024, 2048, 4096])
def test_stockham_radix4_schedule(n):
    x = np.random.default_rng(n).standard_normal(n) + 1j * np.random.default_rng(n + 1).standard_normal(n)
    np.testing.assert_allclose(stockham(x, True), np.fft.fft(x), rtol=0, atol=1e-9 * n)
    np.testing.assert_allclose(stockham(x, False), np.fft.ifft(x) * n, rtol=0, atol=1e-9 * n)
