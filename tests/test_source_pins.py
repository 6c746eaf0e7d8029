"""Pins of the sine-source and analysis-STFT oracles (CPU), each against
something other than itself: a brute-force DFT on tiny inputs, a cosine's
closed form, the round trip through the (separately pinned) iSTFT oracle,
chunked == full, and the sine source's closed form for constant F0."""
from __future__ import annotations

import numpy as np
import pytest

from oracle import istft as I
from oracle import source as O


def test_stft_brute_force_tiny():
    n_fft, hop = 8, 2
    rng = np.random.default_rng(0)
    x = rng.standard_normal(6 * hop)
    X = O.StftStream(n_fft, hop).decode(x)
    buf = np.concatenate([np.zeros(n_fft - hop), x])
    w = [np.sin(np.pi * m / n_fft) ** 2 for m in range(n_fft)]
    for t in range(6):
        for k in range(n_fft // 2 + 1):
            re = sum(w[m] * buf[t * hop + m] * np.cos(2 * np.pi * k * m / n_fft) for m in range(n_fft))
            im = -sum(w[m] * buf[t * hop + m] * np.sin(2 * np.pi * k * m / n_fft) for m in range(n_fft))
            assert abs(X[t, k] - re) < 1e-12 and abs(X[t, n_fft // 2 + 1 + k] - im) < 1e-12


def test_stft_cosine_closed_form():
    """A cosine on bin k0: |X[k0]| = A N / 4 (Hann sums to N / 2), |X[k0 +- 1]| = A N / 8, 0 elsewhere."""
    n_fft, hop, k0, A = 64, 16, 5, 1.7
    n = np.arange(40 * hop)
    x = A * np.cos(2 * np.pi * k0 * n / n_fft + 0.4)
    X = O.StftStream(n_fft, hop).decode(x)[10:]          # frames fully inside the signal
    nb = n_fft // 2 + 1
    mag = np.hypot(X[:, :nb], X[:, nb:])
    np.testing.assert_allclose(mag[:, k0], A * n_fft / 4, rtol=1e-12)
    np.testing.assert_allclose(mag[:, [k0 - 1, k0 + 1]], A * n_fft / 8, rtol=1e-12)
    others = np.delete(mag, [k0 - 1, k0, k0 + 1], axis=1)
    assert others.max() < 1e-10


@pytest.mark.parametrize("n_fft,hop", [(1024, 256), (20, 5), (16, 4), (64, 32)])
def test_stft_istft_round_trip_is_a_delay(n_fft, hop):
    rng = np.random.default_rng(n_fft)
    T = 30
    x = rng.standard_normal(T * hop)
    X = O.StftStream(n_fft, hop).decode(x)
    nb = n_fft // 2 + 1
    spec = np.concatenate([np.log(np.hypot(X[:, :nb], X[:, nb:])), np.arctan2(X[:, nb:], X[:, :nb])], axis=1)
    y = I.istft_full(spec, n_fft, hop)
    d = n_fft - hop
    np.testing.assert_allclose(y[d + d:], x[d:T * hop - d], atol=1e-10)


def test_stft_chunked_equals_full():
    n_fft, hop = 64, 16
    x = np.random.default_rng(1).standard_normal(50 * hop)
    full = O.StftStream(n_fft, hop).decode(x)
    st = O.StftStream(n_fft, hop)
    parts, t = [], 0
    for n in (1, 2, 3, 20, 24):
        parts.append(st.decode(x[t * hop:(t + n) * hop]))
        t += n
    assert np.array_equal(np.concatenate(parts), full)


def test_sine_constant_f0_closed_form():
    upp, fs, H, A, f0 = 256, 24000.0, 4, 0.1, 187.3
    T = 100
    out = O.SineSource(upp, fs, H, A).decode(np.full(T, f0, np.float32))
    n = np.arange(T * upp) + 1                                  # the increment of sample n is included
    f = float(np.float32(f0))
    for h in range(1, H + 1):
        ref = A * np.sin(2 * np.pi * h * f * n / fs)
        bound = A * 2 * np.pi * h * n[-1] * 0.5 / O.TWO32 + 1e-12   # phase quantisation, 1/2 unit per sample
        assert np.abs(out[:, h - 1] - ref).max() <= bound


def test_sine_harmonic_frequencies():
    upp, fs, H, f0 = 100, 8000.0, 3, 250.0                      # 250 Hz: harmonic h on bin h * 250 / (8000 / N)
    out = O.SineSource(upp, fs, H, 1.0).decode(np.full(80, f0, np.float32))
    N = 8000
    for h in range(1, H + 1):
        spec = np.abs(np.fft.rfft(out[:N, h - 1]))
        assert int(np.argmax(spec)) == round(h * f0 * N / fs)


def test_sine_unvoiced_chunked_and_wrap():
    upp, fs, H, A = 64, 16000.0, 2, 0.5
    rng = np.random.default_rng(2)
    f0 = rng.uniform(60, 400, 300).astype(np.float32)
    f0[rng.random(300) < 0.3] = 0.0                             # unvoiced frames
    full = O.SineSource(upp, fs, H, A).decode(f0)
    assert np.all(full[np.repeat(f0 <= 0, upp)] == 0)
    st = O.SineSource(upp, fs, H, A)
    parts, t = [], 0
    for n in (1, 5, 94, 200):
        parts.append(st.decode(f0[t:t + n]))
        t += n
    assert np.array_equal(np.concatenate(parts), full)
    # the integer phase is the float64 running sum of the increments, modulo one cycle
    D = np.repeat(O.phase_increments(f0, fs), upp)
    assert st.phase == int(np.sum(D)) % O.TWO32
