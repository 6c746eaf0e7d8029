"""Pins of the iSTFT-head oracle (CPU): each checks it against something other
than itself - perfect reconstruction of a random signal from an independent
forward STFT, the envelope's closed form, the transposed-convolution form of
the Core AI Kokoro note (conv_transpose1d, stride = hop) through the library
routine, a single-bin closed form, chunked == full, and planted mistakes that
the reconstruction pin catches."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from oracle import istft as O

CONFIGS = [(1024, 256), (20, 5), (16, 4), (64, 16), (64, 32)]


def analysis_spec(s, n_fft, hop, T):
    """Forward STFT (numpy rfft of Hann-windowed frames at t * hop) as
    log-magnitude / phase frames: the input a perfect-reconstruction check
    feeds back."""
    w = O.hann_periodic(n_fft)
    X = np.stack([np.fft.rfft(w * s[t * hop:t * hop + n_fft]) for t in range(T)])
    return np.concatenate([np.log(np.abs(X)), np.angle(X)], axis=1)


@pytest.mark.parametrize("n_fft,hop", CONFIGS)
def test_perfect_reconstruction(n_fft, hop):
    rng = np.random.default_rng(n_fft + hop)
    T = 40
    s = rng.standard_normal(T * hop + n_fft)
    y = O.istft_full(analysis_spec(s, n_fft, hop, T), n_fft, hop)
    lo = n_fft - hop           # from here on every sample is covered by all n_fft / hop frames
    np.testing.assert_allclose(y[lo:], s[lo:T * hop], rtol=0, atol=1e-11)


@pytest.mark.parametrize("K", [3, 4, 5, 8])
def test_envelope_closed_form(K):
    """sum_j sin^4(x + pi j / K) = 3 K / 8 for K >= 3 equally spaced frames."""
    n_fft = 16 * K
    np.testing.assert_allclose(O.envelope(n_fft, n_fft // K), 3 * K / 8, rtol=0, atol=1e-13)


@pytest.mark.parametrize("n_fft,hop", CONFIGS)
def test_conv_transpose_form(n_fft, hop):
    """The iSTFT as one transposed convolution (stride hop, 2 n_bins channels
    -> 1): weight[k][m] = c_k cos(2 pi k m / N) w[m] / (N E[m mod hop]) for the
    real parts and -c_k sin(...) ... for the imaginary parts, c_0 = c_{N/2} = 1,
    else 2; torch's conv_transpose1d in float64 must give the oracle's samples."""
    rng = np.random.default_rng(7)
    nb = n_fft // 2 + 1
    T = 12
    spec = np.concatenate([rng.normal(0, 0.5, (T, nb)), rng.uniform(-np.pi, np.pi, (T, nb))], axis=1)
    mag = np.exp(spec[:, :nb])
    re, im = mag * np.cos(spec[:, nb:]), mag * np.sin(spec[:, nb:])
    k = np.arange(nb)[:, None]
    m = np.arange(n_fft)[None, :]
    c = np.full((nb, 1), 2.0)
    c[0] = 1.0
    if n_fft % 2 == 0:
        c[-1] = 1.0
    scale = O.hann_periodic(n_fft)[None, :] / (n_fft * O.envelope(n_fft, hop)[m % hop])
    wr = c * np.cos(2 * np.pi * k * m / n_fft) * scale
    wi = -c * np.sin(2 * np.pi * k * m / n_fft) * scale
    weight = torch.from_numpy(np.concatenate([wr, wi], axis=0)[:, None, :])
    x = torch.from_numpy(np.concatenate([re, im], axis=1).T[None])
    y = torch.nn.functional.conv_transpose1d(x, weight, stride=hop)[0, 0, :T * hop].numpy()
    np.testing.assert_allclose(O.istft_full(spec, n_fft, hop), y, rtol=0, atol=1e-12)


def test_single_bin_closed_form():
    """Only bin k0 (a multiple of n_fft / hop, so every frame is in phase):
    y[n] = (2 A / N) (sum_j w[p + j hop] / E[p]) cos(2 pi k0 n / N + phi)."""
    n_fft, hop, k0, A, phi = 64, 16, 8, 3.0, 0.7
    nb = n_fft // 2 + 1
    T = 10
    spec = np.full((T, 2 * nb), -np.inf)
    spec[:, nb:] = 0.0
    spec[:, k0] = np.log(A)
    spec[:, nb + k0] = phi
    y = O.istft_full(spec, n_fft, hop)
    n = np.arange(n_fft - hop, T * hop)
    gain = 2.0 / 1.5      # sum of 4 Hann values at spacing N/4 is 2; E = 3/2
    np.testing.assert_allclose(y[n], 2 * A / n_fft * gain * np.cos(2 * np.pi * k0 * n / n_fft + phi), atol=1e-13)


@pytest.mark.parametrize("n_fft,hop", CONFIGS)
def test_chunked_equals_full(n_fft, hop):
    rng = np.random.default_rng(3)
    nb = n_fft // 2 + 1
    T = 30
    spec = np.concatenate([rng.normal(0, 1, (T, nb)), rng.uniform(-np.pi, np.pi, (T, nb))], axis=1)
    full = O.istft_full(spec, n_fft, hop)
    outs = []
    for splits in ([30], [1] * 30, [1, 2, 3, 4, 20], [7, 7, 7, 9]):
        st = O.IstftStream(n_fft, hop)
        parts, t = [], 0
        for n in splits:
            parts.append(st.decode(spec[t:t + n]))
            t += n
        outs.append(np.concatenate(parts))
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])           # the same per-sample order whatever the split
    np.testing.assert_allclose(outs[0], full, rtol=0, atol=1e-12)


def test_reset_and_clip():
    n_fft, hop = 64, 16
    nb = n_fft // 2 + 1
    rng = np.random.default_rng(5)
    spec = np.concatenate([rng.normal(3, 2, (8, nb)), rng.uniform(-np.pi, np.pi, (8, nb))], axis=1)
    st = O.IstftStream(n_fft, hop, mag_clip=20.0)
    a = st.decode(spec)
    st.reset()
    assert np.array_equal(st.decode(spec), a)
    clipped = spec.copy()
    clipped[:, :nb] = np.minimum(clipped[:, :nb], np.log(20.0))
    np.testing.assert_allclose(a, O.istft_full(clipped, n_fft, hop), atol=1e-12)


def test_planted_mistakes_fail_reconstruction():
    """A flipped phase sign, a missing window, or frames placed one hop off all
    break perfect reconstruction (so the pin above would catch them)."""
    n_fft, hop, T = 64, 16, 30
    rng = np.random.default_rng(11)
    s = rng.standard_normal(T * hop + n_fft)
    spec = analysis_spec(s, n_fft, hop, T)
    nb = n_fft // 2 + 1
    lo = n_fft - hop
    flipped = spec.copy()
    flipped[:, nb:] *= -1
    assert np.abs(O.istft_full(flipped, n_fft, hop)[lo:] - s[lo:T * hop]).max() > 0.1
    x = np.fft.irfft(np.exp(spec[:, :nb]) * np.exp(1j * spec[:, nb:]), n=n_fft, axis=1)   # no window
    y = np.zeros(T * hop + n_fft)
    for t in range(T):
        y[t * hop:t * hop + n_fft] += x[t]
    y = y[:T * hop] / np.tile(O.envelope(n_fft, hop), T)
    assert np.abs(y[lo:] - s[lo:T * hop]).max() > 0.1
    shifted = O.istft_full(spec, n_fft, hop)
    assert np.abs(shifted[lo + hop:] - s[lo:T * hop - hop]).max() > 0.1


def test_page_istft_sizes():
    """The Core AI note runs Kokoro's iSTFT as a transposed conv of stride 5
    from 11 channels to 1: n_fft / 2 + 1 = 11 bins at hop 5 is n_fft 20, the
    size the oracle and the GPU tests use; it reconstructs (above)."""
    import json
    from pathlib import Path
    facts = json.loads((Path(__file__).parent / "golden" / "page_facts.json").read_text())
    hop = facts["istft_transposed_conv_stride"]["value"]
    bins = facts["istft_transposed_conv_in_channels"]["value"]
    n_fft = 2 * (bins - 1)
    assert (n_fft, hop) == (20, 5) and (20, 5) in CONFIGS
    assert n_fft % hop == 0 and O.envelope(n_fft, hop).min() > 0
    # 600 samples per Kokoro frame are 120 iSTFT hops
    assert facts["kokoro_samples_per_frame"]["value"] % hop == 0
