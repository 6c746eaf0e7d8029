"""CPU oracle of the streaming iSTFT head (test infrastructure only: the tests,
the smoke check and the bench's CPU baseline use it; the CUDA library never
does).

The pages name an inverse STFT as the last step of the iSTFT-head vocoders:
F5-TTS's Vocos ("Vocos -> iSTFT"), CosyVoice2's and Chatterbox's HiFT ("F0 ->
NSF source, iSTFT"), Kokoro's iSTFTNet generator, whose iSTFT the Core AI
Kokoro note runs as a transposed convolution of stride 5 from 11 channels to
1 (n_fft 20, hop 5).  They fix nothing more, so this module takes the plainest
reading, every step in float64:

  * a frame holds n_bins = n_fft / 2 + 1 log-magnitudes L[k], then n_bins
    phases p[k] (radians);
  * X[k] = min(exp(L[k]), mag_clip) * (cos p[k] + i sin p[k])  (no clip when
    mag_clip <= 0);
  * x = irfft(X, n_fft): the inverse real DFT, which ignores the imaginary
    parts of the DC and Nyquist bins;
  * frame t is multiplied by the periodic Hann window w[m] = sin^2(pi m /
    n_fft) and overlap-added starting at sample t * hop;
  * the sum is divided by the stationary window-square envelope E[n mod hop]
    = sum_j w[(n mod hop) + j hop]^2 (hop divides n_fft), the normalisation
    under which analysis with w and this synthesis reconstruct a signal;
  * streaming is causal: frames before the stream's start are zero, and once
    frame t is in, samples [t hop, (t + 1) hop) are final, so every frame
    yields hop samples; the last n_fft / hop - 1 windowed frames are carried.

The library primitive used is numpy's irfft (one step); the overlap-add and
the envelope are written out.
"""
from __future__ import annotations

import numpy as np


def hann_periodic(n_fft: int) -> np.ndarray:
    """w[m] = sin^2(pi m / n_fft), m = 0 .. n_fft - 1 (the periodic Hann window)."""
    m = np.arange(n_fft, dtype=np.float64)
    return np.sin(np.pi * m / n_fft) ** 2


def envelope(n_fft: int, hop: int) -> np.ndarray:
    """E[p] = sum_j w[p + j hop]^2 for p = 0 .. hop - 1."""
    if n_fft % hop:
        raise ValueError("hop must divide n_fft")
    w2 = hann_periodic(n_fft) ** 2
    return w2.reshape(n_fft // hop, hop).sum(axis=0)


def frames_windowed(spec: np.ndarray, n_fft: int, mag_clip: float = 0.0) -> np.ndarray:
    """spec [T][2 n_bins] (log-magnitudes, then phases) -> w * irfft(X) [T][n_fft]."""
    nb = n_fft // 2 + 1
    spec = np.asarray(spec, dtype=np.float64)
    if spec.ndim != 2 or spec.shape[1] != 2 * nb:
        raise ValueError(f"spec must be [T][{2 * nb}]")
    mag = np.exp(spec[:, :nb])
    if mag_clip > 0:
        mag = np.minimum(mag, mag_clip)
    X = mag * (np.cos(spec[:, nb:]) + 1j * np.sin(spec[:, nb:]))
    return np.fft.irfft(X, n=n_fft, axis=1) * hann_periodic(n_fft)[None, :]


class IstftStream:
    """One stream: feed chunks of frames, get hop samples per frame."""

    def __init__(self, n_fft: int, hop: int, mag_clip: float = 0.0):
        self.n_fft, self.hop, self.mag_clip = n_fft, hop, mag_clip
        self.taps = n_fft // hop
        self.env = envelope(n_fft, hop)
        self.hist = np.zeros((self.taps - 1, n_fft))   # windowed frames -(taps-1) .. -1

    def reset(self):
        self.hist[:] = 0.0

    def decode(self, spec: np.ndarray) -> np.ndarray:
        spec = np.asarray(spec, dtype=np.float64).reshape(-1, self.n_fft + 2)
        T, hop, taps = spec.shape[0], self.hop, self.taps
        F = np.concatenate([self.hist, frames_windowed(spec, self.n_fft, self.mag_clip)], axis=0)
        # F[i] is frame i - (taps - 1); output sample n (this chunk) = frame n // hop
        y = np.zeros(T * hop)
        for t in range(T):
            for j in range(taps):
                # frame t - j covers samples t*hop .. t*hop + hop - 1 at offsets j*hop ..
                y[t * hop:(t + 1) * hop] += F[t - j + taps - 1][j * hop:(j + 1) * hop]
        y /= np.tile(self.env, T)
        self.hist = F[F.shape[0] - (taps - 1):].copy() if taps > 1 else self.hist
        return y


def istft_full(spec: np.ndarray, n_fft: int, hop: int, mag_clip: float = 0.0) -> np.ndarray:
    """The whole sequence at once: y[n] = sum_t w x_t[n - t hop] / E[n mod hop]."""
    f = frames_windowed(spec, n_fft, mag_clip)
    T = f.shape[0]
    y = np.zeros(T * hop + n_fft)
    for t in range(T):
        y[t * hop:t * hop + n_fft] += f[t]
    y = y[:T * hop]
    return y / np.tile(envelope(n_fft, hop), T)
