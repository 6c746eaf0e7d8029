"""CPU oracle of the harmonic sine source and the streaming analysis STFT (test
infrastructure only: the tests and the bench's CPU baseline use it).

The pages give the source path of the iSTFT-head vocoders as "har =
STFT(SineGen(f0_upsamp(F0)))" (the Core AI Kokoro note: the hn-NSF excitation
behind iSTFTNet, also HiFT's "F0 -> NSF source"), and nothing more.  The
plainest reading, every step written out:

Sine source (per stream, F0 in Hz per frame, `upp` samples per frame, sample
rate fs, H harmonics, amplitude A, voiced when F0 > threshold):
  * the frame's F0 is held for its upp samples (nearest upsampling);
  * the per-sample phase increment in cycles is quantised to 2^-32:
    D = rint(F0 * (2^32 / fs)) as an integer (2^32 / fs in float64, round half
    to even; F0 clamped to [0, fs / 2]), so that the phase is an exact integer
    running sum;
  * the phase of sample n is P[n] = (P[-1] + sum_{m <= n} D[m]) mod 2^32 (the
    increment of sample n included), carried between chunks; harmonic h has
    phase h P[n] mod 2^32;
  * out[n][h-1] = A sin(2 pi (h P[n] mod 2^32) / 2^32) where voiced, else 0.

Analysis STFT (causal, per stream): frame t covers input samples
[(t+1) hop - n_fft, (t+1) hop) (samples before the stream's start are zero),
times the periodic Hann window w[m] = sin^2(pi m / n_fft); its output is
X_t[k] = sum_m w[m] x[m] exp(-2 pi i k m / n_fft), k = 0 .. n_fft / 2, stored
as n_fft / 2 + 1 real parts then as many imaginary parts.  Every hop of input
yields one frame; the last n_fft - hop input samples are carried.  Fed to the
iSTFT head (as log-magnitude and phase) it gives the input back delayed by
n_fft - hop samples.
"""
from __future__ import annotations

import numpy as np

TWO32 = 4294967296


def phase_increments(f0: np.ndarray, fs: float) -> np.ndarray:
    """D = rint(min(max(F0, 0), fs / 2) * (2^32 / fs)) per frame, as int64
    (float64 arithmetic; fs is the float32 configuration value)."""
    fs64 = np.float64(np.float32(fs))
    scale = np.float64(TWO32) / fs64
    f = np.clip(np.asarray(f0, dtype=np.float32).astype(np.float64), 0.0, fs64 / 2)
    return np.rint(f * scale).astype(np.int64)


class SineSource:
    def __init__(self, upp: int, fs: float, harmonics: int, amplitude: float, threshold: float = 0.0):
        # amplitude, threshold and fs are float32 configuration values
        self.upp, self.fs, self.H = upp, fs, harmonics
        self.A, self.thr = float(np.float32(amplitude)), np.float32(threshold)
        self.phase = 0            # P[-1], an integer in [0, 2^32)

    def reset(self):
        self.phase = 0

    def decode(self, f0: np.ndarray) -> np.ndarray:
        f0 = np.asarray(f0, dtype=np.float32).reshape(-1)
        D = np.repeat(phase_increments(f0, self.fs), self.upp)
        voiced = np.repeat(f0 > self.thr, self.upp)
        P = (self.phase + np.cumsum(D)) % TWO32
        if P.size:
            self.phase = int(P[-1])
        h = np.arange(1, self.H + 1, dtype=np.int64)
        Ph = (P[:, None] * h[None, :]) % TWO32
        out = self.A * np.sin(2.0 * np.pi * Ph.astype(np.float64) / TWO32)
        return np.where(voiced[:, None], out, 0.0)


def hann_periodic(n_fft: int) -> np.ndarray:
    m = np.arange(n_fft, dtype=np.float64)
    return np.sin(np.pi * m / n_fft) ** 2


class StftStream:
    def __init__(self, n_fft: int, hop: int):
        if n_fft % hop:
            raise ValueError("hop must divide n_fft")
        self.n_fft, self.hop = n_fft, hop
        self.hist = np.zeros(n_fft - hop)    # the last n_fft - hop input samples

    def reset(self):
        self.hist[:] = 0.0

    def decode(self, x: np.ndarray) -> np.ndarray:
        """x: a whole number of hops of input; returns [frames][2 (n_fft / 2 + 1)]."""
        x = np.asarray(x, dtype=np.float64).reshape(-1)
        if x.size % self.hop:
            raise ValueError("input must be a whole number of hops")
        buf = np.concatenate([self.hist, x])
        T = x.size // self.hop
        w = hann_periodic(self.n_fft)
        frames = np.stack([buf[t * self.hop:t * self.hop + self.n_fft] * w for t in range(T)]) if T else \
            np.zeros((0, self.n_fft))
        X = np.fft.rfft(frames, axis=1)
        if self.n_fft > self.hop:
            self.hist = buf[buf.size - (self.n_fft - self.hop):].copy()
        return np.concatenate([X.real, X.imag], axis=1)
