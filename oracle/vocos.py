"""CPU oracle of a Vocos-style generator feeding the streaming iSTFT head
(test infrastructure only: tests, the smoke check and the bench's CPU
baseline use it; the CUDA library never does).

vox's F5-TTS pipeline ends in "Vocos -> iSTFT"; the pages fix nothing of
Vocos itself, so this follows the public Vocos architecture, made causal for
streaming the way the decoder's convolutions are (left context carried, no
look-ahead):

  h = LayerNorm(causal_conv_k(mel) + b)                      embedding
  per block: h = h + gamma * (W2 GELU(W1 LayerNorm(dwconv_k(h) + b_dw) + b1) + b2)
  spec = W_head LayerNorm(h) + b_head                        n_bins log-magnitudes, n_bins phases
  audio = iSTFT head (oracle/istft.py: exp, clip, irfft, Hann, overlap-add)

Every step in float64 (numpy), in the order written; LayerNorm over the
channels with biased variance and eps inside the square root; GELU in its erf
form.  Products with a weight matrix are formed row by row as explicit
products summed over the input channels in ascending order (no BLAS call,
whose rounding can depend on how many rows it is given), so a row's result
never depends on the chunk it came in.  Streaming: the embedding conv carries its last k - 1 mel rows, each
block's depthwise conv the last k - 1 rows of its input, the head its
carried frames, so chunked decoding equals a full decode bit for bit.
"""
from __future__ import annotations

import math

import numpy as np

from .istft import IstftStream


def layer_norm(x, g, b, eps):
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + eps) * g + b


_erf = np.vectorize(math.erf, otypes=[np.float64])


def gelu(x):
    return 0.5 * x * (1.0 + _erf(x / math.sqrt(2.0)))


def rows_times(x, wt):
    """x [T][K] times wt [K][N], each output row summed over k ascending."""
    x = np.asarray(x, np.float64)
    wt = np.asarray(wt, np.float64)
    out = np.empty((x.shape[0], wt.shape[1]))
    for i in range(x.shape[0]):
        acc = np.zeros(wt.shape[1])
        for kk in range(wt.shape[0]):
            acc += x[i, kk] * wt[kk]
        out[i] = acc
    return out


def linear(x, w, b):
    """y = x W^T + b, W [N][K]."""
    return rows_times(x, np.asarray(w, np.float64).T) + b


def causal_conv(x_ext, w, b):
    """x_ext [(k-1) + T][Cin] (history first), w [Cout][Cin][k]:
    y[t][co] = b[co] + sum_j sum_ci w[co][ci][j] x_ext[t + j][ci]."""
    Cout, Cin, k = w.shape
    T = x_ext.shape[0] - (k - 1)
    y = np.tile(np.asarray(b, np.float64), (T, 1))
    for j in range(k):
        y += rows_times(x_ext[j:j + T], np.asarray(w[:, :, j], np.float64).T)
    return y


def depthwise_causal_conv(x_ext, w, b):
    """x_ext [(k-1) + T][C], w [C][1][k]: y[t][c] = b[c] + sum_j w[c][0][j] x_ext[t + j][c]."""
    C, _, k = w.shape
    T = x_ext.shape[0] - (k - 1)
    y = np.tile(np.asarray(b, np.float64), (T, 1))
    for j in range(k):
        y += x_ext[j:j + T] * np.asarray(w[:, 0, j], np.float64)
    return y


class VocosStream:
    """One stream's carried state: the embedding conv's mel rows, each
    block's depthwise-conv input rows, the iSTFT head's carried frames."""

    def __init__(self, cfg, W):
        self.cfg, self.W = cfg, {k: np.asarray(v, np.float64) for k, v in W.items()}
        self.reset()

    def reset(self):
        c = self.cfg
        self.h_mel = np.zeros((c.k - 1, c.n_mels))
        self.h_dw = [np.zeros((c.k - 1, c.d)) for _ in range(c.layers)]
        self.head = IstftStream(c.n_fft, c.hop, c.mag_clip)
        self.frames = 0

    @staticmethod
    def _carry(hist, x):
        ext = np.concatenate([hist, x], axis=0)
        return ext, ext[ext.shape[0] - hist.shape[0]:].copy()

    def spectrum(self, mel):
        """mel [T][n_mels] -> spec [T][2 n_bins] (advances the backbone state)."""
        c, W = self.cfg, self.W
        x = np.asarray(mel, np.float64)
        ext, self.h_mel = self._carry(self.h_mel, x)
        h = layer_norm(causal_conv(ext, W["embed.w"], W["embed.b"]), W["norm.g"], W["norm.b"], c.ln_eps)
        for l in range(c.layers):
            p = f"blk.{l}."
            ext, self.h_dw[l] = self._carry(self.h_dw[l], h)
            y = depthwise_causal_conv(ext, W[p + "dw.w"], W[p + "dw.b"])
            y = layer_norm(y, W[p + "ln.g"], W[p + "ln.b"], c.ln_eps)
            y = gelu(linear(y, W[p + "pw1.w"], W[p + "pw1.b"]))
            y = linear(y, W[p + "pw2.w"], W[p + "pw2.b"])
            h = h + W[p + "gamma"] * y
        h = layer_norm(h, W["final.g"], W["final.b"], c.ln_eps)
        return linear(h, W["head.w"], W["head.b"])

    def decode(self, mel):
        """mel [T][n_mels] -> audio [T hop]."""
        spec = self.spectrum(mel)
        self.frames += spec.shape[0]
        return self.head.decode(spec)


def decode_full(cfg, W, mel):
    return VocosStream(cfg, W).decode(mel)
