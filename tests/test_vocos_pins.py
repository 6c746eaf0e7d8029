"""Pins of the Vocos-style generator oracle (oracle/vocos.py), CPU only.

  * the backbone against an independent float64 PyTorch composition of
    library routines (conv1d with left padding, grouped conv1d, layer_norm,
    exact GELU, linear), the spectrum compared directly;
  * the waveform against the iSTFT oracle applied to that spectrum (the head
    itself is pinned in test_istft_pins.py);
  * LayerNorm's textbook properties (zero mean, unit variance before the
    affine part);
  * chunked decoding equal to a full decode bit for bit, for several splits;
  * causality: a change in mel frame t0 leaves every sample before t0 * hop alone;
  * planted mistakes (depthwise taps reversed, layer scale dropped) fail the
    composition pin.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import istft as OI
from oracle import vocos as V
from streaming_tts_vocoder_gb300.synthetic import make_mels, make_vocos_weights, tiny_vocos_config, vocos_config


def torch_spectrum(cfg, W, mel, flip_dw=False, drop_gamma=False):
    t = lambda a: torch.from_numpy(np.asarray(a, np.float64))
    x = t(mel).t()[None]                                              # [1][n_mels][T]
    k = cfg.k
    h = F.conv1d(F.pad(x, (k - 1, 0)), t(W["embed.w"]), t(W["embed.b"]))[0].t()
    h = F.layer_norm(h, (cfg.d,), t(W["norm.g"]), t(W["norm.b"]), cfg.ln_eps)
    for l in range(cfg.layers):
        p = f"blk.{l}."
        dw = t(W[p + "dw.w"])
        if flip_dw:
            dw = dw.flip(-1)
        y = F.conv1d(F.pad(h.t()[None], (k - 1, 0)), dw, t(W[p + "dw.b"]), groups=cfg.d)[0].t()
        y = F.layer_norm(y, (cfg.d,), t(W[p + "ln.g"]), t(W[p + "ln.b"]), cfg.ln_eps)
        y = F.gelu(F.linear(y, t(W[p + "pw1.w"]), t(W[p + "pw1.b"])))
        y = F.linear(y, t(W[p + "pw2.w"]), t(W[p + "pw2.b"]))
        h = h + (y if drop_gamma else t(W[p + "gamma"]) * y)
    h = F.layer_norm(h, (cfg.d,), t(W["final.g"]), t(W["final.b"]), cfg.ln_eps)
    return F.linear(h, t(W["head.w"]), t(W["head.b"])).numpy()


def relerr(a, b):
    return float(np.linalg.norm(np.asarray(a) - np.asarray(b)) / np.linalg.norm(np.asarray(b)))


@pytest.mark.parametrize("make", [tiny_vocos_config, vocos_config])
def test_backbone_matches_torch_composition(make):
    cfg = make()
    W = make_vocos_weights(cfg, 0)
    mel = make_mels(cfg, 12, 1)
    spec = V.VocosStream(cfg, W).spectrum(mel)
    want = torch_spectrum(cfg, W, mel)
    assert relerr(spec, want) < 1e-12
    audio = V.decode_full(cfg, W, mel)
    assert audio.size == 12 * cfg.hop
    assert relerr(audio, OI.istft_full(want, cfg.n_fft, cfg.hop, cfg.mag_clip)) < 1e-12


def test_layer_norm_textbook():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((5, 64)) * 3 + 2
    y = V.layer_norm(x, np.ones(64), np.zeros(64), 0.0)
    assert np.allclose(y.mean(axis=1), 0, atol=1e-12)
    assert np.allclose((y ** 2).mean(axis=1), 1, atol=1e-12)


@pytest.mark.parametrize("splits", [[1] * 10, [3, 7], [10], [4, 4, 2]])
def test_chunked_equals_full_bit_exact(splits):
    cfg = tiny_vocos_config()
    W = make_vocos_weights(cfg, 0)
    mel = make_mels(cfg, 10, 2)
    full = V.decode_full(cfg, W, mel)
    st = V.VocosStream(cfg, W)
    parts, i = [], 0
    for n in splits:
        parts.append(st.decode(mel[i:i + n]))
        i += n
    assert np.array_equal(np.concatenate(parts), full)


def test_causality():
    cfg = tiny_vocos_config()
    W = make_vocos_weights(cfg, 0)
    mel = make_mels(cfg, 10, 3)
    a = V.decode_full(cfg, W, mel)
    mel2 = mel.copy()
    mel2[6] += 1.0
    b = V.decode_full(cfg, W, mel2)
    assert np.array_equal(a[: 6 * cfg.hop], b[: 6 * cfg.hop])
    assert not np.array_equal(a[6 * cfg.hop:], b[6 * cfg.hop:])


@pytest.mark.parametrize("mistake", ["flip_dw", "drop_gamma"])
def test_pins_catch_planted_mistakes(mistake):
    cfg = tiny_vocos_config()
    W = make_vocos_weights(cfg, 0)
    mel = make_mels(cfg, 8, 1)
    spec = V.VocosStream(cfg, W).spectrum(mel)
    bad = torch_spectrum(cfg, W, mel, **{mistake: True})
    assert relerr(spec, bad) > 1e-3
