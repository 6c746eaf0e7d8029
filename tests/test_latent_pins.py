"""Pins of the latent-input (Mimi-style) decoder variant of the oracle
(blixt/phonon "Weights": denormalise, 1x1 projection without bias, depthwise
x16 transposed-conv upsampling of the codec latents; "Speed" item 7: the codec
transformer at 200 Hz with a 251-position window over a 512-position ring,
chunks of 1, 2, 4 and 8 frames sharing one state).  CPU only.

  * the depthwise causal transposed conv against the library's grouped
    conv_transpose1d (float64, right-trimmed) and its scatter definition;
  * the fold the GPU uses: the projection merged into the upsampling taps,
    one phase GEMM over [z[n-1] | z[n]], equals the three steps in float64;
  * the whole variant against an independent float64 PyTorch composition
    (oracle-check size and the Mimi-shaped size);
  * chunks of 1, 2, 4, 8 frames (and any split) equal a full decode bit for bit;
  * the page's numbers: 12.5 Hz x 16 = 200 Hz, and the ring that holds a
    chunk of up to 8 frames plus the 250 earlier positions is 512 rows;
  * planted mistakes (a tap off by one phase, the history row dropped) fail.
"""
from __future__ import annotations

import json
from pathlib import Path

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import torch_ref_f64 as R
from oracle import oracle as O
from streaming_tts_vocoder_gb300.synthetic import (make_latents, make_weights, mimi_config, pack_blob,
                                                   tiny_mimi_config)

GOLDEN = json.loads((Path(__file__).parent / "golden" / "page_facts.json").read_text())


def relerr(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


@pytest.mark.parametrize("C,s,T", [(8, 16, 5), (3, 5, 7), (64, 2, 9)])
def test_depthwise_convt_matches_library_and_scatter(C, s, T):
    rng = np.random.default_rng(C * 100 + s)
    x = rng.standard_normal((1 + T, C)).astype(np.float32)
    u = rng.standard_normal((C, 1, 2 * s)).astype(np.float32)
    b = rng.standard_normal(C).astype(np.float32)
    got = O.dw_conv_t(x, u, b, s)
    # library: grouped conv_transpose1d over [history | chunk], drop the s
    # outputs the history row alone makes and the k - s tail
    lib = F.conv_transpose1d(torch.from_numpy(x.T.astype(np.float64))[None], torch.from_numpy(u.astype(np.float64)),
                             torch.from_numpy(b.astype(np.float64)), stride=s, groups=C)[0].numpy().T
    want = lib[s: s + T * s]
    assert relerr(got, want) < 1e-6
    # scatter definition: input row i (history = -1) adds u[c][j] x[i][c] to output i s + j
    sc = np.zeros(((T + 2) * s, C))
    for i in range(-1, T):
        for j in range(2 * s):
            sc[(i + 1) * s + j] += u[:, 0, j] * x[i + 1]
    assert relerr(got, sc[s: s + T * s] + b) < 1e-6


def test_fold_of_projection_into_upsampling_is_exact():
    """y[n s + p][c] = b[c] + sum_l (u[c][p+s] Wp[c][l]) z[n-1][l] + (u[c][p] Wp[c][l]) z[n][l]:
    the folded phase GEMM (K = 2 L, N = s d) the GPU runs, in float64, equals the
    oracle's denormalise -> project -> depthwise-upsample front end."""
    cfg = tiny_mimi_config()
    W = make_weights(cfg, 1)
    x = make_latents(cfg, 6, 2).astype(np.float64)
    L, d, s = cfg.latent_dim, cfg.d, cfg.tf_up
    z = x * W["lat.sigma"] + W["lat.mu"]
    zp = np.vstack([np.zeros((1, L)), z])                    # history row: zero after reset
    u, Wp, b = W["lat.up.w"][:, 0, :].astype(np.float64), W["lat.proj"].astype(np.float64), W["lat.up.b"]
    A0 = np.einsum("cp,cl->lpc", u[:, s:], Wp).reshape(L, s * d)    # tap on z[n-1]
    A1 = np.einsum("cp,cl->lpc", u[:, :s], Wp).reshape(L, s * d)    # tap on z[n]
    folded = (zp[:-1] @ A0 + zp[1:] @ A1).reshape(-1, d) + b
    taps = {}
    R.decode_latents(cfg, W, x.astype(np.float32), taps=taps)
    front = taps["front"].numpy()
    assert relerr(folded, front) < 1e-12


@pytest.fixture(scope="module")
def tiny_mimi():
    cfg = tiny_mimi_config()
    W = make_weights(cfg, 0)
    return cfg, W, O.OracleModel(cfg, pack_blob(cfg, W))


def test_latent_decoder_matches_torch_composition(tiny_mimi):
    cfg, W, m = tiny_mimi
    x = make_latents(cfg, 6, 3)
    a, pt = m.decode_latents_full(x, pre_tanh=True)
    taps = {}
    ref = R.decode_latents(cfg, W, x, taps=taps)
    assert a.size == 6 * 1920
    assert relerr(pt, taps["pre_tanh"].numpy()) < 1e-5
    assert relerr(a, ref.numpy()) < 1e-4


def test_mimi_shaped_decoder_matches_torch_composition():
    cfg = mimi_config()
    W = make_weights(cfg, 0)
    m = O.OracleModel(cfg, pack_blob(cfg, W))
    x = make_latents(cfg, 3, 4)
    a, pt = m.decode_latents_full(x, pre_tanh=True)
    taps = {}
    R.decode_latents(cfg, W, x, taps=taps)
    assert relerr(pt, taps["pre_tanh"].numpy()) < 1e-5


@pytest.mark.parametrize("splits", [[1, 2, 4, 8], [1] * 15, [8, 7], [15], [3, 5, 7]])
def test_latent_chunked_equals_full_bit_exact(tiny_mimi, splits):
    cfg, W, m = tiny_mimi
    x = make_latents(cfg, 15, 9)
    full = m.decode_latents_full(x)
    st = m.stream()
    parts, i = [], 0
    for n in splits:
        parts.append(st.decode_latents(x[i:i + n]))
        i += n
    assert np.array_equal(np.concatenate(parts).view(np.uint32), full.view(np.uint32))
    assert st.frames == 15


def test_page_numbers_of_the_phonon_codec():
    cfg = mimi_config()
    assert cfg.window == GOLDEN["phonon_codec_window"]["value"]
    assert 12.5 * cfg.tf_up == GOLDEN["phonon_codec_transformer_rate_hz"]["value"]
    assert cfg.tf_up == GOLDEN["phonon_latent_upsample"]["value"]
    assert cfg.samples_per_frame == 1920
    # the GPU's ring holds the largest chunk plus the W - 1 earlier positions,
    # rounded up to a power of two: the page's 512 positions at 200 Hz
    biggest = max(GOLDEN["phonon_chunk_frames"]["value"]) * cfg.tf_up
    need = biggest + cfg.window - 1
    ring = 1 << (need - 1).bit_length()
    assert ring == GOLDEN["phonon_codec_ring_positions"]["value"]


def test_pins_catch_a_wrong_upsampling_tap():
    """Planted mistake, in a copy of the oracle's front end: the history row
    multiplied by tap p instead of p + s.  The library pin rejects it."""
    rng = np.random.default_rng(0)
    C, s, T = 4, 16, 3
    x = rng.standard_normal((1 + T, C)).astype(np.float32)
    u = rng.standard_normal((C, 1, 2 * s)).astype(np.float32)
    b = np.zeros(C, np.float32)
    bad = np.zeros((T * s, C))
    for m_ in range(T * s):
        n, p = divmod(m_, s)
        bad[m_] = u[:, 0, p] * x[n] + u[:, 0, p] * x[n + 1]
    lib = F.conv_transpose1d(torch.from_numpy(x.T.astype(np.float64))[None], torch.from_numpy(u.astype(np.float64)),
                             torch.from_numpy(b.astype(np.float64)), stride=s, groups=C)[0].numpy().T[s: s + T * s]
    assert relerr(bad, lib) > 1e-2
    assert relerr(O.dw_conv_t(x, u, b, s), lib) < 1e-6


def test_pins_catch_a_dropped_history_row(tiny_mimi):
    """Planted mistake: decoding a chunk without the carried projected row
    (a fresh stream for the second chunk) breaks chunked == full."""
    cfg, W, m = tiny_mimi
    x = make_latents(cfg, 4, 1)
    full = m.decode_latents_full(x)
    a = m.decode_latents_full(x[:2])
    b = m.decode_latents_full(x[2:])
    assert not np.array_equal(np.concatenate([a, b]), full)
