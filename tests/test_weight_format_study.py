"""The blixt/phonon int8 weight format (one f16 scale per 32 values along rows)
on the decoder: pins of the quantiser, then what it costs against the
float64 oracle with the original weights (rel-L2 and PCM SNR of the
waveform), on the tiny and the Qwen3-shaped decoders.  CPU only."""
from __future__ import annotations

import numpy as np
import pytest

from oracle import weights_int8 as Q
from oracle.oracle import OracleModel
from streaming_tts_vocoder_gb300.synthetic import make_codes, make_weights, pack_blob, qwen3_config, tiny_config


def test_group_scale_and_round_half_even():
    # one group: max 1.27 -> scale f16(0.01); 0.015 is 1.5 steps, 0.025 is 2.5: both round to 2
    row = np.zeros((1, 32))
    row[0, 0], row[0, 1], row[0, 2] = 1.27, 0.015, 0.025
    scale = float(np.float16(float(np.float16(1.27)) / 127))     # from the f16-rounded values
    got = Q.quantize_rows(row)[0]
    assert got[0] == np.clip(np.rint(float(np.float16(1.27)) / scale), -127, 127) * scale
    assert got[1] == np.rint(float(np.float16(0.015)) / scale) * scale
    assert got[2] == np.rint(float(np.float16(0.025)) / scale) * scale
    # a value exactly half a step above an even multiple rounds down to the even one
    s = 2.0 ** -6
    row2 = np.zeros((1, 32))
    row2[0, 0] = 127 * s
    row2[0, 1] = 4.5 * s
    row2[0, 2] = 5.5 * s
    got2 = Q.quantize_rows(row2)[0]
    assert got2[1] == 4 * s and got2[2] == 6 * s


def test_groups_are_independent_and_bounded():
    rng = np.random.default_rng(0)
    row = np.concatenate([rng.normal(0, 1e-3, 32), rng.normal(0, 10, 32)])[None]
    got = Q.quantize_rows(row)[0]
    v = Q.f16(row)[0]
    for g in (0, 32):
        scale = float(np.float16(np.abs(v[g:g + 32]).max() / 127))
        assert np.abs(got[g:g + 32] - v[g:g + 32]).max() <= scale / 2 * (1 + 1e-12)
    assert np.abs(got[:32]).max() < 1e-2          # the small group kept its own fine scale


@pytest.mark.parametrize("name,shape", [("st.0.w", (16, 8, 6)), ("up.0.w", (8, 8, 4)), ("st.0.rb.0.0.w", (8, 8, 3)),
                                        ("tf.0.wq", (8, 8)), ("cb.0", (16, 4)), ("st.0.alpha", (8,))])
def test_layouts_round_trip(name, shape):
    a = np.random.default_rng(1).standard_normal(int(np.prod(shape)))
    rows, back = Q.to_rows(name, a, shape)
    assert np.array_equal(back(rows).reshape(-1), a)


def test_conv_rows_group_tap_then_input():
    """A conv's groups run over (tap, in) of one output: a large weight at
    (out 0, in 5, tap 1) raises the scale of out 0's group holding tap 1, in 5
    only."""
    co, ci, k = 2, 32, 3
    w = np.full((co, ci, k), 0.01)
    w[0, 5, 1] = 5.0
    rows, back = Q.to_rows("st.0.rb.0.0.w", w.reshape(-1), (co, ci, k))
    q = back(Q.quantize_rows(rows)).reshape(co, ci, k)
    coarse = np.abs(q - Q.f16(w)) > 1e-4
    assert coarse[0, :, 1].any() and not coarse[0, :, 0].any() and not coarse[0, :, 2].any()
    assert not coarse[1].any()


def snr_db(got, ref):
    return float(10 * np.log10(np.sum(ref ** 2) / np.sum((got - ref) ** 2)))


@pytest.mark.parametrize("which,frames", [("tiny", 8), ("qwen3", 4)])
def test_study_decoder_error(which, frames, capsys):
    cfg = tiny_config() if which == "tiny" else qwen3_config()
    blob = pack_blob(cfg, make_weights(cfg, 0))
    codes = make_codes(cfg, frames, 0)
    ref = OracleModel(cfg, blob).decode_full(codes)
    got = OracleModel(cfg, Q.quantize_blob(cfg, blob)).decode_full(codes)
    rel = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
    with capsys.disabled():
        print(f"\n{which} decoder, {frames} frames, int8 per-32 weights: rel-L2 {rel:.3e}, "
              f"max|err| {np.abs(got - ref).max():.3e}, SNR {snr_db(got, ref):.1f} dB")
    assert np.isfinite(rel) and rel < 1.0
