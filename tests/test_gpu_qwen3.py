"""GPU parity of the Qwen3-TTS-12Hz-shaped decoder (Q=16 x 2048 x 512,
d=1024, 8 layers, window 72, stages 1536 -> 96, MRF k in {3, 7, 11})
through the C ABI.  The oracle checks: the 97-frame decode (25-frame chunk
with 72 frames of context), the first-audio frame and single-frame calls,
a subset of the 64 staggered streams and of the long-form streams, each on
the waveform and on the final conv's output before tanh (which most samples
of these random-weight decoders saturate); every other stream and frame is
checked by GPU chunked == GPU full, bit for bit."""
from __future__ import annotations

import numpy as np
import pytest

from gpu_helpers import assert_close, assert_close_pre_tanh, bits_equal, decode_batch, decode_stream_chunks
from oracle.oracle import OracleModel
from streaming_tts_vocoder_gb300 import codec as C
from streaming_tts_vocoder_gb300.synthetic import (make_codes, make_weights, pack_blob, qwen3_config,
                                                   staggered_schedule)

pytestmark = pytest.mark.gpu

PRECISIONS = [C.PRECISION_FP32, C.PRECISION_FP16X3]


@pytest.fixture(scope="module")
def qwen3():
    cfg = qwen3_config()
    blob = pack_blob(cfg, make_weights(cfg, 0))
    return cfg, blob


@pytest.fixture(scope="module")
def oracle97(qwen3):
    cfg, blob = qwen3
    codes = make_codes(cfg, 97, 0)
    om = OracleModel(cfg, blob)
    audio, pt = om.decode_full(codes, pre_tanh=True)
    return codes, audio, pt


def make_state(cfg, blob, precision, streams=1, chunk=97, batch=None):
    cod = C.Codec(cfg, blob, max_streams=streams, max_chunk_frames=chunk,
                  max_batch_frames=batch if batch is not None else streams * chunk, precision=precision)
    return cod.state()


@pytest.mark.parametrize("precision", PRECISIONS)
def test_97_frames_window_context(qwen3, oracle97, precision):
    """One 25-frame chunk with 72 frames of carried context: 97 frames in,
    the last 48,000 samples out; equal to decoding 72 frames then 25."""
    cfg, blob = qwen3
    codes, ref, ref_pt = oracle97
    st = make_state(cfg, blob, precision)
    (full,), (pt,) = decode_batch(st, [(0, codes)], pre_tanh=True)
    assert full.size == 97 * 1920
    assert_close(full[-48000:], ref[-48000:], "last 48,000 samples")
    assert_close(full, ref, "all 97 frames")
    assert_close_pre_tanh(pt, ref_pt, "97 frames")
    st.reset()
    warm = decode_batch(st, [(0, codes[:, :72])])[0]
    chunk = decode_batch(st, [(0, codes[:, 72:])])[0]
    assert chunk.size == 48000
    assert bits_equal(np.concatenate([warm, chunk]), full)
    assert st.query(0) == (97, 0)


@pytest.mark.parametrize("precision", PRECISIONS)
def test_first_audio_then_single_frames(qwen3, oracle97, precision):
    cfg, blob = qwen3
    codes, ref, ref_pt = oracle97
    st = make_state(cfg, blob, precision, chunk=25)
    (first,), (first_pt,) = decode_batch(st, [(0, codes[:, :1])], pre_tanh=True)
    assert first.size == 1920
    rest, rest_pt = decode_stream_chunks(st, 0, codes[:, 1:25], [1] * 24, pre_tanh=True)
    chunked = np.concatenate([first, rest])
    chunked_pt = np.concatenate([first_pt, rest_pt])
    st.reset()
    full = decode_batch(st, [(0, codes[:, :25])])[0]
    assert bits_equal(chunked, full)
    assert_close(chunked, ref[: 25 * 1920], "25 single-frame calls vs oracle")
    assert_close_pre_tanh(first_pt, ref_pt[:1920], "first-audio frame vs oracle")
    assert_close_pre_tanh(chunked_pt, ref_pt[: 25 * 1920], "25 single-frame calls vs oracle")


@pytest.mark.parametrize("precision", PRECISIONS)
def test_64_staggered_streams(qwen3, precision):
    """64 streams x 250 frames in ragged staggered ticks.  Every stream:
    chunked == its own full GPU decode bit for bit.  Against the oracle, on
    the waveform and before tanh, frames 0-51 of four streams with different
    start offsets (s mod 25 = 0, 13, 12, 24), so each crosses two tick
    boundaries inside the compared frames (at 25 and 50; 12 and 37; 13 and 38;
    1 and 26), with first chunks of 25, 12, 13 and 1 frames."""
    cfg, blob = qwen3
    S, F = 64, 250
    st = make_state(cfg, blob, precision, streams=S, chunk=F, batch=S * 25)
    codes = [make_codes(cfg, F, 1000 + s) for s in range(S)]
    out = [[] for _ in range(S)]
    out_pt = [[] for _ in range(S)]
    for tick in staggered_schedule(S, F, 25):
        entries = [(s, codes[s][:, a:a + n]) for s, a, n in tick]
        audio, pts = decode_batch(st, entries, T_max=25, pre_tanh=True)
        for (s, _), a, p in zip(entries, audio, pts):
            out[s].append(a)
            out_pt[s].append(p)
    got = [np.concatenate(o) for o in out]
    got_pt = [np.concatenate(o) for o in out_pt]
    for s in range(S):
        assert st.query(s) == (F, 0)
    st.reset()
    for s in range(S):
        full = decode_batch(st, [(s, codes[s])])[0]
        assert bits_equal(got[s], full), f"stream {s}: chunked != full"
    om = OracleModel(cfg, blob)
    n = 52
    for s in (0, 13, 37, 49):
        ref, ref_pt = om.decode_full(codes[s][:, :n], pre_tanh=True)
        assert_close(got[s][: n * 1920], ref, f"stream {s} frames 0-{n - 1}")
        assert_close_pre_tanh(got_pt[s][: n * 1920], ref_pt, f"stream {s} frames 0-{n - 1}")


@pytest.mark.parametrize("precision", PRECISIONS)
def test_long_form_8_streams(qwen3, precision):
    """8 streams x 3000 frames as 120 chunks of 25: chunked == one full GPU
    decode per stream, bit for bit; streams 0 and 7 against the oracle on
    their first frames."""
    cfg, blob = qwen3
    S, F = 8, 3000
    st = make_state(cfg, blob, precision, streams=S, chunk=F, batch=F)
    codes = [make_codes(cfg, F, 77 + s) for s in range(S)]
    out = [[] for _ in range(S)]
    out_pt = [[] for _ in range(S)]
    for c in range(F // 25):
        entries = [(s, codes[s][:, c * 25:(c + 1) * 25]) for s in range(S)]
        audio, pts = decode_batch(st, entries, pre_tanh=True)
        for s in range(S):
            out[s].append(audio[s])
            if c < 2:
                out_pt[s].append(pts[s])
    got = [np.concatenate(o) for o in out]
    st.reset()
    for s in range(S):
        full = decode_batch(st, [(s, codes[s])])[0]
        assert bits_equal(got[s], full), f"stream {s}: chunked != full"
    om = OracleModel(cfg, blob)
    for s in (0, 7):
        ref, ref_pt = om.decode_full(codes[s][:, :30], pre_tanh=True)
        assert_close(got[s][: 30 * 1920], ref, f"stream {s} frames 0-29")
        assert_close_pre_tanh(np.concatenate(out_pt[s])[: 30 * 1920], ref_pt, f"stream {s} frames 0-29")
