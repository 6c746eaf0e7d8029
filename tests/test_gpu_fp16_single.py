"""The single-pass fp16 tensor-core mode (CODEC_PRECISION_FP16) through the
C ABI.  It is approximate by design: both operands of every contraction are
rounded to fp16 once, which on the random-weight decoders costs about 1e-2 of
relative L2 error on the waveform (an operand rounding of 2^-11, amplified
by the network), ten times the bound the exact modes meet.  So these tests
pin what the mode does guarantee: the error against the oracle stays at the
size that rounding explains (well under 0.1, above the exact modes' 1e-3),
the output is finite and in tanh's range, the bookkeeping is exact, and
chunked decoding equals a full decode bit for bit."""
from __future__ import annotations

import numpy as np
import pytest

from gpu_helpers import bits_equal, decode_batch, decode_stream_chunks, relerr
from oracle.oracle import OracleModel
from streaming_tts_vocoder_gb300 import codec as C
from streaming_tts_vocoder_gb300.synthetic import make_codes, make_weights, pack_blob, qwen3_config, tiny_config

pytestmark = pytest.mark.gpu

APPROX_REL = 0.1


@pytest.mark.parametrize("name,T", [("tiny", 8), ("qwen3", 4)])
def test_single_pass_error_is_rounding_sized(name, T):
    cfg = tiny_config() if name == "tiny" else qwen3_config()
    blob = pack_blob(cfg, make_weights(cfg, 0))
    codes = make_codes(cfg, T, 0)
    want = OracleModel(cfg, blob).decode_full(codes)
    st = C.Codec(cfg, blob, max_streams=1, max_chunk_frames=T, precision=C.PRECISION_FP16).state()
    (got,) = decode_batch(st, [(0, codes)])
    assert got.size == T * 1920
    assert np.isfinite(got).all() and np.abs(got).max() <= 1.0
    err = relerr(got, want)
    assert err < APPROX_REL, err
    frames, bits = st.query(0)
    assert frames == T and bits == 0


def test_single_pass_chunked_equals_full():
    cfg = qwen3_config()
    blob = pack_blob(cfg, make_weights(cfg, 0))
    codes = make_codes(cfg, 12, 3)
    st = C.Codec(cfg, blob, max_streams=1, max_chunk_frames=12, precision=C.PRECISION_FP16).state()
    (full,) = decode_batch(st, [(0, codes)])
    st.reset()
    chunked = decode_stream_chunks(st, 0, codes, [1, 4, 7])
    assert bits_equal(chunked, full)
