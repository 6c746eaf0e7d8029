"""The int8-per-32 weight file (blixt/phonon "Weights" format) that
codec_create_q8 reads: the converter's output, read back by the layout
stated in include/codec.h, must give exactly the values of the oracle's own
restatement of the format (oracle/weights_int8.quantize_blob), tensor by
tensor; and its size must be the library's codec_q8_bytes.  CPU only."""
from __future__ import annotations

import numpy as np
import pytest

from oracle import weights_int8 as OQ
from streaming_tts_vocoder_gb300 import build as B
from streaming_tts_vocoder_gb300 import codec as C
from streaming_tts_vocoder_gb300.synthetic import make_weights, pack_blob, qwen3_config, tiny_config, weight_manifest
from streaming_tts_vocoder_gb300.weights_q8 import pack_q8


def read_q8(cfg, data: bytes) -> np.ndarray:
    """Expand the file to the fp32 blob by the documented layout."""
    out, off = [], 0
    pad = lambda n: (n + 3) & ~3
    for t in weight_manifest(cfg):
        if t.size < 16384:
            out.append(np.frombuffer(data, np.float16, t.size, off).astype(np.float32))
            off += pad(2 * t.size)
            continue
        shape = t.shape
        transposed = len(shape) == 3 and (t.name.startswith("up.") or (t.name.startswith("st.") and ".rb." not in t.name))
        if transposed:
            cin, cout, k = shape
            R, L = cout, cin * k
        elif len(shape) == 3:
            R, L = shape[0], shape[1] * shape[2]
        else:
            R, L = shape
        G = -(-L // 32)
        q = np.frombuffer(data, np.int8, R * L, off).reshape(R, L).astype(np.float32)
        off += pad(R * L)
        sc = np.frombuffer(data, np.float16, R * G, off).reshape(R, G).astype(np.float32)
        off += pad(2 * R * G)
        v = q * np.repeat(sc, 32, axis=1)[:, :L]
        if transposed:
            s = k // 2
            v = v.reshape(cout, s, 2, cin).transpose(3, 0, 2, 1).reshape(shape)   # [out][p][j][in] -> [in][out][j s + p]
        elif len(shape) == 3:
            v = v.reshape(shape[0], shape[2], shape[1]).transpose(0, 2, 1)        # [out][tap][in] -> [out][in][tap]
        out.append(v.reshape(-1))
    assert off == len(data)
    return np.concatenate(out)


@pytest.fixture(scope="module", autouse=True)
def lib():
    B.build()
    return C._lib()


@pytest.mark.parametrize("make", [tiny_config, qwen3_config])
def test_file_matches_the_oracle_format_bit_for_bit(make):
    cfg = make()
    blob = pack_blob(cfg, make_weights(cfg, 0))
    data = pack_q8(cfg, blob)
    assert len(data) == C.q8_bytes(C.config_c(cfg))
    got = read_q8(cfg, data)
    want = OQ.quantize_blob(cfg, blob)
    assert got.dtype == np.float32 and want.dtype == np.float32
    # an int8 code has no negative zero: a small negative value that rounds to
    # code 0 reads back as +0, where the oracle's float arithmetic keeps -0;
    # adding +0 maps -0 to +0 and leaves every other value's bits alone
    assert np.array_equal((got + np.float32(0)).view(np.uint32), (want + np.float32(0)).view(np.uint32))


def test_size_is_about_a_quarter_of_fp32():
    cfg = qwen3_config()
    n = C.q8_bytes(C.config_c(cfg))
    assert 0.25 < n / (4 * C.weight_floats(C.config_c(cfg))) < 0.30
