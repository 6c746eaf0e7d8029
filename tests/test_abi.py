"""Host-side checks of the C-ABI library (no GPU needed): it builds, loads,
exports every function include/codec.h declares, and its host-only logic
(config validation, blob sizing, status strings) behaves."""
from __future__ import annotations

import ctypes

import pytest

from streaming_tts_vocoder_gb300 import build as B
from streaming_tts_vocoder_gb300 import codec as C
from streaming_tts_vocoder_gb300.synthetic import blob_size, qwen3_config, tiny_config


@pytest.fixture(scope="module")
def lib():
    B.build()
    return C._lib()


def test_exports_every_declared_function(lib):
    names = C.header_functions()
    assert "codec_decode_chunk" in names and "codec_create" in names and "codec_state_reset" in names
    assert "codec_conv1d_noalloc" in names and "codec_state_conv1d" in names
    raw = ctypes.CDLL(str(C.LIB_PATH))
    missing = [n for n in names if not hasattr(raw, n)]
    assert not missing, missing


@pytest.mark.parametrize("make", [tiny_config, qwen3_config])
def test_weight_floats_match_manifest(lib, make):
    cfg = make()
    assert C.weight_floats(C.config_c(cfg)) == blob_size(cfg)


def test_invalid_configs_rejected(lib):
    base = C.config_c(tiny_config())
    assert C.weight_floats(base) > 0
    bad = [
        ("heads", 5),          # d % heads != 0
        ("window", 0),
        ("window", 257),       # the attention kernel takes windows up to 256
        ("up_k", 3),           # kernel must be 2 * stride
        ("E", 6),              # channel counts are multiples of 4
        ("max_batch_frames", 1),
        ("precision", 7),
        ("n_rb", 4),
    ]
    for field, val in bad:
        c = C.config_c(tiny_config())
        setattr(c, field, val)
        assert C.weight_floats(c) == -1, field


def test_status_strings(lib):
    for s in range(9):
        assert lib.codec_status_string(s)
    assert lib.codec_status_string(0) == b"ok"


def test_null_arguments_rejected_without_device(lib):
    h = ctypes.c_void_p()
    assert lib.codec_create(None, None, 0, ctypes.byref(h)) == 1          # CODEC_ERR_NULL
    assert lib.codec_state_create(None, 0, ctypes.byref(h)) == 1
    assert lib.codec_decode_chunk(None, None, None, None, 1, 1, None, None) == 1
    assert lib.codec_state_reset(None, None, 0, None) == 1
    assert lib.codec_samples_per_frame(None) == 0


def test_create_rejects_wrong_blob_length(lib):
    import numpy as np
    cfg = C.config_c(tiny_config())
    n = C.weight_floats(cfg)
    blob = np.zeros(n - 1, np.float32)
    h = ctypes.c_void_p()
    st = lib.codec_create(ctypes.byref(cfg), blob.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), n - 1,
                          ctypes.byref(h))
    assert st == 3 and not h.value                                         # CODEC_ERR_WEIGHTS
