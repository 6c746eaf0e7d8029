"""GPU parity of the int8-per-32 weight mode (codec_create_q8: the
blixt/phonon "Weights" storage format, expanded on the device) through the C
ABI.  The parity target is the oracle decoding the dequantised weights
(oracle/weights_int8.quantize_blob), at the decoder's bound, waveform and
pre-tanh; the device expansion must be exact, so the decode equals bit for
bit that of a codec created from the oracle's dequantised fp32 blob.  The
format's own cost, the SNR against the decoder with the original weights, is
reported (printed), not bounded: random weights amplify the 0.4 % weight
error the way they amplify any rounding."""
from __future__ import annotations

import numpy as np
import pytest

from gpu_helpers import assert_close, assert_close_pre_tanh, bits_equal, decode_batch
from oracle import weights_int8 as OQ
from oracle.oracle import OracleModel
from streaming_tts_vocoder_gb300 import codec as C
from streaming_tts_vocoder_gb300.synthetic import make_codes, make_weights, pack_blob, qwen3_config, tiny_config
from streaming_tts_vocoder_gb300.weights_q8 import pack_q8

pytestmark = pytest.mark.gpu


def snr_db(got, ref):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    return float(20 * np.log10(np.linalg.norm(ref) / np.linalg.norm(got - ref)))


@pytest.mark.parametrize("precision", [C.PRECISION_FP32, C.PRECISION_FP16X3])
def test_q8_tiny_matches_oracle_on_dequantised_weights(precision):
    cfg = tiny_config()
    blob = pack_blob(cfg, make_weights(cfg, 0))
    deq = OQ.quantize_blob(cfg, blob)
    codes = make_codes(cfg, 12, 3)
    cod = C.Codec(cfg, q8=pack_q8(cfg, blob), max_streams=2, max_chunk_frames=12, precision=precision)
    st = cod.state()
    (a,), (pt,) = decode_batch(st, [(0, codes)], pre_tanh=True)
    ref, ref_pt = OracleModel(cfg, deq).decode_full(codes, pre_tanh=True)
    assert_close(a, ref, "q8 weights")
    assert_close_pre_tanh(pt, ref_pt, "q8 weights")
    # the device expansion is exact: same bits as a codec built from the dequantised fp32 blob
    cod2 = C.Codec(cfg, deq, max_streams=2, max_chunk_frames=12, precision=precision)
    assert bits_equal(decode_batch(cod2.state(), [(1, codes)])[0], a)
    full = OracleModel(cfg, blob).decode_full(codes)
    print(f"tiny, int8-per-32 weights: SNR {snr_db(a, full):.1f} dB against the fp32-weight oracle")


def test_q8_qwen3_matches_oracle_on_dequantised_weights():
    cfg = qwen3_config()
    blob = pack_blob(cfg, make_weights(cfg, 0))
    deq = OQ.quantize_blob(cfg, blob)
    codes = make_codes(cfg, 6, 5)
    cod = C.Codec(cfg, q8=pack_q8(cfg, blob), max_streams=1, max_chunk_frames=6, precision=C.PRECISION_FP16X3)
    st = cod.state()
    (a,), (pt,) = decode_batch(st, [(0, codes)], pre_tanh=True)
    ref, ref_pt = OracleModel(cfg, deq).decode_full(codes, pre_tanh=True)
    assert_close(a, ref, "q8 weights")
    assert_close_pre_tanh(pt, ref_pt, "q8 weights")
    full = OracleModel(cfg, blob).decode_full(codes)
    print(f"qwen3, int8-per-32 weights: SNR {snr_db(a, full):.1f} dB against the fp32-weight oracle")


def test_q8_wrong_size_is_rejected():
    cfg = tiny_config()
    data = pack_q8(cfg, pack_blob(cfg, make_weights(cfg, 0)))
    with pytest.raises(C.CodecError) as e:
        C.Codec(cfg, q8=data[:-4], max_streams=1, max_chunk_frames=1)
    assert e.value.status == 3
