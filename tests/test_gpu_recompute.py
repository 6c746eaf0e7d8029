"""GPU parity of the recompute-mode decode (codec_decode_recompute) through
the C ABI: the server schedule of the vllm-omni "Edge TTS design" page,
section 1.4, where each chunk is re-decoded with up to 72 frames of left
context from an empty state and only the new frames' audio is kept.

Checks: the kept audio and pre-tanh output against the oracle decoding the
same window from reset; n_ctx = 0 equal to a carried decode from reset bit
for bit; entries of one batch with different context lengths independent of
each other; an entry with no new frames left untouched; a carried call after a
recompute call continuing the recomputed state bit for bit; argument errors
enqueuing nothing."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from gpu_helpers import assert_close, assert_close_pre_tanh, bits_equal, decode_batch
from oracle.oracle import OracleModel
from streaming_tts_vocoder_gb300 import codec as C
from streaming_tts_vocoder_gb300.synthetic import (make_codes, make_weights, pack_blob, qwen3_config,
                                                   tiny_config)

pytestmark = pytest.mark.gpu
SPF = 1920


def recompute(st, entries, T_max):
    """entries: (stream_id, codes [Q][n_ctx + n_new], n_ctx); one call."""
    cfg = st.codec.cfg
    B = len(entries)
    arr = np.zeros((B, cfg.Q, T_max), np.int32)
    nc, nn = [], []
    for b, (_, c, n_ctx) in enumerate(entries):
        arr[b, :, : c.shape[1]] = c
        nc.append(n_ctx)
        nn.append(c.shape[1] - n_ctx)
    audio = torch.full((B, T_max * SPF), float("nan"), device="cuda")
    pt = torch.full((B, T_max * SPF), float("nan"), device="cuda")
    st.decode_recompute(torch.from_numpy(arr).cuda(), nc, nn, audio, stream_ids=[s for s, _, _ in entries],
                        pre_tanh=pt)
    torch.cuda.synchronize()
    a, p = audio.cpu().numpy(), pt.cpu().numpy()
    return [a[b, : nn[b] * SPF].copy() for b in range(B)], [p[b, : nn[b] * SPF].copy() for b in range(B)], a


@pytest.fixture(scope="module")
def tiny():
    cfg = tiny_config()
    blob = pack_blob(cfg, make_weights(cfg, 0))
    return cfg, blob, OracleModel(cfg, blob)


@pytest.mark.parametrize("precision", [C.PRECISION_FP32, C.PRECISION_FP16X3])
def test_recompute_window_matches_oracle_and_carried(tiny, precision):
    cfg, blob, om = tiny
    cod = C.Codec(cfg, blob, max_streams=4, max_chunk_frames=97, max_batch_frames=4 * 97, precision=precision)
    st = cod.state()
    codes = make_codes(cfg, 140, 21)
    # three entries: the server's 72 + 25 window, a short context, no context
    win = [(0, codes[:, 43:140], 72), (2, codes[:, 10:30], 7), (3, codes[:, 0:12], 0)]
    kept, kept_pt, _ = recompute(st, win, 97)
    for (sid, c, n_ctx), a, p in zip(win, kept, kept_pt):
        ref, ref_pt = om.decode_full(c, pre_tanh=True)
        n_new = c.shape[1] - n_ctx
        assert a.size == n_new * SPF
        assert_close(a, ref[n_ctx * SPF:], f"slot {sid} kept audio")
        assert_close_pre_tanh(p, ref_pt[n_ctx * SPF:], f"slot {sid} kept audio")
        assert st.query(sid) == (c.shape[1], 0)
    # the slot carries the whole window: a carried call continues it
    nxt = codes[:, 30:39]
    cont = decode_batch(st, [(2, nxt)])[0]
    st.reset()
    full = decode_batch(st, [(2, codes[:, 10:39])])[0]
    assert bits_equal(cont, full[20 * SPF:])
    # n_ctx = 0 equals a carried decode from reset, bit for bit
    st.reset()
    carried = decode_batch(st, [(3, codes[:, 0:12])])[0]
    assert bits_equal(kept[2], carried)


def test_recompute_leaves_entries_without_new_frames_alone(tiny):
    cfg, blob, om = tiny
    cod = C.Codec(cfg, blob, max_streams=2, max_chunk_frames=30, precision=C.PRECISION_FP16X3)
    st = cod.state()
    codes = make_codes(cfg, 30, 4)
    first = decode_batch(st, [(1, codes[:, :5])])[0]
    kept, _, raw = recompute(st, [(0, codes[:, :20], 15), (1, codes[:, 5:10], 5)], 20)
    assert st.query(1) == (5, 0)                       # untouched: no reset, no decode
    assert np.isnan(raw[1]).all()                      # nothing written for it
    assert kept[0].size == 5 * SPF
    nxt = decode_batch(st, [(1, codes[:, 5:10])])[0]   # slot 1 still carries its 5 frames
    st.reset()
    assert bits_equal(np.concatenate([first, nxt]), decode_batch(st, [(1, codes[:, :10])])[0])


def test_recompute_argument_errors_enqueue_nothing(tiny):
    cfg, blob, om = tiny
    cod = C.Codec(cfg, blob, max_streams=2, max_chunk_frames=10, precision=C.PRECISION_FP32)
    st = cod.state()
    codes = make_codes(cfg, 10, 1)
    decode_batch(st, [(0, codes[:, :3])])
    arr = torch.zeros(1, cfg.Q, 10, dtype=torch.int32, device="cuda")
    audio = torch.zeros(1, 10 * SPF, device="cuda")
    for nc, nn, want in [([8], [3], 4), ([-1], [2], 4), ([2], [-1], 4)]:
        with pytest.raises(C.CodecError) as e:
            st.decode_recompute(arr, nc, nn, audio, stream_ids=[0])
        assert e.value.status == want
    with pytest.raises(C.CodecError) as e:
        st.decode_recompute(arr, [1], [1], audio, stream_ids=[5])
    assert e.value.status == 4
    assert st.query(0) == (3, 0)                       # no reset was enqueued


def test_recompute_qwen3_72_plus_25_matches_oracle():
    """The page's server call on the Qwen3-shaped decoder: 25 new frames with
    72 frames of left context re-decoded, 48,000 samples kept."""
    cfg = qwen3_config()
    blob = pack_blob(cfg, make_weights(cfg, 0))
    cod = C.Codec(cfg, blob, max_streams=2, max_chunk_frames=97, max_batch_frames=2 * 97,
                  precision=C.PRECISION_FP16X3)
    st = cod.state()
    codes = make_codes(cfg, 110, 7)
    win = codes[:, 13:110]
    kept, kept_pt, _ = recompute(st, [(1, win, 72)], 97)
    assert kept[0].size == 48000
    ref, ref_pt = OracleModel(cfg, blob).decode_full(win, pre_tanh=True)
    assert_close(kept[0], ref[72 * SPF:], "kept 48,000 samples")
    assert_close_pre_tanh(kept_pt[0], ref_pt[72 * SPF:], "kept 48,000 samples")
