"""GPU parity of the latent-input (Mimi-style) decoder variant through the C
ABI (codec_decode_latents): denormalise, the 1x1 projection folded into the
depthwise x16 upsampling's phase GEMM, the transformer at 200 Hz with its
window over a ring of positions, the stages and the final conv (blixt/phonon
"Weights"; "Speed" item 7: window 251 over a 512-position ring at 200 Hz,
chunks of 1, 2, 4 and 8 frames sharing one state).

Against the oracle (which runs the unfolded steps one after the other) on the
waveform and before tanh; chunks of 1, 2, 4, 8 frames equal to a full GPU
decode bit for bit; ragged multi-stream batches; the call errors of the
variant."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from gpu_helpers import assert_close, assert_close_pre_tanh, bits_equal
from oracle.oracle import OracleModel
from streaming_tts_vocoder_gb300 import codec as C
from streaming_tts_vocoder_gb300.synthetic import (make_latents, make_weights, mimi_config, pack_blob,
                                                   tiny_mimi_config)

pytestmark = pytest.mark.gpu
SPF = 1920


def decode_lat(st, entries, T_max=None, pre_tanh=True):
    """entries: (stream_id, latents [n][L]); one codec_decode_latents call."""
    L = st.codec.cfg.latent_dim
    if T_max is None:
        T_max = max(1, max(x.shape[0] for _, x in entries))
    B = len(entries)
    arr = np.zeros((B, T_max, L), np.float32)
    for b, (_, x) in enumerate(entries):
        arr[b, : x.shape[0]] = x
    audio = torch.full((B, T_max * SPF), float("nan"), device="cuda")
    pt = torch.full((B, T_max * SPF), float("nan"), device="cuda")
    st.decode_latents(torch.from_numpy(arr).cuda(), [x.shape[0] for _, x in entries], audio,
                      stream_ids=[s for s, _ in entries], pre_tanh=pt)
    torch.cuda.synchronize()
    a, p = audio.cpu().numpy(), pt.cpu().numpy()
    n = [x.shape[0] * SPF for _, x in entries]
    return [a[b, : n[b]].copy() for b in range(B)], [p[b, : n[b]].copy() for b in range(B)]


def chunked(st, sid, x, splits):
    a_parts, p_parts, i = [], [], 0
    for n in splits:
        (a,), (p,) = decode_lat(st, [(sid, x[i:i + n])])
        a_parts.append(a)
        p_parts.append(p)
        i += n
    return np.concatenate(a_parts), np.concatenate(p_parts)


@pytest.fixture(scope="module")
def tiny_mimi():
    cfg = tiny_mimi_config()
    blob = pack_blob(cfg, make_weights(cfg, 0))
    return cfg, blob, OracleModel(cfg, blob)


@pytest.mark.parametrize("precision", [C.PRECISION_FP32, C.PRECISION_FP16X3])
def test_tiny_latent_decoder_matches_oracle_and_chunks(tiny_mimi, precision):
    cfg, blob, om = tiny_mimi
    cod = C.Codec(cfg, blob, max_streams=3, max_chunk_frames=15, max_batch_frames=45, precision=precision)
    st = cod.state()
    x = make_latents(cfg, 15, 2)
    (full,), (full_pt,) = decode_lat(st, [(0, x)])
    ref, ref_pt = om.decode_latents_full(x, pre_tanh=True)
    assert full.size == 15 * SPF
    assert_close(full, ref, "15 frames")
    assert_close_pre_tanh(full_pt, ref_pt, "15 frames")
    for splits in ([1, 2, 4, 8], [1] * 15, [8, 7]):
        st.reset()
        a, p = chunked(st, 1, x, splits)
        assert bits_equal(a, full) and bits_equal(p, full_pt), splits
    assert st.query(1) == (15, 0)


def test_tiny_latent_ragged_batch(tiny_mimi):
    cfg, blob, om = tiny_mimi
    cod = C.Codec(cfg, blob, max_streams=3, max_chunk_frames=8, max_batch_frames=24, precision=C.PRECISION_FP16X3)
    st = cod.state()
    xs = [make_latents(cfg, 12, 30 + s) for s in range(3)]
    outs = [[] for _ in range(3)]
    # ragged ticks: the streams' chunks differ in size and start
    ticks = [[(0, 0, 1), (1, 0, 4), (2, 0, 8)], [(0, 1, 2), (1, 4, 8), (2, 8, 4)], [(0, 3, 4), (1, 12, 0)],
             [(0, 7, 5)]]
    for tick in ticks:
        entries = [(s, xs[s][a:a + n]) for s, a, n in tick if n]
        audio, _ = decode_lat(st, entries, T_max=8)
        for (s, _), a in zip(entries, audio):
            outs[s].append(a)
    for s in range(3):
        got = np.concatenate(outs[s])
        assert got.size == 12 * SPF
        assert_close(got, om.decode_latents_full(xs[s]), f"stream {s}")


def test_mimi_shaped_decoder_window_251_ring_512():
    """The Mimi-shaped decoder: 8 frames (128 positions at 200 Hz) and then
    chunks 1, 2, 4, 8 on top, so the later queries' 251-key windows reach back
    across calls through the ring."""
    cfg = mimi_config()
    blob = pack_blob(cfg, make_weights(cfg, 0))
    cod = C.Codec(cfg, blob, max_streams=2, max_chunk_frames=8, max_batch_frames=16, precision=C.PRECISION_FP16X3)
    st = cod.state()
    x = make_latents(cfg, 23, 5)
    splits = [8, 1, 2, 4, 8]
    a, p = chunked(st, 0, x, splits)
    ref, ref_pt = OracleModel(cfg, blob).decode_latents_full(x, pre_tanh=True)
    assert_close(a, ref, "23 frames in chunks 8, 1, 2, 4, 8")
    assert_close_pre_tanh(p, ref_pt, "23 frames in chunks 8, 1, 2, 4, 8")
    st.reset()
    b, _ = chunked(st, 1, x, [1, 2, 4, 8, 8])
    assert bits_equal(a, b)


@pytest.mark.parametrize("precision", [C.PRECISION_FP32, C.PRECISION_FP16X3])
def test_long_window_head_64_attention_path(precision):
    """A small latent decoder with 64-wide heads and a 150-position window:
    in the tensor-core modes its attention takes the warp-MMA kernel for long
    windows (keys staged from a 16-aligned position), in fp32 the CUDA-core
    one.  20 frames (320 positions) against the oracle, and every chunking,
    ragged ones included, equal to a full GPU decode bit for bit."""
    import dataclasses
    cfg = dataclasses.replace(tiny_mimi_config(), name="tiny_mimi_h64", d=128, heads=2, ffn=256, window=150)
    blob = pack_blob(cfg, make_weights(cfg, 0))
    cod = C.Codec(cfg, blob, max_streams=2, max_chunk_frames=20, max_batch_frames=40, precision=precision)
    st = cod.state()
    x = make_latents(cfg, 20, 9)
    (full,), (full_pt,) = decode_lat(st, [(0, x)])
    ref, ref_pt = OracleModel(cfg, blob).decode_latents_full(x, pre_tanh=True)
    assert_close(full, ref, "20 frames")
    assert_close_pre_tanh(full_pt, ref_pt, "20 frames")
    for splits in ([1, 2, 4, 8, 5], [3] * 6 + [2], [13, 7]):
        st.reset()
        a, p = chunked(st, 1, x, splits)
        assert bits_equal(a, full) and bits_equal(p, full_pt), splits


def test_latent_variant_call_errors(tiny_mimi):
    cfg, blob, om = tiny_mimi
    cod = C.Codec(cfg, blob, max_streams=1, max_chunk_frames=4, precision=C.PRECISION_FP32)
    st = cod.state()
    codes = torch.zeros(1, 1, 4, dtype=torch.int32, device="cuda")
    audio = torch.zeros(1, 4 * SPF, device="cuda")
    with pytest.raises(C.CodecError) as e:
        st.decode(codes, [1], audio)                       # codes into a latent-input codec
    assert e.value.status == 2
    lat = torch.zeros(1, 5, cfg.latent_dim, device="cuda")
    with pytest.raises(C.CodecError) as e:
        st.decode_latents(lat, [5], torch.zeros(1, 5 * SPF, device="cuda"))   # above max_chunk_frames
    assert e.value.status == 5
    assert st.query(0) == (0, 0)
