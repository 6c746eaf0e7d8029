"""GPU parity of the tiny decoder (Q=4 x 256 x 64, d=64, window 8, channels
64 -> 4) against the CPU oracle, through the C ABI, on the five workloads:
full sequence, first-audio + single-frame calls, 64 ragged staggered streams,
long-form chunking; plus the bookkeeping (bit-exact gather, frame counters,
sticky error bits, reset) and argument errors."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from gpu_helpers import assert_close, assert_close_pre_tanh, bits_equal, decode_batch, decode_stream_chunks
from oracle.oracle import OracleModel
from streaming_tts_vocoder_gb300 import codec as C
from streaming_tts_vocoder_gb300.synthetic import (make_codes, make_weights, pack_blob,
                                                   staggered_schedule, tiny_config)

pytestmark = pytest.mark.gpu

PRECISIONS = [C.PRECISION_FP32, C.PRECISION_FP16X3]


@pytest.fixture(scope="module")
def tiny():
    cfg = tiny_config()
    W = make_weights(cfg, 0)
    blob = pack_blob(cfg, W)
    return cfg, blob, OracleModel(cfg, blob)


def make_state(cfg, blob, precision, streams=1, chunk=97, batch=None):
    cod = C.Codec(cfg, blob, max_streams=streams, max_chunk_frames=chunk,
                  max_batch_frames=batch if batch is not None else streams * chunk, precision=precision)
    return cod.state()


@pytest.mark.parametrize("precision", PRECISIONS)
def test_full_sequence_8_frames(tiny, precision):
    cfg, blob, om = tiny
    codes = make_codes(cfg, 8, 0)
    ref, ref_pt = om.decode_full(codes, pre_tanh=True)
    st = make_state(cfg, blob, precision, chunk=8)
    (a,), (pt,) = decode_batch(st, [(0, codes)], pre_tanh=True)
    assert a.size == 8 * 1920
    assert_close(a, ref, "audio")
    assert_close_pre_tanh(pt, ref_pt, "8 frames")
    assert st.query(0) == (8, 0)


@pytest.mark.parametrize("precision", PRECISIONS)
def test_gather_bit_exact(tiny, precision):
    cfg, blob, om = tiny
    from oracle import oracle as O
    from streaming_tts_vocoder_gb300.synthetic import make_weights as mw
    W = mw(cfg, 0)
    cb = np.stack([W[f"cb.{q}"] for q in range(cfg.Q)])
    st = make_state(cfg, blob, precision, streams=3, chunk=16)
    codes = [make_codes(cfg, n, 10 + n) for n in (5, 16, 1)]
    T_max = 16
    arr = np.zeros((3, cfg.Q, T_max), np.int32)
    for b, c in enumerate(codes):
        arr[b, :, : c.shape[1]] = c
    emb = torch.empty(22, cfg.E, device="cuda")
    st.embed(torch.from_numpy(arr).cuda(), [5, 16, 1], emb, stream_ids=[2, 0, 1])
    torch.cuda.synchronize()
    got = emb.cpu().numpy()
    want = np.concatenate([O.rvq_sum(cb, c)[0] for c in codes])
    assert bits_equal(got, want)


@pytest.mark.parametrize("precision", PRECISIONS)
@pytest.mark.parametrize("splits", [[1] * 12, [2, 3, 1, 6], [5, 7], [4, 4, 4], [11, 1]])
def test_chunked_equals_full(tiny, precision, splits):
    cfg, blob, om = tiny
    codes = make_codes(cfg, 12, 5)
    st = make_state(cfg, blob, precision, chunk=12)
    (full,), (full_pt,) = decode_batch(st, [(0, codes)], pre_tanh=True)
    st.reset()
    chunked, chunked_pt = decode_stream_chunks(st, 0, codes, splits, pre_tanh=True)
    assert bits_equal(chunked, full)
    assert bits_equal(chunked_pt, full_pt)
    ref, ref_pt = om.decode_full(codes, pre_tanh=True)
    assert_close(chunked, ref, "chunked vs oracle")
    assert_close_pre_tanh(chunked_pt, ref_pt, "chunked vs oracle")
    assert st.query(0) == (12, 0)


@pytest.mark.parametrize("precision", PRECISIONS)
def test_first_audio_then_single_frames(tiny, precision):
    """One frame from an empty state (1920 samples), then single-frame calls;
    frames 0..24 equal a 25-frame full decode."""
    cfg, blob, om = tiny
    codes = make_codes(cfg, 25, 3)
    st = make_state(cfg, blob, precision, chunk=25)
    (first,), (first_pt,) = decode_batch(st, [(0, codes[:, :1])], pre_tanh=True)
    assert first.size == 1920
    rest, rest_pt = decode_stream_chunks(st, 0, codes[:, 1:], [1] * 24, pre_tanh=True)
    chunked = np.concatenate([first, rest])
    chunked_pt = np.concatenate([first_pt, rest_pt])
    st.reset()
    full = decode_batch(st, [(0, codes)])[0]
    assert bits_equal(chunked, full)
    ref, ref_pt = om.decode_full(codes, pre_tanh=True)
    assert_close(chunked, ref, "single-frame calls vs oracle")
    assert_close_pre_tanh(chunked_pt, ref_pt, "single-frame calls vs oracle")


@pytest.mark.parametrize("precision", PRECISIONS)
def test_64_staggered_streams(tiny, precision):
    """64 streams x 250 frames, starting at offsets s mod 25, decoded in ragged
    ticks of up to 25 frames per stream."""
    cfg, blob, om = tiny
    S, F = 64, 250
    st = make_state(cfg, blob, precision, streams=S, chunk=25, batch=S * 25)
    codes = [make_codes(cfg, F, 1000 + s) for s in range(S)]
    out = [[] for _ in range(S)]
    out_pt = [[] for _ in range(S)]
    for tick in staggered_schedule(S, F, 25):
        entries = [(s, codes[s][:, a:a + n]) for s, a, n in tick]
        audio, pts = decode_batch(st, entries, T_max=25, pre_tanh=True)
        for (s, _), a, p in zip(entries, audio, pts):
            out[s].append(a)
            out_pt[s].append(p)
    for s in range(S):
        got = np.concatenate(out[s])
        assert got.size == F * 1920
        ref, ref_pt = om.decode_full(codes[s], pre_tanh=True)
        assert_close(got, ref, f"stream {s}")
        assert_close_pre_tanh(np.concatenate(out_pt[s]), ref_pt, f"stream {s}")
        assert st.query(s) == (F, 0)


@pytest.mark.parametrize("precision", PRECISIONS)
def test_long_form_8_streams(tiny, precision):
    """8 streams x 3000 frames as 120 chunks of 25, every stream against a
    full oracle decode, and chunked == one full GPU decode bit for bit."""
    cfg, blob, om = tiny
    S, F = 8, 3000
    st = make_state(cfg, blob, precision, streams=S, chunk=F, batch=S * F)
    codes = [make_codes(cfg, F, 77 + s) for s in range(S)]
    out = [[] for _ in range(S)]
    out_pt = [[] for _ in range(S)]
    for c in range(F // 25):
        entries = [(s, codes[s][:, c * 25:(c + 1) * 25]) for s in range(S)]
        audio, pts = decode_batch(st, entries, pre_tanh=True)
        for s in range(S):
            out[s].append(audio[s])
            out_pt[s].append(pts[s])
    st.reset()
    full = decode_batch(st, [(s, codes[s]) for s in range(S)])
    for s in range(S):
        got = np.concatenate(out[s])
        assert bits_equal(got, full[s]), f"stream {s}: chunked != full"
        ref, ref_pt = om.decode_full(codes[s], pre_tanh=True)
        assert_close(got, ref, f"stream {s}")
        assert_close_pre_tanh(np.concatenate(out_pt[s]), ref_pt, f"stream {s}")


@pytest.mark.parametrize("precision", PRECISIONS)
def test_bad_code_is_sticky_and_reset_clears(tiny, precision):
    cfg, blob, om = tiny
    st = make_state(cfg, blob, precision, streams=2, chunk=4)
    codes = make_codes(cfg, 4, 0)
    bad = codes.copy()
    bad[1, 2] = cfg.V
    (good_a, bad_a), (_, bad_pt) = decode_batch(st, [(0, codes), (1, bad)], pre_tanh=True)
    assert st.query(0) == (4, 0)
    assert st.query(1) == (4, C.STREAM_ERR_BAD_CODE)
    s = om.stream()
    ref, ref_pt = s.decode(bad, pre_tanh=True)
    assert_close(bad_a, ref, "bad-code stream vs oracle (zeroed frame)")
    assert_close_pre_tanh(bad_pt, ref_pt, "bad-code stream vs oracle (zeroed frame)")
    decode_batch(st, [(1, codes)])
    assert st.query(1) == (8, C.STREAM_ERR_BAD_CODE)
    st.reset([1])
    assert st.query(1) == (0, 0)
    again = decode_batch(st, [(1, codes)])[0]
    assert bits_equal(again, good_a)


@pytest.mark.parametrize("precision", PRECISIONS)
def test_reset_equals_fresh_and_isolates_streams(tiny, precision):
    cfg, blob, om = tiny
    st = make_state(cfg, blob, precision, streams=3, chunk=6)
    c0, c1 = make_codes(cfg, 6, 1), make_codes(cfg, 6, 2)
    fresh = decode_batch(st, [(2, c0)])[0]
    decode_batch(st, [(0, c1), (1, c1)])
    st.reset([0])
    a0, a1 = decode_batch(st, [(0, c0), (1, c0)])
    assert bits_equal(a0, fresh)
    assert not bits_equal(a1, fresh)           # stream 1 kept its context
    assert st.query(1) == (12, 0)


def test_host_buffer_entry_point(tiny):
    cfg, blob, om = tiny
    st = make_state(cfg, blob, C.PRECISION_FP32, streams=2, chunk=5)
    codes = np.stack([make_codes(cfg, 5, 9), make_codes(cfg, 5, 10)])
    ch = torch.from_numpy(codes).pin_memory()
    audio = torch.zeros(2, 5 * 1920).pin_memory()
    st.decode_host(ch, [5, 3], audio)
    a = audio.numpy()
    assert_close(a[0], om.decode_full(codes[0]), "host stream 0")
    assert_close(a[1, : 3 * 1920], om.decode_full(codes[1][:, :3]), "host stream 1")


def test_argument_errors_enqueue_nothing(tiny):
    cfg, blob, om = tiny
    st = make_state(cfg, blob, C.PRECISION_FP32, streams=2, chunk=4, batch=6)
    codes = torch.zeros(2, cfg.Q, 4, dtype=torch.int32, device="cuda")
    audio = torch.zeros(2, 4 * 1920, device="cuda")
    cases = [
        (dict(n_frames=[5, 1]), 4),                      # n_frames > T_max
        (dict(n_frames=[1, 1], stream_ids=[1, 1]), 4),   # repeated id
        (dict(n_frames=[1, 1], stream_ids=[0, 2]), 4),   # id out of range
        (dict(n_frames=[-1, 1]), 4),
    ]
    for kw, want in cases:
        with pytest.raises(C.CodecError) as e:
            st.decode(codes, audio=audio, **kw)
        assert e.value.status == want, kw
    codes5 = torch.zeros(2, cfg.Q, 5, dtype=torch.int32, device="cuda")
    audio5 = torch.zeros(2, 5 * 1920, device="cuda")
    with pytest.raises(C.CodecError) as e:
        st.decode(codes5, [5, 0], audio5)             # above max_chunk_frames
    assert e.value.status == 5
    with pytest.raises(C.CodecError) as e:
        st.decode(codes, [4, 4], audio)               # above max_batch_frames
    assert e.value.status == 5
    assert st.query(0) == (0, 0) and st.query(1) == (0, 0)
    st.decode(codes, [0, 0], audio)                   # nothing to do
    assert st.last_launches == 0


def test_kernel_timeout_is_reported_and_reset_recovers(tiny):
    """A decode whose tensor-core GEMMs give up on a bounded wait (each CTA's
    first epilogue wait is pointed at a barrier nothing arrives on) reports
    CODEC_STREAM_ERR_KERNEL_TIMEOUT; a reset of all slots clears it and the
    next decode has its normal bits."""
    cfg, blob, om = tiny
    st = make_state(cfg, blob, C.PRECISION_FP16X3, chunk=8)
    codes = make_codes(cfg, 8, 0)
    good = decode_batch(st, [(0, codes)])[0]
    st.reset()
    try:
        st.set_wait_limit(polls=1000, unarrived_wait=True)
        decode_batch(st, [(0, codes)])
        frames, bits = st.query(0)
        assert frames == 8 and bits & C.STREAM_ERR_KERNEL_TIMEOUT
    finally:
        st.set_wait_limit()
    st.reset()
    assert st.query(0) == (0, 0)
    assert bits_equal(decode_batch(st, [(0, codes)])[0], good)
