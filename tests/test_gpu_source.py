"""GPU parity of the harmonic sine source and the analysis STFT through the C
ABI: against the float64 oracles on ragged multi-stream batches, chunked ==
full bit for bit, the excitation chain STFT(sine source) of the pages, the
GPU STFT -> GPU iSTFT round trip, reset and argument errors."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from oracle import istft as I
from oracle import source as O
from streaming_tts_vocoder_gb300 import codec as C
from streaming_tts_vocoder_gb300.synthetic import make_f0

pytestmark = pytest.mark.gpu

REL_L2, MAX_ABS_REL = 1e-5, 1e-4


def close(got, ref, what):
    rel = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30))
    mx = float(np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-30))
    assert rel <= REL_L2 and mx <= MAX_ABS_REL, f"{what}: rel-L2 {rel:.2e}, max|err|/max|ref| {mx:.2e}"


def sine_call(src, f0s, nf, ids=None):
    B, T = len(f0s), max(max(nf), 1)
    x = np.zeros((B, T), np.float32)
    for b, f in enumerate(f0s):
        x[b, :f.size] = f
    out = torch.full((B, T * src.upp, src.harmonics), float("nan"), device="cuda")
    src.decode(torch.from_numpy(x).cuda(), nf, out, stream_ids=ids)
    torch.cuda.synchronize()
    o = out.cpu().numpy()
    return [o[b, :nf[b] * src.upp] for b in range(B)]


def stft_call(st, xs, nf, ids=None):
    B, T = len(xs), max(max(nf), 1)
    x = np.zeros((B, T, st.hop), np.float32)
    for b, v in enumerate(xs):
        x[b, :v.size // st.hop] = v.reshape(-1, st.hop)
    spec = torch.full((B, T, 2 * st.n_bins), float("nan"), device="cuda")
    st.decode(torch.from_numpy(x).cuda(), nf, spec, stream_ids=ids)
    torch.cuda.synchronize()
    s = spec.cpu().numpy()
    return [s[b, :nf[b]] for b in range(B)]


@pytest.mark.parametrize("upp,fs,H", [(256, 24000.0, 8), (120, 24000.0, 1), (300, 22050.0, 4)])
def test_sine_ragged_vs_oracle_and_chunking(upp, fs, H):
    S, F, chunk = 6, 50, 9
    src = C.SineSource(upp, fs, H, amplitude=0.1, max_streams=S, max_chunk_frames=chunk)
    f0 = [make_f0(F, 40 + s) for s in range(S)]
    outs, t = [[] for _ in range(S)], [0] * S
    tick = 0
    while any(t[s] < F for s in range(S)):
        nf = [0 if tick < s % 3 else min(chunk - s % 4, F - t[s]) for s in range(S)]
        got = sine_call(src, [f0[s][t[s]:t[s] + nf[s]] for s in range(S)], nf)
        for s in range(S):
            outs[s].append(got[s])
            t[s] += nf[s]
        tick += 1
    for s in range(S):
        got = np.concatenate(outs[s])
        ref = O.SineSource(upp, fs, H, 0.1).decode(f0[s])
        assert np.abs(got - ref).max() <= 1e-6, f"stream {s}"
        assert np.all(got[np.repeat(f0[s] <= 0, upp)] == 0)
    # chunked == full, bit for bit (the phase is an exact integer)
    src2 = C.SineSource(upp, fs, H, amplitude=0.1, max_streams=1, max_chunk_frames=F)
    full = sine_call(src2, [f0[0]], [F])[0]
    src2.reset()
    parts = [sine_call(src2, [f0[0][a:b]], [b - a])[0] for a, b in ((0, 1), (1, 4), (4, 30), (30, 50))]
    assert np.array_equal(np.concatenate(parts), full)


@pytest.mark.parametrize("n_fft,hop", [(1024, 256), (20, 5), (16, 4), (48, 24), (32, 8), (512, 128)])
def test_stft_ragged_vs_oracle_and_chunking(n_fft, hop):
    S, F, chunk = 5, 40, 11
    st = C.Stft(n_fft, hop, max_streams=S, max_chunk_frames=chunk)
    rng = np.random.default_rng(n_fft)
    xs = [rng.standard_normal(F * hop).astype(np.float32) for _ in range(S)]
    outs, t = [[] for _ in range(S)], [0] * S
    tick = 0
    while any(t[s] < F for s in range(S)):
        nf = [0 if tick < s % 2 else min(chunk - s % 3, F - t[s]) for s in range(S)]
        got = stft_call(st, [xs[s][t[s] * hop:(t[s] + nf[s]) * hop] for s in range(S)], nf)
        for s in range(S):
            outs[s].append(got[s])
            t[s] += nf[s]
        tick += 1
    for s in range(S):
        close(np.concatenate(outs[s]), O.StftStream(n_fft, hop).decode(xs[s].astype(np.float64)), f"stream {s}")
    st2 = C.Stft(n_fft, hop, max_streams=1, max_chunk_frames=F)
    full = stft_call(st2, [xs[0]], [F])[0]
    st2.reset()
    parts = [stft_call(st2, [xs[0][a * hop:b * hop]], [b - a])[0] for a, b in ((0, 1), (1, 3), (3, 40))]
    assert np.array_equal(np.concatenate(parts), full)


def test_excitation_chain_stft_of_sine():
    """har = STFT(SineGen(f0_upsamp(F0))): the GPU chain against the oracle chain."""
    upp, fs, n_fft, hop, F = 300, 24000.0, 20, 5, 12     # Kokoro-like: iSTFT n_fft 20, hop 5
    f0 = make_f0(F, 9, voiced_fraction=0.9)
    src = C.SineSource(upp, fs, 1, amplitude=0.1, max_streams=1, max_chunk_frames=F)
    exc = sine_call(src, [f0], [F])[0][:, 0]
    st = C.Stft(n_fft, hop, max_streams=1, max_chunk_frames=F * upp // hop)
    got = stft_call(st, [exc], [exc.size // hop])[0]
    ref = O.StftStream(n_fft, hop).decode(O.SineSource(upp, fs, 1, 0.1).decode(f0)[:, 0])
    close(got, ref, "STFT(sine)")


def test_gpu_stft_istft_round_trip():
    n_fft, hop, F = 1024, 256, 30
    x = np.random.default_rng(3).standard_normal(F * hop).astype(np.float32)
    X = stft_call(C.Stft(n_fft, hop, max_streams=1, max_chunk_frames=F), [x], [F])[0]
    nb = n_fft // 2 + 1
    spec = np.concatenate([np.log(np.hypot(X[:, :nb], X[:, nb:])), np.arctan2(X[:, nb:], X[:, :nb])], axis=1)
    ist = C.Istft(n_fft, hop, max_streams=1, max_chunk_frames=F)
    y = torch.empty(1, F * hop, device="cuda")
    ist.decode(torch.from_numpy(spec.astype(np.float32))[None].cuda().contiguous(), [F], y)
    torch.cuda.synchronize()
    d = n_fft - hop
    got = y.cpu().numpy()[0]
    np.testing.assert_allclose(got[d:], x[:F * hop - d], atol=1e-4)


def test_argument_errors():
    src = C.SineSource(64, 16000.0, 2, max_streams=2, max_chunk_frames=4)
    with pytest.raises(C.CodecError):
        src.decode(torch.zeros(3, 4, device="cuda"), [1, 1, 1], torch.zeros(3 * 4 * 64 * 2, device="cuda"))
    with pytest.raises(C.CodecError):
        src.decode(torch.zeros(2, 4, device="cuda"), [1, 1], torch.zeros(2 * 4 * 64 * 2, device="cuda"),
                   stream_ids=[0, 0])
    with pytest.raises(C.CodecError):
        C.SineSource(64, 16000.0, 17)
    st = C.Stft(16, 4, max_streams=1, max_chunk_frames=2)
    with pytest.raises(C.CodecError):
        st.decode(torch.zeros(1, 3, 4, device="cuda"), [3], torch.zeros(1 * 3 * 18, device="cuda"))
    with pytest.raises(C.CodecError):
        C.Stft(18, 4)
