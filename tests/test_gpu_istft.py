"""GPU parity of the streaming iSTFT head through the C ABI: against the
float64 oracle on ragged multi-stream batches (Vocos-, iSTFTNet- and
HiFT-shaped sizes), chunked == full bit for bit, batch composition and
stream ids not changing a stream's bits, reset, magnitude clip, argument
errors."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from oracle import istft as O
from streaming_tts_vocoder_gb300 import codec as C
from streaming_tts_vocoder_gb300.synthetic import make_istft_spec

pytestmark = pytest.mark.gpu

# (n_fft, hop): Vocos at 24 kHz, Kokoro's iSTFTNet (the Core AI note: stride 5, 11 bins), HiFT-sized,
# and a non-power-of-two size with two frames per sample
# powers of two with even log2 (radix-4 stages only) and odd log2 (one radix-2
# stage first: 32, 512), and sizes that take the direct DFT (20, 48)
CONFIGS = [(1024, 256), (20, 5), (16, 4), (48, 24), (32, 8), (512, 128)]
# the oracle is float64; the kernels sum in float32 (FFT, overlap-add): errors are rounding-sized
REL_L2, MAX_ABS_REL = 1e-5, 1e-4


def close(got, ref, what):
    rel = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30))
    mx = float(np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-30))
    assert rel <= REL_L2 and mx <= MAX_ABS_REL, f"{what}: rel-L2 {rel:.2e}, max|err|/max|ref| {mx:.2e}"
    # the decoder's waveform bound, for the record
    assert rel <= 1e-3 and float(np.abs(got - ref).max()) <= 1e-2


def run(ist, specs, n_frames, ids=None):
    """One call: specs [B][T][2 nb] numpy, returns list of B numpy audio arrays."""
    B, T = len(specs), max(max(n_frames), 1)
    nb2 = 2 * ist.n_bins
    x = np.zeros((B, T, nb2), np.float32)
    for b, s in enumerate(specs):
        x[b, :s.shape[0]] = s
    audio = torch.full((B, T * ist.hop), float("nan"), device="cuda")
    ist.decode(torch.from_numpy(x).cuda(), n_frames, audio, stream_ids=ids)
    torch.cuda.synchronize()
    a = audio.cpu().numpy()
    return [a[b, :n_frames[b] * ist.hop] for b in range(B)]


@pytest.mark.parametrize("n_fft,hop", CONFIGS)
def test_ragged_streams_vs_oracle(n_fft, hop):
    S, F, chunk = 8, 60, 11
    ist = C.Istft(n_fft, hop, max_streams=S, max_chunk_frames=chunk)
    specs = [make_istft_spec(n_fft, F, 100 + s) for s in range(S)]
    outs = [[] for _ in range(S)]
    start = [s % chunk for s in range(S)]        # staggered: stream s starts s % chunk ticks late
    t = [0] * S
    tick = 0
    while any(t[s] < F for s in range(S)):
        nf, sp = [], []
        for s in range(S):
            n = 0 if tick < start[s] else min(chunk - (s % 3), F - t[s])
            nf.append(max(n, 0))
            sp.append(specs[s][t[s]:t[s] + nf[-1]])
        got = run(ist, sp, nf)
        for s in range(S):
            outs[s].append(got[s])
            t[s] += nf[s]
        tick += 1
    for s in range(S):
        ref = O.istft_full(specs[s].astype(np.float64), n_fft, hop)
        close(np.concatenate(outs[s]), ref, f"stream {s}")


@pytest.mark.parametrize("n_fft,hop", CONFIGS)
def test_chunked_equals_full_bitwise(n_fft, hop):
    F = 40
    spec = make_istft_spec(n_fft, F, 7)
    ist = C.Istft(n_fft, hop, max_streams=2, max_chunk_frames=F)
    full = run(ist, [spec], [F])[0]
    for splits in ([1] * F, [3, 1, 2, 34], [20, 20]):
        ist.reset()
        parts, t = [], 0
        for n in splits:
            parts.append(run(ist, [spec[t:t + n]], [n])[0])
            t += n
        assert np.array_equal(np.concatenate(parts), full), f"splits {splits[:5]}"


def test_batch_and_ids_do_not_change_bits():
    n_fft, hop, F = 1024, 256, 9
    specs = [make_istft_spec(n_fft, F, 30 + s) for s in range(4)]
    ist = C.Istft(n_fft, hop, max_streams=6, max_chunk_frames=F)
    alone = []
    for s in range(4):
        ist.reset()
        alone.append(run(ist, [specs[s]], [F])[0])
    ist.reset()
    got = run(ist, [specs[2], specs[0], specs[3], specs[1]], [F, F, F, F], ids=[5, 0, 3, 1])
    for g, s in zip(got, [2, 0, 3, 1]):
        assert np.array_equal(g, alone[s])
    # zero-frame entries and a reset of one slot only
    ist.reset([5])
    got = run(ist, [specs[2], specs[0]], [F, 0], ids=[5, 0])
    assert np.array_equal(got[0], alone[2]) and got[1].size == 0


def test_clip_and_reset():
    n_fft, hop, F = 64, 16, 12
    spec = make_istft_spec(n_fft, F, 3, logmag_mean=3.0, logmag_std=2.0)
    ist = C.Istft(n_fft, hop, mag_clip=20.0, max_streams=1, max_chunk_frames=F)
    a = run(ist, [spec], [F])[0]
    ist.reset()
    b = run(ist, [spec], [F])[0]
    assert np.array_equal(a, b)
    close(a, O.istft_full(spec.astype(np.float64), n_fft, hop, mag_clip=20.0), "clipped")


def test_argument_errors():
    ist = C.Istft(16, 4, max_streams=2, max_chunk_frames=4)
    x = torch.zeros(3, 4, 18, device="cuda")
    a = torch.zeros(3, 16, device="cuda")
    with pytest.raises(C.CodecError):
        ist.decode(x, [1, 1, 1], a)                    # B > max_streams
    with pytest.raises(C.CodecError):
        ist.decode(x[:2], [1, 1], a, stream_ids=[1, 1])  # repeated id
    with pytest.raises(C.CodecError):
        ist.decode(torch.zeros(1, 5, 18, device="cuda"), [5], a)   # T_max > max_chunk_frames
    with pytest.raises(C.CodecError):
        C.Istft(18, 4)                                 # hop does not divide n_fft
