"""GPU parity of the streaming Vocos-style generator + iSTFT head
(codec_vocos_*, vox: "Vocos -> iSTFT") through the C ABI, against the float64
oracle (oracle/vocos.py): the waveform at the iSTFT head's tolerance scaled
to the backbone's fp32 / fp16x3 arithmetic (rel-L2 <= 1e-3, max |err| <= 1e-2
of the peak), several ragged streams decoded in chunks, chunked == full bit
for bit, reset, argument errors."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from gpu_helpers import bits_equal, relerr
from oracle import vocos as V
from streaming_tts_vocoder_gb300 import codec as C
from streaming_tts_vocoder_gb300.synthetic import (make_mels, make_vocos_weights, pack_vocos_blob,
                                                   tiny_vocos_config, vocos_config)

pytestmark = pytest.mark.gpu


def run(voc, entries, T_max=None):
    cfg = voc.cfg
    if T_max is None:
        T_max = max(1, max(m.shape[0] for _, m in entries))
    B = len(entries)
    arr = np.zeros((B, T_max, cfg.n_mels), np.float32)
    for b, (_, m) in enumerate(entries):
        arr[b, : m.shape[0]] = m
    audio = torch.full((B, T_max * cfg.hop), float("nan"), device="cuda")
    voc.decode(torch.from_numpy(arr).cuda(), [m.shape[0] for _, m in entries], audio,
               stream_ids=[s for s, _ in entries])
    torch.cuda.synchronize()
    a = audio.cpu().numpy()
    return [a[b, : entries[b][1].shape[0] * cfg.hop].copy() for b in range(B)]


def close(got, want, what):
    r = relerr(got, want)
    m = float(np.abs(np.asarray(got, np.float64) - want).max() / np.abs(want).max())
    assert r <= 1e-3 and m <= 1e-2, f"{what}: rel-L2 {r:.3e}, max |err| / peak {m:.3e}"


@pytest.mark.parametrize("precision", [C.PRECISION_FP32, C.PRECISION_FP16X3])
def test_tiny_vocos_streams_match_oracle(precision):
    cfg = tiny_vocos_config()
    W = make_vocos_weights(cfg, 0)
    voc = C.Vocos(cfg, pack_vocos_blob(cfg, W), max_streams=3, max_chunk_frames=20, max_batch_frames=60,
                  precision=precision)
    mels = [make_mels(cfg, 20, 10 + s) for s in range(3)]
    outs = [[] for _ in range(3)]
    # ragged chunks per tick
    plan = [[(0, 0, 1), (1, 0, 7), (2, 0, 20)], [(0, 1, 19), (1, 7, 13)]]
    for tick in plan:
        entries = [(s, mels[s][a:a + n]) for s, a, n in tick]
        for (s, _), a in zip(entries, run(voc, entries, T_max=20)):
            outs[s].append(a)
    for s in range(3):
        got = np.concatenate(outs[s])
        want = V.decode_full(cfg, W, mels[s])
        close(got, want, f"stream {s}")
    voc.reset()
    full = run(voc, [(2, mels[0])])[0]
    assert bits_equal(np.concatenate(outs[0]), full)


def test_vocos_24khz_shape_matches_oracle():
    cfg = vocos_config()
    W = make_vocos_weights(cfg, 0)
    voc = C.Vocos(cfg, pack_vocos_blob(cfg, W), max_streams=2, max_chunk_frames=24, max_batch_frames=48,
                  precision=C.PRECISION_FP16X3)
    mel = make_mels(cfg, 24, 4)
    a = np.concatenate([run(voc, [(1, mel[i:i + n])])[0] for i, n in ((0, 1), (1, 7), (8, 16))])
    close(a, V.decode_full(cfg, W, mel), "24 frames in chunks 1, 7, 16")
    voc.reset([1])
    assert bits_equal(run(voc, [(1, mel)])[0], a)


def test_vocos_argument_errors():
    cfg = tiny_vocos_config()
    voc = C.Vocos(cfg, pack_vocos_blob(cfg, make_vocos_weights(cfg, 0)), max_streams=2, max_chunk_frames=4)
    mel = torch.zeros(2, 4, cfg.n_mels, device="cuda")
    audio = torch.zeros(2, 4 * cfg.hop, device="cuda")
    for kw, want in [(dict(n_frames=[5, 1]), 4), (dict(n_frames=[1, 1], stream_ids=[1, 1]), 4),
                     (dict(n_frames=[1, 1], stream_ids=[0, 2]), 4)]:
        with pytest.raises(C.CodecError) as e:
            voc.decode(mel, audio=audio, **kw)
        assert e.value.status == want
