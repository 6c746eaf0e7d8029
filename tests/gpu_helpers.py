"""Drivers for the GPU tests: decode through the C ABI (via the binding) and
compare with the oracle.  Test infrastructure only."""
from __future__ import annotations

import numpy as np
import torch

from streaming_tts_vocoder_gb300 import codec as C

TOL_REL = 1e-3     # waveform relative L2 bound
TOL_MAX = 1e-2     # waveform max |err| bound


def relerr(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def assert_close(got, want, what="", rel=TOL_REL, mx=TOL_MAX):
    r = relerr(got, want)
    m = float(np.abs(np.asarray(got, np.float64) - np.asarray(want, np.float64)).max()) if np.size(want) else 0.0
    assert r <= rel and m <= mx, f"{what}: rel-L2 {r:.3e} (<= {rel}), max|err| {m:.3e} (<= {mx})"
    return r, m


def assert_close_pre_tanh(got, want, what=""):
    """The final conv's output before tanh, against the oracle's.  Most samples
    of a random-weight decoder saturate the tanh (|audio| > 0.999), so the
    waveform comparison alone cannot see errors there; this one can.  Same
    relative L2 bound as the waveform; the waveform's max-abs bound of 1e-2
    is stated for a signal of unit scale, so here it scales with the rms of
    the pre-tanh signal (tens on these decoders)."""
    w = np.asarray(want, np.float64)
    scale = max(1.0, float(np.sqrt(np.mean(w * w)))) if w.size else 1.0
    return assert_close(got, want, what + " (pre-tanh)", rel=TOL_REL, mx=TOL_MAX * scale)


def bits_equal(a, b):
    a = np.ascontiguousarray(a, np.float32)
    b = np.ascontiguousarray(b, np.float32)
    return a.shape == b.shape and np.array_equal(a.view(np.uint32), b.view(np.uint32))


def decode_batch(state: C.CodecState, entries, T_max=None, pre_tanh=False):
    """entries: list of (stream_id, codes [Q][n]).  One codec_decode_chunk call;
    returns the list of audio arrays (and pre-tanh arrays)."""
    cod = state.codec
    Q = cod.cfg.Q
    spf = cod.samples_per_frame
    if T_max is None:
        T_max = max(1, max(c.shape[1] for _, c in entries))
    B = len(entries)
    codes = np.zeros((B, Q, T_max), np.int32)
    for b, (_, c) in enumerate(entries):
        codes[b, :, : c.shape[1]] = c
    codes_d = torch.from_numpy(codes).cuda()
    audio = torch.full((B, T_max * spf), float("nan"), device="cuda")
    pt = torch.full((B, T_max * spf), float("nan"), device="cuda") if pre_tanh else None
    state.decode(codes_d, [c.shape[1] for _, c in entries], audio, stream_ids=[s for s, _ in entries],
                 pre_tanh=pt)
    torch.cuda.synchronize()
    a = audio.cpu().numpy()
    out = [a[b, : entries[b][1].shape[1] * spf].copy() for b in range(B)]
    if pre_tanh:
        p = pt.cpu().numpy()
        return out, [p[b, : entries[b][1].shape[1] * spf].copy() for b in range(B)]
    return out


def decode_stream_chunks(state, stream_id, codes, splits, pre_tanh=False):
    """Decode one stream chunk by chunk; returns the concatenated audio."""
    parts, pts, i = [], [], 0
    for n in splits:
        r = decode_batch(state, [(stream_id, codes[:, i:i + n])], pre_tanh=pre_tanh)
        if pre_tanh:
            parts.append(r[0][0])
            pts.append(r[1][0])
        else:
            parts.append(r[0])
        i += n
    assert i == codes.shape[1]
    if pre_tanh:
        return np.concatenate(parts), np.concatenate(pts)
    return np.concatenate(parts)
