"""Converter from the fp32 weight blob to the int8-per-32 storage format that
codec_create_q8 reads (the blixt/phonon "Weights" recipe: tensors of 16,384
values or more become int8 with one f16 scale per 32 values along the rows
of their converted layout, the scale being max |value| / 127 of the
f16-rounded values and the quantised values rounding half to even; other
tensors become f16).  A weight-preparation tool, run once per model; the
decode itself never calls it.  The file layout is documented beside
codec_create_q8 in include/codec.h.
"""
from __future__ import annotations

import numpy as np

from .synthetic import weight_manifest

QUANT_MIN = 16384
GROUP = 32


def _converted_rows(name: str, a: np.ndarray) -> np.ndarray:
    """The tensor as rows of its converted layout: [out][in] for codebooks
    and linears, [out][tap][in] for convolutions, [out][phase][tap][in] for
    transposed convolutions (kernel index = phase + tap * stride)."""
    if a.ndim == 3 and (name.startswith("up.") or (name.startswith("st.") and ".rb." not in name)):
        cin, cout, k = a.shape
        s = k // 2
        # [in][out][tap j][phase p] (k = j s + p) -> [out][p][j][in]
        return a.reshape(cin, cout, 2, s).transpose(1, 3, 2, 0).reshape(cout, 2 * s * cin)
    if a.ndim == 3:
        cout, cin, k = a.shape
        return a.transpose(0, 2, 1).reshape(cout, k * cin)
    return a.reshape(a.shape[0], -1) if a.ndim == 2 else a.reshape(1, -1)


def _pad4(b: bytes) -> bytes:
    return b + b"\0" * (-len(b) % 4)


def quantize_rows(rows: np.ndarray):
    """rows [R][L] -> (int8 q [R][L], f16 scales [R][ceil(L / 32)])."""
    R, L = rows.shape
    G = -(-L // GROUP)
    v = np.zeros((R, G * GROUP), np.float64)
    v[:, :L] = rows.astype(np.float16).astype(np.float64)
    v = v.reshape(R, G, GROUP)
    scale = (np.abs(v).max(axis=2) / 127.0).astype(np.float16)
    s64 = scale.astype(np.float64)[:, :, None]
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(s64 > 0, np.clip(np.rint(v / s64), -127, 127), 0.0)
    return q.reshape(R, G * GROUP)[:, :L].astype(np.int8), scale


def pack_q8(cfg, blob: np.ndarray) -> bytes:
    """fp32 blob (blob order of the decoder config) -> the int8-per-32 file."""
    blob = np.asarray(blob, np.float32)
    parts, off = [], 0
    for t in weight_manifest(cfg):
        a = blob[off:off + t.size].reshape(t.shape)
        off += t.size
        if t.size >= QUANT_MIN:
            q, scale = quantize_rows(_converted_rows(t.name, a))
            parts.append(_pad4(q.tobytes()))
            parts.append(_pad4(scale.tobytes()))
        else:
            parts.append(_pad4(a.astype(np.float16).tobytes()))
    if off != blob.size:
        raise ValueError("blob size does not match the config")
    return b"".join(parts)
