"""The blixt/phonon "Weights" format applied to a decoder weight blob (test
infrastructure: a CPU study of what the format costs against the float64
oracle; the CUDA library does not use it).

The page's recipe, restated: every tensor with 16,384 values or more becomes
int8 with one f16 scale per 32 values along its rows; the scale is max |value|
/ 127 after rounding the values to f16, and quantised values round half to
even; other tensors stay f16; the arithmetic stays f32.  Rows are those of the
page's converted layouts: convolutions [out][tap][in], transposed
convolutions one GEMM per output phase [out][phase][tap][in], linears
[out][in], codebooks [entry][width].  quantize_blob returns the dequantised
values in the blob's own (PyTorch) layouts, so the oracle decodes them as it
decodes any weights.
"""
from __future__ import annotations

import numpy as np

from streaming_tts_vocoder_gb300.synthetic import weight_manifest

MIN_QUANT = 16384
GROUP = 32


def f16(x: np.ndarray) -> np.ndarray:
    return np.asarray(x, dtype=np.float64).astype(np.float16).astype(np.float64)


def quantize_rows(a: np.ndarray) -> np.ndarray:
    """a [rows][L] float64 -> int8-with-f16-scale values, dequantised, per
    group of 32 consecutive values of a row."""
    v = f16(a)
    out = np.empty_like(v)
    for g in range(0, v.shape[1], GROUP):
        blk = v[:, g:g + GROUP]
        scale = f16(np.abs(blk).max(axis=1, keepdims=True) / 127.0)
        q = np.zeros_like(blk)
        nz = scale[:, 0] > 0
        q[nz] = np.clip(np.rint(blk[nz] / scale[nz]), -127, 127)
        out[:, g:g + GROUP] = q * scale
    return out


def to_rows(name: str, a: np.ndarray, shape) -> tuple:
    """(rows [out][...] in the converted layout, inverse map back to the blob layout)."""
    if name.endswith(".w") and len(shape) == 3 and (name.startswith("up.") or
                                                    (name.startswith("st.") and ".rb." not in name)):
        # transposed conv [in][out][2 s] -> [out][phase][tap][in]
        cin, cout, k = shape
        s = k // 2
        r = a.reshape(cin, cout, 2, s).transpose(1, 3, 2, 0)          # [out][phase p][tap j][in], k = p + j s
        return r.reshape(cout, -1), lambda q: q.reshape(cout, s, 2, cin).transpose(3, 0, 2, 1).reshape(shape)
    if len(shape) == 3:
        # conv [out][in][k] -> [out][tap][in]
        co, ci, k = shape
        r = a.reshape(co, ci, k).transpose(0, 2, 1)
        return r.reshape(co, -1), lambda q: q.reshape(co, k, ci).transpose(0, 2, 1).reshape(shape)
    if len(shape) == 2:
        return a.reshape(shape), lambda q: q.reshape(shape)
    return a.reshape(1, -1), lambda q: q.reshape(shape)


def quantize_blob(cfg, blob: np.ndarray) -> np.ndarray:
    """The blob with every tensor in the page's format (dequantised), fp32."""
    out, off = [], 0
    blob = np.asarray(blob, dtype=np.float64)
    for t in weight_manifest(cfg):
        a = blob[off:off + t.size]
        off += t.size
        if t.size >= MIN_QUANT:
            rows, back = to_rows(t.name, a, t.shape)
            out.append(back(quantize_rows(rows)).reshape(-1))
        else:
            out.append(f16(a))
    return np.concatenate(out).astype(np.float32)
