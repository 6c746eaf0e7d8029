"""ctypes front end of the plain C oracle (oracle/codec_oracle.c).

TEST INFRASTRUCTURE ONLY: used by tests/, __graft_entry__.smoke() and the CPU
baseline leg of bench.py.  Never imported by the library.

build() compiles the C source with gcc (-O3 -fopenmp -ffp-contract=off, no
architecture flags, so it builds the same on x86-64 and aarch64).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

HERE = Path(__file__).resolve().parent
SRC = HERE / "codec_oracle.c"
LIB = HERE / "_build" / "libcodec_oracle.so"

_lib = None


def build(force: bool = False) -> Path:
    LIB.parent.mkdir(parents=True, exist_ok=True)
    if force or not LIB.exists() or LIB.stat().st_mtime < SRC.stat().st_mtime:
        tmp = LIB.with_suffix(f".{os.getpid()}.tmp.so")
        cmd = ["gcc", "-std=c11", "-O3", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
               "-fvisibility=hidden", str(SRC), "-o", str(tmp), "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB)
    return LIB


class OcConfig(ctypes.Structure):
    _fields_ = [
        ("Q", ctypes.c_int32), ("V", ctypes.c_int32), ("E", ctypes.c_int32),
        ("pre_k", ctypes.c_int32), ("d", ctypes.c_int32), ("heads", ctypes.c_int32),
        ("ffn", ctypes.c_int32), ("layers", ctypes.c_int32), ("window", ctypes.c_int32),
        ("n_up", ctypes.c_int32), ("up_k", ctypes.c_int32), ("up_s", ctypes.c_int32),
        ("up_ch", ctypes.c_int32 * 4),
        ("n_stages", ctypes.c_int32), ("strides", ctypes.c_int32 * 8), ("ch", ctypes.c_int32 * 8),
        ("n_rb", ctypes.c_int32), ("rb_k", ctypes.c_int32 * 4),
        ("n_dil", ctypes.c_int32), ("dil", ctypes.c_int32 * 4),
        ("final_k", ctypes.c_int32), ("rms_eps", ctypes.c_float),
        ("latent_dim", ctypes.c_int32), ("tf_up", ctypes.c_int32),
    ]


def oc_config(cfg) -> OcConfig:
    c = OcConfig()
    c.Q, c.V, c.E, c.pre_k = cfg.Q, cfg.V, cfg.E, cfg.pre_k
    c.d, c.heads, c.ffn, c.layers, c.window = cfg.d, cfg.heads, cfg.ffn, cfg.layers, cfg.window
    c.n_up, c.up_k, c.up_s = len(cfg.up_channels), cfg.up_k, cfg.up_s
    for i, v in enumerate(cfg.up_channels):
        c.up_ch[i] = v
    c.n_stages = len(cfg.strides)
    for i, (s, ch) in enumerate(zip(cfg.strides, cfg.channels)):
        c.strides[i] = s
        c.ch[i] = ch
    c.n_rb = len(cfg.rb_kernels)
    for i, k in enumerate(cfg.rb_kernels):
        c.rb_k[i] = k
    c.n_dil = len(cfg.dilations)
    for i, dl in enumerate(cfg.dilations):
        c.dil[i] = dl
    c.final_k = cfg.final_k
    c.rms_eps = cfg.rms_eps
    c.latent_dim = cfg.latent_dim
    c.tf_up = cfg.tf_up
    return c


_F = ctypes.POINTER(ctypes.c_float)
_I = ctypes.POINTER(ctypes.c_int32)
_V = ctypes.c_void_p


def lib():
    global _lib
    if _lib is None:
        l = ctypes.CDLL(str(build()))
        i32, i64, u32, f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32, ctypes.c_float
        sig = {
            "oc_op_snake": (None, [_F, i64, i32, _F, _F]),
            "oc_op_causal_conv": (None, [_F, i32, i32, _F, _F, i32, i32, i32, _F, _F, _F]),
            "oc_op_causal_conv_t": (None, [_F, i32, i32, _F, _F, i32, i32, _F, _F]),
            "oc_op_dw_conv_t": (None, [_F, i32, i32, _F, _F, i32, _F]),
            "oc_decode_latents": (u32, [_V, _F, i32, _F, _F]),
            "oc_op_linear": (None, [_F, i32, i32, _F, i32, _F, _F]),
            "oc_op_rms_norm": (None, [_F, i32, i32, _F, f32, _F]),
            "oc_op_gelu": (None, [_F, i64, _F]),
            "oc_op_swa": (None, [_F, _F, _F, i32, i32, i32, i32, i32, i32, _F]),
            "oc_op_rvq_sum": (u32, [_F, i32, i32, i32, _I, i64, i32, _F]),
            "oc_blob_floats": (i64, [ctypes.POINTER(OcConfig)]),
            "oc_model_create": (_V, [ctypes.POINTER(OcConfig), _F, i64]),
            "oc_model_destroy": (None, [_V]),
            "oc_samples_per_frame": (i64, [_V]),
            "oc_state_create": (_V, [_V]),
            "oc_state_reset": (None, [_V]),
            "oc_state_destroy": (None, [_V]),
            "oc_state_frames": (i64, [_V]),
            "oc_state_error": (u32, [_V]),
            "oc_decode": (u32, [_V, _I, i64, i32, _F, _F]),
            "oc_max_threads": (ctypes.c_int, []),
            "oc_set_threads": (None, [ctypes.c_int]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(l, name)
            fn.restype = res
            fn.argtypes = args
        _lib = l
    return _lib


def _f(a):
    return None if a is None else a.ctypes.data_as(_F)


def _c(a, dtype=np.float32):
    return np.ascontiguousarray(a, dtype=dtype)


# ------------------------------------------------------------ single ops --

def snake(x, alpha):
    x = _c(x)
    y = np.empty_like(x)
    lib().oc_op_snake(_f(x), x.shape[0], x.shape[1], _f(_c(alpha)), _f(y))
    return y


def causal_conv(x_ext, w, b, dilation=1, alpha=None, res=None):
    """x_ext [(k-1)*dil + T][Cin] (history rows first), w [Cout][Cin][k]."""
    x_ext, w, b = _c(x_ext), _c(w), _c(b)
    Cout, Cin, k = w.shape
    T = x_ext.shape[0] - (k - 1) * dilation
    y = np.empty((T, Cout), np.float32)
    a = None if alpha is None else _c(alpha)
    r = None if res is None else _c(res)
    lib().oc_op_causal_conv(_f(x_ext), T, Cin, _f(w), _f(b), Cout, k, dilation, _f(a), _f(r), _f(y))
    return y


def causal_conv_t(x_ext, w, b, stride, alpha=None):
    """x_ext [1 + T][Cin] (history row first), w [Cin][Cout][2*stride]."""
    x_ext, w, b = _c(x_ext), _c(w), _c(b)
    Cin, Cout, k = w.shape
    assert k == 2 * stride
    T = x_ext.shape[0] - 1
    y = np.empty((T * stride, Cout), np.float32)
    a = None if alpha is None else _c(alpha)
    lib().oc_op_causal_conv_t(_f(x_ext), T, Cin, _f(w), _f(b), Cout, stride, _f(a), _f(y))
    return y


def dw_conv_t(x_ext, u, b, stride):
    """Causal depthwise transposed conv: x_ext [1 + T][C] (history row first),
    u [C][1][2*stride] -> [T*stride][C]."""
    x_ext, u, b = _c(x_ext), _c(u), _c(b)
    C = x_ext.shape[1]
    T = x_ext.shape[0] - 1
    assert u.shape == (C, 1, 2 * stride)
    y = np.empty((T * stride, C), np.float32)
    lib().oc_op_dw_conv_t(_f(x_ext), T, C, _f(u), _f(b), stride, _f(y))
    return y


def linear(x, w, res=None):
    x, w = _c(x), _c(w)
    y = np.empty((x.shape[0], w.shape[0]), np.float32)
    r = None if res is None else _c(res)
    lib().oc_op_linear(_f(x), x.shape[0], x.shape[1], _f(w), w.shape[0], _f(r), _f(y))
    return y


def rms_norm(x, g, eps):
    x = _c(x)
    y = np.empty_like(x)
    lib().oc_op_rms_norm(_f(x), x.shape[0], x.shape[1], _f(_c(g)), eps, _f(y))
    return y


def gelu(x):
    x = _c(x)
    y = np.empty_like(x)
    lib().oc_op_gelu(_f(x), x.size, _f(y))
    return y


def swa(q, k_ext, v_ext, heads, window, first=0):
    """q [T][d]; k_ext, v_ext [Hk + T][d]; rows before `first` do not exist."""
    q, k_ext, v_ext = _c(q), _c(k_ext), _c(v_ext)
    T, d = q.shape
    Hk = k_ext.shape[0] - T
    o = np.empty_like(q)
    lib().oc_op_swa(_f(q), _f(k_ext), _f(v_ext), T, Hk, first, d, heads, window, _f(o))
    return o


def rvq_sum(cb, codes):
    """cb [Q][V][E], codes [Q][T] -> (e [T][E], error bits)."""
    cb = _c(cb)
    codes = _c(codes, np.int32)
    Q, V, E = cb.shape
    T = codes.shape[1]
    e = np.empty((T, E), np.float32)
    err = lib().oc_op_rvq_sum(_f(cb), Q, V, E, codes.ctypes.data_as(_I), codes.shape[1], T, _f(e))
    return e, err


# ---------------------------------------------------------------- model --

class OracleModel:
    """Weights of one decoder, held by the C oracle (a private copy)."""

    def __init__(self, cfg, blob: np.ndarray):
        self.cfg = cfg
        self._c = oc_config(cfg)
        blob = _c(blob)
        n = lib().oc_blob_floats(ctypes.byref(self._c))
        if n != blob.size:
            raise ValueError(f"blob has {blob.size} floats, config needs {n}")
        self._m = lib().oc_model_create(ctypes.byref(self._c), _f(blob), blob.size)
        if not self._m:
            raise ValueError("oracle rejected the config")
        self.samples_per_frame = lib().oc_samples_per_frame(self._m)

    def __del__(self):
        if getattr(self, "_m", None):
            lib().oc_model_destroy(self._m)
            self._m = None

    def stream(self) -> "OracleStream":
        return OracleStream(self)

    def decode_full(self, codes, pre_tanh=False):
        s = self.stream()
        return s.decode(codes, pre_tanh=pre_tanh)

    def decode_latents_full(self, latents, pre_tanh=False):
        return self.stream().decode_latents(latents, pre_tanh=pre_tanh)


class OracleStream:
    """One stream's carried state (conv histories, last W-1 keys/values)."""

    def __init__(self, model: OracleModel):
        self.model = model
        self._s = lib().oc_state_create(model._m)

    def __del__(self):
        if getattr(self, "_s", None):
            lib().oc_state_destroy(self._s)
            self._s = None

    def reset(self):
        lib().oc_state_reset(self._s)

    @property
    def frames(self) -> int:
        return lib().oc_state_frames(self._s)

    @property
    def error(self) -> int:
        return lib().oc_state_error(self._s)

    def decode_latents(self, latents, pre_tanh=False):
        """latents [n][L] -> audio [n * samples_per_frame] (latent-input decoder)."""
        x = _c(latents)
        n = x.shape[0]
        spf = self.model.samples_per_frame
        audio = np.empty(n * spf, np.float32)
        pt = np.empty(n * spf, np.float32) if pre_tanh else None
        if n:
            lib().oc_decode_latents(self._s, _f(x), n, _f(audio), _f(pt))
        return (audio, pt) if pre_tanh else audio

    def decode(self, codes, pre_tanh=False):
        """codes [Q][n] -> audio [n * samples_per_frame] (and pre-tanh values)."""
        codes = _c(codes, np.int32)
        n = codes.shape[1]
        spf = self.model.samples_per_frame
        audio = np.empty(n * spf, np.float32)
        pt = np.empty(n * spf, np.float32) if pre_tanh else None
        if n:
            lib().oc_decode(self._s, codes.ctypes.data_as(_I), codes.shape[1], n, _f(audio), _f(pt))
        return (audio, pt) if pre_tanh else audio


def max_threads() -> int:
    return lib().oc_max_threads()


def set_threads(n: int) -> None:
    lib().oc_set_threads(n)
