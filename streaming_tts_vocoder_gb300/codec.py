"""Python binding of the C ABI in include/codec.h (argument marshalling only).

Every computation runs in the CUDA library libcodec_gb300.so; this module only
converts configs, numpy weight blobs and torch tensors to the plain pointers
and sizes the C functions take.  It raises if the library is not built: there
is no other code path.
"""
from __future__ import annotations

import ctypes
import re
from pathlib import Path

import numpy as np

PKG = Path(__file__).resolve().parent
LIB_PATH = PKG / "libcodec_gb300.so"
HEADER = PKG.parent / "include" / "codec.h"

PRECISION_FP32 = 0
PRECISION_FP16X3 = 1
PRECISION_FP16 = 2       # single fp16 pass: approximate, outside the parity bound
STREAM_ERR_BAD_CODE = 1
STREAM_ERR_KERNEL_TIMEOUT = 0x80000000

STATUS = {0: "CODEC_OK", 1: "CODEC_ERR_NULL", 2: "CODEC_ERR_CONFIG", 3: "CODEC_ERR_WEIGHTS",
          4: "CODEC_ERR_ARG", 5: "CODEC_ERR_CAPACITY", 6: "CODEC_ERR_OOM", 7: "CODEC_ERR_CUDA",
          8: "CODEC_ERR_NO_DEVICE"}


class CodecError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)} ({_lib().codec_status_string(status).decode()})")


class CodecConfigC(ctypes.Structure):
    _fields_ = [
        ("Q", ctypes.c_int32), ("V", ctypes.c_int32), ("E", ctypes.c_int32), ("pre_k", ctypes.c_int32),
        ("d", ctypes.c_int32), ("heads", ctypes.c_int32), ("ffn", ctypes.c_int32),
        ("layers", ctypes.c_int32), ("window", ctypes.c_int32),
        ("n_up", ctypes.c_int32), ("up_k", ctypes.c_int32), ("up_s", ctypes.c_int32),
        ("up_ch", ctypes.c_int32 * 4),
        ("n_stages", ctypes.c_int32), ("strides", ctypes.c_int32 * 8), ("ch", ctypes.c_int32 * 8),
        ("n_rb", ctypes.c_int32), ("rb_k", ctypes.c_int32 * 4),
        ("n_dil", ctypes.c_int32), ("dil", ctypes.c_int32 * 4),
        ("final_k", ctypes.c_int32), ("rms_eps", ctypes.c_float),
        ("max_streams", ctypes.c_int32), ("max_chunk_frames", ctypes.c_int32),
        ("max_batch_frames", ctypes.c_int32), ("precision", ctypes.c_int32),
        ("latent_dim", ctypes.c_int32), ("tf_up", ctypes.c_int32),
    ]


KERNEL_KINDS = ["gather", "gemm_simt", "gemm_tc", "operand_prep", "rmsnorm", "attention", "final_conv",
                "history", "mrf_sum"]


class KernelStatsC(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("launches", ctypes.c_int32), ("ms", ctypes.c_double),
                ("flops", ctypes.c_double), ("bytes", ctypes.c_double)]


class LaunchRecordC(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("reserved", ctypes.c_int32), ("ms", ctypes.c_double),
                ("flops", ctypes.c_double), ("bytes", ctypes.c_double)]


class IstftConfigC(ctypes.Structure):
    _fields_ = [("n_fft", ctypes.c_int32), ("hop", ctypes.c_int32), ("mag_clip", ctypes.c_float),
                ("max_streams", ctypes.c_int32), ("max_chunk_frames", ctypes.c_int32)]


class SineConfigC(ctypes.Structure):
    _fields_ = [("upp", ctypes.c_int32), ("sample_rate", ctypes.c_float), ("harmonics", ctypes.c_int32),
                ("amplitude", ctypes.c_float), ("voiced_threshold", ctypes.c_float),
                ("max_streams", ctypes.c_int32), ("max_chunk_frames", ctypes.c_int32)]


class StftConfigC(ctypes.Structure):
    _fields_ = [("n_fft", ctypes.c_int32), ("hop", ctypes.c_int32), ("max_streams", ctypes.c_int32),
                ("max_chunk_frames", ctypes.c_int32)]


class ChunkScheduleC(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("first", ctypes.c_int32), ("steady", ctypes.c_int32),
                ("n_ramp", ctypes.c_int32), ("ramp", ctypes.c_int32 * 8)]


SCHEDULE_FIXED, SCHEDULE_RAMP, SCHEDULE_ADAPTIVE = 0, 1, 2


def chunk_schedule(kind: int, first: int = 1, steady: int = 25, ramp=()) -> ChunkScheduleC:
    c = ChunkScheduleC()
    c.kind, c.first, c.steady, c.n_ramp = kind, first, steady, len(ramp)
    for i, v in enumerate(ramp):
        c.ramp[i] = v
    return c


def chunk_frames(schedule: ChunkScheduleC, index: int, frames_delivered: int) -> int:
    """codec_chunk_frames: frames of chunk `index` under the schedule."""
    return _lib().codec_chunk_frames(ctypes.byref(schedule), index, frames_delivered)


def schedule_chunks(schedule: ChunkScheduleC, total_frames: int) -> list:
    """The chunk sizes the schedule gives for a stream of total_frames."""
    out, done = [], 0
    while done < total_frames:
        n = chunk_frames(schedule, len(out), done)
        if n <= 0:
            raise ValueError("invalid chunk schedule")
        n = min(n, total_frames - done)
        out.append(n)
        done += n
    return out


class VocosConfigC(ctypes.Structure):
    _fields_ = [("n_mels", ctypes.c_int32), ("d", ctypes.c_int32), ("ffn", ctypes.c_int32),
                ("layers", ctypes.c_int32), ("k", ctypes.c_int32), ("n_fft", ctypes.c_int32),
                ("hop", ctypes.c_int32), ("ln_eps", ctypes.c_float), ("mag_clip", ctypes.c_float),
                ("max_streams", ctypes.c_int32), ("max_chunk_frames", ctypes.c_int32),
                ("max_batch_frames", ctypes.c_int32), ("precision", ctypes.c_int32)]


class StreamInfoC(ctypes.Structure):
    _fields_ = [("frames_decoded", ctypes.c_int64), ("error_bits", ctypes.c_uint32),
                ("reserved", ctypes.c_int32)]


_L = None
_P = ctypes.c_void_p
_I32P = ctypes.POINTER(ctypes.c_int32)


def _lib():
    global _L
    if _L is None:
        if not LIB_PATH.exists():
            raise RuntimeError(f"CUDA library {LIB_PATH.name} is not built; run __graft_entry__.build()")
        l = ctypes.CDLL(str(LIB_PATH))
        i32, i64 = ctypes.c_int32, ctypes.c_int64
        cfgp = ctypes.POINTER(CodecConfigC)
        sig = {
            "codec_weight_floats": (i64, [cfgp]),
            "codec_create": (i32, [cfgp, ctypes.POINTER(ctypes.c_float), i64, ctypes.POINTER(_P)]),
            "codec_q8_bytes": (i64, [cfgp]),
            "codec_create_q8": (i32, [cfgp, _P, i64, ctypes.POINTER(_P)]),
            "codec_destroy": (None, [_P]),
            "codec_samples_per_frame": (i32, [_P]),
            "codec_state_create": (i32, [_P, i32, ctypes.POINTER(_P)]),
            "codec_state_destroy": (None, [_P]),
            "codec_state_reset": (i32, [_P, _I32P, i32, _P]),
            "codec_decode_chunk": (i32, [_P, _P, _I32P, _I32P, i32, i32, _P, _P]),
            "codec_decode_chunk_ex": (i32, [_P, _P, _I32P, _I32P, i32, i32, _P, _P, _P]),
            "codec_decode_latents": (i32, [_P, _P, _I32P, _I32P, i32, i32, _P, _P, _P]),
            "codec_decode_chunk_host": (i32, [_P, _P, _I32P, _I32P, i32, i32, _P, _P]),
            "codec_decode_recompute": (i32, [_P, _P, _I32P, _I32P, _I32P, i32, i32, _P, _P, _P]),
            "codec_chunk_frames": (i32, [ctypes.POINTER(ChunkScheduleC), i32, i64]),
            "codec_embed_chunk": (i32, [_P, _P, _I32P, _I32P, i32, i32, _P, _P]),
            "codec_state_query": (i32, [_P, i32, ctypes.POINTER(StreamInfoC), _P]),
            "codec_state_streams": (i32, [_P]),
            "codec_state_last_launches": (i32, [_P]),
            "codec_status_string": (ctypes.c_char_p, [i32]),
            "codec_profile_begin": (i32, [_P, i32]),
            "codec_state_set_graphs": (i32, [_P, i32]),
            "codec_state_conv1d": (i32, [_P, _P, i32, i32, _P, _P, _P, i32, i32, i32, _P, _P]),
            "codec_conv1d_noalloc": (i32, [_P, i32, i32, _P, _P, _P, i32, i32, i32, _P, _P]),
            "codec_conv1d_noalloc_status": (i32, [ctypes.POINTER(i32), _P]),
            "codec_state_set_wait_limit": (i32, [_P, ctypes.c_uint32, i32]),
            "codec_profile_end": (i32, [_P, ctypes.POINTER(KernelStatsC), _P]),
            "codec_profile_launches": (i32, [_P, ctypes.POINTER(LaunchRecordC), i32, ctypes.POINTER(i32)]),
            "codec_istft_create": (i32, [ctypes.POINTER(IstftConfigC), ctypes.POINTER(_P)]),
            "codec_istft_destroy": (None, [_P]),
            "codec_istft_reset": (i32, [_P, _I32P, i32, _P]),
            "codec_istft_decode": (i32, [_P, _P, _I32P, _I32P, i32, i32, _P, _P]),
            "codec_sine_create": (i32, [ctypes.POINTER(SineConfigC), ctypes.POINTER(_P)]),
            "codec_sine_destroy": (None, [_P]),
            "codec_sine_reset": (i32, [_P, _I32P, i32, _P]),
            "codec_sine_decode": (i32, [_P, _P, _I32P, _I32P, i32, i32, _P, _P]),
            "codec_vocos_weight_floats": (i64, [ctypes.POINTER(VocosConfigC)]),
            "codec_vocos_create": (i32, [ctypes.POINTER(VocosConfigC), ctypes.POINTER(ctypes.c_float), i64,
                                         ctypes.POINTER(_P)]),
            "codec_vocos_destroy": (None, [_P]),
            "codec_vocos_reset": (i32, [_P, _I32P, i32, _P]),
            "codec_vocos_decode": (i32, [_P, _P, _I32P, _I32P, i32, i32, _P, _P]),
            "codec_stft_create": (i32, [ctypes.POINTER(StftConfigC), ctypes.POINTER(_P)]),
            "codec_stft_destroy": (None, [_P]),
            "codec_stft_reset": (i32, [_P, _I32P, i32, _P]),
            "codec_stft_decode": (i32, [_P, _P, _I32P, _I32P, i32, i32, _P, _P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(l, name)
            fn.restype = res
            fn.argtypes = args
        _L = l
    return _L


def header_functions() -> list:
    """Names of the functions include/codec.h declares."""
    text = HEADER.read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(codec_[a-z0-9_]+)\s*\(", text)))


def config_c(cfg, max_streams=1, max_chunk_frames=97, max_batch_frames=None,
             precision=PRECISION_FP32) -> CodecConfigC:
    c = CodecConfigC()
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
    c.max_streams = max_streams
    c.max_chunk_frames = max_chunk_frames
    c.max_batch_frames = max_batch_frames if max_batch_frames is not None else max_chunk_frames * max_streams
    c.precision = precision
    c.latent_dim = cfg.latent_dim
    c.tf_up = cfg.tf_up
    return c


def weight_floats(cfg_c: CodecConfigC) -> int:
    return _lib().codec_weight_floats(ctypes.byref(cfg_c))


def q8_bytes(cfg_c: CodecConfigC) -> int:
    return _lib().codec_q8_bytes(ctypes.byref(cfg_c))


def _check(status: int, what: str):
    if status != 0:
        raise CodecError(status, what)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _conv1d_shapes(x, w, y, bias, alpha, dilation):
    """Shape and layout checks shared by both conv entry points' wrappers."""
    Cout, Cin, k = w.shape
    T = y.shape[0]
    for name, t in (("x", x), ("w", w), ("y", y), ("bias", bias), ("alpha", alpha)):
        if t is not None and not (t.is_cuda and t.is_contiguous() and str(t.dtype) == "torch.float32"):
            raise ValueError(f"{name} must be a contiguous float32 CUDA tensor")
    if tuple(x.shape) != ((k - 1) * dilation + T, Cin):
        raise ValueError(f"x must be [(k-1)*dilation + T][Cin] = [{(k - 1) * dilation + T}][{Cin}], got {tuple(x.shape)}")
    if tuple(y.shape) != (T, Cout):
        raise ValueError(f"y must be [T][Cout] = [{T}][{Cout}], got {tuple(y.shape)}")
    if bias is not None and bias.numel() != Cout:
        raise ValueError("bias must hold Cout values")
    if alpha is not None and alpha.numel() != Cin:
        raise ValueError("alpha must hold Cin values")
    return T, Cin, Cout, k


def conv1d_noalloc(x, w, y, bias=None, alpha=None, dilation=1, stream=None):
    """codec_conv1d_noalloc: the tensor-core causal conv with no device
    allocation (the library's fixed scratch array); same arguments as
    CodecState.conv1d."""
    T, Cin, Cout, k = _conv1d_shapes(x, w, y, bias, alpha, dilation)
    opt = lambda t: None if t is None else _ptr(t)
    _check(_lib().codec_conv1d_noalloc(_ptr(x), T, Cin, _ptr(w), opt(bias), opt(alpha), Cout, k, dilation,
                                       _ptr(y), _stream_handle(stream)), "codec_conv1d_noalloc")


def conv1d_noalloc_timed_out(stream=None) -> bool:
    """codec_conv1d_noalloc_status: whether the last allocation-free conv on the
    current device gave up on a bounded wait (synchronises the stream)."""
    flag = ctypes.c_int32()
    _check(_lib().codec_conv1d_noalloc_status(ctypes.byref(flag), _stream_handle(stream)),
           "codec_conv1d_noalloc_status")
    return bool(flag.value)


def vocos_config_c(cfg, max_streams=1, max_chunk_frames=64, max_batch_frames=None, precision=PRECISION_FP32):
    c = VocosConfigC()
    c.n_mels, c.d, c.ffn, c.layers, c.k = cfg.n_mels, cfg.d, cfg.ffn, cfg.layers, cfg.k
    c.n_fft, c.hop, c.ln_eps, c.mag_clip = cfg.n_fft, cfg.hop, cfg.ln_eps, cfg.mag_clip
    c.max_streams, c.max_chunk_frames = max_streams, max_chunk_frames
    c.max_batch_frames = max_batch_frames if max_batch_frames is not None else max_streams * max_chunk_frames
    c.precision = precision
    return c


def vocos_weight_floats(cfg_c) -> int:
    return _lib().codec_vocos_weight_floats(ctypes.byref(cfg_c))


class Vocos:
    """codec_vocos_*: the streaming Vocos-style generator + iSTFT head."""

    def __init__(self, cfg, blob, max_streams=1, max_chunk_frames=64, max_batch_frames=None,
                 precision=PRECISION_FP32):
        self.cfg = cfg
        self.cfg_c = vocos_config_c(cfg, max_streams, max_chunk_frames, max_batch_frames, precision)
        blob = np.ascontiguousarray(blob, dtype=np.float32)
        h = _P()
        _check(_lib().codec_vocos_create(ctypes.byref(self.cfg_c), blob.ctypes.data_as(ctypes.POINTER(ctypes.c_float)),
                                         blob.size, ctypes.byref(h)), "codec_vocos_create")
        self._h = h

    def close(self):
        if getattr(self, "_h", None):
            _lib().codec_vocos_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()

    def reset(self, stream_ids=None, stream=None):
        if stream_ids is None:
            _check(_lib().codec_vocos_reset(self._h, None, 0, _stream_handle(stream)), "codec_vocos_reset")
        else:
            ids = np.ascontiguousarray(stream_ids, dtype=np.int32)
            _check(_lib().codec_vocos_reset(self._h, ids.ctypes.data_as(_I32P), ids.size, _stream_handle(stream)),
                   "codec_vocos_reset")

    def decode(self, mel, n_frames, audio, stream_ids=None, stream=None):
        """mel: contiguous float32 CUDA [B][T_max][n_mels]; audio: float32 CUDA
        [B][T_max hop]; n_frames, stream_ids: host sequences of length B."""
        B, T_max, nm = mel.shape
        nf = np.ascontiguousarray(n_frames, dtype=np.int32)
        ids = None if stream_ids is None else np.ascontiguousarray(stream_ids, dtype=np.int32)
        if nf.size != B or (ids is not None and ids.size != B):
            raise ValueError("n_frames / stream_ids must have one entry per batch row")
        if nm != self.cfg.n_mels or not (mel.is_cuda and mel.is_contiguous() and str(mel.dtype) == "torch.float32"):
            raise ValueError(f"mel must be a contiguous float32 CUDA tensor [B][T_max][{self.cfg.n_mels}]")
        if not (audio.is_cuda and audio.is_contiguous() and audio.numel() >= B * T_max * self.cfg.hop):
            raise ValueError("audio must be a contiguous float32 CUDA tensor of B * T_max * hop values")
        ids_p = None if ids is None else ids.ctypes.data_as(_I32P)
        _check(_lib().codec_vocos_decode(self._h, _ptr(mel), nf.ctypes.data_as(_I32P), ids_p, B, T_max, _ptr(audio),
                                         _stream_handle(stream)), "codec_vocos_decode")


class Istft:
    """codec_istft_*: the streaming iSTFT head (log-magnitude / phase frames in,
    hop samples per frame out), with per-slot carried frames."""

    def __init__(self, n_fft: int, hop: int, mag_clip: float = 0.0, max_streams: int = 1,
                 max_chunk_frames: int = 64):
        c = IstftConfigC(n_fft, hop, mag_clip, max_streams, max_chunk_frames)
        h = _P()
        _check(_lib().codec_istft_create(ctypes.byref(c), ctypes.byref(h)), "codec_istft_create")
        self._h = h
        self.n_fft, self.hop, self.n_bins = n_fft, hop, n_fft // 2 + 1

    def close(self):
        if getattr(self, "_h", None):
            _lib().codec_istft_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()

    def reset(self, stream_ids=None, stream=None):
        if stream_ids is None:
            _check(_lib().codec_istft_reset(self._h, None, 0, _stream_handle(stream)), "codec_istft_reset")
        else:
            ids = np.ascontiguousarray(stream_ids, dtype=np.int32)
            _check(_lib().codec_istft_reset(self._h, ids.ctypes.data_as(_I32P), ids.size, _stream_handle(stream)),
                   "codec_istft_reset")

    def decode(self, spec, n_frames, audio, stream_ids=None, stream=None):
        """spec: contiguous float32 CUDA [B][T_max][2 n_bins]; audio: contiguous
        float32 CUDA [B][T_max hop]; n_frames and stream_ids: host sequences of
        length B."""
        B, T_max, width = spec.shape
        nf = np.ascontiguousarray(n_frames, dtype=np.int32)
        ids = None if stream_ids is None else np.ascontiguousarray(stream_ids, dtype=np.int32)
        if nf.size != B or (ids is not None and ids.size != B):
            raise ValueError("n_frames / stream_ids must have one entry per batch row")
        if width != 2 * self.n_bins or not (spec.is_cuda and spec.is_contiguous() and str(spec.dtype) == "torch.float32"):
            raise ValueError(f"spec must be a contiguous float32 CUDA tensor [B][T_max][{2 * self.n_bins}]")
        if not (audio.is_cuda and audio.is_contiguous() and audio.numel() >= B * T_max * self.hop):
            raise ValueError("audio must be a contiguous float32 CUDA tensor of B * T_max * hop values")
        ids_p = None if ids is None else ids.ctypes.data_as(_I32P)
        _check(_lib().codec_istft_decode(self._h, _ptr(spec), nf.ctypes.data_as(_I32P), ids_p, B, T_max,
                                         _ptr(audio), _stream_handle(stream)), "codec_istft_decode")


class _Streamed:
    """Shared marshalling of the per-stream ops (create / reset / decode / destroy)."""
    _prefix = ""

    def _create(self, cfg):
        h = _P()
        _check(getattr(_lib(), self._prefix + "create")(ctypes.byref(cfg), ctypes.byref(h)), self._prefix + "create")
        self._h = h

    def close(self):
        if getattr(self, "_h", None):
            getattr(_lib(), self._prefix + "destroy")(self._h)
            self._h = None

    def __del__(self):
        self.close()

    def reset(self, stream_ids=None, stream=None):
        fn = getattr(_lib(), self._prefix + "reset")
        if stream_ids is None:
            _check(fn(self._h, None, 0, _stream_handle(stream)), self._prefix + "reset")
        else:
            ids = np.ascontiguousarray(stream_ids, dtype=np.int32)
            _check(fn(self._h, ids.ctypes.data_as(_I32P), ids.size, _stream_handle(stream)), self._prefix + "reset")

    def _decode(self, inp, n_frames, out, stream_ids, stream, in_per_frame, out_per_frame):
        B, T_max = inp.shape[0], inp.shape[1] if inp.dim() > 1 else 1
        nf = np.ascontiguousarray(n_frames, dtype=np.int32)
        ids = None if stream_ids is None else np.ascontiguousarray(stream_ids, dtype=np.int32)
        if nf.size != B or (ids is not None and ids.size != B):
            raise ValueError("n_frames / stream_ids must have one entry per batch row")
        for t, per in ((inp, in_per_frame), (out, out_per_frame)):
            if not (t.is_cuda and t.is_contiguous() and str(t.dtype) == "torch.float32"):
                raise ValueError("arguments must be contiguous float32 CUDA tensors")
        if inp.numel() != B * T_max * in_per_frame or out.numel() < B * T_max * out_per_frame:
            raise ValueError("tensor sizes do not match the call")
        ids_p = None if ids is None else ids.ctypes.data_as(_I32P)
        _check(getattr(_lib(), self._prefix + "decode")(self._h, _ptr(inp), nf.ctypes.data_as(_I32P), ids_p, B,
                                                        T_max, _ptr(out), _stream_handle(stream)),
               self._prefix + "decode")


class SineSource(_Streamed):
    """codec_sine_*: harmonic sine source, F0 frames in, [samples][harmonics] out."""
    _prefix = "codec_sine_"

    def __init__(self, upp: int, sample_rate: float, harmonics: int, amplitude: float = 0.1,
                 voiced_threshold: float = 0.0, max_streams: int = 1, max_chunk_frames: int = 64):
        self.upp, self.harmonics = upp, harmonics
        self._create(SineConfigC(upp, sample_rate, harmonics, amplitude, voiced_threshold, max_streams,
                                 max_chunk_frames))

    def decode(self, f0, n_frames, out, stream_ids=None, stream=None):
        """f0: float32 CUDA [B][T_max]; out: float32 CUDA [B][T_max upp][harmonics]."""
        self._decode(f0, n_frames, out, stream_ids, stream, 1, self.upp * self.harmonics)


class Stft(_Streamed):
    """codec_stft_*: causal analysis STFT, hop samples per frame in, 2 (n_fft / 2 + 1) values per frame out."""
    _prefix = "codec_stft_"

    def __init__(self, n_fft: int, hop: int, max_streams: int = 1, max_chunk_frames: int = 64):
        self.n_fft, self.hop, self.n_bins = n_fft, hop, n_fft // 2 + 1
        self._create(StftConfigC(n_fft, hop, max_streams, max_chunk_frames))

    def decode(self, x, n_frames, spec, stream_ids=None, stream=None):
        """x: float32 CUDA [B][T_max][hop]; spec: float32 CUDA [B][T_max][2 n_bins]."""
        self._decode(x, n_frames, spec, stream_ids, stream, self.hop, 2 * self.n_bins)


class Codec:
    """codec_create / codec_destroy: the weights on the current CUDA device."""

    def __init__(self, cfg, blob: np.ndarray = None, q8: bytes = None, **capacity):
        """blob: the fp32 weight blob (codec_create), or q8: the same weights in
        the int8-per-32 storage format (codec_create_q8; see weights_q8.py)."""
        self.cfg = cfg
        self.cfg_c = config_c(cfg, **capacity)
        h = ctypes.c_void_p()
        if q8 is not None:
            buf = np.frombuffer(q8, dtype=np.uint8)
            _check(_lib().codec_create_q8(ctypes.byref(self.cfg_c), buf.ctypes.data_as(ctypes.c_void_p), buf.size,
                                          ctypes.byref(h)), "codec_create_q8")
        else:
            blob = np.ascontiguousarray(blob, dtype=np.float32)
            _check(_lib().codec_create(ctypes.byref(self.cfg_c), blob.ctypes.data_as(ctypes.POINTER(ctypes.c_float)),
                                       blob.size, ctypes.byref(h)), "codec_create")
        self._h = h
        self.samples_per_frame = _lib().codec_samples_per_frame(h)

    def close(self):
        if getattr(self, "_h", None):
            _lib().codec_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()

    def state(self, n_streams: int = 0) -> "CodecState":
        return CodecState(self, n_streams)


class CodecState:
    """codec_state_*: stream slots plus the per-call workspace."""

    def __init__(self, codec: Codec, n_streams: int = 0):
        self.codec = codec
        h = ctypes.c_void_p()
        _check(_lib().codec_state_create(codec._h, n_streams, ctypes.byref(h)), "codec_state_create")
        self._h = h
        self.n_streams = _lib().codec_state_streams(h)

    def close(self):
        if getattr(self, "_h", None):
            _lib().codec_state_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()

    def reset(self, stream_ids=None, stream=None):
        if stream_ids is None:
            _check(_lib().codec_state_reset(self._h, None, 0, _stream_handle(stream)), "codec_state_reset")
        else:
            ids = np.ascontiguousarray(stream_ids, dtype=np.int32)
            _check(_lib().codec_state_reset(self._h, ids.ctypes.data_as(_I32P), ids.size, _stream_handle(stream)),
                   "codec_state_reset")

    def decode(self, codes, n_frames, audio, stream_ids=None, pre_tanh=None, stream=None):
        """codes: device int32 tensor [B][Q][T_max]; audio: device float32
        [B][T_max * spf]; n_frames and stream_ids: host sequences of length B."""
        B, Q, T_max = codes.shape
        nf = np.ascontiguousarray(n_frames, dtype=np.int32)
        ids = None if stream_ids is None else np.ascontiguousarray(stream_ids, dtype=np.int32)
        if nf.size != B or (ids is not None and ids.size != B):
            raise ValueError("n_frames / stream_ids must have one entry per batch row")
        if not (codes.is_cuda and codes.dtype.__str__() == "torch.int32" and codes.is_contiguous()):
            raise ValueError("codes must be a contiguous int32 CUDA tensor")
        if not (audio.is_cuda and audio.is_contiguous() and audio.numel() >= B * T_max * self.codec.samples_per_frame):
            raise ValueError("audio must be a contiguous float32 CUDA tensor of B * T_max * spf values")
        ids_p = None if ids is None else ids.ctypes.data_as(_I32P)
        st = _stream_handle(stream)
        if pre_tanh is None:
            s = _lib().codec_decode_chunk(self._h, _ptr(codes), nf.ctypes.data_as(_I32P), ids_p, B, T_max,
                                          _ptr(audio), st)
        else:
            s = _lib().codec_decode_chunk_ex(self._h, _ptr(codes), nf.ctypes.data_as(_I32P), ids_p, B, T_max,
                                             _ptr(audio), _ptr(pre_tanh), st)
        _check(s, "codec_decode_chunk")

    def decode_latents(self, latents, n_frames, audio, stream_ids=None, pre_tanh=None, stream=None):
        """codec_decode_latents: latents device float32 [B][T_max][L]; audio
        device float32 [B][T_max * spf]; n_frames and stream_ids host, length B."""
        B, T_max, L = latents.shape
        nf = np.ascontiguousarray(n_frames, dtype=np.int32)
        ids = None if stream_ids is None else np.ascontiguousarray(stream_ids, dtype=np.int32)
        if nf.size != B or (ids is not None and ids.size != B):
            raise ValueError("n_frames / stream_ids must have one entry per batch row")
        if not (latents.is_cuda and str(latents.dtype) == "torch.float32" and latents.is_contiguous()):
            raise ValueError("latents must be a contiguous float32 CUDA tensor")
        if L != self.codec.cfg.latent_dim:
            raise ValueError(f"latents must have {self.codec.cfg.latent_dim} channels")
        if not (audio.is_cuda and audio.is_contiguous() and audio.numel() >= B * T_max * self.codec.samples_per_frame):
            raise ValueError("audio must be a contiguous float32 CUDA tensor of B * T_max * spf values")
        ids_p = None if ids is None else ids.ctypes.data_as(_I32P)
        pt = None if pre_tanh is None else _ptr(pre_tanh)
        _check(_lib().codec_decode_latents(self._h, _ptr(latents), nf.ctypes.data_as(_I32P), ids_p, B, T_max,
                                           _ptr(audio), pt, _stream_handle(stream)), "codec_decode_latents")

    def decode_recompute(self, codes, n_ctx, n_new, audio, stream_ids=None, pre_tanh=None, stream=None):
        """codec_decode_recompute: per entry, reset its slot, decode n_ctx + n_new
        frames of its codes row and write only the n_new frames' audio."""
        B, Q, T_max = codes.shape
        nc = np.ascontiguousarray(n_ctx, dtype=np.int32)
        nn = np.ascontiguousarray(n_new, dtype=np.int32)
        ids = None if stream_ids is None else np.ascontiguousarray(stream_ids, dtype=np.int32)
        if nc.size != B or nn.size != B or (ids is not None and ids.size != B):
            raise ValueError("n_ctx / n_new / stream_ids must have one entry per batch row")
        if not (codes.is_cuda and str(codes.dtype) == "torch.int32" and codes.is_contiguous()):
            raise ValueError("codes must be a contiguous int32 CUDA tensor")
        if not (audio.is_cuda and audio.is_contiguous() and audio.numel() >= B * T_max * self.codec.samples_per_frame):
            raise ValueError("audio must be a contiguous float32 CUDA tensor of B * T_max * spf values")
        ids_p = None if ids is None else ids.ctypes.data_as(_I32P)
        pt = None if pre_tanh is None else _ptr(pre_tanh)
        _check(_lib().codec_decode_recompute(self._h, _ptr(codes), nc.ctypes.data_as(_I32P), nn.ctypes.data_as(_I32P),
                                             ids_p, B, T_max, _ptr(audio), pt, _stream_handle(stream)),
               "codec_decode_recompute")

    def embed(self, codes, n_frames, emb, stream_ids=None, stream=None):
        """Codebook sum only: emb device float32 [sum(n_frames)][E]."""
        B, Q, T_max = codes.shape
        nf = np.ascontiguousarray(n_frames, dtype=np.int32)
        ids = None if stream_ids is None else np.ascontiguousarray(stream_ids, dtype=np.int32)
        ids_p = None if ids is None else ids.ctypes.data_as(_I32P)
        _check(_lib().codec_embed_chunk(self._h, _ptr(codes), nf.ctypes.data_as(_I32P), ids_p, B, T_max,
                                        _ptr(emb), _stream_handle(stream)), "codec_embed_chunk")

    def decode_host(self, codes, n_frames, audio, stream_ids=None, stream=None):
        """Host-buffer form: codes int32 [B][Q][T_max] and audio float32
        [B][T_max * spf] are CPU tensors (pinned for asynchronous copies)."""
        B, Q, T_max = codes.shape
        nf = np.ascontiguousarray(n_frames, dtype=np.int32)
        ids = None if stream_ids is None else np.ascontiguousarray(stream_ids, dtype=np.int32)
        ids_p = None if ids is None else ids.ctypes.data_as(_I32P)
        _check(_lib().codec_decode_chunk_host(self._h, _ptr(codes), nf.ctypes.data_as(_I32P), ids_p, B, T_max,
                                              _ptr(audio), _stream_handle(stream)), "codec_decode_chunk_host")

    def conv1d(self, x, w, y, bias=None, alpha=None, dilation=1, stream=None):
        """codec_state_conv1d: x [(k-1) dil + T][Cin], w [Cout][Cin][k], y [T][Cout]
        (contiguous float32 CUDA tensors); bias [Cout], alpha [Cin] optional."""
        T, Cin, Cout, k = _conv1d_shapes(x, w, y, bias, alpha, dilation)
        opt = lambda t: None if t is None else _ptr(t)
        _check(_lib().codec_state_conv1d(self._h, _ptr(x), T, Cin, _ptr(w), opt(bias), opt(alpha), Cout, k,
                                         dilation, _ptr(y), _stream_handle(stream)), "codec_state_conv1d")

    def query(self, stream_id: int, stream=None):
        info = StreamInfoC()
        _check(_lib().codec_state_query(self._h, stream_id, ctypes.byref(info), _stream_handle(stream)),
               "codec_state_query")
        return int(info.frames_decoded), int(info.error_bits)

    def set_wait_limit(self, polls: int = 0, unarrived_wait: bool = False):
        """codec_state_set_wait_limit: polls per bounded wait of the tensor-core
        kernels (0: default); unarrived_wait makes each GEMM CTA's first
        epilogue wait run out, to verify the timeout path."""
        _check(_lib().codec_state_set_wait_limit(self._h, polls, 1 if unarrived_wait else 0),
               "codec_state_set_wait_limit")

    def set_graphs(self, enable: bool):
        _check(_lib().codec_state_set_graphs(self._h, 1 if enable else 0), "codec_state_set_graphs")

    def profile_begin(self, max_records: int = 65536):
        _check(_lib().codec_profile_begin(self._h, max_records), "codec_profile_begin")

    def profile_end(self, stream=None) -> dict:
        """Per kernel kind: launches, summed event ms, algorithmic flops and bytes."""
        arr = (KernelStatsC * len(KERNEL_KINDS))()
        _check(_lib().codec_profile_end(self._h, arr, _stream_handle(stream)), "codec_profile_end")
        return {KERNEL_KINDS[i]: dict(launches=arr[i].launches, ms=arr[i].ms, flops=arr[i].flops,
                                      bytes=arr[i].bytes) for i in range(len(KERNEL_KINDS))}

    def profile_launches(self, max_out: int = 1 << 20) -> list:
        """Per-launch (kind, ms, flops, bytes) of the last profiled interval, in order."""
        arr = (LaunchRecordC * max_out)()
        n = ctypes.c_int32()
        _check(_lib().codec_profile_launches(self._h, arr, max_out, ctypes.byref(n)), "codec_profile_launches")
        return [(KERNEL_KINDS[arr[i].kind], arr[i].ms, arr[i].flops, arr[i].bytes) for i in range(n.value)]

    @property
    def last_launches(self) -> int:
        return _lib().codec_state_last_launches(self._h)
