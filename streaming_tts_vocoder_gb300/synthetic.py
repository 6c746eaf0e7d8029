"""Seeded synthetic inputs for the streaming codec decoder.

This module holds the decoder configurations (layer sizes only), the weight
manifest (tensor names, shapes and initial distributions, in the order of the
flat fp32 weight blob), and the seeded generators for weights and codes.  It
holds none of the decoder's arithmetic: it is the one module that both the CPU
oracle and the CUDA library are fed from.

Sources for the shapes (vllm-omni "Edge TTS design", section 1.3: RVQ
embedding sum, causal conv, 8-layer sliding-window (72 frames) transformer,
2x2 upsampling, BigVGAN/Snake stack, 24 kHz, 1920 samples per frame; section
4: decoder dims 25 + 72 frames).  No trained weights exist here: every tensor
is random, N(0, 1/fan_in) with a fixed seed, Snake alphas U[0.5, 1.5].

Blob order (all fp32, PyTorch layouts):

  cb.{q}                [V][E]               q = 0..Q-1
  pre.w, pre.b          [d][E][pre_k], [d]   Conv1d weight [out][in][tap]
  tf.{l}.n1             [d]                  RMSNorm gain before attention
  tf.{l}.wq/.wk/.wv/.wo [d][d]               Linear weight [out][in]
  tf.{l}.n2             [d]                  RMSNorm gain before the MLP
  tf.{l}.w1, tf.{l}.w2  [F][d], [d][F]
  tf.norm               [d]                  final RMSNorm gain
  up.{u}.w, up.{u}.b    [Cin][Cout][4], [Cout]   ConvTranspose1d [in][out][tap]
  st.{s}.alpha          [C_{s}]              Snake before the stage's ConvT
  st.{s}.w, st.{s}.b    [C_s][C_{s+1}][2*stride], [C_{s+1}]
  st.{s}.rb.{j}.{i}.alpha / .w / .b   [C][C][k_j] resblock j, dilation i
  out.alpha, out.w, out.b             [C_4], [1][C_4][final_k], [1]
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field

import numpy as np

SAMPLE_RATE = 24000
FRAME_RATE_HZ = 12.5


@dataclass(frozen=True)
class CodecConfig:
    name: str
    Q: int                 # codebooks
    V: int                 # entries per codebook
    E: int                 # codebook width
    pre_k: int             # causal pre-conv kernel
    d: int                 # transformer width
    heads: int
    ffn: int
    layers: int
    window: int            # keys per query, including itself
    up_channels: tuple     # outputs of the two latent ConvT(k=4, s=2)
    strides: tuple         # BigVGAN stage strides
    channels: tuple        # stage channels C_1..C_4 (C_0 = up_channels[-1])
    rb_kernels: tuple      # resblock kernel sizes of the MRF
    dilations: tuple
    final_k: int
    rms_eps: float = 1e-5
    up_k: int = 4
    up_s: int = 2

    @property
    def samples_per_frame(self) -> int:
        n = 1
        for _ in self.up_channels:
            n *= self.up_s
        for s in self.strides:
            n *= s
        return n

    @property
    def stage_in_channels(self) -> tuple:
        return (self.up_channels[-1],) + tuple(self.channels[:-1])

    def replace(self, **kw) -> "CodecConfig":
        return dataclasses.replace(self, **kw)


def tiny_config() -> CodecConfig:
    """The oracle-check decoder: Q=4 x 256 x 64, d=64, 1 layer, window 8."""
    return CodecConfig(
        name="tiny", Q=4, V=256, E=64, pre_k=3, d=64, heads=4, ffn=128,
        layers=1, window=8, up_channels=(64, 64), strides=(8, 5, 4, 3),
        channels=(32, 16, 8, 4), rb_kernels=(3,), dilations=(1, 3, 5),
        final_k=7)


def qwen3_config() -> CodecConfig:
    """Qwen3-TTS-12Hz-shaped decoder: Q=16 x 2048 x 512, d=1024, 8 layers,
    window 72, stages 1536 -> 768 -> 384 -> 192 -> 96, MRF k in {3, 7, 11}."""
    return CodecConfig(
        name="qwen3", Q=16, V=2048, E=512, pre_k=3, d=1024, heads=16,
        ffn=4096, layers=8, window=72, up_channels=(1024, 1536),
        strides=(8, 5, 4, 3), channels=(768, 384, 192, 96),
        rb_kernels=(3, 7, 11), dilations=(1, 3, 5), final_k=7)


CONFIGS = {"tiny": tiny_config, "qwen3": qwen3_config}


@dataclass(frozen=True)
class TensorSpec:
    name: str
    shape: tuple
    init: str        # "normal" | "uniform" | "gain"
    std: float = 0.0

    @property
    def size(self) -> int:
        n = 1
        for s in self.shape:
            n *= s
        return n


def weight_manifest(cfg: CodecConfig) -> list:
    """Tensor list in blob order (see the module docstring)."""
    m = []

    def normal(name, shape, fan_in):
        m.append(TensorSpec(name, tuple(shape), "normal", float(fan_in) ** -0.5))

    for q in range(cfg.Q):
        normal(f"cb.{q}", (cfg.V, cfg.E), cfg.Q)          # sum of Q rows has unit variance
    normal("pre.w", (cfg.d, cfg.E, cfg.pre_k), cfg.E * cfg.pre_k)
    normal("pre.b", (cfg.d,), cfg.E * cfg.pre_k)
    for l in range(cfg.layers):
        m.append(TensorSpec(f"tf.{l}.n1", (cfg.d,), "gain"))
        for w in ("wq", "wk", "wv", "wo"):
            normal(f"tf.{l}.{w}", (cfg.d, cfg.d), cfg.d)
        m.append(TensorSpec(f"tf.{l}.n2", (cfg.d,), "gain"))
        normal(f"tf.{l}.w1", (cfg.ffn, cfg.d), cfg.d)
        normal(f"tf.{l}.w2", (cfg.d, cfg.ffn), cfg.ffn)
    m.append(TensorSpec("tf.norm", (cfg.d,), "gain"))
    cin = cfg.d
    for u, cout in enumerate(cfg.up_channels):
        normal(f"up.{u}.w", (cin, cout, cfg.up_k), 2 * cin)   # two taps reach each output
        normal(f"up.{u}.b", (cout,), 2 * cin)
        cin = cout
    for s, (stride, cout) in enumerate(zip(cfg.strides, cfg.channels)):
        m.append(TensorSpec(f"st.{s}.alpha", (cin,), "uniform"))
        normal(f"st.{s}.w", (cin, cout, 2 * stride), 2 * cin)
        normal(f"st.{s}.b", (cout,), 2 * cin)
        for j, k in enumerate(cfg.rb_kernels):
            for i, _ in enumerate(cfg.dilations):
                m.append(TensorSpec(f"st.{s}.rb.{j}.{i}.alpha", (cout,), "uniform"))
                normal(f"st.{s}.rb.{j}.{i}.w", (cout, cout, k), cout * k)
                normal(f"st.{s}.rb.{j}.{i}.b", (cout,), cout * k)
        cin = cout
    m.append(TensorSpec("out.alpha", (cin,), "uniform"))
    normal("out.w", (1, cin, cfg.final_k), cin * cfg.final_k)
    normal("out.b", (1,), cin * cfg.final_k)
    return m


def blob_size(cfg: CodecConfig) -> int:
    return sum(t.size for t in weight_manifest(cfg))


def make_weights(cfg: CodecConfig, seed: int = 0) -> dict:
    """Seeded weights, drawn tensor by tensor in blob order from PCG64(seed)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    out = {}
    for t in weight_manifest(cfg):
        if t.init == "normal":
            a = rng.standard_normal(t.shape) * t.std
        elif t.init == "uniform":
            a = rng.uniform(0.5, 1.5, t.shape)
        elif t.init == "gain":
            a = 1.0 + 0.1 * rng.standard_normal(t.shape)
        else:
            raise ValueError(t.init)
        out[t.name] = np.ascontiguousarray(a, dtype=np.float32)
    return out


def pack_blob(cfg: CodecConfig, weights: dict) -> np.ndarray:
    """Concatenate the tensors in blob order into one contiguous fp32 array."""
    parts = []
    for t in weight_manifest(cfg):
        a = np.asarray(weights[t.name], dtype=np.float32)
        if a.shape != t.shape:
            raise ValueError(f"{t.name}: shape {a.shape} != {t.shape}")
        parts.append(a.reshape(-1))
    return np.ascontiguousarray(np.concatenate(parts))


def make_codes(cfg: CodecConfig, frames: int, seed: int = 0) -> np.ndarray:
    """Codes int32 [Q][frames], uniform in [0, V) from PCG64(seed)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return np.ascontiguousarray(rng.integers(0, cfg.V, size=(cfg.Q, frames)), dtype=np.int32)


def staggered_schedule(n_streams: int, frames: int, chunk: int = 25):
    """Ragged batching workload: stream s starts at global frame s mod chunk and
    is cut into chunks on global chunk boundaries, so its first chunk has
    chunk - (s mod chunk) frames, its last one the remainder.

    Returns a list of ticks; each tick is a list of (stream, first_frame,
    n_frames) with n_frames > 0.
    """
    offsets = [s % chunk for s in range(n_streams)]
    end = max(o + frames for o in offsets)
    ticks = []
    t0 = 0
    while t0 < end:
        tick = []
        for s, o in enumerate(offsets):
            a = max(t0, o) - o
            b = min(t0 + chunk, o + frames) - o
            if b > a:
                tick.append((s, a, b - a))
        if tick:
            ticks.append(tick)
        t0 += chunk
    return ticks


def make_istft_spec(n_fft: int, frames: int, seed: int, logmag_mean: float = -1.0,
                    logmag_std: float = 1.0) -> np.ndarray:
    """Seeded iSTFT-head input [frames][2 (n_fft / 2 + 1)] float32: log-magnitudes
    N(logmag_mean, logmag_std), then phases U[-pi, pi)."""
    nb = n_fft // 2 + 1
    rng = np.random.default_rng(seed)
    lm = rng.normal(logmag_mean, logmag_std, (frames, nb))
    ph = rng.uniform(-np.pi, np.pi, (frames, nb))
    return np.concatenate([lm, ph], axis=1).astype(np.float32)


def make_f0(frames: int, seed: int, voiced_fraction: float = 0.7) -> np.ndarray:
    """Seeded F0 contour [frames] float32 in Hz: voiced runs with F0 drifting in
    [80, 400] Hz, unvoiced frames (0 Hz) with probability 1 - voiced_fraction."""
    rng = np.random.default_rng(seed)
    f = np.clip(200.0 + np.cumsum(rng.normal(0.0, 8.0, frames)), 80.0, 400.0)
    f[rng.random(frames) >= voiced_fraction] = 0.0
    return f.astype(np.float32)
