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

Latent-input variant (latent_dim L > 0; blixt/phonon "Weights": the codec's
latent projection, 1x1 without bias, and its depthwise x16 upsampling; the
codec transformer at the upsampled 200 Hz rate, "Speed" item 7), in place of
cb.* and pre.*:

  lat.mu, lat.sigma     [L], [L]             denormalisation z = x sigma + mu
  lat.proj              [d][L]               1x1 projection, no bias
  lat.up.w, lat.up.b    [d][1][2 tf_up], [d] depthwise ConvTranspose1d (groups = d)

and no latent ConvTs after the transformer (up_channels empty, C_0 = d).
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
    latent_dim: int = 0    # 0: RVQ codes in; L > 0: latent frames of L channels in
    tf_up: int = 1         # latent input: depthwise upsampling stride before the transformer

    @property
    def samples_per_frame(self) -> int:
        n = self.tf_up if self.latent_dim else 1
        for _ in self.up_channels:
            n *= self.up_s
        for s in self.strides:
            n *= s
        return n

    @property
    def stage_in_channels(self) -> tuple:
        c0 = self.up_channels[-1] if self.up_channels else self.d
        return (c0,) + tuple(self.channels[:-1])

    @property
    def rows_per_frame_tf(self) -> int:
        """Transformer rows (positions) per frame."""
        return self.tf_up if self.latent_dim else 1

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


def mimi_config() -> CodecConfig:
    """Latent-input, Mimi-style decoder (the blixt/phonon codec outline): 32
    latent channels at 12.5 Hz, denormalised, projected 1x1 to d = 512 and
    upsampled x16 by a depthwise transposed conv to 200 Hz; 8 transformer
    layers (8 heads, FFN 2048) with a 251-position window at 200 Hz; stages
    x5, x4, x3, x2 (200 Hz -> 24 kHz), channels 512 -> 256 -> 128 -> 64 -> 32,
    one resblock k = 3 with dilations 1, 3, 5 each; final conv k = 7."""
    return CodecConfig(
        name="mimi", Q=0, V=0, E=0, pre_k=0, d=512, heads=8, ffn=2048, layers=8, window=251,
        up_channels=(), strides=(5, 4, 3, 2), channels=(256, 128, 64, 32), rb_kernels=(3,),
        dilations=(1, 3, 5), final_k=7, latent_dim=32, tf_up=16)


def tiny_mimi_config() -> CodecConfig:
    """The latent-input variant at oracle-check size: L = 16, d = 64, one
    layer, window 24 (1.5 frames at 16 rows per frame), stages 5, 4, 3, 2 with
    channels 64 -> 32 -> 16 -> 8 -> 4."""
    return CodecConfig(
        name="tiny_mimi", Q=0, V=0, E=0, pre_k=0, d=64, heads=4, ffn=128, layers=1, window=24,
        up_channels=(), strides=(5, 4, 3, 2), channels=(32, 16, 8, 4), rb_kernels=(3,),
        dilations=(1, 3, 5), final_k=7, latent_dim=16, tf_up=16)


CONFIGS = {"tiny": tiny_config, "qwen3": qwen3_config, "mimi": mimi_config, "tiny_mimi": tiny_mimi_config}


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

    if cfg.latent_dim:
        L = cfg.latent_dim
        m.append(TensorSpec("lat.mu", (L,), "normal", 0.1))
        m.append(TensorSpec("lat.sigma", (L,), "uniform"))
        normal("lat.proj", (cfg.d, L), L)
        normal("lat.up.w", (cfg.d, 1, 2 * cfg.tf_up), 2)     # two taps reach each output
        normal("lat.up.b", (cfg.d,), 2)
    else:
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


def make_latents(cfg: CodecConfig, frames: int, seed: int = 0) -> np.ndarray:
    """Latent frames float32 [frames][L], standard normal from PCG64(seed)
    (the normalised latents a flow head would emit)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return np.ascontiguousarray(rng.standard_normal((frames, cfg.latent_dim)), dtype=np.float32)


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


# ------------------------------------------------------------------ Vocos --
# A Vocos-style generator in front of the streaming iSTFT head (vox: "F5 ->
# Vocos -> iSTFT"): mel frames -> causal embedding conv -> LayerNorm -> L
# ConvNeXt blocks (causal depthwise conv, LayerNorm, pointwise MLP with GELU,
# layer scale, residual) -> LayerNorm -> linear head to n_fft / 2 + 1
# log-magnitudes and as many phases -> iSTFT.  Shapes follow the public
# 24 kHz mel model (100 mels, width 512, MLP 1536, 8 blocks, n_fft 1024, hop
# 256); nothing here holds its arithmetic.

@dataclass(frozen=True)
class VocosConfig:
    name: str
    n_mels: int
    d: int
    ffn: int
    layers: int
    k: int          # embedding and depthwise kernels
    n_fft: int
    hop: int
    ln_eps: float = 1e-6
    mag_clip: float = 100.0

    @property
    def n_bins(self) -> int:
        return self.n_fft // 2 + 1


def vocos_config() -> VocosConfig:
    return VocosConfig(name="vocos", n_mels=100, d=512, ffn=1536, layers=8, k=7, n_fft=1024, hop=256)


def tiny_vocos_config() -> VocosConfig:
    return VocosConfig(name="tiny_vocos", n_mels=32, d=64, ffn=192, layers=2, k=7, n_fft=64, hop=16)


def vocos_manifest(cfg: VocosConfig) -> list:
    """Tensor list in blob order:
      embed.w [d][n_mels][k], embed.b [d], norm.g, norm.b [d];
      per block l: dw.w [d][1][k], dw.b [d], ln.g, ln.b [d], pw1.w [ffn][d], pw1.b [ffn],
                   pw2.w [d][ffn], pw2.b [d], gamma [d];
      final.g, final.b [d]; head.w [n_fft + 2][d], head.b [n_fft + 2]."""
    m = []

    def normal(name, shape, fan_in):
        m.append(TensorSpec(name, tuple(shape), "normal", float(fan_in) ** -0.5))

    normal("embed.w", (cfg.d, cfg.n_mels, cfg.k), cfg.n_mels * cfg.k)
    normal("embed.b", (cfg.d,), cfg.n_mels * cfg.k)
    m.append(TensorSpec("norm.g", (cfg.d,), "gain"))
    m.append(TensorSpec("norm.b", (cfg.d,), "normal", 0.1))
    for l in range(cfg.layers):
        normal(f"blk.{l}.dw.w", (cfg.d, 1, cfg.k), cfg.k)
        normal(f"blk.{l}.dw.b", (cfg.d,), cfg.k)
        m.append(TensorSpec(f"blk.{l}.ln.g", (cfg.d,), "gain"))
        m.append(TensorSpec(f"blk.{l}.ln.b", (cfg.d,), "normal", 0.1))
        normal(f"blk.{l}.pw1.w", (cfg.ffn, cfg.d), cfg.d)
        normal(f"blk.{l}.pw1.b", (cfg.ffn,), cfg.d)
        normal(f"blk.{l}.pw2.w", (cfg.d, cfg.ffn), cfg.ffn)
        normal(f"blk.{l}.pw2.b", (cfg.d,), cfg.ffn)
        m.append(TensorSpec(f"blk.{l}.gamma", (cfg.d,), "scale", 1.0 / cfg.layers))
    m.append(TensorSpec("final.g", (cfg.d,), "gain"))
    m.append(TensorSpec("final.b", (cfg.d,), "normal", 0.1))
    normal("head.w", (cfg.n_fft + 2, cfg.d), cfg.d)
    normal("head.b", (cfg.n_fft + 2,), cfg.d)
    return m


def make_vocos_weights(cfg: VocosConfig, seed: int = 0) -> dict:
    """Seeded weights in blob order from PCG64(seed); layer scales start at
    1 / layers (times 1 + 0.1 N(0, 1), so that folding them into the second
    MLP layer is exercised with distinct values)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    out = {}
    for t in vocos_manifest(cfg):
        if t.init == "normal":
            a = rng.standard_normal(t.shape) * t.std
        elif t.init == "gain":
            a = 1.0 + 0.1 * rng.standard_normal(t.shape)
        elif t.init == "scale":
            a = t.std * (1.0 + 0.1 * rng.standard_normal(t.shape))
        else:
            raise ValueError(t.init)
        out[t.name] = np.ascontiguousarray(a, dtype=np.float32)
    return out


def pack_vocos_blob(cfg: VocosConfig, weights: dict) -> np.ndarray:
    parts = []
    for t in vocos_manifest(cfg):
        a = np.asarray(weights[t.name], dtype=np.float32)
        if a.shape != t.shape:
            raise ValueError(f"{t.name}: shape {a.shape} != {t.shape}")
        parts.append(a.reshape(-1))
    return np.ascontiguousarray(np.concatenate(parts))


def make_mels(cfg: VocosConfig, frames: int, seed: int = 0) -> np.ndarray:
    """Log-mel frames float32 [frames][n_mels], N(-5, 2) from PCG64(seed) (the
    range of natural-log mel magnitudes)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return np.ascontiguousarray(rng.normal(-5.0, 2.0, (frames, cfg.n_mels)), dtype=np.float32)
