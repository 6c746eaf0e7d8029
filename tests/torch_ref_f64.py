"""Second opinion on the oracle: the decoder written as a float64 PyTorch-CPU
composition of library routines (conv1d, conv_transpose1d, masked softmax).

Test infrastructure only.  It is written independently of the C oracle: it
works in PyTorch's [channel][time] layout, realises causality with explicit
left padding and right trimming, and builds attention from a dense band mask,
where the oracle runs plain loops over a carried history.  The stage list
follows vllm-omni "Edge TTS design" section 1.3; the transposed-convolution
form is the library's own conv_transpose1d; Snake is x + sin^2(alpha x)/alpha.
"""
from __future__ import annotations

import math

import numpy as np
import torch
import torch.nn.functional as F


def _t(w, dtype):
    return torch.from_numpy(np.asarray(w)).to(dtype)


def gather_sum(cfg, W, codes):
    """Sum of the Q codebook rows, fp32, q ascending (kept in fp32 on purpose:
    the GPU path must reproduce these bits)."""
    codes = torch.from_numpy(np.asarray(codes)).long()
    e = None
    for q in range(cfg.Q):
        row = torch.from_numpy(W[f"cb.{q}"])[codes[q]]          # [T][E] fp32
        e = row.clone() if e is None else e + row
    return e


def _conv1d(x, w, b, dilation):
    return F.conv1d(x, w, b, dilation=dilation)


def _linear(x, w):
    return x @ w.t()


def _conv_t(x, w, b, stride):
    return F.conv_transpose1d(x, w, b, stride=stride)


def causal_conv(x, w, b, dilation=1):
    """x [C][T]; left pad (k-1)*d zeros, valid correlation."""
    k = w.shape[-1]
    xp = F.pad(x[None], ((k - 1) * dilation, 0))
    return _conv1d(xp, w, b, dilation)[0]


def causal_conv_t(x, w, b, stride):
    """x [C][T] -> [C'][T*stride]: the library transposed conv with the
    right (k - stride) outputs trimmed."""
    T = x.shape[-1]
    y = _conv_t(x[None], w, b, stride)[0]
    return y[:, : T * stride]


def snake(x, alpha):
    a = alpha[:, None]
    return x + torch.sin(a * x) ** 2 / a


def rms_norm(h, g, eps):
    return h * torch.rsqrt((h * h).mean(-1, keepdim=True) + eps) * g


def sliding_attention(q, k, v, heads, window):
    """q,k,v [T][d]; query t sees keys j with t - window < j <= t."""
    T, d = q.shape
    dh = d // heads
    idx = torch.arange(T)
    band = (idx[None, :] <= idx[:, None]) & (idx[None, :] > idx[:, None] - window)
    out = torch.empty_like(q)
    for h in range(heads):
        sl = slice(h * dh, (h + 1) * dh)
        s = (q[:, sl] @ k[:, sl].t()) / math.sqrt(dh)
        s = s.masked_fill(~band, float("-inf"))
        out[:, sl] = torch.softmax(s, dim=-1) @ v[:, sl]
    return out


def decode(cfg, W, codes, dtype=torch.float64, taps=None):
    """Full-sequence decode from an empty state: codes [Q][T] -> audio [T*spf].

    taps, if a dict, receives intermediate tensors by stage name."""
    e = gather_sum(cfg, W, codes).to(dtype).t()               # [E][T]
    h = causal_conv(e, _t(W["pre.w"], dtype), _t(W["pre.b"], dtype)).t()   # [T][d]
    if taps is not None:
        taps["pre"] = h
    return _body(cfg, W, h, dtype, taps)


def decode_latents(cfg, W, latents, dtype=torch.float64, taps=None):
    """Latent-input variant, full sequence from an empty state: latents [T][L]
    -> audio [T*spf].  Denormalise, project 1x1, then the library's grouped
    (depthwise) conv_transpose1d with the right k - s outputs trimmed."""
    x = _t(latents, dtype)
    z = x * _t(W["lat.sigma"], dtype) + _t(W["lat.mu"], dtype)
    p = _linear(z, _t(W["lat.proj"], dtype))                  # [T][d]
    T, s = p.shape[0], cfg.tf_up
    y = F.conv_transpose1d(p.t()[None], _t(W["lat.up.w"], dtype), _t(W["lat.up.b"], dtype), stride=s,
                           groups=cfg.d)[0]
    h = y[:, : T * s].t()                                       # [T s][d]
    if taps is not None:
        taps["front"] = h
    return _body(cfg, W, h, dtype, taps)


def _body(cfg, W, h, dtype, taps):
    for l in range(cfg.layers):
        p = f"tf.{l}."
        u = rms_norm(h, _t(W[p + "n1"], dtype), cfg.rms_eps)
        q = _linear(u, _t(W[p + "wq"], dtype))
        k = _linear(u, _t(W[p + "wk"], dtype))
        v = _linear(u, _t(W[p + "wv"], dtype))
        h = h + _linear(sliding_attention(q, k, v, cfg.heads, cfg.window), _t(W[p + "wo"], dtype))
        u = rms_norm(h, _t(W[p + "n2"], dtype), cfg.rms_eps)
        h = h + _linear(F.gelu(_linear(u, _t(W[p + "w1"], dtype))), _t(W[p + "w2"], dtype))
    h = rms_norm(h, _t(W["tf.norm"], dtype), cfg.rms_eps)
    if taps is not None:
        taps["transformer"] = h
    x = h.t()                                                  # [d][T]
    for u in range(len(cfg.up_channels)):
        x = causal_conv_t(x, _t(W[f"up.{u}.w"], dtype), _t(W[f"up.{u}.b"], dtype), cfg.up_s)
    if taps is not None:
        taps["latent_up"] = x
    for s, stride in enumerate(cfg.strides):
        p = f"st.{s}."
        x = snake(x, _t(W[p + "alpha"], dtype))
        x = causal_conv_t(x, _t(W[p + "w"], dtype), _t(W[p + "b"], dtype), stride)
        branches = []
        for j, _ in enumerate(cfg.rb_kernels):
            r = x
            for i, dil in enumerate(cfg.dilations):
                q = f"{p}rb.{j}.{i}."
                r = r + causal_conv(snake(r, _t(W[q + "alpha"], dtype)),
                                    _t(W[q + "w"], dtype), _t(W[q + "b"], dtype), dil)
            branches.append(r)
        if len(branches) == 1:
            x = branches[0]
        else:
            acc = branches[0]
            for r in branches[1:]:
                acc = acc + r
            x = acc / len(branches)
        if taps is not None:
            taps[f"stage{s}"] = x
    y = causal_conv(snake(x, _t(W["out.alpha"], dtype)), _t(W["out.w"], dtype), _t(W["out.b"], dtype))
    if taps is not None:
        taps["pre_tanh"] = y[0]
    return torch.tanh(y[0])
