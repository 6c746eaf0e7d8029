"""Pins of the CPU oracle against what the pages and the mathematics fix.

Every check compares the oracle with something other than itself: a brute
force written out here in float64 loops, a textbook/library routine (torch CPU
float64), a closed form, an invariant, or a number the pages print
(tests/golden/page_facts.json).  The planted-mistake tests at the end show
that the pins notice a plausible slip (a flipped tap order, a dropped history
term, an off-by-one window).
"""
from __future__ import annotations

import json
import math
from pathlib import Path

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import torch_ref_f64 as R
from oracle import oracle as O
from streaming_tts_vocoder_gb300.synthetic import (
    make_codes, make_weights, pack_blob, qwen3_config, tiny_config, weight_manifest)

GOLDEN = json.loads((Path(__file__).parent / "golden" / "page_facts.json").read_text())
rng = np.random.default_rng(1234)


def rnd(*shape, scale=1.0):
    return (rng.standard_normal(shape) * scale).astype(np.float32)


def relerr(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


# --------------------------------------------------------------- RVQ sum --

def test_rvq_sum_bit_exact_sequential_fp32():
    Q, V, E, T = 5, 37, 24, 9
    cb = rnd(Q, V, E)
    codes = rng.integers(0, V, size=(Q, T)).astype(np.int32)
    e, err = O.rvq_sum(cb, codes)
    assert err == 0
    want = np.zeros((T, E), np.float32)
    for t in range(T):
        acc = np.zeros(E, np.float32)
        for q in range(Q):
            acc = (acc + cb[q, codes[q, t]]).astype(np.float32)
        want[t] = acc
    assert np.array_equal(e.view(np.uint32), want.view(np.uint32))


def test_rvq_sum_equals_one_hot_matmul():
    Q, V, E, T = 4, 50, 16, 11
    cb = rnd(Q, V, E)
    codes = rng.integers(0, V, size=(Q, T)).astype(np.int32)
    e, _ = O.rvq_sum(cb, codes)
    onehot = np.zeros((Q, T, V))
    for q in range(Q):
        onehot[q, np.arange(T), codes[q]] = 1.0
    want = sum(onehot[q] @ cb[q].astype(np.float64) for q in range(Q))
    assert relerr(e, want) < 1e-6


def test_rvq_single_codebook_is_lookup():
    cb = rnd(1, 30, 8)
    codes = rng.integers(0, 30, size=(1, 7)).astype(np.int32)
    e, _ = O.rvq_sum(cb, codes)
    assert np.array_equal(e, cb[0][codes[0]])


def test_rvq_bad_code_zeroes_frame_and_flags():
    cb = rnd(3, 10, 4)
    codes = np.array([[1, 2, 3], [4, 10, 5], [0, 1, -1]], np.int32)
    e, err = O.rvq_sum(cb, codes)
    assert err == 1
    assert np.all(e[1] == 0) and np.all(e[2] == 0)
    assert np.array_equal(e[0], (cb[0, 1] + cb[1, 4] + cb[2, 0]).astype(np.float32))


# ------------------------------------------------------------ causal conv --

@pytest.mark.parametrize("k,dil", [(3, 1), (7, 3), (11, 5), (1, 1)])
def test_causal_conv_matches_library_conv1d(k, dil):
    Cin, Cout, T = 6, 5, 23
    H = (k - 1) * dil
    x = rnd(H + T, Cin)
    w = rnd(Cout, Cin, k, scale=0.3)
    b = rnd(Cout)
    y = O.causal_conv(x, w, b, dil)
    want = F.conv1d(torch.from_numpy(x.T.astype(np.float64))[None], torch.from_numpy(w).double(),
                    torch.from_numpy(b).double(), dilation=dil)[0].T.numpy()
    assert want.shape == y.shape
    assert relerr(y, want) < 1e-6


def test_causal_conv_brute_force_with_snake_and_residual():
    Cin, Cout, T, k, dil = 4, 3, 10, 3, 2
    H = (k - 1) * dil
    x, w, b, alpha = rnd(H + T, Cin), rnd(Cout, Cin, k), rnd(Cout), rng.uniform(0.5, 1.5, Cin).astype(np.float32)
    res = rnd(T, Cout)
    y = O.causal_conv(x, w, b, dil, alpha=alpha, res=res)
    xd = x.astype(np.float64)
    a = xd + np.sin(alpha * xd) ** 2 / alpha
    want = np.zeros((T, Cout))
    for t in range(T):
        for co in range(Cout):
            s = float(b[co]) + float(res[t, co])
            for j in range(k):
                for ci in range(Cin):
                    s += w[co, ci, j] * a[H + t - (k - 1 - j) * dil, ci]
            want[t, co] = s
    assert relerr(y, want) < 1e-6


def test_causal_conv_impulse_response_is_taps():
    Cin, Cout, k, dil, T = 2, 3, 5, 2, 20
    H = (k - 1) * dil
    w, b = rnd(Cout, Cin, k), np.zeros(3, np.float32)
    x = np.zeros((H + T, Cin), np.float32)
    t0, ci = 4, 1
    x[H + t0, ci] = 1.0
    y = O.causal_conv(x, w, b, dil)
    for t in range(T):
        lag = t - t0
        if lag >= 0 and lag % dil == 0 and lag // dil < k:
            assert np.array_equal(y[t], w[:, ci, k - 1 - lag // dil])
        else:
            assert np.all(y[t] == 0)


def test_causal_conv_is_causal():
    Cin, Cout, k, dil, T = 3, 3, 7, 3, 30
    H = (k - 1) * dil
    x, w, b = rnd(H + T, Cin), rnd(Cout, Cin, k), rnd(Cout)
    y0 = O.causal_conv(x, w, b, dil)
    x2 = x.copy()
    x2[H + 17] += 1.0
    y1 = O.causal_conv(x2, w, b, dil)
    assert np.array_equal(y0[:17], y1[:17])
    assert not np.array_equal(y0[17], y1[17])


# --------------------------------------------------- transposed conv ------

def convt_scatter(x, w, b, s):
    """Textbook ConvTranspose1d by scatter: y[n s + j] += W[:, :, j]^T x[n]."""
    T, Cin = x.shape
    _, Cout, k = w.shape
    y = np.zeros(((T - 1) * s + k, Cout))
    for n in range(T):
        for j in range(k):
            y[n * s + j] += x[n].astype(np.float64) @ w[:, :, j].astype(np.float64)
    return y + b


def convt_zero_insert(x, w, b, s):
    """Insert s-1 zeros between inputs, pad k-1 both sides, correlate with the
    flipped kernel (Core AI Kokoro note: ConvTranspose1d = zero insertion +
    conv with the flipped kernel)."""
    T, Cin = x.shape
    _, Cout, k = w.shape
    z = np.zeros(((T - 1) * s + 1, Cin))
    z[::s] = x
    z = np.concatenate([np.zeros((k - 1, Cin)), z, np.zeros((k - 1, Cin))])
    wf = w[:, :, ::-1].astype(np.float64)          # [Cin][Cout][k] flipped
    L = z.shape[0] - k + 1
    y = np.zeros((L, Cout))
    for m in range(L):
        for j in range(k):
            y[m] += z[m + j] @ wf[:, :, j]
    return y + b


@pytest.mark.parametrize("s", [2, 3, 5, 8])
def test_causal_conv_t_four_forms_agree(s):
    Cin, Cout, T = 5, 4, 7
    x = rnd(T, Cin)
    w = rnd(Cin, Cout, 2 * s)
    b = rnd(Cout)
    hist = np.zeros((1, Cin), np.float32)
    y = O.causal_conv_t(np.concatenate([hist, x]), w, b, s)
    assert y.shape == (T * s, Cout)
    full_scatter = convt_scatter(x, w, b, s)
    full_zero = convt_zero_insert(x, w, b, s)
    lib = F.conv_transpose1d(torch.from_numpy(x.T).double()[None], torch.from_numpy(w).double(),
                             torch.from_numpy(b).double(), stride=s)[0].T.numpy()
    assert np.allclose(full_scatter, full_zero, rtol=0, atol=1e-12)
    assert np.allclose(full_scatter, lib, rtol=0, atol=1e-12)
    # causal form keeps the first T*s outputs; the rest belongs to the next chunk
    assert relerr(y, full_scatter[: T * s]) < 1e-6


def test_causal_conv_t_history_row_carries_tail():
    s, Cin, Cout = 4, 3, 2
    x = rnd(9, Cin)
    w, b = rnd(Cin, Cout, 2 * s), rnd(Cout)
    zero = np.zeros((1, Cin), np.float32)
    full = O.causal_conv_t(np.concatenate([zero, x]), w, b, s)
    first = O.causal_conv_t(np.concatenate([zero, x[:4]]), w, b, s)
    second = O.causal_conv_t(np.concatenate([x[3:4], x[4:]]), w, b, s)
    assert np.array_equal(np.concatenate([first, second]), full)


# ---------------------------------------------------------- attention ------

def swa_brute(q, k, v, heads, window, first=0):
    T, d = q.shape
    Hk = k.shape[0] - T
    dh = d // heads
    out = np.zeros((T, d))
    for t in range(T):
        for h in range(heads):
            sl = slice(h * dh, (h + 1) * dh)
            sc = np.full(k.shape[0], -np.inf)
            for i in range(k.shape[0]):
                if i >= first and Hk + t - window < i <= Hk + t:
                    sc[i] = q[t, sl].astype(np.float64) @ k[i, sl].astype(np.float64) / math.sqrt(dh)
            p = np.exp(sc - sc.max())
            p /= p.sum()
            out[t, sl] = p @ v[:, sl].astype(np.float64)
    return out


@pytest.mark.parametrize("T,Hk,first,window", [(6, 0, 0, 3), (5, 4, 0, 5), (5, 4, 2, 5), (9, 7, 7, 8), (3, 7, 0, 8)])
def test_swa_matches_brute_force_mask(T, Hk, first, window):
    d, heads = 8, 2
    q, k, v = rnd(T, d), rnd(Hk + T, d), rnd(Hk + T, d)
    o = O.swa(q, k, v, heads, window, first)
    assert relerr(o, swa_brute(q, k, v, heads, window, first)) < 1e-6


def test_swa_wide_window_is_causal_attention():
    T, d, heads = 8, 16, 4
    q, k, v = rnd(T, d), rnd(T, d), rnd(T, d)
    o = O.swa(q, k, v, heads, window=8)
    qt, kt, vt = (torch.from_numpy(a).double().view(T, heads, d // heads).transpose(0, 1) for a in (q, k, v))
    want = F.scaled_dot_product_attention(qt, kt, vt, is_causal=True).transpose(0, 1).reshape(T, d).numpy()
    assert relerr(o, want) < 1e-6


def test_swa_window_one_returns_own_value():
    T, d = 5, 8
    q, k, v = rnd(T, d), rnd(T, d), rnd(T, d)
    assert np.array_equal(O.swa(q, k, v, 2, window=1), v)


# ------------------------------------------------------- pointwise ops -----

def test_snake_closed_form_and_special_values():
    alpha = rng.uniform(0.5, 1.5, 6).astype(np.float32)
    x = rnd(50, 6, scale=3.0)
    y = O.snake(x, alpha)
    xd, ad = x.astype(np.float64), alpha.astype(np.float64)
    assert np.allclose(y, xd + np.sin(ad * xd) ** 2 / ad, rtol=2e-7, atol=1e-7)
    assert np.all(y >= x)                                   # sin^2 >= 0
    assert np.all(O.snake(np.zeros((3, 6), np.float32), alpha) == 0)
    kpi = (np.arange(1, 4)[:, None] * np.pi / ad[None, :]).astype(np.float32)
    assert np.allclose(O.snake(kpi, alpha), kpi, rtol=1e-6, atol=1e-6)   # sin(k pi) = 0
    small = np.full((1, 6), 1e-3, np.float32)
    assert np.allclose(O.snake(small, alpha), small + alpha * small ** 2, rtol=1e-6)


def test_rms_norm_and_gelu_textbook():
    x = rnd(7, 12)
    g = rnd(12)
    y = O.rms_norm(x, g, 1e-5)
    xd = x.astype(np.float64)
    want = xd / np.sqrt((xd ** 2).mean(-1, keepdims=True) + 1e-5) * g
    assert relerr(y, want) < 1e-6
    z = rnd(100, scale=3.0)
    gz = O.gelu(z)
    assert np.allclose(gz, [0.5 * v * (1 + math.erf(v / math.sqrt(2))) for v in z.astype(np.float64)], rtol=1e-6, atol=1e-7)
    assert np.allclose(gz, F.gelu(torch.from_numpy(z).double()).numpy(), rtol=1e-6, atol=1e-7)


def test_linear_brute_force():
    x, w, res = rnd(4, 9), rnd(6, 9), rnd(4, 6)
    y = O.linear(x, w, res=res)
    assert relerr(y, x.astype(np.float64) @ w.T.astype(np.float64) + res) < 1e-6


# ------------------------------------------------------------ decoder -----

@pytest.fixture(scope="module")
def tiny():
    cfg = tiny_config()
    W = make_weights(cfg, 0)
    return cfg, W, O.OracleModel(cfg, pack_blob(cfg, W))


def test_page_facts_output_lengths(tiny):
    cfg, W, m = tiny
    assert m.samples_per_frame == GOLDEN["samples_per_frame"]["value"]
    assert qwen3_config().samples_per_frame == GOLDEN["samples_per_frame"]["value"]
    assert GOLDEN["sample_rate_hz"]["value"] / GOLDEN["frame_rate_hz"]["value"] == m.samples_per_frame
    for key in ("first_chunk", "steady_chunk"):
        n = GOLDEN[f"{key}_frames"]["value"]
        a = m.decode_full(make_codes(cfg, n, 3))
        assert a.size == GOLDEN[f"{key}_samples"]["value"]
        assert np.all(np.abs(a) <= 1.0)                     # tanh range (fp32 rounds to 1)


def test_page_facts_qwen3_shape():
    cfg = qwen3_config()
    assert cfg.window == GOLDEN["attention_window_frames"]["value"]
    assert cfg.layers == GOLDEN["transformer_layers"]["value"]
    assert cfg.Q == GOLDEN["codebooks_per_frame"]["value"]
    assert cfg.Q * 2 * GOLDEN["frame_rate_hz"]["value"] == GOLDEN["wire_bytes_per_second"]["value"]
    n = sum(t.size for t in weight_manifest(cfg))
    assert abs(n - GOLDEN["decoder_params_approx"]["value"]) / GOLDEN["decoder_params_approx"]["value"] < 0.05


def test_tiny_decoder_matches_independent_torch_composition(tiny):
    cfg, W, m = tiny
    codes = make_codes(cfg, 8, 0)
    a = m.decode_full(codes)
    ref = R.decode(cfg, W, codes).numpy()
    # fp32 storage between ops vs float64 throughout; the random network
    # amplifies fp32 rounding by ~100x (stage gains of 3-8x each)
    assert relerr(a, ref) < 2e-5
    assert np.abs(a - ref).max() < 1e-3


@pytest.mark.parametrize("splits", [[1] * 12, [2, 3, 1, 6], [5, 7], [12], [4, 4, 4], [3, 9]])
def test_tiny_chunked_equals_full_bit_exact(tiny, splits):
    cfg, W, m = tiny
    codes = make_codes(cfg, 12, 5)
    full = m.decode_full(codes)
    s = m.stream()
    parts, i = [], 0
    for n in splits:
        parts.append(s.decode(codes[:, i:i + n]))
        i += n
    assert s.frames == 12
    assert np.array_equal(np.concatenate(parts).view(np.uint32), full.view(np.uint32))


def test_reset_restores_fresh_stream(tiny):
    cfg, W, m = tiny
    codes = make_codes(cfg, 6, 9)
    s = m.stream()
    s.decode(make_codes(cfg, 4, 1))
    s.reset()
    assert s.frames == 0
    assert np.array_equal(s.decode(codes), m.decode_full(codes))


def test_decoder_is_causal(tiny):
    cfg, W, m = tiny
    codes = make_codes(cfg, 10, 2)
    a = m.decode_full(codes)
    c2 = codes.copy()
    c2[:, 6] = (c2[:, 6] + 1) % cfg.V
    b = m.decode_full(c2)
    spf = m.samples_per_frame
    assert np.array_equal(a[: 6 * spf], b[: 6 * spf])
    assert not np.array_equal(a[6 * spf:], b[6 * spf:])


def test_window_limits_attention_reach():
    """A code change more than `window` frames back reaches later frames only
    through the convolutions' finite history; with a zero-layer check that is
    not observable, so test the window on the transformer output directly."""
    cfg = tiny_config().replace(window=3)
    W = make_weights(cfg, 4)
    codes = make_codes(cfg, 10, 4)
    taps_a, taps_b = {}, {}
    R.decode(cfg, W, codes, taps=taps_a)
    c2 = codes.copy()
    c2[:, 2] = (c2[:, 2] + 1) % cfg.V
    R.decode(cfg, W, c2, taps=taps_b)
    # one layer, window 3, pre-conv k=3: frame 2 reaches frames 2..2+2+2 = 6
    diff = np.abs(taps_a["transformer"].numpy() - taps_b["transformer"].numpy()).max(-1)
    assert np.all(diff[:2] == 0) and np.all(diff[7:] == 0) and diff[6] > 0
    m = O.OracleModel(cfg, pack_blob(cfg, W))
    assert relerr(m.decode_full(codes), R.decode(cfg, W, codes).numpy()) < 2e-5


def test_bad_code_flags_stream(tiny):
    cfg, W, m = tiny
    codes = make_codes(cfg, 4, 0)
    codes[2, 1] = cfg.V
    s = m.stream()
    s.decode(codes)
    assert s.error == 1
    s.decode(make_codes(cfg, 2, 0))
    assert s.error == 1                                       # sticky
    s.reset()
    assert s.error == 0


def test_qwen3_decoder_matches_torch_composition():
    cfg = qwen3_config()
    W = make_weights(cfg, 0)
    codes = make_codes(cfg, 2, 0)
    m = O.OracleModel(cfg, pack_blob(cfg, W))
    a = m.decode_full(codes)
    assert a.size == 2 * 1920
    ref = R.decode(cfg, W, codes).numpy()
    assert relerr(a, ref) < 2e-5
    s = m.stream()
    b = np.concatenate([s.decode(codes[:, :1]), s.decode(codes[:, 1:])])
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


# ------------------------------------------------ planted mistakes ---------

def test_pins_catch_flipped_conv_taps():
    """A conv that reads its taps in reverse order fails the library pin."""
    Cin, Cout, k, T = 3, 2, 3, 8
    x, w, b = rnd(k - 1 + T, Cin), rnd(Cout, Cin, k), rnd(Cout)
    wrong = O.causal_conv(x, w[:, :, ::-1], b)
    want = F.conv1d(torch.from_numpy(x.T).double()[None], torch.from_numpy(w).double(),
                    torch.from_numpy(b).double())[0].T.numpy()
    assert relerr(wrong, want) > 1e-2


def test_pins_catch_dropped_convt_history_term():
    s, Cin, Cout, T = 3, 4, 2, 5
    x, w, b = rnd(T, Cin), rnd(Cin, Cout, 2 * s), rnd(Cout)
    w_drop = w.copy()
    w_drop[:, :, s:] = 0                                     # forget the a[n-1] taps
    wrong = O.causal_conv_t(np.concatenate([np.zeros((1, Cin), np.float32), x]), w_drop, b, s)
    assert relerr(wrong, convt_scatter(x, w, b, s)[: T * s]) > 1e-2


def test_pins_catch_window_off_by_one():
    T, d = 10, 8
    q, k, v = rnd(T, d), rnd(T, d), rnd(T, d)
    wrong = O.swa(q, k, v, 2, window=5)
    assert relerr(wrong, swa_brute(q, k, v, 2, 4)) > 1e-3


def test_oracle_independent_of_thread_count():
    """Every GPU parity claim compares against the oracle: its output must not
    depend on how many OpenMP threads compute it (each output's sum runs in
    one thread, in a fixed order)."""
    cfg = tiny_config()
    blob = pack_blob(cfg, make_weights(cfg, 0))
    codes = make_codes(cfg, 8, 3)
    n0 = O.max_threads()
    try:
        O.set_threads(1)
        one = O.OracleModel(cfg, blob).decode_full(codes)
        O.set_threads(max(2, n0))
        many = O.OracleModel(cfg, blob).decode_full(codes)
    finally:
        O.set_threads(n0)
    assert np.array_equal(one, many)
