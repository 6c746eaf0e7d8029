"""GPU parity of the tensor-core conv kernel on its own (codec_state_conv1d)
against the oracle's causal conv, over tap counts, dilations, channel widths
that select each N-tiling of the kernel (two M-tiles sharing N <= 128, one
M-tile with N up to 256, several N-tiles), ragged row counts and Snake on the
input.

Tolerance: the operands are split into fp16 hi + lo (about 2^-22 relative
each) and the products are summed in fp32 in chunks of 8 MMA k-steps, so one
conv lands within a few 1e-7 of the float64-accumulated oracle; 2e-5
relative L2 leaves two orders of margin while still catching a dropped cross
term (about 2^-11 = 5e-4)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from gpu_helpers import relerr
from oracle import oracle as O
from streaming_tts_vocoder_gb300 import codec as C
from streaming_tts_vocoder_gb300.synthetic import make_weights, pack_blob, qwen3_config

pytestmark = pytest.mark.gpu
REL = 2e-5


@pytest.fixture(scope="module")
def state():
    cfg = qwen3_config()
    cod = C.Codec(cfg, pack_blob(cfg, make_weights(cfg, 0)), max_streams=1, max_chunk_frames=1,
                  precision=C.PRECISION_FP16X3)
    return cod.state()


CASES = [
    # k, dil, Cin, Cout, T, snake
    (3, 1, 96, 96, 257, True),      # N <= 128: two M-tiles share the N-tile; ragged last tile
    (11, 5, 192, 192, 300, True),   # one M-tile, N = 192
    (7, 3, 256, 160, 129, False),   # N = 160: one 160-wide tile, second epilogue group on 32 columns
    (1, 1, 512, 1024, 64, False),   # linear: four 256-wide N-tiles
    (2, 1, 64, 288, 200, True),     # 288 = 3 x 96
]


@pytest.mark.parametrize("k,dil,Cin,Cout,T,snake", CASES)
def test_tc_conv_matches_oracle(state, k, dil, Cin, Cout, T, snake):
    rng = np.random.default_rng(k * 1000 + Cout)
    H = (k - 1) * dil
    x = (rng.standard_normal((H + T, Cin)) * 2).astype(np.float32)
    w = (rng.standard_normal((Cout, Cin, k)) / np.sqrt(Cin * k)).astype(np.float32)
    b = rng.standard_normal(Cout).astype(np.float32)
    alpha = rng.uniform(0.5, 1.5, Cin).astype(np.float32) if snake else None
    y = torch.full((T, Cout), float("nan"), device="cuda")
    to = lambda a: None if a is None else torch.from_numpy(a).cuda()
    state.conv1d(to(x), to(w), y, bias=to(b), alpha=to(alpha), dilation=dil)
    torch.cuda.synchronize()
    got = y.cpu().numpy()
    want = O.causal_conv(x, w, b, dil, alpha=alpha)
    assert np.isfinite(got).all()
    assert relerr(got, want) < REL, relerr(got, want)


def test_tc_conv_argument_errors(state):
    x = torch.zeros(10, 64, device="cuda")
    y = torch.zeros(8, 64, device="cuda")
    with pytest.raises(C.CodecError) as e:
        state.conv1d(x[:, :48].contiguous(), torch.zeros(64, 48, 3, device="cuda"), y)   # Cin % 32 != 0
    assert e.value.status == 4
    big = torch.zeros(200000, 64, device="cuda")
    with pytest.raises(C.CodecError) as e:
        state.conv1d(big, torch.zeros(64, 64, 1, device="cuda"), torch.zeros(200000, 64, device="cuda"))
    assert e.value.status == 5
