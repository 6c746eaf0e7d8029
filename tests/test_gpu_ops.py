"""GPU parity of the tensor-core conv kernel on its own (codec_state_conv1d)
against the oracle's causal conv, over tap counts, dilations, channel widths
that select each N-tiling of the kernel (two M-tiles sharing N <= 128, one
M-tile with N up to 256, several N-tiles), ragged row counts and Snake on the
input.

Tolerance: the operands are split into fp16 hi + lo (about 2^-22 relative
each) and the products are summed in fp32 in chunks of 16 MMA k-steps, so one
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


def test_bounded_wait_runs_out_reports_and_recovers(state):
    """Every wait of the tensor-core GEMM is bounded.  With the verification
    switch, each CTA's first epilogue wait targets a barrier nothing arrives
    on, so it gives up after the given polls: the kernel must stop cleanly
    (drain its copies and MMAs, free TMEM), the state must report the timeout,
    and after a reset of all slots the same conv must give its normal bits."""
    rng = np.random.default_rng(5)
    k, dil, Cin, Cout, T = 3, 1, 96, 96, 257
    x = torch.from_numpy((rng.standard_normal(((k - 1) * dil + T, Cin)) * 2).astype(np.float32)).cuda()
    w = torch.from_numpy((rng.standard_normal((Cout, Cin, k)) / np.sqrt(Cin * k)).astype(np.float32)).cuda()
    y0 = torch.full((T, Cout), float("nan"), device="cuda")
    state.conv1d(x, w, y0, dilation=dil)
    state.reset()
    assert state.query(0)[1] == 0
    try:
        state.set_wait_limit(polls=1000, unarrived_wait=True)
        y1 = torch.zeros(T, Cout, device="cuda")
        state.conv1d(x, w, y1, dilation=dil)
        assert state.query(0)[1] & C.STREAM_ERR_KERNEL_TIMEOUT
    finally:
        state.set_wait_limit()
    state.reset()
    assert state.query(0)[1] == 0
    y2 = torch.full((T, Cout), float("nan"), device="cuda")
    state.conv1d(x, w, y2, dilation=dil)
    torch.cuda.synchronize()
    assert np.array_equal(y2.cpu().numpy().view(np.uint32), y0.cpu().numpy().view(np.uint32))
