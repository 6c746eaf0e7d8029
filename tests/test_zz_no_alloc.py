"""The allocation-free conv entry point (codec_conv1d_noalloc) against the
ordinary one (codec_state_conv1d) and the oracle, through the C ABI.

codec_conv1d_noalloc exists for callers that may not allocate device memory
when they need the layer: a real-time audio thread (cudaMalloc can block for
an unbounded time and synchronises the device), an application whose GPU
memory belongs to its own pool allocator, an embedding that only receives
input and output buffers.  It keeps its scratch in one fixed device array of
the library.  Both entry points run the same kernels on the same inputs with
the same launch shapes, so their outputs must agree bit for bit; both are
also held to the oracle's causal conv at the tolerance of test_gpu_ops.py.
Two calls in a row with different shapes check that the shared array carries
nothing from one call into the next, and that the timeout flag reads clear
after each.  This file sorts last so that a run stopping at the first failure
has already run every other test; it also passes on its own in a fresh
process.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from gpu_helpers import bits_equal, relerr
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


def _case(seed, k, dil, Cin, Cout, T, snake):
    rng = np.random.default_rng(seed)
    H = (k - 1) * dil
    x = (rng.standard_normal((H + T, Cin)) * 2).astype(np.float32)
    w = (rng.standard_normal((Cout, Cin, k)) / np.sqrt(Cin * k)).astype(np.float32)
    b = rng.standard_normal(Cout).astype(np.float32)
    a = rng.uniform(0.5, 1.5, Cin).astype(np.float32) if snake else None
    return x, w, b, a, dil, T, Cout


def test_no_alloc_matches_allocating_entry_point_twice(state):
    to = lambda a: None if a is None else torch.from_numpy(a).cuda()
    for args in [(1, 11, 5, 192, 192, 300, True), (2, 3, 1, 96, 96, 257, False)]:
        x, w, b, a, dil, T, Cout = _case(*args)
        want = torch.full((T, Cout), float("nan"), device="cuda")
        got = torch.full((T, Cout), float("nan"), device="cuda")
        state.conv1d(to(x), to(w), want, bias=to(b), alpha=to(a), dilation=dil)
        C.conv1d_noalloc(to(x), to(w), got, bias=to(b), alpha=to(a), dilation=dil)
        assert not C.conv1d_noalloc_timed_out()
        torch.cuda.synchronize()
        g, r = got.cpu().numpy(), want.cpu().numpy()
        assert np.isfinite(g).all()
        assert bits_equal(g, r), (args, relerr(g, r))
        ref = O.causal_conv(x, w, b, dil, alpha=a)
        assert relerr(g, ref) <= REL, (args, relerr(g, ref))


def test_no_alloc_rejects_sizes_beyond_its_array():
    # Cout * Cin * k = 8192 * 64 * 11 = 5.8 M weights > 4,194,304; x is [(k-1) + T][Cin]
    x = torch.zeros(11, 64, device="cuda")
    w = torch.zeros(8192, 64, 11, device="cuda")
    y = torch.zeros(1, 8192, device="cuda")
    with pytest.raises(C.CodecError) as e:
        C.conv1d_noalloc(x, w, y)
    assert e.value.status == 5                              # CODEC_ERR_CAPACITY


def test_no_alloc_argument_error_comes_before_capacity():
    # Cin = 48 is not a multiple of 32 (an argument error) and the weights are
    # also beyond the array: the argument error is reported
    x = torch.zeros(11, 48, device="cuda")
    w = torch.zeros(8192, 48, 11, device="cuda")
    y = torch.zeros(1, 8192, device="cuda")
    with pytest.raises(C.CodecError) as e:
        C.conv1d_noalloc(x, w, y)
    assert e.value.status == 4                              # CODEC_ERR_ARG
