"""The allocation-free conv entry point (codec_conv1d_noalloc) against the
ordinary one (codec_state_conv1d), through the C ABI.

codec_conv1d_noalloc exists for callers that may not allocate device memory
when they need the layer (a real-time audio thread, an application whose GPU
memory belongs to its own pool allocator, an embedding that only receives
input and output buffers); it keeps its scratch in one fixed device array of
the library.  Two calls in a row with different shapes check that the shared
array carries nothing from one call into the next; the outputs must agree
with the ordinary entry point within the conv tolerance of test_gpu_ops.py.
This file sorts last so that a run stopping at the first failure has already
run every other test; it also passes on its own in a fresh process.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from gpu_helpers import relerr
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
    x = torch.from_numpy((rng.standard_normal((H + T, Cin)) * 2).astype(np.float32)).cuda()
    w = torch.from_numpy((rng.standard_normal((Cout, Cin, k)) / np.sqrt(Cin * k)).astype(np.float32)).cuda()
    b = torch.from_numpy(rng.standard_normal(Cout).astype(np.float32)).cuda()
    a = torch.from_numpy(rng.uniform(0.5, 1.5, Cin).astype(np.float32)).cuda() if snake else None
    return x, w, b, a, dil, T, Cout


def test_no_alloc_matches_allocating_entry_point_twice(state):
    for args in [(1, 11, 5, 192, 192, 300, True), (2, 3, 1, 96, 96, 257, False)]:
        x, w, b, a, dil, T, Cout = _case(*args)
        want = torch.full((T, Cout), float("nan"), device="cuda")
        got = torch.full((T, Cout), float("nan"), device="cuda")
        state.conv1d(x, w, want, bias=b, alpha=a, dilation=dil)
        C.conv1d_noalloc(x, w, got, bias=b, alpha=a, dilation=dil)
        torch.cuda.synchronize()
        g, r = got.cpu().numpy(), want.cpu().numpy()
        assert np.isfinite(g).all()
        assert relerr(g, r) <= REL, (args, relerr(g, r))


def test_no_alloc_rejects_sizes_beyond_its_array():
    x = torch.zeros(16, 64, device="cuda")
    w = torch.zeros(8192, 64, 11, device="cuda")          # 5.8 M weights > 4,194,304
    y = torch.zeros(16, 8192, device="cuda")
    with pytest.raises(C.CodecError) as e:
        C.conv1d_noalloc(x[:6], w, y[:1])
    assert e.value.status == 5                              # CODEC_ERR_CAPACITY
