"""Replicas: the decoder shards by stream with no exchange between shards, so
two processes, each with its own codec and its own half of the streams, must
give every stream the same bits as one process decoding all of them together
(one GPU here: the two processes' kernels never wait on each other).  Each
process packs its own ragged ticks, so the row tiles, split counts and
batch positions of a stream differ between the two runs."""
from __future__ import annotations

import os
import subprocess
import sys
import tempfile
from pathlib import Path

import numpy as np
import pytest
import torch

from gpu_helpers import bits_equal, decode_batch
from streaming_tts_vocoder_gb300 import codec as C
from streaming_tts_vocoder_gb300.synthetic import make_codes, make_weights, pack_blob, staggered_schedule, tiny_config

pytestmark = pytest.mark.gpu
S, F, CH = 4, 60, 25


def decode_streams(streams):
    """Decode the given streams of the 4-stream staggered workload in one
    codec; returns {stream: audio}."""
    cfg = tiny_config()
    cod = C.Codec(cfg, pack_blob(cfg, make_weights(cfg, 0)), max_streams=S, max_chunk_frames=CH,
                  max_batch_frames=S * CH, precision=C.PRECISION_FP16X3)
    st = cod.state()
    codes = {s: make_codes(cfg, F, 1000 + s) for s in streams}
    out = {s: [] for s in streams}
    for tick in staggered_schedule(S, F, CH):
        entries = [(s, codes[s][:, a:a + n]) for s, a, n in tick if s in codes]
        if not entries:
            continue
        for (s, _), a in zip(entries, decode_batch(st, entries, T_max=CH)):
            out[s].append(a)
    return {s: np.concatenate(v) for s, v in out.items()}


def worker(streams, path):
    torch.cuda.set_device(0)
    res = decode_streams(streams)
    np.savez(path, **{str(s): a for s, a in res.items()})


def test_two_processes_give_the_bits_of_one():
    here = Path(__file__).resolve().parent
    env = dict(os.environ)
    env["PYTHONPATH"] = os.pathsep.join([str(here), str(here.parent), env.get("PYTHONPATH", "")])
    with tempfile.TemporaryDirectory() as tmp:
        procs, paths = [], []
        for rank, streams in enumerate(([0, 2], [1, 3])):
            p = os.path.join(tmp, f"rank{rank}.npz")
            paths.append(p)
            code = f"import test_gpu_replicas as t; t.worker({streams!r}, {p!r})"
            procs.append(subprocess.Popen([sys.executable, "-c", code], env=env))
        for pr in procs:
            assert pr.wait(timeout=600) == 0
        parts = {}
        for p in paths:
            with np.load(p) as z:
                parts.update({int(k): z[k] for k in z.files})
    one = decode_streams(list(range(S)))
    for s in range(S):
        assert bits_equal(parts[s], one[s]), f"stream {s}"
