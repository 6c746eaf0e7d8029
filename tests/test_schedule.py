"""Chunk schedules of the streaming orchestrator (codec_chunk_frames, host
logic of the C ABI; no GPU): the measured default 1 then 25, the page's
example ramp 4, 4, 8, 16, 25, and the adaptive reading (each chunk as long as
the audio already delivered, capped at the steady size), per the vllm-omni
"Edge TTS design" page, section 2.2 "Orchestrator loop"."""
from __future__ import annotations

import pytest

from streaming_tts_vocoder_gb300 import build as B
from streaming_tts_vocoder_gb300 import codec as C


@pytest.fixture(scope="module", autouse=True)
def lib():
    B.build()
    return C._lib()


def test_fixed_one_then_25():
    s = C.chunk_schedule(C.SCHEDULE_FIXED, first=1, steady=25)
    assert C.schedule_chunks(s, 100) == [1, 25, 25, 25, 24]


def test_ramp_of_the_page():
    s = C.chunk_schedule(C.SCHEDULE_RAMP, steady=25, ramp=(4, 4, 8, 16))
    assert C.schedule_chunks(s, 120) == [4, 4, 8, 16, 25, 25, 25, 13]


def test_adaptive_doubles_to_the_steady_size():
    s4 = C.chunk_schedule(C.SCHEDULE_ADAPTIVE, first=4, steady=25)
    assert C.schedule_chunks(s4, 107) == [4, 4, 8, 16, 25, 25, 25]
    s1 = C.chunk_schedule(C.SCHEDULE_ADAPTIVE, first=1, steady=25)
    assert C.schedule_chunks(s1, 57) == [1, 1, 2, 4, 8, 16, 25]
    # a chunk never exceeds the audio delivered before it (in frames)
    done = 0
    for i in range(12):
        n = C.chunk_frames(s1, i, done)
        if i:
            assert n <= max(1, done)
        done += n


def test_adaptive_chunk_never_outlasts_the_queued_audio():
    """A producer making a frame every half frame period (twice real time)
    and a decoder taking no time: playback started on the first chunk never
    stalls under the adaptive schedule, while 1 then 25 stalls (the cliff the
    page describes)."""
    def stalls(chunks, period=0.5):
        arrived, queued_until, out = 0, None, []
        for n in chunks:
            arrived += n
            t = arrived * period                      # in frame periods
            if queued_until is None:
                queued_until = t + n
            else:
                out.append(max(0.0, t - queued_until))
                queued_until = max(queued_until, t) + n
        return out

    ada = C.schedule_chunks(C.chunk_schedule(C.SCHEDULE_ADAPTIVE, first=1, steady=25), 250)
    assert max(stalls(ada)) == 0.0
    fixed = C.schedule_chunks(C.chunk_schedule(C.SCHEDULE_FIXED, first=1, steady=25), 250)
    assert max(stalls(fixed)) > 0.0


def test_invalid_schedules_give_zero():
    assert C.chunk_frames(C.chunk_schedule(7), 0, 0) == 0
    assert C.chunk_frames(C.chunk_schedule(C.SCHEDULE_FIXED, first=0), 0, 0) == 0
    assert C.chunk_frames(C.chunk_schedule(C.SCHEDULE_FIXED), -1, 0) == 0
