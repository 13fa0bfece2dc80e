"""GPU: wave_step_static, the entry point for callers that cannot allocate
device memory (it runs the step with the library's fixed scratch array
instead of a workspace from cudaMalloc), against wave_step on the same
inputs, for two frames in a row: the same kernel on the same plan, so y and
every appended code and scale are the same bits, and y is within the stated
bound of the oracle.

Collected last on purpose: if it fails, a run that stops at the first
failure has already run every other test.  It must pass both alone in a
fresh process and after the other tests (the scratch keeps the previous
call's contents)."""
import numpy as np
import pytest
import torch

import frame_step_decode_gb300 as fsd
import synth
from gpu_case import DeviceCase, oracle_reference, y_close

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("w", [synth.TINY, synth.MID])
def test_static_scratch_step_matches_wave_step_on_two_frames(w):
    ref = DeviceCase(w)
    new = DeviceCase(w)
    wave = fsd.Wave(ref.cfg, ref.S_max, w.T_max)
    try:
        for frame in range(2):
            if frame == 1:  # the next frame: every session one slot further, fed its own output
                nxt = torch.clamp(ref.pos + 1, max=w.T_max - 1)
                for c in (ref, new):
                    c.pos.copy_(nxt)
                    c.x.copy_(c.y)
                ref.pos_h = nxt.cpu().numpy()
            ref.step(wave)
            assert wave.status() == fsd.WAVE_OK
            rc = fsd.step_static(new.cfg, new.S_max, w.T_max, new.S, new.weights, new.kv, new.sc,
                                 new.pos, new.x, new.y)
            assert rc == fsd.WAVE_OK, fsd.strerror(rc)
            assert np.array_equal(new.y_bits(), ref.y_bits()), f"frame {frame}: y differs from wave_step"
            assert torch.equal(new.kv, ref.kv), f"frame {frame}: history differs from wave_step"
            assert torch.equal(torch.nan_to_num(new.sc, nan=-7.0), torch.nan_to_num(ref.sc, nan=-7.0))
        # and the first frame against the oracle, element-wise
        first = DeviceCase(w)
        rc = fsd.step_static(first.cfg, first.S_max, w.T_max, first.S, first.weights, first.kv, first.sc,
                             first.pos, first.x, first.y)
        assert rc == fsd.WAVE_OK
        _, y_exact, _, _, _ = oracle_reference(w, range(first.S), first.pos_h, first.x_h)
        ok, worst = y_close(first.y_bits(), y_exact)
        assert ok, f"worst error / bound {worst:.3f}"
    finally:
        wave.close()


def test_static_scratch_rejects_a_shape_that_does_not_fit():
    # A one-layer model whose history is long enough that the RoPE table
    # alone (T_max x D/2 x 8 bytes = 51 MB) exceeds the fixed 32 MiB scratch.
    # Every buffer is real and sized for the shape, and the position is 0, so
    # even a wrongly accepted call would stay inside its buffers.
    cfg = fsd.WaveConfig(1, 64, 1, 64, 64, 1e-5, 1e4)
    T = 200_000
    dev = "cuda"
    weights = torch.zeros(fsd.packed_weights_bytes(cfg) // 2, dtype=torch.bfloat16, device=dev)
    kv = torch.zeros((1, 2, 1, 1, T, 64), dtype=torch.uint8, device=dev)
    sc = torch.zeros((1, 2, 1, 1, T), dtype=torch.float32, device=dev)
    pos = torch.zeros(1, dtype=torch.int32, device=dev)
    x = torch.zeros((1, 64), dtype=torch.bfloat16, device=dev)
    y = torch.zeros_like(x)
    rc = fsd.step_static(cfg, 1, T, 1, weights, kv, sc, pos, x, y)
    assert rc == fsd.WAVE_EINVAL
    # the same buffers at a T_max that fits run the step
    rc = fsd.step_static(cfg, 1, 4096, 1, weights, kv, sc, pos, x, y)
    assert rc == fsd.WAVE_OK
