"""GPU: wave_step_static, the entry point for callers that cannot allocate
device memory (it runs the step with the library's fixed scratch array
instead of a workspace from cudaMalloc), against wave_step on the same
inputs, for two frames in a row.

Collected last on purpose: if it fails, a run that stops at the first
failure has already run every other test.  It must pass both alone in a
fresh process and after the other tests (the scratch keeps the previous
call's contents)."""
import numpy as np
import pytest
import torch

import frame_step_decode_gb300 as fsd
import synth
from gpu_case import DeviceCase, y_close, bf16_to_f64

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
            ok, worst = y_close(new.y_bits(), bf16_to_f64(ref.y_bits()))
            assert ok, f"frame {frame}: worst error / bound {worst:.3f}"
            # the appended slot agrees too
            P = ref.pos.long()
            idx = torch.arange(ref.S, device="cuda")
            a = ref.kv[:, :, idx, :, P]
            b = new.kv[:, :, idx, :, P]
            assert (a != b).float().mean().item() < 1e-3
    finally:
        wave.close()


def test_static_scratch_rejects_shapes_that_do_not_fit():
    w = synth.SEVEN_B
    case_cfg = fsd.WaveConfig.of(w)
    dummy = torch.zeros(64, dtype=torch.uint8, device="cuda")
    rc = fsd.step_static(case_cfg, 128, 3000, 1, dummy, dummy, dummy.view(torch.float32), dummy,
                         dummy, dummy)
    assert rc == fsd.WAVE_EINVAL
