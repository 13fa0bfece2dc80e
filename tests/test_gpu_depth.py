"""GPU parity of the inner depth loop (wave_depth) against the oracle: the
6-layer d=1024 (16 x 64 heads, SwiGLU 2816) model, S = 80 sessions, 8
dependent steps per frame over an 8-slot depth cache, x_k = bf16(W_p y_{k-1}).

The oracle recomputes a sample of the sessions (they are independent).  At
this shape one step is already ill-conditioned in the way the 7B-class step
is: the oracle's own output moves by 1.2-1.9% (normwise) when one element of
x0 is nudged by one bf16 ulp, so the element-wise 1e-3 + 2e-2|y| bound is
replaced, for every step, by: y within three times the oracle's own
one-ulp response, normwise, and never above 5e-2.  Later steps also feed
one step's bf16 output into the next through W_p.  Every depth-cache slot
the loop writes is checked to be written, and a rerun to give the same bits.
And every phase of every layer of all 8 steps (with the projection between
steps) is held to the stated element-wise bound and a tight one against the
oracle's functions applied to the GPU's own inputs to that phase."""
import numpy as np
import pytest
import torch

import frame_step_decode_gb300 as fsd
import oracle
import synth
import phase_check
from gpu_case import bf16_to_f64, dump_acts

pytestmark = pytest.mark.gpu

W = synth.DEPTH
STEPS = W.extra["depth_steps"]
SAMPLE = [0, 17, 40, 79]
PHASE_SESSIONS = range(6)   # the activation dump records sessions 0..5


@pytest.fixture(scope="module")
def run():
    w = W
    S, d = w.S, w.d_model
    L, H, T, D = w.n_layers, w.n_heads, w.T_max, w.head_dim
    Wh = synth.weights_host(w)
    wp_h = synth.proj_host(w)
    x0_h = synth.x_bf16(w, S)
    dev = "cuda"
    weights = fsd.pack_weights(fsd.WaveConfig.of(w), torch.from_numpy(Wh.view(np.int16)).to(dev).view(torch.bfloat16))
    wp = torch.from_numpy(wp_h.view(np.int16)).to(dev).view(torch.bfloat16)
    x0 = torch.from_numpy(x0_h.view(np.int16)).to(dev).view(torch.bfloat16)
    kv = torch.full((L, 2, S, H, T, D), 0x7F, dtype=torch.uint8, device=dev)
    sc = torch.full((L, 2, S, H, T), float("nan"), dtype=torch.float32, device=dev)
    xs = torch.zeros((STEPS, S, d), dtype=torch.bfloat16, device=dev)
    y = torch.zeros((STEPS, S, d), dtype=torch.bfloat16, device=dev)
    wave = fsd.Wave(fsd.WaveConfig.of(w), S, T)
    try:
        wave.depth(S, STEPS, weights, wp, kv, sc, x0, xs, y)
        assert wave.status() == fsd.WAVE_OK
        # a second call over the same (now filled) depth cache gives the same bits
        y2 = torch.zeros_like(y)
        wave.depth(S, STEPS, weights, wp, kv, sc, x0, xs, y2)
        assert wave.status() == fsd.WAVE_OK
        same = torch.equal(y.view(torch.int16), y2.view(torch.int16))
        # once more with the activation dump on (its kernel gives the same bits)
        y3 = torch.zeros_like(y)
        recs = dump_acts(wave, len(PHASE_SESSIONS), STEPS,
                         lambda: wave.depth(S, STEPS, weights, wp, kv, sc, x0, xs, y3))
        same = same and torch.equal(y.view(torch.int16), y3.view(torch.int16))
    finally:
        wave.close()
    out = dict(Wh=Wh, wp=wp_h, x0=x0_h, same=same, recs=recs,
               y=y.view(torch.int16).cpu().numpy().view(np.uint16),
               xs=xs.view(torch.int16).cpu().numpy().view(np.uint16),
               kv=kv.cpu().numpy(), sc=sc.cpu().numpy())
    return out


def test_every_depth_slot_written_and_rerun_identical(run):
    assert run["same"]
    assert not np.any(run["kv"][:, :, :, :, :STEPS] == 0x7F)   # 0x7F (NaN) is never a quantiser output
    assert np.all(np.isfinite(run["sc"][:, :, :, :, :STEPS]))


def test_depth_loop_matches_oracle_on_sampled_sessions(run):
    w = W
    ys, ye, xs = oracle.depth_loop(w, run["Wh"], run["wp"], run["x0"][SAMPLE], STEPS)
    x_p = run["x0"][SAMPLE].copy()
    x_p[:, 3] += 1                                   # one bf16 ulp in one element
    _, ye_p, _ = oracle.depth_loop(w, run["Wh"], run["wp"], x_p, STEPS)
    yg = run["y"][:, SAMPLE]
    assert np.array_equal(run["xs"][0][SAMPLE], run["x0"][SAMPLE])
    for k in range(STEPS):
        scale = np.max(np.abs(ye[k]), axis=1)
        err = np.max(np.abs(bf16_to_f64(yg[k]) - ye[k]), axis=1) / scale
        floor = np.max(np.abs(ye_p[k] - ye[k]), axis=1) / scale
        print(f"step {k}: normwise error {err}, oracle one-ulp response {floor}")
        assert np.all(err <= np.maximum(3 * floor, 1e-2)) and np.all(err <= 5e-2)


def test_depth_loop_on_a_ragged_prefix_batch():
    # S = 19 sessions of an S_max = 80 handle; sessions are independent, so
    # each equals its own run in the full batch bit for bit
    w = W
    S, d = 19, w.d_model
    L, H, T, D = w.n_layers, w.n_heads, w.T_max, w.head_dim
    Wh = synth.weights_host(w)
    dev = "cuda"
    weights = fsd.pack_weights(fsd.WaveConfig.of(w), torch.from_numpy(Wh.view(np.int16)).to(dev).view(torch.bfloat16))
    wp = torch.from_numpy(synth.proj_host(w).view(np.int16)).to(dev).view(torch.bfloat16)
    x0 = torch.from_numpy(synth.x_bf16(w, w.S).view(np.int16)).to(dev).view(torch.bfloat16)
    outs = []
    for n in (S, w.S):
        kv = torch.full((L, 2, w.S, H, T, D), 0x7F, dtype=torch.uint8, device=dev)
        sc = torch.full((L, 2, w.S, H, T), float("nan"), dtype=torch.float32, device=dev)
        xs = torch.zeros((STEPS, n, d), dtype=torch.bfloat16, device=dev)
        y = torch.zeros((STEPS, n, d), dtype=torch.bfloat16, device=dev)
        wave = fsd.Wave(fsd.WaveConfig.of(w), w.S, T)
        try:
            wave.depth(n, STEPS, weights, wp, kv, sc, x0[:n].contiguous(), xs, y)
            assert wave.status() == fsd.WAVE_OK
        finally:
            wave.close()
        outs.append(y)
    assert torch.equal(outs[0].view(torch.int16), outs[1][:, :S].view(torch.int16))


def test_every_phase_of_every_step_matches_oracle(run):
    w = W
    worst = {}
    for s in PHASE_SESSIONS:
        kv = np.ascontiguousarray(run["kv"][:, :, s])
        sc = np.ascontiguousarray(run["sc"][:, :, s])
        for k in range(STEPS):
            if k > 0:   # x_k = bf16(W_p y_{k-1}) on the GPU's own y_{k-1}
                yk = synth.bf16_bits_to_f32(run["y"][k - 1, s]).astype(np.float64)
                phase_check.note(worst, "proj", synth.bf16_bits_to_f32(run["xs"][k, s]),
                                 oracle.matvec(run["wp"], yk), True)
            phase_check.check_decoder_frame(w, run["Wh"], run["recs"][k, :, s], k, kv, sc, run["xs"][k, s],
                                            run["y"][k, s], worst)
    print({k: round(v, 3) for k, v in worst.items()})
    assert all(v <= 1.0 for v in worst.values()), worst


def test_depth_loop_with_x0_inside_xs():
    # xs may start at x0 (no copy of x0 then): the same bits as with x0 apart
    w = W
    S, d = 24, w.d_model
    L, H, T, D = w.n_layers, w.n_heads, w.T_max, w.head_dim
    dev = "cuda"
    weights = fsd.pack_weights(fsd.WaveConfig.of(w),
                               torch.from_numpy(synth.weights_host(w).view(np.int16)).to(dev).view(torch.bfloat16))
    wp = torch.from_numpy(synth.proj_host(w).view(np.int16)).to(dev).view(torch.bfloat16)
    x0 = torch.from_numpy(synth.x_bf16(w, S).view(np.int16)).to(dev).view(torch.bfloat16)
    outs = []
    wave = fsd.Wave(fsd.WaveConfig.of(w), S, T)
    try:
        for inside in (False, True):
            kv = torch.full((L, 2, S, H, T, D), 0x7F, dtype=torch.uint8, device=dev)
            sc = torch.full((L, 2, S, H, T), float("nan"), dtype=torch.float32, device=dev)
            xs = torch.zeros((STEPS, S, d), dtype=torch.bfloat16, device=dev)
            y = torch.zeros((STEPS, S, d), dtype=torch.bfloat16, device=dev)
            if inside:
                xs[0].copy_(x0)
                wave.depth(S, STEPS, weights, wp, kv, sc, xs[0], xs, y)
            else:
                wave.depth(S, STEPS, weights, wp, kv, sc, x0, xs, y)
            assert wave.status() == fsd.WAVE_OK
            outs.append((y, xs))
    finally:
        wave.close()
    assert torch.equal(outs[0][0].view(torch.int16), outs[1][0].view(torch.int16))
    assert torch.equal(outs[0][1].view(torch.int16), outs[1][1].view(torch.int16))

