"""GPU parity at the full 7B-class size, in the launch configuration bench.py
times: 32 layers, d = 4096, 32 x 128 heads, F = 11008, S = 80 sessions,
T_max = 3000, inputs drawn on the device.  The oracle recomputes a sample of
the sessions one by one (sessions are independent).

At this depth and width the step is ill-conditioned: the bf16 rounding of
activations turns any arithmetic difference (fp32 against fp64) into
occasional one-ulp flips that cascade through the layers.  The oracle itself
moves its output by ~1.6% (normwise) when one element of x is nudged by one
bf16 ulp.  So the element-wise 1e-3 + 2e-2|y| bound, met on the shallow
shapes of test_gpu_step.py, is replaced here by: (a) every appended FP8 code
and scale bit-exact against the oracle's quantiser on the GPU's own
pre-quantisation rows, (b) layer-0 K/V rows (before any cascade) within
1e-4 of the oracle's, and (c) y within three times the oracle's own
one-ulp sensitivity, normwise, and never above 5e-2.  And (d) every phase of
every one of the 32 layers, for the first sessions, against the oracle's
functions applied to the GPU's own inputs to that phase: no cascade reaches a
phase checked on its own inputs, so each is held to the stated element-wise
bound and to a tight bound that a 1% error anywhere fails.
"""
import numpy as np
import pytest
import torch

import frame_step_decode_gb300 as fsd
import oracle
import synth
import phase_check
from gpu_case import DeviceCase, codes_vs_oracle, dump_acts, y_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def big():
    w = synth.SEVEN_B
    free = torch.cuda.mem_get_info()[0]
    if free < 100e9:
        pytest.skip("needs ~90 GB of device memory")
    case = DeviceCase(w, poison=False, device_gen=True, keep_rowmajor=True)
    # the device generator against the host one, then the row-major blob goes
    W = synth.weights_host(w)
    case.gen_ok = torch.equal(case.weights_rm.view(torch.int16), torch.from_numpy(W.view(np.int16)).to("cuda"))
    del W
    case.weights_rm = None
    torch.cuda.empty_cache()
    wave = fsd.Wave(case.cfg, case.S_max, w.T_max)
    yield case, wave
    wave.close()
    del case
    torch.cuda.empty_cache()


@pytest.fixture(scope="module")
def W7():
    return synth.weights_host(synth.SEVEN_B)


def _sample(pos):
    order = np.argsort(pos)
    return sorted({int(order[0]), int(order[-1]), int(order[len(order) // 2]), 17})


def test_device_generator_matches_host_generator(big):
    case, _ = big
    assert case.gen_ok


def test_full_size_step_matches_oracle_on_sampled_sessions(big, W7):
    case, wave = big
    w = case.w
    sess = _sample(case.pos_h)
    L, H, D = w.n_layers, w.n_heads, w.head_dim
    # the oracle's own history for the sampled sessions equals the GPU's, bit for bit
    kv_o, sc_o = oracle.prefill_history(w, sess, case.pos_h[sess], poison=False)
    for j, s in enumerate(sess):
        P = int(case.pos_h[s])
        g_codes = case.kv[:, :, s, :, :P].cpu().numpy()
        g_sc = case.sc[:, :, s, :, :P].cpu().numpy()
        assert np.array_equal(g_codes, kv_o[:, :, j, :, :P])
        assert np.array_equal(g_sc.view(np.uint32), sc_o[:, :, j, :, :P].view(np.uint32))
    dump = torch.full((L, 2, case.S_max, H, D), float("nan"), device="cuda")
    wave.debug_dump_kv(dump)
    try:
        case.step(wave)
        assert wave.status() == fsd.WAVE_OK
    finally:
        wave.debug_dump_kv(None)
    y = case.y_bits()
    W = W7
    kv_in, sc_in = kv_o.copy(), sc_o.copy()
    _, y_exact, kv_new = oracle.step(w, W, kv_o, sc_o, case.pos_h[sess], case.x_h[sess], want_kv_new=True)
    # the oracle's own sensitivity: one element of x moved by one bf16 ulp
    x_p = case.x_h[sess].copy()
    x_p[:, 5] += 1
    _, y_pert, _ = oracle.step(w, W, kv_in, sc_in, case.pos_h[sess], x_p)
    yg = synth.bf16_bits_to_f32(y[sess]).astype(np.float64)
    scale = np.max(np.abs(y_exact), axis=1)
    gpu_err = np.max(np.abs(yg - y_exact), axis=1) / scale
    floor = np.max(np.abs(y_pert - y_exact), axis=1) / scale
    print("normwise y error per sampled session:", gpu_err, "oracle one-ulp sensitivity:", floor)
    assert np.all(gpu_err <= np.maximum(3 * floor, 1e-3)) and np.all(gpu_err <= 5e-2)
    dump_h = dump.cpu().numpy()
    n_diff = 0
    for j, s in enumerate(sess):
        P = int(case.pos_h[s])
        pre = np.ascontiguousarray(dump_h[:, :, s])          # [L][2][H][D]
        codes, scales = oracle.quantize_rows(pre)
        assert np.array_equal(case.kv[:, :, s, :, P].cpu().numpy(), codes)
        # end to end against the oracle's own codes (written into kv_o by its step)
        n_diff += codes_vs_oracle(codes, pre, kv_o[:, :, j, :, P], sc_o[:, :, j, :, P], kv_new[:, :, j])
        assert np.array_equal(case.sc[:, :, s, :, P].cpu().numpy().view(np.uint32), scales.view(np.uint32))
        err = np.max(np.abs(pre.astype(np.float64) - kv_new[:, :, j]), axis=-1)
        ref = np.max(np.abs(kv_new[:, :, j].astype(np.float64)), axis=-1)
        assert np.all(err[0] <= 1e-4 * ref[0] + 1e-6)   # layer 0: before any cascade
        assert np.all(err <= 5e-2 * ref + 1e-6)
    print(f"{n_diff} of {len(sess) * L * 2 * H * D} appended codes differ from the oracle's own "
          "(each within the two paths' measured difference of the oracle's value)")


def test_full_size_every_phase_of_every_layer_matches_oracle(big, W7):
    case, wave = big
    w = case.w
    n = 4
    case.step(wave)
    assert wave.status() == fsd.WAVE_OK
    y_plain = case.y_bits()
    recs = dump_acts(wave, n, 1, lambda: case.step(wave))
    y = case.y_bits()
    assert np.array_equal(y, y_plain), "the dump's kernel must give the usual kernel's bits"
    worst = {}
    for s in range(n):
        P = int(case.pos_h[s])
        kv = case.kv[:, :, s, :, :P + 1].cpu().numpy()
        sc = case.sc[:, :, s, :, :P + 1].cpu().numpy()
        phase_check.check_decoder_frame(w, W7, recs[0, :, s], P, kv, sc, case.x_h[s], y[s], worst)
    print("positions", case.pos_h[:n], {k: round(v, 3) for k, v in worst.items()})
    assert all(v <= 1.0 for v in worst.values()), worst
