"""GPU parity of the hybrid recurrent step (wave_hybrid_step) against the
oracle: a small shape with every part ragged enough to matter (6 layers, two
groups of two selective-state blocks and one attention block, S = 5), and
the full config (48 layers, d 4096, an attention block every sixth layer,
64 state heads x 64 x 128, S = 56, positions in [0, 1500)) on sampled
sessions, where the model is chaotic (see the full-size test).

Even the small shape is ill-conditioned the way the 7B-class step is: the
oracle's own output, for a one-ulp change of one element of x, exceeds the
element-wise 1e-3 + 2e-2|y| bound by up to 2x on near-zero elements.  So y
is held, normwise, to three times the oracle's own one-ulp response (never
above 5e-2), while the parts before any cascade are held tightly: the first
selective-state block's new state within 1e-3 normwise (its input xn can
differ from the oracle's by a bf16 flip, which moves the state by ~1e-4),
and every appended FP8 code and scale bit for bit against the oracle's
quantiser on the GPU's own rows.  Every phase of every block (norm, the
in-projection, the state update, the gated mixer output, QKV, attention, the
out-projections with their residual) is held, on the small shape and on all
48 blocks of the full config, to the stated element-wise bound and to a tight
one against the oracle's functions applied to the GPU's own inputs to that
phase; at full size, where y itself is chaotic, these phase checks (with
the appended codes and the generators' agreement) are the parity."""
import numpy as np
import pytest
import torch

import frame_step_decode_gb300 as fsd
import oracle
import synth
import phase_check
from gpu_case import HybridCase, bf16_to_f64, dump_acts, y_close

pytestmark = pytest.mark.gpu


def _normwise(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-30))


def _y_within_oracle_sensitivity(w, W, sessions, pos, x, y_bits, elements=(3, 5, 100, 200), cap=5e-2):
    """Normwise y error per session against three times the oracle's own
    response to a one-ulp change of one element of x (the largest over a few
    elements), and at most `cap`."""
    kv, sc, st = oracle.hybrid_prefill(w, list(sessions), pos)
    _, y_exact = oracle.hybrid_step(w, W, kv, sc, st, pos, x)
    scale = np.max(np.abs(y_exact), axis=1)
    floor = np.zeros(len(pos))
    for el in elements:
        kv, sc, st = oracle.hybrid_prefill(w, list(sessions), pos)
        x_p = x.copy()
        x_p[:, el % w.d_model] += 1
        _, y_pert = oracle.hybrid_step(w, W, kv, sc, st, pos, x_p)
        floor = np.maximum(floor, np.max(np.abs(y_pert - y_exact), axis=1) / scale)
    err = np.max(np.abs(bf16_to_f64(y_bits) - y_exact), axis=1) / scale
    ok, worst = y_close(y_bits, y_exact)
    print("normwise y error:", err, "oracle one-ulp response:", floor, "element-wise ratio:", worst)
    assert np.all(err <= np.maximum(3 * floor, 1e-3)) and np.all(err <= cap)


def _run(case, sessions):
    w = case.w
    La, H, D = w.n_attn, w.n_heads, w.head_dim
    wave = fsd.HybridWave(case.cfg, case.S_max, w.T_max)
    dump = torch.full((La, 2, case.S_max, H, D), float("nan"), device="cuda")
    try:
        kv0, sc0, st0 = case.kv.clone(), case.sc.clone(), case.state.clone()
        wave.debug_dump_kv(dump)
        case.step(wave)
        assert wave.status() == fsd.WAVE_OK
    finally:
        wave.debug_dump_kv(None)
        wave.close()
    return kv0, sc0, st0, dump.cpu().numpy()


def _check_phases(case, n):
    """Every phase of every block for sessions 0..n-1 (phase_check), on a
    fresh frame from the case's state; the dump's kernel gives the usual
    kernel's bits."""
    w = case.w
    kv0, sc0, st0 = case.kv.clone(), case.sc.clone(), case.state.clone()
    wave = fsd.HybridWave(case.cfg, case.S_max, w.T_max)
    try:
        case.step(wave)
        assert wave.status() == fsd.WAVE_OK
        y_plain = case.y_bits()
        st_plain = case.state.clone()
        case.kv.copy_(kv0)
        case.sc.copy_(sc0)
        case.state.copy_(st0)
        recs = dump_acts(wave, n, 1, lambda: case.step(wave))
    finally:
        wave.close()
    y = case.y_bits()
    assert np.array_equal(y, y_plain), "the dump's kernel must give the usual kernel's bits"
    assert torch.equal(case.state.view(torch.int32), st_plain.view(torch.int32))
    W = getattr(case, "W_h", None)
    W = synth.hybrid_weights_host(w) if W is None else W
    worst = {}
    st_old = st0.cpu().numpy()
    st_new = case.state.cpu().numpy()
    for s in range(n):
        P = int(case.pos_h[s])
        kv = case.kv[:, :, s, :, :P + 1].cpu().numpy()
        sc = case.sc[:, :, s, :, :P + 1].cpu().numpy()
        phase_check.check_hybrid_frame(w, W, recs[0, :, s], P, kv, sc, st_old[:, s], st_new[:, s], case.x_h[s],
                                       y[s], worst)
    print(w.name, {k: round(v, 3) for k, v in worst.items()})
    assert all(v <= 1.0 for v in worst.values()), worst


def test_small_hybrid_every_phase_matches_oracle():
    w = synth.HYBRID_SMALL
    _check_phases(HybridCase(w), w.S)


def test_small_hybrid_step_matches_oracle():
    w = synth.HYBRID_SMALL
    case = HybridCase(w)
    kv0, sc0, st0, dump = _run(case, range(w.S))
    sess = list(range(w.S))
    W = synth.hybrid_weights_host(w)
    _y_within_oracle_sensitivity(w, W, sess, case.pos_h, case.x_h, case.y_bits())
    kv_o, sc_o, st_o = oracle.hybrid_prefill(w, sess, case.pos_h)
    oracle.hybrid_step(w, W, kv_o, sc_o, st_o, case.pos_h, case.x_h)
    st_g = case.state.cpu().numpy()
    assert _normwise(st_g[0], st_o[0]) <= 1e-3                  # first block: a bf16 flip of xn at most
    for lm in range(w.n_mamba):
        assert _normwise(st_g[lm], st_o[lm]) <= 2e-2, lm
    # appended codes: the oracle's quantiser on the GPU's own pre-quantisation rows
    for s in sess:
        P = int(case.pos_h[s])
        codes, scales = oracle.quantize_rows(np.ascontiguousarray(dump[:, :, s]))
        assert np.array_equal(case.kv[:, :, s, :, P].cpu().numpy(), codes)
        assert np.array_equal(case.sc[:, :, s, :, P].cpu().numpy().view(np.uint32), scales.view(np.uint32))
    # no other history byte moved
    mask = torch.ones_like(case.kv, dtype=torch.bool)
    for s in sess:
        mask[:, :, s, :, int(case.pos_h[s])] = False
    assert torch.equal(case.kv[mask], kv0[mask])


def test_hybrid_empty_slot_leaves_its_state_and_passes_x():
    w = synth.HYBRID_SMALL
    pos = synth.positions(w.attention_view(), w.S).copy()
    pos[2] = -1
    case = HybridCase(w, pos=pos)
    kv0, sc0, st0, _ = _run(case, range(w.S))
    assert np.array_equal(case.y_bits()[2], case.x_h[2])
    assert torch.equal(case.state[:, 2].view(torch.int32), st0[:, 2].view(torch.int32))
    assert torch.equal(case.kv[:, :, 2], kv0[:, :, 2])
    keep = [0, 1, 3, 4]
    W = synth.hybrid_weights_host(w)
    _y_within_oracle_sensitivity(w, W, keep, pos[keep], np.ascontiguousarray(case.x_h[keep]),
                                 case.y_bits()[keep])


def test_hybrid_all_slots_empty():
    # no session at all: y = x, no state, history byte or scale written
    w = synth.HYBRID_SMALL
    pos = np.full(w.S, -1, dtype=np.int32)
    case = HybridCase(w, pos=pos)
    kv0, sc0, st0, _ = _run(case, range(w.S))
    assert np.array_equal(case.y_bits(), case.x_h)
    assert torch.equal(case.state.view(torch.int32), st0.view(torch.int32))
    assert torch.equal(case.kv, kv0)
    assert torch.equal(case.sc.view(torch.int32), sc0.view(torch.int32))


def test_handle_kinds_are_not_interchangeable():
    # the decoder calls refuse a hybrid handle and the hybrid step a decoder
    # handle, before any launch
    w = synth.HYBRID_SMALL
    case = HybridCase(w)
    hw = fsd.HybridWave(case.cfg, case.S_max, w.T_max)
    dw = fsd.Wave(fsd.WaveConfig(2, 256, 4, 64, 688, 1e-5, 1e4), case.S_max, w.T_max)
    try:
        lib = fsd.lib()
        p = [case.weights.data_ptr(), case.kv.data_ptr(), case.sc.data_ptr(), case.pos.data_ptr(),
             case.x.data_ptr(), case.y.data_ptr()]
        assert lib.wave_step(hw.h, case.S, *p, None) == fsd.WAVE_EINVAL
        assert lib.wave_beat(hw.h, case.S, 2, p[0], p[1], p[2], p[3], 0, p[4], p[5], None) == fsd.WAVE_EINVAL
        assert lib.wave_depth(hw.h, case.S, 2, p[0], p[0], p[1], p[2], p[4], p[4], p[5], None) == fsd.WAVE_EINVAL
        assert lib.wave_hybrid_step(dw.h, case.S, p[0], p[1], p[2], case.state.data_ptr(), p[3], p[4], p[5],
                                    None) == fsd.WAVE_EINVAL
        torch.cuda.synchronize()
        assert hw.status() == fsd.WAVE_OK and dw.status() == fsd.WAVE_OK
    finally:
        hw.close()
        dw.close()


def test_hybrid_prefix_batch_in_a_larger_handle_matches_oracle():
    # S < S_max: the state and history are indexed by S_max-strided sessions
    w = synth.HYBRID_SMALL
    case = HybridCase(w, S=3, S_max=7)
    _run(case, range(3))
    W = synth.hybrid_weights_host(w)
    _y_within_oracle_sensitivity(w, W, [0, 1, 2], case.pos_h, np.ascontiguousarray(case.x_h), case.y_bits())
    kv_o, sc_o, st_o = oracle.hybrid_prefill(w, [0, 1, 2], case.pos_h)
    oracle.hybrid_step(w, W, kv_o, sc_o, st_o, case.pos_h, case.x_h)
    st_g = case.state[:, :3].cpu().numpy()
    assert _normwise(st_g[0], st_o[0]) <= 1e-3
    for lm in range(w.n_mamba):
        assert _normwise(st_g[lm], st_o[lm]) <= 2e-2, lm


def test_hybrid_maximum_batch():
    # S = S_max = 128: the projections' MMA at N = 128, three ring stages,
    # and 128 x 4 state items per block; every phase of sessions 0..3, and y
    # of sessions spread over the batch (the last one included)
    w = synth.HYBRID_SMALL
    case = HybridCase(w, S=128, S_max=128)
    _check_phases(case, 4)
    case = HybridCase(w, S=128, S_max=128)
    _run(case, range(128))
    W = synth.hybrid_weights_host(w)
    sess = [0, 1, 64, 126, 127]
    _y_within_oracle_sensitivity(w, W, sess, case.pos_h[sess], np.ascontiguousarray(case.x_h[sess]),
                                 case.y_bits()[sess])


@pytest.mark.parametrize("which", [6, 7, 8, 0])
def test_hybrid_timeout_at_each_hand_over(which):
    # one item never published: a selective-state in-projection tile (the
    # state items wait), one CTA's finished state items (the out-projection
    # waits), an out-projection tile (the next norm waits), an attention
    # block's QKV tile (attention waits).  Every CTA gives up, drains its
    # copies and returns WAVE_ETIMEOUT; the next step on the same context
    # is right again
    w = synth.HYBRID_SMALL
    case = HybridCase(w)
    wave = fsd.HybridWave(case.cfg, case.S_max, w.T_max)
    try:
        assert wave.barriers_per_step == 1
        wave.set_timeout_ns(20_000_000)  # 20 ms
        wave.debug_skip_signal(which, {6: 2, 7: 2, 8: 1, 0: 1}[which])   # items that exist at this shape
        case.step(wave)
        assert wave.status() == fsd.WAVE_ETIMEOUT
        wave.debug_skip_signal(0, -1)
        wave.set_timeout_ns(2_000_000_000)
        fresh = HybridCase(w)
        fresh.step(wave)
        assert wave.status() == fsd.WAVE_OK
    finally:
        wave.close()
    W = synth.hybrid_weights_host(w)
    _y_within_oracle_sensitivity(w, W, list(range(w.S)), fresh.pos_h, fresh.x_h, fresh.y_bits())


@pytest.fixture(scope="module")
def full():
    w = synth.HYBRID
    if torch.cuda.mem_get_info()[0] < 40e9:
        pytest.skip("needs ~20 GB of device memory")
    case = HybridCase(w, device_gen=True, poison=False)
    yield case
    del case
    torch.cuda.empty_cache()


def test_full_hybrid_step_matches_oracle_on_sampled_sessions(full):
    case = full
    w = case.w
    sess = [0, 23, 55]
    st_before = case.state[:, sess].cpu().numpy()
    La, H, D = w.n_attn, w.n_heads, w.head_dim
    dump = torch.full((La, 2, case.S_max, H, D), float("nan"), device="cuda")
    wave = fsd.HybridWave(case.cfg, case.S_max, w.T_max)
    try:
        wave.debug_dump_kv(dump)
        case.step(wave)
        assert wave.status() == fsd.WAVE_OK
    finally:
        wave.debug_dump_kv(None)
        wave.close()
    dump = dump.cpu().numpy()
    for s in sess:  # every appended code and scale: the oracle's quantiser on the GPU's own rows
        P = int(case.pos_h[s])
        codes, scales = oracle.quantize_rows(np.ascontiguousarray(dump[:, :, s]))
        assert np.array_equal(case.kv[:, :, s, :, P].cpu().numpy(), codes)
        assert np.array_equal(case.sc[:, :, s, :, P].cpu().numpy().view(np.uint32), scales.view(np.uint32))
    W = synth.hybrid_weights_host(w)
    kv_o, sc_o, st_o = oracle.hybrid_prefill(w, sess, case.pos_h[sess], poison=False)
    assert np.array_equal(st_o, st_before)                       # the generators agree
    # At this depth the model is chaotic (the oracle's own output moves by
    # 25-55% normwise for a one-ulp change of one element of x), so y is not
    # compared end to end; every phase of every block is, on its own inputs
    # (test_full_hybrid_every_phase_matches_oracle).  The first block, before
    # any cascade, is compared end to end here.
    oracle.hybrid_step(w, W, kv_o, sc_o, st_o, case.pos_h[sess], case.x_h[sess])
    st_g = case.state[:, sess].cpu().numpy()
    assert _normwise(st_g[0], st_o[0]) <= 1e-3                   # first block: a bf16 flip of xn at most


def test_full_hybrid_every_phase_matches_oracle(full):
    case = full
    case.W_h = synth.hybrid_weights_host(case.w)
    _check_phases(case, 3)
