"""GPU parity of wave_step against the CPU oracle, plus its invariants and
error paths.  Shapes: the tiny workload, a 3-layer d=512 shape whose every
dimension has a ragged tail (S = 19, F = 1376, positions up to 319), and
one layer of the 7B-class width (d 4096, 32 x 128 heads, F 11008): every
projection in the launch configuration of the full-size step (stream-K over
all CTAs, split tiles), at a size the oracle finishes in about a second."""
import numpy as np
import pytest
import torch

import frame_step_decode_gb300 as fsd
import synth
import phase_check
from gpu_case import DeviceCase, codes_vs_oracle, dump_acts, oracle_reference, y_close

pytestmark = pytest.mark.gpu

KV_RTOL = 2e-2  # pre-quantisation K/V against the oracle's, per row (normwise)


def _y_within_sensitivity(w, W, pos, x, y_bits, kv, sc):
    """Normwise y error per session at most three times the oracle's own
    response to a one-ulp change of one element of x (the largest over a
    few elements), and at most 5e-2.  kv, sc: the oracle's prefilled history
    (copied, not modified)."""
    import oracle
    _, y_exact, _ = oracle.step(w, W, kv.copy(), sc.copy(), pos, x)
    scale = np.max(np.abs(y_exact), axis=1)
    floor = np.zeros(len(pos))
    for el in (5, 100, 2000):
        xp = x.copy()
        xp[:, el % w.d_model] += 1
        _, y_p, _ = oracle.step(w, W, kv.copy(), sc.copy(), pos, xp)
        floor = np.maximum(floor, np.max(np.abs(y_p - y_exact), axis=1) / scale)
    err = np.max(np.abs(synth.bf16_bits_to_f32(y_bits).astype(np.float64) - y_exact), axis=1) / scale
    assert np.all(err <= np.maximum(3 * floor, 1e-3)) and np.all(err <= 5e-2), (err, floor)


def _check_case(case: DeviceCase, wave, sessions=None, normwise=False):
    """y within the stated bound (normwise=True: within three times the
    oracle's own one-ulp sensitivity, for shapes where even the oracle's
    response to a one-ulp change of x exceeds the element-wise bound); every
    appended code and scale equal, bit for bit, to the oracle quantiser
    applied to the GPU's own pre-quantisation K/V rows; those rows close to
    the oracle's; the codes against the oracle's own end to end (one step
    at most, and only at a rounding boundary); no other history byte moved."""
    import oracle
    w = case.w
    sessions = list(range(case.S)) if sessions is None else sessions
    L, H, D = w.n_layers, w.n_heads, w.head_dim
    kv_before = case.kv.clone()
    sc_before = case.sc.clone()
    dump = torch.full((L, 2, case.S_max, H, D), float("nan"), device="cuda")
    wave.debug_dump_kv(dump)
    try:
        case.step(wave)
        assert wave.status() == fsd.WAVE_OK
    finally:
        wave.debug_dump_kv(None)
    y = case.y_bits()
    pos = case.pos_h[sessions]
    W = getattr(case, "W_h", None)
    W = synth.weights_host(w) if W is None else W
    kv_o, sc_o = oracle.prefill_history(w, sessions, pos, poison=True)
    x_s = np.ascontiguousarray(case.x_h[sessions])
    kv_w, sc_w = kv_o.copy(), sc_o.copy()
    _, y_exact, kv_new = oracle.step(w, W, kv_w, sc_w, pos, x_s, want_kv_new=True)
    if normwise:
        _y_within_sensitivity(w, W, pos, x_s, y[sessions], kv_o, sc_o)
    else:
        ok, worst = y_close(y[sessions], y_exact)
        assert ok, f"y outside |dy| <= 1e-3 + 2e-2|y|: worst ratio {worst:.3f}"
    kv_g = case.kv.cpu().numpy()
    sc_g = case.sc.cpu().numpy()
    dump_h = dump.cpu().numpy()
    idx = np.arange(case.S)
    P = case.pos_h.astype(np.int64)
    got_codes = kv_g[:, :, idx, :, P]          # [S][L][2][H][D] (advanced index first)
    got_sc = sc_g[:, :, idx, :, P]             # [S][L][2][H]
    pre = np.ascontiguousarray(np.moveaxis(dump_h[:, :, :case.S], 2, 0))  # [S][L][2][H][D]
    assert np.all(np.isfinite(pre))
    ref_codes, ref_sc = oracle.quantize_rows(pre)
    assert np.array_equal(got_codes, ref_codes), "appended codes differ from the oracle quantiser"
    assert np.array_equal(got_sc.view(np.uint32), ref_sc.view(np.uint32))
    # end to end against the oracle's own codes (one step, at boundaries only)
    n_diff = 0
    for j, s in enumerate(sessions):
        Pj = int(pos[j])
        n_diff += codes_vs_oracle(got_codes[s], pre[s], kv_w[:, :, j, :, Pj], sc_w[:, :, j, :, Pj], kv_new[:, :, j])
    print(f"{w.name}: {n_diff} of {got_codes[sessions].size} appended codes differ from the oracle's own "
          "(each within the two paths' measured difference of the oracle's value)")
    # the GPU's pre-quantisation rows against the oracle's (fp64 path)
    for j, s in enumerate(sessions):
        a = pre[s].astype(np.float64)
        b = kv_new[:, :, j].astype(np.float64)
        err = np.max(np.abs(a - b), axis=-1)
        ref = np.max(np.abs(b), axis=-1)
        assert np.all(err <= KV_RTOL * ref + 1e-6), float(np.max(err / (ref + 1e-30)))
    # every other byte of the history is untouched
    mask = torch.ones(case.kv.shape[:5], dtype=torch.bool, device="cuda")
    for s in range(case.S):
        mask[:, :, s, :, int(case.pos_h[s])] = False
    assert torch.equal(case.kv[mask], kv_before[mask])
    assert torch.equal(torch.nan_to_num(case.sc[mask], nan=-7.0), torch.nan_to_num(sc_before[mask], nan=-7.0))


@pytest.fixture(scope="module")
def tiny():
    w = synth.TINY
    case = DeviceCase(w)
    wave = fsd.Wave(case.cfg, case.S_max, w.T_max)
    yield case, wave
    wave.close()


@pytest.fixture(scope="module")
def mid():
    w = synth.MID
    case = DeviceCase(w)
    wave = fsd.Wave(case.cfg, case.S_max, w.T_max)
    yield case, wave
    wave.close()


def test_tiny_step_matches_oracle(tiny):
    case, wave = tiny
    _check_case(case, wave)


def test_mid_step_matches_oracle(mid):
    case, wave = mid
    _check_case(case, wave)


@pytest.mark.parametrize("S", [1, 2, 7, 16, 17])
def test_ragged_batch_sizes(S):
    w = synth.MID
    case = DeviceCase(w, S=S, S_max=19)
    wave = fsd.Wave(case.cfg, 19, w.T_max)
    try:
        _check_case(case, wave)
    finally:
        wave.close()


@pytest.mark.parametrize("w", [synth.TINY, synth.MID], ids=["tiny", "mid"])
def test_maximum_batch(w):
    # S = S_max = 128, the largest batch the library takes: the projections'
    # MMA runs at N = 128 and their ring holds three stages instead of four
    case = DeviceCase(w, S=128, S_max=128)
    wave = fsd.Wave(case.cfg, 128, w.T_max)
    try:
        _check_case(case, wave)
    finally:
        wave.close()


def test_edge_positions():
    w = synth.MID
    # 32-token chunk boundaries and the extremes (T_max = 320 is below one
    # 512-token piece, so every history here is a single piece; the split
    # into pieces and their merge are tested on the long shapes below)
    pos = np.array([0, 1, 31, 32, 33, 63, 64, 95, 96, 127, 128, 255, 256, w.T_max - 1, 287, 288, 160],
                   dtype=np.int32)
    case = DeviceCase(w, S=pos.size, pos=pos)
    wave = fsd.Wave(case.cfg, case.S_max, w.T_max)
    try:
        _check_case(case, wave)
    finally:
        wave.close()


def test_batch_invariance_and_determinism():
    w = synth.MID
    big = DeviceCase(w, S=19)
    wave = fsd.Wave(big.cfg, 19, w.T_max)
    try:
        kv0, sc0 = big.kv.clone(), big.sc.clone()
        big.step(wave)
        assert wave.status() == fsd.WAVE_OK
        y_big = big.y.view(torch.int16).clone()
        # same inputs again: identical bits
        big.kv.copy_(kv0)
        big.sc.copy_(sc0)
        big.step(wave)
        assert wave.status() == fsd.WAVE_OK
        assert torch.equal(big.y.view(torch.int16), y_big)
        # a smaller batch (a prefix of the same draws) gives the same bits
        small = DeviceCase(w, S=5, S_max=19)
        small.step(wave)
        assert wave.status() == fsd.WAVE_OK
        assert torch.equal(small.y.view(torch.int16), y_big[:5])
        # changing the other sessions' inputs leaves session 0 unchanged
        big.kv.copy_(kv0)
        big.sc.copy_(sc0)
        big.x[1:] = -big.x[1:]
        big.step(wave)
        assert torch.equal(big.y.view(torch.int16)[0], y_big[0])
    finally:
        wave.close()


def test_invalid_arguments_are_rejected(tiny):
    case, wave = tiny
    for S in (0, -1, case.S_max + 1):
        assert case.step.__self__ is case
        rc = wave.step(S, case.weights, case.kv, case.sc, case.pos, case.x, case.y, check=False)
        assert rc == fsd.WAVE_EINVAL
    rc = wave.step(case.S, 0, case.kv, case.sc, case.pos, case.x, case.y, check=False)
    assert rc == fsd.WAVE_EINVAL
    rc = wave.step(case.S, case.weights.data_ptr() + 2, case.kv, case.sc, case.pos, case.x, case.y,
                   check=False)
    assert rc == fsd.WAVE_EINVAL
    # every buffer off its required alignment (16 bytes; 4 for the positions)
    args = [case.weights.data_ptr(), case.kv.data_ptr(), case.sc.data_ptr(), case.pos.data_ptr(),
            case.x.data_ptr(), case.y.data_ptr()]
    for i, off in ((1, 1), (2, 4), (3, 2), (4, 2), (5, 8)):
        bad_args = list(args)
        bad_args[i] += off
        assert wave.step(case.S, *bad_args, check=False) == fsd.WAVE_EINVAL, i
    for i in range(6):  # and null
        bad_args = list(args)
        bad_args[i] = 0
        assert wave.step(case.S, *bad_args, check=False) == fsd.WAVE_EINVAL, i
    lib = fsd.lib()
    for frames in (0, -1, 65):  # a beat of 1..64 frames
        assert lib.wave_beat(wave.h, case.S, frames, *args[:4], 0, args[4], args[5], None) == fsd.WAVE_EINVAL
    for steps in (0, case.w.T_max + 1, 65):  # a depth loop of 1..min(64, T_max) steps
        assert lib.wave_depth(wave.h, case.S, steps, args[0], args[0], args[1], args[2], args[4], args[4],
                              args[5], None) == fsd.WAVE_EINVAL
    torch.cuda.synchronize()
    assert wave.status() == fsd.WAVE_OK  # nothing was launched
    bad = fsd.WaveConfig(2, 256, 4, 96, 688, 1e-5, 1e4)
    with pytest.raises(fsd.WaveError):
        fsd.Wave(bad, 4, 64)
    with pytest.raises(fsd.WaveError):
        fsd.Wave(case.cfg, 129, 64)
    with pytest.raises(fsd.WaveError):
        fsd.Wave(case.cfg, 4, 62)


def test_empty_slots_pass_x_through_and_touch_no_cache():
    # negative positions: places of the fixed-shape batch with no session
    w = synth.MID
    pos = synth.positions(w, w.S).copy()
    empty = [1, 7, 18]
    pos[empty] = -1
    case = DeviceCase(w, pos=pos)
    wave = fsd.Wave(case.cfg, case.S_max, w.T_max)
    try:
        kv0, sc0 = case.kv.clone(), case.sc.clone()
        case.step(wave)
        assert wave.status() == fsd.WAVE_OK
        y = case.y_bits()
        assert np.array_equal(y[empty], case.x_h[empty])
        assert torch.equal(case.kv[:, :, empty], kv0[:, :, empty])
        assert torch.equal(case.sc[:, :, empty].view(torch.int32), sc0[:, :, empty].view(torch.int32))
        sess = [s for s in range(w.S) if s not in empty]
        _, y_exact, _, _, _ = oracle_reference(w, sess, pos[sess], case.x_h[sess])
        ok, worst = y_close(y[sess], y_exact)
        assert ok, f"worst ratio {worst:.3f}"
    finally:
        wave.close()


def test_shortest_history_capacity():
    # T_max = 4, the smallest the library takes: every chunk and scale copy
    # reaches past the end of a session's history (and of the whole cache)
    from dataclasses import replace
    w = replace(synth.TINY, T_max=4, pos_lo=0, pos_hi=4, name="tiny-2L-d256-h4x64-f688-T4")
    case = DeviceCase(w, S=8, pos=np.array([0, 1, 2, 3, 3, 2, 1, 0], dtype=np.int32))
    wave = fsd.Wave(case.cfg, case.S_max, w.T_max)
    try:
        _check_case(case, wave)
    finally:
        wave.close()


def test_output_may_alias_input():
    # y written over x (the header allows it): the same bits as with a
    # separate y, empty slots included
    w = synth.MID
    pos = synth.positions(w, w.S).copy()
    pos[[3, 11]] = -1
    ref = DeviceCase(w, pos=pos)
    inplace = DeviceCase(w, pos=pos)
    wave = fsd.Wave(ref.cfg, ref.S_max, w.T_max)
    try:
        ref.step(wave)
        assert wave.status() == fsd.WAVE_OK
        wave.step(inplace.S, inplace.weights, inplace.kv, inplace.sc, inplace.pos, inplace.x, inplace.x)
        assert wave.status() == fsd.WAVE_OK
        got = inplace.x.view(torch.int16).cpu().numpy().view(np.uint16)
        assert np.array_equal(got, ref.y_bits())
        assert torch.equal(inplace.kv, ref.kv)
        assert torch.equal(inplace.sc.view(torch.int32), ref.sc.view(torch.int32))
    finally:
        wave.close()


def test_all_slots_empty():
    # a batch with no session at all: no attention work, y = x everywhere,
    # not one history byte or scale written
    w = synth.MID
    pos = np.full(w.S, -1, dtype=np.int32)
    case = DeviceCase(w, pos=pos)
    wave = fsd.Wave(case.cfg, case.S_max, w.T_max)
    try:
        kv0, sc0 = case.kv.clone(), case.sc.clone()
        for _ in range(2):
            case.step(wave)
            assert wave.status() == fsd.WAVE_OK
            assert np.array_equal(case.y_bits(), case.x_h)
            assert torch.equal(case.kv, kv0)
            assert torch.equal(case.sc.view(torch.int32), sc0.view(torch.int32))
    finally:
        wave.close()


@pytest.mark.parametrize("w", [synth.TINY, synth.MID])
def test_two_frame_beat_equals_two_steps_and_rolls_positions(w):
    # one launch of two frames against two single-frame launches with the
    # positions advanced on the host: same kernels, same order -> same bits
    pos = synth.positions(w, w.S).copy()
    pos = np.minimum(pos, w.T_max - 2)
    pos[w.S // 2] = -1  # an empty slot stays empty in both frames
    a = DeviceCase(w, pos=pos)
    b = DeviceCase(w, pos=pos)
    x2 = torch.stack([a.x, a.x.flip(0)])  # frame 1 gets other rows
    y2 = torch.zeros_like(x2)
    wave = fsd.Wave(a.cfg, a.S_max, w.T_max)
    try:
        wave.beat(w.S, 2, a.weights, a.kv, a.sc, a.pos, x2, y2, advance=True)
        assert wave.status() == fsd.WAVE_OK
        ref = []
        for f in range(2):
            xf = x2[f].contiguous()
            yf = torch.zeros_like(xf)
            wave.step(w.S, b.weights, b.kv, b.sc, b.pos, xf, yf)
            assert wave.status() == fsd.WAVE_OK
            ref.append(yf)
            b.pos += (b.pos >= 0).int()
        assert torch.equal(y2[0].view(torch.int16), ref[0].view(torch.int16))
        assert torch.equal(y2[1].view(torch.int16), ref[1].view(torch.int16))
        assert torch.equal(a.kv, b.kv)
        assert torch.equal(a.sc.view(torch.int32), b.sc.view(torch.int32))
        assert torch.equal(a.pos, b.pos)
        assert a.pos[w.S // 2].item() == -1
        # and frame 1 against the oracle, from the oracle's own frame-0 state
        import oracle
        sess = [s for s in range(w.S) if pos[s] >= 0]
        kv_o, sc_o = oracle.prefill_history(w, sess, pos[sess], poison=True)
        W = synth.weights_host(w)
        x_h = x2.view(torch.int16).cpu().numpy().view(np.uint16)
        oracle.step(w, W, kv_o, sc_o, pos[sess], np.ascontiguousarray(x_h[0][sess]))
        _, y1_exact, _ = oracle.step(w, W, kv_o, sc_o, pos[sess] + 1, np.ascontiguousarray(x_h[1][sess]))
        y1 = y2[1].view(torch.int16).cpu().numpy().view(np.uint16)
        ok, worst = y_close(y1[sess], y1_exact)
        assert ok, f"worst ratio {worst:.3f}"
    finally:
        wave.close()


def test_beat_without_advance_and_with_a_frame_past_t_max():
    # frame 1 runs at position + 1: a session at T_max - 1 is out of range
    # there (WAVE_EPOS, nothing written in that frame); positions stay as
    # given when the advance is off; the other sessions match two steps
    w = synth.TINY
    pos = synth.positions(w, w.S).copy()
    pos = np.minimum(pos, w.T_max - 2)
    pos[1] = w.T_max - 1
    a = DeviceCase(w, pos=pos)
    b = DeviceCase(w, pos=pos)
    x2 = torch.stack([a.x, a.x.flip(0)])
    y2 = torch.zeros_like(x2)
    wave = fsd.Wave(a.cfg, a.S_max, w.T_max)
    try:
        wave.beat(w.S, 2, a.weights, a.kv, a.sc, a.pos, x2, y2, advance=False)
        assert wave.status() == fsd.WAVE_EPOS
        assert torch.equal(a.pos.cpu(), torch.from_numpy(pos))
        ys = []
        for f in range(2):
            yf = torch.zeros_like(x2[f])
            wave.step(w.S, b.weights, b.kv, b.sc, b.pos, x2[f].contiguous(), yf)
            wave.status()
            ys.append(yf)
            b.pos += 1
        for f in range(2):
            keep = [s for s in range(w.S) if f == 0 or s != 1]
            assert torch.equal(y2[f][keep].view(torch.int16), ys[f][keep].view(torch.int16))
        assert torch.equal(a.kv, b.kv)
    finally:
        wave.close()


def test_out_of_range_position_is_reported_and_skipped():
    w = synth.TINY
    case = DeviceCase(w)
    wave = fsd.Wave(case.cfg, case.S_max, w.T_max)
    try:
        bad = case.pos.clone()
        bad[2] = w.T_max
        kv0 = case.kv.clone()
        rc = wave.step(case.S, case.weights, case.kv, case.sc, bad, case.x, case.y)
        assert rc == fsd.WAVE_OK
        assert wave.status() == fsd.WAVE_EPOS
        # no cache byte of session 2 changed
        assert torch.equal(case.kv[:, :, 2], kv0[:, :, 2])
        # the other sessions still match the oracle
        y = case.y_bits()
        sess = [0, 1, 3]
        _, y_exact, _, _, _ = oracle_reference(w, sess, case.pos_h[sess], case.x_h[sess])
        ok, worst = y_close(y[sess], y_exact)
        assert ok, worst
        assert wave.status() == fsd.WAVE_OK  # cleared by the previous read
    finally:
        wave.close()


def test_barrier_timeout_is_reported_and_context_survives():
    w = synth.TINY
    case = DeviceCase(w)
    wave = fsd.Wave(case.cfg, case.S_max, w.T_max)
    try:
        wave.set_timeout_ns(20_000_000)  # 20 ms
        wave.debug_skip_barrier(3, 0)
        case.step(wave)
        assert wave.status() == fsd.WAVE_ETIMEOUT
        wave.debug_skip_barrier(-1, -1)
        wave.set_timeout_ns(2_000_000_000)
        fresh = DeviceCase(w)
        fresh.step(wave)
        assert wave.status() == fsd.WAVE_OK
        y = fresh.y_bits()
        _, y_exact, _, _, _ = oracle_reference(w, range(fresh.S), fresh.pos_h, fresh.x_h)
        assert y_close(y, y_exact)[0]
    finally:
        wave.close()


# one decoder layer of the 7B-class width, a few short sessions
WIDE1 = synth.Workload("wide-1L-d4096-h32x128-f11008", 1, 4096, 32, 128, 11008, S=5, T_max=64, pos_lo=1,
                       pos_hi=64)


@pytest.fixture(scope="module")
def wide_weights():
    return synth.weights_host(WIDE1)


def test_wide_layer_matches_oracle(wide_weights):
    # at this width even one layer is ill-conditioned element-wise: the
    # oracle's own y moves by ~15x the element-wise bound for a one-ulp change
    # of one element of x, so y is held normwise to that sensitivity
    case = DeviceCase(WIDE1, device_gen=True)
    case.W_h = wide_weights
    wave = fsd.Wave(case.cfg, case.S_max, WIDE1.T_max)
    try:
        _check_case(case, wave, normwise=True)
    finally:
        wave.close()


SIGNALS = {"qkv": 0, "gate/up": 1, "attention": 2, "o": 3, "norm": 5}


@pytest.mark.parametrize("barrier", [0, "qkv", "gate/up", "attention", "o", "norm"])
def test_timeout_at_each_wait_of_a_wide_layer(barrier, wide_weights):
    # the one grid barrier of a step (after the prologue) and the hand-overs
    # between phases, where one item is never published: a QKV tile
    # (attention waits), a gate/up tile (the down projection waits), a head's
    # attention rows (the output projection waits), an output-projection tile
    # (the second norm waits) or a norm row (gate/up waits).  Every CTA gives
    # up there, drains its copies and returns WAVE_ETIMEOUT, and the next
    # step is exact
    case = DeviceCase(WIDE1, device_gen=True)
    wave = fsd.Wave(case.cfg, case.S_max, WIDE1.T_max)
    try:
        assert wave.barriers_per_step == 1
        wave.set_timeout_ns(20_000_000)  # 20 ms
        if barrier in SIGNALS:
            wave.debug_skip_signal(SIGNALS[barrier], 2)
        else:
            wave.debug_skip_barrier(7, barrier)
        case.step(wave)
        assert wave.status() == fsd.WAVE_ETIMEOUT
        wave.debug_skip_barrier(-1, -1)
        wave.debug_skip_signal(0, -1)
        wave.set_timeout_ns(2_000_000_000)
        fresh = DeviceCase(WIDE1, device_gen=True)
        fresh.step(wave)
        assert wave.status() == fsd.WAVE_OK
        import oracle
        sess = list(range(fresh.S))
        kv_o, sc_o = oracle.prefill_history(WIDE1, sess, fresh.pos_h, poison=True)
        _y_within_sensitivity(WIDE1, wide_weights, fresh.pos_h, np.ascontiguousarray(fresh.x_h), fresh.y_bits(),
                              kv_o, sc_o)
    finally:
        wave.close()


# ----------------------------------------------------------------- phases
def _check_phases(case, wave, n=None):
    """Every phase of every layer of sessions 0..n-1 against the oracle's
    functions on the GPU's own inputs to that phase (tests/phase_check.py),
    under the stated bound and the tight one; and the dump's kernel gives
    the same y bits as the usual kernel."""
    w = case.w
    n = case.S if n is None else n
    kv0, sc0 = case.kv.clone(), case.sc.clone()
    case.step(wave)
    assert wave.status() == fsd.WAVE_OK
    y_plain = case.y_bits()
    case.kv.copy_(kv0)
    case.sc.copy_(sc0)
    recs = dump_acts(wave, n, 1, lambda: case.step(wave))
    y = case.y_bits()
    assert np.array_equal(y, y_plain), "the dump's kernel must give the usual kernel's bits"
    W = getattr(case, "W_h", None)
    W = synth.weights_host(w) if W is None else W
    worst = {}
    for s in range(n):
        P = int(case.pos_h[s])
        kv = case.kv[:, :, s, :, :P + 1].cpu().numpy()
        sc = case.sc[:, :, s, :, :P + 1].cpu().numpy()
        phase_check.check_decoder_frame(w, W, recs[0, :, s], P, kv, sc, case.x_h[s], y[s], worst)
    print(w.name, {k: round(v, 3) for k, v in worst.items()})
    assert all(v <= 1.0 for v in worst.values()), worst


def test_every_phase_matches_oracle_tiny(tiny):
    case, wave = tiny
    _check_phases(case, wave)


def test_every_phase_matches_oracle_mid(mid):
    case, wave = mid
    _check_phases(case, wave)


def test_every_phase_matches_oracle_wide_layer(wide_weights):
    case = DeviceCase(WIDE1, device_gen=True)
    case.W_h = wide_weights
    wave = fsd.Wave(case.cfg, case.S_max, WIDE1.T_max)
    try:
        _check_phases(case, wave)
    finally:
        wave.close()


# ------------------------------------------------ split histories and their merge
# Histories longer than one 512-token piece are cut into several pieces
# whose partial results the merge phase combines: positions at the chunk
# (32) and piece (512) boundaries and both head dims.
MERGE_POS = np.array([0, 31, 32, 511, 512, 513, 1023, 1024, 1535, 1536, 1663, 777], dtype=np.int32)
MERGE128 = synth.Workload("merge-2L-d512-h4x128-f1376", 2, 512, 4, 128, 1376, S=12, T_max=1664, pos_lo=0,
                          pos_hi=1664)
MERGE64 = synth.Workload("merge-2L-d512-h8x64-f1376", 2, 512, 8, 64, 1376, S=12, T_max=1664, pos_lo=0,
                         pos_hi=1664)


@pytest.mark.parametrize("w", [MERGE128, MERGE64], ids=["D128", "D64"])
def test_split_histories_merge_to_the_oracle(w):
    case = DeviceCase(w, pos=MERGE_POS)
    wave = fsd.Wave(case.cfg, case.S_max, w.T_max)
    try:
        _check_case(case, wave)
        _check_phases(case, wave)
    finally:
        wave.close()


# ----------------------------------------------------------------- status
def test_status_reads_without_synchronising():
    # wave_status synchronises nothing: called while the step still waits
    # behind ~100 ms of other work on its stream it returns at once and
    # reports no finished launch; after the caller synchronises it reports
    # the step's error, then nothing (cleared, on the host and the device)
    import time
    w = synth.TINY
    case = DeviceCase(w)
    wave = fsd.Wave(case.cfg, case.S_max, w.T_max)
    stream = torch.cuda.Stream()
    try:
        bad = case.pos.clone()
        bad[1] = w.T_max
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            torch.cuda._sleep(200_000_000)
            wave.step(case.S, case.weights, case.kv, case.sc, bad, case.x, case.y, stream=stream)
            t0 = time.perf_counter()
            rc = fsd.lib().wave_status(wave.h)
            dt = time.perf_counter() - t0
            running = not stream.query()
        assert running and dt < 0.05, (running, dt)
        assert rc == fsd.WAVE_OK
        stream.synchronize()
        assert fsd.lib().wave_status(wave.h) == fsd.WAVE_EPOS
        assert fsd.lib().wave_status(wave.h) == fsd.WAVE_OK
        wave.step(case.S, case.weights, case.kv, case.sc, case.pos, case.x, case.y, stream=stream)
        stream.synchronize()
        assert fsd.lib().wave_status(wave.h) == fsd.WAVE_OK
    finally:
        wave.close()
