"""Shared set-up for the GPU tests: seeded inputs on the device (through the
library's own quantiser for the FP8 history) and the same inputs for the CPU
oracle (through the oracle's quantiser).  Test infrastructure only."""
from __future__ import annotations

import numpy as np
import torch

import frame_step_decode_gb300 as fsd
import oracle
import synth

POISON_CODE = 0x7F


class DeviceCase:
    """Device buffers of one workload at S sessions (S_max = S unless given)."""

    def __init__(self, w, S=None, S_max=None, poison=True, device_gen=False, pos=None, keep_rowmajor=False):
        self.w = w
        self.S = w.S if S is None else S
        self.S_max = self.S if S_max is None else S_max
        self.cfg = fsd.WaveConfig.of(w)
        L, H, T, D = w.n_layers, w.n_heads, w.T_max, w.head_dim
        dev = "cuda"
        self.pos_h = synth.positions(w, self.S) if pos is None else np.asarray(pos, dtype=np.int32)
        self.pos = torch.from_numpy(self.pos_h).to(dev)
        self.x_h = synth.x_bf16(w, self.S)
        self.x = torch.from_numpy(self.x_h.view(np.int16)).to(dev).view(torch.bfloat16)
        self.y = torch.zeros_like(self.x)
        n_w = synth.weight_elems(w)
        if device_gen:
            rm = torch.empty(n_w, dtype=torch.bfloat16, device=dev)
            synth.weights_device(w, rm, torch.cuda.current_stream().cuda_stream)
        else:
            self.W_h = synth.weights_host(w)
            rm = torch.from_numpy(self.W_h.view(np.int16)).to(dev).view(torch.bfloat16)
        # the step reads the packed blob; the row-major one is kept only if asked
        self.weights = fsd.pack_weights(self.cfg, rm)
        self.weights_rm = rm if keep_rowmajor else None
        del rm
        self.kv = torch.zeros((L, 2, self.S_max, H, T, D), dtype=torch.uint8, device=dev)
        self.sc = torch.zeros((L, 2, self.S_max, H, T), dtype=torch.float32, device=dev)
        stream = torch.cuda.current_stream().cuda_stream
        raw = torch.empty((self.S, H, T, D), dtype=torch.float32, device=dev)
        for l in range(L):
            for which in range(2):
                if device_gen:
                    synth.kv_raw_device(w, l, which, 0, self.S, T, raw.data_ptr(), T, stream)
                else:
                    raw.copy_(torch.from_numpy(synth.kv_raw_host(w, l, which, 0, self.S, T)))
                fsd.kv_quantize(raw, self.kv[l, which, :self.S], self.sc[l, which, :self.S])
        del raw
        if poison:
            t = torch.arange(T, device=dev)
            mask = t[None, :] >= self.pos.long()[:, None]  # [S][T]
            m5 = mask[None, None, :, None, :].expand(L, 2, self.S, H, T)
            self.kv[:, :, :self.S][m5] = POISON_CODE
            self.sc[:, :, :self.S][m5] = float("nan")
        torch.cuda.synchronize()

    def y_bits(self) -> np.ndarray:
        """y as bf16 bit patterns (uint16) on the host."""
        return self.y.view(torch.int16).cpu().numpy().view(np.uint16)

    def step(self, wave, S=None, stream=None):
        return wave.step(self.S if S is None else S, self.weights, self.kv, self.sc, self.pos,
                         self.x, self.y, stream=stream)


def oracle_reference(w, sessions, pos, x_rows, W_h=None):
    """Oracle y (bf16 bits), y_exact and the history it wrote, for the listed
    sessions, from the oracle's own quantiser applied to the shared raw
    values."""
    W = synth.weights_host(w) if W_h is None else W_h
    pos = np.asarray(pos, dtype=np.int32)
    kv, sc = oracle.prefill_history(w, list(sessions), pos, poison=True)
    y, y_exact, kv_new = oracle.step(w, W, kv, sc, pos, np.ascontiguousarray(x_rows),
                                     want_kv_new=True)
    return y, y_exact, kv, sc, kv_new


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


def y_close(y_gpu_bits, y_ref_exact, atol=1e-3, rtol=2e-2):
    """Element-wise |y - y_ref| <= atol + rtol * |y_ref| (the stated bound)."""
    y = bf16_to_f64(y_gpu_bits)
    err = np.abs(y - y_ref_exact)
    bound = atol + rtol * np.abs(y_ref_exact)
    return bool(np.all(err <= bound)), float(np.max(err / bound))


class HybridCase:
    """Device buffers of the hybrid step at S sessions: the bf16 blob, the
    attention blocks' FP8 history (the library's own quantiser, poisoned
    beyond pos), the selective-state blocks' fp32 state, positions, x, y."""

    def __init__(self, w, pos=None, device_gen=False, poison=True, S=None, S_max=None, keep_rowmajor=False):
        self.w = w
        self.S = w.S if S is None else S
        self.S_max = self.S if S_max is None else S_max
        aw = w.attention_view()
        self.cfg = fsd.WaveHybridConfig.of(w)
        La, H, T, D = w.n_attn, w.n_heads, w.T_max, w.head_dim
        P, N, Hs = w.ssm_head_dim, w.ssm_state, w.ssm_heads
        dev = "cuda"
        stream = torch.cuda.current_stream().cuda_stream
        self.pos_h = synth.positions(aw, self.S) if pos is None else np.asarray(pos, dtype=np.int32)
        self.pos = torch.from_numpy(self.pos_h).to(dev)
        self.x_h = synth.x_bf16(aw, self.S)
        self.x = torch.from_numpy(self.x_h.view(np.int16)).to(dev).view(torch.bfloat16)
        self.y = torch.zeros_like(self.x)
        n_w = synth.hybrid_weight_elems(w)
        if device_gen:
            rm = torch.empty(n_w, dtype=torch.bfloat16, device=dev)
            synth.hybrid_weights_device(w, rm, stream)
        else:
            self.W_h = synth.hybrid_weights_host(w)
            rm = torch.from_numpy(self.W_h.view(np.int16)).to(dev).view(torch.bfloat16)
        self.weights = fsd.hybrid_pack_weights(self.cfg, rm)   # the packed blob the step reads
        self.weights_rm = rm if keep_rowmajor else None
        del rm
        self.kv = torch.zeros((La, 2, self.S_max, H, T, D), dtype=torch.uint8, device=dev)
        self.sc = torch.zeros((La, 2, self.S_max, H, T), dtype=torch.float32, device=dev)
        raw = torch.empty((self.S, H, T, D), dtype=torch.float32, device=dev)
        for l in range(La):
            for which in range(2):
                if device_gen:
                    synth.kv_raw_device(aw, l, which, 0, self.S, T, raw.data_ptr(), T, stream)
                else:
                    raw.copy_(torch.from_numpy(synth.kv_raw_host(aw, l, which, 0, self.S, T)))
                fsd.kv_quantize(raw, self.kv[l, which, :self.S], self.sc[l, which, :self.S])
        del raw
        if poison:
            t = torch.arange(T, device=dev)
            mask = t[None, :] >= self.pos.long().clamp(min=0)[:, None]
            m5 = mask[None, None, :, None, :].expand(La, 2, self.S, H, T)
            self.kv[:, :, :self.S][m5] = POISON_CODE
            self.sc[:, :, :self.S][m5] = float("nan")
        self.state = torch.empty((w.n_mamba, self.S_max, Hs, P, N), dtype=torch.float32, device=dev)
        for lm in range(w.n_mamba):
            if device_gen:
                synth.hybrid_state_device(w, lm, 0, self.S, self.state[lm].data_ptr(), stream)
            else:
                self.state[lm, :self.S].copy_(torch.from_numpy(synth.hybrid_state_host(w, lm, 0, self.S)))
        torch.cuda.synchronize()

    def y_bits(self) -> np.ndarray:
        return self.y.view(torch.int16).cpu().numpy().view(np.uint16)

    def step(self, wave, stream=None):
        return wave.hybrid_step(self.S, self.weights, self.kv, self.sc, self.state, self.pos, self.x, self.y,
                                stream=stream)


def codes_vs_oracle(gpu_codes, gpu_pre, ora_codes, ora_scales, ora_pre):
    """End-to-end check of one session's appended FP8 codes ([L][2][H][D])
    against the oracle's own codes.  The two paths' pre-quantisation rows
    differ (fp32 against fp64 arithmetic), so where a code differs it must
    be the code of a value within that difference of the oracle's: of some
    v/scale in [u - e, u + e], u the oracle's value in code units and e
    twice the row's measured difference in code units (once for the value,
    once for the row's scale through amax).  With rows that agree closely
    this allows one code step at a rounding boundary and nothing else.
    Returns the number of differing codes."""
    import oracle
    g = np.asarray(gpu_codes, dtype=np.int64)
    o = np.asarray(ora_codes, dtype=np.int64)
    mis = g != o
    n = int(np.count_nonzero(mis))
    if n == 0:
        return 0
    sc = np.asarray(ora_scales, dtype=np.float64)[..., None]
    pre_o = np.asarray(ora_pre, dtype=np.float64)
    safe = np.where(sc > 0, sc, 1.0)
    u = np.where(sc > 0, pre_o / safe, 0.0)
    err_u = np.where(sc > 0, np.max(np.abs(np.asarray(gpu_pre, dtype=np.float64) - pre_o), axis=-1,
                                    keepdims=True) / safe, 0.0)
    e = 2.02 * np.broadcast_to(err_u, u.shape)[mis] + 1e-5 * np.abs(u[mis]) + 1e-12
    lo = oracle.e4m3_encode((u[mis] - e).astype(np.float32)).astype(np.int64)
    hi = oracle.e4m3_encode((u[mis] + e).astype(np.float32)).astype(np.int64)
    signed = lambda c: np.where(c & 0x80, -(c & 0x7F), c & 0x7F)
    gs = signed(g[mis])
    assert np.all((signed(lo) <= gs) & (gs <= signed(hi))), \
        "a code differs by more than the two paths' difference can explain"
    return n


def dump_acts(wave, n, frames, run):
    """Run `run()` (one launch on `wave`) with the activation dump on for
    sessions 0..n-1 and return its records [frames][layers][n][R] (host
    fp32).  The launch's other outputs are the caller's to read."""
    layers = wave.cfg.n_layers
    buf = torch.full((frames, layers, n, wave.act_record_floats), float("nan"), dtype=torch.float32,
                     device="cuda")
    wave.debug_dump_acts(buf, n)
    try:
        run()
        assert wave.status() == fsd.WAVE_OK
    finally:
        wave.debug_dump_acts(None)
    return buf.cpu().numpy()
