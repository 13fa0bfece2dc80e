"""Python binding of libwave.so (include/wave.h): argument marshalling only.

Every step of the frame runs in the library's CUDA kernels; PyTorch is used
only to own device memory and streams.  There is no fallback: if the library
is not built, importing the binding's entry points raises.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libwave.so")

WAVE_OK, WAVE_EINVAL, WAVE_ECUDA, WAVE_ELAUNCH = 0, -1, -2, -3
WAVE_ETIMEOUT, WAVE_EPOS, WAVE_EDEVICE, WAVE_ENOMEM = -4, -5, -6, -7


class WaveConfig(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int), ("d_model", ctypes.c_int), ("n_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("ffn", ctypes.c_int), ("rms_eps", ctypes.c_float),
                ("rope_base", ctypes.c_float)]

    @classmethod
    def of(cls, w) -> "WaveConfig":
        """From any object with the decoder-shape attributes."""
        return cls(w.n_layers, w.d_model, w.n_heads, w.head_dim, w.ffn, w.rms_eps, w.rope_base)


class WaveHybridConfig(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int), ("d_model", ctypes.c_int), ("attn_every", ctypes.c_int),
                ("n_heads", ctypes.c_int), ("head_dim", ctypes.c_int), ("ssm_heads", ctypes.c_int),
                ("ssm_head_dim", ctypes.c_int), ("ssm_state", ctypes.c_int), ("rms_eps", ctypes.c_float),
                ("rope_base", ctypes.c_float)]

    @classmethod
    def of(cls, w) -> "WaveHybridConfig":
        """From any object with the hybrid-shape attributes."""
        return cls(w.n_layers, w.d_model, w.attn_every, w.n_heads, w.head_dim, w.ssm_heads, w.ssm_head_dim,
                   w.ssm_state, w.rms_eps, w.rope_base)


class WaveError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {strerror(code)} ({code})")
        self.code = code


_lib = None
EXPORTS = ("wave_create", "wave_destroy", "wave_weights_bytes", "wave_weight_offset", "wave_packed_weights_bytes",
           "wave_pack_weights", "wave_hybrid_packed_weights_bytes", "wave_hybrid_pack_weights",
           "wave_step", "wave_beat", "wave_depth",
           "wave_status", "wave_strerror", "wave_kv_quantize", "wave_fp8_encode", "wave_step_static",
           "wave_set_timeout_ns", "wave_debug_skip_barrier", "wave_debug_skip_signal", "wave_debug_dump_kv", "wave_debug_dump_acts",
           "wave_debug_act_record_floats", "wave_debug_phase_times", "wave_debug_arrival_times",
           "wave_grid_size", "wave_barriers_per_step", "wave_phases_per_step", "wave_hybrid_create", "wave_hybrid_step",
           "wave_hybrid_weights_bytes", "wave_hybrid_layer_offset")


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built: run frame_step_decode_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
        cfgp = ctypes.POINTER(WaveConfig)
        L.wave_create.argtypes = [cfgp, i32, i32, ctypes.POINTER(vp)]
        L.wave_create.restype = i32
        L.wave_destroy.argtypes = [vp]
        L.wave_destroy.restype = None
        L.wave_weights_bytes.argtypes = [cfgp]
        L.wave_weights_bytes.restype = sz
        L.wave_weight_offset.argtypes = [cfgp, i32, i32]
        L.wave_weight_offset.restype = sz
        L.wave_packed_weights_bytes.argtypes = [cfgp]
        L.wave_packed_weights_bytes.restype = sz
        L.wave_pack_weights.argtypes = [cfgp, vp, vp, vp]
        L.wave_pack_weights.restype = i32
        L.wave_hybrid_packed_weights_bytes.argtypes = [ctypes.POINTER(WaveHybridConfig)]
        L.wave_hybrid_packed_weights_bytes.restype = sz
        L.wave_hybrid_pack_weights.argtypes = [ctypes.POINTER(WaveHybridConfig), vp, vp, vp]
        L.wave_hybrid_pack_weights.restype = i32
        L.wave_step.argtypes = [vp, i32, vp, vp, vp, vp, vp, vp, vp]
        L.wave_step.restype = i32
        L.wave_beat.argtypes = [vp, i32, i32, vp, vp, vp, vp, i32, vp, vp, vp]
        L.wave_beat.restype = i32
        L.wave_depth.argtypes = [vp, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp]
        L.wave_depth.restype = i32
        L.wave_hybrid_create.argtypes = [ctypes.POINTER(WaveHybridConfig), i32, i32, ctypes.POINTER(vp)]
        L.wave_hybrid_create.restype = i32
        L.wave_hybrid_step.argtypes = [vp, i32, vp, vp, vp, vp, vp, vp, vp, vp]
        L.wave_hybrid_step.restype = i32
        L.wave_hybrid_weights_bytes.argtypes = [ctypes.POINTER(WaveHybridConfig)]
        L.wave_hybrid_weights_bytes.restype = ctypes.c_size_t
        L.wave_hybrid_layer_offset.argtypes = [ctypes.POINTER(WaveHybridConfig), i32]
        L.wave_hybrid_layer_offset.restype = ctypes.c_size_t
        L.wave_status.argtypes = [vp]
        L.wave_status.restype = i32
        L.wave_strerror.argtypes = [i32]
        L.wave_strerror.restype = ctypes.c_char_p
        L.wave_kv_quantize.argtypes = [vp, i64, i32, vp, vp, vp]
        L.wave_kv_quantize.restype = i32
        L.wave_fp8_encode.argtypes = [vp, i64, vp, vp]
        L.wave_fp8_encode.restype = i32
        L.wave_step_static.argtypes = [cfgp, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp]
        L.wave_step_static.restype = i32
        L.wave_set_timeout_ns.argtypes = [vp, ctypes.c_longlong]
        L.wave_set_timeout_ns.restype = i32
        L.wave_debug_skip_barrier.argtypes = [vp, i32, i32]
        L.wave_debug_skip_barrier.restype = i32
        L.wave_debug_skip_signal.argtypes = [vp, i32, i32]
        L.wave_debug_skip_signal.restype = i32
        L.wave_debug_dump_kv.argtypes = [vp, vp]
        L.wave_debug_dump_kv.restype = i32
        L.wave_debug_dump_acts.argtypes = [vp, vp, i32]
        L.wave_debug_dump_acts.restype = i32
        L.wave_debug_act_record_floats.argtypes = [vp]
        L.wave_debug_act_record_floats.restype = ctypes.c_longlong
        L.wave_debug_phase_times.argtypes = [vp, vp]
        L.wave_debug_phase_times.restype = i32
        L.wave_debug_arrival_times.argtypes = [vp, vp]
        L.wave_debug_arrival_times.restype = i32
        L.wave_grid_size.argtypes = [vp]
        L.wave_grid_size.restype = i32
        L.wave_barriers_per_step.argtypes = [vp]
        L.wave_barriers_per_step.restype = i32
        L.wave_phases_per_step.argtypes = [vp]
        L.wave_phases_per_step.restype = i32
        _lib = L
    return _lib


def strerror(code: int) -> str:
    return lib().wave_strerror(code).decode()


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def weights_bytes(cfg: WaveConfig) -> int:
    return lib().wave_weights_bytes(ctypes.byref(cfg))


def weight_offset(cfg: WaveConfig, layer: int, which: int) -> int:
    return lib().wave_weight_offset(ctypes.byref(cfg), layer, which)


def packed_weights_bytes(cfg: WaveConfig) -> int:
    return lib().wave_packed_weights_bytes(ctypes.byref(cfg))


def pack_weights(cfg: WaveConfig, src, dst=None, stream=None):
    """wave_pack_weights: the packed blob the step reads, from the row-major
    blob src (a device tensor).  Returns dst (a new bf16 device tensor when
    not given)."""
    import torch
    if dst is None:
        dst = torch.empty(packed_weights_bytes(cfg) // 2, dtype=torch.bfloat16, device=src.device)
    rc = lib().wave_pack_weights(ctypes.byref(cfg), _ptr(src), _ptr(dst), _stream(stream))
    if rc != WAVE_OK:
        raise WaveError(rc, "wave_pack_weights")
    return dst


def hybrid_packed_weights_bytes(cfg: "WaveHybridConfig") -> int:
    return lib().wave_hybrid_packed_weights_bytes(ctypes.byref(cfg))


def hybrid_pack_weights(cfg: "WaveHybridConfig", src, dst=None, stream=None):
    """wave_hybrid_pack_weights (as pack_weights, for the hybrid blob)."""
    import torch
    if dst is None:
        dst = torch.empty(hybrid_packed_weights_bytes(cfg) // 2, dtype=torch.bfloat16, device=src.device)
    rc = lib().wave_hybrid_pack_weights(ctypes.byref(cfg), _ptr(src), _ptr(dst), _stream(stream))
    if rc != WAVE_OK:
        raise WaveError(rc, "wave_hybrid_pack_weights")
    return dst


class Wave:
    """A step context: wave_create / wave_step / wave_status / wave_destroy."""

    def __init__(self, cfg: WaveConfig, S_max: int, T_max: int):
        self.cfg = cfg
        self.S_max, self.T_max = S_max, T_max
        h = ctypes.c_void_p()
        rc = lib().wave_create(ctypes.byref(cfg), S_max, T_max, ctypes.byref(h))
        if rc != WAVE_OK:
            raise WaveError(rc, "wave_create")
        self.h = h

    def step(self, S, weights, kv, kv_scales, positions, x, y, stream=None, check=True) -> int:
        rc = lib().wave_step(self.h, S, _ptr(weights), _ptr(kv), _ptr(kv_scales), _ptr(positions),
                             _ptr(x), _ptr(y), _stream(stream))
        if check and rc != WAVE_OK:
            raise WaveError(rc, "wave_step")
        return rc

    def depth(self, S, steps, weights, w_proj, kv, kv_scales, x0, xs, y, stream=None, check=True) -> int:
        """The inner depth loop: `steps` dependent steps, x_k = bf16(W_p y_{k-1})
        (xs [steps][S][d] scratch, y [steps][S][d])."""
        rc = lib().wave_depth(self.h, S, steps, _ptr(weights), _ptr(w_proj), _ptr(kv), _ptr(kv_scales),
                              _ptr(x0), _ptr(xs), _ptr(y), _stream(stream))
        if check and rc != WAVE_OK:
            raise WaveError(rc, "wave_depth")
        return rc

    def beat(self, S, frames, weights, kv, kv_scales, positions, x, y, advance=True, stream=None,
             check=True) -> int:
        """`frames` frames in one launch (x, y [frames][S][d]); frame f at
        positions + f; positions advanced by `frames` on the device when
        `advance` is set."""
        rc = lib().wave_beat(self.h, S, frames, _ptr(weights), _ptr(kv), _ptr(kv_scales), _ptr(positions),
                             int(bool(advance)), _ptr(x), _ptr(y), _stream(stream))
        if check and rc != WAVE_OK:
            raise WaveError(rc, "wave_beat")
        return rc

    def status(self, sync: bool = True) -> int:
        """wave_status.  The C call synchronises nothing and reports the
        launches already finished; with sync (the default) the device is
        synchronised first, so that it reports every launch made so far."""
        if sync:
            import torch
            torch.cuda.synchronize()
        return lib().wave_status(self.h)

    def set_timeout_ns(self, ns: int) -> None:
        rc = lib().wave_set_timeout_ns(self.h, ns)
        if rc != WAVE_OK:
            raise WaveError(rc, "wave_set_timeout_ns")

    def debug_skip_barrier(self, cta: int, barrier: int) -> None:
        lib().wave_debug_skip_barrier(self.h, cta, barrier)

    def debug_skip_signal(self, which: int, index: int) -> None:
        """Testing hook: later steps never publish item `index` of kind
        `which` (0 QKV tile, 1 gate/up tile, 2 a head's attention rows, 3 O
        tile, 4 down tile, 5 norm row; hybrid: 6 selective-state
        in-projection tile, 7 a CTA's finished state items, 8 selective-state
        out-projection tile); index < 0 disables."""
        rc = lib().wave_debug_skip_signal(self.h, which, index)
        if rc != WAVE_OK:
            raise WaveError(rc, "wave_debug_skip_signal")

    def debug_dump_kv(self, dst) -> None:
        """Testing hook: later steps write their pre-quantisation K/V rows
        into dst ([L][2][S_max][H][D] fp32 on the device); None disables."""
        lib().wave_debug_dump_kv(self.h, _ptr(dst))

    def debug_dump_acts(self, dst, n_sessions: int = 0) -> None:
        """Testing hook: later launches record every phase's input and output
        for sessions 0..n_sessions-1 into dst ([frames][layers][n][R] fp32 on
        the device, R = act_record_floats); None disables."""
        rc = lib().wave_debug_dump_acts(self.h, _ptr(dst), n_sessions if dst is not None else 0)
        if rc != WAVE_OK:
            raise WaveError(rc, "wave_debug_dump_acts")

    @property
    def act_record_floats(self) -> int:
        return lib().wave_debug_act_record_floats(self.h)

    def debug_phase_times(self, dst) -> None:
        """Profiling hook: later steps write globaltimer stamps (int64) at
        entry, after every grid barrier and at exit into dst; None disables."""
        lib().wave_debug_phase_times(self.h, _ptr(dst))

    def debug_arrival_times(self, dst) -> None:
        """Profiling hook: later steps write the globaltimer stamp at which
        each CTA finished each phase into dst ([phases][grid] int64); None
        disables."""
        lib().wave_debug_arrival_times(self.h, _ptr(dst))

    @property
    def grid(self) -> int:
        return lib().wave_grid_size(self.h)

    @property
    def barriers_per_step(self) -> int:
        return lib().wave_barriers_per_step(self.h)

    @property
    def phases_per_step(self) -> int:
        return lib().wave_phases_per_step(self.h)

    def close(self) -> None:
        if getattr(self, "h", None):
            lib().wave_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def step_static(cfg: WaveConfig, S_max: int, T_max: int, S: int, weights, kv, kv_scales, positions,
                x, y, stream=None) -> int:
    """wave_step_static: one frame with the library's fixed scratch instead
    of an allocated workspace, for callers that cannot allocate device memory.
    Waits for the step and returns its status code."""
    return lib().wave_step_static(ctypes.byref(cfg), S_max, T_max, S, _ptr(weights), _ptr(kv),
                                  _ptr(kv_scales), _ptr(positions), _ptr(x), _ptr(y),
                                  _stream(stream))


def kv_quantize(v, codes, scales, stream=None) -> None:
    """FP8 quantiser of the K/V append on rows of v (last dim D)."""
    D = v.shape[-1]
    rows = v.numel() // D
    rc = lib().wave_kv_quantize(_ptr(v), rows, D, _ptr(codes), _ptr(scales), _stream(stream))
    if rc != WAVE_OK:
        raise WaveError(rc, "wave_kv_quantize")


def fp8_encode(inp, out, stream=None, n: int | None = None) -> None:
    n = inp.numel() if n is None else n
    rc = lib().wave_fp8_encode(_ptr(inp), n, _ptr(out), _stream(stream))
    if rc != WAVE_OK:
        raise WaveError(rc, "wave_fp8_encode")


class HybridWave(Wave):
    """A hybrid-step context: wave_hybrid_create / wave_hybrid_step (status,
    hooks and close as Wave)."""

    def __init__(self, cfg: WaveHybridConfig, S_max: int, T_max: int):
        self.cfg = cfg
        self.S_max, self.T_max = S_max, T_max
        h = ctypes.c_void_p()
        rc = lib().wave_hybrid_create(ctypes.byref(cfg), S_max, T_max, ctypes.byref(h))
        if rc != WAVE_OK:
            raise WaveError(rc, "wave_hybrid_create")
        self.h = h

    def hybrid_step(self, S, weights, kv, kv_scales, ssm_state, positions, x, y, stream=None,
                    check=True) -> int:
        rc = lib().wave_hybrid_step(self.h, S, _ptr(weights), _ptr(kv), _ptr(kv_scales), _ptr(ssm_state),
                                    _ptr(positions), _ptr(x), _ptr(y), _stream(stream))
        if check and rc != WAVE_OK:
            raise WaveError(rc, "wave_hybrid_step")
        return rc


def hybrid_weights_bytes(cfg: WaveHybridConfig) -> int:
    return lib().wave_hybrid_weights_bytes(ctypes.byref(cfg))


def hybrid_layer_offset(cfg: WaveHybridConfig, layer: int) -> int:
    return lib().wave_hybrid_layer_offset(ctypes.byref(cfg), layer)
