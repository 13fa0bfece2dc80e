"""An independent PyTorch (CPU, fp64) restatement of the frame step.

Test-only cross-check of the C oracle's structure (weight offsets, q/k/v and
gate/up row order, slot indexing).  It decodes and encodes FP8 with PyTorch's
float8_e4m3fn type rather than the oracle's codec, and rounds to bf16 through
fp32, so it shares nothing with the oracle but the reading of the step.
"""
import numpy as np
import torch

import synth


def _bf16(t: torch.Tensor) -> torch.Tensor:
    """Single round-to-nearest-even of fp64 to bf16 (normal range), done on
    the fp64 bit pattern: keep 7 of the 52 stored mantissa bits."""
    u = t.detach().numpy().astype(np.float64).view(np.uint64)
    u = (u + np.uint64((1 << 44) - 1) + ((u >> np.uint64(45)) & np.uint64(1))) & ~np.uint64((1 << 45) - 1)
    return torch.from_numpy(u.view(np.float64).copy())


def _dec(codes: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).to(torch.float64)


def _rope(v: torch.Tensor, pos: int, base: float) -> torch.Tensor:
    D = v.shape[-1]
    half = D // 2
    i = torch.arange(half, dtype=torch.float64)
    ang = pos * base ** (-2.0 * i / D)
    c, s = torch.cos(ang), torch.sin(ang)
    a, b = v[..., :half], v[..., half:]
    return torch.cat([a * c - b * s, a * s + b * c], dim=-1)


def step(w, weights: np.ndarray, kv: np.ndarray, sc: np.ndarray, pos: np.ndarray, x: np.ndarray):
    """Same contract as oracle.step (kv, sc updated in place); returns y_exact."""
    L, d, H, D, F = w.n_layers, w.d_model, w.n_heads, w.head_dim, w.ffn
    HD = H * D
    lay = synth.layer_layout(w)
    Wall = torch.from_numpy(synth.bf16_bits_to_f32(weights).astype(np.float64))
    n = pos.size
    out = np.empty((n, d))
    for j in range(n):
        P = int(pos[j])
        r = torch.from_numpy(synth.bf16_bits_to_f32(x[j]).astype(np.float64))
        for l in range(L):
            base = l * lay["layer"]
            g_attn = Wall[base + lay["g_attn"]: base + lay["g_attn"] + d]
            wqkv = Wall[base + lay["wqkv"]: base + lay["wqkv"] + 3 * HD * d].view(3 * HD, d)
            wo = Wall[base + lay["wo"]: base + lay["wo"] + d * HD].view(d, HD)
            g_mlp = Wall[base + lay["g_mlp"]: base + lay["g_mlp"] + d]
            wgu = Wall[base + lay["wgu"]: base + lay["wgu"] + 2 * F * d].view(2 * F, d)
            wdown = Wall[base + lay["wdown"]: base + lay["wdown"] + d * F].view(d, F)

            xn = _bf16(r / torch.sqrt((r * r).mean() + w.rms_eps) * g_attn)
            qkv = wqkv @ xn
            q = _rope(qkv[:HD].view(H, D), P, w.rope_base)
            k = _rope(qkv[HD:2 * HD].view(H, D), P, w.rope_base)
            v = qkv[2 * HD:].view(H, D)
            for which, src in ((0, k), (1, v)):
                f = src.to(torch.float32)
                s32 = f.abs().amax(dim=1) / 448.0
                codes = (f / s32[:, None]).to(torch.float8_e4m3fn).view(torch.uint8)
                codes[s32 == 0] = 0
                kv[l, which, j, :, P, :] = codes.numpy()
                sc[l, which, j, :, P] = s32.numpy()
            att = torch.empty(H, D, dtype=torch.float64)
            for h in range(H):
                kd = _dec(kv[l, 0, j, h, :P + 1])
                vd = _dec(kv[l, 1, j, h, :P + 1])
                ks = torch.from_numpy(sc[l, 0, j, h, :P + 1].astype(np.float64))
                vs = torch.from_numpy(sc[l, 1, j, h, :P + 1].astype(np.float64))
                p = torch.softmax((kd @ q[h]) * ks / D ** 0.5, dim=0)
                att[h] = (p * vs) @ vd
            r = r + wo @ _bf16(att.reshape(HD))
            xn = _bf16(r / torch.sqrt((r * r).mean() + w.rms_eps) * g_mlp)
            gu = wgu @ xn
            u = _bf16(torch.nn.functional.silu(gu[:F]) * gu[F:])
            r = r + wdown @ u
        out[j] = r.numpy()
    return out
