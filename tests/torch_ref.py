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


def _softplus(v: torch.Tensor) -> torch.Tensor:
    return torch.nn.functional.softplus(v)


def _hybrid_offsets(w):
    """Element offsets of every layer of the hybrid blob and of the tensors
    inside a layer, worked out from the config alone (not from synth's layout
    helpers): a selective-state block is [g d][W_in R*d][W_out d*di][A_log,
    dt_bias, D: 3*Hs, padded up to a multiple of 8]; an attention block is
    [g d][Wqkv 3HD*d][Wo d*HD]; every attn_every-th layer is an attention block."""
    d, Hs = w.d_model, w.ssm_heads
    di = Hs * w.ssm_head_dim
    R = 2 * di + 2 * w.ssm_state + Hs
    HD = w.n_heads * w.head_dim
    small = 3 * Hs
    small += (-small) % 8
    m_size = d + R * d + d * di + small
    a_size = d + 3 * HD * d + d * HD
    starts, o = [], 0
    for l in range(w.n_layers):
        starts.append(o)
        o += a_size if l % w.attn_every == w.attn_every - 1 else m_size
    return starts, dict(R=R, di=di, HD=HD)


def hybrid_step(w, blob: np.ndarray, kv: np.ndarray, sc: np.ndarray, state: np.ndarray, pos: np.ndarray,
                x: np.ndarray):
    """Same contract as oracle.hybrid_step (kv, sc, state updated in place);
    returns y_exact.  Selective-state block: zxbcdt = W_in xn split
    [z | x | B | C | dt]; dt = softplus(dt + dt_bias); a = exp(-exp(A_log) dt);
    h <- a h + dt B x stored in fp32; y = C.h + D x; r += W_out bf16(y silu(z)).
    Attention block: as step() above, without the MLP."""
    d, H, D = w.d_model, w.n_heads, w.head_dim
    Hs, P, N = w.ssm_heads, w.ssm_head_dim, w.ssm_state
    starts, k = _hybrid_offsets(w)
    R, di, HD = k["R"], k["di"], k["HD"]
    Wall = torch.from_numpy(synth.bf16_bits_to_f32(blob).astype(np.float64))
    n = pos.size
    out = np.empty((n, d))
    for j in range(n):
        p0 = int(pos[j])
        r = torch.from_numpy(synth.bf16_bits_to_f32(x[j]).astype(np.float64))
        if p0 < 0:
            out[j] = r.numpy()
            continue
        la = lm = 0
        for l in range(w.n_layers):
            b = starts[l]
            g = Wall[b:b + d]
            xn = _bf16(r / torch.sqrt((r * r).mean() + w.rms_eps) * g)
            if l % w.attn_every == w.attn_every - 1:
                wqkv = Wall[b + d:b + d + 3 * HD * d].view(3 * HD, d)
                wo = Wall[b + d + 3 * HD * d:b + d + 3 * HD * d + d * HD].view(d, HD)
                qkv = wqkv @ xn
                q = _rope(qkv[:HD].view(H, D), p0, w.rope_base)
                kk = _rope(qkv[HD:2 * HD].view(H, D), p0, w.rope_base)
                v = qkv[2 * HD:].view(H, D)
                for which, src in ((0, kk), (1, v)):
                    f = src.to(torch.float32)
                    s32 = f.abs().amax(dim=1) / 448.0
                    codes = (f / s32[:, None]).to(torch.float8_e4m3fn).view(torch.uint8)
                    codes[s32 == 0] = 0
                    kv[la, which, j, :, p0, :] = codes.numpy()
                    sc[la, which, j, :, p0] = s32.numpy()
                att = torch.empty(H, D, dtype=torch.float64)
                for h in range(H):
                    kd = _dec(kv[la, 0, j, h, :p0 + 1])
                    vd = _dec(kv[la, 1, j, h, :p0 + 1])
                    ks = torch.from_numpy(sc[la, 0, j, h, :p0 + 1].astype(np.float64))
                    vs = torch.from_numpy(sc[la, 1, j, h, :p0 + 1].astype(np.float64))
                    pr = torch.softmax((kd @ q[h]) * ks / D ** 0.5, dim=0)
                    att[h] = (pr * vs) @ vd
                r = r + wo @ _bf16(att.reshape(HD))
                la += 1
            else:
                w_in = Wall[b + d:b + d + R * d].view(R, d)
                w_out = Wall[b + d + R * d:b + d + R * d + d * di].view(d, di)
                prm = b + d + R * d + d * di
                a_log, dt_bias, d_skip = Wall[prm:prm + Hs], Wall[prm + Hs:prm + 2 * Hs], Wall[prm + 2 * Hs:prm + 3 * Hs]
                zx = w_in @ xn
                z, xs = zx[:di].view(Hs, P), zx[di:2 * di].view(Hs, P)
                Bv, Cv, dtr = zx[2 * di:2 * di + N], zx[2 * di + N:2 * di + 2 * N], zx[2 * di + 2 * N:]
                dt = _softplus(dtr + dt_bias)                       # [Hs]
                decay = torch.exp(-torch.exp(a_log) * dt)           # [Hs]
                h_old = torch.from_numpy(state[lm, j].astype(np.float64))   # [Hs][P][N]
                h_new = (decay[:, None, None] * h_old
                         + (dt[:, None] * xs)[:, :, None] * Bv[None, None, :]).to(torch.float32)
                state[lm, j] = h_new.numpy()
                yv = h_new.to(torch.float64) @ Cv + d_skip[:, None] * xs          # [Hs][P]
                gated = _bf16((yv * torch.nn.functional.silu(z)).reshape(di))
                r = r + w_out @ gated
                lm += 1
        out[j] = r.numpy()
    return out
