"""GPU: the library's E4M3 encoder and K/V quantiser against the oracle's,
bit for bit (codes and scales)."""
import numpy as np
import pytest
import torch

import frame_step_decode_gb300 as fsd
import oracle

pytestmark = pytest.mark.gpu


def test_encoder_exhaustive_over_all_fp32_bit_patterns():
    chunk = 1 << 27
    out = torch.empty(chunk, dtype=torch.uint8, device="cuda")
    for c in range((1 << 32) // chunk):
        lo = c * chunk
        bits_h = np.arange(lo, lo + chunk, dtype=np.uint64).astype(np.uint32)
        vals_h = bits_h.view(np.float32)
        vals = torch.from_numpy(vals_h).cuda()
        fsd.fp8_encode(vals, out)
        got = out.cpu().numpy()
        ref = oracle.e4m3_encode(vals_h)
        nan = np.isnan(vals_h)
        assert np.all((got[nan] & 0x7F) == 0x7F), f"chunk {c}: NaN input must give a NaN code"
        bad = np.flatnonzero((got != ref) & ~nan)
        assert bad.size == 0, (f"chunk {c}: {bad.size} mismatches, first input bits "
                               f"{bits_h[bad[0]]:#010x} gpu {got[bad[0]]:#04x} oracle {ref[bad[0]]:#04x}")


@pytest.mark.parametrize("D", [64, 128, 96])
def test_quantiser_matches_oracle_bit_for_bit(D):
    rng = np.random.default_rng(D)
    rows = []
    rows.append(rng.standard_normal((4000, D)).astype(np.float32))
    rows.append((rng.standard_normal((500, D)) * 10.0 ** rng.uniform(-30, 30, (500, 1))).astype(np.float32))
    rows.append(np.zeros((3, D), dtype=np.float32))
    r = np.zeros((4, D), dtype=np.float32)
    r[0, 0] = -0.0
    r[1, :] = -0.0
    r[2, 1] = 1e-45          # scale underflows to 0 -> zero codes
    r[3, :] = 3.0e38         # huge, finite
    rows.append(r)
    dec = oracle.e4m3_decode_all()
    grid = (dec[rng.integers(0, 0x7F, (200, D))] * 0.75).astype(np.float32)
    grid[:, 0] = 448 * 0.75  # exact codes after scaling
    rows.append(grid)
    v = np.concatenate(rows)
    codes_ref, sc_ref = oracle.quantize_rows(v)
    vt = torch.from_numpy(v).cuda()
    codes = torch.empty(v.shape, dtype=torch.uint8, device="cuda")
    sc = torch.empty(v.shape[0], dtype=torch.float32, device="cuda")
    fsd.kv_quantize(vt, codes, sc)
    torch.cuda.synchronize()
    assert np.array_equal(sc.cpu().numpy().view(np.uint32), sc_ref.view(np.uint32))
    assert np.array_equal(codes.cpu().numpy(), codes_ref)


def test_quantiser_rejects_bad_arguments():
    v = torch.zeros((2, 6), device="cuda")
    c = torch.zeros((2, 6), dtype=torch.uint8, device="cuda")
    s = torch.zeros(2, device="cuda")
    with pytest.raises(fsd.WaveError) as e:
        fsd.kv_quantize(v, c, s)
    assert e.value.code == fsd.WAVE_EINVAL
