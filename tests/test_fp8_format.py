"""The E4M3 decoding the FP8 tests rely on (torch.float8_e4m3fn -> float64), checked
against the OCP 8-bit floating point specification's definition of E4M3: sign bit,
4 exponent bits with bias 7, 3 mantissa bits; exponent 0 encodes subnormals m * 2^-9; the
all-ones pattern S.1111.111 is NaN and there are no infinities (largest finite 448)."""
import math

import numpy as np
import torch

import gen


def _ocp_e4m3(code: int) -> float:
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return math.nan
    if e == 0:
        return s * m * 2.0 ** -9
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def test_every_e4m3_code_decodes_as_the_format_defines():
    codes = torch.arange(256, dtype=torch.uint8)
    got = gen.to_f64_numpy(codes.view(torch.float8_e4m3fn))
    for c in range(256):
        ref = _ocp_e4m3(c)
        if math.isnan(ref):
            assert math.isnan(got[c]), c
        else:
            assert got[c] == ref, (c, got[c], ref)
    assert np.nanmax(got) == 448.0 and np.nanmin(got) == -448.0


def test_fp8_inputs_are_the_rounded_normals():
    """Every FP8 workload input is the nearest E4M3 value (ties to even) of the same
    standard-normal draw the 16-bit workloads use."""
    w = gen.custom(1, 2, 33, 17, 128, gen.FP8, seed=7)
    q, k, v = gen.make_qkv(w)
    assert q.dtype == torch.float8_e4m3fn
    wf = gen.custom(1, 2, 33, 17, 128, gen.BF16, seed=7)
    rng = np.random.default_rng([7, 0])
    x = rng.standard_normal(size=(1, 2, 33, 128))
    grid = np.array(sorted({_ocp_e4m3(c) for c in range(256) if not math.isnan(_ocp_e4m3(c))}))
    qd = gen.to_f64_numpy(q)
    idx = np.searchsorted(grid, x)
    lo = grid[np.clip(idx - 1, 0, grid.size - 1)]
    hi = grid[np.clip(idx, 0, grid.size - 1)]
    best = np.minimum(np.abs(x - lo), np.abs(x - hi))
    assert np.all(np.abs(qd - x) == best)
    assert wf.io_bytes > w.io_bytes
