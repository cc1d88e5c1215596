"""The chunked prefills floor each token's log decay before the cumulative sum
(a zero-decay token would otherwise make a difference -inf - (-inf)).  The
floor must give a decay of exactly 0 in fp32 through both exponentials the
kernels use (expf, and 2^x on ex2.approx.ftz, which flushes subnormal results),
so that it changes no decay, and must stay small enough that cumulative sums
after a floored token keep fine fp32 resolution.  This pins the constant the
kernels are built with (CPU only)."""
import os
import re

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "hybrid_linear_attention_gdn_gb300", "csrc", "gdn_common.cuh")


def _floor():
    src = open(HEADER).read()
    m = re.search(r"constexpr float kLogDecayFloor = (-?[0-9.]+)f;", src)
    assert m, "kLogDecayFloor not found"
    # the floor is applied with a comparison that lets NaN through
    assert "return g < kLogDecayFloor ? kLogDecayFloor : g;" in src
    return float(m.group(1))


def test_floor_decays_to_exact_zero_in_fp32():
    f = np.float32(_floor())
    with np.errstate(under="ignore"):
        assert np.exp(f, dtype=np.float32) == 0.0
        # ex2.approx.ftz: 2^(x log2 e); results below the smallest normal flush to 0
        y = np.float32(2.0) ** (f * np.float32(1.4426950408889634))
    assert y < np.finfo(np.float32).tiny


def test_floor_changes_no_finite_decay_that_is_not_already_zero():
    # every log decay between the floor and the largest one whose fp32
    # exponential underflows to 0 already decays to exactly 0
    f = _floor()
    with np.errstate(under="ignore"):
        for g in np.linspace(f, -104.0, 200, dtype=np.float32):
            assert np.exp(g, dtype=np.float32) == 0.0


def test_floor_keeps_cumulative_sums_fine():
    # 64 floored tokens in one chunk: differences of later cumulative sums
    # still resolve 1e-4 relative decay changes
    f = _floor()
    assert -200.0 <= f <= -104.0
    assert np.spacing(np.float32(64 * f)) < 1e-3
