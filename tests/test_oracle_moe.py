"""Pins of the oracle's producer step, the MoE combine + residual add (CPU only).

The step ("nemotron CUDA: RMSNorm rows run on the shared norms and combine
(#548, step 1)", TensorFold pull request #1353, entry tf_nemo_add_moe_norm, and
the author's fix reply, which keeps the routed chain and the shared sum apart):
per hidden lane, an fp32 fma chain over the routed slots taken in index order,
plus the shared slots' own chain, rounded to bf16, added to the bf16 residual
and rounded to bf16.  The pins below do not
restate that formula: hand-worked values (tests/golden/moe_combine_cases.txt,
each derived in the file), bf16 rounding checked by nearest distance in
float64, and sums that are exact in every precision checked against numpy.
"""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "moe_combine_cases.txt")


def _golden_cases():
    cases = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        name, x, sd, slots, weights, routed, want = (f.strip() for f in line.split("|"))
        cases.append((name, int(x, 16), sd, slots, weights, int(routed), int(want, 16)))
    return cases


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c[0])
def test_moe_combine_hand_worked(case):
    name, x, sd, slots, weights, routed, want = case
    vals = [v for v in slots.split(",") if v]
    S = len(vals)
    if sd == "bf16":
        y = np.array([int(v, 16) for v in vals], np.uint16).reshape(1, S, 1)
    else:
        y = np.array([float(v) for v in vals], np.float32).reshape(1, S, 1)
    w = np.array([float(v) for v in weights.split(",") if v], np.float32).reshape(1, S)
    h = oracle.moe_combine(np.array([[x]], np.uint16), y, w, n_routed=routed)
    assert int(h[0, 0]) == want, f"{name}: {int(h[0, 0]):04x} != {want:04x}"


def _bf16_nearest_by_distance(f: float) -> int:
    """bf16 bits nearest to the fp32 value f, ties to the even pattern, by comparing the distances of
    the two bracketing bf16 values in float64 (exact for these magnitudes)."""
    u = int(np.float32(f).view(np.uint32))
    lo = u >> 16
    hi = lo + 1
    vlo = float(np.uint32(lo << 16).view(np.float32))
    vhi = float(np.uint32((hi & 0xFFFF) << 16).view(np.float32))  # the next pattern (inf past the largest)
    d_lo, d_hi = abs(float(np.float32(f)) - vlo), abs(vhi - float(np.float32(f)))
    if d_lo < d_hi:
        return lo
    if d_hi < d_lo:
        return hi & 0xFFFF
    return lo if lo % 2 == 0 else hi & 0xFFFF


def test_bf16_rounding_is_nearest_ties_to_even():
    rng = np.random.default_rng(5)
    vals = list(rng.standard_normal(4000).astype(np.float32))
    vals += list((rng.standard_normal(2000) * np.float32(1e-30)).astype(np.float32))
    # exact midpoints and their neighbours: low 16 bits 0x8000, 0x7fff, 0x8001, odd and even tops
    for top in (0x3F80, 0x3F81, 0xBF80, 0xBF81, 0x0001, 0x7F00):
        for low in (0x7FFF, 0x8000, 0x8001, 0x0000, 0xFFFF):
            vals.append(np.uint32((top << 16) | low).view(np.float32))
    for f in vals:
        assert oracle.f32_to_bf16(float(f)) == _bf16_nearest_by_distance(float(f)), hex(np.float32(f).view(np.uint32))


def _exact_case(seed, sd):
    """Inputs whose combine is exact at every step: integer slots, weights in {-1, 0.5, 1, 2}, small
    integer residuals; every partial sum and the result are bf16-representable."""
    rng = np.random.default_rng(seed)
    B, S, H = 3, 5, 64
    y = rng.integers(-8, 9, size=(B, S, H)).astype(np.float32)
    w = rng.choice(np.array([-1.0, 0.5, 1.0, 2.0], np.float32), size=(B, S))
    x = rng.integers(-16, 17, size=(B, H)).astype(np.float32)
    want = x.astype(np.float64) + np.einsum("bs,bsh->bh", w.astype(np.float64), y.astype(np.float64))
    bits = lambda a: (np.ascontiguousarray(a, np.float32).view(np.uint32) >> 16).astype(np.uint16)
    y_in = bits(y) if sd == "bf16" else y
    return bits(x), y_in, w, bits(want.astype(np.float32))


@pytest.mark.parametrize("sd", ["f32", "bf16"])
def test_moe_combine_exact_sums_match_numpy(sd):
    # exact sums do not depend on how the slots split into routed and shared chains
    for seed in range(4):
        x, y, w, want = _exact_case(seed, sd)
        for n_routed in (None, 0, 2, 5):
            assert np.array_equal(oracle.moe_combine(x, y, w, n_routed=n_routed), want)


def test_moe_combine_without_slots_is_the_residual():
    rng = np.random.default_rng(6)
    x = rng.integers(0, 1 << 16, size=(4, 96), dtype=np.uint16)
    x[(x & 0x7F80) == 0x7F80] = 0x3F80  # no NaN / inf patterns
    h = oracle.moe_combine(x, np.zeros((4, 0, 96), np.float32), np.zeros((4, 0), np.float32))
    # -0 + 0 = +0: the only pattern the add may change
    assert np.array_equal(h, np.where(x == 0x8000, np.uint16(0), x))


def test_moe_combine_rejects_a_routed_count_beyond_the_slots():
    x = np.zeros((1, 8), np.uint16)
    y = np.zeros((1, 2, 8), np.float32)
    w = np.ones((1, 2), np.float32)
    for bad in (-1, 3):
        with pytest.raises(ValueError):
            oracle.moe_combine(x, y, w, n_routed=bad)
