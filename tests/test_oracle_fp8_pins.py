"""Pins of the oracle's e4m3 (FP8) pieces against the format's definition and against the
bf16 routed path, independent of how the oracle implements them.

e4m3 as used by the routed experts' FP8 variant: 1 sign, 4 exponent bits (bias 7), 3
mantissa bits, subnormal step 2^-9, largest finite 448, S.1111.111 = NaN, no infinities;
rounding to nearest with ties to an even mantissa, saturating at 448.  (The pages say only
that SiTU-GLU keeps the activations inside the BF16/FP8 range -- "苏神复盘 Kimi K3",
Stable LatentMoE bullet; the format is the standard OCP FP8 E4M3.)
"""
import numpy as np
import pytest
import torch

FINITE = [c for c in range(256) if (c & 0x7F) != 0x7F]


def _table(oracle_mod):
    return oracle_mod.e4m3_decode(np.arange(256, dtype=np.uint8))


def test_decode_closed_forms(oracle_mod):
    d = _table(oracle_mod)
    assert d[0x00] == 0.0 and np.signbit(d[0x80])
    assert d[0x01] == 2.0 ** -9 and d[0x07] == 7 * 2.0 ** -9      # subnormals
    assert d[0x08] == 2.0 ** -6                                   # smallest normal
    assert d[0x38] == 1.0 and d[0x3C] == 1.5 and d[0x40] == 2.0
    assert d[0x7E] == 448.0 and d[0xFE] == -448.0                 # largest finite
    assert np.isnan(d[0x7F]) and np.isnan(d[0xFF])
    pos = d[[c for c in FINITE if c < 0x80]]
    assert np.all(np.diff(pos) > 0)                               # codes order like values
    assert np.array_equal(d[0x80:0xFF], -d[0x00:0x7F])


def test_encode_round_trips_every_finite_code(oracle_mod):
    d = _table(oracle_mod)
    vals = d[FINITE].astype(np.float32)
    assert np.array_equal(oracle_mod.e4m3_encode(vals), np.array(FINITE, dtype=np.uint8))


def test_ties_go_to_the_even_code(oracle_mod):
    d = _table(oracle_mod)
    pos = [c for c in FINITE if c < 0x7E]
    mids = np.array([(d[c] + d[c + 1]) / 2 for c in pos], dtype=np.float64)
    assert np.all(mids.astype(np.float32) == mids)                # exact in fp32
    got = oracle_mod.e4m3_encode(mids.astype(np.float32))
    want = np.array([c if c % 2 == 0 else c + 1 for c in pos], dtype=np.uint8)
    assert np.array_equal(got, want)
    assert np.array_equal(oracle_mod.e4m3_encode(-mids.astype(np.float32)), want | 0x80)


def test_encode_is_the_nearest_value_by_brute_force(oracle_mod):
    d = _table(oracle_mod)
    codes = np.array(FINITE, dtype=np.int64)
    vals = d[codes]
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.uniform(-460, 460, 20000), rng.uniform(-0.02, 0.02, 20000),
                        rng.standard_normal(20000) * 3.0]).astype(np.float32)
    got = oracle_mod.e4m3_encode(x)
    dist = np.abs(x.astype(np.float64)[:, None] - vals[None, :])
    best = dist.min(axis=1)
    for i in range(len(x)):
        cand = codes[dist[i] == best[i]]
        if x[i] == 0.0:
            continue
        cand = [c for c in cand if (np.signbit(d[c]) == np.signbit(x[i])) or d[c] != 0.0]
        want = [c for c in cand if c % 2 == 0] if len(cand) > 1 else cand
        if abs(x[i]) >= 448.0:
            want = [0x7E | (0x80 if x[i] < 0 else 0)]
        assert got[i] in want, (x[i], got[i], cand)


def test_saturation_and_nan(oracle_mod):
    enc = oracle_mod.e4m3_encode
    big = np.array([448.0, 448.01, 463.9, 464.0, 1e30, np.inf], dtype=np.float32)
    assert np.all(enc(big) == 0x7E) and np.all(enc(-big) == 0xFE)
    assert enc(np.array([np.nan], dtype=np.float32))[0] == 0x7F
    assert enc(np.array([2.0 ** -10], dtype=np.float32))[0] == 0x00  # tie -> even (zero)
    assert enc(np.array([3 * 2.0 ** -10], dtype=np.float32))[0] == 0x02


def test_quantize_rows_scale_and_error_bound(oracle_mod):
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((50, 300)) * rng.uniform(1e-3, 1e3, (50, 1))).astype(np.float32)
    x[3] = 0.0
    q, s = oracle_mod.quantize_rows(x)
    d = oracle_mod.e4m3_decode(q)
    amax = np.abs(x).max(axis=1)
    for r in range(len(x)):
        if amax[r] == 0:
            assert s[r] == 1.0 and np.all(q[r] == 0)
            continue
        assert s[r] == np.float32(amax[r] / np.float32(448.0))
        assert np.abs(d[r]).max() == 448.0              # the largest element maps to +-448
        xs = x[r].astype(np.float64) / np.float64(s[r])
        # half the e4m3 spacing at each value (2^-10 below the normal range)
        e = np.floor(np.log2(np.maximum(np.abs(xs), 2.0 ** -6)))
        half = np.where(np.abs(xs) < 2.0 ** -6, 2.0 ** -10, 2.0 ** (e - 4))
        assert np.all(np.abs(xs - d[r]) <= half * (1 + 1e-6) + 448 * 2.0 ** -24)


def test_bf16_round_is_nearest_even(oracle_mod):
    rng = np.random.default_rng(2)
    x = np.concatenate([rng.standard_normal(3000) * 10.0 ** rng.integers(-8, 8, 3000),
                        [1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8]])
    r = oracle_mod.bf16_round(x).astype(np.float64)
    for xi, ri in zip(x, r):
        e = np.floor(np.log2(abs(xi)))
        ulp = 2.0 ** (e - 7)
        assert abs(xi - ri) <= ulp / 2
        if abs(xi - ri) == ulp / 2:                       # tie: even last mantissa bit
            assert int(np.float32(ri).view(np.uint32) >> 16) % 2 == 0
    assert r[-2] == 1.0 and r[-1] == 1 + 2 * 2.0 ** -7


def _bf16(a):
    return torch.tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)


def _exact_rows(rng, rows, cols, scale_exp):
    """Rows of e4m3 values times 2^scale_exp whose largest magnitude is 448 * 2^scale_exp,
    so that per-row quantisation is exact."""
    codes = rng.choice(FINITE, size=(rows, cols))
    from oracle import e4m3_decode
    vals = e4m3_decode(codes.astype(np.uint8)) * 2.0 ** scale_exp
    vals[:, 0] = 448.0 * 2.0 ** scale_exp * np.where(rng.random(rows) < 0.5, 1, -1)
    return vals


def test_routed_fp8_is_lossless_on_representable_inputs(oracle_mod):
    """Latent and weights built from e4m3 values with a 448 * 2^k maximum per row, and I = 1
    (one SiTU output per pair, quantised to +-448 * its scale): every quantisation is exact
    up to the fp32 rounding of the scale, so the FP8 path must give the bf16 path's result
    with h rounded to bf16.  A dropped or misapplied scale, a wrong weight row or a wrong
    operand would move the result by O(1)."""
    rng = np.random.default_rng(3)
    n, L, E, K, I = 12, 64, 5, 2, 1
    lat = _exact_rows(rng, n, L, -8)
    wg = _exact_rows(rng, E * I, L, -9).reshape(E, I, L)
    wv = _exact_rows(rng, E * I, L, -10).reshape(E, I, L)
    wd = (rng.choice([-1, 1], (E, L, I)) * 2.0 ** rng.integers(-6, 2, (E, L, I)))
    idx = np.stack([rng.choice(E, K, replace=False) for _ in range(n)]).astype(np.int32)
    gate = rng.uniform(0.1, 1.0, (n, K)).astype(np.float32)
    gamma = rng.uniform(0.5, 1.5, L).astype(np.float32)
    w = {"w_gate": _bf16(wg), "w_value": _bf16(wv), "w_edown": _bf16(wd)}
    assert np.array_equal(w["w_gate"].float().numpy(), wg.astype(np.float32))
    wq = oracle_mod.quantize_expert_weights(w["w_gate"], w["w_value"], w["w_edown"])
    z8 = oracle_mod.routed_fp8(lat, idx, gate, wq, gamma, c=100.0, eps=1e-6)
    z = oracle_mod.routed(lat, idx, gate, w["w_gate"], w["w_value"], w["w_edown"], gamma,
                          c=100.0, eps=1e-6)
    rms = np.sqrt(np.mean(z * z))
    # only the bf16 rounding of h (relative 2^-9) and the scales' fp32 rounding remain
    assert np.max(np.abs(z8 - z)) <= 2.0 ** -8 * np.max(np.abs(z)) + 1e-12 * rms
    assert not np.array_equal(z8, z) or np.all(z == 0)


def test_routed_fp8_error_is_that_of_a_3_bit_mantissa(oracle_mod):
    """On generic inputs the FP8 path differs from the bf16 path by the e4m3 rounding of
    every operand: clearly non-zero, and well below the output scale."""
    from latent_compressed_expert_gb300 import synth
    sh = synth.TINY
    w = synth.make_weights(sh, seed=5)
    x = synth.make_x(sh, seed=5)
    r16 = oracle_mod.forward(w, x, sh.K, residual=None)
    r8 = oracle_mod.forward(w, x, sh.K, residual=None, expert_fp8=True)
    assert np.array_equal(r16.idx, r8.idx)             # routing is not quantised
    rel = np.sqrt(np.mean((r8.z - r16.z) ** 2)) / np.sqrt(np.mean(r16.z ** 2))
    assert 1e-3 < rel < 0.1, rel


def test_bf16_tie_distance(oracle_mod):
    d = oracle_mod.bf16_tie_distance(np.array([1.0, 1.0 + 2.0 ** -8, -(1.0 + 2.0 ** -8),
                                               1.75 + 2.0 ** -8, 3.0 + 2.0 ** -7]))
    assert d[0] == pytest.approx(2.0 ** -8)          # a bf16 value: half a spacing away
    assert d[1] == 0.0 and d[2] == 0.0 and d[3] == 0.0 and d[4] == 0.0   # exact ties


def test_routed_fp8_flags_scales_set_at_a_near_tie(oracle_mod):
    """A token whose latent amax sits on a bf16 rounding tie is flagged; the others are
    not (their rows are exact e4m3 multiples of a power of two, far from any tie)."""
    rng = np.random.default_rng(6)
    n, L, E, K, I = 6, 64, 4, 2, 1
    lat = _exact_rows(rng, n, L, -8)
    lat[2, 0] = 1.75 + 2.0 ** -8                    # amax at the midpoint of two bf16 values
    wg = _exact_rows(rng, E * I, L, -9).reshape(E, I, L)
    wv = _exact_rows(rng, E * I, L, -10).reshape(E, I, L)
    wd = np.ones((E, L, I))
    idx = np.stack([rng.choice(E, K, replace=False) for _ in range(n)]).astype(np.int32)
    gate = np.full((n, K), 0.5, dtype=np.float32)
    wq = oracle_mod.quantize_expert_weights(_bf16(wg), _bf16(wv), _bf16(wd))
    _, ties = oracle_mod.routed_fp8(lat, idx, gate, wq, np.ones(L, np.float32),
                                    return_ties=True)
    assert ties.tolist() == [0, 0, 1, 0, 0, 0]
