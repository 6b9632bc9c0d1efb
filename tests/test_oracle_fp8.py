"""Pins of the oracle's 8-bit KV cache pieces (no GPU).

The page on KV cache quantization (P3 §6.2, 量化与压缩的协同优化) names no
format; the oracle reads it as OCP FP8 E4M3 with a per-KV-head scale.  These
pins hold the oracle to that format's definition (hand-derived codes), to a
library routine (torch's float8_e4m3fn cast), and to the unquantized
attention reference on values both formats represent exactly.
"""
import numpy as np
import pytest
import torch

import oracle
from workloads import F16, f32_to_bits


def bits(x, dtype=F16):
    return f32_to_bits(np.asarray(x, dtype=np.float32), dtype)


# ---------------------------------------------------------------- the format
def check_e4m3_known_codes():
    """Codes whose values follow from the definition: bias 7, 3 mantissa bits,
    subnormals at exponent 0, S.1111.111 the only NaN, 448 the largest finite."""
    v = oracle.e4m3_value(np.array([0x00, 0x01, 0x07, 0x08, 0x30, 0x38, 0x3C, 0x78, 0x7E, 0x80, 0xB8, 0xFE],
                                   dtype=np.uint8))
    want = [0.0, 2.0 ** -9, 7 * 2.0 ** -9, 2.0 ** -6, 0.5, 1.0, 1.5, 256.0, 448.0, -0.0, -1.0, -448.0]
    assert v.tolist() == want
    assert np.signbit(v[9])
    nan = oracle.e4m3_value(np.array([0x7F, 0xFF], dtype=np.uint8))
    assert np.isnan(nan).all()
    finite = oracle.e4m3_value(np.arange(0x7F, dtype=np.uint8))
    assert np.all(np.diff(finite) > 0)                        # codes 0x00..0x7E increase
    assert np.isfinite(oracle.e4m3_value(np.arange(256, dtype=np.uint8))).sum() == 254


def check_e4m3_quantize_rules():
    """Exact values keep their code; halfway points go to the even code;
    magnitudes above 448 saturate; NaN is 0x7F; the sign survives underflow."""
    codes = np.arange(0x7F, dtype=np.uint8)
    vals = oracle.e4m3_value(codes)
    assert np.array_equal(oracle.e4m3_quantize(vals.astype(np.float32)), codes)
    assert np.array_equal(oracle.e4m3_quantize(-vals.astype(np.float32)), codes | 0x80)
    mids = (vals[:-1] + vals[1:]) / 2                        # exactly representable in float32
    got = oracle.e4m3_quantize(mids.astype(np.float32))
    lo = codes[:-1]
    assert np.array_equal(got, np.where(lo % 2 == 0, lo, lo + 1))
    assert oracle.e4m3_quantize(np.array([449.0, 1e6, np.inf, -500.0], np.float32)).tolist() == [0x7E, 0x7E, 0x7E, 0xFE]
    assert oracle.e4m3_quantize(np.array([np.nan], np.float32)).tolist() == [0x7F]
    assert oracle.e4m3_quantize(np.array([-1e-9, 1e-9], np.float32)).tolist() == [0x80, 0x00]


def check_e4m3_quantize_matches_torch_cast():
    """In range, the oracle's rounding is the library cast's (torch float8_e4m3fn)."""
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(20000) * 40, rng.standard_normal(20000) * 0.01]).astype(np.float32)
    x = x[np.abs(x) < 448]
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_quantize(x), want)


def check_append_fp8_worked_example():
    """k = (1, 3, -0.1, 500) at scale 2: 0.5 -> 0x30; 1.5 -> 0x3C; -0.05 lies between
    1.5*2^-5 and 1.625*2^-5, nearer the second -> 0x95; 250 lies between 240 and 256,
    nearer 256 -> 0x78.  V at scale 0.5: 0.25 -> 0x28, 3 -> 0x44."""
    kc = np.zeros((2, 4, 1, 4), np.uint8)
    vc = np.zeros_like(kc)
    k = bits([[[1.0, 3.0, -0.1, 500.0]]])
    v = bits([[[0.125, 1.5, 0.0, -0.0]]])
    oracle.append_fp8_ref(kc, vc, k, v, np.array([6]), np.array([2.0], np.float32), np.array([0.5], np.float32), F16)
    assert kc[1, 2, 0].tolist() == [0x30, 0x3C, 0x95, 0x78]
    assert vc[1, 2, 0].tolist() == [0x28, 0x44, 0x00, 0x80]
    assert not kc[0].any() and not kc[1, [0, 1, 3]].any()


def check_fp8_attention_is_attention_on_dequantized_values():
    """Every E4M3 value times a power-of-two scale is exact in fp16, so attention
    over the codes equals the unquantized reference over those fp16 values."""
    rng = np.random.default_rng(4)
    NB, bs, Hkv, d, Hq = 9, 4, 2, 8, 4
    kcode = rng.integers(0x20, 0x50, size=(NB, bs, Hkv, d)).astype(np.uint8) | (rng.integers(0, 2, (NB, bs, Hkv, d)) << 7).astype(np.uint8)
    vcode = rng.integers(0x20, 0x50, size=(NB, bs, Hkv, d)).astype(np.uint8)
    ks = np.array([0.25, 2.0], np.float32)
    vs = np.array([4.0, 0.5], np.float32)
    kf = oracle.e4m3_value(kcode) * ks[None, None, :, None]
    vf = oracle.e4m3_value(vcode) * vs[None, None, :, None]
    tables = np.array([[3, 1, 7], [0, 5, 2]], np.int32)
    lens = np.array([11, 6])
    q = bits(rng.standard_normal((2, Hq, d)))
    got = oracle.attention_fp8_ref(q, kcode, vcode, tables, lens, 0.3, Hkv, F16, ks, vs)
    want = oracle.attention_ref(q, bits(kf), bits(vf), tables, lens, 0.3, Hkv, F16)
    assert np.allclose(got, want, rtol=0, atol=1e-12)


def check_fp8_scales_act_where_stated():
    """Doubling k_scale doubles every score (same as doubling the softmax scale);
    halving v_scale halves the output."""
    rng = np.random.default_rng(5)
    kcode = rng.integers(0x28, 0x48, size=(4, 4, 1, 8)).astype(np.uint8)
    vcode = rng.integers(0x28, 0x48, size=(4, 4, 1, 8)).astype(np.uint8)
    tables = np.array([[2, 0, 3]], np.int32)
    lens = np.array([10])
    q = bits(rng.standard_normal((1, 2, 8)))
    one = np.array([1.0], np.float32)
    base = oracle.attention_fp8_ref(q, kcode, vcode, tables, lens, 0.2, 1, F16, one, one)
    k2 = oracle.attention_fp8_ref(q, kcode, vcode, tables, lens, 0.2, 1, F16, 2 * one, one)
    s2 = oracle.attention_fp8_ref(q, kcode, vcode, tables, lens, 0.4, 1, F16, one, one)
    vh = oracle.attention_fp8_ref(q, kcode, vcode, tables, lens, 0.2, 1, F16, one, 0.5 * one)
    assert np.allclose(k2, s2, atol=1e-12) and not np.allclose(k2, base)
    assert np.allclose(vh, base / 2, atol=1e-12)


def check_fp8_verify_is_verify_on_dequantized_values():
    """Verify (several causal query tokens) over the codes equals the unquantized
    verify reference over the same values held exactly in fp16, token by token."""
    rng = np.random.default_rng(6)
    NB, bs, Hkv, d, Hq, nq = 10, 4, 2, 8, 6, 3
    kcode = rng.integers(0x20, 0x50, size=(NB, bs, Hkv, d)).astype(np.uint8) | (rng.integers(0, 2, (NB, bs, Hkv, d)) << 7).astype(np.uint8)
    vcode = rng.integers(0x20, 0x50, size=(NB, bs, Hkv, d)).astype(np.uint8)
    ks = np.array([0.5, 4.0], np.float32)
    vs = np.array([2.0, 0.25], np.float32)
    kf = oracle.e4m3_value(kcode) * ks[None, None, :, None]
    vf = oracle.e4m3_value(vcode) * vs[None, None, :, None]
    tables = np.array([[6, 1, 9], [0, 5, 2], [4, 8, 3]], np.int32)
    lens = np.array([11, 3, 2])                     # the last: fewer positions than query tokens
    q = bits(rng.standard_normal((3, nq, Hq, d)))
    got = oracle.verify_attention_fp8_ref(q, kcode, vcode, tables, lens, 0.3, Hkv, F16, ks, vs)
    want = oracle.verify_attention_ref(q, bits(kf), bits(vf), tables, lens, 0.3, Hkv, F16)
    assert np.allclose(got, want, rtol=0, atol=1e-12)
    assert not got[2, 0].any()                      # query 0 of a 2-position sequence with 3 queries sees nothing


def check_fp8_verify_one_query_is_decode():
    """One query token per sequence: the single-query E4M3 reference."""
    rng = np.random.default_rng(7)
    kcode = rng.integers(0x28, 0x48, size=(6, 4, 1, 8)).astype(np.uint8)
    vcode = rng.integers(0x28, 0x48, size=(6, 4, 1, 8)).astype(np.uint8)
    tables = np.array([[2, 0, 3], [5, 4, 1]], np.int32)
    lens = np.array([10, 7])
    q = bits(rng.standard_normal((2, 1, 2, 8)))
    one = np.array([1.5], np.float32)
    got = oracle.verify_attention_fp8_ref(q, kcode, vcode, tables, lens, 0.2, 1, F16, one, one)
    want = oracle.attention_fp8_ref(q[:, 0], kcode, vcode, tables, lens, 0.2, 1, F16, one, one)
    assert np.array_equal(got[:, 0], want)


FP8_PINS = [check_e4m3_known_codes, check_e4m3_quantize_rules, check_e4m3_quantize_matches_torch_cast,
            check_append_fp8_worked_example, check_fp8_attention_is_attention_on_dequantized_values,
            check_fp8_scales_act_where_stated, check_fp8_verify_is_verify_on_dequantized_values,
            check_fp8_verify_one_query_is_decode]


@pytest.mark.parametrize("pin", FP8_PINS, ids=lambda f: f.__name__)
def test_fp8_pin(pin):
    pin()


# ---------------------------------------------------------------- planted mistakes
def _value_bias_8(codes):
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    e, m = (c >> 3) & 0xF, (c & 7).astype(np.float64)
    mag = np.where(e == 0, m / 8 * 2.0 ** -7, (1 + m / 8) * np.exp2(e - 8.0))
    return np.where(c >> 7, -mag, mag)


def _quantize_ties_up(x):
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    a = np.abs(x)
    grid = oracle.e4m3_value(np.arange(0x7F, dtype=np.uint8))
    hi = np.clip(np.searchsorted(grid, a, side="left"), 1, 0x7E)
    lo = hi - 1
    code = np.where(a - grid[lo] < grid[hi] - a, lo, hi)
    code = np.where(a >= 448, 0x7E, np.where(a == 0, 0, code)) | np.where(np.signbit(x), 0x80, 0)
    return np.where(np.isnan(x), 0x7F, code).astype(np.uint8)


def _quantize_truncates(x):
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    a = np.abs(x)
    grid = oracle.e4m3_value(np.arange(0x7F, dtype=np.uint8))
    code = np.clip(np.searchsorted(grid, a, side="right") - 1, 0, 0x7E)
    code = code | np.where(np.signbit(x), 0x80, 0)
    return np.where(np.isnan(x), 0x7F, code).astype(np.uint8)


_ATTENTION_FP8 = oracle.attention_fp8_ref


def _attention_fp8_no_v_scale(q, kc, vc, tables, lens, scale, Hkv, q_dtype, ks, vs):
    return _ATTENTION_FP8(q, kc, vc, tables, lens, scale, Hkv, q_dtype, ks, np.ones_like(np.asarray(vs, np.float32)))


def _attention_fp8_k_scale_per_query_head(q, kc, vc, tables, lens, scale, Hkv, q_dtype, ks, vs):
    B, Hq, d = q.shape
    G = Hq // Hkv
    out = np.zeros((B, Hq, d))
    for s in range(B):
        for h in range(Hq):
            g = h // G
            K = oracle.gather_sequence(kc, tables[s], int(lens[s]), g, oracle.E4M3) * float(ks[h % len(ks)])
            V = oracle.gather_sequence(vc, tables[s], int(lens[s]), g, oracle.E4M3) * float(vs[g])
            out[s, h] = oracle.softmax_attention(oracle.decode_bits(q[s, h], q_dtype), K, V, scale)
    return out


def _verify_fp8_with(limit=lambda L, nq, i: L - nq + i + 1, k_scale_of=lambda ks, h, g: ks[g],
                     v_scale_of=lambda vs, g: vs[g]):
    """verify_attention_fp8_ref with the causal limit and the scale lookups as parameters."""
    def run(q, kc, vc, tables, lens, scale, Hkv, q_dtype, ks, vs):
        B, nq, Hq, d = q.shape
        G = Hq // Hkv
        ks = np.asarray(ks, np.float32).astype(np.float64)
        vs = np.asarray(vs, np.float32).astype(np.float64)
        out = np.zeros((B, nq, Hq, d))
        for s in range(B):
            L = int(lens[s])
            for h in range(Hq):
                g = h // G
                K = oracle.gather_sequence(kc, tables[s], L, g, oracle.E4M3) * k_scale_of(ks, h, g)
                V = oracle.gather_sequence(vc, tables[s], L, g, oracle.E4M3) * v_scale_of(vs, g)
                for i in range(nq):
                    vis = min(L, limit(L, nq, i))
                    if L <= 0 or vis <= 0:
                        continue
                    out[s, i, h] = oracle.softmax_attention(oracle.decode_bits(q[s, i, h], q_dtype), K[:vis],
                                                            V[:vis], scale)
        return out
    return run


def _verify_fp8_no_v_scale(*a):
    return _verify_fp8_with(v_scale_of=lambda vs, g: 1.0)(*a)


def _verify_fp8_k_scale_per_query_head(*a):
    return _verify_fp8_with(k_scale_of=lambda ks, h, g: ks[h % len(ks)])(*a)


def _verify_fp8_excludes_itself(*a):
    return _verify_fp8_with(limit=lambda L, nq, i: L - nq + i)(*a)


def test_verify_fp8_mutant_scaffold_unmutated_passes_every_pin(monkeypatch):
    """The verify mutants' scaffold with the right limit and scales passes every pin."""
    monkeypatch.setattr(oracle, "verify_attention_fp8_ref", _verify_fp8_with())
    for pin in FP8_PINS:
        pin()


MUTANTS = [("e4m3_value", _value_bias_8), ("e4m3_quantize", _quantize_ties_up),
           ("e4m3_quantize", _quantize_truncates), ("attention_fp8_ref", _attention_fp8_no_v_scale),
           ("attention_fp8_ref", _attention_fp8_k_scale_per_query_head),
           ("verify_attention_fp8_ref", _verify_fp8_no_v_scale),
           ("verify_attention_fp8_ref", _verify_fp8_k_scale_per_query_head),
           ("verify_attention_fp8_ref", _verify_fp8_excludes_itself)]


@pytest.mark.parametrize("name,mutant", MUTANTS, ids=lambda x: getattr(x, "__name__", x))
def test_planted_fp8_mistakes_are_caught(monkeypatch, name, mutant):
    monkeypatch.setattr(oracle, name, mutant)
    failed = []
    for pin in FP8_PINS:
        try:
            with np.errstate(all="ignore"):
                pin()
        except (AssertionError, ValueError, IndexError, FloatingPointError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake {mutant.__name__}"
