"""Pins for the oracle's FP8 (E4M3) cache: what the format and the mathematics fix.

The pages say only that an FP8 cache halves the bytes per block and that
nothing else about paging changes ("PagedAttention: paging the KV cache",
Fine-tuned models and adapters). The oracle reads that as OCP E4M3 codes with
one float scale per layer for K and for V. These tests pin that reading to
things other than the oracle: torch's own float8_e4m3fn type, closed-form
values of the format, the ties-to-even rule, saturation, the error bound of
one rounding, reduction to the already pinned fp16 path, and the scale
identities.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from workloads import make_random_case
from workloads.configs import FP8_K_SCALE, FP8_V_SCALE, to_bits


def _torch_codes(x32: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32)).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy()


# ----------------------------------------------------------------------------
# the code -> value map


def test_decode_all_codes_match_torch():
    """Every one of the 256 codes widens to torch's float8_e4m3fn value."""
    codes = np.arange(256, dtype=np.uint8)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    got = oracle.e4m3_to_f64(codes)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(want[ok]))


@pytest.mark.parametrize("code,value", [
    (0x00, 0.0), (0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9), (0x08, 2.0 ** -6),
    (0x38, 1.0), (0x39, 1.125), (0x40, 2.0), (0x77, 240.0), (0x7E, 448.0),
    (0xB8, -1.0), (0xFE, -448.0),
])
def test_decode_closed_form_values(code, value):
    """Values fixed by the format: bias 7, three mantissa bits, subnormals
    m * 2^-9, largest finite 1.75 * 2^8 = 448."""
    assert oracle.e4m3_to_f64(np.array([code], dtype=np.uint8))[0] == value


def test_nan_and_negative_zero():
    got = oracle.e4m3_to_f64(np.array([0x7F, 0xFF, 0x80], dtype=np.uint8))
    assert math.isnan(got[0]) and math.isnan(got[1])
    assert got[2] == 0.0 and np.signbit(got[2])


# ----------------------------------------------------------------------------
# the value -> code map (round to nearest even, saturate)


def test_every_finite_code_round_trips():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = oracle.e4m3_to_f64(codes).astype(np.float32)
    assert np.array_equal(oracle.f32_to_e4m3(vals), codes)


def test_encode_matches_torch_in_range():
    """Inside the range torch also converts without overflow (|x| < 464, the
    midpoint between 448 and the next binade step), both round to nearest
    with ties to even, so the codes agree bit for bit."""
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.standard_normal(50000).astype(np.float32) * 60.0,
        rng.standard_normal(20000).astype(np.float32) * 0.01,   # subnormal range
        np.float32(2.0) ** rng.integers(-12, 9, 20000).astype(np.float32)
        * rng.uniform(1.0, 2.0, 20000).astype(np.float32),
    ])
    # every midpoint between adjacent codes, and one float32 step either side
    grid = oracle.e4m3_to_f64(np.arange(0x7F, dtype=np.uint8))
    mids = ((grid[:-1] + grid[1:]) / 2).astype(np.float32)
    x = np.concatenate([x, mids, np.nextafter(mids, np.float32(0)),
                        np.nextafter(mids, np.float32(1000)), -mids])
    x = x[np.abs(x) < 464.0].astype(np.float32)
    assert np.array_equal(oracle.f32_to_e4m3(x), _torch_codes(x))


@pytest.mark.parametrize("x,code", [
    (1.0625, 0x38),        # halfway 1.0 (0x38) / 1.125 (0x39): even code 0x38
    (1.1875, 0x3A),        # halfway 1.125 (0x39) / 1.25 (0x3A): even code 0x3A
    (2.0 ** -10, 0x00),    # halfway 0 / 2^-9: even code 0
    (3 * 2.0 ** -10, 0x02),  # halfway 2^-9 / 2^-8: even code 0x02
    (-1.0625, 0xB8),
    (-1e-30, 0x80),        # rounds to zero, keeps its sign
])
def test_ties_to_even(x, code):
    assert int(oracle.f32_to_e4m3(np.array([x], dtype=np.float32))[0]) == code


@pytest.mark.parametrize("x,code", [(448.0, 0x7E), (449.0, 0x7E), (464.0, 0x7E), (1e30, 0x7E),
                                    (np.inf, 0x7E), (-500.0, 0xFE), (-np.inf, 0xFE)])
def test_saturation(x, code):
    """Magnitudes past the largest finite code clamp to +-448."""
    assert int(oracle.f32_to_e4m3(np.array([x], dtype=np.float32))[0]) == code


def test_nan_encodes_to_nan():
    c = oracle.f32_to_e4m3(np.array([np.nan], dtype=np.float32))
    assert math.isnan(oracle.e4m3_to_f64(c)[0])


def test_one_rounding_error_bound():
    """|value(e4m3(x)) - x| is at most half a code step: 2^(e-4) in binade
    [2^e, 2^(e+1)) for e >= -6, 2^-10 in the subnormal range."""
    rng = np.random.default_rng(11)
    x = (rng.standard_normal(200000) * rng.choice([0.003, 0.3, 30.0], 200000)).astype(np.float32)
    x = x[np.abs(x) <= 448.0]
    err = np.abs(oracle.e4m3_to_f64(oracle.f32_to_e4m3(x)) - x.astype(np.float64))
    ax = np.abs(x.astype(np.float64))
    e = np.floor(np.log2(np.maximum(ax, 2.0 ** -6)))
    bound = np.where(ax < 2.0 ** -6, 2.0 ** -10, 2.0 ** (e - 4))
    assert np.all(err <= bound)


# ----------------------------------------------------------------------------
# quantised writes


def test_quantize_divides_by_the_scale():
    """x = 1.0 with scale 0.5 stores value 2.0 (code 0x40); with scale 4 it
    stores 0.25 (code 0x28)."""
    one = to_bits(np.array([1.0], dtype=np.float32), "f16")
    assert int(oracle.quantize_e4m3(one, "f16", 0.5)[0]) == 0x40
    assert int(oracle.quantize_e4m3(one, "f16", 4.0)[0]) == 0x28


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_quantize_is_a_true_division(dtype):
    """x = 203 * 2^-14 and s = 7 * 2^-10 are exact in both input formats and
    x / s = 1.8125 exactly: the midpoint of 1.75 (code 0x3E) and 1.875 (0x3F),
    so ties-to-even stores 0x3E. Multiplying by the float32-rounded reciprocal
    of s instead lands one float32 step above the midpoint, on 0x3F."""
    x = to_bits(np.array([203.0 / 16384.0], dtype=np.float32), dtype)
    assert oracle.bits_to_f64(x, dtype)[0] == 203.0 / 16384.0
    assert int(oracle.quantize_e4m3(x, dtype, 7.0 / 1024.0)[0]) == 0x3E


def test_quantize_rounds_the_float32_quotient():
    """The code is decided on x / s rounded once to float32 (the precision the
    device divides in), not on the exact real quotient: for inputs whose exact
    quotient sits within one float32 step of a code midpoint the two can
    differ, and the oracle must follow the float32 one."""
    rng = np.random.default_rng(3)
    s = np.float32(FP8_K_SCALE)
    x = rng.standard_normal(400000).astype(np.float32)
    bits = to_bits(x, "bf16")
    xb = oracle.bits_to_f64(bits, "bf16")
    q32 = (xb.astype(np.float32) / s)
    assert np.array_equal(oracle.quantize_e4m3(bits, "bf16", float(s)), _torch_codes(
        np.clip(q32, -448, 448)))


def test_write_e4m3_scatters_quantised_rows():
    """write_kv_e4m3 equals write_kv of the quantised rows; other slots keep
    their bytes."""
    rng = np.random.default_rng(5)
    k = rng.integers(0, 256, size=(6, 4, 2, 16), dtype=np.uint8)
    v = rng.integers(0, 256, size=(6, 4, 2, 16), dtype=np.uint8)
    key = to_bits(rng.standard_normal((3, 2, 16)).astype(np.float32), "f16")
    val = to_bits(rng.standard_normal((3, 2, 16)).astype(np.float32), "f16")
    slots = [5, -1, 17]
    k2, v2 = oracle.write_kv_e4m3(k, v, key, val, slots, "f16", 0.01, 0.02)
    assert np.array_equal(k2[1, 1], _torch_codes(oracle.bits_to_f64(key[0], "f16").astype(np.float32)
                                                 / np.float32(0.01)))
    assert np.array_equal(v2[4, 1], _torch_codes(oracle.bits_to_f64(val[2], "f16").astype(np.float32)
                                                 / np.float32(0.02)))
    mask = np.ones(k.shape[:2], dtype=bool)
    mask[1, 1] = mask[4, 1] = False
    assert np.array_equal(k2[mask], k[mask]) and np.array_equal(v2[mask], v[mask])


# ----------------------------------------------------------------------------
# attention over an E4M3 cache


def _fp8_case(seed=21, **kw):
    args = dict(num_seqs=3, num_q_heads=8, num_kv_heads=2, head_dim=32, block_size=4,
                seq_lens=[1, 9, 30], dtype="f16", kv_dtype="e4m3")
    args.update(kw)
    return make_random_case(seed, **args)


def test_unit_scale_reduces_to_the_fp16_path():
    """Every E4M3 value is exact in fp16, so with unit scales an E4M3 cache and
    the fp16 cache of the same values give identical outputs."""
    w = _fp8_case()
    def as_f16(c):
        return to_bits(oracle.e4m3_to_f64(c).astype(np.float32), "f16")

    got = oracle.decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.scale, "f16",
                        kv_dtype="e4m3", k_scale=1.0, v_scale=1.0)
    want = oracle.decode(w.q, as_f16(w.k_cache), as_f16(w.v_cache), w.block_tables, w.seq_lens,
                         w.scale, "f16")
    assert np.array_equal(got, want)


def test_k_scale_multiplies_the_logits():
    """k_scale * c and softmax scale s act only through their product."""
    w = _fp8_case(seed=22)
    a = oracle.decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.scale * 0.25,
                      "f16", kv_dtype="e4m3", k_scale=4.0, v_scale=w.v_scale)
    b = oracle.decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.scale, "f16",
                      kv_dtype="e4m3", k_scale=1.0, v_scale=w.v_scale)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


def test_v_scale_scales_the_output_linearly():
    w = _fp8_case(seed=23)
    a = oracle.decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.scale, "f16",
                      kv_dtype="e4m3", k_scale=w.k_scale, v_scale=2.0)
    b = oracle.decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.scale, "f16",
                      kv_dtype="e4m3", k_scale=w.k_scale, v_scale=0.5)
    np.testing.assert_allclose(a, 4.0 * b, rtol=1e-13, atol=1e-13)


def test_identity_table_matches_torch_sdpa():
    """Contiguous placement: the oracle equals torch's scaled_dot_product_attention
    in fp64 on torch's own float8_e4m3fn widening of the codes, times the scales."""
    w = _fp8_case(seed=24, block_size=8, seq_lens=[37], num_seqs=1, pool_factor=1.0)
    L = int(w.seq_lens[0])
    table = w.block_tables[0][: -(-L // w.block_size)]
    ident = np.arange(len(table), dtype=np.int32)[None]
    k = w.k_cache[table]
    v = w.v_cache[table]
    got = oracle.decode(w.q, k, v, ident, w.seq_lens, w.scale, "f16", kv_dtype="e4m3",
                        k_scale=w.k_scale, v_scale=w.v_scale)
    kt = torch.from_numpy(k.reshape(-1, w.num_kv_heads, w.head_dim)[:L].copy()).view(
        torch.float8_e4m3fn).double() * float(np.float32(w.k_scale))
    vt = torch.from_numpy(v.reshape(-1, w.num_kv_heads, w.head_dim)[:L].copy()).view(
        torch.float8_e4m3fn).double() * float(np.float32(w.v_scale))
    g = w.group
    kt = kt.permute(1, 0, 2).repeat_interleave(g, dim=0)
    vt = vt.permute(1, 0, 2).repeat_interleave(g, dim=0)
    qt = torch.from_numpy(w.q[0].view(np.float16).astype(np.float64))[:, None, :]
    want = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=w.scale)[:, 0]
    np.testing.assert_allclose(got[0], want.numpy(), rtol=0, atol=1e-12)


def test_workload_scales_are_float32():
    assert float(np.float32(FP8_K_SCALE)) == FP8_K_SCALE
    assert float(np.float32(FP8_V_SCALE)) == FP8_V_SCALE
