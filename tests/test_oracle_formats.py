"""Pins for the oracle's number formats (bf16 and OCP E4M3), against library
casts and the formats' own definitions.  CPU only."""
import numpy as np
import pytest
import torch


def _rand_f32_bits(n, seed):
    rng = np.random.default_rng(seed)
    return rng.integers(0, 2**32, size=n, dtype=np.uint64).astype(np.uint32).view(np.float32)


def test_bf16_rne_matches_library_cast(oracle):
    x = _rand_f32_bits(1 << 20, 1)
    x = x[~np.isnan(x)]
    got = oracle.bf16_from_f32(x)
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_rne_ties_and_specials(oracle):
    cases = {
        0x3F808000: 0x3F80,  # tie, upper even -> stays
        0x3F818000: 0x3F82,  # tie, upper odd -> rounds up
        0x3F808001: 0x3F81,  # above tie -> up
        0x3F807FFF: 0x3F80,  # below tie -> down
        0x7F7FFFFF: 0x7F80,  # max float rounds to +inf
        0x7F800000: 0x7F80,  # +inf
        0xFF800000: 0xFF80,  # -inf
        0x80000000: 0x8000,  # -0
        0x00000001: 0x0000,  # smallest subnormal -> +0
        0x00008000: 0x0000,  # subnormal tie, even -> down
        0x00018000: 0x0002,  # subnormal tie, odd -> up
    }
    x = np.array(list(cases.keys()), dtype=np.uint32).view(np.float32)
    got = oracle.bf16_from_f32(x)
    assert [int(v) for v in got] == list(cases.values())
    nan = np.array([0x7FC00001, 0xFF800001], dtype=np.uint32).view(np.float32)
    g = oracle.bf16_from_f32(nan)
    assert all(((int(v) & 0x7F80) == 0x7F80) and (int(v) & 0x7F) for v in g)
    assert int(g[1]) & 0x8000


def test_bf16_roundtrip_exact(oracle):
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    f = oracle.f32_from_bf16(h)
    finite = ~np.isnan(f)
    assert np.array_equal(oracle.bf16_from_f32(f[finite]), h[finite])


def test_e4m3_decode_all_codes_match_library(oracle):
    codes = np.arange(256, dtype=np.uint16).astype(np.uint8)
    got = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).float().numpy()
    both_nan = np.isnan(got) & np.isnan(ref)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[~both_nan].view(np.uint32), ref[~both_nan].view(np.uint32))


def test_e4m3_decode_ocp_table(oracle):
    # values fixed by the OCP 8-bit floating point E4M3 definition
    table = {0x00: 0.0, 0x01: 2.0**-9, 0x07: 7 * 2.0**-9, 0x08: 2.0**-6, 0x38: 1.0,
             0x39: 1.125, 0x3F: 1.875, 0x40: 2.0, 0x7E: 448.0, 0xFE: -448.0, 0xB8: -1.0}
    codes = np.array(list(table.keys()), dtype=np.uint8)
    assert list(oracle.e4m3_decode(codes)) == list(table.values())
    assert np.isnan(oracle.e4m3_decode(np.array([0x7F, 0xFF], np.uint8))).all()
    assert np.signbit(oracle.e4m3_decode(np.array([0x80], np.uint8)))[0]


def test_e4m3_encode_matches_library_inside_range(oracle):
    # every finite bf16 value below the saturation threshold, plus random fp32
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    xb = oracle.f32_from_bf16(h)
    xr = _rand_f32_bits(1 << 20, 2)
    x = np.concatenate([xb, xr, np.linspace(-470, 470, 200001, dtype=np.float32)])
    x = x[np.isfinite(x) & (np.abs(x) < 464.0)]
    got = oracle.e4m3_encode(x)
    ref = torch.from_numpy(x.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, ref)


def test_e4m3_encode_rounding_and_saturation(oracle):
    cases = [
        (1.0625, 0x38),        # tie between 1.0 and 1.125 -> even mantissa (1.0)
        (1.1875, 0x3A),        # tie between 1.125 and 1.25 -> even (1.25)
        (2.0**-10, 0x00),      # subnormal tie between 0 and 2^-9 -> 0
        (3 * 2.0**-10, 0x02),  # tie between 2^-9 and 2^-8 -> even (2^-8)
        (15 * 2.0**-10, 0x08), # tie between 7*2^-9 and 2^-6 -> even (2^-6 = code 8)
        (432.0, 0x7E),         # tie between 416 and 448 -> even mantissa (448)
        (400.0, 0x7C),         # tie between 384 and 416 -> even mantissa (384)
        (440.0, 0x7E),         # nearer 448
        (448.0, 0x7E),
        (463.99, 0x7E),
        (464.0, 0x7E),         # would round to 480 (not finite in E4M3) -> saturate
        (1e30, 0x7E),
        (float("inf"), 0x7E),
        (-float("inf"), 0xFE),
        (-500.0, 0xFE),
        (-0.0, 0x80),
        (0.0, 0x00),
    ]
    x = np.array([c[0] for c in cases], dtype=np.float32)
    got = oracle.e4m3_encode(x)
    assert [int(v) for v in got] == [c[1] for c in cases]
    assert int(oracle.e4m3_encode(np.array([np.nan], np.float32))[0]) & 0x7F == 0x7F


def test_e4m3_encode_is_nearest(oracle):
    # brute force: the encoded value is the nearest finite E4M3 value (ties even)
    codes = np.arange(256, dtype=np.uint16).astype(np.uint8)
    vals = oracle.e4m3_decode(codes).astype(np.float64)
    finite = ~np.isnan(vals)
    grid = vals[finite]
    gcodes = codes[finite]
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(20000) * rng.choice([1e-3, 1e-1, 1, 10, 100], 20000)).astype(np.float32)
    x = np.clip(x, -448, 448)
    got = oracle.e4m3_decode(oracle.e4m3_encode(x)).astype(np.float64)
    d = np.abs(grid[None, :] - x.astype(np.float64)[:, None])
    best = d.min(axis=1)
    assert np.all(np.abs(got - x) == best)
    del gcodes


def _torch_block_quant(x_bf16_bits):
    """The same per-128 block quantisation written with torch CPU ops."""
    x = torch.from_numpy(x_bf16_bits.view(np.int16).copy()).view(torch.bfloat16).float()
    n, H = x.shape
    xb = x.view(n, H // 128, 128)
    amax = xb.abs().amax(dim=-1, keepdim=True).clamp_min(2.0**-119)
    c448 = torch.full_like(amax, 448.0)
    scale = amax / c448          # tensor / tensor: IEEE division (a scalar operand
    inv = c448 / amax            # would make torch multiply by a reciprocal instead)
    p = xb * inv
    q = p.to(torch.float8_e4m3fn).view(torch.uint8).view(n, H)
    return q.numpy(), scale.view(n, H // 128).numpy()


def test_block_quant_matches_library_ops(oracle):
    rng = np.random.default_rng(5)
    x32 = rng.standard_normal((64, 1024)).astype(np.float32)
    x32[3, :128] = 0.0                            # an all-zero block
    x32[4, 128:256] *= 1e-30                      # a tiny block (amax above the 2^-119 floor)
    x32[6, 512:640] *= 2.0**-140                  # below the floor: bf16 subnormals and zeros
    x32[5, 256:384] = 1e-25                       # constant block
    xb = oracle.bf16_from_f32(x32)
    q, s = oracle.quantize_rows_e4m3(xb)
    q_ref, s_ref = _torch_block_quant(xb)
    assert np.array_equal(s.view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(q, q_ref)


def test_block_quant_error_bound_and_amax_code(oracle):
    rng = np.random.default_rng(6)
    xb = oracle.bf16_from_f32(rng.standard_normal((32, 7168)).astype(np.float32) * 3)
    q, s = oracle.quantize_rows_e4m3(xb)
    x = oracle.f32_from_bf16(xb).astype(np.float64).reshape(32, 56, 128)
    dq = oracle.e4m3_decode(q).astype(np.float64).reshape(32, 56, 128) * s[..., None]
    # the largest magnitude of every block encodes to +-448
    amax_pos = np.abs(x).argmax(axis=-1)
    qa = np.take_along_axis(q.reshape(32, 56, 128), amax_pos[..., None], axis=-1)[..., 0]
    assert np.all((qa & 0x7F) == 0x7E)
    # |dequant - x| <= half an E4M3 spacing at the scaled value, times the scale
    p = np.abs(x) / s[..., None]
    e = np.floor(np.log2(np.maximum(p, 2.0**-6)))
    half = 0.5 * 2.0 ** (e - 3)
    assert np.all(np.abs(dq - x) <= (half * s[..., None]) * (1 + 1e-5) + 1e-30)


# ---------------------------------------------------------------------------
# blocks at and below the amax floor, in exact rational arithmetic
# ---------------------------------------------------------------------------

def _rn_f32(q):
    """The float32 nearest to the rational q (ties to even), subnormals included."""
    from fractions import Fraction
    f = np.float32(float(q))
    cands = [f, np.nextafter(f, np.float32(np.inf)), np.nextafter(f, np.float32(-np.inf))]
    cands = [c for c in cands if np.isfinite(c)]
    best = min(abs(Fraction(float(c)) - q) for c in cands)
    near = [c for c in cands if abs(Fraction(float(c)) - q) == best]
    near.sort(key=lambda c: int(np.array(c, np.float32).view(np.uint32)) & 1)   # even significand first
    return np.float32(near[0])


def _e4m3_nearest_code(p):
    """The E4M3 code nearest to the rational p by brute force over the finite codes (ties
    to the even significand; -0 for a negative value that rounds to zero)."""
    from fractions import Fraction
    best, best_code = None, None
    for c in range(0x7F):                          # 0x00 .. 0x7E: +0 .. 448
        e, m = c >> 3, c & 7
        v = Fraction(m, 8) * Fraction(2) ** -6 if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
        d = abs(v - abs(p))
        if best is None or d < best or (d == best and (c & 1) == 0):
            best, best_code = d, c
    return best_code | (0x80 if p < 0 else 0)


TINY_AMAX = [0.0, 2.0**-70, 2.0**-100, 2.0**-119, float.fromhex("0x1.fep-120"), 2.0**-126, 2.0**-133]


@pytest.mark.parametrize("amax", TINY_AMAX)
def test_block_quant_tiny_blocks_exact(oracle, amax):
    """Blocks whose largest magnitude is 0, 2^-70, 2^-100, 2^-119 (the floor), the bf16 value
    just below it, 2^-126 and the smallest bf16 subnormal 2^-133.  The oracle's codes and
    scale must equal the definition evaluated in exact arithmetic: amax raised to 2^-119,
    scale = RN(amax/448), inv = RN(448/amax), code = the E4M3 value nearest to RN(x * inv).
    Every nonzero bf16 input keeps a nonzero code, and zeros keep their sign."""
    from fractions import Fraction
    rng = np.random.default_rng(int(amax * 2.0**140) % 1000 + 7)
    # 128 bf16 values in [-amax, amax], the largest magnitude exactly amax, with zeros of both signs
    frac = rng.uniform(-1, 1, 128).astype(np.float32)
    x = (frac * np.float32(amax)).astype(np.float32) if amax > 0 else np.zeros(128, np.float32)
    xb = oracle.bf16_from_f32(x)
    xb[5] = oracle.bf16_from_f32(np.array([amax], np.float32))[0]
    xb[6] = 0x0000
    xb[7] = 0x8000
    v = oracle.f32_from_bf16(xb)
    assert np.abs(v).max() == np.float32(amax)
    q, s = oracle.quantize_rows_e4m3(xb.reshape(1, 128))
    a = max(Fraction(float(amax)), Fraction(2) ** -119)
    scale = _rn_f32(a / 448)
    inv = _rn_f32(448 / a)
    assert np.isfinite(inv)
    assert int(s.view(np.uint32)[0, 0]) == int(np.array(scale, np.float32).view(np.uint32))
    want = np.array([_e4m3_nearest_code(Fraction(float(_rn_f32(Fraction(float(vi)) * Fraction(float(inv))))))
                     if vi != 0 else (0x80 if np.signbit(vi) else 0x00) for vi in v], np.uint8)
    assert np.array_equal(q[0], want)
    nz = v != 0
    assert np.all((q[0][nz] & 0x7F) != 0)          # no nonzero input lost to a zero code
    assert q[0][6] == 0x00 and q[0][7] == 0x80
    if amax >= 2.0**-119:                            # at or above the floor: amax maps to 448
        assert (q[0][5] & 0x7F) == 0x7E
