"""Pins for the oracle's MXFP4 quantize and MXFP4 -> FP8 E4M3 conversions (CPU).

MXFP4: the closed form of the power-of-two exponent and reconstruction bounds.
FP4 -> FP8: all 16 codes x 256 scale shifts against (a) a brute-force nearest
E4M3 search and (b) the page's exponent/mantissa bit formula, plus exactness
after decoding both formats; the column form against the row form.
"""
import numpy as np
import pytest

import oracle as ora
from golden_util import load


def test_mxfp4_exponent_closed_form():
    """For block amax in [2^k, 2^(k+1)) the UE8M0 byte is k - 2 + 127."""
    rng = np.random.default_rng(0)
    for k in range(-40, 40, 3):
        x = (rng.uniform(-1, 1, (4, 32)) * 2.0 ** k).astype(np.float32)
        x[:, 5] = np.float32(2.0 ** k) * np.float32(1.0 + rng.uniform(0, 0.99))
        _, scales = ora.mxfp4_quantize(x)
        assert np.all(scales == k - 2 + 127), (k, scales)


def test_mxfp4_codes_and_reconstruction():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((64, 256)).astype(np.float32)
    packed, scales = ora.mxfp4_quantize(x)
    codes = np.stack([packed & 0xF, packed >> 4], axis=-1).reshape(64, 256)
    E = np.repeat(scales.astype(np.int64) - 127, 32, axis=1)
    a = (x.astype(np.float64) * 2.0 ** (-E)).astype(np.float32)
    assert np.all(np.abs(a).reshape(64, 8, 32).max(-1) >= 4.0)
    assert np.all(np.abs(a).reshape(64, 8, 32).max(-1) < 8.0)
    assert np.array_equal(codes, ora.e2m1_rn(a))
    y = ora.e2m1_value(codes) * 2.0 ** E
    # error at most half a grid step (1 in [4, 6]) or the clip from [6, 8) to 6
    assert np.all(np.abs(y - x) <= 2.0 * 2.0 ** E)


def test_mxfp4_zero_and_tiny_blocks():
    x = np.zeros((1, 64), np.float32)
    x[0, 40] = 1e-42          # fp32 subnormal
    x[0, 33] = -0.0
    packed, scales = ora.mxfp4_quantize(x)
    assert scales[0, 0] == 0 and scales[0, 1] == 0     # E clamps to -127
    codes = np.stack([packed & 0xF, packed >> 4], axis=-1).reshape(-1)
    assert np.all(codes[:32] == 0)
    assert codes[33] == 0x8                              # sign of -0 kept


def test_mxfp4_infinite_amax():
    """A block holding an infinity: the exponent is read from the amax's
    exponent field (reading R15), 255 for an infinity, so floor(log2) is 128,
    E = 126 and the UE8M0 byte 253; the infinities saturate to +-6 (R2,
    code 7 with the sign) and the finite elements, scaled by 2^-126, round
    to zero.  A block of finite values beside it keeps its own exponent."""
    x = np.zeros((1, 64), np.float32)
    x[0, :32] = np.linspace(-3.0, 3.0, 32, dtype=np.float32)
    x[0, 3] = np.inf
    x[0, 9] = -np.inf
    x[0, 32:] = 1.5
    packed, scales = ora.mxfp4_quantize(x)
    assert scales[0, 0] == 126 + 127 and scales[0, 1] == 0 - 2 + 127
    codes = np.stack([packed & 0xF, packed >> 4], axis=-1).reshape(-1)
    assert codes[3] == 0x7 and codes[9] == 0xF
    finite = np.r_[0:3, 4:9, 10:32]
    assert np.all((codes[finite] & 0x7) == 0)
    assert np.all(codes[32:] == ora.e2m1_rn(np.full(32, 1.5 * 4.0, np.float32)))


def _brute_e4m3(val: float) -> int:
    table = ora.e4m3_value(np.arange(256))
    fin = np.nonzero(~np.isnan(table))[0]
    if val >= 448.0:
        return 0x7E
    if val <= -448.0:
        return 0xFE
    d = np.abs(table[fin] - val)
    best = fin[d == d.min()]
    if best.size > 1:                                  # tie: even mantissa
        best = best[(best & 1) == 0]
    b = int(best[0]) & 0x7F
    return b | (0x80 if np.signbit(val) else 0)


def test_fp4_to_fp8_all_codes_all_shifts():
    """[MoE-FP4] 核心技术贡献 1, checked on every (code, shift) pair."""
    fix = load("fp8_bitmap.txt")
    bias4, bias8 = int(fix["bias_fp4"][0]), int(fix["bias_fp8"][0])
    shift = int(fix["mantissa_shift"][0])
    for d in range(0, 255):
        # one 128-span whose first block has scale 127 + d and the rest 127:
        # S_t = 127 + d, so block 1..3 get shift d and block 0 shift 0
        packed = np.zeros((1, 64), np.uint8)
        codes = np.tile(np.arange(16, dtype=np.uint8), 8)       # 128 codes
        packed[0] = codes[0::2] | (codes[1::2] << 4)
        scales = np.array([[127 + min(d, 127), 127, 127, 127]], np.uint8) if d <= 127 else \
            np.array([[254, 254 - d, 254 - d, 254 - d]], np.uint8)
        fp8, fsc = ora.fp4_to_fp8_row(packed, scales)
        st = int(scales.max())
        assert fsc[0, 0] == np.float32(2.0 ** (st - 127))
        for k in range(32, 48):                 # block 1, all 16 codes
            c = int(codes[k])
            dd = st - int(scales[0, 1])
            assert dd == d
            val = ora.e2m1_value([c])[0] * 2.0 ** (-dd)
            b = int(fp8[0, k])
            assert b == _brute_e4m3(val), (c, d, b)
            e, m, s = (c >> 1) & 3, c & 1, c >> 3
            if d <= 8:
                # exact after decoding both formats to float
                assert ora.e4m3_value([b])[0] * 2.0 ** (st - 127) == \
                    ora.e2m1_value([c])[0] * 2.0 ** (int(scales[0, 1]) - 127)
            if e >= 1 and e - bias4 + bias8 - d >= 1:
                # the page's formula: exponent re-biased, mantissa shifted,
                # exponent lowered by S_target - S_sub
                want = (s << 7) | ((e - bias4 + bias8 - d) << 3) | (m << shift)
                assert b == want, (c, d, b, want)


def test_fp4_to_fp8_row_target_is_max_of_four():
    rng = np.random.default_rng(3)
    rows, cols = 8, 512
    packed = rng.integers(0, 256, (rows, cols // 2), dtype=np.uint8)
    scales = rng.integers(100, 140, (rows, cols // 32), dtype=np.uint8)
    fp8, fsc = ora.fp4_to_fp8_row(packed, scales)
    st = scales.reshape(rows, -1, 4).max(-1)
    assert np.array_equal(fsc, (2.0 ** (st.astype(np.float64) - 127)).astype(np.float32))
    codes = np.stack([packed & 0xF, packed >> 4], axis=-1).reshape(rows, cols)
    src = ora.e2m1_value(codes) * 2.0 ** (np.repeat(scales, 32, axis=1) - 127.0)
    dst = ora.e4m3_value(fp8) * np.repeat(fsc.astype(np.float64), 128, axis=1)
    dshift = np.repeat(st, 4, axis=1) - scales
    exact = np.repeat(dshift <= 8, 32, axis=1)
    assert np.array_equal(src[exact], dst[exact])


def test_fp4_to_fp8_col_is_transposed_row_when_scales_agree():
    """With every source scale in a token block equal to its neighbours, the
    column form must equal the transposed row form."""
    rng = np.random.default_rng(4)
    R, K = 300, 256
    packed = rng.integers(0, 256, (R, K // 2), dtype=np.uint8)
    scales = np.full((R, K // 32), 130, np.uint8)
    off = np.array([0, 5, 5, 133, 300], np.int64)        # includes an empty segment
    out, osc = ora.fp4_to_fp8_col(packed, scales, off)
    row, rsc = ora.fp4_to_fp8_row(packed, scales)
    so = ora.seg_scale_offsets(off)
    for e in range(len(off) - 1):
        n_e = int(off[e + 1] - off[e])
        seg = out[K * off[e]: K * off[e] + K * n_e].reshape(K, n_e)
        assert np.array_equal(seg, row[off[e]:off[e + 1]].T)
        nb = (n_e + 127) // 128
        s = osc[K * so[e]: K * so[e] + K * nb]
        assert np.all(s == np.float32(2.0 ** 3))


def test_fp4_to_fp8_col_token_block_scale():
    """The target scale of an output block is the largest source scale among
    its <= 128 tokens; smaller source scales shift those tokens down."""
    rng = np.random.default_rng(5)
    R, K = 200, 128
    packed = rng.integers(0, 256, (R, K // 2), dtype=np.uint8)
    scales = rng.integers(120, 135, (R, K // 32), dtype=np.uint8)
    out, osc = ora.fp4_to_fp8_col_segment(packed, scales, 0, R)
    nb = 2
    assert osc.shape == (K, nb)
    codes = np.stack([packed & 0xF, packed >> 4], axis=-1).reshape(R, K)
    for k in (0, 31, 32, 77, 127):
        for b in range(nb):
            toks = np.arange(128 * b, min(128 * b + 128, R))
            st = scales[toks, k // 32].max()
            assert osc[k, b] == np.float32(2.0 ** (int(st) - 127))
            for j in toks[:40]:
                val = ora.e2m1_value([codes[j, k]])[0] * 2.0 ** (int(scales[j, k // 32]) - int(st))
                assert out[k, j] == _brute_e4m3(val)


def test_payload_sizes_match_page():
    """paper-daily review "通信量": FP8 ~1.03*M*K bytes, MXFP4 ~0.53*M*K."""
    s = load("sizes.txt")
    M, K = 32768, 7168
    x = np.zeros((4, K), np.float32)
    packed, scales = ora.mxfp4_quantize(x)
    mx = (packed.nbytes + scales.nbytes) / x.size
    assert mx == 0.53125 and round(mx, 2) == float(s["mxfp4_bytes_per_element_2dp"][0])
    fp8, fsc = ora.fp4_to_fp8_row(packed, scales)
    f8 = (fp8.nbytes + fsc.nbytes) / x.size
    assert f8 == 1.03125 and round(f8, 2) == float(s["fp8_bytes_per_element_2dp"][0])
    assert round(mx * 8, 2) == float(s["mxfp4_bits_per_weight"][0])
