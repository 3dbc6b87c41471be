"""Pins of the oracle's upstream quantizer (per-token-head, quant mode 0) against properties the
definition fixes and against independent conversions: numpy's float16 rounding and torch's
float8_e4m3fn rounding for the two nearest-value searches, error bounds, exact scaling and sign
symmetry, the all-zero vector, and the paged key-cache placement."""
import numpy as np
import pytest

import oracle
import workloads as W


def _bf16(x):
    """float32 array -> bfloat16 bits (truncation; the inputs are then exactly those values)"""
    return (np.ascontiguousarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _f32(b):
    return (b.astype(np.uint32) << 16).view(np.float32)


def _data(seed, shape=(3, 64, 128), sigma=3.0):
    rng = np.random.default_rng(seed)
    return _bf16(rng.normal(0, sigma, size=shape) * rng.uniform(0.01, 100, size=shape[:-1] + (1,)))


@pytest.mark.parametrize("scale_f32", [True, False])
def test_int8_codes_within_half_a_step(scale_f32):
    b = _data(1)
    codes, scales = oracle.quantize(b, False, scale_f32)
    x = _f32(b).astype(np.float64)
    s = scales.astype(np.float64)[..., None]
    err = np.abs(codes.astype(np.float64) * s - x)
    # rounding to the nearest step: at most half a step (plus the scale's own rounding, which can
    # push the largest element one step past 127 before the clamp)
    assert np.all(err <= 0.5 * s * (1 + 2e-3) + np.abs(x) * 2e-3)
    assert np.abs(codes).max() == 127
    amax = np.abs(x).max(-1)
    # the largest element of every vector lands on +-127
    top = np.take_along_axis(np.abs(codes).astype(np.int32), np.abs(x).argmax(-1)[..., None], -1)[..., 0]
    assert np.all(top == 127)
    rel = 2.0 ** -10 if not scale_f32 else 1e-6
    assert np.allclose(scales.astype(np.float64), amax / 127.0, rtol=rel, atol=0)


def test_fp16_scale_is_numpys_rounding():
    b = _data(2)
    _, s16 = oracle.quantize(b, False, False)
    _, s32 = oracle.quantize(b, False, True)
    # the fp16 scale is the fp32 scale rounded to nearest (ties to even): numpy's conversion
    assert np.array_equal(s16, s32.astype(np.float16))


def test_e4m3_codes_are_torchs_rounding_of_x_over_s():
    torch = pytest.importorskip("torch")
    b = _data(3)
    codes, scales = oracle.quantize(b, True, True)
    y = _f32(b) / scales[..., None]                    # fp32 division, as the definition states
    ref = torch.from_numpy(np.ascontiguousarray(y)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes, ref)
    # every vector's largest element saturates at 448 (code 0x7E)
    assert np.all((codes & 0x7F).max(-1) == 0x7E)


def test_zero_vector_and_exact_scaling_and_sign():
    b = _data(4, shape=(2, 4, 128))
    b[0, 1, :] = 0
    for fp8 in (False, True):
        codes, scales = oracle.quantize(b, fp8, True)
        assert scales[0, 1] == 0 and not codes[0, 1].any()
        # x * 2 (exact in bfloat16 here): same codes, doubled scales
        c2, s2 = oracle.quantize(_bf16(_f32(b) * 2), fp8, True)
        assert np.array_equal(c2, codes) and np.array_equal(s2, scales * 2)
        # -x: negated codes, same scales
        cn, sn = oracle.quantize(_bf16(-_f32(b)), fp8, True)
        assert np.array_equal(sn, scales)
        if fp8:
            nz = (codes & 0x7F) != 0
            assert np.array_equal(cn[nz], codes[nz] ^ 0x80)
        else:
            assert np.array_equal(cn, -codes)


def test_key_cache_write_lands_on_its_page_and_slot():
    case = W.make_case("qk", batch=2, s1=1, seq_lens_k=[300, 200], block_size=64, sparse_count=16, seed=5)
    case = W.with_key_stride(case, 32, seed=1)
    before_k, before_s = case.key.copy(), case.k_scale.copy()
    rng = np.random.default_rng(6)
    kb = _bf16(rng.normal(0, 1, size=(3, 128)))
    tok_b = np.array([0, 1, 1], np.int32)
    tok_p = np.array([5, 130, 199], np.int32)
    err = oracle.quantize_keys(case, kb, tok_b, tok_p)
    assert err == 0
    codes, scales = oracle.quantize(kb, False, False)
    page_elems = case.block_size * 128
    touched = np.zeros(case.key.shape, bool)
    for t in range(3):
        page = case.block_table[tok_b[t], tok_p[t] // 64]
        slot = tok_p[t] % 64
        got = case.key[page, slot * 128:(slot + 1) * 128].view(np.int8)
        assert np.array_equal(got, codes[t])
        assert case.k_scale.reshape(case.num_blocks, -1)[page, slot] == scales[t]
        touched[page, slot * 128:(slot + 1) * 128] = True
    assert np.array_equal(case.key[~touched], before_k[~touched])   # nothing else moved (pad too)
    assert page_elems < case.key.shape[1]
    # out-of-range positions and pages are reported and skipped
    case.block_table[0, 0] = case.num_blocks + 3
    k0 = case.key.copy()
    err = oracle.quantize_keys(case, kb[:2], np.array([0, 2], np.int32), np.array([1, 0], np.int32))
    assert err == (oracle.ERR_PAGE | oracle.ERR_LENGTH)
    assert np.array_equal(case.key, k0)


def test_degenerate_vectors_of_the_generator():
    """The generator's special vectors: exact halfway quotients round to even (numpy's rint for
    int8, torch's float8_e4m3fn cast for e4m3), a zero vector, a scale in the float subnormal range
    (which float16 storage rounds to 0, zeroing the codes), and a scale beyond float16's range
    (saturated at 65504, codes then clamp)."""
    torch = pytest.importorskip("torch")
    b = W.bf16_vectors((5, 128), seed=7)
    x = _f32(b)
    c16, s16 = oracle.quantize(b, False, False)
    c32, s32 = oracle.quantize(b, False, True)
    # halfway cases: amax 127 gives s = 1 exactly, so codes are x rounded half to even
    assert s16[3] == 1.0 and s32[3] == 1.0
    assert np.array_equal(c16[3], np.rint(x[3]).astype(np.int8))
    assert np.any(np.abs(x[3] - np.trunc(x[3])) == 0.5)
    e8, se = oracle.quantize(b, True, True)
    assert se[4] == 1.0
    assert np.array_equal(e8[4], torch.from_numpy(x[4].copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy())
    # zero vector
    assert s16[0] == 0 and s32[0] == 0 and not c16[0].any() and not e8[0].any()
    # subnormal scale: kept in float32, rounds to 0 in float16
    assert 0 < s32[1] < np.finfo(np.float32).tiny
    assert s16[1] == 0 and not c16[1].any()
    assert np.abs(c32[1]).max() == 127
    # beyond float16: the stored scale saturates and the codes clamp
    assert s16[2] == np.float16(65504)
    assert np.array_equal(c16[2], np.clip(np.rint(x[2] / np.float32(65504)), -127, 127).astype(np.int8))
    e16, _ = oracle.quantize(b, True, False)
    assert np.all((e16[2] & 0x7F).max() == 0x7E)


def test_signed_zeros_keep_their_sign_in_e4m3():
    """x = -0 (and a negative quotient that underflows to zero) divides to -0, whose nearest e4m3
    value is -0 (code 0x80): torch's float8_e4m3fn cast of x / s says the same; int8 has one zero."""
    torch = pytest.importorskip("torch")
    b = W.bf16_vectors((6, 128), seed=7)              # vector 5: signed zeros beside ~1e30 values
    x = _f32(b[5])
    assert np.any(np.signbit(x) & (x == 0)) and np.any(~np.signbit(x) & (x == 0))
    for scale_f32 in (True, False):
        codes, scales = oracle.quantize(b[5:6], True, scale_f32)
        y = (x / scales[0].astype(np.float32)).astype(np.float32)
        ref = torch.from_numpy(y.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        inside = np.abs(y) <= 448.0               # torch's cast does not saturate: NaN beyond 448
        assert np.array_equal(codes[0][inside], ref[inside])
        assert np.all(codes[0][~inside] == (0x7E | (np.signbit(y[~inside]) << 7)))
        assert np.all(codes[0][np.signbit(x) & (x == 0)] == 0x80)
    c8, _ = oracle.quantize(b[5:6], False, False)
    assert np.all(c8[0][x == 0] == 0)
