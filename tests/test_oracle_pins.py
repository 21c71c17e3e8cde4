"""Pins of the CPU oracle against things other than itself.

Each test fixes part of the oracle with a closed form, an invariant, brute
force on a tiny case, or a library routine (numpy's fp16, ml_dtypes' and
torch's fp8/fp4 tables, torch's float64 matmul).  None of them retypes the
oracle's decoder: blocks are built from fields by the independent test
packer (tests/packers.py) and the expected weights come from hand-chosen
closed forms.
"""
import json
import os

import numpy as np
import pytest

import oracle
from packers import (pack_nvfp4_row, pack_q4k_block, pack_q5k_block, pack_q6k_block,
                     pack_scales_q4k)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ---------------------------------------------------------------- code tables

def test_f16_decode_matches_numpy_all_codes():
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = codes.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_to_f64(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signs of zero and infinities too
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_e4m3_decode_matches_libraries_all_codes():
    ml = pytest.importorskip("ml_dtypes")
    codes = np.arange(256, dtype=np.uint8)
    ref = codes.view(ml.float8_e4m3fn).astype(np.float64)
    got = np.array([oracle.e4m3_to_f64(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan) and nan.sum() == 2
    assert np.array_equal(got[~nan], ref[~nan])
    import torch
    tref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(got[~nan], tref[~nan])


def test_e2m1_decode_matches_ml_dtypes():
    ml = pytest.importorskip("ml_dtypes")
    got = np.array([oracle.e2m1_to_f64(c) for c in range(16)])
    # ml_dtypes stores one e2m1 value per byte in the low nibble
    ref = np.arange(16, dtype=np.uint8).view(ml.float4_e2m1fn).astype(np.float64)
    assert np.array_equal(got, ref)
    assert np.array_equal(got[:8], [0, 0.5, 1, 1.5, 2, 3, 4, 6])


def test_e4m3_generator_code_range_is_2m6_to_16():
    """The synthetic group scales draw codes 0x08..0x58: exactly the 81
    e4m3 values in [2^-6, 16] (checked through the library, not the oracle)."""
    ml = pytest.importorskip("ml_dtypes")
    from skinny_gemm_q4_gb300 import synth
    codes = np.arange(synth.E4M3_CODE_LO, synth.E4M3_CODE_HI + 1, dtype=np.uint8)
    vals = codes.view(ml.float8_e4m3fn).astype(np.float64)
    allpos = np.arange(0, 0x7F, dtype=np.uint8).view(ml.float8_e4m3fn).astype(np.float64)
    inrange = allpos[(allpos >= 2.0 ** -6) & (allpos <= 16.0)]
    assert codes.size == 81 and np.array_equal(np.sort(vals), np.sort(inrange))


# ---------------------------------------------------------- 6-bit packing

def test_scale_min_packing_exhaustive_per_field():
    """Each of the 16 six-bit fields over 0..63, the others at 0 and at 63:
    the oracle's unpacking returns exactly the packed fields."""
    for other in (0, 63):
        for field in range(16):
            for v in range(64):
                sc = [other] * 8
                m = [other] * 8
                if field < 8:
                    sc[field] = v
                else:
                    m[field - 8] = v
                b = pack_scales_q4k(sc, m)
                for s in range(8):
                    assert oracle.unpack_scale_min(b, s) == (sc[s], m[s]), (field, v, s)


def test_scale_min_packing_is_a_bijection_on_12_bytes():
    """96 bits used exactly once: unpack then repack gives back any bytes."""
    rng = np.random.default_rng(7)
    for _ in range(200):
        b = rng.integers(0, 256, 12, dtype=np.uint8)
        fields = [oracle.unpack_scale_min(b, s) for s in range(8)]
        back = pack_scales_q4k([f[0] for f in fields], [f[1] for f in fields])
        assert np.array_equal(back, b)


# ------------------------------------------------------ closed-form blocks

def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_q4k_closed_form_block():
    """d = 1, dmin = 0.5, sc[s] = s+1, m[s] = 2s, q_j = j mod 16 gives
    w_j = (s+1)(j mod 16) - s with s = j // 32 (the sub-block of element j)."""
    g = _golden("q4k_closed_form.json")
    j = np.arange(256)
    q = j % 16
    blk = pack_q4k_block(g["d"], g["dmin"], g["sc"], g["m"], q)
    w = oracle.dequantize(oracle.Q4_K, blk, 1, 256)[0]
    s = j // 32
    assert np.array_equal(w, ((s + 1) * (j % 16) - s).astype(np.float32))


def test_q4k_each_element_lands_at_its_index():
    """Distinct q per element in every sub-block and distinct sc per
    sub-block: w_j = sc[s_j] * q_j identifies each element's slot."""
    rng = np.random.default_rng(3)
    for _ in range(4):
        q = rng.integers(0, 16, 256)
        sc = rng.permutation(np.arange(1, 64))[:8]
        blk = pack_q4k_block(1.0, 0.0, sc, [0] * 8, q)
        w = oracle.dequantize(oracle.Q4_K, blk, 1, 256)[0]
        assert np.array_equal(w, (sc[np.arange(256) // 32] * q).astype(np.float32))


def test_q4k_min_term_per_subblock():
    """d = 0: every weight of sub-block s is -dmin * m[s]."""
    m = [1, 7, 13, 21, 34, 42, 55, 63]
    blk = pack_q4k_block(0.0, 0.25, [63] * 8, m, np.full(256, 15))
    w = oracle.dequantize(oracle.Q4_K, blk, 1, 256)[0]
    assert np.array_equal(w, (-0.25 * np.repeat(m, 32)).astype(np.float32))


def test_q5k_high_bit_adds_16_and_maps_per_element():
    g = _golden("q4k_closed_form.json")
    j = np.arange(256)
    q4 = j % 16
    s = j // 32
    base = pack_q5k_block(g["d"], g["dmin"], g["sc"], g["m"], q4)
    w0 = oracle.dequantize(oracle.Q5_K, base, 1, 256)[0]
    assert np.array_equal(w0, ((s + 1) * q4 - s).astype(np.float32))
    ones = pack_q5k_block(g["d"], g["dmin"], g["sc"], g["m"], q4 + 16)
    assert np.array_equal(ones[16:48], np.full(32, 255, dtype=np.uint8))  # qh all ones
    w1 = oracle.dequantize(oracle.Q5_K, ones, 1, 256)[0]
    assert np.array_equal(w1, ((s + 1) * (q4 + 16) - s).astype(np.float32))
    # one qh bit at a time moves exactly one element by 16 * sc
    for bit in range(8):
        for l in (0, 5, 31):
            blk = base.copy()
            blk[16 + l] |= (1 << bit)
            w = oracle.dequantize(oracle.Q5_K, blk, 1, 256)[0]
            diff = np.nonzero(w != w0)[0]
            c, hi = bit // 2, bit % 2
            e = 64 * c + 32 * hi + l
            assert list(diff) == [e]
            assert w[e] - w0[e] == 16 * (e // 32 + 1)


def test_q6k_all_codes_and_scales():
    """d = 2^-4, scales from {1, 127, -128, -1, ...}: every one of the 64 q
    codes in every 16-group gives 2^-4 * sc * (v - 32) exactly."""
    g = _golden("q6k_closed_form.json")
    scales = np.array(g["scales"], dtype=np.int64)
    for shift in range(4):
        v = (np.arange(256) + 16 * shift) % 64          # all 64 codes per 64 elements
        blk = pack_q6k_block(g["d"], scales, v - 32)
        w = oracle.dequantize(oracle.Q6_K, blk, 1, 256)[0]
        e = np.arange(256)
        h, s, l = e // 128, (e % 128) // 32, e % 32
        sc = scales[8 * h + l // 16 + 2 * s]
        assert np.array_equal(w, (g["d"] * sc * (v - 32)).astype(np.float32))


def test_q6k_each_element_lands_at_its_index():
    rng = np.random.default_rng(11)
    for _ in range(4):
        q = rng.integers(-32, 32, 256)
        scales = np.ones(16, dtype=np.int64)
        blk = pack_q6k_block(1.0, scales, q)
        w = oracle.dequantize(oracle.Q6_K, blk, 1, 256)[0]
        assert np.array_equal(w, q.astype(np.float32))
    # a distinct scale per group: group of element 128h+32s+l is 8h+l/16+2s
    q = np.full(256, 1)
    sc = np.arange(1, 17)
    blk = pack_q6k_block(1.0, sc, q)
    w = oracle.dequantize(oracle.Q6_K, blk, 1, 256)[0]
    e = np.arange(256)
    h, s, l = e // 128, (e % 128) // 32, e % 32
    assert np.array_equal(w, sc[8 * h + l // 16 + 2 * s].astype(np.float32))


def test_nvfp4_every_code_scale_pair():
    """w = e2m1 * e4m3 * g for all 16 x 81 (code, scale) pairs, with both
    tables taken from ml_dtypes; e2m1 * e4m3 has at most six significant
    bits, so it is exact in fp16."""
    ml = pytest.importorskip("ml_dtypes")
    e2m1 = np.arange(16, dtype=np.uint8).view(ml.float4_e2m1fn).astype(np.float64)
    scodes = np.arange(0x08, 0x59, dtype=np.uint8)
    e4m3 = scodes.view(ml.float8_e4m3fn).astype(np.float64)
    g = 0.7109375
    K = 16 * 81
    codes = np.tile(np.arange(16), 81)
    row = pack_nvfp4_row(codes)
    w = oracle.dequantize(oracle.NVFP4, row, 1, K, scales=scodes[None, :], global_scale=g)[0]
    expect = (e2m1[codes] * np.repeat(e4m3, 16) * g).astype(np.float32)
    expect[expect == 0] = 0.0
    assert np.array_equal(w, expect)
    prod = np.outer(e2m1, e4m3).ravel()
    assert np.array_equal(prod.astype(np.float16).astype(np.float64), prod)
    nz = np.abs(prod[prod != 0])
    mant = nz / 2.0 ** np.floor(np.log2(nz))
    assert np.all(np.mod(mant * 32, 1) == 0)                 # <= 6 significant bits


def test_dequant_zero_sign_is_canonical():
    """-0 results (Q6_K with negative scale and q = 0; e2m1 code 8) come
    back as +0."""
    blk = pack_q6k_block(1.0, -np.ones(16, dtype=np.int64), np.zeros(256, dtype=np.int64))
    w = oracle.dequantize(oracle.Q6_K, blk, 1, 256)[0]
    assert np.all(w == 0) and not np.any(np.signbit(w))
    row = pack_nvfp4_row(np.full(16, 8))
    w = oracle.dequantize(oracle.NVFP4, row, 1, 16, scales=np.array([[0x38]], np.uint8),
                          global_scale=1.0)[0]
    assert np.all(w == 0) and not np.any(np.signbit(w))


def test_dequant_equals_any_float32_order_on_random_blocks():
    """Every K-quant weight is an exact product/difference before the final
    rounding, so evaluating the same fields in float32 in another order
    (fma-free numpy) gives the same bits."""
    rng = np.random.default_rng(5)
    for _ in range(20):
        d = np.float16(abs(rng.normal(0, 0.01)))
        dmin = np.float16(abs(rng.normal(0, 0.01)))
        sc = rng.integers(0, 64, 8)
        m = rng.integers(0, 64, 8)
        q = rng.integers(0, 16, 256)
        blk = pack_q4k_block(d, dmin, sc, m, q)
        w = oracle.dequantize(oracle.Q4_K, blk, 1, 256)[0]
        s = np.arange(256) // 32
        alt = (np.float32(d) * sc[s].astype(np.float32)) * q.astype(np.float32) \
            - np.float32(dmin) * m[s].astype(np.float32)
        alt = alt.astype(np.float32)
        alt[alt == 0] = 0.0
        assert np.array_equal(w.view(np.uint32), alt.view(np.uint32))


# ------------------------------------------------------------ the product

def _rand_matrix(qtype, M, K, seed):
    from skinny_gemm_q4_gb300 import synth
    return synth.weights(qtype, M, K, seed=seed, stream=qtype)


@pytest.mark.parametrize("qtype", [oracle.Q4_K, oracle.Q5_K, oracle.Q6_K, oracle.NVFP4])
def test_one_hot_brute_force_k256(qtype):
    """K = 256: x = 2^j e_k for every k gives y[m] = 2^j w[m][k] exactly,
    for every row.  Pins the product's row and column indexing."""
    M, K = 16, 256
    w, sc, g = _rand_matrix(qtype, M, K, seed=1)
    W = oracle.dequantize(qtype, w, M, K, scales=sc, global_scale=g)
    for j in (0, -3, 4):
        x = np.zeros((K, K), dtype=np.float16)
        x[np.arange(K), np.arange(K)] = np.float16(2.0 ** j)
        y, mag = oracle.qgemv(qtype, w, M, K, x, scales=sc, global_scale=g)
        assert np.array_equal(y, (2.0 ** j) * W.T.astype(np.float64))
        assert np.array_equal(mag, np.abs(y))


@pytest.mark.parametrize("qtype", [oracle.Q4_K, oracle.Q5_K, oracle.Q6_K, oracle.NVFP4])
def test_product_matches_torch_float64_matmul(qtype):
    import torch
    M, K, N = 24, 512 if qtype != oracle.NVFP4 else 640, 5
    w, sc, g = _rand_matrix(qtype, M, K, seed=2)
    W = oracle.dequantize(qtype, w, M, K, scales=sc, global_scale=g)
    from skinny_gemm_q4_gb300 import synth
    x = synth.activations(N, K, seed=2)
    y, mag = oracle.qgemv(qtype, w, M, K, x, scales=sc, global_scale=g)
    ref = torch.from_numpy(x.astype(np.float64)) @ torch.from_numpy(W.astype(np.float64)).T
    aref = torch.from_numpy(np.abs(x.astype(np.float64))) @ \
        torch.from_numpy(np.abs(W.astype(np.float64))).T
    assert np.allclose(y, ref.numpy(), rtol=0, atol=1e-12 * aref.numpy().max())
    assert np.allclose(mag, aref.numpy(), rtol=1e-13, atol=0)


def test_q4k_all_q_zero_gives_min_term():
    """All q = 0, uniform m and one dmin per matrix: y = -dmin * m * sum(x)."""
    M, K, N = 8, 1024, 3
    nb = K // 256
    w = np.stack([np.concatenate([pack_q4k_block(0.01171875, 0.0078125, [17] * 8, [37] * 8,
                                                 np.zeros(256, dtype=np.int64))
                                  for _ in range(nb)]) for _ in range(M)])
    from skinny_gemm_q4_gb300 import synth
    x = synth.activations(N, K, seed=4)
    y, _ = oracle.qgemv(oracle.Q4_K, w, M, K, x)
    expect = -0.0078125 * 37 * x.astype(np.float64).sum(axis=1)
    assert np.allclose(y, expect[:, None], rtol=1e-15, atol=1e-15)


def test_q6k_zero_code_gives_zero_and_nvfp4_zero_codes():
    K = 512
    blk = pack_q6k_block(0.5, np.arange(16) - 8, np.zeros(256, dtype=np.int64))
    w = np.concatenate([blk, blk])[None, :]
    from skinny_gemm_q4_gb300 import synth
    x = synth.activations(2, K, seed=5)
    y, _ = oracle.qgemv(oracle.Q6_K, w, 1, K, x)
    assert np.all(y == 0)
    codes = np.where(np.arange(K) % 3 == 0, 0, 8)
    row = pack_nvfp4_row(codes)[None, :]
    sc = np.full((1, K // 16), 0x40, dtype=np.uint8)
    y, _ = oracle.qgemv(oracle.NVFP4, row, 1, K, x, scales=sc, global_scale=0.75)
    assert np.all(y == 0)


@pytest.mark.parametrize("qtype", [oracle.Q4_K, oracle.Q6_K, oracle.NVFP4])
def test_linearity_sign_and_power_of_two(qtype):
    M, K, N = 12, 768 if qtype != oracle.NVFP4 else 800, 4
    w, sc, g = _rand_matrix(qtype, M, K, seed=6)
    from skinny_gemm_q4_gb300 import synth
    x = synth.activations(N, K, seed=6)
    y, mag = oracle.qgemv(qtype, w, M, K, x, scales=sc, global_scale=g)
    yn, _ = oracle.qgemv(qtype, w, M, K, -x, scales=sc, global_scale=g)
    assert np.array_equal(yn, -y)
    y2, mag2 = oracle.qgemv(qtype, w, M, K, (x.astype(np.float32) * 4).astype(np.float16),
                            scales=sc, global_scale=g)
    assert np.array_equal(y2, 4 * y) and np.array_equal(mag2, 4 * mag)


def test_residual_adds_and_enters_mag():
    M, K, N = 10, 512, 3
    w, sc, g = _rand_matrix(oracle.Q4_K, M, K, seed=8)
    from skinny_gemm_q4_gb300 import synth
    x = synth.activations(N, K, seed=8)
    r = synth.residual(N, M, seed=8)
    y, mag = oracle.qgemv(oracle.Q4_K, w, M, K, x)
    yr, magr = oracle.qgemv(oracle.Q4_K, w, M, K, x, residual=r)
    assert np.array_equal(yr, y + r.astype(np.float64))
    assert np.array_equal(magr, mag + np.abs(r.astype(np.float64)))


def test_sampled_rows_equal_full_matrix_rows():
    M, K, N = 40, 512, 2
    w, sc, g = _rand_matrix(oracle.Q5_K, M, K, seed=9)
    from skinny_gemm_q4_gb300 import synth
    x = synth.activations(N, K, seed=9)
    y, mag = oracle.qgemv(oracle.Q5_K, w, M, K, x)
    rows = np.array([39, 0, 17, 17, 5])
    ys, mags = oracle.qgemv(oracle.Q5_K, w, M, K, x, rows=rows)
    assert np.array_equal(ys, y[:, rows]) and np.array_equal(mags, mag[:, rows])


def test_row_bytes_match_block_sizes():
    """Block sizes printed on the pages: block_q4_K is 144 bytes and
    block_q6_K 210 bytes; Q5_K adds qh[32] to Q4_K (176)."""
    facts = _golden("block_sizes.json")
    assert oracle.row_bytes(oracle.Q4_K, 256) == facts["Q4_K"]
    assert oracle.row_bytes(oracle.Q6_K, 256) == facts["Q6_K"]
    assert oracle.row_bytes(oracle.Q5_K, 256) == facts["Q5_K"]
    assert oracle.row_bytes(oracle.Q6_K, 9728) == 7980
    assert oracle.row_bytes(oracle.NVFP4, 5120) == 2560


# --------------------------------------------------------------- SwiGLU
# reflex-llm "docs/kernels.md", SwiGLU section: output = silu(gate) x up,
# silu(x) = x / (1 + exp(-x)).

def test_silu_special_values_and_odd_part_identity():
    """silu(0) = 0; silu(x) - silu(-x) = x (x*s(x) + x*s(-x) = x, s the
    logistic); silu -> x for large x and -> 0 for large -x."""
    assert oracle.silu(0.0) == 0.0
    for v in np.linspace(-30, 30, 241):
        d = oracle.silu(v) - oracle.silu(-v)
        assert abs(d - v) <= 4 * np.finfo(np.float64).eps * max(1.0, abs(v)), v
    assert oracle.silu(50.0) == 50.0
    assert abs(oracle.silu(-50.0)) < 1e-19
    # silu(1) = 1 / (1 + 1/e)
    assert abs(oracle.silu(1.0) - 1.0 / (1.0 + np.exp(-1.0))) <= 2 ** -52


def test_silu_matches_torch_float64():
    torch = pytest.importorskip("torch")
    v = np.random.default_rng(5).normal(0.0, 6.0, size=4096)
    want = torch.nn.functional.silu(torch.from_numpy(v)).numpy()
    got = np.array([oracle.silu(a) for a in v])
    assert np.allclose(got, want, rtol=4 * np.finfo(np.float64).eps, atol=1e-300)


def test_swiglu_is_silu_of_gate_times_up():
    """oracle.swiglu against the definition with numpy's exp, elementwise;
    a planted sign mistake (exp(+v)) keeps the odd-part identity but is
    caught by the closed form silu(1) = 1 / (1 + 1/e)."""
    rng = np.random.default_rng(6)
    g = rng.normal(0, 4, size=(3, 257))
    u = rng.normal(0, 4, size=(3, 257))
    h = oracle.swiglu(g, u)
    want = g / (1.0 + np.exp(-g)) * u
    assert np.allclose(h, want, rtol=4 * np.finfo(np.float64).eps, atol=0)
    bad = lambda v: v / (1.0 + np.exp(v))
    assert abs(bad(1.0) - 1.0 / (1.0 + np.exp(-1.0))) > 0.1


def test_qgemv_swiglu_combines_the_two_products():
    from packers import pack_q4k_block
    M, K = 3, 256
    blk = pack_q4k_block(0.25, 0.0, [1] * 8, [0] * 8, np.full(256, 2, dtype=np.int64))
    wg = np.tile(blk, (M, 1))
    blk_u = pack_q4k_block(0.5, 0.0, [1] * 8, [0] * 8, np.full(256, 1, dtype=np.int64))
    wu = np.tile(blk_u, (M, 1))
    x = np.zeros((1, K), dtype=np.float16)
    x[0, 0] = 1.0  # g = 0.25 * 2 = 0.5, u = 0.5
    h, g, mg, u, mu = oracle.qgemv_swiglu(oracle.Q4_K, wg, oracle.Q4_K, wu, M, K, x)
    assert np.all(g == 0.5) and np.all(u == 0.5)
    assert np.allclose(h, 0.5 / (1 + np.exp(-0.5)) * 0.5, rtol=1e-15)


# --------------------------------------------------------- FP8 block-scaled
# TandemLLM "Kernels", FP8 matrix products: e4m3 codes with one BF16 scale
# per 128 by 128 block.

def test_bf16_decode_matches_numpy_and_torch_all_codes():
    torch = pytest.importorskip("torch")
    codes = np.arange(65536, dtype=np.uint32)
    want = (codes << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    got = np.array([oracle.bf16_to_f64(int(c)) for c in codes])
    fin = np.isfinite(want)
    assert np.array_equal(got[fin], want[fin])
    assert np.all(np.isnan(got[np.isnan(want)]))
    t = torch.from_numpy(codes.astype(np.int32).astype(np.int16)).view(torch.bfloat16)
    assert np.array_equal(got[fin], t.double().numpy()[fin])


def test_fp8_closed_form_blocks_and_scale_indexing():
    """Rows 0..129 (two row blocks) x K = 512 (four k blocks), every weight a
    known e4m3 value times its block's scale; the scale of (m, k) is
    scales[m // 128][k // 128] (a planted transpose of the block index fails)."""
    from packers import bf16_bits, e4m3_code
    M, K = 130, 512
    vals = [0.0, 1.0, -2.0, 448.0, -448.0, 2.0 ** -9, 0.875, 13.0, -0.015625, 240.0]
    rng = np.random.default_rng(7)
    V = np.array(vals)[rng.integers(0, len(vals), size=(M, K))]
    codes = np.vectorize(e4m3_code)(V).astype(np.uint8)
    svals = np.array([[0.25, 3.0, -1.5, 2.0 ** -12], [8.0, 0.125, 1.0, -4.0]])
    scales = np.vectorize(bf16_bits)(svals.astype(np.float32)).astype(np.uint16)
    W = oracle.dequantize(oracle.FP8, codes, M, K, scales=scales)
    expect = V * svals[np.arange(M)[:, None] // 128, np.arange(K)[None, :] // 128]
    assert np.array_equal(W.astype(np.float64), expect)
    wrong = V * svals.T[np.arange(K)[None, :] // 128 % 2, np.arange(M)[:, None] // 128 * 0]
    assert not np.array_equal(W.astype(np.float64), wrong)


def test_fp8_generator_has_no_nan_codes():
    from skinny_gemm_q4_gb300 import synth
    codes, scales, g = synth.fp8_weights(256, 1024, seed=3)
    assert codes.shape == (256, 1024) and scales.shape == (2, 8) and g == 1.0
    assert not np.any((codes & 0x7F) == 0x7F)
    assert len(np.unique(codes)) == 254
    W = oracle.dequantize(oracle.FP8, codes, 256, 1024, scales=scales)
    assert np.isfinite(W).all()


@pytest.mark.parametrize("qtype", [oracle.FP8])
def test_fp8_one_hot_and_torch_matmul(qtype):
    import torch
    M, K = 130, 256
    w, sc, g = _rand_matrix(qtype, M, K, seed=1)
    W = oracle.dequantize(qtype, w, M, K, scales=sc, global_scale=g)
    x = np.eye(K, dtype=np.float16) * np.float16(0.5)
    y, _ = oracle.qgemv(qtype, w, M, K, x, scales=sc, global_scale=g)
    assert np.array_equal(y, 0.5 * W.T.astype(np.float64))
    from skinny_gemm_q4_gb300 import synth
    x = synth.activations(5, K, seed=2)
    y, mag = oracle.qgemv(qtype, w, M, K, x, scales=sc, global_scale=g)
    ref = torch.from_numpy(x.astype(np.float64)) @ torch.from_numpy(W.astype(np.float64)).T
    aref = torch.from_numpy(np.abs(x.astype(np.float64))) @ \
        torch.from_numpy(np.abs(W.astype(np.float64))).T
    assert np.allclose(y, ref.numpy(), rtol=0, atol=1e-12 * aref.numpy().max())
