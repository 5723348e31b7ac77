"""Pins of the CPU oracle against facts fixed outside it (no GPU).

Each test checks the oracle against the format definitions the pages name, values
the pages print, closed forms, special cases that reduce to a library routine, or
brute force on tiny inputs.  A plausible mistake in the oracle (a dropped term, a
wrong sign or index, a transposed operand, a wrong tie rule) fails one of them.
"""
import ctypes
import json
import math
import os

import numpy as np
import pytest
import torch

import csa2_inputs as gen

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def _fnptr(orc, name):
    return ctypes.cast(getattr(orc.lib(), name), ctypes.c_void_p)


# ------------------------------------------------------------------ E2M1 -----------

def test_e2m1_value_set_and_round_trip(orc):
    g = _gold("e2m1_values.json")
    mags = {int(k): v for k, v in g["code_to_magnitude"].items()}
    for c in range(16):
        want = mags[c & 7] * (-1.0 if c & 8 else 1.0)
        got = orc.lib().orc_e2m1_decode(c)
        assert got == want and math.copysign(1.0, got) == math.copysign(1.0, want) or (want == 0 and got == 0)
        # every representable value re-encodes to its own code (negative zero keeps its sign)
        assert orc.lib().orc_e2m1_encode(ctypes.c_float(got)) == c
    values = sorted({abs(orc.lib().orc_e2m1_decode(c)) for c in range(16)})
    assert values == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_exhaustive_vs_brute_force(orc, pins_lib):
    """Every float32 bit pattern: oracle decision table == nearest magnitude, ties to even."""
    mag = (ctypes.c_double * 8)(*[0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    bad = ctypes.c_uint32()
    n_bad = pins_lib.pin_e2m1_sweep(_fnptr(orc, "orc_e2m1_encode"), mag, os.cpu_count() or 4,
                                    ctypes.byref(bad))
    assert n_bad == 0, f"{n_bad} mismatches, first pattern 0x{bad.value:08x}"


# ------------------------------------------------------------------ E4M3 -----------

def _e4m3_table_from_torch():
    codes = torch.arange(256, dtype=torch.uint8)
    vals = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return vals


def test_e4m3_decode_matches_torch_and_anchors(orc):
    vals = _e4m3_table_from_torch()
    for c in range(256):
        got = orc.lib().orc_e4m3_decode(c)
        if c in (0x7F, 0xFF):
            assert math.isnan(got) and math.isnan(vals[c])
        else:
            assert got == vals[c], hex(c)
    for a in _gold("e4m3_anchors.json")["anchors"]:
        assert orc.lib().orc_e4m3_encode(ctypes.c_float(a["value"])) == int(a["code"], 16)
        assert orc.lib().orc_e4m3_decode(int(a["code"], 16)) == a["value"]


def test_e4m3_exhaustive_vs_nearest(orc, pins_lib):
    """Every finite non-negative float32: oracle == nearest finite E4M3 value (ties to
    even code, saturating at 448).  The value table is torch's float8_e4m3fn decode."""
    vals = _e4m3_table_from_torch()[:127]
    assert np.all(np.diff(vals) > 0)
    tab = (ctypes.c_double * 127)(*vals.tolist())
    bad = ctypes.c_uint32()
    n_bad = pins_lib.pin_e4m3_sweep(_fnptr(orc, "orc_e4m3_encode"), tab, os.cpu_count() or 4,
                                    ctypes.byref(bad))
    assert n_bad == 0, f"{n_bad} mismatches, first pattern 0x{bad.value:08x}"


def test_e4m3_full_brute_force_sample(orc, pins_lib):
    """All 127 candidates compared, on random patterns of both signs."""
    vals = _e4m3_table_from_torch()[:127]
    tab = (ctypes.c_double * 127)(*vals.tolist())
    rng = np.random.default_rng(7)
    pats = np.concatenate([rng.integers(0, 2**32, 2_000_000, dtype=np.uint64).astype(np.uint32),
                           np.array([0x80000000, 0x3F880000, 0xBF880000], np.uint32)])
    bad = ctypes.c_uint32()
    n_bad = pins_lib.pin_e4m3_brute(_fnptr(orc, "orc_e4m3_encode"), tab,
                                    pats.ctypes.data_as(ctypes.POINTER(ctypes.c_uint32)), pats.size,
                                    ctypes.byref(bad))
    assert n_bad == 0, f"first bad 0x{bad.value:08x}"


def test_e4m3_encode_matches_torch_in_range(orc):
    """torch's float32 -> float8_e4m3fn cast rounds to nearest even; inside the finite
    range it must agree with the oracle bit for bit."""
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.uniform(0, 448, 500_000), np.exp(rng.uniform(-25, 6, 500_000))])
    x = x[x <= 448].astype(np.float32)
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = orc.e4m3_encode(x)
    assert np.array_equal(got, want)


# ------------------------------------------------------------------ blocks ---------

def test_quant_blocks_worked_by_hand(orc):
    for blk in _gold("quant_blocks.json")["blocks"]:
        x = np.array(blk["x"], dtype=np.float32).reshape(1, 16)
        codes, scales = orc.quantize(x)
        assert scales[0, 0] == int(blk["scale"], 16), blk["name"]
        assert [int(c, 16) for c in blk["codes"]] == codes[0].tolist(), blk["name"]


def test_quant_block_properties(orc):
    """On latent-like data: each block's largest code magnitude is 5, 6 or 7 unless the
    scale is zero; dequantised error stays within half an E2M1 step of y times s."""
    gains = gen.latent_gains(0)
    x = gen.latent_rows(0, 0, 0, np.arange(256), gains)
    codes, scales = orc.quantize(x)
    deq = orc.dequantize(codes, scales)
    nib = np.stack([codes & 0xF, codes >> 4], axis=-1).reshape(256, 512)
    mag = (nib & 7).reshape(256, 32, 16).max(axis=-1)
    s = orc.e4m3_decode(scales.ravel()).reshape(256, 32)
    assert np.all((mag >= 5) | (s == 0))
    # E2M1 gaps: half-step at |y| <= 2 is 0.25, <= 4 is 0.5, <= 6 is 1
    y = np.abs(x.astype(np.float64)) / np.repeat(s, 16, axis=1)
    half = np.where(y <= 2, 0.25, np.where(y <= 4, 0.5, 1.0))
    err = np.abs(x - deq) / np.repeat(s, 16, axis=1)
    assert np.all(err <= half * (1 + 1e-6))


def test_dequant_is_exact_product(orc):
    """Every (code, scale) pair decodes to e2m1 x e4m3, which float32 holds exactly."""
    e2 = np.array([orc.lib().orc_e2m1_decode(c) for c in range(16)])
    e4 = np.array([orc.lib().orc_e4m3_decode(b) for b in range(127)])
    prod = np.outer(e4, e2)
    assert np.array_equal(prod.astype(np.float32).astype(np.float64), prod)
    codes = np.arange(256, dtype=np.uint8).reshape(1, 256).repeat(127, 0)
    codes = np.concatenate([codes, codes], axis=1)[:, :256]
    scales = np.repeat(np.arange(127, dtype=np.uint8).reshape(127, 1), 32, axis=1)
    deq = orc.dequantize(codes, scales)
    for r in (0, 1, 56, 126):
        for c in range(0, 512, 37):
            byte = codes[r, c // 2]
            code = (byte >> 4) if c % 2 else (byte & 0xF)
            assert deq[r, c] == e2[code] * e4[r]


# ------------------------------------------------------------------ MXFP4 variant --
# The OCP Microscaling definition the oracle reads "MXFP4 (E2M1)" as: 32-element blocks,
# E8M0 scale 2^(floor(log2 amax) - emax_elem) with emax_elem = 2 for E2M1 (largest
# power of two 4), elements E2M1 round-to-nearest-even and saturating.

def test_mx_scale_rule_closed_forms(orc):
    """Scale bytes worked by hand from the definition (byte = exponent + 127)."""
    cases = {1.0: 125, 1.5: 125, 0.75: 124, 3.0: 126, 3.999: 126, 4.0: 127, 6.0: 127,
             7.99: 127, 8.0: 128, 100.0: 131, 2.0**-20: 105, 2.0**-125: 0, 2.0**-130: 0,
             1.0e38: 251, 0.0: 0}
    for amax, b in cases.items():
        assert orc.e8m0_scale_for(amax) == b, amax
    # library cross-check away from exact powers of two
    rng = np.random.default_rng(7)
    for amax in np.exp(rng.uniform(-40, 40, 200)).astype(np.float32):
        assert orc.e8m0_scale_for(float(amax)) == int(np.floor(np.log2(np.float64(amax)))) - 2 + 127
    assert list(orc.e8m0_decode([0, 125, 127, 130])) == [2.0**-127, 0.25, 1.0, 8.0]


def test_mx_block_worked_by_hand(orc):
    """amax 6.1 -> X = 2^(2-2) = 1: the elements are coded as plain E2M1 values."""
    x = np.zeros((1, 64), np.float32)
    x[0, :10] = [3.0, -1.5, 0.5, 2.9, 0.2, -0.3, 5.9, 6.1, -5.0, 0.25]
    # second block: amax 0.3 -> X = 2^(-2-2) = 1/16, y = 16 x
    x[0, 32:36] = [0.3, -0.0625, 0.01, 0.2]
    codes, scales = orc.mx_quantize(x)
    assert scales.tolist() == [[127, 123]]
    nib = np.stack([codes[0] & 0xF, codes[0] >> 4], -1).ravel()
    # 3 -> 3 (0b101), -1.5 -> -1.5, 0.5, 2.9 -> 3, 0.2 -> 0, -0.3 -> -0.5, 5.9 -> 6,
    # 6.1 -> 6 (saturated), -5 -> -4 (tie to the even code), 0.25 -> 0 (tie to even)
    assert nib[:10].tolist() == [0x5, 0xB, 0x1, 0x5, 0x0, 0x9, 0x7, 0x7, 0xE, 0x0]
    # 4.8 -> 4 (0b110), -1 -> 0b1010, 0.16 -> 0, 3.2 -> 3
    assert nib[32:36].tolist() == [0x6, 0xA, 0x0, 0x5]
    assert not nib[10:32].any() and not nib[36:].any()
    deq = orc.mx_dequantize(codes, scales)
    assert deq[0, :10].tolist() == [3.0, -1.5, 0.5, 3.0, 0.0, -0.5, 6.0, 6.0, -4.0, 0.0]
    assert deq[0, 32:36].tolist() == [0.25, -0.0625, 0.0, 0.1875]


def test_mx_zero_and_tiny_blocks(orc):
    x = np.zeros((2, 32), np.float32)
    x[1, 0] = 2.0**-130  # below E8M0's range: the scale clamps to 2^-127, y = 1/8 -> 0
    x[1, 1] = -(2.0**-127) * 0.75  # y = -0.75 -> -1 (tie to the even code 0b010)
    codes, scales = orc.mx_quantize(x)
    assert scales[0, 0] == 0 and not codes[0].any()
    assert scales[1, 0] == 0
    assert (codes[1, 0] & 0xF) == 0x0 and (codes[1, 0] >> 4) == 0xA


def test_mx_block_properties_on_latent_rows(orc):
    """Every nonzero block's largest element is coded 4 or 6 (y_max in [4, 8)); the error
    is at most half an E2M1 step times X below 6 and y - 6 above it."""
    gains = gen.latent_gains(0)
    x = gen.latent_rows(0, 0, 0, np.arange(128), gains)
    codes, scales = orc.mx_quantize(x)
    deq = orc.mx_dequantize(codes, scales)
    nib = np.stack([codes & 0xF, codes >> 4], axis=-1).reshape(128, 512)
    mag = (nib & 7).reshape(128, 16, 32).max(axis=-1)
    assert np.all(mag >= 6)
    X = np.repeat(orc.e8m0_decode(scales.ravel()).reshape(128, 16), 32, axis=1)
    y = np.abs(x.astype(np.float64)) / X
    assert np.all(y < 8)
    half = np.where(y <= 2, 0.25, np.where(y <= 4, 0.5, 1.0))
    bound = np.where(y <= 6, half, y - 6)
    err = np.abs(x - deq) / X
    assert np.all(err <= bound * (1 + 1e-9) + 1e-12)


def test_mx_against_e4m3_footprint_and_error(orc):
    """Same latent rows through both formats: MX stores 272 B per 512 channels against
    288 B, and its power-of-two, 32-wide scales cost accuracy."""
    gains = gen.latent_gains(1)
    x = gen.latent_rows(1, 0, 0, np.arange(256), gains).astype(np.float64)
    c4, s4 = orc.quantize(x.astype(np.float32))
    cm, sm = orc.mx_quantize(x.astype(np.float32))
    assert c4.shape[1] + s4.shape[1] == 288 and cm.shape[1] + sm.shape[1] == 272
    e4 = np.sqrt(np.mean((orc.dequantize(c4, s4) - x) ** 2)) / np.sqrt(np.mean(x ** 2))
    em = np.sqrt(np.mean((orc.mx_dequantize(cm, sm) - x) ** 2)) / np.sqrt(np.mean(x ** 2))
    assert 0.05 < e4 < em < 0.3, (e4, em)


# ------------------------------------------------------------------ persistent tier --

def test_pack_pages_worked_by_hand(orc):
    """Two pages with recognisable bytes: each record is the page's 64 code rows, then its
    64 scale rows, then its 64 keys as little-endian bf16; a bad id gives zeros."""
    slots = 3 * 64
    codes = (np.arange(slots * 256) % 251).astype(np.uint8).reshape(slots, 256)
    scales = (np.arange(slots * 16) % 13 + 100).astype(np.uint8).reshape(slots, 16)
    keys = (np.arange(slots * 128) * 7 + 0x1234).astype(np.uint16).reshape(slots, 128)
    packed = orc.pack_pages(codes, scales, keys, [2, 0, 7])
    rec = 64 * (256 + 16 + 256)
    assert packed.shape == (3 * rec,)
    r0 = packed[:rec]
    assert r0[0] == codes[128, 0] and r0[64 * 256 - 1] == codes[191, 255]
    assert r0[64 * 256] == scales[128, 0] and r0[64 * 256 + 64 * 16 - 1] == scales[191, 15]
    k0 = 64 * 256 + 64 * 16
    assert r0[k0] == keys[128, 0] & 0xFF and r0[k0 + 1] == keys[128, 0] >> 8
    assert r0[rec - 1] == keys[191, 127] >> 8
    assert np.array_equal(packed[rec:rec + 64 * 256], codes[:64].ravel())
    assert not packed[2 * rec:].any()


# ------------------------------------------------------------------ projection -----

def _bf16(x):
    return gen.f32_to_bf16_bits(np.asarray(x, np.float32))


def test_projection_identity_reproduces_codec(orc):
    """W = [I_512; 0] makes C = H[:, :512] exactly, so the write path's codes must equal
    the block quantiser applied to H's first 512 columns (tech-report digest CED equation)."""
    rng = np.random.default_rng(11)
    H = _bf16(rng.standard_normal((24, 640)) * 3)
    Wt = np.zeros((512 + 128, 640), np.uint16)
    Wt[np.arange(512), np.arange(512)] = 0x3F80                       # 1.0 in bf16
    Wt[512 + np.arange(128), 512 + np.arange(128)] = 0x3F80
    codes, scales, keys, C = orc.kv_write_rows(H, Wt, 1, 1)
    Hf = gen.bf16_bits_to_f32(H)
    c2, s2 = orc.quantize(Hf[:, :512].copy())
    assert np.array_equal(codes[0], c2) and np.array_equal(scales[0], s2)
    assert np.array_equal(keys[0], H[:, 512:640])                       # bf16 -> fp32 -> bf16 round trip


def test_projection_one_hot_columns_and_library_gemm(orc):
    rng = np.random.default_rng(12)
    H = _bf16(rng.standard_normal((8, 256)))
    Wt = _bf16(rng.standard_normal((64, 256)) / 16)
    perm = rng.permutation(256)[:16]
    Wt[:16] = 0
    Wt[np.arange(16), perm] = 0x3F80
    C = orc.project(H, Wt)
    Hf = gen.bf16_bits_to_f32(H).astype(np.float64)
    Wf = gen.bf16_bits_to_f32(Wt).astype(np.float64)
    assert np.array_equal(C[:, :16], Hf[:, perm].astype(np.float32))  # selects H's columns, not rows
    ref = Hf @ Wf.T                                                     # library GEMM in float64
    np.testing.assert_allclose(C, ref.astype(np.float32), rtol=1e-6, atol=1e-7)


def _bf16_ties():
    """fp32 patterns whose low 16 bits are exactly half a bf16 unit (0x8000), over upper
    halves with an even and an odd last bit, both signs, normal and subnormal exponents,
    plus the patterns one below and one above each tie."""
    uppers = np.array([0x3F80, 0x3F81, 0x3F82, 0x3F83, 0x4000, 0x4001, 0x7F7E, 0x0000, 0x0001,
                       0x0080, 0x0081, 0x1234, 0x1235, 0x4B7F, 0x4B80], np.uint32)
    uppers = np.concatenate([uppers, uppers | 0x8000])
    ties = (uppers << 16) | 0x8000
    return np.concatenate([ties, ties - 1, ties + 1]).view(np.float32)


def test_bf16_store_worked_by_hand(orc):
    """The indexer-key store is fp32 -> bf16 round-to-nearest, ties to even (tech-report
    digest "Causal Encoder-Decoder (CED) アーキテクチャ": the keys are the projection C_l,
    held as bf16).  bf16 keeps 8 significant bits, so at 1.0 one unit is 2^-7:
      1 + 2^-8     lies halfway between 1 (even) and 1 + 2^-7 (odd)      -> 0x3F80
      1 + 3*2^-8   halfway between 1 + 2^-7 (odd) and 1 + 2^-6 (even)    -> 0x3F82
      1 + 2^-8 + 2^-23  just above the first tie                          -> 0x3F81
      -(1 + 2^-8)  the same tie, negative                                 -> 0xBF80
      3.39e38 (0x7F7F8000): halfway to the next power, even side is 0x7F80 = inf
      the smallest positive subnormal rounds to 0, 2^-133 (subnormal, exact in bf16) stays."""
    x = np.array([1 + 2.0**-8, 1 + 3 * 2.0**-8, 1 + 2.0**-8 + 2.0**-23, -(1 + 2.0**-8)],
                 np.float32)
    assert orc.f32_to_bf16_bits(x).tolist() == [0x3F80, 0x3F82, 0x3F81, 0xBF80]
    big = np.array([0x7F7F8000, 0x7F7E8000], np.uint32).view(np.float32)
    assert orc.f32_to_bf16_bits(big).tolist() == [0x7F80, 0x7F7E]
    sub = np.array([0x00000001, 0x00008000, 0x00018000, 0x00010000], np.uint32).view(np.float32)
    assert orc.f32_to_bf16_bits(sub).tolist() == [0x0000, 0x0000, 0x0002, 0x0001]


def test_bf16_store_matches_torch(orc):
    """Against the library's own fp32 -> bf16 conversion (round to nearest even), bit for
    bit, on 2^21 random finite fp32 patterns (every exponent) and on the exact ties."""
    import torch
    rng = np.random.default_rng(21)
    u = rng.integers(0, 2**32, size=1 << 21, dtype=np.uint64).astype(np.uint32)
    u = u[(u & 0x7F800000) != 0x7F800000]                    # finite only
    x = np.concatenate([u.view(np.float32), _bf16_ties()])
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = orc.f32_to_bf16_bits(x)
    bad = np.flatnonzero(got != want)
    assert bad.size == 0, f"{bad.size} mismatches, first fp32 {x[bad[:4]].view(np.uint32)}"


def test_write_path_keys_round_the_fp32_projection(orc):
    """Keys of the write path are bf16(fl32(sum)) of sums that are not bf16 values: two
    nonzero weights per column put C = H[:, a] + H[:, b] / 3 between bf16 neighbours, and the
    stored key must equal torch's rounding of the oracle's fp32 C."""
    import torch
    rng = np.random.default_rng(22)
    H = _bf16(rng.standard_normal((16, 256)))
    Wt = np.zeros((128, 256), np.uint16)
    a, b = rng.permutation(256)[:128], rng.permutation(256)[:128]
    Wt[np.arange(128), a] = 0x3F80                      # 1.0
    Wt[np.arange(128), b] = _bf16(np.float32(1 / 3))    # bf16(1/3), 8 significant bits
    codes, scales, keys, C = orc.kv_write_rows(H, Wt, 0, 1)
    want = torch.from_numpy(C.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy()
    assert np.array_equal(keys[0], want.view(np.uint16))
    assert np.mean(gen.bf16_bits_to_f32(keys[0]) != C) > 0.9   # the rounding is exercised


# ------------------------------------------------------------------ indexer --------

def test_index_score_special_cases(orc):
    """One-hot keys read off one coordinate of each head: score = sum_h max(0, q[h, d])
    (ReLU per head, then a sum over the 4 heads; no transposition of q)."""
    rng = np.random.default_rng(5)
    q = _bf16(rng.standard_normal((4, 128)))
    keys = np.zeros((128, 128), np.uint16)
    keys[np.arange(128), np.arange(128)] = 0x3F80
    s = orc.index_scores(q, keys)
    qf = gen.bf16_bits_to_f32(q).astype(np.float64)
    assert np.array_equal(s, np.maximum(qf, 0).sum(axis=0))
    # doubling a key doubles the score (exact in bf16 and double)
    k = _bf16(rng.standard_normal((16, 128)))
    k2 = _bf16(gen.bf16_bits_to_f32(k) * 2)
    assert np.array_equal(orc.index_scores(q, k2), 2 * orc.index_scores(q, k))
    # permuting heads leaves scores unchanged; negating q flips which heads contribute
    assert np.array_equal(orc.index_scores(q[[2, 0, 3, 1]], k), orc.index_scores(q, k))
    neg = q ^ np.uint16(0x8000)
    both = orc.index_scores(q, k) + orc.index_scores(neg, k)
    dots = np.abs(qf @ gen.bf16_bits_to_f32(k).astype(np.float64).T).sum(axis=0)
    np.testing.assert_allclose(both, dots, rtol=1e-12)


def _brute_topk(scores, tokens, k):
    order = sorted(range(len(scores)), key=lambda i: (-scores[i], tokens[i]))
    sel = sorted(tokens[i] for i in order[:k])
    return np.array(sel + [-1] * (k - len(sel)), np.int32)


@pytest.mark.parametrize("n,k", [(1, 4), (5, 5), (17, 4), (64, 16), (64, 64), (40, 100)])
def test_select_topk_brute_force_with_ties(orc, n, k):
    rng = np.random.default_rng(n * 131 + k)
    scores = rng.integers(0, 4, n).astype(np.float64)      # many exact ties, zeros like ReLU
    tokens = np.sort(rng.choice(1000, n, replace=False)).astype(np.int32)
    assert np.array_equal(orc.select_topk(scores, tokens, k), _brute_topk(scores, tokens, k))


def test_full_mode_pool_contains_topk_and_small_context(orc):
    rng = np.random.default_rng(9)
    keys = _bf16(rng.standard_normal((300, 128)))
    q = _bf16(rng.standard_normal((4, 128)))
    idx, pool, s = orc.index_full(q, keys, 32, 128)
    assert set(idx[idx >= 0]) <= set(pool[pool >= 0])
    assert np.all(np.diff(idx) > 0) and np.all(np.diff(pool) > 0)
    assert s[idx].min() >= np.sort(s)[-32]
    # N <= K selects every token
    idx2, pool2, _ = orc.index_full(q, keys[:20], 32, 128)
    assert np.array_equal(idx2[:20], np.arange(20)) and np.all(idx2[20:] == -1)


def test_reindex_restricted_to_pool_and_equal_to_full(orc):
    """Page 5 Hierarchical Sparse Indexer: Reindex searches only the pool.  With the
    Full layer's own query, Reindex over its pool returns Full's top-K exactly."""
    rng = np.random.default_rng(10)
    keys = _bf16(rng.standard_normal((2000, 128)))
    qf = _bf16(rng.standard_normal((4, 128)))
    idx_full, pool, _ = orc.index_full(qf, keys, 64, 512)
    idx_re, _ = orc.index_reindex(qf, keys, pool, 64)
    assert np.array_equal(idx_re, idx_full)
    q2 = _bf16(rng.standard_normal((4, 128)))
    idx2, _ = orc.index_reindex(q2, keys, pool, 64)
    assert set(idx2[idx2 >= 0]) <= set(pool)
    small = pool.copy()
    small[40:] = -1
    idx3, _ = orc.index_reindex(q2, keys, small, 64)
    assert np.array_equal(idx3[:40], small[:40]) and np.all(idx3[40:] == -1)


def test_reuse_passes_indices_through(orc):
    x = np.array([3, 9, 27, -1], np.int32)
    assert np.array_equal(orc.index_reuse(x), x)


# ------------------------------------------------------------------ attention ------

def test_attention_dense_case_matches_library_sdpa(orc):
    """K = N: sparse attention over every row equals dense scaled-dot-product attention
    (torch's library routine, float64)."""
    rng = np.random.default_rng(21)
    q = _bf16(rng.standard_normal((16, 512)))
    chat = rng.standard_normal((70, 512)).round(3)
    scale = np.float32(1 / math.sqrt(512))
    out, lse = orc.sparse_attention(q, chat, float(scale))
    qt = torch.from_numpy(gen.bf16_bits_to_f32(q).astype(np.float64)).view(1, 16, 512)
    kt = torch.from_numpy(chat).view(1, 1, 70, 512).expand(1, 16, 70, 512)
    ref = torch.nn.functional.scaled_dot_product_attention(qt.view(1, 16, 1, 512), kt, kt,
                                                           scale=float(scale)).view(16, 512)
    np.testing.assert_allclose(out, ref.numpy().astype(np.float32), rtol=2e-6, atol=1e-6)
    ref_lse = torch.logsumexp(float(scale) * (qt.view(16, 512) @ torch.from_numpy(chat).T), dim=-1)
    np.testing.assert_allclose(lse, ref_lse.numpy().astype(np.float32), rtol=1e-6)


def test_attention_closed_forms(orc):
    rng = np.random.default_rng(22)
    q = _bf16(rng.standard_normal((16, 512)))
    row = rng.standard_normal(512)
    # all rows equal -> output is that row, lse = scale*q.row + ln n
    out, lse = orc.sparse_attention(q, np.tile(row, (9, 1)), 0.05)
    np.testing.assert_allclose(out, np.tile(row, (16, 1)).astype(np.float32), rtol=1e-6, atol=1e-7)
    qf = gen.bf16_bits_to_f32(q).astype(np.float64)
    np.testing.assert_allclose(lse, (0.05 * qf @ row + math.log(9)).astype(np.float32), rtol=1e-6)
    # q = 0 -> mean of the rows
    chat = rng.standard_normal((13, 512))
    out0, lse0 = orc.sparse_attention(np.zeros((16, 512), np.uint16), chat, 0.05)
    np.testing.assert_allclose(out0, np.tile(chat.mean(0), (16, 1)).astype(np.float32), rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(lse0, np.float32(math.log(13)), rtol=1e-7)
    # a single row -> that row; no rows -> zeros and -inf
    out1, _ = orc.sparse_attention(q, chat[4:5], 0.05)
    assert np.array_equal(out1, np.tile(chat[4].astype(np.float32), (16, 1)))
    outn, lsen = orc.sparse_attention(q, np.zeros((0, 512)), 0.05)
    assert np.all(outn == 0) and np.all(np.isneginf(lsen))
    # row order does not matter
    perm = rng.permutation(13)
    o_a, _ = orc.sparse_attention(q, chat, 0.05)
    o_b, _ = orc.sparse_attention(q, chat[perm], 0.05)
    np.testing.assert_allclose(o_a, o_b, rtol=1e-6, atol=1e-7)


def test_attention_over_cache_gathers_by_hand(orc):
    """The cache-level oracle: select rows by index (skipping -1), decode each code from the
    E2M1 magnitude table and its scale (E4M3 / 16, or E8M0 = 2^(b - 127) / 32) by hand,
    and attend; duplicates count once per occurrence, an all -1 selection gives zeros."""
    mag = {int(k): v for k, v in _gold("e2m1_values.json")["code_to_magnitude"].items()}
    rng = np.random.default_rng(31)
    n = 40
    codes = rng.integers(0, 256, (n, 256), dtype=np.uint8)
    q = _bf16(rng.standard_normal((16, 512)) * 0.2)

    def by_hand(row_ids, scale_of):
        rows = np.zeros((len(row_ids), 512))
        for i, r in enumerate(row_ids):
            for c in range(512):
                nib = (codes[r, c // 2] >> (4 * (c % 2))) & 0xF
                v = mag[nib & 7] * (-1.0 if nib & 8 else 1.0)
                rows[i, c] = v * scale_of(r, c)
        return rows

    idx = np.array([7, -1, 3, 39, 7, -1, 0], np.int32)
    sel = [7, 3, 39, 7, 0]
    e4 = rng.integers(0x20, 0x50, (n, 32), dtype=np.uint8)  # normal E4M3 scales
    e4_val = lambda b: 2.0 ** ((int(b) >> 3) - 7) * (1 + (int(b) & 7) / 8)
    out, lse = orc.attention_over_cache(q, codes, e4, idx, 0.07)
    ref_o, ref_l = orc.sparse_attention(q, by_hand(sel, lambda r, c: e4_val(e4[r, c // 16])), 0.07)
    assert np.array_equal(out, ref_o) and np.array_equal(lse, ref_l)

    e8 = rng.integers(120, 135, (n, 16), dtype=np.uint8)
    out, lse = orc.attention_over_cache(q, codes, e8, idx, 0.07, mx=True)
    ref_o, ref_l = orc.sparse_attention(q, by_hand(sel, lambda r, c: 2.0 ** (int(e8[r, c // 32]) - 127)),
                                        0.07)
    assert np.array_equal(out, ref_o) and np.array_equal(lse, ref_l)

    out, lse = orc.attention_over_cache(q, codes, e4, np.full(5, -1, np.int32), 0.07)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


def test_attention_large_logit_stability(orc):
    """exp never overflows: a huge logit gap gives one-hot weights."""
    q = _bf16(np.full((16, 512), 4.0))
    chat = np.zeros((3, 512))
    chat[1] = 50.0
    out, _ = orc.sparse_attention(q, chat, 1.0)
    assert np.all(np.isfinite(out)) and np.allclose(out, 50.0)


# ------------------------------------------------------------------ footprint ------

def test_footprint_arithmetic_printed_on_pages(orc):
    g = _gold("footprint.json")
    b = g["bytes_per_token"]
    assert b == orc.PAGES_FOOTPRINT
    assert orc.session_bytes(b["v4.1-flash"], g["session_tokens"]) == g["session_MB_printed"] * 10**6
    assert round(orc.session_bytes(b["v4.1-flash"]) / 1e9, 2) == g["session_GB_printed"]
    assert round(orc.session_bytes(b["v4-flash"]) / 1e9, 1) == g["v4flash_session_GB_printed"]
    assert round(b["v4-flash"] / b["v4.1-flash"], 1) == g["ratio_vs_v4flash_printed"]
    assert round(b["v4-flash"] / b["v4.1-flash"]) == 4
    assert round(b["v1"] / b["v4.1-flash"]) == g["ratio_vs_v1_printed"]
    # this layout: 256 B codes + 32 B scales + 256 B bf16 keys per Full group
    assert orc.layout_bytes_per_token(1) == 544
    assert orc.layout_bytes_per_token(5) == 2720
