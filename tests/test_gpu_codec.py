"""K4 codec parity: FP4 codes and E4M3 scales bit-exact against the oracle on the
same float32 inputs (format: ai2.x.ezic.info blog, "KVを捨てる、共有する、作り直す")."""
import json
import os

import numpy as np
import pytest
import torch

import csa2_inputs as gen
import fp4_compressed_sparse_03_b300 as csa2
import oracle
from gpu_common import dev, gpu_quantize, host, oracle_quantize_parallel

pytestmark = pytest.mark.gpu
GOLD = os.path.join(os.path.dirname(__file__), "golden")


def test_golden_blocks():
    with open(os.path.join(GOLD, "quant_blocks.json")) as f:
        blocks = json.load(f)["blocks"]
    x = np.array([b["x"] for b in blocks], np.float32)
    codes, scales = gpu_quantize(dev(x))
    oc, os_ = oracle.quantize(x)
    assert np.array_equal(host(codes), oc) and np.array_equal(host(scales), os_)
    for i, b in enumerate(blocks):
        assert host(scales)[i, 0] == int(b["scale"], 16)


def test_latent_tiny_workload_bit_exact():
    gains = gen.latent_gains(0)
    x = gen.latent_rows(0, 0, 0, np.arange(4096), gains)
    codes, scales = gpu_quantize(dev(x))
    oc, os_ = oracle_quantize_parallel(x)
    assert np.array_equal(host(codes), oc)
    assert np.array_equal(host(scales), os_)


def _blocks_host(pats: np.ndarray, anchor):
    """float32 blocks [anchor, 15 patterns] (anchor None: [pattern, 0 x 15])."""
    if anchor is None:
        x = np.zeros((pats.size, 16), np.float32)
        x[:, 0] = pats.view(np.float32)
        return x
    nb = (pats.size + 14) // 15
    flat = np.zeros(nb * 15, np.uint32)
    flat[:pats.size] = pats
    x = np.empty((nb, 16), np.float32)
    x[:, 0] = anchor
    x[:, 1:] = flat.view(np.float32).reshape(nb, 15)
    return x


def _blocks_dev(start: int, n: int, sign: int, anchor):
    """The same blocks built on the device from an arange of bit patterns."""
    bits = torch.arange(start, start + n, dtype=torch.int64, device="cuda") | sign
    bits = torch.where(bits >= 2**31, bits - 2**32, bits).to(torch.int32)
    if anchor is None:
        x = torch.zeros((n, 16), dtype=torch.float32, device="cuda")
        x[:, 0] = bits.view(torch.float32)
        return x
    nb = (n + 14) // 15
    flat = torch.zeros(nb * 15, dtype=torch.int32, device="cuda")
    flat[:n] = bits
    x = torch.empty((nb, 16), dtype=torch.float32, device="cuda")
    x[:, 0] = anchor
    x[:, 1:] = flat.view(torch.float32).reshape(nb, 15)
    return x


def test_every_float_up_to_6_at_unit_scale():
    """Blocks [6.0, x_1 .. x_15] have amax 6, so s = E4M3(1) = 1 and y = x: every float32
    with |x| <= 6 (both signs, 2.17e9 values) is encoded by the GPU and the oracle."""
    top = int(np.float32(6.0).view(np.uint32))
    per = 15 * (1 << 22)
    for sign in (0, 0x80000000):
        for start in range(0, top + 1, per):
            n = min(per, top + 1 - start)
            pats = (np.arange(start, start + n, dtype=np.uint64) | sign).astype(np.uint32)
            x = _blocks_host(pats, np.float32(6.0))
            codes, scales = gpu_quantize(_blocks_dev(start, n, sign, 6.0))
            oc, os_ = oracle_quantize_parallel(x)
            assert np.all(os_ == 0x38)
            assert np.array_equal(host(scales), os_), hex(start)
            assert np.array_equal(host(codes), oc), hex(start)


def test_every_amax_scale():
    """Blocks [a, 0, ..., 0] for every float32 a in [0, 8192): the E4M3 scale of a/6,
    including subnormal scales, ties and saturation, plus the code of a/s."""
    top = int(np.float32(8192.0).view(np.uint32))
    per = 1 << 24
    for start in range(0, top, per):
        n = min(per, top - start)
        pats = np.arange(start, start + n, dtype=np.uint64).astype(np.uint32)
        x = _blocks_host(pats, None)
        codes, scales = gpu_quantize(_blocks_dev(start, n, 0, None))
        oc, os_ = oracle_quantize_parallel(x)
        assert np.array_equal(host(scales), os_), hex(start)
        assert np.array_equal(host(codes), oc), hex(start)
    # large amax: saturating scales, sampled
    rng = np.random.default_rng(1)
    big = rng.uniform(8192, 3.0e38, 1 << 20).astype(np.float32)
    y = np.zeros((big.size, 16), np.float32)
    y[:, 0] = big
    y[:, 1] = -big / 3
    codes, scales = gpu_quantize(dev(y))
    oc, os_ = oracle_quantize_parallel(y)
    assert np.array_equal(host(scales), os_) and np.array_equal(host(codes), oc)


def test_dequantize_exact():
    """Every (code byte, scale byte) pair decodes exactly to e2m1 x e4m3."""
    codes = np.tile(np.arange(256, dtype=np.uint8), (127, 1))
    scales = np.repeat(np.arange(127, dtype=np.uint8).reshape(127, 1), 32, axis=1)
    T = 127
    out = torch.zeros((T, 512), dtype=torch.float32, device="cuda")
    slots = torch.arange(T, dtype=torch.int32, device="cuda")
    csa2.check(csa2.csa2_dequantize(dev(codes), dev(scales), slots, out, T, 512, T), "dequantize")
    want = oracle.dequantize(codes, scales)
    assert np.array_equal(host(out).astype(np.float64), want)


def test_bad_slot_is_reported_and_skipped():
    x = np.ones((4, 512), np.float32)
    slots = torch.tensor([0, 7, -1, 2], dtype=torch.int32, device="cuda")
    codes = torch.full((4, 256), 0xAB, dtype=torch.uint8, device="cuda")
    scales = torch.full((4, 32), 0xAB, dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    csa2.check(csa2.csa2_quantize(dev(x), slots, codes, scales, 4, 512, 4, st), "quantize")
    status, bits = csa2.csa2_read_status(st)
    assert status == csa2.CSA2_ERR_DEVICE_FAULT and bits & csa2.CSA2_DEV_BAD_SLOT
    c = host(codes)
    assert np.all(c[1] == 0xAB) and np.all(c[0] != 0xAB) and np.all(c[2] != 0xAB)
    assert csa2.csa2_read_status(st)[0] == csa2.CSA2_OK  # reset by the read


def test_host_argument_errors():
    x = torch.zeros((4, 512), dtype=torch.float32, device="cuda")
    s = torch.zeros(4, dtype=torch.int32, device="cuda")
    c = torch.zeros((4, 256), dtype=torch.uint8, device="cuda")
    sc = torch.zeros((4, 32), dtype=torch.uint8, device="cuda")
    assert csa2.csa2_quantize(x, s, c, sc, 4, 24, 4) == csa2.CSA2_ERR_UNSUPPORTED
    assert csa2.csa2_quantize(None, s, c, sc, 4, 512, 4) == csa2.CSA2_ERR_INVALID_ARGUMENT
    assert csa2.csa2_quantize(x[:, 1:], s, c, sc, 4, 496, 4) == csa2.CSA2_ERR_INVALID_ARGUMENT
    assert csa2.csa2_quantize(x, s, c, sc, 0, 512, 4) == csa2.CSA2_OK


def test_mx_codec_bit_exact_with_special_blocks():
    """MXFP4 variant (OCP MX reading, E8M0 per 32 channels): codes and scales bit-exact
    against the oracle on latent rows plus hand-made blocks (all zero, all negative zero,
    below E8M0's range, amax near 1e31), and the dequantised values equal the oracle's
    exact products."""
    x = gen.latent_rows(3, 0, 0, np.arange(2048), gen.latent_gains(3))
    x[0, :32] = 0.0
    x[1, :32] = 0.0
    x[1, 0] = 2.0**-130
    x[1, 1] = -(2.0**-127) * 0.75
    x[2, :32] *= 1e30
    x[3, 32:64] = -0.0
    x[4, :10] = [3.0, -1.5, 0.5, 2.9, 0.2, -0.3, 5.9, 6.1, -5.0, 0.25]
    T, D = x.shape
    slots = np.random.default_rng(5).permutation(T).astype(np.int32)
    codes = torch.zeros((T, D // 2), dtype=torch.uint8, device="cuda")
    scales = torch.zeros((T, D // 32), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    csa2.check(csa2.csa2_quantize_mx(dev(x), dev(slots), codes, scales, T, D, T, st), "quantize_mx")
    oc, os_ = oracle.mx_quantize(x)
    assert np.array_equal(host(codes)[slots], oc)
    assert np.array_equal(host(scales)[slots], os_)
    out = torch.full((T, D), np.nan, dtype=torch.float32, device="cuda")
    csa2.check(csa2.csa2_dequantize_mx(codes, scales, dev(slots), out, T, D, T, st), "dequantize_mx")
    assert np.array_equal(host(out), oracle.mx_dequantize(oc, os_).astype(np.float32))
    status, bits = csa2.csa2_read_status(st)
    assert status == csa2.CSA2_OK, hex(bits)
