"""Write-path parity: CED projection C = H W (tech-report digest, jiwasawa.github.io,
"Causal Encoder-Decoder (CED) アーキテクチャ", equation C_l = H_{L/2} W_l^KV) quantised on
write (ai2.x.ezic.info blog, "KVを捨てる、共有する、作り直す").  FP4 codes must equal the
oracle's except where the pre-quantisation value lies within 1e-3 of a rounding
boundary; a code whose magnitude rounds to zero on both sides may differ in its sign bit
alone (the code keeps the sign of C, and the sign of a sum that is near zero differs between
fp32 and fp64 accumulation).  E4M3 scales must be equal except where amax/6 lies within
1e-3 of an E4M3 midpoint;
bf16 keys within bf16 rounding of the oracle's value plus the fp32 accumulation error
(|k - C| <= 2^-8 |C| + 1e-4: d = 4096 products of magnitude ~1/64, summed in a
different order in fp32, differ by ~1e-5 typically; near-zero keys can therefore be
several bf16 units apart)."""
import numpy as np
import pytest
import torch

import csa2_inputs as gen
import fp4_compressed_sparse_03_b300 as csa2
import oracle
from fp4_compressed_sparse_03_b300.workload import fill_write_inputs
from gpu_common import _pool, dev, host

pytestmark = pytest.mark.gpu

E2M1_BOUNDS = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
E4M3_VALUES = torch.arange(127, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
E4M3_MIDS = (E4M3_VALUES[1:] + E4M3_VALUES[:-1]) / 2


def run_gpu(H, Wt, slots, T, d, nkv, nidx, num_slots):
    codes = torch.zeros((max(nkv, 1), num_slots, 256), dtype=torch.uint8, device="cuda")
    scales = torch.zeros((max(nkv, 1), num_slots, 32), dtype=torch.uint8, device="cuda")
    keys = torch.zeros((max(nidx, 1), num_slots, 128), dtype=torch.int16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = csa2.csa2_kv_write(H, Wt, codes, scales, keys, T, d, nkv, nidx, slots, num_slots, st)
    assert rc == csa2.CSA2_OK, csa2.status_string(rc)
    status, bits = csa2.csa2_read_status(st)
    assert status == csa2.CSA2_OK, bits
    return host(codes), host(scales), host(keys).view(np.uint16)


def compare(codes_g, scales_g, keys_g, codes_o, scales_o, keys_o, C, what=""):
    """codes_*: [P, R, 256]; scales_*: [P, R, 32]; keys_*: [Pi, R, 128]; C: oracle fp32 [R, n_out]."""
    nkv = codes_o.shape[0]
    R = codes_o.shape[1]
    bad_blocks = 0
    for p in range(nkv):
        Cp = C[:, p * 512:(p + 1) * 512].astype(np.float64).reshape(R, 32, 16)
        amax6 = np.abs(Cp).max(axis=2) / 6.0
        near_mid = np.min(np.abs(amax6[..., None] - E4M3_MIDS) / np.maximum(E4M3_MIDS, 1e-30),
                          axis=-1) <= 1e-3
        sdiff = scales_g[p] != scales_o[p]
        assert np.all(near_mid[sdiff]), f"{what}: scale mismatch away from an E4M3 midpoint"
        s = oracle.e4m3_decode(scales_o[p].ravel()).reshape(R, 32)
        y = np.abs(Cp) / np.where(s > 0, s, 1.0)[..., None]
        near_b = np.min(np.abs(y[..., None] - E2M1_BOUNDS) / E2M1_BOUNDS, axis=-1) <= 1e-3
        cg = np.stack([codes_g[p] & 0xF, codes_g[p] >> 4], -1).reshape(R, 32, 16)
        co = np.stack([codes_o[p] & 0xF, codes_o[p] >> 4], -1).reshape(R, 32, 16)
        # a code that rounds to zero keeps the sign of C: only the sign bit may differ,
        # and only where the magnitude is zero on both sides
        near_b |= ((cg ^ co) == 8) & ((co & 7) == 0)
        cdiff = (cg != co) & ~sdiff[..., None]
        far = np.argwhere(cdiff & ~near_b)
        assert far.size == 0, (f"{what}: code mismatch away from a rounding boundary at "
                               f"(row, block, ch) {far[:4].tolist()}: gpu "
                               f"{[int(cg[tuple(i)]) for i in far[:4]]} oracle "
                               f"{[int(co[tuple(i)]) for i in far[:4]]} C "
                               f"{[float(Cp[tuple(i)]) for i in far[:4]]} y "
                               f"{[float(y[tuple(i)]) for i in far[:4]]}")
        bad_blocks += int(sdiff.sum()) + int(cdiff.any(axis=2).sum())
    if keys_o.size:
        kg_val = gen.bf16_bits_to_f32(keys_g).astype(np.float64)
        base = nkv * 512
        Ck = np.stack([C[:, base + p * 128: base + (p + 1) * 128] for p in range(keys_o.shape[0])])
        assert np.all(np.abs(kg_val - Ck) <= 2.0**-8 * np.abs(Ck) + 1e-4), \
            f"{what}: bf16 key beyond rounding + accumulation error"
        exact = np.mean(keys_g == keys_o)
        assert exact > 0.99, f"{what}: only {exact:.4%} of keys bit-equal"
    return bad_blocks


def _oracle_rows(Hh, Wth, nkv, nidx):
    parts = np.array_split(np.arange(Hh.shape[0]), min(Hh.shape[0], 16))
    res = list(_pool.map(lambda r: oracle.kv_write_rows(Hh[r], Wth, nkv, nidx), parts))
    return (np.concatenate([r[0] for r in res], axis=1), np.concatenate([r[1] for r in res], axis=1),
            np.concatenate([r[2] for r in res], axis=1), np.concatenate([r[3] for r in res], axis=0))


@pytest.mark.parametrize("T,d,nkv,nidx", [(256, 256, 2, 2), (384, 512, 1, 1), (128, 192, 0, 3),
                                          (256, 1024, 3, 0), (64, 256, 2, 2), (200, 512, 1, 1),
                                          (1, 128, 1, 1), (33, 192, 1, 1), (65, 192, 1, 1),
                                          (100, 256, 1, 1)])
def test_small_projections(T, d, nkv, nidx):
    ww = gen.WriteWorkload("small", 50 + T + d, T, d, nkv, nidx)
    H, Wt, slots = fill_write_inputs(ww)
    num_slots = ww.num_pages * 64
    cg, sg, kg = run_gpu(H, Wt, slots, T, d, nkv, nidx, num_slots)
    Hh, Wth = host(H).view(np.uint16), host(Wt).view(np.uint16)
    co, so, ko, C = _oracle_rows(Hh, Wth, nkv, nidx)
    sl = host(slots)
    compare(cg[:nkv, sl], sg[:nkv, sl], kg[:nidx, sl], co, so, ko, C, f"T{T} d{d}")


def test_identity_projection_is_exact():
    """W = [I; 0] makes C equal to H's columns exactly: codes and keys bit-exact."""
    T, d = 128, 640
    rng = np.random.default_rng(3)
    Hh = gen.f32_to_bf16_bits((rng.standard_normal((T, d)) * 4).astype(np.float32))
    Wth = np.zeros((512 + 128, d), np.uint16)
    Wth[np.arange(640), np.arange(640)] = 0x3F80
    slots = np.random.default_rng(4).permutation(T).astype(np.int32)
    cg, sg, kg = run_gpu(dev(Hh), dev(Wth), dev(slots), T, d, 1, 1, T)
    co, so, ko, _ = oracle.kv_write_rows(Hh, Wth, 1, 1)
    assert np.array_equal(cg[0, slots], co[0]) and np.array_equal(sg[0, slots], so[0])
    assert np.array_equal(kg[0, slots], ko[0])


def test_ced_write_32768x4096_sampled_rows():
    """The full write workload (H [32768, 4096]; 20 x 512 latent + 20 x 128 key
    projections); 1024 sampled token rows compared over all 12800 output columns."""
    ww = gen.config_write()
    H, Wt, slots = fill_write_inputs(ww)
    num_slots = ww.num_pages * 64
    cg, sg, kg = run_gpu(H, Wt, slots, ww.T, ww.d_model, ww.n_kv_proj, ww.n_idx_proj, num_slots)
    rows = np.sort(np.random.default_rng(2).choice(ww.T, 1024, replace=False))
    Hh = ww.h_rows(rows)
    Wth = host(Wt).view(np.uint16)
    assert np.array_equal(Wth[[0, 5000, 12799]], ww.w_rows([0, 5000, 12799]))
    co, so, ko, C = _oracle_rows(Hh, Wth, ww.n_kv_proj, ww.n_idx_proj)
    sl = host(slots)[rows]
    bad = compare(cg[:, sl], sg[:, sl], kg[:, sl], co, so, ko, C, "ced write")
    assert bad <= len(rows) * 20 * 32 * 1e-3


def test_decode_append_64_tokens():
    """Decode-time append: one new token per sequence of the 64-sequence batch, each at its
    own page (H [64, 4096]; 20 x 512 latent + 20 x 128 key projections), every row and
    column against the oracle.  The single M-tile is half padding."""
    ww = gen.config_append()
    H, Wt, slots = fill_write_inputs(ww)
    num_slots = ww.num_pages * 64
    cg, sg, kg = run_gpu(H, Wt, slots, ww.T, ww.d_model, ww.n_kv_proj, ww.n_idx_proj, num_slots)
    Hh, Wth = host(H).view(np.uint16), host(Wt).view(np.uint16)
    assert np.array_equal(Hh[[0, 63]], ww.h_rows([0, 63]))
    co, so, ko, C = _oracle_rows(Hh, Wth, ww.n_kv_proj, ww.n_idx_proj)
    sl = host(slots)
    bad = compare(cg[:, sl], sg[:, sl], kg[:, sl], co, so, ko, C, "decode append")
    assert bad <= 64 * 20 * 32 * 1e-3
    # nothing but the 64 new rows was written
    untouched = np.setdiff1d(np.arange(num_slots), sl)
    assert not cg[:, untouched].any() and not sg[:, untouched].any() and not kg[:, untouched].any()


def test_write_host_argument_errors():
    H = torch.zeros((100, 256), dtype=torch.int16, device="cuda")
    Wt = torch.zeros((512, 256), dtype=torch.int16, device="cuda")
    c = torch.zeros((1, 128, 256), dtype=torch.uint8, device="cuda")
    s = torch.zeros((1, 128, 32), dtype=torch.uint8, device="cuda")
    sl = torch.zeros(100, dtype=torch.int32, device="cuda")
    assert csa2.csa2_kv_write(H, Wt, c, s, None, 100, 200, 1, 0, sl, 128) == csa2.CSA2_ERR_UNSUPPORTED
    assert csa2.csa2_kv_write(H, Wt, c, s, None, 128, 256, 1, 1, sl, 128) == \
        csa2.CSA2_ERR_INVALID_ARGUMENT
