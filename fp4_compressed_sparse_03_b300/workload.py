"""Synthetic decode / write workloads placed in HBM.

The random values come from the seeded counter-based generator of ``csa2_inputs``
(device kernels, bit-identical to its host definition); the latent is quantised into
the paged pools by libcsa2's own codec (csa2_quantize), exactly as a serving system
would fill its cache.  Everything here runs before any timed region.
"""
from __future__ import annotations

import numpy as np
import torch

import csa2_inputs as gen
from csa2_inputs import native
from csa2_inputs.native import all_queries_host, layer_queries_host  # noqa: F401  (re-export)

from . import check, csa2_quantize, csa2_quantize_mx
from .decode import DecodeCache

_CHUNK = 1 << 18  # latent rows staged per quantise call (512 MB of fp32)


def fill_decode_cache(wl: gen.DecodeWorkload, n_groups: int | None = None, device="cuda",
                      stream=None, mx: bool = False) -> DecodeCache:
    """A DecodeCache holding every Full group's quantised latent (E4M3 / 16, or the MXFP4
    variant with `mx`) and indexer keys."""
    if n_groups is None:
        n_groups = max(1, sum(1 for m in wl.schedule if m == gen.FULL))
    lay = wl.layout
    cache = DecodeCache(lay.seq_lens, lay.page_table, lay.num_pages, n_groups, device, mx=mx)
    quant = csa2_quantize_mx if mx else csa2_quantize
    B = len(lay.seq_lens)
    max_len = int(lay.seq_lens.max()) if B else 0
    stage = torch.empty((min(_CHUNK, max(max_len, 1)), gen.D_KV), dtype=torch.float32,
                        device=cache.device)
    for g in range(n_groups):
        skeys = torch.as_tensor(native.seq_keys(wl.seed, gen.TAG_KEY, g, B).view(np.int64),
                                device=cache.device)
        native.fill_keys_paged_dev(cache.keys[g], skeys, cache.seq_lens, cache.page_table, stream)
        gains = torch.as_tensor(gen.latent_gains(wl.seed, g), device=cache.device)
        for b in range(B):
            n_b = int(lay.seq_lens[b])
            key = gen.stream_key(wl.seed, gen.TAG_LATENT, (g << 24) | b)
            for t0 in range(0, n_b, _CHUNK):
                n = min(_CHUNK, n_b - t0)
                native.fill_latent_dev(stage[:n], key, t0, gains, stream)
                slots = torch.as_tensor(lay.slots(b, np.arange(t0, t0 + n)).astype(np.int32),
                                        device=cache.device)
                check(quant(stage[:n], slots, cache.codes[g], cache.scales[g], n, gen.D_KV,
                            cache.num_slots, None, stream), "csa2_quantize")
    torch.cuda.synchronize()
    return cache


def fill_write_inputs(ww: gen.WriteWorkload, device="cuda", stream=None):
    """(H [T, d] bf16 bits, Wt [n_out, d] bf16 bits, slot_of_token [T]) on the device."""
    dev = torch.device(device)
    H = torch.empty((ww.T, ww.d_model), dtype=torch.int16, device=dev)
    native.fill_bf16_dev(H, gen.stream_key(ww.seed, gen.TAG_H), 0, 0, stream)
    Wt = torch.empty((ww.n_out, ww.d_model), dtype=torch.int16, device=dev)
    p2 = gen.d_model_pow2_scale(ww.d_model)
    kv = ww.n_kv_proj * gen.D_KV
    if kv:
        native.fill_bf16_dev(Wt[:kv], gen.stream_key(ww.seed, gen.TAG_WKV), 0, p2, stream)
    if ww.n_out > kv:
        native.fill_bf16_dev(Wt[kv:], gen.stream_key(ww.seed, gen.TAG_WIDX), 0, p2, stream)
    slots = torch.as_tensor(ww.slot_of_token(), device=dev)
    torch.cuda.synchronize()
    return H, Wt, slots
