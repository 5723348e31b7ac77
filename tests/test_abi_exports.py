"""The C-ABI library loads and exports every symbol the public header declares; the
host-side argument checks answer before any device work (no GPU needed)."""
import ctypes
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "csa2.h")


def declared_functions():
    src = open(HEADER).read()
    return re.findall(r"CSA2_API\s+[\w\s\*]+?\b(csa2_\w+)\s*\(", src)


def test_header_declares_the_three_calls():
    names = set(declared_functions())
    assert {"csa2_kv_write", "csa2_index", "csa2_sparse_attn"} <= names
    assert len(names) >= 10


def test_library_exports_every_declared_symbol():
    from fp4_compressed_sparse_03_b300 import build
    lib = ctypes.CDLL(build.build())
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_host_side_checks_without_device():
    import fp4_compressed_sparse_03_b300 as csa2
    assert csa2.version() >= 10000
    assert csa2.status_string(csa2.CSA2_ERR_TIMEOUT).startswith("bounded")
    L = csa2._lib
    # null argument blocks are rejected before any CUDA call
    assert L.csa2_index(0, None, None, None, 16, None, None, None, None) == csa2.CSA2_ERR_INVALID_ARGUMENT
    assert L.csa2_quantize(None, None, None, None, -1, 512, 0, None, None) == csa2.CSA2_ERR_INVALID_ARGUMENT
    assert L.csa2_quantize(None, None, None, None, 4, 24, 4, None, None) == csa2.CSA2_ERR_UNSUPPORTED
    assert L.csa2_quantize_mx(None, None, None, None, 4, 48, 4, None, None) == csa2.CSA2_ERR_UNSUPPORTED
    assert L.csa2_dequantize_mx(None, None, None, None, -1, 64, 4, None, None) == \
        csa2.CSA2_ERR_INVALID_ARGUMENT
    assert L.csa2_kv_write(None, None, None, None, None, 4, 64, 1, 0, None, 4, None, None) == \
        csa2.CSA2_ERR_INVALID_ARGUMENT
    assert L.csa2_read_status(None, None, None) == csa2.CSA2_ERR_INVALID_ARGUMENT
    # the bounded-wait diagnostic checks its limit and status word before launching
    fake_st = 1 << 12
    assert L.csa2_check_bounded_wait(0, 1024, None, None) == csa2.CSA2_ERR_INVALID_ARGUMENT
    assert L.csa2_check_bounded_wait(0, 0, fake_st, None) == csa2.CSA2_ERR_INVALID_ARGUMENT
    assert L.csa2_check_bounded_wait(0, (1 << 20) + 1, fake_st, None) == csa2.CSA2_ERR_INVALID_ARGUMENT
    # attention over more than CSA2_ATTN_MAX_TOPK entries per query is refused on the host
    # (fake aligned addresses: nothing is dereferenced before the check)
    fake = 1 << 12
    pages = csa2.Csa2Pages(1, fake, fake, 1, 1, 64)
    for f in (lambda k: L.csa2_sparse_attn(fake, fake, fake, fake, ctypes.byref(pages), fake, None, 1,
                                           fake, k, 0.04, None, 0, None, None),
              lambda k: L.csa2_sparse_attn_static(fake, fake, fake, fake, ctypes.byref(pages), fake,
                                                  None, 1, fake, k, 0.04, None, None)):
        assert f(65536 + 1) == csa2.CSA2_ERR_UNSUPPORTED
    # workspace sizing is host arithmetic
    full = csa2.csa2_index_workspace_size(csa2.CSA2_FULL, 64, 1024, 8192)
    hist = 64 * 2048 * 4                                             # selection histograms
    assert 64 * 1024 * 64 * 4 + hist < full < 64 * 1024 * 64 * 4 + hist + 4096  # + scores, run list
    # beyond 2^18 tokens the wide selection adds (position, key) lists covering every
    # position of the context
    wide = csa2.csa2_index_workspace_size(csa2.CSA2_FULL, 4, 16384, 8192)
    assert wide >= 4 * 16384 * 64 * (4 + 8) + 4 * 2048 * 4
    re = csa2.csa2_index_workspace_size(csa2.CSA2_REINDEX, 64, 2048, 8192)
    assert re == 64 * 8192 * 4                                       # scores only
    assert csa2.csa2_index_workspace_size(csa2.CSA2_REUSE, 64, 2048, 8192) == 0


def test_chunked_attention_host_checks():
    """Argument checks and workspace sizing of csa2_sparse_attn_chunked, before any device
    work (fake aligned addresses are never dereferenced)."""
    import fp4_compressed_sparse_03_b300 as csa2
    L = csa2._lib
    fake = 1 << 12
    pages = csa2.Csa2Pages(1, fake, fake, 1, 1, 64)

    def call(nq, chunk, k, ws=fake, wsb=1 << 30):
        return L.csa2_sparse_attn_chunked(fake, fake, fake, fake, ctypes.byref(pages), fake, None,
                                          nq, fake, chunk, k, ctypes.c_float(0.04), ws, wsb, None,
                                          None)

    assert call(6, 4, 16) == csa2.CSA2_ERR_INVALID_ARGUMENT      # num_q not a multiple of chunk
    assert call(4, 0, 16) == csa2.CSA2_ERR_INVALID_ARGUMENT
    assert call(5, 5, 16) == csa2.CSA2_ERR_UNSUPPORTED           # more than four queries
    assert call(4, 4, 2049) == csa2.CSA2_ERR_UNSUPPORTED         # union above 8192 entries
    assert call(4, 4, 2048, ws=None) == csa2.CSA2_ERR_INVALID_ARGUMENT
    assert call(4, 4, 2048, wsb=1024) == csa2.CSA2_ERR_INVALID_ARGUMENT
    assert call(4, 4, 2048, ws=fake + 8) == csa2.CSA2_ERR_INVALID_ARGUMENT
    assert csa2.csa2_chunk_attn_workspace_size(6, 4, 16) == 0
    assert csa2.csa2_chunk_attn_workspace_size(4, 4, 4096) == 0
    # union slots and masks, then per query and span 16 x 512 partial outputs and 32 (m, l)
    nq, chunk, k = 256, 4, 2048
    ws = csa2.csa2_chunk_attn_workspace_size(nq, chunk, k)
    per_span = nq * (16 * 512 + 32) * 4
    union = (nq // chunk) * chunk * k * 5
    assert union + per_span <= ws <= union + 16 * per_span + 4096
    assert (ws - union) % per_span < 4096


def test_generator_library_host_path():
    import numpy as np
    import csa2_inputs as gen
    from csa2_inputs import native
    assert np.array_equal(native.key_rows_host(3, 1, 2, 10, 50), gen.key_rows(3, 1, 2, np.arange(10, 60)))
    g = gen.latent_gains(3, 1)
    assert np.array_equal(native.latent_rows_host(3, 1, 2, 5, 20, g),
                          gen.latent_rows(3, 1, 2, np.arange(5, 25), g))


def test_overlapping_selections_generator():
    """The multi-query workload's selections: sorted distinct tokens of the context, -1
    padding only at the end, the stated shared part common to every query, and every query
    selecting the whole context when it is shorter than K."""
    import numpy as np
    import csa2_inputs as gen
    sets = gen.overlapping_index_sets(5, 3, 3000, 512, 4, 0.75)
    assert sets.shape == (4, 512) and sets.dtype == np.int32
    for row in sets:
        assert np.all(np.diff(row) > 0) and row.min() >= 0 and row.max() < 3000
    common = set(sets[0]).intersection(*map(set, sets[1:]))
    assert len(common) >= 384  # round(0.75 * 512), plus chance agreements
    assert len(set(sets.ravel())) <= 384 + 4 * 128
    assert np.array_equal(sets, gen.overlapping_index_sets(5, 3, 3000, 512, 4, 0.75))
    short = gen.overlapping_index_sets(5, 4, 300, 512, 3, 0.5)
    for row in short:
        assert np.array_equal(row[:300], np.arange(300)) and np.all(row[300:] == -1)
    none = gen.overlapping_index_sets(5, 6, 4096, 256, 2, 0.0)
    assert len(set(none[0]) & set(none[1])) < 64  # independent draws: about 16 in common


def test_graft_build_entry():
    import __graft_entry__
    __graft_entry__.build()


def test_static_attention_scratch_limit():
    """csa2_sparse_attn_static holds its scratch in a fixed array: at top-K 2048 on 148 SMs
    the decode batch's 64 queries fit (9.8 MiB) and 74 is the most one call takes; a larger
    batch is issued as several calls on one stream.  (Workspace sizes are host arithmetic;
    without a device the library sizes for 148 SMs.)"""
    import fp4_compressed_sparse_03_b300 as csa2
    lim = csa2.ATTN_STATIC_SCRATCH_BYTES
    assert csa2.csa2_attn_workspace_size(64, 2048) <= lim
    assert csa2.csa2_attn_workspace_size(74, 2048) <= lim < csa2.csa2_attn_workspace_size(75, 2048)
