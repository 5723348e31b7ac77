"""Failure detection on the device without a fault: a bounded mbarrier wait that nothing
completes runs out, reports CSA2_DEV_TIMEOUT through the status word, and the kernel
returns with the context still usable (the same wait guards every TMA- and
tcgen05-fed kernel of the library)."""
import time

import numpy as np
import pytest
import torch

import fp4_compressed_sparse_03_b300 as csa2
from gpu_common import dev, host

pytestmark = pytest.mark.gpu


def test_expired_wait_reports_timeout_and_context_survives():
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    csa2.check(csa2.csa2_check_bounded_wait(False, 1 << 16, st), "check_bounded_wait")
    status, bits = csa2.csa2_read_status(st)
    elapsed = time.perf_counter() - t0
    assert status == csa2.CSA2_ERR_TIMEOUT and bits == csa2.CSA2_DEV_TIMEOUT
    assert elapsed < 5.0, elapsed  # bounded: a short limit gives up quickly
    # the status word was reset by the read, and a wait whose phase completes reports nothing
    csa2.check(csa2.csa2_check_bounded_wait(True, 1 << 16, st), "check_bounded_wait")
    assert csa2.csa2_read_status(st) == (csa2.CSA2_OK, 0)
    # the context is intact: a library kernel and a torch kernel still run and agree
    x = np.linspace(-6, 6, 4 * 512, dtype=np.float32).reshape(4, 512)
    slots = torch.arange(4, dtype=torch.int32, device="cuda")
    codes = torch.zeros((4, 256), dtype=torch.uint8, device="cuda")
    scales = torch.zeros((4, 32), dtype=torch.uint8, device="cuda")
    csa2.check(csa2.csa2_quantize(dev(x), slots, codes, scales, 4, 512, 4, st), "quantize")
    assert csa2.csa2_read_status(st)[0] == csa2.CSA2_OK
    assert host(codes).any()
    assert float(torch.ones(8, device="cuda").sum()) == 8.0
