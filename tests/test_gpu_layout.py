"""GEMM scale layout: the device rearrangement equals the oracle's, for the rowwise and
(transposed) columnwise grids of the 16384x6144 weight, ragged grids, padded leading
dimensions and an output that is not 16-byte aligned."""
import numpy as np
import pytest
import torch

import oracle
from mxfp8_master_weight_gb300 import api

from flows import to_host

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("nr,nc,ld,transpose", [
    (16384, 192, 192, False), (512, 6144, 6144, True), (130, 6, 9, False), (33, 65, 65, True),
    (1, 1, 1, False), (1000, 257, 300, True)])
@pytest.mark.parametrize("offset", [0, 3])
def test_swizzle_matches_oracle(nr, nc, ld, transpose, offset):
    rng = np.random.default_rng(nr * 31 + nc)
    S = rng.integers(0, 256, (nr, ld), dtype=np.uint8)
    size = api.mxfp8_swizzled_scales_size(nr, nc, transpose)
    buf = torch.full((size + offset,), 0xCD, dtype=torch.uint8, device="cuda")
    out = buf[offset:]  # offset 3: not 16-byte aligned
    api.mxfp8_swizzle_scales(torch.from_numpy(S).cuda(), out, nr, nc, transpose)
    torch.cuda.synchronize()
    assert np.array_equal(to_host(out), oracle.swizzle_scales(S, nr, nc, transpose))
    assert np.all(to_host(buf[:offset]) == 0xCD)
