"""The library's kernels load on the GPU as sm_103a cubins (GPU)."""
from __future__ import annotations

import pytest
import torch

import h2o_heavy_hitter_decode_gb300 as h2o

pytestmark = pytest.mark.gpu


def test_kernels_load_as_sm103a():
    torch.cuda.init()
    cc = torch.cuda.get_device_capability()
    ptx, binv = h2o.kernel_arch()
    assert cc == (10, 3), cc
    assert (ptx, binv) == (103, 103), (ptx, binv)
