"""The bounded waits of the kernels: a wait that cannot complete gives up,
reports a device fault bit the host can read, and leaves the context usable."""

import numpy as np
import pytest
import torch

from grads_taco_compress_gb300 import binding as tb
from grads_taco_compress_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def test_wait_that_never_completes_times_out():
    tb.taco_get_fault(clear=True)
    assert tb.taco_selftest_wait_timeout(2_000_000) == 1          # 2 ms limit
    bits = tb.taco_get_fault(clear=True)
    assert bits & 4 and not bits & 3
    assert tb.taco_get_fault() == 0
    # the context is still usable
    x = W.make_shards(W.WORKLOADS["tiny-512x1024"], N=8, P=1)
    xd = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda()
    bundle, headers = tb.taco_compress_shards(xd, 128)
    torch.cuda.synchronize()
    assert tb.parse_headers(headers)[0]["N"] == 8
    assert tb.taco_get_fault() == 0
