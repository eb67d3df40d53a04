"""taco_compress_shards_noalloc against taco_compress_shards, through the C ABI.

The no-allocation entry point is for callers that cannot call cudaMalloc
where they compress (a communication library's progress thread or collective
callback, a runtime whose memory belongs to an external pool): it keeps the
header workspace in the library's static device scratch instead of taking one
from the caller. Its output must match the workspace entry point's, call
after call, because every call clears the counters it reuses.
"""

import dataclasses

import numpy as np
import pytest
import torch

import parity
from grads_taco_compress_gb300 import binding as tb
from grads_taco_compress_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _outputs(bundle, headers, P, N, h, block):
    codes, alpha, s = tb.shard_views(bundle, P, N, h, block)
    return codes.cpu().numpy(), alpha.cpu().numpy(), s.cpu().numpy(), tb.parse_headers(headers)


@pytest.mark.parametrize("name,rows,P", [("gpt2-1.5b-act", 300, 4), ("gpt3-6.7b-act", 130, 8)])
def test_noalloc_matches_workspace_entry_point_twice(name, rows, P):
    w = W.WORKLOADS[name]
    N, h, n = rows, w.h, w.block
    sb = tb.shard_bytes(N, h, n)
    # outputs allocated up front: the no-allocation calls themselves allocate nothing
    bundle = torch.empty((P, sb), dtype=torch.uint8, device="cuda")
    headers = torch.empty((P, tb.HEADER_BYTES), dtype=torch.uint8, device="cuda")
    for call in range(2):                                   # two calls in a row
        x_bits = W.make_shards(dataclasses.replace(w, seed=call), N=N, P=P)
        x = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).cuda()
        tb.taco_compress_shards_noalloc(x, n, bundle=bundle, headers=headers)
        ref_bundle, ref_headers = tb.taco_compress_shards(x, n)
        torch.cuda.synchronize()
        got = _outputs(bundle, headers, P, N, h, n)
        ref = _outputs(ref_bundle, ref_headers, P, N, h, n)
        parity.compare_codes(got[0], ref[0], f"call {call} codes")
        parity.compare_scales(got[1], ref[1], f"call {call} alpha")
        parity.compare_scales(got[2], ref[2], f"call {call} s")
        for field in ("N", "h", "block", "variant", "s_max", "n_clamped"):
            assert np.array_equal(got[3][field], ref[3][field]), (call, field)


def test_noalloc_rejects_more_shards_than_its_scratch_holds():
    x = torch.zeros((9, 4, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(tb.TacoError) as err:
        tb.taco_compress_shards_noalloc(x, 128)
    assert err.value.status == 7                            # TACO_ERR_WORKSPACE


def test_noalloc_rejected_call_then_valid_call():
    """A rejected call returns its status before it enqueues anything (not even
    the clear of the static scratch). The next call on the same stream, with
    all 8 shards the scratch holds, writes the outputs and headers of the
    workspace entry point."""
    w = W.WORKLOADS["gpt3-6.7b-act"]
    P, N, h, n = 8, 48, w.h, w.block
    x = torch.from_numpy(W.make_shards(w, N=N, P=P).view(np.int16)).view(torch.bfloat16).cuda()
    sb = tb.shard_bytes(N, h, n)
    bundle = torch.empty((P, sb), dtype=torch.uint8, device="cuda")
    headers = torch.empty((P, tb.HEADER_BYTES), dtype=torch.uint8, device="cuda")
    flat = torch.empty(P * N * h + 8, dtype=torch.bfloat16, device="cuda")
    misaligned = flat[1: 1 + P * N * h].view(P, N, h)          # 2 bytes off a 16-byte boundary
    misaligned.copy_(x)
    for bad, status in (((misaligned, n), 4), ((x, 100), 3)):   # TACO_ERR_ALIGN, TACO_ERR_BLOCK
        with pytest.raises(tb.TacoError) as err:
            tb.taco_compress_shards_noalloc(*bad, bundle=bundle, headers=headers)
        assert err.value.status == status
    tb.taco_compress_shards_noalloc(x, n, bundle=bundle, headers=headers)
    ref_bundle, ref_headers = tb.taco_compress_shards(x, n)
    torch.cuda.synchronize()
    got = _outputs(bundle, headers, P, N, h, n)
    ref = _outputs(ref_bundle, ref_headers, P, N, h, n)
    parity.compare_codes(got[0], ref[0], "codes")
    parity.compare_scales(got[1], ref[1], "alpha")
    parity.compare_scales(got[2], ref[2], "s")
    for field in ("N", "h", "block", "variant", "s_max", "n_clamped"):
        assert np.array_equal(got[3][field], ref[3][field]), field
