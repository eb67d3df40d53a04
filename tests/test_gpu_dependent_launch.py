"""Inputs written by the kernel launched just before, on the same stream.

Every streaming kernel is launched with programmatic dependent launch: its
CTAs may start while the preceding kernel of the stream still runs, ask L2
for the data of their first stages, and only then wait for that kernel to
finish and its writes to become visible. These tests make the preceding
kernel write the very input the next kernel reads, several times over the
same buffers with different data, so that a read of stale data (a first
tile fetched before the writer finished, and used) would show as a wrong
code or element. Every output is compared with the oracle of the data
written last.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import parity
from grads_taco_compress_gb300 import binding as tb
from grads_taco_compress_gb300 import workloads as W
from oracle import taco_oracle as O
from test_gpu_parity import E_STAR, host_bits

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("block", [64, 128, 256])
def test_inputs_written_by_the_previous_kernel(block, oracle_rows):
    """Per round: a torch kernel writes x (x = src_i * 1, exact in bf16), the
    tensor-core compress reads x and writes the bundle, the decompress-reduce
    reads that bundle, the reduce-recompress reads it again. Three rounds
    over the same x, bundle and outputs, with data of a different scale each
    round, all queued without a synchronisation."""
    P, N, h = 4, 1024, 2048
    rng = np.random.default_rng(1000 + block)
    xs = [W.f32_to_bf16_bits(rng.laplace(0, 0.02 * (i + 1), size=(P, N, h)).astype(np.float32))
          for i in range(3)]
    srcs = [torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda() for x in xs]
    x = torch.empty_like(srcs[0])
    bundle = torch.empty((P, tb.shard_bytes(N, h, block)), dtype=torch.uint8, device="cuda")
    out = torch.empty((N, h), dtype=torch.bfloat16, device="cuda")
    rc = torch.empty(tb.shard_bytes(N, h, block), dtype=torch.uint8, device="cuda")
    ws = tb.new_workspace(P)
    ws1 = tb.new_workspace(1)
    torch.cuda.synchronize()
    kept = []
    for i in range(3):
        torch.mul(srcs[i], 1.0, out=x)
        tb.taco_compress_shards_mma(x, block, bundle=bundle, workspace=ws)
        tb.taco_decompress_reduce(bundle, P, N, h, block, out=out)
        tb.taco_reduce_recompress(bundle, P, N, h, block, E_STAR, shard=rc, workspace=ws1)
        kept.append((bundle.clone(), out.clone(), rc.clone()))
    torch.cuda.synchronize()
    for i, (b, y, r) in enumerate(kept):
        codes, alpha, s = (t.cpu().numpy() for t in tb.shard_views(b, P, N, h, block))
        oc, oa, os_ = oracle_rows.compress(xs[i], block, E_STAR)
        for p in range(P):
            parity.compare_codes(codes[p], oc[p], f"round {i} codes[{p}]")
            parity.compare_scales(alpha[p], oa[p], f"round {i} alpha[{p}]")
            parity.compare_scales(s[p], os_[p], f"round {i} s[{p}]")
        # the decompress-reduce of the GPU's own bundle against the oracle's
        # decompress-reduce of that same bundle
        want = oracle_rows.decompress_reduce(codes, alpha, s, block)
        got = host_bits(y)
        assert parity.compare_recon(O.bf16_bits_to_f64(got), O.bf16_bits_to_f64(want)) < 1e-2
        assert float(np.mean(got == want)) > 0.99
        rcodes, ralpha, rs = (t.cpu().numpy() for t in tb.shard_views(r[None], 1, N, h, block))
        qc, qa, qs, _ = O.reduce_recompress(codes, alpha, s, block, E_STAR)
        parity.compare_codes(rcodes[0], qc, f"round {i} recompressed codes")
        parity.compare_scales(ralpha[0], qa, f"round {i} recompressed alpha")
        parity.compare_scales(rs[0], qs, f"round {i} recompressed s")


def test_concurrent_compress_calls_on_two_streams(oracle_rows):
    """Two compress calls of different tensors on two streams, each with its
    own workspace, queued so that they overlap on the GPU several times over:
    the tile pool's counter and the header totals live in each call's own
    workspace, so every output must match the oracle of its own input."""
    P, N, h, block = 4, 1024, 2048, 128
    rng = np.random.default_rng(31)
    xs = [W.f32_to_bf16_bits(rng.laplace(0, 0.03 * (i + 1), size=(P, N, h)).astype(np.float32)) for i in range(2)]
    xd = [torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda() for x in xs]
    streams = [torch.cuda.Stream() for _ in range(2)]
    wss = [tb.new_workspace(P) for _ in range(2)]
    bundles = [torch.empty((P, tb.shard_bytes(N, h, block)), dtype=torch.uint8, device="cuda") for _ in range(2)]
    headers = [torch.empty((P, tb.HEADER_BYTES), dtype=torch.uint8, device="cuda") for _ in range(2)]
    torch.cuda.synchronize()
    for _ in range(5):
        for i in range(2):
            with torch.cuda.stream(streams[i]):
                tb.taco_compress_shards(xd[i], block, bundle=bundles[i], headers=headers[i], workspace=wss[i],
                                        stream=streams[i])
    torch.cuda.synchronize()
    for i in range(2):
        assert int(wss[i].count_nonzero()) == 0
        codes, alpha, s = (t.cpu().numpy() for t in tb.shard_views(bundles[i], P, N, h, block))
        oc, oa, os_ = oracle_rows.compress(xs[i], block, E_STAR)
        hdr = tb.parse_headers(headers[i])
        for p in range(P):
            parity.compare_codes(codes[p], oc[p], f"call {i} codes[{p}]")
            parity.compare_scales(alpha[p], oa[p], f"call {i} alpha[{p}]")
            parity.compare_scales(s[p], os_[p], f"call {i} s[{p}]")
            assert hdr[p]["s_max"] == s[p].max() and hdr[p]["n_clamped"] == np.count_nonzero(s[p] > 1.0)


@pytest.mark.parametrize("entry", ["mma", "reduce_recompress"])
def test_many_back_to_back_launches_on_one_workspace(entry):
    """100 launches queued back to back on one workspace, alternating two
    inputs, each into its own outputs: every launch starts while the previous
    one ends (programmatic dependent launch) and takes the tile pool and the
    header counters the previous one left zeroed. The last outputs of each
    input must equal, bit for bit, those of a single call made alone."""
    w = W.WORKLOADS["gpt2-1.5b-act"]
    P, N, h, n = w.P, 1024, w.h, w.block
    xs = [torch.from_numpy(W.make_shards(w, N=N, P=P).view(np.int16)).view(torch.bfloat16).cuda(),
          torch.from_numpy((W.make_shards(w, N=N, P=P) ^ np.uint16(0x8000)).view(np.int16)).view(torch.bfloat16).cuda()]
    if entry == "mma":
        def run(i, ws, out=None):
            return tb.taco_compress_shards(xs[i % 2], n, workspace=ws, bundle=None if out is None else out[0],
                                           headers=None if out is None else out[1])
    else:
        bundles = [tb.taco_compress_shards(x, n)[0] for x in xs]
        def run(i, ws, out=None):
            sh, hd, _ = tb.taco_reduce_recompress(bundles[i % 2], P, N, h, n, workspace=ws,
                                                 shard=None if out is None else out[0],
                                                 header=None if out is None else out[1])
            return sh, hd
    ref = []
    for i in range(2):
        ref.append(run(i, tb.new_workspace(P)))
        torch.cuda.synchronize()
    ws = tb.new_workspace(P)
    outs = [(torch.empty_like(r[0]), torch.empty_like(r[1])) for r in ref]
    for i in range(100):
        run(i, ws, outs[i % 2])
    torch.cuda.synchronize()
    assert int(ws.count_nonzero()) == 0
    import test_gpu_parity as GP
    shards = P if entry == "mma" else 1
    for i in range(2):
        # codes, (alpha, s) pairs and headers; the alignment padding is never written
        assert GP.same_outputs(outs[i][0].view(shards, -1), outs[i][1], ref[i][0].view(shards, -1), ref[i][1],
                               shards, N, h, n), i
