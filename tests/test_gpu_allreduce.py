"""The emulated compressed two-shot AllReduce against the oracle's pipeline.

The oracle runs the same five steps with its own compress, reduce_recompress
and decompress on the same rank tensors; the GPU result must match it within
the reconstruction tolerance and approximate the exact sum within the error
of two E4M3 quantisations."""

import dataclasses

import numpy as np
import pytest
import torch

import parity
from grads_taco_compress_gb300 import workloads as W
from grads_taco_compress_gb300.allreduce import EmulatedTwoShotAllReduce
from oracle import taco_oracle as O
from test_gpu_parity import dev_bf16, host_bits

pytestmark = pytest.mark.gpu
E_STAR = 4096.0


def oracle_allreduce(xs, block, fmt=O.FORMAT_E4M3, target=E_STAR):
    R, M, h = xs.shape
    c = M // R
    parts = [[O.compress(xs[r, k * c:(k + 1) * c], block, target, O.VARIANT_DUAL, fmt) for k in range(R)]
             for r in range(R)]
    out = []
    for k in range(R):
        codes = np.stack([parts[r][k][0] for r in range(R)])
        alpha = np.stack([parts[r][k][1] for r in range(R)])
        s = np.stack([parts[r][k][2] for r in range(R)])
        rc, ra, rs, _ = O.reduce_recompress(codes, alpha, s, block, target, O.VARIANT_DUAL, fmt)
        out.append(O.decompress_reduce(rc[None], ra[None], rs[None], block, fmt))
    return np.concatenate(out)


@pytest.mark.parametrize("compress", ["mma", "fwht"])
@pytest.mark.parametrize("name,R,M", [("gpt2-1.5b-act", 4, 64), ("gpt3-6.7b-act", 8, 48),
                                      ("gpt3-6.7b-grad", 2, 30), ("tiny-512x1024", 2, 128)])
def test_allreduce_matches_oracle_pipeline(name, R, M, compress):
    w = dataclasses.replace(W.WORKLOADS[name], P=R)
    xs = W.make_shards(w, N=M)                                   # rank r's tensor in xs[r]
    ar = EmulatedTwoShotAllReduce(R, M, w.h, w.block, compress=compress)
    got = host_bits(ar(dev_bf16(xs)))
    want = oracle_allreduce(xs, w.block)
    parity.compare_recon(O.bf16_bits_to_f64(got), O.bf16_bits_to_f64(want), "allreduce output")
    exact = O.bf16_bits_to_f64(xs).sum(axis=0)
    assert parity.rel_rms(O.bf16_bits_to_f64(got), exact) < 0.06


@pytest.mark.parametrize("name,R,M", [("gpt2-1.5b-act", 4, 64), ("gpt3-6.7b-act", 8, 48),
                                      ("gpt3-6.7b-grad", 2, 30)])
def test_allreduce_int8_matches_oracle_pipeline(name, R, M):
    """The INT8 fallback format through all five steps (E* = 900: RMS 30 levels of 127)."""
    w = dataclasses.replace(W.WORKLOADS[name], P=R)
    xs = W.make_shards(w, N=M)
    ar = EmulatedTwoShotAllReduce(R, M, w.h, w.block, target_energy=900.0, fmt="int8")
    got = host_bits(ar(dev_bf16(xs)))
    want = oracle_allreduce(xs, w.block, O.FORMAT_INT8, 900.0)
    parity.compare_recon(O.bf16_bits_to_f64(got), O.bf16_bits_to_f64(want), "int8 allreduce output")
    exact = O.bf16_bits_to_f64(xs).sum(axis=0)
    assert parity.rel_rms(O.bf16_bits_to_f64(got), exact) < 0.12
    from grads_taco_compress_gb300 import binding as tb
    for hd in ar.reduced_headers:
        assert tb.parse_headers(hd.view(1, -1))[0]["q_max"] == 127.0


def test_allreduce_graph_replay_equals_eager():
    w = dataclasses.replace(W.WORKLOADS["gpt2-1.5b-act"], P=4)
    xs = dev_bf16(W.make_shards(w, N=256))
    ar = EmulatedTwoShotAllReduce(4, 256, w.h, w.block)
    eager = ar(xs).clone()
    g = ar.capture(xs)
    ar.out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(ar.out.view(torch.int16), eager.view(torch.int16))


@pytest.mark.parametrize("block,P", [(64, 5), (128, 3), (256, 2)])
def test_decompress_shards_each_shard_alone(block, P):
    from grads_taco_compress_gb300 import binding as tb
    from test_gpu_parity import bundle_from_arrays
    N, h = 19, 3 * block
    codes, alpha, s = W.make_random_bundle(N, h, block, P, seed=block)
    bundle = bundle_from_arrays(codes, alpha, s, block)
    out = tb.taco_decompress_shards(bundle, P, N, h, block)
    for p in range(P):
        single = tb.taco_decompress_reduce(bundle[p], 1, N, h, block)
        torch.cuda.synchronize()
        assert torch.equal(out[p].view(torch.int16), single.view(torch.int16))
        want = O.decompress_reduce(codes[p:p + 1], alpha[p:p + 1], s[p:p + 1], block)
        parity.compare_recon(O.bf16_bits_to_f64(host_bits(out[p])), O.bf16_bits_to_f64(want))


@pytest.mark.parametrize("fmt", ["e4m3", "int8"])
@pytest.mark.parametrize("name,R,M,S", [("gpt2-1.5b-act", 4, 128, 4), ("gpt3-6.7b-act", 8, 64, 2),
                                        ("gpt3-6.7b-grad", 2, 48, 3), ("tiny-512x1024", 2, 128, 8)])
def test_pipelined_allreduce_equals_serial(name, R, M, S, fmt):
    """Segments on three streams give the serial AllReduce's bits (every
    block's arithmetic is the same), eagerly and replayed from a graph."""
    from grads_taco_compress_gb300.allreduce import PipelinedTwoShotAllReduce
    w = dataclasses.replace(W.WORKLOADS[name], P=R)
    xs = dev_bf16(W.make_shards(w, N=M))
    E = 900.0 if fmt == "int8" else E_STAR
    serial = EmulatedTwoShotAllReduce(R, M, w.h, w.block, target_energy=E, fmt=fmt)(xs).clone()
    pipe = PipelinedTwoShotAllReduce(R, M, w.h, w.block, segments=S, target_energy=E, fmt=fmt)
    eager = pipe(xs).clone()
    torch.cuda.synchronize()
    assert torch.equal(eager.view(torch.int16), serial.view(torch.int16))
    g = pipe.capture(xs)
    pipe.out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(pipe.out.view(torch.int16), serial.view(torch.int16))
    if fmt == "e4m3":
        want = oracle_allreduce(W.make_shards(w, N=M), w.block)
        parity.compare_recon(O.bf16_bits_to_f64(host_bits(eager)), O.bf16_bits_to_f64(want), "pipelined output")
