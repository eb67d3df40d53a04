"""Blocks at the ends of the bf16 range, through the C ABI, against the oracle.

alpha = sqrt(E*/E) is kept inside [2^-126, 2^126] ("TACO ...", gist.science pt
summary, §2.B.1 ASH, with alpha stored in fp32): blocks of bf16 subnormals and
the smallest normals are rescaled only part of the way, and the kernels take
the energy of a block whose sum of squares leaves fp32's trusted range from
the block scaled by an exact power of two. Every tensor here mixes such
blocks with ordinary ones; the codes, alpha and s of every block are compared
with the oracle, and the reconstruction block by block (a tensor-wide RMS
would be dominated by the 3e38 blocks).
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import parity
from grads_taco_compress_gb300 import binding as tb
from grads_taco_compress_gb300 import workloads as W
from oracle import taco_oracle as O

pytestmark = pytest.mark.gpu

E_STAR = 4096.0
MAGNITUDES = (1e-38, 1e-30, 1e-20, 1e20, 1e38, 3e38)


def _bits(v: np.ndarray) -> np.ndarray:
    return W.f32_to_bf16_bits(np.clip(v, -3.3e38, 3.3e38).astype(np.float32))


def _extreme_cases(rng, block: int, aligned: bool = False):
    """(name, values) of the extreme blocks, drawn from `rng`."""
    cases = []
    for m in MAGNITUDES:
        if aligned and m > 1e38:
            continue
        cases.append((f"normal x {m:g}", rng.standard_normal(block) * m))
        # magnitudes in [m, 2m) (values above 3.3e38 clipped): a block of
        # one magnitude with random signs would rotate onto exact E4M3
        # midpoints, where a difference of one fp32 ulp decides the tie
        cases.append((f"[1,2) x {m:g}", m * (1.0 + rng.random(block)) * np.sign(rng.standard_normal(block))))
    spike = np.zeros(block)
    spike[3] = 2.0 ** -133                                          # the smallest bf16
    cases.append(("spike 2^-133", spike))
    spike = np.zeros(block)
    spike[block - 1] = -(2.0 ** -126)
    cases.append(("spike -2^-126", spike))
    mixed = rng.laplace(0.0, 0.02, size=block)
    mixed[7] = 1.0e38 if aligned else 3.0e38                        # one huge element
    cases.append(("laplace + one huge element", mixed))
    sub = rng.standard_normal(block) * 1e-30
    sub[::2] = rng.standard_normal(block // 2) * 1e-39              # subnormals beside 1e-30
    cases.append(("1e-30 with subnormals", sub))
    cases.append(("zero", np.zeros(block)))
    return cases


def extreme_tensor(block: int, P: int = 2, N: int = 20, K: int = 4, seed: int = 0, labels: bool = False,
                   aligned: bool = False):
    """bf16 bits [P, N, K * block]: ordinary blocks with extreme ones among them
    (and, with `labels`, the name of every block's case [P, N, K]).

    Shard p puts its extreme blocks on rows r with r % P == p, so no block
    position holds two huge blocks (their sum would overflow bf16). With
    `aligned` every shard puts the same kind of block on the same rows (the
    sums are extreme too) and the cases at 3e38 are left out."""
    rng = np.random.default_rng(seed + block)
    v = rng.laplace(0.0, 0.02, size=(P, N, K, block))
    names = np.full((P, N, K), "ordinary", dtype=object)
    for p in range(P):
        rows = [r for r in range(N) if r % P == (0 if aligned else p)]
        cases = _extreme_cases(rng, block, aligned)
        for i, (name, c) in enumerate(cases):
            r, k = rows[i % len(rows)], (i // len(rows)) % K
            v[p, r, k] = c
            names[p, r, k] = name
    x = _bits(v.reshape(P, N, K * block))
    return (x, names) if labels else x


def _oracle(x, block, variant, fmt, with_ratio=False):
    parts = [O.compress_stages(x[p], block, E_STAR, variant, fmt) for p in range(x.shape[0])]
    out = (np.stack([st["codes"] for st in parts]), np.stack([st["alpha"] for st in parts]),
           np.stack([st["s"] for st in parts]))
    if not with_ratio:
        return out
    # the fp32 value each code rounds: y / s
    ratio = np.stack([(st["y"].astype(np.float64) / st["s"].astype(np.float64)[..., None]).astype(np.float32)
                      for st in parts])
    return out, ratio.reshape(x.shape)


def _steps(codes, fmt):
    if fmt == O.FORMAT_E4M3:
        return parity.e4m3_ordinal(codes)
    return np.asarray(codes, dtype=np.uint8).view(np.int8).astype(np.int64)


def _near_tie(ratio, fmt):
    """The fp32 values y / s that lie within 2^-20 (relative) of a rounding
    midpoint of the code format, where the last bits of the arithmetic
    decide the code."""
    r = np.abs(np.asarray(ratio, dtype=np.float64))
    if fmt == O.FORMAT_E4M3:
        vals = O.e4m3_decode_table()[:127]
        mids = (vals[:-1] + vals[1:]) / 2
    else:
        mids = np.arange(127) + 0.5
    i = np.clip(np.searchsorted(mids, r), 1, len(mids) - 1)
    d = np.minimum(np.abs(r - mids[i - 1]), np.abs(r - mids[i]))
    return d <= np.maximum(r, 2.0 ** -9) * 2.0 ** -20


def _compare_compress(got, want, fmt, what, ratio=None, names=None, block=None, scale_rtol=None):
    """Codes equal to the oracle's except at most one step where the oracle's
    y / s sits on a rounding midpoint (when `ratio` is given; else the
    operator's tolerance); alpha and s within 1e-6 (or `scale_rtol` [P,N,K]
    per block); every mismatch named."""
    codes, alpha, s = got
    oc, oa, os_ = want
    if fmt == O.FORMAT_E4M3:
        assert not np.any((codes & 0x7F) == 0x7F), what
    diff = np.abs(_steps(codes, fmt) - _steps(oc, fmt))
    if ratio is not None:
        bad = (diff > 1) | ((diff == 1) & ~_near_tie(ratio.reshape(diff.shape), fmt))
        if bad.any():
            idx = np.argwhere(bad)[:6]
            detail = []
            for p, r, e in idx:
                k = e // block
                detail.append(f"shard {p} row {r} block {k} ({names[p, r, k]}) element {e % block}: "
                              f"got {int(codes[p, r, e]):#04x}, oracle {int(oc[p, r, e]):#04x}, "
                              f"oracle y/s {float(ratio.reshape(diff.shape)[p, r, e]):.9g}")
            raise AssertionError(f"{what}: {int(bad.sum())} codes off beyond a tie\n" + "\n".join(detail))
    else:
        for p in range(codes.shape[0]):
            if fmt == O.FORMAT_E4M3:
                parity.compare_codes(codes[p], oc[p], f"{what} codes[{p}]")
            else:
                parity.compare_int8_codes(codes[p], oc[p], f"{what} codes[{p}]")
    if scale_rtol is None:
        for p in range(codes.shape[0]):
            parity.compare_scales(alpha[p], oa[p], f"{what} alpha[{p}]")
            parity.compare_scales(s[p], os_[p], f"{what} s[{p}]")
    else:
        for name, g_, w_ in (("alpha", alpha, oa), ("s", s, os_)):
            rel = np.abs(g_.astype(np.float64) - w_) / np.abs(w_.astype(np.float64))
            assert np.all(rel <= scale_rtol), f"{what} {name}: relative difference {rel.max():.3e}"
    assert np.all(np.isfinite(alpha)) and alpha.max() <= 2.0 ** 126 and alpha.min() >= 2.0 ** -126


def _code_blocks_equal(codes, oc, block, fmt):
    """[P * N * K] bool: the block's codes equal the oracle's in value."""
    d = np.abs(_steps(codes, fmt) - _steps(oc, fmt)).reshape(codes.shape[0], -1, block)
    return np.all(d == 0, axis=-1)


def _compare_blocks(got_bits, want_bits, block, what, max_overflow_blocks=0, same_codes=None):
    """Per block: relative RMS within the bar, zero blocks exactly zero.

    A block of values near the bf16 maximum (3e38) can reconstruct beyond the
    bf16 range, since its E4M3 codes round up by as much as 1/16: the oracle
    gives +-inf there, and the GPU's fp32 sums overflow too, in a pattern
    that is not compared. At most `max_overflow_blocks` such blocks."""
    g = O.bf16_bits_to_f64(got_bits).reshape(-1, block)
    w = O.bf16_bits_to_f64(want_bits).reshape(-1, block)
    if same_codes is not None:
        # a block position whose codes broke a rounding tie the other way in
        # some shard (checked at the code level) is not compared here
        keep = np.all(same_codes, axis=0)
        assert keep.sum() >= keep.size - 4, (what, int((~keep).sum()))
        g, w = g[keep], w[keep]
        got_bits = np.asarray(got_bits).reshape(-1, block)[keep]
        want_bits = np.asarray(want_bits).reshape(-1, block)[keep]
    over = ~np.all(np.isfinite(w), axis=-1)
    assert int(over.sum()) <= max_overflow_blocks, (what, int(over.sum()))
    g, w = g[~over], w[~over]
    gb = np.asarray(got_bits).reshape(-1, block)[~over]
    wb = np.asarray(want_bits).reshape(-1, block)[~over]
    assert np.all(np.isfinite(g)), what
    den = np.linalg.norm(w, axis=-1)
    err = np.linalg.norm(g - w, axis=-1)
    zero = den == 0
    assert np.all(err[zero] == 0), what
    rel = np.where(zero, 0.0, err / np.where(zero, 1.0, den))
    # or every element within one bf16 step of the oracle's (blocks of bf16
    # subnormals, where one step is up to a few percent of the value)
    def ordinal(b):
        b = b.astype(np.int64)
        return np.where(b & 0x8000, -(b & 0x7FFF), b & 0x7FFF)
    one_step = np.max(np.abs(ordinal(gb) - ordinal(wb)), axis=-1) <= 1
    ok = (rel <= parity.RECON_REL_RMS) | one_step
    worst = float(np.max(np.where(ok, 0.0, rel)))
    assert ok.all(), f"{what}: worst block relative RMS {worst:.3e}"


COMPRESS_ENTRIES = {
    "mma": (tb.taco_compress_shards_mma, O.FORMAT_E4M3),
    "fwht": (tb.taco_compress_shards_fwht, O.FORMAT_E4M3),
    "int8": (tb.taco_compress_shards_int8, O.FORMAT_INT8),
}


@pytest.mark.parametrize("block", [64, 128, 256])
@pytest.mark.parametrize("variant", [tb.VARIANT_DUAL, tb.VARIANT_ABSMAX, tb.VARIANT_STATIC])
@pytest.mark.parametrize("entry", sorted(COMPRESS_ENTRIES))
def test_compress_extreme_blocks(block, variant, entry):
    fn, fmt = COMPRESS_ENTRIES[entry]
    x, names = extreme_tensor(block, labels=True)
    P, N, h = x.shape
    xd = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda()
    bundle, _ = fn(xd, block, E_STAR, variant)
    codes, alpha, s = (t.cpu().numpy() for t in tb.shard_views(bundle, P, N, h, block))
    want, ratio = _oracle(x, block, variant, fmt, with_ratio=True)
    _compare_compress((codes, alpha, s), want, fmt, f"{entry} n={block} v={variant}", ratio, names, block)
    # decompress-reduce of the GPU's own bundle, block by block against the
    # oracle's reconstruction of the oracle's codes
    dec = tb.taco_decompress_reduce if fmt == O.FORMAT_E4M3 else tb.taco_decompress_reduce_int8
    out = dec(bundle, P, N, h, block)
    got = out.view(torch.int16).cpu().numpy().view(np.uint16)
    ref = O.decompress_reduce(*want, block, fmt)
    same = _code_blocks_equal(codes, want[0], block, fmt)
    _compare_blocks(got, ref, block, f"{entry} n={block} v={variant} decompress-reduce", 2 * P, same)
    if fmt == O.FORMAT_E4M3 and block in (64, 128):
        out = tb.taco_decompress_reduce_mma(bundle, P, N, h, block)
        got = out.view(torch.int16).cpu().numpy().view(np.uint16)
        _compare_blocks(got, ref, block, f"{entry} n={block} v={variant} tensor-core decompress-reduce",
                        2 * P, same)


@pytest.mark.parametrize("block", [64, 256])
@pytest.mark.parametrize("entry", ["mma", "int8"])
def test_compress_extreme_blocks_in_the_shared_tile_pool(block, entry):
    """Four shards of [2048, 16 n], large enough that about a quarter of each
    shard's tiles go to the pool that every CTA of the tensor-core compress
    claims from, so a CTA compresses tiles of other shards than its own.
    Every 128-block tile holds one extreme block (the cases above in turn),
    so blocks that take the rescale and exact paths (the latter re-reads the
    block from its own shard's x) sit in pool tiles too. Codes, alpha and s
    against the oracle as for the small tensors."""
    fn, fmt = COMPRESS_ENTRIES[entry]
    P, N, K = 4, 2048, 16
    rng = np.random.default_rng(77 + block)
    v = rng.laplace(0.0, 0.02, size=(P, N * K, block))
    names = np.full((P, N * K), "ordinary", dtype=object)
    cases = _extreme_cases(rng, block)
    for p in range(P):
        for t in range(N * K // 128):
            name, c = cases[(t + p) % len(cases)]
            b = t * 128 + int(rng.integers(0, 128))
            v[p, b] = c
            names[p, b] = name
    x = _bits(v.reshape(P, N, K * block))
    h = K * block
    xd = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda()
    bundle, _ = fn(xd, block, E_STAR, tb.VARIANT_DUAL)
    codes, alpha, s = (t.cpu().numpy() for t in tb.shard_views(bundle, P, N, h, block))
    want, ratio = _oracle(x, block, tb.VARIANT_DUAL, fmt, with_ratio=True)
    _compare_compress((codes, alpha, s), want, fmt, f"{entry} n={block} pooled", ratio,
                      names.reshape(P, N, K), block)


@pytest.mark.parametrize("target", [E_STAR, 1e-30, 2.0 ** 100])
@pytest.mark.parametrize("variant", [tb.VARIANT_DUAL, tb.VARIANT_ABSMAX, tb.VARIANT_STATIC])
@pytest.mark.parametrize("entry", sorted(COMPRESS_ENTRIES))
def test_compress_extreme_blocks_extreme_target(entry, variant, target):
    """A tiny and a huge target energy E* on the same blocks: the factors the
    kernels form from alpha, s and the codes stay inside the fp32 range."""
    fn, fmt = COMPRESS_ENTRIES[entry]
    block = 128
    x, names = extreme_tensor(block, labels=True, seed=3)
    P, N, h = x.shape
    xd = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda()
    bundle, _ = fn(xd, block, target, variant)
    codes, alpha, s = (t.cpu().numpy() for t in tb.shard_views(bundle, P, N, h, block))
    parts = [O.compress_stages(x[p], block, target, variant, fmt) for p in range(P)]
    want = (np.stack([st["codes"] for st in parts]), np.stack([st["alpha"] for st in parts]),
            np.stack([st["s"] for st in parts]))
    ratio = np.stack([(st["y"].astype(np.float64) / st["s"].astype(np.float64)[..., None]).astype(np.float32)
                      for st in parts]).reshape(x.shape)
    _compare_compress((codes, alpha, s), want, fmt, f"{entry} v={variant} E*={target:g}", ratio, names, block)


@pytest.mark.parametrize("aligned", [False, True])
@pytest.mark.parametrize("variant", [tb.VARIANT_DUAL, tb.VARIANT_ABSMAX, tb.VARIANT_STATIC])
@pytest.mark.parametrize("block", [64, 128, 256])
@pytest.mark.parametrize("fmt", [O.FORMAT_E4M3, O.FORMAT_INT8])
def test_reduce_recompress_extreme_blocks(block, fmt, variant, aligned):
    """Sums of extreme blocks with ordinary ones, and (aligned) sums that are
    themselves tiny or huge, recompressed."""
    x, names = extreme_tensor(block, seed=5, aligned=aligned, labels=True)
    P, N, h = x.shape
    oc, oa, os_ = _oracle(x, block, O.VARIANT_DUAL, fmt)
    sb = tb.shard_bytes(N, h, block)
    off = tb.shard_scales_offset(N, h, block)
    buf = np.zeros((P, sb), dtype=np.uint8)
    for p in range(P):
        buf[p, : N * h] = oc[p].reshape(-1)
        pairs = np.stack([oa[p], os_[p]], axis=-1).astype(np.float32)
        buf[p, off: off + pairs.nbytes] = pairs.view(np.uint8).reshape(-1)
    shards = [torch.from_numpy(buf[p].copy()).cuda() for p in range(P)]
    entry = tb.taco_reduce_recompress_ptrs if fmt == O.FORMAT_E4M3 else tb.taco_reduce_recompress_int8_ptrs
    shard, _, _ = entry(shards, N, h, block, E_STAR, variant)
    rc, ra, rs = (t.cpu().numpy() for t in tb.shard_views(shard[None], 1, N, h, block))
    wc, wa, ws, _ = O.reduce_recompress(oc, oa, os_, block, E_STAR, variant, fmt)
    # the value each recompressed code rounds (the oracle's own steps)
    st = O.compress_values_stages(O.decompress_reduce_f64(oc, oa, os_, block, fmt), block, E_STAR, variant, fmt)
    assert np.array_equal(st["codes"], wc)
    ratio = (st["y"].astype(np.float64) / st["s"].astype(np.float64)[..., None]).astype(np.float32)
    # A shard block whose alpha is clamped at 2^126 decodes with the factor
    # s / (alpha sqrt(n)) below fp32's normal range (about 19 significant
    # bits): where every input block at a position is one, the fp32 sum z
    # carries that precision into the recompressed scales.
    tiny_inputs = np.all(oa == np.float32(2.0 ** 126), axis=0)[None]
    rtol = np.where(tiny_inputs, 1e-5, parity.SCALE_RTOL)
    _compare_compress((rc, ra, rs), (wc[None], wa[None], ws[None]), fmt,
                      f"recompress n={block} v={variant} aligned={aligned}", ratio.reshape(1, N, h),
                      names[:1], block, scale_rtol=rtol)


def test_no_kernel_wait_timed_out_extreme():
    assert tb.taco_get_fault() == 0
