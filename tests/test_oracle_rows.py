"""The oracle split over row ranges in worker processes (tests/oracle_rows.py)
gives exactly what one call of the oracle gives: blocks never straddle rows,
so the ranges are independent. Checked on CPU with uneven ranges (more
pieces than a row count divides evenly) for compress, decompress-reduce and
reduce-recompress, bit for bit."""

from __future__ import annotations

import numpy as np
import pytest

from grads_taco_compress_gb300 import workloads as W
from oracle import taco_oracle as O
from oracle_rows import OracleRows


@pytest.fixture(scope="module")
def pool():
    p = OracleRows(workers=3)
    yield p
    p.close()


@pytest.mark.parametrize("block,variant,fmt", [(64, O.VARIANT_DUAL, O.FORMAT_E4M3),
                                               (256, O.VARIANT_ABSMAX, O.FORMAT_E4M3),
                                               (128, O.VARIANT_DUAL, O.FORMAT_INT8)])
def test_row_ranges_equal_one_call(pool, block, variant, fmt):
    P, N, h, E = 3, 37, 2 * block, 30000.0
    rng = np.random.default_rng(block + fmt)
    x = W.f32_to_bf16_bits(rng.laplace(0, 0.1, size=(P, N, h)).astype(np.float32))
    codes, alpha, s = pool.compress(x, block, E, variant, fmt)
    for p in range(P):
        c, a, sc, _ = O.compress(x[p], block, E, variant, fmt)
        assert np.array_equal(codes[p], c) and np.array_equal(alpha[p], a) and np.array_equal(s[p], sc)
    assert np.array_equal(pool.decompress_reduce(codes, alpha, s, block, fmt),
                          O.decompress_reduce(codes, alpha, s, block, fmt))
    rc, ra, rs = pool.reduce_recompress(codes, alpha, s, block, E, variant, fmt)
    oc, oa, os_, _ = O.reduce_recompress(codes, alpha, s, block, E, variant, fmt)
    assert np.array_equal(rc, oc) and np.array_equal(ra, oa) and np.array_equal(rs, os_)
