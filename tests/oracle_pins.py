"""Pins of the CPU oracle against things other than itself.

Each ``check_*`` takes the oracle module and raises AssertionError when it
disagrees with a closed form, a library routine, a printed format point, an
invariant or a brute-force search. ``tests/test_oracle_pins.py`` runs them
on the oracle; ``tests/test_oracle_mutations.py`` runs them on copies of the
oracle with one planted mistake each and requires some check to fail.
"""

from __future__ import annotations

import math
import pathlib

import numpy as np

GOLDEN = pathlib.Path(__file__).parent / "golden"
E_STAR = 4096.0


def _bf16_bits(v) -> np.ndarray:
    """Exact bf16 bit patterns of values that are bf16 already."""
    v32 = np.asarray(v, dtype=np.float32)
    u = v32.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "value is not a bf16 number"
    return (u >> 16).astype(np.uint16)


def _random_bf16(rng, shape, scale=1.0):
    """Random bf16 bit patterns (truncation of fp32 normals; input only)."""
    v = (rng.standard_normal(shape) * scale).astype(np.float32)
    return (v.view(np.uint32) >> 16).astype(np.uint16)


# --------------------------------------------------------------------------
# Hadamard
# --------------------------------------------------------------------------
def check_hadamard_orthogonal(O):
    for k in range(0, 9):
        n = 1 << k
        H = O.sylvester_hadamard(n)
        assert np.array_equal(H @ H.T, n * np.eye(n, dtype=H.dtype)), n


def check_hadamard_scipy(O):
    scipy_linalg = __import__("scipy.linalg", fromlist=["hadamard"])
    for n in (1, 2, 4, 64, 128, 256):
        assert np.array_equal(O.sylvester_hadamard(n), scipy_linalg.hadamard(n)), n


def check_hadamard_closed_form(O):
    n = 256
    i = np.arange(n)[:, None]
    j = np.arange(n)[None, :]
    pop = np.vectorize(lambda v: bin(int(v)).count("1"))(i & j)
    assert np.array_equal(O.sylvester_hadamard(n), np.where(pop % 2 == 0, 1, -1))


# --------------------------------------------------------------------------
# E4M3 codec
# --------------------------------------------------------------------------
def check_e4m3_decode_torch(O):
    import torch
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = O.e4m3_decode_table()
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], got[ok])


def _torch_e4m3_codes(v32: np.ndarray) -> np.ndarray:
    import torch
    t = torch.from_numpy(np.ascontiguousarray(v32, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def check_e4m3_encode_torch_all_bf16(O):
    """Every bf16 pattern with |v| <= 448 against torch's float8_e4m3fn cast."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    v = (bits.astype(np.uint32) << 16).view(np.float32)
    keep = np.isfinite(v) & (np.abs(v) <= 448.0)
    v = v[keep]
    assert np.array_equal(O.e4m3_encode(v), _torch_e4m3_codes(v))


def check_e4m3_encode_torch_ties(O):
    """Exact midpoints between neighbouring E4M3 values, and random fp32."""
    table = O.e4m3_decode_table()[:127]
    mids = ((table[:-1] + table[1:]) / 2).astype(np.float32)
    assert np.array_equal(mids.astype(np.float64), (table[:-1] + table[1:]) / 2)
    rng = np.random.default_rng(7)
    rnd = (np.exp2(rng.uniform(-12, np.log2(448.0), 200_000))).astype(np.float32)
    v = np.concatenate([mids, -mids, rnd, -rnd])
    v = v[np.abs(v) <= 448.0]
    assert np.array_equal(O.e4m3_encode(v), _torch_e4m3_codes(v))


def check_e4m3_points(O):
    for line in (GOLDEN / "e4m3_points.txt").read_text().splitlines():
        line = line.split("#")[0].strip()
        if not line:
            continue
        expr, code = line.split()
        val = eval(expr, {"__builtins__": {}}, {"float": float})
        got = int(O.e4m3_encode(np.array([val], dtype=np.float32))[0])
        assert got == int(code, 16), (expr, hex(got), code)


def check_e4m3_roundtrip(O):
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = O.e4m3_decode(codes).astype(np.float32)
    assert np.array_equal(O.e4m3_encode(vals), codes)


# --------------------------------------------------------------------------
# bf16 rounding of the reduced output
# --------------------------------------------------------------------------
def check_bf16_round_torch(O):
    import torch
    rng = np.random.default_rng(11)
    u = rng.integers(0, 1 << 32, size=400_000, dtype=np.uint64).astype(np.uint32)
    # include exact ties (low half 0x8000) and values near the top of the range
    u[:50_000] = (u[:50_000] & 0xFFFF0000) | 0x8000
    u[50_000:51_000] = 0x7F7F0000 + rng.integers(0, 0x10000, 1000).astype(np.uint32)
    v = u.view(np.float32)
    v = v[np.isfinite(v)]
    ref = torch.from_numpy(v.copy()).to(torch.bfloat16).to(torch.float64).numpy()
    got = O.round_to_bf16(v.astype(np.float64))
    assert np.array_equal(ref, got)


def check_bf16_round_bruteforce_f64(O):
    """fp64 inputs that fp32 cannot hold: nearest of the two bf16 neighbours."""
    rng = np.random.default_rng(12)
    v = rng.standard_normal(20_000) * np.exp2(rng.uniform(-30, 30, 20_000))
    got = O.round_to_bf16(v)
    for x, g in zip(v[:4000], got[:4000]):
        t = np.float32(x)
        b = int(np.array([t]).view(np.uint32)[0]) >> 16           # a nearby bf16 pattern
        cands = []
        for d in (-2, -1, 0, 1, 2):
            bb = (b + d) & 0xFFFF
            cv = float(np.array([bb << 16], dtype=np.uint32).view(np.float32)[0])
            if math.isfinite(cv):
                cands.append((abs(cv - x), bb & 1, cv))
        cands.sort()
        best = cands[0]
        if len(cands) > 1 and cands[1][0] == best[0]:                # tie: even pattern
            best = min(cands[:2], key=lambda c: c[1])
        assert g == best[2], (x, g, best)


# --------------------------------------------------------------------------
# Energy, rotation and the dual scale
# --------------------------------------------------------------------------
def check_energy_invariant(O):
    rng = np.random.default_rng(3)
    for n in (64, 128, 256):
        for scale in (1e-4, 1e-2, 3.0):
            x = _random_bf16(rng, (16, 4 * n), scale)
            st = O.compress_stages(x, n, E_STAR)
            xb = O.bf16_bits_to_f64(x).reshape(16, 4, n)
            a = st["alpha"].astype(np.float64)[..., None]
            e_after = np.mean((a * xb) ** 2, axis=-1)
            assert np.allclose(e_after, E_STAR, rtol=3e-7, atol=0), (n, scale)
            # the rotated block keeps that energy: sum y^2 = n E*
            y = st["y"].astype(np.float64)
            assert np.allclose(np.sum(y * y, axis=-1), n * E_STAR, rtol=2e-6), (n, scale)


def check_dual_scale_guard(O):
    rng = np.random.default_rng(4)
    for n in (64, 128, 256):
        x = _random_bf16(rng, (64, 2 * n), 0.01)
        # make some blocks concentrated (a Hadamard row times a constant)
        x[:8, :n] = _bf16_bits(np.full(n, 0.5, dtype=np.float32))
        st = O.compress_stages(x, n, E_STAR)
        s = st["s"].astype(np.float64)
        assert np.all(s >= 1.0)
        clamped = st["amax"] > 448.0
        assert np.array_equal(s > 1.0, clamped)
        assert np.allclose(s[clamped], st["amax"][clamped] / 448.0, rtol=1e-7)
        assert np.all(np.abs(O.e4m3_decode(st["codes"])) <= 448.0)
        assert st["header"]["n_clamped"] == int(clamped.sum()) >= 8
        assert st["header"]["s_max"] == float(s.max())


def _closed_form_rows():
    for line in (GOLDEN / "closed_form_blocks.txt").read_text().splitlines():
        line = line.split("#")[0].strip()
        if line:
            n, case, alpha_c, s, code = line.split()
            yield int(n), case, float(alpha_c), float(s), int(code, 16)


def check_spike_and_constant_blocks(O):
    rng = np.random.default_rng(5)
    for n, case, alpha_c, s_ref, code in _closed_form_rows():
        H = O.sylvester_hadamard(n)
        for c in (0.0078125, -3.5, 0.001220703125):
            cb = float(np.float32(c))
            xv = np.zeros(n, dtype=np.float32)
            if case == "spike":
                j = int(rng.integers(n))
                xv[j] = cb
                sign = np.sign(cb) * H[:, j]
                want = np.where(sign > 0, code, code | 0x80)
            else:
                xv[:] = cb
                want = np.zeros(n, dtype=np.int64)
                want[0] = code if cb > 0 else code | 0x80
            x = _bf16_bits(xv)[None, :]
            codes, alpha, s, hdr = O.compress(x, n, E_STAR)
            assert math.isclose(float(alpha[0, 0]) * abs(cb), alpha_c, rel_tol=2e-7), (n, case)
            assert math.isclose(float(s[0, 0]), s_ref, rel_tol=2e-7), (n, case)
            got = codes[0].astype(np.int64)
            nonzero = want & 0x7F != 0
            assert np.array_equal(got[nonzero], want[nonzero]), (n, case)
            assert np.all(got[~nonzero] & 0x7F == 0), (n, case)
            assert hdr["n_clamped"] == (1 if case == "constant" else 0)
            # reconstruction is the input itself
            rec = O.decompress_reduce(codes[None], alpha[None], s[None], n)
            assert np.array_equal(rec, x), (n, case)


def check_zero_block(O):
    for n in (64, 128, 256):
        x = np.zeros((2, 2 * n), dtype=np.uint16)
        x[1, n:] = _bf16_bits(np.full(n, 2.0, np.float32))    # a non-zero neighbour
        codes, alpha, s, _ = O.compress(x, n, E_STAR)
        assert alpha[0, 0] == 1.0 and alpha[0, 1] == 1.0 and alpha[1, 0] == 1.0
        assert s[0, 0] == 1.0 and s[1, 0] == 1.0
        assert np.all(codes[0] & 0x7F == 0) and np.all(codes[1, :n] & 0x7F == 0)
        rec = O.decompress_reduce(codes[None], alpha[None], s[None], n)
        assert np.all(O.bf16_bits_to_f64(rec[0]) == 0.0)
        assert np.all(O.bf16_bits_to_f64(rec[1, :n]) == 0.0)


def check_absmax_variant(O):
    rng = np.random.default_rng(6)
    n = 128
    x = _random_bf16(rng, (32, 4 * n), 0.02)
    c1, _, s1, _ = O.compress(x, n, E_STAR, O.VARIANT_ABSMAX)
    c2, _, _, _ = O.compress(x, n, 3.0, O.VARIANT_ABSMAX)
    mag = np.abs(O.e4m3_decode(c1)).reshape(32, 4, n)
    assert np.all(mag.max(axis=-1) == 448.0)          # the block maximum maps to Q_max
    assert np.mean(c1 == c2) > 0.9999                 # alpha cancels from the codes


def check_static_variant(O):
    """STATIC: one scale sqrt(n E*)/Q_max for every block; Cauchy-Schwarz bound.

    After the energy rescale ||y||^2 = n E*, so |y_i| <= sqrt(n E*): a block
    equal to a scaled Hadamard row reaches the bound (one code +-448, the rest
    zero), a spike block spreads evenly (every code +-448/sqrt(n)), and no
    ratio y/s of any block exceeds 448.
    """
    rng = np.random.default_rng(12)
    for n in (64, 128, 256):
        s_ref = np.float32(math.sqrt(n * E_STAR) / 448.0)
        H = O.sylvester_hadamard(n)
        for c in (0.0078125, -3.5):
            k = int(rng.integers(n))
            row = _bf16_bits(np.float32(c) * H[k].astype(np.float32))[None, :]
            codes, alpha, s, hdr = O.compress(row, n, E_STAR, O.VARIANT_STATIC)
            assert s[0, 0] == s_ref
            want = np.zeros(n, dtype=np.int64)
            want[k] = 0x7E if c > 0 else 0xFE
            got = codes[0].astype(np.int64)
            assert got[k] == want[k], (n, c)
            assert np.all(np.delete(got, k) & 0x7F == 0), (n, c)
            spike = np.zeros(n, dtype=np.float32)
            spike[k] = c
            codes, _, _, _ = O.compress(_bf16_bits(spike)[None, :], n, E_STAR, O.VARIANT_STATIC)
            mag = np.abs(O.e4m3_decode(codes[0]))
            target = 448.0 / math.sqrt(n)
            assert np.all(mag == mag[0])
            if n in (64, 256):
                assert mag[0] == target                     # 56 and 28: exact E4M3 values
            else:
                assert abs(mag[0] - target) <= 2.0 ** (math.floor(math.log2(target)) - 4)
        x = _random_bf16(rng, (16, 4 * n), 0.02)
        x[3, :n] = 0                                          # a zero block keeps alpha = 1
        st = O.compress_stages(x, n, E_STAR, O.VARIANT_STATIC)
        assert np.all(st["s"] == s_ref)
        assert st["alpha"][3, 0] == 1.0 and np.all(st["codes"][3, :n] & 0x7F == 0)
        ratio = np.abs(st["y"].astype(np.float64) / float(s_ref))
        assert ratio.max() <= 448.0 * (1 + 1e-6)
        assert st["header"]["n_clamped"] == (st["s"].size if s_ref > 1.0 else 0)
        assert st["header"]["s_max"] == float(s_ref)


# --------------------------------------------------------------------------
# Blocks at the ends of the bf16 range: alpha kept inside [2^-126, 2^126]
# --------------------------------------------------------------------------
def _exact_pow2_scale(bits: np.ndarray, k: int) -> np.ndarray:
    """bf16 patterns of 2^k x, exact (every |x| and |2^k x| a normal number)."""
    v = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64) * 2.0 ** k
    return _bf16_bits(v.astype(np.float32))


def check_power_of_two_equivariance(O):
    """compress(2^k x) = compress(x) with alpha scaled by exactly 2^-k.

    Energy, alpha and the rotation are homogeneous in x: E(2^k x) = 4^k E(x),
    so sqrt(E*/E) scales by exactly 2^-k, and alpha x, y, s and the codes do
    not change. This holds for k across the whole bf16 exponent range as long
    as alpha stays inside [2^-126, 2^126]; an energy or alpha computed in a
    narrower format than the input's range breaks it at one end.
    """
    rng = np.random.default_rng(22)
    for n in (64, 128, 256):
        v = rng.standard_normal((6, 2 * n)) * np.exp2(rng.uniform(-5, 5, (6, 2 * n)))
        v = np.where(np.abs(v) < 2.0 ** -12, 2.0 ** -12, v)      # every |x| in [2^-12, 2^12]
        x0 = (v.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
        x0[2, :n] = 0                                            # a zero block stays a zero block
        for fmt in (O.FORMAT_E4M3, O.FORMAT_INT8):
            for variant in O.VARIANTS:
                c0, a0, s0, _ = O.compress(x0, n, E_STAR, variant, fmt)
                for k in list(range(-112, 111, 9)) + [-113, 114]:
                    ck, ak, sk, _ = O.compress(_exact_pow2_scale(x0, k), n, E_STAR, variant, fmt)
                    assert np.array_equal(ck, c0), (n, fmt, variant, k)
                    assert np.array_equal(sk, s0), (n, fmt, variant, k)
                    want = np.where(a0 == 1.0, 1.0, a0.astype(np.float64) * 2.0 ** -k)
                    want[2, 0] = 1.0
                    assert np.array_equal(ak.astype(np.float64), want), (n, fmt, variant, k)


def _extreme_rows():
    for line in (GOLDEN / "extreme_blocks.txt").read_text().splitlines():
        line = line.split("#")[0].strip()
        if line:
            n, case, c, E, alpha, s, code, recon = line.split()
            ev = lambda t: float(eval(t, {"__builtins__": {}}, {}))
            yield int(n), case, ev(c), ev(E), ev(alpha), float(s), int(code, 16), recon


def check_alpha_clamp_closed_forms(O):
    """Spike and constant blocks whose sqrt(E*/E) leaves [2^-126, 2^126]."""
    for n, case, c, E, alpha_ref, s_ref, code, recon in _extreme_rows():
        H = O.sylvester_hadamard(n)
        j = 5
        xv = np.zeros(n, dtype=np.float64)
        if case == "spike":
            xv[j] = c
            want = np.where(np.sign(c) * H[:, j] > 0, code, code | 0x80)
        else:
            xv[:] = c
            want = np.zeros(n, dtype=np.int64)
            want[0] = code if c > 0 else code | 0x80
        x = _bf16_bits(xv.astype(np.float32))[None, :]
        codes, alpha, s, _ = O.compress(x, n, E)
        assert float(alpha[0, 0]) == alpha_ref, (n, case, c, float(alpha[0, 0]))
        assert float(s[0, 0]) == s_ref, (n, case, c)
        got = codes[0].astype(np.int64)
        nonzero = want & 0x7F != 0
        assert np.array_equal(got[nonzero], want[nonzero]), (n, case, c)
        assert np.all(got[~nonzero] & 0x7F == 0), (n, case, c)
        rec = O.decompress_reduce(codes[None], alpha[None], s[None], n)
        if recon == "exact":
            assert np.array_equal(rec, x), (n, case, c)
        elif recon == "zero":
            assert np.all(O.bf16_bits_to_f64(rec) == 0.0), (n, case, c)


def check_extreme_magnitudes(O):
    """Blocks anywhere in the bf16 range, subnormals included.

    No finite input gives a NaN code, alpha stays inside [2^-126, 2^126], s is
    finite (>= 1 for the dual scale), and the reconstruction is within the
    E4M3 error of the alpha and s actually stored: per block
      ||x_hat - x||_2 <= (s / alpha) (||max(|r| 2^-4, 2^-10)||_2 + 2^-22 ||r||_2),
    r = y / s the value rounded to E4M3 (half a step: 2^-4 relative in the
    normal range, 2^-10 in the subnormal range; 2^-22 covers the two fp32
    roundings of y and y / s), since the rotation is orthonormal.
    """
    rng = np.random.default_rng(23)
    for n in (64, 128, 256):
        rows, K = 40, 3
        ex = rng.integers(-134, 127, size=(rows, K, 1)).astype(np.float64)
        v = rng.standard_normal((rows, K, n)) * np.exp2(ex)
        v[::5, 1, :] = 0.0
        v[1::5, 1, :] *= np.exp2(rng.uniform(-40, 0, (len(v[1::5]), n)))   # wide range inside a block
        v[2::5, 2, 7] = 3.0e38                                              # one huge element
        v = np.clip(v, -3.3e38, 3.3e38).reshape(rows, K * n)
        x = (v.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
        xv = O.bf16_bits_to_f64(x).reshape(rows, K, n)
        for variant in O.VARIANTS:
            st = O.compress_stages(x, n, E_STAR, variant)
            codes, alpha, s = st["codes"], st["alpha"].astype(np.float64), st["s"].astype(np.float64)
            assert not np.any((codes & 0x7F) == 0x7F), (n, variant)
            assert np.all(np.isfinite(alpha)) and np.all((alpha >= 2.0 ** -126) & (alpha <= 2.0 ** 126))
            assert np.all(np.isfinite(s)) and np.all(s > 0)
            if variant == O.VARIANT_DUAL:
                assert np.all(s >= 1.0)
            rec = O.decompress_reduce_f64(codes[None], st["alpha"][None], st["s"][None], n)
            err = np.linalg.norm(rec.reshape(rows, K, n) - xv, axis=-1)
            r = st["y"].astype(np.float64) / s[..., None]
            half_step = np.maximum(np.abs(r) * 2.0 ** -4, 2.0 ** -10)
            bound = (s / alpha) * (np.linalg.norm(half_step, axis=-1)
                                   + 2.0 ** -22 * np.linalg.norm(r, axis=-1))
            assert np.all(err <= bound * (1 + 1e-9)), (n, variant, float(np.max(err / bound)))


def _nearest_int_tie_even(v: float) -> int:
    """Nearest integer by comparing the two neighbours (no library rounding)."""
    lo = math.floor(v)
    d_lo, d_hi = v - lo, lo + 1 - v
    if d_lo < d_hi:
        return lo
    if d_hi < d_lo:
        return lo + 1
    return lo if lo % 2 == 0 else lo + 1


def check_int8_codec(O):
    """INT8 codes: nearest integer, ties to even, clamp to +-127; two's complement bytes."""
    ints = np.arange(-127, 128)
    assert np.array_equal(O.int8_decode(O.int8_encode(ints.astype(np.float32))), ints)
    assert np.array_equal(O.int8_encode(ints.astype(np.float32)), (ints & 0xFF).astype(np.uint8))
    assert np.array_equal(O.int8_decode(np.arange(256, dtype=np.uint8)),
                          np.concatenate([np.arange(0, 128), np.arange(-128, 0)]).astype(np.float64))
    rng = np.random.default_rng(13)
    v = np.concatenate([np.arange(-130, 130.5, 0.25), rng.uniform(-140, 140, 2000),
                        [0.49999997, -0.49999997, 1e-30, -1e-30, 127.5, -127.5, 1e30, -1e30, np.inf, -np.inf]])
    v = v.astype(np.float32)
    got = O.int8_decode(O.int8_encode(v))
    want = [max(-127, min(127, _nearest_int_tie_even(float(x)))) if np.isfinite(x)
            else (127 if x > 0 else -127) for x in v]
    assert np.array_equal(got, np.array(want, dtype=np.float64))
    assert np.all(O.int8_encode(v) != 0x80)                  # -128 is never produced


def check_int8_closed_forms(O):
    """The FP8 closed forms with Q_max = 127: spike -> +-sqrt(E*) = +-64, constant -> one 127."""
    for n in (64, 128, 256):
        H = O.sylvester_hadamard(n)
        for c in (0.0078125, -3.5):
            j = 5 % n
            spike = np.zeros(n, np.float32)
            spike[j] = c
            x = _bf16_bits(spike)[None, :]
            codes, alpha, s, hdr = O.compress(x, n, E_STAR, O.VARIANT_DUAL, O.FORMAT_INT8)
            assert s[0, 0] == 1.0 and hdr["q_max"] == 127.0
            want = np.where(np.sign(c) * H[:, j] > 0, 64, -64)
            assert np.array_equal(O.int8_decode(codes[0]), want.astype(np.float64))
            assert np.array_equal(O.decompress_reduce(codes[None], alpha[None], s[None], n, O.FORMAT_INT8), x)
            const = _bf16_bits(np.full(n, c, np.float32))[None, :]
            codes, alpha, s, hdr = O.compress(const, n, E_STAR, O.VARIANT_DUAL, O.FORMAT_INT8)
            assert math.isclose(float(s[0, 0]), math.sqrt(n * E_STAR) / 127.0, rel_tol=2e-7)
            q = O.int8_decode(codes[0])
            assert q[0] == (127 if c > 0 else -127) and np.all(q[1:] == 0)
            assert np.array_equal(O.decompress_reduce(codes[None], alpha[None], s[None], n, O.FORMAT_INT8), const)


def check_int8_error_bound(O):
    """Uniform steps of s: every rotated value is off by at most s/2, so a block's
    reconstruction error is at most (s/2) sqrt(n) / alpha (the rotation is orthonormal)."""
    rng = np.random.default_rng(14)
    for n, E in ((64, 4096.0), (128, 900.0), (256, 150.0)):
        x = _random_bf16(rng, (24, 4 * n), 0.01)
        x[:, 3] = _random_bf16(rng, (24,), 2.0)
        codes, alpha, s, _ = O.compress(x, n, E, O.VARIANT_DUAL, O.FORMAT_INT8)
        rec = O.decompress_reduce_f64(codes[None], alpha[None], s[None], n, O.FORMAT_INT8)
        err = (rec - O.bf16_bits_to_f64(x)).reshape(24, 4, n)
        bound = s.astype(np.float64) / 2 * math.sqrt(n) / alpha.astype(np.float64)
        assert np.all(np.linalg.norm(err, axis=-1) <= bound * (1 + 1e-5) + 1e-30)
        assert np.all(np.abs(O.int8_decode(codes)) <= 127)


# --------------------------------------------------------------------------
# Decompress-reduce: sum in the rotated domain, invert once (linearity)
# --------------------------------------------------------------------------
def check_reduce_linearity(O):
    scipy_linalg = __import__("scipy.linalg", fromlist=["hadamard"])
    rng = np.random.default_rng(8)
    for n, P in ((64, 3), (128, 2), (256, 4)):
        N, h = 8, 2 * n
        K = h // n
        codes = rng.integers(0, 256, size=(P, N, h)).astype(np.uint8)
        codes[(codes & 0x7F) == 0x7F] = 0x11                      # no NaN codes
        alpha = np.exp(rng.uniform(-3, 9, size=(P, N, K))).astype(np.float32)
        s = np.maximum(1.0, np.exp(rng.normal(0, 0.5, size=(P, N, K)))).astype(np.float32)
        table = O.e4m3_decode_table()
        vals = table[codes].reshape(P, N, K, n)
        z = np.sum((s.astype(np.float64) / alpha.astype(np.float64))[..., None] * vals, axis=0)
        ref = (z @ scipy_linalg.hadamard(n).astype(np.float64)) / math.sqrt(n)
        got = O.decompress_reduce_f64(codes, alpha, s, n).reshape(N, K, n)
        assert np.allclose(got, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max()), (n, P)


def check_recompress_spike_blocks(O):
    """A reduced spike block is a spike again: the same +-64 codes, exactly."""
    rng = np.random.default_rng(13)
    for n in (64, 128, 256):
        xv = np.zeros((3, 2 * n), dtype=np.float32)
        for r in range(3):
            xv[r, int(rng.integers(2 * n))] = (-1.0) ** r * 0.375 * (r + 1)
        x = _bf16_bits(xv)
        codes, alpha, s, _ = O.compress(x, n, E_STAR)
        rc, ra, rs, _ = O.reduce_recompress(codes[None], alpha[None], s[None], n, E_STAR)
        assert np.array_equal(rc, codes), n
        assert np.allclose(ra, alpha, rtol=2e-7) and np.array_equal(rs, s), n


def check_recompress_scale_invariance(O):
    """Summing a shard with itself doubles x_hat: alpha halves, codes and s stay."""
    rng = np.random.default_rng(14)
    for n in (64, 128, 256):
        N, h = 16, 2 * n
        codes = rng.integers(0, 256, size=(1, N, h)).astype(np.uint8)
        codes[(codes & 0x7F) == 0x7F] = 0x21
        alpha = np.exp(rng.uniform(0, 8, size=(1, N, h // n))).astype(np.float32)
        s = np.maximum(1.0, np.exp(rng.normal(0, 0.3, size=(1, N, h // n)))).astype(np.float32)
        c1, a1, s1, _ = O.reduce_recompress(codes, alpha, s, n, E_STAR)
        c2, a2, s2, _ = O.reduce_recompress(np.concatenate([codes, codes]), np.concatenate([alpha, alpha]),
                                            np.concatenate([s, s]), n, E_STAR)
        assert np.mean(c1 == c2) > 0.9999, n
        assert np.allclose(a2, a1 / 2, rtol=2e-7), n
        assert np.allclose(s2, s1, rtol=2e-7), n


def check_recompress_reconstructs(O):
    """Decoding the recompressed shard gives back x_hat within E4M3 error."""
    rng = np.random.default_rng(15)
    n, P, N, h = 128, 3, 24, 512
    xs = np.stack([_random_bf16(rng, (N, h), 0.02) for _ in range(P)])
    parts = [O.compress(xs[p], n, E_STAR) for p in range(P)]
    codes = np.stack([c for c, _, _, _ in parts])
    alpha = np.stack([a for _, a, _, _ in parts])
    s = np.stack([sc for _, _, sc, _ in parts])
    x_hat = O.decompress_reduce_f64(codes, alpha, s, n)
    rc, ra, rs, hdr = O.reduce_recompress(codes, alpha, s, n, E_STAR)
    back = O.decompress_one_f64(rc, ra, rs, n)
    rel = np.linalg.norm(back - x_hat) / np.linalg.norm(x_hat)
    assert 0.005 < rel < 0.04, rel
    assert hdr["N"] == N and hdr["h"] == h and hdr["n_clamped"] == int(np.count_nonzero(rs > 1))


def check_roundtrip_error(O):
    """One shard round trip: the error of a 3-bit-mantissa code, not more."""
    rng = np.random.default_rng(9)
    for n in (64, 128, 256):
        x = _random_bf16(rng, (64, 4 * n), 0.01)
        codes, alpha, s, _ = O.compress(x, n, E_STAR)
        rec = O.bf16_bits_to_f64(O.decompress_reduce(codes[None], alpha[None], s[None], n))
        ref = O.bf16_bits_to_f64(x)
        rel = np.linalg.norm(rec - ref) / np.linalg.norm(ref)
        assert 0.005 < rel < 0.04, (n, rel)


def check_wire_ratio(O):
    """FP8 codes plus two fp32 scales per block: near the pages' ~45% cut."""
    for n in (64, 128, 256):
        saving = 1.0 - O.wire_bytes_per_element(n) / 2.0
        assert 0.40 < saving < 0.50, (n, saving)


ALL_CHECKS = [v for k, v in sorted(globals().items()) if k.startswith("check_")]
