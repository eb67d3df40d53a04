"""Plant one plausible mistake in a copy of the oracle; some pin must catch it.

Each mutation edits one expression of the oracle's source (a dropped term, a
wrong sign, an inverted ratio, a wrong tie rule ...), loads the edited copy
as a separate module on the CPU and runs every pin against it.
"""

import importlib.util
import pathlib

import pytest

import oracle_pins

SRC = (pathlib.Path(__file__).resolve().parent.parent / "oracle" / "taco_oracle.py").read_text()

MUTATIONS = {
    "rotation_not_normalised": ("y = ((scaled @ H.T) / math.sqrt(n))", "y = ((scaled @ H.T) / 1.0)"),
    "alpha_inverted": ("np.sqrt(target_energy / energy[nz])", "np.sqrt(energy[nz] / target_energy)"),
    "energy_sum_not_mean": ("energy = np.sum(x * x, axis=-1) / n", "energy = np.sum(x * x, axis=-1)"),
    "energy_centred": ("energy = np.sum(x * x, axis=-1) / n",
                       "energy = np.var(x, axis=-1)"),
    "no_overflow_floor": ("np.maximum(1.0, amax / qm)", "(amax / qm)"),
    "qmax_wrong": ("Q_MAX = 448.0", "Q_MAX = 240.0"),
    "hadamard_sign_moved": ("h = np.block([[h, h], [h, -h]])", "h = np.block([[h, -h], [h, h]])"),
    "e4m3_ties_odd": ("(hi % 2 == 0)", "(hi % 2 == 1)"),
    "e4m3_ties_away": ("((d_hi == d_lo) & (hi % 2 == 0))", "(d_hi == d_lo)"),
    "e4m3_bias_8": ("2.0 ** (exp_field - 7)", "2.0 ** (exp_field - 8)"),
    "e4m3_no_subnormal_scale": ("man_field * 2.0 ** -9", "man_field * 2.0 ** -10"),
    "decode_forgets_s": ("w = np.asarray(s, dtype=np.float32).astype(np.float64)[..., None] * q",
                         "w = q"),
    "decode_forgets_alpha": ("xr = u / np.asarray(alpha, dtype=np.float32).astype(np.float64)[..., None]",
                             "xr = u"),
    "decode_not_normalised": ("u = (w @ H) / math.sqrt(n)", "u = (w @ H) / n"),
    "bf16_truncates": ("np.rint(np.ldexp(v[finite], -q))", "np.trunc(np.ldexp(v[finite], -q))"),
    "reduce_drops_last_shard": ("for p in range(P):", "for p in range(P - 1):"),
    "recompress_first_shard_only": ("x_hat = decompress_reduce_f64(codes, alpha, s, block, fmt)",
                                    "x_hat = decompress_reduce_f64(codes[:1], alpha[:1], s[:1], block, fmt)"),
    "static_scale_drops_n": ("math.sqrt(block * float(target_energy)) / q_max(fmt)",
                             "math.sqrt(float(target_energy)) / q_max(fmt)"),
    "static_scale_per_block_amax": ("np.full((N, K), np.float32(static_scale(n, target_energy, fmt)), dtype=np.float32)",
                                    "np.maximum(1.0, amax / qm).astype(np.float32)"),
    "int8_ties_up": ("q = np.rint(np.where(np.isnan(v32), 0.0, v32))",
                     "q = np.floor(np.where(np.isnan(v32), 0.0, v32) + 0.5)"),
    "int8_qmax_128": ("Q_MAX_INT8 = 127.0", "Q_MAX_INT8 = 128.0"),
    "int8_decode_unsigned": ("np.asarray(codes, dtype=np.uint8).view(np.int8).astype(np.float64)",
                             "np.asarray(codes, dtype=np.uint8).astype(np.float64)"),
    "int8_scale_uses_fp8_qmax": ("    qm = q_max(fmt)\n", "    qm = Q_MAX\n"),
    "recompress_skips_alpha": ("    st = compress_values_stages(x_hat, block, target_energy, variant, fmt)\n    return st[\"codes\"], st[\"alpha\"]",
                               "    st = compress_values_stages(x_hat, block, target_energy, variant, fmt)\n    return st[\"codes\"], st[\"alpha\"] * 0 + 1"),
    "energy_in_fp32": ("energy = np.sum(x * x, axis=-1) / n",
                       "energy = np.sum(x.astype(np.float32) ** 2, axis=-1, dtype=np.float32).astype(np.float64) / n"),
    "alpha_unclamped": ("np.clip(np.sqrt(target_energy / energy[nz]), ALPHA_MIN, ALPHA_MAX)",
                        "np.sqrt(target_energy / energy[nz])"),
    "alpha_clamp_at_fp32_max": ("ALPHA_MAX = 2.0 ** 126", "ALPHA_MAX = float(np.finfo(np.float32).max)"),
    "alpha_clamp_low_subnormal": ("ALPHA_MIN = 2.0 ** -126", "ALPHA_MIN = 2.0 ** -149"),
    "alpha_applied_unclamped": ("    scaled = alpha.astype(np.float64)[..., None] * x\n",
                                "    scaled = np.where(energy > 0, np.sqrt(target_energy / np.where(energy > 0, energy, 1.0)), 1.0)[..., None] * x\n"),
}


def _load_mutant(name, tmp_path):
    old, new = MUTATIONS[name]
    assert SRC.count(old) == 1, f"mutation anchor not unique/found: {old!r}"
    path = tmp_path / f"oracle_mutant_{name}.py"
    path.write_text(SRC.replace(old, new))
    spec = importlib.util.spec_from_file_location(path.stem, path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path):
    mod = _load_mutant(name, tmp_path)
    failed = []
    for check in oracle_pins.ALL_CHECKS:
        try:
            check(mod)
        except (AssertionError, ValueError, IndexError, FloatingPointError):
            failed.append(check.__name__)
    assert failed, f"no pin caught the planted mistake {name}"
