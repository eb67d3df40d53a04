"""Seeded synthetic inputs for the TACO operator: shapes and value mixes only.

This module holds none of the operator's arithmetic. It draws bf16 tensors
shaped like the tensor-parallel activations and gradients that the TACO
pages train on (GPT-2-1.5B, GPT-3-6.7B, Qwen-7B; "TACO: Efficient
Communication Compression of Intermediate Tensors ...", euno.news results
table) and, for decompress-reduce inputs that must not come from any
implementation, random shard bundles (codes plus per-block scales).

Every draw is seeded: config-level choices (outlier channels, per-channel
scales) come from ``SeedSequence([seed, 0])`` and shard ``p`` from
``SeedSequence([seed, 1 + p])`` (numpy PCG64). Values are drawn in float64,
rounded to float32 and then to bf16 (both round-to-nearest-even).
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    N: int            # tokens (rows)
    h: int            # hidden size (columns)
    block: int        # Hadamard block size n
    P: int            # shards summed by decompress-reduce
    kind: str         # value mix, see _draw_values
    params: dict = field(default_factory=dict)
    seed: int = 0

    @property
    def K(self) -> int:
        return self.h // self.block

    @property
    def elements(self) -> int:
        return self.N * self.h


WORKLOADS = {
    # [512 tokens, 1024 hidden], n=128, P=2: 99% Laplace(0, 0.01) and
    # 1% Student-t(3) x 0.5 per element; 4 fixed outlier channels x 20.
    "tiny-512x1024": Workload("tiny-512x1024", 512, 1024, 128, 2, "laplace_t_mix",
                              dict(b=0.01, p_t=0.01, nu=3.0, t_scale=0.5,
                                   n_channels=4, channel_gain=20.0)),
    # GPT-2-1.5B TP activation: [8 x 1024 = 8192, 1600], n=64, P=4, same
    # mixture, 16 (1%) outlier channels x 30.
    "gpt2-1.5b-act": Workload("gpt2-1.5b-act", 8192, 1600, 64, 4, "laplace_t_mix",
                              dict(b=0.01, p_t=0.01, nu=3.0, t_scale=0.5,
                                   n_channels=16, channel_gain=30.0)),
    # GPT-3-6.7B TP activation: [4 x 2048 = 8192, 4096], n=128, P=8:
    # Laplace(0, 0.005) with 0.5% of entries replaced by t(2.5) x 0.5.
    "gpt3-6.7b-act": Workload("gpt3-6.7b-act", 8192, 4096, 128, 8, "laplace_t_replace",
                              dict(b=0.005, p_t=0.005, nu=2.5, t_scale=0.5)),
    # TP backward gradient of the same model: [8192, 4096], n=256, P=8:
    # Gaussian(0, 1e-4), 0.1% of entries x 1000, then 10% set to exact zero.
    "gpt3-6.7b-grad": Workload("gpt3-6.7b-grad", 8192, 4096, 256, 8, "gauss_spikes_zeros",
                               dict(sigma=1e-4, p_spike=0.001, spike_gain=1000.0,
                                    p_zero=0.10)),
    # Qwen-7B long sequence: [2 x 8192 = 16384, 3584], n=128, P=8:
    # Laplace(0, 0.01) times a per-channel lognormal(0, 1.5) scale, and
    # 8 massive-activation channels x 100.
    "qwen-7b-long": Workload("qwen-7b-long", 16384, 3584, 128, 8, "laplace_lognormal_channels",
                             dict(b=0.01, ln_sigma=1.5, n_channels=8, channel_gain=100.0)),
}

#: the workload the benchmark's step times at one GPU: the largest one
BENCH_WORKLOAD = "qwen-7b-long"


def f32_to_bf16_bits(v32: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(v32, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def _config_rng(w: Workload) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([w.seed, 0]))


def _shard_rng(w: Workload, p: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([w.seed, 1 + p]))


def _draw_values(w: Workload, rng: np.random.Generator, N: int, h: int,
                 cfg_rng_state: dict) -> np.ndarray:
    k = w.params
    shape = (N, h)
    if w.kind == "laplace_t_mix":
        v = rng.laplace(0.0, k["b"], size=shape)
        m = rng.random(shape) < k["p_t"]
        v[m] = rng.standard_t(k["nu"], size=int(m.sum())) * k["t_scale"]
        v[:, cfg_rng_state["channels"]] *= k["channel_gain"]
    elif w.kind == "laplace_t_replace":
        v = rng.laplace(0.0, k["b"], size=shape)
        m = rng.random(shape) < k["p_t"]
        v[m] = rng.standard_t(k["nu"], size=int(m.sum())) * k["t_scale"]
    elif w.kind == "gauss_spikes_zeros":
        v = rng.normal(0.0, k["sigma"], size=shape)
        m = rng.random(shape) < k["p_spike"]
        v[m] *= k["spike_gain"]
        z = rng.random(shape) < k["p_zero"]
        v[z] = 0.0
    elif w.kind == "laplace_lognormal_channels":
        v = rng.laplace(0.0, k["b"], size=shape)
        v *= cfg_rng_state["channel_scale"][None, :h]
        v[:, cfg_rng_state["channels"]] *= k["channel_gain"]
    else:
        raise ValueError(w.kind)
    return v


def _config_state(w: Workload) -> dict:
    rng = _config_rng(w)
    st = {}
    nch = w.params.get("n_channels", 0)
    st["channels"] = np.sort(rng.choice(w.h, nch, replace=False)) if nch else np.zeros(0, int)
    if w.kind == "laplace_lognormal_channels":
        st["channel_scale"] = rng.lognormal(0.0, w.params["ln_sigma"], size=w.h)
    return st


def make_shard(w: Workload, p: int = 0, N: int | None = None) -> np.ndarray:
    """bf16 bit patterns (uint16) [N, h] of shard ``p``.

    ``N`` overrides the row count (a smaller case of the same mix); the first
    rows of a shorter draw are not the first rows of a longer one.
    """
    N = w.N if N is None else N
    st = _config_state(w)
    rng = _shard_rng(w, p)
    return f32_to_bf16_bits(_draw_values(w, rng, N, w.h, st).astype(np.float32))


def make_shards(w: Workload, N: int | None = None, P: int | None = None) -> np.ndarray:
    """bf16 bit patterns [P, N, h]."""
    P = w.P if P is None else P
    return np.stack([make_shard(w, p, N) for p in range(P)])


def make_random_bundle(N: int, h: int, block: int, P: int, seed: int = 0):
    """Random decompress-reduce inputs: codes u8 [P,N,h], alpha, s f32 [P,N,K].

    Codes are sign-magnitude bytes with the magnitude ordinal drawn from a
    bell shape over 0..126 (0x7F/0xFF, the NaN patterns, never occur);
    alpha is lognormal around 5000 and s is 1 for 90% of blocks and
    1 + |N(0, 0.5)| for the rest. These are shapes only; no encoder runs.
    """
    K = h // block
    rng = np.random.default_rng(np.random.SeedSequence([seed, 0xB0D1E]))
    ordinal = np.clip(np.rint(rng.normal(100.0, 18.0, size=(P, N, h))), 0, 126)
    sign = (rng.random((P, N, h)) < 0.5).astype(np.uint8) << 7
    codes = ordinal.astype(np.uint8) | sign
    alpha = rng.lognormal(np.log(5000.0), 1.0, size=(P, N, K)).astype(np.float32)
    s = np.ones((P, N, K), dtype=np.float32)
    big = rng.random((P, N, K)) < 0.10
    s[big] = (1.0 + np.abs(rng.normal(0.0, 0.5, size=int(big.sum())))).astype(np.float32)
    return codes, alpha, s
