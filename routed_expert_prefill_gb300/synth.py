"""Seeded synthetic inputs for the routed mixture-of-experts FFN.

This module only draws random numbers and packs them into the byte layouts
that both the CUDA path and the CPU oracle consume.  It holds none of the
method's arithmetic: no dequantisation, no routing, no GEMM.

Layouts (shared by every consumer):

* ``x``       bf16 bit patterns, uint16 ``[t, h]`` row-major (the normed rows
  that enter the MoE block).
* ``wr``      bf16 bit patterns, uint16 ``[E, h]`` (router weight; logit
  ``e`` of row ``r`` is the dot product of ``x[r, :]`` and ``wr[e, :]``).
* ``rbias``   float32 ``[E]`` or ``None``: per-expert logit bias (only the
  skewed workload has one).
* ``codes``   uint8 ``[E, 3*inter*h*bits/8]``: one record per expert holding,
  in order, gate ``[inter, h]``, up ``[inter, h]`` and down ``[h, inter]``
  codes of ``bits`` bits (4 unless the workload says otherwise), each row
  K-contiguous and packed least significant bit first: code k of a row
  occupies bits ``[k*bits, k*bits + bits)`` of the row's bytes read as one
  little-endian bit string (at 4 bits: two codes per byte, the low nibble at
  the even K index).
* ``scales``/``biases`` float16 ``[E, 3*inter*h/64]``: per output row and
  per 64-wide K group, same matrix order and row-major ``[rows, K/64]``.
* the shared expert uses the same record layout with ``shared_inter``.
"""

from __future__ import annotations

import dataclasses

import numpy as np

GROUP = 64

# Random streams: default_rng([seed, stream]).
_S_X, _S_WR, _S_CODES, _S_SCALES, _S_SKEW, _S_SH_CODES, _S_SH_SCALES, _S_GATE = range(8)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic routed-MoE workload (sizes and the recipe's seed)."""

    name: str
    t: int
    h: int
    inter: int
    E: int
    k: int
    shared_inter: int
    seed: int
    skew: bool = False
    shared_gate: bool = False
    bits: int = 4  # code width of the expert records (2, 3, 4 or 8)

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workload families of the benchmark recipe.  Seed = family index.
WORKLOADS = {
    "tiny_t16_h256_e8": Workload("tiny_t16_h256_e8", 16, 256, 128, 8, 2, 128, 0),
    "t512_h2048_e128": Workload("t512_h2048_e128", 512, 2048, 768, 128, 8, 768, 1),
    "t4096_h2048_e128_skewed": Workload(
        "t4096_h2048_e128_skewed", 4096, 2048, 768, 128, 8, 768, 2, skew=True
    ),
    "t4096_h4096_e256": Workload("t4096_h4096_e256", 4096, 4096, 1536, 256, 8, 1536, 3),
}
# the headline workload with 2-, 3- and 8-bit expert records (same seed)
for _b in (2, 3, 8):
    WORKLOADS[f"t4096_h4096_e256_b{_b}"] = WORKLOADS["t4096_h4096_e256"].replace(
        name=f"t4096_h4096_e256_b{_b}", bits=_b)
for _t in (1, 2, 4, 8):
    WORKLOADS[f"decode_t{_t}_h2048_e128"] = Workload(
        f"decode_t{_t}_h2048_e128", _t, 2048, 768, 128, 8, 768, 4
    )


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest even); return bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def record_bytes(h: int, inter: int, bits: int = 4) -> int:
    """Bytes of codes in one expert record (gate, up, down)."""
    return 3 * inter * h * bits // 8


def record_groups(h: int, inter: int) -> int:
    """Scale (or bias) entries in one expert record."""
    return 3 * inter * h // GROUP


def _quant_record(rng_codes, rng_scales, n: int, h: int, inter: int, bits: int = 4):
    codes = rng_codes.integers(0, 256, size=(n, record_bytes(h, inter, bits)), dtype=np.uint8)
    # scales 2^(4 - bits) times those of the 4-bit records, so the weights
    # span about the same range at every width
    scales = (rng_scales.uniform(0.005, 0.02, size=(n, record_groups(h, inter))) * 2.0 ** (4 - bits)).astype(
        np.float16)
    # bias = -2^(bits-1) * scale: exact in fp16 (a power-of-two multiple).
    biases = (scales * np.float16(-(2.0 ** (bits - 1)))).astype(np.float16)
    return codes, scales, biases


def skew_bias(E: int, seed: int) -> np.ndarray:
    """Per-expert logit bias of the skewed workload: experts get a random
    permutation of Zipf ranks r = 1..E, and bias_e = 2.0 * ln(r_e ** -1.1)."""
    rng = np.random.default_rng([seed, _S_SKEW])
    ranks = rng.permutation(E).astype(np.float64) + 1.0
    return (2.0 * (-1.1) * np.log(ranks)).astype(np.float32)


def make_inputs(w: Workload, t: int | None = None) -> dict:
    """Draw every input of workload ``w`` (optionally with a different row count).

    Rows are drawn from one stream in order, so the first ``t`` rows of a
    larger draw equal a smaller draw with the same seed.
    """
    t = w.t if t is None else t
    g = lambda s: np.random.default_rng([w.seed, s])  # noqa: E731
    x = f32_to_bf16_bits(g(_S_X).standard_normal((t, w.h)).astype(np.float32))
    wr = f32_to_bf16_bits((g(_S_WR).standard_normal((w.E, w.h)) * 0.02).astype(np.float32))
    codes, scales, biases = _quant_record(g(_S_CODES), g(_S_SCALES), w.E, w.h, w.inter, w.bits)
    s_codes, s_scales, s_biases = _quant_record(
        g(_S_SH_CODES), g(_S_SH_SCALES), 1, w.h, w.shared_inter, w.bits
    )
    out = dict(
        x=x,
        wr=wr,
        rbias=skew_bias(w.E, w.seed) if w.skew else None,
        codes=codes,
        scales=scales,
        biases=biases,
        shared_codes=s_codes[0],
        shared_scales=s_scales[0],
        shared_biases=s_biases[0],
        shared_gate=None,
        bits=w.bits,
    )
    if w.shared_gate:
        out["shared_gate"] = f32_to_bf16_bits(
            (g(_S_GATE).standard_normal(w.h) * 0.02).astype(np.float32)
        )
    return out
