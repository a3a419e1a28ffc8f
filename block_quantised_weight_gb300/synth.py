"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This module only draws random bytes and floats; it holds none of the format's
decoding arithmetic. Both the CUDA path and the CPU oracle receive exactly the
arrays produced here.

Value recipe (the block layouts are the ones page 1 "Rewriting picoLM in
Python" gives for ``dequantize_q4_K`` and page 4 "iq3_pack.py" gives in its
module docstring):

* Q4_K, 144 bytes per 256 weights: the two fp16 fields at bytes 0-3 are
  ``d ~ U(1e-3, 4e-3)`` and ``dmin ~ U(0, 2e-3)``, each rounded to fp16
  (round-to-nearest-even, numpy ``astype``); the other 140 bytes (12 packed
  scale/min bytes and 128 nibble bytes) are uniform uint8.
* IQ3, 98 bytes per 256 weights: bytes 0-95 are uniform uint8 (64 grid-index
  bytes, then eight little-endian uint32 whose 28 sign bits and 4-bit sub-scale
  code are uniform, so the whole word is uniform); bytes 96-97 hold
  ``d ~ U(1e-3, 4e-3)`` rounded to fp16.
* The IQ3 grid is 256 rows x 4 bytes drawn i.i.d. from the doubled-unit
  magnitudes {4, 12, 20, 28, 36, 44, 52, 62}.
* Activations ``x`` are fp32 ``N(0, 1)``, shape ``[M, K]``.
* Page 3's other codebook formats (block sizes, d at bytes 0-1, the rest of
  the bytes uniform uint8, d ~ U(1e-3, 4e-3) rounded to fp16; the codebooks
  are not printed on the pages, so they are drawn too):
  IQ4_NL (18 bytes per 32 weights, eight blocks per 256) and IQ4_XS (136
  bytes per 256) with a table of 16 distinct sorted int8 values drawn from
  [-127, 127]; IQ3_S (110 bytes) with a 512 x 4 grid drawn from
  {1, 3, ..., 15}; IQ2_XXS (66 bytes) with a 256 x 8 grid drawn from
  {8, 24, 40}.  Draw order: codebook, the block bytes, d.

Draw order for one Q4_K matrix: d, dmin, the 12 scale bytes, the 128 qs bytes,
then x. For one IQ3 matrix: grid, the 96 index/word bytes, d, then x.
"""
from __future__ import annotations

import numpy as np

QK = 256                 # weights per super-block (both formats)
Q4K_BLOCK_BYTES = 144    # page 1, dequantize_q4_K docstring
IQ3_BLOCK_BYTES = 98     # page 4, module docstring / BLOCK_BYTES

IQ3_GRID_LEVELS = np.array([4, 12, 20, 28, 36, 44, 52, 62], dtype=np.uint8)


def _rng(seed) -> np.random.Generator:
    if isinstance(seed, np.random.Generator):
        return seed
    return np.random.default_rng(seed)


def _fp16_bytes(values: np.ndarray) -> np.ndarray:
    """fp32/fp64 values -> little-endian fp16 bytes [n, 2] (numpy RNE rounding)."""
    return np.ascontiguousarray(values.astype("<f2")).view(np.uint8).reshape(-1, 2)


def gen_q4k(N: int, K: int, seed) -> np.ndarray:
    """Random Q4_K matrix as uint8 ``[N, K/256*144]`` (row n, then block b)."""
    if K % QK:
        raise ValueError(f"K must be a multiple of {QK}, got {K}")
    rng = _rng(seed)
    nblk = N * (K // QK)
    d = rng.uniform(1e-3, 4e-3, nblk)
    dmin = rng.uniform(0.0, 2e-3, nblk)
    scales = rng.integers(0, 256, (nblk, 12), dtype=np.uint8)
    qs = rng.integers(0, 256, (nblk, 128), dtype=np.uint8)
    blk = np.empty((nblk, Q4K_BLOCK_BYTES), dtype=np.uint8)
    blk[:, 0:2] = _fp16_bytes(d)
    blk[:, 2:4] = _fp16_bytes(dmin)
    blk[:, 4:16] = scales
    blk[:, 16:144] = qs
    return blk.reshape(N, -1)


def gen_iq3_grid(seed) -> np.ndarray:
    """Random IQ3 codebook, uint8 ``[256, 4]`` in doubled units."""
    rng = _rng(seed)
    return IQ3_GRID_LEVELS[rng.integers(0, len(IQ3_GRID_LEVELS), (256, 4))]


def gen_iq3(N: int, K: int, seed, grid_seed=None):
    """Random IQ3 matrix: returns ``(W uint8 [N, K/256*98], grid uint8 [256, 4])``.

    The grid is drawn first from the same generator unless ``grid_seed`` is
    given.
    """
    if K % QK:
        raise ValueError(f"K must be a multiple of {QK}, got {K}")
    rng = _rng(seed)
    grid = gen_iq3_grid(rng if grid_seed is None else grid_seed)
    nblk = N * (K // QK)
    body = rng.integers(0, 256, (nblk, 96), dtype=np.uint8)
    d = rng.uniform(1e-3, 4e-3, nblk)
    blk = np.empty((nblk, IQ3_BLOCK_BYTES), dtype=np.uint8)
    blk[:, 0:96] = body
    blk[:, 96:98] = _fp16_bytes(d)
    return blk.reshape(N, -1), grid


# Page 3's codebook formats: bytes per 256 weights, bytes per fp16 d field
# (one per 32 weights for IQ4_NL, one per 256 otherwise).
CB_UNIT_BYTES = {"iq4nl": 144, "iq4xs": 136, "iq3s": 110, "iq2xxs": 66}


def gen_cb_table(fmt: str, seed) -> np.ndarray:
    """Random codebook of a page-3 format: int8 [16] (IQ4), uint8 [512, 4]
    (IQ3_S) or uint8 [256, 8] (IQ2_XXS)."""
    rng = _rng(seed)
    if fmt in ("iq4nl", "iq4xs"):
        return np.sort(rng.choice(np.arange(-127, 128), 16, replace=False)).astype(np.int8)
    if fmt == "iq3s":
        return (2 * rng.integers(0, 8, (512, 4)) + 1).astype(np.uint8)
    if fmt == "iq2xxs":
        return np.array([8, 24, 40], dtype=np.uint8)[rng.integers(0, 3, (256, 8))]
    raise ValueError(fmt)


def gen_cb(fmt: str, N: int, K: int, seed):
    """Random matrix of a page-3 codebook format: ``(W uint8 [N, K/256*B], table)``."""
    if K % QK:
        raise ValueError(f"K must be a multiple of {QK}, got {K}")
    rng = _rng(seed)
    table = gen_cb_table(fmt, rng)
    units = N * (K // QK)
    if fmt == "iq4nl":   # eight 18-byte blocks per 256 weights, each with its own d
        nblk = 8 * units
        blk = rng.integers(0, 256, (nblk, 18), dtype=np.uint8)
        blk[:, 0:2] = _fp16_bytes(rng.uniform(1e-3, 4e-3, nblk))
    else:
        blk = rng.integers(0, 256, (units, CB_UNIT_BYTES[fmt]), dtype=np.uint8)
        blk[:, 0:2] = _fp16_bytes(rng.uniform(1e-3, 4e-3, units))
    return blk.reshape(N, -1), table


def gen_x(M: int, K: int, seed) -> np.ndarray:
    """Activations, fp32 ``[M, K]`` ~ N(0, 1)."""
    rng = _rng(seed)
    return rng.standard_normal((M, K), dtype=np.float32)


# TinyLlama-1.1B decode pass: 22 layers of q, k, v, o, gate, up, down, then the
# output projection (shapes from page 1's CLI model; 32 q heads, 4 kv heads,
# head_dim 64, hidden 2048, FFN 5632, vocab 32000).
TINYLLAMA_LAYERS = 22
TINYLLAMA_LAYER_SHAPES = (          # (name, K = n_in, N = n_out)
    ("q", 2048, 2048),
    ("k", 2048, 256),
    ("v", 2048, 256),
    ("o", 2048, 2048),
    ("gate", 2048, 5632),
    ("up", 2048, 5632),
    ("down", 5632, 2048),
)
TINYLLAMA_OUTPUT = ("output", 2048, 32000)


def tinyllama_shapes():
    """The 155 (layer, name, K, N) GEMVs of one decode step, in execution order."""
    out = []
    for layer in range(TINYLLAMA_LAYERS):
        for name, K, N in TINYLLAMA_LAYER_SHAPES:
            out.append((layer, name, K, N))
    out.append((TINYLLAMA_LAYERS, *TINYLLAMA_OUTPUT))
    return out


def tinyllama_seeds(seed: int = 1):
    """One child seed per matrix of the pass, spawned from ``seed`` in pass order."""
    shapes = tinyllama_shapes()
    children = np.random.SeedSequence(seed).spawn(len(shapes))
    return [(s, np.random.default_rng(c)) for s, c in zip(shapes, children)]


def q4k_row_bytes(K: int) -> int:
    return K // QK * Q4K_BLOCK_BYTES


def iq3_row_bytes(K: int) -> int:
    return K // QK * IQ3_BLOCK_BYTES
