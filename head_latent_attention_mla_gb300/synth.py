"""Seeded synthetic inputs for one Kimi-K2 MLA layer.

This module only draws and encodes inputs; it holds none of the layer's arithmetic.  Both the
CUDA path (through tests and the benchmark) and the fp64 oracle (through tests) consume the
exact bytes it returns.

Recipe (the model's initializer_range 0.02 and the FP8 quantisation_config on the pages):
  * weights: N(0, 0.02) drawn in float32, one PCG64 stream per matrix (q_a, q_b, kv_a, kv_b,
    o), quantised to OCP e4m3 with one float32 scale per 128x128 block, s = amax/448
    (s = 1 and all-zero codes for an all-zero block); the encode is torch's float8_e4m3fn
    cast (round to nearest even) after clamping to +-448;
  * RMSNorm gains: 1 + U(-0.1, 0.1), rounded to bf16;
  * hidden states: N(0, 1) drawn in float32 and rounded to bf16, one stream per
    (sequence, chunk of 4096 tokens), so any sequence or chunk can be regenerated alone;
  * ragged lengths: U{lo..hi} integers from their own stream.
Every stream is PCG64 seeded by numpy's SeedSequence([seed, tag, ...]).
"""
from __future__ import annotations

import concurrent.futures as _cf
import os

import numpy as np
import torch

HIDDEN, Q_LORA, KV_LORA, HEADS, NOPE, ROPE, VDIM = 7168, 1536, 512, 64, 128, 64, 128
BLOCK = 128
E4M3_MAX = 448.0
CHUNK = 4096

WEIGHT_SHAPES = {
    "q_a": (Q_LORA, HIDDEN),
    "q_b": (HEADS * (NOPE + ROPE), Q_LORA),
    "kv_a": (KV_LORA + ROPE, HIDDEN),
    "kv_b": (HEADS * (NOPE + VDIM), KV_LORA),
    "o": (HIDDEN, HEADS * VDIM),
}
NORM_SIZES = {"q_norm": Q_LORA, "kv_norm": KV_LORA}

_TAG_WEIGHT, _TAG_GAIN, _TAG_HIDDEN, _TAG_LENGTHS = 1, 2, 3, 4


def _rng(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(list(key))))


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 array -> bf16 bit patterns (uint16), round to nearest even (torch's cast)."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def quantise_e4m3_blocks(w: np.ndarray, block: int = BLOCK):
    """float32 [rows, cols] -> (e4m3 codes uint8 [rows, cols], float32 scales
    [ceil(rows/block), ceil(cols/block)]) with s = amax(|block|)/448."""
    rows, cols = w.shape
    rb, cb = -(-rows // block), -(-cols // block)
    pad = np.zeros((rb * block, cb * block), np.float32)
    pad[:rows, :cols] = w
    blocks = torch.from_numpy(pad).reshape(rb, block, cb, block)
    amax = blocks.abs().amax(dim=(1, 3))
    s = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
    scaled = (blocks / s[:, None, :, None]).clamp(-E4M3_MAX, E4M3_MAX)
    q = scaled.to(torch.float8_e4m3fn).view(torch.uint8).reshape(rb * block, cb * block)
    return np.ascontiguousarray(q[:rows, :cols].numpy()), s.numpy().astype(np.float32)


def make_weights(seed: int = 0, shapes: dict | None = None, std: float = 0.02) -> dict:
    """name -> (codes uint8 [out, in], scales float32) for the five projections."""
    shapes = shapes or WEIGHT_SHAPES
    out = {}
    for idx, name in enumerate(("q_a", "q_b", "kv_a", "kv_b", "o")):
        rows, cols = shapes[name]
        w = _rng(seed, _TAG_WEIGHT, idx).standard_normal((rows, cols), dtype=np.float32)
        w *= np.float32(std)
        out[name] = quantise_e4m3_blocks(w)
    return out


def make_gains(seed: int = 0, sizes: dict | None = None) -> dict:
    """name -> bf16 bits of 1 + U(-0.1, 0.1)."""
    sizes = sizes or NORM_SIZES
    out = {}
    for idx, name in enumerate(("q_norm", "kv_norm")):
        u = _rng(seed, _TAG_GAIN, idx).uniform(-0.1, 0.1, size=sizes[name])
        out[name] = to_bf16_bits((1.0 + u).astype(np.float32))
    return out


def make_input_gain(seed: int = 0, hidden: int = HIDDEN) -> np.ndarray:
    """bf16 bits of 1 + U(-0.1, 0.1) for a decoder block's input_layernorm (its own stream)."""
    u = _rng(seed, _TAG_GAIN, 2).uniform(-0.1, 0.1, size=hidden)
    return to_bf16_bits((1.0 + u).astype(np.float32))


def _hidden_chunk(seed: int, seq: int, chunk: int, rows: int, hidden: int) -> np.ndarray:
    x = _rng(seed, _TAG_HIDDEN, seq, chunk).standard_normal((rows, hidden), dtype=np.float32)
    return to_bf16_bits(x)


def hidden_states(seed: int, seq: int, start: int, count: int, hidden: int = HIDDEN,
                  threads: int | None = None) -> np.ndarray:
    """bf16 bits [count, hidden] of sequence `seq`, token indices start..start+count-1.

    Token i of sequence `seq` always has the same value, whatever slice is asked for."""
    if count == 0:
        return np.zeros((0, hidden), np.uint16)
    c0, c1 = start // CHUNK, (start + count - 1) // CHUNK
    threads = threads or min(16, os.cpu_count() or 1)

    def one(c):
        return _hidden_chunk(seed, seq, c, CHUNK, hidden)

    if c1 > c0 and threads > 1:
        with _cf.ThreadPoolExecutor(threads) as ex:
            chunks = list(ex.map(one, range(c0, c1 + 1)))
    else:
        chunks = [one(c) for c in range(c0, c1 + 1)]
    full = np.concatenate(chunks, axis=0) if len(chunks) > 1 else chunks[0]
    off = start - c0 * CHUNK
    return np.ascontiguousarray(full[off: off + count])


def ragged_lengths(seed: int, batch: int, lo: int, hi: int) -> np.ndarray:
    """Integer lengths U{lo..hi} (both ends included) for `batch` sequences."""
    return _rng(seed, _TAG_LENGTHS).integers(lo, hi + 1, size=batch).astype(np.int64)
