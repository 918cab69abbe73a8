"""Shared helpers of the GPU parity tests: seeded inputs, oracle references computed from the
same bytes, and the error measures the parity bar is stated in."""
import functools
import os

import numpy as np
import torch

from head_latent_attention_mla_gb300 import synth
from oracle import mla_oracle as O

REL_FRO_TOL = 1e-2     # relative Frobenius error of layer outputs
MAX_ABS_TOL = 5e-2     # max-abs error of layer outputs
ORACLE_CHUNK = 8192    # tokens per oracle cache-row batch (memory bound only)


@functools.lru_cache(maxsize=1)
def weights_and_gains(seed: int = 0):
    return synth.make_weights(seed), synth.make_gains(seed)


@functools.lru_cache(maxsize=1)
def oracle_weights(seed: int = 0):
    wq, g = weights_and_gains(seed)
    return O.weights_from_quantised(wq, g)


def to_dev(bits: np.ndarray) -> torch.Tensor:
    """bf16 bit patterns (uint16) -> bf16 CUDA tensor."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def errors(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return (float(np.linalg.norm(got - ref) / np.linalg.norm(ref)),
            float(np.max(np.abs(got - ref))))


# (test id, what, rel_fro, max_abs) of every comparison in this process; the terminal summary
# prints them so a run shows how far inside the bar each case sits.
MARGINS: list = []


def assert_close(got, ref, what=""):
    rel, mx = errors(got, ref)
    test = os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0].split("::")[-1]
    MARGINS.append((test, what, rel, mx))
    assert rel <= REL_FRO_TOL and mx <= MAX_ABS_TOL, f"{what}: rel_fro={rel:.3e} max_abs={mx:.3e}"
    return rel, mx


def oracle_cache(seed: int, seq: int, n: int, W) -> np.ndarray:
    """Oracle latent cache [n, 576] of sequence `seq`'s first n tokens."""
    rows = []
    for s0 in range(0, n, ORACLE_CHUNK):
        s1 = min(n, s0 + ORACLE_CHUNK)
        x = O.bf16_to_f64(synth.hidden_states(seed, seq, s0, s1 - s0))
        rows.append(O.cache_rows(x, np.arange(s0, s1), W))
    return np.concatenate(rows, axis=0) if rows else np.zeros((0, 576))


def oracle_rows(x: np.ndarray, rows: np.ndarray, cache: np.ndarray, W) -> np.ndarray:
    """Oracle outputs of tokens at positions `rows` (prefill from position 0, x = all tokens),
    given the full oracle cache of those tokens."""
    xr = x[rows]
    q_nope, q_pe = O.query(xr, W)
    q_rot = np.transpose(O.apply_rope(np.transpose(q_pe, (1, 0, 2)), rows), (1, 0, 2))
    o = O.attend(q_nope, q_rot, rows, cache[: int(rows.max()) + 1], W)
    return O.output(o, W)


def build_caches_gpu(layer, seed: int, lengths, cap: int, chunk: int = 16384):
    """Device caches [B, cap, 576] holding lengths[b] tokens of sequence b, appended through
    mla_cache_append, with device lengths; returns (cache, seq_lens_dev)."""
    B = len(lengths)
    cache = torch.zeros(B, cap, 576, dtype=torch.bfloat16, device="cuda")
    lens = torch.zeros(B, dtype=torch.int32, device="cuda")
    for b in range(B):
        done = 0
        while done < lengths[b]:
            n = min(chunk, lengths[b] - done)
            x = to_dev(synth.hidden_states(seed, b, done, n))[None]
            layer.cache_append(x, cache[b:b + 1], lens[b:b + 1], [done])
            done += n
    torch.cuda.synchronize()
    return cache, lens
