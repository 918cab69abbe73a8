"""Oracle for the forward pass of one Kimi-K2 multi-head latent attention (MLA) layer.

TEST INFRASTRUCTURE ONLY.  This module is plain, slow, double-precision CPU code that
states what the layer computes, in the explicit (non-absorbed) form that the Kimi K2
model-atlas pages print.  Only the tests, the smoke check and the CPU-baseline leg of the
benchmark may import it.  It shares no code with the CUDA path and never imports it.

Sources (page title, then the section or excerpt on it):
  * "Kimi K2 · Key–value latent" page: the `mla-init` excerpt (module layout), the `mla-kv`
    excerpt (joint down-projection, split, latent norm, kv_b up-projection), the `linear`
    excerpt (FP8 e4m3 weights with 128x128 block scales) and the `rmsnorm` excerpt.
  * "Kimi K2 · KV cache" page: the cache excerpt (kv_seq_len bookkeeping, cache update,
    score shape check) and config.json (dimensions, rope_theta, rms_norm_eps).
  * "Kimi K2 · Key content up-projection" page: the k^C = c^KV W_UK equation, the
    Explanation (W_UK is output features 0-127 of each head's 256) and the `mla-prefill`
    excerpt (RoPE call, query/key assembly, scores, mask, fp32 softmax, value contraction).
  * "Kimi K2 · Latent attention (dense block, prefill)" page: the layer's in/out signature,
    the Parameters table, the "In numbers" cache sizes and the `mla-output` excerpt.

Readings where the pages are silent (each is listed in the design notes):
  * RoPE: the body of apply_rotary_pos_emb is not printed.  The rotary slice holds 32 pairs
    (layer signature on the dense-block page); pair j is elements (2j, 2j+1) ("adjacent",
    the default) and turns by pos * theta^(-2j/64).  The rotated pair is written back in
    place.  A "half" pairing (j, j+32) is kept behind the same switch.
  * Softmax scale: 1/sqrt(192) (nope 128 + rope 64); the value is not printed.
  * Mask: key s is visible from query t iff s <= L + t (L = cached length); masked keys get
    -inf, which is the same as leaving them out.
  * FP8 weights: W[o, i] = e4m3(q[o, i]) * s[o // 128, i // 128] (OCP e4m3 "fn": bias 7,
    no infinities, S.1111.111 is NaN); a partial last block shares its block's scale.
  * The cache is held as each position's normalised latent (512) and rotated rotary key
    (64).  Each position's content key and value are rebuilt from it with kv_b_proj exactly
    as the `mla-kv` excerpt builds them when the token is first seen, so the keys and values
    the scores see are the ones the pages' cache would return.

  * YaRN (optional, off by default): config.json on the "KV cache" page declares rope_scaling
    {type yarn, factor 32, original_max_position_embeddings 4096, beta_fast 1, beta_slow 1,
    mscale 1, mscale_all_dim 1} without the formulas.  They follow the published YaRN method
    (Peng et al., 2023, "NTK-by-parts" interpolation with an attention temperature), in the
    parametrisation those config keys name: pair j keeps its frequency while its wavelength
    turns more than beta_fast times over the original context, is divided by the factor
    while it turns fewer than beta_slow times, with a linear ramp between; the score scale
    is multiplied by m(factor, mscale_all_dim)^2 and cos/sin by m(factor, mscale) /
    m(factor, mscale_all_dim), m(s, mu) = 0.1 mu ln s + 1 for s > 1, else 1.

Parity is pinned by tests under tests/ (parameter counts, cache bytes, e4m3 table, RMSNorm and
RoPE closed forms, softmax sums, decode-equals-prefill, prefix consistency, brute-force loops on
tiny sizes, the absorbed form, YaRN's reductions to plain RoPE and its closed-form
boundaries).  Parity unpinned: the RoPE pairing choice itself (no page value decides between
adjacent and half pairing).
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np


# ---------------------------------------------------------------------------------------------
# Dimensions (config.json on the "KV cache" page)
# ---------------------------------------------------------------------------------------------
@dataclass(frozen=True)
class Dims:
    hidden: int = 7168        # hidden_size
    q_lora: int = 1536        # q_lora_rank
    kv_lora: int = 512        # kv_lora_rank
    heads: int = 64           # num_attention_heads
    nope: int = 128           # qk_nope_head_dim
    rope: int = 64            # qk_rope_head_dim (32 pairs)
    vdim: int = 128           # v_head_dim
    block: int = 128          # weight_block_size of the FP8 quantisation_config

    @property
    def q_head(self) -> int:
        return self.nope + self.rope


KIMI_K2 = Dims()
ROPE_THETA = 50000.0          # rope_theta
RMS_EPS = 1e-6                # rms_norm_eps
NUM_LAYERS = 61               # num_hidden_layers (used only by the cache-size figures)
BF16_BYTES = 2                # torch_dtype bfloat16

WEIGHT_NAMES = ("q_a", "q_b", "kv_a", "kv_b", "o")
NORM_NAMES = ("q_norm", "kv_norm")


def softmax_scale(d: Dims = KIMI_K2) -> float:
    """1/sqrt(q_head_dim); the pages use self.softmax_scale without printing it."""
    return 1.0 / math.sqrt(d.nope + d.rope)


def weight_shapes(d: Dims = KIMI_K2) -> dict:
    """[out, in] shapes of the five projections ("Key–value latent" page, `mla-init`; the
    [out, in] storage convention is stated on the "Key content up-projection" page)."""
    return {
        "q_a": (d.q_lora, d.hidden),
        "q_b": (d.heads * d.q_head, d.q_lora),
        "kv_a": (d.kv_lora + d.rope, d.hidden),
        "kv_b": (d.heads * (d.nope + d.vdim), d.kv_lora),
        "o": (d.hidden, d.heads * d.vdim),
    }


def norm_shapes(d: Dims = KIMI_K2) -> dict:
    return {"q_norm": d.q_lora, "kv_norm": d.kv_lora}


# ---------------------------------------------------------------------------------------------
# Weight slices named on the pages
# ---------------------------------------------------------------------------------------------
def split_kv_a(W_kva: np.ndarray, d: Dims = KIMI_K2):
    """Rows [0, kv_lora) give the latent, the last `rope` rows the shared rotary key
    (`mla-kv` excerpt: split into [kv_lora_rank, qk_rope_head_dim])."""
    return W_kva[: d.kv_lora], W_kva[d.kv_lora:]


def split_kv_b(W_kvb: np.ndarray, d: Dims = KIMI_K2):
    """W_UK, W_UV as [heads, nope, kv_lora] and [heads, vdim, kv_lora].

    Each head owns nope+vdim consecutive output rows; the first `nope` are the content key
    (W_UK is output features 0-127 of each head's 256, "Key content up-projection" page,
    Explanation) and the rest the value (`mla-kv` split into [nope, v_head_dim])."""
    per_head = W_kvb.reshape(d.heads, d.nope + d.vdim, d.kv_lora)
    return per_head[:, : d.nope, :], per_head[:, d.nope:, :]


def parameter_counts(d: Dims = KIMI_K2) -> dict:
    """Per-component parameters as grouped in the Parameters table of the dense-block
    attention page, derived from the weight shapes and the weight slices above."""
    ws = weight_shapes(d)
    ns = norm_shapes(d)
    n = lambda shape: shape[0] * shape[1]
    kva_rows, kva_cols = ws["kv_a"]
    latent_rows = split_kv_a(np.empty((kva_rows, 0)), d)[0].shape[0]
    rope_rows = kva_rows - latent_rows
    uk, uv = split_kv_b(np.empty((ws["kv_b"][0], d.kv_lora)), d)
    return {
        "query_compression": n(ws["q_a"]) + ns["q_norm"],
        "kv_compression": latent_rows * kva_cols + ns["kv_norm"],
        "query_heads": n(ws["q_b"]),
        "key_heads": uk.size + rope_rows * kva_cols,
        "value_heads": uv.size,
        "causal_attention": n(ws["o"]),
    }


def cache_values_per_position(d: Dims = KIMI_K2) -> dict:
    """Values one layer keeps per cached position: the pages' rebuilt cache (every head's
    192-wide key and 128-wide value, "KV cache" page) against the latent + rotary key."""
    return {
        "rebuilt": d.heads * d.q_head + d.heads * d.vdim,
        "latent": d.kv_lora + d.rope,
        "flash_padded": d.heads * (d.q_head + d.q_head),
    }


def cache_bytes_per_token_all_layers(d: Dims = KIMI_K2) -> dict:
    """bf16 bytes per token across all layers ("In numbers" on the dense-block page)."""
    v = cache_values_per_position(d)
    return {k: val * BF16_BYTES * NUM_LAYERS for k, val in v.items()}


# ---------------------------------------------------------------------------------------------
# Number formats
# ---------------------------------------------------------------------------------------------
def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    """Decode OCP FP8 e4m3 ("fn": 1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no
    infinities, exponent and mantissa all ones is NaN) to float64, value by value."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where((c >> 7) & 1, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    normal = (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0)
    subnormal = (m / 8.0) * 2.0 ** (1 - 7)
    mag = np.where(e == 0, subnormal, normal)
    mag = np.where((e == 15) & (c & 0x7 == 7), np.nan, mag)
    return sign * mag


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) to float64: the upper half of a float32."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def _expand_scales(s: np.ndarray, rows: int, cols: int, block: int) -> np.ndarray:
    return np.repeat(np.repeat(s, block, axis=0), block, axis=1)[:rows, :cols]


def dequant(q: np.ndarray, s: np.ndarray, d: Dims = KIMI_K2) -> np.ndarray:
    """W[o, i] = e4m3(q[o, i]) * s[o // 128, i // 128], exactly, in float64 (`linear`
    excerpt: fmt e4m3, weight_block_size [128, 128])."""
    rows, cols = q.shape
    return e4m3_to_f64(q) * _expand_scales(np.asarray(s, np.float64), rows, cols, d.block)


def dequant_fp32(q: np.ndarray, s: np.ndarray, d: Dims = KIMI_K2) -> np.ndarray:
    """The same product taken in float32 (one correctly rounded multiply), used to check a
    device-side dequantisation bit for bit."""
    rows, cols = q.shape
    qf = e4m3_to_f64(q).astype(np.float32)            # exact: every e4m3 value is a float32
    return qf * _expand_scales(np.asarray(s, np.float32), rows, cols, d.block)


# ---------------------------------------------------------------------------------------------
# Layer pieces
# ---------------------------------------------------------------------------------------------
def linear(x: np.ndarray, W: np.ndarray) -> np.ndarray:
    """nn.Linear without bias (attention_bias false): y = x W^T, W stored [out, in]."""
    return x @ W.T


def rms_norm(x: np.ndarray, g: np.ndarray, eps: float = RMS_EPS) -> np.ndarray:
    """DeepseekV3RMSNorm (`rmsnorm` excerpt): x * rsqrt(mean(x^2) + eps), times the gain."""
    var = np.mean(x * x, axis=-1, keepdims=True)
    return g * (x / np.sqrt(var + eps))


@dataclass(frozen=True)
class Yarn:
    """rope_scaling of config.json ("KV cache" page); the values are Kimi-K2's."""
    factor: float = 32.0
    original_max_positions: int = 4096
    beta_fast: float = 1.0
    beta_slow: float = 1.0
    mscale: float = 1.0
    mscale_all_dim: float = 1.0


def yarn_m(s: float, mu: float) -> float:
    """YaRN's attention-temperature factor: 0.1 mu ln s + 1 for s > 1, else 1."""
    return 0.1 * mu * np.log(s) + 1.0 if s > 1.0 else 1.0


def yarn_pair_of_rotations(r: float, rope_dim: int, theta: float, original: int) -> float:
    """The (fractional) pair index j whose wavelength 2 pi theta^(2j/rope_dim) fits r times
    into the original context: original * theta^(-2j/rope_dim) / (2 pi) = r."""
    return rope_dim * np.log(original / (2.0 * np.pi * r)) / (2.0 * np.log(theta))


def rope_inv_freq(rope_dim: int, theta: float = ROPE_THETA, yarn: Yarn | None = None):
    """Per-pair angular frequency: theta^(-2j/rope_dim); with YaRN, pairs below the
    fast-rotation boundary keep it, pairs above the slow-rotation boundary take it divided by
    the factor, and a linear ramp in j joins the two."""
    j = np.arange(rope_dim // 2, dtype=np.float64)
    base = theta ** (-2.0 * j / rope_dim)
    if yarn is None:
        return base
    lo = max(np.floor(yarn_pair_of_rotations(yarn.beta_fast, rope_dim, theta,
                                             yarn.original_max_positions)), 0.0)
    hi = min(np.ceil(yarn_pair_of_rotations(yarn.beta_slow, rope_dim, theta,
                                            yarn.original_max_positions)), rope_dim - 1.0)
    width = hi - lo if hi > lo else 1e-3          # one-pair ramp when the bounds meet
    ramp = np.clip((j - lo) / width, 0.0, 1.0)    # 0: keep the frequency, 1: interpolate
    return base * (1.0 - ramp) + (base / yarn.factor) * ramp


def rope_angles(positions: np.ndarray, rope_dim: int, theta: float = ROPE_THETA,
                yarn: Yarn | None = None) -> np.ndarray:
    """angle[p, j] = pos_p * inv_freq_j for the rope_dim/2 pairs (plain: theta^(-2j/rope_dim))."""
    inv_freq = rope_inv_freq(rope_dim, theta, yarn)
    return np.asarray(positions, np.float64)[:, None] * inv_freq[None, :]


def apply_rope(x: np.ndarray, positions: np.ndarray, theta: float = ROPE_THETA,
               pairing: str = "adjacent", yarn: Yarn | None = None) -> np.ndarray:
    """Rotate the rotary slice x[..., P, rope_dim] (P positions on axis -2) by its position.

    "adjacent": pair j = (x[2j], x[2j+1]); "half": pair j = (x[j], x[j + rope_dim/2]).
    Each pair (a, b) becomes (a cos - b sin, b cos + a sin), written back in place."""
    rope_dim = x.shape[-1]
    ang = rope_angles(positions, rope_dim, theta, yarn)
    mag = 1.0 if yarn is None else yarn_m(yarn.factor, yarn.mscale) / yarn_m(yarn.factor,
                                                                                 yarn.mscale_all_dim)
    c, s = mag * np.cos(ang), mag * np.sin(ang)
    out = np.array(x, dtype=np.float64, copy=True)
    if pairing == "adjacent":
        a, b = x[..., 0::2], x[..., 1::2]
        out[..., 0::2] = a * c - b * s
        out[..., 1::2] = b * c + a * s
    elif pairing == "half":
        h = rope_dim // 2
        a, b = x[..., :h], x[..., h:]
        out[..., :h] = a * c - b * s
        out[..., h:] = b * c + a * s
    else:
        raise ValueError(f"unknown pairing {pairing!r}")
    return out


def softmax(scores: np.ndarray, axis: int = -1) -> np.ndarray:
    """Softmax with the row maximum subtracted; -inf entries get weight exactly 0."""
    m = np.max(scores, axis=axis, keepdims=True)
    e = np.exp(scores - m)
    return e / np.sum(e, axis=axis, keepdims=True)


@dataclass
class Weights:
    """Dequantised float64 weights [out, in] and RMSNorm gains."""
    q_a: np.ndarray
    q_b: np.ndarray
    kv_a: np.ndarray
    kv_b: np.ndarray
    o: np.ndarray
    q_norm: np.ndarray
    kv_norm: np.ndarray


def weights_from_quantised(qw: dict, gains: dict, d: Dims = KIMI_K2) -> Weights:
    """qw[name] = (e4m3 codes uint8 [out, in], fp32 scales); gains[name] = bf16 bits."""
    deq = {n: dequant(qw[n][0], qw[n][1], d) for n in WEIGHT_NAMES}
    g = {n: bf16_to_f64(gains[n]) for n in NORM_NAMES}
    return Weights(**deq, **g)


def query(x: np.ndarray, W: Weights, d: Dims = KIMI_K2, eps: float = RMS_EPS):
    """q = q_b_proj(q_a_layernorm(q_a_proj(x))), viewed per head; returns (q_nope, q_pe)
    each [..., heads, nope] and [..., heads, rope] (per head [0:nope] | [nope:nope+rope])."""
    cq = linear(x, W.q_a)
    q = linear(rms_norm(cq, W.q_norm, eps), W.q_b)
    q = q.reshape(*q.shape[:-1], d.heads, d.q_head)
    return q[..., : d.nope], q[..., d.nope:]


def latent(x: np.ndarray, W: Weights, d: Dims = KIMI_K2, eps: float = RMS_EPS):
    """`mla-kv`: compressed_kv, k_pe = split(kv_a_proj_with_mqa(x)); the latent is normalised
    by kv_a_layernorm.  Returns (c_hat [..., kv_lora], k_pe [..., rope]) before RoPE."""
    ckv = linear(x, W.kv_a)
    c, k_pe = ckv[..., : d.kv_lora], ckv[..., d.kv_lora:]
    return rms_norm(c, W.kv_norm, eps), k_pe


def cache_rows(x: np.ndarray, positions: np.ndarray, W: Weights, d: Dims = KIMI_K2,
               eps: float = RMS_EPS, theta: float = ROPE_THETA, pairing: str = "adjacent",
               yarn: Yarn | None = None):
    """What one layer keeps for tokens x [P, hidden] at `positions`: the normalised latent and
    the rotated shared rotary key, concatenated to [P, kv_lora + rope]."""
    c_hat, k_pe = latent(x, W, d, eps)
    k_rot = apply_rope(k_pe, positions, theta, pairing, yarn)
    return np.concatenate([c_hat, k_rot], axis=-1)


def attend(q_nope: np.ndarray, q_pe_rot: np.ndarray, q_pos: np.ndarray, cache: np.ndarray,
           W: Weights, d: Dims = KIMI_K2, scale: float | None = None,
           key_chunk: int = 4096, query_chunk: int = 256, return_probs: bool = False):
    """Explicit attention of one sequence (`mla-prefill` excerpt).

    q_nope [T, heads, nope], q_pe_rot [T, heads, rope], q_pos [T] positions, cache [S, 576]
    (latent | rotated k_pe) for positions 0..S-1.  For every head the keys are
    [k_nope | k_pe] with k_nope = W_UK c_hat and the shared k_pe; values are v = W_UV c_hat.
    scores = q.k * scale, key s visible from query t iff s <= q_pos[t]; fp64 softmax over
    keys; o = sum_s p v.  Returns o [T, heads, vdim] (and the probabilities if asked)."""
    scale = softmax_scale(d) if scale is None else scale
    T, S = q_nope.shape[0], cache.shape[0]
    c_hat, k_rot = cache[:, : d.kv_lora], cache[:, d.kv_lora:]
    W_UK, W_UV = split_kv_b(W.kv_b, d)
    out = np.zeros((T, d.heads, d.vdim))
    probs = np.zeros((d.heads, T, S)) if return_probs else None
    for t0 in range(0, T, query_chunk):
        t1 = min(T, t0 + query_chunk)
        qn = np.transpose(q_nope[t0:t1], (1, 0, 2))          # [H, t, nope]
        qr = np.transpose(q_pe_rot[t0:t1], (1, 0, 2))        # [H, t, rope]
        s_end = min(S, int(np.max(q_pos[t0:t1])) + 1)        # keys past this are masked anyway
        scores = np.empty((d.heads, t1 - t0, s_end))
        for s0 in range(0, s_end, key_chunk):                # each score entry is independent
            s1 = min(s_end, s0 + key_chunk)
            # k_nope[h, n, s] = sum_c W_UK[h, n, c] c_hat[s, c]
            k_nope = (c_hat[s0:s1] @ W_UK.reshape(-1, d.kv_lora).T).T.reshape(
                d.heads, d.nope, s1 - s0)
            scores[:, :, s0:s1] = (np.matmul(qn, k_nope) + np.matmul(qr, k_rot[s0:s1].T)) * scale
        visible = np.arange(s_end)[None, :] <= np.asarray(q_pos[t0:t1])[:, None]   # [t, s]
        scores = np.where(visible[None], scores, -np.inf)
        p = softmax(scores, axis=-1)
        acc = np.zeros((d.heads, t1 - t0, d.vdim))
        for s0 in range(0, s_end, key_chunk):
            s1 = min(s_end, s0 + key_chunk)
            # v[h, s, j] = sum_c W_UV[h, j, c] c_hat[s, c]
            v = (c_hat[s0:s1] @ W_UV.reshape(-1, d.kv_lora).T).reshape(
                s1 - s0, d.heads, d.vdim).transpose(1, 0, 2)
            acc += np.matmul(p[:, :, s0:s1], v)
        out[t0:t1] = np.transpose(acc, (1, 0, 2))
        if return_probs:
            probs[:, t0:t1, :s_end] = p
    return (out, probs) if return_probs else out


def output(o: np.ndarray, W: Weights, d: Dims = KIMI_K2) -> np.ndarray:
    """`mla-output`: merge heads to [..., heads*vdim] and apply o_proj."""
    return linear(o.reshape(*o.shape[:-2], d.heads * d.vdim), W.o)


def forward(x: np.ndarray, cache: np.ndarray | None, W: Weights, d: Dims = KIMI_K2,
            eps: float = RMS_EPS, theta: float = ROPE_THETA, pairing: str = "adjacent",
            scale: float | None = None, return_probs: bool = False, yarn: Yarn | None = None):
    """One layer over T new tokens x [T, hidden] of one sequence whose cache holds
    L = len(cache) positions (None or empty for prefill over an empty cache).

    The new tokens sit at positions L..L+T-1 (kv_seq_len = T + cached length, "KV cache"
    page).  Returns (y [T, hidden], the cache grown to L+T rows[, probabilities])."""
    x = np.asarray(x, np.float64)
    L = 0 if cache is None else cache.shape[0]
    pos = np.arange(L, L + x.shape[0])
    q_nope, q_pe = query(x, W, d, eps)
    q_pe_rot = apply_rope(np.transpose(q_pe, (1, 0, 2)), pos, theta, pairing, yarn)
    q_pe_rot = np.transpose(q_pe_rot, (1, 0, 2))
    new_rows = cache_rows(x, pos, W, d, eps, theta, pairing, yarn)
    if scale is None and yarn is not None:  # YaRN's temperature on the scores
        scale = softmax_scale(d) * yarn_m(yarn.factor, yarn.mscale_all_dim) ** 2
    full = new_rows if L == 0 else np.concatenate([cache, new_rows], axis=0)
    res = attend(q_nope, q_pe_rot, pos, full, W, d, scale, return_probs=return_probs)
    o, probs = res if return_probs else (res, None)
    y = output(o, W, d)
    return (y, full, probs) if return_probs else (y, full)


def block_forward(x: np.ndarray, cache: np.ndarray | None, W: Weights, g_in: np.ndarray,
                  eps: float = RMS_EPS, **kw):
    """The attention half of a decoder block ("Attention input" page, `block` excerpt): the
    input is kept as the residual, normalised by input_layernorm (the `rmsnorm` excerpt with
    the block's own gain over the hidden size), passed through the layer, and the layer's
    output is added back to the residual.  (The post-attention norm and the FFN that follow
    in the block are not part of it.)  Returns (y [T, hidden], the grown cache)."""
    x = np.asarray(x, np.float64)
    h = rms_norm(x, g_in, eps)
    y, full = forward(h, cache, W, eps=eps, **kw)[:2]
    return x + y, full


def prefill(x: np.ndarray, W: Weights, **kw):
    """Prefill over an empty cache: x [T, hidden] -> (y [T, hidden], cache [T, 576])."""
    return forward(x, None, W, **kw)


def decode(x: np.ndarray, cache: np.ndarray, W: Weights, **kw):
    """Decode one token x [hidden] at position len(cache) -> (y [hidden], cache [L+1, 576])."""
    y, full = forward(np.asarray(x)[None, :], cache, W, **kw)[:2]
    return y[0], full
