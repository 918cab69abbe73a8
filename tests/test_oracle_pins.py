"""Pins of the fp64 oracle against what the pages and the mathematics fix (no GPU).

Each test checks the oracle against something other than itself: numbers printed on the
pages (tests/golden/page_numbers.json), closed forms, invariants, library routines, or a
brute-force loop written separately from the pages' equations.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import mla_oracle as O

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_numbers.json")))
G = {k: v["value"] for k, v in GOLDEN.items() if not k.startswith("_")}

TINY = O.Dims(hidden=24, q_lora=12, kv_lora=8, heads=3, nope=4, rope=6, vdim=5, block=8)


def tiny_weights(seed=0, d=TINY):
    rng = np.random.default_rng(seed)
    ws = {n: rng.normal(0, 0.3, s) for n, s in O.weight_shapes(d).items()}
    gs = {n: 1 + rng.uniform(-0.1, 0.1, s) for n, s in O.norm_shapes(d).items()}
    return O.Weights(**ws, **gs)


# ----------------------------------------------------------------------------- page numbers
def test_parameter_counts_match_page_table():
    c = O.parameter_counts()
    for k in ("query_compression", "kv_compression", "query_heads", "key_heads",
              "value_heads", "causal_attention"):
        assert c[k] == G[k], k
    assert sum(c.values()) == G["parameters_per_layer"]


def test_w_uk_slice_matches_page():
    W_kvb = np.zeros(O.weight_shapes()["kv_b"])
    uk, uv = O.split_kv_b(W_kvb)
    assert uk.size == G["w_uk_parameters"] and uv.size == G["value_heads"]
    assert uk.size * 60 == G["w_uk_parameters_60_blocks"]
    assert [uk.shape[2], uk.shape[0] * uk.shape[1]] == G["w_uk_shape_in_out"]
    # W_UK of head h is output rows 256h .. 256h+127 of kv_b_proj.
    marker = np.arange(W_kvb.shape[0], dtype=np.float64)[:, None] * np.ones((1, 512))
    uk, uv = O.split_kv_b(marker)
    assert uk[5, 0, 0] == 5 * 256 and uk[5, 127, 0] == 5 * 256 + 127
    assert uv[5, 0, 0] == 5 * 256 + 128 and uv[63, 127, 0] == 64 * 256 - 1


def test_cache_sizes_match_page():
    v = O.cache_values_per_position()
    assert v["rebuilt"] == G["rebuilt_values_per_position"]
    assert v["latent"] == G["latent_values_per_position"]
    b = O.cache_bytes_per_token_all_layers()
    assert b["rebuilt"] == G["cache_bytes_per_token_rebuilt_61_layers"]
    assert b["latent"] == G["cache_bytes_per_token_latent_61_layers"]
    assert b["flash_padded"] == G["cache_bytes_per_token_flash_padded_61_layers"]
    assert round(b["rebuilt"] / b["latent"]) == 36
    assert O.KIMI_K2.rope // 2 == G["rope_pairs"]


# ----------------------------------------------------------------------------- number formats
def test_e4m3_table_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = O.e4m3_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float32).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9 and ours[0x08] == 2.0 ** -6


def test_bf16_decode_matches_torch():
    rng = np.random.default_rng(1)
    x = torch.from_numpy(rng.normal(0, 3, 1000).astype(np.float32)).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.bf16_to_f64(bits), x.double().numpy())


def test_dequant_blocks_brute_force():
    rng = np.random.default_rng(2)
    rows, cols, blk = 20, 27, 8           # partial last blocks on both axes
    q = rng.integers(0, 256, (rows, cols), dtype=np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x3C          # avoid NaN codes
    s = rng.uniform(1e-4, 2.0, (-(-rows // blk), -(-cols // blk))).astype(np.float32)
    d = O.Dims(block=blk)
    W = O.dequant(q, s, d)
    W32 = O.dequant_fp32(q, s, d)
    table = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).float()
    for o in range(rows):
        for i in range(cols):
            v = float(table[int(q[o, i])])
            assert W[o, i] == v * float(s[o // blk, i // blk])
            assert W32[o, i] == np.float32(np.float32(v) * s[o // blk, i // blk])


# ----------------------------------------------------------------------------- RMSNorm, RoPE
def test_rms_norm_constant_vector():
    for c in (0.0, 1e-4, 0.5, 3.0, -7.0):
        x = np.full(512, c)
        g = np.linspace(0.9, 1.1, 512)
        np.testing.assert_allclose(O.rms_norm(x, g, 1e-6), g * c / math.sqrt(c * c + 1e-6),
                                   rtol=1e-14, atol=0)


def test_rms_norm_loop():
    rng = np.random.default_rng(3)
    x, g = rng.normal(size=37), rng.normal(size=37)
    ms = sum(float(v) * float(v) for v in x) / len(x)
    ref = [float(g[i]) * float(x[i]) / math.sqrt(ms + 1e-6) for i in range(len(x))]
    np.testing.assert_allclose(O.rms_norm(x, g), ref, rtol=1e-13)


def test_rope_position_zero_is_identity():
    x = np.random.default_rng(4).normal(size=(5, 64))
    for pairing in ("adjacent", "half"):
        np.testing.assert_array_equal(O.apply_rope(x, np.zeros(5), pairing=pairing), x)


def test_rope_preserves_pair_norms_and_angles():
    rng = np.random.default_rng(5)
    x = rng.normal(size=(7, 64))
    pos = np.array([1, 2, 17, 999, 1000, 4095, 131072])
    y = O.apply_rope(x, pos)
    for t in range(7):
        for j in range(32):
            a, b = x[t, 2 * j], x[t, 2 * j + 1]
            ang = pos[t] * 50000.0 ** (-2.0 * j / 64)
            ca, sa = math.cos(ang), math.sin(ang)
            assert abs(y[t, 2 * j] - (a * ca - b * sa)) < 1e-12
            assert abs(y[t, 2 * j + 1] - (a * sa + b * ca)) < 1e-12
            assert abs(math.hypot(y[t, 2 * j], y[t, 2 * j + 1]) - math.hypot(a, b)) < 1e-12
    # pair 0 turns by exactly `pos` radians
    e = np.zeros((1, 64)); e[0, 0] = 1.0
    r = O.apply_rope(e, np.array([3]))
    assert abs(r[0, 0] - math.cos(3)) < 1e-15 and abs(r[0, 1] - math.sin(3)) < 1e-15


def half_pairs_turn_by_exact_angles(rope) -> bool:
    """Whether `rope` (the oracle's apply_rope signature) turns pair j = (x[j], x[j+32]) of a
    64-wide slice by +pos * theta^(-2j/64) for the "half" pairing, element by element, with
    every pair's norm kept.  Written out from the rotation itself, one scalar at a time."""
    rng = np.random.default_rng(28)
    x = rng.normal(size=(6, 64))
    pos = np.array([1, 3, 17, 1000, 4095, 131072])
    y = rope(x, pos, pairing="half")
    for t in range(6):
        for j in range(32):
            a, b = x[t, j], x[t, j + 32]
            ang = pos[t] * 50000.0 ** (-2.0 * j / 64)
            ca, sa = math.cos(ang), math.sin(ang)
            if abs(y[t, j] - (a * ca - b * sa)) > 1e-12:
                return False
            if abs(y[t, j + 32] - (a * sa + b * ca)) > 1e-12:
                return False
    return True


def test_rope_half_pairs_turn_by_exact_angles():
    """The half pairing (j, j+32), element by element: a unit vector in element j turns into
    (cos, sin) at elements (j, j+32) by pos * theta^(-2j/64), in the positive direction."""
    assert half_pairs_turn_by_exact_angles(O.apply_rope)
    for j in (0, 1, 13, 31):
        e = np.zeros((1, 64)); e[0, j] = 1.0
        r = O.apply_rope(e, np.array([5]), pairing="half")
        ang = 5 * 50000.0 ** (-2.0 * j / 64)
        expect = np.zeros(64); expect[j] = math.cos(ang); expect[j + 32] = math.sin(ang)
        np.testing.assert_allclose(r[0], expect, rtol=0, atol=1e-15)


def _rope_half_planted(kind):
    """The oracle's apply_rope with one plausible slip planted in its half branch only."""
    orig = O.apply_rope
    def rope(x, positions, theta=O.ROPE_THETA, pairing="adjacent", yarn=None):
        if pairing != "half":
            return orig(x, positions, theta, pairing, yarn)
        if kind == "sign":                     # rotation in the negative direction
            return orig(x, -np.asarray(positions), theta, pairing, yarn)
        if kind == "freq_order":               # pair j given pair 31-j's frequency
            h = x.shape[-1] // 2
            perm = np.concatenate([np.arange(h)[::-1], h + np.arange(h)[::-1]])  # an involution
            return orig(x[..., perm], positions, theta, pairing, yarn)[..., perm]
        if kind == "adjacent_inside":          # the half switch silently ignored
            return orig(x, positions, theta, "adjacent", yarn)
        raise ValueError(kind)
    return rope


@pytest.mark.parametrize("kind", ["sign", "freq_order", "adjacent_inside"])
def test_planted_half_rope_mistakes_are_caught(kind):
    """Each slip planted in the half branch (on the CPU) fails the element-by-element pin."""
    assert not half_pairs_turn_by_exact_angles(_rope_half_planted(kind))


@pytest.mark.parametrize("pairing", ["adjacent", "half"])
def test_rope_dot_depends_on_offset_only(pairing):
    rng = np.random.default_rng(6)
    q, k = rng.normal(size=64), rng.normal(size=64)
    def dot(m, n):
        return float(O.apply_rope(q[None], np.array([m]), pairing=pairing)[0]
                     @ O.apply_rope(k[None], np.array([n]), pairing=pairing)[0])
    for m, n, shift in ((5, 2, 100), (1000, 0, 7), (40, 40, 12345)):
        assert abs(dot(m, n) - dot(m + shift, n + shift)) < 1e-9


# ----------------------------------------------------------------------------- attention
def test_yarn_reduces_to_plain_rope():
    """YaRN with factor 1, or with an original context so long that every pair turns more than
    beta_fast times over it, leaves every frequency (and cos/sin magnitude) unchanged."""
    base = O.rope_inv_freq(64, 50000.0)
    np.testing.assert_array_equal(O.rope_inv_freq(64, 50000.0, O.Yarn(factor=1.0)), base)
    np.testing.assert_allclose(O.rope_inv_freq(64, 50000.0, O.Yarn(original_max_positions=10**15)),
                               base, rtol=0, atol=0)
    x = np.random.default_rng(3).normal(size=(5, 64))
    np.testing.assert_array_equal(O.apply_rope(x, np.arange(5), yarn=O.Yarn(factor=1.0)),
                                  O.apply_rope(x, np.arange(5)))


def test_yarn_boundary_for_kimi_config():
    """Kimi-K2's rope_scaling (factor 32, original 4096, beta_fast = beta_slow = 1): a pair keeps
    its frequency iff its wavelength turns at least once more over the original 4096 positions,
    counted directly as 4096 theta^(-2j/64) / (2 pi); the others run 32 times slower.  The
    temperature is m = 1 + 0.1 ln 32 and the score scale (1/sqrt 192) m^2."""
    j = np.arange(32)
    turns = 4096 * 50000.0 ** (-2.0 * j / 64) / (2 * np.pi)
    keep = turns > 1.0
    assert keep[:20].all() and not keep[20:].any()          # the boundary falls between 19 and 20
    base = 50000.0 ** (-2.0 * j / 64)
    f = O.rope_inv_freq(64, 50000.0, O.Yarn())
    np.testing.assert_array_equal(f[keep], base[keep])
    np.testing.assert_allclose(f[~keep], base[~keep] / 32.0, rtol=1e-15)
    assert abs(O.yarn_m(32.0, 1.0) - (1.0 + 0.1 * np.log(32.0))) < 1e-15
    d, W = TINY, tiny_weights(25)
    x = np.random.default_rng(26).normal(size=(6, d.hidden))
    yy = O.Yarn(factor=4.0, original_max_positions=8)
    y_default, _ = O.prefill(x, W, d=d, yarn=yy)
    y_explicit, _ = O.prefill(x, W, d=d, yarn=yy,
                              scale=O.softmax_scale(d) * (1 + 0.1 * np.log(4.0)) ** 2)
    np.testing.assert_allclose(y_default, y_explicit, rtol=1e-13, atol=1e-15)
    y_plain_scale, _ = O.prefill(x, W, d=d, yarn=yy, scale=O.softmax_scale(d))
    assert np.max(np.abs(y_default - y_plain_scale)) > 1e-6   # the temperature matters


def test_yarn_dot_depends_on_offset_only():
    rng = np.random.default_rng(27)
    q, k = rng.normal(size=64), rng.normal(size=64)
    yy = O.Yarn()
    def dot(m, n):
        return float(O.apply_rope(q[None], np.array([m]), yarn=yy)[0]
                     @ O.apply_rope(k[None], np.array([n]), yarn=yy)[0])
    assert abs(dot(10, 3) - dot(1007, 1000)) < 1e-9
    assert abs(dot(5000, 5000) - dot(0, 0)) < 1e-9


def test_softmax_rows_sum_to_one_and_mask_is_exact():
    d, W = TINY, tiny_weights(7)
    x = np.random.default_rng(8).normal(size=(9, d.hidden))
    y, cache, p = O.prefill(x, W, d=d, return_probs=True)
    np.testing.assert_allclose(p.sum(-1), 1.0, rtol=0, atol=1e-12)
    T = x.shape[0]
    future = np.triu(np.ones((T, T), bool), 1)
    assert np.all(p[:, future] == 0.0)
    assert np.all(p[:, ~future] > 0.0)


def test_single_token_is_value_of_itself():
    """T=1 over an empty cache: softmax over one key is 1, so y = concat_h(v_h(0)) W_o^T."""
    d, W = TINY, tiny_weights(9)
    x = np.random.default_rng(10).normal(size=(1, d.hidden))
    y, cache = O.prefill(x, W, d=d)
    c_hat = cache[0, : d.kv_lora]
    _, W_UV = O.split_kv_b(W.kv_b, d)
    v = np.stack([W_UV[h] @ c_hat for h in range(d.heads)])
    np.testing.assert_allclose(y[0], W.o @ v.reshape(-1), rtol=1e-12, atol=1e-14)


def test_decode_equals_last_prefill_row():
    d, W = TINY, tiny_weights(11)
    x = np.random.default_rng(12).normal(size=(13, d.hidden))
    y_full, cache_full = O.prefill(x, W, d=d)
    _, cache = O.prefill(x[:-1], W, d=d)
    y_dec, cache2 = O.decode(x[-1], cache, W, d=d)
    np.testing.assert_allclose(y_dec, y_full[-1], rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(cache2, cache_full, rtol=1e-12, atol=1e-14)


def test_prefill_in_chunks_equals_one_prefill():
    """Prefill of a prompt in chunks against the growing cache (each chunk at positions
    L..L+T-1 sees keys 0..L+t) equals one causal prefill of the whole prompt, row for row."""
    d, W = TINY, tiny_weights(23)
    x = np.random.default_rng(24).normal(size=(17, d.hidden))
    y_full, cache_full = O.prefill(x, W, d=d)
    cache, ys = None, []
    for a, b in ((0, 5), (5, 6), (6, 13), (13, 17)):
        y, cache = O.forward(x[a:b], cache, W, d=d)
        ys.append(y)
    np.testing.assert_allclose(np.concatenate(ys), y_full, rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(cache, cache_full, rtol=1e-12, atol=1e-14)


def test_prefix_consistency():
    d, W = TINY, tiny_weights(13)
    x = np.random.default_rng(14).normal(size=(10, d.hidden))
    y10, _ = O.prefill(x, W, d=d)
    y6, _ = O.prefill(x[:6], W, d=d)
    np.testing.assert_allclose(y10[:6], y6, rtol=1e-11, atol=1e-14)
    x2 = x.copy(); x2[7:] += 1.0
    y10b, _ = O.prefill(x2, W, d=d)
    np.testing.assert_allclose(y10b[:7], y10[:7], rtol=1e-11, atol=1e-14)


def test_chunked_evaluation_is_the_same_sum():
    d, W = TINY, tiny_weights(15)
    x = np.random.default_rng(16).normal(size=(11, d.hidden))
    y, cache = O.prefill(x, W, d=d)
    q_nope, q_pe = O.query(x, W, d)
    q_rot = np.transpose(O.apply_rope(np.transpose(q_pe, (1, 0, 2)), np.arange(11)), (1, 0, 2))
    o = O.attend(q_nope, q_rot, np.arange(11), cache, W, d, key_chunk=3, query_chunk=2)
    np.testing.assert_allclose(O.output(o, W, d), y, rtol=1e-12, atol=1e-14)


def brute_force_layer(x, W, d, L_cache_x=None, theta=50000.0, eps=1e-6, pairing="adjacent"):
    """The whole layer as plain Python loops over floats, written from the pages' equations:
    q_a -> RMSNorm -> q_b (per head nope|rope); kv_a -> split latent|k_pe -> RMSNorm latent;
    RoPE on adjacent pairs (2j, 2j+1), or with pairing="half" on (j, j + rope/2); k_nope, v
    from kv_b rows (per head: nope rows then v rows); causal scores scaled by
    1/sqrt(nope+rope); softmax; value mix; o_proj."""
    xs = [list(map(float, r)) for r in x]
    def mv(Wm, v):
        return [sum(float(Wm[i][k]) * v[k] for k in range(len(v))) for i in range(len(Wm))]
    def norm(v, g):
        ms = sum(a * a for a in v) / len(v)
        return [float(g[i]) * v[i] / math.sqrt(ms + eps) for i in range(len(v))]
    def rope(v, pos):
        out = list(v)
        for j in range(len(v) // 2):
            ang = pos * theta ** (-2.0 * j / len(v))
            i0, i1 = (2 * j, 2 * j + 1) if pairing == "adjacent" else (j, j + len(v) // 2)
            a, b = v[i0], v[i1]
            out[i0] = a * math.cos(ang) - b * math.sin(ang)
            out[i1] = b * math.cos(ang) + a * math.sin(ang)
        return out
    hd = d.nope + d.vdim
    c_hat, k_rot, qn, qr = [], [], [], []
    for t, xt in enumerate(xs):
        ckv = mv(W.kv_a, xt)
        c_hat.append(norm(ckv[: d.kv_lora], W.kv_norm))
        k_rot.append(rope(ckv[d.kv_lora:], t))
        q = mv(W.q_b, norm(mv(W.q_a, xt), W.q_norm))
        qn.append([q[h * (d.nope + d.rope): h * (d.nope + d.rope) + d.nope] for h in range(d.heads)])
        qr.append([rope(q[h * (d.nope + d.rope) + d.nope: (h + 1) * (d.nope + d.rope)], t)
                   for h in range(d.heads)])
    scale = 1.0 / math.sqrt(d.nope + d.rope)
    ys = []
    for t in range(len(xs)):
        merged = []
        for h in range(d.heads):
            scores = []
            for s in range(t + 1):
                kn = [sum(float(W.kv_b[h * hd + n][c]) * c_hat[s][c] for c in range(d.kv_lora))
                      for n in range(d.nope)]
                sc = sum(qn[t][h][n] * kn[n] for n in range(d.nope))
                sc += sum(qr[t][h][r] * k_rot[s][r] for r in range(d.rope))
                scores.append(sc * scale)
            m = max(scores)
            e = [math.exp(v - m) for v in scores]
            z = sum(e)
            o = [0.0] * d.vdim
            for s in range(t + 1):
                for j in range(d.vdim):
                    v = sum(float(W.kv_b[h * hd + d.nope + j][c]) * c_hat[s][c]
                            for c in range(d.kv_lora))
                    o[j] += e[s] / z * v
            merged.extend(o)
        ys.append(mv(W.o, merged))
    return np.array(ys)


def test_forward_equals_brute_force_loops():
    d, W = TINY, tiny_weights(17)
    x = np.random.default_rng(18).normal(size=(6, d.hidden))
    y, _ = O.prefill(x, W, d=d)
    np.testing.assert_allclose(y, brute_force_layer(x, W, d), rtol=1e-10, atol=1e-13)


def test_forward_half_pairing_equals_brute_force_loops():
    d, W = TINY, tiny_weights(29)
    x = np.random.default_rng(30).normal(size=(6, d.hidden))
    y, _ = O.prefill(x, W, d=d, pairing="half")
    np.testing.assert_allclose(y, brute_force_layer(x, W, d, pairing="half"), rtol=1e-10,
                               atol=1e-13)
    # the two pairings are different layers: the pin tells them apart
    y_adj, _ = O.prefill(x, W, d=d)
    assert not np.allclose(y, y_adj, rtol=1e-6, atol=1e-9)


@pytest.mark.parametrize("kind", ["sign", "freq_order"])
def test_planted_half_rope_mistakes_fail_the_layer_loop(monkeypatch, kind):
    d, W = TINY, tiny_weights(31)
    x = np.random.default_rng(32).normal(size=(5, d.hidden))
    ref = brute_force_layer(x, W, d, pairing="half")
    monkeypatch.setattr(O, "apply_rope", _rope_half_planted(kind))
    y, _ = O.prefill(x, W, d=d, pairing="half")
    assert not np.allclose(y, ref, rtol=1e-6, atol=1e-9)


def absorbed_decode(x_new, cache, W, d):
    """Absorbed form written independently: q~_h = W_UK,h^T q_nope,h scored against the
    latent, o_lat = sum p c_hat, o_h = W_UV,h o_lat."""
    L = cache.shape[0]
    cq = W.q_a @ x_new
    cq = W.q_norm * cq / np.sqrt(np.mean(cq ** 2) + 1e-6)
    q = (W.q_b @ cq).reshape(d.heads, d.nope + d.rope)
    ckv = W.kv_a @ x_new
    c_new = W.kv_norm * ckv[: d.kv_lora] / np.sqrt(np.mean(ckv[: d.kv_lora] ** 2) + 1e-6)
    k_new = O.apply_rope(ckv[None, d.kv_lora:], np.array([L]))[0]
    lat = np.vstack([cache, np.concatenate([c_new, k_new])[None]])
    kvb = W.kv_b.reshape(d.heads, d.nope + d.vdim, d.kv_lora)
    out = []
    for h in range(d.heads):
        q_abs = kvb[h, : d.nope].T @ q[h, : d.nope]
        q_rot = O.apply_rope(q[h, d.nope:][None], np.array([L]))[0]
        s = (lat[:, : d.kv_lora] @ q_abs + lat[:, d.kv_lora:] @ q_rot) / math.sqrt(d.nope + d.rope)
        p = np.exp(s - s.max()); p /= p.sum()
        out.append(kvb[h, d.nope:] @ (p @ lat[:, : d.kv_lora]))
    return W.o @ np.concatenate(out)


def test_absorbed_equals_explicit_tiny():
    d, W = TINY, tiny_weights(19)
    x = np.random.default_rng(20).normal(size=(8, d.hidden))
    _, cache = O.prefill(x[:-1], W, d=d)
    y_exp, _ = O.decode(x[-1], cache, W, d=d)
    np.testing.assert_allclose(absorbed_decode(x[-1], cache, W, d), y_exp, rtol=1e-11, atol=1e-14)


def test_absorbed_equals_explicit_full_dims_short():
    d = O.KIMI_K2
    rng = np.random.default_rng(21)
    ws = {n: rng.normal(0, 0.02, s) for n, s in O.weight_shapes(d).items()}
    gs = {n: 1 + rng.uniform(-0.1, 0.1, s) for n, s in O.norm_shapes(d).items()}
    W = O.Weights(**ws, **gs)
    x = rng.normal(size=(5, d.hidden))
    _, cache = O.prefill(x[:-1], W, d=d)
    y_exp, _ = O.decode(x[-1], cache, W, d=d)
    np.testing.assert_allclose(absorbed_decode(x[-1], cache, W, d), y_exp, rtol=1e-10, atol=1e-14)


# ----------------------------------------------------------------------------- planted mistakes
@pytest.mark.parametrize("mistake", ["swap_kvb_halves", "rope_sign", "no_scale", "mask_off_by_one"])
def test_planted_mistakes_are_caught(monkeypatch, mistake):
    """Each plausible oracle mistake, planted on the CPU, must fail the brute-force pin."""
    d, W = TINY, tiny_weights(22)
    x = np.random.default_rng(23).normal(size=(5, d.hidden))
    ref = brute_force_layer(x, W, d)
    if mistake == "swap_kvb_halves":
        monkeypatch.setattr(O, "split_kv_b", lambda Wk, dd=O.KIMI_K2: _swapped(Wk, dd))
    elif mistake == "rope_sign":
        orig_rope = O.apply_rope
        monkeypatch.setattr(O, "apply_rope",
                            lambda v, p, th=O.ROPE_THETA, pairing="adjacent", yarn=None:
                            orig_rope(v, -np.asarray(p), th, pairing, yarn))
    elif mistake == "no_scale":
        monkeypatch.setattr(O, "softmax_scale", lambda dd=O.KIMI_K2: 1.0)
    elif mistake == "mask_off_by_one":
        orig_attend = O.attend
        def shifted(qn, qr, qp, c, Ww, dd=O.KIMI_K2, *a, **kw):
            qp = np.asarray(qp)
            return orig_attend(qn, qr, qp - 1 + (qp == 0), c, Ww, dd, *a, **kw)
        monkeypatch.setattr(O, "attend", shifted)
    y, _ = O.prefill(x, W, d=d)
    assert not np.allclose(y, ref, rtol=1e-6, atol=1e-9)


def _swapped(W_kvb, d):
    per_head = W_kvb.reshape(d.heads, d.nope + d.vdim, d.kv_lora)
    return per_head[:, d.vdim:, :][:, : d.nope], per_head[:, : d.vdim, :]


# ----------------------------------------------------------------------------- decoder block
def brute_force_block(x, W, d, g_in, eps=1e-6):
    """The attention half of the block as loops: each token normalised by the input gain
    (float arithmetic, one token at a time), the brute-force layer on the normalised tokens,
    and the token itself added back."""
    xs = np.asarray(x, np.float64)
    hs = []
    for row in xs:
        ms = sum(float(v) * float(v) for v in row) / len(row)
        hs.append([float(g_in[i]) * float(row[i]) / math.sqrt(ms + eps) for i in range(len(row))])
    y = brute_force_layer(np.array(hs), W, d, eps=eps)
    return np.array([[float(xs[t][i]) + float(y[t][i]) for i in range(len(xs[t]))]
                     for t in range(len(xs))])


def tiny_input_gain(seed, d=TINY):
    return 1 + np.random.default_rng(seed).uniform(-0.1, 0.1, d.hidden)


def test_block_equals_brute_force_loops():
    d, W = TINY, tiny_weights(33)
    g = tiny_input_gain(34)
    x = np.random.default_rng(35).normal(size=(6, d.hidden)) * 3.0
    y, _ = O.block_forward(x, None, W, g, d=d)
    np.testing.assert_allclose(y, brute_force_block(x, W, d, g), rtol=1e-10, atol=1e-12)


def test_block_with_zero_output_projection_is_the_identity():
    d, W = TINY, tiny_weights(36)
    W = O.Weights(**{**W.__dict__, "o": np.zeros_like(W.o)})
    x = np.random.default_rng(37).normal(size=(5, d.hidden))
    y, _ = O.block_forward(x, None, W, tiny_input_gain(38), d=d)
    np.testing.assert_array_equal(y, x)


def test_block_attention_part_is_scale_invariant_without_eps():
    """With eps = 0 the input norm removes any positive scale of the input, so the block's
    addition to the residual, y - x, is the same for x and 7.5 x."""
    d, W = TINY, tiny_weights(39)
    g = tiny_input_gain(40)
    x = np.random.default_rng(41).normal(size=(5, d.hidden))
    y1, _ = O.block_forward(x, None, W, g, d=d, eps=0.0)
    y2, _ = O.block_forward(7.5 * x, None, W, g, d=d, eps=0.0)
    np.testing.assert_allclose(y2 - 7.5 * x, y1 - x, rtol=1e-9, atol=1e-12)


def test_block_decode_equals_last_block_prefill_row():
    d, W = TINY, tiny_weights(42)
    g = tiny_input_gain(43)
    x = np.random.default_rng(44).normal(size=(9, d.hidden))
    y_full, _ = O.block_forward(x, None, W, g, d=d)
    _, cache = O.block_forward(x[:-1], None, W, g, d=d)
    y_dec, _ = O.block_forward(x[-1:], cache, W, g, d=d)
    np.testing.assert_allclose(y_dec[0], y_full[-1], rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("mistake", ["no_residual", "norm_after", "no_gain"])
def test_planted_block_mistakes_are_caught(monkeypatch, mistake):
    d, W = TINY, tiny_weights(45)
    g = tiny_input_gain(46)
    x = np.random.default_rng(47).normal(size=(4, d.hidden)) * 2.0
    ref = brute_force_block(x, W, d, g)
    orig_forward, orig_norm = O.forward, O.rms_norm
    if mistake == "no_residual":
        monkeypatch.setattr(O, "block_forward", lambda xx, c, Ww, gg, eps=1e-6, **kw:
                            (orig_forward(O.rms_norm(xx, gg, eps), c, Ww, eps=eps, **kw)[0], None))
    elif mistake == "norm_after":
        monkeypatch.setattr(O, "block_forward", lambda xx, c, Ww, gg, eps=1e-6, **kw:
                            (O.rms_norm(xx + orig_forward(xx, c, Ww, eps=eps, **kw)[0], gg, eps),
                             None))
    elif mistake == "no_gain":
        calls = {"n": 0}
        def norm(v, gg, eps=1e-6):
            calls["n"] += 1
            return orig_norm(v, np.ones_like(gg) if calls["n"] == 1 else gg, eps)
        monkeypatch.setattr(O, "rms_norm", norm)
    y, _ = O.block_forward(x, None, W, g, d=d)
    assert not np.allclose(y, ref, rtol=1e-6, atol=1e-9)
