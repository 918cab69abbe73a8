"""The seeded input generators: determinism, slicing and the quantisation recipe (no GPU)."""
import numpy as np

from head_latent_attention_mla_gb300 import synth
from oracle import mla_oracle as O


def test_hidden_states_slices_agree():
    a = synth.hidden_states(0, 3, 4090, 12, hidden=64)
    b = synth.hidden_states(0, 3, 4094, 4, hidden=64)
    assert np.array_equal(a[4:8], b)
    assert not np.array_equal(synth.hidden_states(0, 2, 0, 4, 64), synth.hidden_states(0, 3, 0, 4, 64))


def test_quantisation_recipe():
    rng = np.random.default_rng(0)
    w = (rng.standard_normal((200, 300)) * 0.02).astype(np.float32)
    w[128:, 256:] = 0.0                                   # an all-zero partial block
    q, s = synth.quantise_e4m3_blocks(w)
    assert q.shape == w.shape and s.shape == (2, 3) and s.dtype == np.float32
    assert s[1, 2] == 1.0 and np.all(q[128:, 256:] == 0)
    amax = np.abs(w[:128, :128]).max()
    assert s[0, 0] == np.float32(amax) / np.float32(448.0)
    deq = O.dequant(q, s)
    # e4m3 keeps 3 mantissa bits: relative error at most 2^-4 for normal codes
    big = np.abs(w) > 2.0 ** -6 * s.repeat(128, 0).repeat(128, 1)[:200, :300]
    assert np.all(np.abs(deq - w)[big] <= np.abs(w[big]) * 2.0 ** -4 + 1e-12)
    assert np.max(np.abs(O.e4m3_to_f64(q[:128, :128]))) == 448.0


def test_weights_and_gains_are_seeded():
    shapes = {"q_a": (130, 256), "q_b": (64, 130), "kv_a": (72, 256), "kv_b": (64, 40), "o": (256, 64)}
    a = synth.make_weights(5, shapes)
    b = synth.make_weights(5, shapes)
    for n in a:
        assert np.array_equal(a[n][0], b[n][0]) and np.array_equal(a[n][1], b[n][1])
    g = O.bf16_to_f64(synth.make_gains(0)["q_norm"])
    assert g.shape == (1536,) and np.all(np.abs(g - 1) <= 0.1 + 2 ** -8)


def test_ragged_lengths_range():
    L = synth.ragged_lengths(0, 64, 512, 8192)
    assert L.min() >= 512 and L.max() <= 8192 and len(L) == 64
