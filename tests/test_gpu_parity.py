"""Parity of the CUDA path (through the C ABI) with the fp64 oracle on identical seeded inputs.

Bar: FP8 dequantisation bit-exact; layer outputs within relative Frobenius error 1e-2 and
max-abs error 5e-2.  Small cases compare every element; the full-size workloads compare
sampled outputs that the oracle computes one by one.
"""
import numpy as np
import pytest
import torch

from head_latent_attention_mla_gb300 import mla, synth
from oracle import mla_oracle as O
from tests.mla_cases import (assert_close, build_caches_gpu, oracle_cache, oracle_rows,
                             oracle_weights, to_dev, weights_and_gains)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def layer():
    wq, g = weights_and_gains(0)
    L = mla.MlaLayer(wq, g)
    yield L
    L.close()


def run_prefill(layer, seqs, T, cap=None):
    """GPU prefill of sequences `seqs` (synth sequence ids), T tokens each."""
    B = len(seqs)
    xb = np.stack([synth.hidden_states(0, s, 0, T) for s in seqs])
    x = to_dev(xb)
    cap = cap or T
    cache = torch.zeros(B, cap, 576, dtype=torch.bfloat16, device="cuda")
    lens = torch.zeros(B, dtype=torch.int32, device="cuda")
    y = layer.prefill(x, cache, lens, [0] * B)
    torch.cuda.synchronize()
    assert layer.status() == mla.MLA_OK
    assert lens.tolist() == [T] * B
    return xb, y.float().cpu().numpy(), cache.float().cpu().numpy()


@pytest.mark.parametrize("name", ["q_a", "q_b", "kv_a", "kv_b", "o"])
def test_dequant_bit_exact(layer, name):
    wq, _ = weights_and_gains(0)
    got = layer.dequant(name).cpu().numpy()
    ref = O.dequant_fp32(*wq[name])
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("T", [1, 3, 4, 16, 100, 130, 1200])
def test_prefill_small_every_element(layer, T):
    """Config-1 size (T=16) and tile edge cases (T=1, T=130 = two tiles and a ragged tail).
    T=1 runs the projections as row GEMVs, T=3 and T=4 as mma.sync GEMVs (kv_b among them,
    K = 512 with four tiles per CTA).
    T=100 runs the projections as split-K over one partly filled 128-token tile.
    T=1200 runs the q_a/kv_a and o projections with 256-feature units over ten token tiles
    (the last one ragged), including the kv_a unit whose second weight half lies wholly past
    N=576."""
    W = oracle_weights(0)
    xb, y, cache = run_prefill(layer, [0], T)
    y_ref, cache_ref = O.prefill(O.bf16_to_f64(xb[0]), W)
    assert_close(y[0], y_ref, f"prefill T={T}")
    assert_close(cache[0, :T], cache_ref, f"cache T={T}")


def test_prefill_batch_of_two(layer):
    W = oracle_weights(0)
    xb, y, _ = run_prefill(layer, [3, 4], 70, cap=96)
    for b, s in enumerate([3, 4]):
        y_ref, _ = O.prefill(O.bf16_to_f64(xb[b]), W)
        assert_close(y[b], y_ref, f"batch row {b}")


@pytest.mark.parametrize("T", [16, 200])
def test_half_pairing_prefill_and_decode(T):
    """The half RoPE pairing (j, j+32): prefill (T=16: separate q RoPE kernel; T=200: RoPE in
    the q_b GEMM epilogue) and one decode step after it, every element against the oracle."""
    wq, g = weights_and_gains(0)
    L = mla.MlaLayer(wq, g, rope_pairing=mla.MLA_ROPE_HALF)
    try:
        W = oracle_weights(0)
        xb = synth.hidden_states(0, 5, 0, T + 1)
        cache = torch.zeros(1, T + 1, 576, dtype=torch.bfloat16, device="cuda")
        lens = torch.zeros(1, dtype=torch.int32, device="cuda")
        y = L.prefill(to_dev(xb[None, :T]), cache, lens, [0])
        yd = L.decode(to_dev(xb[T:T + 1]), cache, lens, [T])
        torch.cuda.synchronize()
        assert L.status() == mla.MLA_OK and lens.item() == T + 1
        xf = O.bf16_to_f64(xb)
        y_ref, cache_ref = O.prefill(xf[:T], W, pairing="half")
        yd_ref, full_ref = O.decode(xf[T], cache_ref, W, pairing="half")
        assert_close(y[0].float().cpu().numpy(), y_ref, f"half pairing prefill T={T}")
        assert_close(yd[0].float().cpu().numpy(), yd_ref, f"half pairing decode p={T}")
        assert_close(cache[0].float().cpu().numpy(), full_ref, f"half pairing cache T={T}")
    finally:
        L.close()


@pytest.mark.parametrize("L,T", [(100, 50), (128, 128), (300, 130), (37, 5)])
def test_chunked_prefill_every_element(layer, L, T):
    """A prompt prefilled in two chunks: L tokens over an empty cache, then T tokens against
    the L cached positions (query t at position L + t sees keys 0..L+t, the cached keys and
    values rebuilt from their latent rows).  Every element of the second chunk's output and
    of the whole cache against the oracle's forward over the cached rows."""
    W = oracle_weights(0)
    xb = synth.hidden_states(0, 9, 0, L + T)
    cache = torch.zeros(1, L + T + 3, 576, dtype=torch.bfloat16, device="cuda")
    lens = torch.zeros(1, dtype=torch.int32, device="cuda")
    layer.prefill(to_dev(xb[None, :L]), cache, lens, [0])
    y = layer.prefill(to_dev(xb[None, L:]), cache, lens, [L])
    torch.cuda.synchronize()
    assert layer.status() == mla.MLA_OK and lens.item() == L + T
    xf = O.bf16_to_f64(xb)
    y_ref, full_ref = O.forward(xf[L:], O.cache_rows(xf[:L], np.arange(L), W), W)
    assert_close(y[0].float().cpu().numpy(), y_ref, f"chunk L={L} T={T}")
    assert_close(cache[0, :L + T].float().cpu().numpy(), full_ref, f"cache L={L} T={T}")


def test_chunked_prefill_batch_with_different_offsets(layer):
    """Three sequences with 0, 150 and 260 cached positions take a 70-token chunk together."""
    W = oracle_weights(0)
    Ls, T, seqs = [0, 150, 260], 70, [11, 12, 13]
    xbs = [synth.hidden_states(0, s, 0, Lb + T) for s, Lb in zip(seqs, Ls)]
    cap = max(Ls) + T
    cache = torch.zeros(3, cap, 576, dtype=torch.bfloat16, device="cuda")
    lens = torch.zeros(3, dtype=torch.int32, device="cuda")
    for b, (Lb, xb) in enumerate(zip(Ls, xbs)):
        if Lb:
            one = torch.zeros(1, dtype=torch.int32, device="cuda")
            c1 = torch.zeros(1, cap, 576, dtype=torch.bfloat16, device="cuda")
            layer.prefill(to_dev(xb[None, :Lb]), c1, one, [0])
            cache[b] = c1[0]
    lens.copy_(torch.tensor(Ls, dtype=torch.int32))
    x = torch.cat([to_dev(xb[None, Lb:]) for Lb, xb in zip(Ls, xbs)])
    y = layer.prefill(x, cache, lens, Ls)
    torch.cuda.synchronize()
    assert layer.status() == mla.MLA_OK and lens.tolist() == [Lb + T for Lb in Ls]
    for b, (Lb, xb) in enumerate(zip(Ls, xbs)):
        xf = O.bf16_to_f64(xb)
        cache_ref = O.cache_rows(xf[:Lb], np.arange(Lb), W) if Lb else None
        y_ref, full_ref = O.forward(xf[Lb:], cache_ref, W)
        assert_close(y[b].float().cpu().numpy(), y_ref, f"sequence {b} (L={Lb})")
        assert_close(cache[b, :Lb + T].float().cpu().numpy(), full_ref, f"cache {b}")


def test_yarn_chunk_and_decode_at_6000():
    """YaRN RoPE with Kimi-K2's rope_scaling: a cache of 6000 positions built by append, a
    16-token chunk at positions 6000..6015, then one decode step at 6016 -- far enough that the
    interpolated pairs turn -- every element against the oracle with the same option (which
    also takes the score temperature)."""
    wq, g = weights_and_gains(0)
    Lr = mla.MlaLayer(wq, g, rope_scaling=mla.MLA_ROPE_YARN)
    try:
        W, Y, P = oracle_weights(0), O.Yarn(), 6000
        xb = synth.hidden_states(0, 21, 0, P + 17)
        cache = torch.zeros(1, P + 17, 576, dtype=torch.bfloat16, device="cuda")
        lens = torch.zeros(1, dtype=torch.int32, device="cuda")
        Lr.cache_append(to_dev(xb[None, :P]), cache, lens, [0])
        y = Lr.prefill(to_dev(xb[None, P:P + 16]), cache, lens, [P])
        yd = Lr.decode(to_dev(xb[P + 16:P + 17]), cache, lens, [P + 16])
        torch.cuda.synchronize()
        assert Lr.status() == mla.MLA_OK and lens.item() == P + 17
        xf = O.bf16_to_f64(xb)
        cache_ref = O.cache_rows(xf[:P], np.arange(P), W, yarn=Y)
        y_ref, full = O.forward(xf[P:P + 16], cache_ref, W, yarn=Y)
        yd_ref, full2 = O.decode(xf[P + 16], full, W, yarn=Y)
        assert_close(y[0].float().cpu().numpy(), y_ref, "yarn chunk")
        assert_close(yd[0].float().cpu().numpy(), yd_ref, "yarn decode")
        assert_close(cache[0].float().cpu().numpy(), full2, "yarn cache")
    finally:
        Lr.close()


def test_decode_config2_p1000(layer):
    """Decode at position 1000 over a cache built by a causal prefill of 1000 tokens."""
    W = oracle_weights(0)
    p = 1000
    xb = synth.hidden_states(0, 0, 0, p + 1)
    cache = torch.zeros(1, p + 8, 576, dtype=torch.bfloat16, device="cuda")
    lens = torch.zeros(1, dtype=torch.int32, device="cuda")
    layer.prefill(to_dev(xb[None, :p]), cache, lens, [0])
    yd = layer.decode(to_dev(xb[p:p + 1]), cache, lens, [p])
    torch.cuda.synchronize()
    assert layer.status() == mla.MLA_OK and lens.item() == p + 1
    xf = O.bf16_to_f64(xb)
    cache_ref = O.cache_rows(xf[:p], np.arange(p), W)
    y_ref, full_ref = O.decode(xf[p], cache_ref, W)
    assert_close(yd[0].float().cpu().numpy(), y_ref, "decode p=1000")
    assert_close(cache[0, :p + 1].float().cpu().numpy(), full_ref, "cache after decode")


def test_decode_matches_last_prefill_row_on_gpu(layer):
    """Decode at p equals row p of a causal prefill over p+1 tokens (both on the GPU)."""
    p = 200
    xb = synth.hidden_states(0, 7, 0, p + 1)
    _, y_pre, _ = run_prefill(layer, [7], p + 1)
    cache = torch.zeros(1, p + 1, 576, dtype=torch.bfloat16, device="cuda")
    lens = torch.zeros(1, dtype=torch.int32, device="cuda")
    layer.cache_append(to_dev(xb[None, :p]), cache, lens, [0])
    yd = layer.decode(to_dev(xb[p:p + 1]), cache, lens, [p])
    assert_close(yd[0].float().cpu().numpy(), y_pre[0, p], "decode vs prefill row")


def test_prefill_config3_t4096_sampled(layer):
    """Full-size prefill (T=4096): every cache row, and 160 output rows against the oracle --
    the tile edges of the first, middle and last 128-query tiles plus 128 rows drawn at
    random (seeded) over the whole prompt."""
    W = oracle_weights(0)
    T = 4096
    xb, y, cache = run_prefill(layer, [0], T)
    xf = O.bf16_to_f64(xb[0])
    cache_ref = O.cache_rows(xf, np.arange(T), W)
    assert_close(cache[0], cache_ref, "cache T=4096")
    edges = [0, 1, 63, 64, 65, 127, 128, 129, 2047, 2048, 2049, 3967, 3968, 4094, 4095]
    rnd = np.random.default_rng(40).choice(T, 145, replace=False)
    rows = np.unique(np.concatenate([edges, rnd]))
    assert_close(y[0, rows], oracle_rows(xf, rows, cache_ref, W), f"prefill T=4096 {len(rows)} rows")


def _one_at_a_time(layer, x, cache0, lens0, lengths):
    """mla_decode of each sequence alone (B=1: another split-KV plan and the GEMV
    projections) on copies of the caches as they were before the batched step."""
    outs = []
    for b, n in enumerate(lengths):
        outs.append(layer.decode(x[b:b + 1], cache0[b:b + 1], lens0[b:b + 1], [n])[0])
    torch.cuda.synchronize()
    return torch.stack(outs)


def test_decode_config4_ragged_b64_sampled(layer):
    """Ragged decode, B=64, lengths ~U[512, 8192].  Against the oracle: 16 sequences spread
    over the length range (shortest to longest) and every sequence's appended cache row.
    Against the same layer run one sequence at a time: all 64 outputs and appended rows
    (the batched share plan cuts sequences at places the single-sequence plan does not)."""
    W = oracle_weights(0)
    lengths = synth.ragged_lengths(0, 64, 512, 8192).tolist()
    cap = max(lengths) + 1
    cache, lens = build_caches_gpu(layer, 0, lengths, cap)
    cache0, lens0 = cache.clone(), lens.clone()
    xb = np.stack([synth.hidden_states(0, b, lengths[b], 1)[0] for b in range(64)])
    x = to_dev(xb)
    yd_dev = layer.decode(x, cache, lens, lengths)
    torch.cuda.synchronize()
    assert layer.status() == mla.MLA_OK
    assert lens.tolist() == [n + 1 for n in lengths]
    yd = yd_dev.float().cpu().numpy()
    # every appended row against the oracle
    rows_ref = np.stack([O.cache_rows(O.bf16_to_f64(xb[b])[None], np.array([lengths[b]]), W)[0]
                         for b in range(64)])
    rows_got = torch.stack([cache[b, lengths[b]] for b in range(64)]).float().cpu().numpy()
    assert_close(rows_got, rows_ref, "ragged appended rows (64)")
    order = np.argsort(lengths)
    for b in [int(order[i]) for i in np.linspace(0, 63, 16).round().astype(int)]:
        c_ref = oracle_cache(0, b, lengths[b], W)
        y_ref, _ = O.decode(O.bf16_to_f64(xb[b]), c_ref, W)
        assert_close(yd[b], y_ref, f"ragged decode seq {b} (len {lengths[b]})")
    single = _one_at_a_time(layer, x, cache0, lens0, lengths)
    assert layer.status() == mla.MLA_OK
    assert_close(yd, single.float().cpu().numpy(), "ragged B=64 vs one at a time")
    got1 = torch.stack([cache0[b, lengths[b]] for b in range(64)]).float().cpu().numpy()
    assert_close(got1, rows_got, "ragged appended rows vs one at a time")


def test_decode_config5_long_b8_every_sequence(layer):
    """Long-context decode, B=8 x 131,072 cached positions: all eight outputs and appended
    rows against the oracle, plus sampled cache rows."""
    W = oracle_weights(0)
    L = 131072
    cache, lens = build_caches_gpu(layer, 0, [L] * 8, L + 1)
    xb = np.stack([synth.hidden_states(0, b, L, 1)[0] for b in range(8)])
    yd = layer.decode(to_dev(xb), cache, lens, [L] * 8)
    torch.cuda.synchronize()
    assert layer.status() == mla.MLA_OK
    assert lens.tolist() == [L + 1] * 8
    yd = yd.float().cpu().numpy()
    for b in range(8):
        c_ref = oracle_cache(0, b, L, W)
        y_ref, full = O.decode(O.bf16_to_f64(xb[b]), c_ref, W)
        assert_close(yd[b], y_ref, f"long decode seq {b}")
        idx = [0, 4095, 4096, 77777, L - 1, L]
        assert_close(cache[b, idx].float().cpu().numpy(), full[idx], f"long cache rows seq {b}")


# One sequence and two take the six-kernel decode (fused q-latent norm and cache append, fused
# combine and W_UV, row GEMVs); three and four the separate kernels with the mma.sync GEMV;
# five to eight the tcgen05 projections; nine and more also the batched tcgen05 absorptions
# (nine: one 32-token tile with 23 empty rows; seventeen: a 64-token tile).
@pytest.mark.parametrize("lengths", [[0], [65, 300], [5, 64, 129], [3, 0, 70, 64],
                                     [1, 63, 64, 65, 127, 128, 129, 200],
                                     [1, 63, 64, 65, 127, 128, 129, 200, 0],
                                     [int(v) for v in np.arange(17) * 37 % 300]])
def test_decode_tile_edges_every_sequence(layer, lengths):
    """Empty cache (p=0) and lengths around the 64-position tile edges, all sequences checked,
    with the cache row each decode appends."""
    W = oracle_weights(0)
    cap = max(lengths) + 3
    cache, lens = build_caches_gpu(layer, 0, lengths, cap)
    xb = np.stack([synth.hidden_states(0, b, lengths[b], 1)[0] for b in range(len(lengths))])
    yd = layer.decode(to_dev(xb), cache, lens, lengths)
    torch.cuda.synchronize()
    assert layer.status() == mla.MLA_OK
    assert lens.tolist() == [n + 1 for n in lengths]
    yd = yd.float().cpu().numpy()
    for b, n in enumerate(lengths):
        c_ref = oracle_cache(0, b, n, W) if n else None
        y_ref, _ = O.decode(O.bf16_to_f64(xb[b]), c_ref if n else np.zeros((0, 576)), W)
        assert_close(yd[b], y_ref, f"decode len {n}")
        row_ref = O.cache_rows(O.bf16_to_f64(xb[b])[None], np.array([n]), W)
        assert_close(cache[b, n:n + 1].float().cpu().numpy(), row_ref, f"appended row {n}")


def test_decode_growing_scores_rescale(layer):
    """Later tokens scaled x5: their rotary keys (not normalised by RMSNorm) grow, so the
    running maximum of the scores jumps by far more than 2^8 in late tiles and the output
    kept so far must be rescaled.  (Much larger scales make bf16 rounding of the keys alone
    exceed the tolerance, in any implementation that stores the cache in bf16.)"""
    W = oracle_weights(0)
    n = 700
    xb = synth.hidden_states(0, 11, 0, n + 1)
    xf = O.bf16_to_f64(xb)
    xf[400:] *= 5.0
    from head_latent_attention_mla_gb300.synth import to_bf16_bits
    xb = to_bf16_bits(xf.astype(np.float32))
    xf = O.bf16_to_f64(xb)
    cache = torch.zeros(1, n + 1, 576, dtype=torch.bfloat16, device="cuda")
    lens = torch.zeros(1, dtype=torch.int32, device="cuda")
    layer.cache_append(to_dev(xb[None, :n]), cache, lens, [0])
    yd = layer.decode(to_dev(xb[n:n + 1]), cache, lens, [n])
    torch.cuda.synchronize()
    assert layer.status() == mla.MLA_OK
    c_ref = O.cache_rows(xf[:n], np.arange(n), W)
    y_ref, _ = O.decode(xf[n], c_ref, W)
    assert_close(yd[0].float().cpu().numpy(), y_ref, "rescaled decode")
