"""The attention half of a decoder block (mla_config.block = 1; "Attention input" page, `block`
excerpt): y = x + layer(input_layernorm(x)), against the fp64 oracle's block_forward.

The whole output is held to the bar (rel-Frobenius 1e-2, max-abs 5e-2).  The attention's
contribution y - x is small next to the residual, and the output's final bf16 rounding (up to
2^-9 |y| per element) is the module's own arithmetic, so that part is held to the max-abs bar
only, which a missing or wrong attention term fails."""
import numpy as np
import pytest
import torch

from head_latent_attention_mla_gb300 import mla, synth
from oracle import mla_oracle as O
from tests.mla_cases import (MAX_ABS_TOL, assert_close, errors, oracle_weights, to_dev,
                             weights_and_gains)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def blk():
    wq, g = weights_and_gains(0)
    gains = dict(g, input_norm=synth.make_input_gain(0))
    L = mla.MlaLayer(wq, gains, block=1)
    yield L
    L.close()


def g_in():
    return O.bf16_to_f64(synth.make_input_gain(0))


def check(got, x, ref, what):
    got = np.asarray(got, np.float64)
    assert_close(got, ref, what)
    _, mx = errors(got - x, ref - x)
    assert mx <= MAX_ABS_TOL, f"{what}: attention part max_abs {mx:.3e}"


@pytest.mark.parametrize("T", [1, 16, 130])
def test_block_prefill_every_element(blk, T):
    """T=1: the CUDA-core GEMV epilogue adds the residual; 16: split-K with the residual in the
    reduce; 130: the token-lane tensor-core epilogue."""
    W = oracle_weights(0)
    xb = synth.hidden_states(0, 60, 0, T)
    cache = torch.zeros(1, T + 1, 576, dtype=torch.bfloat16, device="cuda")
    lens = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = blk.prefill(to_dev(xb[None]), cache, lens, [0])
    torch.cuda.synchronize()
    assert blk.status() == mla.MLA_OK and lens.item() == T
    xf = O.bf16_to_f64(xb)
    y_ref, cache_ref = O.block_forward(xf, None, W, g_in())
    check(y[0].float().cpu().numpy(), xf, y_ref, f"block prefill T={T}")
    assert_close(cache[0, :T].float().cpu().numpy(), cache_ref, f"block cache T={T}")


@pytest.mark.parametrize("lengths", [[300], [5, 64, 129, 200, 1]])
def test_block_chunk_then_decode(blk, lengths):
    """A prompt prefilled as two chunks, then one decode step, for one sequence (GEMV chain)
    and five (tensor-core projections with split-K): every output against the oracle."""
    W = oracle_weights(0)
    B = len(lengths)
    cap = max(lengths) + 2
    xbs = [synth.hidden_states(0, 70 + b, 0, n + 1) for b, n in enumerate(lengths)]
    cache = torch.zeros(B, cap, 576, dtype=torch.bfloat16, device="cuda")
    lens = torch.zeros(B, dtype=torch.int32, device="cuda")
    for b, n in enumerate(lengths):   # two chunks per sequence, one sequence at a time
        h = n // 2
        for a0, a1 in ((0, h), (h, n)):
            if a1 > a0:
                blk.prefill(to_dev(xbs[b][None, a0:a1]), cache[b:b + 1], lens[b:b + 1], [a0])
    x = to_dev(np.stack([xbs[b][n] for b, n in enumerate(lengths)]))
    yd = blk.decode(x, cache, lens, lengths)
    torch.cuda.synchronize()
    assert blk.status() == mla.MLA_OK and lens.tolist() == [n + 1 for n in lengths]
    for b, n in enumerate(lengths):
        xf = O.bf16_to_f64(xbs[b])
        _, c_ref = O.block_forward(xf[:n], None, W, g_in())
        y_ref, full = O.block_forward(xf[n:n + 1], c_ref, W, g_in())
        check(yd[b:b + 1].float().cpu().numpy(), xf[n:n + 1], y_ref, f"block decode seq {b}")
        assert_close(cache[b, :n + 1].float().cpu().numpy(), full, f"block cache seq {b}")


def test_block_paged_decode_and_noalloc_refusal(blk):
    W = oracle_weights(0)
    n, page = 500, 64
    xb = synth.hidden_states(0, 80, 0, n + 1)
    pool = torch.zeros(12, page, 576, dtype=torch.bfloat16, device="cuda")
    table = torch.tensor([[7, 3, 11, 0, 5, 9, 1, 2, 4]], dtype=torch.int32, device="cuda")
    lens = torch.zeros(1, dtype=torch.int32, device="cuda")
    blk.prefill_paged(to_dev(xb[None, :n]), pool, table, lens, [0])
    yd = blk.decode_paged(to_dev(xb[n:n + 1]), pool, table, lens, [n])
    torch.cuda.synchronize()
    assert blk.status() == mla.MLA_OK
    xf = O.bf16_to_f64(xb)
    _, c_ref = O.block_forward(xf[:n], None, W, g_in())
    y_ref, _ = O.block_forward(xf[n:], c_ref, W, g_in())
    check(yd.float().cpu().numpy(), xf[n:], y_ref, "block paged decode")
    out = torch.empty_like(yd)
    cache = torch.zeros(1, 4, 576, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(mla.MlaError) as e:
        mla.mla_decode_noalloc(blk.ctx, to_dev(xb[:1]), cache, torch.zeros_like(lens), [0], out)
    assert e.value.status == mla.MLA_ERR_UNSUPPORTED


def test_block_needs_its_input_gain():
    wq, g = weights_and_gains(0)
    L = mla.MlaLayer(wq, g, block=1)   # input_norm gain not uploaded
    try:
        x = to_dev(synth.hidden_states(0, 1, 0, 4))[None]
        cache = torch.zeros(1, 4, 576, dtype=torch.bfloat16, device="cuda")
        lens = torch.zeros(1, dtype=torch.int32, device="cuda")
        with pytest.raises(mla.MlaError) as e:
            L.prefill(x, cache, lens, [0])
        assert e.value.status == mla.MLA_ERR_STATE
    finally:
        L.close()
