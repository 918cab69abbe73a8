"""mla_decode_noalloc: the decode step for callers that cannot allocate GPU memory while they
decode (an arena that owns all device memory, a runtime that forbids allocation after
start-up).  It must give the same outputs and cache as mla_decode with a caller workspace, on
consecutive calls, agree with the oracle, and refuse batches larger than its static scratch
holds.

This file is collected last so that a run stopping at its first failure has run all others."""
import numpy as np
import pytest
import torch

from head_latent_attention_mla_gb300 import mla, synth
from oracle import mla_oracle as O
from tests.mla_cases import assert_close, oracle_cache, oracle_weights, to_dev, weights_and_gains

pytestmark = pytest.mark.gpu


def _caches(layer, lengths, cap, copies):
    """`copies` identical device caches (and lengths) holding lengths[b] tokens of sequence b."""
    out = []
    for _ in range(copies):
        B = len(lengths)
        c = torch.zeros(B, cap, 576, dtype=torch.bfloat16, device="cuda")
        l = torch.zeros(B, dtype=torch.int32, device="cuda")
        for b, n in enumerate(lengths):
            if n:
                layer.cache_append(to_dev(synth.hidden_states(0, b, 0, n))[None], c[b:b + 1],
                                   l[b:b + 1], [0])
        out.append((c, l))
    torch.cuda.synchronize()
    return out


# B=1: the GEMV projections and fused kernels of the one-sequence chain in mla_decode, the
# separate kernels here.  B=3: GEMV projections.  B=4 and 8: tensor-core projections with
# split-K scratch.  Contexts past 48 x 64 positions run with the 48-item cap's longer shares.
@pytest.mark.parametrize("lengths", [[3500], [300, 1, 129], [300, 1, 129, 700],
                                     [5000, 64, 4000, 1, 3100, 128, 2000, 65]])
def test_noalloc_decode_matches_decode_on_two_calls(lengths):
    wq, g = weights_and_gains(0)
    layer = mla.MlaLayer(wq, g)
    try:
        B, cap = len(lengths), max(lengths) + 4
        (c0, l0), (c1, l1) = _caches(layer, lengths, cap, 2)
        host = list(lengths)
        for step in range(2):
            xb = np.stack([synth.hidden_states(0, b, host[b], 1)[0] for b in range(B)])
            x = to_dev(xb)
            ref = layer.decode(x, c0, l0, host)
            got = torch.empty_like(x)
            mla.mla_decode_noalloc(layer.ctx, x, c1, l1, host, got)
            torch.cuda.synchronize()
            assert layer.status() == mla.MLA_OK
            assert_close(got.float().cpu().numpy(), ref.float().cpu().numpy(),
                         f"B={B} step {step} vs mla_decode")
            assert torch.equal(l0, l1)
            # the appended rows (for one or two sequences mla_decode appends them from its
            # fused q_b kernel, so they are compared within the tolerance, not bitwise)
            rows0 = torch.stack([c0[b, host[b]] for b in range(B)]).float().cpu().numpy()
            rows1 = torch.stack([c1[b, host[b]] for b in range(B)]).float().cpu().numpy()
            assert_close(rows1, rows0, f"B={B} step {step} appended rows")
            host = [n + 1 for n in host]
        for b, n in enumerate(lengths):   # rows before the two steps are untouched
            assert torch.equal(c0[b, :n], c1[b, :n])
    finally:
        layer.close()


@pytest.mark.parametrize("lengths", [[3500], [5000, 64, 4000, 1, 3100, 128, 2000, 65]])
def test_noalloc_decode_matches_oracle(lengths):
    """Every sequence's output and appended cache row against the fp64 oracle."""
    wq, g = weights_and_gains(0)
    layer = mla.MlaLayer(wq, g)
    try:
        W = oracle_weights(0)
        B, cap = len(lengths), max(lengths) + 1
        ((c, l),) = _caches(layer, lengths, cap, 1)
        xb = np.stack([synth.hidden_states(0, b, lengths[b], 1)[0] for b in range(B)])
        out = torch.empty(B, 7168, dtype=torch.bfloat16, device="cuda")
        mla.mla_decode_noalloc(layer.ctx, to_dev(xb), c, l, lengths, out)
        torch.cuda.synchronize()
        assert layer.status() == mla.MLA_OK
        assert l.tolist() == [n + 1 for n in lengths]
        y = out.float().cpu().numpy()
        for b, n in enumerate(lengths):
            c_ref = oracle_cache(0, b, n, W)
            y_ref, full = O.decode(O.bf16_to_f64(xb[b]), c_ref, W)
            assert_close(y[b], y_ref, f"noalloc seq {b} (len {n})")
            assert_close(c[b, n:n + 1].float().cpu().numpy(), full[n:n + 1],
                         f"noalloc appended row {b}")
    finally:
        layer.close()


def test_noalloc_rejects_batches_beyond_its_scratch():
    wq, g = weights_and_gains(0)
    layer = mla.MlaLayer(wq, g)
    try:
        B = 9
        x = torch.zeros(B, 7168, dtype=torch.bfloat16, device="cuda")
        cache = torch.zeros(B, 4, 576, dtype=torch.bfloat16, device="cuda")
        lens = torch.zeros(B, dtype=torch.int32, device="cuda")
        out = torch.empty_like(x)
        with pytest.raises(mla.MlaError) as e:
            mla.mla_decode_noalloc(layer.ctx, x, cache, lens, [0] * B, out)
        assert e.value.status == mla.MLA_ERR_CAPACITY
        torch.cuda.synchronize()
        assert lens.abs().sum().item() == 0
    finally:
        layer.close()
