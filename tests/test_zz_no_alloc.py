"""mla_decode_noalloc: the decode step for callers that cannot allocate GPU memory while they
decode (an arena that owns all device memory, a runtime that forbids allocation after
start-up).  It must give the same outputs and cache as mla_decode with a caller workspace, on
consecutive calls, and refuse batches larger than its static scratch holds.

This file is collected last so that a run stopping at its first failure has run all others."""
import numpy as np
import pytest
import torch

from head_latent_attention_mla_gb300 import mla, synth
from tests.mla_cases import assert_close, to_dev, weights_and_gains

pytestmark = pytest.mark.gpu


def test_noalloc_decode_matches_decode_on_two_calls():
    wq, g = weights_and_gains(0)
    layer = mla.MlaLayer(wq, g)
    lengths = [300, 1, 129, 700]
    B, cap = len(lengths), max(lengths) + 4
    caches, lens = [], []
    for _ in range(2):   # identical caches for the two entry points
        c = torch.zeros(B, cap, 576, dtype=torch.bfloat16, device="cuda")
        l = torch.zeros(B, dtype=torch.int32, device="cuda")
        for b, n in enumerate(lengths):
            layer.cache_append(to_dev(synth.hidden_states(0, b, 0, n))[None], c[b:b + 1],
                               l[b:b + 1], [0])
        caches.append(c)
        lens.append(l)
    host = list(lengths)
    for step in range(2):
        xb = np.stack([synth.hidden_states(0, b, host[b], 1)[0] for b in range(B)])
        x = to_dev(xb)
        ref = layer.decode(x, caches[0], lens[0], host)
        got = torch.empty_like(x)
        mla.mla_decode_noalloc(layer.ctx, x, caches[1], lens[1], host, got)
        torch.cuda.synchronize()
        assert layer.status() == mla.MLA_OK
        assert_close(got.float().cpu().numpy(), ref.float().cpu().numpy(), f"step {step}")
        assert torch.equal(lens[0], lens[1])
        assert torch.equal(caches[0], caches[1])
        host = [n + 1 for n in host]
    layer.close()


def test_noalloc_rejects_batches_beyond_its_scratch():
    wq, g = weights_and_gains(0)
    layer = mla.MlaLayer(wq, g)
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
    layer.close()
