"""Boundary behaviour on the GPU: host-side argument checks return status codes before any
launch, and device-side range checks record an error instead of faulting."""
import numpy as np
import pytest
import torch

from head_latent_attention_mla_gb300 import mla, synth
from tests.mla_cases import to_dev, weights_and_gains

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def layer():
    wq, g = weights_and_gains(0)
    L = mla.MlaLayer(wq, g)
    yield L
    L.close()


def test_capacity_and_mode_errors(layer):
    x = to_dev(synth.hidden_states(0, 0, 0, 8))[None]
    cache = torch.zeros(1, 8, 576, dtype=torch.bfloat16, device="cuda")
    lens = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty_like(x)
    ws = layer.workspace(1, 8)
    with pytest.raises(mla.MlaError) as e:
        mla.mla_prefill(layer.ctx, x, cache[:, :4].contiguous(), lens, [0], out, ws)
    assert e.value.status == mla.MLA_ERR_CAPACITY
    with pytest.raises(mla.MlaError) as e:
        mla.mla_prefill(layer.ctx, x, cache, lens, [3], out, ws)
    assert e.value.status in (mla.MLA_ERR_CAPACITY, mla.MLA_ERR_UNSUPPORTED)
    # A chunk after 2000 cached positions needs room for 2002 rebuilt key/value rows: the
    # workspace for an empty cache is refused (before the capacity check).
    small = ws[:mla.mla_workspace_bytes(layer.ctx, 1, 2)]
    assert mla.mla_workspace_bytes_len(layer.ctx, 1, 2, 2002) > small.numel()
    with pytest.raises(mla.MlaError) as e:
        mla.mla_prefill(layer.ctx, x[:, :2].contiguous(), cache, lens, [2000],
                        out[:, :2].contiguous(), small)
    assert e.value.status == mla.MLA_ERR_INVALID_ARG
    with pytest.raises(mla.MlaError) as e:
        mla.mla_decode(layer.ctx, x[0, :1].contiguous(), cache, lens, [8], out[0, :1].contiguous(), ws)
    assert e.value.status == mla.MLA_ERR_CAPACITY
    torch.cuda.synchronize()
    assert lens.item() == 0 and cache.abs().sum().item() == 0   # nothing was written


def test_upload_shape_errors(layer):
    q, s = layer.w["q_a"]
    with pytest.raises(mla.MlaError) as e:
        mla.mla_upload_weights(layer.ctx, mla.MLA_W_Q_B, q, s)
    assert e.value.status == mla.MLA_ERR_SHAPE
    with pytest.raises(mla.MlaError) as e:
        mla.mla_upload_norm(layer.ctx, mla.MLA_NORM_KV, layer.g["q_norm"])
    assert e.value.status == mla.MLA_ERR_SHAPE


def test_device_range_check_flags_instead_of_faulting(layer):
    """Device lengths past the cache (host copy stale): rows are skipped, the error word set."""
    x = to_dev(synth.hidden_states(0, 0, 0, 2))[None]
    cache = torch.zeros(1, 4, 576, dtype=torch.bfloat16, device="cuda")
    lens = torch.full((1,), 4, dtype=torch.int32, device="cuda")   # device says full
    layer.cache_append(x, cache, lens, [0])                           # host says empty
    torch.cuda.synchronize()
    assert layer.status() == mla.MLA_ERR_STATE
    assert cache.abs().sum().item() == 0
    assert layer.status() == mla.MLA_OK                              # the word was cleared


def test_repeat_runs_are_bitwise_identical(layer):
    xb = synth.hidden_states(0, 2, 0, 300)
    outs = []
    for _ in range(2):
        cache = torch.zeros(1, 300, 576, dtype=torch.bfloat16, device="cuda")
        lens = torch.zeros(1, dtype=torch.int32, device="cuda")
        y = layer.prefill(to_dev(xb[None, :299]), cache, lens, [0])
        yd = layer.decode(to_dev(xb[299:300]), cache, lens, [299])
        outs.append((y.clone(), yd.clone(), cache.clone()))
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(a, b)
