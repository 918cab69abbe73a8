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


@pytest.mark.parametrize("B,T", [(1, 299), (8, 16), (1, 16)])
def test_repeat_runs_are_bitwise_identical(layer, B, T):
    """Prefill of T tokens then one decode step, twice on fresh caches: every output and cache
    row bit for bit the same.  B=8 decodes through the tcgen05 projections with split-K, and
    T=16 prefills through the split-K GEMMs, all under programmatic dependent launch (a kernel
    that read its predecessor's data too early would show here)."""
    xb = np.stack([synth.hidden_states(0, 2 + b, 0, T + 1) for b in range(B)])
    outs = []
    for _ in range(2):
        cache = torch.zeros(B, T + 1, 576, dtype=torch.bfloat16, device="cuda")
        lens = torch.zeros(B, dtype=torch.int32, device="cuda")
        y = layer.prefill(to_dev(xb[:, :T]), cache, lens, [0] * B)
        yd = layer.decode(to_dev(xb[:, T]), cache, lens, [T] * B)
        torch.cuda.synchronize()
        assert layer.status() == mla.MLA_OK
        outs.append((y.clone(), yd.clone(), cache.clone()))
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(a, b)
    assert not torch.isnan(outs[0][1].float()).any()


def _injected_layer(n):
    """A layer whose context fails every token call at launch n (MLA_TEST_FAIL_AFTER)."""
    import os
    wq, g = weights_and_gains(0)
    os.environ["MLA_TEST_FAIL_AFTER"] = str(n)
    try:
        return mla.MlaLayer(wq, g)
    finally:
        del os.environ["MLA_TEST_FAIL_AFTER"]


@pytest.mark.parametrize("B,p", [(1, 100), (5, 70)])
def test_injected_launch_failure_never_advances_lengths(layer, B, p):
    """A decode that fails at launch n (host-side injection, for every n the call has):
    MLA_ERR_CUDA reaches the caller, the device lengths stay, the cached rows 0..p-1 are
    untouched, the device status stays clean, and the same state then decodes correctly."""
    xb = np.stack([synth.hidden_states(0, b, 0, p + 1) for b in range(B)])
    cache = torch.zeros(B, p + 1, 576, dtype=torch.bfloat16, device="cuda")
    lens = torch.zeros(B, dtype=torch.int32, device="cuda")
    layer.prefill(to_dev(xb[:, :p]), cache, lens, [0] * B)
    x = to_dev(xb[:, p])
    ref = layer.decode(x, cache.clone(), lens.clone(), [p] * B)
    n_launch = len(mla.mla_last_launches(layer.ctx))
    assert n_launch >= 5
    before = cache[:, :p].clone()
    for n in range(n_launch):
        bad = _injected_layer(n)
        try:
            out = torch.zeros_like(x)
            with pytest.raises(mla.MlaError) as e:
                bad.decode(x, cache, lens, [p] * B, out=out)
            assert e.value.status == mla.MLA_ERR_CUDA
            torch.cuda.synchronize()
            assert bad.status() == mla.MLA_OK
            assert lens.tolist() == [p] * B, f"lengths advanced by a call failed at launch {n}"
            assert torch.equal(cache[:, :p], before)
        finally:
            bad.close()
    got = layer.decode(x, cache, lens, [p] * B)
    torch.cuda.synchronize()
    assert lens.tolist() == [p + 1] * B
    assert torch.equal(got, ref)


def test_injected_failure_in_prefill(layer):
    xb = synth.hidden_states(0, 3, 0, 40)
    x = to_dev(xb[None])
    for n in (0, 2, 5):
        bad = _injected_layer(n)
        try:
            cache = torch.zeros(1, 40, 576, dtype=torch.bfloat16, device="cuda")
            lens = torch.zeros(1, dtype=torch.int32, device="cuda")
            with pytest.raises(mla.MlaError) as e:
                bad.prefill(x, cache, lens, [0])
            assert e.value.status == mla.MLA_ERR_CUDA
            torch.cuda.synchronize()
            assert lens.item() == 0
        finally:
            bad.close()


def test_bounded_wait_gives_up_and_context_stays_usable(layer):
    """The library's bounded wait on an mbarrier nothing arrives at (1 ms limit) records a
    timeout: MLA_ERR_TIMEOUT from the status call, which clears it; a decode then runs
    normally."""
    mla.mla_selftest_wait_timeout(layer.ctx, 1_000_000)
    assert layer.status() == mla.MLA_ERR_TIMEOUT
    assert layer.status() == mla.MLA_OK
    with pytest.raises(mla.MlaError) as e:
        mla.mla_selftest_wait_timeout(layer.ctx, 3_000_000_000)
    assert e.value.status == mla.MLA_ERR_INVALID_ARG
    xb = synth.hidden_states(0, 4, 0, 33)
    cache = torch.zeros(1, 33, 576, dtype=torch.bfloat16, device="cuda")
    lens = torch.zeros(1, dtype=torch.int32, device="cuda")
    layer.prefill(to_dev(xb[None, :32]), cache, lens, [0])
    layer.decode(to_dev(xb[32:33]), cache, lens, [32])
    torch.cuda.synchronize()
    assert layer.status() == mla.MLA_OK and lens.item() == 33


def test_ragged_b64_decode_is_bitwise_repeatable(layer):
    """The B > 8 path (log-sum-exp combine over shares that cut sequences anywhere, tiled
    W_UV absorption, tensor-core projections) gives the same bits on repeated runs."""
    from tests.mla_cases import build_caches_gpu
    lengths = synth.ragged_lengths(1, 64, 100, 1500).tolist()
    cache, lens = build_caches_gpu(layer, 1, lengths, max(lengths) + 1)
    xb = np.stack([synth.hidden_states(1, b, lengths[b], 1)[0] for b in range(64)])
    x = to_dev(xb)
    outs = []
    for _ in range(3):
        c, l = cache.clone(), lens.clone()
        y = layer.decode(x, c, l, lengths)
        torch.cuda.synchronize()
        outs.append((y, torch.stack([c[b, lengths[b]] for b in range(64)])))
    assert layer.status() == mla.MLA_OK
    for y, rows in outs[1:]:
        assert torch.equal(y, outs[0][0]) and torch.equal(rows, outs[0][1])


@pytest.mark.parametrize("B", [1, 3, 9])
@pytest.mark.parametrize("pinned", [True, False])
def test_decode_host_equals_decode(layer, B, pinned):
    """mla_decode_host (input and output in host memory, the copies enqueued by the call: as
    kernels of the chain for page-locked buffers, by cudaMemcpyAsync otherwise) gives the same
    output, cache rows and lengths as mla_decode on device buffers, bit for bit.  B = 1, 3, 9
    cover the row GEMV, the mma.sync GEMV and the tcgen05 projections as the first kernel
    behind the input copy."""
    T = 40
    xb = np.stack([synth.hidden_states(0, 5 + b, 0, T + 1) for b in range(B)])
    res = []
    for host in (False, True):
        cache = torch.zeros(B, T + 1, 576, dtype=torch.bfloat16, device="cuda")
        lens = torch.zeros(B, dtype=torch.int32, device="cuda")
        layer.prefill(to_dev(xb[:, :T]), cache, lens, [0] * B)
        xd = to_dev(xb[:, T])
        if host:
            xh = torch.empty(xd.shape, dtype=xd.dtype, pin_memory=pinned)
            xh.copy_(xd.cpu())
            oh = torch.empty(xd.shape, dtype=xd.dtype, pin_memory=pinned)
            layer.decode_host(xh, cache, lens, [T] * B, oh)
            torch.cuda.synchronize()
            names = [n for n, _ in mla.mla_last_launches(layer.ctx)]
            assert ("copy_in" in names and "copy_out" in names) == pinned, names
            y = oh.clone()
        else:
            y = layer.decode(xd, cache, lens, [T] * B).cpu()
        torch.cuda.synchronize()
        assert layer.status() == mla.MLA_OK
        res.append((y, cache.cpu(), lens.cpu()))
    for a, b in zip(*res):
        assert torch.equal(a, b)
    assert not torch.isnan(res[0][0].float()).any()


def test_decode_host_argument_errors(layer):
    """Host-side checks before anything is enqueued: a short workspace, the same buffer for
    input and output."""
    x = torch.zeros(1, 7168, dtype=torch.bfloat16, pin_memory=True)
    o = torch.zeros_like(x)
    cache = torch.zeros(1, 8, 576, dtype=torch.bfloat16, device="cuda")
    lens = torch.zeros(1, dtype=torch.int32, device="cuda")
    small = torch.empty(mla.mla_decode_host_workspace_bytes(layer.ctx, 1) - 256,
                        dtype=torch.uint8, device="cuda")
    with pytest.raises(mla.MlaError) as e:
        mla.mla_decode_host(layer.ctx, x, cache, lens, [0], o, small)
    assert e.value.status == mla.MLA_ERR_INVALID_ARG
    with pytest.raises(mla.MlaError) as e:
        mla.mla_decode_host(layer.ctx, x, cache, lens, [0], x, layer.workspace_host(1))
    assert e.value.status == mla.MLA_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert lens.item() == 0
