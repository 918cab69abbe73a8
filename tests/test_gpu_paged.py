"""The paged latent cache ("KV cache" page: a cache that grows call by call) against the dense
one and against the fp64 oracle.

The pool is filled with NaN before use and its pages are handed out in a shuffled order, so a
row read from the wrong page, or a row past a sequence's end that reaches the arithmetic,
shows.  The paged calls write the same cache rows as the dense ones, bit for bit.  Prefill
outputs are bitwise equal too; decode outputs agree within the bar (a paged decode reads its
shares in page-aligned tiles, a dense one from each share's first position, so the sums run
in a different order).  Every element is also checked against the oracle."""
import math

import numpy as np
import pytest
import torch

from head_latent_attention_mla_gb300 import mla, synth
from oracle import mla_oracle as O
from tests.mla_cases import assert_close, oracle_weights, to_dev, weights_and_gains

pytestmark = pytest.mark.gpu
BF16_NAN = 0x7FC0


@pytest.fixture(scope="module")
def layer():
    wq, g = weights_and_gains(0)
    L = mla.MlaLayer(wq, g)
    yield L
    L.close()


def make_pool(B, capacity, page, seed):
    """A NaN-filled pool and a block table mapping every logical page of every sequence to a
    distinct pool page, in a seeded random order (plus two pages nobody owns)."""
    max_pages = math.ceil(capacity / page)
    num_pages = B * max_pages + 2
    perm = np.random.default_rng(seed).permutation(num_pages)[: B * max_pages]
    table = torch.from_numpy(perm.reshape(B, max_pages).astype(np.int32)).cuda()
    pool = torch.full((num_pages, page, 576), BF16_NAN, dtype=torch.int16, device="cuda")
    return pool.view(torch.bfloat16), table


def logical_rows(pool, table, b, n):
    """Rows 0..n-1 of sequence b read through the block table (torch indexing)."""
    page = pool.shape[1]
    pos = torch.arange(n, device="cuda")
    return pool[table[b, pos // page].long(), pos % page]


def build_both(layer, lengths, page, capacity, seed=0):
    """Dense and paged caches holding lengths[b] tokens of sequence b, both by cache append."""
    B = len(lengths)
    dense = torch.zeros(B, capacity, 576, dtype=torch.bfloat16, device="cuda")
    dl = torch.zeros(B, dtype=torch.int32, device="cuda")
    pool, table = make_pool(B, capacity, page, seed + 1)
    pl = torch.zeros(B, dtype=torch.int32, device="cuda")
    for b, n in enumerate(lengths):
        if n == 0:
            continue
        x = to_dev(synth.hidden_states(seed, b, 0, n))[None]
        layer.cache_append(x, dense[b:b + 1], dl[b:b + 1], [0])
        # one sequence of the paged batch: its own table row
        layer.cache_append_paged(x, pool, table[b:b + 1].contiguous(), pl[b:b + 1], [0])
    torch.cuda.synchronize()
    assert layer.status() == mla.MLA_OK
    return dense, dl, pool, table, pl


@pytest.mark.parametrize("lengths,page", [([1000], 64), ([130, 64, 700], 128),
                                          ([1, 63, 64, 65, 200, 333, 600, 127, 5], 64)])
def test_paged_decode_matches_dense_and_oracle(layer, lengths, page):
    """One decode step: one sequence (fused six-kernel chain), three (CUDA-core projections) and
    nine (the B > 8 combine and tiled W_UV).  Appended rows equal the dense cache's bit for
    bit and outputs are within the bar of the dense call's; every output and appended row is
    within the bar of the oracle."""
    W = oracle_weights(0)
    B, capacity = len(lengths), max(lengths) + 70
    dense, dl, pool, table, pl = build_both(layer, lengths, page, capacity)
    for b, n in enumerate(lengths):
        assert torch.equal(logical_rows(pool, table, b, n), dense[b, :n])
    xb = np.stack([synth.hidden_states(0, b, lengths[b], 1)[0] for b in range(B)])
    x = to_dev(xb)
    yd = layer.decode(x, dense, dl, lengths)
    yp = layer.decode_paged(x, pool, table, pl, lengths)
    torch.cuda.synchronize()
    assert layer.status() == mla.MLA_OK
    assert pl.tolist() == [n + 1 for n in lengths]
    assert_close(yp.float().cpu().numpy(), yd.float().cpu().numpy(), f"paged vs dense, page {page}")
    for b, n in enumerate(lengths):
        assert torch.equal(logical_rows(pool, table, b, n + 1), dense[b, :n + 1])
    y = yp.float().cpu().numpy()
    for b, n in enumerate(lengths):
        c_ref = O.cache_rows(O.bf16_to_f64(synth.hidden_states(0, b, 0, n)), np.arange(n), W)
        y_ref, full = O.decode(O.bf16_to_f64(xb[b]), c_ref, W)
        assert_close(y[b], y_ref, f"paged decode seq {b} (len {n}, page {page})")
        assert_close(logical_rows(pool, table, b, n + 1)[n:].float().cpu().numpy(), full[n:],
                     f"paged appended row {b}")


def test_paged_prefill_bitwise_equals_dense(layer):
    """Prefill of two 200-token prompts over empty paged caches (64-position pages, so every
    128-key tile of the attention spans two pages)."""
    W = oracle_weights(0)
    T, page = 200, 64
    xb = np.stack([synth.hidden_states(0, s, 0, T) for s in (30, 31)])
    x = to_dev(xb)
    dense = torch.zeros(2, T, 576, dtype=torch.bfloat16, device="cuda")
    dl = torch.zeros(2, dtype=torch.int32, device="cuda")
    pool, table = make_pool(2, T + 64, page, 7)
    pl = torch.zeros(2, dtype=torch.int32, device="cuda")
    yd = layer.prefill(x, dense, dl, [0, 0])
    yp = layer.prefill_paged(x, pool, table, pl, [0, 0])
    torch.cuda.synchronize()
    assert layer.status() == mla.MLA_OK and pl.tolist() == [T, T]
    assert torch.equal(yp, yd)
    for b in range(2):
        assert torch.equal(logical_rows(pool, table, b, T), dense[b])
        y_ref, _ = O.prefill(O.bf16_to_f64(xb[b]), W)
        assert_close(yp[b].float().cpu().numpy(), y_ref, f"paged prefill {b}")


@pytest.mark.parametrize("page", [64, 128])
def test_paged_chunked_prefill_every_element(layer, page):
    """A 70-token chunk for three sequences holding 150, 0 and 77 cached positions on shuffled
    pages: the cached latents are gathered from their pages and their keys and values rebuilt.
    Every element of the chunk's output and of the grown caches against the oracle, and the
    output against the dense chunked call."""
    W = oracle_weights(0)
    Ls, T, seqs = [150, 0, 77], 70, [40, 41, 42]
    xbs = [synth.hidden_states(0, s, 0, Lb + T) for s, Lb in zip(seqs, Ls)]
    capacity = max(Ls) + T + 10
    pool, table = make_pool(3, capacity, page, 3 + page)
    pl = torch.zeros(3, dtype=torch.int32, device="cuda")
    dense = torch.zeros(3, capacity, 576, dtype=torch.bfloat16, device="cuda")
    dl = torch.zeros(3, dtype=torch.int32, device="cuda")
    for b, (Lb, xb) in enumerate(zip(Ls, xbs)):
        if Lb:
            xp = to_dev(xb[None, :Lb])
            layer.cache_append_paged(xp, pool, table[b:b + 1].contiguous(), pl[b:b + 1], [0])
            layer.cache_append(xp, dense[b:b + 1], dl[b:b + 1], [0])
    x = torch.cat([to_dev(xb[None, Lb:]) for Lb, xb in zip(Ls, xbs)])
    yp = layer.prefill_paged(x, pool, table, pl, Ls)
    yd = layer.prefill(x, dense, dl, Ls)
    torch.cuda.synchronize()
    assert layer.status() == mla.MLA_OK and pl.tolist() == [Lb + T for Lb in Ls]
    assert_close(yp.float().cpu().numpy(), yd.float().cpu().numpy(), f"paged vs dense chunk, page {page}")
    for b, (Lb, xb) in enumerate(zip(Ls, xbs)):
        xf = O.bf16_to_f64(xb)
        cache_ref = O.cache_rows(xf[:Lb], np.arange(Lb), W) if Lb else None
        y_ref, full_ref = O.forward(xf[Lb:], cache_ref, W)
        assert_close(yp[b].float().cpu().numpy(), y_ref, f"paged chunk seq {b} (L={Lb}, page {page})")
        assert_close(logical_rows(pool, table, b, Lb + T).float().cpu().numpy(), full_ref,
                     f"paged chunk cache {b}")


def test_paged_decode_after_paged_prefill_long(layer):
    """A 3000-token prompt prefilled into 128-position pages, then three decode steps, each
    checked against the oracle (the decode shares cut the sequence at positions that are not
    multiples of 64, so first tiles start before their share)."""
    W = oracle_weights(0)
    P, page = 3000, 128
    xb = synth.hidden_states(0, 50, 0, P + 3)
    pool, table = make_pool(1, P + 64, page, 11)
    pl = torch.zeros(1, dtype=torch.int32, device="cuda")
    layer.prefill_paged(to_dev(xb[None, :P]), pool, table, pl, [0])
    xf = O.bf16_to_f64(xb)
    cache_ref = O.cache_rows(xf[:P], np.arange(P), W)
    for step in range(3):
        p = P + step
        y = layer.decode_paged(to_dev(xb[p:p + 1]), pool, table, pl, [p])
        torch.cuda.synchronize()
        assert layer.status() == mla.MLA_OK
        y_ref, cache_ref = O.decode(xf[p], cache_ref, W)
        assert_close(y[0].float().cpu().numpy(), y_ref, f"paged decode step {step}")
    assert_close(logical_rows(pool, table, 0, P + 3).float().cpu().numpy(), cache_ref,
                 "paged long cache")


def test_paged_invalid_page_is_flagged_not_followed(layer):
    """A block-table entry outside the pool, for the page a cache append writes: the row is
    skipped (the pool keeps its NaN fill) and the device status reports it."""
    pool, table = make_pool(1, 128, 64, 5)
    before = pool.clone()
    table[0, 0] = pool.shape[0] + 5
    pl = torch.zeros(1, dtype=torch.int32, device="cuda")
    layer.cache_append_paged(to_dev(synth.hidden_states(0, 1, 0, 8))[None], pool, table, pl, [0])
    torch.cuda.synchronize()
    assert layer.status() == mla.MLA_ERR_STATE
    assert torch.equal(pool.view(torch.int16), before.view(torch.int16))
    assert layer.status() == mla.MLA_OK


def test_paged_descriptor_and_capacity_errors(layer):
    pool, table = make_pool(1, 128, 64, 6)
    x = to_dev(synth.hidden_states(0, 2, 0, 4))[None]
    pl = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = layer.workspace(1, 4)
    bad = mla.paged_cache(pool, table)
    bad.page_size = 48                                  # not a multiple of 64
    with pytest.raises(mla.MlaError) as e:
        mla.mla_cache_append_paged(layer.ctx, x, bad, pl, [0], ws)
    assert e.value.status == mla.MLA_ERR_INVALID_ARG
    with pytest.raises(mla.MlaError) as e:              # 126 + 4 > 2 pages x 64
        mla.mla_cache_append_paged(layer.ctx, x, mla.paged_cache(pool, table), pl, [126], ws)
    assert e.value.status == mla.MLA_ERR_CAPACITY
    torch.cuda.synchronize()
    assert pl.item() == 0
