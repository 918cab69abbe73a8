"""The FP8-activation option (mla_config.fp8_activations = 1; "linear" excerpt's
quantization_config, activation_scheme dynamic): projections of more than 64 token rows take
one e4m3 term per activation with one scale per (token, 128-wide group).

This path is lossy by design (e4m3 keeps 3 mantissa bits, a relative rounding error of up to
2^-4 per activation), so it is not held to the layer's bar (relative Frobenius 1e-2, max-abs
5e-2); every case records its error against the fp64 oracle in the margins summary and must
stay within FP8_REL / FP8_ABS, the measured errors with head-room.  The five workloads: prefill
T=16 (no projection takes the option: unchanged), decode at p=1000 over a cache prefilled with
the option, prefill T=4096 (sampled rows), ragged decode B=64 and long decode B=8 x 131,072
over caches appended with it (sampled sequences)."""
import numpy as np
import pytest
import torch

from head_latent_attention_mla_gb300 import mla, synth
from oracle import mla_oracle as O
from tests.mla_cases import (MARGINS, build_caches_gpu, errors, oracle_cache, oracle_rows,
                             oracle_weights, to_dev, weights_and_gains)

pytestmark = pytest.mark.gpu
FP8_REL, FP8_ABS = 0.1, 0.3     # measured at most 5.9e-2 and 1.95e-1


@pytest.fixture(scope="module")
def f8():
    wq, g = weights_and_gains(0)
    L = mla.MlaLayer(wq, g, fp8_activations=1)
    yield L
    L.close()


def record(got, ref, what):
    rel, mx = errors(got, ref)
    MARGINS.append(("fp8_activations", what, rel, mx))
    assert rel <= FP8_REL and mx <= FP8_ABS, f"{what}: rel_fro={rel:.3e} max_abs={mx:.3e}"
    return rel, mx


def test_fp8_prefill_t16_unchanged(f8):
    W = oracle_weights(0)
    xb = synth.hidden_states(0, 0, 0, 16)
    cache = torch.zeros(1, 16, 576, dtype=torch.bfloat16, device="cuda")
    lens = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = f8.prefill(to_dev(xb[None]), cache, lens, [0])
    torch.cuda.synchronize()
    y_ref, _ = O.prefill(O.bf16_to_f64(xb), W)
    rel, _ = record(y[0].float().cpu().numpy(), y_ref, "fp8 config 1 prefill T=16")
    assert rel <= 1e-2   # T = 16 takes no FP8-activation projection


def test_fp8_decode_p1000(f8):
    W = oracle_weights(0)
    p = 1000
    xb = synth.hidden_states(0, 0, 0, p + 1)
    cache = torch.zeros(1, p + 1, 576, dtype=torch.bfloat16, device="cuda")
    lens = torch.zeros(1, dtype=torch.int32, device="cuda")
    f8.prefill(to_dev(xb[None, :p]), cache, lens, [0])
    yd = f8.decode(to_dev(xb[p:p + 1]), cache, lens, [p])
    torch.cuda.synchronize()
    assert f8.status() == mla.MLA_OK
    xf = O.bf16_to_f64(xb)
    y_ref, full = O.decode(xf[p], O.cache_rows(xf[:p], np.arange(p), W), W)
    record(yd[0].float().cpu().numpy(), y_ref, "fp8 config 2 decode p=1000")
    record(cache[0].float().cpu().numpy(), full, "fp8 config 2 cache")


def test_fp8_prefill_t4096_sampled(f8):
    W = oracle_weights(0)
    T = 4096
    xb = synth.hidden_states(0, 0, 0, T)
    cache = torch.zeros(1, T, 576, dtype=torch.bfloat16, device="cuda")
    lens = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = f8.prefill(to_dev(xb[None]), cache, lens, [0])
    torch.cuda.synchronize()
    assert f8.status() == mla.MLA_OK
    xf = O.bf16_to_f64(xb)
    cache_ref = O.cache_rows(xf, np.arange(T), W)
    record(cache[0].float().cpu().numpy(), cache_ref, "fp8 config 3 cache")
    rows = np.unique(np.concatenate([[0, 1, 127, 128, 2048, 4095],
                                     np.random.default_rng(41).choice(T, 58, replace=False)]))
    record(y[0].float().cpu().numpy()[rows], oracle_rows(xf, rows, cache_ref, W),
           "fp8 config 3 prefill T=4096 rows")


def test_fp8_chunked_prefill(f8):
    W = oracle_weights(0)
    L, T = 300, 130
    xb = synth.hidden_states(0, 9, 0, L + T)
    cache = torch.zeros(1, L + T, 576, dtype=torch.bfloat16, device="cuda")
    lens = torch.zeros(1, dtype=torch.int32, device="cuda")
    f8.prefill(to_dev(xb[None, :L]), cache, lens, [0])
    y = f8.prefill(to_dev(xb[None, L:]), cache, lens, [L])
    torch.cuda.synchronize()
    assert f8.status() == mla.MLA_OK
    xf = O.bf16_to_f64(xb)
    y_ref, _ = O.forward(xf[L:], O.cache_rows(xf[:L], np.arange(L), W), W)
    record(y[0].float().cpu().numpy(), y_ref, "fp8 chunk L=300 T=130")


def test_fp8_ragged_b64_sampled(f8):
    W = oracle_weights(0)
    lengths = synth.ragged_lengths(0, 64, 512, 8192).tolist()
    cache, lens = build_caches_gpu(f8, 0, lengths, max(lengths) + 1)
    xb = np.stack([synth.hidden_states(0, b, lengths[b], 1)[0] for b in range(64)])
    yd = f8.decode(to_dev(xb), cache, lens, lengths).float().cpu().numpy()
    torch.cuda.synchronize()
    assert f8.status() == mla.MLA_OK
    order = np.argsort(lengths)
    for b in [int(order[i]) for i in (0, 21, 42, 63)]:
        y_ref, _ = O.decode(O.bf16_to_f64(xb[b]), oracle_cache(0, b, lengths[b], W), W)
        record(yd[b], y_ref, f"fp8 config 4 ragged seq {b} (len {lengths[b]})")


def test_fp8_long_b8_sampled(f8):
    W = oracle_weights(0)
    L = 131072
    cache, lens = build_caches_gpu(f8, 0, [L] * 8, L + 1)
    xb = np.stack([synth.hidden_states(0, b, L, 1)[0] for b in range(8)])
    yd = f8.decode(to_dev(xb), cache, lens, [L] * 8).float().cpu().numpy()
    torch.cuda.synchronize()
    assert f8.status() == mla.MLA_OK
    for b in (0, 7):
        y_ref, _ = O.decode(O.bf16_to_f64(xb[b]), oracle_cache(0, b, L, W), W)
        record(yd[b], y_ref, f"fp8 config 5 long seq {b}")
