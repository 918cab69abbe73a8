"""The C ABI without a GPU: the library loads, exports every function include/mla.h declares,
and the host-only entry points answer (no compute call is made)."""
import ctypes
import os
import re

import pytest

from head_latent_attention_mla_gb300 import mla

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "mla.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(mla.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    return mla.load()


def test_exports_every_declared_function(lib):
    names = declared_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n
        assert n in mla._SIGS, f"binding lacks {n}"


def test_status_strings(lib):
    for code in range(8):
        s = mla.mla_status_string(code)
        assert s.startswith("MLA_")
    assert mla.mla_status_string(99) == "MLA_ERR_UNKNOWN"


def test_default_config_is_kimi_k2(lib):
    c = mla.mla_default_config()
    assert (c.hidden, c.q_lora, c.kv_lora, c.heads, c.nope, c.rope, c.vdim) == \
        (7168, 1536, 512, 64, 128, 64, 128)
    assert abs(c.softmax_scale - 192 ** -0.5) < 1e-7 and c.rope_theta == 50000.0
    assert c.max_positions == 131073 and c.rope_pairing == mla.MLA_ROPE_ADJACENT
    assert c.rope_scaling == mla.MLA_ROPE_PLAIN          # YaRN is off unless asked for
    assert (c.yarn_factor, c.yarn_original_max_positions, c.yarn_beta_fast, c.yarn_beta_slow,
            c.yarn_mscale, c.yarn_mscale_all_dim) == (32.0, 4096, 1.0, 1.0, 1.0, 1.0)
    assert c.block == 0                                  # the layer alone unless asked for


def test_host_argument_checks(lib):
    c = mla.mla_default_config()
    c.heads = 32
    ctx = ctypes.c_void_p()
    assert lib.mla_create(ctypes.byref(c), ctypes.byref(ctx)) == mla.MLA_ERR_UNSUPPORTED
    assert ctx.value is None
    assert lib.mla_create(None, ctypes.byref(ctx)) == mla.MLA_ERR_INVALID_ARG
    c = mla.mla_default_config()
    c.rope_pairing = 7
    assert lib.mla_create(ctypes.byref(c), ctypes.byref(ctx)) == mla.MLA_ERR_INVALID_ARG
    c = mla.mla_default_config()
    c.rope_scaling = 5
    assert lib.mla_create(ctypes.byref(c), ctypes.byref(ctx)) == mla.MLA_ERR_INVALID_ARG
    c = mla.mla_default_config()
    c.rope_scaling, c.yarn_factor = mla.MLA_ROPE_YARN, 0.5
    assert lib.mla_create(ctypes.byref(c), ctypes.byref(ctx)) == mla.MLA_ERR_INVALID_ARG
    c = mla.mla_default_config()
    c.block = 2
    assert lib.mla_create(ctypes.byref(c), ctypes.byref(ctx)) == mla.MLA_ERR_INVALID_ARG
    assert lib.mla_workspace_bytes(None, 1, 1) == 0
    assert lib.mla_workspace_bytes_len(None, 1, 4, 8) == 0
    assert lib.mla_prefill(None, None, 1, 1, None, 1, None, None, None, None, 0, None) == \
        mla.MLA_ERR_INVALID_ARG
    assert lib.mla_decode(None, None, 1, None, 1, None, None, None, None, 0, None) == \
        mla.MLA_ERR_INVALID_ARG
    lib.mla_destroy(None)
