"""Thin ctypes binding of libmla's C ABI (include/mla.h), with the same function names.

Only argument marshalling happens here: torch tensors are passed as raw device pointers and the
current CUDA stream as a cudaStream_t.  Every step of the layer runs in libmla's kernels; if the
library is not built this module raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libmla.so")

MLA_OK, MLA_ERR_INVALID_ARG, MLA_ERR_SHAPE, MLA_ERR_UNSUPPORTED = 0, 1, 2, 3
MLA_ERR_CAPACITY, MLA_ERR_CUDA, MLA_ERR_TIMEOUT, MLA_ERR_STATE = 4, 5, 6, 7
MLA_W_Q_A, MLA_W_Q_B, MLA_W_KV_A, MLA_W_KV_B, MLA_W_O = 0, 1, 2, 3, 4
MLA_NORM_Q, MLA_NORM_KV, MLA_NORM_INPUT = 0, 1, 2
MLA_ROPE_ADJACENT, MLA_ROPE_HALF = 0, 1
MLA_ROPE_PLAIN, MLA_ROPE_YARN = 0, 1
WEIGHT_IDS = {"q_a": MLA_W_Q_A, "q_b": MLA_W_Q_B, "kv_a": MLA_W_KV_A, "kv_b": MLA_W_KV_B,
              "o": MLA_W_O}
NORM_IDS = {"q_norm": MLA_NORM_Q, "kv_norm": MLA_NORM_KV, "input_norm": MLA_NORM_INPUT}


class mla_config(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int), ("q_lora", ctypes.c_int), ("kv_lora", ctypes.c_int),
                ("heads", ctypes.c_int), ("nope", ctypes.c_int), ("rope", ctypes.c_int),
                ("vdim", ctypes.c_int), ("eps", ctypes.c_float), ("rope_theta", ctypes.c_float),
                ("softmax_scale", ctypes.c_float), ("max_positions", ctypes.c_int),
                ("rope_pairing", ctypes.c_int), ("rope_scaling", ctypes.c_int),
                ("yarn_factor", ctypes.c_float), ("yarn_original_max_positions", ctypes.c_int),
                ("yarn_beta_fast", ctypes.c_float), ("yarn_beta_slow", ctypes.c_float),
                ("yarn_mscale", ctypes.c_float), ("yarn_mscale_all_dim", ctypes.c_float),
                ("block", ctypes.c_int), ("fp8_activations", ctypes.c_int)]


class mla_paged_cache(ctypes.Structure):
    _fields_ = [("pool", ctypes.c_void_p), ("num_pages", ctypes.c_int),
                ("page_size", ctypes.c_int), ("block_table", ctypes.c_void_p),
                ("max_pages", ctypes.c_int)]


_P = ctypes.c_void_p
_I = ctypes.c_int
_PC = ctypes.POINTER(mla_paged_cache)
_SIGS = {
    "mla_default_config": (None, [ctypes.POINTER(mla_config)]),
    "mla_create": (_I, [ctypes.POINTER(mla_config), ctypes.POINTER(_P)]),
    "mla_destroy": (None, [_P]),
    "mla_upload_weights": (_I, [_P, _I, _P, _P, _I, _I]),
    "mla_upload_norm": (_I, [_P, _I, _P, _I]),
    "mla_workspace_bytes": (ctypes.c_size_t, [_P, _I, _I]),
    "mla_workspace_bytes_len": (ctypes.c_size_t, [_P, _I, _I, _I]),
    "mla_cache_append": (_I, [_P, _P, _I, _I, _P, _I, _P, _P, _P, ctypes.c_size_t, _P]),
    "mla_prefill": (_I, [_P, _P, _I, _I, _P, _I, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "mla_decode": (_I, [_P, _P, _I, _P, _I, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "mla_decode_host_workspace_bytes": (ctypes.c_size_t, [_P, _I]),
    "mla_decode_host": (_I, [_P, _P, _I, _P, _I, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "mla_cache_append_paged": (_I, [_P, _P, _I, _I, _PC, _P, _P, _P, ctypes.c_size_t, _P]),
    "mla_prefill_paged": (_I, [_P, _P, _I, _I, _PC, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "mla_decode_paged": (_I, [_P, _P, _I, _PC, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "mla_dequant_weight": (_I, [_P, _I, _P, _P]),
    "mla_get_device_status": (_I, [_P, _P]),
    "mla_status_string": (ctypes.c_char_p, [_I]),
    "mla_decode_noalloc": (_I, [_P, _P, _I, _P, _I, _P, _P, _P, _P]),
    "mla_set_profiling": (_I, [_P, _I]),
    "mla_selftest_wait_timeout": (_I, [_P, ctypes.c_ulonglong, _P]),
    "mla_last_launches": (_I, [_P, _I, ctypes.POINTER(ctypes.c_char_p),
                               ctypes.POINTER(ctypes.c_float)]),
}

_lib = None


def load(path: str | None = None) -> ctypes.CDLL:
    """Loads libmla.so (once) and declares every exported signature."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libmla.so is not built ({p}); run __graft_entry__.build()")
    lib = ctypes.CDLL(p)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib


class MlaError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {mla_status_string(status)}")
        self.status = status


def _check(status: int, what: str) -> None:
    if status != MLA_OK:
        raise MlaError(status, what)


def _ptr(t: torch.Tensor | None) -> int | None:
    if t is None:
        return None
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("expected a contiguous CUDA tensor")
    return t.data_ptr()


def _host_ptr(t: torch.Tensor) -> int:
    if t.is_cuda or not t.is_contiguous() or t.dtype != torch.bfloat16:
        raise ValueError("expected a contiguous bf16 host tensor")
    return t.data_ptr()


def _host_i32(t) -> ctypes.Array:
    vals = [int(v) for v in (t.tolist() if hasattr(t, "tolist") else t)]
    return (ctypes.c_int * max(1, len(vals)))(*vals)


def _stream(stream: torch.cuda.Stream | None) -> int:
    return (stream or torch.cuda.current_stream()).cuda_stream


# ---- same-name wrappers of the C functions ------------------------------------------------
def mla_default_config() -> mla_config:
    cfg = mla_config()
    load().mla_default_config(ctypes.byref(cfg))
    return cfg


def mla_create(cfg: mla_config) -> int:
    ctx = _P()
    _check(load().mla_create(ctypes.byref(cfg), ctypes.byref(ctx)), "mla_create")
    return ctx.value


def mla_destroy(ctx: int) -> None:
    load().mla_destroy(ctx)


def mla_upload_weights(ctx: int, which: int, e4m3: torch.Tensor, scale: torch.Tensor) -> None:
    assert e4m3.dtype == torch.uint8 and scale.dtype == torch.float32
    _check(load().mla_upload_weights(ctx, which, _ptr(e4m3), _ptr(scale), e4m3.shape[0],
                                     e4m3.shape[1]), "mla_upload_weights")


def mla_upload_norm(ctx: int, which: int, gain_bf16: torch.Tensor) -> None:
    assert gain_bf16.dtype == torch.bfloat16
    _check(load().mla_upload_norm(ctx, which, _ptr(gain_bf16), gain_bf16.numel()),
           "mla_upload_norm")


def mla_workspace_bytes(ctx: int, B: int, T: int) -> int:
    return int(load().mla_workspace_bytes(ctx, B, T))


def mla_workspace_bytes_len(ctx: int, B: int, T: int, max_len: int) -> int:
    return int(load().mla_workspace_bytes_len(ctx, B, T, max_len))


def mla_cache_append(ctx, x, cache, seq_lens_dev, seq_lens_host, ws, stream=None) -> None:
    B, T = x.shape[0], x.shape[1]
    _check(load().mla_cache_append(ctx, _ptr(x), B, T, _ptr(cache), cache.shape[1],
                                   _ptr(seq_lens_dev), _host_i32(seq_lens_host), _ptr(ws),
                                   ws.numel() * ws.element_size(), _stream(stream)),
           "mla_cache_append")


def mla_prefill(ctx, x, cache, seq_lens_dev, seq_lens_host, out, ws, stream=None) -> None:
    B, T = x.shape[0], x.shape[1]
    _check(load().mla_prefill(ctx, _ptr(x), B, T, _ptr(cache), cache.shape[1],
                              _ptr(seq_lens_dev), _host_i32(seq_lens_host), _ptr(out), _ptr(ws),
                              ws.numel() * ws.element_size(), _stream(stream)), "mla_prefill")


def mla_decode(ctx, x, cache, seq_lens_dev, seq_lens_host, out, ws, stream=None) -> None:
    B = x.shape[0]
    _check(load().mla_decode(ctx, _ptr(x), B, _ptr(cache), cache.shape[1], _ptr(seq_lens_dev),
                             _host_i32(seq_lens_host), _ptr(out), _ptr(ws),
                             ws.numel() * ws.element_size(), _stream(stream)), "mla_decode")


def mla_decode_host_workspace_bytes(ctx: int, B: int) -> int:
    return int(load().mla_decode_host_workspace_bytes(ctx, B))


def mla_decode_host(ctx, x_host, cache, seq_lens_dev, seq_lens_host, out_host, ws,
                    stream=None) -> None:
    """mla_decode with x_host and out_host [B, 7168] bf16 in host memory (page-locked for the
    fast path); the copies are enqueued on the stream with the step."""
    B = x_host.shape[0]
    _check(load().mla_decode_host(ctx, _host_ptr(x_host), B, _ptr(cache), cache.shape[1],
                                  _ptr(seq_lens_dev), _host_i32(seq_lens_host),
                                  _host_ptr(out_host),
                                  _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "mla_decode_host")


def mla_decode_noalloc(ctx, x, cache, seq_lens_dev, seq_lens_host, out, stream=None) -> None:
    """mla_decode without a workspace: scratch comes from a static array in the library."""
    B = x.shape[0]
    _check(load().mla_decode_noalloc(ctx, _ptr(x), B, _ptr(cache), cache.shape[1],
                                     _ptr(seq_lens_dev), _host_i32(seq_lens_host), _ptr(out),
                                     _stream(stream)), "mla_decode_noalloc")


def paged_cache(pool: torch.Tensor, block_table: torch.Tensor) -> mla_paged_cache:
    """Descriptor of a paged latent cache: pool bf16 [num_pages, page_size, 576] and
    block_table int32 [B, max_pages] (both CUDA tensors, kept alive by the caller)."""
    assert pool.dtype == torch.bfloat16 and pool.dim() == 3 and pool.shape[2] == 576
    assert block_table.dtype == torch.int32 and block_table.dim() == 2
    return mla_paged_cache(_ptr(pool), pool.shape[0], pool.shape[1], _ptr(block_table),
                           block_table.shape[1])


def mla_cache_append_paged(ctx, x, cache: mla_paged_cache, seq_lens_dev, seq_lens_host, ws,
                           stream=None) -> None:
    B, T = x.shape[0], x.shape[1]
    _check(load().mla_cache_append_paged(ctx, _ptr(x), B, T, ctypes.byref(cache),
                                         _ptr(seq_lens_dev), _host_i32(seq_lens_host), _ptr(ws),
                                         ws.numel() * ws.element_size(), _stream(stream)),
           "mla_cache_append_paged")


def mla_prefill_paged(ctx, x, cache: mla_paged_cache, seq_lens_dev, seq_lens_host, out, ws,
                      stream=None) -> None:
    B, T = x.shape[0], x.shape[1]
    _check(load().mla_prefill_paged(ctx, _ptr(x), B, T, ctypes.byref(cache), _ptr(seq_lens_dev),
                                    _host_i32(seq_lens_host), _ptr(out), _ptr(ws),
                                    ws.numel() * ws.element_size(), _stream(stream)),
           "mla_prefill_paged")


def mla_decode_paged(ctx, x, cache: mla_paged_cache, seq_lens_dev, seq_lens_host, out, ws,
                     stream=None) -> None:
    B = x.shape[0]
    _check(load().mla_decode_paged(ctx, _ptr(x), B, ctypes.byref(cache), _ptr(seq_lens_dev),
                                   _host_i32(seq_lens_host), _ptr(out), _ptr(ws),
                                   ws.numel() * ws.element_size(), _stream(stream)),
           "mla_decode_paged")


def mla_dequant_weight(ctx: int, which: int, out: torch.Tensor, stream=None) -> None:
    _check(load().mla_dequant_weight(ctx, which, _ptr(out), _stream(stream)),
           "mla_dequant_weight")


def mla_get_device_status(ctx: int, stream=None) -> int:
    return int(load().mla_get_device_status(ctx, _stream(stream)))


def mla_set_profiling(ctx: int, on: bool) -> None:
    _check(load().mla_set_profiling(ctx, int(on)), "mla_set_profiling")


def mla_last_launches(ctx: int, max_launches: int = 32):
    """[(kernel name, device ms or -1)] of the most recent token call."""
    names = (ctypes.c_char_p * max_launches)()
    ms = (ctypes.c_float * max_launches)()
    n = load().mla_last_launches(ctx, max_launches, names, ms)
    return [(names[i].decode(), float(ms[i])) for i in range(min(n, max_launches))]


def mla_selftest_wait_timeout(ctx: int, limit_ns: int, stream=None) -> None:
    """Enqueues the bounded-wait self-test; mla_get_device_status then reports the timeout."""
    _check(load().mla_selftest_wait_timeout(ctx, limit_ns, _stream(stream)),
           "mla_selftest_wait_timeout")


def mla_status_string(status: int) -> str:
    return load().mla_status_string(status).decode()


# ---- convenience owner of one layer's device state ------------------------------------------
class MlaLayer:
    """Holds one context, the device copies of the quantised weights and gains, and a
    workspace.  Methods take and return torch CUDA tensors; all compute is in libmla."""

    def __init__(self, weights: dict, gains: dict, device="cuda", **cfg_overrides):
        cfg = mla_default_config()
        for k, v in cfg_overrides.items():
            setattr(cfg, k, v)
        self.cfg = cfg
        self.ctx = mla_create(cfg)
        self.w = {}
        for name, (codes, scales) in weights.items():
            q = torch.as_tensor(codes).to(device).contiguous()
            s = torch.as_tensor(scales).to(device).contiguous()
            self.w[name] = (q, s)
            mla_upload_weights(self.ctx, WEIGHT_IDS[name], q, s)
        self.g = {}
        for name, bits in gains.items():
            g = torch.as_tensor(bits.view("int16") if hasattr(bits, "view") else bits)
            g = g.view(torch.bfloat16).to(device).contiguous()
            self.g[name] = g
            mla_upload_norm(self.ctx, NORM_IDS[name], g)
        self.ws = torch.empty(0, dtype=torch.uint8, device=device)

    def workspace(self, B: int, T: int, max_len: int | None = None) -> torch.Tensor:
        need = mla_workspace_bytes_len(self.ctx, B, T, max(T, max_len or T))
        if self.ws.numel() < need:
            self.ws = torch.empty(need, dtype=torch.uint8, device=self.ws.device)
        return self.ws

    def prefill(self, x, cache, seq_lens_dev, seq_lens_host, out=None):
        out = torch.empty_like(x) if out is None else out
        T = x.shape[1]
        mla_prefill(self.ctx, x, cache, seq_lens_dev, seq_lens_host, out,
                    self.workspace(x.shape[0], T, max(seq_lens_host) + T))
        return out

    def decode(self, x, cache, seq_lens_dev, seq_lens_host, out=None):
        out = torch.empty_like(x) if out is None else out
        mla_decode(self.ctx, x, cache, seq_lens_dev, seq_lens_host, out,
                   self.workspace(x.shape[0], 1))
        return out

    def workspace_host(self, B: int) -> torch.Tensor:
        need = mla_decode_host_workspace_bytes(self.ctx, B)
        if self.ws.numel() < need:
            self.ws = torch.empty(need, dtype=torch.uint8, device=self.ws.device)
        return self.ws

    def decode_host(self, x_host, cache, seq_lens_dev, seq_lens_host, out_host=None, stream=None):
        """One decode step from and to host memory; synchronise `stream` before reading the
        result."""
        out_host = torch.empty_like(x_host) if out_host is None else out_host
        mla_decode_host(self.ctx, x_host, cache, seq_lens_dev, seq_lens_host, out_host,
                        self.workspace_host(x_host.shape[0]), stream=stream)
        return out_host

    def cache_append(self, x, cache, seq_lens_dev, seq_lens_host):
        mla_cache_append(self.ctx, x, cache, seq_lens_dev, seq_lens_host,
                         self.workspace(x.shape[0], x.shape[1]))

    def prefill_paged(self, x, pool, block_table, seq_lens_dev, seq_lens_host, out=None):
        out = torch.empty_like(x) if out is None else out
        T = x.shape[1]
        mla_prefill_paged(self.ctx, x, paged_cache(pool, block_table), seq_lens_dev,
                          seq_lens_host, out,
                          self.workspace(x.shape[0], T, max(seq_lens_host) + T))
        return out

    def decode_paged(self, x, pool, block_table, seq_lens_dev, seq_lens_host, out=None):
        out = torch.empty_like(x) if out is None else out
        mla_decode_paged(self.ctx, x, paged_cache(pool, block_table), seq_lens_dev,
                         seq_lens_host, out, self.workspace(x.shape[0], 1))
        return out

    def cache_append_paged(self, x, pool, block_table, seq_lens_dev, seq_lens_host):
        mla_cache_append_paged(self.ctx, x, paged_cache(pool, block_table), seq_lens_dev,
                               seq_lens_host, self.workspace(x.shape[0], x.shape[1]))

    def dequant(self, name: str) -> torch.Tensor:
        q, _ = self.w[name]
        out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
        mla_dequant_weight(self.ctx, WEIGHT_IDS[name], out)
        return out

    def status(self) -> int:
        return mla_get_device_status(self.ctx)

    def close(self):
        if self.ctx:
            mla_destroy(self.ctx)
            self.ctx = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
