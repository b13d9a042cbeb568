"""Python binding of the GB300 H2O heavy-hitter KV-cache library (libh2o.so).

Argument marshalling only: every function checks dtypes, devices, shapes and
contiguity, then calls the C-ABI entry point of the same name with raw device
pointers. All work runs in the library's CUDA kernels on the current PyTorch
stream. There is no fallback: if the shared library is missing or CUDA is not
available, the calls raise.

Layouts (see include/h2o.h): a prompt is bf16 [batch, heads, T, d]; a decode
step's q, k_new, v_new are bf16 [batch, heads, d]; outputs are fp32.
"""
from __future__ import annotations

import ctypes
from pathlib import Path

import numpy as np
import torch

__all__ = [
    "H2OError", "H2OContext", "load_library", "h2o_create", "h2o_destroy", "h2o_prefill",
    "h2o_decode_step", "h2o_decode_steps", "h2o_prefill_attention", "h2o_cache_positions", "h2o_last_evicted",
    "h2o_cache_view", "h2o_cache_scales", "h2o_sync_check", "h2o_test_wait_limit", "LIB_PATH",
    "KV_FORMATS", "h2o_reset", "h2o_attention_sync_check", "h2o_attention_test_wait_limit",
    "h2o_test_fail_allocations", "h2o_forget_device_state",
]

LIB_PATH = Path(__file__).resolve().parent / "libh2o.so"

H2O_OK, H2O_EINVAL, H2O_ESTATE, H2O_ENOMEM, H2O_ECUDA, H2O_EDEVICE = 0, -1, -2, -3, -4, -5
_ERR_NAMES = {-1: "EINVAL", -2: "ESTATE", -3: "ENOMEM", -4: "ECUDA", -5: "EDEVICE"}

_lib = None

KV_FORMATS = {"bf16": 0, "fp8": 1}  # H2O_KV_BF16, H2O_KV_FP8


class H2OError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"H2O_{_ERR_NAMES.get(code, code)}: {msg}")
        self.code = code


def load_library() -> ctypes.CDLL:
    """Loads libh2o.so (built in-tree by the package's _build module)."""
    global _lib
    if _lib is not None:
        return _lib
    if not LIB_PATH.exists():
        raise RuntimeError(f"{LIB_PATH} is not built; run h2o_heavy_hitter_gb300._build.build()")
    lib = ctypes.CDLL(str(LIB_PATH))
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(ctypes.c_float)
    I32P = ctypes.POINTER(ctypes.c_int32)
    sig = {
        "h2o_create": (I, [I, I, I, I, I, I, ctypes.POINTER(P)]),
        "h2o_create_ex": (I, [I, I, I, I, I, I, I, ctypes.POINTER(P)]),
        "h2o_cache_scales": (I, [P, I, ctypes.POINTER(P), ctypes.POINTER(P)]),
        "h2o_destroy": (None, [P]),
        "h2o_prefill": (I, [P, I, P, P, P, I, P]),
        "h2o_prefill_ragged": (I, [P, I, P, P, P, I, P, P]),
        "h2o_decode_step": (I, [P, I, P, P, P, P]),
        "h2o_decode_steps": (I, [P, I, I, P, P, P, P, P]),
        "h2o_prefill_attention": (I, [P, P, P, I, I, I, P, P]),
        "h2o_cache_positions": (I, [P, I, I32P]),
        "h2o_last_evicted": (I, [P, I, I32P]),
        "h2o_cache_view": (I, [P, I, ctypes.POINTER(P), ctypes.POINTER(P), ctypes.POINTER(P),
                               ctypes.POINTER(P), ctypes.POINTER(P)]),
        "h2o_cache_dims": (I, [P, ctypes.POINTER(I), ctypes.POINTER(I)]),
        "h2o_sync_check": (I, [P]),
        "h2o_test_wait_limit": (I, [P]),
        "h2o_reset": (I, [P, I]),
        "h2o_attention_sync_check": (I, [P]),
        "h2o_attention_test_wait_limit": (I, [P]),
        "h2o_forget_device_state": (None, []),
        "h2o_test_fail_allocations": (I, [I]),
        "h2o_last_error": (ctypes.c_char_p, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    del F
    _lib = lib
    return lib


def _check(rc: int) -> None:
    if rc != H2O_OK:
        msg = load_library().h2o_last_error().decode(errors="replace")
        raise H2OError(rc, msg)


def _need_cuda():
    if not torch.cuda.is_available():
        raise RuntimeError("the H2O library needs a CUDA device; none is available")
    torch.cuda.init()


def _dev_ptr(t: torch.Tensor, dtype: torch.dtype, shape: tuple, name: str) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"{name} is on {t.device}; the library works on the current device "
                         f"cuda:{torch.cuda.current_device()}")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr() if t.numel() else 0


class H2OContext:
    """Owner of one h2o_ctx handle (cache of `layers` layers)."""

    def __init__(self, handle: int, layers: int, batch: int, heads: int, head_dim: int, h: int,
                 r: int, kv: str = "bf16"):
        self.handle = handle
        self.kv = kv
        self.layers, self.batch, self.heads, self.head_dim = layers, batch, heads, head_dim
        self.h, self.r, self.k = h, r, h + r
        self.rows = batch * heads

    def close(self):
        if self.handle:
            load_library().h2o_destroy(ctypes.c_void_p(self.handle))
            self.handle = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()


H2O_LAYOUT_RING = 0x100


def h2o_create(layers: int, batch: int, heads: int, head_dim: int, h: int, r: int,
               kv: str = "bf16", layout: str = "slots") -> H2OContext:
    """Cache of `layers` layers; kv "bf16" (h2o_create) or "fp8" (E4M3 codes with
    per-token scales, h2o_create_ex); layout "slots" (slot-indexed) or "ring"
    (heavy slots then the recent window as a circular queue, bf16 only)."""
    _need_cuda()
    if kv not in KV_FORMATS:
        raise ValueError(f"kv must be one of {sorted(KV_FORMATS)}")
    if layout not in ("slots", "ring"):
        raise ValueError('layout must be "slots" or "ring"')
    lib = load_library()
    out = ctypes.c_void_p()
    if kv == "bf16" and layout == "slots":
        _check(lib.h2o_create(layers, batch, heads, head_dim, h, r, ctypes.byref(out)))
    else:
        fmt = KV_FORMATS[kv] | (H2O_LAYOUT_RING if layout == "ring" else 0)
        _check(lib.h2o_create_ex(layers, batch, heads, head_dim, h, r, fmt, ctypes.byref(out)))
    ctx = H2OContext(out.value, layers, batch, heads, head_dim, h, r, kv)
    ctx.layout = layout
    return ctx


def h2o_destroy(ctx: H2OContext) -> None:
    ctx.close()


def h2o_prefill(ctx: H2OContext, layer: int, Q, K, V, out=None, lens=None) -> torch.Tensor:
    """Prompt pass of one layer; returns the fp32 attention output [B, H, T, d].

    ``lens``: for a ragged batch, a CUDA int32 tensor [B] of prompt lengths
    (h2o_prefill_ragged); Q, K, V then hold each prompt right-padded to
    T = Q.shape[2] with finite padding, and output rows past a prompt's length
    hold no result."""
    T = Q.shape[2] if Q is not None and Q.dim() == 4 else 0
    shape = (ctx.batch, ctx.heads, T, ctx.head_dim)
    if out is None:
        out = torch.empty(shape, dtype=torch.float32, device=Q.device)
    pq = _dev_ptr(Q, torch.bfloat16, shape, "Q")
    pk = _dev_ptr(K, torch.bfloat16, shape, "K")
    pv = _dev_ptr(V, torch.bfloat16, shape, "V")
    po = _dev_ptr(out, torch.float32, shape, "out")
    lib = load_library()
    if lens is None:
        _check(lib.h2o_prefill(ctypes.c_void_p(ctx.handle), layer, pq, pk, pv, T, po))
    else:
        pl = _dev_ptr(lens, torch.int32, (ctx.batch,), "lens")
        _check(lib.h2o_prefill_ragged(ctypes.c_void_p(ctx.handle), layer, pq, pk, pv, T, pl, po))
    return out


def h2o_reset(ctx: H2OContext, layer: int = -1) -> None:
    """Empties one layer (or every layer with -1) for a new prompt."""
    _check(load_library().h2o_reset(ctypes.c_void_p(ctx.handle), layer))


def h2o_decode_step(ctx: H2OContext, layer: int, q, k_new, v_new, out=None) -> torch.Tensor:
    """One decode step of one layer; returns the fp32 output [B, H, d]."""
    shape = (ctx.batch, ctx.heads, ctx.head_dim)
    if out is None:
        out = torch.empty(shape, dtype=torch.float32, device=q.device)
    pq = _dev_ptr(q, torch.bfloat16, shape, "q")
    pk = _dev_ptr(k_new, torch.bfloat16, shape, "k_new")
    pv = _dev_ptr(v_new, torch.bfloat16, shape, "v_new")
    po = _dev_ptr(out, torch.float32, shape, "out")
    _check(load_library().h2o_decode_step(ctypes.c_void_p(ctx.handle), layer, pq, pk, pv, po))
    return out


def h2o_decode_steps(ctx: H2OContext, layer: int, q, k_new, v_new, out=None,
                     evicted=None) -> torch.Tensor:
    """``S`` decode steps of one layer from inputs [S, B, H, d] known in advance;
    returns the fp32 outputs [S, B, H, d]. ``evicted``: optional CUDA int32
    tensor [S, B * H] receiving each step's evicted position per row."""
    S = q.shape[0]
    shape = (S, ctx.batch, ctx.heads, ctx.head_dim)
    if out is None:
        out = torch.empty(shape, dtype=torch.float32, device=q.device)
    pq = _dev_ptr(q, torch.bfloat16, shape, "q")
    pk = _dev_ptr(k_new, torch.bfloat16, shape, "k_new")
    pv = _dev_ptr(v_new, torch.bfloat16, shape, "v_new")
    po = _dev_ptr(out, torch.float32, shape, "out")
    pe = 0 if evicted is None else _dev_ptr(evicted, torch.int32, (S, ctx.rows), "evicted")
    _check(load_library().h2o_decode_steps(ctypes.c_void_p(ctx.handle), layer, S, pq, pk, pv, po,
                                           pe or None))
    return out


def h2o_prefill_attention(Q, K, V, out=None, score=None):
    """Cache-free causal attention of [rows, T, d] bf16 inputs: (out fp32, column-sum score fp32)."""
    rows, T, d = Q.shape
    if out is None:
        out = torch.empty((rows, T, d), dtype=torch.float32, device=Q.device)
    if score is None:
        score = torch.empty((rows, T), dtype=torch.float32, device=Q.device)
    args = [_dev_ptr(x, torch.bfloat16, (rows, T, d), n) for x, n in ((Q, "Q"), (K, "K"), (V, "V"))]
    po = _dev_ptr(out, torch.float32, (rows, T, d), "out")
    ps = _dev_ptr(score, torch.float32, (rows, T), "score")
    _check(load_library().h2o_prefill_attention(*args, rows, T, d, po, ps))
    return out, score


def h2o_cache_positions(ctx: H2OContext, layer: int) -> np.ndarray:
    """Positions held by every slot, int32 [rows, k] (-1 = empty)."""
    buf = np.empty((ctx.rows, ctx.k), dtype=np.int32)
    _check(load_library().h2o_cache_positions(
        ctypes.c_void_p(ctx.handle), layer, buf.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))))
    return buf


def h2o_last_evicted(ctx: H2OContext, layer: int) -> np.ndarray:
    """Position evicted by the last decode step of each row, int32 [rows] (-1 = none)."""
    buf = np.empty((ctx.rows,), dtype=np.int32)
    _check(load_library().h2o_last_evicted(
        ctypes.c_void_p(ctx.handle), layer, buf.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))))
    return buf


class _DeviceArray:
    """Exposes a library-owned device buffer through __cuda_array_interface__."""

    def __init__(self, ptr: int, shape: tuple, typestr: str):
        self.__cuda_array_interface__ = {"data": (ptr, False), "shape": shape,
                                         "typestr": typestr, "version": 3, "strides": None}


def h2o_cache_view(ctx: H2OContext, layer: int) -> dict:
    """Zero-copy torch views of one layer's cache arrays (library-owned memory).

    K and V are bf16 tensors, or uint8 E4M3 codes for an "fp8" cache (its
    scales: h2o_cache_scales)."""
    ptrs = [ctypes.c_void_p() for _ in range(5)]
    _check(load_library().h2o_cache_view(ctypes.c_void_p(ctx.handle), layer,
                                         *[ctypes.byref(p) for p in ptrs]))
    R, k, d = ctx.rows, ctx.k, ctx.head_dim
    dev = torch.device("cuda", torch.cuda.current_device())
    mk = lambda p, shape, ts: torch.as_tensor(_DeviceArray(p.value, shape, ts), device=dev)
    if ctx.kv == "fp8":
        kv_k, kv_v = mk(ptrs[0], (R, k, d), "|u1"), mk(ptrs[1], (R, k, d), "|u1")
    else:
        kv_k = mk(ptrs[0], (R, k, d), "<i2").view(torch.bfloat16)
        kv_v = mk(ptrs[1], (R, k, d), "<i2").view(torch.bfloat16)
    return {
        "K": kv_k,
        "V": kv_v,
        "score": mk(ptrs[2], (R, k), "<f4"),
        "pos": mk(ptrs[3], (R, k), "<i4"),
        "meta": mk(ptrs[4], (R, 4), "<i4"),
    }


def h2o_cache_scales(ctx: H2OContext, layer: int) -> dict:
    """Zero-copy views of an "fp8" cache's per-slot scales: {"K": fp32 [rows, k],
    "V": fp32 [rows, k]}."""
    ptrs = [ctypes.c_void_p() for _ in range(2)]
    _check(load_library().h2o_cache_scales(ctypes.c_void_p(ctx.handle), layer,
                                           *[ctypes.byref(p) for p in ptrs]))
    dev = torch.device("cuda", torch.cuda.current_device())
    mk = lambda p: torch.as_tensor(_DeviceArray(p.value, (ctx.rows, ctx.k), "<f4"), device=dev)
    return {"K": mk(ptrs[0]), "V": mk(ptrs[1])}


def h2o_test_wait_limit(ctx: H2OContext) -> None:
    """Enqueues a kernel whose bounded wait runs out (the failure path on demand);
    the next h2o_sync_check raises H2O_EDEVICE."""
    _check(load_library().h2o_test_wait_limit(ctypes.c_void_p(ctx.handle)))


def h2o_sync_check(ctx: H2OContext) -> None:
    _check(load_library().h2o_sync_check(ctypes.c_void_p(ctx.handle)))


def _stream_ptr(stream) -> int | None:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream or None


def h2o_attention_sync_check(stream=None) -> None:
    """Synchronises ``stream`` (default: the current stream) and raises
    H2O_EDEVICE if a cache-free prefill call reported a device error."""
    _check(load_library().h2o_attention_sync_check(_stream_ptr(stream)))


def h2o_attention_test_wait_limit(stream=None) -> None:
    """Enqueues a kernel whose bounded wait runs out against the library-level
    error word; the next h2o_attention_sync_check raises H2O_EDEVICE."""
    _check(load_library().h2o_attention_test_wait_limit(_stream_ptr(stream)))


def h2o_test_fail_allocations(n: int) -> None:
    """Makes the library's next ``n`` device allocations fail (0 ends it)."""
    _check(load_library().h2o_test_fail_allocations(n))


def h2o_forget_device_state() -> None:
    """Drops the library's cached per-device state (after a device reset)."""
    load_library().h2o_forget_device_state()
