"""Python binding of libattn.so — exact attention forward with the online softmax on GB300.

The names mirror the C ABI in ``include/attn.h``; this module only marshals arguments
(torch tensors to device pointers, the current torch stream to ``cudaStream_t``). Every step
of the computation runs in the library's CUDA kernels. There is no CPU or PyTorch fallback:
if the library has not been built, importing works but every call raises
:class:`AttnLibraryMissing`.

    import torch, online_softmax_flashattention_gb300 as fa
    o = fa.attn_fwd(q, k, v, causal=True)        # q, k, v: cuda [B, H, N, 64], same dtype

Build with ``python -m online_softmax_flashattention_gb300.build`` (or
``__graft_entry__.build()``).
"""

from __future__ import annotations

import contextlib
import ctypes
import os
import threading

import torch

__all__ = [
    "ATTN_F32", "ATTN_BF16", "ATTN_F16", "AttnError", "AttnLibraryMissing", "library_path",
    "attn_fwd", "attn_fwd_materialized", "attn_materialized_workspace_bytes", "attn_device_status",
    "attn_status_string", "attn_abi_version", "raw", "attn_fwd_materialized_noalloc",
    "ATTN_NOALLOC_MAX_N", "attn_fwd_lse", "attn_bwd", "attn_fwd_kvcache", "attn_kvcache_workspace_bytes",
    "ATTN_KV_MAX_SPLITS", "attn_selftest_wait_timeout", "attn_plan_launch_order", "attn_probe_fp32_fma",
    "attn_probe_sfu_ex2",
]

ATTN_F32, ATTN_BF16, ATTN_F16 = 0, 1, 2
STATUS = {0: "ATTN_OK", 1: "ATTN_ERR_INVALID_ARG", 2: "ATTN_ERR_UNSUPPORTED", 3: "ATTN_ERR_ALIGN",
          4: "ATTN_ERR_ALIAS", 5: "ATTN_ERR_DEVICE", 6: "ATTN_ERR_LAUNCH", 7: "ATTN_ERR_TIMEOUT",
          8: "ATTN_ERR_WORKSPACE"}
_DTYPES = {torch.float32: ATTN_F32, torch.bfloat16: ATTN_BF16, torch.float16: ATTN_F16}

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "_lib", "libattn.so")
_lock = threading.Lock()
_lib = None


class AttnLibraryMissing(RuntimeError):
    """libattn.so has not been built in this checkout."""


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} ({attn_status_string(status)})")


def library_path() -> str:
    return _LIB_PATH


def raw():
    """The loaded ctypes library, with argument types declared (for C-ABI level tests)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise AttnLibraryMissing(
                    f"{_LIB_PATH} is missing: build it with `python -m online_softmax_flashattention_gb300.build`")
            lib = ctypes.CDLL(_LIB_PATH)
            vp, i64, ci, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
            lib.attn_fwd.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, ci, ci, vp]
            lib.attn_fwd.restype = ci
            lib.attn_fwd_lse.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, ci, ci, vp]
            lib.attn_fwd_lse.restype = ci
            lib.attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, ci, ci, vp]
            lib.attn_bwd.restype = ci
            lib.attn_fwd_kvcache.argtypes = [vp, vp, vp, vp, vp, vp, sz, i64, i64, i64, i64, i64, ci, ci, ci, vp]
            lib.attn_fwd_kvcache.restype = ci
            lib.attn_kvcache_workspace_bytes.argtypes = [i64, i64, i64, i64, i64, ci, ci]
            lib.attn_kvcache_workspace_bytes.restype = sz
            lib.attn_fwd_materialized.argtypes = [vp, vp, vp, vp, vp, sz, i64, i64, i64, i64, ci, ci, vp]
            lib.attn_fwd_materialized.restype = ci
            lib.attn_materialized_workspace_bytes.argtypes = [i64, i64, i64]
            lib.attn_materialized_workspace_bytes.restype = sz
            lib.attn_selftest_wait_timeout.argtypes = [ctypes.c_uint64, vp]
            lib.attn_selftest_wait_timeout.restype = ci
            lib.attn_device_status.argtypes = [vp, ci]
            lib.attn_device_status.restype = ci
            lib.attn_status_string.argtypes = [ci]
            lib.attn_status_string.restype = ctypes.c_char_p
            lib.attn_abi_version.argtypes = []
            lib.attn_abi_version.restype = ci
            lib.attn_plan_launch_order.argtypes = [vp, i64, ctypes.c_int32, ctypes.c_int32, vp]
            lib.attn_plan_launch_order.restype = ci
            lib.attn_probe_fp32_fma.argtypes = [vp, i64, i64, ctypes.POINTER(ctypes.c_double), vp]
            lib.attn_probe_fp32_fma.restype = ci
            lib.attn_probe_sfu_ex2.argtypes = [vp, i64, i64, ctypes.POINTER(ctypes.c_double), vp]
            lib.attn_probe_sfu_ex2.restype = ci
            _lib = lib
    return _lib


def attn_probe_fp32_fma(sink: torch.Tensor, iters: int, stream=None) -> float:
    """Enqueue the FFMA throughput probe (see attn_probe_fp32_fma in include/attn.h) on `stream`
    (default: the current stream of sink's device) and return the launch's flop count; the
    caller times the launch with CUDA events. sink: float32 CUDA tensor of >= SMs x 1024."""
    if sink.dtype != torch.float32 or not sink.is_cuda or not sink.is_contiguous():
        raise ValueError("sink must be a contiguous float32 CUDA tensor")
    flop = ctypes.c_double(0.0)
    st = raw().attn_probe_fp32_fma(sink.data_ptr(), sink.numel(), int(iters), ctypes.byref(flop),
                                   _stream(sink.device, stream))
    if st != 0:
        raise AttnError(st, "attn_probe_fp32_fma")
    return float(flop.value)


def attn_probe_sfu_ex2(sink: torch.Tensor, iters: int, stream=None) -> float:
    """Enqueue the exponential (ex2) throughput probe (see attn_probe_sfu_ex2 in include/attn.h)
    on `stream` and return the launch's count of exponentials; the caller times the launch with
    CUDA events. sink: float32 CUDA tensor of >= SMs x 1024."""
    if sink.dtype != torch.float32 or not sink.is_cuda or not sink.is_contiguous():
        raise ValueError("sink must be a contiguous float32 CUDA tensor")
    ops = ctypes.c_double(0.0)
    st = raw().attn_probe_sfu_ex2(sink.data_ptr(), sink.numel(), int(iters), ctypes.byref(ops),
                                  _stream(sink.device, stream))
    if st != 0:
        raise AttnError(st, "attn_probe_sfu_ex2")
    return float(ops.value)


def attn_status_string(status: int) -> str:
    return raw().attn_status_string(int(status)).decode()


def attn_abi_version() -> int:
    return int(raw().attn_abi_version())


def attn_plan_launch_order(weights, fixed: int, num_sms: int) -> list[int]:
    """The launch order the causal kernels use for items of these weights (host only): a list
    of item indices, position -> item. See attn_plan_launch_order in include/attn.h."""
    w = (ctypes.c_int32 * len(weights))(*[int(x) for x in weights])
    out = (ctypes.c_uint16 * max(1, len(weights)))()
    st = raw().attn_plan_launch_order(ctypes.cast(w, ctypes.c_void_p), len(weights), int(fixed), int(num_sms),
                                      ctypes.cast(out, ctypes.c_void_p))
    if st != 0:
        raise AttnError(st, "attn_plan_launch_order")
    return list(out[:len(weights)])


def _check(q, k, v):
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise TypeError(f"{name} must be a CUDA tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous [B, H, N, d]")
    if q.dim() != 4 or q.shape != k.shape or q.shape != v.shape:
        raise ValueError("q, k, v must share one [B, H, N, d] shape")
    if q.dtype != k.dtype or q.dtype != v.dtype or q.dtype not in _DTYPES:
        raise TypeError("q, k, v must share one dtype among float32, bfloat16, float16")
    if q.device != k.device or q.device != v.device:
        raise ValueError("q, k, v must be on one device")


# The current stream's handle without building a Stream object (PyTorch's own raw accessor);
# the public call when a build of PyTorch lacks it.
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(dev, stream):
    if stream is None:
        if _raw_stream is not None:
            return ctypes.c_void_p(_raw_stream(dev.index if dev.index is not None else torch.cuda.current_device()))
        stream = torch.cuda.current_stream(dev)
    return ctypes.c_void_p(stream.cuda_stream)


def _device(dev):
    """The tensors' device made current for the call (the library launches on the current
    device); no switch when it already is."""
    if dev.index is None or dev.index == torch.cuda.current_device():
        return contextlib.nullcontext()
    return torch.cuda.device(dev)


def attn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
             out: torch.Tensor | None = None, stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """o = softmax(q k^T / sqrt(d) + causal mask) v, by the online (flash) kernels."""
    _check(q, k, v)
    if out is None:
        out = torch.empty_like(q)
    elif out.shape != q.shape or out.dtype != q.dtype or out.device != q.device or not out.is_contiguous():
        raise ValueError("out must be a contiguous tensor like q")
    B, H, N, d = q.shape
    lib = raw()
    with _device(q.device):
        st = lib.attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, H, N, d,
                          int(bool(causal)), _DTYPES[q.dtype], _stream(q.device, stream))
    if st != 0:
        raise AttnError(st, "attn_fwd")
    return out


def attn_fwd_lse(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
                 out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                 stream: torch.cuda.Stream | None = None) -> tuple[torch.Tensor, torch.Tensor]:
    """``(o, lse)``: the flash forward and each row's base-2 log-sum-exp,
    ``lse[b, h, i] = log2(sum_j exp(q_i . k_j / sqrt(d)))`` (float32 ``[B, H, N]``)."""
    _check(q, k, v)
    B, H, N, d = q.shape
    if out is None:
        out = torch.empty_like(q)
    elif out.shape != q.shape or out.dtype != q.dtype or out.device != q.device or not out.is_contiguous():
        raise ValueError("out must be a contiguous tensor like q")
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    elif lse.shape != (B, H, N) or lse.dtype != torch.float32 or lse.device != q.device or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 tensor [B, H, N] on q's device")
    lib = raw()
    with _device(q.device):
        st = lib.attn_fwd_lse(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                              B, H, N, d, int(bool(causal)), _DTYPES[q.dtype], _stream(q.device, stream))
    if st != 0:
        raise AttnError(st, "attn_fwd_lse")
    return out, lse


def attn_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor, dout: torch.Tensor,
             lse: torch.Tensor, causal: bool = False,
             stream: torch.cuda.Stream | None = None) -> tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """``(dq, dk, dv)``: gradients for the output gradient ``dout``, given the forward's ``o``
    and base-2 log-sum-exps ``lse`` from :func:`attn_fwd_lse` on the same ``q, k, v``."""
    _check(q, k, v)
    B, H, N, d = q.shape
    for name, t in (("o", o), ("dout", dout)):
        if not isinstance(t, torch.Tensor) or t.shape != q.shape or t.dtype != q.dtype or t.device != q.device \
                or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous tensor like q")
    if lse.shape != (B, H, N) or lse.dtype != torch.float32 or lse.device != q.device or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 tensor [B, H, N] on q's device")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    lib = raw()
    with _device(q.device):
        st = lib.attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(), lse.data_ptr(),
                          dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d, int(bool(causal)),
                          _DTYPES[q.dtype], _stream(q.device, stream))
    if st != 0:
        raise AttnError(st, "attn_bwd")
    return dq, dk, dv


ATTN_KV_MAX_SPLITS = 1024  # include/attn.h: most shares the key range may be cut into


def attn_kvcache_workspace_bytes(B: int, H: int, Nq: int, Nk: int, num_splits: int = 0,
                                 dtype: torch.dtype = torch.bfloat16, device: torch.device | int | None = None,
                                 d: int = 64) -> int:
    """Workspace bytes :func:`attn_fwd_kvcache` needs; for ``num_splits == 0`` (balanced) the plan
    depends on the device, which is queried with ``device`` current."""
    dev = torch.device("cuda", torch.cuda.current_device() if device is None else torch.device(device).index or 0) \
        if num_splits == 0 else None
    if dev is None:
        return int(raw().attn_kvcache_workspace_bytes(B, H, Nq, Nk, d, num_splits, _DTYPES[dtype]))
    with _device(dev):
        return int(raw().attn_kvcache_workspace_bytes(B, H, Nq, Nk, d, num_splits, _DTYPES[dtype]))


def attn_fwd_kvcache(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = True,
                     num_splits: int = 0, workspace: torch.Tensor | None = None,
                     out: torch.Tensor | None = None, lse: torch.Tensor | bool | None = None,
                     stream: torch.cuda.Stream | None = None):
    """Attention of ``q`` ``[B, H, Nq, d]`` (the last Nq positions) against a key-value cache
    ``k, v`` ``[B, H, Nk, d]``, Nq <= Nk; causal: query i sees keys ``0 .. Nk - Nq + i``.
    ``num_splits`` 0 balances the keys of all heads over the whole GPU; S >= 1 cuts every head
    into S shares. When ``workspace`` (a uint8 CUDA tensor) is omitted, one of the needed size
    is allocated here. ``lse=True`` (or a float32 ``[B, H, Nq]`` tensor) also returns the base-2
    log-sum-exps: the result is then ``(o, lse)``, otherwise ``o``."""
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise TypeError(f"{name} must be a CUDA tensor")
        if not t.is_contiguous() or t.dim() != 4:
            raise ValueError(f"{name} must be a contiguous 4-d tensor")
    if k.shape != v.shape or q.shape[:2] != k.shape[:2] or q.shape[3] != k.shape[3]:
        raise ValueError("q must be [B, H, Nq, d] and k, v [B, H, Nk, d]")
    if q.dtype != k.dtype or q.dtype != v.dtype or q.dtype not in _DTYPES:
        raise TypeError("q, k, v must share one dtype among float32, bfloat16, float16")
    if q.device != k.device or q.device != v.device:
        raise ValueError("q, k, v must be on one device")
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if out is None:
        out = torch.empty_like(q)
    elif out.shape != q.shape or out.dtype != q.dtype or out.device != q.device or not out.is_contiguous():
        raise ValueError("out must be a contiguous tensor like q")
    want_lse = lse is not None and lse is not False
    if lse is True:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    elif want_lse and (lse.shape != (B, H, Nq) or lse.dtype != torch.float32 or lse.device != q.device
                       or not lse.is_contiguous()):
        raise ValueError("lse must be a contiguous float32 tensor [B, H, Nq] on q's device")
    lib = raw()
    with _device(q.device):
        if workspace is None:
            need = int(lib.attn_kvcache_workspace_bytes(B, H, Nq, Nk, d, int(num_splits), _DTYPES[q.dtype]))
            workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
        st = lib.attn_fwd_kvcache(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                  lse.data_ptr() if want_lse else None, workspace.data_ptr(),
                                  workspace.numel() * workspace.element_size(), B, H, Nq, Nk, d,
                                  int(bool(causal)), _DTYPES[q.dtype], int(num_splits), _stream(q.device, stream))
    if st != 0:
        raise AttnError(st, "attn_fwd_kvcache")
    return (out, lse) if want_lse else out


def attn_materialized_workspace_bytes(B: int, H: int, N: int) -> int:
    return int(raw().attn_materialized_workspace_bytes(B, H, N))


def attn_fwd_materialized(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
                          workspace: torch.Tensor | None = None, out: torch.Tensor | None = None,
                          stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """The same result through the materialised N x N path (ablation). ``workspace`` is a
    uint8 CUDA tensor; when omitted one big enough for all heads at once is allocated."""
    _check(q, k, v)
    B, H, N, d = q.shape
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = torch.empty(max(1, attn_materialized_workspace_bytes(B, H, N)), dtype=torch.uint8,
                                device=q.device)
    lib = raw()
    with _device(q.device):
        st = lib.attn_fwd_materialized(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                       workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                       B, H, N, d, int(bool(causal)), _DTYPES[q.dtype],
                                       _stream(q.device, stream))
    if st != 0:
        raise AttnError(st, "attn_fwd_materialized")
    return out


def attn_selftest_wait_timeout(timeout_ns: int = 1_000_000, stream: torch.cuda.Stream | None = None,
                               device: torch.device | int | None = None) -> None:
    """Launches the library's timeout self-test: one warp whose only wait runs out after
    ``timeout_ns``; afterwards :func:`attn_device_status` reports ATTN_ERR_TIMEOUT (7)."""
    dev = torch.device("cuda", torch.cuda.current_device() if device is None else torch.device(device).index or 0)
    with _device(dev):
        st = raw().attn_selftest_wait_timeout(int(timeout_ns), _stream(dev, stream))
    if st != 0:
        raise AttnError(st, "attn_selftest_wait_timeout")


def attn_device_status(clear: bool = True, stream: torch.cuda.Stream | None = None,
                       device: torch.device | int | None = None) -> int:
    """Synchronises the stream and returns ATTN_OK (0) or ATTN_ERR_TIMEOUT (7)."""
    dev = torch.device("cuda", torch.cuda.current_device() if device is None else torch.device(device).index or 0)
    with _device(dev):
        return int(raw().attn_device_status(_stream(dev, stream), int(bool(clear))))


ATTN_NOALLOC_MAX_N = 2896  # include/attn.h: largest N whose per-head scratch fits the fixed array


def attn_fwd_materialized_noalloc(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
                                  out: torch.Tensor | None = None,
                                  stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """The materialised path without a workspace: its scratch is a fixed array inside the
    library, so the library allocates nothing. Meant for callers that cannot allocate device
    memory. ``out`` may be passed to avoid the one allocation this Python wrapper would
    otherwise make for the result. N must not exceed ``ATTN_NOALLOC_MAX_N``; concurrent calls
    whose kernels overlap on the GPU share the scratch and race."""
    _check(q, k, v)
    B, H, N, d = q.shape
    if out is None:
        out = torch.empty_like(q)
    lib = raw()
    fn = lib.attn_fwd_materialized_noalloc
    vp, i64, ci = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    fn.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, ci, ci, vp]
    fn.restype = ci
    with _device(q.device):
        st = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, H, N, d, int(bool(causal)),
                _DTYPES[q.dtype], _stream(q.device, stream))
    if st != 0:
        raise AttnError(st, "attn_fwd_materialized_noalloc")
    return out
