"""ctypes binding of libmoe (include/moe.h), same names as the C entry points.

Argument marshalling only: every step of the layer runs in libmoe's CUDA
kernels.  Tensors are torch tensors on the current CUDA device (PyTorch is
used for device memory and streams); they are passed as raw pointers.  If
libmoe.so is missing or cannot be loaded the binding raises instead of
falling back to anything else.
"""
from __future__ import annotations

import ctypes
import re
from pathlib import Path

import torch

PKG = Path(__file__).resolve().parent
LIB_PATH = PKG / "libmoe.so"
HEADER = PKG.parent / "include" / "moe.h"

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_UNSUPPORTED_SHAPE = -2
MOE_ERR_MISALIGNED = -3
MOE_ERR_WORKSPACE_TOO_SMALL = -4
MOE_ERR_CUDA = -5
MOE_ERR_DEVICE_STATUS = -6
MOE_ERR_TIMEOUT = -7
MOE_DEV_BAD_EXPERT_ID = 0x1
MOE_DEV_TIMEOUT = 0x2
MOE_DEV_BAD_OFFSETS = 0x4
MOE_DEV_BAD_MODALITY = 0x8
MOE_DEV_BAD_SOURCE_ROW = 0x10
MOE_FUSE_GATHER = 0x1
MOE_FUSE_GATE = 0x2


class MoeError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} ({code})")


class moe_dims(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("d", ctypes.c_int32), ("n_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("E", ctypes.c_int32), ("inter", ctypes.c_int32),
                ("top_k", ctypes.c_int32)]

    @classmethod
    def make(cls, T, d, E, inter, top_k=6, n_heads=12, head_dim=256):
        return cls(int(T), int(d), int(n_heads), int(head_dim), int(E), int(inter), int(top_k))

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


class moe_ext(ctypes.Structure):
    _fields_ = [("n_shared", ctypes.c_int32), ("n_modalities", ctypes.c_int32),
                ("expert_begin", ctypes.c_int32 * 8), ("expert_end", ctypes.c_int32 * 8),
                ("modality", ctypes.c_void_p)]

    @classmethod
    def make(cls, n_shared=0, ranges=(), modality=None):
        """ranges: ((begin, end), ...) per modality; modality: device int32 [T] tensor or None."""
        e = cls()
        e.n_shared = int(n_shared)
        e.n_modalities = len(ranges)
        for m, (b, en) in enumerate(ranges):
            e.expert_begin[m], e.expert_end[m] = int(b), int(en)
        if modality is not None:
            _dev(modality, dtype=torch.int32)
            e.modality = modality.data_ptr()
        return e


_P = ctypes.c_void_p
_DP = ctypes.POINTER(moe_dims)
_XP = ctypes.POINTER(moe_ext)
_SIGS = {
    "moe_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "moe_check_dims": (ctypes.c_int, [_DP]),
    "moe_scratch_size": (ctypes.c_int, [_DP, ctypes.POINTER(ctypes.c_size_t)]),
    "moe_workspace_size": (ctypes.c_int, [_DP, ctypes.POINTER(ctypes.c_size_t)]),
    "moe_workspace_size_host": (ctypes.c_int, [_DP, ctypes.POINTER(ctypes.c_size_t)]),
    "moe_clear_device_status": (ctypes.c_int, [_P, _P]),
    "moe_get_device_status": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_int32), _P]),
    "moe_prepare_weights": (ctypes.c_int, [_DP, _P, _P, _P, _P]),
    "moe_selftest_timeout": (ctypes.c_int, [_P, ctypes.c_size_t, ctypes.c_uint32, _P]),
    "moe_selftest_timeout_fused": (ctypes.c_int, [_P, ctypes.c_size_t, ctypes.c_uint32, _P]),
    "moe_route": (ctypes.c_int, [_DP, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "moe_route_fused": (ctypes.c_int, [_DP, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "moe_route_two_stage": (ctypes.c_int, [_DP, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "moe_prepare_router": (ctypes.c_int, [_DP, _P, _P, _P, _P]),
    "moe_route_folded": (ctypes.c_int, [_DP, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "moe_forward_folded": (ctypes.c_int, [_DP, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "moe_dispatch": (ctypes.c_int, [_DP, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "moe_dispatch_indices": (ctypes.c_int, [_DP, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "moe_expert_gemm1_gather": (ctypes.c_int, [_DP, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "moe_dispatch_noalloc": (ctypes.c_int, [_DP, _P, _P, _P, _P, _P, _P, _P, _P]),
    "moe_expert_ffn": (ctypes.c_int, [_DP, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "moe_expert_gemm1": (ctypes.c_int, [_DP, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "moe_expert_gemm2": (ctypes.c_int, [_DP, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "moe_combine": (ctypes.c_int, [_DP, _P, _P, _P, _P, _P]),
    "moe_expert_gemm2_gated": (ctypes.c_int, [_DP, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "moe_combine_rows": (ctypes.c_int, [_DP, _P, _P, _P, _P]),
    "moe_forward_fused": (ctypes.c_int, [_DP, _P, _P, _P, _P, _P, _P, _P, ctypes.c_uint32, _P, ctypes.c_size_t,
                                         _P]),
    "moe_forward": (ctypes.c_int, [_DP, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "moe_workspace_size_ext": (ctypes.c_int, [_DP, _XP, ctypes.POINTER(ctypes.c_size_t)]),
    "moe_route_ext": (ctypes.c_int, [_DP, _XP, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "moe_forward_ext": (ctypes.c_int, [_DP, _XP, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "moe_workspace_size_headlocal": (ctypes.c_int, [_DP, ctypes.POINTER(ctypes.c_size_t)]),
    "moe_prepare_weights_headlocal": (ctypes.c_int, [_DP, _P, _P, _P, _P]),
    "moe_forward_headlocal": (ctypes.c_int, [_DP, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "moe_forward_headlocal_staged": (ctypes.c_int, [_DP, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "moe_forward_host": (ctypes.c_int, [_DP, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
}

_lib = None


def header_functions() -> list[str]:
    """Names of the functions declared in include/moe.h."""
    text = HEADER.read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(moe_\w+)\s*\(", text, flags=re.M)))


def lib() -> ctypes.CDLL:
    """Loads libmoe.so (built by fine_grained_moe_02_b300.build); raises if absent."""
    global _lib
    if _lib is None:
        if not LIB_PATH.exists():
            raise RuntimeError(f"{LIB_PATH} is not built; run `python -m fine_grained_moe_02_b300.build`")
        L = ctypes.CDLL(str(LIB_PATH))
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def status_string(code: int) -> str:
    return lib().moe_status_string(int(code)).decode()


def _check(rc: int, where: str) -> None:
    if rc != MOE_OK:
        raise MoeError(rc, where)


def _ptr(t) -> ctypes.c_void_p | None:
    if t is None:
        return None
    if isinstance(t, int):
        return ctypes.c_void_p(t)
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _need(dims, **tensors) -> None:
    """Each named tensor must hold at least the elements its role needs for
    `dims` (the C ABI takes bare pointers and cannot check this; a short
    buffer would be read or written past its end on the device)."""
    T, d, E, I, k = int(dims.T), int(dims.d), int(dims.E), int(dims.inter), int(dims.top_k)
    H, Dh = int(dims.n_heads), int(dims.head_dim)
    L = H * Dh
    sizes = {
        "x": T * d, "out": T * d, "x_host": T * d, "out_host": T * d,
        "w_lat": L * d, "w_head": E * L, "bias": E, "w_router": E * 2 * d,
        "topk_idx": T * k, "topk_gate": T * k, "logits": T * E,
        "w_gate": E * I * d, "w_up": E * I * d, "w13": E * 2 * I * d, "w_down": E * d * I,
        "offsets": E + 1, "row_of": T * k, "src_token": T * k,
        "x_perm": T * k * d, "y_perm": T * k * d, "act": T * k * I, "status": 1,
    }
    for name, t in tensors.items():
        if t is None or isinstance(t, int):
            continue
        need = sizes[name]
        if t.numel() < need:
            raise ValueError(f"{name}: {t.numel()} elements, these dims need {need}")


def _need_n(**named) -> None:
    """name=(tensor, elements needed) pairs, for layouts _need does not cover."""
    for name, (t, need) in named.items():
        if t is not None and not isinstance(t, int) and t.numel() < need:
            raise ValueError(f"{name}: {t.numel()} elements, these dims need {need}")


def _ext_dims(dims, ext):
    """dims with the shared experts added: E + n_shared experts, top_k + n_shared slots."""
    return moe_dims.make(dims.T, dims.d, dims.E + ext.n_shared, dims.inter, dims.top_k + ext.n_shared,
                         dims.n_heads, dims.head_dim)


def _dev(*ts, dtype=None) -> None:
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("expected a CUDA tensor")
        if dtype is not None and t.dtype != dtype:
            raise ValueError(f"expected {dtype}, got {t.dtype}")


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def moe_check_dims(dims: moe_dims) -> int:
    return lib().moe_check_dims(ctypes.byref(dims))


def moe_scratch_size(dims: moe_dims) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().moe_scratch_size(ctypes.byref(dims), ctypes.byref(n)), "moe_scratch_size")
    return n.value


def moe_workspace_size(dims: moe_dims) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().moe_workspace_size(ctypes.byref(dims), ctypes.byref(n)), "moe_workspace_size")
    return n.value


def moe_workspace_size_host(dims: moe_dims) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().moe_workspace_size_host(ctypes.byref(dims), ctypes.byref(n)), "moe_workspace_size_host")
    return n.value


def alloc_workspace(nbytes: int, device=None) -> torch.Tensor:
    """A uint8 device buffer for use as `ws` (PyTorch owns the memory)."""
    return torch.zeros(int(nbytes), dtype=torch.uint8, device=device or "cuda")


def moe_clear_device_status(ws, stream=None) -> None:
    _check(lib().moe_clear_device_status(_ptr(ws), _stream(stream)), "moe_clear_device_status")


def moe_get_device_status(ws, stream=None) -> int:
    v = ctypes.c_int32(0)
    rc = lib().moe_get_device_status(_ptr(ws), ctypes.byref(v), _stream(stream))
    if rc not in (MOE_OK, MOE_ERR_DEVICE_STATUS):
        _check(rc, "moe_get_device_status")
    return v.value


def moe_selftest_timeout(ws, limit_us: int, stream=None) -> None:
    """Runs the GEMM kernel with a loader that issues nothing (waits time out)."""
    _check(lib().moe_selftest_timeout(_ptr(ws), ws.numel(), int(limit_us), _stream(stream)), "moe_selftest_timeout")


def moe_selftest_timeout_fused(ws, limit_us: int, stream=None) -> None:
    """Runs the fused head-local expert kernel with a weight loader that issues nothing."""
    _check(lib().moe_selftest_timeout_fused(_ptr(ws), ws.numel(), int(limit_us), _stream(stream)),
           "moe_selftest_timeout_fused")


def moe_prepare_weights(dims, w_gate, w_up, w13, stream=None) -> None:
    _need(dims, w_gate=w_gate, w_up=w_up, w13=w13)
    _dev(w_gate, w_up, w13, dtype=torch.bfloat16)
    _check(lib().moe_prepare_weights(ctypes.byref(dims), _ptr(w_gate), _ptr(w_up), _ptr(w13), _stream(stream)),
           "moe_prepare_weights")


def moe_route(dims, x, w_lat, w_head, bias, topk_idx, topk_gate, logits, ws, stream=None) -> None:
    _need(dims, x=x, w_lat=w_lat, w_head=w_head, bias=bias, topk_idx=topk_idx, topk_gate=topk_gate, logits=logits)
    _dev(x, w_lat, w_head, dtype=torch.bfloat16)
    _dev(bias, topk_gate, logits, dtype=torch.float32)
    _dev(topk_idx, dtype=torch.int32)
    _check(lib().moe_route(ctypes.byref(dims), _ptr(x), _ptr(w_lat), _ptr(w_head), _ptr(bias), _ptr(topk_idx),
                           _ptr(topk_gate), _ptr(logits), _ptr(ws), ws.numel(), _stream(stream)), "moe_route")


def moe_route_two_stage(dims, x, w_lat, w_head, bias, topk_idx, topk_gate, logits, ws, stream=None) -> None:
    _need(dims, x=x, w_lat=w_lat, w_head=w_head, bias=bias, topk_idx=topk_idx, topk_gate=topk_gate, logits=logits)
    _dev(x, w_lat, w_head, dtype=torch.bfloat16)
    _dev(bias, topk_gate, logits, dtype=torch.float32)
    _dev(topk_idx, dtype=torch.int32)
    _check(lib().moe_route_two_stage(ctypes.byref(dims), _ptr(x), _ptr(w_lat), _ptr(w_head), _ptr(bias),
                                     _ptr(topk_idx), _ptr(topk_gate), _ptr(logits), _ptr(ws), ws.numel(),
                                     _stream(stream)), "moe_route_two_stage")


def moe_route_fused(dims, x, w_lat, w_head, bias, topk_idx, topk_gate, logits, ws, stream=None) -> None:
    _need(dims, x=x, w_lat=w_lat, w_head=w_head, bias=bias, topk_idx=topk_idx, topk_gate=topk_gate, logits=logits)
    _dev(x, w_lat, w_head, dtype=torch.bfloat16)
    _dev(bias, topk_gate, logits, dtype=torch.float32)
    _dev(topk_idx, dtype=torch.int32)
    _check(lib().moe_route_fused(ctypes.byref(dims), _ptr(x), _ptr(w_lat), _ptr(w_head), _ptr(bias), _ptr(topk_idx),
                                 _ptr(topk_gate), _ptr(logits), _ptr(ws), ws.numel(), _stream(stream)),
           "moe_route_fused")


def moe_prepare_router(dims, w_lat, w_head, w_router, stream=None) -> None:
    _need(dims, w_lat=w_lat, w_head=w_head, w_router=w_router)
    _dev(w_lat, w_head, w_router, dtype=torch.bfloat16)
    _check(lib().moe_prepare_router(ctypes.byref(dims), _ptr(w_lat), _ptr(w_head), _ptr(w_router), _stream(stream)),
           "moe_prepare_router")


def moe_route_folded(dims, x, w_router, bias, topk_idx, topk_gate, logits, ws, stream=None) -> None:
    _need(dims, x=x, w_router=w_router, bias=bias, topk_idx=topk_idx, topk_gate=topk_gate, logits=logits)
    _dev(x, w_router, dtype=torch.bfloat16)
    _dev(bias, topk_gate, logits, dtype=torch.float32)
    _dev(topk_idx, dtype=torch.int32)
    _check(lib().moe_route_folded(ctypes.byref(dims), _ptr(x), _ptr(w_router), _ptr(bias), _ptr(topk_idx),
                                  _ptr(topk_gate), _ptr(logits), _ptr(ws), ws.numel(), _stream(stream)),
           "moe_route_folded")


def moe_forward_folded(dims, x, w_router, bias, w13, w_down, out, ws, stream=None) -> None:
    _need(dims, x=x, w_router=w_router, bias=bias, w13=w13, w_down=w_down, out=out)
    _dev(x, w_router, w13, w_down, out, dtype=torch.bfloat16)
    _dev(bias, dtype=torch.float32)
    _check(lib().moe_forward_folded(ctypes.byref(dims), _ptr(x), _ptr(w_router), _ptr(bias), _ptr(w13),
                                    _ptr(w_down), _ptr(out), _ptr(ws), ws.numel(), _stream(stream)),
           "moe_forward_folded")


def moe_dispatch(dims, x, topk_idx, offsets, row_of, src_token, x_perm, ws, stream=None) -> None:
    _need(dims, x=x, topk_idx=topk_idx, offsets=offsets, row_of=row_of, src_token=src_token, x_perm=x_perm)
    _dev(x, x_perm, dtype=torch.bfloat16)
    _dev(topk_idx, offsets, row_of, src_token, dtype=torch.int32)
    _check(lib().moe_dispatch(ctypes.byref(dims), _ptr(x), _ptr(topk_idx), _ptr(offsets), _ptr(row_of),
                              _ptr(src_token), _ptr(x_perm), _ptr(ws), ws.numel(), _stream(stream)), "moe_dispatch")


def moe_dispatch_indices(dims, topk_idx, offsets, row_of, src_token, ws, stream=None) -> None:
    _need(dims, topk_idx=topk_idx, offsets=offsets, row_of=row_of, src_token=src_token)
    _dev(topk_idx, offsets, row_of, src_token, dtype=torch.int32)
    _check(lib().moe_dispatch_indices(ctypes.byref(dims), _ptr(topk_idx), _ptr(offsets), _ptr(row_of),
                                      _ptr(src_token), _ptr(ws), ws.numel(), _stream(stream)), "moe_dispatch_indices")


def moe_expert_gemm1_gather(dims, x, src_token, offsets, w13, act, ws, stream=None) -> None:
    _need(dims, x=x, src_token=src_token, offsets=offsets, w13=w13, act=act)
    _dev(x, w13, act, dtype=torch.bfloat16)
    _dev(src_token, offsets, dtype=torch.int32)
    _check(lib().moe_expert_gemm1_gather(ctypes.byref(dims), _ptr(x), _ptr(src_token), _ptr(offsets), _ptr(w13),
                                         _ptr(act), _ptr(ws), ws.numel(), _stream(stream)), "moe_expert_gemm1_gather")


def moe_dispatch_noalloc(dims, x, topk_idx, offsets, row_of, src_token, x_perm, status=None, stream=None) -> None:
    """moe_dispatch without a workspace (scratch in a fixed array inside libmoe)."""
    _need(dims, x=x, topk_idx=topk_idx, offsets=offsets, row_of=row_of, src_token=src_token, x_perm=x_perm,
          status=status)
    _dev(x, x_perm, dtype=torch.bfloat16)
    _dev(topk_idx, offsets, row_of, src_token, status, dtype=torch.int32)
    _check(lib().moe_dispatch_noalloc(ctypes.byref(dims), _ptr(x), _ptr(topk_idx), _ptr(offsets), _ptr(row_of),
                                      _ptr(src_token), _ptr(x_perm), _ptr(status), _stream(stream)),
           "moe_dispatch_noalloc")


def moe_expert_ffn(dims, x_perm, offsets, w13, w_down, act, y_perm, ws, stream=None) -> None:
    _need(dims, x_perm=x_perm, offsets=offsets, w13=w13, w_down=w_down, act=act, y_perm=y_perm)
    _dev(x_perm, w13, w_down, act, y_perm, dtype=torch.bfloat16)
    _dev(offsets, dtype=torch.int32)
    _check(lib().moe_expert_ffn(ctypes.byref(dims), _ptr(x_perm), _ptr(offsets), _ptr(w13), _ptr(w_down),
                                _ptr(act), _ptr(y_perm), _ptr(ws), ws.numel(), _stream(stream)), "moe_expert_ffn")


def moe_expert_gemm1(dims, x_perm, offsets, w13, act, ws, stream=None) -> None:
    _need(dims, x_perm=x_perm, offsets=offsets, w13=w13, act=act)
    _dev(x_perm, w13, act, dtype=torch.bfloat16)
    _dev(offsets, dtype=torch.int32)
    _check(lib().moe_expert_gemm1(ctypes.byref(dims), _ptr(x_perm), _ptr(offsets), _ptr(w13), _ptr(act),
                                  _ptr(ws), ws.numel(), _stream(stream)), "moe_expert_gemm1")


def moe_expert_gemm2(dims, act, offsets, w_down, y_perm, ws, stream=None) -> None:
    _need(dims, act=act, offsets=offsets, w_down=w_down, y_perm=y_perm)
    _dev(act, w_down, y_perm, dtype=torch.bfloat16)
    _dev(offsets, dtype=torch.int32)
    _check(lib().moe_expert_gemm2(ctypes.byref(dims), _ptr(act), _ptr(offsets), _ptr(w_down), _ptr(y_perm),
                                  _ptr(ws), ws.numel(), _stream(stream)), "moe_expert_gemm2")


def moe_combine(dims, y_perm, row_of, topk_gate, out, stream=None) -> None:
    _need(dims, y_perm=y_perm, row_of=row_of, topk_gate=topk_gate, out=out)
    _dev(y_perm, out, dtype=torch.bfloat16)
    _dev(row_of, dtype=torch.int32)
    _dev(topk_gate, dtype=torch.float32)
    _check(lib().moe_combine(ctypes.byref(dims), _ptr(y_perm), _ptr(row_of), _ptr(topk_gate), _ptr(out),
                             _stream(stream)), "moe_combine")


def moe_expert_gemm2_gated(dims, act, offsets, w_down, src_token, row_of, topk_gate, y_perm, ws,
                           stream=None) -> None:
    _need(dims, act=act, offsets=offsets, w_down=w_down, src_token=src_token, row_of=row_of, topk_gate=topk_gate,
          y_perm=y_perm)
    _dev(act, w_down, y_perm, dtype=torch.bfloat16)
    _dev(offsets, src_token, row_of, dtype=torch.int32)
    _dev(topk_gate, dtype=torch.float32)
    _check(lib().moe_expert_gemm2_gated(ctypes.byref(dims), _ptr(act), _ptr(offsets), _ptr(w_down),
                                        _ptr(src_token), _ptr(row_of), _ptr(topk_gate), _ptr(y_perm), _ptr(ws),
                                        ws.numel(), _stream(stream)), "moe_expert_gemm2_gated")


def moe_combine_rows(dims, y_perm, row_of, out, stream=None) -> None:
    _need(dims, y_perm=y_perm, row_of=row_of, out=out)
    _dev(y_perm, out, dtype=torch.bfloat16)
    _dev(row_of, dtype=torch.int32)
    _check(lib().moe_combine_rows(ctypes.byref(dims), _ptr(y_perm), _ptr(row_of), _ptr(out), _stream(stream)),
           "moe_combine_rows")


def moe_forward_fused(dims, x, w_lat, w_head, bias, w13, w_down, out, fuse, ws, stream=None) -> None:
    _need(dims, x=x, w_lat=w_lat, w_head=w_head, bias=bias, w13=w13, w_down=w_down, out=out)
    _dev(x, w_lat, w_head, w13, w_down, out, dtype=torch.bfloat16)
    _dev(bias, dtype=torch.float32)
    _check(lib().moe_forward_fused(ctypes.byref(dims), _ptr(x), _ptr(w_lat), _ptr(w_head), _ptr(bias), _ptr(w13),
                                   _ptr(w_down), _ptr(out), int(fuse), _ptr(ws), ws.numel(), _stream(stream)),
           "moe_forward_fused")


def moe_forward(dims, x, w_lat, w_head, bias, w13, w_down, out, ws, stream=None) -> None:
    _need(dims, x=x, w_lat=w_lat, w_head=w_head, bias=bias, w13=w13, w_down=w_down, out=out)
    _dev(x, w_lat, w_head, w13, w_down, out, dtype=torch.bfloat16)
    _dev(bias, dtype=torch.float32)
    _check(lib().moe_forward(ctypes.byref(dims), _ptr(x), _ptr(w_lat), _ptr(w_head), _ptr(bias), _ptr(w13),
                             _ptr(w_down), _ptr(out), _ptr(ws), ws.numel(), _stream(stream)), "moe_forward")


def moe_workspace_size_ext(dims, ext) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().moe_workspace_size_ext(ctypes.byref(dims), ctypes.byref(ext), ctypes.byref(n)),
           "moe_workspace_size_ext")
    return n.value


def moe_route_ext(dims, ext, x, w_lat, w_head, bias, topk_idx, topk_gate, logits, ws, stream=None) -> None:
    _need(dims, x=x, w_lat=w_lat, w_head=w_head, bias=bias, logits=logits)
    _need(_ext_dims(dims, ext), topk_idx=topk_idx, topk_gate=topk_gate)
    _dev(x, w_lat, w_head, dtype=torch.bfloat16)
    _dev(bias, topk_gate, logits, dtype=torch.float32)
    _dev(topk_idx, dtype=torch.int32)
    _check(lib().moe_route_ext(ctypes.byref(dims), ctypes.byref(ext), _ptr(x), _ptr(w_lat), _ptr(w_head), _ptr(bias),
                               _ptr(topk_idx), _ptr(topk_gate), _ptr(logits), _ptr(ws), ws.numel(), _stream(stream)),
           "moe_route_ext")


def moe_forward_ext(dims, ext, x, w_lat, w_head, bias, w13, w_down, out, ws, stream=None) -> None:
    _need(dims, x=x, w_lat=w_lat, w_head=w_head, bias=bias, out=out)
    _need(_ext_dims(dims, ext), w13=w13, w_down=w_down)
    _dev(x, w_lat, w_head, w13, w_down, out, dtype=torch.bfloat16)
    _dev(bias, dtype=torch.float32)
    _check(lib().moe_forward_ext(ctypes.byref(dims), ctypes.byref(ext), _ptr(x), _ptr(w_lat), _ptr(w_head),
                                 _ptr(bias), _ptr(w13), _ptr(w_down), _ptr(out), _ptr(ws), ws.numel(),
                                 _stream(stream)), "moe_forward_ext")


def moe_workspace_size_headlocal(dims) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().moe_workspace_size_headlocal(ctypes.byref(dims), ctypes.byref(n)), "moe_workspace_size_headlocal")
    return n.value


def moe_prepare_weights_headlocal(dims, w_gate, w_up, w13, stream=None) -> None:
    H, E, Dh, I, T, k = dims.n_heads, dims.E, dims.head_dim, dims.inter, dims.T, dims.top_k
    _need_n(w_gate=(w_gate, H * E * I * Dh), w_up=(w_up, H * E * I * Dh), w13=(w13, H * E * 2 * I * Dh))
    _dev(w_gate, w_up, w13, dtype=torch.bfloat16)
    _check(lib().moe_prepare_weights_headlocal(ctypes.byref(dims), _ptr(w_gate), _ptr(w_up), _ptr(w13),
                                               _stream(stream)), "moe_prepare_weights_headlocal")


def moe_forward_headlocal(dims, x, w_router, bias, w13, w_down, out, topk_idx, logits, ws, stream=None,
                          staged=False) -> None:
    """staged=True: moe_forward_headlocal_staged (separate expert GEMMs)."""
    H, E, Dh, I, T, k = dims.n_heads, dims.E, dims.head_dim, dims.inter, dims.T, dims.top_k
    _need_n(x=(x, T * dims.d), w_router=(w_router, H * E * Dh), bias=(bias, H * E), w13=(w13, H * E * 2 * I * Dh),
            w_down=(w_down, H * E * Dh * I), out=(out, T * dims.d), topk_idx=(topk_idx, H * T * k),
            logits=(logits, H * T * E))
    _dev(x, w_router, w13, w_down, out, dtype=torch.bfloat16)
    _dev(bias, logits, dtype=torch.float32)
    _dev(topk_idx, dtype=torch.int32)
    name = "moe_forward_headlocal_staged" if staged else "moe_forward_headlocal"
    _check(getattr(lib(), name)(ctypes.byref(dims), _ptr(x), _ptr(w_router), _ptr(bias), _ptr(w13), _ptr(w_down),
                                _ptr(out), _ptr(topk_idx), _ptr(logits), _ptr(ws), ws.numel(), _stream(stream)), name)


def moe_forward_host(dims, x_host, w_lat, w_head, bias, w13, w_down, out_host, ws, stream=None) -> None:
    """x_host/out_host: CPU bf16 tensors (pinned for full bandwidth); weights on the device."""
    _need(dims, x_host=x_host, w_lat=w_lat, w_head=w_head, bias=bias, w13=w13, w_down=w_down,
          out_host=out_host)
    if x_host.is_cuda or out_host.is_cuda:
        raise ValueError("x_host/out_host must be host tensors")
    _dev(w_lat, w_head, w13, w_down, dtype=torch.bfloat16)
    _dev(bias, dtype=torch.float32)
    _check(lib().moe_forward_host(ctypes.byref(dims), _ptr(x_host), _ptr(w_lat), _ptr(w_head), _ptr(bias),
                                  _ptr(w13), _ptr(w_down), _ptr(out_host), _ptr(ws), ws.numel(),
                                  _stream(stream)), "moe_forward_host")


class MoeLayer:
    """Device-resident weights plus a workspace; forward() runs the layer.

    router="latent" (default): moe_forward, the latent projection and head
    scores as the pages define them.  router="folded": the router folded to
    s = x (W_head W_lat)^T + b (moe_prepare_router once, then
    moe_forward_folded; same outputs within the same tolerances).  fuse:
    MOE_FUSE_GATHER and/or MOE_FUSE_GATE runs moe_forward_fused with those
    fusions (latent router only)."""

    def __init__(self, dims: moe_dims, w_lat, w_head, bias, w_gate, w_up, w_down, device="cuda",
                 router: str = "latent", fuse: int = 0):
        if router not in ("latent", "folded"):
            raise ValueError(f"router must be 'latent' or 'folded', not {router!r}")
        if fuse & ~(MOE_FUSE_GATHER | MOE_FUSE_GATE):
            raise ValueError(f"unknown fusion bits {fuse:#x}")
        if router == "folded" and fuse:
            raise ValueError("the folded router runs the unfused layer (fuse=0)")
        self.dims = dims
        self.router = router
        self.fuse = fuse
        dev = torch.device(device)
        self.w_lat = w_lat.to(dev)
        self.w_head = w_head.to(dev)
        self.bias = None if bias is None else bias.to(dev, torch.float32)
        self.w_down = w_down.to(dev)
        wg, wu = w_gate.to(dev), w_up.to(dev)
        self.w13 = torch.empty((dims.E, 2 * dims.inter, dims.d), dtype=torch.bfloat16, device=dev)
        moe_prepare_weights(dims, wg, wu, self.w13)
        del wg, wu
        self.w_router = None
        if router == "folded":
            self.w_router = torch.empty((dims.E, 2 * dims.d), dtype=torch.bfloat16, device=dev)
            moe_prepare_router(dims, self.w_lat, self.w_head, self.w_router)
        self.ws = alloc_workspace(moe_workspace_size(dims), dev)

    def forward(self, x, out=None, stream=None):
        if out is None:
            out = torch.empty((self.dims.T, self.dims.d), dtype=torch.bfloat16, device=x.device)
        if self.router == "folded":
            moe_forward_folded(self.dims, x, self.w_router, self.bias, self.w13, self.w_down, out, self.ws, stream)
        elif self.fuse:
            moe_forward_fused(self.dims, x, self.w_lat, self.w_head, self.bias, self.w13, self.w_down, out,
                              self.fuse, self.ws, stream)
        else:
            moe_forward(self.dims, x, self.w_lat, self.w_head, self.bias, self.w13, self.w_down, out, self.ws, stream)
        return out

    def device_status(self, stream=None) -> int:
        return moe_get_device_status(self.ws, stream)
