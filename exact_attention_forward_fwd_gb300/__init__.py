"""GB300 (sm_103a) exact attention forward -- Python binding of libgb300attn.so.

The binding only marshals arguments: it checks tensor shapes, dtypes and
devices, allocates outputs with torch when the caller gives none, and passes
raw device pointers and the current CUDA stream to the C ABI declared in
``include/attn.h``.  Every step of the computation runs in the library's CUDA
kernels.  There is no CPU fallback: if the library is missing or the device is
not an sm_103 GPU, calls raise.

Functions mirror the C entry points:
  attn_fwd(q, k, v, causal=False, scale=None, out=None, lse=None)
  attn_fwd_ex(q, k, v, causal=False, window=0, scale=None, ...)   (grouped KV heads, window)
  attn_fwd_splitkv(q, k, v, causal=False, window=0, num_splits=None, workspace=None, ...)
  attn_fwd_splitkv_static(q, k, v, causal=False, window=0, num_splits=None, ...)  (no allocation)
  splitkv_workspace_bytes(B, H, N, d, num_splits), splitkv_default_splits(B, H, N, d, causal, num_sms)
  attn_bwd(q, k, v, o, lse, dO, causal=False, window=0, scale=None, ...)  -> (dq, dk, dv)
  bwd_workspace_bytes(B, H, N, d)
  fp8_prep(x, signs=None, transpose=False, out=None, scales=None)
  attn_fwd_fp8(q8, k8, v8t, q_scale, k_scale, v_scale, causal=False, scale=None, ...)
  attn_fwd_fp8_from_bf16(q, k, v, signs, causal=False, scale=None)
  attn_fwd_debug(q, k, v, status, timeout_ns, skip_loads, causal=False, scale=None)
  device_status(clear=True), num_units(B, H, N), grid_size(B, H, N, num_sms)
"""
from __future__ import annotations

import ctypes
import os

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = -1
ATTN_ERR_UNSUPPORTED = -2
ATTN_ERR_ALIGNMENT = -3
ATTN_ERR_CUDA = -4
ATTN_ERR_TIMEOUT = -5
ATTN_BF16 = 0

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libgb300attn.so")
_lib = None


class AttnError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {status_str(status)} (status {status})" if what else
                         f"{status_str(status)} (status {status})")


def lib() -> ctypes.CDLL:
    """The loaded C-ABI library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                           "exact_attention_forward_fwd_gb300.build.build()")
    L = ctypes.CDLL(LIB_PATH)
    vp, i, f, fp = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_void_p
    L.attn_fwd.argtypes = [vp, vp, vp, vp, fp, i, i, i, i, f, i, i, vp]
    L.attn_fwd_ex.argtypes = [vp, vp, vp, vp, fp, i, i, i, i, i, f, i, i, i, vp]
    L.attn_fp8_prep.argtypes = [vp, vp, fp, vp, i, i, i, i, i, vp]
    L.attn_fwd_fp8.argtypes = [vp, vp, vp, fp, fp, fp, vp, fp, i, i, i, i, f, i, vp]
    L.attn_fwd_debug.argtypes = [vp, vp, vp, vp, fp, i, i, i, i, f, i, vp,
                                 ctypes.c_ulonglong, i, vp]
    L.attn_device_status.argtypes = [i]
    L.attn_num_units.argtypes = [i, i, i]
    L.attn_grid_size.argtypes = [i, i, i, i]
    L.attn_fwd_splitkv.argtypes = [vp, vp, vp, vp, fp, i, i, i, i, i, f, i, i, i, i, vp,
                                   ctypes.c_size_t, vp]
    L.attn_fwd_splitkv_static.argtypes = [vp, vp, vp, vp, fp, i, i, i, i, i, f, i, i, i, i, vp]
    L.attn_bwd.argtypes = [vp, vp, vp, vp, fp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp,
                           ctypes.c_size_t, vp]
    L.attn_bwd_workspace_bytes.argtypes = [i, i, i, i]
    L.attn_bwd_workspace_bytes.restype = ctypes.c_size_t
    L.attn_splitkv_workspace_bytes.argtypes = [i, i, i, i, i]
    L.attn_splitkv_workspace_bytes.restype = ctypes.c_size_t
    L.attn_splitkv_default_splits.argtypes = [i, i, i, i, i, i]
    L.attn_status_str.argtypes = [i]
    L.attn_status_str.restype = ctypes.c_char_p
    for name in ("attn_fwd", "attn_fwd_ex", "attn_fp8_prep", "attn_fwd_fp8", "attn_fwd_debug",
                 "attn_device_status", "attn_num_units", "attn_grid_size", "attn_fwd_splitkv",
                 "attn_fwd_splitkv_static", "attn_splitkv_default_splits", "attn_bwd"):
        getattr(L, name).restype = ctypes.c_int
    _lib = L
    return L


def status_str(status: int) -> str:
    try:
        return lib().attn_status_str(int(status)).decode()
    except RuntimeError:
        return "library not loaded"


def _check(rc: int, what: str):
    if rc != ATTN_OK:
        raise AttnError(rc, what)


def _torch():
    import torch
    return torch


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(t):
    torch = _torch()
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _need(t, name, dtype, shape=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (there is no CPU path)")
    if t.dtype != dtype:
        raise ValueError(f"{name} must have dtype {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _qkv_shape(q, k, v):
    if q.dim() != 4:
        raise ValueError("q must be [B, H, N, d]")
    for name, t in (("k", k), ("v", v)):
        if t.shape != q.shape:
            raise ValueError(f"{name} must have the shape of q {tuple(q.shape)}")
        if t.device != q.device:
            raise ValueError(f"{name} must be on {q.device}")
    return tuple(q.shape)


def attn_fwd(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None,
             return_lse: bool = True):
    """Exact attention forward (bf16).  Returns (O, lse); lse is None if not asked for."""
    torch = _torch()
    for name, t in (("q", q), ("k", k), ("v", v)):
        _need(t, name, torch.bfloat16)
    B, H, N, d = _qkv_shape(q, k, v)
    if scale is None:
        scale = d ** -0.5
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, q.shape)
    if lse is None and return_lse:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if lse is not None:
        _need(lse, "lse", torch.float32, (B, H, N))
    with torch.cuda.device(q.device):
        rc = lib().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, N, d,
                            float(scale), int(bool(causal)), ATTN_BF16, _stream(q))
    _check(rc, "attn_fwd")
    return out, lse


def attn_fwd_ex(q, k, v, causal: bool = False, window: int = 0, scale: float | None = None,
                out=None, lse=None, return_lse: bool = True):
    """attn_fwd with grouped-query heads (k, v: [B, H_kv, N, d], H_kv | H) and an
    optional causal sliding window of `window` keys.  Returns (O, lse)."""
    torch = _torch()
    for name, t in (("q", q), ("k", k), ("v", v)):
        _need(t, name, torch.bfloat16)
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("q, k, v must be [B, H, N, d] / [B, H_kv, N, d]")
    B, H, N, d = q.shape
    H_kv = k.shape[1]
    if tuple(k.shape) != (B, H_kv, N, d) or tuple(v.shape) != tuple(k.shape):
        raise ValueError(f"k and v must be [B, H_kv, N, d] = {(B, H_kv, N, d)}")
    if k.device != q.device or v.device != q.device:
        raise ValueError("q, k, v must be on one device")
    scale = d ** -0.5 if scale is None else scale
    out = torch.empty_like(q) if out is None else out
    _need(out, "out", torch.bfloat16, q.shape)
    if lse is None and return_lse:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if lse is not None:
        _need(lse, "lse", torch.float32, (B, H, N))
    with torch.cuda.device(q.device):
        rc = lib().attn_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, H_kv, N, d,
                               float(scale), int(bool(causal)), int(window), ATTN_BF16,
                               _stream(q))
    _check(rc, "attn_fwd_ex")
    return out, lse


def splitkv_workspace_bytes(B: int, H: int, N: int, d: int, num_splits: int) -> int:
    """Bytes of device workspace attn_fwd_splitkv needs (0 for invalid arguments)."""
    return int(lib().attn_splitkv_workspace_bytes(B, H, N, d, num_splits))


def splitkv_default_splits(B: int, H: int, N: int, d: int, causal: bool, num_sms: int) -> int:
    """Split count the library's time model picks for this shape on num_sms
    SMs (1 when the plain schedule fills them; 0 for invalid arguments)."""
    return int(lib().attn_splitkv_default_splits(B, H, N, d, int(bool(causal)), num_sms))


def attn_fwd_splitkv(q, k, v, causal: bool = False, window: int = 0, scale: float | None = None,
                     num_splits: int | None = None, workspace=None, out=None, lse=None,
                     return_lse: bool = True):
    """Split-KV attention forward (k, v may have fewer heads, as attn_fwd_ex).
    num_splits defaults to the count that fills the device; workspace (a CUDA
    uint8 tensor of at least splitkv_workspace_bytes(...) bytes) is allocated
    here when not given.  Returns (O, lse)."""
    torch = _torch()
    for name, t in (("q", q), ("k", k), ("v", v)):
        _need(t, name, torch.bfloat16)
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("q, k, v must be [B, H, N, d] / [B, H_kv, N, d]")
    B, H, N, d = q.shape
    H_kv = k.shape[1]
    if tuple(k.shape) != (B, H_kv, N, d) or tuple(v.shape) != tuple(k.shape):
        raise ValueError(f"k and v must be [B, H_kv, N, d] = {(B, H_kv, N, d)}")
    if k.device != q.device or v.device != q.device:
        raise ValueError("q, k, v must be on one device")
    scale = d ** -0.5 if scale is None else scale
    if num_splits is None:
        sms = torch.cuda.get_device_properties(q.device).multi_processor_count
        num_splits = splitkv_default_splits(B, H, N, d, causal, sms)
    need = splitkv_workspace_bytes(B, H, N, d, num_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    _need(workspace, "workspace", torch.uint8)
    out = torch.empty_like(q) if out is None else out
    _need(out, "out", torch.bfloat16, q.shape)
    if lse is None and return_lse:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if lse is not None:
        _need(lse, "lse", torch.float32, (B, H, N))
    with torch.cuda.device(q.device):
        rc = lib().attn_fwd_splitkv(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, H_kv,
                                    N, d, float(scale), int(bool(causal)), int(window), ATTN_BF16,
                                    int(num_splits), _ptr(workspace), workspace.numel(),
                                    _stream(q))
    _check(rc, "attn_fwd_splitkv")
    return out, lse


def attn_fwd_splitkv_static(q, k, v, causal: bool = False, window: int = 0,
                            scale: float | None = None, num_splits: int | None = None, out=None,
                            lse=None, return_lse: bool = True):
    """attn_fwd_splitkv on the library's own 64 MiB scratch array: the C call
    allocates nothing, for callers that cannot call cudaMalloc (a host program
    that owns all device memory through its own pool, or a loop that must not
    take cudaMalloc's device-wide synchronisation).  Pass ``out`` and ``lse`` to
    keep this wrapper from allocating them through torch.  Calls share the one
    array and must not overlap in time.  Returns (O, lse)."""
    torch = _torch()
    for name, t in (("q", q), ("k", k), ("v", v)):
        _need(t, name, torch.bfloat16)
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("q, k, v must be [B, H, N, d] / [B, H_kv, N, d]")
    B, H, N, d = q.shape
    H_kv = k.shape[1]
    if tuple(k.shape) != (B, H_kv, N, d) or tuple(v.shape) != tuple(k.shape):
        raise ValueError(f"k and v must be [B, H_kv, N, d] = {(B, H_kv, N, d)}")
    scale = d ** -0.5 if scale is None else scale
    if num_splits is None:
        sms = torch.cuda.get_device_properties(q.device).multi_processor_count
        num_splits = splitkv_default_splits(B, H, N, d, causal, sms)
    out = torch.empty_like(q) if out is None else out
    _need(out, "out", torch.bfloat16, q.shape)
    if lse is None and return_lse:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if lse is not None:
        _need(lse, "lse", torch.float32, (B, H, N))
    with torch.cuda.device(q.device):
        rc = lib().attn_fwd_splitkv_static(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H,
                                           H_kv, N, d, float(scale), int(bool(causal)),
                                           int(window), ATTN_BF16, int(num_splits), _stream(q))
    _check(rc, "attn_fwd_splitkv_static")
    return out, lse


def bwd_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    """Bytes of device workspace attn_bwd needs (0 for invalid arguments)."""
    return int(lib().attn_bwd_workspace_bytes(B, H, N, d))


def attn_bwd(q, k, v, o, lse, dO, causal: bool = False, window: int = 0,
             scale: float | None = None, dq=None, dk=None, dv=None, workspace=None):
    """Gradients (dq, dk, dv) of attention given dO and the forward's o, lse.
    k, v may have fewer heads than q (grouped KV heads)."""
    torch = _torch()
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dO", dO)):
        _need(t, name, torch.bfloat16)
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("q, k, v must be [B, H, N, d] / [B, H_kv, N, d]")
    B, H, N, d = q.shape
    H_kv = k.shape[1]
    if tuple(k.shape) != (B, H_kv, N, d) or tuple(v.shape) != tuple(k.shape):
        raise ValueError(f"k and v must be [B, H_kv, N, d] = {(B, H_kv, N, d)}")
    for name, t in (("o", o), ("dO", dO)):
        if tuple(t.shape) != tuple(q.shape):
            raise ValueError(f"{name} must have the shape of q")
    _need(lse, "lse", torch.float32, (B, H, N))
    scale = d ** -0.5 if scale is None else scale
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _need(dq, "dq", torch.bfloat16, q.shape)
    _need(dk, "dk", torch.bfloat16, k.shape)
    _need(dv, "dv", torch.bfloat16, v.shape)
    need = bwd_workspace_bytes(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    _need(workspace, "workspace", torch.uint8)
    with torch.cuda.device(q.device):
        rc = lib().attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq),
                            _ptr(dk), _ptr(dv), B, H, H_kv, N, d, float(scale),
                            int(bool(causal)), int(window), _ptr(workspace), workspace.numel(),
                            _stream(q))
    _check(rc, "attn_bwd")
    return dq, dk, dv


def attn_fwd_debug(q, k, v, status, timeout_ns: int, skip_loads: int, causal: bool = False,
                   scale: float | None = None, out=None, lse=None):
    """attn_fwd with a caller status word (int32 CUDA tensor of 1) and wait limit."""
    torch = _torch()
    for name, t in (("q", q), ("k", k), ("v", v)):
        _need(t, name, torch.bfloat16)
    B, H, N, d = _qkv_shape(q, k, v)
    _need(status, "status", torch.int32, (1,))
    scale = d ** -0.5 if scale is None else scale
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    with torch.cuda.device(q.device):
        rc = lib().attn_fwd_debug(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, N, d,
                                  float(scale), int(bool(causal)), _ptr(status),
                                  int(timeout_ns), int(skip_loads), _stream(q))
    _check(rc, "attn_fwd_debug")
    return out, lse


def fp8_prep(x, signs=None, transpose: bool = False, out=None, scales=None):
    """E4M3 operand preparation.  Returns (codes uint8, block scales f32 [B, H, nblk])."""
    torch = _torch()
    _need(x, "x", torch.bfloat16)
    if x.dim() != 4:
        raise ValueError("x must be [B, H, N, d]")
    B, H, N, d = x.shape
    nblk = (N + 127) // 128
    if signs is not None:
        _need(signs, "signs", torch.int8, (H, d))
    shape = (B, H, d, nblk * 128) if transpose else (B, H, N, d)
    out = torch.empty(shape, dtype=torch.uint8, device=x.device) if out is None else out
    _need(out, "out", torch.uint8, shape)
    scales = torch.empty((B, H, nblk), dtype=torch.float32, device=x.device) if scales is None \
        else scales
    _need(scales, "scales", torch.float32, (B, H, nblk))
    with torch.cuda.device(x.device):
        rc = lib().attn_fp8_prep(_ptr(x), _ptr(out), _ptr(scales), _ptr(signs), B, H, N, d,
                                 int(bool(transpose)), _stream(x))
    _check(rc, "attn_fp8_prep")
    return out, scales


def attn_fwd_fp8(q8, k8, v8t, q_scale, k_scale, v_scale, causal: bool = False,
                 scale: float | None = None, out=None, lse=None, return_lse: bool = True):
    """Exact attention forward on E4M3 operands from fp8_prep.  Returns (O bf16, lse)."""
    torch = _torch()
    _need(q8, "q8", torch.uint8)
    if q8.dim() != 4:
        raise ValueError("q8 must be [B, H, N, d]")
    B, H, N, d = q8.shape
    nblk = (N + 127) // 128
    _need(k8, "k8", torch.uint8, q8.shape)
    _need(v8t, "v8t", torch.uint8, (B, H, d, nblk * 128))
    for name, t in (("q_scale", q_scale), ("k_scale", k_scale), ("v_scale", v_scale)):
        _need(t, name, torch.float32, (B, H, nblk))
    scale = d ** -0.5 if scale is None else scale
    out = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=q8.device) if out is None \
        else out
    _need(out, "out", torch.bfloat16, (B, H, N, d))
    if lse is None and return_lse:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q8.device)
    if lse is not None:
        _need(lse, "lse", torch.float32, (B, H, N))
    with torch.cuda.device(q8.device):
        rc = lib().attn_fwd_fp8(_ptr(q8), _ptr(k8), _ptr(v8t), _ptr(q_scale), _ptr(k_scale),
                                _ptr(v_scale), _ptr(out), _ptr(lse), B, H, N, d, float(scale),
                                int(bool(causal)), _stream(q8))
    _check(rc, "attn_fwd_fp8")
    return out, lse


def attn_fwd_fp8_from_bf16(q, k, v, signs, causal: bool = False, scale: float | None = None):
    """Prepare Q, K (rotated with `signs`) and V (transposed), then run FP8 attention."""
    q8, sq = fp8_prep(q, signs)
    k8, sk = fp8_prep(k, signs)
    v8t, sv = fp8_prep(v, None, transpose=True)
    return attn_fwd_fp8(q8, k8, v8t, sq, sk, sv, causal=causal, scale=scale)


def device_status(clear: bool = True) -> int:
    """Synchronise and return the kernels' status word (ATTN_OK or ATTN_ERR_TIMEOUT)."""
    return lib().attn_device_status(int(bool(clear)))


def num_units(B: int, H: int, N: int) -> int:
    return lib().attn_num_units(B, H, N)


def grid_size(B: int, H: int, N: int, num_sms: int) -> int:
    return lib().attn_grid_size(B, H, N, num_sms)
