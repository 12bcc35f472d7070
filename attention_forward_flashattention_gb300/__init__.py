"""GB300-native (sm_103a) fused attention forward.

A thin ctypes binding over the C ABI in ``include/fa.h``. Every step of the
computation runs in the CUDA library ``_build/libfa_sm103.so``; this module
only marshals arguments (torch tensors -> device pointers, streams -> handles).
There is no fallback: if the library is missing or cannot be loaded, calls
raise.

    import torch
    from attention_forward_flashattention_gb300 import attention_forward
    o, lse = attention_forward(q, k, v, causal=True)   # q, k, v: [B, H, N, d] fp16/bf16 on cuda
"""
from __future__ import annotations

import ctypes
import math
import os
import re
import threading

from . import build as _build

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_CUDA = 3
FA_ERR_ARCH = 4
FA_ERR_TIMEOUT = 5
FA_DTYPE_FP16 = 0
FA_DTYPE_BF16 = 1

HEADER = os.path.join(_build.ROOT, "include", "fa.h")

_lock = threading.Lock()
_lib = None


class FaStrides(ctypes.Structure):
    """fa_strides: element strides of a [B][H][N][d] view (d stride 1)."""
    _fields_ = [("b", ctypes.c_longlong), ("h", ctypes.c_longlong), ("n", ctypes.c_longlong)]


class FaError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} ({status})")
        self.status = status


def header_functions() -> list[str]:
    """Names of the entry points that include/fa.h declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:fa_status|const char\s*\*|int)\s+(fa_\w+)\s*\(", text, flags=re.M)


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Loads libfa_sm103.so (built in-tree by build.build()). Raises if absent."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or _build.lib_path()
        if not os.path.exists(p):
            raise RuntimeError(f"CUDA library not built: {p} (run __graft_entry__.build())")
        lib = ctypes.CDLL(p)
        vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
        lib.fa_fwd.restype = i
        lib.fa_fwd_pair.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
        lib.fa_fwd_pair.restype = i
        if hasattr(lib, "fa_fwd_strided"):
            lib.fa_fwd_strided.argtypes = [vp, vp, vp, vp, vp, i, i, i, i,
                                           ctypes.POINTER(FaStrides), i, f, i, vp]
            lib.fa_fwd_strided.restype = i
        for fn in ("fa_fwd_fp8", "fa_fwd_fp8_pair"):
            if hasattr(lib, fn):
                getattr(lib, fn).argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, vp, f, i, f, vp]
                getattr(lib, fn).restype = i
        if hasattr(lib, "fa_bwd"):
            lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
            lib.fa_bwd.restype = i
            lib.fa_bwd_workspace_size.argtypes = [i, i, i, i, ctypes.POINTER(ctypes.c_size_t)]
            lib.fa_bwd_workspace_size.restype = i
        if hasattr(lib, "fa_fwd_host"):
            lib.fa_fwd_host.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp,
                                        ctypes.c_size_t, vp]
            lib.fa_fwd_host.restype = i
            lib.fa_fwd_host_workspace_size.argtypes = [i, i, i, i,
                                                       ctypes.POINTER(ctypes.c_size_t)]
            lib.fa_fwd_host_workspace_size.restype = i
        lib.fa_fwd_noalloc.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
        lib.fa_fwd_noalloc.restype = i
        lib.fa_check.argtypes = [vp]
        lib.fa_check.restype = i
        lib.fa_sm_clock_read.argtypes = [vp, ctypes.POINTER(ctypes.c_double),
                                         ctypes.POINTER(ctypes.c_ulonglong)]
        lib.fa_sm_clock_read.restype = i
        ip = ctypes.POINTER(ctypes.c_int)
        lib.fa_query_launch.argtypes = [i, i, i, i, i, ip, ip, ip, ip, ip]
        lib.fa_query_launch.restype = i
        lib.fa_sm_clock_probe.argtypes = [vp, ctypes.c_longlong, vp]
        lib.fa_sm_clock_probe.restype = i
        lib.fa_status_string.argtypes = [i]
        lib.fa_status_string.restype = ctypes.c_char_p
        lib.fa_version.argtypes = []
        lib.fa_version.restype = i
        if path is None:
            _lib = lib
        return lib


def status_string(status: int) -> str:
    return load_library().fa_status_string(int(status)).decode()


# ------------------------------------------------------------ raw C ABI

def fa_fwd(q: int, k: int, v: int, o: int, lse: int, B: int, H: int, N: int, d: int,
           causal: bool, scale: float, dtype: int, stream: int = 0) -> int:
    """Same arguments as the C function (device pointers as ints); returns the status."""
    return load_library().fa_fwd(q, k, v, o, lse, B, H, N, d, int(bool(causal)), float(scale),
                                 int(dtype), stream)


def fa_fwd_pair(q: int, k: int, v: int, o: int, lse: int, B: int, H: int, N: int, d: int,
                causal: bool, scale: float, dtype: int, stream: int = 0) -> int:
    """The CTA-pair forward (same arguments as fa_fwd, d = 128); returns the status."""
    return load_library().fa_fwd_pair(q, k, v, o, lse, B, H, N, d, int(bool(causal)),
                                      float(scale), int(dtype), stream)


def fa_fwd_strided(q: int, k: int, v: int, o: int, lse: int, B: int, H: int, N: int, d: int,
                   strides, causal: bool, scale: float, dtype: int, stream: int = 0) -> int:
    """fa_fwd on strided [B][H][N][d] views; strides: 4 (b, h, n) element-stride
    triples for q, k, v, o (None passes a null pointer). Returns the status."""
    arr = None
    if strides is not None:
        arr = (FaStrides * 4)(*[FaStrides(*map(int, s)) for s in strides])
    return load_library().fa_fwd_strided(q, k, v, o, lse, B, H, N, d, arr, int(bool(causal)),
                                         float(scale), int(dtype), stream)


def fa_fwd_fp8(q: int, k: int, vt: int, o: int, lse: int, B: int, H: int, N: int, d: int,
               ldv: int, q_scale: float, k_scales: int, v_scale: float, causal: bool,
               scale: float, stream: int = 0) -> int:
    """Same arguments as the C function (device pointers as ints); returns the status."""
    return load_library().fa_fwd_fp8(q, k, vt, o, lse, B, H, N, d, ldv, float(q_scale), k_scales,
                                     float(v_scale), int(bool(causal)), float(scale), stream)


def fa_fwd_fp8_pair(q: int, k: int, vt: int, o: int, lse: int, B: int, H: int, N: int, d: int,
                    ldv: int, q_scale: float, k_scales: int, v_scale: float, causal: bool,
                    scale: float, stream: int = 0) -> int:
    """fa_fwd_fp8 on CTA pairs; same arguments (device pointers as ints)."""
    return load_library().fa_fwd_fp8_pair(q, k, vt, o, lse, B, H, N, d, ldv, float(q_scale),
                                          k_scales, float(v_scale), int(bool(causal)),
                                          float(scale), stream)


def fa_bwd(q: int, k: int, v: int, o: int, dout: int, lse: int, dq: int, dk: int, dv: int,
           workspace: int, B: int, H: int, N: int, d: int, causal: bool, scale: float,
           dtype: int, stream: int = 0) -> int:
    """Same arguments as the C function (device pointers as ints); returns the status."""
    return load_library().fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, workspace, B, H, N, d,
                                 int(bool(causal)), float(scale), int(dtype), stream)


def fa_bwd_workspace_size(B: int, H: int, N: int, d: int) -> int:
    n = ctypes.c_size_t(0)
    rc = load_library().fa_bwd_workspace_size(B, H, N, d, ctypes.byref(n))
    if rc != FA_OK:
        raise FaError(rc, "fa_bwd_workspace_size")
    return int(n.value)


def fa_fwd_host(q: int, k: int, v: int, o: int, lse: int, B: int, H: int, N: int, d: int,
                causal: bool, scale: float, dtype: int, workspace: int, workspace_size: int,
                stream: int = 0) -> int:
    """Same arguments as the C function (host q, k, v, o, lse and a device
    workspace, pointers as ints); returns the status."""
    return load_library().fa_fwd_host(q, k, v, o, lse, B, H, N, d, int(bool(causal)),
                                      float(scale), int(dtype), workspace, int(workspace_size),
                                      stream)


def fa_fwd_host_workspace_size(B: int, H: int, N: int, d: int) -> int:
    n = ctypes.c_size_t(0)
    rc = load_library().fa_fwd_host_workspace_size(B, H, N, d, ctypes.byref(n))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_host_workspace_size")
    return int(n.value)


def fa_fwd_noalloc(q: int, k: int, v: int, o: int, lse: int, B: int, H: int, N: int, d: int,
                   causal: bool, scale: float, dtype: int, stream: int = 0) -> int:
    """The allocation-free variant of fa_fwd (same arguments); returns the status."""
    return load_library().fa_fwd_noalloc(q, k, v, o, lse, B, H, N, d, int(bool(causal)),
                                         float(scale), int(dtype), stream)


def fa_check(stream: int = 0) -> int:
    return load_library().fa_check(stream)


def fa_sm_clock_read(stream: int = 0) -> tuple[float, int]:
    """(SM MHz the kernels ran at since the last read, CTAs recorded); clears
    the record. Synchronises the stream."""
    mhz, ctas = ctypes.c_double(0.0), ctypes.c_ulonglong(0)
    rc = load_library().fa_sm_clock_read(stream, ctypes.byref(mhz), ctypes.byref(ctas))
    if rc != FA_OK:
        raise FaError(rc, "fa_sm_clock_read")
    return float(mhz.value), int(ctas.value)


def fa_query_launch(B: int, H: int, N: int, d: int, causal: bool = False) -> dict:
    g, t, s, u, c = (ctypes.c_int(0) for _ in range(5))
    rc = load_library().fa_query_launch(B, H, N, d, int(bool(causal)), ctypes.byref(g),
                                        ctypes.byref(t), ctypes.byref(s), ctypes.byref(u),
                                        ctypes.byref(c))
    if rc != FA_OK:
        raise FaError(rc, "fa_query_launch")
    return {"grid": g.value, "threads": t.value, "smem_bytes": s.value, "units": u.value,
            "cluster": c.value}


def fa_sm_clock_probe(out_ptr: int, cycles: int, stream: int = 0) -> int:
    return load_library().fa_sm_clock_probe(out_ptr, int(cycles), stream)


def fa_version() -> int:
    return load_library().fa_version()


# ------------------------------------------------------------ torch helpers

def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float16:
        return FA_DTYPE_FP16
    if t.dtype == torch.bfloat16:
        return FA_DTYPE_BF16
    raise TypeError(f"unsupported dtype {t.dtype} (fp16 or bf16)")


def _allocating_on(stream):
    """Context for the tensors a call creates (outputs, workspace): with an
    explicit stream they are allocated on it, so PyTorch's caching allocator
    reuses their memory only in that stream's order, never while the call's
    kernels may still be running."""
    import contextlib
    import torch
    return torch.cuda.stream(stream) if stream is not None else contextlib.nullcontext()


def _stream_handle(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def attention_forward_into(q, k, v, o, lse, causal: bool = False, scale: float | None = None,
                           stream=None) -> None:
    """Enqueues the forward on torch tensors: q, k, v, o are [B, H, N, d] CUDA
    views with unit stride along d (any other strides that are multiples of 8
    elements, e.g. a [B, N, H, d] tensor passed as .transpose(1, 2)); lse is a
    contiguous [B, H, N] float32 tensor."""
    B, H, N, d = q.shape
    for t in (q, k, v, o):
        if tuple(t.shape) != (B, H, N, d) or t.stride(-1) != 1 or not t.is_cuda:
            raise ValueError("q, k, v, o must be [B, H, N, d] CUDA tensors with unit d stride")
    if tuple(lse.shape) != (B, H, N) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous [B, H, N] float32 CUDA tensor")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if all(t.is_contiguous() for t in (q, k, v, o)):
        rc = fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                    B, H, N, d, causal, scale, _dtype_code(q), _stream_handle(stream))
        what = "fa_fwd"
    else:
        strides = [t.stride()[:3] for t in (q, k, v, o)]
        rc = fa_fwd_strided(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                            lse.data_ptr(), B, H, N, d, strides, causal, scale, _dtype_code(q),
                            _stream_handle(stream))
        what = "fa_fwd_strided"
    if rc != FA_OK:
        raise FaError(rc, what)


def attention_forward_pair_into(q, k, v, o, lse, causal: bool = False,
                                scale: float | None = None, stream=None) -> None:
    """Enqueues fa_fwd_pair (CTA-pair kernel) on contiguous [B, H, N, 128]
    CUDA tensors q, k, v, o (fp16 / bf16) and a contiguous float32 [B, H, N] lse."""
    B, H, N, d = q.shape
    for t in (q, k, v, o):
        if tuple(t.shape) != (B, H, N, d) or not (t.is_cuda and t.is_contiguous()):
            raise ValueError("q, k, v, o must be contiguous [B, H, N, d] CUDA tensors")
    if tuple(lse.shape) != (B, H, N) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous [B, H, N] float32 CUDA tensor")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    rc = fa_fwd_pair(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                     B, H, N, d, causal, scale, _dtype_code(q), _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_pair")


def attention_forward(q, k, v, causal: bool = False, scale: float | None = None, stream=None):
    """Returns (O [B, H, N, d] in q's dtype, LSE [B, H, N] float32)."""
    import torch
    B, H, N, d = q.shape
    with _allocating_on(stream):
        o = torch.empty_like(q)
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    attention_forward_into(q, k, v, o, lse, causal, scale, stream)
    return o, lse


def attention_forward_host_into(q, k, v, o, lse, workspace, causal: bool = False,
                                scale: float | None = None, stream=None) -> None:
    """Enqueues fa_fwd_host: q, k, v, o contiguous CPU tensors [B, H, N, d] of
    one dtype (fp16 / bf16; page-locked for copy / compute overlap), lse a
    contiguous CPU float32 [B, H, N] tensor, workspace a CUDA uint8 tensor of
    at least fa_fwd_host_workspace_size(B, H, N, d) bytes. o and lse hold the
    result once the stream has passed the call."""
    import torch
    B, H, N, d = q.shape
    ok = (all(tuple(t.shape) == (B, H, N, d) and t.dtype == q.dtype for t in (k, v, o))
          and tuple(lse.shape) == (B, H, N) and lse.dtype == torch.float32
          and all(not t.is_cuda and t.is_contiguous() for t in (q, k, v, o, lse))
          and workspace.is_cuda and workspace.is_contiguous())
    if not ok:
        raise ValueError("fa_fwd_host: bad shapes, dtypes or devices")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    nbytes = workspace.numel() * workspace.element_size()
    with torch.cuda.device(workspace.device):
        rc = fa_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                         B, H, N, d, causal, scale, _dtype_code(q), workspace.data_ptr(), nbytes,
                         _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_host")


def attention_forward_host(q, k, v, causal: bool = False, scale: float | None = None,
                           device=None):
    """Forward of CPU tensors on the GPU `device` (default: the current one):
    returns (O, LSE) as page-locked CPU tensors, synchronised."""
    import torch
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None \
        else torch.device(device)
    B, H, N, d = q.shape
    o = torch.empty(q.shape, dtype=q.dtype).pin_memory()
    lse = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    ws = torch.empty(fa_fwd_host_workspace_size(B, H, N, d), dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        stream = torch.cuda.current_stream(dev)
        attention_forward_host_into(q, k, v, o, lse, ws, causal, scale, stream)
        stream.synchronize()
    return o, lse


def attention_forward_fp8_into(q8, k8, vt8, o, lse, q_scale: float, k_scales, v_scale: float,
                               causal: bool = False, scale: float | None = None,
                               stream=None, pair: bool = False) -> None:
    """Enqueues fa_fwd_fp8 (fa_fwd_fp8_pair if `pair`): q8, k8 [B, H, N, 128]
    and vt8 [B, H, 128, ldv] (V transposed) contiguous CUDA tensors of e4m3
    codes (uint8 or float8_e4m3fn), k_scales a contiguous float32
    [B, H, ceil(N / 128)] CUDA tensor, o a contiguous bfloat16 [B, H, N, 128]
    tensor, lse a contiguous float32 [B, H, N] tensor."""
    import torch
    B, H, N, d = q8.shape
    ldv = vt8.shape[-1]
    ok = (tuple(k8.shape) == (B, H, N, d) and tuple(vt8.shape) == (B, H, d, ldv)
          and tuple(o.shape) == (B, H, N, d) and o.dtype == torch.bfloat16
          and tuple(lse.shape) == (B, H, N) and lse.dtype == torch.float32
          and tuple(k_scales.shape) == (B, H, (N + 127) // 128)
          and k_scales.dtype == torch.float32
          and all(t.element_size() == 1 for t in (q8, k8, vt8))
          and all(t.is_cuda and t.is_contiguous() for t in (q8, k8, vt8, o, lse, k_scales)))
    if not ok:
        raise ValueError("fa_fwd_fp8: bad shapes, dtypes or layouts")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    fn = fa_fwd_fp8_pair if pair else fa_fwd_fp8
    rc = fn(q8.data_ptr(), k8.data_ptr(), vt8.data_ptr(), o.data_ptr(), lse.data_ptr(),
            B, H, N, d, ldv, q_scale, k_scales.data_ptr(), v_scale, causal, scale,
            _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, fn.__name__)


def attention_forward_fp8(q8, k8, vt8, q_scale: float, k_scales, v_scale: float,
                          causal: bool = False, scale: float | None = None, stream=None):
    """Returns (O bfloat16 [B, H, N, 128], LSE float32 [B, H, N]) of the 8-bit forward."""
    import torch
    B, H, N, d = q8.shape
    with _allocating_on(stream):
        o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=q8.device)
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q8.device)
    attention_forward_fp8_into(q8, k8, vt8, o, lse, q_scale, k_scales, v_scale, causal, scale,
                               stream)
    return o, lse


def attention_backward(q, k, v, o, lse, dout, causal: bool = False, scale: float | None = None,
                       stream=None):
    """Gradients (dq, dk, dv) of the forward at q, k, v for the output
    gradient dout; o and lse are the forward's outputs. All [B, H, N, d]
    contiguous CUDA tensors of one dtype (fp16 / bf16), lse [B, H, N] float32."""
    import torch
    B, H, N, d = q.shape
    for t in (k, v, o, dout):
        if tuple(t.shape) != (B, H, N, d) or t.dtype != q.dtype:
            raise ValueError("q, k, v, o, dout must share shape [B, H, N, d] and dtype")
    for t in (q, k, v, o, dout, lse):
        if not (t.is_cuda and t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    # the workspace is freed when this returns, possibly before the kernels
    # that use it have run: allocated on their stream, it is reused only after
    with _allocating_on(stream):
        ws = torch.empty(fa_bwd_workspace_size(B, H, N, d) // 4, dtype=torch.float32,
                         device=q.device)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    rc = fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(),
                lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), ws.data_ptr(),
                B, H, N, d, causal, scale, _dtype_code(q), _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_bwd")
    return dq, dk, dv


_autograd_fn = None


def _attention_function():
    """The torch.autograd.Function behind `attention` (built on first use, so
    importing this module does not import torch)."""
    global _autograd_fn
    if _autograd_fn is None:
        import torch

        class _Attention(torch.autograd.Function):
            @staticmethod
            def forward(ctx, q, k, v, causal, scale):
                o, lse = attention_forward(q, k, v, causal=causal, scale=scale)
                ctx.save_for_backward(q, k, v, o, lse)
                ctx.causal, ctx.scale = causal, scale
                return o

            @staticmethod
            def backward(ctx, do):
                q, k, v, o, lse = ctx.saved_tensors
                dq, dk, dv = attention_backward(*(t.contiguous() for t in (q, k, v, o)), lse,
                                                do.contiguous(), causal=ctx.causal,
                                                scale=ctx.scale)
                return dq, dk, dv, None, None

        _autograd_fn = _Attention
    return _autograd_fn


def attention(q, k, v, causal: bool = False, scale: float | None = None):
    """O = softmax(scale q k^T [+ causal mask]) v for [B, H, N, d] fp16 / bf16
    CUDA tensors (d = 64 or 128), differentiable: autograd runs fa_bwd on the
    saved q, k, v, O and LSE. Returns O only (attention_forward also returns
    the LSE)."""
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    return _attention_function().apply(q, k, v, bool(causal), float(scale))
