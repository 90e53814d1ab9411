"""GB300-native fused attention forward (online-softmax tiling), Python binding.

Argument marshalling only: every step of the computation runs in the sm_103a
kernels of ``libfa_gb300.so`` behind the C ABI of ``include/fa.h``.  The names
follow that header: ``fa_fwd``, ``fa_check_device_status``,
``fa_status_string``, ``fa_version`` and ``fa_fwd_debug``.  There is no CPU
fallback: if the library is missing, the first call raises.

``attention_forward`` is a convenience wrapper over ``fa_fwd`` for torch
tensors; torch is used only to allocate device memory and to name the stream.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_MISALIGNED, FA_ERR_CUDA, FA_ERR_TIMEOUT = (
    0, 1, 2, 3, 4, 5)
FA_FP16, FA_BF16 = 0, 1

_HERE = os.path.dirname(os.path.abspath(__file__))
LIBRARY = os.path.join(_HERE, "libfa_gb300.so")
EXPORTS = ("fa_fwd", "fa_check_device_status", "fa_status_string", "fa_version", "fa_fwd_debug",
           "fa_splitkv_num_splits", "fa_splitkv_workspace_size", "fa_fwd_splitkv",
           "fa_fwd_splitkv_noalloc", "fa_fwd_ex", "fa_ceiling_ex2_rate", "fa_ceiling_l2_read",
           "fa_naive_fwd", "fa_naive_workspace_size", "fa_splitkv_num_splits_ex")
FA_CEIL_OK, FA_CEIL_ERR_ARG, FA_CEIL_ERR_CUDA = 0, 1, 4
FA_MASK_NONE, FA_MASK_CAUSAL_TOP_LEFT, FA_MASK_CAUSAL_BOTTOM_RIGHT = 0, 1, 2


class fa_fwd_args(ctypes.Structure):
    """Mirror of `fa_fwd_args` in include/fa.h (same field order and types)."""
    _fields_ = [("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("o", ctypes.c_void_p), ("lse", ctypes.c_void_p),
                ("B", ctypes.c_int), ("H", ctypes.c_int), ("Nq", ctypes.c_int),
                ("Nk", ctypes.c_int), ("d", ctypes.c_int),
                ("q_stride", ctypes.c_longlong * 3), ("k_stride", ctypes.c_longlong * 3),
                ("v_stride", ctypes.c_longlong * 3), ("o_stride", ctypes.c_longlong * 3),
                ("lse_stride", ctypes.c_longlong * 2),
                ("scale", ctypes.c_float), ("mask", ctypes.c_int), ("dtype", ctypes.c_int),
                ("num_splits", ctypes.c_int), ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_size_t), ("stream", ctypes.c_void_p)]
FA_NOALLOC_SCRATCH_BYTES = 16 << 20
FA_MAX_SPLITS = 32

_lock = threading.Lock()
_lib = None


class FaError(RuntimeError):
    def __init__(self, status: int, what: str = "fa_fwd"):
        self.status = status
        super().__init__(f"{what} failed: {fa_status_string(status)} ({status})")


def library() -> ctypes.CDLL:
    """The loaded C-ABI library (built by ``online_softmax_tiling_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIBRARY):
                raise FileNotFoundError(
                    f"{LIBRARY} is missing: build it with "
                    "`python -m online_softmax_tiling_gb300.build` (there is no CPU fallback)")
            lib = ctypes.CDLL(LIBRARY)
            vp, i = ctypes.c_void_p, ctypes.c_int
            lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, ctypes.c_float, i, i, vp]
            lib.fa_fwd.restype = i
            lib.fa_fwd_debug.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, ctypes.c_float, i, i, vp,
                                         i, ctypes.c_double]
            lib.fa_fwd_debug.restype = i
            lib.fa_check_device_status.argtypes = [vp]
            lib.fa_check_device_status.restype = i
            lib.fa_status_string.argtypes = [i]
            lib.fa_status_string.restype = ctypes.c_char_p
            lib.fa_version.argtypes = []
            lib.fa_version.restype = i
            lib.fa_splitkv_num_splits.argtypes = [i, i, i, i, i]
            lib.fa_splitkv_num_splits.restype = i
            lib.fa_splitkv_workspace_size.argtypes = [i, i, i, i, i]
            lib.fa_splitkv_workspace_size.restype = ctypes.c_size_t
            lib.fa_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, ctypes.c_float, i, i, i,
                                           vp, ctypes.c_size_t, vp]
            lib.fa_fwd_splitkv.restype = i
            lib.fa_fwd_splitkv_noalloc.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, ctypes.c_float,
                                                   i, i, i, vp]
            lib.fa_fwd_splitkv_noalloc.restype = i
            lib.fa_fwd_ex.argtypes = [ctypes.POINTER(fa_fwd_args)]
            lib.fa_fwd_ex.restype = i
            lib.fa_splitkv_num_splits_ex.argtypes = [ctypes.POINTER(fa_fwd_args)]
            lib.fa_splitkv_num_splits_ex.restype = i
            lib.fa_ceiling_ex2_rate.argtypes = [ctypes.POINTER(ctypes.c_double), vp]
            lib.fa_ceiling_ex2_rate.restype = i
            lib.fa_ceiling_l2_read.argtypes = [vp, ctypes.c_size_t, ctypes.POINTER(ctypes.c_double), vp]
            lib.fa_ceiling_l2_read.restype = i
            lib.fa_naive_workspace_size.argtypes = [i, i, i]
            lib.fa_naive_workspace_size.restype = ctypes.c_size_t
            lib.fa_naive_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, ctypes.c_float, i, i, vp,
                                         ctypes.c_size_t, vp]
            lib.fa_naive_fwd.restype = i
            _lib = lib
        return _lib


def fa_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, stream) -> int:
    """Raw C call: q, k, v, o, lse and stream are integer addresses (or None)."""
    return library().fa_fwd(q, k, v, o, lse, int(B), int(H), int(N), int(d), float(scale),
                            int(causal), int(dtype), stream)


def fa_fwd_debug(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, stream, fault_mode,
                 timeout_s) -> int:
    return library().fa_fwd_debug(q, k, v, o, lse, int(B), int(H), int(N), int(d), float(scale),
                                  int(causal), int(dtype), stream, int(fault_mode),
                                  float(timeout_s))


def fa_splitkv_num_splits(B, H, N, d, causal) -> int:
    return library().fa_splitkv_num_splits(int(B), int(H), int(N), int(d), int(causal))


def fa_splitkv_workspace_size(B, H, N, d, num_splits) -> int:
    return library().fa_splitkv_workspace_size(int(B), int(H), int(N), int(d), int(num_splits))


def fa_fwd_splitkv(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, num_splits, workspace,
                   workspace_bytes, stream) -> int:
    """Raw C call of the split-KV entry point (addresses as integers or None)."""
    return library().fa_fwd_splitkv(q, k, v, o, lse, int(B), int(H), int(N), int(d),
                                    float(scale), int(causal), int(dtype), int(num_splits),
                                    workspace, int(workspace_bytes), stream)


def fa_fwd_splitkv_noalloc(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, num_splits,
                           stream) -> int:
    """Split-KV with the partials in the library's fixed scratch array, for
    callers that cannot allocate device memory (see include/fa.h)."""
    return library().fa_fwd_splitkv_noalloc(q, k, v, o, lse, int(B), int(H), int(N), int(d),
                                            float(scale), int(causal), int(dtype),
                                            int(num_splits), stream)


def fa_fwd_ex(args: "fa_fwd_args") -> int:
    """Raw C call of the general entry point with a filled `fa_fwd_args`."""
    return library().fa_fwd_ex(ctypes.byref(args))


def fa_naive_workspace_size(B, H, N) -> int:
    return library().fa_naive_workspace_size(int(B), int(H), int(N))


def fa_naive_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, workspace, workspace_bytes,
                 stream) -> int:
    """Raw C call of the step-by-step baseline (include/fa_naive.h)."""
    return library().fa_naive_fwd(q, k, v, o, lse, int(B), int(H), int(N), int(d), float(scale),
                                  int(causal), int(dtype), workspace, int(workspace_bytes), stream)


def _stream_handle(stream):
    """A cudaStream_t address from None, an integer or a torch stream."""
    if stream is None or isinstance(stream, int):
        return stream
    return stream.cuda_stream


def fa_ceiling_ex2_rate(stream=None) -> float:
    """2^x evaluations per second on the current device (include/fa_ceilings.h)."""
    out = ctypes.c_double()
    st = library().fa_ceiling_ex2_rate(ctypes.byref(out), _stream_handle(stream))
    if st != FA_CEIL_OK:
        raise FaError(FA_ERR_CUDA, "fa_ceiling_ex2_rate")
    return out.value


def fa_ceiling_l2_read(buf, nbytes: int, stream=None) -> float:
    """L2 -> SM read bytes per second over `nbytes` at device address `buf`."""
    out = ctypes.c_double()
    st = library().fa_ceiling_l2_read(buf, nbytes, ctypes.byref(out), _stream_handle(stream))
    if st != FA_CEIL_OK:
        raise FaError(FA_ERR_CUDA if st == FA_CEIL_ERR_CUDA else FA_ERR_INVALID_ARG,
                      "fa_ceiling_l2_read")
    return out.value


def fa_splitkv_num_splits_ex(args: "fa_fwd_args") -> int:
    """Split count fa_fwd_ex uses for num_splits = 0 with these arguments."""
    return library().fa_splitkv_num_splits_ex(ctypes.byref(args))


def fa_check_device_status(stream=None) -> int:
    return library().fa_check_device_status(stream)


def fa_status_string(status: int) -> str:
    try:
        return library().fa_status_string(int(status)).decode()
    except FileNotFoundError:
        return f"status {status}"


def fa_version() -> int:
    return library().fa_version()


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float16:
        return FA_FP16
    if t.dtype == torch.bfloat16:
        return FA_BF16
    raise TypeError(f"unsupported dtype {t.dtype} (float16 or bfloat16)")


def _checked(stream_handle, what: str):
    """Wait for the stream and raise FaError if a kernel reported a status."""
    st = fa_check_device_status(stream_handle)
    if st != FA_OK:
        raise FaError(st, what)


def attention_forward(q, k, v, scale: float | None = None, causal: bool = False, out=None,
                      lse=None, stream=None, num_splits: int = 1, check: bool = False):
    """O, LSE for contiguous CUDA tensors q, k, v of shape [B, H, N, d].

    scale defaults to 1/sqrt(d).  Outputs are allocated with torch unless
    given.  num_splits: 1 = one fused launch (fa_fwd); 0 = let the library
    choose a split-KV count for shapes that cannot fill the GPU; >= 2 = that
    many key ranges (fa_fwd_splitkv, with a workspace allocated by torch).
    Raises FaError on any non-OK status of the call.  Asynchronous on
    `stream` (default: torch's current stream).

    IMPORTANT: a kernel whose pipeline wait runs out of time (2 s) leaves its
    outputs unwritten and reports FA_ERR_TIMEOUT only through the device
    status word.  With check=True this call synchronises the stream and raises
    FaError if that happened; otherwise the caller must call
    fa_check_device_status() before trusting the outputs.
    """
    import torch
    if q.dim() != 4 or q.shape != k.shape or q.shape != v.shape:
        raise ValueError("q, k, v must be [B, H, N, d] of one shape")
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out), ("lse", lse)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else stream
    if num_splits == 0:
        num_splits = fa_splitkv_num_splits(B, H, N, d, causal)
    if num_splits == 1:
        st = fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B, H,
                    N, d, scale, causal, _dtype_code(q), handle)
    else:
        nbytes = fa_splitkv_workspace_size(B, H, N, d, num_splits)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
        st = fa_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                            lse.data_ptr(), B, H, N, d, scale, causal, _dtype_code(q), num_splits,
                            ws.data_ptr(), nbytes, handle)
    if st != FA_OK:
        raise FaError(st)
    if check:
        _checked(handle, "fa_fwd")
    return out, lse


def attention_forward_ex(q, k, v, scale: float | None = None, mask: int = FA_MASK_NONE,
                         out=None, lse=None, stream=None, num_splits: int = 1,
                         check: bool = False):
    """General form for CUDA tensors q [B, H, Nq, d], k, v [B, H, Nk, d] of any
    strides with d contiguous (e.g. transposed views of [B, N, H, d] data).

    mask: FA_MASK_NONE, FA_MASK_CAUSAL_TOP_LEFT or FA_MASK_CAUSAL_BOTTOM_RIGHT.
    out (O, [B, H, Nq, d]) and lse ([B, H, Nq], rows contiguous) may be strided
    too; they are allocated contiguous when not given.  num_splits and check
    as in attention_forward (without check, call fa_check_device_status()
    before trusting the outputs).
    """
    import torch
    if q.dim() != 4 or k.dim() != 4 or v.shape != k.shape or q.shape[:2] != k.shape[:2] \
            or q.shape[3] != k.shape[3]:
        raise ValueError("q: [B, H, Nq, d]; k, v: [B, H, Nk, d]")
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, H, Nq, d), dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out)):
        if not t.is_cuda or t.stride(3) != 1:
            raise ValueError(f"{name} must be a CUDA tensor with a contiguous last dimension")
    if not lse.is_cuda or lse.stride(2) != 1:
        raise ValueError("lse must be a CUDA tensor with contiguous rows")
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    a = fa_fwd_args()
    a.q, a.k, a.v, a.o, a.lse = q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), \
        lse.data_ptr()
    a.B, a.H, a.Nq, a.Nk, a.d = B, H, Nq, Nk, d
    for field, t in (("q_stride", q), ("k_stride", k), ("v_stride", v), ("o_stride", out)):
        getattr(a, field)[:] = [t.stride(0), t.stride(1), t.stride(2)]
    a.lse_stride[:] = [lse.stride(0), lse.stride(1)]
    a.scale, a.mask, a.dtype = float(scale), int(mask), _dtype_code(q)
    if num_splits == 0:
        num_splits = fa_splitkv_num_splits_ex(a)
    a.num_splits = num_splits
    ws = None
    if num_splits > 1:
        a.workspace_bytes = fa_splitkv_workspace_size(B, H, Nq, d, num_splits)
        ws = torch.empty(a.workspace_bytes, dtype=torch.uint8, device=q.device)
        a.workspace = ws.data_ptr()
    a.stream = stream.cuda_stream if hasattr(stream, "cuda_stream") else stream
    st = fa_fwd_ex(a)
    if st != FA_OK:
        raise FaError(st, "fa_fwd_ex")
    if check:
        _checked(a.stream, "fa_fwd_ex")
    return out, lse


def naive_attention_forward(q, k, v, scale: float | None = None, causal: bool = False, out=None,
                            lse=None, workspace=None, stream=None):
    """The step-by-step baseline for contiguous CUDA tensors [B, H, N, d]:
    S and P are written to a workspace in HBM (allocated here unless given)."""
    import torch
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    nbytes = fa_naive_workspace_size(B, H, N)
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    st = fa_naive_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                      B, H, N, d, scale, int(causal), _dtype_code(q), workspace.data_ptr(),
                      workspace.numel() * workspace.element_size(), _stream_handle(stream))
    if st != FA_OK:
        raise FaError(st, "fa_naive_fwd")
    return out, lse
