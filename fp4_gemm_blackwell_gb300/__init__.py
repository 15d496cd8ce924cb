"""Python binding of libbsgemm (block-scaled MXFP8 / NVFP4 GEMM for GB300).

Argument marshalling only: every function calls the C entry point of the same name in
``libbsgemm.so`` (declared in include/bsgemm.h); all arithmetic runs in the library's CUDA
kernels.  Pointers may be given as ints or as torch tensors (their ``data_ptr()``);
streams as ints, ``torch.cuda.Stream`` objects or None (torch's current stream).
A missing library raises immediately: there is no fallback.
"""

import ctypes
import os

__all__ = [
    "BSG_MXFP8", "BSG_NVFP4", "BSG_OUT_F16", "BSG_OUT_BF16", "BSG_OUT_NVFP4", "BSG_F_BIAS", "BSG_F_SILU",
    "BSG_F_ALPHA_DEVICE", "BSG_F_C", "BSG_F_ALPHA_ROW", "BSG_F_ALPHA_COL", "BSG_F_GROUPED", "BsgError", "lib", "bsg_sf_bytes", "bsg_quantize", "bsg_quantize_bf16", "bsg_plan_create",
    "bsg_plan_run", "bsg_plan_run_operands", "bsg_plan_destroy", "bsg_plan_check_status", "bsg_plan_variant",
    "bsg_plan_debug_set", "mxfp8_gemm", "nvfp4_gemm", "bsg_cache_clear", "bsg_last_error",
    "bsg_version", "Plan", "bsg_gemm_noalloc", "bsg_noalloc_check_status",
    "bsg_quantize_nvfp4_scaled",
]

BSG_MXFP8, BSG_NVFP4 = 0, 1
BSG_OUT_F16, BSG_OUT_BF16, BSG_OUT_NVFP4 = 0, 1, 2
BSG_F_BIAS, BSG_F_SILU, BSG_F_ALPHA_DEVICE = 1, 2, 4
BSG_F_C, BSG_F_ALPHA_ROW, BSG_F_ALPHA_COL, BSG_F_GROUPED = 8, 16, 32, 64

STATUS_NAMES = {
    0: "BSG_OK", 1: "BSG_ERR_INVALID_ARG", 2: "BSG_ERR_SHAPE", 3: "BSG_ERR_ALIGNMENT",
    4: "BSG_ERR_SCALE_LAYOUT", 5: "BSG_ERR_DTYPE", 6: "BSG_ERR_ARCH", 7: "BSG_ERR_CUDA",
    8: "BSG_ERR_DEVICE_TIMEOUT", 9: "BSG_ERR_NOMEM",
}

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libbsgemm.so")


class BsgError(RuntimeError):
    def __init__(self, status, message):
        self.status = status
        self.name = STATUS_NAMES.get(status, str(status))
        super().__init__("%s: %s" % (self.name, message))


class BsgDesc(ctypes.Structure):
    _fields_ = [
        ("kind", ctypes.c_int), ("out", ctypes.c_int), ("flags", ctypes.c_uint),
        ("M", ctypes.c_int), ("N", ctypes.c_int), ("K", ctypes.c_int),
        ("A", ctypes.c_void_p), ("B", ctypes.c_void_p), ("SFA", ctypes.c_void_p),
        ("SFB", ctypes.c_void_p), ("bias", ctypes.c_void_p), ("D", ctypes.c_void_p),
        ("alpha", ctypes.c_float), ("alpha_dev", ctypes.c_void_p),
        ("C", ctypes.c_void_p), ("beta", ctypes.c_float), ("alpha_row", ctypes.c_void_p),
        ("alpha_col", ctypes.c_void_p), ("L", ctypes.c_int),
        ("stride_A", ctypes.c_longlong), ("stride_B", ctypes.c_longlong), ("stride_SFA", ctypes.c_longlong),
        ("stride_SFB", ctypes.c_longlong), ("stride_D", ctypes.c_longlong), ("stride_C", ctypes.c_longlong),
        ("group_index", ctypes.c_void_p), ("SFD", ctypes.c_void_p), ("d_scale", ctypes.c_void_p),
    ]


class BsgOperands(ctypes.Structure):
    _fields_ = [(name, ctypes.c_void_p) for name in
                ("A", "B", "SFA", "SFB", "D", "bias", "alpha_dev", "C", "alpha_row", "alpha_col", "group_index",
                 "SFD", "d_scale")]


_lib = None


def lib():
    """The loaded ``libbsgemm.so`` (ctypes.CDLL); raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("libbsgemm.so is not built (%s); run __graft_entry__.build() or "
                           "python fp4_gemm_blackwell_gb300/build.py" % LIB_PATH)
    L = ctypes.CDLL(LIB_PATH)
    vp, i, u, f, st = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint, ctypes.c_float, ctypes.c_int
    sig = {
        "bsg_plan_create": (st, [ctypes.POINTER(vp), ctypes.POINTER(BsgDesc)]),
        "bsg_plan_run": (st, [vp, vp]),
        "bsg_plan_run_operands": (st, [vp, ctypes.POINTER(BsgOperands), vp]),
        "bsg_plan_destroy": (st, [vp]),
        "bsg_plan_check_status": (st, [vp]),
        "bsg_plan_variant": (ctypes.c_char_p, [vp]),
        "bsg_plan_debug_set": (st, [vp, i, ctypes.c_ulonglong]),
        "mxfp8_gemm": (st, [vp, vp, vp, vp, vp, f, i, i, i, i, vp]),
        "nvfp4_gemm": (st, [vp, vp, vp, vp, vp, vp, f, u, i, i, i, i, vp]),
        "bsg_cache_clear": (st, []),
        "bsg_gemm_noalloc": (st, [ctypes.POINTER(BsgDesc), vp]),
        "bsg_noalloc_check_status": (st, [vp]),
        "bsg_sf_bytes": (ctypes.c_size_t, [i, i, i]),
        "bsg_quantize": (st, [i, vp, i, i, vp, vp, vp, vp]),
        "bsg_quantize_bf16": (st, [i, vp, i, i, vp, vp, vp, vp]),
        "bsg_quantize_nvfp4_scaled": (st, [vp, i, i, i, vp, vp, vp, vp]),
        "bsg_last_error": (ctypes.c_char_p, []),
        "bsg_version": (ctypes.c_char_p, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(status):
    if status != 0:
        raise BsgError(status, lib().bsg_last_error().decode(errors="replace"))


def bsg_last_error():
    return lib().bsg_last_error().decode(errors="replace")


def bsg_version():
    return lib().bsg_version().decode()


def bsg_sf_bytes(kind, rows, K):
    return int(lib().bsg_sf_bytes(kind, rows, K))


def bsg_quantize(kind, x, rows, K, codes, sf, global_scale=None, stream=None):
    _check(lib().bsg_quantize(kind, _ptr(x), rows, K, _ptr(codes), _ptr(sf), _ptr(global_scale),
                              _stream(stream)))


def bsg_quantize_bf16(kind, x, rows, K, codes, sf, global_scale=None, stream=None):
    """x: rows x K BF16 values (a torch.bfloat16 tensor or 16-bit integer bit patterns)."""
    _check(lib().bsg_quantize_bf16(kind, _ptr(x), rows, K, _ptr(codes), _ptr(sf), _ptr(global_scale),
                                   _stream(stream)))


def bsg_quantize_nvfp4_scaled(x, rows, K, codes, sf, global_scale, bf16_input=False, stream=None):
    """NVFP4 quantisation with the global scale given (device float), one pass; x float32 or BF16."""
    _check(lib().bsg_quantize_nvfp4_scaled(_ptr(x), 1 if bf16_input else 0, rows, K, _ptr(codes), _ptr(sf),
                                           _ptr(global_scale), _stream(stream)))


def bsg_plan_create(kind, out, M, N, K, A, B, SFA, SFB, D, alpha=1.0, flags=0, bias=None, alpha_dev=None,
                    C=None, beta=0.0, alpha_row=None, alpha_col=None, L=0, strides=None, group_index=None,
                    SFD=None, d_scale=None):
    """strides (batched, L >= 2; grouped, stride_B and stride_SFB): dict of byte strides
    stride_A, stride_B, stride_SFA, stride_SFB, stride_D and stride_C between consecutive
    entries.  group_index (grouped, with BSG_F_GROUPED and L groups): M int32 on the device.
    SFD, d_scale (out = BSG_OUT_NVFP4): the output scales and the device global scale."""
    st = strides or {}
    d = BsgDesc(kind, out, flags, M, N, K, _ptr(A), _ptr(B), _ptr(SFA), _ptr(SFB), _ptr(bias), _ptr(D),
                alpha, _ptr(alpha_dev), _ptr(C), beta, _ptr(alpha_row), _ptr(alpha_col), L,
                *(st.get(k, 0) for k in ("stride_A", "stride_B", "stride_SFA", "stride_SFB", "stride_D", "stride_C")),
                _ptr(group_index), _ptr(SFD), _ptr(d_scale))
    h = ctypes.c_void_p()
    _check(lib().bsg_plan_create(ctypes.byref(h), ctypes.byref(d)))
    return h.value


def bsg_plan_run(plan, stream=None):
    _check(lib().bsg_plan_run(plan, _stream(stream)))


def bsg_plan_run_operands(plan, A, B, SFA, SFB, D, bias=None, alpha_dev=None, C=None, alpha_row=None,
                          alpha_col=None, group_index=None, SFD=None, d_scale=None, stream=None):
    ops = BsgOperands(*(_ptr(x) for x in (A, B, SFA, SFB, D, bias, alpha_dev, C, alpha_row, alpha_col,
                                          group_index, SFD, d_scale)))
    _check(lib().bsg_plan_run_operands(plan, ctypes.byref(ops), _stream(stream)))


def bsg_plan_destroy(plan):
    _check(lib().bsg_plan_destroy(plan))


def bsg_plan_check_status(plan):
    _check(lib().bsg_plan_check_status(plan))


def bsg_plan_variant(plan):
    return lib().bsg_plan_variant(plan).decode()


def bsg_plan_debug_set(plan, skip_first_load, wait_limit_ns=0):
    _check(lib().bsg_plan_debug_set(plan, int(skip_first_load), int(wait_limit_ns)))


def mxfp8_gemm(D, A, B, SFA, SFB, alpha, M, N, K, out, stream=None):
    _check(lib().mxfp8_gemm(_ptr(D), _ptr(A), _ptr(B), _ptr(SFA), _ptr(SFB), alpha, M, N, K, out,
                            _stream(stream)))


def nvfp4_gemm(D, A, B, SFA, SFB, bias, alpha, flags, M, N, K, out, stream=None):
    _check(lib().nvfp4_gemm(_ptr(D), _ptr(A), _ptr(B), _ptr(SFA), _ptr(SFB), _ptr(bias), alpha, flags,
                            M, N, K, out, _stream(stream)))


def bsg_gemm_noalloc(kind, out, M, N, K, A, B, SFA, SFB, D, alpha=1.0, flags=0, bias=None, alpha_dev=None,
                     stream=None, C=None, beta=0.0, alpha_row=None, alpha_col=None, L=0, strides=None,
                     group_index=None, SFD=None, d_scale=None):
    """Allocation-free GEMM (no device allocation; shares one static scratch array per GPU).
    The descriptor fields are those of bsg_plan_create."""
    st = strides or {}
    d = BsgDesc(kind, out, flags, M, N, K, _ptr(A), _ptr(B), _ptr(SFA), _ptr(SFB), _ptr(bias), _ptr(D),
                alpha, _ptr(alpha_dev), _ptr(C), beta, _ptr(alpha_row), _ptr(alpha_col), L,
                *(st.get(k, 0) for k in ("stride_A", "stride_B", "stride_SFA", "stride_SFB", "stride_D", "stride_C")),
                _ptr(group_index), _ptr(SFD), _ptr(d_scale))
    _check(lib().bsg_gemm_noalloc(ctypes.byref(d), _stream(stream)))


def bsg_noalloc_check_status(stream=None):
    """Raises BsgError (BSG_ERR_DEVICE_TIMEOUT) if an allocation-free launch on the current
    device gave up a wait since the last check; synchronises `stream` first."""
    _check(lib().bsg_noalloc_check_status(_stream(stream)))


def bsg_cache_clear():
    _check(lib().bsg_cache_clear())


class Plan:
    """Owning wrapper of a bsg_plan_t (destroyed on close / context exit)."""

    def __init__(self, *args, **kwargs):
        self.handle = bsg_plan_create(*args, **kwargs)

    def run(self, stream=None):
        bsg_plan_run(self.handle, stream)

    def run_operands(self, *args, **kwargs):
        bsg_plan_run_operands(self.handle, *args, **kwargs)

    def check_status(self):
        bsg_plan_check_status(self.handle)

    @property
    def variant(self):
        return bsg_plan_variant(self.handle)

    def close(self):
        if self.handle:
            bsg_plan_destroy(self.handle)
            self.handle = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
