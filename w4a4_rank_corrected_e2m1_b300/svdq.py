"""Python binding of libsvdq.so (ctypes): argument marshalling only.

Every step of the layer runs in the library (host pack in C++, kernels in CUDA
for sm_103a).  torch is used only for device memory and streams.  Importing
this module loads the shared library; if it is missing the import fails with
an error that says how to build it -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libsvdq.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "svdq.h")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED_SHAPE, ERR_ARCH, ERR_OOM, ERR_CUDA, ERR_TIMEOUT, ERR_WORKSPACE = range(8)
NO_SMOOTH = 1

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_i32 = ctypes.c_int32


class PackParams(ctypes.Structure):
    _fields_ = [
        ("N", _i64), ("K", _i64), ("rank", _i64),
        ("W_bf16", _vp), ("bias_bf16", _vp), ("Xcal_bf16", _vp), ("Mcal", _i64),
        ("lam", _vp), ("s_gX", ctypes.c_float), ("L1_bf16", _vp), ("L2_bf16", _vp),
        ("flags", ctypes.c_uint32), ("svd_power_iters", _i32), ("svd_oversample", _i32),
        ("svd_seed", ctypes.c_uint64), ("M_max", _i64), ("device", _i32), ("stream", _vp),
    ]


class PackedHost(ctypes.Structure):
    _fields_ = [
        ("lam", _vp), ("inv_lambda", _vp), ("L1_bf16", _vp), ("L2_bf16", _vp),
        ("R_codes", _vp), ("R_scales", _vp), ("bias_bf16", _vp),
        ("s_gW", ctypes.c_float), ("s_gX", ctypes.c_float), ("alpha", ctypes.c_float),
    ]


class Info(ctypes.Structure):
    _fields_ = [
        ("N", _i64), ("K", _i64), ("rank", _i64), ("lora_rank", _i64), ("r_pad", _i64), ("M_max", _i64),
        ("s_gW", ctypes.c_float), ("s_gX", ctypes.c_float), ("alpha", ctypes.c_float),
        ("device", _i32), ("sm_count", _i32),
    ]


class AwqParams(ctypes.Structure):
    _fields_ = [
        ("N", _i64), ("K", _i64), ("W_bf16", _vp), ("bias_bf16", _vp), ("Xcal_bf16", _vp), ("Mcal", _i64),
        ("s", _vp), ("device", _i32), ("stream", _vp),
    ]


class AwqHost(ctypes.Structure):
    _fields_ = [
        ("s", _vp), ("inv_s", _vp), ("codes", _vp), ("scales", _vp), ("zeros", _vp), ("bias_bf16", _vp),
        ("alpha", ctypes.c_float),
    ]


class Int4Host(ctypes.Structure):
    _fields_ = [
        ("lam", _vp), ("inv_lambda", _vp), ("L1_bf16", _vp), ("L2_bf16", _vp), ("R_codes", _vp),
        ("R_scales", _vp), ("bias_bf16", _vp),
    ]


_SIGS = {
    "svdq_pack_host": (_i32, [ctypes.POINTER(PackParams), ctypes.POINTER(PackedHost)]),
    "svdq_pack_weights": (_i32, [ctypes.POINTER(PackParams), ctypes.POINTER(_vp)]),
    "svdq_destroy": (_i32, [_vp]),
    "svdq_get_info": (_i32, [_vp, ctypes.POINTER(Info)]),
    "svdq_export": (_i32, [_vp, ctypes.POINTER(PackedHost)]),
    "svdq_scales_bytes": (_i64, [_i64, _i64]),
    "svdq_workspace_size": (_i32, [_vp, _i64, _i32, ctypes.POINTER(ctypes.c_size_t)]),
    "svdq_reserve": (_i32, [_vp, _i64, _i32]),
    "svdq_set_workspace": (_i32, [_vp, _vp, ctypes.c_size_t, _i64, _i32]),
    "svdq_quantize_act": (_i32, [_vp, _vp, _i64, _vp, _vp, _vp, _vp]),
    "svdq_gemm_quantized": (_i32, [_vp, _vp, _vp, _vp, _vp, _i64, _vp]),
    "svdq_linear_forward": (_i32, [_vp, _vp, _vp, _i64, _vp]),
    "svdq_linear_forward_host": (_i32, [_vp, _vp, _vp, _i64, _vp]),
    "svdq_linear_forward_host_batch": (_i32, [_vp, ctypes.POINTER(_vp), ctypes.POINTER(_vp), _i32, _i64, _vp]),
    "svdq_linear_forward_noalloc": (_i32, [_vp, _vp, _vp, _i64, _vp]),
    "svdq_check_error": (_i32, [_vp]),
    "svdq_set_wait_limit": (_i32, [_vp, ctypes.c_uint64, _i32]),
    "svdq_attach_lora": (_i32, [_vp, _vp, _vp, _i64, ctypes.c_float, _vp]),
    "svdq_awq_pack_host": (_i32, [ctypes.POINTER(AwqParams), ctypes.POINTER(AwqHost)]),
    "svdq_awq_pack": (_i32, [ctypes.POINTER(AwqParams), ctypes.POINTER(_vp)]),
    "svdq_awq_destroy": (_i32, [_vp]),
    "svdq_awq_export": (_i32, [_vp, ctypes.POINTER(AwqHost)]),
    "svdq_awq_forward": (_i32, [_vp, _vp, _vp, _i64, _vp]),
    "svdq_awq_check_error": (_i32, [_vp]),
    "svdq_int4_scale_ld": (_i64, [_i64]),
    "svdq_int4_pack_host": (_i32, [ctypes.POINTER(PackParams), ctypes.POINTER(Int4Host)]),
    "svdq_int4_pack": (_i32, [ctypes.POINTER(PackParams), ctypes.POINTER(_vp)]),
    "svdq_int4_export": (_i32, [_vp, ctypes.POINTER(Int4Host)]),
    "svdq_int4_reserve": (_i32, [_vp, _i64]),
    "svdq_int4_quantize_act": (_i32, [_vp, _vp, _i64, _vp, _vp, _vp, _vp]),
    "svdq_int4_forward": (_i32, [_vp, _vp, _vp, _i64, _vp]),
    "svdq_int4_check_error": (_i32, [_vp]),
    "svdq_int4_destroy": (_i32, [_vp]),
    "svdq_mlp_create": (_i32, [_vp, _vp, _i64, ctypes.POINTER(_vp)]),
    "svdq_mlp_destroy": (_i32, [_vp]),
    "svdq_mlp_up_quantize": (_i32, [_vp, _vp, _i64, _vp, _vp, _vp, _vp]),
    "svdq_mlp_forward": (_i32, [_vp, _vp, _vp, _i64, _vp]),
    "svdq_mlp_check_error": (_i32, [_vp]),
    "svdq_gelu_bf16": (_i32, [_vp, _vp, _i64, _vp]),
    "svdq_status_string": (ctypes.c_char_p, [_i32]),
    "svdq_last_error": (ctypes.c_char_p, []),
}


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with `python -m w4a4_rank_corrected_e2m1_b300.build` "
            "(there is no CPU fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


LIB = _load()


def header_functions(path: str = HEADER):
    """Names of the functions include/svdq.h declares."""
    txt = open(path).read()
    return sorted(set(re.findall(r"^\s*(?:svdq_status_t|int64_t|const char\*)\s+(svdq_\w+)\s*\(", txt, re.M)))


class SvdqError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = LIB.svdq_last_error().decode()
        super().__init__(f"{where}: {LIB.svdq_status_string(status).decode()} ({msg})")


def check(status: int, where: str = "svdq"):
    if status != OK:
        raise SvdqError(status, where)


def _ptr(a) -> Optional[int]:
    """Address of a numpy array (host) or torch tensor (host or device); None stays NULL."""
    if a is None:
        return None
    if isinstance(a, np.ndarray):
        if not a.flags["C_CONTIGUOUS"]:
            raise ValueError("arrays must be C-contiguous")
        return a.ctypes.data
    if hasattr(a, "data_ptr"):
        if not a.is_contiguous():
            raise ValueError("tensors must be contiguous")
        return a.data_ptr()
    if isinstance(a, int):
        return a
    raise TypeError(type(a))


def _stream(stream) -> Optional[int]:
    if stream is None:
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _u16(a):
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("bfloat16 inputs are passed as uint16 bit patterns")
    return a


def make_params(W, rank, bias=None, Xcal=None, lam=None, s_gX=0.0, L1=None, L2=None, smooth=True,
                svd_power_iters=0, svd_oversample=0, svd_seed=0, M_max=0, device=0, stream=None):
    W, bias, Xcal, L1, L2 = _u16(W), _u16(bias), _u16(Xcal), _u16(L1), _u16(L2)
    lam = None if lam is None else np.ascontiguousarray(lam, dtype=np.float32)
    N, K = W.shape
    p = PackParams(N=N, K=K, rank=rank, W_bf16=_ptr(W), bias_bf16=_ptr(bias), Xcal_bf16=_ptr(Xcal),
                   Mcal=0 if Xcal is None else Xcal.shape[0], lam=_ptr(lam), s_gX=s_gX,
                   L1_bf16=_ptr(L1), L2_bf16=_ptr(L2), flags=0 if smooth else NO_SMOOTH,
                   svd_power_iters=svd_power_iters, svd_oversample=svd_oversample, svd_seed=svd_seed,
                   M_max=M_max, device=device, stream=_stream(stream))
    keep = (W, bias, Xcal, lam, L1, L2)
    return p, keep


def _host_out(N, K, rank):
    o = dict(lam=np.zeros(K, np.float32), inv_lambda=np.zeros(K, np.float32),
             L1=np.zeros((K, rank), np.uint16), L2=np.zeros((rank, N), np.uint16),
             R_codes=np.zeros((N, K // 2), np.uint8), R_scales=np.zeros((N, K // 16), np.uint8),
             bias=np.zeros(N, np.uint16))
    s = PackedHost(lam=_ptr(o["lam"]), inv_lambda=_ptr(o["inv_lambda"]), L1_bf16=_ptr(o["L1"]),
                   L2_bf16=_ptr(o["L2"]), R_codes=_ptr(o["R_codes"]), R_scales=_ptr(o["R_scales"]),
                   bias_bf16=_ptr(o["bias"]))
    return o, s


def _finish(o, s, rank):
    o["s_gW"] = np.float32(s.s_gW)
    o["s_gX"] = np.float32(s.s_gX)
    o["alpha"] = np.float32(s.alpha)
    o["rank"] = rank
    return o


def pack_host(W, rank, **kw):
    """svdq_pack_host: the offline step on the CPU; returns the canonical packed layer."""
    p, keep = make_params(W, rank, **kw)
    o, s = _host_out(p.N, p.K, rank)
    check(LIB.svdq_pack_host(ctypes.byref(p), ctypes.byref(s)), "svdq_pack_host")
    return _finish(o, s, rank)


def scales_bytes(M: int, K: int) -> int:
    return int(LIB.svdq_scales_bytes(M, K))


class Layer:
    """A packed SVDQuant layer on one CUDA device (wraps an svdq_handle_t)."""

    def __init__(self, W, rank, **kw):
        p, keep = make_params(W, rank, **kw)
        h = _vp()
        check(LIB.svdq_pack_weights(ctypes.byref(p), ctypes.byref(h)), "svdq_pack_weights")
        self.h = h
        self.N, self.K, self.rank = int(p.N), int(p.K), int(rank)

    def close(self):
        if getattr(self, "h", None):
            LIB.svdq_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def info(self) -> Info:
        i = Info()
        check(LIB.svdq_get_info(self.h, ctypes.byref(i)), "svdq_get_info")
        return i

    def export(self):
        o, s = _host_out(self.N, self.K, self.rank)
        check(LIB.svdq_export(self.h, ctypes.byref(s)), "svdq_export")
        return _finish(o, s, self.rank)

    # host_staging: device staging slots for host X / Y (0, 1, or 2 for forward_host_batch);
    # True / False mean 1 / 0
    def workspace_size(self, M: int, host_staging: int = 0) -> int:
        n = ctypes.c_size_t()
        check(LIB.svdq_workspace_size(self.h, M, int(host_staging), ctypes.byref(n)), "svdq_workspace_size")
        return n.value

    def reserve(self, M_max: int, host_staging: int = 0):
        check(LIB.svdq_reserve(self.h, M_max, int(host_staging)), "svdq_reserve")

    def set_workspace(self, buf, M_max: int, host_staging: int = 0):
        nbytes = 0 if buf is None else buf.numel() * buf.element_size()
        check(LIB.svdq_set_workspace(self.h, _ptr(buf), nbytes, M_max, int(host_staging)), "svdq_set_workspace")

    def quantize_act(self, X, M, x_codes, x_scales, T, stream=None):
        check(LIB.svdq_quantize_act(self.h, _ptr(X), M, _ptr(x_codes), _ptr(x_scales), _ptr(T), _stream(stream)),
              "svdq_quantize_act")

    def gemm_quantized(self, x_codes, x_scales, T, Y, M, stream=None):
        check(LIB.svdq_gemm_quantized(self.h, _ptr(x_codes), _ptr(x_scales), _ptr(T), _ptr(Y), M, _stream(stream)),
              "svdq_gemm_quantized")

    def forward(self, X, Y, M, stream=None):
        check(LIB.svdq_linear_forward(self.h, _ptr(X), _ptr(Y), M, _stream(stream)), "svdq_linear_forward")

    def forward_noalloc(self, X, Y, M, stream=None):
        """The forward on the library's static scratch (no workspace, no allocation)."""
        check(LIB.svdq_linear_forward_noalloc(self.h, _ptr(X), _ptr(Y), M, _stream(stream)),
              "svdq_linear_forward_noalloc")

    def forward_host(self, X_host, Y_host, M, stream=None):
        check(LIB.svdq_linear_forward_host(self.h, _ptr(X_host), _ptr(Y_host), M, _stream(stream)),
              "svdq_linear_forward_host")

    def forward_host_batch(self, X_hosts, Y_hosts, M, stream=None):
        """len(X_hosts) pipelined layer calls on host buffers (workspace with host_staging=2)."""
        if len(X_hosts) != len(Y_hosts):
            raise ValueError("X_hosts and Y_hosts differ in length")
        B = len(X_hosts)
        xs = (_vp * max(B, 1))(*[_ptr(x) for x in X_hosts])
        ys = (_vp * max(B, 1))(*[_ptr(y) for y in Y_hosts])
        check(LIB.svdq_linear_forward_host_batch(self.h, xs, ys, B, M, _stream(stream)),
              "svdq_linear_forward_host_batch")

    def check_error(self):
        check(LIB.svdq_check_error(self.h), "svdq_check_error")

    def set_wait_limit(self, wait_ns: int = 0, stall_kernel: int = 0):
        """Limit of the kernels' bounded waits (0 = default) and the failure-detection stall
        (0 none, 1 kernel 1, 2 kernel 2)."""
        check(LIB.svdq_set_wait_limit(self.h, wait_ns, stall_kernel), "svdq_set_wait_limit")

    def attach_lora(self, A, B, scale: float = 1.0, stream=None):
        """Append a LoRA adapter (A: K x r_lora, B: r_lora x N, bf16 bit patterns on the host)
        to the low-rank branch; A = B = None removes it."""
        if A is None:
            check(LIB.svdq_attach_lora(self.h, None, None, 0, 1.0, _stream(stream)), "svdq_attach_lora")
            return
        A, B = _u16(A), _u16(B)
        r_lora = int(A.shape[1])
        if A.shape != (self.K, r_lora) or B.shape != (r_lora, self.N):
            raise ValueError(f"LoRA factors must be {self.K} x r and r x {self.N}")
        check(LIB.svdq_attach_lora(self.h, A.ctypes.data, B.ctypes.data, r_lora, float(scale), _stream(stream)),
              "svdq_attach_lora")


# ------------------------------------------------------------------ INT4 variant
def _int4_out(N, K, rank):
    o = dict(lam=np.zeros(K, np.float32), inv_lambda=np.zeros(K, np.float32),
             L1=np.zeros((K, rank), np.uint16), L2=np.zeros((rank, N), np.uint16),
             R_codes=np.zeros((N, K // 2), np.uint8), R_scales=np.zeros((N, K // 64), np.float32),
             bias=np.zeros(N, np.uint16), rank=rank, fmt="int4")
    st = Int4Host(lam=_ptr(o["lam"]), inv_lambda=_ptr(o["inv_lambda"]), L1_bf16=_ptr(o["L1"]),
                  L2_bf16=_ptr(o["L2"]), R_codes=_ptr(o["R_codes"]), R_scales=_ptr(o["R_scales"]),
                  bias_bf16=_ptr(o["bias"]))
    return o, st


def int4_pack_host(W, rank, **kw):
    """svdq_int4_pack_host: the INT4 variant's offline step on the CPU (codes two per byte)."""
    p, keep = make_params(W, rank, **kw)
    o, st = _int4_out(int(p.N), int(p.K), rank)
    check(LIB.svdq_int4_pack_host(ctypes.byref(p), ctypes.byref(st)), "svdq_int4_pack_host")
    return o


def int4_scale_ld(rows: int) -> int:
    return int(LIB.svdq_int4_scale_ld(rows))


class Int4Layer:
    """A packed INT4-variant SVDQuant layer on one CUDA device (wraps an svdq_int4_handle_t)."""

    def __init__(self, W, rank, **kw):
        p, keep = make_params(W, rank, **kw)
        h = _vp()
        check(LIB.svdq_int4_pack(ctypes.byref(p), ctypes.byref(h)), "svdq_int4_pack")
        self.h = h
        self.N, self.K, self.rank = int(p.N), int(p.K), int(rank)
        self.r_pad = 0 if rank == 0 else 64 * ((rank + 63) // 64)

    def close(self):
        if getattr(self, "h", None):
            LIB.svdq_int4_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def export(self):
        o, st = _int4_out(self.N, self.K, self.rank)
        check(LIB.svdq_int4_export(self.h, ctypes.byref(st)), "svdq_int4_export")
        return o

    def reserve(self, M_max: int):
        check(LIB.svdq_int4_reserve(self.h, M_max), "svdq_int4_reserve")

    def quantize_act(self, X, M, codes, scales, T=None, stream=None):
        check(LIB.svdq_int4_quantize_act(self.h, _ptr(X), M, _ptr(codes), _ptr(scales), _ptr(T), _stream(stream)),
              "svdq_int4_quantize_act")

    def forward(self, X, Y, M, stream=None):
        check(LIB.svdq_int4_forward(self.h, _ptr(X), _ptr(Y), M, _stream(stream)), "svdq_int4_forward")

    def check_error(self):
        check(LIB.svdq_int4_check_error(self.h), "svdq_int4_check_error")


# ------------------------------------------------------------------ MLP pair
class Mlp:
    """Two packed layers with GELU between them, run with the fused epilogue (wraps an
    svdq_mlp_t).  The layers must outlive the pair and have workspaces for the M they run."""

    def __init__(self, up: Layer, down: Layer, M_max: int):
        h = _vp()
        check(LIB.svdq_mlp_create(up.h, down.h, M_max, ctypes.byref(h)), "svdq_mlp_create")
        self.h = h
        self.up, self.down, self.M_max = up, down, M_max

    def close(self):
        if getattr(self, "h", None):
            LIB.svdq_mlp_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def up_quantize(self, X, M, x_codes, x_scales, T=None, stream=None):
        check(LIB.svdq_mlp_up_quantize(self.h, _ptr(X), M, _ptr(x_codes), _ptr(x_scales), _ptr(T), _stream(stream)),
              "svdq_mlp_up_quantize")

    def forward(self, X, Y, M, stream=None):
        check(LIB.svdq_mlp_forward(self.h, _ptr(X), _ptr(Y), M, _stream(stream)), "svdq_mlp_forward")

    def check_error(self):
        check(LIB.svdq_mlp_check_error(self.h), "svdq_mlp_check_error")


def gelu_bf16(Y, G, n, stream=None):
    """G = bf16(GELU(Y)) elementwise on n bf16 values (the fused epilogue's arithmetic)."""
    check(LIB.svdq_gelu_bf16(_ptr(Y), _ptr(G), n, _stream(stream)), "svdq_gelu_bf16")


# ------------------------------------------------------------------ AWQ-style W4A16 layer
def _awq_params(W, bias=None, Xcal=None, s=None, device=0, stream=None):
    W = _u16(W)
    N, K = W.shape
    bias = _u16(bias)
    Xcal = _u16(Xcal)
    s_arr = None if s is None else np.ascontiguousarray(s, dtype=np.float32)
    p = AwqParams(N=N, K=K, W_bf16=W.ctypes.data, bias_bf16=None if bias is None else bias.ctypes.data,
                  Xcal_bf16=None if Xcal is None else Xcal.ctypes.data, Mcal=0 if Xcal is None else Xcal.shape[0],
                  s=None if s_arr is None else s_arr.ctypes.data, device=device, stream=_stream(stream))
    return p, (W, bias, Xcal, s_arr)


def _awq_out(N, K):
    o = {"s": np.zeros(K, np.float32), "inv_s": np.zeros(K, np.float32), "codes": np.zeros((N, K // 2), np.uint8),
         "scales": np.zeros((N, K // 64), np.float32), "zeros": np.zeros((N, K // 64), np.uint8),
         "bias": np.zeros(N, np.uint16)}
    st = AwqHost(s=o["s"].ctypes.data, inv_s=o["inv_s"].ctypes.data, codes=o["codes"].ctypes.data,
                 scales=o["scales"].ctypes.data, zeros=o["zeros"].ctypes.data, bias_bf16=o["bias"].ctypes.data)
    return o, st


def awq_pack_host(W, bias=None, Xcal=None, s=None):
    """Host quantisation of the AWQ-style layer; codes packed two per byte (low nibble first)."""
    p, keep = _awq_params(W, bias, Xcal, s)
    o, st = _awq_out(int(p.N), int(p.K))
    check(LIB.svdq_awq_pack_host(ctypes.byref(p), ctypes.byref(st)), "svdq_awq_pack_host")
    o["alpha"] = float(st.alpha)
    return o


class AwqLayer:
    """A packed AWQ-style W4A16 layer on one CUDA device (wraps an svdq_awq_handle_t)."""

    def __init__(self, W, bias=None, Xcal=None, s=None, device=0, stream=None):
        p, keep = _awq_params(W, bias, Xcal, s, device, stream)
        h = _vp()
        check(LIB.svdq_awq_pack(ctypes.byref(p), ctypes.byref(h)), "svdq_awq_pack")
        self.h = h
        self.N, self.K = int(p.N), int(p.K)

    def close(self):
        if getattr(self, "h", None):
            LIB.svdq_awq_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def export(self):
        o, st = _awq_out(self.N, self.K)
        check(LIB.svdq_awq_export(self.h, ctypes.byref(st)), "svdq_awq_export")
        o["alpha"] = float(st.alpha)
        return o

    def forward(self, X, Y, M, stream=None):
        check(LIB.svdq_awq_forward(self.h, _ptr(X), _ptr(Y), M, _stream(stream)), "svdq_awq_forward")

    def check_error(self):
        check(LIB.svdq_awq_check_error(self.h), "svdq_awq_check_error")
