"""Python binding of libqmm (ctypes): argument marshalling only.

Every function here has the name of the C entry point it calls (include/qmm.h)
and hands device pointers, sizes and the current CUDA stream to it; all
arithmetic runs in the library's CUDA kernels.  torch is used for device
memory and streams only.  If libqmm.so has not been built the first call
raises -- there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np
import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libqmm.so")

QMM_OK, QMM_EINVAL, QMM_ESHAPE, QMM_EWORKSPACE, QMM_ECUDA, QMM_EALIGN, QMM_ENODEV = \
    0, -1, -2, -3, -4, -5, -6

QMM_PARTIAL_BF16, QMM_PARTIAL_F32 = 0, 1
QMM_PRESET_PAGES, QMM_PRESET_GB300 = 0, 1
QMM_KERNELS_DEFAULT, QMM_KERNELS_MMA_SYNC, QMM_KERNELS_TCGEN05, QMM_KERNELS_LEAN = 0, 1, 2, 3


class qmm_policy(ctypes.Structure):
    _fields_ = [("bm", ctypes.c_int), ("bn", ctypes.c_int), ("target_blocks", ctypes.c_int),
                ("cap", ctypes.c_int), ("min_k_per_split", ctypes.c_int)]

    def as_tuple(self):
        return (self.bm, self.bn, self.target_blocks, self.cap, self.min_k_per_split)

    def __repr__(self):
        return "qmm_policy(bm=%d, bn=%d, target_blocks=%d, cap=%d, min_k_per_split=%d)" % \
            self.as_tuple()


QMM_OPT_DEFAULT = -1
_OPTION_FIELDS = ("kernels", "partitions", "reduce", "weights_static", "pdl",
                  "grouped_schedule", "group_plan")


class qmm_options(ctypes.Structure):
    """Per-call options (see qmm.h); every field defaults to QMM_OPT_DEFAULT."""
    _fields_ = [(f, ctypes.c_int) for f in _OPTION_FIELDS]

    def __init__(self, **kw):
        super().__init__(*([QMM_OPT_DEFAULT] * len(_OPTION_FIELDS)))
        for k, v in kw.items():
            if k not in _OPTION_FIELDS:
                raise TypeError("unknown option %r" % k)
            setattr(self, k, int(v))


def _opt(options):
    return ctypes.byref(options) if options is not None else None


class QmmError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        detail = " [%s]" % qmm_last_cuda_error() if code == QMM_ECUDA else ""
        super().__init__("%s: %s (%d)%s" % (what, qmm_strerror(code), code, detail))


class qmm_stream_call(ctypes.Structure):
    """One chunk of qmm_w4a16_g128_stream (see qmm.h)."""
    _fields_ = [("A_host", ctypes.c_void_p), ("C_host", ctypes.c_void_p),
                ("Wq", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("biases", ctypes.c_void_p), ("M", ctypes.c_int), ("Kred", ctypes.c_int),
                ("Nout", ctypes.c_int)]


class qmm_group_call(ctypes.Structure):
    """One call of qmm_w4a16_g128_grouped (see qmm.h)."""
    _fields_ = [("A", ctypes.c_void_p), ("Wq", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("biases", ctypes.c_void_p), ("C", ctypes.c_void_p), ("M", ctypes.c_int),
                ("Kred", ctypes.c_int), ("Nout", ctypes.c_int)]


_lock = threading.Lock()
_lib = None

_P, _I, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
_SIGS = {
    "qmm_policy_preset": (_I, [_I, _I, _I, ctypes.POINTER(qmm_policy)]),
    "qmm_kernel_tile": (_I, [_I, ctypes.POINTER(_I), ctypes.POINTER(_I)]),
    "qmm_kernel_grouped": (_I, [_I]),
    "qmm_splitk_plan": (_I, [_I, _I, _I, ctypes.POINTER(qmm_policy), ctypes.POINTER(_I)]),
    "qmm_splitk_plan_near_equal": (_I, [_I, _I, _I, ctypes.POINTER(qmm_policy),
                                        ctypes.POINTER(_I)]),
    "qmm_splitk_workspace_bytes": (_SZ, [_I, _I, _I, _I]),
    "qmm_w4a16_g128": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, ctypes.POINTER(qmm_policy),
                            _P, _SZ, _I, _P, ctypes.POINTER(_I)]),
    "qmm_splitk_reduce": (_I, [_P, _I, _I, _I, _I, _P, _P]),
    "qmm_w4a16_g128_partition": (_I, [_P, _P, _P, _P, _P, _SZ, _I, _I, _I, _I, _I, _P]),
    "qmm_gemm_bf16_splitk": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _SZ, _P]),
    "qmm_gemm_workspace_bytes": (_SZ, [_I, _I, _I]),
    "qmm_unpack_probe": (_I, [_P, _I, _I, _P, _P]),
    "qmm_dequant_probe": (_I, [_P, _P, _P, _I, _I, _P, _P]),
    "qmm_strerror": (ctypes.c_char_p, [_I]),
    "qmm_last_cuda_error": (ctypes.c_char_p, []),
    "qmm_options_init": (None, [_P]),
    "qmm_w4a16_g128_ex": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, ctypes.POINTER(qmm_policy),
                               _P, _SZ, _I, _P, ctypes.POINTER(_I), _P]),
    "qmm_splitk_workspace_bytes_ex": (_SZ, [_I, _I, _I, _I, _P]),
    "qmm_call_plan": (_I, [_I, _I, _I, _I, ctypes.POINTER(qmm_policy), _I, _I, _P,
                           ctypes.POINTER(_I), ctypes.POINTER(_I), ctypes.POINTER(_I),
                           ctypes.POINTER(_I)]),
    "qmm_call_workspace_bytes": (_SZ, [_I, _I, _I, _I, ctypes.POINTER(qmm_policy), _I, _I, _P]),
    "qmm_set_kernels": (_I, [_I]),
    "qmm_set_pdl": (_I, [_I]),
    "qmm_set_weights_static": (_I, [_I]),
    "qmm_set_reduce": (_I, [_I]),
    "qmm_set_partitions": (_I, [_I]),
    "qmm_set_grouped_schedule": (_I, [_I]),
    "qmm_set_group_plan": (_I, [_I]),
    "qmm_group_plan": (_I, [ctypes.POINTER(_I), _I, _I, _I, ctypes.POINTER(_I)]),
    "qmm_kernel_status": (_I, [ctypes.POINTER(_I), _I]),
    "qmm_wait_timeout_probe": (_I, [ctypes.c_void_p]),
    "qmm_w4a16_g128_noalloc": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I,
                                    ctypes.POINTER(qmm_policy), _I, _P, ctypes.POINTER(_I)]),
    "qmm_static_scratch_bytes": (_SZ, []),
    "qmm_tc_pipeline_config": (_I, [_I, _I, _I, ctypes.POINTER(_I)]),
    "qmm_tc_persistent_pipeline_config": (_I, [_I, _I, _I, ctypes.POINTER(_I)]),
    "qmm_decode_attention_splits": (_I, [_I, _I, _I, _I, _I, ctypes.POINTER(_I)]),
    "qmm_decode_attention_workspace_bytes": (_SZ, [_I, _I, _I, _I]),
    "qmm_decode_attention": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, ctypes.c_float, _I,
                                  _P, _SZ, _P, ctypes.POINTER(_I)]),
    "qmm_group_workspace_bytes": (_SZ, [ctypes.POINTER(qmm_group_call), _I, _I]),
    "qmm_w4a16_g128_grouped": (_I, [ctypes.POINTER(qmm_group_call), _I, _P, _SZ, _I, _P,
                                    ctypes.POINTER(_I)]),
    "qmm_group_workspace_bytes_ex": (_SZ, [ctypes.POINTER(qmm_group_call), _I, _I, _P]),
    "qmm_w4a16_g128_grouped_ex": (_I, [ctypes.POINTER(qmm_group_call), _I, _P, _SZ, _I, _P,
                                       ctypes.POINTER(_I), _P]),
    "qmm_stream_arena_bytes": (_SZ, [ctypes.POINTER(qmm_stream_call), _I, _I]),
    "qmm_w4a16_g128_stream": (_I, [ctypes.POINTER(qmm_stream_call), _I, _I, _P, _SZ, _P, _P, _P,
                                   ctypes.POINTER(_I)]),
    "qmm_overlap_schedule": (_I, [_I, _I, ctypes.POINTER(ctypes.c_double),
                                  ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double),
                                  _I, ctypes.POINTER(ctypes.c_double),
                                  ctypes.POINTER(ctypes.c_double)]),
}


def lib() -> ctypes.CDLL:
    """The loaded libqmm.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError("libqmm.so is not built; run "
                                   "`python -m split_w4a16_quantized_gb300.build`")
            h = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in _SIGS.items():
                fn = getattr(h, name)
                fn.restype = res
                fn.argtypes = args
            _lib = h
        return _lib


def _check(rc: int, what: str):
    if rc != QMM_OK:
        raise QmmError(rc, what)


# torch's raw current-stream lookup: a plain integer, without building a
# torch.cuda.Stream object (about 3 µs of host time per call on an Arm host)
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)
_cur_device = getattr(torch._C, "_cuda_getDevice", None)


def _stream(stream):
    if stream is None:
        if _raw_stream is not None and _cur_device is not None and torch.cuda.is_initialized():
            return _raw_stream(_cur_device())
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        stream = stream.cuda_stream
    return int(stream)


def _dev(t: torch.Tensor, dtypes, name: str) -> ctypes.c_void_p:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("%s must be a CUDA tensor" % name)
    if t.dtype not in dtypes:
        raise TypeError("%s has dtype %s, expected one of %s" % (name, t.dtype, dtypes))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return ctypes.c_void_p(t.data_ptr())


def _ptr(t: torch.Tensor, dtypes, name: str) -> int:
    """_dev's checks in one expression for the per-call entry points; the
    pointer as a plain integer.  Any failed check is reported by _dev."""
    try:
        if t.is_cuda and t.dtype in dtypes and t.is_contiguous():
            return t.data_ptr()
    except AttributeError:
        pass
    _dev(t, dtypes, name)
    raise TypeError("%s is not a usable CUDA tensor" % name)


_BF16 = (torch.bfloat16,)
_WORDS = (torch.int32, torch.uint32) if hasattr(torch, "uint32") else (torch.int32,)


# ---- host-only entry points ---------------------------------------------

def qmm_strerror(code: int) -> str:
    return lib().qmm_strerror(code).decode()


def qmm_last_cuda_error() -> str:
    """Name of the CUDA error behind this thread's latest QMM_ECUDA."""
    return lib().qmm_last_cuda_error().decode()


def qmm_policy_preset(which: int, M: int = 1, num_sms: int = 0) -> qmm_policy:
    out = qmm_policy()
    _check(lib().qmm_policy_preset(which, M, num_sms, ctypes.byref(out)), "qmm_policy_preset")
    return out


def qmm_set_kernels(which: int) -> int:
    """Select the kernel table (QMM_KERNELS_*); returns the previous one."""
    prev = lib().qmm_set_kernels(which)
    if prev < 0:
        raise QmmError(prev, "qmm_set_kernels")
    return prev


def qmm_set_pdl(enable: bool) -> int:
    """Programmatic dependent launch on/off; returns the previous setting."""
    return lib().qmm_set_pdl(int(bool(enable)))


QMM_REDUCE_KERNEL, QMM_REDUCE_FUSED, QMM_REDUCE_CLUSTER = 0, 1, 2


def qmm_set_reduce(mode: int) -> int:
    """Separate reduce kernel (default), the fused last-CTA reduce or the
    cluster reduce (see qmm.h)."""
    prev = lib().qmm_set_reduce(mode)
    if prev < 0:
        raise QmmError(prev, "qmm_set_reduce")
    return prev


QMM_PARTITIONS_EQUAL, QMM_PARTITIONS_NEAR_EQUAL = 0, 1


def qmm_set_partitions(mode: int) -> int:
    """Equal partitions (default) or near-equal ones for any split (see qmm.h)."""
    prev = lib().qmm_set_partitions(mode)
    if prev < 0:
        raise QmmError(prev, "qmm_set_partitions")
    return prev


QMM_GROUPED_TILES, QMM_GROUPED_PERSISTENT = 0, 1


def qmm_set_grouped_schedule(mode: int) -> int:
    """Schedule of the grouped call's tcgen05 launches (QMM_GROUPED_*, the
    persistent one by default); returns the previous one."""
    prev = lib().qmm_set_grouped_schedule(mode)
    if prev < 0:
        raise QmmError(prev, "qmm_set_grouped_schedule")
    return prev


QMM_GROUP_PLAN_CALLS, QMM_GROUP_PLAN_GROUP = 0, 1
QMM_SPLIT_PLANNED = -1  # split_req of qmm_w4a16_g128: the group plan for the call alone
QMM_SPLIT_BALANCED = -2  # split_req: whole waves unsplit, the partial wave's rows split


def qmm_set_group_plan(mode: int) -> int:
    """Split plan of the grouped call (QMM_GROUP_PLAN_*); returns the previous one."""
    prev = lib().qmm_set_group_plan(mode)
    if prev < 0:
        raise QmmError(prev, "qmm_set_group_plan")
    return prev


def qmm_group_plan(shapes, num_sms: int = 0, partial_dtype: int = QMM_PARTIAL_BF16) -> list:
    """The group plan's splits for shapes [(M, Kred, Nout), ...] (host only)."""
    n = len(shapes)
    flat = (_I * (3 * n))(*[int(v) for shp in shapes for v in shp])
    out = (_I * n)()
    _check(lib().qmm_group_plan(flat, n, num_sms, partial_dtype, out), "qmm_group_plan")
    return list(out)


def qmm_set_weights_static(enable: bool) -> int:
    """Promise that no earlier kernel on the stream writes the weights (see qmm.h)."""
    return int(lib().qmm_set_weights_static(1 if enable else 0))


def qmm_kernel_status(clear: bool = True) -> int:
    """0, or 1 if a bounded wait inside a tcgen05 kernel ran out (synchronizes)."""
    st = _I(0)
    _check(lib().qmm_kernel_status(ctypes.byref(st), int(clear)), "qmm_kernel_status")
    return st.value


def qmm_wait_timeout_probe(stream=None) -> None:
    """Launch one CTA whose bounded wait runs out (test hook; see qmm.h)."""
    _check(lib().qmm_wait_timeout_probe(_stream(stream)), "qmm_wait_timeout_probe")


def qmm_kernel_tile(M: int):
    bm, bn = _I(0), _I(0)
    _check(lib().qmm_kernel_tile(M, ctypes.byref(bm), ctypes.byref(bn)), "qmm_kernel_tile")
    return bm.value, bn.value


def qmm_kernel_grouped(M: int) -> bool:
    """True if the grouped call runs calls with M rows in shared launches."""
    rc = lib().qmm_kernel_grouped(M)
    if rc < 0:
        _check(rc, "qmm_kernel_grouped")
    return rc == 1


def qmm_splitk_plan(M: int, Kred: int, Nout: int, pol: qmm_policy) -> int:
    s = _I(0)
    _check(lib().qmm_splitk_plan(M, Kred, Nout, ctypes.byref(pol), ctypes.byref(s)),
           "qmm_splitk_plan")
    return s.value


def qmm_splitk_plan_near_equal(M: int, Kred: int, Nout: int, pol: qmm_policy) -> int:
    s = _I(0)
    _check(lib().qmm_splitk_plan_near_equal(M, Kred, Nout, ctypes.byref(pol), ctypes.byref(s)),
           "qmm_splitk_plan_near_equal")
    return s.value


def qmm_splitk_workspace_bytes(M: int, Nout: int, split: int,
                               partial_dtype: int = QMM_PARTIAL_BF16, options=None) -> int:
    if options is not None:
        return int(lib().qmm_splitk_workspace_bytes_ex(M, Nout, split, partial_dtype,
                                                        _opt(options)))
    return int(lib().qmm_splitk_workspace_bytes(M, Nout, split, partial_dtype))


def qmm_call_plan(M: int, Kred: int, Nout: int, split_req: int = 0, pol=None,
                  partial_dtype: int = QMM_PARTIAL_BF16, num_sms: int = 0, options=None,
                  with_head: bool = False):
    """(split, bm, bn) that qmm_w4a16_g128_ex would dispatch (host only);
    with_head: (split, bm, bn, head_rows), head_rows > 0 when
    QMM_SPLIT_BALANCED cuts the call."""
    s, bm, bn, hd = _I(0), _I(0), _I(0), _I(0)
    _check(lib().qmm_call_plan(M, Kred, Nout, split_req,
                               ctypes.byref(pol) if pol is not None else None, partial_dtype,
                               num_sms, _opt(options), ctypes.byref(s), ctypes.byref(bm),
                               ctypes.byref(bn), ctypes.byref(hd)), "qmm_call_plan")
    return (s.value, bm.value, bn.value, hd.value) if with_head else (s.value, bm.value, bn.value)


def qmm_call_workspace_bytes(M: int, Kred: int, Nout: int, split_req: int = 0, pol=None,
                             partial_dtype: int = QMM_PARTIAL_BF16, num_sms: int = 0,
                             options=None) -> int:
    return int(lib().qmm_call_workspace_bytes(M, Kred, Nout, split_req,
                                              ctypes.byref(pol) if pol is not None else None,
                                              partial_dtype, num_sms, _opt(options)))


def qmm_gemm_workspace_bytes(M: int, N: int, split: int) -> int:
    return int(lib().qmm_gemm_workspace_bytes(M, N, split))


# ---- device entry points -------------------------------------------------

def qmm_w4a16_g128(A: torch.Tensor, Wq: torch.Tensor, scales: torch.Tensor,
                   biases: torch.Tensor, C: torch.Tensor, split_req: int = 0,
                   pol: qmm_policy | None = None, workspace: torch.Tensor | None = None,
                   partial_dtype: int = QMM_PARTIAL_BF16, stream=None, options=None) -> int:
    """C = A @ W^T (W in the W4A16-g128 format); returns the split dispatched.
    Shapes: A [M, Kred] bf16, Wq [Nout, Kred/8] int32, scales/biases
    [Nout, Kred/128] bf16, C [M, Nout] bf16; workspace any contiguous CUDA
    tensor of at least qmm_splitk_workspace_bytes(...) bytes.  options: a
    qmm_options for this call only (qmm_w4a16_g128_ex), else the process-wide
    settings."""
    M, Kred = A.shape
    Nout = Wq.shape[0]
    g = Kred // 128
    if Wq.shape != (Nout, Kred // 8) or C.shape != (M, Nout) or \
            scales.shape != (Nout, g) or biases.shape != (Nout, g):
        raise ValueError("qmm_w4a16_g128: inconsistent shapes")
    ws, ws_bytes = None, 0
    if workspace is not None:
        if not workspace.is_cuda or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous CUDA tensor")
        ws, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    used = _I(0)
    args = (_ptr(A, _BF16, "A"), _ptr(Wq, _WORDS, "Wq"), _ptr(scales, _BF16, "scales"),
            _ptr(biases, _BF16, "biases"), _ptr(C, _BF16, "C"), M, Kred, Nout, split_req,
            ctypes.byref(pol) if pol is not None else None, ws, ws_bytes, partial_dtype,
            _stream(stream), ctypes.byref(used))
    if options is not None:
        _check(lib().qmm_w4a16_g128_ex(*args, _opt(options)), "qmm_w4a16_g128_ex")
    else:
        rc = (_lib or lib()).qmm_w4a16_g128(*args)
        if rc != QMM_OK:
            raise QmmError(rc, "qmm_w4a16_g128")
    return used.value


def qmm_w4a16_g128_partition(A: torch.Tensor, Wq: torch.Tensor, scales: torch.Tensor,
                             biases: torch.Tensor, partials: torch.Tensor, split: int,
                             partial_dtype: int = QMM_PARTIAL_BF16, stream=None) -> None:
    """The partition kernel alone: partials [split, M, Nout] (bf16 or float32
    to match partial_dtype) receives one rounded plane per partition."""
    M, Kred = A.shape
    Nout = Wq.shape[0]
    if tuple(Wq.shape) != (Nout, Kred // 8) or \
            tuple(scales.shape) != (Nout, Kred // 128) or tuple(biases.shape) != (Nout, Kred // 128):
        raise ValueError("qmm_w4a16_g128_partition: inconsistent shapes")
    want = (torch.float32,) if partial_dtype == QMM_PARTIAL_F32 else _BF16
    rc = lib().qmm_w4a16_g128_partition(
        _dev(A, _BF16, "A"), _dev(Wq, _WORDS, "Wq"), _dev(scales, _BF16, "scales"),
        _dev(biases, _BF16, "biases"), _dev(partials, want, "partials"),
        partials.numel() * partials.element_size(), M, Kred, Nout, split, partial_dtype,
        _stream(stream))
    _check(rc, "qmm_w4a16_g128_partition")


TC_PIPELINE_FIELDS = ("issuers", "dequant_sets", "a_buffers", "weight_stage_groups",
                      "act_stage_groups", "act_stages", "weight_stages", "threads", "smem")


def qmm_tc_pipeline_config(bm: int, gpp: int, smem_limit: int = 232432) -> dict:
    """The tcgen05 kernel's pipeline shape for a tile and partition (host only)."""
    out = (_I * 9)()
    _check(lib().qmm_tc_pipeline_config(bm, gpp, smem_limit, out), "qmm_tc_pipeline_config")
    return dict(zip(TC_PIPELINE_FIELDS, list(out)))


def qmm_tc_persistent_pipeline_config(bm: int, gpp: int, smem_limit: int = 231408) -> dict:
    """The persistent grouped launch's pipeline shape (host only)."""
    out = (_I * 9)()
    _check(lib().qmm_tc_persistent_pipeline_config(bm, gpp, smem_limit, out),
           "qmm_tc_persistent_pipeline_config")
    return dict(zip(TC_PIPELINE_FIELDS, list(out)))


def qmm_static_scratch_bytes() -> int:
    return int(lib().qmm_static_scratch_bytes())


def qmm_w4a16_g128_noalloc(A: torch.Tensor, Wq: torch.Tensor, scales: torch.Tensor,
                           biases: torch.Tensor, C: torch.Tensor, split_req: int = 0,
                           pol: qmm_policy | None = None, partial_dtype: int = QMM_PARTIAL_BF16,
                           stream=None) -> int:
    """qmm_w4a16_g128 with the partial planes in the library's fixed device
    buffer (no workspace argument, no allocation); returns the split."""
    M, Kred = A.shape
    Nout = Wq.shape[0]
    if Wq.shape != (Nout, Kred // 8) or C.shape != (M, Nout) or \
            scales.shape != (Nout, Kred // 128) or biases.shape != (Nout, Kred // 128):
        raise ValueError("qmm_w4a16_g128_noalloc: inconsistent shapes")
    used = _I(0)
    rc = lib().qmm_w4a16_g128_noalloc(
        _ptr(A, _BF16, "A"), _ptr(Wq, _WORDS, "Wq"), _ptr(scales, _BF16, "scales"),
        _ptr(biases, _BF16, "biases"), _ptr(C, _BF16, "C"), M, Kred, Nout, split_req,
        ctypes.byref(pol) if pol is not None else None, partial_dtype, _stream(stream),
        ctypes.byref(used))
    _check(rc, "qmm_w4a16_g128_noalloc")
    return used.value


def qmm_splitk_reduce(partials: torch.Tensor, partial_dtype: int, split: int, M: int, Nout: int,
                      C: torch.Tensor, stream=None) -> None:
    want = (torch.float32,) if partial_dtype == QMM_PARTIAL_F32 else _BF16
    if partials.numel() < split * M * Nout or C.numel() < M * Nout:
        raise ValueError("qmm_splitk_reduce: buffers too small")
    _check(lib().qmm_splitk_reduce(_dev(partials, want, "partials"), partial_dtype, split, M, Nout,
                                   _dev(C, _BF16, "C"), _stream(stream)), "qmm_splitk_reduce")


def qmm_gemm_bf16_splitk(A: torch.Tensor, W: torch.Tensor, C: torch.Tensor, split: int,
                         workspace: torch.Tensor | None = None, stream=None) -> None:
    M, K = A.shape
    N = W.shape[0]
    if W.shape[1] != K or tuple(C.shape) != (M, N):
        raise ValueError("qmm_gemm_bf16_splitk: inconsistent shapes")
    ws, ws_bytes = None, 0
    if workspace is not None:
        ws, ws_bytes = ctypes.c_void_p(workspace.data_ptr()), \
            workspace.numel() * workspace.element_size()
    _check(lib().qmm_gemm_bf16_splitk(_dev(A, _BF16, "A"), _dev(W, _BF16, "W"),
                                      _dev(C, _BF16, "C"), M, N, K, split, ws, ws_bytes,
                                      _stream(stream)), "qmm_gemm_bf16_splitk")


def qmm_unpack_probe(Wq: torch.Tensor, Kred: int, q: torch.Tensor, stream=None) -> None:
    Nout = Wq.shape[0]
    if q.numel() < Nout * Kred:
        raise ValueError("qmm_unpack_probe: q too small")
    _check(lib().qmm_unpack_probe(_dev(Wq, _WORDS, "Wq"), Nout, Kred,
                                  _dev(q, (torch.uint8,), "q"), _stream(stream)),
           "qmm_unpack_probe")


def qmm_dequant_probe(Wq: torch.Tensor, scales: torch.Tensor, biases: torch.Tensor, Kred: int,
                      w: torch.Tensor, stream=None) -> None:
    Nout = Wq.shape[0]
    if w.numel() < Nout * Kred:
        raise ValueError("qmm_dequant_probe: w too small")
    _check(lib().qmm_dequant_probe(_dev(Wq, _WORDS, "Wq"), _dev(scales, _BF16, "scales"),
                                   _dev(biases, _BF16, "biases"), Nout, Kred,
                                   _dev(w, _BF16, "w"), _stream(stream)), "qmm_dequant_probe")


# ---- convenience ---------------------------------------------------------

def w4a16_matmul(A, Wq, scales, biases, split_req: int = 0, pol=None,
                 partial_dtype: int = QMM_PARTIAL_BF16, stream=None):
    """Allocate C (and the workspace the plan needs) with torch and call
    qmm_w4a16_g128.  Returns (C, split_used)."""
    M, Kred = A.shape
    Nout = Wq.shape[0]
    C = torch.empty((M, Nout), dtype=torch.bfloat16, device=A.device)
    # the workspace of the call as the library plans it, for any split_req
    # (policy, forced, QMM_SPLIT_PLANNED or QMM_SPLIT_BALANCED)
    nbytes = qmm_call_workspace_bytes(M, Kred, Nout, split_req, pol, partial_dtype)
    # zeroed: under QMM_REDUCE_FUSED the workspace's tail holds tile counters
    # that must start at zero
    ws = torch.zeros(max(nbytes, 16), dtype=torch.uint8, device=A.device) if nbytes else None
    used = qmm_w4a16_g128(A, Wq, scales, biases, C, split_req=split_req, pol=pol, workspace=ws,
                          partial_dtype=partial_dtype, stream=stream)
    return C, used


def to_device(problem: dict, device="cuda") -> dict:
    """Move a problem from split_w4a16_quantized_gb300.inputs to the GPU as the
    tensors qmm_w4a16_g128 takes."""
    import numpy as np

    def bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16) \
            .to(device)

    return {
        "A": bf16(problem["A"]),
        "Wq": torch.from_numpy(np.ascontiguousarray(problem["Wq"]).view(np.int32)).to(device),
        "scales": bf16(problem["scales"]),
        "biases": bf16(problem["biases"]),
    }


# ---- streaming host activations (copy in / compute / copy out) -------------

def _host(t: torch.Tensor, name: str) -> int:
    if not isinstance(t, torch.Tensor) or t.is_cuda or t.dtype != torch.bfloat16:
        raise TypeError("%s must be a host BF16 tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return t.data_ptr()


def stream_calls(chunks) -> "ctypes.Array":
    """chunks: sequence of dicts with host A and C (BF16, pinned to overlap) and
    device Wq, scales, biases.  Returns the qmm_stream_call array."""
    arr = (qmm_stream_call * len(chunks))()
    for i, c in enumerate(chunks):
        M, Kred = c["A"].shape
        Nout = c["Wq"].shape[0]
        if tuple(c["C"].shape) != (M, Nout):
            raise ValueError("chunk %d: C must be [M, Nout]" % i)
        arr[i] = qmm_stream_call(_host(c["A"], "A"), _host(c["C"], "C"),
                                 _dev(c["Wq"], _WORDS, "Wq").value,
                                 _dev(c["scales"], _BF16, "scales").value,
                                 _dev(c["biases"], _BF16, "biases").value, M, Kred, Nout)
    return arr


def qmm_stream_arena_bytes(calls, buffers: int) -> int:
    return int(lib().qmm_stream_arena_bytes(calls, len(calls), buffers))


def qmm_w4a16_g128_stream(calls, buffers: int, arena: torch.Tensor, stream_in=None,
                          stream_compute=None, stream_out=None):
    """Enqueue the copy-in / compute / copy-out pipeline; returns the splits used.
    Synchronize stream_out before reading the host outputs."""
    n = len(calls)
    used = (_I * n)()
    _check(lib().qmm_w4a16_g128_stream(calls, n, buffers, _dev(arena, (torch.uint8,), "arena"),
                                       arena.numel(), _stream(stream_in),
                                       _stream(stream_compute), _stream(stream_out), used),
           "qmm_w4a16_g128_stream")
    return list(used)


def qmm_overlap_schedule(n: int, buffers: int, t_load, t_comp, t_store, out_reuse=False,
                         with_events=False):
    """The pipeline's schedule model: end of the last store (and the [n, 6] events)."""
    import numpy as np
    t = [np.ascontiguousarray(np.broadcast_to(np.asarray(x, np.float64), (n,)))
         for x in (t_load, t_comp, t_store)]
    D = ctypes.POINTER(ctypes.c_double)
    T = ctypes.c_double(0.0)
    ev = np.empty((n, 6), np.float64) if with_events else None
    _check(lib().qmm_overlap_schedule(n, buffers, *(a.ctypes.data_as(D) for a in t),
                                      int(bool(out_reuse)), ctypes.byref(T),
                                      ev.ctypes.data_as(D) if ev is not None else None),
           "qmm_overlap_schedule")
    return (T.value, ev) if with_events else T.value


# ---- several independent calls in few launches ----------------------------

def group_calls(calls) -> "ctypes.Array":
    """calls: sequence of dicts of device tensors A, Wq, scales, biases, C.
    Returns the qmm_group_call array (shapes checked here)."""
    arr = (qmm_group_call * len(calls))()
    for i, c in enumerate(calls):
        M, Kred = c["A"].shape
        Nout = c["Wq"].shape[0]
        if tuple(c["Wq"].shape) != (Nout, Kred // 8) or tuple(c["C"].shape) != (M, Nout) or \
                tuple(c["scales"].shape) != (Nout, Kred // 128) or \
                tuple(c["biases"].shape) != (Nout, Kred // 128):
            raise ValueError("group call %d: inconsistent shapes" % i)
        arr[i] = qmm_group_call(_dev(c["A"], _BF16, "A").value, _dev(c["Wq"], _WORDS, "Wq").value,
                                _dev(c["scales"], _BF16, "scales").value,
                                _dev(c["biases"], _BF16, "biases").value,
                                _dev(c["C"], _BF16, "C").value, M, Kred, Nout)
    return arr


def qmm_group_workspace_bytes(calls, partial_dtype: int = QMM_PARTIAL_BF16,
                              options=None) -> int:
    if options is not None:
        return int(lib().qmm_group_workspace_bytes_ex(calls, len(calls), partial_dtype,
                                                       _opt(options)))
    return int(lib().qmm_group_workspace_bytes(calls, len(calls), partial_dtype))


def qmm_w4a16_g128_grouped(calls, workspace: torch.Tensor | None = None,
                           partial_dtype: int = QMM_PARTIAL_BF16, stream=None, options=None):
    """Every call's C with its policy split, in few launches; returns the splits."""
    n = len(calls)
    used = (_I * n)()
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr = _dev(workspace, (workspace.dtype,), "workspace")
        ws_bytes = workspace.numel() * workspace.element_size()
    args = (calls, n, ws_ptr, ws_bytes, partial_dtype, _stream(stream), used)
    if options is not None:
        _check(lib().qmm_w4a16_g128_grouped_ex(*args, _opt(options)), "qmm_w4a16_g128_grouped_ex")
    else:
        _check(lib().qmm_w4a16_g128_grouped(*args), "qmm_w4a16_g128_grouped")
    return list(used)


# ---- split-KV decode attention ---------------------------------------------

def qmm_decode_attention_splits(B: int, Hq: int, Hkv: int, Lmax: int, num_sms: int = 0) -> int:
    s = _I(0)
    _check(lib().qmm_decode_attention_splits(B, Hq, Hkv, Lmax, num_sms, ctypes.byref(s)),
           "qmm_decode_attention_splits")
    return s.value


def qmm_decode_attention_workspace_bytes(B: int, Hq: int, D: int, splits: int) -> int:
    return int(lib().qmm_decode_attention_workspace_bytes(B, Hq, D, splits))


def qmm_decode_attention(q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, lens: torch.Tensor,
                         O: torch.Tensor, scale: float = 0.0, splits_req: int = 0,
                         workspace: torch.Tensor | None = None, stream=None) -> int:
    """O = split-KV decode attention (see qmm.h); returns the split used.
    q [B, Hq, D], K/V [B, Hkv, Lmax, D] bf16, lens int32 [B] (device), O [B, Hq, D] bf16."""
    B, Hq, D = q.shape
    _, Hkv, Lmax, _ = K.shape
    if tuple(K.shape) != (B, Hkv, Lmax, D) or tuple(V.shape) != tuple(K.shape) or \
            tuple(O.shape) != (B, Hq, D) or tuple(lens.shape) != (B,):
        raise ValueError("qmm_decode_attention: inconsistent shapes")
    used = _I(0)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr = _dev(workspace, (workspace.dtype,), "workspace")
        ws_bytes = workspace.numel() * workspace.element_size()
    _check(lib().qmm_decode_attention(_dev(q, _BF16, "q"), _dev(K, _BF16, "K"),
                                      _dev(V, _BF16, "V"), _dev(lens, (torch.int32,), "lens"),
                                      _dev(O, _BF16, "O"), B, Hq, Hkv, Lmax, D, float(scale),
                                      splits_req, ws_ptr, ws_bytes, _stream(stream),
                                      ctypes.byref(used)), "qmm_decode_attention")
    return used.value


def attention_to_device(problem: dict, device="cuda") -> dict:
    """Upload an inputs.make_attention problem: q, K, V as bf16, lens as int32."""
    def bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16) \
            .to(device)
    return {"q": bf16(problem["q"]), "K": bf16(problem["K"]), "V": bf16(problem["V"]),
            "lens": torch.from_numpy(problem["lens"]).to(device)}
