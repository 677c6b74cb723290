"""Python binding of the qmuon C ABI (``include/qmuon.h``).

Argument marshalling only: every function below converts its arguments to
the C types of the entry point with the same name, calls ``libqmuon.so``
and raises :class:`QmuonError` on a non-OK status.  All arithmetic runs in
the library's CUDA kernels; there is no Python or CPU fallback, and calling
any entry point without the built library raises.

Device buffers are passed as torch tensors (their ``data_ptr()``) or as raw
integer addresses; ``stream`` is a ``torch.cuda.Stream``, a raw
``cudaStream_t`` integer, or ``None`` for torch's current stream.
"""

from __future__ import annotations

import ctypes as C
import os
from typing import Iterable, Optional, Sequence

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqmuon.so")

QMUON_OK = 0
QMUON_ERR_INVALID_ARGUMENT = 1
QMUON_ERR_MISALIGNED_SEGMENT = 2
QMUON_ERR_UNSUPPORTED = 3
QMUON_ERR_WORKSPACE_TOO_SMALL = 4
QMUON_ERR_CUDA = 5
QMUON_ERR_TIMEOUT = 6
QMUON_ERR_OUT_OF_MEMORY = 7

QMUON_Q8_INT8, QMUON_Q8_UINT8 = 0, 1
QMUON_BF16, QMUON_FP16, QMUON_FP32 = 0, 1, 2
QMUON_WS_UPDATE, QMUON_WS_STEP = 0, 1
QMUON_NS_BF16, QMUON_NS_MXFP8 = 0, 1

Q8_KINDS = {"int8": QMUON_Q8_INT8, "uint8": QMUON_Q8_UINT8}
DTYPES = {"bf16": QMUON_BF16, "f16": QMUON_FP16, "f32": QMUON_FP32}


class QmuonError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        detail = ""
        try:
            detail = lib().qmuon_last_error().decode()
        except Exception:
            pass
        super().__init__(f"{where}: {status_string(status)} (status {status})" + (f" -- {detail}" if detail else ""))


class qmuon_tensor(C.Structure):
    _fields_ = [("q8", C.c_void_p), ("absmax", C.c_void_p), ("grad", C.c_void_p),
                ("rows", C.c_int64), ("cols", C.c_int64)]


class qmuon_norm_segment(C.Structure):
    _fields_ = [("tensor_index", C.c_int32), ("group_id", C.c_int32),
                ("start", C.c_int64), ("length", C.c_int64)]


class qmuon_ns_problem(C.Structure):
    _fields_ = [("x", C.c_void_p), ("rows", C.c_int64), ("cols", C.c_int64), ("ld", C.c_int64),
                ("inv_norm", C.c_void_p), ("input", C.c_int32), ("reserved", C.c_int32),
                ("payload", C.c_void_p), ("scale_inv", C.c_void_p)]


class qmuon_grasp_matrix(C.Structure):
    _fields_ = [("rows", C.c_int64), ("cols", C.c_int64), ("res", C.c_void_p), ("res_rmax", C.c_void_p),
                ("res_cmax", C.c_void_p), ("p", C.c_void_p), ("p_rmax", C.c_void_p), ("p_cmax", C.c_void_p),
                ("r", C.c_void_p), ("r_rmax", C.c_void_p), ("r_cmax", C.c_void_p), ("grad", C.c_void_p)]


GRASP_RANK, GRASP_BLOCK = 8, 64

COUNTER_FIELDS = (
    "update_calls", "update_sr_calls", "carrier_calls", "ns_calls", "step_block_calls", "step_full_calls",
    "step_sr_calls", "step_host_fed_calls", "grasp_calls", "grad_bf16_tensors", "grad_fp16_tensors",
    "grad_fp32_tensors", "state_int8_tensors", "state_uint8_tensors", "carrier_payload_u8_tensors",
    "carrier_scale_u8_tensors", "carrier_inv_norm_f32_values", "ns_bf16_problems", "ns_mxfp8_problems",
    "ns_bf16_handoff_bytes", "weight_f32_tensors", "grasp_matrices", "host_pulled_bytes", "host_copied_bytes")


class qmuon_counters(C.Structure):
    _fields_ = [(f, C.c_uint64) for f in COUNTER_FIELDS]

_lib_handle = None


def lib() -> C.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib_handle
    if _lib_handle is not None:
        return _lib_handle
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"qmuon CUDA library not built ({LIB_PATH} missing); "
                           "run `python -m memory_reduced_muon_gb300.build`")
    L = C.CDLL(LIB_PATH)
    vp, i32, i64, f32, sz = C.c_void_p, C.c_int32, C.c_int64, C.c_float, C.c_size_t
    sig = {
        "qmuon_plan_create": (i32, [C.POINTER(qmuon_tensor), i32, i32, i32, C.POINTER(qmuon_norm_segment),
                                    i32, i32, i32, i32, C.POINTER(vp)]),
        "qmuon_plan_destroy": (None, [vp]),
        "qmuon_plan_info": (i32, [vp, C.POINTER(i64), C.POINTER(i32), C.POINTER(i32), C.POINTER(i32)]),
        "qmuon_workspace_size": (sz, [vp, i32]),
        "qmuon_update_multi_normalize_groups": (i32, [vp, f32, i32, vp, vp, vp, sz, vp]),
        "qmuon_update_multi_normalize_groups_sr": (i32, [vp, f32, i32, C.c_uint64, i64, vp, vp, vp, sz, vp]),
        "qmuon_plan_set_stochastic_rounding": (i32, [vp, i32, C.c_uint64]),
        "qmuon_plan_set_host_ingest": (i32, [vp, i32]),
        "qmuon_grasp_workspace_size": (sz, [C.POINTER(qmuon_grasp_matrix), i32]),
        "qmuon_grasp_step": (i32, [C.POINTER(qmuon_grasp_matrix), i32, f32, vp, sz, vp]),
        "qmuon_carrier_workspace_size": (sz, [i64, i64]),
        "qmuon_update_mxfp8_carrier": (i32, [C.POINTER(qmuon_tensor), i32, i32, f32, vp, vp, vp, vp, sz, vp]),
        "qmuon_update_mxfp8_carrier_multi": (i32, [vp, f32, C.POINTER(vp), C.POINTER(vp), vp, vp, vp, sz, vp]),
        "qmuon_ns_workspace_size": (sz, [C.POINTER(qmuon_ns_problem), i32]),
        "qmuon_newton_schulz_batched": (i32, [C.POINTER(qmuon_ns_problem), i32, i32, C.POINTER(f32), vp, sz, vp]),
        "qmuon_step": (i32, [vp, i64, i32, f32, f32, f32, C.POINTER(vp), C.POINTER(f32), i32, vp, vp, sz, vp]),
        "qmuon_sync_status": (i32, [vp, vp]),
        "qmuon_status_string": (C.c_char_p, [i32]),
        "qmuon_version": (C.c_char_p, []),
        "qmuon_last_error": (C.c_char_p, []),
        "qmuon_update_normalize_noalloc": (i32, [C.POINTER(qmuon_tensor), i32, i32, f32, vp, vp, vp]),
        "qmuon_step_prepare": (i32, [vp, C.POINTER(vp), vp, sz]),
        "qmuon_step_from_host": (i32, [vp, i64, i32, f32, f32, f32, C.POINTER(vp), C.POINTER(f32), i32,
                                       C.POINTER(vp), vp, vp, vp, sz, vp, vp]),
        "qmuon_plan_set_nonfinite_counter": (i32, [vp, vp]),
        "qmuon_noalloc_sync_status": (i32, [vp]),
        "qmuon_noalloc_inject_status": (i32, [i32, C.c_uint32]),
        "qmuon_get_counters": (i32, [C.POINTER(qmuon_counters), sz]),
        "qmuon_reset_counters": (None, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib_handle = L
    return L


def exported_symbols() -> list:
    return ["qmuon_plan_create", "qmuon_plan_destroy", "qmuon_plan_info", "qmuon_workspace_size",
            "qmuon_update_multi_normalize_groups", "qmuon_carrier_workspace_size",
            "qmuon_update_mxfp8_carrier", "qmuon_ns_workspace_size", "qmuon_newton_schulz_batched",
            "qmuon_step", "qmuon_sync_status", "qmuon_status_string", "qmuon_version", "qmuon_last_error",
            "qmuon_update_normalize_noalloc", "qmuon_step_prepare", "qmuon_update_multi_normalize_groups_sr",
            "qmuon_plan_set_stochastic_rounding", "qmuon_update_mxfp8_carrier_multi",
            "qmuon_grasp_workspace_size", "qmuon_grasp_step", "qmuon_step_from_host",
            "qmuon_plan_set_nonfinite_counter", "qmuon_noalloc_sync_status", "qmuon_noalloc_inject_status",
            "qmuon_get_counters", "qmuon_reset_counters", "qmuon_plan_set_host_ingest"]


# --------------------------------------------------------------------------
# marshalling helpers
# --------------------------------------------------------------------------

def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def _nbytes(x) -> int:
    return int(x.numel() * x.element_size())


def _check(status: int, where: str):
    if status != QMUON_OK:
        raise QmuonError(status, where)


def status_string(status: int) -> str:
    try:
        return lib().qmuon_status_string(int(status)).decode()
    except RuntimeError:
        return "library not built"


qmuon_status_string = status_string


def qmuon_version() -> str:
    return lib().qmuon_version().decode()


def qmuon_last_error() -> str:
    return lib().qmuon_last_error().decode()


class Plan:
    """An owned ``qmuon_plan*`` (destroyed with the object)."""

    def __init__(self, handle: int, keepalive):
        self.handle = handle
        self._keep = keepalive

    def __del__(self):
        h, self.handle = getattr(self, "handle", None), None
        if h and _lib_handle is not None:
            _lib_handle.qmuon_plan_destroy(h)


def tensor_desc(q8, absmax, grad, rows: int, cols: int) -> qmuon_tensor:
    return qmuon_tensor(_ptr(q8), _ptr(absmax), _ptr(grad), int(rows), int(cols))


def qmuon_plan_create(tensors: Sequence, q8_kind="int8", grad_dtype="bf16", segments=None,
                      n_groups: int = 0, tile=(1, 1)) -> Plan:
    """``tensors``: ``(q8, absmax, grad, rows, cols)`` tuples or ``qmuon_tensor``;
    ``segments``: ``(tensor_index, start, length, group_id)`` tuples."""
    descs = [t if isinstance(t, qmuon_tensor) else tensor_desc(*t) for t in tensors]
    arr = (qmuon_tensor * max(1, len(descs)))(*descs)
    segs = None
    nseg = 0
    if segments:
        nseg = len(segments)
        segs = (qmuon_norm_segment * nseg)(*[
            s if isinstance(s, qmuon_norm_segment) else
            qmuon_norm_segment(int(s[0]), int(s[3]), int(s[1]), int(s[2])) for s in segments])
    out = C.c_void_p()
    q = Q8_KINDS.get(q8_kind, q8_kind)
    d = DTYPES.get(grad_dtype, grad_dtype)
    st = lib().qmuon_plan_create(arr, len(descs), q, d, segs, nseg, int(n_groups), int(tile[0]), int(tile[1]),
                                 C.byref(out))
    _check(st, "qmuon_plan_create")
    return Plan(out.value, (tensors, segments))


def qmuon_plan_destroy(plan: Plan):
    if plan.handle:
        lib().qmuon_plan_destroy(plan.handle)
        plan.handle = None


def qmuon_plan_info(plan: Plan) -> dict:
    nb, g, gf, gb = C.c_int64(), C.c_int32(), C.c_int32(), C.c_int32()
    _check(lib().qmuon_plan_info(plan.handle, C.byref(nb), C.byref(g), C.byref(gf), C.byref(gb)),
           "qmuon_plan_info")
    return {"n_blocks": nb.value, "n_groups": g.value, "n_full_groups": gf.value, "n_block_groups": gb.value}


def qmuon_workspace_size(plan: Plan, which: int = QMUON_WS_UPDATE) -> int:
    return int(lib().qmuon_workspace_size(plan.handle, int(which)))


def qmuon_update_multi_normalize_groups(plan: Plan, beta: float, normalize_mode: int, group_sumsq, group_inv_norm,
                                        ws, ws_bytes: Optional[int] = None, stream=None):
    st = lib().qmuon_update_multi_normalize_groups(
        plan.handle, float(beta), int(normalize_mode), _ptr(group_sumsq), _ptr(group_inv_norm), _ptr(ws),
        _nbytes(ws) if ws_bytes is None else int(ws_bytes), _stream(stream))
    _check(st, "qmuon_update_multi_normalize_groups")


def qmuon_update_multi_normalize_groups_sr(plan: Plan, beta: float, normalize_mode: int, seed: int, step: int,
                                           group_sumsq, group_inv_norm, ws, ws_bytes: Optional[int] = None,
                                           stream=None):
    st = lib().qmuon_update_multi_normalize_groups_sr(
        plan.handle, float(beta), int(normalize_mode), int(seed) & 0xFFFFFFFFFFFFFFFF, int(step),
        _ptr(group_sumsq), _ptr(group_inv_norm), _ptr(ws), _nbytes(ws) if ws_bytes is None else int(ws_bytes),
        _stream(stream))
    _check(st, "qmuon_update_multi_normalize_groups_sr")


def qmuon_plan_set_nonfinite_counter(plan: Plan, counter):
    """``counter``: a device uint32/int32 tensor of one element, or None."""
    _check(lib().qmuon_plan_set_nonfinite_counter(plan.handle, _ptr(counter)), "qmuon_plan_set_nonfinite_counter")


QMUON_INGEST_PULL = 0
QMUON_INGEST_COPY = 1


def qmuon_plan_set_host_ingest(plan: Plan, mode: int):
    """QMUON_INGEST_PULL (default) or QMUON_INGEST_COPY for qmuon_step_from_host."""
    _check(lib().qmuon_plan_set_host_ingest(plan.handle, int(mode)), "qmuon_plan_set_host_ingest")


def qmuon_plan_set_stochastic_rounding(plan: Plan, enable: bool, seed: int = 0):
    _check(lib().qmuon_plan_set_stochastic_rounding(plan.handle, 1 if enable else 0,
                                                    int(seed) & 0xFFFFFFFFFFFFFFFF),
           "qmuon_plan_set_stochastic_rounding")


def qmuon_carrier_workspace_size(rows: int, cols: int) -> int:
    return int(lib().qmuon_carrier_workspace_size(int(rows), int(cols)))


def qmuon_update_mxfp8_carrier(q8, absmax, grad, rows: int, cols: int, q8_kind, grad_dtype, beta: float,
                               payload, scale_inv, inv_norm, ws, ws_bytes: Optional[int] = None, stream=None):
    t = tensor_desc(q8, absmax, grad, rows, cols)
    st = lib().qmuon_update_mxfp8_carrier(
        C.byref(t), Q8_KINDS.get(q8_kind, q8_kind), DTYPES.get(grad_dtype, grad_dtype), float(beta),
        _ptr(payload), _ptr(scale_inv), _ptr(inv_norm), _ptr(ws),
        _nbytes(ws) if ws_bytes is None else int(ws_bytes), _stream(stream))
    _check(st, "qmuon_update_mxfp8_carrier")


def qmuon_update_mxfp8_carrier_multi(plan: Plan, beta: float, payloads: Sequence, scale_invs: Sequence, inv_norms,
                                     ws, group_sumsq=None, ws_bytes: Optional[int] = None, stream=None):
    n = len(payloads)
    pp = (C.c_void_p * max(1, n))(*[_ptr(x) for x in payloads])
    sp = (C.c_void_p * max(1, n))(*[_ptr(x) for x in scale_invs])
    st = lib().qmuon_update_mxfp8_carrier_multi(plan.handle, float(beta), pp, sp, _ptr(inv_norms), _ptr(group_sumsq),
                                                _ptr(ws), _nbytes(ws) if ws_bytes is None else int(ws_bytes),
                                                _stream(stream))
    _check(st, "qmuon_update_mxfp8_carrier_multi")


def ns_problem(x, rows: int, cols: int, ld: Optional[int] = None, inv_norm=None, input_kind=QMUON_NS_BF16,
               payload=None, scale_inv=None) -> qmuon_ns_problem:
    return qmuon_ns_problem(_ptr(x), int(rows), int(cols), int(cols if ld is None else ld), _ptr(inv_norm),
                            int(input_kind), 0, _ptr(payload), _ptr(scale_inv))


def _problems(problems: Iterable):
    ps = [p if isinstance(p, qmuon_ns_problem) else ns_problem(*p) for p in problems]
    return (qmuon_ns_problem * max(1, len(ps)))(*ps), len(ps)


def qmuon_ns_workspace_size(problems) -> int:
    arr, n = _problems(problems)
    return int(lib().qmuon_ns_workspace_size(arr, n))


def qmuon_newton_schulz_batched(problems, iters: int, coeffs, ws, ws_bytes: Optional[int] = None, stream=None):
    arr, n = _problems(problems)
    cf = (C.c_float * 3)(*[float(c) for c in coeffs])
    st = lib().qmuon_newton_schulz_batched(arr, n, int(iters), cf, _ptr(ws),
                                           _nbytes(ws) if ws_bytes is None else int(ws_bytes), _stream(stream))
    _check(st, "qmuon_newton_schulz_batched")


def qmuon_step(plan: Plan, t: int, P: int, beta: float, eta_full: float, eta_block: float, weights,
               coeffs, iters: int, group_sumsq, ws, ws_bytes: Optional[int] = None, stream=None):
    wp = (C.c_void_p * max(1, len(weights)))(*[_ptr(w) for w in weights])
    cf = (C.c_float * 3)(*[float(c) for c in coeffs])
    st = lib().qmuon_step(plan.handle, int(t), int(P), float(beta), float(eta_full), float(eta_block), wp, cf,
                          int(iters), _ptr(group_sumsq), _ptr(ws),
                          _nbytes(ws) if ws_bytes is None else int(ws_bytes), _stream(stream))
    _check(st, "qmuon_step")


def qmuon_step_from_host(plan: Plan, t: int, P: int, beta: float, eta_full: float, eta_block: float, weights,
                         coeffs, iters: int, host_grads, host_group_sumsq, group_sumsq, ws,
                         ws_bytes: Optional[int] = None, stream=None, copy_stream=None):
    """``host_grads``: host tensors (page-locked for overlap) or raw host
    addresses, one per plan tensor; ``host_group_sumsq``: a host fp32 tensor
    or None."""
    wp = (C.c_void_p * max(1, len(weights)))(*[_ptr(w) for w in weights])
    hp = (C.c_void_p * max(1, len(host_grads)))(*[_ptr(h) for h in host_grads])
    cf = (C.c_float * 3)(*[float(c) for c in coeffs])
    st = lib().qmuon_step_from_host(plan.handle, int(t), int(P), float(beta), float(eta_full), float(eta_block), wp,
                                    cf, int(iters), hp, _ptr(host_group_sumsq), _ptr(group_sumsq), _ptr(ws),
                                    _nbytes(ws) if ws_bytes is None else int(ws_bytes), _stream(stream),
                                    _stream(copy_stream))
    _check(st, "qmuon_step_from_host")


def qmuon_update_normalize_noalloc(q8, absmax, grad, rows: int, cols: int, q8_kind, grad_dtype, beta: float,
                                   sumsq=None, inv_norm=None, stream=None):
    """The single-tensor update whose scratch is a static array in the
    library (no plan, no workspace, no device allocation)."""
    t = tensor_desc(q8, absmax, grad, rows, cols)
    st = lib().qmuon_update_normalize_noalloc(C.byref(t), Q8_KINDS.get(q8_kind, q8_kind),
                                              DTYPES.get(grad_dtype, grad_dtype), float(beta), _ptr(sumsq),
                                              _ptr(inv_norm), _stream(stream))
    _check(st, "qmuon_update_normalize_noalloc")


def qmuon_noalloc_sync_status(stream=None):
    """Waits for the stream and raises if a kernel of the allocation-free
    update recorded a failure since the last read (the record is cleared)."""
    _check(lib().qmuon_noalloc_sync_status(_stream(stream)), "qmuon_noalloc_sync_status")


def qmuon_noalloc_inject_status(status: int, site: int = 0):
    """Records ``status`` as if a kernel of the allocation-free update had
    failed at ``site`` (for testing a caller's failure handling)."""
    _check(lib().qmuon_noalloc_inject_status(int(status), int(site)), "qmuon_noalloc_inject_status")


def qmuon_get_counters() -> dict:
    """The library's path and dtype tallies (calls that returned OK, and the
    tensors they read or wrote), field name -> count."""
    c = qmuon_counters()
    _check(lib().qmuon_get_counters(C.byref(c), C.sizeof(c)), "qmuon_get_counters")
    return {f: int(getattr(c, f)) for f in COUNTER_FIELDS}


def qmuon_reset_counters():
    lib().qmuon_reset_counters()


def qmuon_step_prepare(plan: Plan, weights, ws, ws_bytes: Optional[int] = None):
    wp = (C.c_void_p * max(1, len(weights)))(*[_ptr(w) for w in weights])
    _check(lib().qmuon_step_prepare(plan.handle, wp, _ptr(ws), _nbytes(ws) if ws_bytes is None else int(ws_bytes)),
           "qmuon_step_prepare")


def qmuon_sync_status(ws, stream=None):
    _check(lib().qmuon_sync_status(_ptr(ws), _stream(stream)), "qmuon_sync_status")


# --------------------------------------------------------------------------
# 4-bit GRASP momentum state
# --------------------------------------------------------------------------

def grasp_matrix(rows: int, cols: int, res, res_rmax, res_cmax, p, p_rmax, p_cmax, r, r_rmax, r_cmax,
                 grad) -> qmuon_grasp_matrix:
    return qmuon_grasp_matrix(int(rows), int(cols), _ptr(res), _ptr(res_rmax), _ptr(res_cmax), _ptr(p), _ptr(p_rmax),
                              _ptr(p_cmax), _ptr(r), _ptr(r_rmax), _ptr(r_cmax), _ptr(grad))


def _grasp_array(matrices: Sequence):
    arr = (qmuon_grasp_matrix * max(1, len(matrices)))(*matrices)
    return arr, len(matrices)


def qmuon_grasp_workspace_size(matrices: Sequence) -> int:
    arr, n = _grasp_array(matrices)
    return int(lib().qmuon_grasp_workspace_size(arr, n))


def qmuon_grasp_step(matrices: Sequence, mu: float, ws, ws_bytes: Optional[int] = None, stream=None):
    arr, n = _grasp_array(matrices)
    _check(lib().qmuon_grasp_step(arr, n, float(mu), _ptr(ws), _nbytes(ws) if ws_bytes is None else int(ws_bytes),
                                  _stream(stream)), "qmuon_grasp_step")
