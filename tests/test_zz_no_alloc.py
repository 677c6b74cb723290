"""The allocation-free update entry point against the planned entry point.

``qmuon_update_normalize_noalloc`` serves callers that cannot allocate device
memory when they update (no plan, no workspace: its scratch is a static array
inside the library).  Its outputs must equal those of
``qmuon_update_multi_normalize_groups`` on a one-tensor plan: codes, absmax
and stored momentum bit for bit, the sum of squares and inverse norm within
the relative 1e-5 the other GPU tests use -- on two calls in a row, so that
the second call starts from the array's leftover contents.  A failure that a
kernel records on the GPU comes back through ``qmuon_noalloc_sync_status``:
after clean calls it returns QMUON_OK, and a recorded status survives later
calls until it is read, then is cleared.  This file sorts last so a
stop-at-first-failure run has executed every other test first.
"""

import ctypes as C

import numpy as np
import pytest
import torch

import memory_reduced_muon_gb300 as q
import workloads

from gpu_util import random_grad

pytestmark = pytest.mark.gpu


def _noalloc(t, q8_kind, grad_dtype, s, i):
    return q.lib().qmuon_update_normalize_noalloc(C.byref(t), q.Q8_KINDS[q8_kind], q.DTYPES[grad_dtype],
                                                  C.c_float(0.95), None if s is None else s.data_ptr(),
                                                  None if i is None else i.data_ptr(),
                                                  torch.cuda.current_stream().cuda_stream)


def _sync_status():
    return q.lib().qmuon_noalloc_sync_status(torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("shape,q8_kind,grad_dtype,sums", [
    ((1000, 777), "int8", "bf16", True),      # ragged: the last quantization block is partial
    ((4096, 4096), "uint8", "bf16", True),    # several waves of CTAs
    ((64, 256), "int8", "f32", True),
    ((333, 512), "uint8", "f16", True),
    ((1000, 777), "int8", "bf16", False),     # no sums asked for: the launch skips the reduction
])
def test_noalloc_matches_planned_update_twice(shape, q8_kind, grad_dtype, sums):
    rows, cols = shape
    m = workloads.Matrix("t", rows, cols)
    q_a, a_a = workloads.random_state(m, 321, q8_kind, device="cuda")
    q_b, a_b = q_a.clone(), a_a.clone()
    plan = None
    ws = None
    for call in range(2):
        g = random_grad(rows * cols, grad_dtype, 55 + call)
        g_a, g_b = g.clone(), g.clone()
        s_a = torch.full((1,), -1.0, device="cuda")
        i_a = torch.full((1,), -1.0, device="cuda")
        s_b = torch.full((1,), -1.0, device="cuda")
        i_b = torch.full((1,), -1.0, device="cuda")
        # the existing entry point, with a plan and a workspace
        plan = q.qmuon_plan_create([(q_a, a_a, g_a, rows, cols)], q8_kind, grad_dtype)
        ws = torch.empty(q.qmuon_workspace_size(plan), dtype=torch.uint8, device="cuda")
        q.qmuon_update_multi_normalize_groups(plan, 0.95, 2, s_a, i_a, ws)
        # the allocation-free one, called through the C ABI
        t = q.tensor_desc(q_b, a_b, g_b, rows, cols)
        st = _noalloc(t, q8_kind, grad_dtype, s_b if sums else None, i_b if sums else None)
        assert st == q.QMUON_OK, q.qmuon_last_error()
        assert _sync_status() == q.QMUON_OK, q.qmuon_last_error()
        torch.cuda.synchronize()
        assert torch.equal(q_a, q_b)
        assert torch.equal(a_a, a_b)
        assert torch.equal(g_a.view(torch.uint8), g_b.view(torch.uint8))
        if sums:
            np.testing.assert_allclose(s_b.item(), s_a.item(), rtol=1e-5)
            np.testing.assert_allclose(i_b.item(), i_a.item(), rtol=1e-5)
            assert s_b.item() > 0
        else:
            assert s_b.item() == -1.0 and i_b.item() == -1.0   # untouched


def test_noalloc_status_is_kept_until_read_then_cleared():
    # a status recorded in the static array (here written from the host, as a
    # kernel would record a wait that expired) is reported once and cleared
    assert _sync_status() == q.QMUON_OK, q.qmuon_last_error()
    assert q.lib().qmuon_noalloc_inject_status(q.QMUON_ERR_TIMEOUT, 0x1300) == q.QMUON_OK
    assert _sync_status() == q.QMUON_ERR_TIMEOUT
    assert "0x1300" in q.qmuon_last_error()
    assert _sync_status() == q.QMUON_OK
    # later calls neither erase it nor stop because of it: they compute as usual
    rows, cols = 700, 512
    m = workloads.Matrix("t", rows, cols)
    q_a, a_a = workloads.random_state(m, 9, "int8", device="cuda")
    q_b, a_b = q_a.clone(), a_a.clone()
    assert q.lib().qmuon_noalloc_inject_status(q.QMUON_ERR_TIMEOUT, 0x1100) == q.QMUON_OK
    for call in range(2):
        g = random_grad(rows * cols, "bf16", 77 + call)
        g_a, g_b = g.clone(), g.clone()
        s_a, i_a = torch.zeros(1, device="cuda"), torch.zeros(1, device="cuda")
        s_b, i_b = torch.zeros(1, device="cuda"), torch.zeros(1, device="cuda")
        plan = q.qmuon_plan_create([(q_a, a_a, g_a, rows, cols)], "int8", "bf16")
        ws = torch.empty(q.qmuon_workspace_size(plan), dtype=torch.uint8, device="cuda")
        q.qmuon_update_multi_normalize_groups(plan, 0.95, 2, s_a, i_a, ws)
        assert _noalloc(q.tensor_desc(q_b, a_b, g_b, rows, cols), "int8", "bf16", s_b, i_b) == q.QMUON_OK
        torch.cuda.synchronize()
        assert torch.equal(q_a, q_b) and torch.equal(a_a, a_b)
        assert torch.equal(g_a.view(torch.uint8), g_b.view(torch.uint8))
        np.testing.assert_allclose(i_b.item(), i_a.item(), rtol=1e-5)
    assert _sync_status() == q.QMUON_ERR_TIMEOUT
    assert "0x1100" in q.qmuon_last_error()
    assert _sync_status() == q.QMUON_OK


def test_noalloc_rejects_oversized_and_bad_args():
    L = q.lib()
    too_big = q.qmuon_tensor(0x7F0000000000, 0x7F0000100000, 0x7F0000200000, 1 << 16, (1 << 15) + 1)
    st = L.qmuon_update_normalize_noalloc(C.byref(too_big), 0, 0, C.c_float(0.9), None, None, None)
    assert st == q.QMUON_ERR_INVALID_ARGUMENT
    assert "QMUON_NOALLOC_MAX_ELEMS" in q.qmuon_last_error()
    assert L.qmuon_update_normalize_noalloc(None, 0, 0, C.c_float(0.9), None, None, None) == \
        q.QMUON_ERR_INVALID_ARGUMENT
    assert L.qmuon_noalloc_inject_status(q.QMUON_OK, 0) == q.QMUON_ERR_INVALID_ARGUMENT
    assert _sync_status() == q.QMUON_OK
