"""The C ABI on the CPU: the library loads, exports every symbol the header
declares, and rejects invalid arguments on the host (status codes, nothing
launched) -- none of these calls needs a GPU."""

import ctypes as C
import os
import re
import subprocess
import sys

import pytest

import memory_reduced_muon_gb300 as q

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qmuon.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(q.LIB_PATH):
        from memory_reduced_muon_gb300 import build
        build.build()
    return q.lib()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"QMUON_API\s+[\w\s\*]+?\b(qmuon_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_symbols()
    for must in ["qmuon_update_multi_normalize_groups", "qmuon_update_mxfp8_carrier",
                 "qmuon_newton_schulz_batched", "qmuon_step", "qmuon_plan_create"]:
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", q.LIB_PATH], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in declared_symbols():
        assert name in exported, name
        assert hasattr(lib, name)
    assert set(q.exported_symbols()) == set(declared_symbols())   # the binding covers the whole header


def test_status_strings_and_version(lib):
    assert q.qmuon_version().startswith("qmuon")
    for code in range(8):
        s = q.status_string(code)
        assert s and s != "unknown status"
    assert q.status_string(99) == "unknown status"


FAKE = 0x7F0000000000  # a 16-byte-aligned address that is never dereferenced


def _tensor(rows, cols, base=FAKE):
    return q.qmuon_tensor(base, base + 0x100000, base + 0x200000, rows, cols)


def _plan_status(tensors, segments=None, n_groups=0, tile=(1, 1), q8=0, dt=0):
    arr = (q.qmuon_tensor * max(1, len(tensors)))(*tensors)
    segs = None
    if segments:
        segs = (q.qmuon_norm_segment * len(segments))(*[q.qmuon_norm_segment(t, g, s, l) for t, s, l, g in segments])
    out = C.c_void_p()
    return q.lib().qmuon_plan_create(arr, len(tensors), q8, dt, segs, len(segments or []), n_groups,
                                     tile[0], tile[1], C.byref(out))


def test_plan_create_rejects_on_host(lib):
    INV, MIS = q.QMUON_ERR_INVALID_ARGUMENT, q.QMUON_ERR_MISALIGNED_SEGMENT
    assert _plan_status([]) == INV
    assert _plan_status([_tensor(16, 16)], q8=7) == INV                      # bad enum
    assert _plan_status([_tensor(16, 16)], dt=9) == INV
    assert _plan_status([q.qmuon_tensor(FAKE + 8, FAKE, FAKE, 16, 16)]) == INV   # q8 not 16-byte aligned
    assert _plan_status([q.qmuon_tensor(0, FAKE, FAKE, 16, 16)]) == INV          # null pointer
    assert _plan_status([_tensor(-1, 16)]) == INV
    assert _plan_status([_tensor(0, 16), _tensor(16, 0)]) == INV             # no quantization block at all
    # norm segments ("Grouped QKV And Sharding"): 256-element alignment
    t = [_tensor(8, 512)]
    assert _plan_status(t, segments=[(0, 100, 256, 0)], n_groups=1) == MIS
    assert _plan_status(t, segments=[(0, 0, 300, 0)], n_groups=1) == MIS
    assert _plan_status(t, segments=[(0, 0, 512, 0), (0, 256, 512, 1)], n_groups=2) == INV  # overlap
    assert _plan_status(t, segments=[(0, 0, 512, 3)], n_groups=2) == INV                    # group id
    assert _plan_status(t, segments=[(1, 0, 512, 0)], n_groups=1) == INV                    # tensor index
    assert _plan_status(t, segments=[(0, 0, 5000, 0)], n_groups=1) == INV                   # past the end
    # MuonBP tiling: must divide the matrix, column tiles must be 256-aligned
    assert _plan_status([_tensor(8, 512)], tile=(3, 1)) == INV
    assert _plan_status([_tensor(8, 512)], tile=(1, 4)) == MIS
    assert _plan_status([_tensor(8, 512)], tile=(0, 1)) == INV
    assert _plan_status([_tensor(8, 512)], n_groups=5) == INV  # per-tensor groups need n_groups == n


def test_entries_reject_null_plan_and_bad_args(lib):
    L = q.lib()
    INV = q.QMUON_ERR_INVALID_ARGUMENT
    assert L.qmuon_update_multi_normalize_groups(None, 0.9, 0, None, None, FAKE, 1 << 20, None) == INV
    assert L.qmuon_workspace_size(None, 0) == 0
    cf = (C.c_float * 3)(3.4445, -4.775, 2.0315)
    w = (C.c_void_p * 1)(FAKE)
    assert L.qmuon_step(None, 1, 5, 0.9, 0.02, 0.01, w, cf, 5, None, FAKE, 1 << 20, None) == INV
    h = (C.c_void_p * 1)(FAKE)
    assert L.qmuon_step_from_host(None, 1, 5, 0.9, 0.02, 0.01, w, cf, 5, h, None, None, FAKE, 1 << 20, None,
                                  None) == INV
    assert L.qmuon_sync_status(None, None) == INV
    assert L.qmuon_plan_set_nonfinite_counter(None, None) == INV
    assert L.qmuon_sync_status(FAKE + 16, None) == INV   # not 256-byte aligned


def test_noalloc_status_calls_on_host(lib):
    # the injector refuses a non-failure code before any CUDA call; with no
    # usable device both status calls answer QMUON_ERR_CUDA with the detail
    import torch
    L = q.lib()
    assert L.qmuon_noalloc_inject_status(q.QMUON_OK, 0) == q.QMUON_ERR_INVALID_ARGUMENT
    assert L.qmuon_noalloc_inject_status(99, 0) == q.QMUON_ERR_INVALID_ARGUMENT
    assert "not a failure status" in q.qmuon_last_error()
    if torch.cuda.is_available():
        return
    assert L.qmuon_noalloc_sync_status(None) == q.QMUON_ERR_CUDA
    assert q.qmuon_last_error().startswith("qmuon_noalloc_sync_status")
    assert L.qmuon_noalloc_inject_status(q.QMUON_ERR_TIMEOUT, 7) == q.QMUON_ERR_CUDA
    assert q.qmuon_last_error().startswith("qmuon_noalloc_inject_status")


def test_carrier_rejects_on_host(lib):
    L = q.lib()
    t = _tensor(4, 48)   # 48 columns: not a multiple of 32
    r = L.qmuon_update_mxfp8_carrier(C.byref(t), 0, 0, 0.9, FAKE, FAKE, FAKE, FAKE, 1 << 20, None)
    assert r == q.QMUON_ERR_UNSUPPORTED
    t = _tensor(4, 64)
    r = L.qmuon_update_mxfp8_carrier(C.byref(t), 0, 0, 0.9, FAKE + 4, FAKE, FAKE, FAKE, 1 << 20, None)
    assert r == q.QMUON_ERR_INVALID_ARGUMENT   # payload not 16-byte aligned
    r = L.qmuon_update_mxfp8_carrier(C.byref(t), 3, 0, 0.9, FAKE, FAKE, FAKE, FAKE, 1 << 20, None)
    assert r == q.QMUON_ERR_INVALID_ARGUMENT


def test_newton_schulz_rejects_on_host(lib):
    L = q.lib()
    cf = (C.c_float * 3)(3.4445, -4.775, 2.0315)

    def call(probs, iters=5, ws_bytes=1 << 30):
        arr = (q.qmuon_ns_problem * len(probs))(*probs)
        return L.qmuon_newton_schulz_batched(arr, len(probs), iters, cf, FAKE, ws_bytes, None)

    ok = q.ns_problem(FAKE, 64, 64)
    assert call([q.ns_problem(FAKE, 0, 64)]) == q.QMUON_ERR_INVALID_ARGUMENT
    assert call([q.ns_problem(FAKE, 64, 60)]) == q.QMUON_ERR_UNSUPPORTED       # cols % 8
    assert call([q.ns_problem(FAKE, 64, 64, ld=32)]) == q.QMUON_ERR_INVALID_ARGUMENT
    assert call([q.ns_problem(FAKE + 8, 64, 64)]) == q.QMUON_ERR_INVALID_ARGUMENT
    assert call([ok], iters=0) == q.QMUON_ERR_INVALID_ARGUMENT
    assert call([ok], ws_bytes=100) == q.QMUON_ERR_WORKSPACE_TOO_SMALL
    for bad in (q.ns_problem(FAKE, -5, 64), q.ns_problem(FAKE, 64, 60), q.ns_problem(FAKE, 64, 64, ld=32),
                q.ns_problem(FAKE, 64, 48, input_kind=q.QMUON_NS_MXFP8), q.ns_problem(FAKE, 64, 64, input_kind=7)):
        assert q.qmuon_ns_workspace_size([ok, bad]) == 0
    assert q.qmuon_ns_workspace_size([q.ns_problem(None, 64, 64)]) > 0      # pointers not needed
    need = q.qmuon_ns_workspace_size([ok])
    # A, B (64x64 bf16) and two 64x64 scratch copies, plus the problem table
    assert need >= 4 * 64 * 64 * 2


def test_binding_raises_when_library_missing(monkeypatch):
    monkeypatch.setattr(q, "LIB_PATH", "/nonexistent/libqmuon.so")
    monkeypatch.setattr(q, "_lib_handle", None)
    with pytest.raises(RuntimeError, match="not built"):
        q.lib()


_OOM_CHILD = r"""
import ctypes as C, resource, sys
sys.path.insert(0, sys.argv[1])
import memory_reduced_muon_gb300 as q
L = q.lib()
vm_kb = int([l for l in open('/proc/self/status') if l.startswith('VmSize')][0].split()[1])
lim = vm_kb * 1024 + (2 << 30)
resource.setrlimit(resource.RLIMIT_AS, (lim, lim))
FAKE = 0x7F0000000000
# one row of (2^31 - 1) * 256 elements: the most quantization blocks a plan
# accepts, whose host group tables (about 26 GB) cannot fit in 2 GB
t = q.qmuon_tensor(FAKE, FAKE + 0x100000, FAKE + 0x200000, 1, ((1 << 31) - 1) * 256)
arr = (q.qmuon_tensor * 1)(t)
out = C.c_void_p()
st = L.qmuon_plan_create(arr, 1, 0, 0, None, 0, 0, 1, 1, C.byref(out))
print(st, out.value, L.qmuon_last_error().decode())
"""


@pytest.mark.skipif(not os.path.exists("/proc/self/status"), reason="needs Linux /proc")
def test_host_allocation_failure_returns_status(lib):
    # A plan whose host tables cannot be allocated (address space capped in a
    # child process) must come back as QMUON_ERR_OUT_OF_MEMORY, with no plan
    # and no exception escaping the C ABI (that would abort the process).
    import sys
    r = subprocess.run([sys.executable, "-c", _OOM_CHILD, ROOT], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr[-2000:]
    status, handle, detail = r.stdout.strip().split(" ", 2)
    assert int(status) == q.QMUON_ERR_OUT_OF_MEMORY
    assert handle == "None"
    assert "host memory allocation failed" in detail


def test_cuda_failures_carry_detail(lib):
    # with no usable device, the first CUDA call of a valid request fails:
    # the status is QMUON_ERR_CUDA and qmuon_last_error names the entry
    import torch
    if torch.cuda.is_available():
        pytest.skip("needs a machine without a usable GPU")
    L = q.lib()
    assert _plan_status([_tensor(16, 256)]) == q.QMUON_ERR_CUDA
    assert q.qmuon_last_error().startswith("qmuon_plan_create")
    t = _tensor(4, 64)
    r = L.qmuon_update_mxfp8_carrier(C.byref(t), 0, 0, 0.9, FAKE, FAKE, FAKE, FAKE, 1 << 20, None)
    assert r == q.QMUON_ERR_CUDA
    assert q.qmuon_last_error().startswith("qmuon_update_mxfp8_carrier")


_C_CALLER = r"""
/* A plain C99 caller of the library: the header must compile as C, and the
 * entries must link and answer without a GPU. */
#include <stddef.h>
#include <stdio.h>
#include <string.h>
#include "qmuon.h"

int main(void) {
  qmuon_plan* plan = (qmuon_plan*)0x1;
  qmuon_tensor t;
  memset(&t, 0, sizeof(t));
  if (qmuon_plan_create(&t, 0, QMUON_Q8_INT8, QMUON_BF16, NULL, 0, 0, 1, 1, &plan) != QMUON_ERR_INVALID_ARGUMENT)
    return 1;
  if (plan != NULL) return 2;
  if (qmuon_workspace_size(NULL, QMUON_WS_STEP) != 0) return 3;
  if (strcmp(qmuon_status_string(QMUON_OK), "ok") != 0) return 4;
  if (strncmp(qmuon_version(), "qmuon", 5) != 0) return 5;
  if (sizeof(qmuon_tensor) != 40 || sizeof(qmuon_norm_segment) != 24 || sizeof(qmuon_ns_problem) != 64 ||
      sizeof(qmuon_grasp_matrix) != 96)
    return 6;
  /* the audit tallies: no CUDA call, and the failed plan_create above added nothing */
  qmuon_counters c;
  memset(&c, 0xff, sizeof(c));
  if (sizeof(qmuon_counters) != 192 || offsetof(qmuon_counters, grasp_matrices) != 168 ||
      offsetof(qmuon_counters, host_copied_bytes) != 184)
    return 7;
  if (qmuon_get_counters(&c, sizeof(c)) != QMUON_OK || c.update_calls != 0 || c.grasp_matrices != 0) return 8;
  qmuon_reset_counters();
  if (qmuon_get_counters(NULL, sizeof(c)) != QMUON_ERR_INVALID_ARGUMENT) return 9;
  printf("%s\n", qmuon_version());
  return 0;
}
"""


def test_header_compiles_as_c_and_links(lib, tmp_path):
    # the boundary is a C ABI: a C99 program built with gcc against the header
    # and the shared library calls it directly, without Python or torch
    import shutil
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    src = tmp_path / "caller.c"
    src.write_text(_C_CALLER)
    exe = tmp_path / "caller"
    libdir = os.path.dirname(q.LIB_PATH)
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                        str(src), "-o", str(exe), "-L", libdir, "-lqmuon", "-Wl,-rpath," + libdir],
                       capture_output=True, text=True)
    if r.returncode != 0 and "cannot find -lqmuon" in r.stderr:
        r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                            str(src), "-o", str(exe), q.LIB_PATH, "-Wl,-rpath," + libdir],
                           capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert run.returncode == 0, (run.returncode, run.stderr)
    assert run.stdout.startswith("qmuon")
    # the binding's structures have the sizes the C compiler gave them
    assert [C.sizeof(t) for t in (q.qmuon_tensor, q.qmuon_norm_segment, q.qmuon_ns_problem,
                                  q.qmuon_grasp_matrix, q.qmuon_counters)] == [40, 24, 64, 96, 192]


def _header_counter_fields():
    text = open(HEADER).read()
    body = text[text.index("typedef struct qmuon_counters {"):text.index("} qmuon_counters;")]
    return re.findall(r"uint64_t\s+(\w+);", body)


def test_counters_on_host(lib):
    # the binding names the header's fields in the header's order
    assert tuple(_header_counter_fields()) == q.COUNTER_FIELDS
    L = q.lib()
    q.qmuon_reset_counters()
    assert set(q.qmuon_get_counters().values()) == {0}
    # calls rejected on the host add nothing
    t = _tensor(4, 48)
    assert L.qmuon_update_mxfp8_carrier(C.byref(t), 0, 0, 0.9, FAKE, FAKE, FAKE, FAKE, 1 << 20, None) \
        == q.QMUON_ERR_UNSUPPORTED
    assert L.qmuon_update_normalize_noalloc(None, 0, 0, 0.9, None, None, None) == q.QMUON_ERR_INVALID_ARGUMENT
    cf = (C.c_float * 3)(3.4445, -4.775, 2.0315)
    arr = (q.qmuon_ns_problem * 1)(q.ns_problem(FAKE, 64, 60))
    assert L.qmuon_newton_schulz_batched(arr, 1, 5, cf, FAKE, 1 << 30, None) == q.QMUON_ERR_UNSUPPORTED
    assert set(q.qmuon_get_counters().values()) == {0}
    # a shorter struct (an older caller's) receives only its own prefix
    buf = (C.c_uint64 * 3)(7, 7, 7)
    assert L.qmuon_get_counters(C.cast(buf, C.POINTER(q.qmuon_counters)), 16) == q.QMUON_OK
    assert list(buf) == [0, 0, 7]
    assert L.qmuon_get_counters(None, 192) == q.QMUON_ERR_INVALID_ARGUMENT


def test_host_ingest_mode_is_checked_on_host(lib):
    L = q.lib()
    assert L.qmuon_plan_set_host_ingest(None, q.QMUON_INGEST_COPY) == q.QMUON_ERR_INVALID_ARGUMENT


def _declared_arities():
    # QMUON_API <ret> name(<params>);  -> number of parameters ("void" = 0)
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    out = {}
    for m in re.finditer(r"QMUON_API\s+[\w\s\*]+?\b(qmuon_\w+)\s*\(([^)]*)\)\s*;", text):
        params = m.group(2).strip()
        out[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_signatures_match_the_header(lib):
    # every entry the binding sets up takes as many arguments as the header
    # declares (ctypes would otherwise pass garbage or drop arguments)
    arity = _declared_arities()
    assert set(arity) == set(declared_symbols())
    L = q.lib()
    for name in q.exported_symbols():
        fn = getattr(L, name)
        assert fn.argtypes is not None, name
        assert len(fn.argtypes) == arity[name], (name, len(fn.argtypes), arity[name])


def test_product_path_never_touches_the_oracle():
    # the binding and the library sources name nothing of the oracle, and
    # importing and loading the product leaves the oracle package unimported
    pkg = os.path.join(ROOT, "memory_reduced_muon_gb300")
    for dirpath, _, names in os.walk(pkg):
        for n in names:
            if n.endswith((".py", ".cu", ".h", ".cuh", ".cpp")):
                text = open(os.path.join(dirpath, n)).read()
                assert "oracle" not in text, os.path.join(dirpath, n)
    code = ("import sys; sys.path.insert(0, sys.argv[1]); import memory_reduced_muon_gb300 as q; q.lib(); "
            "print(any(m == 'oracle' or m.startswith('oracle.') for m in sys.modules))")
    r = subprocess.run([sys.executable, "-c", code, ROOT], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr[-1000:]
    assert r.stdout.strip() == "False"


def test_oracle_shares_nothing_with_the_product():
    # the oracle's code imports neither the library's binding, ctypes nor
    # torch, and touches no CUDA attribute (its docstrings may name them)
    import ast
    for n in sorted(os.listdir(os.path.join(ROOT, "oracle"))):
        if not n.endswith(".py"):
            continue
        tree = ast.parse(open(os.path.join(ROOT, "oracle", n)).read())
        for node in ast.walk(tree):
            mods = []
            if isinstance(node, ast.Import):
                mods = [a.name for a in node.names]
            elif isinstance(node, ast.ImportFrom) and node.module:
                mods = [node.module]
            for m in mods:
                assert m.split(".")[0] not in ("memory_reduced_muon_gb300", "ctypes", "torch"), (n, m)
            if isinstance(node, ast.Attribute):
                assert node.attr != "cuda", n


def _grasp(rows, cols, base=FAKE, grad=None):
    p = [base + 0x10000 * i for i in range(10)]
    return q.qmuon_grasp_matrix(rows, cols, p[0], p[1], p[2], p[3], p[4], p[5], p[6], p[7], p[8],
                                p[9] if grad is None else grad)


def test_grasp_rejects_on_host(lib):
    L = q.lib()
    INV, UNS = q.QMUON_ERR_INVALID_ARGUMENT, q.QMUON_ERR_UNSUPPORTED

    def call(mats, ws=FAKE, ws_bytes=1 << 40):
        arr = (q.qmuon_grasp_matrix * max(1, len(mats)))(*mats)
        return L.qmuon_grasp_step(arr if mats else None, len(mats), 0.9, ws, ws_bytes, None)

    assert call([]) == INV
    assert call([_grasp(7, 64)]) == INV                  # fewer rows than the rank 8
    assert call([_grasp(64, 96)]) == UNS                 # cols not a multiple of 64
    assert call([_grasp(64, 0)]) == INV
    assert call([_grasp(64, 64, grad=FAKE + 8)]) == INV  # gradient not 16-byte aligned
    bad = _grasp(64, 64)
    bad.r_cmax = None
    assert call([bad]) == INV                            # a missing state array
    assert call([_grasp(64, 64)], ws=FAKE + 16) == INV   # workspace not 256-byte aligned
    need = q.qmuon_grasp_workspace_size([_grasp(64, 64), _grasp(100, 128)])
    assert need > q.qmuon_grasp_workspace_size([_grasp(64, 64)]) > 0
    assert call([_grasp(64, 64), _grasp(100, 128)], ws_bytes=need - 1) == q.QMUON_ERR_WORKSPACE_TOO_SMALL
    assert q.qmuon_grasp_workspace_size([]) == 0
    for rows, cols in ((7, 64), (64, 96), (64, 0), (-1, 64)):
        assert q.qmuon_grasp_workspace_size([_grasp(64, 64), _grasp(rows, cols)]) == 0, (rows, cols)
    assert q.qmuon_grasp_workspace_size([q.qmuon_grasp_matrix(64, 64)]) > 0   # pointers not needed
