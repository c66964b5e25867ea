"""The C ABI without a GPU: the library loads, exports every declared symbol, and
rejects bad arguments before touching the device."""
import ctypes
import os
import re
import subprocess

import pytest

from dspark_draft_sampling_gb300 import api

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "dspark.h")

INVALID, UNSUPPORTED = api.DSPARK_ERR_INVALID, api.DSPARK_ERR_UNSUPPORTED
FAKE = ctypes.c_void_p(0x10000)        # never dereferenced: every case fails validation first
FAKE_ODD = ctypes.c_void_p(0x10002)    # not 16-byte aligned
NULL = None


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dspark_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_three_operations():
    names = declared_functions()
    for n in ("dspark_markov_draft", "dspark_conf_probe", "dspark_ws_matvec"):
        assert n in names


def test_exports_every_declared_symbol(dspark_lib):
    names = declared_functions()
    assert set(names) == set(api.SIGNATURES), "binding and header disagree"
    out = subprocess.run(["nm", "-D", "--defined-only", api.lib_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (dspark_\w+)", out))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        assert getattr(dspark_lib, n) is not None


def test_version(dspark_lib):
    assert dspark_lib.dspark_version().decode().startswith("libdspark")


def test_workspace_bytes(dspark_lib):
    a = dspark_lib.dspark_markov_workspace_bytes(1, 15, 248320, 256)
    b = dspark_lib.dspark_markov_workspace_bytes(8, 15, 248320, 256)
    assert a == b and a % 256 == 0 and a >= 256 + 15 * 8 * 8
    assert dspark_lib.dspark_markov_workspace_bytes(1, 0, 10, 64) == 256
    # the matvecs' workspaces hold only the status word
    assert dspark_lib.dspark_ws_matvec_workspace_bytes(7, 4096, 4096) == 256


def _markov(lib, *, base=FAKE, w1=FAKE, w2=FAKE, d2t=NULL, prev=FAKE, B=1, k=4, V=4096, R=64,
            out=FAKE, ws=FAKE, wsb=1 << 20):
    return lib.dspark_markov_draft(base, w1, w2, d2t, prev, B, k, V, R, out, NULL, NULL, ws, wsb,
                                   NULL)


def test_markov_validation(dspark_lib):
    lib = dspark_lib
    assert _markov(lib, R=100) == UNSUPPORTED
    assert _markov(lib, R=512) == UNSUPPORTED
    assert _markov(lib, B=9) == UNSUPPORTED
    assert _markov(lib, B=-1) == INVALID
    assert _markov(lib, V=0) == INVALID
    assert _markov(lib, base=NULL) == INVALID
    assert _markov(lib, w2=NULL) == INVALID
    assert _markov(lib, prev=NULL) == INVALID
    assert _markov(lib, out=NULL) == INVALID
    assert _markov(lib, ws=NULL) == INVALID
    assert _markov(lib, w2=FAKE_ODD) == INVALID
    assert _markov(lib, w1=FAKE_ODD) == INVALID
    assert _markov(lib, ws=FAKE_ODD) == INVALID
    assert _markov(lib, wsb=16) == INVALID
    assert "workspace" in lib.dspark_last_error().decode()
    # nothing to do: accepted without launching anything
    assert _markov(lib, k=0) == 0
    assert _markov(lib, B=0) == 0
    assert lib.dspark_last_error().decode() == ""


def test_markov_kernel_choice(dspark_lib):
    lib = dspark_lib
    k_ = lib.dspark_markov_draft_kernel
    # an unknown kernel is refused before anything else is looked at
    assert k_(FAKE, FAKE, FAKE, NULL, FAKE, 1, 4, 4096, 64, FAKE, NULL, NULL, FAKE, 1 << 20, 7,
              NULL) == INVALID
    assert k_(FAKE, FAKE, FAKE, NULL, FAKE, 1, 4, 4096, 64, FAKE, NULL, NULL, FAKE, 1 << 20, -1,
              NULL) == INVALID
    assert k_(FAKE, FAKE, FAKE, NULL, FAKE, 1, 4, 4096, 100, FAKE, NULL, NULL, FAKE, 1 << 20, 2,
              NULL) == UNSUPPORTED
    grid, cluster = 1, 2
    kf = lib.dspark_markov_kernel_for
    # small vocabularies with one or two requests go to the single-cluster kernel
    assert {kf(B, 4, 4096, 64) for B in (1, 2)} == {cluster}
    assert kf(8, 4, 4096, 64) == grid
    assert kf(1, 3, 1024, 256) == cluster
    # the 27B and reduced-vocab lanes, and a vocabulary that is not a multiple of 4, do not
    assert kf(8, 15, 248320, 256) == grid
    assert kf(1, 9, 32000, 256) == grid
    assert kf(1, 4, 4098, 64) == grid
    assert kf(1, 4, 4096, 100) == grid


def test_markov_debug_and_plan_validation(dspark_lib):
    lib = dspark_lib
    assert lib.dspark_markov_draft_debug(FAKE, FAKE, FAKE, NULL, FAKE, 1, 4, 64, 64, FAKE, FAKE,
                                         4096, 1, 0, NULL) == INVALID
    assert lib.dspark_markov_plan_create(FAKE, FAKE, FAKE, NULL, FAKE, 1, 4, 64, 64, FAKE, FAKE,
                                         4096, None) == INVALID
    assert lib.dspark_markov_plan_launch(NULL, NULL) == INVALID
    lib.dspark_markov_plan_destroy(NULL)
    assert lib.dspark_markov_status(NULL, NULL) == INVALID


def test_draft_plan_validation(dspark_lib):
    lib = dspark_lib
    f = lib.dspark_draft_plan_create
    h = api.ctypes.c_void_p()
    args = lambda B, k: (FAKE, FAKE, 256, FAKE, FAKE, NULL, FAKE, B, k, 1000, 64, FAKE, FAKE, FAKE,
                         1 << 20, FAKE, 1 << 20)
    assert f(*args(1, 4), None) == INVALID
    assert f(*args(2, 9), api.ctypes.byref(h)) == UNSUPPORTED
    assert f(*args(0, 4), api.ctypes.byref(h)) == INVALID
    assert lib.dspark_draft_plan_launch(NULL, NULL) == INVALID
    lib.dspark_draft_plan_destroy(NULL)


def test_gated_plan_validation(dspark_lib):
    lib = dspark_lib
    f = lib.dspark_gated_draft_plan_create
    h = api.ctypes.c_void_p()
    args = lambda K, B, k: (FAKE, FAKE, K, 0.0, 0.5, FAKE, FAKE, FAKE, FAKE, FAKE, NULL, FAKE, B, k,
                            1000, 64, FAKE, FAKE, 1 << 20)
    assert f(*args(7424, 1, 4), None) == INVALID
    assert f(*args(7425, 1, 4), api.ctypes.byref(h)) == INVALID
    assert f(*args(7424, 0, 4), api.ctypes.byref(h)) == INVALID
    assert lib.dspark_gated_draft_plan_launch(NULL, NULL) == INVALID
    lib.dspark_gated_draft_plan_destroy(NULL)


def test_probe_split_validation(dspark_lib):
    f = dspark_lib.dspark_conf_probe_split
    assert f(FAKE, FAKE, 7168, 7168, FAKE, 250, 256, 0.0, 0.5, 1, NULL, FAKE, NULL) == INVALID
    assert f(FAKE, FAKE, 7168, 7000, FAKE, 256, 256, 0.0, 0.5, 1, NULL, FAKE, NULL) == INVALID
    assert f(FAKE, FAKE, 7168, 7168, NULL, 256, 256, 0.0, 0.5, 1, NULL, FAKE, NULL) == INVALID
    assert f(FAKE, FAKE, 7168, 7168, FAKE, 256, 256, 0.0, 0.5, 0, NULL, FAKE, NULL) == 0


def test_probe_validation(dspark_lib):
    lib = dspark_lib
    f = lib.dspark_conf_probe
    assert f(FAKE, FAKE, 0.0, 0.5, 33, 1, NULL, FAKE, NULL) == INVALID
    assert f(FAKE, FAKE, 0.0, 0.5, 0, 1, NULL, FAKE, NULL) == INVALID
    assert f(FAKE, FAKE, 0.0, 1.0, 64, 1, NULL, FAKE, NULL) == INVALID
    assert f(FAKE, FAKE, 0.0, 0.0, 64, 1, NULL, FAKE, NULL) == INVALID
    assert f(FAKE, FAKE, 0.0, 0.5, 64, -1, NULL, FAKE, NULL) == INVALID
    assert f(FAKE, FAKE, 0.0, 0.5, 64, 1, NULL, NULL, NULL) == INVALID
    assert f(FAKE, FAKE_ODD, 0.0, 0.5, 64, 1, NULL, FAKE, NULL) == INVALID
    assert f(FAKE, FAKE, 0.0, 0.5, 64, 0, NULL, FAKE, NULL) == 0


def test_ws_validation(dspark_lib):
    lib = dspark_lib
    f = lib.dspark_ws_matvec
    B = 1 << 20
    assert f(FAKE, FAKE, FAKE, 0, 17, 64, 64, FAKE, B, NULL) == UNSUPPORTED
    assert f(FAKE, FAKE, FAKE, 0, 7, 64, 12, FAKE, B, NULL) == INVALID
    assert f(FAKE, FAKE, FAKE, 0, 7, 64, 0, FAKE, B, NULL) == INVALID
    assert f(FAKE, FAKE, FAKE, 0, -1, 64, 64, FAKE, B, NULL) == INVALID
    assert f(NULL, FAKE, FAKE, 0, 7, 64, 64, FAKE, B, NULL) == INVALID
    assert f(FAKE, FAKE, FAKE, 0, 7, 64, 64, NULL, B, NULL) == INVALID
    assert f(FAKE_ODD, FAKE, FAKE, 0, 7, 64, 64, FAKE, B, NULL) == INVALID
    assert f(FAKE, FAKE, ctypes.c_void_p(0x10001), 0, 7, 64, 64, FAKE, B, NULL) == INVALID
    assert f(FAKE, FAKE, FAKE, 0, 7, 64, 64, FAKE_ODD, B, NULL) == INVALID
    assert f(FAKE, FAKE, FAKE, 1, 0, 64, 64, FAKE, B, NULL) == 0
    assert f(FAKE, FAKE, FAKE, 1, 7, 0, 64, FAKE, B, NULL) == 0


def test_python_binding_rejects_cpu_tensors(dspark_lib):
    import torch

    with pytest.raises(ValueError):
        api.ws_matvec(torch.zeros(4, 8, dtype=torch.float16), torch.zeros(1, 8, dtype=torch.float16))


def test_ws_q8_validation(dspark_lib):
    lib = dspark_lib
    f = lib.dspark_ws_matvec_q8
    B = 1 << 20

    def g(q=FAKE, d=FAKE, x=FAKE, y=FAKE, yf=0, M=7, N=64, K=256, ws=FAKE, wsb=B):
        return f(q, d, x, y, yf, M, N, K, ws, wsb, NULL)

    assert g(M=17) == UNSUPPORTED
    assert g(K=288) == UNSUPPORTED   # K % 256 != 0
    assert g(K=0) == UNSUPPORTED
    assert g(M=-1) == INVALID
    assert g(N=-1) == INVALID
    assert g(q=NULL) == INVALID
    assert g(d=NULL) == INVALID
    assert g(y=NULL) == INVALID
    assert g(ws=NULL) == INVALID
    assert g(q=FAKE_ODD) == INVALID
    assert g(d=FAKE_ODD) == INVALID
    assert g(x=FAKE_ODD) == INVALID
    assert g(y=ctypes.c_void_p(0x10002), yf=1) == INVALID
    assert g(ws=FAKE_ODD) == INVALID
    assert g(M=0) == 0
    assert g(N=0) == 0
    assert lib.dspark_ws_matvec_q8_workspace_bytes(7, 0, 256) == 256  # the status word
    r = lib.dspark_q8_0_repack
    assert r(FAKE, FAKE, FAKE, 4, 48, NULL) == INVALID
    assert r(FAKE, FAKE, FAKE, -1, 64, NULL) == INVALID
    assert r(NULL, FAKE, FAKE, 4, 64, NULL) == INVALID
    assert r(FAKE, FAKE_ODD, FAKE, 4, 64, NULL) == INVALID
    assert r(FAKE, FAKE, ctypes.c_void_p(0x10001), 4, 64, NULL) == INVALID
    assert r(NULL, NULL, NULL, 0, 64, NULL) == 0


def test_python_q8_binding_rejects_cpu_tensors(dspark_lib):
    import torch

    with pytest.raises(ValueError):
        api.ws_matvec_q8(torch.zeros(4, 256, dtype=torch.int8), torch.zeros(4, 8, dtype=torch.int16),
                         torch.zeros(1, 256, dtype=torch.float16), workspace=torch.zeros(16))
    with pytest.raises(ValueError):
        api.q8_0_repack(torch.zeros(4 * 2 * 34, dtype=torch.uint8), 4, 64)


def test_host_form_validation(dspark_lib):
    """Argument errors of the host-buffer forms are caught before any copy is enqueued."""
    lib = dspark_lib
    m = lib.dspark_markov_draft_host
    nb = lib.dspark_markov_draft_host_scratch_bytes(1, 4, 4096, 64)
    assert nb >= 4 * 4096 * 4 and nb % 256 == 0
    assert m(FAKE, FAKE, FAKE, NULL, FAKE, 1, 4, 4096, 100, FAKE, FAKE, nb, NULL, NULL) == UNSUPPORTED
    assert m(FAKE, FAKE, FAKE, NULL, FAKE, 9, 4, 4096, 64, FAKE, FAKE, nb, NULL, NULL) == UNSUPPORTED
    assert m(NULL, FAKE, FAKE, NULL, FAKE, 1, 4, 4096, 64, FAKE, FAKE, nb, NULL, NULL) == INVALID
    assert m(FAKE, FAKE, FAKE, NULL, NULL, 1, 4, 4096, 64, FAKE, FAKE, nb, NULL, NULL) == INVALID
    assert m(FAKE, FAKE, FAKE, NULL, FAKE, 1, 4, 4096, 64, FAKE, FAKE_ODD, nb, NULL, NULL) == INVALID
    assert m(FAKE, FAKE, FAKE, NULL, FAKE, 1, 4, 4096, 64, FAKE, FAKE, nb - 256, NULL, NULL) == INVALID
    assert "scratch" in lib.dspark_last_error().decode()
    assert m(FAKE, FAKE, FAKE, NULL, FAKE, 1, 0, 4096, 64, FAKE, FAKE, nb, NULL, NULL) == 0
    p = lib.dspark_conf_probe_host
    pb = lib.dspark_conf_probe_host_scratch_bytes(7424, 3)
    assert pb >= 3 * 7424 * 4
    assert p(FAKE, FAKE, 0.0, 0.5, 48, 3, NULL, FAKE, FAKE, pb, NULL, NULL) == INVALID
    assert p(FAKE, FAKE, 0.0, 1.5, 7424, 3, NULL, FAKE, FAKE, pb, NULL, NULL) == INVALID
    assert p(FAKE, NULL, 0.0, 0.5, 7424, 3, NULL, FAKE, FAKE, pb, NULL, NULL) == INVALID
    assert p(FAKE, FAKE, 0.0, 0.5, 7424, 3, NULL, NULL, FAKE, pb, NULL, NULL) == INVALID
    assert p(FAKE, FAKE, 0.0, 0.5, 7424, 3, NULL, FAKE, FAKE, pb - 1, NULL, NULL) == INVALID
    assert p(FAKE, FAKE, 0.0, 0.5, 7424, 0, NULL, FAKE, FAKE, pb, NULL, NULL) == 0
    w = lib.dspark_ws_matvec_host
    assert w(FAKE, FAKE, FAKE, 0, 17, 64, 64, FAKE, 1 << 20, NULL, NULL) == UNSUPPORTED
    assert w(FAKE, FAKE, FAKE, 0, 7, 64, 12, FAKE, 1 << 20, NULL, NULL) == INVALID
    assert w(FAKE, NULL, FAKE, 0, 7, 64, 64, FAKE, 1 << 20, NULL, NULL) == INVALID
    assert w(FAKE, FAKE, FAKE, 0, 7, 64, 64, FAKE_ODD, 1 << 20, NULL, NULL) == INVALID
    assert w(FAKE, FAKE, FAKE, 0, 0, 64, 64, FAKE, 1 << 20, NULL, NULL) == 0


def test_ws_status_and_debug_validation(dspark_lib):
    lib = dspark_lib
    assert lib.dspark_ws_matvec_status(NULL, NULL) == INVALID
    assert lib.dspark_ws_matvec_debug(FAKE, FAKE, FAKE, 0, 7, 64, 64, FAKE, 1 << 20, 0, NULL) == INVALID
    assert lib.dspark_ws_matvec_debug(NULL, FAKE, FAKE, 0, 7, 64, 64, FAKE, 1 << 20, 100, NULL) == INVALID
    assert lib.dspark_ws_matvec_q8_debug(FAKE, FAKE, FAKE, FAKE, 0, 7, 64, 256, FAKE, 1 << 20, 0, NULL) == INVALID
    assert lib.dspark_ws_matvec_q8_debug(FAKE, FAKE, FAKE, FAKE, 0, 17, 64, 256, FAKE, 1 << 20, 100, NULL) == UNSUPPORTED


def test_ws_grouped_validation(dspark_lib):
    lib = dspark_lib
    arr = (api.WsProblem * 9)()
    for i in range(9):
        arr[i] = api.WsProblem(FAKE.value, FAKE.value, FAKE.value, 0, 7, 64, 64)
    g = lib.dspark_ws_matvec_grouped
    p = ctypes.cast(arr, ctypes.c_void_p)
    assert g(p, 9, FAKE, 1 << 20, NULL) == UNSUPPORTED
    assert g(NULL, 2, FAKE, 1 << 20, NULL) == INVALID
    assert g(p, 0, NULL, 0, NULL) == 0
    arr[1] = api.WsProblem(FAKE.value, FAKE.value, FAKE.value, 0, 17, 64, 64)
    assert g(p, 2, FAKE, 1 << 20, NULL) == UNSUPPORTED
    arr[1] = api.WsProblem(FAKE.value, None, FAKE.value, 0, 7, 64, 64)
    assert g(p, 2, FAKE, 1 << 20, NULL) == INVALID
    arr[0] = api.WsProblem(FAKE.value, FAKE.value, FAKE.value, 0, 0, 64, 64)
    arr[1] = api.WsProblem(FAKE.value, FAKE.value, FAKE.value, 0, 7, 0, 64)
    assert g(p, 2, NULL, 0, NULL) == 0  # every problem empty: nothing to enqueue
    arr[0] = api.WsProblem(FAKE.value, FAKE.value, FAKE.value, 0, 7, 64, 64)
    assert g(p, 1, NULL, 1 << 20, NULL) == INVALID


def test_ws_q8_grouped_validation(dspark_lib):
    lib = dspark_lib
    P = api.WsQ8Problem
    arr = (P * 9)()
    for i in range(9):
        arr[i] = P(FAKE.value, FAKE.value, FAKE.value, FAKE.value, 0, 7, 64, 256)
    g = lib.dspark_ws_matvec_q8_grouped
    p = ctypes.cast(arr, ctypes.c_void_p)
    assert g(p, 9, FAKE, 1 << 20, NULL) == UNSUPPORTED
    assert g(NULL, 2, FAKE, 1 << 20, NULL) == INVALID
    assert g(p, 0, NULL, 0, NULL) == 0
    arr[1] = P(FAKE.value, FAKE.value, FAKE.value, FAKE.value, 0, 17, 64, 256)
    assert g(p, 2, FAKE, 1 << 20, NULL) == UNSUPPORTED
    arr[1] = P(FAKE.value, FAKE.value, FAKE.value, FAKE.value, 0, 7, 64, 288)
    assert g(p, 2, FAKE, 1 << 20, NULL) == UNSUPPORTED
    arr[1] = P(FAKE.value, None, FAKE.value, FAKE.value, 0, 7, 64, 256)
    assert g(p, 2, FAKE, 1 << 20, NULL) == INVALID
    arr[1] = P(FAKE.value, FAKE_ODD.value, FAKE.value, FAKE.value, 0, 7, 64, 256)
    assert g(p, 2, FAKE, 1 << 20, NULL) == INVALID
    arr[0] = P(FAKE.value, FAKE.value, FAKE.value, FAKE.value, 0, 0, 64, 256)
    arr[1] = P(FAKE.value, FAKE.value, FAKE.value, FAKE.value, 0, 7, 0, 256)
    assert g(p, 2, NULL, 0, NULL) == 0  # every problem empty: nothing to enqueue
    arr[0] = P(FAKE.value, FAKE.value, FAKE.value, FAKE.value, 0, 7, 64, 256)
    assert g(p, 1, NULL, 1 << 20, NULL) == INVALID
    assert g(p, 1, FAKE, 16, NULL) == INVALID
    # status word, one flag and one partial row block per SM (0 without a device)
    n = lib.dspark_ws_matvec_q8_grouped_workspace_bytes(p, 2)
    assert n == 0 or n >= 256 + 256 + 8192
    # the fault-injection hook: a wait limit, a CTA number and two non-empty problems
    d = lib.dspark_ws_matvec_q8_grouped_debug
    arr[1] = P(FAKE.value, FAKE.value, FAKE.value, FAKE.value, 0, 7, 64, 256)
    assert d(p, 2, FAKE, 1 << 20, 1, 0, NULL) == INVALID
    assert d(p, 2, FAKE, 1 << 20, -1, 100, NULL) == INVALID
    assert d(p, 1, FAKE, 1 << 20, 1, 100, NULL) == INVALID
    arr[1] = P(FAKE.value, FAKE.value, FAKE.value, FAKE.value, 0, 0, 64, 256)
    assert d(p, 2, FAKE, 1 << 20, 1, 100, NULL) == INVALID


def test_ws_grouped_host_validation(dspark_lib):
    lib = dspark_lib
    arr = (api.WsProblem * 2)()
    arr[0] = api.WsProblem(FAKE.value, FAKE.value, FAKE.value, 0, 7, 64, 64)
    arr[1] = api.WsProblem(FAKE.value, FAKE.value, FAKE.value, 0, 17, 64, 64)
    g = lib.dspark_ws_matvec_grouped_host
    p = ctypes.cast(arr, ctypes.c_void_p)
    assert g(p, 9, FAKE, 1 << 20, NULL, NULL) == UNSUPPORTED
    assert g(NULL, 1, FAKE, 1 << 20, NULL, NULL) == INVALID
    assert g(p, 2, FAKE, 1 << 20, NULL, NULL) == UNSUPPORTED
    assert g(p, 1, NULL, 1 << 20, NULL, NULL) == INVALID
    assert g(p, 1, FAKE_ODD, 1 << 20, NULL, NULL) == INVALID
    assert g(p, 0, NULL, 0, NULL, NULL) == 0


def test_bench_library_exports_its_header():
    """libdspark_bench.so (measurement kernels used by bench.py) exports what its header
    declares."""
    from dspark_draft_sampling_gb300 import build

    build.build()
    hdr = os.path.join(os.path.dirname(HEADER), "dspark_bench.h")
    text = re.sub(r"/\*.*?\*/", "", open(hdr).read(), flags=re.S)
    names = sorted(set(re.findall(r"\b(dspark_bench_[a-z0-9_]+)\s*\(", text)))
    assert names == ["dspark_bench_empty", "dspark_bench_empty_smem", "dspark_bench_read"]
    out = subprocess.run(["nm", "-D", "--defined-only", build.bench_lib_file()], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (dspark_\w+)", out))
    assert set(names) <= exported
    lib = ctypes.CDLL(build.bench_lib_file())
    # argument checks reject before launching anything (cudaErrorInvalidValue = 1)
    lib.dspark_bench_read.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p,
                                      ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    assert lib.dspark_bench_read(FAKE, 24, 1, FAKE, 1, 32, NULL) == 1
    assert lib.dspark_bench_read(FAKE_ODD, 32, 1, FAKE, 1, 32, NULL) == 1
    assert lib.dspark_bench_read(FAKE, 32, 0, FAKE, 1, 32, NULL) == 1
