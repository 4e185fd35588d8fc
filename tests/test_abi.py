"""The C ABI library on the CPU: it builds, loads, exports every symbol that
include/flp.h declares, and rejects bad arguments before touching a device."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "flp.h")


@pytest.fixture(scope="module")
def lib():
    from entropy_loss_gb300 import build, flp
    build.build()
    return flp.load()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:flp_status|const char\s*\*)\s*(flp_\w+)\s*\(", text, re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("flp_workspace_query", "flp_forward", "flp_backward", "flp_get_error"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    from entropy_loss_gb300 import build
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\bT\s+(flp_\w+)", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, f"declared but not exported: {missing}"
    for n in declared_functions():
        assert hasattr(lib, n)


def test_binding_lists_the_same_exports():
    from entropy_loss_gb300 import flp
    assert sorted(flp.EXPORTS) == declared_functions()


def test_status_strings(lib):
    for code in range(0, 7):
        assert lib.flp_status_string(code)
    assert b"unknown" in lib.flp_status_string(99)


def _fwd(lib, **over):
    buf = ctypes.create_string_buffer(4096 + 16)
    base = (ctypes.addressof(buf) + 15) // 16 * 16
    a = dict(X=base, W=base, y=base, M=4, H=64, V=10, ign=-100, s=1.0, ent=1, lp=base, lse=base,
             en=base, ws=base, wsb=4096, stream=None)
    a.update(over)
    return lib.flp_forward(a["X"], a["W"], a["y"], a["M"], a["H"], a["V"], a["ign"], a["s"], a["ent"],
                           a["lp"], a["lse"], a["en"], a["ws"], a["wsb"], a["stream"])


def test_forward_argument_checks_need_no_device(lib):
    from entropy_loss_gb300 import flp
    assert _fwd(lib, M=-1) == flp.FLP_ERR_INVALID_ARG
    assert _fwd(lib, V=0) == flp.FLP_ERR_INVALID_ARG
    assert _fwd(lib, H=60) == flp.FLP_ERR_UNSUPPORTED
    assert _fwd(lib, X=None) == flp.FLP_ERR_INVALID_ARG
    assert _fwd(lib, W=None) == flp.FLP_ERR_INVALID_ARG
    assert _fwd(lib, y=None) == flp.FLP_ERR_INVALID_ARG
    buf = ctypes.create_string_buffer(64)
    odd = (ctypes.addressof(buf) + 15) // 16 * 16 + 4
    assert _fwd(lib, X=odd) == flp.FLP_ERR_INVALID_ARG
    assert _fwd(lib, en=None) == flp.FLP_ERR_INVALID_ARG          # entropy on but no buffer
    assert _fwd(lib, ent=0) == flp.FLP_ERR_INVALID_ARG            # entropy off but a buffer
    assert _fwd(lib, s=float("nan")) == flp.FLP_ERR_INVALID_ARG
    assert _fwd(lib, M=2**31) == flp.FLP_ERR_UNSUPPORTED


def test_backward_argument_checks_need_no_device(lib):
    from entropy_loss_gb300 import flp
    buf = ctypes.create_string_buffer(4096 + 16)
    b = (ctypes.addressof(buf) + 15) // 16 * 16

    def call(**o):
        a = dict(X=b, W=b, y=b, M=4, H=64, V=10, ent=1, lse=b, en=b, g1=b, g2=b, dX=b, dxt=1, dW=b,
                 dwt=0, acc=0, ws=b, wsb=4096)
        a.update(o)
        return lib.flp_backward(a["X"], a["W"], a["y"], a["M"], a["H"], a["V"], -100, 1.0, a["ent"],
                                a["lse"], a["en"], a["g1"], a["g2"], a["dX"], a["dxt"], a["dW"],
                                a["dwt"], a["acc"], a["ws"], a["wsb"], None)

    assert call(dX=None) == flp.FLP_ERR_INVALID_ARG
    assert call(dW=None) == flp.FLP_ERR_INVALID_ARG
    assert call(dxt=7) == flp.FLP_ERR_INVALID_ARG
    assert call(dwt=7) == flp.FLP_ERR_INVALID_ARG
    assert call(dwt=1, acc=1) == flp.FLP_ERR_UNSUPPORTED  # bf16 dW cannot be accumulated into
    assert call(lse=None) == flp.FLP_ERR_INVALID_ARG
    assert call(en=None) == flp.FLP_ERR_INVALID_ARG
    assert call(H=12) == flp.FLP_ERR_UNSUPPORTED


def test_phase_event_count_checked(lib):
    from entropy_loss_gb300 import flp
    assert lib.flp_set_phase_events(None, 11) == flp.FLP_ERR_INVALID_ARG
    assert lib.flp_set_phase_events(None, -1) == flp.FLP_ERR_INVALID_ARG
    assert lib.flp_set_phase_events(None, 0) == flp.FLP_OK


def test_product_path_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "entropy_loss_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", text, re.M), f
                assert "flp_oracle" not in text and "libflp_oracle" not in text, f


def test_selftest_argument_checks_need_no_device(lib):
    from entropy_loss_gb300 import flp
    buf = ctypes.create_string_buffer(64)
    base = (ctypes.addressof(buf) + 15) // 16 * 16
    assert lib.flp_selftest_wait_timeout(None, 1 << 20, 1, 1000, None) == flp.FLP_ERR_WORKSPACE
    assert lib.flp_selftest_wait_timeout(base, 1024, 1, 1000, None) == flp.FLP_ERR_WORKSPACE
    assert lib.flp_selftest_wait_timeout(base, 1 << 20, 1, 0, None) == flp.FLP_ERR_INVALID_ARG
    assert lib.flp_selftest_wait_timeout(base, 1 << 20, 1, 61 * 10**9, None) == flp.FLP_ERR_INVALID_ARG


def test_dependency_selftest_argument_checks_need_no_device(lib):
    from entropy_loss_gb300 import flp
    buf = ctypes.create_string_buffer(64)
    base = (ctypes.addressof(buf) + 15) // 16 * 16
    assert lib.flp_selftest_dependency_timeout(None, 1 << 20, 1, 1000, None) == flp.FLP_ERR_WORKSPACE
    assert lib.flp_selftest_dependency_timeout(base, 1024, 1, 1000, None) == flp.FLP_ERR_WORKSPACE
    assert lib.flp_selftest_dependency_timeout(base, 1 << 20, 1, 0, None) == flp.FLP_ERR_INVALID_ARG


def test_dz_selftest_argument_checks_need_no_device(lib):
    from entropy_loss_gb300 import flp
    buf = ctypes.create_string_buffer(64)
    base = (ctypes.addressof(buf) + 15) // 16 * 16
    assert lib.flp_selftest_dz_wait_timeout(None, 1 << 20, 1, 1000, None) == flp.FLP_ERR_WORKSPACE
    assert lib.flp_selftest_dz_wait_timeout(base, 1024, 1, 1000, None) == flp.FLP_ERR_WORKSPACE
    assert lib.flp_selftest_dz_wait_timeout(base, 1 << 20, 1, 0, None) == flp.FLP_ERR_INVALID_ARG
    assert lib.flp_selftest_dz_wait_timeout(base, 1 << 20, 1, 61 * 10**9, None) == flp.FLP_ERR_INVALID_ARG


def test_loss_argument_checks_need_no_device(lib):
    from entropy_loss_gb300 import flp
    import ctypes as C
    buf = C.create_string_buffer(64)
    b = (C.addressof(buf) + 15) // 16 * 16
    f = C.c_float
    assert lib.flp_loss(b, b, 4, -100, 7, b, b, None, f(0.2), f(0.2), f(0), b, b, b, None) == flp.FLP_ERR_INVALID_ARG
    assert lib.flp_loss(b, b, -1, -100, 1, None, None, None, f(0.2), f(0.2), f(0), b, b, b, None) == flp.FLP_ERR_INVALID_ARG
    assert lib.flp_loss(b, b, 4, -100, 2, None, b, None, f(0.2), f(0.2), f(0), b, b, b, None) == flp.FLP_ERR_INVALID_ARG
    assert lib.flp_loss(b, b, 4, -100, 2, b, b, None, f(-0.1), f(0.2), f(0), b, b, b, None) == flp.FLP_ERR_INVALID_ARG
    assert lib.flp_loss(b, b, 4, -100, 1, None, None, None, f(0.2), f(0.2), f(0), b, b, None, None) == flp.FLP_ERR_INVALID_ARG


def test_a_caller_of_the_contract_compiles_and_links(tmp_path):
    """A C program written against include/flp.h, calling the six-argument
    flp_workspace_query of the boundary contract and its wave-size variant,
    compiles, links against the library and runs on a machine without a GPU:
    negative sizes are rejected before any device is touched, and a valid
    query reports that no sm_103 device can be queried."""
    from entropy_loss_gb300 import build
    build.build()
    src = tmp_path / "caller.c"
    src.write_text(r'''
#include <stdio.h>
#include "flp.h"
int main(void) {
    size_t f = 0, b = 0;
    flp_status a = flp_workspace_query(-1, 64, 10, 1, &f, &b);
    flp_status c = flp_workspace_query_ex(4, 64, 10, 1, -5, NULL, NULL);
    flp_status d = flp_workspace_query(4, 64, 10, 0, &f, NULL);
    printf("%d %d %d\n", (int)a, (int)c, (int)d);
    return 0;
}
''')
    exe = tmp_path / "caller"
    libdir = os.path.dirname(build.LIB)
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    str(src), "-o", str(exe), f"-L{libdir}", "-l:libflp.so",
                    f"-Wl,-rpath,{libdir}"], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()
    from entropy_loss_gb300 import flp
    assert int(out[0]) == flp.FLP_ERR_INVALID_ARG
    assert int(out[1]) in (flp.FLP_ERR_CUDA, flp.FLP_ERR_UNSUPPORTED, flp.FLP_OK)
    assert int(out[2]) in (flp.FLP_ERR_CUDA, flp.FLP_ERR_UNSUPPORTED, flp.FLP_OK)


def test_policy_loss_argument_checks_need_no_device(lib):
    from entropy_loss_gb300 import flp
    import ctypes as C
    buf = C.create_string_buffer(64)
    b = (C.addressof(buf) + 15) // 16 * 16
    f, dd = C.c_float, C.c_double

    def call(**o):
        a = dict(lp=b, y=b, M=4, off=None, B=0, old=b, adv=b, ref=None, lo=0.2, hi=0.2, beta=0.0,
                 lvl=0, agg=0, norm=0.0, per=b, grad=b, loss=b)
        a.update(o)
        return lib.flp_policy_loss(a["lp"], a["y"], a["M"], -100, a["off"], a["B"], a["old"], a["adv"],
                                   a["ref"], f(a["lo"]), f(a["hi"]), f(a["beta"]), a["lvl"], a["agg"],
                                   dd(a["norm"]), a["per"], a["grad"], a["loss"], None)
    assert call(M=-1) == flp.FLP_ERR_INVALID_ARG
    assert call(lvl=2) == flp.FLP_ERR_INVALID_ARG
    assert call(agg=3) == flp.FLP_ERR_INVALID_ARG
    assert call(old=None) == flp.FLP_ERR_INVALID_ARG
    assert call(adv=None) == flp.FLP_ERR_INVALID_ARG
    assert call(loss=None) == flp.FLP_ERR_INVALID_ARG
    assert call(off=b, B=0) == flp.FLP_ERR_INVALID_ARG
    assert call(lo=1.5) == flp.FLP_ERR_INVALID_ARG
    assert call(norm=float("inf")) == flp.FLP_ERR_INVALID_ARG
