"""The C ABI without a GPU: the library builds and loads, exports every
symbol the header declares, and its host-side checks answer without any
compute call."""
import ctypes
import os
import re

import pytest
import torch

import moe_finalize_residual_rmsnorm_gb300 as mfr

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")


@pytest.fixture(scope="module")
def lib():
    mfr.build()
    return mfr.load_library()


def declared_functions():
    names = set()
    for fn in os.listdir(HEADER_DIR):
        if fn.endswith(".h"):
            text = open(os.path.join(HEADER_DIR, fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(moe_finalize_\w+)\s*\(", text))
    return names


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("moe_finalize_rmsnorm_plan", "moe_finalize_rmsnorm_run", "moe_finalize_rmsnorm_destroy",
              "moe_finalize_rmsnorm_supports", "moe_finalize_rmsnorm_get_status",
              "moe_finalize_rmsnorm_strerror"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    # and the binding knows a signature for each
    assert declared_functions() <= set(mfr.SIGNATURES)


def test_supports_truth_table(lib):
    s = lib.moe_finalize_rmsnorm_supports
    assert s(4096, 8) == 1 and s(8192, 8) == 1 and s(8, 1) == 1 and s(16384, 16) == 1
    assert s(0, 8) == 0 and s(4, 8) == 0 and s(4100, 8) == 0 and s(16392, 8) == 0
    assert s(4096, 0) == 0 and s(4096, 17) == 0 and s(-8, 8) == 0


def test_default_options(lib):
    o = mfr.Options(7, 7, 7, 7, 7)
    lib.moe_finalize_rmsnorm_default_options(ctypes.byref(o))
    assert (o.enable_pdl, o.force_variant, o.cluster_size, o.debug_checks, o.sentinel_skip) == (1, 0, 0, 0, 0)


def test_strerror_covers_every_code(lib):
    for code in [0, *mfr.ERROR_CODES]:
        msg = lib.moe_finalize_rmsnorm_strerror(code).decode()
        assert msg and msg != "unknown error code"
    assert lib.moe_finalize_rmsnorm_strerror(99).decode() == "unknown error code"


def _plan(lib, T, H, k, R, opt=None):
    h = ctypes.c_void_p(123)
    rc = lib.moe_finalize_rmsnorm_plan(ctypes.byref(h), T, H, k, R, ctypes.byref(opt) if opt else None)
    return rc, h


def test_plan_rejects_bad_shapes_before_touching_a_device(lib):
    for T, H, k, R in [(4, 4100, 8, 32), (4, 4096, 0, 32), (4, 4096, 17, 64), (4, 20000, 8, 32)]:
        rc, h = _plan(lib, T, H, k, R)
        assert rc == 2 and not h.value
        assert "unsupported shape" in lib.moe_finalize_rmsnorm_last_error().decode()
    rc, h = _plan(lib, -1, 4096, 8, 0)
    assert rc == 1 and not h.value
    assert lib.moe_finalize_rmsnorm_plan(None, 1, 4096, 8, 8, None) == 1


def test_plan_rejects_bad_options(lib):
    rc, _ = _plan(lib, 4, 4096, 8, 32, mfr.Options(1, 9, 0, 0, 0))
    assert rc == 1
    rc, _ = _plan(lib, 4, 4096, 8, 32, mfr.Options(1, 0, 3, 0, 0))
    assert rc == 1


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU answer")
def test_plan_without_a_gpu_reports_bad_device(lib):
    rc, h = _plan(lib, 16, 4096, 8, 128)
    assert rc == 4 and not h.value
    assert lib.moe_finalize_rmsnorm_last_error().decode()


def test_null_handles_are_rejected(lib):
    assert lib.moe_finalize_rmsnorm_run(None, None, None, None, None, None, None, 1e-6, None, None) == 1
    st = ctypes.c_int(0)
    assert lib.moe_finalize_rmsnorm_get_status(None, None, ctypes.byref(st)) == 1
    info = mfr.PlanInfo()
    assert lib.moe_finalize_rmsnorm_plan_info(None, ctypes.byref(info)) == 1
    lib.moe_finalize_rmsnorm_destroy(None)


def test_binding_fails_loudly_without_the_library(tmp_path, monkeypatch):
    monkeypatch.setattr(mfr, "_lib", None)
    monkeypatch.setattr(mfr, "LIBRARY", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        mfr.load_library()
    with pytest.raises(ImportError):
        mfr.Plan(1, 4096, 8)


def test_header_compiles_as_c_and_links_from_a_c_program(lib, tmp_path):
    """The boundary is plain C: a C99 program that includes only the header
    compiles with gcc, links against the library and gets the host-side
    answers (no GPU here: a plan reports MFR_ERR_BAD_DEVICE)."""
    import importlib
    import subprocess
    libpath = importlib.import_module("moe_finalize_residual_rmsnorm_gb300.build").LIBRARY
    src = tmp_path / "use_abi.c"
    src.write_text(r"""
#include <stdio.h>
#include <string.h>
#include "moe_finalize_rmsnorm.h"
int main(void) {
    mfr_options o;
    mfr_plan_t plan = NULL;
    moe_finalize_rmsnorm_default_options(&o);
    if (moe_finalize_rmsnorm_supports(4096, 8) != 1 || moe_finalize_rmsnorm_supports(4100, 8) != 0) return 1;
    if (strcmp(moe_finalize_rmsnorm_strerror(MFR_OK), "ok") != 0) return 2;
    int rc = moe_finalize_rmsnorm_plan(&plan, 8, 4096, 8, 64, &o);
    if (rc != MFR_OK && plan != NULL) return 3;
    printf("%d\n", rc);
    if (plan) moe_finalize_rmsnorm_destroy(plan);
    return 0;
}
""")
    exe = tmp_path / "use_abi"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", f"-I{HEADER_DIR}", str(src), "-o", str(exe),
                    libpath, f"-Wl,-rpath,{os.path.dirname(libpath)}"], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, out
    rc = int(out.stdout.strip())
    expected = mfr.MFR_OK if torch.cuda.is_available() else 4    # MFR_ERR_BAD_DEVICE
    assert rc == expected
