"""The C-ABI library builds for sm_103a, loads, and exports every entry point
that include/ibp.h declares.  Only calls that return before touching the GPU
(argument errors, strings) are made here."""

import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ibp.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ibp_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from host_transfer_gb300 import build, ibp

    build.build()
    return ibp.load()


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("ibp_preprocess", "ibp_plan_create", "ibp_compress", "ibp_gather_decompress",
              "ibp_decompress_contig", "ibp_get_status"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from host_transfer_gb300 import ibp

    out = subprocess.run(["nm", "-D", "--defined-only", ibp.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (ibp_\w+)", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    for n in declared_functions():
        assert hasattr(lib, n)


def test_library_is_built_for_sm_103a_only():
    """Every translation unit is compiled with the one sm_103a target."""
    from host_transfer_gb300 import build

    import inspect

    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
    src = inspect.getsource(build.build)
    assert src.count("*ARCH") == 2  # every object and the device link


def test_version_and_strings(lib):
    hdr = open(os.path.join(ROOT, "include", "ibp.h")).read()
    assert lib.ibp_version() == int(re.search(r"#define IBP_VERSION (\d+)", hdr).group(1))
    for code in range(7):
        s = lib.ibp_strerror(code).decode()
        assert s.startswith("IBP_")
    assert lib.ibp_strerror(99).decode().startswith("IBP_?")


def test_argument_errors_without_gpu(lib):
    vp = ctypes.c_void_p
    null = vp(0)
    EINVAL = 1
    # W = 0 and W > IBP_MAX_W
    assert lib.ibp_preprocess(null, 1, 0, 0.5, null, null, null) == EINVAL
    assert lib.ibp_preprocess(null, 1, 8193, 0.5, null, null, null) == EINVAL
    # T outside (0, 1], no rows
    assert lib.ibp_preprocess(null, 4, 4, 0.0, null, null, null) == EINVAL
    assert lib.ibp_preprocess(null, 4, 4, 1.5, null, null, null) == EINVAL
    assert lib.ibp_preprocess(null, 0, 4, 0.5, null, null, null) == EINVAL
    # no plan
    assert lib.ibp_compress(null, null, null, 1, null, null, null) == EINVAL
    assert lib.ibp_gather_decompress(null, null, 1, null, null, 1, null, null) == EINVAL
    assert lib.ibp_decompress_contig(null, null, 1, null, 0, 1, null, null) == EINVAL
    assert lib.ibp_get_status(null, null) == EINVAL
    assert lib.ibp_plan_get_info(null, None) == EINVAL
    assert lib.ibp_plan_create(null, null, 4, 0, ctypes.POINTER(ctypes.c_void_p)()) == EINVAL
    assert lib.ibp_plan_destroy(null) == 0
    assert lib.ibp_gather_raw(null, 1, 0, null, 1, null, null) == EINVAL


def test_product_path_has_no_oracle_dependency():
    """The package never imports the oracle, and the library never links it."""
    pkg = os.path.join(ROOT, "host_transfer_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".cpp", ".h")):
                text = open(os.path.join(dirpath, f), encoding="utf-8").read()
                for pat in (r"\bfrom\s+oracle\b", r"\bimport\s+oracle\b", r"ibp_ref", r"oracle_c",
                            r"libibp_oracle", r"ibp_oracle"):
                    assert not re.search(pat, text), (f, pat)


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    from host_transfer_gb300 import ibp

    monkeypatch.setattr(ibp, "_lib", None)
    monkeypatch.setattr(ibp, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        ibp.load()
