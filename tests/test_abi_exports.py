"""The C ABI library loads and exports every entry point include/fi.h declares
(no compute calls: this runs without a GPU)."""
import os
import re
import subprocess

import pytest

import paged_kv_attention_13_gb300 as fi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            text = open(os.path.join(ROOT, "include", f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(fi_[a-z0-9_]+)\s*\(", text))
    return names


def test_header_declares_the_four_named_entry_points():
    d = _declared()
    for n in ("fi_plan", "fi_batch_prefill_paged", "fi_batch_decode_paged", "fi_merge_state"):
        assert n in d


def test_library_exports_every_declared_symbol():
    from paged_kv_attention_13_gb300 import build
    build.build()
    lib = fi.load()
    declared = _declared()
    for name in declared:
        assert hasattr(lib, name), name
    assert declared <= set(fi.EXPORTED) | declared
    out = subprocess.run(["nm", "-D", "--defined-only", fi.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (fi_[a-z0-9_]+)$", out, flags=re.M))
    assert declared <= exported, declared - exported
    assert set(fi.EXPORTED) == declared


def test_status_strings():
    lib = fi.load()
    assert lib.fi_status_str(0) == b"FI_OK"
    assert lib.fi_status_str(4) == b"FI_ERR_GQA_INDIVISIBLE"


def test_plain_c_caller(tmp_path):
    """The header compiles as C99 (no CUDA headers) and a C program can plan
    and read refusals through libfi.so without a GPU (tests/c_abi_host.c)."""
    import shutil
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    libdir = os.path.dirname(fi._lib.LIB_PATH)
    exe = str(tmp_path / "c_abi_host")
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                        "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c_abi_host.c"),
                        "-o", exe, "-L", libdir, "-lfi", "-Wl,-rpath," + libdir],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and "c abi ok" in r.stdout, r.stdout + r.stderr
