"""Host-side checks of the C ABI (no GPU needed).

The library must load on a machine without a GPU, export every function
include/*.h declares, and reject bad arguments before touching the device.
"""
import ctypes
import glob
import os
import re

import pytest

from quantised_gguf_weight_gb300 import build as qbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    qbuild.build()
    from quantised_gguf_weight_gb300 import qk
    return qk.load()


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s*([a-z_][a-z0-9_]*)\s*\(",
                            text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("qmatvec_q8_0", "qmatvec_q4_k", "qmatvec_swiglu_q8_0", "qmatvec_swiglu_q4_k",
              "qmatvec_experts_q8_0", "qmatvec_experts_q4_k", "qgemm_q4_k", "qgemm_q4_k_acc",
              "qgemm_swiglu_q4_k", "qgemm_q8_0", "qgemm_q8_0_acc", "qgemm_swiglu_q8_0",
              "qgemm_q4_k_workspace_bytes", "qk_status_string", "qk_device_error"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for s in range(10):
        assert lib.qk_status_string(s) and lib.qk_status_string(s) != b"unknown status"
    assert lib.qk_status_string(99) == b"unknown status"


def test_row_bytes(lib):
    assert lib.qk_row_bytes_q8_0(576) == 18 * 34
    assert lib.qk_row_bytes_q8_0(40) == 2 * 34
    assert lib.qk_row_bytes_q4_k(896) == 4 * 144
    assert lib.qk_row_bytes_q4_k(4096) == 16 * 144
    assert lib.qk_row_bytes_q6_k(4096) == 16 * 210
    assert lib.qk_row_bytes_q6_k(300) == 2 * 210
    assert lib.qk_row_bytes_q4_k(0) == 0


FAKE = 0x10000  # never dereferenced: validation fails first


@pytest.mark.parametrize("name", ["qmatvec_q8_0", "qmatvec_q4_k", "qmatvec_q6_k"])
def test_argument_validation_without_gpu(lib, name):
    f = getattr(lib, name)
    ok_args = dict(w=FAKE, off=0, rows=16, K=256, x=FAKE, batch=1, y=FAKE, ldy=0)

    def call(**kw):
        a = dict(ok_args, **kw)
        return f(a["w"], a["off"], a["rows"], a["K"], a["x"], a["batch"], a["y"], a["ldy"], None)

    assert call(w=None) == 1
    assert call(x=None) == 1
    assert call(y=None) == 1
    assert call(rows=0) == 2
    assert call(K=0) == 2
    assert call(K=-5) == 2
    assert call(off=-1) == 2
    assert call(ldy=8) == 2          # ldy < rows
    assert call(batch=0) == 4
    assert call(batch=9) == 4
    assert call(x=FAKE + 2) == 3     # x not 4-byte aligned
    assert call(y=FAKE + 1) == 3
    assert call(w=FAKE + 1) == 3     # odd w
    if name == "qmatvec_q4_k":
        assert call(w=FAKE + 8) == 3     # Q4_K rows need 16-byte alignment


@pytest.mark.parametrize("name", ["qmatvec_swiglu_q8_0", "qmatvec_swiglu_q4_k", "qmatvec_swiglu_q6_k"])
def test_swiglu_argument_validation_without_gpu(lib, name):
    f = getattr(lib, name)
    f.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                  ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
    ok_args = dict(w=FAKE, gate=0, up=16, F=16, K=256, x=FAKE, batch=1, h=FAKE, ldh=0)

    def call(**kw):
        a = dict(ok_args, **kw)
        return f(a["w"], a["gate"], a["up"], a["F"], a["K"], a["x"], a["batch"], a["h"], a["ldh"], None)

    assert call(w=None) == 1
    assert call(h=None) == 1
    assert call(up=-1) == 2
    assert call(gate=-1) == 2
    assert call(F=0) == 2
    assert call(ldh=8) == 2          # ldh < F
    assert call(batch=9) == 4
    assert call(x=FAKE + 2) == 3


@pytest.mark.parametrize("name", ["qmatvec_experts_q8_0", "qmatvec_experts_q4_k", "qmatvec_experts_q6_k"])
def test_experts_argument_validation_without_gpu(lib, name):
    f = getattr(lib, name)
    f.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int,
                  ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
    ok_args = dict(w=FAKE, E=4, rows=16, K=256, x=FAKE, xk=2, ids=FAKE, n=4, y=FAKE, ldy=0)

    def call(**kw):
        a = dict(ok_args, **kw)
        return f(a["w"], a["E"], a["rows"], a["K"], a["x"], a["xk"], a["ids"], a["n"], a["y"], a["ldy"], None)

    assert call(ids=None) == 1
    assert call(w=None) == 1
    assert call(E=0) == 2
    assert call(xk=0) == 2
    assert call(n=0) == 2
    assert call(rows=0) == 2
    assert call(ldy=3) == 2
    assert call(ids=FAKE + 2) == 3
    assert call(x=FAKE + 1) == 3


def test_wait_limit_roundtrip(lib):
    old = lib.qk_set_wait_limit_ns(12345)
    assert lib.qk_set_wait_limit_ns(old) == 12345


def test_product_path_does_not_import_the_oracle():
    """Nothing in the package imports, loads or builds anything under oracle/."""
    pkg = os.path.join(ROOT, "quantised_gguf_weight_gb300")
    pat = re.compile(r"^\s*(from\s+oracle\b|import\s+oracle\b)|qk_oracle|libqk_oracle", re.M)
    for path in glob.glob(os.path.join(pkg, "**", "*.py"), recursive=True) + \
            glob.glob(os.path.join(pkg, "csrc", "*")):
        assert not pat.search(open(path, errors="replace").read()), path


@pytest.mark.parametrize("name", ["qgemm_q4_k", "qgemm_q4_k_acc", "qgemm_q8_0", "qgemm_q8_0_acc"])
def test_gemm_argument_validation_without_gpu(lib, name):
    f = getattr(lib, name)
    f.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64,
                  ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    ok = dict(w=FAKE, off=0, N=128, K=256, x=FAKE, M=4, y=FAKE, ldy=0, ws=FAKE, wsb=1 << 20)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["w"], a["off"], a["N"], a["K"], a["x"], a["M"], a["y"], a["ldy"], a["ws"], a["wsb"], None)

    assert call(w=None) == 1
    assert call(y=None) == 1
    assert call(N=0) == 2
    assert call(M=0) == 2
    assert call(K=-1) == 2
    assert call(ldy=64) == 2
    assert call(w=FAKE + (8 if "q4_k" in name else 1)) == 3   # Q4_K: 16-byte, Q8_0: 2-byte alignment
    assert call(ws=None) == 7
    assert call(ws=FAKE + 16) == 7
    assert call(wsb=100) == 7
    assert lib.qgemm_q4_k_workspace_bytes(512, 14336, 4096) >= 512 * 4096 * 2


# K that is not a whole number of blocks, and one that is, per format
STRICT_K = {"q8_0": (40, 64), "q4_k": (896, 1024), "q6_k": (300, 512)}


@pytest.fixture
def strict(lib):
    old = lib.qk_set_strict_blocks(1)
    yield lib
    lib.qk_set_strict_blocks(old)


def strict_calls(lib):
    """(format, call(K, x)) for every compute entry point.  The tests pass a
    misaligned x to every call, so no call can get past validation to a launch
    whatever the strict-blocks check does; the fake pointers are never
    dereferenced."""
    P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    out = []
    for fmt in ("q8_0", "q4_k", "q6_k"):
        f = getattr(lib, "qmatvec_" + fmt)
        out.append((fmt, lambda K, x, f=f: f(FAKE, 0, 16, K, x, 1, FAKE, 0, None)))
        f = getattr(lib, "qmatvec_swiglu_" + fmt)
        f.argtypes = [P, I64, I64, I64, I64, P, I, P, I64, P]
        out.append((fmt, lambda K, x, f=f: f(FAKE, 0, 16, 16, K, x, 1, FAKE, 0, None)))
        f = getattr(lib, "qmatvec_experts_" + fmt)
        f.argtypes = [P, I64, I64, I64, P, I, P, I64, P, I64, P]
        out.append((fmt, lambda K, x, f=f: f(FAKE, 4, 16, K, x, 1, FAKE, 2, FAKE, 0, None)))
    gemm_types = [P, I64, I64, I64, P, I64, P, I64, P, ctypes.c_size_t, P]
    for fmt, names in (("q4_k", ("qgemm_q4_k", "qgemm_q4_k_acc")), ("q8_0", ("qgemm_q8_0", "qgemm_q8_0_acc"))):
        for n in names:
            f = getattr(lib, n)
            f.argtypes = gemm_types
            out.append((fmt, lambda K, x, f=f: f(FAKE, 0, 128, K, x, 4, FAKE, 0, FAKE, 1 << 20, None)))
        f = getattr(lib, "qgemm_swiglu_" + fmt)
        f.argtypes = [P, I64, I64, I64, I64, P, I64, P, I64, P, ctypes.c_size_t, P]
        out.append((fmt, lambda K, x, f=f: f(FAKE, 0, 128, 128, K, x, 4, FAKE, 0, FAKE, 1 << 20, None)))
    f = lib.qgemm_q4_k_noalloc
    f.argtypes = [P, I64, I64, I64, P, I64, P, I64, P]
    out.append(("q4_k", lambda K, x, f=f: f(FAKE, 0, 128, K, x, 4, FAKE, 0, None)))
    return out


def test_strict_blocks_mode_refuses_partial_blocks(strict):
    calls = strict_calls(strict)
    assert len(calls) == 16
    for fmt, call in calls:
        bad, good = STRICT_K[fmt]
        assert call(bad, FAKE + 2) == 2, fmt        # refused before the pointer checks
        assert call(good, FAKE + 2) == 3, fmt       # a whole number of blocks passes on to them


def test_strict_blocks_mode_off_accepts_partial_blocks(lib):
    old = lib.qk_set_strict_blocks(0)
    try:
        for fmt, call in strict_calls(lib):
            bad, _ = STRICT_K[fmt]
            assert call(bad, FAKE + 2) == 3, fmt    # K passes; the misaligned x is what is refused
    finally:
        lib.qk_set_strict_blocks(old)


def test_strict_blocks_mode_from_environment(lib):
    """QK_STRICT=1 in the environment turns the mode on when the library loads."""
    import subprocess
    import sys
    from quantised_gguf_weight_gb300 import qk
    code = ("import ctypes, sys; lib = ctypes.CDLL(sys.argv[1]); "
            "print(lib.qk_set_strict_blocks(0), lib.qk_set_strict_blocks(0))")
    path = qk.library_path()
    for env_value, first in (("1", "1"), ("0", "0"), (None, "0")):
        env = {k: v for k, v in os.environ.items() if k != "QK_STRICT"}
        if env_value is not None:
            env["QK_STRICT"] = env_value
        out = subprocess.run([sys.executable, "-c", code, path], env=env, capture_output=True, text=True,
                             check=True).stdout.split()
        assert out == [first, "0"], (env_value, out)


def test_binding_refuses_host_tensors():
    """The Python binding hands the library device pointers only: a tensor in
    host memory is refused before the library is called."""
    import torch
    from quantised_gguf_weight_gb300 import qk
    K = 256
    w = torch.zeros(qk._fmt_row_bytes("q4_k", K) * 4, dtype=torch.uint8)
    x = torch.zeros((1, K))
    ids = torch.zeros(2, dtype=torch.int32)
    calls = [
        lambda: qk.qmatvec_q8_0(w, 0, 4, K, x),
        lambda: qk.qmatvec_q4_k(w, 0, 4, K, x),
        lambda: qk.qmatvec_q6_k(w, 0, 4, K, x),
        lambda: qk.qmatvec_swiglu("q4_k", w, 0, 2, 2, K, x),
        lambda: qk.qmatvec_experts("q4_k", w, 2, 2, K, x, 2, ids),
        lambda: qk.qgemm_q4_k(w, 0, 4, K, x),
        lambda: qk.qgemm_q8_0(w, 0, 4, K, x),
        lambda: qk.qgemm_acc("q4_k", w, 0, 4, K, x, torch.zeros((1, 4))),
        lambda: qk.qgemm_swiglu("q4_k", w, 0, 2, 2, K, x),
    ]
    for call in calls:
        with pytest.raises(ValueError, match="CUDA tensor"):
            call()


def test_binding_row_bytes_match_the_library(lib):
    from quantised_gguf_weight_gb300 import qk
    for K in (1, 31, 32, 33, 255, 256, 257, 896, 4096, 14336):
        assert qk._fmt_row_bytes("q8_0", K) == lib.qk_row_bytes_q8_0(K)
        assert qk._fmt_row_bytes("q4_k", K) == lib.qk_row_bytes_q4_k(K)
        assert qk._fmt_row_bytes("q6_k", K) == lib.qk_row_bytes_q6_k(K)


def test_header_compiles_as_c99_and_the_library_answers_from_c(lib, tmp_path):
    """A plain C client (tests/c_abi_check.c) builds against include/qk.h with
    strict C99 warnings as errors, links libqk.so and sees the documented
    statuses; every compute call there fails validation, so nothing launches."""
    import shutil
    import subprocess
    from quantised_gguf_weight_gb300 import qk
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    libdir = os.path.dirname(qk.library_path())
    exe = str(tmp_path / "c_abi_check")
    subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "c_abi_check.c"), "-o", exe, "-L", libdir, "-lqk",
                    "-Wl,-rpath," + libdir], check=True, capture_output=True, text=True)
    env = {k: v for k, v in os.environ.items() if k != "QK_STRICT"}
    r = subprocess.run([exe], env=env, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip().endswith("failures 0")


def test_missing_library_fails_loudly(tmp_path):
    """Without the built CUDA library there is no fallback: loading it raises."""
    import subprocess
    import sys
    code = ("import sys; sys.path.insert(0, sys.argv[1]); "
            "from quantised_gguf_weight_gb300 import qk\n"
            "try:\n"
            "    qk.load(sys.argv[2])\n"
            "except RuntimeError as e:\n"
            "    print('refused:', e)\n"
            "else:\n"
            "    print('loaded')\n")
    r = subprocess.run([sys.executable, "-c", code, ROOT, str(tmp_path / "libqk.so")], capture_output=True,
                       text=True, check=True)
    assert r.stdout.startswith("refused:") and "not built" in r.stdout
