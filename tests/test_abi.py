"""CPU tests of the C ABI: the library loads, exports every function that
include/iha.h declares, and rejects bad arguments on the host before any
launch (no GPU is touched: every call here fails validation)."""
import ctypes as C
import os
import re

import pytest

import transformer_attention_iha_gb300 as T

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    T.build()
    return T.lib()


def declared_functions():
    names = []
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(L, n), f"{n} declared in include/ but not exported"
    assert set(T.SYMBOLS) <= set(names)


def test_status_strings(L):
    for s in range(5):
        assert L.iha_status_string(s)
    assert L.iha_status_string(99) == b"unknown status"


FAKE = C.c_void_p(0x10000)       # never dereferenced: every call below fails validation
MISALIGNED = C.c_void_p(0x10008)


def _err(L):
    return L.iha_last_error().decode()


def test_premix_validation(L):
    assert L.iha_premix_fwd(None, FAKE, FAKE, 1, 8, 4, 2, 32, T.BF16, 0, 1e4, None) == 1
    assert L.iha_premix_fwd(FAKE, FAKE, FAKE, 0, 8, 4, 2, 32, T.BF16, 0, 1e4, None) == 1
    assert L.iha_premix_fwd(FAKE, FAKE, FAKE, 1, 8, 4, 2, 32, 7, 0, 1e4, None) == 1
    assert L.iha_premix_fwd(FAKE, FAKE, FAKE, 1, 8, 33, 1, 32, T.BF16, 0, 1e4, None) == 2
    assert L.iha_premix_fwd(FAKE, FAKE, FAKE, 1, 8, 20, 7, 32, T.BF16, 0, 1e4, None) == 2
    assert L.iha_premix_fwd(FAKE, FAKE, FAKE, 1, 8, 4, 2, 12, T.BF16, 0, 1e4, None) == 2
    assert L.iha_premix_fwd(FAKE, FAKE, FAKE, 1, 8, 4, 2, 96, T.BF16, 1, 1e4, None) == 2
    assert "RoPE" in _err(L)
    assert L.iha_premix_fwd(FAKE, FAKE, FAKE, 1, 8, 4, 2, 64, T.BF16, 1, -1.0, None) == 1
    assert L.iha_premix_fwd(MISALIGNED, FAKE, FAKE, 1, 8, 4, 2, 32, T.BF16, 0, 1e4, None) == 3
    assert L.iha_premix_bwd_dx(FAKE, None, FAKE, 1, 8, 4, 2, 32, T.BF16, 0, 1e4, None) == 1
    assert L.iha_premix_bwd_dw(FAKE, FAKE, MISALIGNED, 1, 8, 4, 2, 32, T.BF16, 0, 1e4, None) == 3
    # output overlapping an input
    assert L.iha_premix_fwd(FAKE, FAKE, FAKE, 1, 8, 4, 2, 32, T.BF16, 0, 1e4, None) == 1
    assert "overlap" in _err(L)


def _s(b_outer, b_inner, seq, head):
    return T.Strides(b_outer, b_inner, seq, head)


def test_attention_validation(L):
    s = _s(8 * 64 * 2, 8 * 64 * 2, 64 * 2, 64)
    ok = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE)

    def call(q=FAKE, o=FAKE, Bo=1, Bi=1, Hh=2, Nq=8, Nk=8, d=64, sq=s, mask=0, window=0,
             dt=T.BF16):
        return L.mha_fwd(q, FAKE, FAKE, o, None, Bo, Bi, Hh, Nq, Nk, d, sq, s, s, s, 0.0,
                         mask, window, dt, None)

    assert call(q=None) == 1
    assert call(Nq=0) == 1
    assert call(mask=5) == 1
    assert call(mask=2, window=0) == 1
    assert call(mask=1, Nk=9) == 2
    assert call(d=256) == 2
    assert call(d=12) == 2
    assert call(q=MISALIGNED) == 3
    assert call(sq=_s(8 * 64 * 2, 8 * 64 * 2, 68 * 2, 68)) == 3
    assert call(Bo=300, Bi=300) == 2


def test_mask_unit_validation(L):
    assert L.mu_gather(FAKE, FAKE, FAKE, 1, 10, 10, 3, 3, 1, 8, 2, None) == 1   # 10 % 3
    assert L.mu_gather(FAKE, FAKE, FAKE, 1, 8, 8, 4, 4, 5, 8, 2, None) == 1     # 5 > 4 units
    assert L.mu_scatter(None, FAKE, FAKE, 1, 8, 8, 4, 4, 1, 8, 2, None) == 1
    assert L.mu_scatter(FAKE, FAKE, FAKE, 1, 8, 8, 4, 4, 1, 8, 2, None) == 1    # aliasing


def test_python_binding_refuses_to_run_without_library(monkeypatch, tmp_path):
    """The product path fails loudly when the extension is missing."""
    import importlib
    mod = importlib.import_module("transformer_attention_iha_gb300")
    monkeypatch.setattr(mod, "_lib", None)
    monkeypatch.setattr(mod._build, "LIB", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError):
        mod.lib()


def test_premix_qkv_backward_validation(L):
    """iha_premix_bwd_qkv checks all fifteen buffers on the host."""
    def call(dyk=FAKE, H=4, P=2, d=32, dt=T.BF16, dwv=FAKE, rope=0):
        return L.iha_premix_bwd_qkv(FAKE, dyk, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                    FAKE, FAKE, FAKE, FAKE, FAKE, dwv, 1, 8, H, P, d, dt, rope,
                                    1e4, None)
    assert call(dyk=None) == 1
    assert call(H=33, P=1) == 2
    assert call(H=20, P=7) == 2
    assert call(dt=7) == 1
    assert call(d=96, rope=1) == 2                # RoPE needs d a power of two
    assert call(dwv=MISALIGNED) == 3
    assert call() == 1                            # every buffer at one address
    assert "overlap" in _err(L)


def test_qpool_attention_validation(L):
    """mha_fwd_qpool rejects what the pooled mask-unit kernel cannot run."""
    s = _s(64 * 96 * 2, 64 * 96 * 2, 96, 96)

    def call(q=FAKE, T_=64, d=96, qs=4, dt=T.BF16, lse=None, sq=s):
        return L.mha_fwd_qpool(q, FAKE, FAKE, FAKE, lse, 1, 1, 1, T_, d, qs, sq, s, s, s, 0.0,
                               dt, None)
    assert call(q=None) == 1
    assert call(qs=0) == 1
    assert call(qs=3) == 1                        # 3 does not divide 64
    assert "q_stride" in _err(L)
    assert call(dt=T.F32) == 2
    assert call(T_=128, qs=4) == 2                # more than 64 tokens per unit
    assert call(d=12, qs=4) == 2
    assert call(q=MISALIGNED) == 3
    assert call(lse=C.c_void_p(0x10002)) == 3
    assert call(sq=_s(64 * 96 * 2, 64 * 96 * 2, 100, 96)) == 3   # stride not 8-aligned


def _declarations():
    """{name: (return type, [parameter types])} of every function in include/."""
    out = {}
    for f in os.listdir(os.path.join(ROOT, "include")):
        if not f.endswith(".h"):
            continue
        src = open(os.path.join(ROOT, "include", f)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for ret, name, params in re.findall(
                r"^\s*((?:const\s+)?\w+\s*\*?)\s*(\w+)\s*\(([^)]*)\)\s*;", src, flags=re.M):
            types = []
            for prm in params.split(","):
                prm = " ".join(prm.split())
                if prm in ("", "void"):
                    continue
                types.append(re.sub(r"\s*\w+$", "", prm).replace(" *", "*"))
            out[name] = (" ".join(ret.split()).replace(" *", "*"), types)
    return out


_CTYPE = {"int": C.c_int, "float": C.c_float, "size_t": C.c_size_t,
          "iha_dtype": C.c_int, "iha_mask": C.c_int, "iha_status": C.c_int,
          "const char*": C.c_char_p, "iha_strides": T.Strides}


def _expected(ctype: str):
    return C.c_void_p if ctype.endswith("*") and ctype != "const char*" else _CTYPE[ctype]


def test_binding_signatures_match_the_header(L):
    """Every ctypes argtypes / restype the binding sets agrees, parameter by
    parameter, with the C declaration: a pointer is a c_void_p, an enum or int
    a c_int, a float a c_float, size_t a c_size_t, iha_strides the struct."""
    decl = _declarations()
    assert set(T.SYMBOLS) <= set(decl)
    checked = 0
    for name, (ret, params) in decl.items():
        fn = getattr(L, name)
        assert fn.argtypes is not None, f"{name}: argtypes not set"
        assert len(fn.argtypes) == len(params), (name, params, fn.argtypes)
        for i, (got, ctype) in enumerate(zip(fn.argtypes, params)):
            assert got is _expected(ctype), f"{name} parameter {i}: {ctype} bound as {got}"
        assert fn.restype is _expected(ret), f"{name}: returns {ret}, bound as {fn.restype}"
        checked += 1
    assert checked == len(decl) >= 19


def test_strides_struct_matches_the_header():
    src = open(os.path.join(ROOT, "include", "iha.h")).read()
    body = re.search(r"typedef struct \{(.*?)\} iha_strides;", src, flags=re.S).group(1)
    fields = re.findall(r"int64_t\s+(\w+);", body)
    assert [(n, t) for n, t in T.Strides._fields_] == [(f, C.c_int64) for f in fields]


@pytest.mark.parametrize("compiler,std", [("gcc", "-std=c99"), ("g++", "-std=c++11")])
def test_header_is_plain_c_and_cpp(compiler, std, tmp_path):
    import shutil
    import subprocess
    if shutil.which(compiler) is None:
        pytest.skip(f"{compiler} not found")
    src = tmp_path / ("t.c" if compiler == "gcc" else "t.cpp")
    src.write_text('#include "iha.h"\nint main(void) { return IHA_OK; }\n')
    r = subprocess.run([compiler, std, "-Wall", "-Werror", "-pedantic", "-fsyntax-only",
                        "-I", os.path.join(ROOT, "include"), str(src)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
