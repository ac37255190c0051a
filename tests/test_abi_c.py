"""The C ABI from C: include/moge.h compiles as strict C99 (and as C++17), a program that takes the
address of every declared entry point links against libmoge.so, and the calls that need no GPU
(version, status text, workspace sizing, argument rejection before any launch) behave as the
header states.  No GPU is needed: nothing here enqueues device work.
"""
import os
import re
import shutil
import subprocess

import pytest

import sparse_router_gemm_global_b300 as moge

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")
HEADER = os.path.join(INCLUDE, "moge.h")


def declared_functions():
    src = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    return sorted(set(re.findall(r"\b(moge_\w+)\s*\(", src)))


PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "moge.h"

typedef void (*any_fn)(void);

int main(void) {
    any_fn fns[] = { %(fns)s };
    moge_config_t c;
    memset(&c, 0, sizeof c);
    c.T = 32; c.d = 64; c.N = 16; c.M = 4; c.k_per_group = 1; c.I = 32;
    c.act_dtype = MOGE_BF16; c.weight_dtype = MOGE_BF16;
    if (moge_abi_version() != MOGE_ABI_VERSION) return 10;
    if (strcmp(moge_status_string(MOGE_OK), "ok") != 0) return 11;
    size_t ws = moge_workspace_bytes(&c);
    if (ws == 0 || ws %% 256 != 0) return 12;
    if (moge_workspace_bytes_shared(&c, 4) <= ws) return 13;
    c.N = 15;  /* N %% M != 0 */
    if (moge_workspace_bytes(&c) != 0) return 14;
    c.N = 16;
    /* null x, weights, output: rejected on the host before any launch */
    if (moge_layer_forward(&c, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 0, NULL)
        != MOGE_ERR_INVALID_ARGUMENT) return 15;
    if (moge_layer_forward_residual(&c, 0, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 0, NULL)
        != MOGE_ERR_INVALID_ARGUMENT) return 16;
    printf("%%d entry points, workspace %%zu bytes\n", (int)(sizeof fns / sizeof fns[0]), ws);
    return 0;
}
"""


@pytest.fixture(scope="module")
def program_source():
    names = declared_functions()
    assert len(names) >= 19
    return PROGRAM % {"fns": ", ".join(f"(any_fn){n}" for n in names)}, len(names)


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_header_is_c99_and_links_every_entry_point(tmp_path, program_source):
    src, n = program_source
    c_file = tmp_path / "abi_check.c"
    c_file.write_text(src)
    exe = tmp_path / "abi_check"
    lib_dir = os.path.dirname(moge.library_path())
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-Wno-pedantic", "-I", INCLUDE, str(c_file), "-o",
                    str(exe), "-L", lib_dir, "-lmoge", f"-Wl,-rpath,{lib_dir}"], check=True,
                   capture_output=True, text=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, (out.returncode, out.stdout, out.stderr)
    assert out.stdout.startswith(f"{n} entry points")


@pytest.mark.skipif(shutil.which("g++") is None, reason="needs g++")
def test_header_compiles_as_cpp(tmp_path, program_source):
    src, _ = program_source
    cpp = tmp_path / "abi_check.cpp"
    cpp.write_text(src.replace("typedef void (*any_fn)(void);", "typedef void (*any_fn)();"))
    subprocess.run(["g++", "-std=c++17", "-fsyntax-only", "-Wall", "-Werror", "-I", INCLUDE, str(cpp)], check=True,
                   capture_output=True, text=True)


def declared_parameter_counts():
    """{function: number of parameters} from the prototypes in include/moge.h."""
    src = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    out = {}
    for m in re.finditer(r"\b(moge_\w+)\s*\(([^;{]*?)\)\s*;", src, flags=re.S):
        params = m.group(2).strip()
        out[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_declares_every_prototype_with_its_parameter_count():
    """ctypes trusts argtypes: a binding that passes more or fewer arguments than the C prototype
    would hand the library garbage.  Every function the binding declares matches the header."""
    from sparse_router_gemm_global_b300 import binding
    lib = binding.load()
    want = declared_parameter_counts()
    assert len(want) >= 19
    checked = 0
    for name, n in want.items():
        fn = getattr(lib, name)
        assert fn.argtypes is not None, f"{name}: no argtypes declared"
        assert len(fn.argtypes) == n, (name, len(fn.argtypes), n)
        checked += 1
    assert checked == len(want)
