"""The C ABI library builds, loads and exports every symbol include/hc_gr.h declares.

CPU only: no call here reaches the GPU (the argument checks used below
return before any CUDA call).
"""
import ctypes
import os
import re

import pytest

from hyper_connection_gated_gb300 import _native


@pytest.fixture(scope="module")
def lib(root):
    if not os.path.exists(_native.LIB_PATH):
        from hyper_connection_gated_gb300 import build
        build.build()
    return _native.load()


def declared(root):
    with open(os.path.join(root, "include", "hc_gr.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:int|const char\*)\s+(hc_gr_\w+)\s*\(", text, re.M)))


def test_header_declares_the_boundary(root):
    names = declared(root)
    assert set(_native.EXPORTS) == set(names), names


def test_library_exports_every_declared_symbol(lib, root):
    for name in declared(root):
        assert hasattr(lib, name), name


def test_exports_are_c_symbols(root, lib):
    # extern "C": names are unmangled in the dynamic symbol table
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", _native.LIB_PATH],
                         capture_output=True, text=True).stdout
    for name in declared(root):
        assert re.search(rf"\bT {name}$", out, re.M), name


def test_strerror_and_null_handles(lib):
    assert lib.hc_gr_strerror(0) == b"ok"
    assert b"overlap" in lib.hc_gr_strerror(_native.ERR_ALIAS)
    assert lib.hc_gr_strerror(99) == b"unknown status"
    assert lib.hc_gr_destroy(None) == _native.OK
    assert lib.hc_gr_check(None, None) == _native.ERR_INVALID_ARG
    assert lib.hc_gr_forward_ex(None, None, None) == _native.ERR_INVALID_ARG
    assert lib.hc_gr_create(None, 0, 1, 4, 2560, 320) == _native.ERR_INVALID_ARG
    h = ctypes.c_void_p()
    assert lib.hc_gr_create(ctypes.byref(h), 0, 0, 4, 2560, 320) == _native.ERR_INVALID_ARG
    assert lib.hc_gr_create(ctypes.byref(h), 0, 8, 4, 2561, 320) == _native.ERR_UNSUPPORTED
    assert h.value is None
    # the size limits are checked before any CUDA call
    assert lib.hc_gr_create(ctypes.byref(h), 0, _native.MAX_TOKENS + 1, 4, 2560, 320) == \
        _native.ERR_UNSUPPORTED
    assert lib.hc_gr_create(ctypes.byref(h), 0, 8, 2, (1 << 29) + 8, 320) == _native.ERR_UNSUPPORTED
    assert h.value is None


def test_args_struct_matches_header_layout(root):
    # Field order and types of hc_gr_args in the header and in the ctypes mirror.
    with open(os.path.join(root, "include", "hc_gr.h")) as f:
        text = f.read()
    body = re.search(r"typedef struct hc_gr_args \{(.*?)\} hc_gr_args;", text, re.S).group(1)
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    fields = []
    for decl in body.split(";"):
        decl = decl.strip()
        if not decl:
            continue
        names = [n.strip().lstrip("*") for n in re.sub(r"^(const\s+)?\w+\s*\**", "", decl).split(",")]
        fields += names
    assert fields == [f for f, _ in _native.Args._fields_]


def test_args_struct_offsets_match_c(root, tmp_path):
    # Compile a C program against the header and compare every field offset
    # and the struct size with the ctypes mirror.
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    names = [f for f, _ in _native.Args._fields_]
    src = tmp_path / "off.c"
    src.write_text(
        "#include <stdio.h>\n#include <stddef.h>\n#include \"hc_gr.h\"\n"
        "int main(void){printf(\"%zu\\n\", sizeof(hc_gr_args));\n"
        + "".join(f'printf("%zu\\n", offsetof(hc_gr_args, {n}));\n' for n in names)
        + "return 0;}\n")
    exe = tmp_path / "off"
    subprocess.run([cc, "-I", os.path.join(root, "include"), str(src), "-o", str(exe)], check=True)
    vals = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True,
                                           check=True).stdout.split()]
    assert vals[0] == ctypes.sizeof(_native.Args)
    assert vals[1:] == [getattr(_native.Args, n).offset for n in names]


C_CONSUMER = r"""
#include <stdio.h>
#include <string.h>
#include "hc_gr.h"

/* A plain C caller: every rejection below happens in the argument checks,
   before any CUDA call, so this runs without a GPU. */
int main(void) {
  int fails = 0;
  hc_gr_handle h = NULL;
  hc_gr_args a;
  memset(&a, 0, sizeof(a));
#define EXPECT(call, want) do { int st_ = (call); if (st_ != (want)) { \
    printf("%s -> %d (want %d)\n", #call, st_, (want)); ++fails; } } while (0)
  EXPECT(hc_gr_create(NULL, 0, 8, 4, 2560, 320), HC_GR_ERR_INVALID_ARG);
  EXPECT(hc_gr_create(&h, 0, 0, 4, 2560, 320), HC_GR_ERR_INVALID_ARG);
  EXPECT(hc_gr_create(&h, 0, HC_GR_MAX_TOKENS + 1, 4, 2560, 320), HC_GR_ERR_UNSUPPORTED);
  EXPECT(hc_gr_forward_noalloc(0, 4, 2560, 320, 1e-6f, NULL, NULL, NULL, NULL, NULL, NULL, NULL,
                               NULL, NULL, NULL, NULL, NULL, NULL), HC_GR_ERR_INVALID_ARG);
  EXPECT(hc_gr_forward_ex(NULL, &a, NULL), HC_GR_ERR_INVALID_ARG);
  EXPECT(hc_gr_forward(NULL, 4, 4, 2560, 320, 1e-6f, NULL, NULL, NULL, NULL, NULL, NULL, NULL,
                       NULL, NULL, NULL, NULL, NULL, NULL), HC_GR_ERR_INVALID_ARG);
  EXPECT(hc_gr_combine(NULL, 4, 4, 2560, NULL, NULL, NULL, 0, NULL, NULL), HC_GR_ERR_INVALID_ARG);
  EXPECT(hc_gr_mix(NULL, 4, 4, 2560, 320, 1e-6f, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL,
                   NULL, NULL), HC_GR_ERR_INVALID_ARG);
  EXPECT(hc_gr_check(NULL, NULL), HC_GR_ERR_INVALID_ARG);
  EXPECT(hc_gr_destroy(NULL), HC_GR_OK);
  if (strcmp(hc_gr_strerror(HC_GR_OK), "ok") != 0) { printf("strerror\n"); ++fails; }
  printf("%s\n", fails ? "FAIL" : "PASS");
  return fails != 0;
}
"""


def test_plain_c_caller_links_and_gets_rejections(root, lib, tmp_path):
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "caller.c"
    src.write_text(C_CONSUMER)
    exe = tmp_path / "caller"
    libdir = os.path.dirname(_native.LIB_PATH)
    subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(root, "include"), str(src),
                    "-L", libdir, "-lhc_gr", "-Wl,-rpath," + libdir, "-o", str(exe)], check=True)
    res = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert res.returncode == 0 and res.stdout.strip().endswith("PASS"), res.stdout + res.stderr
