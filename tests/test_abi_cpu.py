"""CPU checks of the C ABI: the library loads, exports every function that
include/moe_dispatch.h declares, and rejects invalid arguments on the host
before any CUDA call (so these run without a GPU)."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "moe_dispatch.h")


@pytest.fixture(scope="module")
def lib():
    from expert_dispatch_planning_gb300 import _lib
    from expert_dispatch_planning_gb300 import build as b
    if not os.path.exists(_lib.LIB_PATH):
        b.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", text)


def test_header_declares_the_four_steps():
    names = declared_functions()
    for n in ("moe_route_topk", "moe_plan", "moe_permute", "moe_combine"):
        assert n in names
    assert len(names) == len(set(names))


def test_library_exports_every_declared_symbol(lib):
    from expert_dispatch_planning_gb300 import _lib
    names = declared_functions()
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(n for n, _, _ in _lib.SIGNATURES) == sorted(names)


def test_library_hides_internal_symbols(lib):
    # only moe_* entry points are visible
    out = os.popen("nm -D --defined-only %s" % lib._name).read().split("\n")
    exported = [ln.split()[-1] for ln in out if " T " in ln]
    assert exported and all(s.startswith("moe_") for s in exported), exported


def test_status_strings(lib):
    assert lib.moe_status_string(0) == b"ok"
    assert lib.moe_status_string(5) == b"device wait timed out"
    assert lib.moe_status_string(99) == b"unknown status"


def test_sizes(lib):
    assert lib.moe_plan_capacity_rows(4, 4, 2, 2) == 12
    assert lib.moe_plan_capacity_rows(65536, 256, 8, 128) == 65536 * 8 + 256 * 127
    assert lib.moe_plan_capacity_rows(0, 4, 2, 2) == 4      # an empty batch: E*(a-1) rows
    assert lib.moe_plan_capacity_rows(-1, 4, 2, 2) == -1
    assert lib.moe_plan_workspace_size(0, 8, 2, 2) > 0
    assert lib.moe_plan_launch_count(0, 8, 2, 2) == 1        # the empty-plan kernel
    assert lib.moe_plan_launch_count(-1, 8, 2, 2) == -1
    ws = lib.moe_plan_workspace_size(4096, 256, 8, 8)
    assert ws > 0 and ws % 16 == 0
    assert lib.moe_plan_workspace_size(4096, 256, 8, 7) == 0      # E % R
    assert lib.moe_plan_workspace_size(4096, 256, 8, 256) == 0    # R > 128
    assert lib.moe_plan_workspace_size(1 << 28, 8, 8, 2) == 0     # N*K >= 2^30


P = ctypes.c_void_p
FAKE = P(0x10000)  # never dereferenced: validation fails first


def test_route_rejects_bad_arguments(lib):
    f = lib.moe_route_topk
    ok = dict(logits=FAKE, bias=None, N=4, E=8, K=2, scoring=0, renorm=1, ng=1, tg=1, sc=1.0,
              idx=FAKE, w=FAKE, stream=None)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["logits"], a["bias"], a["N"], a["E"], a["K"], a["scoring"], a["renorm"], a["ng"],
                 a["tg"], a["sc"], a["idx"], a["w"], a["stream"])
    assert call(logits=None) == 1
    assert call(N=-1) == 1
    assert call(N=0, E=2048) == 1                     # an empty batch is still validated
    # an empty batch is valid, launches nothing (so it runs without a GPU),
    # and its zero-sized arrays may be NULL
    assert call(N=0) == 0
    assert call(N=0, logits=None, idx=None, w=None) == 0
    assert call(K=9) == 1
    assert call(K=33, E=64) == 1
    assert call(E=2048) == 1
    assert call(scoring=2) == 1
    assert call(ng=3, scoring=1) == 1                 # E % n_group
    assert call(ng=2, tg=1, scoring=0) == 2           # groups need sigmoid
    assert call(ng=4, tg=1, K=3, scoring=1) == 1      # K > kept experts
    assert call(bias=FAKE, scoring=0) == 2            # bias needs sigmoid
    assert call(logits=P(0x10004)) == 1               # rows must be 16-byte aligned


def _plan_struct(ptr=FAKE):
    from expert_dispatch_planning_gb300._lib import MoePlanOut
    return MoePlanOut(*([ptr.value] * 14))


def test_plan_rejects_bad_arguments(lib):
    out = _plan_struct()
    f = lib.moe_plan

    def call(N=4, E=8, K=2, R=2, a=2, ws_bytes=1 << 20, topk=FAKE, ws=FAKE, o=ctypes.byref(out)):
        return f(topk, N, E, K, R, a, ws, ws_bytes, o, None)
    assert call(R=3) == 1
    assert call(a=0) == 1
    assert call(K=0) == 1
    assert call(topk=None) == 1
    assert call(o=None) == 1
    assert call(ws=P(0x10008)) == 1
    assert call(ws_bytes=16) == 3                      # workspace too small
    bad = _plan_struct()
    bad.dst = None
    assert call(o=ctypes.byref(bad)) == 1
    assert call(N=-1) == 1
    # an empty batch: still validated (its kernel needs a GPU, so only the
    # rejections run here)
    assert call(N=0, o=None) == 1
    assert call(N=0, R=3) == 1
    no_cu = _plan_struct()
    no_cu.cu_seqlens = None
    assert call(N=0, o=ctypes.byref(no_cu)) == 1
    no_slots = _plan_struct()
    no_slots.src_of_slot = None                        # capacity E*(a-1) = 8 rows
    assert call(N=0, o=ctypes.byref(no_slots)) == 1


def test_rows_reject_bad_arguments(lib):
    out = _plan_struct()
    assert lib.moe_permute(FAKE, 4, 12, 2, 8, 2, ctypes.byref(out), FAKE, 0, None) == 1     # H % 8
    assert lib.moe_permute(P(0x10008), 4, 16, 2, 8, 2, ctypes.byref(out), FAKE, 0, None) == 1
    assert lib.moe_permute(FAKE, 4, 65536, 2, 8, 2, ctypes.byref(out), FAKE, 0, None) == 2  # row > 96 KB
    assert lib.moe_permute(FAKE, 4, 16, 2, 8, 2, ctypes.byref(out), FAKE, 2, None) == 1     # unknown flag
    assert lib.moe_combine(FAKE, FAKE, 4, 2, 12, 8, 2, ctypes.byref(out), FAKE, None) == 1
    assert lib.moe_combine(FAKE, FAKE, 4, 9, 16, 8, 2, ctypes.byref(out), FAKE, None) == 1  # K > E
    assert lib.moe_combine(FAKE, FAKE, 4, 2, 16, 8, 2, None, FAKE, None) == 1
    assert lib.moe_permute(FAKE, -1, 16, 2, 8, 2, ctypes.byref(out), FAKE, 0, None) == 1
    assert lib.moe_combine(FAKE, FAKE, -1, 2, 16, 8, 2, ctypes.byref(out), FAKE, None) == 1
    # an empty batch moves no rows: valid, nothing launched, N-sized arrays may be NULL
    empty = _plan_struct()
    empty.dst = None
    assert lib.moe_permute(None, 0, 16, 2, 8, 2, ctypes.byref(empty), FAKE, 0, None) == 0
    assert lib.moe_permute(None, 0, 16, 2, 8, 1, ctypes.byref(empty), None, 0, None) == 0   # no capacity rows
    assert lib.moe_permute(None, 4, 16, 2, 8, 2, ctypes.byref(out), FAKE, 0, None) == 1     # x needed
    assert lib.moe_permute(None, 0, 12, 2, 8, 2, ctypes.byref(empty), FAKE, 0, None) == 1    # H % 8
    assert lib.moe_combine(FAKE, None, 0, 2, 16, 8, 2, ctypes.byref(empty), None, None) == 0
    assert lib.moe_combine(FAKE, None, 0, 9, 16, 8, 2, ctypes.byref(empty), None, None) == 1  # K > E


def test_debug_hook_validates(lib):
    assert lib.moe_debug_set_plan_fault(-2, 0) == 1
    assert lib.moe_debug_set_plan_fault(-1, 0) == 0


def test_rank_layout_workspace_and_validation(lib):
    n = lib.moe_rank_layout_workspace_size(65536, 64)
    assert n > 0 and n % 4 == 0
    assert lib.moe_rank_layout_workspace_size(1, 1) > 0
    assert lib.moe_rank_layout_workspace_size(0, 4) > 0        # an empty batch
    assert lib.moe_rank_layout_workspace_size(-1, 4) == 0
    assert lib.moe_rank_layout_workspace_size(0, 129) == 0
    assert lib.moe_rank_layout_workspace_size(16, 129) == 0
    out = _plan_struct()
    f = lib.moe_rank_layout

    def call(N=64, R=4, C=3, ws=P(0x10000), ws_bytes=1 << 20, cpm=FAKE, trs=FAKE):
        return f(ctypes.byref(out), N, R, C, ws, ws_bytes, cpm, trs, None)
    assert call(C=0) == 1
    assert call(R=129) == 1
    assert call(ws=None) == 1
    assert call(ws=P(0x10010)) == 1                   # 256-byte alignment
    assert call(ws_bytes=4) == 3                      # too small
    assert call(trs=None) == 1
    assert call(N=-1) == 1
    assert call(N=0, C=0) == 1                        # an empty batch is still validated
    assert call(N=0, R=129) == 1
    assert call(N=0, cpm=None) == 1


def _header_prototypes():
    """name -> list of parameter declarations, parsed from the header."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    protos = {}
    for m in re.finditer(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(([^)]*)\)\s*;", text, flags=re.S):
        params = [p.strip() for p in m.group(2).split(",") if p.strip()]
        if params == ["void"]:
            params = []
        protos[m.group(1)] = params
    return protos


def test_binding_signatures_match_the_header():
    # every ctypes declaration has the header's argument count, and pointer
    # parameters are passed as pointers (a drift here would shift arguments)
    import ctypes
    from expert_dispatch_planning_gb300 import _lib
    protos = _header_prototypes()
    assert sorted(protos) == sorted(n for n, _, _ in _lib.SIGNATURES)
    for name, _, argtypes in _lib.SIGNATURES:
        params = protos[name]
        assert len(argtypes) == len(params), (name, len(argtypes), params)
        for decl, t in zip(params, argtypes):
            is_ptr = "*" in decl or decl.startswith("cudaStream_t")
            t_is_ptr = t in (ctypes.c_void_p, ctypes.c_char_p) or hasattr(t, "_type_") and t.__name__.startswith("LP_")
            assert is_ptr == t_is_ptr, (name, decl, t)


def test_header_is_plain_c_and_links(lib, tmp_path):
    # a C99 caller: every declared entry point referenced, compiled by a C
    # compiler and linked against the library (nothing is run)
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    cuda_inc = "/usr/local/cuda/include"
    names = declared_functions()
    src = tmp_path / "caller.c"
    src.write_text('#include "moe_dispatch.h"\n#include <stdio.h>\n'
                   "int main(void) {\n    const void* fns[] = {\n" +
                   "".join("        (const void*)&%s,\n" % n for n in names) +
                   "    };\n    printf(\"%%s\\n\", moe_status_string(MOE_OK));\n"
                   "    return (int)(sizeof(fns) / sizeof(fns[0])) == %d ? 0 : 1;\n}\n" % len(names))
    libdir = os.path.dirname(lib._name)
    cmd = [gcc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
           "-I", cuda_inc, str(src), "-o", str(tmp_path / "caller"), "-L", libdir, "-lmoe_dispatch",
           "-Wl,-rpath," + libdir]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
