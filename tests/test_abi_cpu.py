"""Host-only checks of the C ABI: the library builds for sm_103a, loads
without a GPU, exports every entry point include/moe.h declares, and rejects
bad arguments before touching CUDA."""
import ctypes
import os
import re

import pytest

import moe_expert_ffn_02_gb300 as moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:moe_status|const char\s*\*|int32_t)\s*(moe_\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    return moe.load(build_if_missing=True)


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("moe_create", "moe_destroy", "moe_workspace_bytes", "moe_route", "moe_route_from_logits",
              "moe_forward_prefill", "moe_forward_decode", "moe_forward_host", "moe_get_device_status",
              "moe_status_string", "moe_last_error"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    assert moe.moe_abi_version() == 1


def test_library_exports_nothing_else(lib):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", moe.library_path()], capture_output=True, text=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    assert {n for n in exported if n.startswith("moe_")} == set(declared_functions())


def _w():
    # distinct, 16-byte aligned fake device addresses: moe_create must reject
    # the descriptor before it dereferences or copies anything
    return moe.MoeWeights(*[0x10000 * (i + 1) for i in range(14)])


@pytest.mark.parametrize("desc,code", [
    ((100, 256, 8, 2, 1, 256), 2),        # hidden not a multiple of 128
    ((256, 200, 8, 2, 1, 200), 2),        # inter not a multiple of 128
    ((256, 256, 8, 0, 1, 256), 2),        # top_k < 1
    ((256, 256, 8, 9, 1, 256), 2),        # top_k > E
    ((256, 256, 2048, 8, 1, 256), 2),     # E > 1024
    ((256, 256, 64, 33, 1, 256), 2),      # top_k > 32
    ((256, 256, 8, 2, 2, 256), 2),        # two shared experts
    ((256, 256, 8, 2, 1, 384), 2),        # shared_inter != inter
])
def test_create_rejects_bad_descriptors_without_cuda(lib, desc, code):
    d = moe.MoeDesc(*desc)
    h = ctypes.c_void_p()
    st = lib.moe_create(ctypes.byref(d), ctypes.byref(_w()), None, ctypes.byref(h))
    assert st == code and h.value is None
    assert moe.moe_last_error()


def test_create_rejects_null_and_misaligned_weights(lib):
    d = moe.MoeDesc(256, 256, 8, 2, 1, 256)
    h = ctypes.c_void_p()
    w = _w()
    w.w_gate = None
    assert lib.moe_create(ctypes.byref(d), ctypes.byref(w), None, ctypes.byref(h)) == 1
    w = _w()
    w.s_down = 0x10008
    assert lib.moe_create(ctypes.byref(d), ctypes.byref(w), None, ctypes.byref(h)) == 1
    assert lib.moe_create(None, ctypes.byref(w), None, ctypes.byref(h)) == 1


def test_null_handle_calls_fail_cleanly(lib):
    n = ctypes.c_size_t()
    assert lib.moe_workspace_bytes(None, 8, 1, ctypes.byref(n)) == 1
    assert lib.moe_forward_prefill(None, None, 0, None, None, None, 0, None) == 1
    assert lib.moe_forward_decode(None, None, 1, None, None, None, 0, None) == 1
    assert lib.moe_route(None, None, 0, None, None, 0, None) == 1
    assert lib.moe_destroy(None) == 1
    assert lib.moe_debug_inject(None, 1) == 1
    assert moe.moe_status_string(3) == "MOE_ERR_WORKSPACE"


def test_device_check_comes_before_any_other_use_of_the_handle(lib):
    """Entries that enqueue work first compare the current device with the
    one the layer was created on, and return before touching anything else.
    The stand-in handle records device 7 and holds nothing else (its
    pointers are NULL): without a GPU the device query itself fails
    (MOE_ERR_CUDA), on a machine with fewer than 8 GPUs the devices differ
    (MOE_ERR_INVALID_ARG); either way the call returns cleanly."""
    import torch
    fake = (ctypes.c_int32 * 4096)()
    fake[6] = 7                                 # the device field follows the 24-byte descriptor
    no_gpu = not torch.cuda.is_available()
    for st in (lib.moe_forward_prefill(fake, 0x1000, 8, 0x1000, None, 0x1000, 1 << 30, None),
               lib.moe_forward_decode(fake, 0x1000, 8, 0x1000, None, 0x1000, 1 << 30, None),
               lib.moe_route_from_logits_noalloc(fake, 0x1000, 8, None, None),
               lib.moe_tiles_load(fake, 0x1000, None)):
        msg = moe.moe_last_error()
        if no_gpu:
            assert st == 4 and "cudaGetDevice" in msg, (st, msg)
        else:
            assert st == 1 and "is not the layer's device (7)" in msg, (st, msg)


def test_plain_c_caller_compiles_links_and_gets_a_status(lib, tmp_path):
    """The boundary is a C ABI: a C99 program (no C++, no CUDA headers)
    includes include/moe.h with every warning an error, links libmoe.so and
    gets a status and a message back for a rejected call."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "caller.c"
    src.write_text(
        '#include <stdio.h>\n#include "moe.h"\n'
        "int main(void) {\n"
        "    moe_desc d = {0};\n"
        "    moe_layer* layer = 0;\n"
        "    d.hidden = 256; d.inter = 256; d.n_experts = 8; d.top_k = 2; d.n_shared = 1; d.shared_inter = 256;\n"
        "    moe_status st = moe_create(&d, 0, 0, &layer);\n"
        '    printf("%d|%s|%s\\n", (int)st, moe_status_string(st), moe_last_error());\n'
        "    return layer != 0;\n"
        "}\n")
    exe = tmp_path / "caller"
    libdir = os.path.dirname(moe.library_path())
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(ROOT, "include"),
                        str(src), "-L", libdir, "-lmoe", f"-Wl,-rpath,{libdir}", "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    code, name, msg = r.stdout.strip().split("|", 2)
    assert int(code) == 1 and name == "MOE_ERR_INVALID_ARG" and msg
