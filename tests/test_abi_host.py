"""The C-ABI library loads, exports every declared symbol, and rejects bad
arguments on the host before any launch (no GPU needed).

Every call here that carries made-up pointers is one the library must reject
during argument checking, so nothing is ever launched with them.
"""
import ctypes
import os
import re
import shutil
import subprocess
import sys

import pytest

from tests.util import build_lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_w4.h")

OK, INVALID, MISALIGNED, UNSUPPORTED, WORKSPACE = 0, 1, 2, 3, 4


@pytest.fixture(scope="module")
def M():
    try:
        build_lib()
    except RuntimeError as e:  # pragma: no cover
        pytest.skip(f"cannot build: {e}")
    import bit_quantized_expert_moe_gb300 as M
    return M


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:moe_status_t|size_t|uint64_t|const char\*)\s+(moe_\w+)\s*\(", text, re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("moe_route_topk", "moe_permute", "moe_expert_ffn_w4a16", "moe_combine", "moe_layer_forward"):
        assert n in names


def test_library_exports_every_declared_symbol(M):
    lib = M.lib()
    for n in declared_functions():
        assert hasattr(lib, n), n


def test_status_strings_and_version(M):
    for code, name in M.STATUS.items():
        assert M.status_str(code) == name
    assert "sm_103a" in M.version()


FAKE = 0x100000  # 16-byte aligned, never dereferenced (every call below fails validation)


def fake_layer(M, E=8, d=256, f=512, group=128, ptr=FAKE):
    return M.moe_w4_layer(E, d, f, group, ptr, ptr, ptr, ptr, ptr, ptr)


def test_workspace_sizes(M):
    lib = M.lib()
    L = fake_layer(M)
    a = lib.moe_layer_workspace_size(ctypes.byref(L), 8, 2)
    b = lib.moe_layer_workspace_size(ctypes.byref(L), 4096, 2)
    assert 256 < a < b
    assert lib.moe_layer_workspace_size(ctypes.byref(fake_layer(M, group=64)), 8, 2) == 0
    assert lib.moe_permute_workspace_size(8, 2, 8) >= 256
    assert lib.moe_expert_ffn_workspace_size(ctypes.byref(L), 16) > 256


def test_layer_forward_rejects_bad_arguments(M):
    lib = M.lib()
    P = FAKE
    big = 1 << 40

    def call(L, T=8, k=2, x=P, lg=P, out=P, ids=None, ws=P, wsb=big):
        return lib.moe_layer_forward(ctypes.byref(L), x, lg, T, k, out, ids, ws, wsb, None)

    assert call(fake_layer(M, group=64)) == UNSUPPORTED
    assert call(fake_layer(M, d=384)) == UNSUPPORTED          # not a multiple of 256
    assert call(fake_layer(M, f=128 + 256)) == UNSUPPORTED
    assert call(fake_layer(M, E=0)) == INVALID
    assert call(fake_layer(M, E=2000)) == INVALID
    assert call(fake_layer(M, ptr=0)) == INVALID
    assert call(fake_layer(M, ptr=FAKE + 4)) == MISALIGNED
    assert call(fake_layer(M), k=9) == INVALID                 # k > E
    assert call(fake_layer(M), k=0) == INVALID
    assert call(fake_layer(M), T=-1) == INVALID
    assert call(fake_layer(M), x=None) == INVALID
    assert call(fake_layer(M), ws=None) == INVALID
    assert call(fake_layer(M), x=P + 8) == MISALIGNED
    assert call(fake_layer(M), ids=P + 2) == MISALIGNED
    assert call(fake_layer(M), wsb=100) == WORKSPACE
    assert call(fake_layer(M), T=0) == OK                      # empty batch: no-op, nothing launched


def test_stage_entry_points_reject_bad_arguments(M):
    lib = M.lib()
    P = FAKE
    assert lib.moe_route_topk(P, 4, 8, 9, P, P, None) == INVALID
    assert lib.moe_route_topk(P, 4, 2000, 2, P, P, None) == INVALID
    assert lib.moe_route_topk(P + 4, 4, 8, 2, P, P, None) == MISALIGNED
    assert lib.moe_route_topk(None, 4, 8, 2, P, P, None) == INVALID
    assert lib.moe_route_topk(None, 0, 8, 2, None, None, None) == OK
    assert lib.moe_permute(P, 4, 9, 8, None, 0, P, P, P, P, None, P, 1 << 30, None) == INVALID
    assert lib.moe_permute(P, 4, 2, 8, None, 0, P, P, P, P, None, P, 16, None) == WORKSPACE
    assert lib.moe_permute(P, 4, 2, 8, None, 0, P + 4, P, P, P, None, P, 1 << 30, None) == MISALIGNED
    assert lib.moe_permute(P, 4, 2, 8, None, 0, P, P, P, P, P, P, 1 << 30, None) == INVALID  # x_perm without x
    assert lib.moe_combine(P, P, P, 4, 2, 12, P, None) == INVALID   # d % 8
    assert lib.moe_combine(P, P, P, 4, 0, 16, P, None) == INVALID
    assert lib.moe_combine(P, P + 4, P, 4, 2, 16, P, None) == MISALIGNED
    assert lib.moe_combine(None, None, None, 0, 2, 16, None, None) == OK
    L = fake_layer(M)
    assert lib.moe_expert_ffn_w4a16(ctypes.byref(L), P, P, 16, None, P, P, 8, None) == WORKSPACE
    assert lib.moe_expert_ffn_w4a16(ctypes.byref(L), P, None, 16, None, P, P, 1 << 30, None) == INVALID
    assert lib.moe_expert_ffn_w4a16(ctypes.byref(L), P + 2, P, 16, None, P, P, 1 << 30, None) == MISALIGNED
    assert lib.moe_get_device_error(None, None) == INVALID


C_CONSUMER = r"""
#include <stdio.h>
#include <string.h>
#include "moe_w4.h"

int main(void) {
    moe_w4_layer L;
    memset(&L, 0, sizeof L);
    L.E = 8;
    L.d_model = 256;
    L.d_ff = 512;
    L.group = 128;
    /* sizes are checked against a complete, aligned layer; nothing is read */
    L.w13_q = L.w2_q = (const uint32_t*)(uintptr_t)0x100000;
    L.w13_s = L.w13_z = L.w2_s = L.w2_z = (const uint16_t*)(uintptr_t)0x100000;
    const size_t ws = moe_layer_workspace_size(&L, 8, 2);
    /* a null layer is rejected on the host, before anything is launched */
    const moe_status_t st = moe_layer_forward(NULL, NULL, NULL, 8, 2, NULL, NULL, NULL, 0, NULL);
    printf("%s|%s|%zu|%d\n", moe_version(), moe_status_str(MOE_OK), ws, (int)st);
    return (ws > 256 && st == MOE_ERR_INVALID_ARG) ? 0 : 1;
}
"""


def test_header_compiles_as_c99_and_links(M, tmp_path):
    """The boundary is usable from plain C: the header compiles as C99 with
    warnings as errors, a program links against the library, and its host-side
    calls behave as documented."""
    gcc = shutil.which("gcc")
    if gcc is None:  # pragma: no cover
        pytest.skip("gcc not found")
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    cuda_lib = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "lib64")
    lib_dir = os.path.dirname(M.LIB_PATH)
    src = tmp_path / "consumer.c"
    src.write_text(C_CONSUMER)
    exe = tmp_path / "consumer"
    cmd = [gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"), "-I", cuda_inc,
           str(src), M.LIB_PATH, f"-Wl,-rpath,{lib_dir}", f"-Wl,-rpath,{cuda_lib}", f"-Wl,-rpath-link,{cuda_lib}",
           "-o", str(exe)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, (r.stdout, r.stderr)
    version, ok, ws, st = r.stdout.strip().split("|")
    assert version == M.version() and ok == M.status_str(OK)
    assert int(ws) == M.lib().moe_layer_workspace_size(ctypes.byref(fake_layer(M)), 8, 2)
    assert int(st) == INVALID


def test_binding_fails_loudly_without_the_library():
    """No CPU fallback: without the built library every call raises."""
    code = ("import bit_quantized_expert_moe_gb300 as M\n"
            "M.LIB_PATH = '/nonexistent/libmoe_w4.so'\n"
            "M._lib = None\n"
            "try:\n"
            "    M.lib()\n"
            "    print('loaded')\n"
            "except RuntimeError as e:\n"
            "    print('raised', 'no CPU fallback' in str(e))\n")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == "raised True"


def test_binding_rejects_host_tensors(M):
    """Host (CPU) tensors are refused before any library call: the layer runs
    only on the device."""
    import torch
    E, d, f = 8, 256, 512
    w = lambda *s: torch.zeros(s, dtype=torch.int32)
    h = lambda *s: torch.zeros(s, dtype=torch.float16)
    layer = M.Layer(E=E, d_model=d, d_ff=f, w13_q=w(E, 2 * f, d // 8), w13_s=h(E, 2 * f, d // 128),
                    w13_z=h(E, 2 * f, d // 128), w2_q=w(E, d, f // 8), w2_s=h(E, d, f // 128), w2_z=h(E, d, f // 128))
    with pytest.raises(ValueError, match="device tensor"):
        M.LayerCall(layer, 2, 2)
