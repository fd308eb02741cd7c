"""moe_permute_noalloc: the permutation for callers that cannot allocate.

Some callers cannot give the library a workspace (a serving runtime whose
device memory is fixed at start-up, code running where allocating CUDA calls
are forbidden), so this entry point keeps its scratch in a fixed array inside
the library image.  These tests call it through the C ABI and check it
against the oracle's permutation (and the workspace-taking moe_permute) on
two calls in a row (a multi-block case, then a small one that reuses the
shared scratch the first call left behind), at the largest size its scratch
accepts (T*k = 32768 with E = 1024), with T = 0, with ids outside [0, E), and
that a request beyond its fixed scratch is refused.  A fresh process checks
that a first call made during a stream capture is refused without harming
the capture.  The file is named to be collected last.
"""
import ctypes
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest

import moe_synth as S
from oracle import moe_oracle as OM
from tests.util import build_lib, i32_to_dev, x_to_dev

pytestmark = pytest.mark.gpu

MOE_OK, MOE_ERR_SCRATCH_LIMIT, MOE_ERR_CAPTURE = 0, 9, 10
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def M():
    build_lib()
    import bit_quantized_expert_moe_gb300 as M
    return M


def _noalloc_fn(M):
    fn = M.lib().moe_permute_noalloc
    V, I32 = ctypes.c_void_p, ctypes.c_int32
    fn.restype = I32
    fn.argtypes = [V, I32, I32, I32, V, I32, V, V, V, V, V, V]
    return fn


def _case(T, E, k, d, seed, skew):
    rng = np.random.default_rng(seed)
    if skew:
        p = np.arange(1, E + 1, dtype=np.float64) ** -1.2
        p /= p.sum()
        ids = np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    else:
        ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    x = S.f32_to_bf16_bits(rng.standard_normal((T, d)).astype(np.float32))
    return ids, x


def _call(M, fn, ids, E, x):
    """One moe_permute_noalloc call; returns (status, outputs as numpy)."""
    import torch
    T, k = ids.shape
    R, d = T * k, x.shape[1]
    ids_d, x_d = i32_to_dev(ids.reshape(max(T, 1), k) if T else np.zeros((1, k), np.int32)), x_to_dev(
        x if T else np.zeros((1, max(d, 8)), np.uint16))
    counts = torch.full((E,), -1, dtype=torch.int32, device="cuda")
    offsets = torch.full((E + 1,), -1, dtype=torch.int32, device="cuda")
    sorted_ = torch.full((max(R, 1),), -1, dtype=torch.int32, device="cuda")
    inv = torch.full((max(R, 1),), -1, dtype=torch.int32, device="cuda")
    x_perm = torch.zeros((max(R, 1), max(d, 8)), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    st = fn(ids_d.data_ptr(), T, k, E, x_d.data_ptr() if T else None, d if T else 0, counts.data_ptr(),
            offsets.data_ptr(), sorted_.data_ptr(), inv.data_ptr(), x_perm.data_ptr() if T else None, stream)
    torch.cuda.synchronize()
    out = {"counts": counts.cpu().numpy(), "offsets": offsets.cpu().numpy(),
           "sorted": sorted_.cpu().numpy()[:R], "inv": inv.cpu().numpy()[:R],
           "x_perm": x_perm.view(torch.int16).cpu().numpy().view(np.uint16)[:R]}
    return st, out


def test_noalloc_permute_matches_oracle_twice(M):
    fn = _noalloc_fn(M)
    for T, E, k, d, seed, skew in [(4096, 128, 8, 512, 1, True), (37, 64, 6, 256, 2, False)]:
        ids, x = _case(T, E, k, d, seed, skew)
        st, got = _call(M, fn, ids, E, x)
        assert st == MOE_OK, M.status_str(st)
        counts, offsets, sorted_, inv = OM.permute(ids, E)
        for name, ref in (("counts", counts), ("offsets", offsets), ("sorted", sorted_), ("inv", inv)):
            assert np.array_equal(got[name], ref), name
        assert np.array_equal(got["x_perm"], x[sorted_ // k])
        # and the workspace-taking entry point agrees on the same inputs
        w = M.permute(i32_to_dev(ids), E)
        assert np.array_equal(w["sorted"].cpu().numpy(), got["sorted"])


def test_noalloc_permute_at_its_largest_size(M):
    """T*k = MOE_NOALLOC_MAX_ROWS with E = 1024: the largest layout the fixed
    scratch holds must be accepted and correct."""
    fn = _noalloc_fn(M)
    ids, x = _case(4096, 1024, 8, 256, 5, True)
    st, got = _call(M, fn, ids, 1024, x)
    assert st == MOE_OK, M.status_str(st)
    counts, offsets, sorted_, inv = OM.permute(ids, 1024)
    for name, ref in (("counts", counts), ("offsets", offsets), ("sorted", sorted_), ("inv", inv)):
        assert np.array_equal(got[name], ref), name
    assert np.array_equal(got["x_perm"], x[sorted_ // 8])


def test_noalloc_permute_zero_tokens(M):
    fn = _noalloc_fn(M)
    st, got = _call(M, fn, np.zeros((0, 4), np.int32), 16, np.zeros((0, 64), np.uint16))
    assert st == MOE_OK, M.status_str(st)
    assert np.all(got["counts"] == 0) and np.all(got["offsets"] == 0)


def test_noalloc_permute_skips_out_of_range_ids(M):
    """Ids outside [0, E) are skipped: counts hold only the valid ids (so they
    sum to less than T*k) and the valid assignments keep their stable order."""
    fn = _noalloc_fn(M)
    E = 8
    ids = np.array([[0, 3], [9, 1], [3, -1], [7, 3], [2, 8]], dtype=np.int32)
    x = S.f32_to_bf16_bits(np.random.default_rng(3).standard_normal((5, 64)).astype(np.float32))
    st, got = _call(M, fn, ids, E, x)
    assert st == MOE_OK, M.status_str(st)
    flat = ids.reshape(-1)
    valid = (flat >= 0) & (flat < E)
    assert np.array_equal(got["counts"], np.bincount(flat[valid], minlength=E))
    assert got["counts"].sum() == valid.sum() < flat.size
    assert np.array_equal(got["offsets"][1:], np.cumsum(got["counts"]))
    a_valid = np.nonzero(valid)[0]
    order = a_valid[np.argsort(flat[valid], kind="stable")]  # the oracle's rule on the valid ids
    assert np.array_equal(got["sorted"][:valid.sum()], order)
    assert np.array_equal(got["inv"][order], np.arange(valid.sum()))


def test_noalloc_permute_refuses_more_rows_than_its_scratch(M):
    fn = _noalloc_fn(M)
    P = 0x100000  # never dereferenced: the size check fails first
    assert fn(P, 32769, 1, 8, None, 0, P, P, P, P, None, None) == MOE_ERR_SCRATCH_LIMIT
    assert M.status_str(MOE_ERR_SCRATCH_LIMIT) == "MOE_ERR_SCRATCH_LIMIT"


def test_noalloc_first_call_inside_a_capture_is_refused(M):
    """In a fresh process, where the scratch address is not yet known, a first
    call made while the stream captures returns MOE_ERR_CAPTURE and leaves the
    capture usable; the next call outside the capture works."""
    script = textwrap.dedent(f"""
        import ctypes, sys
        import numpy as np, torch
        sys.path.insert(0, {ROOT!r})
        import bit_quantized_expert_moe_gb300 as M
        from oracle import moe_oracle as OM
        fn = M.lib().moe_permute_noalloc
        V, I32 = ctypes.c_void_p, ctypes.c_int32
        fn.restype = I32
        fn.argtypes = [V, I32, I32, I32, V, I32, V, V, V, V, V, V]
        ids = torch.tensor([[1, 0], [0, 2], [2, 1]], dtype=torch.int32, device="cuda")
        buf = [torch.zeros(8, dtype=torch.int32, device="cuda") for _ in range(4)]
        y = torch.zeros(16, device="cuda")
        s = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            st = fn(ids.data_ptr(), 3, 2, 3, None, 0, *[b.data_ptr() for b in buf], None, s.cuda_stream)
            y.add_(1.0)
        g.replay()
        torch.cuda.synchronize()
        assert st == {MOE_ERR_CAPTURE}, st
        assert float(y.sum()) == 16.0, "capture was harmed"
        st = fn(ids.data_ptr(), 3, 2, 3, None, 0, *[b.data_ptr() for b in buf], None,
                torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        assert st == 0, st
        counts, offsets, sorted_, inv = OM.permute(ids.cpu().numpy(), 3)
        assert np.array_equal(buf[0].cpu().numpy()[:3], counts)
        assert np.array_equal(buf[2].cpu().numpy()[:6], sorted_)
        print("capture-refusal ok")
    """)
    r = subprocess.run([sys.executable, "-c", script], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and "capture-refusal ok" in r.stdout, r.stdout + r.stderr
