"""moe_permute_noalloc: the permutation for callers that cannot allocate.

Some callers cannot give the library a workspace (a serving runtime whose
device memory is fixed at start-up, code running where allocating CUDA calls
are forbidden), so this entry point keeps its scratch in a fixed array inside
the library image.  This test calls it through the C ABI and checks its
outputs against the workspace-taking moe_permute on the same inputs, on two
calls in a row (a multi-block case, then a small one that reuses the shared
scratch the first call left behind), and checks that a request beyond its
fixed scratch is refused.  The file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest

import moe_synth as S
from tests.util import build_lib, i32_to_dev, x_to_dev

pytestmark = pytest.mark.gpu

MOE_OK, MOE_ERR_SCRATCH_LIMIT = 0, 9


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


def test_noalloc_permute_matches_workspace_entry_point_twice(M):
    import torch
    fn = _noalloc_fn(M)
    for T, E, k, d, seed, skew in [(4096, 128, 8, 512, 1, True), (37, 64, 6, 256, 2, False)]:
        ids, x = _case(T, E, k, d, seed, skew)
        ids_d, x_d = i32_to_dev(ids), x_to_dev(x)
        ref = M.permute(ids_d, E, x=x_d, want_x_perm=True)  # the workspace-taking entry point
        R = T * k
        counts = torch.full((E,), -1, dtype=torch.int32, device="cuda")
        offsets = torch.full((E + 1,), -1, dtype=torch.int32, device="cuda")
        sorted_ = torch.full((R,), -1, dtype=torch.int32, device="cuda")
        inv = torch.full((R,), -1, dtype=torch.int32, device="cuda")
        x_perm = torch.zeros((R, d), dtype=torch.bfloat16, device="cuda")
        stream = torch.cuda.current_stream().cuda_stream
        st = fn(ids_d.data_ptr(), T, k, E, x_d.data_ptr(), d, counts.data_ptr(), offsets.data_ptr(),
                sorted_.data_ptr(), inv.data_ptr(), x_perm.data_ptr(), stream)
        assert st == MOE_OK, M.status_str(st)
        torch.cuda.synchronize()
        for name, got in (("counts", counts), ("offsets", offsets), ("sorted", sorted_), ("inv", inv)):
            assert torch.equal(got, ref[name]), name
        assert torch.equal(x_perm.view(torch.int16), ref["x_perm"].view(torch.int16))


def test_noalloc_permute_refuses_more_rows_than_its_scratch(M):
    fn = _noalloc_fn(M)
    P = 0x100000  # never dereferenced: the size check fails first
    assert fn(P, 32769, 1, 8, None, 0, P, P, P, P, None, None) == MOE_ERR_SCRATCH_LIMIT
    assert M.status_str(MOE_ERR_SCRATCH_LIMIT) == "MOE_ERR_SCRATCH_LIMIT"
