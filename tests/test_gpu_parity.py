"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Integer outputs (routing ids, counts, offsets, permutation) are compared
bit-exactly; floating outputs within the stated bar: max|err| <= 2e-2 rms(ref)
and mean|err| / mean|ref| <= 5e-3 for bf16 outputs; combine weights within a
relative 1e-6 of the fp64 softmax.
"""
import os

import numpy as np
import pytest

import moe_synth as S
from oracle import moe_oracle as OM
from tests.util import assert_close, bf16_to_f64, build_lib, f32_to_dev, i32_to_dev, x_to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    build_lib()
    import bit_quantized_expert_moe_gb300 as M
    return M


@pytest.fixture
def regime():
    """Force the GEMM regime for one test (the library reads MOE_W4_REGIME per call)."""
    old = os.environ.get("MOE_W4_REGIME")

    def set_(v):
        if v is None:
            os.environ.pop("MOE_W4_REGIME", None)
        else:
            os.environ["MOE_W4_REGIME"] = v
    yield set_
    set_(old)


@pytest.fixture
def decode_kernel():
    """Force the decode-regime layer kernel for one test: "fused" (one kernel
    for the whole layer) or "split" (routing/permutation + two GEMV kernels)."""
    old = os.environ.get("MOE_W4_DECODE_KERNEL")

    def set_(v):
        if v is None:
            os.environ.pop("MOE_W4_DECODE_KERNEL", None)
        else:
            os.environ["MOE_W4_DECODE_KERNEL"] = v
    yield set_
    set_(old)


def _getter(W):
    return lambda e: {key: v[e] for key, v in W.items()}


_layer_cache = {}


def _layer(cfg, layer=0):
    key = (cfg.name, cfg.cfg_id, cfg.T, cfg.d, cfg.f, cfg.E, layer, cfg.seed)
    if key not in _layer_cache:
        _layer_cache.clear()
        _layer_cache[key] = S.layer_weights(cfg, layer)
    return _layer_cache[key]


# ------------------------------------------------------------------ stage 1
@pytest.mark.parametrize("name", ["tiny", "decode", "prefill", "skew", "large_decode", "large_prefill"])
def test_route_topk_matches_oracle(M, name):
    cfg = S.CONFIGS[name]
    lg = S.router_logits(cfg)
    ids_ref, w_ref = OM.route_topk(lg, cfg.k)
    ids, w = M.route_topk(f32_to_dev(lg), cfg.k)
    assert np.array_equal(ids.cpu().numpy(), ids_ref)
    np.testing.assert_allclose(w.cpu().numpy(), w_ref, rtol=1e-6, atol=0)


@pytest.mark.parametrize("T,E,k", [(1, 1, 1), (7, 8, 8), (33, 64, 1), (100, 1024, 8), (5, 1000, 40), (300, 256, 8)])
def test_route_topk_ties_and_shapes(M, T, E, k):
    rng = np.random.default_rng(T * 1000 + E)
    lg = np.round(rng.standard_normal((T, E)), 1).astype(np.float32)  # many exact ties
    lg[0, :] = 0.25                                                      # a fully tied row
    if T > 1:
        lg[1, :] = -0.0
        lg[1, ::2] = 0.0                                                 # +0 / -0 ties
    ids_ref, w_ref = OM.route_topk(lg, k)
    ids, w = M.route_topk(f32_to_dev(lg), k)
    assert np.array_equal(ids.cpu().numpy(), ids_ref)
    np.testing.assert_allclose(w.cpu().numpy(), w_ref, rtol=1e-6, atol=0)


# ------------------------------------------------------------------ stage 2
@pytest.mark.parametrize("T,E,k,skew", [(8, 8, 2, False), (2, 128, 8, False), (512, 128, 8, False),
                                        (4096, 128, 8, True), (300, 1024, 7, False), (2048, 16, 1, True),
                                        (1024, 1024, 8, True), (2600, 3, 3, False), (257, 3, 3, False),
                                        (1, 1, 1, False)])
def test_permute_bit_exact(M, T, E, k, skew):
    rng = np.random.default_rng(T + E + k)
    if skew:
        p = np.arange(1, E + 1, dtype=np.float64) ** -1.5
        p[-1] = 0.0
        p /= p.sum()
        ids = np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    else:
        ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    d = 256
    x = S.f32_to_bf16_bits(rng.standard_normal((T, d)).astype(np.float32))
    counts, offsets, sorted_, inv = OM.permute(ids, E)
    out = M.permute(i32_to_dev(ids), E, x=x_to_dev(x), want_x_perm=True)
    assert np.array_equal(out["counts"].cpu().numpy(), counts)
    assert np.array_equal(out["offsets"].cpu().numpy(), offsets)
    assert np.array_equal(out["sorted"].cpu().numpy(), sorted_)
    assert np.array_equal(out["inv"].cpu().numpy(), inv)
    xp = out["x_perm"].view(__import__("torch").int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(xp, x[sorted_ // k])
    assert M.get_device_error(out["ws"]) == 0


def test_permute_reports_out_of_range_ids(M):
    ids = np.array([[0, 1], [2, 9], [-1, 3]], dtype=np.int32)  # 9 and -1 are outside [0, 4)
    out = M.permute(i32_to_dev(ids), 4)
    assert M.get_device_error(out["ws"]) == 6  # MOE_ERR_DEVICE_RANGE
    assert M.get_device_error(out["ws"]) == 0  # read-and-clear
    counts = out["counts"].cpu().numpy()
    assert counts.tolist() == [1, 1, 1, 1]


@pytest.mark.parametrize("T", [600, 2600])
def test_permute_multiblock_skips_out_of_range_ids(M, T):
    """Multi-block permutation (T*k > 2048 assignments; at T = 2600 the placing
    CTAs also copy the rows): ids outside [0, E) set the range error and are
    skipped; the valid assignments keep their stable order by expert and their
    activation rows."""
    rng = np.random.default_rng(T)
    E, k, d = 64, 8, 256
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    flat = ids.reshape(-1)
    bad = rng.choice(flat.size, size=37, replace=False)
    flat[bad[:20]] = E + rng.integers(0, 5, size=20)
    flat[bad[20:]] = -1 - rng.integers(0, 5, size=17)
    x = S.f32_to_bf16_bits(rng.standard_normal((T, d)).astype(np.float32))
    out = M.permute(i32_to_dev(ids), E, x=x_to_dev(x), want_x_perm=True)
    assert M.get_device_error(out["ws"]) == 6  # MOE_ERR_DEVICE_RANGE
    valid = (flat >= 0) & (flat < E)
    nv = int(valid.sum())
    counts = out["counts"].cpu().numpy()
    assert np.array_equal(counts, np.bincount(flat[valid], minlength=E))
    assert np.array_equal(out["offsets"].cpu().numpy(), np.concatenate([[0], np.cumsum(counts)]))
    a_valid = np.nonzero(valid)[0]
    order = a_valid[np.argsort(flat[valid], kind="stable")]  # stable sort of the valid assignments
    assert np.array_equal(out["sorted"].cpu().numpy()[:nv], order)
    assert np.array_equal(out["inv"].cpu().numpy()[order], np.arange(nv))
    xp = out["x_perm"].view(__import__("torch").int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(xp[:nv], x[order // k])


# ------------------------------------------------------------------ stage 3
def _ffn_case(cfg, W, rows_by_expert, seed=0):
    """x_perm rows grouped by expert with the given counts, plus oracle y."""
    rng = np.random.default_rng(seed)
    counts = np.asarray(rows_by_expert, np.int32)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    R = int(offsets[-1])
    x = S.f32_to_bf16_bits(rng.standard_normal((R, cfg.d)).astype(np.float32))
    row_w = rng.uniform(0.1, 1.0, size=R)
    y_ref = OM.expert_ffn(OM.bf16_bits_to_f64(x), offsets, _getter(W), cfg.d, cfg.f)
    return x, offsets, row_w, y_ref


@pytest.mark.parametrize("regime_name", ["decode", "prefill"])
def test_expert_ffn_small_both_regimes(M, regime, regime_name):
    cfg = S.CONFIGS["tiny"]
    W = _layer(cfg)
    layer = M.Layer.from_numpy(W)
    x, offsets, row_w, y_ref = _ffn_case(cfg, W, [3, 0, 1, 5, 2, 0, 4, 1])
    regime(regime_name)
    y = M.expert_ffn_w4a16(layer, x_to_dev(x), i32_to_dev(offsets))
    assert_close(bf16_to_f64(y), y_ref, f"ffn {regime_name}")
    yw = M.expert_ffn_w4a16(layer, x_to_dev(x), i32_to_dev(offsets), row_w=f32_to_dev(row_w))
    # compare row by row in units of the row weight (the bar is relative to rms)
    rw = row_w.astype(np.float32).astype(np.float64)[:, None]
    assert_close(bf16_to_f64(yw) / rw, y_ref, f"ffn row_w {regime_name}")


def test_expert_ffn_prefill_ragged_tiles(M, regime):
    # one expert spanning three token tiles (256 + 256 + 91), tails of 1..33 rows, empty experts
    cfg = S.custom("ragged", T=1, d=512, f=768, E=7, k=1, cfg_id=80)
    W = S.layer_weights(cfg, 0)
    layer = M.Layer.from_numpy(W)
    x, offsets, row_w, y_ref = _ffn_case(cfg, W, [603, 0, 1, 33, 16, 0, 17], seed=3)
    regime("prefill")
    y = M.expert_ffn_w4a16(layer, x_to_dev(x), i32_to_dev(offsets), row_w=f32_to_dev(row_w))
    rw = row_w.astype(np.float32).astype(np.float64)[:, None]
    assert_close(bf16_to_f64(y) / rw, y_ref, "ragged")


def test_expert_ffn_decode_many_rows_per_expert(M, regime):
    # more rows of one expert than a GEMV pass holds (passes of 2 rows)
    cfg = S.custom("passes", T=1, d=768, f=512, E=5, k=1, cfg_id=81)
    W = S.layer_weights(cfg, 0)
    layer = M.Layer.from_numpy(W)
    x, offsets, _, y_ref = _ffn_case(cfg, W, [5, 1, 0, 7, 3], seed=4)
    regime("decode")
    y = M.expert_ffn_w4a16(layer, x_to_dev(x), i32_to_dev(offsets))
    assert_close(bf16_to_f64(y), y_ref, "gemv passes")


# ------------------------------------------------------------------ stage 4
def test_combine_matches_oracle(M):
    import torch
    rng = np.random.default_rng(7)
    T, k, d = 333, 6, 1024
    R = T * k
    y = S.f32_to_bf16_bits(rng.standard_normal((R, d)).astype(np.float32))
    inv = rng.permutation(R).astype(np.int32)
    w = rng.uniform(0, 1, size=(T, k)).astype(np.float32)
    ref = OM.combine(OM.bf16_bits_to_f64(y), inv, w.astype(np.float64), T, k)
    out = M.combine(x_to_dev(y), i32_to_dev(inv), f32_to_dev(w))
    got = bf16_to_f64(out)
    # only the final bf16 rounding separates the two: |err| <= 2^-8 |ref| (+ fp32 noise)
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-6 * np.abs(ref).max())
    assert out.dtype == torch.bfloat16


# ------------------------------------------------------------- whole layer
def _run_layer(M, cfg, layer_idx=0):
    W = _layer(cfg, layer_idx)
    layer = M.Layer.from_numpy(W)
    x = S.activations(cfg, layer_idx)
    lg = S.router_logits(cfg, layer_idx)
    import torch
    ids = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device="cuda")
    call = M.LayerCall(layer, cfg.T, cfg.k)
    out = torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16, device="cuda")
    call(x_to_dev(x), f32_to_dev(lg), out, ids)
    assert M.get_device_error(call.ws) == 0
    return W, x, lg, ids.cpu().numpy(), bf16_to_f64(out)


@pytest.mark.parametrize("name", ["tiny", "decode", "prefill", "skew", "large_decode", "large_prefill"])
def test_layer_forward_full(M, name):
    """Every output element of the whole layer at each workload's full size
    (the oracle's cost is dominated by dequantising the touched experts, so the
    4096-token skewed layer and the 512-token large layer are affordable)."""
    cfg = S.CONFIGS[name]
    W, x, lg, ids, out = _run_layer(M, cfg)
    ref, inter = OM.layer_forward(x, lg, _getter(W), cfg.E, cfg.d, cfg.f, cfg.k, want_intermediates=True)
    assert np.array_equal(ids, inter["ids"])
    assert_close(out, ref, f"layer {name}")


def test_decode_layers_of_the_stack(M):
    cfg = S.CONFIGS["decode"]
    for layer_idx in (1, 47):
        W, x, lg, ids, out = _run_layer(M, cfg, layer_idx)
        ref = OM.layer_forward(x, lg, _getter(W), cfg.E, cfg.d, cfg.f, cfg.k)
        assert_close(out, ref, f"decode layer {layer_idx}")


def test_regimes_agree_on_the_same_input(M, regime):
    cfg = S.CONFIGS["decode"]
    regime("decode")
    W, x, lg, ids_a, out_a = _run_layer(M, cfg)
    regime("prefill")
    _, _, _, ids_b, out_b = _run_layer(M, cfg)
    regime(None)
    assert np.array_equal(ids_a, ids_b)
    ref = OM.layer_forward(x, lg, _getter(W), cfg.E, cfg.d, cfg.f, cfg.k)
    assert_close(out_a, ref, "decode regime")
    assert_close(out_b, ref, "prefill regime")


def test_deterministic_and_graph_replay_equals_eager(M):
    import torch
    for name in ("decode", "prefill"):
        cfg = S.CONFIGS[name]
        W = _layer(cfg)
        layer = M.Layer.from_numpy(W)
        x = x_to_dev(S.activations(cfg))
        lg = f32_to_dev(S.router_logits(cfg))
        call = M.LayerCall(layer, cfg.T, cfg.k)
        o1 = torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16, device="cuda")
        o2 = torch.empty_like(o1)
        o3 = torch.empty_like(o1)
        call(x, lg, o1)
        call(x, lg, o2)
        torch.cuda.synchronize()
        assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)), name
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            call(x, lg, o3, stream=s)  # warm-up on the capture stream
            torch.cuda.synchronize()
            o3.zero_()
            with torch.cuda.graph(g, stream=s):
                call(x, lg, o3, stream=s)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(o1.view(torch.int16), o3.view(torch.int16)), name


@pytest.mark.parametrize("T,E,k,d,f", [(1, 1, 1, 256, 256), (3, 4, 4, 256, 512), (70, 16, 1, 512, 256),
                                       (9, 32, 8, 1024, 256)])
def test_layer_edge_shapes(M, T, E, k, d, f):
    cfg = S.custom("edge", T=T, d=d, f=f, E=E, k=k, cfg_id=90 + T)
    W = S.layer_weights(cfg, 0)
    _layer_cache.clear()
    layer = M.Layer.from_numpy(W)
    x = S.activations(cfg)
    lg = S.router_logits(cfg)
    out = M.layer_forward(layer, x_to_dev(x), f32_to_dev(lg), k)
    ref = OM.layer_forward(x, lg, _getter(W), E, d, f, k)
    assert_close(bf16_to_f64(out), ref, f"edge {T},{E},{k},{d},{f}")


def test_zero_tokens_is_a_no_op(M):
    import torch
    cfg = S.CONFIGS["tiny"]
    layer = M.Layer.from_numpy(_layer(cfg))
    x = torch.empty((0, cfg.d), dtype=torch.bfloat16, device="cuda")
    lg = torch.empty((0, cfg.E), dtype=torch.float32, device="cuda")
    out = M.layer_forward(layer, x, lg, cfg.k, out=torch.empty((0, cfg.d), dtype=torch.bfloat16, device="cuda"))
    assert out.shape == (0, cfg.d)


# ------------------------------------------- decode regime: one-kernel layer
@pytest.mark.parametrize("kernel", ["fused", "split"])
@pytest.mark.parametrize("name", ["tiny", "decode", "large_decode"])
def test_decode_layer_kernels_match_oracle(M, decode_kernel, kernel, name):
    cfg = S.CONFIGS[name]
    decode_kernel(kernel)
    W, x, lg, ids, out = _run_layer(M, cfg)
    decode_kernel(None)
    ref, inter = OM.layer_forward(x, lg, _getter(W), cfg.E, cfg.d, cfg.f, cfg.k, want_intermediates=True)
    assert np.array_equal(ids, inter["ids"])
    assert_close(out, ref, f"{name} {kernel}")


@pytest.mark.parametrize("T,E,k,d,f,ties", [
    (1, 1, 1, 256, 256, False),     # one expert, one token
    (3, 4, 4, 256, 512, False),     # every token on every expert
    (8, 8, 8, 512, 256, False),     # 8 tokens per expert: all MMA columns used
    (8, 16, 8, 1280, 768, True),    # ragged chunks (10 and 6 groups), tied logits
    (2, 1024, 32, 256, 256, False), # E = 1024, R = 64
    (5, 64, 2, 2048, 1024, True),
    (1, 256, 40, 512, 256, False),  # k > 32: slots j and j + 32 per lane in the router
    (8, 16, 8, 7168, 2048, False),  # the smallest ring: 8 slots, 2 per producer pipeline
])
def test_fused_decode_layer_shapes(M, T, E, k, d, f, ties):
    import torch
    cfg = S.custom("fused", T=T, d=d, f=f, E=E, k=k, cfg_id=70 + T + k)
    W = S.layer_weights(cfg, 0)
    _layer_cache.clear()
    layer = M.Layer.from_numpy(W)
    x = S.activations(cfg)
    lg = S.router_logits(cfg)
    if ties:
        lg = np.round(lg * 2.0).astype(np.float32) / 2.0  # many equal logits
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    call = M.LayerCall(layer, T, k)
    out = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
    call(x_to_dev(x), f32_to_dev(lg), out, ids)
    assert M.get_device_error(call.ws) == 0
    ref, inter = OM.layer_forward(x, lg, _getter(W), E, d, f, k, want_intermediates=True)
    assert np.array_equal(ids.cpu().numpy(), inter["ids"])
    assert_close(bf16_to_f64(out), ref, f"fused {T},{E},{k},{d},{f}")


def test_fused_decode_repeated_calls_share_the_grid_barrier(M, decode_kernel):
    """The grid-barrier layer kernel counts arrivals in the workspace header;
    every call must add exactly one arrival per CTA and leave nothing pending,
    so calls on one workspace keep working and agree."""
    import torch
    decode_kernel("fused")
    cfg = S.CONFIGS["decode"]
    W = _layer(cfg)
    layer = M.Layer.from_numpy(W)
    call = M.LayerCall(layer, cfg.T, cfg.k)
    outs = []
    for layer_idx in (0, 1, 0, 1, 0):
        x = x_to_dev(S.activations(cfg, layer_idx))
        lg = f32_to_dev(S.router_logits(cfg, layer_idx))
        o = torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16, device="cuda")
        call(x, lg, o)
        outs.append(o)
    torch.cuda.synchronize()
    assert M.get_device_error(call.ws) == 0
    arrivals = int(call.ws[64:72].view(torch.int64).item())
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    assert arrivals == 5 * n_sm
    for a, b in ((0, 2), (0, 4), (1, 3)):
        assert torch.equal(outs[a].view(torch.int16), outs[b].view(torch.int16))


def test_fused_decode_barrier_wait_that_runs_out_reports_a_timeout(M, decode_kernel):
    """The grid-barrier kernel's bounded wait running out: the workspace's
    arrival counter is set one short of a multiple of the grid size, so only
    the first CTA to arrive passes the barrier and every other CTA waits until
    the 2 s limit.  The call must end (no hang), report MOE_ERR_TIMEOUT, and
    after moe_get_device_error has cleared the header the next call on the
    same workspace must match the oracle again."""
    import torch
    decode_kernel("fused")
    cfg = S.CONFIGS["decode"]
    W = _layer(cfg, 0)
    layer = M.Layer.from_numpy(W)
    call = M.LayerCall(layer, cfg.T, cfg.k)
    x, lg = x_to_dev(S.activations(cfg, 0)), f32_to_dev(S.router_logits(cfg, 0))
    out = torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16, device="cuda")
    call(x, lg, out)
    assert M.get_device_error(call.ws) == 0
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    arrivals = int(call.ws[64:72].view(torch.int64).item())
    assert arrivals % n_sm == 0
    call.ws[64:72].view(torch.int64).fill_(arrivals + n_sm - 1)
    call(x, lg, out)
    assert M.get_device_error(call.ws) == 7  # MOE_ERR_TIMEOUT
    assert int(call.ws[:256].count_nonzero()) == 0
    out.zero_()
    call(x, lg, out)
    assert M.get_device_error(call.ws) == 0
    ref = OM.layer_forward(S.activations(cfg, 0), S.router_logits(cfg, 0), _getter(W), cfg.E, cfg.d, cfg.f, cfg.k)
    assert_close(bf16_to_f64(out), ref, "fused after a timeout")


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["decode", "large_decode"])
def test_fused_decode_back_to_back_calls_on_one_workspace(M, name):
    """Consecutive one-kernel decode calls overlap their launches (each waits
    for the previous kernel before it touches global memory) and share one
    workspace, whose h rows and grid-barrier counter every call rewrites.  A
    stream of calls over alternating layers, eager and replayed as a CUDA
    graph, must give bit-for-bit the outputs of the same calls made one at a
    time with a synchronisation between them, and report no device error."""
    import torch
    cfg = S.CONFIGS[name]
    nl = 3 if name == "decode" else 2
    layers = [M.Layer.from_numpy(_layer(cfg, l)) for l in range(nl)]
    xs = [x_to_dev(S.activations(cfg, l)) for l in range(nl)]
    lgs = [f32_to_dev(S.router_logits(cfg, l)) for l in range(nl)]
    ws = M.workspace(max(M.layer_workspace_size(ly, cfg.T, cfg.k) for ly in layers))
    calls = [M.LayerCall(ly, cfg.T, cfg.k, ws=ws) for ly in layers]
    ref = []
    for l in range(nl):
        o = torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16, device="cuda")
        calls[l](xs[l], lgs[l], o)
        torch.cuda.synchronize()
        ref.append(o)
        # the single calls are themselves held to the oracle
        W = _layer(cfg, l)
        ora = OM.layer_forward(S.activations(cfg, l), S.router_logits(cfg, l), _getter(W), cfg.E, cfg.d, cfg.f,
                               cfg.k)
        assert_close(bf16_to_f64(o), ora, f"{name} layer {l}, single call")
    seq = [i % nl for i in range(24)]
    outs = [torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16, device="cuda") for _ in seq]
    for o, l in zip(outs, seq):
        calls[l](xs[l], lgs[l], o)
    torch.cuda.synchronize()
    assert M.get_device_error(ws) == 0
    for o, l in zip(outs, seq):
        assert torch.equal(o.view(torch.int16), ref[l].view(torch.int16))
    # the same stream of calls captured once and replayed twice
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    for o in outs:
        o.zero_()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for o, l in zip(outs, seq):
                calls[l](xs[l], lgs[l], o, stream=s)
        g.replay()
        g.replay()
    s.synchronize()
    assert M.get_device_error(ws) == 0
    for o, l in zip(outs, seq):
        assert torch.equal(o.view(torch.int16), ref[l].view(torch.int16))
