"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test checks the oracle against a closed form, a brute-force evaluation on
tiny inputs, an invariant, a special case that reduces to a textbook routine,
or a value the pages print.  The `planted_*` tests swap a plausible mistake
into the oracle (on the CPU) and check that a pin then fails.
"""
import math
import os

import numpy as np
import pytest

import moe_synth as S

from oracle import moe_oracle as OM

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- helpers --
def _tiny_layer(E=4, d=128, f=128, seed=0):
    cfg = S.custom("pin", T=6, d=d, f=f, E=E, k=2, seed=seed, cfg_id=77)
    return cfg, S.layer_weights(cfg, 0, threads=1)


def _getter(W):
    return lambda e: {key: v[e] for key, v in W.items()}


def _brute_codes(word_rows, K):
    """Pure-Python nibble extraction (independent of unpack_int4)."""
    rows = []
    for wr in word_rows:
        r = []
        for k in range(K):
            r.append((int(wr[k // 8]) >> (4 * (k % 8))) & 15)
        rows.append(r)
    return np.array(rows, dtype=np.float64)


def _brute_dense(q, s_bits, z_bits, K):
    codes = _brute_codes(q, K)
    s = np.asarray(s_bits, np.uint16).view(np.float16).astype(np.float64)
    z = np.asarray(z_bits, np.uint16).view(np.float16).astype(np.float64)
    out = np.empty_like(codes)
    for n in range(codes.shape[0]):
        for k in range(K):
            out[n, k] = (codes[n, k] - z[n, k // 128]) * s[n, k // 128]
    return out


def _brute_topk(logits, k):
    """Repeated argmax with ties to the lower id (independent of argsort)."""
    T, E = logits.shape
    ids = np.zeros((T, k), np.int32)
    for t in range(T):
        left = list(range(E))
        for j in range(k):
            best = left[0]
            for e in left[1:]:
                if logits[t, e] > logits[t, best]:
                    best = e
            ids[t, j] = best
            left.remove(best)
    return ids


def _dense_masked_forward(x_bits, logits, W, E, d, f, k):
    """Brute force: every expert evaluated for every token, masked by routing.

    out[t] = sum_e mask[t,e] * softmax_sel[t,e] * FFN_e(x_t), with weights
    built from pure-Python dequantisation and the routing from repeated argmax.
    """
    T = x_bits.shape[0]
    x = (np.asarray(x_bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ids = _brute_topk(logits, k)
    out = np.zeros((T, d))
    for e in range(E):
        w13 = _brute_dense(W["w13_q"][e], W["w13_s"][e], W["w13_z"][e], d)
        w2 = _brute_dense(W["w2_q"][e], W["w2_s"][e], W["w2_z"][e], f)
        for t in range(T):
            if e not in ids[t]:
                continue
            sel = [float(logits[t, i]) for i in ids[t]]
            m = max(sel)
            den = sum(math.exp(v - m) for v in sel)
            wt = math.exp(float(logits[t, e]) - m) / den
            g = w13[:f] @ x[t]
            u = w13[f:] @ x[t]
            h = np.array([gi / (1 + math.exp(-gi)) for gi in g]) * u
            out[t] += wt * (w2 @ h)
    return out


# ------------------------------------------------------------ pack/unpack --
def test_unpack_hand_built_words():
    w = np.array([[0x76543210, 0xFEDCBA98]], dtype=np.uint32)
    assert OM.unpack_int4(w, 16).tolist() == [list(range(16))]


def test_pack_unpack_round_trip():
    rng = np.random.default_rng(1)
    codes = rng.integers(0, 16, size=(7, 256)).astype(np.uint8)
    codes[0, :] = 0
    codes[1, :] = 15
    assert np.array_equal(OM.unpack_int4(OM.pack_int4(codes), 256), codes)
    words = rng.integers(0, 2**32, size=(5, 32), dtype=np.uint32)
    assert np.array_equal(OM.pack_int4(OM.unpack_int4(words, 256)), words)


# ---------------------------------------------------------------- format --
def _golden_kv(name):
    kv = {}
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.strip()
            if line and not line.startswith("#"):
                key, *vals = line.split()
                kv.setdefault(key, []).append(vals)
    return kv


def test_format_bits_per_weight_matches_page():
    kv = _golden_kv("format_bits_per_weight.txt")
    bits = float(kv["bits_per_weight"][0][0])
    group = int(kv["group"][0][0])
    assert group == OM.GROUP
    cfg = S.CONFIGS["tiny"]
    w = S.expert_weights(cfg, 0, 0)
    n_weights = 3 * cfg.d * cfg.f
    nbytes = sum(v.nbytes for v in w.values())
    assert nbytes * 8 / n_weights == pytest.approx(bits, abs=0)
    assert cfg.expert_weight_bytes() == nbytes


def test_dequant_group_index_closed_form():
    # codes all 9, zero 8 -> (q - z) = 1; scale of group g = 2^-g
    K = 512
    q = OM.pack_int4(np.full((3, K), 9, np.uint8))
    s = np.array([[1.0, 0.5, 0.25, 0.125]] * 3, np.float16).view(np.uint16)
    z = np.full((3, 4), 8.0, np.float16).view(np.uint16)
    w = OM.dequant(q, s, z, K)
    expect = 2.0 ** -(np.arange(K) // 128)
    assert np.array_equal(w, np.broadcast_to(expect, (3, K)))


def test_dequant_against_bruteforce():
    cfg, W = _tiny_layer(E=1, d=128, f=128)
    a = OM.dequant(W["w13_q"][0], W["w13_s"][0], W["w13_z"][0], 128)
    b = _brute_dense(W["w13_q"][0], W["w13_s"][0], W["w13_z"][0], 128)
    assert np.array_equal(a, b)


# ----------------------------------------------------------------- top-k --
def test_topk_matches_repeated_argmax_with_ties():
    rng = np.random.default_rng(2)
    lg = np.round(rng.standard_normal((64, 16)), 1).astype(np.float32)  # many exact ties
    lg[0, :] = 0.5  # all tied: ids must be 0..k-1
    for k in (1, 3, 8, 16):
        ids, _ = OM.route_topk(lg, k)
        assert np.array_equal(ids, _brute_topk(lg, k))
        assert ids[0].tolist() == list(range(k))


def test_topk_invariants_and_weights():
    rng = np.random.default_rng(3)
    lg = rng.standard_normal((200, 32)).astype(np.float32)
    ids, w = OM.route_topk(lg, 6)
    for t in range(200):
        assert len(set(ids[t].tolist())) == 6
        sel = lg[t, ids[t]]
        rest = np.delete(lg[t], ids[t])
        assert sel.min() >= rest.max()
        assert np.all(np.diff(sel) <= 0)
    assert np.all(w > 0)
    assert np.allclose(w.sum(1), 1.0, rtol=0, atol=1e-12)
    assert np.all(np.diff(w, axis=1) <= 0)  # monotone with the logits
    _, w1 = OM.route_topk(lg, 1)
    assert np.array_equal(w1, np.ones((200, 1)))


def test_topk_golden_examples():
    kv = _golden_kv("softmax_top2.txt")
    for lgs, ks, ids_s, ws in zip(kv["logits"], kv["k"], kv["ids"], kv["w"]):
        lg = np.array([[float(v) for v in lgs]], np.float32)
        ids, w = OM.route_topk(lg, int(ks[0]))
        assert ids[0].tolist() == [int(v) for v in ids_s]
        assert np.allclose(w[0], [float(v) for v in ws], rtol=0, atol=1e-15)


# ----------------------------------------------------------- permutation --
def test_permutation_matches_python_sorted_and_invariants():
    rng = np.random.default_rng(4)
    for E, T, k in ((8, 50, 2), (128, 33, 8), (5, 1, 5)):
        ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
        counts, offsets, sorted_, inv = OM.permute(ids, E)
        R = T * k
        flat = ids.reshape(-1).tolist()
        ref = sorted(range(R), key=lambda a: (flat[a], a))
        assert sorted_.tolist() == ref
        assert counts.sum() == R and offsets[-1] == R and offsets[0] == 0
        assert np.array_equal(np.diff(offsets), counts)
        assert sorted(sorted_.tolist()) == list(range(R))
        assert np.array_equal(sorted_[inv], np.arange(R))
        for e in range(E):
            seg = sorted_[offsets[e]:offsets[e + 1]]
            assert all(flat[a] == e for a in seg)
            assert np.all(np.diff(seg) > 0)


# ------------------------------------------------------------ FFN/layer --
def test_layer_matches_dense_masked_bruteforce():
    cfg, W = _tiny_layer(E=4, d=128, f=128)
    x = S.activations(cfg)
    lg = S.router_logits(cfg)
    lg[1, :] = lg[1, 0]  # a token whose logits all tie
    got = OM.layer_forward(x, lg, _getter(W), cfg.E, cfg.d, cfg.f, cfg.k)
    ref = _dense_masked_forward(x, lg, W, cfg.E, cfg.d, cfg.f, cfg.k)
    assert np.max(np.abs(got - ref)) <= 1e-12 * np.max(np.abs(ref))


def test_single_expert_is_textbook_mlp():
    # E = 1, k = 1: the layer is a dense W4 MLP, out = Wd (SiLU(Wg x) * (Wu x))
    cfg = S.custom("e1", T=5, d=256, f=128, E=1, k=1, cfg_id=78)
    W = S.layer_weights(cfg, 0, threads=1)
    x = S.activations(cfg)
    lg = S.router_logits(cfg)
    got = OM.layer_forward(x, lg, _getter(W), 1, cfg.d, cfg.f, 1)
    xf = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    w13 = _brute_dense(W["w13_q"][0], W["w13_s"][0], W["w13_z"][0], cfg.d)
    w2 = _brute_dense(W["w2_q"][0], W["w2_s"][0], W["w2_z"][0], cfg.f)
    g = np.einsum("td,fd->tf", xf, w13[:cfg.f])
    u = np.einsum("td,fd->tf", xf, w13[cfg.f:])
    ref = np.einsum("tf,df->td", g * 0.5 * (1 + np.tanh(g / 2)) * u, w2)  # SiLU = g*sigmoid(g)
    assert np.max(np.abs(got - ref)) <= 1e-12 * np.max(np.abs(ref))


def _perm_structured_expert(d, f, shifts, amps):
    """Weights with exactly one nonzero dequantised entry per row.

    gate row m: nonzero at k = (m + sg) % d; up row m at (m + su) % d;
    down row n: nonzero at m = (n + sd) % f.  Codes 8 (zero) elsewhere.
    """
    sg, su, sd = shifts
    cg, cu, cd = amps  # codes at the nonzero (zero point 8)
    c13 = np.full((2 * f, d), 8, np.uint8)
    c2 = np.full((d, f), 8, np.uint8)
    for m in range(f):
        c13[m, (m + sg) % d] = cg
        c13[f + m, (m + su) % d] = cu
    for n in range(d):
        c2[n, (n + sd) % f] = cd
    s13 = np.full((2 * f, d // 128), 0.25, np.float16).view(np.uint16)
    s2 = np.full((d, f // 128), 0.5, np.float16).view(np.uint16)
    return {
        "w13_q": OM.pack_int4(c13), "w13_s": s13, "w13_z": np.full_like(s13, 0x4800),
        "w2_q": OM.pack_int4(c2), "w2_s": s2, "w2_z": np.full_like(s2, 0x4800),
    }


def test_closed_form_on_permutation_structured_weights():
    # out[t][n] = sum_j w_tj * 0.5*(cd-8) * SiLU(0.25*(cg-8)*x[t][(m+sg)%d]) * 0.25*(cu-8)*x[t][(m+su)%d]
    # with m = (n + sd) % f.  A transposed matrix, a gate/up swap or a wrong
    # row split changes the result.
    d, f, E, k, T = 256, 128, 3, 2, 4
    shifts = [(5, 17, 3), (100, 2, 64), (7, 7, 1)]
    amps = [(12, 5, 15), (3, 14, 1), (9, 10, 13)]
    experts = [_perm_structured_expert(d, f, shifts[e], amps[e]) for e in range(E)]
    rng = np.random.default_rng(5)
    x = S.f32_to_bf16_bits(rng.standard_normal((T, d)).astype(np.float32))
    lg = rng.standard_normal((T, E)).astype(np.float32)
    got = OM.layer_forward(x, lg, lambda e: experts[e], E, d, f, k)
    xf = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    order = np.argsort(-lg, axis=1, kind="stable")[:, :k]
    ref = np.zeros((T, d))
    for t in range(T):
        sel = lg[t, order[t]].astype(np.float64)
        wts = np.exp(sel - sel.max()) / np.exp(sel - sel.max()).sum()
        for j, e in enumerate(order[t]):
            (sg, su, sd), (cg, cu, cd) = shifts[e], amps[e]
            for n in range(d):
                m = (n + sd) % f
                g = 0.25 * (cg - 8) * xf[t, (m + sg) % d]
                u = 0.25 * (cu - 8) * xf[t, (m + su) % d]
                ref[t, n] += wts[j] * 0.5 * (cd - 8) * (g / (1 + math.exp(-g))) * u
    assert np.max(np.abs(got - ref)) <= 1e-13 * np.max(np.abs(ref))


def test_special_cases_zero_and_linearity():
    cfg, W = _tiny_layer(E=4, d=128, f=256)
    x = S.activations(cfg)
    lg = S.router_logits(cfg)
    base = OM.layer_forward(x, lg, _getter(W), cfg.E, cfg.d, cfg.f, cfg.k)
    assert np.any(base != 0)
    # x = 0 -> out = 0
    z = OM.layer_forward(np.zeros_like(x), lg, _getter(W), cfg.E, cfg.d, cfg.f, cfg.k)
    assert np.all(z == 0)
    # codes equal to the zero point -> out = 0
    Wq = dict(W)
    Wq["w2_q"] = np.full_like(W["w2_q"], 0x88888888)
    z2 = OM.layer_forward(x, lg, _getter(Wq), cfg.E, cfg.d, cfg.f, cfg.k)
    assert np.all(z2 == 0)
    # doubling every down-projection scale doubles the output exactly
    W2 = dict(W)
    W2["w2_s"] = (W["w2_s"].view(np.float16) * np.float16(2)).view(np.uint16)
    dbl = OM.layer_forward(x, lg, _getter(W2), cfg.E, cfg.d, cfg.f, cfg.k)
    assert np.array_equal(dbl, 2 * base)


def test_sampled_tokens_agree_with_full_layer():
    cfg, W = _tiny_layer(E=4, d=128, f=128)
    x = S.activations(cfg)
    lg = S.router_logits(cfg)
    full = OM.layer_forward(x, lg, _getter(W), cfg.E, cfg.d, cfg.f, cfg.k)
    toks = [0, 3, 5]
    part = OM.layer_forward_tokens(x, lg, _getter(W), cfg.E, cfg.d, cfg.f, cfg.k, toks)
    assert np.allclose(part, full[toks], rtol=0, atol=1e-12 * np.abs(full).max())


def test_skew_workload_shape():
    cfg = S.CONFIGS["skew"]
    ids, _ = OM.route_topk(S.router_logits(cfg), cfg.k)
    c = np.bincount(ids.ravel(), minlength=cfg.E)
    assert c.max() / c.mean() > 10 and (c == 0).sum() >= 1


# ------------------------------------------------------- planted mistakes --
def _pins_fail(monkeypatch, name, fn, check):
    monkeypatch.setattr(OM, name, fn)
    with pytest.raises(AssertionError):
        check()


def test_planted_swapped_nibble_order(monkeypatch):
    real = OM.unpack_int4

    def swapped(words, K):
        c = real(words, K).reshape(-1, K // 8, 8)
        return c[..., ::-1].reshape(np.asarray(words).shape[:-1] + (K,))
    _pins_fail(monkeypatch, "unpack_int4", swapped, test_unpack_hand_built_words)
    _pins_fail(monkeypatch, "unpack_int4", swapped, test_layer_matches_dense_masked_bruteforce)


def test_planted_group_off_by_one(monkeypatch):
    def bad(q, s_bits, z_bits, K):
        codes = OM.unpack_int4(q, K).astype(np.float32)
        s = np.roll(OM.fp16_bits_to_f32(s_bits), 1, axis=-1)
        z = OM.fp16_bits_to_f32(z_bits)
        return ((codes - np.repeat(z, 128, -1)) * np.repeat(s, 128, -1)).astype(np.float64)
    _pins_fail(monkeypatch, "dequant", bad, test_dequant_group_index_closed_form)


def test_planted_tie_break_flipped(monkeypatch):
    def bad(logits, k):
        lg = np.asarray(logits, np.float32)
        E = lg.shape[1]
        order = (E - 1 - np.argsort(-lg[:, ::-1], axis=1, kind="stable"))  # ties to the higher id
        ids = order[:, :k].astype(np.int32)
        sel = np.take_along_axis(lg, ids, 1).astype(np.float64)
        ex = np.exp(sel - sel.max(1, keepdims=True))
        return ids, ex / ex.sum(1, keepdims=True)
    _pins_fail(monkeypatch, "route_topk", bad, test_topk_matches_repeated_argmax_with_ties)


def test_planted_unstable_permutation(monkeypatch):
    def bad(ids, E):
        flat = np.asarray(ids, np.int64).reshape(-1)
        counts = np.bincount(flat, minlength=E).astype(np.int32)
        offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
        sorted_ = np.lexsort((-np.arange(flat.size), flat)).astype(np.int32)  # descending a in a segment
        inv = np.empty(flat.size, np.int32)
        inv[sorted_] = np.arange(flat.size)
        return counts, offsets, sorted_, inv
    _pins_fail(monkeypatch, "permute", bad, test_permutation_matches_python_sorted_and_invariants)


def test_planted_transposed_down_and_gate_up_swap(monkeypatch):
    real = OM.expert_matrices

    def transposed(wts, d, f):
        g, u, dn = real(wts, d, f)
        # a square-block transpose of the down matrix (keeps shapes valid)
        dn2 = dn.copy()
        dn2[:f, :f] = dn[:f, :f].T
        return g, u, dn2

    def swapped(wts, d, f):
        g, u, dn = real(wts, d, f)
        return u, g, dn
    _pins_fail(monkeypatch, "expert_matrices", transposed,
               test_closed_form_on_permutation_structured_weights)
    _pins_fail(monkeypatch, "expert_matrices", swapped,
               test_closed_form_on_permutation_structured_weights)


def test_planted_dropped_silu(monkeypatch):
    _pins_fail(monkeypatch, "silu", lambda g: g, test_single_expert_is_textbook_mlp)


def test_planted_full_softmax_not_renormalised(monkeypatch):
    # combine weights taken from a softmax over all E logits, not over the k
    # selected ones
    real = OM.route_topk

    def bad(logits, k):
        ids, _ = real(logits, k)
        lg = np.asarray(logits, np.float64)
        ex = np.exp(lg - lg.max(1, keepdims=True))
        full = ex / ex.sum(1, keepdims=True)
        return ids, np.take_along_axis(full, ids.astype(np.int64), 1)
    _pins_fail(monkeypatch, "route_topk", bad, test_topk_invariants_and_weights)
    _pins_fail(monkeypatch, "route_topk", bad, test_topk_golden_examples)


def test_planted_combine_slot_weights_reversed(monkeypatch):
    real = OM.combine

    def bad(y_perm, inv, w, T, k):
        return real(y_perm, inv, np.ascontiguousarray(w[:, ::-1]), T, k)
    _pins_fail(monkeypatch, "combine", bad, test_layer_matches_dense_masked_bruteforce)


def test_planted_combine_reads_through_sorted(monkeypatch):
    # rows fetched with the forward permutation instead of its inverse
    def bad(y_perm, inv, w, T, k):
        sorted_ = np.argsort(inv)
        out = np.zeros((T, y_perm.shape[1]))
        for j in range(k):
            out += w[:, j:j + 1] * y_perm[sorted_[np.arange(T) * k + j]]
        return out
    _pins_fail(monkeypatch, "combine", bad, test_layer_matches_dense_masked_bruteforce)
