"""CPU oracle of the routed W4A16 mixture-of-experts FFN layer.

TEST INFRASTRUCTURE ONLY.  This module is imported by the tests, by
`__graft_entry__.smoke()` and by the CPU-baseline leg of `bench.py`; the
product path (the CUDA library and its Python binding) never imports, links or
calls it, and it imports nothing from the product path.

It is deliberately plain: numpy, float64 for all floating-point work except
the one step the method fixes in float32 (the group dequantisation), library
matmuls as steps, no blocking, fusion or reordering beyond the definitions.

Sources.  The pages that describe the method print no formula or code for the
layer; they fix the weight format and the shape of the computation:
  * "Measured results" (vllm-omni docs/edge/results.md), sections Memory,
    Speed and Fidelity: W4A16 with groups of 128 along the reduction axis,
    4.25 bits per weight (a 4-bit code plus a 16-bit scale and a 16-bit zero
    per group of 128), 4-bit codes stored packed eight to a 32-bit word
    (`unpack_nibbles` expands them 8x into int32).
  * "Performance and verification" (bloomery docs/performance.md), section
    "Why it is fast": the tokens of a batch are grouped by expert so that an
    expert's weights are fetched a single time per batch, and the experts'
    matrix products are grouped; section "How it is verified": the router's
    expert ids are integers and are held to exact equality (ties aside).
The remaining definitions are the plainest reading of the problem statement:
top-k by descending logit with ties to the lower expert id, combine weights =
softmax over the k selected logits, SiLU(gate) * up, a stable counting-sort
permutation and the router-weighted combine.  Each function below says which
reading it implements.

Parity status per function (see the pins in tests/test_oracle_pins.py):
  unpack_int4 / pack_int4 ... pinned (hand-built word, round trip)
  dequant ................... pinned (hand-derived values, 4.25 bits/weight)
  route_topk ................ pinned (brute-force repeated argmax, ties, invariants)
  permute ................... pinned (Python sorted(), invariants)
  expert_ffn / combine ...... pinned (dense masked brute force, E=1 textbook MLP,
                              closed form on permutation-structured weights,
                              zero/linearity special cases)
"""
from __future__ import annotations

import numpy as np

GROUP = 128


# --------------------------------------------------------------------------
# Storage formats
# --------------------------------------------------------------------------
def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns -> float64 (exact: bf16 is the top half of fp32)."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def fp16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """IEEE fp16 bit patterns -> float32 (exact)."""
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float32)


def unpack_int4(words: np.ndarray, K: int) -> np.ndarray:
    """Codes [rows, K] (uint8, 0..15) from packed words [rows, K/8] (uint32).

    Code k of a row sits in word k // 8 at bits 4*(k % 8) .. 4*(k % 8)+3:
    eight 4-bit codes per 32-bit word, the lowest k in the lowest nibble.
    """
    words = np.asarray(words, dtype=np.uint32)
    assert words.shape[-1] * 8 == K
    shifts = (4 * np.arange(8, dtype=np.uint32))
    codes = (words[..., :, None] >> shifts) & np.uint32(0xF)  # [rows, K/8, 8]
    return codes.reshape(*words.shape[:-1], K).astype(np.uint8)


def pack_int4(codes: np.ndarray) -> np.ndarray:
    """Inverse of unpack_int4: codes [rows, K] (0..15) -> words [rows, K/8]."""
    codes = np.asarray(codes, dtype=np.uint32)
    K = codes.shape[-1]
    assert K % 8 == 0 and codes.max(initial=0) < 16
    c = codes.reshape(*codes.shape[:-1], K // 8, 8)
    shifts = (4 * np.arange(8, dtype=np.uint32))
    return np.bitwise_or.reduce(c << shifts, axis=-1).astype(np.uint32)


def dequant(q: np.ndarray, s_bits: np.ndarray, z_bits: np.ndarray, K: int) -> np.ndarray:
    """Group dequantisation of one packed matrix -> float64 [rows, K].

    w[n, k] = (code[n, k] - z[n, k // 128]) * s[n, k // 128], evaluated in
    float32 as the method states, then widened to float64.  The zero is in
    code units (the workloads store z = 8, i.e. zero-centred codes).
    """
    codes = unpack_int4(q, K).astype(np.float32)
    s = fp16_bits_to_f32(s_bits)
    z = fp16_bits_to_f32(z_bits)
    assert s.shape[-1] * GROUP == K and z.shape == s.shape
    s_k = np.repeat(s, GROUP, axis=-1)
    z_k = np.repeat(z, GROUP, axis=-1)
    w32 = (codes - z_k) * s_k
    return w32.astype(np.float64)


# --------------------------------------------------------------------------
# Stage 1: top-k routing
# --------------------------------------------------------------------------
def route_topk(logits: np.ndarray, k: int):
    """Top-k expert selection and combine weights.

    For each token: order the experts by (-logit, expert id) ascending and keep
    the first k, so slot 0 holds the largest logit and equal logits go to the
    lower id (router ids are integer outputs that must match exactly).  The
    selection compares the float32 values only; no arithmetic touches them.
    Combine weights: softmax over the k selected logits, in float64.
    Returns ids int32 [T, k] and w float64 [T, k].
    """
    logits = np.asarray(logits, dtype=np.float32)
    T, E = logits.shape
    assert 1 <= k <= E
    order = np.argsort(-logits, axis=1, kind="stable")  # stable: ties keep ascending id
    ids = order[:, :k].astype(np.int32)
    sel = np.take_along_axis(logits, ids, axis=1).astype(np.float64)
    m = sel.max(axis=1, keepdims=True)
    ex = np.exp(sel - m)
    w = ex / ex.sum(axis=1, keepdims=True)
    return ids, w


# --------------------------------------------------------------------------
# Stage 2: token -> expert permutation
# --------------------------------------------------------------------------
def permute(ids: np.ndarray, E: int):
    """Expert histogram, exclusive prefix sum and stable permutation.

    Assignment a = t*k + j (token t, slot j) goes to expert ids[t, j].
    counts[e]   = number of assignments to e
    offsets     = exclusive prefix sum of counts, length E+1
    sorted[i]   = the assignment at permuted position i: assignments grouped by
                  expert, ascending a inside each expert's segment (stable)
    inv[a]      = position of assignment a, so sorted[inv[a]] = a
    """
    flat = np.asarray(ids, dtype=np.int64).reshape(-1)
    R = flat.size
    counts = np.bincount(flat, minlength=E).astype(np.int32)
    offsets = np.zeros(E + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    sorted_ = np.argsort(flat, kind="stable").astype(np.int32)
    inv = np.empty(R, dtype=np.int32)
    inv[sorted_] = np.arange(R, dtype=np.int32)
    return counts, offsets, sorted_, inv


# --------------------------------------------------------------------------
# Stage 3: grouped expert FFN
# --------------------------------------------------------------------------
def silu(g: np.ndarray) -> np.ndarray:
    """SiLU(g) = g / (1 + exp(-g)) in float64."""
    return g / (1.0 + np.exp(-g))


def expert_matrices(wts: dict, d: int, f: int):
    """Dequantised (gate, up, down) of one expert: [f, d], [f, d], [d, f]."""
    w13 = dequant(wts["w13_q"], wts["w13_s"], wts["w13_z"], d)  # [2f, d]
    w2 = dequant(wts["w2_q"], wts["w2_s"], wts["w2_z"], f)      # [d, f]
    return w13[:f], w13[f:], w2


def expert_ffn_rows(X: np.ndarray, wts: dict, d: int, f: int, want_h: bool = False):
    """FFN of one expert on rows X [m, d] (float64).

    G = X Wg^T, U = X Wu^T, H = SiLU(G) * U, Y = H Wd^T, all float64
    (the intermediate H is not rounded).
    """
    wg, wu, wd = expert_matrices(wts, d, f)
    G = X @ wg.T
    U = X @ wu.T
    H = silu(G) * U
    Y = H @ wd.T
    return (Y, H) if want_h else Y


def expert_ffn(x_perm: np.ndarray, offsets: np.ndarray, get_expert, d: int, f: int,
               row_w: np.ndarray | None = None, want_h: bool = False):
    """Grouped FFN over permuted rows: segment e = rows offsets[e]..offsets[e+1].

    get_expert(e) returns the six storage arrays of expert e.  Experts with an
    empty segment are not touched.  Optional row_w scales row i of the output.
    """
    R = x_perm.shape[0]
    E = len(offsets) - 1
    Y = np.zeros((R, d), dtype=np.float64)
    H = np.zeros((R, f), dtype=np.float64) if want_h else None
    for e in range(E):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if b == a:
            continue
        r = expert_ffn_rows(x_perm[a:b], get_expert(e), d, f, want_h=want_h)
        if want_h:
            Y[a:b], H[a:b] = r
        else:
            Y[a:b] = r
    if row_w is not None:
        Y = Y * np.asarray(row_w, dtype=np.float64)[:, None]
    return (Y, H) if want_h else Y


# --------------------------------------------------------------------------
# Stage 4: combine
# --------------------------------------------------------------------------
def combine(y_perm: np.ndarray, inv: np.ndarray, w: np.ndarray, T: int, k: int) -> np.ndarray:
    """out[t] = sum over slots j of w[t, j] * y_perm[inv[t*k + j]] (float64)."""
    d = y_perm.shape[1]
    out = np.zeros((T, d), dtype=np.float64)
    for j in range(k):
        out += w[:, j:j + 1] * y_perm[inv[np.arange(T) * k + j]]
    return out


# --------------------------------------------------------------------------
# Whole layer
# --------------------------------------------------------------------------
def layer_forward(x_bits: np.ndarray, logits: np.ndarray, get_expert, E: int, d: int, f: int,
                  k: int, want_intermediates: bool = False):
    """The layer, stage by stage: route, permute, gather, grouped FFN, combine."""
    T = x_bits.shape[0]
    ids, w = route_topk(logits, k)
    counts, offsets, sorted_, inv = permute(ids, E)
    x = bf16_bits_to_f64(x_bits)
    x_perm = x[sorted_ // k]
    y_perm, h = expert_ffn(x_perm, offsets, get_expert, d, f, want_h=True)
    out = combine(y_perm, inv, w, T, k)
    if want_intermediates:
        return out, dict(ids=ids, w=w, counts=counts, offsets=offsets, sorted=sorted_,
                         inv=inv, h=h, y_perm=y_perm)
    return out


def layer_forward_tokens(x_bits: np.ndarray, logits: np.ndarray, get_expert, E: int, d: int,
                         f: int, k: int, tokens) -> np.ndarray:
    """Output rows of selected tokens only (same definition as layer_forward,
    evaluated for a sample of tokens so that full-size layers stay cheap)."""
    tokens = np.asarray(tokens, dtype=np.int64)
    ids, w = route_topk(logits[tokens], k)
    x = bf16_bits_to_f64(x_bits[tokens])
    out = np.zeros((tokens.size, d), dtype=np.float64)
    for e in np.unique(ids):
        rows, slots = np.nonzero(ids == e)
        y = expert_ffn_rows(x[rows], get_expert(int(e)), d, f)
        out[rows] += w[rows, slots][:, None] * y
    return out
