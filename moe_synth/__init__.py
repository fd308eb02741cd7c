"""Seeded synthetic inputs for the routed W4A16 MoE layer.

This module is the ONLY code shared by the CUDA path's callers (tests, bench)
and the CPU oracle.  It draws random numbers and stores them in the layer's
storage formats; it holds none of the layer's arithmetic (no dequantisation,
no routing, no matmul).  Every array it returns is plain numpy.

Workloads (shapes follow the MoE models that the "bloomery" performance page
and the "Measured results" page of vllm-omni describe; the weight format is
their W4A16 group-128 scheme, 4.25 bits/weight):

  tiny     T=8    d=256  f=512  E=8   k=2   logits N(0,1)
  decode   T=2    d=2048 f=768  E=128 k=8   logits N(0,1), 48 layers
  prefill  T=512  d=2048 f=768  E=128 k=8   logits N(0,1) + per-expert bias N(0,0.5)
  skew     T=4096 d=2048 f=768  E=128 k=8   Zipf(1.1) expert popularity (Gumbel-top-k)
  large_decode  T=2   d=7168 f=2048 E=256 k=8   logits N(0,1)
  large_prefill T=512 d=7168 f=2048 E=256 k=8   logits N(0,1)

Storage (all little-endian):
  w13_q [E][2f][d/8]  uint32  int4 codes, 8 per word, low nibble = lowest k;
                              rows 0..f-1 are the gate projection, f..2f-1 up
  w13_s, w13_z [E][2f][d/128] uint16 = IEEE fp16 bit patterns (scale, zero)
  w2_q  [E][d][f/8]   uint32  down projection, same packing along f
  w2_s, w2_z   [E][d][f/128]  uint16 fp16 bits
  x      [T][d]  uint16 bf16 bit patterns (N(0,1) rounded to nearest even)
  logits [T][E]  float32

Random streams: numpy PCG64 seeded by SeedSequence([seed, cfg_id, layer,
expert, tag]) so each expert's matrices can be regenerated alone.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np

GROUP = 128
ZERO_FP16_BITS = np.uint16(0x4800)  # fp16 8.0: the zero point of every group

# stream tags
_T_W13Q, _T_W13S, _T_W2Q, _T_W2S = 0, 1, 2, 3
_T_X, _T_LOGITS, _T_BIAS, _T_PERM, _T_GUMBEL = 10, 11, 12, 13, 14


@dataclass(frozen=True)
class Config:
    name: str
    cfg_id: int
    T: int
    d: int
    f: int
    E: int
    k: int
    layers: int = 1
    logits: str = "normal"  # "normal" | "biased" | "zipf"
    seed: int = 0

    @property
    def R(self) -> int:
        return self.T * self.k

    def expert_weight_bytes(self) -> int:
        """Packed codes + fp16 scale + fp16 zero of one expert (3 matrices)."""
        n = 3 * self.d * self.f
        return n // 2 + 2 * 2 * (n // GROUP)


CONFIGS = {
    "tiny": Config("tiny", 0, T=8, d=256, f=512, E=8, k=2),
    "decode": Config("decode", 1, T=2, d=2048, f=768, E=128, k=8, layers=48),
    "prefill": Config("prefill", 2, T=512, d=2048, f=768, E=128, k=8, logits="biased"),
    "skew": Config("skew", 3, T=4096, d=2048, f=768, E=128, k=8, logits="zipf"),
    "large_decode": Config("large_decode", 4, T=2, d=7168, f=2048, E=256, k=8),
    "large_prefill": Config("large_prefill", 4, T=512, d=7168, f=2048, E=256, k=8),
}


def custom(name: str, T: int, d: int, f: int, E: int, k: int, logits: str = "normal",
           layers: int = 1, seed: int = 0, cfg_id: int = 99) -> Config:
    """A workload outside the named set (used for edge-case tests)."""
    return Config(name, cfg_id, T=T, d=d, f=f, E=E, k=k, layers=layers, logits=logits, seed=seed)


def _rng(cfg: Config, layer: int, expert: int, tag: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([cfg.seed, cfg.cfg_id, layer, expert, tag]))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns uint16 bits."""
    b = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return b.astype(np.uint16)


def _scales(rng: np.random.Generator, shape) -> np.ndarray:
    s = rng.uniform(0.002, 0.02, size=shape).astype(np.float16)
    return s.view(np.uint16)


def expert_weights(cfg: Config, layer: int, e: int) -> dict:
    """All six arrays of expert `e` of `layer` (no leading E axis)."""
    d, f = cfg.d, cfg.f
    w13_q = _rng(cfg, layer, e, _T_W13Q).integers(0, 2**32, size=(2 * f, d // 8), dtype=np.uint32)
    w13_s = _scales(_rng(cfg, layer, e, _T_W13S), (2 * f, d // GROUP))
    w2_q = _rng(cfg, layer, e, _T_W2Q).integers(0, 2**32, size=(d, f // 8), dtype=np.uint32)
    w2_s = _scales(_rng(cfg, layer, e, _T_W2S), (d, f // GROUP))
    return {
        "w13_q": w13_q,
        "w13_s": w13_s,
        "w13_z": np.full_like(w13_s, ZERO_FP16_BITS),
        "w2_q": w2_q,
        "w2_s": w2_s,
        "w2_z": np.full_like(w2_s, ZERO_FP16_BITS),
    }


def layer_weights(cfg: Config, layer: int, threads: int | None = None) -> dict:
    """Stacked [E, ...] arrays of one layer, generated expert by expert."""
    d, f, E = cfg.d, cfg.f, cfg.E
    out = {
        "w13_q": np.empty((E, 2 * f, d // 8), np.uint32),
        "w13_s": np.empty((E, 2 * f, d // GROUP), np.uint16),
        "w13_z": np.empty((E, 2 * f, d // GROUP), np.uint16),
        "w2_q": np.empty((E, d, f // 8), np.uint32),
        "w2_s": np.empty((E, d, f // GROUP), np.uint16),
        "w2_z": np.empty((E, d, f // GROUP), np.uint16),
    }

    def fill(e):
        w = expert_weights(cfg, layer, e)
        for key, v in w.items():
            out[key][e] = v

    threads = threads or min(32, os.cpu_count() or 1)
    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(fill, range(E)))
    return out


def activations(cfg: Config, layer: int = 0) -> np.ndarray:
    """x [T, d] as bf16 bits: N(0,1) in float32 rounded to nearest-even bf16."""
    x = _rng(cfg, layer, 0, _T_X).standard_normal((cfg.T, cfg.d), dtype=np.float32)
    return f32_to_bf16_bits(x)


def zipf_probabilities(E: int, s: float = 1.1, zero_tail: int = 8) -> np.ndarray:
    """Expert popularity by rank: p_r proportional to r^-s, the last `zero_tail` ranks 0."""
    r = np.arange(1, E + 1, dtype=np.float64)
    p = r ** (-s)
    if zero_tail:
        p[E - zero_tail:] = 0.0
    return p / p.sum()


def router_logits(cfg: Config, layer: int = 0) -> np.ndarray:
    """Router logits [T, E] float32 for the workload's distribution."""
    T, E = cfg.T, cfg.E
    if cfg.logits == "normal":
        return _rng(cfg, layer, 0, _T_LOGITS).standard_normal((T, E), dtype=np.float32)
    if cfg.logits == "biased":
        z = _rng(cfg, layer, 0, _T_LOGITS).standard_normal((T, E), dtype=np.float32)
        bias = _rng(cfg, layer, 0, _T_BIAS).normal(0.0, 0.5, size=E).astype(np.float32)
        return (z + bias[None, :]).astype(np.float32)
    if cfg.logits == "zipf":
        # Gumbel-top-k: the k largest of log p + Gumbel(0,1) are k draws without
        # replacement with probability proportional to p.  Experts of rank with
        # p = 0 get a very negative logit and are never chosen.
        p = zipf_probabilities(E)
        perm = _rng(cfg, layer, 0, _T_PERM).permutation(E)  # rank of expert e is perm[e]
        g = _rng(cfg, layer, 0, _T_GUMBEL).gumbel(0.0, 1.0, size=(T, E))
        pe = p[perm]
        with np.errstate(divide="ignore"):
            lp = np.where(pe > 0, np.log(np.where(pe > 0, pe, 1.0)), -1e4)
        out = np.where(pe[None, :] > 0, lp[None, :] + g, -1e4)
        return out.astype(np.float32)
    raise ValueError(cfg.logits)

