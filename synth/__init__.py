"""Seeded synthetic inputs for the split-residency MoE layer.

This module is shared by the CUDA-path tests/bench and by the CPU oracle's
tests.  It draws inputs only: MXFP4 expert weights in the logical layout,
bf16 activations, fp32 router logits, per-layer Zipf rankings and the hot/cold
placement derived from them.  It holds none of the layer's arithmetic (no
dequantisation, routing, FFN or combine).

Generators
----------
* Bytes: SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014) in counter mode, ``out_i = mix64(key + (i+1)*gamma)``.
  Counter mode makes every tensor's stream independent of how it is split
  across threads, so generation can use all host cores.
* Normals: Box-Muller on two 53-bit uniforms from the same stream, rounded to
  fp32 (and from fp32 to bf16 with round-to-nearest-even for activations).

Workloads (the write-ups' decode and prefill shapes; see ``CONFIGS``)
--------------------------------------------------------------------
* e2m1 nibbles uniform over all 16 codes; e8m0 block-scale bytes uniform over
  123..127, i.e. scales 2^-4 .. 2^0, one per 32 contiguous K elements.
* activations: bf16(N(0,1)).
* logits: fp32(N(0,1) + bias_e), with bias_e = beta * ln p_rank(e) for a
  Zipf(s) popularity law over a seeded per-layer ranking of the experts
  (the write-ups measure the top-25% of experts taking ~71% of decode picks).
* router weights (for the router GEMM that produces logits from hidden
  states): bf16(N(0,1)/sqrt(H)) [E][H], with the same per-expert bias.
* hot bank: the ``n_hot`` experts with the best Zipf rank; cold bank: the rest.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field, replace

import numpy as np

__all__ = [
    "Config", "CONFIGS", "get_config", "stream_u64", "stream_bytes",
    "expert_weights", "layer_weights", "activations", "router_logits", "router_weights", "router_bias",
    "zipf_ranks", "zipf_bias", "hot_mask", "shifted_ranks", "spearman",
    "bf16_bits_to_f32", "expert_bytes",
]

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


@dataclass(frozen=True)
class Config:
    """One workload.  Sizes follow the MoE-layer notation of the write-ups:
    E routed experts, top-k routing, hidden size H, expert intermediate size I,
    T tokens per layer-step, L MoE layers."""
    name: str
    L: int
    E: int
    k: int
    H: int
    I: int
    T: int
    n_hot: int                      # experts per layer in the HBM bank
    zipf_s: float = 0.0             # 0 => no bias (near-uniform routing)
    beta: float = 0.0               # bias scale on ln p_rank
    scale_lo: int = 123             # e8m0 byte range (inclusive)
    scale_hi: int = 127
    # "unit-scale" variants: subtracted from every W13 / W2 scale byte, so
    # the layer's outputs are O(1) (0 = the drawn bytes as they are)
    w13_scale_shift: int = 0
    w2_scale_shift: int = 0
    hbm_layers: tuple = ()          # layers kept all-HBM regardless of n_hot
    steps: int = 1
    shift_at: int = -1              # step at which the Zipf ranking is re-drawn
    shift_rho: float = 0.0          # correlation knob of the re-drawn ranking
    count_on: bool = True
    seed: int = 0
    extra: dict = field(default_factory=dict)


# beta = 0.35 puts ~70% of the top-6 picks on the top 25% of experts at E=384
# (measured by tests/test_synth.py); the write-ups' histogram shows 71.4%.
_BETA = 0.35

CONFIGS = {
    # 1 layer, 16 experts, top-2, H=256, I=128, 8 tokens; hot = 12, cold = 4.
    "tiny": Config("tiny", L=1, E=16, k=2, H=256, I=128, T=8, n_hot=12,
                   zipf_s=1.1, beta=1.0),
    # one-user decode step (7-token speculative verify window), 1 layer.
    "decode1": Config("decode1", L=1, E=384, k=6, H=4096, I=2880, T=7,
                      n_hot=295, zipf_s=1.1, beta=_BETA),
    # 16 streams x 7 tokens, 4 layers; odd layers all-HBM, even layers split.
    "decode16": Config("decode16", L=4, E=384, k=6, H=4096, I=2880, T=112,
                       n_hot=295, zipf_s=1.1, beta=_BETA, hbm_layers=(1, 3),
                       steps=200),
    # 128 decode steps, ranking re-drawn at step 64 (Spearman ~0.15).  The
    # printed defaults pair a minimum average of 8 with reads every 64 steps;
    # this workload reads every 16 steps, so its minimum is the same rate per
    # read: 8 * 16 / 64 = 2 picks.
    "adaptive": Config("adaptive", L=1, E=384, k=6, H=4096, I=2880, T=7,
                       n_hot=295, zipf_s=1.1, beta=_BETA, steps=128,
                       shift_at=64, shift_rho=0.115,
                       extra=dict(read_every=16, half_life=500.0, max_per_read=8,
                                  max_per_step=8, hysteresis=1.5, min_avg=2.0)),
    # prefill chunk: 8192 tokens, all experts in HBM, no bias, no counting.
    "prefill": Config("prefill", L=1, E=384, k=6, H=4096, I=2880, T=8192,
                      n_hot=384, zipf_s=0.0, beta=0.0, count_on=False),
}


def get_config(name: str, **over) -> Config:
    cfg = CONFIGS[name]
    return replace(cfg, **over) if over else cfg


def expert_bytes(H: int, I: int) -> int:
    """Bytes of one MXFP4 expert: W13 [2I x H] and W2 [H x I] at 4 bits per
    element plus one e8m0 byte per 32 elements."""
    n = 2 * I * H + H * I
    return n // 2 + n // 32


# --------------------------------------------------------------------------
# counter-mode SplitMix64
# --------------------------------------------------------------------------

def _mix(z: np.ndarray) -> np.ndarray:
    z = z ^ (z >> np.uint64(30))
    z = z * _M1
    z = z ^ (z >> np.uint64(27))
    z = z * _M2
    return z ^ (z >> np.uint64(31))


def _key(*parts) -> np.uint64:
    """Fold integers/strings into one 64-bit stream key."""
    h = np.uint64(0x243F6A8885A308D3)
    with np.errstate(over="ignore"):
        for p in parts:
            if isinstance(p, str):
                v = 0
                for ch in p.encode():
                    v = (v * 131 + ch) & 0xFFFFFFFFFFFFFFFF
            else:
                v = int(p) & 0xFFFFFFFFFFFFFFFF
            h = _mix(np.array([h ^ np.uint64(v)], dtype=np.uint64) + _GAMMA)[0]
    return h


def _u64_block(key: np.uint64, start: int, n: int) -> np.ndarray:
    with np.errstate(over="ignore"):
        c = np.arange(start + 1, start + n + 1, dtype=np.uint64) * _GAMMA + key
        return _mix(c)


_POOL = None


def _pool():
    global _POOL
    if _POOL is None:
        _POOL = ThreadPoolExecutor(max(1, min(32, os.cpu_count() or 1)))
    return _POOL


def stream_u64(key: np.uint64, n: int) -> np.ndarray:
    """n 64-bit outputs of the counter-mode stream keyed by ``key``."""
    chunk = 1 << 22
    if n <= chunk:
        return _u64_block(key, 0, n)
    out = np.empty(n, dtype=np.uint64)

    def fill(s):
        e = min(n, s + chunk)
        out[s:e] = _u64_block(key, s, e - s)

    list(_pool().map(fill, range(0, n, chunk)))
    return out


def stream_bytes(key: np.uint64, n: int) -> np.ndarray:
    words = stream_u64(key, (n + 7) // 8)
    return words.astype("<u8", copy=False).view(np.uint8)[:n]


def _uniform01(key, n):
    """53-bit uniforms in (0, 1]."""
    r = stream_u64(key, n)
    return ((r >> np.uint64(11)).astype(np.float64) + 1.0) * (1.0 / 9007199254740992.0)


def _normal(key, n) -> np.ndarray:
    """Box-Muller: z = sqrt(-2 ln u1) cos(2 pi u2), in float64."""
    u = _uniform01(key, 2 * n)
    u1, u2 = u[0::2], u[1::2]
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)


def _f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit pattern, round to nearest even (inputs are finite)."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# --------------------------------------------------------------------------
# weights
# --------------------------------------------------------------------------

def _scales(key, n, lo, hi):
    b = stream_bytes(key, n).astype(np.uint16)
    span = hi - lo + 1
    return (lo + ((b * span) >> 8)).astype(np.uint8)


def expert_weights(cfg: Config, layer: int, expert: int, seed: int | None = None):
    """(w13_q [2I][H/2], w13_s [2I][H/32], w2_q [H][I/2], w2_s [H][I/32]) uint8.

    Logical MXFP4 layout: byte b of a row packs K elements 2b (low nibble) and
    2b+1 (high nibble); rows 0..I-1 of W13 are the gate projection and rows
    I..2I-1 the up projection; scales run along K in blocks of 32."""
    s = cfg.seed if seed is None else seed
    H, I = cfg.H, cfg.I
    w13_q = stream_bytes(_key(s, "w13q", layer, expert), 2 * I * H // 2).reshape(2 * I, H // 2)
    w13_s = _scales(_key(s, "w13s", layer, expert), 2 * I * H // 32, cfg.scale_lo, cfg.scale_hi).reshape(2 * I, H // 32)
    w2_q = stream_bytes(_key(s, "w2q", layer, expert), H * I // 2).reshape(H, I // 2)
    w2_s = _scales(_key(s, "w2s", layer, expert), H * I // 32, cfg.scale_lo, cfg.scale_hi).reshape(H, I // 32)
    if cfg.w13_scale_shift:
        w13_s = (w13_s.astype(np.int16) - cfg.w13_scale_shift).astype(np.uint8)
    if cfg.w2_scale_shift:
        w2_s = (w2_s.astype(np.int16) - cfg.w2_scale_shift).astype(np.uint8)
    return w13_q, w13_s, w2_q, w2_s


def layer_weights(cfg: Config, layer: int, seed: int | None = None, experts=None):
    """Stacked [E, ...] logical arrays for one layer (all experts unless a
    subset of expert ids is given)."""
    ids = range(cfg.E) if experts is None else list(experts)
    H, I = cfg.H, cfg.I
    n = len(ids)
    w13_q = np.empty((n, 2 * I, H // 2), np.uint8)
    w13_s = np.empty((n, 2 * I, H // 32), np.uint8)
    w2_q = np.empty((n, H, I // 2), np.uint8)
    w2_s = np.empty((n, H, I // 32), np.uint8)
    for i, e in enumerate(ids):
        a, b, c, d = expert_weights(cfg, layer, e, seed)
        w13_q[i], w13_s[i], w2_q[i], w2_s[i] = a, b, c, d
    return w13_q, w13_s, w2_q, w2_s


# --------------------------------------------------------------------------
# activations and router logits
# --------------------------------------------------------------------------

def activations(cfg: Config, layer: int = 0, step: int = 0, T: int | None = None,
                seed: int | None = None) -> np.ndarray:
    """bf16(N(0,1)) activations [T][H] as uint16 bit patterns."""
    s = cfg.seed if seed is None else seed
    T = cfg.T if T is None else T
    z = _normal(_key(s, "x", layer, step), T * cfg.H).astype(np.float32)
    return _f32_to_bf16_bits(z).reshape(T, cfg.H)


def zipf_ranks(cfg: Config, layer: int, phase: int = 0, seed: int | None = None) -> np.ndarray:
    """rank[e] in 1..E: a seeded permutation giving each expert its popularity
    rank (1 = most popular)."""
    s = cfg.seed if seed is None else seed
    keys = stream_u64(_key(s, "rank", layer, phase), cfg.E)
    order = np.argsort(keys, kind="stable")
    rank = np.empty(cfg.E, np.int64)
    rank[order] = np.arange(1, cfg.E + 1)
    return rank


def shifted_ranks(cfg: Config, layer: int, base_rank: np.ndarray, seed: int | None = None) -> np.ndarray:
    """Re-drawn ranking with a weak rank correlation to ``base_rank``:
    z_e = rho * std(rank_e) + sqrt(1 - rho^2) * N(0,1); new rank = rank of z."""
    s = cfg.seed if seed is None else seed
    r = base_rank.astype(np.float64)
    zr = (r - r.mean()) / r.std()
    noise = _normal(_key(s, "shift", layer), cfg.E)
    rho = cfg.shift_rho
    z = rho * zr + math.sqrt(1.0 - rho * rho) * noise
    order = np.argsort(z, kind="stable")
    rank = np.empty(cfg.E, np.int64)
    rank[order] = np.arange(1, cfg.E + 1)
    return rank


def spearman(a: np.ndarray, b: np.ndarray) -> float:
    """Spearman rank correlation of two rankings without ties."""
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    n = a.size
    d = a - b
    return 1.0 - 6.0 * float(np.sum(d * d)) / (n * (n * n - 1.0))


def zipf_bias(cfg: Config, rank: np.ndarray) -> np.ndarray:
    """bias_e = beta * ln p_rank(e), p_r proportional to r^-s (0 if no skew)."""
    if cfg.zipf_s == 0.0 or cfg.beta == 0.0:
        return np.zeros(cfg.E, np.float64)
    r = np.arange(1, cfg.E + 1, dtype=np.float64)
    p = r ** (-cfg.zipf_s)
    p /= p.sum()
    return cfg.beta * np.log(p[rank - 1])


def _step_bias(cfg: Config, layer: int, step: int, s: int) -> np.ndarray:
    rank = zipf_ranks(cfg, layer, 0, s)
    if cfg.shift_at >= 0 and step >= cfg.shift_at:
        rank = shifted_ranks(cfg, layer, rank, s)
    return zipf_bias(cfg, rank)


def router_logits(cfg: Config, layer: int = 0, step: int = 0, T: int | None = None,
                  seed: int | None = None) -> np.ndarray:
    """fp32 logits [T][E] = N(0,1) + bias_e (bias from the layer's Zipf
    ranking, re-drawn at ``cfg.shift_at`` when set)."""
    s = cfg.seed if seed is None else seed
    T = cfg.T if T is None else T
    bias = _step_bias(cfg, layer, step, s)
    z = _normal(_key(s, "logit", layer, step), T * cfg.E).reshape(T, cfg.E)
    return (z + bias[None, :]).astype(np.float32)


def router_weights(cfg: Config, layer: int = 0, seed: int | None = None) -> np.ndarray:
    """bf16(N(0,1) / sqrt(H)) router weights [E][H] as uint16 bit patterns.
    With bf16(N(0,1)) activations each score is then about N(0,1), the same
    law as ``router_logits`` before its bias."""
    s = cfg.seed if seed is None else seed
    z = _normal(_key(s, "router", layer), cfg.E * cfg.H) / math.sqrt(cfg.H)
    return _f32_to_bf16_bits(z.astype(np.float32)).reshape(cfg.E, cfg.H)


def router_bias(cfg: Config, layer: int = 0, step: int = 0, seed: int | None = None) -> np.ndarray:
    """fp32 per-expert router bias [E]: the layer's Zipf bias (as in
    ``router_logits``)."""
    s = cfg.seed if seed is None else seed
    return _step_bias(cfg, layer, step, s).astype(np.float32)


def hot_mask(cfg: Config, layer: int, seed: int | None = None) -> np.ndarray:
    """uint8[E]: 1 for the n_hot best-ranked experts (HBM bank), 0 for the
    cold bank; all ones for layers kept all-HBM."""
    if layer in cfg.hbm_layers or cfg.n_hot >= cfg.E:
        return np.ones(cfg.E, np.uint8)
    rank = zipf_ranks(cfg, layer, 0, seed)
    return (rank <= cfg.n_hot).astype(np.uint8)
