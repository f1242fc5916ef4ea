"""Shared set-up for the GPU tests: contexts, banks and layer-steps on seeded
inputs, plus the comparison rules.  Inputs come from ``synth``; expected
values come from ``oracle`` only."""
from __future__ import annotations

import numpy as np

import synth

try:
    import torch
except ImportError:       # pragma: no cover
    torch = None

# FFN output tolerance (bf16): relative L2 <= 5e-3 and max |diff| <= 2e-2
# measured in units of the largest |reference| value of the compared tensor
# (raw outputs are O(1e5), where one bf16 ulp already exceeds 2e-2).
REL_L2 = 5e-3
MAX_REL = 2e-2


def f32(bits):
    return synth.bf16_bits_to_f32(np.asarray(bits).view(np.uint16)).astype(np.float64)


def close_bf16(got_bits, ref_bits):
    g, r = f32(got_bits), f32(ref_bits)
    rel_l2 = float(np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30))
    max_rel = float(np.abs(g - r).max() / max(np.abs(r).max(), 1e-30))
    return rel_l2, max_rel


def assert_close_bf16(got_bits, ref_bits, what=""):
    rel_l2, max_rel = close_bf16(got_bits, ref_bits)
    assert np.all(np.isfinite(f32(got_bits))), f"{what}: non-finite output"
    assert rel_l2 <= REL_L2 and max_rel <= MAX_REL, f"{what}: rel_l2={rel_l2:.3g} max_rel={max_rel:.3g}"
    return rel_l2, max_rel


def assert_rows_close_bf16(got_bits, ref_bits, what="", rel=REL_L2):
    """Relative L2 <= rel in every row (last axis) with a nonzero reference:
    a wrong K block or a wrong token in one row cannot hide in the norm of
    the whole tensor."""
    g = f32(got_bits).reshape(-1, np.asarray(got_bits).shape[-1])
    r = f32(ref_bits).reshape(g.shape)
    nr = np.linalg.norm(r, axis=1)
    err = np.linalg.norm(g - r, axis=1)
    ok = nr > 0
    worst = float((err[ok] / nr[ok]).max()) if ok.any() else 0.0
    assert np.all(err[~ok] == 0), f"{what}: rows with a zero reference differ"
    assert worst <= rel, f"{what}: worst row rel_l2={worst:.3g}"
    return worst


def tile_edge_slots(ids, widths):
    """Slots s = t*k + j of the first and last pick of each token tile of
    each expert: an expert's picks in slot order (the order of its bank
    list), cut into tiles of each width in `widths` (the FFN's token tiles).
    Rows at these slots exercise every (expert, token tile) unit of both
    GEMMs and every tile's first and last token row."""
    flat = np.asarray(ids).reshape(-1)
    order = np.argsort(flat, kind="stable")          # grouped by expert, slot order within
    e_sorted = flat[order]
    starts = np.flatnonzero(np.r_[True, e_sorted[1:] != e_sorted[:-1]])
    ends = np.r_[starts[1:], flat.size]
    sel = set()
    for a, b in zip(starts.tolist(), ends.tolist()):
        for W in widths:
            for t0 in range(a, b, W):
                sel.add(int(order[t0]))
                sel.add(int(order[min(t0 + W, b) - 1]))
    return np.array(sorted(sel), np.int32)


def bf16_ulp(v):
    """Spacing of bf16 numbers at |v| (8 significant bits)."""
    a = np.maximum(np.abs(np.asarray(v, np.float64)), 2.0 ** -126)
    return np.exp2(np.floor(np.log2(a)) - 7)


def ffn_error_bound(weights, e, x_bits):
    """Per-element bound on |Y_gpu - Y_oracle| for one pick (expert e of the
    stacked logical weights, token row x_bits), from the CUDA path's
    arithmetic:
      - a row v carried as two e4m3 pieces after a power-of-two scaling that
        puts max|v| in (224, 448]: |dv| <= 2^-8 |v| + 2^-14 * max|v| / 224
        (e4m3 has 3 mantissa bits; the second piece holds 16x the first's
        error; subnormal pieces leave at most 2^-14 of the scaled unit);
      - fp32 accumulation of exact products: at most K * 2^-24 of sum |W||v|;
      - SwiGLU: |d silu/dz| <= 1.1, and a few fp32 ulps for exp and divide;
      - both sides round y to bf16: one bf16 ulp.
    First order in the errors, widened by 1.25 for the second-order terms."""
    import oracle
    w13_q, w13_s, w2_q, w2_s = (np.asarray(a[e]) for a in weights)
    I2, H = w13_q.shape[0], w13_q.shape[1] * 2
    I = I2 // 2
    W13 = oracle.dequant(w13_q, w13_s)
    W2 = oracle.dequant(w2_q, w2_s)
    x = f32(x_bits).reshape(H)
    ax = np.abs(x)
    floor_x = 2.0 ** -14 * ax.max() / 224.0
    A13 = np.abs(W13)
    S = A13 @ ax
    R = A13.sum(axis=1)
    B13 = (2.0 ** -8 + H * 2.0 ** -24) * S + floor_x * R
    gu = W13 @ x
    g, u = gu[:I], gu[I:]
    Bg, Bu = B13[:I], B13[I:]
    sg = g / (1.0 + np.exp(-np.clip(g, -700, 700)))
    h = sg * u
    Bh = 1.1 * Bg * (np.abs(u) + Bu) + np.abs(sg) * Bu + 2.0 ** -20 * np.abs(h)
    hm = np.abs(h) + Bh
    Bh_rep = Bh + 2.0 ** -8 * hm + 2.0 ** -14 * hm.max() / 224.0
    A2 = np.abs(W2)
    By = A2 @ Bh_rep + I * 2.0 ** -24 * (A2 @ hm)
    y = W2 @ h
    return 1.25 * By + bf16_ulp(np.abs(y) + By)


def assert_within_elem_bound(got_bits, ref_bits, bound, what=""):
    g, r = f32(got_bits).ravel(), f32(ref_bits).ravel()
    d = np.abs(g - r)
    b = np.asarray(bound, np.float64).ravel()
    bad = np.flatnonzero(~(d <= b))
    assert bad.size == 0, (f"{what}: {bad.size} elements over their bound; first at {bad[0]}: "
                           f"|d|={d[bad[0]]:.4g} bound={b[bad[0]]:.4g}")
    return float((d / b).max())


def to_dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.cuda()


class Harness:
    """A context for one config with banks placed from the config's hot mask
    (or an explicit mask), and a LayerStep to run steps."""

    def __init__(self, cfg, T_max=None, layers=None, masks=None, weights=None, impl=None):
        import cold_expert_residency_gb300 as moe
        from cold_expert_residency_gb300.runtime import LayerStep
        self.moe = moe
        self.cfg = cfg
        self.L = cfg.L if layers is None else layers
        self.T_max = cfg.T if T_max is None else T_max
        self.ctx = moe.moe_create(self.L, cfg.E, cfg.k, cfg.H, cfg.I, self.T_max)
        if impl is not None:
            moe.moe_set_ffn_impl(self.ctx, impl)
        self.weights = {}
        for l in range(self.L):
            w = weights[l] if weights is not None else synth.layer_weights(cfg, l)
            self.weights[l] = w
            mask = masks[l] if masks is not None else synth.hot_mask(cfg, l)
            moe.moe_init_banks(self.ctx, l, *w, mask)
        self.step = LayerStep(self.ctx, cfg.E, cfg.k, cfg.H, self.T_max)

    def load(self, logits, x):
        T = logits.shape[0]
        b = self.step.buf
        b.logits[:T].copy_(torch.from_numpy(np.ascontiguousarray(logits)))
        b.x[:T].copy_(torch.from_numpy(np.ascontiguousarray(x).view(np.int16)))
        return T

    def run(self, layer, logits, x, count_on=True, split=True, fused=True):
        T = self.load(logits, x)
        self.step.run(layer, T, count_on=count_on, split=split, fused=fused)
        torch.cuda.synchronize()
        b = self.step.buf
        return dict(ids=b.ids[:T].cpu().numpy(), w=b.w[:T].cpu().numpy(),
                    Y=b.Y[:T].cpu().numpy().view(np.uint16), out=b.out[:T].cpu().numpy().view(np.uint16))

    def split_lists(self, T):
        return [self.moe.moe_read_split(self.ctx, self.step.buf.ws_ptr, T, self.cfg.k, b) for b in (0, 1)]

    def close(self):
        if self.ctx:
            torch.cuda.synchronize()
            self.moe.moe_destroy(self.ctx)
            self.ctx = None
