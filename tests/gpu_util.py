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
