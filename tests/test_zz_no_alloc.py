"""The allocation-free FFN entry point (moe_expert_ffn_bank_static).

It exists for callers that may not allocate device memory (a plugin with a
fixed memory budget, a serving loop that must not call cudaMalloc).  Its rows
must match the workspace-based entry point's, on two calls in a row (the
static scratch area keeps the previous call's contents), and a step too big
for the area must be refused.  Kept in a file of its own that runs last."""
import numpy as np
import pytest

import synth
from gpu_util import assert_close_bf16

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import cold_expert_residency_gb300 as m
    m.build()
    return m


def _routed(moe, cfg, T_max):
    from cold_expert_residency_gb300.runtime import StepBuffers
    ctx = moe.moe_create(cfg.L, cfg.E, cfg.k, cfg.H, cfg.I, T_max)
    moe.moe_init_banks(ctx, 0, *synth.layer_weights(cfg, 0), synth.hot_mask(cfg, 0))
    buf = StepBuffers(ctx, cfg.E, cfg.k, cfg.H, T_max)
    return ctx, buf


@pytest.mark.parametrize("name", ["tiny", "decode1"])
def test_static_scratch_matches_workspace_path_twice(moe, name):
    cfg = synth.get_config(name)
    ctx, buf = _routed(moe, cfg, cfg.T)
    try:
        T = cfg.T
        for step in range(2):   # two calls in a row share the static area
            buf.logits[:T].copy_(torch.from_numpy(synth.router_logits(cfg, 0, step)))
            buf.x[:T].copy_(torch.from_numpy(synth.activations(cfg, 0, step).view(np.int16)))
            moe.moe_route_split_count(ctx, 0, buf.logits, T, True, buf.ids, buf.w, buf.ws_ptr)
            Y_ref = torch.zeros_like(buf.Y)
            Y_new = torch.full_like(buf.Y, 0x7FC0)          # bf16 NaN: every routed row must be written
            for bank in (moe.MOE_BANK_HOT, moe.MOE_BANK_COLD):
                moe.moe_expert_ffn_bank(ctx, 0, bank, buf.x, T, buf.ws_ptr, Y_ref)
            for bank in (moe.MOE_BANK_HOT, moe.MOE_BANK_COLD):
                moe.moe_expert_ffn_bank_static(ctx, 0, bank, buf.x, T, buf.ws_ptr, Y_new)
            torch.cuda.synchronize()
            a = Y_new[:T].cpu().numpy().view(np.uint16)
            b = Y_ref[:T].cpu().numpy().view(np.uint16)
            assert_close_bf16(a, b, f"{name} call {step}")
        assert moe.moe_device_status(ctx) == 0
    finally:
        torch.cuda.synchronize()
        moe.moe_destroy(ctx)


def test_static_scratch_refuses_oversized_steps(moe):
    cfg = synth.get_config("tiny")
    T = 8192                       # T*k*(2H + 6I) is well past the 16 MiB area
    ctx = moe.moe_create(1, cfg.E, cfg.k, cfg.H, cfg.I, T)
    try:
        moe.moe_init_banks(ctx, 0, *synth.layer_weights(cfg, 0), synth.hot_mask(cfg, 0))
        with pytest.raises(moe.MoeError) as ei:   # refused before any device work
            moe.moe_expert_ffn_bank_static(ctx, 0, moe.MOE_BANK_HOT, 16, T, 256, 16)
        assert ei.value.code == moe.MOE_EINVAL and "static area" in str(ei.value)
    finally:
        moe.moe_destroy(ctx)
