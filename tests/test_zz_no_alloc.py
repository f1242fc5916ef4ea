"""The allocation-free FFN entry point (moe_expert_ffn_bank_static).

It exists for callers that may not allocate device memory (a plugin with a
fixed memory budget, a serving loop that must not call cudaMalloc).  It runs
the same kernels on the same inputs as the workspace-based entry point, so
its rows must equal that entry point's bit for bit, on two calls in a row
(the static scratch area keeps the previous call's contents), at every
decode tile width that fits the area; one call is also checked against the
oracle; a step too big for the area must be refused.  Kept in a file of its
own that runs last."""
import numpy as np
import pytest

import oracle
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


def _routed(moe, cfg, T_max, weights):
    from cold_expert_residency_gb300.runtime import StepBuffers
    ctx = moe.moe_create(cfg.L, cfg.E, cfg.k, cfg.H, cfg.I, T_max)
    moe.moe_init_banks(ctx, 0, *weights, synth.hot_mask(cfg, 0))
    buf = StepBuffers(ctx, cfg.E, cfg.k, cfg.H, T_max)
    return ctx, buf


# (config, tokens): tiny at the 8- and 32-token tiles; the decode geometry
# (H=4096, I=2880; 48 experts) at the 8-, 16- and 32-token tiles, the last
# one with 24 tokens (144 picks, about 9 MB of scratch)
CASES = [("tiny", 8), ("tiny", 40), ("decode1", 7), ("decode1", 12), ("decode1", 24)]


@pytest.mark.parametrize("name,T", CASES)
def test_static_scratch_matches_workspace_path_twice(moe, name, T):
    cfg = synth.get_config(name, T=T) if name == "tiny" else synth.get_config(name, T=T, E=48, n_hot=37)
    weights = synth.layer_weights(cfg, 0)
    ctx, buf = _routed(moe, cfg, T, weights)
    try:
        for step in range(2):   # two calls in a row share the static area
            lg = synth.router_logits(cfg, 0, step)
            x = synth.activations(cfg, 0, step)
            buf.logits[:T].copy_(torch.from_numpy(lg))
            buf.x[:T].copy_(torch.from_numpy(x.view(np.int16)))
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
            assert np.array_equal(a, b), f"{name} T={T} call {step}: rows differ from the workspace path"
            if step == 0:
                ids = buf.ids[:T].cpu().numpy()
                slots = np.arange(0, T * cfg.k, max(1, T * cfg.k // 12), dtype=np.int32)
                ref = oracle.rows_for_slots(weights, ids, x, slots)
                assert_close_bf16(a.reshape(-1, cfg.H)[slots], ref, f"{name} T={T} vs oracle")
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
