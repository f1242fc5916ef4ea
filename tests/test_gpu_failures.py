"""Failure handling on the GPU, in forms that never fault, trap or hang it.

- A bounded wait that runs out: the host asks the next FFN call to withhold
  one K group's copies in one CTA (moe_inject_fault) and shortens the wait
  bound to a few milliseconds.  Every role of that CTA must give up, let its
  issued copies land, free its tensor memory and return; the call ends, the
  status word reads MOE_ETIMEOUT, and the next step (default bound) equals a
  clean step bit for bit.  Each FFN kernel is covered: 8- and 32-token decode
  tiles and the 144-token prefill tile, over both banks and one bank.
- Allocation failures ("a host-memory floor instead of an out-of-memory
  kill"): with MOE_INJECT_ALLOC_FAIL naming an allocation site,
  moe_init_banks returns MOE_ENOMEM, leaves the layer unplaced and holds no
  more device or pinned memory than before; placing the layer again works.
- Repeatability (race detection without a sanitizer): the same step ten
  times gives the same bits every time."""
import os
import time

import numpy as np
import pytest

import synth
from gpu_util import Harness

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import cold_expert_residency_gb300 as moe
    moe.build()


@pytest.mark.parametrize("T,fused", [(8, True), (40, True), (300, True), (8, False), (300, False)])
def test_withheld_copy_times_out_and_next_step_is_clean(T, fused):
    cfg = synth.get_config("tiny", T=T)
    h = Harness(cfg)
    moe = h.moe
    try:
        lg = synth.router_logits(cfg, 0, 1, T=T)
        x = synth.activations(cfg, 0, 1, T=T)
        clean = h.run(0, lg, x, fused=fused)
        assert moe.moe_device_status(h.ctx) == 0
        moe.moe_set_wait_limit(h.ctx, 5_000_000)            # 5 ms
        moe.moe_inject_fault(h.ctx, moe.MOE_FAULT_WITHHOLD_COPY)
        t0 = time.perf_counter()
        h.run(0, lg, x, fused=fused)
        dt = time.perf_counter() - t0
        assert moe.moe_device_status(h.ctx) == moe.MOE_ETIMEOUT
        assert dt < 5.0, f"the timed-out call took {dt:.2f} s"
        moe.moe_set_wait_limit(h.ctx, 0)                    # back to the default bound
        again = h.run(0, lg, x, fused=fused)
        assert moe.moe_device_status(h.ctx) == 0
        assert np.array_equal(again["Y"], clean["Y"]) and np.array_equal(again["out"], clean["out"])
        # an injection not yet consumed can be withdrawn
        moe.moe_inject_fault(h.ctx, moe.MOE_FAULT_WITHHOLD_COPY)
        moe.moe_inject_fault(h.ctx, moe.MOE_FAULT_NONE)
        third = h.run(0, lg, x, fused=fused)
        assert moe.moe_device_status(h.ctx) == 0
        assert np.array_equal(third["out"], clean["out"])
    finally:
        h.close()


def _mem(moe):
    torch.cuda.synchronize()
    return moe.moe_memory_in_use(), torch.cuda.mem_get_info()[0]


@pytest.mark.parametrize("site", ["cold_bank", "hot_bank", "rowmap", "init_staging"])
def test_alloc_failure_in_placement_leaves_nothing(site):
    """Decode geometry with 16 experts (12 hot, 4 cold: about 300 MB), so a
    leaked bank would show in the device's free memory too."""
    import cold_expert_residency_gb300 as moe
    cfg = synth.get_config("decode1", E=16, n_hot=12)
    w = synth.layer_weights(cfg, 0)
    mask = synth.hot_mask(cfg, 0)
    ctx = moe.moe_create(1, cfg.E, cfg.k, cfg.H, cfg.I, cfg.T)
    try:
        lib0, free0 = _mem(moe)
        os.environ["MOE_INJECT_ALLOC_FAIL"] = site
        try:
            with pytest.raises(moe.MoeError) as ei:
                moe.moe_init_banks(ctx, 0, *w, mask)
        finally:
            del os.environ["MOE_INJECT_ALLOC_FAIL"]
        assert ei.value.code == moe.MOE_ENOMEM
        lib1, free1 = _mem(moe)
        assert lib1 == lib0
        assert abs(free1 - free0) < (8 << 20)
        with pytest.raises(moe.MoeError) as ei:
            moe.moe_bank_rows(ctx, 0)
        assert ei.value.code == moe.MOE_ESTATE
        # placed again without the injection: the layer works and a second
        # failed placement frees the first one's banks too
        moe.moe_init_banks(ctx, 0, *w, mask)
        assert moe.moe_bank_rows(ctx, 0) == (12, 4)
        lib2, _ = _mem(moe)
        assert lib2[0] > lib0[0] and lib2[1] > lib0[1]
        os.environ["MOE_INJECT_ALLOC_FAIL"] = site
        try:
            with pytest.raises(moe.MoeError):
                moe.moe_init_banks(ctx, 0, *w, mask)
        finally:
            del os.environ["MOE_INJECT_ALLOC_FAIL"]
        assert _mem(moe)[0] == lib0
    finally:
        moe.moe_destroy(ctx)


@pytest.mark.parametrize("site", ["create_counts", "create_status"])
def test_alloc_failure_in_create_leaves_nothing(site):
    """The first and the last of the context's allocations (the last one
    fails after the usage table and the swap staging row exist)."""
    import cold_expert_residency_gb300 as moe
    cfg = synth.get_config("decode1")
    lib0, _ = _mem(moe)
    os.environ["MOE_INJECT_ALLOC_FAIL"] = site
    try:
        with pytest.raises(moe.MoeError) as ei:
            moe.moe_create(1, cfg.E, cfg.k, cfg.H, cfg.I, cfg.T)
    finally:
        del os.environ["MOE_INJECT_ALLOC_FAIL"]
    assert ei.value.code == moe.MOE_ENOMEM
    assert _mem(moe)[0] == lib0


@pytest.mark.parametrize("T", [8, 40, 300])
def test_same_step_ten_times_same_bits(T):
    cfg = synth.get_config("tiny", T=T)
    h = Harness(cfg)
    try:
        lg = synth.router_logits(cfg, 0, 6, T=T)
        x = synth.activations(cfg, 0, 6, T=T)
        first = h.run(0, lg, x)
        for _ in range(9):
            r = h.run(0, lg, x)
            for key in ("ids", "w", "Y", "out"):
                assert np.array_equal(r[key], first[key]), key
    finally:
        h.close()
