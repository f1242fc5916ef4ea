"""Big-batch cold staging (moe_set_cold_staging), through the C ABI.

The cold bank here holds the most popular experts (a placement right after a
domain shift), so a step routes more picks to some cold experts than one
token tile holds.  With a staging pool those rows are copied once into HBM
and read from there.  Checked:
- the rows of Y and the layer output are bit-identical to the unstaged step
  and to an all-HBM placement, for 32-token and prefill-sized tiles, both
  activation formats, one call over both banks and two calls on two streams;
- the device picks the rows the rule names: cold active rows with more picks
  than one tile, most picks first, ties to the lower row, at most the pool's
  slots (computed here from the oracle's split lists);
- a pool smaller than the candidates stages only the first of them, still
  bitwise equal."""
import numpy as np
import pytest

import oracle
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


def _popular_cold(cfg):
    """Hot mask with the 4 best-ranked experts in the cold bank."""
    rank = synth.zipf_ranks(cfg, 0)
    return (rank > 4).astype(np.uint8)


def _expected_stage(h, lg, T, slots, fmt=0):
    cfg = h.cfg
    ids, _ = oracle.route(lg, cfg.k)
    rm = h.moe.moe_get_rowmap(h.ctx, 0, cfg.E)
    cold = oracle.split(rm, ids)[1]
    W = 8 if T <= 8 else 16 if T <= 16 else 32 if T <= 256 else (160 if fmt else 144)
    n = np.diff(cold["act_off"])
    cand = [(-int(c), a) for a, c in enumerate(n) if c > W]
    cand.sort()
    rows = [int(cold["act_row"][a]) for _, a in cand[:slots]]
    return rows + [-1] * (64 - len(rows)), len(cand)


@pytest.mark.parametrize("T,fmt", [(100, 0), (2048, 0), (2048, 1)])
def test_staged_rows_are_bit_identical(T, fmt):
    cfg = synth.get_config("tiny", T=T)
    w = synth.layer_weights(cfg, 0)
    mask = _popular_cold(cfg)
    staged = Harness(cfg, weights={0: w}, masks={0: mask})
    plain = Harness(cfg, weights={0: w}, masks={0: mask})
    hbm = Harness(cfg, weights={0: w}, masks={0: np.ones(cfg.E, np.uint8)})
    moe = staged.moe
    try:
        for h in (staged, plain, hbm):
            moe.moe_set_act_format(h.ctx, fmt)
        moe.moe_set_cold_staging(staged.ctx, 8)
        lg = synth.router_logits(cfg, 0, 3, T=T)
        x = synth.activations(cfg, 0, 3, T=T)
        a = staged.run(0, lg, x)
        exp_rows, n_cand = _expected_stage(staged, lg, T, 8, fmt)
        assert n_cand > 0, "the workload should route several tiles to a cold expert"
        got_rows = moe.moe_read_stage(staged.ctx, staged.step.buf.ws_ptr, T)
        assert got_rows.tolist() == exp_rows
        b = plain.run(0, lg, x)
        c = hbm.run(0, lg, x)
        d = staged.run(0, lg, x, fused=False)      # the two banks' calls on two streams
        for r in (b, c, d):
            assert np.array_equal(a["Y"], r["Y"]) and np.array_equal(a["out"], r["out"])
        assert moe.moe_device_status(staged.ctx) == 0
    finally:
        staged.close()
        plain.close()
        hbm.close()


def test_pool_smaller_than_the_candidates():
    T = 2048
    cfg = synth.get_config("tiny", T=T)
    w = synth.layer_weights(cfg, 0)
    mask = _popular_cold(cfg)
    staged = Harness(cfg, weights={0: w}, masks={0: mask})
    plain = Harness(cfg, weights={0: w}, masks={0: mask})
    try:
        staged.moe.moe_set_cold_staging(staged.ctx, 1)
        lg = synth.router_logits(cfg, 0, 5, T=T)
        x = synth.activations(cfg, 0, 5, T=T)
        a = staged.run(0, lg, x)
        exp_rows, n_cand = _expected_stage(staged, lg, T, 1)
        assert n_cand >= 2
        assert staged.moe.moe_read_stage(staged.ctx, staged.step.buf.ws_ptr, T).tolist() == exp_rows
        b = plain.run(0, lg, x)
        assert np.array_equal(a["Y"], b["Y"]) and np.array_equal(a["out"], b["out"])
        # turning staging off again gives the same rows too
        staged.moe.moe_set_cold_staging(staged.ctx, 0)
        c = staged.run(0, lg, x)
        assert np.array_equal(a["out"], c["out"])
    finally:
        staged.close()
        plain.close()


def test_staging_arguments():
    import cold_expert_residency_gb300 as moe
    cfg = synth.get_config("tiny")
    h = Harness(cfg)
    try:
        for bad in (-1, 65):
            with pytest.raises(moe.MoeError) as ei:
                moe.moe_set_cold_staging(h.ctx, bad)
            assert ei.value.code == moe.MOE_EINVAL
        d0, _ = moe.moe_memory_in_use()
        moe.moe_set_cold_staging(h.ctx, 4)
        d1, _ = moe.moe_memory_in_use()
        assert d1 - d0 == 4 * moe.moe_expert_bytes(cfg.H, cfg.I)
        moe.moe_set_cold_staging(h.ctx, 0)
        assert moe.moe_memory_in_use()[0] == d0
    finally:
        h.close()
