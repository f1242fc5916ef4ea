"""Full-size workloads on the GPU against the oracle.

- adaptive residency under a domain shift: 128 decode steps, counts read every
  16 steps, the native policy's swaps applied between steps; every step's
  output is bitwise equal to an all-HBM (unsplit) layer, the policy takes the
  oracle policy's decisions on the GPU's counts, and counts and row maps match
  the oracle's bookkeeping exactly;
- 16-stream decode (112 tokens, 32-token tiles) on a split layer and an
  all-HBM layer: routing/split bit-exact, every expert row within tolerance;
- prefill (8192 tokens, the multi-kernel routing path, no counting): routing
  and split bit-exact; within tolerance, the first and last pick of every
  token tile of every expert (so every (expert, tile) unit of both GEMMs and
  every ragged tile end is checked)."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import Harness, assert_close_bf16, assert_rows_close_bf16, tile_edge_slots

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import cold_expert_residency_gb300 as moe
    moe.build()


def _check_split(h, layer, ids, T):
    rm = h.moe.moe_get_rowmap(h.ctx, layer, h.cfg.E)
    assert np.array_equal(h.moe.moe_read_rowmap_device(h.ctx, layer, h.cfg.E), rm)
    ref = oracle.split(rm, ids)
    got = h.split_lists(T)
    for b in range(2):
        for key in ("act_row", "act_off", "picks"):
            assert np.array_equal(got[b][key], ref[b][key]), (layer, b, key)


def test_adaptive_domain_shift_swaps_are_bit_identical():
    cfg = synth.get_config("adaptive")
    ex = cfg.extra
    w = synth.layer_weights(cfg, 0)
    split = Harness(cfg, weights={0: w})
    unsplit = Harness(cfg, weights={0: w}, masks={0: np.ones(cfg.E, np.uint8)})
    moe = split.moe
    try:
        params = dict(read_every=ex["read_every"], half_life=ex["half_life"], hysteresis=ex["hysteresis"],
                      min_avg=ex["min_avg"], max_pairs=ex["max_per_read"])
        nat = moe.moe_policy(cfg.E, **params)
        ref = oracle.Policy(cfg.E, **params)
        rm = moe.moe_get_rowmap(split.ctx, 0, cfg.E).copy()
        counts_ref = np.zeros(cfg.E, np.int32)
        swaps, cold_picks = 0, []
        for step in range(cfg.steps):
            lg = synth.router_logits(cfg, 0, step)
            x = synth.activations(cfg, 0, step)
            a = split.run(0, lg, x)
            b = unsplit.run(0, lg, x, count_on=False)
            assert np.array_equal(a["out"], b["out"]), step
            assert np.array_equal(a["Y"], b["Y"]), step
            ids_ref, _ = oracle.route(lg, cfg.k)
            assert np.array_equal(a["ids"], ids_ref), step
            oracle.count(counts_ref, ids_ref, True, 256)
            cold_picks.append(int((rm[a["ids"]] < 0).sum()))
            if (step + 1) % ex["read_every"] == 0:
                counts = moe.moe_read_counts(split.ctx, 1, cfg.E)[0]
                assert np.array_equal(counts, counts_ref), step
                pro_n, dem_n = nat.read(counts, rm)
                pro_r, dem_r = ref.read(counts, rm)
                assert np.array_equal(pro_n, pro_r) and np.array_equal(dem_n, dem_r), step
                for i in range(0, len(pro_n), ex["max_per_step"]):
                    n, applied = moe.moe_swap_rows(split.ctx, 0, pro_n[i:i + 8], dem_n[i:i + 8])
                    exp = oracle.swap(rm, pro_n[i:i + 8], dem_n[i:i + 8])
                    assert applied.tolist() == exp.tolist()
                    swaps += n
                assert np.array_equal(moe.moe_get_rowmap(split.ctx, 0, cfg.E), rm)
        assert swaps > 0, "the domain shift should trigger swaps"
        # adaptation moves the new domain's experts in: fewer cold picks at the end
        late = np.mean(cold_picks[-16:])
        just_after = np.mean(cold_picks[cfg.shift_at:cfg.shift_at + 16])
        assert late <= just_after
        assert moe.moe_device_status(split.ctx) == 0
    finally:
        split.close()
        unsplit.close()


def _rows(h, layer, x, res, slots):
    """The GPU's expert rows of `slots` against the oracle's: within tolerance
    over the rows together and in every row."""
    ref = oracle.rows_for_slots(h.weights[layer], res["ids"], x, slots)
    got = res["Y"].reshape(-1, h.cfg.H)[slots]
    assert_close_bf16(got, ref, f"layer {layer}: {slots.size} rows")
    assert_rows_close_bf16(got, ref, f"layer {layer}: {slots.size} rows")


def test_decode16_split_and_hbm_layers():
    cfg = synth.get_config("decode16")
    h = Harness(cfg, layers=2)          # layer 0 split 295/89, layer 1 all-HBM
    try:
        for layer in (0, 1):
            lg = synth.router_logits(cfg, layer, 0)
            x = synth.activations(cfg, layer, 0)
            res = h.run(layer, lg, x)
            ids_ref, w_ref = oracle.route(lg, cfg.k)
            assert np.array_equal(res["ids"], ids_ref)
            _check_split(h, layer, ids_ref, cfg.T)
            _rows(h, layer, x, res, np.arange(cfg.T * cfg.k, dtype=np.int32))    # every row
            assert np.array_equal(res["out"], oracle.finalize(res["Y"], res["w"]))
        counts = h.moe.moe_read_counts(h.ctx, 2, cfg.E)
        assert counts.sum(axis=1).tolist() == [cfg.T * cfg.k] * 2
    finally:
        h.close()


def test_prefill_chunk_every_tile_end():
    cfg = synth.get_config("prefill")
    h = Harness(cfg)
    try:
        lg = synth.router_logits(cfg, 0, 0)
        x = synth.activations(cfg, 0, 0)
        res = h.run(0, lg, x, count_on=True)
        ids_ref, w_ref = oracle.route(lg, cfg.k)
        assert np.array_equal(res["ids"], ids_ref)
        assert np.allclose(res["w"], w_ref, rtol=4e-7, atol=0)
        _check_split(h, 0, ids_ref, cfg.T)
        assert h.moe.moe_read_counts(h.ctx, 1, cfg.E).sum() == 0      # 8192 tokens > 256: not counted
        # both formats' tile widths: two-piece rows 144 tokens, MXFP8 rows 160
        _rows(h, 0, x, res, tile_edge_slots(res["ids"], (144, 160)))
        # finalize bit-exact on a slice of tokens
        assert np.array_equal(res["out"][:64], oracle.finalize(res["Y"][:64], res["w"][:64]))
    finally:
        h.close()
