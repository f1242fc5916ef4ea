"""Routing at its edge cases, through the C ABI, bit-exact against the oracle.

- Tied logits: values drawn from {0, 1, 2, 3} with +0.0 and -0.0 mixed, so
  most picks are decided by the tie rule (lower expert id first); ids, the
  residency split lists and the usage table must equal the oracle's.
- NaN logits, which the routing reads as -infinity: every id stays a valid
  expert id and equals the oracle's.
- The usage counter inside a captured CUDA graph ("We Built the Counter",
  section 5, "Is it still the same model?"): after N replays with fresh
  inputs the table equals the sum of the oracle's N histograms, and every
  replayed output equals the eager step's bit for bit.
Both routing paths run: one CTA for steps of at most 32 tokens, three
kernels beyond."""
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


def _wide_cfg(T):
    """384 experts, top-6 (the decode routing shape) with small experts."""
    return synth.get_config("tiny", E=384, k=6, n_hot=295, beta=0.35, T=T)


def _check_route_split_count(h, res, lg, T, counts_before):
    cfg = h.cfg
    ids_ref, w_ref = oracle.route(lg, cfg.k)
    assert np.array_equal(res["ids"], ids_ref)
    # host and device expf may differ in the last ulp; NaN weights must match NaN
    np.testing.assert_allclose(res["w"], w_ref, rtol=4e-7, atol=0, equal_nan=True)
    assert np.all((res["ids"] >= 0) & (res["ids"] < cfg.E))
    rm = h.moe.moe_get_rowmap(h.ctx, 0, cfg.E)
    sp_ref = oracle.split(rm, ids_ref)
    sp = h.split_lists(T)
    for b in range(2):
        for key in ("n_act", "n_picks"):
            assert sp[b][key] == sp_ref[b][key], (b, key)
        for key in ("act_row", "act_off", "picks"):
            assert np.array_equal(sp[b][key], sp_ref[b][key]), (b, key)
    counts = counts_before.copy()
    oracle.count(counts, ids_ref, True, 256)
    assert np.array_equal(h.moe.moe_read_counts(h.ctx, 1, cfg.E)[0], counts)
    return counts


@pytest.mark.parametrize("T", [7, 40, 300])
def test_tied_logits_bit_exact(T):
    cfg = _wide_cfg(T)
    h = Harness(cfg)
    try:
        rng = np.random.default_rng(100 + T)
        counts = np.zeros(cfg.E, np.int32)
        for step in range(2):
            lg = rng.integers(0, 4, size=(T, cfg.E)).astype(np.float32)
            zero = lg == 0
            lg[zero & (rng.random(lg.shape) < 0.5)] = np.float32(-0.0)
            if step == 1:
                lg[:, ::5] = 3.0            # many ties at the top value
            x = synth.activations(cfg, 0, step, T=T)
            res = h.run(0, lg, x)
            counts = _check_route_split_count(h, res, lg, T, counts)
            np.testing.assert_array_equal(res["out"], oracle.finalize(res["Y"], res["w"]))
    finally:
        h.close()


@pytest.mark.parametrize("T", [7, 300])
def test_nan_logits_route_to_valid_ids(T):
    cfg = _wide_cfg(T)
    h = Harness(cfg)
    try:
        rng = np.random.default_rng(7 + T)
        lg = synth.router_logits(cfg, 0, 0, T=T).copy()
        lg[rng.random(lg.shape) < 0.3] = np.nan      # NaN sprinkled through every row
        lg[1, :] = np.nan                            # one row of NaN only: ids 0..k-1, weights NaN
        lg[2, : cfg.E - 3] = np.nan                  # fewer finite logits than k
        x = synth.activations(cfg, 0, 0, T=T)
        res = h.run(0, lg, x)
        _check_route_split_count(h, res, lg, T, np.zeros(cfg.E, np.int32))
        assert res["ids"][1].tolist() == list(range(cfg.k))
        assert h.moe.moe_device_status(h.ctx) == 0
    finally:
        h.close()


@pytest.mark.parametrize("T", [8, 300])
def test_counter_inside_captured_graph(T):
    cfg = synth.get_config("tiny", T=T)
    h = Harness(cfg)
    N = 5
    try:
        b = h.step.buf
        inputs = [(synth.router_logits(cfg, 0, s, T=T), synth.activations(cfg, 0, s, T=T)) for s in range(N)]
        eager = [h.run(0, lg, x) for lg, x in inputs]
        h.moe.moe_reset_counts(h.ctx)
        torch.cuda.synchronize()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph, stream=side):
                h.step.run(0, T)
        torch.cuda.synchronize()
        assert h.moe.moe_read_counts(h.ctx, 1, cfg.E).sum() == 0      # capture runs nothing
        expect = np.zeros(cfg.E, np.int32)
        for (lg, x), ref in zip(inputs, eager):
            h.load(lg, x)
            graph.replay()
            torch.cuda.synchronize()
            assert np.array_equal(b.ids[:T].cpu().numpy(), ref["ids"])
            assert np.array_equal(b.out[:T].cpu().numpy().view(np.uint16), ref["out"])
            oracle.count(expect, oracle.route(lg, cfg.k)[0], True, 256)
        got = h.moe.moe_read_counts(h.ctx, 1, cfg.E)[0]
        assert np.array_equal(got, expect)
        assert got.sum() == (N * T * cfg.k if T <= 256 else 0)
    finally:
        h.close()
