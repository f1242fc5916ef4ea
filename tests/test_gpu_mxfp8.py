"""The opt-in MXFP8 activation format of prefill-sized steps
(moe_set_act_format(MOE_ACT_MXFP8)), through the C ABI.

Token rows and h rows become OCP MXFP8 (32-element blocks sharing an e8m0
scale, e4m3 elements) and each product takes one block-scaled MMA instead of
two.  Checked against:
- the oracle's MXFP8 reading of the same layer (expert_ffn_mx8): relative L2
  <= 5e-3 in every row and <= 2e-3 over the tensor -- the GPU and the oracle
  quantize x identically; only fp32 accumulation order and, rarely, an h
  value that rounds to a neighbouring e4m3 code separate them;
- the exact oracle, with the format's own stated tolerance: relative L2
  <= 8e-2 and max |diff| <= 0.15 max |ref| (e4m3 keeps 3 mantissa bits: about
  2.7% RMS per element, on x and again on h; the model of this arithmetic
  gives 4.7-5.7% per row);
- the layer's invariants: split equals unsplit bit for bit, one-bank calls
  equal the call over both banks, and decode-sized steps ignore the format."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import Harness, assert_rows_close_bf16, f32

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

MX_REL_EXACT = 8e-2
MX_MAX_EXACT = 0.15


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import cold_expert_residency_gb300 as moe
    moe.build()


def _harness(cfg, **kw):
    h = Harness(cfg, **kw)
    h.moe.moe_set_act_format(h.ctx, h.moe.MOE_ACT_MXFP8)
    return h


def _vs_exact(got, ref, what):
    g, r = f32(got), f32(ref)
    rel = float(np.linalg.norm(g - r) / np.linalg.norm(r))
    mx = float(np.abs(g - r).max() / np.abs(r).max())
    assert rel <= MX_REL_EXACT and mx <= MX_MAX_EXACT, f"{what}: rel_l2={rel:.3g} max={mx:.3g}"
    return rel


def _vs_mx8(got, ref, what):
    assert_rows_close_bf16(got, ref, what)
    g, r = f32(got), f32(ref)
    rel = float(np.linalg.norm(g - r) / np.linalg.norm(r))
    assert rel <= 2e-3, f"{what}: rel_l2={rel:.3g}"


@pytest.mark.parametrize("T", [300, 2048])
def test_mxfp8_rows_against_both_oracles(T):
    cfg = synth.get_config("tiny", T=T)
    h = _harness(cfg)
    try:
        lg = synth.router_logits(cfg, 0, 1, T=T)
        x = synth.activations(cfg, 0, 1, T=T)
        res = h.run(0, lg, x)
        ids_ref, w_ref = oracle.route(lg, cfg.k)
        assert np.array_equal(res["ids"], ids_ref)
        slots = np.arange(T * cfg.k, dtype=np.int32)
        Y_mx = oracle.rows_for_slots(h.weights[0], ids_ref, x, slots, mx8=True)
        Y_ex = oracle.rows_for_slots(h.weights[0], ids_ref, x, slots)
        got = res["Y"].reshape(-1, cfg.H)
        _vs_mx8(got, Y_mx, f"T={T} vs MXFP8 oracle")
        _vs_exact(got, Y_ex, f"T={T} vs exact oracle")
        _vs_exact(res["out"], oracle.finalize(Y_ex.reshape(T, cfg.k, cfg.H), w_ref), f"T={T} out vs exact")
        assert np.array_equal(res["out"], oracle.finalize(res["Y"], res["w"]))
        assert h.moe.moe_device_status(h.ctx) == 0
    finally:
        h.close()


def test_mxfp8_split_unsplit_and_bank_calls_bitwise():
    cfg = synth.get_config("tiny", T=300)
    w = synth.layer_weights(cfg, 0)
    split = _harness(cfg, weights={0: w})
    unsplit = _harness(cfg, weights={0: w}, masks={0: np.ones(cfg.E, np.uint8)})
    try:
        for step in range(2):
            lg = synth.router_logits(cfg, 0, step, T=300)
            x = synth.activations(cfg, 0, step, T=300)
            a = split.run(0, lg, x)
            b = unsplit.run(0, lg, x)
            c = split.run(0, lg, x, fused=False)               # two streams
            d = split.run(0, lg, x, fused=False, split=False)  # one bank after the other
            for r in (b, c, d):
                assert np.array_equal(a["Y"], r["Y"]) and np.array_equal(a["out"], r["out"])
    finally:
        split.close()
        unsplit.close()


def test_decode_sized_steps_ignore_the_format():
    cfg = synth.get_config("tiny", T=40)
    w = synth.layer_weights(cfg, 0)
    mx = _harness(cfg, weights={0: w})
    two = Harness(cfg, weights={0: w})
    try:
        lg = synth.router_logits(cfg, 0, 2, T=40)
        x = synth.activations(cfg, 0, 2, T=40)
        a, b = mx.run(0, lg, x), two.run(0, lg, x)
        assert np.array_equal(a["Y"], b["Y"])
    finally:
        mx.close()
        two.close()


@pytest.mark.slow
def test_mxfp8_prefill_chunk_sampled():
    """The 8192-token prefill chunk (all 384 experts in HBM): sampled rows
    against both oracles."""
    cfg = synth.get_config("prefill")
    h = _harness(cfg)
    try:
        lg = synth.router_logits(cfg, 0, 0)
        x = synth.activations(cfg, 0, 0)
        res = h.run(0, lg, x, count_on=False)
        ids_ref, _ = oracle.route(lg, cfg.k)
        assert np.array_equal(res["ids"], ids_ref)
        rng = np.random.default_rng(1)
        slots = np.sort(rng.choice(cfg.T * cfg.k, size=24, replace=False)).astype(np.int32)
        got = res["Y"].reshape(-1, cfg.H)[slots]
        _vs_mx8(got, oracle.rows_for_slots(h.weights[0], ids_ref, x, slots, mx8=True), "prefill vs MXFP8 oracle")
        _vs_exact(got, oracle.rows_for_slots(h.weights[0], ids_ref, x, slots), "prefill vs exact oracle")
    finally:
        h.close()
