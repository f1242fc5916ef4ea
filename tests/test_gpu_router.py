"""Router GEMM on the GPU against the oracle, through the C ABI.

Logits: every element within the error bound of an fp32 summation around the
oracle's once-rounded exact sum.  Both kernels are covered: the CUDA-core one
(up to 32 tokens) and the tensor-core one with narrow (32) and wide (192)
expert tiles, with ragged token tiles, ragged expert tiles and K ending in a
partial 64-wide slice.  Routing from the GPU's logits: ids bit-exact against
the oracle's routing of those same logits, and a layer-step that starts with
the router equals, bit for bit, the step fed those logits directly."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import Harness, to_dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import cold_expert_residency_gb300 as moe
    moe.build()


@pytest.fixture(scope="module")
def ctx():
    import cold_expert_residency_gb300 as moe
    c = moe.moe_create(1, 16, 2, 256, 128, 8)
    yield c
    torch.cuda.synchronize()
    assert moe.moe_device_status(c) == moe.MOE_OK
    moe.moe_destroy(c)


def _bound(xb, wb, bias):
    """First-order bound on |fp32 sum - exact| for a sum of H products and
    the bias taken in at most n = H/8 + 16 steps, each rounding (or, in the
    tensor cores' accumulator, truncating) to within two units (2^-23) of the
    running sum of |terms|."""
    H = xb.shape[1]
    S = np.abs(synth.bf16_bits_to_f32(xb).astype(np.float64)) @ \
        np.abs(synth.bf16_bits_to_f32(wb).astype(np.float64)).T
    if bias is not None:
        S += np.abs(bias.astype(np.float64))[None, :]
    n = H // 8 + 16
    return n * 2.0 ** -23 * S


def _run(ctx, xb, wb, bias):
    import cold_expert_residency_gb300 as moe
    T, H = xb.shape
    E = wb.shape[0]
    x = to_dev(xb.view(np.int16))
    w = to_dev(wb.view(np.int16))
    b = None if bias is None else to_dev(bias)
    out = torch.full((T, E), float("nan"), dtype=torch.float32, device="cuda")
    moe.moe_router_logits(ctx, x, w, b, T, E, H, out)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def _check(got, xb, wb, bias):
    ref = oracle.router_logits(xb, wb, bias)
    assert np.all(np.isfinite(got))
    err = np.abs(got.astype(np.float64) - ref.astype(np.float64))
    bound = _bound(xb, wb, bias) + np.abs(ref.astype(np.float64)) * 2.0 ** -24
    bad = np.argwhere(err > bound)
    assert bad.size == 0, f"{len(bad)} logits outside the bound, first {bad[:3].tolist()}"


@pytest.mark.parametrize("T,E,H", [(1, 16, 256), (8, 16, 256), (13, 16, 256), (32, 10, 264),
                                   (7, 384, 4096), (40, 10, 264), (112, 384, 4096), (300, 384, 4096),
                                   (5000, 200, 520)])
def test_router_logits_within_summation_bound(ctx, T, E, H):
    # T <= 32: CUDA cores (13: a ragged token group; E = 10: few CTAs;
    # H = 264: 33 sixteen-byte columns).  T > 32: tensor cores, narrow expert
    # tiles (40 x 10: one tile, zero-filled rows and experts, K = 264 ends in a
    # partial slice; 300: a ragged third token tile), and at 5000 x 200 wide
    # tiles (the second expert tile holds 8 experts)
    cfg = synth.get_config("tiny", E=E, H=H)
    xb = synth.activations(cfg, 0, 0, T=T)
    wb = synth.router_weights(cfg, 0)
    bias = synth.router_bias(cfg, 0)
    _check(_run(ctx, xb, wb, bias), xb, wb, bias)
    _check(_run(ctx, xb, wb, None), xb, wb, None)


def test_router_prefill_sampled_rows(ctx):
    cfg = synth.get_config("prefill")
    xb = synth.activations(cfg, 0, 0)
    wb = synth.router_weights(cfg, 0)
    bias = synth.router_bias(cfg, 0)
    got = _run(ctx, xb, wb, bias)
    rows = np.unique(np.concatenate([[0, cfg.T - 1],
                                     np.random.default_rng(0).choice(cfg.T, 46, replace=False)]))
    _check(got[rows], xb[rows], wb, bias)


def test_step_with_router_equals_step_from_its_logits():
    cfg = synth.get_config("tiny", T=13)
    h = Harness(cfg)
    try:
        wb = synth.router_weights(cfg, 0)
        bias = synth.router_bias(cfg, 0)
        x = synth.activations(cfg, 0, 0)
        T = h.load(np.zeros((cfg.T, cfg.E), np.float32), x)
        h.step.run(0, T, router=(to_dev(wb.view(np.int16)), to_dev(bias)))
        torch.cuda.synchronize()
        b = h.step.buf
        lg = b.logits[:T].cpu().numpy()
        ids = b.ids[:T].cpu().numpy()
        out = b.out[:T].cpu().numpy().view(np.uint16)
        _check(lg, x, wb, bias)
        ids_ref, _ = oracle.route(lg, cfg.k)
        assert np.array_equal(ids, ids_ref)
        direct = h.run(0, lg, x)
        assert np.array_equal(direct["ids"], ids) and np.array_equal(direct["out"], out)
    finally:
        h.close()
