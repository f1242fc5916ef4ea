"""CUDA path vs the CPU oracle, through the C ABI, on seeded inputs.

Bit-exact: routing ids, the residency split (pick lists), the usage table,
the finalize given the same Y and w, split vs unsplit and swapped vs unsplit
outputs.  Tolerance (relative L2 <= 5e-3, max |diff| <= 2e-2 of max |ref|):
the FFN rows Y and the layer output against the oracle."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import Harness, assert_close_bf16, f32

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

IMPLS = [0, 1]   # MOE_FFN_TCGEN05, MOE_FFN_SIMT


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import cold_expert_residency_gb300 as moe
    moe.build()


def _check_routing(h, cfg, res, lg, T, counts_before=None, count_on=True):
    ids_ref, w_ref = oracle.route(lg, cfg.k)
    assert np.array_equal(res["ids"], ids_ref)
    assert np.allclose(res["w"], w_ref, rtol=4e-7, atol=0)
    assert np.all(np.abs(res["w"].astype(np.float64).sum(1) - 1.0) <= 1e-6)
    rm = h.moe.moe_get_rowmap(h.ctx, 0, cfg.E)
    assert np.array_equal(h.moe.moe_read_rowmap_device(h.ctx, 0, cfg.E), rm)
    sp_ref = oracle.split(rm, ids_ref)
    sp = h.split_lists(T)
    for b in range(2):
        for key in ("n_act", "n_picks"):
            assert sp[b][key] == sp_ref[b][key], (b, key)
        for key in ("act_row", "act_off", "picks"):
            assert np.array_equal(sp[b][key], sp_ref[b][key]), (b, key)
    return ids_ref, w_ref


@pytest.mark.parametrize("impl", IMPLS)
def test_tiny_layer_step_matches_oracle(impl):
    cfg = synth.get_config("tiny")
    h = Harness(cfg, impl=impl)
    try:
        lg = synth.router_logits(cfg, 0, 0)
        x = synth.activations(cfg, 0, 0)
        res = h.run(0, lg, x)
        _check_routing(h, cfg, res, lg, cfg.T)
        counts = np.zeros(cfg.E, np.int32)
        ids_ref, w_ref, Y_ref, out_ref = oracle.layer_step(h.weights[0], lg, x, cfg.k, counts=counts)
        got = h.moe.moe_read_counts(h.ctx, 1, cfg.E)[0]
        assert np.array_equal(got, counts)
        assert_close_bf16(res["Y"], Y_ref, "Y")
        assert_close_bf16(res["out"], out_ref, "out")
        # the finalize is bit-exact given the same Y and w
        assert np.array_equal(res["out"], oracle.finalize(res["Y"], res["w"]))
    finally:
        h.close()


@pytest.mark.parametrize("impl", IMPLS)
def test_split_equals_unsplit_bitwise(impl):
    cfg = synth.get_config("tiny")
    w = synth.layer_weights(cfg, 0)
    split = Harness(cfg, weights={0: w}, impl=impl)
    unsplit = Harness(cfg, weights={0: w}, masks={0: np.ones(cfg.E, np.uint8)}, impl=impl)
    try:
        for step in range(3):
            lg = synth.router_logits(cfg, 0, step)
            x = synth.activations(cfg, 0, step)
            a = split.run(0, lg, x)                            # one call over both banks
            b = unsplit.run(0, lg, x)
            c = split.run(0, lg, x, fused=False, split=False)  # one bank after the other
            d = split.run(0, lg, x, fused=False)               # the two banks on two streams
            assert np.array_equal(a["Y"], b["Y"]) and np.array_equal(a["out"], b["out"])
            for r in (c, d):
                assert np.array_equal(a["Y"], r["Y"]) and np.array_equal(a["out"], r["out"])
    finally:
        split.close()
        unsplit.close()


def test_tc_and_simt_agree_within_tolerance():
    cfg = synth.get_config("tiny")
    w = synth.layer_weights(cfg, 0)
    a = Harness(cfg, weights={0: w}, impl=0)
    b = Harness(cfg, weights={0: w}, impl=1)
    try:
        lg = synth.router_logits(cfg, 0, 1)
        x = synth.activations(cfg, 0, 1)
        ra, rb = a.run(0, lg, x), b.run(0, lg, x)
        assert_close_bf16(ra["Y"], rb["Y"], "tc vs simt")
    finally:
        a.close()
        b.close()


@pytest.mark.parametrize("impl", IMPLS)
def test_swaps_bit_identical_and_negative_control(impl):
    cfg = synth.get_config("tiny")
    w = synth.layer_weights(cfg, 0)
    mask = synth.hot_mask(cfg, 0)
    h = Harness(cfg, weights={0: w}, impl=impl)
    ref = Harness(cfg, weights={0: w}, masks={0: np.ones(cfg.E, np.uint8)}, impl=impl)
    try:
        lg = synth.router_logits(cfg, 0, 0)
        x = synth.activations(cfg, 0, 0)
        base = ref.run(0, lg, x)
        cold = [int(e) for e in np.flatnonzero(mask == 0)]
        hot = [int(e) for e in np.flatnonzero(mask == 1)]
        rm = h.moe.moe_get_rowmap(h.ctx, 0, cfg.E).copy()
        for i in range(5):     # five ordered swaps, output checked after each
            pro, dem = cold[i % len(cold)], hot[i]
            n, applied = h.moe.moe_swap_rows(h.ctx, 0, [pro], [dem])
            exp = oracle.swap(rm, [pro], [dem])
            assert applied.tolist() == exp.tolist()
            assert np.array_equal(h.moe.moe_get_rowmap(h.ctx, 0, cfg.E), rm)
            res = h.run(0, lg, x)
            assert np.array_equal(h.moe.moe_read_rowmap_device(h.ctx, 0, cfg.E), rm)
            assert np.array_equal(res["out"], base["out"]) and np.array_equal(res["Y"], base["Y"])
        # a stale pair is refused and changes nothing
        n, applied = h.moe.moe_swap_rows(h.ctx, 0, [hot[-1]], [cold[-1]])
        assert n == 0 and applied.tolist() == [0]
        # bank contents follow the map: a fresh placement with the final map
        # holds the same bytes row for row
        eb = h.moe.moe_expert_bytes(cfg.H, cfg.I)
        fresh = Harness(cfg, weights={0: w}, masks={0: (rm >= 0).astype(np.uint8)}, impl=impl)
        try:
            frm = fresh.moe.moe_get_rowmap(fresh.ctx, 0, cfg.E)
            for e in range(cfg.E):
                bank_a, row_a = (0, rm[e]) if rm[e] >= 0 else (1, -1 - rm[e])
                bank_b, row_b = (0, frm[e]) if frm[e] >= 0 else (1, -1 - frm[e])
                ra = h.moe.moe_read_bank_row(h.ctx, 0, bank_a, int(row_a), eb)
                rb = fresh.moe.moe_read_bank_row(fresh.ctx, 0, bank_b, int(row_b), eb)
                assert np.array_equal(ra, rb), e
        finally:
            fresh.close()
        # negative control: a map that names the other expert's rows (a map
        # flip without the copies) changes the output
        bad = list(w)
        e0, e1 = int(base["ids"][0, 0]), int(base["ids"][0, 1])
        for arr in bad:
            tmp = arr[e0].copy()
            arr[e0] = arr[e1]
            arr[e1] = tmp
        neg = Harness(cfg, weights={0: bad}, impl=impl)
        try:
            r = neg.run(0, lg, x)
            assert not np.array_equal(r["out"], base["out"])
        finally:
            neg.close()
    finally:
        h.close()
        ref.close()


@pytest.mark.parametrize("impl", IMPLS)
def test_restore_round_trip_is_lossless(impl):
    """Wander away from the boot placement with swaps, restore its hot set in
    budgets of three swaps, then check every expert's bank row byte for byte
    against its packing and the output against the all-HBM layer."""
    from cold_expert_residency_gb300.runtime import restore_placement
    cfg = synth.get_config("tiny")
    w = synth.layer_weights(cfg, 0)
    h = Harness(cfg, weights={0: w}, impl=impl)
    ref = Harness(cfg, weights={0: w}, masks={0: np.ones(cfg.E, np.uint8)}, impl=impl)
    try:
        lg = synth.router_logits(cfg, 0, 1)
        x = synth.activations(cfg, 0, 1)
        base = ref.run(0, lg, x)
        boot = h.moe.moe_get_rowmap(h.ctx, 0, cfg.E).copy()
        rng = np.random.default_rng(5)
        rm = boot.copy()
        for _ in range(3):       # three adaptation rounds of up to four swaps each
            pro = rng.permutation(np.flatnonzero(rm < 0))[:4]
            dem = rng.permutation(np.flatnonzero(rm >= 0))[:pro.size]
            n, applied = h.moe.moe_swap_rows(h.ctx, 0, pro, dem)
            assert applied.tolist() == oracle.swap(rm, pro, dem).tolist()
            assert np.array_equal(h.run(0, lg, x)["out"], base["out"])
        away = int(np.count_nonzero((rm >= 0) & (boot < 0)))
        assert away > 0
        total, calls = 0, 0
        while True:
            n = restore_placement(h.ctx, 0, boot, budget=3)
            if n == 0:
                break
            total += n
            calls += 1
            assert np.array_equal(h.run(0, lg, x)["out"], base["out"])
        assert total == away and calls == -(-away // 3)
        rm = h.moe.moe_get_rowmap(h.ctx, 0, cfg.E)
        assert np.array_equal(rm >= 0, boot >= 0)
        assert np.array_equal(h.moe.moe_read_rowmap_device(h.ctx, 0, cfg.E), rm)
        eb = h.moe.moe_expert_bytes(cfg.H, cfg.I)
        for e in range(cfg.E):
            bank, row = (0, rm[e]) if rm[e] >= 0 else (1, -1 - rm[e])
            got = h.moe.moe_read_bank_row(h.ctx, 0, bank, int(row), eb)
            want = h.moe.moe_pack_expert(cfg.H, cfg.I, *(a[e] for a in w))
            assert np.array_equal(got, want), e
        r = h.run(0, lg, x)
        assert np.array_equal(r["out"], base["out"]) and np.array_equal(r["Y"], base["Y"])
    finally:
        h.close()
        ref.close()


def test_workspace_serves_every_smaller_step():
    """A workspace (and a host-buffer step's scratch area) sized for T_max
    serves every step of at most T_max tokens: the size is non-decreasing in T
    although steps of at most 256 tokens hold extra fp32 partial-sum rows that
    larger steps do not."""
    import cold_expert_residency_gb300 as moe
    for name in ("tiny", "decode1"):
        cfg = synth.get_config(name)
        ctx = moe.moe_create(1, cfg.E, cfg.k, cfg.H, cfg.I, 600)
        try:
            sizes = [moe.moe_workspace_bytes(ctx, T) for T in range(0, 601)]
            assert all(b >= a for a, b in zip(sizes, sizes[1:])), name
            # the host-buffer step's scratch area likewise
            sizes = [moe.moe_step_scratch_bytes(ctx, T) for T in range(0, 601)]
            assert all(b >= a for a, b in zip(sizes, sizes[1:])), name
        finally:
            moe.moe_destroy(ctx)


def test_counts_only_for_small_steps_and_when_on():
    cfg = synth.get_config("tiny")
    h = Harness(cfg, T_max=300)
    try:
        x = synth.activations(cfg, 0, 0, T=300)
        lg = synth.router_logits(cfg, 0, 0, T=300)
        h.run(0, lg[:256], x[:256], count_on=True)
        c1 = h.moe.moe_read_counts(h.ctx, 1, cfg.E)[0]
        assert c1.sum() == 256 * cfg.k
        h.run(0, lg[:8], x[:8], count_on=False)
        assert np.array_equal(h.moe.moe_read_counts(h.ctx, 1, cfg.E)[0], c1)
        res = h.run(0, lg, x, count_on=True)          # 300 tokens: not counted
        assert np.array_equal(h.moe.moe_read_counts(h.ctx, 1, cfg.E)[0], c1)
        # the multi-kernel route/split path (T > 256) matches the oracle too
        _check_routing(h, cfg, res, lg, 300)
        ids_ref, w_ref, Y_ref, out_ref = oracle.layer_step(h.weights[0], lg, x, cfg.k)
        assert_close_bf16(res["out"], out_ref, "out T=300")
        h.moe.moe_reset_counts(h.ctx)
        assert h.moe.moe_read_counts(h.ctx, 1, cfg.E).sum() == 0
    finally:
        h.close()


@pytest.mark.parametrize("T", [1, 5, 33, 64, 65, 130])
def test_token_counts_and_ragged_tiles(T):
    """Several N-tile widths (16 / 64 / 256 variants) and ragged token counts."""
    cfg = synth.get_config("tiny", T=T)
    h = Harness(cfg)
    try:
        lg = synth.router_logits(cfg, 0, 3, T=T)
        x = synth.activations(cfg, 0, 3, T=T)
        res = h.run(0, lg, x)
        _check_routing(h, cfg, res, lg, T)
        _, _, Y_ref, out_ref = oracle.layer_step(h.weights[0], lg, x, cfg.k)
        assert_close_bf16(res["Y"], Y_ref, f"Y T={T}")
        assert_close_bf16(res["out"], out_ref, f"out T={T}")
    finally:
        h.close()


@pytest.mark.parametrize("T,impl", [(3, 0), (3, 1), (12, 0), (40, 0), (300, 0)])
def test_half_group_geometry(T, impl):
    """I = 192: the down GEMM's K ends in half a 128-wide K group, which
    M-tiles 2p and 2p+1 share in the device layout.  Every tile width against
    the oracle, and the split banks bit-identical to an all-HBM placement."""
    cfg = synth.get_config("tiny", I=192, T=T)
    w = synth.layer_weights(cfg, 0)
    h = Harness(cfg, weights={0: w}, impl=impl)
    ref = Harness(cfg, weights={0: w}, masks={0: np.ones(cfg.E, np.uint8)}, impl=impl)
    try:
        lg = synth.router_logits(cfg, 0, 5, T=T)
        x = synth.activations(cfg, 0, 5, T=T)
        res = h.run(0, lg, x)
        _check_routing(h, cfg, res, lg, T)
        _, _, Y_ref, out_ref = oracle.layer_step(h.weights[0], lg, x, cfg.k)
        assert_close_bf16(res["Y"], Y_ref, f"Y T={T}")
        assert_close_bf16(res["out"], out_ref, f"out T={T}")
        r2 = ref.run(0, lg, x)
        assert np.array_equal(res["Y"], r2["Y"]) and np.array_equal(res["out"], r2["out"])
    finally:
        h.close()
        ref.close()


def test_all_cold_and_all_hot_banks():
    cfg = synth.get_config("tiny")
    w = synth.layer_weights(cfg, 0)
    lg = synth.router_logits(cfg, 0, 0)
    x = synth.activations(cfg, 0, 0)
    outs = []
    for mask in (np.zeros(cfg.E, np.uint8), np.ones(cfg.E, np.uint8)):
        h = Harness(cfg, weights={0: w}, masks={0: mask})
        try:
            outs.append(h.run(0, lg, x)["out"])
        finally:
            h.close()
    assert np.array_equal(outs[0], outs[1])


def test_empty_step_is_a_no_op():
    """A step of zero tokens routes nothing, counts nothing, writes no row and
    leaves the next step unchanged."""
    cfg = synth.get_config("tiny")
    h = Harness(cfg)
    try:
        lg = synth.router_logits(cfg, 0, 0)
        x = synth.activations(cfg, 0, 0)
        first = h.run(0, lg, x)
        c1 = h.moe.moe_read_counts(h.ctx, 1, cfg.E)
        empty = h.run(0, np.zeros((0, cfg.E), np.float32), np.zeros((0, cfg.H), np.uint16))
        assert empty["ids"].shape == (0, cfg.k) and empty["out"].shape == (0, cfg.H)
        assert np.array_equal(h.moe.moe_read_counts(h.ctx, 1, cfg.E), c1)
        for b in range(2):
            sp = h.moe.moe_read_split(h.ctx, h.step.buf.ws_ptr, 0, cfg.k, b)
            assert sp["n_act"] == 0 and sp["n_picks"] == 0
        again = h.run(0, lg, x)
        assert np.array_equal(again["Y"], first["Y"]) and np.array_equal(again["out"], first["out"])
        assert h.moe.moe_read_counts(h.ctx, 1, cfg.E).sum() == c1.sum() + cfg.T * cfg.k
        assert h.moe.moe_device_status(h.ctx) == 0
    finally:
        h.close()


def test_device_status_clean_after_steps():
    cfg = synth.get_config("tiny")
    h = Harness(cfg)
    try:
        h.run(0, synth.router_logits(cfg, 0, 0), synth.activations(cfg, 0, 0))
        assert h.moe.moe_device_status(h.ctx) == 0
    finally:
        h.close()


@pytest.mark.slow
def test_decode1_full_size_against_oracle():
    """One-user decode step at full geometry (E=384, k=6, H=4096, I=2880,
    T=7, hot 295 / cold 89): every routed row against the oracle."""
    cfg = synth.get_config("decode1")
    h = Harness(cfg)
    try:
        lg = synth.router_logits(cfg, 0, 0)
        x = synth.activations(cfg, 0, 0)
        res = h.run(0, lg, x)
        ids_ref, w_ref = _check_routing(h, cfg, res, lg, cfg.T)
        slots = np.arange(cfg.T * cfg.k, dtype=np.int32)
        Y_ref = oracle.rows_for_slots(h.weights[0], ids_ref, x, slots).reshape(cfg.T, cfg.k, cfg.H)
        assert_close_bf16(res["Y"], Y_ref, "Y decode1")
        out_ref = oracle.finalize(Y_ref, w_ref)
        assert_close_bf16(res["out"], out_ref, "out decode1")
        assert np.array_equal(res["out"], oracle.finalize(res["Y"], res["w"]))
        sp = h.split_lists(cfg.T)
        assert sp[1]["n_picks"] > 0, "decode step should touch the cold bank"
    finally:
        h.close()


@pytest.mark.parametrize("T", [7, 40, 300])
def test_host_buffer_step_equals_the_device_calls(T):
    """moe_layer_step_host (host logits and hidden states in, host output rows
    out) gives the same bits as the device calls it stands for, at 8-, 32- and
    prefill-sized tiles, on a split layer; a scratch area sized for the
    largest step serves a smaller one; T = 0 is a no-op."""
    cfg = synth.get_config("tiny", T=T)
    h = Harness(cfg, T_max=300)
    moe = h.moe
    try:
        lg = synth.router_logits(cfg, 0, 11, T=T)
        x = synth.activations(cfg, 0, 11, T=T)
        ref = h.run(0, lg, x)
        scratch = torch.empty(moe.moe_step_scratch_bytes(h.ctx, 300) + 256, dtype=torch.uint8, device="cuda")
        sp = (scratch.data_ptr() + 255) // 256 * 256
        h_lg = torch.from_numpy(np.ascontiguousarray(lg)).pin_memory()
        h_x = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).pin_memory()
        h_out = torch.full((T, cfg.H), -1, dtype=torch.int16).pin_memory()
        moe.moe_layer_step_host(h.ctx, 0, h_lg, h_x, T, True, h_out, sp)
        torch.cuda.synchronize()
        assert np.array_equal(h_out.numpy().view(np.uint16), ref["out"])
        moe.moe_layer_step_host(h.ctx, 0, h_lg, h_x, 0, True, h_out, sp)   # T = 0: nothing changes
        torch.cuda.synchronize()
        assert np.array_equal(h_out.numpy().view(np.uint16), ref["out"])
        assert moe.moe_device_status(h.ctx) == 0
    finally:
        h.close()
