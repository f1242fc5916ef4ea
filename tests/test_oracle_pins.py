"""Pins of the CPU oracle against values fixed by the pages and by mathematics
(not against itself): hand-decoded MXFP4 codes, the printed byte model, exact
rational arithmetic for the fma finalize, brute-force dense evaluation of all
experts, a textbook dense SwiGLU special case, and invariants of routing,
split, counting, swaps and the policy.  CPU only."""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth
from conftest import load_golden

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ------------------------------------------------------------------ helpers

def golden_e2m1():
    return {int(r[1], 16): float(r[5]) for r in load_golden("mxfp4_codes.txt") if r[0] == "e2m1"}


def golden_e8m0():
    return {int(r[1], 16): float(r[5]) for r in load_golden("mxfp4_codes.txt") if r[0] == "e8m0"}


def np_dequant(q, s):
    """Independent dequantisation from the hand-decoded table."""
    table = np.array([golden_e2m1()[c] for c in range(16)], np.float64)
    q = np.asarray(q, np.uint8)
    lo = table[q & 0x0F]
    hi = table[q >> 4]
    vals = np.empty(q.shape[:-1] + (q.shape[-1] * 2,), np.float64)
    vals[..., 0::2] = lo
    vals[..., 1::2] = hi
    scale = np.ldexp(1.0, np.asarray(s, np.int64) - 127)
    return vals * np.repeat(scale, 32, axis=-1)


def bf16_to_f64(b):
    return synth.bf16_bits_to_f32(b).astype(np.float64)


def f32_round(x: Fraction) -> Fraction:
    """Exact round-to-nearest-even of a rational to IEEE binary32 (normal and
    subnormal range, no overflow in these tests)."""
    if x == 0:
        return Fraction(0)
    sign = -1 if x < 0 else 1
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    e = max(e, -126)
    ulp = Fraction(2) ** (e - 23)
    q, r = divmod(a, ulp)
    q = int(q)
    if r > ulp / 2 or (r == ulp / 2 and q % 2 == 1):
        q += 1
    return sign * q * ulp


# --------------------------------------------------------------- MXFP4 codes

def test_e2m1_hand_table():
    for code, val in golden_e2m1().items():
        got = oracle.e2m1_value(code)
        assert got == val and math.copysign(1, got) == math.copysign(1, val), (code, got, val)


def test_e8m0_hand_table():
    for byte, val in golden_e8m0().items():
        got = oracle.e8m0_value(byte)
        if math.isnan(val):
            assert math.isnan(got)
        else:
            assert got == val, (byte, got, val)


def test_nibble_order_low_is_even_k():
    # byte 0x2F: low nibble 0xF (-6) is K element 0, high nibble 0x2 (+1) is K element 1
    q = np.zeros((1, 16), np.uint8)
    q[0, 0] = 0x2F
    s = np.array([[0x7E]], np.uint8)          # scale 0.5
    d = oracle.dequant(q, s)
    assert d[0, 0] == -3.0 and d[0, 1] == 0.5 and np.all(d[0, 2:] == 0.0)


def test_scale_blocks_run_along_k():
    rng = np.random.default_rng(1)
    q = rng.integers(0, 256, (3, 64), dtype=np.uint8)       # K = 128: 4 blocks per row
    s = rng.integers(120, 130, (3, 4), dtype=np.uint8)
    assert np.array_equal(oracle.dequant(q, s), np_dequant(q, s))


# ------------------------------------------------------------- byte model

def test_byte_model_matches_printed_sizes():
    g = {r[0]: float(r[1]) for r in load_golden("byte_model.txt")}
    b = oracle.expert_bytes(4096, 2880)
    assert b == 18_800_640
    assert round(b / 2**20, 2) == g["expert_mib"]
    assert math.floor(b / 2**20 * 100) / 100 == g["expert_mib_alt"]
    assert round(384 * b / 2**30, 2) == g["layer_gib"]
    assert round(40 * 384 * b / 2**30) == g["model_gib"]
    # one expert over a ~340 GB/s host link takes ~55 us
    assert round(b / 2**20 * 2**20 / 340e9 * 1e6) == pytest.approx(g["c2c_expert_us"], abs=1)
    assert synth.expert_bytes(4096, 2880) == b


# ----------------------------------------------------------------- routing

def _route_case(T=64, E=48, k=6, seed=3):
    rng = np.random.default_rng(seed)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    return lg, oracle.route(lg, k)


# --------------------------------------------------------------------- bf16

def _f32(bits):
    return float(np.array([bits], np.uint32).view(np.float32)[0])


def test_bf16_rounding_hand_cases():
    # bf16 keeps the top 16 bits of a binary32; hand-worked round-to-nearest-even
    cases = [
        (0x3F800000, 0x3F80),   # 1.0 exact
        (0x3F808000, 0x3F80),   # 1 + 2^-8: halfway, even neighbour below
        (0x3F818000, 0x3F82),   # 1 + 3*2^-8: halfway, even neighbour above
        (0x3F808001, 0x3F81),   # just above halfway
        (0x3F807FFF, 0x3F80),   # just below halfway
        (0xBF808000, 0xBF80),   # sign does not change the tie rule
        (0x7F7FFFFF, 0x7F80),   # largest binary32 rounds up to +inf
        (0x00008000, 0x0000),   # tiny subnormal halfway: to even (zero)
        (0x80000000, 0x8000),   # -0 stays -0
    ]
    for f_bits, want in cases:
        assert oracle.f32_to_bf16(_f32(f_bits)) == want, hex(f_bits)
    nan = oracle.f32_to_bf16(float("nan"))
    assert (nan & 0x7F80) == 0x7F80 and (nan & 0x007F) != 0          # stays a NaN
    for b in (0x0000, 0x3F80, 0xC2F7, 0x7F80, 0x0001):
        assert np.array([oracle.bf16_to_f32(b)], np.float32).view(np.uint32)[0] == b << 16


# ------------------------------------------------------------------- router

def _bf16_bits(a):
    return synth._f32_to_bf16_bits(np.asarray(a, np.float32))


def test_router_integer_case_is_exact():
    # small integers are exact in bf16 and every partial sum is exact in
    # fp32, so the logits are the integer matrix product; T != E catches a
    # transposed operand, distinct values a wrong index
    rng = np.random.default_rng(3)
    T, E, H = 5, 7, 96
    xi = rng.integers(-8, 9, size=(T, H))
    wi = rng.integers(-8, 9, size=(E, H))
    bi = rng.integers(-50, 51, size=E)
    got = oracle.router_logits(_bf16_bits(xi), _bf16_bits(wi), bi.astype(np.float32))
    assert np.array_equal(got.astype(np.int64), xi @ wi.T + bi[None, :])
    got0 = oracle.router_logits(_bf16_bits(xi), _bf16_bits(wi), None)
    assert np.array_equal(got0.astype(np.int64), xi @ wi.T)


def test_router_one_hot_rows_pick_weight_columns():
    E, H = 6, 40
    w = synth.router_weights(synth.get_config("tiny", E=E, H=H), 0)
    x = np.zeros((H, H), np.float32)
    x[np.arange(H), np.arange(H)] = 1.0
    b = np.linspace(-1, 1, E).astype(np.float32)
    got = oracle.router_logits(_bf16_bits(x), w, b)
    want = synth.bf16_bits_to_f32(w).T.astype(np.float64) + b[None, :].astype(np.float64)
    assert np.array_equal(got, want.astype(np.float32))


def test_router_rounds_the_exact_sum_once():
    rng = np.random.default_rng(11)
    T, E, H = 3, 4, 24
    xb = _bf16_bits(rng.standard_normal((T, H)))
    wb = _bf16_bits(rng.standard_normal((E, H)))
    bias = rng.standard_normal(E).astype(np.float32)
    got = oracle.router_logits(xb, wb, bias)
    xf = [[Fraction(float(v)) for v in row] for row in synth.bf16_bits_to_f32(xb)]
    wf = [[Fraction(float(v)) for v in row] for row in synth.bf16_bits_to_f32(wb)]
    for t in range(T):
        for e in range(E):
            exact = Fraction(float(bias[e])) + sum(a * b for a, b in zip(xf[t], wf[e]))
            assert Fraction(float(got[t, e])) == f32_round(exact), (t, e)


def test_route_topk_matches_full_sort():
    lg, (ids, w) = _route_case()
    order = np.argsort(-lg, axis=1, kind="stable")[:, :6]      # stable: ties -> lower id
    assert np.array_equal(ids, order)


def test_route_ties_lower_id_first():
    lg = np.array([[1.0, 3.0, 3.0, 2.0, 3.0, 0.5]], np.float32)
    ids, w = oracle.route(lg, 4)
    assert ids.tolist() == [[1, 2, 4, 3]]
    assert w[0, 0] == w[0, 1] == w[0, 2]


def test_route_nan_logits_rank_below_every_number():
    """A NaN logit is read as -infinity: it is never picked while k finite
    logits remain, an all-NaN row yields the k lowest ids, and a pick read as
    -infinity gets weight 0 beside a finite first pick."""
    nan = np.float32(np.nan)
    lg = np.array([[nan, 0.5, nan, 2.0, -1.0, nan],
                   [nan, nan, nan, nan, nan, nan],
                   [nan, -np.inf, 1.0, nan, nan, nan]], np.float32)
    ids, w = oracle.route(lg, 3)
    assert ids[0].tolist() == [3, 1, 4]
    assert np.allclose(w[0], np.exp([0.0, -1.5, -3.0]) / np.exp([0.0, -1.5, -3.0]).sum(), rtol=2e-6)
    assert ids[1].tolist() == [0, 1, 2] and np.all(np.isnan(w[1]))
    # finite 1.0 first, then the -inf logit and the NaN ones tie at -inf: lower id first
    assert ids[2].tolist() == [2, 0, 1]
    assert w[2].tolist() == [1.0, 0.0, 0.0]


def test_route_weights_are_softmax_over_picks():
    lg, (ids, w) = _route_case()
    sel = np.take_along_axis(lg, ids, axis=1).astype(np.float64)
    assert np.all(np.diff(sel, axis=1) <= 0)
    ref = np.exp(sel - sel[:, :1])
    ref /= ref.sum(axis=1, keepdims=True)
    assert np.allclose(w, ref, rtol=2e-6, atol=0)
    assert np.all(np.abs(w.astype(np.float64).sum(axis=1) - 1.0) <= 1e-6)
    for row in ids:
        assert len(set(row.tolist())) == len(row)


def test_route_softmax_equals_full_softmax_renormalised():
    lg, (ids, w) = _route_case(T=8, E=16, k=3)
    full = np.exp(lg.astype(np.float64) - lg.max(axis=1, keepdims=True))
    full /= full.sum(axis=1, keepdims=True)
    top = np.take_along_axis(full, ids, axis=1)
    assert np.allclose(w, top / top.sum(axis=1, keepdims=True), rtol=2e-6)


# ------------------------------------------------------------ split / count

def _split_case(T=9, E=20, k=3, seed=5):
    rng = np.random.default_rng(seed)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    ids, _ = oracle.route(lg, k)
    is_hot = (rng.random(E) < 0.6).astype(np.uint8)
    rm, nh, nc = oracle.initial_rowmap(is_hot)
    return ids, is_hot, rm, nh, nc


def test_initial_rowmap_is_a_bijection_in_id_order():
    _, is_hot, rm, nh, nc = _split_case()
    assert nh == int(is_hot.sum()) and nc == len(is_hot) - nh
    hot_ids = np.flatnonzero(is_hot)
    cold_ids = np.flatnonzero(is_hot == 0)
    assert rm[hot_ids].tolist() == list(range(nh))
    assert (-1 - rm[cold_ids]).tolist() == list(range(nc))


def test_split_partitions_every_slot_once_in_row_order():
    ids, is_hot, rm, nh, nc = _split_case()
    sp = oracle.split(rm, ids)
    T, k = ids.shape
    assert sp[0]["n_picks"] + sp[1]["n_picks"] == T * k
    allp = np.concatenate([sp[0]["picks"], sp[1]["picks"]])
    assert sorted(allp.tolist()) == list(range(T * k))
    flat = ids.reshape(-1)
    for b, bank in enumerate(sp):
        rows = bank["act_row"]
        assert np.all(np.diff(rows) > 0)
        for a, r in enumerate(rows):
            seg = bank["picks"][bank["act_off"][a]:bank["act_off"][a + 1]]
            assert len(seg) > 0 and np.all(np.diff(seg) > 0)
            for s in seg:
                m = rm[flat[s]]
                assert (m >= 0) == (b == 0)
                assert (m if b == 0 else -1 - m) == r
        # every slot whose expert maps to this bank appears
        in_bank = [s for s in range(T * k) if (rm[flat[s]] >= 0) == (b == 0)]
        assert sorted(bank["picks"].tolist()) == in_bank


def test_count_histogram_and_prefill_rule():
    ids, *_ = _split_case()
    E = 20
    c = np.zeros(E, np.int32)
    oracle.count(c, ids, True, 256)
    assert np.array_equal(c, np.bincount(ids.reshape(-1), minlength=E).astype(np.int32))
    assert c.sum() == ids.size
    c2 = np.zeros(E, np.int32)
    oracle.count(c2, ids, False, 256)
    assert c2.sum() == 0
    big = np.zeros((300, 2), np.int32)
    c3 = np.zeros(E, np.int32)
    oracle.count(c3, big, True, 256)         # 300 tokens > 256: not counted
    assert c3.sum() == 0
    edge = np.zeros((256, 2), np.int32)
    oracle.count(c3, edge, True, 256)        # exactly 256: counted
    assert c3.sum() == 512


# ----------------------------------------------------------------- finalize

def test_finalize_fma_chain_is_exactly_rounded_in_k_order():
    rng = np.random.default_rng(7)
    T, k, H = 5, 6, 33
    Y = synth._f32_to_bf16_bits(rng.standard_normal((T, k, H)).astype(np.float32) * 1000)
    w = rng.random((T, k)).astype(np.float32)
    out = oracle.finalize(Y, w)
    for t in range(T):
        for c in range(H):
            acc = Fraction(0)
            for j in range(k):
                acc = f32_round(Fraction(float(w[t, j])) * Fraction(float(bf16_to_f64(Y[t, j, c]))) + acc)
            ref = synth._f32_to_bf16_bits(np.array([float(acc)], np.float32))[0]
            assert out[t, c] == ref, (t, c)


def test_finalize_uses_a_fused_multiply_add():
    # w1*y1 = 1 + 2^-7 + 2^-23 + 2^-30 is not an fp32 value; acc1 = -(1 + 2^-7 + 2^-23).
    # One rounding of w1*y1 + acc1 leaves 2^-30; multiply-then-add leaves 0.
    w = np.array([[-(1 + 2.0**-7 + 2.0**-23), 1 + 2.0**-23]], np.float32)
    Y = synth._f32_to_bf16_bits(np.array([[[1.0], [1 + 2.0**-7]]], np.float32))
    out = oracle.finalize(Y, w)
    assert bf16_to_f64(out[0, 0]) == 2.0**-30


def test_finalize_order_matters_and_k1_is_identity():
    # values where summing in another order changes the fp32 result
    Y = synth._f32_to_bf16_bits(np.array([[[1.0], [2.0**-24 * 3], [-1.0]]], np.float32))
    w = np.ones((1, 3), np.float32)
    fwd = oracle.finalize(Y, w)
    rev = oracle.finalize(Y[:, ::-1].copy(), w)
    assert fwd[0, 0] != rev[0, 0]
    Y1 = synth._f32_to_bf16_bits(np.random.default_rng(0).standard_normal((4, 1, 16)).astype(np.float32))
    assert np.array_equal(oracle.finalize(Y1, np.ones((4, 1), np.float32)), Y1[:, 0, :])


# ---------------------------------------------------------------------- FFN

def np_swiglu_ffn(Wg, Wu, W2, x):
    """Textbook dense SwiGLU FFN in float64: W2 (silu(Wg x) * (Wu x))."""
    g = Wg @ x
    u = Wu @ x
    return W2 @ (g / (1.0 + np.exp(-g)) * u)


def test_single_expert_equals_textbook_dense_swiglu():
    cfg = synth.get_config("tiny")
    w13_q, w13_s, w2_q, w2_s = synth.expert_weights(cfg, 0, 3)
    x = synth.activations(cfg, 0, 0)[:1]
    y = oracle.expert_ffn(w13_q, w13_s, w2_q, w2_s, x)
    W13 = np_dequant(w13_q, w13_s)
    W2 = np_dequant(w2_q, w2_s)
    I = cfg.I
    ref = np_swiglu_ffn(W13[:I], W13[I:], W2, bf16_to_f64(x[0]))
    got = bf16_to_f64(y[0])
    # bf16 output rounding (2^-9 relative) plus fp32 intermediates
    assert np.all(np.abs(got - ref) <= 2.0**-8 * np.abs(ref) + 1e-6 * np.abs(ref).max())
    # a swapped gate/up would not pass
    bad = np_swiglu_ffn(W13[I:], W13[:I], W2, bf16_to_f64(x[0]))
    assert np.abs(bad - ref).max() > 0.1 * np.abs(ref).max()


def test_layer_step_equals_bruteforce_dense_all_experts():
    """Evaluate every expert densely for every token (numpy float64), then
    combine the top-k with softmax weights: the routed layer must agree."""
    cfg = synth.get_config("tiny")
    weights = synth.layer_weights(cfg, 0)
    x = synth.activations(cfg, 0, 0)
    lg = synth.router_logits(cfg, 0, 0)
    counts = np.zeros(cfg.E, np.int32)
    ids, w, Y, out = oracle.layer_step(weights, lg, x, cfg.k, counts=counts)
    X = bf16_to_f64(x)
    I = cfg.I
    dense = np.empty((cfg.E, cfg.T, cfg.H))
    for e in range(cfg.E):
        W13 = np_dequant(weights[0][e], weights[1][e])
        W2 = np_dequant(weights[2][e], weights[3][e])
        for t in range(cfg.T):
            dense[e, t] = np_swiglu_ffn(W13[:I], W13[I:], W2, X[t])
    sel = np.argsort(-lg.astype(np.float64), axis=1, kind="stable")[:, :cfg.k]
    assert np.array_equal(ids, sel)
    l = np.take_along_axis(lg.astype(np.float64), sel, axis=1)
    p = np.exp(l - l[:, :1])
    p /= p.sum(axis=1, keepdims=True)
    ref = np.einsum("tj,tjh->th", p, dense[sel, np.arange(cfg.T)[:, None]])
    got = bf16_to_f64(out)
    rel_l2 = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert rel_l2 < 3e-3
    assert np.abs(got - ref).max() <= 2e-2 * np.abs(ref).max()
    # per-pick rows too
    for t in range(cfg.T):
        for j in range(cfg.k):
            r = dense[sel[t, j], t]
            assert np.abs(bf16_to_f64(Y[t, j]) - r).max() <= 2.0**-8 * np.abs(r).max()
    assert counts.sum() == cfg.T * cfg.k


def test_rows_for_slots_matches_layer_step():
    cfg = synth.get_config("tiny")
    weights = synth.layer_weights(cfg, 0)
    x = synth.activations(cfg, 0, 0)
    lg = synth.router_logits(cfg, 0, 0)
    ids, w, Y, out = oracle.layer_step(weights, lg, x, cfg.k)
    slots = np.array([0, 5, 7, 15, 3], np.int32)
    Ys = oracle.rows_for_slots(weights, ids, x, slots)
    assert np.array_equal(Ys, Y.reshape(-1, cfg.H)[slots])


# -------------------------------------------------------------------- swaps

def test_swap_exchanges_rows_and_refuses_stale_pairs():
    is_hot = np.array([1, 1, 0, 1, 0, 0, 1], np.uint8)
    rm, nh, nc = oracle.initial_rowmap(is_hot)
    before = rm.copy()
    applied = oracle.swap(rm, [2, 2, 4, 0], [1, 3, 0, 5])
    # pair 0: 2 (cold row 0) <-> 1 (hot row 1); pair 1 is stale (2 is hot now);
    # pair 2: 4 (cold row 1) <-> 0 (hot row 0); pair 3 stale (0 is cold now)
    assert applied.tolist() == [1, 0, 1, 0]
    assert rm[2] == before[1] and rm[1] == before[2]
    assert rm[4] == before[0] and rm[0] == before[4]
    hot_rows = sorted(rm[rm >= 0].tolist())
    cold_rows = sorted((-1 - rm[rm < 0]).tolist())
    assert hot_rows == list(range(nh)) and cold_rows == list(range(nc))
    back = oracle.swap(rm, [1, 0], [2, 4])
    assert back.tolist() == [1, 1] and np.array_equal(rm, before)


def test_swap_rejects_bad_ids_and_self_pairs():
    rm, _, _ = oracle.initial_rowmap(np.array([1, 0, 1], np.uint8))
    before = rm.copy()
    assert oracle.swap(rm, [1, -1, 1, 7], [1, 0, 9, 0]).tolist() == [0, 0, 0, 0]
    assert np.array_equal(rm, before)


# ------------------------------------------------------------------- policy

def test_policy_constant_rate_average_is_exact():
    E = 6
    is_hot = np.array([1, 1, 1, 0, 0, 0], np.uint8)
    rm, _, _ = oracle.initial_rowmap(is_hot)
    pol = oracle.Policy(E, read_every=16, half_life=500, hysteresis=1.5, min_avg=8, max_pairs=8)
    rate = np.array([20, 1, 10, 30, 2, 9], np.int64)
    counts = np.zeros(E, np.int64)
    for _ in range(5):
        counts += rate
        pro, dem = pol.read(counts.astype(np.int32), rm)
    # a decaying average of a constant is that constant
    assert np.allclose(pol.acc / pol.st.wsum, rate, rtol=1e-12)
    # cold by avg desc with avg >= 8: 3 (30), 5 (9); hot by avg asc: 1 (1), 2 (10)
    # pairs: 30 > 1.5*1 yes; 9 > 1.5*10 no -> one pair
    assert pro.tolist() == [3] and dem.tolist() == [1]


def test_policy_decay_closed_form_and_limits():
    E = 4
    rm, _, _ = oracle.initial_rowmap(np.array([1, 1, 0, 0], np.uint8))
    pol = oracle.Policy(E, read_every=64, half_life=128, hysteresis=1.5, min_avg=8, max_pairs=1)
    d = 0.5 ** (64 / 128)
    seq = [np.array([0, 0, 0, 0]), np.array([4, 4, 100, 100])]
    counts = np.zeros(E, np.int64)
    counts += seq[1]
    pro, dem = pol.read(counts.astype(np.int32), rm)          # first read: avg = delta
    assert np.allclose(pol.acc / pol.st.wsum, [4, 4, 100, 100])
    assert pro.tolist() == [2] and dem.tolist() == [0]      # max_pairs=1, ties -> lower id
    counts += 0
    pol.read(counts.astype(np.int32), rm)                    # a read with no picks
    want = np.array([4, 4, 100, 100]) * d / (d + 1.0)
    assert np.allclose(pol.acc / pol.st.wsum, want, rtol=1e-12)


def test_policy_hysteresis_boundary_is_strict():
    E = 2
    rm, _, _ = oracle.initial_rowmap(np.array([1, 0], np.uint8))
    pol = oracle.Policy(E, read_every=1, half_life=1e9, hysteresis=1.5, min_avg=8, max_pairs=4)
    pro, _ = pol.read(np.array([10, 15], np.int32), rm)      # 15 == 1.5 * 10: no swap
    assert pro.size == 0
    pol2 = oracle.Policy(E, read_every=1, half_life=1e9, hysteresis=1.5, min_avg=8, max_pairs=4)
    pro, dem = pol2.read(np.array([10, 16], np.int32), rm)
    assert pro.tolist() == [1] and dem.tolist() == [0]
    pol3 = oracle.Policy(E, read_every=1, half_life=1e9, hysteresis=1.5, min_avg=8, max_pairs=4)
    pro, _ = pol3.read(np.array([0, 7], np.int32), rm)        # below minimum average
    assert pro.size == 0


# ------------------------------------------------------------------ restore

def test_restore_plan_hand_example():
    # now hot {0, 1, 3, 6}; saved hot {1, 2, 3, 4}: 2 and 4 come in, 0 and 6 go out
    now, _, _ = oracle.initial_rowmap(np.array([1, 1, 0, 1, 0, 0, 1], np.uint8))
    saved, _, _ = oracle.initial_rowmap(np.array([0, 1, 1, 1, 1, 0, 0], np.uint8))
    pro, dem = oracle.plan_restore(now, saved, 8)
    assert pro.tolist() == [2, 4] and dem.tolist() == [0, 6]
    pro, dem = oracle.plan_restore(now, saved, 1)
    assert pro.tolist() == [2] and dem.tolist() == [0]
    assert [a.tolist() for a in oracle.plan_restore(now, now, 8)] == [[], []]
    bigger, _, _ = oracle.initial_rowmap(np.array([1, 1, 1, 1, 1, 0, 0], np.uint8))
    assert oracle.plan_restore(now, bigger, 8) is None        # hot counts differ


@pytest.mark.parametrize("seed", range(6))
def test_restore_reaches_the_saved_hot_set_in_the_fewest_swaps(seed):
    rng = np.random.default_rng(seed)
    E = int(rng.integers(2, 200))
    n_hot = int(rng.integers(1, E))
    saved_mask = np.zeros(E, np.uint8)
    saved_mask[rng.permutation(E)[:n_hot]] = 1
    saved, _, _ = oracle.initial_rowmap(saved_mask)
    rm = saved.copy()
    # wander away with random valid swaps
    for _ in range(int(rng.integers(0, 3 * E))):
        hot, cold = np.flatnonzero(rm >= 0), np.flatnonzero(rm < 0)
        oracle.swap(rm, [rng.choice(cold)], [rng.choice(hot)])
    # each swap moves one expert in and one out, so no plan can be shorter
    # than the number of experts hot now and cold in the saved map
    need = int(np.count_nonzero((rm >= 0) & (saved < 0)))
    budget = int(rng.integers(1, 9))
    rounds, total = 0, 0
    while True:
        pro, dem = oracle.plan_restore(rm, saved, budget)
        if pro.size == 0:
            break
        assert pro.size <= budget
        assert np.all(rm[pro] < 0) and np.all(saved[pro] >= 0)
        assert np.all(rm[dem] >= 0) and np.all(saved[dem] < 0)
        assert oracle.swap(rm, pro, dem).tolist() == [1] * pro.size
        rounds += 1
        total += pro.size
    assert total == need and rounds == -(-need // budget)
    assert np.array_equal(rm >= 0, saved >= 0)
    hot_rows = sorted(rm[rm >= 0].tolist())
    assert hot_rows == list(range(n_hot))                   # still a bijection onto the bank rows


# ------------------------------------------------------- MXFP8 activations

def test_e4m3_rounding_matches_torch_float8():
    """The oracle's E4M3 rounding, written from the format's definition,
    against torch's float32 -> float8_e4m3fn cast on values inside +-448:
    random magnitudes across the normal and subnormal binades, and every
    midpoint between neighbouring E4M3 values (the ties)."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(11)
    v = (rng.standard_normal(20000) * np.exp2(rng.integers(-14, 9, 20000))).astype(np.float32)
    v = v[np.abs(v) <= 448]
    grid = torch.arange(0, 256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    grid = np.unique(np.abs(grid[np.isfinite(grid)]))
    mids = ((grid[1:] + grid[:-1]) / 2).astype(np.float32)
    vals = np.concatenate([v, mids, -mids, grid.astype(np.float32)])
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).float().numpy()
    got = np.array([oracle.e4m3(float(a)) for a in vals])
    assert np.array_equal(got, ref.astype(np.float64))


def test_e4m3_hand_values():
    # 1.0625 lies halfway between 1.0 and 1.125: ties to the even mantissa 1.0
    assert oracle.e4m3(1.0625) == 1.0
    # 1.1875 lies halfway between 1.125 (odd) and 1.25 (even)
    assert oracle.e4m3(1.1875) == 1.25
    # subnormal spacing 2^-9: 2^-10 ties to 0, 3 * 2^-10 ties to 2^-8
    assert oracle.e4m3(2.0 ** -10) == 0.0 and oracle.e4m3(3 * 2.0 ** -10) == 2.0 ** -8
    assert oracle.e4m3(448.0) == 448.0 and oracle.e4m3(464.0) == 448.0 and oracle.e4m3(-1e6) == -448.0
    assert oracle.e4m3(-0.3) == -0.3125          # 0.3 / 2^-5 = 9.6 -> 10 steps


def test_mx8_block_exponent_boundaries():
    # the smallest e with amax * 2^-e <= 448
    assert oracle.mx8_block_exponent(0.0) == 0
    assert oracle.mx8_block_exponent(448.0) == 0
    assert oracle.mx8_block_exponent(448.0001) == 1
    assert oracle.mx8_block_exponent(224.0) == -1        # 224 * 2 = 448 still fits
    assert oracle.mx8_block_exponent(224.0001) == 0
    assert oracle.mx8_block_exponent(1.0) == -8          # 256 <= 448 < 512
    assert oracle.mx8_block_exponent(2.0 ** -20) == -28
    # held to the e8m0 scale's range
    assert oracle.mx8_block_exponent(2.0 ** -200) == -127 and oracle.mx8_block_exponent(2.0 ** 200) == 127


def test_mx8_quantize_blocks_are_independent_and_exact_values_stay():
    rng = np.random.default_rng(3)
    # values with 4 significant bits, within one binade of the block max:
    # exactly representable after the shared scaling
    v = (rng.integers(8, 16, 64) * np.exp2(rng.integers(-3, 0, 64)) * rng.choice([-1, 1], 64)).astype(np.float64)
    assert np.array_equal(oracle.mx8_quantize(v), v)
    # a large value in block 0 coarsens block 0 only
    w = v.copy()
    w[0] = 2.0 ** 20
    q = oracle.mx8_quantize(w)
    assert np.array_equal(q[32:], v[32:])
    assert not np.array_equal(q[1:32], v[1:32])
    e = oracle.mx8_block_exponent(2.0 ** 20)
    for a, b in zip(q[:32], w[:32]):      # each element is its own e4m3 rounding at the block's scale
        assert a == np.ldexp(oracle.e4m3(np.ldexp(b, -e)), e)


def test_expert_ffn_mx8_composition():
    """qx = qh = 0 is the pinned FFN bit for bit; qx alone is the pinned FFN
    applied to the MXFP8 reading of x (exact in bf16: 4 significant bits);
    adding qh changes the rows by e4m3-level relative error."""
    cfg = synth.get_config("tiny")
    w = synth.expert_weights(cfg, 0, 3)
    x = synth.activations(cfg, 0, 0)[:4]
    base = oracle.expert_ffn(*w, x)
    assert np.array_equal(oracle.expert_ffn_mx8(*w, x, qx=False, qh=False), base)
    xq = np.stack([oracle.mx8_quantize(synth.bf16_bits_to_f32(r).astype(np.float64)) for r in x])
    xq_bits = synth._f32_to_bf16_bits(xq.astype(np.float32))
    assert np.array_equal(synth.bf16_bits_to_f32(xq_bits).astype(np.float64), xq)
    only_x = oracle.expert_ffn_mx8(*w, x, qx=True, qh=False)
    assert np.array_equal(only_x, oracle.expert_ffn(*w, xq_bits))
    both = oracle.expert_ffn_mx8(*w, x, qx=True, qh=True)
    a = synth.bf16_bits_to_f32(both).astype(np.float64)
    b = synth.bf16_bits_to_f32(only_x).astype(np.float64)
    rel = np.linalg.norm(a - b) / np.linalg.norm(b)
    assert 1e-3 < rel < 0.08
