"""The C ABI without a GPU: the library builds for sm_103a and loads, every
symbol include/moe_residency.h declares is exported, argument validation
fails cleanly, and the native host policy and restore planner take the
oracle's decisions."""
import ctypes as C

import numpy as np
import pytest

import cold_expert_residency_gb300 as moe
import oracle


@pytest.fixture(scope="module")
def lib():
    moe.build()
    return moe.lib()


def test_every_declared_symbol_is_exported(lib):
    names = moe.exported_symbols()
    assert len(names) >= 20
    for n in ["moe_init_banks", "moe_route_split_count", "moe_expert_ffn_bank", "moe_finalize",
              "moe_swap_rows", "moe_read_counts"]:
        assert n in names
    for n in names:
        assert hasattr(lib, n), n


def test_expert_bytes(lib):
    assert moe.moe_expert_bytes(4096, 2880) == 18_800_640
    assert moe.moe_expert_bytes(256, 128) == oracle.expert_bytes(256, 128)


def test_bad_geometry_is_rejected(lib):
    bad = [dict(layers=0), dict(experts=1), dict(top_k=0), dict(top_k=17), dict(hidden=100),
           dict(inter=96), dict(max_tokens=0), dict(experts=2000),
           dict(hidden=384, inter=192)]   # W2 tiles odd in number and K ending in half a group
    base = dict(layers=1, experts=16, top_k=2, hidden=256, inter=128, max_tokens=8)
    for b in bad:
        kw = dict(base, **b)
        with pytest.raises(moe.MoeError) as ei:
            moe.moe_create(kw["layers"], kw["experts"], kw["top_k"], kw["hidden"], kw["inter"], kw["max_tokens"])
        assert ei.value.code == moe.MOE_EINVAL


def test_null_and_shape_checks_fail_cleanly(lib):
    assert lib.moe_finalize(None, None, 4, 0, 64, None, None) == moe.MOE_EINVAL
    assert lib.moe_finalize(None, None, 4, 2, 60, None, None) == moe.MOE_EINVAL
    assert lib.moe_finalize(None, None, 0, 2, 64, None, None) == moe.MOE_OK     # empty step
    assert lib.moe_swap_rows(None, 0, 0, None, None, None, None) == moe.MOE_EINVAL
    assert lib.moe_read_counts(None, None, None) == moe.MOE_EINVAL
    assert b"context" in lib.moe_last_error()
    assert lib.moe_policy_create(0, 64.0, 500.0, 1.5, 8.0, 2, None, C.byref(C.c_void_p())) == moe.MOE_EINVAL
    # router: context, shape and pointer checks come before any device work
    assert lib.moe_router_logits(None, None, None, None, 0, 16, 256, None, None) == moe.MOE_EINVAL
    assert lib.moe_step_scratch_bytes(None, 8, C.byref(C.c_size_t())) == moe.MOE_EINVAL
    assert lib.moe_layer_step_host(None, 0, None, None, 8, 1, None, None, None) == moe.MOE_EINVAL
    assert b"context" in lib.moe_last_error()


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_native_policy_matches_oracle_policy(lib, seed):
    rng = np.random.default_rng(seed)
    E = 64
    is_hot = np.zeros(E, np.uint8)
    is_hot[rng.permutation(E)[:48]] = 1
    rm, _, _ = oracle.initial_rowmap(is_hot)
    params = dict(read_every=16.0, half_life=200.0, hysteresis=1.5, min_avg=8.0, max_pairs=8)
    ref = oracle.Policy(E, **params)
    nat = moe.moe_policy(E, **params)
    counts = np.zeros(E, np.int64)
    p = rng.dirichlet(np.full(E, 0.3))
    for read in range(12):
        if read == 6:
            p = rng.dirichlet(np.full(E, 0.3))       # traffic shift
        counts += rng.multinomial(16 * 42, p)
        a = ref.read(counts.astype(np.int32), rm)
        b = nat.read(counts.astype(np.int32), rm)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1]), read
        oracle.swap(rm, a[0], a[1])


def test_policy_counts_wrap_as_uint32(lib):
    rm, _, _ = oracle.initial_rowmap(np.array([1, 0], np.uint8))
    start = np.array([2**31 - 5, 2**31 - 5], np.int64).astype(np.int32)
    nat = moe.moe_policy(2, read_every=1, half_life=1e9, min_avg=8, max_pairs=1, counts_now=start)
    ref = oracle.Policy(2, counts=start, read_every=1, half_life=1e9, min_avg=8, max_pairs=1)
    now = (np.array([2**31 - 5 + 2, 2**31 - 5 + 40], np.int64) & 0xFFFFFFFF).astype(np.uint32).view(np.int32)
    assert [x.tolist() for x in nat.read(now, rm)] == [[1], [0]]
    assert [x.tolist() for x in ref.read(now, rm)] == [[1], [0]]


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_native_restore_plan_matches_oracle(lib, seed):
    rng = np.random.default_rng(seed)
    E = 384
    mask = np.zeros(E, np.uint8)
    mask[rng.permutation(E)[:295]] = 1
    saved, _, _ = oracle.initial_rowmap(mask)
    rm = saved.copy()
    for _ in range(40):
        hot, cold = np.flatnonzero(rm >= 0), np.flatnonzero(rm < 0)
        oracle.swap(rm, [rng.choice(cold)], [rng.choice(hot)])
    for budget in (0, 1, 8, E):
        a = oracle.plan_restore(rm, saved, budget)
        b = moe.moe_plan_restore(rm, saved, budget)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1]), budget


def test_native_restore_plan_rejects_a_different_hot_count(lib):
    now, _, _ = oracle.initial_rowmap(np.array([1, 0, 0], np.uint8))
    other, _, _ = oracle.initial_rowmap(np.array([1, 1, 0], np.uint8))
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_plan_restore(now, other, 4)
    assert ei.value.code == moe.MOE_EINVAL and "hot experts" in str(ei.value)


def _declared_param_counts():
    """Parameter count of every function the header declares, read from the
    header text (comments stripped)."""
    import os
    import re
    hdr = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "moe_residency.h")
    text = re.sub(r"/\*.*?\*/", "", open(hdr).read(), flags=re.S)
    counts = {}
    for m in re.finditer(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(moe_[a-z_0-9]+)\s*\(([^)]*)\)\s*;", text, re.M):
        params = m.group(2).strip()
        counts[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return counts


def test_binding_signatures_match_the_header(lib):
    counts = _declared_param_counts()
    assert set(counts) == set(moe.exported_symbols())
    for name, n in counts.items():
        fn = getattr(lib, name)
        assert fn.argtypes is not None, f"{name} has no ctypes signature"
        assert len(fn.argtypes) == n, f"{name}: header has {n} parameters, binding {len(fn.argtypes)}"


def test_restore_plan_argument_checks(lib):
    rm = np.array([0, -1, 1, -2], np.int32)
    tg = np.array([-1, 0, 1, -2], np.int32)
    assert [a.tolist() for a in moe.moe_plan_restore(rm, tg, 0)] == [[], []]       # zero budget: no pairs
    assert lib.moe_plan_restore(4, moe._ptr(rm), moe._ptr(tg), 2, None, None) == moe.MOE_EINVAL
    assert lib.moe_plan_restore(0, moe._ptr(rm), moe._ptr(tg), 2, None, None) == moe.MOE_EINVAL
    assert lib.moe_plan_restore(4, None, moe._ptr(tg), 0, None, None) == moe.MOE_EINVAL
    pro, dem = moe.moe_plan_restore(rm, tg, 4)
    assert pro.tolist() == [1] and dem.tolist() == [0]


def test_policy_and_counter_defaults_are_the_printed_ones(lib):
    import inspect
    from conftest import load_golden
    g = {r[0]: float(r[1]) for r in load_golden("policy_defaults.txt")}
    for fn in (moe.moe_policy.__init__, oracle.Policy.__init__):
        p = inspect.signature(fn).parameters
        assert p["read_every"].default == g["read_every"]
        assert p["half_life"].default == g["half_life"]
        assert p["hysteresis"].default == g["hysteresis"]
        assert p["min_avg"].default == g["min_avg"]
        assert p["max_pairs"].default == g["max_pairs_per_read"]
    assert inspect.signature(moe.moe_create).parameters["count_tmax"].default == g["count_tmax"]
    # the restore helper's per-call budget is the per-step swap budget
    from cold_expert_residency_gb300.runtime import restore_placement
    assert inspect.signature(restore_placement).parameters["budget"].default == g["max_swaps_per_step"]
    # the usage table: int32 per (layer, expert), 40 x 384 x 4 B = 61 KB (rounded down)
    assert int(g["table_layers"] * g["table_experts"] * 4 / 1000) == g["table_kb"]


def test_failure_hooks_without_a_device(lib):
    """The memory accounting and the failure-path hooks load and validate
    their arguments without a GPU (no context can exist here)."""
    d, p = moe.moe_memory_in_use()
    assert d >= 0 and p >= 0
    for fn, args in ((lib.moe_set_wait_limit, (None, 1000)), (lib.moe_inject_fault, (None, 1))):
        assert fn(*args) == moe.MOE_EINVAL
    assert lib.moe_memory_in_use(None, None) == moe.MOE_OK
