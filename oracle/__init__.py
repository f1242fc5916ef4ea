"""CPU oracle for the split-residency routed MoE layer -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The CUDA library (``cold_expert_residency_gb300``)
never imports it and shares no code with it.

The arithmetic lives in ``moe_oracle.c`` (plain C, built with gcc,
``-ffp-contract=off``, OpenMP only across independent output rows); this
module builds it on first use and wraps it with numpy arrays.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_HDR = os.path.join(_HERE, "moe_oracle.h")
_SO = os.path.join(_HERE, "_build", "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc into oracle/_build/ and return the path."""
    os.makedirs(os.path.dirname(_SO), exist_ok=True)
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < newest:
        tmp = _SO + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
               "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = C.CDLL(build())
        P = C.c_void_p
        i32, i64, f64 = C.c_int, C.c_int64, C.c_double
        sig = {
            "orc_e2m1_value": (f64, [C.c_uint]),
            "orc_e8m0_value": (f64, [C.c_uint]),
            "orc_dequant": (None, [P, P, i64, i64, P]),
            "orc_bf16_to_f32": (C.c_float, [C.c_uint16]),
            "orc_f32_to_bf16": (C.c_uint16, [C.c_float]),
            "orc_router_logits": (None, [P, P, P, i32, i32, i32, P]),
            "orc_route": (None, [P, i32, i32, i32, P, P]),
            "orc_initial_rowmap": (None, [P, i32, P, P, P]),
            "orc_split": (None, [P, i32, P, i32, i32, P]),
            "orc_count": (None, [P, i32, P, i32, i32, i32, i32]),
            "orc_expert_ffn": (None, [P, P, P, P, i32, i32, P, i32, P]),
            "orc_finalize": (None, [P, P, i32, i32, i32, P]),
            "orc_layer_step": (None, [P, P, P, P, i32, i32, i32, i32, P, P, i32, P, P, P, P, P, i32, i32]),
            "orc_rows_for_slots": (None, [P, P, P, P, i32, i32, i32, P, P, P, i32, P]),
            "orc_rows_for_slots_fmt": (None, [P, P, P, P, i32, i32, i32, P, P, P, i32, P, i32]),
            "orc_e4m3_rne": (f64, [f64]),
            "orc_mx8_block_exponent": (i32, [f64]),
            "orc_mx8_quantize": (None, [P, i64, P]),
            "orc_expert_ffn_mx8": (None, [P, P, P, P, i32, i32, P, i32, P, i32, i32]),
            "orc_swap": (i32, [P, i32, i32, P, P, P]),
            "orc_plan_restore": (i32, [P, P, i32, i32, P, P]),
            "orc_policy_init": (None, [P, i32, P, P, P]),
            "orc_policy_read": (i32, [P, P, P, f64, f64, f64, f64, i32, P, P]),
            "orc_expert_bytes": (i64, [i32, i32]),
            "orc_num_threads": (i32, []),
            "orc_set_num_threads": (None, [i32]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(C.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ------------------------------------------------------------------ decode

def e2m1_value(code: int) -> float:
    return _load().orc_e2m1_value(code)


def e8m0_value(byte: int) -> float:
    return _load().orc_e8m0_value(byte)


def dequant(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """[rows][K/2] e2m1 bytes + [rows][K/32] e8m0 -> float64 [rows][K]."""
    q = _c(q, np.uint8)
    s = _c(s, np.uint8)
    rows, half = q.shape
    out = np.empty((rows, 2 * half), np.float64)
    _load().orc_dequant(_p(q), _p(s), rows, 2 * half, _p(out))
    return out


def bf16_to_f32(b: int) -> float:
    return _load().orc_bf16_to_f32(b)


def f32_to_bf16(f: float) -> int:
    return _load().orc_f32_to_bf16(f)


# ----------------------------------------------------------------- routing

def router_logits(x_bits: np.ndarray, w_router_bits: np.ndarray, bias=None) -> np.ndarray:
    """x bf16 bits [T][H], router weight bf16 bits [E][H], bias fp32 [E] or
    None -> logits float32 [T][E]."""
    x = _c(x_bits, np.uint16)
    w = _c(w_router_bits, np.uint16)
    T, H = x.shape
    E = w.shape[0]
    assert w.shape[1] == H
    b = None if bias is None else _c(bias, np.float32)
    out = np.empty((T, E), np.float32)
    _load().orc_router_logits(_p(x), _p(w), None if b is None else _p(b), T, E, H, _p(out))
    return out


def route(logits: np.ndarray, k: int):
    """-> ids int32 [T][k], w float32 [T][k]."""
    lg = _c(logits, np.float32)
    T, E = lg.shape
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float32)
    _load().orc_route(_p(lg), T, E, k, _p(ids), _p(w))
    return ids, w


def initial_rowmap(is_hot: np.ndarray):
    m = _c(is_hot, np.uint8)
    rm = np.empty(m.size, np.int32)
    nh, nc = C.c_int(), C.c_int()
    _load().orc_initial_rowmap(_p(m), m.size, _p(rm), C.byref(nh), C.byref(nc))
    return rm, nh.value, nc.value


class _Split(C.Structure):
    _fields_ = [("n_picks", C.c_int32 * 2), ("n_act", C.c_int32 * 2),
                ("act_row", C.c_void_p * 2), ("act_off", C.c_void_p * 2),
                ("picks", C.c_void_p * 2)]


def split(row_map: np.ndarray, ids: np.ndarray):
    """-> dict per bank (0 hot, 1 cold): act_row, act_off, picks (int32)."""
    rm = _c(row_map, np.int32)
    ids = _c(ids, np.int32)
    T, k = ids.shape
    P = T * k
    bufs = [[np.zeros(max(P, 1), np.int32), np.zeros(P + 1, np.int32), np.zeros(max(P, 1), np.int32)]
            for _ in range(2)]
    st = _Split()
    for b in range(2):
        st.act_row[b] = bufs[b][0].ctypes.data
        st.act_off[b] = bufs[b][1].ctypes.data
        st.picks[b] = bufs[b][2].ctypes.data
    _load().orc_split(_p(rm), rm.size, _p(ids), T, k, C.byref(st))
    out = []
    for b in range(2):
        na, npk = st.n_act[b], st.n_picks[b]
        out.append(dict(n_act=na, n_picks=npk, act_row=bufs[b][0][:na].copy(),
                        act_off=bufs[b][1][:na + 1].copy(), picks=bufs[b][2][:npk].copy()))
    return out


def count(counts: np.ndarray, ids: np.ndarray, count_on: bool, count_tmax: int = 256):
    """Updates ``counts`` (int32 [E]) in place."""
    assert counts.dtype == np.int32 and counts.flags.c_contiguous
    ids = _c(ids, np.int32)
    T, k = ids.shape
    _load().orc_count(_p(counts), counts.size, _p(ids), T, k, int(count_on), count_tmax)


# --------------------------------------------------------------------- FFN

def expert_ffn(w13_q, w13_s, w2_q, w2_s, x: np.ndarray) -> np.ndarray:
    """One expert (logical layout), x bf16 bits [n][H] -> y bf16 bits [n][H]."""
    w13_q, w13_s, w2_q, w2_s = (_c(a, np.uint8) for a in (w13_q, w13_s, w2_q, w2_s))
    x = _c(x, np.uint16)
    n, H = x.shape
    I = w2_q.shape[1] * 2
    y = np.empty((n, H), np.uint16)
    _load().orc_expert_ffn(_p(w13_q), _p(w13_s), _p(w2_q), _p(w2_s), H, I, _p(x), n, _p(y))
    return y


def finalize(Y: np.ndarray, w: np.ndarray) -> np.ndarray:
    """Y bf16 bits [T][k][H], w float32 [T][k] -> out bf16 bits [T][H]."""
    Y = _c(Y, np.uint16)
    w = _c(w, np.float32)
    T, k, H = Y.shape
    out = np.empty((T, H), np.uint16)
    _load().orc_finalize(_p(Y), _p(w), T, k, H, _p(out))
    return out


def layer_step(weights, logits: np.ndarray, x: np.ndarray, k: int, counts=None,
               count_on: bool = True, count_tmax: int = 256):
    """Whole unsplit layer-step.  weights = stacked logical (w13_q, w13_s,
    w2_q, w2_s) over all E experts.  Returns ids, w, Y [T][k][H], out [T][H]."""
    w13_q, w13_s, w2_q, w2_s = (_c(a, np.uint8) for a in weights)
    lg = _c(logits, np.float32)
    x = _c(x, np.uint16)
    T, E = lg.shape
    H = x.shape[1]
    I = w2_q.shape[2] * 2
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float32)
    Y = np.empty((T, k, H), np.uint16)
    out = np.empty((T, H), np.uint16)
    cp = None if counts is None else _p(counts)
    if counts is not None:
        assert counts.dtype == np.int32 and counts.flags.c_contiguous
    _load().orc_layer_step(_p(w13_q), _p(w13_s), _p(w2_q), _p(w2_s), E, k, H, I, _p(lg), _p(x), T,
                           _p(ids), _p(w), _p(Y), _p(out), cp, int(count_on), count_tmax)
    return ids, w, Y, out


def rows_for_slots(weights, ids: np.ndarray, x: np.ndarray, slots, mx8: bool = False) -> np.ndarray:
    """Expert rows Y[s] for the given slot indices s = t*k + j only; with
    mx8, the token rows and h read as MXFP8 (expert_ffn_mx8)."""
    w13_q, w13_s, w2_q, w2_s = (_c(a, np.uint8) for a in weights)
    ids = _c(ids, np.int32)
    x = _c(x, np.uint16)
    slots = _c(slots, np.int32)
    k = ids.shape[1]
    H = x.shape[1]
    I = w2_q.shape[2] * 2
    Y = np.empty((slots.size, H), np.uint16)
    _load().orc_rows_for_slots_fmt(_p(w13_q), _p(w13_s), _p(w2_q), _p(w2_s), H, I, k, _p(ids), _p(x),
                                   _p(slots), slots.size, _p(Y), 1 if mx8 else 0)
    return Y


def e4m3(v: float) -> float:
    """FP8 E4M3 value nearest v (ties to even), saturated at +-448."""
    return float(_load().orc_e4m3_rne(float(v)))


def mx8_block_exponent(amax: float) -> int:
    return int(_load().orc_mx8_block_exponent(float(amax)))


def mx8_quantize(v: np.ndarray) -> np.ndarray:
    """MXFP8 reading of a vector (length a multiple of 32), float64."""
    v = _c(v, np.float64)
    out = np.empty_like(v)
    _load().orc_mx8_quantize(_p(v), v.size, _p(out))
    return out


def expert_ffn_mx8(w13_q, w13_s, w2_q, w2_s, x: np.ndarray, qx: bool = True, qh: bool = True) -> np.ndarray:
    """expert_ffn with the token rows (qx) and h (qh) read as MXFP8."""
    w13_q, w13_s, w2_q, w2_s = (_c(a, np.uint8) for a in (w13_q, w13_s, w2_q, w2_s))
    x = _c(x, np.uint16)
    n, H = x.shape
    I = w2_q.shape[1] * 2
    y = np.empty((n, H), np.uint16)
    _load().orc_expert_ffn_mx8(_p(w13_q), _p(w13_s), _p(w2_q), _p(w2_s), H, I, _p(x), n, _p(y), int(qx), int(qh))
    return y


# ------------------------------------------------------------ swaps/policy

def swap(row_map: np.ndarray, promote, demote):
    """Applies pairs in order to ``row_map`` (int32, in place).
    Returns the applied flags."""
    assert row_map.dtype == np.int32 and row_map.flags.c_contiguous
    promote = _c(promote, np.int32)
    demote = _c(demote, np.int32)
    applied = np.zeros(promote.size, np.int32)
    _load().orc_swap(_p(row_map), row_map.size, promote.size, _p(promote), _p(demote), _p(applied))
    return applied


def plan_restore(row_map, target, max_pairs: int):
    """Swap pairs that bring ``row_map``'s hot set back to ``target``'s
    (see moe_oracle.h).  Returns (promote, demote) int32 arrays, or None when
    the two maps hold different numbers of hot experts."""
    rm = _c(row_map, np.int32)
    tg = _c(target, np.int32)
    assert rm.size == tg.size
    pro = np.zeros(max(rm.size, 1), np.int32)
    dem = np.zeros(max(rm.size, 1), np.int32)
    n = _load().orc_plan_restore(_p(rm), _p(tg), rm.size, int(max_pairs), _p(pro), _p(dem))
    if n < 0:
        return None
    return pro[:n].copy(), dem[:n].copy()


class _Policy(C.Structure):
    _fields_ = [("E", C.c_int), ("last", C.c_void_p), ("acc", C.c_void_p), ("wsum", C.c_double)]


class Policy:
    """Decaying-average swap policy of one layer (see moe_oracle.h)."""

    def __init__(self, E: int, counts=None, read_every=64.0, half_life=500.0,
                 hysteresis=1.5, min_avg=8.0, max_pairs=2):
        self.E = E
        self.last = np.zeros(E, np.uint32)
        self.acc = np.zeros(E, np.float64)
        self.params = (float(read_every), float(half_life), float(hysteresis), float(min_avg), int(max_pairs))
        self.st = _Policy()
        c = None if counts is None else _c(counts, np.int32)
        _load().orc_policy_init(C.byref(self.st), E, _p(self.last), _p(self.acc),
                                None if c is None else _p(c))

    def read(self, counts: np.ndarray, row_map: np.ndarray):
        c = _c(counts, np.int32)
        rm = _c(row_map, np.int32)
        pro = np.zeros(self.E, np.int32)
        dem = np.zeros(self.E, np.int32)
        re, hl, hy, ma, mp = self.params
        n = _load().orc_policy_read(C.byref(self.st), _p(c), _p(rm), re, hl, hy, ma, mp, _p(pro), _p(dem))
        return pro[:n].copy(), dem[:n].copy()


def expert_bytes(H: int, I: int) -> int:
    return int(_load().orc_expert_bytes(H, I))


def num_threads() -> int:
    return int(_load().orc_num_threads())


def set_num_threads(n: int) -> None:
    _load().orc_set_num_threads(int(n))
