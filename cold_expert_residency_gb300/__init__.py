"""Split-residency routed MoE layer for one GB300 GPU -- Python binding.

A thin ctypes binding over ``libmoe_residency.so`` (C ABI declared in
``include/moe_residency.h``).  Functions keep the C names; arguments are
marshalled only: torch tensors and numpy arrays become pointers, a torch
stream becomes its ``cudaStream_t``.  Every step of the layer runs in the
library's CUDA kernels; there is no Python or CPU fallback -- a missing
library raises ``LibraryMissing``.

PyTorch is used by callers for device memory and streams only.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from ._build import LIB as _LIB_PATH, build  # noqa: F401

MOE_OK, MOE_EINVAL, MOE_ENOMEM, MOE_ECUDA, MOE_ESTALE, MOE_ETIMEOUT, MOE_ESTATE = 0, -1, -2, -3, -4, -5, -6
MOE_BANK_HOT, MOE_BANK_COLD, MOE_BANK_BOTH = 0, 1, 2
MOE_FFN_TCGEN05, MOE_FFN_SIMT = 0, 1
MOE_FAULT_NONE, MOE_FAULT_WITHHOLD_COPY = 0, 1
MOE_ACT_E4M3X2, MOE_ACT_MXFP8 = 0, 1

_lib = None


class LibraryMissing(RuntimeError):
    pass


class MoeError(RuntimeError):
    def __init__(self, fn, code, msg):
        super().__init__(f"{fn} failed ({code}): {msg}")
        self.code = code


class moe_geom(C.Structure):
    _fields_ = [("layers", C.c_int32), ("experts", C.c_int32), ("top_k", C.c_int32),
                ("hidden", C.c_int32), ("inter", C.c_int32), ("count_tmax", C.c_int32),
                ("max_tokens", C.c_int32)]


def lib():
    """The loaded library; raises LibraryMissing if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise LibraryMissing(f"{_LIB_PATH} is missing: run cold_expert_residency_gb300.build() "
                             "(the CUDA library is required; there is no fallback)")
    L = C.CDLL(_LIB_PATH)
    P, i32, i64, sz = C.c_void_p, C.c_int, C.c_int64, C.c_size_t
    sig = {
        "moe_last_error": (C.c_char_p, []),
        "moe_expert_bytes": (i64, [C.c_int32, C.c_int32]),
        "moe_pack_expert": (i32, [C.c_int32, C.c_int32, P, P, P, P, P]),
        "moe_create": (i32, [C.POINTER(moe_geom), i32, C.POINTER(P)]),
        "moe_destroy": (i32, [P]),
        "moe_set_ffn_impl": (i32, [P, i32]),
        "moe_set_act_format": (i32, [P, i32]),
        "moe_set_cold_staging": (i32, [P, i32]),
        "moe_read_stage": (i32, [P, P, i32, P, P]),
        "moe_init_banks": (i32, [P, i32, P, P, P, P, P, P]),
        "moe_workspace_bytes": (i32, [P, i32, C.POINTER(sz)]),
        "moe_route_split_count": (i32, [P, i32, P, i32, i32, P, P, P, P]),
        "moe_read_split": (i32, [P, P, i32, i32, P, P, P, P, P, P]),
        "moe_expert_ffn_bank": (i32, [P, i32, i32, P, i32, P, P, P]),
        "moe_expert_ffn_bank_static": (i32, [P, i32, i32, P, i32, P, P, P]),
        "moe_static_scratch_bytes": (sz, []),
        "moe_finalize": (i32, [P, P, i32, i32, i32, P, P]),
        "moe_router_logits": (i32, [P, P, P, P, i32, i32, i32, P, P]),
        "moe_step_scratch_bytes": (i32, [P, i32, C.POINTER(sz)]),
        "moe_layer_step_host": (i32, [P, i32, P, P, i32, i32, P, P, P]),
        "moe_swap_rows": (i32, [P, i32, i32, P, P, P, P]),
        "moe_read_counts": (i32, [P, P, P]),
        "moe_reset_counts": (i32, [P, P]),
        "moe_bank_rows": (i32, [P, i32, P, P]),
        "moe_get_rowmap": (i32, [P, i32, P]),
        "moe_read_rowmap_device": (i32, [P, i32, P, P]),
        "moe_read_bank_row": (i32, [P, i32, i32, i32, P, P]),
        "moe_probe_link": (i32, [P, sz, i32, C.POINTER(C.c_double), C.POINTER(C.c_double)]),
        "moe_device_status": (i32, [P, C.POINTER(C.c_int32)]),
        "moe_kernel_launches": (i64, []),
        "moe_memory_in_use": (i32, [C.POINTER(i64), C.POINTER(i64)]),
        "moe_set_wait_limit": (i32, [P, C.c_uint64]),
        "moe_inject_fault": (i32, [P, i32]),
        "moe_policy_create": (i32, [i32, C.c_double, C.c_double, C.c_double, C.c_double, i32, P, C.POINTER(P)]),
        "moe_policy_destroy": (i32, [P]),
        "moe_policy_read": (i32, [P, P, P, P, P]),
        "moe_plan_restore": (i32, [i32, P, P, i32, P, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


def exported_symbols():
    """Names the C header declares (used by the ABI tests)."""
    hdr = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                       "moe_residency.h")
    import re
    names = []
    with open(hdr) as f:
        for m in re.finditer(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(moe_[a-z_0-9]+)\s*\(", f.read(), re.M):
            names.append(m.group(1))
    return names


# --------------------------------------------------------------- marshalling

def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if isinstance(x, np.ndarray):
        if not x.flags.c_contiguous:
            raise ValueError("arrays must be C-contiguous")
        return x.ctypes.data
    if hasattr(x, "data_ptr"):
        if hasattr(x, "is_contiguous") and not x.is_contiguous():
            raise ValueError("tensors must be contiguous")
        return x.data_ptr()
    raise TypeError(f"cannot pass {type(x)} as a pointer")


def _stream(s):
    if s is None:
        try:
            import torch
            if torch.cuda.is_available():
                return torch.cuda.current_stream().cuda_stream
        except ImportError:
            pass
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _err(fn, rc):
    if rc < 0:
        raise MoeError(fn, rc, lib().moe_last_error().decode())
    return rc


# ------------------------------------------------------------------- the ABI

def moe_expert_bytes(hidden, inter):
    return int(lib().moe_expert_bytes(hidden, inter))


def moe_pack_expert(hidden, inter, w13_q, w13_s, w2_q, w2_s):
    """One expert's logical MXFP4 arrays (host numpy uint8) -> the bytes of
    its bank row (numpy uint8 [moe_expert_bytes(hidden, inter)])."""
    import numpy as np
    arrs = [np.ascontiguousarray(a, dtype=np.uint8) for a in (w13_q, w13_s, w2_q, w2_s)]
    out = np.empty(moe_expert_bytes(hidden, inter), np.uint8)
    _err("moe_pack_expert", lib().moe_pack_expert(hidden, inter, *[a.ctypes.data for a in arrs], out.ctypes.data))
    return out


def moe_create(layers, experts, top_k, hidden, inter, max_tokens, count_tmax=256, device=0):
    g = moe_geom(layers, experts, top_k, hidden, inter, count_tmax, max_tokens)
    out = C.c_void_p()
    _err("moe_create", lib().moe_create(C.byref(g), device, C.byref(out)))
    return out.value


def moe_destroy(ctx):
    return _err("moe_destroy", lib().moe_destroy(ctx))


def moe_set_ffn_impl(ctx, impl):
    return _err("moe_set_ffn_impl", lib().moe_set_ffn_impl(ctx, impl))


def moe_set_cold_staging(ctx, slots):
    return _err("moe_set_cold_staging", lib().moe_set_cold_staging(ctx, slots))


def moe_read_stage(ctx, ws, T, stream=None):
    """Cold-bank rows copied into the staging pool's slots by the last staged
    FFN call on this workspace (-1: slot unused)."""
    rows = np.zeros(64, np.int32)
    _err("moe_read_stage", lib().moe_read_stage(ctx, _ptr(ws), T, _ptr(rows), _stream(stream)))
    return rows


def moe_set_act_format(ctx, fmt):
    return _err("moe_set_act_format", lib().moe_set_act_format(ctx, fmt))


def moe_init_banks(ctx, layer, w13_q, w13_s, w2_q, w2_s, is_hot, stream=None):
    arrs = [np.ascontiguousarray(a, dtype=np.uint8) for a in (w13_q, w13_s, w2_q, w2_s, is_hot)]
    return _err("moe_init_banks", lib().moe_init_banks(ctx, layer, *(_ptr(a) for a in arrs), _stream(stream)))


def moe_workspace_bytes(ctx, T):
    n = C.c_size_t()
    _err("moe_workspace_bytes", lib().moe_workspace_bytes(ctx, T, C.byref(n)))
    return n.value


def moe_route_split_count(ctx, layer, logits, T, count_on, ids, w, ws, stream=None):
    return _err("moe_route_split_count", lib().moe_route_split_count(
        ctx, layer, _ptr(logits), T, int(count_on), _ptr(ids), _ptr(w), _ptr(ws), _stream(stream)))


def moe_read_split(ctx, ws, T, k, bank, stream=None):
    """One bank's pick lists: dict(n_act, n_picks, act_row, act_off, picks)."""
    P = T * k
    na, npk = C.c_int32(), C.c_int32()
    act_row = np.zeros(max(P, 1), np.int32)
    act_off = np.zeros(P + 1, np.int32)
    picks = np.zeros(max(P, 1), np.int32)
    _err("moe_read_split", lib().moe_read_split(ctx, _ptr(ws), T, bank, C.byref(na), C.byref(npk), _ptr(act_row),
                                                _ptr(act_off), _ptr(picks), _stream(stream)))
    return dict(n_act=na.value, n_picks=npk.value, act_row=act_row[:na.value].copy(),
                act_off=act_off[:na.value + 1].copy(), picks=picks[:npk.value].copy())


def moe_expert_ffn_bank(ctx, layer, bank, x, T, ws, Y, stream=None):
    return _err("moe_expert_ffn_bank", lib().moe_expert_ffn_bank(
        ctx, layer, bank, _ptr(x), T, _ptr(ws), _ptr(Y), _stream(stream)))


def moe_expert_ffn_bank_static(ctx, layer, bank, x, T, split_ws, Y, stream=None):
    """Allocation-free FFN over one bank: scratch lives in the library's
    static device area (see the C header)."""
    return _err("moe_expert_ffn_bank_static", lib().moe_expert_ffn_bank_static(
        ctx, layer, bank, _ptr(x), T, _ptr(split_ws), _ptr(Y), _stream(stream)))


def moe_static_scratch_bytes():
    return int(lib().moe_static_scratch_bytes())


def moe_step_scratch_bytes(ctx, T):
    n = C.c_size_t()
    _err("moe_step_scratch_bytes", lib().moe_step_scratch_bytes(ctx, T, C.byref(n)))
    return n.value


def moe_layer_step_host(ctx, layer, logits, x, T, count_on, out, scratch, stream=None):
    """One layer-step from host buffers (logits fp32 [T][E], x bf16 bits
    [T][H] in, out bf16 bits [T][H]); out is valid once the stream has
    reached the end of the call."""
    return _err("moe_layer_step_host", lib().moe_layer_step_host(
        ctx, layer, _ptr(logits), _ptr(x), T, int(count_on), _ptr(out), _ptr(scratch), _stream(stream)))


def moe_finalize(Y, w, T, k, H, out, stream=None):
    return _err("moe_finalize", lib().moe_finalize(_ptr(Y), _ptr(w), T, k, H, _ptr(out), _stream(stream)))


def moe_router_logits(ctx, x, w_router, bias, T, E, H, logits, stream=None):
    return _err("moe_router_logits", lib().moe_router_logits(ctx, _ptr(x), _ptr(w_router), _ptr(bias), T, E, H,
                                                             _ptr(logits), _stream(stream)))


def moe_swap_rows(ctx, layer, promote, demote, stream=None):
    """Returns (number applied, applied flags as an int32 array)."""
    pro = np.ascontiguousarray(promote, dtype=np.int32)
    dem = np.ascontiguousarray(demote, dtype=np.int32)
    applied = np.zeros(pro.size, np.int32)
    n = _err("moe_swap_rows", lib().moe_swap_rows(ctx, layer, pro.size, _ptr(pro), _ptr(dem), _ptr(applied),
                                                  _stream(stream)))
    return n, applied


def moe_read_counts(ctx, layers, experts, stream=None):
    out = np.zeros((layers, experts), np.int32)
    _err("moe_read_counts", lib().moe_read_counts(ctx, _ptr(out), _stream(stream)))
    return out


def moe_reset_counts(ctx, stream=None):
    return _err("moe_reset_counts", lib().moe_reset_counts(ctx, _stream(stream)))


def moe_bank_rows(ctx, layer):
    h, c = C.c_int32(), C.c_int32()
    _err("moe_bank_rows", lib().moe_bank_rows(ctx, layer, C.byref(h), C.byref(c)))
    return h.value, c.value


def moe_get_rowmap(ctx, layer, experts):
    out = np.zeros(experts, np.int32)
    _err("moe_get_rowmap", lib().moe_get_rowmap(ctx, layer, _ptr(out)))
    return out


def moe_read_rowmap_device(ctx, layer, experts, stream=None):
    out = np.zeros(experts, np.int32)
    _err("moe_read_rowmap_device", lib().moe_read_rowmap_device(ctx, layer, _ptr(out), _stream(stream)))
    return out


def moe_read_bank_row(ctx, layer, bank, row, nbytes, stream=None):
    out = np.zeros(nbytes, np.uint8)
    _err("moe_read_bank_row", lib().moe_read_bank_row(ctx, layer, bank, row, _ptr(out), _stream(stream)))
    return out


def moe_probe_link(ctx, nbytes=1 << 30, iters=5):
    """(host-link read GB/s, HBM read GB/s) measured by the library's probe kernel."""
    a, b = C.c_double(), C.c_double()
    _err("moe_probe_link", lib().moe_probe_link(ctx, nbytes, iters, C.byref(a), C.byref(b)))
    return a.value, b.value


def moe_device_status(ctx):
    s = C.c_int32()
    _err("moe_device_status", lib().moe_device_status(ctx, C.byref(s)))
    return s.value


def moe_kernel_launches():
    return int(lib().moe_kernel_launches())


def moe_memory_in_use():
    """(device bytes, pinned host bytes) the library holds in this process."""
    d, p = C.c_int64(), C.c_int64()
    _err("moe_memory_in_use", lib().moe_memory_in_use(C.byref(d), C.byref(p)))
    return d.value, p.value


def moe_set_wait_limit(ctx, ns):
    return _err("moe_set_wait_limit", lib().moe_set_wait_limit(ctx, int(ns)))


def moe_inject_fault(ctx, kind):
    return _err("moe_inject_fault", lib().moe_inject_fault(ctx, kind))


def moe_plan_restore(row_map, target, max_pairs):
    """Swap pairs (promote, demote) that bring row_map's hot set back to
    target's, at most max_pairs of them (moe_plan_restore ABI)."""
    rm = np.ascontiguousarray(row_map, dtype=np.int32)
    tg = np.ascontiguousarray(target, dtype=np.int32)
    if rm.shape != tg.shape:
        raise ValueError("row_map and target differ in length")
    pro = np.zeros(max(int(max_pairs), 1), np.int32)
    dem = np.zeros(max(int(max_pairs), 1), np.int32)
    n = _err("moe_plan_restore", lib().moe_plan_restore(rm.size, _ptr(rm), _ptr(tg), int(max_pairs),
                                                        _ptr(pro), _ptr(dem)))
    return pro[:n].copy(), dem[:n].copy()


class moe_policy:
    """Native decaying-average swap policy of one layer (moe_policy_* ABI)."""

    def __init__(self, experts, read_every=64.0, half_life=500.0, hysteresis=1.5, min_avg=8.0,
                 max_pairs=2, counts_now=None):
        self.E = experts
        h = C.c_void_p()
        c = None if counts_now is None else np.ascontiguousarray(counts_now, dtype=np.int32)
        _err("moe_policy_create", lib().moe_policy_create(experts, read_every, half_life, hysteresis, min_avg,
                                                          max_pairs, _ptr(c), C.byref(h)))
        self.h = h.value

    def read(self, counts, row_map):
        c = np.ascontiguousarray(counts, dtype=np.int32)
        rm = np.ascontiguousarray(row_map, dtype=np.int32)
        pro = np.zeros(self.E, np.int32)
        dem = np.zeros(self.E, np.int32)
        n = _err("moe_policy_read", lib().moe_policy_read(self.h, _ptr(c), _ptr(rm), _ptr(pro), _ptr(dem)))
        return pro[:n].copy(), dem[:n].copy()

    def __del__(self):
        try:
            if self.h:
                lib().moe_policy_destroy(self.h)
        except Exception:
            pass
