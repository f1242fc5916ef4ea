"""Layer-step orchestration over the C ABI (streams and buffers only).

One layer-step ("vLLM: Pin Hot Experts", Results):
    [router GEMM                     (moe_router_logits, optional)]
    route + split + count            (moe_route_split_count, main stream)
    expert FFN over both banks       (moe_expert_ffn_bank with MOE_BANK_BOTH:
                                      one launch per GEMM, main stream)
    finalize                         (moe_finalize, main stream)
The hot bank streams HBM and the cold bank streams the host link, so the two
run concurrently: inside the one call by default, or as two calls on two
streams joined by events.  Both forms, and the two calls one after the other,
give bit-identical rows.  PyTorch provides the device buffers and streams.
"""
from __future__ import annotations

import torch

from . import (MOE_BANK_BOTH, MOE_BANK_COLD, MOE_BANK_HOT, moe_expert_ffn_bank, moe_finalize,
               moe_get_rowmap, moe_plan_restore, moe_route_split_count, moe_router_logits, moe_swap_rows,
               moe_workspace_bytes)


class StepBuffers:
    """Device buffers of one layer-step of up to T_max tokens."""

    def __init__(self, ctx, E, k, H, T_max, device="cuda"):
        self.E, self.k, self.H, self.T_max = E, k, H, T_max
        dev = torch.device(device)
        self.logits = torch.zeros((T_max, E), dtype=torch.float32, device=dev)
        self.x = torch.zeros((T_max, H), dtype=torch.int16, device=dev)        # bf16 bits
        self.ids = torch.zeros((T_max, k), dtype=torch.int32, device=dev)
        self.w = torch.zeros((T_max, k), dtype=torch.float32, device=dev)
        self.Y = torch.zeros((T_max, k, H), dtype=torch.int16, device=dev)     # bf16 bits
        self.out = torch.zeros((T_max, H), dtype=torch.int16, device=dev)      # bf16 bits
        nbytes = moe_workspace_bytes(ctx, T_max)
        self.ws = torch.zeros(nbytes + 256, dtype=torch.uint8, device=dev)
        off = (-self.ws.data_ptr()) % 256
        self.ws_ptr = self.ws.data_ptr() + off


class LayerStep:
    """Runs layer-steps on a main stream plus a second stream for the cold bank."""

    def __init__(self, ctx, E, k, H, T_max, device="cuda"):
        self.ctx = ctx
        self.buf = StepBuffers(ctx, E, k, H, T_max, device)
        # high priority: the cold bank's few CTAs get SM slots first and keep
        # the host link busy while the hot bank fills the rest of the GPU
        self.cold_stream = torch.cuda.Stream(device=device, priority=-1)
        self.ev_routed = torch.cuda.Event()
        self.ev_cold = torch.cuda.Event()

    def run(self, layer, T, count_on=True, stream=None, split=True, fused=True, router=None):
        """Enqueue one layer-step of T tokens from buf.logits / buf.x into
        buf.out (and buf.ids, buf.w, buf.Y).  By default one FFN call covers
        both banks (its launches stream the cold bank from one CTA per SM
        and the hot bank from the others); ``fused=False`` runs the two banks'
        calls on two streams at once, and with ``split=False`` one after the
        other on the main stream.  ``router=(w_router, bias)`` (device bf16
        [E][H] and fp32 [E] or None) first computes buf.logits from buf.x by
        the router GEMM."""
        b = self.buf
        main = stream if stream is not None else torch.cuda.current_stream()
        if router is not None:
            w_router, bias = router
            moe_router_logits(self.ctx, b.x, w_router, bias, T, b.E, b.H, b.logits, main)
        moe_route_split_count(self.ctx, layer, b.logits, T, count_on, b.ids, b.w, b.ws_ptr, main)
        if fused:
            moe_expert_ffn_bank(self.ctx, layer, MOE_BANK_BOTH, b.x, T, b.ws_ptr, b.Y, main)
        elif split:
            self.ev_routed.record(main)
            self.cold_stream.wait_event(self.ev_routed)
            moe_expert_ffn_bank(self.ctx, layer, MOE_BANK_COLD, b.x, T, b.ws_ptr, b.Y, self.cold_stream)
            self.ev_cold.record(self.cold_stream)
            moe_expert_ffn_bank(self.ctx, layer, MOE_BANK_HOT, b.x, T, b.ws_ptr, b.Y, main)
            main.wait_event(self.ev_cold)
        else:
            moe_expert_ffn_bank(self.ctx, layer, MOE_BANK_HOT, b.x, T, b.ws_ptr, b.Y, main)
            moe_expert_ffn_bank(self.ctx, layer, MOE_BANK_COLD, b.x, T, b.ws_ptr, b.Y, main)
        moe_finalize(b.Y, b.w, T, b.k, b.H, b.out, main)


def restore_placement(ctx, layer, saved, budget=8, stream=None):
    """Between steps: queue at most ``budget`` swaps that move the layer's
    hot set toward the saved row map's (one saved by moe_get_rowmap, e.g. at
    boot).  Returns the number of swaps applied; 0 once the hot set is
    restored.  "We Built the Counter", section 2: a return to the start-up
    placement, at most 8 swaps per step."""
    row_map = moe_get_rowmap(ctx, layer, len(saved))
    promote, demote = moe_plan_restore(row_map, saved, budget)
    if promote.size == 0:
        return 0
    n, _ = moe_swap_rows(ctx, layer, promote, demote, stream)
    return n
