// Route, split and count: top-k routing with softmax weights, the residency
// split into per-bank pick lists, and the masked relaxed usage counter.
//
// Write-ups: "vLLM: Pin Hot Experts", Results (split each token's k expert ids
// by residency and remap through the row map); "We Built the Counter",
// section 2 (one masked relaxed atomic add per routed pick into the
// [layers x experts] table inside the split kernel; only steps of at most 256
// tokens are counted).
//
// Pick lists: for each bank, the active rows in increasing row order and, per
// row, its picks as slot indices s = t*k + j in increasing order.  The order
// is a pure function of (ids, row map), so the FFN that consumes it sees the
// same token order for an expert whichever bank holds it.
#include "moe_internal.cuh"

#include <climits>

namespace moe {

namespace {

constexpr int kMaxLanesVals = 32;   // E <= 1024 => at most 32 logits per lane
constexpr int kMaxK = 16;

struct WsPtrs {
    int32_t *hdr, *act_row, *act_off, *picks, *epos;
    int P;
};

__device__ __forceinline__ void red_relaxed_add(int32_t *p, int v) {
    asm volatile("red.relaxed.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ bool better(float va, int ea, float vb, int eb) {
    return va > vb || (va == vb && ea < eb);
}

// One warp routes one token: k rounds of a warp-wide argmax (larger logit
// first, ties to the lower expert id), then fp32 softmax over the k picks.
// A NaN logit is read as -infinity (ranked below every number, weight
// exp(-inf) = 0 beside a finite first pick), so the k ids are always valid.
// Lane j < k returns pick j in (*id_out, *w_out); other lanes return -1.
__device__ __forceinline__ void warp_route_token(const float *__restrict__ l, int E, int k, int lane,
                                                 int *id_out, float *w_out) {
    float lv[kMaxLanesVals];
    uint32_t taken = 0;
#pragma unroll
    for (int i = 0; i < kMaxLanesVals; ++i) {
        int e = lane + 32 * i;
        const float v = e < E ? l[e] : -INFINITY;
        lv[i] = isnan(v) ? -INFINITY : v;
        if (e >= E) taken |= 1u << i;
    }
    float sel_v[kMaxK];
    int sel_e[kMaxK];
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
        if (j < k) {
            float bv = -INFINITY;
            int be = INT_MAX;
#pragma unroll
            for (int i = 0; i < kMaxLanesVals; ++i) {
                int e = lane + 32 * i;
                if (!((taken >> i) & 1u) && better(lv[i], e, bv, be)) {
                    bv = lv[i];
                    be = e;
                }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                float ov = __shfl_xor_sync(0xffffffffu, bv, off);
                int oe = __shfl_xor_sync(0xffffffffu, be, off);
                if (better(ov, oe, bv, be)) {
                    bv = ov;
                    be = oe;
                }
            }
            if ((be & 31) == lane) taken |= 1u << (be >> 5);
            sel_v[j] = bv;
            sel_e[j] = be;
        }
    }
    // softmax over the picks, shifted by the largest (pick 0), summed in j order
    float ex[kMaxK];
    float sum = 0.0f;
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
        if (j < k) {
            ex[j] = expf(sel_v[j] - sel_v[0]);
            sum = sum + ex[j];
        }
    }
    int myid = -1;
    float myw = 0.0f;
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
        if (j < k && j == lane) {
            myid = sel_e[j];
            myw = __fdiv_rn(ex[j], sum);
        }
    }
    *id_out = myid;
    *w_out = myw;
}

// Build the active-row lists of bank b from per-expert pick counts.
// Warp-level: rows in increasing order, chunks of 32 with ballot + scan.
__device__ void warp_scan_bank(int b, int rows, int E, const int32_t *rowexp, const int32_t *cnt,
                               int32_t *epos, WsPtrs ws, int lane) {
    const int P = ws.P;
    int na = 0, np = 0;
    for (int base = 0; base < rows; base += 32) {
        int r = base + lane;
        int e = r < rows ? rowexp[b * E + r] : -1;
        int c = e >= 0 ? cnt[e] : 0;
        unsigned act = __ballot_sync(0xffffffffu, c > 0);
        int inc = c;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            int v = __shfl_up_sync(0xffffffffu, inc, off);
            if (lane >= off) inc += v;
        }
        if (c > 0) {
            int a = na + __popc(act & ((1u << lane) - 1u));
            ws.act_row[b * P + a] = r;
            ws.act_off[b * (P + 1) + a + 1] = np + inc;
            epos[e] = np + inc - c;
        }
        na += __popc(act);
        np += __shfl_sync(0xffffffffu, inc, 31);
    }
    if (lane == 0) {
        ws.act_off[b * (P + 1)] = 0;
        ws.hdr[kHdrNAct + b] = na;
        ws.hdr[kHdrNPicks + b] = np;
    }
}

// Fill expert e's picks (in slot order) starting at pos in bank b's list.
__device__ __forceinline__ void warp_fill_expert(int e, int b, int pos, const int32_t *ids, WsPtrs ws,
                                                 int lane) {
    const int P = ws.P;
    for (int base = 0; base < P; base += 32) {
        int s = base + lane;
        bool hit = s < P && ids[s] == e;
        unsigned msk = __ballot_sync(0xffffffffu, hit);
        if (hit) ws.picks[b * P + pos + __popc(msk & ((1u << lane) - 1u))] = s;
        pos += __popc(msk);
    }
}

// Small steps (T <= 32, T*k <= 4096): route, count, scan and fill in one
// CTA of 8 warps.
__global__ void __launch_bounds__(256) route_split_small(
    const float *__restrict__ logits, int T, int E, int k, const int32_t *__restrict__ rowmap,
    int n_hot, int n_cold, int32_t *counts, int32_t *__restrict__ ids, float *__restrict__ w, WsPtrs ws) {
    extern __shared__ int32_t sm[];
    const int P = ws.P;
    int32_t *s_ids = sm;            // [P]
    int32_t *cnt = s_ids + P;       // [E]
    int32_t *rmap = cnt + E;        // [E]
    int32_t *rowexp = rmap + E;     // [2][E]
    int32_t *epos = rowexp + 2 * E; // [E]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;

    for (int t = warp; t < T; t += nwarps) {
        int id;
        float wv;
        warp_route_token(logits + (size_t)t * E, E, k, lane, &id, &wv);
        if (lane < k) {
            ids[t * k + lane] = id;
            w[t * k + lane] = wv;
            s_ids[t * k + lane] = id;
            if (counts) red_relaxed_add(counts + id, 1);
        }
    }
    for (int e = tid; e < E; e += blockDim.x) {
        cnt[e] = 0;
        int m = rowmap[e];
        rmap[e] = m;
        if (m >= 0) rowexp[m] = e;
        else rowexp[E + (-1 - m)] = e;
    }
    __syncthreads();
    for (int s = tid; s < P; s += blockDim.x) atomicAdd(&cnt[s_ids[s]], 1);
    __syncthreads();
    if (warp < 2) warp_scan_bank(warp, warp == 0 ? n_hot : n_cold, E, rowexp, cnt, epos, ws, lane);
    __syncthreads();
    for (int e = warp; e < E; e += nwarps) {
        if (cnt[e] == 0) continue;
        int m = rmap[e];
        warp_fill_expert(e, m >= 0 ? 0 : 1, epos[e], s_ids, ws, lane);
    }
}

// Large steps, stage 1: one warp per token.
__global__ void __launch_bounds__(256) route_tokens(const float *__restrict__ logits, int T, int E, int k,
                                                   int32_t *counts, int32_t *__restrict__ ids,
                                                   float *__restrict__ w, int32_t *ecnt) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (t >= T) return;
    int id;
    float wv;
    warp_route_token(logits + (size_t)t * E, E, k, lane, &id, &wv);
    if (lane < k) {
        ids[t * k + lane] = id;
        w[t * k + lane] = wv;
        if (counts) red_relaxed_add(counts + id, 1);
        red_relaxed_add(ecnt + id, 1);   // picks per expert for the split (order-free)
    }
}

// Large steps, stage 2: the active-row scan over the per-expert counts (one CTA).
__global__ void __launch_bounds__(1024) split_scan(const int32_t *__restrict__ ecnt, int E,
                                                   const int32_t *__restrict__ rowmap, int n_hot,
                                                   int n_cold, WsPtrs ws) {
    extern __shared__ int32_t sm[];
    int32_t *cnt = sm;              // [E]
    int32_t *rowexp = cnt + E;      // [2][E]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int e = tid; e < E; e += blockDim.x) {
        cnt[e] = ecnt[e];
        ws.epos[e] = -1;
        int m = rowmap[e];
        if (m >= 0) rowexp[m] = e;
        else rowexp[E + (-1 - m)] = e;
    }
    __syncthreads();
    if (warp < 2) warp_scan_bank(warp, warp == 0 ? n_hot : n_cold, E, rowexp, cnt, ws.epos, ws, lane);
}

// Large steps, stage 3: one warp per active expert fills its picks.
__global__ void __launch_bounds__(256) split_fill(const int32_t *__restrict__ ids, int E,
                                                  const int32_t *__restrict__ rowmap, WsPtrs ws) {
    const int lane = threadIdx.x & 31;
    const int e = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (e >= E) return;
    int pos = ws.epos[e];
    if (pos < 0) return;
    warp_fill_expert(e, rowmap[e] >= 0 ? 0 : 1, pos, ids, ws, lane);
}

}  // namespace

int launch_route_split(moe_ctx *ctx, int layer, const float *logits, int T, int count_on,
                       int32_t *ids, float *w, uint8_t *ws_base, cudaStream_t s) {
    const Geom &g = ctx->g;
    const Layer &L = ctx->layers[layer];
    WsLayout lay = ws_layout(g, T);
    WsPtrs ws;
    ws.hdr = (int32_t *)(ws_base + lay.hdr);
    ws.act_row = (int32_t *)(ws_base + lay.act_row);
    ws.act_off = (int32_t *)(ws_base + lay.act_off);
    ws.picks = (int32_t *)(ws_base + lay.picks);
    ws.epos = (int32_t *)(ws_base + lay.epos);
    ws.P = T * g.k;
    if (T == 0) {
        MOE_CUDA_TRY(cudaMemsetAsync(ws.hdr, 0, kHdrWords * 4, s));
        return MOE_OK;
    }
    int32_t *counts = (count_on && T <= g.count_tmax) ? ctx->counts_dev + (size_t)layer * g.E : nullptr;
    const int P = ws.P;
    if (T <= 32 && P <= 4096) {
        size_t smem = sizeof(int32_t) * ((size_t)P + 5 * (size_t)g.E);
        route_split_small<<<1, 256, smem, s>>>(logits, T, g.E, g.k, L.rowmap_dev, L.n_hot, L.n_cold,
                                                counts, ids, w, ws);
        MOE_LAUNCH_CHECK();
        return MOE_OK;
    }
    int32_t *ecnt = (int32_t *)(ws_base + lay.ecnt);
    MOE_CUDA_TRY(cudaMemsetAsync(ecnt, 0, sizeof(int32_t) * g.E, s));
    route_tokens<<<(T + 7) / 8, 256, 0, s>>>(logits, T, g.E, g.k, counts, ids, w, ecnt);
    MOE_LAUNCH_CHECK();
    split_scan<<<1, 1024, sizeof(int32_t) * 3 * (size_t)g.E, s>>>(ecnt, g.E, L.rowmap_dev, L.n_hot,
                                                                  L.n_cold, ws);
    MOE_LAUNCH_CHECK();
    split_fill<<<(g.E + 7) / 8, 256, 0, s>>>(ids, g.E, L.rowmap_dev, ws);
    MOE_LAUNCH_CHECK();
    return MOE_OK;
}

// Two-element row-map write, ordered on the stream after a swap's copies.
__global__ void rowmap_write_kernel(int32_t *rowmap, int32_t e0, int32_t v0, int32_t e1, int32_t v1) {
    if (threadIdx.x == 0 && blockIdx.x == 0) {
        rowmap[e0] = v0;
        rowmap[e1] = v1;
    }
}

int launch_rowmap_write(int32_t *rowmap_dev, int32_t e0, int32_t v0, int32_t e1, int32_t v1,
                        cudaStream_t s) {
    rowmap_write_kernel<<<1, 32, 0, s>>>(rowmap_dev, e0, v0, e1, v1);
    MOE_LAUNCH_CHECK();
    return MOE_OK;
}

}  // namespace moe
