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
//
// Decode steps (at most 256 tokens) build the lists in one CTA of 512 threads
// whose work is sized by the step's picks, not by the experts: one
// block-wide scan over the per-row pick counts gives every active row its
// list position and offset, and each pick's place adds the number of earlier
// picks of its expert (read from the expert's token mask up to 32 tokens,
// counted beyond).  Steps of at most 32 tokens route in the same CTA; larger
// decode steps route with one warp per token across CTAs first.  Larger
// steps (prefill) route the same way, counting picks per expert and per
// (expert, 32-token chunk), then build the lists in three more kernels: the
// active-row scan, each chunk's first place per expert, and the placement of
// each chunk's picks in slot order.
#include "moe_internal.cuh"

#include <climits>

namespace moe {

namespace {

constexpr int kSmallThreads = 512;
constexpr int kFusedMaxT = 32;      // one CTA routes and splits
constexpr int kSmallMaxT = 256;     // routing over many CTAs, then one CTA splits
constexpr int kSmallMaxP = 4096;

struct WsPtrs {
    int32_t *hdr, *act_row, *act_off, *picks, *epos;
    int P;
};

__device__ __forceinline__ void red_relaxed_add(int32_t *p, int v) {
    asm volatile("red.relaxed.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// A token's logits as one lane holds them: experts lane, lane+32, ... (NV
// values, NV*32 >= E), loaded together so their latencies overlap.  A NaN
// logit is read as -infinity.
template <int NV>
__device__ __forceinline__ void load_logits(const float *__restrict__ l, int E, int lane, float (&v)[NV]) {
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int e = lane + 32 * i;
        const float raw = e < E ? l[e] : -INFINITY;
        v[i] = isnan(raw) ? -INFINITY : raw;
    }
}

// Order-preserving 32-bit key of a logit: a larger key for a larger value,
// -0.0 read as +0.0 (equal logits must tie, so the lower expert id decides).
__device__ __forceinline__ uint32_t logit_key(float f) {
    const uint32_t b = __float_as_uint(f == 0.0f ? 0.0f : f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_logit(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// A lane's best two values not yet picked, as (value, index) with index NV
// for none: higher value first, the lower index on equal values (a lane's
// expert ids rise with the index).  One pass in index order.
template <int NV>
__device__ __forceinline__ void lane_top2(const float (&v)[NV], uint32_t taken, float &v1, int &i1, float &v2,
                                          int &i2) {
    v1 = -INFINITY;
    v2 = -INFINITY;
    i1 = NV;
    i2 = NV;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        if ((taken >> i) & 1u) continue;
        if (i1 == NV || v[i] > v1) {
            v2 = v1;
            i2 = i1;
            v1 = v[i];
            i1 = i;
        } else if (i2 == NV || v[i] > v2) {
            v2 = v[i];
            i2 = i;
        }
    }
}

// One warp routes one token from its logits in registers, in k rounds.  Each
// lane offers its best value not yet picked; one warp reduction takes the
// largest key over the lanes, a second the lowest expert id among the lanes
// that offer it, and the lane that held the pick marks it picked and offers
// its second best next.  A lane whose second best is used up too finds its
// next two again (the warp takes that branch only when some lane needs it).
// NaN logits arrive as -infinity (ranked below every number, weight
// exp(-inf) = 0 beside a finite first pick), so the k ids are always valid.
// Then fp32 softmax over the k picks, shifted by the first and summed in pick
// order.  Lane j < k returns pick j in (*id_out, *w_out); other lanes
// return -1.
template <int KM, int NV>
__device__ __forceinline__ void warp_route_token(const float (&v)[NV], int E, int k, int lane, int *id_out,
                                                 float *w_out) {
    uint32_t taken = 0;   // bit i: value i of this lane picked, or past E
#pragma unroll
    for (int i = 0; i < NV; ++i)
        if (lane + 32 * i >= E) taken |= 1u << i;
    float v1, v2;
    int i1, i2;
    lane_top2<NV>(v, taken, v1, i1, v2, i2);
    bool second = true;   // (v2, i2) is this lane's second best
    float sel_v[KM];
    int sel_e[KM];
#pragma unroll
    for (int j = 0; j < KM; ++j) {
        if (j < k) {
            // a lane without a candidate offers key 0, below every logit's key
            const bool has = i1 < NV;
            const uint32_t key = has ? logit_key(v1) : 0u;
            const uint32_t mk = __reduce_max_sync(0xffffffffu, key);
            const uint32_t be = __reduce_min_sync(0xffffffffu, has && key == mk ? (uint32_t)(lane + 32 * i1) : 0xFFFFFFFFu);
            bool refill = false;
            if ((int)(be & 31u) == lane) {   // this lane held the pick
                taken |= 1u << (be >> 5);
                if (second) {
                    v1 = v2;
                    i1 = i2;
                    second = false;
                } else {
                    refill = true;
                }
            }
            if (__any_sync(0xffffffffu, refill) && refill) {
                lane_top2<NV>(v, taken, v1, i1, v2, i2);
                second = true;
            }
            sel_v[j] = key_logit(mk);
            sel_e[j] = (int)be;
        }
    }
    float ex[KM];
    float sum = 0.0f;
#pragma unroll
    for (int j = 0; j < KM; ++j) {
        if (j < k) {
            ex[j] = expf(sel_v[j] - sel_v[0]);
            sum = sum + ex[j];
        }
    }
    int myid = -1;
    float myex = 0.0f;
#pragma unroll
    for (int j = 0; j < KM; ++j) {
        if (j < k && j == lane) {
            myid = sel_e[j];
            myex = ex[j];
        }
    }
    *id_out = myid;
    *w_out = lane < k ? __fdiv_rn(myex, sum) : 0.0f;
}

// Route token t from logits in registers and write its picks (and, in the
// one-CTA path, each pick's expert and the token's bit in its expert's token
// mask in shared memory).
template <int KM, int NV>
__device__ __forceinline__ void route_one(const float (&v)[NV], int t, int E, int k, int lane, int32_t *counts,
                                          int32_t *ids, float *w, int32_t *s_ids, uint32_t *s_tmask) {
    int id;
    float wv;
    warp_route_token<KM, NV>(v, E, k, lane, &id, &wv);
    if (lane < k) {
        ids[t * k + lane] = id;
        w[t * k + lane] = wv;
        if (s_ids) s_ids[t * k + lane] = id;
        if (s_tmask) atomicOr(&s_tmask[id], 1u << t);
        if (counts) red_relaxed_add(counts + id, 1);
    }
}

// Block-wide inclusive scan of one int per thread (blockDim.x = 512).
__device__ __forceinline__ int block_scan(int v, int *warp_tot) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += o;
    }
    if (lane == 31) warp_tot[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int t = lane < kSmallThreads / 32 ? warp_tot[lane] : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, t, off);
            if (lane >= off) t += o;
        }
        if (lane < kSmallThreads / 32) warp_tot[lane] = t;
    }
    __syncthreads();
    return v + (warp ? warp_tot[warp - 1] : 0);
}

// Both banks' pick lists from the step's picks, in one CTA of 512 threads.
// On entry: s_ids [P] holds each pick's expert, s_rm [E] the row map, s_cnt
// [E] zeros, base1 zero, and for steps of at most 32 tokens s_tmask [E] each
// expert's token mask (else null) -- all visible after a barrier.
//  - each pick adds 1 to its row's count (rows of both banks in one array:
//    hot row r at r, cold row r at n_hot + r)
//  - one scan over that array (two rows per thread), the count in the low 16
//    bits and "active" in the high 16: a row's exclusive prefix gives its
//    offset in its bank's pick list and its index among its bank's active rows
//  - each pick's place: its row's offset + the number of earlier picks (lower
//    slots) of the same expert -- a token picks an expert at most once, so
//    with a token mask that is the mask's bits below the pick's token.
__device__ __forceinline__ void build_lists(const int32_t *s_ids, const int32_t *s_rm, int32_t *s_cnt, int *warp_tot,
                                            int &base1, int P, int E, int k, int n_hot, const uint32_t *s_tmask,
                                            WsPtrs ws) {
    const int tid = threadIdx.x;
    for (int s = tid; s < P; s += kSmallThreads) {
        const int m = s_rm[s_ids[s]];
        atomicAdd(&s_cnt[m >= 0 ? m : n_hot + (-1 - m)], 1);
    }
    __syncthreads();
    // the scan: E <= 1024 rows, rows 2*tid and 2*tid+1 in this thread
    const int r0 = 2 * tid, r1 = r0 + 1;
    const int c0 = r0 < E ? s_cnt[r0] : 0, c1 = r1 < E ? s_cnt[r1] : 0;
    const int v0 = c0 | ((c0 > 0) << 16), v1 = c1 | ((c1 > 0) << 16);
    const int incl1 = block_scan(v0 + v1, warp_tot);   // through row r1
    const int incl0 = incl1 - v1;                      // through row r0
    if (n_hot > 0) {   // the thread holding row n_hot - 1 publishes bank 0's totals
        if (r0 == n_hot - 1) base1 = incl0;
        if (r1 == n_hot - 1) base1 = incl1;
    }
    __syncthreads();
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int r = h ? r1 : r0, c = h ? c1 : c0, incl = h ? incl1 : incl0, v = h ? v1 : v0;
        if (r >= E) continue;
        const int b = r >= n_hot;
        const int excl = incl - v - (b ? base1 : 0);
        const int off = excl & 0xFFFF, a = excl >> 16;
        s_cnt[r] = off;   // this row's offset in its bank's pick list
        if (c > 0) {
            ws.act_row[b * P + a] = b ? r - n_hot : r;
            ws.act_off[b * (P + 1) + a + 1] = off + c;
        }
        if (r == E - 1) {   // the thread of the last row holds both banks' totals
            const int tot1 = incl - base1;
            ws.hdr[kHdrNAct + 0] = base1 >> 16;
            ws.hdr[kHdrNPicks + 0] = base1 & 0xFFFF;
            ws.hdr[kHdrNAct + 1] = tot1 >> 16;
            ws.hdr[kHdrNPicks + 1] = tot1 & 0xFFFF;
            ws.act_off[0] = 0;
            ws.act_off[P + 1] = 0;
        }
    }
    __syncthreads();
    for (int s = tid; s < P; s += kSmallThreads) {
        const int e = s_ids[s];
        const int m = s_rm[e];
        const int b = m < 0;
        int pos = 0;
        if (s_tmask) {
            pos = __popc(s_tmask[e] & ((1u << (s / k)) - 1u));
        } else {
            for (int q = 0; q < s; ++q) pos += s_ids[q] == e;
        }
        ws.picks[b * P + s_cnt[b ? n_hot + (-1 - m) : m] + pos] = s;
    }
}

// One-user steps (T <= 32): route, count and build both banks' lists in one
// CTA of 512 threads; warp w routes tokens w and w+16, loading the second
// token's logits while it routes the first.
template <int KM, int NV>
__global__ void __launch_bounds__(kSmallThreads) route_split_small(
    const float *__restrict__ logits, int T, int E, int k, const int32_t *__restrict__ rowmap,
    int n_hot, int32_t *counts, int32_t *__restrict__ ids, float *__restrict__ w, WsPtrs ws) {
    extern __shared__ int32_t sm[];
    __shared__ int warp_tot[32];
    __shared__ int base1;           // bank 0's totals: the prefix bank 1's rows start from
    const int P = ws.P;
    int32_t *s_ids = sm;            // [P] expert of each pick
    int32_t *s_rm = s_ids + P;      // [E] row map
    int32_t *s_cnt = s_rm + E;      // [E] picks per row (both banks), then row offsets
    uint32_t *s_tmask = (uint32_t *)(s_cnt + E);   // [E] tokens that picked each expert
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // the row map is read only by the list building: its loads (E <= 1024,
    // two per thread) stay in flight while the tokens are routed
    const int rm0 = tid < E ? rowmap[tid] : 0;
    const int rm1 = tid + kSmallThreads < E ? rowmap[tid + kSmallThreads] : 0;
    for (int e = tid; e < E; e += kSmallThreads) {
        s_cnt[e] = 0;
        s_tmask[e] = 0u;
    }
    __syncthreads();   // the masks are zero before any token sets a bit
    if (tid == 0) base1 = 0;
    {
        constexpr int kWarps = kSmallThreads / 32;
        float cur[NV], nxt[NV];
        if (warp < T) load_logits<NV>(logits + (size_t)warp * E, E, lane, cur);
        for (int t = warp; t < T; t += kWarps) {
            if (t + kWarps < T) load_logits<NV>(logits + (size_t)(t + kWarps) * E, E, lane, nxt);
            route_one<KM, NV>(cur, t, E, k, lane, counts, ids, w, s_ids, s_tmask);
#pragma unroll
            for (int i = 0; i < NV; ++i) cur[i] = nxt[i];
        }
    }
    if (tid < E) s_rm[tid] = rm0;
    if (tid + kSmallThreads < E) s_rm[tid + kSmallThreads] = rm1;
    __syncthreads();
    build_lists(s_ids, s_rm, s_cnt, warp_tot, base1, P, E, k, n_hot, s_tmask, ws);
}

// Decode steps of 33..256 tokens, after route_tokens: both banks' lists in
// one CTA from the routed ids.
__global__ void __launch_bounds__(kSmallThreads) split_picks(const int32_t *__restrict__ ids, int E,
                                                            const int32_t *__restrict__ rowmap, int n_hot, WsPtrs ws) {
    extern __shared__ int32_t sm[];
    __shared__ int warp_tot[32];
    __shared__ int base1;
    const int P = ws.P;
    int32_t *s_ids = sm;
    int32_t *s_rm = s_ids + P;
    int32_t *s_cnt = s_rm + E;
    const int tid = threadIdx.x;
    for (int e = tid; e < E; e += kSmallThreads) {
        s_rm[e] = rowmap[e];
        s_cnt[e] = 0;
    }
    for (int q = tid; q < P; q += kSmallThreads) s_ids[q] = ids[q];
    if (tid == 0) base1 = 0;
    __syncthreads();
    build_lists(s_ids, s_rm, s_cnt, warp_tot, base1, P, E, 1, n_hot, nullptr, ws);
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

// Large steps, stage 1: one warp per token.  For the split it also counts,
// order-free, the picks of each expert and of each (expert, 32-token chunk).
template <int KM, int NV>
__global__ void __launch_bounds__(256) route_tokens(const float *__restrict__ logits, int T, int E, int k,
                                                   int32_t *counts, int32_t *__restrict__ ids,
                                                   float *__restrict__ w, int32_t *ecnt, int32_t *ccnt) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (t >= T) return;
    float v[NV];
    load_logits<NV>(logits + (size_t)t * E, E, lane, v);
    route_one<KM, NV>(v, t, E, k, lane, counts, ids, w, nullptr, nullptr);
    if (ecnt && lane < k) {
        const int e = ids[t * k + lane];
        red_relaxed_add(ecnt + e, 1);
        red_relaxed_add(ccnt + (size_t)e * ((T + 31) / 32) + t / 32, 1);
    }
}

// Large steps, stage 2 (one CTA): the active-row scan over the per-expert counts.
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

// Large steps, stage 3: one warp per active expert turns its chunk counts
// into the first place of each 32-token chunk's picks in its bank list (the
// expert's list start plus the earlier chunks' counts), over the counts.
__global__ void __launch_bounds__(256) split_chunks(int32_t *ccnt, int nch, int E, WsPtrs ws) {
    const int lane = threadIdx.x & 31;
    const int e = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (e >= E) return;
    int base = ws.epos[e];
    if (base < 0) return;   // no picks
    int32_t *row = ccnt + (size_t)e * nch;
    for (int c0 = 0; c0 < nch; c0 += 32) {
        const int c = c0 + lane;
        const int v = c < nch ? row[c] : 0;
        int inc = v;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, inc, off);
            if (lane >= off) inc += o;
        }
        if (c < nch) row[c] = base + inc - v;
        base += __shfl_sync(0xffffffffu, inc, 31);
    }
}

// Large steps, stage 4: one warp per 32-token chunk places the chunk's picks,
// 32 slots at a time in slot order: the lanes holding the same expert
// (__match_any_sync) take consecutive places from that expert's cursor for
// this chunk, lower slots first, so each expert's picks stay in slot order.
__global__ void __launch_bounds__(32) split_place(const int32_t *__restrict__ ids, int T, int k, int E,
                                                   const int32_t *__restrict__ coff, const int32_t *__restrict__ rowmap,
                                                   WsPtrs ws) {
    extern __shared__ int32_t cur[];   // [E] the chunk's next place per expert
    const int lane = threadIdx.x, c = blockIdx.x, nch = (T + 31) / 32;
    for (int e = lane; e < E; e += 32) cur[e] = coff[(size_t)e * nch + c];
    __syncwarp();
    const int P = ws.P;
    const int s0 = c * 32 * k, s1 = min(P, s0 + 32 * k);
    for (int base = s0; base < s1; base += 32) {
        const int s = base + lane;
        const bool live = s < s1;
        const int e = live ? ids[s] : -1;
        const unsigned grp = __match_any_sync(0xffffffffu, e);
        const int rank = __popc(grp & ((1u << lane) - 1u));
        const int start = live ? cur[e] : 0;
        __syncwarp();
        if (live) {
            ws.picks[(rowmap[e] < 0 ? P : 0) + start + rank] = s;
            if (rank == 0) cur[e] = start + __popc(grp);
        }
        __syncwarp();
    }
}

template <int KM, int NV>
int launch_route_km(const moe_ctx *ctx, const Layer &L, const float *logits, int T, int32_t *counts, int32_t *ids,
                    float *w, WsPtrs ws, int32_t *ecnt, int32_t *ccnt, cudaStream_t s) {
    const Geom &g = ctx->g;
    const int P = ws.P;
    const size_t smem = sizeof(int32_t) * ((size_t)P + 2 * (size_t)g.E);
    if (T <= kFusedMaxT) {
        route_split_small<KM, NV><<<1, kSmallThreads, smem + sizeof(uint32_t) * g.E, s>>>(
            logits, T, g.E, g.k, L.rowmap_dev, L.n_hot, counts, ids, w, ws);
        MOE_LAUNCH_CHECK();
        return MOE_OK;
    }
    if (T <= kSmallMaxT && P <= kSmallMaxP) {
        route_tokens<KM, NV><<<(T + 7) / 8, 256, 0, s>>>(logits, T, g.E, g.k, counts, ids, w, nullptr, nullptr);
        MOE_LAUNCH_CHECK();
        split_picks<<<1, kSmallThreads, smem, s>>>(ids, g.E, L.rowmap_dev, L.n_hot, ws);
        MOE_LAUNCH_CHECK();
        return MOE_OK;
    }
    const int nch = (T + 31) / 32;
    MOE_CUDA_TRY(cudaMemsetAsync(ecnt, 0, sizeof(int32_t) * g.E, s));
    MOE_CUDA_TRY(cudaMemsetAsync(ccnt, 0, sizeof(int32_t) * g.E * nch, s));
    route_tokens<KM, NV><<<(T + 7) / 8, 256, 0, s>>>(logits, T, g.E, g.k, counts, ids, w, ecnt, ccnt);
    MOE_LAUNCH_CHECK();
    split_scan<<<1, 1024, sizeof(int32_t) * 3 * (size_t)g.E, s>>>(ecnt, g.E, L.rowmap_dev, L.n_hot, L.n_cold, ws);
    MOE_LAUNCH_CHECK();
    split_chunks<<<(g.E + 7) / 8, 256, 0, s>>>(ccnt, nch, g.E, ws);
    MOE_LAUNCH_CHECK();
    split_place<<<nch, 32, sizeof(int32_t) * (size_t)g.E, s>>>(ids, T, g.k, g.E, ccnt, L.rowmap_dev, ws);
    MOE_LAUNCH_CHECK();
    return MOE_OK;
}

template <int KM>
int launch_route_nv(const moe_ctx *ctx, const Layer &L, const float *logits, int T, int32_t *counts, int32_t *ids,
                    float *w, WsPtrs ws, int32_t *ecnt, int32_t *ccnt, cudaStream_t s) {
    const int E = ctx->g.E;
    if (E <= 128) return launch_route_km<KM, 4>(ctx, L, logits, T, counts, ids, w, ws, ecnt, ccnt, s);
    if (E <= 256) return launch_route_km<KM, 8>(ctx, L, logits, T, counts, ids, w, ws, ecnt, ccnt, s);
    if (E <= 384) return launch_route_km<KM, 12>(ctx, L, logits, T, counts, ids, w, ws, ecnt, ccnt, s);
    if (E <= 512) return launch_route_km<KM, 16>(ctx, L, logits, T, counts, ids, w, ws, ecnt, ccnt, s);
    return launch_route_km<KM, 32>(ctx, L, logits, T, counts, ids, w, ws, ecnt, ccnt, s);
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
    int32_t *ecnt = (int32_t *)(ws_base + lay.ecnt);
    int32_t *ccnt = (int32_t *)(ws_base + lay.ccnt);
    // the lanes' sorted lists hold KM >= k entries; each lane holds NV >= E/32
    // of a token's logits
    if (g.k <= 4) return launch_route_nv<4>(ctx, L, logits, T, counts, ids, w, ws, ecnt, ccnt, s);
    if (g.k <= 8) return launch_route_nv<8>(ctx, L, logits, T, counts, ids, w, ws, ecnt, ccnt, s);
    return launch_route_nv<16>(ctx, L, logits, T, counts, ids, w, ws, ecnt, ccnt, s);
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
