// Big-batch cold staging: copy-on-miss for cold experts that a step routes
// more tokens than one token tile holds.
//
// "We Built the Counter", section 6 (copying an expert on a miss is a tool
// for big batches; between steps, swaps move rows for good) and "Should a
// GB300 Prefetch Its Cold Experts?" section 6 (staging offloaded experts for
// prefill-sized steps): the FFN kernels stream a unit's weights once per
// token tile, so a cold expert with picks in n tiles crosses the host link n
// times.  When the context has a staging pool (moe_set_cold_staging), every
// FFN call that covers the cold bank first
//   1. selects, on the device, the cold active rows whose pick count exceeds
//      the step's tile width -- most picks first, ties to the lower row, up
//      to the pool's slots -- into the workspace (slot per active row, and
//      the cold row held by each slot), and
//   2. copies each selected row once from the pinned host bank into its HBM
//      slot (16-byte loads over the host link, many CTAs).
// The FFN's units of those rows then read the slot instead of the host bank.
// The bytes are the same, so the rows of Y are bit-identical to unstaged
// (and unsplit) steps.
#include "moe_internal.cuh"

namespace moe {

namespace {

// One CTA of 1024 threads: cold active rows a < n_act (<= 1024).
__global__ void __launch_bounds__(1024) stage_select_kernel(BankLists L, int W, int slots, int32_t *__restrict__ slot_of,
                                                            int32_t *__restrict__ src_of) {
    __shared__ int s_n[1024];
    const int na = L.hdr[kHdrNAct + 1];
    const int a = threadIdx.x;
    const int n = a < na ? L.act_off[a + 1] - L.act_off[a] : 0;
    s_n[a] = n > W ? n : 0;   // candidates: more picks than one tile holds
    for (int s = a; s < kMaxStageSlots; s += blockDim.x) src_of[s] = -1;
    __syncthreads();
    if (a >= na) return;
    int slot = -1;
    if (s_n[a] > 0) {
        int rank = 0;
        for (int q = 0; q < na; ++q) rank += s_n[q] > s_n[a] || (s_n[q] == s_n[a] && s_n[q] > 0 && q < a);
        if (rank < slots) slot = rank;
    }
    slot_of[a] = slot;
    if (slot >= 0) src_of[slot] = L.act_row[a];
}

// Copy the selected cold rows into their slots: 16-byte chunks, four loads in
// flight per thread before their stores.
__global__ void __launch_bounds__(256) stage_copy_kernel(const uint4 *__restrict__ cold, uint4 *__restrict__ pool,
                                                         const int32_t *__restrict__ src_of, int slots, int64_t eb16) {
    const int64_t total = (int64_t)slots * eb16;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t c0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c0 < total; c0 += 4 * stride) {
        uint4 v[4];
        int64_t dst[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int64_t c = c0 + u * stride;
            dst[u] = -1;
            if (c < total) {
                const int slot = (int)(c / eb16);
                const int32_t row = src_of[slot];
                if (row >= 0) {
                    v[u] = __ldcs(cold + (int64_t)row * eb16 + (c - (int64_t)slot * eb16));
                    dst[u] = c;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (dst[u] >= 0) pool[dst[u]] = v[u];
    }
}

}  // namespace

int launch_cold_staging(moe_ctx *ctx, const Layer &layer, int W, const BankLists &cold_lists, int32_t *slot_of,
                        int32_t *src_of, cudaStream_t s) {
    stage_select_kernel<<<1, 1024, 0, s>>>(cold_lists, W, ctx->stage_slots, slot_of, src_of);
    MOE_LAUNCH_CHECK();
    const int64_t eb16 = ctx->g.eb / 16;
    stage_copy_kernel<<<4 * ctx->sms, 256, 0, s>>>((const uint4 *)layer.cold_dev, (uint4 *)ctx->stage_pool, src_of,
                                                   ctx->stage_slots, eb16);
    MOE_LAUNCH_CHECK();
    return MOE_OK;
}

}  // namespace moe
