// Router GEMM: the step that produces the routing logits from the layer's
// hidden states.
//
// "vLLM: Pin Hot Experts", Where the experts live today: every MoE layer's
// router scores all experts for every token and keeps its top-6, whichever
// bank the experts sit in.  Here the scores are
//     logits[t][e] = bias[e] + sum_h x[t][h] * w_router[e][h]
// with bf16 hidden states and router weights, exact products, fp32 sums and
// fp32 logits written where the routing kernel reads them.
//
// Two kernels:
//  * up to 32 tokens (decode): CUDA cores.  A cluster of four CTAs per
//    (group of 4 experts, group of 8 tokens); CTA q of the cluster takes the
//    q-th quarter of K, 64 threads per expert.  One thread issues a bulk
//    asynchronous copy of each expert row's quarter and of each token row's
//    quarter into shared memory (at H = 4096: 4 x 2 KB and up to 8 x 2 KB), so
//    the 3 MB of router weights (E = 384) move from HBM across the whole GPU
//    in about one memory latency, without one 16-byte request per thread.  A
//    thread sums its columns in order; a butterfly adds the 32 lanes; the
//    expert's two warps are added in warp order; CTA 0 of the cluster adds
//    the four quarters in order through distributed shared memory, then the
//    bias -- a fixed order, so the logits are reproducible.
//  * more tokens: a dense bf16 GEMM on the tensor cores (tcgen05.mma
//    kind::f16, fp32 accumulator in tensor memory).  One CTA per (128-token
//    tile, BN-expert tile); one thread issues TMA loads of 64-wide K slices of
//    both operands (128-byte swizzle) into a ring of stages, one thread
//    issues the MMAs, four warps read the accumulator back and add the bias.
//    Tokens and experts past the ends are zero-filled by the TMA and never
//    stored.  At 8192 tokens the GEMM is 25.8 GFLOP.
//
// Every mbarrier wait is bounded; on timeout the kernel sets the status word
// to MOE_ETIMEOUT, lets its own copies and MMAs in flight finish, frees its
// tensor memory and returns.
#include "moe_internal.cuh"
#include "sm103_ptx.cuh"

#include <cooperative_groups.h>
#include <cudaTypedefs.h>

namespace moe {

namespace {

// ---------------------------------------------------------------- CUDA cores

constexpr int kTok = 8;       // tokens per CTA
constexpr int kRE = 4;        // experts per CTA (64 threads each)
constexpr int kKParts = 4;    // CTAs per cluster: the quarters of K
constexpr int kRThreads = 64 * kRE;

__device__ __forceinline__ void bf16x8(const uint4 v, float (&f)[8]) {
    const uint32_t p[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        f[2 * q] = __uint_as_float(p[q] << 16);
        f[2 * q + 1] = __uint_as_float(p[q] & 0xFFFF0000u);
    }
}

constexpr int kSpan = 224;                     // 16-byte columns of a K quarter staged at a time
constexpr uint64_t kSimtWaitNs = 1000000000ull;   // bound of the copies' wait

__global__ void __cluster_dims__(kKParts, 1, 1) __launch_bounds__(kRThreads)
    router_simt_kernel(const uint4 *__restrict__ x, const uint4 *__restrict__ w, const float *__restrict__ bias, int T,
                       int E, int H8, float *__restrict__ logits, int32_t *status) {
    namespace cg = cooperative_groups;
    __shared__ __align__(128) uint4 wsm[kRE][kSpan];   // the CTA's experts over a span of its K quarter
    __shared__ __align__(128) uint4 xs[kTok][kSpan];   // its tokens over the same span
    __shared__ float part[kRE][2][kTok];                // [expert][its warp][token]
    __shared__ __align__(8) uint64_t full;
    cg::cluster_group cluster = cg::this_cluster();
    const int kp = (int)cluster.block_rank();   // this CTA's quarter of K
    const int grp = blockIdx.x / kKParts;
    const int tid = threadIdx.x, el = tid >> 6, r = tid & 63, lane = tid & 31, wp = (tid >> 5) & 1;
    const int e = grp * kRE + el;
    const int ne = min(kRE, E - grp * kRE);   // experts of this group, >= 1
    const int t0 = blockIdx.y * kTok;
    const int nt = min(kTok, T - t0);         // >= 1: the grid covers T exactly
    const int c0 = kp * H8 / kKParts, c1 = (kp + 1) * H8 / kKParts;
    const uint32_t bar = ptx::smem_addr(&full);
    if (tid == 0) {
        ptx::mbar_init(bar, 1);
        ptx::fence_mbar_init();
    }
    __syncthreads();
    float acc[kTok];
#pragma unroll
    for (int j = 0; j < kTok; ++j) acc[j] = 0.0f;
    bool ok = true;
    uint32_t phase = 0;
    for (int cs = c0; ok && cs < c1; cs += kSpan, phase ^= 1u) {
        const int len = min(c1, cs + kSpan) - cs;   // 16-byte columns in this span
        if (tid == 0) {
            // one bulk copy per expert row and per token row of the span
            ptx::mbar_arrive_expect_tx(bar, (uint32_t)((ne + nt) * len * 16));
            for (int q = 0; q < ne; ++q)
                ptx::bulk_g2s(ptx::smem_addr(&wsm[q][0]), w + (size_t)(grp * kRE + q) * H8 + cs, (uint32_t)len * 16, bar);
            for (int j = 0; j < nt; ++j)
                ptx::bulk_g2s(ptx::smem_addr(&xs[j][0]), x + (size_t)(t0 + j) * H8 + cs, (uint32_t)len * 16, bar);
        }
        uint64_t tw = 0;
        for (uint32_t i = 0;; ++i) {   // bounded wait for the span
            if (ptx::mbar_try_wait(bar, phase)) break;
            if ((i & 255u) == 0u) {
                const uint64_t now = ptx::globaltimer_ns();
                if (i == 0) {
                    tw = now;
                } else if (now - tw > kSimtWaitNs) {
                    atomicCAS(status, 0, MOE_ETIMEOUT);
                    ok = false;
                    break;
                }
            }
        }
        if (!ok) break;
        if (e < E) {
            for (int c = r; c < len; c += 64) {   // this thread's columns in increasing order
                float wf[8], xf[8];
                bf16x8(wsm[el][c], wf);
#pragma unroll
                for (int j = 0; j < kTok; ++j) {
                    if (j < nt) {
                        bf16x8(xs[j][c], xf);
#pragma unroll
                        for (int q = 0; q < 8; ++q) acc[j] = __fmaf_rn(xf[q], wf[q], acc[j]);
                    }
                }
            }
        }
        __syncthreads();   // the span is read before the next one is copied over it
    }
    if (!ok) {
        // let this CTA's copies land before it goes away (bounded)
        for (uint32_t i = 0; i < (1u << 22); ++i)
            if (ptx::mbar_try_wait(bar, phase)) break;
    }
#pragma unroll
    for (int j = 0; j < kTok; ++j) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc[j] += __shfl_xor_sync(0xFFFFFFFFu, acc[j], o);
        if (lane == 0) part[el][wp][j] = acc[j];
    }
    cluster.sync();   // every quarter's sums are in its CTA's shared memory
    if (kp == 0 && tid < kRE * kTok && ok) {
        const int el2 = tid / kTok, j = tid % kTok, e2 = grp * kRE + el2;
        if (e2 < E && j < nt) {
            float sum = 0.0f;
#pragma unroll
            for (int q = 0; q < kKParts; ++q) {
                const float *rp = cluster.map_shared_rank(&part[0][0][0], q);
                sum += rp[(el2 * 2 + 0) * kTok + j] + rp[(el2 * 2 + 1) * kTok + j];
            }
            logits[(size_t)(t0 + j) * E + e2] = sum + (bias ? __ldg(bias + e2) : 0.0f);
        }
    }
    cluster.sync();   // the other quarters' shared memory stays until CTA 0 has read it
}

// -------------------------------------------------------------- tensor cores

constexpr int kBM = 128;                 // tokens per tile (MMA M)
constexpr int kBK = 64;                  // K elements per stage (128 bytes of bf16: one swizzle row)
constexpr int kAStage = kBM * kBK * 2;   // 16 KB
constexpr uint64_t kWaitNs = 1000000000ull;
constexpr uint32_t kDrainPolls = 1u << 22;

template <int BN>
struct RouterCfg {
    static_assert(BN % 16 == 0 && BN >= 32 && BN <= 256, "MMA N");
    static constexpr int kStages = BN >= 128 ? 5 : 8;
    static constexpr int kBStage = BN * kBK * 2;
    static constexpr int kStage = kAStage + kBStage;
    static constexpr uint32_t kCols = BN <= 32 ? 32 : BN <= 64 ? 64 : BN <= 128 ? 128 : 256;   // TMEM columns
    static constexpr size_t kSmem = 1024 + (size_t)kStages * kStage + (2 * kStages + 1) * 8 + 16;
};

// Bounded mbarrier wait (one thread): false once kWaitNs of wall-clock time
// have passed or another role gave up.
__device__ __forceinline__ bool rwait(uint32_t bar, uint32_t parity, volatile int *abort_flag, int32_t *status) {
    uint64_t t0 = 0;
    for (uint32_t i = 0;; ++i) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if ((i & 255u) == 0u) {
            if (*abort_flag) return false;
            const uint64_t now = ptx::globaltimer_ns();
            if (i == 0) {
                t0 = now;
            } else if (now - t0 > kWaitNs) {
                *abort_flag = 1;
                atomicCAS(status, 0, MOE_ETIMEOUT);
                return false;
            }
        }
    }
}

template <int BN>
__global__ void __launch_bounds__(192, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                     const float *__restrict__ bias, int T, int E, int H, float *__restrict__ logits,
                     int32_t *status) {
    using C = RouterCfg<BN>;
    constexpr int S = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (ptx::smem_addr(smem_raw) & 1023u)) & 1023u);
    uint64_t *bars = (uint64_t *)(smem + (size_t)S * C::kStage);   // FULL[S], DONE[S], ACC
    uint32_t *holder = (uint32_t *)(bars + 2 * S + 1);
    volatile int *abort_flag = (volatile int *)(holder + 1);
    auto bar = [&](int i) { return ptx::smem_addr(bars + i); };
    const int FULL = 0, DONE = S, ACC = 2 * S;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int m0 = blockIdx.x * kBM, n0 = blockIdx.y * BN;
    const int nk = (H + kBK - 1) / kBK;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(bar(FULL + s), 1);
            ptx::mbar_init(bar(DONE + s), 1);
        }
        ptx::mbar_init(bar(ACC), 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 4 && lane == 0) {
        ptx::prefetch_tmap(&tmX);
        ptx::prefetch_tmap(&tmW);
    }
    if (warp == 5) {
        ptx::tmem_alloc(ptx::smem_addr(holder), C::kCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *holder;

    if (warp < 4) {
        // ---------------------------------------------------------- epilogue
        // thread 32 w + l reads accumulator row (token) m0 + 32 w + l
        const bool ok = rwait(bar(ACC), 0, abort_flag, status);
        if (__all_sync(0xFFFFFFFFu, ok)) {
            ptx::tc_fence_after();
            const int t = m0 + warp * 32 + lane;
            float *row = logits + (size_t)t * E;
            const bool vec = (E % 4) == 0 && ((uintptr_t)logits % 16) == 0;
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += 32) {
                uint32_t r[32];
                ptx::tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c0, r);
                ptx::tmem_wait_ld();
                if (t < T) {
                    const int e0 = n0 + c0;
                    if (vec && e0 + 32 <= E) {
#pragma unroll
                        for (int i = 0; i < 32; i += 4) {
                            float4 v;
                            v.x = __uint_as_float(r[i]) + (bias ? __ldg(bias + e0 + i) : 0.0f);
                            v.y = __uint_as_float(r[i + 1]) + (bias ? __ldg(bias + e0 + i + 1) : 0.0f);
                            v.z = __uint_as_float(r[i + 2]) + (bias ? __ldg(bias + e0 + i + 2) : 0.0f);
                            v.w = __uint_as_float(r[i + 3]) + (bias ? __ldg(bias + e0 + i + 3) : 0.0f);
                            *reinterpret_cast<float4 *>(row + e0 + i) = v;
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (e0 + i < E) row[e0 + i] = __uint_as_float(r[i]) + (bias ? __ldg(bias + e0 + i) : 0.0f);
                    }
                }
            }
        }
    } else if (warp == 4 && lane == 0) {
        // ---------------------------------------------------------- producer
        int it = 0;
        bool ok = true;
        for (; it < nk; ++it) {
            const int st = it % S;
            if (it >= S && !rwait(bar(DONE + st), ((it / S) - 1) & 1, abort_flag, status)) {
                ok = false;
                break;
            }
            uint8_t *a = smem + (size_t)st * C::kStage;
            // out-of-range rows and columns are zero-filled and still counted
            ptx::mbar_arrive_expect_tx(bar(FULL + st), (uint32_t)C::kStage);
            ptx::tma_load_2d(ptx::smem_addr(a), &tmX, it * kBK, m0, bar(FULL + st));
            ptx::tma_load_2d(ptx::smem_addr(a + kAStage), &tmW, it * kBK, n0, bar(FULL + st));
        }
        if (!ok) {
            // let the copies this thread issued land before the CTA goes away
            for (int i = it > S ? it - S : 0; i < it; ++i)
                for (uint32_t p = 0; p < kDrainPolls; ++p)
                    if (ptx::mbar_try_wait(bar(FULL + i % S), (i / S) & 1)) break;
        }
    } else if (warp == 5 && lane == 0) {
        // --------------------------------------------------------- MMA issue
        constexpr uint32_t idesc = ptx::idesc_bf16_f32(kBM, BN);
        int it = 0;
        bool ok = true;
        for (; it < nk; ++it) {
            const int st = it % S;
            if (!rwait(bar(FULL + st), (it / S) & 1, abort_flag, status)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            const uint32_t a_addr = ptx::smem_addr(smem + (size_t)st * C::kStage);
            const uint32_t b_addr = a_addr + kAStage;
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)   // 16 bf16 = 32 bytes per MMA
                ptx::mma_f16_ss(tmem, ptx::smem_desc_sw128(a_addr + kk * 32), ptx::smem_desc_sw128(b_addr + kk * 32),
                                idesc, (it | kk) != 0);
            ptx::mma_commit(bar(DONE + st));
        }
        if (ok) {
            ptx::mma_commit(bar(ACC));
        } else if (it > 0) {
            // wait until the MMAs already issued have retired (bounded)
            const int last = it - 1;
            for (uint32_t p = 0; p < kDrainPolls; ++p)
                if (ptx::mbar_try_wait(bar(DONE + last % S), (last / S) & 1)) break;
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, C::kCols);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
    }
    return fn;
}

// Row-major bf16 [rows][H] as (column, row) boxes of 64 columns x box_rows
// rows, 128-byte swizzle, zero fill outside.
int bf16_rows_map(CUtensorMap *map, const uint16_t *base, int rows, int H, int box_rows) {
    auto enc = encoder();
    if (!enc) return set_error(MOE_ECUDA, "cuTensorMapEncodeTiled unavailable");
    cuuint64_t dims[2] = {(cuuint64_t)H, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)H * 2};
    cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return set_error(MOE_ECUDA, "cuTensorMapEncodeTiled (router) failed: " + std::to_string((int)r));
    return MOE_OK;
}

template <int BN>
int launch_router_tc(const uint16_t *x, const uint16_t *w_router, const float *bias, int T, int E, int H,
                     float *logits, int32_t *status, cudaStream_t s) {
    using C = RouterCfg<BN>;
    CUtensorMap tmX, tmW;
    if (int r = bf16_rows_map(&tmX, x, T, H, kBM)) return r;
    if (int r = bf16_rows_map(&tmW, w_router, E, H, BN)) return r;
    auto kern = router_tc_kernel<BN>;
    MOE_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem));
    const dim3 grid((T + kBM - 1) / kBM, (E + BN - 1) / BN);
    kern<<<grid, 192, C::kSmem, s>>>(tmX, tmW, bias, T, E, H, logits, status);
    MOE_LAUNCH_CHECK();
    return MOE_OK;
}

}  // namespace

int launch_router(const uint16_t *x, const uint16_t *w_router, const float *bias, int T, int E, int H,
                  float *logits, int32_t *status, int sms, cudaStream_t s) {
    if (T <= 32) {
        const dim3 grid(kKParts * ((E + kRE - 1) / kRE), (T + kTok - 1) / kTok);
        router_simt_kernel<<<grid, kRThreads, 0, s>>>((const uint4 *)x, (const uint4 *)w_router, bias, T, E, H / 8,
                                                      logits, status);
        MOE_LAUNCH_CHECK();
        return MOE_OK;
    }
    // wide expert tiles once they alone fill half the SMs; narrow ones
    // spread a few token tiles over more CTAs
    const int mtiles = (T + kBM - 1) / kBM;
    if (2 * mtiles * ((E + 191) / 192) >= sms)
        return launch_router_tc<192>(x, w_router, bias, T, E, H, logits, status, s);
    return launch_router_tc<32>(x, w_router, bias, T, E, H, logits, status, s);
}

}  // namespace moe
