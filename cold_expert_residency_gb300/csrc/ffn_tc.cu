// MXFP4 expert FFN on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// "vLLM: Pin Hot Experts", Results: the routed MXFP4 expert FFN (gate/up
// GEMM, SwiGLU, down GEMM) runs once per residency bank without finalize.
// Here one launch per GEMM covers one bank:
//
//   unit = (active bank row = one expert, 128-row M-tile [, N-tile]);
//   D[128 x N] = A[128 x K] * B[N x K]^T accumulated in TMEM (fp32), with
//   A = the expert's MXFP4 weights dequantised exactly to f16 and
//   B = the expert's token rows (f16, each row scaled by a power of two so its
//   largest element lies in [2^13, 2^14); the epilogue undoes the scale).
//
// Warp roles (192 threads):
//   warp 4      producer: hot bank -> one bulk async copy (TMA) of each
//               4352-byte (M-tile, K-chunk) weight block into a shared-memory
//               ring; cold bank -> 16-byte cp.async reads of the mapped host
//               bank (the host-link streaming path); token rows of the chunk
//               into the canonical no-swizzle K-major layout.
//   warps 0-3   dequant: thread m owns weight row m = TMEM lane m; converts 64
//               e2m1 codes with the hardware e2m1x2 -> f16x2 conversion,
//               applies the e8m0 block scale (exact in f16), and stores the
//               32 f16x2 columns to a double-buffered A operand in TMEM;
//               then the epilogue (tcgen05.ld of D, SwiGLU or bf16 store).
//   warp 5      TMEM allocation; lane 0 issues tcgen05.mma (A from TMEM,
//               B from shared memory) and tcgen05.commit.
//
// The arithmetic of a pick depends only on its expert's weights, its token
// row and the expert's token count (which fixes N), never on the bank, so the
// hot and cold banks and any swap give bit-identical rows.
//
// Every mbarrier wait is bounded; on timeout the kernel sets the status word
// to MOE_ETIMEOUT, drains its own copies in flight, frees TMEM and returns.
#include "moe_internal.cuh"
#include "sm103_ptx.cuh"

namespace moe {

namespace {

constexpr uint32_t kWaitLimit = 1u << 22;

struct TcArgs {
    const uint8_t *bank;
    int64_t eb, part_off;
    int mt_count, kc;
    BankLists lists;
    int b, k, H, I;
    const __half *bsrc;     // phase 1: scaled x rows [T][H]; phase 2: scaled h rows [P][I]
    int bsrc_ld;
    const int32_t *bexp;    // phase 1: per token; phase 2: per slot
    float *h_out;           // phase 1 output [P][I]
    uint16_t *Y;            // phase 2 output [P][H]
    int32_t *status;
};

__device__ __forceinline__ bool wait_one(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                         int32_t *status) {
    for (uint32_t i = 0;; ++i) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if ((i & 255u) == 255u) {
            if (*abort_flag) return false;
            if (i >= kWaitLimit) {
                *abort_flag = 1;
                atomicCAS(status, 0, MOE_ETIMEOUT);
                return false;
            }
        }
    }
}

__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                          int32_t *status) {
    bool ok = wait_one(bar, parity, abort_flag, status);
    return __all_sync(0xffffffffu, ok);
}

// e8m0 byte (104..140, checked at bank init) -> the same power of two in f16.
__device__ __forceinline__ uint32_t e8m0_f16x2(uint32_t s) {
    uint32_t h = s >= 113u ? (s - 112u) << 10 : 1u << (s - 103u);
    return h | (h << 16);
}

// 8 e2m1 codes (one 32-bit word, low nibble first) -> 4 f16x2, scaled.
__device__ __forceinline__ void dequant_word(uint32_t w, uint32_t scale2, uint32_t *o) {
    uint32_t c0, c1, c2, c3;
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
        " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
        " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
        : "=r"(c0), "=r"(c1), "=r"(c2), "=r"(c3)
        : "r"(w));
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(o[0]) : "r"(c0), "r"(scale2));
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(o[1]) : "r"(c1), "r"(scale2));
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(o[2]) : "r"(c2), "r"(scale2));
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(o[3]) : "r"(c3), "r"(scale2));
}

template <int NMAX>
struct TcCfg {
    static constexpr int kStages = NMAX <= 16 ? 8 : (NMAX <= 64 ? 6 : 4);
    static constexpr int kBStage = NMAX * 128;              // bytes of one B chunk
    static constexpr uint32_t kLBO = NMAX * 16;             // core-matrix stride along K
    static constexpr uint32_t kCols = NMAX <= 64 ? 128 : 512;
    static constexpr uint32_t kDCol = 64;                   // D after two 32-column A buffers
    static constexpr int kBars = 2 * kStages + 6;
    static constexpr size_t kSmem = (size_t)kStages * (kChunkBytes + kBStage) + kBars * 8 + 16;
};

template <int NMAX, int PHASE, bool COLD>
__global__ void __launch_bounds__(192, 1) ffn_tc_kernel(TcArgs args) {
    using C = TcCfg<NMAX>;
    constexpr int S = C::kStages;
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t *sA = smem;
    uint8_t *sB = smem + S * kChunkBytes;
    uint64_t *bars = (uint64_t *)(sB + S * C::kBStage);
    uint32_t *holder = (uint32_t *)(bars + C::kBars);
    volatile int *abort_flag = (volatile int *)(holder + 1);
    auto bar = [&](int i) { return ptx::smem_addr(bars + i); };
    // barrier indices
    const int FULL = 0, EMPTY = S, AREADY = 2 * S, AFREE = 2 * S + 2, ACCREADY = 2 * S + 4, ACCFREE = 2 * S + 5;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(bar(FULL + s), COLD ? 33 : 1);
            ptx::mbar_init(bar(EMPTY + s), 1);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(bar(AREADY + i), 128);
            ptx::mbar_init(bar(AFREE + i), 1);
        }
        ptx::mbar_init(bar(ACCREADY), 1);
        ptx::mbar_init(bar(ACCFREE), 128);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 5) {
        ptx::tmem_alloc(ptx::smem_addr(holder), C::kCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *holder;

    const BankLists &L = args.lists;
    const int n_act = L.hdr[kHdrNAct + args.b];
    const int units = n_act * args.mt_count;
    const int kc = args.kc;

    if (warp < 4) {
        // ------------------------------------------------ dequant + epilogue
        const int m = tid;
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        uint32_t it = 0, j = 0;
        bool ok = true;
        for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
            const int a = u / args.mt_count, mt = u % args.mt_count;
            const int p0 = L.act_off[a], n = L.act_off[a + 1] - p0;
            for (int n0 = 0; ok && n0 < n; n0 += NMAX, ++j) {
                const int nn = min(NMAX, n - n0);
                for (int c = 0; c < kc; ++c, ++it) {
                    const int st = it % S;
                    if (!wait_warp(bar(FULL + st), (it / S) & 1, abort_flag, args.status)) { ok = false; break; }
                    const uint8_t *a_st = sA + st * kChunkBytes;
                    const uint4 q0 = *(const uint4 *)(a_st + m * 16);
                    const uint4 q1 = *(const uint4 *)(a_st + 2048 + m * 16);
                    const uint32_t sc = *(const uint16_t *)(a_st + kChunkQBytes + 2 * m);
                    const uint32_t s0 = e8m0_f16x2(sc & 0xFFu), s1 = e8m0_f16x2(sc >> 8);
                    uint32_t r[32];
                    dequant_word(q0.x, s0, r + 0);
                    dequant_word(q0.y, s0, r + 4);
                    dequant_word(q0.z, s0, r + 8);
                    dequant_word(q0.w, s0, r + 12);
                    dequant_word(q1.x, s1, r + 16);
                    dequant_word(q1.y, s1, r + 20);
                    dequant_word(q1.z, s1, r + 24);
                    dequant_word(q1.w, s1, r + 28);
                    const int abuf = it & 1;
                    const uint32_t ua = it >> 1;
                    if (ua > 0 && !wait_warp(bar(AFREE + abuf), (ua - 1) & 1, abort_flag, args.status)) {
                        ok = false;
                        break;
                    }
                    ptx::tmem_st32(tmem + lane_base + abuf * 32, r);
                    ptx::tmem_wait_st();
                    ptx::tc_fence_before();
                    ptx::mbar_arrive(bar(AREADY + abuf));
                }
                if (!ok) break;
                if (!wait_warp(bar(ACCREADY), j & 1, abort_flag, args.status)) { ok = false; break; }
                ptx::tc_fence_after();
                const int w = warp, l = lane;
                const int Nr = (nn + 15) & ~15;
                for (int c0 = 0; c0 < Nr; c0 += 16) {
                    uint32_t v[16];
                    ptx::tmem_ld16(tmem + lane_base + C::kDCol + c0, v);
                    ptx::tmem_wait_ld();
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        const int col = c0 + q;
                        if (col < nn) {   // warp-uniform
                            const int slot = L.picks[p0 + n0 + col];
                            if (PHASE == 1) {
                                const float d = ldexpf(__uint_as_float(v[q]), args.bexp[slot / args.k]);
                                const float o = __shfl_xor_sync(0xffffffffu, d, 16);
                                if (l < 16) {
                                    const float hv = __fmul_rn(__fdiv_rn(d, 1.0f + expf(-d)), o);
                                    args.h_out[(int64_t)slot * args.I + 64 * mt + 16 * w + l] = hv;
                                }
                            } else {
                                const float d = ldexpf(__uint_as_float(v[q]), args.bexp[slot]);
                                args.Y[(int64_t)slot * args.H + kMT * mt + m] =
                                    __bfloat16_as_ushort(__float2bfloat16_rn(d));
                            }
                        }
                    }
                }
                ptx::tc_fence_before();
                ptx::mbar_arrive(bar(ACCFREE));
            }
        }
    } else if (warp == 4) {
        // ------------------------------------------------------------ producer
        uint32_t it = 0;
        bool ok = true;
        for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
            const int a = u / args.mt_count, mt = u % args.mt_count;
            const int row = L.act_row[a];
            const int p0 = L.act_off[a], n = L.act_off[a + 1] - p0;
            const uint8_t *tile = args.bank + (int64_t)row * args.eb + args.part_off +
                                  (int64_t)mt * kc * kChunkBytes;
            for (int n0 = 0; ok && n0 < n; n0 += NMAX) {
                const int nn = min(NMAX, n - n0);
                const int Nr = (nn + 15) & ~15;
                for (int c = 0; c < kc; ++c, ++it) {
                    const int st = it % S;
                    const uint32_t rnd = it / S;
                    if (rnd > 0 && !wait_warp(bar(EMPTY + st), (rnd - 1) & 1, abort_flag, args.status)) {
                        ok = false;
                        break;
                    }
                    const uint32_t b_addr = ptx::smem_addr(sB + st * C::kBStage);
                    for (int idx = lane; idx < Nr * 8; idx += 32) {
                        const int nr = idx >> 3, kb = idx & 7;
                        uint4 v = make_uint4(0u, 0u, 0u, 0u);
                        if (nr < nn) {
                            const int slot = L.picks[p0 + n0 + nr];
                            const int src = PHASE == 1 ? slot / args.k : slot;
                            v = ptx::ld_nc_v4(args.bsrc + (int64_t)src * args.bsrc_ld + c * kKC + kb * 8);
                        }
                        ptx::st_shared_v4(b_addr + kb * C::kLBO + (nr >> 3) * 128 + (nr & 7) * 16, v);
                    }
                    const uint32_t a_addr = ptx::smem_addr(sA + st * kChunkBytes);
                    const uint8_t *src_chunk = tile + (int64_t)c * kChunkBytes;
                    if (COLD) {
                        for (int i = lane; i < kChunkBytes / 16; i += 32) ptx::cp_async16(a_addr + i * 16, src_chunk + i * 16);
                    }
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    if (COLD) {
                        ptx::cp_async_arrive_noinc(bar(FULL + st));
                        if (lane == 0) ptx::mbar_arrive(bar(FULL + st));
                    } else if (lane == 0) {
                        ptx::mbar_arrive_expect_tx(bar(FULL + st), kChunkBytes);
                        ptx::bulk_g2s(a_addr, src_chunk, kChunkBytes, bar(FULL + st));
                    }
                }
            }
        }
        if (!ok) {
            // let the copies this warp issued land before the CTA goes away
            const uint32_t first = it > (uint32_t)S ? it - S : 0u;
            for (uint32_t i = first; i < it; ++i) {
                for (uint32_t t = 0; t < kWaitLimit; ++t)
                    if (ptx::mbar_try_wait(bar(FULL + i % S), (i / S) & 1)) break;
            }
        }
    } else if (lane == 0) {
        // ----------------------------------------------------------- MMA issue
        uint32_t it = 0, j = 0;
        bool ok = true;
        for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
            const int a = u / args.mt_count;
            const int n = L.act_off[a + 1] - L.act_off[a];
            for (int n0 = 0; ok && n0 < n; n0 += NMAX, ++j) {
                const int nn = min(NMAX, n - n0);
                const int Nr = (nn + 15) & ~15;
                const uint32_t idesc = ptx::idesc_f16_f32(128, Nr);
                if (j > 0 && !wait_one(bar(ACCFREE), (j - 1) & 1, abort_flag, args.status)) { ok = false; break; }
                ptx::tc_fence_after();
                for (int c = 0; c < kc; ++c, ++it) {
                    const int st = it % S, abuf = it & 1;
                    if (!wait_one(bar(AREADY + abuf), (it >> 1) & 1, abort_flag, args.status)) { ok = false; break; }
                    ptx::tc_fence_after();
                    ptx::fence_proxy_async_smem();
                    const uint32_t b_addr = ptx::smem_addr(sB + st * C::kBStage);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t bd = ptx::smem_desc_noswizzle(b_addr + 2 * kk * C::kLBO, C::kLBO, 128);
                        ptx::mma_f16_ts(tmem + C::kDCol, tmem + abuf * 32 + kk * 8, bd, idesc, (c | kk) != 0);
                    }
                    ptx::mma_commit(bar(EMPTY + st));
                    ptx::mma_commit(bar(AFREE + abuf));
                }
                if (!ok) break;
                ptx::mma_commit(bar(ACCREADY));
            }
        }
        if (!ok && it > 0) {
            // wait until the MMAs already issued have retired (bounded)
            const uint32_t last = it - 1;
            for (uint32_t t = 0; t < kWaitLimit; ++t)
                if (ptx::mbar_try_wait(bar(AFREE + (last & 1)), (last >> 1) & 1)) break;
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, C::kCols);
    }
}

// Per-token power-of-two scaling of x into f16: largest |x| -> [2^13, 2^14).
__global__ void __launch_bounds__(256) prep_x_kernel(const uint16_t *__restrict__ x, int H,
                                                     __half *__restrict__ xs, int32_t *__restrict__ xexp) {
    __shared__ float red[8];
    const int t = blockIdx.x;
    const uint16_t *row = x + (int64_t)t * H;
    float mx = 0.0f;
    for (int h = threadIdx.x; h < H; h += blockDim.x) mx = fmaxf(mx, fabsf(__uint_as_float((uint32_t)row[h] << 16)));
    for (int off = 16; off; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
    __syncthreads();
    mx = red[0];
    for (int i = 1; i < (int)(blockDim.x >> 5); ++i) mx = fmaxf(mx, red[i]);
    int e = 0;
    frexpf(mx, &e);
    const int c = mx > 0.0f ? e - 14 : 0;
    for (int h = threadIdx.x; h < H; h += blockDim.x)
        xs[(int64_t)t * H + h] = __float2half_rn(ldexpf(__uint_as_float((uint32_t)row[h] << 16), -c));
    if (threadIdx.x == 0) xexp[t] = c;
}

// Per-pick power-of-two scaling of the gate/up output h into f16.
__global__ void __launch_bounds__(256) prep_h_kernel(BankLists lists, int b, int I,
                                                     const float *__restrict__ h32, __half *__restrict__ h16,
                                                     int32_t *__restrict__ hexp) {
    __shared__ float red[8];
    const int p = blockIdx.x;
    if (p >= lists.hdr[kHdrNPicks + b]) return;
    const int slot = lists.picks[p];
    const float *row = h32 + (int64_t)slot * I;
    float mx = 0.0f;
    for (int i = threadIdx.x; i < I; i += blockDim.x) mx = fmaxf(mx, fabsf(row[i]));
    for (int off = 16; off; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
    __syncthreads();
    mx = red[0];
    for (int i = 1; i < (int)(blockDim.x >> 5); ++i) mx = fmaxf(mx, red[i]);
    int e = 0;
    frexpf(mx, &e);
    const int c = mx > 0.0f ? e - 14 : 0;
    for (int i = threadIdx.x; i < I; i += blockDim.x) h16[(int64_t)slot * I + i] = __float2half_rn(ldexpf(row[i], -c));
    if (threadIdx.x == 0) hexp[slot] = c;
}

template <int NMAX, int PHASE, bool COLD>
int launch_one(moe_ctx *ctx, const TcArgs &args, int units_max, cudaStream_t s) {
    using C = TcCfg<NMAX>;
    auto kern = ffn_tc_kernel<NMAX, PHASE, COLD>;
    MOE_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem));
    const int per_sm = NMAX <= 64 ? 4 : 1;   // TMEM: 128 columns per CTA, or 512
    int blocks = std::min(units_max, ctx->sms * per_sm);
    if (blocks < 1) return MOE_OK;
    kern<<<blocks, 192, C::kSmem, s>>>(args);
    MOE_LAUNCH_CHECK();
    return MOE_OK;
}

template <int NMAX>
int launch_bank(moe_ctx *ctx, bool cold, TcArgs a1, TcArgs a2, int units1, int units2, BankLists lists, int b,
                int T, int P, const WsLayout &lay, uint8_t *ws, const uint16_t *x, cudaStream_t s) {
    const Geom &g = ctx->g;
    __half *xs16 = (__half *)(ws + lay.xs16) + (size_t)b * T * g.H;
    int32_t *xexp = (int32_t *)(ws + lay.xexp) + (size_t)b * T;
    prep_x_kernel<<<T, 256, 0, s>>>(x, g.H, xs16, xexp);
    MOE_LAUNCH_CHECK();
    int r = cold ? launch_one<NMAX, 1, true>(ctx, a1, units1, s) : launch_one<NMAX, 1, false>(ctx, a1, units1, s);
    if (r) return r;
    prep_h_kernel<<<P, 256, 0, s>>>(lists, b, g.I, (const float *)(ws + lay.h32), (__half *)(ws + lay.h16),
                                    (int32_t *)(ws + lay.hexp));
    MOE_LAUNCH_CHECK();
    return cold ? launch_one<NMAX, 2, true>(ctx, a2, units2, s) : launch_one<NMAX, 2, false>(ctx, a2, units2, s);
}

}  // namespace

int launch_ffn_tc(moe_ctx *ctx, const uint8_t *bank, int b, const uint16_t *x, int T, uint8_t *ws, uint16_t *Y,
                  cudaStream_t s) {
    const Geom &g = ctx->g;
    WsLayout lay = ws_layout(g, T);
    const int P = T * g.k;
    BankLists lists;
    lists.hdr = (const int32_t *)(ws + lay.hdr);
    lists.act_row = (const int32_t *)(ws + lay.act_row) + (size_t)b * P;
    lists.act_off = (const int32_t *)(ws + lay.act_off) + (size_t)b * (P + 1);
    lists.picks = (const int32_t *)(ws + lay.picks) + (size_t)b * P;

    TcArgs a1{};
    a1.bank = bank;
    a1.eb = g.eb;
    a1.part_off = 0;
    a1.mt_count = g.mt13;
    a1.kc = g.kc13;
    a1.lists = lists;
    a1.b = b;
    a1.k = g.k;
    a1.H = g.H;
    a1.I = g.I;
    a1.bsrc = (const __half *)(ws + lay.xs16) + (size_t)b * T * g.H;
    a1.bsrc_ld = g.H;
    a1.bexp = (const int32_t *)(ws + lay.xexp) + (size_t)b * T;
    a1.h_out = (float *)(ws + lay.h32);
    a1.status = ctx->status_dev;
    TcArgs a2 = a1;
    a2.part_off = g.w2_off;
    a2.mt_count = g.mt2;
    a2.kc = g.kc2;
    a2.bsrc = (const __half *)(ws + lay.h16);
    a2.bsrc_ld = g.I;
    a2.bexp = (const int32_t *)(ws + lay.hexp);
    a2.h_out = nullptr;
    a2.Y = Y;

    const bool cold = b == MOE_BANK_COLD;
    const int rows = P;   // active rows never exceed the picks
    const int units1 = rows * g.mt13, units2 = rows * g.mt2;
    // the token-tile width depends only on T, so an expert's arithmetic is
    // the same in either bank
    if (T <= 16) return launch_bank<16>(ctx, cold, a1, a2, units1, units2, lists, b, T, P, lay, ws, x, s);
    if (T <= 64) return launch_bank<64>(ctx, cold, a1, a2, units1, units2, lists, b, T, P, lay, ws, x, s);
    return launch_bank<256>(ctx, cold, a1, a2, units1, units2, lists, b, T, P, lay, ws, x, s);
}

}  // namespace moe
