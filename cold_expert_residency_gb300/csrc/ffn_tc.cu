// MXFP4 expert FFN on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// "vLLM: Pin Hot Experts", Results: the routed MXFP4 expert FFN (gate/up
// GEMM, SwiGLU, down GEMM) runs once per residency bank without finalize.
// Here one launch per GEMM covers one bank:
//
//   unit = (active bank row = one expert, 128-row M-tile [, token tile]);
//   D[128 x N] = A[128 x K] * B[N x K]^T accumulated in TMEM (fp32), with
//   A = the expert's MXFP4 weights dequantised exactly to f16 and
//   B = the expert's token rows (f16, each row scaled by a power of two so its
//   largest element lies in [2^13, 2^14); the epilogue undoes the scale).
//
// Warp roles:
//   producer    Weights: hot bank -> one 1-D bulk async copy (TMA) of each
//               4352-byte (M-tile, K-chunk) block; cold bank -> 16-byte
//               cp.async reads of the mapped host bank (the host-link
//               streaming path).  Token rows: 2-D tensor TMA boxes of 64 f16
//               per row with 128-byte swizzle from the pick-ordered row
//               array.  All into a shared-memory ring, completion on one
//               mbarrier per stage.
//   dequant     Thread m of a 4-warp group owns weight row m = TMEM lane m;
//               it converts 64 e2m1 codes with the hardware e2m1x2 -> f16x2
//               conversion, applies the e8m0 block scale (exact in f16) and
//               stores the 32 f16x2 columns into the group's TMEM A buffer.
//   epilogue    tcgen05.ld of D, the row's power of two undone, then SwiGLU
//               (gate and up rows meet in lanes l and l^16) or the bf16 row.
//   MMA         TMEM allocation; one lane issues tcgen05.mma (A from TMEM, B
//               from shared memory) and tcgen05.commit.
// Decode tiles (16 or 64 tokens): one dequant group that also runs the
// epilogue, 3-4 CTAs per SM.  Prefill tiles (192 tokens): one CTA per SM with
// four dequant groups (group g takes the chunks c = g mod 4, so four chunks
// are in flight), four dedicated epilogue warps and a double-buffered
// accumulator, so one tile's epilogue overlaps the next tile's MMAs.
//
// The arithmetic of a pick depends only on its expert's weights, its token
// row and the expert's token count (which fixes the tile), never on the bank,
// so the hot and cold banks and any swap give bit-identical rows.
//
// Every mbarrier wait is bounded; on timeout the kernel sets the status word
// to MOE_ETIMEOUT, lets its own copies in flight land, frees TMEM and returns.
#include "moe_internal.cuh"
#include "sm103_ptx.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

namespace moe {

namespace {

constexpr uint32_t kWaitLimit = 1u << 22;        // polls of the teardown drains
constexpr uint64_t kWaitNs = 1000000000ull;      // 1 s bound of a pipeline wait

struct TcArgs {
    const uint8_t *bank;
    int64_t eb, part_off;
    int mt_count, kc;
    BankLists lists;
    int b, k, H, I, P;
    const int32_t *bexp;    // [P] scale exponent of B row g
    float *h_out;           // phase 1 output [P][I] by g
    uint16_t *Y;            // phase 2 output [T*k][H] by slot
    int32_t *status;
    int32_t *sched;         // work counter of this launch (zeroed before it)
};

constexpr int kQ = 4;       // unit queue depth (producer -> the other roles)

// Bounded mbarrier wait: gives up after kWaitNs of wall-clock time, raising
// the CTA's abort flag and the launch status.  SUSP: each poll may suspend the
// thread (up to 20 us) instead of returning at once -- used by the decode
// tiles, whose 3-4 CTAs per SM otherwise spend issue slots polling.
template <bool SUSP>
__device__ __forceinline__ bool wait_one(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                         int32_t *status) {
    uint64_t t0 = 0;
    for (uint32_t i = 0;; ++i) {
        if (SUSP ? ptx::mbar_try_wait_suspend(bar, parity, 20000u) : ptx::mbar_try_wait(bar, parity)) return true;
        if ((i & (SUSP ? 3u : 255u)) == 0u) {
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

template <bool SUSP>
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                          int32_t *status) {
    bool ok = wait_one<SUSP>(bar, parity, abort_flag, status);
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

__device__ __forceinline__ int bank_offset(const BankLists &L, int b, int P) {
    return b == 0 ? 0 : P - L.hdr[kHdrNPicks + 1];
}

template <int NMAX>
struct TcCfg {
    static constexpr int kStages = NMAX <= 16 ? 8 : (NMAX <= 64 ? 5 : 7);
    static constexpr int kBStage = NMAX * 128;              // bytes of one B chunk (NMAX rows x 128 B)
    static constexpr bool kWide = NMAX >= 128;
    static constexpr int kDq = kWide ? 16 : 4;              // dequant warps
    static constexpr int kGroups = kDq / 4;                 // dequant groups (one TMEM lane set each)
    static constexpr int kABufs = kGroups > 1 ? kGroups : (NMAX <= 16 ? 3 : 2);
    static constexpr int kEpi = kWide ? 4 : 0;              // dedicated epilogue warps
    static constexpr int kDBufs = kEpi ? 2 : 1;             // accumulators in TMEM
    // token rows per tensor-TMA box: few large boxes for wide tiles (the TMA
    // engine's cost is per box), 16-row boxes for the few tokens of decode
    static constexpr int kBoxRows = kWide ? 64 : 16;
    static constexpr int kBoxBytes = kBoxRows * 128;
    static constexpr uint32_t kDCol = kABufs * 32;          // first D column (after the A buffers)
    static constexpr uint32_t kColsUsed = kDCol + kDBufs * NMAX;
    static constexpr uint32_t kCols = kColsUsed <= 128 ? 128 : (kColsUsed <= 256 ? 256 : 512);
    static_assert(kColsUsed <= 512, "tile does not fit in tensor memory");
    static constexpr int kProducer = kDq + kEpi;            // producer warp; the MMA warp follows
    static constexpr int kThreads = 32 * (kDq + kEpi + 2);
    static constexpr int kBars = 2 * kStages + 2 * kABufs + 2 * kDBufs + 2 * kQ;
    static constexpr size_t kSmem = 1024 + (size_t)kStages * (kBStage + kChunkBytes) + kBars * 8 + 16 + 4 * kQ;
};

// Epilogue metadata of NBLK column blocks of 16: lane q of block i holds, for
// column (blk0 + i*bstride)*16 + q, its slot and the exact power of two that
// undoes its row's scaling (0 past the tile's last column).
template <int NBLK>
__device__ __forceinline__ void load_meta(const BankLists &L, const TcArgs &args, int blk0, int bstride, int nn,
                                          int p, int g, int lane, int (&rs)[NBLK], float (&rsc)[NBLK]) {
#pragma unroll
    for (int i = 0; i < NBLK; ++i) {
        const int col = (blk0 + i * bstride) * 16 + (lane & 15);
        rs[i] = col < nn ? L.picks[p + col] : 0;
        rsc[i] = col < nn ? ldexpf(1.0f, args.bexp[g + col]) : 0.0f;
    }
}

// Drain NBLK column blocks of D (TMEM address dt = this warp's lane quarter,
// first D column) into h rows (phase 1) or bf16 Y rows (phase 2).  All 16
// columns of a block are computed together; only the stores are predicated.
template <int PHASE, int NBLK>
__device__ __forceinline__ void epilogue_cols(const TcArgs &args, uint32_t dt, int blk0, int bstride, int nn, int g,
                                              int mt, int quarter, int lane, const int (&rs)[NBLK],
                                              const float (&rsc)[NBLK]) {
    const int Nr = (nn + 15) & ~15;
    const int m = quarter * 32 + lane;
    uint32_t vv[32];
#pragma unroll
    for (int i = 0; i < NBLK; ++i) {
        const int c0 = (blk0 + i * bstride) * 16;
        if (c0 >= Nr) break;   // warp-uniform
        // contiguous column blocks are read 32 columns per TMEM load
        const bool pair = bstride == 1 && (i & 1) == 0 && i + 1 < NBLK && c0 + 16 < Nr;
        if ((i & 1) == 0 || bstride != 1) {
            if (pair) {
                ptx::tmem_ld32(dt + c0, vv);
            } else {
                uint32_t (&lo)[16] = *reinterpret_cast<uint32_t(*)[16]>(&vv[0]);
                ptx::tmem_ld16(dt + c0, lo);
            }
            ptx::tmem_wait_ld();
        }
        const uint32_t *v = vv + (bstride == 1 ? (i & 1) * 16 : 0);
        float d[16];
#pragma unroll
        for (int q = 0; q < 16; ++q)   // undo the row's power of two (exact)
            d[q] = __fmul_rn(__uint_as_float(v[q]), __shfl_sync(0xffffffffu, rsc[i], q));
        if (PHASE == 1) {
            float o[16];
#pragma unroll
            for (int q = 0; q < 16; ++q) o[q] = __shfl_xor_sync(0xffffffffu, d[q], 16);
            if (lane < 16) {
                float *dst = args.h_out + (int64_t)(g + c0) * args.I + 64 * mt + 16 * quarter + lane;
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                    // silu(gate) * up with silu(z) = z / (1 + e^-z)
                    const float hv = __fmul_rn(__fdividef(d[q], 1.0f + __expf(-d[q])), o[q]);
                    if (c0 + q < nn) dst[(int64_t)q * args.I] = hv;
                }
            }
        } else {
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                const int slot = __shfl_sync(0xffffffffu, rs[i], q);
                if (c0 + q < nn)
                    args.Y[(int64_t)slot * args.H + kMT * mt + m] = __bfloat16_as_ushort(__float2bfloat16_rn(d[q]));
            }
        }
    }
}

template <int NMAX, int PHASE, bool COLD>
__global__ void __launch_bounds__(TcCfg<NMAX>::kThreads, 1) ffn_tc_kernel(const __grid_constant__ CUtensorMap tmap,
                                                                         TcArgs args) {
    using C = TcCfg<NMAX>;
    constexpr int DQ = C::kDq, NA = C::kABufs, DB = C::kDBufs, S = C::kStages, G = C::kGroups;
    extern __shared__ uint8_t smem_raw[];
    // 128-byte-swizzled B stages need 1024-byte alignment
    uint8_t *smem = smem_raw + ((1024u - (ptx::smem_addr(smem_raw) & 1023u)) & 1023u);
    uint8_t *sB = smem;
    uint8_t *sA = sB + S * C::kBStage;
    uint64_t *bars = (uint64_t *)(sA + S * kChunkBytes);
    uint32_t *holder = (uint32_t *)(bars + C::kBars);
    volatile int *abort_flag = (volatile int *)(holder + 1);
    volatile int *uq = (volatile int *)(holder + 2);   // [kQ] unit queue
    auto bar = [&](int i) { return ptx::smem_addr(bars + i); };
    const int FULL = 0, EMPTY = S, AREADY = 2 * S, AFREE = 2 * S + NA, ACCREADY = 2 * S + 2 * NA,
              ACCFREE = ACCREADY + DB, UQFULL = ACCFREE + DB, UQEMPTY = UQFULL + kQ;
    constexpr int kEpiThreads = C::kEpi ? 32 * C::kEpi : 32 * DQ;   // threads that drain D
    constexpr int kQueueReaders = 32 * DQ + 32 * C::kEpi + 1;       // + the MMA thread
    constexpr int PROD = C::kProducer, MMAW = C::kProducer + 1;
    constexpr bool SUSP = !C::kWide;   // suspend-hinted waits for the decode tiles

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(bar(FULL + s), COLD ? 33 : 1);
            ptx::mbar_init(bar(EMPTY + s), 1);
        }
        for (int q = 0; q < kQ; ++q) {
            ptx::mbar_init(bar(UQFULL + q), 1);
            ptx::mbar_init(bar(UQEMPTY + q), kQueueReaders);
        }
        for (int i = 0; i < NA; ++i) {
            ptx::mbar_init(bar(AREADY + i), 128);   // the four warps of the chunk's group
            ptx::mbar_init(bar(AFREE + i), 1);
        }
        for (int i = 0; i < DB; ++i) {
            ptx::mbar_init(bar(ACCREADY + i), 1);
            ptx::mbar_init(bar(ACCFREE + i), kEpiThreads);
        }
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == PROD && lane == 0) ptx::prefetch_tmap(&tmap);
    if (warp == MMAW) {
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
    const int goff = bank_offset(L, args.b, args.P);

    // every role but the producer reads the unit sequence from the queue
    auto take_unit = [&](uint32_t ui, bool warp_wide, bool &ok) -> int {
        const int qs = ui % kQ;
        const bool w = warp_wide ? wait_warp<SUSP>(bar(UQFULL + qs), (ui / kQ) & 1, abort_flag, args.status)
                                 : wait_one<SUSP>(bar(UQFULL + qs), (ui / kQ) & 1, abort_flag, args.status);
        if (!w) {
            ok = false;
            return -1;
        }
        const int u = uq[qs];
        ptx::mbar_arrive(bar(UQEMPTY + qs));
        return u;
    };

    if (warp < DQ) {
        // ------------------------------------------------ dequant (+ epilogue)
        const int quarter = warp & 3, group = warp >> 2;
        const int m = quarter * 32 + lane;
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        constexpr int NB = (NMAX / 16 + G - 1) / G;   // this warp's D column blocks when it drains D
        uint32_t it = 0, j = 0;
        bool ok = true;
        for (uint32_t ui = 0; ok; ++ui) {
            const int u = take_unit(ui, true, ok);
            if (u < 0) break;
            const int a = u / args.mt_count, mt = u % args.mt_count;
            const int p0 = L.act_off[a], n = L.act_off[a + 1] - p0;
            for (int n0 = 0; ok && n0 < n; n0 += NMAX, ++j) {
                const int nn = min(NMAX, n - n0);
                int rs[NB];
                float re[NB];
                if (C::kEpi == 0) load_meta<NB>(L, args, group, G, nn, p0 + n0, goff + p0 + n0, lane, rs, re);
                for (int c = 0; c < kc; ++c, ++it) {
                    if (G > 1 && (int)(it % G) != group) continue;   // another group's chunk
                    const int st = it % S;
                    if (!wait_warp<SUSP>(bar(FULL + st), (it / S) & 1, abort_flag, args.status)) { ok = false; break; }
                    const uint8_t *a_st = sA + st * kChunkBytes;
                    const int abuf = it % NA;
                    const uint32_t ua = it / NA;
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
                    if (ua > 0 && !wait_warp<SUSP>(bar(AFREE + abuf), (ua - 1) & 1, abort_flag, args.status)) {
                        ok = false;
                        break;
                    }
                    ptx::tmem_st32(tmem + lane_base + abuf * 32, r);
                    ptx::tmem_wait_st();
                    ptx::tc_fence_before();
                    ptx::mbar_arrive(bar(AREADY + abuf));
                }
                if (!ok) break;
                if (C::kEpi == 0) {
                    if (!wait_warp<SUSP>(bar(ACCREADY), j & 1, abort_flag, args.status)) { ok = false; break; }
                    ptx::tc_fence_after();
                    epilogue_cols<PHASE, NB>(args, tmem + lane_base + C::kDCol, group, G, nn, goff + p0 + n0, mt,
                                             quarter, lane, rs, re);
                    ptx::tc_fence_before();
                    ptx::mbar_arrive(bar(ACCFREE));
                }
            }
        }
    } else if (C::kEpi && warp < DQ + C::kEpi) {
        // -------------------------------------------------------- epilogue
        const int quarter = warp & 3;
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        constexpr int NB = NMAX / 16;
        uint32_t j = 0;
        bool ok = true;
        for (uint32_t ui = 0; ok; ++ui) {
            const int u = take_unit(ui, true, ok);
            if (u < 0) break;
            const int a = u / args.mt_count, mt = u % args.mt_count;
            const int p0 = L.act_off[a], n = L.act_off[a + 1] - p0;
            for (int n0 = 0; ok && n0 < n; n0 += NMAX, ++j) {
                const int nn = min(NMAX, n - n0);
                int rs[NB];
                float re[NB];
                load_meta<NB>(L, args, 0, 1, nn, p0 + n0, goff + p0 + n0, lane, rs, re);
                const int db = j % DB;
                if (!wait_warp<SUSP>(bar(ACCREADY + db), (j / DB) & 1, abort_flag, args.status)) { ok = false; break; }
                ptx::tc_fence_after();
                epilogue_cols<PHASE, NB>(args, tmem + lane_base + C::kDCol + db * NMAX, 0, 1, nn, goff + p0 + n0,
                                         mt, quarter, lane, rs, re);
                ptx::tc_fence_before();
                ptx::mbar_arrive(bar(ACCFREE + db));
            }
        }
    } else if (warp == PROD) {
        // ------------------------------------------------------------ producer
        uint32_t it = 0;
        bool ok = true;
        for (uint32_t ui = 0; ok; ++ui) {
            // take the next unit from the launch's work counter and publish it
            const int qs = ui % kQ;
            if (ui >= (uint32_t)kQ &&
                !wait_warp<SUSP>(bar(UQEMPTY + qs), ((ui / kQ) - 1) & 1, abort_flag, args.status)) {
                ok = false;
                break;
            }
            int u = 0;
            if (lane == 0) {
                u = atomicAdd(args.sched, 1);
                if (u >= units) u = -1;
                uq[qs] = u;
                ptx::mbar_arrive(bar(UQFULL + qs));
            }
            u = __shfl_sync(0xffffffffu, u, 0);
            if (u < 0) break;
            const int a = u / args.mt_count, mt = u % args.mt_count;
            const int row = L.act_row[a];
            const int p0 = L.act_off[a], n = L.act_off[a + 1] - p0;
            const uint8_t *tile = args.bank + (int64_t)row * args.eb + args.part_off +
                                  (int64_t)mt * kc * kChunkBytes;
            for (int n0 = 0; ok && n0 < n; n0 += NMAX) {
                const int nn = min(NMAX, n - n0);
                const int nbox = (nn + C::kBoxRows - 1) / C::kBoxRows;
                const int brow = goff + p0 + n0;
                for (int c = 0; c < kc; ++c, ++it) {
                    const int st = it % S;
                    const uint32_t rnd = it / S;
                    if (rnd > 0 && !wait_warp<SUSP>(bar(EMPTY + st), (rnd - 1) & 1, abort_flag, args.status)) {
                        ok = false;
                        break;
                    }
                    const uint32_t a_addr = ptx::smem_addr(sA + st * kChunkBytes);
                    const uint32_t b_addr = ptx::smem_addr(sB + st * C::kBStage);
                    const uint8_t *src_chunk = tile + (int64_t)c * kChunkBytes;
                    if (COLD) {
                        for (int i = lane; i < kChunkBytes / 16; i += 32) ptx::cp_async16(a_addr + i * 16, src_chunk + i * 16);
                        ptx::cp_async_arrive_noinc(bar(FULL + st));
                    }
                    if (lane == 0) {
                        ptx::mbar_arrive_expect_tx(bar(FULL + st), (COLD ? 0u : (uint32_t)kChunkBytes) + nbox * C::kBoxBytes);
                        if (!COLD) ptx::bulk_g2s(a_addr, src_chunk, kChunkBytes, bar(FULL + st));
                        for (int q = 0; q < nbox; ++q)
                            ptx::tma_load_2d(b_addr + q * C::kBoxBytes, &tmap, c * kKC, brow + q * C::kBoxRows,
                                             bar(FULL + st));
                    }
                    __syncwarp();
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
    } else if (warp == MMAW && lane == 0) {
        // ----------------------------------------------------------- MMA issue
        uint32_t it = 0, j = 0;
        bool ok = true;
        for (uint32_t ui = 0; ok; ++ui) {
            const int u = take_unit(ui, false, ok);
            if (u < 0) break;
            const int a = u / args.mt_count;
            const int n = L.act_off[a + 1] - L.act_off[a];
            for (int n0 = 0; ok && n0 < n; n0 += NMAX, ++j) {
                const int nn = min(NMAX, n - n0);
                const int Nr = (nn + 15) & ~15;
                const uint32_t idesc = ptx::idesc_f16_f32(128, Nr);
                const int db = j % DB;
                if (j >= (uint32_t)DB &&
                    !wait_one<SUSP>(bar(ACCFREE + db), ((j / DB) - 1) & 1, abort_flag, args.status)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem + C::kDCol + db * NMAX;
                for (int c = 0; c < kc; ++c, ++it) {
                    const int st = it % S, abuf = it % NA;
                    if (!wait_one<SUSP>(bar(AREADY + abuf), (it / NA) & 1, abort_flag, args.status)) { ok = false; break; }
                    ptx::tc_fence_after();
                    const uint32_t b_addr = ptx::smem_addr(sB + st * C::kBStage);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t bd = ptx::smem_desc_sw128(b_addr + kk * 32);
                        ptx::mma_f16_ts(d_tmem, tmem + abuf * 32 + kk * 8, bd, idesc, (c | kk) != 0);
                    }
                    ptx::mma_commit(bar(EMPTY + st));
                    ptx::mma_commit(bar(AFREE + abuf));
                }
                if (!ok) break;
                ptx::mma_commit(bar(ACCREADY + db));
            }
        }
        if (!ok && it > 0) {
            // wait until the MMAs already issued have retired (bounded)
            const uint32_t last = it - 1;
            for (uint32_t t = 0; t < kWaitLimit; ++t)
                if (ptx::mbar_try_wait(bar(AFREE + (last % NA)), (last / NA) & 1)) break;
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == MMAW) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, C::kCols);
    }
}

// Gather this bank's token rows in pick order, each scaled by a power of two
// into f16 (largest |x| -> [2^13, 2^14)): row g = offset + p of xg.
__global__ void __launch_bounds__(256) prep_x_kernel(const uint16_t *__restrict__ x, int H, int k, BankLists L,
                                                     int b, int P, __half *__restrict__ xg,
                                                     int32_t *__restrict__ xgexp, int32_t *sched) {
    __shared__ float red[8];
    const int p = blockIdx.x;
    // reset the work counters of this bank's two GEMM launches (stream-ordered before them)
    if (p == 0 && threadIdx.x < 2) sched[threadIdx.x] = 0;
    if (p >= L.hdr[kHdrNPicks + b]) return;
    const int g = bank_offset(L, b, P) + p;
    const int t = L.picks[p] / k;
    const uint4 *row = (const uint4 *)(x + (int64_t)t * H);
    const int n8 = H / 8;
    float mx = 0.0f;
    for (int i = threadIdx.x; i < n8; i += blockDim.x) {
        const uint4 v = row[i];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q)
            mx = fmaxf(mx, fmaxf(fabsf(__uint_as_float(w[q] << 16)), fabsf(__uint_as_float(w[q] & 0xFFFF0000u))));
    }
    for (int off = 16; off; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
    __syncthreads();
    mx = red[0];
    for (int i = 1; i < (int)(blockDim.x >> 5); ++i) mx = fmaxf(mx, red[i]);
    int e = 0;
    frexpf(mx, &e);
    const int c = mx > 0.0f ? e - 14 : 0;
    uint4 *dst = (uint4 *)(xg + (int64_t)g * H);
    for (int i = threadIdx.x; i < n8; i += blockDim.x) {
        const uint4 v = row[i];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            __half2 h = __floats2half2_rn(ldexpf(__uint_as_float(w[q] << 16), -c),
                                          ldexpf(__uint_as_float(w[q] & 0xFFFF0000u), -c));
            o[q] = *reinterpret_cast<uint32_t *>(&h);
        }
        dst[i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
    if (threadIdx.x == 0) xgexp[g] = c;
}

// Scale this bank's gate/up rows h (fp32, row g) into f16 the same way.
__global__ void __launch_bounds__(256) prep_h_kernel(BankLists L, int b, int P, int I,
                                                     const float *__restrict__ h32, __half *__restrict__ h16,
                                                     int32_t *__restrict__ hexp) {
    __shared__ float red[8];
    const int p = blockIdx.x;
    if (p >= L.hdr[kHdrNPicks + b]) return;
    const int g = bank_offset(L, b, P) + p;
    const float4 *row = (const float4 *)(h32 + (int64_t)g * I);
    const int n4 = I / 4;
    float mx = 0.0f;
    for (int i = threadIdx.x; i < n4; i += blockDim.x) {
        const float4 v = row[i];
        mx = fmaxf(mx, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
    for (int off = 16; off; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
    __syncthreads();
    mx = red[0];
    for (int i = 1; i < (int)(blockDim.x >> 5); ++i) mx = fmaxf(mx, red[i]);
    int e = 0;
    frexpf(mx, &e);
    const int c = mx > 0.0f ? e - 14 : 0;
    uint2 *dst = (uint2 *)(h16 + (int64_t)g * I);
    for (int i = threadIdx.x; i < n4; i += blockDim.x) {
        const float4 v = row[i];
        __half2 a = __floats2half2_rn(ldexpf(v.x, -c), ldexpf(v.y, -c));
        __half2 bb = __floats2half2_rn(ldexpf(v.z, -c), ldexpf(v.w, -c));
        dst[i] = make_uint2(*reinterpret_cast<uint32_t *>(&a), *reinterpret_cast<uint32_t *>(&bb));
    }
    if (threadIdx.x == 0) hexp[g] = c;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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

// Tensor map over a [rows][K] f16 array: boxes of box_rows rows x 64
// elements, 128-byte swizzle, zero fill past the last row.
int make_row_map(CUtensorMap *map, const void *base, int K, int rows, int box_rows) {
    auto enc = tensor_map_encoder();
    if (!enc) return set_error(MOE_ECUDA, "cuTensorMapEncodeTiled unavailable");
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    cuuint32_t box[2] = {(cuuint32_t)kKC, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return set_error(MOE_ECUDA, "cuTensorMapEncodeTiled failed: " + std::to_string((int)r));
    return MOE_OK;
}

template <int NMAX, int PHASE, bool COLD>
int launch_one(const CUtensorMap &map, const TcArgs &args, int blocks, cudaStream_t s) {
    using C = TcCfg<NMAX>;
    auto kern = ffn_tc_kernel<NMAX, PHASE, COLD>;
    MOE_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem));
    if (blocks < 1) return MOE_OK;
    kern<<<blocks, C::kThreads, C::kSmem, s>>>(map, args);
    MOE_LAUNCH_CHECK();
    return MOE_OK;
}

// Grid of one GEMM launch.  Units are handed out dynamically, so the grid
// only sets how many CTAs stream at once.  A cold-bank launch needs few CTAs
// to keep the host link busy; when the layer also has a hot bank, the hot
// launch leaves room on every SM for those, so both banks run concurrently.
template <int NMAX>
int grid_for(const moe_ctx *ctx, bool cold, bool shared, int units_max) {
    const int per_sm = NMAX <= 16 ? 4 : (NMAX <= 64 ? 3 : 1);   // shared memory and TMEM both fit
    const int cold_ctas = NMAX <= 64 ? 64 : 32;
    int blocks;
    if (cold) blocks = cold_ctas;
    else if (!shared) blocks = ctx->sms * per_sm;
    else if (per_sm > 1) blocks = ctx->sms * (per_sm - 1);
    else blocks = ctx->sms - cold_ctas;
    return std::max(1, std::min(units_max, blocks));
}

template <int NMAX>
int launch_bank(moe_ctx *ctx, bool cold, bool shared, const TcArgs &a1, const TcArgs &a2, int units1, int units2,
                const uint16_t *x, const WsLayout &lay, uint8_t *ws, cudaStream_t s) {
    const Geom &g = ctx->g;
    const int P = a1.P;
    CUtensorMap m1, m2;
    if (int r = make_row_map(&m1, ws + lay.xg16, g.H, P, TcCfg<NMAX>::kBoxRows)) return r;
    if (int r = make_row_map(&m2, ws + lay.h16, g.I, P, TcCfg<NMAX>::kBoxRows)) return r;
    prep_x_kernel<<<P, 256, 0, s>>>(x, g.H, g.k, a1.lists, a1.b, P, (__half *)(ws + lay.xg16),
                                    (int32_t *)(ws + lay.xgexp), a1.sched);
    MOE_LAUNCH_CHECK();
    const int b1 = grid_for<NMAX>(ctx, cold, shared, units1), b2 = grid_for<NMAX>(ctx, cold, shared, units2);
    int r = cold ? launch_one<NMAX, 1, true>(m1, a1, b1, s) : launch_one<NMAX, 1, false>(m1, a1, b1, s);
    if (r) return r;
    prep_h_kernel<<<P, 256, 0, s>>>(a1.lists, a1.b, P, g.I, (const float *)(ws + lay.h32), (__half *)(ws + lay.h16),
                                    (int32_t *)(ws + lay.hexp));
    MOE_LAUNCH_CHECK();
    return cold ? launch_one<NMAX, 2, true>(m2, a2, b2, s) : launch_one<NMAX, 2, false>(m2, a2, b2, s);
}

}  // namespace

int launch_ffn_tc(moe_ctx *ctx, const uint8_t *bank, int b, const uint16_t *x, int T, uint8_t *ws, uint16_t *Y,
                  cudaStream_t s, bool shared) {
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
    a1.P = P;
    a1.bexp = (const int32_t *)(ws + lay.xgexp);
    a1.h_out = (float *)(ws + lay.h32);
    a1.status = ctx->status_dev;
    a1.sched = (int32_t *)(ws + lay.hdr) + kHdrSched + 2 * b;
    TcArgs a2 = a1;
    a2.sched = a1.sched + 1;
    a2.part_off = g.w2_off;
    a2.mt_count = g.mt2;
    a2.kc = g.kc2;
    a2.bexp = (const int32_t *)(ws + lay.hexp);
    a2.h_out = nullptr;
    a2.Y = Y;

    const bool cold = b == MOE_BANK_COLD;
    const int units1 = P * g.mt13, units2 = P * g.mt2;   // active rows never exceed the picks
    // The token-tile width depends only on T, so an expert's arithmetic is
    // the same in either bank.  Decode-sized steps use narrow tiles with
    // several CTAs per SM (an expert with more tokens than the tile loops over
    // token tiles); prefill-sized steps use 192-wide tiles (an expert's
    // ~T*k/E tokens in one tile), one CTA per SM.
    if (T <= 16) return launch_bank<16>(ctx, cold, shared, a1, a2, units1, units2, x, lay, ws, s);
    if (T <= 256) return launch_bank<64>(ctx, cold, shared, a1, a2, units1, units2, x, lay, ws, s);
    return launch_bank<192>(ctx, cold, shared, a1, a2, units1, units2, x, lay, ws, s);
}

}  // namespace moe
