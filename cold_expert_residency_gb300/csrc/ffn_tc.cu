// MXFP4 expert FFN on the 5th-generation tensor cores (tcgen05 + TMEM),
// block-scaled.
//
// "vLLM: Pin Hot Experts", Results: the routed MXFP4 expert FFN (gate/up
// GEMM, SwiGLU, down GEMM) runs once per residency bank without finalize.
// Here one launch per GEMM covers one bank:
//
//   unit = (active bank row = one expert, 128-row M-tile [, token tile]);
//   D[128 x N] = sum over 32-wide K blocks of (SFA * A) (SFB * B)^T, fp32 in
//   TMEM, by tcgen05.mma kind::mxf8f6f4 with e8m0 block scales, where
//   A = the expert's e2m1 weights with their own e8m0 scales (exact), and
//   B = the expert's token rows (bf16 x, or the fp32 gate/up output h), each
//       row scaled by a power of two so its largest |value| lies in (224, 448]
//       and carried as two e4m3 pieces: q1 = e4m3(v), q2 = e4m3(16 (v - q1)).
//       B's scales are constants (2^0 for q1, 2^-4 for q2); both pieces
//       accumulate into the same D, so v is represented to about 2^-8 of
//       itself; the epilogue undoes the row's power of two.
//
// Warp roles:
//   producer    Weights: one 1-D bulk async copy (TMA) of each 4352-byte
//               (M-tile, K-chunk) block, from HBM for the hot bank and from
//               the mapped pinned host bank for the cold bank (the
//               host-link streaming path: the copy engine of the SM reads
//               the host memory in place).  Token rows: 2-D tensor TMA boxes of 128
//               bytes (the chunk's two e4m3 pieces) per row with 128-byte
//               swizzle from the pick-ordered row array.  All into a
//               shared-memory ring, completion on one mbarrier per stage.
//   unpack      Thread m of a 4-warp group owns weight row m = TMEM lane m;
//               per chunk it spreads its 64 e2m1 codes to one byte each
//               (two masked shifts per 8 codes, thanks to the device nibble
//               order) into the group's TMEM A slot, and its two e8m0 scale
//               bytes into the slot's scale column.
//   epilogue    tcgen05.ld of D, the row's power of two undone, then SwiGLU
//               (gate and up rows meet in lanes l and l^16) or the bf16 row.
//   MMA         TMEM allocation; one lane issues tcgen05.mma (A and the
//               scales from TMEM, B from shared memory) and tcgen05.commit.
// Decode tiles (16 or 64 tokens): one unpack group that also runs the
// epilogue, 3-4 CTAs per SM.  Prefill tiles (192 tokens): one CTA per SM with
// two unpack groups (group g takes the chunks c = g mod 2), four dedicated
// epilogue warps and a double-buffered accumulator, so one tile's epilogue
// overlaps the next tile's MMAs.
//
// The arithmetic of a pick depends only on its expert's weights, its token
// row and the step's token count (which fixes the tile), never on the bank,
// so the hot and cold banks and any swap give bit-identical rows.
//
// Every mbarrier wait is bounded; on timeout the kernel sets the status word
// to MOE_ETIMEOUT, lets its own copies in flight land, frees TMEM and returns.
#include "moe_internal.cuh"
#include "sm103_ptx.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp8.h>

namespace moe {

namespace {

constexpr uint32_t kWaitLimit = 1u << 22;        // polls of the teardown drains
constexpr uint64_t kWaitNs = 1000000000ull;      // 1 s bound of a pipeline wait

struct TcArgs {
    const uint8_t *bank[2];  // device-visible base of the hot (HBM) and cold (mapped host) bank
    int64_t eb, part_off;
    int mt_count, kc;
    BankLists lists[2];      // both banks' split lists
    int b;                   // the bank this launch covers, or -1: both banks in one launch
    int k, H, I, P;
    const int32_t *bexp;    // [P] scale exponent of B row g
    float *h_out;           // phase 1 output [P][I] by g
    uint16_t *Y;            // phase 2 output [T*k][H] by slot
    float *gu_out;          // split units, phase 1: [P][2I] gate/up sums by g (fp32, atomically added)
    float *y_out;           // split units, phase 2: [T*k][H] sums by slot (fp32, atomically added)
    int32_t *status;
    int32_t *sched;         // [2 banks][2 phases] work counters (zeroed before the launch)
    int32_t *claim;         // both banks: [SM] first-CTA claims (zeroed before the launch)
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

// 8 e2m1 codes in the device nibble order (byte i: codes i and 4+i) -> two
// TMEM columns of one code per byte, code in bits 5..2.
__device__ __forceinline__ void unpack_word(uint32_t w, uint32_t &lo, uint32_t &hi) {
    lo = (w << 2) & 0x3C3C3C3Cu;
    hi = (w >> 2) & 0x3C3C3C3Cu;
}

// Unit u -> active row a, M-tile mt and its K-chunk range [c0, c1) (one of
// ks equal K parts).
__device__ __forceinline__ void unit_pos(int u, int mt_count, int kc, int ks, int &a, int &mt, int &c0, int &c1) {
    const int per = mt_count * ks;
    a = u / per;
    const int r = u - a * per;
    mt = r / ks;
    const int h = r - mt * ks;
    c0 = h * kc / ks;
    c1 = (h + 1) * kc / ks;
}

__device__ __forceinline__ int bank_offset(const BankLists &L, int b, int P) {
    return b == 0 ? 0 : P - L.hdr[kHdrNPicks + 1];
}

template <int NMAX>
struct TcCfg {
    static constexpr bool kWide = NMAX >= 128;
    // 16-token tiles stack the two e4m3 pieces as token rows [0, Nr) and
    // [Nr, 2 Nr) of one MMA (half the MMA instructions); wider tiles issue
    // one MMA per piece.
    static constexpr bool kStack = NMAX <= 16;
    static constexpr int kStages = NMAX <= 8 ? 8 : (NMAX <= 16 ? 6 : (NMAX <= 64 ? 5 : 7));
    static constexpr int kBStage = (kStack ? 2 : 1) * NMAX * 128;   // bytes of one B chunk (rows x 128 B)
    static constexpr int kDq = kWide ? 8 : 4;               // unpack warps
    static constexpr int kGroups = kDq / 4;                 // unpack groups (one TMEM lane set each)
    static constexpr int kABufs = kWide ? 4 : (NMAX <= 16 ? 3 : 2);   // TMEM A slots
    static constexpr int kEpi = kWide ? 4 : 0;              // dedicated epilogue warps
    static constexpr int kDBufs = kEpi ? 2 : 1;             // accumulators in TMEM
    // token rows per tensor-TMA box: few large boxes for wide tiles (the TMA
    // engine's cost is per box), 16-row boxes for the few tokens of decode
    static constexpr int kBoxRows = kWide ? 64 : (NMAX <= 8 ? 8 : 16);
    static constexpr int kBoxBytes = kBoxRows * 128;
    // token rows of one piece are padded to a multiple of kRowQ (8-token tiles:
    // pieces at rows [0, 8) and [8, 16) of an N = 16 MMA)
    static constexpr int kRowQ = kStack ? kBoxRows : 16;
    // Tensor memory columns.  Slot s owns the 32-column block at
    // kBlk + 32 s: its A scale columns at +0 (quarter q reads +q), its A
    // codes (64 bytes = 16 columns) at +16; blocks 0 and 1 also hold the B
    // scale columns of e4m3 piece 0 and 1 at +8 (one per 32 B rows; stacked
    // tiles use block 0's for both pieces).  The accumulators (kDW columns
    // each) take their own range.
    static constexpr int kDW = (kStack ? 2 : 1) * NMAX;
    static constexpr int kNCol = (kDW + 31) / 32;
    static constexpr uint32_t kBlk = kWide ? kDBufs * NMAX : 0;
    static constexpr uint32_t kDCol = kWide ? 0 : 32 * kABufs;
    static constexpr uint32_t kSfaCol = kBlk;
    static constexpr uint32_t kACol = kBlk + 16;
    static constexpr uint32_t kSfbCol = kBlk + 8;
    static constexpr uint32_t kSfbStride = 32;              // piece 1 in the next block
    static constexpr uint32_t kColsUsed = kWide ? kBlk + 32 * kABufs : kDCol + kDBufs * kDW;
    static constexpr uint32_t kCols = kColsUsed <= 128 ? 128 : (kColsUsed <= 256 ? 256 : 512);
    static_assert(kColsUsed <= 512, "tile does not fit in tensor memory");
    static_assert(kABufs >= 2 && kNCol <= 8, "B scale columns");
    static_assert(NMAX % 8 == 0 && kDW % 16 == 0 && kBlk % 32 == 0 && kDCol % 32 == 0, "column alignment");
    static constexpr int kPerSm = NMAX <= 16 ? 4 : (NMAX <= 64 ? 3 : 1);   // resident CTAs per SM
    // Narrow tiles split each (expert, M-tile) unit into two K halves: a
    // decode step has only a few units per CTA, and halving them halves the
    // tail of the launch.  Two partial sums added onto zero in either order
    // give the same fp32 result, so the split stays deterministic.
    static constexpr int kSplit = kWide ? 1 : 2;
    static constexpr int kProducer = kDq + kEpi;            // producer warp; the MMA warp follows
    static constexpr int kThreads = 32 * (kDq + kEpi + 2);
    static constexpr int kBars = 2 * kStages + kABufs + 2 * kDBufs + 2 * kQ;
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
// STACK: column n + Nr holds the second e4m3 piece's product (16x scaled),
// so the token's value is D[n] + 2^-4 D[n + Nr].
template <int PHASE, int NBLK, bool STACK, int KS, int RQ>
__device__ __forceinline__ void epilogue_cols(const TcArgs &args, uint32_t dt, int blk0, int bstride, int nn, int g,
                                              int mt, int quarter, int lane, const int (&rs)[NBLK],
                                              const float (&rsc)[NBLK]) {
    const int Nr = (nn + RQ - 1) / RQ * RQ;
    const int m = quarter * 32 + lane;
    uint32_t vv[32];
#pragma unroll
    for (int i = 0; i < NBLK; ++i) {
        const int c0 = (blk0 + i * bstride) * 16;
        if (c0 >= Nr) break;   // warp-uniform
        float d[16];
        if (STACK && RQ == 8) {
            // 8-token tile: one load of the 16 columns, pieces at q and 8 + q
            uint32_t (&v)[16] = *reinterpret_cast<uint32_t(*)[16]>(&vv[0]);
            ptx::tmem_ld16(dt, v);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int q = 0; q < 16; ++q)
                d[q] = q < 8 ? __fmul_rn(__fmaf_rn(__uint_as_float(v[8 + (q & 7)]), 0.0625f, __uint_as_float(v[q & 7])),
                                         __shfl_sync(0xffffffffu, rsc[i], q))
                             : 0.0f;
        } else if (STACK) {
            uint32_t (&lo)[16] = *reinterpret_cast<uint32_t(*)[16]>(&vv[0]);
            uint32_t (&hi)[16] = *reinterpret_cast<uint32_t(*)[16]>(&vv[16]);
            ptx::tmem_ld16(dt + c0, lo);
            ptx::tmem_ld16(dt + Nr + c0, hi);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int q = 0; q < 16; ++q)   // pieces combined, then the row's power of two undone (exact)
                d[q] = __fmul_rn(__fmaf_rn(__uint_as_float(hi[q]), 0.0625f, __uint_as_float(lo[q])),
                                 __shfl_sync(0xffffffffu, rsc[i], q));
        } else {
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
#pragma unroll
            for (int q = 0; q < 16; ++q)   // undo the row's power of two (exact)
                d[q] = __fmul_rn(__uint_as_float(v[q]), __shfl_sync(0xffffffffu, rsc[i], q));
        }
        if (KS > 1) {
            // partial sums of one K half: added into fp32 rows; SwiGLU and the
            // bf16 rounding follow once both halves are in
            if (PHASE == 1) {
                // tile row m = W13 row (lane < 16 ? gate : up) of unit 64 mt + 16 quarter + lane % 16
                float *dst = args.gu_out + (int64_t)(g + c0) * (2 * args.I) + (lane < 16 ? 0 : args.I) + 64 * mt +
                             16 * quarter + (lane & 15);
#pragma unroll
                for (int q = 0; q < 16; ++q)
                    if (c0 + q < nn) atomicAdd(dst + (int64_t)q * (2 * args.I), d[q]);
            } else {
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                    const int slot = __shfl_sync(0xffffffffu, rs[i], q);
                    if (c0 + q < nn) atomicAdd(&args.y_out[(int64_t)slot * args.H + kMT * mt + m], d[q]);
                }
            }
        } else if (PHASE == 1) {
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

// BANKS names the launch (0 hot bank, 1 cold bank, 2 both banks); the code
// is the same, every unit carries its bank.
template <int NMAX, int PHASE, int BANKS>
__global__ void __launch_bounds__(TcCfg<NMAX>::kThreads, TcCfg<NMAX>::kPerSm) ffn_tc_kernel(const __grid_constant__ CUtensorMap tmap,
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
    // FULL: stage landed.  DONE: the chunk's MMAs completed (its stage and
    // its A slot are free again).  AREADY: A slot written.
    const int FULL = 0, DONE = S, AREADY = 2 * S, ACCREADY = 2 * S + NA, ACCFREE = ACCREADY + DB,
              UQFULL = ACCFREE + DB, UQEMPTY = UQFULL + kQ;
    constexpr int kEpiThreads = C::kEpi ? 32 * C::kEpi : 32 * DQ;   // threads that drain D
    constexpr int kQueueReaders = 32 * DQ + 32 * C::kEpi + 1;       // + the MMA thread
    constexpr int PROD = C::kProducer, MMAW = C::kProducer + 1;
    constexpr bool SUSP = !C::kWide;   // suspend-hinted waits for the decode tiles

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (BANKS == 1) {
        // A cold-bank launch keeps one host-link streamer per SM: a CTA placed
        // on an SM that already holds one leaves at once (two streamers on one
        // SM slow the hot-bank CTAs beside them).
        __shared__ int extra;
        if (tid == 0) {
            uint32_t smid;
            asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
            extra = atomicAdd(&args.claim[smid & 1023u], 1) > 0;
        }
        __syncthreads();
        if (extra) return;
    }
    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(bar(FULL + s), 1);
            ptx::mbar_init(bar(DONE + s), 1);
        }
        for (int q = 0; q < kQ; ++q) {
            ptx::mbar_init(bar(UQFULL + q), 1);
            ptx::mbar_init(bar(UQEMPTY + q), kQueueReaders);
        }
        for (int i = 0; i < NA; ++i) ptx::mbar_init(bar(AREADY + i), 128);   // the four warps of the chunk's group
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
    if (warp < 4) {
        // B scale columns, constant, in every lane quarter (each quarter
        // reads its own): 2^0; wide tiles scale the second piece by 2^-4
        // here, stacked tiles in the epilogue
        const uint32_t lb = (uint32_t)(warp * 32) << 16;
#pragma unroll
        for (int j = 0; j < C::kNCol; ++j) {
            ptx::tmem_st1(tmem + lb + C::kSfbCol + j, 0x7F7F7F7Fu);
            if (!C::kStack) ptx::tmem_st1(tmem + lb + C::kSfbCol + C::kSfbStride + j, 0x7B7B7B7Bu);
        }
        ptx::tmem_wait_st();   // made visible to the MMA by the first A-slot handoff
    }

    const int kc = args.kc;
    auto units_of = [&](int bk) { return args.lists[0].hdr[kHdrNAct + bk] * args.mt_count * C::kSplit; };

    // every role but the producer reads the unit sequence from the queue:
    // entry 2u + bank (unit u of that bank), or -1 at the end
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
        // ------------------------------------------------- unpack (+ epilogue)
        const int quarter = warp & 3, group = warp >> 2;
        const int m = quarter * 32 + lane;
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        constexpr int NB = ((NMAX + 15) / 16 + G - 1) / G;   // this warp's D column blocks when it drains D
        uint32_t it = 0, j = 0;
        bool ok = true;
        for (uint32_t ui = 0; ok; ++ui) {
            const int e = take_unit(ui, true, ok);
            if (e < 0) break;
            const int bk = e & 1;
            const BankLists &L = args.lists[bk];
            const int goff = bank_offset(L, bk, args.P);
            int a, mt, c0, c1;
            unit_pos(e >> 1, args.mt_count, kc, C::kSplit, a, mt, c0, c1);
            const int p0 = L.act_off[a], n = L.act_off[a + 1] - p0;
            for (int n0 = 0; ok && n0 < n; n0 += NMAX, ++j) {
                const int nn = min(NMAX, n - n0);
                int rs[NB];
                float re[NB];
                if (C::kEpi == 0) load_meta<NB>(L, args, group, G, nn, p0 + n0, goff + p0 + n0, lane, rs, re);
                for (int c = c0; c < c1; ++c, ++it) {
                    if (G > 1 && (int)(it % G) != group) continue;   // another group's chunk
                    const int st = it % S;
                    if (!wait_warp<SUSP>(bar(FULL + st), (it / S) & 1, abort_flag, args.status)) { ok = false; break; }
                    const uint8_t *a_st = sA + st * kChunkBytes;
                    const int abuf = it % NA;
                    const uint4 q0 = *(const uint4 *)(a_st + m * 16);
                    const uint4 q1 = *(const uint4 *)(a_st + 2048 + m * 16);
                    const uint32_t sc = *(const uint16_t *)(a_st + kChunkQBytes + 2 * m);
                    uint32_t r[16];
                    unpack_word(q0.x, r[0], r[1]);
                    unpack_word(q0.y, r[2], r[3]);
                    unpack_word(q0.z, r[4], r[5]);
                    unpack_word(q0.w, r[6], r[7]);
                    unpack_word(q1.x, r[8], r[9]);
                    unpack_word(q1.y, r[10], r[11]);
                    unpack_word(q1.z, r[12], r[13]);
                    unpack_word(q1.w, r[14], r[15]);
                    // the slot's previous chunk (it - NA) must have been consumed
                    if (it >= (uint32_t)NA && !wait_warp<SUSP>(bar(DONE + (it - NA) % S), ((it - NA) / S) & 1,
                                                               abort_flag, args.status)) {
                        ok = false;
                        break;
                    }
                    ptx::tmem_st16(tmem + lane_base + C::kACol + abuf * 32, r);
                    // the chunk's two K blocks' scales in bytes 0 and 1 of this quarter's column
                    ptx::tmem_st1(tmem + lane_base + C::kSfaCol + abuf * 32 + quarter, sc);
                    ptx::tmem_wait_st();
                    ptx::tc_fence_before();
                    ptx::mbar_arrive(bar(AREADY + abuf));
                }
                if (!ok) break;
                if (C::kEpi == 0) {
                    if (!wait_warp<SUSP>(bar(ACCREADY), j & 1, abort_flag, args.status)) { ok = false; break; }
                    ptx::tc_fence_after();
                    epilogue_cols<PHASE, NB, C::kStack, C::kSplit, C::kRowQ>(args, tmem + lane_base + C::kDCol, group, G, nn,
                                                        goff + p0 + n0, mt, quarter, lane, rs, re);
                    ptx::tc_fence_before();
                    ptx::mbar_arrive(bar(ACCFREE));
                }
            }
        }
    } else if (C::kEpi && warp < DQ + C::kEpi) {
        // -------------------------------------------------------- epilogue
        const int quarter = warp & 3;
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        constexpr int NB = (NMAX + 15) / 16;
        uint32_t j = 0;
        bool ok = true;
        for (uint32_t ui = 0; ok; ++ui) {
            const int e = take_unit(ui, true, ok);
            if (e < 0) break;
            const int bk = e & 1;
            const BankLists &L = args.lists[bk];
            const int goff = bank_offset(L, bk, args.P);
            int a, mt, c0, c1;
            unit_pos(e >> 1, args.mt_count, kc, C::kSplit, a, mt, c0, c1);
            const int p0 = L.act_off[a], n = L.act_off[a + 1] - p0;
            for (int n0 = 0; ok && n0 < n; n0 += NMAX, ++j) {
                const int nn = min(NMAX, n - n0);
                int rs[NB];
                float re[NB];
                load_meta<NB>(L, args, 0, 1, nn, p0 + n0, goff + p0 + n0, lane, rs, re);
                const int db = j % DB;
                if (!wait_warp<SUSP>(bar(ACCREADY + db), (j / DB) & 1, abort_flag, args.status)) { ok = false; break; }
                ptx::tc_fence_after();
                epilogue_cols<PHASE, NB, C::kStack, C::kSplit, C::kRowQ>(args, tmem + lane_base + C::kDCol + db * C::kDW, 0, 1, nn,
                                                    goff + p0 + n0, mt, quarter, lane, rs, re);
                ptx::tc_fence_before();
                ptx::mbar_arrive(bar(ACCFREE + db));
            }
        }
    } else if (warp == PROD) {
        // ------------------------------------------------------------ producer
        // A launch over both banks prefers, in the first CTA that reaches each
        // SM, the cold bank's units (one host-link streamer per SM) and in the
        // others the hot bank's; each turns to the other bank's queue once
        // its own is empty.
        int pref = args.b;
        if (args.b < 0) {
            if (lane == 0) {
                uint32_t smid;
                asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
                pref = atomicAdd(&args.claim[smid & 1023u], 1) == 0 ? MOE_BANK_COLD : MOE_BANK_HOT;
            }
            pref = __shfl_sync(0xffffffffu, pref, 0);
        }
        bool dry_pref = false, dry_other = args.b >= 0;   // lane 0's view of the queues
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
            int e = -1;
            if (lane == 0) {
                if (!dry_pref) {
                    const int u = atomicAdd(&args.sched[2 * pref + PHASE - 1], 1);
                    if (u < units_of(pref)) e = 2 * u + pref;
                    else dry_pref = true;
                }
                if (e < 0 && !dry_other) {
                    const int u = atomicAdd(&args.sched[2 * (1 - pref) + PHASE - 1], 1);
                    if (u < units_of(1 - pref)) e = 2 * u + (1 - pref);
                    else dry_other = true;
                }
                uq[qs] = e;
                ptx::mbar_arrive(bar(UQFULL + qs));
            }
            e = __shfl_sync(0xffffffffu, e, 0);
            if (e < 0) break;
            const int bk = e & 1;
            const BankLists &L = args.lists[bk];
            const int goff = bank_offset(L, bk, args.P);
            int a, mt, c0, c1;
            unit_pos(e >> 1, args.mt_count, kc, C::kSplit, a, mt, c0, c1);
            const int row = L.act_row[a];
            const int p0 = L.act_off[a], n = L.act_off[a + 1] - p0;
            const uint8_t *tile = args.bank[bk] + (int64_t)row * args.eb + args.part_off +
                                  (int64_t)mt * kc * kChunkBytes;
            for (int n0 = 0; ok && n0 < n; n0 += NMAX) {
                const int nn = min(NMAX, n - n0);
                const int nbox = (nn + C::kBoxRows - 1) / C::kBoxRows;
                const int brow = goff + p0 + n0;
                for (int c = c0; c < c1; ++c, ++it) {
                    const int st = it % S;
                    const uint32_t rnd = it / S;
                    if (rnd > 0 && !wait_warp<SUSP>(bar(DONE + st), (rnd - 1) & 1, abort_flag, args.status)) {
                        ok = false;
                        break;
                    }
                    const uint32_t a_addr = ptx::smem_addr(sA + st * kChunkBytes);
                    const uint32_t b_addr = ptx::smem_addr(sB + st * C::kBStage);
                    const uint8_t *src_chunk = tile + (int64_t)c * kChunkBytes;
                    if (lane == 0) {
                        ptx::mbar_arrive_expect_tx(bar(FULL + st),
                                                   (uint32_t)kChunkBytes + (C::kStack ? 2 : 1) * nbox * C::kBoxBytes);
                        // one bulk copy per weight chunk, from HBM or, for the cold
                        // bank, from the mapped host bank over the host link
                        ptx::bulk_g2s(a_addr, src_chunk, kChunkBytes, bar(FULL + st));
                        for (int q = 0; q < nbox; ++q)
                            ptx::tma_load_2d(b_addr + q * C::kBoxBytes, &tmap, c * 128, brow + q * C::kBoxRows,
                                             bar(FULL + st));
                        // stacked: the same rows again, 64 bytes further, so the
                        // second piece starts each row (rows nbox*16 ...; the last
                        // chunk's box reads past the row end: zero fill, unused)
                        if (C::kStack)
                            for (int q = 0; q < nbox; ++q)
                                ptx::tma_load_2d(b_addr + (nbox + q) * C::kBoxBytes, &tmap, c * 128 + 64,
                                                 brow + q * C::kBoxRows, bar(FULL + st));
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
            const int e = take_unit(ui, false, ok);
            if (e < 0) break;
            const BankLists &L = args.lists[e & 1];
            int a, mt, c0, c1;
            unit_pos(e >> 1, args.mt_count, kc, C::kSplit, a, mt, c0, c1);
            const int n = L.act_off[a + 1] - L.act_off[a];
            for (int n0 = 0; ok && n0 < n; n0 += NMAX, ++j) {
                const int nn = min(NMAX, n - n0);
                const int Nr = (nn + C::kRowQ - 1) / C::kRowQ * C::kRowQ;
                const int Nm = C::kStack ? 2 * Nr : Nr;                              // B rows of one MMA
                const uint32_t idesc0 = ptx::idesc_mx_e2m1_e4m3(128, Nm, 0, 0);   // K block 0 of the chunk
                const uint32_t idesc1 = ptx::idesc_mx_e2m1_e4m3(128, Nm, 1, 0);   // K block 1
                const int db = j % DB;
                if (j >= (uint32_t)DB &&
                    !wait_one<SUSP>(bar(ACCFREE + db), ((j / DB) - 1) & 1, abort_flag, args.status)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem + C::kDCol + db * C::kDW;
                for (int c = c0; c < c1; ++c, ++it) {
                    const int st = it % S, abuf = it % NA;
                    if (!wait_one<SUSP>(bar(AREADY + abuf), (it / NA) & 1, abort_flag, args.status)) { ok = false; break; }
                    ptx::tc_fence_after();
                    const uint32_t b_addr = ptx::smem_addr(sB + st * C::kBStage);
                    const uint32_t a_tm = tmem + C::kACol + abuf * 32;
                    const uint32_t sfa = tmem + C::kSfaCol + abuf * 32;
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk) {
#pragma unroll
                        for (int pc = 0; pc < (C::kStack ? 1 : 2); ++pc) {   // e4m3 piece of B (wide tiles)
                            const uint64_t bd = ptx::smem_desc_sw128(b_addr + pc * 64 + kk * 32);
                            ptx::mma_mxf8f6f4_ts(d_tmem, a_tm + kk * 8, bd, kk ? idesc1 : idesc0, sfa,
                                                 tmem + C::kSfbCol + pc * C::kSfbStride, (c != c0) | kk | pc);
                        }
                    }
                    ptx::mma_commit(bar(DONE + st));
                }
                if (!ok) break;
                ptx::mma_commit(bar(ACCREADY + db));
            }
        }
        if (!ok && it > 0) {
            // wait until the MMAs already issued have retired (bounded)
            const uint32_t last = it - 1;
            for (uint32_t t = 0; t < kWaitLimit; ++t)
                if (ptx::mbar_try_wait(bar(DONE + (last % S)), (last / S) & 1)) break;
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == MMAW) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, C::kCols);
    }
}

// Exponent e of a row whose largest |value| is mx: mx * 2^-e lies in
// (224, 448], the top binade of e4m3 (largest finite 448 = 0.875 * 2^9).
__device__ __forceinline__ int row_exponent(float mx) {
    if (!(mx > 0.0f)) return 0;
    int ex = 0;
    const float f = frexpf(mx, &ex);   // mx = f * 2^ex, f in [0.5, 1)
    return ex - 9 + (f > 0.875f ? 1 : 0);
}

// Eight scaled values -> the two e4m3 pieces (8 bytes each, value i in byte
// i): q1 = e4m3(v), q2 = e4m3(16 (v - q1)); v - q1 is exact in fp32.
__device__ __forceinline__ void split_e4m3x8(const float (&v)[8], uint2 &q1, uint2 &q2) {
    uint32_t a[4], r[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __nv_fp8x2_storage_t h = __nv_cvt_float2_to_fp8x2(make_float2(v[2 * i], v[2 * i + 1]), __NV_SATFINITE,
                                                               __NV_E4M3);
        const float2 back = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(h, __NV_E4M3)));
        const __nv_fp8x2_storage_t l = __nv_cvt_float2_to_fp8x2(
            make_float2(__fmul_rn(__fsub_rn(v[2 * i], back.x), 16.0f), __fmul_rn(__fsub_rn(v[2 * i + 1], back.y), 16.0f)),
            __NV_SATFINITE, __NV_E4M3);
        a[i] = h;
        r[i] = l;
    }
    q1 = make_uint2(a[0] | (a[1] << 16), a[2] | (a[3] << 16));
    q2 = make_uint2(r[0] | (r[1] << 16), r[2] | (r[3] << 16));
}

// Store values 8i..8i+7 of a row (K element 8i = chunk i/8, byte 8*(i%8)) as
// the two pieces of that chunk's 128-byte record.
__device__ __forceinline__ void store_pieces(uint8_t *row, int i, const float (&v)[8]) {
    uint2 q1, q2;
    split_e4m3x8(v, q1, q2);
    uint8_t *rec = row + (i >> 3) * 128 + (i & 7) * 8;
    *(uint2 *)rec = q1;
    *(uint2 *)(rec + 64) = q2;
}

__device__ __forceinline__ float block_max(float mx, float *red) {
    for (int off = 16; off; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
    __syncthreads();
    mx = red[0];
    for (int i = 1; i < (int)(blockDim.x >> 5); ++i) mx = fmaxf(mx, red[i]);
    return mx;
}

// Gather the bank's token rows in pick order (row g = offset + p of xq) as
// two e4m3 pieces per 64-wide chunk, each row scaled by 2^-e (e in xgexp).
// b0 >= 0: that bank; b0 < 0: both banks, bank = blockIdx.y.
__global__ void __launch_bounds__(256) prep_x_kernel(const uint16_t *__restrict__ x, int H, int k, BankLists L0,
                                                     BankLists L1, int b0, int P, uint8_t *__restrict__ xq,
                                                     int32_t *__restrict__ xgexp, int32_t *sched, int32_t *claim,
                                                     float *__restrict__ gu32, int I) {
    __shared__ float red[8];
    const int p = blockIdx.x, b = b0 >= 0 ? b0 : (int)blockIdx.y;
    const BankLists &L = b ? L1 : L0;
    if (p == 0 && blockIdx.y == 0) {
        // reset the work counters (and SM claims) of this call's GEMM launches,
        // stream-ordered before them; a one-bank call leaves the other bank's alone
        if (threadIdx.x < 4 && (b0 < 0 || (int)threadIdx.x / 2 == b0)) sched[threadIdx.x] = 0;
        if (claim)
            for (int i = threadIdx.x; i < 1024; i += blockDim.x) claim[i] = 0;
    }
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
    const int e = row_exponent(block_max(mx, red));
    uint8_t *dst = xq + (int64_t)g * H * 2;
    for (int i = threadIdx.x; i < n8; i += blockDim.x) {
        const uint4 v = row[i];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        float f[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            f[2 * q] = ldexpf(__uint_as_float(w[q] << 16), -e);
            f[2 * q + 1] = ldexpf(__uint_as_float(w[q] & 0xFFFF0000u), -e);
        }
        store_pieces(dst, i, f);
    }
    if (threadIdx.x == 0) xgexp[g] = e;
    if (gu32) {   // split units: clear this pick's gate/up sums before the gate/up GEMM adds into them
        float4 *z = (float4 *)(gu32 + (int64_t)g * 2 * I);
        for (int i = threadIdx.x; i < I / 2; i += blockDim.x) z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

// silu(gate) * up, silu(z) = z / (1 + e^-z)
__device__ __forceinline__ float swiglu(float gate, float up) {
    return __fmul_rn(__fdividef(gate, 1.0f + __expf(-gate)), up);
}

// Values 8i..8i+7 of row g of h: read from h32, or (split units) formed from
// the row's gate/up sums.
__device__ __forceinline__ void h_values(const float *h32, const float *gu32, int64_t g, int I, int i, float (&f)[8]) {
    if (gu32) {
        const float4 *gr = (const float4 *)(gu32 + g * 2 * I) + 2 * i, *ur = (const float4 *)(gu32 + g * 2 * I + I) + 2 * i;
        const float4 g0 = gr[0], g1 = gr[1], u0 = ur[0], u1 = ur[1];
        f[0] = swiglu(g0.x, u0.x); f[1] = swiglu(g0.y, u0.y); f[2] = swiglu(g0.z, u0.z); f[3] = swiglu(g0.w, u0.w);
        f[4] = swiglu(g1.x, u1.x); f[5] = swiglu(g1.y, u1.y); f[6] = swiglu(g1.z, u1.z); f[7] = swiglu(g1.w, u1.w);
    } else {
        const float4 *row = (const float4 *)(h32 + g * I) + 2 * i;
        const float4 a = row[0], c = row[1];
        f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = c.x; f[5] = c.y; f[6] = c.z; f[7] = c.w;
    }
}

// The same for this bank's gate/up rows h (row g).  Split units: h is formed
// here from the gate/up sums, and the pick's down-GEMM sum row is cleared.
__global__ void __launch_bounds__(256) prep_h_kernel(BankLists L0, BankLists L1, int b0, int P, int I,
                                                     const float *__restrict__ h32, const float *__restrict__ gu32,
                                                     uint8_t *__restrict__ hq, int32_t *__restrict__ hexp,
                                                     float *__restrict__ y32, int H, int32_t *claim) {
    __shared__ float red[8];
    const int p = blockIdx.x, b = b0 >= 0 ? b0 : (int)blockIdx.y;
    const BankLists &L = b ? L1 : L0;
    if (claim && p == 0 && blockIdx.y == 0)   // SM claims of the down GEMM's launch
        for (int i = threadIdx.x; i < 1024; i += blockDim.x) claim[i] = 0;
    if (p >= L.hdr[kHdrNPicks + b]) return;
    const int g = bank_offset(L, b, P) + p;
    const int n8 = I / 8;
    float mx = 0.0f;
    for (int i = threadIdx.x; i < n8; i += blockDim.x) {
        float f[8];
        h_values(h32, gu32, g, I, i, f);
#pragma unroll
        for (int q = 0; q < 8; ++q) mx = fmaxf(mx, fabsf(f[q]));
    }
    const int e = row_exponent(block_max(mx, red));
    uint8_t *dst = hq + (int64_t)g * I * 2;
    for (int i = threadIdx.x; i < n8; i += blockDim.x) {
        float f[8];
        h_values(h32, gu32, g, I, i, f);
#pragma unroll
        for (int q = 0; q < 8; ++q) f[q] = ldexpf(f[q], -e);
        store_pieces(dst, i, f);
    }
    if (threadIdx.x == 0) hexp[g] = e;
    if (y32) {
        float4 *z = (float4 *)(y32 + (int64_t)L.picks[p] * H);
        for (int i = threadIdx.x; i < H / 4; i += blockDim.x) z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

// Split units: this bank's down-GEMM sums (fp32, by slot) -> the bf16 rows of Y.
__global__ void __launch_bounds__(256) round_y_kernel(BankLists L0, BankLists L1, int b0, int H,
                                                      const float *__restrict__ y32, uint16_t *__restrict__ Y) {
    const int p = blockIdx.x, b = b0 >= 0 ? b0 : (int)blockIdx.y;
    const BankLists &L = b ? L1 : L0;
    if (p >= L.hdr[kHdrNPicks + b]) return;
    const int64_t slot = L.picks[p];
    const float4 *src = (const float4 *)(y32 + slot * H);
    uint2 *dst = (uint2 *)(Y + slot * H);
    for (int i = threadIdx.x; i < H / 4; i += blockDim.x) {
        const float4 v = src[i];
        const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
        dst[i] = make_uint2(*reinterpret_cast<const uint32_t *>(&lo), *reinterpret_cast<const uint32_t *>(&hi));
    }
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

// Tensor map over the [rows][K/64][128 B] piece records of K-element rows:
// boxes of box_rows rows x one 128-byte record, 128-byte swizzle, zero fill
// past the last row.
int make_row_map(CUtensorMap *map, const void *base, int K, int rows, int box_rows) {
    auto enc = tensor_map_encoder();
    if (!enc) return set_error(MOE_ECUDA, "cuTensorMapEncodeTiled unavailable");
    cuuint64_t dims[2] = {(cuuint64_t)K * 2, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    cuuint32_t box[2] = {128u, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return set_error(MOE_ECUDA, "cuTensorMapEncodeTiled failed: " + std::to_string((int)r));
    return MOE_OK;
}

template <int NMAX, int PHASE, int BANKS>
int launch_one(const CUtensorMap &map, const TcArgs &args, int blocks, cudaStream_t s) {
    using C = TcCfg<NMAX>;
    auto kern = ffn_tc_kernel<NMAX, PHASE, BANKS>;
    MOE_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem));
    if (blocks < 1) return MOE_OK;
    kern<<<blocks, C::kThreads, C::kSmem, s>>>(map, args);
    MOE_LAUNCH_CHECK();
    return MOE_OK;
}

// Grid of one GEMM launch.  Units are handed out dynamically, so the grid
// only sets how many CTAs stream at once.  A launch over both banks fills
// every SM with kPerSm CTAs.  One-bank launches: the host link needs a few
// MB in flight, so a cold-bank launch of narrow tiles takes one CTA per SM;
// when the layer also has a hot bank, the hot launch takes the SM's other
// slots, so two concurrent one-bank launches fit.
template <int NMAX>
int grid_for(const moe_ctx *ctx, int b, bool shared, int units_max) {
    const int per_sm = TcCfg<NMAX>::kPerSm;   // shared memory, registers and TMEM all fit
    const int cold_ctas = per_sm > 1 ? ctx->sms : 32;
    int blocks;
    if (b < 0) blocks = ctx->sms * per_sm;
    else if (b == MOE_BANK_COLD) blocks = cold_ctas;
    else if (!shared) blocks = ctx->sms * per_sm;
    else if (per_sm > 1) blocks = ctx->sms * (per_sm - 1);
    else blocks = ctx->sms - cold_ctas;
    return std::max(1, std::min(units_max, blocks));
}

template <int NMAX, int PHASE>
int launch_gemm(const CUtensorMap &map, const TcArgs &a, int blocks, cudaStream_t s) {
    if (a.b < 0) return launch_one<NMAX, PHASE, 2>(map, a, blocks, s);
    if (a.b == MOE_BANK_COLD) return launch_one<NMAX, PHASE, 1>(map, a, blocks, s);
    return launch_one<NMAX, PHASE, 0>(map, a, blocks, s);
}

template <int NMAX>
int launch_bank(moe_ctx *ctx, bool shared, const TcArgs &a1, const TcArgs &a2, int units1, int units2,
                const uint16_t *x, const WsLayout &lay, uint8_t *ws, cudaStream_t s) {
    const Geom &g = ctx->g;
    const int P = a1.P;
    const dim3 grid_p(P, a1.b < 0 ? 2 : 1);   // one block per pick (of each bank)
    CUtensorMap m1, m2;
    if (int r = make_row_map(&m1, ws + lay.xq, g.H, P, TcCfg<NMAX>::kBoxRows)) return r;
    if (int r = make_row_map(&m2, ws + lay.hq, g.I, P, TcCfg<NMAX>::kBoxRows)) return r;
    prep_x_kernel<<<grid_p, 256, 0, s>>>(x, g.H, g.k, a1.lists[0], a1.lists[1], a1.b, P, ws + lay.xq,
                                         (int32_t *)(ws + lay.xgexp), a1.sched, a1.claim, a1.gu_out, g.I);
    MOE_LAUNCH_CHECK();
    const int b1 = grid_for<NMAX>(ctx, a1.b, shared, units1), b2 = grid_for<NMAX>(ctx, a1.b, shared, units2);
    if (int r = launch_gemm<NMAX, 1>(m1, a1, b1, s)) return r;
    prep_h_kernel<<<grid_p, 256, 0, s>>>(a1.lists[0], a1.lists[1], a1.b, P, g.I, (const float *)(ws + lay.h32),
                                         a1.gu_out, ws + lay.hq, (int32_t *)(ws + lay.hexp), a2.y_out, g.H, a1.claim);
    MOE_LAUNCH_CHECK();
    if (int r = launch_gemm<NMAX, 2>(m2, a2, b2, s)) return r;
    if (!a2.y_out) return MOE_OK;
    round_y_kernel<<<grid_p, 256, 0, s>>>(a2.lists[0], a2.lists[1], a2.b, g.H, a2.y_out, a2.Y);
    MOE_LAUNCH_CHECK();
    return MOE_OK;
}

}  // namespace

int launch_ffn_tc(moe_ctx *ctx, const uint8_t *hot, const uint8_t *cold, int b, const uint16_t *x, int T,
                  uint8_t *ws, uint16_t *Y, cudaStream_t s, bool shared) {
    const Geom &g = ctx->g;
    WsLayout lay = ws_layout(g, T);
    const int P = T * g.k;

    TcArgs a1{};
    a1.bank[MOE_BANK_HOT] = hot;
    a1.bank[MOE_BANK_COLD] = cold;
    for (int bk = 0; bk < 2; ++bk) {
        BankLists &L = a1.lists[bk];
        L.hdr = (const int32_t *)(ws + lay.hdr);
        L.act_row = (const int32_t *)(ws + lay.act_row) + (size_t)bk * P;
        L.act_off = (const int32_t *)(ws + lay.act_off) + (size_t)bk * (P + 1);
        L.picks = (const int32_t *)(ws + lay.picks) + (size_t)bk * P;
    }
    a1.eb = g.eb;
    a1.part_off = 0;
    a1.mt_count = g.mt13;
    a1.kc = g.kc13;
    a1.b = b == MOE_BANK_BOTH ? -1 : b;
    a1.k = g.k;
    a1.H = g.H;
    a1.I = g.I;
    a1.P = P;
    a1.bexp = (const int32_t *)(ws + lay.xgexp);
    a1.h_out = (float *)(ws + lay.h32);
    a1.status = ctx->status_dev;
    a1.sched = (int32_t *)(ws + lay.hdr) + kHdrSched;
    // SM claims: a launch over both banks, or a cold-bank launch (one each;
    // the hot bank's concurrent launches never read them)
    a1.claim = (a1.b < 0 || a1.b == MOE_BANK_COLD) ? (int32_t *)(ws + lay.claim) : nullptr;
    TcArgs a2 = a1;
    a2.part_off = g.w2_off;
    a2.mt_count = g.mt2;
    a2.kc = g.kc2;
    a2.bexp = (const int32_t *)(ws + lay.hexp);
    a2.h_out = nullptr;
    a2.Y = Y;
    // narrow-tile steps: two K halves per unit, summed in fp32 rows
    const bool split = split_k_steps(T);
    a1.gu_out = split ? (float *)(ws + lay.gu32) : nullptr;
    a1.y_out = nullptr;
    a2.gu_out = nullptr;
    a2.y_out = split ? (float *)(ws + lay.y32) : nullptr;

    const int units1 = 4 * P * g.mt13, units2 = 4 * P * g.mt2;   // bound: active rows never exceed the picks
    // The token-tile width depends only on T, so an expert's arithmetic is
    // the same in either bank.  Decode-sized steps use narrow tiles with
    // several CTAs per SM (an expert with more tokens than the tile loops over
    // token tiles); prefill-sized steps use 192-wide tiles (an expert's
    // ~T*k/E tokens in one tile), one CTA per SM.
    if (T <= 8) return launch_bank<8>(ctx, shared, a1, a2, units1, units2, x, lay, ws, s);
    if (T <= 16) return launch_bank<16>(ctx, shared, a1, a2, units1, units2, x, lay, ws, s);
    if (T <= kNarrowMaxT) return launch_bank<64>(ctx, shared, a1, a2, units1, units2, x, lay, ws, s);
    return launch_bank<192>(ctx, shared, a1, a2, units1, units2, x, lay, ws, s);
}

}  // namespace moe
