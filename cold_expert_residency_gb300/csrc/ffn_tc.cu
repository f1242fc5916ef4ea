// MXFP4 expert FFN on the 5th-generation tensor cores (tcgen05 + TMEM),
// block-scaled.  This file holds the prefill-tile kernel, whose weights are
// moved only by the tensor memory accelerator, the row kernels around the
// GEMMs, and the launch code; decode tiles run the kernel in
// ffn_tc_decode.cuh (included below).
//
// "vLLM: Pin Hot Experts", Results: the routed MXFP4 expert FFN (gate/up
// GEMM, SwiGLU, down GEMM) runs once per residency bank without finalize.
// Here one launch per GEMM covers one bank (or both):
//
//   unit = (active bank row = one expert, 128-row M-tile [, K half for decode
//          tiles]);
//   D[128 x N] = sum over 32-wide K blocks of (SFA * A) (SFB * B)^T, fp32 in
//   TMEM, by tcgen05.mma kind::mxf8f6f4 with e8m0 block scales, where
//   A = the expert's e2m1 weights with their own e8m0 scales (exact), read
//       by the tensor cores from shared memory, and
//   B = the expert's token rows (bf16 x, or the gate/up output h), each
//       row scaled by a power of two so its largest |value| lies in (224, 448]
//       and carried as two e4m3 pieces: q1 = e4m3(v), q2 = e4m3(16 (v - q1)).
//       B's scales are constants (2^0 for q1, 2^-4 for q2); both pieces
//       accumulate into the same D, so v is represented to about 2^-8 of
//       itself; the epilogue undoes the row's power of two.
//
// No SM instruction touches a weight byte.  Warp roles:
//   producer  Per K group of 128: one tensor-TMA box of the padded 4-bit
//             type (the group's 8 KB code block becomes 16 KB of shared
//             memory in the layout the MMA reads, 128-byte swizzle), one bulk
//             copy of its 512-byte scale atom, and one box of the tile's
//             token rows (4-D tensor TMA, both e4m3 pieces of both 64-wide
//             chunks, 64-byte swizzle, from the pick-ordered row array); from
//             HBM for the hot bank, over the host link from the mapped pinned
//             host bank for the cold bank.  All into a ring of stages with one
//             mbarrier each; one thread issues them.
//   MMA       One warp runs the loop and one elected lane issues: per landed
//             stage, tcgen05.cp of its scale atom into the stage's
//             tensor-memory scale slot, the group's MMAs (four K blocks per
//             e4m3 piece, two for a half group), tcgen05.commit to free the
//             stage; it goes on through every following stage that has
//             landed too (one burst) before it waits again.  After a token
//             tile's last group, a commit hands its accumulator over.
//   epilogue  Four warps (thread m = accumulator row m): tcgen05.ld of D, the
//             row's power of two undone, then SwiGLU (gate and up rows meet
//             in lanes l and l^16) or the bf16 row.  Two accumulators, so a
//             tile's epilogue overlaps the next tile's MMAs.
// Prefill tiles (144 tokens with two-piece rows, 160 with MXFP8 rows) run one
// CTA per SM, the ring as deep as shared and tensor memory allow.
//
// The arithmetic of a pick depends only on its expert's weights, its token
// row and the step's token count (which fixes the tile), never on the bank,
// so the hot and cold banks and any swap give bit-identical rows.
//
// Every mbarrier wait is bounded; on timeout the kernel sets the status word
// to MOE_ETIMEOUT, lets its own copies in flight land, frees TMEM and returns.
#include "moe_internal.cuh"
#include "sm103_ptx.cuh"

#include <cudaTypedefs.h>
#include <cuda_fp8.h>

namespace moe {

namespace {

constexpr uint32_t kWaitLimit = 1u << 22;        // polls of the teardown drains

struct TcArgs {
    const uint8_t *bank[2];  // device-visible base of the hot (HBM) and cold (mapped host) bank
    int64_t eb;              // bytes per expert
    PartLayout part;         // this GEMM's part of an expert (W13 or W2)
    int ks;                  // K parts per (expert, M-tile) unit
    BankLists lists[2];      // both banks' split lists
    int b;                   // the bank this launch covers, or -1: both banks in one launch
    int k, H, I, P;
    const int32_t *bexp;    // [P] scale exponent of B row g
    float *h_out;           // phase 1 output [P][I] by g
    uint16_t *Y;            // phase 2 output [T*k][H] by slot
    float *gu_out;          // narrow tiles, phase 1: [P][2I] gate/up sums by g (fp32, atomically added)
    float *y_out;           // narrow tiles, phase 2: [T*k][H] sums by slot (fp32, atomically added)
    int32_t *status;
    int32_t *sched;         // [2 banks][2 phases] work counters (zeroed before the launch)
    int32_t *claim;         // [SM] first-CTA claims (zeroed before the launch)
    uint64_t wait_ns;       // bound of every pipeline wait (wall-clock ns)
    int32_t withhold;       // fault injection: the CTA that takes unit 0 of a bank skips its first group's copies
    // MXFP8 prefill tiles: per bank, the first tile of each active row and
    // the tiles' B-operand block scales [tile][group][kSfbGroupBytes]
    const int32_t *tile_off[2];
    const uint8_t *sfb[2];
    int sf_groups;          // K groups per tile in sfb
    // cold staging: the pool slot of each cold active row (or -1; null: no
    // staging in this call) and the pool's base
    const int32_t *stage_slot;
    const uint8_t *stage_pool;
};

// The pool slot that holds unit row a of bank bk this call, or -1.
__device__ __forceinline__ int staged_slot(const TcArgs &args, int bk, int a) {
    return (bk == 1 && args.stage_slot) ? args.stage_slot[a] : -1;
}

constexpr int kQ = 4;       // unit queue depth (producer -> the other roles)

// Position in a ring of S stages: the stage and the parity of its round,
// advanced without dividing by the launch-time S (a division by a runtime
// value costs about as much as the rest of a K step's bookkeeping).
struct RingPos {
    uint32_t st = 0, ph = 0;
    __device__ __forceinline__ void next(uint32_t S) {
        if (++st == S) {
            st = 0;
            ph ^= 1u;
        }
    }
};

// Bounded mbarrier wait: gives up after limit_ns of wall-clock time, raising
// the CTA's abort flag and the launch status.  SUSP: each poll may suspend the
// thread (up to 20 us) instead of returning at once -- used by the decode
// tiles, whose CTAs share an SM.
template <bool SUSP>
__device__ __forceinline__ bool wait_one(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                         int32_t *status, uint64_t limit_ns) {
    uint64_t t0 = 0;
    for (uint32_t i = 0;; ++i) {
        if (SUSP ? ptx::mbar_try_wait_suspend(bar, parity, 20000u) : ptx::mbar_try_wait(bar, parity)) return true;
        if ((i & (SUSP ? 3u : 255u)) == 0u) {
            if (*abort_flag) return false;
            const uint64_t now = ptx::globaltimer_ns();
            if (i == 0) {
                t0 = now;
            } else if (now - t0 > limit_ns) {
                *abort_flag = 1;
                atomicCAS(status, 0, MOE_ETIMEOUT);
                return false;
            }
        }
    }
}

template <bool SUSP>
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                          int32_t *status, uint64_t limit_ns) {
    // the warps that spread the weights mostly find their phase complete: a
    // non-blocking check costs less than a suspend-hinted wait
    bool ok = (SUSP && ptx::mbar_test_wait(bar, parity)) || wait_one<SUSP>(bar, parity, abort_flag, status, limit_ns);
    return __all_sync(0xffffffffu, ok);
}

// Unit u -> active row a, M-tile mt and its K-step range [s0, s1) (one of ks
// equal parts of the tile's ns K groups).
__device__ __forceinline__ void unit_pos(int u, int mt_count, int ns, int ks, int &a, int &mt, int &s0, int &s1) {
    const int per = mt_count * ks;
    a = u / per;
    const int r = u - a * per;
    mt = r / ks;
    const int h = r - mt * ks;
    s0 = h * ns / ks;
    s1 = (h + 1) * ns / ks;
}

__device__ __forceinline__ int bank_offset(const BankLists &L, int b, int P) {
    return b == 0 ? 0 : P - L.hdr[kHdrNPicks + 1];
}

template <int NMAX, bool MX = false>
struct TcCfg {
    // This kernel runs the prefill tiles; decode tiles run ffn_tc_decode_kernel.
    static_assert(NMAX >= 128 && NMAX <= 256 && NMAX % 16 == 0, "prefill tile");
    static constexpr bool kStack = false;                   // one MMA per e4m3 piece
    // One 4-D tensor-TMA box per stage brings the tile's token rows: the
    // e4m3 pieces (two, or one in the MXFP8 format) of both 64-wide chunks, as
    // [chunk][piece][NMAX rows][64 B] with 64-byte swizzle (rows past the
    // tile's tokens are loaded and unused).
    static constexpr int kPieces = MX ? 1 : 2;
    static constexpr int kBChunk = kPieces * NMAX * 64;     // one chunk: its pieces
    static constexpr int kBStage = 2 * kBChunk;
    static constexpr int kRowQ = 16;                        // token rows of a piece, padded to 16
    static constexpr int kAStage = 2 * kGroupQBytes;        // padded code block: 16 KB
    static constexpr int kSfbStage = MX ? kSfbGroupBytes : 0;   // the tile's B block scales of one group
    // One stage holds a group's 8.5 KB of weights as 16.5 KB of padded codes
    // and scales, plus the token rows (and their block scales).
    static constexpr int kStageBytes = kAStage + kBStage + kSfAtomBytes + kSfbStage;
    static constexpr int kDBufs = 2;                        // accumulators in TMEM
    static constexpr int kDW = NMAX;                        // columns of one accumulator
    static constexpr int kNCol = (kDW + 31) / 32;           // B scale columns of one piece
    // Ring stages, each with its own scale slot in tensor memory: stage s's
    // scales are copied into slot s, so a slot is rewritten only after the
    // producer has seen the stage's previous MMAs complete (the MMA warp
    // needs no wait of its own).  As many stages as shared memory holds (one
    // CTA per SM: 227 KB, less alignment slack, barriers and a few static
    // words), up to what tensor memory leaves for 32-column slots beside the
    // accumulators.
    static constexpr size_t kFixedSmem = 1024 + (2 * 8 + 2 * kDBufs + 2 * kQ) * 8 + 16 + 16 * kQ + 64;
    static constexpr int kSmemStages = (int)((227u * 1024u - kFixedSmem) / kStageBytes);
    static constexpr int kTmemStages = (512 - kDBufs * kDW) / 32;
    static constexpr int kStages = kSmemStages < kTmemStages ? (kSmemStages < 8 ? kSmemStages : 8)
                                                             : (kTmemStages < 8 ? kTmemStages : 8);
    static_assert(kStages >= 2, "ring too shallow");
    // Tensor memory columns: slot i's A scales at 32 i (four columns written
    // by tcgen05.cp); slot 0's block also holds the constant B scale columns
    // of piece 0 at +8 and of piece 1 at +16 -- in the MXFP8 format, slot i's
    // own B scale columns sit at 32 i + 8 (token blocks 0..7, one tcgen05.cp
    // per four blocks); then the accumulators.
    static constexpr uint32_t kSfbCol = 8;
    static constexpr uint32_t kSfbStride = 8;
    static constexpr uint32_t kDCol = 32 * kStages;
    static constexpr uint32_t kColsUsed = kDCol + kDBufs * kDW;
    static constexpr uint32_t kCols = 512;                  // one CTA per SM
    static_assert(kColsUsed <= kCols, "tile does not fit in tensor memory");
    static_assert(kNCol <= 8 && kSfbCol + kSfbStride + kNCol <= 32, "B scale columns");
    static constexpr int kSplit = 1;                        // whole-K units
    static constexpr int kProducer = 4, kMmaWarp = 5;
    static constexpr int kThreads = 192;
    static constexpr int kBars = 2 * kStages + 2 * kDBufs + 2 * kQ;
    static constexpr size_t kSmem = 1024 + (size_t)kStages * kStageBytes + kBars * 8 + 16 + 16 * kQ;
    static_assert(kSmem + 64 <= 227u * 1024u, "ring does not fit in shared memory");
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
// is the same, every unit carries its bank.  tmA0 / tmA1: the hot and cold
// bank's code-block maps of this GEMM's part; tmB: the token-row records.
template <int NMAX, int PHASE, int BANKS, bool MX>
__global__ void __launch_bounds__(TcCfg<NMAX, MX>::kThreads, 1)
    ffn_tc_kernel(const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmA0,
                  const __grid_constant__ CUtensorMap tmA1, const __grid_constant__ CUtensorMap tmA2, TcArgs args) {
    using C = TcCfg<NMAX, MX>;
    constexpr int DB = C::kDBufs, S = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    // 128-byte-swizzled stages need 1024-byte alignment
    uint8_t *smem = smem_raw + ((1024u - (ptx::smem_addr(smem_raw) & 1023u)) & 1023u);
    uint8_t *sA = smem;                          // [S][16 KB] padded code blocks
    uint8_t *sB = sA + S * C::kAStage;           // [S][2 chunks][2 pieces][NMAX rows][64 B] token rows
    uint8_t *sSF = sB + S * C::kBStage;          // [S][512] scale atoms
    uint8_t *sSFB = sSF + S * kSfAtomBytes;      // [S][kSfbStage] token rows' block scales (MXFP8)
    uint64_t *bars = (uint64_t *)(sSFB + S * C::kSfbStage);
    uint32_t *holder = (uint32_t *)(bars + C::kBars);
    volatile int *abort_flag = (volatile int *)(holder + 1);
    volatile int *uq = (volatile int *)(holder + 4);   // [kQ][4] unit queue
    auto bar = [&](int i) { return ptx::smem_addr(bars + i); };
    // FULL: stage landed.  DONE: the stage's MMAs completed (stage and scale
    // slot free again).  ACCREADY / ACCFREE: accumulator handover.
    const int FULL = 0, DONE = S, ACCREADY = 2 * S, ACCFREE = ACCREADY + DB, UQFULL = ACCFREE + DB,
              UQEMPTY = UQFULL + kQ;
    constexpr int kQueueReaders = 128 + 1;   // the epilogue warps and the MMA warp's lane 0
    constexpr bool SUSP = false;             // one CTA per SM: plain polling

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
        for (int i = 0; i < DB; ++i) {
            ptx::mbar_init(bar(ACCREADY + i), 1);
            ptx::mbar_init(bar(ACCFREE + i), 128);
        }
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == C::kProducer && lane == 0) {
        ptx::prefetch_tmap(&tmB);
        ptx::prefetch_tmap(&tmA0);
        ptx::prefetch_tmap(&tmA1);
        if (args.stage_slot) ptx::prefetch_tmap(&tmA2);
    }
    if (warp == C::kMmaWarp) {
        ptx::tmem_alloc(ptx::smem_addr(holder), C::kCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *holder;
    if (warp < 4 && !MX) {
        // B scale columns, constant, in every lane quarter (each quarter
        // reads its own): 2^0; wide tiles scale the second piece by 2^-4
        // here, stacked tiles in the epilogue
        const uint32_t lb = (uint32_t)(warp * 32) << 16;
#pragma unroll
        for (int j = 0; j < C::kNCol; ++j) {
            ptx::tmem_st1(tmem + lb + C::kSfbCol + j, 0x7F7F7F7Fu);
            if (!C::kStack) ptx::tmem_st1(tmem + lb + C::kSfbCol + C::kSfbStride + j, 0x7B7B7B7Bu);
        }
        ptx::tmem_wait_st();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();

    const PartLayout &part = args.part;
    const int ns = part.steps();
    auto units_of = [&](int bk) { return args.lists[0].hdr[kHdrNAct + bk] * part.tiles * args.ks; };

    // every role but the producer reads the unit sequence from the queue.
    // An entry is the unit as the producer resolved it: 2u + bank (unit u
    // of that bank, -1 at the end), its token count n, its first pick p0 and
    // its M-tile and K-step range -- so the other roles load nothing to
    // start a unit.  The epilogue warps wait with a suspend hint (a spinning
    // warp takes issue slots from the producer and MMA warps that share its
    // scheduler); the MMA warp spins, and only its lane 0 counts as a reader.
    struct Unit {
        int e, n, p0, mt, s0, s1;
    };
    auto take_unit = [&](uint32_t ui, bool epilogue, bool &ok) -> Unit {
        const int qs = ui % kQ;
        const uint32_t ph = (ui / kQ) & 1;
        const bool w = epilogue ? wait_warp<true>(bar(UQFULL + qs), ph, abort_flag, args.status, args.wait_ns)
                                : wait_warp<SUSP>(bar(UQFULL + qs), ph, abort_flag, args.status, args.wait_ns);
        Unit u{-1, 0, 0, 0, 0, 0};
        if (!w) {
            ok = false;
            return u;
        }
        // lane 0's reads, so the warp holds the values uniformly
        u.e = __shfl_sync(0xffffffffu, uq[4 * qs + 0], 0);
        u.n = __shfl_sync(0xffffffffu, uq[4 * qs + 1], 0);
        u.p0 = __shfl_sync(0xffffffffu, uq[4 * qs + 2], 0);
        const int r = __shfl_sync(0xffffffffu, uq[4 * qs + 3], 0);
        u.mt = r & 0xFF;
        u.s0 = (r >> 8) & 0xFF;
        u.s1 = r >> 16;
        if (epilogue || lane == 0) ptx::mbar_arrive(bar(UQEMPTY + qs));
        return u;
    };

    if (warp < 4) {
        // -------------------------------------------------------- epilogue
        const int quarter = warp;
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        constexpr int NB = (NMAX + 15) / 16;
        uint32_t j = 0;
        bool ok = true;
        for (uint32_t ui = 0; ok; ++ui) {
            const Unit un = take_unit(ui, true, ok);
            if (un.e < 0) break;
            const int bk = un.e & 1;
            const BankLists &L = args.lists[bk];
            const int goff = bank_offset(L, bk, args.P);
            const int mt = un.mt, p0 = un.p0, n = un.n;
            for (int n0 = 0; ok && n0 < n; n0 += NMAX, ++j) {
                const int nn = min(NMAX, n - n0);
                int rs[NB];
                float re[NB];
                load_meta<NB>(L, args, 0, 1, nn, p0 + n0, goff + p0 + n0, lane, rs, re);
                const int db = j % DB;
                if (!wait_warp<true>(bar(ACCREADY + db), (j / DB) & 1, abort_flag, args.status, args.wait_ns)) { ok = false; break; }
                ptx::tc_fence_after();
                epilogue_cols<PHASE, NB, C::kStack, C::kSplit, C::kRowQ>(args, tmem + lane_base + C::kDCol + db * C::kDW, 0, 1,
                                                                        nn, goff + p0 + n0, mt, quarter, lane, rs, re);
                ptx::tc_fence_before();
                ptx::mbar_arrive(bar(ACCFREE + db));
            }
        }
    } else if (warp == C::kProducer && lane == 0) {
        // ------------------------------------------------------------ producer
        // A launch over both banks prefers, in the first CTA that reaches each
        // SM, the cold bank's units (one host-link streamer per SM) and in the
        // others the hot bank's; each turns to the other bank's queue once
        // its own is empty.
        int pref = args.b;
        if (args.b < 0) {
            uint32_t smid;
            asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
            pref = atomicAdd(&args.claim[smid & 1023u], 1) == 0 ? MOE_BANK_COLD : MOE_BANK_HOT;
        }
        bool dry_pref = false, dry_other = args.b >= 0;
        uint32_t it = 0;
        RingPos pos;   // stage of iteration it
        bool ok = true, withheld = false;
        for (uint32_t ui = 0; ok; ++ui) {
            // take the next unit from the launch's work counter and publish it
            const int qs = ui % kQ;
            if (ui >= (uint32_t)kQ &&
                !wait_one<SUSP>(bar(UQEMPTY + qs), ((ui / kQ) - 1) & 1, abort_flag, args.status, args.wait_ns)) {
                ok = false;
                break;
            }
            int e = -1;
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
            if (e < 0) {
                uq[4 * qs] = -1;
                ptx::mbar_arrive(bar(UQFULL + qs));
                break;
            }
            const int bk = e & 1;
            const BankLists &L = args.lists[bk];
            const int goff = bank_offset(L, bk, args.P);
            int a, mt, s0, s1;
            unit_pos(e >> 1, part.tiles, ns, args.ks, a, mt, s0, s1);
            const int p0 = L.act_off[a], n = L.act_off[a + 1] - p0;
            uq[4 * qs + 0] = e;
            uq[4 * qs + 1] = n;
            uq[4 * qs + 2] = p0;
            uq[4 * qs + 3] = mt | (s0 << 8) | (s1 << 16);
            ptx::mbar_arrive(bar(UQFULL + qs));
            // a staged cold row is read from its pool slot (tmA2), not the host bank
            const int sslot = staged_slot(args, bk, a);
            const int row = sslot >= 0 ? sslot : L.act_row[a];
            const CUtensorMap *tmA = sslot >= 0 ? &tmA2 : (bk ? &tmA1 : &tmA0);
            const uint8_t *expert = (sslot >= 0 ? args.stage_pool : args.bank[bk]) + (int64_t)row * args.eb;
            for (int n0 = 0; ok && n0 < n; n0 += NMAX) {
                const int brow = goff + p0 + n0;
                for (int s = s0; s < s1; ++s, ++it, pos.next(S)) {
                    const int st = pos.st;
                    // the stage's previous round must have been consumed
                    if (it >= (uint32_t)S && !wait_one<SUSP>(bar(DONE + st), pos.ph ^ 1u, abort_flag, args.status, args.wait_ns)) {
                        ok = false;
                        break;
                    }
                    int slot, tidx, kb0, nkb;
                    part.group(mt, s, slot, tidx, kb0, nkb);
                    if (args.withhold && it == 0 && (e >> 1) == 0) {
                        // injected fault: this stage's copies are never issued, so
                        // the roles waiting for it time out
                        withheld = true;
                        continue;
                    }
                    // the code block counts its packed (global) bytes; the token-row
                    // box counts in full (a half group's second chunk is past the
                    // rows' end: zero fill, unused)
                    ptx::mbar_arrive_expect_tx(bar(FULL + st),
                                               (uint32_t)(kGroupQBytes + kSfAtomBytes + C::kBStage + C::kSfbStage));
                    ptx::tma_load_5d(ptx::smem_addr(sA + st * C::kAStage), tmA, 0, 0, slot, tidx, row, bar(FULL + st));
                    ptx::bulk_g2s(ptx::smem_addr(sSF + st * kSfAtomBytes), expert + part.group_off(slot, tidx) + kGroupQBytes,
                                  kSfAtomBytes, bar(FULL + st));
                    ptx::tma_load_4d(ptx::smem_addr(sB + st * C::kBStage), &tmB, 0, brow, 0, 2 * s, bar(FULL + st));
                    if (MX) {   // the tile's block scales of this group
                        const int64_t tile = args.tile_off[bk][a] + n0 / NMAX;
                        ptx::bulk_g2s(ptx::smem_addr(sSFB + st * C::kSfbStage),
                                      args.sfb[bk] + (tile * args.sf_groups + s) * kSfbGroupBytes, kSfbGroupBytes,
                                      bar(FULL + st));
                    }
                }
            }
        }
        if (!ok) {
            // let the copies this thread issued land before the CTA goes away
            const uint32_t first = it > (uint32_t)S ? it - S : 0u;
            for (uint32_t i = first; i < it; ++i) {
                if (withheld && i == 0) continue;   // nothing was issued for it
                for (uint32_t t = 0; t < kWaitLimit; ++t)
                    if (ptx::mbar_try_wait(bar(FULL + i % S), (i / S) & 1)) break;
            }
        }
    } else if (warp == C::kMmaWarp) {
        // ----------------------------------------------------------- MMA issue
        // The whole warp runs the loop (holding the unit's values uniformly);
        // one elected lane issues the tensor-core instructions.  Once a
        // stage has landed, that lane keeps issuing the following groups
        // whose stages have landed too (a non-blocking check each), so the
        // per-group handshakes of the warp are paid once per burst.
        uint32_t it = 0, j = 0;
        RingPos pos;   // stage of iteration it
        bool ok = true;
        for (uint32_t ui = 0; ok; ++ui) {
            const Unit un = take_unit(ui, false, ok);
            if (un.e < 0) break;
            const int mt = un.mt, s0 = un.s0, s1 = un.s1, n = un.n;
            for (int n0 = 0; ok && n0 < n; n0 += NMAX, ++j) {
                const int nn = min(NMAX, n - n0);
                const int Nr = (nn + C::kRowQ - 1) / C::kRowQ * C::kRowQ;
                const int Nm = C::kStack ? 2 * Nr : Nr;   // B rows of one MMA
                const uint32_t idesc0 = ptx::idesc_mx_e2m1_e4m3(128, Nm, 0, 0);   // | (K block << 29): A scale byte
                const int db = j % DB;
                if (j >= (uint32_t)DB &&
                    !wait_warp<SUSP>(bar(ACCFREE + db), ((j / DB) - 1) & 1, abort_flag, args.status, args.wait_ns)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem + C::kDCol + db * C::kDW;
                for (int s = s0; s < s1;) {
                    if (!wait_warp<SUSP>(bar(FULL + pos.st), pos.ph, abort_flag, args.status, args.wait_ns)) { ok = false; break; }
                    ptx::tc_fence_after();
                    int issued = 0;
                    if (ptx::elect_one()) {
                        RingPos p = pos;
                        for (int ss = s;;) {
                            const int st = p.st;
                            int slot, tidx, kb0, nkb;
                            part.group(mt, ss, slot, tidx, kb0, nkb);
                            // the group's scales -> the stage's own slot
                            const uint32_t sfa = tmem + 32u * st;
                            ptx::tmem_cp_32x128b_warpx4(
                                sfa, ptx::smem_desc_noswizzle(ptx::smem_addr(sSF + st * kSfAtomBytes), 128, 128));
                            if (MX) {   // token blocks 0-3 and (tiles past 128 rows) 4-7 of the tile's block scales
                                const uint32_t sb = ptx::smem_addr(sSFB + st * C::kSfbStage);
                                ptx::tmem_cp_32x128b_warpx4(sfa + C::kSfbCol, ptx::smem_desc_noswizzle(sb, 128, 128));
                                if (Nm > 128)
                                    ptx::tmem_cp_32x128b_warpx4(sfa + C::kSfbCol + 4,
                                                                ptx::smem_desc_noswizzle(sb + 512, 128, 128));
                            }
                            const uint32_t a_addr = ptx::smem_addr(sA + st * C::kAStage);
                            for (int i = 0; i < nkb; ++i) {
                                const int kb = kb0 + i;   // K block of the group (A bytes kb*32.., scale byte kb)
                                const uint64_t ad = ptx::smem_desc_sw128(a_addr + kb * 32);
                                // this tile's chunk i/2 of the group, its K block i%2
                                const uint32_t b_addr =
                                    ptx::smem_addr(sB + st * C::kBStage + (i >> 1) * C::kBChunk) + (i & 1) * 32;
#pragma unroll
                                for (int pc = 0; pc < (C::kStack ? 1 : C::kPieces); ++pc) {   // e4m3 piece of B
                                    const uint64_t bd = ptx::smem_desc_sw64(b_addr + pc * NMAX * 64);
                                    if (MX)   // B's scale: byte i (the token rows' K block) of the slot's own columns
                                        ptx::mma_mxf8f6f4_ss(d_tmem, ad, bd, idesc0 | ((uint32_t)kb << 29) | ((uint32_t)i << 4),
                                                             sfa, sfa + C::kSfbCol, (ss != s0) | i);
                                    else
                                        ptx::mma_mxf8f6f4_ss(d_tmem, ad, bd, idesc0 | ((uint32_t)kb << 29), sfa,
                                                             tmem + C::kSfbCol + pc * C::kSfbStride, (ss != s0) | i | pc);
                                }
                            }
                            ptx::mma_commit(bar(DONE + st));
                            ++issued;
                            ++ss;
                            p.next(S);
                            if (ss >= s1 || !ptx::mbar_test_wait(bar(FULL + p.st), p.ph)) break;
                            ptx::tc_fence_after();
                        }
                    }
                    issued = __reduce_max_sync(0xffffffffu, issued);
                    s += issued;
                    it += issued;
                    for (int k = 0; k < issued; ++k) pos.next(S);
                }
                if (!ok) break;
                if (ptx::elect_one()) ptx::mma_commit(bar(ACCREADY + db));
                __syncwarp();
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
    if (warp == C::kMmaWarp) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, C::kCols);
    }
}

#include "ffn_tc_decode.cuh"

constexpr int kKeep = 4;   // 16-byte (x) or 8-value (h) columns a prep thread keeps in registers

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
// the two pieces of that chunk's 128-byte record.  PERM: in the order
// 0,2,4,6,1,3,5,7 -- the K order in which the decode-tile kernel spreads an
// expert's codes into tensor memory.
template <bool PERM>
__device__ __forceinline__ void store_pieces(uint8_t *row, int i, const float (&v)[8]) {
    uint2 q1, q2;
    if (PERM) {
        const float w[8] = {v[0], v[2], v[4], v[6], v[1], v[3], v[5], v[7]};
        split_e4m3x8(w, q1, q2);
    } else {
        split_e4m3x8(v, q1, q2);
    }
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
// b0 >= 0: that bank; b0 < 0: both banks, bank = blockIdx.y.  PERM: decode
// tiles' K order (see store_pieces).
constexpr int kPrepWarps = 8;    // picks per prep_x block (one warp each) on large steps; 1 on small ones
constexpr int kLaneCols = 16;    // 16-byte columns of a row a lane keeps (H <= 4096)

// Gather one pick's token row, scale it by the power of two that puts its
// largest |value| in (224, 448], split it into the two e4m3 pieces: one warp
// per pick, the row in the lanes' registers, the maximum a warp reduction.
// Blocks of blockDim.x / 32 picks (a small step spreads its picks over more
// blocks).
template <bool PERM>
__global__ void __launch_bounds__(32 * kPrepWarps) prep_x_kernel(const uint16_t *__restrict__ x, int H, int k,
                                                                BankLists L0, BankLists L1, int b0, int P,
                                                                uint8_t *__restrict__ xq, int32_t *__restrict__ xgexp,
                                                                int32_t *sched, int32_t *claim,
                                                                float *__restrict__ gu32, int I) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int p = blockIdx.x * (int)(blockDim.x >> 5) + warp, b = b0 >= 0 ? b0 : (int)blockIdx.y;
    const BankLists &L = b ? L1 : L0;
    if (blockIdx.x == 0 && blockIdx.y == 0) {
        // reset the work counters (and both GEMMs' SM claims) of this call's launches,
        // stream-ordered before them; a one-bank call leaves the other bank's alone
        if (threadIdx.x < 4 && (b0 < 0 || (int)threadIdx.x / 2 == b0)) sched[threadIdx.x] = 0;
        if (claim)
            for (int i = threadIdx.x; i < 2 * 1024; i += blockDim.x) claim[i] = 0;
    }
    if (p >= L.hdr[kHdrNPicks + b]) return;   // warp-uniform
    const int g = bank_offset(L, b, P) + p;
    const int t = L.picks[p] / k;
    const uint4 *row = (const uint4 *)(x + (int64_t)t * H);
    const int n8 = H / 8;
    // a row of up to kLaneCols 16-byte columns per lane is read once and kept
    // for the conversion; a wider one is read twice
    const bool keep = n8 <= 32 * kLaneCols;
    uint4 kv[kLaneCols];
    float mx = 0.0f;
    auto row_max = [&](const uint4 v) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q)
            mx = fmaxf(mx, fmaxf(fabsf(__uint_as_float(w[q] << 16)), fabsf(__uint_as_float(w[q] & 0xFFFF0000u))));
    };
    if (keep) {
#pragma unroll
        for (int c = 0; c < kLaneCols; ++c) {
            const int i = lane + 32 * c;
            kv[c] = i < n8 ? row[i] : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int c = 0; c < kLaneCols; ++c) row_max(kv[c]);   // zero columns past the row change no maximum
    } else {
        for (int i = lane; i < n8; i += 32) row_max(row[i]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const int e = row_exponent(mx);
    uint8_t *dst = xq + (int64_t)g * H * 2;
    auto convert = [&](const uint4 v, int i) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        float f[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            f[2 * q] = ldexpf(__uint_as_float(w[q] << 16), -e);
            f[2 * q + 1] = ldexpf(__uint_as_float(w[q] & 0xFFFF0000u), -e);
        }
        store_pieces<PERM>(dst, i, f);
    };
    if (keep) {
#pragma unroll
        for (int c = 0; c < kLaneCols; ++c) {
            const int i = lane + 32 * c;
            if (i < n8) convert(kv[c], i);
        }
    } else {
        for (int i = lane; i < n8; i += 32) convert(row[i], i);
    }
    if (lane == 0) xgexp[g] = e;
    if (gu32) {   // split units: clear this pick's gate/up sums before the gate/up GEMM adds into them
        float4 *z = (float4 *)(gu32 + (int64_t)g * 2 * I);
        for (int i = lane; i < I / 2; i += 32) z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
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
template <bool PERM>
__global__ void __launch_bounds__(256) prep_h_kernel(BankLists L0, BankLists L1, int b0, int P, int I,
                                                     const float *__restrict__ h32, const float *__restrict__ gu32,
                                                     uint8_t *__restrict__ hq, int32_t *__restrict__ hexp,
                                                     float *__restrict__ y32, int H) {
    __shared__ float red[8];
    const int p = blockIdx.x, b = b0 >= 0 ? b0 : (int)blockIdx.y;
    const BankLists &L = b ? L1 : L0;
    // Launched as a programmatic dependent of the gate/up GEMM: wait for its
    // sums, and let the down GEMM launch at once (it streams weights, and
    // waits for these rows before it reads them).
    ptx::gdc_wait();
    ptx::gdc_launch_dependents();
    if (p >= L.hdr[kHdrNPicks + b]) return;
    const int g = bank_offset(L, b, P) + p;
    const int n8 = I / 8;
    // a row of up to kKeep 8-value columns per thread (I <= 8192) is read once
    // and kept in registers for the conversion; a wider one is read twice
    const bool keep = n8 <= kKeep * (int)blockDim.x;
    float kf[kKeep][8];
    float mx = 0.0f;
    if (keep) {
#pragma unroll
        for (int c = 0; c < kKeep; ++c) {
            const int i = threadIdx.x + c * blockDim.x;
            if (i < n8) {
                h_values(h32, gu32, g, I, i, kf[c]);
#pragma unroll
                for (int q = 0; q < 8; ++q) mx = fmaxf(mx, fabsf(kf[c][q]));
            }
        }
    } else {
        for (int i = threadIdx.x; i < n8; i += blockDim.x) {
            float f[8];
            h_values(h32, gu32, g, I, i, f);
#pragma unroll
            for (int q = 0; q < 8; ++q) mx = fmaxf(mx, fabsf(f[q]));
        }
    }
    const int e = row_exponent(block_max(mx, red));
    uint8_t *dst = hq + (int64_t)g * I * 2;
    if (keep) {
#pragma unroll
        for (int c = 0; c < kKeep; ++c) {
            const int i = threadIdx.x + c * blockDim.x;
            if (i < n8) {
                float f[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) f[q] = ldexpf(kf[c][q], -e);
                store_pieces<PERM>(dst, i, f);
            }
        }
    } else {
        for (int i = threadIdx.x; i < n8; i += blockDim.x) {
            float f[8];
            h_values(h32, gu32, g, I, i, f);
#pragma unroll
            for (int q = 0; q < 8; ++q) f[q] = ldexpf(f[q], -e);
            store_pieces<PERM>(dst, i, f);
        }
    }
    if (threadIdx.x == 0) hexp[g] = e;
    if (y32) {
        float4 *z = (float4 *)(y32 + (int64_t)L.picks[p] * H);
        for (int i = threadIdx.x; i < H / 4; i += blockDim.x) z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

constexpr int kHLaneCols = 12;   // 8-value columns of an h row a lane keeps (I <= 3072)

// prep_h for prefill-sized steps: one warp per pick, the row in the lanes'
// registers, the maximum a warp reduction; the same values and rounding as
// prep_h_kernel.
template <bool PERM>
__global__ void __launch_bounds__(32 * kPrepWarps) prep_h_warp_kernel(BankLists L0, BankLists L1, int b0, int P, int I,
                                                                     const float *__restrict__ h32,
                                                                     const float *__restrict__ gu32,
                                                                     uint8_t *__restrict__ hq,
                                                                     int32_t *__restrict__ hexp,
                                                                     float *__restrict__ y32, int H) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int p = blockIdx.x * (int)(blockDim.x >> 5) + warp, b = b0 >= 0 ? b0 : (int)blockIdx.y;
    const BankLists &L = b ? L1 : L0;
    if (p >= L.hdr[kHdrNPicks + b]) return;   // warp-uniform
    const int g = bank_offset(L, b, P) + p;
    const int n8 = I / 8;
    const bool keep = n8 <= 32 * kHLaneCols;
    float kf[kHLaneCols][8];
    float mx = 0.0f;
    if (keep) {
#pragma unroll
        for (int c = 0; c < kHLaneCols; ++c) {
            const int i = lane + 32 * c;
            if (i < n8) {
                h_values(h32, gu32, g, I, i, kf[c]);
#pragma unroll
                for (int q = 0; q < 8; ++q) mx = fmaxf(mx, fabsf(kf[c][q]));
            }
        }
    } else {
        for (int i = lane; i < n8; i += 32) {
            float f[8];
            h_values(h32, gu32, g, I, i, f);
#pragma unroll
            for (int q = 0; q < 8; ++q) mx = fmaxf(mx, fabsf(f[q]));
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const int e = row_exponent(mx);
    uint8_t *dst = hq + (int64_t)g * I * 2;
    if (keep) {
#pragma unroll
        for (int c = 0; c < kHLaneCols; ++c) {
            const int i = lane + 32 * c;
            if (i < n8) {
                float f[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) f[q] = ldexpf(kf[c][q], -e);
                store_pieces<PERM>(dst, i, f);
            }
        }
    } else {
        for (int i = lane; i < n8; i += 32) {
            float f[8];
            h_values(h32, gu32, g, I, i, f);
#pragma unroll
            for (int q = 0; q < 8; ++q) f[q] = ldexpf(f[q], -e);
            store_pieces<PERM>(dst, i, f);
        }
    }
    if (lane == 0) hexp[g] = e;
    if (y32) {
        float4 *z = (float4 *)(y32 + (int64_t)L.picks[p] * H);
        for (int i = lane; i < H / 4; i += 32) z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
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

// ---------------------------------------------------------------------------
// MXFP8 rows for prefill tiles (moe_set_act_format(MOE_ACT_MXFP8))
// ---------------------------------------------------------------------------

// The first prefill tile of each active row, per bank: tile_off[b][a] =
// sum over a' < a of ceil(n_a' / kPrefillTileMx); tile_off[b][n_act] = the bank's tiles.
// One warp per bank.
__global__ void __launch_bounds__(64) tile_scan_kernel(BankLists L0, BankLists L1, int b0, int P, int32_t *tile_off) {
    const int b = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (b0 >= 0 && b != b0) return;
    const BankLists &L = b ? L1 : L0;
    const int na = L.hdr[kHdrNAct + b];
    int32_t *to = tile_off + (size_t)b * (P + 1);
    int run = 0;
    for (int base = 0; base < na; base += 32) {
        const int a = base + lane;
        const int n = a < na ? L.act_off[a + 1] - L.act_off[a] : 0;
        const int t = (n + kPrefillTileMx - 1) / kPrefillTileMx;
        int incl = t;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += v;
        }
        if (a < na) to[a] = run + incl - t;
        run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) to[na] = run;
}

// Values 8i..8i+7 of a row -> MXFP8: the 32-element block of these values
// lies in lanes 4j..4j+3 of the warp (all 32 lanes call this together); the
// block's exponent e makes its largest |value| fit 448 (the same rule as a
// row's exponent, held to the e8m0 range), and each value becomes
// e4m3(v 2^-e), rounded to nearest even.  Returns the 8 bytes and the
// block's e.
__device__ __forceinline__ uint2 mx8_values(const float (&v)[8], int &e) {
    float mx = 0.0f;
#pragma unroll
    for (int q = 0; q < 8; ++q) mx = fmaxf(mx, fabsf(v[q]));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    e = min(127, max(-127, row_exponent(mx)));   // an e8m0 scale spans 2^-127 .. 2^127
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
        w[q] = __nv_cvt_float2_to_fp8x2(make_float2(ldexpf(v[2 * q], -e), ldexpf(v[2 * q + 1], -e)), __NV_SATFINITE,
                                        __NV_E4M3);
    return make_uint2(w[0] | (w[1] << 16), w[2] | (w[3] << 16));
}

// Where pick p of bank b sits among the prefill tiles: its active row a (the
// largest a with act_off[a] <= p), its tile and its row in the tile.
__device__ __forceinline__ void pick_tile(const BankLists &L, int b, int p, const int32_t *tile_off, int P, int &tile,
                                          int &r) {
    int lo = 0, hi = L.hdr[kHdrNAct + b] - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (L.act_off[mid] <= p) lo = mid;
        else hi = mid - 1;
    }
    const int q = p - L.act_off[lo];
    tile = tile_off[(size_t)b * (P + 1) + lo] + q / kPrefillTileMx;
    r = q % kPrefillTileMx;
}

// Byte of a tile's block-scale slab holding token row r's scale for K block
// kblk of the row (group kblk / 4, block kblk % 4).
__device__ __forceinline__ int sfb_byte(int r, int kblk) {
    const int j = r >> 5, l = r & 31;
    return (kblk >> 2) * kSfbGroupBytes + (j >> 2) * 512 + l * 16 + (j & 3) * 4 + (kblk & 3);
}

// One row of K values (8 per thread per pass; n8 = K / 8, a multiple of 4)
// to its MXFP8 bytes (dst, K bytes, logical order) and its block scales in
// the tile's slab.
template <class Load8>
__device__ __forceinline__ void mx8_row(int n8, Load8 load8, uint8_t *__restrict__ dst, uint8_t *__restrict__ slab,
                                        int r) {
    // one warp per row: every lane takes part in each pass (warp shuffles)
    const int lane = threadIdx.x & 31;
    for (int i0 = 0; i0 < n8; i0 += 32) {
        const int i = i0 + lane;
        float v[8];
        if (i < n8) {
            load8(i, v);
        } else {
#pragma unroll
            for (int q = 0; q < 8; ++q) v[q] = 0.0f;
        }
        int e;
        const uint2 q8 = mx8_values(v, e);
        if (i < n8) {
            *(uint2 *)(dst + (int64_t)i * 8) = q8;
            if ((i & 3) == 0) slab[sfb_byte(r, i >> 2)] = (uint8_t)(127 + e);
        }
    }
}

// One warp per pick, blockDim.x / 32 picks per block.
__global__ void __launch_bounds__(256) prep_x_mx8_kernel(const uint16_t *__restrict__ x, int H, int k, BankLists L0,
                                                         BankLists L1, int b0, int P, uint8_t *__restrict__ xq,
                                                         int32_t *__restrict__ xgexp, int32_t *sched, int32_t *claim,
                                                         const int32_t *__restrict__ tile_off, uint8_t *__restrict__ sfx,
                                                         int max_tiles) {
    const int p = blockIdx.x * (int)(blockDim.x >> 5) + (int)(threadIdx.x >> 5), b = b0 >= 0 ? b0 : (int)blockIdx.y;
    const BankLists &L = b ? L1 : L0;
    if (blockIdx.x == 0 && blockIdx.y == 0) {
        if (threadIdx.x < 4 && (b0 < 0 || (int)threadIdx.x / 2 == b0)) sched[threadIdx.x] = 0;
        if (claim)
            for (int i = threadIdx.x; i < 2 * 1024; i += blockDim.x) claim[i] = 0;
    }
    if (p >= L.hdr[kHdrNPicks + b]) return;
    const int g = bank_offset(L, b, P) + p;
    int tile, r;
    pick_tile(L, b, p, tile_off, P, tile, r);
    const int groups = H / kKG;
    uint8_t *slab = sfx + ((int64_t)b * max_tiles + tile) * groups * kSfbGroupBytes;
    const uint4 *row = (const uint4 *)(x + (int64_t)(L.picks[p] / k) * H);
    mx8_row(H / 8, [&](int i, float (&v)[8]) {
        const uint4 u = row[i];
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            v[2 * q] = __uint_as_float(w[q] << 16);
            v[2 * q + 1] = __uint_as_float(w[q] & 0xFFFF0000u);
        }
    }, xq + (int64_t)g * H, slab, r);
    if ((threadIdx.x & 31) == 0) xgexp[g] = 0;   // the block scales carry the magnitudes
}

__global__ void __launch_bounds__(256) prep_h_mx8_kernel(BankLists L0, BankLists L1, int b0, int P, int I,
                                                         const float *__restrict__ h32, uint8_t *__restrict__ hq,
                                                         int32_t *__restrict__ hexp, const int32_t *__restrict__ tile_off,
                                                         uint8_t *__restrict__ sfh, int max_tiles) {
    // one warp per pick, blockDim.x / 32 picks per block
    const int p = blockIdx.x * (int)(blockDim.x >> 5) + (int)(threadIdx.x >> 5), b = b0 >= 0 ? b0 : (int)blockIdx.y;
    const BankLists &L = b ? L1 : L0;
    if (p >= L.hdr[kHdrNPicks + b]) return;
    const int g = bank_offset(L, b, P) + p;
    int tile, r;
    pick_tile(L, b, p, tile_off, P, tile, r);
    const int groups = (I + kKG - 1) / kKG;
    uint8_t *slab = sfh + ((int64_t)b * max_tiles + tile) * groups * kSfbGroupBytes;
    const float4 *row = (const float4 *)(h32 + (int64_t)g * I);
    mx8_row(I / 8, [&](int i, float (&v)[8]) {
        const float4 a = row[2 * i], c = row[2 * i + 1];
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = c.x; v[5] = c.y; v[6] = c.z; v[7] = c.w;
    }, hq + (int64_t)g * I, slab, r);
    if ((threadIdx.x & 31) == 0) hexp[g] = 0;
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

// Tensor map over the [rows][K/64][pieces][64 B] records of K-element rows
// (two e4m3 pieces, or one in the MXFP8 format), viewed as (byte, row,
// piece, chunk): a box of box_rows rows x every piece x two chunks lands as
// [chunk][piece][row][64 B], 64-byte swizzle, zero fill past the last row or
// chunk.
int make_piece_map(CUtensorMap *map, const void *base, int K, int rows, int box_rows, int pieces = 2) {
    auto enc = tensor_map_encoder();
    if (!enc) return set_error(MOE_ECUDA, "cuTensorMapEncodeTiled unavailable");
    cuuint64_t dims[4] = {64, (cuuint64_t)rows, (cuuint64_t)pieces, (cuuint64_t)K / 64};
    cuuint64_t strides[3] = {(cuuint64_t)K * pieces, 64, (cuuint64_t)64 * pieces};
    cuuint32_t box[4] = {64u, (cuuint32_t)box_rows, (cuuint32_t)pieces, 2};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return set_error(MOE_ECUDA, "cuTensorMapEncodeTiled failed: " + std::to_string((int)r));
    return MOE_OK;
}

template <int NMAX, int PHASE, int BANKS, bool MX>
int launch_one(const CUtensorMap &mB, const CUtensorMap &mA0, const CUtensorMap &mA1, const CUtensorMap &mA2,
               const TcArgs &args, int blocks, cudaStream_t s) {
    using C = TcCfg<NMAX, MX>;
    auto kern = ffn_tc_kernel<NMAX, PHASE, BANKS, MX>;
    const size_t smem = C::kSmem;
    MOE_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    if (blocks < 1) return MOE_OK;
    kern<<<blocks, C::kThreads, smem, s>>>(mB, mA0, mA1, mA2, args);
    MOE_LAUNCH_CHECK();
    return MOE_OK;
}

// Grid of one prefill GEMM launch: one CTA per SM (32 SMs' worth for a cold
// bank when the layer has both banks, so the two banks' launches run side by
// side).
int prefill_blocks(const moe_ctx *ctx, int b, bool shared, int units_max) {
    const int cold_ctas = 32;
    int blocks;
    if (b < 0 || !shared) blocks = ctx->sms;
    else blocks = b == MOE_BANK_COLD ? cold_ctas : ctx->sms - cold_ctas;
    return std::max(1, std::min(units_max, blocks));
}

template <int NMAX, int PHASE, bool MX>
int launch_gemm(const CUtensorMap &mB, const CUtensorMap &mA0, const CUtensorMap &mA1, const CUtensorMap &mA2,
                const TcArgs &a, int blocks, cudaStream_t s) {
    if (a.b < 0) return launch_one<NMAX, PHASE, 2, MX>(mB, mA0, mA1, mA2, a, blocks, s);
    if (a.b == MOE_BANK_COLD) return launch_one<NMAX, PHASE, 1, MX>(mB, mA0, mA1, mA2, a, blocks, s);
    return launch_one<NMAX, PHASE, 0, MX>(mB, mA0, mA1, mA2, a, blocks, s);
}

template <int NMAX, bool MX>
int launch_bank(moe_ctx *ctx, const Layer &layer, bool shared, TcArgs a1, TcArgs a2, int units1, int units2,
                const uint16_t *x, const WsLayout &lay, uint8_t *ws, cudaStream_t s) {
    const Geom &g = ctx->g;
    const int P = a1.P;
    a1.ks = std::min(TcCfg<NMAX, MX>::kSplit, a1.part.steps());
    a2.ks = std::min(TcCfg<NMAX, MX>::kSplit, a2.part.steps());
    const int blocks1 = prefill_blocks(ctx, a1.b, shared, units1), blocks2 = prefill_blocks(ctx, a1.b, shared, units2);
    const dim3 grid_p(P, a1.b < 0 ? 2 : 1);   // one block per pick (of each bank)
    const int xw = P >= 4096 ? kPrepWarps : 1;   // picks per prep_x block
    const dim3 grid_x((P + xw - 1) / xw, a1.b < 0 ? 2 : 1);
    const int pieces = MX ? 1 : 2;
    CUtensorMap m1, m2;
    if (int r = make_piece_map(&m1, ws + lay.xq, g.H, P, NMAX, pieces)) return r;
    if (int r = make_piece_map(&m2, ws + lay.hq, g.I, P, NMAX, pieces)) return r;
    if (MX) {
        int32_t *tile_off = (int32_t *)(ws + lay.tile_off);
        const int gx = g.H / kKG, gh = (g.I + kKG - 1) / kKG;
        for (int bk = 0; bk < 2; ++bk) {
            a1.tile_off[bk] = a2.tile_off[bk] = tile_off + (size_t)bk * (P + 1);
            a1.sfb[bk] = ws + lay.sfx + (size_t)bk * lay.max_tiles * gx * kSfbGroupBytes;
            a2.sfb[bk] = ws + lay.sfh + (size_t)bk * lay.max_tiles * gh * kSfbGroupBytes;
        }
        a1.sf_groups = gx;
        a2.sf_groups = gh;
        tile_scan_kernel<<<1, 64, 0, s>>>(a1.lists[0], a1.lists[1], a1.b, P, tile_off);
        MOE_LAUNCH_CHECK();
        prep_x_mx8_kernel<<<grid_x, 32 * xw, 0, s>>>(x, g.H, g.k, a1.lists[0], a1.lists[1], a1.b, P, ws + lay.xq,
                                                 (int32_t *)(ws + lay.xgexp), a1.sched, a1.claim, tile_off, ws + lay.sfx,
                                                 lay.max_tiles);
    } else {
        prep_x_kernel<false><<<grid_x, 32 * xw, 0, s>>>(x, g.H, g.k, a1.lists[0], a1.lists[1], a1.b, P, ws + lay.xq,
                                                    (int32_t *)(ws + lay.xgexp), a1.sched, a1.claim, a1.gu_out, g.I);
    }
    MOE_LAUNCH_CHECK();
    // the staging pool's maps stand in for units read from it (the cold maps
    // where no pool exists: then no unit reads them)
    const CUtensorMap &sm1 = ctx->stage_pool ? ctx->stage_map[0] : layer.wmap[1][0];
    const CUtensorMap &sm2 = ctx->stage_pool ? ctx->stage_map[1] : layer.wmap[1][1];
    if (int r = launch_gemm<NMAX, 1, MX>(m1, layer.wmap[0][0], layer.wmap[1][0], sm1, a1, blocks1, s)) return r;
    if (MX) {
        prep_h_mx8_kernel<<<grid_x, 32 * xw, 0, s>>>(a1.lists[0], a1.lists[1], a1.b, P, g.I, (const float *)(ws + lay.h32),
                                                 ws + lay.hq, (int32_t *)(ws + lay.hexp),
                                                 (const int32_t *)(ws + lay.tile_off), ws + lay.sfh, lay.max_tiles);
    } else {
        prep_h_warp_kernel<false><<<grid_x, 32 * xw, 0, s>>>(a1.lists[0], a1.lists[1], a1.b, P, g.I,
                                                    (const float *)(ws + lay.h32), a1.gu_out, ws + lay.hq,
                                                    (int32_t *)(ws + lay.hexp), a2.y_out, g.H);
    }
    MOE_LAUNCH_CHECK();
    if (int r = launch_gemm<NMAX, 2, MX>(m2, layer.wmap[0][1], layer.wmap[1][1], sm2, a2, blocks2, s)) return r;
    if (!a2.y_out) return MOE_OK;
    round_y_kernel<<<grid_p, 256, 0, s>>>(a2.lists[0], a2.lists[1], a2.b, g.H, a2.y_out, a2.Y);
    MOE_LAUNCH_CHECK();
    return MOE_OK;
}

// Launch `kern` on `s` as a programmatic dependent of the kernel before it:
// it may start once every block of that kernel has started or finished, and
// synchronizes with it through griddepcontrol.wait.
template <class T>
struct same_type {
    using type = T;
};

template <typename... KArgs>
cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                             typename same_type<KArgs>::type... args) {
    void *pargs[] = {(void *)&args...};   // each argument in the kernel's own parameter type
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, (const void *)kern, pargs);
}

template <int NMAX, int PHASE, int BANKS>
int launch_decode_one(const CUtensorMap &mB, const TcArgs &args, int blocks, bool dependent, cudaStream_t s) {
    using C = DecCfg<NMAX>;
    auto kern = ffn_tc_decode_kernel<NMAX, PHASE, BANKS>;
    MOE_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem));
    if (blocks < 1) return MOE_OK;
    if (PHASE == 2 && dependent) {
        // the down GEMM depends on prep_h programmatically: it claims units
        // and streams weights before prep_h's rows exist
        MOE_CUDA_TRY(launch_dependent(kern, dim3(blocks), dim3(C::kThreads), C::kSmem, s, mB, args));
    } else {
        kern<<<blocks, C::kThreads, C::kSmem, s>>>(mB, args);
    }
    MOE_LAUNCH_CHECK();
    return MOE_OK;
}

template <int NMAX, int PHASE>
int launch_decode_gemm(const CUtensorMap &mB, const TcArgs &a, int blocks, bool dependent, cudaStream_t s) {
    if (a.b < 0) return launch_decode_one<NMAX, PHASE, 2>(mB, a, blocks, dependent, s);
    if (a.b == MOE_BANK_COLD) return launch_decode_one<NMAX, PHASE, 1>(mB, a, blocks, dependent, s);
    return launch_decode_one<NMAX, PHASE, 0>(mB, a, blocks, dependent, s);
}

// Grid of a decode-tile GEMM launch: kPerSm CTAs per SM fill the SM; a
// cold-bank launch takes one per SM (the host link needs a few MB in flight
// GPU-wide) and, beside it, a hot-bank launch the SM's other slots, so the
// two banks' launches run side by side.
template <int NMAX>
int decode_blocks(const moe_ctx *ctx, int b, bool shared, int units_max) {
    const int per_sm = DecCfg<NMAX>::kPerSm;
    int blocks;
    if (b < 0 || (b == MOE_BANK_HOT && !shared)) blocks = ctx->sms * per_sm;
    else if (b == MOE_BANK_COLD) blocks = ctx->sms;
    else blocks = ctx->sms * (per_sm - 1);
    return std::max(1, std::min(units_max, blocks));
}

template <int NMAX>
int launch_bank_decode(moe_ctx *ctx, bool shared, bool cold_rows, TcArgs a1, TcArgs a2, int units1, int units2,
                       const uint16_t *x, const WsLayout &lay, uint8_t *ws, cudaStream_t s) {
    const Geom &g = ctx->g;
    const int P = a1.P;
    a1.ks = std::min(DecCfg<NMAX>::kSplit, a1.part.steps());
    a2.ks = std::min(DecCfg<NMAX>::kSplit, a2.part.steps());
    const dim3 grid_p(P, a1.b < 0 ? 2 : 1);   // one block per pick (of each bank)
    const int xw = P >= 4096 ? kPrepWarps : 1;   // picks per prep_x block
    const dim3 grid_x((P + xw - 1) / xw, a1.b < 0 ? 2 : 1);
    CUtensorMap m1, m2;
    if (int r = make_piece_map(&m1, ws + lay.xq, g.H, P, NMAX)) return r;
    if (int r = make_piece_map(&m2, ws + lay.hq, g.I, P, NMAX)) return r;
    prep_x_kernel<true><<<grid_x, 32 * xw, 0, s>>>(x, g.H, g.k, a1.lists[0], a1.lists[1], a1.b, P, ws + lay.xq,
                                               (int32_t *)(ws + lay.xgexp), a1.sched, a1.claim, a1.gu_out, g.I);
    MOE_LAUNCH_CHECK();
    if (int r = launch_decode_gemm<NMAX, 1>(m1, a1, decode_blocks<NMAX>(ctx, a1.b, shared, units1), false, s)) return r;
    // A call that streams the cold bank chains prep_h and the down GEMM to
    // the gate/up GEMM as programmatic dependents, so the host link restarts
    // before prep_h ends; an HBM-only call measured faster without.
    const bool dependent = a1.b != MOE_BANK_HOT && cold_rows;
    if (dependent) {
        MOE_CUDA_TRY(launch_dependent(prep_h_kernel<true>, grid_p, dim3(256), 0, s, a1.lists[0], a1.lists[1], a1.b, P,
                                      g.I, (const float *)(ws + lay.h32), (const float *)a1.gu_out, ws + lay.hq,
                                      (int32_t *)(ws + lay.hexp), a2.y_out, g.H));
    } else {
        prep_h_kernel<true><<<grid_p, 256, 0, s>>>(a1.lists[0], a1.lists[1], a1.b, P, g.I, (const float *)(ws + lay.h32),
                                                   a1.gu_out, ws + lay.hq, (int32_t *)(ws + lay.hexp), a2.y_out, g.H);
    }
    MOE_LAUNCH_CHECK();
    if (int r = launch_decode_gemm<NMAX, 2>(m2, a2, decode_blocks<NMAX>(ctx, a1.b, shared, units2), dependent, s)) return r;
    round_y_kernel<<<grid_p, 256, 0, s>>>(a2.lists[0], a2.lists[1], a2.b, g.H, a2.y_out, a2.Y);
    MOE_LAUNCH_CHECK();
    return MOE_OK;
}

}  // namespace

int make_weight_map(CUtensorMap *map, const uint8_t *bank, const Geom &g, const PartLayout &part, int rows) {
    auto enc = tensor_map_encoder();
    if (!enc) return set_error(MOE_ECUDA, "cuTensorMapEncodeTiled unavailable");
    // (code, row, slot, tile index, expert): 128 4-bit codes of a row, the
    // block's 128 rows of 64 bytes, the groups of a tile (or tile pair), the
    // tiles, the bank's experts
    cuuint64_t dims[5] = {(cuuint64_t)kKG, (cuuint64_t)kMT, (cuuint64_t)part.slots(), (cuuint64_t)part.tile_index_count(),
                          (cuuint64_t)rows};
    cuuint64_t strides[4] = {(cuuint64_t)kKG / 2, (cuuint64_t)kGroupBytes, (cuuint64_t)part.tile_stride, (cuuint64_t)g.eb};
    cuuint32_t box[5] = {(cuuint32_t)kKG, (cuuint32_t)kMT, 1, 1, 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 5, const_cast<uint8_t *>(bank + part.off), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return set_error(MOE_ECUDA, "cuTensorMapEncodeTiled (weights) failed: " + std::to_string((int)r));
    return MOE_OK;
}

int launch_ffn_tc(moe_ctx *ctx, const Layer &layer, int b, const uint16_t *x, int T, uint8_t *ws, uint16_t *Y,
                  cudaStream_t s) {
    const Geom &g = ctx->g;
    WsLayout lay = ws_layout(g, T);
    const int P = T * g.k;
    const bool shared = layer.n_hot > 0 && layer.n_cold > 0;

    TcArgs a1{};
    a1.bank[MOE_BANK_HOT] = layer.hot;
    a1.bank[MOE_BANK_COLD] = layer.cold_dev;
    for (int bk = 0; bk < 2; ++bk) {
        BankLists &L = a1.lists[bk];
        L.hdr = (const int32_t *)(ws + lay.hdr);
        L.act_row = (const int32_t *)(ws + lay.act_row) + (size_t)bk * P;
        L.act_off = (const int32_t *)(ws + lay.act_off) + (size_t)bk * (P + 1);
        L.picks = (const int32_t *)(ws + lay.picks) + (size_t)bk * P;
    }
    a1.eb = g.eb;
    a1.part = g.w13;
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
    a1.wait_ns = ctx->wait_ns;
    a1.withhold = ctx->inject_withhold ? 1 : 0;   // test hook, consumed by this call's gate/up GEMM
    ctx->inject_withhold = false;
    // Big-batch cold staging: a call that covers the cold bank copies the cold
    // rows with more picks than one token tile into the pool first (steps of
    // at most 16 tokens never route more picks to an expert than one tile).
    a1.stage_slot = nullptr;
    a1.stage_pool = nullptr;
    if (ctx->stage_slots > 0 && layer.n_cold > 0 && a1.b != MOE_BANK_HOT && T > 16) {
        int32_t *slot_of = (int32_t *)(ws + lay.stage_slot);
        if (int r = launch_cold_staging(ctx, layer, tile_width(T, ctx->act_format == MOE_ACT_MXFP8), a1.lists[1], slot_of,
                                        (int32_t *)(ws + lay.stage_src), s))
            return r;
        a1.stage_slot = slot_of;
        a1.stage_pool = ctx->stage_pool;
    }
    TcArgs a2 = a1;
    a2.withhold = 0;
    a2.claim = a1.claim ? a1.claim + 1024 : nullptr;   // the down GEMM's own claims
    a2.part = g.w2;
    a2.bexp = (const int32_t *)(ws + lay.hexp);
    a2.h_out = nullptr;
    a2.Y = Y;
    // narrow-tile steps: K parts per unit, summed in fp32 rows
    const bool split = split_k_steps(T);
    a1.gu_out = split ? (float *)(ws + lay.gu32) : nullptr;
    a1.y_out = nullptr;
    a2.gu_out = nullptr;
    a2.y_out = split ? (float *)(ws + lay.y32) : nullptr;

    const int units1 = 4 * P * g.mt13, units2 = 4 * P * g.mt2;   // bound: active rows never exceed the picks
    // The token-tile width depends only on T (and the activation format), so
    // an expert's arithmetic is the same in either bank.  Decode-sized steps
    // use narrow tiles (8, 16 or 32 tokens; an expert with more tokens loops
    // over token tiles) in the decode-tile kernel, which keeps more weight
    // bytes in flight per SM; prefill-sized steps use 144- or 160-wide tiles
    // (an 8192-token step's ~128 tokens per expert in one tile) in the
    // shared-memory-A kernel, one CTA per SM.
    const bool cold_rows = layer.n_cold > 0;
    if (T <= 8) return launch_bank_decode<8>(ctx, shared, cold_rows, a1, a2, units1, units2, x, lay, ws, s);
    if (T <= 16) return launch_bank_decode<16>(ctx, shared, cold_rows, a1, a2, units1, units2, x, lay, ws, s);
    if (T <= kNarrowMaxT) return launch_bank_decode<32>(ctx, shared, cold_rows, a1, a2, units1, units2, x, lay, ws, s);
    if (ctx->act_format == MOE_ACT_MXFP8)
        return launch_bank<kPrefillTileMx, true>(ctx, layer, shared, a1, a2, units1, units2, x, lay, ws, s);
    return launch_bank<kPrefillTile, false>(ctx, layer, shared, a1, a2, units1, units2, x, lay, ws, s);
}

}  // namespace moe
