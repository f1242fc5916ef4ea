// Decode-tile expert FFN with the weights spread into tensor memory by the
// tensor memory accelerator (included by ffn_tc.cu).
//
// The same tiles, units and arithmetic as ffn_tc_decode_kernel, but no SM
// instruction touches a weight byte:
//   producer  one thread: per K group, a tensor-TMA box of the padded 4-bit
//             type (the 8 KB code block lands as 16 KB of padded codes, 128-
//             byte swizzle), a bulk copy of its 512-byte scale atom, and the
//             tile's token rows (4-D box, [chunk][piece][row], 64-byte
//             swizzle); from HBM, the mapped pinned host bank, or the staging
//             pool.
//   MMA       one thread: per 64-wide chunk, tcgen05.cp of the scale atom into
//             a tensor-memory slot and two decompressing copies
//             (tcgen05.cp .128x256b .b8x16.b4x16_p64) of the chunk's K blocks
//             from the padded codes into the slot -- one code per byte in bits
//             5..2, K order kept -- then the MMAs with A from tensor memory.
//             A slot is handed back once its MMAs completed, the stage once
//             the group's copies and MMAs did (the MMAs read its token rows).
//   epilogue  four warps: the accumulator's rows, as in the other kernels.
// The K order is the logical one, so these tiles take token rows in logical
// order.  Bounded waits and teardown as in the other kernels.

template <int NMAX>
struct DecCpCfg {
    static constexpr bool kStack = NMAX <= 16;              // both e4m3 pieces as rows of one MMA
    static constexpr int kBChunk = 2 * NMAX * 64;           // one chunk's token rows: [piece][NMAX rows][64 B]
    static constexpr int kBStage = 2 * kBChunk;
    static constexpr int kRowQ = kStack ? NMAX : 16;
    static constexpr int kAStage = 2 * kGroupQBytes;        // padded code block: 16 KB
    static constexpr int kStageBytes = kAStage + kSfAtomBytes + kBStage;
    static constexpr int kPerSm = NMAX <= 16 ? 3 : 2;       // resident CTAs per SM
    static constexpr int kABufs = 3;                        // TMEM A slots, one chunk each
    static constexpr int kDW = (kStack ? 2 : 1) * NMAX;     // accumulator columns
    static constexpr int kNCol = (kDW + 31) / 32;           // B scale columns of one piece
    // Tensor memory: slot s owns the 32-column block at 32 s: its A scale
    // columns at +0 (four, one per lane quarter's rows), its codes (16
    // columns: two K blocks) at +16; blocks 0 and 1 also hold the B scale
    // columns of piece 0 and 1 at +8 (stacked tiles use block 0's for both).
    static constexpr uint32_t kSfaCol = 0, kSfbCol = 8, kACol = 16, kSfbStride = 32;
    static constexpr uint32_t kDCol = 32 * kABufs;
    static constexpr uint32_t kColsUsed = kDCol + kDW;
    static constexpr uint32_t kCols = kColsUsed <= 64 ? 64 : (kColsUsed <= 128 ? 128 : 256);
    static_assert(kCols * kPerSm <= 512 && kNCol <= 8, "tensor memory");
    static constexpr int kSplit = 2;                        // K halves per unit
    static constexpr int kProducer = 4, kMmaWarp = 5;
    static constexpr int kThreads = 192;
    static constexpr size_t kFixed = 2048;                  // alignment slack, barriers, queue
    // as many stages as the SM's shared memory holds for kPerSm CTAs
    static constexpr int kStages = (int)((228u * 1024u / kPerSm - 1024u - kFixed) / kStageBytes);
    static_assert(kStages >= 2 && kStages <= 8, "ring depth");
    static constexpr int kBars = 2 * kStages + 2 * kABufs + 2 + 2 * kQ;
    static constexpr size_t kSmem = 1024 + (size_t)kStages * kStageBytes + kBars * 8 + 16 + 4 * kQ;
    static_assert(kSmem <= kFixed + (size_t)kStages * kStageBytes, "fixed part");
};

template <int NMAX, int PHASE, int BANKS>
__global__ void __launch_bounds__(DecCpCfg<NMAX>::kThreads, DecCpCfg<NMAX>::kPerSm)
    ffn_tc_decode_cp_kernel(const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmA0,
                            const __grid_constant__ CUtensorMap tmA1, const __grid_constant__ CUtensorMap tmA2,
                            TcArgs args) {
    using C = DecCpCfg<NMAX>;
    constexpr int S = C::kStages, NA = C::kABufs;
    extern __shared__ uint8_t smem_raw[];
    // 128-byte-swizzled code blocks need 1024-byte alignment
    uint8_t *smem = smem_raw + ((1024u - (ptx::smem_addr(smem_raw) & 1023u)) & 1023u);
    uint8_t *sA = smem;                          // [S][16 KB] padded code blocks
    uint8_t *sB = sA + S * C::kAStage;           // [S][2 chunks][2 pieces][NMAX rows][64 B]
    uint8_t *sSF = sB + S * C::kBStage;          // [S][512] scale atoms
    uint64_t *bars = (uint64_t *)(sSF + S * kSfAtomBytes);
    uint32_t *holder = (uint32_t *)(bars + C::kBars);
    volatile int *abort_flag = (volatile int *)(holder + 1);
    volatile int *uq = (volatile int *)(holder + 2);
    auto bar = [&](int i) { return ptx::smem_addr(bars + i); };
    // FULL: group landed.  DONEG: the group's copies and MMAs completed
    // (stage free).  ADONE: an A slot's MMAs completed.
    const int FULL = 0, DONEG = S, ADONE = 2 * S, ACCREADY = 2 * S + NA, ACCFREE = ACCREADY + 1, UQFULL = ACCFREE + 1,
              UQEMPTY = UQFULL + kQ;
    constexpr int kQueueReaders = 128 + 1;
    constexpr bool SUSP = true;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (BANKS == 1) {
        // A cold-bank launch keeps one host-link streamer per SM.
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
            ptx::mbar_init(bar(DONEG + s), 1);
        }
        for (int i = 0; i < NA; ++i) ptx::mbar_init(bar(ADONE + i), 1);
        ptx::mbar_init(bar(ACCREADY), 1);
        ptx::mbar_init(bar(ACCFREE), 128);
        for (int q = 0; q < kQ; ++q) {
            ptx::mbar_init(bar(UQFULL + q), 1);
            ptx::mbar_init(bar(UQEMPTY + q), kQueueReaders);
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
    if (warp < 4) {
        // B scale columns, constant, in every lane quarter: 2^0; unstacked
        // tiles scale the second piece by 2^-4 here, stacked tiles in the
        // epilogue
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
    auto take_unit = [&](uint32_t ui, bool warp_wide, bool &ok) -> int {
        const int qs = ui % kQ;
        const bool w = warp_wide ? wait_warp<SUSP>(bar(UQFULL + qs), (ui / kQ) & 1, abort_flag, args.status, args.wait_ns)
                                 : wait_one<SUSP>(bar(UQFULL + qs), (ui / kQ) & 1, abort_flag, args.status, args.wait_ns);
        if (!w) {
            ok = false;
            return -1;
        }
        const int u = uq[qs];
        ptx::mbar_arrive(bar(UQEMPTY + qs));
        return u;
    };

    if (warp < 4) {
        // ---------------------------------------------------------- epilogue
        const int quarter = warp;
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        constexpr int NB = (NMAX + 15) / 16;
        uint32_t j = 0;
        bool ok = true;
        for (uint32_t ui = 0; ok; ++ui) {
            const int e = take_unit(ui, true, ok);
            if (e < 0) break;
            // the down GEMM reads prep_h's row exponents and adds into the rows
            // it cleared: wait for it (once)
            if (PHASE == 2 && ui == 0) ptx::gdc_wait();
            const int bk = e & 1;
            const BankLists &L = args.lists[bk];
            const int goff = bank_offset(L, bk, args.P);
            int a, mt, s0, s1;
            unit_pos(e >> 1, part.tiles, ns, args.ks, a, mt, s0, s1);
            const int p0 = L.act_off[a], n = L.act_off[a + 1] - p0;
            for (int n0 = 0; ok && n0 < n; n0 += NMAX, ++j) {
                const int nn = min(NMAX, n - n0);
                int rs[NB];
                float re[NB];
                load_meta<NB>(L, args, 0, 1, nn, p0 + n0, goff + p0 + n0, lane, rs, re);
                if (!wait_warp<SUSP>(bar(ACCREADY), j & 1, abort_flag, args.status, args.wait_ns)) { ok = false; break; }
                ptx::tc_fence_after();
                epilogue_cols<PHASE, NB, C::kStack, C::kSplit, C::kRowQ>(args, tmem + lane_base + C::kDCol, 0, 1, nn,
                                                                        goff + p0 + n0, mt, quarter, lane, rs, re);
                ptx::tc_fence_before();
                ptx::mbar_arrive(bar(ACCFREE));
            }
        }
    } else if (warp == C::kProducer && lane == 0) {
        // ------------------------------------------------------------ producer
        int pref = args.b;
        if (args.b < 0) {
            uint32_t smid;
            asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
            pref = atomicAdd(&args.claim[smid & 1023u], 1) == 0 ? MOE_BANK_COLD : MOE_BANK_HOT;
        }
        bool dry_pref = false, dry_other = args.b >= 0;
        uint32_t it = 0;
        bool ok = true, withheld = false;
        // The down GEMM's token rows are prep_h's output: the ring's first round
        // of weight copies goes out at once, its token-row boxes once prep_h
        // has finished (before any stage is reused, and at the end).
        bool rows_ready = PHASE == 1;
        int def_brow[S], def_s[S], ndef = 0;
        auto release_rows = [&]() {
            if (rows_ready) return;
            ptx::gdc_wait();
            rows_ready = true;
            for (int i = 0; i < ndef; ++i)
                ptx::tma_load_4d(ptx::smem_addr(sB + i * C::kBStage), &tmB, 0, def_brow[i], 0, 2 * def_s[i], bar(FULL + i));
        };
        for (uint32_t ui = 0; ok; ++ui) {
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
            uq[qs] = e;
            ptx::mbar_arrive(bar(UQFULL + qs));
            if (e < 0) break;
            const int bk = e & 1;
            const BankLists &L = args.lists[bk];
            const int goff = bank_offset(L, bk, args.P);
            int a, mt, s0, s1;
            unit_pos(e >> 1, part.tiles, ns, args.ks, a, mt, s0, s1);
            // a staged cold row is read from its pool slot (tmA2), not the host bank
            const int sslot = staged_slot(args, bk, a);
            const int row = sslot >= 0 ? sslot : L.act_row[a];
            const int p0 = L.act_off[a], n = L.act_off[a + 1] - p0;
            const CUtensorMap *tmA = sslot >= 0 ? &tmA2 : (bk ? &tmA1 : &tmA0);
            const uint8_t *expert = (sslot >= 0 ? args.stage_pool : args.bank[bk]) + (int64_t)row * args.eb;
            for (int n0 = 0; ok && n0 < n; n0 += NMAX) {
                const int brow = goff + p0 + n0;
                for (int s = s0; s < s1; ++s, ++it) {
                    const int st = it % S;
                    const uint32_t rnd = it / S;
                    if (rnd > 0) release_rows();
                    if (rnd > 0 &&
                        !wait_one<SUSP>(bar(DONEG + st), (rnd - 1) & 1, abort_flag, args.status, args.wait_ns)) {
                        ok = false;
                        break;
                    }
                    int slot, tidx, kb0, nkb;
                    part.group(mt, s, slot, tidx, kb0, nkb);
                    if (PHASE == 1 && args.withhold && it == 0 && (e >> 1) == 0) {
                        // injected fault: this stage's copies are never issued, so
                        // the roles waiting for it time out
                        withheld = true;
                        continue;
                    }
                    // the code block counts its packed (global) bytes; a half
                    // group's second token-row chunk is past the rows' end: zero
                    // fill, counted, unused
                    ptx::mbar_arrive_expect_tx(bar(FULL + st), (uint32_t)(kGroupQBytes + kSfAtomBytes + C::kBStage));
                    ptx::tma_load_5d(ptx::smem_addr(sA + st * C::kAStage), tmA, 0, 0, slot, tidx, row, bar(FULL + st));
                    ptx::bulk_g2s(ptx::smem_addr(sSF + st * kSfAtomBytes), expert + part.group_off(slot, tidx) + kGroupQBytes,
                                  kSfAtomBytes, bar(FULL + st));
                    if (rows_ready) {
                        ptx::tma_load_4d(ptx::smem_addr(sB + st * C::kBStage), &tmB, 0, brow, 0, 2 * s, bar(FULL + st));
                    } else {   // first round: stage st == ndef
                        def_brow[ndef] = brow;
                        def_s[ndef] = s;
                        ++ndef;
                    }
                }
            }
        }
        release_rows();
        if (!ok) {
            // let the copies this thread issued land before the CTA goes away
            const uint32_t first = it > (uint32_t)S ? it - S : 0u;
            for (uint32_t i = first; i < it; ++i) {
                if (withheld && i == 0) continue;   // nothing was issued for it
                for (uint32_t t = 0; t < kWaitLimit; ++t)
                    if (ptx::mbar_try_wait(bar(FULL + i % S), (i / S) & 1)) break;
            }
        }
    } else if (warp == C::kMmaWarp && lane == 0) {
        // ----------------------------------------------------------- MMA issue
        uint32_t it = 0, ci = 0, j = 0;
        bool ok = true, issued = false;
        for (uint32_t ui = 0; ok; ++ui) {
            const int e = take_unit(ui, false, ok);
            if (e < 0) break;
            const BankLists &L = args.lists[e & 1];
            int a, mt, s0, s1;
            unit_pos(e >> 1, part.tiles, ns, args.ks, a, mt, s0, s1);
            const int n = L.act_off[a + 1] - L.act_off[a];
            for (int n0 = 0; ok && n0 < n; n0 += NMAX, ++j) {
                const int nn = min(NMAX, n - n0);
                const int Nr = (nn + C::kRowQ - 1) / C::kRowQ * C::kRowQ;
                const int Nm = C::kStack ? 2 * Nr : Nr;   // B rows of one MMA
                const uint32_t idesc0 = ptx::idesc_mx_e2m1_e4m3(128, Nm, 0, 0);   // | (scale byte << 29)
                if (j >= 1u && !wait_one<SUSP>(bar(ACCFREE), (j - 1) & 1, abort_flag, args.status, args.wait_ns)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem + C::kDCol;
                for (int s = s0; ok && s < s1; ++s, ++it) {
                    const int st = it % S;
                    if (!wait_one<SUSP>(bar(FULL + st), (it / S) & 1, abort_flag, args.status, args.wait_ns)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    int slot, tidx, kb0, nkb;
                    part.group(mt, s, slot, tidx, kb0, nkb);
                    const int nch = nkb / 2;
                    // the chunks' slots must be free (their previous MMAs completed)
                    for (int ch = 0; ok && ch < nch; ++ch) {
                        const uint32_t c = ci + ch;
                        if (c >= (uint32_t)NA &&
                            !wait_one<SUSP>(bar(ADONE + c % NA), ((c / NA) - 1) & 1, abort_flag, args.status, args.wait_ns))
                            ok = false;
                    }
                    if (!ok) break;
                    // copies into the slots: the scale atom, and the chunk's two K
                    // blocks decompressed (padded 4-bit -> one code per byte)
                    const uint32_t a_addr = ptx::smem_addr(sA + st * C::kAStage);
                    const uint64_t sfd = ptx::smem_desc_noswizzle(ptx::smem_addr(sSF + st * kSfAtomBytes), 128, 128);
                    for (int ch = 0; ch < nch; ++ch) {
                        const uint32_t sb = tmem + 32u * ((ci + ch) % NA);
                        ptx::tmem_cp_32x128b_warpx4(sb + C::kSfaCol, sfd);
#pragma unroll
                        for (int kk = 0; kk < 2; ++kk)
                            ptx::tmem_cp_128x256b_unpack4(sb + C::kACol + 8 * kk,
                                                          ptx::smem_desc_sw128(a_addr + (kb0 + 2 * ch + kk) * 32));
                    }
                    issued = true;
                    for (int ch = 0; ch < nch; ++ch, ++ci) {
                        const uint32_t sb = tmem + 32u * (ci % NA);
                        const uint32_t b_addr = ptx::smem_addr(sB + st * C::kBStage + ch * C::kBChunk);
#pragma unroll
                        for (int kk = 0; kk < 2; ++kk) {
                            const uint32_t idesc = idesc0 | ((uint32_t)(kb0 + 2 * ch + kk) << 29);
#pragma unroll
                            for (int pc = 0; pc < (C::kStack ? 1 : 2); ++pc) {
                                const uint64_t bd = ptx::smem_desc_sw64(b_addr + pc * NMAX * 64 + kk * 32);
                                ptx::mma_mxf8f6f4_ts(d_tmem, sb + C::kACol + kk * 8, bd, idesc, sb + C::kSfaCol,
                                                     tmem + C::kSfbCol + pc * C::kSfbStride, (s != s0) | ch | kk | pc);
                            }
                        }
                        ptx::mma_commit(bar(ADONE + ci % NA));
                    }
                    // the stage (codes, scales and the token rows the MMAs read) is
                    // free once this group's copies and MMAs completed
                    ptx::mma_commit(bar(DONEG + st));
                }
                if (!ok) break;
                ptx::mma_commit(bar(ACCREADY));
            }
        }
        if (!ok && issued) {
            // wait until the copies and MMAs already issued have retired
            // (bounded); the latest commit covers every earlier one
            const uint32_t last = it > 0 ? it - 1 : 0;
            for (uint32_t t = 0; t < kWaitLimit; ++t)
                if (ptx::mbar_try_wait(bar(DONEG + (last % S)), (last / S) & 1)) break;
            if (ci > 0) {
                const uint32_t lc = ci - 1;
                for (uint32_t t = 0; t < kWaitLimit; ++t)
                    if (ptx::mbar_try_wait(bar(ADONE + (lc % NA)), (lc / NA) & 1)) break;
            }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == C::kMmaWarp) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, C::kCols);
    }
}
