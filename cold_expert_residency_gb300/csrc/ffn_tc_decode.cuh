// Decode-tile variant of the tensor-core expert FFN (included by ffn_tc.cu).
//
// A decode step streams each active expert once for a handful of tokens, so
// the GEMMs are bound by how many weight bytes each SM keeps in flight.  The
// padded shared-memory form of e2m1 that the MMA reads from shared memory
// costs two bytes of shared memory per weight byte; here the weights land
// packed (one 1-D bulk copy of the 8704-byte group: code block and scale
// atom) and the SM spreads them into tensor memory, where the MMA reads A:
//
//   producer  one thread: per K group, a bulk copy of the group from HBM (hot
//             bank) or the mapped pinned host bank (cold bank), and one 4-D
//             tensor-TMA box of the tile's token rows ([chunk][piece][row]).
//   unpack    four warps, thread m = weight row m = TMEM lane m: per 64-wide
//             chunk, the row's 32 code bytes become 16 TMEM columns of one
//             code per byte (bits 5..2) -- element 8j+2b in byte b of column
//             2j and element 8j+2b+1 in byte b of column 2j+1, two masked
//             shifts per word -- plus the row's four scale bytes.  The K
//             order inside each group of eight elements is thus permuted;
//             the token rows of decode tiles are written with the same
//             permutation, so every dot product is unchanged.  The same warps
//             run the epilogue.
//   MMA       one warp, one elected lane issuing: per chunk, tcgen05.mma
//             kind::mxf8f6f4 with A and its scales from TMEM, B from shared
//             memory; commits free the A slot (per chunk) and the stage (per
//             group).
//
// Bounded waits and teardown as in the shared-memory-A kernel.

template <int NMAX>
struct DecCfg {
    static constexpr bool kStack = NMAX <= 16;              // both e4m3 pieces as rows of one MMA
    static constexpr int kBChunk = 2 * NMAX * 64;           // one chunk's token rows: [piece][NMAX rows][64 B]
    static constexpr int kBStage = 2 * kBChunk;
    static constexpr int kRowQ = kStack ? NMAX : 16;
    static constexpr int kStages = NMAX <= 8 ? 5 : (NMAX <= 16 ? 4 : 3);   // K groups in the ring
    static constexpr int kPerSm = 4;                        // resident CTAs per SM
    static constexpr int kABufs = 3;                        // TMEM A slots, one chunk each
    static constexpr int kDW = (kStack ? 2 : 1) * NMAX;     // accumulator columns
    static constexpr int kNCol = (kDW + 31) / 32;           // B scale columns of one piece
    // Tensor memory: slot s owns the 32-column block at 32 s: its A scale
    // columns at +0 (quarter q at +q), its codes (16 columns) at +16; blocks
    // 0 and 1 also hold the B scale columns of piece 0 and 1 at +8 (stacked
    // tiles use block 0's for both).  The accumulator follows the slots.
    static constexpr uint32_t kSfaCol = 0, kSfbCol = 8, kACol = 16, kSfbStride = 32;
    static constexpr uint32_t kDCol = 32 * kABufs;
    static constexpr uint32_t kColsUsed = kDCol + kDW;
    static constexpr uint32_t kCols = kColsUsed <= 64 ? 64 : (kColsUsed <= 128 ? 128 : 256);
    static_assert(kCols * kPerSm <= 512 && kNCol <= 8 && kABufs >= 2, "tensor memory");
    static_assert(NMAX % 8 == 0 && kDW % 16 == 0, "tile alignment");
    static constexpr int kSplit = 2;                        // K halves per unit
    static constexpr int kProducer = 4, kMmaWarp = 5;
    static constexpr int kThreads = 192;
    static constexpr int kBars = 2 * kStages + 2 * kABufs + 2 + 2 * kQ;
    static constexpr size_t kSmem = 1024 + (size_t)kStages * (kBStage + kGroupBytes) + kBars * 8 + 16 + 4 * kQ;
    static_assert((kSmem + 1024) * kPerSm <= 228u * 1024u, "shared memory");
};

// 8 e2m1 codes (element 2i in the low nibble of byte i) -> the even elements
// in bytes 0..3 of `ev`, the odd ones in bytes 0..3 of `od`, each code in
// bits 5..2 of its byte.
__device__ __forceinline__ void unpack_word(uint32_t w, uint32_t &ev, uint32_t &od) {
    ev = (w << 2) & 0x3C3C3C3Cu;
    od = (w >> 2) & 0x3C3C3C3Cu;
}

template <int NMAX, int PHASE, int BANKS>
__global__ void __launch_bounds__(DecCfg<NMAX>::kThreads, DecCfg<NMAX>::kPerSm)
    ffn_tc_decode_kernel(const __grid_constant__ CUtensorMap tmB, TcArgs args) {
    using C = DecCfg<NMAX>;
    constexpr int S = C::kStages, NA = C::kABufs;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (ptx::smem_addr(smem_raw) & 1023u)) & 1023u);
    uint8_t *sB = smem;                          // [S][2 chunks][2 pieces][NMAX rows][64 B], 64-byte swizzle
    uint8_t *sA = sB + S * C::kBStage;           // [S][8704]: code block and scale atom
    uint64_t *bars = (uint64_t *)(sA + S * kGroupBytes);
    uint32_t *holder = (uint32_t *)(bars + C::kBars);
    volatile int *abort_flag = (volatile int *)(holder + 1);
    volatile int *uq = (volatile int *)(holder + 2);
    auto bar = [&](int i) { return ptx::smem_addr(bars + i); };
    // FULL: group landed.  DONEG: the group's MMAs completed (stage free).
    // AREADY / ADONE: A slot written / its MMAs completed.
    const int FULL = 0, DONEG = S, AREADY = 2 * S, ADONE = 2 * S + NA, ACCREADY = 2 * S + 2 * NA,
              ACCFREE = ACCREADY + 1, UQFULL = ACCFREE + 1, UQEMPTY = UQFULL + kQ;
    constexpr int kQueueReaders = 128 + 1;
    constexpr bool SUSP = true;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (BANKS == 1) {
        // A cold-bank launch keeps one host-link streamer per SM: a CTA placed
        // on an SM that already holds one leaves at once.
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
        for (int i = 0; i < NA; ++i) {
            ptx::mbar_init(bar(AREADY + i), 128);
            ptx::mbar_init(bar(ADONE + i), 1);
        }
        ptx::mbar_init(bar(ACCREADY), 1);
        ptx::mbar_init(bar(ACCFREE), 128);
        for (int q = 0; q < kQ; ++q) {
            ptx::mbar_init(bar(UQFULL + q), 1);
            ptx::mbar_init(bar(UQEMPTY + q), kQueueReaders);
        }
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == C::kProducer && lane == 0) ptx::prefetch_tmap(&tmB);
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
        ptx::tmem_wait_st();   // made visible to the MMA by the first A-slot handoff
    }

    const PartLayout &part = args.part;
    const int ns = part.steps();
    auto units_of = [&](int bk) { return args.lists[0].hdr[kHdrNAct + bk] * part.tiles * args.ks; };
    // the unpack warps and the MMA warp read the unit sequence warp-wide;
    // of the MMA warp only lane 0 counts as a reader
    auto take_unit = [&](uint32_t ui, bool all_lanes, bool &ok) -> int {
        const int qs = ui % kQ;
        if (!wait_warp<SUSP>(bar(UQFULL + qs), (ui / kQ) & 1, abort_flag, args.status, args.wait_ns)) {
            ok = false;
            return -1;
        }
        const int u = uq[qs];
        if (all_lanes || lane == 0) ptx::mbar_arrive(bar(UQEMPTY + qs));
        return u;
    };

    if (warp < 4) {
        // ------------------------------------------------- unpack + epilogue
        const int quarter = warp, m = quarter * 32 + lane;
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        constexpr int NB = (NMAX + 15) / 16;
        uint32_t it = 0, ci = 0, j = 0;
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
                for (int s = s0; ok && s < s1; ++s, ++it) {
                    const int st = it % S;
                    if (!wait_warp<SUSP>(bar(FULL + st), (it / S) & 1, abort_flag, args.status, args.wait_ns)) { ok = false; break; }
                    int slot, tidx, kb0, nkb;
                    part.group(mt, s, slot, tidx, kb0, nkb);
                    const uint8_t *grp = sA + st * kGroupBytes;
                    // this row's four scale bytes (K blocks 0..3 of the group)
                    const uint32_t sf = *(const uint32_t *)(grp + kGroupQBytes + (m % 32) * 16 + 4 * (m / 32));
                    for (int ch = 0; ch < nkb / 2; ++ch, ++ci) {
                        const uint8_t *src = grp + m * 64 + (kb0 / 2 + ch) * 32;
                        const uint4 q0 = *(const uint4 *)src;
                        const uint4 q1 = *(const uint4 *)(src + 16);
                        uint32_t r[16];
                        unpack_word(q0.x, r[0], r[1]);
                        unpack_word(q0.y, r[2], r[3]);
                        unpack_word(q0.z, r[4], r[5]);
                        unpack_word(q0.w, r[6], r[7]);
                        unpack_word(q1.x, r[8], r[9]);
                        unpack_word(q1.y, r[10], r[11]);
                        unpack_word(q1.z, r[12], r[13]);
                        unpack_word(q1.w, r[14], r[15]);
                        const int abuf = ci % NA;
                        // the slot's previous chunk (ci - NA) must have been consumed
                        if (ci >= (uint32_t)NA &&
                            !wait_warp<SUSP>(bar(ADONE + abuf), ((ci / NA) - 1) & 1, abort_flag, args.status, args.wait_ns)) {
                            ok = false;
                            break;
                        }
                        ptx::tmem_st16(tmem + lane_base + C::kACol + abuf * 32, r);
                        ptx::tmem_st1(tmem + lane_base + C::kSfaCol + abuf * 32 + quarter, sf);
                        ptx::tmem_wait_st();
                        ptx::tc_fence_before();
                        ptx::mbar_arrive(bar(AREADY + abuf));
                    }
                }
                if (!ok) break;
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
        // A launch over both banks prefers, in the first CTA that reaches each
        // SM, the cold bank's units and in the others the hot bank's; each
        // turns to the other bank's queue once its own is empty.
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
            const int row = L.act_row[a];
            const int p0 = L.act_off[a], n = L.act_off[a + 1] - p0;
            // a staged cold row is read from its pool slot in HBM, not the host bank
            const int sslot = staged_slot(args, bk, a);
            const uint8_t *expert = sslot >= 0 ? args.stage_pool + (int64_t)sslot * args.eb
                                               : args.bank[bk] + (int64_t)row * args.eb;
            for (int n0 = 0; ok && n0 < n; n0 += NMAX) {
                const int brow = goff + p0 + n0;
                for (int s = s0; s < s1; ++s, ++it) {
                    const int st = it % S;
                    const uint32_t rnd = it / S;
                    if (rnd > 0) release_rows();
                    if (rnd > 0 && !wait_one<SUSP>(bar(DONEG + st), (rnd - 1) & 1, abort_flag, args.status, args.wait_ns)) {
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
                    // a half group's second token-row chunk is past the rows' end:
                    // zero fill, counted, unused
                    ptx::mbar_arrive_expect_tx(bar(FULL + st), (uint32_t)(kGroupBytes + C::kBStage));
                    ptx::bulk_g2s(ptx::smem_addr(sA + st * kGroupBytes), expert + part.group_off(slot, tidx), kGroupBytes,
                                  bar(FULL + st));
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
    } else if (warp == C::kMmaWarp) {
        // ----------------------------------------------------------- MMA issue
        // the whole warp runs the loop; one elected lane issues
        uint32_t it = 0, ci = 0, j = 0;
        bool ok = true;
        for (uint32_t ui = 0; ok; ++ui) {
            const int e = __shfl_sync(0xffffffffu, take_unit(ui, false, ok), 0);
            if (e < 0) break;
            const BankLists &L = args.lists[e & 1];
            int a, mt, s0, s1;
            unit_pos(e >> 1, part.tiles, ns, args.ks, a, mt, s0, s1);
            const int n = __shfl_sync(0xffffffffu, L.act_off[a + 1] - L.act_off[a], 0);
            for (int n0 = 0; ok && n0 < n; n0 += NMAX, ++j) {
                const int nn = min(NMAX, n - n0);
                const int Nr = (nn + C::kRowQ - 1) / C::kRowQ * C::kRowQ;
                const int Nm = C::kStack ? 2 * Nr : Nr;   // B rows of one MMA
                const uint32_t idesc0 = ptx::idesc_mx_e2m1_e4m3(128, Nm, 0, 0);   // | (scale byte << 29)
                if (j >= 1u && !wait_warp<SUSP>(bar(ACCFREE), (j - 1) & 1, abort_flag, args.status, args.wait_ns)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem + C::kDCol;
                for (int s = s0; ok && s < s1; ++s, ++it) {
                    const int st = it % S;
                    int slot, tidx, kb0, nkb;
                    part.group(mt, s, slot, tidx, kb0, nkb);
                    for (int ch = 0; ch < nkb / 2; ++ch, ++ci) {
                        const int abuf = ci % NA;
                        if (!wait_warp<SUSP>(bar(AREADY + abuf), (ci / NA) & 1, abort_flag, args.status, args.wait_ns)) {
                            ok = false;
                            break;
                        }
                        ptx::tc_fence_after();
                        const uint32_t a_tm = tmem + C::kACol + abuf * 32, sfa = tmem + C::kSfaCol + abuf * 32;
                        const uint32_t b_addr = ptx::smem_addr(sB + st * C::kBStage + ch * C::kBChunk);
                        if (ptx::elect_one()) {
#pragma unroll
                            for (int kk = 0; kk < 2; ++kk) {
                                const uint32_t idesc = idesc0 | ((uint32_t)(kb0 + 2 * ch + kk) << 29);
#pragma unroll
                                for (int pc = 0; pc < (C::kStack ? 1 : 2); ++pc) {
                                    const uint64_t bd = ptx::smem_desc_sw64(b_addr + pc * NMAX * 64 + kk * 32);
                                    ptx::mma_mxf8f6f4_ts(d_tmem, a_tm + kk * 8, bd, idesc, sfa,
                                                         tmem + C::kSfbCol + pc * C::kSfbStride,
                                                         (s != s0) | ch | kk | pc);
                                }
                            }
                            ptx::mma_commit(bar(ADONE + abuf));
                        }
                        __syncwarp();
                    }
                    if (!ok) break;
                    if (ptx::elect_one()) ptx::mma_commit(bar(DONEG + st));
                    __syncwarp();
                }
                if (!ok) break;
                if (ptx::elect_one()) ptx::mma_commit(bar(ACCREADY));
                __syncwarp();
            }
        }
        if (!ok && ci > 0) {
            // wait until the MMAs already issued have retired (bounded); the
            // last chunk's commit covers every earlier MMA of the issuing
            // lane (elect.sync over the converged warp elects the same lane
            // each time)
            const uint32_t last = ci - 1;
            for (uint32_t t = 0; t < kWaitLimit; ++t)
                if (ptx::mbar_try_wait(bar(ADONE + (last % NA)), (last / NA) & 1)) break;
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == C::kMmaWarp) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, C::kCols);
    }
}
