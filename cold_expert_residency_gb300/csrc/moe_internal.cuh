// Internal definitions of the split-residency MoE library (not part of the
// C ABI).  Device layout of an expert, workspace layout, context state and
// launch helpers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <string>
#include <vector>

#include "../../include/moe_residency.h"

namespace moe {

// ---------------------------------------------------------------------------
// Device layout of one expert ("tiled MXFP4")
//
// Both GEMMs of an expert are cut into M-tiles of 128 weight rows and K-groups
// of 128 elements.  One (M-tile, K-group) is stored contiguously as
//     [row m = 0..127][64 bytes]    (8192 B: the row's 128 e2m1 codes, element
//                                    2i in the low nibble of byte i, as in
//                                    the logical MXFP4 rows)
//     [512-byte scale atom]          (the e8m0 scale of row m and 32-element K
//                                    block kb at byte (m%32)*16 + 4*(m/32) + kb)
// = 8704 bytes.  The code block is what one tensor-TMA box of the padded 4-bit
// type moves into shared memory in the layout the tensor cores read; the
// scale atom is what one tensor-memory copy (32 lanes x 16 bytes, repeated in
// all four lane quarters) puts where the block-scaled MMA reads A's scales.
//
// W13 M-tile mt covers gate units i = 64*mt .. 64*mt+63 and their up rows:
// tile row m = 32*w + l (w = m/32, l = m%32) holds W13 row
//     (l < 16 ? 0 : I) + 64*mt + 16*w + (l % 16),
// so within a warp lane l (gate) and lane l^16 (up) hold the same unit.
// W2 M-tile mt row m holds W2 row 128*mt + m.
//
// A part (W13 or W2) is a sequence of tile slots: tile t's groups in K order.
// W2's K (= I) may end in half a group (I % 128 == 64).  Then M-tiles 2p and
// 2p+1 are stored as a pair: tile 2p's full groups, tile 2p+1's full groups,
// and one shared group whose K blocks 0-1 hold tile 2p's last 64 columns and
// blocks 2-3 tile 2p+1's.  Either way an expert holds exactly its logical
// MXFP4 bytes (18,800,640 at H=4096, I=2880), permuted.
// ---------------------------------------------------------------------------
constexpr int kKC = 64;                       // K elements per chunk (one token-row record)
constexpr int kKG = 128;                      // K elements per group
constexpr int kMT = 128;                      // weight rows per M-tile
constexpr int kGroupQBytes = kMT * kKG / 2;   // 8192
constexpr int kSfAtomBytes = 512;
constexpr int kGroupBytes = kGroupQBytes + kSfAtomBytes;   // 8704

struct PartLayout {
    int64_t off;           // byte offset of the part in an expert
    int64_t tile_stride;   // bytes per tile index (a tile, or a pair of tiles)
    int tiles;             // M-tiles
    int gfull;             // full K groups per tile
    int paired;            // 1: the last K group is half, shared by tiles 2p and 2p+1
    int kchunks;           // K / 64
    __host__ __device__ int steps() const { return gfull + paired; }
    __host__ __device__ int tile_index_count() const { return paired ? tiles / 2 : tiles; }
    __host__ __device__ int slots() const { return paired ? 2 * gfull + 1 : gfull; }
    // K step s of tile mt: its group's slot and tile index, and the first and
    // number of the group's 32-wide K blocks that belong to this tile
    __host__ __device__ void group(int mt, int s, int &slot, int &tidx, int &kb0, int &nkb) const {
        if (!paired) {
            slot = s; tidx = mt; kb0 = 0; nkb = 4;
        } else {
            tidx = mt >> 1;
            if (s < gfull) { slot = (mt & 1) * gfull + s; kb0 = 0; nkb = 4; }
            else { slot = 2 * gfull; kb0 = 2 * (mt & 1); nkb = 2; }
        }
    }
    __host__ __device__ int64_t group_off(int slot, int tidx) const {
        return off + (int64_t)tidx * tile_stride + (int64_t)slot * kGroupBytes;
    }
};

struct Geom {
    int L, E, k, H, I, count_tmax, Tmax;
    int64_t eb;                // bytes per expert
    PartLayout w13, w2;
    int mt13, mt2;             // M-tiles of W13 (I/64) and W2 (H/128)
    int64_t w2_off;            // byte offset of the W2 part in an expert
};

inline Geom make_geom(const moe_geom &g) {
    Geom o;
    o.L = g.layers; o.E = g.experts; o.k = g.top_k; o.H = g.hidden; o.I = g.inter;
    o.count_tmax = g.count_tmax; o.Tmax = g.max_tokens;
    o.mt13 = g.inter / 64;
    o.mt2 = g.hidden / kMT;
    o.w13.off = 0;
    o.w13.tiles = o.mt13;
    o.w13.gfull = g.hidden / kKG;
    o.w13.paired = 0;
    o.w13.kchunks = g.hidden / kKC;
    o.w13.tile_stride = (int64_t)o.w13.gfull * kGroupBytes;
    o.w2_off = (int64_t)o.mt13 * o.w13.tile_stride;
    o.w2.off = o.w2_off;
    o.w2.tiles = o.mt2;
    o.w2.gfull = g.inter / kKG;
    o.w2.paired = (g.inter / kKC) % 2;
    o.w2.kchunks = g.inter / kKC;
    o.w2.tile_stride = (int64_t)o.w2.slots() * kGroupBytes;
    o.eb = o.w2_off + (int64_t)o.w2.tile_index_count() * o.w2.tile_stride;
    return o;
}

// ---------------------------------------------------------------------------
// Workspace (caller-owned device memory) for a step of T tokens, P = T*k.
// Every region starts on a 256-byte boundary.
// ---------------------------------------------------------------------------
// Rows of the FFN's intermediate arrays are indexed by the pick's global
// position g: hot picks take g = p, cold picks g = P - n_cold + p (p = the
// pick's index in its bank's list), so the two banks never share a row and
// each expert's rows are contiguous.
struct WsLayout {
    size_t hdr, act_row, act_off, picks, epos, ecnt, ccnt, xq, xgexp, h32, hq, hexp, gu32, y32, claim;
    // prefill-sized steps with MXFP8 activations: per bank, the first token
    // tile of each active row, and the tiles' B-operand block scales
    size_t tile_off, sfx, sfh;
    int max_tiles;          // token tiles per bank, at most
    // cold staging: the slot of each cold active row (or -1), the cold row of
    // each slot (or -1)
    size_t stage_slot, stage_src;
    size_t total;
};
// header words
// kHdrSched + 2*bank + phase: work counters of the FFN kernels' dynamic
// unit scheduler (zeroed by the bank's first FFN kernel).
enum { kHdrNPicks = 0, kHdrNAct = 2, kHdrSched = 8, kHdrWords = 64 };

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Steps of at most this many tokens run the FFN with narrow token tiles and
// two K halves per unit.
constexpr int kNarrowMaxT = 256;
inline bool split_k_steps(int T) { return T <= kNarrowMaxT; }

// Token rows per prefill tile: 144 with two e4m3 pieces per value (a ring of
// four 53 KB stages), 160 in the MXFP8 format (six 38 KB stages); an expert
// with more picks takes further tiles.  And the bytes of one K group's
// B-operand block scales of one tile in the MXFP8 format: two 32-row x
// 16-byte atoms, row l of atom c holding tokens 32*(4c + q) + l (q = 0..3),
// 4 bytes each (the group's four 32-wide K blocks) -- what tcgen05.cp puts
// where the block-scaled MMA reads token n's scale (column n/32, lane n%32).
constexpr int kPrefillTile = 144;
constexpr int kPrefillTileMx = 160;
constexpr int kSfbGroupBytes = 1024;

// Slots of a context's cold-staging pool, at most.
constexpr int kMaxStageSlots = 64;

// Token rows per tile of the FFN kernels for a step of T tokens (mx: the
// MXFP8 activation format).
inline int tile_width(int T, bool mx) {
    return T <= 8 ? 8 : T <= 16 ? 16 : T <= kNarrowMaxT ? 32 : (mx ? kPrefillTileMx : kPrefillTile);
}

inline WsLayout ws_layout(const Geom &g, int T) {
    WsLayout w;
    size_t P = (size_t)T * g.k;
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t o = off; off = align256(off + bytes); return o; };
    w.hdr = take(kHdrWords * 4);
    w.act_row = take(2 * P * 4);              // [2][P]
    w.act_off = take(2 * (P + 1) * 4);        // [2][P+1]
    w.picks = take(2 * P * 4);                // [2][P]
    w.epos = take((size_t)g.E * 4);           // [E] start of expert e's picks in its bank list
    w.ecnt = take((size_t)g.E * 4);           // [E] picks per expert (large-step routing path)
    // large steps: picks per expert in each 32-token chunk, then each chunk's
    // first place in its expert's list ([E][chunks], expert-major)
    w.ccnt = take(split_k_steps(T) ? 0 : (size_t)g.E * ((T + 31) / 32) * 4);
    w.xq = take(P * (size_t)g.H * 2);         // [P][H/64][2][64] e4m3 token rows in pick order (two pieces)
    w.xgexp = take(P * 4);                    // [P] int32 scale exponents of those rows
    w.h32 = take(P * (size_t)g.I * 4);        // [P][I] fp32 gate/up output (by g; by slot on CUDA cores)
    w.hq = take(P * (size_t)g.I * 2);         // [P][I/64][2][64] e4m3 h rows (two pieces), by g
    w.hexp = take(P * 4);                     // [P] int32
    // Narrow-tile steps split each GEMM unit into two K halves whose partial
    // sums meet in these fp32 rows (see the tensor-core FFN).
    const size_t ks = split_k_steps(T) ? 1 : 0;
    w.gu32 = take(ks * P * (size_t)g.I * 2 * 4); // [P][2I] gate/up sums before SwiGLU, by g
    w.y32 = take(ks * P * (size_t)g.H * 4);     // [P][H] down-GEMM sums, by slot
    w.claim = take(2 * 1024 * 4);               // [GEMM][SM] first-CTA claims of a launch over both banks
    // prefill tiles, MXFP8 format: a bank's tiles are at most one per active
    // row (<= min(P, E) rows) plus P / kPrefillTileMx
    const size_t wide = split_k_steps(T) ? 0 : 1;
    w.max_tiles = (int)(wide * (std::min<size_t>(P, (size_t)g.E) + P / kPrefillTileMx + 1));
    w.tile_off = take(wide * 2 * (P + 1) * 4);  // [2][P+1] int32
    w.sfx = take((size_t)2 * w.max_tiles * (g.H / kKG) * kSfbGroupBytes);
    w.sfh = take((size_t)2 * w.max_tiles * ((g.I + kKG - 1) / kKG) * kSfbGroupBytes);
    w.stage_slot = take(P * 4);
    w.stage_src = take(kMaxStageSlots * 4);
    w.total = off;
    return w;
}

// Device-side view of one bank's split lists.
struct BankLists {
    const int32_t *hdr;        // n_picks at [kHdrNPicks + b], n_act at [kHdrNAct + b]
    const int32_t *act_row;    // [P]
    const int32_t *act_off;    // [P+1]
    const int32_t *picks;      // [P]
};

// ---------------------------------------------------------------------------
// Context
// ---------------------------------------------------------------------------
struct Layer {
    bool init = false;
    int n_hot = 0, n_cold = 0;
    uint8_t *hot = nullptr;        // device: n_hot * eb
    uint8_t *cold_host = nullptr;  // pinned host: n_cold * eb
    uint8_t *cold_dev = nullptr;   // device view of cold_host
    void *cold_map = nullptr;      // the huge-page mapping holding cold_host (null: cudaHostAlloc)
    size_t cold_map_bytes = 0;
    int32_t *rowmap_dev = nullptr; // device int32[E]
    // tensor maps of the weight code blocks: [bank][part] (part 0 = W13,
    // 1 = W2); valid where the bank has rows
    CUtensorMap wmap[2][2];
    std::vector<int32_t> rowmap;   // CPU copy
};

}  // namespace moe

namespace moe {
constexpr uint64_t kDefaultWaitNs = 1000000000ull;   // 1 s bound of a device pipeline wait
}

struct moe_ctx {
    moe::Geom g;
    int device = 0;
    int sms = 0;
    int ffn_impl = MOE_FFN_TCGEN05;
    int act_format = MOE_ACT_E4M3X2;          // token rows of prefill-sized steps
    int stage_slots = 0;                      // cold-staging pool: slots (0 = off)
    uint8_t *stage_pool = nullptr;            // stage_slots expert rows in HBM
    CUtensorMap stage_map[2];                 // code-block maps over the pool (W13, W2)
    uint64_t wait_ns = moe::kDefaultWaitNs;   // bound of every FFN pipeline wait
    bool inject_withhold = false;             // test hook: the next FFN call withholds one copy
    int32_t *counts_dev = nullptr;   // [L][E]
    uint8_t *staging = nullptr;      // two expert rows in HBM (swaps alternate between them)
    cudaStream_t swap_stream = nullptr;   // a swap's copy back to the host bank
    cudaEvent_t swap_in[2] = {nullptr, nullptr}, swap_out[2] = {nullptr, nullptr};
    int32_t *status_dev = nullptr;   // bounded-wait status word
    uint8_t *probe_host = nullptr;   // pinned probe buffer for moe_probe_link
    uint8_t *probe_dev = nullptr;
    size_t probe_bytes = 0;
    std::vector<moe::Layer> layers;
};

namespace moe {

// error reporting (per thread)
int set_error(int code, const std::string &msg);
int cuda_error(cudaError_t e, const char *what);
// argument checks shared by the entry points: a non-null context; a layer
// index in range (and, with need_init, a layer whose banks are placed)
int check_ctx(const moe_ctx *ctx);
int check_layer(moe_ctx *ctx, int layer, bool need_init);

// Makes `dev` the calling thread's current device for the guard's lifetime
// and restores the previous one after.  status() is the cudaSetDevice result
// (cudaSuccess when the device was already current).
struct DeviceGuard {
    int prev = -1;
    cudaError_t err = cudaSuccess;
    explicit DeviceGuard(int dev) {
        err = cudaGetDevice(&prev);
        if (err == cudaSuccess && prev != dev) err = cudaSetDevice(dev);
    }
    cudaError_t status() const { return err; }
    ~DeviceGuard() {
        int cur;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};
// An entry point's device switch: the context's device is current for the
// rest of the enclosing function, or the function returns the failure.
#define MOE_ON_DEVICE(dev)                                  \
    moe::DeviceGuard moe_dev_guard_(dev);                    \
    if (moe_dev_guard_.status() != cudaSuccess)              \
    return moe::cuda_error(moe_dev_guard_.status(), "cudaSetDevice(context device)")
#define MOE_CUDA_TRY(call)                                   \
    do {                                                     \
        cudaError_t e_ = (call);                             \
        if (e_ != cudaSuccess) return moe::cuda_error(e_, #call); \
    } while (0)
// process-wide count of kernels this library launched
extern std::atomic<int64_t> g_launches;
#define MOE_LAUNCH_CHECK()                                                 \
    do {                                                                   \
        cudaError_t e_ = cudaGetLastError();                               \
        if (e_ != cudaSuccess) return moe::cuda_error(e_, "kernel launch"); \
        moe::g_launches.fetch_add(1, std::memory_order_relaxed);           \
    } while (0)

// kernels' host launchers (defined in their .cu files)
int launch_route_split(moe_ctx *ctx, int layer, const float *logits, int T, int count_on,
                       int32_t *ids, float *w, uint8_t *ws, cudaStream_t s);
int launch_ffn_simt(moe_ctx *ctx, const uint8_t *bank, int bank_id, const uint16_t *x, int T,
                    uint8_t *ws, uint16_t *Y, cudaStream_t s);
// bank_id: MOE_BANK_HOT, MOE_BANK_COLD, or MOE_BANK_BOTH (one launch per GEMM
// over both banks); a layer with rows in both banks sizes one-bank launches so
// that the two banks' launches can run side by side
int launch_ffn_tc(moe_ctx *ctx, const Layer &layer, int bank_id, const uint16_t *x, int T, uint8_t *ws,
                  uint16_t *Y, cudaStream_t s);
// Tensor map over one part's code blocks in a bank of `rows` experts at `bank`
// (device-visible address; 16U4_ALIGN16B boxes of 128 x 128 codes, 128-byte
// swizzle).
int make_weight_map(CUtensorMap *map, const uint8_t *bank, const Geom &g, const PartLayout &part, int rows);
int launch_finalize(const uint16_t *Y, const float *w, int T, int k, int H, uint16_t *out,
                    cudaStream_t s);
int launch_router(const uint16_t *x, const uint16_t *w_router, const float *bias, int T, int E, int H,
                  float *logits, int32_t *status, int sms, cudaStream_t s);
int launch_rowmap_write(int32_t *rowmap_dev, int32_t e0, int32_t v0, int32_t e1, int32_t v1,
                        cudaStream_t s);
// Select the step's cold rows to stage (tile width W) and copy them into the
// context's pool (cold_stage.cu).
int launch_cold_staging(moe_ctx *ctx, const Layer &layer, int W, const BankLists &cold_lists, int32_t *slot_of,
                        int32_t *src_of, cudaStream_t s);
int launch_probe_read(const uint8_t *src, size_t bytes, uint64_t *sink, int blocks,
                      cudaStream_t s);

}  // namespace moe
