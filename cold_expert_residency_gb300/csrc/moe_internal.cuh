// Internal definitions of the split-residency MoE library (not part of the
// C ABI).  Device layout of an expert, workspace layout, context state and
// launch helpers.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>

#include <atomic>
#include <cstdint>
#include <string>
#include <vector>

#include "../../include/moe_residency.h"

namespace moe {

// ---------------------------------------------------------------------------
// Device layout of one expert ("tiled MXFP4")
//
// Both GEMMs of an expert are cut into M-tiles of 128 weight rows and K-chunks
// of 64 elements.  One (M-tile, K-chunk) is stored contiguously as
//     [half h = 0,1][row m = 0..127][16 bytes]   (4096 B: 32 e2m1 codes per
//                                                  16 B, i.e. one MX block)
//     [row m][2 scale bytes]                      (256 B: the row's two e8m0
//                                                  scales of this chunk)
// Inside a half, 32-bit word j (bytes 4j..4j+3) holds the block's elements
// 8j..8j+7: byte i carries element 8j+i in its low nibble and element
// 8j+4+i in its high nibble.  Two masked shifts of the word then give the
// one-code-per-byte form the tensor cores read from tensor memory.
// = 4352 bytes, exactly the logical bytes of those 128 x 64 elements.  Chunks
// of a tile follow in K order, tiles in M order; the W13 tiles come first,
// then the W2 tiles.  So the bank stores the same bytes the logical layout
// holds (18,800,640 per expert at H=4096, I=2880), permuted so that a warp's
// 16-byte loads are contiguous and one tile's chunk is one bulk copy.
//
// W13 M-tile mt covers gate units i = 64*mt .. 64*mt+63 and their up rows:
// tile row m = 32*w + l (w = m/32, l = m%32) holds W13 row
//     (l < 16 ? 0 : I) + 64*mt + 16*w + (l % 16),
// so within a warp lane l (gate) and lane l^16 (up) hold the same unit.
// W2 M-tile mt row m holds W2 row 128*mt + m.
// ---------------------------------------------------------------------------
constexpr int kKC = 64;                       // K elements per chunk
constexpr int kMT = 128;                      // weight rows per M-tile
constexpr int kChunkQBytes = kMT * kKC / 2;   // 4096
constexpr int kChunkBytes = kChunkQBytes + kMT * 2;  // 4352

struct Geom {
    int L, E, k, H, I, count_tmax, Tmax;
    int64_t eb;                // bytes per expert
    int mt13, kc13;            // W13: M-tiles (I/64) and K-chunks (H/64)
    int mt2, kc2;              // W2:  M-tiles (H/128) and K-chunks (I/64)
    int64_t w2_off;            // byte offset of the W2 tiles in an expert
};

inline Geom make_geom(const moe_geom &g) {
    Geom o;
    o.L = g.layers; o.E = g.experts; o.k = g.top_k; o.H = g.hidden; o.I = g.inter;
    o.count_tmax = g.count_tmax; o.Tmax = g.max_tokens;
    o.mt13 = g.inter / 64; o.kc13 = g.hidden / kKC;
    o.mt2 = g.hidden / kMT; o.kc2 = g.inter / kKC;
    o.w2_off = (int64_t)o.mt13 * o.kc13 * kChunkBytes;
    o.eb = o.w2_off + (int64_t)o.mt2 * o.kc2 * kChunkBytes;
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
    size_t hdr, act_row, act_off, picks, epos, ecnt, xq, xgexp, h32, hq, hexp, gu32, y32, claim, total;
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
    w.claim = take(1024 * 4);                   // [SM] first-CTA claims of a launch over both banks
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
    std::vector<int32_t> rowmap;   // CPU copy
};

}  // namespace moe

struct moe_ctx {
    moe::Geom g;
    int device = 0;
    int sms = 0;
    int ffn_impl = MOE_FFN_TCGEN05;
    int32_t *counts_dev = nullptr;   // [L][E]
    uint8_t *staging = nullptr;      // one expert row in HBM
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
// over both banks); hot/cold: the banks' device-visible bases (null if
// unused); shared: the layer has rows in both banks (one-bank launches may
// overlap)
int launch_ffn_tc(moe_ctx *ctx, const uint8_t *hot, const uint8_t *cold, int bank_id, const uint16_t *x, int T,
                  uint8_t *ws, uint16_t *Y, cudaStream_t s, bool shared);
int launch_finalize(const uint16_t *Y, const float *w, int T, int k, int H, uint16_t *out,
                    cudaStream_t s);
int launch_rowmap_write(int32_t *rowmap_dev, int32_t e0, int32_t v0, int32_t e1, int32_t v1,
                        cudaStream_t s);
int launch_probe_read(const uint8_t *src, size_t bytes, uint64_t *sink, int blocks,
                      cudaStream_t s);

}  // namespace moe
