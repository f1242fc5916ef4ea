// C ABI of the split-residency MoE layer: context, banks, row maps, usage
// table, swaps and probes.  Kernels live in route_split.cu, ffn_simt.cu,
// ffn_tc.cu and finalize.cu.
#include "moe_internal.cuh"

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <sys/mman.h>
#include <thread>
#include <unordered_map>

namespace moe {

std::atomic<int64_t> g_launches{0};
static thread_local std::string g_last_error = "ok";

int set_error(int code, const std::string &msg) {
    g_last_error = msg;
    return code;
}

int cuda_error(cudaError_t e, const char *what) {
    std::string m = std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
    if (e == cudaErrorMemoryAllocation) return set_error(MOE_ENOMEM, m);
    return set_error(MOE_ECUDA, m);
}

// ---- library-owned memory, tracked process-wide (moe_memory_in_use) -------
static std::mutex g_mem_mu;
static std::unordered_map<const void *, std::pair<size_t, int>> g_mem;   // address -> (bytes, 0 device / 1 pinned)
static int64_t g_mem_bytes[2] = {0, 0};

static void track(const void *p, size_t n, int kind) {
    std::lock_guard<std::mutex> lock(g_mem_mu);
    g_mem[p] = {n, kind};
    g_mem_bytes[kind] += (int64_t)n;
}

static void untrack(const void *p) {
    std::lock_guard<std::mutex> lock(g_mem_mu);
    auto it = g_mem.find(p);
    if (it == g_mem.end()) return;
    g_mem_bytes[it->second.second] -= (int64_t)it->second.first;
    g_mem.erase(it);
}

// Test hook for the failure path of allocations: when the environment
// variable MOE_INJECT_ALLOC_FAIL names an allocation site, that site reports
// cudaErrorMemoryAllocation without allocating.
static bool injected_failure(const char *site) {
    const char *v = std::getenv("MOE_INJECT_ALLOC_FAIL");
    return v && std::strcmp(v, site) == 0;
}

static cudaError_t dev_alloc(void **p, size_t n, const char *site) {
    if (injected_failure(site)) return cudaErrorMemoryAllocation;
    cudaError_t e = cudaMalloc(p, n);
    if (e == cudaSuccess) track(*p, n, 0);
    return e;
}

static void dev_free(void *p) {
    if (!p) return;
    untrack(p);
    cudaFree(p);
}

static cudaError_t pinned_alloc(void **p, size_t n, unsigned flags, const char *site) {
    if (injected_failure(site)) return cudaErrorMemoryAllocation;
    cudaError_t e = cudaHostAlloc(p, n, flags);
    if (e == cudaSuccess) track(*p, n, 1);
    return e;
}

static void pinned_free(void *p) {
    if (!p) return;
    untrack(p);
    cudaFreeHost(p);
}

// Run f(i) for i in [0, n) on up to 32 host threads, the calling one
// included.  If a thread cannot be started, the ones that did (and the
// caller) take its share: nothing throws out of here.
template <class F>
static void parallel_for(int n, F f) {
    int threads = (int)std::max(1u, std::min(32u, std::thread::hardware_concurrency()));
    threads = std::min(threads, n);
    std::atomic<int> next{0};
    auto work = [&]() {
        for (int i = next.fetch_add(1); i < n; i = next.fetch_add(1)) f(i);
    };
    std::vector<std::thread> pool;
    for (int t = 1; t < threads; ++t) {
        try {
            pool.emplace_back(work);
        } catch (...) {
            break;
        }
    }
    work();
    for (auto &th : pool) th.join();
}

// The first GPU read of a page of mapped host memory sets up its address
// translation, which is far slower than the reads that follow it.  Touching
// every 4 KB of a cold bank once at placement takes that cost out of the
// layer-steps (a decode step would otherwise pay it for each cold expert the
// first time a token routes to it).
__global__ void touch_host_bank_kernel(const uint8_t *__restrict__ p, size_t bytes, uint32_t *sink) {
    uint32_t acc = 0;
    for (size_t off = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) * 4096; off < bytes;
         off += (size_t)gridDim.x * blockDim.x * 4096)
        acc ^= *(const volatile uint32_t *)(p + off);
    if (acc == 0x9E3779B9u && sink) *sink = acc;   // keeps the reads; almost never taken
}

// Logical MXFP4 expert -> tiled device layout (see moe_internal.cuh).
// q: [rows][K/2] codes, sc: [rows][K/32] e8m0 scales of one part; row_of(mt,
// m) names the logical row held by tile row m.  Every byte of the part is
// written.  Returns false if a scale byte lies outside [104, 140].
template <class RowOf>
static bool repack_part(const PartLayout &part, int K, const uint8_t *q, const uint8_t *sc, RowOf row_of, uint8_t *dst) {
    bool ok = true;
    for (int mt = 0; mt < part.tiles; ++mt) {
        for (int s = 0; s < part.steps(); ++s) {
            int slot, tidx, kb0, nkb;
            part.group(mt, s, slot, tidx, kb0, nkb);
            uint8_t *grp = dst + part.group_off(slot, tidx);
            for (int m = 0; m < kMT; ++m) {
                const int64_t row = row_of(mt, m);
                for (int i = 0; i < nkb; ++i) {
                    const int kb = kb0 + i, blk = 4 * s + i;   // the group's K block, the row's 32-element block
                    std::memcpy(grp + m * 64 + kb * 16, q + row * (K / 2) + blk * 16, 16);
                    const uint8_t e = sc[row * (K / 32) + blk];
                    grp[kGroupQBytes + (m % 32) * 16 + 4 * (m / 32) + kb] = e;
                    ok &= e >= 104 && e <= 140;
                }
            }
        }
    }
    return ok;
}

static bool repack_expert(const Geom &g, const uint8_t *w13_q, const uint8_t *w13_s,
                          const uint8_t *w2_q, const uint8_t *w2_s, uint8_t *dst) {
    const int I = g.I;
    std::memset(dst, 0, (size_t)g.eb);
    bool ok = repack_part(g.w13, g.H, w13_q, w13_s, [&](int mt, int m) {
        const int w = m / 32, l = m % 32;
        return (int64_t)(l < 16 ? 0 : I) + 64 * mt + 16 * w + (l % 16);
    }, dst);
    ok &= repack_part(g.w2, g.I, w2_q, w2_s, [&](int mt, int m) { return (int64_t)kMT * mt + m; }, dst);
    return ok;
}

// Pinned, device-mapped host memory for a cold bank.  The GPU reaches host
// memory through the host's page tables, and a bank of 64 KB pages needs
// tens of thousands of translations: more than the GPU keeps, so steps that
// route to rarely used cold experts stall on translation misses.  Large
// banks therefore go into an anonymous mapping aligned to 512 MB with huge
// pages requested (best effort), pinned with cudaHostRegister; anything that
// fails falls back to cudaHostAlloc.
static cudaError_t alloc_cold_bank(size_t bytes, moe::Layer &L) {
    constexpr size_t kAlign = 512ull << 20;
    if (injected_failure("cold_bank")) return cudaErrorMemoryAllocation;
    if (bytes >= (256ull << 20)) {
        const size_t span = (bytes + kAlign - 1) / kAlign * kAlign;
        void *m = mmap(nullptr, span + kAlign, PROT_READ | PROT_WRITE, MAP_PRIVATE | MAP_ANONYMOUS | MAP_NORESERVE,
                       -1, 0);
        if (m != MAP_FAILED) {
            uint8_t *a = (uint8_t *)(((uintptr_t)m + kAlign - 1) & ~(uintptr_t)(kAlign - 1));
            madvise(a, span, MADV_HUGEPAGE);
            if (cudaHostRegister(a, span, cudaHostRegisterMapped | cudaHostRegisterPortable) == cudaSuccess) {
                if (cudaHostGetDevicePointer((void **)&L.cold_dev, a, 0) == cudaSuccess) {
                    L.cold_host = a;
                    L.cold_map = m;
                    L.cold_map_bytes = span + kAlign;
                    track(a, span, 1);
                    return cudaSuccess;
                }
                cudaHostUnregister(a);
            }
            cudaGetLastError();   // the fallback below reports its own errors
            munmap(m, span + kAlign);
        }
    }
    cudaError_t e = pinned_alloc((void **)&L.cold_host, bytes, cudaHostAllocMapped | cudaHostAllocPortable, "cold_bank");
    if (e == cudaSuccess) e = cudaHostGetDevicePointer((void **)&L.cold_dev, L.cold_host, 0);
    return e;
}

static void free_layer(moe::Layer &L) {
    dev_free(L.hot);
    if (L.cold_map) {
        untrack(L.cold_host);
        cudaHostUnregister(L.cold_host);
        munmap(L.cold_map, L.cold_map_bytes);
    } else {
        pinned_free(L.cold_host);
    }
    dev_free(L.rowmap_dev);
    L = moe::Layer();
}

int check_ctx(const moe_ctx *ctx) {
    if (!ctx) return set_error(MOE_EINVAL, "null context");
    return MOE_OK;
}

int check_layer(moe_ctx *ctx, int layer, bool need_init) {
    if (int r = check_ctx(ctx)) return r;
    if (layer < 0 || layer >= ctx->g.L) return set_error(MOE_EINVAL, "layer out of range");
    if (need_init && !ctx->layers[layer].init)
        return set_error(MOE_ESTATE, "layer has no banks (call moe_init_banks first)");
    return MOE_OK;
}

}  // namespace moe

using namespace moe;

extern "C" {

const char *moe_last_error(void) { return g_last_error.c_str(); }

int64_t moe_expert_bytes(int32_t hidden, int32_t inter) {
    int64_t n = 2LL * inter * hidden + (int64_t)hidden * inter;
    return n / 2 + n / 32;
}

int moe_pack_expert(int32_t hidden, int32_t inter, const uint8_t *w13_q, const uint8_t *w13_s,
                    const uint8_t *w2_q, const uint8_t *w2_s, uint8_t *out) {
    if (!w13_q || !w13_s || !w2_q || !w2_s || !out) return set_error(MOE_EINVAL, "null argument");
    if (hidden < 128 || hidden % 128 || inter < 64 || inter % 64 || (hidden % 256 && inter % 128))
        return set_error(MOE_EINVAL, "invalid geometry (need H % 128 == 0, I % 64 == 0, "
                                     "H % 256 == 0 or I % 128 == 0)");
    moe_geom mg{};
    mg.layers = 1;
    mg.experts = 2;
    mg.top_k = 1;
    mg.hidden = hidden;
    mg.inter = inter;
    mg.max_tokens = 1;
    const Geom g = make_geom(mg);
    if (!repack_expert(g, w13_q, w13_s, w2_q, w2_s, out))
        return set_error(MOE_EINVAL, "e8m0 scale byte outside [104, 140]");
    return MOE_OK;
}

int moe_create(const moe_geom *geom, int device, moe_ctx **out) {
    if (!geom || !out) return set_error(MOE_EINVAL, "null argument");
    *out = nullptr;
    const moe_geom &g = *geom;
    if (g.layers < 1 || g.experts < 2 || g.experts > 1024 || g.top_k < 1 || g.top_k > 16 ||
        g.top_k > g.experts || g.hidden < 128 || g.hidden % 128 || g.inter < 64 || g.inter % 64 ||
        (g.hidden % 256 && g.inter % 128) ||
        g.max_tokens < 1 || g.count_tmax < 0)
        return set_error(MOE_EINVAL, "invalid geometry (need E in 2..1024, k in 1..min(16,E), "
                                     "H % 128 == 0, I % 64 == 0, H % 256 == 0 or I % 128 == 0, T_max >= 1)");
    if ((int64_t)g.max_tokens * g.top_k > (1 << 24))
        return set_error(MOE_EINVAL, "max_tokens * top_k too large");
    int ndev = 0;
    MOE_CUDA_TRY(cudaGetDeviceCount(&ndev));
    if (device < 0 || device >= ndev) return set_error(MOE_EINVAL, "no such CUDA device");
    MOE_ON_DEVICE(device);
    moe_ctx *ctx = new (std::nothrow) moe_ctx();
    if (!ctx) return set_error(MOE_ENOMEM, "out of host memory");
    ctx->g = make_geom(g);
    ctx->device = device;
    try {
        ctx->layers.resize(g.layers);
    } catch (const std::bad_alloc &) {
        delete ctx;
        return set_error(MOE_ENOMEM, "out of host memory");
    }
    cudaDeviceProp prop;
    cudaError_t e = cudaGetDeviceProperties(&prop, device);
    if (e == cudaSuccess) ctx->sms = prop.multiProcessorCount;
    if (e == cudaSuccess) e = dev_alloc((void **)&ctx->counts_dev, sizeof(int32_t) * g.layers * g.experts, "create_counts");
    if (e == cudaSuccess) e = cudaMemset(ctx->counts_dev, 0, sizeof(int32_t) * g.layers * g.experts);
    if (e == cudaSuccess) e = dev_alloc((void **)&ctx->staging, 2 * ctx->g.eb, "create_staging");
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&ctx->swap_stream, cudaStreamNonBlocking);
    for (int i = 0; i < 2 && e == cudaSuccess; ++i) {
        e = cudaEventCreateWithFlags(&ctx->swap_in[i], cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ctx->swap_out[i], cudaEventDisableTiming);
    }
    if (e == cudaSuccess) e = dev_alloc((void **)&ctx->status_dev, sizeof(int32_t) * 4, "create_status");
    if (e == cudaSuccess) e = cudaMemset(ctx->status_dev, 0, sizeof(int32_t) * 4);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        int r = cuda_error(e, "moe_create allocation");
        moe_destroy(ctx);
        return r;
    }
    *out = ctx;
    return MOE_OK;
}

int moe_destroy(moe_ctx *ctx) {
    if (!ctx) return MOE_OK;
    DeviceGuard guard(ctx->device);
    cudaDeviceSynchronize();
    for (auto &L : ctx->layers) free_layer(L);
    dev_free(ctx->counts_dev);
    dev_free(ctx->staging);
    for (int i = 0; i < 2; ++i) {
        if (ctx->swap_in[i]) cudaEventDestroy(ctx->swap_in[i]);
        if (ctx->swap_out[i]) cudaEventDestroy(ctx->swap_out[i]);
    }
    if (ctx->swap_stream) cudaStreamDestroy(ctx->swap_stream);
    dev_free(ctx->status_dev);
    pinned_free(ctx->probe_host);
    dev_free(ctx->probe_dev);
    dev_free(ctx->stage_pool);
    delete ctx;
    return MOE_OK;
}

int moe_set_ffn_impl(moe_ctx *ctx, int impl) {
    if (int r = check_ctx(ctx)) return r;
    if (impl != MOE_FFN_TCGEN05 && impl != MOE_FFN_SIMT) return set_error(MOE_EINVAL, "unknown FFN impl");
    ctx->ffn_impl = impl;
    return MOE_OK;
}

int moe_set_cold_staging(moe_ctx *ctx, int slots) {
    if (int r = check_ctx(ctx)) return r;
    if (slots < 0 || slots > kMaxStageSlots) return set_error(MOE_EINVAL, "staging slots out of range (0..64)");
    MOE_ON_DEVICE(ctx->device);
    MOE_CUDA_TRY(cudaDeviceSynchronize());   // no call in flight may still read the old pool
    dev_free(ctx->stage_pool);
    ctx->stage_pool = nullptr;
    ctx->stage_slots = 0;
    if (slots == 0) return MOE_OK;
    uint8_t *pool = nullptr;
    MOE_CUDA_TRY(dev_alloc((void **)&pool, (size_t)slots * ctx->g.eb, "stage_pool"));
    int r = make_weight_map(&ctx->stage_map[0], pool, ctx->g, ctx->g.w13, slots);
    if (r == MOE_OK) r = make_weight_map(&ctx->stage_map[1], pool, ctx->g, ctx->g.w2, slots);
    if (r != MOE_OK) {
        dev_free(pool);
        return r;
    }
    ctx->stage_pool = pool;
    ctx->stage_slots = slots;
    return MOE_OK;
}

int moe_read_stage(moe_ctx *ctx, const void *ws, int T, int32_t *rows, void *stream) {
    if (int r = check_ctx(ctx)) return r;
    if (!ws || !rows || T < 0 || T > ctx->g.Tmax) return set_error(MOE_EINVAL, "bad moe_read_stage arguments");
    MOE_ON_DEVICE(ctx->device);
    cudaStream_t s = (cudaStream_t)stream;
    const WsLayout lay = ws_layout(ctx->g, T);
    MOE_CUDA_TRY(cudaMemcpyAsync(rows, (const uint8_t *)ws + lay.stage_src, sizeof(int32_t) * kMaxStageSlots,
                                 cudaMemcpyDeviceToHost, s));
    MOE_CUDA_TRY(cudaStreamSynchronize(s));
    return MOE_OK;
}

int moe_set_act_format(moe_ctx *ctx, int format) {
    if (int r = check_ctx(ctx)) return r;
    if (format != MOE_ACT_E4M3X2 && format != MOE_ACT_MXFP8) return set_error(MOE_EINVAL, "unknown activation format");
    ctx->act_format = format;
    return MOE_OK;
}

int moe_init_banks(moe_ctx *ctx, int layer, const uint8_t *w13_q, const uint8_t *w13_s,
                   const uint8_t *w2_q, const uint8_t *w2_s, const uint8_t *is_hot, void *stream) {
    if (int r = check_layer(ctx, layer, false)) return r;
    if (!w13_q || !w13_s || !w2_q || !w2_s || !is_hot) return set_error(MOE_EINVAL, "null weight pointer");
    MOE_ON_DEVICE(ctx->device);
    cudaStream_t s = (cudaStream_t)stream;
    const Geom &g = ctx->g;
    Layer &L = ctx->layers[layer];
    MOE_CUDA_TRY(cudaStreamSynchronize(s));
    free_layer(L);

    std::vector<int32_t> rowmap(g.E);
    std::vector<int> hot_ids, cold_ids;
    for (int e = 0; e < g.E; ++e) {
        if (is_hot[e]) { rowmap[e] = (int32_t)hot_ids.size(); hot_ids.push_back(e); }
        else { rowmap[e] = -1 - (int32_t)cold_ids.size(); cold_ids.push_back(e); }
    }
    const size_t q13 = (size_t)2 * g.I * (g.H / 2), s13 = (size_t)2 * g.I * (g.H / 32);
    const size_t q2 = (size_t)g.H * (g.I / 2), s2 = (size_t)g.H * (g.I / 32);
    auto repack = [&](int e, uint8_t *dst) {
        return repack_expert(g, w13_q + e * q13, w13_s + e * s13, w2_q + e * q2, w2_s + e * s2, dst);
    };

    Layer nl;
    nl.n_hot = (int)hot_ids.size();
    nl.n_cold = (int)cold_ids.size();
    cudaError_t e = cudaSuccess;
    std::atomic<bool> scales_ok{true};
    if (nl.n_hot) e = dev_alloc((void **)&nl.hot, (size_t)nl.n_hot * g.eb, "hot_bank");
    if (e == cudaSuccess && nl.n_cold) {
        e = alloc_cold_bank((size_t)nl.n_cold * g.eb, nl);
    }
    if (e == cudaSuccess) e = dev_alloc((void **)&nl.rowmap_dev, sizeof(int32_t) * g.E, "rowmap");
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(nl.rowmap_dev, rowmap.data(), sizeof(int32_t) * g.E, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) {
        int r = cuda_error(e, "moe_init_banks allocation");
        free_layer(nl);
        return r;
    }
    // cold rows: repack straight into the pinned bank
    parallel_for((int)cold_ids.size(), [&](int i) {
        if (!repack(cold_ids[i], nl.cold_host + (size_t)i * g.eb)) scales_ok = false;
    });
    // hot rows: repack into pinned staging, batch by batch, then copy to HBM
    if (nl.n_hot) {
        const int batch = std::min(nl.n_hot, 16);
        uint8_t *pin = nullptr;
        e = pinned_alloc((void **)&pin, (size_t)batch * g.eb, cudaHostAllocDefault, "init_staging");
        for (int b0 = 0; e == cudaSuccess && b0 < nl.n_hot; b0 += batch) {
            int nb = std::min(batch, nl.n_hot - b0);
            parallel_for(nb, [&](int i) {
                if (!repack(hot_ids[b0 + i], pin + (size_t)i * g.eb)) scales_ok = false;
            });
            e = cudaMemcpyAsync(nl.hot + (size_t)b0 * g.eb, pin, (size_t)nb * g.eb, cudaMemcpyHostToDevice, s);
            if (e == cudaSuccess) e = cudaStreamSynchronize(s);
        }
        pinned_free(pin);
    }
    if (e == cudaSuccess && nl.n_cold) {
        touch_host_bank_kernel<<<4 * ctx->sms, 256, 0, s>>>(nl.cold_dev, (size_t)nl.n_cold * g.eb, nullptr);
        e = cudaGetLastError();
        if (e == cudaSuccess) g_launches.fetch_add(1, std::memory_order_relaxed);
    }
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) {
        int r = cuda_error(e, "moe_init_banks copy");
        free_layer(nl);
        return r;
    }
    if (!scales_ok) {
        free_layer(nl);
        return set_error(MOE_EINVAL, "e8m0 scale byte outside [104, 140]");
    }
    // tensor maps of each bank's code blocks, fixed for the banks' lifetime
    // (swaps move rows, never the banks)
    std::memset(nl.wmap, 0, sizeof(nl.wmap));
    for (int bk = 0; bk < 2; ++bk) {
        const int rows = bk == MOE_BANK_HOT ? nl.n_hot : nl.n_cold;
        const uint8_t *base = bk == MOE_BANK_HOT ? nl.hot : nl.cold_dev;
        if (!rows) continue;
        int r = make_weight_map(&nl.wmap[bk][0], base, g, g.w13, rows);
        if (r == MOE_OK) r = make_weight_map(&nl.wmap[bk][1], base, g, g.w2, rows);
        if (r != MOE_OK) {
            free_layer(nl);
            return r;
        }
    }
    nl.rowmap = std::move(rowmap);
    nl.init = true;
    L = std::move(nl);
    return MOE_OK;
}

int moe_workspace_bytes(const moe_ctx *ctx, int T, size_t *bytes) {
    if (int r = check_ctx(ctx)) return r;
    if (!bytes || T < 0 || T > ctx->g.Tmax) return set_error(MOE_EINVAL, "T out of range");
    // The layout is not monotonic in T: steps of at most kNarrowMaxT tokens
    // also hold fp32 partial-sum rows.  Size for the largest step of each kind.
    *bytes = std::max(ws_layout(ctx->g, T).total, ws_layout(ctx->g, std::min(T, kNarrowMaxT)).total);
    return MOE_OK;
}

int moe_route_split_count(moe_ctx *ctx, int layer, const float *logits, int T, int count_on,
                          int32_t *ids, float *w, void *ws, void *stream) {
    if (int r = check_layer(ctx, layer, true)) return r;
    if (T < 0 || T > ctx->g.Tmax) return set_error(MOE_EINVAL, "T out of range");
    if (T > 0 && (!logits || !ids || !w || !ws)) return set_error(MOE_EINVAL, "null pointer");
    if (!ws) return set_error(MOE_EINVAL, "null workspace");
    if ((uintptr_t)ws % 256) return set_error(MOE_EINVAL, "workspace must be 256-byte aligned");
    MOE_ON_DEVICE(ctx->device);
    return launch_route_split(ctx, layer, logits, T, count_on, ids, w, (uint8_t *)ws, (cudaStream_t)stream);
}

int moe_read_split(moe_ctx *ctx, const void *ws, int T, int bank, int32_t *n_act, int32_t *n_picks,
                   int32_t *act_row, int32_t *act_off, int32_t *picks, void *stream) {
    if (int r = check_ctx(ctx)) return r;
    if (!ws || T < 0 || T > ctx->g.Tmax || (bank != 0 && bank != 1) || !n_act || !n_picks || !act_row ||
        !act_off || !picks)
        return set_error(MOE_EINVAL, "bad moe_read_split arguments");
    MOE_ON_DEVICE(ctx->device);
    cudaStream_t s = (cudaStream_t)stream;
    const WsLayout lay = ws_layout(ctx->g, T);
    const size_t P = (size_t)T * ctx->g.k;
    const uint8_t *base = (const uint8_t *)ws;
    int32_t hdr[kHdrWords];
    MOE_CUDA_TRY(cudaMemcpyAsync(hdr, base + lay.hdr, sizeof hdr, cudaMemcpyDeviceToHost, s));
    MOE_CUDA_TRY(cudaStreamSynchronize(s));
    *n_act = hdr[kHdrNAct + bank];
    *n_picks = hdr[kHdrNPicks + bank];
    if (*n_act < 0 || (size_t)*n_act > P || *n_picks < 0 || (size_t)*n_picks > P)
        return set_error(MOE_ESTATE, "workspace does not hold a routed step of this T");
    MOE_CUDA_TRY(cudaMemcpyAsync(act_row, base + lay.act_row + bank * P * 4, sizeof(int32_t) * *n_act,
                                 cudaMemcpyDeviceToHost, s));
    MOE_CUDA_TRY(cudaMemcpyAsync(act_off, base + lay.act_off + bank * (P + 1) * 4, sizeof(int32_t) * (*n_act + 1),
                                 cudaMemcpyDeviceToHost, s));
    MOE_CUDA_TRY(cudaMemcpyAsync(picks, base + lay.picks + bank * P * 4, sizeof(int32_t) * *n_picks,
                                 cudaMemcpyDeviceToHost, s));
    MOE_CUDA_TRY(cudaStreamSynchronize(s));
    return MOE_OK;
}

int moe_expert_ffn_bank(moe_ctx *ctx, int layer, int bank, const uint16_t *x, int T, void *ws,
                        uint16_t *Y, void *stream) {
    if (int r = check_layer(ctx, layer, true)) return r;
    if (bank != MOE_BANK_HOT && bank != MOE_BANK_COLD && bank != MOE_BANK_BOTH)
        return set_error(MOE_EINVAL, "bank must be 0, 1 or 2");
    if (T < 0 || T > ctx->g.Tmax) return set_error(MOE_EINVAL, "T out of range");
    if (!ws || (uintptr_t)ws % 256) return set_error(MOE_EINVAL, "workspace must be non-null and 256-byte aligned");
    if (T > 0 && (!x || !Y)) return set_error(MOE_EINVAL, "null pointer");
    if (((uintptr_t)x | (uintptr_t)Y) % 16) return set_error(MOE_EINVAL, "x and Y must be 16-byte aligned");
    Layer &L = ctx->layers[layer];
    // a both-bank call over a layer with one empty bank is a one-bank call
    if (bank == MOE_BANK_BOTH && (L.n_hot == 0 || L.n_cold == 0)) bank = L.n_hot ? MOE_BANK_HOT : MOE_BANK_COLD;
    const int rows = bank == MOE_BANK_HOT ? L.n_hot : (bank == MOE_BANK_COLD ? L.n_cold : L.n_hot + L.n_cold);
    if (T == 0 || rows == 0) return MOE_OK;
    MOE_ON_DEVICE(ctx->device);
    cudaStream_t s = (cudaStream_t)stream;
    if (ctx->ffn_impl == MOE_FFN_SIMT) {
        for (int bk = 0; bk < 2; ++bk) {
            if (bank != MOE_BANK_BOTH && bank != bk) continue;
            const uint8_t *base = bk == MOE_BANK_HOT ? L.hot : L.cold_dev;
            if (int r = launch_ffn_simt(ctx, base, bk, x, T, (uint8_t *)ws, Y, s)) return r;
        }
        return MOE_OK;
    }
    return launch_ffn_tc(ctx, L, bank, x, T, (uint8_t *)ws, Y, s);
}

int moe_finalize(const uint16_t *Y, const float *w, int T, int k, int H, uint16_t *out, void *stream) {
    if (T < 0 || k < 1 || k > 16 || H < 8 || H % 8) return set_error(MOE_EINVAL, "bad finalize shape (H % 8 == 0)");
    if (T == 0) return MOE_OK;
    if (!Y || !w || !out) return set_error(MOE_EINVAL, "null pointer");
    if (((uintptr_t)Y | (uintptr_t)out) % 16) return set_error(MOE_EINVAL, "Y and out must be 16-byte aligned");
    return launch_finalize(Y, w, T, k, H, out, (cudaStream_t)stream);
}

namespace {

// Parts of a host-buffer step's scratch area for a step of T tokens, each on
// a 256-byte boundary: the workspace, then the step's device buffers.
struct StepScratch {
    size_t ws, logits, x, ids, w, Y, out, total;
};

StepScratch step_scratch(const moe_ctx *ctx, int T, size_t ws_bytes) {
    const moe::Geom &g = ctx->g;
    StepScratch p;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = (off + bytes + 255) / 256 * 256;
        return o;
    };
    p.ws = take(ws_bytes);
    p.logits = take((size_t)T * g.E * 4);
    p.x = take((size_t)T * g.H * 2);
    p.ids = take((size_t)T * g.k * 4);
    p.w = take((size_t)T * g.k * 4);
    p.Y = take((size_t)T * g.k * g.H * 2);
    p.out = take((size_t)T * g.H * 2);
    p.total = off;
    return p;
}

}  // namespace

int moe_step_scratch_bytes(const moe_ctx *ctx, int T, size_t *bytes) {
    if (int r = check_ctx(ctx)) return r;
    if (!bytes || T < 0 || T > ctx->g.Tmax) return set_error(MOE_EINVAL, "T out of range");
    size_t ws = 0;
    if (int r = moe_workspace_bytes(ctx, T, &ws)) return r;
    *bytes = step_scratch(ctx, T, ws).total;
    return MOE_OK;
}

int moe_layer_step_host(moe_ctx *ctx, int layer, const float *logits, const uint16_t *x, int T, int count_on,
                        uint16_t *out, void *scratch, void *stream) {
    if (int r = check_layer(ctx, layer, true)) return r;
    if (T < 0 || T > ctx->g.Tmax) return set_error(MOE_EINVAL, "T out of range");
    if (T == 0) return MOE_OK;
    if (!logits || !x || !out || !scratch) return set_error(MOE_EINVAL, "null pointer");
    if ((uintptr_t)scratch % 256) return set_error(MOE_EINVAL, "scratch must be 256-byte aligned");
    const moe::Geom &g = ctx->g;
    size_t ws = 0;
    if (int r = moe_workspace_bytes(ctx, T, &ws)) return r;
    const StepScratch p = step_scratch(ctx, T, ws);
    uint8_t *base = (uint8_t *)scratch;
    float *d_logits = (float *)(base + p.logits);
    uint16_t *d_x = (uint16_t *)(base + p.x), *d_Y = (uint16_t *)(base + p.Y), *d_out = (uint16_t *)(base + p.out);
    int32_t *d_ids = (int32_t *)(base + p.ids);
    float *d_w = (float *)(base + p.w);
    MOE_ON_DEVICE(ctx->device);
    cudaStream_t s = (cudaStream_t)stream;
    MOE_CUDA_TRY(cudaMemcpyAsync(d_logits, logits, (size_t)T * g.E * 4, cudaMemcpyHostToDevice, s));
    MOE_CUDA_TRY(cudaMemcpyAsync(d_x, x, (size_t)T * g.H * 2, cudaMemcpyHostToDevice, s));
    if (int r = moe_route_split_count(ctx, layer, d_logits, T, count_on, d_ids, d_w, base + p.ws, stream)) return r;
    if (int r = moe_expert_ffn_bank(ctx, layer, MOE_BANK_BOTH, d_x, T, base + p.ws, d_Y, stream)) return r;
    if (int r = moe_finalize(d_Y, d_w, T, g.k, g.H, d_out, stream)) return r;
    MOE_CUDA_TRY(cudaMemcpyAsync(out, d_out, (size_t)T * g.H * 2, cudaMemcpyDeviceToHost, s));
    return MOE_OK;
}

int moe_router_logits(moe_ctx *ctx, const uint16_t *x, const uint16_t *w_router, const float *bias, int T, int E,
                      int H, float *logits, void *stream) {
    if (!ctx) return set_error(MOE_EINVAL, "null context");
    if (T < 0 || E < 1 || E > (1 << 20) || H < 8 || H % 8)
        return set_error(MOE_EINVAL, "bad router shape (H % 8 == 0, 1 <= E <= 2^20)");
    if (T == 0) return MOE_OK;
    if (!x || !w_router || !logits) return set_error(MOE_EINVAL, "null pointer");
    if (((uintptr_t)x | (uintptr_t)w_router) % 16 || (uintptr_t)logits % 4 || (uintptr_t)bias % 4)
        return set_error(MOE_EINVAL, "x and w_router must be 16-byte aligned, logits and bias 4-byte aligned");
    MOE_ON_DEVICE(ctx->device);
    return launch_router(x, w_router, bias, T, E, H, logits, ctx->status_dev, ctx->sms, (cudaStream_t)stream);
}

int moe_swap_rows(moe_ctx *ctx, int layer, int n, const int32_t *promote, const int32_t *demote,
                  int32_t *applied, void *stream) {
    if (int r = check_layer(ctx, layer, true)) return r;
    if (n < 0 || (n > 0 && (!promote || !demote))) return set_error(MOE_EINVAL, "bad swap list");
    MOE_ON_DEVICE(ctx->device);
    cudaStream_t s = (cudaStream_t)stream;
    Layer &L = ctx->layers[layer];
    const Geom &g = ctx->g;
    int done = 0;
    if (applied)
        for (int i = 0; i < n; ++i) applied[i] = 0;
    // Applied pairs alternate between two staging rows.  Pair k: hot row ->
    // staging[k % 2] and cold row -> hot slot on `stream`; staging -> cold
    // slot on the swap stream, after those two (so it overlaps pair k+1's
    // copy into HBM: the host link carries both directions at once).  Pair
    // k's row-map write goes on `stream` once its copy back has landed:
    // before pair k+2 reuses its staging row, or at the end.
    struct Pending {
        int32_t c, hot_row, h, cold_row;
    };
    Pending pend[2];
    int npend = 0;   // pairs whose copy back is not yet joined (the last one or two)
    int32_t last_cold = -1;
    auto fail = [&](int r) {
        L.init = false;
        return set_error(r, std::string(moe_last_error()) + "; layer " + std::to_string(layer) +
                                " must be placed again with moe_init_banks");
    };
    // join the oldest pending pair: wait for its copy back, then write its two map entries
    auto join_oldest = [&]() -> int {
        const Pending q = pend[0];
        const int buf = (done - npend) % 2;
        cudaError_t e = cudaStreamWaitEvent(s, ctx->swap_out[buf], 0);
        if (e != cudaSuccess) return cuda_error(e, "moe_swap_rows join");
        if (int r = launch_rowmap_write(L.rowmap_dev, q.c, q.hot_row, q.h, -1 - q.cold_row, s)) return r;
        pend[0] = pend[1];
        --npend;
        return MOE_OK;
    };
    for (int i = 0; i < n; ++i) {
        int32_t c = promote[i], h = demote[i];
        bool ok = c >= 0 && c < g.E && h >= 0 && h < g.E && c != h && L.rowmap[c] < 0 && L.rowmap[h] >= 0;
        if (!ok) continue;
        int32_t hot_row = L.rowmap[h];
        int32_t cold_row = -1 - L.rowmap[c];
        uint8_t *hot_p = L.hot + (size_t)hot_row * g.eb;
        uint8_t *cold_p = L.cold_host + (size_t)cold_row * g.eb;
        const int buf = done % 2;
        uint8_t *stage = ctx->staging + (size_t)buf * g.eb;
        // this staging row's previous pair must be joined first; so must the
        // pair before whose copy back still writes the cold row read here
        if (npend == 2)
            if (int r = join_oldest()) return fail(r);
        if (npend == 1 && pend[0].cold_row == cold_row)
            if (int r = join_oldest()) return fail(r);
        // A failure after the first copy may leave a bank row holding neither
        // expert whole: the layer is then marked as needing moe_init_banks,
        // and this pair is not reported as applied.
        cudaError_t e = cudaMemcpyAsync(stage, hot_p, g.eb, cudaMemcpyDeviceToDevice, s);
        if (e == cudaSuccess) e = cudaMemcpyAsync(hot_p, cold_p, g.eb, cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess) e = cudaEventRecord(ctx->swap_in[buf], s);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(ctx->swap_stream, ctx->swap_in[buf], 0);
        if (e == cudaSuccess) e = cudaMemcpyAsync(cold_p, stage, g.eb, cudaMemcpyDeviceToHost, ctx->swap_stream);
        if (e == cudaSuccess) e = cudaEventRecord(ctx->swap_out[buf], ctx->swap_stream);
        if (e != cudaSuccess) return fail(cuda_error(e, "moe_swap_rows copy"));
        pend[npend++] = Pending{c, hot_row, h, cold_row};
        L.rowmap[c] = hot_row;
        L.rowmap[h] = -1 - cold_row;
        if (applied) applied[i] = 1;
        ++done;
    }
    while (npend > 0)
        if (int r = join_oldest()) return fail(r);
    return done;
}

int moe_read_counts(moe_ctx *ctx, int32_t *host_out, void *stream) {
    if (int r = check_ctx(ctx)) return r;
    if (!host_out) return set_error(MOE_EINVAL, "null output");
    MOE_ON_DEVICE(ctx->device);
    cudaStream_t s = (cudaStream_t)stream;
    MOE_CUDA_TRY(cudaMemcpyAsync(host_out, ctx->counts_dev, sizeof(int32_t) * ctx->g.L * ctx->g.E,
                                 cudaMemcpyDeviceToHost, s));
    MOE_CUDA_TRY(cudaStreamSynchronize(s));
    return MOE_OK;
}

int moe_reset_counts(moe_ctx *ctx, void *stream) {
    if (int r = check_ctx(ctx)) return r;
    MOE_ON_DEVICE(ctx->device);
    MOE_CUDA_TRY(cudaMemsetAsync(ctx->counts_dev, 0, sizeof(int32_t) * ctx->g.L * ctx->g.E, (cudaStream_t)stream));
    return MOE_OK;
}

int moe_bank_rows(moe_ctx *ctx, int layer, int32_t *n_hot, int32_t *n_cold) {
    if (int r = check_layer(ctx, layer, true)) return r;
    if (n_hot) *n_hot = ctx->layers[layer].n_hot;
    if (n_cold) *n_cold = ctx->layers[layer].n_cold;
    return MOE_OK;
}

int moe_get_rowmap(moe_ctx *ctx, int layer, int32_t *host_out) {
    if (int r = check_layer(ctx, layer, true)) return r;
    if (!host_out) return set_error(MOE_EINVAL, "null output");
    std::memcpy(host_out, ctx->layers[layer].rowmap.data(), sizeof(int32_t) * ctx->g.E);
    return MOE_OK;
}

int moe_read_rowmap_device(moe_ctx *ctx, int layer, int32_t *host_out, void *stream) {
    if (int r = check_layer(ctx, layer, true)) return r;
    if (!host_out) return set_error(MOE_EINVAL, "null output");
    MOE_ON_DEVICE(ctx->device);
    cudaStream_t s = (cudaStream_t)stream;
    MOE_CUDA_TRY(cudaMemcpyAsync(host_out, ctx->layers[layer].rowmap_dev, sizeof(int32_t) * ctx->g.E,
                                 cudaMemcpyDeviceToHost, s));
    MOE_CUDA_TRY(cudaStreamSynchronize(s));
    return MOE_OK;
}

int moe_read_bank_row(moe_ctx *ctx, int layer, int bank, int row, uint8_t *host_out, void *stream) {
    if (int r = check_layer(ctx, layer, true)) return r;
    Layer &L = ctx->layers[layer];
    int rows = bank == MOE_BANK_HOT ? L.n_hot : (bank == MOE_BANK_COLD ? L.n_cold : -1);
    if (row < 0 || row >= rows || !host_out) return set_error(MOE_EINVAL, "bank/row out of range");
    MOE_ON_DEVICE(ctx->device);
    cudaStream_t s = (cudaStream_t)stream;
    MOE_CUDA_TRY(cudaStreamSynchronize(s));
    if (bank == MOE_BANK_HOT) {
        MOE_CUDA_TRY(cudaMemcpyAsync(host_out, L.hot + (size_t)row * ctx->g.eb, ctx->g.eb, cudaMemcpyDeviceToHost, s));
        MOE_CUDA_TRY(cudaStreamSynchronize(s));
    } else {
        std::memcpy(host_out, L.cold_host + (size_t)row * ctx->g.eb, ctx->g.eb);
    }
    return MOE_OK;
}

int moe_probe_link(moe_ctx *ctx, size_t bytes, int iters, double *gbps, double *hbm_gbps) {
    if (int r = check_ctx(ctx)) return r;
    if (!gbps || bytes < (1 << 20) || iters < 1) return set_error(MOE_EINVAL, "bad probe arguments");
    bytes &= ~size_t(4095);
    MOE_ON_DEVICE(ctx->device);
    if (ctx->probe_bytes < bytes) {
        pinned_free(ctx->probe_host);
        dev_free(ctx->probe_dev);
        ctx->probe_host = nullptr;
        ctx->probe_dev = nullptr;
        ctx->probe_bytes = 0;
        MOE_CUDA_TRY(pinned_alloc((void **)&ctx->probe_host, bytes, cudaHostAllocMapped | cudaHostAllocPortable, "probe"));
        std::memset(ctx->probe_host, 0x5A, bytes);
        MOE_CUDA_TRY(dev_alloc((void **)&ctx->probe_dev, bytes, "probe"));
        MOE_CUDA_TRY(cudaMemset(ctx->probe_dev, 0x5A, bytes));
        ctx->probe_bytes = bytes;
    }
    uint8_t *host_dev = nullptr;
    MOE_CUDA_TRY(cudaHostGetDevicePointer((void **)&host_dev, ctx->probe_host, 0));
    uint64_t *sink = nullptr;
    MOE_CUDA_TRY(dev_alloc((void **)&sink, sizeof(uint64_t) * 65536, "probe"));
    cudaEvent_t a, b;
    cudaEventCreate(&a);
    cudaEventCreate(&b);
    int blocks = ctx->sms * 8;
    auto measure = [&](const uint8_t *src, double *best) -> int {
        *best = 0.0;
        for (int it = 0; it < iters + 1; ++it) {
            cudaEventRecord(a, 0);
            if (int r = launch_probe_read(src, bytes, sink, blocks, 0)) return r;
            cudaEventRecord(b, 0);
            MOE_CUDA_TRY(cudaEventSynchronize(b));
            float ms = 0.f;
            cudaEventElapsedTime(&ms, a, b);
            if (it > 0) *best = std::max(*best, (double)bytes / (ms * 1e-3) / 1e9);
        }
        return MOE_OK;
    };
    int r = measure(host_dev, gbps);
    if (!r && hbm_gbps) r = measure(ctx->probe_dev, hbm_gbps);
    cudaEventDestroy(a);
    cudaEventDestroy(b);
    dev_free(sink);
    return r;
}

int moe_device_status(moe_ctx *ctx, int32_t *status) {
    if (int r = check_ctx(ctx)) return r;
    MOE_ON_DEVICE(ctx->device);
    int32_t v[4] = {0, 0, 0, 0};
    MOE_CUDA_TRY(cudaDeviceSynchronize());
    MOE_CUDA_TRY(cudaMemcpy(v, ctx->status_dev, sizeof v, cudaMemcpyDeviceToHost));
    MOE_CUDA_TRY(cudaMemset(ctx->status_dev, 0, sizeof v));
    if (status) *status = v[0];
    return MOE_OK;
}

int64_t moe_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

int moe_memory_in_use(int64_t *device_bytes, int64_t *pinned_bytes) {
    std::lock_guard<std::mutex> lock(g_mem_mu);
    if (device_bytes) *device_bytes = g_mem_bytes[0];
    if (pinned_bytes) *pinned_bytes = g_mem_bytes[1];
    return MOE_OK;
}

int moe_set_wait_limit(moe_ctx *ctx, uint64_t ns) {
    if (int r = check_ctx(ctx)) return r;
    ctx->wait_ns = ns ? ns : kDefaultWaitNs;
    return MOE_OK;
}

int moe_inject_fault(moe_ctx *ctx, int kind) {
    if (int r = check_ctx(ctx)) return r;
    if (kind != MOE_FAULT_NONE && kind != MOE_FAULT_WITHHOLD_COPY) return set_error(MOE_EINVAL, "unknown fault kind");
    ctx->inject_withhold = kind == MOE_FAULT_WITHHOLD_COPY;
    return MOE_OK;
}

}  // extern "C"
