// Allocation-free variant of the expert-FFN entry point.
//
// moe_expert_ffn_bank keeps its intermediate rows (the token rows as e4m3
// pieces, the gate/up output and its pieces, fp32 partial-sum rows of
// decode-sized steps, the scheduler counters) in a workspace the
// caller allocates.  Some callers cannot allocate device memory at all: a
// plugin handed a fixed memory budget by its host framework, or a serving
// loop that must not call cudaMalloc because the call can synchronize the
// device and can fail under memory pressure.  For them this file keeps one
// scratch area in a file-scope __device__ array, which every GPU that loads
// the library holds from module load until the process exits.
//
// The entry point copies the routed step's pick lists from the caller's
// workspace into the front of that area (a device-to-device copy, not an
// allocation) and runs the same FFN kernels with the area as their
// workspace, so its output equals moe_expert_ffn_bank's.
#include "moe_internal.cuh"

#include <mutex>

namespace moe {
namespace {

constexpr size_t kStaticScratchBytes = 16u << 20;   // 16 MiB

static __device__ __align__(256) uint8_t g_ffn_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
uint8_t *g_scratch_ptr[kMaxDevices] = {};

// Device address of this device's copy of g_ffn_scratch.  The host-side name
// of the array is only a stand-in, so the address is looked up once per
// device, with that device current.
int scratch_for_device(int device, uint8_t **out) {
    if (device < 0 || device >= kMaxDevices) return set_error(MOE_EINVAL, "device index out of range");
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[device]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_ffn_scratch);
        if (e != cudaSuccess) return cuda_error(e, "cudaGetSymbolAddress(static FFN scratch)");
        g_scratch_ptr[device] = (uint8_t *)p;
    }
    *out = g_scratch_ptr[device];
    return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

size_t moe_static_scratch_bytes(void) { return kStaticScratchBytes; }

int moe_expert_ffn_bank_static(moe_ctx *ctx, int layer, int bank, const uint16_t *x, int T, const void *split_ws,
                               uint16_t *Y, void *stream) {
    if (int r = check_layer(ctx, layer, true)) return r;
    if (bank != MOE_BANK_HOT && bank != MOE_BANK_COLD && bank != MOE_BANK_BOTH)
        return set_error(MOE_EINVAL, "bank must be 0, 1 or 2");
    if (T < 0 || T > ctx->g.Tmax) return set_error(MOE_EINVAL, "T out of range");
    if (!split_ws || (uintptr_t)split_ws % 256) return set_error(MOE_EINVAL, "split workspace must be non-null and 256-byte aligned");
    if (T > 0 && (!x || !Y)) return set_error(MOE_EINVAL, "null pointer");
    if (((uintptr_t)x | (uintptr_t)Y) % 16) return set_error(MOE_EINVAL, "x and Y must be 16-byte aligned");
    const WsLayout lay = ws_layout(ctx->g, T);
    if (lay.total > kStaticScratchBytes)
        return set_error(MOE_EINVAL, "step needs " + std::to_string(lay.total) + " bytes of FFN scratch; the static area holds " +
                                         std::to_string(kStaticScratchBytes));
    Layer &L = ctx->layers[layer];
    if (bank == MOE_BANK_BOTH && (L.n_hot == 0 || L.n_cold == 0)) bank = L.n_hot ? MOE_BANK_HOT : MOE_BANK_COLD;
    const int rows = bank == MOE_BANK_HOT ? L.n_hot : (bank == MOE_BANK_COLD ? L.n_cold : L.n_hot + L.n_cold);
    if (T == 0 || rows == 0) return MOE_OK;

    MOE_ON_DEVICE(ctx->device);
    uint8_t *scratch = nullptr;
    if (int r = scratch_for_device(ctx->device, &scratch)) return r;
    cudaStream_t s = (cudaStream_t)stream;
    // the pick lists are the front of the workspace (header, rows, offsets, picks, positions)
    MOE_CUDA_TRY(cudaMemcpyAsync(scratch, split_ws, lay.xq, cudaMemcpyDeviceToDevice, s));
    if (ctx->ffn_impl == MOE_FFN_SIMT) {
        for (int bk = 0; bk < 2; ++bk)
            if (bank == MOE_BANK_BOTH || bank == bk)
                if (int r = launch_ffn_simt(ctx, bk == MOE_BANK_HOT ? L.hot : L.cold_dev, bk, x, T, scratch, Y, s))
                    return r;
        return MOE_OK;
    }
    return launch_ffn_tc(ctx, L, bank, x, T, scratch, Y, s);
}

}  // extern "C"
