// Finalize and the host-link probe.
//
// Finalize ("vLLM: Pin Hot Experts", Results and the F4 split): every token's
// k bf16 expert rows are accumulated in fp32 with a fused multiply-add in the
// original k order, starting from +0, and cast to bf16 once.  Because the
// order never depends on which bank produced a row, the split layer and any
// row swap give bit-identical outputs.
//
// HBM-bound: reads T*k*H*2 + T*k*4 bytes and writes T*H*2; each thread owns
// eight consecutive columns (16-byte loads and stores).
#include "moe_internal.cuh"

namespace moe {

namespace {

__global__ void __launch_bounds__(256) finalize_kernel(const uint4 *__restrict__ Y,
                                                       const float *__restrict__ w, int T, int k,
                                                       int H8, uint4 *__restrict__ out) {
    const long long n = (long long)T * H8;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x) {
        const int t = (int)(i / H8), c = (int)(i % H8);
        float acc[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
        for (int j = 0; j < k; ++j) {
            const float wj = __ldg(w + (size_t)t * k + j);
            const uint4 v = __ldg(Y + ((size_t)t * k + j) * H8 + c);
            const uint32_t p[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                acc[2 * q] = __fmaf_rn(wj, __uint_as_float(p[q] << 16), acc[2 * q]);
                acc[2 * q + 1] = __fmaf_rn(wj, __uint_as_float(p[q] & 0xFFFF0000u), acc[2 * q + 1]);
            }
        }
        uint32_t o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * q], acc[2 * q + 1]);
            o[q] = *reinterpret_cast<uint32_t *>(&b);
        }
        out[(size_t)t * H8 + c] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// Streams `bytes` from src with 16-byte loads; folds them into a sink so the
// loads are not removed.
__global__ void __launch_bounds__(256) probe_read_kernel(const uint4 *__restrict__ src, size_t n16,
                                                         uint64_t *sink) {
    uint32_t acc = 0;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
    for (; i + 3 * stride < n16; i += 4 * stride) {
        uint4 a = __ldcs(src + i), b = __ldcs(src + i + stride);
        uint4 c = __ldcs(src + i + 2 * stride), d = __ldcs(src + i + 3 * stride);
        acc ^= a.x ^ a.y ^ a.z ^ a.w ^ b.x ^ b.y ^ b.z ^ b.w ^ c.x ^ c.y ^ c.z ^ c.w ^ d.x ^ d.y ^ d.z ^ d.w;
    }
    for (; i < n16; i += stride) {
        uint4 a = __ldcs(src + i);
        acc ^= a.x ^ a.y ^ a.z ^ a.w;
    }
    if (acc == 0x12345678u) sink[(blockIdx.x * blockDim.x + threadIdx.x) & 65535] = acc;
}

}  // namespace

int launch_finalize(const uint16_t *Y, const float *w, int T, int k, int H, uint16_t *out, cudaStream_t s) {
    const int H8 = H / 8;
    const long long n = (long long)T * H8;
    int blocks = (int)std::min<long long>((n + 255) / 256, 152LL * 8);
    finalize_kernel<<<blocks, 256, 0, s>>>((const uint4 *)Y, w, T, k, H8, (uint4 *)out);
    MOE_LAUNCH_CHECK();
    return MOE_OK;
}

int launch_probe_read(const uint8_t *src, size_t bytes, uint64_t *sink, int blocks, cudaStream_t s) {
    probe_read_kernel<<<blocks, 256, 0, s>>>((const uint4 *)src, bytes / 16, sink);
    MOE_LAUNCH_CHECK();
    return MOE_OK;
}

}  // namespace moe
