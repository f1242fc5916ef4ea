// MXFP4 expert FFN on CUDA cores (cross-check implementation).
//
// Same work decomposition and device layout as the tensor-core kernel: a unit
// is (active bank row, 128-row M-tile); thread m of the 128-thread block owns
// tile row m, reads its 32 packed bytes and two e8m0 scales per 64-wide
// K-chunk (two K blocks of the chunk's group), dequantises them exactly to
// fp32 and accumulates up to 8 tokens with fp32 fma in K order.  Phase 1 (gate/up) writes h = silu(g) * u in fp32
// per slot; phase 2 (down) writes the bf16 expert row into Y.
#include "moe_internal.cuh"

namespace moe {

namespace {

constexpr int kTok = 8;   // tokens per pass

__device__ __forceinline__ float e2m1_to_f32(uint32_t c) {
    const uint32_t e = (c >> 1) & 3u, m = c & 1u;
    float mag = e == 0 ? 0.5f * (float)m : (1.0f + 0.5f * (float)m) * (float)(1u << (e - 1));
    return (c & 8u) ? -mag : mag;
}

template <int PHASE>
__global__ void __launch_bounds__(128) ffn_simt_kernel(const uint8_t *__restrict__ bank, int64_t eb,
                                                       PartLayout part, BankLists lists, int b, int k, int H, int I,
                                                       const uint16_t *__restrict__ x,
                                                       const float *__restrict__ h_in,
                                                       float *__restrict__ h_out,
                                                       uint16_t *__restrict__ Y) {
    __shared__ float sx[kTok][kKC];
    const int m = threadIdx.x;
    const int n_act = lists.hdr[kHdrNAct + b];
    const int mt_count = part.tiles, kc = part.kchunks;
    const int units = n_act * mt_count;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
        const int a = u / mt_count, mt = u % mt_count;
        const int row = lists.act_row[a];
        const int p0 = lists.act_off[a], n = lists.act_off[a + 1] - p0;
        const uint8_t *expert = bank + (int64_t)row * eb;
        for (int ng = 0; ng < n; ng += kTok) {
            const int nn = min(kTok, n - ng);
            float acc[kTok];
#pragma unroll
            for (int q = 0; q < kTok; ++q) acc[q] = 0.0f;
            for (int c = 0; c < kc; ++c) {
                __syncthreads();
                for (int idx = m; idx < nn * kKC; idx += blockDim.x) {
                    const int tn = idx / kKC, kk = idx % kKC;
                    const int slot = lists.picks[p0 + ng + tn];
                    float v;
                    if (PHASE == 1) v = __uint_as_float((uint32_t)x[(int64_t)(slot / k) * H + c * kKC + kk] << 16);
                    else v = h_in[(int64_t)slot * I + c * kKC + kk];
                    sx[tn][kk] = v;
                }
                __syncthreads();
                int slot, tidx, kb0, nkb;
                part.group(mt, c >> 1, slot, tidx, kb0, nkb);
                const uint8_t *grp = expert + part.group_off(slot, tidx);
                const int kb = kb0 + 2 * (c & 1);   // the chunk's first K block in its group
                const uint4 q[2] = {*(const uint4 *)(grp + m * 64 + kb * 16), *(const uint4 *)(grp + m * 64 + kb * 16 + 16)};
                const uint8_t *sa = grp + kGroupQBytes + (m % 32) * 16 + 4 * (m / 32) + kb;
                const float sc[2] = {ldexpf(1.0f, (int)sa[0] - 127), ldexpf(1.0f, (int)sa[1] - 127)};
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const uint32_t wd[4] = {q[hh].x, q[hh].y, q[hh].z, q[hh].w};
#pragma unroll
                    for (int wi = 0; wi < 4; ++wi) {
#pragma unroll
                        for (int ni = 0; ni < 8; ++ni) {
                            const int kk = hh * 32 + wi * 8 + ni;
                            const int sh = 4 * ni;   // element 2i in the low nibble of byte i
                            const float wv = e2m1_to_f32((wd[wi] >> sh) & 15u) * sc[hh];
#pragma unroll
                            for (int tn = 0; tn < kTok; ++tn)
                                if (tn < nn) acc[tn] = __fmaf_rn(wv, sx[tn][kk], acc[tn]);
                        }
                    }
                }
            }
            // epilogue
            const int w = m >> 5, l = m & 31;
#pragma unroll
            for (int tn = 0; tn < kTok; ++tn) {
                const float other = __shfl_xor_sync(0xffffffffu, acc[tn], 16);
                if (tn < nn) {
                    const int slot = lists.picks[p0 + ng + tn];
                    if (PHASE == 1) {
                        if (l < 16) {
                            const float g = acc[tn], uu = other;
                            const float hv = __fmul_rn(__fdiv_rn(g, 1.0f + expf(-g)), uu);
                            h_out[(int64_t)slot * I + 64 * mt + 16 * w + l] = hv;
                        }
                    } else {
                        Y[(int64_t)slot * H + kMT * mt + m] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[tn]));
                    }
                }
            }
        }
    }
}

}  // namespace

int launch_ffn_simt(moe_ctx *ctx, const uint8_t *bank, int b, const uint16_t *x, int T, uint8_t *ws,
                    uint16_t *Y, cudaStream_t s) {
    const Geom &g = ctx->g;
    WsLayout lay = ws_layout(g, T);
    const int P = T * g.k;
    BankLists lists;
    lists.hdr = (const int32_t *)(ws + lay.hdr);
    lists.act_row = (const int32_t *)(ws + lay.act_row) + (size_t)b * P;
    lists.act_off = (const int32_t *)(ws + lay.act_off) + (size_t)b * (P + 1);
    lists.picks = (const int32_t *)(ws + lay.picks) + (size_t)b * P;
    float *h32 = (float *)(ws + lay.h32);
    const int max_rows = P;   // active rows never exceed the picks
    int blocks1 = (int)std::min<long long>((long long)max_rows * g.mt13, (long long)ctx->sms * 8);
    ffn_simt_kernel<1><<<blocks1, 128, 0, s>>>(bank, g.eb, g.w13, lists, b, g.k, g.H, g.I, x,
                                               nullptr, h32, nullptr);
    MOE_LAUNCH_CHECK();
    int blocks2 = (int)std::min<long long>((long long)max_rows * g.mt2, (long long)ctx->sms * 8);
    ffn_simt_kernel<2><<<blocks2, 128, 0, s>>>(bank, g.eb, g.w2, lists, b, g.k, g.H, g.I,
                                               nullptr, h32, nullptr, Y);
    MOE_LAUNCH_CHECK();
    return MOE_OK;
}

}  // namespace moe
