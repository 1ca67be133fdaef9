// gq4_embed.cu -- int4 embedding gather (gq4_embedding).
//
// The decode step's first dispatch (EmbeddingInt4) and the executor's
// per-layer-embedding stream gather the rows of an int4 table for the step's
// token ids and dequantize them: the table is V rows of width K in the
// matvec's format (row v owns K/8 words and K/gs scale/zero groups), and
//   out[t][k] = fl(fl(q(ids[t], k) - zero) * scale)
// one binary32 rounding per operation, as the dequant test kernel.  An id
// outside [0, V) gives a NaN row and sets device error bit 4 (no table
// access is made for it).
//
// Work item = one 1024-element segment of one output row, taken by one
// warp: lane l writes float4 i*32 + l of the segment (i = 0..7), so every
// store instruction writes 512 contiguous bytes.  A float4 covers 4 codes,
// half of one packed word and always inside one scale group.  The kernel is
// bound by HBM (or L2) writes: 4 bytes out per 0.5 + 8/gs bytes in.
#include <cstdint>

#include "gq4_device.cuh"
#include "gq4_internal.h"

namespace gq4 {
namespace {

__device__ unsigned int g_embed_error = 0;
constexpr unsigned int kEmbedBadId = 1u << 4;

constexpr int kEmbedThreads = 256;
constexpr int kSegFloat4 = 256;  // float4 per work item (1024 elements)

struct EmbedParams {
    const int32_t *ids;
    const uint32_t *Bq;
    const float *scales;
    const float *zeros;
    float4 *out;
    unsigned long long group_magic;  // ceil(2^40 / (gs / 32))
    long long n_items;               // T * segs
    int K, V, G, segs;               // segs = ceil((K / 4) / 256)
};

__global__ void __launch_bounds__(kEmbedThreads) embedding_kernel(EmbedParams p)
{
    const int lane = threadIdx.x & 31;
    const long long warp0 = ((long long)blockIdx.x * kEmbedThreads + threadIdx.x) >> 5;
    const long long n_warps = ((long long)gridDim.x * kEmbedThreads) >> 5;
    const int row_f4 = p.K >> 2;
    for (long long item = warp0; item < p.n_items; item += n_warps) {
        const long long t = item / p.segs;
        const int seg = (int)(item - t * p.segs);
        const int v = __ldg(p.ids + t);  // uniform across the warp
        float4 *orow = p.out + t * (long long)row_f4;
        const int f0 = seg * kSegFloat4;
        if (v < 0 || v >= p.V) {
            const float nan = __int_as_float(0x7fc00000);
#pragma unroll
            for (int i = 0; i < kSegFloat4 / 32; ++i) {
                const int f = f0 + i * 32 + lane;
                if (f < row_f4) orow[f] = make_float4(nan, nan, nan, nan);
            }
            if (lane == 0) atomicOr(&g_embed_error, kEmbedBadId);
            continue;
        }
        const uint32_t *wrow = p.Bq + (long long)v * (p.K >> 3);
        const float *srow = p.scales + (long long)v * p.G;
        const float *zrow = p.zeros + (long long)v * p.G;
        // all loads of the segment first
        uint32_t w[kSegFloat4 / 32];
        float s[kSegFloat4 / 32], z[kSegFloat4 / 32];
#pragma unroll
        for (int i = 0; i < kSegFloat4 / 32; ++i) {
            const int f = f0 + i * 32 + lane;
            if (f < row_f4) {
                const int g = chunk_group(f >> 3, p.group_magic);  // 8 float4 per 32-code chunk
                w[i] = __ldg(wrow + (f >> 1));
                s[i] = __ldg(srow + g);
                z[i] = __ldg(zrow + g);
            }
        }
#pragma unroll
        for (int i = 0; i < kSegFloat4 / 32; ++i) {
            const int f = f0 + i * 32 + lane;
            if (f >= row_f4) break;
            const uint32_t h = w[i] >> (16 * (f & 1));  // this float4's 4 codes
            float4 o;
            o.x = __fmul_rn(__fsub_rn((float)(h & 0xFu), z[i]), s[i]);
            o.y = __fmul_rn(__fsub_rn((float)((h >> 4) & 0xFu), z[i]), s[i]);
            o.z = __fmul_rn(__fsub_rn((float)((h >> 8) & 0xFu), z[i]), s[i]);
            o.w = __fmul_rn(__fsub_rn((float)((h >> 12) & 0xFu), z[i]), s[i]);
            orow[f] = o;
        }
    }
}

}  // namespace

cudaError_t launch_embedding(int T, int K, int V, int gs, const int32_t *ids, const uint32_t *Bq,
                             const float *scales, const float *zeros, float *out,
                             cudaStream_t stream)
{
    static const int resident = [] {
        int b = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, embedding_kernel, kEmbedThreads, 0) !=
            cudaSuccess)
            return 1;
        return b > 0 ? b : 1;
    }();
    int dev = 0, sms = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
    EmbedParams p{};
    p.ids = ids;
    p.Bq = Bq;
    p.scales = scales;
    p.zeros = zeros;
    p.out = reinterpret_cast<float4 *>(out);
    const unsigned long long cpg = (unsigned long long)(gs / 32);
    p.group_magic = ((1ull << 40) + cpg - 1) / cpg;
    p.K = K;
    p.V = V;
    p.G = K / gs;
    p.segs = (K / 4 + kSegFloat4 - 1) / kSegFloat4;
    p.n_items = (long long)T * p.segs;
    const long long warps_per_block = kEmbedThreads / 32;
    const long long want = (p.n_items + warps_per_block - 1) / warps_per_block;
    const long long cap = (long long)sms * resident;
    const unsigned grid = (unsigned)(want < cap ? want : cap);
    embedding_kernel<<<grid, kEmbedThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t read_embed_device_error(unsigned int *bits, bool clear)
{
    cudaError_t err = cudaMemcpyFromSymbol(bits, g_embed_error, sizeof(unsigned int));
    if (err != cudaSuccess || !clear) return err;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_embed_error, &zero, sizeof(unsigned int));
}

}  // namespace gq4
