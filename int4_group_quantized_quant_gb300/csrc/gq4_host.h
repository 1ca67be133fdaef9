// gq4_host.h -- small host-side helpers shared by the launchers: integer
// arithmetic for the shared-memory plans and, for the tensor-core kernels,
// the driver's tensor-map encoder and the scale groups a K stage spans.
#pragma once

#include <cuda.h>

#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

namespace gq4 {

inline int gcd_int(int a, int b)
{
    while (b) {
        const int t = a % b;
        a = b;
        b = t;
    }
    return a;
}

inline uint32_t round_up(uint32_t x, uint32_t a)
{
    return (x + a - 1) / a * a;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against libcuda); nullptr when the driver does not provide it.
inline EncodeTiledFn encode_tiled_fn()
{
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, []() {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    });
    return fn;
}

// Most scale groups one stage of `stage_k` codes (starting at a multiple of
// stage_k) spans, counted without clipping at K, so every K-block of a stage
// -- including those past K in the last stage -- finds its constant row in
// the stage.
inline int groups_per_stage(int gs, int stage_k)
{
    int most = 1;
    for (int k0 = 0; k0 < stage_k * gs; k0 += stage_k) {
        const int g = (k0 + stage_k - 1) / gs - k0 / gs + 1;
        most = g > most ? g : most;
        if (k0 % gs == 0 && k0 > 0) break;  // the pattern repeats
    }
    return most;
}

}  // namespace gq4
