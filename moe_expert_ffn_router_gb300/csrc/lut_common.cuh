// Lookup-table helpers of the decode GEMV kernels (lut_gemv.cu): code bytes
// -> shared-memory table addresses and fp32 sums.
#pragma once

#include <stdint.h>

#include "internal.cuh"

namespace rvq {

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}
__device__ __forceinline__ uint64_t pk2(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1,%2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ float2 upk2(uint64_t v) {
    float2 r;
    asm("mov.b64 {%0,%1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint32_t word_of(const uint4 &v, int q) {
    return q == 0 ? v.x : q == 1 ? v.y : q == 2 ? v.z : v.w;
}

// One-token lookups of one tile with more independent work in flight: the 16
// lookups of a 16-byte code plane are issued before any is added, and four
// accumulators split the add chain (for warps that cannot rely on other
// warps to hide the shared-memory latency).
__device__ __forceinline__ float tile_lookups1_ilp(const uint4 (&c)[6], const uint32_t (&aux2)[16],
                                                   const uint8_t *lut) {
    uint64_t acc[4] = {0, 0, 0, 0};
#pragma unroll
    for (int s = 0; s < 3; ++s)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float v[16];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint32_t w = word_of(c[s * 2 + h], q);
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    const int t = h * 16 + q * 4 + b;
                    const uint32_t idx = prmt(w, aux2[t >> 1], 0x7600u | (b << 4) | (4 + (t & 1)));
                    v[q * 4 + b] = *reinterpret_cast<const float *>(lut + s * kLutStageBytes + idx);
                }
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                acc[q] = fadd2(acc[q], pk2(v[q * 4], v[q * 4 + 1]));
                acc[q] = fadd2(acc[q], pk2(v[q * 4 + 2], v[q * 4 + 3]));
            }
        }
    const float2 a0 = upk2(fadd2(acc[0], acc[1])), a1 = upk2(fadd2(acc[2], acc[3]));
    return (a0.x + a0.y) + (a1.x + a1.y);
}

}  // namespace rvq
