// Offline RVQ encoder on the device: residual k-means, one stage at a time.
//
// The pages' converter encodes every expert matrix once, offline, into the
// 3-stage RVQ format (8-dim sub-vectors, 256-entry codebooks) [GeekNews
// topic 32035, sections "Quantization and accuracy" and "Conversion"]; they
// give no algorithm.  This is the plainest residual quantiser: per stage,
// codebook = 256 evenly spaced residual sub-vectors, then `iters` Lloyd
// rounds (nearest codeword, ties to the lower index; each codeword with
// members replaced by their mean), a last assignment for the codes, and the
// residual minus the chosen codewords.
//
// Reproducible by construction:
//  * the nearest codeword is decided in fp32 with the 8 squared differences
//    accumulated by fused multiply-adds in dimension order;
//  * a mean is an int64 fixed-point sum (each value times 2^32, rounded to
//    nearest even) divided by the member count in double: integer atomics
//    make the sum independent of the order the threads add in.  With
//    |w| < 128 every residual stays below 1024 = 2^10, so at most 2^21
//    sub-vectors keep a sum below 2^63.
// Per stage and round: one assignment pass (codebook in shared memory, one
// thread per two sub-vectors, per-block fixed-point partial sums in shared memory,
// one global atomic per block and entry) and one update of the 2048 entries.
#include "internal.cuh"

#include <algorithm>

namespace rvq {
namespace {

constexpr int ENC_NT = 256;
constexpr int ENC_SV = 2;  // sub-vectors per thread in the search

struct EncWs {
    float *R;             // [N][8] residual
    int32_t *a;           // [N] assignment
    unsigned long long *sum;  // [256][8] fixed-point sums
    unsigned long long *cnt;  // [256]
};

__global__ void __launch_bounds__(ENC_NT) enc_init_codebook(const float *__restrict__ R,
                                                            int64_t N, float *__restrict__ C) {
    const int t = blockIdx.x * ENC_NT + threadIdx.x;  // 256 x 8 entries
    if (t >= 256 * 8) return;
    const int k = t >> 3, d = t & 7;
    C[t] = R[((int64_t)k * N / 256) * 8 + d];
}

// One thread per ENC_SV sub-vectors (i, i + ENC_NT, ... of the block's
// ENC_SV x ENC_NT): the nearest codeword of each, and (do_sums) their
// fixed-point sums and counts.  The sub-vectors' distances are independent
// chains that share each codeword load; each chain still accumulates its 8
// squared differences in dimension order.
__global__ void __launch_bounds__(ENC_NT) enc_assign(const float *__restrict__ R, int64_t N,
                                                     const float *__restrict__ C,
                                                     int32_t *__restrict__ a, int do_sums,
                                                     unsigned long long *__restrict__ gsum,
                                                     unsigned long long *__restrict__ gcnt) {
    __shared__ __align__(16) float cb[256 * 8];
    __shared__ unsigned long long ssum[256 * 8];
    __shared__ unsigned long long scnt[256];
    for (int i = threadIdx.x; i < 256 * 8; i += ENC_NT) {
        cb[i] = C[i];
        ssum[i] = 0ull;
    }
    for (int i = threadIdx.x; i < 256; i += ENC_NT) scnt[i] = 0ull;
    __syncthreads();
    for (int64_t i0 = (int64_t)blockIdx.x * ENC_SV * ENC_NT + threadIdx.x; i0 < N;
         i0 += (int64_t)gridDim.x * ENC_SV * ENC_NT) {
        float r[ENC_SV][8];
#pragma unroll
        for (int v = 0; v < ENC_SV; ++v) {
            const int64_t i = i0 + v * ENC_NT;
            const float4 *p = reinterpret_cast<const float4 *>(R + (i < N ? i : i0) * 8);
            const float4 x0 = p[0], x1 = p[1];
            r[v][0] = x0.x; r[v][1] = x0.y; r[v][2] = x0.z; r[v][3] = x0.w;
            r[v][4] = x1.x; r[v][5] = x1.y; r[v][6] = x1.z; r[v][7] = x1.w;
        }
        float bd[ENC_SV], dk[ENC_SV];
        int best[ENC_SV];
        auto dist = [&](int k, float (&dd)[ENC_SV]) {
            const float4 c0 = *reinterpret_cast<const float4 *>(cb + k * 8);
            const float4 c1 = *reinterpret_cast<const float4 *>(cb + k * 8 + 4);
            const float c[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
            for (int v = 0; v < ENC_SV; ++v) dd[v] = 0.f;
#pragma unroll
            for (int d = 0; d < 8; ++d)
#pragma unroll
                for (int v = 0; v < ENC_SV; ++v) {
                    const float t = __fsub_rn(r[v][d], c[d]);
                    dd[v] = __fmaf_rn(t, t, dd[v]);
                }
        };
        dist(0, bd);
#pragma unroll
        for (int v = 0; v < ENC_SV; ++v) best[v] = 0;
#pragma unroll 3
        for (int k = 1; k < 256; ++k) {
            dist(k, dk);
#pragma unroll
            for (int v = 0; v < ENC_SV; ++v)
                if (dk[v] < bd[v]) {
                    bd[v] = dk[v];
                    best[v] = k;
                }
        }
#pragma unroll
        for (int v = 0; v < ENC_SV; ++v) {
            const int64_t i = i0 + v * ENC_NT;
            if (i >= N) continue;
            a[i] = best[v];
            if (do_sums) {
                atomicAdd(&scnt[best[v]], 1ull);
#pragma unroll
                for (int d = 0; d < 8; ++d)
                    atomicAdd(&ssum[best[v] * 8 + d],
                              (unsigned long long)__double2ll_rn((double)r[v][d] * 4294967296.0));
            }
        }
    }
    if (!do_sums) return;
    __syncthreads();
    for (int i = threadIdx.x; i < 256 * 8; i += ENC_NT)
        if (ssum[i] != 0ull) atomicAdd(&gsum[i], ssum[i]);
    for (int i = threadIdx.x; i < 256; i += ENC_NT)
        if (scnt[i] != 0ull) atomicAdd(&gcnt[i], scnt[i]);
}

// Codewords with members become their mean; the sums are cleared for the
// next round.
__global__ void __launch_bounds__(ENC_NT) enc_update(float *__restrict__ C,
                                                     unsigned long long *__restrict__ gsum,
                                                     unsigned long long *__restrict__ gcnt) {
    // launched as 8 x 256 threads: one per entry, the 8 entries of a codeword
    // in one block, so the barrier orders their count reads before the clear
    const int t = blockIdx.x * ENC_NT + threadIdx.x;
    const int k = t >> 3;
    const long long n = (long long)gcnt[k];
    if (n > 0)
        C[t] = (float)(((double)(long long)gsum[t] * (1.0 / 4294967296.0)) / (double)n);
    gsum[t] = 0ull;
    __syncthreads();
    if ((t & 7) == 0) gcnt[k] = 0ull;
}

// codes[i][s] = a[i]; R[i] -= C[a[i]]
__global__ void __launch_bounds__(ENC_NT) enc_finish(float *__restrict__ R, int64_t N,
                                                     const float *__restrict__ C,
                                                     const int32_t *__restrict__ a,
                                                     uint8_t *__restrict__ codes, int s) {
    for (int64_t i = (int64_t)blockIdx.x * ENC_NT + threadIdx.x; i < N;
         i += (int64_t)gridDim.x * ENC_NT) {
        const int k = a[i];
        codes[i * 3 + s] = (uint8_t)k;
#pragma unroll
        for (int d = 0; d < 8; ++d) R[i * 8 + d] = __fsub_rn(R[i * 8 + d], C[k * 8 + d]);
    }
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

size_t encode_workspace_bytes(int rows, int cols) {
    const size_t N = (size_t)rows * (cols / 8);
    return align256(N * 32) + align256(N * 4) + align256(256 * 8 * 8) + align256(256 * 8);
}

rvq_status launch_rvq_encode(const float *w, int rows, int cols, int iters, uint8_t *codes,
                             float *codebooks, void *ws, cudaStream_t stream) {
    const int64_t N = (int64_t)rows * (cols / 8);
    uint8_t *p = (uint8_t *)ws;
    EncWs W;
    W.R = (float *)p;
    p += align256((size_t)N * 32);
    W.a = (int32_t *)p;
    p += align256((size_t)N * 4);
    W.sum = (unsigned long long *)p;
    p += align256(256 * 8 * 8);
    W.cnt = (unsigned long long *)p;
    RVQ_CUDA(cudaMemcpyAsync(W.R, w, (size_t)N * 32, cudaMemcpyDeviceToDevice, stream));
    RVQ_CUDA(cudaMemsetAsync(W.sum, 0, 256 * 8 * 8, stream));
    RVQ_CUDA(cudaMemsetAsync(W.cnt, 0, 256 * 8, stream));
    // one wave of resident blocks (a persistent grid-stride loop)
    int per_sm = 0;
    RVQ_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, enc_assign, ENC_NT, 0));
    const int grid = (int)std::min<int64_t>((N + ENC_SV * ENC_NT - 1) / (ENC_SV * ENC_NT),
                                            (int64_t)std::max(1, per_sm) * num_sms());
    for (int s = 0; s < 3; ++s) {
        float *C = codebooks + (size_t)s * 256 * 8;
        enc_init_codebook<<<8, ENC_NT, 0, stream>>>(W.R, N, C);
        for (int it = 0; it <= iters; ++it) {
            const int sums = it < iters;
            enc_assign<<<grid, ENC_NT, 0, stream>>>(W.R, N, C, W.a, sums, W.sum, W.cnt);
            if (!sums) break;
            enc_update<<<8, ENC_NT, 0, stream>>>(C, W.sum, W.cnt);
        }
        enc_finish<<<grid, ENC_NT, 0, stream>>>(W.R, N, C, W.a, codes, s);
    }
    RVQ_LAUNCHED("rvq_encode");
    return RVQ_OK;
}

}  // namespace rvq
