// Expert-record checksums on the device: CRC-32 of each record's payload.
//
// The pages check every expert record's header on read and offer an opt-in
// CRC of the payload (a few percent of a read from disk) [GeekNews topic
// 32035, section "Disk streaming structure"].  The variant is not named; this
// is the common CRC-32 (ISO-HDLC): reflected polynomial 0xEDB88320, register
// preset to all ones, result complemented, over bytes [128, record_bytes) of
// each record (everything after the header, alignment padding included).
//
// GPU form: one block per record, each thread takes the CRC of one contiguous
// segment with a zero register (slice-by-4 tables in shared memory, 16-byte
// loads).  CRC arithmetic is linear over GF(2): the register after A || B is
// reg(A) * x^(8|B|) + reg(B) (mod the polynomial), and a preset P adds
// P * x^(8 n).  So each segment's register is multiplied by x^(8 * bytes after
// it) -- a product of precomputed x^(8 * 2^j) factors -- and the block XORs
// them together.
#include "internal.cuh"

namespace rvq {
namespace {

constexpr int CRC_NT = 512;
constexpr uint32_t kCrcPoly = 0xEDB88320u;
constexpr uint32_t kHdrCrcOffset = 28;  // rvq_expert_header.crc32
constexpr uint32_t kHdrFlagsOffset = 24;

// x^(8 * 2^j) mod P in the reflected representation (bit 31 - i holds the
// coefficient of x^i), j = 0..31.
__constant__ uint32_t c_xpow[32];

// a * b mod P, reflected: Horner over a's coefficients from x^31 (bit 0) down.
__host__ __device__ inline uint32_t gf2_mulmod(uint32_t a, uint32_t b) {
    uint32_t p = 0;
    for (int i = 0; i < 32; ++i) {
        p = (p >> 1) ^ ((p & 1u) ? kCrcPoly : 0u);  // p * x
        if ((a >> i) & 1u) p ^= b;
    }
    return p;
}

// reg * x^(8 n) mod P
__device__ inline uint32_t crc_shift(uint32_t reg, uint64_t n) {
    for (int j = 0; n != 0 && j < 32; ++j, n >>= 1)
        if (n & 1u) reg = gf2_mulmod(reg, c_xpow[j]);
    return reg;
}

// mode 0: verify (crc_out[e] = computed; a sealed header with another value
// sets RVQ_DEV_ERR_CORRUPT); mode 1: seal (header crc32 = computed, flag set).
__global__ void __launch_bounds__(CRC_NT) record_crc_kernel(uint8_t *base, uint64_t record_bytes,
                                                            int mode, uint32_t *crc_out,
                                                            uint32_t *status) {
    __shared__ uint32_t T[4][256];
    __shared__ uint32_t red[CRC_NT / 32];
    for (int i = threadIdx.x; i < 256; i += CRC_NT) {
        uint32_t c = (uint32_t)i;
        for (int b = 0; b < 8; ++b) c = (c >> 1) ^ ((c & 1u) ? kCrcPoly : 0u);
        T[0][i] = c;
    }
    __syncthreads();
    for (int k = 1; k < 4; ++k) {
        for (int i = threadIdx.x; i < 256; i += CRC_NT)
            T[k][i] = (T[k - 1][i] >> 8) ^ T[0][T[k - 1][i] & 0xFFu];
        __syncthreads();
    }
    const int e = blockIdx.x;
    uint8_t *rec = base + (uint64_t)e * record_bytes;
    const uint8_t *p = rec + 128;
    const uint64_t len = record_bytes - 128;
    // this thread's segment, 16-byte multiples (the last one ends at len)
    const uint64_t seg = ((len + CRC_NT - 1) / CRC_NT + 15) & ~(uint64_t)15;
    const uint64_t s0 = min(len, (uint64_t)threadIdx.x * seg), s1 = min(len, s0 + seg);
    uint32_t c = 0;
    auto word = [&](uint32_t w) {
        c ^= w;
        c = T[3][c & 0xFFu] ^ T[2][(c >> 8) & 0xFFu] ^ T[1][(c >> 16) & 0xFFu] ^ T[0][c >> 24];
    };
    uint64_t q = s0;
    for (; q + 16 <= s1; q += 16) {
        const uint4 v = __ldg(reinterpret_cast<const uint4 *>(p + q));
        word(v.x);
        word(v.y);
        word(v.z);
        word(v.w);
    }
    for (; q < s1; ++q) c = T[0][(c ^ p[q]) & 0xFFu] ^ (c >> 8);
    c = crc_shift(c, len - s1);
    for (int o = 16; o > 0; o >>= 1) c ^= __shfl_xor_sync(0xffffffffu, c, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = c;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t r = 0;
        for (int w = 0; w < CRC_NT / 32; ++w) r ^= red[w];
        const uint32_t crc = ~(r ^ crc_shift(0xFFFFFFFFu, len));
        uint32_t *hcrc = reinterpret_cast<uint32_t *>(rec + kHdrCrcOffset);
        uint32_t *hflags = reinterpret_cast<uint32_t *>(rec + kHdrFlagsOffset);
        if (mode == 1) {
            *hcrc = crc;
            *hflags |= RVQ_HDR_FLAG_CRC32;
        } else {
            if (crc_out) crc_out[e] = crc;
            if ((*hflags & RVQ_HDR_FLAG_CRC32) && *hcrc != crc)
                set_dev_error(status, RVQ_DEV_ERR_CORRUPT);
        }
    }
}

}  // namespace

rvq_status launch_record_crc(uint8_t *base, uint64_t record_bytes, int n_records, int mode,
                             uint32_t *crc_out, uint32_t *status, cudaStream_t stream) {
    static std::atomic<int> table_done[64];  // per device; copying twice is harmless
    int dev = 0;
    RVQ_CUDA(cudaGetDevice(&dev));
    if (dev >= 64 || !table_done[dev]) {
        uint32_t xp[32];
        xp[0] = 1u << (31 - 8);  // x^8
        for (int j = 1; j < 32; ++j) xp[j] = gf2_mulmod(xp[j - 1], xp[j - 1]);
        RVQ_CUDA(cudaMemcpyToSymbol(c_xpow, xp, sizeof(xp)));
        if (dev < 64) table_done[dev] = 1;
    }
    if (n_records <= 0) return RVQ_OK;
    record_crc_kernel<<<n_records, CRC_NT, 0, stream>>>(base, record_bytes, mode, crc_out, status);
    RVQ_LAUNCHED("record_crc");
    return RVQ_OK;
}

}  // namespace rvq
