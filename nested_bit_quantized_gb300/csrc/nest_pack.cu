// Packing of codes and scales into the unit storage format, and its inverse.
// Storage: feedman.me/posts/wZBTJ, POC recipe step 2 (2-bit base, one fp16
// scale per 128 weights) and step 3 (b-bit residual, one fp16 scale per
// (row, 128-group)); base and residual in separate buffers (BitNest,
// section 3.3).  The bit layout is the one the GEMM decoder reads; it is
// spelled out in include/nest.h.
#include "nest_device.cuh"
#include "nest_internal.h"

namespace nest {
namespace {

__device__ __forceinline__ size_t word_off(int r, int w) {
    return ((size_t)(w >> 2) * kRows + r) * 16 + (size_t)(w & 3) * 4;
}

// one thread per (unit, row, code word)
__global__ void k_pack_base(const uint8_t* __restrict__ codes, const uint16_t* __restrict__ scales,
                            int M, int K, long long n_items, uint8_t* __restrict__ out) {
    const int G = K / kGroup;
    for (long long it = blockIdx.x * (long long)blockDim.x + threadIdx.x; it < n_items;
         it += (long long)gridDim.x * blockDim.x) {
        const int w = (int)(it & 7);
        const int r = (int)((it >> 3) & 127);
        const long long unit = it >> 10;
        const int tile = (int)(unit / G), g = (int)(unit % G);
        const int m = tile * kRows + r;
        uint8_t* u = out + unit * kBaseUnit;
        uint32_t word = 0;
        if (m < M) {
            const uint8_t* c = codes + (size_t)m * K + (size_t)g * kGroup + 16 * w;
#pragma unroll
            for (int j = 0; j < 16; ++j) word |= (uint32_t)(c[j] & 3u) << (8 * (j & 3) + 2 * (j >> 2));
        }
        *reinterpret_cast<uint32_t*>(u + word_off(r, w)) = word;
        if (w == 0) *reinterpret_cast<uint16_t*>(u + 4096 + 2 * r) = m < M ? scales[(size_t)m * G + g] : (uint16_t)0;
    }
}

// one thread per (unit, row, residual word)
__global__ void k_pack_resid(const int8_t* __restrict__ codes, const uint16_t* __restrict__ scales,
                             int M, int K, int bits, long long n_items, uint8_t* __restrict__ out) {
    const int G = K / kGroup;
    const int wpr = 4 * bits;                 // words per row
    const int off = 1 << (bits - 1);
    const size_t ub = (size_t)resid_unit_bytes(bits);
    for (long long it = blockIdx.x * (long long)blockDim.x + threadIdx.x; it < n_items;
         it += (long long)gridDim.x * blockDim.x) {
        const int w = (int)(it % wpr);
        const int r = (int)((it / wpr) % kRows);
        const long long unit = it / ((long long)wpr * kRows);
        const int tile = (int)(unit / G), g = (int)(unit % G);
        const int m = tile * kRows + r;
        const bool valid = m < M;
        const int8_t* c = codes + (size_t)(valid ? m : 0) * K + (size_t)g * kGroup;
        auto u_of = [&](int j) -> uint32_t { return (uint32_t)((valid ? (int)c[j] : 0) + off); };
        uint32_t word = 0;
        if (bits == 8) {
#pragma unroll
            for (int q = 0; q < 4; ++q) word |= u_of(4 * w + q) << (8 * q);
        } else if (w < 16) {
#pragma unroll
            for (int j = 0; j < 8; ++j) word |= (u_of(8 * w + j) & 15u) << (8 * (j & 3) + 4 * (j >> 2));
        } else if (w < 24) {
            const int a = w - 16;
#pragma unroll
            for (int j = 0; j < 16; ++j) word |= ((u_of(16 * a + j) >> 4) & 3u) << (8 * (j & 3) + 2 * (j >> 2));
        } else {
            const int a = w - 24;
#pragma unroll
            for (int j = 0; j < 32; ++j) word |= ((u_of(32 * a + j) >> 6) & 1u) << (8 * (j & 3) + (j >> 2));
        }
        uint8_t* u = out + unit * ub;
        *reinterpret_cast<uint32_t*>(u + word_off(r, w)) = word;
        if (w == 0)
            *reinterpret_cast<uint16_t*>(u + 2048 * bits + 2 * r) = valid ? scales[(size_t)m * G + g] : (uint16_t)0;
    }
}

__device__ __forceinline__ uint32_t rd_word(const uint8_t* u, int r, int w) {
    return *reinterpret_cast<const uint32_t*>(u + word_off(r, w));
}

// one thread per weight (test path)
__global__ void k_unpack(const uint8_t* __restrict__ base, const uint8_t* __restrict__ resid, int M, int K, int bits,
                         uint8_t* __restrict__ bc, uint16_t* __restrict__ bs, int8_t* __restrict__ rc,
                         uint16_t* __restrict__ rs) {
    const int G = K / kGroup;
    const long long total = (long long)M * K;
    for (long long it = blockIdx.x * (long long)blockDim.x + threadIdx.x; it < total;
         it += (long long)gridDim.x * blockDim.x) {
        const int m = (int)(it / K), k = (int)(it % K);
        const int tile = m / kRows, r = m % kRows, g = k / kGroup, j = k % kGroup;
        const long long unit = (long long)tile * G + g;
        const uint8_t* ub = base + unit * kBaseUnit;
        const int jj = j & 15;
        bc[it] = (uint8_t)((rd_word(ub, r, j >> 4) >> (8 * (jj & 3) + 2 * (jj >> 2))) & 3u);
        if (j == 0) bs[(size_t)m * G + g] = *reinterpret_cast<const uint16_t*>(ub + 4096 + 2 * r);
        if (bits) {
            const uint8_t* ur = resid + unit * (size_t)resid_unit_bytes(bits);
            uint32_t u;
            if (bits == 8) {
                u = (rd_word(ur, r, j >> 2) >> (8 * (j & 3))) & 255u;
            } else {
                const int j8 = j & 7, j16 = j & 15, j32 = j & 31;
                u = (rd_word(ur, r, j >> 3) >> (8 * (j8 & 3) + 4 * (j8 >> 2))) & 15u;
                u |= ((rd_word(ur, r, 16 + (j >> 4)) >> (8 * (j16 & 3) + 2 * (j16 >> 2))) & 3u) << 4;
                if (bits == 7) u |= ((rd_word(ur, r, 24 + (j >> 5)) >> (8 * (j32 & 3) + (j32 >> 2))) & 1u) << 6;
            }
            rc[it] = (int8_t)((int)u - (1 << (bits - 1)));
            if (j == 0) rs[(size_t)m * G + g] = *reinterpret_cast<const uint16_t*>(ur + 2048 * bits + 2 * r);
        }
    }
}

// W4/W8 dual-plane storage (BitNest, section 3.3): one thread per (unit, row, nibble
// word); word w of a row holds columns 8w..8w+7, column 8w + 4h + q in bits 8q + 4h.
// Stored nibble u = code + 8.  The base plane carries the fp16 scale s4 of each row at
// byte 8192 + 2r of its unit; the refinement plane has no scale.
__global__ void k_pack_nib(const int8_t* __restrict__ codes, const uint16_t* __restrict__ scales, int M, int K,
                           long long n_items, size_t unit_bytes, uint8_t* __restrict__ out) {
    const int G = K / kGroup;
    for (long long it = blockIdx.x * (long long)blockDim.x + threadIdx.x; it < n_items;
         it += (long long)gridDim.x * blockDim.x) {
        const int w = (int)(it & 15);
        const int r = (int)((it >> 4) & 127);
        const long long unit = it >> 11;
        const int tile = (int)(unit / G), g = (int)(unit % G);
        const int m = tile * kRows + r;
        const bool valid = m < M;
        const int8_t* c = codes + (size_t)(valid ? m : 0) * K + (size_t)g * kGroup + 8 * w;
        uint32_t word = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) word |= (((uint32_t)((valid ? (int)c[j] : 0) + 8)) & 15u) << (8 * (j & 3) + 4 * (j >> 2));
        uint8_t* u = out + unit * unit_bytes;
        *reinterpret_cast<uint32_t*>(u + word_off(r, w)) = word;
        if (scales != nullptr && w == 0)
            *reinterpret_cast<uint16_t*>(u + 8192 + 2 * r) = valid ? scales[(size_t)m * G + g] : (uint16_t)0;
    }
}

// one thread per weight (test path)
__global__ void k_unpack_w4w8(const uint8_t* __restrict__ base, const uint8_t* __restrict__ ref, int M, int K,
                              int8_t* __restrict__ q4, uint16_t* __restrict__ s4, int8_t* __restrict__ qr) {
    const int G = K / kGroup;
    const long long total = (long long)M * K;
    for (long long it = blockIdx.x * (long long)blockDim.x + threadIdx.x; it < total;
         it += (long long)gridDim.x * blockDim.x) {
        const int m = (int)(it / K), k = (int)(it % K);
        const int tile = m / kRows, r = m % kRows, g = k / kGroup, j = k % kGroup;
        const long long unit = (long long)tile * G + g;
        const int j8 = j & 7, sh = 8 * (j8 & 3) + 4 * (j8 >> 2);
        const uint8_t* ub = base + unit * kW4BaseUnit;
        q4[it] = (int8_t)((int)((rd_word(ub, r, j >> 3) >> sh) & 15u) - 8);
        if (j == 0) s4[(size_t)m * G + g] = *reinterpret_cast<const uint16_t*>(ub + 8192 + 2 * r);
        if (ref != nullptr) {
            const uint8_t* ur = ref + unit * kW4RefUnit;
            qr[it] = (int8_t)((int)((rd_word(ur, r, j >> 3) >> sh) & 15u) - 8);
        }
    }
}

int grid_for(long long items, int threads) {
    long long g = (items + threads - 1) / threads;
    return (int)(g < 65535 * 16 ? (g < 1 ? 1 : g) : 65535 * 16);
}

}  // namespace

cudaError_t launch_pack(const uint8_t* bc, const uint16_t* bs, const int8_t* rc, const uint16_t* rs,
                        int M, int K, int bits, uint8_t* base_out, uint8_t* resid_out, cudaStream_t stream) {
    const long long units = (long long)n_tiles(M) * (K / kGroup);
    const long long nb = units * kRows * 8;
    k_pack_base<<<grid_for(nb, 256), 256, 0, stream>>>(bc, bs, M, K, nb, base_out);
    if (bits) {
        const long long nr = units * kRows * 4 * bits;
        k_pack_resid<<<grid_for(nr, 256), 256, 0, stream>>>(rc, rs, M, K, bits, nr, resid_out);
    }
    return cudaGetLastError();
}

cudaError_t launch_unpack(const uint8_t* base, const uint8_t* resid, int M, int K, int bits,
                          uint8_t* bc, uint16_t* bs, int8_t* rc, uint16_t* rs, cudaStream_t stream) {
    const long long total = (long long)M * K;
    k_unpack<<<grid_for(total, 256), 256, 0, stream>>>(base, resid, M, K, bits, bc, bs, rc, rs);
    return cudaGetLastError();
}

}  // namespace nest

namespace nest {

cudaError_t launch_pack_w4w8(const int8_t* q4, const uint16_t* s4, const int8_t* qr, int M, int K,
                             uint8_t* base_out, uint8_t* ref_out, cudaStream_t stream) {
    const long long units = (long long)n_tiles(M) * (K / kGroup);
    const long long n = units * kRows * 16;
    k_pack_nib<<<grid_for(n, 256), 256, 0, stream>>>(q4, s4, M, K, n, kW4BaseUnit, base_out);
    if (qr != nullptr) k_pack_nib<<<grid_for(n, 256), 256, 0, stream>>>(qr, nullptr, M, K, n, kW4RefUnit, ref_out);
    return cudaGetLastError();
}

cudaError_t launch_unpack_w4w8(const uint8_t* base, const uint8_t* ref, int M, int K, int8_t* q4, uint16_t* s4,
                               int8_t* qr, cudaStream_t stream) {
    const long long total = (long long)M * K;
    k_unpack_w4w8<<<grid_for(total, 256), 256, 0, stream>>>(base, ref, M, K, q4, s4, qr);
    return cudaGetLastError();
}

}  // namespace nest
