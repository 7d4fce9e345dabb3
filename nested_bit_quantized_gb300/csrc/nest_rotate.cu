// Randomized Hadamard rotation of activations (feedman.me/posts/wZBTJ, POC
// recipe step 1 for the transform, step 4 for where it is applied):
//   input side : x' = H S x   (signs, then the block-diagonal Sylvester FWHT)
//   output side: y  = S H z   (FWHT, then the signs)
// with blocks of size b = largest power of two dividing n (at most 4096), each
// scaled by 1/sqrt(b).
//
// A CTA takes 4096 consecutive elements of the token-major [T][n] array (a
// whole number of blocks, since b divides both n and 4096), views them as a
// 64 x 64 tile in shared memory, and runs the butterflies in two phases with
// warp shuffles: phase 1 along rows (index bits 0..5), phase 2 along columns
// (index bits 6..11).  Each warp holds 64 elements, two per lane.
#include "nest_device.cuh"
#include "nest_internal.h"

namespace nest {
namespace {

constexpr int kSeg = 4096;
constexpr int kThreads = 512;

// Butterflies over the low `nbits` bits of a 64-element warp vector:
// element `lane` in v0, element `lane + 32` in v1.
__device__ __forceinline__ void warp_fwht(float& v0, float& v1, int nbits, int lane) {
    const int lane_bits = nbits < 5 ? nbits : 5;
    for (int s = 0; s < lane_bits; ++s) {
        const int m = 1 << s;
        const float o0 = __shfl_xor_sync(0xffffffffu, v0, m);
        const float o1 = __shfl_xor_sync(0xffffffffu, v1, m);
        const bool upper = (lane & m) != 0;
        v0 = upper ? o0 - v0 : v0 + o0;
        v1 = upper ? o1 - v1 : v1 + o1;
    }
    if (nbits >= 6) {
        const float a = v0 + v1, b = v0 - v1;
        v0 = a;
        v1 = b;
    }
}

template <int MODE, bool BF16>
__global__ void __launch_bounds__(kThreads)
k_rotate(const void* __restrict__ x, const int8_t* __restrict__ signs, unsigned n, unsigned total, int L,
         float scale, float* __restrict__ y, uint16_t* __restrict__ xop, int NB, float* __restrict__ zero_out,
         long long zero_count) {
    __shared__ float buf[64][65];
    grid_dep_launch_dependents();
    grid_dep_wait();                      // x may be the previous kernel's output; y may be its input
    if (zero_out != nullptr) {            // clear the accumulator of the GEMM that follows
        const long long per = (zero_count + gridDim.x - 1) / gridDim.x;
        const long long lo = per * blockIdx.x, hi = lo + per < zero_count ? lo + per : zero_count;
        for (long long i = lo + threadIdx.x; i < hi; i += kThreads) zero_out[i] = 0.0f;
    }
    const unsigned seg0 = blockIdx.x * (unsigned)kSeg;
    const unsigned rem = total - seg0;
    const int count = rem < (unsigned)kSeg ? (int)rem : kSeg;

    for (int f = threadIdx.x; f < kSeg; f += kThreads) {
        float v = 0.0f;
        if (f < count) {
            const unsigned idx = seg0 + f;
            if constexpr (BF16) v = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(x)[idx]);
            else v = reinterpret_cast<const float*>(x)[idx];
            if constexpr (MODE == 0) v *= (float)signs[idx % n];
        }
        buf[f >> 6][f & 63] = v;
    }
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int L1 = L < 6 ? L : 6;
    if (L1 > 0) {
        for (int row = warp; row < 64; row += kThreads / 32) {
            float v0 = buf[row][lane], v1 = buf[row][lane + 32];
            warp_fwht(v0, v1, L1, lane);
            buf[row][lane] = v0;
            buf[row][lane + 32] = v1;
        }
        __syncthreads();
    }
    if (L > 6) {
        for (int col = warp; col < 64; col += kThreads / 32) {
            float v0 = buf[lane][col], v1 = buf[lane + 32][col];
            warp_fwht(v0, v1, L - 6, lane);
            buf[lane][col] = v0;
            buf[lane + 32][col] = v1;
        }
        __syncthreads();
    }

    if (y != nullptr) {
        for (int f = threadIdx.x; f < count; f += kThreads) {
            const unsigned idx = seg0 + f;
            float v = buf[f >> 6][f & 63] * scale;
            if constexpr (MODE == 1) v *= (float)signs[idx % n];
            y[idx] = v;
        }
    }
    if (MODE == 0 && xop != nullptr) {
        // eight consecutive columns of one token -> one 16-byte store into the operand layout
        for (int j = threadIdx.x; j < count / 8; j += kThreads) {
            const int f = 8 * j;
            const unsigned idx = seg0 + f;
            const unsigned t = idx / n, k = idx - t * n;
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float a = buf[(f + 2 * e) >> 6][(f + 2 * e) & 63] * scale;
                const float b = buf[(f + 2 * e + 1) >> 6][(f + 2 * e + 1) & 63] * scale;
                w[e] = h2_as_u32(__floats2half2_rn(a, b));
            }
            const int g = k >> 7, c = (k & 127) >> 3;
            const size_t off = (size_t)g * 2048 * NB + ((size_t)(c * NB + (t >> 3)) * 8 + (t & 7)) * 16;
            *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(xop) + off) = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
}

}  // namespace

int hadamard_block(int n) {
    if (n < 1) return 0;
    int b = 1;
    while (n % (2 * b) == 0 && 2 * b <= kHadCap) b *= 2;
    return b;
}

cudaError_t launch_rotate(const void* x, int x_dtype, const int8_t* signs, int n, int T, int mode,
                          float* y, uint16_t* xop, float* zero_out, long long zero_count, cudaStream_t stream) {
    const int b = hadamard_block(n);
    int L = 0;
    while ((1 << L) < b) ++L;
    const float scale = (float)(1.0 / sqrt((double)b));
    const unsigned total = (unsigned)T * (unsigned)n;     // the entry point keeps T * n < 2^31
    const int grid = (int)((total + kSeg - 1) / kSeg);
    const int NB = n_pad(T) / 8;
    const dim3 g(grid), blk(kThreads);
    if (mode == 0) {
        if (x_dtype == 1)
            return launch_pdl(k_rotate<0, true>, g, blk, 0, stream, x, signs, (unsigned)n, total, L, scale, y, xop, NB,
                              zero_out, zero_count);
        return launch_pdl(k_rotate<0, false>, g, blk, 0, stream, x, signs, (unsigned)n, total, L, scale, y, xop, NB,
                          zero_out, zero_count);
    }
    if (x_dtype == 1)
        return launch_pdl(k_rotate<1, true>, g, blk, 0, stream, x, signs, (unsigned)n, total, L, scale, y,
                          (uint16_t*)nullptr, NB, zero_out, zero_count);
    return launch_pdl(k_rotate<1, false>, g, blk, 0, stream, x, signs, (unsigned)n, total, L, scale, y,
                      (uint16_t*)nullptr, NB, zero_out, zero_count);
}

}  // namespace nest
