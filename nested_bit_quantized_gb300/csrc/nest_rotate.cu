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

template <int MODE, bool BF16>
__global__ void __launch_bounds__(kThreads)
k_rotate(const __grid_constant__ RotArgs args) {
    __shared__ float buf[64][65];
    grid_dep_launch_dependents();
    int k = 0;                            // the vector set this CTA works on
    while (k + 1 < args.ntasks && args.task[k + 1].cta_begin <= (int)blockIdx.x) ++k;
    const RotTask& tk = args.task[k];
    const void* __restrict__ x = tk.x;
    const int8_t* __restrict__ signs = tk.signs;
    const unsigned n = tk.n, total = tk.total;
    const int L = tk.L, NB = tk.NB;
    const float scale = tk.scale;
    float* __restrict__ y = tk.y;
    uint16_t* __restrict__ xop = tk.xop;
    const unsigned cta = blockIdx.x - tk.cta_begin;
    const unsigned nctas = (total + kSeg - 1) / kSeg;
    grid_dep_wait();                      // x may be the previous kernel's output; y may be its input
    if (tk.zero_out != nullptr) {         // clear the accumulator of the GEMM that follows
        const long long per = (tk.zero_count + nctas - 1) / nctas;
        const long long lo = per * cta, hi = lo + per < tk.zero_count ? lo + per : tk.zero_count;
        for (long long i = lo + threadIdx.x; i < hi; i += kThreads) tk.zero_out[i] = 0.0f;
    }
    const unsigned seg0 = cta * (unsigned)kSeg;
    const unsigned rem = total - seg0;
    const int count = rem < (unsigned)kSeg ? (int)rem : kSeg;

    // all loads of this thread in flight together, then into shared memory
    constexpr int kPer = kSeg / kThreads;
    float v[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const int f = threadIdx.x + j * kThreads;
        v[j] = 0.0f;
        if (f < count) {
            const unsigned idx = seg0 + f;
            if constexpr (BF16) v[j] = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(x)[idx]);
            else v[j] = reinterpret_cast<const float*>(x)[idx];
            if constexpr (MODE == 0) v[j] *= (float)signs[idx % n];
        }
    }
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const int f = threadIdx.x + j * kThreads;
        buf[f >> 6][f & 63] = v[j];
    }
    __syncthreads();

    tile_fwht<kThreads>(buf, L);

    if (y != nullptr) {
        float sg[kPer];
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            const int f = threadIdx.x + j * kThreads;
            sg[j] = (MODE == 1 && f < count) ? (float)signs[(seg0 + f) % n] : 1.0f;
        }
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            const int f = threadIdx.x + j * kThreads;
            if (f < count) y[seg0 + f] = buf[f >> 6][f & 63] * scale * sg[j];
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
            *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(xop) + xop_offset(k, t, NB)) =
                make_uint4(w[0], w[1], w[2], w[3]);
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

cudaError_t launch_rotate_group(RotArgs& a, int x_dtype, int mode, int T, cudaStream_t stream) {
    int ctas = 0;
    for (int k = 0; k < a.ntasks; ++k) {
        RotTask& t = a.task[k];
        const int b = hadamard_block((int)t.n);
        int L = 0;
        while ((1 << L) < b) ++L;
        t.L = L;
        t.scale = (float)(1.0 / sqrt((double)b));
        t.total = (unsigned)T * t.n;                     // the entry points keep T * n < 2^31
        t.NB = n_pad(T) / 8;
        t.cta_begin = ctas;
        ctas += (int)((t.total + kSeg - 1) / kSeg);
    }
    const dim3 g(ctas), blk(kThreads);
    if (mode == 0)
        return x_dtype == 1 ? launch_pdl(k_rotate<0, true>, g, blk, 0, stream, a)
                            : launch_pdl(k_rotate<0, false>, g, blk, 0, stream, a);
    return x_dtype == 1 ? launch_pdl(k_rotate<1, true>, g, blk, 0, stream, a)
                        : launch_pdl(k_rotate<1, false>, g, blk, 0, stream, a);
}

cudaError_t launch_rotate(const void* x, int x_dtype, const int8_t* signs, int n, int T, int mode,
                          float* y, uint16_t* xop, float* zero_out, long long zero_count, cudaStream_t stream) {
    RotArgs a = {};
    a.ntasks = 1;
    a.task[0].x = x;
    a.task[0].signs = signs;
    a.task[0].y = y;
    a.task[0].xop = mode == 0 ? xop : nullptr;
    a.task[0].zero_out = zero_out;
    a.task[0].zero_count = zero_count;
    a.task[0].n = (unsigned)n;
    return launch_rotate_group(a, x_dtype, mode, T, stream);
}

}  // namespace nest
