// Randomized Hadamard rotation of activations (feedman.me/posts/wZBTJ, POC
// recipe step 1 for the transform, step 4 for where it is applied):
//   input side : x' = H S x   (signs, then the block-diagonal Sylvester FWHT)
//   output side: y  = S H z   (FWHT, then the signs)
// with blocks of size b = largest power of two dividing n (at most 4096), each
// scaled by 1/sqrt(b).
//
// Three ways, chosen per vector set of a launch:
// - blocks of at most 512 (and n % 8 == 0, 16-byte aligned vectors, 8-byte aligned
//   signs): each warp takes one (token, chunk of max(b, 256) elements) and runs the
//   butterflies in registers and warp shuffles, with no shared memory and no barrier
//   (in CTAs of one warp, k_rotate_small, when every set of the launch takes this path);
// - blocks of 1024 to 4096 (aligned output and signs): one CTA per (token, 4096-element
//   segment), butterflies over the high index bits per column, one pass through shared
//   memory, then the low 8 bits along rows (rotate_seg);
// - otherwise a CTA takes 4096 consecutive elements of the token-major [T][n] array (a
//   whole number of blocks, since b divides both n and 4096), views them as a 64 x 64
//   tile in shared memory, and runs the butterflies in two phases with warp shuffles:
//   phase 1 along rows (index bits 0..5), phase 2 along columns (index bits 6..11).
#include "nest_device.cuh"
#include "nest_internal.h"

namespace nest {
namespace {

constexpr int kSeg = 4096;
constexpr int kThreads = 512;
constexpr int kRegWarps = kThreads / 32;

constexpr long long kClearPerCta = 8192;     // floats a register-path CTA clears at most

// Register path: one warp per (token, chunk of W = max(b, 256) consecutive elements, b <=
// 512).  Lane l holds elements 256 h + 8 l + i of the chunk (i < 8, h < W / 256), so each
// lane's loads and stores are 16- or 32-byte pieces (chunk_fwht).  The signs are constants
// of the layer, not outputs of the previous kernel, so they are loaded before waiting for
// it; the clearing stores are issued after the loads.
template <int MODE, bool BF16, int H, int WARPS = kRegWarps>
__device__ __forceinline__ void rotate_reg(const RotTask& tk, unsigned cta) {
    constexpr int W = 256 * H, NR = 8 * H;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const unsigned n = tk.n, T = tk.total / tk.n;
    const unsigned nchunk = (n + W - 1) / W;
    const unsigned item = cta * WARPS + warp;
    const bool active = item < T * nchunk;             // the same for the whole warp
    const unsigned tok = active ? item / nchunk : 0, c0 = active ? (item - tok * nchunk) * W : 0;
    bool have[H];
    uint2 sg[H];
#pragma unroll
    for (int h = 0; h < H; ++h) {
        const unsigned col = c0 + 256 * h + 8 * lane;
        have[h] = active && col < n;
        sg[h] = have[h] ? *reinterpret_cast<const uint2*>(tk.signs + col) : make_uint2(0u, 0u);
    }
    grid_dep_wait();                      // x may be the previous kernel's output; y may be its input
    float v[NR];
#pragma unroll
    for (int h = 0; h < H; ++h) {
        const size_t idx = (size_t)tok * n + c0 + 256 * h + 8 * lane;
        if (have[h]) {
            if constexpr (BF16) {
                const uint4 u = __ldcg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(tk.x) + idx));
                const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    v[8 * h + 2 * e] = __uint_as_float(w[e] << 16);
                    v[8 * h + 2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
                }
            } else {
                const float4* xp = reinterpret_cast<const float4*>(static_cast<const float*>(tk.x) + idx);
                const float4 a = __ldcg(xp), b = __ldcg(xp + 1);
                v[8 * h + 0] = a.x; v[8 * h + 1] = a.y; v[8 * h + 2] = a.z; v[8 * h + 3] = a.w;
                v[8 * h + 4] = b.x; v[8 * h + 5] = b.y; v[8 * h + 6] = b.z; v[8 * h + 7] = b.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) v[8 * h + i] = 0.0f;
        }
    }
    // clear the accumulator of the GEMM that follows (the task may have CTAs for this alone)
    if (tk.zero_out != nullptr) clear_share<32 * WARPS>(tk.zero_out, tk.zero_count, cta, tk.nctas);
    if (!active) return;
    auto sign = [&](int j) { return (float)(int8_t)((((j & 7) < 4 ? sg[j >> 3].x : sg[j >> 3].y) >> (8 * (j & 3))) & 0xFFu); };
    if constexpr (MODE == 0) {
#pragma unroll
        for (int j = 0; j < NR; ++j) v[j] *= sign(j);
    }
    chunk_fwht<H>(v, tk.L, lane);
    const float scale = tk.scale;
#pragma unroll
    for (int j = 0; j < NR; ++j) v[j] *= MODE == 1 ? scale * sign(j) : scale;
#pragma unroll
    for (int h = 0; h < H; ++h) {
        if (!have[h]) continue;
        const unsigned col = c0 + 256 * h + 8 * lane;
        if (tk.y != nullptr) {
            float4* yp = reinterpret_cast<float4*>(tk.y + (size_t)tok * n + col);
            yp[0] = make_float4(v[8 * h + 0], v[8 * h + 1], v[8 * h + 2], v[8 * h + 3]);
            yp[1] = make_float4(v[8 * h + 4], v[8 * h + 5], v[8 * h + 6], v[8 * h + 7]);
        }
        if (MODE == 0 && tk.xop != nullptr) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) w[e] = h2_as_u32(__floats2half2_rn(v[8 * h + 2 * e], v[8 * h + 2 * e + 1]));
            *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(tk.xop) + xop_offset((int)col, (int)tok, tk.NB)) =
                make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
}

// Segment path (blocks of 1024 .. 4096, 16-byte aligned y, 8-byte aligned signs): one CTA
// per (token, 4096-element segment of the vector), see seg_col in nest_device.cuh.  Phase A
// loads each thread's rows of one column (coalesced scalar loads; input-side signs applied
// there), phase B stores each warp's row as 16- or 32-byte pieces.  One barrier.
template <int MODE, bool BF16>
__device__ __forceinline__ void rotate_seg(const RotTask& tk, unsigned cta, float* sm) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const unsigned n = tk.n, T = tk.total / tk.n;
    const unsigned nseg = (n + 4095) / 4096;
    const bool work = cta < T * nseg;                  // the same for the whole CTA
    const unsigned tok = work ? cta / nseg : 0, s0 = work ? (cta - tok * nseg) * 4096 : 0;
    const int L = tk.L;
    const SegCol sc = seg_col(L);
    float sgA[16];
    uint2 sgB = make_uint2(0u, 0u);
    const unsigned eB = s0 + 256 * warp + 8 * lane;    // phase B: this lane's 8 elements
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const unsigned e = s0 + 256 * (sc.r0 + k) + sc.c;
        sgA[k] = (MODE == 0 && work && k < sc.nr && e < n) ? (float)tk.signs[e] : 0.0f;
    }
    if (MODE == 1 && work && eB < n) sgB = *reinterpret_cast<const uint2*>(tk.signs + eB);
    grid_dep_wait();                      // x may be the previous kernel's output; y may be its input
    float v[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const unsigned e = s0 + 256 * (sc.r0 + k) + sc.c;
        float x = 0.0f;
        if (work && k < sc.nr && e < n) {
            const size_t idx = (size_t)tok * n + e;
            if constexpr (BF16) x = __bfloat162float(__ldcg(static_cast<const __nv_bfloat16*>(tk.x) + idx));
            else x = __ldcg(static_cast<const float*>(tk.x) + idx);
        }
        v[k] = MODE == 0 ? x * sgA[k] : x;
    }
    // clear the accumulator of the GEMM that follows (the task may have CTAs for this alone)
    if (tk.zero_out != nullptr) clear_share<kThreads>(tk.zero_out, tk.zero_count, cta, tk.nctas);
    if (!work) return;
    seg_rows_fwht(v, L);
    seg_col_store(sm, sc, v);
    __syncthreads();
    float w[8];
    seg_row_load(sm, warp, lane, w);
    chunk_fwht<1>(w, 8, lane);
    if (eB >= n) return;                  // n is a multiple of 1024: whole groups of 8
    const float scale = tk.scale;
    if constexpr (MODE == 1) {
        const uint2 sg[1] = {sgB};
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i] *= scale * chunk_sign<1>(sg, i);
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i] *= scale;
    }
    if (tk.y != nullptr) {
        float4* yp = reinterpret_cast<float4*>(tk.y + (size_t)tok * n + eB);
        yp[0] = make_float4(w[0], w[1], w[2], w[3]);
        yp[1] = make_float4(w[4], w[5], w[6], w[7]);
    }
    if (MODE == 0 && tk.xop != nullptr) {
        uint32_t q[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) q[e] = h2_as_u32(__floats2half2_rn(w[2 * e], w[2 * e + 1]));
        *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(tk.xop) + xop_offset((int)eB, (int)tok, tk.NB)) =
            make_uint4(q[0], q[1], q[2], q[3]);
    }
}

// Launches whose vector sets all take the register path: CTAs of one warp with no shared
// memory, small enough that two become resident on an SM beside the GEMM's two CTAs, so
// that the launch's CTAs are in place, signs loaded, when the GEMM before them completes
// (and leave the GEMM after them every SM).
constexpr int kSmallWarps = 1;
constexpr long long kSmallClear = 1024;      // floats a small CTA clears at most

template <int MODE, bool BF16>
__global__ void __launch_bounds__(32 * kSmallWarps)
k_rotate_small(const __grid_constant__ RotArgs args) {
    grid_dep_launch_dependents();
    int k = 0;
    while (k + 1 < args.ntasks && args.task[k + 1].cta_begin <= (int)blockIdx.x) ++k;
    const RotTask& tk = args.task[k];
    const unsigned cta = blockIdx.x - tk.cta_begin;
    if (tk.L <= 8) rotate_reg<MODE, BF16, 1, kSmallWarps>(tk, cta);
    else rotate_reg<MODE, BF16, 2, kSmallWarps>(tk, cta);
}

template <int MODE, bool BF16>
__global__ void __launch_bounds__(kThreads)
k_rotate(const __grid_constant__ RotArgs args) {
    __shared__ __align__(16) float buf[64][65];
    grid_dep_launch_dependents();
    int k = 0;                            // the vector set this CTA works on
    while (k + 1 < args.ntasks && args.task[k + 1].cta_begin <= (int)blockIdx.x) ++k;
    const RotTask& tk = args.task[k];
    if (tk.path != 0) {                   // the same for every thread of the CTA
        const unsigned cta = blockIdx.x - tk.cta_begin;
        if (tk.path == 2) rotate_seg<MODE, BF16>(tk, cta, &buf[0][0]);
        else if (tk.L <= 8) rotate_reg<MODE, BF16, 1>(tk, cta);
        else rotate_reg<MODE, BF16, 2>(tk, cta);
        return;
    }
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
    // clear the accumulator of the GEMM that follows (after the loads)
    if (tk.zero_out != nullptr) clear_share<kThreads>(tk.zero_out, tk.zero_count, cta, nctas);
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

static bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

cudaError_t launch_rotate_group(RotArgs& a, int x_dtype, int mode, int T, cudaStream_t stream) {
    bool small = true;                                   // every set takes the register path
    for (int k = 0; k < a.ntasks; ++k) {
        const RotTask& t = a.task[k];
        const int b = hadamard_block((int)t.n);
        small = small && b <= 512 && t.n % 8 == 0 && aligned(t.x, 16) && aligned(t.y, 16) && aligned(t.signs, 8);
    }
    const int warps = small ? kSmallWarps : kRegWarps;
    const long long clear_per = small ? kSmallClear : kClearPerCta;
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
        if (b <= 512 && t.n % 8 == 0 && aligned(t.x, 16) && aligned(t.y, 16) && aligned(t.signs, 8)) t.path = 1;
        else if (b >= 1024 && aligned(t.y, 16) && aligned(t.signs, 8)) t.path = 2;
        else t.path = 0;
        t.cta_begin = ctas;
        long long c;
        if (t.path != 0) {
            const long long items = t.path == 1 ? (long long)T * ((t.n + reg_chunk(L) - 1) / reg_chunk(L)) : 0;
            c = t.path == 1 ? (items + warps - 1) / warps : (long long)T * ((t.n + 4095) / 4096);
            const long long cz = t.zero_out != nullptr ? (t.zero_count + clear_per - 1) / clear_per : 0;
            if (cz > c) c = cz;
        } else {
            c = (t.total + kSeg - 1) / kSeg;
        }
        t.nctas = (unsigned)c;
        ctas += (int)c;
    }
    if (small) {
        const dim3 g(ctas), blk(32 * kSmallWarps);
        if (mode == 0)
            return x_dtype == 1 ? launch_pdl(k_rotate_small<0, true>, g, blk, 0, stream, a)
                                : launch_pdl(k_rotate_small<0, false>, g, blk, 0, stream, a);
        return x_dtype == 1 ? launch_pdl(k_rotate_small<1, true>, g, blk, 0, stream, a)
                            : launch_pdl(k_rotate_small<1, false>, g, blk, 0, stream, a);
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
