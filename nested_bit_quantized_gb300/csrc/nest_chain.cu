// Glue between the linears of a chained decoder layer, fused with the
// rotations on both sides of it:
//   h    = S_o H_o z_a           (output rotation of linear a)
//      or  (S_o H_o z_a) * (S_o' H_o' z_b)   (elementwise product, e.g. gate * up)
//   h'   = bf16(h / rms(h))      (unit-RMS rescale per token, then the bf16 cast)
//   x'_j = H_j S_j h'            (input rotation of each next linear j, into its
//                                 fp16 GEMM operand)
// The rotations follow feedman.me/posts/wZBTJ, POC recipe steps 1 and 4.  The
// chaining itself (which output feeds which linear, and the RMS rescale standing
// in for the normalisation between them) is not on the pages; it is the plain
// reading used by the chained-layer workload.
//
// Two launches, both spread over every (token, 4096-element segment) pair so that
// a single token still occupies many SMs:
//   k_glue_out: one CTA per (t, segment) rotates its segment of z_a (and z_b) in a
//               64 x 64 shared-memory tile, writes h and the segment's sum of
//               squares.  A segment is a whole number of Hadamard blocks (the block
//               size divides both M and 4096).
//   k_glue_in : one CTA per (next linear, t, segment) adds up the token's segment
//               sums in a fixed order (so the result does not depend on timing),
//               rescales and rounds its segment of h, applies S_j, rotates and
//               writes the fp16 operand; it also clears a share of the next GEMM's
//               accumulator.
#include "nest_device.cuh"
#include "nest_internal.h"

namespace nest {
namespace {

constexpr int kSeg = 4096;
constexpr int kThreads = 512;
constexpr int kPer = kSeg / kThreads;

template <bool PROD>
__global__ void __launch_bounds__(kThreads) k_glue_out(const __grid_constant__ GlueArgs a) {
    __shared__ float buf[64][65];
    __shared__ float buf2[PROD ? 64 : 1][65];
    __shared__ float red[32];
    grid_dep_launch_dependents();
    const int t = blockIdx.x / a.nseg, s = blockIdx.x - t * a.nseg;
    const int seg0 = s * kSeg;
    const int count = a.M - seg0 < kSeg ? a.M - seg0 : kSeg;
    const size_t row = (size_t)t * a.M + seg0;
    grid_dep_wait();                 // z_a, z_b come from the GEMM before this launch

    float v[kPer], w[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const int f = threadIdx.x + j * kThreads;
        v[j] = f < count ? a.za[row + f] : 0.0f;
        if constexpr (PROD) w[j] = f < count ? a.zb[row + f] : 0.0f;
    }
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const int f = threadIdx.x + j * kThreads;
        buf[f >> 6][f & 63] = v[j];
        if constexpr (PROD) buf2[f >> 6][f & 63] = w[j];
    }
    __syncthreads();
    tile_fwht<kThreads>(buf, a.L);
    if constexpr (PROD) tile_fwht<kThreads>(buf2, a.L);

    // h may overwrite z_a: every element of this segment was read above, by this CTA
    float ss = 0.0f;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const int f = threadIdx.x + j * kThreads;
        if (f < count) {
            float h = buf[f >> 6][f & 63] * a.scale * (float)a.sa[seg0 + f];
            if constexpr (PROD) h *= buf2[f >> 6][f & 63] * a.scale * (float)a.sb[seg0 + f];
            a.h[row + f] = h;
            ss += h * h;
        }
    }
    ss = cta_sum<kThreads>(ss, red);
    if (threadIdx.x == 0) a.work[blockIdx.x] = ss;
}

__global__ void __launch_bounds__(kThreads) k_glue_in(const __grid_constant__ GlueArgs a) {
    __shared__ float buf[64][65];
    __shared__ float s_inv;
    grid_dep_launch_dependents();
    const int per_next = a.T * a.nseg;
    const int jn = blockIdx.x / per_next;
    const int rem = blockIdx.x - jn * per_next;
    const int t = rem / a.nseg, s = rem - t * a.nseg;
    const int seg0 = s * kSeg;
    const int count = a.M - seg0 < kSeg ? a.M - seg0 : kSeg;
    const size_t row = (size_t)t * a.M + seg0;
    const GlueNext& nx = a.next[jn];
    grid_dep_wait();                 // h and the segment sums come from k_glue_out

    if (nx.zero_out != nullptr) {    // this CTA's share of the next GEMM's accumulator
        const long long per = (nx.zero_count + per_next - 1) / per_next;
        const long long lo = per * rem, hi = lo + per < nx.zero_count ? lo + per : nx.zero_count;
        for (long long i = lo + threadIdx.x; i < hi; i += kThreads) nx.zero_out[i] = 0.0f;
    }
    if (threadIdx.x == 0) {
        float ss = 0.0f;
        for (int i = 0; i < a.nseg; ++i) ss += a.work[t * a.nseg + i];
        const float rms = sqrtf(ss / (float)a.M);
        s_inv = rms > 0.0f ? 1.0f / rms : 0.0f;
    }
    float v[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const int f = threadIdx.x + j * kThreads;
        v[j] = f < count ? a.h[row + f] : 0.0f;
    }
    __syncthreads();
    const float inv = s_inv;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const int f = threadIdx.x + j * kThreads;
        float x = 0.0f;
        if (f < count) x = __bfloat162float(__float2bfloat16_rn(v[j] * inv)) * (float)nx.sign_in[seg0 + f];
        buf[f >> 6][f & 63] = x;
    }
    __syncthreads();
    tile_fwht<kThreads>(buf, a.L);

    // eight consecutive columns -> one 16-byte store into the operand layout (count % 128 == 0)
    for (int c8 = threadIdx.x; c8 < count / 8; c8 += kThreads) {
        const int f = 8 * c8;
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int f0 = f + 2 * e, f1 = f0 + 1;
            w[e] = h2_as_u32(__floats2half2_rn(buf[f0 >> 6][f0 & 63] * a.scale, buf[f1 >> 6][f1 & 63] * a.scale));
        }
        *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(nx.xop) + xop_offset(seg0 + f, t, a.NB)) =
            make_uint4(w[0], w[1], w[2], w[3]);
    }
}

}  // namespace

int glue_segments(int M) { return (M + kSeg - 1) / kSeg; }

cudaError_t launch_glue(GlueArgs& a, cudaStream_t stream) {
    const int b = hadamard_block(a.M);
    int L = 0;
    while ((1 << L) < b) ++L;
    a.L = L;
    a.scale = (float)(1.0 / sqrt((double)b));
    a.NB = n_pad(a.T) / 8;
    a.nseg = glue_segments(a.M);
    const dim3 blk(kThreads);
    cudaError_t e = a.zb != nullptr ? launch_pdl(k_glue_out<true>, dim3(a.T * a.nseg), blk, 0, stream, a)
                                    : launch_pdl(k_glue_out<false>, dim3(a.T * a.nseg), blk, 0, stream, a);
    if (e != cudaSuccess || a.nnext == 0) return e;
    return launch_pdl(k_glue_in, dim3(a.nnext * a.T * a.nseg), blk, 0, stream, a);
}

}  // namespace nest
