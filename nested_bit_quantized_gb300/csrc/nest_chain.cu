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
// Two launches (out, then in), both spread over the token's elements so that a single
// token still occupies many SMs.  For blocks of up to 512 elements the butterflies run in
// registers, one warp per (token, chunk of max(b, 256) elements), in CTAs of one warp
// without shared memory (the register path below; one partial sum of squares per chunk);
// for blocks of 1024 to 4096 one CTA takes a (token, 4096-element segment) as 16 rows x 256
// columns with one pass through shared memory (the segment path); otherwise:
//   k_glue_out: one CTA per (t, segment) rotates its segment of z_a (and z_b) in a
//               64 x 64 shared-memory tile, writes h and the segment's sum of
//               squares.  A segment is a whole number of Hadamard blocks (the block
//               size divides both M and 4096).
//   k_glue_in : one CTA per (next linear, t, segment) adds up the token's segment
//               sums in a fixed order (so the result does not depend on timing),
//               rescales and rounds its segment of h, applies S_j, rotates and
//               writes the fp16 operand; it also clears a share of the next GEMM's
//               accumulator.
// Side tasks: up to two plain output rotations y = S_o H_o z of other linears (the k and v
// outputs beside the q glue) run as extra CTAs of the first launch, on the glue's own path,
// so they add no launch to the chain (OutJob below; no sum of squares is kept for them).
#include "nest_device.cuh"
#include "nest_internal.h"

namespace nest {
namespace {

constexpr int kSeg = 4096;
constexpr int kThreads = 512;
constexpr int kPer = kSeg / kThreads;
constexpr int kWarps = kThreads / 32;

// Register path (GlueArgs::path 3: b <= 512, M % 8 == 0, 16-byte aligned vectors, 8-byte
// aligned signs): a warp keeps a chunk of W = max(b, 256) elements in registers (chunk_fwht:
// lane l holds elements 256 h + 8 l + i) and needs no shared memory or barrier for the
// butterflies.  The signs are layer constants and are loaded before waiting for the
// previous kernel.

// Load the 8 H fp32 values of a warp's chunk that starts at element c0 of row `row`.
template <int H>
__device__ __forceinline__ void load_chunk(const float* base, const bool (&have)[H], int lane, float (&v)[8 * H]) {
#pragma unroll
    for (int h = 0; h < H; ++h) {
        if (have[h]) {
            const float4* p = reinterpret_cast<const float4*>(base + 256 * h + 8 * lane);
            const float4 x = __ldcg(p), y = __ldcg(p + 1);
            v[8 * h + 0] = x.x; v[8 * h + 1] = x.y; v[8 * h + 2] = x.z; v[8 * h + 3] = x.w;
            v[8 * h + 4] = y.x; v[8 * h + 5] = y.y; v[8 * h + 6] = y.z; v[8 * h + 7] = y.w;
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) v[8 * h + i] = 0.0f;
        }
    }
}

// Segment path (GlueArgs::path 2: b = 1024 .. 4096, 16-byte aligned h, 8-byte aligned
// signs): the CTA's (token, 4096-element segment) as 16 rows x 256 columns (seg_col in
// nest_device.cuh): coalesced column loads and the butterflies over the high index bits,
// one pass through shared memory, then the low 8 bits along the rows, one row per warp.
// What an out-rotation CTA (register path: warp) works on: the glue's linear a (and its
// product partner), or an extra output rotation run in the same launch (no partner, and its
// sums of squares are not kept).
struct OutJob {
    const float* za;
    const int8_t* sa;
    const float* zb;
    const int8_t* sb;
    float* h;
    float* work;              // partial sums of squares, or nullptr
    int M, L;
    float scale;
};
__device__ __forceinline__ OutJob glue_job(const GlueArgs& a) {
    return OutJob{a.za, a.sa, a.zb, a.sb, a.h, a.work, a.M, a.L, a.scale};
}
__device__ __forceinline__ OutJob side_job(const GlueSide& d) {
    return OutJob{d.z, d.s, nullptr, nullptr, d.y, nullptr, d.M, d.L, d.scale};
}
// The side task of a launch that holds CTA (warp item) i, i past the glue's own.
__device__ __forceinline__ const GlueSide& side_of(const GlueArgs& a, int i) {
    int k = 0;
    while (k + 1 < a.nside && a.side[k + 1].cta_begin <= i) ++k;
    return a.side[k];
}

template <bool PROD>
__device__ __forceinline__ void glue_out_seg(const OutJob& a, int t, int seg0, int slot, float* sm, float* sm2,
                                             float* red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int L = a.L, M = a.M;
    const SegCol sc = seg_col(L);
    const int eB = seg0 + 256 * warp + 8 * lane;       // phase B: this lane's 8 elements
    uint2 sa[1] = {make_uint2(0u, 0u)}, sb[1] = {make_uint2(0u, 0u)};
    if (eB < M) {
        sa[0] = *reinterpret_cast<const uint2*>(a.sa + eB);
        if constexpr (PROD) sb[0] = *reinterpret_cast<const uint2*>(a.sb + eB);
    }
    grid_dep_wait();                 // z_a, z_b come from the GEMM before this launch
    const size_t row = (size_t)t * M;
    float v[16], w[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const int e = seg0 + 256 * (sc.r0 + k) + sc.c;
        const bool in = k < sc.nr && e < M;
        v[k] = in ? __ldcg(a.za + row + e) : 0.0f;
        w[k] = (PROD && in) ? __ldcg(a.zb + row + e) : 0.0f;
    }
    seg_rows_fwht(v, L);
    seg_col_store(sm, sc, v);
    if constexpr (PROD) {
        seg_rows_fwht(w, L);
        seg_col_store(sm2, sc, w);
    }
    __syncthreads();                 // every load of the segment is done: h may overwrite z_a
    float hv[8], wb[8];
    seg_row_load(sm, warp, lane, hv);
    chunk_fwht<1>(hv, 8, lane);
    if constexpr (PROD) {
        seg_row_load(sm2, warp, lane, wb);
        chunk_fwht<1>(wb, 8, lane);
    }
    float ss = 0.0f;
    if (eB < M) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            hv[i] *= a.scale * chunk_sign<1>(sa, i);
            if constexpr (PROD) hv[i] *= wb[i] * a.scale * chunk_sign<1>(sb, i);
            ss += hv[i] * hv[i];
        }
        float4* hp = reinterpret_cast<float4*>(a.h + row + eB);
        hp[0] = make_float4(hv[0], hv[1], hv[2], hv[3]);
        hp[1] = make_float4(hv[4], hv[5], hv[6], hv[7]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) red[warp] = ss;
    __syncthreads();
    if (threadIdx.x == 0 && a.work != nullptr) {      // the warps' sums in a fixed order
        float tot = 0.0f;
        for (int i = 0; i < kWarps; ++i) tot += red[i];
        a.work[slot] = tot;
    }
}

__device__ __forceinline__ void glue_in_seg(const GlueArgs& a, const GlueNext& nx, int t, int seg0, int rem,
                                            int per_next, float* sm) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int L = a.L, M = a.M;
    const SegCol sc = seg_col(L);
    float sg[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const int e = seg0 + 256 * (sc.r0 + k) + sc.c;
        sg[k] = (k < sc.nr && e < M) ? (float)nx.sign_in[e] : 0.0f;
    }
    grid_dep_wait();                 // h and the segment sums come from k_glue_out
    const size_t row = (size_t)t * M;
    float v[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const int e = seg0 + 256 * (sc.r0 + k) + sc.c;
        v[k] = (k < sc.nr && e < M) ? __ldcg(a.h + row + e) : 0.0f;
    }
    // this CTA's share of the next GEMM's accumulator, after the loads
    if (nx.zero_out != nullptr) clear_share<kThreads>(nx.zero_out, nx.zero_count, rem, per_next);
    // the token's sum of squares: every warp adds the segment sums in the same tree order
    float ss = 0.0f;
    for (int i = lane; i < a.nseg; i += 32) ss += __ldcg(a.work + t * a.nseg + i);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float rms = sqrtf(ss / (float)M);
    const float inv = rms > 0.0f ? 1.0f / rms : 0.0f;
#pragma unroll
    for (int k = 0; k < 16; ++k) v[k] = __bfloat162float(__float2bfloat16_rn(v[k] * inv)) * sg[k];
    seg_rows_fwht(v, L);
    seg_col_store(sm, sc, v);
    __syncthreads();
    float w[8];
    seg_row_load(sm, warp, lane, w);
    chunk_fwht<1>(w, 8, lane);
    const int eB = seg0 + 256 * warp + 8 * lane;
    if (eB >= M) return;
    uint32_t q[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) q[e] = h2_as_u32(__floats2half2_rn(w[2 * e] * a.scale, w[2 * e + 1] * a.scale));
    *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(nx.xop) + xop_offset(eB, t, a.NB)) =
        make_uint4(q[0], q[1], q[2], q[3]);
}

// Small launch shape for the register path (GlueArgs::path 3): CTAs of one warp with no
// shared memory, each warp one (token, chunk of W = max(b, 256) elements), small enough to
// become resident beside a running GEMM.  With no CTA-wide reduction, k_glue_out_small
// writes one sum of squares per (token, chunk) (work [T][nchunk]) and k_glue_in_small adds a
// token's nchunk partial sums with a fixed shuffle tree in every warp.
constexpr int kSmallWarps = 1;

template <bool PROD, int H>
__device__ __forceinline__ void glue_out_small(const OutJob& a, int item, int nchunk) {
    constexpr int W = 256 * H, NR = 8 * H;
    const int lane = threadIdx.x & 31;
    const int t = item / nchunk, c = item - t * nchunk;
    const int c0 = c * W, M = a.M;
    bool have[H];
    uint2 sa[H], sb[H];
#pragma unroll
    for (int h = 0; h < H; ++h) {
        const int col = c0 + 256 * h + 8 * lane;
        have[h] = col < M;
        sa[h] = have[h] ? *reinterpret_cast<const uint2*>(a.sa + col) : make_uint2(0u, 0u);
        sb[h] = (PROD && have[h]) ? *reinterpret_cast<const uint2*>(a.sb + col) : make_uint2(0u, 0u);
    }
    grid_dep_wait();                 // z_a, z_b come from the GEMM before this launch
    const size_t row = (size_t)t * M + c0;
    float v[NR], w[NR];
    load_chunk<H>(a.za + row, have, lane, v);
    if constexpr (PROD) load_chunk<H>(a.zb + row, have, lane, w);
    chunk_fwht<H>(v, a.L, lane);
    if constexpr (PROD) chunk_fwht<H>(w, a.L, lane);
    float ss = 0.0f;
#pragma unroll
    for (int j = 0; j < NR; ++j) {
        v[j] *= a.scale * chunk_sign<H>(sa, j);
        if constexpr (PROD) v[j] *= w[j] * a.scale * chunk_sign<H>(sb, j);
        ss += v[j] * v[j];
    }
    // h may overwrite z_a: this warp read its whole chunk above
#pragma unroll
    for (int h = 0; h < H; ++h) {
        if (!have[h]) continue;
        float4* hp = reinterpret_cast<float4*>(a.h + row + 256 * h + 8 * lane);
        hp[0] = make_float4(v[8 * h + 0], v[8 * h + 1], v[8 * h + 2], v[8 * h + 3]);
        hp[1] = make_float4(v[8 * h + 4], v[8 * h + 5], v[8 * h + 6], v[8 * h + 7]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0 && a.work != nullptr) a.work[item] = ss;
}

template <int H>
__device__ __forceinline__ void glue_in_small(const GlueArgs& a) {
    constexpr int W = 256 * H, NR = 8 * H;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int per_next = (a.T * a.nchunk + kSmallWarps - 1) / kSmallWarps;   // CTAs of one next linear
    const int jn = blockIdx.x / per_next, lc = blockIdx.x - jn * per_next;
    const GlueNext& nx = a.next[jn];
    const int item = lc * kSmallWarps + warp;
    const bool active = item < a.T * a.nchunk;         // the same for the whole warp
    const int t = active ? item / a.nchunk : 0, c = active ? item - t * a.nchunk : 0;
    const int c0 = c * W, M = a.M;
    bool have[H];
    uint2 sg[H];
#pragma unroll
    for (int h = 0; h < H; ++h) {
        const int col = c0 + 256 * h + 8 * lane;
        have[h] = active && col < M;
        sg[h] = have[h] ? *reinterpret_cast<const uint2*>(nx.sign_in + col) : make_uint2(0u, 0u);
    }
    grid_dep_wait();                 // h and the chunk sums come from k_glue_out_small
    float v[NR];
    if (active) load_chunk<H>(a.h + (size_t)t * M + c0, have, lane, v);
    // this CTA's share of the next GEMM's accumulator, after the loads
    if (nx.zero_out != nullptr) clear_share<32 * kSmallWarps>(nx.zero_out, nx.zero_count, lc, per_next);
    if (!active) return;
    float ss = 0.0f;
    for (int i = lane; i < a.nchunk; i += 32) ss += __ldcg(a.work + t * a.nchunk + i);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float rms = sqrtf(ss / (float)M);
    const float inv = rms > 0.0f ? 1.0f / rms : 0.0f;
#pragma unroll
    for (int j = 0; j < NR; ++j)
        v[j] = __bfloat162float(__float2bfloat16_rn(v[j] * inv)) * chunk_sign<H>(sg, j);
    chunk_fwht<H>(v, a.L, lane);
#pragma unroll
    for (int h = 0; h < H; ++h) {
        if (!have[h]) continue;
        const int col = c0 + 256 * h + 8 * lane;
        uint32_t q[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
            q[e] = h2_as_u32(__floats2half2_rn(v[8 * h + 2 * e] * a.scale, v[8 * h + 2 * e + 1] * a.scale));
        *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(nx.xop) + xop_offset(col, t, a.NB)) =
            make_uint4(q[0], q[1], q[2], q[3]);
    }
}

template <bool PROD>
__global__ void __launch_bounds__(32 * kSmallWarps) k_glue_out_small(const __grid_constant__ GlueArgs a) {
    grid_dep_launch_dependents();
    const int item = blockIdx.x * kSmallWarps + (threadIdx.x >> 5);   // the same for the whole warp
    if (item < a.glue_ctas) {
        if (a.L <= 8) glue_out_small<PROD, 1>(glue_job(a), item, a.nchunk);
        else glue_out_small<PROD, 2>(glue_job(a), item, a.nchunk);
        return;
    }
    if (a.nside == 0) return;
    const GlueSide& d = side_of(a, item);
    const int it = item - d.cta_begin;
    if (it >= a.T * d.nchunk) return;
    if (d.L <= 8) glue_out_small<false, 1>(side_job(d), it, d.nchunk);
    else glue_out_small<false, 2>(side_job(d), it, d.nchunk);
}

__global__ void __launch_bounds__(32 * kSmallWarps) k_glue_in_small(const __grid_constant__ GlueArgs a) {
    grid_dep_launch_dependents();
    if (a.L <= 8) glue_in_small<1>(a);
    else glue_in_small<2>(a);
}

template <bool PROD>
__global__ void __launch_bounds__(kThreads) k_glue_out(const __grid_constant__ GlueArgs a) {
    __shared__ __align__(16) float buf[64][65];
    __shared__ __align__(16) float buf2[PROD ? 64 : 1][65];
    __shared__ float red[32];
    grid_dep_launch_dependents();
    if ((int)blockIdx.x >= a.glue_ctas) {             // an extra output rotation (segment path)
        const GlueSide& d = side_of(a, blockIdx.x);
        const int l = blockIdx.x - d.cta_begin, td = l / d.nseg;
        glue_out_seg<false>(side_job(d), td, (l - td * d.nseg) * kSeg, 0, &buf[0][0], &buf2[0][0], red);
        return;
    }
    const int t = blockIdx.x / a.nseg, s = blockIdx.x - t * a.nseg;
    const int seg0 = s * kSeg;
    if (a.path == 2) {
        glue_out_seg<PROD>(glue_job(a), t, seg0, blockIdx.x, &buf[0][0], &buf2[0][0], red);
        return;
    }
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
    __shared__ __align__(16) float buf[64][65];
    __shared__ float s_inv;
    grid_dep_launch_dependents();
    const int per_next = a.T * a.nseg;
    const int jn = blockIdx.x / per_next;
    const int rem = blockIdx.x - jn * per_next;
    const int t = rem / a.nseg, s = rem - t * a.nseg;
    const int seg0 = s * kSeg;
    const GlueNext& nx = a.next[jn];
    if (a.path == 2) {
        glue_in_seg(a, nx, t, seg0, rem, per_next, &buf[0][0]);
        return;
    }
    const int count = a.M - seg0 < kSeg ? a.M - seg0 : kSeg;
    const size_t row = (size_t)t * a.M + seg0;
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
int glue_work_floats(int M, int T) {
    // one partial sum per (token, chunk) on the register path (b <= 512), else per (token,
    // 4096-element segment); a call may fall back from the register path to the tile path
    const int segs = glue_segments(M), b = hadamard_block(M);
    if (b > 512) return T * segs;
    int L = 0;
    while ((1 << L) < b) ++L;
    const int chunks = (M + reg_chunk(L) - 1) / reg_chunk(L);
    return T * (chunks > segs ? chunks : segs);
}

cudaError_t launch_glue(GlueArgs& a, cudaStream_t stream) {
    const int b = hadamard_block(a.M);
    int L = 0;
    while ((1 << L) < b) ++L;
    a.L = L;
    a.scale = (float)(1.0 / sqrt((double)b));
    a.NB = n_pad(a.T) / 8;
    a.nseg = glue_segments(a.M);
    auto al = [](const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) & (n - 1)) == 0; };
    bool reg = b <= 512 && a.M % 8 == 0 && al(a.za, 16) && al(a.zb, 16) && al(a.h, 16) && al(a.sa, 8) && al(a.sb, 8);
    for (int j = 0; j < a.nnext; ++j) reg = reg && al(a.next[j].sign_in, 8);
    const bool seg = b >= 1024 && al(a.h, 16) && al(a.sa, 8) && al(a.sb, 8);
    a.path = reg ? 3 : (seg ? 2 : 0);
    a.nchunk = (a.M + reg_chunk(L) - 1) / reg_chunk(L);
    // Side rotations whose block size puts them on the glue's path (register or segment) ride
    // in its first launch as extra CTAs; any other runs in a grouped rotation launch of its own.
    a.glue_ctas = a.path == 3 ? a.T * a.nchunk : a.T * a.nseg;
    long long items = a.glue_ctas;
    RotArgs rest = {};
    int keep = 0;
    for (int k = 0; k < a.nside; ++k) {
        GlueSide d = a.side[k];
        const int bs = hadamard_block(d.M);
        int Ls = 0;
        while ((1 << Ls) < bs) ++Ls;
        d.L = Ls;
        d.scale = (float)(1.0 / sqrt((double)bs));
        d.nseg = glue_segments(d.M);
        d.nchunk = (d.M + reg_chunk(Ls) - 1) / reg_chunk(Ls);
        const bool ok = a.path == 3 ? (bs <= 512 && d.M % 8 == 0 && al(d.z, 16) && al(d.y, 16) && al(d.s, 8))
                                    : (a.path == 2 && bs >= 1024 && al(d.y, 16) && al(d.s, 8));
        if (ok) {
            d.cta_begin = (int)items;
            items += (long long)a.T * (a.path == 3 ? d.nchunk : d.nseg);
            a.side[keep++] = d;
        } else {
            RotTask& r = rest.task[rest.ntasks++];
            r = RotTask{};
            r.x = d.z;
            r.signs = d.s;
            r.y = d.y;
            r.n = (unsigned)d.M;
        }
    }
    a.nside = keep;
    if (items >= (1LL << 31)) return cudaErrorInvalidValue;
    cudaError_t e;
    if (a.path == 3) {                 // one-warp CTAs, one (token, chunk) per warp
        const int ctas = (int)((items + kSmallWarps - 1) / kSmallWarps);
        const int glue = (a.glue_ctas + kSmallWarps - 1) / kSmallWarps;
        const dim3 sblk(32 * kSmallWarps);
        e = a.zb != nullptr ? launch_pdl(k_glue_out_small<true>, dim3(ctas), sblk, 0, stream, a)
                            : launch_pdl(k_glue_out_small<false>, dim3(ctas), sblk, 0, stream, a);
        if (e == cudaSuccess && a.nnext > 0) e = launch_pdl(k_glue_in_small, dim3(a.nnext * glue), sblk, 0, stream, a);
    } else {
        const dim3 blk(kThreads);
        e = a.zb != nullptr ? launch_pdl(k_glue_out<true>, dim3((unsigned)items), blk, 0, stream, a)
                            : launch_pdl(k_glue_out<false>, dim3((unsigned)items), blk, 0, stream, a);
        if (e == cudaSuccess && a.nnext > 0) e = launch_pdl(k_glue_in, dim3(a.nnext * a.T * a.nseg), blk, 0, stream, a);
    }
    if (e == cudaSuccess && rest.ntasks > 0) e = launch_rotate_group(rest, 0, 1, a.T, stream);
    return e;
}

}  // namespace nest
