// Nested KV4/KV8 cache (BitNest paper, Section 3.4 and Appendix A.2, Eq. (11)-(14)):
// quantise-on-write of the key or value vectors of new tokens, and decode attention that
// reads either view of the same cache.
//
// Cache layout (one for keys, one for values), d = 128 per head:
//   base  [H][Lmax][64]: byte i of a row holds dims 2i (low nibble) and 2i+1 (high
//                        nibble), stored q4 + 8;
//   ref   [H][Lmax][64]: the refinement codes q_r + 8, same layout;
//   scale [H][Lmax]:     fp16 s = max|x| / 7.
// The KV4 view reads base + scale (66 bytes per row), the KV8 view base + ref + scale
// (130 bytes per row): the draft never touches the refinement plane.
#include <type_traits>

#include "nest_device.cuh"
#include "nest_internal.h"

namespace nest {
namespace {

constexpr int kD = 128;

// One warp per (token, head): lane l owns dims 4l .. 4l+3.  Decisions in fp32 with
// each operation rounded on its own (no contraction), so that the codes are those of
// the definition, bit for bit:  s = fp16(max|x| / 7);  q4 = clip(rint(x / s), -8, 7);
// q_r = clip(rint((x - q4 s) / (s / 16)), -8, 7).
template <bool BF16>
__global__ void k_kv_write(const void* __restrict__ x, int T, int H, int pos0, int Lmax,
                           uint8_t* __restrict__ base, uint8_t* __restrict__ ref, uint16_t* __restrict__ scale) {
    grid_dep_launch_dependents();
    const int w = (int)((blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    grid_dep_wait();
    if (w >= T * H) return;
    const int t = w / H, h = w - t * H;
    const size_t src = ((size_t)t * H + h) * kD + 4 * lane;
    float v[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
        v[e] = BF16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(x)[src + e])
                    : reinterpret_cast<const float*>(x)[src + e];
    float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const __half s16 = __float2half_rn(__fdiv_rn(amax, 7.0f));
    const float s = __half2float(s16);
    const float sref = __fdiv_rn(s, 16.0f);
    uint32_t u4 = 0, ur = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        float a = 0.0f, b = 0.0f;
        if (s > 0.0f) {
            a = fminf(fmaxf(rintf(__fdiv_rn(v[e], s)), -8.0f), 7.0f);
            const float r = __fsub_rn(v[e], __fmul_rn(a, s));
            b = fminf(fmaxf(rintf(__fdiv_rn(r, sref)), -8.0f), 7.0f);
        }
        u4 |= (uint32_t)((int)a + 8) << (4 * e);
        ur |= (uint32_t)((int)b + 8) << (4 * e);
    }
    const size_t row = (size_t)h * Lmax + pos0 + t;
    *reinterpret_cast<uint16_t*>(base + row * (kD / 2) + 2 * lane) = (uint16_t)u4;
    *reinterpret_cast<uint16_t*>(ref + row * (kD / 2) + 2 * lane) = (uint16_t)ur;
    if (lane == 0) scale[row] = __half_as_ushort(s16);
}

constexpr int kAttnWarps = 4;
constexpr int kAttnThreads = 32 * kAttnWarps;
constexpr int kRowsPerTile = 16;           // query rows (token, head-in-group) per CTA

// The 4-bit value pairs of one byte, as floats: code - 8 for the low and high nibble.
__device__ __forceinline__ void nib2(uint32_t byte, float& lo, float& hi) {
    lo = (float)((int)(byte & 15u) - 8);
    hi = (float)((int)((byte >> 4) & 15u) - 8);
}

// Split over positions: CTA (h, split, tile) handles KV head h, a contiguous range of
// positions and up to 16 query rows (token t, group member g) of that head.  Per warp,
// 32 positions at a time: lane j computes the scores of position j for every row
// (dequantising the key row on the fly), the warp updates its online softmax, then
// lane l accumulates dims 4l..4l+3 of p * v over the 32 positions.  The warps' states
// are merged in shared memory; the split's (max, sum, output) go to `work`.
template <int NR>
__global__ void __launch_bounds__(kAttnThreads, NR <= 4 ? 4 : 2)
k_kv_attn(const __grid_constant__ KvAttnArgs a) {
    __shared__ float sq[NR][kD];                    // queries of the tile, scaled by log2(e)/sqrt(d)
    __shared__ float sm[kAttnWarps][NR];
    __shared__ float sl[kAttnWarps][NR];
    __shared__ float so[kAttnWarps][NR][kD];
    grid_dep_launch_dependents();
    const int h = blockIdx.x, split = blockIdx.y, tile = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int R = a.T * a.G;                        // rows of this KV head
    const int r0 = tile * kRowsPerTile;
    const int nr = R - r0 < NR ? R - r0 : NR;
    const int per = (a.L + a.nsplit - 1) / a.nsplit;
    const int p0 = split * per, p1 = p0 + per < a.L ? p0 + per : a.L;
    grid_dep_wait();                                // queries and cache come from earlier kernels

    const float qscale = 1.4426950408889634f / sqrtf((float)kD);
    for (int i = threadIdx.x; i < NR * kD; i += kAttnThreads) {
        const int rr = i / kD, dd = i % kD;
        float val = 0.0f;
        if (rr < nr) {
            const int row = r0 + rr, t = row / a.G, g = row % a.G;
            const size_t qi = ((size_t)t * a.Hq + (size_t)h * a.G + g) * kD + dd;
            val = a.q_bf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(a.q)[qi])
                           : reinterpret_cast<const float*>(a.q)[qi];
        }
        sq[rr][dd] = val * qscale;
    }
    __syncthreads();

    int vis[NR];                          // positions visible to each row
#pragma unroll
    for (int rr = 0; rr < NR; ++rr) vis[rr] = rr < nr ? a.L - a.T + (r0 + rr) / a.G + 1 : 0;
    float m[NR], l[NR], o[NR][4];
#pragma unroll
    for (int rr = 0; rr < NR; ++rr) {
        m[rr] = -INFINITY;
        l[rr] = 0.0f;
        o[rr][0] = o[rr][1] = o[rr][2] = o[rr][3] = 0.0f;
    }
    const size_t hrow = (size_t)h * a.Lmax;
    const int recent0 = a.L - a.recent_n;           // positions >= recent0 read at KV8 in the draft view

    for (int pt = p0 + 32 * warp; pt < p1; pt += 32 * kAttnWarps) {
        // scores of position p = pt + lane
        const int p = pt + lane;
        const bool valid = p < p1;
        float sc[NR];
#pragma unroll
        for (int rr = 0; rr < NR; ++rr) sc[rr] = 0.0f;
        if (valid) {
            float part[kD / 32][NR];                 // one partial sum per 32-dim chunk: four independent chains
#pragma unroll
            for (int c = 0; c < kD / 32; ++c)
#pragma unroll
                for (int rr = 0; rr < NR; ++rr) part[c][rr] = 0.0f;
            const bool kv8 = a.view == 8 || p >= recent0;
            const uint8_t* kb = a.kbase + (hrow + p) * (kD / 2);
            const uint8_t* kr = a.kref + (hrow + p) * (kD / 2);
            const float ks = __half2float(__ushort_as_half(a.kscale[hrow + p]));
#pragma unroll
            for (int c = 0; c < kD / 32; ++c) {      // 32 dims = 16 bytes per step
                const uint4 bb = *reinterpret_cast<const uint4*>(kb + 16 * c);
                uint4 rb = make_uint4(0u, 0u, 0u, 0u);
                if (kv8) rb = *reinterpret_cast<const uint4*>(kr + 16 * c);
                const uint32_t bw[4] = {bb.x, bb.y, bb.z, bb.w};
                const uint32_t rw[4] = {rb.x, rb.y, rb.z, rb.w};
#pragma unroll
                for (int wd = 0; wd < 4; ++wd) {
#pragma unroll
                    for (int by = 0; by < 4; ++by) {
                        float b0, b1;
                        nib2(bw[wd] >> (8 * by), b0, b1);
                        float k0 = b0, k1 = b1;
                        if (kv8) {
                            float r0f, r1f;
                            nib2(rw[wd] >> (8 * by), r0f, r1f);
                            k0 = fmaf(b0, 16.0f, r0f) * 0.0625f;
                            k1 = fmaf(b1, 16.0f, r1f) * 0.0625f;
                        }
                        const int dd = 32 * c + 8 * wd + 2 * by;
#pragma unroll
                        for (int rr = 0; rr < NR; ++rr) {
                            if (rr < nr) part[c][rr] = fmaf(sq[rr][dd], k0, fmaf(sq[rr][dd + 1], k1, part[c][rr]));
                        }
                    }
                }
            }
#pragma unroll
            for (int rr = 0; rr < NR; ++rr) sc[rr] = ((part[0][rr] + part[1][rr]) + (part[2][rr] + part[3][rr])) * ks;
        }
        // online softmax per row (base 2), then p * v
        float pj[NR];
#pragma unroll
        for (int rr = 0; rr < NR; ++rr) {
            if (rr >= nr) { pj[rr] = 0.0f; continue; }
            const float s = (valid && p < vis[rr]) ? sc[rr] : -INFINITY;
            float mx = s;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            const float mn = fmaxf(m[rr], mx);
            if (mn == -INFINITY) { pj[rr] = 0.0f; continue; }
            const float corr = exp2f(m[rr] - mn);
            const float pv = s == -INFINITY ? 0.0f : exp2f(s - mn);
            float sum = pv;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
            l[rr] = l[rr] * corr + sum;
            o[rr][0] *= corr; o[rr][1] *= corr; o[rr][2] *= corr; o[rr][3] *= corr;
            m[rr] = mn;
            pj[rr] = pv;
        }
        const int nvalid = p1 - pt < 32 ? p1 - pt : 32;
        for (int jb = 0; jb < nvalid; jb += 8) {
            // the next 8 positions' value bytes, loaded before any is used
            uint16_t vb[8], vr[8];
            float vs[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int pp = pt + jb + u;
                vb[u] = vr[u] = 0x8888u;
                vs[u] = 0.0f;
                if (jb + u < nvalid) {
                    vb[u] = *reinterpret_cast<const uint16_t*>(a.vbase + (hrow + pp) * (kD / 2) + 2 * lane);
                    if (a.view == 8 || pp >= recent0)
                        vr[u] = *reinterpret_cast<const uint16_t*>(a.vref + (hrow + pp) * (kD / 2) + 2 * lane);
                    vs[u] = __half2float(__ushort_as_half(a.vscale[hrow + pp]));
                }
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int pp = pt + jb + u;
                const bool kv8 = a.view == 8 || pp >= recent0;
                float b0, b1, b2, b3;
                nib2(vb[u], b0, b1);
                nib2((uint32_t)vb[u] >> 8, b2, b3);
                float vv[4] = {b0, b1, b2, b3};
                if (kv8) {
                    float c0, c1, c2, c3;
                    nib2(vr[u], c0, c1);
                    nib2((uint32_t)vr[u] >> 8, c2, c3);
                    vv[0] = fmaf(b0, 16.0f, c0) * 0.0625f;
                    vv[1] = fmaf(b1, 16.0f, c1) * 0.0625f;
                    vv[2] = fmaf(b2, 16.0f, c2) * 0.0625f;
                    vv[3] = fmaf(b3, 16.0f, c3) * 0.0625f;
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) vv[e] *= vs[u];
#pragma unroll
                for (int rr = 0; rr < NR; ++rr) {
                    if (rr >= nr) continue;
                    const float w = __shfl_sync(0xffffffffu, pj[rr], (jb + u) & 31);
                    o[rr][0] = fmaf(w, vv[0], o[rr][0]);
                    o[rr][1] = fmaf(w, vv[1], o[rr][1]);
                    o[rr][2] = fmaf(w, vv[2], o[rr][2]);
                    o[rr][3] = fmaf(w, vv[3], o[rr][3]);
                }
            }
        }
    }

    // merge the warps' states, then write this split's partial result
#pragma unroll
    for (int rr = 0; rr < NR; ++rr) {
        if (lane == 0) { sm[warp][rr] = m[rr]; sl[warp][rr] = l[rr]; }
#pragma unroll
        for (int e = 0; e < 4; ++e) so[warp][rr][4 * lane + e] = o[rr][e];
    }
    __syncthreads();
    for (int i = threadIdx.x; i < nr * kD; i += kAttnThreads) {
        const int rr = i / kD, dd = i % kD;
        float M = -INFINITY;
        for (int w2 = 0; w2 < kAttnWarps; ++w2) M = fmaxf(M, sm[w2][rr]);
        float L = 0.0f, O = 0.0f;
        if (M != -INFINITY) {
            for (int w2 = 0; w2 < kAttnWarps; ++w2) {
                const float f = sm[w2][rr] == -INFINITY ? 0.0f : exp2f(sm[w2][rr] - M);
                L += f * sl[w2][rr];
                O += f * so[w2][rr][dd];
            }
        }
        const size_t slot = (((size_t)h * a.ntiles + tile) * a.nsplit + split) * kRowsPerTile + rr;
        float* wp = a.work + slot * (kD + 2);
        wp[2 + dd] = O;
        if (dd == 0) { wp[0] = M; wp[1] = L; }
    }
}

// ---------------------------------------------------------------------------
// Tensor-core decode attention (mma.sync m16n8k16), 16 positions per warp step.
//
// QK: S[pos][row] = K[pos][:] . Q[row][:] with A = the key codes (16 positions x 16 dims
// per k-step), B = the queries (16 dims x 8 rows).  A dot product may take its dims in any
// order shared by both operands, and the decode below is cheapest when each 32-bit word of
// a row (dims 8w .. 8w+7, byte i = dims 2i | 2i+1) comes out as the fp16 pairs
// (8w + j, 8w + j + 4), j = 0..3.  Thread q of a quad owns bytes 16q .. 16q+15 of its two
// key rows (one 16-byte load per row, the quad reading the row's 64 bytes); word w of
// them feeds k-steps 2w (pairs j = 0, 1) and 2w + 1 (pairs j = 2, 3), and the query
// fragments are packed in the same order.
// Codes: the byte (u4 << 4) | u_r minus 136 is the KV8 code 16 q4 + q_r, and a position
// read at KV4 takes u_r = 8, giving 16 q4, so every position's scale is s / 16, applied to
// its scores (keys) and to its probabilities (values).  Blocks read wholly at KV4 take a
// shorter decode of the base word alone.
// PV: O^T[dim][row] += V^T[dim][pos] P^T[pos][row]: A = V^T loaded with ldmatrix.trans
// from the block's values decoded to fp16 in shared memory (each 8-dim group in the pair
// order above, undone when the output is written), B = P^T from the score fragments
// transposed in registers with movmatrix.
// ---------------------------------------------------------------------------

constexpr int kTcWarps = 4;
constexpr float kLazy = 8.0f;             // log2 headroom before the outputs are rescaled
constexpr int kTcThreads = 32 * kTcWarps;
constexpr int kVPitch = 272;              // bytes per position row of a warp's fp16 value block (bank-conflict free)

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
    return h2_as_u32(__floats2half2_rn(lo, hi));
}

__device__ __forceinline__ void mma16816f(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                                  uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

// Logic helpers with one immediate each.  A single lop3 takes one 32-bit immediate, so
// an expression with two constants (a mask and the fp16 exponent bytes) costs two; the
// kernels keep the second constant in a register (see kv_consts) and use these.
template <uint32_t M>
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t c) {      // (a & M) | c
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "n"(M), "r"(c));
    return d;
}
__device__ __forceinline__ uint32_t select_bits(uint32_t a, uint32_t b, uint32_t m) {   // (a & m) | (b & ~m)
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xE4;" : "=r"(d) : "r"(a), "r"(b), "r"(m));
    return d;
}

// Constants of the decode, held in registers: the fp16 exponent bytes 0x64 of a pair
// (e64), of four bytes (e6464) and the high-nibble mask (mhi).  They are built from a
// kernel parameter (x >> 31 of a non-negative count is 0) so that they are not folded
// back into immediates.
struct KvConsts {
    uint32_t e64, e6464, mhi;
};
__device__ __forceinline__ KvConsts kv_consts(int nonneg) {
    const uint32_t z = (uint32_t)nonneg >> 31;
    return {0x64006400u | z, 0x64646464u | z, 0xF0F0F0F0u | z};
}

// One 32-bit base word b and refinement word r (dims 8w .. 8w+7 of a row, byte i = dims
// 2i | 2i+1) as the fp16 codes 16 u4 + u_r - 136 in pairs out[j] = (dim j, dim j + 4).
__device__ __forceinline__ void dec8(uint32_t b, uint32_t r, const KvConsts& k, uint32_t (&out)[4]) {
    const uint32_t ev = select_bits(b << 4, r, k.mhi);          // byte i: dim 2i
    const uint32_t od = select_bits(b, r >> 4, k.mhi);          // byte i: dim 2i + 1
    const __half2 off = __float2half2_rn(1024.0f + 136.0f);
    out[0] = h2_as_u32(__hsub2(u32_as_h2(prmt(ev, k.e6464, 0x4240u)), off));   // dims 0, 4
    out[1] = h2_as_u32(__hsub2(u32_as_h2(prmt(od, k.e6464, 0x4240u)), off));   // dims 1, 5
    out[2] = h2_as_u32(__hsub2(u32_as_h2(prmt(ev, k.e6464, 0x4341u)), off));   // dims 2, 6
    out[3] = h2_as_u32(__hsub2(u32_as_h2(prmt(od, k.e6464, 0x4341u)), off));   // dims 3, 7
}

// The same word read at KV4 (u_r = 8): 16 u4 - 128 in the same pair order.  A nibble in
// bits 0-3 of an fp16 with exponent field 0x64 reads as 1024 + u4, one in bits 4-7 as
// 1024 + 16 u4; both are mapped to 16 u4 - 128 exactly by one fp16 operation.
__device__ __forceinline__ void dec4(uint32_t b, const KvConsts& k, uint32_t (&out)[4]) {
    const uint32_t b8 = b >> 8;
    const __half2 x16 = __float2half2_rn(16.0f), o16 = __float2half2_rn(-16.0f * 1024.0f - 128.0f);
    const __half2 o1 = __float2half2_rn(1024.0f + 128.0f);
    out[0] = h2_as_u32(__hfma2(u32_as_h2(and_or<0x000F000Fu>(b, k.e64)), x16, o16));    // dims 0, 4
    out[1] = h2_as_u32(__hsub2(u32_as_h2(and_or<0x00F000F0u>(b, k.e64)), o1));          // dims 1, 5
    out[2] = h2_as_u32(__hfma2(u32_as_h2(and_or<0x000F000Fu>(b8, k.e64)), x16, o16));   // dims 2, 6
    out[3] = h2_as_u32(__hsub2(u32_as_h2(and_or<0x00F000F0u>(b8, k.e64)), o1));         // dims 3, 7
}

// Dim of slot x of the decoded order (pairs (j, j + 4) inside each group of 8).
__device__ __forceinline__ int slot_dim(int x) { return (x & ~7) | ((x >> 1) & 3) | ((x & 1) << 2); }

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <int NRT>
constexpr int kv_tc_smem() {
    constexpr int v = kTcWarps * 16 * kVPitch, o = kTcWarps * 8 * NRT * (kD + 1) * 4;
    return (v > o ? v : o) + 2 * kTcWarps * 8 * NRT * 4;
}

template <int NRT>
__global__ void __launch_bounds__(kTcThreads, NRT == 1 ? 4 : 2)
k_kv_attn_tc(const __grid_constant__ KvAttnArgs a) {
    constexpr int NRm = 8 * NRT;          // query rows per CTA
    // dynamic shared memory: the warps' fp16 value blocks, later reused for the merge of
    // the warps' outputs; the warps' softmax states after the larger of the two
    extern __shared__ __align__(16) uint8_t dsm[];
    constexpr int kVBytes = kTcWarps * 16 * kVPitch;
    constexpr int kOBytes = kTcWarps * NRm * (kD + 1) * 4;
    constexpr int kFront = kVBytes > kOBytes ? kVBytes : kOBytes;
    uint8_t (*svb)[16 * kVPitch] = reinterpret_cast<uint8_t (*)[16 * kVPitch]>(dsm);
    float (*so)[NRm][kD + 1] = reinterpret_cast<float (*)[NRm][kD + 1]>(dsm);
    float (*sm)[NRm] = reinterpret_cast<float (*)[NRm]>(dsm + kFront);
    float (*sl)[NRm] = reinterpret_cast<float (*)[NRm]>(dsm + kFront + kTcWarps * NRm * 4);
    grid_dep_launch_dependents();
    const int h = blockIdx.x, split = blockIdx.y, tile = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, q = lane & 3;
    const int R = a.T * a.G;
    const int r0 = tile * NRm;
    const int per = (a.L + a.nsplit - 1) / a.nsplit;
    const int p0 = split * per, p1 = p0 + per < a.L ? p0 + per : a.L;
    const size_t hrow = (size_t)h * a.Lmax;
    const int recent0 = a.L - a.recent_n;
    grid_dep_wait();

    // B fragments of the queries (fp16, scaled by log2(e) / sqrt(d)), rows 8nt + g
    uint32_t qb[NRT][8][2];
    const float qscale = 1.4426950408889634f / sqrtf((float)kD);
#pragma unroll
    for (int nt = 0; nt < NRT; ++nt) {
        const int row = r0 + 8 * nt + g;
        const bool ok = row < R;
        const int t = ok ? row / a.G : 0, gg = ok ? row % a.G : 0;
        const size_t qi = ((size_t)t * a.Hq + (size_t)h * a.G + gg) * kD;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            float v[8];                       // dims 32q + 8w .. +7
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int dd = 32 * q + 8 * w + e;
                float x = 0.0f;
                if (ok) x = a.q_bf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(a.q)[qi + dd])
                                     : reinterpret_cast<const float*>(a.q)[qi + dd];
                v[e] = x * qscale;
            }
            qb[nt][2 * w][0] = pack_h2(v[0], v[4]);
            qb[nt][2 * w][1] = pack_h2(v[1], v[5]);
            qb[nt][2 * w + 1][0] = pack_h2(v[2], v[6]);
            qb[nt][2 * w + 1][1] = pack_h2(v[3], v[7]);
        }
    }
    // visible positions of the thread's two rows per n-tile (rows 8nt + 2q, 8nt + 2q + 1)
    int vis[NRT][2];
#pragma unroll
    for (int nt = 0; nt < NRT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int row = r0 + 8 * nt + 2 * q + e;
            vis[nt][e] = row < R ? a.L - a.T + row / a.G + 1 : 0;
        }

    // positions below vis_all are inside the split and visible to every row of the CTA
    const int vis_r0 = a.L - a.T + r0 / a.G + 1;     // row r0 (the CTA's earliest token) sees the fewest
    const int vis_all = vis_r0 < p1 ? vis_r0 : p1;
    float m[NRT][2], l[NRT][2], o[NRT][8][4];
#pragma unroll
    for (int nt = 0; nt < NRT; ++nt) {
        m[nt][0] = m[nt][1] = -INFINITY;
        l[nt][0] = l[nt][1] = 0.0f;
#pragma unroll
        for (int dt = 0; dt < 8; ++dt) o[nt][dt][0] = o[nt][dt][1] = o[nt][dt][2] = o[nt][dt][3] = 0.0f;
    }
    uint8_t* vblk = svb[warp];
    const uint32_t vblk_s = smem_u32(vblk);
    // ldmatrix row addresses of matrix i/8, row i%8: positions (i%8) + 8*((i/8)/2), dims +8*((i/8)%2)
    const int lm = lane >> 3, lr = lane & 7;
    const uint32_t lda = vblk_s + (uint32_t)((lr + 8 * (lm >> 1)) * kVPitch + 16 * (lm & 1));

    // Raw words of one 16-position block: keys (rows g, g+8; bytes 16q..16q+15) and values
    // (position lane/2, dims 64*(lane&1) ..), base and refinement planes, and the fp16
    // scales of positions g, g+8.  The next block's value words are loaded as soon as the
    // current ones are decoded, its key words as soon as the scores are issued, so one
    // set of registers carries both with a full iteration of lead time.
    struct Blk {
        uint4 kb[2], kr[2], vb[2], vr[2];
        uint16_t ks[2], vs[2];
    };
    const uint4 z8 = make_uint4(0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u);
    // per-lane 32-bit offsets of position 0 of the head (a plane holds fewer than 2^32
    // bytes); a block at pb adds pb rows.  The plane pointers stay kernel parameters.
    const bool view8 = a.view == 8;
    const KvConsts kc = kv_consts(a.T);
    const uint32_t krow = (uint32_t)((hrow + g) * (kD / 2)) + 16u * q;
    const uint32_t vrow = (uint32_t)((hrow + (lane >> 1)) * (kD / 2)) + 32u * (lane & 1);
    const uint32_t srow = (uint32_t)(hrow + g);
    auto ld16 = [](const uint8_t* p) { return *reinterpret_cast<const uint4*>(p); };
    // Key words of the block at pb.  Whole blocks inside the split take unguarded loads; the
    // refinement words are read only where the block's decode uses them (every position
    // at KV8, or the Recent-N window), other positions of a straddling block read u_r = 8.
    auto load_k = [&](int pb, Blk& B) {
        const bool need_ref = view8 || pb + 15 >= recent0;
        if (pb + 16 <= p1) {
            const uint32_t o = krow + (uint32_t)pb * (kD / 2);
            B.kb[0] = ld16(a.kbase + o);
            B.kb[1] = ld16(a.kbase + o + 8 * (kD / 2));
            B.ks[0] = a.kscale[srow + pb];
            B.ks[1] = a.kscale[srow + pb + 8];
            if (need_ref) {
                const bool all = view8 || pb >= recent0;
                B.kr[0] = (all || pb + g >= recent0) ? ld16(a.kref + o) : z8;
                B.kr[1] = (all || pb + g + 8 >= recent0) ? ld16(a.kref + o + 8 * (kD / 2)) : z8;
            }
            return;
        }
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int p = pb + g + 8 * e;
            const uint32_t o = krow + (uint32_t)(pb + 8 * e) * (kD / 2);
            B.kb[e] = z8;
            B.kr[e] = z8;
            B.ks[e] = 0;
            if (p < p1) {
                B.kb[e] = ld16(a.kbase + o);
                if (view8 || p >= recent0) B.kr[e] = ld16(a.kref + o);
                B.ks[e] = a.kscale[srow + pb + 8 * e];
            }
        }
    };
    auto load_v = [&](int pb, Blk& B) {
        const bool need_ref = view8 || pb + 15 >= recent0;
        const int p = pb + (lane >> 1);
        const uint32_t o = vrow + (uint32_t)pb * (kD / 2);
        if (pb + 16 <= p1) {
            B.vb[0] = ld16(a.vbase + o);
            B.vb[1] = ld16(a.vbase + o + 16);
            B.vs[0] = a.vscale[srow + pb];
            B.vs[1] = a.vscale[srow + pb + 8];
            if (need_ref) {
                const bool use = view8 || p >= recent0;
                B.vr[0] = use ? ld16(a.vref + o) : z8;
                B.vr[1] = use ? ld16(a.vref + o + 16) : z8;
            }
            return;
        }
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            B.vb[c] = z8;
            B.vr[c] = z8;
            if (p < p1) {
                B.vb[c] = ld16(a.vbase + o + 16 * c);
                if (view8 || p >= recent0) B.vr[c] = ld16(a.vref + o + 16 * c);
            }
        }
#pragma unroll
        for (int e = 0; e < 2; ++e) B.vs[e] = pb + g + 8 * e < p1 ? a.vscale[srow + pb + 8 * e] : (uint16_t)0;
    };
    Blk buf;
    int pb = p0 + 16 * warp;                  // this warp's current block
    if (pb < p1) {
        load_k(pb, buf);
        load_v(pb, buf);
    }

    // One 16-position block.  DEC: 0 decodes the base words alone (a block wholly read at
    // KV4), 1 base + refinement (KV8, or a KV4 read's Recent-N window, where positions
    // outside the window carry u_r = 8), 2 picks one of the two at run time.  MASK: the
    // block may hold positions past the split's end or past some row's causal limit.
    auto step = [&](auto dec_c, auto mask_c) {
        constexpr int DEC = decltype(dec_c)::value;
        constexpr bool MASK = decltype(mask_c)::value;
        const int pn = pb + 16 * kTcWarps;    // the warp's next block
        const bool kv8 = DEC == 1 || (DEC == 2 && (view8 || pb + 15 >= recent0));
        float ks[2], vsc[2];                  // zero past the split's end
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            ks[e] = __half2float(__ushort_as_half(buf.ks[e])) * 0.0625f;
            vsc[e] = __half2float(__ushort_as_half(buf.vs[e])) * 0.0625f;
        }
        // ---- values: thread lane decodes position pb + lane/2, dims 64*(lane&1) .. +63 into fp16 ----
        {
            uint8_t* dst = vblk + (lane >> 1) * kVPitch + 128 * (lane & 1);
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const uint32_t bw[4] = {buf.vb[c].x, buf.vb[c].y, buf.vb[c].z, buf.vb[c].w};
                const uint32_t rw[4] = {buf.vr[c].x, buf.vr[c].y, buf.vr[c].z, buf.vr[c].w};
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    uint32_t cv[4];
                    if (kv8) dec8(bw[w], rw[w], kc, cv);
                    else dec4(bw[w], kc, cv);
                    *reinterpret_cast<uint4*>(dst + 64 * c + 16 * w) = make_uint4(cv[0], cv[1], cv[2], cv[3]);
                }
            }
        }
        if (pn < p1) load_v(pn, buf);
        __syncwarp();

        // ---- scores S[pos][row]: each key word is decoded right before its two k-steps ----
        // A fragments: rows g (a0, a2), g + 8 (a1, a3); word w holds dims 32q + 8w .. +7
        float scs[NRT][2][4];                 // two independent accumulation chains per n-tile
#pragma unroll
        for (int nt = 0; nt < NRT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) scs[nt][0][e] = scs[nt][1][e] = 0.0f;
        {
            const uint32_t b0w[4] = {buf.kb[0].x, buf.kb[0].y, buf.kb[0].z, buf.kb[0].w};
            const uint32_t r0w[4] = {buf.kr[0].x, buf.kr[0].y, buf.kr[0].z, buf.kr[0].w};
            const uint32_t b1w[4] = {buf.kb[1].x, buf.kb[1].y, buf.kb[1].z, buf.kb[1].w};
            const uint32_t r1w[4] = {buf.kr[1].x, buf.kr[1].y, buf.kr[1].z, buf.kr[1].w};
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                uint32_t c0[4], c1[4];
                if (kv8) {
                    dec8(b0w[w], r0w[w], kc, c0);
                    dec8(b1w[w], r1w[w], kc, c1);
                } else {
                    dec4(b0w[w], kc, c0);
                    dec4(b1w[w], kc, c1);
                }
#pragma unroll
                for (int nt = 0; nt < NRT; ++nt) {
                    mma16816f(scs[nt][0], c0[0], c1[0], c0[1], c1[1], qb[nt][2 * w][0], qb[nt][2 * w][1]);
                    mma16816f(scs[nt][1], c0[2], c1[2], c0[3], c1[3], qb[nt][2 * w + 1][0],
                              qb[nt][2 * w + 1][1]);
                }
            }
        }
        if (pn < p1) load_k(pn, buf);
#pragma unroll
        for (int nt = 0; nt < NRT; ++nt) {
            // sc: (pos g, rows 2q, 2q+1), (pos g+8, rows 2q, 2q+1)
            float sc[4], pr[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) sc[e] = (scs[nt][0][e] + scs[nt][1][e]) * ks[e >> 1];
            if constexpr (!MASK) {
                float mx[2];
#pragma unroll
                for (int re = 0; re < 2; ++re) {
                    mx[re] = fmaxf(sc[re], sc[2 + re]);
#pragma unroll
                    for (int off = 4; off < 32; off <<= 1)
                        mx[re] = fmaxf(mx[re], __shfl_xor_sync(0xffffffffu, mx[re], off));
                }
                // The outputs are rescaled only when some row's block max exceeds its running
                // max by more than kLazy (log2 units): in between, the probabilities against the
                // kept max stay below 2^kLazy, which fp16 P and the fp32 sums hold without loss,
                // and the final merge divides by the sum taken against the same max.
                if (__any_sync(0xffffffffu, mx[0] > m[nt][0] + kLazy || mx[1] > m[nt][1] + kLazy)) {
#pragma unroll
                    for (int re = 0; re < 2; ++re) {
                        const float mn = fmaxf(m[nt][re], mx[re]);
                        const float corr = ex2(m[nt][re] - mn);  // m = -inf before the first block: 0
                        l[nt][re] *= corr;
                        m[nt][re] = mn;
#pragma unroll
                        for (int dt = 0; dt < 8; ++dt) { o[nt][dt][re] *= corr; o[nt][dt][2 + re] *= corr; }
                    }
                }
#pragma unroll
                for (int re = 0; re < 2; ++re) {
                    const float e0 = ex2(sc[re] - m[nt][re]), e1 = ex2(sc[2 + re] - m[nt][re]);
                    // per-lane partial sum under the row's common max; lanes are summed at the end
                    l[nt][re] += e0 + e1;
                    pr[re] = e0 * vsc[0];
                    pr[2 + re] = e1 * vsc[1];
                }
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int pe = pb + g + 8 * (e >> 1), re = e & 1;
                    if (!(pe < p1 && pe < vis[nt][re])) sc[e] = -INFINITY;
                }
#pragma unroll
                for (int re = 0; re < 2; ++re) {
                    float mx = fmaxf(sc[re], sc[2 + re]);
#pragma unroll
                    for (int off = 4; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
                    const float mn = fmaxf(m[nt][re], mx);
                    const float corr = mn == -INFINITY ? 1.0f : ex2(m[nt][re] - mn);
                    const float e0 = sc[re] == -INFINITY ? 0.0f : ex2(sc[re] - mn);
                    const float e1 = sc[2 + re] == -INFINITY ? 0.0f : ex2(sc[2 + re] - mn);
                    l[nt][re] = l[nt][re] * corr + (e0 + e1);
                    m[nt][re] = mn;
#pragma unroll
                    for (int dt = 0; dt < 8; ++dt) { o[nt][dt][re] *= corr; o[nt][dt][2 + re] *= corr; }
                    pr[re] = e0 * vsc[0];
                    pr[2 + re] = e1 * vsc[1];
                }
            }
            // B fragments of P^T: b0 = positions 2q, 2q+1 of row g; b1 = positions 2q+8, 2q+9
            const uint32_t pb0 = movmatrix_trans(pack_h2(pr[0], pr[1]));
            const uint32_t pb1 = movmatrix_trans(pack_h2(pr[2], pr[3]));
#pragma unroll
            for (int dt = 0; dt < 8; ++dt) {
                uint32_t v0, v1, v2, v3;
                ldmatrix_x4_trans(lda + 32 * dt, v0, v1, v2, v3);
                mma16816f(o[nt][dt], v0, v1, v2, v3, pb0, pb1);
            }
        }
        __syncwarp();
        pb = pn;
    };
    using Dec4 = std::integral_constant<int, 0>;
    using Dec8 = std::integral_constant<int, 1>;
    using DecAny = std::integral_constant<int, 2>;
    // interior blocks (inside the split, visible to every row): first those wholly before
    // a KV4 read's Recent-N window, then the rest; the last few blocks take the masked step
    if (!view8) {
        const int lim = vis_all < recent0 ? vis_all : recent0;
        while (pb + 16 <= lim) step(Dec4{}, std::false_type{});
    }
    while (pb + 16 <= vis_all) step(Dec8{}, std::false_type{});
    while (pb < p1) step(DecAny{}, std::true_type{});

    // o[nt][dt]: (dim 16dt + g, rows 2q, 2q+1), (dim 16dt + g + 8, rows 2q, 2q+1) of the n-tile
#pragma unroll
    for (int nt = 0; nt < NRT; ++nt)
#pragma unroll
        for (int re = 0; re < 2; ++re)
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) l[nt][re] += __shfl_xor_sync(0xffffffffu, l[nt][re], off);
    __syncthreads();                          // every warp is done with its value block (aliased below)
#pragma unroll
    for (int nt = 0; nt < NRT; ++nt) {
#pragma unroll
        for (int re = 0; re < 2; ++re) {
            const int rr = 8 * nt + 2 * q + re;
            if (g == 0) { sm[warp][rr] = m[nt][re]; sl[warp][rr] = l[nt][re]; }
#pragma unroll
            for (int dt = 0; dt < 8; ++dt) {
                so[warp][rr][slot_dim(16 * dt + g)] = o[nt][dt][re];
                so[warp][rr][slot_dim(16 * dt + g + 8)] = o[nt][dt][2 + re];
            }
        }
    }
    __syncthreads();
    const int nr = R - r0 < NRm ? R - r0 : NRm;
    for (int i = threadIdx.x; i < nr * kD; i += kTcThreads) {
        const int rr = i / kD, dd = i % kD;
        float M = -INFINITY;
        for (int w2 = 0; w2 < kTcWarps; ++w2) M = fmaxf(M, sm[w2][rr]);
        float L = 0.0f, O = 0.0f;
        if (M != -INFINITY) {
            for (int w2 = 0; w2 < kTcWarps; ++w2) {
                const float f = sm[w2][rr] == -INFINITY ? 0.0f : exp2f(sm[w2][rr] - M);
                L += f * sl[w2][rr];
                O += f * so[w2][rr][dd];
            }
        }
        const int rg = r0 + rr;            // row within the head
        const int tile16 = rg / kRowsPerTile, r16 = rg % kRowsPerTile;
        const size_t slot = (((size_t)h * a.ntiles + tile16) * a.nsplit + split) * kRowsPerTile + r16;
        float* wp = a.work + slot * (kD + 2);
        wp[2 + dd] = O;
        if (dd == 0) { wp[0] = M; wp[1] = L; }
    }
}

// ---------------------------------------------------------------------------
// Paired variant for more than 16 query rows per KV head (the verify's T tokens x G heads):
// a CTA of four warps in two pairs takes 32 rows.  Both warps of a pair walk the same
// 16-position blocks; warp 0 decodes the block's keys and warp 1 its values into fp16 tiles
// in shared memory (slot order as above), and each warp then computes the scores, softmax
// and PV of its own 16 rows from the two tiles (ldmatrix for the keys as A, ldmatrix.trans
// for the values).  The cache is read and decoded once per 32 rows instead of once per 16.
// A pair alternates between two tile buffers, so one pair barrier per block orders the
// writes of a block after the partner's reads of the block two steps back.
// ---------------------------------------------------------------------------
constexpr int kPairWarps = 4;
constexpr int kPairThreads = 32 * kPairWarps;
constexpr int kPairRows = 32;
constexpr int kPairTile = 16 * kVPitch;                          // one decoded 16-position tile
constexpr int kPairBuf = 2 * kPairTile + 2 * 16 * 4;             // key tile, value tile, their scales
constexpr int kPairFront = (kPairWarps / 2) * 2 * kPairBuf;      // two pairs, two buffers each
constexpr int kPairMerge = kPairWarps * 16 * (kD + 1) * 4;
constexpr int kPairFrontMax = kPairFront > kPairMerge ? kPairFront : kPairMerge;
constexpr int kPairSmem = kPairFrontMax + 2 * kPairWarps * 16 * 4;

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

__global__ void __launch_bounds__(kPairThreads, 3)
k_kv_attn_pair(const __grid_constant__ KvAttnArgs a) {
    // dynamic shared memory: the pairs' tile buffers, later reused for the merge of the
    // warps' outputs; the warps' softmax states after the larger of the two
    extern __shared__ __align__(16) uint8_t dsm[];
    float (*so)[16][kD + 1] = reinterpret_cast<float (*)[16][kD + 1]>(dsm);
    float (*sm)[16] = reinterpret_cast<float (*)[16]>(dsm + kPairFrontMax);
    float (*sl)[16] = reinterpret_cast<float (*)[16]>(dsm + kPairFrontMax + kPairWarps * 16 * 4);
    grid_dep_launch_dependents();
    const int h = blockIdx.x, split = blockIdx.y, tile = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int pair = warp >> 1, role = warp & 1;       // role 0 decodes the keys, 1 the values
    const int g = lane >> 2, q = lane & 3;
    const int R = a.T * a.G;
    const int r0 = tile * kPairRows + 16 * role;       // the warp's first row
    const int per = (a.L + a.nsplit - 1) / a.nsplit;
    const int p0 = split * per, p1 = p0 + per < a.L ? p0 + per : a.L;
    const size_t hrow = (size_t)h * a.Lmax;
    const int recent0 = a.L - a.recent_n;
    const bool view8 = a.view == 8;
    const KvConsts kc = kv_consts(a.T);
    uint8_t* pbuf = dsm + pair * 2 * kPairBuf;
    grid_dep_wait();

    // B fragments of the queries in the tiles' slot order: in k-step s, slots 16s + 2q + e
    // and 16s + 8 + 2q + e hold dims 16s + q + 4e and 16s + 8 + q + 4e
    uint32_t qb[2][8][2];
    const float qscale = 1.4426950408889634f / sqrtf((float)kD);
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        const int row = r0 + 8 * nt + g;
        const bool ok = row < R;
        const int t = ok ? row / a.G : 0, gg = ok ? row % a.G : 0;
        const size_t qi = ((size_t)t * a.Hq + (size_t)h * a.G + gg) * kD;
        auto qv = [&](int dd) {
            float x = 0.0f;
            if (ok) x = a.q_bf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(a.q)[qi + dd])
                                 : reinterpret_cast<const float*>(a.q)[qi + dd];
            return x * qscale;
        };
#pragma unroll
        for (int st = 0; st < 8; ++st) {
            qb[nt][st][0] = pack_h2(qv(16 * st + q), qv(16 * st + q + 4));
            qb[nt][st][1] = pack_h2(qv(16 * st + 8 + q), qv(16 * st + 12 + q));
        }
    }
    int vis[2][2];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int row = r0 + 8 * nt + 2 * q + e;
            vis[nt][e] = row < R ? a.L - a.T + row / a.G + 1 : 0;
        }
    const int vis_r0 = a.L - a.T + r0 / a.G + 1;
    const int vis_all = vis_r0 < p1 ? vis_r0 : p1;

    float m[2][2], l[2][2], o[2][8][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        m[nt][0] = m[nt][1] = -INFINITY;
        l[nt][0] = l[nt][1] = 0.0f;
#pragma unroll
        for (int dt = 0; dt < 8; ++dt) o[nt][dt][0] = o[nt][dt][1] = o[nt][dt][2] = o[nt][dt][3] = 0.0f;
    }

    // The warp's loads: role 0 the key rows, role 1 the value rows of a block; lane reads
    // position pb + lane/2, bytes 32 (lane & 1) .. +31 of the base and refinement rows, and
    // the scale of position pb + (lane & 15).
    const uint8_t* bplane = role ? a.vbase : a.kbase;
    const uint8_t* rplane = role ? a.vref : a.kref;
    const uint16_t* splane = role ? a.vscale : a.kscale;
    const uint32_t wrow = (uint32_t)((hrow + (lane >> 1)) * (kD / 2)) + 32u * (lane & 1);
    const uint32_t srow = (uint32_t)hrow;
    const uint4 z8 = make_uint4(0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u);
    auto ld16 = [](const uint8_t* ptr) { return *reinterpret_cast<const uint4*>(ptr); };
    struct Blk {
        uint4 b[2], r[2];
        uint16_t sc;
    };
    auto load = [&](int pb, Blk& B) {
        const int p = pb + (lane >> 1), ps = pb + (lane & 15);
        const uint32_t o_ = wrow + (uint32_t)pb * (kD / 2);
        const bool need_ref = view8 || pb + 15 >= recent0;
        B.sc = ps < p1 ? splane[srow + ps] : (uint16_t)0;
        if (pb + 16 <= p1) {
            B.b[0] = ld16(bplane + o_);
            B.b[1] = ld16(bplane + o_ + 16);
            if (need_ref) {
                const bool use = view8 || p >= recent0;
                B.r[0] = use ? ld16(rplane + o_) : z8;
                B.r[1] = use ? ld16(rplane + o_ + 16) : z8;
            }
            return;
        }
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            B.b[c] = z8;
            B.r[c] = z8;
            if (p < p1) {
                B.b[c] = ld16(bplane + o_ + 16 * c);
                if (view8 || p >= recent0) B.r[c] = ld16(rplane + o_ + 16 * c);
            }
        }
    };
    // ldmatrix row addresses inside a tile: keys (A, rows = positions) and values (A = V^T)
    const uint32_t koff = (uint32_t)(((lane & 7) + 8 * ((lane >> 3) & 1)) * kVPitch + 16 * (lane >> 4));
    const int lm = lane >> 3, lr = lane & 7;
    const uint32_t voff = (uint32_t)((lr + 8 * (lm >> 1)) * kVPitch + 16 * (lm & 1));

    int pb = p0 + 16 * pair, it = 0;
    Blk buf;
    if (pb < p1) load(pb, buf);

    auto step = [&](auto dec_c, auto mask_c) {
        constexpr int DEC = decltype(dec_c)::value;
        constexpr bool MASK = decltype(mask_c)::value;
        const int pn = pb + 16 * (kPairWarps / 2);
        const bool kv8 = DEC == 1 || (DEC == 2 && (view8 || pb + 15 >= recent0));
        uint8_t* bt = pbuf + (it & 1) * kPairBuf;
        float* ssc = reinterpret_cast<float*>(bt + 2 * kPairTile);     // 16 key scales, 16 value scales
        {
            uint8_t* dst = bt + role * kPairTile + (lane >> 1) * kVPitch + 128 * (lane & 1);
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const uint32_t bw[4] = {buf.b[c].x, buf.b[c].y, buf.b[c].z, buf.b[c].w};
                const uint32_t rw[4] = {buf.r[c].x, buf.r[c].y, buf.r[c].z, buf.r[c].w};
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    uint32_t cv[4];
                    if (kv8) dec8(bw[w], rw[w], kc, cv);
                    else dec4(bw[w], kc, cv);
                    *reinterpret_cast<uint4*>(dst + 64 * c + 16 * w) = make_uint4(cv[0], cv[1], cv[2], cv[3]);
                }
            }
            if (lane < 16) ssc[16 * role + lane] = __half2float(__ushort_as_half(buf.sc)) * 0.0625f;
        }
        if (pn < p1) load(pn, buf);
        named_sync(1 + pair, 64);             // both tiles of the block are in place

        const uint32_t kt = smem_u32(bt), vt = kt + kPairTile;
        float scs[2][2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) scs[nt][0][e] = scs[nt][1][e] = 0.0f;
#pragma unroll
        for (int st = 0; st < 8; ++st) {
            uint32_t a0, a1, a2, a3;
            ldmatrix_x4(kt + koff + 32 * st, a0, a1, a2, a3);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) mma16816f(scs[nt][st & 1], a0, a1, a2, a3, qb[nt][st][0], qb[nt][st][1]);
        }
        float ks[2], vsc[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            ks[e] = ssc[g + 8 * e];
            vsc[e] = ssc[16 + g + 8 * e];
        }
        uint32_t pf[2][2];                    // P^T fragments of both row groups
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            float sc[4], pr[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) sc[e] = (scs[nt][0][e] + scs[nt][1][e]) * ks[e >> 1];
            if constexpr (!MASK) {
                float mx[2];
#pragma unroll
                for (int re = 0; re < 2; ++re) {
                    mx[re] = fmaxf(sc[re], sc[2 + re]);
#pragma unroll
                    for (int off = 4; off < 32; off <<= 1)
                        mx[re] = fmaxf(mx[re], __shfl_xor_sync(0xffffffffu, mx[re], off));
                }
                if (__any_sync(0xffffffffu, mx[0] > m[nt][0] + kLazy || mx[1] > m[nt][1] + kLazy)) {   // see k_kv_attn_tc
#pragma unroll
                    for (int re = 0; re < 2; ++re) {
                        const float mn = fmaxf(m[nt][re], mx[re]);
                        const float corr = ex2(m[nt][re] - mn);
                        l[nt][re] *= corr;
                        m[nt][re] = mn;
#pragma unroll
                        for (int dt = 0; dt < 8; ++dt) { o[nt][dt][re] *= corr; o[nt][dt][2 + re] *= corr; }
                    }
                }
#pragma unroll
                for (int re = 0; re < 2; ++re) {
                    const float e0 = ex2(sc[re] - m[nt][re]), e1 = ex2(sc[2 + re] - m[nt][re]);
                    l[nt][re] += e0 + e1;
                    pr[re] = e0 * vsc[0];
                    pr[2 + re] = e1 * vsc[1];
                }
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int pe = pb + g + 8 * (e >> 1), re = e & 1;
                    if (!(pe < p1 && pe < vis[nt][re])) sc[e] = -INFINITY;
                }
#pragma unroll
                for (int re = 0; re < 2; ++re) {
                    float mx = fmaxf(sc[re], sc[2 + re]);
#pragma unroll
                    for (int off = 4; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
                    const float mn = fmaxf(m[nt][re], mx);
                    const float corr = mn == -INFINITY ? 1.0f : ex2(m[nt][re] - mn);
                    const float e0 = sc[re] == -INFINITY ? 0.0f : ex2(sc[re] - mn);
                    const float e1 = sc[2 + re] == -INFINITY ? 0.0f : ex2(sc[2 + re] - mn);
                    l[nt][re] = l[nt][re] * corr + (e0 + e1);
                    m[nt][re] = mn;
#pragma unroll
                    for (int dt = 0; dt < 8; ++dt) { o[nt][dt][re] *= corr; o[nt][dt][2 + re] *= corr; }
                    pr[re] = e0 * vsc[0];
                    pr[2 + re] = e1 * vsc[1];
                }
            }
            pf[nt][0] = movmatrix_trans(pack_h2(pr[0], pr[1]));
            pf[nt][1] = movmatrix_trans(pack_h2(pr[2], pr[3]));
        }
        // each value fragment is read from the tile once, for both row groups
#pragma unroll
        for (int dt = 0; dt < 8; ++dt) {
            uint32_t v0, v1, v2, v3;
            ldmatrix_x4_trans(vt + voff + 32 * dt, v0, v1, v2, v3);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) mma16816f(o[nt][dt], v0, v1, v2, v3, pf[nt][0], pf[nt][1]);
        }
        pb = pn;
        ++it;
    };
    using Dec4 = std::integral_constant<int, 0>;
    using Dec8 = std::integral_constant<int, 1>;
    using DecAny = std::integral_constant<int, 2>;
    // Both warps of a pair take every block of the pair in the same order (one pair barrier
    // each); the specialised steps only change what a warp does inside a block.
    if (!view8) {
        const int lim = vis_all < recent0 ? vis_all : recent0;
        while (pb + 16 <= lim) step(Dec4{}, std::false_type{});
    }
    while (pb + 16 <= vis_all) step(Dec8{}, std::false_type{});
    while (pb < p1) step(DecAny{}, std::true_type{});

#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int re = 0; re < 2; ++re)
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) l[nt][re] += __shfl_xor_sync(0xffffffffu, l[nt][re], off);
    __syncthreads();                          // every warp is done with the tiles (aliased below)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
        for (int re = 0; re < 2; ++re) {
            const int rr = 8 * nt + 2 * q + re;
            if (g == 0) { sm[warp][rr] = m[nt][re]; sl[warp][rr] = l[nt][re]; }
#pragma unroll
            for (int dt = 0; dt < 8; ++dt) {
                so[warp][rr][slot_dim(16 * dt + g)] = o[nt][dt][re];
                so[warp][rr][slot_dim(16 * dt + g + 8)] = o[nt][dt][2 + re];
            }
        }
    }
    __syncthreads();
    const int rbase = tile * kPairRows;
    const int nr = R - rbase < kPairRows ? R - rbase : kPairRows;
    for (int i = threadIdx.x; i < nr * kD; i += kPairThreads) {
        const int rr = i / kD, dd = i % kD;
        const int rl = rr & 15, w0 = rr >> 4;     // the row's warps: w0 (pair 0), w0 + 2 (pair 1)
        float M = -INFINITY;
        for (int w2 = w0; w2 < kPairWarps; w2 += 2) M = fmaxf(M, sm[w2][rl]);
        float L = 0.0f, O = 0.0f;
        if (M != -INFINITY) {
            for (int w2 = w0; w2 < kPairWarps; w2 += 2) {
                const float f = sm[w2][rl] == -INFINITY ? 0.0f : exp2f(sm[w2][rl] - M);
                L += f * sl[w2][rl];
                O += f * so[w2][rl][dd];
            }
        }
        const int rg = rbase + rr;
        const int tile16 = rg / kRowsPerTile, r16 = rg % kRowsPerTile;
        const size_t slot = (((size_t)h * a.ntiles + tile16) * a.nsplit + split) * kRowsPerTile + r16;
        float* wp = a.work + slot * (kD + 2);
        wp[2 + dd] = O;
        if (dd == 0) { wp[0] = M; wp[1] = L; }
    }
}

// out[t][h*G+g][:] = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s over the splits.
// The splits' (max, sum) pairs are read in parallel into shared memory first, so the
// per-dim pass below issues independent loads.
constexpr int kMaxSplits = 1024;
__global__ void __launch_bounds__(128) k_kv_combine(const __grid_constant__ KvAttnArgs a) {
    __shared__ float sw[kMaxSplits];          // weight 2^(m_s - M) of each split
    __shared__ float red[4];
    grid_dep_launch_dependents();
    const int h = blockIdx.x, row = blockIdx.y;     // row = t * G + g
    grid_dep_wait();
    const int tile = row / kRowsPerTile, rr = row % kRowsPerTile;
    const int t = row / a.G, g = row % a.G;
    auto slot = [&](int s) { return (((size_t)h * a.ntiles + tile) * a.nsplit + s) * kRowsPerTile + rr; };
    float mloc = -INFINITY;
    for (int s = threadIdx.x; s < a.nsplit; s += blockDim.x) {
        const float ms = a.work[slot(s) * (kD + 2)];
        sw[s] = ms;
        mloc = fmaxf(mloc, ms);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mloc;
    __syncthreads();
    const float M = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
    __syncthreads();
    float lloc = 0.0f;
    for (int s = threadIdx.x; s < a.nsplit; s += blockDim.x) {
        const float f = sw[s] == -INFINITY ? 0.0f : exp2f(sw[s] - M);
        sw[s] = f;
        lloc += f * a.work[slot(s) * (kD + 2) + 1];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lloc += __shfl_xor_sync(0xffffffffu, lloc, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = lloc;
    __syncthreads();
    const float L = (red[0] + red[1]) + (red[2] + red[3]);
    const int dd = threadIdx.x;                     // one output dim per thread (128 threads)
    float O = 0.0f;
#pragma unroll 8
    for (int s = 0; s < a.nsplit; ++s) O += sw[s] * a.work[slot(s) * (kD + 2) + 2 + dd];
    a.out[((size_t)t * a.Hq + (size_t)h * a.G + g) * kD + dd] = L > 0.0f ? O / L : 0.0f;
}

}  // namespace

cudaError_t launch_kv_write(const void* x, int bf16, int T, int H, int pos0, int Lmax, uint8_t* base, uint8_t* ref,
                            uint16_t* scale, cudaStream_t stream) {
    const long long threads = (long long)T * H * 32;
    const dim3 grid((unsigned)((threads + 255) / 256)), blk(256);
    return bf16 ? launch_pdl(k_kv_write<true>, grid, blk, 0, stream, x, T, H, pos0, Lmax, base, ref, scale)
                : launch_pdl(k_kv_write<false>, grid, blk, 0, stream, x, T, H, pos0, Lmax, base, ref, scale);
}

int kv_rows_per_tile() { return kRowsPerTile; }

// Resident CTAs per SM of the tensor-core kernel for 8 (kind 1) or 16 (kind 2) query rows,
// or of the paired kernel for 32 (kind 3).
int tc_resident(int kind) {
    static int cached[4] = {0, 0, 0, 0};
    if (cached[kind] == 0) {
        int n = 0;
        const cudaError_t e =
            kind == 1   ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_kv_attn_tc<1>, kTcThreads, kv_tc_smem<1>())
            : kind == 2 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_kv_attn_tc<2>, kTcThreads, kv_tc_smem<2>())
                        : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_kv_attn_pair, kPairThreads, kPairSmem);
        if (e != cudaSuccess) (void)cudaGetLastError();
        cached[kind] = (e == cudaSuccess && n > 0) ? n : 1;
    }
    return cached[kind];
}

// Position splits: the smallest count whose CTAs fill the resident slots (SMs x CTAs per
// SM) to 95 % over whole waves, else the best fill up to four waves; at least 128
// positions per split and at most kMaxSplits splits.
int kv_kind(int R) { return R <= 8 ? 1 : R <= 16 ? 2 : 3; }
int kv_rows_per_cta(int kind) { return kind == 1 ? 8 : kind == 2 ? 16 : kPairRows; }

int kv_splits(int T, int G, int Hkv, int L, int sms) {
    const int R = T * G;
    const int kind = kv_kind(R), rows = kv_rows_per_cta(kind);
    const long long base = (long long)Hkv * ((R + rows - 1) / rows);
    const long long slots = (long long)tc_resident(kind) * (sms > 0 ? sms : 1);
    long long cap = (L + 127) / 128;
    cap = cap < kMaxSplits ? cap : kMaxSplits;
    const long long by_waves = (4 * slots + base - 1) / base;
    cap = cap < by_waves ? cap : by_waves;
    int best = 1;
    double best_eff = -1.0;
    for (int n = 1; n <= cap; ++n) {
        const long long ctas = base * n, waves = (ctas + slots - 1) / slots;
        const double eff = (double)ctas / (double)(waves * slots);
        if (eff >= 0.95) return n;
        if (eff > best_eff + 1e-9) { best_eff = eff; best = n; }
    }
    return best;
}

cudaError_t launch_kv_attention(KvAttnArgs& a, int sms, cudaStream_t stream) {
    const int R = a.T * a.G;
    a.ntiles = (R + kRowsPerTile - 1) / kRowsPerTile;
    a.nsplit = kv_splits(a.T, a.Hq / a.Hkv, a.Hkv, a.L, sms);
    const int rows = R < kRowsPerTile ? R : kRowsPerTile;
    cudaError_t e;
    if (a.impl == 1) {                        // CUDA-core kernel (kept for measurement)
        const dim3 grid(a.Hkv, a.nsplit, a.ntiles), blk(kAttnThreads);
        e = rows <= 2   ? launch_pdl(k_kv_attn<2>, grid, blk, 0, stream, a)
            : rows <= 4 ? launch_pdl(k_kv_attn<4>, grid, blk, 0, stream, a)
            : rows <= 8 ? launch_pdl(k_kv_attn<8>, grid, blk, 0, stream, a)
                        : launch_pdl(k_kv_attn<16>, grid, blk, 0, stream, a);
    } else {                                  // tensor cores: 8, 16 or (paired) 32 rows per CTA
        const int kind = kv_kind(R);
        if (kind == 1) {
            const dim3 grid(a.Hkv, a.nsplit, (R + 7) / 8), blk(kTcThreads);
            e = launch_pdl(k_kv_attn_tc<1>, grid, blk, kv_tc_smem<1>(), stream, a);
        } else if (kind == 2 || a.impl == 2) {  // impl 2: 16-row CTAs only (kept for measurement)
            const dim3 grid(a.Hkv, a.nsplit, a.ntiles), blk(kTcThreads);
            e = launch_pdl(k_kv_attn_tc<2>, grid, blk, kv_tc_smem<2>(), stream, a);
        } else {
            const dim3 grid(a.Hkv, a.nsplit, (R + kPairRows - 1) / kPairRows), blk(kPairThreads);
            e = launch_pdl(k_kv_attn_pair, grid, blk, kPairSmem, stream, a);
        }
    }
    if (e != cudaSuccess) return e;
    return launch_pdl(k_kv_combine, dim3(a.Hkv, R), dim3(kD), 0, stream, a);
}

}  // namespace nest
