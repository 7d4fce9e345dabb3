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
#include "nest_device.cuh"
#include "nest_internal.h"

namespace nest {
namespace {

constexpr int kD = 128;

// One warp per (token, head): lane l owns dims 4l .. 4l+3.  Decisions in fp32 with
// each operation rounded on its own (no contraction), so that they match the
// reference bit for bit:  s = fp16(max|x| / 7);  q4 = clip(rint(x / s), -8, 7);
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

// out[t][h*G+g][:] = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s over the splits
__global__ void k_kv_combine(const __grid_constant__ KvAttnArgs a) {
    grid_dep_launch_dependents();
    const int h = blockIdx.x, row = blockIdx.y;     // row = t * G + g
    grid_dep_wait();
    const int tile = row / kRowsPerTile, rr = row % kRowsPerTile;
    const int t = row / a.G, g = row % a.G;
    for (int dd = threadIdx.x; dd < kD; dd += blockDim.x) {
        float M = -INFINITY;
        for (int s = 0; s < a.nsplit; ++s) {
            const size_t slot = (((size_t)h * a.ntiles + tile) * a.nsplit + s) * kRowsPerTile + rr;
            M = fmaxf(M, a.work[slot * (kD + 2)]);
        }
        float L = 0.0f, O = 0.0f;
        for (int s = 0; s < a.nsplit; ++s) {
            const size_t slot = (((size_t)h * a.ntiles + tile) * a.nsplit + s) * kRowsPerTile + rr;
            const float* wp = a.work + slot * (kD + 2);
            const float f = wp[0] == -INFINITY ? 0.0f : exp2f(wp[0] - M);
            L += f * wp[1];
            O += f * wp[2 + dd];
        }
        a.out[((size_t)t * a.Hq + (size_t)h * a.G + g) * kD + dd] = L > 0.0f ? O / L : 0.0f;
    }
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

// Position splits: enough CTAs for eight per SM (many loads in flight), at least 128
// positions (one 32-position tile per warp) per split.
int kv_splits(int T, int G, int Hkv, int L, int sms) {
    const int tiles = (T * G + kRowsPerTile - 1) / kRowsPerTile;
    const int base = Hkv * tiles;
    int ns = (8 * sms + base - 1) / base;
    const int by_len = (L + 127) / 128;
    ns = ns < by_len ? ns : by_len;
    return ns < 1 ? 1 : ns;
}

cudaError_t launch_kv_attention(KvAttnArgs& a, int sms, cudaStream_t stream) {
    const int R = a.T * a.G;
    a.ntiles = (R + kRowsPerTile - 1) / kRowsPerTile;
    a.nsplit = kv_splits(a.T, a.Hq / a.Hkv, a.Hkv, a.L, sms);
    const int rows = R < kRowsPerTile ? R : kRowsPerTile;
    const dim3 grid(a.Hkv, a.nsplit, a.ntiles), blk(kAttnThreads);
    cudaError_t e = rows <= 2   ? launch_pdl(k_kv_attn<2>, grid, blk, 0, stream, a)
                    : rows <= 4 ? launch_pdl(k_kv_attn<4>, grid, blk, 0, stream, a)
                    : rows <= 8 ? launch_pdl(k_kv_attn<8>, grid, blk, 0, stream, a)
                                : launch_pdl(k_kv_attn<16>, grid, blk, 0, stream, a);
    if (e != cudaSuccess) return e;
    return launch_pdl(k_kv_combine, dim3(a.Hkv, R), dim3(kD), 0, stream, a);
}

}  // namespace nest
