// Glue between the linears of a chained decoder layer, fused with the
// rotations on both sides of it:
//   y   = S_o H_o z_a               (output rotation of linear a)
//   h   = y            or  y * (S_o' H_o' z_b)   (elementwise product, e.g. gate * up)
//   h  <- bf16(h / rms(h))          (unit-RMS rescale per token, then the bf16 cast)
//   x'_j = H_j S_j h                 (input rotation of each next linear j, into its
//                                     fp16 GEMM operand)
// The rotations follow feedman.me/posts/wZBTJ, POC recipe steps 1 and 4.  The
// chaining itself (which output feeds which linear, and the RMS rescale standing
// in for the normalisation between them) is not on the pages; it is the plain
// reading used by the chained-layer workload.
//
// One CTA handles one token's whole vector in shared memory (two buffers of M
// floats), so the RMS needs no cross-CTA reduction.  FWHT: butterflies over index
// bits 0..5 with warp shuffles on 64-element rows, the higher bits as
// shared-memory butterfly stages.
#include "nest_device.cuh"
#include "nest_internal.h"

namespace nest {
namespace {

constexpr int kThreads = 1024;

// In-place block-diagonal FWHT (blocks of 2^L, unnormalised) of buf[0..M).
__device__ void fwht_smem(float* buf, int M, int L) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
    const int L1 = L < 6 ? L : 6;
    if (L1 > 0) {
        const int rows = (M + 63) / 64;
        for (int row = warp; row < rows; row += nwarps) {
            const int i0 = row * 64 + lane, i1 = i0 + 32;
            float v0 = i0 < M ? buf[i0] : 0.0f, v1 = i1 < M ? buf[i1] : 0.0f;
            warp_fwht(v0, v1, L1, lane);
            if (i0 < M) buf[i0] = v0;
            if (i1 < M) buf[i1] = v1;
        }
        __syncthreads();
    }
    for (int s = 6; s < L; ++s) {
        const int h = 1 << s;
        for (int q = threadIdx.x; q < M / 2; q += blockDim.x) {
            const int i = ((q >> s) << (s + 1)) | (q & (h - 1));
            const float a = buf[i], b = buf[i + h];
            buf[i] = a + b;
            buf[i + h] = a - b;
        }
        __syncthreads();
    }
}

__device__ float block_sum(float v, float* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float t = 0.0f;
    if (warp == 0) {
        t = lane < (int)(blockDim.x >> 5) ? red[lane] : 0.0f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
        if (lane == 0) red[0] = t;
    }
    __syncthreads();
    t = red[0];
    __syncthreads();
    return t;
}

__global__ void __launch_bounds__(kThreads) k_chain(const __grid_constant__ ChainArgs a) {
    extern __shared__ __align__(16) float sh[];
    float* buf = sh;                 // h
    float* tmp = sh + a.M;           // second operand / per-next-linear work
    float* red = sh + 2 * a.M;       // 32 floats
    const int t = blockIdx.x, M = a.M;
    grid_dep_launch_dependents();
    grid_dep_wait();                 // z comes from the previous kernel; the operands may be its input

    for (int j = 0; j < a.nnext; ++j) {          // clear the accumulators of the GEMMs that follow
        const ChainNext& nx = a.next[j];
        if (nx.zero_out == nullptr) continue;
        const long long per = (nx.zero_count + gridDim.x - 1) / gridDim.x;
        const long long lo = per * t, hi = lo + per < nx.zero_count ? lo + per : nx.zero_count;
        for (long long i = lo + threadIdx.x; i < hi; i += blockDim.x) nx.zero_out[i] = 0.0f;
    }

    // y = S_o H_o z_a (and the product partner)
    for (int i = threadIdx.x; i < M; i += blockDim.x) buf[i] = a.za[(size_t)t * M + i];
    if (a.zb != nullptr)
        for (int i = threadIdx.x; i < M; i += blockDim.x) tmp[i] = a.zb[(size_t)t * M + i];
    __syncthreads();
    fwht_smem(buf, M, a.L);
    if (a.zb != nullptr) fwht_smem(tmp, M, a.L);
    float ss = 0.0f;
    for (int i = threadIdx.x; i < M; i += blockDim.x) {
        float v = buf[i] * a.scale * (float)a.sa[i];
        if (a.zb != nullptr) v *= tmp[i] * a.scale * (float)a.sb[i];
        buf[i] = v;
        if (a.y != nullptr) a.y[(size_t)t * M + i] = v;
        ss += v * v;
    }
    ss = block_sum(ss, red);
    const float rms = sqrtf(ss / (float)M);
    const float inv = rms > 0.0f ? 1.0f / rms : 0.0f;
    for (int i = threadIdx.x; i < M; i += blockDim.x) buf[i] = __bfloat162float(__float2bfloat16_rn(buf[i] * inv));
    __syncthreads();

    // x'_j = H_j S_j h for every next linear, written as its fp16 GEMM operand
    for (int j = 0; j < a.nnext; ++j) {
        const ChainNext& nx = a.next[j];
        for (int i = threadIdx.x; i < M; i += blockDim.x) tmp[i] = buf[i] * (float)nx.sign_in[i];
        __syncthreads();
        fwht_smem(tmp, M, a.L);
        for (int c8 = threadIdx.x; c8 < M / 8; c8 += blockDim.x) {
            const int k = 8 * c8;
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
                w[e] = h2_as_u32(__floats2half2_rn(tmp[k + 2 * e] * a.scale, tmp[k + 2 * e + 1] * a.scale));
            const int g = k >> 7, c = (k & 127) >> 3;
            const size_t off = (size_t)g * 2048 * a.NB + ((size_t)(c * a.NB + (t >> 3)) * 8 + (t & 7)) * 16;
            *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(nx.xop) + off) = make_uint4(w[0], w[1], w[2], w[3]);
        }
        __syncthreads();
    }
}

}  // namespace

size_t chain_smem_bytes(int M) { return (size_t)(2 * M + 32) * sizeof(float); }

cudaError_t launch_chain(ChainArgs& a, cudaStream_t stream) {
    const int b = hadamard_block(a.M);
    int L = 0;
    while ((1 << L) < b) ++L;
    a.L = L;
    a.scale = (float)(1.0 / sqrt((double)b));
    a.NB = n_pad(a.T) / 8;
    const size_t smem = chain_smem_bytes(a.M);
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(k_chain, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    return launch_pdl(k_chain, dim3(a.T), dim3(kThreads), smem, stream, a);
}

}  // namespace nest
