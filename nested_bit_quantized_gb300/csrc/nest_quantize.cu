// Offline RTN quantizer of one layer, in fp64 (feedman.me/posts/wZBTJ, POC
// recipe steps 1-3, without the calibration-based GPTQ/LDLQ feedback):
//   W~ = H_o S_o W S_i H_i            (block-diagonal Sylvester Hadamard / sqrt(b))
//   base:     s_b = fp16(RMS of each (row, 128-group) block), code = nearest
//             level of W~/s_b among -1.5104, -0.4528, +0.4528, +1.5104
//   residual: R = W~ - L[code] s_b, s_r = fp16(max|R| / qm),
//             q = clip(rint(R / s_r), -qm, qm), qm = 2^(b-1) - 1
// Ties: |u| exactly at the inner/outer midpoint takes the inner level, u == 0
// the positive inner level, a zero scale gives code 2 / residual 0; rint is
// round-half-to-even.  Codes are decided in fp64 like the CPU oracle.
#include "nest_device.cuh"
#include "nest_internal.h"

namespace nest {
namespace {

// W S_i H_i along each row: one CTA per (row, Hadamard block of the input side)
__global__ void k_q_rows(const float* __restrict__ W, const int8_t* __restrict__ si, int K, int b,
                         double scale, double* __restrict__ out) {
    extern __shared__ double sh[];
    const int nblk = K / b;
    const long long m = blockIdx.x / nblk;
    const int j = blockIdx.x % nblk;
    const float* src = W + m * K + (long long)j * b;
    for (int i = threadIdx.x; i < b; i += blockDim.x) sh[i] = (double)src[i] * (double)si[j * b + i];
    __syncthreads();
    for (int h = 1; h < b; h <<= 1) {
        for (int p = threadIdx.x; p < b / 2; p += blockDim.x) {
            const int i = (p / h) * 2 * h + (p % h);
            const double a = sh[i], c = sh[i + h];
            sh[i] = a + c;
            sh[i + h] = a - c;
        }
        __syncthreads();
    }
    double* dst = out + m * K + (long long)j * b;
    for (int i = threadIdx.x; i < b; i += blockDim.x) dst[i] = sh[i] * scale;
}

// one butterfly stage of H_o S_o (.) along the rows (output side); the first
// stage applies S_o, the last one the 1/sqrt(b) normalisation
__global__ void k_q_cols(double* __restrict__ w, const int8_t* __restrict__ so, int M, int K, int h,
                         int first, double scale) {
    const long long n = (long long)(M / 2) * K;
    for (long long it = blockIdx.x * (long long)blockDim.x + threadIdx.x; it < n;
         it += (long long)gridDim.x * blockDim.x) {
        const int p = (int)(it / K), k = (int)(it % K);
        const int i = (p / h) * 2 * h + (p % h), j = i + h;
        double a = w[(long long)i * K + k], c = w[(long long)j * K + k];
        if (first) { a *= (double)so[i]; c *= (double)so[j]; }
        w[(long long)i * K + k] = (a + c) * scale;
        w[(long long)j * K + k] = (a - c) * scale;
    }
}

// output side with block size 1 (odd M): signs only
__global__ void k_q_signs(double* __restrict__ w, const int8_t* __restrict__ so, int M, int K) {
    const long long n = (long long)M * K;
    for (long long it = blockIdx.x * (long long)blockDim.x + threadIdx.x; it < n;
         it += (long long)gridDim.x * blockDim.x)
        w[it] *= (double)so[it / K];
}

__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ double warp_max(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmax(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// one warp per (row, group): 4 consecutive columns per lane
__global__ void k_q_quant(const double* __restrict__ wr, int M, int K, int bits,
                          uint8_t* __restrict__ bc, uint16_t* __restrict__ bs,
                          int8_t* __restrict__ rc, uint16_t* __restrict__ rs) {
    const int G = K / kGroup;
    const long long wid = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (wid >= (long long)M * G) return;
    const long long m = wid / G;
    const int g = (int)(wid % G);
    const long long col = (long long)g * kGroup + 4 * lane;
    double v[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) v[e] = wr[m * K + col + e];

    const double ss = warp_sum(v[0] * v[0] + v[1] * v[1] + v[2] * v[2] + v[3] * v[3]);
    const __half sb16 = __double2half(sqrt(ss / 128.0));
    const double s = (double)__half2float(sb16);
    constexpr double thr = (level_d(2) + level_d(3)) / 2.0;
    int code[4];
    double R[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        int c = 2;
        if (s > 0.0) {
            const double u = v[e] / s;
            const bool outer = fabs(u) > thr;
            c = (u < 0.0) ? (outer ? 0 : 1) : (outer ? 3 : 2);
        }
        code[e] = c;
        R[e] = v[e] - level_d(c) * s;
    }
    bc[m * K + col + 0] = (uint8_t)code[0];
    bc[m * K + col + 1] = (uint8_t)code[1];
    bc[m * K + col + 2] = (uint8_t)code[2];
    bc[m * K + col + 3] = (uint8_t)code[3];
    if (lane == 0) bs[m * G + g] = __half_as_ushort(sb16);
    if (bits == 0) return;

    const int qm = (1 << (bits - 1)) - 1;
    const double amax = warp_max(fmax(fmax(fabs(R[0]), fabs(R[1])), fmax(fabs(R[2]), fabs(R[3]))));
    const __half sr16 = __double2half(amax / (double)qm);
    const double sr = (double)__half2float(sr16);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        int q = 0;
        if (sr > 0.0) {
            double t = rint(R[e] / sr);
            t = fmin(fmax(t, (double)-qm), (double)qm);
            q = (int)t;
        }
        rc[m * K + col + e] = (int8_t)q;
    }
    if (lane == 0) rs[m * G + g] = __half_as_ushort(sr16);
}

// BitNest W4/W8 (Eq. (5)-(10) of the BitNest paper, RTN base): one warp per (row,
// group), 4 consecutive columns per lane.  s4 = fp16(max|W'| / 7); q4 = clip(rint(W'/s4),
// -8, 7); dW = W' - q4 s4; s_ref = s4 / 16; q_r = clip(rint(dW / s_ref), q4 == -8 ? 0 : -8, 7).
__global__ void k_q_w4w8(const double* __restrict__ wr, int M, int K, int8_t* __restrict__ q4,
                         uint16_t* __restrict__ s4, int8_t* __restrict__ qr) {
    const int G = K / kGroup;
    const long long wid = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (wid >= (long long)M * G) return;
    const long long m = wid / G;
    const int g = (int)(wid % G);
    const long long col = (long long)g * kGroup + 4 * lane;
    double v[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) v[e] = wr[m * K + col + e];
    const double amax = warp_max(fmax(fmax(fabs(v[0]), fabs(v[1])), fmax(fabs(v[2]), fabs(v[3]))));
    const __half s16 = __double2half(amax / 7.0);
    const double s = (double)__half2float(s16);
    const double sref = s / 16.0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        int a = 0, b = 0;
        if (s > 0.0) {
            a = (int)fmin(fmax(rint(v[e] / s), -8.0), 7.0);
            const double t = rint((v[e] - (double)a * s) / sref);
            b = (int)fmin(fmax(t, a == -8 ? 0.0 : -8.0), 7.0);
        }
        q4[m * K + col + e] = (int8_t)a;
        if (qr != nullptr) qr[m * K + col + e] = (int8_t)b;
    }
    if (lane == 0) s4[m * G + g] = __half_as_ushort(s16);
}

int grid_for(long long items, int threads) {
    long long g = (items + threads - 1) / threads;
    return (int)(g < 65535 * 16 ? (g < 1 ? 1 : g) : 65535 * 16);
}

// W' = H_o S_o W S_i H_i in fp64 into `work` (the rotation both quantizers start from)
void rotate_stage(const float* W, const int8_t* so, const int8_t* si, int M, int K, double* work,
                  cudaStream_t stream) {
    const int b_in = hadamard_block(K), b_out = hadamard_block(M);
    const int thr_rows = b_in >= 512 ? 256 : (b_in / 2 > 32 ? b_in / 2 : 32);
    k_q_rows<<<(unsigned)((long long)M * (K / b_in)), thr_rows, b_in * sizeof(double), stream>>>(
        W, si, K, b_in, 1.0 / sqrt((double)b_in), work);
    if (b_out == 1) {
        k_q_signs<<<grid_for((long long)M * K, 256), 256, 0, stream>>>(work, so, M, K);
    } else {
        const double sc = 1.0 / sqrt((double)b_out);
        for (int h = 1; h < b_out; h <<= 1)
            k_q_cols<<<grid_for((long long)(M / 2) * K, 256), 256, 0, stream>>>(
                work, so, M, K, h, h == 1 ? 1 : 0, (2 * h == b_out) ? sc : 1.0);
    }
}

}  // namespace

cudaError_t launch_quantize(const float* W, const int8_t* so, const int8_t* si, int M, int K, int bits,
                            double* work, uint8_t* bc, uint16_t* bs, int8_t* rc, uint16_t* rs,
                            cudaStream_t stream) {
    rotate_stage(W, so, si, M, K, work, stream);
    const long long warps = (long long)M * (K / kGroup);
    k_q_quant<<<(unsigned)((warps * 32 + 255) / 256), 256, 0, stream>>>(work, M, K, bits, bc, bs, rc, rs);
    return cudaGetLastError();
}

cudaError_t launch_quantize_w4w8(const float* W, const int8_t* so, const int8_t* si, int M, int K, double* work,
                                 int8_t* q4, uint16_t* s4, int8_t* qr, cudaStream_t stream) {
    rotate_stage(W, so, si, M, K, work, stream);
    const long long warps = (long long)M * (K / kGroup);
    k_q_w4w8<<<(unsigned)((warps * 32 + 255) / 256), 256, 0, stream>>>(work, M, K, q4, s4, qr);
    return cudaGetLastError();
}

}  // namespace nest
