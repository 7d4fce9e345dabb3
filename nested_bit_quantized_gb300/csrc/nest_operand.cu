// The GEMM activation operand from an already-rotated fp32 block x' [T][K].
//
// The draft and verify GEMMs read x' as fp16 in the tensor-core operand layout
// (include/nest.h, "Activation operand").  nest_rotate writes that layout while it
// rotates; a caller that already holds x' = H_i S_i x in fp32 (the plain form of
// the POC recipe's step 4, x' then y_b = Q_base x', y_r = Q_resid x') uses this call
// instead.  Each thread converts 8 consecutive columns of one token (round to
// nearest) and writes them as one 16-byte row of a core matrix; padding tokens
// T <= t < Np get zeros.
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/nest.h"
#include "nest_device.cuh"
#include "nest_internal.h"

namespace nest {
namespace {

constexpr int kOpThreads = 256;

__global__ void __launch_bounds__(kOpThreads) k_operand(const float* __restrict__ x, uint16_t* __restrict__ xop,
                                                        int K, int T, int Np) {
    grid_dep_launch_dependents();
    grid_dep_wait();                          // x' may come from the previous kernel in the stream
    const int chunks = K >> 3;                // 8-column pieces per token
    const long long total = (long long)Np * chunks;
    const int NB = Np >> 3;
    for (long long i = (long long)blockIdx.x * kOpThreads + threadIdx.x; i < total;
         i += (long long)gridDim.x * kOpThreads) {
        const int t = (int)(i / chunks), k = (int)(i - (long long)t * chunks) * 8;
        uint32_t w[4] = {0u, 0u, 0u, 0u};
        if (t < T) {
            const float* p = x + (size_t)t * K + k;
#pragma unroll
            for (int e = 0; e < 4; ++e) w[e] = h2_as_u32(__floats2half2_rn(p[2 * e], p[2 * e + 1]));
        }
        *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(xop) + xop_offset(k, t, NB)) =
            make_uint4(w[0], w[1], w[2], w[3]);
    }
}

}  // namespace
}  // namespace nest

extern "C" nest_status nest_operand(const float* x_rot, int32_t K, int32_t T, uint16_t* x_op, void* stream) {
    using namespace nest;
    if (x_rot == nullptr || x_op == nullptr || K < 1 || T < 1) return NEST_ERR_INVALID_ARG;
    if (K % 128 != 0 || T > kMaxT) return NEST_ERR_UNSUPPORTED;
    if ((long long)K * T >= (1LL << 31)) return NEST_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(x_rot) & 3u) || (reinterpret_cast<uintptr_t>(x_op) & 15u))
        return NEST_ERR_MISALIGNED;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return NEST_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
        return NEST_ERR_CUDA;
    const int Np = n_pad(T);
    const long long total = (long long)Np * (K / 8);
    long long grid = (total + kOpThreads - 1) / kOpThreads;
    if (grid > 4LL * sms) grid = 4LL * sms;
    const cudaError_t e = launch_pdl(k_operand, dim3((unsigned)grid), dim3(kOpThreads), 0,
                                     reinterpret_cast<cudaStream_t>(stream), x_rot, x_op, (int)K, (int)T, Np);
    return e == cudaSuccess ? NEST_OK : NEST_ERR_CUDA;
}
