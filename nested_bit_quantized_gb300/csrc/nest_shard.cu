// Reorder of the all-gathered output blocks of a row-sharded linear.
//
// Row-sharded tensor parallelism over the output rows: each of `world` ranks
// holds whole 128-row tiles of the packed layer (Mp rows per rank, the last
// rank's share possibly shorter or empty), rotates the replicated input
// itself, and computes its rows of the rotated-basis output z.  One all-gather
// blocks (rank r's [T][M_r] rows, M_r = min(Mp, M - r Mp), at the start of a
// block of T * Mp floats) gives every rank [world][T * Mp]; the output rotation
// needs each token's whole row of z, so this kernel writes it back token-major:
//   z[t][r Mp + j] = gathered[r T Mp + t M_r + j],   j < M_r.
// The source pages run on one device; this is the library's multi-GPU split.
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/nest.h"
#include "nest_device.cuh"
#include "nest_internal.h"

namespace nest {
namespace {

constexpr int kShardThreads = 256;

__global__ void __launch_bounds__(kShardThreads) k_shard_gather(const float* __restrict__ in, float* __restrict__ out,
                                                                 int T, int Mp, int M) {
    grid_dep_launch_dependents();
    grid_dep_wait();                          // the gathered blocks come from the previous work in the stream
    const long long total = (long long)T * M;
    for (long long i = (long long)blockIdx.x * kShardThreads + threadIdx.x; i < total;
         i += (long long)gridDim.x * kShardThreads) {
        const int t = (int)(i / M), m = (int)(i - (long long)t * M);
        const int r = m / Mp, j = m - r * Mp;
        const int Mr = M - r * Mp < Mp ? M - r * Mp : Mp;     // rows of rank r
        out[i] = in[(long long)r * T * Mp + (long long)t * Mr + j];
    }
}

}  // namespace
}  // namespace nest

extern "C" nest_status nest_shard_gather(const float* gathered, float* z, int32_t world, int32_t T, int32_t Mp,
                                         int32_t M, void* stream) {
    using namespace nest;
    if (gathered == nullptr || z == nullptr) return NEST_ERR_INVALID_ARG;
    if (world < 1 || T < 1 || Mp < 1 || M < 1) return NEST_ERR_INVALID_ARG;
    if ((long long)world * Mp < M) return NEST_ERR_INVALID_ARG;
    if ((long long)world * T * Mp >= (1LL << 31)) return NEST_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(gathered) & 3u) || (reinterpret_cast<uintptr_t>(z) & 3u))
        return NEST_ERR_MISALIGNED;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return NEST_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
        return NEST_ERR_CUDA;
    const long long total = (long long)T * M;
    long long grid = (total + kShardThreads - 1) / kShardThreads;
    if (grid > 2LL * sms) grid = 2LL * sms;
    const cudaError_t e = launch_pdl(k_shard_gather, dim3((unsigned)grid), dim3(kShardThreads), 0,
                                     reinterpret_cast<cudaStream_t>(stream), gathered, z, (int)T, (int)Mp, (int)M);
    return e == cudaSuccess ? NEST_OK : NEST_ERR_CUDA;
}
