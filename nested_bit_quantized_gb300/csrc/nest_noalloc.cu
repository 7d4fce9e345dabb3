// nest_linear_static: the whole-linear call for callers that cannot allocate
// device memory.
//
// Who needs it: a process whose device memory is carved up once at start-up by
// its own pool (a serving engine that claims the GPU's memory before taking
// traffic, or an embedding framework whose allocator the library must not go
// around), plain C callers with no allocator of their own, and latency-critical
// loops that cannot afford cudaMalloc's implicit synchronisation.  Such callers
// can still pass their inputs and outputs, but not the intermediate buffers the
// linear needs between its kernels (the fp16 activation operand and the fp32
// accumulator).  This entry point keeps those buffers in one fixed array in the
// library's own device memory instead.
//
// The array is a file-scope __device__ variable of kStaticScratchBytes: every GPU
// that loads the library holds it until the process exits.  Host code cannot use
// its name as a device pointer; the address is looked up once per device with
// cudaGetSymbolAddress (on the first call made with that device current) and
// cached.  All calls share the one array and it keeps the last call's contents;
// the path clears the accumulator itself, so nothing has to start at zero on
// entry, but calls whose kernels overlap on the GPU (other streams, other host
// threads) race on the array and must be serialised by the caller.  The cached
// address belongs to the device's primary context: after cudaDeviceReset the
// array lives elsewhere (or nowhere), so the entry point must not be called on a
// device that this process has reset.
#include <atomic>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/nest.h"
#include "nest_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(8) << 20;      // 8 MiB
constexpr int kMaxDevices = 64;

__device__ __align__(256) uint8_t g_linear_scratch[kStaticScratchBytes];

std::atomic<void*> g_scratch_addr[kMaxDevices];

// Device address of g_linear_scratch on the current device (looked up once per device).
nest_status scratch_for_current_device(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NEST_ERR_CUDA;
    void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
        const cudaError_t e = cudaGetSymbolAddress(&p, g_linear_scratch);
        if (e != cudaSuccess || p == nullptr) return NEST_ERR_CUDA;
        g_scratch_addr[dev].store(p, std::memory_order_release);
    }
    *out = p;
    return NEST_OK;
}

}  // namespace

extern "C" nest_status nest_linear_static(const nest_layer* layer, int32_t verify, const void* x, int32_t x_dtype,
                                          int32_t T, float* y, void* stream) {
    if (layer == nullptr || x == nullptr || y == nullptr) return NEST_ERR_INVALID_ARG;
    if (layer->M < 1 || layer->K < 1 || T < 1) return NEST_ERR_INVALID_ARG;
    const size_t need = nest_linear_scratch_bytes(layer->M, layer->K, T);
    if (need == 0) return NEST_ERR_UNSUPPORTED;               // K % 128 != 0 or T > 256
    if (need > kStaticScratchBytes) return NEST_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    const nest_status st = scratch_for_current_device(&scratch);
    if (st != NEST_OK) return st;
    return nest_linear(layer, verify, x, x_dtype, T, y, scratch, stream);
}
