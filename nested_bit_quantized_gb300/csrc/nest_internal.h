// Host-side declarations shared between the C-ABI layer and the kernel files.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>
#include <utility>

namespace nest {

// Arguments of one draft/verify GEMM launch.
struct GemmArgs {
    const uint8_t* base;      // packed base units
    const uint8_t* resid;     // packed residual units (verify only)
    const uint16_t* xop;      // activation operand
    float* z;                 // [T][M] output, accumulated into
    int M, K, T, G;           // G = K / 128
    long long units;          // row tiles * G
};

constexpr int kMaxGrid = 1024;
constexpr int kGemmCtasPerSm = 2;     // resident GEMM CTAs per SM (matches the kernel's launch bounds)

inline int n_tiles(int M) { return (M + 127) / 128; }
inline int n_pad(int T) { return T <= 16 ? 16 : (T <= 32 ? 32 : 64); }

// Launch with programmatic stream serialization: the kernel may start while
// the previous kernel in the stream is still running; it must call
// griddepcontrol.wait before touching anything that kernel produces or reads.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

cudaError_t launch_gemm(const GemmArgs& a, int bits, int grid, cudaStream_t stream);
cudaError_t read_and_clear_error(int* flag, cudaStream_t stream);

// zero_out (optional): a buffer of zero_count floats the kernel also clears (the
// accumulator of the GEMM that follows it).
cudaError_t launch_rotate(const void* x, int x_dtype, const int8_t* signs, int n, int T, int mode,
                          float* y, uint16_t* xop, float* zero_out, long long zero_count, cudaStream_t stream);

cudaError_t launch_pack(const uint8_t* bc, const uint16_t* bs, const int8_t* rc, const uint16_t* rs,
                        int M, int K, int bits, uint8_t* base_out, uint8_t* resid_out, cudaStream_t stream);
cudaError_t launch_unpack(const uint8_t* base, const uint8_t* resid, int M, int K, int bits,
                          uint8_t* bc, uint16_t* bs, int8_t* rc, uint16_t* rs, cudaStream_t stream);

cudaError_t launch_quantize(const float* W, const int8_t* so, const int8_t* si, int M, int K, int bits,
                            double* work, uint8_t* bc, uint16_t* bs, int8_t* rc, uint16_t* rs,
                            cudaStream_t stream);

int hadamard_block(int n);

}  // namespace nest
