// Host-side declarations shared between the C-ABI layer and the kernel files.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace nest {

// Arguments of one draft/verify GEMM launch.
struct GemmArgs {
    const uint8_t* base;      // packed base units
    const uint8_t* resid;     // packed residual units (verify only)
    const uint16_t* xop;      // activation operand
    float* z;                 // [T][M] output
    float* partial;           // workspace: 2 slots per CTA of T x 128 partial sums
    int* counters;            // workspace: 4 counters per row tile
    int M, K, T, G;           // G = K / 128
    long long units;          // row tiles * G
};

constexpr int kMaxGrid = 1024;

inline int n_tiles(int M) { return (M + 127) / 128; }
inline int n_pad(int T) { return T <= 16 ? 16 : (T <= 32 ? 32 : 64); }

// workspace layout: counters first (4 per tile, 256-byte aligned), then partials
inline size_t ws_counter_bytes(int M) { return ((size_t)4 * n_tiles(M) * sizeof(int) + 255) / 256 * 256; }
inline size_t ws_partial_bytes(int M, int K, int T) {
    long long units = (long long)n_tiles(M) * (K / 128);
    long long g = units < kMaxGrid ? units : kMaxGrid;
    return (size_t)2 * g * T * 128 * sizeof(float);
}

cudaError_t launch_gemm(const GemmArgs& a, int bits, int grid, cudaStream_t stream);
cudaError_t read_and_clear_error(int* flag, cudaStream_t stream);

cudaError_t launch_rotate(const void* x, int x_dtype, const int8_t* signs, int n, int T, int mode,
                          float* y, uint16_t* xop, cudaStream_t stream);

cudaError_t launch_pack(const uint8_t* bc, const uint16_t* bs, const int8_t* rc, const uint16_t* rs,
                        int M, int K, int bits, uint8_t* base_out, uint8_t* resid_out, cudaStream_t stream);
cudaError_t launch_unpack(const uint8_t* base, const uint8_t* resid, int M, int K, int bits,
                          uint8_t* bc, uint16_t* bs, int8_t* rc, uint16_t* rs, cudaStream_t stream);

cudaError_t launch_quantize(const float* W, const int8_t* so, const int8_t* si, int M, int K, int bits,
                            double* work, uint8_t* bc, uint16_t* bs, int8_t* rc, uint16_t* rs,
                            cudaStream_t stream);

int hadamard_block(int n);

}  // namespace nest
