// Host-side declarations shared between the C-ABI layer and the kernel files.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>
#include <utility>

namespace nest {

constexpr int kMaxTasks = 64;          // vector sets in one grouped rotation; linears of nest_linear_group
constexpr int kMaxGemmTasks = 64;      // linears in one grouped draft/verify GEMM launch

// One linear of a grouped draft/verify GEMM launch.
struct GemmTask {
    const uint8_t* base;      // packed base units
    const uint8_t* resid;     // packed residual units (verify only)
    const uint16_t* xop;      // activation operand
    float* z;                 // [T][M] output, accumulated into
    int M, G, tiles;          // G = K / 128, tiles = ceil(M / 128)
    long long ubegin;         // index of the task's first unit in the launch's unit range
};

// Arguments of one grouped launch: the tasks' (tile, group) units are concatenated.
struct GemmArgs {
    GemmTask task[kMaxGemmTasks];
    int ntasks, T;
    long long units;          // total units of all tasks
};

// One set of vectors of a grouped rotation launch (see launch_rotate).
struct RotTask {
    const void* x;
    const int8_t* signs;
    float* y;
    uint16_t* xop;
    float* zero_out;
    long long zero_count;
    unsigned n, total;        // vector length, T * n
    int L, NB, cta_begin;     // log2 block size, operand token blocks, first CTA of the task
    float scale;
    int path;                 // 0 shared-memory tile, 1 register (b <= 512), 2 segment (b >= 1024)
    unsigned nctas;           // CTAs of the task
};

struct RotArgs {
    RotTask task[kMaxTasks];
    int ntasks;
};

constexpr int kMaxGrid = 1024;
constexpr int kGemmCtasPerSm = 2;     // resident GEMM CTAs per SM (matches the kernel's launch bounds)

inline int n_tiles(int M) { return (M + 127) / 128; }
constexpr int kMaxT = 256;                // tokens per call (verify trees up to prefill-size chunks)
inline int n_pad(int T) { return T <= 16 ? 16 : (T <= 32 ? 32 : (T <= 64 ? 64 : (T <= 128 ? 128 : 256))); }
int gemm_ctas_per_sm(int T);              // resident CTAs per SM of the GEMM launched for T tokens

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

cudaError_t launch_gemm(const GemmArgs& a, int bits, int grid, int sms, cudaStream_t stream);
// The one-token 2-bit draft by table look-up (nest_lut.cu), and its error flag.
cudaError_t launch_lut(const GemmArgs& a, int sms, cudaStream_t stream);
cudaError_t read_and_clear_lut_error(int* flag, cudaStream_t stream);
cudaError_t read_and_clear_error(int* flag, cudaStream_t stream);
cudaError_t launch_wait_selftest(cudaStream_t stream);
cudaError_t launch_lut_wait_selftest(cudaStream_t stream);

// zero_out (optional): a buffer of zero_count floats the kernel also clears (the
// accumulator of the GEMM that follows it).
cudaError_t launch_rotate(const void* x, int x_dtype, const int8_t* signs, int n, int T, int mode,
                          float* y, uint16_t* xop, float* zero_out, long long zero_count, cudaStream_t stream);
// Rotation of several vector sets in one launch (same mode and input type); fills the
// tasks' L, NB, scale, total and cta_begin.
cudaError_t launch_rotate_group(RotArgs& a, int x_dtype, int mode, int T, cudaStream_t stream);

// Glue between chained linears (nest_chain): see nest_chain.cu.
struct GlueNext {
    const int8_t* sign_in;    // S_i of the next linear (length M)
    uint16_t* xop;            // its GEMM operand (out)
    float* zero_out;          // its GEMM accumulator, cleared here (optional)
    long long zero_count;
};
constexpr int kMaxChainNext = 3;
// An output rotation y = S_o H_o z of another linear run by extra CTAs (one-warp CTAs on the
// register path: warps) of the glue's first launch.
struct GlueSide {
    const float* z;
    const int8_t* s;
    float* y;
    int M, L, nseg, nchunk;   // length, log2 block size, 4096-segments and register chunks per token
    float scale;
    int cta_begin;            // first CTA (register path: first warp item) of the task in the launch
};
constexpr int kMaxChainSide = 2;
struct GlueArgs {
    const float* za;          // accumulator of linear a, [T][M], rotated basis
    const int8_t* sa;         // S_o of linear a
    const float* zb;          // optional product partner (same M)
    const int8_t* sb;
    float* h;                 // glue output before the RMS rescale, [T][M] (may be za)
    float* work;              // [T][nseg] segment sums of squares
    GlueNext next[kMaxChainNext];
    GlueSide side[kMaxChainSide];
    int nnext, nside, M, T, L, NB, nseg, nchunk;
    int glue_ctas;            // CTAs (register path: warp items) of the glue itself in the first launch
    float scale;
    int path;                 // 0 shared-memory tile, 2 segment (b >= 1024), 3 register with one-warp CTAs (b <= 512)
};
int glue_segments(int M);     // 4096-element segments per token
int glue_work_floats(int M, int T);   // floats of the work buffer of a glue call
cudaError_t launch_glue(GlueArgs& a, cudaStream_t stream);

cudaError_t launch_pack(const uint8_t* bc, const uint16_t* bs, const int8_t* rc, const uint16_t* rs,
                        int M, int K, int bits, uint8_t* base_out, uint8_t* resid_out, cudaStream_t stream);
cudaError_t launch_unpack(const uint8_t* base, const uint8_t* resid, int M, int K, int bits,
                          uint8_t* bc, uint16_t* bs, int8_t* rc, uint16_t* rs, cudaStream_t stream);

cudaError_t launch_pack_w4w8(const int8_t* q4, const uint16_t* s4, const int8_t* qr, int M, int K,
                             uint8_t* base_out, uint8_t* ref_out, cudaStream_t stream);
cudaError_t launch_unpack_w4w8(const uint8_t* base, const uint8_t* ref, int M, int K, int8_t* q4, uint16_t* s4,
                               int8_t* qr, cudaStream_t stream);
cudaError_t launch_quantize_w4w8(const float* W, const int8_t* so, const int8_t* si, int M, int K, double* work,
                                 int8_t* q4, uint16_t* s4, int8_t* qr, cudaStream_t stream);

cudaError_t launch_quantize(const float* W, const int8_t* so, const int8_t* si, int M, int K, int bits,
                            double* work, uint8_t* bc, uint16_t* bs, int8_t* rc, uint16_t* rs,
                            cudaStream_t stream);

int hadamard_block(int n);

// Nested KV cache (nest_kv.cu).
struct KvAttnArgs {
    const void* q;            // [T][Hq][128] queries
    int q_bf16;
    const uint8_t *kbase, *kref, *vbase, *vref;
    const uint16_t *kscale, *vscale;
    float* out;               // [T][Hq][128]
    float* work;              // per (head, tile, split, row): max, sum, 128 partial outputs
    int T, Hq, Hkv, G, L, Lmax, view, recent_n, nsplit, ntiles;
    int impl;                 // 0 tensor cores, 1 CUDA cores
};
cudaError_t launch_kv_write(const void* x, int bf16, int T, int H, int pos0, int Lmax, uint8_t* base, uint8_t* ref,
                            uint16_t* scale, cudaStream_t stream);
cudaError_t launch_kv_attention(KvAttnArgs& a, int sms, cudaStream_t stream);
int kv_rows_per_tile();
int kv_splits(int T, int G, int Hkv, int L, int sms);

}  // namespace nest
