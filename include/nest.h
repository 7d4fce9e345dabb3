/*
 * libnest -- nested-bit quantized linear layer for GB300 (sm_103a).
 *
 * One weight matrix W (M = d_out rows, K = d_in columns) is stored once, in
 * a randomized-Hadamard-rotated basis W~ = H_o S_o W S_i H_i, as
 *   - a 2-bit base: 4 Lloyd-Max levels (+-0.4528, +-1.5104) times an fp16
 *     scale per (row, 128-column group), the scale being the RMS of the block;
 *   - a b-bit residual (b = 6, 7, 8): the error W~ - Q_base on a uniform
 *     symmetric grid -qm..qm, qm = 2^(b-1) - 1, with an fp16 scale
 *     max|block|/qm per (row, 128-group).
 * Source: feedman.me/posts/wZBTJ (2-bit base in VRAM + residual in RAM
 * post), POC recipe steps 1-4.  The draft pass reads the base alone
 * (z = Q_base x'); the verify pass reads both parts in one weight-streaming
 * pass over all T tokens of a draft tree (z = (Q_base + Q_resid) x').  Base
 * and residual are separate buffers so the draft never fetches residual
 * bytes (BitNest, arXiv 2610.02800, section 3.3 "Dual-Plane Weight
 * Storage").
 *
 * Conventions for every entry point:
 *   - All data pointers are DEVICE pointers owned by the caller, except
 *     where an argument says "host".  The library allocates no memory.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t passed as
 *     void*; NULL is the legacy default stream).  No entry point
 *     synchronises, except nest_error_check.  Kernels are launched with
 *     programmatic dependent launch: each waits for the previous kernel in
 *     the stream before it reads that kernel's results or writes its outputs.
 *   - Arguments are validated on the host before any launch; a bad argument
 *     returns an error status and launches nothing.
 *   - Pointers must be 16-byte aligned unless stated otherwise
 *     (NEST_ERR_MISALIGNED otherwise).
 *   - Inputs and outputs must not overlap.
 *   - Supported envelope of the GEMMs: K % 128 == 0, any M >= 1,
 *     1 <= T <= 256.  Device: compute capability 10.3 (sm_103a).
 *
 * Storage format (packed buffers): arrays of UNITS, one unit per (tile of
 * 128 output rows, 128-column group), tile-major.  A base unit is 4352 bytes
 * (4096 bytes of 2-bit codes for 128 rows x 128 columns + 128 fp16 scales);
 * a residual unit is 2048*b + 256 bytes.  The bit layout inside a unit is
 * specified in nest_pack below.  Rows past M in the last tile are padding.
 *
 * Activation operand ("x_op"): the rotated activations x' = H_i S_i x in
 * fp16, laid out as the GEMM reads them: per 128-column group g, a block of
 * 256*Np bytes (Np = T rounded up to 16, 32, 64, 128 or 256); inside it, the fp16
 * value of token t, column k = 128 g + 8 c + e sits at byte
 * ((c * Np/8 + t/8) * 8 + t%8) * 16 + 2 e.  Rows t >= T are never read
 * into an output.
 */
#ifndef NEST_H
#define NEST_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    NEST_OK = 0,
    NEST_ERR_INVALID_ARG = 1,   /* null pointer, negative or zero size, bad enum */
    NEST_ERR_UNSUPPORTED = 2,   /* outside the supported envelope (K % 128, T > 256, bits, device) */
    NEST_ERR_MISALIGNED = 3,    /* a pointer is not 16-byte aligned */
    NEST_ERR_CUDA = 4,          /* a CUDA runtime call or a launch failed */
    NEST_ERR_TIMEOUT = 5        /* a kernel gave up waiting on a pipeline barrier (nest_error_check) */
} nest_status;

/* Weight codecs. */
#define NEST_CODEC_L2 0   /* 2-bit Lloyd-Max base + b-bit uniform residual (POC recipe steps 2, 3) */
#define NEST_CODEC_W4W8 1 /* BitNest W4 base + 4-bit refinement at s4/16, dual planes (BitNest 3.2, 3.3) */

/* A packed layer.  Plain descriptor; the pointers are device pointers owned by the caller. */
typedef struct {
    int32_t M;                  /* d_out, >= 1 */
    int32_t K;                  /* d_in, multiple of 128 */
    int32_t resid_bits;         /* NEST_CODEC_L2: 6, 7 or 8; NEST_CODEC_W4W8: 4; 0 = base only (draft-only layer) */
    const uint8_t* base;        /* nest_base_bytes(M, K) (L2) or nest_w4_base_bytes(M, K) (W4W8) bytes */
    const uint8_t* resid;       /* nest_resid_bytes(M, K, resid_bits) (L2) or nest_w4_ref_bytes(M, K) (W4W8)
                                   bytes, or NULL if resid_bits == 0 */
    const int8_t* sign_out;     /* S_o, M entries of +-1 */
    const int8_t* sign_in;      /* S_i, K entries of +-1 */
    int32_t codec;              /* NEST_CODEC_L2 (0, the default of a zeroed descriptor) or NEST_CODEC_W4W8 */
    int32_t group;              /* columns per scale group: 128, the storage format's group (0, the default of a
                                   zeroed descriptor, means 128); any other value returns NEST_ERR_UNSUPPORTED */
} nest_layer;

/* Human-readable name of a status. */
const char* nest_status_string(nest_status s);

/* ---- sizes (host-only, no device work) --------------------------------- */

/* Hadamard block size of a dimension n: the largest power of two dividing n,
 * capped at 4096 (feedman.me/posts/wZBTJ, POC recipe step 1).  0 if n < 1. */
int32_t nest_hadamard_block(int32_t n);

/* Bytes of the packed base buffer: ceil(M/128) * (K/128) * 4352.  0 if the shape is unsupported. */
size_t nest_base_bytes(int32_t M, int32_t K);

/* Bytes of the packed residual buffer: ceil(M/128) * (K/128) * (2048*bits + 256). */
size_t nest_resid_bytes(int32_t M, int32_t K, int32_t bits);

/* BitNest W4/W8 dual planes (NEST_CODEC_W4W8): ceil(M/128) * (K/128) units of 8448 bytes
 * (4-bit base codes + fp16 scales s4) and of 8192 bytes (4-bit refinement codes). */
size_t nest_w4_base_bytes(int32_t M, int32_t K);
size_t nest_w4_ref_bytes(int32_t M, int32_t K);

/* Bytes of the activation operand for K columns and T tokens: (K/128) * 256 * Np. */
size_t nest_xop_bytes(int32_t K, int32_t T);

/* ---- offline: quantize and pack --------------------------------------- */

/* RTN quantizer of one layer (feedman.me/posts/wZBTJ, POC recipe steps 1-3,
 * without the GPTQ/LDLQ error feedback), computed in fp64:
 *   W~ = H_o S_o W S_i H_i (block-diagonal Sylvester Hadamard, 1/sqrt(b));
 *   base: s_b = fp16(RMS of the (row, group) block), code = nearest level of
 *         W~/s_b (index 0..3 into -1.5104, -0.4528, +0.4528, +1.5104; |u| at the
 *         inner/outer midpoint goes inner, u == 0 goes to +0.4528; s_b == 0 gives code 2);
 *   residual: R = W~ - L[code] s_b; s_r = fp16(max|R| / qm);
 *             q = clip(rint(R / s_r), -qm, qm) (half to even; s_r == 0 gives 0).
 * W          float32 [M][K] (device).
 * sign_out   int8 [M] +-1; sign_in int8 [K] +-1.
 * work       fp64 scratch of M*K doubles (device, 16-byte aligned), overwritten.
 * base_codes uint8 [M][K] out (0..3); base_scales fp16 bits [M][K/128] out.
 * resid_codes int8 [M][K] out; resid_scales fp16 bits [M][K/128] out
 *            (both may be NULL when bits == 0).
 * Pointers to uint8/int8/fp16 arrays need only natural alignment. */
nest_status nest_quantize(const float* W, const int8_t* sign_out, const int8_t* sign_in,
                          int32_t M, int32_t K, int32_t bits, double* work,
                          uint8_t* base_codes, uint16_t* base_scales,
                          int8_t* resid_codes, uint16_t* resid_scales, void* stream);

/* Pack codes and scales into the unit format (storage of POC recipe steps 2-3).
 * base_codes  uint8 [M][K], values 0..3 (level index, ascending).
 * base_scales fp16 bits [M][K/128].
 * resid_codes int8 [M][K] in [-qm, qm]; resid_scales fp16 bits [M][K/128]
 *             (NULL with bits == 0 to pack the base alone).
 * base_out    nest_base_bytes(M, K) bytes; resid_out nest_resid_bytes(M, K, bits).
 * Unit bit layout (row r = 0..127 of the tile, a row's words are 32-bit little endian,
 * word w of row r at unit byte ((w/4)*128 + r)*16 + (w%4)*4):
 *   base: words 0..7; column 16w + 4p + q (p, q in 0..3) at bits 8q + 2p..8q + 2p + 1;
 *         fp16 scale of row r at unit byte 4096 + 2r.
 *   residual, stored u = q + 2^(b-1):
 *     b = 8: words 0..31, column 4w + q in byte q of word w;
 *     b = 6, 7: words 0..15 hold u & 15, column 8a + 4h + q of word a at bits 8q + 4h;
 *               words 16..23 hold (u >> 4) & 3, column 16a + 4p + q of word 16 + a at bits 8q + 2p;
 *               b = 7 only: words 24..27 hold (u >> 6) & 1, column 32a + 4p + q of word 24 + a at bit 8q + p;
 *     fp16 scale of row r at unit byte 2048*b + 2r.
 *   Rows past M: codes 0, residual q = 0, scales 0. */
nest_status nest_pack(const uint8_t* base_codes, const uint16_t* base_scales,
                      const int8_t* resid_codes, const uint16_t* resid_scales,
                      int32_t M, int32_t K, int32_t bits,
                      uint8_t* base_out, uint8_t* resid_out, void* stream);

/* BitNest W4/W8 offline quantizer (BitNest paper, Eq. (5)-(10)): rotate W as
 * nest_quantize does, then per (row, 128-group) s4 = fp16(max|W'| / 7), q4 =
 * clip(rint(W'/s4), -8, 7) (an RTN base: GPTQ needs calibration data), and
 * q_r = clip(rint((W' - q4 s4) / (s4/16)), q4 == -8 ? 0 : -8, 7), all in fp64.
 * work: M*K doubles (16-byte aligned).  q4, q_r: int8 [M][K] (q_r may be NULL: base only);
 * s4: fp16 bits [M][K/128]. */
nest_status nest_quantize_w4w8(const float* W, const int8_t* sign_out, const int8_t* sign_in,
                               int32_t M, int32_t K, double* work, int8_t* q4, uint16_t* s4, int8_t* q_r,
                               void* stream);

/* Dual-plane packing of W4/W8 codes.  q4 in [-8, 7], q_r in [-8, 7] (NULL: no refinement
 * plane, and ref_out may be NULL).  Unit layout (row r, 32-bit little-endian words, word w
 * of row r at unit byte ((w/4)*128 + r)*16 + (w%4)*4): word w holds columns 8w..8w+7,
 * column 8w + 4k + j in bits 8j + 4k .. 8j + 4k + 3, stored as code + 8; the base unit's
 * fp16 s4 of row r at byte 8192 + 2r.  Rows past M hold code 0 and scale 0. */
nest_status nest_pack_w4w8(const int8_t* q4, const uint16_t* s4, const int8_t* q_r, int32_t M, int32_t K,
                           uint8_t* base_out, uint8_t* ref_out, void* stream);

/* Inverse of nest_pack_w4w8 (tests).  q_r may be NULL. */
nest_status nest_unpack_w4w8(const nest_layer* layer, int8_t* q4, uint16_t* s4, int8_t* q_r, void* stream);

/* Inverse of nest_pack (used by tests).  resid_* may be NULL when layer->resid_bits == 0. */
nest_status nest_unpack(const nest_layer* layer, uint8_t* base_codes, uint16_t* base_scales,
                        int8_t* resid_codes, uint16_t* resid_scales, void* stream);

/* ---- per-forward kernels ----------------------------------------------- */

/* Randomized Hadamard rotation of T vectors of length n (POC recipe steps 1 and 4).
 * mode 0 (input side):  out_t = H S x_t   (signs first, then the block FWHT);
 * mode 1 (output side): out_t = S H x_t   (block FWHT first, then the signs).
 * H is block-diagonal with Sylvester blocks of size nest_hadamard_block(n), each scaled by 1/sqrt(b).
 * x        [T][n], fp32 (x_dtype 0) or bf16 bits (x_dtype 1); T * n < 2^31.
 * signs    int8 [n] +-1 (natural alignment).
 * y        fp32 [T][n] out, or NULL.
 * x_op     activation operand out (mode 0 only, n % 128 == 0, T <= 256), or NULL.
 * At least one of y, x_op must be given.  n >= 1, T >= 1. */
nest_status nest_rotate(const void* x, int32_t x_dtype, const int8_t* signs, int32_t n, int32_t T,
                        int32_t mode, float* y, uint16_t* x_op, void* stream);

/* The GEMM operand from an already-rotated activation block (POC recipe step 4, with x'
 * computed by the caller): x_op = fp16(x') in the operand layout above, round to nearest;
 * the padding tokens T <= t < Np are written as zeros.  nest_rotate produces the same
 * operand while it rotates; this call serves callers that hold x' = H_i S_i x in fp32.
 * x_rot  device fp32 [T][K] (4-byte aligned); x_op  nest_xop_bytes(K, T) bytes (16-byte aligned).
 * Limits: K % 128 == 0, 1 <= T <= 256, K * T < 2^31.  |x'| must stay within the fp16 range. */
nest_status nest_operand(const float* x_rot, int32_t K, int32_t T, uint16_t* x_op, void* stream);

/* Draft GEMV/GEMM: z[t][m] += sum_k Q_base[m][k] x'[t][k] for t < T, in the rotated
 * output basis (POC recipe step 4: the draft forward is the verifier's without y_r).
 * Reads the base buffer only.  For NEST_CODEC_W4W8 layers Q_base = q4 s4 (BitNest
 * Eq. (6)) and the verify below uses Q = (16 q4 + q_r) s4/16 (Eq. (10)).  A grouped
 * launch takes layers of one codec.
 * x_op  activation operand from nest_rotate or nest_operand (T tokens).
 * z     fp32 [T][M], ACCUMULATED into: clear it first for a plain product.  The
 *       128-column groups of a row are split across CTAs and each part is added with
 *       fp32 atomics, so the order of those additions (and the last bits of z) may
 *       differ between calls.  Calls that write the same z must not run concurrently
 *       unless that accumulation is intended. */
nest_status nest_draft_gemv(const nest_layer* layer, const uint16_t* x_op, float* z, int32_t T, void* stream);

/* Verify GEMM: z[t][m] += sum_k (Q_base + Q_resid)[m][k] x'[t][k] for t < T, one pass over
 * both buffers for all T tokens (POC recipe step 4: y_b + y_r before the output rotation).
 * Needs layer->resid_bits in {6, 7, 8}.  Arguments as nest_draft_gemv. */
nest_status nest_verify_gemm(const nest_layer* layer, const uint16_t* x_op, float* z, int32_t T, void* stream);

/* Grouped GEMMs: `count` (1..64) independent linears in ONE launch, e.g. the q/k/v
 * projections or the gate/up projections of a decoder layer, which read the same input,
 * or the independent linears of a batch of layers whose inputs are all ready.  Their
 * (row tile, group) units are concatenated and split evenly over the CTAs, which stay
 * resident and stream their contiguous ranges, so the launch's start-up and tail are
 * paid once for all of them.  layers: host array of `count` descriptors
 * (for verify, all with the same resid_bits); x_ops, z: host arrays of `count` device
 * pointers; each z[k] is fp32 [T][layers[k].M] and is accumulated into, as in
 * nest_draft_gemv / nest_verify_gemm.  T is shared. */
nest_status nest_draft_gemv_group(const nest_layer* layers, int32_t count, const uint16_t* const* x_ops,
                                  float* const* z, int32_t T, void* stream);
nest_status nest_verify_gemm_group(const nest_layer* layers, int32_t count, const uint16_t* const* x_ops,
                                   float* const* z, int32_t T, void* stream);

/* Whole linear: y = S_o H_o (Q x'), x' = H_i S_i x (rotate in, GEMM, rotate out).
 * verify  0 = draft (base only), 1 = verify (base + residual).
 * x       [T][K] fp32 (x_dtype 0) or bf16 bits (x_dtype 1).
 * y       fp32 [T][M] out.
 * scratch nest_linear_scratch_bytes(M, K, T) bytes of device memory (operand and
 *         accumulator; no initial contents needed).  Calls sharing a scratch buffer
 *         must be ordered (one stream). */
size_t nest_linear_scratch_bytes(int32_t M, int32_t K, int32_t T);
nest_status nest_linear(const nest_layer* layer, int32_t verify, const void* x, int32_t x_dtype,
                        int32_t T, float* y, void* scratch, void* stream);

/* Whole linears for `count` (1..64) independent layers in three launches (one grouped
 * rotation in, one grouped GEMM, one grouped rotation out).  layers: host array; xs, ys:
 * host arrays of device pointers ([T][K_k] inputs, [T][M_k] fp32 outputs); scratch:
 * nest_linear_group_scratch_bytes(layers, count, T) bytes of device memory. */
size_t nest_linear_group_scratch_bytes(const nest_layer* layers, int32_t count, int32_t T);
nest_status nest_linear_group(const nest_layer* layers, int32_t count, int32_t verify, const void* const* xs,
                              int32_t x_dtype, int32_t T, float* const* ys, void* scratch, void* stream);

/* Grouped rotation: `count` (1..64) independent nest_rotate calls sharing x_dtype, T and mode,
 * in ONE launch (e.g. one layer input rotated into the q, k and v operands, or the k and v
 * outputs rotated back).  Each task may also clear a buffer of zero_count floats (e.g. the
 * accumulator of the GEMM that reads its operand), which saves a separate fill launch.
 * Task fields have nest_rotate's meaning and limits; zero_out may be NULL when zero_count
 * is 0 and must not overlap any other buffer of the call. */
typedef struct {
    const void* x;          /* [T][n] fp32 or bf16 bits */
    const int8_t* signs;    /* int8 [n] */
    int32_t n;
    float* y;               /* fp32 [T][n] out, or NULL */
    uint16_t* x_op;         /* operand out (mode 0), or NULL */
    float* zero_out;        /* cleared here, or NULL */
    int64_t zero_count;     /* floats to clear */
} nest_rotate_task;
nest_status nest_rotate_group(const nest_rotate_task* tasks, int32_t count, int32_t x_dtype, int32_t T,
                              int32_t mode, void* stream);

/* Glue between chained linears, fused with the rotations on both sides of it:
 *   h = S_o H_o z_a  (or the elementwise product h_a * h_b of two linears' outputs, e.g. gate * up),
 *   h' = bf16(h / rms(h)) per token (unit-RMS rescale standing in for the normalisation
 *        between linears, then the bf16 cast),
 *   and for each of n_next (0..3) next linears j: x'_j = H_i S_i h' written as its GEMM operand.
 * The rotations are those of POC recipe steps 1 and 4 (feedman.me/posts/wZBTJ); the chaining
 * and the RMS rescale are the chained-layer workload's reading, not the pages'.
 * Two launches (rotation out with partial sums of squares per token and chunk or segment;
 * rescale, cast and rotation in).
 * z_a           fp32 [T][M] GEMM accumulator of linear a (rotated basis).  When y is NULL, h
 *               overwrites z_a.
 * z_b           NULL, or the accumulator of the product partner (fp32 [T][M], read only);
 *               sign_out_b is NULL exactly when z_b is.  z_b must differ from z_a and y.
 * sign_out_a/b  S_o of those linears (int8 [M]).
 * y             NULL, or fp32 [T][M] out: h (the product when z_b is given), kept by the caller.
 * next          host array of n_next layer descriptors; each must have K == M (its sign_in is used).
 * x_ops         host array of n_next operand buffers (out, nest_xop_bytes(M, T) bytes each).
 * z_next        NULL, or host array of n_next accumulators (fp32 [T][next[j].M], or NULL entries)
 *               that are cleared here for the GEMMs that follow.
 * work          nest_chain_work_bytes(M, T) bytes of device memory (one fp32 partial sum of
 *               squares per token and 256/512-element chunk when the block size is at most 512,
 *               else per token and 4096-element segment), no initial contents; calls whose work
 *               may overlap on the GPU need separate work buffers.
 * side          NULL, or host array of n_side (0..2) output rotations y = S_o H_o z of other
 *               linears (e.g. the k and v outputs of the layer whose q output this glue reads),
 *               run as extra CTAs of the glue's first launch, so they add no launch to the
 *               chain.  Each task: x = z (fp32 [T][n], read only), signs = its S_o, y (fp32
 *               [T][n] out), x_op and zero_out NULL; n >= 1, n * T < 2^31, 4-byte aligned.
 *               A task whose block size falls on another path than the glue's runs in a
 *               launch of its own.  Its z and y must not overlap z_a, z_b, y or each other.
 * Limits: T <= 256, M * T < 2^31, M % 128 == 0 when n_next > 0. */
size_t nest_chain_work_bytes(int32_t M, int32_t T);
nest_status nest_chain(float* z_a, const int8_t* sign_out_a, const float* z_b, const int8_t* sign_out_b,
                       int32_t M, int32_t T, float* y, const nest_layer* next, int32_t n_next,
                       uint16_t* const* x_ops, float* const* z_next, float* work,
                       const nest_rotate_task* side, int32_t n_side, void* stream);

/* nest_linear without caller scratch, for callers that cannot allocate device memory
 * (a process whose memory pool is fixed at start-up, a plain C caller without an
 * allocator, a loop that cannot afford cudaMalloc's implicit synchronisation).  None of
 * the source pages has a counterpart; this is a library convenience.  Arguments as
 * nest_linear minus `scratch`: the operand and the accumulator live in one fixed 8 MiB
 * array of the library's device memory, held by every GPU that loads the library until
 * the process exits.  Shapes with nest_linear_scratch_bytes(M, K, T) > 8 MiB return
 * NEST_ERR_UNSUPPORTED without launching.  The first call on a device looks up the
 * array's address for that device (make that call before any stream capture).  Calls
 * share the array: calls whose work overlaps on the GPU (other streams or threads) race
 * and must be serialised by the caller; nothing needs clearing between calls.  The looked-up
 * address is cached per device: cudaDeviceReset on a device ends the context holding the
 * array, so do not call this entry point on that device again in the same process.
 * Allocates nothing (no cudaMalloc, cudaFree or allocating library routine). */
nest_status nest_linear_static(const nest_layer* layer, int32_t verify, const void* x, int32_t x_dtype,
                               int32_t T, float* y, void* stream);

/* ---- row-sharded linears (several GPUs) ---------------------------------- */

/* Reorder of a row-sharded linear's all-gathered output.  No page has a counterpart
 * (the pages run on one device); this is the library's split of one linear over `world`
 * GPUs by output rows.  Rank r holds whole 128-row tiles of the packed layer: rows
 * [r * Mp, min((r + 1) * Mp, M)) with Mp = 128 * ceil(ceil(M / 128) / world), a view of
 * its tiles' units (the packed buffers are tile-major).  Every rank rotates the
 * replicated input itself (nest_rotate) and runs the draft or verify GEMM on its M_r =
 * min(Mp, M - r * Mp) rows into the first T * M_r floats ([T][M_r]) of a block of T * Mp
 * floats; one all-gather of those blocks (e.g. NCCL) gives every rank gathered =
 * [world][T * Mp].  This call writes
 *   z[t][r * Mp + j] = gathered[r * T * Mp + t * M_r + j]   for j < M_r,
 * the token-major [T][M] rotated-basis output that nest_rotate (mode 1) turns into y.
 * gathered: device fp32, world * T * Mp floats; z: device fp32 [T][M], not overlapping it.
 * Limits: world, T, Mp, M >= 1, M <= world * Mp, world * T * Mp < 2^31; 4-byte aligned. */
nest_status nest_shard_gather(const float* gathered, float* z, int32_t world, int32_t T, int32_t Mp, int32_t M,
                              void* stream);

/* ---- nested KV4/KV8 cache (BitNest paper, Section 3.4, Appendix A.2) ------ */

/* One cache (keys or values) of H heads x Lmax positions, head dimension 128.
 *   base  [H][Lmax][64] bytes: byte i of a row holds dims 2i (low nibble) and 2i+1
 *                              (high nibble) as q4 + 8;
 *   ref   [H][Lmax][64] bytes: the refinement codes q_r + 8, same layout;
 *   scale [H][Lmax] fp16 bits: s = max|x| / 7 of the row.
 * base and ref 16-byte aligned, scale 2-byte aligned; nest_kv_plane_bytes(H, Lmax)
 * bytes each for base and ref, 2*H*Lmax bytes for scale.  A plane holds fewer than
 * 2^32 bytes (H * Lmax < 2^26); larger caches give NEST_ERR_UNSUPPORTED. */
typedef struct {
    uint8_t* base;
    uint8_t* ref;
    uint16_t* scale;
    int32_t H;
    int32_t Lmax;
} nest_kv_cache;

size_t nest_kv_plane_bytes(int32_t H, int32_t Lmax);

/* Quantise-on-write (Eq. (11), (13)): the key or value vectors x [T][H][128] (fp32 for
 * x_dtype 0, bf16 bits for 1) of T new tokens are stored at positions pos0 .. pos0+T-1:
 * s = fp16(max|x| / 7), q4 = clip(rint(x / s), -8, 7), q_r = clip(rint((x - q4 s) /
 * (s / 16)), -8, 7), decided in fp32 with each operation rounded on its own.
 * Needs 0 <= pos0, pos0 + T <= Lmax, 1 <= T. */
nest_status nest_kv_write(const void* x, int32_t x_dtype, int32_t T, const nest_kv_cache* cache, int32_t pos0,
                          void* stream);

/* Decode attention over the nested caches (grouped-query: query head h reads KV head
 * h / (Hq / Hkv)).  q [T][Hq][128] (fp32 or bf16 bits per q_dtype) are the queries of
 * the T newest tokens, whose keys and values are already written at positions
 * L-T .. L-1; query t sees positions 0 .. L-T+t (causal), scores q.k / sqrt(128),
 * softmax, out [T][Hq][128] fp32 = sum p v.
 * view 8: the KV8 view (16 q4 + q_r) s / 16 everywhere (verification);
 * view 4: the KV4 view q4 s (drafting), except positions >= L - recent_n, read at KV8
 *         (the Recent-N policy; recent_n = 0 is pure KV4).
 * work: nest_kv_attention_work_bytes(T, Hq, Hkv, L) bytes of device memory (no
 * initial contents); two launches (position splits, then their combination).
 * Needs Hq % Hkv == 0, k->H == v->H == Hkv, k->Lmax == v->Lmax, T <= L <= Lmax. */
size_t nest_kv_attention_work_bytes(int32_t T, int32_t Hq, int32_t Hkv, int32_t L);
nest_status nest_kv_attention(const void* q, int32_t q_dtype, int32_t T, int32_t Hq, const nest_kv_cache* k,
                              const nest_kv_cache* v, int32_t L, int32_t view, int32_t recent_n, float* out,
                              float* work, void* stream);

/* Reads and clears the device-side error flags that kernels set when a pipeline
 * wait runs past its limit (one for the tensor-core and register-fragment GEMM
 * kernels, one for the one-token look-up kernel).  Synchronises `stream`.  Returns
 * NEST_ERR_TIMEOUT if either flag was set, NEST_ERR_CUDA on a CUDA error, NEST_OK
 * otherwise. */
nest_status nest_error_check(void* stream);

/* The give-up path of the kernels' bounded waits, exercised without a fault: launches
 * one warp that waits, through the same bounded wait as the pipelines of the GEMM
 * kernels (which = 0) or of the one-token look-up kernel (which = 1), on a barrier that
 * nothing arrives on.  The wait gives up after its limit (2 s), raises that kernel
 * family's device error flag and the kernel returns, so the context stays usable and
 * the next nest_error_check returns NEST_ERR_TIMEOUT (and clears the flag).
 * Asynchronous on `stream`; NEST_ERR_INVALID_ARG for another `which`, NEST_ERR_CUDA if
 * the launch fails. */
nest_status nest_wait_selftest(int32_t which, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* NEST_H */
