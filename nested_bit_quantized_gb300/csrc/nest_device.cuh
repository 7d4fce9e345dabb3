// Device-side building blocks shared by the libnest kernels: constants of the
// storage format and mbarrier / bulk-copy / tcgen05 wrappers in inline PTX.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_bf16.h>

namespace nest {

constexpr int kRows = 128;           // output rows per tile (one TMEM lane each)
constexpr int kGroup = 128;          // columns per quantisation group
constexpr int kBaseUnit = 4096 + 256;
__host__ __device__ constexpr int resid_unit_bytes(int bits) { return bits ? 2048 * bits + 256 : 0; }
// W4/W8 dual-plane units (BitNest section 3.3): 4-bit base codes + fp16 scales, 4-bit refinement codes
constexpr int kW4BaseUnit = 8192 + 256;
constexpr int kW4RefUnit = 8192;
constexpr int kHadCap = 4096;

// Levels of the 2-bit base, ascending (the Gaussian 4-level Lloyd-Max set).
__host__ __device__ constexpr double level_d(int c) {
    return c == 0 ? -1.5104 : (c == 1 ? -0.4528 : (c == 2 ? 0.4528 : 1.5104));
}
__host__ __device__ constexpr float level_f(int c) { return (float)level_d(c); }

// ---------------------------------------------------------------------------
// shared-memory addresses, mbarriers, bulk copies
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.shared::cta.b64 st, [%0];\n}" :: "r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}"
                 :: "r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
                 " selp.u32 %0, 1, 0, p;\n}" : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}

// Non-blocking test of a barrier phase.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
                 " selp.u32 %0, 1, 0, p;\n}" : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}

// 1-D bulk copy global -> shared, completing transaction bytes on `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 :: "r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

// programmatic dependent launch: wait for the previous grid in the stream to
// complete (and its writes to be visible); allow the next grid to launch
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// bounded waits
// ---------------------------------------------------------------------------

constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait for a whole warp (all 32 lanes converged); the result is the
// same on every lane.  Gives up after kWaitLimitNs, or at once when another
// role of the CTA has given up (*abort != 0) unless `honour_abort` is false
// (used while draining in-flight copies and MMAs); on a timeout it raises the
// CTA's abort flag and the device error flag *err.
__device__ inline bool warp_wait_flag(uint32_t bar, uint32_t parity, volatile int* abort, int* err,
                                      bool honour_abort = true) {
    bool ok = mbar_try_wait(bar, parity);
    if (__all_sync(0xffffffffu, ok)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t it = 0;; ++it) {
        if (!ok) ok = mbar_try_wait(bar, parity);
        if (__all_sync(0xffffffffu, ok)) return true;
        const bool timed_out = (it & 31u) == 31u && globaltimer() - t0 > kWaitLimitNs;
        const bool stop = timed_out || (honour_abort && *abort != 0);
        if (__any_sync(0xffffffffu, stop)) {
            if (__any_sync(0xffffffffu, timed_out) && (threadIdx.x & 31) == 0) {
                *abort = 1;
                atomicExch(err, 1);
            }
            return false;
        }
    }
}

// named barrier over `count` threads
__device__ __forceinline__ void named_sync(uint32_t id, uint32_t count) {
    asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(count) : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory, MMA, commit
// ---------------------------------------------------------------------------

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(dst_smem), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tc_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Arrive on `bar` once all tcgen05 operations issued so far by this thread have completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 :: "r"(bar) : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc], kind::f16 (fp16 inputs, fp32 accumulate).
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
    asm volatile("{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
                 " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}"
                 :: "r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}

// Shared-memory matrix descriptor, no swizzle, K-major core matrices of 8 rows x 16 bytes:
// lbo = byte distance between core matrices adjacent along K,
// sbo = byte distance between core matrices adjacent along M/N.
__device__ __forceinline__ uint64_t smem_desc_noswizzle(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((addr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;            // descriptor version for tcgen05
    return d;                          // base offset 0, lbo mode 0, swizzle none
}

// Instruction descriptor, kind::f16: A = B = fp16, D = fp32, both K-major.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
    return (1u << 4)                       // D format f32
         | (0u << 7) | (0u << 10)          // A, B format f16
         | ((uint32_t)(N >> 3) << 17)
         | ((uint32_t)(M >> 4) << 24);
}

// 32 lanes x 32 bit, 32 columns: each thread writes registers v[0..31] to its lane.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {"
                 "%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
                 "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
                 :: "r"(taddr),
                    "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
                    "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]),
                    "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]),
                    "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
                 : "memory");
}

// 32 lanes x 32 bit, 16 columns: each thread writes registers v[0..15] to its lane.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {"
                 "%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
                 :: "r"(taddr),
                    "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
                    "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
                 : "memory");
}

// 32 lanes x 32 bit, 16 columns: each thread reads its lane's 16 columns.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {"
                 "%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                 : "r"(taddr) : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// ---------------------------------------------------------------------------
// fast Walsh-Hadamard butterflies
// ---------------------------------------------------------------------------

// Butterflies over the low `nbits` bits of a 64-element warp vector:
// element `lane` in v0, element `lane + 32` in v1 (unnormalised Sylvester order).
__device__ __forceinline__ void warp_fwht(float& v0, float& v1, int nbits, int lane) {
    const int lane_bits = nbits < 5 ? nbits : 5;
    for (int s = 0; s < lane_bits; ++s) {
        const int m = 1 << s;
        const float o0 = __shfl_xor_sync(0xffffffffu, v0, m);
        const float o1 = __shfl_xor_sync(0xffffffffu, v1, m);
        const bool upper = (lane & m) != 0;
        v0 = upper ? o0 - v0 : v0 + o0;
        v1 = upper ? o1 - v1 : v1 + o1;
    }
    if (nbits >= 6) {
        const float a = v0 + v1, b = v0 - v1;
        v0 = a;
        v1 = b;
    }
}

// This CTA's share (of nctas CTAs of THREADS threads) of clearing `count` floats at p:
// 16-byte stores when p and count allow them.
template <int THREADS>
__device__ __forceinline__ void clear_share(float* p, long long count, unsigned cta, unsigned nctas) {
    if ((reinterpret_cast<uintptr_t>(p) & 15u) == 0 && (count & 3) == 0) {
        float4* q = reinterpret_cast<float4*>(p);
        const long long c4 = count >> 2, per = (c4 + nctas - 1) / nctas;
        const long long lo = per * cta, hi = lo + per < c4 ? lo + per : c4;
        for (long long i = lo + threadIdx.x; i < hi; i += THREADS) q[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    } else {
        const long long per = (count + nctas - 1) / nctas;
        const long long lo = per * cta, hi = lo + per < count ? lo + per : count;
        for (long long i = lo + threadIdx.x; i < hi; i += THREADS) p[i] = 0.0f;
    }
}

// Sign j (0 <= j < 8 H) of a register chunk whose lane holds 8 signs per h in sg[h].
template <int H>
__device__ __forceinline__ float chunk_sign(const uint2 (&sg)[H], int j) {
    return (float)(int8_t)((((j & 7) < 4 ? sg[j >> 3].x : sg[j >> 3].y) >> (8 * (j & 3))) & 0xFFu);
}

// Block-diagonal FWHT (unnormalised Sylvester order, blocks of 2^L <= 256 H elements) of
// one warp's chunk of 256 H consecutive elements held in registers: element 256 h + 8 l + i
// of the chunk in v[8 h + i] of lane l (i < 8, h < H).  Index bits 0-2 and 8 and up are
// butterflies inside the lane, bits 3-7 warp shuffles.  All 32 lanes call it.
template <int H>
__device__ __forceinline__ void chunk_fwht(float (&v)[8 * H], int L, int lane) {
    constexpr int NR = 8 * H;
#pragma unroll
    for (int b = 0; b < 3; ++b) {
        if (b < L) {
#pragma unroll
            for (int j = 0; j < NR; ++j) {
                if (j & (1 << b)) continue;
                const float a = v[j], d = v[j + (1 << b)];
                v[j] = a + d;
                v[j + (1 << b)] = a - d;
            }
        }
    }
    for (int b = 3; b < 8 && b < L; ++b) {
        const int m = 1 << (b - 3);
        const bool upper = (lane & m) != 0;
#pragma unroll
        for (int j = 0; j < NR; ++j) {
            const float o = __shfl_xor_sync(0xffffffffu, v[j], m);
            v[j] = upper ? o - v[j] : v[j] + o;
        }
    }
#pragma unroll
    for (int q = 0; (8 << q) < NR; ++q) {
        if (8 + q < L) {
#pragma unroll
            for (int j = 0; j < NR; ++j) {
                if (j & (8 << q)) continue;
                const float a = v[j], d = v[j + (8 << q)];
                v[j] = a + d;
                v[j + (8 << q)] = a - d;
            }
        }
    }
}

// Segment path of the FWHT for blocks of 2^L, 10 <= L <= 12: one CTA of 512 threads per
// 4096-element segment, seen as 16 rows x 256 columns (element 256 r + c).  The butterflies
// over index bits 8 .. L-1 run first, each thread holding rows of one column in registers
// (phase A, seg_col and seg_rows_fwht); one pass through shared memory; then bits 0 .. 7
// along the rows, warp w holding row w in the chunk layout (phase B, seg_row_load and
// chunk_fwht<1>).  The stage order does not change the transform.
struct SegCol {
    int c, r0, nr;            // column, first row, rows held (0: idle in phase A)
};
__device__ __forceinline__ SegCol seg_col(int L) {
    const int t = threadIdx.x;
    if (L >= 12) return SegCol{t & 255, 0, t < 256 ? 16 : 0};
    return SegCol{t & 255, 8 * (t >> 8), 8};
}
// v[k] holds row r0 + k of the thread's column; butterflies over row bits 0 .. L-9.
__device__ __forceinline__ void seg_rows_fwht(float (&v)[16], int L) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        if (q < L - 8) {
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                if (k & (1 << q)) continue;
                const float a = v[k], d = v[k + (1 << q)];
                v[k] = a + d;
                v[k + (1 << q)] = a - d;
            }
        }
    }
}
__device__ __forceinline__ void seg_col_store(float* sm, const SegCol& sc, const float (&v)[16]) {
#pragma unroll
    for (int k = 0; k < 16; ++k)
        if (k < sc.nr) sm[(sc.r0 + k) * 256 + sc.c] = v[k];
}
// Phase B input of warp w: row w, lane l's elements 8 l .. 8 l + 7.
__device__ __forceinline__ void seg_row_load(const float* sm, int w, int lane, float (&v)[8]) {
    const float4 a = *reinterpret_cast<const float4*>(sm + w * 256 + 8 * lane);
    const float4 b = *reinterpret_cast<const float4*>(sm + w * 256 + 8 * lane + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// Chunk of the register-path FWHT for blocks of 2^L (L <= 9): 256 or 512 elements.
__host__ __device__ constexpr int reg_chunk(int L) { return L <= 8 ? 256 : 512; }

// Block-diagonal FWHT (unnormalised, blocks of 2^L, 0 <= L <= 12) of the 4096 values
// of a 64 x 64 shared-memory tile, value f at tile[f / 64][f % 64]: butterflies over
// index bits 0..5 along rows, then bits 6..11 along columns (the padding column keeps
// the column pass free of bank conflicts).  Every thread of the CTA (THREADS of them)
// calls it; the tile is complete on return.
template <int THREADS>
__device__ __forceinline__ void tile_fwht(float (*tile)[65], int L) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int L1 = L < 6 ? L : 6;
    if (L1 > 0) {
        for (int row = warp; row < 64; row += THREADS / 32) {
            float v0 = tile[row][lane], v1 = tile[row][lane + 32];
            warp_fwht(v0, v1, L1, lane);
            tile[row][lane] = v0;
            tile[row][lane + 32] = v1;
        }
        __syncthreads();
    }
    if (L > 6) {
        for (int col = warp; col < 64; col += THREADS / 32) {
            float v0 = tile[lane][col], v1 = tile[lane + 32][col];
            warp_fwht(v0, v1, L - 6, lane);
            tile[lane][col] = v0;
            tile[lane + 32][col] = v1;
        }
        __syncthreads();
    }
}

// Sum over all THREADS threads of the CTA; every thread gets the total.  red: 32 floats
// of shared memory.
template <int THREADS>
__device__ __forceinline__ float cta_sum(float v, float* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float t = lane < THREADS / 32 ? red[lane] : 0.0f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    __syncthreads();
    return t;
}

// Offset in bytes of token t, columns k..k+7 (k % 8 == 0) in the fp16 GEMM operand of
// NB token blocks: per 128-column group g, core matrices of 8 tokens x 8 columns (16-byte
// rows), column-block c major, token block minor.
__device__ __forceinline__ size_t xop_offset(int k, int t, int NB) {
    const int g = k >> 7, c = (k & 127) >> 3;
    return (size_t)g * 2048 * NB + ((size_t)(c * NB + (t >> 3)) * 8 + (t & 7)) * 16;
}

// ---------------------------------------------------------------------------
// small integer / half helpers
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u32_as_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

}  // namespace nest
