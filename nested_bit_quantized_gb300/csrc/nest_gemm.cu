// Draft and verify GEMMs of the nested-bit linear layer on tcgen05 tensor cores.
//
//   draft : z[t][m] = sum_k Q_base[m][k] x'[t][k]
//   verify: z[t][m] = sum_k (Q_base + Q_resid)[m][k] x'[t][k]
// (feedman.me/posts/wZBTJ, POC recipe step 4: y_b = Q_base x', y_r = Q_resid x';
//  the draft is the same without y_r.)  All T tokens share one pass over the
// packed weights, so the weight bytes are streamed from HBM once per call.
//
// Design (warp-specialised pipeline; two CTAs per SM up to 64 tokens, one at 128 and 256):
//   producer warp  : 1-D bulk copies (TMA engine) of one unit per stage -- the
//                    base unit, the residual unit and the fp16 activation block
//                    of the unit's 128-column group -- into shared memory.
//   dequant warps  : two warpgroups (four at 128 and 256 tokens); thread r of a
//                    warpgroup owns row r of the tile.  It decodes its row's 128 weights of the unit into
//                    fp16 w = s_b*L[code] + s_r*q in registers (PRMT look-up of
//                    the four scaled levels, fp16 magic-number decode of the
//                    residual) and stores them to tensor memory with tcgen05.st.
//   MMA thread     : tcgen05.mma kind::f16, A = the dequantised weights in tensor
//                    memory (128 x 16 per instruction), B = the activation block
//                    in shared memory (Np x 16), D = fp32 accumulators in tensor
//                    memory (128 lanes x Np columns).
//   epilogue       : warpgroup 0 (at 128 tokens and more every warpgroup, each
//                    for its share of the columns) reads D with tcgen05.ld and
//                    adds it into z.
// Work split: the (tile, group) units, tile-major, are cut into equal
// contiguous ranges, one per CTA ("stream-K").  Every CTA adds the sums of
// each row-tile segment it covers into z with fp32 reductions (z += ...), so a
// tile split across CTAs needs no workspace and no inter-CTA handshake; the
// order in which the split parts land is not fixed.
// Launches use programmatic dependent launch: a CTA sets up its barriers and
// tensor memory and starts streaming weights before the previous kernel in the
// stream has finished; it waits for it (griddepcontrol.wait) only before it
// reads the activation operand or touches z.
#include <cstdlib>

#include "nest_device.cuh"
#include "nest_internal.h"

namespace nest {

__device__ int g_nest_error;

namespace {

// Bounded wait of a whole warp (see warp_wait_flag); a timeout raises g_nest_error.
__device__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort, bool honour_abort = true) {
    return warp_wait_flag(bar, parity, abort, &g_nest_error, honour_abort);
}

// The give-up path of the bounded wait, on its own: one warp waits on a barrier that
// nothing arrives on, so the wait runs out after kWaitLimitNs, raises the CTA's abort
// flag and the device error flag, and the kernel returns normally.
__global__ void __launch_bounds__(32) k_wait_selftest() {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    warp_wait(smem_u32(&bar), 0, &abort_flag);
}

// Weight codecs of the GEMM kernels (template parameter BITS):
//   0        2-bit Lloyd-Max base only (draft)
//   6, 7, 8  2-bit base + b-bit uniform residual (verify)
//   40       BitNest W4 base only (draft)
//   48       BitNest W4 base + 4-bit refinement, the W8 target (verify)
__host__ __device__ constexpr bool is_w4(int codec) { return codec >= 40; }
__host__ __device__ constexpr int base_unit_bytes(int codec) { return is_w4(codec) ? kW4BaseUnit : kBaseUnit; }
__host__ __device__ constexpr int second_unit_bytes(int codec) {
    return codec == 48 ? kW4RefUnit : (is_w4(codec) ? 0 : resid_unit_bytes(codec));
}

template <int BITS, int NP>
struct Cfg {
    // Up to 64 tokens two CTAs share an SM: each has its own MMA issuer, so the gaps
    // in one CTA's MMA stream (barrier waits, commits) are filled by the other's.
    // 128 and 256 tokens (prefill-size trees) take a whole SM: its 512 tensor-memory
    // columns hold the 128 x Np accumulator(s) and the A buffers, and 220 KB of shared
    // memory the 32-64 KB activation blocks.
    static constexpr int kCtasPerSm = NP >= 128 ? 1 : 2;
    static constexpr int kBaseBytes = base_unit_bytes(BITS);
    static constexpr int kResUnit = second_unit_bytes(BITS);
    static constexpr int kWStage = kBaseBytes + kResUnit;    // packed weights of one unit
    static constexpr int kXBytes = 256 * NP;                 // Np tokens x 128 columns of fp16
    static constexpr int kTmemCols = 512 / kCtasPerSm;
    static constexpr int kNumD = NP >= 256 ? 1 : 2;          // accumulator buffers
    static constexpr int kColA = kNumD * NP;                 // A buffers after the D buffers
    static constexpr int kNumARaw = (kTmemCols - kColA) / 64;
    static constexpr int kMaxA = NP >= 256 ? 2 : (NP >= 128 ? 4 : 8);   // activation slots the smem holds
    static constexpr int kNumA = kNumARaw < kMaxA ? kNumARaw : kMaxA;   // A buffers (64 columns) = activation slots
    static constexpr int kXRing = kNumA * kXBytes;
    static constexpr int kSmemBudget = kCtasPerSm == 1 ? 220 * 1024 : 110 * 1024;
    static constexpr int kStagesRaw = (kSmemBudget - 512 - kXRing) / kWStage;
    static constexpr int kStages = kStagesRaw > 16 ? 16 : kStagesRaw;
    // dequantising warpgroups: a CTA that has the SM to itself (128 and 256 tokens) runs
    // four, so that the decode keeps up with the longer MMAs.  At 128 tokens each takes
    // whole units (one per activation slot); at 256 the smem holds only two activation
    // slots, so two warpgroups share each unit, one 64-column half each.
    static constexpr int kDeqWG = NP >= 128 ? 4 : 2;
    static constexpr int kUnitWG = NP >= 256 ? 2 : 1;        // warpgroups per unit
    // warpgroups that run the epilogues: all of them at 128 tokens and more (each reads
    // and reduces its share of the accumulator columns), warpgroup 0 alone below
    static constexpr int kEpiWG = NP >= 128 ? kDeqWG : 1;
    static constexpr int kProducerWarp = 4 * kDeqWG;
    static constexpr int kMmaWarp = 4 * kDeqWG + 1;
    static constexpr int kThreads = 32 * (4 * kDeqWG + 2);
    // barriers: full_w[S], empty_w[S], full_x[NA], a_full[NA], done[NA], d_full[ND], d_empty[ND], drain
    static constexpr int kNumBars = 2 * kStages + 3 * kNumA + 2 * kNumD + 1;
    static constexpr int kSmemBytes = kStages * kWStage + kXRing + kNumBars * 8 + 16;
    static_assert(kNumA >= 2, "tensor memory budget");
    static_assert(kStages >= 2, "stage too large");
    static_assert(kStages % kDeqWG == 0 || kStages >= kNumA, "weight-stage phase order needs S >= NA when S is odd");
    static_assert(kDeqWG % kUnitWG == 0 && (kUnitWG == 1 || kUnitWG == 2), "warpgroups per unit");
    static_assert(kSmemBytes <= kSmemBudget, "shared memory budget");
    static_assert(kWStage % 128 == 0 && kXBytes % 128 == 0, "stage alignment");
    static_assert(NP < 128 || (NP / kEpiWG) % 32 == 0, "epilogue columns per warpgroup");
};

// W4/W8: decode 64 columns (half h) of row r into 32 fp16x2 registers, w = c * s4 with
// c = q4 (draft) or 16 q4 + q_r (verify; the epilogue applies the 1/16 of s_ref = s4/16).
// Word w of a row's nibble plane holds columns 8w..8w+7 (column 8w + 4k + j in bits
// 8j + 4k), so for Q = 16h + qd the four columns 4Q..4Q+3 are the k = qd & 1 nibbles of
// word 8h + qd/2.  With offset nibbles u4 = q4 + 8, u_r = q_r + 8 the byte u4 * 16 + u_r
// equals 16 q4 + q_r + 136, so one shift and one masked select build four target codes.
template <int BITS>
__device__ __forceinline__ void dequant_half_w4(const uint8_t* sb, const uint8_t* sr, int r, int h, __half2 s2,
                                                __half2 off2, uint32_t (&out)[32]) {
    uint32_t bw[8], rw[8];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        const uint4 v = *reinterpret_cast<const uint4*>(sb + ((2 * h + c) * kRows + r) * 16);
        bw[4 * c] = v.x; bw[4 * c + 1] = v.y; bw[4 * c + 2] = v.z; bw[4 * c + 3] = v.w;
        if constexpr (BITS == 48) {
            const uint4 u = *reinterpret_cast<const uint4*>(sr + ((2 * h + c) * kRows + r) * 16);
            rw[4 * c] = u.x; rw[4 * c + 1] = u.y; rw[4 * c + 2] = u.z; rw[4 * c + 3] = u.w;
        }
    }
#pragma unroll
    for (int qd = 0; qd < 16; ++qd) {
        const uint32_t wb = bw[qd >> 1];
        uint32_t b4;
        if constexpr (BITS == 48) {
            const uint32_t wr = rw[qd >> 1];
            b4 = (qd & 1) ? ((wb & 0xF0F0F0F0u) | ((wr >> 4) & 0x0F0F0F0Fu))
                          : (((wb << 4) & 0xF0F0F0F0u) | (wr & 0x0F0F0F0Fu));
        } else {
            b4 = (qd & 1) ? ((wb >> 4) & 0x0F0F0F0Fu) : (wb & 0x0F0F0F0Fu);
        }
        // 1024 + byte as fp16 (exact), minus 1024 + offset, times s4
        const __half2 c01 = __hsub2(u32_as_h2(prmt(b4, 0x64646464u, 0x5140u)), off2);
        const __half2 c23 = __hsub2(u32_as_h2(prmt(b4, 0x64646464u, 0x7362u)), off2);
        out[2 * qd] = h2_as_u32(__hmul2(c01, s2));
        out[2 * qd + 1] = h2_as_u32(__hmul2(c23, s2));
    }
}

// Decode 32 columns (quarter qq of half h of the 128-column group) of row r of one unit
// into 16 fp16x2 registers: w = s_b * L[code] (+ s_r * q).  Quarter-size pieces keep 16
// results live instead of 32, which takes the kernel from 96 to 79 registers at b = 7 and
// leaves room on the SM for the small rotation CTAs that run beside it.  Local index l
// stands for qd = 8 qq + l of the half; every shift below depends on qd & 7 = l only.
template <int BITS>
__device__ __forceinline__ void dequant_quarter(const uint8_t* sb, const uint8_t* sr, int r, int h, int qq,
                                                uint32_t lut_lo, uint32_t lut_hi, __half2 sr2, __half2 off2,
                                                uint32_t (&out)[16]) {
    const uint2 bw2 = *reinterpret_cast<const uint2*>(sb + (h * kRows + r) * 16 + 8 * qq);
    const uint32_t bw[2] = {bw2.x, bw2.y};
    uint32_t rw[8];
    uint32_t mid[2], hi = 0;
    if constexpr (BITS == 8) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const uint4 v = *reinterpret_cast<const uint4*>(sr + ((4 * h + 2 * qq + c) * kRows + r) * 16);
            rw[4 * c] = v.x; rw[4 * c + 1] = v.y; rw[4 * c + 2] = v.z; rw[4 * c + 3] = v.w;
        }
    } else if constexpr (BITS == 6 || BITS == 7) {
        const uint4 v = *reinterpret_cast<const uint4*>(sr + ((2 * h + qq) * kRows + r) * 16);
        rw[0] = v.x; rw[1] = v.y; rw[2] = v.z; rw[3] = v.w;
        const uint2 m = *reinterpret_cast<const uint2*>(sr + ((4 + h) * kRows + r) * 16 + 8 * qq);
        mid[0] = m.x; mid[1] = m.y;
        if constexpr (BITS == 7) hi = *reinterpret_cast<const uint32_t*>(sr + (6 * kRows + r) * 16 + 8 * h + 4 * qq);
    }
#pragma unroll
    for (int l = 0; l < 8; ++l) {
        // base: bytes of v hold the codes of columns 4Q .. 4Q+3 (Q = 16h + 8qq + l)
        const uint32_t v = (bw[l >> 2] >> (2 * (l & 3))) & 0x03030303u;
        const uint32_t sel = v * 0x11u + 0x40404040u;
        const uint32_t b01 = prmt(lut_lo, lut_hi, sel);
        const uint32_t b23 = prmt(lut_lo, lut_hi, sel >> 16);
        if constexpr (BITS == 0) {
            out[2 * l] = b01;
            out[2 * l + 1] = b23;
        } else {
            uint32_t u;
            if constexpr (BITS == 8) {
                u = rw[l];
            } else {
                const uint32_t lo = (rw[l >> 1] >> (4 * (l & 1))) & 0x0F0F0F0Fu;
                const int pm = l & 3;
                const uint32_t ms = pm < 2 ? (mid[l >> 2] << (4 - 2 * pm)) : (mid[l >> 2] >> (2 * pm - 4));
                u = lo | (ms & 0x30303030u);
                if constexpr (BITS == 7) {
                    const uint32_t hs = l < 7 ? (hi << (6 - l)) : (hi >> 1);
                    u |= hs & 0x40404040u;
                }
            }
            // 1024 + u as fp16 (exact), minus 1024 + 2^(b-1), gives q exactly
            const __half2 q01 = __hsub2(u32_as_h2(prmt(u, 0x64646464u, 0x5140u)), off2);
            const __half2 q23 = __hsub2(u32_as_h2(prmt(u, 0x64646464u, 0x7362u)), off2);
            out[2 * l] = h2_as_u32(__hfma2(q01, sr2, u32_as_h2(b01)));
            out[2 * l + 1] = h2_as_u32(__hfma2(q23, sr2, u32_as_h2(b23)));
        }
    }
}

__device__ __forceinline__ void tmem_st32_wait(uint32_t taddr, const uint32_t (&v)[32]) {
    tmem_st32(taddr, v);
    tc_wait_st();
}

// Load NP accumulator columns of this thread's lane and wait for them.
template <int NP>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float (&v)[NP]) {
#pragma unroll
    for (int j = 0; j < NP / 16; ++j) {
        float t[16];
        uint32_t r[16];
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {"
                     "%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
                     "tcgen05.wait::ld.sync.aligned;"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                       "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
                       "=r"(r[14]), "=r"(r[15])
                     : "r"(taddr + 16 * j) : "memory");
#pragma unroll
        for (int i = 0; i < 16; ++i) t[i] = __uint_as_float(r[i]);
#pragma unroll
        for (int i = 0; i < 16; ++i) v[16 * j + i] = t[i];
    }
}

__device__ __forceinline__ long long unit_begin(int c, long long units, int grid) {
    return (long long)c * units / grid;
}

// Position in the concatenated unit range of a grouped launch: task k, row tile, group g.
struct UnitCursor {
    int k, tile, g;
    __device__ __forceinline__ void init(const GemmArgs& p, long long u) {
        k = 0;
        while (k + 1 < p.ntasks && p.task[k + 1].ubegin <= u) ++k;
        const long long l = u - p.task[k].ubegin;
        tile = (int)(l / p.task[k].G);
        g = (int)(l - (long long)tile * p.task[k].G);
    }
    __device__ __forceinline__ void next(const GemmArgs& p) {
        if (++g == p.task[k].G) {
            g = 0;
            if (++tile == p.task[k].tiles) { tile = 0; ++k; }
        }
    }
    __device__ __forceinline__ long long local(const GemmArgs& p) const { return (long long)tile * p.task[k].G + g; }
    __device__ __forceinline__ bool group_end(const GemmArgs& p) const { return g == p.task[k].G - 1; }
};

template <int BITS, int NP>
__global__ void __launch_bounds__(Cfg<BITS, NP>::kThreads, Cfg<BITS, NP>::kCtasPerSm)
k_nest_gemm(const __grid_constant__ GemmArgs p) {
    using C = Cfg<BITS, NP>;
    constexpr int S = C::kStages, NA = C::kNumA;
    extern __shared__ __align__(1024) uint8_t smem[];

    uint8_t* xring = smem + S * C::kWStage;
    uint64_t* bars = reinterpret_cast<uint64_t*>(xring + C::kXRing);
    const uint32_t bar0 = smem_u32(bars);
    auto full_w = [&](int s) { return bar0 + 8u * s; };
    auto empty_w = [&](int s) { return bar0 + 8u * (S + s); };
    auto full_x = [&](int a) { return bar0 + 8u * (2 * S + a); };
    auto a_full = [&](int a) { return bar0 + 8u * (2 * S + NA + a); };
    auto done = [&](int a) { return bar0 + 8u * (2 * S + 2 * NA + a); };
    constexpr int ND = C::kNumD;
    auto d_full = [&](int d) { return bar0 + 8u * (2 * S + 3 * NA + d); };
    auto d_empty = [&](int d) { return bar0 + 8u * (2 * S + 3 * NA + ND + d); };
    const uint32_t drain_bar = bar0 + 8u * (2 * S + 3 * NA + 2 * ND);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    auto st_base = [&](int s) { return smem + s * C::kWStage; };
    auto st_res = [&](int s) { return smem + s * C::kWStage + C::kBaseBytes; };
    auto st_x = [&](int a) { return xring + a * C::kXBytes; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) { mbar_init(full_w(s), 1); mbar_init(empty_w(s), C::kUnitWG * kRows); }
        for (int a = 0; a < NA; ++a) {
            mbar_init(full_x(a), 1);
            mbar_init(a_full(a), C::kUnitWG * kRows);
            mbar_init(done(a), 1);
        }
        for (int d = 0; d < ND; ++d) { mbar_init(d_full(d), 1); mbar_init(d_empty(d), C::kEpiWG * kRows); }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == C::kMmaWarp) {
        tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    grid_dep_launch_dependents();

    // this CTA's contiguous range of units (tasks, row tiles, groups concatenated)
    const long long units = p.units;
    const int grid = gridDim.x;
    const long long u0 = unit_begin(blockIdx.x, units, grid);
    const int n = (int)(unit_begin(blockIdx.x + 1, units, grid) - u0);
    UnitCursor start;
    start.init(p, u0);

    if (warp == C::kProducerWarp) {
        UnitCursor cw = start;               // next unit whose weights are fetched
        auto issue_w = [&](int i) {
            const int s = i % S;
            const GemmTask& t = p.task[cw.k];
            const long long lu = cw.local(p);
            mbar_arrive_expect_tx(full_w(s), C::kWStage);
            bulk_g2s(smem_u32(st_base(s)), t.base + lu * C::kBaseBytes, C::kBaseBytes, full_w(s));
            if constexpr (C::kResUnit != 0)
                bulk_g2s(smem_u32(st_res(s)), t.resid + lu * C::kResUnit, C::kResUnit, full_w(s));
            cw.next(p);
        };
        // weights do not depend on the previous kernel: fill the weight ring now
        const int pre = n < S ? n : S;
        for (int i = 0; i < pre; ++i) {
            if (lane == 0) issue_w(i);
            else cw.next(p);
        }
        __syncwarp();
        grid_dep_wait();                     // the activation operand comes from the previous kernel
        // Two independent rings: activation block of unit ix goes to slot ix % NA once unit
        // ix - NA's MMAs are done; weights of unit iw go to stage iw % S once unit iw - S has
        // been decoded.  Poll both so neither waits behind the other.
        int iw = pre, ix = 0;
        UnitCursor cx = start;               // next unit whose activation block is fetched
        uint64_t t_last = globaltimer();
        while (ix < n || iw < n) {
            bool moved = false;
            if (ix < n) {
                bool ready = ix < NA;
                if (!ready && lane == 0) ready = mbar_test_wait(done(ix % NA), ((ix / NA) - 1) & 1);
                if (__shfl_sync(0xffffffffu, ready, 0)) {
                    if (lane == 0) {
                        const int a = ix % NA;
                        mbar_arrive_expect_tx(full_x(a), C::kXBytes);
                        bulk_g2s(smem_u32(st_x(a)), p.task[cx.k].xop + (size_t)cx.g * (C::kXBytes / 2), C::kXBytes,
                                 full_x(a));
                    }
                    cx.next(p);
                    ++ix;
                    moved = true;
                }
            }
            if (iw < n) {
                bool ready = false;
                if (lane == 0) ready = mbar_test_wait(empty_w(iw % S), ((iw / S) - 1) & 1);
                if (__shfl_sync(0xffffffffu, ready, 0)) {
                    if (lane == 0) issue_w(iw);
                    else cw.next(p);
                    ++iw;
                    moved = true;
                }
            }
            if (moved) {
                t_last = globaltimer();
            } else {
                __nanosleep(64);           // nothing to issue yet: back off the barrier words
                const bool stop = (*abort_flag != 0) || (globaltimer() - t_last > kWaitLimitNs);
                if (__shfl_sync(0xffffffffu, stop, 0)) {
                    if (lane == 0 && *abort_flag == 0) { *abort_flag = 1; atomicExch(&g_nest_error, 1); }
                    break;
                }
            }
        }
        __syncwarp();
        // every issued copy has landed before the CTA may leave
        for (int j = iw > S ? iw - S : 0; j < iw; ++j) warp_wait(full_w(j % S), (j / S) & 1, abort_flag, false);
        for (int j = ix > NA ? ix - NA : 0; j < ix; ++j) warp_wait(full_x(j % NA), (j / NA) & 1, abort_flag, false);
    } else if (warp == C::kMmaWarp) {
        constexpr uint32_t idesc = idesc_f16_f32(128, NP);
        // B descriptor of activation slot 0, k-step 0; slot a adds a * kXBytes, k-step kk adds kk * NP * 32 bytes
        const uint64_t bdesc0 = smem_desc_noswizzle(smem_u32(xring), (NP / 8) * 128, 128);
        int seg = -1;
        UnitCursor cu = start;
        bool issued_any = false;
        for (int i = 0; i < n; ++i) {
            const bool first = (i == 0) || cu.g == 0;
            const bool last = (i == n - 1) || cu.group_end(p);
            if (first) {
                ++seg;
                if (seg >= ND && !warp_wait(d_empty(seg % ND), ((seg / ND) - 1) & 1, abort_flag)) break;
            }
            const int a = i % NA, d = seg % ND;
            // a_full also covers the activation block: its warpgroup waited for full_x before arriving
            if (!warp_wait(a_full(a), (i / NA) & 1, abort_flag)) break;
            tc_fence_after();
            if (lane == 0) {
                const uint64_t bd = bdesc0 + (uint64_t)((a * C::kXBytes) >> 4);
                const uint32_t ta = tmem + C::kColA + 64 * a, td = tmem + d * NP;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_f16_ts(td, ta + 8 * kk, bd + (uint64_t)(kk * NP * 2), idesc, (first && kk == 0) ? 0u : 1u);
                tc_commit(done(a));
                if (last) tc_commit(d_full(d));
            }
            __syncwarp();
            issued_any = true;
            cu.next(p);
        }
        if (issued_any) {              // all MMAs finished before tensor memory is released
            if (lane == 0) tc_commit(drain_bar);
            __syncwarp();
            warp_wait(drain_bar, 0, abort_flag, false);
        }
    } else {
        // dequantisation warpgroups; they (warpgroup 0 alone below 128 tokens) also run the epilogues
        const int wg = warp >> 2;
        const int r = 32 * (warp & 3) + lane;               // row of the tile == TMEM lane
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        // magic-number offsets: 1024 + the stored offset of the codes
        const __half2 off2 = __float2half2_rn(
            1024.0f + (BITS == 48 ? 136.0f : BITS == 40 ? 8.0f : (BITS ? (float)(1 << (BITS - 1)) : 0.0f)));
        constexpr float kOutScale = BITS == 48 ? 0.0625f : 1.0f;     // s_ref = s4 / 16
        int seg = -1;
        UnitCursor cu = start;
        bool dep_done = false;
        for (int i = 0; i < n; ++i) {
            const bool first = (i == 0) || cu.g == 0;
            const bool last = (i == n - 1) || cu.group_end(p);
            if (first) ++seg;
            if (i % (C::kDeqWG / C::kUnitWG) == wg / C::kUnitWG) {
                const int s = i % S, a = i % NA;
                // Order matters when S is odd: stage s then alternates between the two
                // warpgroups, and a parity wait cannot tell phase k+1 from phase k-1.  The
                // wait on done(a) for unit i-NA comes first: its MMAs were issued after
                // the a_full of unit i-S (S >= NA), so every thread that consumed unit i-S
                // has already seen full_w(s) complete, and the phase this wait tests is the
                // next one.  Unit i+1's copy can land before unit i's, so without this the
                // warpgroup of unit i+S could read a stage that is still being filled.
                if (i >= NA && !warp_wait(done(a), ((i / NA) - 1) & 1, abort_flag)) break;
                if (!warp_wait(full_w(s), (i / S) & 1, abort_flag)) break;
                tc_fence_after();
                const uint8_t* sb = st_base(s);
                const uint8_t* sr = st_res(s);
                constexpr int kHalves = 2 / C::kUnitWG;          // the 64-column halves this warpgroup decodes
                const int h_first = (wg % C::kUnitWG) * kHalves;
                if constexpr (is_w4(BITS)) {
                    const __half2 s2 = __half2half2(*reinterpret_cast<const __half*>(sb + 8192 + 2 * r));
#pragma unroll
                    for (int j = 0; j < kHalves; ++j) {
                        const int hh = h_first + j;
                        uint32_t w[32];
                        dequant_half_w4<BITS>(sb, sr, r, hh, s2, off2, w);
                        tmem_st32_wait(tmem + lane_base + C::kColA + 64 * a + 32 * hh, w);
                    }
                } else {
                    const float s_b = __half2float(*reinterpret_cast<const __half*>(sb + 4096 + 2 * r));
                    // scaled levels as fp16, low bytes in lut_lo and high bytes in lut_hi
                    uint32_t h[4];
#pragma unroll
                    for (int c = 0; c < 4; ++c) h[c] = __half_as_ushort(__float2half_rn(s_b * level_f(c)));
                    const uint32_t lut_lo = (h[0] & 0xFFu) | ((h[1] & 0xFFu) << 8) | ((h[2] & 0xFFu) << 16) | ((h[3] & 0xFFu) << 24);
                    const uint32_t lut_hi = (h[0] >> 8) | ((h[1] >> 8) << 8) | ((h[2] >> 8) << 16) | ((h[3] >> 8) << 24);
                    __half2 sr2 = __float2half2_rn(0.0f);
                    if constexpr (BITS != 0)
                        sr2 = __half2half2(*reinterpret_cast<const __half*>(sr + 2048 * BITS + 2 * r));
#pragma unroll
                    for (int j = 0; j < kHalves; ++j) {
                        const int hh = h_first + j;
#pragma unroll
                        for (int qq = 0; qq < 2; ++qq) {
                            uint32_t w[16];
                            dequant_quarter<BITS>(sb, sr, r, hh, qq, lut_lo, lut_hi, sr2, off2, w);
                            tmem_st16(tmem + lane_base + C::kColA + 64 * a + 32 * hh + 16 * qq, w);
                        }
                        tc_wait_st();
                    }
                }
                mbar_arrive(empty_w(s));             // this thread is done with the weight stage
                tc_fence_before();
                // the MMA issuer waits on a_full alone, so a_full must also imply the activation block
                if (!warp_wait(full_x(a), (i / NA) & 1, abort_flag)) break;
                mbar_arrive(a_full(a));
            }
            if (wg < C::kEpiWG && last) {
                const int d = seg % ND;
                if (!warp_wait(d_full(d), (seg / ND) & 1, abort_flag)) break;
                tc_fence_after();
                const GemmTask& task = p.task[cu.k];
                const int m = cu.tile * kRows + r;
                const int T = p.T, M = task.M;
                float* zp = task.z + m;
                if constexpr (NP <= 64) {
                    float v[NP];
                    tmem_ld_cols<NP>(tmem + lane_base + d * NP, v);
                    tc_fence_before();
                    mbar_arrive(d_empty(d));
                    if (!dep_done) { grid_dep_wait(); dep_done = true; }
                    if (m < M) {
#pragma unroll
                        for (int t = 0; t < NP; ++t)
                            if (t < T) atomicAdd(zp + (size_t)t * M, v[t] * kOutScale);   // fire-and-forget reduction
                    }
                } else {
                    // warpgroup wg takes its kEpiCols accumulator columns, 32 at a time; it
                    // releases the buffer after its last load
                    constexpr int kEpiCols = NP / C::kEpiWG;
                    if (!dep_done) { grid_dep_wait(); dep_done = true; }
                    for (int c0 = wg * kEpiCols; c0 < (wg + 1) * kEpiCols; c0 += 32) {
                        float v[32];
                        tmem_ld_cols<32>(tmem + lane_base + d * NP + c0, v);
                        if (c0 + 32 == (wg + 1) * kEpiCols) {
                            tc_fence_before();
                            mbar_arrive(d_empty(d));
                        }
                        if (m < M) {
#pragma unroll
                            for (int t = 0; t < 32; ++t)
                                if (c0 + t < T) atomicAdd(zp + (size_t)(c0 + t) * M, v[t] * kOutScale);
                        }
                    }
                }
            }
            cu.next(p);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == C::kMmaWarp) tmem_dealloc(tmem, C::kTmemCols);
}

// ---------------------------------------------------------------------------
// Register-fragment GEMM for few tokens (T <= 8 * NT): mma.sync m16n8k16.
//
// With N = 8..16 tokens a tcgen05.mma of 128 x N x 16 costs a fixed issue time
// that does not shrink with N, and one thread issues all of a CTA's MMAs.  Here
// every warp decodes its weights straight into mma.sync A fragments (no tensor
// memory, no MMA thread, no hand-off), so the weight rate is set by the decode
// ALU work and the memory pipe.
//
// K order inside a fragment.  mma.sync sums over its 16 k indices in any order,
// so the k index a thread's fragment slot stands for may be any column, as long
// as the B fragment uses the same one.  Thread (g, q) of a warp (g = lane / 4,
// q = lane % 4) takes, in k-step s of half h, the four columns 4Q .. 4Q+3 with
// Q = 16h + 4q + s.  In the packed unit those are exactly the four codes that
// word q of the row's half-h base vector holds at bit offset 2s, and residual
// word Q - 16h; the B fragment is x'[token][4Q .. 4Q+3], eight contiguous bytes
// of the operand.  So the kernel reads the same packed layout and operand as
// the tcgen05 kernel, each byte once.
//
// Scales are applied in fp32 per (row, group): the base fragment holds the
// unscaled fp16 levels, the residual fragment the integer codes q (exact in
// fp16), each summed into its own fp32 accumulator by the MMA, then
//   z += s_b * sum(L[c] x') + s_r * sum(q x').
//
// Copies.  A 1-D bulk copy costs a CTA about the same time whether it moves 2 KB
// or 8 KB, so a copy of one 4 KB unit caps a CTA far below its share of HBM
// bandwidth.  A stage therefore holds up to KU consecutive units of one row tile
// (contiguous in the packed buffers and, group after group, in the operand), each
// part fetched by one copy.  With T <= 8 the activation is not staged at all:
// the B fragments are read from global memory, the next unit's while the current
// one is decoded, so the only copies are the weights'.
//
// Pipeline: one producer warp fills a ring of S stages.  Two teams of four warps
// take alternate units of each stage; every compute warp waits for every stage in
// order and releases it, so each barrier phase is waited in order by the same
// warps.  Warp w of a team owns rows 32w .. 32w+31 of a unit (two 16-row slabs);
// partial sums of a row tile are added into z with fp32 reductions when the
// team's next unit starts another tile.
// ---------------------------------------------------------------------------

template <int BITS, int NT>
struct RfCfg {
    static constexpr int kCtasPerSm = NT >= 4 ? 1 : 2;       // 32 tokens need the registers of a whole SM
    static constexpr int kNB = NT < 2 ? 2 : NT;              // operand token blocks (n_pad / 8)
    static constexpr bool kStageX = NT >= 2;                 // T <= 8 reads its B fragments from global memory
    static constexpr int kXBytes = kStageX ? 2048 * kNB : 0; // one group of the operand
    static constexpr int kBaseBytes = base_unit_bytes(BITS);
    static constexpr int kResUnit = second_unit_bytes(BITS);
    static constexpr int kUnit = kBaseBytes + kResUnit + kXBytes;
    static constexpr int kSmemBudget = kCtasPerSm == 1 ? 220 * 1024 : 110 * 1024;
    static constexpr int kAvail = kSmemBudget - 512;
    static constexpr int kKURaw = kAvail / (4 * kUnit);      // room for two stages per team
    static constexpr int kKU = kKURaw > 4 ? 4 : (kKURaw < 1 ? 1 : kKURaw);   // units per stage
    static constexpr int kStageBytes = kKU * kUnit;
    static constexpr int kStagesRaw = kAvail / kStageBytes;
    static constexpr int kStages = (kStagesRaw > 8 ? 8 : kStagesRaw) & ~1;   // even: a stage keeps its team
    static constexpr int kResOff = kKU * kBaseBytes;         // parts of a stage: bases, residuals, operand
    static constexpr int kXOff = kResOff + kKU * kResUnit;
    static constexpr int kTeams = 2;
    static constexpr int kWarpsPerTeam = 4;
    static constexpr int kComputeWarps = kTeams * kWarpsPerTeam;
    static constexpr int kProducerWarp = kComputeWarps;
    static constexpr int kThreads = 32 * (kComputeWarps + 1);
    static constexpr int kSmemBytes = kStages * kStageBytes + 2 * kStages * 8 + 16;
    static_assert(kStages >= 2 * kTeams, "stage too large");
    static_assert(kStageBytes % 128 == 0 && kResOff % 16 == 0 && kXOff % 16 == 0, "stage alignment");
    static_assert(kSmemBytes <= kSmemBudget, "shared memory budget");
};

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint4 ld_cg_v4(const void* ptr) {
    uint4 v;
    asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(ptr));
    return v;
}

// Residual words of one row and half for thread q: everything the four k-steps need.
template <int BITS>
struct ResidWords {
    uint32_t w[4];
    __device__ __forceinline__ void load(const uint8_t* sr, int r, int h, int q) {
        if constexpr (BITS == 8) {
            const uint4 v = *reinterpret_cast<const uint4*>(sr + ((4 * h + q) * kRows + r) * 16);
            w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
        } else if constexpr (BITS == 6 || BITS == 7) {
            const uint2 lo = *reinterpret_cast<const uint2*>(sr + ((2 * h + (q >> 1)) * kRows + r) * 16 + 8 * (q & 1));
            w[0] = lo.x;
            w[1] = lo.y;
            w[2] = *reinterpret_cast<const uint32_t*>(sr + ((4 + h) * kRows + r) * 16 + 4 * q);
            w[3] = BITS == 7 ? *reinterpret_cast<const uint32_t*>(sr + (6 * kRows + r) * 16 + 8 * h + 4 * (q >> 1)) : 0u;
        }
    }
    // offset-binary residual codes of columns 4Q .. 4Q+3, Q = 16h + 4q + s, one per byte
    __device__ __forceinline__ uint32_t codes(int s, int q) const {
        if constexpr (BITS == 8) {
            return w[s];
        } else {
            const uint32_t lo = ((s < 2 ? w[0] : w[1]) >> (4 * (s & 1))) & 0x0F0F0F0Fu;
            const uint32_t ms = (s < 2 ? (w[2] << (4 - 2 * s)) : (w[2] >> (2 * s - 4))) & 0x30303030u;
            uint32_t u = lo | ms;
            if constexpr (BITS == 7) {
                const int ph = 4 * (q & 1) + s;
                u |= (ph < 7 ? (w[3] << (6 - ph)) : (w[3] >> 1)) & 0x40404040u;
            }
            return u;
        }
    }
};

// Units in the chunk that starts at cursor c: at most ku, at most `left`, never past the row tile.
__device__ __forceinline__ int chunk_len(const GemmArgs& p, const UnitCursor& c, int left, int ku) {
    const int in_tile = p.task[c.k].G - c.g;
    const int l = left < ku ? left : ku;
    return l < in_tile ? l : in_tile;
}

template <int BITS, int NT>
__global__ void __launch_bounds__(RfCfg<BITS, NT>::kThreads, RfCfg<BITS, NT>::kCtasPerSm)
k_nest_rf(const __grid_constant__ GemmArgs p) {
    using C = RfCfg<BITS, NT>;
    constexpr int S = C::kStages, KU = C::kKU;
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * C::kStageBytes);
    const uint32_t bar0 = smem_u32(bars);
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (S + s); };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * S);
    auto stage = [&](int s) { return smem + s * C::kStageBytes; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) { mbar_init(full(s), 1); mbar_init(empty(s), C::kWarpsPerTeam); }
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    grid_dep_launch_dependents();

    const long long units = p.units;
    const int grid = gridDim.x;
    const long long u0 = unit_begin(blockIdx.x, units, grid);
    const int n = (int)(unit_begin(blockIdx.x + 1, units, grid) - u0);
    UnitCursor start;
    start.init(p, u0);

    if (warp == C::kProducerWarp) {
        // chunk j holds units [i, i + kc) of this CTA, starting at cursor c
        auto issue_w = [&](int j, const UnitCursor& c, int kc) {
            const int s = j % S;
            const GemmTask& t = p.task[c.k];
            const long long lu = c.local(p);
            mbar_arrive_expect_tx(full(s), kc * C::kUnit);
            bulk_g2s(smem_u32(stage(s)), t.base + lu * C::kBaseBytes, kc * C::kBaseBytes, full(s));
            if constexpr (C::kResUnit != 0)
                bulk_g2s(smem_u32(stage(s) + C::kResOff), t.resid + lu * C::kResUnit, kc * C::kResUnit, full(s));
        };
        auto issue_x = [&](int j, const UnitCursor& c, int kc) {
            if constexpr (C::kStageX)
                bulk_g2s(smem_u32(stage(j % S) + C::kXOff), p.task[c.k].xop + (size_t)c.g * (C::kXBytes / 2),
                         kc * C::kXBytes, full(j % S));
        };
        UnitCursor cw = start;
        int i = 0, j = 0;
        while (j < S && i < n) {             // weights do not depend on the previous kernel: start them now
            const int kc = chunk_len(p, cw, n - i, KU);
            if (lane == 0) issue_w(j, cw, kc);
            for (int u = 0; u < kc; ++u) cw.next(p);
            i += kc;
            ++j;
        }
        grid_dep_wait();                     // the activation operand comes from the previous kernel
        {
            UnitCursor cx = start;
            int ii = 0;
            for (int jj = 0; jj < j; ++jj) {
                const int kc = chunk_len(p, cx, n - ii, KU);
                if (lane == 0) issue_x(jj, cx, kc);
                for (int u = 0; u < kc; ++u) cx.next(p);
                ii += kc;
            }
        }
        uint64_t t_last = globaltimer();
        while (i < n) {
            bool ready = false;
            if (lane == 0) ready = mbar_test_wait(empty(j % S), ((j / S) - 1) & 1);
            if (__shfl_sync(0xffffffffu, ready, 0)) {
                const int kc = chunk_len(p, cw, n - i, KU);
                if (lane == 0) { issue_w(j, cw, kc); issue_x(j, cw, kc); }
                for (int u = 0; u < kc; ++u) cw.next(p);
                i += kc;
                ++j;
                t_last = globaltimer();
            } else {
                __nanosleep(64);
                const bool stop = (*abort_flag != 0) || (globaltimer() - t_last > kWaitLimitNs);
                if (__shfl_sync(0xffffffffu, stop, 0)) {
                    if (lane == 0 && *abort_flag == 0) { *abort_flag = 1; atomicExch(&g_nest_error, 1); }
                    break;
                }
            }
        }
        __syncwarp();
        // every issued copy has landed before the CTA may leave
        for (int jj = j > S ? j - S : 0; jj < j; ++jj) warp_wait(full(jj % S), (jj / S) & 1, abort_flag, false);
        return;
    }

    const int team = warp / C::kWarpsPerTeam, wq = warp % C::kWarpsPerTeam;
    const int g = lane >> 2, q = lane & 3;
    const int T = p.T;
    uint32_t lut_lo, lut_hi;                  // unscaled fp16 levels: low bytes, high bytes
    {
        uint32_t hv[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) hv[c] = __half_as_ushort(__float2half_rn(level_f(c)));
        lut_lo = (hv[0] & 0xFFu) | ((hv[1] & 0xFFu) << 8) | ((hv[2] & 0xFFu) << 16) | ((hv[3] & 0xFFu) << 24);
        lut_hi = (hv[0] >> 8) | ((hv[1] >> 8) << 8) | ((hv[2] >> 8) << 16) | ((hv[3] >> 8) << 24);
    }
    const __half2 off2 = __float2half2_rn(1024.0f + ((BITS && !is_w4(BITS)) ? (float)(1 << (BITS - 1)) : 0.0f));
    const __half2 off4 = __float2half2_rn(1024.0f + 8.0f);   // W4: 1024 + the nibble offset
    float zacc[2][NT][4];
#pragma unroll
    for (int sl = 0; sl < 2; ++sl)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) zacc[sl][nt][e] = 0.0f;

    grid_dep_wait();                          // the operand and z come from / are cleared by the previous kernel

    // T <= 8: B fragments x'[g][4Q .. 4Q+7] (token block 0) straight from global memory
    auto load_bx = [&](const uint16_t* xop, int grp, uint4 (&dst)[2][2]) {
        const uint8_t* xg = reinterpret_cast<const uint8_t*>(xop) + (size_t)grp * 4096;
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int pp = 0; pp < 2; ++pp)
                dst[h][pp] = g < T ? ld_cg_v4(xg + ((8 * h + 2 * q + pp) * 16 + g) * 16) : make_uint4(0u, 0u, 0u, 0u);
    };
    auto advance = [&](UnitCursor& c, int m) {
        for (int u = 0; u < m; ++u) c.next(p);
    };
    uint4 bxg[2][2];

    // Chunks go to the teams in turn (chunk j -> team j % 2); S is even, so a stage always
    // belongs to the same team.  cj / i: cursor and unit index of chunk j's first unit.
    UnitCursor cj = start;
    int i = 0, j = 0;
    if constexpr (!C::kStageX) {
        UnitCursor c0 = start;
        if (team == 1 && n > 0) advance(c0, chunk_len(p, start, n, KU));
        if (team == 0 ? n > 0 : chunk_len(p, start, n, KU) < n) load_bx(p.task[c0.k].xop, c0.g, bxg);
    }
    while (i < n) {
        const int kc = chunk_len(p, cj, n - i, KU);
        UnitCursor c1 = cj;
        advance(c1, kc);
        const int i1 = i + kc;
        if ((j % C::kTeams) == team) {
            const int s_ = j % S;
            if (!warp_wait(full(s_), (j / S) & 1, abort_flag)) break;
            // the team's next chunk, j + 2: where its partial sums go, and its first operand block
            const int kc1 = i1 < n ? chunk_len(p, c1, n - i1, KU) : 0;
            UnitCursor c2 = c1;
            advance(c2, kc1);
            const bool has_next = i1 + kc1 < n;
            const bool flush = !has_next || c2.k != cj.k || c2.tile != cj.tile;
            const GemmTask& task = p.task[cj.k];
            for (int u = 0; u < kc; ++u) {
                uint4 bxn[2][2];
                if constexpr (!C::kStageX) {
                    if (u + 1 < kc) load_bx(task.xop, cj.g + u + 1, bxn);
                    else if (has_next) load_bx(p.task[c2.k].xop, c2.g, bxn);
                }
                const uint8_t* sb = stage(s_) + u * C::kBaseBytes;
                const uint8_t* sr = stage(s_) + C::kResOff + u * C::kResUnit;
                const uint8_t* sx = stage(s_) + C::kXOff + u * C::kXBytes;
#pragma unroll
                for (int sl = 0; sl < 2; ++sl) {
                    const int r0 = 32 * wq + 16 * sl + g, r1 = r0 + 8;
                    // 2-bit base: one word per row and half (codes of columns 4Q.., Q = 16h + 4q + s,
                    // in bits 2s of each byte).  W4: the row's nibble words 8h + 2q and 8h + 2q + 1
                    // (column 8w + 4k + j in bits 8j + 4k of word w).
                    uint32_t bw0[2][2], bw1[2][2];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        if constexpr (is_w4(BITS)) {
                            const uint2 v0 = *reinterpret_cast<const uint2*>(sb + ((2 * h + (q >> 1)) * kRows + r0) * 16 + 8 * (q & 1));
                            const uint2 v1 = *reinterpret_cast<const uint2*>(sb + ((2 * h + (q >> 1)) * kRows + r1) * 16 + 8 * (q & 1));
                            bw0[h][0] = v0.x; bw0[h][1] = v0.y; bw1[h][0] = v1.x; bw1[h][1] = v1.y;
                        } else {
                            bw0[h][0] = *reinterpret_cast<const uint32_t*>(sb + (h * kRows + r0) * 16 + 4 * q);
                            bw1[h][0] = *reinterpret_cast<const uint32_t*>(sb + (h * kRows + r1) * 16 + 4 * q);
                        }
                    }
                    constexpr int kScaleOff = is_w4(BITS) ? 8192 : 4096;   // s4 (W4) or s_b
                    const float sb0 = __half2float(*reinterpret_cast<const __half*>(sb + kScaleOff + 2 * r0));
                    const float sb1 = __half2float(*reinterpret_cast<const __half*>(sb + kScaleOff + 2 * r1));
                    float sr0 = 0.0f, sr1 = 0.0f;
                    if constexpr (C::kResUnit != 0) {
                        sr0 = __half2float(*reinterpret_cast<const __half*>(sr + 2048 * BITS + 2 * r0));
                        sr1 = __half2float(*reinterpret_cast<const __half*>(sr + 2048 * BITS + 2 * r1));
                    }
                    float db[NT][4], dr[NT][4];
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) { db[nt][e] = 0.0f; dr[nt][e] = 0.0f; }
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        ResidWords<is_w4(BITS) ? 0 : BITS> rw0, rw1;
                        if constexpr (C::kResUnit != 0) { rw0.load(sr, r0, h, q); rw1.load(sr, r1, h, q); }
#pragma unroll
                        for (int pp = 0; pp < 2; ++pp) {
                            // B fragments of k-steps 2pp and 2pp+1: x'[8nt + g][4Q .. 4Q+7], Q = 16h + 4q + 2pp
                            uint4 bx[NT];
                            if constexpr (C::kStageX) {
#pragma unroll
                                for (int nt = 0; nt < NT; ++nt)
                                    bx[nt] = *reinterpret_cast<const uint4*>(
                                        sx + (((8 * h + 2 * q + pp) * C::kNB + nt) * 8 + g) * 16);
                            } else {
                                bx[0] = bxg[h][pp];
                            }
#pragma unroll
                            for (int s2 = 0; s2 < 2; ++s2) {
                                const int s = 2 * pp + s2;
                                uint32_t a0, a1, a2, a3;
                                if constexpr (is_w4(BITS)) {
                                    // u4 = q4 + 8 of columns 4Q .. 4Q+3, one per byte, as fp16 q4
                                    const uint32_t b0 = (bw0[h][s >> 1] >> (4 * (s & 1))) & 0x0F0F0F0Fu;
                                    const uint32_t b1 = (bw1[h][s >> 1] >> (4 * (s & 1))) & 0x0F0F0F0Fu;
                                    a0 = h2_as_u32(__hsub2(u32_as_h2(prmt(b0, 0x64646464u, 0x5140u)), off4));
                                    a2 = h2_as_u32(__hsub2(u32_as_h2(prmt(b0, 0x64646464u, 0x7362u)), off4));
                                    a1 = h2_as_u32(__hsub2(u32_as_h2(prmt(b1, 0x64646464u, 0x5140u)), off4));
                                    a3 = h2_as_u32(__hsub2(u32_as_h2(prmt(b1, 0x64646464u, 0x7362u)), off4));
                                } else {
                                    const uint32_t v0 = (bw0[h][0] >> (2 * s)) & 0x03030303u;
                                    const uint32_t v1 = (bw1[h][0] >> (2 * s)) & 0x03030303u;
                                    const uint32_t sel0 = v0 * 0x11u + 0x40404040u, sel1 = v1 * 0x11u + 0x40404040u;
                                    a0 = prmt(lut_lo, lut_hi, sel0);
                                    a2 = prmt(lut_lo, lut_hi, sel0 >> 16);
                                    a1 = prmt(lut_lo, lut_hi, sel1);
                                    a3 = prmt(lut_lo, lut_hi, sel1 >> 16);
                                }
#pragma unroll
                                for (int nt = 0; nt < NT; ++nt)
                                    mma16816(db[nt], a0, a1, a2, a3, s2 ? bx[nt].z : bx[nt].x, s2 ? bx[nt].w : bx[nt].y);
                                if constexpr (C::kResUnit != 0) {
                                    const uint32_t u0 = rw0.codes(s, q), u1 = rw1.codes(s, q);
                                    const uint32_t q0 = h2_as_u32(__hsub2(u32_as_h2(prmt(u0, 0x64646464u, 0x5140u)), off2));
                                    const uint32_t q2 = h2_as_u32(__hsub2(u32_as_h2(prmt(u0, 0x64646464u, 0x7362u)), off2));
                                    const uint32_t q1 = h2_as_u32(__hsub2(u32_as_h2(prmt(u1, 0x64646464u, 0x5140u)), off2));
                                    const uint32_t q3 = h2_as_u32(__hsub2(u32_as_h2(prmt(u1, 0x64646464u, 0x7362u)), off2));
#pragma unroll
                                    for (int nt = 0; nt < NT; ++nt)
                                        mma16816(dr[nt], q0, q1, q2, q3, s2 ? bx[nt].z : bx[nt].x, s2 ? bx[nt].w : bx[nt].y);
                                }
                            }
                        }
                    }
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        zacc[sl][nt][0] += sb0 * db[nt][0] + sr0 * dr[nt][0];
                        zacc[sl][nt][1] += sb0 * db[nt][1] + sr0 * dr[nt][1];
                        zacc[sl][nt][2] += sb1 * db[nt][2] + sr1 * dr[nt][2];
                        zacc[sl][nt][3] += sb1 * db[nt][3] + sr1 * dr[nt][3];
                    }
                }
                if constexpr (!C::kStageX) {
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int pp = 0; pp < 2; ++pp) bxg[h][pp] = bxn[h][pp];
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty(s_));     // this warp is done with the stage
            if (flush) {
                const int M = task.M;
#pragma unroll
                for (int sl = 0; sl < 2; ++sl) {
                    const int m0 = cj.tile * kRows + 32 * wq + 16 * sl + g, m1 = m0 + 8;
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        const int t0 = 8 * nt + 2 * q, t1 = t0 + 1;
                        if (m0 < M) {
                            if (t0 < T) atomicAdd(task.z + (size_t)t0 * M + m0, zacc[sl][nt][0]);
                            if (t1 < T) atomicAdd(task.z + (size_t)t1 * M + m0, zacc[sl][nt][1]);
                        }
                        if (m1 < M) {
                            if (t0 < T) atomicAdd(task.z + (size_t)t0 * M + m1, zacc[sl][nt][2]);
                            if (t1 < T) atomicAdd(task.z + (size_t)t1 * M + m1, zacc[sl][nt][3]);
                        }
#pragma unroll
                        for (int e = 0; e < 4; ++e) zacc[sl][nt][e] = 0.0f;
                    }
                }
            }
        }
        cj = c1;
        i = i1;
        ++j;
    }
}

template <int BITS, int NT>
cudaError_t launch_rf(const GemmArgs& a, int grid, cudaStream_t stream) {
    using C = RfCfg<BITS, NT>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(k_nest_rf<BITS, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::kSmemBytes);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    return launch_pdl(k_nest_rf<BITS, NT>, dim3(grid), dim3(C::kThreads), C::kSmemBytes, stream, a);
}

template <int BITS, int NP>
cudaError_t launch_t(const GemmArgs& a, int grid, cudaStream_t stream) {
    using C = Cfg<BITS, NP>;
    static bool configured = false;       // the attribute is per function; set it on first use
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(k_nest_gemm<BITS, NP>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    return launch_pdl(k_nest_gemm<BITS, NP>, dim3(grid), dim3(C::kThreads), C::kSmemBytes, stream, a);
}

// Kernel choice, from measurements on GB300 (a 128 x N x 16 tcgen05.mma costs a
// fixed ~50 cycles to issue whatever N is; mma.sync m16n8k16 runs ~0.47 per cycle
// per SM): the 2-bit draft at one token on the table look-up kernel; the drafts
// (2-bit base or W4 alone) at T <= 8 otherwise on the register-fragment kernel,
// where the decode and not the MMA issue bounds them; everything else on tcgen05,
// which is faster for the verify at every T (and the only kernel with the W8
// decode).  NEST_GEMM_PATH=tc or =rf in the environment forces one kernel (rf up to
// 32 tokens, not for W8), for measuring one against the other.
int path_override() {
    const char* e = getenv("NEST_GEMM_PATH");
    return (e && e[0] == 't') ? 1 : (e && e[0] == 'r') ? 2 : 0;
}

template <int BITS>
cudaError_t launch_bits(const GemmArgs& a, int grid, int sms, cudaStream_t stream) {
    if constexpr (BITS == 0) {                // the 2-bit draft at one token: table look-up
        if (a.T == 1 && path_override() == 0) return launch_lut(a, sms, stream);
    }
    if constexpr (BITS != 48) {               // the register-fragment kernel has no W8 decode
        const int ov = path_override();
        const bool rf = ov == 2 ? a.T <= 32 : (ov == 0 && (BITS == 0 || BITS == 40) && a.T <= 8);
        if (rf) {
            if (a.T <= 8) return launch_rf<BITS, 1>(a, grid, stream);
            if (a.T <= 16) return launch_rf<BITS, 2>(a, grid, stream);
            return launch_rf<BITS, 4>(a, grid, stream);
        }
    }
    if (a.T <= 16) return launch_t<BITS, 16>(a, grid, stream);
    if (a.T <= 32) return launch_t<BITS, 32>(a, grid, stream);
    if (a.T <= 64) return launch_t<BITS, 64>(a, grid, stream);
    if (a.T <= 128) return launch_t<BITS, 128>(a, grid, stream);
    return launch_t<BITS, 256>(a, grid, stream);
}

}  // namespace

cudaError_t launch_gemm(const GemmArgs& a, int bits, int grid, int sms, cudaStream_t stream) {
    switch (bits) {
        case 0: return launch_bits<0>(a, grid, sms, stream);
        case 6: return launch_bits<6>(a, grid, sms, stream);
        case 7: return launch_bits<7>(a, grid, sms, stream);
        case 8: return launch_bits<8>(a, grid, sms, stream);
        case 40: return launch_bits<40>(a, grid, sms, stream);
        case 48: return launch_bits<48>(a, grid, sms, stream);
        default: return cudaErrorInvalidValue;
    }
}

int gemm_ctas_per_sm(int T) { return T > 64 ? 1 : kGemmCtasPerSm; }

cudaError_t launch_wait_selftest(cudaStream_t stream) {
    k_wait_selftest<<<1, 32, 0, stream>>>();
    return cudaGetLastError();
}

cudaError_t read_and_clear_error(int* flag, cudaStream_t stream) {
    cudaError_t e = cudaMemcpyFromSymbolAsync(flag, g_nest_error, sizeof(int), 0, cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    if (*flag) {
        const int zero = 0;
        e = cudaMemcpyToSymbolAsync(g_nest_error, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    }
    return e;
}

}  // namespace nest
