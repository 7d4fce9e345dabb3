// The draft GEMV at one token by table look-up (k_nest_lut): z = Q_base x', the draft
// forward of the "2-bit base in VRAM, residual in RAM" post (feedman.me/posts/wZBTJ), POC
// recipe step 4, "the same but without y_r".  See the description below.
#include <cstdlib>
#include <cstring>
#include <utility>

#include "nest_device.cuh"
#include "nest_internal.h"

namespace nest {

__device__ int g_lut_error;    // raised when a bounded wait of this kernel gives up

namespace {

__device__ __forceinline__ long long unit_begin(int c, long long units, int grid) {
    return (long long)c * units / grid;
}

__device__ bool lut_wait(uint32_t bar, uint32_t parity, volatile int* abort, bool honour_abort = true) {
    return warp_wait_flag(bar, parity, abort, &g_lut_error, honour_abort);
}

// ---------------------------------------------------------------------------
// k_nest_lut: the draft GEMV at one token, by table look-up.
//
// At T = 1 the draft is a matrix-vector product whose weights take one of four
// level values per (row, group) scale, so a pair of columns (k0, k1) carries
// only 16 possible weight pairs.  The CTA builds, per pair, the 16 partial
// sums L[c0] x'[k0] + L[c1] x'[k1] in fp32 once, and every row then reads its
// pair's sum with the 4-bit index its packed codes already form: one
// shared-memory load per two weights and one packed two-lane fp32 FMA (with the
// row's scale) per four, no per-weight decode.
// Pairing, from the packed layout: byte b of code word w (w = 0..7) holds at
// bit offsets 2s the codes of columns 16w + 4s + b, so its nibble n (bits
// 4n..4n+3) is the pair (8C + b, 8C + b + 4) with C = 2w + n, index
// c0 + 4 c1.  Both columns sit in chunk C of the activation operand (token 0:
// 8 fp16 values at byte 256 C of the group's block).  Table (C, b) holds the
// pair's 16 sums at byte 64 (4C + b) of a table buffer.  All 32 lanes of a
// warp (32 rows) read one pair's 64-byte table at a time: 16 words in 16
// banks, no bank conflicts.
//
// Work: super-units of (block of kTiles row tiles, group) -- 2 tiles = 256 rows
// in the default shape -- in task / row-block / group order, split into equal
// contiguous ranges over the resident CTAs (four per SM by default).  Warp roles:
//   producer : bulk copies of the block's base units into a ring of stages (the
//              weights do not depend on the previous kernel, so the first
//              stages are requested before it has finished);
//   table    : reads the group's 128 activations of token 0 itself (plain
//              loads, one super-unit ahead) and builds super-unit j's 1024
//              sums into table buffer j % 4, up to four super-units ahead of
//              the row warps and independent of the stage ring;
//   row warps: R rows per lane (2 by default); each row's 64 look-ups, times its
//              (row, group) scale, go into eight register partial sums that are
//              added into z when the CTA's range leaves the row block.
// Each row warp waits only for its stage and its table, so the row warps run
// independently of each other.  All waits are bounded.
// ---------------------------------------------------------------------------

// Shape of the look-up kernel: WARPS row warps, R rows per lane, CPS resident CTAs per SM;
// a super-unit covers WARPS * 32 * R rows = kTiles row tiles.
template <int WARPS, int R, int CPS = 1>
struct LutCfg {
    static constexpr int kCtasPerSm = CPS;
    static constexpr int kTiles = WARPS * 32 * R / kRows;
    static constexpr int kStage = kTiles * kBaseUnit;     // the block's base units of one group
    static constexpr int kTable = 64 * 16 * 4;            // 64 pairs x 16 sums x fp32
    static constexpr int kTables = 4;                     // table buffers
    static constexpr int kSmemBudget = CPS == 1 ? 227 * 1024 : (CPS == 2 ? 110 * 1024 : 54 * 1024);
    static constexpr int kStagesRaw = (kSmemBudget - kTables * kTable - 512) / kStage;
    static constexpr int kStages = kStagesRaw > 8 ? 8 : kStagesRaw;
    static constexpr int kProducer = WARPS;
    static constexpr int kTableWarp = WARPS + 1;
    static constexpr int kThreads = 32 * (WARPS + 2);
    // stages, tables, barriers: full[S], empty[S], tfull[NT], tempty[NT], abort flag
    static constexpr int kSmem = kStages * kStage + kTables * kTable + (2 * kStages + 2 * kTables) * 8 + 16;
    static_assert(WARPS % (kRows / 32) == 0 && kStages >= 4, "look-up GEMV shape");
    static_assert(kStage % 16 == 0 && (kStages * kStage) % 256 == 0 && kTable % 256 == 0 && kSmem <= 227 * 1024,
                  "look-up GEMV shared memory (table buffers 256-byte aligned)");
};

// Position in the super-unit range of a grouped launch: task k, row block rb, group g.
template <int TILES>
struct LutCursor {
    int k, rb, g;
    __device__ __forceinline__ static int blocks(const GemmTask& t) { return (t.tiles + TILES - 1) / TILES; }
    __device__ __forceinline__ void init(const GemmArgs& p, long long u) {
        k = 0;
        long long base = 0;
        while (k + 1 < p.ntasks && base + (long long)blocks(p.task[k]) * p.task[k].G <= u) {
            base += (long long)blocks(p.task[k]) * p.task[k].G;
            ++k;
        }
        const long long l = u - base;
        rb = (int)(l / p.task[k].G);
        g = (int)(l - (long long)rb * p.task[k].G);
    }
    __device__ __forceinline__ void next(const GemmArgs& p) {
        if (++g == p.task[k].G) {
            g = 0;
            if (++rb == blocks(p.task[k])) { rb = 0; ++k; }
        }
    }
};

// One look-up: byte J of x holds a pair index times 4 (bits 2..5, the rest zero); a byte
// permute puts it under the upper three bytes of the 256-byte aligned table base, and the
// sum is read at byte offset OFF (the pair's table).
template <int J, int OFF>
__device__ __forceinline__ float lut_load(uint32_t x, uint32_t tbase) {
    float v;
    asm volatile("{\n\t.reg .b32 t;\n\tprmt.b32 t, %1, %2, %3;\n\tld.shared.f32 %0, [t+%4];\n\t}"
                 : "=f"(v) : "r"(x), "r"(tbase), "n"(0x7650 | J), "n"(OFF));
    return v;
}

// The eight look-ups of code word W: the low nibbles of its four bytes (pairs C = 2W, b = J)
// and the high nibbles (C = 2W + 1), each moved to bits 2..5 of its byte by one shift and
// one mask for all four bytes.  Byte J's two sums, times the row's scale, add into part[J]
// with one packed two-lane fp32 FMA.
template <int W, int... J>
__device__ __forceinline__ void lut_word(uint32_t w, uint32_t tbase, float2 sc, float2 (&part)[4],
                                         std::integer_sequence<int, J...>) {
    const uint32_t x0 = (w << 2) & 0x3C3C3C3Cu, x1 = (w >> 2) & 0x3C3C3C3Cu;
    const float v0[4] = {lut_load<J, 64 * (4 * (2 * W) + J)>(x0, tbase)...};
    const float v1[4] = {lut_load<J, 64 * (4 * (2 * W + 1) + J)>(x1, tbase)...};
    ((part[J] = __ffma2_rn(make_float2(v0[J], v1[J]), sc, part[J])), ...);
}

// R rows' look-ups, word by word, the rows interleaved.
template <int R, int... W>
__device__ __forceinline__ void lut_rows(const uint32_t (&wd)[R][8], uint32_t tbase, const float2 (&sc)[R],
                                         float2 (&part)[R][4], std::integer_sequence<int, W...>) {
    auto one = [&](auto wc) {
        constexpr int w = decltype(wc)::value;
#pragma unroll
        for (int k = 0; k < R; ++k)
            lut_word<w>(wd[k][w], tbase, sc[k], part[k], std::make_integer_sequence<int, 4>{});
    };
    (one(std::integral_constant<int, W>{}), ...);
}

template <int WARPS, int R, int CPS>
__global__ void __launch_bounds__(LutCfg<WARPS, R, CPS>::kThreads, CPS)
k_nest_lut(const __grid_constant__ GemmArgs p) {
    using C = LutCfg<WARPS, R, CPS>;
    constexpr int S = C::kStages, NT = C::kTables, TILES = C::kTiles;
    using Cursor = LutCursor<TILES>;
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t* tables = smem + S * C::kStage;
    uint64_t* bars = reinterpret_cast<uint64_t*>(tables + NT * C::kTable);
    const uint32_t bar0 = smem_u32(bars);
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (S + s); };
    auto tfull = [&](int b) { return bar0 + 8u * (2 * S + b); };
    auto tempty = [&](int b) { return bar0 + 8u * (2 * S + NT + b); };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * S + 2 * NT);
    auto stage = [&](int s) { return smem + s * C::kStage; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) { mbar_init(full(s), 1); mbar_init(empty(s), WARPS); }
        for (int b = 0; b < NT; ++b) { mbar_init(tfull(b), 1); mbar_init(tempty(b), WARPS); }
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    grid_dep_launch_dependents();

    long long units = 0;
    for (int k = 0; k < p.ntasks; ++k) units += (long long)Cursor::blocks(p.task[k]) * p.task[k].G;
    const int grid = gridDim.x;
    const long long u0 = unit_begin(blockIdx.x, units, grid);
    const int n = (int)(unit_begin(blockIdx.x + 1, units, grid) - u0);
    Cursor start;
    start.init(p, u0);

    if (warp == C::kProducer) {
        auto tiles_of = [&](const Cursor& c) {
            const int left = p.task[c.k].tiles - c.rb * TILES;
            return left < TILES ? left : TILES;
        };
        auto issue_w = [&](int j, const Cursor& c) {        // lane 0: the block's base units
            const int s = j % S;
            const GemmTask& t = p.task[c.k];
            const int nt = tiles_of(c);
            mbar_arrive_expect_tx(full(s), nt * kBaseUnit);
            for (int i = 0; i < nt; ++i)
                bulk_g2s(smem_u32(stage(s) + i * kBaseUnit),
                         t.base + ((long long)(c.rb * TILES + i) * t.G + c.g) * kBaseUnit, kBaseUnit, full(s));
        };
        Cursor cw = start;
        int j = 0;
        while (j < S && j < n) {             // weights do not depend on the previous kernel: start them now
            if (lane == 0) issue_w(j, cw);
            __syncwarp();
            cw.next(p);
            ++j;
        }
        uint64_t t_last = globaltimer();
        while (j < n) {
            // a blocking test: the lane sleeps in the barrier until the stage is free (or a
            // hardware time limit passes), so the waiting warp takes no issue slots
            bool ready = false;
            if (lane == 0) ready = mbar_try_wait(empty(j % S), ((j / S) - 1) & 1);
            if (__shfl_sync(0xffffffffu, ready, 0)) {
                if (lane == 0) issue_w(j, cw);
                __syncwarp();
                cw.next(p);
                ++j;
                t_last = globaltimer();
            } else {
                const bool stop = (*abort_flag != 0) || (globaltimer() - t_last > kWaitLimitNs);
                if (__shfl_sync(0xffffffffu, stop, 0)) {
                    if (lane == 0 && *abort_flag == 0) { *abort_flag = 1; atomicExch(&g_lut_error, 1); }
                    break;
                }
            }
        }
        __syncwarp();
        // every issued copy has landed before the CTA may leave
        for (int jj = j > S ? j - S : 0; jj < j; ++jj) lut_wait(full(jj % S), (jj / S) & 1, abort_flag, false);
        return;
    }

    if (warp == C::kTableWarp) {
        // lane l builds the sums of pairs l and l + 32: pair P = 4 C + b reads x'[8C + b], x'[8C + b + 4],
        // token 0's values at halves 128 C + b and 128 C + b + 4 of the group's operand block.
        // Sums 4q .. 4q + 3 (c1 = q) go out as one 16-byte store, q rotated by lane / 2 so that the
        // eight lanes of a quarter-warp write eight different 16-byte bank groups.
        float lv[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) lv[c] = level_f(c);
        const int off = 128 * (lane >> 2) + (lane & 3);      // pair `lane`; pair lane + 32 is 8 chunks on
        auto fetch = [&](const Cursor& c, unsigned short (&h)[4]) {
            const unsigned short* x = p.task[c.k].xop + (size_t)c.g * 2048;
            h[0] = __ldcg(x + off);
            h[1] = __ldcg(x + off + 4);
            h[2] = __ldcg(x + off + 1024);
            h[3] = __ldcg(x + off + 1028);
        };
        grid_dep_wait();                     // the activation operand comes from the previous kernel
        Cursor ct = start;
        unsigned short xv[4] = {0, 0, 0, 0}, xn[4] = {0, 0, 0, 0};
        if (n > 0) fetch(ct, xv);
        for (int j = 0; j < n; ++j) {
            const int tb = j % NT;
            Cursor cn = ct;
            cn.next(p);
            if (j + 1 < n) fetch(cn, xn);        // the next super-unit's values, in flight meanwhile
            if (j >= NT && !lut_wait(tempty(tb), ((j / NT) - 1) & 1, abort_flag)) break;
            float* t = reinterpret_cast<float*>(tables + tb * C::kTable);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int P = lane + 32 * h;
                const float x0 = __half2float(__ushort_as_half(xv[2 * h])),
                            x1 = __half2float(__ushort_as_half(xv[2 * h + 1]));
                float a[4], c1[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) { a[c] = lv[c] * x0; c1[c] = lv[c] * x1; }
#pragma unroll
                for (int it = 0; it < 4; ++it) {   // sums 4q .. 4q + 3: c1 = q, c0 = 0..3
                    const int q = (it + (lane >> 1)) & 3;
                    const float cq = (q & 2) ? ((q & 1) ? c1[3] : c1[2]) : ((q & 1) ? c1[1] : c1[0]);
                    *reinterpret_cast<float4*>(t + 16 * P + 4 * q) =
                        make_float4(a[0] + cq, a[1] + cq, a[2] + cq, a[3] + cq);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(tfull(tb));
            ct = cn;
#pragma unroll
            for (int i = 0; i < 4; ++i) xv[i] = xn[i];
        }
        return;
    }

    // row warps: row k of a lane is row 32 (w % 4) + lane of tile w / 4 + k WARPS / 4 of the block
    int tile[R];
#pragma unroll
    for (int k = 0; k < R; ++k) tile[k] = warp / (kRows / 32) + k * (WARPS / (kRows / 32));
    const int rr = 32 * (warp % (kRows / 32)) + lane;
    const uint32_t tables_u32 = smem_u32(tables);
    // scaled sums of the current row block, eight partial sums per row (four lane pairs)
    float2 part[R][4];
#pragma unroll
    for (int k = 0; k < R; ++k)
#pragma unroll
        for (int i = 0; i < 4; ++i) part[k][i] = make_float2(0.0f, 0.0f);

    grid_dep_wait();                          // z is cleared by the previous kernel

    Cursor cj = start;
    int cur_k = -1, t_tiles = 0, t_G = 0, t_M = 0, t_blocks = 0;   // fields of task cj.k
    float* t_z = nullptr;
    int s = 0, ph = 0, tb = 0, tph = 0;       // stage and table ring positions and phases
    for (int j = 0; j < n; ++j) {
        if (!lut_wait(full(s), ph, abort_flag)) break;
        if (!lut_wait(tfull(tb), tph, abort_flag)) break;
        if (cj.k != cur_k) {
            cur_k = cj.k;
            t_tiles = p.task[cur_k].tiles;
            t_G = p.task[cur_k].G;
            t_M = p.task[cur_k].M;
            t_z = p.task[cur_k].z;
            t_blocks = (t_tiles + TILES - 1) / TILES;
        }
        const int live_tiles = t_tiles - cj.rb * TILES;   // tiles of this block that exist
        uint32_t wd[R][8];
        float2 sc[R];
        const uint8_t* st = stage(s);
#pragma unroll
        for (int k = 0; k < R; ++k) {
            if (tile[k] < live_tiles) {
                const uint8_t* un = st + tile[k] * kBaseUnit;
                const uint4 wa = *reinterpret_cast<const uint4*>(un + rr * 16);
                const uint4 wb = *reinterpret_cast<const uint4*>(un + 2048 + rr * 16);
                wd[k][0] = wa.x; wd[k][1] = wa.y; wd[k][2] = wa.z; wd[k][3] = wa.w;
                wd[k][4] = wb.x; wd[k][5] = wb.y; wd[k][6] = wb.z; wd[k][7] = wb.w;
                const float f = __half2float(*reinterpret_cast<const __half*>(un + 4096 + 2 * rr));
                sc[k] = make_float2(f, f);
            } else {                          // a tile past the end of the task: any codes, scale 0
#pragma unroll
                for (int w = 0; w < 8; ++w) wd[k][w] = 0u;
                sc[k] = make_float2(0.0f, 0.0f);
            }
        }
        lut_rows<R>(wd, tables_u32 + tb * C::kTable, sc, part, std::make_integer_sequence<int, 8>{});
        __syncwarp();
        if (lane == 0) { mbar_arrive(empty(s)); mbar_arrive(tempty(tb)); }   // done with the stage and table
        // next super-unit; the row block's sums go out when the range leaves the block
        const int rb_done = cj.rb;
        bool flush = j + 1 == n;
        if (++cj.g == t_G) {
            cj.g = 0;
            flush = true;
            if (++cj.rb == t_blocks) { cj.rb = 0; ++cj.k; }
        }
        if (flush) {
#pragma unroll
            for (int k = 0; k < R; ++k) {
                const int m = (rb_done * TILES + tile[k]) * kRows + rr;
                const float sum = ((part[k][0].x + part[k][0].y) + (part[k][1].x + part[k][1].y)) +
                                  ((part[k][2].x + part[k][2].y) + (part[k][3].x + part[k][3].y));
                if (tile[k] < live_tiles && m < t_M) atomicAdd(t_z + m, sum);
#pragma unroll
                for (int i = 0; i < 4; ++i) part[k][i] = make_float2(0.0f, 0.0f);
            }
        }
        if (++s == S) { s = 0; ph ^= 1; }
        if (++tb == NT) { tb = 0; tph ^= 1; }
    }
}

template <int WARPS, int R, int CPS>
cudaError_t launch_lut_shape(const GemmArgs& a, int sms, cudaStream_t stream) {
    using C = LutCfg<WARPS, R, CPS>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(k_nest_lut<WARPS, R, CPS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::kSmem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    long long units = 0;
    for (int k = 0; k < a.ntasks; ++k)
        units += (long long)((a.task[k].tiles + C::kTiles - 1) / C::kTiles) * a.task[k].G;
    const long long slots = (long long)CPS * sms;
    long long grid = units < slots ? units : slots;
    if (grid > kMaxGrid) grid = kMaxGrid;
    return launch_pdl(k_nest_lut<WARPS, R, CPS>, dim3((unsigned)grid), dim3(C::kThreads), C::kSmem, stream, a);
}

// NEST_LUT_SHAPE=16x2x1 or 8x2x2 picks another compiled shape, for measurement.
}  // namespace

cudaError_t launch_lut(const GemmArgs& a, int sms, cudaStream_t stream) {
    // 4 row warps x 2 rows in four CTAs per SM (256-row blocks): equal to the larger shapes
    // on a long grouped launch, faster on small launches and in the chained layer, where
    // the finer super-units shorten each launch's tail
    const char* e = getenv("NEST_LUT_SHAPE");
    if (e && strcmp(e, "16x2x1") == 0) return launch_lut_shape<16, 2, 1>(a, sms, stream);
    if (e && strcmp(e, "8x2x2") == 0) return launch_lut_shape<8, 2, 2>(a, sms, stream);
    return launch_lut_shape<4, 2, 4>(a, sms, stream);
}

namespace {
// One warp waiting, through the look-up kernel's bounded wait, on a barrier nothing arrives
// on: the give-up path (error flag raised, kernel returns) without a fault.
__global__ void __launch_bounds__(32) k_lut_wait_selftest() {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    lut_wait(smem_u32(&bar), 0, &abort_flag);
}
}  // namespace

cudaError_t launch_lut_wait_selftest(cudaStream_t stream) {
    k_lut_wait_selftest<<<1, 32, 0, stream>>>();
    return cudaGetLastError();
}

cudaError_t read_and_clear_lut_error(int* flag, cudaStream_t stream) {
    cudaError_t e = cudaMemcpyFromSymbolAsync(flag, g_lut_error, sizeof(int), 0, cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    if (*flag) {
        const int zero = 0;
        e = cudaMemcpyToSymbolAsync(g_lut_error, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    }
    return e;
}

}  // namespace nest
