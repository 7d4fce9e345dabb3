// C-ABI entry points of libnest (declared in include/nest.h): host-side
// argument validation, launch configuration, and status codes.  No entry
// point allocates memory or synchronises (except nest_error_check).
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <cuda_runtime.h>

#include "../../include/nest.h"
#include "nest_device.cuh"
#include "nest_internal.h"

using namespace nest;

namespace {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

nest_status from_cuda(cudaError_t e) { return e == cudaSuccess ? NEST_OK : NEST_ERR_CUDA; }

// number of SMs of the current device (queried once per device)
int device_sms() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cached[dev] == 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cached[dev] = v;
    }
    return cached[dev];
}

// the tcgen05 kernels are built for sm_103a only
bool device_supported() {
    static int cached[64] = {0};   // 0 unknown, 1 yes, 2 no
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    if (cached[dev] == 0) {
        int major = 0, minor = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        cached[dev] = (major == 10 && minor == 3) ? 1 : 2;
    }
    return cached[dev] == 1;
}

bool bits_ok(int bits) { return bits == 6 || bits == 7 || bits == 8; }

nest_status check_layer(const nest_layer* L, bool need_resid) {
    if (L == nullptr) return NEST_ERR_INVALID_ARG;
    if (L->M < 1 || L->K < 1) return NEST_ERR_INVALID_ARG;
    if (L->group != 0 && L->group != 128) return NEST_ERR_UNSUPPORTED;   // the format's group is 128 columns
    if (L->K % 128 != 0) return NEST_ERR_UNSUPPORTED;
    if (L->base == nullptr) return NEST_ERR_INVALID_ARG;
    if (!aligned16(L->base)) return NEST_ERR_MISALIGNED;
    if (L->codec == NEST_CODEC_W4W8) {
        if (L->resid_bits != 0 && L->resid_bits != 4) return NEST_ERR_UNSUPPORTED;
        if (need_resid) {
            if (L->resid_bits != 4 || L->resid == nullptr) return NEST_ERR_INVALID_ARG;
            if (!aligned16(L->resid)) return NEST_ERR_MISALIGNED;
        }
        return NEST_OK;
    }
    if (L->codec != NEST_CODEC_L2) return NEST_ERR_UNSUPPORTED;
    if (need_resid) {
        if (!bits_ok(L->resid_bits)) return L->resid_bits == 0 ? NEST_ERR_INVALID_ARG : NEST_ERR_UNSUPPORTED;
        if (L->resid == nullptr) return NEST_ERR_INVALID_ARG;
        if (!aligned16(L->resid)) return NEST_ERR_MISALIGNED;
    } else if (L->resid_bits != 0 && !bits_ok(L->resid_bits)) {
        return NEST_ERR_UNSUPPORTED;
    }
    return NEST_OK;
}

// One launch over `count` independent linears (same residual width, same T).
nest_status run_gemm_group(const nest_layer* layers, int count, bool verify, const uint16_t* const* xops,
                           float* const* zs, int T, void* stream) {
    if (layers == nullptr || xops == nullptr || zs == nullptr) return NEST_ERR_INVALID_ARG;
    if (count < 1) return NEST_ERR_INVALID_ARG;
    if (count > kMaxGemmTasks) return NEST_ERR_UNSUPPORTED;
    if (T < 1) return NEST_ERR_INVALID_ARG;
    if (T > kMaxT) return NEST_ERR_UNSUPPORTED;
    const int codec = layers[0].codec;
    const int bits = verify ? layers[0].resid_bits : 0;
    if (verify && bits == 0) return NEST_ERR_INVALID_ARG;
    // kernel codec: 0 / 6 / 7 / 8 (2-bit base, residual width) or 40 / 48 (W4 draft / W8 target)
    const int kcodec = codec == NEST_CODEC_W4W8 ? (verify ? 48 : 40) : bits;
    GemmArgs a = {};
    a.ntasks = count;
    a.T = T;
    long long units = 0;
    for (int k = 0; k < count; ++k) {
        const nest_layer* L = &layers[k];
        nest_status st = check_layer(L, verify);
        if (st != NEST_OK) return st;
        if (L->codec != codec || (verify && L->resid_bits != bits)) return NEST_ERR_INVALID_ARG;
        if (xops[k] == nullptr || zs[k] == nullptr) return NEST_ERR_INVALID_ARG;
        if (!aligned16(xops[k]) || (reinterpret_cast<uintptr_t>(zs[k]) & 3u)) return NEST_ERR_MISALIGNED;
        GemmTask& t = a.task[k];
        t.base = L->base;
        t.resid = verify ? L->resid : nullptr;
        t.xop = xops[k];
        t.z = zs[k];
        t.M = L->M;
        t.G = L->K / 128;
        t.tiles = n_tiles(L->M);
        t.ubegin = units;
        units += (long long)t.tiles * t.G;
    }
    a.units = units;
    if (!device_supported()) return NEST_ERR_UNSUPPORTED;
    const int sms = device_sms();
    if (sms <= 0) return NEST_ERR_CUDA;
    const long long slots = (long long)gemm_ctas_per_sm(T) * sms;   // every CTA resident at once
    long long grid = units < slots ? units : slots;
    if (grid > kMaxGrid) grid = kMaxGrid;
    return from_cuda(launch_gemm(a, kcodec, (int)grid, sms, as_stream(stream)));
}

}  // namespace

extern "C" {

const char* nest_status_string(nest_status s) {
    switch (s) {
        case NEST_OK: return "ok";
        case NEST_ERR_INVALID_ARG: return "invalid argument";
        case NEST_ERR_UNSUPPORTED: return "unsupported shape, bit width or device";
        case NEST_ERR_MISALIGNED: return "pointer not 16-byte aligned";
        case NEST_ERR_CUDA: return "CUDA error";
        case NEST_ERR_TIMEOUT: return "kernel pipeline wait timed out";
    }
    return "unknown status";
}

int32_t nest_hadamard_block(int32_t n) { return hadamard_block(n); }

size_t nest_base_bytes(int32_t M, int32_t K) {
    if (M < 1 || K < 1 || K % 128) return 0;
    return (size_t)n_tiles(M) * (K / 128) * 4352;
}

size_t nest_resid_bytes(int32_t M, int32_t K, int32_t bits) {
    if (M < 1 || K < 1 || K % 128 || !bits_ok(bits)) return 0;
    return (size_t)n_tiles(M) * (K / 128) * (2048 * (size_t)bits + 256);
}

size_t nest_w4_base_bytes(int32_t M, int32_t K) {
    if (M < 1 || K < 1 || K % 128) return 0;
    return (size_t)n_tiles(M) * (K / 128) * kW4BaseUnit;
}

size_t nest_w4_ref_bytes(int32_t M, int32_t K) {
    if (M < 1 || K < 1 || K % 128) return 0;
    return (size_t)n_tiles(M) * (K / 128) * kW4RefUnit;
}

nest_status nest_quantize_w4w8(const float* W, const int8_t* sign_out, const int8_t* sign_in, int32_t M, int32_t K,
                               double* work, int8_t* q4, uint16_t* s4, int8_t* q_r, void* stream) {
    if (!W || !sign_out || !sign_in || !work || !q4 || !s4) return NEST_ERR_INVALID_ARG;
    if (M < 1 || K < 1) return NEST_ERR_INVALID_ARG;
    if (K % 128) return NEST_ERR_UNSUPPORTED;
    if (!aligned16(W) || !aligned16(work)) return NEST_ERR_MISALIGNED;
    if (reinterpret_cast<uintptr_t>(s4) & 1u) return NEST_ERR_MISALIGNED;
    if ((long long)M * (K / hadamard_block(K)) > 0x7fffffffLL) return NEST_ERR_UNSUPPORTED;
    return from_cuda(launch_quantize_w4w8(W, sign_out, sign_in, M, K, work, q4, s4, q_r, as_stream(stream)));
}

nest_status nest_pack_w4w8(const int8_t* q4, const uint16_t* s4, const int8_t* q_r, int32_t M, int32_t K,
                           uint8_t* base_out, uint8_t* ref_out, void* stream) {
    if (!q4 || !s4 || !base_out) return NEST_ERR_INVALID_ARG;
    if (q_r != nullptr && ref_out == nullptr) return NEST_ERR_INVALID_ARG;
    if (M < 1 || K < 1) return NEST_ERR_INVALID_ARG;
    if (K % 128) return NEST_ERR_UNSUPPORTED;
    if (!aligned16(base_out) || (q_r && !aligned16(ref_out))) return NEST_ERR_MISALIGNED;
    if (reinterpret_cast<uintptr_t>(s4) & 1u) return NEST_ERR_MISALIGNED;
    return from_cuda(launch_pack_w4w8(q4, s4, q_r, M, K, base_out, q_r ? ref_out : nullptr, as_stream(stream)));
}

nest_status nest_unpack_w4w8(const nest_layer* layer, int8_t* q4, uint16_t* s4, int8_t* q_r, void* stream) {
    if (layer == nullptr || layer->codec != NEST_CODEC_W4W8) return NEST_ERR_INVALID_ARG;
    nest_status st = check_layer(layer, q_r != nullptr);
    if (st != NEST_OK) return st;
    if (!q4 || !s4) return NEST_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(s4) & 1u) return NEST_ERR_MISALIGNED;
    return from_cuda(launch_unpack_w4w8(layer->base, q_r ? layer->resid : nullptr, layer->M, layer->K, q4, s4, q_r,
                                        as_stream(stream)));
}

size_t nest_xop_bytes(int32_t K, int32_t T) {
    if (K < 1 || K % 128 || T < 1 || T > kMaxT) return 0;
    return (size_t)(K / 128) * 256 * n_pad(T);
}

nest_status nest_quantize(const float* W, const int8_t* sign_out, const int8_t* sign_in, int32_t M, int32_t K,
                          int32_t bits, double* work, uint8_t* base_codes, uint16_t* base_scales,
                          int8_t* resid_codes, uint16_t* resid_scales, void* stream) {
    if (!W || !sign_out || !sign_in || !work || !base_codes || !base_scales) return NEST_ERR_INVALID_ARG;
    if (M < 1 || K < 1) return NEST_ERR_INVALID_ARG;
    if (K % 128) return NEST_ERR_UNSUPPORTED;
    if (bits != 0 && !bits_ok(bits)) return NEST_ERR_UNSUPPORTED;
    if (bits != 0 && (!resid_codes || !resid_scales)) return NEST_ERR_INVALID_ARG;
    if (!aligned16(W) || !aligned16(work)) return NEST_ERR_MISALIGNED;
    if ((reinterpret_cast<uintptr_t>(base_scales) & 1u) || (bits && (reinterpret_cast<uintptr_t>(resid_scales) & 1u)))
        return NEST_ERR_MISALIGNED;
    if ((long long)M * (K / hadamard_block(K)) > 0x7fffffffLL) return NEST_ERR_UNSUPPORTED;
    return from_cuda(launch_quantize(W, sign_out, sign_in, M, K, bits, work, base_codes, base_scales,
                                     resid_codes, resid_scales, as_stream(stream)));
}

nest_status nest_pack(const uint8_t* base_codes, const uint16_t* base_scales, const int8_t* resid_codes,
                      const uint16_t* resid_scales, int32_t M, int32_t K, int32_t bits, uint8_t* base_out,
                      uint8_t* resid_out, void* stream) {
    if (!base_codes || !base_scales || !base_out) return NEST_ERR_INVALID_ARG;
    if (M < 1 || K < 1) return NEST_ERR_INVALID_ARG;
    if (K % 128) return NEST_ERR_UNSUPPORTED;
    if (bits != 0 && !bits_ok(bits)) return NEST_ERR_UNSUPPORTED;
    if (bits != 0 && (!resid_codes || !resid_scales || !resid_out)) return NEST_ERR_INVALID_ARG;
    if (!aligned16(base_out) || (bits && !aligned16(resid_out))) return NEST_ERR_MISALIGNED;
    if ((reinterpret_cast<uintptr_t>(base_scales) & 1u) || (bits && (reinterpret_cast<uintptr_t>(resid_scales) & 1u)))
        return NEST_ERR_MISALIGNED;
    return from_cuda(launch_pack(base_codes, base_scales, resid_codes, resid_scales, M, K, bits, base_out,
                                 resid_out, as_stream(stream)));
}

nest_status nest_unpack(const nest_layer* layer, uint8_t* base_codes, uint16_t* base_scales, int8_t* resid_codes,
                        uint16_t* resid_scales, void* stream) {
    if (layer != nullptr && layer->codec != NEST_CODEC_L2) return NEST_ERR_INVALID_ARG;
    nest_status st = check_layer(layer, false);
    if (st != NEST_OK) return st;
    const int bits = layer->resid_bits;
    if (!base_codes || !base_scales) return NEST_ERR_INVALID_ARG;
    if (bits && (!layer->resid || !resid_codes || !resid_scales)) return NEST_ERR_INVALID_ARG;
    if (bits && !aligned16(layer->resid)) return NEST_ERR_MISALIGNED;
    if ((reinterpret_cast<uintptr_t>(base_scales) & 1u) || (bits && (reinterpret_cast<uintptr_t>(resid_scales) & 1u)))
        return NEST_ERR_MISALIGNED;
    return from_cuda(launch_unpack(layer->base, bits ? layer->resid : nullptr, layer->M, layer->K, bits, base_codes,
                                   base_scales, resid_codes, resid_scales, as_stream(stream)));
}

nest_status nest_rotate(const void* x, int32_t x_dtype, const int8_t* signs, int32_t n, int32_t T, int32_t mode,
                        float* y, uint16_t* x_op, void* stream) {
    if (!x || !signs || (!y && !x_op)) return NEST_ERR_INVALID_ARG;
    if (n < 1 || T < 1) return NEST_ERR_INVALID_ARG;
    if ((long long)n * T >= (1LL << 31)) return NEST_ERR_UNSUPPORTED;
    if ((x_dtype != 0 && x_dtype != 1) || (mode != 0 && mode != 1)) return NEST_ERR_INVALID_ARG;
    if (x_op != nullptr) {
        if (mode != 0) return NEST_ERR_INVALID_ARG;
        if (n % 128 || T > kMaxT) return NEST_ERR_UNSUPPORTED;
        if (!aligned16(x_op)) return NEST_ERR_MISALIGNED;
    }
    if ((reinterpret_cast<uintptr_t>(x) & (x_dtype == 1 ? 1u : 3u)) || (y && (reinterpret_cast<uintptr_t>(y) & 3u)))
        return NEST_ERR_MISALIGNED;
    return from_cuda(launch_rotate(x, x_dtype, signs, n, T, mode, y, x_op, nullptr, 0, as_stream(stream)));
}

nest_status nest_draft_gemv(const nest_layer* layer, const uint16_t* x_op, float* z, int32_t T, void* stream) {
    return run_gemm_group(layer, 1, false, &x_op, &z, T, stream);
}

nest_status nest_verify_gemm(const nest_layer* layer, const uint16_t* x_op, float* z, int32_t T, void* stream) {
    return run_gemm_group(layer, 1, true, &x_op, &z, T, stream);
}

nest_status nest_draft_gemv_group(const nest_layer* layers, int32_t count, const uint16_t* const* x_ops,
                                  float* const* z, int32_t T, void* stream) {
    return run_gemm_group(layers, count, false, x_ops, z, T, stream);
}

nest_status nest_verify_gemm_group(const nest_layer* layers, int32_t count, const uint16_t* const* x_ops,
                                   float* const* z, int32_t T, void* stream) {
    return run_gemm_group(layers, count, true, x_ops, z, T, stream);
}

// scratch of nest_linear: [x_op][z], each 256-byte aligned; of nest_linear_group: one such pair per linear
static size_t round256(size_t v) { return (v + 255) / 256 * 256; }

size_t nest_linear_scratch_bytes(int32_t M, int32_t K, int32_t T) {
    if (M < 1 || K < 1 || K % 128 || T < 1 || T > kMaxT) return 0;
    return round256(nest_xop_bytes(K, T)) + round256((size_t)T * M * sizeof(float));
}

size_t nest_linear_group_scratch_bytes(const nest_layer* layers, int32_t count, int32_t T) {
    if (layers == nullptr || count < 1 || count > kMaxTasks) return 0;
    size_t total = 0;
    for (int k = 0; k < count; ++k) {
        const size_t b = nest_linear_scratch_bytes(layers[k].M, layers[k].K, T);
        if (b == 0) return 0;
        total += b;
    }
    return total;
}

nest_status nest_linear_group(const nest_layer* layers, int32_t count, int32_t verify, const void* const* xs,
                              int32_t x_dtype, int32_t T, float* const* ys, void* scratch, void* stream) {
    if (layers == nullptr || xs == nullptr || ys == nullptr || scratch == nullptr) return NEST_ERR_INVALID_ARG;
    if (count < 1) return NEST_ERR_INVALID_ARG;
    if (count > kMaxTasks) return NEST_ERR_UNSUPPORTED;
    if (x_dtype != 0 && x_dtype != 1) return NEST_ERR_INVALID_ARG;
    if (T < 1) return NEST_ERR_INVALID_ARG;
    if (T > kMaxT) return NEST_ERR_UNSUPPORTED;
    if (!aligned16(scratch)) return NEST_ERR_MISALIGNED;
    RotArgs rin = {}, rout = {};
    const uint16_t* xops[kMaxTasks];
    float* zs[kMaxTasks];
    uint8_t* s = reinterpret_cast<uint8_t*>(scratch);
    for (int k = 0; k < count; ++k) {
        const nest_layer* L = &layers[k];
        nest_status st = check_layer(L, verify != 0);
        if (st != NEST_OK) return st;
        if (!L->sign_in || !L->sign_out || !xs[k] || !ys[k]) return NEST_ERR_INVALID_ARG;
        if ((reinterpret_cast<uintptr_t>(xs[k]) & (x_dtype == 1 ? 1u : 3u)) || (reinterpret_cast<uintptr_t>(ys[k]) & 3u))
            return NEST_ERR_MISALIGNED;
        uint16_t* xop = reinterpret_cast<uint16_t*>(s);
        float* z = reinterpret_cast<float*>(s + round256(nest_xop_bytes(L->K, T)));
        s += nest_linear_scratch_bytes(L->M, L->K, T);
        xops[k] = xop;
        zs[k] = z;
        // rotate in, writing the GEMM operand and clearing the accumulator z
        rin.task[k] = RotTask{xs[k], L->sign_in, nullptr, xop, z, (long long)T * L->M, (unsigned)L->K};
        // rotate out
        rout.task[k] = RotTask{z, L->sign_out, ys[k], nullptr, nullptr, 0, (unsigned)L->M};
    }
    rin.ntasks = rout.ntasks = count;
    if (launch_rotate_group(rin, x_dtype, 0, T, as_stream(stream)) != cudaSuccess) return NEST_ERR_CUDA;
    nest_status st = run_gemm_group(layers, count, verify != 0, xops, zs, T, stream);
    if (st != NEST_OK) return st;
    if (launch_rotate_group(rout, 0, 1, T, as_stream(stream)) != cudaSuccess) return NEST_ERR_CUDA;
    return NEST_OK;
}

nest_status nest_linear(const nest_layer* layer, int32_t verify, const void* x, int32_t x_dtype, int32_t T, float* y,
                        void* scratch, void* stream) {
    return nest_linear_group(layer, 1, verify, &x, x_dtype, T, &y, scratch, stream);
}

size_t nest_chain_work_bytes(int32_t M, int32_t T) {
    if (M < 1 || T < 1 || T > kMaxT) return 0;
    return round256((size_t)glue_work_floats(M, T) * sizeof(float));
}

nest_status nest_chain(float* z_a, const int8_t* sign_out_a, const float* z_b, const int8_t* sign_out_b,
                       int32_t M, int32_t T, float* y, const nest_layer* next, int32_t n_next,
                       uint16_t* const* x_ops, float* const* z_next, float* work,
                       const nest_rotate_task* side, int32_t n_side, void* stream) {
    if (z_a == nullptr || sign_out_a == nullptr || work == nullptr) return NEST_ERR_INVALID_ARG;
    if (n_side < 0 || (n_side > 0 && side == nullptr)) return NEST_ERR_INVALID_ARG;
    if (n_side > kMaxChainSide) return NEST_ERR_UNSUPPORTED;
    if ((z_b == nullptr) != (sign_out_b == nullptr)) return NEST_ERR_INVALID_ARG;
    if (z_b == z_a || (y != nullptr && y == z_b)) return NEST_ERR_INVALID_ARG;
    if (M < 1 || T < 1 || n_next < 0) return NEST_ERR_INVALID_ARG;
    if (T > kMaxT || n_next > kMaxChainNext) return NEST_ERR_UNSUPPORTED;
    if ((long long)M * T >= (1LL << 31)) return NEST_ERR_UNSUPPORTED;
    if (n_next > 0 && (next == nullptr || x_ops == nullptr)) return NEST_ERR_INVALID_ARG;
    if (n_next > 0 && M % 128) return NEST_ERR_UNSUPPORTED;
    for (int j = 0; j < n_next; ++j)
        if (next[j].group != 0 && next[j].group != 128) return NEST_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(z_a) & 3u) || (z_b && (reinterpret_cast<uintptr_t>(z_b) & 3u)) ||
        (y && (reinterpret_cast<uintptr_t>(y) & 3u)) || (reinterpret_cast<uintptr_t>(work) & 3u))
        return NEST_ERR_MISALIGNED;
    GlueArgs c = {};
    c.za = z_a;
    c.sa = sign_out_a;
    c.zb = z_b;
    c.sb = sign_out_b;
    c.h = y != nullptr ? y : z_a;
    c.work = work;
    c.nnext = n_next;
    c.M = M;
    c.T = T;
    for (int j = 0; j < n_next; ++j) {
        const nest_layer& L = next[j];
        if (L.K != M || L.sign_in == nullptr || x_ops[j] == nullptr) return NEST_ERR_INVALID_ARG;
        if (!aligned16(x_ops[j])) return NEST_ERR_MISALIGNED;
        float* zn = z_next ? z_next[j] : nullptr;
        if (zn && (reinterpret_cast<uintptr_t>(zn) & 3u)) return NEST_ERR_MISALIGNED;
        c.next[j] = GlueNext{L.sign_in, x_ops[j], zn, zn ? (long long)T * L.M : 0};
    }
    // side output rotations: plain z -> y tasks on buffers of their own
    for (int k = 0; k < n_side; ++k) {
        const nest_rotate_task& r = side[k];
        if (!r.x || !r.signs || !r.y || r.x_op || r.zero_out || r.zero_count || r.n < 1) return NEST_ERR_INVALID_ARG;
        if ((long long)r.n * T >= (1LL << 31)) return NEST_ERR_UNSUPPORTED;
        if ((reinterpret_cast<uintptr_t>(r.x) & 3u) || (reinterpret_cast<uintptr_t>(r.y) & 3u))
            return NEST_ERR_MISALIGNED;
        const void* mine[2] = {r.x, r.y};
        for (const void* p : mine) {
            if (p == z_a || (z_b && p == z_b) || (y && p == y)) return NEST_ERR_INVALID_ARG;
            for (int o = 0; o < k; ++o)
                if (p == side[o].x || p == side[o].y) return NEST_ERR_INVALID_ARG;
        }
        if (r.x == r.y) return NEST_ERR_INVALID_ARG;
        c.side[k] = GlueSide{static_cast<const float*>(r.x), r.signs, r.y, r.n, 0, 0, 0, 0.0f, 0};
    }
    c.nside = n_side;
    return from_cuda(launch_glue(c, as_stream(stream)));
}

nest_status nest_rotate_group(const nest_rotate_task* tasks, int32_t count, int32_t x_dtype, int32_t T,
                              int32_t mode, void* stream) {
    if (tasks == nullptr || count < 1 || T < 1) return NEST_ERR_INVALID_ARG;
    if (count > kMaxTasks) return NEST_ERR_UNSUPPORTED;
    if ((x_dtype != 0 && x_dtype != 1) || (mode != 0 && mode != 1)) return NEST_ERR_INVALID_ARG;
    RotArgs a = {};
    a.ntasks = count;
    long long ctas = 0;
    for (int k = 0; k < count; ++k) {
        const nest_rotate_task& r = tasks[k];
        if (!r.x || !r.signs || (!r.y && !r.x_op) || r.n < 1) return NEST_ERR_INVALID_ARG;
        if ((long long)r.n * T >= (1LL << 31)) return NEST_ERR_UNSUPPORTED;
        if (r.x_op != nullptr) {
            if (mode != 0) return NEST_ERR_INVALID_ARG;
            if (r.n % 128 || T > kMaxT) return NEST_ERR_UNSUPPORTED;
            if (!aligned16(r.x_op)) return NEST_ERR_MISALIGNED;
        }
        if ((reinterpret_cast<uintptr_t>(r.x) & (x_dtype == 1 ? 1u : 3u)) ||
            (r.y && (reinterpret_cast<uintptr_t>(r.y) & 3u)))
            return NEST_ERR_MISALIGNED;
        if (r.zero_count < 0 || (r.zero_count > 0 && r.zero_out == nullptr)) return NEST_ERR_INVALID_ARG;
        if (r.zero_out && (reinterpret_cast<uintptr_t>(r.zero_out) & 3u)) return NEST_ERR_MISALIGNED;
        // at most one CTA per 512 elements, or per 2048 floats to clear (the launch's bound)
        const long long c_rot = ((long long)r.n * T + 511) / 512, c_clr = (r.zero_count + 2047) / 2048;
        ctas += c_rot > c_clr ? c_rot : c_clr;
        a.task[k].x = r.x;
        a.task[k].signs = r.signs;
        a.task[k].y = r.y;
        a.task[k].xop = r.x_op;
        a.task[k].zero_out = r.zero_count > 0 ? r.zero_out : nullptr;
        a.task[k].zero_count = r.zero_count;
        a.task[k].n = (unsigned)r.n;
    }
    if (ctas >= (1LL << 31)) return NEST_ERR_UNSUPPORTED;
    return from_cuda(launch_rotate_group(a, x_dtype, mode, T, as_stream(stream)));
}

size_t nest_kv_plane_bytes(int32_t H, int32_t Lmax) {
    if (H < 1 || Lmax < 1) return 0;
    return (size_t)H * Lmax * 64;
}

static nest_status check_kv(const nest_kv_cache* c) {
    if (c == nullptr || !c->base || !c->ref || !c->scale) return NEST_ERR_INVALID_ARG;
    if (c->H < 1 || c->Lmax < 1) return NEST_ERR_INVALID_ARG;
    if ((long long)c->H * c->Lmax >= (1LL << 26)) return NEST_ERR_UNSUPPORTED;   // 32-bit plane offsets
    if (!aligned16(c->base) || !aligned16(c->ref) || (reinterpret_cast<uintptr_t>(c->scale) & 1u))
        return NEST_ERR_MISALIGNED;
    return NEST_OK;
}

nest_status nest_kv_write(const void* x, int32_t x_dtype, int32_t T, const nest_kv_cache* cache, int32_t pos0,
                          void* stream) {
    nest_status st = check_kv(cache);
    if (st != NEST_OK) return st;
    if (x == nullptr || T < 1 || pos0 < 0 || (x_dtype != 0 && x_dtype != 1)) return NEST_ERR_INVALID_ARG;
    if ((long long)pos0 + T > cache->Lmax) return NEST_ERR_INVALID_ARG;
    if ((long long)T * cache->H * 32 >= (1LL << 31)) return NEST_ERR_UNSUPPORTED;
    if (reinterpret_cast<uintptr_t>(x) & (x_dtype == 1 ? 1u : 3u)) return NEST_ERR_MISALIGNED;
    return from_cuda(launch_kv_write(x, x_dtype, T, cache->H, pos0, cache->Lmax, cache->base, cache->ref,
                                     cache->scale, as_stream(stream)));
}

size_t nest_kv_attention_work_bytes(int32_t T, int32_t Hq, int32_t Hkv, int32_t L) {
    if (T < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || L < T) return 0;
    const int sms = device_sms();
    if (sms <= 0) return 0;
    const int G = Hq / Hkv;
    const int rows = kv_rows_per_tile();
    const long long tiles = ((long long)T * G + rows - 1) / rows;
    const long long ns = kv_splits(T, G, Hkv, L, sms);
    return (size_t)Hkv * tiles * ns * rows * (128 + 2) * sizeof(float);
}

nest_status nest_kv_attention(const void* q, int32_t q_dtype, int32_t T, int32_t Hq, const nest_kv_cache* k,
                              const nest_kv_cache* v, int32_t L, int32_t view, int32_t recent_n, float* out,
                              float* work, void* stream) {
    nest_status st = check_kv(k);
    if (st == NEST_OK) st = check_kv(v);
    if (st != NEST_OK) return st;
    if (!q || !out || !work || T < 1 || Hq < 1 || (q_dtype != 0 && q_dtype != 1)) return NEST_ERR_INVALID_ARG;
    if (view != 4 && view != 8) return NEST_ERR_INVALID_ARG;
    if (recent_n < 0) return NEST_ERR_INVALID_ARG;
    const int Hkv = k->H;
    if (v->H != Hkv || Hq % Hkv) return NEST_ERR_INVALID_ARG;
    if (L < T || L > k->Lmax || L > v->Lmax) return NEST_ERR_INVALID_ARG;
    if ((long long)T * (Hq / Hkv) > 65535LL * kv_rows_per_tile()) return NEST_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(q) & (q_dtype == 1 ? 1u : 3u)) || (reinterpret_cast<uintptr_t>(out) & 3u) ||
        (reinterpret_cast<uintptr_t>(work) & 3u))
        return NEST_ERR_MISALIGNED;
    if (!device_supported()) return NEST_ERR_UNSUPPORTED;
    const int sms = device_sms();
    if (sms <= 0) return NEST_ERR_CUDA;
    KvAttnArgs a = {};
    a.q = q;
    a.q_bf16 = q_dtype;
    a.kbase = k->base; a.kref = k->ref; a.kscale = k->scale;
    a.vbase = v->base; a.vref = v->ref; a.vscale = v->scale;
    a.out = out;
    a.work = work;
    a.T = T; a.Hq = Hq; a.Hkv = Hkv; a.G = Hq / Hkv; a.L = L;
    if (k->Lmax != v->Lmax) return NEST_ERR_INVALID_ARG;
    a.Lmax = k->Lmax;
    a.view = view;
    a.recent_n = recent_n;
    // for measurement: "cuda" the CUDA-core kernel, "tc16" tensor-core CTAs of at most 16 rows
    const char* impl = getenv("NEST_KV_IMPL");
    a.impl = (impl && impl[0] == 'c') ? 1 : (impl && strncmp(impl, "tc16", 4) == 0) ? 2 : 0;
    return from_cuda(launch_kv_attention(a, sms, as_stream(stream)));
}

nest_status nest_error_check(void* stream) {
    int flag = 0, lut_flag = 0;
    cudaError_t e = read_and_clear_error(&flag, as_stream(stream));
    if (e == cudaSuccess) e = read_and_clear_lut_error(&lut_flag, as_stream(stream));
    if (e != cudaSuccess) return NEST_ERR_CUDA;
    return (flag || lut_flag) ? NEST_ERR_TIMEOUT : NEST_OK;
}

nest_status nest_wait_selftest(int32_t which, void* stream) {
    if (which == 0) return from_cuda(launch_wait_selftest(as_stream(stream)));
    if (which == 1) return from_cuda(launch_lut_wait_selftest(as_stream(stream)));
    return NEST_ERR_INVALID_ARG;
}

}  // extern "C"
