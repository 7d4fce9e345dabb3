/* A plain C11 caller of the library: the header must compile as C on its own, and the
 * host-only entry points (sizes, status names, argument validation) must answer without a
 * GPU.  Every call below either computes a size or is refused by validation before any
 * device work, so the program runs on a machine without a GPU.  Exit status 0 = all
 * checks held; otherwise the number of the first failed check. */
#include "nest.h"

#include <stdint.h>
#include <stdio.h>
#include <string.h>

#define CHECK(n, cond)                                       \
    do {                                                     \
        if (!(cond)) {                                       \
            fprintf(stderr, "check %d failed: %s\n", n, #cond); \
            return n;                                        \
        }                                                    \
    } while (0)

int main(void) {
    /* sizes: base ceil(M/128)*(K/128)*4352, residual ceil(M/128)*(K/128)*(2048 b + 256) */
    CHECK(1, nest_base_bytes(9728, 2560) == (size_t)76 * 20 * 4352);
    CHECK(2, nest_resid_bytes(9728, 2560, 7) == (size_t)76 * 20 * (2048 * 7 + 256));
    CHECK(3, nest_base_bytes(1, 128) == 4352);
    CHECK(4, nest_base_bytes(128, 100) == 0);
    CHECK(5, nest_resid_bytes(128, 128, 5) == 0);
    CHECK(6, nest_hadamard_block(5376) == 256 && nest_hadamard_block(8192) == 4096);
    CHECK(7, nest_xop_bytes(256, 1) == (size_t)2 * 256 * 16 && nest_xop_bytes(128, 257) == 0);
    CHECK(8, nest_linear_scratch_bytes(4096, 4096, 16) == nest_xop_bytes(4096, 16) + (size_t)16 * 4096 * 4);

    /* status names */
    for (int s = NEST_OK; s <= NEST_ERR_TIMEOUT; ++s) {
        const char* name = nest_status_string((nest_status)s);
        CHECK(9, name != NULL && strlen(name) > 0);
    }

    /* validation refuses before any launch: descriptors point at addresses that are never read */
    nest_layer L;
    memset(&L, 0, sizeof(L));
    L.M = 256;
    L.K = 512;
    L.resid_bits = 8;
    L.base = (const uint8_t*)(uintptr_t)0x10000;
    L.resid = (const uint8_t*)(uintptr_t)0x20000;
    L.sign_out = (const int8_t*)(uintptr_t)0x30000;
    L.sign_in = (const int8_t*)(uintptr_t)0x40000;
    const uint16_t* xop = (const uint16_t*)(uintptr_t)0x50000;
    float* z = (float*)(uintptr_t)0x60000;
    CHECK(10, nest_verify_gemm(NULL, xop, z, 16, NULL) == NEST_ERR_INVALID_ARG);
    CHECK(11, nest_verify_gemm(&L, xop, z, 0, NULL) == NEST_ERR_INVALID_ARG);
    CHECK(12, nest_verify_gemm(&L, xop, z, 257, NULL) == NEST_ERR_UNSUPPORTED);
    CHECK(13, nest_verify_gemm(&L, (const uint16_t*)(uintptr_t)0x50008, z, 4, NULL) == NEST_ERR_MISALIGNED);
    L.K = 200;
    CHECK(14, nest_verify_gemm(&L, xop, z, 4, NULL) == NEST_ERR_UNSUPPORTED);
    L.K = 512;
    L.resid_bits = 0;
    CHECK(15, nest_verify_gemm(&L, xop, z, 4, NULL) == NEST_ERR_INVALID_ARG);
    CHECK(16, nest_rotate(NULL, 1, L.sign_in, 128, 4, 0, z, NULL, NULL) == NEST_ERR_INVALID_ARG);
    CHECK(17, nest_linear(&L, 1, NULL, 1, 4, z, (float*)(uintptr_t)0x70000, NULL) == NEST_ERR_INVALID_ARG);

    /* the operand from an already-rotated x', and the row-shard reorder */
    const float* xr = (const float*)(uintptr_t)0x80000;
    uint16_t* xo = (uint16_t*)(uintptr_t)0x90000;
    CHECK(18, nest_operand(NULL, 512, 4, xo, NULL) == NEST_ERR_INVALID_ARG);
    CHECK(19, nest_operand(xr, 500, 4, xo, NULL) == NEST_ERR_UNSUPPORTED);
    CHECK(20, nest_operand(xr, 512, 4, (uint16_t*)(uintptr_t)0x90008, NULL) == NEST_ERR_MISALIGNED);
    CHECK(21, nest_shard_gather(xr, z, 2, 4, 128, 300, NULL) == NEST_ERR_INVALID_ARG);   /* 2 x 128 < 300 rows */
    CHECK(22, nest_shard_gather(xr, z, 0, 4, 128, 100, NULL) == NEST_ERR_INVALID_ARG);

    /* the scale group: 0 (zeroed) and 128 are the format's; others are refused */
    L.resid_bits = 8;
    L.group = 8;
    CHECK(23, nest_verify_gemm(&L, xop, z, 4, NULL) == NEST_ERR_UNSUPPORTED);
    L.group = 128;
    CHECK(24, nest_verify_gemm(&L, (const uint16_t*)(uintptr_t)0x50008, z, 4, NULL) == NEST_ERR_MISALIGNED);

    printf("ok\n");
    return 0;
}
