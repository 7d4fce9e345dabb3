/*
 * Reference packer for the nested-bit storage format.  TEST INFRASTRUCTURE:
 * loaded only by the test suite (through oracle/pack.py); the CUDA library
 * has its own packer and shares nothing with this file.
 *
 * Storage (the 2-bit-base post, POC recipe steps 2 and 3: "2 bit-planes plus
 * an fp16 scale per 128 weights" for the base; a separate b-bit residual with
 * an fp16 scale per (row, 128-group)).  Base and residual live in two
 * separate buffers so a draft pass reads the base alone (the dual-plane
 * principle of BitNest, section 3.3).
 *
 * Both buffers are arrays of UNITS.  A unit covers one tile of 128 output
 * rows and one 128-column group; units are ordered tile-major
 * (unit = tile * (K/128) + group).  Rows past M in the last tile hold code 0,
 * residual 0 and scale 0.
 *
 * Base unit (4352 bytes):
 *   bytes [0, 4096): the 2-bit codes, chunk-major: the 16-byte chunk c (0..1)
 *                    of row r sits at byte (c*128 + r)*16.  A row's 32 code
 *                    bytes are 8 little-endian 32-bit words; word w (chunk
 *                    w/4, word w%4 of the chunk) holds columns 16w..16w+15:
 *                    column 16w + 4p + q sits at bits 8q + 2p .. 8q + 2p + 1.
 *                    A code is the index 0..3 of the level, levels ascending.
 *   bytes [4096, 4352): the fp16 scale of row r at byte 4096 + 2r.
 *
 * Residual unit (2048*b + 256 bytes), stored value u = q + 2^(b-1) (1..2^b-1):
 *   bytes [0, 2048*b): a row's 16*b bytes as 4*b words, chunk-major as above
 *                    (word w of row r at byte ((w/4)*128 + r)*16 + (w%4)*4).
 *     b = 8: word w holds columns 4w..4w+3, column 4w + q in byte q.
 *     b = 6, 7: u split into a 4-bit low part, a 2-bit middle part
 *               (bits 4..5) and, for b = 7, a 1-bit high part (bit 6):
 *       words  0..15: low nibbles; word a holds columns 8a..8a+7, column
 *                     8a + 4h + q in bits 8q + 4h .. 8q + 4h + 3;
 *       words 16..23: middle pairs; word 16+a holds columns 16a..16a+15,
 *                     column 16a + 4p + q in bits 8q + 2p .. 8q + 2p + 1;
 *       words 24..27 (b = 7): high bits; word 24+a holds columns
 *                     32a..32a+31, column 32a + 4p + q in bit 8q + p.
 *   bytes [2048*b, 2048*b + 256): fp16 scale of row r at 2048*b + 2r.
 */
#include <stdint.h>
#include <stddef.h>
#include <string.h>

#define ROWS 128
#define GROUP 128

static size_t n_tiles(int M) { return (size_t)((M + ROWS - 1) / ROWS); }

size_t ref_base_unit_bytes(void) { return 4096 + 256; }
size_t ref_resid_unit_bytes(int bits) { return (size_t)2048 * bits + 256; }

size_t ref_base_bytes(int M, int K) {
    return n_tiles(M) * (size_t)(K / GROUP) * ref_base_unit_bytes();
}

size_t ref_resid_bytes(int M, int K, int bits) {
    return n_tiles(M) * (size_t)(K / GROUP) * ref_resid_unit_bytes(bits);
}

/* byte offset, inside a unit, of word w of row r */
static size_t word_offset(int r, int w) {
    return ((size_t)(w / 4) * ROWS + r) * 16 + (size_t)(w % 4) * 4;
}

static void set_bits(uint8_t* unit, int r, int w, int bit, uint32_t value) {
    uint8_t* p = unit + word_offset(r, w);
    uint32_t word = (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
    word |= value << bit;
    p[0] = (uint8_t)word; p[1] = (uint8_t)(word >> 8); p[2] = (uint8_t)(word >> 16); p[3] = (uint8_t)(word >> 24);
}

static uint32_t get_bits(const uint8_t* unit, int r, int w, int bit, uint32_t mask) {
    const uint8_t* p = unit + word_offset(r, w);
    uint32_t word = (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
    return (word >> bit) & mask;
}

/* where column j (0..127) of a row lives in the base code words */
static void base_pos(int j, int* w, int* bit) {
    int jj = j % 16;
    *w = j / 16;
    *bit = 8 * (jj % 4) + 2 * (jj / 4);
}

void ref_pack_base(const uint8_t* codes, const uint16_t* scales, int M, int K, uint8_t* out) {
    int G = K / GROUP;
    size_t ub = ref_base_unit_bytes();
    memset(out, 0, ref_base_bytes(M, K));
    for (size_t t = 0; t < n_tiles(M); ++t)
        for (int g = 0; g < G; ++g) {
            uint8_t* unit = out + (t * G + g) * ub;
            for (int r = 0; r < ROWS; ++r) {
                size_t m = t * ROWS + r;
                if (m >= (size_t)M) continue;
                for (int j = 0; j < GROUP; ++j) {
                    int w, bit;
                    base_pos(j, &w, &bit);
                    set_bits(unit, r, w, bit, codes[m * K + (size_t)g * GROUP + j] & 3u);
                }
                uint16_t s = scales[m * G + g];
                unit[4096 + 2 * r] = (uint8_t)s;
                unit[4096 + 2 * r + 1] = (uint8_t)(s >> 8);
            }
        }
}

void ref_unpack_base(const uint8_t* packed, int M, int K, uint8_t* codes, uint16_t* scales) {
    int G = K / GROUP;
    size_t ub = ref_base_unit_bytes();
    for (size_t t = 0; t < n_tiles(M); ++t)
        for (int g = 0; g < G; ++g) {
            const uint8_t* unit = packed + (t * G + g) * ub;
            for (int r = 0; r < ROWS; ++r) {
                size_t m = t * ROWS + r;
                if (m >= (size_t)M) continue;
                for (int j = 0; j < GROUP; ++j) {
                    int w, bit;
                    base_pos(j, &w, &bit);
                    codes[m * K + (size_t)g * GROUP + j] = (uint8_t)get_bits(unit, r, w, bit, 3u);
                }
                scales[m * G + g] = (uint16_t)(unit[4096 + 2 * r] | (unit[4096 + 2 * r + 1] << 8));
            }
        }
}

/* store or load the residual value u of column j of row r */
static void resid_put(uint8_t* unit, int r, int j, int bits, uint32_t u) {
    if (bits == 8) {
        set_bits(unit, r, j / 4, 8 * (j % 4), u);
        return;
    }
    int j8 = j % 8, j16 = j % 16, j32 = j % 32;
    set_bits(unit, r, j / 8, 8 * (j8 % 4) + 4 * (j8 / 4), u & 15u);
    set_bits(unit, r, 16 + j / 16, 8 * (j16 % 4) + 2 * (j16 / 4), (u >> 4) & 3u);
    if (bits == 7)
        set_bits(unit, r, 24 + j / 32, 8 * (j32 % 4) + j32 / 4, (u >> 6) & 1u);
}

static uint32_t resid_get(const uint8_t* unit, int r, int j, int bits) {
    if (bits == 8) return get_bits(unit, r, j / 4, 8 * (j % 4), 255u);
    int j8 = j % 8, j16 = j % 16, j32 = j % 32;
    uint32_t u = get_bits(unit, r, j / 8, 8 * (j8 % 4) + 4 * (j8 / 4), 15u);
    u |= get_bits(unit, r, 16 + j / 16, 8 * (j16 % 4) + 2 * (j16 / 4), 3u) << 4;
    if (bits == 7) u |= get_bits(unit, r, 24 + j / 32, 8 * (j32 % 4) + j32 / 4, 1u) << 6;
    return u;
}

int ref_pack_resid(const int8_t* codes, const uint16_t* scales, int M, int K, int bits, uint8_t* out) {
    if (bits < 6 || bits > 8) return 1;
    int G = K / GROUP;
    int off = 1 << (bits - 1);
    size_t ub = ref_resid_unit_bytes(bits);
    memset(out, 0, ref_resid_bytes(M, K, bits));
    for (size_t t = 0; t < n_tiles(M); ++t)
        for (int g = 0; g < G; ++g) {
            uint8_t* unit = out + (t * G + g) * ub;
            for (int r = 0; r < ROWS; ++r) {
                size_t m = t * ROWS + r;
                int valid = m < (size_t)M;
                for (int j = 0; j < GROUP; ++j) {
                    int q = valid ? codes[m * K + (size_t)g * GROUP + j] : 0;
                    resid_put(unit, r, j, bits, (uint32_t)(q + off));
                }
                uint16_t s = valid ? scales[m * G + g] : 0;
                unit[2048 * bits + 2 * r] = (uint8_t)s;
                unit[2048 * bits + 2 * r + 1] = (uint8_t)(s >> 8);
            }
        }
    return 0;
}

int ref_unpack_resid(const uint8_t* packed, int M, int K, int bits, int8_t* codes, uint16_t* scales) {
    if (bits < 6 || bits > 8) return 1;
    int G = K / GROUP;
    int off = 1 << (bits - 1);
    size_t ub = ref_resid_unit_bytes(bits);
    for (size_t t = 0; t < n_tiles(M); ++t)
        for (int g = 0; g < G; ++g) {
            const uint8_t* unit = packed + (t * G + g) * ub;
            for (int r = 0; r < ROWS; ++r) {
                size_t m = t * ROWS + r;
                if (m >= (size_t)M) continue;
                for (int j = 0; j < GROUP; ++j)
                    codes[m * K + (size_t)g * GROUP + j] = (int8_t)((int)resid_get(unit, r, j, bits) - off);
                scales[m * G + g] = (uint16_t)(unit[2048 * bits + 2 * r] | (unit[2048 * bits + 2 * r + 1] << 8));
            }
        }
    return 0;
}

/*
 * BitNest W4/W8 dual-plane storage (BitNest paper, Section 3.3: the base and the
 * refinement codes in two independently packed 4-bit planes, N/2 bytes each for
 * N weights, the refinement without scale metadata).  Same unit grid as above.
 *
 * W4 base unit (8448 bytes), stored value u4 = q4 + 8 (0..15):
 *   bytes [0, 8192): a row's 64 bytes as 16 words, chunk-major (word w of row r at
 *                    byte ((w/4)*128 + r)*16 + (w%4)*4); word w holds columns
 *                    8w..8w+7, column 8w + 4h + q in bits 8q + 4h .. 8q + 4h + 3.
 *   bytes [8192, 8448): fp16 s4 of row r at 8192 + 2r.
 * Refinement unit (8192 bytes): the same nibble layout with u_r = q_r + 8.
 * Rows past M hold q4 = q_r = 0 and scale 0.
 */
size_t ref_w4_unit_bytes(void) { return 8192 + 256; }
size_t ref_w4ref_unit_bytes(void) { return 8192; }

size_t ref_w4_bytes(int M, int K) { return n_tiles(M) * (size_t)(K / GROUP) * ref_w4_unit_bytes(); }
size_t ref_w4ref_bytes(int M, int K) { return n_tiles(M) * (size_t)(K / GROUP) * ref_w4ref_unit_bytes(); }

static void nib_put(uint8_t* unit, int r, int j, uint32_t u) {
    int j8 = j % 8;
    set_bits(unit, r, j / 8, 8 * (j8 % 4) + 4 * (j8 / 4), u & 15u);
}

static uint32_t nib_get(const uint8_t* unit, int r, int j) {
    int j8 = j % 8;
    return get_bits(unit, r, j / 8, 8 * (j8 % 4) + 4 * (j8 / 4), 15u);
}

void ref_pack_w4w8(const int8_t* q4, const uint16_t* s4, const int8_t* qr, int M, int K,
                   uint8_t* base_out, uint8_t* ref_out) {
    int G = K / GROUP;
    memset(base_out, 0, ref_w4_bytes(M, K));
    if (ref_out) memset(ref_out, 0, ref_w4ref_bytes(M, K));
    for (size_t t = 0; t < n_tiles(M); ++t)
        for (int g = 0; g < G; ++g) {
            uint8_t* bu = base_out + (t * G + g) * ref_w4_unit_bytes();
            uint8_t* ru = ref_out ? ref_out + (t * G + g) * ref_w4ref_unit_bytes() : NULL;
            for (int r = 0; r < ROWS; ++r) {
                size_t m = t * ROWS + r;
                int valid = m < (size_t)M;
                for (int j = 0; j < GROUP; ++j) {
                    size_t i = m * K + (size_t)g * GROUP + j;
                    nib_put(bu, r, j, (uint32_t)((valid ? q4[i] : 0) + 8));
                    if (ru) nib_put(ru, r, j, (uint32_t)((valid ? qr[i] : 0) + 8));
                }
                uint16_t s = valid ? s4[m * G + g] : 0;
                bu[8192 + 2 * r] = (uint8_t)s;
                bu[8192 + 2 * r + 1] = (uint8_t)(s >> 8);
            }
        }
}

void ref_unpack_w4w8(const uint8_t* base, const uint8_t* ref, int M, int K, int8_t* q4, uint16_t* s4, int8_t* qr) {
    int G = K / GROUP;
    for (size_t t = 0; t < n_tiles(M); ++t)
        for (int g = 0; g < G; ++g) {
            const uint8_t* bu = base + (t * G + g) * ref_w4_unit_bytes();
            const uint8_t* ru = ref ? ref + (t * G + g) * ref_w4ref_unit_bytes() : NULL;
            for (int r = 0; r < ROWS; ++r) {
                size_t m = t * ROWS + r;
                if (m >= (size_t)M) continue;
                for (int j = 0; j < GROUP; ++j) {
                    size_t i = m * K + (size_t)g * GROUP + j;
                    q4[i] = (int8_t)((int)nib_get(bu, r, j) - 8);
                    if (ru) qr[i] = (int8_t)((int)nib_get(ru, r, j) - 8);
                }
                s4[m * G + g] = (uint16_t)(bu[8192 + 2 * r] | (bu[8192 + 2 * r + 1] << 8));
            }
        }
}
