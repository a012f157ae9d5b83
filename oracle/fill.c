/*
 * oracle/fill.c -- the producer's hashed values, element by element, in plain C.
 * TEST INFRASTRUCTURE ONLY: the CPU oracle (see oracle/__init__.py).  Neither the library nor
 * any product path links or calls this file; the tests load it through oracle/cfill.py.
 *
 * The same definition as oracle/hashfill.py, written out as scalar loops so that whole
 * full-size buffers can be checked byte for byte (numpy needs seconds per 32 MiB slice).  The
 * pages fix no value formula ("Triggered Plans", section Model: the producer "computes and
 * stores the tile"); this is the build's own definition:
 *   fmix32     MurmurHash3's 32-bit finaliser (Austin Appleby, public domain): xor-shift 16,
 *              multiply 0x85EBCA6B, xor-shift 13, multiply 0xC2B2AE35, xor-shift 16;
 *   salt       fmix32(seed ^ fmix32(rank ^ fmix32(round)));
 *   h          fmix32(((row * N + col) mod 2^32) ^ salt), row local to the rank's slice;
 *   u          ((h >> 8) - 2^23) * 2^-23, an exact float in [-1, 1);
 *   bf16       u rounded to nearest, ties to even, by bit arithmetic; f32 keeps u; u8 = h & 0xFF.
 * Bytes are written little-endian with shifts, whatever the host's byte order.
 */
#include <stdint.h>
#include <string.h>

enum { ORACLE_BF16 = 0, ORACLE_F32 = 1, ORACLE_U8 = 2 };

static uint32_t fmix32(uint32_t h) {
    h ^= h >> 16;
    h *= 0x85EBCA6Bu;
    h ^= h >> 13;
    h *= 0xC2B2AE35u;
    h ^= h >> 16;
    return h;
}

static uint32_t salt_of(uint32_t seed, uint32_t rank, uint32_t round) {
    return fmix32(seed ^ fmix32(rank ^ fmix32(round)));
}

/* The uniform value as float32 bits: k = (h >> 8) - 2^23 has |k| <= 2^23, so (float)k is exact,
 * and so is the product with the power of two 2^-23. */
static uint32_t uniform_bits(uint32_t h) {
    const int32_t k = (int32_t)(h >> 8) - (int32_t)(1 << 23);
    const float u = (float)k * (1.0f / 8388608.0f);
    uint32_t b;
    memcpy(&b, &u, sizeof b);
    return b;
}

/* float32 bits -> bfloat16 bits, round to nearest, ties to even (finite inputs). */
static uint32_t bf16_of(uint32_t b) {
    const uint32_t lsb = (b >> 16) & 1u;
    return ((b + 0x7FFFu + lsb) >> 16) & 0xFFFFu;
}

uint32_t oracle_fmix32(uint32_t h) { return fmix32(h); }
uint32_t oracle_salt(uint32_t seed, uint32_t rank, uint32_t round) { return salt_of(seed, rank, round); }
uint32_t oracle_uniform_bits(uint32_t h) { return uniform_bits(h); }
uint32_t oracle_bf16_bits(uint32_t f32_bits) { return bf16_of(f32_bits); }

/* Rows [row0, row1) of rank `rank`'s M x N slice in round `round`, as raw bytes at `out`
 * ((row1 - row0) * N * element bytes).  Returns 0, or -1 for an unknown dtype. */
int oracle_fill_rows(int dtype, uint32_t seed, uint32_t rank, uint32_t round, uint64_t N,
                     uint64_t row0, uint64_t row1, uint8_t* out) {
    if (dtype != ORACLE_BF16 && dtype != ORACLE_F32 && dtype != ORACLE_U8) return -1;
    const uint32_t salt = salt_of(seed, rank, round);
    uint64_t o = 0;
    for (uint64_t row = row0; row < row1; ++row) {
        for (uint64_t col = 0; col < N; ++col) {
            const uint32_t idx = (uint32_t)(row * N + col);   /* mod 2^32 */
            const uint32_t h = fmix32(idx ^ salt);
            if (dtype == ORACLE_U8) {
                out[o++] = (uint8_t)(h & 0xFFu);
            } else if (dtype == ORACLE_F32) {
                const uint32_t b = uniform_bits(h);
                out[o++] = (uint8_t)(b & 0xFFu);
                out[o++] = (uint8_t)((b >> 8) & 0xFFu);
                out[o++] = (uint8_t)((b >> 16) & 0xFFu);
                out[o++] = (uint8_t)(b >> 24);
            } else {
                const uint32_t b = bf16_of(uniform_bits(h));
                out[o++] = (uint8_t)(b & 0xFFu);
                out[o++] = (uint8_t)(b >> 8);
            }
        }
    }
    return 0;
}
