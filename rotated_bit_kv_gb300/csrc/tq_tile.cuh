// The 16-token tile layout of the packed cache (the caches the tensor-core decode
// kernel reads: every format without mixed-rate keys, at most 8 query heads per
// KV head).  Shared by the write kernels (which scatter each token's codes into
// it) and the decode kernel (which reads whole tiles).  The layout is documented
// for users in include/tq.h; the code values themselves are those of the packed
// record ([TQ-MNN] §3.3: 3-bit indices eight per three bytes, 4-bit two per byte).
//
// A tile holds 16 consecutive positions of one (batch, KV head).  Its codes are
// 32 "lane" pieces L = 4 r + c (r = 0..7, c = 0..3) of 2W words (W = 3 for 3-bit,
// 4 for 4-bit codes): words 0..3 of lane L at byte 16 L, words 4 .. 2W-1 at byte
// 512 + 8 (W - 2) L.  A "field" is the pair of codes of coordinates (2i, 2i+1)
// (3-bit: low code in bits 0-2, high in 3-5; 4-bit: low nibble, high nibble).
//
//   Keys:   words 0..W-1 of lane L hold token r, words W..2W-1 token r + 8; the
//           W words of a token in lane L hold the 16 fields of pairs
//           i = 8 (s >> 1) + c + 4 (s & 1), s = 0..15.
//   Values: words 0..W-1 hold tokens 2c (low 16-bit halves) and 2c + 1 (high
//           halves), words W..2W-1 tokens 2c + 8 and 2c + 9; the three or four
//           halves of a token in lane L hold the 8 fields of pairs
//           16 (q >> 1) + r + 8 (q & 1), q = 0..7.
//
// Inside a token's words the fields sit in bytes.  4-bit: field s of a key is byte
// s & 3 of word s >> 2; field q of a value is byte q & 1 of half q >> 1.  3-bit:
// 12 (key) or 6 (value) fields have a byte of their own, the last 4 (key) or 2
// (value) are spread over two-bit pieces of the bytes of the token's three words:
//   word 0 and 2 bytes: field bits 0-5 in byte bits 0-5; word 1 bytes: field
//   bits 0-1 in byte bits 0-1, field bits 2-5 in byte bits 4-7;
//   spread field number g (byte lane g of the three words): bits 0-1 in bits 6-7
//   of the word-0 byte, bits 2-3 in bits 2-3 of the word-1 byte, bits 4-5 in bits
//   6-7 of the word-2 byte.
// Keys: fields 0..11 in byte (s & 3) of word (s >> 2), fields 12..15 spread over
// byte lanes 0..3.  Values: fields q = 0..5 in byte lane (q & 1) of word (q >> 1),
// fields 6, 7 spread over byte lanes 0, 1 (of the token's 16-bit halves).
//
// Norms (one tile = 16 tokens x slots): one slot: token t at 2 (t & 7) + (t >> 3);
// four slots, keys: (2 (t & 7) + (t >> 3)) * 4 + b; values:
// ((((t & 7) >> 1) * 2 + (t >> 3)) * 4 + b) * 2 + (t & 1).
#pragma once
#include <stdint.h>

namespace tqtile {

constexpr int kTok = 16;

__host__ __device__ constexpr int group_words(int bits) { return bits == 3 ? 3 : 4; }
__host__ __device__ constexpr int tile_bytes(int bits) { return bits == 3 ? 768 : 1024; }

// byte offset of word i (0 .. 2W-1) of lane L within a code tile
__host__ __device__ constexpr int word_off(int bits, int L, int i) {
    return i < 4 ? 16 * L + 4 * i : 512 + 8 * (group_words(bits) - 2) * L + 4 * (i - 4);
}

// coordinate pair of key field s held by lane column c, and of value field q
// held by lane row r
__host__ __device__ constexpr int k_pair(int c, int s) { return 8 * (s >> 1) + c + 4 * (s & 1); }
__host__ __device__ constexpr int v_pair(int r, int q) { return 16 * (q >> 1) + r + 8 * (q & 1); }

// norm element positions within a tile's norms
__host__ __device__ constexpr int norm_pos1(int t) { return 2 * (t & 7) + (t >> 3); }
__host__ __device__ constexpr int norm_pos4_k(int t, int b) { return (2 * (t & 7) + (t >> 3)) * 4 + b; }
__host__ __device__ constexpr int norm_pos4_v(int t, int b) {
    return ((((t & 7) >> 1) * 2 + (t >> 3)) * 4 + b) * 2 + (t & 1);
}

// positions per (batch, KV head): the capacity rounded up to whole tiles
__host__ __device__ constexpr long long alloc_tokens(long long cap) { return (cap + kTok - 1) / kTok * kTok; }

#ifdef __CUDACC__
// ---- write side: the tile words of one token from its packed record (held as
// 32-bit little-endian words, LSB-first codes)

// 6-bit field of pair i of a 3-bit record
__device__ __forceinline__ uint32_t rec_field3(const uint32_t* rec, int i) {
    const int bit = 6 * i, w = bit >> 5, sh = bit & 31;
    const uint32_t v = sh <= 26 ? rec[w] >> sh : __funnelshift_r(rec[w], rec[w + 1], sh);
    return v & 63u;
}
// byte j of a 4-bit record (the field of pair j)
__device__ __forceinline__ uint32_t rec_byte(const uint32_t* rec, int j) { return (rec[j >> 2] >> (8 * (j & 3))) & 255u; }

// a 3-bit field in the byte of word w, and the piece of a spread field in it
__device__ __forceinline__ uint32_t byte3(uint32_t f, int w) { return w == 1 ? (f & 3u) | ((f & 0x3Cu) << 2) : f; }
__device__ __forceinline__ uint32_t piece3(uint32_t F, int w) {
    return w == 0 ? (F & 3u) << 6 : w == 1 ? ((F >> 2) & 3u) << 2 : ((F >> 4) & 3u) << 6;
}

// key word w (0 .. W-1) of a token for lane column c
template <int BITS>
__device__ __forceinline__ uint32_t key_word(const uint32_t* rec, int c, int w) {
    uint32_t x = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        uint32_t b;
        if constexpr (BITS == 3)
            b = byte3(rec_field3(rec, k_pair(c, 4 * w + k)), w) | piece3(rec_field3(rec, k_pair(c, 12 + k)), w);
        else
            b = rec_byte(rec, k_pair(c, 4 * w + k));
        x |= b << (8 * k);
    }
    return x;
}

// value half w (0 .. W-1) of a token for lane row r
template <int BITS>
__device__ __forceinline__ uint32_t value_half(const uint32_t* rec, int r, int w) {
    uint32_t x = 0;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        uint32_t b;
        if constexpr (BITS == 3)
            b = byte3(rec_field3(rec, v_pair(r, 2 * w + j)), w) | piece3(rec_field3(rec, v_pair(r, 6 + j)), w);
        else
            b = rec_byte(rec, v_pair(r, 2 * w + j));
        x |= b << (8 * j);
    }
    return x;
}

// Scatter the packed record `rec` (warp-visible memory) of the token at tile
// position t (0..15) into the key tile `tile`: lanes 0 .. 4W-1 write one word each.
template <int BITS>
__device__ __forceinline__ void store_key(uint8_t* tile, const uint32_t* rec, int t, int lane) {
    constexpr int W = group_words(BITS);
    if (lane < 4 * W) {
        const int c = lane / W, w = lane - c * W;
        const uint32_t x = key_word<BITS>(rec, c, w);
        *reinterpret_cast<uint32_t*>(tile + word_off(BITS, 4 * (t & 7) + c, W * (t >> 3) + w)) = x;
    }
}

// ... and into the value tile: lanes 0 .. 8W-1 write one 16-bit half each.
template <int BITS>
__device__ __forceinline__ void store_value(uint8_t* tile, const uint32_t* rec, int t, int lane) {
    constexpr int W = group_words(BITS);
    if (lane < 8 * W) {
        const int r = lane / W, w = lane - r * W;
        const uint32_t x = value_half<BITS>(rec, r, w);
        *reinterpret_cast<uint16_t*>(tile + word_off(BITS, 4 * r + ((t & 7) >> 1), W * (t >> 3) + w) + 2 * (t & 1)) =
            (uint16_t)x;
    }
}
#endif

}  // namespace tqtile
