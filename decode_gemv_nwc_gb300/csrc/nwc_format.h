// nwc_format.h -- layout constants of the NWC blob shared by the library's host code and
// kernels (not by the CPU oracle, which restates the format on its own).
//
// Layout (little-endian): 64-byte header, 16-byte rank table, u32 block table (16-byte units
// from the data section), fp32 row scales (fp8 only), then one region per 8x512 block in
// row-block-major order:
//   u8 lane_words[32] | 32 code streams (u32 words, most significant bit first) | zero pad to
//   16 B | raw section | escape list (u32 t | lane << 7 | v << 12 per listed element, lanes in
//   order, t increasing, padded to 16 B with kEscPad).
// A lane's stream holds its 64 row pairs (rows 2i, 2i+1 of column c = j / 4, i = j % 4, for
// pair j): each element's code is its exponent's unary rank code (rank p: p ones and a zero;
// an unranked exponent: n_ranked ones; a filler: the rank-0 code), and a pair whose two codes
// exceed kPeek bits keeps the first code followed by ones up to kPeek bits, its second element
// being listed. The sign and the mantissa are raw: a byte s << 7 | m per BF16 element, a
// nibble s << 3 | m per fp8 element. Raw section of a block whose 512 columns lie inside K:
// 16-byte unit u of lane l at 16 (32 u + l); BF16 units hold columns 2u, 2u + 1 (a byte per
// row), fp8 units columns 4u .. 4u + 3 (a byte per row pair, the even row in the low nibble).
// Other blocks: each lane's real columns in order (8, resp. 4, bytes a column), padded to 16
// bytes, the lanes one after another. Rows past N hold zero raw bits.
#pragma once
#include <stdint.h>

#if defined(__CUDACC__)
#define NWC_HD __host__ __device__ __forceinline__
#else
#define NWC_HD inline
#endif

namespace nwcf {

constexpr uint32_t kMagic = 0x3143574Eu;  // "NWC1"
constexpr uint32_t kVersion = 4;
constexpr int kRows = 8, kCols = 512, kLanes = 32, kLaneCols = 16, kSyms = 128, kPairs = 64;
constexpr int kMaxRanked = 12;
constexpr int kPeek = 13;          // bits of one table lookup; a pair's codes never exceed it
constexpr int kMaxLaneWords = 26;  // 64 pairs x 13 bits / 32, rounded up
constexpr uint32_t kEscPad = 0xFFFFFFFFu;
constexpr uint64_t kHeaderBytes = 64, kRankOff = 64, kBlockTabOff = 80;

// header field offsets
constexpr int H_MAGIC = 0, H_VERSION = 4, H_ELEM = 6, H_NR = 7, H_N = 8, H_K = 16, H_NB = 24,
              H_OFF_BLOCKS = 32, H_OFF_SCALES = 40, H_OFF_DATA = 48, H_TOTAL = 56;

NWC_HD int exp_bits(int elem) { return elem == 0 ? 8 : 4; }
NWC_HD uint64_t cdiv(uint64_t a, uint64_t b) { return (a + b - 1) / b; }
NWC_HD uint64_t up16(uint64_t a) { return (a + 15) & ~uint64_t(15); }

// Real rows / columns covered by lane l of block (rb, cb).
NWC_HD int real_rows(uint64_t n, uint64_t rb) {
    uint64_t r0 = rb * kRows;
    return r0 >= n ? 0 : (n - r0 >= (uint64_t)kRows ? kRows : (int)(n - r0));
}
NWC_HD int real_cols(uint64_t k, uint64_t cb, int lane) {
    uint64_t c0 = cb * kCols + (uint64_t)lane * kLaneCols;
    return c0 >= k ? 0 : (k - c0 >= (uint64_t)kLaneCols ? kLaneCols : (int)(k - c0));
}
// Raw bytes per column (8 rows): a byte per BF16 element, a nibble per fp8 element.
NWC_HD uint32_t col_bytes(int elem) { return elem == 0 ? 8u : 4u; }
// A block whose columns all lie inside K has the interleaved (full) raw layout.
NWC_HD bool raw_full(uint64_t k, uint64_t cb) { return (cb + 1) * (uint64_t)kCols <= k; }
// Bytes of lane l's raw region in a block without the full layout.
NWC_HD uint32_t lane_raw_bytes(uint64_t k, uint64_t cb, int lane, int elem) {
    return (uint32_t)up16((uint64_t)real_cols(k, cb, lane) * col_bytes(elem));
}
// Bytes of a block's raw section.
NWC_HD uint32_t raw_section_bytes(uint64_t k, uint64_t cb, int elem) {
    if (raw_full(k, cb)) return (uint32_t)(kLanes * kLaneCols) * col_bytes(elem);
    uint32_t s = 0;
    for (int l = 0; l < kLanes; l++) s += lane_raw_bytes(k, cb, l, elem);
    return s;
}

// Escape-list entry fields.
NWC_HD uint32_t esc_entry(uint32_t t, uint32_t lane, uint32_t v) { return t | (lane << 7) | (v << 12); }
NWC_HD uint32_t esc_t(uint32_t e) { return e & 127u; }
NWC_HD uint32_t esc_lane(uint32_t e) { return (e >> 7) & 31u; }
NWC_HD uint32_t esc_v(uint32_t e) { return e >> 12; }

// Leading one-bits of x.
NWC_HD int lead_ones(uint32_t x) {
#if defined(__CUDA_ARCH__)
    return __clz(~x);
#else
    return ~x == 0u ? 32 : __builtin_clz(~x);
#endif
}

// Exponent field that the decoders place for exponent value v: BF16 the value itself; fp8
// the exponent of the same number as a BF16 (v + 120; 0 stays 0, exact for zeros, and the
// subnormal and NaN codes are listed).
NWC_HD uint32_t bf16_exp_field(int elem, uint32_t v) { return elem == 0 ? v : (v ? v + 120u : 0u); }

// Decode-table entry for a kPeek-bit peek p (first stream bit = bit kPeek - 1): the row pair
// that the peek holds. Bits 0..4 the pair's length in bits, bits 7..14 the first element's
// exponent field as a BF16 high part (escape or cut: 0, the placeholder that the escape list
// corrects), bits 23..30 the second element's, bits 16..17 the number of the pair's elements
// that the escape list must hold (an escape code, or the tail of a cut pair); all other bits
// zero (bits 5..6 are zero so that whole entries can be subtracted from a bit counter).
// First code: leading ones up to nr (nr ones: an escape, no terminating zero), else the count
// and a zero. Second code: the same on the rest of the peek, except that ones running to the
// end of the peek before nr of them are the tail of a cut pair.
NWC_HD uint32_t table_entry(uint32_t p, int nr, int elem, const uint8_t *rank_exp) {
    const uint32_t bits = p << (32 - kPeek);
    const int a = lead_ones(bits);
    uint32_t e1, len1, nesc = 0;
    if (a >= nr) {
        e1 = 0;
        len1 = (uint32_t)nr;
        nesc++;
    } else {
        e1 = bf16_exp_field(elem, rank_exp[a]);
        len1 = (uint32_t)a + 1u;
    }
    const uint32_t rest = (uint32_t)kPeek - len1;
    const int b = lead_ones(bits << len1);
    uint32_t e2, len2;
    if (b >= nr) {
        e2 = 0;
        len2 = (uint32_t)nr;
        nesc++;
    } else if ((uint32_t)b < rest) {
        e2 = bf16_exp_field(elem, rank_exp[b]);
        len2 = (uint32_t)b + 1u;
    } else {
        e2 = 0;
        len2 = rest;
        nesc++;
    }
    return (len1 + len2) | (e1 << 7) | (nesc << 16) | (e2 << 23);
}

}  // namespace nwcf
