// nwc_format.h -- layout constants of the NWC blob shared by the library's host code and
// kernels (not by the CPU oracle, which restates the format on its own).
//
// Layout (little-endian): 64-byte header, 16-byte rank table, u32 block table (16-byte units
// from the data section), fp32 row scales (fp8 only), then one region per 8x512 block in
// row-block-major order: u8 lane_words[32] | 32 code streams (u32 words, most significant bit
// first) | zero pad to 16 B | 32 mantissa regions (even-t half-stream in the low halves, odd-t
// half-stream in the high halves, F-bit fields least significant bit first, 16-byte multiple;
// when all lanes have the same word count W, word k of lane l is word 32k + l of the section,
// otherwise the regions follow one another) |
// escape list (u32 t | lane << 7 | element bits << 12 per escaped element, lanes in order, t
// increasing, padded to 16 B with kEscPad). An escape code in a lane stream is n_ranked ones and
// the sign; the escaped element's exponent (with the rest of its bits) is in the list.
#pragma once
#include <stdint.h>

#if defined(__CUDACC__)
#define NWC_HD __host__ __device__ __forceinline__
#else
#define NWC_HD inline
#endif

namespace nwcf {

constexpr uint32_t kMagic = 0x3143574Eu;  // "NWC1"
constexpr uint32_t kVersion = 3;
constexpr int kRows = 8, kCols = 512, kLanes = 32, kLaneCols = 16, kSyms = 128;
constexpr int kMaxRanked = 11;
constexpr int kMaxLaneWords = 48;  // 128 codes x 12 bits / 32
constexpr uint32_t kEscPad = 0xFFFFFFFFu;
constexpr uint64_t kHeaderBytes = 64, kRankOff = 64, kBlockTabOff = 80;

// header field offsets
constexpr int H_MAGIC = 0, H_VERSION = 4, H_ELEM = 6, H_NR = 7, H_N = 8, H_K = 16, H_NB = 24,
              H_OFF_BLOCKS = 32, H_OFF_SCALES = 40, H_OFF_DATA = 48, H_TOTAL = 56;

NWC_HD int exp_bits(int elem) { return elem == 0 ? 8 : 4; }
NWC_HD int man_bits(int elem) { return elem == 0 ? 7 : 3; }
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
// Mantissa region words of a lane: even-t elements are rows 0,2,4,6.
NWC_HD uint32_t man_words(int rows, int cols, int F) {
    uint32_t n_even = (uint32_t)cols * (uint32_t)((rows + 1) / 2);
    uint32_t half_words = (uint32_t)cdiv((uint64_t)F * n_even, 16);
    return (uint32_t)(cdiv(half_words, 4) * 4);
}

// Escape-list entry fields.
NWC_HD uint32_t esc_entry(uint32_t t, uint32_t lane, uint32_t bits) { return t | (lane << 7) | (bits << 12); }
NWC_HD uint32_t esc_t(uint32_t e) { return e & 127u; }
NWC_HD uint32_t esc_lane(uint32_t e) { return (e >> 7) & 31u; }
NWC_HD uint32_t esc_bits(uint32_t e) { return e >> 12; }

}  // namespace nwcf
