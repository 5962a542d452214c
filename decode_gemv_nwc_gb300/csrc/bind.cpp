// bind.cpp -- host-side validation of an NWC blob and binding of its device copy.
//
// Validation covers everything the kernels trust without checking: header fields, the rank
// table (exponents ranked by frequency, at most 12 ranked values), the block table, each
// block region's size, which must equal its 32 lane code streams (at most 26 words each: 64
// row pairs of at most 13 bits) plus the raw section implied by the block's real columns
// (fillers past K carry no raw bits, as the "How it works" section of "NWC -- Neural Weight
// Compression" states for padding) plus its escape list, and the escape list itself: every
// entry names a real element of the block, in (lane, t) order without repeats, with an
// exponent field of the element's width, followed by fewer than four padding words.
// Lane stream contents are checked on the device while decoding.
#include <cstring>
#include <string>

#include "nwc.h"
#include "nwc_format.h"

using namespace nwcf;

namespace {

inline uint64_t rd64(const uint8_t *p) {
    uint64_t v;
    std::memcpy(&v, p, 8);
    return v;
}
inline uint32_t rd32(const uint8_t *p) {
    uint32_t v;
    std::memcpy(&v, p, 4);
    return v;
}

struct Parsed {
    int elem, nr;
    uint64_t n, k, rb, cb, nb, off_blocks, off_scales, off_data, total, max_block, data_bytes;
    uint8_t rank_exp[16];
};

nwc_status parse_and_check(const uint8_t *b, uint64_t bytes, Parsed &p) {
    if (!b || bytes < kBlockTabOff + 8) return NWC_ERR_FORMAT;
    if (rd32(b + H_MAGIC) != kMagic || b[H_VERSION] != kVersion || b[H_VERSION + 1] != 0)
        return NWC_ERR_FORMAT;
    p.elem = b[H_ELEM];
    p.nr = b[H_NR];
    p.n = rd64(b + H_N);
    p.k = rd64(b + H_K);
    p.nb = rd64(b + H_NB);
    p.off_blocks = rd64(b + H_OFF_BLOCKS);
    p.off_scales = rd64(b + H_OFF_SCALES);
    p.off_data = rd64(b + H_OFF_DATA);
    p.total = rd64(b + H_TOTAL);
    if (p.elem != NWC_ELEM_BF16 && p.elem != NWC_ELEM_FP8_E4M3) return NWC_ERR_FORMAT;
    if (p.nr < 1 || p.nr > kMaxRanked) return NWC_ERR_FORMAT;
    if (p.n == 0 || p.k == 0 || p.n >= (1ull << 40) || p.k >= (1ull << 40)) return NWC_ERR_FORMAT;
    p.rb = cdiv(p.n, kRows);
    p.cb = cdiv(p.k, kCols);
    // the block count must stay below 2^31; checked before the product so that it cannot wrap
    if (p.rb > ((1ull << 31) - 1) / p.cb) return NWC_ERR_FORMAT;
    if (p.nb != p.rb * p.cb || p.nb >= (1ull << 31)) return NWC_ERR_FORMAT;
    if (p.total != bytes || p.off_blocks != kBlockTabOff) return NWC_ERR_FORMAT;
    const uint64_t tab_end = p.off_blocks + 4 * (p.nb + 1);
    if (tab_end > bytes) return NWC_ERR_FORMAT;
    if (p.elem == NWC_ELEM_FP8_E4M3) {
        if (p.off_scales != up16(tab_end) || p.off_data != up16(p.off_scales + 4 * p.n)) return NWC_ERR_FORMAT;
    } else if (p.off_scales != 0 || p.off_data != up16(tab_end)) {
        return NWC_ERR_FORMAT;
    }
    if (p.off_data > bytes) return NWC_ERR_FORMAT;
    std::memcpy(p.rank_exp, b + kRankOff, 16);
    const int nv = 1 << exp_bits(p.elem);
    bool seen[256] = {false};
    for (int i = 0; i < p.nr; i++) {
        int v = p.rank_exp[i];
        if (v >= nv || seen[v]) return NWC_ERR_FORMAT;
        seen[v] = true;
    }
    for (int i = p.nr; i < 16; i++)
        if (p.rank_exp[i] != 0) return NWC_ERR_FORMAT;
    const uint8_t *tab = b + p.off_blocks;
    if (rd32(tab) != 0) return NWC_ERR_FORMAT;
    if (p.off_data + 16 * (uint64_t)rd32(tab + 4 * p.nb) != bytes) return NWC_ERR_FORMAT;
    const int eb = exp_bits(p.elem);
    p.max_block = 0;
    for (uint64_t i = 0; i < p.nb; i++) {
        uint64_t s = rd32(tab + 4 * i), e = rd32(tab + 4 * (i + 1));
        if (e < s) return NWC_ERR_FORMAT;
        uint64_t start = p.off_data + 16 * s, len = 16 * (e - s);
        if (len < 32 || start + len > bytes) return NWC_ERR_FORMAT;
        const uint8_t *lw = b + start;
        uint64_t rb = i / p.cb, cb = i % p.cb, words = 0;
        int rows = real_rows(p.n, rb);
        for (int l = 0; l < kLanes; l++) {
            if (lw[l] > kMaxLaneWords) return NWC_ERR_FORMAT;
            words += lw[l];
        }
        const uint64_t esc_off = up16(32 + 4 * words) + raw_section_bytes(p.k, cb, p.elem);
        if (esc_off > len) return NWC_ERR_FORMAT;
        const uint64_t slots = (len - esc_off) / 4;
        int64_t last = -1;
        uint64_t entries = 0;
        for (uint64_t j = 0; j < slots; j++) {
            const uint32_t e = rd32(lw + esc_off + 4 * j);
            if (e == kEscPad) continue;
            if (entries != j) return NWC_ERR_FORMAT;  // an entry after padding
            const int64_t key = (int64_t)esc_lane(e) * kSyms + esc_t(e);
            if (key <= last) return NWC_ERR_FORMAT;
            last = key;
            const int t = (int)esc_t(e);
            if (t % kRows >= rows || t / kRows >= real_cols(p.k, cb, (int)esc_lane(e))) return NWC_ERR_FORMAT;
            if (esc_v(e) >> eb) return NWC_ERR_FORMAT;  // exponent field wider than the element's
            entries++;
        }
        if (slots - entries > 3) return NWC_ERR_FORMAT;
        if (len > p.max_block) p.max_block = len;
    }
    p.data_bytes = bytes - p.off_data;
    return NWC_OK;
}

}  // namespace

extern "C" const char *nwc_status_str(nwc_status s) {
    switch (s) {
        case NWC_OK: return "ok";
        case NWC_ERR_INVALID_ARG: return "invalid argument";
        case NWC_ERR_FORMAT: return "malformed blob";
        case NWC_ERR_CUDA: return "CUDA error";
        case NWC_ERR_TIMEOUT: return "device wait timed out";
        case NWC_ERR_DEVICE_FLAG: return "device error flag raised";
        case NWC_ERR_UNSUPPORTED: return "unsupported";
        case NWC_ERR_IO: return "file could not be opened, read or written";
    }
    return "unknown status";
}

extern "C" const char *nwc_version(void) {
    static const std::string v = "nwc " + std::to_string(kVersion) + " (format " + std::to_string(kVersion) + ", sm_103a)";
    return v.c_str();
}

extern "C" nwc_status nwc_validate(const void *blob_host, size_t bytes) {
    Parsed p;
    return parse_and_check(static_cast<const uint8_t *>(blob_host), bytes, p);
}

extern "C" nwc_status nwc_bind(const void *blob_host, size_t bytes, const void *blob_dev, nwc_matrix *out) {
    if (!blob_host || !blob_dev || !out) return NWC_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(blob_dev) % 16) return NWC_ERR_INVALID_ARG;
    Parsed p;
    nwc_status st = parse_and_check(static_cast<const uint8_t *>(blob_host), bytes, p);
    if (st != NWC_OK) return st;
    const uint8_t *d = static_cast<const uint8_t *>(blob_dev);
    nwc_matrix m;
    std::memset(&m, 0, sizeof(m));
    m.elem = p.elem;
    m.n_ranked = p.nr;
    m.n = (int64_t)p.n;
    m.k = (int64_t)p.k;
    m.row_blocks = (int64_t)p.rb;
    m.col_blocks = (int64_t)p.cb;
    std::memcpy(m.rank_exp, p.rank_exp, 16);
    m.block_tab = reinterpret_cast<const uint32_t *>(d + p.off_blocks);
    m.data = d + p.off_data;
    m.scales = p.elem == NWC_ELEM_FP8_E4M3 ? reinterpret_cast<const float *>(d + p.off_scales) : nullptr;
    m.blob_bytes = p.total;
    m.max_block_bytes = p.max_block;
    m.data_bytes = p.data_bytes;
    *out = m;
    return NWC_OK;
}
