// encoder.cpp -- host encoder of the NWC blob and the fp8 e4m3 quantizer.
//
// "NWC -- Neural Weight Compression", section "How it works": a BF16 weight is split into a
// raw part and an entropy-coded exponent; the exponent is ranked by frequency and written as a
// unary rank code, the sign is a raw bit (kept here beside the raw mantissa, a byte per
// element), with an escape for rare values (n_ranked ones in the stream, the exponent in the
// block's escape list); a 12-bit peek yields up to two codes: here every row pair of a lane is
// written so that one 13-bit peek holds it (a longer pair keeps its first code and ones up to
// 13 bits, and its second element is listed); every lane of a block of 8 rows x 512 columns
// has its own bit stream; padding to any shape costs a one-bit code per filler weight and no
// raw bits past K.
// "Qwen3-4B-NWC-fp8": weight-only e4m3, symmetric per-output-channel scale, bytes coded
// losslessly with the same code (4-bit exponent; sign and 3-bit mantissa raw, a nibble). The
// subnormal and NaN codes are listed as well, so that the kernels can treat every other e4m3
// value as a BF16 pattern.
//
// Work is split over row-blocks across host threads. Pass 1 sizes every block region, pass 2
// writes each region at its prefix-summed offset, so the bytes do not depend on the thread
// count.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <thread>
#include <vector>

#include "nwc.h"
#include "nwc_format.h"

using namespace nwcf;

namespace {

struct Codebook {
    int elem = 0, nr = 0;
    uint32_t code[256];  // code bits of the exponent value, most significant bit first
    uint8_t len[256];    // code length
    uint8_t rank_exp[16];
    bool escaped[256];
};

// Ranking: values with a nonzero count, most frequent first, ties to the lower value;
// at most kMaxRanked of them get a unary code, the rest escape.
Codebook make_codebook(const uint64_t *hist, int elem) {
    Codebook cb;
    cb.elem = elem;
    const int nv = 1 << exp_bits(elem);
    std::vector<int> vals;
    for (int v = 0; v < nv; v++)
        if (hist[v]) vals.push_back(v);
    std::stable_sort(vals.begin(), vals.end(), [&](int a, int b) { return hist[a] > hist[b]; });
    cb.nr = std::min<int>((int)vals.size(), kMaxRanked);
    std::memset(cb.rank_exp, 0, sizeof(cb.rank_exp));
    for (int v = 0; v < nv; v++) {  // escape: nr ones
        cb.code[v] = (1u << cb.nr) - 1u;
        cb.len[v] = (uint8_t)cb.nr;
        cb.escaped[v] = true;
    }
    for (int p = 0; p < cb.nr; p++) {  // rank p: p ones, a zero
        const int v = vals[p];
        cb.rank_exp[p] = (uint8_t)v;
        cb.code[v] = ((1u << p) - 1u) << 1;
        cb.len[v] = (uint8_t)(p + 1);
        cb.escaped[v] = false;
    }
    return cb;
}

template <class E>
struct Src {
    const E *e;
    int64_t ld;
    uint64_t n, k;
    uint32_t at(uint64_t r, uint64_t c) const { return (uint32_t)e[r * (uint64_t)ld + c]; }
};

inline void fields(int elem, uint32_t x, uint32_t &s, uint32_t &v, uint32_t &m) {
    if (elem == 0) { s = x >> 15; v = (x >> 7) & 0xFF; m = x & 0x7F; }
    else { s = (x >> 7) & 1; v = (x >> 3) & 0xF; m = x & 7; }
}

// fp8 codes the kernels cannot treat as a rebiased BF16 pattern: subnormals and NaN.
inline bool fp8_listed(uint32_t v, uint32_t m) { return (v == 0 && m != 0) || (v == 15 && m == 7); }

// MSB-first bit sink into 32-bit words (out == nullptr: count only).
struct CodeSink {
    uint32_t *out;
    uint64_t acc = 0;
    int nacc = 0;
    uint32_t nw = 0;
    void put(uint32_t bits, int n) {
        acc = (acc << n) | bits;
        nacc += n;
        if (nacc >= 32) {
            nacc -= 32;
            const uint32_t w = (uint32_t)(acc >> nacc);
            if (out) out[nw] = w;
            nw++;
        }
    }
    void flush() {
        if (nacc > 0) {
            const uint32_t w = (uint32_t)(acc << (32 - nacc));
            if (out) out[nw] = w;
            nw++;
            nacc = 0;
        }
    }
};

// Lane l of block (rb, cbi): writes (or, with out == nullptr, counts) its code stream and
// appends its listed elements (t | lane << 7 | v << 12) to esc (when non-null). Returns the
// lane's word count; *n_list receives the number of listed elements.
template <class E>
uint32_t lane_stream(const Src<E> &src, const Codebook &cbk, uint64_t rb, uint64_t cbi, int l, uint32_t *out,
                     uint32_t *esc, uint32_t *n_list) {
    const int rows = real_rows(src.n, rb), cols = real_cols(src.k, cbi, l);
    CodeSink cs;
    cs.out = out;
    uint32_t listed = 0;
    for (int j = 0; j < kPairs; j++) {
        const int c = j >> 2, r0 = 2 * (j & 3);
        uint32_t code[2], v[2] = {0, 0};
        int len[2];
        bool real[2], lst[2] = {false, false};
        for (int h = 0; h < 2; h++) {
            real[h] = r0 + h < rows && c < cols;
            if (!real[h]) {  // filler: the rank-0 code, a zero bit
                code[h] = 0;
                len[h] = 1;
                continue;
            }
            uint32_t s, m;
            fields(cbk.elem, src.at(rb * kRows + r0 + h, cbi * kCols + (uint64_t)l * kLaneCols + c), s, v[h], m);
            code[h] = cbk.code[v[h]];
            len[h] = cbk.len[v[h]];
            lst[h] = cbk.escaped[v[h]] || (cbk.elem == 1 && fp8_listed(v[h], m));
        }
        cs.put(code[0], len[0]);
        if (len[0] + len[1] <= kPeek) {
            cs.put(code[1], len[1]);
        } else {  // the pair is cut: ones up to kPeek bits, the second element listed
            const int tail = kPeek - len[0];
            cs.put((1u << tail) - 1u, tail);
            lst[1] = real[1];
        }
        for (int h = 0; h < 2; h++)
            if (lst[h]) {
                if (esc) esc[listed] = esc_entry((uint32_t)(8 * c + r0 + h), (uint32_t)l, v[h]);
                listed++;
            }
    }
    cs.flush();
    *n_list = listed;
    return cs.nw;
}

// Size in bytes of block (rb, cb)'s region.
template <class E>
uint64_t block_size(const Src<E> &src, const Codebook &cbk, uint64_t rb, uint64_t cbi) {
    uint64_t code_words = 0, n_esc = 0;
    for (int l = 0; l < kLanes; l++) {
        uint32_t nl;
        code_words += lane_stream(src, cbk, rb, cbi, l, nullptr, nullptr, &nl);
        n_esc += nl;
    }
    return up16(32 + 4 * code_words) + raw_section_bytes(src.k, cbi, cbk.elem) + up16(4 * n_esc);
}

// Writes block (rb, cb)'s region of `size` bytes at dst (16-byte aligned, zeroed).
template <class E>
void write_block(const Src<E> &src, const Codebook &cbk, uint64_t rb, uint64_t cbi, uint8_t *dst, uint64_t size) {
    const int rows = real_rows(src.n, rb);
    uint32_t *words = reinterpret_cast<uint32_t *>(dst + 32);
    std::vector<uint32_t> esc;
    esc.reserve(kSyms);
    uint32_t pos = 0, lane_list[kSyms];
    for (int l = 0; l < kLanes; l++) {
        uint32_t nl;
        const uint32_t nw = lane_stream(src, cbk, rb, cbi, l, words + pos, lane_list, &nl);
        dst[l] = (uint8_t)nw;
        pos += nw;
        esc.insert(esc.end(), lane_list, lane_list + nl);
    }
    uint8_t *raw = dst + up16(32 + 4 * (uint64_t)pos);
    const bool full = raw_full(src.k, cbi);
    uint32_t lane_off = 0;
    for (int l = 0; l < kLanes; l++) {
        const int cols = real_cols(src.k, cbi, l);
        for (int c = 0; c < cols; c++)
            for (int r = 0; r < rows; r++) {
                uint32_t s, v, m;
                fields(cbk.elem, src.at(rb * kRows + r, cbi * kCols + (uint64_t)l * kLaneCols + c), s, v, m);
                if (cbk.elem == 0) {
                    const uint32_t at = full ? 16u * (32u * (uint32_t)(c >> 1) + (uint32_t)l) + 8u * (uint32_t)(c & 1) + (uint32_t)r
                                             : lane_off + 8u * (uint32_t)c + (uint32_t)r;
                    raw[at] = (uint8_t)((s << 7) | m);
                } else {
                    const uint32_t at = full ? 16u * (32u * (uint32_t)(c >> 2) + (uint32_t)l) + 4u * (uint32_t)(c & 3) + (uint32_t)(r >> 1)
                                             : lane_off + 4u * (uint32_t)c + (uint32_t)(r >> 1);
                    raw[at] |= (uint8_t)(((s << 3) | m) << (4 * (r & 1)));
                }
            }
        if (!full) lane_off += lane_raw_bytes(src.k, cbi, l, cbk.elem);
    }
    uint32_t *list = reinterpret_cast<uint32_t *>(raw + raw_section_bytes(src.k, cbi, cbk.elem));
    uint32_t *list_end = reinterpret_cast<uint32_t *>(dst + size);
    for (uint32_t e : esc) *list++ = e;
    while (list < list_end) *list++ = kEscPad;
}

int pick_threads(int threads) {
    if (threads > 0) return threads;
    unsigned h = std::thread::hardware_concurrency();
    return h ? (int)h : 1;
}

template <class F>
void parallel_for(uint64_t count, int threads, F &&fn) {
    threads = (int)std::min<uint64_t>((uint64_t)threads, std::max<uint64_t>(count, 1));
    if (threads <= 1) {
        for (uint64_t i = 0; i < count; i++) fn(i);
        return;
    }
    std::atomic<uint64_t> next{0};
    std::vector<std::thread> pool;
    const uint64_t chunk = 16;
    for (int t = 0; t < threads; t++)
        pool.emplace_back([&] {
            for (;;) {
                uint64_t s = next.fetch_add(chunk);
                if (s >= count) break;
                uint64_t e = std::min(count, s + chunk);
                for (uint64_t i = s; i < e; i++) fn(i);
            }
        });
    for (auto &th : pool) th.join();
}

inline void put64(uint8_t *p, uint64_t v) { std::memcpy(p, &v, 8); }  // little-endian hosts

template <class E>
nwc_status encode_impl(const Src<E> &src, int elem, const float *scales, int threads, void *blob,
                       size_t *blob_bytes) {
    threads = pick_threads(threads);
    const uint64_t RB = cdiv(src.n, kRows), CB = cdiv(src.k, kCols), NB = RB * CB;
    if (NB >= (1ull << 31)) return NWC_ERR_INVALID_ARG;
    // histogram of exponent values over the real elements, per row-block then summed
    std::vector<uint64_t> hist_rb(RB * 256, 0);
    parallel_for(RB, threads, [&](uint64_t rb) {
        uint64_t *h = &hist_rb[rb * 256];
        int rows = real_rows(src.n, rb);
        for (int r = 0; r < rows; r++)
            for (uint64_t c = 0; c < src.k; c++) {
                uint32_t s, v, m;
                fields(elem, src.at(rb * kRows + r, c), s, v, m);
                h[v]++;
            }
    });
    uint64_t hist[256] = {0};
    for (uint64_t rb = 0; rb < RB; rb++)
        for (int v = 0; v < 256; v++) hist[v] += hist_rb[rb * 256 + v];
    const Codebook cbk = make_codebook(hist, elem);

    std::vector<uint64_t> size(NB);
    parallel_for(RB, threads, [&](uint64_t rb) {
        for (uint64_t c = 0; c < CB; c++) size[rb * CB + c] = block_size(src, cbk, rb, c);
    });
    std::vector<uint64_t> off(NB + 1, 0);
    for (uint64_t b = 0; b < NB; b++) off[b + 1] = off[b] + size[b];
    if (off[NB] / 16 >= (1ull << 32)) return NWC_ERR_INVALID_ARG;
    const uint64_t off_blocks = kBlockTabOff;
    const uint64_t tab_end = off_blocks + 4 * (NB + 1);
    const uint64_t off_scales = elem == 1 ? up16(tab_end) : 0;
    const uint64_t off_data = elem == 1 ? up16(off_scales + 4 * src.n) : up16(tab_end);
    const uint64_t total = off_data + off[NB];
    if (!blob) {
        *blob_bytes = (size_t)total;
        return NWC_OK;
    }
    if (*blob_bytes < total) return NWC_ERR_INVALID_ARG;
    uint8_t *b = static_cast<uint8_t *>(blob);
    std::memset(b, 0, (size_t)off_data);
    uint32_t magic = kMagic;
    std::memcpy(b + H_MAGIC, &magic, 4);
    b[H_VERSION] = (uint8_t)kVersion;
    b[H_VERSION + 1] = 0;
    b[H_ELEM] = (uint8_t)elem;
    b[H_NR] = (uint8_t)cbk.nr;
    put64(b + H_N, src.n);
    put64(b + H_K, src.k);
    put64(b + H_NB, NB);
    put64(b + H_OFF_BLOCKS, off_blocks);
    put64(b + H_OFF_SCALES, off_scales);
    put64(b + H_OFF_DATA, off_data);
    put64(b + H_TOTAL, total);
    std::memcpy(b + kRankOff, cbk.rank_exp, 16);
    for (uint64_t i = 0; i <= NB; i++) {
        uint32_t u = (uint32_t)(off[i] / 16);
        std::memcpy(b + off_blocks + 4 * i, &u, 4);
    }
    if (elem == 1 && scales) std::memcpy(b + off_scales, scales, 4 * src.n);
    // Regions are written at 16-byte aligned offsets into a 16-byte aligned scratch when the
    // caller's buffer is not aligned; otherwise in place.
    const bool aligned = (reinterpret_cast<uintptr_t>(b + off_data) % 16) == 0;
    parallel_for(RB, threads, [&](uint64_t rb) {
        std::vector<uint32_t> tmp;
        for (uint64_t c = 0; c < CB; c++) {
            uint64_t bi = rb * CB + c;
            uint8_t *dst = b + off_data + off[bi];
            if (aligned) {
                std::memset(dst, 0, size[bi]);
                write_block(src, cbk, rb, c, dst, size[bi]);
            } else {
                tmp.assign(size[bi] / 4, 0);
                write_block(src, cbk, rb, c, reinterpret_cast<uint8_t *>(tmp.data()), size[bi]);
                std::memcpy(dst, tmp.data(), size[bi]);
            }
        }
    });
    *blob_bytes = (size_t)total;
    return NWC_OK;
}

// FP32 -> e4m3, round to nearest even, saturating at +-448 (OCP FP8 e4m3: bias 7, no
// infinities). Written from the format definition with frexp/nearbyint (default rounding
// mode is to-nearest-even).
uint8_t e4m3_rne_sat(float f) {
    uint8_t sign = std::signbit(f) ? 0x80 : 0x00;
    float a = std::fabs(f);
    if (a > 448.0f) return sign | 0x7E;
    if (a < 0.015625f) {  // below 2^-6: subnormal step 2^-9 (the result 8 is the first normal)
        int m = (int)std::nearbyint(std::ldexp(a, 9));
        return sign | (uint8_t)m;
    }
    int ex;
    float fr = std::frexp(a, &ex);  // a = fr * 2^ex, fr in [0.5, 1)
    int e = ex - 1;                  // a = (2 fr) * 2^e
    int m = (int)std::nearbyint((2.0f * fr - 1.0f) * 8.0f);
    if (m == 8) { m = 0; e++; }
    int code = ((e + 7) << 3) | m;
    if (code > 0x7E) code = 0x7E;
    return sign | (uint8_t)code;
}

inline float bf16_to_f32(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    std::memcpy(&f, &u, 4);
    return f;
}

}  // namespace

extern "C" nwc_status nwc_quantize_fp8(const uint16_t *w, int64_t n, int64_t k, int64_t ld,
                                       uint8_t *q, int64_t ldq, float *scales) {
    if (!w || !q || !scales || n <= 0 || k <= 0 || ld < k || ldq < k) return NWC_ERR_INVALID_ARG;
    for (int64_t r = 0; r < n; r++) {
        float a = 0.0f;
        for (int64_t c = 0; c < k; c++) {
            float f = bf16_to_f32(w[r * ld + c]);
            if (!std::isfinite(f)) return NWC_ERR_INVALID_ARG;
            a = std::max(a, std::fabs(f));
        }
        float s = a == 0.0f ? 1.0f : a / 448.0f;
        scales[r] = s;
        for (int64_t c = 0; c < k; c++) q[r * ldq + c] = e4m3_rne_sat(bf16_to_f32(w[r * ld + c]) / s);
    }
    return NWC_OK;
}

extern "C" nwc_status nwc_encode_fp8(const uint8_t *q, const float *scales, int64_t n, int64_t k,
                                     int64_t ld, int threads, void *blob, size_t *blob_bytes) {
    if (!q || !scales || !blob_bytes || n <= 0 || k <= 0 || ld < k) return NWC_ERR_INVALID_ARG;
    Src<uint8_t> src{q, ld, (uint64_t)n, (uint64_t)k};
    return encode_impl(src, NWC_ELEM_FP8_E4M3, scales, threads, blob, blob_bytes);
}

extern "C" nwc_status nwc_encode(const uint16_t *w, int64_t n, int64_t k, int64_t ld, int elem,
                                 int threads, void *blob, size_t *blob_bytes) {
    if (!w || !blob_bytes || n <= 0 || k <= 0 || ld < k) return NWC_ERR_INVALID_ARG;
    if (elem == NWC_ELEM_BF16) {
        Src<uint16_t> src{w, ld, (uint64_t)n, (uint64_t)k};
        return encode_impl(src, NWC_ELEM_BF16, nullptr, threads, blob, blob_bytes);
    }
    if (elem != NWC_ELEM_FP8_E4M3) return NWC_ERR_INVALID_ARG;
    std::vector<uint8_t> q((size_t)(n * k));
    std::vector<float> s((size_t)n);
    nwc_status st = nwc_quantize_fp8(w, n, k, ld, q.data(), k, s.data());
    if (st != NWC_OK) return st;
    return nwc_encode_fp8(q.data(), s.data(), n, k, k, threads, blob, blob_bytes);
}
