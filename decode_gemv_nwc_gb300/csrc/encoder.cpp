// encoder.cpp -- host encoder of the NWC blob and the fp8 e4m3 quantizer.
//
// "NWC -- Neural Weight Compression", section "How it works": a BF16 weight is split into a
// raw mantissa plane and an exponent/sign part; the exponent is ranked by frequency and
// written as a unary rank code plus a raw sign bit, with an escape for rare values (in the
// stream n_ranked ones and the sign; the element's bits go to the block's escape list, so that
// no in-stream code is longer than 12 bits); every lane of a block of 8 rows x 512 columns has
// its own bit stream; padding to any shape costs 2 bits per filler weight and no mantissa.
// Mantissa regions are interleaved word by word across the lanes when all lanes have the same
// word count (every block whose 512 columns are all inside K).
// "Qwen3-4B-NWC-fp8": weight-only e4m3, symmetric per-output-channel scale, bytes coded
// losslessly with the same code (4-bit exponent, 3-bit raw mantissa).
//
// Work is split over row-blocks across host threads. Pass 1 sizes every block region from a
// per-exponent code-length table, pass 2 writes each region at its prefix-summed offset, so
// the bytes do not depend on the thread count.
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
    int elem = 0, nr = 0, eb = 8, F = 7;
    uint32_t code[256];  // code of the exponent value with its sign slot (sign bit = 0)
    uint8_t len[256];    // code length including the sign bit
    uint8_t rank_exp[16];
    bool escaped[256];
};

// Ranking: values with a nonzero count, most frequent first, ties to the lower value;
// at most kMaxRanked of them get a unary code, the rest escape.
Codebook make_codebook(const uint64_t *hist, int elem) {
    Codebook cb;
    cb.elem = elem;
    cb.eb = exp_bits(elem);
    cb.F = man_bits(elem);
    int nv = 1 << cb.eb;
    std::vector<int> vals;
    for (int v = 0; v < nv; v++)
        if (hist[v]) vals.push_back(v);
    std::stable_sort(vals.begin(), vals.end(), [&](int a, int b) { return hist[a] > hist[b]; });
    cb.nr = std::min<int>((int)vals.size(), kMaxRanked);
    std::memset(cb.rank_exp, 0, sizeof(cb.rank_exp));
    for (int v = 0; v < nv; v++) {  // escape: nr ones, sign
        cb.code[v] = ((1u << cb.nr) - 1u) << 1;
        cb.len[v] = (uint8_t)(cb.nr + 1);
        cb.escaped[v] = true;
    }
    for (int p = 0; p < cb.nr; p++) {  // rank p: p ones, a zero, sign
        int v = vals[p];
        cb.rank_exp[p] = (uint8_t)v;
        cb.code[v] = ((1u << p) - 1u) << 2;
        cb.len[v] = (uint8_t)(p + 2);
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

// MSB-first bit sink into 32-bit words.
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
            uint32_t w = (uint32_t)(acc >> nacc);
            if (out) out[nw] = w;
            nw++;
        }
    }
    void flush() {
        if (nacc > 0) {
            uint32_t w = (uint32_t)(acc << (32 - nacc));
            if (out) out[nw] = w;
            nw++;
            nacc = 0;
        }
    }
};

// LSB-first F-bit fields into 16-bit half-words.
struct HalfSink {
    uint16_t h[kSyms];
    uint32_t acc = 0;
    int nacc = 0, nh = 0;
    void put(uint32_t m, int F) {
        acc |= m << nacc;
        nacc += F;
        if (nacc >= 16) {
            h[nh++] = (uint16_t)acc;
            acc >>= 16;
            nacc -= 16;
        }
    }
    void flush() {
        if (nacc > 0) { h[nh++] = (uint16_t)acc; acc = 0; nacc = 0; }
    }
};

// Size in bytes of block (rb, cb)'s region; with lane word counts.
template <class E>
uint64_t block_size(const Src<E> &src, const Codebook &cbk, uint64_t rb, uint64_t cbi, uint8_t *lw) {
    int rows = real_rows(src.n, rb);
    uint64_t code_words = 0, man = 0, n_esc = 0;
    for (int l = 0; l < kLanes; l++) {
        int cols = real_cols(src.k, cbi, l);
        uint32_t bits = 2u * (uint32_t)(kSyms - rows * cols);  // fillers
        for (int c = 0; c < cols; c++)
            for (int r = 0; r < rows; r++) {
                uint32_t s, v, m;
                fields(cbk.elem, src.at(rb * kRows + r, cbi * kCols + (uint64_t)l * kLaneCols + c), s, v, m);
                bits += cbk.len[v];
                n_esc += cbk.escaped[v];
            }
        uint32_t nw = (bits + 31) / 32;
        if (lw) lw[l] = (uint8_t)nw;
        code_words += nw;
        man += man_words(rows, cols, cbk.F);
    }
    return up16(32 + 4 * code_words) + 4 * man + up16(4 * n_esc);
}

template <class E>
void write_block(const Src<E> &src, const Codebook &cbk, uint64_t rb, uint64_t cbi, uint8_t *dst, uint64_t size) {
    int rows = real_rows(src.n, rb);
    uint32_t *words = reinterpret_cast<uint32_t *>(dst + 32);  // dst is 16-byte aligned
    uint32_t pos = 0;
    for (int l = 0; l < kLanes; l++) {
        int cols = real_cols(src.k, cbi, l);
        CodeSink cs;
        cs.out = words + pos;
        for (int t = 0; t < kSyms; t++) {
            int c = t / kRows, r = t % kRows;
            if (r >= rows || c >= cols) { cs.put(0, 2); continue; }
            uint32_t s, v, m;
            fields(cbk.elem, src.at(rb * kRows + r, cbi * kCols + (uint64_t)l * kLaneCols + c), s, v, m);
            cs.put(cbk.code[v] | s, cbk.len[v]);
        }
        cs.flush();
        dst[l] = (uint8_t)cs.nw;
        pos += cs.nw;
    }
    uint8_t *man = dst + up16(32 + 4 * (uint64_t)pos);
    // all lanes with the same word count: word k of lane l at 32k + l (interleaved)
    bool uniform = true;
    for (int l = 1; l < kLanes; l++)
        uniform &= man_words(rows, real_cols(src.k, cbi, l), cbk.F) == man_words(rows, real_cols(src.k, cbi, 0), cbk.F);
    uint32_t *man0 = reinterpret_cast<uint32_t *>(man);
    for (int l = 0; l < kLanes; l++) {
        int cols = real_cols(src.k, cbi, l);
        HalfSink ev, od;
        for (int t = 0; t < kSyms; t++) {
            int c = t / kRows, r = t % kRows;
            if (r >= rows || c >= cols) continue;
            uint32_t s, v, m;
            fields(cbk.elem, src.at(rb * kRows + r, cbi * kCols + (uint64_t)l * kLaneCols + c), s, v, m);
            (r % 2 == 0 ? ev : od).put(m, cbk.F);
        }
        ev.flush();
        od.flush();
        uint32_t mw = man_words(rows, cols, cbk.F);
        uint32_t *mwp = reinterpret_cast<uint32_t *>(man);
        for (uint32_t i = 0; i < mw; i++) {
            uint32_t lo = (int)i < ev.nh ? ev.h[i] : 0, hi = (int)i < od.nh ? od.h[i] : 0;
            if (uniform) man0[i * kLanes + (uint32_t)l] = lo | (hi << 16);
            else mwp[i] = lo | (hi << 16);
        }
        man += 4 * mw;
    }
    // escape list: lanes in order, t increasing; padding to the region's end
    uint32_t *esc = reinterpret_cast<uint32_t *>(man);
    uint32_t *esc_end = reinterpret_cast<uint32_t *>(dst + size);
    for (int l = 0; l < kLanes; l++) {
        int cols = real_cols(src.k, cbi, l);
        for (int t = 0; t < kSyms; t++) {
            int c = t / kRows, r = t % kRows;
            if (r >= rows || c >= cols) continue;
            uint32_t x = src.at(rb * kRows + r, cbi * kCols + (uint64_t)l * kLaneCols + c), s, v, m;
            fields(cbk.elem, x, s, v, m);
            if (cbk.escaped[v]) *esc++ = esc_entry((uint32_t)t, (uint32_t)l, x);
        }
    }
    while (esc < esc_end) *esc++ = kEscPad;
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
        for (uint64_t c = 0; c < CB; c++) size[rb * CB + c] = block_size(src, cbk, rb, c, nullptr);
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
