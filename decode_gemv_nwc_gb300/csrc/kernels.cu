// kernels.cu -- sm_103a kernels and C-ABI launchers: decode to BF16/e4m3, embedding gather,
// the fused decode-GEMV (one or two vectors) and the small-batch GEMV (up to 16 vectors).
//
// "NWC -- Neural Weight Compression", section "How it works":
//   * each lane decodes its own bit stream for a block of 8 rows x 512 columns (16 columns
//     x 8 rows per lane), keeps the 16 matching activations in registers and accumulates
//     eight row sums; a transposed shuffle reduction produces partial sums per (row, column
//     block);
//   * a 12-bit peek into a 16 KB shared-memory lookup table yields two complete codes per
//     step; the bit window is shifted and refilled from the lane's words;
//   * dequantization and embedding lookup run on the same decoder.
// Escapes (the pages' escape for rare exponents): the stream holds n_ranked ones and the sign, the element's
// bits are in the block's escape list. Every in-stream code thus fits the 12-bit peek and the
// GEMV's hot loop has no escape branch: it multiplies a placeholder (the sign and raw mantissa
// with exponent field 0, a subnormal) and the warp adds (true - placeholder) * x for each list
// entry before its row reduction. Decode and gather write the listed elements over the
// placeholders.
// "Qwen3-4B-NWC-fp8": the per-channel scale is applied at the end of the matvec.
//
// GB300 choices: the GEMV is a persistent grid of one 32-warp CTA per SM (block b on CTA
// b % grid); each warp streams whole block regions (counts, code streams, mantissas, escape
// list) from HBM into its own shared-memory stage with one TMA bulk copy (cp.async.bulk,
// completion on an mbarrier, bounded waits) and prefetches its next region into L2; every CTA
// builds the 4096-entry table in shared memory while its first copies are in flight; a lane
// decodes four codes per window refill (the table yields one code per peek: a second code from
// the same peek would be incomplete too often for a SIMT warp); the LUT
// entry carries the code as a BF16 high half so that one LOP3 merges a row pair's two raw
// mantissas (stored 16 bits apart) into a BF16x2, which feeds FMAs with BF16 operands and FP32
// accumulators (fp8: packed FP32 FMA). Cross-column-block sums are done by the last warp to
// finish a row block (one counter per row block, reset by that warp), in a fixed order. The
// kernel is launched with programmatic stream serialization: it may start while the previous
// kernel on the stream drains and waits for it before touching x, the workspace or y.
// The small-batch GEMV keeps the decoder and moves the products with three or more vectors to
// the tensor cores (mma.sync on decoded tiles staged in shared memory).
// Blocks that reach past K or N (filler codes, mantissas of real elements only) take the same
// decoders, in kernel instantiations of their own; a generic one-code-at-a-time decoder serves
// regions too large for a stage and blocks whose fillers could decode to Inf or NaN.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "nwc.h"
#include "nwc_format.h"

using namespace nwcf;

// Device error word: bit 0 = malformed stream (a lane read past its words, or an escape list
// that does not match the lane streams), bit 1 = gather id out of range, bit 2 = a bounded wait
// ran out. Read and cleared by nwc_check.
__device__ uint32_t g_nwc_error;

namespace {

constexpr uint32_t kErrFormat = 1u, kErrId = 2u, kErrTimeout = 4u;

struct Mat {
    int elem, nr;
    uint64_t n, k, rbs, cbs, nb;
    const uint32_t *tab;
    const uint8_t *data;
    const float *scales;
    uint8_t rank_exp[16];
};

Mat to_mat(const nwc_matrix &m) {
    Mat t;
    t.elem = m.elem;
    t.nr = m.n_ranked;
    t.n = (uint64_t)m.n;
    t.k = (uint64_t)m.k;
    t.rbs = (uint64_t)m.row_blocks;
    t.cbs = (uint64_t)m.col_blocks;
    t.nb = t.rbs * t.cbs;
    t.tab = m.block_tab;
    t.data = m.data;
    t.scales = m.scales;
    for (int i = 0; i < 16; i++) t.rank_exp[i] = m.rank_exp[i];
    return t;
}

__device__ __forceinline__ void raise_error(uint32_t bits) { atomicOr(&g_nwc_error, bits); }

// Copies the rank table into shared memory without indexing the kernel parameter
// dynamically (which would spill the whole parameter struct to local memory).
__device__ __forceinline__ void load_rank_table(const Mat &m, uint8_t *rexp) {
    if (threadIdx.x < 16) {
        uint32_t v = 0;
#pragma unroll
        for (int i = 0; i < 16; i++)
            if ((int)threadIdx.x == i) v = m.rank_exp[i];
        rexp[threadIdx.x] = (uint8_t)v;
    }
}

// ------------------------------------------------------------------ lane bit stream
// 64-bit window, most significant bit = next stream bit; nb valid bits at the top. The word
// pointer may point into shared memory (a staged block) or global memory; after inlining the
// compiler emits shared or global loads accordingly.
struct LaneStream {
    const uint32_t *p, *start, *end;
    int nb;
    uint64_t win;

    __device__ __forceinline__ void init(const uint32_t *ptr, uint32_t n) {
        p = start = ptr;
        end = ptr + n;
        nb = 0;
        win = 0;
        refill();
        refill();
    }
    // Ensures at least 33 valid bits. Past the lane's last word, zero words are inserted
    // without reading memory; overrun() reports whether such bits were consumed.
    __device__ __forceinline__ void refill() {
        if (nb <= 32) {
            const uint32_t w = p < end ? *p : 0u;
            p++;
            win |= (uint64_t)w << (32 - nb);
            nb += 32;
        }
    }
    __device__ __forceinline__ void consume(uint32_t L) {
        win <<= L;
        nb -= (int)L;
    }
    __device__ __forceinline__ uint32_t top() const { return (uint32_t)(win >> 32); }
    __device__ __forceinline__ bool overrun() const {
        return (uint64_t)(p - start) * 32u - (uint64_t)nb > (uint64_t)(end - start) * 32u;
    }
};

// One code: rank p < nr is p ones, a zero, the sign; an escape is nr ones and the sign (its
// exponent is in the escape list; v is returned as 0). Returns whether it was an escape.
template <class S>
__device__ __forceinline__ bool decode_one(S &ls, int nr, const uint8_t *rexp, uint32_t &s, uint32_t &v) {
    ls.refill();
    const uint32_t top = ls.top();
    const int ones = __clz(~top);
    const bool esc = ones >= nr;
    if (!esc) {
        v = rexp[ones];
        s = (top >> (30 - ones)) & 1u;
        ls.consume((uint32_t)ones + 2u);
    } else {
        v = 0;
        s = (top >> (31 - nr)) & 1u;
        ls.consume((uint32_t)nr + 1u);
    }
    return esc;
}

__device__ __forceinline__ bool stream_decode(LaneStream &ls, int nr, const uint8_t *rexp, uint32_t &s, uint32_t &v) {
    return decode_one(ls, nr, rexp, s, v);
}

// Field j of the even (odd = 0) or odd (odd = 1) mantissa half-stream of a lane region whose
// word k is man[k * stride] (stride 32 when the block's lane regions are interleaved).
template <int F>
__device__ __forceinline__ uint32_t half_field(const uint32_t *man, uint32_t stride, int odd, uint32_t j) {
    const uint32_t bit = (uint32_t)F * j, k = bit >> 4, o = bit & 15u;
    uint32_t w = man[k * stride];
    uint32_t h = odd ? (w >> 16) : (w & 0xFFFFu);
    if (o + F > 16) {
        uint32_t w1 = man[(k + 1) * stride];
        h |= (odd ? (w1 >> 16) : (w1 & 0xFFFFu)) << 16;
    }
    return (h >> o) & ((1u << F) - 1u);
}

// Element value as FP32 from its fields.
template <int ELEM>
__device__ __forceinline__ float elem_value(uint32_t s, uint32_t v, uint32_t m) {
    if (ELEM == 0) return __uint_as_float(((s << 15) | (v << 7) | m) << 16);
    // e4m3: bias 7, subnormals at v == 0, S.1111.111 is NaN
    if (v == 0) {
        float f = (float)m * 0.001953125f;  // m * 2^-9, exact
        return s ? -f : f;
    }
    if (v == 15 && m == 7) return __uint_as_float(0x7FC00000u);
    return __uint_as_float((s << 31) | ((v + 120u) << 23) | (m << 20));
}

template <int ELEM>
__device__ __forceinline__ uint32_t elem_bits(uint32_t s, uint32_t v, uint32_t m) {
    return ELEM == 0 ? ((s << 15) | (v << 7) | m) : ((s << 7) | (v << 3) | m);
}

// Generic decode of one lane of one block, column loop rolled and rows unrolled: calls
// fn(c, r, s, v, m, esc) for each real element (column c, row r of the lane). rows/cols are the
// lane's real extent. Returns the number of escape codes in the lane's 128 codes.
template <int ELEM, class S, class Fn>
__device__ __forceinline__ uint32_t lane_rolled(S &ls, const uint32_t *man, uint32_t stride, int rows,
                                                int cols, int nr,
                                                const uint8_t *rexp, Fn &&fn) {
    constexpr int F = ELEM == 0 ? 7 : 3;
    uint32_t je = 0, jo = 0, n_esc = 0;
#pragma unroll 1
    for (int c = 0; c < kLaneCols; c++) {
#pragma unroll
        for (int r = 0; r < kRows; r++) {
            uint32_t s, v;
            const bool esc = stream_decode(ls, nr, rexp, s, v);
            n_esc += esc;
            if (r < rows && c < cols) {
                uint32_t m;
                if (r & 1) m = half_field<F>(man, stride, 1, jo++);
                else m = half_field<F>(man, stride, 0, je++);
                fn(c, r, s, v, m, esc);
            }
        }
    }
    return n_esc;
}

// Layout facts of one block region at `reg` (`bytes` long) for this lane.
struct LaneRegion {
    const uint32_t *code, *man, *esc;
    uint32_t nwords, slots;  // slots = escape-list words (entries and padding)
    uint32_t man_stride;     // 32 when the lanes' mantissa words are interleaved, else 1
};

__device__ __forceinline__ LaneRegion lane_region(const uint8_t *reg, uint32_t bytes, int lane, int rows,
                                                  uint64_t k, uint64_t cb, int F) {
    const uint32_t lw = reg[lane];
    uint32_t incl = lw;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        uint32_t o = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        if (lane >= d) incl += o;
    }
    const uint32_t total = __shfl_sync(0xFFFFFFFFu, incl, 31);
    LaneRegion lr;
    lr.code = reinterpret_cast<const uint32_t *>(reg + 32) + (incl - lw);
    lr.nwords = lw;
    // mantissa regions in lane order; sizes from the real extents of lanes before this one
    uint32_t mw = man_words(rows, real_cols(k, cb, lane), F);
    uint32_t mincl = mw;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        uint32_t o = __shfl_up_sync(0xFFFFFFFFu, mincl, d);
        if (lane >= d) mincl += o;
    }
    const uint32_t man0 = (uint32_t)up16(32 + 4 * (uint64_t)total);
    const bool uniform = __all_sync(0xFFFFFFFFu, mw == __shfl_sync(0xFFFFFFFFu, mw, 0));
    lr.man = reinterpret_cast<const uint32_t *>(reg + man0) + (uniform ? (uint32_t)lane : mincl - mw);
    lr.man_stride = uniform ? (uint32_t)kLanes : 1u;
    const uint32_t esc0 = man0 + 4 * __shfl_sync(0xFFFFFFFFu, mincl, 31);
    lr.esc = reinterpret_cast<const uint32_t *>(reg + esc0);
    lr.slots = esc0 <= bytes ? (bytes - esc0) / 4 : 0;
    return lr;
}

// This lane's slice [start, start + cnt) of the block's escape list, from the lanes' escape
// counts; flags a list whose entry count differs from the streams' total or that is followed by
// more than three padding words.
__device__ __forceinline__ uint32_t esc_slice(const LaneRegion &lr, uint32_t cnt, int lane, bool &bad) {
    uint32_t incl = cnt;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        uint32_t o = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        if (lane >= d) incl += o;
    }
    const uint32_t total = __shfl_sync(0xFFFFFFFFu, incl, 31);
    if (lane == 0) {
        if (total > lr.slots || lr.slots - total > 3) bad = true;
        else if (total < lr.slots && lr.esc[total] != kEscPad) bad = true;
    }
    return incl - cnt;
}

// Writes this lane's escape-list entries [start, start + cnt) over their placeholders in the
// output: element (r, c) of the lane goes to out[(row0 + r) * ld_out + col0 + c], only for
// r == want when want >= 0. Checks that each entry names this lane and a real element of it;
// returns false if one does not. Kept out of line: inlined after the fully unrolled lane
// decode it more than doubled the decoders' register use.
template <int ELEM>
__device__ __noinline__ bool esc_patch(const uint32_t *esc, uint32_t slots, uint32_t start, uint32_t cnt, int lane,
                                       int rows, int cols, int want, void *out, int64_t ld_out, int64_t row0,
                                       uint64_t col0) {
    bool ok = true;
    for (uint32_t i = 0; i < cnt; i++) {
        const uint32_t j = start + i;
        const uint32_t e = j < slots ? esc[j] : kEscPad;
        const int t = (int)esc_t(e), c = t >> 3, r = t & 7;
        if (e == kEscPad || (int)esc_lane(e) != lane || r >= rows || c >= cols) {
            ok = false;
            continue;
        }
        if (want >= 0 && r != want) continue;
        const uint64_t at = (uint64_t)(row0 + r) * (uint64_t)ld_out + col0 + (uint64_t)c;
        if (ELEM == 0) static_cast<uint16_t *>(out)[at] = (uint16_t)esc_bits(e);
        else static_cast<uint8_t *>(out)[at] = (uint8_t)esc_bits(e);
    }
    return ok;
}

// =================================================================== GEMV kernel
// Warps per CTA (one CTA per SM) and block-region stages per warp. With one stage the next
// region is prefetched into L2 while the current one is decoded, then copied in.
#ifndef NWC_GEMV_WARPS
#define NWC_GEMV_WARPS 32
#endif
#ifndef NWC_GEMV_STAGES
#define NWC_GEMV_STAGES 1
#endif
constexpr int kGemvWarps = NWC_GEMV_WARPS;

constexpr int kStagesPerWarp = NWC_GEMV_STAGES;
constexpr int kStageBytes = 6144;
constexpr int kLutEntries = 4096;
constexpr int kLutBytes = kLutEntries * 4;
constexpr int kRexpOff = kLutBytes;
constexpr int kBarOff = kRexpOff + 16;
constexpr int kStageOff = (kBarOff + kGemvWarps * 2 * 8 + 127) / 128 * 128;
// A lane's fast decoder reads at most about 200 bytes past its first code word whatever the code
// bits (128 codes of at most 12 bits through a 64-bit window with one word of lookahead), and
// validation caps a lane at 48 words, so the last lane of a staged region can read up to
// 32 + 31 * 48 * 4 + 200 = 6184 bytes past the stage's start (a stage holds 6144): the slack
// after the last stage keeps those reads inside the allocation.
constexpr int kStageSlack = 256;
constexpr int kGemvSmem = kStageOff + kGemvWarps * kStagesPerWarp * kStageBytes + kStageSlack;
static_assert(kStagesPerWarp == 1 || kStagesPerWarp == 2, "stages");
static_assert(kGemvSmem <= 232448, "shared memory per CTA");
// CTAs per SM: 32 warps at 64 registers, and what 228 KB of shared memory holds (1 KB of it
// reserved per CTA)
constexpr int kCtasPerSm = (32 / kGemvWarps) < (233472 / (kGemvSmem + 1024)) ? (32 / kGemvWarps)
                                                                               : (233472 / (kGemvSmem + 1024));
static_assert(kCtasPerSm >= 1, "one CTA per SM at least");
// The GEMV kernel for NB vectors at once (1 or 2): two vectors need a second accumulator set, so
// 24 warps per SM with up to 85 registers each and one stage per warp.
template <int NB>
struct GemvCfg {
    static constexpr int kWarps = NB == 1 ? kGemvWarps : 24;
    static constexpr int kStages = NB == 1 ? kStagesPerWarp : 1;
    static constexpr int kStageOff = (kBarOff + kWarps * 2 * 8 + 127) / 128 * 128;
    static constexpr int kSmem = kStageOff + kWarps * kStages * kStageBytes + kStageSlack;
    static constexpr int kCtas = NB == 1 ? kCtasPerSm : 1;
};
static_assert(GemvCfg<2>::kSmem <= 232448, "shared memory per CTA");
// Decode: 16 warps per SM with up to 128 registers each, so that a lane holds its whole 8x16
// output tile and writes every 32-byte row segment with full-sector stores. Gather keeps one
// row per lane and runs 32 warps.
template <int MODE>
struct UnpackCfg {
    static constexpr int kWarps = MODE == 0 ? 16 : kGemvWarps;
    static constexpr int kStageOff = (kBarOff + kWarps * 2 * 8 + 127) / 128 * 128;
    static constexpr int kSmem = kStageOff + kWarps * kStageBytes + kStageSlack;
};
static_assert(UnpackCfg<0>::kSmem <= 232448 && UnpackCfg<1>::kSmem <= 232448, "shared memory per CTA");

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t phase) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(phase)
        : "memory");
    return ok != 0;
}
// Bounded wait: gives up after about 2^32 SM clocks (1-3 s) and reports failure.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t phase) {
    const long long t0 = clock64();
    for (;;) {
        if (mbar_try(bar, phase)) return true;
        if (clock64() - t0 > (1ll << 32)) return false;
    }
}
__device__ __forceinline__ void tma_load_1d(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// LUT entry for a 12-bit peek P (first stream bit = bit 11), one code per entry:
//   bits 0..4   code length L (rank + 2; an escape n_ranked + 1)
//   bits 5..6   zero (whole entries may be subtracted from the bit counter)
//   bits 7..15  BF16: the code as a BF16 high part (s << 15 | exponent << 7);
//               fp8: s << 15 | v << 11, so that with the 3-bit mantissa at bits 8..10 each
//               half's high byte is the e4m3 code itself.
//               An escape gets exponent field 0, the placeholder that the escape list corrects.
//   bit 24      set for an escape (sums of up to 128 entries stay below it, so a running sum
//               counts a lane's escapes in its top byte)
// A 12-bit peek holds any code (at most n_ranked + 1 <= 12 bits), which is why at most 11
// exponents are ranked.
template <int ELEM>
__device__ __forceinline__ uint32_t lut_entry(uint32_t P, int nr, const uint32_t (&rank4)[3]) {
    const uint32_t bits = P << 20;
    const int ones = __clz(~bits);
    if (ones >= nr) return (1u << 24) | (((bits >> (31 - nr)) & 1u) << 15) | (uint32_t)(nr + 1);
    const uint32_t word = ones < 4 ? rank4[0] : (ones < 8 ? rank4[1] : rank4[2]);
    const uint32_t s = (bits >> (30 - ones)) & 1u, v = (word >> (8 * (ones & 3))) & 0xFFu;
    return (s << 15) | (v << (ELEM == 0 ? 7 : 11)) | ((uint32_t)ones + 2);
}

// Builds the 4096-entry table in shared memory with all threads of the CTA; the rank table is
// read from the kernel parameter with static offsets only (packed four values per word).
template <int ELEM>
__device__ __forceinline__ void build_lut(const Mat &m, uint32_t *lut) {
    uint32_t rank4[3];
#pragma unroll
    for (int i = 0; i < 3; i++)
        rank4[i] = (uint32_t)m.rank_exp[4 * i] | (uint32_t)m.rank_exp[4 * i + 1] << 8 |
                   (uint32_t)m.rank_exp[4 * i + 2] << 16 | (uint32_t)m.rank_exp[4 * i + 3] << 24;
    for (uint32_t i = threadIdx.x; i < (uint32_t)kLutEntries; i += blockDim.x)
        lut[i] = lut_entry<ELEM>(i, m.nr, rank4);
}

// Pair q's two mantissas (even t at bits 0.., odd t at bits 16..) from a group's words.
template <int F>
__device__ __forceinline__ uint32_t xpair(const uint32_t *mw, int q) {
    const int bit = F * q, k = bit >> 4, o = bit & 15;
    if (o + F <= 16) return mw[k] >> o;
    const uint32_t M = (0xFFFFu >> o) * 0x10001u;
    return ((mw[k] >> o) & M) | ((mw[k + 1] << (16 - o)) & ~M);
}

// Row-ragged block (only the first `rows` < 8 rows real): the region stores mantissa fields of
// real elements only, he = (rows + 1) / 2 per column in the even half-stream and ho = rows / 2 in
// the odd one, where a full block has 4 and 4. Column c's fields start at field c he (c ho), and
// the 4 F bits from there hold its real fields followed by the next column's: taken whole into
// the column's place in the full-block layout, the real fields land where the full-block decoder
// reads them and the rest fall on rows past N, whose values are never stored. Reads stay inside
// the lane's nw mantissa words (word k at man + k mstride bytes); missing bits read as 0.
template <int F>
__device__ __forceinline__ uint32_t col_fields(uint32_t man, uint32_t mstride, uint32_t nw, int odd, uint32_t first) {
    const uint32_t bit = (uint32_t)F * first, k = bit >> 4, o = bit & 15u;
    uint64_t v = 0;
#pragma unroll
    for (int i = 0; i < 3; i++) {  // o + 4 F <= 43 bits
        uint32_t w = 0;
        if (k + i < nw) asm volatile("ld.shared.u32 %0, [%1];" : "=r"(w) : "r"(man + (k + i) * mstride));
        v |= (uint64_t)(odd ? w >> 16 : w & 0xFFFFu) << (16 * i);
    }
    return (uint32_t)(v >> o) & ((1u << (4 * F)) - 1u);
}

// Group g (columns 4g .. 4g + 3) of a row-ragged block in the full-block word layout: word i =
// even half-word F g + i | odd half-word F g + i << 16.
template <int F>
__device__ __forceinline__ void group_fields_ragged(uint32_t man, uint32_t mstride, uint32_t nw, int g, int rows,
                                                    uint32_t (&mw)[F]) {
    const uint32_t he = (uint32_t)(rows + 1) >> 1, ho = (uint32_t)rows >> 1;
#pragma unroll
    for (int i = 0; i < F; i++) mw[i] = 0;
#pragma unroll
    for (int cl = 0; cl < 4; cl++) {
        const uint32_t c = 4u * (uint32_t)g + (uint32_t)cl;
        const int P = 4 * F * cl, k = P >> 4, o = P & 15;  // the column's place in the group (static)
#pragma unroll
        for (int odd = 0; odd < 2; odd++) {
            const uint64_t v = (uint64_t)col_fields<F>(man, mstride, nw, odd, c * (odd ? ho : he)) << o;
#pragma unroll
            for (int h = 0; h < 3; h++)
                if (k + h < F) mw[k + h] |= ((uint32_t)(v >> (16 * h)) & 0xFFFFu) << (16 * odd);
        }
    }
}

// Transposed reduction of acc[8] over the 32 lanes: afterwards lanes with (lane & 3) == 0
// hold the sum of row rowsel(lane) = bit4<<2 | bit3<<1 | bit2 of the lane id.
__device__ __forceinline__ float transpose_reduce(float (&acc)[8], int lane) {
    float a4[4];
    const bool up16 = lane & 16;
#pragma unroll
    for (int i = 0; i < 4; i++) {
        float send = up16 ? acc[i] : acc[i + 4];
        float keep = up16 ? acc[i + 4] : acc[i];
        a4[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 16);
    }
    float a2[2];
    const bool up8 = lane & 8;
#pragma unroll
    for (int i = 0; i < 2; i++) {
        float send = up8 ? a4[i] : a4[i + 2];
        float keep = up8 ? a4[i + 2] : a4[i];
        a2[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 8);
    }
    const bool up4 = lane & 4;
    float send = up4 ? a2[0] : a2[1];
    float keep = up4 ? a2[1] : a2[0];
    float a1 = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 4);
    a1 += __shfl_xor_sync(0xFFFFFFFFu, a1, 2);
    a1 += __shfl_xor_sync(0xFFFFFFFFu, a1, 1);
    return a1;
}

// Fast-path stream state in registers: window wh:wl (most significant bit first); V holds
// (valid bits - 1) in its low 7 bits (at most 64 bits are buffered), so whole LUT entries,
// whose bits 5..6 are zero and whose low five bits are the length, can be subtracted from it;
// pa = shared-memory address of the next code word. Reads past a lane's words stay inside the
// staged region (its mantissa regions follow the code streams), so a malformed stream yields
// garbage but no out-of-bounds access; the bit count check flags it.
struct Fs32 {
    uint32_t wh, wl, V, pa, nw;  // nw = the word at pa, loaded one refill ahead
};

// Branch-free refill: when at most 32 bits are valid the next word is added right below them
// by a multiply-add with 2^(32 - valid) (the pages refill with one wide multiply-add; here it
// is split into its low and high halves: the bits below the valid ones are zero, so no carry crosses);
// otherwise the multiplier is 0. The word was loaded by the previous refill, so the shared-memory
// latency of the following word's load is off the decode chain.
__device__ __forceinline__ void fs_refill(Fs32 &s) {
    asm("{\n\t"
        ".reg .pred q;\n\t"
        ".reg .u32 t, mul;\n\t"
        "and.b32 t, %3, 127;\n\t"
        "shf.r.clamp.b32 mul, 0x80000000, 0, t;\n\t"
        "setp.ne.u32 q, mul, 0;\n\t"
        "mad.lo.u32 %1, %4, mul, %1;\n\t"
        "mad.hi.u32 %0, %4, mul, %0;\n\t"
        "@q add.u32 %2, %2, 4;\n\t"
        "@q add.u32 %3, %3, 32;\n\t"
        "@q ld.shared.u32 %4, [%2];\n\t"
        "}"
        : "+r"(s.wh), "+r"(s.wl), "+r"(s.pa), "+r"(s.V), "+r"(s.nw));
}

__device__ __forceinline__ void fs_consume(Fs32 &s, uint32_t e) {  // e mod 32 bits
    const uint32_t h = __funnelshift_l(s.wl, s.wh, e);
    s.wl = __funnelshift_l(0u, s.wl, e);
    s.wh = h;
    s.V -= e;
}

__device__ __forceinline__ uint32_t lut_at(const Fs32 &s, uint32_t lutb) {
    uint32_t e;
    asm("{\n\t.reg .u32 a;\n\tshr.u32 a, %1, 20;\n\tmad.lo.u32 a, a, 4, %2;\n\tld.shared.u32 %0, [a];\n\t}"
        : "=r"(e)
        : "r"(s.wh), "r"(lutb));
    return e;
}

// The generic decoder's stream over a staged region: the fast path's window and table, one
// lookup per code. It serves malformed streams too, so every word read is checked against
// `limit` (the last word of the warp's stage); past it the stream reads zeros.
template <int ELEM>
struct LutStream {
    Fs32 f;
    uint32_t code, lw, lutb, limit;
    __device__ __forceinline__ uint32_t word(uint32_t a) const {
        uint32_t w = 0;
        if (a <= limit) asm("ld.shared.u32 %0, [%1];" : "=r"(w) : "r"(a));
        return w;
    }
    __device__ __forceinline__ void init(uint32_t code_, uint32_t lw_, uint32_t lutb_, uint32_t limit_) {
        code = code_;
        lw = lw_;
        lutb = lutb_;
        limit = limit_;
        f.wh = lw > 0 ? word(code) : 0u;
        f.wl = lw > 1 ? word(code + 4) : 0u;
        f.pa = code + 8;
        f.V = 63u;
        f.nw = word(f.pa);
    }
    // at most 32 valid bits: the preloaded word goes right below them (as fs_refill)
    __device__ __forceinline__ void refill() {
        const uint32_t t = f.V & 127u;  // valid bits - 1
        if (t < 32u) {
            f.wl += f.nw << (31u - t);
            f.wh += t == 31u ? 0u : f.nw >> (t + 1u);
            f.pa += 4;
            f.V += 32;
            f.nw = word(f.pa);
        }
    }
    __device__ __forceinline__ bool overrun() const {
        const uint32_t valid = (f.V & 127u) + 1u, inserted = (f.pa - code) * 8u;
        return inserted - valid > 32u * lw;
    }
};

template <int ELEM>
__device__ __forceinline__ bool stream_decode(LutStream<ELEM> &ls, int, const uint8_t *, uint32_t &s, uint32_t &v) {
    ls.refill();  // a refill leaves at least 33 valid bits; a code takes at most 12
    const uint32_t e = lut_at(ls.f, ls.lutb);
    fs_consume(ls.f, e);
    s = (e >> 15) & 1u;
    v = ELEM == 0 ? (e >> 7) & 0xFFu : (e >> 11) & 0xFu;
    return (e >> 24) & 1u;
}

// fp8: the row pair's two e4m3 codes (the high bytes of the halves) widened exactly to FP32
// through the hardware e4m3x2 -> f16x2 conversion (subnormals included).
__device__ __forceinline__ void e4m3_pair_to_f32(uint32_t bf, float &w0, float &w1) {
    const uint32_t codes = __byte_perm(bf, 0u, 0x0031u);
    asm("{\n\t.reg .b16 c, l, u;\n\t.reg .b32 h;\n\t"
        "cvt.u16.u32 c, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 h, c;\n\t"
        "mov.b32 {l, u}, h;\n\t"
        "cvt.f32.f16 %0, l;\n\t"
        "cvt.f32.f16 %1, u;\n\t}"
        : "=f"(w0), "=f"(w1)
        : "r"(codes));
}

// Row pair from its two table entries and raw mantissas X (even t at bits 0.., odd t at 16..):
// packed BF16 (row r in the low half; fp8: each half's high byte is the e4m3 code); fp8 also
// returns the two values as FP32 in w0, w1.
template <int ELEM>
__device__ __forceinline__ uint32_t pair_bits(uint32_t e1, uint32_t e2, uint32_t X, float &w0, float &w1) {
    const uint32_t e = __byte_perm(e1, e2, 0x5410);
    uint32_t bf;
    if (ELEM == 0) {
        bf = (e & 0xFF80FF80u) | (X & 0x007F007Fu);
    } else {
        bf = (e & 0xFF80FF80u) | ((X & 0x00070007u) << 8);
        e4m3_pair_to_f32(bf, w0, w1);
    }
    return bf;
}

// One row pair: refill, two single-code lookups, assembly with the raw mantissas (the batch
// GEMV's decoder; the single-vector GEMV decodes four codes per refill, below).
template <int ELEM>
__device__ __forceinline__ uint32_t pair_step(Fs32 &s, uint32_t lutb, uint32_t X, float &w0, float &w1) {
    fs_refill(s);  // two codes take at most 24 bits; a refill leaves at least 33
    const uint32_t e1 = lut_at(s, lutb);
    fs_consume(s, e1);
    const uint32_t e2 = lut_at(s, lutb);
    fs_consume(s, e2);
    return pair_bits<ELEM>(e1, e2, X, w0, w1);
}

// Four codes (two row pairs) on one refill: the refill leaves at least 33 valid bits, which four
// codes (at most 12 bits each) exceed only rarely. No escape branch: an escape yields its
// placeholder, corrected from the block's escape list. A lane that ran past its valid bits (the low seven
// bits of V wrapped: bit 6 set) finds code 3's bit position from the words it inserted and the
// valid count before code 3, reloads its window there from the staged stream and decodes codes 3
// and 4 again. code = shared address of the lane's first code word.
__device__ __forceinline__ void fs_quad(Fs32 &s, uint32_t lutb, uint32_t code, uint32_t (&e)[4]) {
    fs_refill(s);
#pragma unroll
    for (int c = 0; c < 4; c++) {
        e[c] = lut_at(s, lutb);
        fs_consume(s, e[c]);
    }
    if (__any_sync(0xFFFFFFFFu, (s.V & 64u) != 0u) && (s.V & 64u)) {
        const uint32_t V2 = s.V + e[2] + e[3];  // V before code 3 (low seven bits)
        const uint32_t pos = (s.pa - code) * 8u - ((V2 & 127u) + 1u);
        const uint32_t a = code + 4u * (pos >> 5), o = pos & 31u;
        uint32_t w0, w1;
        asm("ld.shared.u32 %0, [%1];" : "=r"(w0) : "r"(a));
        asm("ld.shared.u32 %0, [%1];" : "=r"(w1) : "r"(a + 4));
        s.wh = __funnelshift_l(w1, w0, o);
        s.wl = w1 << o;
        s.V = 63u - o;  // 64 - o >= 33 valid bits
        s.pa = a + 8;
        asm("ld.shared.u32 %0, [%1];" : "=r"(s.nw) : "r"(s.pa));
        e[2] = lut_at(s, lutb);
        fs_consume(s, e[2]);
        e[3] = lut_at(s, lutb);
        fs_consume(s, e[3]);
    }
}

// acc0 += lo(w2) * x, acc1 += hi(w2) * x with BF16 operands and FP32 accumulation: the BF16
// product is exact in FP32, so each equals an FP32 FMA of the widened values.
__device__ __forceinline__ void fma_bf16x2(uint32_t w2, uint32_t x16, float &acc0, float &acc1) {
    asm("{\n\t.reg .b16 lo, hi, xx;\n\t"
        "mov.b32 {lo, hi}, %2;\n\t"
        "cvt.u16.u32 xx, %3;\n\t"
        "fma.rn.f32.bf16 %0, lo, xx, %0;\n\t"
        "fma.rn.f32.bf16 %1, hi, xx, %1;\n\t}"
        : "+f"(acc0), "+f"(acc1)
        : "r"(w2), "r"(x16));
}

// Placeholder that the decoders produce for an escaped element with the given bits: its sign
// and raw mantissa under exponent field 0 (BF16: a subnormal of order 2^-133; fp8: the e4m3
// subnormal +-m 2^-9).
template <int ELEM>
__device__ __forceinline__ float esc_placeholder(uint32_t bits) {
    if (ELEM == 0) return __uint_as_float((bits & 0x807Fu) << 16);
    const float f = (float)(bits & 7u) * 0.001953125f;
    return (bits & 0x80u) ? -f : f;
}

// Adds (w - placeholder) * x to acc[row] for every entry of a block's escape list (`slots`
// words at `list`), the entries spread over the lanes; the transposed reduction then sums them
// with the rows. xb = activations from the block's first column; rows, kc = the block's real
// extent.
template <int ELEM>
__device__ __forceinline__ void esc_correct(const uint32_t *list, uint32_t slots, int lane, const uint16_t *xb,
                                            int rows, int kc, float (&acc)[8], bool &bad) {
    for (uint32_t j = (uint32_t)lane; j < slots; j += 32) {
        const uint32_t e = list[j];
        if (e == kEscPad) continue;
        const uint32_t t = esc_t(e), bits = esc_bits(e);
        const int r = (int)(t & 7u), c = (int)esc_lane(e) * kLaneCols + (int)(t >> 3);
        if (r >= rows || c >= kc) {
            bad = true;
            continue;
        }
        const float xv = __uint_as_float((uint32_t)__ldg(xb + c) << 16);
        const float w = ELEM == 0 ? __uint_as_float(bits << 16) : elem_value<1>(bits >> 7, (bits >> 3) & 15u, bits & 7u);
        const float d = fmaf(w, xv, -(esc_placeholder<ELEM>(bits) * xv));
#pragma unroll
        for (int i = 0; i < 8; i++)
            if (i == r) acc[i] += d;
    }
}

// Four activations (columns c0 .. c0 + 3 of a column block starting at xv) as BF16 pairs;
// columns at or past kc (the block's real columns) read as 0.
__device__ __forceinline__ uint2 x4_load(const uint16_t *xv, int c0, int kc) {
    if (c0 + 4 <= kc) return __ldg(reinterpret_cast<const uint2 *>(xv + c0));
    uint32_t e[4];
#pragma unroll
    for (int j = 0; j < 4; j++) e[j] = c0 + j < kc ? (uint32_t)__ldg(xv + c0 + j) : 0u;
    return make_uint2(e[0] | e[1] << 16, e[2] | e[3] << 16);
}

// Block from its staged region (`bytes` long), all 8 rows real: 4 groups of 4 columns (16 row
// pairs each); the group loop stays rolled so the hot loop fits the instruction cache.
// EDGE: the block's real extent is kc <= 512 columns and rows <= 8 rows, not both full. Every
// lane still holds 128 codes (fillers for elements past K or N). Past K: the real columns'
// mantissa fields sit where they sit in a full block, but the lanes' mantissa regions follow one
// another unless all have the same word count; activations past K read as 0, so the fillers add
// nothing. Past N: each group's fields are gathered into the full-block layout first; the rows
// past N accumulate filler values that are never stored.
template <int ELEM, int NB, bool EDGE = false>
__device__ __forceinline__ void block_fast(const uint8_t *reg, uint32_t bytes, int lane, const uint32_t *lut,
                                           const uint16_t *xb, int64_t ld_x, uint2 (&xq)[NB], float (&acc)[NB][8],
                                           bool &bad, int kc = kCols, int rows = kRows) {
    constexpr int F = ELEM == 0 ? 7 : 3;
    constexpr int MW = ELEM == 0 ? 28 : 12;  // words of a full lane's mantissa region
    constexpr int MWG = MW / 4;              // words per group of 4 columns
    const uint32_t lw = reg[lane];
    uint32_t incl = lw;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        uint32_t o = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        if (lane >= d) incl += o;
    }
    const uint32_t total = __shfl_sync(0xFFFFFFFFu, incl, 31);
    const uint32_t regs = (uint32_t)__cvta_generic_to_shared(reg);
    const uint32_t code = regs + 32 + 4 * (incl - lw);
    // full block: every lane has MW mantissa words, interleaved (word k of lane l at 32k + l)
    const uint32_t man0 = (uint32_t)up16(32 + 4 * (uint64_t)total);
    uint32_t man = regs + man0 + (uint32_t)lane * 4, mstride = 4 * kLanes, esc0 = man0 + kLanes * MW * 4;
    uint32_t mwords = MW;  // this lane's mantissa words (EDGE: only these are read)
    if (EDGE) {
        const int cols = kc - lane * kLaneCols < 0 ? 0 : (kc - lane * kLaneCols > kLaneCols ? kLaneCols : kc - lane * kLaneCols);
        const uint32_t mw = man_words(rows, cols, F);
        mwords = mw;
        uint32_t mincl = mw;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            uint32_t o = __shfl_up_sync(0xFFFFFFFFu, mincl, d);
            if (lane >= d) mincl += o;
        }
        const bool uniform = __all_sync(0xFFFFFFFFu, mw == __shfl_sync(0xFFFFFFFFu, mw, 0));
        if (!uniform) {
            man = regs + man0 + 4 * (mincl - mw);
            mstride = 4;
        }
        esc0 = man0 + 4 * __shfl_sync(0xFFFFFFFFu, mincl, 31);
    }
    Fs32 s;
    {
        uint32_t w0 = 0, w1 = 0;
        if (lw > 0) asm("ld.shared.u32 %0, [%1];" : "=r"(w0) : "r"(code));
        if (lw > 1) asm("ld.shared.u32 %0, [%1];" : "=r"(w1) : "r"(code + 4));
        s.wh = w0;
        s.wl = w1;
        s.pa = code + 8;
        s.V = 63u;
        asm("ld.shared.u32 %0, [%1];" : "=r"(s.nw) : "r"(s.pa));
    }
    const uint32_t lutb = (uint32_t)__cvta_generic_to_shared(lut);
#pragma unroll 1
    for (int g = 0; g < 4; g++) {
        uint2 xn[NB];
        uint32_t x16[NB][4];  // the group's four activations of each vector: BF16 bits (BF16 path)
        float xf[NB][4];      // and FP32 (fp8 path)
#pragma unroll
        for (int v = 0; v < NB; v++) {
            if (EDGE) xn[v] = x4_load(xb + v * ld_x, lane * kLaneCols + 4 * (g < 3 ? g + 1 : 3), kc);
            else xn[v] = __ldg(reinterpret_cast<const uint2 *>(xb + v * ld_x + lane * kLaneCols) + (g < 3 ? g + 1 : 3));
            x16[v][0] = xq[v].x & 0xFFFFu;
            x16[v][1] = xq[v].x >> 16;
            x16[v][2] = xq[v].y & 0xFFFFu;
            x16[v][3] = xq[v].y >> 16;
            xf[v][0] = __uint_as_float(xq[v].x << 16);
            xf[v][1] = __uint_as_float(xq[v].x & 0xFFFF0000u);
            xf[v][2] = __uint_as_float(xq[v].y << 16);
            xf[v][3] = __uint_as_float(xq[v].y & 0xFFFF0000u);
        }
        uint32_t mw[MWG];
        if (EDGE && rows < kRows) {
            group_fields_ragged<F>(man, mstride, mwords, g, rows, mw);
        } else {
#pragma unroll
            for (int i = 0; i < MWG; i++) {
                const uint32_t kw = (uint32_t)(MWG * g + i);
                mw[i] = 0;
                if (!EDGE || kw < mwords)
                    asm("ld.shared.u32 %0, [%1];" : "=r"(mw[i]) : "r"(man + (EDGE ? mstride : 4 * kLanes) * kw));
            }
        }
        uint32_t e4[4];  // table entries of row pairs q, q + 1 (q even)
#pragma unroll
        for (int q = 0; q < 16; q++) {
            const int pp = q & 3;
            const uint32_t X = xpair<F>(mw, q);
            float w0, w1;
            if ((q & 1) == 0) fs_quad(s, lutb, code, e4);
            const uint32_t w2 = pair_bits<ELEM>(e4[2 * (q & 1)], e4[2 * (q & 1) + 1], X, w0, w1);
#pragma unroll
            for (int v = 0; v < NB; v++) {
                if (ELEM == 0) {
                    fma_bf16x2(w2, x16[v][q >> 2], acc[v][2 * pp], acc[v][2 * pp + 1]);
                } else {
                    const float xc = xf[v][q >> 2];
                    const float2 r = __ffma2_rn(make_float2(w0, w1), make_float2(xc, xc),
                                                make_float2(acc[v][2 * pp], acc[v][2 * pp + 1]));
                    acc[v][2 * pp] = r.x;
                    acc[v][2 * pp + 1] = r.y;
                }
            }
        }
#pragma unroll
        for (int v = 0; v < NB; v++) xq[v] = xn[v];
    }
    // consumed bits = 32 * words inserted - valid bits
    const uint32_t valid = (s.V & 127u) + 1u;
    const uint32_t inserted = (s.pa - code) * 8u;
    bad |= inserted - valid > 32u * lw;
#pragma unroll
    for (int v = 0; v < NB; v++)
        esc_correct<ELEM>(reinterpret_cast<const uint32_t *>(reg + esc0), esc0 <= bytes ? (bytes - esc0) / 4 : 0, lane,
                          xb + v * ld_x, rows, kc, acc[v], bad);
}

// Any block (edge, or a region too large to stage) from shared or global memory; escaped
// elements contribute the same placeholder as on the fast path, which the list corrects (first,
// so that the list's registers are free before the decode).
template <int ELEM>
__device__ __forceinline__ void block_generic(const uint8_t *reg, uint32_t bytes, int lane, const uint8_t *rexp,
                                              int nr, int rows, uint64_t k, uint64_t cb, const uint16_t *xb,
                                              float (&acc)[8], bool &bad, bool staged = false, uint32_t lutb = 0) {
    constexpr int F = ELEM == 0 ? 7 : 3;
    const int cols = real_cols(k, cb, lane);
    LaneRegion lr = lane_region(reg, bytes, lane, rows, k, cb, F);
    const uint64_t kc = k - cb * kCols;
    esc_correct<ELEM>(lr.esc, lr.slots, lane, xb, rows, kc < (uint64_t)kCols ? (int)kc : kCols, acc, bad);
    const uint16_t *xl = xb + lane * kLaneCols;
    auto fma_elem = [&](int c, int r, uint32_t s, uint32_t v, uint32_t mm, bool esc) {
        const float w = esc ? esc_placeholder<ELEM>(elem_bits<ELEM>(s, 0, mm)) : elem_value<ELEM>(s, v, mm);
        acc[r] = fmaf(w, __uint_as_float((uint32_t)__ldg(xl + c) << 16), acc[r]);
    };
    if (staged) {  // codes through the shared table
        LutStream<ELEM> ls;
        ls.init((uint32_t)__cvta_generic_to_shared(lr.code), lr.nwords, lutb,
                (uint32_t)__cvta_generic_to_shared(reg) + kStageBytes - 4);
        lane_rolled<ELEM>(ls, lr.man, lr.man_stride, rows, cols, nr, rexp, fma_elem);
        bad |= ls.overrun();
    } else {
        LaneStream ls;
        ls.init(lr.code, lr.nwords);
        lane_rolled<ELEM>(ls, lr.man, lr.man_stride, rows, cols, nr, rexp, fma_elem);
        bad |= ls.overrun();
    }
}

// y[v] = W x[v] for NB vectors (1 or 2; vector v at x + v ld_x, its result at y + v ld_y, its
// partial sums at partial + v col_blocks n_pad). RAG: N % 8 != 0, and the blocks of the last row
// block take the fast decoder too, in a kernel of their own so that the others keep their
// registers.
template <int ELEM, int NB, bool RAG = false>
__global__ void __launch_bounds__(GemvCfg<NB>::kWarps * 32, GemvCfg<NB>::kCtas)
    gemv_kernel(Mat m, const uint16_t *__restrict__ x, int64_t ld_x, float *__restrict__ y, int64_t ld_y,
                float *partial, uint32_t *counters, uint64_t n_pad) {
    using C = GemvCfg<NB>;
    // A kernel launched after this one with programmatic stream serialization may start as soon
    // as SMs free up; it waits (griddepcontrol.wait) before touching anything this one writes.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    extern __shared__ __align__(128) uint8_t smem[];
    uint32_t *lut = reinterpret_cast<uint32_t *>(smem);
    uint8_t *rexp = smem + kRexpOff;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t bar0 = smem_u32(smem + kBarOff + warp * 16), bar1 = bar0 + 8;
    uint8_t *stage0 = smem + C::kStageOff + warp * C::kStages * kStageBytes,
            *stage1 = stage0 + (C::kStages - 1) * kStageBytes;

    // Block b goes to CTA b % grid, so every SM gets within one block of the same count.
    const uint64_t total_warps = (uint64_t)gridDim.x * C::kWarps;
    uint64_t b = (uint64_t)blockIdx.x + (uint64_t)gridDim.x * warp;
    uint32_t phase = 0;  // bit i: parity of the next completion of stage i
    bool bad = false, timed_out = false;

    // Region bounds of block bb, read by lane 0 and broadcast.
    auto region = [&](uint64_t bb, const uint8_t *&ptr, uint32_t &bytes) {
        uint32_t s = 0, e = 0;
        if (lane == 0) {
            s = m.tab[bb];
            e = m.tab[bb + 1];
        }
        s = __shfl_sync(0xFFFFFFFFu, s, 0);
        e = __shfl_sync(0xFFFFFFFFu, e, 0);
        ptr = m.data + 16 * (uint64_t)s;
        bytes = 16 * (e - s);
    };
    // reuse = the stage held an earlier region that this warp read through the generic proxy
    auto issue = [&](uint64_t bb, int which, bool reuse) {
        const uint8_t *src;
        uint32_t bytes;
        region(bb, src, bytes);
        if (bytes <= (uint32_t)kStageBytes && lane == 0) {
            const uint32_t bar = which ? bar1 : bar0;
            if (reuse) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_expect_tx(bar, bytes);
            tma_load_1d(smem_u32(which ? stage1 : stage0), src, bytes, bar);
        }
    };

    // The warp's own barriers and first region copy go first, so that the copy is in flight
    // while the CTA builds the decode table.
    if (lane == 0) {
        mbar_init(bar0);
        mbar_init(bar1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    if (b < m.nb) issue(b, 0, false);
    load_rank_table(m, rexp);
    build_lut<ELEM>(m, lut);
    __syncthreads();
    // Up to here only the matrix and the kernel parameters were read. x, the workspace and y may
    // belong to the kernel before this one on the stream: wait for it to complete.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    for (int it = 0; b < m.nb; it++) {
        const int cur = C::kStages == 2 ? (it & 1) : 0;
        const uint64_t nxt = b + total_warps;
        __syncwarp();
        if (C::kStages == 2) {
            if (nxt < m.nb) issue(nxt, cur ^ 1, it > 0);
        } else if (nxt < m.nb && lane == 0) {
            const uint8_t *nsrc;
            uint32_t nbytes;
            const uint32_t s0 = m.tab[nxt], s1 = m.tab[nxt + 1];
            nsrc = m.data + 16 * (uint64_t)s0;
            nbytes = 16 * (s1 - s0);
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(nsrc), "r"(nbytes) : "memory");
        }
        const uint8_t *src;
        uint32_t bytes;
        region(b, src, bytes);
        const uint8_t *reg = src;
        const bool staged = bytes <= (uint32_t)kStageBytes;
        const uint64_t rb = b / m.cbs, cb = b % m.cbs;
        const int rows = real_rows(m.n, rb);
        const uint64_t kc64 = m.k - cb * kCols;
        const int kc = kc64 < (uint64_t)kCols ? (int)kc64 : kCols;  // the block's real columns
        // the fast decoder; for a block past K or N only when filler codes, which decode to rank
        // 0 with a garbage mantissa, cannot be Inf or NaN (times a zero activation they add 0)
        const bool full = rows == kRows && kc == kCols;
        const bool fast = staged && (RAG || rows == kRows) && (full || m.rank_exp[0] != (ELEM == 0 ? 0xFFu : 0xFu));
        // the fast path's first activations, loaded while the region copy completes
        uint2 xq0[NB];
#pragma unroll
        for (int v = 0; v < NB; v++) {
            xq0[v] = make_uint2(0u, 0u);
            if (fast) xq0[v] = x4_load(x + v * ld_x + cb * kCols, lane * kLaneCols, kc);
        }
        if (staged) {
            const uint32_t bar = cur ? bar1 : bar0;
            if (!mbar_wait(bar, (phase >> cur) & 1u)) {
                timed_out = true;
                break;
            }
            phase ^= 1u << cur;
            reg = cur ? stage1 : stage0;
        }
        float acc[NB][8];
#pragma unroll
        for (int v = 0; v < NB; v++)
#pragma unroll
            for (int r = 0; r < 8; r++) acc[v][r] = 0.0f;
        if (fast && full) {
            block_fast<ELEM, NB>(cur ? stage1 : stage0, bytes, lane, lut, x + cb * kCols, ld_x, xq0, acc, bad);
        } else if (fast) {
            block_fast<ELEM, NB, true>(cur ? stage1 : stage0, bytes, lane, lut, x + cb * kCols, ld_x, xq0, acc, bad, kc,
                                       RAG ? rows : kRows);
        } else {
#pragma unroll
            for (int v = 0; v < NB; v++)
                block_generic<ELEM>(reg, bytes, lane, rexp, m.nr, rows, m.k, cb, x + v * ld_x + cb * kCols, acc[v],
                                    bad, staged, smem_u32(lut));
        }
        const int row_in = ((lane >> 4) & 1) << 2 | ((lane >> 3) & 1) << 1 | ((lane >> 2) & 1);
        const uint64_t row = rb * kRows + (uint64_t)row_in;
        const bool writer = (lane & 3) == 0 && row < m.n;
#pragma unroll
        for (int v = 0; v < NB; v++) {
            const float sum = transpose_reduce(acc[v], lane);
            if (m.cbs == 1) {
                if (writer) y[v * ld_y + (int64_t)row] = ELEM == 0 ? sum : sum * m.scales[row];
            } else {
                if (writer) partial[(v * m.cbs + cb) * n_pad + row] = sum;
            }
        }
        if (m.cbs > 1) {
            __syncwarp();
            uint32_t ticket = 0;
            // Release: the warp's partial sums (ordered before lane 0 by the warp barrier) are
            // visible to whoever takes the last ticket. Acquire: the last taker's lane 0 gets
            // it from the same atomic, and the warp barrier orders the other lanes' loads after.
            if (lane == 0)
                asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], 1;" : "=r"(ticket) : "l"(counters + rb) : "memory");
            ticket = __shfl_sync(0xFFFFFFFFu, ticket, 0);
            if (ticket == (uint32_t)m.cbs - 1) {
                __syncwarp();
                // row lane % 8; lane / 8 sums column blocks lane / 8, + 4, ... (loads in
                // parallel across the warp), then a fixed shuffle order adds the four
                const uint64_t r2 = rb * kRows + (uint64_t)(lane & 7);
#pragma unroll
                for (int v = 0; v < NB; v++) {
                    const float *pv = partial + (uint64_t)v * m.cbs * n_pad;
                    float s = 0.0f;
                    if (r2 < m.n)
                        for (uint64_t c2 = (uint64_t)(lane >> 3); c2 < m.cbs; c2 += 4) s += __ldcg(pv + c2 * n_pad + r2);
                    s += __shfl_xor_sync(0xFFFFFFFFu, s, 8);
                    s += __shfl_xor_sync(0xFFFFFFFFu, s, 16);
                    if (lane < kRows && r2 < m.n) y[v * ld_y + (int64_t)r2] = ELEM == 0 ? s : s * m.scales[r2];
                }
                if (lane == 0) counters[rb] = 0;
            }
        }
        if (C::kStages == 1) {
            __syncwarp();
            if (nxt < m.nb) issue(nxt, 0, true);
        }
        b = nxt;
    }
    if (timed_out) {
        raise_error(kErrTimeout);
        // let this warp's own copies land before the CTA's shared memory goes away
        mbar_wait(bar0, phase & 1u);
        if (C::kStages == 2) mbar_wait(bar1, (phase >> 1) & 1u);
    }
    if (bad) raise_error(kErrFormat);
}

// =================================================================== small-batch GEMV
// Y[v] = W x[v] for up to 16 activation vectors (a few tokens per step) in one pass over the
// matrix: each weight is decoded once, as in the single-vector GEMV, and the products with all
// vectors are a dense contraction per block ([vectors x 512] . [512 x 8 rows]), done by the
// tensor cores. Per group of 4 columns the warp writes its decoded 8 x 128 tile to shared memory
// and runs eight m16n8k16 BF16 products with FP32 accumulation; the vectors are the M side, so
// any count up to 16 costs about the same. Escaped elements are written into the tile with their
// true values, so no correction is needed. Each CTA takes a contiguous range of blocks in
// column-block-major order and stages the activations of its (at most two) column blocks in
// shared memory once; 20 warps per SM with up to 102 registers.
#ifndef NWC_BATCH_WARPS
#define NWC_BATCH_WARPS 20
#endif
constexpr int kBatchWarps = NWC_BATCH_WARPS;
constexpr int kTileRow = 32 * 8 + 32;  // 32 lanes x 4 columns x BF16, padded by 32 bytes
constexpr int kTileBytes = 8 * kTileRow;
constexpr int kBatchStageOff = (kBarOff + kBatchWarps * 2 * 8 + 127) / 128 * 128;
constexpr int kBatchTileOff = kBatchStageOff + kBatchWarps * kStageBytes;
constexpr int kBatchMax = 16;
constexpr int kXSlice = kBatchMax * kCols * 2;  // one column block of every vector, BF16
constexpr int kBatchXOff = kBatchTileOff + kBatchWarps * kTileBytes;
constexpr int kBatchSmem = kBatchXOff + 2 * kXSlice;
static_assert(kBatchSmem <= 232448, "shared memory per CTA");
static_assert(kBatchMax == NWC_GEMV_BATCH_MAX, "vectors per call");

// Byte offset in a staged activation slice of vector v, columns 4u..4u+3 of the column block
// (u = 4 * lane + group): 8-byte unit u ^ (v & 3), so the operand loads of one product (vectors
// gid, four lanes) fall in 16 distinct units per half-warp.
__device__ __forceinline__ uint32_t xs_off(uint32_t v, uint32_t u) { return v * (uint32_t)(kCols * 2) + 8u * (u ^ (v & 3u)); }

// Byte offset in a warp's tile of row r, lane L's 4 columns (8 bytes). Rows are 288 bytes apart
// (36 8-byte units, 4 mod 16): a row's stores (32 consecutive units) and an mma operand load
// (rows 0..3 or 4..7 of a half-warp, four consecutive lanes each) both touch 16 distinct bank
// pairs per half-warp, and the operand of product j sits 32 j bytes after that of product 0.
__device__ __forceinline__ uint32_t tile_off(uint32_t r, uint32_t L) { return r * (uint32_t)kTileRow + 8u * L; }

// d += A . B for one m16n8k16 tile: a0..a3 and b0, b1 in the PTX fragment layout (BF16 pairs),
// FP32 accumulators.
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two FP32 values (exact in BF16) packed as BF16x2, lo in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// BF16 bits of an escaped element's true value (fp8: the e4m3 value, exact in BF16).
template <int ELEM>
__device__ __forceinline__ uint32_t esc_bf16(uint32_t bits) {
    if (ELEM == 0) return bits & 0xFFFFu;
    return __float_as_uint(elem_value<1>(bits >> 7, (bits >> 3) & 15u, bits & 7u)) >> 16;
}

// Interior block from its staged region, all vectors: d[0..3] receive the block's sums in the
// m16n8k16 accumulator layout (vector lane/4 rows 2(lane%4), +1 in d0, d1; vector lane/4 + 8 in
// d2, d3). The activations come from the CTA's staged slice at xs (shared address) when the
// block's column block is staged, else from global memory at x0/x1 (this thread's two vectors
// from the block's first column); v0/v1: those vectors exist (< nb).
// EDGE: the block's real extent is kc <= 512 columns and rows <= 8 rows, not both full. Past K:
// lane-contiguous mantissa regions unless all lanes have the same word count, and activations
// past K are 0 (the staged slice is zero-filled there, global loads are masked), so filler codes
// add nothing. Past N: each group's fields are gathered into the full-block layout first; the
// tile rows past N hold filler values whose products are never stored.
template <int ELEM, bool EDGE = false>
__device__ __forceinline__ void block_mma(const uint8_t *reg, uint32_t bytes, int lane, const uint32_t *lut,
                                          uint32_t tile, bool staged_x, uint32_t xs, const uint16_t *x0,
                                          const uint16_t *x1, bool v0, bool v1, float (&d)[4], bool &bad,
                                          int kc = kCols, int rows = kRows) {
    constexpr int F = ELEM == 0 ? 7 : 3;
    constexpr int MW = ELEM == 0 ? 28 : 12;
    constexpr int MWG = MW / 4;
    const uint32_t lw = reg[lane];
    uint32_t incl = lw;
#pragma unroll
    for (int dd = 1; dd < 32; dd <<= 1) {
        uint32_t o = __shfl_up_sync(0xFFFFFFFFu, incl, dd);
        if (lane >= dd) incl += o;
    }
    const uint32_t total = __shfl_sync(0xFFFFFFFFu, incl, 31);
    const uint32_t regs = (uint32_t)__cvta_generic_to_shared(reg);
    const uint32_t code = regs + 32 + 4 * (incl - lw);
    const uint32_t man0 = (uint32_t)up16(32 + 4 * (uint64_t)total);
    uint32_t man = regs + man0 + (uint32_t)lane * 4, mstride = 4 * kLanes, mwords = MW;
    uint32_t esc0 = man0 + kLanes * MW * 4;
    if (EDGE) {
        const int cols = kc - lane * kLaneCols < 0 ? 0 : (kc - lane * kLaneCols > kLaneCols ? kLaneCols : kc - lane * kLaneCols);
        const uint32_t mw = man_words(rows, cols, F);
        mwords = mw;
        uint32_t mincl = mw;
#pragma unroll
        for (int dd = 1; dd < 32; dd <<= 1) {
            uint32_t o = __shfl_up_sync(0xFFFFFFFFu, mincl, dd);
            if (lane >= dd) mincl += o;
        }
        const bool uniform = __all_sync(0xFFFFFFFFu, mw == __shfl_sync(0xFFFFFFFFu, mw, 0));
        if (!uniform) {
            man = regs + man0 + 4 * (mincl - mw);
            mstride = 4;
        }
        esc0 = man0 + 4 * __shfl_sync(0xFFFFFFFFu, mincl, 31);
    }
    Fs32 s;
    {
        uint32_t w0 = 0, w1 = 0;
        if (lw > 0) asm("ld.shared.u32 %0, [%1];" : "=r"(w0) : "r"(code));
        if (lw > 1) asm("ld.shared.u32 %0, [%1];" : "=r"(w1) : "r"(code + 4));
        s.wh = w0;
        s.wl = w1;
        s.pa = code + 8;
        s.V = 63u;
        asm("ld.shared.u32 %0, [%1];" : "=r"(s.nw) : "r"(s.pa));
    }
    const uint32_t lutb = (uint32_t)__cvta_generic_to_shared(lut);
    const uint32_t slots = esc0 <= bytes ? (bytes - esc0) / 4 : 0;
    const uint32_t *list = reinterpret_cast<const uint32_t *>(reg + esc0);
    const uint32_t gid = (uint32_t)lane >> 2, t = (uint32_t)lane & 3u;
    // this thread's B operand of product j in every group: row gid, lane 4j + t (32 j bytes on)
    const uint32_t bbase = tile + tile_off(gid, t);
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll 1
    for (int g = 0; g < 4; g++) {
        uint32_t mw[MWG];
        if (EDGE && rows < kRows) {
            group_fields_ragged<F>(man, mstride, mwords, g, rows, mw);
        } else {
#pragma unroll
            for (int i = 0; i < MWG; i++) {
                const uint32_t kw = (uint32_t)(MWG * g + i);
                mw[i] = 0;
                if (!EDGE || kw < mwords)
                    asm("ld.shared.u32 %0, [%1];" : "=r"(mw[i]) : "r"(man + (EDGE ? mstride : 4 * kLanes) * kw));
            }
        }
        uint32_t w2[16];
#pragma unroll
        for (int q = 0; q < 16; q++) {
            float f0, f1;
            w2[q] = pair_step<ELEM>(s, lutb, xpair<F>(mw, q), f0, f1);
            if (ELEM == 1) w2[q] = pack_bf16x2(f0, f1);
        }
        // rows 2pp (low halves) and 2pp + 1 (high halves) of columns 0..3 (w2[4 c + pp])
#pragma unroll
        for (int pp = 0; pp < 4; pp++) {
            const uint32_t lo0 = __byte_perm(w2[pp], w2[4 + pp], 0x5410), lo1 = __byte_perm(w2[8 + pp], w2[12 + pp], 0x5410);
            const uint32_t hi0 = __byte_perm(w2[pp], w2[4 + pp], 0x7632), hi1 = __byte_perm(w2[8 + pp], w2[12 + pp], 0x7632);
            asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(tile + tile_off(2 * pp, lane)), "r"(lo0), "r"(lo1)
                         : "memory");
            asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(tile + tile_off(2 * pp + 1, lane)), "r"(hi0),
                         "r"(hi1)
                         : "memory");
        }
        __syncwarp();
        // escaped elements of this group: their true values over the placeholders
        for (uint32_t j = (uint32_t)lane; j < slots; j += 32) {
            const uint32_t e = list[j];
            if (e == kEscPad) continue;
            const uint32_t te = esc_t(e), c = te >> 3;
            if ((c >> 2) != (uint32_t)g) continue;
            if (EDGE && ((int)(te & 7u) >= rows || (int)(esc_lane(e) * kLaneCols + c) >= kc)) {
                bad = true;
                continue;
            }
            const uint32_t a = tile + tile_off(te & 7u, esc_lane(e)) + 2u * (c & 3u);
            asm volatile("st.shared.u16 [%0], %1;" ::"r"(a), "h"((unsigned short)esc_bf16<ELEM>(esc_bits(e))) : "memory");
        }
        __syncwarp();
        // A operands: columns 4g..4g+3 of lane 4j + t as BF16 pairs (cols 0, 1 -> k = 2t, 2t + 1;
        // cols 2, 3 -> k = 2t + 8, 2t + 9); B: the same columns of row gid, from the tile. In the
        // staged slice these are units 16 j + 4 t + g, whose swizzle (^ (gid & 3)) touches only the
        // low two bits: product j's A operand sits 128 j bytes after product 0's.
        const uint32_t abase = xs + xs_off(gid, 4u * t + (uint32_t)g);
#pragma unroll
        for (int j = 0; j < 8; j++) {
            const uint32_t L = 4u * (uint32_t)j + t;
            uint32_t b0, b1;
            asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];"
                         : "=r"(b0), "=r"(b1)
                         : "r"(bbase + 32u * (uint32_t)j)
                         : "memory");
            uint2 a = make_uint2(0u, 0u), a8 = make_uint2(0u, 0u);
            if (staged_x) {
                const uint32_t aj = abase + 128u * (uint32_t)j;
                if (v0) asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(a.x), "=r"(a.y) : "r"(aj) : "memory");
                if (v1)
                    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];"
                                 : "=r"(a8.x), "=r"(a8.y)
                                 : "r"(aj + 8u * (uint32_t)kCols * 2u)
                                 : "memory");
            } else {
                const int col = (int)L * kLaneCols + 4 * g;
                if (v0) a = EDGE ? x4_load(x0, col, kc) : __ldg(reinterpret_cast<const uint2 *>(x0 + col));
                if (v1) a8 = EDGE ? x4_load(x1, col, kc) : __ldg(reinterpret_cast<const uint2 *>(x1 + col));
            }
            mma_bf16(acc[j & 1], a.x, a8.x, a.y, a8.y, b0, b1);
        }
        __syncwarp();
    }
    const uint32_t valid = (s.V & 127u) + 1u;
    const uint32_t inserted = (s.pa - code) * 8u;
    bad |= inserted - valid > 32u * lw;
#pragma unroll
    for (int i = 0; i < 4; i++) d[i] = acc[0][i] + acc[1][i];
}

// RAG: N % 8 != 0, and the blocks of the last row block take the tensor-core path too, in a kernel
// of their own so that the others keep the regular kernel's code.
template <int ELEM, bool RAG = false>
__global__ void __launch_bounds__(kBatchWarps * 32, 1)
    gemv_batch_kernel(Mat m, const uint16_t *__restrict__ x, int64_t ld_x, int nb, float *__restrict__ y,
                      int64_t ld_y, float *partial, uint32_t *counters, uint64_t n_pad) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    extern __shared__ __align__(128) uint8_t smem[];
    uint32_t *lut = reinterpret_cast<uint32_t *>(smem);
    uint8_t *rexp = smem + kRexpOff;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t bar0 = smem_u32(smem + kBarOff + warp * 16);
    uint8_t *stage = smem + kBatchStageOff + warp * kStageBytes;
    const uint32_t tile = smem_u32(smem + kBatchTileOff + warp * kTileBytes);
    const uint32_t xs0 = smem_u32(smem + kBatchXOff);
    // The CTA takes a contiguous range of positions p in column-block-major order (block
    // (rb, cb) at p = cb * rbs + rb), so its warps mostly share one column block, whose
    // activations it stages once in shared memory (two slices: the range may cross one
    // boundary). Warp w takes positions start + w, start + w + warps, ...
    const uint64_t per = (m.nb + gridDim.x - 1) / gridDim.x;
    const uint64_t start = (uint64_t)blockIdx.x * per;
    const uint64_t end = start + per < m.nb ? start + per : m.nb;
    const uint64_t cb_first = start / m.rbs;
    uint64_t p = start + (uint64_t)warp;
    // (rb, cb) of position p, stepped without division; (rbn, cbn) of the next position
    uint64_t cb = p / m.rbs, rb = p % m.rbs;
    auto step = [&](uint64_t &r, uint64_t &c) {
        r += kBatchWarps;
        while (r >= m.rbs) {
            r -= m.rbs;
            c += 1;
        }
    };
    uint32_t phase = 0;
    bool bad = false, timed_out = false;
    const int gid = lane >> 2, t = lane & 3;

    auto region = [&](uint64_t bb, const uint8_t *&ptr, uint32_t &bytes) {
        uint32_t s0 = 0, s1 = 0;
        if (lane == 0) {
            s0 = m.tab[bb];
            s1 = m.tab[bb + 1];
        }
        s0 = __shfl_sync(0xFFFFFFFFu, s0, 0);
        s1 = __shfl_sync(0xFFFFFFFFu, s1, 0);
        ptr = m.data + 16 * (uint64_t)s0;
        bytes = 16 * (s1 - s0);
    };
    auto issue = [&](uint64_t bb, bool reuse) {
        const uint8_t *src;
        uint32_t bytes;
        region(bb, src, bytes);
        if (bytes <= (uint32_t)kStageBytes && lane == 0) {
            if (reuse) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_expect_tx(bar0, bytes);
            tma_load_1d(smem_u32(stage), src, bytes, bar0);
        }
    };
    // result of vector v, row `row` (< n) of column block cb
    auto emit = [&](int v, uint64_t row, uint64_t cb, float val) {
        if (m.cbs == 1) y[(int64_t)v * ld_y + (int64_t)row] = ELEM == 0 ? val : val * m.scales[row];
        else partial[((uint64_t)v * m.cbs + cb) * n_pad + row] = val;
    };

    if (lane == 0) {
        mbar_init(bar0);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    if (p < end) issue(rb * m.cbs + cb, false);
    load_rank_table(m, rexp);
    build_lut<ELEM>(m, lut);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // stage the activations of column blocks cb_first and cb_first + 1 (whole 16-byte pieces
    // inside K; the rest of a slice is only read for interior blocks, which lie inside K)
    for (uint32_t i = threadIdx.x; i < 2u * (uint32_t)nb * (kCols / 8); i += blockDim.x) {
        const uint32_t slot = i / ((uint32_t)nb * (kCols / 8)), rem = i % ((uint32_t)nb * (kCols / 8));
        const uint32_t v = rem / (kCols / 8), c8 = rem % (kCols / 8);  // columns 8 c8 .. 8 c8 + 7
        const uint64_t col = (cb_first + slot) * kCols + 8 * (uint64_t)c8;
        uint4 q = make_uint4(0u, 0u, 0u, 0u);  // past K: zeros (the fillers of a ragged K meet them)
        if (col + 8 <= m.k) {
            q = __ldg(reinterpret_cast<const uint4 *>(x + (int64_t)v * ld_x + (int64_t)col));
        } else if (col < m.k) {
            uint32_t e[8];
#pragma unroll
            for (int j = 0; j < 8; j++) e[j] = col + j < m.k ? (uint32_t)__ldg(x + (int64_t)v * ld_x + (int64_t)(col + j)) : 0u;
            q = make_uint4(e[0] | e[1] << 16, e[2] | e[3] << 16, e[4] | e[5] << 16, e[6] | e[7] << 16);
        }
        // columns 8 c8.. are lane c8 / 2, groups 2 (c8 & 1) and 2 (c8 & 1) + 1: units 2 c8, 2 c8 + 1
        const uint32_t xs = xs0 + slot * (uint32_t)kXSlice;
        asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(xs + xs_off(v, 2 * c8)), "r"(q.x), "r"(q.y) : "memory");
        asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(xs + xs_off(v, 2 * c8 + 1)), "r"(q.z), "r"(q.w) : "memory");
    }
    __syncthreads();

    while (p < end) {
        const uint64_t b = rb * m.cbs + cb;
        const uint64_t pn = p + kBatchWarps;
        uint64_t rbn = rb, cbn = cb;
        step(rbn, cbn);
        const uint64_t bn = rbn * m.cbs + cbn;
        __syncwarp();
        if (pn < end && lane == 0) {
            const uint32_t s0 = m.tab[bn], s1 = m.tab[bn + 1];
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(m.data + 16 * (uint64_t)s0),
                         "r"(16 * (s1 - s0))
                         : "memory");
        }
        const uint8_t *src;
        uint32_t bytes;
        region(b, src, bytes);
        const uint8_t *reg = src;
        const bool staged = bytes <= (uint32_t)kStageBytes;
        if (staged) {
            if (!mbar_wait(bar0, phase & 1u)) {
                timed_out = true;
                break;
            }
            phase ^= 1u;
            reg = stage;
        }
        const int rows = real_rows(m.n, rb);
        const uint64_t kc64 = m.k - cb * kCols;
        const int kc = kc64 < (uint64_t)kCols ? (int)kc64 : kCols;  // the block's real columns
        // the tensor-core path; for a block past K or N only when filler codes cannot decode to
        // Inf or NaN (times a zero activation they add 0)
        const bool full = rows == kRows && kc == kCols;
        if (staged && (RAG || rows == kRows) && (full || m.rank_exp[0] != (ELEM == 0 ? 0xFFu : 0xFu))) {
            const uint16_t *xc = x + cb * kCols;
            const bool v0 = gid < nb, v1 = gid + 8 < nb;
            const uint16_t *x0 = xc + (int64_t)(v0 ? gid : 0) * ld_x;
            const uint16_t *x1 = xc + (int64_t)(v1 ? gid + 8 : 0) * ld_x;
            const bool staged_x = cb == cb_first || cb == cb_first + 1;
            const uint32_t xs = xs0 + (cb == cb_first ? 0u : (uint32_t)kXSlice);
            float d[4];
            if (full) block_mma<ELEM>(stage, bytes, lane, lut, tile, staged_x, xs, x0, x1, v0, v1, d, bad);
            else block_mma<ELEM, true>(stage, bytes, lane, lut, tile, staged_x, xs, x0, x1, v0, v1, d, bad, kc,
                                       RAG ? rows : kRows);
            const uint64_t r0 = rb * kRows + 2 * (uint64_t)t;
            const bool in0 = !RAG || r0 < m.n, in1 = !RAG || r0 + 1 < m.n;
            if (v0) {
                if (in0) emit(gid, r0, cb, d[0]);
                if (in1) emit(gid, r0 + 1, cb, d[1]);
            }
            if (v1) {
                if (in0) emit(gid + 8, r0, cb, d[2]);
                if (in1) emit(gid + 8, r0 + 1, cb, d[3]);
            }
        } else {
            // regions too large to stage, and edge blocks whose fillers could decode to Inf or NaN:
            // the single-vector decoder per vector
            const int row_in = ((lane >> 4) & 1) << 2 | ((lane >> 3) & 1) << 1 | ((lane >> 2) & 1);
            const uint64_t row = rb * kRows + (uint64_t)row_in;
            for (int v = 0; v < nb; v++) {
                float a1[8];
#pragma unroll
                for (int r = 0; r < 8; r++) a1[r] = 0.0f;
                block_generic<ELEM>(reg, bytes, lane, rexp, m.nr, rows, m.k, cb, x + (int64_t)v * ld_x + cb * kCols,
                                    a1, bad, staged, smem_u32(lut));
                const float sum = transpose_reduce(a1, lane);
                if ((lane & 3) == 0 && row < m.n) emit(v, row, cb, sum);
            }
        }
        if (m.cbs > 1) {
            __syncwarp();
            uint32_t ticket = 0;
            // release / acquire as in the single-vector GEMV
            if (lane == 0)
                asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], 1;" : "=r"(ticket) : "l"(counters + rb) : "memory");
            ticket = __shfl_sync(0xFFFFFFFFu, ticket, 0);
            if (ticket == (uint32_t)m.cbs - 1) {
                __syncwarp();
                // (vector, row) pairs i, vector i / 8, row i % 8, summed over the column blocks in a
                // fixed order with all loads in flight together. Up to 16 pairs (nb <= 2): lanes
                // i + np * sub (np = 8 or 16) sum column blocks sub, sub + 32 / np, ... and two or
                // one shuffle steps add those; more pairs: lane sums pairs lane + 32 k whole.
                const int pairs = nb * kRows;
                if (pairs <= 16) {
                    const int np = pairs <= 8 ? 8 : 16, S = 32 / np;
                    const int i = lane & (np - 1), sub = lane / np;
                    const uint64_t r2 = rb * kRows + (uint64_t)(i & 7);
                    const bool live = i < pairs && r2 < m.n;
                    const float *pp = partial + (uint64_t)(i >> 3) * m.cbs * n_pad + r2;
                    float sv = 0.0f;
#pragma unroll 4
                    for (uint64_t c2 = (uint64_t)sub; c2 < m.cbs; c2 += (uint64_t)S)
                        if (live) sv += __ldcg(pp + c2 * n_pad);
                    if (S == 4) sv += __shfl_xor_sync(0xFFFFFFFFu, sv, 8);
                    sv += __shfl_xor_sync(0xFFFFFFFFu, sv, 16);
                    if (sub == 0 && live)
                        y[(int64_t)(i >> 3) * ld_y + (int64_t)r2] = ELEM == 0 ? sv : sv * m.scales[r2];
                } else {
                    float sv[kBatchMax * kRows / 32];
                    bool live[kBatchMax * kRows / 32];
                    const float *pp[kBatchMax * kRows / 32];
#pragma unroll
                    for (int k2 = 0; k2 < kBatchMax * kRows / 32; k2++) {
                        const int i = lane + 32 * k2, v = i >> 3;
                        const uint64_t r2 = rb * kRows + (uint64_t)(i & 7);
                        live[k2] = v < nb && r2 < m.n;
                        pp[k2] = partial + (uint64_t)v * m.cbs * n_pad + r2;
                        sv[k2] = 0.0f;
                    }
#pragma unroll 4
                    for (uint64_t c2 = 0; c2 < m.cbs; c2++) {
#pragma unroll
                        for (int k2 = 0; k2 < kBatchMax * kRows / 32; k2++)
                            if (live[k2]) sv[k2] += __ldcg(pp[k2] + c2 * n_pad);
                    }
#pragma unroll
                    for (int k2 = 0; k2 < kBatchMax * kRows / 32; k2++) {
                        if (!live[k2]) continue;
                        const int i = lane + 32 * k2, v = i >> 3;
                        const uint64_t r2 = rb * kRows + (uint64_t)(i & 7);
                        y[(int64_t)v * ld_y + (int64_t)r2] = ELEM == 0 ? sv[k2] : sv[k2] * m.scales[r2];
                    }
                }
                if (lane == 0) counters[rb] = 0;
            }
        }
        __syncwarp();
        if (pn < end) issue(bn, true);
        p = pn;
        rb = rbn;
        cb = cbn;
    }
    if (timed_out) {
        raise_error(kErrTimeout);
        mbar_wait(bar0, phase & 1u);
    }
    if (bad) raise_error(kErrFormat);
}

// =================================================================== decode and gather
// The pages run dequantization and the tied lm_head's embedding lookup on the GEMV's decoder;
// here too: the same CTA
// layout, table and staged regions as the GEMV. MODE 0 decodes every block to BF16 (fp8: e4m3
// bytes); MODE 1 writes, for each id, that row of the block row, one block per warp item.

// One row pair of the unpack path: returns rows (2pp, 2pp+1) at one column as two 16-bit
// halves (BF16 bits; fp8: the e4m3 code in each half's high byte) and adds both entries to
// `flags`, whose top byte then counts the lane's escapes.
template <int ELEM>
__device__ __forceinline__ uint32_t unpack_pair(Fs32 &s, uint32_t lutb, uint32_t X, uint32_t &flags) {
    fs_refill(s);
    const uint32_t e1 = lut_at(s, lutb);
    fs_consume(s, e1);
    const uint32_t e2 = lut_at(s, lutb);
    fs_consume(s, e2);
    flags += e1 + e2;
    const uint32_t e = __byte_perm(e1, e2, 0x5410);
    return ELEM == 0 ? (e & 0xFF80FF80u) | (X & 0x007F007Fu) : (e & 0xFF80FF80u) | ((X & 0x00070007u) << 8);
}

// Row word of 4 columns from the group's pairs p[c4 * 4 + pp]: BF16 rows give two words (cols
// 0-1, 2-3), fp8 rows one word of four bytes. hi selects row 2pp + 1.
template <int ELEM>
__device__ __forceinline__ uint2 row_words(uint32_t a, uint32_t b, uint32_t c, uint32_t d, bool hi) {
    if (ELEM == 0) {
        const uint32_t sel = hi ? 0x7632u : 0x5410u;
        return make_uint2(__byte_perm(a, b, sel), __byte_perm(c, d, sel));
    }
    const uint32_t sel = hi ? 0x0073u : 0x0051u;
    return make_uint2(__byte_perm(__byte_perm(a, b, sel), __byte_perm(c, d, sel), 0x5410), 0u);
}

// One lane's 16-column row segment (BF16: 8 words, fp8: 4 words) to out[at ..] with stores of
// vec bytes (16, 8 or 4: out and the row stride keep that alignment), else element-wise.
template <int ELEM>
__device__ __forceinline__ void store_row16(void *out, uint64_t at, const uint32_t (&w)[8], int vec) {
    constexpr int NW = ELEM == 0 ? 8 : 4;  // words in the segment
    void *o = ELEM == 0 ? static_cast<void *>(static_cast<uint16_t *>(out) + at)
                        : static_cast<void *>(static_cast<uint8_t *>(out) + at);
    if (vec == 16) {
#pragma unroll
        for (int i = 0; i < NW / 4; i++)
            reinterpret_cast<uint4 *>(o)[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
    } else if (vec == 8) {
#pragma unroll
        for (int i = 0; i < NW / 2; i++) reinterpret_cast<uint2 *>(o)[i] = make_uint2(w[2 * i], w[2 * i + 1]);
    } else if (vec == 4) {
#pragma unroll
        for (int i = 0; i < NW; i++) reinterpret_cast<uint32_t *>(o)[i] = w[i];
    } else if (ELEM == 0) {
#pragma unroll
        for (int i = 0; i < 16; i++) static_cast<uint16_t *>(o)[i] = (uint16_t)(w[i >> 1] >> (16 * (i & 1)));
    } else {
#pragma unroll
        for (int i = 0; i < 16; i++) static_cast<uint8_t *>(o)[i] = (uint8_t)(w[i >> 2] >> (8 * (i & 3)));
    }
}

// The first `cols` columns (< 16) of a lane's row segment, element by element.
template <int ELEM>
__device__ __forceinline__ void store_row_part(void *out, uint64_t at, const uint32_t (&w)[8], int cols) {
#pragma unroll
    for (int i = 0; i < 16; i++) {
        if (i >= cols) break;
        if (ELEM == 0) static_cast<uint16_t *>(out)[at + i] = (uint16_t)(w[i >> 1] >> (16 * (i & 1)));
        else static_cast<uint8_t *>(out)[at + i] = (uint8_t)(w[i >> 2] >> (8 * (i & 3)));
    }
}

// Block from its staged region, all 8 rows real. Decode writes rows row0 .. row0 + 7; gather
// writes row `want` of the block to output row row0. col0 = the lane's first column. EDGE: the
// block's real extent is kc <= 512 columns and rows <= 8 rows, not both full: lane-contiguous
// mantissa regions unless all lanes have the same word count, the fields of a row-ragged block
// gathered into the full-block layout per group, and only real elements written.
template <int ELEM, int MODE, bool EDGE = false>
__device__ __forceinline__ void unpack_fast(const uint8_t *reg, uint32_t bytes, int lane, const uint32_t *lut,
                                            void *out, int64_t ld_out, uint64_t row0, uint64_t col0, int want,
                                            int vec, bool &bad, int kc = kCols, int rows = kRows) {
    constexpr int F = ELEM == 0 ? 7 : 3;
    constexpr int MW = ELEM == 0 ? 28 : 12;
    constexpr int MWG = MW / 4;
    const uint32_t lw = reg[lane];
    uint32_t incl = lw;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        uint32_t o = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        if (lane >= d) incl += o;
    }
    const uint32_t total = __shfl_sync(0xFFFFFFFFu, incl, 31);
    const uint32_t regs = (uint32_t)__cvta_generic_to_shared(reg);
    const uint32_t code = regs + 32 + 4 * (incl - lw);
    // full block: every lane has MW mantissa words, interleaved (word k of lane l at 32k + l)
    const uint32_t man0 = (uint32_t)up16(32 + 4 * (uint64_t)total);
    uint32_t man = regs + man0 + (uint32_t)lane * 4, mstride = 4 * kLanes, esc0e = 0;
    uint32_t mwords = MW;
    int cols = kLaneCols;
    if (EDGE) {
        cols = kc - lane * kLaneCols < 0 ? 0 : (kc - lane * kLaneCols > kLaneCols ? kLaneCols : kc - lane * kLaneCols);
        const uint32_t mw = man_words(rows, cols, F);
        mwords = mw;
        uint32_t mincl = mw;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            uint32_t o = __shfl_up_sync(0xFFFFFFFFu, mincl, d);
            if (lane >= d) mincl += o;
        }
        const bool uniform = __all_sync(0xFFFFFFFFu, mw == __shfl_sync(0xFFFFFFFFu, mw, 0));
        if (!uniform) {
            man = regs + man0 + 4 * (mincl - mw);
            mstride = 4;
        }
        esc0e = man0 + 4 * __shfl_sync(0xFFFFFFFFu, mincl, 31);
    }
    Fs32 s;
    {
        uint32_t w0 = 0, w1 = 0;
        if (lw > 0) asm("ld.shared.u32 %0, [%1];" : "=r"(w0) : "r"(code));
        if (lw > 1) asm("ld.shared.u32 %0, [%1];" : "=r"(w1) : "r"(code + 4));
        s.wh = w0;
        s.wl = w1;
        s.pa = code + 8;
        s.V = 63u;
        asm("ld.shared.u32 %0, [%1];" : "=r"(s.nw) : "r"(s.pa));
    }
    const uint32_t lutb = (uint32_t)__cvta_generic_to_shared(lut);
    uint32_t flags = 0;
    const int wpp = want >> 1;
    const bool whi = want & 1;
    // the lane's output tile: o[r][k] = row r, words k (BF16: 2 columns a word, fp8: 4)
    uint32_t o[MODE == 0 ? 8 : 1][8];
    auto group = [&](int g) {
        uint32_t mw[MWG];
        if (EDGE && rows < kRows) {
            group_fields_ragged<F>(man, mstride, mwords, g, rows, mw);
        } else {
#pragma unroll
            for (int i = 0; i < MWG; i++) {
                const uint32_t kw = (uint32_t)(MWG * g + i);
                mw[i] = 0;
                if (!EDGE || kw < mwords)
                    asm("ld.shared.u32 %0, [%1];" : "=r"(mw[i]) : "r"(man + (EDGE ? mstride : 4 * kLanes) * kw));
            }
        }
        uint32_t p[16];  // p[c4 * 4 + pp]: rows (2pp, 2pp + 1) at column 4g + c4
#pragma unroll
        for (int q = 0; q < 16; q++) p[q] = unpack_pair<ELEM>(s, lutb, xpair<F>(mw, q), flags);
        if (MODE == 0) {  // g static here (unrolled)
#pragma unroll
            for (int pp = 0; pp < 4; pp++) {
                const uint2 lo = row_words<ELEM>(p[pp], p[4 + pp], p[8 + pp], p[12 + pp], false);
                const uint2 hi = row_words<ELEM>(p[pp], p[4 + pp], p[8 + pp], p[12 + pp], true);
                if (ELEM == 0) {
                    o[2 * pp][2 * g] = lo.x;
                    o[2 * pp][2 * g + 1] = lo.y;
                    o[2 * pp + 1][2 * g] = hi.x;
                    o[2 * pp + 1][2 * g + 1] = hi.y;
                } else {
                    o[2 * pp][g] = lo.x;
                    o[2 * pp + 1][g] = hi.x;
                }
            }
        } else {  // g dynamic: the wanted row's words shift in from the top
            uint32_t v[4];
#pragma unroll
            for (int c4 = 0; c4 < 4; c4++)
                v[c4] = wpp == 0 ? p[c4 * 4] : (wpp == 1 ? p[c4 * 4 + 1] : (wpp == 2 ? p[c4 * 4 + 2] : p[c4 * 4 + 3]));
            const uint2 wd = row_words<ELEM>(v[0], v[1], v[2], v[3], whi);
            if (ELEM == 0) {
#pragma unroll
                for (int i = 0; i < 6; i++) o[0][i] = o[0][i + 2];
                o[0][6] = wd.x;
                o[0][7] = wd.y;
            } else {
#pragma unroll
                for (int i = 0; i < 3; i++) o[0][i] = o[0][i + 1];
                o[0][3] = wd.x;
            }
        }
    };
    if (MODE == 0) {
#pragma unroll
        for (int g = 0; g < 4; g++) group(g);
    } else {
#pragma unroll 1
        for (int g = 0; g < 4; g++) group(g);
    }
    if (!EDGE || cols == kLaneCols) {
        if (MODE == 0) {
#pragma unroll
            for (int r = 0; r < 8; r++)
                if (!EDGE || r < rows) store_row16<ELEM>(out, (row0 + (uint64_t)r) * (uint64_t)ld_out + col0, o[r], vec);
        } else {
            store_row16<ELEM>(out, row0 * (uint64_t)ld_out + col0, o[0], vec);
        }
    } else if (cols > 0) {
        if (MODE == 0) {
#pragma unroll
            for (int r = 0; r < 8; r++)
                if (r < rows) store_row_part<ELEM>(out, (row0 + (uint64_t)r) * (uint64_t)ld_out + col0, o[r], cols);
        } else {
            store_row_part<ELEM>(out, row0 * (uint64_t)ld_out + col0, o[0], cols);
        }
    }
    const uint32_t valid = (s.V & 127u) + 1u;
    const uint32_t inserted = (s.pa - code) * 8u;
    bad |= inserted - valid > 32u * lw;
    // escaped elements over their placeholders: this lane's slice of the list
    LaneRegion lr;
    const uint32_t esc0 = EDGE ? esc0e : (uint32_t)up16(32 + 4 * (uint64_t)total) + kLanes * MW * 4;
    lr.esc = reinterpret_cast<const uint32_t *>(reg + esc0);
    lr.slots = esc0 <= bytes ? (bytes - esc0) / 4 : 0;
    const uint32_t n_esc = flags >> 24;
    const uint32_t start = esc_slice(lr, n_esc, lane, bad);
    const uint64_t lane_col = col0;
    if (!esc_patch<ELEM>(lr.esc, lr.slots, start, n_esc, lane, rows, cols, MODE == 0 ? -1 : want, out, ld_out,
                         MODE == 0 ? (int64_t)row0 : (int64_t)row0 - want, lane_col))
        bad = true;
}

// Any block (edge, or a region too large to stage), element by element.
template <int ELEM, int MODE>
__device__ __forceinline__ void unpack_generic(const uint8_t *reg, uint32_t bytes, int lane, const uint8_t *rexp,
                                               int nr, int rows, uint64_t k, uint64_t cb, void *out, int64_t ld_out,
                                               uint64_t row0, uint64_t col0, int want, bool &bad, bool staged = false,
                                               uint32_t lutb = 0) {
    constexpr int F = ELEM == 0 ? 7 : 3;
    const int cols = real_cols(k, cb, lane);
    LaneRegion lr = lane_region(reg, bytes, lane, rows, k, cb, F);
    auto put = [&](int c, int r, uint32_t sg, uint32_t v, uint32_t mm, bool esc) {
        if (MODE == 1 && r != want) return;
        const uint64_t row = MODE == 0 ? row0 + (uint64_t)r : row0;
        const uint32_t e = elem_bits<ELEM>(sg, esc ? 0u : v, mm);
        if (ELEM == 0) static_cast<uint16_t *>(out)[row * (uint64_t)ld_out + col0 + (uint64_t)c] = (uint16_t)e;
        else static_cast<uint8_t *>(out)[row * (uint64_t)ld_out + col0 + (uint64_t)c] = (uint8_t)e;
    };
    uint32_t n_esc;
    if (staged) {  // codes through the shared table
        LutStream<ELEM> ls;
        ls.init((uint32_t)__cvta_generic_to_shared(lr.code), lr.nwords, lutb,
                (uint32_t)__cvta_generic_to_shared(reg) + kStageBytes - 4);
        n_esc = lane_rolled<ELEM>(ls, lr.man, lr.man_stride, rows, cols, nr, rexp, put);
        bad |= ls.overrun();
    } else {
        LaneStream ls;
        ls.init(lr.code, lr.nwords);
        n_esc = lane_rolled<ELEM>(ls, lr.man, lr.man_stride, rows, cols, nr, rexp, put);
        bad |= ls.overrun();
    }
    const uint32_t start = esc_slice(lr, n_esc, lane, bad);
    if (!esc_patch<ELEM>(lr.esc, lr.slots, start, n_esc, lane, rows, cols, MODE == 0 ? -1 : want, out, ld_out,
                         MODE == 0 ? (int64_t)row0 : (int64_t)row0 - want, col0))
        bad = true;
}

template <int ELEM, int MODE, bool EDGEK = false>
__global__ void __launch_bounds__(UnpackCfg<MODE>::kWarps * 32, 1)
    unpack_kernel(Mat m, const int32_t *ids, uint64_t n_items, void *out, int64_t ld_out, int vec) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint32_t *lut = reinterpret_cast<uint32_t *>(smem);
    uint8_t *rexp = smem + kRexpOff;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t bar0 = smem_u32(smem + kBarOff + warp * 16);
    uint8_t *stage = smem + UnpackCfg<MODE>::kStageOff + warp * kStageBytes;
    const uint64_t stride = (uint64_t)gridDim.x * UnpackCfg<MODE>::kWarps;
    uint32_t phase = 0;
    bool bad = false, timed_out = false;

    // Work item it -> block b, wanted row (gather) and first output row. Gather ids are read by
    // lane 0 and broadcast; an out-of-range id gives ok = false.
    auto locate = [&](uint64_t it, uint64_t &b, int &want, uint64_t &orow, bool &ok) {
        if (MODE == 0) {
            b = it;
            want = -1;
            orow = (it / m.cbs) * kRows;
            ok = true;
        } else {
            const uint64_t i = it / m.cbs, cb = it % m.cbs;
            int32_t id = 0;
            if (lane == 0) id = ids[i];
            id = __shfl_sync(0xFFFFFFFFu, id, 0);
            ok = id >= 0 && (uint64_t)id < m.n;
            const uint64_t uid = ok ? (uint64_t)id : 0;
            b = (uid >> 3) * m.cbs + cb;
            want = (int)(uid & 7);
            orow = i;
        }
    };
    auto region = [&](uint64_t bb, const uint8_t *&ptr, uint32_t &bytes) {
        uint32_t s0 = 0, s1 = 0;
        if (lane == 0) {
            s0 = m.tab[bb];
            s1 = m.tab[bb + 1];
        }
        s0 = __shfl_sync(0xFFFFFFFFu, s0, 0);
        s1 = __shfl_sync(0xFFFFFFFFu, s1, 0);
        ptr = m.data + 16 * (uint64_t)s0;
        bytes = 16 * (s1 - s0);
    };
    auto issue = [&](uint64_t bb) {
        const uint8_t *src;
        uint32_t bytes;
        region(bb, src, bytes);
        if (bytes <= (uint32_t)kStageBytes && lane == 0) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_expect_tx(bar0, bytes);
            tma_load_1d(smem_u32(stage), src, bytes, bar0);
        }
    };

    if (lane == 0) {
        mbar_init(bar0);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    uint64_t it = (uint64_t)blockIdx.x + (uint64_t)gridDim.x * warp;
    uint64_t b = 0, orow = 0;
    int want = 0;
    bool ok = false;
    if (it < n_items) {
        locate(it, b, want, orow, ok);
        if (ok) issue(b);
    }
    load_rank_table(m, rexp);
    build_lut<ELEM>(m, lut);
    __syncthreads();

    while (it < n_items) {
        const uint64_t nxt = it + stride;
        uint64_t nb_ = 0, norow = 0;
        int nwant = 0;
        bool nok = false;
        if (nxt < n_items) {
            locate(nxt, nb_, nwant, norow, nok);
            if (nok && lane == 0) {
                const uint32_t s0 = m.tab[nb_], s1 = m.tab[nb_ + 1];
                asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(m.data + 16 * (uint64_t)s0),
                             "r"(16 * (s1 - s0))
                             : "memory");
            }
        }
        const uint64_t cb = MODE == 0 ? it % m.cbs : (it % m.cbs);
        const uint64_t col0 = cb * kCols + (uint64_t)lane * kLaneCols;
        if (!ok) {
            // gather id out of range: a zero row, and the error word
            if (lane == 0 && cb == 0) raise_error(kErrId);
            const int cols = real_cols(m.k, cb, lane);
            for (int c = 0; c < cols; c++) {
                if (ELEM == 0) static_cast<uint16_t *>(out)[orow * (uint64_t)ld_out + col0 + c] = 0;
                else static_cast<uint8_t *>(out)[orow * (uint64_t)ld_out + col0 + c] = 0;
            }
        } else {
            const uint8_t *src;
            uint32_t bytes;
            region(b, src, bytes);
            const uint8_t *reg = src;
            const bool staged = bytes <= (uint32_t)kStageBytes;
            if (staged) {
                if (!mbar_wait(bar0, phase & 1u)) {
                    timed_out = true;
                    break;
                }
                phase ^= 1u;
                reg = stage;
            }
            const uint64_t rb = b / m.cbs;
            const int rows = real_rows(m.n, rb);
            const uint64_t kc64 = m.k - cb * kCols;
            const int kc = kc64 < (uint64_t)kCols ? (int)kc64 : kCols;  // the block's real columns
            bool done = false;
            if (rows == kRows && staged && kc == kCols) {
                unpack_fast<ELEM, MODE>(stage, bytes, lane, lut, out, ld_out, orow, col0, want, vec, bad);
                done = true;
            }
            // blocks past K or N: the fast decoder, in a kernel of their own (EDGEK) so that the
            // regular decode and gather keep their registers
            if constexpr (EDGEK) {
                if (!done && staged) {
                    unpack_fast<ELEM, MODE, true>(stage, bytes, lane, lut, out, ld_out, orow, col0, want, vec, bad, kc,
                                                  rows);
                    done = true;
                }
            }
            if (!done)
                unpack_generic<ELEM, MODE>(reg, bytes, lane, rexp, m.nr, rows, m.k, cb, out, ld_out, orow, col0, want,
                                           bad, staged, smem_u32(lut));
        }
        __syncwarp();
        if (nxt < n_items && nok) issue(nb_);
        it = nxt;
        b = nb_;
        want = nwant;
        orow = norow;
        ok = nok;
    }
    if (timed_out) {
        raise_error(kErrTimeout);
        mbar_wait(bar0, phase & 1u);  // let this warp's copy land before shared memory goes away
    }
    if (bad) raise_error(kErrFormat);
}

// =================================================================== host side
int g_sm_count = -1;
std::mutex g_mu;

int sm_count() {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_sm_count < 0) {
        int dev = 0, n = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return 0;
        g_sm_count = n;
    }
    return g_sm_count;
}

template <class K>
bool set_smem(K kernel, int bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) == cudaSuccess;
}

nwc_status launched() { return cudaGetLastError() == cudaSuccess ? NWC_OK : NWC_ERR_CUDA; }

uint64_t pad_rows(const nwc_matrix &m) { return (uint64_t)m.row_blocks * kRows; }

}  // namespace

extern "C" int nwc_sm_count(void) { return sm_count(); }

namespace {
template <int ELEM, int MODE, bool EDGEK = false>
nwc_status launch_unpack(const Mat &m, const int32_t *ids, uint64_t n_items, void *out, int64_t ld_out, int vec,
                         cudaStream_t s) {
    const int sms = sm_count();
    if (sms <= 0) return NWC_ERR_CUDA;
    static bool smem_ok = false;
    static std::once_flag once;
    using C = UnpackCfg<MODE>;
    std::call_once(once, [] { smem_ok = set_smem(unpack_kernel<ELEM, MODE, EDGEK>, C::kSmem); });
    if (!smem_ok) return NWC_ERR_CUDA;
    const int grid = (int)(n_items < (uint64_t)sms ? n_items : (uint64_t)sms);
    unpack_kernel<ELEM, MODE, EDGEK><<<grid, C::kWarps * 32, C::kSmem, s>>>(m, ids, n_items, out, ld_out, vec);
    return launched();
}

// A lane's 16-column row segment is stored with 16-byte stores when every row start keeps that
// alignment (2), with 8-byte stores when rows keep 8-byte alignment (1), else element by element.
// Widest store (16, 8 or 4 bytes; 0: element-wise) that every 16-column row segment of out allows:
// segments start at out + (r ld_out + 16 j) elements.
int vec_ok(const void *out, int64_t ld_out, int elem) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(out);
    const int64_t esz = elem == NWC_ELEM_BF16 ? 2 : 1;
    for (int v = 16; v >= 4; v /= 2)
        if ((a % v) == 0 && ((ld_out * esz) % v) == 0) return v;
    return 0;
}

}  // namespace

extern "C" nwc_status nwc_decode(const nwc_matrix *mp, void *out, int64_t ld_out, float *scales_out, nwc_stream stream) {
    if (!mp || !out || ld_out < mp->k) return NWC_ERR_INVALID_ARG;
    const Mat m = to_mat(*mp);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int vec = vec_ok(out, ld_out, m.elem);
    const bool ragged = (m.k % kCols) != 0 || (m.n % kRows) != 0;
    nwc_status st;
    if (m.elem == NWC_ELEM_BF16)
        st = ragged ? launch_unpack<0, 0, true>(m, nullptr, m.nb, out, ld_out, vec, s)
                    : launch_unpack<0, 0>(m, nullptr, m.nb, out, ld_out, vec, s);
    else
        st = ragged ? launch_unpack<1, 0, true>(m, nullptr, m.nb, out, ld_out, vec, s)
                    : launch_unpack<1, 0>(m, nullptr, m.nb, out, ld_out, vec, s);
    if (st != NWC_OK) return st;
    if (m.elem == NWC_ELEM_FP8_E4M3 && scales_out) {
        if (cudaMemcpyAsync(scales_out, m.scales, 4 * m.n, cudaMemcpyDeviceToDevice, s) != cudaSuccess)
            return NWC_ERR_CUDA;
    }
    return NWC_OK;
}

extern "C" nwc_status nwc_gather(const nwc_matrix *mp, const int32_t *ids, int64_t n_ids, void *out, int64_t ld_out,
                                 nwc_stream stream) {
    if (!mp || n_ids < 0 || ld_out < mp->k) return NWC_ERR_INVALID_ARG;
    if (n_ids == 0) return NWC_OK;
    if (!ids || !out) return NWC_ERR_INVALID_ARG;
    const Mat m = to_mat(*mp);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int vec = vec_ok(out, ld_out, m.elem);
    const uint64_t items = (uint64_t)n_ids * m.cbs;
    const bool ragged = (m.k % kCols) != 0 || (m.n % kRows) != 0;
    if (m.elem == NWC_ELEM_BF16)
        return ragged ? launch_unpack<0, 1, true>(m, ids, items, out, ld_out, vec, s)
                      : launch_unpack<0, 1>(m, ids, items, out, ld_out, vec, s);
    return ragged ? launch_unpack<1, 1, true>(m, ids, items, out, ld_out, vec, s)
                  : launch_unpack<1, 1>(m, ids, items, out, ld_out, vec, s);
}

namespace {
// Workspace: [partials fp32 col_blocks x n_pad][counters u32 row_blocks]; both only when K > 512.
uint64_t ws_counter_off(const nwc_matrix &m) {
    return m.col_blocks > 1 ? 4 * (uint64_t)m.col_blocks * pad_rows(m) : 0;
}
}  // namespace

extern "C" size_t nwc_gemv_workspace_bytes(const nwc_matrix *mp) {
    if (!mp) return 0;
    uint64_t b = ws_counter_off(*mp);
    if (mp->col_blocks > 1) b += 4 * (uint64_t)mp->row_blocks;
    return (size_t)up16(b < 16 ? 16 : b);
}

extern "C" nwc_status nwc_gemv_prepare(const nwc_matrix *mp, void *ws, size_t ws_bytes, nwc_stream stream) {
    if (!mp || !ws || ws_bytes < nwc_gemv_workspace_bytes(mp) || (reinterpret_cast<uintptr_t>(ws) & 15))
        return NWC_ERR_INVALID_ARG;
    if (mp->col_blocks <= 1) return NWC_OK;
    uint8_t *counters = static_cast<uint8_t *>(ws) + ws_counter_off(*mp);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return cudaMemsetAsync(counters, 0, 4 * (size_t)mp->row_blocks, s) == cudaSuccess ? NWC_OK : NWC_ERR_CUDA;
}

namespace {
template <int ELEM, int NB>
cudaError_t launch_gemv_nb(const Mat &m, const uint16_t *x, int64_t ld_x, float *y, int64_t ld_y, float *partial,
                           uint32_t *counters, uint64_t n_pad, int sms, cudaStream_t stream) {
    using C = GemvCfg<NB>;
    static bool smem_ok = false;
    static std::once_flag once;
    std::call_once(once, [] {
        smem_ok = set_smem(gemv_kernel<ELEM, NB>, C::kSmem) && set_smem(gemv_kernel<ELEM, NB, true>, C::kSmem);
    });
    if (!smem_ok) return cudaErrorInvalidConfiguration;
    const uint64_t slots = (uint64_t)sms * C::kCtas;
    const int grid = (int)(m.nb < slots ? m.nb : slots);
    // Programmatic dependent launch: the kernel may start while the previous kernel on the stream
    // finishes; it streams its first block regions and builds its decode table meanwhile.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(C::kWarps * 32);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (m.n % kRows != 0)
        return cudaLaunchKernelEx(&cfg, gemv_kernel<ELEM, NB, true>, m, x, ld_x, y, ld_y, partial, counters, n_pad);
    return cudaLaunchKernelEx(&cfg, gemv_kernel<ELEM, NB>, m, x, ld_x, y, ld_y, partial, counters, n_pad);
}

// The GEMV for nb = 1 or 2 vectors on `partial` (nb x col_blocks x n_pad floats) and `counters`
// (row_blocks, zero); arguments already checked.
nwc_status launch_gemv(const Mat &m, const uint16_t *x, int64_t ld_x, float *y, int64_t ld_y, int nb, float *partial,
                       uint32_t *counters, uint64_t n_pad, cudaStream_t stream) {
    const int sms = sm_count();
    if (sms <= 0) return NWC_ERR_CUDA;
    cudaError_t rc;
    if (nb == 1)
        rc = m.elem == NWC_ELEM_BF16 ? launch_gemv_nb<0, 1>(m, x, ld_x, y, ld_y, partial, counters, n_pad, sms, stream)
                                     : launch_gemv_nb<1, 1>(m, x, ld_x, y, ld_y, partial, counters, n_pad, sms, stream);
    else
        rc = m.elem == NWC_ELEM_BF16 ? launch_gemv_nb<0, 2>(m, x, ld_x, y, ld_y, partial, counters, n_pad, sms, stream)
                                     : launch_gemv_nb<1, 2>(m, x, ld_x, y, ld_y, partial, counters, n_pad, sms, stream);
    return rc == cudaSuccess ? NWC_OK : NWC_ERR_CUDA;
}
}  // namespace

extern "C" nwc_status nwc_gemv(const nwc_matrix *mp, const uint16_t *x, float *y, void *ws, size_t ws_bytes,
                               nwc_stream stream) {
    if (!mp || !x || !y || !ws) return NWC_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(x) & 15) || (reinterpret_cast<uintptr_t>(ws) & 15)) return NWC_ERR_INVALID_ARG;
    if (ws_bytes < nwc_gemv_workspace_bytes(mp)) return NWC_ERR_INVALID_ARG;
    uint8_t *w8 = static_cast<uint8_t *>(ws);
    return launch_gemv(to_mat(*mp), x, 0, y, 0, 1, reinterpret_cast<float *>(w8),
                       reinterpret_cast<uint32_t *>(w8 + ws_counter_off(*mp)), pad_rows(*mp),
                       reinterpret_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------- small-batch GEMV
namespace {
// Batch workspace: [counters u32 row_blocks, padded to 16 B][partials fp32 nb x col_blocks x
// n_pad]; both only when K > 512. The counters come first, so a workspace prepared for nb
// vectors serves every smaller count.
uint64_t wsb_partial_off(const nwc_matrix &m) { return up16(4 * (uint64_t)m.row_blocks); }

template <int ELEM>
cudaError_t launch_batch(const Mat &m, const uint16_t *x, int64_t ld_x, int nb, float *y, int64_t ld_y, void *ws,
                         uint64_t n_pad, int grid, cudaStream_t s) {
    static bool smem_ok = false;
    static std::once_flag once;
    std::call_once(once, [] {
        smem_ok = set_smem(gemv_batch_kernel<ELEM>, kBatchSmem) && set_smem(gemv_batch_kernel<ELEM, true>, kBatchSmem);
    });
    if (!smem_ok) return cudaErrorInvalidConfiguration;
    uint8_t *w8 = static_cast<uint8_t *>(ws);
    uint32_t *counters = reinterpret_cast<uint32_t *>(w8);
    float *partial = reinterpret_cast<float *>(w8 + (m.cbs > 1 ? up16(4 * m.rbs) : 0));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kBatchWarps * 32);
    cfg.dynamicSmemBytes = kBatchSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (m.n % kRows != 0)
        return cudaLaunchKernelEx(&cfg, gemv_batch_kernel<ELEM, true>, m, x, ld_x, nb, y, ld_y, partial, counters,
                                  n_pad);
    return cudaLaunchKernelEx(&cfg, gemv_batch_kernel<ELEM>, m, x, ld_x, nb, y, ld_y, partial, counters, n_pad);
}
}  // namespace

extern "C" size_t nwc_gemv_batch_workspace_bytes(const nwc_matrix *mp, int nb) {
    if (!mp || nb < 1 || nb > NWC_GEMV_BATCH_MAX) return 0;
    if (mp->col_blocks <= 1) return 16;
    return (size_t)up16(wsb_partial_off(*mp) + 4 * (uint64_t)nb * mp->col_blocks * pad_rows(*mp));
}

extern "C" nwc_status nwc_gemv_batch_prepare(const nwc_matrix *mp, int nb, void *ws, size_t ws_bytes,
                                             nwc_stream stream) {
    const size_t need = nwc_gemv_batch_workspace_bytes(mp, nb);
    if (need == 0 || !ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 15)) return NWC_ERR_INVALID_ARG;
    if (mp->col_blocks <= 1) return NWC_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return cudaMemsetAsync(ws, 0, 4 * (size_t)mp->row_blocks, s) == cudaSuccess ? NWC_OK : NWC_ERR_CUDA;
}

extern "C" nwc_status nwc_gemv_batch(const nwc_matrix *mp, const uint16_t *x, int64_t ld_x, int nb, float *y,
                                     int64_t ld_y, void *ws, size_t ws_bytes, nwc_stream stream) {
    if (!mp || !x || !y || !ws || nb < 1 || nb > NWC_GEMV_BATCH_MAX) return NWC_ERR_INVALID_ARG;
    if (ld_x < (int64_t)mp->k || ld_y < (int64_t)mp->n || (ld_x % 8) != 0) return NWC_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(x) & 15) || (reinterpret_cast<uintptr_t>(ws) & 15)) return NWC_ERR_INVALID_ARG;
    if (ws_bytes < nwc_gemv_batch_workspace_bytes(mp, nb)) return NWC_ERR_INVALID_ARG;
    const Mat m = to_mat(*mp);
    const uint64_t n_pad = pad_rows(*mp);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (nb <= 2) {
        // one or two vectors: the GEMV kernel (FMA per vector), on the batch workspace's counters
        // and partials
        uint8_t *w8 = static_cast<uint8_t *>(ws);
        return launch_gemv(m, x, ld_x, y, ld_y, nb, reinterpret_cast<float *>(w8 + (m.cbs > 1 ? up16(4 * m.rbs) : 0)),
                           reinterpret_cast<uint32_t *>(w8), n_pad, s);
    }
    const int sms = sm_count();
    if (sms <= 0) return NWC_ERR_CUDA;
    const int grid = (int)(m.nb < (uint64_t)sms ? m.nb : (uint64_t)sms);
    const cudaError_t rc = m.elem == NWC_ELEM_BF16 ? launch_batch<0>(m, x, ld_x, nb, y, ld_y, ws, n_pad, grid, s)
                                                   : launch_batch<1>(m, x, ld_x, nb, y, ld_y, ws, n_pad, grid, s);
    return rc == cudaSuccess ? NWC_OK : NWC_ERR_CUDA;
}

// ---------------------------------------------------------------- allocation-free GEMV
// Scratch of nwc_gemv_noalloc: the partial sums and counters of one call live in
// this file-scope array, which every GPU that loads the library holds until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;  // 4 MiB
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void *g_noalloc_ptr[kMaxDevices] = {nullptr};
}  // namespace

extern "C" nwc_status nwc_gemv_noalloc(const nwc_matrix *mp, const uint16_t *x, float *y, nwc_stream stream) {
    if (!mp || !x || !y) return NWC_ERR_INVALID_ARG;
    const size_t need = nwc_gemv_workspace_bytes(mp);
    if (need == 0 || need > kNoAllocScratchBytes) return NWC_ERR_INVALID_ARG;  // matrix too large for the array
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return NWC_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return NWC_ERR_UNSUPPORTED;
    void *ptr = nullptr;
    {
        // Host code cannot use the array's name as a device address: resolve it once per device,
        // with that device current.
        std::lock_guard<std::mutex> lk(g_noalloc_mu);
        if (!g_noalloc_ptr[dev]) {
            void *p = nullptr;
            if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return NWC_ERR_CUDA;
            g_noalloc_ptr[dev] = p;
        }
        ptr = g_noalloc_ptr[dev];
    }
    // The array keeps whatever the previous call left: zero the counters for this matrix, then
    // run the GEMV on the same stream.
    nwc_status st = nwc_gemv_prepare(mp, ptr, kNoAllocScratchBytes, stream);
    if (st != NWC_OK) return st;
    return nwc_gemv(mp, x, y, ptr, kNoAllocScratchBytes, stream);
}

extern "C" nwc_status nwc_check(nwc_stream stream, uint32_t *flags) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return NWC_ERR_CUDA;
    uint32_t f = 0;
    if (cudaMemcpyFromSymbol(&f, g_nwc_error, 4) != cudaSuccess) return NWC_ERR_CUDA;
    if (f) {
        const uint32_t zero = 0;
        if (cudaMemcpyToSymbol(g_nwc_error, &zero, 4) != cudaSuccess) return NWC_ERR_CUDA;
    }
    if (flags) *flags = f;
    if (f & kErrTimeout) return NWC_ERR_TIMEOUT;
    return f ? NWC_ERR_DEVICE_FLAG : NWC_OK;
}
