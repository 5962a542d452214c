// kernels.cu -- sm_103a kernels and C-ABI launchers: decode to BF16/e4m3, embedding gather,
// the fused decode-GEMV (one or two vectors) and the small-batch GEMV (up to 16 vectors).
//
// "NWC -- Neural Weight Compression", section "How it works":
//   * each lane decodes its own bit stream for a block of 8 rows x 512 columns (16 columns
//     x 8 rows per lane), keeps the 16 matching activations in registers and accumulates
//     eight row sums; a transposed shuffle reduction produces partial sums per (row, column
//     block);
//   * a peek into a shared-memory lookup table yields two complete codes per step; the bit
//     window is shifted with funnel shifts and refilled with a wide multiply-add;
//   * dequantization and embedding lookup run on the same decoder.
// Format (version 4): the exponent's unary rank code is the only coded part; the sign and
// the mantissa are a raw byte per BF16 element (a nibble per fp8 element). A lane's stream is
// its 64 row pairs, each at most 13 bits, so one 13-bit peek into an 8192-entry table returns
// both exponents of a row pair, already in BF16 position, and the pair's length. Escapes (the
// pages' escape for rare exponents) and the second element of a pair too long for the peek
// decode to exponent field 0, a placeholder: the GEMV adds (true - placeholder) * x for each
// entry of the block's escape list before its row reduction; decode and gather write the
// listed elements over the placeholders.
// "Qwen3-4B-NWC-fp8": the per-channel scale is applied at the end of the matvec; an e4m3 value
// is a BF16 with exponent field v + 120 and mantissa m << 4 (zeros keep field 0, subnormal and
// NaN codes are listed), so fp8 runs through the same BF16 arithmetic.
//
// GB300 choices: the GEMV is a persistent grid of one CTA per SM (block b on CTA b % grid) with
// up to 32 warps, as few as keep the number of rounds of blocks so that no warp of the last
// round decodes alone; each warp streams whole block regions from HBM into its own shared-memory stage
// with one TMA bulk copy (cp.async.bulk, completion on an mbarrier, bounded waits) and
// prefetches its next region into L2; the decode table is copied in by TMA from a device copy
// prepared once per matrix (or built by the CTA when there is none) while the first regions
// are in flight. Per row pair a lane does one table load, a 64-bit funnel shift, a PRMT that
// spreads the two raw bytes (sign replicated into the high byte) and a LOP3 that merges them
// with the table's exponents into a BF16x2, then two FMAs with BF16 operands and FP32
// accumulators; the window is refilled every two pairs. Cross-column-block sums: every warp
// stores its partial sums and takes a ticket; the warp with the last ticket adds the column
// blocks' partial sums of its row block in a fixed order, writes y and resets the slots. When
// warps have further blocks, each loads the other partials while its ticket is in flight
// (partials not yet visible read as a sentinel and are loaded again); otherwise the ticket is an
// acquire-release atomic and only the last warp loads. The list kernel sums the row blocks that
// lie wholly in one SM's share inside one warp, without partial sums.
// The kernel is launched with programmatic stream serialization: it may start while the
// previous kernel on the stream drains and waits for it before touching x, the workspace or y.
// The small-batch GEMV keeps the decoder and moves the products with three or more vectors to
// the tensor cores (mma.sync on decoded tiles staged in shared memory).
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <mutex>
#include <utility>
#include <vector>

#include "nwc.h"
#include "nwc_format.h"

using namespace nwcf;

// Device error word: bit 0 = malformed stream (a lane read past its words, or an escape list
// that does not match the lane streams), bit 1 = gather id out of range, bit 2 = a bounded wait
// ran out. Read and cleared by nwc_check.
__device__ uint32_t g_nwc_error;

namespace {

constexpr uint32_t kErrFormat = 1u, kErrId = 2u, kErrTimeout = 4u;
constexpr uint32_t kSentinel = 0xFFFFFFFFu;  // an empty partial-sum slot (no float sum has these bits)

// floor(n / d) for 0 <= n < 2^31 by one wide multiply and a shift: m = ceil(2^(31+l) / d) with
// l = ceil(log2 d) fits 32 bits, and (n m) >> (31 + l) is exact for every such n (Granlund and
// Montgomery, "Division by invariant integers using multiplication", 1994, theorem 4.2, with
// 31-bit dividends). Block indices stay below 2^31 (validation bounds the block count), so every
// per-block division by the column-block count takes this form.
struct Div {
    uint32_t m, s;
};
Div make_div(uint64_t d) {
    uint32_t l = 0;
    while ((1ull << l) < d) l++;
    return Div{(uint32_t)(((1ull << (31 + l)) + d - 1) / d), 31u + l};
}
__device__ __forceinline__ uint32_t div_q(uint32_t n, Div v) { return (uint32_t)(((uint64_t)n * v.m) >> v.s); }

struct Mat {
    int elem, nr;
    uint64_t n, k, rbs, cbs, nb;
    Div cdiv;  // division by cbs
    const uint32_t *tab;
    const uint8_t *data;
    const float *scales;
    const uint32_t *table;
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
    t.cdiv = make_div(t.cbs);
    t.tab = m.block_tab;
    t.data = m.data;
    t.scales = m.scales;
    t.table = m.table;
    for (int i = 0; i < 16; i++) t.rank_exp[i] = m.rank_exp[i];
    return t;
}

__device__ __forceinline__ void raise_error(uint32_t bits) { atomicOr(&g_nwc_error, bits); }

// ------------------------------------------------------------------ shared memory, TMA
__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t lds8(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
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
__device__ __forceinline__ void l2_prefetch(const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// ------------------------------------------------------------------ geometry of the CTAs
constexpr int kStageBytes = 6144;  // a block region up to this size is staged, else read in place
constexpr int kLutEntries = 1 << kPeek;
constexpr int kLutBytes = kLutEntries * 4;
static_assert(kLutEntries == NWC_TABLE_ENTRIES && kLutBytes == NWC_TABLE_BYTES, "decode table size");
// A lane's fast decoder consumes at most 64 x 13 = 832 bits (every table entry's length is at
// most 13); its window moves on by a word only after 32 of them, so it takes in at most 26
// words after the first two and reads one word ahead: at most 29 words (116 bytes) from its
// first code word, whatever the code bits.
// Validation caps a lane at 26 words, so every lane's reads stay below 32 + 31 * 26 * 4 + 116
// = 3372 bytes of its stage; raw and list reads stay inside the region. The slack after the
// last stage is kept for good measure.
constexpr int kStageSlack = 256;
// Shared memory of a kernel with W warps: the table at 0, then an mbarrier per warp and one
// for the table, then the stages (and whatever else the kernel adds after them).
template <int W>
struct Smem {
    static constexpr int kBar = kLutBytes;
    static constexpr int kLutBar = kBar + 8 * W;
    static constexpr int kStage = (kLutBar + 8 + 127) / 128 * 128;
    static constexpr int kEnd = kStage + W * kStageBytes;
};
constexpr int kGemvWarps = 32;
constexpr int kGemv2Warps = 28;  // two vectors: a second accumulator set, up to 72 registers
constexpr int kGemvSmem = Smem<kGemvWarps>::kEnd + kStageSlack;
constexpr int kGemv2Smem = Smem<kGemv2Warps>::kEnd + kStageSlack;
static_assert(kGemvSmem <= 232448 && kGemv2Smem <= 232448, "shared memory per CTA");
template <int NB>
struct GemvCfg {
    static constexpr int kWarps = NB == 1 ? kGemvWarps : kGemv2Warps;
    static constexpr int kSmem = NB == 1 ? kGemvSmem : kGemv2Smem;
};

// The decode table in shared memory: a TMA copy of the matrix's table when there is one
// (issued by thread 0 on the table barrier; every thread later waits for it with
// lut_ready), else built by all threads of the CTA from the rank table (read from the kernel
// parameter with static offsets only, so the parameter is not copied to local memory).
__device__ __forceinline__ void lut_start(const Mat &m, uint8_t *smem, uint32_t lut_bar) {
    if (m.table) {
        if (threadIdx.x == 0) {
            mbar_init(lut_bar);
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
            mbar_expect_tx(lut_bar, kLutBytes);
#pragma unroll
            for (int q = 0; q < 4; q++)
                tma_load_1d(smem_u32(smem) + q * (kLutBytes / 4), m.table + q * (kLutEntries / 4), kLutBytes / 4, lut_bar);
        }
        return;
    }
    __shared__ uint8_t rexp[16];
    if (threadIdx.x < 16) {
        uint32_t v = 0;
#pragma unroll
        for (int i = 0; i < 16; i++)
            if ((int)threadIdx.x == i) v = m.rank_exp[i];
        rexp[threadIdx.x] = (uint8_t)v;
    }
    __syncthreads();
    uint32_t *lut = reinterpret_cast<uint32_t *>(smem);
    for (uint32_t i = threadIdx.x; i < (uint32_t)kLutEntries; i += blockDim.x) lut[i] = table_entry(i, m.nr, m.elem, rexp);
}
// After a __syncthreads that follows lut_start: the table is complete in shared memory.
__device__ __forceinline__ bool lut_ready(const Mat &m, uint32_t lut_bar) {
    return m.table ? mbar_wait(lut_bar, 0) : true;
}

// ------------------------------------------------------------------ the lane decoder
// Window state in registers: the 64 stream bits wh:wl (most significant bit first) and the
// offset o of the next unread bit in them; pa = shared-memory address of the next word to
// insert, nw = that word (loaded one refill ahead, off the decode chain). Whole table entries
// are added to o: their low five bits are the pair's length and bits 5..6 are zero, and o stays
// below 64, so o's low six bits are exact and the bits above them are ignored.
struct Fs {
    uint32_t wh, wl, o, pa, nw;
};

// First two words of a lane's stream at shared address `code` (lw words).
__device__ __forceinline__ void fs_init(Fs &s, uint32_t code, uint32_t lw) {
    s.wh = lw > 0 ? lds32(code) : 0u;
    s.wl = lw > 1 ? lds32(code + 4) : 0u;
    s.pa = code + 8;
    s.o = 0u;
    s.nw = lds32(s.pa);
}

// Before every second row pair: once the offset has passed the first word, the window moves on
// by a word (wh:wl <- wl:nw). Leaves o < 32, so the window holds at least 33 unread bits: two
// row pairs.
__device__ __forceinline__ void fs_refill(Fs &s) {
    asm("{\n\t"
        ".reg .pred q;\n\t"
        ".reg .u32 t;\n\t"
        "and.b32 t, %2, 32;\n\t"
        "setp.ne.u32 q, t, 0;\n\t"
        "@q mov.b32 %0, %1;\n\t"
        "@q mov.b32 %1, %4;\n\t"
        "@q xor.b32 %2, %2, 32;\n\t"
        "@q add.u32 %3, %3, 4;\n\t"
        "@q ld.shared.u32 %4, [%3];\n\t"
        "}"
        : "+r"(s.wh), "+r"(s.wl), "+r"(s.o), "+r"(s.pa), "+r"(s.nw));
}

// One row pair: the table entry of the next 13 bits; the offset moves past the pair.
__device__ __forceinline__ uint32_t fs_pair(Fs &s, uint32_t lutb) {
    uint32_t e;
    asm volatile("{\n\t.reg .u32 a, h, n;\n\t.reg .b64 w;\n\t"
                 "and.b32 n, %3, 63;\n\t"
                 "mov.b64 w, {%2, %1};\n\t"
                 "shl.b64 w, w, n;\n\t"
                 "mov.b64 {a, h}, w;\n\t"
                 "shr.u32 a, h, 19;\n\t"
                 "mad.lo.u32 a, a, 4, %4;\n\t"
                 "ld.shared.u32 %0, [a];\n\t}"
                 : "=r"(e)
                 : "r"(s.wh), "r"(s.wl), "r"(s.o), "r"(lutb));
    s.o += e;
    return e;
}

// Whether the lane consumed more bits than its lw words hold (a malformed stream): the window
// holds the two words before pa, o bits of them read.
__device__ __forceinline__ bool fs_overrun(const Fs &s, uint32_t code, uint32_t lw) {
    const uint32_t consumed = (s.pa - code) * 8u - 64u + (s.o & 63u);
    return consumed > 32u * lw;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// The raw bits of a row pair spread into a BF16x2's sign and mantissa positions (row 2i in the
// low half), the sign replicated over the high byte of each half (the merge masks it).
// BF16: `w` holds rows 4h .. 4h + 3 of a column, a byte each; pair i picks bytes 2(i%2) and
// 2(i%2) + 1. fp8: `rl` and `rh` are a column's four row-pair bytes with the even rows' nibbles
// (rl) and the odd rows' nibbles (rh) moved to bits 4..7 of each byte (the mantissa then sits
// at BF16 mantissa bits 4..6, the sign at bit 7); pair i picks byte i of each.
template <int ELEM>
__device__ __forceinline__ uint32_t raw_pair(uint32_t w, uint32_t rh, int i) {
    if (ELEM == 0) return prmt(w, 0u, (i & 1) ? 0xB3A2u : 0x9180u);
    return prmt(w, rh, 0xC480u + 0x1111u * (uint32_t)i);
}
__device__ __forceinline__ uint32_t merge_pair(uint32_t rp, uint32_t e) {
    return (rp & 0x807F807Fu) | (e & 0x7F807F80u);
}

// acc0 += lo(w2) * x, acc1 += hi(w2) * x with BF16 operands and FP32 accumulation, x being the
// low (H = 0) or high (H = 1) half of the activation pair xp. A BF16 product is exact in FP32,
// so each equals an FP32 FMA of the widened values.
template <int H>
__device__ __forceinline__ void fma_bf16x2(uint32_t w2, uint32_t xp, float &acc0, float &acc1) {
    if (H == 0)
        asm("{\n\t.reg .b16 lo, hi, xl, xh;\n\t"
            "mov.b32 {lo, hi}, %2;\n\t"
            "mov.b32 {xl, xh}, %3;\n\t"
            "fma.rn.f32.bf16 %0, lo, xl, %0;\n\t"
            "fma.rn.f32.bf16 %1, hi, xl, %1;\n\t}"
            : "+f"(acc0), "+f"(acc1)
            : "r"(w2), "r"(xp));
    else
        asm("{\n\t.reg .b16 lo, hi, xl, xh;\n\t"
            "mov.b32 {lo, hi}, %2;\n\t"
            "mov.b32 {xl, xh}, %3;\n\t"
            "fma.rn.f32.bf16 %0, lo, xh, %0;\n\t"
            "fma.rn.f32.bf16 %1, hi, xh, %1;\n\t}"
            : "+f"(acc0), "+f"(acc1)
            : "r"(w2), "r"(xp));
}

// Value of an element from its raw bits and exponent field (the true value of a listed
// element): BF16 raw byte s << 7 | m; fp8 raw nibble s << 3 | m (e4m3: bias 7, subnormals at
// v = 0, S.1111.111 is NaN).
template <int ELEM>
__device__ __forceinline__ float elem_value(uint32_t raw, uint32_t v) {
    if (ELEM == 0) return __uint_as_float(((raw & 0x80u) << 24) | (v << 23) | ((raw & 0x7Fu) << 16));
    const uint32_t s = (raw >> 3) & 1u, m = raw & 7u;
    if (v == 0) {
        const float f = (float)m * 0.001953125f;  // m * 2^-9, exact
        return s ? -f : f;
    }
    if (v == 15 && m == 7) return __uint_as_float(0x7FC00000u);
    return __uint_as_float((s << 31) | ((v + 120u) << 23) | (m << 20));
}
// The placeholder that the decoders produce for a listed element: exponent field 0 with the
// element's raw sign and mantissa (BF16: a subnormal of order 2^-133; fp8: mantissa m << 4).
template <int ELEM>
__device__ __forceinline__ float placeholder(uint32_t raw) {
    if (ELEM == 0) return __uint_as_float(((raw & 0x80u) << 24) | ((raw & 0x7Fu) << 16));
    return __uint_as_float(((raw & 8u) << 28) | ((raw & 7u) << 20));
}
// BF16 bits of an element's value (fp8: the e4m3 value, exact in BF16; NaN 0x7FC0).
template <int ELEM>
__device__ __forceinline__ uint32_t elem_bf16(uint32_t raw, uint32_t v) {
    return __float_as_uint(elem_value<ELEM>(raw, v)) >> 16;
}

// Where the raw bits of row r, column c of lane l sit in a block's raw section, as a byte
// offset from the section start (fp8: the byte holding rows r & ~1, r | 1, nibble r & 1).
// kc = the block's real columns (the layout is the full one when kc == 512).
template <int ELEM>
__device__ __forceinline__ uint32_t raw_offset(int kc, uint32_t l, uint32_t c, uint32_t r) {
    constexpr uint32_t CB = ELEM == 0 ? 8u : 4u;  // bytes per column
    const uint32_t rb = ELEM == 0 ? r : r >> 1;
    if (kc == kCols) {
        if (ELEM == 0) return 16u * (32u * (c >> 1) + l) + 8u * (c & 1u) + rb;
        return 16u * (32u * (c >> 2) + l) + 4u * (c & 3u) + rb;
    }
    // lanes before l: full lanes of 16 columns, then the one partial lane (if any)
    const uint32_t full = (uint32_t)kc >> 4, part = (uint32_t)kc & 15u;
    const uint32_t before = (l < full ? l : full) * 16u * CB + (l > full && part ? (uint32_t)up16(part * CB) : 0u);
    return before + CB * c + rb;
}
// Bytes of a block's raw section for kc real columns.
template <int ELEM>
__device__ __forceinline__ uint32_t raw_bytes(int kc) {
    constexpr uint32_t CB = ELEM == 0 ? 8u : 4u;
    if (kc == kCols) return 512u * CB;
    const uint32_t full = (uint32_t)kc >> 4, part = (uint32_t)kc & 15u;
    return full * 16u * CB + (part ? (uint32_t)up16(part * CB) : 0u);
}

// ------------------------------------------------------------------ row sums
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
__device__ __forceinline__ int rowsel(int lane) { return ((lane >> 4) & 1) << 2 | ((lane >> 3) & 1) << 1 | ((lane >> 2) & 1); }
// The lane holding row r's sum after transpose_reduce.
__device__ __forceinline__ int row_holder(int r) { return ((r >> 2) & 1) << 4 | ((r >> 1) & 1) << 3 | (r & 1) << 2; }

__device__ __forceinline__ uint32_t ld_relaxed(const float *p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed(float *p, uint32_t v) {
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// A partial sum as stored: any NaN as the canonical quiet NaN, so that no stored sum has the
// sentinel's bits.
__device__ __forceinline__ uint32_t canon(float f) { return f != f ? 0x7FC00000u : __float_as_uint(f); }

// Row block rb done for NB vectors (sum[v] in the lanes that transpose_reduce left it in):
// one column block writes y directly; otherwise every warp stores its partial sums and takes a
// ticket, and the warp that took the last ticket loads the other column blocks' partials of its
// row block (lane i: row i % 8, column blocks i / 8, i / 8 + 4, ...), adds them in that fixed
// order, writes y (times the row scale for fp8), and puts the sentinels and the counter back for
// the next call. Two ways to reach the loads, with the same sums bit for bit:
//   SPEC: every warp loads the other partials while its (relaxed) ticket is in flight, so the
//     last warp usually has them at once; a slot still holding the sentinel is loaded again (a
//     bounded number of times). Best when warps have further blocks to decode meanwhile.
//   otherwise: the ticket is an acquire-release atomic after a warp barrier (the writer lanes'
//     stores precede it), and only the last warp loads, after it; far fewer loads reach L2 at a
//     launch's end, which is what a launch with at most one block per warp waits for.
// Partial slots: partial[(v cbs + cb) n_pad + row].
template <int ELEM, int NB, bool SPEC>
__device__ __forceinline__ void finish_rows(const Mat &m, const float (&sum)[NB], int lane, uint64_t rb, uint64_t cb,
                                            float *y, int64_t ld_y, float *partial, uint32_t *counters,
                                            uint64_t n_pad, bool &timed_out) {
    const uint64_t row = rb * kRows + (uint64_t)rowsel(lane);
    const bool writer = (lane & 3) == 0 && row < m.n;
    if (m.cbs == 1) {
#pragma unroll
        for (int v = 0; v < NB; v++)
            if (writer) y[v * ld_y + (int64_t)row] = ELEM == 0 ? sum[v] : sum[v] * m.scales[row];
        return;
    }
    const uint64_t r2 = rb * kRows + (uint64_t)(lane & 7);
    const bool live = r2 < m.n;
    const uint64_t c0 = (uint64_t)(lane >> 3);
    constexpr int kSpec = 4;  // loads per lane in one round: column blocks up to 16
#pragma unroll
    for (int v = 0; v < NB; v++)
        if (writer) st_relaxed(partial + ((uint64_t)v * m.cbs + cb) * n_pad + row, canon(sum[v]));
    uint32_t pv[NB][kSpec];
    auto load_round = [&]() {
#pragma unroll
        for (int v = 0; v < NB; v++)
#pragma unroll
            for (int q = 0; q < kSpec; q++) {
                const uint64_t c2 = c0 + 4 * q;
                pv[v][q] = kSentinel;
                if (live && c2 < m.cbs && c2 != cb) pv[v][q] = ld_relaxed(partial + ((uint64_t)v * m.cbs + c2) * n_pad + r2);
            }
    };
    uint32_t ticket = 0;
    if (SPEC) {
        load_round();
        if (lane == 0) asm volatile("atom.relaxed.gpu.global.add.u32 %0, [%1], 1;" : "=r"(ticket) : "l"(counters + rb) : "memory");
    } else {
        __syncwarp();
        if (lane == 0) asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(ticket) : "l"(counters + rb) : "memory");
    }
    ticket = __shfl_sync(0xFFFFFFFFu, ticket, 0);
    if (ticket != (uint32_t)m.cbs - 1) return;
    if (!SPEC) {
        __syncwarp();  // lane 0's acquire precedes every lane's loads
        load_round();
    }
    float own[NB];
#pragma unroll
    for (int v = 0; v < NB; v++) own[v] = __shfl_sync(0xFFFFFFFFu, sum[v], row_holder(lane & 7));
    const long long t0 = clock64();
#pragma unroll
    for (int v = 0; v < NB; v++) {
        float s = 0.0f;
        if (live) {
            // slots c0 + 4q in a fixed order: the first kSpec from the loads above, the rest
            // (more than 16 column blocks) kSpec at a time with their loads in flight together;
            // a slot still holding the sentinel is loaded again (bounded)
            for (uint64_t q0 = 0; c0 + 4 * q0 < m.cbs; q0 += kSpec) {
                uint32_t bits[kSpec];
#pragma unroll
                for (int qq = 0; qq < kSpec; qq++) {
                    const uint64_t c2 = c0 + 4 * (q0 + qq);
                    bits[qq] = q0 == 0 ? pv[v][qq] : kSentinel;
                    if (q0 != 0 && c2 < m.cbs && c2 != cb) bits[qq] = ld_relaxed(partial + ((uint64_t)v * m.cbs + c2) * n_pad + r2);
                }
#pragma unroll
                for (int qq = 0; qq < kSpec; qq++) {
                    const uint64_t c2 = c0 + 4 * (q0 + qq);
                    if (c2 >= m.cbs) break;
                    if (c2 == cb) {
                        s += own[v];
                        continue;
                    }
                    while (bits[qq] == kSentinel) {
                        bits[qq] = ld_relaxed(partial + ((uint64_t)v * m.cbs + c2) * n_pad + r2);
                        if (bits[qq] == kSentinel && clock64() - t0 > (1ll << 32)) {
                            timed_out = true;
                            bits[qq] = 0u;
                        }
                    }
                    s += __uint_as_float(bits[qq]);
                }
            }
        }
        s += __shfl_xor_sync(0xFFFFFFFFu, s, 8);
        s += __shfl_xor_sync(0xFFFFFFFFu, s, 16);
        if (lane < kRows && live) y[v * ld_y + (int64_t)r2] = ELEM == 0 ? s : s * m.scales[r2];
    }
    // every slot read goes back to the sentinel (the warp's own slot below, after its writer)
#pragma unroll
    for (int v = 0; v < NB; v++)
        if (live)
            for (uint64_t c2 = c0; c2 < m.cbs; c2 += 4)
                if (c2 != cb) st_relaxed(partial + ((uint64_t)v * m.cbs + c2) * n_pad + r2, kSentinel);
    // the warp's own slots: written by the writer lanes above, reset here after them
    __syncwarp();
#pragma unroll
    for (int v = 0; v < NB; v++)
        if (writer) st_relaxed(partial + ((uint64_t)v * m.cbs + cb) * n_pad + row, kSentinel);
    if (lane == 0) counters[rb] = 0;
}

// ------------------------------------------------------------------ block geometry
// Facts of one staged block region for this lane (all shared addresses).
struct LaneBlock {
    uint32_t code, lw;   // the lane's first code word and its word count
    uint32_t raw0;       // start of the raw section
    uint32_t ubase;      // the lane's first 16-byte raw unit
    uint32_t ustride;    // bytes from one of the lane's units to the next
    uint32_t units;      // units the lane may read (its region; full layout: all)
    uint32_t list0;      // start of the escape list
    int cols;            // the lane's real columns
};
// kc = the block's real columns (512: the full layout).
template <int ELEM, bool EDGE>
__device__ __forceinline__ LaneBlock lane_block(uint32_t stage, int lane, int kc) {
    LaneBlock b;
    b.lw = lds8(stage + (uint32_t)lane);
    uint32_t incl = b.lw;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t o = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        if (lane >= d) incl += o;
    }
    const uint32_t total = __shfl_sync(0xFFFFFFFFu, incl, 31);
    b.code = stage + 32u + 4u * (incl - b.lw);
    b.raw0 = stage + (uint32_t)up16(32u + 4u * total);
    constexpr uint32_t CBY = ELEM == 0 ? 8u : 4u;
    if (!EDGE) {
        b.ubase = b.raw0 + 16u * (uint32_t)lane;
        b.ustride = 512u;
        b.units = ELEM == 0 ? 8u : 4u;
        b.list0 = b.raw0 + 512u * CBY;
        b.cols = kLaneCols;
    } else {
        const int c = kc - kLaneCols * lane;
        b.cols = c < 0 ? 0 : (c > kLaneCols ? kLaneCols : c);
        b.ubase = b.raw0 + raw_offset<ELEM>(kc, (uint32_t)lane, 0, 0);
        b.ustride = 16u;
        b.units = (uint32_t)up16((uint32_t)b.cols * CBY) / 16u;
        b.list0 = b.raw0 + raw_bytes<ELEM>(kc);
    }
    return b;
}

// Decodes columns 4g .. 4g + 3 of the lane (16 row pairs) into w2[4 cc + i] = rows (2i, 2i + 1)
// of column 4g + cc as BF16x2 (row 2i in the low half). EDGE: columns at or past the lane's real
// ones give 0 and only the lane's own raw units are read. COUNT: adds each pair's listed-element
// count (table bits 16..17) to *nesc.
template <int ELEM, bool EDGE, bool COUNT = false>
__device__ __forceinline__ void decode_group(Fs &s, uint32_t lutb, const LaneBlock &lb, int g, uint32_t (&w2)[16],
                                             uint32_t *nesc = nullptr) {
    uint32_t cw[8];  // BF16: column cc's rows 0..3 in cw[2cc], rows 4..7 in cw[2cc + 1]; fp8: cw[cc]
    constexpr int NU = ELEM == 0 ? 2 : 1;
#pragma unroll
    for (int q = 0; q < NU; q++) {
        const uint32_t u = (uint32_t)(NU * g + q);
        uint4 r = make_uint4(0u, 0u, 0u, 0u);
        if (!EDGE || u < lb.units) r = lds128(lb.ubase + u * lb.ustride);
        cw[4 * q] = r.x;
        cw[4 * q + 1] = r.y;
        cw[4 * q + 2] = r.z;
        cw[4 * q + 3] = r.w;
    }
#pragma unroll
    for (int cc = 0; cc < 4; cc++) {
        uint32_t rl = 0, rh = 0;
        if (ELEM == 1) {
            rl = (cw[cc] << 4) & 0xF0F0F0F0u;
            rh = cw[cc] & 0xF0F0F0F0u;
        }
#pragma unroll
        for (int i = 0; i < 4; i++) {
            if ((i & 1) == 0) fs_refill(s);
            const uint32_t e = fs_pair(s, lutb);
            if (COUNT) *nesc += (e >> 16) & 3u;
            const uint32_t rp = ELEM == 0 ? raw_pair<0>(cw[2 * cc + (i >> 1)], 0u, i) : raw_pair<1>(rl, rh, i);
            uint32_t bf = merge_pair(rp, e);
            if (EDGE && 4 * g + cc >= lb.cols) bf = 0u;
            w2[4 * cc + i] = bf;
        }
    }
}

// The 16 activations of a lane (columns c0 .. c0 + 15 of a vector) as BF16 pairs; columns at
// or past `cols` read as 0 (and are not loaded).
__device__ __forceinline__ void load_x16(const uint16_t *xl, int cols, uint32_t (&xs)[8]) {
    if (cols == kLaneCols) {
        const uint4 a = __ldg(reinterpret_cast<const uint4 *>(xl));
        const uint4 b = __ldg(reinterpret_cast<const uint4 *>(xl) + 1);
        xs[0] = a.x; xs[1] = a.y; xs[2] = a.z; xs[3] = a.w;
        xs[4] = b.x; xs[5] = b.y; xs[6] = b.z; xs[7] = b.w;
        return;
    }
#pragma unroll
    for (int k = 0; k < 8; k++) {
        const uint32_t lo = 2 * k < cols ? (uint32_t)__ldg(xl + 2 * k) : 0u;
        const uint32_t hi = 2 * k + 1 < cols ? (uint32_t)__ldg(xl + 2 * k + 1) : 0u;
        xs[k] = lo | hi << 16;
    }
}

// Adds (true - placeholder) * x to acc[v][row] for every entry of a block's escape list (`slots`
// words from shared address list0, or from global memory at glist when that is not null), the
// entries spread over the lanes; the transposed reduction then sums them with the rows. The raw
// bits come from the raw section at raw0 (shared) or graw (global). xb = activations from the
// block's first column; kc, rows = the block's real extent. An entry naming no real element
// raises `bad`.
template <int ELEM, int NB>
__device__ __forceinline__ void esc_correct(uint32_t list0, uint32_t raw0, const uint32_t *glist, const uint8_t *graw,
                                            uint32_t slots, int lane, const uint16_t *xb, int64_t ld_x, int kc, int rows,
                                            float (&acc)[NB][8], bool &bad) {
    for (uint32_t j = (uint32_t)lane; j < slots; j += 32) {
        const uint32_t e = glist ? __ldg(glist + j) : lds32(list0 + 4u * j);
        if (e == kEscPad) continue;
        const uint32_t t = esc_t(e), l = esc_lane(e), v = esc_v(e);
        const uint32_t r = t & 7u, c = t >> 3;
        if ((int)r >= rows || (int)(kLaneCols * l + c) >= kc || (v >> exp_bits(ELEM))) {
            bad = true;
            continue;
        }
        const uint32_t at = raw_offset<ELEM>(kc, l, c, r);
        uint32_t rawb = graw ? (uint32_t)__ldg(graw + at) : lds8(raw0 + at);
        if (ELEM == 1) rawb = (rawb >> (4u * (r & 1u))) & 0xFu;
        const float w = elem_value<ELEM>(rawb, v), ph = placeholder<ELEM>(rawb);
#pragma unroll
        for (int q = 0; q < NB; q++) {
            const float xv = __uint_as_float((uint32_t)__ldg(xb + q * ld_x + kLaneCols * l + c) << 16);
            const float d = fmaf(w, xv, -(ph * xv));
#pragma unroll
            for (int i = 0; i < 8; i++)
                if (i == (int)r) acc[q][i] += d;
        }
    }
}

// Block from its staged region (shared address `stage`, `bytes` long) for NB vectors (vector v
// at xb + v ld_x from the block's first column; xs = the lane's 16 activations of each, loaded
// by the caller while the region lands, zero past K). EDGE: the block's real columns kc < 512 (the
// lanes' raw regions follow one another; columns past K give 0). rows = the block's real rows:
// rows past N decode to finite fillers whose sums are never stored.
template <int ELEM, int NB, bool EDGE>
__device__ __forceinline__ void gemv_block(uint32_t stage, uint32_t bytes, int lane, uint32_t lutb, const uint16_t *xb,
                                           int64_t ld_x, const uint32_t (&xs)[NB][8], float (&acc)[NB][8], bool &bad,
                                           int kc, int rows) {
    const LaneBlock lb = lane_block<ELEM, EDGE>(stage, lane, kc);
    Fs s;
    fs_init(s, lb.code, lb.lw);
#pragma unroll
    for (int g = 0; g < 4; g++) {
        uint32_t w2[16];
        decode_group<ELEM, EDGE>(s, lutb, lb, g, w2);
#pragma unroll
        for (int cc = 0; cc < 4; cc++) {
            const int c = 4 * g + cc;
#pragma unroll
            for (int i = 0; i < 4; i++)
#pragma unroll
                for (int v = 0; v < NB; v++) {
                    if (c & 1) fma_bf16x2<1>(w2[4 * cc + i], xs[v][c >> 1], acc[v][2 * i], acc[v][2 * i + 1]);
                    else fma_bf16x2<0>(w2[4 * cc + i], xs[v][c >> 1], acc[v][2 * i], acc[v][2 * i + 1]);
                }
        }
    }
    bad |= fs_overrun(s, lb.code, lb.lw);
    const uint32_t lo = lb.list0 - stage;
    const uint32_t slots = lo <= bytes ? (bytes - lo) / 4u : 0u;
    esc_correct<ELEM, NB>(lb.list0, lb.raw0, nullptr, nullptr, slots, lane, xb, ld_x, EDGE ? kc : kCols, rows, acc, bad);
}

// Any block read in place from global memory (a region too large for a stage): the same
// arithmetic, one row pair at a time, every word read bounded by the lane's own words (zeros
// past them) and every raw read by the region.
template <int ELEM, int NB>
__device__ __forceinline__ void gemv_block_global(const uint8_t *reg, uint32_t bytes, int lane, uint32_t lutb,
                                               const uint16_t *xb, int64_t ld_x, float (&acc)[NB][8], bool &bad, int kc,
                                               int rows) {
    const uint32_t lw = reg[lane];
    uint32_t incl = lw;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t o = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        if (lane >= d) incl += o;
    }
    const uint32_t total = __shfl_sync(0xFFFFFFFFu, incl, 31);
    const uint32_t *code = reinterpret_cast<const uint32_t *>(reg + 32) + (incl - lw);
    const uint32_t raw0 = (uint32_t)up16(32u + 4u * total);
    const uint32_t list0 = raw0 + raw_bytes<ELEM>(kc);
    if (list0 > bytes) {
        bad = true;
        return;
    }
    const int cl = kc - kLaneCols * lane, cols = cl < 0 ? 0 : (cl > kLaneCols ? kLaneCols : cl);
    uint64_t win = 0;
    int nbits = 0;
    uint32_t wi = 0, used = 0;
#pragma unroll 1
    for (int c = 0; c < kLaneCols; c++) {
        float xv[NB];
#pragma unroll
        for (int v = 0; v < NB; v++)
            xv[v] = c < cols ? __uint_as_float((uint32_t)__ldg(xb + v * ld_x + kLaneCols * lane + c) << 16) : 0.0f;
#pragma unroll
        for (int i = 0; i < 4; i++) {
            while (nbits <= 32) {
                const uint32_t w = wi < lw ? __ldg(code + wi) : 0u;
                wi++;
                win |= (uint64_t)w << (32 - nbits);
                nbits += 32;
            }
            const uint32_t e = lds32(lutb + 4u * (uint32_t)(win >> (64 - kPeek)));
            const uint32_t L = e & 31u;
            win <<= L;
            nbits -= (int)L;
            used += L;
            if (c >= cols) continue;
            const uint32_t at = raw_offset<ELEM>(kc, (uint32_t)lane, (uint32_t)c, 2u * i);
            uint32_t b0, b1;
            if (ELEM == 0) {
                b0 = reg[raw0 + at];
                b1 = reg[raw0 + at + 1];
            } else {
                const uint32_t byte = reg[raw0 + at];
                b0 = byte & 0xFu;
                b1 = byte >> 4;
            }
            const uint32_t E0 = (e >> 7) & 0xFFu, E1 = (e >> 23) & 0xFFu;
            const uint32_t h0 = ELEM == 0 ? ((b0 & 0x80u) << 8) | (E0 << 7) | (b0 & 0x7Fu)
                                          : ((b0 & 8u) << 12) | (E0 << 7) | ((b0 & 7u) << 4);
            const uint32_t h1 = ELEM == 0 ? ((b1 & 0x80u) << 8) | (E1 << 7) | (b1 & 0x7Fu)
                                          : ((b1 & 8u) << 12) | (E1 << 7) | ((b1 & 7u) << 4);
#pragma unroll
            for (int v = 0; v < NB; v++) {
                acc[v][2 * i] = fmaf(__uint_as_float(h0 << 16), xv[v], acc[v][2 * i]);
                acc[v][2 * i + 1] = fmaf(__uint_as_float(h1 << 16), xv[v], acc[v][2 * i + 1]);
            }
        }
    }
    bad |= used > 32u * lw;
    esc_correct<ELEM, NB>(0u, 0u, reinterpret_cast<const uint32_t *>(reg + list0), reg + raw0, (bytes - list0) / 4u, lane,
                          xb, ld_x, kc, rows, acc, bad);
}

// =================================================================== GEMV kernel
// y[v] = W x[v] for NB vectors (1 or 2; vector v at x + v ld_x, its result at y + v ld_y, its
// partial sums at partial + v col_blocks n_pad). KR: K % 512 != 0, and the last column block's
// blocks take the fast decoder with the ragged raw layout, in a kernel of its own so that the
// others keep their registers.
// The matrix multiplied after this one, whose bytes this kernel brings into L2 once its own
// first regions have landed (its decode phase leaves HBM idle): the block regions, the block
// table and the decode table. bytes == 0: nothing to prefetch.
struct Prefetch {
    const uint8_t *data;
    uint64_t bytes;
    const uint32_t *tab;
    uint64_t tab_bytes;
    const uint32_t *table;
};

// This warp's share of the prefetch: the regions split evenly (16-byte pieces) over the `ways`
// warps that have a block; warp 0 also takes the block table and the decode table.
__device__ __forceinline__ void prefetch_share(const Prefetch &pf, uint64_t w, uint64_t ways) {
    if (pf.bytes == 0 || w >= ways) return;
    const uint64_t units = pf.bytes / 16, per = (units + ways - 1) / ways;
    const uint64_t u0 = w * per, u1 = u0 + per < units ? u0 + per : units;
    // one bulk prefetch per 64 KB at most
    for (uint64_t u = u0; u < u1; u += 4096) {
        const uint64_t n = u1 - u < 4096 ? u1 - u : 4096;
        l2_prefetch(pf.data + 16 * u, (uint32_t)(16 * n));
    }
    if (w == 0) {
        for (uint64_t o = 0; o < pf.tab_bytes; o += 65536)
            l2_prefetch(reinterpret_cast<const uint8_t *>(pf.tab) + o,
                        (uint32_t)(pf.tab_bytes - o < 65536 ? pf.tab_bytes - o : 65536));
        if (pf.table) l2_prefetch(pf.table, kLutBytes);
    }
}

template <int ELEM, int NB, bool KR, bool SPEC>
__global__ void __launch_bounds__(GemvCfg<NB>::kWarps * 32, 1)
    gemv_kernel(Mat m, const uint16_t *__restrict__ x, int64_t ld_x, float *__restrict__ y, int64_t ld_y,
                float *partial, uint32_t *counters, uint64_t n_pad, Prefetch pf) {
    using C = GemvCfg<NB>;
    using S = Smem<C::kWarps>;
    // A kernel launched after this one with programmatic stream serialization may start as soon
    // as SMs free up; it waits (griddepcontrol.wait) before touching anything this one writes.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t bar = smem_u32(smem + S::kBar + 8 * warp), lut_bar = smem_u32(smem + S::kLutBar);
    const uint32_t stage = smem_u32(smem + S::kStage + warp * kStageBytes);

    // Block b goes to CTA b % grid, so every SM gets within one block of the same count. The CTA
    // may have fewer warps than its shared memory is laid out for (the launch picks the count).
    const uint64_t total_warps = (uint64_t)gridDim.x * (blockDim.x >> 5);
    uint64_t b = (uint64_t)blockIdx.x + (uint64_t)gridDim.x * warp;
    uint32_t phase = 0;
    bool bad = false, timed_out = false, inflight = false;

    // Block bounds (16-byte units from the data section) travel with the warp: c0/c1 of block b
    // in every lane; n0/n1 of the warp's next block in lane 0, read one iteration ahead, so that
    // no read of the block table sits on the decode path.
    uint32_t c0 = 0, c1 = 0, n0 = 0, n1 = 0;
    if (lane == 0 && b < m.nb) {
        c0 = m.tab[b];
        c1 = m.tab[b + 1];
    }
    if (lane == 0 && b + total_warps < m.nb) {
        n0 = m.tab[b + total_warps];
        n1 = m.tab[b + total_warps + 1];
    }
    c0 = __shfl_sync(0xFFFFFFFFu, c0, 0);
    c1 = __shfl_sync(0xFFFFFFFFu, c1, 0);
    // reuse = the stage held an earlier region that this warp read through the generic proxy
    auto issue = [&](uint32_t s0, uint32_t s1, bool reuse) {
        const uint32_t bytes = 16 * (s1 - s0);
        if (bytes <= (uint32_t)kStageBytes) {
            if (lane == 0) {
                if (reuse) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                mbar_expect_tx(bar, bytes);
                tma_load_1d(stage, m.data + 16 * (uint64_t)s0, bytes, bar);
            }
            inflight = true;
        }
    };

    // The warp's own barrier and first region copy go first, so that the copy is in flight
    // while the CTA brings in (or builds) the decode table.
    if (lane == 0) {
        mbar_init(bar);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    if (b < m.nb) issue(c0, c1, false);
    lut_start(m, smem, lut_bar);
    __syncthreads();
    // Up to here only the matrix and its table were read. x, the workspace and y may belong to
    // the kernel before this one on the stream: wait for it to complete. The table copy is
    // waited for only before the first decode, so that it lands while the activations load
    // and the first region arrives.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const uint32_t lutb = smem_u32(smem);
    const uint64_t w_id = (uint64_t)blockIdx.x + (uint64_t)gridDim.x * warp;  // = the warp's first block
    const uint64_t ways = m.nb < total_warps ? m.nb : total_warps;
    bool prefetched = false, lut_ok = false;
    while (b < m.nb && !timed_out) {
        const uint64_t nxt = b + total_warps, nn = nxt + total_warps;
        uint32_t f0 = 0, f1 = 0;  // bounds of block nn, for the next iteration
        if (lane == 0) {
            if (nn < m.nb) {
                f0 = m.tab[nn];
                f1 = m.tab[nn + 1];
            }
            if (nxt < m.nb) l2_prefetch(m.data + 16 * (uint64_t)n0, 16 * (n1 - n0));
        }
        const uint32_t bytes = 16 * (c1 - c0);
        const uint8_t *src = m.data + 16 * (uint64_t)c0;
        const uint32_t rb32 = div_q((uint32_t)b, m.cdiv);
        const uint64_t rb = rb32, cb = b - (uint64_t)rb32 * m.cbs;
        const int rows = real_rows(m.n, rb);
        const uint64_t kc64 = m.k - cb * kCols;
        const int kc = kc64 < (uint64_t)kCols ? (int)kc64 : kCols;  // the block's real columns
        const uint16_t *xb = x + cb * kCols;
        float acc[NB][8];
#pragma unroll
        for (int v = 0; v < NB; v++)
#pragma unroll
            for (int r = 0; r < 8; r++) acc[v][r] = 0.0f;
        if (bytes <= (uint32_t)kStageBytes) {
            // the lane's activations, loaded while the region lands
            uint32_t xs[NB][8];
            const int cl = kc - kLaneCols * lane, cols = cl < 0 ? 0 : (cl > kLaneCols ? kLaneCols : cl);
#pragma unroll
            for (int v = 0; v < NB; v++) load_x16(xb + v * ld_x + kLaneCols * lane, cols, xs[v]);
            if (!mbar_wait(bar, phase & 1u)) {
                timed_out = true;
                break;
            }
            inflight = false;
            phase ^= 1u;
            if (!lut_ok) {
                if (!lut_ready(m, lut_bar)) {
                    timed_out = true;
                    break;
                }
                lut_ok = true;
            }
            if (!prefetched && lane == 0) prefetch_share(pf, w_id, ways);
            prefetched = true;
            if (KR && kc < kCols) gemv_block<ELEM, NB, KR>(stage, bytes, lane, lutb, xb, ld_x, xs, acc, bad, kc, rows);
            else gemv_block<ELEM, NB, false>(stage, bytes, lane, lutb, xb, ld_x, xs, acc, bad, kCols, rows);
        } else {
            if (!lut_ok) {
                if (!lut_ready(m, lut_bar)) {
                    timed_out = true;
                    break;
                }
                lut_ok = true;
            }
            if (!prefetched && lane == 0) prefetch_share(pf, w_id, ways);
            prefetched = true;
            gemv_block_global<ELEM, NB>(src, bytes, lane, lutb, xb, ld_x, acc, bad, kc, rows);
        }
        float sum[NB];
#pragma unroll
        for (int v = 0; v < NB; v++) sum[v] = transpose_reduce(acc[v], lane);
        finish_rows<ELEM, NB, SPEC>(m, sum, lane, rb, cb, y, ld_y, partial, counters, n_pad, timed_out);
        __syncwarp();
        c0 = __shfl_sync(0xFFFFFFFFu, n0, 0);
        c1 = __shfl_sync(0xFFFFFFFFu, n1, 0);
        if (nxt < m.nb) issue(c0, c1, true);
        n0 = f0;
        n1 = f1;
        b = nxt;
    }
    if (timed_out) {
        raise_error(kErrTimeout);
        // let this warp's own copy land before the CTA's shared memory goes away
        if (inflight) mbar_wait(bar, phase & 1u);
    }
    if (m.table) mbar_wait(lut_bar, 0);  // the table copy has landed (a no-op unless it timed out)
    if (bad) raise_error(kErrFormat);
}

// =================================================================== GEMV list
// y_i = W_i x_i for up to kListMax independent products in one launch. The items' blocks are
// numbered one after another (item by item, each in its blob's row-block-major order) and CTA c
// takes the contiguous range [c T / G, (c + 1) T / G) of the T blocks; its warps take the range's
// blocks item by item, warp w every kGemvWarps-th block from the item's first one in the range.
// A CTA thus meets only the few items its range crosses and brings in each one's decode table
// once: at an item boundary all warps meet at a barrier and thread 0 copies the next table over
// the previous one (each warp's first copy of the next item is already in flight). Each block
// is decoded, and its row block reduced, exactly as by gemv_kernel (the same code, the same
// fixed-order sum over column blocks, on the item's own workspace), so every y_i equals
// nwc_gemv's bit for bit.
constexpr int kListMax = NWC_GEMV_LIST_MAX;
struct ListItem {
    const uint32_t *tab;
    const uint8_t *data;
    const float *scales;
    const uint32_t *table;
    const uint16_t *x;
    float *y;
    float *partial;
    uint32_t *counters;
    uint64_t n, k, cbs, n_pad, start;  // start: the item's first block in the list's numbering
    Div cdiv;                          // division by cbs
};
struct ListParams {
    uint64_t total;  // blocks of all items
    int count;
    ListItem items[kListMax];
};
static_assert(sizeof(ListParams) <= 32764, "kernel parameters");

template <int ELEM, bool KR, bool SPEC>
__global__ void __launch_bounds__(kGemvWarps * 32, 1) gemv_list_kernel(const __grid_constant__ ListParams p) {
    using S = Smem<kGemvWarps>;
    constexpr uint64_t W = kGemvWarps;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t bar = smem_u32(smem + S::kBar + 8 * warp), lut_bar = smem_u32(smem + S::kLutBar);
    const uint32_t stage = smem_u32(smem + S::kStage + warp * kStageBytes);
    const uint32_t lutb = smem_u32(smem);
    const uint64_t s0 = p.total * blockIdx.x / gridDim.x, s1 = p.total * (blockIdx.x + 1) / gridDim.x;
    if (s0 >= s1) return;
    // the items the range crosses: f .. l
    int f = 0;
    while (f + 1 < p.count && p.items[f + 1].start <= s0) f++;
    int l = f;
    while (l + 1 < p.count && p.items[l + 1].start < s1) l++;
    auto load_table = [&](int j) {
        mbar_expect_tx(lut_bar, kLutBytes);
#pragma unroll
        for (int q = 0; q < 4; q++)
            tma_load_1d(lutb + q * (kLutBytes / 4), p.items[j].table + q * (kLutEntries / 4), kLutBytes / 4, lut_bar);
    };

    // The CTA's share of item j, [r0, r1) in the item's own block numbering, as work units taken
    // by the warps in turn (warp w: units w, w + W, ...). The first L units are whole row blocks
    // lying inside the share, L a multiple of W (every warp gets the same number): one warp
    // decodes all of such a row block's column blocks and sums them itself, in the order the
    // final sums of finish_rows use, so every y is bit for bit the same. The remaining units are
    // single blocks (those of the row blocks cut by the share's ends, and of the whole row blocks
    // left over), each with finish_rows' ticket; they keep the warps' shares within one block of
    // each other.
    // (block indices stay below 2^31, so the plan is kept in 32 bits)
    struct Plan {
        uint32_t r0, ra, L, nhead, single0, units, cbs;
    };
    auto plan_of = [&](int j) {
        const ListItem &it = p.items[j];
        const uint64_t e = j + 1 < p.count ? p.items[j + 1].start : p.total;
        Plan q;
        q.r0 = (uint32_t)((it.start > s0 ? it.start : s0) - it.start);
        const uint32_t r1 = (uint32_t)((e < s1 ? e : s1) - it.start);
        q.cbs = (uint32_t)it.cbs;
        const uint32_t ra = div_q(q.r0 + q.cbs - 1, it.cdiv), rz = div_q(r1, it.cdiv);
        const uint32_t whole = q.cbs > 1 && rz > ra ? rz - ra : 0;
        q.L = whole / W * W;
        if (q.L > 0) {
            q.ra = ra;
            q.nhead = ra * q.cbs - q.r0;
            q.single0 = (ra + q.L) * q.cbs;
        } else {
            q.ra = 0;
            q.nhead = r1 - q.r0;
            q.single0 = r1;
        }
        q.units = q.L + q.nhead + (r1 - q.single0);
        return q;
    };
    // A warp's walk through its units: step (u, k) is block k of unit u, in the item's block
    // numbering; next() moves to the following step.
    struct Walk {
        uint32_t u, k, b;
    };
    auto at = [&](const Plan &q, uint32_t u, uint32_t k) -> Walk {
        Walk w;
        w.u = u;
        w.k = k;
        if (u < q.L) {
            w.b = (q.ra + u) * q.cbs + k;
        } else {
            const uint32_t e = u - q.L;
            w.b = e < q.nhead ? q.r0 + e : q.single0 + (e - q.nhead);
        }
        return w;
    };
    auto next = [&](const Plan &q, const Walk &w) -> Walk {
        if (w.u < q.L && w.k + 1 < q.cbs) return Walk{w.u, w.k + 1, w.b + 1};
        return at(q, w.u + (uint32_t)W, 0);
    };

    uint32_t phase = 0;
    bool bad = false, timed_out = false, inflight = false;
    auto issue = [&](const uint8_t *data, uint32_t s0u, uint32_t s1u, bool reuse) {
        const uint32_t bytes = 16 * (s1u - s0u);
        if (bytes <= (uint32_t)kStageBytes) {
            if (lane == 0) {
                if (reuse) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                mbar_expect_tx(bar, bytes);
                tma_load_1d(stage, data + 16 * (uint64_t)s0u, bytes, bar);
            }
            inflight = true;
        }
    };
    // Bounds of the warp's current block (c0/c1, every lane) and of its next one (n0/n1, lane 0),
    // for the warp's first step in item j.
    uint32_t c0 = 0, c1 = 0, n0 = 0, n1 = 0;
    auto first_bounds = [&](int j) {
        const ListItem &it = p.items[j];
        const Plan q = plan_of(j);
        const Walk w0 = at(q, (uint32_t)warp, 0);
        c0 = c1 = n0 = n1 = 0;
        const bool have = w0.u < q.units;
        if (lane == 0 && have) {
            c0 = it.tab[w0.b];
            c1 = it.tab[w0.b + 1];
            const Walk w1 = next(q, w0);
            if (w1.u < q.units) {
                n0 = it.tab[w1.b];
                n1 = it.tab[w1.b + 1];
            }
        }
        c0 = __shfl_sync(0xFFFFFFFFu, c0, 0);
        c1 = __shfl_sync(0xFFFFFFFFu, c1, 0);
        return have;
    };

    // the warp's barrier and first copy, and the first item's table, before anything else
    if (lane == 0) {
        mbar_init(bar);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    if (first_bounds(f)) issue(p.items[f].data, c0, c1, false);
    if (threadIdx.x == 0) {
        mbar_init(lut_bar);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        load_table(f);
    }
    __syncthreads();
    // x, the workspaces and y may belong to the kernel before this one on the stream
    asm volatile("griddepcontrol.wait;" ::: "memory");

    for (int j = f; j <= l; j++) {
        const ListItem &it = p.items[j];
        Mat m;  // the fields finish_rows reads
        m.n = it.n;
        m.cbs = it.cbs;
        m.scales = it.scales;
        const Plan q = plan_of(j);
        if (j > f) {
            __syncthreads();  // every warp is done with the previous table
            if (threadIdx.x == 0) {
                // the previous copy has landed (already waited for, unless a wait timed out)
                mbar_wait(lut_bar, (uint32_t)(j - 1 - f) & 1u);
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                load_table(j);
            }
        }
        bool lut_ok = false;
        float sloc = 0.0f;  // a whole row block's sum so far (lane i: column blocks i / 8 mod 4)
        Walk w = at(q, (uint32_t)warp, 0), w1 = next(q, w), w2 = next(q, w1);
        while (w.u < q.units && !timed_out) {
            const bool has1 = w1.u < q.units, has2 = w2.u < q.units;
            uint32_t f0 = 0, f1 = 0;  // bounds of the step after next, for the next iteration
            if (lane == 0) {
                if (has2) {
                    f0 = it.tab[w2.b];
                    f1 = it.tab[w2.b + 1];
                }
                if (has1) l2_prefetch(it.data + 16 * (uint64_t)n0, 16 * (n1 - n0));
            }
            const uint32_t bytes = 16 * (c1 - c0);
            const uint32_t rb32 = div_q(w.b, it.cdiv);
            const uint64_t rb = rb32, cb = w.b - rb32 * q.cbs;
            const int rows = real_rows(it.n, rb);
            const uint64_t kc64 = it.k - cb * kCols;
            const int kc = kc64 < (uint64_t)kCols ? (int)kc64 : kCols;
            const uint16_t *xb = it.x + cb * kCols;
            float acc[1][8];
#pragma unroll
            for (int r = 0; r < 8; r++) acc[0][r] = 0.0f;
            if (bytes <= (uint32_t)kStageBytes) {
                uint32_t xs[1][8];
                const int cl = kc - kLaneCols * lane, cols = cl < 0 ? 0 : (cl > kLaneCols ? kLaneCols : cl);
                load_x16(xb + kLaneCols * lane, cols, xs[0]);
                if (!mbar_wait(bar, phase & 1u)) {
                    timed_out = true;
                    break;
                }
                inflight = false;
                phase ^= 1u;
                if (!lut_ok) {
                    if (!mbar_wait(lut_bar, (uint32_t)(j - f) & 1u)) {
                        timed_out = true;
                        break;
                    }
                    lut_ok = true;
                }
                if (KR && kc < kCols) gemv_block<ELEM, 1, KR>(stage, bytes, lane, lutb, xb, 0, xs, acc, bad, kc, rows);
                else gemv_block<ELEM, 1, false>(stage, bytes, lane, lutb, xb, 0, xs, acc, bad, kCols, rows);
            } else {
                if (!lut_ok) {
                    if (!mbar_wait(lut_bar, (uint32_t)(j - f) & 1u)) {
                        timed_out = true;
                        break;
                    }
                    lut_ok = true;
                }
                gemv_block_global<ELEM, 1>(it.data + 16 * (uint64_t)c0, bytes, lane, lutb, xb, 0, acc, bad, kc, rows);
            }
            float sum[1] = {transpose_reduce(acc[0], lane)};
            if (w.u >= q.L) {
                finish_rows<ELEM, 1, SPEC>(m, sum, lane, rb, cb, it.y, 0, it.partial, it.counters, it.n_pad, timed_out);
            } else {
                const float v = __shfl_sync(0xFFFFFFFFu, sum[0], row_holder(lane & 7));
                if ((uint32_t)(cb & 3u) == (uint32_t)(lane >> 3)) sloc += v;
                if (cb + 1 == it.cbs) {
                    sloc += __shfl_xor_sync(0xFFFFFFFFu, sloc, 8);
                    sloc += __shfl_xor_sync(0xFFFFFFFFu, sloc, 16);
                    const uint64_t r2 = rb * kRows + (uint64_t)(lane & 7);
                    if (lane < kRows && r2 < it.n) it.y[r2] = ELEM == 0 ? sloc : sloc * it.scales[r2];
                    sloc = 0.0f;
                }
            }
            __syncwarp();
            c0 = __shfl_sync(0xFFFFFFFFu, n0, 0);
            c1 = __shfl_sync(0xFFFFFFFFu, n1, 0);
            if (has1) issue(it.data, c0, c1, true);
            n0 = f0;
            n1 = f1;
            w = w1;
            w1 = w2;
            w2 = next(q, w2);
        }
        // the warp's first copy of the next item goes out before the barrier
        if (j < l && first_bounds(j + 1) && !timed_out) issue(p.items[j + 1].data, c0, c1, true);
    }
    if (timed_out) {
        raise_error(kErrTimeout);
        if (inflight) mbar_wait(bar, phase & 1u);
    }
    mbar_wait(lut_bar, (uint32_t)(l - f) & 1u);  // the last table copy has landed
    if (bad) raise_error(kErrFormat);
}

// =================================================================== small-batch GEMV
// Y[v] = W x[v] for up to 16 activation vectors (a few tokens per step) in one pass over the
// matrix: each weight is decoded once, as in the single-vector GEMV, and the products with all
// vectors are a dense contraction per block ([vectors x 512] . [512 x 8 rows]), done by the
// tensor cores. Per group of 4 columns the warp writes its decoded 8 x 128 tile to shared memory
// and runs eight m16n8k16 BF16 products with FP32 accumulation; the vectors are the M side, so
// any count up to 16 costs about the same. Listed elements are written into the tile with their
// true values, so no correction is needed. Each CTA takes a contiguous range of blocks in
// column-block-major order and stages the activations of its (at most two) column blocks in
// shared memory once.
constexpr int kBatchWarps = 19;
constexpr int kTileRow = 32 * 8 + 32;  // 32 lanes x 4 columns x BF16, padded by 32 bytes
constexpr int kTileBytes = 8 * kTileRow;
constexpr int kBatchTileOff = Smem<kBatchWarps>::kEnd;
constexpr int kBatchMax = 16;
constexpr int kXSlice = kBatchMax * kCols * 2;  // one column block of every vector, BF16
constexpr int kBatchXOff = kBatchTileOff + kBatchWarps * kTileBytes;
constexpr int kBatchSmem = kBatchXOff + 2 * kXSlice;
static_assert(kBatchSmem <= 232448, "shared memory per CTA");
static_assert(kBatchMax == NWC_GEMV_BATCH_MAX, "vectors per call");

// Byte offset in a staged activation slice of vector v, columns 4u..4u+3 of the column block
// (u = 4 * lane + group): 8-byte unit u ^ (v & 3), so the operand loads of one product (vectors
// gid, four lanes) fall in 16 distinct units per half-warp.
__device__ __forceinline__ uint32_t xs_off(uint32_t v, uint32_t u) { return v * (uint32_t)(kCols * 2) + 8u * (u ^ (v & 3)); }

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

// Four activations (columns c0 .. c0 + 3 of a column block starting at xv) as BF16 pairs;
// columns at or past kc (the block's real columns) read as 0.
__device__ __forceinline__ uint2 x4_load(const uint16_t *xv, int c0, int kc) {
    if (c0 + 4 <= kc) return __ldg(reinterpret_cast<const uint2 *>(xv + c0));
    uint32_t e[4];
#pragma unroll
    for (int j = 0; j < 4; j++) e[j] = c0 + j < kc ? (uint32_t)__ldg(xv + c0 + j) : 0u;
    return make_uint2(e[0] | e[1] << 16, e[2] | e[3] << 16);
}

// Block from its staged region, all vectors: d[0..3] receive the block's sums in the
// m16n8k16 accumulator layout (vector lane/4 rows 2(lane%4), +1 in d0, d1; vector lane/4 + 8 in
// d2, d3). The activations come from the CTA's staged slice at xs (shared address) when the
// block's column block is staged, else from global memory at x0/x1 (this thread's two vectors
// from the block's first column); v0/v1: those vectors exist (< nb). EDGE: the block's real
// columns kc < 512 (columns past K give 0 weights and 0 activations).
template <int ELEM, bool EDGE>
__device__ __forceinline__ void block_mma(uint32_t stage, uint32_t bytes, int lane, uint32_t lutb, uint32_t tile,
                                          bool staged_x, uint32_t xs, const uint16_t *x0, const uint16_t *x1, bool v0,
                                          bool v1, float (&d)[4], bool &bad, int kc, int rows) {
    const LaneBlock lb = lane_block<ELEM, EDGE>(stage, lane, kc);
    Fs s;
    fs_init(s, lb.code, lb.lw);
    const uint32_t lo = lb.list0 - stage;
    const uint32_t slots = lo <= bytes ? (bytes - lo) / 4u : 0u;
    const uint32_t gid = (uint32_t)lane >> 2, t = (uint32_t)lane & 3u;
    // this thread's B operand of product j in every group: row gid, lane 4j + t (32 j bytes on)
    const uint32_t bbase = tile + tile_off(gid, t);
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll 1
    for (int g = 0; g < 4; g++) {
        uint32_t w2[16];
        decode_group<ELEM, EDGE>(s, lutb, lb, g, w2);
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
        // listed elements of this group: their true values over the placeholders
        for (uint32_t j = (uint32_t)lane; j < slots; j += 32) {
            const uint32_t e = lds32(lb.list0 + 4u * j);
            if (e == kEscPad) continue;
            const uint32_t te = esc_t(e), c = te >> 3, r = te & 7u, l = esc_lane(e), v = esc_v(e);
            if ((c >> 2) != (uint32_t)g) continue;
            if ((int)r >= rows || (int)(kLaneCols * l + c) >= (EDGE ? kc : kCols) || (v >> exp_bits(ELEM))) {
                bad = true;
                continue;
            }
            uint32_t rawb = lds8(lb.raw0 + raw_offset<ELEM>(EDGE ? kc : kCols, l, c, r));
            if (ELEM == 1) rawb = (rawb >> (4u * (r & 1u))) & 0xFu;
            const uint32_t a = tile + tile_off(r, l) + 2u * (c & 3u);
            asm volatile("st.shared.u16 [%0], %1;" ::"r"(a), "h"((unsigned short)elem_bf16<ELEM>(rawb, v)) : "memory");
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
            asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(b0), "=r"(b1) : "r"(bbase + 32u * (uint32_t)j) : "memory");
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
    bad |= fs_overrun(s, lb.code, lb.lw);
#pragma unroll
    for (int i = 0; i < 4; i++) d[i] = acc[0][i] + acc[1][i];
}

// KR: K % 512 != 0, and the last column block's blocks take the tensor-core path with the
// ragged raw layout, in a kernel of its own so that the others keep the regular kernel's code.
template <int ELEM, bool KR = false>
__global__ void __launch_bounds__(kBatchWarps * 32, 1)
    gemv_batch_kernel(Mat m, const uint16_t *__restrict__ x, int64_t ld_x, int nb, float *__restrict__ y,
                      int64_t ld_y, float *partial, uint32_t *counters, uint64_t n_pad) {
    using S = Smem<kBatchWarps>;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t bar = smem_u32(smem + S::kBar + 8 * warp), lut_bar = smem_u32(smem + S::kLutBar);
    const uint32_t stage = smem_u32(smem + S::kStage + warp * kStageBytes);
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
    const uint32_t warps = blockDim.x >> 5;
    uint64_t p = start + (uint64_t)warp;
    // (rb, cb) of position p, stepped without division; (rbn, cbn) of the next position
    uint64_t cb = p / m.rbs, rb = p % m.rbs;
    auto step = [&](uint64_t &r, uint64_t &c) {
        r += warps;
        while (r >= m.rbs) {
            r -= m.rbs;
            c += 1;
        }
    };
    uint32_t phase = 0;
    bool bad = false, timed_out = false, inflight = false;
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
        if (bytes <= (uint32_t)kStageBytes) {
            if (lane == 0) {
                if (reuse) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                mbar_expect_tx(bar, bytes);
                tma_load_1d(stage, src, bytes, bar);
            }
            inflight = true;
        }
    };
    // result of vector v, row `row` (< n) of column block cb
    auto emit = [&](int v, uint64_t row, uint64_t cb2, float val) {
        if (m.cbs == 1) y[(int64_t)v * ld_y + (int64_t)row] = ELEM == 0 ? val : val * m.scales[row];
        else partial[((uint64_t)v * m.cbs + cb2) * n_pad + row] = val;
    };

    if (lane == 0) {
        mbar_init(bar);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    if (p < end) issue(rb * m.cbs + cb, false);
    lut_start(m, smem, lut_bar);
    __syncthreads();
    if (!lut_ready(m, lut_bar)) timed_out = true;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // stage the activations of column blocks cb_first and cb_first + 1 (whole 16-byte pieces
    // inside K; past K zeros, which the fillers of a ragged K meet)
    for (uint32_t i = threadIdx.x; i < 2u * (uint32_t)nb * (kCols / 8); i += blockDim.x) {
        const uint32_t slot = i / ((uint32_t)nb * (kCols / 8)), rem = i % ((uint32_t)nb * (kCols / 8));
        const uint32_t v = rem / (kCols / 8), c8 = rem % (kCols / 8);  // columns 8 c8 .. 8 c8 + 7
        const uint64_t col = (cb_first + slot) * kCols + 8 * (uint64_t)c8;
        uint4 q = make_uint4(0u, 0u, 0u, 0u);
        if (col + 8 <= m.k) {
            q = __ldg(reinterpret_cast<const uint4 *>(x + (int64_t)v * ld_x + (int64_t)col));
        } else if (col < m.k) {
            uint32_t e[8];
#pragma unroll
            for (int j = 0; j < 8; j++) e[j] = col + j < m.k ? (uint32_t)__ldg(x + (int64_t)v * ld_x + (int64_t)(col + j)) : 0u;
            q = make_uint4(e[0] | e[1] << 16, e[2] | e[3] << 16, e[4] | e[5] << 16, e[6] | e[7] << 16);
        }
        // columns 8 c8.. are lane c8 / 2, groups 2 (c8 & 1) and 2 (c8 & 1) + 1: units 2 c8, 2 c8 + 1
        const uint32_t xsl = xs0 + slot * (uint32_t)kXSlice;
        asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(xsl + xs_off(v, 2 * c8)), "r"(q.x), "r"(q.y) : "memory");
        asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(xsl + xs_off(v, 2 * c8 + 1)), "r"(q.z), "r"(q.w) : "memory");
    }
    __syncthreads();
    const uint32_t lutb = smem_u32(smem);

    while (p < end && !timed_out) {
        const uint64_t b = rb * m.cbs + cb;
        const uint64_t pn = p + warps;
        uint64_t rbn = rb, cbn = cb;
        step(rbn, cbn);
        const uint64_t bn = rbn * m.cbs + cbn;
        __syncwarp();
        if (pn < end && lane == 0) {
            const uint32_t s0 = m.tab[bn], s1 = m.tab[bn + 1];
            l2_prefetch(m.data + 16 * (uint64_t)s0, 16 * (s1 - s0));
        }
        const uint8_t *src;
        uint32_t bytes;
        region(b, src, bytes);
        const bool staged = bytes <= (uint32_t)kStageBytes;
        if (staged) {
            if (!mbar_wait(bar, phase & 1u)) {
                timed_out = true;
                break;
            }
            inflight = false;
            phase ^= 1u;
        }
        const int rows = real_rows(m.n, rb);
        const uint64_t kc64 = m.k - cb * kCols;
        const int kc = kc64 < (uint64_t)kCols ? (int)kc64 : kCols;  // the block's real columns
        if (staged && (KR || kc == kCols)) {
            const uint16_t *xc = x + cb * kCols;
            const bool v0 = gid < nb, v1 = gid + 8 < nb;
            const uint16_t *x0 = xc + (int64_t)(v0 ? gid : 0) * ld_x;
            const uint16_t *x1 = xc + (int64_t)(v1 ? gid + 8 : 0) * ld_x;
            const bool staged_x = cb == cb_first || cb == cb_first + 1;
            const uint32_t xs = xs0 + (cb == cb_first ? 0u : (uint32_t)kXSlice);
            float d[4];
            if (kc == kCols) block_mma<ELEM, false>(stage, bytes, lane, lutb, tile, staged_x, xs, x0, x1, v0, v1, d, bad, kCols, rows);
            else block_mma<ELEM, KR>(stage, bytes, lane, lutb, tile, staged_x, xs, x0, x1, v0, v1, d, bad, kc, rows);
            const uint64_t r0 = rb * kRows + 2 * (uint64_t)t;
            const bool in0 = r0 < m.n, in1 = r0 + 1 < m.n;
            if (v0) {
                if (in0) emit(gid, r0, cb, d[0]);
                if (in1) emit(gid, r0 + 1, cb, d[1]);
            }
            if (v1) {
                if (in0) emit(gid + 8, r0, cb, d[2]);
                if (in1) emit(gid + 8, r0 + 1, cb, d[3]);
            }
        } else {
            // regions read in place: the single-vector decoder per vector
            const uint64_t row = rb * kRows + (uint64_t)rowsel(lane);
            for (int v = 0; v < nb; v++) {
                float a1[1][8];
#pragma unroll
                for (int r = 0; r < 8; r++) a1[0][r] = 0.0f;
                gemv_block_global<ELEM, 1>(src, bytes, lane, lutb, x + (int64_t)v * ld_x + cb * kCols, 0, a1, bad, kc,
                                           rows);
                const float sum = transpose_reduce(a1[0], lane);
                if ((lane & 3) == 0 && row < m.n) emit(v, row, cb, sum);
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
                // (vector, row) pairs i, vector i / 8, row i % 8, summed over the column blocks in a
                // fixed order, every pair's loads of a round in flight together (4 pairs a lane at
                // 16 vectors); then each slot read goes back to the sentinel that the single- and
                // two-vector kernel expect of a prepared workspace.
                constexpr int PL = kBatchMax * kRows / 32;
                float sv[PL];
                bool live[PL];
                float *pp[PL];
#pragma unroll
                for (int k2 = 0; k2 < PL; k2++) {
                    const int i = lane + 32 * k2, v = i >> 3;
                    const uint64_t r2 = rb * kRows + (uint64_t)(i & 7);
                    live[k2] = v < nb && r2 < m.n;
                    pp[k2] = partial + (uint64_t)(live[k2] ? v : 0) * m.cbs * n_pad + r2;
                    sv[k2] = 0.0f;
                }
#pragma unroll 4
                for (uint64_t c2 = 0; c2 < m.cbs; c2++) {
#pragma unroll
                    for (int k2 = 0; k2 < PL; k2++)
                        if (live[k2]) sv[k2] += __ldcg(pp[k2] + c2 * n_pad);
                }
#pragma unroll
                for (int k2 = 0; k2 < PL; k2++) {
                    if (!live[k2]) continue;
                    const int i = lane + 32 * k2, v = i >> 3;
                    const uint64_t r2 = rb * kRows + (uint64_t)(i & 7);
                    y[(int64_t)v * ld_y + (int64_t)r2] = ELEM == 0 ? sv[k2] : sv[k2] * m.scales[r2];
                    for (uint64_t c2 = 0; c2 < m.cbs; c2++) __stcg(pp[k2] + c2 * n_pad, __uint_as_float(kSentinel));
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
        if (inflight) mbar_wait(bar, phase & 1u);
    }
    if (m.table) mbar_wait(lut_bar, 0);
    if (bad) raise_error(kErrFormat);
}

// =================================================================== decode and gather
// The pages run dequantization and the tied lm_head's embedding lookup on the GEMV's decoder;
// here too: the same table, staged regions and row-pair decoder. MODE 0 decodes every block to
// BF16 (fp8: e4m3 bytes); MODE 1 writes, for each id, that row of the block row, one block per
// warp item.

// e4m3 codes of a decoded fp8 row pair (a BF16x2 with exponent field v + 120, or 0): low byte
// row 2i, next byte row 2i + 1. Listed elements (placeholders here) are written afterwards.
__device__ __forceinline__ uint32_t e4m3_pair(uint32_t w2) {
    uint32_t q = 0;
#pragma unroll
    for (int h = 0; h < 2; h++) {
        const uint32_t b = w2 >> (16 * h), E = (b >> 7) & 0xFFu;
        const uint32_t v = E ? E - 120u : 0u;
        q |= (((b >> 8) & 0x80u) | ((v & 15u) << 3) | ((b >> 4) & 7u)) << (8 * h);
    }
    return q;
}

// Row words of 4 columns from a group's pairs p[4 c + pp] (rows 2pp, 2pp + 1 of column c):
// BF16 rows give two words (columns 0-1, 2-3), fp8 rows one word of four bytes (p holds the
// e4m3 pairs). hi selects row 2pp + 1.
template <int ELEM>
__device__ __forceinline__ uint2 row_words(uint32_t a, uint32_t b, uint32_t c, uint32_t d, bool hi) {
    if (ELEM == 0) {
        const uint32_t sel = hi ? 0x7632u : 0x5410u;
        return make_uint2(__byte_perm(a, b, sel), __byte_perm(c, d, sel));
    }
    const uint32_t sel = hi ? 0x0051u : 0x0040u;
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

// Writes the block's listed elements (`slots` list words at list0 / glist, raw bits at raw0 /
// graw) over their placeholders: element (r, c) of lane l to out[(row0 + r) ld_out + col0 + 16 l
// + c], only r == want when want >= 0 (then to row row0). Checks that the entries name real
// elements and that there are as many as the streams' escape and cut codes (nesc, summed over
// the warp; fp8 lists its subnormal and NaN codes as well, so it may hold more).
template <int ELEM>
__device__ __forceinline__ void unpack_patch(uint32_t list0, uint32_t raw0, const uint32_t *glist, const uint8_t *graw,
                                             uint32_t slots, int lane, uint32_t nesc, int kc, int rows, int want, void *out,
                                             int64_t ld_out, uint64_t row0, uint64_t col0, bool &bad) {
    uint32_t cnt = 0;
    for (uint32_t j = (uint32_t)lane; j < slots; j += 32) {
        const uint32_t e = glist ? __ldg(glist + j) : lds32(list0 + 4u * j);
        if (e == kEscPad) continue;
        cnt++;
        const uint32_t t = esc_t(e), l = esc_lane(e), v = esc_v(e), r = t & 7u, c = t >> 3;
        if ((int)r >= rows || (int)(kLaneCols * l + c) >= kc || (v >> exp_bits(ELEM))) {
            bad = true;
            continue;
        }
        if (want >= 0 && (int)r != want) continue;
        const uint32_t at = raw_offset<ELEM>(kc, l, c, r);
        uint32_t rawb = graw ? (uint32_t)__ldg(graw + at) : lds8(raw0 + at);
        const uint64_t o = (row0 + (want >= 0 ? 0u : r)) * (uint64_t)ld_out + col0 + kLaneCols * l + c;
        if (ELEM == 0) {
            static_cast<uint16_t *>(out)[o] = (uint16_t)(((rawb & 0x80u) << 8) | (v << 7) | (rawb & 0x7Fu));
        } else {
            rawb = (rawb >> (4u * (r & 1u))) & 0xFu;
            static_cast<uint8_t *>(out)[o] = (uint8_t)(((rawb & 8u) << 4) | (v << 3) | (rawb & 7u));
        }
    }
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) {
        cnt += __shfl_xor_sync(0xFFFFFFFFu, cnt, d);
        nesc += __shfl_xor_sync(0xFFFFFFFFu, nesc, d);
    }
    if (ELEM == 0 ? cnt != nesc : cnt < nesc) bad = true;
}

// Block from its staged region. Decode writes rows row0 .. row0 + rows - 1; gather writes row
// `want` of the block to output row row0. colb = the block's first column. EDGE: the block's
// real columns kc < 512.
template <int ELEM, int MODE, bool EDGE>
__device__ __forceinline__ void unpack_fast(uint32_t stage, uint32_t bytes, int lane, uint32_t lutb, void *out,
                                            int64_t ld_out, uint64_t row0, uint64_t colb, int want, int vec, bool &bad,
                                            int kc, int rows) {
    const LaneBlock lb = lane_block<ELEM, EDGE>(stage, lane, kc);
    Fs s;
    fs_init(s, lb.code, lb.lw);
    uint32_t nesc = 0;
    const int wpp = want >> 1;
    const bool whi = want & 1;
    // the lane's output tile: o[r][k] = row r, words k (BF16: 2 columns a word, fp8: 4)
    uint32_t o[MODE == 0 ? 8 : 1][8];
    auto group = [&](int g) {
        uint32_t p[16];  // p[4 c + pp]: rows (2pp, 2pp + 1) at column 4g + c
        decode_group<ELEM, EDGE, true>(s, lutb, lb, g, p, &nesc);
        if (ELEM == 1) {
#pragma unroll
            for (int q = 0; q < 16; q++) p[q] = e4m3_pair(p[q]);
        }
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
    const uint64_t col0 = colb + (uint64_t)(kLaneCols * lane);
    const int cols = EDGE ? lb.cols : kLaneCols;
    if (cols == kLaneCols) {
        if (MODE == 0) {
#pragma unroll
            for (int r = 0; r < 8; r++)
                if (r < rows) store_row16<ELEM>(out, (row0 + (uint64_t)r) * (uint64_t)ld_out + col0, o[r], vec);
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
    bad |= fs_overrun(s, lb.code, lb.lw);
    __syncwarp();  // the tile stores before any lane's patch of a listed element
    const uint32_t lo = lb.list0 - stage;
    const uint32_t slots = lo <= bytes ? (bytes - lo) / 4u : 0u;
    unpack_patch<ELEM>(lb.list0, lb.raw0, nullptr, nullptr, slots, lane, nesc, EDGE ? kc : kCols, rows,
                       MODE == 0 ? -1 : want, out, ld_out, row0, colb, bad);
}

// Any block read in place from global memory (a region too large for a stage), element by
// element: every word read bounded by the lane's own words, every raw read by the region.
template <int ELEM, int MODE>
__device__ __noinline__ bool unpack_global(const uint8_t *reg, uint32_t bytes, int lane, uint32_t lutb, void *out,
                                           int64_t ld_out, uint64_t row0, uint64_t colb, int want, int kc, int rows) {
    bool bad = false;
    const uint32_t lw = reg[lane];
    uint32_t incl = lw;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t o = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        if (lane >= d) incl += o;
    }
    const uint32_t total = __shfl_sync(0xFFFFFFFFu, incl, 31);
    const uint32_t *code = reinterpret_cast<const uint32_t *>(reg + 32) + (incl - lw);
    const uint32_t raw0 = (uint32_t)up16(32u + 4u * total);
    const uint32_t list0 = raw0 + raw_bytes<ELEM>(kc);
    if (list0 > bytes) return true;
    const int cl = kc - kLaneCols * lane, cols = cl < 0 ? 0 : (cl > kLaneCols ? kLaneCols : cl);
    const uint64_t col0 = colb + (uint64_t)(kLaneCols * lane);
    uint64_t win = 0;
    int nbits = 0;
    uint32_t wi = 0, used = 0, nesc = 0;
#pragma unroll 1
    for (int c = 0; c < kLaneCols; c++) {
#pragma unroll
        for (int i = 0; i < 4; i++) {
            while (nbits <= 32) {
                const uint32_t w = wi < lw ? __ldg(code + wi) : 0u;
                wi++;
                win |= (uint64_t)w << (32 - nbits);
                nbits += 32;
            }
            const uint32_t e = lds32(lutb + 4u * (uint32_t)(win >> (64 - kPeek)));
            const uint32_t L = e & 31u;
            win <<= L;
            nbits -= (int)L;
            used += L;
            nesc += (e >> 16) & 3u;
            if (c >= cols) continue;
            const uint32_t at = raw_offset<ELEM>(kc, (uint32_t)lane, (uint32_t)c, 2u * i);
#pragma unroll
            for (int h = 0; h < 2; h++) {
                const int r = 2 * i + h;
                if (r >= rows || (MODE == 1 && r != want)) continue;
                const uint32_t E = (e >> (h ? 23 : 7)) & 0xFFu;
                const uint64_t o = (MODE == 0 ? row0 + (uint64_t)r : row0) * (uint64_t)ld_out + col0 + (uint64_t)c;
                if (ELEM == 0) {
                    const uint32_t b = reg[raw0 + at + h];
                    static_cast<uint16_t *>(out)[o] = (uint16_t)(((b & 0x80u) << 8) | (E << 7) | (b & 0x7Fu));
                } else {
                    const uint32_t b = (reg[raw0 + at] >> (4 * h)) & 0xFu;
                    const uint32_t v = E ? E - 120u : 0u;
                    static_cast<uint8_t *>(out)[o] = (uint8_t)(((b & 8u) << 4) | ((v & 15u) << 3) | (b & 7u));
                }
            }
        }
    }
    bad |= used > 32u * lw;
    __syncwarp();
    unpack_patch<ELEM>(0u, 0u, reinterpret_cast<const uint32_t *>(reg + list0), reg + raw0, (bytes - list0) / 4u, lane,
                       nesc, kc, rows, MODE == 0 ? -1 : want, out, ld_out, row0, colb, bad);
    return bad;
}

// Decode: 16 warps per SM with up to 128 registers each, so that a lane holds its whole 8x16
// output tile and writes every 32-byte row segment with full-sector stores. Gather keeps one
// row per lane and runs 32 warps.
template <int MODE>
struct UnpackCfg {
    static constexpr int kWarps = MODE == 0 ? 16 : 32;
    static constexpr int kSmem = Smem<kWarps>::kEnd + kStageSlack;
};
static_assert(UnpackCfg<0>::kSmem <= 232448 && UnpackCfg<1>::kSmem <= 232448, "shared memory per CTA");

// KR: K % 512 != 0 (the last column block takes the fast decoder with the ragged raw layout, in
// a kernel of its own so that the regular decode and gather keep their registers).
template <int ELEM, int MODE, bool KR = false>
__global__ void __launch_bounds__(UnpackCfg<MODE>::kWarps * 32, 1)
    unpack_kernel(Mat m, const int32_t *ids, uint64_t n_items, void *out, int64_t ld_out, int vec) {
    using S = Smem<UnpackCfg<MODE>::kWarps>;
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t bar = smem_u32(smem + S::kBar + 8 * warp), lut_bar = smem_u32(smem + S::kLutBar);
    const uint32_t stage = smem_u32(smem + S::kStage + warp * kStageBytes);
    const uint64_t stride = (uint64_t)gridDim.x * UnpackCfg<MODE>::kWarps;
    uint32_t phase = 0;
    bool bad = false, timed_out = false, inflight = false;

    // Work item it -> block b, wanted row (gather) and first output row. Gather ids are read by
    // lane 0 and broadcast; an out-of-range id gives ok = false.
    auto locate = [&](uint64_t it, uint64_t &b, int &want, uint64_t &orow, bool &ok) {
        if (MODE == 0) {
            b = it;
            want = -1;
            orow = (uint64_t)div_q((uint32_t)it, m.cdiv) * kRows;
            ok = true;
        } else {
            const uint64_t i = div_q((uint32_t)it, m.cdiv), cb = it - i * m.cbs;
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
        if (bytes <= (uint32_t)kStageBytes) {
            if (lane == 0) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                mbar_expect_tx(bar, bytes);
                tma_load_1d(stage, src, bytes, bar);
            }
            inflight = true;
        }
    };

    if (lane == 0) {
        mbar_init(bar);
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
    lut_start(m, smem, lut_bar);
    __syncthreads();
    if (!lut_ready(m, lut_bar)) timed_out = true;
    const uint32_t lutb = smem_u32(smem);

    while (it < n_items && !timed_out) {
        const uint64_t nxt = it + stride;
        uint64_t nb_ = 0, norow = 0;
        int nwant = 0;
        bool nok = false;
        if (nxt < n_items) {
            locate(nxt, nb_, nwant, norow, nok);
            if (nok && lane == 0) {
                const uint32_t s0 = m.tab[nb_], s1 = m.tab[nb_ + 1];
                l2_prefetch(m.data + 16 * (uint64_t)s0, 16 * (s1 - s0));
            }
        }
        const uint64_t cb = it - (uint64_t)div_q((uint32_t)it, m.cdiv) * m.cbs;
        const uint64_t colb = cb * kCols;
        if (!ok) {
            // gather id out of range: a zero row, and the error word
            if (lane == 0 && cb == 0) raise_error(kErrId);
            const int cols = real_cols(m.k, cb, lane);
            const uint64_t col0 = colb + (uint64_t)(kLaneCols * lane);
            for (int c = 0; c < cols; c++) {
                if (ELEM == 0) static_cast<uint16_t *>(out)[orow * (uint64_t)ld_out + col0 + c] = 0;
                else static_cast<uint8_t *>(out)[orow * (uint64_t)ld_out + col0 + c] = 0;
            }
        } else {
            const uint8_t *src;
            uint32_t bytes;
            region(b, src, bytes);
            const uint64_t rb = div_q((uint32_t)b, m.cdiv);
            const int rows = real_rows(m.n, rb);
            const uint64_t kc64 = m.k - cb * kCols;
            const int kc = kc64 < (uint64_t)kCols ? (int)kc64 : kCols;  // the block's real columns
            if (bytes <= (uint32_t)kStageBytes) {
                if (!mbar_wait(bar, phase & 1u)) {
                    timed_out = true;
                    break;
                }
                inflight = false;
                phase ^= 1u;
                if (KR && kc < kCols)
                    unpack_fast<ELEM, MODE, KR>(stage, bytes, lane, lutb, out, ld_out, orow, colb, want, vec, bad, kc, rows);
                else
                    unpack_fast<ELEM, MODE, false>(stage, bytes, lane, lutb, out, ld_out, orow, colb, want, vec, bad, kCols,
                                                   rows);
            } else {
                bad |= unpack_global<ELEM, MODE>(src, bytes, lane, lutb, out, ld_out, orow, colb, want, kc, rows);
            }
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
        if (inflight) mbar_wait(bar, phase & 1u);  // let this warp's copy land before shared memory goes away
    }
    if (m.table) mbar_wait(lut_bar, 0);
    if (bad) raise_error(kErrFormat);
}

// =================================================================== host side
// Per-device state: every device the process uses gets its own SM count and its own
// raised shared-memory limit for each kernel (a function attribute applies to the current
// device's context only).
constexpr int kMaxDevices = 64;
std::mutex g_mu;
int g_sm_count[kMaxDevices];
bool g_sm_known[kMaxDevices];

int current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
}

int sm_count() {
    const int dev = current_device();
    if (dev < 0) return 0;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_sm_known[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 0;
        g_sm_count[dev] = n;
        g_sm_known[dev] = true;
    }
    return g_sm_count[dev];
}

// Raises kernel K's dynamic shared-memory limit on the current device, once per device.
template <auto K>
bool smem_ready(int bytes) {
    static bool done[kMaxDevices];
    static std::mutex mu;
    const int dev = current_device();
    if (dev < 0) return false;
    std::lock_guard<std::mutex> lk(mu);
    if (!done[dev]) {
        if (cudaFuncSetAttribute(K, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) return false;
        done[dev] = true;
    }
    return true;
}

nwc_status launched() { return cudaGetLastError() == cudaSuccess ? NWC_OK : NWC_ERR_CUDA; }

uint64_t pad_rows(const nwc_matrix &m) { return (uint64_t)m.row_blocks * kRows; }

// Launch with programmatic stream serialization: the kernel may start while the previous
// kernel on the stream finishes; it streams its first block regions and brings in its decode
// table meanwhile.
template <class... A>
cudaError_t launch_pdl(void (*kernel)(A...), int grid, int threads, int smem, cudaStream_t s, A... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <int ELEM, int MODE, bool KR>
nwc_status launch_unpack(const Mat &m, const int32_t *ids, uint64_t n_items, void *out, int64_t ld_out, int vec,
                         cudaStream_t s) {
    const int sms = sm_count();
    if (sms <= 0) return NWC_ERR_CUDA;
    using C = UnpackCfg<MODE>;
    if (!smem_ready<unpack_kernel<ELEM, MODE, KR>>(C::kSmem)) return NWC_ERR_CUDA;
    const int grid = (int)(n_items < (uint64_t)sms ? n_items : (uint64_t)sms);
    unpack_kernel<ELEM, MODE, KR><<<grid, C::kWarps * 32, C::kSmem, s>>>(m, ids, n_items, out, ld_out, vec);
    return launched();
}

// Widest store (16, 8 or 4 bytes; 0: element-wise) that every 16-column row segment of out allows:
// segments start at out + (r ld_out + 16 j) elements.
int vec_ok(const void *out, int64_t ld_out, int elem) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(out);
    const int64_t esz = elem == NWC_ELEM_BF16 ? 2 : 1;
    for (int v = 16; v >= 4; v /= 2)
        if ((a % v) == 0 && ((ld_out * esz) % v) == 0) return v;
    return 0;
}

bool k_ragged(const Mat &m) { return (m.k % kCols) != 0; }

}  // namespace

extern "C" int nwc_sm_count(void) { return sm_count(); }

extern "C" nwc_status nwc_decode_table(const nwc_matrix *mp, uint32_t *table_host) {
    if (!mp || !table_host) return NWC_ERR_INVALID_ARG;
    if (mp->n_ranked < 1 || mp->n_ranked > kMaxRanked || (mp->elem != NWC_ELEM_BF16 && mp->elem != NWC_ELEM_FP8_E4M3))
        return NWC_ERR_INVALID_ARG;
    for (uint32_t i = 0; i < (uint32_t)kLutEntries; i++) table_host[i] = table_entry(i, mp->n_ranked, mp->elem, mp->rank_exp);
    return NWC_OK;
}

extern "C" nwc_status nwc_decode(const nwc_matrix *mp, void *out, int64_t ld_out, float *scales_out, nwc_stream stream) {
    if (!mp || !out || ld_out < mp->k) return NWC_ERR_INVALID_ARG;
    const Mat m = to_mat(*mp);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int vec = vec_ok(out, ld_out, m.elem);
    const bool kr = k_ragged(m);
    nwc_status st;
    if (m.elem == NWC_ELEM_BF16)
        st = kr ? launch_unpack<0, 0, true>(m, nullptr, m.nb, out, ld_out, vec, s)
                : launch_unpack<0, 0, false>(m, nullptr, m.nb, out, ld_out, vec, s);
    else
        st = kr ? launch_unpack<1, 0, true>(m, nullptr, m.nb, out, ld_out, vec, s)
                : launch_unpack<1, 0, false>(m, nullptr, m.nb, out, ld_out, vec, s);
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
    // work items (id, column block) are numbered below 2^31
    if ((uint64_t)n_ids >= ((1ull << 31) - 1) / m.cbs) return NWC_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int vec = vec_ok(out, ld_out, m.elem);
    const uint64_t items = (uint64_t)n_ids * m.cbs;
    const bool kr = k_ragged(m);
    if (m.elem == NWC_ELEM_BF16)
        return kr ? launch_unpack<0, 1, true>(m, ids, items, out, ld_out, vec, s)
                  : launch_unpack<0, 1, false>(m, ids, items, out, ld_out, vec, s);
    return kr ? launch_unpack<1, 1, true>(m, ids, items, out, ld_out, vec, s)
              : launch_unpack<1, 1, false>(m, ids, items, out, ld_out, vec, s);
}

namespace {
// Workspace: [partial sums fp32 col_blocks x n_pad, every slot the sentinel][counters u32
// row_blocks, zero]; both only when K > 512.
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
    uint8_t *w8 = static_cast<uint8_t *>(ws);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(w8, 0xFF, (size_t)ws_counter_off(*mp), s) != cudaSuccess) return NWC_ERR_CUDA;
    return cudaMemsetAsync(w8 + ws_counter_off(*mp), 0, 4 * (size_t)mp->row_blocks, s) == cudaSuccess ? NWC_OK
                                                                                                      : NWC_ERR_CUDA;
}

namespace {
template <int ELEM, int NB, bool KR, bool SPEC>
cudaError_t launch_gemv_k(const Mat &m, const uint16_t *x, int64_t ld_x, float *y, int64_t ld_y, float *partial,
                          uint32_t *counters, uint64_t n_pad, const Prefetch &pf, int grid, int warps,
                          cudaStream_t stream) {
    using C = GemvCfg<NB>;
    if (!smem_ready<gemv_kernel<ELEM, NB, KR, SPEC>>(C::kSmem)) return cudaErrorInvalidConfiguration;
    return launch_pdl(gemv_kernel<ELEM, NB, KR, SPEC>, grid, warps * 32, C::kSmem, stream, m, x, ld_x, y, ld_y,
                      partial, counters, n_pad, pf);
}

template <int ELEM, int NB>
cudaError_t launch_gemv_nb(const Mat &m, const uint16_t *x, int64_t ld_x, float *y, int64_t ld_y, float *partial,
                           uint32_t *counters, uint64_t n_pad, const Prefetch &pf, int sms, cudaStream_t stream) {
    using C = GemvCfg<NB>;
    const int grid = (int)(m.nb < (uint64_t)sms ? m.nb : (uint64_t)sms);
    // The fewest warps per CTA that keep the number of rounds (blocks per warp) of a full CTA, so
    // that every warp of a round has a block: 6080 blocks on 152 SMs take 20 warps with two blocks
    // each instead of 32 warps of which a quarter decode a second block alone.
    const uint64_t rounds = cdiv(m.nb, (uint64_t)grid * C::kWarps);
    const int warps = (int)cdiv(m.nb, rounds * (uint64_t)grid);
    const bool spec = rounds > 1;  // some warps decode more than one block
    if (k_ragged(m))
        return spec ? launch_gemv_k<ELEM, NB, true, true>(m, x, ld_x, y, ld_y, partial, counters, n_pad, pf, grid, warps, stream)
                    : launch_gemv_k<ELEM, NB, true, false>(m, x, ld_x, y, ld_y, partial, counters, n_pad, pf, grid, warps, stream);
    return spec ? launch_gemv_k<ELEM, NB, false, true>(m, x, ld_x, y, ld_y, partial, counters, n_pad, pf, grid, warps, stream)
                : launch_gemv_k<ELEM, NB, false, false>(m, x, ld_x, y, ld_y, partial, counters, n_pad, pf, grid, warps, stream);
}

template <int ELEM, bool KR>
cudaError_t launch_list(const ListParams &p, int grid, cudaStream_t s);

// The list launch's parameters (28 KB) for the calling thread, kept off the stack.
ListParams &list_params() {
    static thread_local ListParams p;
    return p;
}
// Item i of a list launch: matrix m with x, y and its workspace's partial sums and counters.
void set_item(ListParams &p, int i, const Mat &m, const uint16_t *x, float *y, float *partial, uint32_t *counters,
              uint64_t n_pad) {
    ListItem &d = p.items[i];
    d.tab = m.tab;
    d.data = m.data;
    d.scales = m.scales;
    d.table = m.table;
    d.x = x;
    d.y = y;
    d.partial = partial;
    d.counters = counters;
    d.n = m.n;
    d.k = m.k;
    d.cbs = m.cbs;
    d.n_pad = n_pad;
    d.start = p.total;
    d.cdiv = m.cdiv;
    p.total += m.nb;
}

// Which kernel the GEMV of m for nb vectors (with a next matrix to prefetch or not) launches.
// A tall matrix (every SM's share of the blocks holds at least 32 whole row blocks) runs the
// list kernel with one item: its whole row blocks are summed by one warp each, without partial
// sums, with the same y bit for bit (the list kernel needs the device decode table).
int route_of(const Mat &m, int nb, bool next, int sms) {
    if (nb == 1 && !next && m.table && m.cbs > 1 && m.rbs >= 33 * (uint64_t)sms) return NWC_ROUTE_LIST;
    return NWC_ROUTE_GEMV;
}

// The GEMV for nb = 1 or 2 vectors on `partial` (nb x col_blocks x n_pad floats, sentinels) and
// `counters` (row_blocks, zero); arguments already checked. next: the matrix to prefetch, or null.
nwc_status launch_gemv(const Mat &m, const uint16_t *x, int64_t ld_x, float *y, int64_t ld_y, int nb, float *partial,
                       uint32_t *counters, uint64_t n_pad, cudaStream_t stream, const nwc_matrix *next = nullptr) {
    const int sms = sm_count();
    if (sms <= 0) return NWC_ERR_CUDA;
    if (route_of(m, nb, next != nullptr, sms) == NWC_ROUTE_LIST) {
        ListParams &p = list_params();
        p.count = 1;
        p.total = 0;
        set_item(p, 0, m, x, y, partial, counters, n_pad);
        const int grid = sms;
        const bool kr = k_ragged(m);
        cudaError_t rc;
        if (m.elem == NWC_ELEM_BF16) rc = kr ? launch_list<0, true>(p, grid, stream) : launch_list<0, false>(p, grid, stream);
        else rc = kr ? launch_list<1, true>(p, grid, stream) : launch_list<1, false>(p, grid, stream);
        return rc == cudaSuccess ? NWC_OK : NWC_ERR_CUDA;
    }
    Prefetch pf = {nullptr, 0, nullptr, 0, nullptr};
    if (next && next->data && next->block_tab) {
        pf.data = next->data;
        pf.bytes = next->data_bytes & ~uint64_t(15);
        pf.tab = next->block_tab;
        pf.tab_bytes = up16(4 * ((uint64_t)next->row_blocks * (uint64_t)next->col_blocks + 1)) & ~uint64_t(15);
        pf.table = next->table;
    }
    cudaError_t rc;
    if (nb == 1)
        rc = m.elem == NWC_ELEM_BF16 ? launch_gemv_nb<0, 1>(m, x, ld_x, y, ld_y, partial, counters, n_pad, pf, sms, stream)
                                     : launch_gemv_nb<1, 1>(m, x, ld_x, y, ld_y, partial, counters, n_pad, pf, sms, stream);
    else
        rc = m.elem == NWC_ELEM_BF16 ? launch_gemv_nb<0, 2>(m, x, ld_x, y, ld_y, partial, counters, n_pad, pf, sms, stream)
                                     : launch_gemv_nb<1, 2>(m, x, ld_x, y, ld_y, partial, counters, n_pad, pf, sms, stream);
    return rc == cudaSuccess ? NWC_OK : NWC_ERR_CUDA;
}
}  // namespace

extern "C" nwc_status nwc_gemv_next(const nwc_matrix *mp, const uint16_t *x, float *y, void *ws, size_t ws_bytes,
                                    const nwc_matrix *next, nwc_stream stream) {
    if (!mp || !x || !y || !ws) return NWC_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(x) & 15) || (reinterpret_cast<uintptr_t>(ws) & 15)) return NWC_ERR_INVALID_ARG;
    if (ws_bytes < nwc_gemv_workspace_bytes(mp)) return NWC_ERR_INVALID_ARG;
    uint8_t *w8 = static_cast<uint8_t *>(ws);
    return launch_gemv(to_mat(*mp), x, 0, y, 0, 1, reinterpret_cast<float *>(w8),
                       reinterpret_cast<uint32_t *>(w8 + ws_counter_off(*mp)), pad_rows(*mp),
                       reinterpret_cast<cudaStream_t>(stream), next);
}

extern "C" nwc_status nwc_gemv(const nwc_matrix *mp, const uint16_t *x, float *y, void *ws, size_t ws_bytes,
                               nwc_stream stream) {
    return nwc_gemv_next(mp, x, y, ws, ws_bytes, nullptr, stream);
}

extern "C" nwc_status nwc_gemv_route(const nwc_matrix *mp, int *route) {
    if (!mp || !route) return NWC_ERR_INVALID_ARG;
    const int sms = sm_count();
    if (sms <= 0) return NWC_ERR_CUDA;
    *route = route_of(to_mat(*mp), 1, false, sms);
    return NWC_OK;
}

// ---------------------------------------------------------------- GEMV list
namespace {
template <int ELEM, bool KR, bool SPEC>
cudaError_t launch_list_k(const ListParams &p, int grid, cudaStream_t s) {
    if (!smem_ready<gemv_list_kernel<ELEM, KR, SPEC>>(kGemvSmem)) return cudaErrorInvalidConfiguration;
    return launch_pdl(gemv_list_kernel<ELEM, KR, SPEC>, grid, kGemvWarps * 32, kGemvSmem, s, p);
}
template <int ELEM, bool KR>
cudaError_t launch_list(const ListParams &p, int grid, cudaStream_t s) {
    // some warps decode more than one block: the final sums' speculative loads (finish_rows)
    return p.total > (uint64_t)grid * kGemvWarps ? launch_list_k<ELEM, KR, true>(p, grid, s)
                                                 : launch_list_k<ELEM, KR, false>(p, grid, s);
}
}  // namespace

extern "C" nwc_status nwc_gemv_list(const nwc_gemv_item *items, int count, nwc_stream stream) {
    if (!items || count < 1 || count > kListMax) return NWC_ERR_INVALID_ARG;
    ListParams &p = list_params();
    std::vector<std::pair<uintptr_t, uintptr_t>> used;  // workspace bytes the items touch
    p.count = count;
    p.total = 0;
    int elem = -1;
    bool kr = false;
    for (int i = 0; i < count; i++) {
        const nwc_gemv_item &it = items[i];
        if (!it.m || !it.x || !it.y || !it.ws) return NWC_ERR_INVALID_ARG;
        const nwc_matrix &m = *it.m;
        if (!m.table || (reinterpret_cast<uintptr_t>(m.table) & 15)) return NWC_ERR_INVALID_ARG;
        if ((reinterpret_cast<uintptr_t>(it.x) & 15) || (reinterpret_cast<uintptr_t>(it.ws) & 15)) return NWC_ERR_INVALID_ARG;
        if (it.ws_bytes < nwc_gemv_workspace_bytes(&m)) return NWC_ERR_INVALID_ARG;
        if (elem >= 0 && m.elem != elem) return NWC_ERR_INVALID_ARG;
        elem = m.elem;
        kr |= (m.k % kCols) != 0;
        set_item(p, i, to_mat(m), it.x, it.y, static_cast<float *>(it.ws),
                 reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(it.ws) + ws_counter_off(m)), pad_rows(m));
        if (m.col_blocks > 1) {
            const uintptr_t a = reinterpret_cast<uintptr_t>(it.ws);
            used.push_back({a, a + nwc_gemv_workspace_bytes(&m)});
        }
    }
    std::sort(used.begin(), used.end());
    for (size_t i = 1; i < used.size(); i++)
        if (used[i].first < used[i - 1].second) return NWC_ERR_INVALID_ARG;  // two items share workspace
    const int sms = sm_count();
    if (sms <= 0) return NWC_ERR_CUDA;
    const int grid = (int)(p.total < (uint64_t)sms ? p.total : (uint64_t)sms);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t rc;
    if (elem == NWC_ELEM_BF16) rc = kr ? launch_list<0, true>(p, grid, s) : launch_list<0, false>(p, grid, s);
    else rc = kr ? launch_list<1, true>(p, grid, s) : launch_list<1, false>(p, grid, s);
    return rc == cudaSuccess ? NWC_OK : NWC_ERR_CUDA;
}

// ---------------------------------------------------------------- small-batch GEMV
namespace {
// Batch workspace: [counters u32 row_blocks, padded to 16 B, zero][partials fp32 nb x col_blocks
// x n_pad, sentinels]; both only when K > 512. The counters come first, so a workspace prepared
// for nb vectors serves every smaller count.
uint64_t wsb_partial_off(const nwc_matrix &m) { return up16(4 * (uint64_t)m.row_blocks); }

template <int ELEM>
cudaError_t launch_batch(const Mat &m, const uint16_t *x, int64_t ld_x, int nb, float *y, int64_t ld_y, void *ws,
                         uint64_t n_pad, int grid, cudaStream_t s) {
    uint8_t *w8 = static_cast<uint8_t *>(ws);
    uint32_t *counters = reinterpret_cast<uint32_t *>(w8);
    float *partial = reinterpret_cast<float *>(w8 + (m.cbs > 1 ? up16(4 * m.rbs) : 0));
    // a CTA's range of `per` positions takes r = ceil(per / kBatchWarps) rounds of its warps;
    // the fewest warps that keep r rounds leave no warp of the last round decoding alone
    const uint64_t per = (m.nb + (uint64_t)grid - 1) / (uint64_t)grid;
    const uint64_t rounds = (per + kBatchWarps - 1) / kBatchWarps;
    const int warps = rounds == 0 ? kBatchWarps : (int)((per + rounds - 1) / rounds);
    if (k_ragged(m)) {
        if (!smem_ready<gemv_batch_kernel<ELEM, true>>(kBatchSmem)) return cudaErrorInvalidConfiguration;
        return launch_pdl(gemv_batch_kernel<ELEM, true>, grid, warps * 32, kBatchSmem, s, m, x, ld_x, nb, y, ld_y,
                          partial, counters, n_pad);
    }
    if (!smem_ready<gemv_batch_kernel<ELEM, false>>(kBatchSmem)) return cudaErrorInvalidConfiguration;
    return launch_pdl(gemv_batch_kernel<ELEM, false>, grid, warps * 32, kBatchSmem, s, m, x, ld_x, nb, y, ld_y,
                      partial, counters, n_pad);
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
    uint8_t *w8 = static_cast<uint8_t *>(ws);
    if (cudaMemsetAsync(w8, 0, (size_t)wsb_partial_off(*mp), s) != cudaSuccess) return NWC_ERR_CUDA;
    return cudaMemsetAsync(w8 + wsb_partial_off(*mp), 0xFF, need - (size_t)wsb_partial_off(*mp), s) == cudaSuccess
               ? NWC_OK
               : NWC_ERR_CUDA;
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
    // The array keeps whatever the previous call left: put this matrix's slots and counters in
    // their starting state, then run the GEMV on the same stream.
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
