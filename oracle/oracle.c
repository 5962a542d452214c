/*
 * oracle.c -- plain, slow CPU reference for the NWC entropy-coded matrix format.
 *
 * TEST INFRASTRUCTURE ONLY. The product library never links, loads or calls this
 * file; only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg use it.
 * It shares no code with the library (decode_gemv_nwc_gb300/csrc): both are written
 * independently from the format definition below.
 *
 * Sources (the pages this restates; reading choices are marked READING):
 *   [P1] "NWC -- Neural Weight Compression" (PyPI project page, v0.9.0),
 *        section "How it works":
 *          - byte planes: the mantissa is stored raw, the exponent/sign part is
 *            entropy coded;
 *          - prefix code: exponent ranked by frequency, written as a unary rank code
 *            plus a raw sign bit, escape for rare values;
 *          - fused kernel: each lane decodes its own bit stream for a block of
 *            8 rows x 512 columns (16 columns x 8 rows per lane); any shape works,
 *            padding costs 2 bits per filler weight and no mantissa.
 *   [P2] "Qwen3-4B-NWC-fp8" (model card): weight-only fp8 e4m3 with a symmetric
 *        per-output-channel scale; the fp8 bytes are coded losslessly.
 *
 * FORMAT (little-endian):
 *   header, 64 bytes
 *     0  u32 magic 0x3143574E ("NWC1")      4  u16 version = 3
 *     6  u8  elem (0 = BF16, 1 = FP8 e4m3)  7  u8  n_ranked (1..11)
 *     8  u64 N    16 u64 K    24 u64 n_blocks = ceil(N/8) * ceil(K/512)
 *     32 u64 off_blocks   40 u64 off_scales (0 for BF16)   48 u64 off_data
 *     56 u64 total_bytes
 *   64: u8 rank_exp[16]  -- exponent value of rank 0..n_ranked-1, rest zero
 *   off_blocks: u32 tab[n_blocks + 1]; block b occupies bytes
 *        [off_data + 16*tab[b], off_data + 16*tab[b+1]); padded to 16 bytes
 *   off_scales (FP8 only): f32 scale[N]; padded to 16 bytes
 *   off_data: block regions, row-block-major (b = rb * CB + cb)
 *   block region: u8 lane_words[32]; then the 32 lane code streams (lane 0 first),
 *     each a whole number of u32 words; zero padding to 16 bytes; then the 32 lane
 *     mantissa regions (lane 0 first), each a multiple of 16 bytes; then the block's
 *     escape list: one u32 per escaped element, t | lane << 7 | value << 12 (value =
 *     the element's full bit pattern), lanes in order and t increasing within a lane,
 *     padded to 16 bytes with 0xFFFFFFFF.
 *
 *   Fields of one element (READING: BF16 splits into a raw 7-bit mantissa and a
 *   coded 8-bit exponent with a raw sign; fp8 likewise with 4-bit exponent, 3-bit
 *   mantissa):  BF16 b: s = b>>15, v = (b>>7)&0xFF, m = b&0x7F
 *               FP8  q: s = q>>7,  v = (q>>3)&0xF,  m = q&7
 *   Ranking: histogram of v over the N*K real elements; ranks by (count desc,
 *     v asc) over values with count > 0; n_ranked = min(11, #distinct values).
 *     (READING: tie-break by ascending value; at most 11 ranked values so that any
 *     ranked code with its sign fits a 12-bit peek.)
 *   Code of one element, bits appended in order:
 *     ranked (rank p < n_ranked): p one-bits, one zero-bit, the sign bit;
 *     escape (v unranked): n_ranked one-bits, the sign bit; the element's exponent
 *     bits (8 BF16 / 4 fp8, with the rest of the element) are in the block's escape
 *     list. (READING: the pages' escape for rare exponents, with the raw exponent kept outside the
 *     lane stream, so that every in-stream code is at most 12 bits.)
 *     filler (row >= N or col >= K): the rank-0 code with sign 0, i.e. two zero
 *     bits, and no mantissa.
 *   Lane stream of block (rb, cb), lane l: elements t = 8c + r, c = 0..15,
 *     r = 0..7, at row 8rb + r, column 512cb + 16l + c (READING: column-outer
 *     order). Bits fill u32 words most significant bit first (stream bit i is bit
 *     31 - i%32 of word i/32); the last word is zero padded.
 *   Lane mantissa region: the mantissas of the lane's REAL elements with even t
 *     form the even half-stream, those with odd t the odd half-stream, each in
 *     increasing t. Field j of a half-stream (F = 7 or 3 bits) occupies half-stream
 *     bits [F*j, F*j + F), least significant bit first; half-stream bit i is bit
 *     i%16 of half-word i/16. Word k of the region = even half-word k |
 *     (odd half-word k << 16). Word count = ceil(max(F*n_even, F*n_odd) / 16)
 *     rounded up to a multiple of 4. (READING: bit packed, so that the raw plane
 *     costs F bits per element; even/odd halves so that the two mantissas of a row
 *     pair sit 16 bits apart.)
 *   Mantissa regions of a block: when all 32 lanes have the same word count W, word k of
 *     lane l is word 32k + l of the block's mantissa section (interleaved, so that the 32
 *     lanes reading their word k touch 32 consecutive words); otherwise the lanes' regions
 *     follow one another, lane 0 first. (READING: a layout choice with no size cost.)
 *   FP8 quantization of row n (READING of [P2]): a = max_k |w[n,k]| in FP32;
 *     s_n = a / 448 in FP32 (s_n = 1 when a = 0); q = e4m3 nearest to
 *     fp32(w) / s_n (FP32 division), ties to even, saturating at +-448.
 *
 *   Matrix-vector product (the plain definition): y_n = sum_k w[n,k] * x[k] with
 *   every product and the sum taken in FP64 (FP8: y_n = s_n * sum_k q[n,k] x[k]).
 *
 *   FP8 dequantization for prefill (READING of [P2]): BF16 nearest (ties to even) to the FP32
 *   product e4m3(q[n,k]) * s_n; NaN codes give 0x7FC0.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_MAGIC 0x3143574Eu
#define ORC_VERSION 3
#define ORC_R 11
#define ORC_ROWS 8
#define ORC_COLS 512
#define ORC_LANES 32
#define ORC_LANE_COLS 16
#define ORC_SYMS 128
#define ORC_MAX_LANE_WORDS 80 /* 128 codes * 20 bits / 32 */

enum { ORC_BF16 = 0, ORC_FP8 = 1 };

/* ------------------------------------------------------------------ helpers */

static uint64_t ceil_div(uint64_t a, uint64_t b) { return (a + b - 1) / b; }
static uint64_t pad16(uint64_t a) { return ceil_div(a, 16) * 16; }

static void put_u16(uint8_t *p, uint32_t v) { p[0] = v & 0xFF; p[1] = (v >> 8) & 0xFF; }
static void put_u32(uint8_t *p, uint32_t v) {
    for (int i = 0; i < 4; i++) p[i] = (v >> (8 * i)) & 0xFF;
}
static void put_u64(uint8_t *p, uint64_t v) {
    for (int i = 0; i < 8; i++) p[i] = (v >> (8 * i)) & 0xFF;
}
static uint32_t get_u32(const uint8_t *p) {
    uint32_t v = 0;
    for (int i = 0; i < 4; i++) v |= (uint32_t)p[i] << (8 * i);
    return v;
}
static uint64_t get_u64(const uint8_t *p) {
    uint64_t v = 0;
    for (int i = 0; i < 8; i++) v |= (uint64_t)p[i] << (8 * i);
    return v;
}

/* Fields of one element. */
static void split(int elem, uint32_t e, uint32_t *s, uint32_t *v, uint32_t *m) {
    if (elem == ORC_BF16) {
        *s = (e >> 15) & 1; *v = (e >> 7) & 0xFF; *m = e & 0x7F;
    } else {
        *s = (e >> 7) & 1; *v = (e >> 3) & 0xF; *m = e & 7;
    }
}
static uint32_t join(int elem, uint32_t s, uint32_t v, uint32_t m) {
    if (elem == ORC_BF16) return (s << 15) | (v << 7) | m;
    return (s << 7) | (v << 3) | m;
}
static int exp_bits(int elem) { return elem == ORC_BF16 ? 8 : 4; }
static int man_bits(int elem) { return elem == ORC_BF16 ? 7 : 3; }

/* Position of element t of lane l in block (rb, cb). */
static void position(uint64_t rb, uint64_t cb, int l, int t, uint64_t *row, uint64_t *col) {
    int c = t / ORC_ROWS, r = t % ORC_ROWS;
    *row = rb * ORC_ROWS + (uint64_t)r;
    *col = cb * ORC_COLS + (uint64_t)l * ORC_LANE_COLS + (uint64_t)c;
}

/* --------------------------------------------------------------- bit writer */
typedef struct { uint32_t w[ORC_MAX_LANE_WORDS]; int nbits; } bitw;

static void bw_put(bitw *b, uint32_t bit) {
    int word = b->nbits / 32, pos = 31 - b->nbits % 32;
    if (bit) b->w[word] |= 1u << pos;
    b->nbits++;
}

/* half-stream writer: bit i -> bit i%16 of half-word i/16 */
typedef struct { uint16_t h[ORC_SYMS]; int nbits; } halfw;

static void hw_put_field(halfw *h, uint32_t value, int width) {
    for (int i = 0; i < width; i++) {
        int bit = h->nbits + i;
        if ((value >> i) & 1) h->h[bit / 16] |= (uint16_t)(1u << (bit % 16));
    }
    h->nbits += width;
}

/* ------------------------------------------------------------------ ranking */
/* Ranks by (count desc, value asc) over values with count > 0, at most ORC_R. */
static int make_ranks(const uint64_t *count, int nvals, uint8_t *rank_exp, int *rank_of) {
    int chosen[256] = {0}, n = 0;
    for (int v = 0; v < nvals; v++) rank_of[v] = -1;
    while (n < ORC_R) {
        int best = -1;
        for (int v = 0; v < nvals; v++) {
            if (chosen[v] || count[v] == 0) continue;
            if (best < 0 || count[v] > count[best]) best = v; /* strict > keeps lowest v */
        }
        if (best < 0) break;
        chosen[best] = 1; rank_exp[n] = (uint8_t)best; rank_of[best] = n; n++;
    }
    return n;
}

/* ----------------------------------------------------------------- encoder */
/*
 * Encodes an N x K matrix of BF16 bit patterns (elem 0, e[] holds uint16) or fp8
 * bytes (elem 1, e[] holds the byte values, scale[] the N row scales). Returns a
 * malloc'd blob in *out and its size in *bytes; 0 on success.
 */
int orc_encode(const uint16_t *e, const float *scale, uint64_t N, uint64_t K, int elem,
               uint8_t **out, uint64_t *bytes) {
    if (N == 0 || K == 0 || (elem != ORC_BF16 && elem != ORC_FP8)) return -1;
    uint64_t RB = ceil_div(N, ORC_ROWS), CB = ceil_div(K, ORC_COLS), NB = RB * CB;
    int nvals = 1 << exp_bits(elem);
    uint64_t count[256] = {0};
    for (uint64_t i = 0; i < N * K; i++) {
        uint32_t s, v, m;
        split(elem, e[i], &s, &v, &m);
        count[v]++;
    }
    uint8_t rank_exp[16] = {0};
    int rank_of[256];
    int nr = make_ranks(count, nvals, rank_exp, rank_of);

    /* Pass 1 builds every block region in its own buffer. */
    uint8_t **reg = (uint8_t **)calloc(NB, sizeof(uint8_t *));
    uint64_t *reg_len = (uint64_t *)calloc(NB, sizeof(uint64_t));
    if (!reg || !reg_len) return -2;
    for (uint64_t b = 0; b < NB; b++) {
        uint64_t rb = b / CB, cb = b % CB;
        static bitw code[ORC_LANES];
        static halfw even[ORC_LANES], odd[ORC_LANES];
        static uint32_t esc[ORC_LANES * ORC_SYMS];
        uint64_t n_esc = 0;
        memset(code, 0, sizeof(code));
        memset(even, 0, sizeof(even));
        memset(odd, 0, sizeof(odd));
        int F = man_bits(elem);
        for (int l = 0; l < ORC_LANES; l++) {
            for (int t = 0; t < ORC_SYMS; t++) {
                uint64_t row, col;
                position(rb, cb, l, t, &row, &col);
                if (row >= N || col >= K) { /* filler: rank-0 code, sign 0 */
                    bw_put(&code[l], 0);
                    bw_put(&code[l], 0);
                    continue;
                }
                uint32_t s, v, m;
                split(elem, e[row * K + col], &s, &v, &m);
                int p = rank_of[v];
                if (p >= 0) {
                    for (int i = 0; i < p; i++) bw_put(&code[l], 1);
                    bw_put(&code[l], 0);
                } else {
                    for (int i = 0; i < nr; i++) bw_put(&code[l], 1);
                    esc[n_esc++] = (uint32_t)t | ((uint32_t)l << 7) | ((uint32_t)e[row * K + col] << 12);
                }
                bw_put(&code[l], s);
                if (t % 2 == 0) hw_put_field(&even[l], m, F);
                else hw_put_field(&odd[l], m, F);
            }
        }
        uint64_t code_words = 0, man_words[ORC_LANES];
        for (int l = 0; l < ORC_LANES; l++) {
            code_words += ceil_div((uint64_t)code[l].nbits, 32);
            uint64_t bits = (uint64_t)(even[l].nbits > odd[l].nbits ? even[l].nbits : odd[l].nbits);
            man_words[l] = ceil_div(ceil_div(bits, 16), 4) * 4;
        }
        uint64_t len = pad16(32 + 4 * code_words);
        for (int l = 0; l < ORC_LANES; l++) len += 4 * man_words[l];
        uint64_t esc_at = len;
        len += pad16(4 * n_esc);
        uint8_t *r = (uint8_t *)calloc(len, 1);
        if (!r) return -2;
        uint64_t pos = 32;
        for (int l = 0; l < ORC_LANES; l++) {
            uint64_t nw = ceil_div((uint64_t)code[l].nbits, 32);
            r[l] = (uint8_t)nw;
            for (uint64_t i = 0; i < nw; i++, pos += 4) put_u32(r + pos, code[l].w[i]);
        }
        pos = pad16(pos);
        int uniform = 1;
        for (int l = 1; l < ORC_LANES; l++) uniform &= man_words[l] == man_words[0];
        uint64_t man0 = pos;
        for (int l = 0; l < ORC_LANES; l++) {
            for (uint64_t k = 0; k < man_words[l]; k++, pos += 4) {
                uint64_t at = uniform ? man0 + 4 * (k * ORC_LANES + (uint64_t)l) : pos;
                put_u32(r + at, (uint32_t)even[l].h[k] | ((uint32_t)odd[l].h[k] << 16));
            }
        }
        for (uint64_t i = 0; esc_at + 4 * i < len; i++)
            put_u32(r + esc_at + 4 * i, i < n_esc ? esc[i] : 0xFFFFFFFFu);
        reg[b] = r;
        reg_len[b] = len;
    }

    /* Pass 2 lays out header, tables and data. */
    uint64_t off_blocks = 80;
    uint64_t off_scales = elem == ORC_FP8 ? pad16(off_blocks + 4 * (NB + 1)) : 0;
    uint64_t off_data = elem == ORC_FP8 ? pad16(off_scales + 4 * N) : pad16(off_blocks + 4 * (NB + 1));
    uint64_t data_len = 0;
    for (uint64_t b = 0; b < NB; b++) data_len += reg_len[b];
    uint64_t total = off_data + data_len;
    uint8_t *blob = (uint8_t *)calloc(total, 1);
    if (!blob) return -2;
    put_u32(blob + 0, ORC_MAGIC);
    put_u16(blob + 4, ORC_VERSION);
    blob[6] = (uint8_t)elem;
    blob[7] = (uint8_t)nr;
    put_u64(blob + 8, N);
    put_u64(blob + 16, K);
    put_u64(blob + 24, NB);
    put_u64(blob + 32, off_blocks);
    put_u64(blob + 40, off_scales);
    put_u64(blob + 48, off_data);
    put_u64(blob + 56, total);
    memcpy(blob + 64, rank_exp, 16);
    uint64_t acc = 0;
    for (uint64_t b = 0; b < NB; b++) {
        put_u32(blob + off_blocks + 4 * b, (uint32_t)(acc / 16));
        memcpy(blob + off_data + acc, reg[b], reg_len[b]);
        acc += reg_len[b];
        free(reg[b]);
    }
    put_u32(blob + off_blocks + 4 * NB, (uint32_t)(acc / 16));
    if (elem == ORC_FP8)
        for (uint64_t n = 0; n < N; n++) memcpy(blob + off_scales + 4 * n, &scale[n], 4);
    free(reg);
    free(reg_len);
    *out = blob;
    *bytes = total;
    return 0;
}

void orc_free(void *p) { free(p); }

/* ----------------------------------------------------------------- decoder */
typedef struct {
    int elem, nr;
    uint64_t N, K, NB, RB, CB, off_blocks, off_scales, off_data, total;
    uint8_t rank_exp[16];
} orc_hdr;

static int parse(const uint8_t *blob, uint64_t bytes, orc_hdr *h) {
    if (bytes < 80 || get_u32(blob) != ORC_MAGIC || blob[4] != ORC_VERSION || blob[5] != 0) return -1;
    h->elem = blob[6];
    h->nr = blob[7];
    h->N = get_u64(blob + 8);
    h->K = get_u64(blob + 16);
    h->NB = get_u64(blob + 24);
    h->off_blocks = get_u64(blob + 32);
    h->off_scales = get_u64(blob + 40);
    h->off_data = get_u64(blob + 48);
    h->total = get_u64(blob + 56);
    if (h->elem > 1 || h->nr < 1 || h->nr > ORC_R || h->N == 0 || h->K == 0) return -1;
    h->RB = ceil_div(h->N, ORC_ROWS);
    h->CB = ceil_div(h->K, ORC_COLS);
    if (h->NB != h->RB * h->CB || h->total != bytes) return -1;
    if (h->off_blocks + 4 * (h->NB + 1) > bytes || h->off_data > bytes) return -1;
    memcpy(h->rank_exp, blob + 64, 16);
    return 0;
}

/* bit reader over one lane stream */
typedef struct { const uint8_t *p; uint64_t nwords; uint64_t pos; int bad; } bitr;

static uint32_t br_get(bitr *b) {
    uint64_t word = b->pos / 32;
    int bitpos = 31 - (int)(b->pos % 32);
    b->pos++;
    if (word >= b->nwords) { b->bad = 1; return 0; }
    return (get_u32(b->p + 4 * word) >> bitpos) & 1;
}

/* field j of a lane's even (odd = 0) or odd half-stream; the lane's word k is at
   region + 4 * k * stride */
static uint32_t half_field(const uint8_t *region, uint64_t stride, int odd, uint64_t j, int F) {
    uint32_t v = 0;
    for (int i = 0; i < F; i++) {
        uint64_t bit = (uint64_t)F * j + (uint64_t)i;
        uint32_t word = get_u32(region + 4 * (bit / 16) * stride);
        uint32_t half = odd ? (word >> 16) : (word & 0xFFFF);
        v |= ((half >> (bit % 16)) & 1u) << i;
    }
    return v;
}

/*
 * Decodes block b into tile[r][c] (8 x 512 element values; fillers left 0).
 * Returns 0, or -1 if a stream or region is malformed.
 */
static int decode_block(const uint8_t *blob, const orc_hdr *h, uint64_t b, uint16_t tile[ORC_ROWS][ORC_COLS]) {
    uint64_t rb = b / h->CB, cb = b % h->CB;
    uint64_t start = h->off_data + 16 * (uint64_t)get_u32(blob + h->off_blocks + 4 * b);
    uint64_t end = h->off_data + 16 * (uint64_t)get_u32(blob + h->off_blocks + 4 * (b + 1));
    if (end > h->total || start + 32 > end) return -1;
    const uint8_t *reg = blob + start;
    uint64_t pos = 32;
    const uint8_t *lane_code[ORC_LANES];
    for (int l = 0; l < ORC_LANES; l++) {
        lane_code[l] = reg + pos;
        pos += 4 * (uint64_t)reg[l];
    }
    pos = pad16(pos);
    int F = man_bits(h->elem);
    int ok = 0;
    /* the mantissa regions' sizes follow from the real extents; the escape list follows them */
    uint64_t man_at = pos, esc_at = pos, mwords[ORC_LANES];
    for (int l = 0; l < ORC_LANES; l++) {
        uint64_t n_even = 0, n_odd = 0;
        for (int t = 0; t < ORC_SYMS; t++) {
            uint64_t row, col;
            position(rb, cb, l, t, &row, &col);
            if (row < h->N && col < h->K) { if (t % 2 == 0) n_even++; else n_odd++; }
        }
        uint64_t bits = (uint64_t)F * (n_even > n_odd ? n_even : n_odd);
        mwords[l] = ceil_div(ceil_div(bits, 16), 4) * 4;
        esc_at += 4 * mwords[l];
    }
    int uniform = 1;
    for (int l = 1; l < ORC_LANES; l++) uniform &= mwords[l] == mwords[0];
    if (start + esc_at > end) return -1;
    static uint32_t esc_value[ORC_LANES][ORC_SYMS];
    static int esc_seen[ORC_LANES][ORC_SYMS];
    memset(esc_seen, 0, sizeof(esc_seen));
    for (uint64_t at = esc_at; start + at + 4 <= end; at += 4) {
        uint32_t ent = get_u32(reg + at);
        if (ent == 0xFFFFFFFFu) continue;
        int t = (int)(ent & 127u), l = (int)((ent >> 7) & 31u);
        esc_value[l][t] = ent >> 12;
        esc_seen[l][t] = 1;
    }
    pos = man_at;
    for (int l = 0; l < ORC_LANES; l++) {
        bitr br = {lane_code[l], reg[l], 0, 0};
        uint32_t sv[ORC_SYMS], vv[ORC_SYMS];
        int real[ORC_SYMS], escaped[ORC_SYMS];
        uint64_t n_even = 0, n_odd = 0;
        for (int t = 0; t < ORC_SYMS; t++) {
            uint64_t row, col;
            position(rb, cb, l, t, &row, &col);
            real[t] = row < h->N && col < h->K;
            int ones = 0;
            while (ones < h->nr && br_get(&br) == 1) ones++;
            escaped[t] = ones >= h->nr;
            vv[t] = escaped[t] ? 0 : h->rank_exp[ones];
            sv[t] = br_get(&br);
            if (real[t]) { if (t % 2 == 0) n_even++; else n_odd++; }
        }
        if (br.bad) ok = -1;
        uint64_t bits = (uint64_t)F * (n_even > n_odd ? n_even : n_odd);
        uint64_t words = ceil_div(ceil_div(bits, 16), 4) * 4;
        const uint8_t *man = uniform ? reg + man_at + 4 * (uint64_t)l : reg + pos;
        uint64_t stride = uniform ? ORC_LANES : 1;
        uint64_t je = 0, jo = 0;
        for (int t = 0; t < ORC_SYMS; t++) {
            if (!real[t]) continue;
            uint32_t m = (t % 2 == 0) ? half_field(man, stride, 0, je++, F) : half_field(man, stride, 1, jo++, F);
            uint32_t value = join(h->elem, sv[t], vv[t], m);
            if (escaped[t]) {
                if (!esc_seen[l][t]) return -1;
                value = esc_value[l][t];
            }
            tile[t % ORC_ROWS][l * ORC_LANE_COLS + t / ORC_ROWS] = (uint16_t)value;
        }
        pos += 4 * words;
    }
    return ok;
}

/* Header facts for the Python side: out[0..5] = elem, n_ranked, N, K, n_blocks, total. */
int orc_info(const uint8_t *blob, uint64_t bytes, uint64_t *out, uint8_t *rank_exp) {
    orc_hdr h;
    if (parse(blob, bytes, &h)) return -1;
    out[0] = (uint64_t)h.elem; out[1] = (uint64_t)h.nr; out[2] = h.N; out[3] = h.K;
    out[4] = h.NB; out[5] = h.total;
    memcpy(rank_exp, h.rank_exp, 16);
    return 0;
}

/* Decodes the whole matrix into e[N*K] (BF16 bits or fp8 bytes widened to uint16)
 * and, for fp8, the scales into scale[N]. */
int orc_decode(const uint8_t *blob, uint64_t bytes, uint16_t *e, float *scale) {
    orc_hdr h;
    if (parse(blob, bytes, &h)) return -1;
    static uint16_t tile[ORC_ROWS][ORC_COLS];
    for (uint64_t b = 0; b < h.NB; b++) {
        memset(tile, 0, sizeof(tile));
        if (decode_block(blob, &h, b, tile)) return -1;
        uint64_t rb = b / h.CB, cb = b % h.CB;
        for (int r = 0; r < ORC_ROWS; r++) {
            uint64_t row = rb * ORC_ROWS + (uint64_t)r;
            if (row >= h.N) continue;
            for (int c = 0; c < ORC_COLS; c++) {
                uint64_t col = cb * ORC_COLS + (uint64_t)c;
                if (col < h.K) e[row * h.K + col] = tile[r][c];
            }
        }
    }
    if (h.elem == ORC_FP8 && scale)
        for (uint64_t n = 0; n < h.N; n++) memcpy(&scale[n], blob + h.off_scales + 4 * n, 4);
    return 0;
}

/* ------------------------------------------------------------- arithmetic */
static double bf16_value(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* OCP fp8 e4m3: bias 7, no infinities, S.1111.111 is NaN. */
static double e4m3_value(uint8_t q) {
    int s = q >> 7, e = (q >> 3) & 0xF, m = q & 7;
    double mag;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) mag = ldexp((double)m / 8.0, -6);
    else mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* Value of an element of the given kind. */
static double elem_value(int elem, uint16_t e) {
    return elem == ORC_BF16 ? bf16_value(e) : e4m3_value((uint8_t)e);
}

/* Nearest e4m3 to a finite float, ties to even, saturating at +-448: a search
 * over every finite non-negative code. */
uint8_t orc_e4m3_from_f32(float x) {
    double ax = fabs((double)x);
    int best = 0;
    double best_err = INFINITY;
    for (int c = 0; c <= 126; c++) {
        double err = fabs(ax - e4m3_value((uint8_t)c));
        if (err < best_err || (err == best_err && (c & 1) == 0)) { best = c; best_err = err; }
    }
    return (uint8_t)(best | (signbit(x) ? 0x80 : 0));
}

/* Per-row symmetric quantization of BF16 weights to e4m3 with scale absmax/448.
 * Returns -1 if any weight is not finite. */
int orc_quantize_fp8(const uint16_t *w, uint64_t N, uint64_t K, uint8_t *q, float *scale) {
    for (uint64_t n = 0; n < N; n++) {
        float a = 0.0f;
        for (uint64_t k = 0; k < K; k++) {
            float f = (float)bf16_value(w[n * K + k]);
            if (!isfinite(f)) return -1;
            if (fabsf(f) > a) a = fabsf(f);
        }
        float s = a == 0.0f ? 1.0f : a / 448.0f;
        scale[n] = s;
        for (uint64_t k = 0; k < K; k++) {
            float f = (float)bf16_value(w[n * K + k]);
            q[n * K + k] = orc_e4m3_from_f32(f / s);
        }
    }
    return 0;
}

/* BF16 nearest to a float, ties to even; every NaN gives the quiet NaN 0x7FC0. */
static uint16_t bf16_nearest(float f) {
    if (isnan(f)) return 0x7FC0;
    uint32_t u;
    memcpy(&u, &f, 4);
    uint32_t low = u & 0xFFFFu, high = u >> 16;
    if (low > 0x8000u || (low == 0x8000u && (high & 1u))) high += 1; /* carries into the exponent */
    return (uint16_t)high;
}

/* Dequantization of fp8 rows to BF16 for prefill (READING of [P2], whose prefill turns the
 * weights back into BF16 for a BF16 GEMM):
 * out[n,k] = the BF16 nearest (ties to even) to the FP32 product of the e4m3 value (exact in
 * FP32) and s_n; a NaN code gives 0x7FC0. */
void orc_dequantize_fp8(const uint8_t *q, const float *scale, uint64_t N, uint64_t K, uint16_t *out) {
    for (uint64_t n = 0; n < N; n++)
        for (uint64_t k = 0; k < K; k++) {
            float v = (float)e4m3_value(q[n * K + k]);
            float p = v * scale[n];
            out[n * K + k] = bf16_nearest(p);
        }
}

/* y[i] = sum_k value(W[rows[i], k]) * x[k] in FP64 (times s_n for fp8), for the
 * listed rows (all rows when rows == NULL, n_rows == N). Decodes only the
 * row-blocks it needs. */
int orc_gemv_rows(const uint8_t *blob, uint64_t bytes, const uint16_t *x, const int64_t *rows,
                  uint64_t n_rows, double *y) {
    orc_hdr h;
    if (parse(blob, bytes, &h)) return -1;
    uint16_t *rowbuf = (uint16_t *)malloc(sizeof(uint16_t) * ORC_ROWS * h.K);
    if (!rowbuf) return -2;
    static uint16_t tile[ORC_ROWS][ORC_COLS];
    uint64_t have_rb = UINT64_MAX;
    for (uint64_t i = 0; i < n_rows; i++) {
        uint64_t row = rows ? (uint64_t)rows[i] : i;
        if (row >= h.N) { free(rowbuf); return -1; }
        uint64_t rb = row / ORC_ROWS;
        if (rb != have_rb) {
            for (uint64_t cb = 0; cb < h.CB; cb++) {
                memset(tile, 0, sizeof(tile));
                if (decode_block(blob, &h, rb * h.CB + cb, tile)) { free(rowbuf); return -1; }
                for (int r = 0; r < ORC_ROWS; r++)
                    for (int c = 0; c < ORC_COLS; c++) {
                        uint64_t col = cb * ORC_COLS + (uint64_t)c;
                        if (col < h.K) rowbuf[(uint64_t)r * h.K + col] = tile[r][c];
                    }
            }
            have_rb = rb;
        }
        double acc = 0.0;
        const uint16_t *wr = rowbuf + (row % ORC_ROWS) * h.K;
        for (uint64_t k = 0; k < h.K; k++) acc += elem_value(h.elem, wr[k]) * bf16_value(x[k]);
        if (h.elem == ORC_FP8) {
            float s;
            memcpy(&s, blob + h.off_scales + 4 * row, 4);
            acc *= (double)s;
        }
        y[i] = acc;
    }
    free(rowbuf);
    return 0;
}

/* FP64 sum of |w x| per listed row: the scale of the matrix-vector tolerance. */
int orc_abs_dot_rows(const uint8_t *blob, uint64_t bytes, const uint16_t *x, const int64_t *rows,
                     uint64_t n_rows, double *out) {
    orc_hdr h;
    if (parse(blob, bytes, &h)) return -1;
    uint16_t *xa = (uint16_t *)malloc(sizeof(uint16_t) * h.K);
    if (!xa) return -2;
    for (uint64_t k = 0; k < h.K; k++) xa[k] = x[k] & 0x7FFF; /* |x| */
    /* |w x| = |w| |x|: decode, take |value| per element. */
    uint16_t *rowbuf = (uint16_t *)malloc(sizeof(uint16_t) * ORC_ROWS * h.K);
    if (!rowbuf) { free(xa); return -2; }
    static uint16_t tile[ORC_ROWS][ORC_COLS];
    uint64_t have_rb = UINT64_MAX;
    for (uint64_t i = 0; i < n_rows; i++) {
        uint64_t row = rows ? (uint64_t)rows[i] : i;
        if (row >= h.N) { free(xa); free(rowbuf); return -1; }
        uint64_t rb = row / ORC_ROWS;
        if (rb != have_rb) {
            for (uint64_t cb = 0; cb < h.CB; cb++) {
                memset(tile, 0, sizeof(tile));
                if (decode_block(blob, &h, rb * h.CB + cb, tile)) { free(xa); free(rowbuf); return -1; }
                for (int r = 0; r < ORC_ROWS; r++)
                    for (int c = 0; c < ORC_COLS; c++) {
                        uint64_t col = cb * ORC_COLS + (uint64_t)c;
                        if (col < h.K) rowbuf[(uint64_t)r * h.K + col] = tile[r][c];
                    }
            }
            have_rb = rb;
        }
        double acc = 0.0;
        const uint16_t *wr = rowbuf + (row % ORC_ROWS) * h.K;
        for (uint64_t k = 0; k < h.K; k++) acc += fabs(elem_value(h.elem, wr[k])) * bf16_value(xa[k]);
        if (h.elem == ORC_FP8) {
            float s;
            memcpy(&s, blob + h.off_scales + 4 * row, 4);
            acc *= fabs((double)s);
        }
        out[i] = acc;
    }
    free(xa);
    free(rowbuf);
    return 0;
}
