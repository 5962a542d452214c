/*
 * oracle.c -- plain, slow CPU reference for the NWC entropy-coded matrix format.
 *
 * TEST INFRASTRUCTURE ONLY. The product library never links, loads or calls this
 * file; only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline legs use it.
 * It shares no code with the library (decode_gemv_nwc_gb300/csrc): both are written
 * independently from the format definition below.
 *
 * Sources (the pages this restates; reading choices are marked READING):
 *   [P1] "NWC -- Neural Weight Compression" (PyPI project page, v0.9.0),
 *        section "How it works":
 *          - byte planes: the mantissa is stored raw, the exponent is entropy coded;
 *          - prefix code: exponent ranked by frequency, written as a unary rank code
 *            plus a raw sign bit, escape for rare values;
 *          - a 12-bit peek into a shared-memory table yields up to two complete codes;
 *          - fused kernel: each lane decodes its own bit stream for a block of
 *            8 rows x 512 columns (16 columns x 8 rows per lane); any shape works,
 *            padding costs a short code per filler weight and no mantissa.
 *   [P2] "Qwen3-4B-NWC-fp8" (model card): weight-only fp8 e4m3 with a symmetric
 *        per-output-channel scale; the fp8 bytes are coded losslessly.
 *
 * FORMAT, version 4 (little-endian):
 *   header, 64 bytes
 *     0  u32 magic 0x3143574E ("NWC1")      4  u16 version = 4
 *     6  u8  elem (0 = BF16, 1 = FP8 e4m3)  7  u8  n_ranked R (1..12)
 *     8  u64 N    16 u64 K    24 u64 n_blocks = ceil(N/8) * ceil(K/512)
 *     32 u64 off_blocks   40 u64 off_scales (0 for BF16)   48 u64 off_data
 *     56 u64 total_bytes
 *   64: u8 rank_exp[16]  -- exponent field value of rank 0..R-1, rest zero
 *   off_blocks: u32 tab[n_blocks + 1]; block b occupies bytes
 *        [off_data + 16*tab[b], off_data + 16*tab[b+1]); padded to 16 bytes
 *   off_scales (FP8 only): f32 scale[N]; padded to 16 bytes
 *   off_data: block regions, row-block-major (b = rb * CB + cb)
 *   block region: u8 lane_words[32]; the 32 lane code streams (lane 0 first), each
 *     a whole number of u32 words; zero padding to 16 bytes; the raw section; the
 *     escape list (u32 entries, padded to 16 bytes with 0xFFFFFFFF).
 *
 *   Fields of one element (READING: the sign is a raw bit and is stored beside the
 *   raw mantissa, so the raw plane is a whole byte per BF16 element and the coded
 *   stream holds only the exponent's rank code):
 *       BF16 b: s = b>>15, v = (b>>7)&0xFF, m = b&0x7F, raw byte   = s<<7 | m
 *       FP8  q: s = q>>7,  v = (q>>3)&0xF,  m = q&7,    raw nibble = s<<3 | m
 *   Ranking: histogram of v over the N*K real elements; ranks by (count desc,
 *     v asc) over values with count > 0; R = min(12, #distinct values).
 *     (READING: tie-break by ascending value.)
 *   Code of one symbol: ranked v (rank p < R): p one-bits then a zero-bit (p + 1
 *     bits); unranked v (escape): R one-bits; filler (row >= N or col >= K): the
 *     rank-0 code, one zero-bit. (READING: an escape for rare exponents whose raw
 *     exponent sits in the block's escape list, outside the stream.)
 *   Lane stream of block (rb, cb), lane l: symbols t = 8c + r, c = 0..15, r = 0..7,
 *     at row 8rb + r, column 512cb + 16l + c, taken in pairs j = 0..63 of symbols
 *     (2j, 2j+1) (rows 2i, 2i+1 of column c = j/4, i = j%4). A pair with codes of
 *     lengths La, Lb is written as both codes when La + Lb <= 13; otherwise as the
 *     first code followed by 13 - La one-bits, and the second symbol's exponent goes
 *     to the escape list (READING: the pages' peek yields up to two codes; here a
 *     13-bit peek always holds one pair, and a pair too long for it is cut).
 *     Bits fill u32 words most significant bit first (stream bit i is bit
 *     31 - i%32 of word i/32); the last word is zero padded.
 *   Escape list: one u32 per listed element, t | lane << 7 | v << 12, lanes in order
 *     and t increasing within a lane. Listed are the real elements whose exponent is
 *     unranked, the real second elements of cut pairs, and (FP8 only) the real
 *     elements with v = 0 and m != 0 (subnormals) or v = 15 and m = 7 (NaN).
 *     (READING: the FP8 exceptions are listed so that every other e4m3 value is a
 *     BF16 bit pattern with exponent field v + 120.)
 *   Raw section: a block whose 512 columns are all < K is "full": BF16 4096 bytes,
 *     the byte of row r, column c of lane l at 16*(32*(c/2) + l) + 8*(c%2) + r;
 *     FP8 2048 bytes, the byte holding rows 2i (low nibble) and 2i+1 (high nibble) of
 *     column c of lane l at 16*(32*(c/4) + l) + 4*(c%4) + i. Any other block: the
 *     lanes' regions follow one another (lane 0 first), lane l's region holding its
 *     real columns in order (8 bytes, resp. 4 bytes, per column as above) and zero
 *     padding to 16 bytes. Rows >= N of a real column hold zero.
 *     (READING: the filler rows of the last row block keep a zero raw byte, so that
 *     every real column has the same raw layout; fillers past K have none.)
 *   FP8 quantization of row n (READING of [P2]): a = max_k |w[n,k]| in FP32;
 *     s_n = a / 448 in FP32 (s_n = 1 when a = 0); q = e4m3 nearest to
 *     fp32(w) / s_n (FP32 division), ties to even, saturating at +-448.
 *
 *   Decoding a pair from the stream: count one-bits up to R: R of them is an escape,
 *   fewer end at a zero-bit (rank = the count). The second code is read the same way
 *   but if the first code took La bits and 13 - La < R one-bits follow with no zero
 *   among them, the pair was cut: those bits are its tail and the second symbol is
 *   listed. A listed element takes its exponent from the list, any other real element
 *   the ranked exponent of its code.
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
#define ORC_VERSION 4
#define ORC_R 12
#define ORC_PEEK 13
#define ORC_ROWS 8
#define ORC_COLS 512
#define ORC_LANES 32
#define ORC_LANE_COLS 16
#define ORC_SYMS 128
#define ORC_MAX_LANE_WORDS 26 /* 64 pairs * 13 bits / 32, rounded up */

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

/* The raw bits of an element: BF16 a byte s<<7 | m, FP8 a nibble s<<3 | m. */
static uint32_t raw_of(int elem, uint32_t s, uint32_t m) { return elem == ORC_BF16 ? (s << 7) | m : (s << 3) | m; }

/* FP8 values that the format always lists: subnormals and NaN. */
static int fp8_special(uint32_t v, uint32_t m) { return (v == 0 && m != 0) || (v == 15 && m == 7); }

/* Position of element t of lane l in block (rb, cb). */
static void position(uint64_t rb, uint64_t cb, int l, int t, uint64_t *row, uint64_t *col) {
    int c = t / ORC_ROWS, r = t % ORC_ROWS;
    *row = rb * ORC_ROWS + (uint64_t)r;
    *col = cb * ORC_COLS + (uint64_t)l * ORC_LANE_COLS + (uint64_t)c;
}

/* Real columns of lane l in column block cb. */
static int lane_cols(uint64_t K, uint64_t cb, int l) {
    uint64_t c0 = cb * ORC_COLS + (uint64_t)l * ORC_LANE_COLS;
    if (c0 >= K) return 0;
    return K - c0 >= ORC_LANE_COLS ? ORC_LANE_COLS : (int)(K - c0);
}

/* Bytes of raw data per column: 8 rows of a byte (BF16) or of a nibble (FP8). */
static int col_bytes(int elem) { return elem == ORC_BF16 ? 8 : 4; }

/* Offset of the raw bits of row r, column c of lane l inside the raw section, and the
 * nibble (0 low, 1 high; always 0 for BF16). `full` selects the full-block layout;
 * otherwise lane_off is the start of lane l's region. */
static uint64_t raw_at(int elem, int full, int l, int c, int r, uint64_t lane_off, int *nib) {
    if (elem == ORC_BF16) {
        *nib = 0;
        if (full) return 16 * (uint64_t)(32 * (c / 2) + l) + 8 * (uint64_t)(c % 2) + (uint64_t)r;
        return lane_off + 8 * (uint64_t)c + (uint64_t)r;
    }
    *nib = r % 2;
    if (full) return 16 * (uint64_t)(32 * (c / 4) + l) + 4 * (uint64_t)(c % 4) + (uint64_t)(r / 2);
    return lane_off + 4 * (uint64_t)c + (uint64_t)(r / 2);
}

/* Size of a block's raw section; lane_off[l] receives each lane's region start
 * (ragged layout). */
static uint64_t raw_section(int elem, uint64_t K, uint64_t cb, uint64_t lane_off[ORC_LANES], int *full) {
    *full = (cb + 1) * ORC_COLS <= K;
    if (*full) {
        for (int l = 0; l < ORC_LANES; l++) lane_off[l] = 0;
        return (uint64_t)ORC_LANES * ORC_LANE_COLS * (uint64_t)col_bytes(elem);
    }
    uint64_t at = 0;
    for (int l = 0; l < ORC_LANES; l++) {
        lane_off[l] = at;
        at += pad16((uint64_t)lane_cols(K, cb, l) * (uint64_t)col_bytes(elem));
    }
    return at;
}

/* --------------------------------------------------------------- bit writer */
typedef struct { uint32_t w[ORC_MAX_LANE_WORDS]; int nbits; } bitw;

static void bw_put(bitw *b, uint32_t bit) {
    int word = b->nbits / 32, pos = 31 - b->nbits % 32;
    if (bit) b->w[word] |= 1u << pos;
    b->nbits++;
}
static void bw_ones(bitw *b, int n) {
    for (int i = 0; i < n; i++) bw_put(b, 1);
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
/* Code of one symbol: *len bits, most significant first in *code. */
static void symbol_code(int nr, int rank, uint32_t *code, int *len) {
    if (rank < 0) { *code = (1u << nr) - 1u; *len = nr; return; }      /* escape */
    *code = ((1u << rank) - 1u) << 1; *len = rank + 1;                  /* rank ones, a zero */
}
static void put_code(bitw *b, uint32_t code, int len) {
    for (int i = len - 1; i >= 0; i--) bw_put(b, (code >> i) & 1);
}

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
        static uint32_t esc[ORC_LANES * ORC_SYMS];
        uint64_t n_esc = 0;
        memset(code, 0, sizeof(code));
        for (int l = 0; l < ORC_LANES; l++) {
            int listed[ORC_SYMS] = {0};
            uint32_t vals[ORC_SYMS] = {0};
            for (int j = 0; j < ORC_SYMS / 2; j++) {
                uint32_t c2[2];
                int len[2], real[2];
                for (int h = 0; h < 2; h++) {
                    int t = 2 * j + h;
                    uint64_t row, col;
                    position(rb, cb, l, t, &row, &col);
                    real[h] = row < N && col < K;
                    if (!real[h]) { symbol_code(nr, 0, &c2[h], &len[h]); continue; }
                    uint32_t s, v, m;
                    split(elem, e[row * K + col], &s, &v, &m);
                    vals[t] = v;
                    symbol_code(nr, rank_of[v], &c2[h], &len[h]);
                    if (rank_of[v] < 0) listed[t] = 1;
                    if (elem == ORC_FP8 && fp8_special(v, m)) listed[t] = 1;
                }
                put_code(&code[l], c2[0], len[0]);
                if (len[0] + len[1] <= ORC_PEEK) {
                    put_code(&code[l], c2[1], len[1]);
                } else {                      /* cut pair: the tail, the second symbol listed */
                    bw_ones(&code[l], ORC_PEEK - len[0]);
                    if (real[1]) listed[2 * j + 1] = 1;
                }
            }
            for (int t = 0; t < ORC_SYMS; t++)
                if (listed[t]) esc[n_esc++] = (uint32_t)t | ((uint32_t)l << 7) | (vals[t] << 12);
        }
        uint64_t code_words = 0;
        for (int l = 0; l < ORC_LANES; l++) code_words += ceil_div((uint64_t)code[l].nbits, 32);
        uint64_t lane_off[ORC_LANES];
        int full;
        uint64_t raw_len = raw_section(elem, K, cb, lane_off, &full);
        uint64_t raw0 = pad16(32 + 4 * code_words);
        uint64_t esc_at = raw0 + raw_len;
        uint64_t len = esc_at + pad16(4 * n_esc);
        uint8_t *r = (uint8_t *)calloc(len, 1);
        if (!r) return -2;
        uint64_t pos = 32;
        for (int l = 0; l < ORC_LANES; l++) {
            uint64_t nw = ceil_div((uint64_t)code[l].nbits, 32);
            r[l] = (uint8_t)nw;
            for (uint64_t i = 0; i < nw; i++, pos += 4) put_u32(r + pos, code[l].w[i]);
        }
        for (int l = 0; l < ORC_LANES; l++)
            for (int t = 0; t < ORC_SYMS; t++) {
                uint64_t row, col;
                position(rb, cb, l, t, &row, &col);
                if (col >= K) continue;                 /* no raw bits past K */
                uint32_t raw = 0;                       /* rows past N: zero */
                if (row < N) {
                    uint32_t s, v, m;
                    split(elem, e[row * K + col], &s, &v, &m);
                    raw = raw_of(elem, s, m);
                }
                int nib;
                uint64_t at = raw0 + raw_at(elem, full, l, t / ORC_ROWS, t % ORC_ROWS, lane_off[l], &nib);
                r[at] |= (uint8_t)(raw << (4 * nib));
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

/* One code: counts one-bits up to `limit`; returns the count and whether a zero-bit
 * ended it (*ended). */
static int read_ones(bitr *b, int limit, int *ended) {
    int ones = 0;
    *ended = 0;
    while (ones < limit) {
        if (br_get(b) == 0) { *ended = 1; return ones; }
        ones++;
    }
    return ones;
}

/*
 * Decodes block b into tile[r][c] (8 x 512 element values; fillers left 0).
 * Returns 0, or -1 if a stream, the raw section or the escape list is malformed.
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
    uint64_t raw0 = pad16(pos), lane_off[ORC_LANES];
    int full;
    uint64_t esc_at = raw0 + raw_section(h->elem, h->K, cb, lane_off, &full);
    if (start + esc_at > end) return -1;
    /* the escape list: entry per (lane, t) */
    static uint32_t esc_v[ORC_LANES][ORC_SYMS];
    static int esc_seen[ORC_LANES][ORC_SYMS];
    memset(esc_seen, 0, sizeof(esc_seen));
    for (uint64_t at = esc_at; start + at + 4 <= end; at += 4) {
        uint32_t ent = get_u32(reg + at);
        if (ent == 0xFFFFFFFFu) continue;
        int t = (int)(ent & 127u), l = (int)((ent >> 7) & 31u);
        if (esc_seen[l][t] || (ent >> 12) >> exp_bits(h->elem)) return -1;
        esc_v[l][t] = ent >> 12;
        esc_seen[l][t] = 1;
    }
    int ok = 0;
    for (int l = 0; l < ORC_LANES; l++) {
        bitr br = {lane_code[l], reg[l], 0, 0};
        for (int j = 0; j < ORC_SYMS / 2; j++) {
            int rank[2], ended;
            int a = read_ones(&br, h->nr, &ended);
            rank[0] = ended ? a : -1;                    /* -1: escape */
            int used = ended ? a + 1 : a;
            int room = ORC_PEEK - used;                  /* bits of the peek left */
            int lim = room < h->nr ? room : h->nr;
            int bcount = read_ones(&br, lim, &ended);
            if (ended) rank[1] = bcount;
            else rank[1] = -1;                           /* an escape, or the tail of a cut pair */
            for (int q = 0; q < 2; q++) {
                int t = 2 * j + q;
                uint64_t row, col;
                position(rb, cb, l, t, &row, &col);
                if (row >= h->N || col >= h->K) continue;
                uint32_t v;
                if (esc_seen[l][t]) v = esc_v[l][t];
                else if (rank[q] >= 0) v = h->rank_exp[rank[q]];
                else return -1;                          /* escaped but not listed */
                int nib;
                uint64_t at = raw0 + raw_at(h->elem, full, l, t / ORC_ROWS, t % ORC_ROWS, lane_off[l], &nib);
                uint32_t raw = (reg[at] >> (4 * nib)) & (h->elem == ORC_BF16 ? 0xFFu : 0xFu);
                uint32_t s = h->elem == ORC_BF16 ? raw >> 7 : raw >> 3;
                uint32_t m = h->elem == ORC_BF16 ? raw & 0x7F : raw & 7;
                tile[t % ORC_ROWS][l * ORC_LANE_COLS + t / ORC_ROWS] = (uint16_t)join(h->elem, s, v, m);
            }
        }
        if (br.bad) ok = -1;
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
