/*
 * ep_oracle.c -- plain, slow, single-threaded CPU oracle for MoE expert-parallel
 * Dispatch and Combine.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call this
 * file; only the tests, the smoke check and the benchmark's CPU-baseline leg do.  It shares
 * no code, header, table or helper with the CUDA implementation.
 *
 * What it computes (MORI-EP gfx1201 PR "feat(ep): add opt-in gfx1201 EP2/EP4 support",
 * section "How the gfx1201 kernels work", Dispatch and Combine bullets; MORI-EP guide,
 * section 3 "Operator API", dispatch(), combine(), get_dispatch_src_token_pos()):
 *
 *   Dispatch.  Every token t < n_tok[s] of source rank s names k experts idx[s][t][0..k).
 *   Expert e lives on rank floor(e / E) (contiguous blocks of E experts per rank; the pages
 *   only say "num_experts_per_rank").  The token gets ONE receive row on each DISTINCT
 *   destination rank (experts on the same rank share one hidden payload).  The row holds
 *   the token's whole hidden vector, its whole top-k index row, its FP32 weight row (if
 *   given) and its FP32 scale row (if scale_dim > 0).  Rows are handed out per destination
 *   rank in (source rank ascending, token ascending) order.  The reverse map entry of the
 *   row is src_rank * (W * M) + src_token (guide, get_dispatch_src_token_pos()).  Receive
 *   capacity per rank is W * M rows (each source sends at most one row per token).
 *
 *   Combine.  For each source token the rows it was sent to are read back, in ascending
 *   destination-rank order, converted to FP32, summed starting from +0.0f with plain float
 *   additions (no fused multiply-add; compiled with -ffp-contract=off), and the sum is
 *   rounded to nearest even into BF16 or FP16 (the Combine bullet: FP32 accumulation of the
 *   local and received contributions, one conversion at the end).  Optional FP32 weight
 *   rows are summed the same way, separately; routing weights are never applied to the
 *   payload (the Combine bullet leaves scaling expert outputs by routing weights to the
 *   caller).
 *
 *   Expert ids outside [0, W*E) route nowhere and make dispatch return EP_ORACLE_ERR_INDEX.
 *
 * Conversions are written from the IEEE 754 binary16 / bfloat16 definitions
 * (round to nearest, ties to even; overflow to infinity; NaN stays NaN).
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define EP_ORACLE_OK 0
#define EP_ORACLE_ERR_ARG (-1)
#define EP_ORACLE_ERR_INDEX (-6)

/* ---- IEEE conversions ------------------------------------------------------------- */

static uint32_t f32_bits(float f) { uint32_t b; memcpy(&b, &f, 4); return b; }
static float bits_f32(uint32_t b) { float f; memcpy(&f, &b, 4); return f; }

/* float -> bfloat16, round to nearest even.  bfloat16 is the top half of a binary32, so
 * rounding drops the low 16 bits: add half of the dropped range, plus one more when the
 * kept part is odd (ties go to the even neighbour), then truncate.  A carry out of the
 * mantissa correctly bumps the exponent; past the largest finite value it lands on Inf. */
uint16_t ep_oracle_bf16_from_f32(float f)
{
    uint32_t b = f32_bits(f);
    if ((b & 0x7FFFFFFFu) > 0x7F800000u)        /* NaN: keep sign, force a quiet NaN */
        return (uint16_t)(((b >> 16) & 0x8000u) | 0x7FC0u);
    uint32_t kept_lsb = (b >> 16) & 1u;
    b += 0x7FFFu + kept_lsb;
    return (uint16_t)(b >> 16);
}

float ep_oracle_f32_from_bf16(uint16_t h) { return bits_f32((uint32_t)h << 16); }

/* float -> binary16 (1 sign, 5 exponent bits with bias 15, 10 fraction bits), RNE. */
uint16_t ep_oracle_f16_from_f32(float f)
{
    uint32_t b = f32_bits(f);
    uint16_t sign = (uint16_t)((b >> 16) & 0x8000u);
    uint32_t a = b & 0x7FFFFFFFu;
    if (a > 0x7F800000u) return (uint16_t)(sign | 0x7E00u);     /* NaN */
    if (a >= 0x477FF000u) return (uint16_t)(sign | 0x7C00u);    /* >= 65520: rounds to Inf */
    if (a >= 0x38800000u) {                                     /* >= 2^-14: normal half */
        uint32_t exp = (a >> 23) - 127u + 15u;
        uint32_t h = (exp << 10) | ((a & 0x7FFFFFu) >> 13);
        uint32_t rem = a & 0x1FFFu;                             /* 13 dropped bits */
        if (rem > 0x1000u || (rem == 0x1000u && (h & 1u))) h += 1u;
        return (uint16_t)(sign | h);
    }
    /* subnormal half: value / 2^-24 rounded to an integer.  With the binary32 significand
     * m (implicit bit included) and biased exponent E, value = m * 2^(E - 150), so the
     * integer is m * 2^(E - 126), i.e. m shifted right by 126 - E. */
    uint32_t E = a >> 23;
    if (E < 102u) return sign;                                  /* below 2^-25: rounds to 0 */
    uint32_t m = (a & 0x7FFFFFu) | 0x800000u;
    uint32_t shift = 126u - E;                                  /* 14 .. 24 */
    uint32_t h = m >> shift;
    uint32_t rem = m & ((1u << shift) - 1u);
    uint32_t half = 1u << (shift - 1u);
    if (rem > half || (rem == half && (h & 1u))) h += 1u;       /* may carry into 0x400 */
    return (uint16_t)(sign | h);
}

/* binary16 -> float, exact. */
float ep_oracle_f32_from_f16(uint16_t h)
{
    uint32_t sign = ((uint32_t)h & 0x8000u) << 16;
    uint32_t exp = ((uint32_t)h >> 10) & 0x1Fu;
    uint32_t frac = (uint32_t)h & 0x3FFu;
    if (exp == 0x1Fu) return bits_f32(sign | 0x7F800000u | (frac << 13));
    if (exp == 0) {
        /* subnormal: frac * 2^-24, exact in binary32 */
        float v = (float)frac * bits_f32(0x33800000u);          /* 2^-24 */
        return sign ? -v : v;
    }
    return bits_f32(sign | ((exp - 15u + 127u) << 23) | (frac << 13));
}

/* float -> FP8 e4m3fn (OCP: 1 sign, 4 exponent bits with bias 7, 3 fraction bits; no
 * infinities; largest finite 448; all-ones exponent and fraction is NaN), round to nearest
 * even, saturating: magnitudes that round above 448 give 448. */
uint8_t ep_oracle_e4m3_from_f32(float f)
{
    uint32_t b = f32_bits(f);
    uint8_t sign = (uint8_t)((b >> 24) & 0x80u);
    uint32_t a = b & 0x7FFFFFFFu;
    if (a > 0x7F800000u) return (uint8_t)(sign | 0x7Fu);              /* NaN */
    if (a >= 0x43E00000u) return (uint8_t)(sign | 0x7Eu);             /* >= 448 (and Inf): 448 */
    if (a >= 0x3C800000u) {                                           /* >= 2^-6: normal e4m3 */
        uint32_t exp = (a >> 23) - 127u + 7u;
        uint32_t h = (exp << 3) | ((a & 0x7FFFFFu) >> 20);
        uint32_t rem = a & 0xFFFFFu;                                  /* 20 dropped bits */
        if (rem > 0x80000u || (rem == 0x80000u && (h & 1u))) h += 1u;
        if (h > 0x7Eu) h = 0x7Eu;                                     /* 464 > v > 448 rounds up: saturate */
        return (uint8_t)(sign | h);
    }
    /* subnormal e4m3: value / 2^-9 rounded to an integer = m * 2^(E - 150 + 9) with the binary32
     * significand m and biased exponent E, i.e. m shifted right by 141 - E */
    uint32_t E = a >> 23;
    if (E < 117u) return sign;                                        /* below 2^-10: rounds to 0 */
    uint32_t m = (a & 0x7FFFFFu) | 0x800000u;
    uint32_t shift = 141u - E;                                        /* 21 .. 24 */
    uint32_t h = m >> shift;
    uint32_t rem = m & ((1u << shift) - 1u);
    uint32_t half = 1u << (shift - 1u);
    if (rem > half || (rem == half && (h & 1u))) h += 1u;             /* may carry into 0x08 */
    return (uint8_t)(sign | h);
}

/* FP8 e4m3fn -> float, exact. */
float ep_oracle_f32_from_e4m3(uint8_t q)
{
    uint32_t sign = ((uint32_t)q & 0x80u) << 24;
    uint32_t exp = ((uint32_t)q >> 3) & 0xFu;
    uint32_t frac = (uint32_t)q & 0x7u;
    if (exp == 0xFu && frac == 0x7u) return bits_f32(sign | 0x7FC00000u);
    if (exp == 0) {
        float v = (float)frac * bits_f32(0x3B000000u);                /* frac * 2^-9 */
        return sign ? -v : v;
    }
    return bits_f32(sign | ((exp - 7u + 127u) << 23) | (frac << 20));
}

/*
 * Block-wise FP8 quantisation of BF16 rows (the FP8 wire of the MORI-EP tuning matrix, read as
 * one FP32 scale per 128-element block).  For every block of 128 elements of a row:
 *   amax  = max |x| (exact, in FP32)
 *   scale = amax / 448 (FP32 division, round to nearest even), or 1 when amax is 0
 *   q[i]  = e4m3 RNE saturating of (x[i] / scale) (FP32 division, round to nearest even)
 * x [rows][H] BF16 bits, q [rows][H], scales [rows][H/128]; H must be a multiple of 128.
 */
int ep_oracle_quantize_e4m3_blockwise(int64_t rows, int H, const uint16_t* x, uint8_t* q, float* scales)
{
    if (H < 128 || H % 128 != 0 || rows < 0) return EP_ORACLE_ERR_ARG;
    const int nb = H / 128;
    for (int64_t r = 0; r < rows; ++r) {
        for (int b = 0; b < nb; ++b) {
            const uint16_t* xb = x + r * H + b * 128;
            float amax = 0.0f;
            for (int i = 0; i < 128; ++i) {
                float v = ep_oracle_f32_from_bf16(xb[i]);
                float m = v < 0.0f ? -v : v;
                if (m > amax) amax = m;
            }
            float scale = amax > 0.0f ? amax / 448.0f : 1.0f;
            scales[r * nb + b] = scale;
            for (int i = 0; i < 128; ++i)
                q[r * H + b * 128 + i] = ep_oracle_e4m3_from_f32(ep_oracle_f32_from_bf16(xb[i]) / scale);
        }
    }
    return EP_ORACLE_OK;
}

void ep_oracle_e4m3_from_f32_array(const float* in, uint8_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = ep_oracle_e4m3_from_f32(in[i]);
}

void ep_oracle_f32_from_e4m3_array(const uint8_t* in, float* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = ep_oracle_f32_from_e4m3(in[i]);
}

void ep_oracle_bf16_from_f32_array(const float* in, uint16_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = ep_oracle_bf16_from_f32(in[i]);
}

void ep_oracle_f16_from_f32_array(const float* in, uint16_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = ep_oracle_f16_from_f32(in[i]);
}

void ep_oracle_f32_from_f16_array(const uint16_t* in, float* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = ep_oracle_f32_from_f16(in[i]);
}

/* ---- Dispatch ---------------------------------------------------------------------- */

/*
 * Arguments (all host pointers, row-major):
 *   x        [W][M][H] elements of elem_bytes bytes (raw bits)
 *   w        [W][M][k] float or NULL
 *   scales   [W][M][sd] float, NULL iff sd == 0
 *   idx      [W][M][k] int32
 *   n_tok    [W] tokens per source rank, each in 0..M
 * Outputs (caller-allocated):
 *   recv_x      [W][W*M][H]      recv_idx [W][W*M][k]      recv_w [W][W*M][k] (if w)
 *   recv_scales [W][W*M][sd] (if sd)
 *   src_pos     [W][W*M]         reverse map, src_rank * (W*M) + src_token
 *   slot_of     [W][M][W]        slot_of[s][t][r] = row of (s,t) on rank r, or -1
 *   recv_count  [W]
 */
int ep_oracle_dispatch(int W, int E, int k, int H, int elem_bytes, int sd, int M,
                       const void* x, const float* w, const float* scales, const int32_t* idx,
                       const int32_t* n_tok,
                       void* recv_x, int32_t* recv_idx, float* recv_w, float* recv_scales,
                       int32_t* src_pos, int32_t* slot_of, int32_t* recv_count)
{
    if (W < 1 || E < 1 || k < 1 || H < 1 || M < 1 || sd < 0) return EP_ORACLE_ERR_ARG;
    if (elem_bytes != 1 && elem_bytes != 2) return EP_ORACLE_ERR_ARG;
    const int64_t rows = (int64_t)W * M;                 /* receive rows per rank */
    const int64_t n_experts = (int64_t)W * E;
    const size_t row_bytes = (size_t)H * (size_t)elem_bytes;
    int64_t* cnt = (int64_t*)calloc((size_t)W, sizeof(int64_t));
    unsigned char* in_D = (unsigned char*)malloc((size_t)W);
    if (!cnt || !in_D) { free(cnt); free(in_D); return EP_ORACLE_ERR_ARG; }
    int status = EP_ORACLE_OK;

    for (int s = 0; s < W; ++s) {
        if (n_tok[s] < 0 || n_tok[s] > M) { status = EP_ORACLE_ERR_ARG; break; }
        for (int t = 0; t < n_tok[s]; ++t) {
            const int64_t tok = (int64_t)s * M + t;
            const int32_t* ids = idx + tok * k;
            /* D(s,t): the distinct destination ranks of the token's experts */
            memset(in_D, 0, (size_t)W);
            for (int j = 0; j < k; ++j) {
                int64_t e = ids[j];
                if (e < 0 || e >= n_experts) { status = EP_ORACLE_ERR_INDEX; continue; }
                in_D[e / E] = 1;
            }
            for (int r = 0; r < W; ++r) {
                slot_of[tok * W + r] = -1;
                if (!in_D[r]) continue;
                const int64_t slot = cnt[r]++;
                const int64_t row = (int64_t)r * rows + slot;
                memcpy((char*)recv_x + (size_t)row * row_bytes,
                       (const char*)x + (size_t)tok * row_bytes, row_bytes);
                memcpy(recv_idx + row * k, ids, (size_t)k * sizeof(int32_t));
                if (w) memcpy(recv_w + row * k, w + tok * k, (size_t)k * sizeof(float));
                if (sd > 0) memcpy(recv_scales + row * sd, scales + tok * sd, (size_t)sd * sizeof(float));
                src_pos[(int64_t)r * rows + slot] = (int32_t)((int64_t)s * rows + t);
                slot_of[tok * W + r] = (int32_t)slot;
            }
        }
    }
    for (int r = 0; r < W; ++r) recv_count[r] = (int32_t)cnt[r];
    free(cnt);
    free(in_D);
    return status;
}

/* ---- Combine ----------------------------------------------------------------------- */

/*
 *   expert_out [W][W*M][H] 16-bit elements (BF16 if out_fp16 == 0, FP16 otherwise)
 *   w_in       [W][W*M][k] float or NULL
 *   slot_of    [W][M][W] as written by ep_oracle_dispatch
 *   out        [W][M][H] 16-bit elements; rows t >= n_tok[s] are left untouched
 *   out_w      [W][M][k] float or NULL (written iff w_in and out_w are both given)
 */
int ep_oracle_combine(int W, int k, int H, int out_fp16, int M, const int32_t* n_tok,
                      const int32_t* slot_of, const uint16_t* expert_out, const float* w_in,
                      uint16_t* out, float* out_w)
{
    if (W < 1 || k < 1 || H < 1 || M < 1) return EP_ORACLE_ERR_ARG;
    const int64_t rows = (int64_t)W * M;
    float* acc = (float*)malloc((size_t)H * sizeof(float));
    float* accw = (float*)malloc((size_t)k * sizeof(float));
    if (!acc || !accw) { free(acc); free(accw); return EP_ORACLE_ERR_ARG; }
    for (int s = 0; s < W; ++s) {
        for (int t = 0; t < n_tok[s]; ++t) {
            const int64_t tok = (int64_t)s * M + t;
            for (int h = 0; h < H; ++h) acc[h] = 0.0f;
            for (int j = 0; j < k; ++j) accw[j] = 0.0f;
            for (int r = 0; r < W; ++r) {                 /* ascending destination rank */
                const int32_t slot = slot_of[tok * W + r];
                if (slot < 0) continue;
                const int64_t row = (int64_t)r * rows + slot;
                const uint16_t* src = expert_out + row * H;
                for (int h = 0; h < H; ++h) {
                    float v = out_fp16 ? ep_oracle_f32_from_f16(src[h]) : ep_oracle_f32_from_bf16(src[h]);
                    acc[h] = acc[h] + v;
                }
                if (w_in)
                    for (int j = 0; j < k; ++j) accw[j] = accw[j] + w_in[row * k + j];
            }
            uint16_t* dst = out + tok * H;
            for (int h = 0; h < H; ++h)
                dst[h] = out_fp16 ? ep_oracle_f16_from_f32(acc[h]) : ep_oracle_bf16_from_f32(acc[h]);
            if (w_in && out_w)
                for (int j = 0; j < k; ++j) out_w[tok * k + j] = accw[j];
        }
    }
    free(acc);
    free(accw);
    return EP_ORACLE_OK;
}

/* ---- Combine over an FP8 wire ------------------------------------------------------ */

/*
 * Combine of expert outputs sent as FP8 e4m3 codes with one FP32 scale per 128 elements (the
 * fp8_blockwise combine of the MORI-EP gfx1250 EPv2 pages).  For each source token and element
 * h: acc = +0.0f; for each destination rank r holding the token, ascending:
 *   v = float(q[r][row][h]) * scales[r][row][h / 128]     (one FP32 multiply, rounded)
 *   acc = acc + v                                         (one FP32 add, rounded)
 * out = BF16 RNE of acc.  Weights, when given, are summed exactly as in ep_oracle_combine.
 *   q [W][W*M][H] codes, scales [W][W*M][H/128], out [W][M][H] BF16 bits.
 */
int ep_oracle_combine_fp8(int W, int k, int H, int M, const int32_t* n_tok, const int32_t* slot_of,
                          const uint8_t* q, const float* scales, const float* w_in, uint16_t* out,
                          float* out_w)
{
    if (W < 1 || k < 1 || H < 128 || H % 128 != 0 || M < 1) return EP_ORACLE_ERR_ARG;
    const int64_t rows = (int64_t)W * M;
    const int nb = H / 128;
    float* acc = (float*)malloc((size_t)H * sizeof(float));
    float* accw = (float*)malloc((size_t)k * sizeof(float));
    if (!acc || !accw) { free(acc); free(accw); return EP_ORACLE_ERR_ARG; }
    for (int s = 0; s < W; ++s) {
        for (int t = 0; t < n_tok[s]; ++t) {
            const int64_t tok = (int64_t)s * M + t;
            for (int h = 0; h < H; ++h) acc[h] = 0.0f;
            for (int j = 0; j < k; ++j) accw[j] = 0.0f;
            for (int r = 0; r < W; ++r) {
                const int32_t slot = slot_of[tok * W + r];
                if (slot < 0) continue;
                const int64_t row = (int64_t)r * rows + slot;
                for (int h = 0; h < H; ++h) {
                    float v = ep_oracle_f32_from_e4m3(q[row * H + h]) * scales[row * nb + h / 128];
                    acc[h] = acc[h] + v;
                }
                if (w_in)
                    for (int j = 0; j < k; ++j) accw[j] = accw[j] + w_in[row * k + j];
            }
            for (int h = 0; h < H; ++h) out[tok * H + h] = ep_oracle_bf16_from_f32(acc[h]);
            if (w_in && out_w)
                for (int j = 0; j < k; ++j) out_w[tok * k + j] = accw[j];
        }
    }
    free(acc);
    free(accw);
    return EP_ORACLE_OK;
}


/* ---- Expert-grouped ("standard MoE") layout ---------------------------------------- */

/*
 * The dispatch output regrouped by local expert (MORI-EP guide, section 4 "Standard MoE
 * Compatibility", convert_dispatch_output(): packed_recv_x, packed_recv_count,
 * packed_recv_src_info, packed_recv_layout_range).  The guide names the outputs only; the
 * reading taken: on rank r, the list of local expert e (global id r*E + e) holds, in receive-row
 * order, every received row whose top-k names that expert (once per row, even if named twice);
 *   packed_x[r][e][slot]        the row's payload (cap = W*M slots per expert)
 *   packed_count[r][e]          length of the list
 *   packed_src_info[r][e][slot] the row's source token index within its source rank
 *   layout_range[r][e][s]       (first slot of source rank s) << 32 | (number of its slots);
 *                               rows arrive in source-rank order, so each source's slots are
 *                               contiguous and its first slot is the count of earlier sources
 *   packed_row[r][e][slot]      the receive row (kept for the inverse below)
 */
int ep_oracle_group_by_expert(int W, int E, int k, int H, int elem_bytes, int M, const void* recv_x,
                              const int32_t* recv_idx, const int32_t* recv_count,
                              const int32_t* src_pos, void* packed_x, int32_t* packed_count,
                              int32_t* packed_src_info, int64_t* layout_range, int32_t* packed_row)
{
    if (W < 1 || E < 1 || k < 1 || H < 1 || M < 1 || (elem_bytes != 1 && elem_bytes != 2))
        return EP_ORACLE_ERR_ARG;
    const int64_t rows = (int64_t)W * M;
    const size_t row_bytes = (size_t)H * (size_t)elem_bytes;
    int64_t* per_src = (int64_t*)malloc((size_t)W * sizeof(int64_t));
    if (!per_src) return EP_ORACLE_ERR_ARG;
    for (int r = 0; r < W; ++r) {
        for (int e = 0; e < E; ++e) {
            const int32_t ge = r * E + e;
            const int64_t list = (int64_t)r * E + e;
            int64_t cnt = 0;
            for (int s = 0; s < W; ++s) per_src[s] = 0;
            for (int64_t i = 0; i < recv_count[r]; ++i) {
                const int32_t* ids = recv_idx + ((int64_t)r * rows + i) * k;
                int named = 0;
                for (int j = 0; j < k; ++j) named |= ids[j] == ge;
                if (!named) continue;
                const int64_t slot = cnt++;
                memcpy((char*)packed_x + (size_t)(list * rows + slot) * row_bytes,
                       (const char*)recv_x + (size_t)((int64_t)r * rows + i) * row_bytes, row_bytes);
                const int32_t pos = src_pos[(int64_t)r * rows + i];
                packed_src_info[list * rows + slot] = (int32_t)(pos % rows);
                packed_row[list * rows + slot] = (int32_t)i;
                per_src[pos / rows] += 1;
            }
            packed_count[list] = (int32_t)cnt;
            int64_t first = 0;
            for (int s = 0; s < W; ++s) {
                layout_range[list * W + s] = (first << 32) | per_src[s];
                first += per_src[s];
            }
        }
    }
    free(per_src);
    return EP_ORACLE_OK;
}

/*
 * The inverse (guide, convert_combine_input()): the per-rank combine input of every received
 * row is the sum of its local experts' outputs, taken in ascending expert id, in FP32 from
 * +0.0f, rounded to nearest even into BF16 (out_fp16 == 0) or FP16.
 *   packed_y [W][E][W*M][H] 16-bit expert outputs, packed_row / packed_count as written above,
 *   out [W][W*M][H]; rows at or past recv_count[r] are left untouched.
 */
int ep_oracle_ungroup_by_expert(int W, int E, int H, int out_fp16, int M, const int32_t* recv_count,
                                const int32_t* packed_count, const int32_t* packed_row,
                                const uint16_t* packed_y, uint16_t* out)
{
    if (W < 1 || E < 1 || H < 1 || M < 1) return EP_ORACLE_ERR_ARG;
    const int64_t rows = (int64_t)W * M;
    for (int r = 0; r < W; ++r) {
        const int64_t n = recv_count[r];
        float* acc = (float*)calloc((size_t)(n > 0 ? n : 1) * (size_t)H, sizeof(float));
        if (!acc) return EP_ORACLE_ERR_ARG;
        for (int e = 0; e < E; ++e) {                  /* ascending expert id */
            const int64_t list = (int64_t)r * E + e;
            for (int64_t slot = 0; slot < packed_count[list]; ++slot) {
                const int64_t i = packed_row[list * rows + slot];
                const uint16_t* y = packed_y + (list * rows + slot) * H;
                for (int h = 0; h < H; ++h) {
                    float v = out_fp16 ? ep_oracle_f32_from_f16(y[h]) : ep_oracle_f32_from_bf16(y[h]);
                    acc[i * H + h] = acc[i * H + h] + v;
                }
            }
        }
        for (int64_t i = 0; i < n; ++i)
            for (int h = 0; h < H; ++h)
                out[((int64_t)r * rows + i) * H + h] =
                    out_fp16 ? ep_oracle_f16_from_f32(acc[i * H + h]) : ep_oracle_bf16_from_f32(acc[i * H + h]);
        free(acc);
    }
    return EP_ORACLE_OK;
}

/* ---- Combine over an FP4 (MX) wire -------------------------------------------------- */

/*
 * FP4 e2m1 (1 sign, 2 exponent bits with bias 1, 1 fraction bit): magnitudes 0, 0.5, 1, 1.5,
 * 2, 3, 4, 6.  Round to nearest; a tie goes to the code with a zero fraction bit (even);
 * magnitudes past 6 saturate to 6; NaN maps to 6 with its sign (the format has no NaN).
 * Written by comparing against the eight magnitudes, from the definition of the format.
 */
uint8_t ep_oracle_e2m1_from_f32(float f)
{
    static const float mag[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};
    uint32_t b = f32_bits(f);
    uint8_t sign = (uint8_t)((b >> 28) & 0x8u);
    float a = bits_f32(b & 0x7FFFFFFFu);
    if (!(a <= 6.0f)) return (uint8_t)(sign | 0x7u);            /* > 6, Inf, NaN */
    int best = 0;
    for (int c = 1; c < 8; ++c) {
        float dc = a - mag[c] < 0 ? mag[c] - a : a - mag[c];
        float db = a - mag[best] < 0 ? mag[best] - a : a - mag[best];
        if (dc < db || (dc == db && (c & 1) == 0)) best = c;
    }
    return (uint8_t)(sign | best);
}

float ep_oracle_f32_from_e2m1(uint8_t q)
{
    static const float mag[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};
    float v = mag[q & 0x7u];
    return (q & 0x8u) ? -v : v;
}

/* e8m0 scale code -> 2^(code - 127) (code 255 would be NaN; never produced here) */
float ep_oracle_f32_from_e8m0(uint8_t c)
{
    if (c == 0) return bits_f32(0x00400000u);                   /* 2^-127 */
    return bits_f32((uint32_t)c << 23);
}

/*
 * MX FP4 quantisation of BF16 rows (the "mxfp4" wire of the MORI-EP pages, read as the OCP
 * microscaling layout): blocks of 32 elements; with amax = max |x| of the block,
 *   shared exponent e = floor(log2(amax)) - 2   (2 = exponent of e2m1's largest value, 6)
 *   scale code       = e + 127, clamped to 0..254; an all-zero block uses code 127 (scale 1)
 *   codes            = e2m1 of (x / 2^e), exact division by a power of two, then RNE above
 * q [rows][H/2]: element 2i in the low nibble of byte i, 2i+1 in the high nibble;
 * scales [rows][H/32] e8m0 codes.  H must be a multiple of 32.
 */
int ep_oracle_quantize_mxfp4(int64_t rows, int H, const uint16_t* x, uint8_t* q, uint8_t* scales)
{
    if (H < 32 || H % 32 != 0 || rows < 0) return EP_ORACLE_ERR_ARG;
    const int nb = H / 32;
    for (int64_t r = 0; r < rows; ++r) {
        for (int b = 0; b < nb; ++b) {
            const uint16_t* xb = x + r * H + b * 32;
            float amax = 0.0f;
            for (int i = 0; i < 32; ++i) {
                float v = ep_oracle_f32_from_bf16(xb[i]);
                float m = v < 0.0f ? -v : v;
                if (m > amax) amax = m;
            }
            int code = 127;
            if (amax > 0.0f) {
                uint32_t ab = f32_bits(amax);
                int e2 = (int)(ab >> 23) - 127;                 /* floor(log2) of a normal */
                if ((ab >> 23) == 0) {                          /* subnormal amax */
                    uint32_t m = ab & 0x7FFFFFu;
                    e2 = -127;
                    while (!(m & 0x400000u)) { m <<= 1; --e2; }
                }
                code = e2 - 2 + 127;
                if (code < 0) code = 0;
                if (code > 254) code = 254;
            }
            scales[r * nb + b] = (uint8_t)code;
            const float s = ep_oracle_f32_from_e8m0((uint8_t)code);
            for (int i = 0; i < 32; i += 2) {
                uint8_t lo = ep_oracle_e2m1_from_f32(ep_oracle_f32_from_bf16(xb[i]) / s);
                uint8_t hi = ep_oracle_e2m1_from_f32(ep_oracle_f32_from_bf16(xb[i + 1]) / s);
                q[r * (H / 2) + b * 16 + i / 2] = (uint8_t)(lo | (hi << 4));
            }
        }
    }
    return EP_ORACLE_OK;
}

/*
 * Combine over the MX FP4 wire: as ep_oracle_combine_fp8, with each term
 *   v = float(code) * 2^(scale_code - 127)    (exact: a 2-bit significand times a power of two)
 * added in ascending rank order in FP32 from +0.0f; BF16 RNE output.
 *   q [W][W*M][H/2], scales [W][W*M][H/32].
 */
int ep_oracle_combine_fp4(int W, int k, int H, int M, const int32_t* n_tok, const int32_t* slot_of,
                          const uint8_t* q, const uint8_t* scales, const float* w_in, uint16_t* out,
                          float* out_w)
{
    if (W < 1 || k < 1 || H < 32 || H % 32 != 0 || M < 1) return EP_ORACLE_ERR_ARG;
    const int64_t rows = (int64_t)W * M;
    const int nb = H / 32;
    float* acc = (float*)malloc((size_t)H * sizeof(float));
    float* accw = (float*)malloc((size_t)k * sizeof(float));
    if (!acc || !accw) { free(acc); free(accw); return EP_ORACLE_ERR_ARG; }
    for (int s = 0; s < W; ++s) {
        for (int t = 0; t < n_tok[s]; ++t) {
            const int64_t tok = (int64_t)s * M + t;
            for (int h = 0; h < H; ++h) acc[h] = 0.0f;
            for (int j = 0; j < k; ++j) accw[j] = 0.0f;
            for (int r = 0; r < W; ++r) {
                const int32_t slot = slot_of[tok * W + r];
                if (slot < 0) continue;
                const int64_t row = (int64_t)r * rows + slot;
                for (int h = 0; h < H; ++h) {
                    uint8_t byte = q[row * (H / 2) + h / 2];
                    uint8_t code = (h & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xFu);
                    float v = ep_oracle_f32_from_e2m1(code) * ep_oracle_f32_from_e8m0(scales[row * nb + h / 32]);
                    acc[h] = acc[h] + v;
                }
                if (w_in)
                    for (int j = 0; j < k; ++j) accw[j] = accw[j] + w_in[row * k + j];
            }
            for (int h = 0; h < H; ++h) out[tok * H + h] = ep_oracle_bf16_from_f32(acc[h]);
            if (w_in && out_w)
                for (int j = 0; j < k; ++j) out_w[tok * k + j] = accw[j];
        }
    }
    free(acc);
    free(accw);
    return EP_ORACLE_OK;
}
