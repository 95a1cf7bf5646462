/*
 * moe_ref.c -- CPU oracle for MoE expert-parallel dispatch and combine.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously correct
 * statement of what the GPU path computes.  Only the test suite, the smoke
 * check and the benchmark's CPU-baseline leg load it.  It shares no code,
 * header, table or constant with the CUDA library.
 *
 * Every step is plain loops in the order the pages describe it:
 *
 *   "Enabling trillion-parameter models on AWS EFA" (Perplexity blog):
 *     - Introduction: dispatch sends each token to the ranks hosting its
 *       experts; combine returns the expert outputs and takes their weighted
 *       average.
 *     - "Send and receive buffers": N ranks, T tokens each, R experts per
 *       token out of E; senders lay out their writes contiguously per peer,
 *       which needs per-expert token counts exchanged first; a rank receives
 *       at most N*T*max(R, E/N) tokens.
 *     - "Dispatch and combine": per-expert counts with atomics in one block,
 *       a cumulative sum gives the offsets into contiguous per-peer send
 *       buffers, tokens are packed, receivers compute offsets once all
 *       routing info is in, and shuffle received tokens into the tensor
 *       handed to the grouped GEMM; combine shuffles outputs back, one write
 *       per peer, and accumulates the weighted average from the receive
 *       buffer.
 *     - "Evaluation: dispatch/combine latency": block-scaled fp8 dispatch,
 *       bf16 combine.
 *
 * Readings where the pages leave a step open:
 *   - one row per (token, expert) assignment, no per-rank de-duplication;
 *   - expert e lives on rank e / (E/N) (contiguous blocks of E/N experts);
 *   - within one expert, rows keep ascending flattened index t*R + k;
 *   - fp8 is OCP E4M3 ("E4M3FN": max 448, no infinities, S.1111.111 = NaN),
 *     per 128-element block: scale = amax / 448 in fp32, q = RNE satfinite
 *     e4m3 of (x / scale) in fp32; a block with amax == 0 has scale 0 and
 *     all-zero bytes;
 *   - the grouped layout orders rows by local expert, then sender, then
 *     the sender's order; no padding;
 *   - combine accumulates w_k * y_k in fp32 with one fused multiply-add per
 *     slot k = 0..R-1 in order, then rounds once to bf16 (nearest even);
 *   - an expert id outside [0, E) is skipped and flagged; a grouped or
 *     combine row at or beyond the capacity is dropped and flagged, and a
 *     dropped assignment contributes zero to the combine;
 *   - the send-side reduction (an alternative combine, see below) sums a
 *     token's weighted outputs per expert rank in slot order, rounds that
 *     partial once to bf16, and the receiver adds the partials in ascending
 *     rank order in fp32 and rounds once more.
 *
 * Precision: the pages fix fp32 scales, fp8 payload, bf16 outputs and fp32
 * accumulation, so those steps run in exactly those types here.  The
 * encoder and decoder work in double, where every step is exact.
 *
 * Build: gcc -O2 -std=c11 -fPIC -shared -ffp-contract=off -fno-fast-math
 * (contraction off: every multiply and add rounds as written).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define REF_ST_BAD_EXPERT 1
#define REF_ST_CAPACITY 2

/* ---------------------------------------------------------------- numbers */

/* bf16 -> fp32: a bf16 value is the upper half of an fp32 bit pattern. */
float ref_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* fp32 -> bf16, round to nearest, ties to even: keep the upper 16 bits and
 * look at the 16 bits dropped. */
uint16_t ref_f32_to_bf16_rn(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0)
        return (uint16_t)((u >> 16) | 0x0040u); /* NaN stays NaN (quiet) */
    uint32_t hi = u >> 16;
    uint32_t lo = u & 0xffffu;
    if (lo > 0x8000u || (lo == 0x8000u && (hi & 1u)))
        hi += 1u; /* carry into the exponent is the correct rounding */
    return (uint16_t)hi;
}

void ref_f32_to_bf16_array(const float *v, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = ref_f32_to_bf16_rn(v[i]);
}

/* Round half to even on a double that holds an exactly representable real. */
static double round_half_even(double v)
{
    double f = floor(v);
    double d = v - f;
    if (d > 0.5)
        return f + 1.0;
    if (d < 0.5)
        return f;
    return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;
}

/* OCP 8-bit floating point, E4M3 variant: 1 sign bit, 4 exponent bits with
 * bias 7, 3 mantissa bits; exponent field 0 holds subnormals m * 2^-9;
 * S.1111.111 is NaN; there is no infinity; largest finite 1.75 * 2^8 = 448. */
double ref_e4m3_decode(uint8_t c)
{
    int s = c >> 7, ef = (c >> 3) & 0xf, m = c & 7;
    double v;
    if (ef == 15 && m == 7)
        return NAN;
    if (ef == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp(1.0 + m / 8.0, ef - 7);
    return s ? -v : v;
}

/* Encode with round-to-nearest-even and saturation to the largest finite
 * value ("satfinite").  NaN maps to S.1111.111.  Magnitudes at or above 448
 * (448 itself, values that round up past it, infinity) saturate to 448. */
uint8_t ref_e4m3_encode(float v)
{
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    if (isnan(v))
        return (uint8_t)(sign | 0x7f);
    double a = fabs((double)v);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7e);
    if (a < ldexp(1.0, -6)) {
        /* subnormal spacing 2^-9; n == 8 is exactly the smallest normal,
         * whose code (exponent field 1, mantissa 0) is also 8 */
        double n = round_half_even(a / ldexp(1.0, -9));
        return (uint8_t)(sign | (uint8_t)n);
    }
    int k;
    frexp(a, &k); /* a = f * 2^k, f in [0.5, 1) */
    int E = k - 1; /* a in [2^E, 2^(E+1)) */
    double n = round_half_even(a / ldexp(1.0, E - 3)); /* in [8, 16] */
    if (n == 16.0) {
        E += 1;
        n = 8.0;
    }
    return (uint8_t)(sign | ((E + 7) << 3) | ((int)n - 8));
}

void ref_e4m3_encode_array(const float *v, uint8_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = ref_e4m3_encode(v[i]);
}

void ref_e4m3_decode_array(const uint8_t *c, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = ref_e4m3_decode(c[i]);
}

/* ---------------------------------------------------------------- dispatch */

/* Per-expert counts, per-peer and per-expert exclusive scans, stable slots.
 *
 *   cnt[s][e]         = #{(t,k) : idx[s][t][k] == e}
 *   expert_send_off[s][e] = sum_{e' < e} cnt[s][e'], last entry = total
 *   send_off[s][p]    = sum over peers p' < p of the tokens rank s sends to p'
 *   slot_row[s][t][k] = expert_send_off[s][e] + number of earlier (t',k')
 *                       (in flattened order) with the same expert; -1 if the
 *                       id is outside [0, E)
 *
 * Returns status bits (REF_ST_BAD_EXPERT). */
int ref_route_count(int N, int T, int E, int R, const int32_t *idx, int32_t *cnt,
                    int32_t *send_off, int32_t *expert_send_off, int32_t *slot_row)
{
    int st = 0;
    int Er = E / N;
    int32_t *fill = (int32_t *)calloc((size_t)E, sizeof(int32_t));
    for (int s = 0; s < N; ++s) {
        const int32_t *id = idx + (size_t)s * T * R;
        int32_t *c = cnt + (size_t)s * E;
        int32_t *eso = expert_send_off + (size_t)s * (E + 1);
        int32_t *so = send_off + (size_t)s * (N + 1);
        int32_t *slot = slot_row + (size_t)s * T * R;

        /* counts */
        for (int e = 0; e < E; ++e)
            c[e] = 0;
        for (int i = 0; i < T * R; ++i) {
            int e = id[i];
            if (e < 0 || e >= E) {
                st |= REF_ST_BAD_EXPERT;
                continue;
            }
            c[e] += 1;
        }
        /* exclusive scan over experts */
        int32_t acc = 0;
        for (int e = 0; e < E; ++e) {
            eso[e] = acc;
            acc += c[e];
        }
        eso[E] = acc;
        /* per-peer counts, exclusive scan over peers */
        acc = 0;
        for (int p = 0; p < N; ++p) {
            so[p] = acc;
            for (int j = 0; j < Er; ++j)
                acc += c[p * Er + j];
        }
        so[N] = acc;
        /* stable slot of every assignment */
        for (int e = 0; e < E; ++e)
            fill[e] = 0;
        for (int i = 0; i < T * R; ++i) {
            int e = id[i];
            if (e < 0 || e >= E) {
                slot[i] = -1;
                continue;
            }
            slot[i] = eso[e] + fill[e];
            fill[e] += 1;
        }
    }
    free(fill);
    return st;
}

/* Routing-information exchange and receive-side offsets.
 *
 * Receiver r hosts experts e = r*Er + j, j = 0..Er-1.
 *   seg_off[r][j][s] = offset of sender s's run of expert j in r's grouped
 *                      layout (order: j, then s)
 *   grp_off[r][j]    = first grouped row of local expert j; grp_off[r][Er]
 *                      is the number of rows r receives
 *   m_sizes[r][j]    = rows of local expert j
 *   csend_off[r][s]  = offset in r's combine send buffer of the rows going
 *                      back to s (order: s); csend_off[r][N] = total
 * Returns REF_ST_CAPACITY if some rank receives more than cap rows. */
int ref_exchange(int N, int E, int cap, const int32_t *cnt, const int32_t *send_off,
                 int32_t *grp_off, int32_t *seg_off, int32_t *csend_off, int32_t *m_sizes)
{
    int st = 0;
    int Er = E / N;
    for (int r = 0; r < N; ++r) {
        int32_t acc = 0;
        for (int j = 0; j < Er; ++j) {
            int e = r * Er + j;
            int32_t m = 0;
            grp_off[(size_t)r * (Er + 1) + j] = acc;
            for (int s = 0; s < N; ++s) {
                int32_t n = cnt[(size_t)s * E + e];
                seg_off[((size_t)r * Er + j) * N + s] = acc;
                acc += n;
                m += n;
            }
            m_sizes[(size_t)r * Er + j] = m;
        }
        grp_off[(size_t)r * (Er + 1) + Er] = acc;
        if (acc > cap)
            st |= REF_ST_CAPACITY;

        int32_t acc2 = 0;
        for (int s = 0; s < N; ++s) {
            const int32_t *so = send_off + (size_t)s * (N + 1);
            csend_off[(size_t)r * (N + 1) + s] = acc2;
            acc2 += so[r + 1] - so[r];
        }
        csend_off[(size_t)r * (N + 1) + N] = acc2;
    }
    return st;
}

/* Block-scaled fp8 quantisation of one token row of H bf16 values.
 * For block b of 128 elements:
 *   amax  = max |x|
 *   scale = amax / 448            (fp32 division)
 *   q     = e4m3(x / scale)       (fp32 division, then RNE satfinite)
 * A block with amax == 0 gets scale 0 and all-zero bytes. */
void ref_quant_token(int H, const uint16_t *xr, uint8_t *q, float *scales)
{
    int Sb = H / 128;
    for (int b = 0; b < Sb; ++b) {
        float amax = 0.0f;
        for (int u = 0; u < 128; ++u) {
            float v = fabsf(ref_bf16_to_f32(xr[b * 128 + u]));
            if (v > amax)
                amax = v;
        }
        float scale = amax / 448.0f;
        scales[b] = scale;
        for (int u = 0; u < 128; ++u) {
            if (amax == 0.0f) {
                q[b * 128 + u] = 0;
            } else {
                float v = ref_bf16_to_f32(xr[b * 128 + u]) / scale;
                q[b * 128 + u] = ref_e4m3_encode(v);
            }
        }
    }
}

/* Quantisation fused with the pack into the send buffer: the token's R
 * copies go to rows slot_row[s][t][k] of rank s's send buffer, with the
 * scales beside them and the token id in send_tok. */
void ref_dispatch_send(int N, int T, int R, int H, const uint16_t *x,
                       const int32_t *slot_row, uint8_t *send_q, float *send_s,
                       int32_t *send_tok)
{
    int Sb = H / 128;
    uint8_t *q = (uint8_t *)malloc((size_t)H);
    float *sc = (float *)malloc((size_t)Sb * sizeof(float));
    for (int s = 0; s < N; ++s) {
        for (int t = 0; t < T; ++t) {
            const int32_t *slot = slot_row + ((size_t)s * T + t) * R;
            ref_quant_token(H, x + ((size_t)s * T + t) * H, q, sc);
            for (int k = 0; k < R; ++k) {
                if (slot[k] < 0)
                    continue;
                size_t row = (size_t)s * T * R + slot[k];
                memcpy(send_q + row * H, q, (size_t)H);
                memcpy(send_s + row * Sb, sc, (size_t)Sb * sizeof(float));
                send_tok[row] = t;
            }
        }
    }
    free(q);
    free(sc);
}

/* Receive-side shuffle into the expert-grouped layout.  For every receiver r,
 * local expert j and sender s, the contiguous run of cnt[s][e] rows that s
 * packed for expert e (starting at expert_send_off[s][e]) is copied to r's
 * grouped rows starting at seg_off[r][j][s]; grp_src records (s, t).  Rows at
 * or beyond cap are dropped. */
void ref_dispatch_recv(int N, int T, int E, int R, int H, int cap,
                       const uint8_t *send_q, const float *send_s,
                       const int32_t *send_tok, const int32_t *cnt,
                       const int32_t *expert_send_off, const int32_t *seg_off,
                       uint8_t *grp_q, float *grp_s, int32_t *grp_src)
{
    int Er = E / N, Sb = H / 128;
    for (int r = 0; r < N; ++r) {
        for (int j = 0; j < Er; ++j) {
            int e = r * Er + j;
            for (int s = 0; s < N; ++s) {
                int32_t n = cnt[(size_t)s * E + e];
                int32_t src0 = expert_send_off[(size_t)s * (E + 1) + e];
                int32_t dst0 = seg_off[((size_t)r * Er + j) * N + s];
                for (int32_t u = 0; u < n; ++u) {
                    int32_t g = dst0 + u;
                    if (g >= cap)
                        continue;
                    size_t srow = (size_t)s * T * R + src0 + u;
                    size_t drow = (size_t)r * cap + g;
                    memcpy(grp_q + drow * H, send_q + srow * H, (size_t)H);
                    memcpy(grp_s + drow * Sb, send_s + srow * Sb, (size_t)Sb * sizeof(float));
                    grp_src[drow * 2 + 0] = s;
                    grp_src[drow * 2 + 1] = send_tok[srow];
                }
            }
        }
    }
}

/* Stand-in for the grouped GEMM (not part of the timed path), one row of
 * expert e:  y = bf16_rn((decode(q) * scale) * s_e)  with fp32 multiplies,
 * s_e = 1 (mode 0, identity) or 2^((e mod 3) - 1) (mode 1, per-expert scale). */
void ref_standin_row(int H, int mode, int e, const uint8_t *q, const float *scales,
                     uint16_t *y)
{
    float se = (mode == 0) ? 1.0f : (float)ldexp(1.0, (e % 3) - 1);
    for (int h = 0; h < H; ++h) {
        float dq = (float)ref_e4m3_decode(q[h]);
        float v = dq * scales[h / 128];
        v = v * se;
        y[h] = ref_f32_to_bf16_rn(v);
    }
}

/* The stand-in over every received row of every rank; rows beyond the
 * received count (and beyond cap) are left untouched. */
void ref_expert_standin(int N, int E, int H, int cap, int mode, const uint8_t *grp_q,
                        const float *grp_s, const int32_t *grp_off, uint16_t *y)
{
    int Er = E / N, Sb = H / 128;
    for (int r = 0; r < N; ++r) {
        for (int j = 0; j < Er; ++j) {
            int e = r * Er + j;
            int32_t g0 = grp_off[(size_t)r * (Er + 1) + j];
            int32_t g1 = grp_off[(size_t)r * (Er + 1) + j + 1];
            for (int32_t g = g0; g < g1 && g < cap; ++g) {
                size_t row = (size_t)r * cap + g;
                ref_standin_row(H, mode, e, grp_q + row * H, grp_s + row * Sb, y + row * H);
            }
        }
    }
}

/* ----------------------------------------------------------------- combine */

/* Combine send: expert rank r copies, for every local expert j and source s,
 * the run of outputs y (grouped rows from seg_off[r][j][s]) into its combine
 * send buffer at csend_off[r][s] + (expert_send_off[s][e] - send_off[s][r]),
 * so the rows going back to s are contiguous and in s's own send order.  A
 * row whose grouped position was dropped (>= cap) is sent as zeros; a row
 * whose combine position is >= cap is dropped. */
void ref_combine_send(int N, int T, int E, int R, int H, int cap, const uint16_t *y,
                      const int32_t *cnt, const int32_t *expert_send_off,
                      const int32_t *send_off, const int32_t *seg_off,
                      const int32_t *csend_off, uint16_t *csend)
{
    (void)T;
    (void)R;
    int Er = E / N;
    for (int r = 0; r < N; ++r) {
        for (int j = 0; j < Er; ++j) {
            int e = r * Er + j;
            for (int s = 0; s < N; ++s) {
                int32_t n = cnt[(size_t)s * E + e];
                int32_t g0 = seg_off[((size_t)r * Er + j) * N + s];
                int32_t c0 = csend_off[(size_t)r * (N + 1) + s] +
                             (expert_send_off[(size_t)s * (E + 1) + e] -
                              send_off[(size_t)s * (N + 1) + r]);
                for (int32_t u = 0; u < n; ++u) {
                    int32_t g = g0 + u, c = c0 + u;
                    if (c >= cap)
                        continue;
                    uint16_t *dst = csend + ((size_t)r * cap + c) * H;
                    if (g >= cap)
                        memset(dst, 0, (size_t)H * sizeof(uint16_t));
                    else
                        memcpy(dst, y + ((size_t)r * cap + g) * H, (size_t)H * sizeof(uint16_t));
                }
            }
        }
    }
}

/* Weighted sum of one token's R rows (bf16, R x H, row k at rows + k*H):
 *   acc = 0;  for k = 0..R-1 with use[k]:  acc = fma(w[k], row_k, acc)
 *   out = bf16_rn(acc) */
void ref_weighted_sum(int R, int H, const uint16_t *rows, const float *w,
                      const int32_t *use, uint16_t *out)
{
    for (int h = 0; h < H; ++h) {
        float acc = 0.0f;
        for (int k = 0; k < R; ++k)
            if (use[k])
                acc = fmaf(w[k], ref_bf16_to_f32(rows[(size_t)k * H + h]), acc);
        out[h] = ref_f32_to_bf16_rn(acc);
    }
}

/* Combine receive: for token t of rank s, row k is read from the combine
 * send buffer of the expert's rank p at
 *   csend_off[p][s] + (slot_row[s][t][k] - send_off[s][p])
 * and the R rows are reduced by ref_weighted_sum.  Skipped (bad id) and
 * dropped (>= cap) assignments contribute nothing. */
void ref_combine_recv(int N, int T, int E, int R, int H, int cap, const uint16_t *csend,
                      const int32_t *idx, const float *w, const int32_t *slot_row,
                      const int32_t *send_off, const int32_t *csend_off, uint16_t *out)
{
    int Er = E / N;
    uint16_t *rows = (uint16_t *)calloc((size_t)R * H, sizeof(uint16_t));
    int32_t *use = (int32_t *)calloc((size_t)R, sizeof(int32_t));
    for (int s = 0; s < N; ++s) {
        for (int t = 0; t < T; ++t) {
            size_t tok = (size_t)s * T + t;
            for (int k = 0; k < R; ++k) {
                int e = idx[tok * R + k];
                int32_t slot = slot_row[tok * R + k];
                use[k] = 0;
                if (e < 0 || e >= E || slot < 0)
                    continue;
                int p = e / Er;
                int32_t q = slot - send_off[(size_t)s * (N + 1) + p];
                int32_t c = csend_off[(size_t)p * (N + 1) + s] + q;
                if (c >= cap)
                    continue;
                memcpy(rows + (size_t)k * H, csend + ((size_t)p * cap + c) * H,
                       (size_t)H * sizeof(uint16_t));
                use[k] = 1;
            }
            ref_weighted_sum(R, H, rows, w + tok * R, use, out + tok * H);
        }
    }
    free(rows);
    free(use);
}

/* ------------------------------------------------------------ send-side reduction */

/* Send-side accumulation for the combine: the alternative that the EFA page's
 * evaluation ("Evaluation: dispatch/combine latency", prefill) contrasts with
 * its own receive-side-only accumulation -- another implementation sums on
 * the sending side to cut the bytes transferred, with some risk to accuracy.
 * On expert rank r, for every token t of every sender s with at least one
 * assignment to an expert of r (valid id, slot_row >= 0), the weighted
 * outputs of those experts are summed before they leave r:
 *   acc = 0;  for k = 0..R-1 in order with e_k / Er == r:
 *               acc = fma(w_k, y_k, acc)        (y_k = 0 if its grouped row
 *                                                 was dropped at capacity)
 *   part[r][s][t] = bf16_rn(acc)
 * one partial row per (r, s, t) in the fixed layout [N][N][T][H]; the rows of
 * an (r, s, t) without such an assignment are not written. */
void ref_combine_partial_send(int N, int T, int E, int R, int H, int cap, const uint16_t *y,
                              const int32_t *idx, const float *w, const int32_t *slot_row,
                              const int32_t *expert_send_off, const int32_t *seg_off,
                              uint16_t *part)
{
    int Er = E / N;
    float *acc = (float *)calloc((size_t)H, sizeof(float));
    for (int r = 0; r < N; ++r) {
        for (int s = 0; s < N; ++s) {
            for (int t = 0; t < T; ++t) {
                size_t tok = (size_t)s * T + t;
                int has = 0;
                for (int h = 0; h < H; ++h)
                    acc[h] = 0.0f;
                for (int k = 0; k < R; ++k) {
                    int e = idx[tok * R + k];
                    int32_t slot = slot_row[tok * R + k];
                    if (e < 0 || e >= E || slot < 0 || e / Er != r)
                        continue;
                    has = 1;
                    int j = e - r * Er;
                    int32_t g = seg_off[((size_t)r * Er + j) * N + s] +
                                (slot - expert_send_off[(size_t)s * (E + 1) + e]);
                    if (g >= cap)
                        continue; /* dropped: the expert output is zero */
                    const uint16_t *row = y + ((size_t)r * cap + g) * H;
                    for (int h = 0; h < H; ++h)
                        acc[h] = fmaf(w[tok * R + k], ref_bf16_to_f32(row[h]), acc[h]);
                }
                if (!has)
                    continue;
                uint16_t *dst = part + (((size_t)r * N + s) * T + t) * H;
                for (int h = 0; h < H; ++h)
                    dst[h] = ref_f32_to_bf16_rn(acc[h]);
            }
        }
    }
    free(acc);
}

/* The receiving side of the send-side reduction: token t of rank s adds the
 * partial rows of the ranks its experts live on, in ascending rank order, in
 * fp32, and rounds once:
 *   acc = 0;  for r = 0..N-1 with a partial row:  acc = acc + float(part[r][s][t])
 *   out[s][t] = bf16_rn(acc)                      (0 for a token with none) */
void ref_combine_partial_recv(int N, int T, int E, int R, int H, const uint16_t *part,
                              const int32_t *idx, const int32_t *slot_row, uint16_t *out)
{
    int Er = E / N;
    float *acc = (float *)calloc((size_t)H, sizeof(float));
    for (int s = 0; s < N; ++s) {
        for (int t = 0; t < T; ++t) {
            size_t tok = (size_t)s * T + t;
            for (int h = 0; h < H; ++h)
                acc[h] = 0.0f;
            for (int r = 0; r < N; ++r) {
                int present = 0;
                for (int k = 0; k < R; ++k) {
                    int e = idx[tok * R + k];
                    if (e >= 0 && e < E && slot_row[tok * R + k] >= 0 && e / Er == r)
                        present = 1;
                }
                if (!present)
                    continue;
                const uint16_t *row = part + (((size_t)r * N + s) * T + t) * H;
                for (int h = 0; h < H; ++h)
                    acc[h] = acc[h] + ref_bf16_to_f32(row[h]);
            }
            for (int h = 0; h < H; ++h)
                out[tok * H + h] = ref_f32_to_bf16_rn(acc[h]);
        }
    }
    free(acc);
}

/* ------------------------------------------------------------ low latency */

/* Low-latency layout, after the fixed-size receive buffers of the
 * low-latency mode the RoCE->EFA page describes (section 4.4: a preset
 * per-rank token limit, one kernel, no count-then-allocate round):
 * receiver r keeps, for each local expert j and sender s, a region of T rows.
 * Assignment (t, k) of sender s with expert e = r*Er + j takes row
 *   ll_row = ((r*Er + j)*N + s)*T + u,
 * u = number of earlier (t', k') of rank s, in flattened order, with the same
 * expert (the same stable order as slot_row).  u >= T cannot happen when a
 * token's experts are distinct; otherwise the row is dropped (-1) and
 * REF_ST_CAPACITY is returned.  Bad ids give -1 and REF_ST_BAD_EXPERT.
 * ll_count[r][j][s] = number of assignments of s to expert r*Er + j. */
int ref_ll_rows(int N, int T, int E, int R, const int32_t *idx, int32_t *ll_row,
                int32_t *ll_count)
{
    int st = 0;
    int Er = E / N;
    int32_t *seen = (int32_t *)calloc((size_t)E, sizeof(int32_t));
    for (int i = 0; i < N * E; ++i)
        ll_count[i] = 0;
    for (int s = 0; s < N; ++s) {
        for (int e = 0; e < E; ++e)
            seen[e] = 0;
        for (int i = 0; i < T * R; ++i) {
            size_t a = (size_t)s * T * R + i;
            int e = idx[a];
            if (e < 0 || e >= E) {
                ll_row[a] = -1;
                st |= REF_ST_BAD_EXPERT;
                continue;
            }
            int r = e / Er, j = e % Er;
            int u = seen[e];
            seen[e] += 1;
            ll_count[((size_t)r * Er + j) * N + s] += 1;
            if (u >= T) {
                ll_row[a] = -1;
                st |= REF_ST_CAPACITY;
                continue;
            }
            ll_row[a] = (int32_t)((((size_t)r * Er + j) * N + s) * T + u);
        }
    }
    free(seen);
    return st;
}

/* Quantise each token (ref_quant_token) and place its copies at the
 * low-latency rows, with the source token id beside them. */
void ref_dispatch_ll(int N, int T, int R, int H, const uint16_t *x, const int32_t *ll_row,
                     uint8_t *ll_q, float *ll_s, int32_t *ll_src)
{
    int Sb = H / 128;
    uint8_t *q = (uint8_t *)malloc((size_t)H);
    float *sc = (float *)malloc((size_t)Sb * sizeof(float));
    for (int s = 0; s < N; ++s) {
        for (int t = 0; t < T; ++t) {
            size_t tok = (size_t)s * T + t;
            ref_quant_token(H, x + tok * H, q, sc);
            for (int k = 0; k < R; ++k) {
                int32_t row = ll_row[tok * R + k];
                if (row < 0)
                    continue;
                memcpy(ll_q + (size_t)row * H, q, (size_t)H);
                memcpy(ll_s + (size_t)row * Sb, sc, (size_t)Sb * sizeof(float));
                ll_src[row] = t;
            }
        }
    }
    free(q);
    free(sc);
}

/* Stand-in expert over the low-latency layout: rows u < min(count, T) of
 * every region (r, j, s) of expert e = r*Er + j. */
void ref_standin_ll(int N, int T, int E, int H, int mode, const uint8_t *ll_q,
                    const float *ll_s, const int32_t *ll_count, uint16_t *y_ll)
{
    int Er = E / N, Sb = H / 128;
    for (int r = 0; r < N; ++r)
        for (int j = 0; j < Er; ++j)
            for (int s = 0; s < N; ++s) {
                size_t reg = ((size_t)r * Er + j) * N + s;
                int n = ll_count[reg] < T ? ll_count[reg] : T;
                for (int u = 0; u < n; ++u) {
                    size_t row = reg * T + u;
                    ref_standin_row(H, mode, r * Er + j, ll_q + row * H, ll_s + row * Sb,
                                    y_ll + row * H);
                }
            }
}

/* Combine over the low-latency layout: token (s, t) reduces its R rows
 * y_ll[ll_row[s][t][k]] with ref_weighted_sum (dropped rows contribute
 * nothing). */
void ref_combine_ll(int N, int T, int R, int H, const uint16_t *y_ll, const float *w,
                    const int32_t *ll_row, uint16_t *out)
{
    uint16_t *rows = (uint16_t *)calloc((size_t)R * H, sizeof(uint16_t));
    int32_t *use = (int32_t *)calloc((size_t)R, sizeof(int32_t));
    for (int s = 0; s < N; ++s)
        for (int t = 0; t < T; ++t) {
            size_t tok = (size_t)s * T + t;
            for (int k = 0; k < R; ++k) {
                int32_t row = ll_row[tok * R + k];
                use[k] = row >= 0;
                if (row >= 0)
                    memcpy(rows + (size_t)k * H, y_ll + (size_t)row * H, (size_t)H * 2);
            }
            ref_weighted_sum(R, H, rows, w + tok * R, use, out + tok * H);
        }
    free(rows);
    free(use);
}
