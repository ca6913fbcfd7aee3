/*
 * oracle.c — plain, slow, CPU reference for GGUF block-quantized GEMV and the
 * decode-time MoE FFN.  TEST INFRASTRUCTURE ONLY: the test suite, the smoke
 * check and the benchmark's CPU-baseline leg are the only callers.  The
 * product path (the CUDA library) never links, loads or calls this file, and
 * this file shares no code, header, table or helper with it.
 *
 * Sources (page titles; sections are the Rust/CUDA items on those pages):
 *   [ferrox gpu.rs]  "ferrox-cuda 0.14.0 — src/gpu.rs": the CUDA C kernel
 *       sources Q8_0_MATVEC_KERNEL_SRC, Q4_0_MATVEC_KERNEL_SRC,
 *       Q4_K_MATVEC_KERNEL_SRC (with ferrox_f16_to_f32 and
 *       ferrox_q4_k_scale_min), Q5_K_MATVEC_KERNEL_SRC, Q6_K_MATVEC_KERNEL_SRC
 *       and SILU_MUL_KERNEL_SRC; launch_dense_ffn_swiglu.
 *   [ferrox weight_matrix.rs] "ferrox-core 0.16.0 — weight_matrix.rs":
 *       block_bytes_per_row, dequant_row, apply.
 *   [aprender qwen3 moe] "aprender-serve 0.70.2 —
 *       forward_qwen3_moe_resident.rs": module doc (op order, "Kernels"),
 *       ExpertStack::expert, moe_layer, last_routes.
 *   [ferrox gpu.rs] also gives FUSED_ADD_RMSNORM_KERNEL_SRC (ffn_norm).
 *
 * Precision: block values are formed in f32 in the order the page kernels
 * write them; every dot product and every MoE intermediate is carried in
 * double; outputs are returned as double and the caller rounds.
 *
 * Build: gcc -O2 -std=c99 -ffp-contract=off -fPIC -shared (no fast-math, no
 * explicit SIMD) — see oracle/__init__.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Format codes understood by this oracle (its own numbering). */
enum { ORC_F32 = 0, ORC_Q8_0 = 1, ORC_Q4_0 = 2, ORC_Q4_K = 3, ORC_Q5_K = 4, ORC_Q6_K = 5 };

/* Elements and bytes per block — [ferrox gpu.rs] kernel doc comments:
 * Q8_0 34-byte blocks of 32; Q4_0 18-byte blocks of 32; Q4_K 144-byte
 * super-blocks of 256; Q5_K 176 of 256; Q6_K 210 of 256. */
int orc_block_elems(int qt) {
    switch (qt) {
    case ORC_F32: return 1;
    case ORC_Q8_0: case ORC_Q4_0: return 32;
    case ORC_Q4_K: case ORC_Q5_K: case ORC_Q6_K: return 256;
    default: return 0;
    }
}
int orc_block_bytes(int qt) {
    switch (qt) {
    case ORC_F32: return 4;
    case ORC_Q8_0: return 34;
    case ORC_Q4_0: return 18;
    case ORC_Q4_K: return 144;
    case ORC_Q5_K: return 176;
    case ORC_Q6_K: return 210;
    default: return 0;
    }
}
/* [ferrox weight_matrix.rs] block_bytes_per_row: (cols / elems) * bytes. */
int64_t orc_row_bytes(int qt, int64_t cols) {
    int be = orc_block_elems(qt);
    if (be <= 0 || cols % be) return -1;
    return (cols / be) * orc_block_bytes(qt);
}

/* IEEE 754 binary16 -> binary32, from the definition of the format
 * (sign 1, exponent 5 biased by 15, fraction 10), as ferrox_f16_to_f32 in
 * [ferrox gpu.rs] states it: exponent 0 is subnormal (fraction * 2^-24),
 * exponent 31 is Inf (fraction 0) or NaN, otherwise (1024+fraction)*2^(e-25).
 * Bytes are little-endian. */
float orc_f16_to_f32(uint16_t h) {
    unsigned sign = (h >> 15) & 1u;
    unsigned e = (h >> 10) & 31u;
    unsigned f = h & 1023u;
    float v;
    if (e == 0)
        v = ldexpf((float)f, -24);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexpf((float)(f + 1024u), (int)e - 25);
    return sign ? -v : v;
}

static uint16_t le16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }

/* 6-bit (scale, min) pair j of a Q4_K / Q5_K super-block, from 12 packed
 * bytes — ferrox_q4_k_scale_min in [ferrox gpu.rs]. */
void orc_k_scale_min(int j, const uint8_t *s, uint8_t *sc, uint8_t *m) {
    if (j < 4) {
        *sc = s[j] & 63;
        *m = s[j + 4] & 63;
    } else {
        *sc = (uint8_t)((s[j + 4] & 15) | ((s[j - 4] >> 6) << 4));
        *m = (uint8_t)((s[j + 4] >> 4) | ((s[j] >> 6) << 4));
    }
}

/* ---- one block -> f32 values, in the page kernels' expression order ---- */

/* Q8_0_MATVEC_KERNEL_SRC: f16 d, then 32 signed bytes; value d * q. */
static void dec_q8_0(const uint8_t *b, float *out) {
    float d = orc_f16_to_f32(le16(b));
    for (int i = 0; i < 32; i++) out[i] = d * (float)(int8_t)b[2 + i];
}

/* Q4_0_MATVEC_KERNEL_SRC: f16 d, 16 bytes; byte i low nibble -> element i,
 * high nibble -> element i+16; value (nibble - 8) * d. */
static void dec_q4_0(const uint8_t *b, float *out) {
    float d = orc_f16_to_f32(le16(b));
    for (int i = 0; i < 16; i++) {
        int lo = (b[2 + i] & 15) - 8;
        int hi = (b[2 + i] >> 4) - 8;
        out[i] = (float)lo * d;
        out[i + 16] = (float)hi * d;
    }
}

/* Q4_K_MATVEC_KERNEL_SRC: d @0, dmin @2, scales[12] @4, qs[128] @16.
 * Group oi (0..3) uses pairs 2oi and 2oi+1; qs[32oi+l] low nibble is
 * element 64oi+l, high nibble element 64oi+32+l;
 * value (d*sc)*q - dmin*m. */
static void dec_q4_k(const uint8_t *b, float *out) {
    float d = orc_f16_to_f32(le16(b));
    float dmin = orc_f16_to_f32(le16(b + 2));
    const uint8_t *scales = b + 4, *qs = b + 16;
    for (int oi = 0; oi < 4; oi++) {
        uint8_t sc1, m1, sc2, m2;
        orc_k_scale_min(2 * oi, scales, &sc1, &m1);
        orc_k_scale_min(2 * oi + 1, scales, &sc2, &m2);
        float d1 = d * (float)sc1, min1 = dmin * (float)m1;
        float d2 = d * (float)sc2, min2 = dmin * (float)m2;
        for (int l = 0; l < 32; l++) {
            float p1 = d1 * (float)(qs[32 * oi + l] & 15);
            float p2 = d2 * (float)(qs[32 * oi + l] >> 4);
            out[64 * oi + l] = p1 - min1;
            out[64 * oi + 32 + l] = p2 - min2;
        }
    }
}

/* Q5_K_MATVEC_KERNEL_SRC: d @0, dmin @2, scales[12] @4, qh[32] @16,
 * qs[128] @48.  As Q4_K, plus 16 when bit 2oi (low half) or 2oi+1 (high
 * half) of qh[l] is set. */
static void dec_q5_k(const uint8_t *b, float *out) {
    float d = orc_f16_to_f32(le16(b));
    float dmin = orc_f16_to_f32(le16(b + 2));
    const uint8_t *scales = b + 4, *qh = b + 16, *qs = b + 48;
    for (int oi = 0; oi < 4; oi++) {
        uint8_t sc1, m1, sc2, m2;
        orc_k_scale_min(2 * oi, scales, &sc1, &m1);
        orc_k_scale_min(2 * oi + 1, scales, &sc2, &m2);
        float d1 = d * (float)sc1, min1 = dmin * (float)m1;
        float d2 = d * (float)sc2, min2 = dmin * (float)m2;
        unsigned u1 = 1u << (2 * oi), u2 = 2u << (2 * oi);
        for (int l = 0; l < 32; l++) {
            int q1 = (qs[32 * oi + l] & 15) + ((qh[l] & u1) ? 16 : 0);
            int q2 = (qs[32 * oi + l] >> 4) + ((qh[l] & u2) ? 16 : 0);
            float p1 = d1 * (float)q1;
            float p2 = d2 * (float)q2;
            out[64 * oi + l] = p1 - min1;
            out[64 * oi + 32 + l] = p2 - min2;
        }
    }
}

/* Q6_K_MATVEC_KERNEL_SRC: ql[128] @0, qh[64] @128, signed int8 sc[16] @192,
 * f16 d @208.  Two halves of 128; in half h, for l < 32 with is = l/16,
 * four 6-bit values (4 bits of ql, 2 bits of qh) minus 32 land at
 * elements 128h + l, +32, +64, +96 with scales sc[is], sc[is+2], sc[is+4],
 * sc[is+6]; value (d*sc)*q. */
static void dec_q6_k(const uint8_t *b, float *out) {
    float d = orc_f16_to_f32(le16(b + 208));
    for (int h = 0; h < 2; h++) {
        const uint8_t *ql = b + 64 * h, *qh = b + 128 + 32 * h;
        const int8_t *sc = (const int8_t *)(b + 192 + 8 * h);
        for (int l = 0; l < 32; l++) {
            int is = l / 16;
            int q1 = ((ql[l] & 15) | ((qh[l] & 3) << 4)) - 32;
            int q2 = ((ql[l + 32] & 15) | (((qh[l] >> 2) & 3) << 4)) - 32;
            int q3 = ((ql[l] >> 4) | (((qh[l] >> 4) & 3) << 4)) - 32;
            int q4 = ((ql[l + 32] >> 4) | (((qh[l] >> 6) & 3) << 4)) - 32;
            out[128 * h + l] = (d * (float)sc[is]) * (float)q1;
            out[128 * h + l + 32] = (d * (float)sc[is + 2]) * (float)q2;
            out[128 * h + l + 64] = (d * (float)sc[is + 4]) * (float)q3;
            out[128 * h + l + 96] = (d * (float)sc[is + 6]) * (float)q4;
        }
    }
}

/* Decode one block of format qt into orc_block_elems(qt) floats. */
int orc_decode_block(int qt, const uint8_t *blk, float *out) {
    switch (qt) {
    case ORC_F32: memcpy(out, blk, 4); return 0;
    case ORC_Q8_0: dec_q8_0(blk, out); return 0;
    case ORC_Q4_0: dec_q4_0(blk, out); return 0;
    case ORC_Q4_K: dec_q4_k(blk, out); return 0;
    case ORC_Q5_K: dec_q5_k(blk, out); return 0;
    case ORC_Q6_K: dec_q6_k(blk, out); return 0;
    default: return -1;
    }
}

/* [ferrox weight_matrix.rs] dequant_row: one row of `cols` values. */
int orc_dequant_row(int qt, const uint8_t *row, int64_t cols, float *out) {
    int be = orc_block_elems(qt), bb = orc_block_bytes(qt);
    if (be <= 0 || cols % be) return -1;
    for (int64_t b = 0; b < cols / be; b++)
        if (orc_decode_block(qt, row + b * bb, out + b * be)) return -1;
    return 0;
}

/* Dense y = W x ([ferrox weight_matrix.rs] apply: out[r] = row_r . x), by
 * decode-then-dot: each row is decoded to f32, then summed in double.
 * Optionally also returns sabs[r] = sum_j |w_rj * x_j| (the tolerance
 * scale of one GEMV output). */
int orc_matvec(int qt, const uint8_t *W, int64_t rows, int64_t cols, const float *x,
               double *y, double *sabs) {
    int64_t rb = orc_row_bytes(qt, cols);
    if (rb < 0) return -1;
    float *w = (float *)malloc(sizeof(float) * (size_t)cols);
    if (!w) return -2;
    for (int64_t r = 0; r < rows; r++) {
        orc_dequant_row(qt, W + r * rb, cols, w);
        double acc = 0.0, aabs = 0.0;
        for (int64_t j = 0; j < cols; j++) {
            double p = (double)w[j] * (double)x[j];
            acc += p;
            aabs += fabs(p);
        }
        y[r] = acc;
        if (sabs) sabs[r] = aabs;
    }
    free(w);
    return 0;
}

/* The same product computed the "fused" way the page kernels and the CPU
 * scalar dots do it: each block is decoded inside the dot loop, value by
 * value, without materialising the row.  Written separately from the
 * decoders above (same formulas, restated inline) so the two paths check
 * each other. */
int orc_matvec_fused(int qt, const uint8_t *W, int64_t rows, int64_t cols, const float *x,
                     double *y) {
    int64_t rb = orc_row_bytes(qt, cols);
    if (rb < 0) return -1;
    int be = orc_block_elems(qt), bb = orc_block_bytes(qt);
    int64_t nb = cols / be;
    for (int64_t r = 0; r < rows; r++) {
        const uint8_t *row = W + r * rb;
        double acc = 0.0;
        for (int64_t bi = 0; bi < nb; bi++) {
            const uint8_t *b = row + bi * bb;
            const float *xb = x + bi * be;
            if (qt == ORC_F32) {
                float v;
                memcpy(&v, b, 4);
                acc += (double)v * (double)xb[0];
            } else if (qt == ORC_Q8_0) {
                float d = orc_f16_to_f32(le16(b));
                for (int i = 0; i < 32; i++)
                    acc += (double)(d * (float)(int8_t)b[2 + i]) * (double)xb[i];
            } else if (qt == ORC_Q4_0) {
                float d = orc_f16_to_f32(le16(b));
                for (int i = 0; i < 32; i++) {
                    int nib = i < 16 ? (b[2 + i] & 15) : (b[2 + i - 16] >> 4);
                    acc += (double)((float)(nib - 8) * d) * (double)xb[i];
                }
            } else if (qt == ORC_Q4_K || qt == ORC_Q5_K) {
                float d = orc_f16_to_f32(le16(b));
                float dmin = orc_f16_to_f32(le16(b + 2));
                const uint8_t *qs = b + (qt == ORC_Q4_K ? 16 : 48);
                const uint8_t *qh = b + 16;
                for (int e = 0; e < 256; e++) {
                    int oi = e / 64, hi = (e % 64) >= 32, l = e % 32;
                    int j = 2 * oi + hi;
                    uint8_t sc, m;
                    orc_k_scale_min(j, b + 4, &sc, &m);
                    int q = hi ? (qs[32 * oi + l] >> 4) : (qs[32 * oi + l] & 15);
                    if (qt == ORC_Q5_K && ((qh[l] >> j) & 1)) q += 16;
                    float ds = d * (float)sc, mn = dmin * (float)m;
                    float p = ds * (float)q;
                    acc += (double)(p - mn) * (double)xb[e];
                }
            } else if (qt == ORC_Q6_K) {
                float d = orc_f16_to_f32(le16(b + 208));
                for (int e = 0; e < 256; e++) {
                    int h = e / 128, t = e % 128, quarter = t / 32, l = t % 32;
                    const uint8_t *ql = b + 64 * h, *qh = b + 128 + 32 * h;
                    int lowbits = (quarter & 1) ? ql[l + 32] : ql[l];
                    lowbits = (quarter >= 2) ? (lowbits >> 4) : (lowbits & 15);
                    int highbits = (qh[l] >> (2 * quarter)) & 3;
                    int q = (lowbits | (highbits << 4)) - 32;
                    int8_t s = (int8_t)b[192 + 8 * h + l / 16 + 2 * quarter];
                    acc += (double)((d * (float)s) * (float)q) * (double)xb[e];
                }
            } else {
                return -1;
            }
        }
        y[r] = acc;
    }
    return 0;
}

/* ------------------------------ routing ---------------------------------
 * [aprender qwen3 moe] module doc and moe_layer: router logits -> softmax
 * over all experts -> the k largest -> renormalise over those k; the
 * routes come back as (expert, weight) pairs in rank order (last_routes).
 * Readings (the routing function's body is not on the pages): softmax in
 * double with the maximum subtracted; ranking by probability, descending,
 * equal probabilities ranked by the lower expert index; w_s = p_s / sum
 * of the k selected p.
 * renorm = 0 skips the last step (w_s = p_s, the softmax probability over
 * all E experts): the pages do not say whether the OLMoE-shaped layer
 * renormalises, so both readings are available. */
int orc_route(const double *logits, int E, int k, int renorm, int32_t *idx, double *w) {
    if (E <= 0 || k <= 0 || k > E) return -1;
    double mx = logits[0];
    for (int e = 1; e < E; e++)
        if (logits[e] > mx) mx = logits[e];
    double *p = (double *)malloc(sizeof(double) * (size_t)E);
    int *order = (int *)malloc(sizeof(int) * (size_t)E);
    if (!p || !order) { free(p); free(order); return -2; }
    double z = 0.0;
    for (int e = 0; e < E; e++) { p[e] = exp(logits[e] - mx); z += p[e]; }
    for (int e = 0; e < E; e++) p[e] /= z;
    /* stable insertion sort by descending probability: equal values keep
     * ascending expert order */
    for (int e = 0; e < E; e++) order[e] = e;
    for (int i = 1; i < E; i++) {
        int v = order[i], j = i - 1;
        while (j >= 0 && p[order[j]] < p[v]) { order[j + 1] = order[j]; j--; }
        order[j + 1] = v;
    }
    double s = 0.0;
    for (int i = 0; i < k; i++) s += p[order[i]];
    if (!renorm) s = 1.0;
    for (int i = 0; i < k; i++) { idx[i] = order[i]; w[i] = p[order[i]] / s; }
    free(p);
    free(order);
    return 0;
}

/* ------------------------------ ffn_norm -------------------------------
 * RMSNorm as FUSED_ADD_RMSNORM_KERNEL_SRC in [ferrox gpu.rs] writes it,
 * applied to the hidden state alone (moe_layer in [aprender qwen3 moe] norms
 * `hidden` with ffn_norm before the router):
 *   out[i] = h[i] * w[i] / sqrt(mean_j h[j]^2 + eps).
 * Carried in double. */
int orc_rmsnorm(const float *h, const float *w, int64_t n, double eps, double *out) {
    if (n <= 0 || eps < 0.0) return -1;
    double ss = 0.0;
    for (int64_t i = 0; i < n; i++) ss += (double)h[i] * (double)h[i];
    const double denom = sqrt(ss / (double)n + eps);
    for (int64_t i = 0; i < n; i++) out[i] = (double)h[i] * (double)w[i] / denom;
    return 0;
}

/* silu(g) = g / (1 + e^-g) — SILU_MUL_KERNEL_SRC in [ferrox gpu.rs]. */
static double silu(double g) { return g / (1.0 + exp(-g)); }

/* -------------------------- MoE FFN (per token) --------------------------
 * [aprender qwen3 moe] moe_layer, after ffn_norm (x is the normed input):
 *   logits = R x  (F32 router [E][hidden])
 *   routes = route(logits, k)
 *   for each routed (expert e, weight w) in rank order:
 *       g = G_e x, u = U_e x           (G_e = gate_base + e * stride)
 *       a = silu(g) * u                 (fused_swiglu_into)
 *       b = a * w                       (elementwise_mul_into, route_w)
 *       residual += D_e b               (down GEMV, residual_add_into)
 * All intermediates in double; out[t][i] is the final residual.
 *
 * Tolerance (tol may be NULL): first-order propagation of the per-GEMV
 * bound |gpu - ref| <= 1e-3 * sum_j |w_ij x_j| + 1e-6 through the op order:
 *   tol_i = 1e-3 * sum_s sum_j |D[i,j] b_s[j]|
 *         + sum_s sum_j |D[i,j]| (w_s da_s[j] + dw_s |a_s[j]|)
 *         + 2^-22 |out_i| + 1e-6
 *   da = |silu'(g) u| dg + |silu(g)| du,  dg_j = 1e-3 S^G_j + 1e-6 (du alike)
 *   dw_s = 2 w_s (1 - w_s) max_t dl_t,  dl_t = 1e-3 sum_j |R_tj x_j| + 1e-6
 *   (dw_s/dl_t = w_s (delta_st - w_t) over the k renormalised weights, or
 *   over all E softmax probabilities without renormalisation; either way
 *   |dw_s| <= 2 w_s (1 - w_s) max |dl|).
 * route_idx/route_w (nullable) receive [T][k]; logit_gap (nullable)
 * receives per token the smallest gap among the top k+1 sorted logits
 * divided by max_t sum_j |R_tj x_j| (the ambiguity measure for ties);
 * logits_out / lscale_out (nullable) receive [T][E] logits and per token
 * max_t sum_j |R_tj x_j|. */
typedef struct {
    int32_t hidden, expert_dim, num_experts, top_k;
    int32_t gate_qt, up_qt, down_qt;
    int32_t no_renorm;  /* 1: routing weights are not renormalised (orc_route) */
} orc_moe_shape;

static double dsilu(double g) {
    double s = 1.0 / (1.0 + exp(-g));
    return s * (1.0 + g * (1.0 - s));
}

int orc_moe_ffn(const orc_moe_shape *sh, int64_t T, const float *router, const uint8_t *gate,
                const uint8_t *up, const uint8_t *down, const float *x, const float *residual,
                double *out, double *tol, int32_t *route_idx, double *route_w,
                double *logit_gap, double *logits_out, double *lscale_out) {
    int H = sh->hidden, F = sh->expert_dim, E = sh->num_experts, K = sh->top_k;
    if (H <= 0 || F <= 0 || E <= 0 || K <= 0 || K > E) return -1;
    int64_t grb = orc_row_bytes(sh->gate_qt, H), urb = orc_row_bytes(sh->up_qt, H);
    int64_t drb = orc_row_bytes(sh->down_qt, F);
    if (grb < 0 || urb < 0 || drb < 0) return -1;
    /* ExpertStack::expert: base + e * stride, stride = one [n][k] matrix */
    int64_t gstride = grb * F, ustride = urb * F, dstride = drb * H;

    double *logits = malloc(sizeof(double) * E), *lab = malloc(sizeof(double) * E);
    double *g = malloc(sizeof(double) * F), *u = malloc(sizeof(double) * F);
    double *sg = malloc(sizeof(double) * F), *su = malloc(sizeof(double) * F);
    double *a = malloc(sizeof(double) * F), *da = malloc(sizeof(double) * F);
    float *wrow = malloc(sizeof(float) * (size_t)(H > F ? H : F));
    int32_t *idx = malloc(sizeof(int32_t) * K);
    double *w = malloc(sizeof(double) * K);
    double *acc = malloc(sizeof(double) * H), *t1 = malloc(sizeof(double) * H),
           *t2 = malloc(sizeof(double) * H);
    double *sorted = malloc(sizeof(double) * E);
    if (!logits || !lab || !g || !u || !sg || !su || !a || !da || !wrow || !idx || !w || !acc ||
        !t1 || !t2 || !sorted)
        return -2;

    for (int64_t t = 0; t < T; t++) {
        const float *xt = x + t * H;
        /* router GEMV, F32 rows */
        double dl = 0.0;
        for (int e = 0; e < E; e++) {
            double s = 0.0, sa = 0.0;
            for (int j = 0; j < H; j++) {
                double p = (double)router[(int64_t)e * H + j] * (double)xt[j];
                s += p;
                sa += fabs(p);
            }
            logits[e] = s;
            lab[e] = sa;
            double d = 1e-3 * sa + 1e-6;
            if (d > dl) dl = d;
        }
        orc_route(logits, E, K, !sh->no_renorm, idx, w);
        if (logits_out)
            for (int e = 0; e < E; e++) logits_out[t * E + e] = logits[e];
        if (lscale_out) {
            double mx = 0.0;
            for (int e = 0; e < E; e++) if (lab[e] > mx) mx = lab[e];
            lscale_out[t] = mx;
        }
        if (route_idx)
            for (int s = 0; s < K; s++) route_idx[t * K + s] = idx[s];
        if (route_w)
            for (int s = 0; s < K; s++) route_w[t * K + s] = w[s];
        if (logit_gap) {
            /* logits sorted descending; smallest adjacent gap among the top
             * k+1 (k+1 capped at E) relative to the largest router scale */
            for (int e = 0; e < E; e++) sorted[e] = logits[e];
            for (int i = 1; i < E; i++) {
                double v = sorted[i];
                int j = i - 1;
                while (j >= 0 && sorted[j] < v) { sorted[j + 1] = sorted[j]; j--; }
                sorted[j + 1] = v;
            }
            double mx = 0.0;
            for (int e = 0; e < E; e++) if (lab[e] > mx) mx = lab[e];
            int lim = K + 1 < E ? K + 1 : E;
            double gap = INFINITY;
            for (int i = 0; i + 1 < lim; i++)
                if (sorted[i] - sorted[i + 1] < gap) gap = sorted[i] - sorted[i + 1];
            logit_gap[t] = mx > 0 ? gap / mx : gap;
        }
        for (int i = 0; i < H; i++) { acc[i] = 0.0; t1[i] = 0.0; t2[i] = 0.0; }
        for (int s = 0; s < K; s++) {
            int e = idx[s];
            const uint8_t *G = gate + (int64_t)e * gstride, *U = up + (int64_t)e * ustride;
            const uint8_t *D = down + (int64_t)e * dstride;
            for (int f = 0; f < F; f++) {
                double gs = 0, gsa = 0, us = 0, usa = 0;
                orc_dequant_row(sh->gate_qt, G + f * grb, H, wrow);
                for (int j = 0; j < H; j++) {
                    double p = (double)wrow[j] * (double)xt[j];
                    gs += p; gsa += fabs(p);
                }
                orc_dequant_row(sh->up_qt, U + f * urb, H, wrow);
                for (int j = 0; j < H; j++) {
                    double p = (double)wrow[j] * (double)xt[j];
                    us += p; usa += fabs(p);
                }
                g[f] = gs; u[f] = us; sg[f] = gsa; su[f] = usa;
                a[f] = silu(gs) * us;
                double dg = 1e-3 * gsa + 1e-6, du = 1e-3 * usa + 1e-6;
                da[f] = fabs(dsilu(gs) * us) * dg + fabs(silu(gs)) * du;
            }
            double dws = 2.0 * w[s] * (1.0 - w[s]) * dl;
            for (int i = 0; i < H; i++) {
                orc_dequant_row(sh->down_qt, D + i * drb, F, wrow);
                double ys = 0, ya = 0, yp = 0;
                for (int f = 0; f < F; f++) {
                    double b = a[f] * w[s];
                    double p = (double)wrow[f] * b;
                    ys += p;
                    ya += fabs(p);
                    yp += fabs((double)wrow[f]) * (w[s] * da[f] + dws * fabs(a[f]));
                }
                acc[i] += ys;
                t1[i] += ya;
                t2[i] += yp;
            }
        }
        for (int i = 0; i < H; i++) {
            double o = (double)residual[t * H + i] + acc[i];
            out[t * H + i] = o;
            if (tol) tol[t * H + i] = 1e-3 * t1[i] + t2[i] + ldexp(fabs(o), -22) + 1e-6;
        }
    }
    free(logits); free(lab); free(g); free(u); free(sg); free(su); free(a); free(da);
    free(wrow); free(idx); free(w); free(acc); free(t1); free(t2); free(sorted);
    return 0;
}

/* Dense SwiGLU FFN — [ferrox gpu.rs] launch_dense_ffn_swiglu: gate and up
 * GEMVs on x, silu(gate) * up, down GEMV; the result is added to the
 * residual (the layer's residual update, as in the MoE op order with one
 * expert of weight 1).  tol as for orc_moe_ffn with w = 1, dw = 0. */
int orc_ffn_swiglu(int gate_qt, int up_qt, int down_qt, int64_t H, int64_t F,
                   const uint8_t *gate, const uint8_t *up, const uint8_t *down, const float *x,
                   const float *residual, double *out, double *tol) {
    int64_t grb = orc_row_bytes(gate_qt, H), urb = orc_row_bytes(up_qt, H);
    int64_t drb = orc_row_bytes(down_qt, F);
    if (H <= 0 || F <= 0 || grb < 0 || urb < 0 || drb < 0) return -1;
    double *a = malloc(sizeof(double) * F), *da = malloc(sizeof(double) * F);
    float *wrow = malloc(sizeof(float) * (size_t)(H > F ? H : F));
    if (!a || !da || !wrow) return -2;
    for (int64_t f = 0; f < F; f++) {
        double gs = 0, gsa = 0, us = 0, usa = 0;
        orc_dequant_row(gate_qt, gate + f * grb, H, wrow);
        for (int64_t j = 0; j < H; j++) {
            double p = (double)wrow[j] * (double)x[j];
            gs += p; gsa += fabs(p);
        }
        orc_dequant_row(up_qt, up + f * urb, H, wrow);
        for (int64_t j = 0; j < H; j++) {
            double p = (double)wrow[j] * (double)x[j];
            us += p; usa += fabs(p);
        }
        a[f] = silu(gs) * us;
        da[f] = fabs(dsilu(gs) * us) * (1e-3 * gsa + 1e-6) + fabs(silu(gs)) * (1e-3 * usa + 1e-6);
    }
    for (int64_t i = 0; i < H; i++) {
        orc_dequant_row(down_qt, down + i * drb, F, wrow);
        double ys = 0, ya = 0, yp = 0;
        for (int64_t f = 0; f < F; f++) {
            double p = (double)wrow[f] * a[f];
            ys += p;
            ya += fabs(p);
            yp += fabs((double)wrow[f]) * da[f];
        }
        double o = (double)residual[i] + ys;
        out[i] = o;
        if (tol) tol[i] = 1e-3 * ya + yp + ldexp(fabs(o), -22) + 1e-6;
    }
    free(a); free(da); free(wrow);
    return 0;
}
