/* colimoe_oracle.c — CPU oracle for the quantized MoE feed-forward block.
 *
 * TEST INFRASTRUCTURE ONLY: loaded by the test suite, the smoke check and the benchmark's
 * CPU-baseline leg; never by the product library. Plain C99, single thread, no intrinsics.
 * See colimoe_oracle.h for the sources cited below and the precision convention.
 */
#include "colimoe_oracle.h"
#include <math.h>
#include <stdlib.h>
#include <string.h>

/* [glm.c] QT struct and qt_bytes(): a row of In elements takes In*4 bytes (f32), In bytes
 * (int8), ceil(In/2) bytes (int4, two per byte) or ceil(In/4) bytes (int2, four per byte). */
int64_t oracle_row_bytes(int fmt, int64_t In) {
    switch (fmt) {
    case ORACLE_FMT_F32:  return In * 4;
    case ORACLE_FMT_INT8: return In;
    case ORACLE_FMT_INT4:
    case ORACLE_FMT_INT4G: return (In + 1) / 2;
    case ORACLE_FMT_INT2: return (In + 3) / 4;
    default: return -1;
    }
}

/* Dequantisation of one element, from the scalar tails of [glm.c] matmul_q (signed byte),
 * matmul_i4 (element i lives in byte i/2: low nibble for even i, high nibble for odd i,
 * value = nibble - 8; an odd last element uses the low nibble only) and matmul_i2 (element i
 * lives in byte i/4 at bit 2*(i%4), value = 2-bit field - 2). */
float oracle_deq(int fmt, const uint8_t *row, int64_t i) {
    switch (fmt) {
    case ORACLE_FMT_F32: {
        float f;
        memcpy(&f, row + 4 * i, 4);
        return f;
    }
    case ORACLE_FMT_INT8:
        return (float)(int8_t)row[i];
    case ORACLE_FMT_INT4:
    case ORACLE_FMT_INT4G: {
        uint8_t b = row[i / 2];
        int nib = (i % 2 == 0) ? (b & 0x0F) : (b >> 4);
        return (float)(nib - 8);
    }
    case ORACLE_FMT_INT2: {
        uint8_t b = row[i / 4];
        int v = (b >> (2 * (i % 4))) & 0x3;
        return (float)(v - 2);
    }
    default:
        return NAN;
    }
}

/* Quantised GEMV, [glm.c] matmul_q / matmul_i4 / matmul_i2 and [metal] mm_gemv:
 * y[o] = (sum_i deq(W[o,i]) * v[i]) * scale[o].  The scale multiplies the finished sum. */
void oracle_qgemv(int fmt, const void *W, const float *s, const float *v, int O, int In, float *y) {
    int64_t rb = oracle_row_bytes(fmt, In);
    for (int o = 0; o < O; o++) {
        const uint8_t *row = (const uint8_t *)W + (int64_t)o * rb;
        double acc = 0.0;
        for (int64_t i = 0; i < In; i++)
            acc += (double)oracle_deq(fmt, row, i) * (double)v[i];
        float a = (float)acc;
        y[o] = s ? a * s[o] : a;
    }
}

/* The int4-grouped tensor ([glm.c, quick-start diff] qt_resolve_fmt, qt_from_disk,
 * expert_load_impl: format 4 keeps the int4 weight bytes and O * ceil(In/gs) fp32 scales, one per
 * group of gs consecutive inputs of a row). The scale changes inside the sum, so it multiplies
 * each group's partial sum: y[o] = sum_g s[o*ng + g] * (sum_{i in group g} deq(W[o,i]) * v[i]),
 * ng = ceil(In/gs), the last group holding the remainder; accumulated in double, rounded once. */
void oracle_qgemv_grouped(const void *W, const float *s, int gs, const float *v, int O, int In, float *y) {
    int64_t rb = oracle_row_bytes(ORACLE_FMT_INT4G, In);
    int ng = (In + gs - 1) / gs;
    for (int o = 0; o < O; o++) {
        const uint8_t *row = (const uint8_t *)W + (int64_t)o * rb;
        double acc = 0.0;
        for (int g = 0; g < ng; g++) {
            double part = 0.0;
            int64_t i1 = (int64_t)(g + 1) * gs < In ? (int64_t)(g + 1) * gs : In;
            for (int64_t i = (int64_t)g * gs; i < i1; i++)
                part += (double)oracle_deq(ORACLE_FMT_INT4G, row, i) * (double)v[i];
            acc += (double)s[(int64_t)o * ng + g] * part;
        }
        y[o] = (float)acc;
    }
}

/* [glm.c] qrow_i8 (the IDOT kernels' activation quantiser): amax = max |x_i| in float,
 * s = amax / 127 (at least 1e-12), q_i = lrintf(x_i * (1 / s)) as a signed byte; returns s. */
float oracle_qrow_i8(const float *x, int8_t *q, int n) {
    float amax = 0.f;
    for (int i = 0; i < n; i++) {
        float a = fabsf(x[i]);
        if (a > amax) amax = a;
    }
    float s = amax / 127.f;
    if (s < 1e-12f) s = 1e-12f;
    float inv = 1.f / s;
    for (int i = 0; i < n; i++) q[i] = (int8_t)lrintf(x[i] * inv);
    return s;
}

/* [glm.c] matmul_q_idot / matmul_i4_idot (dot_i8i8, dot_i4i8): the integer dot of the
 * dequantised weights with the int8 activations, then y[o] = (float)dot * scale[o] * sx,
 * multiplied left to right. int8 and int4 weights only. */
void oracle_qgemv_idot(int fmt, const void *W, const float *s, const int8_t *q, float sx, int O, int In,
                       float *y) {
    int64_t rb = oracle_row_bytes(fmt, In);
    for (int o = 0; o < O; o++) {
        const uint8_t *row = (const uint8_t *)W + (int64_t)o * rb;
        int64_t dot = 0;
        for (int64_t i = 0; i < In; i++) dot += (int64_t)oracle_deq(fmt, row, i) * (int64_t)q[i];
        y[o] = ((float)dot * s[o]) * sx;
    }
}

/* one quantized matrix-vector product: the int4-grouped layout, the IDOT kernels (when idot is
 * set, for int8 and int4 weights only, as glm.c's matmul_qt selects them; int2 and format 4 keep
 * the exact path), or the exact per-row path */
static void matvec(int fmt, int gs, int idot, const void *W, const float *s, const float *v, int O, int In,
                   float *y) {
    if (fmt == ORACLE_FMT_INT4G) {
        oracle_qgemv_grouped(W, s, gs, v, O, In, y);
    } else if (idot && (fmt == ORACLE_FMT_INT8 || fmt == ORACLE_FMT_INT4)) {
        int8_t *q = (int8_t *)malloc((size_t)In);
        float sx = oracle_qrow_i8(v, q, In);
        oracle_qgemv_idot(fmt, W, s, q, sx, O, In, y);
        free(q);
    } else {
        oracle_qgemv(fmt, W, s, v, O, In, y);
    }
}

/* [glm.c] sigmoidf and siluf */
static float sigmoid_f(float z) { return 1.f / (1.f + expf(-z)); }
static float silu_f(float z) { return z / (1.f + expf(-z)); }

/* Phase A of [glm.c] moe(), first half, and [metal] r_router: logit = x . Wr_e in full
 * precision (the f32 matmul), sig = sigmoid(logit), choice = sig + bias[e]. */
int oracle_router(const float *x, int T, int H, const float *Wr, const float *bias, int E,
                  float *sig, float *choice) {
    if (T < 0 || H < 1 || E < 1) return -1;
    for (int t = 0; t < T; t++) {
        float *lg = (float *)malloc(sizeof(float) * (size_t)E);
        oracle_qgemv(ORACLE_FMT_F32, Wr, NULL, x + (int64_t)t * H, E, H, lg);
        for (int e = 0; e < E; e++) {
            float s = sigmoid_f(lg[e]);
            float c = s + bias[e];
            sig[(int64_t)t * E + e] = s;
            choice[(int64_t)t * E + e] = c;
            if (!isfinite(s) || !isfinite(c)) { free(lg); return -1; }
        }
        free(lg);
    }
    return 0;
}

/* Phase A of [glm.c] moe(), second half, and [metal] r_top8:
 *  1. Greedy selection of Ksel experts: each round scans e = 0..E-1 and keeps the first
 *     not-yet-taken expert whose choice is strictly greater than the best so far, so equal
 *     choices go to the lower expert index.  w[k] = sig[idx[k]] (the bias only steers the
 *     selection).  Ksel = min(ksel, K) when the TOPK override is set, else K.
 *  2. Adaptive top-p (TOPP), when 0 < top_p < 1: insertion-sort the selected pairs by w,
 *     descending (equal w keep their order), tot = 1e-20 + sum w, and keep the shortest prefix
 *     whose running sum reaches top_p * tot.
 *  3. If norm_topk: w /= (sum of the kept w + 1e-20).  4. w *= routed_scale. */
int oracle_select(const float *sig, const float *choice, int T, int E, int K, int ksel,
                  float top_p, int norm_topk, float routed_scale,
                  int32_t *idx, float *w, int32_t *keff) {
    if (T < 0 || E < 1 || K < 1 || K > E || ksel < 0) return -1;
    int Ksel = (ksel > 0 && ksel < K) ? ksel : K;
    for (int t = 0; t < T; t++) {
        const float *sg = sig + (int64_t)t * E, *ch = choice + (int64_t)t * E;
        int32_t *id = idx + (int64_t)t * K;
        float *ww = w + (int64_t)t * K;
        for (int k = 0; k < K; k++) { id[k] = -1; ww[k] = 0.f; }
        for (int k = 0; k < Ksel; k++) {
            int best = -1;
            float bv = -1e30f;
            for (int e = 0; e < E; e++) {
                int taken = 0;
                for (int j = 0; j < k; j++)
                    if (id[j] == e) { taken = 1; break; }
                if (!taken && ch[e] > bv) { bv = ch[e]; best = e; }
            }
            if (best < 0) return -1;
            id[k] = best;
            ww[k] = sg[best];
        }
        int Ke = Ksel;
        if (top_p > 0.f && top_p < 1.f) {
            for (int a = 1; a < Ksel; a++) {
                int ia = id[a];
                float wa = ww[a];
                int b = a - 1;
                while (b >= 0 && ww[b] < wa) { ww[b + 1] = ww[b]; id[b + 1] = id[b]; b--; }
                ww[b + 1] = wa;
                id[b + 1] = ia;
            }
            float tot = 1e-20f;
            for (int k = 0; k < Ksel; k++) tot += ww[k];
            float cum = 0.f;
            for (int k = 0; k < Ksel; k++) {
                cum += ww[k];
                if (cum >= top_p * tot) { Ke = k + 1; break; }
            }
            for (int k = Ke; k < Ksel; k++) { id[k] = -1; ww[k] = 0.f; }
        }
        if (norm_topk) {
            float sm = 0.f;
            for (int k = 0; k < Ke; k++) sm += ww[k];
            sm += 1e-20f;
            for (int k = 0; k < Ke; k++) ww[k] /= sm;
        }
        for (int k = 0; k < Ke; k++) ww[k] *= routed_scale;
        if (keff) keff[t] = Ke;
    }
    return 0;
}

/* Phase B of [glm.c] moe() (batch union: each expert is read once for all rows that use it)
 * and the row gather of phases C/D (rows of one expert in token order), restated as a
 * counting sort of the assignment ids a = t*K + k by expert, stable in a. */
int oracle_buckets(const int32_t *idx, const int32_t *keff, int T, int K, int E,
                   int32_t *counts, int32_t *offsets, int32_t *perm) {
    if (T < 0 || K < 1 || E < 1) return -1;
    for (int e = 0; e < E; e++) counts[e] = 0;
    for (int t = 0; t < T; t++) {
        int ke = keff ? keff[t] : K;
        for (int k = 0; k < ke; k++) {
            int e = idx[(int64_t)t * K + k];
            if (e < 0 || e >= E) return -1;
            counts[e]++;
        }
    }
    offsets[0] = 0;
    for (int e = 0; e < E; e++) offsets[e + 1] = offsets[e] + counts[e];
    int32_t *fill = (int32_t *)calloc((size_t)E, sizeof(int32_t));
    for (int t = 0; t < T; t++) {
        int ke = keff ? keff[t] : K;
        for (int k = 0; k < ke; k++) {
            int e = idx[(int64_t)t * K + k];
            perm[offsets[e] + fill[e]] = t * K + k;
            fill[e]++;
        }
    }
    free(fill);
    return offsets[E];
}

/* Phases C/D of [glm.c] moe() for one row (also [metal] moe_gemv + moe_silu):
 * g = gate.x, u = up.x, h = silu(g) * u, y = down.h. */
void oracle_expert(int fmt, int gs, int idot, const void *gate_w, const float *gate_s, const void *up_w,
                   const float *up_s, const void *down_w, const float *down_s,
                   int H, int Iin, const float *x, float *y) {
    float *g = (float *)malloc(sizeof(float) * (size_t)Iin);
    float *u = (float *)malloc(sizeof(float) * (size_t)Iin);
    matvec(fmt, gs, idot, gate_w, gate_s, x, Iin, H, g);
    matvec(fmt, gs, idot, up_w, up_s, x, Iin, H, u);
    for (int j = 0; j < Iin; j++) g[j] = silu_f(g[j]) * u[j];
    matvec(fmt, gs, idot, down_w, down_s, g, H, Iin, y);
    free(g);
    free(u);
}

/* [glm.c] rmsnorm(), the normalisation that feeds moe() in the layer forward (post_ln after
 * the attention residual): the mean square in double, its reciprocal root in float, then each
 * element times r times its weight, in that order. */
void oracle_rmsnorm(const float *x, const float *w, int D, float eps, float *out) {
    double ms = 0.0;
    for (int i = 0; i < D; i++) ms += (double)x[i] * x[i];
    const float r = 1.f / sqrtf((float)(ms / D) + eps);
    for (int i = 0; i < D; i++) out[i] = x[i] * r * w[i];
}

/* The block, [glm.c] moe(): per token, route (phase A), run each kept routed expert in
 * selection order and accumulate out += w * y (phases C/D), then add the shared expert with
 * weight 1 (phase E).  Tokens are independent rows, so the per-token loop gives the same
 * values as the batch-union loop up to the order of the routed additions: selection order
 * is used here. */
int oracle_moe_forward(int T, int H, int I, int E, int K, int ksel, float top_p,
                       int norm_topk, float routed_scale, int routed_fmt,
                       const float *x, const float *Wr, const float *bias,
                       const void *const *gate_w, const float *const *gate_s,
                       const void *const *up_w, const float *const *up_s,
                       const void *const *down_w, const float *const *down_s,
                       int I_shared, int shared_fmt, int group_size, int idot,
                       const void *sh_gate_w, const float *sh_gate_s,
                       const void *sh_up_w, const float *sh_up_s,
                       const void *sh_down_w, const float *sh_down_s,
                       float *out, int32_t *idx_out, float *w_out, int32_t *keff_out) {
    if (T < 0 || H < 1 || I < 1 || E < 1 || K < 1 || K > E || I_shared < 0) return -1;
    if (oracle_row_bytes(routed_fmt, 1) < 0) return -1;
    if (I_shared > 0 && oracle_row_bytes(shared_fmt, 1) < 0) return -1;
    if ((routed_fmt == ORACLE_FMT_INT4G || (I_shared > 0 && shared_fmt == ORACLE_FMT_INT4G)) && group_size < 1)
        return -1;
    float *sig = (float *)malloc(sizeof(float) * (size_t)E);
    float *ch = (float *)malloc(sizeof(float) * (size_t)E);
    int32_t *id = (int32_t *)malloc(sizeof(int32_t) * (size_t)K);
    float *ww = (float *)malloc(sizeof(float) * (size_t)K);
    float *y = (float *)malloc(sizeof(float) * (size_t)H);
    int rc = 0;
    for (int t = 0; t < T && rc == 0; t++) {
        const float *xt = x + (int64_t)t * H;
        float *ot = out + (int64_t)t * H;
        int32_t ke = 0;
        if (oracle_router(xt, 1, H, Wr, bias, E, sig, ch) != 0 ||
            oracle_select(sig, ch, 1, E, K, ksel, top_p, norm_topk, routed_scale, id, ww, &ke) != 0) {
            rc = -1;
            break;
        }
        for (int d = 0; d < H; d++) ot[d] = 0.f;
        for (int k = 0; k < ke; k++) {
            int e = id[k];
            oracle_expert(routed_fmt, group_size, idot, gate_w[e], gate_s[e], up_w[e], up_s[e], down_w[e],
                          down_s[e], H, I, xt, y);
            for (int d = 0; d < H; d++) ot[d] += ww[k] * y[d];
        }
        if (I_shared > 0) {
            oracle_expert(shared_fmt, group_size, idot, sh_gate_w, sh_gate_s, sh_up_w, sh_up_s, sh_down_w,
                          sh_down_s, H, I_shared, xt, y);
            for (int d = 0; d < H; d++) ot[d] += y[d];
        }
        if (idx_out) memcpy(idx_out + (int64_t)t * K, id, sizeof(int32_t) * (size_t)K);
        if (w_out) memcpy(w_out + (int64_t)t * K, ww, sizeof(float) * (size_t)K);
        if (keff_out) keff_out[t] = ke;
    }
    free(sig);
    free(ch);
    free(id);
    free(ww);
    free(y);
    return rc;
}
