/* colimoe_oracle.h — CPU oracle for the quantized MoE feed-forward block.
 *
 * TEST INFRASTRUCTURE ONLY. This is the plain, slow, obviously-correct statement of what the
 * block computes, used to check the CUDA library. Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load it; the product path (libcolimoe) never links or calls
 * it, and the two share no code, headers or tables.
 *
 * Source of the definitions (cited per function in colimoe_oracle.c):
 *   [glm.c]   colibri-strix, c/glm.c @98759bf — QT tensor formats, matmul/matmul_q/matmul_i4/
 *             matmul_i2, sigmoidf/siluf, moe() phases A–E.
 *   [glm.c']  colibri-strix, c/glm.c @97c756a — same file, later revision (matmul_i4_pair).
 *   [metal]   colibri, c/backend_metal.mm @93cde63 — shaders mm_gemv, moe_gemv, moe_silu,
 *             r_router, r_top8, r_top8_par; host moe_submit/moe_finish.
 *   [glm.c, quick-start diff]  colibri, compare main...docs-quickstart — c/glm.c qt_resolve_fmt,
 *             qt_from_disk, expert_load_impl: tensor format 4 (int4 with per-group scales).
 *   [glm.c] also: qrow_i8, dot_i8i8 / dot_i4i8, matmul_q_idot / matmul_i4_idot, matmul_qt —
 *             the IDOT kernels (int8 activations, integer dot), the lossy default of the engine.
 *
 * Precision: dot products accumulate in double and are rounded once to float, then multiplied
 * by the float row scale (the pages apply the scale after the sum). For format 4 the scale
 * changes inside the sum: each group's double partial sum is multiplied by its scale, the
 * products are summed in double and the total is rounded once. Every elementwise step
 * (sigmoid, bias add, renormalisation, SiLU·mul, weighted combine) runs in float, in the order
 * the pages give, because the pages hold those values in float and the router's comparisons
 * decide integers (the selected expert ids) in that precision.
 *
 * Parity status: every function here is pinned by tests against hand-worked examples, closed
 * forms, brute force or invariants (see tests/test_oracle_pins.py). No function is unpinned.
 */
#ifndef COLIMOE_ORACLE_H
#define COLIMOE_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* weight formats of the QT tensor ([glm.c] QT struct): 0 f32, 1 int8, 2 int4, 3 int2, and
 * 4 int4-grouped ([glm.c, quick-start diff] qt_resolve_fmt: int4 bytes, one fp32 scale per group
 * of gs inputs of a row) */
#define ORACLE_FMT_F32  0
#define ORACLE_FMT_INT8 1
#define ORACLE_FMT_INT4 2
#define ORACLE_FMT_INT2 3
#define ORACLE_FMT_INT4G 4

/* bytes of one packed row of In elements */
int64_t oracle_row_bytes(int fmt, int64_t In);

/* dequantised value of element i of one packed row (no scale) */
float oracle_deq(int fmt, const uint8_t *row, int64_t i);

/* y[o] = (float)(sum_i deq(W[o,i]) * v[i]) * s[o]   for o in [0,O); W is [O][row_bytes(In)]
 * (f32 weights: s may be NULL, meaning scale 1). */
void oracle_qgemv(int fmt, const void *W, const float *s, const float *v, int O, int In, float *y);

/* int4-grouped: y[o] = (float)(sum_g s[o*ng + g] * sum_{i in group g} deq(W[o,i]) * v[i]) with
 * ng = ceil(In/gs); s is [O][ng]. */
void oracle_qgemv_grouped(const void *W, const float *s, int gs, const float *v, int O, int In, float *y);

/* IDOT activation quantiser: q[i] = lrintf(x[i] / s) with s = max(max|x| / 127, 1e-12); returns s. */
float oracle_qrow_i8(const float *x, int8_t *q, int n);

/* IDOT GEMV (int8 or int4 weights): y[o] = ((float)sum_i deq(W[o,i]) * q[i]) * s[o] * sx. */
void oracle_qgemv_idot(int fmt, const void *W, const float *s, const int8_t *q, float sx, int O, int In,
                       float *y);

/* Router scores for T tokens: sig[t,e] = sigmoid(x_t . Wr_e), choice[t,e] = sig + bias[e].
 * Returns 0, or -1 if any score or choice is not finite. */
int oracle_router(const float *x, int T, int H, const float *Wr, const float *bias, int E,
                  float *sig, float *choice);

/* Top-K selection with optional TOPK override (ksel, 0 = K) and adaptive top-p (top_p in (0,1),
 * 0 = off), then optional renormalisation and routed scaling.  idx/w are [T,K]; entries beyond
 * keff[t] are set to -1 / 0.  keff may be NULL.  Returns 0 or -1 on bad arguments. */
int oracle_select(const float *sig, const float *choice, int T, int E, int K, int ksel,
                  float top_p, int norm_topk, float routed_scale,
                  int32_t *idx, float *w, int32_t *keff);

/* Token->expert buckets.  counts[E]; offsets[E+1] (exclusive prefix sum); perm[N] lists the
 * assignment ids a = t*K + k (k < keff[t]) grouped by expert, ascending a within a group;
 * N = sum keff.  keff may be NULL (all K).  Returns N, or -1 on an out-of-range index. */
int oracle_buckets(const int32_t *idx, const int32_t *keff, int T, int K, int E,
                   int32_t *counts, int32_t *offsets, int32_t *perm);

/* One SwiGLU expert on one vector: g = gate.x, u = up.x, h = silu(g)*u, y = down.h.
 * gate/up are [Iin][row_bytes(H)], down is [H][row_bytes(Iin)]; gs is the group size of
 * format 4 (its scales are [Iin][ceil(H/gs)] and [H][ceil(Iin/gs)]), ignored otherwise; idot:
 * int8 and int4 products through the IDOT kernels (int8 activations). */
void oracle_expert(int fmt, int gs, int idot, const void *gate_w, const float *gate_s, const void *up_w,
                   const float *up_s, const void *down_w, const float *down_s,
                   int H, int Iin, const float *x, float *y);

/* RMS normalisation of one row, [glm.c] rmsnorm(): ms = sum_i x[i]^2 accumulated in double;
 * r = 1 / sqrtf((float)(ms / D) + eps); out[i] = (x[i] * r) * w[i] in float. out may be x. */
void oracle_rmsnorm(const float *x, const float *w, int D, float eps, float *out);

/* The whole block for T tokens.  Experts are given as host pointer tables of length E.
 * shared_* may be NULL when I_shared == 0.  idx_out/w_out/keff_out optional ([T,K], [T]).
 * Returns 0, or -1 on bad arguments or non-finite router scores. */
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
                       float *out, int32_t *idx_out, float *w_out, int32_t *keff_out);

#ifdef __cplusplus
}
#endif
#endif
