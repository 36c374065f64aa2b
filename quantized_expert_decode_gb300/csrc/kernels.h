// kernels.h — host-side launchers of libcolimoe's kernels (internal, not part of the ABI).
#pragma once

#include "common.cuh"

namespace colimoe {

// Everything the expert kernels need to find their work; device pointers into the workspace.
struct ExpertWork {
    const coli_moe_expert *experts;  // device [E]
    coli_moe_expert shared;          // by value; unused when I_shared == 0
    const float *x;                  // [T][H]
    const int32_t *counts;           // [E]
    const int32_t *offsets;          // [E+1]
    const int32_t *perm;             // [T*K]
    const int32_t *act;              // [E]
    const int32_t *meta;             // [0] = U
    float *h;                        // [(T*K + T)][ldh]
    float *y;                        // [(T*K + T)][H]
    int32_t *err;
    int T, H, I, E, K, I_shared, routed_fmt, shared_fmt;
    int ldh;                         // row stride of h in floats (max(I, I_shared))
    int slots;                       // grid.y: max active routed experts + (shared ? 1 : 0)
    int group_size;                  // inputs per scale of COLI_FMT_INT4G experts
    int idot;                        // int8 and int4 experts through the IDOT kernels
};

// ---------------------------------------------------------------- decode.cu
constexpr int kDecMaxT = 64;              // the persistent decode kernel serves T <= 64
constexpr int kTokSlices = 32;            // T > 8: router partial slices the token CTAs sum

// Counters of one decode call (zeroed before each launch; err stays the first word, which is
// also the workspace error word read by coli_moe_check).
struct DecCtrl {
    int err, router_done, dn_done;
    int gu_all;                        // single-token kernel: finished gate/up units, all slots
    int q_b, q_c, q_d;                 // token-group kernel: next chunk of phases B, C, D
    int routed_done;                   // token-group kernel, T > 8: tokens routed by their CTA
    int pad[8];
    unsigned long long call;           // single-token kernel: id of the call whose counters these are
    int hmax[kMaxK + 1];               // single-token kernel: max |h| per slot (float bits)
    int gu_done[kMaxE + 1];            // finished gate/up units per slot (shared: index kMaxE)
};

struct DecParams {
    const float *x, *Wr, *bias;
    // the layer tail: out = resid + block; the single-token kernel also normalises resid itself
    // (x = rmsnorm(resid) * norm_w); the other kernels take x already normalised
    const float *resid, *norm_w;
    float eps;
    const coli_moe_expert *experts;
    coli_moe_expert shared;
    float *out;
    float *part;               // router partial logits [nks][T][E]
    float *sig, *choice, *w;
    int32_t *idx, *keff, *counts, *offsets, *perm, *pos, *act;
    float *h, *y;
    DecCtrl *ctrl;
    int T, H, I, E, K, Is, rfmt, sfmt, Ksel, norm_topk;
    int rgs, sgs;              // inputs per scale of int4-grouped routed / shared weights (0: per-row scales)
    int rq8, sq8;              // single-token kernel: routed / shared products on int8 activations (IDOT)
    float top_p, rscale;
    int ldh;
    int NV, xs_stride, xs_bytes, rt_bytes;
    int R, route_only;         // router items; route_only: logits come from a separate launch
    int neb, nks, rks_floats;  // router expert blocks, k-slices, floats per k-slice
    int groups_sh, G_sh;       // shared expert token groups and gate/up units
    // single-token kernel (decode1.cu): shared-memory offsets (activation limbs, routing
    // scratch, per-CTA down results, expert table, bias, end), the bytes of one slot's staged h,
    // and the row pairs of the down phase per CTA at most
    int single, d1_act_off, d1_rsc_off, d1_ylo_off, d1_tab_off, d1_bias_off, d1_xf_off, d1_end, d1_hs, d1_pairs;
    unsigned long long call_id;  // single-token kernel: unique per call (counters reset in-kernel)
};

bool decode_plan(const coli_moe_desc &d, DecParams &P, int grid);
bool decode_supported(const coli_moe_desc &d);
size_t decode_smem_bytes(const DecParams &P);
int decode_ctas_per_sm(const DecParams &P);
cudaError_t launch_decode(const DecParams &P, int grid, cudaStream_t s);

// decode1.cu: the single-token kernel
bool decode1_plan(const coli_moe_desc &d, DecParams &P, int grid);
int decode1_ctas_per_sm(const DecParams &P);
cudaError_t launch_decode1(const DecParams &P, int grid, cudaStream_t s);

// prefill.cu: the tensor-core expert GEMMs for T > 64
struct PrefillWork {
    const coli_moe_expert *experts;  // device [E]
    coli_moe_expert shared;
    const float *x;
    const int32_t *counts, *offsets, *perm;
    uint16_t *xb, *hb;               // f16 activations (row p scaled by 2^xe[p]) / bf16 h (block-permuted K order)
    int32_t *xe;                     // [T*K + T] exponents of the activation rows' scales
    void *tmaps;                     // [E + 1][3] tensor maps of the expert matrices (workspace)
    float *y;
    int32_t *err;
    int T, H, I, E, K, I_shared, routed_fmt, shared_fmt, ldh, grid;
};
bool prefill_supported(const coli_moe_desc &d);
// part 0: activation pre-pass + gate/up GEMM; part 1: down GEMM
cudaError_t launch_prefill(const PrefillWork &w, int part, cudaStream_t s);

// router.cu
cudaError_t launch_router_partial(const float *x, const float *W_r, float *part, int T, int H,
                                  int E, int splits, cudaStream_t s);
cudaError_t launch_select(const float *part, int splits, const float *bias, int T, int E, int K,
                          int ksel, float top_p, int norm_topk, float routed_scale, float *sig,
                          float *choice, int32_t *idx, float *w, int32_t *keff, int32_t *err,
                          cudaStream_t s);
cudaError_t launch_bucket(const int32_t *idx, const int32_t *keff, int T, int K, int E,
                          int32_t *counts, int32_t *offsets, int32_t *perm, int32_t *pos,
                          int32_t *act, int32_t *meta, int32_t *err, cudaStream_t s);

// expert.cu
cudaError_t launch_gateup(const ExpertWork &w, cudaStream_t s);
cudaError_t launch_down(const ExpertWork &w, cudaStream_t s);
// resid: the layer tail's residual added to the block (NULL: the block alone)
cudaError_t launch_combine(const float *y, const float *wts, const int32_t *keff,
                           const int32_t *pos, int T, int H, int K, int has_shared, const float *resid,
                           float *out, cudaStream_t s);
// xn[t] = rmsnorm(resid[t]) * w for T rows of H (H a multiple of 4)
cudaError_t launch_rmsnorm(const float *resid, const float *w, float eps, int T, int H, float *xn, cudaStream_t s);
// gs: inputs per scale when fmt is COLI_FMT_INT4G (sc is then [O][ceil(In/gs)]), else unused
cudaError_t launch_qgemv(int fmt, const void *W, const float *sc, int gs, const float *x, float *y, int O,
                         int In, int T, cudaStream_t st);

}  // namespace colimoe
