// decode1.cu — the whole MoE block for ONE token (T = 1) in one persistent launch.
//
// The single-token call is the decode step of the engine (colibri-strix c/glm.c @98759bf
// moe() with S = 1; the Metal path's moe_gemv). Its work is small per CTA, so the kernel is
// built around the dependent memory round trips between its phases rather than around tiling:
// every phase issues its independent loads together. Phases, split statically over the CTAs
// (two per SM, cooperative launch):
//   A  router items: partial logits of 32 experts over one slice of H (r_router shader), the
//      slice's router rows and x in flight together
//   X  the expert table and the bias copied into shared memory; the token's x in 24-bit block
//      fixed point (idot.cuh), in the layout of each weight format the block uses (int8 bytes
//      instead for the sides that run on int8 activations, IDOT)
//   B  shared expert gate/up rows (independent of routing), spread over every CTA: here only
//      when the shared expert's walk differs from the routed experts' (another format); else
//      its units follow each CTA's routed units in phase C, one stream of loads through both
//   R  routing by EVERY CTA from the partial logits: logits summed in a fixed order, sigmoid,
//      bias, greedy top-K with ties to the lower index (select.cuh), TOPK/TOPP, renorm, routed
//      scale. The kept experts become slots 0..U-1 in ascending id order; the shared expert is
//      slot U. Their weight pointers come from the shared-memory copy of the table.
//   C  routed gate/up units (rows j of gate and up of one slot): h = silu(gate.x * s_g) *
//      (up.x * s_u); each CTA keeps the largest |h| of every slot it wrote, the exponent of the
//      down step's fixed point (or the scale of its int8 quantisation); the CTA then raises
//      one counter.
//   D  once every gate/up unit is in (that counter): (slot, 4-row group) units split
//      slot-major over the CTAs, so each stages only the one or two h vectors its units read
//      (h and the slots' maxima in one round trip); y rows go to the workspace. Routed and
//      shared units are one stream when their rows have the same walk and length.
//   E  once every down row is in (one counter): each CTA's rows of
//      out[d] = sum_k w_k y[pos_k][d] in selection order, + y[U][d]  (moe() phases C/D/E)
// Warps walk their gate/up and down units without CTA barriers. Every wait is bounded.
// Instances: <routed format, shared format, GRP>, GRP marking int4-grouped sides (a scale per
// group of inputs, applied per 16-byte chunk) and sides on int8 activations (IDOT).
#include <algorithm>

#include "decode_parts.cuh"
#include "select.cuh"

namespace colimoe {

namespace {

struct Rec {  // one expert's weight pointers
    const uint8_t *gw, *uw, *dw;
    const float *gs, *us, *ds;
};

constexpr int kShSlot = kMaxK;  // index of the shared expert in rec[] and hmax[]
constexpr int kInfl1 = 8;       // 16-byte loads in flight per lane in the streaming phases
constexpr int kRtQ = 4;         // float4 steps per lane and router row held at once
constexpr int kHB = 2;          // staged h items (16 elements each) per thread per round trip
constexpr int kMaxSlices = 16;  // router slices of H per expert block
constexpr int kGuRows = 4;      // rows per gate/up unit: gate j, up j, gate j + 1, up j + 1 (or 2)
constexpr bool kOnce = false;   // true: expert rows stream with an evict-first L2 policy

struct D1S {  // the fixed part of the CTA's shared memory
    Rec rec[kMaxK + 1];
    int slot_e[kMaxK];
    int pos[kMaxK];     // slot of selection k, -1 beyond keff
    float w[kMaxK];     // kept routing weights, 0 beyond keff
    int sel_i[kMaxK];
    int ncand, nok;     // selection: candidates, selectable experts
    int U;
    int xshift;
    float xinv;
    int hshift[kMaxK + 1];  // per slot (shared: at U) in the down phase
    float hinv[kMaxK + 1];
    float hamax[kMaxK + 1]; // max |h| of each staged slot (the int8 quantisation's amax)
    float hsq[kMaxK + 1];   // ... and its int8 scale
    float xsq;              // the int8 scale of x
    int hmax[kMaxK + 1];    // this CTA's max |h| per slot (float bits); shared at kShSlot
    float redf[kNW];
    double redd[kNW];
};

__device__ __forceinline__ Rec rec_of(const coli_moe_expert &e) {
    Rec r;
    r.gw = static_cast<const uint8_t *>(e.gate_w);
    r.uw = static_cast<const uint8_t *>(e.up_w);
    r.dw = static_cast<const uint8_t *>(e.down_w);
    r.gs = e.gate_s;
    r.us = e.up_s;
    r.ds = e.down_s;
    return r;
}


// A: partial logits of 32 experts (4 per warp) over one slice of H. Each lane holds up to kRtQ
// float4 steps of the four router rows and of x, so a slice of up to 512 floats is one round
// trip; the sums run in the same order for every expert (equal rows give equal partials).
// xsrc: x in global memory, or the normalised row in shared memory (the layer tail)
__device__ __noinline__ void router_item1(const DecParams &P, int item, const float *xsrc) {
    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
    const int eb = item % P.neb, ks = item / P.neb;
    const int kb = ks * P.rks_floats, ke = min(P.H, kb + P.rks_floats), nq = (ke - kb) / 4;
    const float *xs = xsrc + kb;
    const float *wr[4];
#pragma unroll
    for (int r = 0; r < 4; r++) wr[r] = P.Wr + (size_t)min(eb * kRtE + warp * 4 + r, P.E - 1) * P.H + kb;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    const uint64_t pol = policy_evict_first();
    for (int q0 = 0; q0 < nq; q0 += kWarp * kRtQ) {
        uint4 wv[4][kRtQ];
        float4 xv[kRtQ];
#pragma unroll
        for (int j = 0; j < kRtQ; j++) {
            const int q = q0 + lane + kWarp * j;
            const bool in = q < nq;
#pragma unroll
            for (int r = 0; r < 4; r++) wv[r][j] = in ? ld_once_16(wr[r] + 4 * q, pol) : make_uint4(0, 0, 0, 0);
            xv[j] = in ? reinterpret_cast<const float4 *>(xs)[q] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int j = 0; j < kRtQ; j++)
#pragma unroll
            for (int r = 0; r < 4; r++) {
                float a = acc[r];
                a = fmaf(__uint_as_float(wv[r][j].x), xv[j].x, a);
                a = fmaf(__uint_as_float(wv[r][j].y), xv[j].y, a);
                a = fmaf(__uint_as_float(wv[r][j].z), xv[j].z, a);
                a = fmaf(__uint_as_float(wv[r][j].w), xv[j].w, a);
                acc[r] = a;
            }
    }
#pragma unroll
    for (int r = 0; r < 4; r++) {
        float s = acc[r];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(kFull, s, o);
        const int er = eb * kRtE + warp * 4 + r;
        if (lane == 0 && er < P.E) P.part[(size_t)ks * P.E + er] = s;
    }
}

// X: x -> limbs in the routed layout (and the shared one when it differs). A thread's items
// (16 elements each) are loaded once and kept in registers across the max reduction when it
// has at most two of them (H <= 8192); larger H reloads them for the conversion.
template <int FMT>
__device__ __forceinline__ void limbs_from_regs(const float4 (&v)[4], uint8_t *xq, int CPR, int p,
                                                const FixedScale &fx) {
    using G = QGeom<FMT>;
    using I = IQ<FMT>;
    const int c = p % CPR, ss = p / CPR;
    int X[16];
#pragma unroll
    for (int k = 0; k < 4; k++) {
        X[4 * k + 0] = fx(v[k].x);
        X[4 * k + 1] = fx(v[k].y);
        X[4 * k + 2] = fx(v[k].z);
        X[4 * k + 3] = fx(v[k].w);
    }
    uint32_t o[12];
#pragma unroll
    for (int wl = 0; wl < I::WPSS; wl++)
#pragma unroll
        for (int g = 0; g < I::NGW; g++) {
            const int e0 = wl * G::EPW + g, u = (wl * I::NGW + g) * 3;
            pack_limbs(X[e0], X[e0 + I::NGW], X[e0 + 2 * I::NGW], X[e0 + 3 * I::NGW], o[u], o[u + 1], o[u + 2]);
        }
    uint4 *xq4 = reinterpret_cast<uint4 *>(xq);
#pragma unroll
    for (int j = 0; j < 3; j++)
        xq4[(ss * 3 + j) * CPR + c] = make_uint4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
}

// RQ / SQ: the routed / shared side takes int8 bytes (the IDOT quantisation) instead of limbs
template <int RF, int SF, bool RQ, bool SQ>
__device__ void stage_x(const DecParams &P, const float *xsrc, uint8_t *xq_r, uint8_t *xq_s, bool two, D1S &m) {
    const int tid = threadIdx.x, lane = tid % kWarp, warp = tid / kWarp;
    const int n16 = P.H / 16;  // 16-element groups; group q is item q of every layout ordering
    const float4 *x4 = reinterpret_cast<const float4 *>(xsrc);
    const bool in_regs = n16 <= 2 * kNT;
    float4 v[2][4];
    float mx = 0.f;
    for (int q0 = tid; q0 < n16; q0 += 2 * kNT) {
#pragma unroll
        for (int j = 0; j < 2; j++) {
            const int q = q0 + j * kNT;
            if (q < n16)
#pragma unroll
                for (int k = 0; k < 4; k++) v[j][k] = x4[4 * q + k];
        }
#pragma unroll
        for (int j = 0; j < 2; j++)
            if (q0 + j * kNT < n16)
#pragma unroll
                for (int k = 0; k < 4; k++)
                    mx = fmaxf(mx, fmaxf(fmaxf(fabsf(v[j][k].x), fabsf(v[j][k].y)),
                                         fmaxf(fabsf(v[j][k].z), fabsf(v[j][k].w))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
    if (lane == 0) m.redf[warp] = mx;
    __syncthreads();
    mx = m.redf[0];
#pragma unroll
    for (int w = 1; w < kNW; w++) mx = fmaxf(mx, m.redf[w]);
    const int s = fixed_shift(mx);
    const FixedScale fx(s);
    const Q8Scale qs(mx);
    // the 16 elements of group q are item q of a layout whose items are (ss, c) with
    // p = ss * CPR + c covering elements c * EPC + ss * 16: map q to that p
    auto item_of = [&](int fmt_epc, int fmt_nss, int q) {
        const int cpr = P.H / fmt_epc;
        const int c = q / fmt_nss, ss = q % fmt_nss;
        return ss * cpr + c;
    };
    for (int q0 = tid; q0 < n16; q0 += 2 * kNT) {
        if (!in_regs) {
#pragma unroll
            for (int j = 0; j < 2; j++) {
                const int q = q0 + j * kNT;
                if (q < n16)
#pragma unroll
                    for (int k = 0; k < 4; k++) v[j][k] = x4[4 * q + k];
            }
        }
#pragma unroll
        for (int j = 0; j < 2; j++) {
            const int q = q0 + j * kNT;
            if (q < n16) {
                const int pr = item_of(QGeom<RF>::EPC, IQ<RF>::NSS, q);
                if constexpr (RQ) q8_from_regs<RF>(v[j], xq_r, P.H / QGeom<RF>::EPC, pr, qs);
                else limbs_from_regs<RF>(v[j], xq_r, P.H / QGeom<RF>::EPC, pr, fx);
                if (two) {
                    const int ps = item_of(QGeom<SF>::EPC, IQ<SF>::NSS, q);
                    if constexpr (SQ) q8_from_regs<SF>(v[j], xq_s, P.H / QGeom<SF>::EPC, ps, qs);
                    else limbs_from_regs<SF>(v[j], xq_s, P.H / QGeom<SF>::EPC, ps, fx);
                }
            }
        }
    }
    if (tid == 0) {
        m.xshift = s;
        m.xinv = ldexpf(1.f, -s);
        m.xsq = qs.s;
    }
    __syncthreads();
}

// The layer tail's normalised row, by this CTA into shared memory (xf, H floats):
// xf = (resid * r) * norm_w with r = 1 / sqrtf(mean square of resid + eps), the squares summed
// in double (per thread in a fixed stride order, then over the warps in a fixed order), as
// glm.c's rmsnorm computes the post-attention norm that feeds moe().
__device__ __noinline__ void stage_xn(const DecParams &P, float *xf, D1S &m) {
    const int tid = threadIdx.x, lane = tid % kWarp, warp = tid / kWarp;
    const float4 *r4 = reinterpret_cast<const float4 *>(P.resid);
    const float4 *w4 = reinterpret_cast<const float4 *>(P.norm_w);
    double ms = 0.0;
    for (int q = tid; q < P.H / 4; q += kNT) {
        const float4 v = __ldg(r4 + q);
        ms += (double)v.x * v.x;
        ms += (double)v.y * v.y;
        ms += (double)v.z * v.z;
        ms += (double)v.w * v.w;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ms += __shfl_xor_sync(kFull, ms, o);
    if (lane == 0) m.redd[warp] = ms;
    __syncthreads();
    double tot = 0.0;
#pragma unroll
    for (int k = 0; k < kNW; k++) tot += m.redd[k];
    const float r = 1.f / sqrtf((float)(tot / P.H) + P.eps);
    float4 *o4 = reinterpret_cast<float4 *>(xf);
    for (int q = tid; q < P.H / 4; q += kNT) {
        const float4 v = __ldg(r4 + q), g = __ldg(w4 + q);
        o4[q] = make_float4(v.x * r * g.x, v.y * r * g.y, v.z * r * g.z, v.w * r * g.w);
    }
    __syncthreads();
}

// R: the routing of the token by this CTA (sg/ch: shared scratch of sel_padded(E) floats each,
// cand: sel_cand_cap(E, Ksel) float2; bias and tab: the bias and the expert table, in shared
// memory when they fit). Inlined into the kernel: its code then follows the wait before it.
__device__ __forceinline__ void route1(const DecParams &P, D1S &m, float *sg, float *ch, float2 *cand,
                                       const float *bias, const coli_moe_expert *tab) {
    const int tid = threadIdx.x, lane = tid % kWarp, warp = tid / kWarp;
    const bool out = blockIdx.x == 0;
    const int E = P.E, Ep = sel_padded(E);
    // 1. logits (fixed-order sum of the partial slices) -> sigmoid scores and choices
    for (int e = tid; e < Ep; e += kNT) {
        if (e < E) {
            float a[kMaxSlices];
#pragma unroll
            for (int k = 0; k < kMaxSlices; k++)
                if (k < P.nks) a[k] = __ldcg(P.part + (size_t)k * E + e);
            float lg = 0.f;
#pragma unroll
            for (int k = 0; k < kMaxSlices; k++)
                if (k < P.nks) lg += a[k];
            const float sv = 1.f / (1.f + expf(-lg));
            const float cv = sv + bias[e];
            sg[e] = sv;
            ch[e] = cv;
            if (out) {
                P.sig[e] = sv;
                P.choice[e] = cv;
            }
        } else {
            sg[e] = 0.f;
            ch[e] = -INFINITY;
        }
    }
    if (tid == 0) m.ncand = m.nok = 0;
    __syncthreads();
    // 2. the picks, by the whole CTA (select.cuh)
    sel_topk_cta(ch, E, P.Ksel, cand, &m.ncand, &m.nok, m.sel_i);
    // 3. the kept experts, their weights and slots (warp 0, one pick per lane)
    if (warp == 0) {
        const int K = P.K, Ksel = P.Ksel;
        const int nsel = min(m.nok, Ksel);
        if (nsel < Ksel && out && lane == 0) flag_error(P.ctrl, kErrNoCandidate);
        const int pick = lane < nsel ? m.sel_i[lane] : -1;
        const SelKept kp = sel_finish_warp(nsel, pick, lane < nsel ? sg[pick] : 0.f, P.top_p, P.norm_topk, P.rscale);
        const int Ke = kp.ke, id = kp.id;
        const bool kept = lane < Ke;
        coli_moe_expert ex{};
        if (kept) ex = tab[id];
        int slot = 0;
        for (int k = 0; k < Ke; k++) slot += __shfl_sync(kFull, id, k) < id;
        if (lane < K) {
            m.w[lane] = kp.w;
            m.pos[lane] = kept ? slot : -1;
            if (kept) {
                m.slot_e[slot] = id;
                if (bad16(ex.gate_w) || bad16(ex.up_w) || bad16(ex.down_w)) flag_error(P.ctrl, kErrBadExpert);
                m.rec[slot] = rec_of(ex);
            }
            if (out) {
                P.idx[lane] = id;
                P.w[lane] = kp.w;
                P.pos[lane] = kept ? slot : -1;
                if (kept) {
                    P.perm[slot] = lane;
                    P.act[slot] = id;
                }
            }
        }
        if (lane == 0) {
            m.U = Ke;
            if (out) P.keff[0] = Ke;
        }
    }
    __syncthreads();
    // 4. bucket counts (CTA 0 only; nothing in this CTA reads them)
    if (out) {
        const int U = m.U;
        for (int e = tid; e < E; e += kNT) {
            int cnt = 0, o = 0;
            for (int u = 0; u < U; u++) {
                const int se = m.slot_e[u];
                cnt += se == e;
                o += se < e;
            }
            P.counts[e] = cnt;
            P.offsets[e] = o;
        }
        if (tid == 0) P.offsets[E] = U;
    }
}

// The CTA's gate/up units: routed units [rb0, re0) of the slot-major routed space (kGuRows / 2
// row pairs j, j + 1 .. of gate and of up of one slot per unit), then the shared expert's units
// [sb0, se0). Warps take the combined list round-robin, with no barriers, so one stream of loads
// runs through both when the formats agree.
// list entry w -> slot (kShSlot for the shared expert) and first row j; per: units per routed
// slot, nr: routed units in the list
__device__ __forceinline__ void gu_unit(int per, int rb, int nr, int sb, int w, int &slot, int &j) {
    constexpr int NP = kGuRows / 2;
    if (w < nr) {
        const int l = rb + w;
        slot = l / per;
        j = NP * (l - slot * per);
    } else {
        slot = kShSlot;
        j = NP * (sb + w - nr);
    }
}

// B / C: the units of g; warps wfirst .. wfirst + wcount - 1 of the CTA take part
// Q8: int8 activations (the IDOT quantisation; x at m.xsq), else limbs
template <int FMT, bool Q8>
__device__ __noinline__ void gateup_run(const DecParams &P, D1S &m, const uint8_t *xq, int rb0, int re0, int sb0,
                                        int se0, int wfirst = 0, int wcount = kNW) {
    constexpr int NP = kGuRows / 2;  // row pairs per unit
    const int warp = threadIdx.x / kWarp - wfirst, lane = threadIdx.x % kWarp;
    const int nr = re0 - rb0, nu = nr + (se0 - sb0);
    const int mine = nu > warp ? (nu - warp + wcount - 1) / wcount : 0;
    const int64_t rb = row_bytes(FMT, P.H);
    const float xinv = m.xinv;
    const int per = (P.I + NP - 1) / NP;
    auto unit = [&](int i, int &slot, int &j) { gu_unit(per, rb0, nr, sb0, warp + wcount * i, slot, j); };
    auto rows_of = [&](int i, const uint8_t *(&rr)[kGuRows]) {
        int slot, j;
        unit(i, slot, j);
        const Rec &r = m.rec[slot];
        const int inter = slot == kShSlot ? P.Is : P.I;
#pragma unroll
        for (int q = 0; q < NP; q++) {
            const int jq = min(j + q, inter - 1);
            rr[2 * q] = r.gw + (size_t)jq * rb;
            rr[2 * q + 1] = r.uw + (size_t)jq * rb;
        }
    };
    auto xq_of = [&](int) { return reinterpret_cast<const uint4 *>(xq); };
    auto pre = [&](int i) {  // lane 16 q: the scales of gate row and up row j + q
        int slot, j;
        unit(i, slot, j);
        const Rec &r = m.rec[slot];
        const int inter = slot == kShSlot ? P.Is : P.I;
        const int jq = min(j + (NP > 1 ? lane >> 4 : 0), inter - 1);
        const bool ld = NP > 1 ? (lane & 15) == 0 : lane == 0;
        return ld ? make_float2(__ldg(r.gs + jq), __ldg(r.us + jq)) : make_float2(0.f, 0.f);
    };
    // 2 rows: lanes 0-15 hold gate j, 16-31 up j; 4 rows: lanes 8 r hold row r of (gate j, up j,
    // gate j + 1, up j + 1); gv / uv are the gate and up values of the lane's row pair
    auto finish = [&](int i, float gv, float uv) {
        int slot, j;
        unit(i, slot, j);
        const int inter = slot == kShSlot ? P.Is : P.I;
        const int q = kGuRows == 2 ? 0 : (lane >> 4);
        const bool mine_row = kGuRows == 2 ? lane == 0 : (lane & 15) == 0;
        if (mine_row && j + q < inter) {
            const float hv = gv / (1.f + expf(-gv)) * uv;
            P.h[(size_t)(slot == kShSlot ? P.K : slot) * P.ldh + j + q] = hv;
            atomicMax(&m.hmax[slot], __float_as_int(fabsf(hv)));
        }
    };
    constexpr int UPD = kGuRows == 2 ? 16 : 8;
    if constexpr (Q8) {
        static_assert(kGuRows == 4, "the int8 walk takes four rows per unit");
        const float sx = m.xsq;
        warp_stream_q8<FMT, kInfl1>(mine, (int)(rb / 16), lane, rows_of, xq_of, pre, [&](int i, int dot, float2 sc) {
            const int up = __shfl_down_sync(kFull, dot, UPD);
            finish(i, __fmul_rn(__fmul_rn(__int2float_rn(dot), sc.x), sx),
                   __fmul_rn(__fmul_rn(__int2float_rn(up), sc.y), sx));
        });
    } else {
        warp_stream_int<FMT, kGuRows, kInfl1, kOnce>(
            mine, (int)(rb / 16), lane, rows_of, xq_of, pre, [&](int i, long long tot, float2 sc) {
                const long long up = __shfl_down_sync(kFull, tot, UPD);
                finish(i, (__ll2float_rn(tot) * xinv) * sc.x, (__ll2float_rn(up) * xinv) * sc.y);
            });
    }
}

// B / C for int4-grouped weights (one fp32 scale per gs inputs of a row): the units of
// gateup_run (two row pairs each), every 16-byte chunk's integer sum scaled by its group
__device__ __noinline__ void gateup_run_grouped(const DecParams &P, D1S &m, const uint8_t *xq, int rb0, int re0,
                                                int sb0, int se0) {
    static_assert(kGuRows == 4, "the grouped walk takes four rows per unit");
    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
    const int nr = re0 - rb0, nu = nr + (se0 - sb0);
    const int mine = nu > warp ? (nu - warp + kNW - 1) / kNW : 0;
    const int64_t rb = row_bytes(COLI_FMT_INT4, P.H);
    const float xinv = m.xinv;
    const int per = (P.I + 1) / 2;
    auto unit = [&](int i, int &slot, int &j) { gu_unit(per, rb0, nr, sb0, warp + kNW * i, slot, j); };
    // both lists of one call are int4-grouped with the same group size
    const int gs = nr > 0 ? P.rgs : P.sgs;
    const int ng = (P.H + gs - 1) / gs;
    warp_stream_int_grouped<COLI_FMT_INT4, kInfl1>(
        mine, (int)(rb / 16), gs, lane,
        [&](int i, const uint8_t *(&rr)[4]) {
            int slot, j;
            unit(i, slot, j);
            const Rec &r = m.rec[slot];
            const int j1 = min(j + 1, (slot == kShSlot ? P.Is : P.I) - 1);
            rr[0] = r.gw + (size_t)j * rb;
            rr[1] = r.uw + (size_t)j * rb;
            rr[2] = r.gw + (size_t)j1 * rb;
            rr[3] = r.uw + (size_t)j1 * rb;
        },
        [&](int i, const float *(&sr)[4]) {
            int slot, j;
            unit(i, slot, j);
            const Rec &r = m.rec[slot];
            const int j1 = min(j + 1, (slot == kShSlot ? P.Is : P.I) - 1);
            sr[0] = r.gs + (size_t)j * ng;
            sr[1] = r.us + (size_t)j * ng;
            sr[2] = r.gs + (size_t)j1 * ng;
            sr[3] = r.us + (size_t)j1 * ng;
        },
        [&](int) { return reinterpret_cast<const uint4 *>(xq); },
        [&](int i, float tot) {  // lanes 0 / 16 hold gate j / j + 1, lanes 8 / 24 up, scaled
            const float up = __shfl_down_sync(kFull, tot, 8);
            int slot, j;
            unit(i, slot, j);
            const int q = lane >> 4;
            if ((lane & 15) == 0 && j + q < (slot == kShSlot ? P.Is : P.I)) {
                const float gv = tot * xinv, uv = up * xinv;
                const float hv = gv / (1.f + expf(-gv)) * uv;
                P.h[(size_t)(slot == kShSlot ? P.K : slot) * P.ldh + j + q] = hv;
                atomicMax(&m.hmax[slot], __float_as_int(fabsf(hv)));
            }
        });
}

// D: down units [lo, hi) of the slot-major space (unit l: slot l / ngr, rows 4 (l % ngr) .. +3);
// slot u's staged h sits at hq + (u - s0) * hs. y goes to the workspace row of the slot.
// rot rotates the warp order so that two calls share the warps evenly.
// Q8: int8 activations (the IDOT quantisation; slot u's h at m.hsq[u - s0]), else limbs
template <int FMT, bool Q8>
__device__ __noinline__ void down_run(const DecParams &P, D1S &m, const uint8_t *hq, int hs, int s0, int lo, int hi,
                                      int ngr, int rot) {
    const int lane = threadIdx.x % kWarp;
    const int warp = (threadIdx.x / kWarp + kNW - rot) % kNW;
    const int nu = hi - lo;
    const int mine = nu > warp ? (nu - warp + kNW - 1) / kNW : 0;
    const bool sh = P.Is > 0 && lo / ngr == m.U;
    const int inter = sh ? P.Is : P.I;
    const int64_t rb = row_bytes(FMT, inter);
    auto unit = [&](int i, int &slot, int &grp) {
        const int l = lo + warp + kNW * i;
        slot = l / ngr;
        grp = l - slot * ngr;
    };
    auto rows_of = [&](int i, const uint8_t *(&rr)[4]) {
        int slot, grp;
        unit(i, slot, grp);
        const Rec &r = m.rec[slot == m.U ? kShSlot : slot];
#pragma unroll
        for (int q = 0; q < 4; q++) rr[q] = r.dw + (size_t)min(4 * grp + q, P.H - 1) * rb;
    };
    auto xq_of = [&](int i) {
        int slot, grp;
        unit(i, slot, grp);
        return reinterpret_cast<const uint4 *>(hq + (size_t)(slot - s0) * hs);
    };
    auto pre = [&](int i) {
        int slot, grp;
        unit(i, slot, grp);
        const Rec &r = m.rec[slot == m.U ? kShSlot : slot];
        return (lane & 7) == 0 ? __ldg(r.ds + min(4 * grp + (lane >> 3), P.H - 1)) : 0.f;
    };
    auto store = [&](int i, auto value_of) {  // lane 8q holds row q
        int slot, grp;
        unit(i, slot, grp);
        const int d = 4 * grp + (lane >> 3);
        if ((lane & 7) == 0 && d < P.H) P.y[(size_t)(slot == m.U ? P.K : slot) * P.H + d] = value_of(slot);
    };
    if constexpr (Q8) {
        warp_stream_q8<FMT, kInfl1>(mine, (int)(rb / 16), lane, rows_of, xq_of, pre, [&](int i, int dot, float sc) {
            store(i, [&](int slot) { return __fmul_rn(__fmul_rn(__int2float_rn(dot), sc), m.hsq[slot - s0]); });
        });
    } else {
        warp_stream_int<FMT, 4, kInfl1, kOnce>(mine, (int)(rb / 16), lane, rows_of, xq_of, pre,
                                               [&](int i, long long tot, float sc) {
                                                   store(i, [&](int slot) {
                                                       return (__ll2float_rn(tot) * m.hinv[slot - s0]) * sc;
                                                   });
                                               });
    }
}

// D for int4-grouped weights: the units of down_run, every chunk scaled by its group
__device__ __noinline__ void down_run_grouped(const DecParams &P, D1S &m, const uint8_t *hq, int hs, int s0, int lo,
                                              int hi, int ngr, int rot) {
    const int lane = threadIdx.x % kWarp;
    const int warp = (threadIdx.x / kWarp + kNW - rot) % kNW;
    const int nu = hi - lo;
    const int mine = nu > warp ? (nu - warp + kNW - 1) / kNW : 0;
    const bool sh = P.Is > 0 && lo / ngr == m.U;
    const int inter = sh ? P.Is : P.I;
    const int64_t rb = row_bytes(COLI_FMT_INT4, inter);
    const int gs = sh ? P.sgs : P.rgs;
    auto unit = [&](int i, int &slot, int &grp) {
        const int l = lo + warp + kNW * i;
        slot = l / ngr;
        grp = l - slot * ngr;
    };
    const int ng = (inter + gs - 1) / gs;
    warp_stream_int_grouped<COLI_FMT_INT4, kInfl1>(
        mine, (int)(rb / 16), gs, lane,
        [&](int i, const uint8_t *(&rr)[4]) {
            int slot, grp;
            unit(i, slot, grp);
            const Rec &r = m.rec[slot == m.U ? kShSlot : slot];
#pragma unroll
            for (int q = 0; q < 4; q++) rr[q] = r.dw + (size_t)min(4 * grp + q, P.H - 1) * rb;
        },
        [&](int i, const float *(&sr)[4]) {
            int slot, grp;
            unit(i, slot, grp);
            const Rec &r = m.rec[slot == m.U ? kShSlot : slot];
#pragma unroll
            for (int q = 0; q < 4; q++) sr[q] = r.ds + (size_t)min(4 * grp + q, P.H - 1) * ng;
        },
        [&](int i) {
            int slot, grp;
            unit(i, slot, grp);
            return reinterpret_cast<const uint4 *>(hq + (size_t)(slot - s0) * hs);
        },
        [&](int i, float tot) {  // lane 8q holds row q, scaled
            int slot, grp;
            unit(i, slot, grp);
            const int d = 4 * grp + (lane >> 3);
            if ((lane & 7) == 0 && d < P.H)
                P.y[(size_t)(slot == m.U ? P.K : slot) * P.H + d] = tot * m.hinv[slot - s0];
        });
}

// D: the h vectors of slots s0 .. s0 + ns - 1 as limbs (slot s0 + j at act + j * hs, in the
// routed layout, or the shared one for slot U), each in block fixed point from the largest |h|
// of the slot over all CTAs. A thread loads up to kHB 16-element items while threads below ns
// read the slots' maxima: one round trip for the usual one or two vectors.
template <int RF, int SF, bool RQ, bool SQ>
__device__ void stage_h(const DecParams &P, D1S &m, uint8_t *act, int hs, int s0, int ns) {
    const int tid = threadIdx.x;
    const int U = m.U;
    const int items_r = limb_items<RF>(P.I), items_s = P.Is > 0 ? limb_items<SF>(P.Is) : 0;
    const int cpr_r = P.I / QGeom<RF>::EPC, cpr_s = P.Is > 0 ? P.Is / QGeom<SF>::EPC : 1;
    // items of staged vector j start at ib[j]
    int total = 0;
    for (int j = 0; j < ns; j++) total += s0 + j < U ? items_r : items_s;
    for (int b0 = 0; b0 < total; b0 += kNT * kHB) {
        float4 v[kHB][4];
        int jv[kHB], pv[kHB];
#pragma unroll
        for (int k = 0; k < kHB; k++) {
            int i = b0 + tid + kNT * k;
            jv[k] = -1;
            if (i < total) {
                int j = 0;
                while (true) {  // at most kMaxK + 1 vectors, usually one or two
                    const int n = s0 + j < U ? items_r : items_s;
                    if (i < n) break;
                    i -= n;
                    j++;
                }
                const int u = s0 + j;
                const bool rt = u < U;
                const int cpr = rt ? cpr_r : cpr_s, epc = rt ? QGeom<RF>::EPC : QGeom<SF>::EPC;
                const int c = i % cpr, ss = i / cpr;
                const float4 *src = reinterpret_cast<const float4 *>(P.h + (size_t)(rt ? u : P.K) * P.ldh + c * epc + ss * 16);
#pragma unroll
                for (int q = 0; q < 4; q++) v[k][q] = __ldcg(src + q);
                jv[k] = j;
                pv[k] = i;
            }
        }
        if (b0 == 0 && tid < ns) {  // the exponent of each staged slot, read while the items are in flight
            const int u = s0 + tid;
            const float amax = __int_as_float(__ldcg(&P.ctrl->hmax[u < U ? u : kShSlot]));
            const int sh = fixed_shift(amax);
            m.hshift[tid] = sh;
            m.hinv[tid] = ldexpf(1.f, -sh);
            m.hamax[tid] = amax;
            m.hsq[tid] = Q8Scale(amax).s;
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < kHB; k++) {
            if (jv[k] >= 0) {
                uint8_t *dst = act + (size_t)jv[k] * hs;
                if (s0 + jv[k] < U) {
                    if constexpr (RQ) q8_from_regs<RF>(v[k], dst, cpr_r, pv[k], Q8Scale(m.hamax[jv[k]]));
                    else limbs_from_regs<RF>(v[k], dst, cpr_r, pv[k], FixedScale(m.hshift[jv[k]]));
                } else {
                    if constexpr (SQ) q8_from_regs<SF>(v[k], dst, cpr_s, pv[k], Q8Scale(m.hamax[jv[k]]));
                    else limbs_from_regs<SF>(v[k], dst, cpr_s, pv[k], FixedScale(m.hshift[jv[k]]));
                }
            }
        }
    }
    __syncthreads();
}

// GRP: bit 0 the routed experts, bit 1 the shared expert are int4-grouped (RF / SF then int4);
// bit 2 the routed experts, bit 3 the shared expert take int8 activations (IDOT)
template <int RF, int SF, int GRP>
__global__ void __launch_bounds__(kNT, 2) moe_decode1_kernel(const __grid_constant__ DecParams P) {
    extern __shared__ __align__(128) uint8_t smem[];
    D1S &m = *reinterpret_cast<D1S *>(smem);
    uint8_t *act = smem + P.d1_act_off;
    float *rsg = reinterpret_cast<float *>(smem + P.d1_rsc_off);
    float *rch = rsg + sel_padded(P.E);
    float2 *rcand = reinterpret_cast<float2 *>(rch + sel_padded(P.E));
    const int tid = threadIdx.x, G = gridDim.x, c = blockIdx.x;
    const bool two = P.Is > 0 && SF != RF;
    uint8_t *xq_r = act, *xq_s = two ? act + 3 * P.H : act;

    if (tid <= kMaxK) m.hmax[tid] = 0;
    if (tid == 0 && P.Is > 0) m.rec[kShSlot] = rec_of(P.shared);
    // CTA 0 resets this call's counters and publishes the call id; every CTA sees the id before
    // its first counter operation (a workspace's earlier contents never hold this id)
    if (c == 0) {
        if (tid <= kMaxK) P.ctrl->hmax[tid] = 0;
        if (tid == 0) {
            P.ctrl->err = 0;
            P.ctrl->router_done = 0;
            P.ctrl->gu_all = 0;
            P.ctrl->dn_done = 0;
        }
        __syncthreads();
        if (tid == 0) {
            __threadfence();
            *reinterpret_cast<volatile unsigned long long *>(&P.ctrl->call) = P.call_id;
        }
    }
    auto await_call = [&]() {  // thread 0
        const volatile unsigned long long *cp = &P.ctrl->call;
        if (*cp == P.call_id) return;
        const uint64_t t0 = globaltimer_ns();
        while (*cp != P.call_id) {
            __nanosleep(32);
            if (globaltimer_ns() - t0 > kWaitNs) {
                flag_error(P.ctrl, kErrWaitExpired);
                return;
            }
        }
        __threadfence();
    };
    // the shared expert's gate/up units, spread over every CTA
    const int bb = range_lo(P.G_sh, c, G), be = range_lo(P.G_sh, c + 1, G);
    __syncthreads();

    // the layer tail normalises resid into shared memory first; else x is read where it is
    const float *xsrc = P.x;
    if (P.resid) {
        float *xf = reinterpret_cast<float *>(smem + P.d1_xf_off);
        stage_xn(P, xf, m);
        xsrc = xf;
    }

    // ---------------- A: router partial logits
    if (c < P.R) {
        router_item1(P, c, xsrc);
        __syncthreads();
        if (tid == 0) {
            await_call();
            __threadfence();
            atomicAdd(&P.ctrl->router_done, 1);
        }
    }
    // ---------------- X: the expert table and the bias into shared memory, then x as limbs
    // (read by routing only, after the barriers below). A thread's share of the copy is held in
    // registers while x loads, so the two share one round trip; a table too large for that is
    // copied first.
    const float *bias_s = P.bias;
    const coli_moe_expert *tab_s = P.experts;
    constexpr int kTabRegs = 8;  // 8-byte table words per thread held across the x staging
    const int n8 = P.E * (int)(sizeof(coli_moe_expert) / 8);
    uint2 *ts = reinterpret_cast<uint2 *>(smem + P.d1_tab_off);
    float *bs = reinterpret_cast<float *>(smem + P.d1_bias_off);
    const uint2 *tg = reinterpret_cast<const uint2 *>(P.experts);
    const bool tab_regs = P.d1_tab_off > 0 && n8 <= kTabRegs * kNT && P.E <= kNT;
    uint2 tv[kTabRegs];
    float bv = 0.f;
    if (tab_regs) {
#pragma unroll
        for (int k = 0; k < kTabRegs; k++)
            if (tid + k * kNT < n8) tv[k] = __ldg(tg + tid + k * kNT);
        if (tid < P.E) bv = __ldg(P.bias + tid);
    } else if (P.d1_tab_off > 0) {
        for (int i = tid; i < n8; i += kNT) ts[i] = __ldg(tg + i);
        for (int i = tid; i < P.E; i += kNT) bs[i] = __ldg(P.bias + i);
    }
    if (P.d1_tab_off > 0) {
        bias_s = bs;
        tab_s = reinterpret_cast<const coli_moe_expert *>(ts);
    }
    constexpr bool RQ = (GRP & 4) != 0, SQ = (GRP & 8) != 0;
    stage_x<RF, SF, RQ, SQ>(P, xsrc, xq_r, xq_s, two, m);
    if (tab_regs) {
#pragma unroll
        for (int k = 0; k < kTabRegs; k++)
            if (tid + k * kNT < n8) ts[tid + k * kNT] = tv[k];
        if (tid < P.E) bs[tid] = bv;
    }
    // ---------------- B: the shared expert's gate/up, here only when its walk differs from the
    // routed experts' (else its units follow the routed ones in one stream, phase C)
    constexpr bool kMerged = RF == SF && ((GRP & 1) != 0) == ((GRP & 2) != 0) && RQ == SQ;
    if (!kMerged && be > bb) {
        if constexpr ((GRP & 2) != 0) gateup_run_grouped(P, m, xq_s, 0, 0, bb, be);
        else gateup_run<SF, SQ>(P, m, xq_s, 0, 0, bb, be);
    }

    // ---------------- R: routing
    if (tid == 0) {
        await_call();
        wait_at_least(&P.ctrl->router_done, P.R, P.ctrl);
        __threadfence();
    }
    __syncthreads();
    route1(P, m, rsg, rch, rcand, bias_s, tab_s);
    const int U = m.U;
    const int nsl = U + (P.Is > 0 ? 1 : 0);
    const int ngr = (P.H + 3) / 4, ND = nsl * ngr;
    const int db = range_lo(ND, c, G), de = range_lo(ND, c + 1, G);

    // ---------------- C: routed gate/up (then the shared expert's, one stream, when merged)
    const int gu_per = (P.I + kGuRows / 2 - 1) / (kGuRows / 2);  // units per routed slot
    const int gu_tot = U * gu_per;
    const int cb = range_lo(gu_tot, c, G), ce = range_lo(gu_tot, c + 1, G);
    if constexpr ((GRP & 1) != 0) gateup_run_grouped(P, m, xq_r, cb, ce, kMerged ? bb : 0, kMerged ? be : 0);
    else gateup_run<RF, RQ>(P, m, xq_r, cb, ce, kMerged ? bb : 0, kMerged ? be : 0);
    __syncthreads();
    if (tid < U || (tid == kShSlot && P.Is > 0))
        if (m.hmax[tid] != 0) atomicMax(&P.ctrl->hmax[tid], m.hmax[tid]);
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        atomicAdd(&P.ctrl->gu_all, (be - bb) + (ce - cb));
    }

    // ---------------- D: down rows, (slot, 4-row group) units split slot-major over the CTAs
    if (tid == 0) {
        wait_at_least(&P.ctrl->gu_all, P.G_sh + gu_tot, P.ctrl);
        __threadfence();
    }
    __syncthreads();
    const int s0 = db / ngr, ns = de > db ? (de - 1) / ngr - s0 + 1 : 0;
    const int hs = P.d1_hs;
    stage_h<RF, SF, RQ, SQ>(P, m, act, hs, s0, ns);
    {
        // one stream through routed and shared units when their rows have the same walk and length
        const int split = (kMerged && P.I == P.Is) ? de : U * ngr;  // routed units below, shared from here
        const int rlo = db, rhi = min(de, split), slo = max(db, split), shi = de;
        const int rot = rhi > rlo ? (rhi - rlo) % kNW : 0;
        if (rhi > rlo) {
            if constexpr ((GRP & 1) != 0) down_run_grouped(P, m, act, hs, s0, rlo, rhi, ngr, 0);
            else down_run<RF, RQ>(P, m, act, hs, s0, rlo, rhi, ngr, 0);
        }
        if (shi > slo) {
            if constexpr ((GRP & 2) != 0) down_run_grouped(P, m, act, hs, s0, slo, shi, ngr, rot);
            else down_run<SF, SQ>(P, m, act, hs, s0, slo, shi, ngr, rot);
        }
    }
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        atomicAdd(&P.ctrl->dn_done, de - db);
    }

    // ---------------- E: this CTA's rows of out, selection order then the shared expert
    if (tid == 0) {
        wait_at_least(&P.ctrl->dn_done, ND, P.ctrl);
        __threadfence();
    }
    __syncthreads();
    const int r_lo = range_lo(P.H, c, G), r_hi = range_lo(P.H, c + 1, G);
    for (int d = r_lo + tid; d < r_hi; d += kNT) {
        float yv[kMaxK + 1];
#pragma unroll
        for (int k = 0; k <= kMaxK; k++)
            if (k < U) yv[k] = __ldcg(P.y + (size_t)m.pos[k] * P.H + d);
            else if (k == U && P.Is > 0) yv[k] = __ldcg(P.y + (size_t)P.K * P.H + d);
        float a = 0.f;
#pragma unroll
        for (int k = 0; k < kMaxK; k++)
            if (k < U) a = __fadd_rn(a, __fmul_rn(m.w[k], yv[k]));
        if (P.Is > 0) {
#pragma unroll
            for (int k = 0; k <= kMaxK; k++)
                if (k == U) a = __fadd_rn(a, yv[k]);
        }
        if (P.resid) a = __fadd_rn(P.resid[d], a);  // the layer tail: x += tmp
        P.out[d] = a;
    }
}

using KernelFn = void (*)(DecParams);

// rf, sf: the formats of the instance (int4-grouped weights run as int4); grp as in the kernel
KernelFn kernel_for(int rf, int sf, int grp) {
    constexpr int I8 = COLI_FMT_INT8, I4 = COLI_FMT_INT4, I2 = COLI_FMT_INT2;
    auto pick = [](int f) { return f == COLI_FMT_INT8 ? 0 : f == COLI_FMT_INT4 ? 1 : 2; };
    static const KernelFn plain[3][3] = {
        {moe_decode1_kernel<I8, I8, 0>, moe_decode1_kernel<I8, I4, 0>, moe_decode1_kernel<I8, I2, 0>},
        {moe_decode1_kernel<I4, I8, 0>, moe_decode1_kernel<I4, I4, 0>, moe_decode1_kernel<I4, I2, 0>},
        {moe_decode1_kernel<I2, I8, 0>, moe_decode1_kernel<I2, I4, 0>, moe_decode1_kernel<I2, I2, 0>},
    };
    // routed grouped (by the shared format), shared grouped (by the routed format), both
    static const KernelFn rgrp[3] = {moe_decode1_kernel<I4, I8, 1>, moe_decode1_kernel<I4, I4, 1>,
                                     moe_decode1_kernel<I4, I2, 1>};
    static const KernelFn sgrp[3] = {moe_decode1_kernel<I8, I4, 2>, moe_decode1_kernel<I4, I4, 2>,
                                     moe_decode1_kernel<I2, I4, 2>};
    // int8 activations (IDOT): routed and shared (int8 / int4 each), routed only, shared only
    static const KernelFn q8both[2][2] = {{moe_decode1_kernel<I8, I8, 12>, moe_decode1_kernel<I8, I4, 12>},
                                          {moe_decode1_kernel<I4, I8, 12>, moe_decode1_kernel<I4, I4, 12>}};
    static const KernelFn q8r[2] = {moe_decode1_kernel<I8, I2, 4>, moe_decode1_kernel<I4, I2, 4>};
    static const KernelFn q8s[2] = {moe_decode1_kernel<I2, I8, 8>, moe_decode1_kernel<I2, I4, 8>};
    if (grp == 12) return q8both[pick(rf)][pick(sf)];
    if (grp == 4) return q8r[pick(rf)];
    if (grp == 8) return q8s[pick(sf)];
    if (grp == 3) return moe_decode1_kernel<I4, I4, 3>;
    if (grp == 1) return rgrp[pick(sf)];
    if (grp == 2) return sgrp[pick(rf)];
    return plain[pick(rf)][pick(sf)];
}

// the grouped bits of a plan
int grp_of(const DecParams &P) {
    return (P.rgs > 0 ? 1 : 0) | (P.sgs > 0 ? 2 : 0) | (P.rq8 ? 4 : 0) | (P.sq8 ? 8 : 0);
}

size_t decode1_smem_bytes(const DecParams &P) { return (size_t)P.d1_end; }

}  // namespace

// Host-side geometry of the single-token launch for a grid of `grid` CTAs.
bool decode1_plan(const coli_moe_desc &d, DecParams &P, int grid) {
    if (d.T != 1 || d.K > kMaxK || d.E > kMaxE) return false;
    P.single = 1;
    P.K = d.K;
    // int4-grouped weights run in the int4 instances, their scales applied per 16-byte chunk
    P.rfmt = d.routed_fmt == COLI_FMT_INT4G ? COLI_FMT_INT4 : d.routed_fmt;
    P.sfmt = d.shared_fmt == COLI_FMT_INT4G ? COLI_FMT_INT4 : d.shared_fmt;
    P.rgs = d.routed_fmt == COLI_FMT_INT4G ? d.group_size : 0;
    P.sgs = d.I_shared > 0 && d.shared_fmt == COLI_FMT_INT4G ? d.group_size : 0;
    // IDOT: int8 activations for the int8 and int4 experts (int2 and int4-grouped keep limbs)
    auto q8 = [&](int f) { return d.idot != 0 && (f == COLI_FMT_INT8 || f == COLI_FMT_INT4); };
    P.rq8 = q8(d.routed_fmt) ? 1 : 0;
    P.sq8 = d.I_shared > 0 && q8(d.shared_fmt) ? 1 : 0;
    if ((P.rgs > 0 || P.sgs > 0) && (P.rq8 || P.sq8)) return false;  // the general kernels take those
    P.NV = 1;
    P.route_only = 0;
    P.neb = (d.E + kRtE - 1) / kRtE;
    const int max_slices = std::max(1, d.H / 128);
    int nks = std::max(1, std::min({grid / P.neb, max_slices, kMaxSlices}));
    P.rks_floats = (d.H / nks + 3) / 4 * 4;
    nks = (d.H + P.rks_floats - 1) / P.rks_floats;
    P.nks = nks;
    P.R = P.neb * nks;
    if (P.R > grid) return false;
    P.groups_sh = d.I_shared > 0 ? 1 : 0;
    P.G_sh = d.I_shared > 0 ? (d.I_shared + kGuRows / 2 - 1) / (kGuRows / 2) : 0;  // shared gate/up units
    const bool two = d.I_shared > 0 && P.sfmt != P.rfmt;
    const size_t x_bytes = (size_t)3 * d.H * (two ? 2 : 1);
    P.d1_hs = 3 * std::max(d.I, d.I_shared);  // limbs of one staged h vector (a multiple of 16)
    // the slots one CTA's down units can touch: its share of (K + 1) * ngr units over `grid`
    const int ngr = (d.H + 3) / 4;
    const int share = ((d.K + 1) * ngr + grid - 1) / grid;
    const int ns_max = std::min(d.K + 1, (share + ngr - 1) / ngr + 1);
    const size_t h_bytes = (size_t)P.d1_hs * ns_max;
    const int ksel = (d.ksel > 0 && d.ksel < d.K) ? d.ksel : d.K;
    const size_t sel_bytes = (size_t)2 * sel_padded(d.E) * 4 + (size_t)sel_cand_cap(d.E, ksel) * 8;
    size_t o = align_up(sizeof(D1S), 128);
    P.d1_act_off = (int)o;
    o += align_up(std::max(x_bytes, h_bytes), 128);
    P.d1_rsc_off = (int)o;
    o += align_up(sel_bytes, 128);
    P.d1_ylo_off = 0;
    P.d1_pairs = 0;
    // the expert table and the bias in shared memory when they are small
    const size_t tab_bytes = (size_t)d.E * sizeof(coli_moe_expert);
    if (tab_bytes + (size_t)d.E * 4 <= 32 * 1024) {
        P.d1_tab_off = (int)o;
        o += align_up(tab_bytes, 128);
        P.d1_bias_off = (int)o;
        o += align_up((size_t)d.E * 4, 128);
    } else {
        P.d1_tab_off = P.d1_bias_off = 0;
    }
    // the layer tail's normalised row (H floats), reserved by every plan: the kernel reads it
    // only when it is given a residual
    P.d1_xf_off = (int)o;
    o += align_up((size_t)d.H * 4, 128);
    P.d1_end = (int)o;
    return decode1_smem_bytes(P) <= 113u * 1024;
}

int decode1_ctas_per_sm(const DecParams &P) {
    int n = 0;
    const void *fn = (const void *)kernel_for(P.rfmt, P.sfmt, grp_of(P));
    const size_t smem = decode1_smem_bytes(P);
    // the query counts against the kernel's dynamic shared-memory limit: raise it first
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kNT, smem) != cudaSuccess) return 0;
    return n;
}

cudaError_t launch_decode1(const DecParams &P, int grid, cudaStream_t st) {
    const size_t smem = decode1_smem_bytes(P);
    const void *fn = (const void *)kernel_for(P.rfmt, P.sfmt, grp_of(P));
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    void *args[] = {const_cast<DecParams *>(&P)};
    return cudaLaunchCooperativeKernel(fn, dim3(grid), dim3(kNT), args, smem, st);
}

}  // namespace colimoe
