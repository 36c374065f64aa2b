// decode1.cu — the whole MoE block for ONE token (T = 1) in one persistent launch.
//
// The single-token call is the decode step of the engine (colibri-strix c/glm.c @98759bf
// moe() with S = 1; the Metal path's moe_gemv). Its work is tiny per CTA — a few row chunks per
// warp — so the kernel is built around the number of dependent memory round trips rather than
// around tiling. Phases, split statically over the CTAs (two per SM, cooperative launch):
//   X  the token's x in 24-bit block fixed point (idot.cuh), staged once per CTA, in the
//      layout of each weight format the block uses
//   A  router items: partial logits of 32 experts over one slice of H (r_router shader)
//   B  shared expert gate/up rows (independent of routing)
//   R  routing by EVERY CTA from the partial logits: logits summed in a fixed order, sigmoid,
//      bias, greedy top-K with ties to the lower index (select.cuh: an expert's place in the
//      greedy order is the number of experts that beat it, counted over candidates),
//      TOPK/TOPP, renorm, routed scale. The kept experts become slots 0..U-1 in ascending id
//      order; the shared expert is slot U. Their weight pointers are loaded by the lanes that
//      hold them.
//   C  routed gate/up rows: h = silu(gate.x * s_g) * (up.x * s_u); every CTA also records the
//      largest |h| of each slot it wrote, the block fixed-point exponent of the down step
//   D  once every gate/up row is in (one counter): (slot, 4-row group) units split slot-major
//      over the CTAs, so each stages only the one or two h vectors its units read; y rows
//      go to the workspace
//   E  once every down row is in (one counter): each CTA's rows of
//      out[d] = sum_k w_k y[pos_k][d] in selection order, + y[U][d]  (moe() phases C/D/E)
//      (staging every h vector in every CTA to combine without y was measured slower)
// Warps walk their gate/up and down units without CTA barriers. (Asking L2 for each phase's
// rows ahead with cp.async.bulk.prefetch was measured: it slowed large decode by 11 %, so the
// loads go straight to HBM.) Every wait is bounded.
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

struct D1S {  // the fixed part of the CTA's shared memory
    Rec rec[kMaxK + 1];
    int slot_e[kMaxK];
    int pos[kMaxK];     // slot of selection k, -1 beyond keff
    float w[kMaxK];     // kept routing weights, 0 beyond keff
    int sel_i[kMaxK];
    int ncand, nok;  // selection: candidates, selectable experts
    int U;
    int xshift;
    float xinv;
    int hshift[kMaxK + 1];
    float hinv[kMaxK + 1];
    int hmax[kMaxK + 1];  // this CTA's max |h| per slot (float bits); shared at kShSlot
    float redf[kNW];
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

template <int RF, int SF>
__device__ void stage_x(const DecParams &P, uint8_t *xq_r, uint8_t *xq_s, bool two, D1S &m) {
    const int tid = threadIdx.x, lane = tid % kWarp, warp = tid / kWarp;
    const int n16 = P.H / 16;  // 16-element groups; group q is item q of every layout ordering
    const float4 *x4 = reinterpret_cast<const float4 *>(P.x);
    const bool in_regs = n16 <= 2 * kNT;
    float4 v[2][4];
    float mx = 0.f;
    for (int q0 = tid; q0 < n16; q0 += 2 * kNT) {
#pragma unroll
        for (int j = 0; j < 2; j++) {
            const int q = q0 + j * kNT;
            if (q < n16)
#pragma unroll
                for (int k = 0; k < 4; k++) v[j][k] = __ldg(x4 + 4 * q + k);
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
                    for (int k = 0; k < 4; k++) v[j][k] = __ldg(x4 + 4 * q + k);
            }
        }
#pragma unroll
        for (int j = 0; j < 2; j++) {
            const int q = q0 + j * kNT;
            if (q < n16) {
                limbs_from_regs<RF>(v[j], xq_r, P.H / QGeom<RF>::EPC, item_of(QGeom<RF>::EPC, IQ<RF>::NSS, q), fx);
                if (two)
                    limbs_from_regs<SF>(v[j], xq_s, P.H / QGeom<SF>::EPC, item_of(QGeom<SF>::EPC, IQ<SF>::NSS, q), fx);
            }
        }
    }
    if (tid == 0) {
        m.xshift = s;
        m.xinv = ldexpf(1.f, -s);
    }
    __syncthreads();
}

// R: the routing of the token by this CTA (sg/ch: shared scratch of sel_padded(E) floats each,
// cand: sel_cand_cap(E, Ksel) float2)
__device__ __noinline__ void route1(const DecParams &P, D1S &m, float *sg, float *ch, float2 *cand) {
    const int tid = threadIdx.x, lane = tid % kWarp, warp = tid / kWarp;
    const bool out = blockIdx.x == 0;
    const int E = P.E, Ep = sel_padded(E);
    // 1. logits (fixed-order sum of the partial slices) -> sigmoid scores and choices
    for (int e = tid; e < Ep; e += kNT) {
        if (e < E) {
            float a[16];
#pragma unroll
            for (int k = 0; k < 16; k++)
                if (k < P.nks) a[k] = __ldcg(P.part + (size_t)k * E + e);
            float lg = 0.f;
#pragma unroll
            for (int k = 0; k < 16; k++)
                if (k < P.nks) lg += a[k];
            const float sv = 1.f / (1.f + expf(-lg));
            const float cv = sv + __ldg(P.bias + e);
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
        // each kept lane asks for its expert's weight pointers
        coli_moe_expert ex{};
        if (lane < Ke) ex = P.experts[id];
        const bool kept = lane < Ke;
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

// B / C: gate/up units [b, e) (shared: the shared expert's, else slot-major over the routed
// slots), each two rows j, j+1 of gate and of up; warps take units round-robin, no barriers
template <int FMT>
__device__ __noinline__ void gateup_run(const DecParams &P, D1S &m, const uint8_t *xq, int b, int e, bool shared) {
    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
    const int nu = e - b;
    const int mine = nu > warp ? (nu - warp + kNW - 1) / kNW : 0;
    const int inter = shared ? P.Is : P.I;
    const int per = (inter + 1) / 2;
    const int64_t rb = row_bytes(FMT, P.H);
    const float xinv = m.xinv;
    auto unit = [&](int i, int &slot, int &j) {
        const int l = b + warp + kNW * i;
        slot = shared ? kShSlot : l / per;
        j = 2 * (shared ? l : l - slot * per);
    };
    warp_stream_int<FMT, 4, kInfl1>(
        mine, (int)(rb / 16), lane,
        [&](int i, const uint8_t *(&rr)[4]) {
            int slot, j;
            unit(i, slot, j);
            const Rec &r = m.rec[slot];
            const int j1 = min(j + 1, inter - 1);
            rr[0] = r.gw + (size_t)j * rb;
            rr[1] = r.uw + (size_t)j * rb;
            rr[2] = r.gw + (size_t)j1 * rb;
            rr[3] = r.uw + (size_t)j1 * rb;
        },
        [&](int) { return reinterpret_cast<const uint4 *>(xq); },
        [&](int i) {  // lanes 0 and 16: the scales of rows j and j + 1
            int slot, j;
            unit(i, slot, j);
            const Rec &r = m.rec[slot];
            const int jq = min(j + (lane >> 4), inter - 1);
            return (lane & 15) == 0 ? make_float2(__ldg(r.gs + jq), __ldg(r.us + jq)) : make_float2(0.f, 0.f);
        },
        [&](int i, long long tot, float2 sc) {  // lanes 0 / 16 hold gate j / j+1, lanes 8 / 24 up
            const long long up = __shfl_down_sync(kFull, tot, 8);
            int slot, j;
            unit(i, slot, j);
            const int jq = j + (lane >> 4);
            if ((lane & 15) == 0 && jq < inter) {
                const float gv = (__ll2float_rn(tot) * xinv) * sc.x;
                const float uv = (__ll2float_rn(up) * xinv) * sc.y;
                const float hv = gv / (1.f + expf(-gv)) * uv;
                P.h[(size_t)(shared ? P.K : slot) * P.ldh + jq] = hv;
                atomicMax(&m.hmax[slot], __float_as_int(fabsf(hv)));
            }
        });
}

// D: down units [lo, hi) of the slot-major space (unit l: slot l / ngr, rows 4 (l % ngr) .. +3);
// slot u's staged h sits at hq + (u - s0) * hs. y goes to the workspace row of the slot.
// rot rotates the warp order so that two calls share the warps evenly.
template <int FMT>
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
    warp_stream_int<FMT, 4, kInfl1>(
        mine, (int)(rb / 16), lane,
        [&](int i, const uint8_t *(&rr)[4]) {
            int slot, grp;
            unit(i, slot, grp);
            const Rec &r = m.rec[sh ? kShSlot : slot];
#pragma unroll
            for (int q = 0; q < 4; q++) rr[q] = r.dw + (size_t)min(4 * grp + q, P.H - 1) * rb;
        },
        [&](int i) {
            int slot, grp;
            unit(i, slot, grp);
            return reinterpret_cast<const uint4 *>(hq + (size_t)(slot - s0) * hs);
        },
        [&](int i) {
            int slot, grp;
            unit(i, slot, grp);
            const Rec &r = m.rec[sh ? kShSlot : slot];
            return (lane & 7) == 0 ? __ldg(r.ds + min(4 * grp + (lane >> 3), P.H - 1)) : 0.f;
        },
        [&](int i, long long tot, float sc) {  // lane 8q holds row q
            int slot, grp;
            unit(i, slot, grp);
            const int d = 4 * grp + (lane >> 3);
            if ((lane & 7) == 0 && d < P.H)
                P.y[(size_t)(sh ? P.K : slot) * P.H + d] = (__ll2float_rn(tot) * m.hinv[slot - s0]) * sc;
        });
}

template <int RF, int SF>
__global__ void __launch_bounds__(kNT, 2) moe_decode1_kernel(const DecParams P) {
    extern __shared__ __align__(128) uint8_t smem[];
    D1S &m = *reinterpret_cast<D1S *>(smem);
    uint8_t *act = smem + P.d1_act_off;
    float *rsg = reinterpret_cast<float *>(smem + P.d1_rsc_off);
    float *rch = rsg + sel_padded(P.E);
    float2 *rcand = reinterpret_cast<float2 *>(rch + sel_padded(P.E));
    const int tid = threadIdx.x, G = gridDim.x, c = blockIdx.x;
    const bool two = P.Is > 0 && SF != RF;
    uint8_t *xq_r = act, *xq_s = two ? act + 3 * P.H : act;
    const int GUPER = (P.I + 1) / 2;

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
    __syncthreads();
    // the shared expert's gate/up goes to the CTAs without a router item, so that every CTA
    // reaches the routing wait at about the same time
    const int nb = G - P.R > 0 ? G - P.R : G, cb0 = G - P.R > 0 ? c - P.R : c;
    const int bb = cb0 < 0 ? 0 : range_lo(P.G_sh, cb0, nb), be = cb0 < 0 ? 0 : range_lo(P.G_sh, cb0 + 1, nb);
    // routing reads the bias and the expert table right after its wait: warm them in L2
    {
        const int lb = (P.E * 4 + 127) / 128, lt = (P.E * (int)sizeof(coli_moe_expert) + 127) / 128;
        const int per = (lb + lt + G - 1) / G;
        for (int i = c * per + tid; i < min(lb + lt, (c + 1) * per) && tid < per; i += kNT) {
            if (i < lb) prefetch_line_l2(reinterpret_cast<const uint8_t *>(P.bias) + 128 * i);
            else prefetch_line_l2(reinterpret_cast<const uint8_t *>(P.experts) + 128 * (i - lb));
        }
    }

    // ---------------- A: router partial logits
    if (c < P.R) {
        router_item<1>(P, c);
        __syncthreads();
        if (tid == 0) {
            await_call();
            __threadfence();
            atomicAdd(&P.ctrl->router_done, 1);
        }
    }
    // ---------------- X, then B: the shared expert's gate/up
    stage_x<RF, SF>(P, xq_r, xq_s, two, m);
    if (be > bb) gateup_run<SF>(P, m, xq_s, bb, be, true);

    // ---------------- R: routing
    if (tid == 0) {
        await_call();
        wait_at_least(&P.ctrl->router_done, P.R, P.ctrl);
        __threadfence();
    }
    __syncthreads();
    route1(P, m, rsg, rch, rcand);
    const int U = m.U;

    // ---------------- C: routed gate/up
    const int gu_tot = U * GUPER;
    const int cb = range_lo(gu_tot, c, G), ce = range_lo(gu_tot, c + 1, G);
    gateup_run<RF>(P, m, xq_r, cb, ce, false);
    __syncthreads();
    if (tid < U || (tid == kShSlot && P.Is > 0))
        if (m.hmax[tid] != 0) atomicMax(&P.ctrl->hmax[tid], m.hmax[tid]);
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        atomicAdd(&P.ctrl->gu_all, (be - bb) + (ce - cb));
    }

    // ---------------- D: down rows, (slot, 4-row group) units split slot-major over the CTAs, so
    // a CTA stages only the one or two h vectors its units read
    if (tid == 0) {
        wait_at_least(&P.ctrl->gu_all, P.G_sh + gu_tot, P.ctrl);
        __threadfence();
    }
    __syncthreads();
    const int nsl = U + (P.Is > 0 ? 1 : 0);
    const int ngr = P.H / 4, ND = nsl * ngr;
    const int db = range_lo(ND, c, G), de = range_lo(ND, c + 1, G);
    const int s0 = db / ngr, ns = de > db ? (de - 1) / ngr - s0 + 1 : 0;
    const int hs = 3 * (P.I > P.Is ? P.I : P.Is);  // staged bytes per h vector
    if (tid < ns) {
        const int u = s0 + tid;
        const int s = fixed_shift(__int_as_float(__ldcg(&P.ctrl->hmax[u < U ? u : kShSlot])));
        m.hshift[tid] = s;
        m.hinv[tid] = ldexpf(1.f, -s);
    }
    __syncthreads();
    for (int j = 0; j < ns; j++) {
        const int u = s0 + j;
        const FixedScale fx(m.hshift[j]);
        if (u < U) stage_limbs_vec<RF>(P.h + (size_t)u * P.ldh, P.I, true, act + (size_t)j * hs, fx, tid, kNT);
        else stage_limbs_vec<SF>(P.h + (size_t)P.K * P.ldh, P.Is, true, act + (size_t)j * hs, fx, tid, kNT);
    }
    __syncthreads();
    {
        const int split = U * ngr;  // routed units below, shared units from here
        const int rlo = db, rhi = min(de, split), slo = max(db, split), shi = de;
        if (rhi > rlo) down_run<RF>(P, m, act, hs, s0, rlo, rhi, ngr, 0);
        if (shi > slo) down_run<SF>(P, m, act, hs, s0, slo, shi, ngr, rhi > rlo ? (rhi - rlo) % kNW : 0);
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
        P.out[d] = a;
    }
}

using KernelFn = void (*)(DecParams);

KernelFn kernel_for(int rf, int sf) {
    auto pick = [](int f) { return f == COLI_FMT_INT8 ? 0 : f == COLI_FMT_INT4 ? 1 : 2; };
    static const KernelFn table[3][3] = {
        {moe_decode1_kernel<COLI_FMT_INT8, COLI_FMT_INT8>, moe_decode1_kernel<COLI_FMT_INT8, COLI_FMT_INT4>,
         moe_decode1_kernel<COLI_FMT_INT8, COLI_FMT_INT2>},
        {moe_decode1_kernel<COLI_FMT_INT4, COLI_FMT_INT8>, moe_decode1_kernel<COLI_FMT_INT4, COLI_FMT_INT4>,
         moe_decode1_kernel<COLI_FMT_INT4, COLI_FMT_INT2>},
        {moe_decode1_kernel<COLI_FMT_INT2, COLI_FMT_INT8>, moe_decode1_kernel<COLI_FMT_INT2, COLI_FMT_INT4>,
         moe_decode1_kernel<COLI_FMT_INT2, COLI_FMT_INT2>},
    };
    return table[pick(rf)][pick(sf)];
}

size_t decode1_smem_bytes(const DecParams &P) { return (size_t)P.d1_y_off; }

}  // namespace

// Host-side geometry of the single-token launch for a grid of `grid` CTAs.
bool decode1_plan(const coli_moe_desc &d, DecParams &P, int grid) {
    if (d.T != 1 || d.K > kMaxK || d.E > kMaxE) return false;
    P.single = 1;
    P.K = d.K;
    P.rfmt = d.routed_fmt;
    P.sfmt = d.shared_fmt;
    P.NV = 1;
    P.route_only = 0;
    P.neb = (d.E + kRtE - 1) / kRtE;
    const int max_slices = std::max(1, d.H / 128);
    int nks = std::max(1, std::min({grid / P.neb, max_slices, 16}));
    P.rks_floats = (d.H / nks + 3) / 4 * 4;
    nks = (d.H + P.rks_floats - 1) / P.rks_floats;
    P.nks = nks;
    P.R = P.neb * nks;
    if (P.R > grid) return false;
    P.groups_sh = d.I_shared > 0 ? 1 : 0;
    P.G_sh = d.I_shared > 0 ? (d.I_shared + 1) / 2 : 0;
    const bool two = d.I_shared > 0 && d.shared_fmt != d.routed_fmt;
    const size_t x_bytes = (size_t)3 * d.H * (two ? 2 : 1);
    const size_t h_bytes = (size_t)3 * (d.K + 1) * std::max(d.I, d.I_shared);
    P.d1_act_off = (int)align_up(sizeof(D1S), 128);
    P.d1_rsc_off = P.d1_act_off + (int)align_up(std::max(x_bytes, h_bytes), 128);
    const int ksel = (d.ksel > 0 && d.ksel < d.K) ? d.ksel : d.K;
    const size_t sel_bytes = (size_t)2 * sel_padded(d.E) * 4 + (size_t)sel_cand_cap(d.E, ksel) * 8;
    P.d1_y_off = P.d1_rsc_off + (int)align_up(sel_bytes, 128);  // end of smem
    P.d1_rows = 0;
    return decode1_smem_bytes(P) <= 113u * 1024;
}

int decode1_ctas_per_sm(const DecParams &P) {
    int n = 0;
    const void *fn = (const void *)kernel_for(P.rfmt, P.sfmt);
    const size_t smem = decode1_smem_bytes(P);
    // the query counts against the kernel's dynamic shared-memory limit: raise it first
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kNT, smem) != cudaSuccess) return 0;
    return n;
}

cudaError_t launch_decode1(const DecParams &P, int grid, cudaStream_t st) {
    const size_t smem = decode1_smem_bytes(P);
    const void *fn = (const void *)kernel_for(P.rfmt, P.sfmt);
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    void *args[] = {const_cast<DecParams *>(&P)};
    return cudaLaunchCooperativeKernel(fn, dim3(grid), dim3(kNT), args, smem, st);
}

}  // namespace colimoe
