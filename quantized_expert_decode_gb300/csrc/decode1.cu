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
//      bias, greedy top-K with ties to the lower index (found as ranks: an expert's place in
//      the greedy order is the number of experts that beat it), TOPK/TOPP, renorm, routed
//      scale. The kept experts become slots 0..U-1 in ascending id order; the shared expert
//      is slot U. Their weight pointers go to shared memory in one round trip.
//   C  routed gate/up rows: h = silu(gate.x * s_g) * (up.x * s_u); every CTA also records the
//      largest |h| of each slot it wrote, the block fixed-point exponent of the down step
//   D  once every gate/up row is in (one counter), each CTA stages ALL h vectors and computes,
//      for its own block of output rows d, y[slot][d] for every slot, then
//      out[d] = sum_k w_k y[pos_k][d] in selection order, + y[U][d]  (moe() phases C/D/E)
//      — the combine needs no y round trip through memory and no final wait.
// Warps walk their gate/up and down units without CTA barriers. (Asking L2 for each phase's
// rows ahead with cp.async.bulk.prefetch was measured: it slowed large decode by 11 %, so the
// loads go straight to HBM.) Every wait is bounded.
#include <algorithm>

#include "decode_parts.cuh"

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
    float sel_w[kMaxK];
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

// X: x -> limbs in the routed layout (and the shared one when it differs)
template <int RF, int SF>
__device__ void stage_x(const DecParams &P, uint8_t *xq_r, uint8_t *xq_s, bool two, D1S &m) {
    const int tid = threadIdx.x, lane = tid % kWarp, warp = tid / kWarp;
    const int n4 = P.H / 4;
    const float4 *x4 = reinterpret_cast<const float4 *>(P.x);
    constexpr int B = 4;
    float mx = 0.f;
    for (int q0 = tid; q0 < n4; q0 += kNT * B) {
        float4 v[B];
#pragma unroll
        for (int j = 0; j < B; j++)
            if (q0 + j * kNT < n4) v[j] = __ldg(x4 + q0 + j * kNT);
#pragma unroll
        for (int j = 0; j < B; j++)
            if (q0 + j * kNT < n4)
                mx = fmaxf(mx, fmaxf(fmaxf(fabsf(v[j].x), fabsf(v[j].y)), fmaxf(fabsf(v[j].z), fabsf(v[j].w))));
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
    stage_limbs_vec<RF>(P.x, P.H, false, xq_r, fx, tid, kNT);
    if (two) stage_limbs_vec<SF>(P.x, P.H, false, xq_s, fx, tid, kNT);
    if (tid == 0) {
        m.xshift = s;
        m.xinv = ldexpf(1.f, -s);
    }
    __syncthreads();
}

// TOPP on the nsel selected (one per lane, selection order): sort by weight, descending and
// stable (the insertion sort of the pages' top-p step), then keep the shortest prefix whose
// running sum reaches top_p * (1e-20 + total). Returns the kept count; id/wv come back sorted.
__device__ __noinline__ int top_p_cut(float top_p, int nsel, int &id, float &wv) {
    const int lane = threadIdx.x % kWarp;
    int p = 0;
    for (int k = 0; k < nsel; k++) {
        const float o = __shfl_sync(kFull, wv, k);
        p += (o > wv) || (o == wv && k < lane);
    }
    int nid = id;
    float nwv = wv;
    for (int k = 0; k < nsel; k++) {
        const int pk = __shfl_sync(kFull, p, k);
        const int ik = __shfl_sync(kFull, id, k);
        const float wk = __shfl_sync(kFull, wv, k);
        if (pk == lane && lane < nsel) {
            nid = ik;
            nwv = wk;
        }
    }
    id = nid;
    wv = nwv;
    float tot = 1e-20f;
    for (int k = 0; k < nsel; k++) tot = __fadd_rn(tot, __shfl_sync(kFull, wv, k));
    const float lim = __fmul_rn(top_p, tot);
    float cum = 0.f;
    int ke = nsel;
    for (int k = 0; k < nsel; k++) {
        cum = __fadd_rn(cum, __shfl_sync(kFull, wv, k));
        if (cum >= lim) {
            ke = k + 1;
            break;
        }
    }
    return ke;
}

// R: the routing of the token by this CTA (sg/ch: shared scratch of E rounded up to 4 floats)
__device__ __noinline__ void route1(const DecParams &P, D1S &m, float *sg, float *ch) {
    const int tid = threadIdx.x, lane = tid % kWarp, warp = tid / kWarp;
    const bool out = blockIdx.x == 0;
    const int E = P.E, E4 = (E + 3) & ~3;
    // 1. logits (fixed-order sum of the partial slices) -> sigmoid scores and choices
    for (int e = tid; e < E4; e += kNT) {
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
    if (tid < kMaxK) m.sel_i[tid] = -1;
    __syncthreads();
    // 2. greedy top-Ksel as ranks: an expert beaten by r others (a higher choice, or an equal
    //    choice and a lower id) is the (r+1)-th pick of the serial scan, which starts at -1e30
    const float4 *c4 = reinterpret_cast<const float4 *>(ch);
    for (int e = tid; e < E; e += kNT) {
        const float cv = ch[e];
        if (!(cv > -1e30f)) continue;
        int r = 0;
        for (int q = 0; q < E4 / 4; q++) {
            const float4 v = c4[q];
            const int e0 = 4 * q;
            r += (v.x > cv) || (v.x == cv && e0 < e);
            r += (v.y > cv) || (v.y == cv && e0 + 1 < e);
            r += (v.z > cv) || (v.z == cv && e0 + 2 < e);
            r += (v.w > cv) || (v.w == cv && e0 + 3 < e);
        }
        if (r < P.Ksel) {
            m.sel_i[r] = e;
            m.sel_w[r] = sg[e];
        }
    }
    __syncthreads();
    // 3. the kept experts, their weights and slots (warp 0, one selection per lane)
    if (warp == 0) {
        const int K = P.K, Ksel = P.Ksel;
        int id = lane < Ksel ? m.sel_i[lane] : -1;
        float wv = lane < Ksel ? m.sel_w[lane] : 0.f;
        const int nsel = __popc(__ballot_sync(kFull, id >= 0));
        if (nsel < Ksel && out && lane == 0) flag_error(P.ctrl, kErrNoCandidate);
        int Ke = nsel;
        if (P.top_p > 0.f && P.top_p < 1.f) Ke = top_p_cut(P.top_p, nsel, id, wv);
        float sm = 1.f;
        if (P.norm_topk) {
            sm = 0.f;
            for (int k = 0; k < Ke; k++) sm = __fadd_rn(sm, __shfl_sync(kFull, wv, k));
            sm = __fadd_rn(sm, 1e-20f);
        }
        const bool kept = lane < Ke;
        const float wn = kept ? (P.norm_topk ? __fdiv_rn(wv, sm) : wv) : 0.f;
        const float wk = kept ? __fmul_rn(wn, P.rscale) : 0.f;
        id = kept ? id : -1;
        int slot = 0;
        for (int k = 0; k < Ke; k++) slot += __shfl_sync(kFull, id, k) < id;
        if (lane < K) {
            m.w[lane] = wk;
            m.pos[lane] = kept ? slot : -1;
            if (kept) m.slot_e[slot] = id;
            if (out) {
                P.idx[lane] = id;
                P.w[lane] = wk;
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
    // 4. bucket counts (CTA 0) and the kept experts' weight pointers (every CTA)
    const int U = m.U;
    if (out) {
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
    if (tid < U) {
        const coli_moe_expert ex = P.experts[m.slot_e[tid]];
        if (bad16(ex.gate_w) || bad16(ex.up_w) || bad16(ex.down_w)) flag_error(P.ctrl, kErrBadExpert);
        m.rec[tid] = rec_of(ex);
    }
    __syncthreads();
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
        [&](int i) {
            int slot, j;
            unit(i, slot, j);
            const Rec &r = m.rec[slot];
            const int jq = min(j + (lane & 1), inter - 1);
            return lane < 2 ? make_float2(__ldg(r.gs + jq), __ldg(r.us + jq)) : make_float2(0.f, 0.f);
        },
        [&](int i, const long long (&s)[4], float2 sc) {
            int slot, j;
            unit(i, slot, j);
            const int jq = j + lane;
            if (lane < 2 && jq < inter) {
                const long long sgt = lane ? s[2] : s[0], sut = lane ? s[3] : s[1];
                const float gv = (__ll2float_rn(sgt) * xinv) * sc.x;
                const float uv = (__ll2float_rn(sut) * xinv) * sc.y;
                const float hv = gv / (1.f + expf(-gv)) * uv;
                P.h[(size_t)(shared ? P.K : slot) * P.ldh + jq] = hv;
                atomicMax(&m.hmax[slot], __float_as_int(fabsf(hv)));
            }
        });
}

// D: down units of `nsl` slots starting at slot0 over this CTA's row groups [gb, gb + ng);
// unit i -> slot slot0 + i / ng, rows 4*(gb + i % ng) .. +3; y goes to ybuf[slot][row - 4*gb].
// rot rotates the warp order so that two calls share the warps evenly.
template <int FMT>
__device__ __noinline__ void down_run(const DecParams &P, D1S &m, const uint8_t *hq, int hq_stride, int slot0, int nsl,
                         int gb, int ng, int rot, float *ybuf) {
    const int lane = threadIdx.x % kWarp;
    const int warp = (threadIdx.x / kWarp + kNW - rot) % kNW;
    const int nu = nsl * ng;
    const int mine = nu > warp ? (nu - warp + kNW - 1) / kNW : 0;
    const bool sh = P.Is > 0 && slot0 == m.U;
    const int inter = sh ? P.Is : P.I;
    const int64_t rb = row_bytes(FMT, inter);
    auto unit = [&](int i, int &slot, int &grp) {
        const int l = warp + kNW * i;
        slot = slot0 + l / ng;
        grp = gb + l % ng;
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
            return reinterpret_cast<const uint4 *>(hq + (size_t)(slot - slot0) * hq_stride);
        },
        [&](int i) {
            int slot, grp;
            unit(i, slot, grp);
            const Rec &r = m.rec[sh ? kShSlot : slot];
            return lane < 4 ? __ldg(r.ds + min(4 * grp + lane, P.H - 1)) : 0.f;
        },
        [&](int i, const long long (&s)[4], float sc) {
            int slot, grp;
            unit(i, slot, grp);
            const int d = 4 * grp + lane;
            if (lane < 4 && d < P.H) {
                const long long sv = lane == 0 ? s[0] : lane == 1 ? s[1] : lane == 2 ? s[2] : s[3];
                ybuf[slot * P.d1_rows + d - 4 * gb] = (__ll2float_rn(sv) * m.hinv[slot]) * sc;
            }
        });
}

template <int RF, int SF>
__global__ void __launch_bounds__(kNT, 2) moe_decode1_kernel(const DecParams P) {
    extern __shared__ __align__(128) uint8_t smem[];
    D1S &m = *reinterpret_cast<D1S *>(smem);
    uint8_t *act = smem + P.d1_act_off;
    float *rsg = reinterpret_cast<float *>(smem + P.d1_rsc_off);
    float *rch = rsg + ((P.E + 3) & ~3);
    float *ybuf = reinterpret_cast<float *>(smem + P.d1_y_off);
    const int tid = threadIdx.x, G = gridDim.x, c = blockIdx.x;
    const bool two = P.Is > 0 && SF != RF;
    uint8_t *xq_r = act, *xq_s = two ? act + 3 * P.H : act;
    const int GUPER = (P.I + 1) / 2;

    if (tid <= kMaxK) m.hmax[tid] = 0;
    if (tid == 0 && P.Is > 0) m.rec[kShSlot] = rec_of(P.shared);
    __syncthreads();
    const int bb = range_lo(P.G_sh, c, G), be = range_lo(P.G_sh, c + 1, G);
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
            __threadfence();
            atomicAdd(&P.ctrl->router_done, 1);
        }
    }
    // ---------------- X, then B: the shared expert's gate/up
    stage_x<RF, SF>(P, xq_r, xq_s, two, m);
    if (be > bb) gateup_run<SF>(P, m, xq_s, bb, be, true);

    // ---------------- R: routing
    if (tid == 0) {
        wait_at_least(&P.ctrl->router_done, P.R, P.ctrl);
        __threadfence();
    }
    __syncthreads();
    route1(P, m, rsg, rch);
    const int U = m.U;

    // ---------------- C: routed gate/up
    const int gu_tot = U * GUPER;
    const int cb = range_lo(gu_tot, c, G), ce = range_lo(gu_tot, c + 1, G);
    gateup_run<RF>(P, m, xq_r, cb, ce, false);
    __syncthreads();
    if (tid < U || (tid == kShSlot && P.Is > 0))
        if (m.hmax[tid] != 0) atomicMax(&P.ctrl->hmax[tid], m.hmax[tid]);
    __syncthreads();
    const int ngr = P.H / 4;
    const int gb = range_lo(ngr, c, G), ge = range_lo(ngr, c + 1, G), ng = ge - gb;
    if (tid == 0) {
        __threadfence();
        atomicAdd(&P.ctrl->gu_all, (be - bb) + (ce - cb));
    }

    // ---------------- D: all h staged, this CTA's output rows for every slot, combine
    if (tid == 0) {
        wait_at_least(&P.ctrl->gu_all, P.G_sh + gu_tot, P.ctrl);
        __threadfence();
    }
    __syncthreads();
    const int nsl = U + (P.Is > 0 ? 1 : 0);
    if (tid < nsl) {
        const int hi = tid < U ? tid : kShSlot;
        const int s = fixed_shift(__int_as_float(__ldcg(&P.ctrl->hmax[hi])));
        m.hshift[tid] = s;
        m.hinv[tid] = ldexpf(1.f, -s);
    }
    __syncthreads();
    const int hs_r = 3 * P.I;  // staged bytes per routed h vector
    uint8_t *hq_s = act + (size_t)U * hs_r;
    {
        const int ir = limb_items<RF>(P.I), is = P.Is > 0 ? limb_items<SF>(P.Is) : 0;
        const int cpr_r = P.I / QGeom<RF>::EPC, cpr_s = P.Is / QGeom<SF>::EPC;
        for (int p = tid; p < U * ir + is; p += kNT) {
            if (p < U * ir) {
                const int u = p / ir;
                stage_limb_item<RF>(P.h + (size_t)u * P.ldh, cpr_r, true,
                                    reinterpret_cast<uint4 *>(act + (size_t)u * hs_r), FixedScale(m.hshift[u]), p - u * ir);
            } else {
                stage_limb_item<SF>(P.h + (size_t)P.K * P.ldh, cpr_s, true, reinterpret_cast<uint4 *>(hq_s),
                                    FixedScale(m.hshift[U]), p - U * ir);
            }
        }
    }
    __syncthreads();
    if (ng > 0) {
        down_run<RF>(P, m, act, hs_r, 0, U, gb, ng, 0, ybuf);
        if (P.Is > 0) down_run<SF>(P, m, hq_s, 0, U, 1, gb, ng, (U * ng) % kNW, ybuf);
    }
    __syncthreads();
    for (int r = tid; r < 4 * ng; r += kNT) {
        const int d = 4 * gb + r;
        float a = 0.f;
        for (int k = 0; k < U; k++) a = __fadd_rn(a, __fmul_rn(m.w[k], ybuf[m.pos[k] * P.d1_rows + r]));
        if (P.Is > 0) a = __fadd_rn(a, ybuf[U * P.d1_rows + r]);
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

size_t decode1_smem_bytes(const DecParams &P) { return (size_t)P.d1_y_off + (size_t)(P.K + 1) * P.d1_rows * 4; }

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
    const size_t h_bytes = (size_t)3 * ((size_t)d.K * d.I + d.I_shared);
    P.d1_act_off = (int)align_up(sizeof(D1S), 128);
    P.d1_rsc_off = P.d1_act_off + (int)align_up(std::max(x_bytes, h_bytes), 128);
    P.d1_y_off = P.d1_rsc_off + (int)align_up((size_t)2 * ((d.E + 3) & ~3) * 4, 128);
    const int ngr = d.H / 4;
    P.d1_rows = 4 * ((ngr + grid - 1) / grid);
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
