// decode.cu — the whole MoE block for decode-sized batches (T <= 64) in ONE persistent launch.
//
// Phases, each split statically and contiguously over the CTAs (two per SM, cooperative
// launch, so every CTA is resident and a wait is only ever on an earlier phase):
//   A  router logits (colibri-strix c/glm.c @98759bf moe() phase A; r_router shader):
//      T <= 8: router items — partial logits of 32 experts over one slice of H; T > 8: the
//      partials come from a router launch before this kernel, and CTA t routes token t alone
//      (logits, picks, kept weights: route_token), writing its row of the routing outputs.
//   B  shared expert gate/up rows (independent of routing: runs while A completes)
//   R  routing, by EVERY CTA for itself once all partials are in (one counter wait; T > 8: once
//      every token CTA has written its picks, which every CTA then loads): logits
//      summed in a fixed order, sigmoid, bias, greedy top-K with ties to the lower index
//      (select.cuh, one warp per token), TOPK/TOPP, renorm, routed scale, stable token->expert buckets and
//      the unit tables — all in shared memory; CTA 0 also writes the routing outputs. Running
//      it everywhere keeps a cold, single-CTA step off the critical path.
//   C  routed gate/up rows: h = silu(gate.x * s_g) * (up.x * s_u)   (moe() phases C/D)
//   D  down rows: y = (down.h) * s_d, for every selected expert and the shared one
//   E  combine: out = sum_k w_k y_k in selection order + y_shared   (moe() phases C/D/E)
// Units of B/C are two row pairs (gate and up rows j, j+1) of one expert for one group of up to
// NV tokens; units of D are four down rows. Each phase's units are handed out in chunks by an
// atomic counter (CTAs whose units are cheaper take more). A CTA walks its share in pieces that
// have the same expert and tokens: the piece's activations are staged once in shared memory,
// then each warp streams its units' rows with 16-byte loads kept ahead in registers across unit
// boundaries. A single-token group runs the integer core (x as fixed-point limbs, idot.cuh);
// a group of 2-4 tokens runs the tensor-core core (x as f16 hi + lo parts, mma.cuh) on blocks
// of 16 rows.
// Dependencies are counters in the workspace: router items -> routing, gate/up -> down (raised
// once per CTA per expert), down -> combine (once per CTA). Every wait is bounded (2 s of
// %globaltimer); on expiry the kernel records kErrWaitExpired and carries on, so a fault in the
// schedule can not hang the GPU.
#include <algorithm>

#include "decode_parts.cuh"
#include "select.cuh"

namespace colimoe {

namespace {

// ------------------------------------------------------------------ routing
// This CTA's copy of the routing result (shared memory, alive until the kernel ends).
struct RTab {
    int *slot_e, *slot_n, *slot_pbase, *slot_groups;  // [E+1]: slot u < U routed, U shared
    int *gu_off, *dn_off;                             // [E+2]: units before slot u
    int *perm, *pos;                                  // [T*K]
    float *w;                                         // [T*K] kept weights (0 beyond keff)
    int *keff;                                        // [T]
    int *U;
};

size_t rtab_bytes(int T, int E, int K) {
    return (size_t)(4 * (E + 1) + 2 * (E + 2) + 3 * T * K + T + 16) * 4;
}

__device__ __forceinline__ RTab rtab_of(void *base, int T, int E, int K) {
    RTab r;
    int *p = static_cast<int *>(base);
    r.slot_e = p;
    r.slot_n = r.slot_e + (E + 1);
    r.slot_pbase = r.slot_n + (E + 1);
    r.slot_groups = r.slot_pbase + (E + 1);
    r.gu_off = r.slot_groups + (E + 1);
    r.dn_off = r.gu_off + (E + 2);
    r.perm = r.dn_off + (E + 2);
    r.pos = r.perm + T * K;
    r.w = reinterpret_cast<float *>(r.pos + T * K);
    r.keff = reinterpret_cast<int *>(r.w + T * K);
    r.U = r.keff + T;
    return r;
}

// Scratch of the routing step (inside the activation staging buffer).
struct RScratch {
    float *sg, *ch;          // [T][sel_padded(E)] sigmoid scores, choices (-inf past E)
    int *sel_i;              // [T][K] picks in selection order, then the kept ids (-1 past keff)
    float2 *cand;            // [kNW][sel_cand_cap(E, Ksel)] selection candidates of each warp
    int *cnt, *off, *fill, *chk, *actv, *wc, *tmp;
};

__device__ __forceinline__ RScratch rscratch_of(void *base, const DecParams &P) {
    RScratch s;
    const int TE = P.T * sel_padded(P.E), TK = P.T * P.K, E = P.E;
    s.sg = static_cast<float *>(base);
    s.ch = s.sg + TE;
    s.cand = reinterpret_cast<float2 *>(s.ch + TE);
    s.sel_i = reinterpret_cast<int *>(s.cand + kNW * sel_cand_cap(E, P.Ksel));
    s.cnt = s.sel_i + TK;
    s.off = s.cnt + E;
    s.fill = s.off + E;
    s.chk = s.fill + E;
    s.actv = s.chk + E;
    s.wc = s.actv + E;
    s.tmp = s.wc + kNW * E;
    return s;
}

size_t rscratch_bytes(int T, int E, int K, int Ksel) {
    return (size_t)(2 * T * sel_padded(E) + 2 * kNW * sel_cand_cap(E, Ksel) + T * K + 5 * E + kNW * E + 16 + 16) * 4;
}

// exclusive scan in place of n <= 2048 ints in shared memory by the CTA; returns the total
__device__ int scan_smem(int *a, int n, int *tmp) {
    const int tid = threadIdx.x, lane = tid % kWarp, warp = tid / kWarp;
    int loc[8], sum = 0;
#pragma unroll
    for (int i = 0; i < 8; i++) {
        const int j = tid * 8 + i;
        loc[i] = j < n ? a[j] : 0;
        sum += loc[i];
    }
    int inc = sum;
#pragma unroll
    for (int o = 1; o < kWarp; o <<= 1) {
        const int v = __shfl_up_sync(kFull, inc, o);
        if (lane >= o) inc += v;
    }
    if (lane == kWarp - 1) tmp[warp] = inc;
    __syncthreads();
    if (tid == 0) {
        int run = 0;
        for (int w = 0; w < kNW; w++) {
            const int v = tmp[w];
            tmp[w] = run;
            run += v;
        }
        tmp[kNW] = run;
    }
    __syncthreads();
    int run = tmp[warp] + inc - sum;
#pragma unroll
    for (int i = 0; i < 8; i++) {
        const int j = tid * 8 + i;
        if (j < n) a[j] = run;
        run += loc[i];
    }
    const int total = tmp[kNW];
    __syncthreads();
    return total;
}

// T > 8: CTA t routes token t alone, with all its threads (at most kTokSlices partial slices): the logits are the fixed-order sum
// of the nks partial slices, then sigmoid and bias; the picks by the whole CTA (select.cuh), the
// kept weights by warp 0. The token's rows of the routing outputs go to the workspace / caller,
// then the CTA raises routed_done. scratch: shared memory of at least rscratch_bytes.
__device__ __noinline__ void route_token(const DecParams &P, int t, float *scratch) {
    const int tid = threadIdx.x, lane = tid % kWarp, warp = tid / kWarp;
    const int T = P.T, E = P.E, K = P.K, Ep = sel_padded(E);
    float *sg = scratch, *ch = sg + Ep;
    float2 *cand = reinterpret_cast<float2 *>(ch + Ep);
    int *nc = reinterpret_cast<int *>(cand + sel_cand_cap(E, P.Ksel));  // candidates, selectable
    int *sel_i = nc + 2;
    for (int e = tid; e < Ep; e += kNT) {
        float sv = 0.f, cv = -INFINITY;
        if (e < E) {
            float a[kTokSlices];
            const size_t j = (size_t)t * E + e;
#pragma unroll
            for (int k = 0; k < kTokSlices; k++)
                if (k < P.nks) a[k] = __ldcg(P.part + (size_t)k * T * E + j);
            float lg = 0.f;
#pragma unroll
            for (int k = 0; k < kTokSlices; k++)
                if (k < P.nks) lg += a[k];
            sv = 1.f / (1.f + expf(-lg));
            cv = sv + __ldg(P.bias + e);
            P.sig[j] = sv;
            P.choice[j] = cv;
        }
        sg[e] = sv;
        ch[e] = cv;
    }
    if (tid == 0) nc[0] = nc[1] = 0;
    __syncthreads();
    sel_topk_cta(ch, E, P.Ksel, cand, &nc[0], &nc[1], sel_i);
    if (warp == 0) {
        const int nsel = min(nc[1], P.Ksel);
        if (nsel < P.Ksel && lane == 0) flag_error(P.ctrl, kErrNoCandidate);
        const int pick = lane < nsel ? sel_i[lane] : -1;
        const SelKept kp = sel_finish_warp(nsel, pick, lane < nsel ? sg[pick] : 0.f, P.top_p, P.norm_topk, P.rscale);
        if (lane < K) {
            P.idx[(size_t)t * K + lane] = kp.id;
            P.w[(size_t)t * K + lane] = kp.w;
        }
        if (lane == 0) P.keff[t] = kp.ke;
    }
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        atomicAdd(&P.ctrl->routed_done, 1);
    }
}

// The routing of all T tokens into this CTA's tables: from the logits (the fixed-order sum of
// the nks partial slices, T <= 8) or, from_tokens, from the kept picks and weights the token
// CTAs wrote (T > 8). Results go to rt; CTA 0 also writes the routing outputs of the workspace /
// caller that the token CTAs do not.
__device__ __noinline__ void route_local(const DecParams &P, float *scratch, const RTab &rt, bool from_tokens) {
    const int tid = threadIdx.x, lane = tid % kWarp, warp = tid / kWarp;
    const bool out = blockIdx.x == 0;
    const RScratch s = rscratch_of(scratch, P);
    const int T = P.T, E = P.E, K = P.K, Ep = sel_padded(E), TE = T * Ep;
    if (from_tokens) {
        for (int i = tid; i < T * K; i += kNT) {
            s.sel_i[i] = __ldcg(P.idx + i);
            rt.w[i] = __ldcg(P.w + i);
        }
        for (int t = tid; t < T; t += kNT) rt.keff[t] = __ldcg(P.keff + t);
    } else {
        // 1. logits -> sigmoid scores and choices, rows padded to whole selection blocks
        for (int i = tid; i < TE; i += kNT) {
            const int t = i / Ep, e = i - t * Ep;
            float sv = 0.f, cv = -INFINITY;
            if (e < E) {
                float a[16];
                const size_t j = (size_t)t * E + e;
#pragma unroll
                for (int k = 0; k < 16; k++)
                    if (k < P.nks) a[k] = __ldcg(P.part + (size_t)k * T * E + j);
                float lg = 0.f;
#pragma unroll
                for (int k = 0; k < 16; k++)
                    if (k < P.nks) lg += a[k];
                sv = 1.f / (1.f + expf(-lg));
                cv = sv + P.bias[e];
                if (out) {
                    P.sig[j] = sv;
                    P.choice[j] = cv;
                }
            }
            s.sg[i] = sv;
            s.ch[i] = cv;
        }
        __syncthreads();
        // 2. per token, one warp: the picks (select.cuh), then TOPP, renormalisation and routed
        //    scale in the serial code's float order
        float2 *cand = s.cand + warp * sel_cand_cap(E, P.Ksel);
        for (int t = warp; t < T; t += kNW) {
            int *id = s.sel_i + t * K;
            const int nsel = sel_topk_warp(s.ch + t * Ep, E, P.Ksel, cand, id);
            if (nsel < P.Ksel && out && lane == 0) flag_error(P.ctrl, kErrNoCandidate);
            const int pick = lane < nsel ? id[lane] : -1;
            const SelKept kp = sel_finish_warp(nsel, pick, lane < nsel ? s.sg[t * Ep + pick] : 0.f, P.top_p,
                                               P.norm_topk, P.rscale);
            __syncwarp();
            if (lane < K) {
                id[lane] = kp.id;
                rt.w[t * K + lane] = kp.w;
                if (out) {
                    P.idx[(size_t)t * K + lane] = kp.id;
                    P.w[(size_t)t * K + lane] = kp.w;
                }
            }
            if (lane == 0) {
                rt.keff[t] = kp.ke;
                if (out) P.keff[t] = kp.ke;
            }
        }
    }
    __syncthreads();
    // 4. buckets and the unit tables (slot u < U: u-th active expert, ascending id; U: shared)
    const int GUPER = (P.I + 1) / 2, DNPER = (P.H + 3) / 4;
    int U;
    if (T == 1) {  // one token: its kept experts are distinct
        const int Ke = rt.keff[0];
        if (out) {
            for (int e = tid; e < E; e += kNT) {
                int c = 0, o = 0;
                for (int k = 0; k < Ke; k++) {
                    const int ek = s.sel_i[k];
                    c += ek == e;
                    o += ek < e;
                }
                P.counts[e] = c;
                P.offsets[e] = o;
            }
            if (tid == 0) P.offsets[E] = Ke;
        }
        if (tid < K) {
            if (tid < Ke) {
                const int e = s.sel_i[tid];
                int slot = 0;
                for (int k = 0; k < Ke; k++) slot += s.sel_i[k] < e;
                rt.slot_e[slot] = e;
                rt.slot_n[slot] = 1;
                rt.slot_pbase[slot] = slot;
                rt.slot_groups[slot] = 1;
                rt.perm[slot] = tid;
                rt.pos[tid] = slot;
                if (out) {
                    P.act[slot] = e;
                    P.perm[slot] = tid;
                    P.pos[tid] = slot;
                }
            } else {
                rt.pos[tid] = -1;
                if (out) P.pos[tid] = -1;
            }
        }
        U = Ke;
        for (int u = tid; u <= U + 1; u += kNT) {
            rt.gu_off[u] = min(u, U) * GUPER;
            rt.dn_off[u] = min(u, U) * DNPER + (u > U && P.Is > 0 ? P.groups_sh * DNPER : 0);
        }
    } else {
        const int N = T * K;
        for (int e = tid; e < E; e += kNT) {
            s.cnt[e] = 0;
            s.fill[e] = 0;
        }
        __syncthreads();
        auto expert_of = [&](int a) -> int { return a < N ? s.sel_i[a] : -1; };  // -1 when not kept
        for (int a = tid; a < N; a += kNT) {
            const int e = expert_of(a);
            if (e >= 0) atomicAdd(&s.cnt[e], 1);
        }
        __syncthreads();
        for (int e = tid; e < E; e += kNT) {
            s.off[e] = s.cnt[e];
            s.actv[e] = s.cnt[e] > 0 ? 1 : 0;
            if (out) P.counts[e] = s.cnt[e];
        }
        __syncthreads();
        const int total = scan_smem(s.off, E, s.tmp);
        U = scan_smem(s.actv, E, s.tmp);
        for (int e = tid; e < E; e += kNT) {
            if (out) P.offsets[e] = s.off[e];
            if (s.cnt[e] > 0) {
                const int u = s.actv[e];
                const int g = (s.cnt[e] + P.NV - 1) / P.NV;
                rt.slot_e[u] = e;
                rt.slot_n[u] = s.cnt[e];
                rt.slot_pbase[u] = s.off[e];
                rt.slot_groups[u] = g;
                rt.gu_off[u] = g * GUPER;
                rt.dn_off[u] = g * DNPER;
                if (out) P.act[u] = e;
            }
        }
        if (tid == 0) {
            if (out) P.offsets[E] = total;
            rt.gu_off[U] = 0;
            rt.dn_off[U] = P.Is > 0 ? P.groups_sh * DNPER : 0;
        }
        __syncthreads();
        const int gu_tot = scan_smem(rt.gu_off, U + 1, s.tmp);
        const int dn_tot = scan_smem(rt.dn_off, U + 1, s.tmp);
        if (tid == 0) {
            rt.gu_off[U + 1] = gu_tot;
            rt.dn_off[U + 1] = dn_tot;
        }
        // stable perm / pos: 256-assignment chunks in order; inside a chunk, rank within the
        // warp from a match-any mask, then the warps' per-expert counts are scanned
        for (int a0 = 0; a0 < N; a0 += kNT) {
            for (int i = tid; i < kNW * E; i += kNT) s.wc[i] = 0;
            __syncthreads();
            const int a = a0 + tid;
            const int e = expert_of(a);
            const unsigned peers = __match_any_sync(kFull, e);
            const int rank = __popc(peers & ((1u << lane) - 1u));
            if (e >= 0 && rank == 0) s.wc[warp * E + e] = __popc(peers);
            __syncthreads();
            for (int x = tid; x < E; x += kNT) {
                int run = 0;
                for (int w = 0; w < kNW; w++) {
                    const int v = s.wc[w * E + x];
                    s.wc[w * E + x] = run;
                    run += v;
                }
                s.chk[x] = run;
            }
            __syncthreads();
            if (a < N) {
                const int p = e >= 0 ? s.off[e] + s.fill[e] + s.wc[warp * E + e] + rank : -1;
                if (e >= 0) rt.perm[p] = a;
                rt.pos[a] = p;
                if (out) {
                    if (e >= 0) P.perm[p] = a;
                    P.pos[a] = p;
                }
            }
            __syncthreads();
            for (int x = tid; x < E; x += kNT) s.fill[x] += s.chk[x];
            __syncthreads();
        }
    }
    if (tid == 0) {
        *rt.U = U;
        rt.slot_e[U] = -1;  // the shared expert
        rt.slot_n[U] = T;
        rt.slot_pbase[U] = 0;
        rt.slot_groups[U] = P.groups_sh;
    }
    __syncthreads();
}

// ------------------------------------------------------------------ expert phases
constexpr int kScCap = 64;  // units per segment piece: their row scales are staged in smem

struct Seg {  // one segment piece: units of one expert and token group (broadcast in smem)
    const uint8_t *w0, *w1;  // gate and up rows, or down rows in w0
    const float *s0, *s1;    // their row scales
    int fmt, inter, n, pbase, shared, tg, key, need, nv;
    int ulo, uhi;            // units [ulo, uhi) of this CTA in the piece
    int ubase;               // unit index of the token group's first unit
};

// per-CTA scratch next to the staged activations and the routing tables
struct Misc {
    Seg sg;
    int skey[4];
    int chunk;                // the chunk this CTA took from a phase queue
    int xshift;               // integer core: X = round(x * 2^xshift)
    float xinv;               // 2^-xshift
    float redf[kNW];
    float redv[4][kNW];       // tensor-core staging: per-token max |x| of each warp
    float vf[4][2];           // ... the two exact factors of 2^e of each token
    float vinv[4];            // ... and 2^-e
    float sc[2][4 * kScCap];  // row scales of the piece's units (gate/up: gate, up; down: [0])
};

// One vector in 24-bit block fixed point for the integer core (idot.cuh); leaves s and 2^-s in
// m (published by the caller's next barrier).
template <int FMT>
__device__ void stage_limbs(const float *__restrict__ src, int len, bool coherent, uint8_t *xq, Misc &m) {
    const int tid = threadIdx.x, lane = tid % kWarp, warp = tid / kWarp;
    const int CPR = len / QGeom<FMT>::EPC, n4 = len / 4;
    constexpr int B = 4;
    float mx = 0.f;
    for (int q0 = tid; q0 < n4; q0 += kNT * B) {
        float4 v[B];
#pragma unroll
        for (int j = 0; j < B; j++) {
            const int q = q0 + j * kNT;
            if (q < n4) v[j] = ld_act4(src, q, coherent);
        }
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
    stage_limbs_vec<FMT>(src, len, coherent, xq, FixedScale(s), tid, kNT);
    if (tid == 0) {
        m.xshift = s;
        m.xinv = ldexpf(1.f, -s);
    }
}

// Multi-token groups: the group's vectors as f16 hi/lo parts in the tensor-core layout
// (mma.cuh), token v scaled by its own 2^e so that max|x_v| * 2^e lies in [2^14, 2^15).
template <int FMT, class SrcOf>
__device__ void stage_mma(SrcOf src_of, int nv, int len, bool coherent, uint8_t *xs, size_t stride, Misc &m) {
    const int tid = threadIdx.x, lane = tid % kWarp, warp = tid / kWarp;
    const int n4 = len / 4;
    for (int v = 0; v < nv; v++) {
        const float *src = src_of(v);
        float mx = 0.f;
        for (int q = tid; q < n4; q += kNT) {
            const float4 a = ld_act4(src, q, coherent);
            mx = fmaxf(mx, fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(a.z), fabsf(a.w))));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
        if (lane == 0) m.redv[v][warp] = mx;
    }
    __syncthreads();
    if (tid < nv) {
        float mx = m.redv[tid][0];
#pragma unroll
        for (int w = 1; w < kNW; w++) mx = fmaxf(mx, m.redv[tid][w]);
        int e = 0;
        if (mx > 0.f) {
            const int ex = (int)((__float_as_uint(mx) >> 23) & 255u);
            e = 14 - (ex == 0 ? -126 : ex - 127);
        }
        const int e1 = max(-126, min(126, e)), e2 = e - e1;
        m.vf[tid][0] = __int_as_float((e1 + 127) << 23);
        m.vf[tid][1] = __int_as_float((e2 + 127) << 23);
        m.vinv[tid] = ldexpf(1.f, -e);
    }
    __syncthreads();
    const int items = mma_items<FMT>(len);
    for (int idx = tid; idx < nv * items; idx += kNT) {
        const int v = idx / items, it = idx - v * items;
        stage_mma_item<FMT>(src_of(v), len, coherent, xs + (size_t)v * stride, m.vf[v][0], m.vf[v][1], it);
    }
}

__device__ __noinline__ void stage_acts(const DecParams &P, const RTab &rt, const Seg &g, bool down, void *xs,
                                        Misc &m) {
    const int len = down ? g.inter : P.H;
    auto src_of = [&](int v) -> const float * {
        const int pv = g.tg * P.NV + v;
        if (down) {
            const int row = g.shared ? P.T * P.K + pv : g.pbase + pv;
            return P.h + (size_t)row * P.ldh;
        }
        const int t = g.shared ? pv : rt.perm[g.pbase + pv] / P.K;
        return P.x + (size_t)t * P.H;
    };
    uint8_t *xq = static_cast<uint8_t *>(xs);
    if (g.nv == 1) {
        if (g.fmt == COLI_FMT_INT4) stage_limbs<COLI_FMT_INT4>(src_of(0), len, down, xq, m);
        else if (g.fmt == COLI_FMT_INT8) stage_limbs<COLI_FMT_INT8>(src_of(0), len, down, xq, m);
        else stage_limbs<COLI_FMT_INT2>(src_of(0), len, down, xq, m);
        return;
    }
    const size_t stride = (size_t)P.xs_stride * 4;
    if (g.fmt == COLI_FMT_INT4) stage_mma<COLI_FMT_INT4>(src_of, g.nv, len, down, xq, stride, m);
    else if (g.fmt == COLI_FMT_INT8) stage_mma<COLI_FMT_INT8>(src_of, g.nv, len, down, xq, stride, m);
    else stage_mma<COLI_FMT_INT2>(src_of, g.nv, len, down, xq, stride, m);
}

// h or y row of token v of the piece's group
__device__ __forceinline__ int act_row(const DecParams &P, const Seg &g, int v) {
    const int pv = g.tg * P.NV + v;
    return g.shared ? P.T * P.K + pv : g.pbase + pv;
}

// gate/up: a unit is two row pairs (rows j and j+1 of gate and of up)
template <int FMT>
__device__ void gateup_units_int(const DecParams &P, const Seg &g, const void *xs, const Misc &m) {
    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
    const int nu = g.uhi - g.ulo;
    const int mine = nu > warp ? (nu - warp + kNW - 1) / kNW : 0;
    const int64_t rb = row_bytes(FMT, P.H);
    const int ubase = g.ulo - g.ubase;
    const float xinv = m.xinv;
    float *hrow = P.h + (size_t)act_row(P, g, 0) * P.ldh;
    warp_stream_int<FMT, 4>(
        mine, (int)(rb / 16), lane,
        [&](int i, const uint8_t *(&rr)[4]) {
            const int j = 2 * (ubase + warp + kNW * i);
            const int j1 = min(j + 1, g.inter - 1);
            rr[0] = g.w0 + (size_t)j * rb;
            rr[1] = g.w1 + (size_t)j * rb;
            rr[2] = g.w0 + (size_t)j1 * rb;
            rr[3] = g.w1 + (size_t)j1 * rb;
        },
        [&](int) { return static_cast<const uint4 *>(xs); }, [](int) { return 0; },
        [&](int i, long long tot, int) {  // lanes 0 / 16 hold gate j / j+1, lanes 8 / 24 up
            const long long su = __shfl_down_sync(kFull, tot, 8);
            const int lj = 2 * (warp + kNW * i) + (lane >> 4);  // row within the piece's scales
            const int jq = 2 * ubase + lj;
            if ((lane & 15) == 0 && jq < g.inter) {
                const float gv = (__ll2float_rn(tot) * xinv) * m.sc[0][lj];
                const float uv = (__ll2float_rn(su) * xinv) * m.sc[1][lj];
                hrow[jq] = gv / (1.f + expf(-gv)) * uv;
            }
        });
}

// Multi-token groups (tensor cores): blocks of 8 row pairs, gate row j in MMA row g and up
// row j in row g + 8, so lane (g, c < 2) ends with gate and up of row pair g for tokens 2c, 2c + 1.
template <int FMT>
__device__ void gateup_units_mma(const DecParams &P, const Seg &g, const uint8_t *xs, const Misc &m) {
    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
    const int gq = lane >> 2, c = lane & 3;
    const int jlo = 2 * (g.ulo - g.ubase);                    // first row pair of the piece
    const int np = min(2 * (g.uhi - g.ulo), g.inter - jlo);  // row pairs of the piece
    const int nb = (np + 7) / 8;
    const int mine = nb > warp ? (nb - warp + kNW - 1) / kNW : 0;
    const int64_t rb = row_bytes(FMT, P.H);
    const int tok = (gq & 3) < g.nv ? (gq & 3) : 0;
    const uint8_t *xb = xs + (size_t)tok * P.xs_stride * 4 + (gq >> 2) * 64 + c * 16;
    warp_stream_mma<FMT>(
        mine, (int)(rb / 16), xb, lane,
        [&](int i, const uint8_t *(&rr)[2]) {
            const int j = min(jlo + 8 * (warp + kNW * i) + gq, g.inter - 1);
            rr[0] = g.w0 + (size_t)j * rb;
            rr[1] = g.w1 + (size_t)j * rb;
        },
        [&](int i, float (&d)[4]) {
#pragma unroll
            for (int q = 0; q < 4; q++) d[q] += __shfl_xor_sync(kFull, d[q], 2);  // hi + lo columns
            const int lj = 8 * (warp + kNW * i) + gq;
            if (c < 2 && lj < np) {
#pragma unroll
                for (int t = 0; t < 2; t++) {
                    const int v = 2 * c + t;
                    if (v < g.nv) {
                        const float gv = (d[t] * m.vinv[v]) * m.sc[0][lj];
                        const float uv = (d[2 + t] * m.vinv[v]) * m.sc[1][lj];
                        P.h[(size_t)act_row(P, g, v) * P.ldh + jlo + lj] = gv / (1.f + expf(-gv)) * uv;
                    }
                }
            }
        });
}

// down: a unit is four consecutive rows
template <int FMT>
__device__ void down_units_int(const DecParams &P, const Seg &g, const void *xs, const Misc &m) {
    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
    const int nu = g.uhi - g.ulo;
    const int mine = nu > warp ? (nu - warp + kNW - 1) / kNW : 0;
    const int64_t rb = row_bytes(FMT, g.inter);
    const int ubase = g.ulo - g.ubase;
    const float xinv = m.xinv;
    float *yrow = P.y + (size_t)act_row(P, g, 0) * P.H;
    warp_stream_int<FMT, 4>(
        mine, (int)(rb / 16), lane,
        [&](int i, const uint8_t *(&rr)[4]) {
            const int d = 4 * (ubase + warp + kNW * i);
#pragma unroll
            for (int q = 0; q < 4; q++) rr[q] = g.w0 + (size_t)min(d + q, P.H - 1) * rb;
        },
        [&](int) { return static_cast<const uint4 *>(xs); }, [](int) { return 0; },
        [&](int i, long long tot, int) {  // lane 8q holds row q
            const int ld = 4 * (warp + kNW * i) + (lane >> 3);
            const int d = 4 * ubase + ld;
            if ((lane & 7) == 0 && d < P.H) yrow[d] = (__ll2float_rn(tot) * xinv) * m.sc[0][ld];
        });
}

// Multi-token groups (tensor cores): blocks of 16 consecutive down rows.
template <int FMT>
__device__ void down_units_mma(const DecParams &P, const Seg &g, const uint8_t *xs, const Misc &m) {
    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
    const int gq = lane >> 2, c = lane & 3;
    const int dlo = 4 * (g.ulo - g.ubase);
    const int nr = min(4 * (g.uhi - g.ulo), P.H - dlo);
    const int nb = (nr + 15) / 16;
    const int mine = nb > warp ? (nb - warp + kNW - 1) / kNW : 0;
    const int64_t rb = row_bytes(FMT, g.inter);
    const int tok = (gq & 3) < g.nv ? (gq & 3) : 0;
    const uint8_t *xb = xs + (size_t)tok * P.xs_stride * 4 + (gq >> 2) * 64 + c * 16;
    warp_stream_mma<FMT>(
        mine, (int)(rb / 16), xb, lane,
        [&](int i, const uint8_t *(&rr)[2]) {
            const int r = dlo + 16 * (warp + kNW * i) + gq;
            rr[0] = g.w0 + (size_t)min(r, P.H - 1) * rb;
            rr[1] = g.w0 + (size_t)min(r + 8, P.H - 1) * rb;
        },
        [&](int i, float (&d)[4]) {
#pragma unroll
            for (int q = 0; q < 4; q++) d[q] += __shfl_xor_sync(kFull, d[q], 2);
            const int ld = 16 * (warp + kNW * i) + gq;
            if (c < 2) {
#pragma unroll
                for (int t = 0; t < 2; t++) {
                    const int v = 2 * c + t;
                    if (v < g.nv) {
                        float *yrow = P.y + (size_t)act_row(P, g, v) * P.H + dlo;
                        if (ld < nr) yrow[ld] = (d[t] * m.vinv[v]) * m.sc[0][ld];
                        if (ld + 8 < nr) yrow[ld + 8] = (d[2 + t] * m.vinv[v]) * m.sc[0][ld + 8];
                    }
                }
            }
        });
}

template <int FMT>
__device__ void run_units_mma_fmt(const DecParams &P, const Seg &g, bool down, const uint8_t *xs, const Misc &m) {
    if (down) down_units_mma<FMT>(P, g, xs, m);
    else gateup_units_mma<FMT>(P, g, xs, m);
}

template <int NV>
__device__ void run_units(const DecParams &P, const Seg &g, bool down, const void *xs, const Misc &m) {
    if (g.nv == 1) {
        if (down) {
            if (g.fmt == COLI_FMT_INT4) down_units_int<COLI_FMT_INT4>(P, g, xs, m);
            else if (g.fmt == COLI_FMT_INT8) down_units_int<COLI_FMT_INT8>(P, g, xs, m);
            else down_units_int<COLI_FMT_INT2>(P, g, xs, m);
        } else {
            if (g.fmt == COLI_FMT_INT4) gateup_units_int<COLI_FMT_INT4>(P, g, xs, m);
            else if (g.fmt == COLI_FMT_INT8) gateup_units_int<COLI_FMT_INT8>(P, g, xs, m);
            else gateup_units_int<COLI_FMT_INT2>(P, g, xs, m);
        }
        return;
    }
    if constexpr (NV > 1) {
        const uint8_t *xq = static_cast<const uint8_t *>(xs);
        if (g.fmt == COLI_FMT_INT4) run_units_mma_fmt<COLI_FMT_INT4>(P, g, down, xq, m);
        else if (g.fmt == COLI_FMT_INT8) run_units_mma_fmt<COLI_FMT_INT8>(P, g, down, xq, m);
        else run_units_mma_fmt<COLI_FMT_INT2>(P, g, down, xq, m);
    }
}

// first index i in [0, n) with off[i+1] > x, off in shared memory
__device__ __forceinline__ int upper_slot_smem(const int *off, int n, int x) {
    int lo = 0, hi = n - 1;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (off[mid + 1] > x) hi = mid;
        else lo = mid + 1;
    }
    return lo;
}

// fill the piece of unit l (thread 0 only). Unit spaces run slot by
// slot, then token group, then unit; shared_phase: the shared expert's gate/up before routing.
__device__ __noinline__ void make_seg(const DecParams &P, const RTab &rt, int slot, int U, int slot_base, int l,
                                      int e_share, bool down, bool shared_phase, Seg &g) {
    const int GUPER = (P.I + 1) / 2, GUPER_SH = (P.Is + 1) / 2, DNPER = (P.H + 3) / 4;
    const bool shared = shared_phase || slot == U;
    coli_moe_expert ex;
    int n, pbase, groups;
    if (shared) {
        ex = P.shared;
        n = P.T;
        pbase = 0;
        groups = P.groups_sh;
    } else {
        ex = P.experts[rt.slot_e[slot]];
        n = rt.slot_n[slot];
        pbase = rt.slot_pbase[slot];
        groups = rt.slot_groups[slot];
        if (bad16(ex.gate_w) || bad16(ex.up_w) || bad16(ex.down_w)) flag_error(P.ctrl, kErrBadExpert);
    }
    g.w0 = static_cast<const uint8_t *>(down ? ex.down_w : ex.gate_w);
    g.w1 = static_cast<const uint8_t *>(ex.up_w);
    g.s0 = down ? ex.down_s : ex.gate_s;
    g.s1 = ex.up_s;
    g.fmt = shared ? P.sfmt : P.rfmt;
    g.inter = shared ? P.Is : P.I;
    g.n = n;
    g.pbase = pbase;
    g.shared = shared ? 1 : 0;
    g.key = shared ? kSharedKey : slot;
    g.need = shared ? P.G_sh : groups * GUPER;
    const int per = down ? DNPER : (shared ? GUPER_SH : GUPER);
    const int local = l - slot_base;
    g.tg = local / per;
    g.nv = min(P.NV, n - g.tg * P.NV);
    g.ubase = slot_base + g.tg * per;
    g.ulo = l;
    g.uhi = min(min(e_share, g.ubase + per), l + kScCap);
}

// walk this CTA's share [b, e) of a unit space piece by piece; off/nslots: the unit prefix
// over the slots (shared memory), unused in the shared phase
template <int NV>
__device__ void run_share(const DecParams &P, const RTab &rt, int b, int e, bool down, bool shared_phase,
                          const int *off, int nslots, int U, void *xs, Misc &m) {
    const int tid = threadIdx.x;
    if (b >= e) return;
    int slot = 0, slot_base = 0, slot_end = 0, done_in_slot = 0;
    if (tid == 0) {
        if (shared_phase) {
            slot_end = P.G_sh;
        } else {
            slot = upper_slot_smem(off, nslots, b);
            slot_base = off[slot];
            slot_end = off[slot + 1];
        }
    }
    int l = b;
    while (l < e) {
        __syncthreads();  // the previous piece's units are done with xs, sg and sc
        if (tid == 0) {
            while (l >= slot_end) {
                slot++;
                slot_base = slot_end;
                slot_end = off[slot + 1];
            }
            make_seg(P, rt, slot, U, slot_base, l, min(e, slot_end), down, shared_phase, m.sg);
        }
        __syncthreads();
        const Seg g = m.sg;
        // row scales of the piece (loads issued before any wait or staging)
        const int nrow = down ? 4 * (g.uhi - g.ulo) : 2 * (g.uhi - g.ulo);
        const int r0 = (down ? 4 : 2) * (g.ulo - g.ubase);
        const int rlim = down ? P.H : g.inter;
        float sv0 = 0.f, sv1 = 0.f;
        if (tid < nrow && r0 + tid < rlim) {
            sv0 = __ldg(g.s0 + r0 + tid);
            if (!down) sv1 = __ldg(g.s1 + r0 + tid);
        }
        if (down) {  // this expert's h rows must all be written
            if (tid == 0) {
                wait_at_least(&P.ctrl->gu_done[g.key], g.need, P.ctrl);
                __threadfence();
            }
            __syncthreads();
        }
        // activations: skip restaging when xs already holds them (same kind, tokens and format)
        const int k0 = (down ? 2 : 1) + (g.nv == 1 ? 4 : 0);
        const int k1 = down ? g.key : (P.T == 1 ? 0 : (g.shared ? -1 : g.pbase));
        const int k2 = (P.T == 1 && !down) ? g.fmt : g.tg * 8 + g.fmt;
        if (!(m.skey[0] == k0 && m.skey[1] == k1 && m.skey[2] == k2)) {
            stage_acts(P, rt, g, down, xs, m);
            if (tid == 0) {
                m.skey[0] = k0;
                m.skey[1] = k1;
                m.skey[2] = k2;
            }
        }
        if (tid < nrow) {
            m.sc[0][tid] = sv0;
            m.sc[1][tid] = sv1;
        }
        __syncthreads();
        run_units<NV>(P, g, down, xs, m);
        l = g.uhi;
        if (!down) {  // publish this CTA's gate/up units of the expert when its run ends
            __syncthreads();  // every warp's h stores precede thread 0's release
            if (tid == 0) {
                done_in_slot += g.uhi - g.ulo;
                if (l >= e || l >= slot_end) {
                    __threadfence();
                    atomicAdd(&P.ctrl->gu_done[g.key], done_in_slot);
                    done_in_slot = 0;
                }
            }
        }
    }
    __syncthreads();
}

constexpr int kChunk = 128;  // units per chunk of a phase queue (two pieces of one group share a staging)

// Dynamic shares: chunks of kChunk units, handed out in order by the phase's counter, so that a
// CTA whose units are cheaper (single-token groups on the integer core) takes more of them.
// A chunk is taken only when the CTA is about to work on it. Returns the units this CTA did.
template <int NV>
__device__ int run_queue(const DecParams &P, const RTab &rt, int tot, int *q, bool down, bool shared_phase,
                         const int *off, int nslots, int U, void *xs, Misc &m) {
    int done = 0;
    for (;;) {
        if (threadIdx.x == 0) m.chunk = atomicAdd(q, 1);
        __syncthreads();
        const int b = m.chunk * kChunk;
        __syncthreads();  // every thread has read the chunk before thread 0 takes the next
        if (b >= tot) break;
        const int e = min(tot, b + kChunk);
        run_share<NV>(P, rt, b, e, down, shared_phase, off, nslots, U, xs, m);
        done += e - b;
    }
    return done;
}

template <int NV>
__global__ void __launch_bounds__(kNT, 2) moe_decode_kernel(const __grid_constant__ DecParams P) {
    extern __shared__ __align__(128) uint8_t smem[];
    void *xs = smem;
    const RTab rt = rtab_of(smem + P.xs_bytes, P.T, P.E, P.K);
    Misc &m = *reinterpret_cast<Misc *>(smem + P.xs_bytes + P.rt_bytes);
    const int tid = threadIdx.x, G = gridDim.x, c = blockIdx.x;
    if (tid == 0) m.skey[0] = m.skey[1] = m.skey[2] = -1;

    // ---------------- A: router partial logits
    if (!P.route_only) {
        if (c < P.R) {
            router_item<NV == 1 ? 1 : (NV == 2 ? 2 : 8)>(P, c);
            __syncthreads();
            if (tid == 0) {
                __threadfence();
                atomicAdd(&P.ctrl->router_done, 1);
            }
        }
    } else if (c < P.T) {  // the partials come from the router launch before this kernel
        route_token(P, c, static_cast<float *>(xs));
    }

    // ---------------- B: the shared expert's gate/up (independent of routing)
    if (P.Is > 0)
        run_queue<NV>(P, rt, P.G_sh, &P.ctrl->q_b, false, true, nullptr, 0, -1, xs, m);

    // ---------------- R: routing, by this CTA for itself
    if (tid == 0) {
        if (P.route_only) wait_at_least(&P.ctrl->routed_done, P.T, P.ctrl);
        else wait_at_least(&P.ctrl->router_done, P.R, P.ctrl);
        __threadfence();
        m.skey[0] = -1;  // xs becomes routing scratch
    }
    __syncthreads();
    route_local(P, static_cast<float *>(xs), rt, P.route_only != 0);
    const int U = *rt.U;

    // ---------------- C: routed gate/up
    const int gu_tot = rt.gu_off[U];
    run_queue<NV>(P, rt, gu_tot, &P.ctrl->q_c, false, false, rt.gu_off, U, U, xs, m);

    // ---------------- D: down rows of every expert
    const int nslots = U + (P.Is > 0 ? 1 : 0);
    const int dn_tot = rt.dn_off[nslots];
    const int dn_mine = run_queue<NV>(P, rt, dn_tot, &P.ctrl->q_d, true, false, rt.dn_off, nslots, U, xs, m);
    if (tid == 0) {
        __threadfence();
        atomicAdd(&P.ctrl->dn_done, dn_mine);
    }

    // ---------------- E: combine this CTA's rows of out
    if (tid == 0) {
        wait_at_least(&P.ctrl->dn_done, dn_tot, P.ctrl);
        __threadfence();
    }
    __syncthreads();
    const int r_lo = range_lo(P.H, c, G), r_hi = range_lo(P.H, c + 1, G), nd = r_hi - r_lo;
    for (int i = tid; i < P.T * nd; i += kNT) {
        const int t = i / nd, d = r_lo + i % nd;
        const int ke = rt.keff[t];
        float a = 0.f;
        for (int k = 0; k < ke; k++)
            a = __fadd_rn(a, __fmul_rn(rt.w[t * P.K + k], __ldcg(P.y + (size_t)rt.pos[t * P.K + k] * P.H + d)));
        if (P.Is > 0) a = __fadd_rn(a, __ldcg(P.y + ((size_t)P.T * P.K + t) * P.H + d));
        if (P.resid) a = __fadd_rn(P.resid[(size_t)t * P.H + d], a);  // the layer tail: x += tmp
        P.out[(size_t)t * P.H + d] = a;
    }
}

}  // namespace

size_t decode_ctrl_bytes() { return sizeof(DecCtrl); }

size_t decode_smem_bytes(const DecParams &P) { return (size_t)P.xs_bytes + P.rt_bytes + sizeof(Misc) + 64; }

// Host-side geometry of the decode launch for a grid of `grid` CTAs.
bool decode_plan(const coli_moe_desc &d, DecParams &P, int grid) {
    const int T = d.T;
    P.NV = T == 1 ? 1 : (T <= 2 ? 2 : 4);
    const int maxdim = std::max(d.H, std::max(d.I, d.I_shared));
    // per-token stride of the tensor-core staging, in 4-byte words: 4 bytes (f16 hi + lo) per
    // element over whole 64-byte weight segments, plus 64 bytes so that consecutive tokens
    // start 64 bytes apart modulo 128 (distinct shared-memory banks for a quarter-warp)
    P.xs_stride = (int)align_up((size_t)maxdim, 256) + 16;
    const size_t xs_vec = (size_t)P.NV * P.xs_stride * sizeof(float);
    const int ksel = (d.ksel > 0 && d.ksel < d.K) ? d.ksel : d.K;
    const size_t scratch = rscratch_bytes(T, d.E, d.K, ksel);
    P.xs_bytes = (int)align_up(std::max(xs_vec, scratch), 128);
    P.rt_bytes = (int)align_up(rtab_bytes(T, d.E, d.K), 128);
    P.route_only = T <= 8 ? 0 : 1;
    P.neb = (d.E + kRtE - 1) / kRtE;
    if (!P.route_only) {
        // router items: expert blocks x k-slices of whole float4 groups, at most one per CTA
        const int max_slices = std::max(1, d.H / 128);
        int nks = std::max(1, std::min({grid / P.neb, max_slices, 16}));
        P.rks_floats = (d.H / nks + 3) / 4 * 4;
        nks = (d.H + P.rks_floats - 1) / P.rks_floats;
        P.nks = nks;
        P.R = P.neb * nks;
        if (P.R > grid) return false;
    } else {
        P.R = 0;  // P.nks is the separate router launch's split count
    }
    P.groups_sh = d.I_shared > 0 ? (T + P.NV - 1) / P.NV : 0;
    P.G_sh = d.I_shared > 0 ? P.groups_sh * ((d.I_shared + 1) / 2) : 0;
    return decode_smem_bytes(P) <= 113u * 1024;
}

bool decode_supported(const coli_moe_desc &d) {
    return d.T >= 1 && d.T <= kDecMaxT && (d.E + kRtE - 1) / kRtE <= 32;
}

cudaError_t launch_decode(const DecParams &P, int grid, cudaStream_t st) {
    const size_t smem = decode_smem_bytes(P);
    const void *fn = P.NV == 1 ? (const void *)moe_decode_kernel<1>
                   : P.NV == 2 ? (const void *)moe_decode_kernel<2> : (const void *)moe_decode_kernel<4>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    // cooperative: every CTA of the static schedule is resident at once
    void *args[] = {const_cast<DecParams *>(&P)};
    return cudaLaunchCooperativeKernel(fn, dim3(grid), dim3(kNT), args, smem, st);
}

int decode_ctas_per_sm(const DecParams &P) {
    int n = 0;
    const void *fn = P.NV == 1 ? (const void *)moe_decode_kernel<1>
                   : P.NV == 2 ? (const void *)moe_decode_kernel<2> : (const void *)moe_decode_kernel<4>;
    const size_t smem = decode_smem_bytes(P);
    // the query counts against the kernel's dynamic shared-memory limit: raise it first
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kNT, smem) != cudaSuccess) return 0;
    return n;
}

}  // namespace colimoe
