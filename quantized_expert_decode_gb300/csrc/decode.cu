// decode.cu — the whole MoE block for decode-sized batches (T <= 64) in ONE persistent launch.
//
// Phases, each split statically and contiguously over the CTAs (two per SM, cooperative
// launch, so every CTA is resident and a wait is only ever on an earlier phase):
//   A  routing (colibri-strix c/glm.c @98759bf moe() phase A; r_router / r_top8_par shaders):
//      T <= 8: router items — logits of 32 experts over one slice of H — write partial logits;
//      the last item of each 32-expert block (atomic ticket) sums that block's partials in a
//      fixed order; the last block runs the selection. T > 8: the partial logits come from a
//      router launch before this kernel; every CTA sums a share, the last one selects.
//      Selection (one CTA, everything in shared memory): sigmoid, bias, greedy top-K with ties
//      to the lower index, TOPK/TOPP, renorm, routed scale, token->expert buckets (stable) and
//      the unit table of the expert phases; then a flag is published.
//   B  shared expert gate/up rows (known before routing: overlaps phase A)
//   C  routed gate/up rows: h = silu(gate.x * s_g) * (up.x * s_u)   (moe() phases C/D)
//   D  down rows: y = (down.h) * s_d, for every selected expert and the shared one
//   E  combine: out = sum_k w_k y_k in selection order + y_shared   (moe() phases C/D/E)
// Units of B/C are one row pair (gate row j, up row j) of one expert for one group of up to
// NV tokens; units of D are one down row. A CTA walks its share in segments that have the same
// expert and tokens: the segment's activations are staged once in shared memory (pre-scaled and
// permuted, see qdot.cuh), then each warp streams its units' rows with 16-byte loads kept
// several chunks ahead in registers, across unit boundaries.
// Dependencies are counters in the workspace, raised once per CTA per expert (gate/up -> down)
// or per CTA (down -> combine). Every wait is bounded (2 s of %globaltimer); on expiry the kernel
// records kErrWaitExpired and carries on, so a fault in the schedule can not hang the GPU.
#include <algorithm>

#include "kernels.h"
#include "ptx.cuh"
#include "qdot.cuh"

namespace colimoe {

namespace {

constexpr int kNT = 256;                 // threads per CTA
constexpr int kNW = kNT / kWarp;         // warps per CTA
constexpr int kRtE = 32;                 // experts per router item (4 per warp)
constexpr int kDepth = 4;                // 16-byte chunks kept in flight per lane and row
constexpr unsigned long long kWaitNs = 2000000000ull;
constexpr int kSharedKey = kMaxE;        // gu_done index of the shared expert

__device__ __forceinline__ void flag_error(DecCtrl *c, int code) { atomicCAS(&c->err, 0, code); }

// bounded wait until *p >= target; false (and flagged) on timeout
__device__ bool wait_at_least(const int *p, int target, DecCtrl *c) {
    if (ld_volatile(p) >= target) return true;
    const uint64_t t0 = globaltimer_ns();
    while (ld_volatile(p) < target) {
        __nanosleep(64);
        if (globaltimer_ns() - t0 > kWaitNs) {
            flag_error(c, kErrWaitExpired);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ int range_lo(int n, int c, int G) { return (int)((long long)n * c / G); }

// first index i in [0, n) with off[i+1] > x (off: nondecreasing prefix array, off[0] = 0)
__device__ int upper_slot(const int *off, int n, int x) {
    int lo = 0, hi = n - 1;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (__ldcg(off + mid + 1) > x) hi = mid;
        else lo = mid + 1;
    }
    return lo;
}

__device__ __forceinline__ bool bad16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

// ------------------------------------------------------------------ the streaming core
// One warp streams `nunits` units of NR packed rows each (CPR 16-byte chunks per row), lane l
// taking chunks l, l+32, ... of every row, with kDepth chunk-steps of loads in flight across unit
// boundaries. rows_of(i, rows) gives unit i's row pointers; epi(i, sums) gets the finished
// warp-reduced dot products with the NV staged vectors.
template <int FMT, int NR, int NV, class RowsOf, class Epi>
__device__ __forceinline__ void warp_stream(int nunits, int CPR, const float *xs, int xstride, int lane,
                                            RowsOf rows_of, Epi epi) {
    using G = QGeom<FMT>;
    if (nunits <= 0) return;
    const int S = (CPR + kWarp - 1) / kWarp;  // steps per unit
    const int total = nunits * S;
    uint4 buf[kDepth][NR];
    int iu = 0, ik = 0;  // issue cursor: unit, step within unit
    auto issue = [&](uint4 (&b)[NR]) {
        if (iu < nunits) {
            const int c = lane + kWarp * ik;
            const uint8_t *rr[NR];
            rows_of(iu, rr);
#pragma unroll
            for (int r = 0; r < NR; r++) b[r] = c < CPR ? ld_stream_16(rr[r] + 16 * c) : make_uint4(0, 0, 0, 0);
            if (++ik == S) {
                ik = 0;
                iu++;
            }
        }
    };
#pragma unroll
    for (int j = 0; j < kDepth; j++) issue(buf[j]);
    float2 acc[NR][NV];
#pragma unroll
    for (int r = 0; r < NR; r++)
#pragma unroll
        for (int v = 0; v < NV; v++) acc[r][v] = make_float2(0.f, 0.f);
    const float4 *xs4 = reinterpret_cast<const float4 *>(xs);
    const int xstride4 = xstride / 4;
    int cu = 0, ck = 0;  // compute cursor
    for (int s0 = 0; s0 < total; s0 += kDepth) {
#pragma unroll
        for (int j = 0; j < kDepth; j++) {
            if (s0 + j < total) {
                const int c = lane + kWarp * ck;
                if (c < CPR) {
#pragma unroll
                    for (int wi = 0; wi < 4; wi++) {
                        float4 xv[NV][G::F4W];
#pragma unroll
                        for (int v = 0; v < NV; v++)
#pragma unroll
                            for (int q = 0; q < G::F4W; q++)
                                xv[v][q] = xs4[v * xstride4 + (wi * G::F4W + q) * CPR + c];
#pragma unroll
                        for (int r = 0; r < NR; r++) {
                            const uint32_t w = word_of(buf[j][r], wi);
                            const uint32_t wh = w >> 16;
#pragma unroll
                            for (int m = 0; m < G::HALF; m++) {
                                const uint32_t lo = lop3_and_xor(w, G::mask(m), G::xorv(m));
                                const uint32_t hi = lop3_and_xor(wh, G::mask(m), G::xorv(m));
                                const float2 d = __fadd2_rn(make_float2(__uint_as_float(lo), __uint_as_float(hi)),
                                                            make_float2(-G::magic(m), -G::magic(m)));
#pragma unroll
                                for (int v = 0; v < NV; v++) {
                                    const float4 &x4 = xv[v][m >> 1];
                                    const float2 x2 = (m & 1) ? make_float2(x4.z, x4.w) : make_float2(x4.x, x4.y);
                                    acc[r][v] = __ffma2_rn(d, x2, acc[r][v]);
                                }
                            }
                        }
                    }
                }
                issue(buf[j]);
                if (++ck == S) {
                    float sums[NR][NV];
                    warp_reduce_acc<NR, NV>(acc, sums);
                    epi(cu, sums);
#pragma unroll
                    for (int r = 0; r < NR; r++)
#pragma unroll
                        for (int v = 0; v < NV; v++) acc[r][v] = make_float2(0.f, 0.f);
                    ck = 0;
                    cu++;
                }
            }
        }
    }
}

// ------------------------------------------------------------------ routing
struct Scratch {  // shared-memory layout of the selection step (inside the staging buffer)
    int *cnt, *off, *fill, *chk, *actv, *wc, *tmp, *idx, *keff, *gu, *dn;
    float *w;
};

__device__ __forceinline__ Scratch scratch_of(void *base, int E, int T, int K) {
    Scratch s;
    int *p = static_cast<int *>(base);
    s.cnt = p;
    s.off = s.cnt + E;
    s.fill = s.off + E;
    s.chk = s.fill + E;
    s.actv = s.chk + E;
    s.wc = s.actv + E;
    s.tmp = s.wc + kNW * E;
    s.idx = s.tmp + 16;
    s.keff = s.idx + T * K;
    s.gu = s.keff + T;
    s.dn = s.gu + (E + 2);
    s.w = reinterpret_cast<float *>(s.dn + (E + 2));
    return s;
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

// one warp: selection of token t from its logits (sigmoid, bias, greedy top-K, TOPP, renorm,
// scale). Lane l owns experts [l*PER, l*PER + PER), so the lane-local strict '>' ascending scan
// plus a cross-lane argmax preferring the lower index reproduce the serial first-max-wins order.
template <int PER>
__device__ void select_token(const DecParams &P, int t, int lane, const Scratch &sc) {
    const int base = lane * PER;
    float ch[PER], sg[PER];
#pragma unroll
    for (int j = 0; j < PER; j++) {
        const int e = base + j;
        ch[j] = e < P.E ? __ldcg(P.sig + (size_t)t * P.E + e) : 0.f;  // logits, all loads in flight
    }
#pragma unroll
    for (int j = 0; j < PER; j++) {
        const int e = base + j;
        if (e < P.E) {
            const float sv = 1.f / (1.f + expf(-ch[j]));
            const float cv = sv + P.bias[e];
            P.sig[(size_t)t * P.E + e] = sv;
            P.choice[(size_t)t * P.E + e] = cv;
            sg[j] = sv;
            ch[j] = cv;
        } else {
            sg[j] = 0.f;
            ch[j] = -INFINITY;
        }
    }
    uint32_t taken = 0;
    int nsel = 0, my_i = -1;
    float my_w = 0.f;
    for (int k = 0; k < P.Ksel; k++) {
        float bv = -1e30f, bs = 0.f;
        int bi = 0x7fffffff;
#pragma unroll
        for (int j = 0; j < PER; j++)
            if (!((taken >> j) & 1u) && ch[j] > bv) {
                bv = ch[j];
                bi = base + j;
                bs = sg[j];
            }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_down_sync(kFull, bv, o);
            const int oi = __shfl_down_sync(kFull, bi, o);
            const float os = __shfl_down_sync(kFull, bs, o);
            if (ov > bv || (ov == bv && oi < bi)) {
                bv = ov;
                bi = oi;
                bs = os;
            }
        }
        bi = __shfl_sync(kFull, bi, 0);
        bs = __shfl_sync(kFull, bs, 0);
        if (bi == 0x7fffffff) {
            if (lane == 0) flag_error(P.ctrl, kErrNoCandidate);
            break;
        }
        if (bi >= base && bi < base + PER) taken |= 1u << (bi - base);
        if (lane == k) {
            my_i = bi;
            my_w = bs;
        }
        nsel = k + 1;
    }
    float ww[kMaxK];
    int id[kMaxK];
    for (int k = 0; k < nsel; k++) {
        ww[k] = __shfl_sync(kFull, my_w, k);
        id[k] = __shfl_sync(kFull, my_i, k);
    }
    if (lane != 0) return;
    int Ke = nsel;
    if (P.top_p > 0.f && P.top_p < 1.f) {
        for (int a = 1; a < nsel; a++) {
            const int ia = id[a];
            const float wa = ww[a];
            int b = a - 1;
            while (b >= 0 && ww[b] < wa) {
                ww[b + 1] = ww[b];
                id[b + 1] = id[b];
                b--;
            }
            ww[b + 1] = wa;
            id[b + 1] = ia;
        }
        float tot = 1e-20f;
        for (int k = 0; k < nsel; k++) tot = __fadd_rn(tot, ww[k]);
        float cum = 0.f;
        for (int k = 0; k < nsel; k++) {
            cum = __fadd_rn(cum, ww[k]);
            if (cum >= __fmul_rn(P.top_p, tot)) {
                Ke = k + 1;
                break;
            }
        }
    }
    if (P.norm_topk) {
        float sm = 0.f;
        for (int k = 0; k < Ke; k++) sm = __fadd_rn(sm, ww[k]);
        sm = __fadd_rn(sm, 1e-20f);
        for (int k = 0; k < Ke; k++) ww[k] = __fdiv_rn(ww[k], sm);
    }
    for (int k = 0; k < P.K; k++) {
        const bool kept = k < Ke;
        const int vi = kept ? id[k] : -1;
        const float vw = kept ? __fmul_rn(ww[k], P.rscale) : 0.f;
        P.idx[(size_t)t * P.K + k] = vi;
        P.w[(size_t)t * P.K + k] = vw;
        sc.idx[t * P.K + k] = vi;
        sc.w[t * P.K + k] = vw;
    }
    P.keff[t] = Ke;
    sc.keff[t] = Ke;
}

// selection, buckets and the unit table, by one CTA, from the logits in P.sig
__device__ void route_final(const DecParams &P, void *scratch) {
    const int tid = threadIdx.x, lane = tid % kWarp, warp = tid / kWarp;
    const Scratch sc = scratch_of(scratch, P.E, P.T, P.K);
    const int per = (P.E + kWarp - 1) / kWarp;
    for (int t = warp; t < P.T; t += kNW) {
        if (per <= 1) select_token<1>(P, t, lane, sc);
        else if (per <= 2) select_token<2>(P, t, lane, sc);
        else if (per <= 4) select_token<4>(P, t, lane, sc);
        else if (per <= 8) select_token<8>(P, t, lane, sc);
        else if (per <= 16) select_token<16>(P, t, lane, sc);
        else select_token<32>(P, t, lane, sc);
    }
    const int E = P.E, N = P.T * P.K;
    for (int e = tid; e < E; e += kNT) {
        sc.cnt[e] = 0;
        sc.fill[e] = 0;
    }
    __syncthreads();
    auto expert_of = [&](int a) -> int {
        if (a >= N) return -1;
        return (a % P.K) < sc.keff[a / P.K] ? sc.idx[a] : -1;
    };
    for (int a = tid; a < N; a += kNT) {
        const int e = expert_of(a);
        if (e >= 0) atomicAdd(&sc.cnt[e], 1);
    }
    __syncthreads();
    for (int e = tid; e < E; e += kNT) {
        sc.off[e] = sc.cnt[e];
        sc.actv[e] = sc.cnt[e] > 0 ? 1 : 0;
        P.counts[e] = sc.cnt[e];
    }
    __syncthreads();
    const int total = scan_smem(sc.off, E, sc.tmp);
    const int U = scan_smem(sc.actv, E, sc.tmp);
    for (int e = tid; e < E; e += kNT) {
        P.offsets[e] = sc.off[e];
        if (sc.cnt[e] > 0) {
            P.act[sc.actv[e]] = e;
            sc.chk[sc.actv[e]] = e;  // active experts, ascending (chk is free until the chunk loop)
        }
    }
    if (tid == 0) P.offsets[E] = total;
    __syncthreads();
    // unit table: slot u < U is the u-th active expert; slot U the shared expert
    for (int u = tid; u < U + 1; u += kNT) {
        int g = 0;
        if (u < U) {
            const int e = sc.chk[u];
            g = (sc.cnt[e] + P.NV - 1) / P.NV;
            P.tab->slot_e[u] = e;
            P.tab->slot_n[u] = sc.cnt[e];
            P.tab->slot_pbase[u] = sc.off[e];
            P.tab->slot_groups[u] = g;
            sc.gu[u] = g * P.I;
            sc.dn[u] = g * P.H;
        } else {
            sc.gu[u] = 0;
            sc.dn[u] = P.Is > 0 ? P.groups_sh * P.H : 0;
        }
    }
    __syncthreads();
    const int gu_tot = scan_smem(sc.gu, U + 1, sc.tmp);
    const int dn_tot = scan_smem(sc.dn, U + 1, sc.tmp);
    for (int u = tid; u < U + 1; u += kNT) {
        P.tab->gu_off[u] = sc.gu[u];
        P.tab->dn_off[u] = sc.dn[u];
    }
    if (tid == 0) {
        P.tab->gu_off[U + 1] = gu_tot;
        P.tab->dn_off[U + 1] = dn_tot;
        P.tab->U = U;
        P.tab->gu_tot = gu_tot;
        P.tab->dn_tot = dn_tot;
    }
    // stable perm / pos: 256-assignment chunks in order; inside a chunk, rank within the warp
    // from a match-any mask, then the warps' per-expert counts are scanned
    for (int a0 = 0; a0 < N; a0 += kNT) {
        for (int i = tid; i < kNW * E; i += kNT) sc.wc[i] = 0;
        __syncthreads();
        const int a = a0 + tid;
        const int e = expert_of(a);
        const unsigned peers = __match_any_sync(kFull, e);
        const int rank = __popc(peers & ((1u << lane) - 1u));
        if (e >= 0 && rank == 0) sc.wc[warp * E + e] = __popc(peers);
        __syncthreads();
        for (int x = tid; x < E; x += kNT) {
            int run = 0;
            for (int w = 0; w < kNW; w++) {
                const int v = sc.wc[w * E + x];
                sc.wc[w * E + x] = run;
                run += v;
            }
            sc.chk[x] = run;
        }
        __syncthreads();
        if (a < N) {
            if (e >= 0) {
                const int p = sc.off[e] + sc.fill[e] + sc.wc[warp * E + e] + rank;
                P.perm[p] = a;
                P.pos[a] = p;
            } else {
                P.pos[a] = -1;
            }
        }
        __syncthreads();
        for (int x = tid; x < E; x += kNT) sc.fill[x] += sc.chk[x];
        __syncthreads();
    }
    if (tid == 0) {
        __threadfence();
        atomicExch(&P.ctrl->routing_ready, 1);
    }
}

// T <= 8: partial logits of 32 experts (4 per warp) over one slice of H
__device__ void router_item(const DecParams &P, int item) {
    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
    const int eb = item % P.neb, ks = item / P.neb;
    const int kb = ks * P.rks_floats, ke = min(P.H, kb + P.rks_floats);
    float acc[4][8];
#pragma unroll
    for (int r = 0; r < 4; r++)
#pragma unroll
        for (int t = 0; t < 8; t++) acc[r][t] = 0.f;
    int e[4];
#pragma unroll
    for (int r = 0; r < 4; r++) e[r] = min(eb * kRtE + warp * 4 + r, P.E - 1);
    for (int k = kb + 4 * lane; k < ke; k += 4 * kWarp) {
        float4 wv[4];
#pragma unroll
        for (int r = 0; r < 4; r++) {
            const uint4 u = ld_stream_16(P.Wr + (size_t)e[r] * P.H + k);
            wv[r] = make_float4(__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z), __uint_as_float(u.w));
        }
#pragma unroll
        for (int t = 0; t < 8; t++) {
            if (t >= P.T) break;
            const float4 xv = __ldg(reinterpret_cast<const float4 *>(P.x + (size_t)t * P.H + k));
#pragma unroll
            for (int r = 0; r < 4; r++) {
                float a = acc[r][t];
                a = fmaf(wv[r].x, xv.x, a);
                a = fmaf(wv[r].y, xv.y, a);
                a = fmaf(wv[r].z, xv.z, a);
                a = fmaf(wv[r].w, xv.w, a);
                acc[r][t] = a;
            }
        }
    }
#pragma unroll
    for (int r = 0; r < 4; r++)
#pragma unroll
        for (int t = 0; t < 8; t++) {
            if (t >= P.T) break;
            float s = acc[r][t];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(kFull, s, o);
            const int er = eb * kRtE + warp * 4 + r;
            if (lane == 0 && er < P.E) P.part[((size_t)ks * P.T + t) * P.E + er] = s;
        }
}

// logits = fixed-order sums of the partials, for flat logit indices [lo, hi) (t-major)
__device__ void reduce_logits(const DecParams &P, int lo, int hi) {
    for (int i = lo + (int)threadIdx.x; i < hi; i += kNT) {
        float s = 0.f;
        int k = 0;
        for (; k + 4 <= P.nks; k += 4) {
            const float a0 = __ldcg(P.part + (size_t)(k + 0) * P.T * P.E + i);
            const float a1 = __ldcg(P.part + (size_t)(k + 1) * P.T * P.E + i);
            const float a2 = __ldcg(P.part + (size_t)(k + 2) * P.T * P.E + i);
            const float a3 = __ldcg(P.part + (size_t)(k + 3) * P.T * P.E + i);
            s += a0;
            s += a1;
            s += a2;
            s += a3;
        }
        for (; k < P.nks; k++) s += __ldcg(P.part + (size_t)k * P.T * P.E + i);
        P.sig[i] = s;
    }
}

// ------------------------------------------------------------------ expert phases
struct Seg {  // one segment of units with the same expert and tokens (broadcast in smem)
    const uint8_t *w0, *w1;  // gate/up rows, or down rows in w0
    const float *s0, *s1;    // their row scales
    int fmt, inter, n, pbase, shared, tg, key, need;
    int ulo, uhi;            // units [ulo, uhi) of this CTA in the segment
    int ubase;               // unit index of the segment's first unit (row 0)
};

// stage the activations of token group tg (x rows for gate/up, h rows for down) into xs
__device__ void stage_acts(const DecParams &P, const Seg &g, bool down, float *xs) {
    const int nv = min(P.NV, g.n - g.tg * P.NV);
    const int len = down ? g.inter : P.H;
    const int gran = g.fmt == COLI_FMT_INT4 ? 32 : g.fmt == COLI_FMT_INT8 ? 16 : 64;
    const int CPR = len / gran;
    for (int v = 0; v < P.NV; v++) {
        float *dst = xs + (size_t)v * P.xs_stride;
        if (v < nv) {
            const int pv = g.tg * P.NV + v;
            const float *src;
            if (down) {
                const int row = g.shared ? P.T * P.K + pv : g.pbase + pv;
                src = P.h + (size_t)row * P.ldh;
            } else {
                const int t = g.shared ? pv : __ldcg(P.perm + g.pbase + pv) / P.K;
                src = P.x + (size_t)t * P.H;
            }
            for (int i = threadIdx.x; i < len; i += kNT) {
                float sc;
                int at;
                if (g.fmt == COLI_FMT_INT4) at = staged_index<COLI_FMT_INT4>(i, CPR, sc);
                else if (g.fmt == COLI_FMT_INT8) at = staged_index<COLI_FMT_INT8>(i, CPR, sc);
                else at = staged_index<COLI_FMT_INT2>(i, CPR, sc);
                dst[at] = (down ? __ldcg(src + i) : __ldg(src + i)) * sc;
            }
        } else {
            for (int i = threadIdx.x; i < len; i += kNT) dst[i] = 0.f;
        }
    }
}

template <int FMT, int NV>
__device__ void gateup_units(const DecParams &P, const Seg &g, const float *xs) {
    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
    const int nu = g.uhi - g.ulo;
    const int mine = nu > warp ? (nu - warp + kNW - 1) / kNW : 0;
    const int64_t rb = row_bytes(FMT, P.H);
    const int nv = min(P.NV, g.n - g.tg * P.NV);
    const int jbase = g.ulo - g.ubase;  // row of the segment's first unit of this CTA
    warp_stream<FMT, 2, NV>(
        mine, (int)(rb / 16), xs, P.xs_stride, lane,
        [&](int i, const uint8_t *(&rr)[2]) {
            const int j = jbase + warp + kNW * i;
            rr[0] = g.w0 + (size_t)j * rb;
            rr[1] = g.w1 + (size_t)j * rb;
        },
        [&](int i, const float (&s)[2][NV]) {
            const int j = jbase + warp + kNW * i;
#pragma unroll
            for (int v = 0; v < NV; v++) {
                if (lane == v && v < nv) {
                    const float gv = s[0][v] * g.s0[j];
                    const float uv = s[1][v] * g.s1[j];
                    const int pv = g.tg * P.NV + v;
                    const int row = g.shared ? P.T * P.K + pv : g.pbase + pv;
                    P.h[(size_t)row * P.ldh + j] = gv / (1.f + expf(-gv)) * uv;
                }
            }
        });
}

template <int FMT, int NV>
__device__ void down_units(const DecParams &P, const Seg &g, const float *xs) {
    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
    const int nu = g.uhi - g.ulo;
    const int mine = nu > warp ? (nu - warp + kNW - 1) / kNW : 0;
    const int64_t rb = row_bytes(FMT, g.inter);
    const int nv = min(P.NV, g.n - g.tg * P.NV);
    const int dbase = g.ulo - g.ubase;
    warp_stream<FMT, 1, NV>(
        mine, (int)(rb / 16), xs, P.xs_stride, lane,
        [&](int i, const uint8_t *(&rr)[1]) { rr[0] = g.w0 + (size_t)(dbase + warp + kNW * i) * rb; },
        [&](int i, const float (&s)[1][NV]) {
            const int d = dbase + warp + kNW * i;
#pragma unroll
            for (int v = 0; v < NV; v++) {
                if (lane == v && v < nv) {
                    const int pv = g.tg * P.NV + v;
                    const int row = g.shared ? P.T * P.K + pv : g.pbase + pv;
                    P.y[(size_t)row * P.H + d] = s[0][v] * g.s0[d];
                }
            }
        });
}

template <int NV>
__device__ void run_units(const DecParams &P, const Seg &g, bool down, const float *xs) {
    if (down) {
        if (g.fmt == COLI_FMT_INT4) down_units<COLI_FMT_INT4, NV>(P, g, xs);
        else if (g.fmt == COLI_FMT_INT8) down_units<COLI_FMT_INT8, NV>(P, g, xs);
        else down_units<COLI_FMT_INT2, NV>(P, g, xs);
    } else {
        if (g.fmt == COLI_FMT_INT4) gateup_units<COLI_FMT_INT4, NV>(P, g, xs);
        else if (g.fmt == COLI_FMT_INT8) gateup_units<COLI_FMT_INT8, NV>(P, g, xs);
        else gateup_units<COLI_FMT_INT2, NV>(P, g, xs);
    }
}

// fill the segment of unit l (thread 0 only): unit spaces are slot-major, then token group,
// then row; routed slots come from the table, the shared expert is slot U (or the static
// shared phase when U < 0)
__device__ void make_seg(const DecParams &P, int slot, int U, int slot_base, int l, int e_share, bool down, Seg &g) {
    const bool shared = U < 0 || slot == U;
    const int rows_per_group = down ? P.H : (shared ? P.Is : P.I);
    if (shared) {
        g.w0 = static_cast<const uint8_t *>(down ? P.shared.down_w : P.shared.gate_w);
        g.w1 = static_cast<const uint8_t *>(P.shared.up_w);
        g.s0 = down ? P.shared.down_s : P.shared.gate_s;
        g.s1 = P.shared.up_s;
        g.fmt = P.sfmt;
        g.inter = P.Is;
        g.n = P.T;
        g.pbase = 0;
        g.key = kSharedKey;
        g.need = P.G_sh;
    } else {
        const int e = __ldcg(&P.tab->slot_e[slot]);
        const coli_moe_expert ex = P.experts[e];
        g.w0 = static_cast<const uint8_t *>(down ? ex.down_w : ex.gate_w);
        g.w1 = static_cast<const uint8_t *>(ex.up_w);
        g.s0 = down ? ex.down_s : ex.gate_s;
        g.s1 = ex.up_s;
        g.fmt = P.rfmt;
        g.inter = P.I;
        g.n = __ldcg(&P.tab->slot_n[slot]);
        g.pbase = __ldcg(&P.tab->slot_pbase[slot]);
        g.key = slot;
        g.need = __ldcg(&P.tab->slot_groups[slot]) * P.I;
        if (bad16(ex.gate_w) || bad16(ex.up_w) || bad16(ex.down_w)) flag_error(P.ctrl, kErrBadExpert);
    }
    g.shared = shared ? 1 : 0;
    const int local = l - slot_base;
    g.tg = local / rows_per_group;
    g.ubase = slot_base + g.tg * rows_per_group;
    g.ulo = l;
    g.uhi = min(e_share, g.ubase + rows_per_group);
}

// walk this CTA's share [b, e) of a unit space (gate/up or down) segment by segment
template <int NV>
__device__ void run_share(const DecParams &P, int b, int e, bool down, bool shared_phase, float *xs, Seg *sg,
                          int *skey) {
    const int tid = threadIdx.x;
    if (b >= e) return;
    int U = -1, slot = 0, slot_base = 0, slot_end = 0, done_in_slot = 0;
    const int *off = down ? P.tab->dn_off : P.tab->gu_off;
    if (!shared_phase) U = __ldcg(&P.tab->U);
    const int nslots = shared_phase ? 1 : (down ? U + (P.Is > 0 ? 1 : 0) : U);
    if (tid == 0) {
        if (shared_phase) {
            slot_base = 0;
            slot_end = P.G_sh;
        } else {
            slot = upper_slot(off, nslots, b);
            slot_base = __ldcg(off + slot);
            slot_end = __ldcg(off + slot + 1);
        }
    }
    int l = b;
    while (l < e) {
        __syncthreads();  // the previous segment's units are done with xs and sg
        if (tid == 0) {
            while (l >= slot_end) {  // next slot (thread 0's cursor)
                slot++;
                slot_base = slot_end;
                slot_end = __ldcg(off + slot + 1);
            }
            make_seg(P, slot, shared_phase ? -1 : U, slot_base, l, min(e, slot_end), down, *sg);
            if (down) {  // this expert's h rows must all be written
                wait_at_least(&P.ctrl->gu_done[sg->key], sg->need, P.ctrl);
                __threadfence();
            }
        }
        __syncthreads();
        const Seg g = *sg;
        // activations: skip restaging when xs already holds them (same kind, tokens and format)
        const int k0 = down ? 2 : 1;
        const int k1 = down ? g.key : (P.T == 1 ? 0 : (g.shared ? -1 : g.pbase));
        const int k2 = (P.T == 1 && !down) ? g.fmt : g.tg * 8 + g.fmt;
        if (!(skey[0] == k0 && skey[1] == k1 && skey[2] == k2)) {
            stage_acts(P, g, down, xs);
            __syncthreads();
            if (tid == 0) {
                skey[0] = k0;
                skey[1] = k1;
                skey[2] = k2;
            }
        }
        run_units<NV>(P, g, down, xs);
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

template <int NV>
__global__ void __launch_bounds__(kNT, 2) moe_decode_kernel(const DecParams P) {
    extern __shared__ __align__(128) uint8_t smem[];
    float *xs = reinterpret_cast<float *>(smem);
    Seg *sg = reinterpret_cast<Seg *>(smem + P.xs_bytes);
    int *skey = reinterpret_cast<int *>(sg + 1);
    int *sflag = skey + 3;
    const int tid = threadIdx.x, G = gridDim.x, c = blockIdx.x;
    if (tid == 0) skey[0] = skey[1] = skey[2] = -1;

    // ---------------- A: routing
    if (!P.route_only) {
        if (c < P.R) {
            router_item(P, c);
            __syncthreads();
            const int eb = c % P.neb;
            if (tid == 0) {
                __threadfence();
                const bool last = atomicAdd(&P.ctrl->eb_done[eb], 1) == P.nks - 1;
                if (last) __threadfence();
                *sflag = last;
            }
            __syncthreads();
            if (*sflag) {  // last k-slice of this expert block: its logits
                const int e0 = eb * kRtE, e1 = min(P.E, e0 + kRtE);
                for (int t = 0; t < P.T; t++) reduce_logits(P, t * P.E + e0, t * P.E + e1);
                __syncthreads();
                if (tid == 0) {
                    __threadfence();
                    const bool last = atomicAdd(&P.ctrl->router_done, 1) == P.neb - 1;
                    if (last) __threadfence();
                    *sflag = last;
                }
                __syncthreads();
                if (*sflag) route_final(P, xs);
            }
            __syncthreads();
        }
    } else {
        reduce_logits(P, range_lo(P.T * P.E, c, G), range_lo(P.T * P.E, c + 1, G));
        __syncthreads();
        if (tid == 0) {
            __threadfence();
            const bool last = atomicAdd(&P.ctrl->router_done, 1) == G - 1;
            if (last) __threadfence();
            *sflag = last;
        }
        __syncthreads();
        if (*sflag) route_final(P, xs);
        __syncthreads();
    }
    if (tid == 0) skey[0] = -1;  // xs may have served as routing scratch

    // ---------------- B: the shared expert's gate/up (independent of routing)
    if (P.Is > 0) run_share<NV>(P, range_lo(P.G_sh, c, G), range_lo(P.G_sh, c + 1, G), false, true, xs, sg, skey);

    // ---------------- C: routed gate/up
    if (tid == 0) {
        wait_at_least(&P.ctrl->routing_ready, 1, P.ctrl);
        __threadfence();
    }
    __syncthreads();
    const int gu_tot = __ldcg(&P.tab->gu_tot);
    run_share<NV>(P, range_lo(gu_tot, c, G), range_lo(gu_tot, c + 1, G), false, false, xs, sg, skey);

    // ---------------- D: down rows of every expert
    const int dn_tot = __ldcg(&P.tab->dn_tot);
    const int db = range_lo(dn_tot, c, G), de = range_lo(dn_tot, c + 1, G);
    run_share<NV>(P, db, de, true, false, xs, sg, skey);
    if (tid == 0) {
        __threadfence();
        atomicAdd(&P.ctrl->dn_done, de - db);
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
        const int ke = __ldcg(P.keff + t);
        float a = 0.f;
        for (int k = 0; k < ke; k++) {
            const float wk = __ldcg(P.w + (size_t)t * P.K + k);
            const int p = __ldcg(P.pos + (size_t)t * P.K + k);
            a = __fadd_rn(a, __fmul_rn(wk, __ldcg(P.y + (size_t)p * P.H + d)));
        }
        if (P.Is > 0) a = __fadd_rn(a, __ldcg(P.y + ((size_t)P.T * P.K + t) * P.H + d));
        P.out[(size_t)t * P.H + d] = a;
    }
}

}  // namespace

size_t decode_ctrl_bytes() { return sizeof(DecCtrl); }
size_t decode_table_bytes() { return sizeof(DecTable); }

size_t decode_smem_bytes(const DecParams &P) { return (size_t)P.xs_bytes + sizeof(Seg) + 64; }

// Host-side geometry of the decode launch for a grid of `grid` CTAs.
bool decode_plan(const coli_moe_desc &d, DecParams &P, int grid) {
    const int T = d.T;
    P.NV = T == 1 ? 1 : (T <= 2 ? 2 : 4);
    const int maxdim = std::max(d.H, std::max(d.I, d.I_shared));
    P.xs_stride = maxdim;
    const size_t xs_vec = (size_t)P.NV * maxdim * sizeof(float);
    const size_t scratch = (size_t)(5 * d.E + kNW * d.E + 16 + 2 * T * d.K + T + 2 * (d.E + 2) + 16) * sizeof(int);
    P.xs_bytes = (int)align_up(std::max(xs_vec, scratch), 128);
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
    P.G_sh = d.I_shared > 0 ? P.groups_sh * d.I_shared : 0;
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
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kNT, decode_smem_bytes(P)) != cudaSuccess) return 0;
    return n;
}

}  // namespace colimoe
