// decode_parts.cuh — device pieces shared by the persistent decode kernels (decode.cu for
// token groups, decode1.cu for one token): bounded waits, the router item, the integer and
// tensor-core streaming walks, activation loads and an L2 line warm-up. Internal to
// libcolimoe; every translation unit gets its own copy (anonymous namespace).
#pragma once

#include "idot.cuh"
#include "kernels.h"
#include "mma.cuh"
#include "ptx.cuh"
#include "qdot.cuh"

namespace colimoe {
namespace {

constexpr int kNT = 256;                 // threads per CTA
constexpr int kNW = kNT / kWarp;         // warps per CTA
constexpr int kRtE = 32;                 // experts per router item (4 per warp)
constexpr int kInflight = 8;             // 16-byte loads in flight per lane (rows x depth)
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

__device__ __forceinline__ bool bad16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

// weight rows read once per call can be streamed with an evict-first L2 policy, so that they do
// not push out lines that were asked of L2 ahead of their use
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ uint4 ld_once_16(const void *p, uint64_t pol) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(pol));
    return v;
}

// ------------------------------------------------------------------ the streaming cores
// Single-token groups on the integer core (idot.cuh), four or two rows per unit. One warp
// streams `nunits` units of NR packed rows (CPR 16-byte chunks per row), lane l taking chunks
// l, l+32, ... of every row, with INFL / NR chunk-steps of loads in flight across unit
// boundaries; rows_of(i, rows) gives unit i's row pointers;
// xq_of(i) gives the staged activation limbs unit i is dotted with; epi(i, tot, d) gets, in
// lane l, the exact warp total S of row l / (32 / NR) of unit i, and d = pre(i), the unit's
// epilogue operands (row scales), which are loaded two units ahead.
template <int FMT, int NR, int INFL = kInflight, bool ONCE = false, class RowsOf, class XqOf, class Pre, class Epi>
__device__ __forceinline__ void warp_stream_int(int nunits, int CPR, int lane, RowsOf rows_of, XqOf xq_of, Pre pre,
                                                Epi epi) {
    constexpr int kDepth = INFL / NR;
    if (nunits <= 0) return;
    const uint64_t pol = ONCE ? policy_evict_first() : 0;  // ONCE: the rows are read once (evict first)
    const int S = (CPR + kWarp - 1) / kWarp;
    const int total = nunits * S;
    uint4 buf[kDepth][NR];
    int iu = 0, ik = 0;
    const uint8_t *rr[NR];  // row pointers of the unit being issued (looked up once per unit)
    rows_of(0, rr);
    auto issue = [&](uint4 (&b)[NR]) {
        if (iu < nunits) {
            const int c = lane + kWarp * ik;
#pragma unroll
            for (int r = 0; r < NR; r++)
                b[r] = c < CPR ? (ONCE ? ld_once_16(rr[r] + 16 * c, pol) : ld_stream_16(rr[r] + 16 * c))
                               : make_uint4(0, 0, 0, 0);
            if (++ik == S) {
                ik = 0;
                if (++iu < nunits) rows_of(iu, rr);
            }
        }
    };
#pragma unroll
    for (int j = 0; j < kDepth; j++) issue(buf[j]);
    auto d0 = pre(0);
    decltype(d0) d1 = d0;
    if (nunits > 1) d1 = pre(1);
    int acc[NR][3];
#pragma unroll
    for (int r = 0; r < NR; r++) acc[r][0] = acc[r][1] = acc[r][2] = 0;
    int cu = 0, ck = 0;
    const uint4 *xq4 = xq_of(0);
    for (int s0 = 0; s0 < total; s0 += kDepth) {
#pragma unroll
        for (int j = 0; j < kDepth; j++) {
            if (s0 + j < total) {
                const int c = lane + kWarp * ck;
                if (c < CPR) idot_chunk<FMT, NR>(buf[j], xq4, CPR, c, acc);
                issue(buf[j]);
                if (++ck == S) {
                    static_assert(NR == 4 || NR == 2, "the integer walk reduces four or two rows per unit");
                    if constexpr (NR == 4) epi(cu, idot_reduce4<FMT>(acc, lane), d0);
                    else epi(cu, idot_reduce2<FMT>(acc, lane), d0);
                    d0 = d1;
                    if (cu + 2 < nunits) d1 = pre(cu + 2);
#pragma unroll
                    for (int r = 0; r < NR; r++) acc[r][0] = acc[r][1] = acc[r][2] = 0;
                    ck = 0;
                    cu++;
                    if (cu < nunits) xq4 = xq_of(cu);
                }
            }
        }
    }
}

// The same walk for int8 activations (the IDOT quantisation, idot.cuh q8_chunk): four rows per
// unit, one int accumulator per row; epi(i, dot, pre) gets, in lane l, the exact dot of row l / 8.
template <int FMT, int INFL, class RowsOf, class XqOf, class Pre, class Epi>
__device__ __forceinline__ void warp_stream_q8(int nunits, int CPR, int lane, RowsOf rows_of, XqOf xq_of, Pre pre,
                                               Epi epi) {
    constexpr int NR = 4, kDepth = INFL / NR;
    if (nunits <= 0) return;
    const int S = (CPR + kWarp - 1) / kWarp;
    const int total = nunits * S;
    uint4 buf[kDepth][NR];
    int iu = 0, ik = 0;
    const uint8_t *rr[NR];
    rows_of(0, rr);
    auto issue = [&](uint4 (&b)[NR]) {
        if (iu < nunits) {
            const int c = lane + kWarp * ik;
#pragma unroll
            for (int r = 0; r < NR; r++) b[r] = c < CPR ? ld_stream_16(rr[r] + 16 * c) : make_uint4(0, 0, 0, 0);
            if (++ik == S) {
                ik = 0;
                if (++iu < nunits) rows_of(iu, rr);
            }
        }
    };
#pragma unroll
    for (int j = 0; j < kDepth; j++) issue(buf[j]);
    auto d0 = pre(0);
    decltype(d0) d1 = d0;
    if (nunits > 1) d1 = pre(1);
    int acc[NR] = {0, 0, 0, 0};
    int cu = 0, ck = 0;
    const uint4 *xq4 = xq_of(0);
    for (int s0 = 0; s0 < total; s0 += kDepth) {
#pragma unroll
        for (int j = 0; j < kDepth; j++) {
            if (s0 + j < total) {
                const int c = lane + kWarp * ck;
                if (c < CPR) q8_chunk<FMT, NR>(buf[j], xq4, CPR, c, acc);
                issue(buf[j]);
                if (++ck == S) {
                    epi(cu, q8_reduce4<FMT>(acc, lane), d0);
                    d0 = d1;
                    if (cu + 2 < nunits) d1 = pre(cu + 2);
#pragma unroll
                    for (int r = 0; r < NR; r++) acc[r] = 0;
                    ck = 0;
                    cu++;
                    if (cu < nunits) xq4 = xq_of(cu);
                }
            }
        }
    }
}

// Four rows of float lane partials at once, transposing as it reduces (the shuffle pattern of
// idot_reduce4): every lane ends with the total of row lane / 8.
__device__ __forceinline__ float freduce4(const float (&p)[4], int lane) {
    const bool h16 = (lane & 16) != 0, h8 = (lane & 8) != 0;
    float k0 = h16 ? p[2] : p[0], k1 = h16 ? p[3] : p[1];
    const float s0 = h16 ? p[0] : p[2], s1 = h16 ? p[1] : p[3];
    k0 += __shfl_xor_sync(kFull, s0, 16);
    k1 += __shfl_xor_sync(kFull, s1, 16);
    float k = h8 ? k1 : k0;
    k += __shfl_xor_sync(kFull, h8 ? k0 : k1, 8);
    k += __shfl_xor_sync(kFull, k, 4);
    k += __shfl_xor_sync(kFull, k, 2);
    k += __shfl_xor_sync(kFull, k, 1);
    return k;
}

// The integer walk for int4-grouped rows (one fp32 scale per gs inputs of a row, gs a multiple of
// 32, so a 16-byte chunk lies in one group): each chunk's limb sums (exact integers, multiples of
// 2^LOG_SC) are converted to float, joined and multiplied by the chunk's group scale as the chunk
// is consumed; the rows' float partials are reduced across the warp at the unit's end. Lane l
// takes chunks l + 32 k, whose group it tracks incrementally (no division per chunk), and loads
// each chunk's scale with its weights. scl_of(i, sr) gives unit i's rows' scale rows
// ([ceil(In / gs)] floats each); epi(i, tot) gets, in lane l, the scaled total of row l / 8 (in
// units of the activations' fixed point).
template <int FMT, int INFL, class RowsOf, class SclOf, class XqOf, class Epi>
__device__ __forceinline__ void warp_stream_int_grouped(int nunits, int CPR, int gs, int lane, RowsOf rows_of,
                                                        SclOf scl_of, XqOf xq_of, Epi epi) {
    constexpr int NR = 4, kDepth = INFL / NR;
    constexpr int LS = IQ<FMT>::LOG_SC;
    constexpr float k0 = 1.f / (1 << LS), k1 = 256.f / (1 << LS), k2 = 65536.f / (1 << LS);
    if (nunits <= 0) return;
    const int S = (CPR + kWarp - 1) / kWarp;
    const int total = nunits * S;
    const int cpg = gs / 32;  // 16-byte int4 chunks per group
    // group of chunk lane + 32 k: starts at lane / cpg and advances by 32 chunks a step
    const int g0 = lane / cpg, r0 = lane - g0 * cpg, gq = kWarp / cpg, gr = kWarp - gq * cpg;
    int ig = g0, irem = r0;
    uint4 buf[kDepth][NR];
    float sbuf[kDepth][NR];
    int iu = 0, ik = 0;
    const uint8_t *rr[NR];
    const float *sr[NR];
    rows_of(0, rr);
    scl_of(0, sr);
    auto issue = [&](uint4 (&b)[NR], float (&sb)[NR]) {
        if (iu < nunits) {
            const int c = lane + kWarp * ik;
#pragma unroll
            for (int r = 0; r < NR; r++) {
                b[r] = c < CPR ? ld_stream_16(rr[r] + 16 * c) : make_uint4(0, 0, 0, 0);
                sb[r] = c < CPR ? __ldg(sr[r] + ig) : 0.f;
            }
            if (++ik == S) {
                ik = 0;
                ig = g0;
                irem = r0;
                if (++iu < nunits) {
                    rows_of(iu, rr);
                    scl_of(iu, sr);
                }
            } else {
                ig += gq;
                irem += gr;
                if (irem >= cpg) {
                    irem -= cpg;
                    ig++;
                }
            }
        }
    };
#pragma unroll
    for (int j = 0; j < kDepth; j++) issue(buf[j], sbuf[j]);
    float facc[NR] = {0.f, 0.f, 0.f, 0.f};
    int cu = 0, ck = 0;
    const uint4 *xq4 = xq_of(0);
    for (int s0 = 0; s0 < total; s0 += kDepth) {
#pragma unroll
        for (int j = 0; j < kDepth; j++) {
            if (s0 + j < total) {
                const int c = lane + kWarp * ck;
                if (c < CPR) {
                    int acc[NR][3];
#pragma unroll
                    for (int r = 0; r < NR; r++) acc[r][0] = acc[r][1] = acc[r][2] = 0;
                    idot_chunk<FMT, NR>(buf[j], xq4, CPR, c, acc);
#pragma unroll
                    for (int r = 0; r < NR; r++) {
                        const float v = fmaf((float)acc[r][2], k2, fmaf((float)acc[r][1], k1, (float)acc[r][0] * k0));
                        facc[r] = fmaf(v, sbuf[j][r], facc[r]);
                    }
                }
                issue(buf[j], sbuf[j]);
                if (++ck == S) {
                    epi(cu, freduce4(facc, lane));
#pragma unroll
                    for (int r = 0; r < NR; r++) facc[r] = 0.f;
                    ck = 0;
                    cu++;
                    if (cu < nunits) xq4 = xq_of(cu);
                }
            }
        }
    }
}

// The walk for multi-token groups on the tensor-core core (mma.cuh): blocks of 16 rows, lane
// (g, c) streaming chunk 4*sigma + c of rows g and g + 8 (rows_of(i, rr) gives block i's two row
// pointers for this lane), two segments of loads in flight across block boundaries (deeper
// register buffers spill at the kernel's 128-register budget and measured slower).
// xb: this lane's staged B column (token and part) at its chunk column; epi(i, d) gets block i's
// accumulators (columns 2c, 2c + 1 of rows g and g + 8).
template <int FMT, class RowsOf, class Epi>
__device__ __forceinline__ void warp_stream_mma(int nblk, int CPR, const uint8_t *xb, int lane, RowsOf rows_of,
                                                Epi epi) {
    using M = MQ<FMT>;
    constexpr int kDepth = 2;
    if (nblk <= 0) return;
    const int NSEG = (CPR + 3) / 4;
    const int total = nblk * NSEG;
    const int c = lane & 3;
    uint4 buf[kDepth][2];
    int iu = 0, is = 0;
    const uint8_t *rr[2];
    rows_of(0, rr);
    auto issue = [&](uint4 (&b)[2]) {
        if (iu < nblk) {
            const int ch = 4 * is + c;
            b[0] = ch < CPR ? ld_stream_16(rr[0] + 16 * ch) : make_uint4(0, 0, 0, 0);
            b[1] = ch < CPR ? ld_stream_16(rr[1] + 16 * ch) : make_uint4(0, 0, 0, 0);
            if (++is == NSEG) {
                is = 0;
                if (++iu < nblk) rows_of(iu, rr);
            }
        }
    };
#pragma unroll
    for (int j = 0; j < kDepth; j++) issue(buf[j]);
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    int cu = 0, cs = 0;
    for (int s0 = 0; s0 < total; s0 += kDepth) {
#pragma unroll
        for (int j = 0; j < kDepth; j++) {
            if (s0 + j < total) {
                seg_mma<FMT>(buf[j], xb + (size_t)cs * M::SEGB, d);
                issue(buf[j]);
                if (++cs == NSEG) {
                    epi(cu, d);
                    d[0] = d[1] = d[2] = d[3] = 0.f;
                    cs = 0;
                    cu++;
                }
            }
        }
    }
}

// ------------------------------------------------------------------ router items
// T <= 8: partial logits of 32 experts (4 per warp) over one slice of H; each lane keeps two
// float4 steps of W_r and x loads in flight
template <int TM>  // tokens handled: P.T <= TM
__device__ __noinline__ void router_item(const DecParams &P, int item) {
    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
    const int eb = item % P.neb, ks = item / P.neb;
    const int kb = ks * P.rks_floats, ke = min(P.H, kb + P.rks_floats);
    float acc[4][TM];
#pragma unroll
    for (int r = 0; r < 4; r++)
#pragma unroll
        for (int t = 0; t < TM; t++) acc[r][t] = 0.f;
    int e[4];
#pragma unroll
    for (int r = 0; r < 4; r++) e[r] = min(eb * kRtE + warp * 4 + r, P.E - 1);
    constexpr int B = 2;
    for (int k0 = kb + 4 * lane; k0 < ke; k0 += 4 * kWarp * B) {
        float4 wv[B][4];
#pragma unroll
        for (int b = 0; b < B; b++) {
            const int k = k0 + b * 4 * kWarp;
#pragma unroll
            for (int r = 0; r < 4; r++) {
                uint4 u = make_uint4(0, 0, 0, 0);
                if (k < ke) u = ld_stream_16(P.Wr + (size_t)e[r] * P.H + k);
                wv[b][r] = make_float4(__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z),
                                       __uint_as_float(u.w));
            }
        }
#pragma unroll
        for (int t = 0; t < TM; t++) {
            if (t >= P.T) break;
            float4 xv[B];
#pragma unroll
            for (int b = 0; b < B; b++) {
                const int k = k0 + b * 4 * kWarp;
                xv[b] = k < ke ? __ldg(reinterpret_cast<const float4 *>(P.x + (size_t)t * P.H + k))
                               : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int b = 0; b < B; b++)
#pragma unroll
                for (int r = 0; r < 4; r++) {
                    float a = acc[r][t];
                    a = fmaf(wv[b][r].x, xv[b].x, a);
                    a = fmaf(wv[b][r].y, xv[b].y, a);
                    a = fmaf(wv[b][r].z, xv[b].z, a);
                    a = fmaf(wv[b][r].w, xv[b].w, a);
                    acc[r][t] = a;
                }
        }
    }
#pragma unroll
    for (int r = 0; r < 4; r++)
#pragma unroll
        for (int t = 0; t < TM; t++) {
            if (t >= P.T) break;
            float s = acc[r][t];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(kFull, s, o);
            const int er = eb * kRtE + warp * 4 + r;
            if (lane == 0 && er < P.E) P.part[((size_t)ks * P.T + t) * P.E + er] = s;
        }
}

// ------------------------------------------------------------------ staging
__device__ __forceinline__ float4 ld_act4(const float *src, int q, bool coherent) {
    return coherent ? __ldcg(reinterpret_cast<const float4 *>(src) + q)
                    : __ldg(reinterpret_cast<const float4 *>(src) + q);
}

}  // namespace
}  // namespace colimoe
