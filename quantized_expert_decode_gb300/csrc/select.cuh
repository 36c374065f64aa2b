// select.cuh — top-K selection of the router choices and the kept weights, shared by the
// router kernel (router.cu), the token-group decode kernel (decode.cu) and the single-token
// kernel (decode1.cu). Internal to libcolimoe.
//
// What it computes (colibri-strix c/glm.c @98759bf, moe() phase A): the greedy K-max of
// choice = sig + bias, scanning experts in ascending id with a strict '>' from -1e30, so equal
// choices go to the lower id; the weights are the sigmoid scores of the picks; then the TOPP
// cut, the renormalisation (+1e-20) and routed_scale.
//
// How: by candidate ranks. Say a beats b when a's choice is higher, or equal and a's id is
// lower. On the selectable experts (choice > -1e30; a NaN choice is never selectable) this is a
// strict total order, and the greedy scan's k-th pick is the expert that exactly k others beat.
//   stage 1  experts in blocks of 32, one per lane: an expert is a candidate when fewer than
//            Ksel of its block-mates beat it. Everything that beats a member of the global top
//            Ksel is itself in the top Ksel, hence in its own block's top Ksel: every top-Ksel
//            member is a candidate, and so is everything that beats it.
//   stage 2  each candidate counts the candidates that beat it. For a top-Ksel member that is
//            its global rank; for any other candidate it is at least Ksel (the whole top Ksel
//            beats it). So rank r < Ksel names the r-th pick.
// Stage 1 costs 32 comparisons per expert, stage 2 (#candidates) per candidate: at E = 256,
// K = 8, 8 blocks leave at most 64 candidates.
#pragma once

#include "common.cuh"

namespace colimoe {
namespace {

// experts per selection block and the padded row length of a choice vector
constexpr int kSelBlock = 32;
__host__ __device__ __forceinline__ int sel_padded(int E) { return (E + kSelBlock - 1) / kSelBlock * kSelBlock; }
// candidate slots one token can need: min(Ksel, 32) per block
__host__ __device__ __forceinline__ int sel_cand_cap(int E, int Ksel) {
    return sel_padded(E) / kSelBlock * (Ksel < kSelBlock ? Ksel : kSelBlock);
}

__device__ __forceinline__ bool sel_beats(float ca, int ea, float cb, int eb) {
    return ca > cb || (ca == cb && ea < eb);
}

// the serial scan starts from -1e30 with a strict '>': only choices above it can be picked
__device__ __forceinline__ bool sel_selectable(float c) { return c > -1e30f; }

// number of the 32 experts of a block (chb: their choices, 16-byte aligned, in shared memory)
// that beat the block's expert `lane`, whose choice is c
__device__ __forceinline__ int sel_block_rank(const float *chb, float c, int lane) {
    const float4 *c4 = reinterpret_cast<const float4 *>(chb);
    int r = 0;
#pragma unroll
    for (int q = 0; q < kSelBlock / 4; q++) {
        const float4 v = c4[q];
        r += sel_beats(v.x, 4 * q + 0, c, lane);
        r += sel_beats(v.y, 4 * q + 1, c, lane);
        r += sel_beats(v.z, 4 * q + 2, c, lane);
        r += sel_beats(v.w, 4 * q + 3, c, lane);
    }
    return r;
}

// number of the n candidates (choice, id bits) that beat (c, e); unrolled so that several
// shared-memory loads are in flight
__device__ __forceinline__ int sel_cand_rank(const float2 *cand, int n, float c, int e) {
    int r = 0;
#pragma unroll 8
    for (int j = 0; j < n; j++) {
        const float2 o = cand[j];
        r += sel_beats(o.x, __float_as_int(o.y), c, e);
    }
    return r;
}

// One warp selects for one token. ch: the token's choices in shared memory, sel_padded(E)
// entries with -inf beyond E; cand: this warp's scratch of sel_cand_cap(E, Ksel) float2.
// Writes the ids of picks 0..n-1 to sel_i (shared or global) and returns n = min(Ksel, number
// of selectable experts), the same in every lane.
__device__ int sel_topk_warp(const float *ch, int E, int Ksel, float2 *cand, int *sel_i) {
    const int lane = threadIdx.x % kWarp;
    const int nb = sel_padded(E) / kSelBlock;
    int n = 0, nok = 0;
    for (int b = 0; b < nb; b++) {
        const float *chb = ch + b * kSelBlock;
        const float c = chb[lane];
        const bool ok = sel_selectable(c);
        const bool is_cand = ok && sel_block_rank(chb, c, lane) < Ksel;
        const unsigned m = __ballot_sync(kFull, is_cand);
        if (is_cand) cand[n + __popc(m & ((1u << lane) - 1u))] = make_float2(c, __int_as_float(b * kSelBlock + lane));
        n += __popc(m);
        nok += __popc(__ballot_sync(kFull, ok));
    }
    __syncwarp();
    for (int i = lane; i < n; i += kWarp) {
        const float2 me = cand[i];
        const int e = __float_as_int(me.y);
        const int r = sel_cand_rank(cand, n, me.x, e);
        if (r < Ksel) sel_i[r] = e;
    }
    __syncwarp();
    return nok < Ksel ? nok : Ksel;
}

// The whole CTA selects for one token (stage 1 over the warps, stage 2 over the threads).
// ch as above; cand: sel_cand_cap(E, Ksel) float2 and ncand / nok: two ints, all in shared
// memory, the ints zeroed before the call and published by a barrier. Picks go to sel_i;
// after the call's closing barrier *nok is the number of selectable experts.
__device__ void sel_topk_cta(const float *ch, int E, int Ksel, float2 *cand, int *ncand, int *nok, int *sel_i) {
    const int lane = threadIdx.x % kWarp, warp = threadIdx.x / kWarp, nw = blockDim.x / kWarp;
    const int nb = sel_padded(E) / kSelBlock;
    for (int b = warp; b < nb; b += nw) {
        const float *chb = ch + b * kSelBlock;
        const float c = chb[lane];
        const bool ok = sel_selectable(c);
        const bool is_cand = ok && sel_block_rank(chb, c, lane) < Ksel;
        const unsigned m = __ballot_sync(kFull, is_cand);
        const unsigned mo = __ballot_sync(kFull, ok);
        int base = 0;
        if (lane == 0) {
            base = atomicAdd(ncand, __popc(m));
            atomicAdd(nok, __popc(mo));
        }
        base = __shfl_sync(kFull, base, 0);
        if (is_cand) cand[base + __popc(m & ((1u << lane) - 1u))] = make_float2(c, __int_as_float(b * kSelBlock + lane));
    }
    __syncthreads();
    const int n = *ncand;
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const float2 me = cand[i];
        const int e = __float_as_int(me.y);
        const int r = sel_cand_rank(cand, n, me.x, e);
        if (r < Ksel) sel_i[r] = e;
    }
    __syncthreads();
}

// The kept experts of one token and their weights, one warp: on entry lane k < nsel holds pick
// k (id, sigmoid score) in selection order. TOPP (top_p in (0,1)): the picks sorted by score,
// descending and stable (the pages' insertion sort), keep the shortest prefix whose running
// sum reaches top_p * (1e-20 + total). Then, if norm_topk, each weight is divided by
// (sum of the kept weights in order + 1e-20), and multiplied by routed_scale. On return lane
// k < Ke holds kept pick k (its id and final weight); other lanes hold id -1 and weight 0.
// Returns Ke. The float operations and their order are the serial code's.
struct SelKept {
    int id;
    float w;
    int ke;
};

__device__ SelKept sel_finish_warp(int nsel, int id, float wv, float top_p, int norm_topk, float rscale) {
    const int lane = threadIdx.x % kWarp;
    if (lane >= nsel) {
        id = -1;
        wv = 0.f;
    }
    int ke = nsel;
    if (top_p > 0.f && top_p < 1.f && nsel > 0) {
        int p = 0;  // place of this pick in the stable descending order of scores
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
        for (int k = 0; k < nsel; k++) {
            cum = __fadd_rn(cum, __shfl_sync(kFull, wv, k));
            if (cum >= lim) {
                ke = k + 1;
                break;
            }
        }
    }
    float sm = 1.f;
    if (norm_topk) {
        sm = 0.f;
        for (int k = 0; k < ke; k++) sm = __fadd_rn(sm, __shfl_sync(kFull, wv, k));
        sm = __fadd_rn(sm, 1e-20f);
    }
    const bool kept = lane < ke;
    const float wn = kept ? (norm_topk ? __fdiv_rn(wv, sm) : wv) : 0.f;
    SelKept r;
    r.id = kept ? id : -1;
    r.w = kept ? __fmul_rn(wn, rscale) : 0.f;
    r.ke = ke;
    return r;
}

}  // namespace
}  // namespace colimoe
