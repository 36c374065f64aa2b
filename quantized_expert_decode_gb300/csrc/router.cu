// router.cu — router logits, top-K selection and token->expert bucketing.
//
// Phase A of moe() in colibri-strix c/glm.c @98759bf (and the r_router
// shader of colibri c/backend_metal.mm @93cde63): logit = x . W_r[e] in fp32,
// sig = 1/(1+exp(-logit)), choice = sig + bias[e], greedy top-K over choice with ties to the
// lower expert index, w = sig of the chosen experts, optional TOPK / TOPP, renormalisation
// and routed_scale. Phase B (batch union) becomes a stable counting sort of the assignment
// ids a = t*K + k by expert.
#include <cmath>

#include "kernels.h"
#include "select.cuh"

namespace colimoe {

// ---------------------------------------------------------------- router partial logits
// part[s][t][e] = sum over the s-th slice of H of x[t][h] * W_r[e][h]. A 32-token x 64-expert
// output tile per CTA, k staged through shared memory 32 at a time; the k range is split
// into `splits` slices so that small T still fills the GPU. Partials are summed in a fixed
// order by the selection kernel (no atomics: the logits are reproducible run to run).
__global__ void __launch_bounds__(256)
router_partial_kernel(const float *__restrict__ x, const float *__restrict__ Wr,
                      float *__restrict__ part, int T, int H, int E, int kslice) {
    constexpr int TM = kRouterTM, TE = kRouterTE, TK = kRouterTK;
    __shared__ float xs[TK][TM + 4];
    __shared__ __align__(16) float wsm[TK][TE + 4];
    const int tid = threadIdx.x;
    const int t0 = blockIdx.x * TM, e0 = blockIdx.y * TE, s = blockIdx.z;
    const int kb = s * kslice;
    const int ke = min(H, kb + kslice);
    const int tx = tid % 16, ty = tid / 16;  // experts tx*4..+3, tokens ty*2..+1
    float acc[2][4] = {};
    for (int k0 = kb; k0 < ke; k0 += TK) {
        {   // x tile: 32 tokens x 32 k, one float4 per thread, stored k-major
            const int r = tid / 8, kc = (tid % 8) * 4;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (t0 + r < T && k0 + kc < ke)
                v = *reinterpret_cast<const float4 *>(x + (size_t)(t0 + r) * H + k0 + kc);
            xs[kc + 0][r] = v.x;
            xs[kc + 1][r] = v.y;
            xs[kc + 2][r] = v.z;
            xs[kc + 3][r] = v.w;
        }
#pragma unroll
        for (int half = 0; half < 2; half++) {  // W_r tile: 64 experts x 32 k
            const int r = half * 32 + tid / 8, kc = (tid % 8) * 4;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (e0 + r < E && k0 + kc < ke)
                v = *reinterpret_cast<const float4 *>(Wr + (size_t)(e0 + r) * H + k0 + kc);
            wsm[kc + 0][r] = v.x;
            wsm[kc + 1][r] = v.y;
            wsm[kc + 2][r] = v.z;
            wsm[kc + 3][r] = v.w;
        }
        __syncthreads();
#pragma unroll 8
        for (int k = 0; k < TK; k++) {
            const float a0 = xs[k][ty * 2], a1 = xs[k][ty * 2 + 1];
            const float4 b = *reinterpret_cast<const float4 *>(&wsm[k][tx * 4]);
            acc[0][0] = fmaf(a0, b.x, acc[0][0]);
            acc[0][1] = fmaf(a0, b.y, acc[0][1]);
            acc[0][2] = fmaf(a0, b.z, acc[0][2]);
            acc[0][3] = fmaf(a0, b.w, acc[0][3]);
            acc[1][0] = fmaf(a1, b.x, acc[1][0]);
            acc[1][1] = fmaf(a1, b.y, acc[1][1]);
            acc[1][2] = fmaf(a1, b.z, acc[1][2]);
            acc[1][3] = fmaf(a1, b.w, acc[1][3]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 2; i++) {
        const int t = t0 + ty * 2 + i;
        if (t >= T) continue;
#pragma unroll
        for (int j = 0; j < 4; j++) {
            const int e = e0 + tx * 4 + j;
            if (e < E) part[((size_t)s * T + t) * E + e] = acc[i][j];
        }
    }
}

// The same partials for many tokens: a 128-token x 128-expert tile per CTA over one k slice,
// each thread 8 tokens x 8 experts (tokens 4 ty + i and 64 + 4 ty + i, experts 4 tx + j and
// 64 + 4 tx + j), k staged through shared memory kRgK at a time in two buffers (the next stage's
// loads in registers while this one is used). Each partial is a plain fp32 sum in k order.
__global__ void __launch_bounds__(256)
router_gemm_kernel(const float *__restrict__ x, const float *__restrict__ Wr, float *__restrict__ part, int T,
                   int H, int E, int kslice) {
    __shared__ __align__(16) float xs[2][kRgK][kRgT + 4];
    __shared__ __align__(16) float ws[2][kRgK][kRgE + 4];
    const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
    const int t0 = blockIdx.x * kRgT, e0 = blockIdx.y * kRgE, s = blockIdx.z;
    const int kb = s * kslice, ke = min(H, kb + kslice);
    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; i++)
#pragma unroll
        for (int j = 0; j < 8; j++) acc[i][j] = 0.f;
    // global loads: row r = tid / 4 + 64 i of each operand tile, float4 q = tid % 4 of the stage
    const int lr = tid / 4, lq = tid % 4;
    float4 xv[2], wv[2];
    auto gload = [&](int k0) {
        const int k = k0 + 4 * lq;  // H and the slices are multiples of 16: k < ke covers k + 3
#pragma unroll
        for (int i = 0; i < 2; i++) {
            const int r = lr + 64 * i;
            const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
            xv[i] = (t0 + r < T && k < ke) ? __ldg(reinterpret_cast<const float4 *>(x + (size_t)(t0 + r) * H + k)) : z;
            wv[i] = (e0 + r < E && k < ke) ? __ldg(reinterpret_cast<const float4 *>(Wr + (size_t)(e0 + r) * H + k)) : z;
        }
    };
    auto sstore = [&](int b) {
#pragma unroll
        for (int i = 0; i < 2; i++) {
            const int r = lr + 64 * i;
            xs[b][4 * lq + 0][r] = xv[i].x;
            xs[b][4 * lq + 1][r] = xv[i].y;
            xs[b][4 * lq + 2][r] = xv[i].z;
            xs[b][4 * lq + 3][r] = xv[i].w;
            ws[b][4 * lq + 0][r] = wv[i].x;
            ws[b][4 * lq + 1][r] = wv[i].y;
            ws[b][4 * lq + 2][r] = wv[i].z;
            ws[b][4 * lq + 3][r] = wv[i].w;
        }
    };
    int buf = 0;
    if (kb < ke) {
        gload(kb);
        sstore(0);
    }
    __syncthreads();
    for (int k0 = kb; k0 < ke; k0 += kRgK) {
        const bool more = k0 + kRgK < ke;
        if (more) gload(k0 + kRgK);
#pragma unroll
        for (int k = 0; k < kRgK; k++) {
            const float4 a0 = *reinterpret_cast<const float4 *>(&xs[buf][k][4 * ty]);
            const float4 a1 = *reinterpret_cast<const float4 *>(&xs[buf][k][64 + 4 * ty]);
            const float4 b0 = *reinterpret_cast<const float4 *>(&ws[buf][k][4 * tx]);
            const float4 b1 = *reinterpret_cast<const float4 *>(&ws[buf][k][64 + 4 * tx]);
            const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int i = 0; i < 8; i++)
#pragma unroll
                for (int j = 0; j < 8; j++) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        if (more) sstore(buf ^ 1);  // the other buffer: every thread is past its last use
        __syncthreads();
        buf ^= 1;
    }
#pragma unroll
    for (int i = 0; i < 8; i++) {
        const int t = t0 + (i < 4 ? 4 * ty + i : 64 + 4 * ty + i - 4);
        if (t >= T) continue;
#pragma unroll
        for (int j = 0; j < 8; j++) {
            const int e = e0 + (j < 4 ? 4 * tx + j : 64 + 4 * tx + j - 4);
            if (e < E) part[((size_t)s * T + t) * E + e] = acc[i][j];
        }
    }
}

cudaError_t launch_router_partial(const float *x, const float *W_r, float *part, int T, int H,
                                  int E, int splits, cudaStream_t st) {
    if (T >= kRouterBigT) {
        int kslice = (H + splits - 1) / splits;
        kslice = (kslice + kRgK - 1) / kRgK * kRgK;
        dim3 grid((T + kRgT - 1) / kRgT, (E + kRgE - 1) / kRgE, splits);
        router_gemm_kernel<<<grid, 256, 0, st>>>(x, W_r, part, T, H, E, kslice);
        return cudaGetLastError();
    }
    int kslice = (H + splits - 1) / splits;
    kslice = (kslice + kRouterTK - 1) / kRouterTK * kRouterTK;
    dim3 grid((T + kRouterTM - 1) / kRouterTM, (E + kRouterTE - 1) / kRouterTE, splits);
    router_partial_kernel<<<grid, 256, 0, st>>>(x, W_r, part, T, H, E, kslice);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- top-K selection
// One warp per token (eight per CTA): the logits are the partial slices summed in a fixed
// order, then sigmoid and bias; the selection and the kept weights are select.cuh's (candidate
// ranks over blocks of 32 experts, then the TOPP / renorm / scale tail in the serial code's
// float order). Per warp, shared memory holds the token's choices and scores (padded to whole
// blocks), the candidates and the picks.
constexpr int kSelWarps = 8;

__host__ __device__ __forceinline__ int select_warp_floats(int E, int Ksel) {
    return (2 * sel_padded(E) + 2 * sel_cand_cap(E, Ksel) + kMaxK + 3) / 4 * 4;
}

__global__ void __launch_bounds__(kSelWarps * kWarp)
select_kernel(const float *__restrict__ part, int S, const float *__restrict__ bias, int T, int E,
              int K, int Ksel, float top_p, int norm_topk, float routed_scale,
              float *__restrict__ sig_out, float *__restrict__ ch_out, int32_t *__restrict__ idx,
              float *__restrict__ w, int32_t *__restrict__ keff, int32_t *__restrict__ err) {
    extern __shared__ __align__(16) float sel_smem[];
    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
    const int t = blockIdx.x * kSelWarps + warp;
    if (t >= T) return;  // the whole warp: nothing below synchronises the CTA
    const int Ep = sel_padded(E), cap = sel_cand_cap(E, Ksel);
    float *ch = sel_smem + (size_t)warp * select_warp_floats(E, Ksel);
    float *sg = ch + Ep;
    float2 *cand = reinterpret_cast<float2 *>(sg + Ep);
    int *sel_i = reinterpret_cast<int *>(cand + cap);
    // the lane's experts e = lane + 32 j, kEL at a time, their partial slices summed in slice
    // order; the loads of kSB slices of all kEL experts are in flight together
    constexpr int kEL = 8, kSB = 8;
    for (int e0 = lane; e0 < Ep; e0 += kWarp * kEL) {
        float lg[kEL];
#pragma unroll
        for (int j = 0; j < kEL; j++) lg[j] = 0.f;
        for (int s0 = 0; s0 < S; s0 += kSB) {
            float v[kEL][kSB];
#pragma unroll
            for (int j = 0; j < kEL; j++)
#pragma unroll
                for (int b = 0; b < kSB; b++) {
                    const int e = e0 + kWarp * j, s = s0 + b;
                    v[j][b] = (e < E && s < S) ? part[((size_t)s * T + t) * E + e] : 0.f;
                }
#pragma unroll
            for (int j = 0; j < kEL; j++)
#pragma unroll
                for (int b = 0; b < kSB; b++)
                    if (s0 + b < S) lg[j] += v[j][b];
        }
#pragma unroll
        for (int j = 0; j < kEL; j++) {
            const int e = e0 + kWarp * j;
            if (e >= Ep) break;
            if (e < E) {
                const float sv = 1.f / (1.f + expf(-lg[j]));
                const float cv = sv + bias[e];
                sig_out[(size_t)t * E + e] = sv;
                ch_out[(size_t)t * E + e] = cv;
                sg[e] = sv;
                ch[e] = cv;
            } else {
                sg[e] = 0.f;
                ch[e] = -INFINITY;
            }
        }
    }
    __syncwarp();
    const int nsel = sel_topk_warp(ch, E, Ksel, cand, sel_i);
    if (nsel < Ksel && lane == 0) atomicCAS(err, 0, (int)kErrNoCandidate);
    const int id = lane < nsel ? sel_i[lane] : -1;
    const SelKept kp = sel_finish_warp(nsel, id, lane < nsel ? sg[id] : 0.f, top_p, norm_topk, routed_scale);
    if (lane < K) {
        idx[(size_t)t * K + lane] = kp.id;
        w[(size_t)t * K + lane] = kp.w;
    }
    if (lane == 0 && keff) keff[t] = kp.ke;
}

cudaError_t launch_select(const float *part, int splits, const float *bias, int T, int E, int K,
                          int ksel, float top_p, int norm_topk, float routed_scale, float *sig,
                          float *choice, int32_t *idx, float *w, int32_t *keff, int32_t *err,
                          cudaStream_t st) {
    const int Ksel = (ksel > 0 && ksel < K) ? ksel : K;
    const size_t smem = (size_t)kSelWarps * select_warp_floats(E, Ksel) * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    select_kernel<<<(T + kSelWarps - 1) / kSelWarps, kSelWarps * kWarp, smem, st>>>(
        part, splits, bias, T, E, K, Ksel, top_p, norm_topk, routed_scale, sig, choice, idx, w, keff, err);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- buckets
// Exclusive scan over the 1024 threads of the block; returns this thread's prefix and the
// block total in *total.
__device__ int block_excl_scan_1024(int v, int *scratch /* >= 33 ints */, int *total) {
    const int lane = threadIdx.x % kWarp, warp = threadIdx.x / kWarp;
    int inc = v;
#pragma unroll
    for (int o = 1; o < kWarp; o <<= 1) {
        const int n = __shfl_up_sync(kFull, inc, o);
        if (lane >= o) inc += n;
    }
    if (lane == kWarp - 1) scratch[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        int ws = scratch[lane];
        int wi = ws;
#pragma unroll
        for (int o = 1; o < kWarp; o <<= 1) {
            const int n = __shfl_up_sync(kFull, wi, o);
            if (lane >= o) wi += n;
        }
        scratch[lane] = wi - ws;  // exclusive prefix of warp totals
        if (lane == kWarp - 1) scratch[32] = wi;
    }
    __syncthreads();
    const int r = scratch[warp] + inc - v;
    *total = scratch[32];
    __syncthreads();
    return r;
}

// Single CTA of 1024 threads. counts[e] = assignments of expert e; offsets = exclusive scan;
// perm lists the kept assignments a (k < keff[t]) grouped by expert, ascending a within an
// expert (each 1024-assignment chunk is placed in order: rank inside the warp from a
// match-any mask, then the warps' per-expert counts are scanned); pos[a] is a's slot in
// perm (-1 when not kept); act lists the experts with a non-empty bucket, ascending;
// meta = {U, N}.
__global__ void __launch_bounds__(1024)
bucket_kernel(const int32_t *__restrict__ idx, const int32_t *__restrict__ keff, int T, int K,
              int E, int32_t *__restrict__ counts, int32_t *__restrict__ offsets,
              int32_t *__restrict__ perm, int32_t *__restrict__ pos, int32_t *__restrict__ act,
              int32_t *__restrict__ meta, int32_t *__restrict__ err) {
    extern __shared__ int sm[];
    int *cnt = sm;                 // [E]
    int *off = cnt + E;            // [E]
    int *fill = off + E;           // [E]
    int *chunk = fill + E;         // [E]
    int *wc = chunk + E;           // [32][E]
    int *scratch = wc + 32 * E;    // [33]
    const int tid = threadIdx.x, lane = tid % kWarp, warp = tid / kWarp;
    const int N = T * K;
    auto expert_of = [&](int a) -> int {
        if (a >= N) return -1;
        const int t = a / K, k = a % K;
        if (keff && k >= keff[t]) return -1;
        const int e = idx[a];
        if (e < 0 || e >= E) {
            atomicCAS(err, 0, (int)kErrBadExpert);
            return -1;
        }
        return e;
    };
    for (int e = tid; e < E; e += blockDim.x) {
        cnt[e] = 0;
        fill[e] = 0;
    }
    __syncthreads();
    for (int a = tid; a < N; a += blockDim.x) {
        const int e = expert_of(a);
        if (e >= 0) atomicAdd(&cnt[e], 1);
    }
    __syncthreads();
    // offsets and the active list (E <= 1024: one expert per thread)
    {
        const int c = tid < E ? cnt[tid] : 0;
        int tot;
        const int ex = block_excl_scan_1024(c, scratch, &tot);
        if (tid < E) {
            off[tid] = ex;
            counts[tid] = c;
            offsets[tid] = ex;
        }
        if (tid == 0) offsets[E] = tot;
        int nact;
        const int ax = block_excl_scan_1024(c > 0 ? 1 : 0, scratch, &nact);
        if (tid < E && c > 0) act[ax] = tid;
        if (tid == 0) {
            meta[0] = nact;
            meta[1] = tot;
        }
    }
    __syncthreads();
    for (int a0 = 0; a0 < N; a0 += blockDim.x) {
        for (int i = tid; i < 32 * E; i += blockDim.x) wc[i] = 0;
        __syncthreads();
        const int a = a0 + tid;
        const int e = expert_of(a);
        const unsigned peers = __match_any_sync(kFull, e);
        const int rank = __popc(peers & ((1u << lane) - 1u));
        if (e >= 0 && rank == 0) wc[warp * E + e] = __popc(peers);
        __syncthreads();
        for (int x = tid; x < E; x += blockDim.x) {
            int run = 0;
            for (int w = 0; w < 32; w++) {
                const int v = wc[w * E + x];
                wc[w * E + x] = run;
                run += v;
            }
            chunk[x] = run;
        }
        __syncthreads();
        if (a < N) {
            if (e >= 0) {
                const int p = off[e] + fill[e] + wc[warp * E + e] + rank;
                perm[p] = a;
                pos[a] = p;
            } else {
                pos[a] = -1;
            }
        }
        __syncthreads();
        for (int x = tid; x < E; x += blockDim.x) fill[x] += chunk[x];
        __syncthreads();
    }
}

cudaError_t launch_bucket(const int32_t *idx, const int32_t *keff, int T, int K, int E,
                          int32_t *counts, int32_t *offsets, int32_t *perm, int32_t *pos,
                          int32_t *act, int32_t *meta, int32_t *err, cudaStream_t st) {
    const size_t smem = (size_t)(4 * E + 32 * E + 33) * sizeof(int);
    cudaError_t e = cudaFuncSetAttribute(bucket_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    bucket_kernel<<<1, 1024, smem, st>>>(idx, keff, T, K, E, counts, offsets, perm, pos, act, meta,
                                         err);
    return cudaGetLastError();
}

}  // namespace colimoe
