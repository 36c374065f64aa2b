// expert.cu — dequant-on-use expert GEMVs (gate+up with SiLU*mul, down), the weighted combine,
// and the standalone quantized GEMV.
//
// Phases C/D/E of moe() in colibri-strix c/glm.c @98759bf (per unique expert: gather its rows,
// g = gate.x, u = up.x, h = silu(g)*u, y = down.h, out[row] += w*y; then the shared expert with
// weight 1) and the moe_gemv / moe_silu shaders of colibri c/backend_metal.mm @93cde63.
// Gate and up are fused in one pass over x (the idea of matmul_i4_pair in the later glm.c).
#include "idot.cuh"
#include "kernels.h"
#include "qdot.cuh"

namespace colimoe {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / kWarp;
constexpr int kNV = 4;              // activation vectors per pass
constexpr int kGuRowsPerCta = 16;   // gate/up row pairs per CTA (2 per warp)
constexpr int kDnRowsPerCta = 32;   // down rows per CTA (4 per warp)

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.f + expf(-g)) * u; }

__device__ __forceinline__ bool misaligned16(const void *p) {
    return (reinterpret_cast<uintptr_t>(p) & 15u) != 0;
}

// Work of one slot of the expert grid: which expert, its tokens, where its rows go.
struct Slot {
    coli_moe_expert ex;
    int fmt, inter;  // weight format and intermediate size of this expert
    int n;           // tokens using it
    int pbase;       // first bucket position (routed) — h/y rows are pbase + v
    bool shared;
};

__device__ __forceinline__ bool resolve_slot(const ExpertWork &W, int slot, Slot &s) {
    const bool has_shared = W.I_shared > 0;
    if (has_shared && slot == 0) {
        s.ex = W.shared;
        s.fmt = W.shared_fmt;
        s.inter = W.I_shared;
        s.n = W.T;
        s.pbase = 0;
        s.shared = true;
        return true;
    }
    const int r = has_shared ? slot - 1 : slot;
    if (r >= W.meta[0]) return false;
    const int e = W.act[r];
    s.ex = W.experts[e];
    s.fmt = W.routed_fmt;
    s.inter = W.I;
    s.n = W.counts[e];
    s.pbase = W.offsets[e];
    s.shared = false;
    if (misaligned16(s.ex.gate_w) || misaligned16(s.ex.up_w) || misaligned16(s.ex.down_w) ||
        (reinterpret_cast<uintptr_t>(s.ex.gate_s) & 3u) || (reinterpret_cast<uintptr_t>(s.ex.up_s) & 3u) ||
        (reinterpret_cast<uintptr_t>(s.ex.down_s) & 3u)) {
        if (threadIdx.x == 0) atomicCAS(W.err, 0, (int)kErrBadExpert);
        return false;
    }
    return true;
}

// ---------------------------------------------------------------- IDOT (int8 activations)
// glm.c's IDOT kernels (qrow_i8, dot_i8i8 / dot_i4i8, matmul_q_idot / matmul_i4_idot): each
// activation row is quantised to int8 with one scale, s = max(max|x| / 127, 1e-12) and
// q = round-half-even(x * (1/s)), every division and product rounded as IEEE fp32; the dot with
// the dequantised weights is an exact integer sum, and y[o] = ((float)dot * scale[o]) * s.
// Staged layout (one u32 = four activation bytes per token): u32 (wi * NGW + g) * CPR + c holds
// the elements that meet field group g of word wi of chunk c (idot.cuh signed_fields), so the
// 32 lanes of a warp, on consecutive chunks, read consecutive u32s.
template <int FMT>
__device__ void stage_idot(const float *__restrict__ src, int len, uint32_t *xq, float *sx_out) {
    using G = QGeom<FMT>;
    using I = IQ<FMT>;
    __shared__ float red[kWarps];
    const int tid = threadIdx.x, lane = tid % kWarp, warp = tid / kWarp;
    float mx = 0.f;
    for (int i = tid; i < len / 4; i += kThreads) {
        const float4 v = __ldg(reinterpret_cast<const float4 *>(src) + i);
        mx = fmaxf(mx, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
    if (lane == 0) red[warp] = mx;
    __syncthreads();
    float amax = red[0];
#pragma unroll
    for (int w = 1; w < kWarps; w++) amax = fmaxf(amax, red[w]);
    __syncthreads();  // red is reused by the next vector
    float sq = __fdiv_rn(amax, 127.f);
    if (sq < 1e-12f) sq = 1e-12f;
    const float inv = __fdiv_rn(1.f, sq);
    const int CPR = len / G::EPC, n = 4 * I::NGW * CPR;
    for (int it = tid; it < n; it += kThreads) {
        const int c = it % CPR, rest = it / CPR, g = rest % I::NGW, wi = rest / I::NGW;
        uint32_t word = 0;
#pragma unroll
        for (int b = 0; b < 4; b++) {
            const int el = c * G::EPC + wi * G::EPW + (FMT == COLI_FMT_INT4 ? 2 * b + g : b);
            const int q = __float2int_rn(__fmul_rn(__ldg(src + el), inv));
            word |= (uint32_t)(q & 0xFF) << (8 * b);
        }
        xq[it] = word;
    }
    if (tid == 0) *sx_out = sq;
}

// exact integer dots of NR packed rows (int8 or int4) with NV staged int8 vectors (xq, xstride
// u32 per vector), lane share of the chunks reduced across the warp: every lane gets the totals
template <int FMT, int NR, int NV>
__device__ __forceinline__ void idot_rows(const uint8_t *const (&rows)[NR], const uint32_t *xq, int xstride, int CPR,
                                          int lane, int (&out)[NR][NV]) {
    using I = IQ<FMT>;
    int acc[NR][NV];
#pragma unroll
    for (int r = 0; r < NR; r++)
#pragma unroll
        for (int v = 0; v < NV; v++) acc[r][v] = 0;
    for (int c = lane; c < CPR; c += kWarp) {
        uint4 w[NR];
#pragma unroll
        for (int r = 0; r < NR; r++) w[r] = ld_stream_16(rows[r] + 16 * c);
#pragma unroll
        for (int wi = 0; wi < 4; wi++)
#pragma unroll
            for (int g = 0; g < I::NGW; g++) {
                uint32_t a[NR];
#pragma unroll
                for (int r = 0; r < NR; r++) a[r] = signed_fields<FMT>(word_of(w[r], wi), g);
#pragma unroll
                for (int v = 0; v < NV; v++) {
                    const uint32_t xv = xq[v * xstride + (wi * I::NGW + g) * CPR + c];
#pragma unroll
                    for (int r = 0; r < NR; r++) acc[r][v] = dp4a_s<true>(a[r], xv, acc[r][v]);
                }
            }
    }
#pragma unroll
    for (int r = 0; r < NR; r++)
#pragma unroll
        for (int v = 0; v < NV; v++) {
            int t = acc[r][v];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(kFull, t, o);
            out[r][v] = t >> I::LOG_SC;  // every product carries the exact factor 2^LOG_SC
        }
}

__device__ __forceinline__ float idot_scale(int dot, float sc, float sx) {
    return __fmul_rn(__fmul_rn(__int2float_rn(dot), sc), sx);
}

// Row of h / y that holds token v of the slot (routed: its bucket position; shared: T*K + t).
__device__ __forceinline__ int slot_row(const ExpertWork &W, const Slot &s, int v) {
    return s.shared ? W.T * W.K + v : s.pbase + v;
}
__device__ __forceinline__ int slot_token(const ExpertWork &W, const Slot &s, int v) {
    return s.shared ? v : W.perm[s.pbase + v] / W.K;
}

// GRP: COLI_FMT_INT4G weights (FMT is then the int4 layout): per-group scales inside the sum
template <int FMT, int NV, bool GRP>
__device__ __forceinline__ void gateup_pass(const ExpertWork &W, const Slot &s, int j0, int v0, int nv,
                                            const float *xs, int CPR) {
    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
    const int64_t rb = row_bytes(FMT, W.H);
    int jp[2];
    const uint8_t *rows[4];
#pragma unroll
    for (int p = 0; p < 2; p++) {
        jp[p] = j0 + 2 * warp + p;
        const int jc = min(jp[p], s.inter - 1);
        rows[2 * p] = static_cast<const uint8_t *>(s.ex.gate_w) + jc * rb;
        rows[2 * p + 1] = static_cast<const uint8_t *>(s.ex.up_w) + jc * rb;
    }
    float out[4][NV];
    if constexpr (GRP) {
        const int ng = (W.H + W.group_size - 1) / W.group_size;
        const float *srows[4];
#pragma unroll
        for (int p = 0; p < 2; p++) {
            const int jc = min(jp[p], s.inter - 1);
            srows[2 * p] = s.ex.gate_s + (size_t)jc * ng;
            srows[2 * p + 1] = s.ex.up_s + (size_t)jc * ng;
        }
        qdot_rows_grouped<4, NV>(rows, srows, W.group_size / 32, xs, W.H, CPR, lane, out);
    } else {
        qdot_rows<FMT, 4, NV>(rows, xs, W.H, CPR, lane, out);
    }
#pragma unroll
    for (int v = 0; v < NV; v++) {
        if (lane != v || v >= nv) continue;
        const int hr = slot_row(W, s, v0 + v);
#pragma unroll
        for (int p = 0; p < 2; p++) {
            if (jp[p] >= s.inter) continue;
            const float g = GRP ? out[2 * p][v] : out[2 * p][v] * s.ex.gate_s[jp[p]];
            const float u = GRP ? out[2 * p + 1][v] : out[2 * p + 1][v] * s.ex.up_s[jp[p]];
            W.h[(size_t)hr * W.ldh + jp[p]] = silu_mul(g, u);
        }
    }
}

template <int FMT, bool GRP = false>
__device__ void gateup_slot(const ExpertWork &W, const Slot &s, float *xs) {
    using G = QGeom<FMT>;
    const int j0 = blockIdx.x * kGuRowsPerCta;
    if (j0 >= s.inter) return;
    const int CPR = W.H / G::EPC;
    for (int v0 = 0; v0 < s.n; v0 += kNV) {
        const int nv = min(kNV, s.n - v0);
        __syncthreads();
        for (int v = 0; v < nv; v++)
            stage_vec<FMT>(W.x + (size_t)slot_token(W, s, v0 + v) * W.H, xs + v * W.H, W.H, CPR,
                           threadIdx.x, kThreads);
        if (nv == 3)
            for (int i = threadIdx.x; i < W.H; i += kThreads) xs[3 * W.H + i] = 0.f;
        __syncthreads();
        if (nv == 1) gateup_pass<FMT, 1, GRP>(W, s, j0, v0, nv, xs, CPR);
        else if (nv == 2) gateup_pass<FMT, 2, GRP>(W, s, j0, v0, nv, xs, CPR);
        else gateup_pass<FMT, 4, GRP>(W, s, j0, v0, nv, xs, CPR);
    }
}

template <int FMT, int NV>
__device__ __forceinline__ void gateup_pass_idot(const ExpertWork &W, const Slot &s, int j0, int v0, int nv,
                                                 const uint32_t *xq, const float *sxv, int CPR) {
    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
    const int64_t rb = row_bytes(FMT, W.H);
    int jp[2];
    const uint8_t *rows[4];
#pragma unroll
    for (int p = 0; p < 2; p++) {
        jp[p] = j0 + 2 * warp + p;
        const int jc = min(jp[p], s.inter - 1);
        rows[2 * p] = static_cast<const uint8_t *>(s.ex.gate_w) + jc * rb;
        rows[2 * p + 1] = static_cast<const uint8_t *>(s.ex.up_w) + jc * rb;
    }
    int out[4][NV];
    idot_rows<FMT, 4, NV>(rows, xq, W.H / 4, CPR, lane, out);
#pragma unroll
    for (int v = 0; v < NV; v++) {
        if (lane != v || v >= nv) continue;
        const int hr = slot_row(W, s, v0 + v);
#pragma unroll
        for (int p = 0; p < 2; p++) {
            if (jp[p] >= s.inter) continue;
            const float g = idot_scale(out[2 * p][v], s.ex.gate_s[jp[p]], sxv[v]);
            const float u = idot_scale(out[2 * p + 1][v], s.ex.up_s[jp[p]], sxv[v]);
            W.h[(size_t)hr * W.ldh + jp[p]] = silu_mul(g, u);
        }
    }
}

template <int FMT>
__device__ void gateup_slot_idot(const ExpertWork &W, const Slot &s, float *xs) {
    __shared__ float sxv[kNV];
    const int j0 = blockIdx.x * kGuRowsPerCta;
    if (j0 >= s.inter) return;
    const int CPR = W.H / QGeom<FMT>::EPC;
    uint32_t *xq = reinterpret_cast<uint32_t *>(xs);
    for (int v0 = 0; v0 < s.n; v0 += kNV) {
        const int nv = min(kNV, s.n - v0);
        __syncthreads();
        for (int v = 0; v < nv; v++)
            stage_idot<FMT>(W.x + (size_t)slot_token(W, s, v0 + v) * W.H, W.H, xq + v * (W.H / 4), &sxv[v]);
        __syncthreads();
        // (a missing fourth vector leaves stale integers in its slot; its sums are not stored)
        if (nv == 1) gateup_pass_idot<FMT, 1>(W, s, j0, v0, nv, xq, sxv, CPR);
        else if (nv == 2) gateup_pass_idot<FMT, 2>(W, s, j0, v0, nv, xq, sxv, CPR);
        else gateup_pass_idot<FMT, 4>(W, s, j0, v0, nv, xq, sxv, CPR);
    }
}

// grid = (ceil(max inter / 16), slots); slot 0 is the shared expert when there is one.
// Two CTAs per SM (128 registers): measured faster than the unbounded 218-register build
// (large decode with int4-grouped weights 175 -> 135 us, batch-32 2.50 -> 1.66 ms).
__global__ void __launch_bounds__(kThreads, 2) gateup_kernel(ExpertWork W) {
    extern __shared__ __align__(16) float xs[];
    Slot s;
    if (!resolve_slot(W, blockIdx.y, s)) return;
    if (W.idot && s.fmt == COLI_FMT_INT4) gateup_slot_idot<COLI_FMT_INT4>(W, s, xs);
    else if (W.idot && s.fmt == COLI_FMT_INT8) gateup_slot_idot<COLI_FMT_INT8>(W, s, xs);
    else if (s.fmt == COLI_FMT_INT4) gateup_slot<COLI_FMT_INT4>(W, s, xs);
    else if (s.fmt == COLI_FMT_INT4G) gateup_slot<COLI_FMT_INT4, true>(W, s, xs);
    else if (s.fmt == COLI_FMT_INT8) gateup_slot<COLI_FMT_INT8>(W, s, xs);
    else gateup_slot<COLI_FMT_INT2>(W, s, xs);
}

template <int FMT, int NV, bool GRP>
__device__ __forceinline__ void down_pass(const ExpertWork &W, const Slot &s, int d0, int v0, int nv,
                                          const float *xs, int CPR) {
    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
    const int64_t rb = row_bytes(FMT, s.inter);
    int d[4];
    const uint8_t *rows[4];
#pragma unroll
    for (int r = 0; r < 4; r++) {
        d[r] = d0 + 4 * warp + r;
        rows[r] = static_cast<const uint8_t *>(s.ex.down_w) + min(d[r], W.H - 1) * rb;
    }
    float out[4][NV];
    if constexpr (GRP) {
        const int ng = (s.inter + W.group_size - 1) / W.group_size;
        const float *srows[4];
#pragma unroll
        for (int r = 0; r < 4; r++) srows[r] = s.ex.down_s + (size_t)min(d[r], W.H - 1) * ng;
        qdot_rows_grouped<4, NV>(rows, srows, W.group_size / 32, xs, s.inter, CPR, lane, out);
    } else {
        qdot_rows<FMT, 4, NV>(rows, xs, s.inter, CPR, lane, out);
    }
#pragma unroll
    for (int v = 0; v < NV; v++) {
        if (lane != v || v >= nv) continue;
        const int yr = slot_row(W, s, v0 + v);
#pragma unroll
        for (int r = 0; r < 4; r++)
            if (d[r] < W.H) W.y[(size_t)yr * W.H + d[r]] = GRP ? out[r][v] : out[r][v] * s.ex.down_s[d[r]];
    }
}

template <int FMT, bool GRP = false>
__device__ void down_slot(const ExpertWork &W, const Slot &s, float *xs) {
    using G = QGeom<FMT>;
    const int d0 = blockIdx.x * kDnRowsPerCta;
    if (d0 >= W.H) return;
    const int CPR = s.inter / G::EPC;
    for (int v0 = 0; v0 < s.n; v0 += kNV) {
        const int nv = min(kNV, s.n - v0);
        __syncthreads();
        for (int v = 0; v < nv; v++)
            stage_vec<FMT>(W.h + (size_t)slot_row(W, s, v0 + v) * W.ldh, xs + v * s.inter, s.inter, CPR,
                           threadIdx.x, kThreads);
        if (nv == 3)
            for (int i = threadIdx.x; i < s.inter; i += kThreads) xs[3 * s.inter + i] = 0.f;
        __syncthreads();
        if (nv == 1) down_pass<FMT, 1, GRP>(W, s, d0, v0, nv, xs, CPR);
        else if (nv == 2) down_pass<FMT, 2, GRP>(W, s, d0, v0, nv, xs, CPR);
        else down_pass<FMT, 4, GRP>(W, s, d0, v0, nv, xs, CPR);
    }
}

template <int FMT, int NV>
__device__ __forceinline__ void down_pass_idot(const ExpertWork &W, const Slot &s, int d0, int v0, int nv,
                                               const uint32_t *xq, const float *sxv, int CPR) {
    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
    const int64_t rb = row_bytes(FMT, s.inter);
    int d[4];
    const uint8_t *rows[4];
#pragma unroll
    for (int r = 0; r < 4; r++) {
        d[r] = d0 + 4 * warp + r;
        rows[r] = static_cast<const uint8_t *>(s.ex.down_w) + min(d[r], W.H - 1) * rb;
    }
    int out[4][NV];
    idot_rows<FMT, 4, NV>(rows, xq, s.inter / 4, CPR, lane, out);
#pragma unroll
    for (int v = 0; v < NV; v++) {
        if (lane != v || v >= nv) continue;
        const int yr = slot_row(W, s, v0 + v);
#pragma unroll
        for (int r = 0; r < 4; r++)
            if (d[r] < W.H) W.y[(size_t)yr * W.H + d[r]] = idot_scale(out[r][v], s.ex.down_s[d[r]], sxv[v]);
    }
}

template <int FMT>
__device__ void down_slot_idot(const ExpertWork &W, const Slot &s, float *xs) {
    __shared__ float sxv[kNV];
    const int d0 = blockIdx.x * kDnRowsPerCta;
    if (d0 >= W.H) return;
    const int CPR = s.inter / QGeom<FMT>::EPC;
    uint32_t *xq = reinterpret_cast<uint32_t *>(xs);
    for (int v0 = 0; v0 < s.n; v0 += kNV) {
        const int nv = min(kNV, s.n - v0);
        __syncthreads();
        for (int v = 0; v < nv; v++)
            stage_idot<FMT>(W.h + (size_t)slot_row(W, s, v0 + v) * W.ldh, s.inter, xq + v * (s.inter / 4), &sxv[v]);
        __syncthreads();
        if (nv == 1) down_pass_idot<FMT, 1>(W, s, d0, v0, nv, xq, sxv, CPR);
        else if (nv == 2) down_pass_idot<FMT, 2>(W, s, d0, v0, nv, xq, sxv, CPR);
        else down_pass_idot<FMT, 4>(W, s, d0, v0, nv, xq, sxv, CPR);
    }
}

// grid = (ceil(H / 32), slots)
__global__ void __launch_bounds__(kThreads, 2) down_kernel(ExpertWork W) {
    extern __shared__ __align__(16) float xs[];
    Slot s;
    if (!resolve_slot(W, blockIdx.y, s)) return;
    if (W.idot && s.fmt == COLI_FMT_INT4) down_slot_idot<COLI_FMT_INT4>(W, s, xs);
    else if (W.idot && s.fmt == COLI_FMT_INT8) down_slot_idot<COLI_FMT_INT8>(W, s, xs);
    else if (s.fmt == COLI_FMT_INT4) down_slot<COLI_FMT_INT4>(W, s, xs);
    else if (s.fmt == COLI_FMT_INT4G) down_slot<COLI_FMT_INT4, true>(W, s, xs);
    else if (s.fmt == COLI_FMT_INT8) down_slot<COLI_FMT_INT8>(W, s, xs);
    else down_slot<COLI_FMT_INT2>(W, s, xs);
}

static size_t expert_smem(const ExpertWork &w, int dim) {
    const int nv = w.T < kNV ? w.T : kNV;
    return (size_t)(nv == 3 ? 4 : nv) * dim * sizeof(float);
}

cudaError_t launch_gateup(const ExpertWork &w, cudaStream_t st) {
    const size_t smem = expert_smem(w, w.H);
    cudaError_t e = cudaFuncSetAttribute(gateup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    const int imax = w.I > w.I_shared ? w.I : w.I_shared;
    dim3 grid((imax + kGuRowsPerCta - 1) / kGuRowsPerCta, w.slots);
    gateup_kernel<<<grid, kThreads, smem, st>>>(w);
    return cudaGetLastError();
}

cudaError_t launch_down(const ExpertWork &w, cudaStream_t st) {
    const int imax = w.I > w.I_shared ? w.I : w.I_shared;
    const size_t smem = expert_smem(w, imax);
    cudaError_t e = cudaFuncSetAttribute(down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((w.H + kDnRowsPerCta - 1) / kDnRowsPerCta, w.slots);
    down_kernel<<<grid, kThreads, smem, st>>>(w);
    return cudaGetLastError();
}

// out[t][d] = sum_{k < keff[t]} w[t][k] * y[pos[t*K+k]][d]  (selection order)  + y_shared[t][d]
__global__ void __launch_bounds__(256)
combine_kernel(const float *__restrict__ y, const float *__restrict__ wts,
               const int32_t *__restrict__ keff, const int32_t *__restrict__ pos, int T, int H,
               int K, int has_shared, const float *resid, float *out) {
    const int t = blockIdx.y;
    const int d = 4 * (blockIdx.x * blockDim.x + threadIdx.x);
    if (d >= H) return;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    const int ke = keff[t];
    for (int k = 0; k < ke; k++) {
        const float wk = wts[(size_t)t * K + k];
        const float4 v = *reinterpret_cast<const float4 *>(y + (size_t)pos[(size_t)t * K + k] * H + d);
        acc.x = __fadd_rn(acc.x, __fmul_rn(wk, v.x));
        acc.y = __fadd_rn(acc.y, __fmul_rn(wk, v.y));
        acc.z = __fadd_rn(acc.z, __fmul_rn(wk, v.z));
        acc.w = __fadd_rn(acc.w, __fmul_rn(wk, v.w));
    }
    if (has_shared) {
        const float4 v = *reinterpret_cast<const float4 *>(y + ((size_t)T * K + t) * H + d);
        acc.x = __fadd_rn(acc.x, v.x);
        acc.y = __fadd_rn(acc.y, v.y);
        acc.z = __fadd_rn(acc.z, v.z);
        acc.w = __fadd_rn(acc.w, v.w);
    }
    if (resid) {  // the layer tail: the residual plus the block (x += tmp)
        const float4 r = *reinterpret_cast<const float4 *>(resid + (size_t)t * H + d);
        acc = make_float4(__fadd_rn(r.x, acc.x), __fadd_rn(r.y, acc.y), __fadd_rn(r.z, acc.z), __fadd_rn(r.w, acc.w));
    }
    *reinterpret_cast<float4 *>(out + (size_t)t * H + d) = acc;
}

cudaError_t launch_combine(const float *y, const float *wts, const int32_t *keff,
                           const int32_t *pos, int T, int H, int K, int has_shared, const float *resid,
                           float *out, cudaStream_t st) {
    dim3 grid((H / 4 + 255) / 256, T);
    combine_kernel<<<grid, 256, 0, st>>>(y, wts, keff, pos, T, H, K, has_shared, resid, out);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- RMS normalisation of the rows
// xn[t] = (resid[t] * r_t) * w with r_t = 1 / sqrtf(mean square of resid[t] + eps), the mean
// square summed in double (colibri-strix c/glm.c @98759bf rmsnorm, applied with the post-attention
// norm before moe() in the layer forward). One CTA per row; the squares are summed per thread in
// a fixed stride order, then over the warps in a fixed order.
__global__ void __launch_bounds__(256) rmsnorm_rows_kernel(const float *__restrict__ resid, const float *__restrict__ w,
                                                           float eps, int H, float *__restrict__ xn) {
    __shared__ double red[8];
    const int t = blockIdx.x, tid = threadIdx.x, lane = tid % kWarp, warp = tid / kWarp;
    const float4 *r4 = reinterpret_cast<const float4 *>(resid + (size_t)t * H);
    double ms = 0.0;
    for (int q = tid; q < H / 4; q += 256) {
        const float4 v = r4[q];
        ms += (double)v.x * v.x;
        ms += (double)v.y * v.y;
        ms += (double)v.z * v.z;
        ms += (double)v.w * v.w;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ms += __shfl_xor_sync(kFull, ms, o);
    if (lane == 0) red[warp] = ms;
    __syncthreads();
    double tot = 0.0;
#pragma unroll
    for (int k = 0; k < 8; k++) tot += red[k];
    const float r = 1.f / sqrtf((float)(tot / H) + eps);
    const float4 *w4 = reinterpret_cast<const float4 *>(w);
    float4 *o4 = reinterpret_cast<float4 *>(xn + (size_t)t * H);
    for (int q = tid; q < H / 4; q += 256) {
        const float4 v = r4[q], g = w4[q];
        o4[q] = make_float4(v.x * r * g.x, v.y * r * g.y, v.z * r * g.z, v.w * r * g.w);
    }
}

cudaError_t launch_rmsnorm(const float *resid, const float *w, float eps, int T, int H, float *xn, cudaStream_t st) {
    rmsnorm_rows_kernel<<<T, 256, 0, st>>>(resid, w, eps, H, xn);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- standalone quantized GEMV
// gs > 0: COLI_FMT_INT4G (FMT is the int4 layout), sc is [O][ceil(In/gs)]
template <int FMT, int NV, bool GRP>
__device__ __forceinline__ void qgemv_pass(const uint8_t *W, const float *sc, int gs, float *y, int O, int In,
                                           int o0, int t0, int nv, const float *xs, int CPR) {
    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
    const int64_t rb = row_bytes(FMT, In);
    int o[4];
    const uint8_t *rows[4];
#pragma unroll
    for (int r = 0; r < 4; r++) {
        o[r] = o0 + 4 * warp + r;
        rows[r] = W + min(o[r], O - 1) * rb;
    }
    float out[4][NV];
    if constexpr (GRP) {
        const int ng = (In + gs - 1) / gs;
        const float *srows[4];
#pragma unroll
        for (int r = 0; r < 4; r++) srows[r] = sc + (size_t)min(o[r], O - 1) * ng;
        qdot_rows_grouped<4, NV>(rows, srows, gs / 32, xs, In, CPR, lane, out);
    } else {
        qdot_rows<FMT, 4, NV>(rows, xs, In, CPR, lane, out);
    }
#pragma unroll
    for (int v = 0; v < NV; v++) {
        if (lane != v || v >= nv) continue;
#pragma unroll
        for (int r = 0; r < 4; r++)
            if (o[r] < O) y[(size_t)(t0 + v) * O + o[r]] = GRP ? out[r][v] : out[r][v] * sc[o[r]];
    }
}

template <int FMT, bool GRP>
__global__ void __launch_bounds__(kThreads)
qgemv_kernel(const uint8_t *__restrict__ W, const float *__restrict__ sc, int gs, const float *__restrict__ x,
             float *__restrict__ y, int O, int In, int T) {
    extern __shared__ __align__(16) float xs[];
    using G = QGeom<FMT>;
    const int CPR = In / G::EPC;
    const int o0 = blockIdx.x * kDnRowsPerCta, t0 = blockIdx.y * kNV;
    const int nv = min(kNV, T - t0);
    for (int v = 0; v < nv; v++)
        stage_vec<FMT>(x + (size_t)(t0 + v) * In, xs + v * In, In, CPR, threadIdx.x, kThreads);
    if (nv == 3)
        for (int i = threadIdx.x; i < In; i += kThreads) xs[3 * In + i] = 0.f;
    __syncthreads();
    if (nv == 1) qgemv_pass<FMT, 1, GRP>(W, sc, gs, y, O, In, o0, t0, nv, xs, CPR);
    else if (nv == 2) qgemv_pass<FMT, 2, GRP>(W, sc, gs, y, O, In, o0, t0, nv, xs, CPR);
    else qgemv_pass<FMT, 4, GRP>(W, sc, gs, y, O, In, o0, t0, nv, xs, CPR);
}

cudaError_t launch_qgemv(int fmt, const void *W, const float *sc, int gs, const float *x, float *y, int O,
                         int In, int T, cudaStream_t st) {
    const int nv = T < kNV ? T : kNV;
    const size_t smem = (size_t)(nv == 3 ? 4 : nv) * In * sizeof(float);
    dim3 grid((O + kDnRowsPerCta - 1) / kDnRowsPerCta, (T + kNV - 1) / kNV);
    auto go = [&](auto kern) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        kern<<<grid, kThreads, smem, st>>>(static_cast<const uint8_t *>(W), sc, gs, x, y, O, In, T);
        return cudaGetLastError();
    };
    if (fmt == COLI_FMT_INT8) return go(qgemv_kernel<COLI_FMT_INT8, false>);
    if (fmt == COLI_FMT_INT4) return go(qgemv_kernel<COLI_FMT_INT4, false>);
    if (fmt == COLI_FMT_INT4G) return go(qgemv_kernel<COLI_FMT_INT4, true>);
    return go(qgemv_kernel<COLI_FMT_INT2, false>);
}

}  // namespace colimoe
