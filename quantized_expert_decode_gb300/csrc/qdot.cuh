// qdot.cuh — the dequant-on-use dot-product core shared by the expert kernels.
//
// Computes, for NR packed weight rows and NV activation vectors, the fp32 dot products
//   sum_i deq(W[r, i]) * v[i]
// where deq is the glm.c QT format (int8: signed byte; int4: two per byte, low nibble first,
// value = nibble - 8; int2: four per byte from bit 0, value = field - 2). The row scale is
// applied by the caller after the sum, as matmul_q / matmul_i4 / matmul_i2 do.
//
// Unpacking without integer->float conversions. A b-bit field f at bit position b*m of a
// 32-bit word is masked and OR-ed into the mantissa of 2^23 (0x4B000000): the float is then
// exactly 2^23 + f * 2^(b*m). Subtracting the constant 2^23 + off * 2^(b*m) (off = 8 for int4,
// 2 for int2; for int8 the byte's sign bit is flipped in the same LOP3 and off = 128) leaves
// exactly (value) * 2^(b*m). The activation that multiplies it was staged in shared memory
// pre-multiplied by 2^-(b*m), so every product is value * x up to the usual fp32 rounding.
// One LOP3 per element, one FADD2 per two elements, one FFMA2 per two elements per vector.
// Fields m (low half-word) and m + EPW/2 (high half-word, after one shift by 16) share the
// same scale and form the two lanes of one f32x2 operation.
//
// Staged activation layout (per vector, In floats): element i of chunk c (EPC elements per
// 16-byte weight chunk) is stored at float4 slot k of chunk c at smem float4 index k*CPR + c,
// so that the 32 lanes of a warp, which read consecutive chunks, hit consecutive float4s
// (no bank conflicts). Inside a chunk, word wi's EPW elements are ordered
// [x_0, x_h, x_1 2^-b, x_{h+1} 2^-b, ...] with h = EPW/2.
#pragma once

#include "common.cuh"

namespace colimoe {

template <int FMT>
struct Q;
template <>
struct Q<COLI_FMT_INT8> {
    static constexpr int BITS = 8, OFF = 128;
    static constexpr bool FLIP = true;
};
template <>
struct Q<COLI_FMT_INT4> {
    static constexpr int BITS = 4, OFF = 8;
    static constexpr bool FLIP = false;
};
template <>
struct Q<COLI_FMT_INT2> {
    static constexpr int BITS = 2, OFF = 2;
    static constexpr bool FLIP = false;
};

template <int FMT>
struct QGeom {
    static constexpr int BITS = Q<FMT>::BITS;
    static constexpr int EPW = 32 / BITS;   // elements per 32-bit word
    static constexpr int HALF = EPW / 2;    // f32x2 pairs per word
    static constexpr int EPC = 4 * EPW;     // elements per 16-byte chunk
    static constexpr int F4W = EPW / 4;     // staged float4s per word
    __host__ __device__ static constexpr uint32_t mask(int m) {
        return ((1u << BITS) - 1u) << (BITS * m);
    }
    __host__ __device__ static constexpr uint32_t xorv(int m) {
        return 0x4B000000u | (Q<FMT>::FLIP ? (0x80u << (BITS * m)) : 0u);
    }
    __host__ __device__ static constexpr float magic(int m) {
        return 8388608.0f + (float)Q<FMT>::OFF * (float)(1u << (BITS * m));
    }
    __host__ __device__ static constexpr float xscale(int m) {
        return 1.0f / (float)(1u << (BITS * m));
    }
};

// (a & b) ^ c in one LOP3
__device__ __forceinline__ uint32_t lop3_and_xor(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ uint4 ld_stream_16(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t word_of(const uint4 &v, int wi) {
    return wi == 0 ? v.x : wi == 1 ? v.y : wi == 2 ? v.z : v.w;
}

// Index in the staged layout of element i of a vector whose packed rows have CPR chunks.
template <int FMT>
__host__ __device__ __forceinline__ int staged_index(int i, int CPR, float &scale) {
    using G = QGeom<FMT>;
    const int c = i / G::EPC, r = i % G::EPC;
    const int wi = r / G::EPW, q = r % G::EPW;
    const int m = q % G::HALF, hi = q / G::HALF;
    const int f = wi * G::EPW + 2 * m + hi;
    scale = 1.0f / (float)(1u << (G::BITS * m));
    return ((f >> 2) * CPR + c) * 4 + (f & 3);
}

// Stage one fp32 vector of In elements (In a multiple of EPC) into shared memory.
template <int FMT>
__device__ __forceinline__ void stage_vec(const float *__restrict__ src, float *dst, int In, int CPR,
                                          int tid, int nthreads) {
    for (int i = tid; i < In; i += nthreads) {
        float sc;
        const int at = staged_index<FMT>(i, CPR, sc);
        dst[at] = src[i] * sc;
    }
}

// Dot products of NR packed rows with NV staged vectors, for the lane's share of the chunks.
// rows[r] points at the row's first byte (16-byte aligned). xs points at vector 0 in shared
// memory; vector v starts at xs + v * xstride floats. The result is reduced across the warp:
// every lane returns the full sums.
template <int FMT, int NR, int NV>
__device__ __forceinline__ void qdot_rows(const uint8_t *const (&rows)[NR], const float *xs,
                                          int xstride, int CPR, int lane, float (&out)[NR][NV]) {
    using G = QGeom<FMT>;
    float2 acc[NR][NV];
#pragma unroll
    for (int r = 0; r < NR; r++)
#pragma unroll
        for (int v = 0; v < NV; v++) acc[r][v] = make_float2(0.f, 0.f);

    const float4 *xs4 = reinterpret_cast<const float4 *>(xs);
    const int xstride4 = xstride / 4;
    uint4 cur[NR], nxt[NR];
    int c = lane;
    if (c < CPR) {
#pragma unroll
        for (int r = 0; r < NR; r++) cur[r] = ld_stream_16(rows[r] + 16 * c);
    }
    for (; c < CPR; c += kWarp) {
        const int cn = c + kWarp;
        if (cn < CPR) {
#pragma unroll
            for (int r = 0; r < NR; r++) nxt[r] = ld_stream_16(rows[r] + 16 * cn);
        }
#pragma unroll
        for (int wi = 0; wi < 4; wi++) {
            float4 xv[NV][G::F4W];
#pragma unroll
            for (int v = 0; v < NV; v++)
#pragma unroll
                for (int j = 0; j < G::F4W; j++)
                    xv[v][j] = xs4[v * xstride4 + (wi * G::F4W + j) * CPR + c];
#pragma unroll
            for (int r = 0; r < NR; r++) {
                const uint32_t q = word_of(cur[r], wi);
                const uint32_t qh = q >> 16;
#pragma unroll
                for (int m = 0; m < G::HALF; m++) {
                    const uint32_t lo = lop3_and_xor(q, G::mask(m), G::xorv(m));
                    const uint32_t hi = lop3_and_xor(qh, G::mask(m), G::xorv(m));
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
        if (cn < CPR) {
#pragma unroll
            for (int r = 0; r < NR; r++) cur[r] = nxt[r];
        }
    }
#pragma unroll
    for (int r = 0; r < NR; r++)
#pragma unroll
        for (int v = 0; v < NV; v++) {
            float s = acc[r][v].x + acc[r][v].y;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(kFull, s, o);
            out[r][v] = s;
        }
}

// The int4-grouped form (COLI_FMT_INT4G: int4 bytes, one scale per group of gs inputs): each
// 16-byte chunk (32 inputs) lies in one group when gs is a multiple of 32, so a lane forms the
// chunk's partial sums, multiplies them by the group scale srows[r][c / cpg] (cpg = gs / 32
// chunks per group) and adds them to its accumulators. The staged layout is the int4 one.
template <int NR, int NV>
__device__ __forceinline__ void qdot_rows_grouped(const uint8_t *const (&rows)[NR], const float *const (&srows)[NR],
                                                  int cpg, const float *xs, int xstride, int CPR, int lane,
                                                  float (&out)[NR][NV]) {
    using G = QGeom<COLI_FMT_INT4>;
    float2 acc[NR][NV];
#pragma unroll
    for (int r = 0; r < NR; r++)
#pragma unroll
        for (int v = 0; v < NV; v++) acc[r][v] = make_float2(0.f, 0.f);
    const float4 *xs4 = reinterpret_cast<const float4 *>(xs);
    const int xstride4 = xstride / 4;
    for (int c = lane; c < CPR; c += kWarp) {
        uint4 cur[NR];
        float sg[NR];
#pragma unroll
        for (int r = 0; r < NR; r++) {
            cur[r] = ld_stream_16(rows[r] + 16 * c);
            sg[r] = __ldg(srows[r] + c / cpg);
        }
        float2 part[NR][NV];
#pragma unroll
        for (int r = 0; r < NR; r++)
#pragma unroll
            for (int v = 0; v < NV; v++) part[r][v] = make_float2(0.f, 0.f);
#pragma unroll
        for (int wi = 0; wi < 4; wi++) {
            float4 xv[NV][G::F4W];
#pragma unroll
            for (int v = 0; v < NV; v++)
#pragma unroll
                for (int j = 0; j < G::F4W; j++) xv[v][j] = xs4[v * xstride4 + (wi * G::F4W + j) * CPR + c];
#pragma unroll
            for (int r = 0; r < NR; r++) {
                const uint32_t q = word_of(cur[r], wi);
                const uint32_t qh = q >> 16;
#pragma unroll
                for (int m = 0; m < G::HALF; m++) {
                    const uint32_t lo = lop3_and_xor(q, G::mask(m), G::xorv(m));
                    const uint32_t hi = lop3_and_xor(qh, G::mask(m), G::xorv(m));
                    const float2 d = __fadd2_rn(make_float2(__uint_as_float(lo), __uint_as_float(hi)),
                                                make_float2(-G::magic(m), -G::magic(m)));
#pragma unroll
                    for (int v = 0; v < NV; v++) {
                        const float4 &x4 = xv[v][m >> 1];
                        const float2 x2 = (m & 1) ? make_float2(x4.z, x4.w) : make_float2(x4.x, x4.y);
                        part[r][v] = __ffma2_rn(d, x2, part[r][v]);
                    }
                }
            }
        }
#pragma unroll
        for (int r = 0; r < NR; r++)
#pragma unroll
            for (int v = 0; v < NV; v++) acc[r][v] = __ffma2_rn(part[r][v], make_float2(sg[r], sg[r]), acc[r][v]);
    }
#pragma unroll
    for (int r = 0; r < NR; r++)
#pragma unroll
        for (int v = 0; v < NV; v++) {
            float s = acc[r][v].x + acc[r][v].y;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(kFull, s, o);
            out[r][v] = s;
        }
}

}  // namespace colimoe
