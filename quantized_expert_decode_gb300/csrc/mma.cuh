// mma.cuh — the tensor-core dot-product core for multi-token groups of the decode kernel.
//
// For a group of up to four activation vectors x_t (tokens) and a block of 16 packed weight
// rows, it computes the fp32 sums
//   S[r][t] = sum_i deq(W[r, i]) * x_t[i]
// (deq as in the glm.c QT formats: int8 signed byte, int4 nibble - 8, int2 field - 2; the row
// scale is applied by the caller after the sum, as matmul_q / matmul_i4 / matmul_i2 do) with
// warp-level mma.sync m16n8k16 (f16 x f16 -> f32).
//
// Why: a group of n tokens shares every dequantised weight, and on the CUDA cores each weight
// still costs one FMA per token on top of its unpack. Here the unpack is the only per-weight
// CUDA-core work (per 32-bit word of int4: one shift, four LOP3 and four f16x2 FMA, all
// exact), and the products and sums over the group run on the tensor cores.
//
// Exactness. A dequantised weight is a small integer, exact in f16. Each vector is staged as
// two f16 parts of x * 2^e (e per vector, so that max|x| * 2^e lies in [2^14, 2^15)):
//   hi = f16(x * 2^e),  lo = f16(x * 2^e - hi)
// which together carry 22 significant bits of x. The eight columns of the MMA are the four
// tokens' hi parts (columns 0..3) and their lo parts (columns 4..7); products are exact and
// accumulate in fp32, and S = (D[:, t] + D[:, 4 + t]) * 2^-e.
//
// Weight f16 pairs come straight out of the packed word: OR-ing a field into the mantissa of
// 1024.0 (f16 0x6400) gives 1024 + f * 2^p exactly; one f16x2 FMA with (2^-p, -(1024 * 2^-p +
// offset)) leaves the dequantised value. For int4, word bits [0,4) and [16,20) (elements 0 and
// 4) form one pair; pair q of a word holds elements (q, q + EPW/2).
//
// K order. Lane (g, c) of the warp (g = lane / 4, c = lane % 4) holds, in each MMA step, the
// k-slots {2c, 2c+1} and {2c+8, 2c+9} of rows g and g+8 (A) and of column g (B). It loads the
// 16-byte chunk 4*sigma + c of its two rows in segment sigma (64 bytes of each row), and its
// pairs 2r and 2r+1 of a word feed step r of that word. The activation element that meets a
// weight element is staged at the same place, so each lane's B operand for two steps is one
// 16-byte shared-memory load. Staged layout, per token (stride ≡ 64 mod 128 bytes so that the
// eight lanes of a quarter-warp hit distinct banks): uint4 index ((sigma * NSPC + sp) * 2 +
// part) * 4 + c, part 0 = hi, 1 = lo, sp = step pair, holding {B(step 2sp), B(step 2sp+1)}.
#pragma once

#include <cuda_fp16.h>

#include "idot.cuh"

namespace colimoe {

template <int FMT>
struct MQ {
    static constexpr int EPW = QGeom<FMT>::EPW;  // elements per 32-bit word
    static constexpr int EPC = 4 * EPW;          // elements per 16-byte chunk
    static constexpr int NP = EPW / 2;           // f16 pairs per word
    static constexpr int SPW = NP / 2;           // MMA steps per word
    static constexpr int NSPC = 2 * SPW;         // step pairs per chunk (4 words)
    static constexpr int SEGB = NSPC * 128;      // staged bytes per segment per token
};

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ uint32_t hfma2_bits(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// The NP dequantised f16 pairs of one packed word (pair q = elements q and q + EPW/2).
template <int FMT>
__device__ __forceinline__ void deq_pairs(uint32_t w, uint32_t (&p)[MQ<FMT>::NP]) {
    if constexpr (FMT == COLI_FMT_INT4) {
        const uint32_t w8 = w >> 8;
        p[0] = hfma2_bits(lop3_and_or(w, 0x000F000Fu, 0x64006400u), 0x3C003C00u, 0xE408E408u);   // x1, -1032
        p[1] = hfma2_bits(lop3_and_or(w, 0x00F000F0u, 0x64006400u), 0x2C002C00u, 0xD480D480u);   // x1/16, -72
        p[2] = hfma2_bits(lop3_and_or(w8, 0x000F000Fu, 0x64006400u), 0x3C003C00u, 0xE408E408u);
        p[3] = hfma2_bits(lop3_and_or(w8, 0x00F000F0u, 0x64006400u), 0x2C002C00u, 0xD480D480u);
    } else if constexpr (FMT == COLI_FMT_INT8) {
        const uint32_t u = w ^ 0x80808080u;  // signed byte b -> b + 128
        p[0] = hfma2_bits(prmt(u, 0x64646464u, 0x4240u), 0x3C003C00u, 0xE480E480u);  // bytes 0, 2; -1152
        p[1] = hfma2_bits(prmt(u, 0x64646464u, 0x4341u), 0x3C003C00u, 0xE480E480u);  // bytes 1, 3
    } else {
        const uint32_t w8 = w >> 8;
        constexpr uint32_t mul[4] = {0x3C003C00u, 0x34003400u, 0x2C002C00u, 0x24002400u};  // 1, 1/4, 1/16, 1/64
        constexpr uint32_t add[4] = {0xE402E402u, 0xDC08DC08u, 0xD420D420u, 0xCC80CC80u};  // -1026, -258, -66, -18
#pragma unroll
        for (int q = 0; q < 4; q++) {
            p[q] = hfma2_bits(lop3_and_or(w, 0x00030003u << (2 * q), 0x64006400u), mul[q], add[q]);
            p[4 + q] = hfma2_bits(lop3_and_or(w8, 0x00030003u << (2 * q), 0x64006400u), mul[q], add[q]);
        }
    }
}

// D (16x8 f32) += A (16x16 f16) * B (16x8 f16)
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// One 64-byte segment of the lane's two rows (wv[0]: row g, wv[1]: row g + 8) against the staged
// activations of the segment (xseg: this lane's part and chunk column).
template <int FMT>
__device__ __forceinline__ void seg_mma(const uint4 (&wv)[2], const uint8_t *xseg, float (&d)[4]) {
    using M = MQ<FMT>;
    uint32_t p0[M::NP], p1[M::NP];
#pragma unroll
    for (int sp = 0; sp < M::NSPC; sp++) {
        const uint4 u = *reinterpret_cast<const uint4 *>(xseg + sp * 128);
#pragma unroll
        for (int t = 0; t < 2; t++) {
            const int s = 2 * sp + t, w = s / M::SPW, r = s % M::SPW;
            if (r == 0) {
                deq_pairs<FMT>(word_of(wv[0], w), p0);
                deq_pairs<FMT>(word_of(wv[1], w), p1);
            }
            mma_16816(d, p0[2 * r], p1[2 * r], p0[2 * r + 1], p1[2 * r + 1], t ? u.z : u.x, t ? u.w : u.y);
        }
    }
}

// Stage item `it` of one token: the two 16-byte B words (hi and lo) of step pair sp of chunk
// column c in segment sigma. Elements past the vector's end (a ragged last segment) stage 0.
template <int FMT>
__device__ __forceinline__ void stage_mma_item(const float *__restrict__ src, int len, bool coherent, uint8_t *tok,
                                               float f1, float f2, int it) {
    using M = MQ<FMT>;
    const int c = it & 3, rest = it >> 2;
    const int sp = rest % M::NSPC, sigma = rest / M::NSPC;
    const int ch = 4 * sigma + c;
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int t = 0; t < 2; t++) {
        const int s = 2 * sp + t, w = s / M::SPW, r = s % M::SPW;
#pragma unroll
        for (int qq = 0; qq < 2; qq++) {
            const int q = 2 * r + qq;
            uint32_t hb[2], lb[2];
#pragma unroll
            for (int j = 0; j < 2; j++) {
                const int el = ch * M::EPC + w * M::EPW + q + (M::EPW / 2) * j;
                float x = 0.f;
                if (el < len) x = coherent ? __ldcg(src + el) : __ldg(src + el);
                const float xs = (x * f1) * f2;
                const __half h = __float2half_rn(xs);
                const __half l = __float2half_rn(xs - __half2float(h));
                hb[j] = __half_as_ushort(h);
                lb[j] = __half_as_ushort(l);
            }
            hw[2 * t + qq] = hb[0] | (hb[1] << 16);
            lw[2 * t + qq] = lb[0] | (lb[1] << 16);
        }
    }
    uint4 *row = reinterpret_cast<uint4 *>(tok + (size_t)(sigma * M::NSPC + sp) * 128);
    row[c] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    row[4 + c] = make_uint4(lw[0], lw[1], lw[2], lw[3]);
}

// staged items per token of a vector of len elements (segments of 4 chunks)
template <int FMT>
__host__ __device__ __forceinline__ int mma_items(int len) {
    const int cpr = (len + MQ<FMT>::EPC - 1) / MQ<FMT>::EPC;
    return (cpr + 3) / 4 * MQ<FMT>::NSPC * 4;
}

}  // namespace colimoe
