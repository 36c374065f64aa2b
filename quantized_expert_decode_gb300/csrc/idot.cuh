// idot.cuh — the integer dot-product core for single-token groups.
//
// Computes, for NR packed weight rows and ONE activation vector x, the exact integer sums
//   S_r = sum_i v[r, i] * X[i]
// where v is the dequantised integer of the glm.c QT format (int8: the signed byte; int4:
// nibble - 8; int2: field - 2) and X is x in 24-bit block fixed point:
//   X[i] = round(x[i] * 2^s),  s chosen per vector so that max|x| * 2^s < 2^22.
// The dot product is then S_r * 2^-s, formed exactly in int64 before its one conversion to
// float; the caller applies the row scale, as matmul_q / matmul_i4 / matmul_i2 do.
//
// Why integers: the float route spends one LOP3 per weight plus an f32x2 subtract and FMA per
// two, and LOP3 issues at half rate, so on GB300 it cannot unpack int4 as fast as HBM delivers
// it. DP4A multiplies four signed weight bytes by four activation bytes and accumulates into an
// int32 in one (half-rate) instruction: with X split into three byte limbs
//   X = X2 * 2^16 + X1 * 2^8 + X0   (X0, X1 unsigned, X2 signed)
// a 32-bit word of int4 costs one shift, two LOP3 and six DP4A.
//
// Signed fields in place: a field f of b bits moved to the top of its byte and XOR-ed with
// 0x80 reads, as a signed byte, 2^(8-b) * (f - 2^(b-1)) — the dequantised value times a power of
// two. For int4, (w & 0xF0F0F0F0) ^ 0x80808080 gives the odd nibbles as 16 * (f - 8) and the
// same after w << 4 gives the even ones; int2 shifts each of its four fields to the top; int8
// bytes are used as they are. Every product carries the same factor SC (16, 64 or 1), which
// the final sum drops with an exact arithmetic shift.
//
// Staged activation layout (per vector, bytes): for the 16-byte weight chunk c of a row (EPC
// elements), the activation limbs are grouped by the word of the chunk they meet; NSS sub-steps
// of WPSS words each use three uint4 of limbs, stored at uint4 index (ss*3 + j)*CPR + c so
// that the 32 lanes of a warp, which take consecutive chunks, read consecutive uint4s. Inside
// a sub-step, u32 number u = (wl*NGW + g)*3 + l holds limb l of the four elements of field
// group g of word wl (byte b of the u32 = the element in byte b of the weight word).
#pragma once

#include "qdot.cuh"

namespace colimoe {

template <int FMT>
struct IQ;
template <>
struct IQ<COLI_FMT_INT8> {
    static constexpr int NSS = 1, WPSS = 4, NGW = 1, LOG_SC = 0;
};
template <>
struct IQ<COLI_FMT_INT4> {
    static constexpr int NSS = 2, WPSS = 2, NGW = 2, LOG_SC = 4;
};
template <>
struct IQ<COLI_FMT_INT2> {
    static constexpr int NSS = 4, WPSS = 1, NGW = 4, LOG_SC = 6;
};

// d = c + dot(signed bytes of a, bytes of b); SB: the bytes of b are signed
template <bool SB>
__device__ __forceinline__ int dp4a_s(uint32_t a, uint32_t b, int c) {
    int d;
    if (SB) asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    else asm("dp4a.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// field group g of weight word w as signed bytes SC * value
template <int FMT>
__device__ __forceinline__ uint32_t signed_fields(uint32_t w, int g) {
    if (FMT == COLI_FMT_INT4) return lop3_and_xor(g == 0 ? (w << 4) : w, 0xF0F0F0F0u, 0x80808080u);
    if (FMT == COLI_FMT_INT2) return lop3_and_xor(w << (6 - 2 * g), 0xC0C0C0C0u, 0x80808080u);
    return w;
}

// accumulate one 16-byte chunk of NR rows (w[r]) against the staged limbs: acc[r][limb]
template <int FMT, int NR>
__device__ __forceinline__ void idot_chunk(const uint4 (&w)[NR], const uint4 *xq4, int CPR, int c,
                                           int (&acc)[NR][3]) {
    using I = IQ<FMT>;
#pragma unroll
    for (int ss = 0; ss < I::NSS; ss++) {
        const uint4 xa = xq4[(ss * 3 + 0) * CPR + c];
        const uint4 xb = xq4[(ss * 3 + 1) * CPR + c];
        const uint4 xc = xq4[(ss * 3 + 2) * CPR + c];
        const uint32_t xv[12] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w, xc.x, xc.y, xc.z, xc.w};
#pragma unroll
        for (int r = 0; r < NR; r++) {
#pragma unroll
            for (int wl = 0; wl < I::WPSS; wl++) {
                const uint32_t wd = word_of(w[r], ss * I::WPSS + wl);
#pragma unroll
                for (int g = 0; g < I::NGW; g++) {
                    const uint32_t a = signed_fields<FMT>(wd, g);
                    const int u = (wl * I::NGW + g) * 3;
                    acc[r][0] = dp4a_s<false>(a, xv[u + 0], acc[r][0]);
                    acc[r][1] = dp4a_s<false>(a, xv[u + 1], acc[r][1]);
                    acc[r][2] = dp4a_s<true>(a, xv[u + 2], acc[r][2]);
                }
            }
        }
    }
}

// Four rows at once, transposing as it reduces: rows {0,1} and {2,3} are split between the lane
// halves, then between the quarters, so 12 shuffles (instead of 40) leave every lane with the
// exact total of row lane / 8.
template <int FMT>
__device__ __forceinline__ long long idot_reduce4(const int (&acc)[4][3], int lane) {
    constexpr int LS = IQ<FMT>::LOG_SC;
    long long p[4];
#pragma unroll
    for (int r = 0; r < 4; r++)
        p[r] = ((long long)(acc[r][2] >> LS) << 16) + ((long long)(acc[r][1] >> LS) << 8) +
               (long long)(acc[r][0] >> LS);
    const bool h16 = (lane & 16) != 0, h8 = (lane & 8) != 0;
    long long k0 = h16 ? p[2] : p[0], k1 = h16 ? p[3] : p[1];
    const long long s0 = h16 ? p[0] : p[2], s1 = h16 ? p[1] : p[3];
    k0 += __shfl_xor_sync(kFull, s0, 16);
    k1 += __shfl_xor_sync(kFull, s1, 16);
    long long k = h8 ? k1 : k0;
    k += __shfl_xor_sync(kFull, h8 ? k0 : k1, 8);
    k += __shfl_xor_sync(kFull, k, 4);
    k += __shfl_xor_sync(kFull, k, 2);
    k += __shfl_xor_sync(kFull, k, 1);
    return k;
}

// Two rows: the lane halves split the rows, then a butterfly over the half; every lane ends
// with the exact total of row lane / 16.
template <int FMT>
__device__ __forceinline__ long long idot_reduce2(const int (&acc)[2][3], int lane) {
    constexpr int LS = IQ<FMT>::LOG_SC;
    long long p[2];
#pragma unroll
    for (int r = 0; r < 2; r++)
        p[r] = ((long long)(acc[r][2] >> LS) << 16) + ((long long)(acc[r][1] >> LS) << 8) +
               (long long)(acc[r][0] >> LS);
    const bool h16 = (lane & 16) != 0;
    long long k = h16 ? p[1] : p[0];
    k += __shfl_xor_sync(kFull, h16 ? p[0] : p[1], 16);
    k += __shfl_xor_sync(kFull, k, 8);
    k += __shfl_xor_sync(kFull, k, 4);
    k += __shfl_xor_sync(kFull, k, 2);
    k += __shfl_xor_sync(kFull, k, 1);
    return k;
}

// the shift s of a vector whose largest magnitude is mx (0 for an all-zero vector)
__device__ __forceinline__ int fixed_shift(float mx) {
    if (!(mx > 0.f)) return 0;
    const int ex = (int)((__float_as_uint(mx) >> 23) & 255u);
    return 21 - (ex == 0 ? -126 : ex - 127);
}

// X = round(x * 2^s), with 2^s applied as two exact factors (s reaches 147 for subnormal input)
struct FixedScale {
    float f1, f2;
    __device__ __forceinline__ explicit FixedScale(int s) {
        const int s1 = max(-126, min(126, s)), s2 = s - s1;
        f1 = __int_as_float((s1 + 127) << 23);
        f2 = __int_as_float((s2 + 127) << 23);
    }
    __device__ __forceinline__ int operator()(float x) const { return __float2int_rn((x * f1) * f2); }
};

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// limbs of four values: w0 = their bytes 0, w1 = bytes 1, w2 = bytes 2 (X2 for |X| < 2^22)
__device__ __forceinline__ void pack_limbs(int a, int b, int c, int d, uint32_t &w0, uint32_t &w1, uint32_t &w2) {
    const uint32_t ab = prmt(a, b, 0x5140u), cd = prmt(c, d, 0x5140u);  // a0 b0 a1 b1 / c0 d0 c1 d1
    w0 = prmt(ab, cd, 0x5410u);
    w1 = prmt(ab, cd, 0x7632u);
    w2 = prmt(prmt(a, b, 0x0062u), prmt(c, d, 0x0062u), 0x5410u);
}

// Stage item p of a vector (n a multiple of EPC, CPR = n / EPC): p = ss * CPR + c takes the 16
// elements of sub-step ss of chunk c, packs their limbs and writes the three uint4 of the
// layout, so consecutive items write consecutive uint4s.
template <int FMT>
__device__ __forceinline__ void stage_limb_item(const float *__restrict__ src, int CPR, bool coherent, uint4 *xq4,
                                                const FixedScale &fx, int p) {
    using G = QGeom<FMT>;
    using I = IQ<FMT>;
    const int c = p % CPR, ss = p / CPR;
    const float4 *s4 = reinterpret_cast<const float4 *>(src + c * G::EPC + ss * 16);
    float4 v[4];
#pragma unroll
    for (int k = 0; k < 4; k++) v[k] = coherent ? __ldcg(s4 + k) : __ldg(s4 + k);
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
#pragma unroll
    for (int j = 0; j < 3; j++)
        xq4[(ss * 3 + j) * CPR + c] = make_uint4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
}

// ---------------------------------------------------------------- IDOT activations (int8)
// glm.c's IDOT kernels quantise an activation row to int8 with one scale (qrow_i8):
// s = max(max|x| / 127, 1e-12), q = round-half-even(x * (1 / s)), every division and product
// rounded as IEEE fp32; the dot with the dequantised weights is an exact integer sum, and
// y[o] = ((float)dot * scale[o]) * s. For the single-token walk the bytes sit in the layout of
// the limbs with one limb: item p = ss * CPR + c (the 16 elements of sub-step ss of chunk c) is
// one uint4 at p, u32 number u = wl * NGW + g holding the four elements that meet field group g
// of word wl (byte b: element wl * EPW + g + b * NGW of the item).
struct Q8Scale {
    float s, inv;
    __device__ __forceinline__ explicit Q8Scale(float amax) {
        s = __fdiv_rn(amax, 127.f);
        if (s < 1e-12f) s = 1e-12f;
        inv = __fdiv_rn(1.f, s);
    }
    __device__ __forceinline__ int operator()(float x) const { return __float2int_rn(__fmul_rn(x, inv)); }
};

// item p of a vector as int8 bytes (v: its 16 elements)
template <int FMT>
__device__ __forceinline__ void q8_from_regs(const float4 (&v)[4], uint8_t *xq, int CPR, int p, const Q8Scale &qs) {
    using G = QGeom<FMT>;
    using I = IQ<FMT>;
    int X[16];
#pragma unroll
    for (int k = 0; k < 4; k++) {
        X[4 * k + 0] = qs(v[k].x);
        X[4 * k + 1] = qs(v[k].y);
        X[4 * k + 2] = qs(v[k].z);
        X[4 * k + 3] = qs(v[k].w);
    }
    static_assert(I::WPSS * I::NGW == 4, "one uint4 of int8 bytes per item");
    uint32_t o[4];
#pragma unroll
    for (int wl = 0; wl < I::WPSS; wl++)
#pragma unroll
        for (int g = 0; g < I::NGW; g++) {
            const int e0 = wl * G::EPW + g;
            const uint32_t ab = prmt(X[e0], X[e0 + I::NGW], 0x0040u), cd = prmt(X[e0 + 2 * I::NGW], X[e0 + 3 * I::NGW], 0x0040u);
            o[wl * I::NGW + g] = prmt(ab, cd, 0x5410u);
        }
    reinterpret_cast<uint4 *>(xq)[p] = make_uint4(o[0], o[1], o[2], o[3]);
}

// one 16-byte chunk of NR rows against the int8 bytes: acc[r] += sum of SC * deq * q
template <int FMT, int NR>
__device__ __forceinline__ void q8_chunk(const uint4 (&w)[NR], const uint4 *xq4, int CPR, int c, int (&acc)[NR]) {
    using I = IQ<FMT>;
#pragma unroll
    for (int ss = 0; ss < I::NSS; ss++) {
        const uint4 xa = xq4[ss * CPR + c];
        const uint32_t xv[4] = {xa.x, xa.y, xa.z, xa.w};
#pragma unroll
        for (int r = 0; r < NR; r++)
#pragma unroll
            for (int wl = 0; wl < I::WPSS; wl++) {
                const uint32_t wd = word_of(w[r], ss * I::WPSS + wl);
#pragma unroll
                for (int g = 0; g < I::NGW; g++)
                    acc[r] = dp4a_s<true>(signed_fields<FMT>(wd, g), xv[wl * I::NGW + g], acc[r]);
            }
    }
}

// four rows of lane partials at once (the transposing pattern of idot_reduce4): every lane ends
// with the exact dot of row lane / 8, the factor SC dropped
template <int FMT>
__device__ __forceinline__ int q8_reduce4(const int (&p)[4], int lane) {
    const bool h16 = (lane & 16) != 0, h8 = (lane & 8) != 0;
    int k0 = h16 ? p[2] : p[0], k1 = h16 ? p[3] : p[1];
    const int s0 = h16 ? p[0] : p[2], s1 = h16 ? p[1] : p[3];
    k0 += __shfl_xor_sync(kFull, s0, 16);
    k1 += __shfl_xor_sync(kFull, s1, 16);
    int k = h8 ? k1 : k0;
    k += __shfl_xor_sync(kFull, h8 ? k0 : k1, 8);
    k += __shfl_xor_sync(kFull, k, 4);
    k += __shfl_xor_sync(kFull, k, 2);
    k += __shfl_xor_sync(kFull, k, 1);
    return k >> IQ<FMT>::LOG_SC;
}

// items per vector of n elements
template <int FMT>
__host__ __device__ __forceinline__ int limb_items(int n) {
    return n / QGeom<FMT>::EPC * IQ<FMT>::NSS;
}

// the whole vector, items p0, p0 + dp, ...
template <int FMT>
__device__ __forceinline__ void stage_limbs_vec(const float *__restrict__ src, int n, bool coherent, uint8_t *xq,
                                                const FixedScale &fx, int p0, int dp) {
    const int CPR = n / QGeom<FMT>::EPC, items = limb_items<FMT>(n);
    for (int p = p0; p < items; p += dp) stage_limb_item<FMT>(src, CPR, coherent, reinterpret_cast<uint4 *>(xq), fx, p);
}

}  // namespace colimoe
