// prefill.cu — the expert GEMMs of large batches (T > 64) on the 5th-generation tensor cores.
//
// With tens of tokens per expert the gate/up and down products are real dense contractions
// (colibri-strix c/glm.c @98759bf moe() phases C/D, batched over the tokens of one expert), so
// they run as grouped bf16 GEMMs with fp32 accumulation in tensor memory:
//   gate/up: for each expert slot, A = its gate and up rows (dequantised to bf16 on the fly,
//            interleaved so that row 2r is gate row j0+r and row 2r+1 is up row j0+r),
//            B = the slot's tokens' activations in bf16; epilogue h = silu(g*s_g) * (u*s_u)
//   down:    A = the slot's down rows, B = its h rows in bf16; epilogue y = acc * s_d
// Swap-AB: weight rows are the MMA's M = 128 (the long dimension), tokens its N (16..128).
//
// One persistent CTA per SM walks the tiles (slot, token block, row block) of a launch, its
// warps specialised:
//   warp 0     weight copies: for each 128-byte K-chunk of the tile's 128 weight rows (four
//              K-steps of int4, two of int8, eight of int2), 2-D tensor copies (64 gate rows and
//              64 up rows, or 128 down rows; 128-byte swizzle) into a raw stage, completed on
//              that stage's `rfull` mbarrier. Every expert matrix has its own tensor map, written
//              on the device by a prologue launch from a host-encoded template (only the base
//              address differs: the expert table holds device pointers the host cannot read)
//   warp 1     activation copies: for each K-step, 2-D tensor copies (cp.async.bulk.tensor, a
//              tensor map over the workspace's activation rows, 128-byte swizzle) of the tile's
//              token rows straight into the B stage, in the K-major layout the MMA reads
//   warps 2-9  dequant warps: thread (r, half) turns its half of raw row r's K-step into 16
//              columns of 16-bit pairs and stores them to the A tile in tensor memory (row r =
//              TMEM lane r, tcgen05.st), then arrives on the A tile's `full`
//   warp 10    one thread issues four tcgen05.mma (K = 16 each, A from tensor memory, B from
//              shared memory) per K-step into one of two TMEM accumulators and commits the A
//              tile's and the B stage's `empty` mbarriers to their completion; after a tile's
//              last step it commits that accumulator's `accf`
//   warps 11-14 epilogue: tcgen05.ld of the 128 x N tile (warp w reads TMEM lanes 32 (w % 4)..),
//              the fused epilogue, then `tfree` hands the accumulator back to the MMA warp, so
//              the next tile's MMAs run while the epilogue reads this one
// The copies are issued by single threads and land without any instruction of the dequant
// warps; the dequant warps only dequantise. A lives in tensor memory, so the 16-bit A tile never
// passes through shared memory (at N ~ 64 tokens per expert the operand traffic of shared memory
// is what limits the MMA rate).
// K order: the dot product does not depend on the order of K, so within each block of 8 (int4)
// or 16 (int2) elements K is permuted the same way in A and B — the order in which the
// magic-number unpack produces bf16 pairs — and no byte shuffles are needed. The activations
// (x, and h written by the gate/up epilogue) are stored in that order.
// Every mbarrier wait is bounded; on expiry the CTA flags the error, drains the copies and the
// MMAs it issued (waits no other warp's abort cuts short), frees its tensor memory and returns.
#include <algorithm>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "tc.cuh"

namespace colimoe {

namespace {

constexpr int kTcM = 128;        // MMA M: weight rows per tile
constexpr int kTcN = 128;        // max tokens per tile (MMA N, multiple of 16)
constexpr int kTcKB = 64;        // K per step (one 128-byte swizzle row of 16-bit values)
constexpr int kTcA = 4;          // A tiles in tensor memory (32 columns each, after the accumulators)
constexpr int kTcBS = 6;         // B stages, one K-step of up to 128 token rows each
constexpr int kTcRS = 4;         // raw weight stages, one 128-byte K-chunk of the 128 rows each
constexpr int kChunkB = 128;     // packed bytes of a row per raw stage (128-byte swizzled rows)
constexpr int kBoxRows = 32;     // token rows per tensor copy of a B stage
constexpr int kTcThreads = 480;  // warps: 0 weights, 1 activations, 2-9 dequant, 10 MMA, 11-14 epilogue
constexpr int kTcDeq = 256, kTcEpi = 128;
constexpr int kWarpB = 1, kDeq0 = 2, kTcMmaWarp = 10;
constexpr int kTileCap = 128;    // tiles per CTA whose parameters are kept in shared memory
constexpr unsigned long long kTcWaitNs = 2000000000ull;

struct PfParams {
    const coli_moe_expert *experts;  // device [E]
    coli_moe_expert shared;
    const int32_t *counts, *offsets; // routed buckets
    const uint16_t *xb;              // f16 activations [T*K + T][H], row p scaled by 2^xe[p] (block-permuted per format)
    const int32_t *xe;               // [T*K + T] the exponent of each activation row's scale
    uint16_t *hb;                    // bf16 h [T*K + T][ldh] (block-permuted per format)
    const CUtensorMap *tmaps;        // [E + 1][3]: gate, up, down of every expert, the shared one last
    float *y;                        // [T*K + T][H]
    int32_t *err;
    int T, H, I, E, K, Is, rfmt, sfmt, ldh;
    int down;                        // 0: gate/up GEMM, 1: down GEMM
};

struct Tile {
    const uint8_t *w0, *w1;  // gate/up rows (or down rows in w0)
    const float *s0, *s1;
    int fmt, inter, n0, ncur, N, pbase, row0;  // row0: first j (gate/up) or d (down)
    int slot, sh;                              // expert slot (E: the shared expert)
};

struct TcSmem {  // after the 1024-aligned stage buffers
    uint64_t rfull[kTcRS], rempty[kTcRS], bfull[kTcBS], bempty[kTcBS], full[kTcA], emptya[kTcA], accf[2], tfree[2],
        drain;
    uint32_t tmem_base;
    int abort;
    int pref[kMaxE + 2];  // tiles before slot g (slots 0..E-1 routed, E shared)
    Tile tiles[kTileCap]; // this CTA's tiles blockIdx.x + i * gridDim.x, looked up once
};

constexpr size_t kStageB = (size_t)kTcN * 128, kStageRaw = (size_t)kTcM * kChunkB;
constexpr size_t tc_smem_bytes() { return 1024 + kTcBS * kStageB + kTcRS * kStageRaw + sizeof(TcSmem); }
constexpr uint32_t kTmemCols = 512;  // two accumulators of kTcN columns, then the A tiles
constexpr uint32_t kTmemA = 2 * kTcN;
static_assert(kTmemA + 32 * kTcA <= kTmemCols, "tensor memory holds the accumulators and the A tiles");

// position of element j of a K block in the permuted order of format fmt
__host__ __device__ __forceinline__ int kperm(int fmt, int j) {
    if (fmt == COLI_FMT_INT4) return (j & ~7) | ((j & 3) << 1) | ((j >> 2) & 1);
    if (fmt == COLI_FMT_INT2) return (j & ~15) | ((j & 7) << 1) | ((j >> 3) & 1);
    return j;
}

__device__ __forceinline__ uint32_t bf16x2_fma(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));  // (a & b) | c
    return d;
}

// bf16 pair (lo, hi) of two floats, round to nearest even
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

__device__ __forceinline__ uint32_t f16x2_fma(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// f16 pair (lo, hi) of two floats, round to nearest even
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// Dequantise 16 consecutive weights to 8 pairs of 16-bit floats (F16: IEEE half, else bf16) in
// the permuted K order. The magic: a field f in the low bits of a halfword OR-ed with the bits of
// 2^m (f16: 1024, 0x6400; bf16: 128, 0x4300) is the float 2^m + f exactly (f < 2^m fits the
// mantissa); one fused multiply-add by 1 and -(2^m + 8) (int2: -(2^m + 2)) leaves f - 8
// (f - 2) exactly. int8 bytes go through float (every int8 value is exact in both types).
template <int FMT, bool F16>
__device__ __forceinline__ void deq16(const uint32_t *w, uint32_t (&out)[8]) {
    // 16 consecutive weights (int4: 2 words, int2: 1, int8: 4) -> 8 pairs, permuted K order
    const uint32_t base = F16 ? 0x64006400u : 0x43004300u, one = F16 ? 0x3C003C00u : 0x3F803F80u;
    auto fma2 = [&](uint32_t a, uint32_t c) { return F16 ? f16x2_fma(a, one, c) : bf16x2_fma(a, one, c); };
    if (FMT == COLI_FMT_INT4) {
        const uint32_t off = F16 ? 0xE408E408u : 0xC308C308u;  // -(1024 + 8) / -(128 + 8)
#pragma unroll
        for (int i = 0; i < 2; i++)
#pragma unroll
            for (int m = 0; m < 4; m++) out[4 * i + m] = fma2(lop3_and_or(w[i] >> (4 * m), 0x000F000Fu, base), off);
    } else if (FMT == COLI_FMT_INT2) {
        const uint32_t off = F16 ? 0xE402E402u : 0xC302C302u;  // -(1024 + 2) / -(128 + 2)
#pragma unroll
        for (int m = 0; m < 8; m++) out[m] = fma2(lop3_and_or(w[0] >> (2 * m), 0x00030003u, base), off);
    } else {
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const int v = (int)w[i];
            const float a = (float)((v << 24) >> 24), b = (float)((v << 16) >> 24);
            const float c = (float)((v << 8) >> 24), d = (float)(v >> 24);
            out[2 * i] = F16 ? pack_f16(a, b) : pack_bf16(a, b);
            out[2 * i + 1] = F16 ? pack_f16(c, d) : pack_bf16(c, d);
        }
    }
}

__device__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, TcSmem &ts, int32_t *err) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (*reinterpret_cast<volatile int *>(&ts.abort)) return false;
        if (globaltimer_ns() - t0 > kTcWaitNs) {
            *reinterpret_cast<volatile int *>(&ts.abort) = 1;
            atomicCAS(err, 0, (int)kErrWaitExpired);
            return false;
        }
    }
    return true;
}


// the final drain of a CTA's MMAs: bounded, but not cut short by another warp's abort
__device__ bool mbar_wait_drain(uint64_t *bar, uint32_t parity, int32_t *err) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > kTcWaitNs) {
            atomicCAS(err, 0, (int)kErrWaitExpired);
            return false;
        }
    }
    return true;
}

__device__ int slot_rows(const PfParams &P, int g) { return g < P.E ? P.counts[g] : P.T; }

__device__ Tile make_tile(const PfParams &P, const TcSmem &ts, int t) {
    // slot of tile t: last g with pref[g] <= t
    int lo = 0, hi = P.E + (P.Is > 0 ? 1 : 0) - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (ts.pref[mid] <= t) lo = mid;
        else hi = mid - 1;
    }
    const int g = lo;
    const bool sh = g == P.E;
    const coli_moe_expert ex = sh ? P.shared : P.experts[g];
    Tile T;
    T.fmt = sh ? P.sfmt : P.rfmt;
    T.inter = sh ? P.Is : P.I;
    const int mt = P.down ? (P.H + kTcM - 1) / kTcM : (T.inter + 63) / 64;
    const int local = t - ts.pref[g];
    const int nb = local / mt, mb = local % mt;
    const int n = slot_rows(P, g);
    T.n0 = nb * kTcN;
    T.ncur = min(kTcN, n - T.n0);
    T.N = (T.ncur + 15) & ~15;
    T.pbase = sh ? P.T * P.K : P.offsets[g];
    T.row0 = P.down ? mb * kTcM : mb * 64;
    T.w0 = static_cast<const uint8_t *>(P.down ? ex.down_w : ex.gate_w);
    T.w1 = static_cast<const uint8_t *>(ex.up_w);
    T.s0 = P.down ? ex.down_s : ex.gate_s;
    T.s1 = ex.up_s;
    T.slot = g;
    T.sh = sh ? 1 : 0;
    return T;
}

// a tensor map written by the generic proxy is made visible to this thread's later tensor copies
__device__ __forceinline__ void tmap_acquire(const CUtensorMap *map) {
    asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(map) : "memory");
}

__device__ __forceinline__ int qbytes(int fmt) { return fmt == COLI_FMT_INT4 ? 32 : fmt == COLI_FMT_INT2 ? 16 : 64; }

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

// 2-D tensor copy of the box at (x = innermost element, y = row) into shared memory, counted on bar
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// dequantise half h of K-step kin of a raw row into the 16 columns (16-bit K pairs, permuted K
// order) it fills in the A tile. The raw stage holds the tensor copy of 128 rows of 128 bytes with
// the 128-byte swizzle (16-byte chunk c of raw row rr at chunk c ^ (rr % 8)); gate/up tiles keep
// gate row j0 + i in raw row i and up row j0 + i in raw row 64 + i, down tiles row d0 + r in
// raw row r.
template <int FMT, bool F16>
__device__ __forceinline__ void dequant_half(const uint8_t *raw, int rr, int kin, int h, uint32_t (&col)[16]) {
    constexpr int QH = (FMT == COLI_FMT_INT4 ? 32 : FMT == COLI_FMT_INT2 ? 16 : 64) / 2;  // bytes of the half step
    const uint8_t *row = raw + rr * kChunkB;
    const int o = kin * 2 * QH + h * QH;  // byte offset of the half step in the logical row
    auto at = [&](int off) { return row + ((((off >> 4) ^ (rr & 7)) << 4) | (off & 15)); };
    uint32_t w[8];
    if (QH == 8) {
        const uint2 v = *reinterpret_cast<const uint2 *>(at(o));
        w[0] = v.x;
        w[1] = v.y;
    } else {
#pragma unroll
        for (int i = 0; i < QH / 16; i++) {
            const uint4 v = *reinterpret_cast<const uint4 *>(at(o + 16 * i));
            w[4 * i] = v.x;
            w[4 * i + 1] = v.y;
            w[4 * i + 2] = v.z;
            w[4 * i + 3] = v.w;
        }
    }
    constexpr int WPQ = QH / 8;  // words per 16 weights
#pragma unroll
    for (int c2 = 0; c2 < 2; c2++) {
        uint32_t out[8];
        deq16<FMT, F16>(w + c2 * WPQ, out);
#pragma unroll
        for (int k = 0; k < 8; k++) col[8 * c2 + k] = out[k];
    }
}

// 2^-e for the exponents the prepass writes (e in [-113, 275]): two exact factors
__device__ __forceinline__ float exp2_neg(int e) {
    const int e1 = max(-126, min(126, -e)), e2 = -e - e1;
    return __int_as_float((e1 + 127) << 23) * __int_as_float((max(-126, e2) + 127) << 23);
}

__device__ __forceinline__ uint16_t bf16_bits(float f) {
    return (uint16_t)(pack_bf16(f, 0.f) & 0xFFFFu);
}

__global__ void __launch_bounds__(kTcThreads, 1)
moe_prefill_tc_kernel(const PfParams P, const __grid_constant__ CUtensorMap tmB) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    uint8_t *sB = smem, *sR = sB + kTcBS * kStageB;
    TcSmem &ts = *reinterpret_cast<TcSmem *>(sR + kTcRS * kStageRaw);
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int nslots = P.E + (P.Is > 0 ? 1 : 0);

    // tile prefix over the slots: per-thread chunk sums, a warp scan of the chunk sums, then
    // every thread writes its chunk's prefix entries
    {
        constexpr int kChunks = 160;
        const int per = (nslots + kChunks - 1) / kChunks;
        auto tiles_of = [&](int g) {
            const int inter = g == P.E ? P.Is : P.I;
            const int mt = P.down ? (P.H + kTcM - 1) / kTcM : (inter + 63) / 64;
            return mt * ((slot_rows(P, g) + kTcN - 1) / kTcN);
        };
        int loc[8], sum = 0;  // per <= 8: nslots <= kMaxE + 1 = 1025 <= 8 * 160
#pragma unroll
        for (int i = 0; i < 8; i++) {
            const int g = tid * per + i;
            loc[i] = (tid < kChunks && i < per && g < nslots) ? tiles_of(g) : 0;
            sum += loc[i];
        }
        if (tid < kChunks) ts.pref[tid] = sum;  // scratch: chunk sums (pref is rewritten below)
        __syncthreads();
        if (warp == 0) {
            int v[5], s5 = 0;
#pragma unroll
            for (int i = 0; i < 5; i++) {
                v[i] = ts.pref[5 * lane + i];
                s5 += v[i];
            }
            int inc = s5;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, inc, o);
                if (lane >= o) inc += u;
            }
            int run = inc - s5;
#pragma unroll
            for (int i = 0; i < 5; i++) {
                const int vi = v[i];
                ts.pref[5 * lane + i] = run;
                run += vi;
            }
            if (lane == 31) ts.pref[kMaxE + 1] = inc;  // total
        }
        __syncthreads();
        int run = tid < kChunks ? ts.pref[tid] : 0;
        const int total_tiles = ts.pref[kMaxE + 1];
        __syncthreads();
        if (tid < kChunks) {
#pragma unroll
            for (int i = 0; i < 8; i++) {
                const int g = tid * per + i;
                if (i < per && g < nslots) ts.pref[g] = run;
                run += loc[i];
            }
        }
        if (tid == 0) ts.pref[nslots] = total_tiles;
    }
    __syncthreads();
    {  // this CTA's tile parameters, looked up in parallel once
        const int total0 = ts.pref[nslots];
        const int t = blockIdx.x + tid * gridDim.x;
        if (tid < kTileCap && t < total0) ts.tiles[tid] = make_tile(P, ts, t);
    }
    if (tid == 0) {
        ts.abort = 0;
        for (int s = 0; s < kTcRS; s++) {
            mbar_init(&ts.rfull[s], 1);
            mbar_init(&ts.rempty[s], kTcDeq);
        }
        for (int s = 0; s < kTcBS; s++) {
            mbar_init(&ts.bfull[s], 1);
            mbar_init(&ts.bempty[s], 1);
        }
        for (int s = 0; s < kTcA; s++) {
            mbar_init(&ts.full[s], kTcDeq);
            mbar_init(&ts.emptya[s], 1);
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(&ts.accf[b], 1);
            mbar_init(&ts.tfree[b], kTcEpi);
        }
        mbar_init(&ts.drain, 1);
        fence_mbar_init();
    }
    if (warp == kTcMmaWarp) {
        tmem_alloc(&ts.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tbase = ts.tmem_base;
    const int total = ts.pref[nslots];
    const int G = gridDim.x;
    auto nkb_of = [&](const Tile &T) { return (P.down ? T.inter : P.H) / kTcKB; };
    auto spc_of = [&](const Tile &T) { return kChunkB / qbytes(T.fmt); };  // K-steps per raw chunk
    auto tile_at = [&](int t) {  // t = blockIdx.x + i * G
        const int i = (t - (int)blockIdx.x) / G;
        return i < kTileCap ? ts.tiles[i] : make_tile(P, ts, t);
    };

    if (warp == 0) {
        // ---------------- weight copies: 2-D tensor copies of 128-byte K-chunks of the rows
        uint32_t gc = 0;  // chunks issued
        if (lane == 0) {
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += G) {
                const Tile T = tile_at(t);
                const int nkb = nkb_of(T), spc = spc_of(T), qb = qbytes(T.fmt);
                const CUtensorMap *maps = P.tmaps + 3 * (T.sh ? P.E : T.slot);
                const CUtensorMap *m0 = P.down ? maps + 2 : maps, *m1 = maps + 1;
                tmap_acquire(m0);
                if (!P.down) tmap_acquire(m1);
                for (int kb0 = 0; kb0 < nkb; kb0 += spc, gc++) {
                    const int s = gc % kTcRS;
                    const uint32_t use = gc / kTcRS;
                    if (use > 0 && !mbar_wait_bounded(&ts.rempty[s], (use - 1) & 1, ts, P.err)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&ts.rfull[s], (uint32_t)kStageRaw);
                    uint8_t *dst = sR + s * kStageRaw;
                    if (P.down) {
                        tma_load_2d(dst, m0, kb0 * qb, T.row0, &ts.rfull[s]);
                    } else {
                        tma_load_2d(dst, m0, kb0 * qb, T.row0, &ts.rfull[s]);
                        tma_load_2d(dst + 64 * kChunkB, m1, kb0 * qb, T.row0, &ts.rfull[s]);
                    }
                }
            }
            // every copy issued has landed before the CTA can end
            for (uint32_t q = gc > (uint32_t)kTcRS ? gc - kTcRS : 0; q < gc; q++)
                mbar_wait_drain(&ts.rfull[q % kTcRS], (q / kTcRS) & 1, P.err);
        }
        __syncwarp();
    } else if (warp == kWarpB) {
        // ---------------- activation copies: 2-D tensor copies of 32 token rows each
        uint32_t gb = 0;  // K-steps issued
        if (lane == 0) {
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += G) {
                const Tile T = tile_at(t);
                const int nkb = nkb_of(T), nbox = (T.N + kBoxRows - 1) / kBoxRows, row = T.pbase + T.n0;
                for (int kb = 0; kb < nkb; kb++, gb++) {
                    const int s = gb % kTcBS;
                    const uint32_t use = gb / kTcBS;
                    if (use > 0 && !mbar_wait_bounded(&ts.bempty[s], (use - 1) & 1, ts, P.err)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&ts.bfull[s], (uint32_t)(nbox * kBoxRows * 128));
                    for (int i = 0; i < nbox; i++)
                        tma_load_2d(sB + s * kStageB + i * kBoxRows * 128, &tmB, kb * kTcKB, row + i * kBoxRows,
                                    &ts.bfull[s]);
                }
            }
            for (uint32_t q = gb > (uint32_t)kTcBS ? gb - kTcBS : 0; q < gb; q++)
                mbar_wait_drain(&ts.bfull[q % kTcBS], (q / kTcBS) & 1, P.err);
        }
        __syncwarp();
    } else if (warp < kTcMmaWarp) {
        // ---------------- dequant warps
        // TMEM lanes 32 (w % 4) .. + 31 belong to warp w: row r = lane of that quarter, and
        // warps 2-5 / 6-9 take the two halves of the K-step
        const int r = 32 * (warp % 4) + lane, h = (warp - kDeq0) / 4;
        const uint32_t tlane = (uint32_t)(32 * (warp % 4)) << 16;
        // Software-pipelined: the store of step g to tensor memory completes while step g + 1 is
        // dequantised; only then is step g announced to the MMA warp.
        uint32_t g = 0, gc = 0;  // K-steps and raw chunks consumed
        int pend = -1;            // the A tile whose store is in flight, not yet announced
        bool ok = true;
        auto announce = [&]() {
            if (pend < 0) return;
            tmem_st_wait();
            tc_fence_before_sync();
            mbar_arrive(&ts.full[pend]);
            pend = -1;
        };
        for (int t = blockIdx.x; t < total && ok; t += G) {
            const Tile T = tile_at(t);
            const int fmt = T.fmt, nkb = nkb_of(T), spc = spc_of(T);
            for (int kb = 0; kb < nkb; kb++, g++) {
                const int kin = kb % spc, s = gc % kTcRS, a = g % kTcA;
                if (kin == 0 && !mbar_wait_bounded(&ts.rfull[s], (gc / kTcRS) & 1, ts, P.err)) {
                    ok = false;
                    break;
                }
                if (g >= (uint32_t)kTcA && !mbar_wait_bounded(&ts.emptya[a], ((g / kTcA) - 1) & 1, ts, P.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();  // the MMAs that read this A tile have completed
                const uint8_t *raw = sR + s * kStageRaw;
                const int rr = P.down ? r : (r & 1) * 64 + (r >> 1);  // raw row of A row r
                uint32_t col[16];
                // gate/up: f16 (the activations are per-token scaled f16); down: bf16 (h)
                if (!P.down) {
                    if (fmt == COLI_FMT_INT4) dequant_half<COLI_FMT_INT4, true>(raw, rr, kin, h, col);
                    else if (fmt == COLI_FMT_INT8) dequant_half<COLI_FMT_INT8, true>(raw, rr, kin, h, col);
                    else dequant_half<COLI_FMT_INT2, true>(raw, rr, kin, h, col);
                } else {
                    if (fmt == COLI_FMT_INT4) dequant_half<COLI_FMT_INT4, false>(raw, rr, kin, h, col);
                    else if (fmt == COLI_FMT_INT8) dequant_half<COLI_FMT_INT8, false>(raw, rr, kin, h, col);
                    else dequant_half<COLI_FMT_INT2, false>(raw, rr, kin, h, col);
                }
                if (kin == spc - 1 || kb == nkb - 1) {  // the chunk's last step is read: the raw stage is free
                    mbar_arrive(&ts.rempty[s]);
                    gc++;
                }
                announce();  // the previous step's store has had this step's dequantisation to land
                tmem_st_x16(tbase + tlane + kTmemA + 32 * a + 16 * h, col);
                pend = a;
            }
        }
        if (ok) announce();
    } else if (warp == kTcMmaWarp) {
        // ---------------- MMA issuer
        if (lane == 0) {
            uint32_t gk = 0;
            int it = 0;
            for (int t = blockIdx.x; t < total && !ts.abort; t += G, it++) {
                const Tile T = tile_at(t);
                const int nkb = nkb_of(T), b = it & 1;
                if (it >= 2 && !mbar_wait_bounded(&ts.tfree[b], ((it >> 1) - 1) & 1, ts, P.err)) break;
                tc_fence_after_sync();
                const uint32_t idesc = idesc_f32acc(kTcM, T.N, P.down != 0), dcol = tbase + b * kTcN;
                for (int kb = 0; kb < nkb; kb++, gk++) {
                    const int s = gk % kTcBS, a = gk % kTcA;
                    if (!mbar_wait_bounded(&ts.full[a], (gk / kTcA) & 1, ts, P.err)) break;
                    if (!mbar_wait_bounded(&ts.bfull[s], (gk / kTcBS) & 1, ts, P.err)) break;
                    tc_fence_after_sync();
                    const uint32_t ta = tbase + kTmemA + 32 * a, b0 = smem_u32(sB + s * kStageB);
#pragma unroll
                    for (int k = 0; k < kTcKB / 16; k++)  // K = 16: 8 columns of A, 32 bytes of each B row
                        tc_mma_f16kind_ta(dcol, ta + 8 * k, sdesc_k_sw128(b0 + 32 * k), idesc, (kb | k) != 0);
                    tc_commit(&ts.bempty[s]);
                    tc_commit(&ts.emptya[a]);
                }
                tc_commit(&ts.accf[b]);
            }
            // every MMA issued has completed before the tensor memory is freed: this wait ignores
            // the abort flag (an aborted CTA still drains what it issued). The MMAs in flight
            // are a few microseconds of work; should even this bounded wait expire, the error
            // word already says so and the context's results are undefined from then on.
            tc_commit(&ts.drain);
            mbar_wait_drain(&ts.drain, 0, P.err);
        }
        __syncwarp();
    } else {
        // ---------------- epilogue
        const int R = 32 * (warp % 4) + lane;  // accumulator row = TMEM lane of this thread
        int it = 0;
        for (int t = blockIdx.x; t < total && !ts.abort; t += G, it++) {
            const Tile T = tile_at(t);
            const int b = it & 1;
            float sc0 = 0.f, sc1 = 0.f;
            if (P.down) {
                sc0 = __ldg(T.s0 + min(T.row0 + R, P.H - 1));
            } else if ((R & 1) == 0) {
                const int j = min(T.row0 + (R >> 1), T.inter - 1);
                sc0 = __ldg(T.s0 + j);
                sc1 = __ldg(T.s1 + j);
            }
            if (!mbar_wait_bounded(&ts.accf[b], (it >> 1) & 1, ts, P.err)) break;
            tc_fence_after_sync();
            const uint32_t trow = tbase + b * kTcN + ((uint32_t)(32 * (warp % 4)) << 16);
            for (int c0 = 0; c0 < T.N; c0 += 16) {
                uint32_t v[16];
                tmem_ld_x16(trow + c0, v);
                tmem_ld_wait();
                if (P.down) {
                    const int d = T.row0 + R;
                    if (d < P.H) {
#pragma unroll
                        for (int i = 0; i < 16; i++) {
                            const int n = c0 + i;
                            if (n < T.ncur) P.y[(size_t)(T.pbase + T.n0 + n) * P.H + d] = __uint_as_float(v[i]) * sc0;
                        }
                    }
                } else {
                    uint32_t pv[16];
#pragma unroll
                    for (int i = 0; i < 16; i++) pv[i] = __shfl_xor_sync(0xffffffffu, v[i], 1);
                    const int j = T.row0 + (R >> 1);
                    if ((R & 1) == 0 && j < T.inter) {
                        const int col = kperm(T.fmt, j);
#pragma unroll
                        for (int i = 0; i < 16; i++) {
                            const int n = c0 + i;
                            if (n < T.ncur) {
                                // undo the token's 2^e of the f16 staging (exact), then the row scale
                                const float inv = exp2_neg(__ldg(P.xe + T.pbase + T.n0 + n));
                                const float gv = (__uint_as_float(v[i]) * inv) * sc0;
                                const float uv = (__uint_as_float(pv[i]) * inv) * sc1;
                                const float hv = gv / (1.f + expf(-gv)) * uv;
                                P.hb[(size_t)(T.pbase + T.n0 + n) * P.ldh + col] = bf16_bits(hv);
                            }
                        }
                    }
                }
            }
            tc_fence_before_sync();
            mbar_arrive(&ts.tfree[b]);
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == kTcMmaWarp) {
        tc_fence_after_sync();
        tmem_dealloc(tbase, kTmemCols);
    }
}

// The tensor maps of every expert matrix: templates encoded on the host (the matrix shapes: routed
// gate/up, routed down, shared gate/up, shared down) with each expert's base address put in on the
// device, one warp per map, written to the workspace table with the fence that orders them before
// any tensor copy that reads them.
struct TmapTemplates {
    CUtensorMap t[4];
};

__global__ void __launch_bounds__(96) tmap_build_kernel(const __grid_constant__ TmapTemplates tp,
                                                        const coli_moe_expert *experts, coli_moe_expert shared,
                                                        int E, CUtensorMap *out) {
    __shared__ __align__(128) CUtensorMap sm[3];
    const int slot = blockIdx.x, warp = threadIdx.x / 32, lane = threadIdx.x % 32;  // warp: gate, up, down
    const bool sh = slot == E;
    const coli_moe_expert ex = sh ? shared : experts[slot];
    const CUtensorMap &src = tp.t[(sh ? 2 : 0) + (warp == 2 ? 1 : 0)];
    reinterpret_cast<uint32_t *>(&sm[warp])[lane] = reinterpret_cast<const uint32_t *>(&src)[lane];
    __syncwarp();
    if (lane == 0) {
        const void *addr = warp == 0 ? ex.gate_w : warp == 1 ? ex.up_w : ex.down_w;
        asm volatile("tensormap.replace.tile.global_address.shared::cta.b1024.b64 [%0], %1;" ::"r"(smem_u32(&sm[warp])),
                     "l"(addr)
                     : "memory");
    }
    __syncwarp();
    asm volatile(
        "tensormap.cp_fenceproxy.global.shared::cta.tensormap::generic.release.gpu.sync.aligned [%0], [%1], 128;" ::"l"(
            out + 3 * slot + warp),
        "r"(smem_u32(&sm[warp]))
        : "memory");
}

// x (fp32) -> f16 rows in bucket order (rows p < T*K: token perm[p] / K, up to offsets[E]) and
// plain order for the shared expert (rows T*K + t), K-permuted per the rows' weight format. One
// warp per row: row p is scaled by 2^xe[p], chosen from the row's max |x| so that the largest
// element lands in [2^14, 2^15), then rounded to f16 (nearest even): every element keeps an
// 11-bit significand unless it is below 2^-24 of the row's largest.
__global__ void __launch_bounds__(256) prefill_prepass_kernel(const float *__restrict__ x, const int32_t *__restrict__ perm,
                                                              const int32_t *__restrict__ offsets, uint16_t *xb,
                                                              int32_t *xe, int T, int H, int K, int E, int rfmt,
                                                              int sfmt, int has_shared) {
    const int lane = threadIdx.x % 32;
    const int warp0 = (blockIdx.x * blockDim.x + threadIdx.x) / 32, nwarps = gridDim.x * blockDim.x / 32;
    const int rows = T * K + (has_shared ? T : 0);
    const int kept = offsets[E];
    for (int p = warp0; p < rows; p += nwarps) {
        int t, fmt;
        if (p < T * K) {
            if (p >= kept) continue;
            t = perm[p] / K;
            fmt = rfmt;
        } else {
            t = p - T * K;
            fmt = sfmt;
        }
        const float4 *src = reinterpret_cast<const float4 *>(x + (size_t)t * H);
        float mx = 0.f;
        for (int q = lane; q < H / 4; q += 32) {
            const float4 v = __ldg(src + q);
            mx = fmaxf(mx, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        int e = 0;
        if (mx > 0.f) {
            const int ex = (int)((__float_as_uint(mx) >> 23) & 255u);
            e = 14 - (ex == 0 ? -126 : ex - 127);
        }
        const int e1 = max(-126, min(126, e)), e2 = e - e1;  // 2^e as two exact factors
        const float f1 = __int_as_float((e1 + 127) << 23), f2 = __int_as_float((e2 + 127) << 23);
        for (int b = lane; b < H / 16; b += 32) {
            float v[16];
#pragma unroll
            for (int q = 0; q < 4; q++) {
                const float4 f = __ldg(src + 4 * b + q);
                v[4 * q] = f.x;
                v[4 * q + 1] = f.y;
                v[4 * q + 2] = f.z;
                v[4 * q + 3] = f.w;
            }
            float o[16];
#pragma unroll
            for (int j = 0; j < 16; j++) o[kperm(fmt, j)] = (v[j] * f1) * f2;
            uint32_t w[8];
#pragma unroll
            for (int j = 0; j < 8; j++) w[j] = pack_f16(o[2 * j], o[2 * j + 1]);
            uint4 *dst = reinterpret_cast<uint4 *>(xb + (size_t)p * H + b * 16);
            dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
            dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
        }
        if (lane == 0) xe[p] = e;
    }
}

}  // namespace

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link against libcuda)
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

bool prefill_supported(const coli_moe_desc &d) {
    return d.H % 64 == 0 && d.I % 64 == 0 && d.I_shared % 64 == 0 && d.E <= kMaxE;
}


cudaError_t launch_prefill(const PrefillWork &w, int part, cudaStream_t st) {
    cudaError_t e;
    if (part == 0) {
        const long long rows = (long long)w.T * w.K + (w.I_shared > 0 ? w.T : 0);
        const int blocks = (int)std::min<long long>((rows + 7) / 8, (long long)w.grid * 16);
        prefill_prepass_kernel<<<blocks, 256, 0, st>>>(w.x, w.perm, w.offsets, w.xb, w.xe, w.T, w.H, w.K, w.E,
                                                       w.routed_fmt, w.shared_fmt, w.I_shared > 0);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode) return cudaErrorNotSupported;
    // a 2-D map of 16-bit or 8-bit rows, boxes of 128 bytes x box_rows, 128-byte swizzle; the base
    // address is a placeholder for the weight templates (replaced per expert on the device)
    auto map2d = [&](CUtensorMap *m, CUtensorMapDataType dt, size_t esize, const void *base, size_t cols, size_t rows,
                     uint32_t box_rows) {
        const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
        const cuuint64_t strides[1] = {(cuuint64_t)(cols * esize)};
        const cuuint32_t box[2] = {(cuuint32_t)(128 / esize), box_rows};
        const cuuint32_t estr[2] = {1, 1};
        return encode(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    };
    if (part == 0) {
        TmapTemplates tp;
        const int sfmt = w.I_shared > 0 ? w.shared_fmt : w.routed_fmt, Is = w.I_shared > 0 ? w.I_shared : w.I;
        if (!map2d(&tp.t[0], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, w.xb, row_bytes(w.routed_fmt, w.H), w.I, 64) ||
            !map2d(&tp.t[1], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, w.xb, row_bytes(w.routed_fmt, w.I), w.H, 128) ||
            !map2d(&tp.t[2], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, w.xb, row_bytes(sfmt, w.H), Is, 64) ||
            !map2d(&tp.t[3], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, w.xb, row_bytes(sfmt, Is), w.H, 128))
            return cudaErrorInvalidValue;
        coli_moe_expert sh = w.shared;
        if (w.I_shared == 0) sh = coli_moe_expert{w.xb, w.xb, w.xb, nullptr, nullptr, nullptr};  // unused slot
        tmap_build_kernel<<<w.E + 1, 96, 0, st>>>(tp, w.experts, sh, w.E, static_cast<CUtensorMap *>(w.tmaps));
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    PfParams P{};
    P.tmaps = static_cast<const CUtensorMap *>(w.tmaps);
    P.experts = w.experts;
    P.shared = w.shared;
    P.counts = w.counts;
    P.offsets = w.offsets;
    P.xb = w.xb;
    P.xe = w.xe;
    P.hb = w.hb;
    P.y = w.y;
    P.err = w.err;
    P.T = w.T;
    P.H = w.H;
    P.I = w.I;
    P.E = w.E;
    P.K = w.K;
    P.Is = w.I_shared;
    P.rfmt = w.routed_fmt;
    P.sfmt = w.shared_fmt;
    P.ldh = w.ldh;
    P.down = part;
    // the tensor map of the B operand: the activation rows (f16, gate/up) or h (bf16, down),
    // [rows][cols] 16-bit values, copied 64 columns (128 bytes) x 32 rows at a time with the
    // 128-byte swizzle of the MMA's K-major layout; rows past the end read as zeros
    const size_t rows = (size_t)w.T * w.K + (w.I_shared > 0 ? w.T : 0);
    const size_t cols = part == 0 ? (size_t)w.H : (size_t)w.ldh;
    CUtensorMap tmB;
    if (!map2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, part == 0 ? (const void *)w.xb : (const void *)w.hb, cols, rows,
               kBoxRows))
        return cudaErrorInvalidValue;
    const size_t smem = tc_smem_bytes();
    if ((e = cudaFuncSetAttribute(moe_prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
        cudaSuccess)
        return e;
    moe_prefill_tc_kernel<<<w.grid, kTcThreads, smem, st>>>(P, tmB);
    return cudaGetLastError();
}

}  // namespace colimoe
