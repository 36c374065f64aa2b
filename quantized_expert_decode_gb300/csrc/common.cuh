// common.cuh — shared definitions of libcolimoe's kernels and host code (not part of the ABI).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "colimoe.h"

namespace colimoe {

constexpr int kWarp = 32;
constexpr unsigned kFull = 0xffffffffu;
constexpr int kMaxK = 32;
constexpr int kMaxE = 1024;
constexpr int kMaxT = 65536;
constexpr int kMaxDim = 65536;

// Kernel-side error codes written to the workspace error word (first error wins).
enum KernelError : int {
    kErrNone = 0,
    kErrNoCandidate = 1,   // no expert had a finite choice above -1e30
    kErrBadExpert = 2,     // an expert id outside [0, E) reached the bucketing step
    kErrWaitExpired = 3,   // a bounded spin-wait gave up
};

__host__ __device__ inline size_t align_up(size_t n, size_t a) { return (n + a - 1) / a * a; }

// Bytes of one packed row of n elements.
__host__ __device__ inline int64_t row_bytes(int fmt, int64_t n) {
    return fmt == COLI_FMT_INT8 ? n : (fmt == COLI_FMT_INT4 || fmt == COLI_FMT_INT4G) ? (n + 1) / 2 : (n + 3) / 4;
}

// Elements per 16-byte chunk and the element-count granule the kernels need per format.
__host__ __device__ inline int elems_per_chunk(int fmt) {
    return fmt == COLI_FMT_INT8 ? 16 : (fmt == COLI_FMT_INT4 || fmt == COLI_FMT_INT4G) ? 32 : 64;
}

// Device workspace layout. Every region starts on a 256-byte boundary.
struct WsLayout {
    size_t err;       // control block of the call; its first int32 is the error word
    size_t part;      // f32 [S][T][E] router partial logits
    size_t sig;       // f32 [T][E]
    size_t choice;    // f32 [T][E]
    size_t idx;       // i32 [T][K]
    size_t w;         // f32 [T][K]
    size_t keff;      // i32 [T]
    size_t counts;    // i32 [E]
    size_t offsets;   // i32 [E+1]
    size_t perm;      // i32 [T*K]
    size_t pos;       // i32 [T*K]  position of assignment a in perm, -1 if not kept
    size_t act;       // i32 [E]    active routed experts, ascending
    size_t meta;      // i32 [4]    [0] = active count U, [1] = kept assignments N
    size_t h;         // f32 [T*K + T][max(I, I_shared)]  SiLU(gate)*up rows
    size_t y;         // f32 [T*K + T][H]                 down-projection rows
    size_t xstage;    // f32 [T][H]  device copy of a host x
    size_t ostage;    // f32 [T][H]  device staging of a host out
    size_t tmaps;     // 128-byte tensor maps [E + 1][3] (gate, up, down of every expert; the
                      // shared expert last), written on the device for the tensor-core GEMMs
    size_t total;
    int router_splits;
};

// Router GEMM tiling (router.cu); the split count decides the partial-logit buffer size.
constexpr int kRouterTM = 32;   // tokens per tile
constexpr int kRouterTE = 64;   // experts per tile
constexpr int kRouterTK = 32;   // k per smem stage

constexpr int kRouterTargetCtas = 304;  // two per SM of a 152-SM GB300

// From kRouterBigT tokens the logits run as 128-token x 128-expert tiles with 8 x 8 outputs per
// thread (router_gemm_kernel), k in steps of kRgK.
constexpr int kRouterBigT = 128;
constexpr int kRgT = 128, kRgE = 128, kRgK = 16;

inline int router_splits(const coli_moe_desc &d) {
    const bool big = d.T >= kRouterBigT;
    const int tm = big ? kRgT : kRouterTM, te = big ? kRgE : kRouterTE;
    long tiles = (long)((d.T + tm - 1) / tm) * ((d.E + te - 1) / te);
    // the big tiles fill one wave of two CTAs per SM without a partial second one
    long want = big ? kRouterTargetCtas / tiles : (kRouterTargetCtas + tiles - 1) / tiles;
    // at least one k-stage per split (four of the big tiles' shorter stages)
    long max_s = big ? (d.H + 4 * kRgK - 1) / (4 * kRgK) : (d.H + kRouterTK - 1) / kRouterTK;
    if (want > max_s) want = max_s;
    if (want < 1) want = 1;
    if (want > 128) want = 128;
    return (int)want;
}

size_t decode_ctrl_bytes();

inline WsLayout ws_layout(const coli_moe_desc &d) {
    WsLayout L{};
    size_t p = 0;
    auto take = [&](size_t bytes) {
        size_t at = p;
        p = align_up(p + (bytes ? bytes : 1), 256);
        return at;
    };
    const size_t T = d.T, E = d.E, K = d.K, H = d.H;
    const size_t rows = T * K + (d.I_shared > 0 ? T : 0);
    const size_t imax = (size_t)(d.I > d.I_shared ? d.I : d.I_shared);
    L.router_splits = router_splits(d);
    L.err = take(decode_ctrl_bytes());
    L.part = take((size_t)L.router_splits * T * E * 4);
    L.sig = take(T * E * 4);
    L.choice = take(T * E * 4);
    L.idx = take(T * K * 4);
    L.w = take(T * K * 4);
    L.keff = take(T * 4);
    L.counts = take(E * 4);
    L.offsets = take((E + 1) * 4);
    L.perm = take(T * K * 4);
    L.pos = take(T * K * 4);
    L.act = take(E * 4);
    L.meta = take(16);
    L.h = take(rows * imax * 4);
    L.y = take(rows * H * 4);
    L.xstage = take(T * H * 4);
    L.ostage = take(T * H * 4);
    L.tmaps = take((E + 1) * 3 * 128);
    L.total = p;
    return L;
}

template <typename T>
inline T *ws_ptr(void *ws, size_t off) {
    return reinterpret_cast<T *>(static_cast<char *>(ws) + off);
}

}  // namespace colimoe
