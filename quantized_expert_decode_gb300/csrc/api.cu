// api.cu — the C ABI of libcolimoe (include/colimoe.h): argument validation, workspace layout
// and the launch sequence of the block. No allocation, no synchronisation except where the
// header says so (coli_moe_forward_host, coli_moe_check).
#include <algorithm>
#include <cmath>
#include <cstddef>
#include <cstring>
#include <mutex>

#include <atomic>
#include <chrono>
#include <random>

#include "kernels.h"

using namespace colimoe;

namespace {

thread_local int g_last_cuda = 0;

int cuda_fail(cudaError_t e) {
    g_last_cuda = (int)e;
    return COLI_MOE_ECUDA;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_device() {
    static int cache[64];  // 0 unknown, 1 ok, 2 wrong device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev >= 0 && dev < 64 && cache[dev]) return cache[dev] == 1 ? COLI_MOE_OK : COLI_MOE_EDEVICE;
    int maj = 0, min = 0;
    if ((e = cudaDeviceGetAttribute(&maj, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&min, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
        return cuda_fail(e);
    const bool ok = maj == 10 && min == 3;
    if (dev >= 0 && dev < 64) cache[dev] = ok ? 1 : 2;
    return ok ? COLI_MOE_OK : COLI_MOE_EDEVICE;
}

int check_fmt(int fmt) {
    if (fmt == COLI_FMT_INT8 || fmt == COLI_FMT_INT4 || fmt == COLI_FMT_INT2 || fmt == COLI_FMT_INT4G)
        return COLI_MOE_OK;
    if (fmt == 0) return COLI_MOE_ENOTSUP;  // f32 experts: a glm.c format this library does not take
    return COLI_MOE_EINVAL;
}

// an expert of the block is int4-grouped (those run the general kernels)
bool grouped(const coli_moe_desc &d) {
    return d.routed_fmt == COLI_FMT_INT4G || (d.I_shared > 0 && d.shared_fmt == COLI_FMT_INT4G);
}

// blocks that run the general launches for T > 1: a grouped expert, or the IDOT kernels requested
bool general_only(const coli_moe_desc &d) { return grouped(d) || d.idot != 0; }

// group sizes the grouped kernels take: whole 16-byte chunks (32 int4 inputs) per group
bool group_size_ok(int gs) { return gs >= 32 && gs <= kMaxDim && gs % 32 == 0; }

int validate_desc(const coli_moe_desc *d) {
    if (!d) return COLI_MOE_EINVAL;
    if (d->T < 1 || d->T > kMaxT || d->H < 1 || d->H > kMaxDim || d->I < 1 || d->I > kMaxDim ||
        d->E < 1 || d->E > kMaxE || d->K < 1 || d->K > d->E || d->K > kMaxK || d->I_shared < 0 ||
        d->I_shared > kMaxDim || (d->norm_topk != 0 && d->norm_topk != 1) || d->ksel < 0 ||
        d->ksel > d->K || !(d->top_p >= 0.f && d->top_p < 1.f) || !std::isfinite(d->routed_scale) ||
        (d->idot != 0 && d->idot != 1))
        return COLI_MOE_EINVAL;
    int rc = check_fmt(d->routed_fmt);
    if (rc) return rc;
    const int g = elems_per_chunk(d->routed_fmt);
    if (d->H % g || d->I % g) return COLI_MOE_ENOTSUP;
    if (d->I_shared > 0) {
        if ((rc = check_fmt(d->shared_fmt))) return rc;
        const int gs = elems_per_chunk(d->shared_fmt);
        if (d->H % gs || d->I_shared % gs) return COLI_MOE_ENOTSUP;
    }
    if (grouped(*d) && !group_size_ok(d->group_size)) return COLI_MOE_EINVAL;
    return COLI_MOE_OK;
}

int check_ws(const coli_moe_desc *d, void *ws, size_t ws_bytes) {
    if (!ws || !aligned(ws, 256)) return COLI_MOE_EWORKSPACE;
    if (ws_bytes < ws_layout(*d).total) return COLI_MOE_EWORKSPACE;
    return COLI_MOE_OK;
}

int ksel_of(const coli_moe_desc *d) { return (d->ksel > 0 && d->ksel < d->K) ? d->ksel : d->K; }

// Router + selection (+ buckets when want_buckets). Outputs default to the workspace.
int run_route(const coli_moe_desc *d, const float *x, const float *W_r, const float *bias,
              int32_t *idx, float *w, int32_t *keff, int32_t *counts, int32_t *offsets,
              int32_t *perm, bool want_buckets, void *ws, cudaStream_t st) {
    const WsLayout L = ws_layout(*d);
    int32_t *err = ws_ptr<int32_t>(ws, L.err);
    // the error word starts each call at zero (a plain 4-byte memset node in a graph)
    cudaError_t e = cudaMemsetAsync(err, 0, sizeof(int32_t), st);
    if (e != cudaSuccess) return cuda_fail(e);
    if (!idx) idx = ws_ptr<int32_t>(ws, L.idx);
    if (!w) w = ws_ptr<float>(ws, L.w);
    if (!keff) keff = ws_ptr<int32_t>(ws, L.keff);
    float *part = ws_ptr<float>(ws, L.part);
    if ((e = launch_router_partial(x, W_r, part, d->T, d->H, d->E, L.router_splits, st)) != cudaSuccess)
        return cuda_fail(e);
    if ((e = launch_select(part, L.router_splits, bias, d->T, d->E, d->K, d->ksel, d->top_p,
                           d->norm_topk, d->routed_scale, ws_ptr<float>(ws, L.sig),
                           ws_ptr<float>(ws, L.choice), idx, w, keff, err, st)) != cudaSuccess)
        return cuda_fail(e);
    if (!want_buckets) return COLI_MOE_OK;
    if (!counts) counts = ws_ptr<int32_t>(ws, L.counts);
    if (!offsets) offsets = ws_ptr<int32_t>(ws, L.offsets);
    if (!perm) perm = ws_ptr<int32_t>(ws, L.perm);
    if ((e = launch_bucket(idx, keff, d->T, d->K, d->E, counts, offsets, perm, ws_ptr<int32_t>(ws, L.pos),
                           ws_ptr<int32_t>(ws, L.act), ws_ptr<int32_t>(ws, L.meta), err, st)) != cudaSuccess)
        return cuda_fail(e);
    return COLI_MOE_OK;
}

int validate_expert_ptrs(const coli_moe_expert *s) {
    if (!s->gate_w || !s->up_w || !s->down_w || !s->gate_s || !s->up_s || !s->down_s) return COLI_MOE_EINVAL;
    if (!aligned(s->gate_w, 16) || !aligned(s->up_w, 16) || !aligned(s->down_w, 16) ||
        !aligned(s->gate_s, 4) || !aligned(s->up_s, 4) || !aligned(s->down_s, 4))
        return COLI_MOE_EALIGN;
    return COLI_MOE_OK;
}

int record(void *const *events, int i, cudaStream_t st) {
    if (!events) return COLI_MOE_OK;
    cudaError_t e = cudaEventRecord(static_cast<cudaEvent_t>(events[i]), st);
    return e == cudaSuccess ? COLI_MOE_OK : cuda_fail(e);
}

int num_sms() {
    static int cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 152;
    if (dev >= 0 && dev < 64 && cache[dev]) return cache[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 152;
    if (dev >= 0 && dev < 64) cache[dev] = n;
    return n;
}

// Call ids of the single-token kernel: a random 64-bit base per process (so that ids left in a
// workspace by another process never match) plus a counter.
uint64_t next_call_id() {
    static std::atomic<uint64_t> next{[] {
        std::random_device rd;
        uint64_t b = ((uint64_t)rd() << 32) ^ (uint64_t)rd();
        b ^= (uint64_t)std::chrono::steady_clock::now().time_since_epoch().count() * 0x9E3779B97F4A7C15ull;
        return b | 1ull;
    }()};
    return next.fetch_add(2, std::memory_order_relaxed);
}

// The layer tail (coli_moe_forward_tail): the block runs on rmsnorm(resid) * norm_w and adds
// resid to its output. NULL when the call is the block alone.
struct Tail {
    const float *resid, *norm_w;
    float eps;
};

// T <= 64: router, selection, buckets, experts and combine in one persistent launch
// (decode.cu); T > 8 computes the router logits in a preceding launch.
int run_forward_decode(const coli_moe_desc *d, const float *x, const float *W_r, const float *bias,
                       const coli_moe_expert *experts, const coli_moe_expert *shared, float *out,
                       int32_t *idx_out, float *w_out, void *ws, cudaStream_t st,
                       void *const *events, const DecParams &plan, int grid, const Tail *tail) {
    const WsLayout L = ws_layout(*d);
    DecParams P = plan;
    P.x = x;
    if (tail) {  // the single-token kernel normalises resid itself; the others get x normalised
        P.resid = tail->resid;
        P.norm_w = tail->norm_w;
        P.eps = tail->eps;
    }
    P.Wr = W_r;
    P.bias = bias;
    P.experts = experts;
    if (shared) P.shared = *shared;
    P.out = out;
    P.part = ws_ptr<float>(ws, L.part);
    P.sig = ws_ptr<float>(ws, L.sig);
    P.choice = ws_ptr<float>(ws, L.choice);
    P.w = w_out ? w_out : ws_ptr<float>(ws, L.w);
    P.idx = idx_out ? idx_out : ws_ptr<int32_t>(ws, L.idx);
    P.keff = ws_ptr<int32_t>(ws, L.keff);
    P.counts = ws_ptr<int32_t>(ws, L.counts);
    P.offsets = ws_ptr<int32_t>(ws, L.offsets);
    P.perm = ws_ptr<int32_t>(ws, L.perm);
    P.pos = ws_ptr<int32_t>(ws, L.pos);
    P.act = ws_ptr<int32_t>(ws, L.act);
    P.h = ws_ptr<float>(ws, L.h);
    P.y = ws_ptr<float>(ws, L.y);
    P.ctrl = ws_ptr<DecCtrl>(ws, L.err);
    P.T = d->T;
    P.H = d->H;
    P.I = d->I;
    P.E = d->E;
    P.K = d->K;
    P.Is = d->I_shared;
    // int4-grouped weights run in the int4 instances, their scales applied by group (rgs, sgs)
    P.rfmt = d->routed_fmt == COLI_FMT_INT4G ? COLI_FMT_INT4 : d->routed_fmt;
    P.sfmt = d->shared_fmt == COLI_FMT_INT4G ? COLI_FMT_INT4 : d->shared_fmt;
    P.Ksel = ksel_of(d);
    P.norm_topk = d->norm_topk;
    P.top_p = d->top_p;
    P.rscale = d->routed_scale;
    P.ldh = d->I > d->I_shared ? d->I : d->I_shared;
    const int splits = std::min(L.router_splits, kTokSlices);
    if (P.route_only) P.nks = splits;
    if ((size_t)P.nks * d->T * d->E * sizeof(float) > L.sig - L.part) return COLI_MOE_ENOTSUP;
    int rc;
    if ((rc = record(events, 0, st))) return rc;
    cudaError_t e = cudaSuccess;
    if (P.single) {
        // the single-token kernel resets its own counters: CTA 0 zeroes them and publishes this
        // call's id, which no earlier call (of this or another process) has used
        P.call_id = next_call_id();
    } else if ((e = cudaMemsetAsync(P.ctrl, 0, sizeof(DecCtrl), st)) != cudaSuccess) {
        return cuda_fail(e);
    }
    if (P.route_only &&
        (e = launch_router_partial(x, W_r, P.part, d->T, d->H, d->E, splits, st)) != cudaSuccess)
        return cuda_fail(e);
    if ((rc = record(events, 1, st))) return rc;
    if ((e = P.single ? launch_decode1(P, grid, st) : launch_decode(P, grid, st)) != cudaSuccess) return cuda_fail(e);
    if ((rc = record(events, 2, st))) return rc;
    if ((rc = record(events, 3, st))) return rc;
    return record(events, 4, st);
}

// the persistent decode kernel's plan and grid for this description (false: not applicable):
// the single-token kernel for T = 1 when its shared memory fits, else the token-group kernel.
// IDOT and int4-grouped blocks run the single-token kernel at T = 1 (not both at once) and the
// general launches otherwise.
bool decode_plan_for(const coli_moe_desc &d, DecParams &P, int &grid) {
    if (general_only(d) && d.T != 1) return false;
    const int sms0 = num_sms();
    for (int per_sm = 2; per_sm >= 1 && d.T == 1; per_sm--) {
        DecParams Q{};
        grid = per_sm * sms0;
        if (decode1_plan(d, Q, grid) && decode1_ctas_per_sm(Q) >= per_sm) {
            P = Q;
            return true;
        }
    }
    if (!decode_supported(d) || general_only(d)) return false;
    const int sms = num_sms();
    grid = 2 * sms;
    if (!decode_plan(d, P, grid)) return false;
    const int occ = decode_ctas_per_sm(P);
    if (occ < 1) return false;
    if (occ < 2) {
        grid = sms;
        if (!decode_plan(d, P, grid)) return false;
    }
    return true;
}

int run_forward(const coli_moe_desc *d, const float *x, const float *W_r, const float *bias,
                const coli_moe_expert *experts, const coli_moe_expert *shared, float *out,
                int32_t *idx_out, float *w_out, void *ws, cudaStream_t st,
                void *const *events = nullptr, const Tail *tail = nullptr) {
    const WsLayout L = ws_layout(*d);
    const float *resid = tail ? tail->resid : nullptr;
    // the layer tail outside the single-token kernel: a prologue launch writes the normalised
    // rows into the workspace's staging rows, which the rest of the block reads as x
    auto normalise = [&]() -> int {
        float *xn = ws_ptr<float>(ws, L.xstage);
        cudaError_t e = launch_rmsnorm(tail->resid, tail->norm_w, tail->eps, d->T, d->H, xn, st);
        if (e != cudaSuccess) return cuda_fail(e);
        x = xn;
        return COLI_MOE_OK;
    };
    {
        DecParams plan{};
        int grid = 0;
        if (decode_plan_for(*d, plan, grid)) {
            if (tail && !plan.single) {
                if (int rc = normalise()) return rc;
            }
            return run_forward_decode(d, x, W_r, bias, experts, shared, out, idx_out, w_out, ws, st, events,
                                      plan, grid, tail);
        }
    }
    if (tail) {
        if (int rc = normalise()) return rc;
    }
    if (int rc0 = record(events, 0, st)) return rc0;
    int32_t *idx = idx_out ? idx_out : ws_ptr<int32_t>(ws, L.idx);
    float *w = w_out ? w_out : ws_ptr<float>(ws, L.w);
    int32_t *keff = ws_ptr<int32_t>(ws, L.keff);
    int rc = run_route(d, x, W_r, bias, idx, w, keff, nullptr, nullptr, nullptr, true, ws, st);
    if (rc) return rc;
    if ((rc = record(events, 1, st))) return rc;
    if (d->T > kDecMaxT && !general_only(*d) && prefill_supported(*d)) {
        PrefillWork pw{};
        pw.experts = experts;
        if (shared) pw.shared = *shared;
        pw.x = x;
        pw.counts = ws_ptr<int32_t>(ws, L.counts);
        pw.offsets = ws_ptr<int32_t>(ws, L.offsets);
        pw.perm = ws_ptr<int32_t>(ws, L.perm);
        // the f16 activations and their row exponents live in the y region: only the gate/up
        // GEMM reads them, before the down GEMM writes y
        pw.xb = ws_ptr<uint16_t>(ws, L.y);
        const size_t rows = (size_t)d->T * d->K + (d->I_shared > 0 ? d->T : 0);  // the rows of y
        pw.xe = ws_ptr<int32_t>(ws, L.y + align_up(rows * d->H * sizeof(uint16_t), 256));
        pw.hb = ws_ptr<uint16_t>(ws, L.h);
        pw.y = ws_ptr<float>(ws, L.y);
        pw.err = ws_ptr<int32_t>(ws, L.err);
        pw.T = d->T;
        pw.H = d->H;
        pw.I = d->I;
        pw.E = d->E;
        pw.K = d->K;
        pw.I_shared = d->I_shared;
        pw.routed_fmt = d->routed_fmt;
        pw.shared_fmt = d->shared_fmt;
        pw.ldh = d->I > d->I_shared ? d->I : d->I_shared;
        pw.grid = num_sms();
        pw.tmaps = ws_ptr<void>(ws, L.tmaps);
        cudaError_t e;
        if ((e = launch_prefill(pw, 0, st)) != cudaSuccess) return cuda_fail(e);
        if ((rc = record(events, 2, st))) return rc;
        if ((e = launch_prefill(pw, 1, st)) != cudaSuccess) return cuda_fail(e);
        if ((rc = record(events, 3, st))) return rc;
        if ((e = launch_combine(pw.y, w, keff, ws_ptr<int32_t>(ws, L.pos), d->T, d->H, d->K,
                                d->I_shared > 0, resid, out, st)) != cudaSuccess)
            return cuda_fail(e);
        return record(events, 4, st);
    }
    ExpertWork W{};
    W.experts = experts;
    if (shared) W.shared = *shared;
    W.x = x;
    W.counts = ws_ptr<int32_t>(ws, L.counts);
    W.offsets = ws_ptr<int32_t>(ws, L.offsets);
    W.perm = ws_ptr<int32_t>(ws, L.perm);
    W.act = ws_ptr<int32_t>(ws, L.act);
    W.meta = ws_ptr<int32_t>(ws, L.meta);
    W.h = ws_ptr<float>(ws, L.h);
    W.y = ws_ptr<float>(ws, L.y);
    W.err = ws_ptr<int32_t>(ws, L.err);
    W.T = d->T;
    W.H = d->H;
    W.I = d->I;
    W.E = d->E;
    W.K = d->K;
    W.I_shared = d->I_shared;
    W.routed_fmt = d->routed_fmt;
    W.shared_fmt = d->shared_fmt;
    W.ldh = d->I > d->I_shared ? d->I : d->I_shared;
    W.group_size = d->group_size;
    W.idot = d->idot;
    const long max_active = std::min<long>((long)d->E, (long)d->T * ksel_of(d));
    W.slots = (int)max_active + (d->I_shared > 0 ? 1 : 0);
    cudaError_t e;
    if ((e = launch_gateup(W, st)) != cudaSuccess) return cuda_fail(e);
    if ((rc = record(events, 2, st))) return rc;
    if ((e = launch_down(W, st)) != cudaSuccess) return cuda_fail(e);
    if ((rc = record(events, 3, st))) return rc;
    if ((e = launch_combine(W.y, w, keff, ws_ptr<int32_t>(ws, L.pos), d->T, d->H, d->K,
                            d->I_shared > 0, resid, out, st)) != cudaSuccess)
        return cuda_fail(e);
    return record(events, 4, st);
}

int validate_forward(const coli_moe_desc *desc, const float *x, const float *W_r, const float *bias,
                     const coli_moe_expert *experts, const coli_moe_expert *shared, const float *out,
                     void *ws, size_t ws_bytes) {
    int rc = validate_desc(desc);
    if (rc) return rc;
    if (!x || !W_r || !bias || !experts || !out) return COLI_MOE_EINVAL;
    if ((desc->I_shared > 0) != (shared != nullptr)) return COLI_MOE_EINVAL;
    if (shared && (rc = validate_expert_ptrs(shared))) return rc;
    if (!aligned(W_r, 16) || !aligned(bias, 4) || !aligned(experts, 8)) return COLI_MOE_EALIGN;
    return check_ws(desc, ws, ws_bytes);
}

}  // namespace

extern "C" {

size_t coli_moe_workspace_bytes(const coli_moe_desc *desc) {
    if (validate_desc(desc) != COLI_MOE_OK) return 0;
    return ws_layout(*desc).total;
}

int coli_moe_route(const coli_moe_desc *desc, const float *x, const float *W_r, const float *bias,
                   int32_t *idx, float *w, int32_t *keff, int32_t *counts, int32_t *offsets,
                   int32_t *perm, void *ws, size_t ws_bytes, coli_stream_t stream) {
    int rc = validate_desc(desc);
    if (rc) return rc;
    if (!x || !W_r || !bias || !idx || !w) return COLI_MOE_EINVAL;
    if (!aligned(x, 16) || !aligned(W_r, 16) || !aligned(bias, 4) || !aligned(idx, 4) || !aligned(w, 4) ||
        (keff && !aligned(keff, 4)) || (counts && !aligned(counts, 4)) ||
        (offsets && !aligned(offsets, 4)) || (perm && !aligned(perm, 4)))
        return COLI_MOE_EALIGN;
    if ((rc = check_ws(desc, ws, ws_bytes))) return rc;
    if ((rc = check_device())) return rc;
    const bool buckets = counts || offsets || perm;
    return run_route(desc, x, W_r, bias, idx, w, keff, counts, offsets, perm, buckets, ws,
                     reinterpret_cast<cudaStream_t>(stream));
}

int coli_moe_forward(const coli_moe_desc *desc, const float *x, const float *W_r, const float *bias,
                     const coli_moe_expert *experts, const coli_moe_expert *shared, float *out,
                     int32_t *idx_out, float *w_out, void *ws, size_t ws_bytes, coli_stream_t stream) {
    int rc = validate_forward(desc, x, W_r, bias, experts, shared, out, ws, ws_bytes);
    if (rc) return rc;
    if (!aligned(x, 16) || !aligned(out, 16) || (idx_out && !aligned(idx_out, 4)) ||
        (w_out && !aligned(w_out, 4)))
        return COLI_MOE_EALIGN;
    if ((rc = check_device())) return rc;
    return run_forward(desc, x, W_r, bias, experts, shared, out, idx_out, w_out, ws,
                       reinterpret_cast<cudaStream_t>(stream));
}

int coli_moe_forward_profiled(const coli_moe_desc *desc, const float *x, const float *W_r,
                              const float *bias, const coli_moe_expert *experts,
                              const coli_moe_expert *shared, float *out, void *const *events,
                              int n_events, void *ws, size_t ws_bytes, coli_stream_t stream) {
    int rc = validate_forward(desc, x, W_r, bias, experts, shared, out, ws, ws_bytes);
    if (rc) return rc;
    if (!events || n_events != 5) return COLI_MOE_EINVAL;
    for (int i = 0; i < 5; i++)
        if (!events[i]) return COLI_MOE_EINVAL;
    if (!aligned(x, 16) || !aligned(out, 16)) return COLI_MOE_EALIGN;
    if ((rc = check_device())) return rc;
    return run_forward(desc, x, W_r, bias, experts, shared, out, nullptr, nullptr, ws,
                       reinterpret_cast<cudaStream_t>(stream), events);
}

int coli_moe_forward_tail(const coli_moe_desc *desc, const float *resid, const float *norm_w, float eps,
                          const float *W_r, const float *bias, const coli_moe_expert *experts,
                          const coli_moe_expert *shared, float *out, int32_t *idx_out, float *w_out, void *ws,
                          size_t ws_bytes, coli_stream_t stream) {
    int rc = validate_forward(desc, resid, W_r, bias, experts, shared, out, ws, ws_bytes);
    if (rc) return rc;
    if (!norm_w || !std::isfinite(eps) || eps < 0.f) return COLI_MOE_EINVAL;
    if (!aligned(resid, 16) || !aligned(out, 16) || !aligned(norm_w, 16) || (idx_out && !aligned(idx_out, 4)) ||
        (w_out && !aligned(w_out, 4)))
        return COLI_MOE_EALIGN;
    if ((rc = check_device())) return rc;
    const Tail tail{resid, norm_w, eps};
    return run_forward(desc, resid, W_r, bias, experts, shared, out, idx_out, w_out, ws,
                       reinterpret_cast<cudaStream_t>(stream), nullptr, &tail);
}

int coli_moe_rmsnorm(const float *resid, const float *norm_w, float eps, float *xn, int32_t T, int32_t H,
                     coli_stream_t stream) {
    if (!resid || !norm_w || !xn || T < 1 || H < 4 || H > kMaxDim || T > kMaxT || !std::isfinite(eps) || eps < 0.f)
        return COLI_MOE_EINVAL;
    if (H % 4) return COLI_MOE_ENOTSUP;
    if (!aligned(resid, 16) || !aligned(norm_w, 16) || !aligned(xn, 16)) return COLI_MOE_EALIGN;
    int rc = check_device();
    if (rc) return rc;
    cudaError_t e = launch_rmsnorm(resid, norm_w, eps, T, H, xn, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? COLI_MOE_OK : cuda_fail(e);
}

int coli_moe_forward_host(const coli_moe_desc *desc, const float *x_host, const float *W_r,
                          const float *bias, const coli_moe_expert *experts,
                          const coli_moe_expert *shared, float *out_host, void *ws, size_t ws_bytes,
                          coli_stream_t stream) {
    int rc = validate_forward(desc, x_host, W_r, bias, experts, shared, out_host, ws, ws_bytes);
    if (rc) return rc;
    if ((rc = check_device())) return rc;
    const WsLayout L = ws_layout(*desc);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    float *xd = ws_ptr<float>(ws, L.xstage);
    float *od = ws_ptr<float>(ws, L.ostage);
    const size_t bytes = (size_t)desc->T * desc->H * sizeof(float);
    cudaError_t e = cudaMemcpyAsync(xd, x_host, bytes, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return cuda_fail(e);
    if ((rc = run_forward(desc, xd, W_r, bias, experts, shared, od, nullptr, nullptr, ws, st))) return rc;
    if ((e = cudaMemcpyAsync(out_host, od, bytes, cudaMemcpyDeviceToHost, st)) != cudaSuccess)
        return cuda_fail(e);
    if ((e = cudaStreamSynchronize(st)) != cudaSuccess) return cuda_fail(e);
    return COLI_MOE_OK;
}

int coli_moe_qgemv(int32_t fmt, const void *W, const float *s, const float *x, float *y, int32_t O,
                   int32_t In, int32_t T, coli_stream_t stream) {
    int rc = check_fmt(fmt);
    if (rc) return rc;
    if (fmt == COLI_FMT_INT4G) return COLI_MOE_ENOTSUP;  // needs the group size: coli_moe_qgemv_grouped
    if (!W || !s || !x || !y || O < 1 || In < 1 || T < 1 || O > (1 << 24) || In > kMaxDim ||
        T > (1 << 24))
        return COLI_MOE_EINVAL;
    if (In % elems_per_chunk(fmt)) return COLI_MOE_ENOTSUP;
    if (!aligned(W, 16) || !aligned(s, 4) || !aligned(x, 4) || !aligned(y, 4)) return COLI_MOE_EALIGN;
    if ((rc = check_device())) return rc;
    cudaError_t e = launch_qgemv(fmt, W, s, 0, x, y, O, In, T, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? COLI_MOE_OK : cuda_fail(e);
}

int coli_moe_qgemv_grouped(const void *W, const float *s, int32_t group_size, const float *x, float *y,
                           int32_t O, int32_t In, int32_t T, coli_stream_t stream) {
    if (!W || !s || !x || !y || O < 1 || In < 1 || T < 1 || O > (1 << 24) || In > kMaxDim ||
        T > (1 << 24) || !group_size_ok(group_size))
        return COLI_MOE_EINVAL;
    if (In % elems_per_chunk(COLI_FMT_INT4G)) return COLI_MOE_ENOTSUP;
    if (!aligned(W, 16) || !aligned(s, 4) || !aligned(x, 4) || !aligned(y, 4)) return COLI_MOE_EALIGN;
    int rc = check_device();
    if (rc) return rc;
    cudaError_t e = launch_qgemv(COLI_FMT_INT4G, W, s, group_size, x, y, O, In, T,
                                 reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? COLI_MOE_OK : cuda_fail(e);
}

int coli_moe_check(void *ws, coli_stream_t stream) {
    if (!ws) return COLI_MOE_EWORKSPACE;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    int32_t word = 0;
    cudaError_t e = cudaMemcpyAsync(&word, ws, sizeof(word), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e);
    if (word == 0) return COLI_MOE_OK;
    const int32_t zero = 0;
    e = cudaMemcpyAsync(ws, &zero, sizeof(zero), cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e);
    return COLI_MOE_EKERNEL;
}

const char *coli_moe_strerror(int code) {
    switch (code) {
    case COLI_MOE_OK: return "ok";
    case COLI_MOE_EINVAL: return "invalid argument (null pointer or out-of-range size/option)";
    case COLI_MOE_ENOTSUP: return "not supported (weight format or dimension granule)";
    case COLI_MOE_EALIGN: return "pointer or row stride not aligned (16 bytes)";
    case COLI_MOE_EWORKSPACE: return "workspace missing, misaligned (256 bytes) or too small";
    case COLI_MOE_ECUDA: return "CUDA runtime error (see coli_moe_last_cuda_error)";
    case COLI_MOE_EDEVICE: return "current device is not compute capability 10.3 (GB300)";
    case COLI_MOE_EKERNEL: return "a kernel flagged an error (no selectable expert, bad expert id or pointer, or an expired wait)";
    default: return "unknown error code";
    }
}

int coli_moe_last_cuda_error(void) { return g_last_cuda; }

}  // extern "C"

// ---------------------------------------------------------------- no-allocation forward
// Scratch of coli_moe_forward_noalloc: a fixed array in this module's device image, so a
// caller that cannot allocate device memory can still run the block. Host code never uses the
// name as an address (on the host it is only a stand-in for the symbol); the device address
// is looked up once per device with cudaGetSymbolAddress while that device is current.
static __device__ __align__(256) unsigned char g_noalloc_scratch[COLI_MOE_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kNoallocDevices = 64;
std::mutex g_noalloc_mu;
void *g_noalloc_ptr[kNoallocDevices];

int noalloc_scratch(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kNoallocDevices) return COLI_MOE_ENOTSUP;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail(e);
        if (!p) return COLI_MOE_EWORKSPACE;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return COLI_MOE_OK;
}
}  // namespace

extern "C" int coli_moe_forward_noalloc(const coli_moe_desc *desc, const float *x,
                                        const float *W_r, const float *bias,
                                        const coli_moe_expert *experts,
                                        const coli_moe_expert *shared, float *out,
                                        coli_stream_t stream) {
    int rc = validate_desc(desc);
    if (rc) return rc;
    if (ws_layout(*desc).total > COLI_MOE_NOALLOC_SCRATCH_BYTES) return COLI_MOE_EWORKSPACE;
    if ((rc = check_device())) return rc;
    void *ws = nullptr;
    if ((rc = noalloc_scratch(&ws))) return rc;
    return coli_moe_forward(desc, x, W_r, bias, experts, shared, out, nullptr, nullptr, ws,
                            COLI_MOE_NOALLOC_SCRATCH_BYTES, stream);
}

// the error word is the first int32 of the array, as of every workspace
extern "C" int coli_moe_noalloc_check(coli_stream_t stream) {
    int rc = check_device();
    if (rc) return rc;
    void *ws = nullptr;
    if ((rc = noalloc_scratch(&ws))) return rc;
    return coli_moe_check(ws, stream);
}
