// decode.cu — the whole MoE block for decode-sized batches (T <= 64) in ONE persistent launch.
//
// Work is a list of items, each CTA taking a static share (see Producer::run):
//   router items       logits of 32 experts over one slice of H, for T <= 8 tokens
//                      (colibri-strix c/glm.c @98759bf moe() phase A; r_router shader)
//   shared gate/up     8 rows of the shared expert's gate and up (phase E)
//   routed gate/up     8 rows of one selected expert's gate and up, for up to NV tokens
//                      (phases C/D: g = gate.x, u = up.x, h = silu(g)*u; moe_gemv + moe_silu)
//   down               each CTA owns a slice of the H output rows: for every selected expert
//                      and the shared one it computes its rows of y = down.h into shared
//                      memory, then combines them in selection order plus the shared expert
//                      and writes out (phases C/D/E) — no atomics, no global y
// The item ids of routed work are only known after routing: the CTA that finishes the last
// router item (an atomic ticket) runs the top-K selection (r_top8_par's lane-blocked warp
// argmax, ties to the lower index, TOPK/TOPP, renorm, routed scale), the token->expert
// buckets and the item table, then publishes a flag.
//
// Each CTA has 8 consumer warps and 1 producer warp. The producer claims items and streams
// their weights into a ring of 16 KB shared-memory stages with bulk asynchronous copies
// (cp.async.bulk, completion counted on an mbarrier per stage); consumers dequantise from
// shared memory (qdot.cuh) against activations staged, pre-scaled and permuted, in shared
// memory. Dependencies (routing -> routed work, an expert's gate/up -> its down) are counters
// in the workspace, raised once per CTA per expert. Every
// CTA finishes all of its earlier-phase items before it waits on a later phase, and the launch
// is cooperative (all CTAs resident), so progress is guaranteed; every wait is still bounded
// (2 s of %globaltimer), after which the kernel records kErrWaitExpired and goes on without
// blocking the GPU.
#include <algorithm>

#include "kernels.h"
#include "ptx.cuh"
#include "qdot.cuh"

namespace colimoe {

namespace {

constexpr int kCW = 8;                          // consumer warps
constexpr int kCT = kCW * kWarp;                // consumer threads
constexpr int kDecThreads = kCT + kWarp;        // + one producer warp
constexpr int kSB = 16384;                      // bytes per ring stage
constexpr int kGuPairs = 8;                     // gate/up row pairs per item (one per consumer warp)
constexpr int kGuKc = kSB / (2 * kGuPairs);     // 1024 bytes of each row per stage
constexpr int kRtE = 32;                        // experts per router item (4 per consumer warp)
constexpr int kRtKc = kSB / kRtE;               // 512 bytes (128 floats) of each W_r row per stage
constexpr int kRtStages = 4;                    // stages per router item
constexpr unsigned long long kWaitNs = 2000000000ull;
constexpr int kSharedSlotKey = kMaxE;           // gu_done index of the shared expert

enum Kind : int { kEnd = 0, kRouter = 1, kGateUp = 2, kDown = 3, kRouteOnly = 4 };

// What the consumers need about the expert of an item (filled in by the producer, so that
// consumers make no global lookups per item).
struct ItemSlot {
    const float *s0, *s1;  // gate/up: gate and up row scales; down: down row scales
    int fmt, inter;        // weight format, intermediate size of this expert
    int n, pbase;          // tokens using it, first bucket position (routed)
    int key;               // gu_done index: routed slot, or kSharedSlotKey
    int need;              // gate/up items of this expert that its down work waits for
    int shared;
};

struct StageDesc {
    int kind;
    int sidx, nst;   // stage index in the item, stages in the item
    int slot;        // routed slot (0..U-1) or U = shared; router: expert block
    int rb;          // row block (gate/up: 8 pairs, down: 64 rows); router: k-slice
    int tg;          // token group
    int row0, nrows; // rows carried by this stage (gate/up: pairs; down: rows; router: experts)
    int k0, kbytes;  // byte range of each row carried (gate/up, router); down: whole rows
    int sig;         // gate/up: >0 on the last stage of this CTA's run of items of one expert
                     // (the number of items in the run, added to that expert's counter)
    ItemSlot it;
};

__device__ __forceinline__ void flag_error(DecCtrl *c, int code) { atomicCAS(&c->err, 0, code); }

// bounded wait until *p >= target; returns false (and flags) on timeout
__device__ bool wait_at_least(const int *p, int target, DecCtrl *c) {
    if (ld_volatile(p) >= target) return true;
    const uint64_t t0 = globaltimer_ns();
    while (ld_volatile(p) < target) {
        __nanosleep(128);
        if (globaltimer_ns() - t0 > kWaitNs) {
            flag_error(c, kErrWaitExpired);
            return false;
        }
    }
    return true;
}

__device__ bool mbar_wait(uint64_t *bar, uint32_t parity, DecCtrl *c) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > kWaitNs) {
            flag_error(c, kErrWaitExpired);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ void consumer_bar() { named_bar(1, kCT); }

// first index i in [0, n) with off[i+1] > x (off is a prefix array of length n+1)
__device__ int upper_slot(const int *off, int n, int x) {
    int lo = 0, hi = n - 1;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (__ldcg(off + mid + 1) > x) hi = mid;
        else lo = mid + 1;
    }
    return lo;
}

struct SlotInfo {
    const uint8_t *gw, *uw, *dw;
    const float *gs, *us, *ds;
    int fmt, inter, n, pbase, groups, key;
    bool shared;
};

__device__ SlotInfo slot_info(const DecParams &P, int slot, int U) {
    SlotInfo s;
    if (P.Is > 0 && slot == U) {
        s.gw = static_cast<const uint8_t *>(P.shared.gate_w);
        s.uw = static_cast<const uint8_t *>(P.shared.up_w);
        s.dw = static_cast<const uint8_t *>(P.shared.down_w);
        s.gs = P.shared.gate_s;
        s.us = P.shared.up_s;
        s.ds = P.shared.down_s;
        s.fmt = P.sfmt;
        s.inter = P.Is;
        s.n = P.T;
        s.pbase = 0;
        s.groups = P.groups_sh;
        s.key = kSharedSlotKey;
        s.shared = true;
        return s;
    }
    const DecTable *tb = P.tab;
    const int e = __ldcg(&tb->slot_e[slot]);
    const coli_moe_expert ex = P.experts[e];
    s.gw = static_cast<const uint8_t *>(ex.gate_w);
    s.uw = static_cast<const uint8_t *>(ex.up_w);
    s.dw = static_cast<const uint8_t *>(ex.down_w);
    s.gs = ex.gate_s;
    s.us = ex.up_s;
    s.ds = ex.down_s;
    s.fmt = P.rfmt;
    s.inter = P.I;
    s.n = __ldcg(&tb->slot_n[slot]);
    s.pbase = __ldcg(&tb->slot_pbase[slot]);
    s.groups = __ldcg(&tb->slot_groups[slot]);
    s.key = slot;
    s.shared = false;
    return s;
}

__device__ __forceinline__ bool bad_ptr16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

// ------------------------------------------------------------------ producer
__device__ __forceinline__ int range_lo(int n, int c, int G) { return (int)((long long)n * c / G); }

struct Producer {
    const DecParams &P;
    uint8_t *ring;
    uint64_t *full, *empty;
    StageDesc *desc;
    int lane;
    int seq = 0;

    __device__ __forceinline__ uint8_t *stage_buf(int s) { return ring + (size_t)s * kSB; }

    // wait for ring stage `seq` to be free, return its index
    __device__ __forceinline__ int acquire() {
        const int s = seq % P.nst, use = seq / P.nst;
        if (use > 0) {
            if (lane == 0) mbar_wait(&empty[s], (use - 1) & 1, P.ctrl);
            __syncwarp();
        }
        return s;
    }

    __device__ __forceinline__ void publish_end() {
        const int s = acquire();
        if (lane == 0) {
            desc[s].kind = kEnd;
            mbar_arrive(&full[s]);
        }
        __syncwarp();
        seq++;
    }

    // before the producer leaves, every copy it issued has landed (each stage's last use has
    // completed its phase), so no bulk copy is in flight when the CTA exits
    __device__ __forceinline__ void drain() {
        if (lane == 0) {
            for (int s = 0; s < P.nst && s < seq; s++) {
                const int last = s + ((seq - 1 - s) / P.nst) * P.nst;
                mbar_wait(&full[s], (last / P.nst) & 1, P.ctrl);
            }
        }
        __syncwarp();
    }

    __device__ __forceinline__ ItemSlot item_slot(const SlotInfo &si, bool down) const {
        ItemSlot it;
        it.s0 = down ? si.ds : si.gs;
        it.s1 = si.us;
        it.fmt = si.fmt;
        it.inter = si.inter;
        it.n = si.n;
        it.pbase = si.pbase;
        it.key = si.key;
        it.need = si.shared ? P.G_sh : P.gu_rb * si.groups;
        it.shared = si.shared ? 1 : 0;
        return it;
    }

    // T > 8: the logits come from an earlier launch; one item only runs the selection
    __device__ __forceinline__ void route_only_item() {
        const int s = acquire();
        if (lane == 0) {
            desc[s].kind = kRouteOnly;
            desc[s].sidx = 0;
            desc[s].nst = 1;
            mbar_arrive(&full[s]);
        }
        __syncwarp();
        seq++;
    }

    __device__ __forceinline__ void router_item(int item) {
        const int eb = item % P.neb, ks = item / P.neb;
        const int e0 = eb * kRtE;
        const int kbeg = ks * P.rks_floats;
        const int kend = min(P.H, kbeg + P.rks_floats);
        const int nst = (kend - kbeg + kRtKc / 4 - 1) / (kRtKc / 4);
        const int ne = min(kRtE, P.E - e0);
        for (int st = 0; st < nst; st++) {
            const int s = acquire();
            const int kf = kbeg + st * (kRtKc / 4);
            const int nf = min(kRtKc / 4, kend - kf);
            if (lane == 0) {
                StageDesc &d = desc[s];
                d.kind = kRouter;
                d.sidx = st;
                d.nst = nst;
                d.slot = eb;
                d.rb = ks;
                d.tg = 0;
                d.row0 = e0;
                d.nrows = ne;
                d.k0 = kf * 4;
                d.kbytes = nf * 4;
                d.sig = 0;
                mbar_arrive_expect_tx(&full[s], (uint32_t)(ne * nf * 4));
            }
            __syncwarp();
            if (lane < ne)
                bulk_g2s(stage_buf(s) + lane * kRtKc, P.Wr + (size_t)(e0 + lane) * P.H + kf, nf * 4, &full[s]);
            seq++;
        }
    }

    // 8 row pairs (gate row j, up row j) of one expert for token group tg; `sig` is set on the
    // item's last stage when it closes this CTA's run of items of that expert
    __device__ __forceinline__ void gateup_item(int slot, int rb, int tg, const SlotInfo &si, int sig) {
        const int64_t rbytes = row_bytes(si.fmt, P.H);
        const int j0 = rb * kGuPairs;
        const int np = min(kGuPairs, si.inter - j0);
        const int nst = (int)((rbytes + kGuKc - 1) / kGuKc);
        const ItemSlot it = item_slot(si, false);
        for (int st = 0; st < nst; st++) {
            const int s = acquire();
            const int k0 = st * kGuKc;
            const int kb = (int)((rbytes - k0) < kGuKc ? (rbytes - k0) : kGuKc);
            if (lane == 0) {
                StageDesc &d = desc[s];
                d.kind = kGateUp;
                d.sidx = st;
                d.nst = nst;
                d.slot = slot;
                d.rb = rb;
                d.tg = tg;
                d.row0 = j0;
                d.nrows = np;
                d.k0 = k0;
                d.kbytes = kb;
                d.sig = st == nst - 1 ? sig : 0;
                d.it = it;
                mbar_arrive_expect_tx(&full[s], (uint32_t)(2 * np * kb));
            }
            __syncwarp();
            if (lane < 2 * kGuPairs) {
                const int p = lane % kGuPairs, m = lane / kGuPairs;
                if (p < np) {
                    const uint8_t *src = (m ? si.uw : si.gw) + (size_t)(j0 + p) * rbytes + k0;
                    bulk_g2s(stage_buf(s) + (m * kGuPairs + p) * kGuKc, src, kb, &full[s]);
                }
            }
            seq++;
        }
    }

    // rows [r_lo, r_hi) of one expert's down projection for token group tg, whole rows per stage
    __device__ __forceinline__ void down_rows(int slot, int tg, int r_lo, int r_hi, const SlotInfo &si) {
        const int64_t rbytes = row_bytes(si.fmt, si.inter);
        const int64_t rfit = kSB / rbytes;
        const int rps = rfit < 1 ? 1 : (rfit > 16 ? 16 : (int)rfit);
        const int nst = (r_hi - r_lo + rps - 1) / rps;
        const ItemSlot it = item_slot(si, true);
        for (int st = 0; st < nst; st++) {
            const int s = acquire();
            const int r0 = r_lo + st * rps;
            const int nr = min(rps, r_hi - r0);
            if (lane == 0) {
                StageDesc &d = desc[s];
                d.kind = kDown;
                d.sidx = st;
                d.nst = nst;
                d.slot = slot;
                d.rb = 0;
                d.tg = tg;
                d.row0 = r0;
                d.nrows = nr;
                d.k0 = r_lo;
                d.kbytes = (int)rbytes;
                d.sig = 0;
                d.it = it;
                mbar_arrive_expect_tx(&full[s], (uint32_t)(nr * rbytes));
                bulk_g2s(stage_buf(s), si.dw + (size_t)r0 * rbytes, (uint32_t)(nr * rbytes), &full[s]);
            }
            __syncwarp();
            seq++;
        }
    }

    __device__ __forceinline__ bool slot_ok(const SlotInfo &si) {
        if (bad_ptr16(si.gw) || bad_ptr16(si.uw) || bad_ptr16(si.dw)) {
            if (lane == 0) flag_error(P.ctrl, kErrBadExpert);
            return false;
        }
        return true;
    }

    // Static schedule. CTA c takes router items c, c+G, ...; its contiguous share of the shared
    // expert's gate/up items; after routing, its contiguous share of the routed gate/up items;
    // then its slice of the H down-projection rows for every expert. Each phase finishes in a CTA
    // before it waits on the next, and all CTAs are resident (cooperative launch), so every wait
    // is on work some running CTA reaches first.
    __device__ __forceinline__ void run() {
        const int G = gridDim.x, c = blockIdx.x;
        for (int r = c; r < P.R; r += G) {
            if (P.route_only) route_only_item();
            else router_item(r);
        }
        if (P.G_sh > 0) {
            const int b = range_lo(P.G_sh, c, G), e = range_lo(P.G_sh, c + 1, G);
            const SlotInfo si = slot_info(P, 0, 0);
            for (int l = b; l < e; l++)
                gateup_item(-1, l % P.G_sh_rb, l / P.G_sh_rb, si, l == e - 1 ? e - b : 0);
        }
        int ready = 1;
        if (lane == 0) ready = wait_at_least(&P.ctrl->routing_ready, 1, P.ctrl) ? 1 : 0;
        ready = __shfl_sync(kFull, ready, 0);
        __threadfence();
        if (ready) {
            const DecTable *tb = P.tab;
            const int U = __ldcg(&tb->U);
            const int gu_tot = __ldcg(&tb->gu_off[U]);
            const int b = range_lo(gu_tot, c, G), e = range_lo(gu_tot, c + 1, G);
            if (b < e) {
                int slot = upper_slot(tb->gu_off, U, b);
                int lo = __ldcg(&tb->gu_off[slot]), hi = __ldcg(&tb->gu_off[slot + 1]);
                SlotInfo si = slot_info(P, slot, U);
                bool ok = slot_ok(si);
                int run_start = b;
                for (int l = b; l < e; l++) {
                    while (l >= hi) {
                        slot++;
                        lo = hi;
                        hi = __ldcg(&tb->gu_off[slot + 1]);
                        si = slot_info(P, slot, U);
                        ok = slot_ok(si);
                        run_start = l;
                    }
                    if (!ok) continue;
                    const int ll = l - lo;
                    const bool run_end = (l == e - 1) || (l + 1 >= hi);
                    gateup_item(slot, ll % P.gu_rb, ll / P.gu_rb, si, run_end ? l + 1 - run_start : 0);
                }
            }
            // this CTA's rows of every expert's down projection (routed slots, then shared)
            const int r_lo = range_lo(P.H, c, G), r_hi = range_lo(P.H, c + 1, G);
            const int nslots = U + (P.Is > 0 ? 1 : 0);
            if (r_lo < r_hi) {
                for (int slot = 0; slot < nslots; slot++) {
                    const SlotInfo si = slot_info(P, slot, U);
                    if (!slot_ok(si)) continue;
                    for (int tg = 0; tg < si.groups; tg++) down_rows(slot, tg, r_lo, r_hi, si);
                }
            }
        }
        publish_end();
        drain();
    }
};

// ------------------------------------------------------------------ routing (one CTA)
template <int PER>
__device__ void select_token(const DecParams &P, int t, int lane, int nks) {
    const int base = lane * PER;
    float ch[PER], sg[PER];
#pragma unroll
    for (int j = 0; j < PER; j++) {
        const int e = base + j;
        if (e < P.E) {
            float lg = 0.f;
            for (int s = 0; s < nks; s++) lg += __ldcg(P.part + ((size_t)s * P.T + t) * P.E + e);
            const float sv = 1.f / (1.f + expf(-lg));
            const float cv = sv + P.bias[e];
            P.sig[(size_t)t * P.E + e] = sv;
            P.choice[(size_t)t * P.E + e] = cv;
            sg[j] = sv;
            ch[j] = cv;
        } else {
            sg[j] = 0.f;
            ch[j] = -INFINITY;
        }
    }
    uint32_t taken = 0;
    int nsel = 0, my_i = -1;
    float my_w = 0.f;
    for (int k = 0; k < P.Ksel; k++) {
        float bv = -1e30f, bs = 0.f;
        int bi = 0x7fffffff;
#pragma unroll
        for (int j = 0; j < PER; j++)
            if (!((taken >> j) & 1u) && ch[j] > bv) {
                bv = ch[j];
                bi = base + j;
                bs = sg[j];
            }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_down_sync(kFull, bv, o);
            const int oi = __shfl_down_sync(kFull, bi, o);
            const float os = __shfl_down_sync(kFull, bs, o);
            if (ov > bv || (ov == bv && oi < bi)) {
                bv = ov;
                bi = oi;
                bs = os;
            }
        }
        bi = __shfl_sync(kFull, bi, 0);
        bs = __shfl_sync(kFull, bs, 0);
        if (bi == 0x7fffffff) {
            if (lane == 0) flag_error(P.ctrl, kErrNoCandidate);
            break;
        }
        if (bi >= base && bi < base + PER) taken |= 1u << (bi - base);
        if (lane == k) {  // lane k keeps selection k
            my_i = bi;
            my_w = bs;
        }
        nsel = k + 1;
    }
    // tail on lane 0 with the pages' float operations and order (TOPP, renorm, scale)
    float ww[kMaxK];
    int id[kMaxK];
    for (int k = 0; k < nsel; k++) {
        ww[k] = __shfl_sync(kFull, my_w, k);
        id[k] = __shfl_sync(kFull, my_i, k);
    }
    if (lane != 0) return;
    int Ke = nsel;
    if (P.top_p > 0.f && P.top_p < 1.f) {
        for (int a = 1; a < nsel; a++) {
            const int ia = id[a];
            const float wa = ww[a];
            int b = a - 1;
            while (b >= 0 && ww[b] < wa) {
                ww[b + 1] = ww[b];
                id[b + 1] = id[b];
                b--;
            }
            ww[b + 1] = wa;
            id[b + 1] = ia;
        }
        float tot = 1e-20f;
        for (int k = 0; k < nsel; k++) tot = __fadd_rn(tot, ww[k]);
        float cum = 0.f;
        for (int k = 0; k < nsel; k++) {
            cum = __fadd_rn(cum, ww[k]);
            if (cum >= __fmul_rn(P.top_p, tot)) {
                Ke = k + 1;
                break;
            }
        }
    }
    if (P.norm_topk) {
        float sm = 0.f;
        for (int k = 0; k < Ke; k++) sm = __fadd_rn(sm, ww[k]);
        sm = __fadd_rn(sm, 1e-20f);
        for (int k = 0; k < Ke; k++) ww[k] = __fdiv_rn(ww[k], sm);
    }
    for (int k = 0; k < P.K; k++) {
        const bool kept = k < Ke;
        P.idx[(size_t)t * P.K + k] = kept ? id[k] : -1;
        P.w[(size_t)t * P.K + k] = kept ? __fmul_rn(ww[k], P.rscale) : 0.f;
    }
    P.keff[t] = Ke;
}

// exclusive scan of n <= 1024 ints held in shared memory, in place, by the 256 consumer threads;
// returns the total
__device__ int scan_smem(int *a, int n, int *tmp /* >= 9 ints */) {
    const int tid = threadIdx.x, lane = tid % kWarp, warp = tid / kWarp;
    int loc[8], sum = 0;  // n <= 2048
#pragma unroll
    for (int i = 0; i < 8; i++) {
        const int j = tid * 8 + i;
        loc[i] = j < n ? a[j] : 0;
        sum += loc[i];
    }
    int inc = sum;
#pragma unroll
    for (int o = 1; o < kWarp; o <<= 1) {
        const int v = __shfl_up_sync(kFull, inc, o);
        if (lane >= o) inc += v;
    }
    if (lane == kWarp - 1) tmp[warp] = inc;
    consumer_bar();
    if (tid == 0) {
        int run = 0;
        for (int w = 0; w < kCW; w++) {
            const int v = tmp[w];
            tmp[w] = run;
            run += v;
        }
        tmp[kCW] = run;
    }
    consumer_bar();
    int run = tmp[warp] + inc - sum;
#pragma unroll
    for (int i = 0; i < 8; i++) {
        const int j = tid * 8 + i;
        if (j < n) a[j] = run;
        run += loc[i];
    }
    const int total = tmp[kCW];
    consumer_bar();
    return total;
}

__device__ void route_final(const DecParams &P, int *scr) {
    const int tid = threadIdx.x, lane = tid % kWarp, warp = tid / kWarp;
    const int per = (P.E + kWarp - 1) / kWarp;
    for (int t = warp; t < P.T; t += kCW) {
        if (per <= 1) select_token<1>(P, t, lane, P.nks);
        else if (per <= 2) select_token<2>(P, t, lane, P.nks);
        else if (per <= 4) select_token<4>(P, t, lane, P.nks);
        else if (per <= 8) select_token<8>(P, t, lane, P.nks);
        else if (per <= 16) select_token<16>(P, t, lane, P.nks);
        else select_token<32>(P, t, lane, P.nks);
    }
    consumer_bar();  // the buckets below read idx/keff through L2 (ld.cg) in the same CTA
    if (tid == 0) __threadfence();
    consumer_bar();
    // buckets: counts, offsets, active list, stable perm / pos
    const int E = P.E, N = P.T * P.K;
    int *cnt = scr, *off = cnt + E, *fill = off + E, *chk = fill + E, *actv = chk + E;
    int *wc = actv + E, *tmp = wc + kCW * E;
    for (int e = tid; e < E; e += kCT) {
        cnt[e] = 0;
        fill[e] = 0;
    }
    consumer_bar();
    auto expert_of = [&](int a) -> int {
        if (a >= N) return -1;
        const int t = a / P.K, k = a % P.K;
        if (k >= __ldcg(P.keff + t)) return -1;
        return __ldcg(P.idx + a);
    };
    for (int a = tid; a < N; a += kCT) {
        const int e = expert_of(a);
        if (e >= 0) atomicAdd(&cnt[e], 1);
    }
    consumer_bar();
    for (int e = tid; e < E; e += kCT) {
        off[e] = cnt[e];
        actv[e] = cnt[e] > 0 ? 1 : 0;
        P.counts[e] = cnt[e];
    }
    consumer_bar();
    const int total = scan_smem(off, E, tmp);
    const int U = scan_smem(actv, E, tmp);
    for (int e = tid; e < E; e += kCT) {
        P.offsets[e] = off[e];
        if (cnt[e] > 0) P.act[actv[e]] = e;
    }
    if (tid == 0) P.offsets[E] = total;
    consumer_bar();
    for (int a0 = 0; a0 < N; a0 += kCT) {
        for (int i = tid; i < kCW * E; i += kCT) wc[i] = 0;
        consumer_bar();
        const int a = a0 + tid;
        const int e = expert_of(a);
        const unsigned peers = __match_any_sync(kFull, e);
        const int rank = __popc(peers & ((1u << lane) - 1u));
        if (e >= 0 && rank == 0) wc[warp * E + e] = __popc(peers);
        consumer_bar();
        for (int x = tid; x < E; x += kCT) {
            int run = 0;
            for (int w = 0; w < kCW; w++) {
                const int v = wc[w * E + x];
                wc[w * E + x] = run;
                run += v;
            }
            chk[x] = run;
        }
        consumer_bar();
        if (a < N) {
            if (e >= 0) {
                const int p = off[e] + fill[e] + wc[warp * E + e] + rank;
                P.perm[p] = a;
                P.pos[a] = p;
            } else {
                P.pos[a] = -1;
            }
        }
        consumer_bar();
        for (int x = tid; x < E; x += kCT) fill[x] += chk[x];
        consumer_bar();
    }
    // item table: slots 0..U-1 routed (ascending expert id), slot U shared
    DecTable *tb = P.tab;
    const bool sh = P.Is > 0;
    int *gu = wc;  // reuse: per-slot gate/up item counts, scanned
    for (int u = tid; u < U + 1; u += kCT) {
        int g = 0;
        if (u < U) {
            const int e = __ldcg(P.act + u);
            const int n = cnt[e];
            g = (n + P.NV - 1) / P.NV;
            tb->slot_e[u] = e;
            tb->slot_n[u] = n;
            tb->slot_pbase[u] = off[e];
            tb->slot_groups[u] = g;
        }
        gu[u] = u < U ? P.gu_rb * g : 0;
    }
    consumer_bar();
    const int gu_tot = scan_smem(gu, U + 1, tmp);
    for (int u = tid; u < U + 1; u += kCT) tb->gu_off[u] = gu[u];
    if (tid == 0) {
        tb->gu_off[U + 1] = gu_tot;
        tb->U = U;
    }
    consumer_bar();
    if (tid == 0) {
        __threadfence();
        atomicExch(&P.ctrl->routing_ready, 1);
    }
}

// ------------------------------------------------------------------ consumers
struct Consumer {
    const DecParams &P;
    uint8_t *ring;
    uint64_t *full, *empty;
    StageDesc *desc;
    float *xs;     // activation staging / routing scratch
    float *ybuf;   // this CTA's rows of y: [T*K + T][rows_cta]
    int *sflag;    // shared flag word
    int tid, lane, warp;
    int seq = 0;
    int key0 = -1, key1 = -1, key2 = -1;  // what XS currently holds (kind, slot/bucket, group)
    float2 acc[2][4];
    float racc[4][8];

    // activations of token group tg of the item's expert, staged pre-scaled and permuted for
    // its format (x for gate/up, h for down); skipped when XS already holds them
    __device__ __forceinline__ void stage_acts(const ItemSlot &it, int tg, bool down) {
        const int k0 = down ? 2 : 1;
        const int k1 = down ? it.key : (P.T == 1 ? 0 : (it.shared ? -1 : it.pbase));
        const int k2 = (P.T == 1 && !down) ? it.fmt : tg * 8 + it.fmt;
        if (key0 == k0 && key1 == k1 && key2 == k2) return;
        const int nv = min(P.NV, it.n - tg * P.NV);
        const int len = down ? it.inter : P.H;
        const int gran = it.fmt == COLI_FMT_INT4 ? 32 : it.fmt == COLI_FMT_INT8 ? 16 : 64;
        const int CPR = len / gran;
        consumer_bar();
        for (int v = 0; v < P.NV; v++) {
            float *dst = xs + (size_t)v * P.xs_stride;
            if (v < nv) {
                const int pv = tg * P.NV + v;
                const float *src;
                if (down) {
                    const int row = it.shared ? P.T * P.K + pv : it.pbase + pv;
                    src = P.h + (size_t)row * P.ldh;
                } else {
                    const int t = it.shared ? pv : __ldcg(P.perm + it.pbase + pv) / P.K;
                    src = P.x + (size_t)t * P.H;
                }
                for (int i = tid; i < len; i += kCT) {
                    float sc;
                    int at;
                    if (it.fmt == COLI_FMT_INT4) at = staged_index<COLI_FMT_INT4>(i, CPR, sc);
                    else if (it.fmt == COLI_FMT_INT8) at = staged_index<COLI_FMT_INT8>(i, CPR, sc);
                    else at = staged_index<COLI_FMT_INT2>(i, CPR, sc);
                    dst[at] = (down ? __ldcg(src + i) : __ldg(src + i)) * sc;
                }
            } else {
                for (int i = tid; i < len; i += kCT) dst[i] = 0.f;
            }
        }
        key0 = k0;
        key1 = k1;
        key2 = k2;
        consumer_bar();
    }

    // ---------------- router stage: 4 experts per warp, up to 8 tokens, one float4 per lane
    __device__ __forceinline__ void router_stage(const StageDesc &d, const uint8_t *buf) {
        if (d.sidx == 0) {
#pragma unroll
            for (int r = 0; r < 4; r++)
#pragma unroll
                for (int t = 0; t < 8; t++) racc[r][t] = 0.f;
        }
        const int nf4 = d.kbytes / 16;
        const int kf = d.k0 / 4 + lane * 4;
        if (lane < nf4) {
            float4 wv[4];
#pragma unroll
            for (int r = 0; r < 4; r++) {
                const int er = warp * 4 + r;
                wv[r] = er < d.nrows ? *reinterpret_cast<const float4 *>(buf + er * kRtKc + lane * 16)
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int t = 0; t < 8; t++) {
                if (t >= P.T) break;
                const float4 xv = __ldg(reinterpret_cast<const float4 *>(P.x + (size_t)t * P.H + kf));
#pragma unroll
                for (int r = 0; r < 4; r++) {
                    float a = racc[r][t];
                    a = fmaf(wv[r].x, xv.x, a);
                    a = fmaf(wv[r].y, xv.y, a);
                    a = fmaf(wv[r].z, xv.z, a);
                    a = fmaf(wv[r].w, xv.w, a);
                    racc[r][t] = a;
                }
            }
        }
    }

    __device__ __forceinline__ void router_finish(const StageDesc &d) {
        // d.slot = expert block, d.rb = k-slice
#pragma unroll
        for (int r = 0; r < 4; r++)
#pragma unroll
            for (int t = 0; t < 8; t++) {
                if (t >= P.T) break;
                float s = racc[r][t];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(kFull, s, o);
                const int e = d.row0 + warp * 4 + r;
                if (lane == 0 && warp * 4 + r < d.nrows) P.part[((size_t)d.rb * P.T + t) * P.E + e] = s;
            }
        consumer_bar();
        if (tid == 0) {
            __threadfence();
            const bool lastone = atomicAdd(&P.ctrl->router_done, 1) == P.R - 1;
            if (lastone) __threadfence();
            *sflag = lastone;
        }
        consumer_bar();
        const bool last = *sflag;
        consumer_bar();
        if (last) {
            route_final(P, reinterpret_cast<int *>(xs));
            key0 = -1;
        }
    }

    // ---------------- gate/up stages: warp w owns row pair w (gate row, up row)
    template <int FMT, int NV>
    __device__ __forceinline__ void gateup_stage_t(const StageDesc &d, const uint8_t *buf) {
        if (warp >= d.nrows) return;
        const uint8_t *rows[2] = {buf + warp * kGuKc, buf + (kGuPairs + warp) * kGuKc};
        float2 a[2][NV];
#pragma unroll
        for (int r = 0; r < 2; r++)
#pragma unroll
            for (int v = 0; v < NV; v++) a[r][v] = acc[r][v];
        qdot_smem_acc<FMT, 2, NV>(rows, d.k0 / 16, d.kbytes / 16, xs, P.xs_stride, P.H / QGeom<FMT>::EPC,
                                  lane, a);
#pragma unroll
        for (int r = 0; r < 2; r++)
#pragma unroll
            for (int v = 0; v < NV; v++) acc[r][v] = a[r][v];
    }

    template <int NV>
    __device__ __forceinline__ void gateup_finish_t(const StageDesc &d) {
        float2 a[2][NV];
#pragma unroll
        for (int r = 0; r < 2; r++)
#pragma unroll
            for (int v = 0; v < NV; v++) a[r][v] = acc[r][v];
        float sum[2][NV];
        warp_reduce_acc<2, NV>(a, sum);
        const ItemSlot &it = d.it;
        const int j = d.row0 + warp;
        const int nv = min(P.NV, it.n - d.tg * P.NV);
        if (warp < d.nrows) {
#pragma unroll
            for (int v = 0; v < NV; v++) {
                if (lane == v && v < nv) {
                    const float g = sum[0][v] * it.s0[j];
                    const float u = sum[1][v] * it.s1[j];
                    const int pv = d.tg * P.NV + v;
                    const int row = it.shared ? P.T * P.K + pv : it.pbase + pv;
                    P.h[(size_t)row * P.ldh + j] = g / (1.f + expf(-g)) * u;
                }
            }
        }
    }

    // ---------------- down stages: each warp owns whole rows of the stage; y goes to ybuf
    template <int FMT, int NV>
    __device__ __forceinline__ void down_stage_t(const StageDesc &d, const uint8_t *buf) {
        const ItemSlot &it = d.it;
        const int rbytes = d.kbytes;
        const int CPR = it.inter / QGeom<FMT>::EPC;
        const int nv = min(P.NV, it.n - d.tg * P.NV);
        for (int r = warp; r < d.nrows; r += kCW) {
            const uint8_t *rows[1] = {buf + r * rbytes};
            float2 a[1][NV];
#pragma unroll
            for (int v = 0; v < NV; v++) a[0][v] = make_float2(0.f, 0.f);
            qdot_smem_acc<FMT, 1, NV>(rows, 0, CPR, xs, P.xs_stride, CPR, lane, a);
            float sum[1][NV];
            warp_reduce_acc<1, NV>(a, sum);
            const int dd = d.row0 + r;
#pragma unroll
            for (int v = 0; v < NV; v++) {
                if (lane == v && v < nv) {
                    const int pv = d.tg * P.NV + v;
                    const int row = it.shared ? P.T * P.K + pv : it.pbase + pv;
                    ybuf[(size_t)row * P.rows_cta + (dd - d.k0)] = sum[0][v] * it.s0[dd];
                }
            }
        }
    }

    // out rows of this CTA's slice: selection order, then the shared expert
    __device__ __forceinline__ void combine_rows() {
        const int G = gridDim.x, c = blockIdx.x;
        const int r_lo = range_lo(P.H, c, G), r_hi = range_lo(P.H, c + 1, G);
        const int nd = r_hi - r_lo;
        consumer_bar();
        for (int i = tid; i < P.T * nd; i += kCT) {
            const int t = i / nd, rr = i % nd;
            const int ke = __ldcg(P.keff + t);
            float a = 0.f;
            for (int k = 0; k < ke; k++) {
                const float wk = __ldcg(P.w + (size_t)t * P.K + k);
                const int p = __ldcg(P.pos + (size_t)t * P.K + k);
                a = __fadd_rn(a, __fmul_rn(wk, ybuf[(size_t)p * P.rows_cta + rr]));
            }
            if (P.Is > 0) a = __fadd_rn(a, ybuf[((size_t)P.T * P.K + t) * P.rows_cta + rr]);
            P.out[(size_t)t * P.H + r_lo + rr] = a;
        }
    }

    template <int NV>
    __device__ __forceinline__ void process_nv(const StageDesc &d, const uint8_t *buf) {
        const int fmt = d.it.fmt;
        if (d.kind == kGateUp) {
            if (d.sidx == 0) {
#pragma unroll
                for (int r = 0; r < 2; r++)
#pragma unroll
                    for (int v = 0; v < 4; v++) acc[r][v] = make_float2(0.f, 0.f);
            }
            if (fmt == COLI_FMT_INT4) gateup_stage_t<COLI_FMT_INT4, NV>(d, buf);
            else if (fmt == COLI_FMT_INT8) gateup_stage_t<COLI_FMT_INT8, NV>(d, buf);
            else gateup_stage_t<COLI_FMT_INT2, NV>(d, buf);
        } else {
            if (fmt == COLI_FMT_INT4) down_stage_t<COLI_FMT_INT4, NV>(d, buf);
            else if (fmt == COLI_FMT_INT8) down_stage_t<COLI_FMT_INT8, NV>(d, buf);
            else down_stage_t<COLI_FMT_INT2, NV>(d, buf);
        }
    }

    __device__ __forceinline__ void run() {
        bool did_down = false;
        for (;;) {
            const int s = seq % P.nst, use = seq / P.nst;
            if (!mbar_wait(&full[s], use & 1, P.ctrl)) break;  // flagged; the producer drains
            const StageDesc d = desc[s];
            if (d.kind == kEnd) break;
            const uint8_t *buf = ring + (size_t)s * kSB;
            if (d.kind == kRouteOnly) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
                seq++;
                route_final(P, reinterpret_cast<int *>(xs));
                key0 = -1;
                continue;
            }
            if (d.kind == kRouter) {
                router_stage(d, buf);
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
                seq++;
                if (d.sidx == d.nst - 1) router_finish(d);
                continue;
            }
            if (d.sidx == 0) {
                if (d.kind == kGateUp) {
                    stage_acts(d.it, d.tg, false);
                } else {
                    did_down = true;
                    // this expert's h rows must be complete before they are staged
                    if (key0 != 2 || key1 != d.it.key || key2 != d.tg * 8 + d.it.fmt) {
                        if (tid == 0) {
                            wait_at_least(&P.ctrl->gu_done[d.it.key], d.it.need, P.ctrl);
                            __threadfence();
                        }
                        consumer_bar();
                    }
                    stage_acts(d.it, d.tg, true);
                }
            }
            if (P.NV == 1) process_nv<1>(d, buf);
            else if (P.NV == 2) process_nv<2>(d, buf);
            else process_nv<4>(d, buf);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            seq++;
            if (d.kind == kGateUp && d.sidx == d.nst - 1) {
                if (P.NV == 1) gateup_finish_t<1>(d);
                else if (P.NV == 2) gateup_finish_t<2>(d);
                else gateup_finish_t<4>(d);
                if (d.sig > 0) {  // this CTA's run of items of the expert is done: publish it
                    consumer_bar();
                    if (tid == 0) {
                        __threadfence();
                        atomicAdd(&P.ctrl->gu_done[d.it.key], d.sig);
                    }
                }
            }
        }
        if (did_down) combine_rows();
    }
};

__global__ void __launch_bounds__(kDecThreads, 1) moe_decode_kernel(const DecParams P) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *ring = smem;
    float *xs = reinterpret_cast<float *>(smem + (size_t)P.nst * kSB);
    float *ybuf = reinterpret_cast<float *>(smem + (size_t)P.nst * kSB + P.xs_bytes);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)P.nst * kSB + P.xs_bytes + P.ybuf_bytes);
    uint64_t *empty = full + P.nst;
    StageDesc *desc = reinterpret_cast<StageDesc *>(empty + P.nst);
    int *sflag = reinterpret_cast<int *>(desc + P.nst);
    const int tid = threadIdx.x, warp = tid / kWarp, lane = tid % kWarp;
    if (tid == 0) {
        for (int s = 0; s < P.nst; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kCW);
        }
        fence_mbar_init();
    }
    __syncthreads();
    if (warp == kCW) {
        Producer pr{P, ring, full, empty, desc, lane};
        pr.run();
    } else {
        Consumer co{P, ring, full, empty, desc, xs, ybuf, sflag, tid, lane, warp};
        co.run();
    }
}

}  // namespace

size_t decode_ctrl_bytes() { return sizeof(DecCtrl); }
size_t decode_table_bytes() { return sizeof(DecTable); }

size_t decode_smem_bytes(const DecParams &P) {
    return (size_t)P.nst * kSB + P.xs_bytes + P.ybuf_bytes + 2 * P.nst * sizeof(uint64_t) +
           P.nst * sizeof(StageDesc) + 16;
}

// Host-side geometry of the decode launch (static item counts, staging sizes).
void decode_plan(const coli_moe_desc &d, DecParams &P) {
    const int T = d.T;
    P.NV = T == 1 ? 1 : (T <= 2 || T > 32 ? 2 : 4);
    P.nst = 2;  // set by decode_plan_grid
    const int maxdim = std::max(d.H, std::max(d.I, d.I_shared));
    P.xs_stride = maxdim;
    const size_t xs_vec = (size_t)P.NV * maxdim * sizeof(float);
    const size_t xs_route = (size_t)(5 * d.E + kCW * d.E + 2 * (d.E + 2) + 16) * sizeof(int);
    P.xs_bytes = (int)align_up(std::max(xs_vec, xs_route), 128);
    const bool in_kernel_router = T <= 8;
    P.neb = (d.E + kRtE - 1) / kRtE;
    // about 64 router items: split H into k-slices of whole 128-float stages
    const int max_slices = (d.H + kRtKc / 4 - 1) / (kRtKc / 4);
    int nks = std::min(max_slices, std::max(1, (64 + P.neb - 1) / P.neb));
    const int stages = (max_slices + nks - 1) / nks;
    P.rks_floats = stages * (kRtKc / 4);
    nks = (d.H + P.rks_floats - 1) / P.rks_floats;
    P.route_only = in_kernel_router ? 0 : 1;
    P.nks = in_kernel_router ? nks : 0;  // T > 8: set by the caller to the router launch's splits
    P.R = in_kernel_router ? P.neb * nks : 1;
    P.groups_sh = d.I_shared > 0 ? (T + P.NV - 1) / P.NV : 0;
    P.G_sh_rb = d.I_shared > 0 ? (d.I_shared + kGuPairs - 1) / kGuPairs : 0;
    P.G_sh = P.G_sh_rb * P.groups_sh;
    P.gu_rb = (d.I + kGuPairs - 1) / kGuPairs;
}

// the grid is one CTA per SM; each owns ceil(H / grid) rows of the down projection
// and as many 16 KB ring stages (2..6) as fit beside the staging and y buffers
bool decode_plan_grid(const coli_moe_desc &d, DecParams &P, int grid) {
    P.rows_cta = (d.H + grid - 1) / grid;
    const size_t rows = (size_t)d.T * d.K + (d.I_shared > 0 ? d.T : 0);
    P.ybuf_bytes = (int)align_up(rows * P.rows_cta * sizeof(float), 128);
    const long budget = 227L * 1024 - P.xs_bytes - P.ybuf_bytes - 1024;
    const long nst = std::min(6L, budget / kSB);
    if (nst < 2) return false;
    P.nst = (int)nst;
    return decode_smem_bytes(P) <= 227u * 1024;
}

bool decode_supported(const coli_moe_desc &d) {
    if (d.T > kDecMaxT || d.T < 1) return false;
    // every gate/up row k-chunk and every down row must fit a 16 KB ring stage
    const int64_t dn_r = row_bytes(d.routed_fmt, d.I);
    const int64_t dn_s = d.I_shared > 0 ? row_bytes(d.shared_fmt, d.I_shared) : 0;
    if (dn_r > kSB || dn_s > kSB) return false;
    return true;
}

cudaError_t launch_decode(const DecParams &P, int grid, cudaStream_t st) {
    const size_t smem = decode_smem_bytes(P);
    cudaError_t e = cudaFuncSetAttribute(moe_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    // cooperative: every CTA of the static schedule is resident at once
    void *args[] = {const_cast<DecParams *>(&P)};
    return cudaLaunchCooperativeKernel((const void *)moe_decode_kernel, dim3(grid), dim3(kDecThreads), args,
                                       smem, st);
}

int decode_ctas_per_sm(const DecParams &P) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, moe_decode_kernel, kDecThreads, decode_smem_bytes(P)) !=
        cudaSuccess)
        return 1;
    return n < 1 ? 1 : n;
}

}  // namespace colimoe
