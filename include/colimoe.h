/* colimoe.h — C ABI of libcolimoe: one MoE feed-forward block on quantized expert weights,
 * computed by hand-written CUDA kernels for GB300 (sm_103a).
 *
 * What the block computes (colibri-strix c/glm.c @98759bf, function moe(); colibri
 * c/backend_metal.mm @93cde63, shaders r_router / r_top8 / moe_gemv / moe_silu):
 *   for every token t (a row of x[T,H]):
 *     logit[e]  = x_t . W_r[e]                       (fp32 router, moe() phase A)
 *     sig[e]    = 1 / (1 + exp(-logit[e]))          (sigmoidf)
 *     choice[e] = sig[e] + bias[e]                  (noaux_tc selection bias, n_group = 1)
 *     idx[0..K) = greedy top-K of choice, ties to the lower expert index (r_top8 / r_top8_par)
 *     w[k]      = sig[idx[k]]; optional adaptive top-p truncation (TOPP) and TOPK override;
 *                 if norm_topk: w /= (sum w + 1e-20); then w *= routed_scale
 *     for each kept k, expert e = idx[k] (moe() phases C/D):
 *       g = G_e x_t, u = U_e x_t, h = silu(g) * u, y = D_e h
 *       out_t += w[k] * y                            (in selection order)
 *     out_t += shared expert SwiGLU(x_t)             (weight 1, moe() phase E)
 *   A quantized matrix W[O][In] with per-row scale s[O] is used as
 *     (W v)[o] = (sum_i deq(W[o,i]) * v[i]) * s[o]     (matmul_q / matmul_i4 / matmul_i2)
 *   deq: COLI_FMT_INT8 — signed byte; COLI_FMT_INT4 — element i in byte i/2, low nibble for
 *   even i, value = nibble - 8; COLI_FMT_INT2 — element i in byte i/4 at bit 2*(i%4),
 *   value = field - 2 (the QT tensor formats of glm.c).
 *   COLI_FMT_INT4G (int4-grouped, tensor format 4 of glm.c's qt_resolve_fmt on the colibri
 *   "compare main...docs-quickstart" page): the int4 bytes with one fp32 scale per group of
 *   gs = desc->group_size consecutive inputs of a row, scales [O][ceil(In/gs)] row-major, and
 *     (W v)[o] = sum_g s[o][g] * (sum_{i in group g} deq(W[o,i]) * v[i])
 *   (the last group of a row holds In - (ceil(In/gs) - 1) * gs inputs).
 *
 * Conventions for every entry point:
 *  - All tensors are row-major and live in DEVICE memory unless the argument says HOST.
 *    The caller owns every buffer, including the workspace; the library never allocates,
 *    frees or synchronises inside coli_moe_route / coli_moe_forward / coli_moe_qgemv: work is
 *    enqueued on `stream` (a cudaStream_t; NULL = the legacy default stream) on the current
 *    device, and the call returns when it is enqueued.
 *  - Return value: COLI_MOE_OK (0) or a negative COLI_MOE_E* code. Arguments are validated
 *    on the host before anything is launched; on an error nothing is enqueued.
 *    Faults that happen while the kernels run surface at the caller's next synchronisation;
 *    kernel-detected conditions (no selectable expert, a misaligned routed-expert pointer,
 *    an expired bounded wait) set an error word in the workspace that coli_moe_check reads.
 *    route / forward calls clear that word when they start, so it reports the latest call.
 *  - There is no CPU fallback: every step runs in this library's kernels.
 *  - Packed weight rows must start on 16-byte boundaries: H and I must be multiples of 16
 *    (int8), 32 (int4, int4-grouped) or 64 (int2), and every weight and scale pointer 16-byte aligned;
 *    x and out must be 16-byte aligned. Violations return COLI_MOE_EALIGN / COLI_MOE_ENOTSUP.
 *  - Limits: 1 <= K <= min(E, 32), E <= 1024, T <= 65536, H, I <= 65536.
 */
#ifndef COLIMOE_H
#define COLIMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *coli_stream_t; /* the same type as cudaStream_t */

/* weight formats (glm.c QT struct; 0 = f32 is not an expert format here) */
#define COLI_FMT_INT8 1
#define COLI_FMT_INT4 2
#define COLI_FMT_INT2 3
#define COLI_FMT_INT4G 4 /* int4 with per-group scales; group size in coli_moe_desc.group_size */

/* return codes */
#define COLI_MOE_OK 0
#define COLI_MOE_EINVAL (-1)     /* a null required pointer or an out-of-range size/option */
#define COLI_MOE_ENOTSUP (-2)    /* a valid request this build does not implement (format, dims) */
#define COLI_MOE_EALIGN (-3)     /* a pointer or row stride is not 16-byte aligned */
#define COLI_MOE_EWORKSPACE (-4) /* ws is NULL, misaligned (256 B) or smaller than required */
#define COLI_MOE_ECUDA (-5)      /* a CUDA runtime call failed; see coli_moe_last_cuda_error */
#define COLI_MOE_EDEVICE (-6)    /* the current device is not compute capability 10.3 */
#define COLI_MOE_EKERNEL (-7)    /* a kernel flagged an error in the workspace (coli_moe_check) */

/* Block description (the config.json fields moe() reads: hidden_size, moe_intermediate_size,
 * n_routed_experts, num_experts_per_tok, n_shared_experts * moe_intermediate_size,
 * norm_topk_prob, routed_scaling_factor; plus glm.c's TOPK and TOPP switches). */
typedef struct {
    int32_t T;            /* tokens (rows of x and out), >= 1 */
    int32_t H;            /* hidden size */
    int32_t I;            /* routed expert intermediate size */
    int32_t E;            /* routed experts */
    int32_t K;            /* experts per token */
    int32_t I_shared;     /* shared expert intermediate size; 0 = no shared expert */
    int32_t norm_topk;    /* 1: renormalise the kept weights to sum 1 before scaling */
    float routed_scale;   /* routed_scaling_factor, multiplies the kept weights */
    int32_t routed_fmt;   /* COLI_FMT_* of every routed expert */
    int32_t shared_fmt;   /* COLI_FMT_* of the shared expert (may differ from routed_fmt) */
    int32_t ksel;         /* TOPK override: keep min(ksel, K) experts; 0 = K */
    float top_p;          /* adaptive top-p in (0,1); 0 = off */
    int32_t group_size;   /* inputs per scale of COLI_FMT_INT4G tensors (routed and shared alike):
                             a positive multiple of 32; ignored when neither format is 4.
                             Blocks with an int4-grouped expert run the single-token kernel at
                             T = 1 (unless idot is also set) and the general kernels (router
                             launch, gate/up, down and combine launches) for every other T. */
    int32_t idot;         /* 0: exact products (the default, IDOT=0 in glm.c). 1: glm.c's IDOT
                             kernels for int8 and int4 experts (qrow_i8 / matmul_q_idot /
                             matmul_i4_idot): each activation row x (x for gate and up, h for
                             down) is quantised to q = round-half-even(x / s) with
                             s = max(max|x| / 127, 1e-12), the integer sum of deq(W) * q is exact,
                             and y[o] = ((float)sum * scale[o]) * s — lossy (about 0.3 % RMS per
                             product, as the pages state). int2 and int4-grouped experts keep the
                             exact path. T = 1 runs the single-token kernel (int8 bytes on the
                             DP4A core; with an int4-grouped expert in the block, the general
                             kernels); other T the general kernels. */
} coli_moe_desc;

/* One expert's six device pointers: gate/up are [I][row_bytes(H)] with fp32 scales [I];
 * down is [H][row_bytes(I)] with fp32 scales [H] (I = I_shared for the shared expert).
 * For COLI_FMT_INT4G the scales are [I][ceil(H/gs)] (gate, up) and [H][ceil(I/gs)] (down). */
typedef struct {
    const void *gate_w;
    const void *up_w;
    const void *down_w;
    const float *gate_s;
    const float *up_s;
    const float *down_s;
} coli_moe_expert;

/* Bytes of device workspace coli_moe_route / coli_moe_forward / coli_moe_forward_host need
 * for this description (256-byte aligned base required). Returns 0 if desc is invalid. */
size_t coli_moe_workspace_bytes(const coli_moe_desc *desc);

/* Router + selection + buckets (moe() phases A and B; r_router + r_top8_par).
 *   x [T,H] fp32, W_r [E,H] fp32, bias [E] fp32                           (inputs)
 *   idx [T,K] int32, w [T,K] fp32: the kept experts in selection order and their weights;
 *     slots beyond keff[t] hold -1 / 0                                       (outputs)
 *   keff [T] int32: experts kept per token (K unless ksel/top_p cut it)    (output, may be NULL)
 *   counts [E], offsets [E+1], perm [T*K] int32: token->expert buckets — perm lists the
 *     assignment ids a = t*K + k grouped by expert, ascending a within each expert,
 *     offsets is the exclusive prefix sum of counts                         (outputs, may be NULL)
 *   ws / ws_bytes: workspace of at least coli_moe_workspace_bytes(desc) bytes. */
int coli_moe_route(const coli_moe_desc *desc, const float *x, const float *W_r,
                   const float *bias, int32_t *idx, float *w, int32_t *keff, int32_t *counts,
                   int32_t *offsets, int32_t *perm, void *ws, size_t ws_bytes,
                   coli_stream_t stream);

/* The whole block: out[T,H] (fp32, overwritten) = routed experts combined in selection order
 * with their weights, plus the shared expert.
 *   experts: DEVICE array [E] of coli_moe_expert (device pointers inside).
 *   shared:  HOST pointer to one coli_moe_expert holding device pointers; NULL iff
 *            desc->I_shared == 0.
 *   idx_out / w_out: optional DEVICE [T,K] copies of the routing (may be NULL).
 * Arithmetic. The router (logits, sigmoid, bias, selection, renorm) is fp32 on every path;
 * expert ids are decided exactly as the serial scan decides them on the fp32 choices. The
 * dequantised weights are always exact (small integers times the fp32 row scale, applied after
 * the sum). The expert products depend on the path the description selects:
 *  - T = 1, formats 1-3: one persistent launch. Each activation vector (x for gate/up, h for
 *    down) is put in 24-bit block fixed point, X = round(v * 2^s) with s set by max|v|, so
 *    every element is exact to 2^-23 of max|v|; the integer products and their sums are exact
 *    (int32 lanes, int64 totals), then one conversion to float and the row scale. Output error
 *    within 1e-4 * rms(out) of the exact block.
 *  - T = 1 with a COLI_FMT_INT4G expert (the rest formats 1-4): the same launch and activation
 *    fixed point; each 16-byte chunk of a row (32 inputs, inside one group) gets its exact
 *    integer sum, converted to float and multiplied by its group's scale, and the row's chunk
 *    products are summed in fp32. Output error within 1e-4 * rms(out).
 *  - 2 <= T <= 64, formats 1-3: one persistent launch (plus a router launch for T > 8).
 *    Single-token expert groups run as above; groups of 2-4 tokens run on the tensor cores
 *    (mma.sync f16) with each token's vector split into two f16 parts (hi + lo, 22 significant
 *    bits relative to that token's max|v|), exact f16 weights, exact products and fp32
 *    accumulation. Output error within 1e-4 * rms(out).
 *  - T > 64 with H, I, I_shared multiples of 64, formats 1-3: x and h are rounded to bf16
 *    (round to nearest even) and the expert products run as tcgen05 bf16 GEMMs with fp32
 *    accumulation in tensor memory; scales and SiLU are fp32. Output error within
 *    2e-2 * rms(out).
 *  - T = 1 with desc->idot set: the same launch on the IDOT quantisation (int8 activations, one
 *    scale per vector, exact int32 sums, y = ((float)dot * scale) * s), as described at
 *    coli_moe_desc.idot; within 2e-3 * rms(out) of the IDOT definition.
 *  - A block with a COLI_FMT_INT4G expert at T > 1, or with desc->idot set at T > 1, and T > 64
 *    shapes the GEMMs do not take: separate router, selection, bucket, gate/up, down and combine launches with
 *    fp32 products and fp32 accumulation (1e-4 * rms(out)); with idot, the IDOT quantisation
 *    described at coli_moe_desc.idot (2e-3 * rms(out) of the IDOT definition).
 * Results are deterministic: the same inputs give the same bits (fixed summation orders, no
 * float atomics). */
int coli_moe_forward(const coli_moe_desc *desc, const float *x, const float *W_r,
                     const float *bias, const coli_moe_expert *experts,
                     const coli_moe_expert *shared, float *out, int32_t *idx_out,
                     float *w_out, void *ws, size_t ws_bytes, coli_stream_t stream);

/* Same work as coli_moe_forward, and it records caller-created CUDA events (cudaEvent_t,
 * passed as void*) on `stream` at the stage boundaries: events[0] before the router,
 * events[1] after routing and bucketing, events[2] after the gate/up (+SiLU*mul) kernel,
 * events[3] after the down kernel, events[4] after the combine. n_events must be 5.
 * Meant for live per-stage timing; the events are only recorded, never synchronised. */
int coli_moe_forward_profiled(const coli_moe_desc *desc, const float *x, const float *W_r,
                              const float *bias, const coli_moe_expert *experts,
                              const coli_moe_expert *shared, float *out, void *const *events,
                              int n_events, void *ws, size_t ws_bytes, coli_stream_t stream);

/* The block as the tail of a decoder layer (colibri-strix c/glm.c @98759bf, the layer forward
 * after the attention residual: rmsnorm with post_ln, moe(), x += tmp; the Metal path runs the
 * norm, the router and the shared expert in one command buffer, coli_metal_layer_decode):
 *   xn[t]  = resid[t] * r_t * norm_w,   r_t = 1 / sqrtf(mean_i resid[t][i]^2 + eps)
 *            (the mean square accumulated in double, the rest in float, in that order)
 *   out[t] = resid[t] + block(xn)[t]   (the block exactly as coli_moe_forward computes it)
 *   resid [T,H] fp32, norm_w [H] fp32 (16-byte aligned), eps >= 0 (rms_norm_eps); out may be
 *   resid itself (an in-place residual update). Other arguments as coli_moe_forward.
 * T = 1 runs as one launch: the single-token kernel normalises resid itself in every CTA.
 * Other T add one small launch that writes the normalised rows into the workspace. */
int coli_moe_forward_tail(const coli_moe_desc *desc, const float *resid, const float *norm_w, float eps,
                          const float *W_r, const float *bias, const coli_moe_expert *experts,
                          const coli_moe_expert *shared, float *out, int32_t *idx_out, float *w_out, void *ws,
                          size_t ws_bytes, coli_stream_t stream);

/* The normalisation of coli_moe_forward_tail on its own: xn[t] = resid[t] * r_t * norm_w for
 * T rows of H (H a multiple of 4; resid, norm_w, xn 16-byte aligned; xn may be resid). Uses no
 * workspace. */
int coli_moe_rmsnorm(const float *resid, const float *norm_w, float eps, float *xn, int32_t T, int32_t H,
                     coli_stream_t stream);

/* Same as coli_moe_forward, but x_host and out_host are HOST buffers (page-locked memory
 * gives asynchronous copies). The copies go through the workspace; the call synchronises
 * `stream` before it returns, so out_host is ready on return. */
int coli_moe_forward_host(const coli_moe_desc *desc, const float *x_host, const float *W_r,
                          const float *bias, const coli_moe_expert *experts,
                          const coli_moe_expert *shared, float *out_host, void *ws,
                          size_t ws_bytes, coli_stream_t stream);

/* Quantized GEMV/GEMM building block: y[t][o] = (sum_i deq(W[o,i]) * x[t][i]) * s[o] for
 * t < T, o < O (matmul_q / matmul_i4 / matmul_i2; mm_gemv). W is [O][row_bytes(In)], s [O],
 * x [T][In] fp32, y [T][O] fp32. Uses no workspace. */
int coli_moe_qgemv(int32_t fmt, const void *W, const float *s, const float *x, float *y,
                   int32_t O, int32_t In, int32_t T, coli_stream_t stream);

/* The same for an int4-grouped matrix (COLI_FMT_INT4G; coli_moe_qgemv refuses that format with
 * COLI_MOE_ENOTSUP because it needs the group size): W is [O][In/2] int4 bytes, s is
 * [O][ceil(In/group_size)] fp32, y[t][o] = sum_g s[o][g] * sum_{i in group g} deq(W[o,i]) * x[t][i].
 * group_size: a positive multiple of 32 (else COLI_MOE_EINVAL). Uses no workspace. */
int coli_moe_qgemv_grouped(const void *W, const float *s, int32_t group_size, const float *x, float *y,
                           int32_t O, int32_t In, int32_t T, coli_stream_t stream);

/* Synchronises `stream`, reads and clears the workspace error word. Returns COLI_MOE_OK,
 * COLI_MOE_EKERNEL if a kernel flagged an error since the last check, or COLI_MOE_ECUDA. */
int coli_moe_check(void *ws, coli_stream_t stream);

/* Static description of a return code. */
const char *coli_moe_strerror(int code);

/* The cudaError_t of the last COLI_MOE_ECUDA returned on this thread (0 if none). */
int coli_moe_last_cuda_error(void);

/* ---- Forward without any caller-provided or allocated scratch ----
 * The pages have no counterpart of this entry point; it exists for callers that cannot call
 * cudaMalloc: code running where device allocation is forbidden or unavailable (a host
 * application whose memory pool owns all device memory, a plugin or sandbox that may only
 * launch work, a latency-critical loop that must never enter the allocator), and that
 * therefore cannot provide the workspace coli_moe_forward asks for.
 *
 * It computes exactly what coli_moe_forward computes, with the same arguments minus the
 * workspace and the optional routing outputs, and its result is bit-identical to that call's.
 * Its scratch is one fixed array of COLI_MOE_NOALLOC_SCRATCH_BYTES inside the library's device
 * image: every GPU on which the library is loaded holds that much memory until the process
 * exits. The caller still owns and passes x, the weights and out.
 *   - Sizes: a description whose coli_moe_workspace_bytes() exceeds
 *     COLI_MOE_NOALLOC_SCRATCH_BYTES is rejected with COLI_MOE_EWORKSPACE before anything is
 *     launched. At H = 6144, I = I_shared = 2048, E = 256, K = 8 that admits T <= 89 (T up to
 *     64 on the persistent decode kernels, 65..89 on the tensor-core GEMMs).
 *   - Set-up: the first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and keeps it for the life of the
 *     process; make that first call before any stream capture. The kept address belongs to
 *     the device's primary context: after cudaDeviceReset (or any teardown of that context) do
 *     not call this entry point again in the same process.
 *   - Sharing: all calls, on every stream and thread, use the same array, which keeps the last
 *     call's contents (each call clears what must start at zero). Calls whose work overlaps on
 *     the GPU — on different streams, or from different threads without ordering — race on
 *     it and give wrong results; order them on one stream.
 *   - Errors: kernel-detected conditions (no selectable expert, a misaligned expert pointer,
 *     an expired bounded wait) land in the array's error word; coli_moe_noalloc_check reads
 *     and clears it.
 *   - It calls no cudaMalloc, cudaFree or other allocating routine. */
#define COLI_MOE_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
int coli_moe_forward_noalloc(const coli_moe_desc *desc, const float *x, const float *W_r,
                             const float *bias, const coli_moe_expert *experts,
                             const coli_moe_expert *shared, float *out, coli_stream_t stream);

/* coli_moe_check for the fixed array of coli_moe_forward_noalloc, on the current device:
 * synchronises `stream`, reads and clears the array's error word. Returns COLI_MOE_OK,
 * COLI_MOE_EKERNEL if a kernel flagged an error since the last check, or COLI_MOE_ECUDA.
 * Allocates nothing. */
int coli_moe_noalloc_check(coli_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* COLIMOE_H */
