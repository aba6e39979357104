/*
 * pw.h -- C ABI of libpw.so: a GB300-native (sm_103a) fused mixed-precision MoE layer
 * that reads Any-Precision bit-planes and per-row centroid LUTs directly, with a
 * device-resident weight page table, asynchronous page offload/reload and a greedy
 * quality-aware planner.
 *
 * Source of every operation: "PagedWeight: Efficient MoE LLM Serving with Dynamic
 * Quality-Aware Weight Quantization" (arXiv 2607.16184).
 *
 * Conventions shared by every call
 *   - Every call returns pw_status; nothing throws across the ABI.  pw_last_error()
 *     gives a message for the last failing call on a context (or, with ctx == NULL,
 *     on the calling thread).
 *   - A CUDA error met asynchronously (a failed kernel or copy) is sticky: the next call
 *     on the same context returns PW_ERR_CUDA.
 *   - Host inputs are copied; the caller keeps ownership.  Device pointers handed to a
 *     call (x, y, ids, w) are borrowed and must stay valid until the stream reaches the
 *     work.  The context owns planes, LUTs, the page table, pinned host pages and scratch.
 *   - A context is used by one host thread at a time.
 *   - Linear block i = (layer, expert, u), u = 0 gate_up, 1 down, is addressed by the
 *     block id (layer * E + expert) * 2 + u.
 *   - A gate_up block has N = 2*I rows (gate rows 0..I-1, then up rows I..2I-1) and K = H
 *     columns; a down block has N = H rows and K = I columns.
 *   - Bitwidths: a block stores bmax <= 8 bit-planes, plane 0 the most significant bit,
 *     so a b-bit code is the top b planes.  Supported bitwidths are the set bits of
 *     bits_mask (each between 1 and bmax).  A LUT for bitwidth b holds 2^b fp16
 *     centroids per output row.
 *   - Page p of a block is bit-plane p together with LUT_{p+1} when p+1 is supported.
 *     At committed bitwidth q the GPU holds planes 0..q-1 and LUT_c for supported c <= q;
 *     M^b (Eq. 3 of the paper) counts exactly those bytes.
 */
#ifndef PW_H
#define PW_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PW_OK = 0,
    PW_ERR_INVALID = 1, /* bad argument: nothing was changed */
    PW_ERR_CUDA = 2,    /* a CUDA call failed (message in pw_last_error) */
    PW_ERR_OOM = 3,     /* device or pinned-host memory exhausted: nothing was changed */
    PW_ERR_STATE = 4,   /* the page state forbids the request (e.g. a page in transfer) */
    PW_ERR_TIMEOUT = 5, /* a bounded device wait gave up */
    PW_ERR_BUSY = 6,    /* an earlier transfer of the same block has not landed yet */
    PW_ERR_RANGE = 7    /* an fp16 activation overflowed or an output is not finite */
} pw_status;

typedef struct pw_ctx pw_ctx;
typedef void *pw_stream; /* a cudaStream_t; NULL means the legacy default stream */

enum {
    PW_FLAG_POISON = 1 /* fill retired device pages with 0xFF before reuse (testing) */
};

enum {
    PW_ACCUMULATE = 1, /* pw_moe_forward: y <- bf16(y + layer(x)); y may alias x */
    PW_PRENORM = 2     /* the layer reads RMSNorm(x) = x / sqrt(mean_h x^2 + 1e-6) (unit gain), the
                          way the pre-norm models of the paper's Table 1 feed their MoE blocks */
};

typedef struct {
    int L, E, H, I, K; /* layers, routed experts, hidden, expert intermediate, top-K */
    int Is;            /* shared-expert intermediate; 0 = no shared expert */
    int bmax;          /* bit-planes per block, 1..8 */
    uint32_t bits_mask;/* bit b set <=> bitwidth b supported */
    int renorm;        /* 1: routing weights renormalised over the chosen K */
    int device;        /* CUDA device ordinal */
    int max_tokens;    /* largest T accepted by the forward calls */
    int flags;         /* PW_FLAG_* */
} pw_desc;

/* ---------------------------------------------------------------- lifetime */

/* Create a context on desc->device.  The context holds the state the paper describes for one
 * model: the per-block weight pages and the device weight page table of Sec. 3.1 ("Paged
 * Weight Representation": committed bitwidth q_i, desired bitwidth d_i, per-page residency),
 * the compute and side streams of Sec. 3.3 ("Asynchronous Page Movement"), and the forward
 * scratch of the fused layer of Sec. 3.3.  The paper specifies no API; the call and its
 * plain-C signature are this library's own.  Requires H % 16 == 0, I % 8 == 0, Is % 8 == 0,
 * K <= E <= 256, K <= 8.  Allocates the page table, scratch for max_tokens tokens and
 * the two streams (compute stream = a new non-blocking stream, side stream for page
 * copies).  Errors: PW_ERR_INVALID on bad shapes, PW_ERR_CUDA / PW_ERR_OOM otherwise. */
pw_status pw_create(const pw_desc *desc, pw_ctx **out);
/* Release everything the context owns (device pages, pinned host pages, scratch, streams it
 * created); waits for its streams first.  NULL is ignored. */
void pw_destroy(pw_ctx *ctx);
/* Message of the last failing call on ctx (or of the calling thread when ctx is NULL); owned
 * by the library, valid until the next call on the same context or thread. */
const char *pw_last_error(const pw_ctx *ctx);
/* Library version string (static storage). */
const char *pw_version(void);

/* Stream on which commits (pw_set_bits, pw_offload's lowering, pw_commit's raising) and
 * the context's own copies are enqueued; by default a non-blocking stream the context
 * created.  Forward calls should run on the same stream so that a commit lands between
 * launches (PagedWeight Sec. 3.3: commit only at safe boundaries).  Switching waits for
 * the previous stream.  The caller keeps ownership of a stream it sets. */
pw_status pw_set_stream(pw_ctx *ctx, pw_stream stream);
pw_status pw_get_stream(pw_ctx *ctx, pw_stream *stream);

/* ---------------------------------------------------------------- weights */

/* Pack one linear block (PagedWeight Sec. 3.1 paged weight representation; APL overlaid
 * bit-planes, Sec. 2.2).
 *   idx: uint8 [N][K] codes < 2^bmax, row-major.
 *   lut: fp16 bits, the LUTs of every supported b in ascending b, concatenated:
 *        [N][2^b] for the smallest b, then the next, ...; entries in any order.
 *   q_init: initial committed bitwidth (supported).
 * idx and lut may both be host memory or both be device memory (detected).  Pages
 * 0..q_init-1 become GPU-resident, the rest CPU-resident in pinned host memory.
 * Re-packing a block replaces it (its pages must not be in transfer: PW_ERR_BUSY).
 * The device copy uses a kernel-private tiling of each plane; pw_unpack_indices
 * reproduces the plain codes. */
pw_status pw_pack(pw_ctx *ctx, int layer, int expert, int u, const uint8_t *idx,
                  const uint16_t *lut, int q_init);

/* Router of a layer (Sec. 2.1): Wr fp32 [E][H]; bias fp32 [E] or NULL.
 * Host or device pointers (detected). */
pw_status pw_set_router(pw_ctx *ctx, int layer, const float *Wr, const float *bias);

/* Shared expert of a layer (Table 1 counts shared experts): wgu bf16 bits [2*Is][H]
 * (gate rows, then up rows), wd bf16 bits [H][Is].  Host or device pointers.  The device
 * copy is fp16 (exact for bf16 values in [2^-14, 65504]; smaller ones keep an absolute
 * error below 2^-25); PW_ERR_INVALID if a weight exceeds 65504 in magnitude. */
pw_status pw_set_shared(pw_ctx *ctx, int layer, const uint16_t *wgu, const uint16_t *wd);

/* Gate the shared expert of `layer`: its output for token t is scaled by
 * sigmoid(x_t . wsg), x_t the layer input as the experts read it (RMS-normalised under
 * PW_PRENORM), computed in fp32 by the router.  This is the shared-expert gate of the
 * Qwen1.5-MoE model in Table 1; the pages describe no gating, so layers are ungated until
 * this is called.  wsg: fp32 [H], host or device, copied; NULL removes the gate.  Waits for
 * the context's stream.  PW_ERR_INVALID if the context has no shared expert. */
pw_status pw_set_shared_gate(pw_ctx *ctx, int layer, const float *wsg);

/* ---------------------------------------------------------------- forward */

/* One fused MoE layer (Sec. 3.3 "fused mixed-precision MoE kernel"): router logits in
 * fp32, softmax over E, top-K (ties to the lower expert id, listed by descending
 * probability), token-to-expert bucketing, gate_up with SiLU(gate)*up, down projection
 * and the routing-weighted combine y_t = sum_k r_tk o_tk (k order), plus the shared
 * expert.  Each block is read at the committed bitwidth q_i held in the device page
 * table when the launch runs.
 *   x: device bf16 [T][H]; y: device bf16 [T][H] (with PW_ACCUMULATE, y += layer(x);
 *   y may equal x).  ids (int32 [T][K]) and w (fp32 [T][K]) are optional device
 *   outputs (NULL to skip).  1 <= T <= max_tokens.  Asynchronous on `stream`; no host
 *   synchronisation and no allocation, so it can be captured in a CUDA graph.
 * Activations are handled in fp16 inside the expert kernels: |x| (after the RMS norm under
 * PW_PRENORM) and |h| must stay below 65504.  A value that rounds past it (or a NaN), and a
 * y that is not finite, set a flag in the context that pw_check reports as PW_ERR_RANGE. */
pw_status pw_moe_forward(pw_ctx *ctx, int layer, const void *x, int T, void *y,
                         int32_t *ids, float *w, int flags, pw_stream stream);

/* Wait for the compute stream and report whether a bounded wait inside an expert kernel
 * expired since the last check (PW_ERR_TIMEOUT; the outputs of that launch are invalid),
 * else whether an fp16 activation (x as the experts read it, or h) overflowed or a y came out
 * infinite or NaN (PW_ERR_RANGE; the outputs since the last check are invalid).  Both
 * flags are cleared by the call.  Also reports sticky CUDA errors.  No counterpart in the paper: the fused kernel of
 * Sec. 3.3 synchronises its warps on device barriers, and this library bounds every such
 * wait and reports the ones that gave up here. */
pw_status pw_check(pw_ctx *ctx);

/* The whole stack in place: for l = 0..L-1, x <- bf16(x + layer_l(RMSNorm(x))), i.e.
 * pw_moe_forward with PW_ACCUMULATE | PW_PRENORM and y = x.  x: device bf16 [T][H].  Asynchronous; launched as a CUDA graph replay after the first call
 * for a given (x, T, stream). */
pw_status pw_stack_forward(pw_ctx *ctx, void *x, int T, pw_stream stream);

/* End-to-end variant with host buffers: copies x_host (bf16 [T][H]) to the device,
 * runs pw_stack_forward, copies the result to y_host and waits for it.  Pinned host
 * buffers give full copy bandwidth; pageable ones work too. */
pw_status pw_stack_forward_host(pw_ctx *ctx, const void *x_host, int T, void *y_host);

/* Online routing statistics (Sec. 3.2 "Routing statistics"): per expert of `layer`, the
 * number of (token, k) selections and the sum of their routing weights since the last
 * reset, accumulated by every forward call.  Outputs are host double [E].  Waits for
 * the compute stream. */
pw_status pw_routing_stats(pw_ctx *ctx, int layer, double *count, double *weight_sum,
                           int reset);

/* Routed-input features phi of Eq. 5 (Sec. 3.2 "Prompt residual"), per expert of `layer`,
 * over every forward call since the last reset: with n_t the L2 norm of token t's input as
 * the experts read it (RMS-normalised under PW_PRENORM) and r the routing weight of each
 * (token, k) selection of the expert, phi[e] = (sum r n / sum r, sqrt(sum r n^2 / sum r),
 * max n); zeros for an expert no token reached.  Both linear blocks of an expert share its
 * phi.  Output host double [E][3].  Waits for the compute stream. */
pw_status pw_routing_features(pw_ctx *ctx, int layer, double *phi, int reset);

/* Decode kernel choice (no counterpart in the paper: its fused kernel, Sec. 3.3, has one
 * path; this switch offers a CUDA-core bit-plane GEMV for items too small to fill a tensor-core
 * tile in the memory-bound decode regime).  At decode batch sizes (T < 512) a routed work item -- a 128-row
 * tile of one expert's block times the tokens routed to that expert -- with at most
 * `max_tokens` tokens is computed on the CUDA cores (packed fp16 products of the decoded
 * centroids and the activations, summed in fp32 per 32 columns); larger items go to the
 * tensor cores.  0 sends every item to the tensor cores.  Default 0 (on GB300 the
 * tensor-core items measured faster at every decode size); valid 0..8, else
 * PW_ERR_INVALID.  Takes effect at the next forward launch (captured stack graphs are
 * dropped). */
pw_status pw_set_gemv_tokens(pw_ctx *ctx, int max_tokens);

/* Tracing (no counterpart in the paper; measurement only): while on, every forward records
 * five CUDA timing events per layer, before,
 * between and after its four kernels (router, gate_up, down, combine), on the launch
 * stream; stack graphs captured while on contain the event records.  The events are
 * owned by the context.  pw_profile_read waits for the latest recording of `layer` and
 * writes the four kernel durations in milliseconds to ms[0..3]. */
pw_status pw_set_profiling(pw_ctx *ctx, int on);
pw_status pw_profile_read(pw_ctx *ctx, int layer, float *ms);

/* Routing without allocation.  The paper has no counterpart: this entry point exists for
 * callers that cannot call cudaMalloc (or anything that allocates) where they route, e.g.
 * code running under a memory budget or allocator it does not own.  It runs the same
 * router kernel as pw_moe_forward -- fp32 logits, softmax, top-K, bucketing -- for layer
 * `layer` on device x (bf16 [T][H], 16-byte aligned), writing ids (int32 [T][K]) and w
 * (fp32 [T][K]) to the caller's device buffers.  flags: PW_PRENORM or 0.
 * Its scratch is a static device array of 8 MiB inside libpw.so (held by every GPU that
 * loads the library until the process exits); T is limited by it, and a T whose scratch
 * does not fit returns PW_ERR_INVALID.  The first call on a device looks up the array's
 * device address, so make it before any stream capture.  Calls share the array: calls
 * that overlap on the GPU (e.g. on two streams) race.  Online routing statistics are not
 * updated.  The call returns before the router runs: if the router's bounded wait for its
 * input copies gives up, a pw_check on the context made after the call's stream has run it
 * reports PW_ERR_TIMEOUT (and the ids and w of that call are invalid).  No cudaMalloc, cudaFree or other allocation happens
 * in the call. */
pw_status pw_route_noalloc(pw_ctx *ctx, int layer, const void *x, int T, int32_t *ids, float *w,
                           int flags, pw_stream stream);

/* ---------------------------------------------------------------- page table */

enum { PW_PAGE_GPU = 0, PW_PAGE_CPU = 1, PW_PAGE_TO_CPU = 2, PW_PAGE_TO_GPU = 3 };

typedef struct {
    int layer, expert, u;
    int N, K;
    int q;          /* committed bitwidth (read by the kernels) */
    int d;          /* desired bitwidth (set by the planner and by offload/reload) */
    int pending_q;  /* reload target waiting for its pages, or 0 */
    int state[8];   /* PW_PAGE_* per page 0..bmax-1 */
    int64_t M[9];   /* M^b bytes for b = 0..8 (-1 when b is not supported) */
} pw_block_info;

/* Commit bitwidth q for a block now (stream-ordered write of the device table entry on
 * the ctx stream).  Sec. 3.1 ("Paged Weight Representation"): the page table row holds the
 * committed bitwidth q_i the kernels read, and q_i may only name pages the GPU holds;
 * Sec. 3.3: a bitwidth changes only at a safe boundary, here between launches on the ctx
 * stream.  Every page below q must be GPU-resident (else PW_ERR_STATE, as for an unpacked
 * block); PW_ERR_BUSY while a transfer of the block is in flight; PW_ERR_INVALID if q is not
 * a supported bitwidth or block is out of range. */
pw_status pw_set_bits(pw_ctx *ctx, int block, int q);

/* Offload (Sec. 3.1, Sec. 3.3): lower the committed bitwidth of `block` to q_new first
 * (enqueued on the ctx stream), then copy pages q_new..q-1 to pinned host memory on the
 * side stream after the compute stream has passed the lowering.  The device pages are
 * released by the pw_commit call that sees the copy landed.  PW_ERR_STATE if q_new is
 * not a supported bitwidth below q or a page of the range is not GPU-resident;
 * PW_ERR_BUSY if a transfer of the block is in flight. */
pw_status pw_offload(pw_ctx *ctx, int block, int q_new);

/* Reload: allocate device pages q..q_new-1 and copy them in from pinned host memory on
 * the side stream; q stays unchanged until pw_commit sees the copy landed and then
 * raises q (Sec. 3.1: raise only once GPU-resident).  PW_ERR_OOM if device memory is
 * exhausted (nothing changed); PW_ERR_STATE / PW_ERR_BUSY as for pw_offload. */
pw_status pw_reload(pw_ctx *ctx, int block, int q_new);

/* Apply every transfer that has landed: retire offloaded device pages and commit the
 * raises of landed reloads on the ctx stream (Sec. 3.1: q_i rises only once the pages are
 * GPU-resident; Sec. 3.3 and Fig. 4: a reload becomes visible to the kernels at a later safe
 * commit point, and retired pages become free device memory).  *n_applied (may be NULL) receives the
 * number of raises committed.  Never blocks.  A failed copy rolls its block back
 * (pages stay or become CPU-resident, q is not raised) and returns PW_ERR_CUDA. */
pw_status pw_commit(pw_ctx *ctx, int *n_applied);

/* Wait for every transfer in flight (then pw_commit applies them).  Sec. 3.3's page movement
 * is asynchronous; this is the blocking point a caller uses before teardown or a test. */
pw_status pw_sync_io(pw_ctx *ctx);

/* One row of the weight page table and its host-side state (Sec. 3.1: the committed bitwidth
 * q_i, the desired bitwidth d_i, where each page lives, and M_i^b of Eq. 3 for every b).
 * info: caller storage.  PW_ERR_INVALID if block is out of range.  Does not wait. */
pw_status pw_query(pw_ctx *ctx, int block, pw_block_info *info);

typedef struct {
    int64_t resident_bytes;   /* sum over blocks of M_i^{q_i} (routed planes + LUTs) */
    int64_t device_pool_bytes;/* bytes reserved from cudaMalloc for pages */
    int64_t device_pool_free; /* of which free for reuse */
    int64_t pinned_bytes;     /* pinned host bytes reserved for CPU-resident pages */
    int64_t scratch_bytes;    /* forward scratch */
    int64_t held_bytes;       /* device bytes of the weight pages the GPU holds: resident, in
                                 transfer, or lowered but not yet retired by pw_commit */
} pw_mem_info;
/* Memory accounting of the context (Sec. 3.1 and Eq. 3: the GPU holds M_i^{q_i} bytes of
 * block i; Sec. 3.3: retired pages return to the device budget).  Does not wait. */
pw_status pw_memory(pw_ctx *ctx, pw_mem_info *info);

/* Host-side fault injection for testing the page I/O paths (no GPU fault is ever made; no
 * counterpart in the paper):
 * kind 1 = the n-th next page copy is reported failed instead of issued;
 * kind 2 = the n-th next device page allocation fails;
 * kind 3 = while n != 0, no transfer is observed as landed (the copies still run), so a
 * test can act while pages are in transfer;
 * kind 4 = with n != 0, the next forward's gate_up kernel withholds one barrier arrival of
 *   its first routed chunk (nothing asynchronous is held back), so that the bounded device
 *   wait on it expires: the launch's outputs are invalid and pw_check reports
 *   PW_ERR_TIMEOUT, after which the context is usable as before;
 * kind 5 = bounded device waits of the expert kernels give up after about n microseconds
 *   (n = 0: the default, about 2 s).
 * n = 0 clears kinds 1-4. */
pw_status pw_set_fault(pw_ctx *ctx, int kind, int n);

/* ---------------------------------------------------------------- planner */

typedef struct {
    int T_blk;          /* free-block threshold (Eq. 7) */
    int F_blk;          /* current number of free KV blocks (Eq. 7) */
    double B_KV;        /* bytes of one KV block (Eq. 7) */
    int R;              /* reload margin in blocks (reload when F_blk >= T_blk + R) */
    const double *mass; /* [L][E] routing mass (Eq. 1), or NULL: use the context's
                           online routing statistics (pw_plan_step only) */
    const double *phi;  /* [n_blocks][3] routed-input features (Eq. 5), or NULL: the
                           context's device features, pw_routing_features (pw_plan_step only) */
    const double *rho_hat; /* [n_blocks][n_bits-1] prompt residuals, transition j = bits[j+1] ->
                           bits[j], or NULL: Eq. 5 from phi.  A batch-level table from
                           pw_merge_requests (Sec. 3.2, batched serving); phi is then unused */
} pw_obs;

typedef struct {
    int n_bits;             /* number of supported bitwidths */
    const double *s;        /* [n_blocks][n_bits] offline sensitivity s_i^b (Eq. 2), b ascending */
    const double *head_w;   /* [2][n_bits-1][3] residual heads w_u^{b->b'} (Eq. 5); transition j: bits[j+1] -> bits[j] */
    const double *head_a;   /* [2][n_bits-1] */
    const double *head_c;   /* [2][n_bits-1] confidence c_u^{b->b'} (Eq. 6) */
    double alpha, rho_min, rho_max, eps; /* Eq. 6, Eq. 8 */
    int n_buckets;
    const double *mu;       /* [n_buckets] damage multipliers, bucket 0 hottest (Eq. 8) */
    const int *floors;      /* [n_buckets] bitwidth floors */
    int n_stages;           /* bitwidth-floor stages: stage s allows s+1 levels below q_i */
} pw_offline;

typedef struct {
    int block, from_bits, to_bits;
    double delta;           /* bytes released (offload) or restored (reload) */
} pw_plan_entry;

typedef struct {
    pw_plan_entry *entries; /* caller storage */
    int capacity;           /* entries available; PW_ERR_INVALID if too small */
    int n;                  /* entries written */
    int kind;               /* 0 no plan, 1 offload plan, 2 reload plan */
    int stage;              /* stage of the chosen offload plan, -1 otherwise */
    double D;               /* Eq. 7 byte target */
    double total;           /* bytes of the chosen plan */
} pw_plan;

/* A planner problem over explicit arrays (no context, no GPU). */
typedef struct {
    int n_blocks, n_bits, L, E;
    const int *bits;        /* [n_bits] ascending supported bitwidths */
    const int *q;           /* [n_blocks] committed bitwidths */
    const int *q_init;      /* [n_blocks] bitwidths reloads may restore up to */
    const int *utype;       /* [n_blocks] 0 gate_up, 1 down */
    const int *layer;       /* [n_blocks] */
    const int *expert;      /* [n_blocks] */
    const double *M;        /* [n_blocks][n_bits] M^b bytes (Eq. 3) */
} pw_plan_problem;

/* PlanStep (Algorithm 1 of Sec. 3.2) on an explicit problem: D from Eq. 7; for every
 * stage: score the legal single-level steps with Eqs. 4-6, 8, greedily take the lowest
 * d_hat / Delta until D is met (ties: larger Delta, then lower block); keep each stage's
 * plan; when D > 0 return the lowest stage meeting D, else the largest reduction.  When
 * D == 0 and F_blk >= T_blk + R, returns a reload plan instead (most damaging reduction
 * restored first while the bytes fit in (F_blk - T_blk - R) * B_KV).  Host only. */
pw_status pw_plan_host(const pw_plan_problem *prob, const pw_obs *obs,
                       const pw_offline *off, pw_plan *out);

/* One request's planner signals, for the batch-level merge. */
typedef struct {
    const double *mass;      /* [L][E] the request's routing mass (Eq. 1) */
    const double *rho_hat;   /* [n_blocks][n_bits-1] its prompt residuals (Eq. 5) */
    const double *conf;      /* [2][n_bits-1] its confidence scores c_u^{b->b'} (Eq. 6) */
    double rho_min, rho_max; /* its clipping bounds (Eq. 6) */
    double kv_blocks;        /* KV blocks the request holds: its weight in the merge */
} pw_request_signals;

/* Batched serving (Sec. 3.2): before planning, the signals of the batch's requests are
 * merged into a single batch-level table.  Routing masses, prompt residuals, confidence scores and clipping
 * bounds are each averaged with weights kv_blocks / sum(kv_blocks), requests summed in
 * order.  Outputs (caller storage): mass [L][E], rho_hat [n_blocks][n_bits-1], conf
 * [2][n_bits-1], *rho_min, *rho_max; plan with them by passing rho_hat in pw_obs and conf
 * and the bounds in pw_offline.  PW_ERR_INVALID if n_req < 1, a pointer is NULL, a weight
 * is negative or the weights do not sum to a positive number.  Host only. */
pw_status pw_merge_requests(const pw_request_signals *req, int n_req, int L, int E, int n_blocks,
                            int n_bits, double *mass, double *rho_hat, double *conf, double *rho_min,
                            double *rho_max);

/* PlanStep on the context's page table (q_i, M_i^b) and, when obs->mass is NULL, its
 * online routing statistics (Eq. 1).  Blocks with a page transfer in flight, or a landed
 * reload not yet committed, take no step (they are left out of the problem), so every
 * entry of the plan can be applied at once.  Writes the desired bitwidth d_i of every
 * planned block.  Applying the plan is the caller's pw_offload / pw_reload. */
pw_status pw_plan_step(pw_ctx *ctx, const pw_obs *obs, const pw_offline *off, pw_plan *out);

/* ---------------------------------------------------------------- KV-block allocator */

/* The KV blocks of a paged KV cache and the weight pages share one device budget: the pages
 * an offload retires become headroom for KV blocks, and the planner follows the free KV
 * blocks, the allocator headroom and the pending KV growth (Sec. 3.3).  This allocator hands
 * out logical block ids and keeps the free-block count F_blk that Eq. 7 (Sec. 3.2) turns into
 * the planner's byte target, with S the budget, W the weight-page bytes and B the block size:
 *   capacity  C = floor(max(0, S - W) / B) blocks
 *   U = blocks held by requests, P = blocks announced as pending growth
 *   F_blk = C - U - P  (negative when the budget is overcommitted; pass it as pw_obs.F_blk)
 *   headroom = S - W - U * B bytes
 * W is either set by the caller or read, on every call that needs it, from an attached
 * context (its pw_mem_info.held_bytes, so pages count until pw_commit retires them).  A
 * request is any int64 key.  Host only; an allocator is used by one thread at a time. */
typedef struct pw_kv pw_kv;

typedef struct {
    int64_t budget_bytes;     /* S */
    int64_t block_bytes;      /* B */
    int64_t weight_bytes;     /* W */
    int64_t capacity_blocks;  /* C */
    int64_t used_blocks;      /* U */
    int64_t pending_blocks;   /* P */
    int64_t free_blocks;      /* F_blk = C - U - P */
    int64_t headroom_bytes;   /* S - W - U * B */
} pw_kv_stats;

/* budget_bytes >= 0, block_bytes > 0 and budget_bytes / block_bytes < 2^31 (ids are int32),
 * else PW_ERR_INVALID.  W starts at 0. */
pw_status pw_kv_create(int64_t budget_bytes, int64_t block_bytes, pw_kv **out);
void pw_kv_destroy(pw_kv *kv);
/* W = weight_bytes (>= 0) from now on; detaches a context. */
pw_status pw_kv_set_weight_bytes(pw_kv *kv, int64_t weight_bytes);
/* W = ctx's held weight-page bytes from now on (ctx must outlive the attachment; NULL
 * detaches and keeps the last value read).  PW_ERR_* of pw_memory when reading fails. */
pw_status pw_kv_attach(pw_kv *kv, pw_ctx *ctx);
/* Request r expects to need n_blocks (>= 0) more blocks soon; replaces its previous
 * announcement.  The announced blocks count as taken in F_blk. */
pw_status pw_kv_announce(pw_kv *kv, int64_t request, int64_t n_blocks);
/* Grow request r by n_blocks (>= 0): c = min(n, r's announcement) of them come out of the
 * announcement, the other n - c must fit in F_blk, else PW_ERR_OOM and nothing changes.
 * The granted ids -- the lowest free ones, ascending -- go to ids_out[0..n-1] (NULL: not
 * written). */
pw_status pw_kv_grow(pw_kv *kv, int64_t request, int64_t n_blocks, int32_t *ids_out);
/* Return every block of request r and drop its announcement; the count to *n_released
 * (may be NULL).  An unknown request releases nothing. */
pw_status pw_kv_release(pw_kv *kv, int64_t request, int64_t *n_released);
/* Blocks request r holds and has announced (0 and 0 for an unknown request); either
 * pointer may be NULL.  The held count is the request's weight in pw_merge_requests. */
pw_status pw_kv_request(const pw_kv *kv, int64_t request, int64_t *held, int64_t *announced);
/* Request r's block table in the order granted: *n = its block count, and the first
 * min(*n, capacity) ids go to ids_out. */
pw_status pw_kv_blocks(const pw_kv *kv, int64_t request, int32_t *ids_out, int64_t capacity, int64_t *n);
pw_status pw_kv_get_stats(pw_kv *kv, pw_kv_stats *out);

/* ---------------------------------------------------------------- inspection */

/* b-bit codes of a block as the GPU kernels read them (the same device extraction code
 * as the forward): host uint8 [N][K].  Sec. 2.2 (Any-Precision LLM's overlaid bit-planes):
 * the b-bit code of an element is its top b bit-planes, plane 0 the most significant.
 * Pages 0..b-1 must be GPU-resident, else PW_ERR_STATE; PW_ERR_INVALID for a bad block or
 * b outside 1..bmax.  Waits for the ctx stream. */
pw_status pw_unpack_indices(pw_ctx *ctx, int block, int b, uint8_t *host_out);

/* Dequantised weights W^(b)[n][k] = LUT_b[n][code] as the GPU kernels produce them:
 * host fp16 bits [N][K].  Sec. 2.2: each output row has its own table of 2^b centroids per
 * supported bitwidth b, indexed by the b-bit code.  Pages 0..b-1 and LUT_b must be
 * GPU-resident, else PW_ERR_STATE; PW_ERR_INVALID for a bad block or unsupported b.
 * Waits for the ctx stream. */
pw_status pw_dequant(pw_ctx *ctx, int block, int b, uint16_t *host_out);

/* Self-check of the 5th-generation tensor-core path (tcgen05) on one CTA: D[128][N] =
 * A[128][K] * B[N][K]^T with fp16 A, B (row-major, device) and fp32 D (row-major, device),
 * 16 <= N <= 256 and 16 <= K <= 128, both multiples of 16.  flags bit 0: A goes through
 * tensor memory (written with tcgen05.st, read by the MMA from there) as the expert kernels'
 * dequantised weights do; otherwise both operands come from shared memory.  Other flag
 * bits are invalid.  *err (device int) is set to 1 if the bounded wait for the MMAs
 * expired.  Asynchronous on `stream`.  No counterpart in the paper: a hardware check. */
pw_status pw_tc_selftest(const uint16_t *A, const uint16_t *B, int N, int K, int flags, float *D, int *err,
                         pw_stream stream);

/* Pure host helpers (no context, no GPU) for checking the packer (Sec. 2.2 bit-planes,
 * Sec. 3.1 one page per plane).
 * pw_pack_planes_host: the plain plane layout -- planes [bmax][N][W] uint32,
 *   W = ceil(K/128)*4 words per row, bit j of word w is column 32w+j, plane 0 = MSB.
 * pw_tile_planes_host / pw_untile_planes_host: the kernel-private device tiling of
 *   those planes for a block of type u (gate_up rows are interleaved per 16-row tile)
 *   and its inverse.  Sizes: bmax * N * W words each. */
pw_status pw_pack_planes_host(const uint8_t *idx, int N, int K, int bmax, uint32_t *planes);
pw_status pw_tile_planes_host(const uint32_t *planes, int N, int K, int nplanes, int u,
                              uint32_t *tiled);
pw_status pw_untile_planes_host(const uint32_t *tiled, int N, int K, int nplanes, int u,
                                uint32_t *planes);

#ifdef __cplusplus
}
#endif
#endif /* PW_H */
