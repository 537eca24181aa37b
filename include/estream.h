/*
 * estream.h -- C ABI of the GB300 MoE-layer prefill library (libestream.so).
 *
 * One MoE layer's prefill over T prompt tokens, as described in "EStream:
 * Fast and Memory-Efficient MoE Prefill through Expert Virtualization on
 * Mobile NPUs" (arXiv 2609.06551):
 *   - section 3.2, Eq. 2: Y_t = A_t + sum over (e, alpha) in R_l(t) of
 *     alpha * F_e(X_t), with Eq. 1: F_e(x) = W_e^d (SiLU(W_e^g x) (*) W_e^u x);
 *   - section 3.2, "Composed Sparse Route and Parameter Binding" and
 *     Algorithm 1: routes (e_i, t_i, alpha_i), slots psi_i = Phi_l(e_i), a
 *     CSR of records (t_i, i) by slot, and slot addresses p_s^j = p_{B^j} +
 *     s*S_j (Eq. 3) for the three parameter planes j in {g, u, d};
 *   - section 3.3: a bounded arena of P = B*G fixed-address slots organised
 *     in B banks of G slots; storage groups of G experts in an offline order
 *     pi_l; placement Phi_l(e) = b*G + (pi_l(e) mod G) (Eq. 4); slot states
 *     Available -> Filling -> Ready -> InUse -> Available;
 *   - section 3.4: loading overlapped with execution; after routing, groups
 *     with no routes are skipped.
 *
 * Conventions for every call:
 *   - Every entry point returns an estream_status; nothing throws, exits or
 *     aborts. Argument errors are reported before anything is enqueued.
 *   - "device pointer" arguments are CUDA device memory owned by the caller;
 *     the library never frees them. "host pointer" arguments are host memory.
 *   - Calls taking `cuda_stream` (a cudaStream_t; NULL = legacy default
 *     stream) enqueue their GPU work on it and return without waiting, except
 *     where a call says it synchronises.
 *   - Errors found by a kernel while it runs (a slot id out of range, a
 *     bounded wait that ran out) are written to a device error word and
 *     reported by estream_get_device_error / estream_workspace_error.
 *   - Only sm_100-family GPUs built for here (sm_103a) are supported; other
 *     devices get ESTREAM_ERR_UNSUPPORTED.
 *   - Tracing: the calling thread's work is marked with NVTX ranges in the
 *     domain "estream" ("layer", "route build", "route from X", "routed
 *     experts", "shared experts", "combine", "bank fill", "preload"; payload:
 *     the layer, or layer * 65536 + group for a bank fill). They cost nothing
 *     measurable unless a tool is attached.
 */
#ifndef ESTREAM_H
#define ESTREAM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ESTREAM_OK = 0,
    ESTREAM_ERR_INVALID_ARG = 1,  /* bad pointer, size, alignment or shape */
    ESTREAM_ERR_CAPACITY = 2,     /* T or k beyond what the context was bound for */
    ESTREAM_ERR_NOT_BOUND = 3,    /* null or unbound context */
    ESTREAM_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed */
    ESTREAM_ERR_PAGER = 5,        /* the pager failed to fill a bank */
    ESTREAM_ERR_TIMEOUT = 6,      /* a kernel's bounded wait ran out */
    ESTREAM_ERR_DEVICE = 7,       /* a kernel found bad data (e.g. a slot id out of range) */
    ESTREAM_ERR_UNSUPPORTED = 8   /* device or data type not supported */
} estream_status;

/* Arithmetic types of a context. F32: X and weights fp32 (CUDA cores).
 * BF16: X and weights bf16 (tensor cores; the down weights are converted to
 * fp16 at pack time). Q4: X bf16; every expert weight 4-bit -- blocks of 32
 * weights along the reduction share one scale, value = (code - 8) * scale
 * (the paper stores expert matrices as weight-only GGUF Q4_0, section 4);
 * packed from bf16 master weights by estream_pack_experts /
 * estream_pack_shared. */
typedef enum { ESTREAM_F32 = 0, ESTREAM_BF16 = 1, ESTREAM_Q4 = 2 } estream_dtype;

/* Short English name of a status code (static storage). */
const char* estream_status_string(estream_status s);

/* ABI version of this header: major*10000 + minor*100 + patch. */
int estream_version(void);

/* ---------------------------------------------------------------------- */
/* Routing and route map                                                   */
/* ---------------------------------------------------------------------- */

/* Bytes of device workspace estream_route_build needs for these sizes. */
size_t estream_route_workspace_bytes(int T, int E, int k, int P);

/*
 * Router top-k and the route map of section 3.2 / Algorithm 1.
 *
 * logits    device, [T][E] fp32 row-major, finite values.
 * T, E, k   tokens, experts, routes per token: T >= 0, 1 <= k <= E <= 1024, k <= 32.
 * renorm    0: alpha = softmax probability; 1: alpha divided by the sum of
 *           the token's k selected probabilities (summed in rank order).
 * phi       device, [E] int32: Phi(e) = slot in [0, P), or -1 when expert e
 *           is not resident; NULL means the identity and needs P == E.
 * P         physical slots, 0 <= P <= 4096.
 * topk_ids  device, [T*k] int32 out: route i = t*k + j is the token's j-th
 *           expert, larger logit first, equal logits -> lower expert id.
 * alpha     device, [T*k] fp32 out: the routing weight of route i.
 * offsets   device, [P+2] int32 out: slot s owns records
 *           [offsets[s], offsets[s+1]); the trailing bucket P holds the
 *           routes whose expert is not resident; offsets[P+1] = T*k.
 * rec_tok   device, [T*k] int32 out: t_i of the record at each position.
 * rec_route device, [T*k] int32 out: route index i of the record; records
 *           of one slot are in ascending i.
 * workspace device, >= estream_route_workspace_bytes(T, E, k, P) bytes,
 *           256-byte aligned; its contents need no initialisation (the call
 *           clears the error word estream_workspace_error reads).
 * The softmax uses a written fp32 exponential (Cody & Waite range
 * reduction + degree-7 Taylor polynomial) so that alpha is reproducible bit
 * for bit. Nothing is synchronised. A phi entry outside [-1, P) is reported
 * through estream_workspace_error.
 */
estream_status estream_route_build(const float* logits, int T, int E, int k, int renorm,
                                   const int32_t* phi, int P,
                                   int32_t* topk_ids, float* alpha, int32_t* offsets,
                                   int32_t* rec_tok, int32_t* rec_route,
                                   void* workspace, size_t workspace_bytes,
                                   void* cuda_stream);

/* Synchronises `cuda_stream` and returns the error a route-build or
 * router-logits kernel recorded in `workspace` (ESTREAM_OK if none), then
 * clears it. */
estream_status estream_workspace_error(void* workspace, void* cuda_stream);

/* Bytes of device workspace estream_router_logits needs for these sizes on
 * the current device (>= 256); 0 for invalid sizes. */
size_t estream_router_workspace_bytes(int T, int H, int E);

/*
 * Router logits upstream of the top-k: logits[t][e] = sum over h of
 * X[t][h] * W_r[e][h]. The pages name the router (a token goes to the top-k
 * of E experts, section 1) and run routing on the accelerator from the layer
 * input (section 4) without giving its form; this is the bias-free linear
 * router of top-k MoE layers. The output feeds estream_route_build or
 * estream_moe_layer_prefill.
 *
 * X         device, [T][H] bf16 row-major, 16-byte aligned.
 * W_r       device, [E][H] bf16 row-major (one row per expert), 16-byte aligned.
 * T, H, E   T >= 0; H a multiple of 64; 1 <= E <= 1024.
 * logits    device, [T][E] fp32 out.
 * workspace device, >= estream_router_workspace_bytes(T, H, E) bytes,
 *           256-byte aligned; no initialisation needed. Its first word is the
 *           error word estream_workspace_error reads (a bounded wait that ran
 *           out is reported there).
 * Computed on the tensor cores (bf16 products, fp32 accumulation) with the
 * K range split into chunks whose fp32 partial sums are added in a fixed
 * order: the result does not depend on timing, but its rounding differs
 * from a sequential fp32 sum. Nothing is synchronised.
 */
estream_status estream_router_logits(const void* X, int T, int H, const void* W_r, int E,
                                     float* logits, void* workspace, size_t workspace_bytes,
                                     void* cuda_stream);

/*
 * Router logits and route map in one call: logits = X W_r^T as
 * estream_router_logits computes them (bf16 products, fp32 accumulation,
 * the K range split into chunks whose partial sums are added in a fixed
 * order), then the top-k and route map of estream_route_build on those
 * logits, which are also written to `logits`. The pages run routing on the
 * accelerator from the layer input (section 1, section 4); this is that
 * operator as one kernel: a cooperative launch of thread-block clusters in
 * which each cluster computes a 128-token tile of logits on the tensor cores,
 * sums the chunks' partials in shared memory, ranks the tile's tokens there
 * and then joins the grid-wide route-map construction -- the logits never
 * make a round trip through device memory before the top-k. Shapes the
 * single launch cannot take (E > 128, or more 128-token tiles than clusters
 * the device holds at once) run the router kernel and the route build as
 * two launches on the same stream, with the same results;
 * estream_route_build_from_x_fused tells which form a shape gets.
 *
 * X, W_r, T, H, E  as in estream_router_logits (H a multiple of 64).
 * k, renorm, phi, P, topk_ids, alpha, offsets, rec_tok, rec_route, workspace,
 *           workspace_bytes: as in estream_route_build (the workspace size is
 *           estream_route_workspace_bytes(T, E, k, P)).
 * logits    device, [T][E] fp32 out.
 * Errors the kernels find (a phi entry out of range, a bounded wait that ran
 * out) are reported by estream_workspace_error; a wait that ran out leaves
 * an empty route map. Nothing is synchronised.
 */
estream_status estream_route_build_from_x(const void* X, int T, int H, const void* W_r, int E,
                                          int k, int renorm, const int32_t* phi, int P,
                                          float* logits, int32_t* topk_ids, float* alpha,
                                          int32_t* offsets, int32_t* rec_tok, int32_t* rec_route,
                                          void* workspace, size_t workspace_bytes,
                                          void* cuda_stream);

/* 1 if estream_route_build_from_x (and estream_moe_layer_prefill_from_x)
 * run these sizes as one fused launch on the current device, 0 if as two. */
int estream_route_build_from_x_fused(int T, int H, int E, int P);

/*
 * estream_route_build without a workspace argument, for callers that cannot
 * give this library device scratch memory (for example a serving process
 * that reserved all device memory up front and allows no cudaMalloc on its
 * request path, since an allocation there can synchronise the device or fail
 * once the budget is carved up). The paper has no counterpart of this call.
 * Inputs, outputs and results are those of estream_route_build; it allocates
 * nothing. Its scratch is a 1 MiB file-scope device array held by every GPU
 * that loads the library until the process exits:
 *   - sizes whose estream_route_workspace_bytes(T, E, k, P) exceeds 1 MiB are
 *     rejected with ESTREAM_ERR_CAPACITY before anything is enqueued;
 *   - all calls on a device share the array, which keeps the previous call's
 *     contents; each call clears what must start at zero on its own stream;
 *     calls whose GPU work overlaps (other streams, unordered threads) race
 *     on it and give wrong results;
 *   - the first call on a device looks the array's address up (with that
 *     device current); make it before any stream capture on the device;
 *   - errors found by the kernel (a phi entry outside [-1, P), a grid
 *     barrier that gave up) are kept in the array's error word, which
 *     estream_route_noalloc_error reads;
 *   - logits and the outputs must be memory of the current device
 *     (ESTREAM_ERR_INVALID_ARG otherwise).
 */
estream_status estream_route_build_noalloc(const float* logits, int T, int E, int k, int renorm,
                                           const int32_t* phi, int P,
                                           int32_t* topk_ids, float* alpha, int32_t* offsets,
                                           int32_t* rec_tok, int32_t* rec_route,
                                           void* cuda_stream);

/* Synchronises `cuda_stream`, then returns and clears the error word that
 * estream_route_build_noalloc calls on the current device recorded in the
 * static scratch array: ESTREAM_OK if none, ESTREAM_ERR_DEVICE for a phi
 * entry outside [-1, P) (that route was filed under the trailing bucket),
 * ESTREAM_ERR_TIMEOUT when a grid barrier of the route build gave up after
 * its 1 s bound (that call left an empty route map: offsets all zero).
 * Every call of estream_route_build_noalloc clears the word when it starts,
 * so it reports the latest call on the device: read it after the call whose
 * result matters, before the next one. */
estream_status estream_route_noalloc_error(void* cuda_stream);

/* ---------------------------------------------------------------------- */
/* Expert arena, pager and layer prefill                                   */
/* ---------------------------------------------------------------------- */

enum {
    ESTREAM_SCHED_AFTER_ROUTING = 0, /* start copies once the routes are known */
    ESTREAM_SCHED_PREFETCH = 1       /* also fill free banks in storage order before routing */
};

/* Form of the bf16 fused expert kernel (no counterpart in the paper, whose
 * NPU has one matrix unit per core). SINGLE: 128-record tiles, one SM each.
 * PAIR: 256-record tiles on a cluster of two SMs (tcgen05.mma.cta_group::2),
 * each SM holding half of every weight tile: less shared-memory and L2
 * traffic per FLOP, but up to 255 padded rows per expert instead of 127.
 * AUTO: PAIR when an expert segment holds on average at least
 * ESTREAM_PAIR_MIN_ROWS records (T*k/E for routed experts, T for shared
 * ones; the measured crossover lies between 128 and 192), else SINGLE. */
enum {
    ESTREAM_FFN_AUTO = 0,
    ESTREAM_FFN_SINGLE = 1,
    ESTREAM_FFN_PAIR = 2
};
#define ESTREAM_PAIR_MIN_ROWS 160

typedef struct {
    int L;                  /* sparse layers whose experts stream through this arena */
    int E, H, F;            /* routed experts per layer, hidden size, expert FFN size */
    int G, B;               /* experts per storage group (= slots per bank), banks; P = B*G */
    int Q;                  /* reads in flight: Q copy streams, group fill k on stream k mod Q (>= 1) */
    estream_dtype wdtype;   /* arithmetic types of X and the weights (estream_dtype) */
    void* arena_dev;        /* device, >= estream_arena_bytes(...) bytes, 1024-byte aligned */
    size_t arena_bytes;
    const void* const* host_pool;   /* host array [L] of pinned pools, each laid out by
                                       estream_pack_experts */
    const int32_t* perm;    /* host, [L*E]: pi_l(e), the storage order; NULL = identity */
    int n_shared, F_shared; /* always-on shared experts per layer (weight 1), their FFN size */
    const void* const* shared_dev;  /* host array [L] of device pointers, each to one layer's
                                       shared experts as laid out by estream_pack_shared;
                                       NULL if none */
    int T_max, k_max;       /* largest T and k a layer call will see (workspace capacity) */
    int deterministic;      /* 1: per-route outputs + fixed-order combine (bit-reproducible Y) */
    int schedule;           /* ESTREAM_SCHED_* */
    int ffn_form;           /* ESTREAM_FFN_* (fp32 ignores it; Q4 follows the same rule, its
                               CTA-pair form expanding half of every packed weight tile per SM) */
} estream_arena_desc;

typedef struct estream_ctx estream_ctx;

/* Bytes of arena for P = B*G slots of one expert each (gate, up, down). */
size_t estream_arena_bytes(int E, int H, int F, int G, int B, estream_dtype wdtype);

/* Bytes of one layer's pinned host pool: E experts, group-contiguous, then
 * E fp32 down-weight scales in storage order (see estream_pack_experts). */
size_t estream_pool_bytes(int E, int H, int F, estream_dtype wdtype);

/* Bytes of one layer's packed shared experts (see estream_pack_shared). */
size_t estream_shared_bytes(int n_shared, int H, int F_shared, estream_dtype wdtype);

/*
 * Validate `d`, compute the slot addresses of Eq. 3 and their TMA
 * descriptors, create the copy stream and the per-bank events, and allocate
 * the library workspace (sized for T_max, k_max). Copies no weights.
 * Shapes: H % 256 == 0, F % 128 == 0, F_shared % 128 == 0, 1 <= G, 1 <= B,
 * 1 <= E <= 1024. On success *out is a context owned by the caller, to be
 * released with estream_unbind. The current CUDA device is the one used;
 * every later call on the context must be made with that device current
 * (ESTREAM_ERR_INVALID_ARG otherwise).
 */
estream_status estream_bind_arena(estream_ctx** out, const estream_arena_desc* d);

/*
 * Offline repack (host -> host) of one layer's expert weights into the
 * layout the kernels consume and the pager streams (section 3.3, "Offline
 * NPU-Consumable Weight Layout", restated for GB300). For storage group q
 * (experts with pi(e) in [q*G, q*G+G)), in pi order, at byte offset q*G*W_e:
 * [gate n_q x F x H][up n_q x F x H][down n_q x H x F], W_e = 3*H*F*elem.
 * After the last group: E fp32 scales, one per storage position.
 * bf16 layers: gate and up are copied unchanged; the down plane is stored
 * as fp16 of (W_d * 2^s_e), with s_e = 15 - (binary exponent of max|W_d[e]|)
 * so the largest magnitude lands in [2^14, 2^15); the stored scale is 2^-s_e
 * and the down GEMM multiplies it back in. The conversion is exact for every
 * weight within a factor 2^32 of the expert's largest one. fp32 layers are
 * copied unchanged with scale 1.
 * Q4 layers (from bf16 master weights): each plane is quantised in blocks of
 * 32 weights along its reduction dimension (H for gate and up, F for down;
 * the down weights first multiplied by 2^s_e as above). Block scale: the
 * element of largest magnitude m (the first on ties) gives d = m / -8
 * rounded to 5 significant bits (ties to even), then to bf16 (gate, up) or
 * fp16 (down); codes q = clamp(rint(w / d) + 8, 0, 15) (fp32 division, ties
 * to even); a zero block has d = 0 and codes 8. The weight used is
 * (q - 8) * d, exact in the operand type. Layout: tile-major boxes of
 * (R = 128 rows of gate/up or 256 rows of down) x 64 weights, each box
 * being two column blocks of codes -- block j holds every row's 16 bytes of
 * weights 32j..32j+31 (in byte-word w of a row, bits 4i..4i+3 hold weight
 * 32j + 8w + 2i and bits 16 + 4i.. weight 32j + 8w + 2i + 1) -- followed by
 * the rows' two block scales (uint16 bits); W_e = 3 * H * F * 9 / 16 bytes.
 * wg, wu: host [E][F][H]; wd: host [E][H][F] (fp32 for F32, bf16 for BF16 and Q4);
 * host_pool_out: host, estream_pool_bytes(...) bytes (pinned if streamed).
 * Only d->E, H, F, G, wdtype and perm (row `layer`) are read. Pools must be
 * packed before estream_bind_arena (which reads their scales).
 */
estream_status estream_pack_experts(const estream_arena_desc* d, int layer,
                                    const void* wg, const void* wu, const void* wd,
                                    void* host_pool_out);

/*
 * Repack (host -> host) of one layer's shared experts into
 * [gate n_shared x F_shared x H][up (same)][down n_shared x H x F_shared]
 * [n_shared fp32 scales], with the down plane converted as in
 * estream_pack_experts. The caller copies the result to device memory and
 * passes it in estream_arena_desc.shared_dev. sg, su: host
 * [n_shared][F_shared][H]; sd: host [n_shared][H][F_shared];
 * out: host, estream_shared_bytes(...) bytes. Reads d->n_shared, F_shared,
 * H and wdtype.
 */
estream_status estream_pack_shared(const estream_arena_desc* d, const void* sg,
                                   const void* su, const void* sd, void* out);

/*
 * Load every group of `layer` into the arena and keep it there (needs
 * B*G >= E, i.e. ceil(E/G) <= B). Later calls for that layer copy nothing
 * and run each kernel once over all experts. Enqueued on the copy stream;
 * the first layer call waits for it.
 */
estream_status estream_arena_preload(estream_ctx* c, int layer, void* cuda_stream);

/* Forget every bank's contents (the next call streams again). Waits for
 * in-flight work on the library's streams. */
estream_status estream_arena_invalidate(estream_ctx* c);

/*
 * One MoE layer's prefill: Y += sum_j alpha_{t,j} F_{e_{t,j}}(X_t) (+ the
 * shared experts with weight 1), i.e. Eq. 2 with Y holding A_t on entry.
 * X       device, [T][H] of d->wdtype, 16-byte aligned.
 * logits  device, [T][E] fp32 (the router's logits for this layer).
 * T, k    1 <= T <= T_max, 1 <= k <= min(k_max, E); renorm as in route_build.
 * Y       device, [T][H] fp32, read and written.
 * Steps: routing + route map over the storage order (K1), then per group
 * with routes: bank fill on the copy stream (skipped when already resident),
 * gate/up GEMM with the row gather and SiLU-mul fused (K2), down GEMM with
 * the alpha-weighted scatter-add into Y (K3). When some group is not
 * resident, the call copies the per-slot offsets to the host and
 * synchronises `cuda_stream` once (after routing). All later GPU work of the
 * call is ordered before any later work on `cuda_stream`.
 */
estream_status estream_moe_layer_prefill(estream_ctx* c, int layer, const void* X,
                                         const float* logits, int T, int k, int renorm,
                                         float* Y, void* cuda_stream);

/*
 * The same layer with the residual of Eq. 2 given explicitly:
 * Y = A + sum_j alpha_{t,j} F_{e_{t,j}}(X_t) (+ shared experts). Y is written,
 * not read: the call initialises the rows from A itself -- the route build
 * beside its ranking of the tokens' experts, or, when T exceeds the rows it
 * covers there (bf16 and Q4 contexts), the first expert kernel before its
 * first tile -- so the caller needs no separate copy of A into Y.
 * A       device, [T][H] in X's type (bf16, or fp32 for ESTREAM_F32), 16-byte
 *         aligned; A == X (the usual residual stream) is allowed.
 * The other arguments and the behaviour are those of
 * estream_moe_layer_prefill.
 */
estream_status estream_moe_layer_prefill_residual(estream_ctx* c, int layer, const void* X,
                                                  const float* logits, int T, int k, int renorm,
                                                  const void* A, float* Y, void* cuda_stream);

/*
 * The layer call with routing from the layer input: router logits
 * X W_r^T, top-k and route map in one launch (estream_route_build_from_x),
 * then the experts as in estream_moe_layer_prefill.
 * W_r        device, [E][H] bf16 (one row per expert), 16-byte aligned.
 * A          NULL: Y is accumulated into (Y += ...); else the residual of
 *            Eq. 2 as in estream_moe_layer_prefill_residual (Y written; the
 *            routing launch initialises the rows beside its router tile, or
 *            past the rows it covers there, the first expert kernel does).
 * logits_out device, [T][E] fp32, or NULL: receives the router logits.
 * Contexts of type ESTREAM_F32 are refused (ESTREAM_ERR_INVALID_ARG). The
 * other arguments and the behaviour are those of estream_moe_layer_prefill.
 */
estream_status estream_moe_layer_prefill_from_x(estream_ctx* c, int layer, const void* X,
                                                const void* W_r, int T, int k, int renorm,
                                                const void* A, float* Y, float* logits_out,
                                                void* cuda_stream);

/* Timings and counters accumulated since the last estream_reset_stats. The
 * per-kernel times are CUDA-event times on the launching stream, recorded
 * only while timing is on (estream_set_timing); reading them synchronises. */
typedef struct {
    int calls;
    int launches;            /* kernels this library enqueued (memsets and copies not counted) */
    double ms_route;         /* routing + route map (memset + one kernel) */
    double ms_ffn;           /* routed fused expert kernel (gather, gate/up, SwiGLU, down, scatter) */
    double ms_shared;        /* shared experts (identity map + fused expert kernel) */
    double ms_combine;       /* deterministic combine */
    double ms_total;         /* first to last event of each call, summed */
    int n_ffn;               /* routed fused expert launches counted in ms_ffn */
    double h2d_bytes;        /* bytes copied into the arena */
    int groups_loaded, groups_skipped, groups_hit;
    double ms_io_busy;       /* copy-stream busy time (timing on) */
    /* Overlap of loading and execution over the same calls (timing on), with
     * T_io = ms_io_busy, T_exec = ms_route + ms_ffn + ms_shared + ms_combine
     * and T_total = ms_total:
     *   hidden_fraction = (T_io + T_exec - T_total) / T_io, clamped to [0, 1]:
     *     the share of the copy time that ran under execution (0 when nothing
     *     was copied);
     *   bubble_rate = 1 - max(T_io, T_exec) / T_total, clamped to [0, 1]: the
     *     paper's bubble rate (section 3.4, Fig. 6 caption). */
    double hidden_fraction;
    double bubble_rate;
} estream_stats;

estream_status estream_set_timing(estream_ctx* c, int on);
estream_status estream_reset_stats(estream_ctx* c);
estream_status estream_last_stats(estream_ctx* c, estream_stats* out);

/* Test aid for the cross-CTA ordering of the fused kernels: enqueues on
 * `cuda_stream` a fill of every per-call buffer of the context's workspace
 * (top-k ids, alpha, route records and offsets, the route build's scratch,
 * the h intermediates, the deterministic mode's row buffers) with all-ones
 * bytes -- NaN for the floating-point buffers -- and of the m-block
 * completion counters and tile tickets with 0x7f bytes (a count past every
 * target). A layer call after it must give the same Y as without it: every
 * buffer is written before it is read, and every counter is zeroed by the
 * call before it is waited on. The bind-time tables (storage order, down
 * scales) and the error word are left alone. Not for production use. */
estream_status estream_poison_workspace(estream_ctx* c, void* cuda_stream);

/* Synchronises the library's streams, returns and clears the device error
 * words (ESTREAM_OK, ESTREAM_ERR_TIMEOUT or ESTREAM_ERR_DEVICE): the
 * context's, set by the expert kernels and kept until read, and the route
 * build's, set by the latest call's routing. A route build whose grid
 * barrier gave up leaves an empty route map, so the call computes no routed
 * experts and this call reports ESTREAM_ERR_TIMEOUT. */
estream_status estream_get_device_error(estream_ctx* c);

/* Residency-table trace for tests: writes up to `cap` events as
 * (bank, layer, group, state) int32 quadruples and returns their count in
 * *n (states: 0 Available, 1 Filling, 2 Ready, 3 InUse). Tracing is kept for
 * the last call only. */
estream_status estream_residency_trace(estream_ctx* c, int32_t* out, int cap, int* n);

/* Per-group pipeline trace of the last paged layer call made with timing on
 * (estream_set_timing): for each group filled by that call, in order, the
 * times in ms since the call began at which its read started (a) and ended
 * (d) on its copy stream and its execution started (s) and ended (f) on the
 * compute stream -- the quantities of EStream section 3.4, Eq. 5 (a group
 * filled before routing and then found empty has s = f, no execution). adsf:
 * host [cap][4]; *n receives the number of groups; *t_ne (optional) the time
 * routing finished. Synchronises on the recorded events. */
estream_status estream_pipeline_trace(estream_ctx* c, double* adsf, int cap, int* n,
                                      double* t_ne);

/* ---------------------------------------------------------------------- */
/* Pipeline model and automatic configuration (host only)                 */
/* ---------------------------------------------------------------------- */

/*
 * Max-plus recurrence of EStream section 3.4, Eq. 5, over K groups:
 *   a_k = max(d_{k-q}, f_{k-b}), d_k = a_k + L_k,
 *   s_k = max(d_k, T_ne, f_{k-1}), f_k = s_k + X_k, with d_j = f_j = 0 for j <= 0.
 * L, X: host [K] read and execution times; q >= 1 reads in flight; b >= 1
 * banks. Returns T_pipe = f_K (T_ne when K = 0; -1 on bad arguments) and,
 * if adsf is not NULL, writes (a_k, d_k, s_k, f_k) to adsf[4(k-1) .. +3].
 */
double estream_maxplus_pipeline(const double* L, const double* X, int K, int q, int b,
                                double T_ne, double* adsf);

/* Eq. 8: largest feasible bank count for group size g under a memory budget:
 * min(floor((M_max - M_other) / (g * W_e)), ceil(N_e / g)); 0 if none. */
int estream_bank_bound(int g, double M_max, double M_other, double W_e, int N_e);

/*
 * Eqs. 9-10: for each candidate group size g_values[i] (with its calibrated
 * per-group read times L_per_g[i][0..K_per_g[i]) and execution times
 * X_per_g[i][...] from one profiled call, e.g. estream_pipeline_trace),
 * choose B*(g) = argmin over Q0 <= b <= B_max(g) of T_pipe, then G* =
 * argmin over feasible g of T_pipe(g, Q0, B*(g)). Ties keep the smaller b
 * and the earlier g. M_other_per_g may be NULL (0). Writes *G_out, *B_out
 * and (if not NULL) the predicted *T_out; ESTREAM_ERR_CAPACITY if no g is
 * feasible (B_max(g) < Q0 for all).
 */
estream_status estream_autoconfig(int n_g, const int* g_values, const int* K_per_g,
                                  const double* const* L_per_g, const double* const* X_per_g,
                                  double T_ne, int Q0, double M_max, const double* M_other_per_g,
                                  double W_e, int N_e, int* G_out, int* B_out, double* T_out);

/* Test of the route build's bounded grid barrier: in the next layer call one
 * CTA of the route build does not arrive at its first grid barrier, so the
 * other CTAs' wait (1 s) runs out. That call leaves an empty route map
 * (no routed expert is computed; the residual rows, if given, are written),
 * returns ESTREAM_OK, and estream_get_device_error then reports
 * ESTREAM_ERR_TIMEOUT. Later calls are unaffected. No GPU fault is involved. */
estream_status estream_inject_route_timeout(estream_ctx* c);

/* Test of the expert kernels' bounded waits: the next layer call runs the
 * routed expert kernels' down tiles without their gate/up tiles, so each down
 * tile's wait for its m-block's h rows (2 s) runs out. Every CTA then stops,
 * lets the copies and MMAs it issued complete, frees its tensor memory and
 * returns; the call returns ESTREAM_OK and estream_get_device_error reports
 * ESTREAM_ERR_TIMEOUT. Y then holds no routed contribution. Later calls are
 * unaffected. No GPU fault is involved. */
estream_status estream_inject_expert_timeout(estream_ctx* c);

/* Host-side fault injection for tests: the pager refuses to fill group
 * `group` of `layer` (before any copy is issued) and the call returns
 * ESTREAM_ERR_PAGER with the streams drained. group < 0 turns it off. */
estream_status estream_inject_pager_fault(estream_ctx* c, int layer, int group);

/* Drains the library's streams and frees everything the library owns
 * (workspace, streams, events, the context). Caller memory is untouched. */
void estream_unbind(estream_ctx* c);

/* fp32 -> bf16 (round to nearest even) of n elements, device to device;
 * used to chain layers (X_{l+1} = bf16(Y_l)). */
estream_status estream_cast_f32_bf16(const float* src, void* dst, size_t n, void* cuda_stream);

#ifdef __cplusplus
}
#endif

#endif /* ESTREAM_H */
