// Internal declarations shared by the CUDA translation units of libestream.
// Not installed; the public ABI is include/estream.h.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "estream.h"

namespace es {

// Rows of one GEMM M tile (route records per tile).
constexpr int kBM = 128;
// Limits checked at the boundary.
constexpr int kMaxE = 1024;
constexpr int kMaxK = 32;
constexpr int kMaxP = 4096;

// Device error word values (first error wins).
constexpr int kDevErrNone = 0;
constexpr int kDevErrSlotRange = 1;  // a phi entry outside [-1, P)
constexpr int kDevErrTimeout = 2;    // a bounded wait ran out
constexpr int kDevErrRange = 3;      // an intermediate h value outside the fp16 range
constexpr int kDevErrLaunch = 4;     // a cluster kernel launched without its cluster shape

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Layout of the route-build workspace (all offsets 256-byte aligned).
struct RouteWorkspace {
    size_t err_off;      // int32 device error word
    size_t sync_off;     // int32 grid-barrier counter of the fused route kernel
    size_t hist_off;     // int32 [P+1][nchunk]: per-chunk counts, then bases inside the slot
    size_t mblk_off;     // int32 [P+2]: exclusive prefix of ceil(count[s]/kBM), s < P
    size_t tot_off;      // int32 [P+1]: per-slot totals
    size_t total;
    int nchunk;
};
RouteWorkspace route_workspace_layout(int T, int k, int P);

// Optional fused initialisation Y[t][:] = fp32(A[t][:]) (the residual of
// Eq. 2), done by the route build's token warps; H a multiple of 256.
struct ResidualInit {
    const void* A;   // [T][H], bf16 (elem_bytes 2) or fp32 (4)
    int elem_bytes;
    float* Y;        // [T][H]
    int H;
};

// Enqueue the full route build (K1). `ws` holds ws_bytes bytes, which must
// cover route_workspace_layout(T,k,P) (cudaErrorInvalidValue otherwise, before
// anything is enqueued: a second guard behind every entry point's own check).
// rec_pos (optional, [T*k]) receives, for route i, its position in the CSR.
// done (optional) is zeroed over the route map's m-blocks (mblk[P] ints) for
// the fused expert kernel's m-block counters, and tickets[0..n_tickets) (the
// dynamic tile counters of the call's expert-kernel launches) as well.
cudaError_t launch_route_build(const float* logits, int T, int E, int k, int renorm,
                               const int32_t* phi, int P, int32_t* topk_ids, float* alpha,
                               int32_t* offsets, int32_t* rec_tok, int32_t* rec_route,
                               int32_t* rec_pos, int32_t* done, int32_t* tickets, int n_tickets,
                               void* ws, size_t ws_bytes, cudaStream_t stream, int* n_launches,
                               const ResidualInit* resid = nullptr, int withhold_arrival = 0,
                               bool clear_err = true);

// Router logits fused with the route build: one cooperative launch of
// clusters from X [T][H] and W_r [E][H] (bf16) to the route map (and, when
// `logits` is given, the logits [T][E] fp32), with the same outputs, optional
// residual rows and test hook as launch_route_build. Shapes it
// cannot take (E > 128, H not a multiple of 64, more token tiles than
// resident clusters) return cudaErrorNotSupported before anything is
// enqueued; the caller then runs the router and the route build separately.
struct FusedRoutePlan {
    bool ok;
    int S, N, m_tiles, KB;  // CTAs per token tile (cluster), experts per tile, tiles, k-blocks
    size_t smem;
};
FusedRoutePlan fused_route_plan(int T, int H, int E, int P);
cudaError_t launch_route_from_x(const void* X, int T, int H, const void* W_r, int E, int k,
                                int renorm, const int32_t* phi, int P, float* logits,
                                int32_t* topk_ids, float* alpha, int32_t* offsets,
                                int32_t* rec_tok, int32_t* rec_route, int32_t* rec_pos,
                                int32_t* done, int32_t* tickets, int n_tickets, void* ws,
                                size_t ws_bytes, cudaStream_t stream, int* n_launches,
                                const ResidualInit* resid = nullptr, int withhold_arrival = 0);

// Identity route map for the shared experts: n_shared segments of T rows,
// rec_tok[p] = p mod T, offsets[s] = s*T, mblk[s] = s*ceil(T/kBM); zeroes
// done[0 .. n_shared*ceil(T/kBM)).
cudaError_t launch_identity_map(int T, int n_shared, int32_t* offsets, int32_t* rec_tok,
                                int32_t* mblk, int32_t* done, cudaStream_t stream);

// ---------------------------------------------------------------------------
// Grouped expert GEMMs (K2 gate/up + SwiGLU, K3 down + weighted scatter-add)
// ---------------------------------------------------------------------------

struct GemmSegments {
    const int32_t* offsets;    // CSR offsets (indexed by segment)
    const int32_t* mblk;       // exclusive prefix of m-blocks per segment
    const int32_t* rec_tok;    // token of each record
    const int32_t* rec_route;  // route of each record (K3 alpha lookup; may be null)
    const float* alpha;        // route weights, or null for weight 1
    const float* seg_scale;    // per segment: 2^-s of the down weights' offline scale
    int seg_begin, seg_count;  // segments [seg_begin, seg_begin+seg_count)
    int slot_base;             // arena slot of segment seg_begin
    int max_tiles_m;           // host upper bound on m-blocks in the range
    // Residual rows Y = A, written by this launch's epilogue warps before
    // their first tile (the first expert launch of a layer call with a
    // residual; resid_A null otherwise): A [resid_T][H] with resid_elem bytes
    // per element (bf16 2, fp32 4) into resid_Y [resid_T][H]. Each epilogue warp then adds 1 to
    // *resid_done (zeroed by the route build), and a down epilogue waits for
    // every epilogue warp of the launch before it adds into Y.
    const void* resid_A;
    float* resid_Y;
    int resid_elem, resid_T;
    int* resid_done;
};

// Residual rows (T given) that the route build copies beside its top-k on
// CTAs it adds for them; rows beyond it are copied by the chunk CTAs after
// the top-k, ahead of the route build's grid barriers.
int route_residual_overlap_rows(int T);

// Y[t][:] = fp32(A[t][:]) for t < T (A bf16 or fp32 by elem_bytes): the
// residual rows of a layer call whose expert launches did not write them.
cudaError_t launch_residual_rows(const void* A, int elem_bytes, float* Y, int T, int H,
                                 cudaStream_t stream);

// Fused expert FFN (one cooperative launch), phases bit 0 / bit 1:
//   gate/up: h[p, :] = fp16(SiLU(X[tok(p)] Wg_slot^T) * (X[tok(p)] Wu_slot^T)) (bf16 MMA);
//   down:    Y[tok(p), :] += alpha(p) * scale(seg) * (h[p] Wd_slot^T) (fp16 MMA), or
//            out_rows[p, :] = ... when out_rows != null (deterministic mode).
// X: device [T][H] bf16 (16-byte aligned rows); h: [rows][F] fp16; done: one
// zeroed int per absolute m-block of the route map (mblk indices); ticket: a
// zeroed int for this launch's dynamic tile hand-out, or null for a static
// assignment.
// tm_h: TMA map of h ([rows][F] fp16, 64 x 128 boxes, 128-byte swizzle).
cudaError_t launch_expert_ffn(const CUtensorMap* tm_wg, const CUtensorMap* tm_wu,
                              const CUtensorMap* tm_wd, const CUtensorMap* tm_h,
                              const GemmSegments& seg, const void* X,
                              void* h, float* Y, float* out_rows, int* done, int* ticket, int H,
                              int F, int phases, int* dev_err, int num_sms, cudaStream_t stream);

// The same operator on CTA pairs (clusters of two, tcgen05.mma.cta_group::2,
// 256-record pair tiles, and 128-record half tiles for segment remainders);
// tm_wd_half maps the down planes with 64 x 128 boxes (each CTA loads half of
// a 256-row W_d box); tm_wg64 / tm_wu64 map the gate / up planes with 64 x 64
// boxes (a half tile's CTA loads 64 gate and 64 up rows of an n-block).
// m_first: tiles m-block-major inside a segment (for weights that stay in L2
// across m-blocks, as a shared expert's do), else n-block-major.
cudaError_t launch_expert_ffn_pair(const CUtensorMap* tm_wg, const CUtensorMap* tm_wu,
                                   const CUtensorMap* tm_wd_half, const CUtensorMap* tm_h,
                                   const CUtensorMap* tm_wg64, const CUtensorMap* tm_wu64,
                                   const GemmSegments& seg, const void* X, void* h, float* Y,
                                   float* out_rows, int* done, int H, int F, int phases,
                                   int* dev_err, bool m_first, cudaStream_t stream);

// The same operator on 4-bit weights (single-SM form): planes hold
// Q4_0-style packed boxes (see estream_pack_experts), slot s of a plane at
// plane + s * S_gu (gate, up) or s * S_d (down).
cudaError_t launch_expert_ffn_q4(const uint8_t* plane_g, const uint8_t* plane_u, const uint8_t* plane_d,
                                 size_t S_gu, size_t S_d, const CUtensorMap* tm_h,
                                 const GemmSegments& seg, const void* X, void* h, float* Y,
                                 float* out_rows, int* done, int* ticket, int H, int F, int phases,
                                 int* dev_err, int num_sms, cudaStream_t stream);

// The 4-bit operator on CTA pairs: each CTA streams and expands its half of
// every packed weight box (the pair form's tiles, without half tiles).
cudaError_t launch_expert_ffn_pair_q4(const uint8_t* plane_g, const uint8_t* plane_u,
                                      const uint8_t* plane_d, size_t S_gu, size_t S_d,
                                      const CUtensorMap* tm_h, const GemmSegments& seg,
                                      const void* X, void* h, float* Y, float* out_rows, int* done,
                                      int H, int F, int phases, int* dev_err, cudaStream_t stream);

// fp32 path (CUDA-core FMA): the same two steps for fp32 X and weights.
// Weight planes are [slots][F][H] (gate, up) and [slots][H][F] (down).
cudaError_t launch_gateup_f32(const float* X, const float* wg, const float* wu,
                              const GemmSegments& seg, float* h, int H, int F, int max_rows,
                              cudaStream_t stream);
cudaError_t launch_down_f32(const float* h, const float* wd, const GemmSegments& seg, float* Y,
                            float* out_rows, int H, int F, int max_rows, cudaStream_t stream);

// K4: Y[t, :] += sum_j rows[pos[t*k+j], :] (j ascending), then
// + sum_s shared_rows[s*T + t, :] (s ascending) when n_shared > 0.
cudaError_t launch_combine(const float* rows, const int32_t* pos, int T, int k, int H,
                           const float* shared_rows, int n_shared, float* Y,
                           cudaStream_t stream);

// Router logits l[T][E] = X[T][H] W_r[E][H]^T (bf16 in, fp32 out) on the
// tensor cores, K split S <= 8 ways across the CTAs of one cluster.
struct RouterPlan {
    int N;              // experts per tile (multiple of 16, <= 256)
    int m_tiles, n_tiles, KB, S;
    size_t partial_bytes;  // device scratch beyond the error word (0)
};
RouterPlan router_plan(int T, int H, int E, int num_sms);
cudaError_t launch_router_logits(const void* X, int T, int H, const void* W_r, int E, float* logits,
                                 const RouterPlan& p, int* dev_err, cudaStream_t stream);

cudaError_t launch_cast_f32_bf16(const float* src, void* dst, size_t n, cudaStream_t stream);

// Tensor-map helper (driver entry point resolved at run time).
CUresult encode_tmap_2d(CUtensorMap* tm, CUtensorMapDataType dtype, const void* base,
                        uint64_t inner, uint64_t outer, uint64_t row_stride_bytes,
                        uint32_t box_inner, uint32_t box_outer);

}  // namespace es
