// K1: router top-k and the route map (CSR of records by physical slot).
//
// "EStream: Fast and Memory-Efficient MoE Prefill through Expert
// Virtualization on Mobile NPUs", section 3.2 ("Composed Sparse Route and
// Parameter Binding") and Algorithm 1 (route-map construction): every route i
// (token t_i, logical expert e_i, weight alpha_i) is resolved to its slot
// psi_i = Phi(e_i); routes are counted per slot, an exclusive prefix sum
// gives where each slot's records begin, and a second pass stores (t_i, i)
// contiguously by slot, in ascending i. Routes whose expert is not resident
// (Phi = -1) are filed under a trailing bucket P.
//
// GPU form: one 8-byte memset, then one cooperative kernel (k_route_fused)
// in three phases separated by bounded grid barriers. Routes are processed in
// chunks of kChunkTokens tokens (16 * k routes):
//   1. one CTA per chunk, one warp per token: softmax top-k, alpha, and the
//      chunk's slot counts (shared-memory atomics; counts are order-free),
//      written bucket-major as hist[slot][chunk]; with a residual A the
//      rows Y[t] = A[t] are written in the same phase, by the warps of CTAs
//      added for them first (those CTAs then leave: the later phases and
//      their grid barriers involve the chunks' CTAs only);
//   2. every warp of the chunks' CTAs scans whole slots (a warp per slot):
//      each chunk's base inside the slot, and the slot's total;
//   3. every CTA forms the slot offsets and the m-block prefix (the expert
//      kernel schedules by it) from the slot totals with block scans in its
//      shared memory -- CTA 0 also stores them -- then, one CTA per chunk,
//      places the chunk's records: ranks inside a warp by __match_any_sync,
//      across warps in ascending order, so the placement is the stable one
//      Algorithm 1 produces.
// A grid barrier that gives up (1 s) records a timeout in the error word and
// leaves an empty route map, so that kernels reading it find no records.
#include <cuda_bf16.h>

#include <algorithm>
#include <mutex>

#include "estream_internal.h"

namespace es {
namespace {
#include "tc_ptx.cuh"
#include "router_tile.cuh"
}  // namespace

// ---------------------------------------------------------------------------
// Written fp32 exponential, the same written definition the CPU oracle uses,
// implemented here on its own so both sides round identically:
//   x < -87 -> 0; n = nearest-even(fl(x * LOG2E));
//   r = fma(-n, LN2_HI, x); r = fma(-n, LN2_LO, r)   (Cody & Waite, 1980)
//   p = Horner of sum_{j<=7} r^j/j!, one fma per step;  result = p * 2^n.
// LN2_HI = fp32(ln 2) with its 8 low significand bits cleared, LN2_LO =
// fp32(ln 2 - LN2_HI); LOG2E and 1/j! are round-to-nearest fp32 values.
// Every operation is an explicit round-to-nearest intrinsic (no contraction).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float route_exp(float x) {
    if (x < -87.0f) return 0.0f;
    const float kLog2e = 0x1.715476p+0f;
    const float kLn2Hi = 0x1.62e4p-1f;
    const float kLn2Lo = 0x1.7f7d1cp-20f;
    const int n = __float2int_rn(__fmul_rn(x, kLog2e));
    const float nf = static_cast<float>(n);
    float r = __fmaf_rn(-nf, kLn2Hi, x);
    r = __fmaf_rn(-nf, kLn2Lo, r);
    float p = 0x1.a01a02p-13f;           // 1/7!
    p = __fmaf_rn(p, r, 0x1.6c16c2p-10f);  // 1/6!
    p = __fmaf_rn(p, r, 0x1.111112p-7f);   // 1/5!
    p = __fmaf_rn(p, r, 0x1.555556p-5f);   // 1/4!
    p = __fmaf_rn(p, r, 0x1.555556p-3f);   // 1/3!
    p = __fmaf_rn(p, r, 0.5f);             // 1/2!
    p = __fmaf_rn(p, r, 1.0f);             // 1/1!
    p = __fmaf_rn(p, r, 1.0f);             // 1/0!
    return __fmul_rn(p, __int_as_float((n + 127) << 23));
}

// One warp per token; lane l holds the logits of experts l, l+32, l+64, ...
// The softmax denominator is summed in ascending expert order (the same
// sequence of fp32 additions as the written definition): the warp streams the
// per-expert exponentials to every lane with shuffles, one expert at a time.
// Selection walks the strict total order (logit descending, expert id
// ascending): round j takes the best expert after round j-1's pick in that
// order. Each logit is mapped to an unsigned key of the same order (-0 taken
// as +0, which compares equal to it), so a round is one warp-wide max of the
// keys and one min of the ids holding it. Lane j then forms route j's weight.
constexpr int kMaxPerLane = kMaxE / 32;
constexpr int kRouteThreads = 512;
constexpr int kChunkTokens = kRouteThreads / 32;  // one token per warp
constexpr uint64_t kGridWaitLimitNs = 1000000000ull;  // 1 s

// kJ: logits held per lane (E <= 32 kJ), so that small E keeps the arrays in
// registers.
// l: the token's E logits (global or shared memory).
template <int kJ>
__device__ __forceinline__ void topk_token(
    int t, const float* l, int E, int k, int renorm,
    const int32_t* __restrict__ phi, int P, int32_t* __restrict__ topk_ids,
    float* __restrict__ alpha, int* counts, int* __restrict__ err) {
    const int lane = threadIdx.x & 31;
    const int nj = (E + 31) >> 5;
    const float kNegInf = __int_as_float(0xff800000);
    float v[kJ];
#pragma unroll
    for (int j = 0; j < kJ; ++j) {
        const int e = lane + 32 * j;
        v[j] = (j < nj && e < E) ? l[e] : kNegInf;
    }
    float m = kNegInf;
#pragma unroll
    for (int j = 0; j < kJ; ++j) m = fmaxf(m, v[j]);
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, d));

    // denominator: sequential fp32 sum over e = 0, 1, ..., E-1
    float s = 0.0f;
#pragma unroll
    for (int j = 0; j < kJ; ++j) {
        if (j >= nj) break;
        const int e = lane + 32 * j;
        const float p = (e < E) ? route_exp(__fsub_rn(v[j], m)) : 0.0f;
        const int n_here = min(32, E - 32 * j);
        if (n_here == 32) {
#pragma unroll
            for (int src = 0; src < 32; ++src) s = __fadd_rn(s, __shfl_sync(0xffffffffu, p, src));
        } else {
            for (int src = 0; src < n_here; ++src)
                s = __fadd_rn(s, __shfl_sync(0xffffffffu, p, src));
        }
    }

    // order-preserving keys (entries past E are never candidates)
    uint32_t key[kJ];
#pragma unroll
    for (int j = 0; j < kJ; ++j) {
        const uint32_t b = __float_as_uint(__fadd_rn(v[j], 0.0f));  // -0 -> +0
        key[j] = (j < nj && lane + 32 * j < E) ? ((b & 0x80000000u) ? ~b : (b | 0x80000000u)) : 0u;
    }
    uint32_t prev_k = 0xffffffffu;  // every expert comes after it
    uint32_t prev_i = 0u;           // with prev_k = max, ids compare as "after" from 0 on
    bool first = true;
    uint32_t key_mine = 0u;  // lane j keeps route j's key and expert
    int id_mine = -1;
    for (int r = 0; r < k; ++r) {
        uint32_t bk = 0u, bi = 0xffffffffu;
#pragma unroll
        for (int j = 0; j < kJ; ++j) {
            if (j >= nj) break;
            const uint32_t e = static_cast<uint32_t>(lane + 32 * j);
            if (static_cast<int>(e) >= E) break;
            const bool after_prev =
                first || key[j] < prev_k || (key[j] == prev_k && e > prev_i);
            if (after_prev && (key[j] > bk || (key[j] == bk && e < bi))) {
                bk = key[j];
                bi = e;
            }
        }
        const uint32_t mk = __reduce_max_sync(0xffffffffu, bk);
        const uint32_t mi = __reduce_min_sync(0xffffffffu, bk == mk ? bi : 0xffffffffu);
        prev_k = mk;
        prev_i = mi;
        first = false;
        if (lane == r) {
            key_mine = mk;
            id_mine = static_cast<int>(mi);
        }
    }
    float a_mine = 0.0f;
    if (lane < k) {
        const float bv = __uint_as_float((key_mine & 0x80000000u) ? (key_mine & 0x7fffffffu) : ~key_mine);
        a_mine = __fdiv_rn(route_exp(__fsub_rn(bv, m)), s);
    }
    if (renorm) {
        float z = 0.0f;  // summed in rank order
        for (int r = 0; r < k; ++r) z = __fadd_rn(z, __shfl_sync(0xffffffffu, a_mine, r));
        a_mine = __fdiv_rn(a_mine, z);
    }
    if (lane < k) {
        const int i = t * k + lane;
        topk_ids[i] = id_mine;
        alpha[i] = a_mine;
        // no candidate is selected only for logits outside the contract (a
        // row of NaNs with every bit set): file the route as unresolved
        int slot = id_mine < 0 ? P + 1 : (phi ? phi[id_mine] : id_mine);
        if (slot < -1 || slot >= P) {
            record_error(err, kDevErrSlotRange);
            slot = -1;
        }
        const int b = slot < 0 ? P : slot;
        atomicAdd(&counts[b], 1);
    }
}

// Y[t][:] = fp32(A[t][:]), one warp per row (16-byte vectors; H % 256 == 0).
// The first kResidStageBytes of the row are fetched into a per-warp
// shared-memory stage with cp.async before the warp ranks its token, so the
// load latency overlaps the top-k; the rest of a longer row is copied
// directly afterwards.
constexpr int kResidStageBytes = 4096;
constexpr int kResidStageCta = kChunkTokens * kResidStageBytes;  // per CTA: one stage per warp

// Issues the copies of row t's first bytes into `stage`; returns their count.
__device__ __forceinline__ int stage_residual_row(int t, const ResidualInit& r, char* stage) {
    const int lane = threadIdx.x & 31;
    const int row_bytes = r.H * r.elem_bytes;
    const int staged = min(row_bytes, kResidStageBytes);
    const char* src = static_cast<const char*>(r.A) + static_cast<size_t>(t) * row_bytes;
    const uint32_t dst = static_cast<uint32_t>(__cvta_generic_to_shared(stage));
    for (int off = lane * 16; off < staged; off += 32 * 16)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst + off), "l"(src + off)
                     : "memory");
    asm volatile("cp.async.commit_group;" ::: "memory");
    return staged;
}

// Widens bytes [b0, b1) of row t (taken from `src`, shared or global) into Y.
__device__ __forceinline__ void widen_residual(const ResidualInit& r, int t, const char* src,
                                               int b0, int b1) {
    const int lane = threadIdx.x & 31;
    float* y = r.Y + static_cast<size_t>(t) * r.H;
    for (int off = b0 + lane * 16; off < b1; off += 32 * 16) {
        const uint4 v = *reinterpret_cast<const uint4*>(src + off);
        if (r.elem_bytes == 2) {  // 8 bf16: a bf16 is the high half of its fp32
            float4* d = reinterpret_cast<float4*>(y + off / 2);
            d[0] = make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xFFFF0000u),
                               __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xFFFF0000u));
            d[1] = make_float4(__uint_as_float(v.z << 16), __uint_as_float(v.z & 0xFFFF0000u),
                               __uint_as_float(v.w << 16), __uint_as_float(v.w & 0xFFFF0000u));
        } else {
            *reinterpret_cast<uint4*>(y + off / 4) = v;
        }
    }
}

// Completes row t: the staged bytes from shared memory, the rest from A.
__device__ __forceinline__ void finish_residual_row(int t, const ResidualInit& r, const char* stage,
                                                    int staged) {
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncwarp();
    widen_residual(r, t, stage, 0, staged);
    const int row_bytes = r.H * r.elem_bytes;
    if (staged < row_bytes)
        widen_residual(r, t, static_cast<const char*>(r.A) + static_cast<size_t>(t) * row_bytes,
                       staged, row_bytes);
}

// In-place exclusive scan of n ints in shared memory by one CTA of
// blockDim.x (multiple of 32, <= 1024) threads. Returns the total.
__device__ int block_exclusive_scan(int* data, int n, int* warp_sums) {
    const int tid = threadIdx.x;
    const int nthr = blockDim.x;
    const int per = (n + nthr - 1) / nthr;
    const int lo = min(n, tid * per);
    const int hi = min(n, lo + per);
    int local = 0;
    for (int x = lo; x < hi; ++x) local += data[x];
    const int lane = tid & 31, warp = tid >> 5;
    int incl = local;
    for (int d = 1; d < 32; d <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += v;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int nw = nthr >> 5;
        int w = lane < nw ? warp_sums[lane] : 0;
        int wi = w;
        for (int d = 1; d < 32; d <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, wi, d);
            if (lane >= d) wi += v;
        }
        if (lane < nw) warp_sums[lane] = wi - w;  // exclusive warp offsets
        if (lane == 31) warp_sums[32] = wi;       // grand total
    }
    __syncthreads();
    int run = warp_sums[warp] + incl - local;
    for (int x = lo; x < hi; ++x) {
        const int v = data[x];
        data[x] = run;
        run += v;
    }
    const int total = warp_sums[32];
    __syncthreads();
    return total;
}

// Grid-wide: warp g of the grid scans slots g, g + (warps in the grid), ...:
// hist[b][c] (counts, bucket-major) becomes the base of chunk c's first
// record inside slot b, and totals[b] the slot's count. Lane l handles a
// contiguous run of chunks, so its loads are independent of one another.
__device__ void scan_slots(int32_t* __restrict__ hist, int nchunk, int nb,
                           int32_t* __restrict__ totals, int n_part) {
    const int lane = threadIdx.x & 31;
    const int gw = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int nw = n_part * (blockDim.x >> 5);
    const int per = (nchunk + 31) / 32;
    constexpr int kRegs = 16;  // a lane's counts kept in registers up to this many
    for (int b = gw; b < nb; b += nw) {
        int32_t* row = hist + static_cast<size_t>(b) * nchunk;
        const int lo = min(nchunk, lane * per);
        const int hi = min(nchunk, lo + per);
        int vals[kRegs];
        int local = 0;
        if (per <= kRegs) {
            // every load in flight at once
#pragma unroll
            for (int j = 0; j < kRegs; ++j) vals[j] = lo + j < hi ? __ldcg(row + lo + j) : 0;
#pragma unroll
            for (int j = 0; j < kRegs; ++j) local += vals[j];
        } else {
            for (int c = lo; c < hi; ++c) local += __ldcg(row + c);
        }
        int incl = local;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl += o;
        }
        int run = incl - local;
        if (per <= kRegs) {
#pragma unroll
            for (int j = 0; j < kRegs; ++j)
                if (lo + j < hi) {
                    row[lo + j] = run;
                    run += vals[j];
                }
        } else {
            for (int c = lo; c < hi; ++c) {
                const int v = __ldcg(row + c);
                row[c] = run;
                run += v;
            }
        }
        if (lane == 31) totals[b] = incl;
    }
}

// Places the records of chunk c (the routes of tokens [c*kChunkTokens,
// (c+1)*kChunkTokens)) in passes of one route per thread.
__device__ void scatter_chunk(int c, int nchunk, const int32_t* __restrict__ topk_ids,
                              const int32_t* __restrict__ phi, int P, int k, int R,
                              const int32_t* __restrict__ base, const int* slot_off,
                              int32_t* __restrict__ rec_tok, int32_t* __restrict__ rec_route,
                              int32_t* __restrict__ rec_pos, int* cnt) {
    const int nb = P + 1;
    for (int b = threadIdx.x; b < nb; b += blockDim.x) cnt[b] = 0;
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    const int r0 = c * kChunkTokens * k;
    const int r1 = min(R, r0 + kChunkTokens * k);
    for (int pass = r0; pass < r1; pass += blockDim.x) {
        const int i = pass + threadIdx.x;
        const bool valid = i < r1;
        int b = P;
        if (valid) {
            const int e = topk_ids[i];
            const int slot = e < 0 ? -1 : (phi ? phi[e] : e);
            b = (slot < 0 || slot >= P) ? P : slot;
        }
        // the chunk's base inside the slot, loaded by every thread before the
        // warps take their turns
        const int cbase = valid ? __ldcg(base + static_cast<size_t>(b) * nchunk + c) : 0;
        const int key = valid ? b : -(lane + 1);  // invalid lanes match nobody
        const unsigned peers = __match_any_sync(0xffffffffu, key);
        const unsigned lt_mask = (1u << lane) - 1u;
        const int rank = __popc(peers & lt_mask);
        const int leader = __ffs(peers) - 1;
        int pos = 0;
        const int active_warps = min(nwarps, (r1 - pass + 31) >> 5);
        for (int w = 0; w < active_warps; ++w) {
            if (warp == w) {
                const int before = valid ? cnt[b] : 0;
                __syncwarp();
                if (valid && lane == leader) cnt[b] = before + __popc(peers);
                pos = slot_off[b] + cbase + before + rank;
            }
            __syncthreads();
        }
        if (valid) {
            rec_tok[pos] = i / k;
            rec_route[pos] = i;
            if (rec_pos) rec_pos[i] = pos;
        }
    }
    __syncthreads();
}

// Grid-wide barrier for a cooperative launch, bounded in time: returns false
// (after recording a timeout) if the other CTAs did not arrive within the limit.
// withhold: this CTA does not arrive (a test of the bounded wait: the other
// CTAs' wait runs out and records a timeout; so does this CTA's own).
// Barrier of the first n_part CTAs of the grid (those that take part in the
// route map).
__device__ bool grid_barrier(int* counter, int generation, int n_part, int* err, int* ok_flag,
                             bool withhold = false) {
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        if (!withhold) atomicAdd(counter, 1);
        const int target = generation * n_part;
        uint64_t t0;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
        int seen;
        bool ok = true;
        while (true) {
            asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(seen) : "l"(counter) : "memory");
            if (seen >= target) break;
            uint64_t t1;
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t1));
            if (t1 - t0 > kGridWaitLimitNs) {
                record_error(err, kDevErrTimeout);
                ok = false;
                break;
            }
        }
        __threadfence();
        *ok_flag = ok ? 1 : 0;
    }
    __syncthreads();
    return *ok_flag != 0;
}

// Shared memory of k_route_fused before the residual stages: slot counts /
// offsets, m-block prefix and scan scratch, rounded up to 16 bytes.
__host__ __device__ constexpr size_t route_scratch_bytes(int nb) {
    return (sizeof(int) * (2 * static_cast<size_t>(nb) + 33) + 15) & ~static_cast<size_t>(15);
}

// After a grid barrier gave up (recorded as a timeout) CTA 0 leaves an empty
// route map, so that kernels reading it find no records.
__device__ void empty_route_map(int32_t* offsets, int32_t* mblk, int P) {
    if (blockIdx.x != 0) return;
    for (int b = threadIdx.x; b < P + 2; b += blockDim.x) {
        offsets[b] = 0;
        mblk[b] = 0;
    }
}

__global__ void __launch_bounds__(kRouteThreads, 2) k_route_fused(
    const float* __restrict__ logits, int T, int E, int k, int renorm,
    const int32_t* __restrict__ phi, int P, int32_t* __restrict__ topk_ids,
    float* __restrict__ alpha, int32_t* __restrict__ offsets, int32_t* __restrict__ rec_tok,
    int32_t* __restrict__ rec_route, int32_t* __restrict__ rec_pos, int32_t* __restrict__ hist,
    int32_t* __restrict__ mblk, int32_t* __restrict__ totals, int32_t* __restrict__ done,
    int32_t* __restrict__ tickets, int n_tickets, int* __restrict__ sync, int* __restrict__ err,
    int nchunk, ResidualInit resid, int withhold_arrival) {
    extern __shared__ int smem[];
    __shared__ int ok_flag;
    const int R = T * k;
    const int nb = P + 1;
    // residual stages after the counters and scan scratch (16-byte aligned)
    const int warp = threadIdx.x >> 5;
    char* rstage = reinterpret_cast<char*>(smem) + route_scratch_bytes(nb) +
                   static_cast<size_t>(warp) * kResidStageBytes;
    // Residual rows go to every warp of the grid, those of the CTAs without a
    // top-k chunk first (the launch adds such CTAs when a residual is given),
    // so that the copies run beside the top-k instead of after it. Those CTAs
    // stage their first row at once; CTAs with chunks start theirs after the
    // top-k, so that their copies do not queue ahead of the logits loads.
    const int grid = static_cast<int>(gridDim.x);
    const int nc = min(nchunk, grid);  // CTAs holding top-k chunks
    const int cta = static_cast<int>(blockIdx.x);
    const int n_workers = grid * kChunkTokens;
    int rrow = resid.A ? (cta >= nc ? cta - nc : cta + grid - nc) * kChunkTokens + warp : T;
    bool pre = rrow < T && cta >= nc;
    int staged = pre ? stage_residual_row(rrow, resid, rstage) : 0;
    // 1. router + the chunk's slot counts, one warp per token
    for (int c = blockIdx.x; c < nchunk; c += gridDim.x) {
        for (int x = threadIdx.x; x < nb; x += blockDim.x) smem[x] = 0;
        __syncthreads();
        const int t = c * kChunkTokens + warp;
        if (t < T) {
            const float* l = logits + static_cast<size_t>(t) * E;
            if (E <= 32)
                topk_token<1>(t, l, E, k, renorm, phi, P, topk_ids, alpha, smem, err);
            else if (E <= 64)
                topk_token<2>(t, l, E, k, renorm, phi, P, topk_ids, alpha, smem, err);
            else if (E <= 128)
                topk_token<4>(t, l, E, k, renorm, phi, P, topk_ids, alpha, smem, err);
            else if (E <= 256)
                topk_token<8>(t, l, E, k, renorm, phi, P, topk_ids, alpha, smem, err);
            else
                topk_token<kMaxPerLane>(t, l, E, k, renorm, phi, P, topk_ids, alpha, smem, err);
        }
        __syncthreads();
        for (int x = threadIdx.x; x < nb; x += blockDim.x)
            hist[static_cast<size_t>(x) * nchunk + c] = smem[x];
        __syncthreads();
    }
    for (; rrow < T; rrow += n_workers, pre = false) {
        if (!pre) staged = stage_residual_row(rrow, resid, rstage);
        finish_residual_row(rrow, resid, rstage, staged);
    }
    // CTAs added for residual rows take no part in the route map
    if (cta >= nc) return;
    if (!grid_barrier(sync, 1, nc, err, &ok_flag, withhold_arrival != 0 && blockIdx.x == 0)) {
        empty_route_map(offsets, mblk, P);
        return;
    }
    // 2. per-slot scans over chunks, spread over every warp of the chunks' CTAs
    scan_slots(hist, nchunk, nb, totals, nc);
    if (!grid_barrier(sync, 2, nc, err, &ok_flag)) {
        empty_route_map(offsets, mblk, P);
        return;
    }
    // 3. slot offsets and m-block prefix from the totals (in every CTA), then
    //    stable placement, one chunk per CTA at a time; the expert kernel's
    //    per-m-block counters start from zero
    int* off = smem;                 // [nb] slot offsets
    int* mb = smem + nb;             // [nb] m-block prefix, then the placement's counters
    int* warp_sums = smem + 2 * nb;  // [33]
    for (int b = threadIdx.x; b < nb; b += blockDim.x) {
        const int v = __ldcg(totals + b);
        off[b] = v;
        mb[b] = b < P ? (v + kBM - 1) / kBM : 0;
    }
    __syncthreads();
    block_exclusive_scan(off, nb, warp_sums);
    const int mb_total = block_exclusive_scan(mb, nb, warp_sums);
    if (blockIdx.x == 0) {
        for (int b = threadIdx.x; b < nb; b += blockDim.x) {
            offsets[b] = off[b];
            mblk[b] = mb[b];
        }
        if (tickets)
            for (int x = threadIdx.x; x < n_tickets; x += blockDim.x) tickets[x] = 0;
        if (threadIdx.x == 0) {
            offsets[P + 1] = R;
            mblk[P + 1] = mb_total;
        }
    }
    if (done)
        for (int m = blockIdx.x * blockDim.x + threadIdx.x; m < mb_total; m += nc * blockDim.x)
            done[m] = 0;
    __syncthreads();
    for (int c = blockIdx.x; c < nchunk; c += gridDim.x)
        scatter_chunk(c, nchunk, topk_ids, phi, P, k, R, hist, off, rec_tok, rec_route, rec_pos, mb);
}

// ---------------------------------------------------------------------------
// Router logits fused with the route build: one cooperative launch of
// clusters, from X and W_r to the route map.
//
// Cluster m (S CTAs) owns tokens [128 m, 128 m + 128). CTA s of the cluster
// multiplies the tile's X rows by W_r over its share of the k-blocks on the
// tensor cores (router_tile.cuh: TMA ring, tcgen05.mma, fp32 accumulator in
// TMEM, partial sums to shared memory) while its warps 6-15 write the tile's
// residual rows Y = A. After a cluster barrier CTA s takes the tile's 16-token
// chunks s, s + S, ...: a warp per token adds the S partials of each of its
// logits in ascending chunk order over distributed shared memory (the
// standalone router's order), keeps the row in shared memory (and writes it
// out when asked), and runs the same top-k and slot counting as k_route_fused
// on it. The rest is k_route_fused's route map: bounded grid barrier, per-slot
// scans over chunks, barrier, slot offsets and m-block prefix, stable
// placement of the CTA's chunks.
// ---------------------------------------------------------------------------
struct FusedRouter {
    int KB, S, N;        // k-blocks of H, CTAs per tile (the cluster), experts per tile
    uint32_t tx_bytes;   // bytes one ring stage's two boxes deliver
    float* logits;       // [T][E] out, or null
};

constexpr int kFusedMaxE = 128;
constexpr int kFusedChunksPerTile = 128 / kChunkTokens;

__host__ __device__ constexpr size_t fused_ring_bytes(int N) {
    return router_ring_bytes(N) > router_part_bytes(N) ? router_ring_bytes(N) : router_part_bytes(N);
}
__host__ __device__ constexpr size_t fused_rows_bytes(int N) {
    return static_cast<size_t>(kChunkTokens) * N * sizeof(float);
}
__host__ __device__ constexpr size_t fused_smem_bytes(int N, int P) {
    return 1024 + fused_ring_bytes(N) + fused_rows_bytes(N) + route_scratch_bytes(P + 1) +
           8 * (2 * kRStages + 1) + 16;
}

__global__ void __launch_bounds__(kRouteThreads, 1) k_route_from_x(
    const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
    const FusedRouter fr, int T, int E, int k, int renorm, const int32_t* __restrict__ phi, int P,
    int32_t* __restrict__ topk_ids, float* __restrict__ alpha, int32_t* __restrict__ offsets,
    int32_t* __restrict__ rec_tok, int32_t* __restrict__ rec_route, int32_t* __restrict__ rec_pos,
    int32_t* __restrict__ hist, int32_t* __restrict__ mblk, int32_t* __restrict__ totals,
    int32_t* __restrict__ done, int32_t* __restrict__ tickets, int n_tickets, int* __restrict__ sync,
    int* __restrict__ err, int nchunk, ResidualInit resid, int withhold_arrival) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ int ok_flag;
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const int R = T * k;
    const int nb = P + 1;
    const int S = fr.S, N = fr.N;
    // the partial sums are read across a cluster of S CTAs: any other launch
    // shape leaves an empty route map before any cluster or tensor access
    if (cluster_num_ctas() != static_cast<uint32_t>(S)) {
        if (threadIdx.x == 0) record_error(err, kDevErrLaunch);
        empty_route_map(offsets, mblk, P);
        return;
    }
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    uint32_t s_rank;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(s_rank));
    const int s = static_cast<int>(s_rank);
    const int m = static_cast<int>(blockIdx.x) / S;  // the cluster's token tile

    const uint32_t sbase = smem_addr(smem);
    const size_t ring = fused_ring_bytes(N);
    float* lrows = reinterpret_cast<float*>(smem + ring);                            // [16][N]
    int* scratch = reinterpret_cast<int*>(smem + ring + fused_rows_bytes(N));         // route scratch
    const size_t bar_off = ring + fused_rows_bytes(N) + route_scratch_bytes(nb);
    uint8_t* misc = smem + bar_off + 8 * (2 * kRStages + 1);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 4);
    RouterTile rt;
    rt.sA = sbase;
    rt.sB = sbase + kRStages * kRTileA;
    rt.bar0 = sbase + static_cast<uint32_t>(bar_off);
    rt.part = reinterpret_cast<float*>(smem);
    rt.m0 = m * 128;
    rt.n0 = 0;
    rt.N = N;
    rt.tx_bytes = fr.tx_bytes;
    rt.kb0 = static_cast<int>(static_cast<long long>(s) * fr.KB / S);
    rt.kb1 = static_cast<int>(static_cast<long long>(s + 1) * fr.KB / S);
    const uint32_t tmem_cols = router_tmem_cols(N);

    if (threadIdx.x == 0) {
        router_tile_init(rt);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(tmem_slot), tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    // 1. logits tile on the tensor cores; beside it, the residual rows
    if (warp < 6) {
        router_tile_roles(rt, &tm_x, &tm_w, tmem_base, abort_flag, err);
    } else if (resid.A) {
        const int rows_per = (128 + S - 1) / S;
        const int r0 = rt.m0 + s * rows_per;
        const int r1 = min(T, min(rt.m0 + 128, r0 + rows_per));
        const int row_bytes = resid.H * resid.elem_bytes;
        for (int t = r0 + (warp - 6); t < r1; t += kRouteThreads / 32 - 6)
            widen_residual(resid, t, static_cast<const char*>(resid.A) + static_cast<size_t>(t) * row_bytes,
                           0, row_bytes);
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // every CTA's partial is in place
    const bool gemm_ok = !*abort_flag;

    // 2. the logits of this CTA's chunks (fixed-order sums over the cluster),
    //    their top-k, and the chunks' slot counts
    int* counts = scratch;
    for (int j = s; j < kFusedChunksPerTile; j += S) {
        const int c = m * kFusedChunksPerTile + j;
        if (c >= nchunk) break;
        for (int x = threadIdx.x; x < nb; x += blockDim.x) counts[x] = 0;
        __syncthreads();
        const int t = c * kChunkTokens + warp;
        if (t < T) {
            float* row = lrows + warp * N;
            const int r = t - rt.m0;
            for (int e = lane; e < E; e += 32) {
                const uint32_t off = sbase + static_cast<uint32_t>((r * (N + 1) + e) * 4);
                const float v = gemm_ok ? sum_cluster_partials(off, S) : 0.0f;
                row[e] = v;
                if (fr.logits) fr.logits[static_cast<size_t>(t) * E + e] = v;
            }
            __syncwarp();
            if (E <= 32)
                topk_token<1>(t, row, E, k, renorm, phi, P, topk_ids, alpha, counts, err);
            else if (E <= 64)
                topk_token<2>(t, row, E, k, renorm, phi, P, topk_ids, alpha, counts, err);
            else
                topk_token<4>(t, row, E, k, renorm, phi, P, topk_ids, alpha, counts, err);
        }
        __syncthreads();
        for (int x = threadIdx.x; x < nb; x += blockDim.x)
            hist[static_cast<size_t>(x) * nchunk + c] = counts[x];
        __syncthreads();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // the peers have read this CTA's partials
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, tmem_cols);
    }

    // 3. the route map, as in k_route_fused over every CTA of the grid
    const int ncta = static_cast<int>(gridDim.x);
    if (!grid_barrier(sync, 1, ncta, err, &ok_flag, withhold_arrival != 0 && blockIdx.x == 0)) {
        empty_route_map(offsets, mblk, P);
        return;
    }
    // a tile whose logits did not complete (a bounded wait ran out, recorded
    // before the barrier) leaves the whole route map empty
    int e0;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(e0) : "l"(err) : "memory");
    if (e0 == kDevErrTimeout) {
        empty_route_map(offsets, mblk, P);
        return;
    }
    scan_slots(hist, nchunk, nb, totals, ncta);
    if (!grid_barrier(sync, 2, ncta, err, &ok_flag)) {
        empty_route_map(offsets, mblk, P);
        return;
    }
    int* off = scratch;
    int* mb = scratch + nb;
    int* warp_sums = scratch + 2 * nb;
    for (int b = threadIdx.x; b < nb; b += blockDim.x) {
        const int v = __ldcg(totals + b);
        off[b] = v;
        mb[b] = b < P ? (v + kBM - 1) / kBM : 0;
    }
    __syncthreads();
    block_exclusive_scan(off, nb, warp_sums);
    const int mb_total = block_exclusive_scan(mb, nb, warp_sums);
    if (blockIdx.x == 0) {
        for (int b = threadIdx.x; b < nb; b += blockDim.x) {
            offsets[b] = off[b];
            mblk[b] = mb[b];
        }
        if (tickets)
            for (int x = threadIdx.x; x < n_tickets; x += blockDim.x) tickets[x] = 0;
        if (threadIdx.x == 0) {
            offsets[P + 1] = R;
            mblk[P + 1] = mb_total;
        }
    }
    if (done)
        for (int q = blockIdx.x * blockDim.x + threadIdx.x; q < mb_total; q += ncta * blockDim.x)
            done[q] = 0;
    __syncthreads();
    for (int j = s; j < kFusedChunksPerTile; j += S) {
        const int c = m * kFusedChunksPerTile + j;
        if (c >= nchunk) break;
        scatter_chunk(c, nchunk, topk_ids, phi, P, k, R, hist, off, rec_tok, rec_route, rec_pos, mb);
    }
}

__global__ void k_identity_map(int T, int n_shared, int32_t* __restrict__ offsets,
                               int32_t* __restrict__ rec_tok, int32_t* __restrict__ mblk,
                               int32_t* __restrict__ done) {
    const int p = blockIdx.x * blockDim.x + threadIdx.x;
    if (p < T * n_shared) rec_tok[p] = p % T;
    if (done && p < n_shared * ((T + kBM - 1) / kBM)) done[p] = 0;
    if (p <= n_shared) {
        offsets[p] = p * T;
        mblk[p] = p * ((T + kBM - 1) / kBM);
    }
}

// Y = fp32(A), one warp per row (grid-stride over rows).
__global__ void k_residual_rows(ResidualInit r, int T) {
    const int warp = static_cast<int>((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    const int n_warps = static_cast<int>((gridDim.x * blockDim.x) >> 5);
    const int row_bytes = r.H * r.elem_bytes;
    for (int t = warp; t < T; t += n_warps)
        widen_residual(r, t, static_cast<const char*>(r.A) + static_cast<size_t>(t) * row_bytes, 0,
                       row_bytes);
}

__global__ void k_cast_f32_bf16(const float* __restrict__ src, __nv_bfloat16* __restrict__ dst,
                                size_t n) {
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    for (size_t x = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; x < n; x += stride)
        dst[x] = __float2bfloat16_rn(src[x]);
}

// CTAs of k_route_fused that fit on the current device at once, at its
// largest shared-memory size (the bound for every smaller launch). Looked up
// once per device, under a lock; the kernel's shared-memory attribute is set
// on each device as it is first seen (a device's attributes are its own).
static int route_co_resident() {
    constexpr int kMaxDevices = 64;
    static std::mutex mu;
    static int cache[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev] > 0) return cache[dev];
    int sms = 0, per_sm = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    const size_t max_smem = route_scratch_bytes(kMaxP + 1) + kResidStageCta;
    if (cudaFuncSetAttribute(k_route_fused, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(max_smem)) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_route_fused, kRouteThreads,
                                                      max_smem) != cudaSuccess ||
        per_sm <= 0)
        return 0;
    cache[dev] = sms * per_sm;
    return cache[dev];
}

// Residual rows the route build copies on CTAs it adds beside the top-k
// chunks (those copies overlap the top-k; later rows follow it on the chunk
// CTAs, ahead of the grid barriers).
int route_residual_overlap_rows(int T) {
    const int co = route_co_resident();
    const int nchunk = (T + kChunkTokens - 1) / kChunkTokens;
    const int grid = std::max(1, std::min(co, 2 * nchunk));
    return std::max(0, grid - std::min(nchunk, grid)) * kChunkTokens;
}

RouteWorkspace route_workspace_layout(int T, int k, int P) {
    RouteWorkspace w;
    (void)k;
    w.nchunk = (T + kChunkTokens - 1) / kChunkTokens;
    size_t off = 0;
    w.err_off = off;
    w.sync_off = off + sizeof(int32_t);
    off = align_up(off + 2 * sizeof(int32_t), 256);
    w.hist_off = off;
    off = align_up(off + sizeof(int32_t) * static_cast<size_t>(w.nchunk > 0 ? w.nchunk : 1) * (P + 1), 256);
    w.mblk_off = off;
    off = align_up(off + sizeof(int32_t) * static_cast<size_t>(P + 2), 256);
    w.tot_off = off;
    off = align_up(off + sizeof(int32_t) * static_cast<size_t>(P + 1), 256);
    w.total = off;
    return w;
}

cudaError_t launch_route_build(const float* logits, int T, int E, int k, int renorm,
                               const int32_t* phi, int P, int32_t* topk_ids, float* alpha,
                               int32_t* offsets, int32_t* rec_tok, int32_t* rec_route,
                               int32_t* rec_pos, int32_t* done, int32_t* tickets, int n_tickets,
                               void* ws, size_t ws_bytes, cudaStream_t stream, int* n_launches,
                               const ResidualInit* resid_in, int withhold_arrival,
                               bool clear_err) {
    const RouteWorkspace w = route_workspace_layout(T, k, P);
    if (!ws || w.total > ws_bytes) return cudaErrorInvalidValue;
    char* base = static_cast<char*>(ws);
    int* err = reinterpret_cast<int*>(base + w.err_off);
    int32_t* hist = reinterpret_cast<int32_t*>(base + w.hist_off);
    int32_t* mblk = reinterpret_cast<int32_t*>(base + w.mblk_off);
    int32_t* totals = reinterpret_cast<int32_t*>(base + w.tot_off);
    const int R = T * k;
    const int nb = P + 1;
    int launches = 0;
    cudaError_t rc;
    if (R == 0) {
        rc = cudaMemsetAsync(err, 0, sizeof(int), stream);
        if (rc == cudaSuccess) rc = cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (P + 2), stream);
        if (rc == cudaSuccess) rc = cudaMemsetAsync(mblk, 0, sizeof(int32_t) * (P + 2), stream);
        return rc;
    }
    // clear the error word (unless an earlier kernel of the same call wrote
    // it) and the grid-barrier counter; the kernel writes every per-chunk
    // count itself
    rc = clear_err ? cudaMemsetAsync(base + w.err_off, 0, 2 * sizeof(int32_t), stream)
                   : cudaMemsetAsync(base + w.sync_off, 0, sizeof(int32_t), stream);
    if (rc != cudaSuccess) return rc;
    int* sync = reinterpret_cast<int*>(base + w.sync_off);
    ResidualInit resid{nullptr, 0, nullptr, 0};
    if (resid_in) resid = *resid_in;
    const int co_resident = route_co_resident();
    if (co_resident <= 0) return cudaErrorLaunchOutOfResources;
    // with a residual, up to as many CTAs again for its rows
    const int grid = std::max(1, std::min(co_resident, resid.A ? 2 * w.nchunk : w.nchunk));
    const size_t smem = route_scratch_bytes(nb) + (resid.A ? kResidStageCta : 0);
    void* args[] = {&logits, &T, &E, &k, &renorm, &phi, &P, &topk_ids, &alpha, &offsets,
                    &rec_tok, &rec_route, &rec_pos, &hist, &mblk, &totals, &done, &tickets,
                    &n_tickets, &sync, &err, const_cast<int*>(&w.nchunk), &resid,
                    &withhold_arrival};
    rc = cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(k_route_fused), grid,
                                     kRouteThreads, args, smem, stream);
    if (rc != cudaSuccess) return rc;
    ++launches;
    if (n_launches) *n_launches += launches;
    return cudaGetLastError();
}

// Largest number of clusters of S CTAs (each with smem bytes of dynamic shared
// memory) that the current device holds at once, cached per (device, S, smem).
static int fused_max_clusters(int S, size_t smem) {
    struct Key { int dev, S; size_t smem; int n; };
    static std::mutex mu;
    static Key cache[64];
    static int n_cache = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n_cache; ++i)
        if (cache[i].dev == dev && cache[i].S == S && cache[i].smem == smem) return cache[i].n;
    if (cudaFuncSetAttribute(k_route_from_x, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
        return 0;
    if (S > 8 && cudaFuncSetAttribute(k_route_from_x, cudaFuncAttributeNonPortableClusterSizeAllowed,
                                      1) != cudaSuccess)
        return 0;
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = static_cast<unsigned>(S);
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(sms / S * S));
    cfg.blockDim = dim3(kRouteThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void*>(k_route_from_x), &cfg) !=
        cudaSuccess) {
        (void)cudaGetLastError();
        n = 0;
    }
    if (n_cache < 64) cache[n_cache++] = {dev, S, smem, n};
    return n;
}

FusedRoutePlan fused_route_plan(int T, int H, int E, int P) {
    FusedRoutePlan p{};
    p.ok = false;
    if (T <= 0 || H < 64 || H % 64 != 0 || E < 1 || E > kFusedMaxE || P < 0 || P > kMaxP) return p;
    p.N = ((E + 15) / 16) * 16;
    p.m_tiles = (T + 127) / 128;
    p.KB = H / 64;
    p.smem = fused_smem_bytes(p.N, P);
    int dev = 0, sms = 0, max_smem = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return p;
    if (p.smem > static_cast<size_t>(max_smem)) return p;
    // about one wave of CTAs, at least four k-blocks per CTA, a portable
    // cluster, and every cluster resident at once (cooperative launch)
    long long S = (sms + p.m_tiles - 1) / p.m_tiles;
    if (S > p.KB / 4) S = p.KB / 4;
    if (S > kRMaxSplit) S = kRMaxSplit;
    if (S < 1) S = 1;
    for (; S >= 1; --S)
        if (fused_max_clusters(static_cast<int>(S), p.smem) >= p.m_tiles) break;
    if (S < 1) return p;
    p.S = static_cast<int>(S);
    p.ok = true;
    return p;
}

cudaError_t launch_route_from_x(const void* X, int T, int H, const void* W_r, int E, int k,
                                int renorm, const int32_t* phi, int P, float* logits,
                                int32_t* topk_ids, float* alpha, int32_t* offsets,
                                int32_t* rec_tok, int32_t* rec_route, int32_t* rec_pos,
                                int32_t* done, int32_t* tickets, int n_tickets, void* ws,
                                size_t ws_bytes, cudaStream_t stream, int* n_launches,
                                const ResidualInit* resid_in, int withhold_arrival) {
    const RouteWorkspace w = route_workspace_layout(T, k, P);
    if (!ws || w.total > ws_bytes) return cudaErrorInvalidValue;
    char* base = static_cast<char*>(ws);
    int* err = reinterpret_cast<int*>(base + w.err_off);
    int32_t* hist = reinterpret_cast<int32_t*>(base + w.hist_off);
    int32_t* mblk = reinterpret_cast<int32_t*>(base + w.mblk_off);
    int32_t* totals = reinterpret_cast<int32_t*>(base + w.tot_off);
    int* sync = reinterpret_cast<int*>(base + w.sync_off);
    cudaError_t rc;
    if (T * k == 0) {
        rc = cudaMemsetAsync(err, 0, sizeof(int), stream);
        if (rc == cudaSuccess) rc = cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (P + 2), stream);
        if (rc == cudaSuccess) rc = cudaMemsetAsync(mblk, 0, sizeof(int32_t) * (P + 2), stream);
        return rc;
    }
    const FusedRoutePlan p = fused_route_plan(T, H, E, P);
    if (!p.ok) return cudaErrorNotSupported;
    // boxes no taller than the tensors; the MMA still reads 128 x N rows, the
    // rows past T or E hold stale data whose results are never used
    CUtensorMap tm_x, tm_w;
    const CUtensorMapDataType BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const uint32_t box_x = static_cast<uint32_t>(T < 128 ? T : 128);
    const uint32_t box_w = static_cast<uint32_t>(E < p.N ? E : p.N);
    if (encode_tmap_2d(&tm_x, BF, X, static_cast<uint64_t>(H), static_cast<uint64_t>(T),
                       static_cast<uint64_t>(H) * 2, 64, box_x) != CUDA_SUCCESS ||
        encode_tmap_2d(&tm_w, BF, W_r, static_cast<uint64_t>(H), static_cast<uint64_t>(E),
                       static_cast<uint64_t>(H) * 2, 64, box_w) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    rc = cudaMemsetAsync(base + w.err_off, 0, 2 * sizeof(int32_t), stream);
    if (rc != cudaSuccess) return rc;
    rc = cudaFuncSetAttribute(k_route_from_x, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(p.smem));
    if (rc != cudaSuccess) return rc;
    FusedRouter fr;
    fr.KB = p.KB;
    fr.S = p.S;
    fr.N = p.N;
    fr.tx_bytes = (box_x + box_w) * 128u;
    fr.logits = logits;
    ResidualInit resid{nullptr, 0, nullptr, 0};
    if (resid_in) resid = *resid_in;
    int nchunk = w.nchunk;
    void* args[] = {&tm_x, &tm_w, &fr, &T, &E, &k, &renorm, &phi, &P, &topk_ids, &alpha, &offsets,
                    &rec_tok, &rec_route, &rec_pos, &hist, &mblk, &totals, &done, &tickets,
                    &n_tickets, &sync, &err, &nchunk, &resid, &withhold_arrival};
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = static_cast<unsigned>(p.S);
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeCooperative;
    at[1].val.cooperative = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(p.m_tiles * p.S));
    cfg.blockDim = dim3(kRouteThreads);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = stream;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    rc = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(k_route_from_x), args);
    if (rc != cudaSuccess) return rc;
    if (n_launches) *n_launches += 1;
    return cudaGetLastError();
}

cudaError_t launch_identity_map(int T, int n_shared, int32_t* offsets, int32_t* rec_tok,
                                int32_t* mblk, int32_t* done, cudaStream_t stream) {
    const int n = T * n_shared > n_shared + 1 ? T * n_shared : n_shared + 1;
    k_identity_map<<<(n + 255) / 256, 256, 0, stream>>>(T, n_shared, offsets, rec_tok, mblk, done);
    return cudaGetLastError();
}

cudaError_t launch_residual_rows(const void* A, int elem_bytes, float* Y, int T, int H,
                                 cudaStream_t stream) {
    if (T <= 0) return cudaSuccess;
    const ResidualInit r{A, elem_bytes, Y, H};
    const int blocks = (T + 7) / 8 < 1024 ? (T + 7) / 8 : 1024;   // 8 warps of 32 per block
    k_residual_rows<<<blocks, 256, 0, stream>>>(r, T);
    return cudaGetLastError();
}

cudaError_t launch_cast_f32_bf16(const float* src, void* dst, size_t n, cudaStream_t stream) {
    if (n == 0) return cudaSuccess;
    size_t blocks = (n + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    k_cast_f32_bf16<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        src, static_cast<__nv_bfloat16*>(dst), n);
    return cudaGetLastError();
}

}  // namespace es
