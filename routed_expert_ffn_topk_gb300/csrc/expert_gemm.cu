// The routed expert FFN as one fused, persistent operator on the
// 5th-generation tensor cores (tcgen05 + TMEM), fed by TMA and cp.async.
//
// "EStream: Fast and Memory-Efficient MoE Prefill through Expert
// Virtualization on Mobile NPUs", section 3.2 ("Fused Expert Execution with
// Intra-NPU Pipelining") and Eq. 1: for every non-empty slot s the routed
// rows of X are gathered, the gate and up projections are evaluated as tile
// pairs, SiLU(g) * u is applied to completed pairs, the down projection is
// evaluated, and completed down tiles are multiplied by the route weight and
// scatter-added into the token accumulator Y (Eq. 2) -- one route-aware
// operator, as the paper builds it.
//
// GB300 form. One cooperative kernel per call walks a list of 128-row tiles
// built from the route map: first every gate/up tile (segment, n-block of 128
// h columns, m-block), then every down tile (segment, n-block of 256 Y
// columns, m-block). Warp roles per CTA (one CTA per SM):
//   warp 0     TMA producer into a 4-stage ring: the weight tiles (gate + up
//              2 x 16 KB, or down 32 KB, per stage; evict-first in L2 when the
//              segment has a single m-block, their only reader) and, for down
//              tiles, the 16 KB A tile of h once the m-block's gate/up tiles
//              have all published (records are contiguous by slot, so a plain
//              box).
//   warp 1     allocates 512 TMEM columns (two 128x256 fp32 accumulators);
//              one lane issues tcgen05.mma (M=128, N=256, K=16 per
//              instruction, kind::f16), committing stages back to the
//              producers and finished accumulators to the epilogue.
//   warps 2-5  epilogue: tcgen05.ld of the accumulator. Gate/up tiles write
//              h = SiLU(g) * u as fp16 and publish "m-block done" counters;
//              down tiles scale by alpha times the expert's down-weight scale
//              and add into Y[t] with vector fp32 reductions (or store the
//              scaled row for the deterministic combine). Rows go out through
//              a per-warp shared-memory stage, four whole rows per
//              instruction.
//   warps 6-9  row gather of gate/up tiles: each record's 128-byte slice of
//              X[tok] for the stage's K range is copied with 16-byte cp.async
//              into the 128-byte-swizzled layout the MMA reads (chunk c of row
//              r at c ^ (r mod 8)). TMA tile::gather4 moves only four rows per
//              instruction and measured ~2.3x slower here. For down tiles
//              these warps only pass the stages through.
// The gate and up weight tiles of one n-block sit back to back in shared
// memory, so a single N=256 instruction produces both halves of a pair.
// Operand types: gate/up multiply bf16 X by bf16 W_g / W_u; down multiplies
// fp16 h by fp16 W_d, which the offline packer converted from bf16 with an
// exact per-expert power-of-two scale: fp16 keeps 3 more significand bits of
// h than bf16 would, which is what keeps Y within the accuracy bound.
// Every wait is bounded: on timeout the kernel records an error word, lets
// outstanding copies and MMAs land, frees TMEM and returns. The cross-CTA
// wait (down tile on gate/up tiles) is deadlock-free because the launch is
// cooperative (all CTAs resident) and every gate/up tile precedes every down
// tile in each CTA's tile order.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <mutex>

#include "estream_internal.h"

namespace es {
namespace {

constexpr int kStages = 4;
constexpr int kRowBytes = 128;                    // one swizzle row of K
constexpr int kTileABytes = kBM * kRowBytes;      // 16 KB
constexpr int kTileBBytes = 256 * kRowBytes;      // 32 KB
constexpr int kAccCols = 256;
constexpr int kTmemCols = 512;
constexpr int kThreads = 320;           // TMA, MMA, 4 epilogue warps, 4 A-loader warps
constexpr int kLoaderWarp0 = 6;
constexpr int kLoaderDepth = 2;         // cp.async groups kept in flight per loader thread
constexpr float kHalfMax = 65504.0f;

// Shared-memory map (offsets from a 1024-byte aligned base).
constexpr int kOffA = 0;
constexpr int kOffB = kStages * kTileABytes;
constexpr int kOffStg = kOffB + kStages * kTileBBytes;  // epilogue stages, 4 x 4 KB
constexpr int kOffBar = kOffStg + 4 * 32 * 128;
// barriers: full[kStages], empty[kStages], acc_full[2], acc_empty[2], drain
// + tile ring: tile_full[4], tile_empty[4]
constexpr int kNumBars = 2 * kStages + 5 + 2 * 4;
constexpr int kOffMisc = kOffBar + 8 * kNumBars;  // tmem base, abort flag
constexpr int kOffRing = kOffMisc + 16;           // tile ring: 4 ints
constexpr int kOffTable = kOffRing + 16;

size_t gemm_smem_bytes(int seg_count) {
    return 1024 + kOffTable + sizeof(int) * static_cast<size_t>(seg_count + 1);
}

#include "tc_ptx.cuh"

__device__ __forceinline__ float silu_mul(float g, float u) {
    return __fdividef(g, 1.0f + __expf(-g)) * u;
}

struct Tile {
    int seg;   // segment index relative to seg_begin
    int mb;    // m-block inside the segment
    int nb;    // n-block
    int row0;  // first record of the tile
    int rows;  // valid records in the tile (1..kBM)
};

// Tiles are numbered segment by segment; inside a segment n-block-major with
// the m-blocks fastest, so the CTAs running at the same time share one
// weight n-block (read from HBM about once) while the gathered rows of the
// segment stay in L2.
__device__ __forceinline__ Tile decode_tile(int t, const int* table, int seg_count, int NB,
                                            const int32_t* offsets, int seg_begin) {
    int lo = 0, hi = seg_count;  // largest lo with table[lo] * NB <= t
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (table[mid] * NB <= t) lo = mid; else hi = mid;
    }
    Tile ti;
    ti.seg = lo;
    const int nmb = table[lo + 1] - table[lo];
    const int l = t - table[lo] * NB;
    ti.nb = l / nmb;
    ti.mb = l - ti.nb * nmb;
    const int s_lo = offsets[seg_begin + lo];
    const int s_hi = offsets[seg_begin + lo + 1];
    ti.row0 = s_lo + ti.mb * kBM;
    ti.rows = min(kBM, s_hi - ti.row0);
    return ti;
}

// The idx-th tile of worker b (a CTA, or a CTA pair) among G workers, or -1
// past its last. Gate/up tiles [0, TA) go round-robin (worker b gets b,
// b + G, ...). Down tiles [TA, TA + TB) first top up the workers that got one
// gate/up tile fewer, KBA / KBB tiles each (round-robin over those), then go
// round-robin over all workers starting at the first of them, so that the
// k-blocks per worker (KBA per gate/up tile, KBB per down tile) even out.
// Each worker runs all its gate/up tiles before its down tiles, which keeps
// the cross-CTA wait of a down tile deadlock-free.
__device__ __forceinline__ int tile_of(int b, int G, int TA, int TB, int KBA, int KBB, int idx) {
    const int q = TA / G, rem = TA - q * G;
    const int n_gu = q + (b < rem ? 1 : 0);
    if (idx < n_gu) return b + idx * G;
    idx -= n_gu;
    const int lows = G - rem;
    const int n_extra = rem ? KBA / KBB : 0;
    const int A = static_cast<int>(min(static_cast<long long>(TB), static_cast<long long>(n_extra) * lows));
    if (b >= rem && b - rem < A) {
        const int nA = (A - (b - rem) + lows - 1) / lows;
        if (idx < nA) return TA + (b - rem) + idx * lows;
        idx -= nA;
    }
    const long long j = static_cast<long long>(A) + (b - rem + G) % G + static_cast<long long>(idx) * G;
    return j < TB ? TA + static_cast<int>(j) : -1;
}

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// Make this thread's completed generic-proxy shared-memory writes visible to
// the async proxy (the tensor cores read operands through it).
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Acquire load of a counter another CTA publishes.
__device__ __forceinline__ int ld_acquire(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void red_release_add(int* p, int v) {
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

struct FfnArgs {
    GemmSegments seg;
    const __nv_bfloat16* x;  // [T][H]: gate/up A rows (gathered)
    __half* h;               // [rows][F]: written by gate/up tiles, read by down tiles
    float* Y;                // [T][H] accumulator
    float* out_rows;         // deterministic mode: [rows][H], else null
    int* done;               // per absolute m-block: epilogue-warp publications of gate/up tiles
    int* ticket;             // dynamic tile counter (zero at launch), or null for the static order
    int* dev_err;
    int H, F;
    int phases;              // bit 0: gate/up tiles, bit 1: down tiles
};

// Orders this thread's generic-proxy global accesses with its async-proxy
// (TMA) accesses: h is written with st.global and read back with TMA.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Epilogue of a gate/up tile for one TMEM lane (one record): columns
// [0, 128) of the accumulator hold the gate half and [128, 256) the up half
// of 128 h columns; h = fp16(SiLU(g) * u) goes to dst[0 .. 128). Values
// outside fp16's range are reported through dev_err.
__device__ __forceinline__ void epilogue_gate_up(uint32_t tacc, bool valid, __half* dst,
                                                 int* dev_err) {
    bool in_range = true;
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
        uint32_t g[32], u[32];
        tmem_ld32(tacc + c * 32, g);
        tmem_ld32(tacc + 128 + c * 32, u);
        tmem_ld_wait();
        if (valid) {
            uint32_t packed[16];
#pragma unroll
            for (int v = 0; v < 16; ++v) {
                const float h0 = silu_mul(__uint_as_float(g[2 * v]), __uint_as_float(u[2 * v]));
                const float h1 = silu_mul(__uint_as_float(g[2 * v + 1]), __uint_as_float(u[2 * v + 1]));
                in_range = in_range && fabsf(h0) <= kHalfMax && fabsf(h1) <= kHalfMax;
                const __half2 p2 = __floats2half2_rn(h0, h1);
                packed[v] = *reinterpret_cast<const uint32_t*>(&p2);
            }
#pragma unroll
            for (int v = 0; v < 4; ++v)
                st_v4(dst + c * 32 + 8 * v, packed[4 * v], packed[4 * v + 1], packed[4 * v + 2],
                      packed[4 * v + 3]);
        }
    }
    if (!in_range) record_error(dev_err, kDevErrRange);
}

// Epilogue of a down tile for one TMEM lane: the 256 accumulator columns
// times `al` are added into y_row[col0 ..] with vector reductions, or stored
// to out_row[col0 ..] when out_row is given (deterministic mode).
__device__ __forceinline__ void epilogue_down(uint32_t tacc, bool valid, float al, float* out_row,
                                              float* y_row, int col0) {
#pragma unroll 1
    for (int c = 0; c < 8; ++c) {
        uint32_t v[32];
        tmem_ld32(tacc + c * 32, v);
        tmem_ld_wait();
        if (valid) {
            const int col = col0 + c * 32;
            if (out_row) {
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    st_v4(out_row + col + 4 * q, __float_as_uint(al * __uint_as_float(v[4 * q])),
                          __float_as_uint(al * __uint_as_float(v[4 * q + 1])),
                          __float_as_uint(al * __uint_as_float(v[4 * q + 2])),
                          __float_as_uint(al * __uint_as_float(v[4 * q + 3])));
            } else {
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    red_add_v4(y_row + col + 4 * q, al * __uint_as_float(v[4 * q]),
                               al * __uint_as_float(v[4 * q + 1]), al * __uint_as_float(v[4 * q + 2]),
                               al * __uint_as_float(v[4 * q + 3]));
            }
        }
    }
}

// Coalesced write-out. A tcgen05.ld gives each thread one record's row, so
// storing straight from registers makes every warp instruction touch 32
// different rows of h or Y with 16 bytes each. The staged epilogues instead
// pass each 32 x 128-byte chunk of the warp's accumulator rows through a
// 4 KB shared-memory stage and write it out row by row: one instruction then
// covers four whole 128-byte rows (for Y, four full lines of vector
// reductions). The stage stores 16-byte chunk j of row r at chunk
// j ^ (r mod 8), which keeps both the row-wise writes and the column-wise
// reads free of bank conflicts.
constexpr int kStageWarpBytes = 32 * 128;

__device__ __forceinline__ uint32_t stage_off(int r, int j) {
    return static_cast<uint32_t>(r * 128 + ((j ^ (r & 7)) << 4));
}

// Row pointer of the record that lane `lane` writes in read-out step i
// (rows 4 i .. 4 i + 3, eight lanes per row).
template <typename T>
__device__ __forceinline__ T* row_of_step(T* my_row, int i, int lane) {
    return reinterpret_cast<T*>(
        __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(my_row), 4 * i + (lane >> 3)));
}

// Gate/up epilogue through the stage: h = fp16(SiLU(g) u) of this lane's
// record goes to dst_row[0 .. 64 n_halves) (null for a padding record), 64
// columns (128 bytes) per pass. The gate value of h column j is accumulator
// column j and the up value column u_off + j (u_off = 128 for a full tile's
// 128 columns; 64 for the 64 columns a lane holds in a half pair tile).
__device__ __forceinline__ void epilogue_gate_up_staged(uint32_t tacc, __half* dst_row,
                                                        uint32_t stg, int lane, int* dev_err,
                                                        int n_halves = 2, uint32_t u_off = 128) {
    bool in_range = true;
    __half* dst[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) dst[i] = row_of_step(dst_row, i, lane);
    const int j = lane & 7;
#pragma unroll 1
    for (int half = 0; half < n_halves; ++half) {
#pragma unroll 1
        for (int c2 = 0; c2 < 2; ++c2) {
            const int c = 2 * half + c2;
            uint32_t g[32], u[32];
            tmem_ld32(tacc + c * 32, g);
            tmem_ld32(tacc + u_off + c * 32, u);
            tmem_ld_wait();
            uint32_t packed[16];
#pragma unroll
            for (int v = 0; v < 16; ++v) {
                const float h0 = silu_mul(__uint_as_float(g[2 * v]), __uint_as_float(u[2 * v]));
                const float h1 = silu_mul(__uint_as_float(g[2 * v + 1]), __uint_as_float(u[2 * v + 1]));
                in_range = in_range && fabsf(h0) <= kHalfMax && fabsf(h1) <= kHalfMax;
                const __half2 p2 = __floats2half2_rn(h0, h1);
                packed[v] = *reinterpret_cast<const uint32_t*>(&p2);
            }
#pragma unroll
            for (int v = 0; v < 4; ++v)
                st_shared_v4(stg + stage_off(lane, 4 * c2 + v), packed[4 * v], packed[4 * v + 1],
                             packed[4 * v + 2], packed[4 * v + 3]);
        }
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint4 x = ld_shared_v4(stg + stage_off(4 * i + (lane >> 3), j));
            if (dst[i]) st_v4(dst[i] + half * 64 + 8 * j, x.x, x.y, x.z, x.w);
        }
        __syncwarp();
    }
    if (dst_row && !in_range) record_error(dev_err, kDevErrRange);
}

// Down epilogue through the stage: the first 32 n_chunks accumulator columns
// of this lane's record (256 in a full tile, the 128 a lane holds in a half
// pair tile) times `al` are added into dst_row[0 .. 32 n_chunks) with vector
// reductions (reduce) or stored there (the scaled-row buffer of the
// deterministic mode); dst_row is null for a padding record.
__device__ __forceinline__ void epilogue_down_staged(uint32_t tacc, float al, float* dst_row,
                                                     bool reduce, uint32_t stg, int lane,
                                                     int n_chunks = 8) {
    float* dst[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) dst[i] = row_of_step(dst_row, i, lane);
    const int j = lane & 7;
#pragma unroll 1
    for (int c = 0; c < n_chunks; ++c) {
        uint32_t v[32];
        tmem_ld32(tacc + c * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 8; ++q)
            st_shared_v4(stg + stage_off(lane, q), __float_as_uint(al * __uint_as_float(v[4 * q])),
                         __float_as_uint(al * __uint_as_float(v[4 * q + 1])),
                         __float_as_uint(al * __uint_as_float(v[4 * q + 2])),
                         __float_as_uint(al * __uint_as_float(v[4 * q + 3])));
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint4 x = ld_shared_v4(stg + stage_off(4 * i + (lane >> 3), j));
            if (dst[i]) {
                float* d = dst[i] + c * 32 + 4 * j;
                if (reduce)
                    red_add_v4(d, __uint_as_float(x.x), __uint_as_float(x.y), __uint_as_float(x.z),
                               __uint_as_float(x.w));
                else
                    st_v4(d, x.x, x.y, x.z, x.w);
            }
        }
        __syncwarp();
    }
}

// ----------------------------------------------------------------------------
// Roles shared by the single-SM kernels (bf16 weights and 4-bit weights)
// ----------------------------------------------------------------------------

// Barriers of a stage ring: full[s] at full0 + 8 s, empty[s] at empty0 + 8 s.
struct Ring {
    uint32_t full0, empty0;
    __device__ __forceinline__ uint32_t full(int s) const { return full0 + 8u * s; }
    __device__ __forceinline__ uint32_t empty(int s) const { return empty0 + 8u * s; }
};

// This CTA's walk over the tile list and the decode of a tile. With a ticket
// counter (zero at launch) tiles are handed out dynamically: the producer
// thread takes tickets from the counter -- CTAs that run faster take more
// tiles, absorbing the spread of tile times -- and publishes each in a
// shared-memory ring that every other role reads in order. Tickets are taken in list order and
// every gate/up tile precedes every down tile in the list, so a CTA takes all
// its gate/up tiles before any down tile and the cross-CTA wait of a down
// tile stays deadlock-free. Without a counter the static tile_of order is used.
constexpr int kTileRing = 4;

struct TileWalk {
    const GemmSegments* seg;
    const int* table;  // m-block prefix of the segment range, in shared memory
    int TA, TB, NBA, NBB, KBA, KBB;
    int* ticket;                 // per-launch counter, or null for the static order
    volatile int* ring;          // [kTileRing] published tile ids (-1: no more)
    uint32_t tfull0, tempty0;    // ring barriers, kTileRing each
    volatile int* abort_flag;
    int* dev_err;

    __device__ __forceinline__ Tile decode(int t) const {
        const bool gu = t < TA;
        return decode_tile(gu ? t : t - TA, table, seg->seg_count, gu ? NBA : NBB, seg->offsets,
                           seg->seg_begin);
    }
    // Consumer side, one thread: the it-th tile of this CTA, or -1 after the last.
    __device__ int tile_thread(int it) const {
        if (!ticket) return tile_of(blockIdx.x, gridDim.x, TA, TB, KBA, KBB, it);
        const int r = it % kTileRing;
        const uint32_t ph = static_cast<uint32_t>(it / kTileRing) & 1u;
        if (!mbar_wait(tfull0 + 8u * r, ph, abort_flag, dev_err)) return -1;
        const int t = ring[r];
        mbar_arrive(tempty0 + 8u * r);
        return t;
    }
    // The same for a whole warp (lane 0 reads the ring).
    __device__ int tile(int it) const {
        if (!ticket) return tile_of(blockIdx.x, gridDim.x, TA, TB, KBA, KBB, it);
        int t = -1;
        if ((threadIdx.x & 31) == 0) t = tile_thread(it);
        return __shfl_sync(0xffffffffu, t, 0);
    }
    // Producer side, one thread: publish the it-th tile. `pending` holds the
    // ticket requested one tile earlier (first request before the walk).
    __device__ int publish(int it, int& pending) const {
        if (!ticket) return tile_of(blockIdx.x, gridDim.x, TA, TB, KBA, KBB, it);
        const int r = it % kTileRing;
        const uint32_t ph = static_cast<uint32_t>(it / kTileRing) & 1u;
        if (!mbar_wait(tempty0 + 8u * r, ph ^ 1u, abort_flag, dev_err)) return -1;
        int t = pending;
        if (t >= 0 && t < TA + TB) {
            pending = atomicAdd(ticket, 1);
        } else {
            t = -1;
        }
        ring[r] = t;
        mbar_arrive(tfull0 + 8u * r);
        return t;
    }
    __device__ int first_ticket() const { return ticket ? atomicAdd(ticket, 1) : 0; }
};

// Lane 0: bounded wait until *cnt >= target (an m-block's gate/up tiles have
// all published). Returns false on abort or timeout (recorded).
__device__ bool wait_counter(const int* cnt, int target, volatile int* abort_flag, int* dev_err) {
    if (ld_acquire(cnt) >= target) return true;
    const uint64_t t0 = global_ns();
    while (ld_acquire(cnt) < target) {
        if (*abort_flag) return false;
        if (global_ns() - t0 > kWaitLimitNs) {
            *abort_flag = 1;
            record_error(dev_err, kDevErrTimeout);
            return false;
        }
    }
    return true;
}

// A-operand loader (4 warps): the row gather of gate/up tiles. Loader warp
// gw covers rows [32 gw, 32 gw + 32) of every A stage; in copy instruction i
// lane l moves 16-byte chunk (l mod 8) of row 32 gw + 4i + l/8, so each
// warp-instruction reads four whole 128-byte rows. Every thread arrives on a
// stage once its own copies are complete (wait_group) and fenced to the async
// proxy; kDepth stages stay in flight per thread, and the pending ones are
// published before a down tile (whose A comes by TMA) so the CTA never waits
// on a counter with its own stages unpublished. Down tiles' stages are only
// passed on (one arrival per thread).
template <int kSt, int kDepth>
__device__ void role_gather(const FfnArgs& a, const TileWalk& w, Ring ring, uint32_t sA,
                            volatile int* abort_flag, int gw, int lane) {
    const GemmSegments& seg = *w.seg;
    const uint32_t chunk = static_cast<uint32_t>(lane & 7);
    int stage = 0;
    uint32_t phase = 0;
    int pend[kDepth + 1];
    int npend = 0;
    bool ok = true;
    for (int it = 0, t; ok && (t = w.tile(it)) >= 0; ++it) {
        const bool gu = t < w.TA;
        const Tile ti = w.decode(t);
        const int num_kb = gu ? w.KBA : w.KBB;
        if (!gu) {
            if (npend > 0) {
                cp_async_wait<0>();
                fence_proxy_async();
                for (int q = 0; q < npend; ++q) mbar_arrive(ring.full(pend[q]));
                npend = 0;
            }
            for (int kb = 0; kb < num_kb; ++kb) {
                bool wt = true;
                if (lane == 0) wt = mbar_wait(ring.empty(stage), phase ^ 1u, abort_flag, a.dev_err);
                wt = __shfl_sync(0xffffffffu, wt, 0);
                if (!wt) {
                    ok = false;
                    break;
                }
                mbar_arrive(ring.full(stage));
                if (++stage == kSt) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            continue;
        }
        const uint8_t* src_row[8];
        uint32_t dst_off[8];
        unsigned live = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int r = gw * 32 + 4 * i + (lane >> 3);
            dst_off[i] = static_cast<uint32_t>(r) * kRowBytes +
                         ((chunk ^ static_cast<uint32_t>(r & 7)) << 4);
            const bool lv = r < ti.rows;
            live |= lv ? (1u << i) : 0u;
            const uint8_t* row = reinterpret_cast<const uint8_t*>(a.x);
            if (lv)
                row = reinterpret_cast<const uint8_t*>(
                    a.x + static_cast<size_t>(seg.rec_tok[ti.row0 + r]) * a.H);
            src_row[i] = row + chunk * 16;
        }
        for (int kb = 0; kb < num_kb; ++kb) {
            bool wt = true;
            if (lane == 0) wt = mbar_wait(ring.empty(stage), phase ^ 1u, abort_flag, a.dev_err);
            wt = __shfl_sync(0xffffffffu, wt, 0);
            if (!wt) {
                ok = false;
                break;
            }
            const uint32_t base = sA + stage * kTileABytes;
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (live & (1u << i)) cp_async_16(base + dst_off[i], src_row[i] + kb * kRowBytes);
            cp_async_commit();
            pend[npend++] = stage;
            if (npend > kDepth) {
                cp_async_wait<kDepth>();
                fence_proxy_async();
                mbar_arrive(ring.full(pend[0]));
#pragma unroll
                for (int q = 0; q < kDepth; ++q) pend[q] = pend[q + 1];
                --npend;
            }
            if (++stage == kSt) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
    // the stages still pending: complete, fence, publish
    cp_async_wait<0>();
    fence_proxy_async();
    for (int q = 0; q < npend; ++q) mbar_arrive(ring.full(pend[q]));
}

// MMA issuer (one thread): per tile, wait for a free accumulator, then per
// stage tcgen05.mma M=128 N=256 K=16 x 4, commit the stage back to the
// producers and the finished accumulator to the epilogue. Gate/up tiles are
// bf16 x bf16, down tiles fp16 x fp16.
template <int kSt>
__device__ void role_mma(const FfnArgs& a, const TileWalk& w, Ring ring, uint32_t sA, uint32_t sB,
                         uint32_t accf0, uint32_t acce0, uint32_t drain_bar, uint32_t tmem_base,
                         volatile int* abort_flag) {
    const uint32_t idesc_gu = make_idesc(true, 128, 256);
    const uint32_t idesc_dn = make_idesc(false, 128, 256);
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    bool issued_any = false;
    for (int it = 0, t; ok && (t = w.tile_thread(it)) >= 0; ++it) {
        const bool gu = t < w.TA;
        const int num_kb = gu ? w.KBA : w.KBB;
        const uint32_t idesc = gu ? idesc_gu : idesc_dn;
        if (!mbar_wait(acce0 + 8u * acc, acc_phase ^ 1u, abort_flag, a.dev_err)) {
            ok = false;
            break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kAccCols);
        for (int kb = 0; kb < num_kb; ++kb) {
            if (!mbar_wait(ring.full(stage), phase, abort_flag, a.dev_err)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint64_t adesc = sw128_desc(sA + stage * kTileABytes);
            const uint64_t bdesc = sw128_desc(sB + stage * kTileBBytes);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)  // 4 x 32 bytes of K per stage
                umma_f16(d_tmem, adesc + 2u * kk, bdesc + 2u * kk, idesc, (kb | kk) != 0 ? 1u : 0u);
            issued_any = true;
            umma_commit(ring.empty(stage));
            if (++stage == kSt) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (!ok) break;
        umma_commit(accf0 + 8u * acc);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
    }
    if (!ok && issued_any) {
        // wait (bounded) for the MMAs already issued before TMEM is freed
        umma_commit(drain_bar);
        mbar_wait_drain(drain_bar, 0);
    }
}

// The launch's residual rows (GemmSegments::resid_A), by its epilogue warps
// before their first tile (they wait for the first accumulator anyway; no
// tile adds into Y before the gate/up phase ends): epilogue warp w of n_warps
// writes Y[t] = fp32(A[t]) for t = w, w + n_warps, ..., four 16-byte loads
// per lane in flight, then publishes its rows with one release-add.
__device__ void residual_rows(const GemmSegments& seg, int H, int w, int n_warps, int lane) {
    float* Y = seg.resid_Y;
    const int row_bytes = H * seg.resid_elem;
    for (int t = w; t < seg.resid_T; t += n_warps) {
        const char* src = static_cast<const char*>(seg.resid_A) + static_cast<size_t>(t) * row_bytes;
        float* y = Y + static_cast<size_t>(t) * H;
        for (int base = lane * 16; base < row_bytes; base += 4 * 32 * 16) {
            uint4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int off = base + u * 32 * 16;
                if (off < row_bytes) v[u] = __ldg(reinterpret_cast<const uint4*>(src + off));
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int off = base + u * 32 * 16;
                if (off >= row_bytes) continue;
                if (seg.resid_elem == 2) {  // 8 bf16: a bf16 is the high half of its fp32
                    float4* d = reinterpret_cast<float4*>(y + off / 2);
                    d[0] = make_float4(__uint_as_float(v[u].x << 16), __uint_as_float(v[u].x & 0xFFFF0000u),
                                       __uint_as_float(v[u].y << 16), __uint_as_float(v[u].y & 0xFFFF0000u));
                    d[1] = make_float4(__uint_as_float(v[u].z << 16), __uint_as_float(v[u].z & 0xFFFF0000u),
                                       __uint_as_float(v[u].w << 16), __uint_as_float(v[u].w & 0xFFFF0000u));
                } else {
                    *reinterpret_cast<uint4*>(y + off / 4) = v[u];
                }
            }
        }
    }
    __threadfence();
    __syncwarp();
    if (lane == 0) red_release_add(seg.resid_done, 1);
}

// Before a down epilogue's first addition into Y: wait (bounded) until every
// epilogue warp of the launch has published its residual rows.
__device__ __forceinline__ bool residual_ready(const GemmSegments& seg, int n_warps, int lane,
                                               volatile int* abort_flag, int* dev_err) {
    bool ok = true;
    if (lane == 0) ok = wait_counter(seg.resid_done, n_warps, abort_flag, dev_err);
    return __shfl_sync(0xffffffffu, ok, 0);
}

// Epilogue (4 warps, TMEM lanes = records): gate/up tiles write
// h = fp16(SiLU(g) u) and publish the m-block counter; down tiles add
// alpha * scale * acc into Y (or store the row in deterministic mode).
// With a stage (shared address of 4 x kStageWarpBytes, else 0) the rows are
// written out coalesced through it.
__device__ void role_epilogue(const FfnArgs& a, const TileWalk& w, uint32_t accf0, uint32_t acce0,
                              uint32_t tmem_base, volatile int* abort_flag, int warp, int lane,
                              uint32_t stage0) {
    const GemmSegments& seg = *w.seg;
    const int quarter = warp & 3;  // TMEM lanes this warp may read
    const int row = quarter * 32 + lane;
    const uint32_t stg = stage0 + static_cast<uint32_t>(quarter * kStageWarpBytes);
    const int n_epi = static_cast<int>(gridDim.x) * 4;   // epilogue warps of the launch
    if (seg.resid_A) residual_rows(seg, a.H, static_cast<int>(blockIdx.x) * 4 + warp - 2, n_epi, lane);
    // the deterministic mode adds into Y only in the combine, a later launch
    bool resid_ok = !seg.resid_A || a.out_rows;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int it = 0, t; (t = w.tile(it)) >= 0; ++it) {
        const bool gu = t < w.TA;
        const Tile ti = w.decode(t);
        if (!gu && !resid_ok) {
            if (!residual_ready(seg, n_epi, lane, abort_flag, a.dev_err)) break;
            resid_ok = true;
        }
        bool wt = true;
        if (lane == 0) wt = mbar_wait(accf0 + 8u * acc, acc_phase, abort_flag, a.dev_err);
        wt = __shfl_sync(0xffffffffu, wt, 0);
        if (!wt) break;
        tc_fence_after();
        const bool valid = row < ti.rows;
        const int p = ti.row0 + row;
        const uint32_t tacc = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                              static_cast<uint32_t>(acc * kAccCols);
        if (gu) {
            __half* dst = a.h + static_cast<size_t>(p) * a.F + static_cast<size_t>(ti.nb) * 128;
            if (stage0)
                epilogue_gate_up_staged(tacc, valid ? dst : nullptr, stg, lane, a.dev_err);
            else
                epilogue_gate_up(tacc, valid, dst, a.dev_err);
            // publish this warp's rows of the tile to the down tiles (which
            // read h through TMA, the async proxy)
            fence_proxy_async_global();
            __threadfence();
            __syncwarp();
            if (lane == 0 && (a.phases & 2))
                red_release_add(a.done + seg.mblk[seg.seg_begin + ti.seg] + ti.mb, 1);
        } else {
            int tok = 0;
            float al = 0.0f;
            if (valid) {
                tok = seg.rec_tok[p];
                al = seg.alpha ? seg.alpha[seg.rec_route[p]] : 1.0f;
                al *= seg.seg_scale[seg.seg_begin + ti.seg];  // undo the W_d scale
            }
            float* out_row = a.out_rows ? a.out_rows + static_cast<size_t>(p) * a.H : nullptr;
            float* y_row = a.Y + static_cast<size_t>(tok) * a.H;
            if (stage0) {
                float* dst = out_row ? out_row : y_row;
                epilogue_down_staged(tacc, al, valid ? dst + ti.nb * 256 : nullptr, !out_row, stg,
                                     lane);
            } else {
                epilogue_down(tacc, valid, al, out_row, y_row, ti.nb * 256);
            }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acce0 + 8u * acc);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
    }
}

__global__ void __launch_bounds__(kThreads, 1)
    k_expert_ffn(const __grid_constant__ CUtensorMap tm_wg, const __grid_constant__ CUtensorMap tm_wu,
                 const __grid_constant__ CUtensorMap tm_wd, const __grid_constant__ CUtensorMap tm_h,
                 const FfnArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const GemmSegments& seg = a.seg;
    const uint32_t sbase = smem_addr(smem);
    const uint32_t sA = sbase + kOffA;
    const uint32_t sB = sbase + kOffB;
    const uint32_t bar0 = sbase + kOffBar;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kStages + s); };
    auto accf_bar = [&](int q) { return bar0 + 8u * (2 * kStages + q); };
    auto acce_bar = [&](int q) { return bar0 + 8u * (2 * kStages + 2 + q); };
    const uint32_t drain_bar = bar0 + 8u * (2 * kStages + 4);
    const uint32_t tfull0 = bar0 + 8u * (2 * kStages + 5);
    const uint32_t tempty0 = tfull0 + 8u * kTileRing;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
    volatile int* tile_ring = reinterpret_cast<volatile int*>(smem + kOffRing);
    int* table = reinterpret_cast<int*>(smem + kOffTable);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // m-block prefix of the segment range, relative to its first segment
    const int m0 = seg.mblk[seg.seg_begin];
    for (int s = threadIdx.x; s <= seg.seg_count; s += blockDim.x)
        table[s] = seg.mblk[seg.seg_begin + s] - m0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full_bar(s), 1 + kBM);  // producer's expect_tx + one per loader thread
            mbar_init(empty_bar(s), 1);
        }
        for (int q = 0; q < 2; ++q) {
            mbar_init(accf_bar(q), 1);
            mbar_init(acce_bar(q), 4);  // one arrival per epilogue warp
        }
        mbar_init(drain_bar, 1);
        for (int r = 0; r < kTileRing; ++r) {
            mbar_init(tfull0 + 8u * r, 1);
            mbar_init(tempty0 + 8u * r, 4 + 1 + 4);  // loader warps, MMA thread, epilogue warps
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int H = a.H, F = a.F;
    const int NBA = F / 128, NBB = H / 256;   // n-blocks of gate/up and of down tiles
    const int KBA = H / 64, KBB = F / 64;     // k-blocks (64 elements = 128 bytes)
    const int MB = table[seg.seg_count];
    const int TA = (a.phases & 1) ? MB * NBA : 0;
    const int TB = (a.phases & 2) ? MB * NBB : 0;
    const int done_target = 4 * NBA;          // every epilogue warp of every gate/up n-block
    const TileWalk walk{&seg,     table,     TA,     TB,         NBA,       NBB, KBA,
                        KBB,      a.ticket,  tile_ring, tfull0, tempty0, abort_flag, a.dev_err};
    const Ring ring{full_bar(0), empty_bar(0)};

    if (warp == 0) {
        // ------------------------------ TMA producer (weights) ------------------------------
        int stage = 0;
        uint32_t phase = 0;
        const uint64_t evict_first = policy_evict_first();
        int issued[kStages];
        for (int s = 0; s < kStages; ++s) issued[s] = -1;
        bool ok = true;
        int pending = lane == 0 ? walk.first_ticket() : 0;
        auto next_tile = [&](int it) {
            int t = 0;
            if (lane == 0) t = walk.publish(it, pending);
            return __shfl_sync(0xffffffffu, t, 0);
        };
        for (int it = 0, t; ok && (t = next_tile(it)) >= 0; ++it) {
            const bool gu = t < TA;
            const Tile ti = walk.decode(t);
            const int slot = seg.slot_base + ti.seg;
            // weight planes are tile-major: the (n-block, k-block) box of a slot
            // is one contiguous run of 128 (gate/up) or 256 (down) rows of 128 B
            const int num_kb = gu ? KBA : KBB;
            const int tile_rows = gu ? 128 : 256;
            const int brow0 = (slot * (gu ? NBA : NBB) + ti.nb) * num_kb * tile_rows;
            // a segment of one m-block is its weight tiles' only reader: those
            // tiles are loaded evict-first (tiles read by further m-blocks keep
            // the default policy; marking them measured slower)
            const bool only_reader = table[ti.seg + 1] - table[ti.seg] == 1;
            if (!gu) {
                // the m-block's h rows are complete once every epilogue warp of
                // every gate/up n-block has published
                const int* cnt = a.done + seg.mblk[seg.seg_begin + ti.seg] + ti.mb;
                bool w = true;
                if (lane == 0) w = wait_counter(cnt, done_target, abort_flag, a.dev_err);
                if (lane == 0) fence_proxy_async_global();  // before the TMA reads of h
                w = __shfl_sync(0xffffffffu, w, 0);
                if (!w) {
                    ok = false;
                    break;
                }
            }
            for (int kb = 0; kb < num_kb; ++kb) {
                bool w = true;
                if (lane == 0) w = mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, a.dev_err);
                w = __shfl_sync(0xffffffffu, w, 0);
                if (!w) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    mbar_arrive_expect_tx(full_bar(stage),
                                          gu ? kTileBBytes : kTileBBytes + kTileABytes);
                    issued[stage] = static_cast<int>(phase);
                    const uint32_t b_dst = sB + stage * kTileBBytes;
                    const int brow = brow0 + kb * tile_rows;
                    if (gu) {
                        if (only_reader) {
                            tma_load_2d_hint(b_dst, &tm_wg, 0, brow, full_bar(stage), evict_first);
                            tma_load_2d_hint(b_dst + 128 * kRowBytes, &tm_wu, 0, brow,
                                             full_bar(stage), evict_first);
                        } else {
                            tma_load_2d(b_dst, &tm_wg, 0, brow, full_bar(stage));
                            tma_load_2d(b_dst + 128 * kRowBytes, &tm_wu, 0, brow, full_bar(stage));
                        }
                    } else {
                        tma_load_2d(sA + stage * kTileABytes, &tm_h, kb * 64, ti.row0,
                                    full_bar(stage));
                        if (only_reader)
                            tma_load_2d_hint(b_dst, &tm_wd, 0, brow, full_bar(stage), evict_first);
                        else
                            tma_load_2d(b_dst, &tm_wd, 0, brow, full_bar(stage));
                    }
                }
                __syncwarp();
                if (++stage == kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (!ok && lane == 0) {
            // let every copy already issued land before the CTA goes away
            for (int s = 0; s < kStages; ++s)
                if (issued[s] >= 0) mbar_wait_drain(full_bar(s), static_cast<uint32_t>(issued[s]));
        }
    } else if (warp >= kLoaderWarp0) {
        role_gather<kStages, kLoaderDepth>(a, walk, ring, sA, abort_flag, warp - kLoaderWarp0, lane);
    } else if (warp == 1) {
        if (lane == 0)
            role_mma<kStages>(a, walk, ring, sA, sB, accf_bar(0), acce_bar(0), drain_bar, tmem_base,
                              abort_flag);
        __syncwarp();
    } else {
        role_epilogue(a, walk, accf_bar(0), acce_bar(0), tmem_base, abort_flag, warp, lane,
                      sbase + kOffStg);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

// ----------------------------------------------------------------------------
// 4-bit expert weights, single-SM form
// ----------------------------------------------------------------------------
// The weight planes hold Q4_0-style blocks (section 4 of the paper stores
// expert matrices as weight-only GGUF Q4_0): per (n-block, k-block) box of
// R rows, two column blocks of codes -- block j holds each row's 16 bytes of
// weights 32j..32j+31 (in byte-word w, bits 4i..4i+3 hold k = 32j + 8w + 2i
// and bits 16 + 4i.. hold k = 32j + 8w + 2i + 1), so a row's halves sit
// R * 16 bytes apart -- followed by the rows' two block scales (bf16 for gate
// and up, fp16 for down), a value being (q - 8) * d. Roles: warp 0 streams packed boxes with plain bulk
// copies into a 3-deep ring (a stage is 9 KB instead of 32 KB of bf16);
// warps 10-13 expand each packed stage into the 128-byte-swizzled bf16/fp16
// B tile of the 4-deep MMA ring -- the paper's "vector workers decode them into
// matrix-engine operands" (section 3.2) -- and, for down tiles, wait for the
// m-block's h rows and load them with TMA; the gather, MMA and epilogue roles
// are the bf16 kernel's. Every expanded operand is exact: (q - 8) and d each
// have at most 5 significant bits, so their product fits bf16 and fp16.
constexpr int kQStages = 4;                   // MMA ring (expanded operands)
constexpr int kQPStages = 3;                  // packed-weight ring
constexpr int kQMaxSegs = kMaxE;              // segments are experts of one layer
constexpr int kQBoxGU = 128 * 32 + 128 * 4;   // 4608 B: one gate or up box
constexpr int kQBoxDn = 256 * 32 + 256 * 4;   // 9216 B: one down box
constexpr int kQPBytes = kQBoxDn;             // a packed stage: gate + up, or down
constexpr int kConvWarps = 8;                 // one B row per converter thread and stage
constexpr int kQThreads = 320 + 32 * kConvWarps;
constexpr int kConvWarp0 = 10;
constexpr int kQOffA = 0;
constexpr int kQOffB = kQStages * kTileABytes;
constexpr int kQOffP = kQOffB + kQStages * kTileBBytes;
constexpr int kQOffBar = kQOffP + kQPStages * kQPBytes;
// barriers: full[4], empty[4], pfull[3], pempty[3], acc_full[2], acc_empty[2], drain,
// tile_full[4], tile_empty[4]
constexpr int kQNumBars = 2 * kQStages + 2 * kQPStages + 5 + 2 * 4;
constexpr int kQOffMisc = kQOffBar + 8 * kQNumBars;
constexpr int kQOffRing = kQOffMisc + 16;
constexpr int kQOffTable = kQOffRing + 16;

size_t q4_smem_bytes(int seg_count) {
    return 1024 + kQOffTable + sizeof(int) * static_cast<size_t>(seg_count + 1);
}

struct Q4Planes {
    const uint8_t* g;  // slot s of the gate plane at g + s * S_gu
    const uint8_t* u;
    const uint8_t* d;  // slot s of the down plane at d + s * S_d
    size_t S_gu, S_d;
};

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Expand one packed row (64 codes: 16 bytes at codes_lo, 16 at codes_hi; two
// block scales) into 64 operands of B-tile row r: 8 chunks of 16 bytes,
// chunk c at (c ^ (r mod 8)) * 16. A code
// q becomes the number 128 + q (bf16 0x4300 | q) or 1024 + q (fp16
// 0x6400 | q) by bit placement; subtracting 136 (1032) gives q - 8 and the
// multiplication by d the weight, both exact.
template <bool kFp16>
__device__ __forceinline__ void expand_row(uint32_t codes_lo, uint32_t codes_hi, uint32_t scales,
                                           uint32_t dst_row, int r) {
    uint32_t w[8], sc;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]) : "r"(codes_lo));
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7]) : "r"(codes_hi));
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(sc) : "r"(scales));
    const uint32_t magic = kFp16 ? 0x64006400u : 0x43004300u;
    const uint32_t offset = kFp16 ? 0x64086408u : 0x43084308u;
    const uint32_t d_lo = (sc & 0xFFFFu) * 0x10001u;  // block 0's scale in both halves
    const uint32_t d_hi = (sc >> 16) * 0x10001u;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const uint32_t d2 = c < 4 ? d_lo : d_hi;
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t v = ((w[c] >> (4 * i)) & 0x000F000Fu) | magic;
            uint32_t t;
            if (kFp16) {
                asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(t) : "r"(v), "r"(offset));
                asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(o[i]) : "r"(t), "r"(d2));
            } else {
                asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(t) : "r"(v), "r"(offset));
                asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(o[i]) : "r"(t), "r"(d2));
            }
        }
        const uint32_t dst = dst_row + ((static_cast<uint32_t>(c) ^ static_cast<uint32_t>(r & 7)) << 4);
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(o[0]), "r"(o[1]),
                     "r"(o[2]), "r"(o[3])
                     : "memory");
    }
}

// Converter warps (cw = 0..7, thread ct = 32 cw + lane expands B row ct of
// every stage: rows 0-127 the gate box, 128-255 the up box, or the 256 rows
// of the down box).
__device__ void role_convert(const FfnArgs& a, const TileWalk& w, Ring ring, Ring pring, uint32_t sA,
                             uint32_t sB, uint32_t sP, const CUtensorMap* tm_h, int done_target,
                             volatile int* abort_flag, int cw, int lane) {
    const GemmSegments& seg = *w.seg;
    const int ct = cw * 32 + lane;
    int g = 0;
    bool ok = true;
    for (int it = 0, t; ok && (t = w.tile(it)) >= 0; ++it) {
        const bool gu = t < w.TA;
        const Tile ti = w.decode(t);
        const int num_kb = gu ? w.KBA : w.KBB;
        for (int kb = 0; kb < num_kb; ++kb, ++g) {
            const int s = g % kQStages;
            const uint32_t ph = static_cast<uint32_t>(g / kQStages) & 1u;
            const int ps = g % kQPStages;
            const uint32_t pph = static_cast<uint32_t>(g / kQPStages) & 1u;
            bool wt = true;
            if (lane == 0)
                wt = mbar_wait(pring.full(ps), pph, abort_flag, a.dev_err) &&
                     mbar_wait(ring.empty(s), ph ^ 1u, abort_flag, a.dev_err);
            if (!gu && kb == 0 && cw == 0 && lane == 0 && wt) {
                // the m-block's h rows are complete once every epilogue warp
                // of every gate/up n-block has published
                wt = wait_counter(a.done + seg.mblk[seg.seg_begin + ti.seg] + ti.mb, done_target,
                                  abort_flag, a.dev_err);
                fence_proxy_async_global();  // before the TMA reads of h
            }
            wt = __shfl_sync(0xffffffffu, wt, 0);
            if (!wt) {
                ok = false;
                break;
            }
            const uint32_t pb = sP + ps * kQPBytes;
            const uint32_t bb = sB + s * kTileBBytes;
            if (gu) {
                const uint32_t box = pb + (ct < 128 ? 0u : static_cast<uint32_t>(kQBoxGU));
                const int r = ct & 127;
                expand_row<false>(box + r * 16, box + 2048 + r * 16, box + 4096 + r * 4,
                                  bb + ct * kRowBytes, ct);
            } else {
                expand_row<true>(pb + ct * 16, pb + 4096 + ct * 16, pb + 8192 + ct * 4,
                                 bb + ct * kRowBytes, ct);
            }
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) {
                if (!gu && cw == 0) {
                    mbar_arrive_expect_tx(ring.full(s), kTileABytes);
                    tma_load_2d(sA + s * kTileABytes, tm_h, kb * 64, ti.row0, ring.full(s));
                } else {
                    mbar_arrive(ring.full(s));
                }
                mbar_arrive(pring.empty(ps));
            }
        }
    }
    if (!ok && cw == 0 && lane == 0) {
        // give an h load already issued time to land before the CTA goes away
        const uint64_t t0 = global_ns();
        while (global_ns() - t0 < kDrainLimitNs / 100) {
        }
    }
}

__global__ void __launch_bounds__(kQThreads, 1)
    k_expert_ffn_q4(const __grid_constant__ CUtensorMap tm_h, const Q4Planes planes, const FfnArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const GemmSegments& seg = a.seg;
    const uint32_t sbase = smem_addr(smem);
    const uint32_t sA = sbase + kQOffA;
    const uint32_t sB = sbase + kQOffB;
    const uint32_t sP = sbase + kQOffP;
    const uint32_t bar0 = sbase + kQOffBar;
    const Ring ring{bar0, bar0 + 8u * kQStages};
    const Ring pring{bar0 + 8u * (2 * kQStages), bar0 + 8u * (2 * kQStages + kQPStages)};
    const uint32_t accf0 = bar0 + 8u * (2 * kQStages + 2 * kQPStages);
    const uint32_t acce0 = accf0 + 16u;
    const uint32_t drain_bar = acce0 + 16u;
    const uint32_t tfull0 = drain_bar + 8u;
    const uint32_t tempty0 = tfull0 + 8u * kTileRing;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kQOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kQOffMisc + 4);
    volatile int* tile_ring = reinterpret_cast<volatile int*>(smem + kQOffRing);
    int* table = reinterpret_cast<int*>(smem + kQOffTable);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    const int m0 = seg.mblk[seg.seg_begin];
    for (int s = threadIdx.x; s <= seg.seg_count; s += blockDim.x)
        table[s] = seg.mblk[seg.seg_begin + s] - m0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kQStages; ++s) {
            mbar_init(ring.full(s), kBM + kConvWarps);  // one per loader thread + one per converter warp
            mbar_init(ring.empty(s), 1);
        }
        for (int s = 0; s < kQPStages; ++s) {
            mbar_init(pring.full(s), 1);   // the producer's expect_tx
            mbar_init(pring.empty(s), kConvWarps);  // one per converter warp
        }
        for (int q = 0; q < 2; ++q) {
            mbar_init(accf0 + 8u * q, 1);
            mbar_init(acce0 + 8u * q, 4);
        }
        mbar_init(drain_bar, 1);
        for (int r = 0; r < kTileRing; ++r) {
            mbar_init(tfull0 + 8u * r, 1);
            // loader warps, MMA thread, epilogue warps, converter warps
            mbar_init(tempty0 + 8u * r, 4 + 1 + 4 + kConvWarps);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int H = a.H, F = a.F;
    const int NBA = F / 128, NBB = H / 256;
    const int KBA = H / 64, KBB = F / 64;
    const int MB = table[seg.seg_count];
    const int TA = (a.phases & 1) ? MB * NBA : 0;
    const int TB = (a.phases & 2) ? MB * NBB : 0;
    const TileWalk walk{&seg,     table,     TA,     TB,         NBA,       NBB, KBA,
                        KBB,      a.ticket,  tile_ring, tfull0, tempty0, abort_flag, a.dev_err};

    if (warp == 0) {
        // ------------------------------ packed-weight producer ------------------------------
        if (lane == 0) {
            int issued[kQPStages];
            for (int s = 0; s < kQPStages; ++s) issued[s] = -1;
            bool ok = true;
            int g = 0;
            int pending = walk.first_ticket();
            for (int it = 0, t; ok && (t = walk.publish(it, pending)) >= 0; ++it) {
                const bool gu = t < TA;
                const Tile ti = walk.decode(t);
                const size_t slot = static_cast<size_t>(seg.slot_base + ti.seg);
                const int num_kb = gu ? KBA : KBB;
                const uint8_t* src0 = gu ? planes.g + slot * planes.S_gu + static_cast<size_t>(ti.nb) * KBA * kQBoxGU
                                         : planes.d + slot * planes.S_d + static_cast<size_t>(ti.nb) * KBB * kQBoxDn;
                const uint8_t* src1 = planes.u + slot * planes.S_gu + static_cast<size_t>(ti.nb) * KBA * kQBoxGU;
                for (int kb = 0; kb < num_kb; ++kb, ++g) {
                    const int ps = g % kQPStages;
                    const uint32_t pph = static_cast<uint32_t>(g / kQPStages) & 1u;
                    if (!mbar_wait(pring.empty(ps), pph ^ 1u, abort_flag, a.dev_err)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(pring.full(ps), kQPBytes);
                    issued[ps] = static_cast<int>(pph);
                    const uint32_t dst = sP + ps * kQPBytes;
                    if (gu) {
                        bulk_load(dst, src0 + static_cast<size_t>(kb) * kQBoxGU, kQBoxGU, pring.full(ps));
                        bulk_load(dst + kQBoxGU, src1 + static_cast<size_t>(kb) * kQBoxGU, kQBoxGU,
                                  pring.full(ps));
                    } else {
                        bulk_load(dst, src0 + static_cast<size_t>(kb) * kQBoxDn, kQBoxDn, pring.full(ps));
                    }
                }
            }
            if (!ok)
                for (int s = 0; s < kQPStages; ++s)
                    if (issued[s] >= 0) mbar_wait_drain(pring.full(s), static_cast<uint32_t>(issued[s]));
        }
        __syncwarp();
    } else if (warp >= kConvWarp0) {
        role_convert(a, walk, ring, pring, sA, sB, sP, &tm_h, 4 * NBA, abort_flag, warp - kConvWarp0, lane);
    } else if (warp >= kLoaderWarp0) {
        role_gather<kQStages, kLoaderDepth>(a, walk, ring, sA, abort_flag, warp - kLoaderWarp0, lane);
    } else if (warp == 1) {
        if (lane == 0)
            role_mma<kQStages>(a, walk, ring, sA, sB, accf0, acce0, drain_bar, tmem_base, abort_flag);
        __syncwarp();
    } else {
        role_epilogue(a, walk, accf0, acce0, tmem_base, abort_flag, warp, lane, 0u);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

// ----------------------------------------------------------------------------
// CTA-pair form: tcgen05.mma.cta_group::2, M = 256 rows over two SMs.
// ----------------------------------------------------------------------------
// A pair tile is (segment, n-block, pair m-block of 256 records). CTA r of the
// cluster pair owns records [128r, 128r+128) of the pair m-block: it gathers
// (gate/up) or TMA-loads (down, h) its 128 A rows, and holds half of the
// N = 256 B tile -- rank 0 the gate rows, rank 1 the up rows of the h n-block;
// or rows [128r, 128r+128) of the 256-row W_d box. The leader (rank 0) issues
// the MMAs, which read both CTAs' shared memory; each CTA receives its 128
// rows of the 128 x 256 fp32 result in its own TMEM, so the epilogue is the
// single-CTA one. Per SM a stage is 32 KB (A 16 KB + half of B 16 KB) instead
// of 48 KB for the same 128 x 256 x 64 of MMA work per SM, so the ring holds
// six stages and each weight byte crosses from L2 to the SMs once per pair.
// Completion: every stage's TMA bytes and loader arrivals land on the
// leader's full barrier; the leader's commits are multicast to both CTAs'
// empty and accumulator-full barriers; both CTAs' epilogue warps arrive on
// the leader's accumulator-empty barrier.
constexpr int kPStages = 6;                            // MMA ring of the bf16 form
constexpr int kPHalf = 128 * kRowBytes;                // 16 KB
constexpr int kPOffA = 0;
constexpr int kPairRows = 2 * kBM;
constexpr int kLoaderWarps = 4;
constexpr int kEpiWarps = 4;
constexpr int kSplitMinKb = 128;   // down tiles of at least this many k-blocks are split in K

// 4-bit weights in the pair form: each CTA streams only its half of a packed
// box (the gate box on rank 0 and the up box on rank 1, or rows
// [128 r, 128 r + 128) of the down box: 4608 bytes either way) into a
// 3-deep packed ring, and four converter warps (one B row per thread)
// expand it into the CTA's half of the operand tile -- half of the
// conversion of the single-SM 4-bit kernel per SM.
constexpr int kPQConvWarps = 4;
constexpr int kPQConvWarp0 = 10;
constexpr int kPQThreads = kThreads + 32 * kPQConvWarps;
// Measured: five MMA stages with nine packed stages are no faster, and eight
// converter warps of half a row each are slower (the block's registers then
// spill): the conversion is bound by the SM's instruction issue, shared with
// the other roles.
constexpr int kPQStages = 6;    // MMA ring of the 4-bit form
constexpr int kPQPStages = 3;   // packed-weight ring
constexpr int kPQBox = 128 * 32 + 128 * 4;  // 4608 B

// Shared-memory map of a pair-kernel form: A and B halves of the MMA ring,
// the epilogue stages, the packed ring (4-bit form), barriers, misc, table.
struct PairLayout {
    int stages, pstages, off_b, off_stg, off_pk, off_bar, num_bars, off_misc, off_table;
};
__host__ __device__ constexpr PairLayout pair_layout(bool q4) {
    const int st = q4 ? kPQStages : kPStages;
    const int pst = q4 ? kPQPStages : 0;
    const int off_b = st * kPHalf;
    const int off_stg = off_b + st * kPHalf;
    const int off_pk = off_stg + 4 * 32 * 128;
    const int off_bar = off_pk + pst * kPQBox;
    const int num_bars = 2 * st + 5 + 2 * pst;
    const int off_misc = off_bar + 8 * num_bars;
    return PairLayout{st, pst, off_b, off_stg, off_pk, off_bar, num_bars, off_misc, off_misc + 16};
}

// The launch's segment offsets are copied next to the segment table when
// that fits the shared memory of the largest table (seg_count + 1 at most
// half of it), so a tile decode reads no global memory.
constexpr int pair_seg_cap(bool q4) { return q4 ? kQMaxSegs : kMaxP; }
__host__ __device__ constexpr bool pair_offsets_cached(int seg_count, bool q4) {
    return 2 * (seg_count + 1) <= (q4 ? kQMaxSegs : kMaxP) + 1;
}
size_t pair_smem_bytes(int seg_count, bool q4 = false) {
    const size_t n = static_cast<size_t>(seg_count + 1);
    return 1024 + pair_layout(q4).off_table + sizeof(int) * n +
           (pair_offsets_cached(seg_count, q4) ? sizeof(int) * n : 0);
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Address of the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_rank(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cl(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// mbar_wait with cluster-scope acquire (arrivals come from the peer CTA).
// The cluster-scope form of mbar_wait_drain (ignores the abort flag).
__device__ bool mbar_wait_cl_drain(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait_cl(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait_cl(bar, parity))
        if (global_ns() - t0 > kDrainLimitNs) return false;
    return true;
}

__device__ bool mbar_wait_cl(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* dev_err) {
    if (mbar_try_wait_cl(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    uint32_t spins = 0;
    while (true) {
        if (mbar_try_wait_cl(bar, parity)) return true;
        if ((++spins & 63u) == 0) {
            if (*abort_flag) return false;
            if (global_ns() - t0 > kWaitLimitNs) {
                *abort_flag = 1;
                record_error(dev_err, kDevErrTimeout);
                return false;
            }
        }
    }
}
// Release of this thread's shared-memory writes at cluster scope, restricted
// to shared::cta memory (lighter than a full cluster-scope release, which
// also waits for the thread's global-memory traffic), followed by a relaxed
// arrival on a barrier of the peer CTA: the hand-off of a shared-memory
// payload to the other CTA of the pair.
__device__ __forceinline__ void mbar_arrive_remote_smem_release(uint32_t cl_addr) {
    asm volatile(
        "fence.release.sync_restrict::shared::cta.cluster;\n\t"
        "mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cl_addr)
        : "memory");
}
// Arrive on a barrier given by its shared::cluster address (either CTA).
__device__ __forceinline__ void mbar_arrive_cl(uint32_t cl_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cl_addr)
                 : "memory");
}
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* tm, int x, int y,
                                                 uint32_t cl_bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(cl_bar)
        : "memory");
}
__device__ __forceinline__ void tma_load_2d_pair_hint(uint32_t dst, const CUtensorMap* tm, int x,
                                                      int y, uint32_t cl_bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(cl_bar), "l"(policy)
        : "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void umma_f16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                              uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive once on the barrier at offset `bar` in both CTAs of the pair when
// the MMAs issued so far have completed.
__device__ __forceinline__ void umma_commit_pair(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(bar),
        "h"(static_cast<uint16_t>(3))
        : "memory");
}

// A pair tile covers 256 records (M = 256: 128 per CTA), except the last one
// of a segment whose remainder fits 128 records: that one is a half tile
// (M = 128: 64 records per CTA), which costs half the MMA time -- so a
// segment pads to a multiple of 128 records, not 256. In a half tile the
// accumulator rows land in TMEM lanes 0-63 of each CTA, read by the epilogue
// warps of quarters 0 and 1; the other quarters hold no valid rows.
struct PairTile {
    int seg;     // segment index relative to seg_begin
    int pm;      // pair m-block inside the segment
    int nb;      // n-block
    int row0;    // first record of this CTA's part
    int rows;    // valid records in this CTA's part (0..kBM, 0..kBM/2 in a half tile)
    int rows1;   // valid records in rank 1's part
    bool half;   // M = 128 tile
    int cnt;     // m-block counter of this CTA's h rows, relative to the segment's first
    int npub;    // CTAs whose epilogues publish on that counter per gate/up tile
};

// kMFirst: inside a segment the tiles run m-block-major (all n-blocks of pair
// m-block 0, then of m-block 1, ...) instead of n-block-major.
template <bool kMFirst>
__device__ __forceinline__ PairTile decode_pair(int t, const int* table, int seg_count, int NB,
                                                const int32_t* offsets, int seg_begin, int rank,
                                                bool allow_half = true) {
    int lo = 0, hi = seg_count;  // largest lo with table[lo] * NB <= t
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (table[mid] * NB <= t) lo = mid; else hi = mid;
    }
    PairTile ti;
    ti.seg = lo;
    const int npm = table[lo + 1] - table[lo];
    const int l = t - table[lo] * NB;
    if (kMFirst) {
        ti.pm = l / NB;
        ti.nb = l - ti.pm * NB;
    } else {
        ti.nb = l / npm;
        ti.pm = l - ti.nb * npm;
    }
    const int s_lo = offsets[seg_begin + lo];
    const int s_hi = offsets[seg_begin + lo + 1];
    const int pr0 = s_lo + ti.pm * kPairRows;
    const int tot = min(kPairRows, s_hi - pr0);
    ti.half = allow_half && tot <= kBM;
    // records [pr0, pr0 + tot) are the single m-blocks 2 pm (and 2 pm + 1):
    // in a full tile rank r's rows are m-block 2 pm + r with its own counter;
    // a half tile is one m-block whose counter both ranks publish on
    const int part = ti.half ? kBM / 2 : kBM;
    ti.row0 = pr0 + part * rank;
    ti.rows = max(0, min(part, tot - part * rank));
    ti.rows1 = max(0, min(part, tot - part));
    ti.cnt = 2 * ti.pm + (ti.half ? 0 : rank);
    ti.npub = ti.half ? 1 + (tot > part ? 1 : 0) : 1;
    return ti;
}

// kQ4: 4-bit weights (Q4Planes, packed producer and converter warps in
// place of the weight TMA; no half tiles, whose B half mixes gate and up
// rows). The bf16 form ignores `planes`, the 4-bit form the weight maps.
// kMFirst: the m-block-major tile order (decode_pair), for launches whose
// weights stay in L2 across m-blocks (shared experts): a down tile needs
// every gate/up n-block of its m-block, and in this order the first m-blocks
// complete early, so pairs that finish their gate/up tiles find down tiles
// ready instead of waiting for the end of the gate/up phase.
template <bool kQ4, bool kMFirst>
__global__ void __launch_bounds__(kQ4 ? kPQThreads : kThreads, 1)
    k_expert_ffn_pair(const __grid_constant__ CUtensorMap tm_wg,
                      const __grid_constant__ CUtensorMap tm_wu,
                      const __grid_constant__ CUtensorMap tm_wd,
                      const __grid_constant__ CUtensorMap tm_h,
                      const __grid_constant__ CUtensorMap tm_wg64,
                      const __grid_constant__ CUtensorMap tm_wu64, const Q4Planes planes,
                      const FfnArgs a) {
    constexpr int kNT = kQ4 ? kPQThreads : kThreads;
    constexpr bool kHalfTiles = !kQ4;
    extern __shared__ uint8_t smem_raw[];
    __shared__ int warp_total[kNT / 32];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    // The cta_group::2 tensor-memory and MMA instructions, the peer-CTA
    // addresses and the leader's barriers all assume a cluster of exactly two
    // CTAs. A launch of any other shape (for example a tool relaunching the
    // kernel without its cluster attribute) returns here, before any of them,
    // with an error recorded, instead of executing pair instructions outside
    // a pair. The test is uniform over the grid.
    if (cluster_num_ctas() != 2) {
        if (threadIdx.x == 0) record_error(a.dev_err, kDevErrLaunch);
        return;
    }
    const GemmSegments& seg = a.seg;
    const uint32_t rank = cluster_rank();
    const int pair = static_cast<int>(blockIdx.x >> 1);
    const int n_pairs = static_cast<int>(gridDim.x >> 1);
    constexpr PairLayout kL = pair_layout(kQ4);
    constexpr int kST = kL.stages;      // MMA ring stages
    constexpr int kPST = kL.pstages;    // packed ring stages (4-bit form)
    constexpr int kPSTm = kPST > 0 ? kPST : 1;  // its modulus (the bf16 form never uses it)
    constexpr int kOffMisc = kL.off_misc;
    constexpr int kOffTable = kL.off_table;
    const uint32_t sbase = smem_addr(smem);
    const uint32_t sA = sbase + kPOffA;
    const uint32_t sB = sbase + kL.off_b;
    const uint32_t sPk = sbase + kL.off_pk;  // packed ring (4-bit form)
    const uint32_t bar0 = sbase + kL.off_bar;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kST + s); };
    auto accf_bar = [&](int q) { return bar0 + 8u * (2 * kST + q); };
    auto acce_bar = [&](int q) { return bar0 + 8u * (2 * kST + 2 + q); };
    const uint32_t drain_bar = bar0 + 8u * (2 * kST + 4);
    auto pfull_bar = [&](int s) { return bar0 + 8u * (2 * kST + 5 + s); };
    auto pempty_bar = [&](int s) { return bar0 + 8u * (2 * kST + 5 + kPST + s); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
    int* table = reinterpret_cast<int*>(smem + kOffTable);
    // the segment offsets (relative to seg_begin), in shared memory when cached
    const bool offs_cached = pair_offsets_cached(seg.seg_count, kQ4);
    int* offs_cache = table + seg.seg_count + 1;
    const int32_t* offs = offs_cached ? offs_cache : seg.offsets + seg.seg_begin;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // pair m-blocks per segment (ceil(count / 256)), exclusive prefix in table
    {
        const int n = seg.seg_count;
        const int per = (n + kNT - 1) / kNT;
        const int lo = min(n, static_cast<int>(threadIdx.x) * per);
        const int hi = min(n, lo + per);
        int sum = 0;
        for (int s = lo; s < hi; ++s) {
            const int s0 = seg.offsets[seg.seg_begin + s];
            const int cnt = seg.offsets[seg.seg_begin + s + 1] - s0;
            if (offs_cached) offs_cache[s] = s0;
            sum += (cnt + kPairRows - 1) / kPairRows;
        }
        if (offs_cached && threadIdx.x == kNT - 1) offs_cache[n] = seg.offsets[seg.seg_begin + n];
        int incl = sum;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl += v;
        }
        if (lane == 31) warp_total[warp] = incl;
        __syncthreads();
        int run = incl - sum;
        for (int w = 0; w < warp; ++w) run += warp_total[w];
        for (int s = lo; s < hi; ++s) {
            table[s] = run;
            const int cnt = seg.offsets[seg.seg_begin + s + 1] - seg.offsets[seg.seg_begin + s];
            run += (cnt + kPairRows - 1) / kPairRows;
        }
        if (threadIdx.x == kNT - 1) table[n] = run;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < kST; ++s) {
            // leader: the expect_tx (producer, or converter warp 0 in the 4-bit
            // form) + one arrival per loader warp -- and per converter warp --
            // of both CTAs (the peer's full barriers stay unused)
            mbar_init(full_bar(s), 1 + 2 * kLoaderWarps + (kQ4 ? 2 * kPQConvWarps : 0));
            mbar_init(empty_bar(s), 1);
        }
        if (kQ4)
            for (int s = 0; s < kPST; ++s) {
                mbar_init(pfull_bar(s), 1);                // the packed producer's expect_tx
                mbar_init(pempty_bar(s), kPQConvWarps);   // one per converter warp
            }
        for (int q = 0; q < 2; ++q) {
            mbar_init(accf_bar(q), 1);
            mbar_init(acce_bar(q), 2 * kEpiWarps);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_addr(tmem_slot), kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // both CTAs' barriers exist before any remote arrival
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int H = a.H, F = a.F;
    const int NBA = F / 128, NBB = H / 256;
    const int KBA = H / 64, KBB = F / 64;
    // A long down tile is split in two halves of its K range, each adding its
    // partial product into Y (not in the deterministic mode, which stores
    // rows): the unit the tile hand-out balances halves (on the Mixtral shape
    // a whole down tile is 224 k-blocks, ~5% of a pair's work). Down tile
    // column v is n-block v / KS, K half v % KS.
    const int KS = (!kQ4 && !a.out_rows && KBB >= kSplitMinKb && KBB % 2 == 0) ? 2 : 1;
    const int NBBv = NBB * KS;
    const int KBBs = KBB / KS;   // k-blocks of a down tile
    const int PM = table[seg.seg_count];
    const int TA = (a.phases & 1) ? PM * NBA : 0;
    const int TB = (a.phases & 2) ? PM * NBBv : 0;
    const int done_target = kEpiWarps * NBA;

    if (kQ4 && warp == 0) {
        // ------------------------------ packed-weight producer (4-bit) ------------------------------
        // this CTA's half of every packed box: the gate (rank 0) or up (rank 1)
        // box of the n-block, or rows [128 r, 128 r + 128) of the down box,
        // laid out in the stage as [codes 0-31: 2 KB][codes 32-63: 2 KB][scales: 512 B]
        if (lane == 0) {
            int issued[kPST > 0 ? kPST : 1];
            for (int q = 0; q < kPST; ++q) issued[q] = -1;
            bool ok = true;
            int g = 0;
            for (int it = 0, t; ok && (t = tile_of(pair, n_pairs, TA, TB, KBA, KBBs, it)) >= 0; ++it) {
                const bool gu = t < TA;
                const PairTile ti = decode_pair<kMFirst>(gu ? t : t - TA, table, seg.seg_count,
                                                gu ? NBA : NBBv, offs, 0,
                                                static_cast<int>(rank), kHalfTiles);
                const size_t slot = static_cast<size_t>(seg.slot_base + ti.seg);
                const int num_kb = gu ? KBA : KBBs;
                const uint8_t* box0 =
                    gu ? (rank == 0 ? planes.g : planes.u) + slot * planes.S_gu +
                             static_cast<size_t>(ti.nb) * KBA * kQBoxGU
                       : planes.d + slot * planes.S_d + static_cast<size_t>(ti.nb) * KBB * kQBoxDn;
                for (int kb = 0; kb < num_kb; ++kb, ++g) {
                    const int ps = g % kPSTm;
                    const uint32_t pph = static_cast<uint32_t>(g / kPSTm) & 1u;
                    if (!mbar_wait(pempty_bar(ps), pph ^ 1u, abort_flag, a.dev_err)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(pfull_bar(ps), kPQBox);
                    issued[ps] = static_cast<int>(pph);
                    const uint32_t dst = sPk + ps * kPQBox;
                    if (gu) {
                        bulk_load(dst, box0 + static_cast<size_t>(kb) * kQBoxGU, kPQBox, pfull_bar(ps));
                    } else {
                        const uint8_t* box = box0 + static_cast<size_t>(kb) * kQBoxDn;
                        bulk_load(dst, box + 2048 * rank, 2048, pfull_bar(ps));
                        bulk_load(dst + 2048, box + 4096 + 2048 * rank, 2048, pfull_bar(ps));
                        bulk_load(dst + 4096, box + 8192 + 512 * rank, 512, pfull_bar(ps));
                    }
                }
            }
            if (!ok)
                for (int q = 0; q < kPST; ++q)
                    if (issued[q] >= 0) mbar_wait_drain(pfull_bar(q), static_cast<uint32_t>(issued[q]));
        }
        __syncwarp();
    } else if (kQ4 && warp >= kPQConvWarp0) {
        // ------------------------------ converters (4-bit) ------------------------------
        // thread ct expands B row ct of this CTA's half of every stage; converter
        // warp 0 also loads the h rows of down tiles (after the m-block's gate/up
        // tiles have published), and on the leader posts the stage's expected bytes
        const int cw = warp - kPQConvWarp0;
        const int ct = cw * 32 + lane;
        int g = 0;
        bool ok = true;
        for (int it = 0, t; ok && (t = tile_of(pair, n_pairs, TA, TB, KBA, KBBs, it)) >= 0; ++it) {
            const bool gu = t < TA;
            const PairTile ti = decode_pair<kMFirst>(gu ? t : t - TA, table, seg.seg_count, gu ? NBA : NBBv,
                                            offs, 0, static_cast<int>(rank),
                                            kHalfTiles);
            const int num_kb = gu ? KBA : KBBs;
            const bool load_h = !gu && ti.rows > 0;
            const uint32_t tx = gu ? 0u : static_cast<uint32_t>(kPHalf * (1 + (ti.rows1 > 0 ? 1 : 0)));
            for (int kb = 0; kb < num_kb; ++kb, ++g) {
                const int s = g % kST;
                const uint32_t ph = static_cast<uint32_t>(g / kST) & 1u;
                const int ps = g % kPSTm;
                const uint32_t pph = static_cast<uint32_t>(g / kPSTm) & 1u;
                bool wt = true;
                if (lane == 0)
                    wt = mbar_wait(pfull_bar(ps), pph, abort_flag, a.dev_err) &&
                         mbar_wait_cl(empty_bar(s), ph ^ 1u, abort_flag, a.dev_err);
                if (cw == 0 && lane == 0 && wt && load_h && kb == 0) {
                    wt = wait_counter(a.done + seg.mblk[seg.seg_begin + ti.seg] + ti.cnt,
                                      ti.npub * done_target, abort_flag, a.dev_err);
                    fence_proxy_async_global();  // before the TMA reads of h
                }
                wt = __shfl_sync(0xffffffffu, wt, 0);
                if (!wt) {
                    ok = false;
                    break;
                }
                const uint32_t pb = sPk + ps * kPQBox;
                const uint32_t bb = sB + s * kPHalf;
                if (gu)
                    expand_row<false>(pb + ct * 16, pb + 2048 + ct * 16, pb + 4096 + ct * 4,
                                      bb + ct * kRowBytes, ct);
                else
                    expand_row<true>(pb + ct * 16, pb + 2048 + ct * 16, pb + 4096 + ct * 4,
                                     bb + ct * kRowBytes, ct);
                fence_proxy_async();
                __syncwarp();
                if (lane == 0) {
                    const uint32_t lbar = map_rank(full_bar(s), 0);
                    if (cw == 0) {
                        if (rank == 0) mbar_arrive_expect_tx(full_bar(s), tx);
                        if (load_h) tma_load_2d_pair(sA + s * kPHalf, &tm_h, kb * 64, ti.row0, lbar);
                    }
                    if (rank == 0)
                        mbar_arrive(full_bar(s));
                    else
                        mbar_arrive_remote_smem_release(lbar);
                    mbar_arrive(pempty_bar(ps));
                }
            }
        }
        if (!ok && cw == 0 && lane == 0) {
            // give an h load already issued time to land before the CTA goes away
            const uint64_t t0 = global_ns();
            while (global_ns() - t0 < kDrainLimitNs / 100) {
            }
        }
    } else if (warp == 0) {
        // ------------------------------ TMA producer ------------------------------
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int it = 0, t; ok && (t = tile_of(pair, n_pairs, TA, TB, KBA, KBBs, it)) >= 0; ++it) {
            const bool gu = t < TA;
            const PairTile ti = decode_pair<kMFirst>(gu ? t : t - TA, table, seg.seg_count, gu ? NBA : NBBv,
                                            offs, 0, static_cast<int>(rank),
                                            kHalfTiles);
            const int slot = seg.slot_base + ti.seg;
            const int num_kb = gu ? KBA : KBBs;
            // tile-major planes: the (n-block, k-block) box of a slot is one
            // contiguous run of 128 (gate, up) or 256 (down) rows of 128 bytes
            int brow0;
            const CUtensorMap* tm_b;
            const int kb0 = gu ? 0 : (ti.nb % KS) * KBBs;   // first k-block of the tile
            if (gu) {
                brow0 = (slot * NBA + ti.nb) * KBA * 128;
                tm_b = rank == 0 ? &tm_wg : &tm_wu;
            } else {
                brow0 = (slot * NBB + ti.nb / KS) * KBB * 256 + kBM * static_cast<int>(rank);
                tm_b = &tm_wd;
            }
            const int brow_step = gu ? 128 : 256;
            const bool load_h = !gu && ti.rows > 0;
            // a segment of one pair m-block is its weight tiles' only reader
            const bool only_reader = table[ti.seg + 1] - table[ti.seg] == 1;
            if (load_h) {
                // this half's h rows are complete once every epilogue warp of
                // every gate/up n-block of its m-block has published
                const int* cnt = a.done + seg.mblk[seg.seg_begin + ti.seg] + ti.cnt;
                const int target = ti.npub * done_target;
                bool w = true;
                if (lane == 0 && ld_acquire(cnt) < target) {
                    const uint64_t t0 = global_ns();
                    while (ld_acquire(cnt) < target) {
                        if (*abort_flag) {
                            w = false;
                            break;
                        }
                        if (global_ns() - t0 > kWaitLimitNs) {
                            *abort_flag = 1;
                            record_error(a.dev_err, kDevErrTimeout);
                            w = false;
                            break;
                        }
                    }
                }
                if (lane == 0) fence_proxy_async_global();  // before the TMA reads of h
                w = __shfl_sync(0xffffffffu, w, 0);
                if (!w) {
                    ok = false;
                    break;
                }
            }
            const uint32_t tx = 2 * kPHalf + (gu ? 0 : kPHalf * (1 + (ti.rows1 > 0 ? 1 : 0)));
            for (int kb = 0; kb < num_kb; ++kb) {
                bool w = true;
                if (lane == 0) w = mbar_wait_cl(empty_bar(stage), phase ^ 1u, abort_flag, a.dev_err);
                w = __shfl_sync(0xffffffffu, w, 0);
                if (!w) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    if (rank == 0) mbar_arrive_expect_tx(full_bar(stage), tx);
                    const uint32_t lbar = map_rank(full_bar(stage), 0);
                    if (gu && ti.half) {
                        // half tile: CTA r's B half = gate rows [64 r, 64 r + 64) of the
                        // n-block, then up rows [64 r, 64 r + 64) (8 KB each)
                        const int r64 = brow0 + kb * brow_step + 64 * static_cast<int>(rank);
                        const uint32_t dst = sB + stage * kPHalf;
                        if (only_reader) {
                            tma_load_2d_pair_hint(dst, &tm_wg64, 0, r64, lbar, policy_evict_first());
                            tma_load_2d_pair_hint(dst + kPHalf / 2, &tm_wu64, 0, r64, lbar,
                                                  policy_evict_first());
                        } else {
                            tma_load_2d_pair(dst, &tm_wg64, 0, r64, lbar);
                            tma_load_2d_pair(dst + kPHalf / 2, &tm_wu64, 0, r64, lbar);
                        }
                    } else if (only_reader)
                        tma_load_2d_pair_hint(sB + stage * kPHalf, tm_b, 0,
                                              brow0 + (kb0 + kb) * brow_step, lbar,
                                              policy_evict_first());
                    else
                        tma_load_2d_pair(sB + stage * kPHalf, tm_b, 0, brow0 + (kb0 + kb) * brow_step,
                                         lbar);
                    if (load_h)
                        tma_load_2d_pair(sA + stage * kPHalf, &tm_h, (kb0 + kb) * 64, ti.row0, lbar);
                }
                __syncwarp();
                if (++stage == kST) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (!ok && lane == 0) {
            // give copies already issued time to land before the CTA goes away
            const uint64_t t0 = global_ns();
            while (global_ns() - t0 < kDrainLimitNs / 100) {
            }
        }
    } else if (warp >= kLoaderWarp0 && warp < kLoaderWarp0 + kLoaderWarps) {
        // ------------------------------ A-operand loader ------------------------------
        // As in the single-CTA kernel, but each warp arrives once per stage
        // (after every lane's copies completed and were fenced) on the
        // leader's full barrier: a local arrival in the leader, a restricted
        // shared-memory release and a relaxed remote arrival in the peer.
        const int gw = warp - kLoaderWarp0;
        const uint32_t chunk = static_cast<uint32_t>(lane & 7);
        int stage = 0;
        uint32_t phase = 0;
        int pend[kLoaderDepth + 1];
        int npend = 0;
        bool ok = true;
        auto publish = [&](int s) {
            __syncwarp();
            if (lane == 0) {
                if (rank == 0)
                    mbar_arrive(full_bar(s));
                else
                    mbar_arrive_remote_smem_release(map_rank(full_bar(s), 0));
            }
        };
        for (int it = 0, t; ok && (t = tile_of(pair, n_pairs, TA, TB, KBA, KBBs, it)) >= 0; ++it) {
            const bool gu = t < TA;
            const PairTile ti = decode_pair<kMFirst>(gu ? t : t - TA, table, seg.seg_count, gu ? NBA : NBBv,
                                            offs, 0, static_cast<int>(rank),
                                            kHalfTiles);
            const int num_kb = gu ? KBA : KBBs;
            if (!gu) {
                if (npend > 0) {
                    cp_async_wait<0>();
                    fence_proxy_async();
                    for (int q = 0; q < npend; ++q) publish(pend[q]);
                    npend = 0;
                }
                for (int kb = 0; kb < num_kb; ++kb) {
                    bool w = true;
                    if (lane == 0) w = mbar_wait_cl(empty_bar(stage), phase ^ 1u, abort_flag, a.dev_err);
                    w = __shfl_sync(0xffffffffu, w, 0);
                    if (!w) {
                        ok = false;
                        break;
                    }
                    publish(stage);
                    if (++stage == kST) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                continue;
            }
            const uint8_t* src_row[8];
            uint32_t dst_off[8];
            unsigned live = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int r = gw * 32 + 4 * i + (lane >> 3);
                dst_off[i] = static_cast<uint32_t>(r) * kRowBytes +
                             ((chunk ^ static_cast<uint32_t>(r & 7)) << 4);
                const bool lv = r < ti.rows;
                live |= lv ? (1u << i) : 0u;
                const uint8_t* row = reinterpret_cast<const uint8_t*>(a.x);
                if (lv)
                    row = reinterpret_cast<const uint8_t*>(
                        a.x + static_cast<size_t>(seg.rec_tok[ti.row0 + r]) * H);
                src_row[i] = row + chunk * 16;
            }
            for (int kb = 0; kb < num_kb; ++kb) {
                bool w = true;
                if (lane == 0) w = mbar_wait_cl(empty_bar(stage), phase ^ 1u, abort_flag, a.dev_err);
                w = __shfl_sync(0xffffffffu, w, 0);
                if (!w) {
                    ok = false;
                    break;
                }
                const uint32_t base = sA + stage * kPHalf;
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (live & (1u << i)) cp_async_16(base + dst_off[i], src_row[i] + kb * kRowBytes);
                cp_async_commit();
                pend[npend++] = stage;
                if (npend > kLoaderDepth) {
                    cp_async_wait<kLoaderDepth>();
                    fence_proxy_async();
                    publish(pend[0]);
#pragma unroll
                    for (int q = 0; q < kLoaderDepth; ++q) pend[q] = pend[q + 1];
                    --npend;
                }
                if (++stage == kST) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        cp_async_wait<0>();
        fence_proxy_async();
        for (int q = 0; q < npend; ++q) publish(pend[q]);
    } else if (warp == 1) {
        // ------------------------------ MMA issuer (leader CTA) ------------------------------
        if (lane == 0 && rank == 0) {
            const uint32_t idesc_gu = make_idesc(true, kPairRows, 256);   // bf16 x bf16
            const uint32_t idesc_dn = make_idesc(false, kPairRows, 256);  // fp16 x fp16
            const uint32_t idesc_gu_half = make_idesc(true, kBM, 256);    // half tiles: M = 128
            const uint32_t idesc_dn_half = make_idesc(false, kBM, 256);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            bool issued_any = false;
            for (int it = 0, t; ok && (t = tile_of(pair, n_pairs, TA, TB, KBA, KBBs, it)) >= 0; ++it) {
                const bool gu = t < TA;
                const int num_kb = gu ? KBA : KBBs;
                const PairTile ti = decode_pair<kMFirst>(gu ? t : t - TA, table, seg.seg_count, gu ? NBA : NBBv,
                                                offs, 0, 0, kHalfTiles);
                const uint32_t idesc = gu ? (ti.half ? idesc_gu_half : idesc_gu)
                                          : (ti.half ? idesc_dn_half : idesc_dn);
                if (!mbar_wait_cl(acce_bar(acc), acc_phase ^ 1u, abort_flag, a.dev_err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kAccCols);
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait_cl(full_bar(stage), phase, abort_flag, a.dev_err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t adesc = sw128_desc(sA + stage * kPHalf);
                    const uint64_t bdesc = sw128_desc(sB + stage * kPHalf);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_f16_pair(d_tmem, adesc + 2u * kk, bdesc + 2u * kk, idesc,
                                      (kb | kk) != 0 ? 1u : 0u);
                    issued_any = true;
                    umma_commit_pair(empty_bar(stage));
                    if (++stage == kST) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit_pair(accf_bar(acc));
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
            if (!ok && issued_any) {
                umma_commit_pair(drain_bar);
                mbar_wait_cl_drain(drain_bar, 0);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------ epilogue (warps 2-5) ------------------------------
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t stg = sbase + kL.off_stg + static_cast<uint32_t>(quarter * kStageWarpBytes);
        const uint32_t leader_acce0 = map_rank(acce_bar(0), 0);
        const uint32_t leader_acce1 = map_rank(acce_bar(1), 0);
        const int n_epi = static_cast<int>(gridDim.x) * kEpiWarps;   // epilogue warps of the launch
        if (seg.resid_A)
            residual_rows(seg, a.H, static_cast<int>(blockIdx.x) * kEpiWarps + warp - 2, n_epi, lane);
        // the deterministic mode adds into Y only in the combine, a later launch
        bool resid_ok = !seg.resid_A || a.out_rows;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int it = 0, t; (t = tile_of(pair, n_pairs, TA, TB, KBA, KBBs, it)) >= 0; ++it) {
            const bool gu = t < TA;
            if (!gu && !resid_ok) {
                if (!residual_ready(seg, n_epi, lane, abort_flag, a.dev_err)) break;
                resid_ok = true;
            }
            const PairTile ti = decode_pair<kMFirst>(gu ? t : t - TA, table, seg.seg_count, gu ? NBA : NBBv,
                                            offs, 0, static_cast<int>(rank),
                                            kHalfTiles);
            bool w = true;
            if (lane == 0) w = mbar_wait_cl(accf_bar(acc), acc_phase, abort_flag, a.dev_err);
            w = __shfl_sync(0xffffffffu, w, 0);
            if (!w) break;
            tc_fence_after();
            // A half tile's 64 rows per CTA fill TMEM lanes 0-63 with accumulator
            // columns 0-127 and lanes 64-127 with columns 128-255 of the same
            // rows: quarters q and q + 2 hold one row range, different columns.
            const int trow = ti.half ? (quarter & 1) * 32 + lane : row;
            const int cpart = ti.half ? quarter >> 1 : 0;   // column half of a half tile
            const bool valid = trow < ti.rows;
            const int p = ti.row0 + trow;
            const uint32_t tacc = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                  static_cast<uint32_t>(acc * kAccCols);
            if (gu) {
                // half tiles: the B half of each CTA is 64 gate rows then 64 up
                // rows, so a lane holds g in columns 0-63 and u in 64-127 of h
                // columns 64 cpart .. 64 cpart + 63 of the n-block
                __half* dst = a.h + static_cast<size_t>(p) * F + static_cast<size_t>(ti.nb) * 128 +
                              64 * cpart;
                if (ti.half)
                    epilogue_gate_up_staged(tacc, valid ? dst : nullptr, stg, lane, a.dev_err, 1, 64);
                else
                    epilogue_gate_up_staged(tacc, valid ? dst : nullptr, stg, lane, a.dev_err);
                fence_proxy_async_global();
                __threadfence();
                __syncwarp();
                if (lane == 0 && (a.phases & 2) && ti.rows > 0)
                    red_release_add(a.done + seg.mblk[seg.seg_begin + ti.seg] + ti.cnt, 1);
            } else {
                float al = 0.0f;
                int tok = 0;
                if (valid) {
                    tok = seg.rec_tok[p];
                    al = seg.alpha ? seg.alpha[seg.rec_route[p]] : 1.0f;
                    al *= seg.seg_scale[seg.seg_begin + ti.seg];
                }
                float* dst = a.out_rows ? a.out_rows + static_cast<size_t>(p) * H
                                        : a.Y + static_cast<size_t>(tok) * H;
                epilogue_down_staged(tacc, al, valid ? dst + (ti.nb / KS) * 256 + 128 * cpart : nullptr,
                                     !a.out_rows, stg, lane, ti.half ? 4 : 8);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (rank == 0)
                    mbar_arrive(acce_bar(acc));
                else
                    mbar_arrive_cl(acc == 0 ? leader_acce0 : leader_acce1);
            }
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();  // the peer's shared memory and TMEM stay until the pair is done
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, kTmemCols);
    }
}

// Deterministic combine: one thread per 4 columns of one token.
__global__ void k_combine(const float* __restrict__ rows, const int32_t* __restrict__ pos, int T,
                          int k, int H, const float* __restrict__ shared_rows, int n_shared,
                          float* __restrict__ Y) {
    const int H4 = H / 4;
    const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= static_cast<long long>(T) * H4) return;
    const int t = static_cast<int>(idx / H4);
    const int c = static_cast<int>(idx % H4) * 4;
    float4 y = *reinterpret_cast<const float4*>(Y + static_cast<size_t>(t) * H + c);
    for (int j = 0; j < k; ++j) {
        const int p = pos[t * k + j];
        if (p < 0 || p >= T * k) continue;  // not placed (a route build that gave up)
        const float4 v = *reinterpret_cast<const float4*>(rows + static_cast<size_t>(p) * H + c);
        y.x += v.x; y.y += v.y; y.z += v.z; y.w += v.w;
    }
    for (int s = 0; s < n_shared; ++s) {
        const float4 v = *reinterpret_cast<const float4*>(
            shared_rows + (static_cast<size_t>(s) * T + t) * H + c);
        y.x += v.x; y.y += v.y; y.z += v.z; y.w += v.w;
    }
    *reinterpret_cast<float4*>(Y + static_cast<size_t>(t) * H + c) = y;
}

}  // namespace

cudaError_t launch_expert_ffn(const CUtensorMap* tm_wg, const CUtensorMap* tm_wu,
                              const CUtensorMap* tm_wd, const CUtensorMap* tm_h,
                              const GemmSegments& seg, const void* X,
                              void* h, float* Y, float* out_rows, int* done, int* ticket, int H,
                              int F, int phases, int* dev_err, int num_sms, cudaStream_t stream) {
    const long long max_tiles = static_cast<long long>(seg.max_tiles_m) *
                                (((phases & 1) ? F / 128 : 0) + ((phases & 2) ? H / 256 : 0));
    if (max_tiles <= 0 || seg.seg_count <= 0) return cudaSuccess;
    const int grid = static_cast<int>(max_tiles < num_sms ? max_tiles : num_sms);
    const size_t smem = gemm_smem_bytes(seg.seg_count);
    cudaError_t rc = cudaFuncSetAttribute(k_expert_ffn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          static_cast<int>(smem));
    if (rc != cudaSuccess) return rc;
    FfnArgs args;
    args.seg = seg;
    args.x = static_cast<const __nv_bfloat16*>(X);
    args.h = static_cast<__half*>(h);
    args.Y = Y;
    args.out_rows = out_rows;
    args.done = done;
    args.ticket = ticket;
    args.dev_err = dev_err;
    args.H = H;
    args.F = F;
    args.phases = phases;
    void* kargs[] = {const_cast<CUtensorMap*>(tm_wg), const_cast<CUtensorMap*>(tm_wu),
                     const_cast<CUtensorMap*>(tm_wd), const_cast<CUtensorMap*>(tm_h), &args};
    // cooperative: every CTA is resident, so a down tile may wait for the
    // gate/up tiles of its m-block that other CTAs own
    rc = cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(k_expert_ffn), grid, kThreads,
                                     kargs, smem, stream);
    if (rc != cudaSuccess) return rc;
    return cudaGetLastError();
}

// Co-resident CTA pairs of a pair kernel form at its largest shared-memory
// size (the bound for every smaller launch), per device and form.
template <bool kQ4, bool kMFirst>
static int max_pairs(int device) {
    static std::mutex mu;
    static int cache[64] = {0};
    if (device < 0 || device >= 64) return 0;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[device] > 0) return cache[device];
    // the largest segment count a launch of this form takes: slots of an arena,
    // or the experts of one layer for 4-bit weights
    const size_t smem = pair_smem_bytes(pair_seg_cap(kQ4), kQ4);
    if (cudaFuncSetAttribute(k_expert_ffn_pair<kQ4, kMFirst>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    int nsm = 0;
    cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, device);
    cfg.gridDim = dim3(static_cast<unsigned>(nsm & ~1));
    cfg.blockDim = dim3(kQ4 ? kPQThreads : kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void*>(k_expert_ffn_pair<kQ4, kMFirst>),
                                       &cfg) != cudaSuccess)
        return 0;
    cache[device] = n;
    return n;
}

// One cooperative launch of clusters of two CTAs: every pair is resident, so
// a down tile may wait for gate/up tiles that other pairs own.
template <bool kQ4, bool kMFirst>
static cudaError_t launch_pair(const CUtensorMap* tm_wg, const CUtensorMap* tm_wu,
                               const CUtensorMap* tm_wd_half, const CUtensorMap* tm_h,
                               const CUtensorMap* tm_wg64, const CUtensorMap* tm_wu64,
                               const Q4Planes& planes, const GemmSegments& seg, const void* X,
                               void* h, float* Y, float* out_rows, int* done, int H, int F,
                               int phases, int* dev_err, cudaStream_t stream) {
    const long long max_tiles = static_cast<long long>(seg.max_tiles_m) *
                                (((phases & 1) ? F / 128 : 0) + ((phases & 2) ? H / 256 : 0));
    if (max_tiles <= 0 || seg.seg_count <= 0) return cudaSuccess;
    int device = 0;
    cudaError_t rc = cudaGetDevice(&device);
    if (rc != cudaSuccess) return rc;
    const int cap = max_pairs<kQ4, kMFirst>(device);
    if (cap <= 0) return cudaErrorLaunchOutOfResources;
    const int pairs = static_cast<int>(max_tiles < cap ? max_tiles : cap);
    const size_t smem = pair_smem_bytes(seg.seg_count, kQ4);
    rc = cudaFuncSetAttribute(k_expert_ffn_pair<kQ4, kMFirst>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(smem));
    if (rc != cudaSuccess) return rc;
    FfnArgs args;
    args.seg = seg;
    args.x = static_cast<const __nv_bfloat16*>(X);
    args.h = static_cast<__half*>(h);
    args.Y = Y;
    args.out_rows = out_rows;
    args.done = done;
    args.ticket = nullptr;
    args.dev_err = dev_err;
    args.H = H;
    args.F = F;
    args.phases = phases;
    Q4Planes pl = planes;
    void* kargs[] = {const_cast<CUtensorMap*>(tm_wg), const_cast<CUtensorMap*>(tm_wu),
                     const_cast<CUtensorMap*>(tm_wd_half), const_cast<CUtensorMap*>(tm_h),
                     const_cast<CUtensorMap*>(tm_wg64), const_cast<CUtensorMap*>(tm_wu64), &pl,
                     &args};
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeCooperative;
    at[1].val.cooperative = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs));
    cfg.blockDim = dim3(kQ4 ? kPQThreads : kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    rc = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(k_expert_ffn_pair<kQ4, kMFirst>), kargs);
    if (rc != cudaSuccess) return rc;
    return cudaGetLastError();
}

cudaError_t launch_expert_ffn_pair(const CUtensorMap* tm_wg, const CUtensorMap* tm_wu,
                                   const CUtensorMap* tm_wd_half, const CUtensorMap* tm_h,
                                   const CUtensorMap* tm_wg64, const CUtensorMap* tm_wu64,
                                   const GemmSegments& seg, const void* X, void* h, float* Y,
                                   float* out_rows, int* done, int H, int F, int phases,
                                   int* dev_err, bool m_first, cudaStream_t stream) {
    const Q4Planes none{nullptr, nullptr, nullptr, 0, 0};
    if (m_first)
        return launch_pair<false, true>(tm_wg, tm_wu, tm_wd_half, tm_h, tm_wg64, tm_wu64, none, seg,
                                        X, h, Y, out_rows, done, H, F, phases, dev_err, stream);
    return launch_pair<false, false>(tm_wg, tm_wu, tm_wd_half, tm_h, tm_wg64, tm_wu64, none, seg, X,
                                     h, Y, out_rows, done, H, F, phases, dev_err, stream);
}

cudaError_t launch_expert_ffn_pair_q4(const uint8_t* plane_g, const uint8_t* plane_u,
                                      const uint8_t* plane_d, size_t S_gu, size_t S_d,
                                      const CUtensorMap* tm_h, const GemmSegments& seg,
                                      const void* X, void* h, float* Y, float* out_rows, int* done,
                                      int H, int F, int phases, int* dev_err, cudaStream_t stream) {
    if (seg.seg_count > kQMaxSegs) return cudaErrorInvalidValue;
    const Q4Planes planes{plane_g, plane_u, plane_d, S_gu, S_d};
    // the weight maps are not read by the 4-bit form; h's map stands in for them
    return launch_pair<true, false>(tm_h, tm_h, tm_h, tm_h, tm_h, tm_h, planes, seg, X, h, Y,
                                    out_rows, done, H, F, phases, dev_err, stream);
}

cudaError_t launch_expert_ffn_q4(const uint8_t* plane_g, const uint8_t* plane_u, const uint8_t* plane_d,
                                 size_t S_gu, size_t S_d, const CUtensorMap* tm_h,
                                 const GemmSegments& seg, const void* X, void* h, float* Y,
                                 float* out_rows, int* done, int* ticket, int H, int F, int phases,
                                 int* dev_err, int num_sms, cudaStream_t stream) {
    const long long max_tiles = static_cast<long long>(seg.max_tiles_m) *
                                (((phases & 1) ? F / 128 : 0) + ((phases & 2) ? H / 256 : 0));
    if (max_tiles <= 0 || seg.seg_count <= 0) return cudaSuccess;
    if (seg.seg_count > kQMaxSegs) return cudaErrorInvalidValue;
    const int grid = static_cast<int>(max_tiles < num_sms ? max_tiles : num_sms);
    const size_t smem = q4_smem_bytes(seg.seg_count);
    cudaError_t rc = cudaFuncSetAttribute(k_expert_ffn_q4, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          static_cast<int>(smem));
    if (rc != cudaSuccess) return rc;
    Q4Planes planes{plane_g, plane_u, plane_d, S_gu, S_d};
    FfnArgs args;
    args.seg = seg;
    args.x = static_cast<const __nv_bfloat16*>(X);
    args.h = static_cast<__half*>(h);
    args.Y = Y;
    args.out_rows = out_rows;
    args.done = done;
    args.ticket = ticket;
    args.dev_err = dev_err;
    args.H = H;
    args.F = F;
    args.phases = phases;
    void* kargs[] = {const_cast<CUtensorMap*>(tm_h), &planes, &args};
    // cooperative: every CTA is resident, so a down tile may wait for the
    // gate/up tiles of its m-block that other CTAs own
    rc = cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(k_expert_ffn_q4), grid, kQThreads,
                                     kargs, smem, stream);
    if (rc != cudaSuccess) return rc;
    return cudaGetLastError();
}

cudaError_t launch_combine(const float* rows, const int32_t* pos, int T, int k, int H,
                           const float* shared_rows, int n_shared, float* Y, cudaStream_t stream) {
    const long long n = static_cast<long long>(T) * (H / 4);
    if (n == 0) return cudaSuccess;
    k_combine<<<static_cast<unsigned>((n + 255) / 256), 256, 0, stream>>>(rows, pos, T, k, H,
                                                                          shared_rows, n_shared, Y);
    return cudaGetLastError();
}

// ----------------------------------------------------------------------------
// Tensor maps
// ----------------------------------------------------------------------------
namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}
}  // namespace

CUresult encode_tmap_2d(CUtensorMap* tm, CUtensorMapDataType dtype, const void* base, uint64_t inner,
                        uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner,
                        uint32_t box_outer) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return CUDA_ERROR_NOT_FOUND;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_stride_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return fn(tm, dtype, 2,
              const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace es
