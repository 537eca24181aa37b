// One CTA's share of a router-logits tile on the tensor cores, shared by the
// standalone router kernel (router.cu) and the fused router + route-build
// kernel (route.cu): tokens [m0, m0+128) x experts [n0, n0+N) over k-blocks
// [kb0, kb1) of 64 hidden elements, bf16 operands TMA-loaded with the 128-byte
// swizzle through a kRStages ring, tcgen05.mma.kind::f16 into an fp32 TMEM
// accumulator, and the partial sums written to `part` in shared memory as
// rows of N + 1 floats (token r at part[r * (N + 1)], padded against bank
// conflicts). Warp roles: warp 0 TMA producer, warp 1 MMA issue, warps 2-5
// TMEM read-out (TMEM lanes = tokens); other warps return at once. Every wait
// is bounded; after an abort the MMAs already issued still complete before
// the caller frees TMEM, and the partial is left unwritten (the abort flag
// tells the caller).
// Included inside `namespace es { namespace { ... } }` after tc_ptx.cuh.
#pragma once

constexpr int kRStages = 4;
constexpr int kRTileA = 128 * 128;  // 128 tokens x 64 bf16
constexpr int kRMaxSplit = 8;       // portable cluster size

// Shared memory of the stage ring for N experts per tile (the partial sums
// reuse it once every MMA has completed).
__host__ __device__ constexpr size_t router_ring_bytes(int N) {
    return static_cast<size_t>(kRStages) * (kRTileA + static_cast<size_t>(N) * 128);
}
__host__ __device__ constexpr size_t router_part_bytes(int N) {
    return static_cast<size_t>(128) * (N + 1) * sizeof(float);
}
// TMEM columns of an N-wide fp32 accumulator (a power of two >= 32).
__host__ __device__ constexpr uint32_t router_tmem_cols(int N) {
    return N <= 32 ? 32u : (N <= 64 ? 64u : (N <= 128 ? 128u : 256u));
}

struct RouterTile {
    uint32_t sA, sB;        // stage ring: kRStages A tiles, then kRStages B tiles (N x 128 B)
    uint32_t bar0;          // full[kRStages], empty[kRStages], acc: 2 kRStages + 1 barriers
    float* part;            // partial sums (overlaps the ring)
    int m0, n0, kb0, kb1, N;
    uint32_t tx_bytes;      // bytes one stage's two boxes deliver
};

// Barrier initialisation, one thread (before the CTA's first __syncthreads).
__device__ __forceinline__ void router_tile_init(const RouterTile& rt) {
    for (int q = 0; q < kRStages; ++q) {
        mbar_init(rt.bar0 + 8u * q, 1);
        mbar_init(rt.bar0 + 8u * (kRStages + q), 1);
    }
    mbar_init(rt.bar0 + 8u * (2 * kRStages), 1);
}

// The roles of warps 0-5 over the tile (see the file comment).
__device__ void router_tile_roles(const RouterTile& rt, const CUtensorMap* tm_x,
                                  const CUtensorMap* tm_w, uint32_t tmem_base,
                                  volatile int* abort_flag, int* dev_err) {
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int tileB = rt.N * 128;
    auto full_bar = [&](int s) { return rt.bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return rt.bar0 + 8u * (kRStages + s); };
    const uint32_t acc_bar = rt.bar0 + 8u * (2 * kRStages);
    if (warp == 0) {
        if (lane == 0) {
            int issued[kRStages];
            for (int q = 0; q < kRStages; ++q) issued[q] = -1;
            bool ok = true;
            for (int kb = rt.kb0, i = 0; kb < rt.kb1; ++kb, ++i) {
                const int st = i % kRStages;
                const uint32_t ph = static_cast<uint32_t>(i / kRStages) & 1u;
                if (!mbar_wait(empty_bar(st), ph ^ 1u, abort_flag, dev_err)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(full_bar(st), rt.tx_bytes);
                issued[st] = static_cast<int>(ph);
                tma_load_2d(rt.sA + st * kRTileA, tm_x, kb * 64, rt.m0, full_bar(st));
                tma_load_2d(rt.sB + st * tileB, tm_w, kb * 64, rt.n0, full_bar(st));
            }
            if (!ok)
                for (int q = 0; q < kRStages; ++q)
                    if (issued[q] >= 0)
                        mbar_wait_drain(full_bar(q), static_cast<uint32_t>(issued[q]));
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = make_idesc(true, 128, rt.N);
            bool any = false;
            for (int kb = rt.kb0, i = 0; kb < rt.kb1; ++kb, ++i) {
                const int st = i % kRStages;
                const uint32_t ph = static_cast<uint32_t>(i / kRStages) & 1u;
                if (!mbar_wait(full_bar(st), ph, abort_flag, dev_err)) break;
                tc_fence_after();
                const uint64_t adesc = sw128_desc(rt.sA + st * kRTileA);
                const uint64_t bdesc = sw128_desc(rt.sB + st * tileB);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    umma_f16(tmem_base, adesc + 2u * kk, bdesc + 2u * kk, idesc, (i | kk) != 0 ? 1u : 0u);
                any = true;
                umma_commit(empty_bar(st));
            }
            // the accumulator barrier completes once every MMA issued so far
            // has finished (also after an abort, so TMEM can be freed)
            if (any) umma_commit(acc_bar);
            else mbar_arrive(acc_bar);
        }
        __syncwarp();
    } else if (warp < 6) {
        // the tile's partial sums into shared memory (the stage buffers are
        // free once every MMA has completed)
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        bool w = true;
        if (lane == 0) {
            w = mbar_wait(acc_bar, 0, abort_flag, dev_err);
            // after an abort the MMAs already issued still complete (the MMA
            // thread always commits this barrier) before TMEM is freed
            if (!w) mbar_wait_drain(acc_bar, 0);
        }
        w = __shfl_sync(0xffffffffu, w, 0);
        tc_fence_after();
        if (w && !*abort_flag) {
            float* part = rt.part + row * (rt.N + 1);
            for (int c0 = 0; c0 < rt.N; c0 += 32) {
                uint32_t v[32];
                tmem_ld32(tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + c0, v);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (c0 + j < rt.N) part[c0 + j] = __uint_as_float(v[j]);
            }
        }
    }
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t local_addr, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}
// Sum of the S partials of one logit (partial element at shared offset `off`
// in every CTA of the cluster), loaded together, then added in ascending
// chunk order -- the same order whichever CTA sums it.
__device__ __forceinline__ float sum_cluster_partials(uint32_t off, int S) {
    float v[kRMaxSplit];
#pragma unroll
    for (int q = 0; q < kRMaxSplit; ++q)
        if (q < S) v[q] = ld_cluster_f32(off, static_cast<uint32_t>(q));
    float acc = v[0];
#pragma unroll
    for (int q = 1; q < kRMaxSplit; ++q)
        if (q < S) acc += v[q];
    return acc;
}
