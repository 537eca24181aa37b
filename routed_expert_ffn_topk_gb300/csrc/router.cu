// Router logits upstream of the top-k: l[t][e] = sum_h X[t][h] * W_r[e][h].
//
// "EStream: Fast and Memory-Efficient MoE Prefill through Expert
// Virtualization on Mobile NPUs", section 1 (a router assigns each token to
// the top-k of E experts) and section 4 (routing is one of the operators run
// on the accelerator, on the layer input). The form of the router is not on
// the pages; this is the bias-free linear router of top-k MoE layers.
//
// GB300 form. The contraction is [T, H] x [H, E] with E small (8..1024), so
// one 128-token tile per CTA would leave most SMs idle. The K range is split
// into S <= 8 chunks so that about one wave of CTAs covers the GPU: CTA
// (m, n, s) multiplies tokens [128m, 128m+128) by experts [N n, N n + N)
// over its k-blocks with tcgen05.mma.kind::f16 (bf16, fp32 accumulate in
// TMEM), both operands TMA-loaded with 128-byte swizzle through a 4-stage
// ring. The S CTAs of a tile form one thread-block cluster: each stages its
// fp32 partial in its own shared memory, and after a cluster barrier CTA s
// adds, for its slice of the tile's rows, the S partials read through
// distributed shared memory in ascending chunk order -- one kernel, no
// partial sums in HBM, and logits that do not depend on timing.
// Warp roles: warp 0 TMA producer, warp 1 TMEM allocation and the MMA issue,
// warps 2-5 epilogue (TMEM lanes = tokens). Every wait is bounded.
#include <cuda.h>
#include <cuda_bf16.h>

#include "estream_internal.h"

namespace es {
namespace {

#include "tc_ptx.cuh"

#include "router_tile.cuh"

constexpr int kRThreads = 192;

struct RouterArgs {
    float* logits;      // [T][E]
    int* dev_err;       // optional
    int T, E, KB, S, N;
    uint32_t tx_bytes;  // bytes one stage's two boxes deliver
};

size_t router_smem_bytes(int N) {
    return 1024 + router_ring_bytes(N) + 8 * (2 * kRStages + 1) + 16;
}

__global__ void __launch_bounds__(kRThreads, 1)
    k_router_partial(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                     const RouterArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    // the fixed-order sum reads the partials of a.S CTAs of one cluster: a
    // launch without that cluster shape returns before any cluster access
    if (cluster_num_ctas() != static_cast<uint32_t>(a.S)) {
        if (threadIdx.x == 0 && a.dev_err) atomicCAS(a.dev_err, kDevErrNone, kDevErrLaunch);
        return;
    }
    const int N = a.N;
    const uint32_t sbase = smem_addr(smem);
    RouterTile rt;
    rt.sA = sbase;
    rt.sB = sbase + kRStages * kRTileA;
    rt.bar0 = sbase + static_cast<uint32_t>(router_ring_bytes(N));
    rt.part = reinterpret_cast<float*>(smem);
    rt.m0 = blockIdx.x * 128;
    rt.n0 = blockIdx.y * N;
    rt.N = N;
    rt.tx_bytes = a.tx_bytes;
    const int s = blockIdx.z;
    rt.kb0 = static_cast<int>(static_cast<long long>(s) * a.KB / a.S);
    rt.kb1 = static_cast<int>(static_cast<long long>(s + 1) * a.KB / a.S);
    uint8_t* misc = smem + router_ring_bytes(N) + 8 * (2 * kRStages + 1);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 4);
    const int warp = threadIdx.x >> 5;
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
    router_tile_roles(rt, &tm_x, &tm_w, tmem_base, abort_flag, a.dev_err);
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // every chunk's partial is in place
    {
        // CTA s of the cluster sums rows [r0, r1) of the tile over the chunks
        const int rows_per = (128 + a.S - 1) / a.S;
        const int r0 = s * rows_per;
        const int r1 = min(128, r0 + rows_per);
        const bool ok = !*abort_flag;
        for (int i = threadIdx.x; ok && i < (r1 - r0) * N; i += kRThreads) {
            const int r = r0 + i / N, c = i % N;
            const int t = rt.m0 + r, e = rt.n0 + c;
            if (t >= a.T || e >= a.E) continue;
            const uint32_t off = sbase + static_cast<uint32_t>((r * (N + 1) + c) * 4);
            a.logits[static_cast<size_t>(t) * a.E + e] = sum_cluster_partials(off, a.S);
        }
    }
    cluster_sync_all();  // no CTA leaves while its partial may still be read
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, tmem_cols);
    }
}

}  // namespace

RouterPlan router_plan(int T, int H, int E, int num_sms) {
    RouterPlan p{};
    p.N = E >= 256 ? 256 : ((E + 15) / 16) * 16;
    p.m_tiles = (T + 127) / 128;
    p.n_tiles = (E + p.N - 1) / p.N;
    p.KB = H / 64;
    // enough K chunks to fill about one wave, but at least four k-blocks per
    // chunk (a CTA's fixed cost -- barriers, TMEM, the first TMA round trip --
    // is that of a few k-blocks, and every chunk adds a partial to the sum)
    const long long tiles = static_cast<long long>(p.m_tiles) * p.n_tiles;
    long long S = tiles > 0 ? (num_sms + tiles - 1) / tiles : 1;
    if (S > p.KB / 4) S = p.KB / 4;
    if (S > kRMaxSplit) S = kRMaxSplit;
    if (S < 1) S = 1;
    p.S = static_cast<int>(S);
    p.partial_bytes = 0;  // partial sums stay in shared memory
    return p;
}

cudaError_t launch_router_logits(const void* X, int T, int H, const void* W_r, int E, float* logits,
                                 const RouterPlan& p, int* dev_err, cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    // boxes no taller than the tensors; the MMA still reads 128 x N rows, the
    // rows past T or E hold stale data whose results are never stored
    CUtensorMap tm_x, tm_w;
    const CUtensorMapDataType BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const uint32_t box_x = static_cast<uint32_t>(T < 128 ? T : 128);
    const uint32_t box_w = static_cast<uint32_t>(E < p.N ? E : p.N);
    if (encode_tmap_2d(&tm_x, BF, X, static_cast<uint64_t>(H), static_cast<uint64_t>(T),
                       static_cast<uint64_t>(H) * 2, 64, box_x) != CUDA_SUCCESS ||
        encode_tmap_2d(&tm_w, BF, W_r, static_cast<uint64_t>(H), static_cast<uint64_t>(E),
                       static_cast<uint64_t>(H) * 2, 64, box_w) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    const size_t smem = router_smem_bytes(p.N);
    cudaError_t rc = cudaFuncSetAttribute(k_router_partial, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          static_cast<int>(smem));
    if (rc != cudaSuccess) return rc;
    RouterArgs args;
    args.logits = logits;
    args.dev_err = dev_err;
    args.T = T;
    args.E = E;
    args.KB = p.KB;
    args.S = p.S;
    args.N = p.N;
    args.tx_bytes = (box_x + box_w) * 128u;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 1;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = static_cast<unsigned>(p.S);
    cfg.gridDim = dim3(static_cast<unsigned>(p.m_tiles), static_cast<unsigned>(p.n_tiles),
                       static_cast<unsigned>(p.S));
    cfg.blockDim = dim3(kRThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    void* kargs[] = {&tm_x, &tm_w, &args};
    rc = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(k_router_partial), kargs);
    if (rc != cudaSuccess) return rc;
    return cudaGetLastError();
}

}  // namespace es

// ----------------------------------------------------------------------------
// C ABI
// ----------------------------------------------------------------------------
namespace {

constexpr size_t kRouterErrBytes = 256;  // the error word

int router_current_sms() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

bool router_shape_ok(int T, int H, int E) {
    return T >= 0 && H >= 64 && H % 64 == 0 && E >= 1 && E <= es::kMaxE;
}

bool router_aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" size_t estream_router_workspace_bytes(int T, int H, int E) {
    if (!router_shape_ok(T, H, E)) return 0;
    const int sms = router_current_sms();
    if (sms <= 0) return 0;
    return kRouterErrBytes + es::router_plan(T, H, E, sms).partial_bytes;
}

extern "C" estream_status estream_router_logits(const void* X, int T, int H, const void* W_r, int E,
                                                float* logits, void* workspace,
                                                size_t workspace_bytes, void* cuda_stream) {
    if (!router_shape_ok(T, H, E) || !workspace || !router_aligned(workspace, 256))
        return ESTREAM_ERR_INVALID_ARG;
    if (T > 0 && (!X || !W_r || !logits || !router_aligned(X, 16) || !router_aligned(W_r, 16) ||
                  !router_aligned(logits, 4)))
        return ESTREAM_ERR_INVALID_ARG;
    int dev = 0, major = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess)
        return ESTREAM_ERR_CUDA;
    if (major != 10) return ESTREAM_ERR_UNSUPPORTED;
    const int sms = router_current_sms();
    if (sms <= 0) return ESTREAM_ERR_CUDA;
    const es::RouterPlan plan = es::router_plan(T, H, E, sms);
    if (workspace_bytes < kRouterErrBytes + plan.partial_bytes) return ESTREAM_ERR_CAPACITY;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    char* ws = static_cast<char*>(workspace);
    if (cudaMemsetAsync(ws, 0, sizeof(int), s) != cudaSuccess) return ESTREAM_ERR_CUDA;
    const cudaError_t rc =
        es::launch_router_logits(X, T, H, W_r, E, logits, plan, reinterpret_cast<int*>(ws), s);
    return rc == cudaSuccess ? ESTREAM_OK : ESTREAM_ERR_CUDA;
}
