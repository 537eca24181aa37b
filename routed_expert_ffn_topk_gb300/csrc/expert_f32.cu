// fp32 expert FFN on the CUDA cores (layers whose X and weights are fp32).
//
// Same two steps as the tensor-core path -- gate/up with the row gather and
// SiLU-mul fused, then down with the weighted scatter-add (Eq. 1 and Eq. 2 of
// "EStream: Fast and Memory-Efficient MoE Prefill through Expert
// Virtualization on Mobile NPUs", section 3.2) -- in full fp32 FMA. The
// tensor cores offer fp32 inputs only as tf32, whose rounding of X, W and h
// does not keep Y inside the accuracy bound, so fp32 layers take this path.
// One CTA handles one record row and 128 output columns; the row's input
// vector is staged in shared memory.
#include "estream_internal.h"

namespace es {
namespace {

// Largest s in [0, seg_count) with offsets[seg_begin + s] <= p.
__device__ __forceinline__ int find_segment(const int32_t* offsets, int seg_begin, int seg_count,
                                            int p) {
    int lo = 0, hi = seg_count;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (offsets[seg_begin + mid] <= p) lo = mid; else hi = mid;
    }
    return lo;
}

__global__ void __launch_bounds__(128) k_gateup_f32(const float* __restrict__ X,
                                                    const float* __restrict__ wg,
                                                    const float* __restrict__ wu,
                                                    const GemmSegments seg, float* __restrict__ h,
                                                    int H, int F) {
    extern __shared__ float xs[];
    const int r0 = seg.offsets[seg.seg_begin];
    const int r1 = seg.offsets[seg.seg_begin + seg.seg_count];
    const int p = r0 + blockIdx.x;
    if (p >= r1) return;
    const int s = find_segment(seg.offsets, seg.seg_begin, seg.seg_count, p);
    const size_t slot = static_cast<size_t>(seg.slot_base + s);
    const float* x = X + static_cast<size_t>(seg.rec_tok[p]) * H;
    for (int k = threadIdx.x; k < H; k += blockDim.x) xs[k] = x[k];
    __syncthreads();
    const int f = blockIdx.y * blockDim.x + threadIdx.x;
    if (f >= F) return;
    const float* rg = wg + (slot * F + f) * H;
    const float* ru = wu + (slot * F + f) * H;
    float g = 0.0f, u = 0.0f;
    for (int k = 0; k < H; ++k) {
        g = fmaf(rg[k], xs[k], g);
        u = fmaf(ru[k], xs[k], u);
    }
    h[static_cast<size_t>(p) * F + f] = g / (1.0f + expf(-g)) * u;
}

__global__ void __launch_bounds__(128) k_down_f32(const float* __restrict__ h,
                                                  const float* __restrict__ wd,
                                                  const GemmSegments seg, float* __restrict__ Y,
                                                  float* __restrict__ out_rows, int H, int F) {
    extern __shared__ float hs[];
    const int r0 = seg.offsets[seg.seg_begin];
    const int r1 = seg.offsets[seg.seg_begin + seg.seg_count];
    const int p = r0 + blockIdx.x;
    if (p >= r1) return;
    const int s = find_segment(seg.offsets, seg.seg_begin, seg.seg_count, p);
    const size_t slot = static_cast<size_t>(seg.slot_base + s);
    for (int k = threadIdx.x; k < F; k += blockDim.x) hs[k] = h[static_cast<size_t>(p) * F + k];
    __syncthreads();
    const int o = blockIdx.y * blockDim.x + threadIdx.x;
    if (o >= H) return;
    const float* rd = wd + (slot * H + o) * F;
    float y = 0.0f;
    for (int k = 0; k < F; ++k) y = fmaf(rd[k], hs[k], y);
    float a = seg.alpha ? seg.alpha[seg.rec_route[p]] : 1.0f;
    a *= seg.seg_scale[seg.seg_begin + s];
    if (out_rows)
        out_rows[static_cast<size_t>(p) * H + o] = a * y;
    else
        atomicAdd(&Y[static_cast<size_t>(seg.rec_tok[p]) * H + o], a * y);
}

}  // namespace

cudaError_t launch_gateup_f32(const float* X, const float* wg, const float* wu,
                              const GemmSegments& seg, float* h, int H, int F, int max_rows,
                              cudaStream_t stream) {
    if (max_rows <= 0 || seg.seg_count <= 0) return cudaSuccess;
    const dim3 grid(static_cast<unsigned>(max_rows), static_cast<unsigned>((F + 127) / 128));
    const size_t smem = sizeof(float) * H;
    if (smem > 48 * 1024) {
        cudaError_t rc = cudaFuncSetAttribute(k_gateup_f32, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              static_cast<int>(smem));
        if (rc != cudaSuccess) return rc;
    }
    k_gateup_f32<<<grid, 128, smem, stream>>>(X, wg, wu, seg, h, H, F);
    return cudaGetLastError();
}

cudaError_t launch_down_f32(const float* h, const float* wd, const GemmSegments& seg, float* Y,
                            float* out_rows, int H, int F, int max_rows, cudaStream_t stream) {
    if (max_rows <= 0 || seg.seg_count <= 0) return cudaSuccess;
    const dim3 grid(static_cast<unsigned>(max_rows), static_cast<unsigned>((H + 127) / 128));
    const size_t smem = sizeof(float) * F;
    if (smem > 48 * 1024) {
        cudaError_t rc = cudaFuncSetAttribute(k_down_f32, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              static_cast<int>(smem));
        if (rc != cudaSuccess) return rc;
    }
    k_down_f32<<<grid, 128, smem, stream>>>(h, wd, seg, Y, out_rows, H, F);
    return cudaGetLastError();
}

}  // namespace es
