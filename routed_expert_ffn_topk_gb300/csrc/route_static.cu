// Route build without caller-provided scratch: the allocation-free variant of
// estream_route_build.
//
// Some callers cannot hand this library device scratch memory: a serving
// process that reserved all of its device memory up front for a fixed
// budget (weights, arena, activations) and allows no cudaMalloc afterwards,
// because an allocation at request time can synchronise the whole device
// and stall other streams, or can fail once the budget is carved up; or a
// host framework that owns every device allocation and gives plugins no
// allocator. For them this entry point keeps its scratch (the per-chunk
// route counts, the m-block prefix and an error word) in a file-scope
// device array that every GPU loading the library holds until the process
// exits. It calls no cudaMalloc, cudaFree or allocating library routine.
//
// Limits and sharing rules:
//   - the array holds kStaticScratchBytes (1 MiB); a call whose route-build
//     workspace (estream_route_workspace_bytes(T, E, k, P)) is larger is
//     rejected with ESTREAM_ERR_CAPACITY before anything is enqueued;
//   - every call on a device uses the same array, which keeps the previous
//     call's contents; the call clears the parts that must start at zero
//     (the counts and the error word) on its stream before using them;
//   - calls whose GPU work overlaps (different streams, or different host
//     threads without ordering) race on the array and give wrong results;
//     order them on one stream or serialise them;
//   - the first call on a device looks up the array's device address
//     (cudaGetSymbolAddress, with that device current); make that first call
//     before any stream capture begins on the device;
//   - errors the kernel finds (a phi entry outside [-1, P), a grid barrier
//     that gave up) stay in the array's error word until
//     estream_route_noalloc_error reads and clears it.
#include <mutex>

#include "estream_internal.h"

namespace es {
namespace {

constexpr size_t kStaticScratchBytes = size_t(1) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_route_scratch[kStaticScratchBytes];

std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_route_scratch on the current device (looked up once per
// device). Returns nullptr on failure.
void* scratch_on_current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess) return nullptr;
        g_scratch_addr[dev] = p;
    }
    return g_scratch_addr[dev];
}

}  // namespace
}  // namespace es

using namespace es;

namespace {

// True when p is device memory of the current device (or managed memory),
// the only memory the route kernel can be given.
bool on_current_device(const void* p) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    return (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) && at.device == dev;
}

}  // namespace

extern "C" estream_status estream_route_build_noalloc(const float* logits, int T, int E, int k,
                                                      int renorm, const int32_t* phi, int P,
                                                      int32_t* topk_ids, float* alpha,
                                                      int32_t* offsets, int32_t* rec_tok,
                                                      int32_t* rec_route, void* cuda_stream) {
    if (T < 0 || E < 1 || E > kMaxE || k < 1 || k > E || k > kMaxK || P < 0 || P > kMaxP)
        return ESTREAM_ERR_INVALID_ARG;
    if (!phi && P != E) return ESTREAM_ERR_INVALID_ARG;
    if (!offsets) return ESTREAM_ERR_INVALID_ARG;
    if (T > 0 && (!logits || !topk_ids || !alpha || !rec_tok || !rec_route))
        return ESTREAM_ERR_INVALID_ARG;
    if (static_cast<long long>(T) * k > (1ll << 30)) return ESTREAM_ERR_CAPACITY;
    if (route_workspace_layout(T, k, P).total > kStaticScratchBytes) return ESTREAM_ERR_CAPACITY;
    if (!on_current_device(offsets) || (T > 0 && !on_current_device(logits)) ||
        (phi && !on_current_device(phi)))
        return ESTREAM_ERR_INVALID_ARG;
    void* ws = scratch_on_current_device();
    if (!ws) return ESTREAM_ERR_CUDA;
    cudaError_t rc = launch_route_build(logits, T, E, k, renorm, phi, P, topk_ids, alpha, offsets,
                                        rec_tok, rec_route, nullptr, nullptr, nullptr, 0, ws,
                                        kStaticScratchBytes, static_cast<cudaStream_t>(cuda_stream),
                                        nullptr);
    return rc == cudaSuccess ? ESTREAM_OK : ESTREAM_ERR_CUDA;
}

// The error word sits at the start of the static array (the route build's
// workspace layout puts it at offset 0).
extern "C" estream_status estream_route_noalloc_error(void* cuda_stream) {
    void* ws = scratch_on_current_device();
    if (!ws) return ESTREAM_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    int word = 0;
    int* err = reinterpret_cast<int*>(static_cast<char*>(ws) + route_workspace_layout(0, 1, 0).err_off);
    if (cudaStreamSynchronize(s) != cudaSuccess ||
        cudaMemcpy(&word, err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return ESTREAM_ERR_CUDA;
    if (word == kDevErrNone) return ESTREAM_OK;
    if (cudaMemset(err, 0, sizeof(int)) != cudaSuccess) return ESTREAM_ERR_CUDA;
    return word == kDevErrTimeout ? ESTREAM_ERR_TIMEOUT : ESTREAM_ERR_DEVICE;
}
