// Host runtime of libestream: the C ABI, the bounded expert arena, the pager
// and the sequencing of one MoE layer's prefill.
//
// "EStream: Fast and Memory-Efficient MoE Prefill through Expert
// Virtualization on Mobile NPUs":
//   - section 3.2 / Eq. 3: the arena has three parameter planes B^g, B^u,
//     B^d with fixed bases; slot s of plane j sits at p_{B^j} + s*S_j. Here
//     each plane is described once, at bind time, by a TMA tensor map whose
//     row coordinate s*F (or s*H) addresses the slot: only coordinates change
//     per invocation, never descriptors.
//   - section 3.3: P = B*G slots in B banks of G; storage group q of G
//     experts in the order pi fills one bank; residency states Available ->
//     Filling -> Ready -> InUse -> Available; a Ready bank with no routed
//     work is released directly.
//   - section 3.4: loading overlaps execution; after routing, groups with no
//     routes are skipped; optionally the first banks are filled in storage
//     order before the routes are known.
// GB300 form: the loader is a copy stream issuing cudaMemcpyAsync from pinned
// host memory; "published after fill" is a CUDA event recorded after a
// bank's copies and waited on by the compute stream; "released after the
// last consumer" is an event recorded after the bank's down GEMM and waited
// on by the copy stream before the bank is refilled.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <deque>
#include <new>
#include <vector>

#include "estream_internal.h"

using namespace es;

namespace {

enum BankState { kAvailable = 0, kFilling = 1, kReady = 2, kInUse = 3 };

struct Bank {
    int layer = -1, group = -1;  // contents (valid while layer >= 0)
    bool release_pending = false;
    cudaEvent_t ready = nullptr;
    cudaEvent_t released = nullptr;
};

enum TimedKind { kTRoute = 0, kTFfn, kTShared, kTCombine, kTTotal, kTIo, kTKinds };

// NVTX ranges (domain "estream") for timeline tools: one per layer call, route
// build, expert launch, combine and bank fill, and per standalone route build
// or preload. Names are registered once, so a range costs no formatting; the
// payload carries the layer (bank fills: layer * 65536 + group). Without an
// attached tool NVTX's calls are no-ops.
enum NvtxName {
    kNvRoute = kTRoute, kNvRouted = kTFfn, kNvShared = kTShared, kNvCombine = kTCombine,
    kNvLayer = kTTotal, kNvBankFill = kTIo, kNvRouteFromX, kNvPreload, kNvNames
};
struct NvtxNames {
    nvtxDomainHandle_t dom = nullptr;
    nvtxStringHandle_t name[kNvNames] = {};
};
const NvtxNames& nvtx_names() {
    static const NvtxNames n = [] {
        NvtxNames r;
        r.dom = nvtxDomainCreateA("estream");
        const char* text[kNvNames] = {"route build",  "routed experts", "shared experts",
                                      "combine",      "layer",          "bank fill",
                                      "route from X", "preload"};
        for (int i = 0; i < kNvNames; ++i) r.name[i] = nvtxDomainRegisterStringA(r.dom, text[i]);
        return r;
    }();
    return n;
}
void nvtx_push(int name, long long payload) {
    static const uint32_t color[kNvNames] = {0xff2e9e44, 0xff2a6fdb, 0xff1aa3a3, 0xff8a4fd0,
                                             0xff808080, 0xffe08a1e, 0xff2e9e44, 0xffe08a1e};
    const NvtxNames& n = nvtx_names();
    nvtxEventAttributes_t at = {};
    at.version = NVTX_VERSION;
    at.size = NVTX_EVENT_ATTRIB_STRUCT_SIZE;
    at.colorType = NVTX_COLOR_ARGB;
    at.color = color[name];
    at.payloadType = NVTX_PAYLOAD_TYPE_INT64;
    at.payload.llValue = payload;
    at.messageType = NVTX_MESSAGE_TYPE_REGISTERED;
    at.message.registered = n.name[name];
    nvtxDomainRangePushEx(n.dom, &at);
}
void nvtx_pop() { nvtxDomainRangePop(nvtx_names().dom); }
struct NvtxRange {
    bool on;
    NvtxRange(int name, long long payload, bool on_ = true) : on(on_) {
        if (on) nvtx_push(name, payload);
    }
    ~NvtxRange() {
        if (on) nvtx_pop();
    }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};

struct Timed {
    int kind;
    cudaEvent_t a, b;
};

}  // namespace

struct estream_ctx {
    estream_arena_desc d{};
    int P = 0, n_groups = 0, es = 2, num_sms = 0, device = 0;
    size_t S_gu = 0, S_d = 0, W_e = 0;
    std::vector<const void*> host_pool;
    std::vector<int32_t> perm;
    std::vector<const void*> shared_dev;
    char *plane_g = nullptr, *plane_u = nullptr, *plane_d = nullptr;
    CUtensorMap tm_wg{}, tm_wu{}, tm_wd{}, tm_wd_half{}, tm_h{}, tm_hs{};
    CUtensorMap tm_wg64{}, tm_wu64{};   // 64-row boxes of the gate / up planes (half pair tiles)
    std::vector<CUtensorMap> tm_sg, tm_su, tm_sd, tm_sd_half, tm_sg64, tm_su64;

    // library-owned device workspace
    char* ws = nullptr;
    size_t ws_bytes = 0;
    int32_t *d_perm = nullptr, *topk_ids = nullptr, *rec_tok = nullptr, *rec_route = nullptr,
            *rec_pos = nullptr, *offsets = nullptr, *sh_offsets = nullptr, *sh_mblk = nullptr,
            *sh_rec_tok = nullptr;
    float *alpha = nullptr, *out_rows = nullptr, *out_shared = nullptr;
    float* d_scale = nullptr;                  // [L*E] down-weight scales, storage order
    int32_t *done = nullptr, *sh_done = nullptr;  // per-m-block counters of the fused expert kernel
    int32_t* tickets = nullptr;  // [E+3] zeroed per call: [0] shared experts' and [1+i] the i-th routed
                                 // launch's tile counters, [E+2] the residual rows' counter
    // per-call part of the workspace (everything after the bind-time tables),
    // and the counter regions inside it (for estream_poison_workspace)
    size_t ws_call_off = 0;
    size_t route_ws_bytes = 0;   // the route build's part of the workspace
    float* logits_buf = nullptr; // [T_max][E]: router logits of a layer call from X (two-launch form)
    size_t n_done = 0, n_sh_done = 0, n_tickets = 0;
    int n_ffn_launch = 0;        // routed expert-kernel launches so far in the current layer call
    std::vector<const float*> shared_scale;    // [L] device pointers into shared buffers
    void *route_ws = nullptr, *h = nullptr, *h_shared = nullptr;
    int* dev_err = nullptr;
    int32_t* h_offsets = nullptr;  // pinned host copy of offsets

    cudaStream_t copy_stream = nullptr;        // copy_streams[0]
    std::vector<cudaStream_t> copy_streams;    // Q streams: group k is read on stream k mod Q
    cudaEvent_t copy_done = nullptr, preload_done = nullptr;
    bool preload_pending = false;
    std::vector<Bank> banks;

    bool timing = false;
    estream_stats stats{};
    std::vector<Timed> timed;
    std::vector<cudaEvent_t> event_pool;
    std::vector<int32_t> trace;
    // per-group pipeline events of the last timed paged call (Eq. 5 a/d/s/f)
    struct GroupEvents { cudaEvent_t a, d, s, f; };
    std::vector<GroupEvents> pipe;
    cudaEvent_t pipe_t0 = nullptr, pipe_tne = nullptr;
    int fault_layer = -1, fault_group = -1;
    bool route_withhold_next = false;  // test: the next route build withholds an arrival
    int ffn_phases = 3;                // routed expert kernels: bit 0 gate/up tiles, bit 1 down tiles
    // residual rows of the current call still to be written by an expert
    // launch (the first one takes them; estream_moe_layer_prefill_residual)
    bool resid_pending = false;
    const void* resid_A = nullptr;
    float* resid_Y = nullptr;
    int resid_T = 0;
    bool ffn_down_only_next = false;   // test: the next call runs the down tiles alone
};

namespace {

cudaEvent_t pool_event(estream_ctx* c) {
    if (!c->event_pool.empty()) {
        cudaEvent_t e = c->event_pool.back();
        c->event_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

// Record a (start, end) pair around some work when timing is on.
struct TimedScope {
    estream_ctx* c;
    cudaStream_t s;
    int kind;
    cudaEvent_t a = nullptr;
    bool open = true;  // its NVTX range (same name as the kind) is pushed
    TimedScope(estream_ctx* c_, cudaStream_t s_, int kind_, long long payload)
        : c(c_), s(s_), kind(kind_) {
        nvtx_push(kind, payload);
        if (c->timing) {
            a = pool_event(c);
            if (a) cudaEventRecord(a, s);
        }
    }
    TimedScope(const TimedScope&) = delete;
    TimedScope& operator=(const TimedScope&) = delete;
    void end() {
        if (open) {
            nvtx_pop();
            open = false;
        }
        if (!a) return;
        cudaEvent_t b = pool_event(c);
        if (b) {
            cudaEventRecord(b, s);
            c->timed.push_back({kind, a, b});
        } else {
            c->event_pool.push_back(a);
        }
        a = nullptr;
    }
    ~TimedScope() { end(); }
};

void trace_state(estream_ctx* c, int bank, int layer, int group, int state) {
    c->trace.push_back(bank);
    c->trace.push_back(layer);
    c->trace.push_back(group);
    c->trace.push_back(state);
}

bool device_supported(int dev) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess)
        return false;
    if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return false;
    return major == 10 && minor == 3;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

// The context's device is the current one (its kernels, tensor maps and
// workspace live there; a call made with another device current would launch
// on that device with this device's pointers).
static bool on_bound_device(const estream_ctx* c) {
    int dev = -1;
    return cudaGetDevice(&dev) == cudaSuccess && dev == c->device;
}

namespace {

float bf16_bits_to_float(uint16_t b) {
    uint32_t u = static_cast<uint32_t>(b) << 16;
    float f;
    std::memcpy(&f, &u, sizeof(f));
    return f;
}

// Element size of X and of the h intermediate (bf16 X and fp16 h unless fp32).
size_t elem_size(estream_dtype t) { return t == ESTREAM_F32 ? 4 : 2; }

// Bytes of one expert's [rows][cols] plane as stored in the arena: 4 or 2
// bytes per weight, or for 4-bit weights half a byte per weight plus a 2-byte
// scale per 32 weights (9/16 of a byte per weight).
size_t plane_slot_bytes(estream_dtype t, int rows, int cols) {
    const size_t n = static_cast<size_t>(rows) * cols;
    if (t == ESTREAM_Q4) return n / 16 * 9;
    return n * elem_size(t);
}

// Bytes of one expert's master weights as the packers read them (4-bit
// experts are packed from bf16).
size_t master_bytes(estream_dtype t, int rows, int cols) {
    return static_cast<size_t>(rows) * cols * (t == ESTREAM_F32 ? 4 : 2);
}

// ---- 4-bit packing (Q4_0-style blocks of 32 weights along the reduction) ----
// Scale of a block: the element of largest magnitude m (the first on ties)
// gives d = m / -8, rounded to 5 significant bits (ties to even), then to the
// operand type; code q = clamp(rint(x / d) + 8, 0, 15) (fp32 division, ties
// to even); a zero block has d = 0 and codes 8. With 5 significant bits in d
// every (q - 8) * d is exact in bf16 and in fp16.
float round_to_5_bits(float x) {
    uint32_t u;
    std::memcpy(&u, &x, sizeof(u));
    const uint32_t keep_from = 19;  // fp32 keeps 23 fraction bits, d keeps 4
    const uint32_t low = u & ((1u << keep_from) - 1u);
    const uint32_t half = 1u << (keep_from - 1);
    u &= ~((1u << keep_from) - 1u);
    if (low > half || (low == half && ((u >> keep_from) & 1u))) u += 1u << keep_from;
    float y;
    std::memcpy(&y, &u, sizeof(y));
    return y;
}

uint16_t float_to_bf16_bits_rne(float x) {
    uint32_t u;
    std::memcpy(&u, &x, sizeof(u));
    const uint32_t lsb = (u >> 16) & 1u;
    return static_cast<uint16_t>((u + 0x7FFFu + lsb) >> 16);
}

// One (n-block, k-block) box of a 4-bit plane: tile_rows rows x 64 weights of
// src (fp32 values, row stride cols), written as two column blocks of codes --
// block j holds, for every row, the 16 bytes of weights 32j..32j+31 (byte-word
// w of a block row: bits 4i..4i+3 = code of weight 32j + 8w + 2i, bits
// 16 + 4i.. = code of weight 32j + 8w + 2i + 1) -- then tile_rows x 2 scales
// (uint16 bits of bf16, or of fp16 when fp16 is set). A row's two 16-byte
// halves sit tile_rows * 16 bytes apart, so threads reading consecutive rows
// read consecutive 16-byte words.
void pack_q4_box(const float* src, int cols, int tile_rows, bool fp16, uint8_t* dst) {
    uint8_t* codes = dst;
    uint16_t* scales = reinterpret_cast<uint16_t*>(dst + static_cast<size_t>(tile_rows) * 32);
    for (int r = 0; r < tile_rows; ++r) {
        const float* row = src + static_cast<size_t>(r) * cols;
        uint8_t q[64];
        for (int b = 0; b < 2; ++b) {
            const float* x = row + 32 * b;
            float m = 0.0f;
            for (int j = 0; j < 32; ++j)
                if (std::fabs(x[j]) > std::fabs(m)) m = x[j];
            float d = 0.0f;
            uint16_t bits = 0;
            if (m != 0.0f) {
                const float d5 = round_to_5_bits(m / -8.0f);
                if (fp16) {
                    const __half hd = __float2half_rn(d5);
                    d = __half2float(hd);
                    std::memcpy(&bits, &hd, sizeof(bits));
                } else {
                    bits = float_to_bf16_bits_rne(d5);
                    d = bf16_bits_to_float(bits);
                }
            }
            scales[2 * r + b] = bits;
            for (int j = 0; j < 32; ++j) {
                int c = 8;
                if (d != 0.0f) c = std::min(15, std::max(0, static_cast<int>(std::nearbyint(x[j] / d)) + 8));
                q[32 * b + j] = static_cast<uint8_t>(c);
            }
        }
        for (int w = 0; w < 8; ++w) {
            uint32_t word = 0;
            for (int i = 0; i < 4; ++i) {
                word |= static_cast<uint32_t>(q[8 * w + 2 * i]) << (4 * i);
                word |= static_cast<uint32_t>(q[8 * w + 2 * i + 1]) << (16 + 4 * i);
            }
            const size_t block = static_cast<size_t>(w / 4) * tile_rows * 16;
            std::memcpy(codes + block + static_cast<size_t>(r) * 16 + 4 * (w % 4), &word, sizeof(word));
        }
    }
}

// A whole [rows][cols] bf16 plane, times 2^scale_exp, into tile-major 4-bit
// boxes ([rows/tile_rows][cols/64] boxes of tile_rows rows).
void pack_q4_plane(const uint16_t* src, int rows, int cols, int tile_rows, bool fp16, int scale_exp,
                   uint8_t* dst) {
    const size_t box = static_cast<size_t>(tile_rows) * 36;
    std::vector<float> tile(static_cast<size_t>(tile_rows) * 64);
    size_t o = 0;
    for (int nb = 0; nb < rows / tile_rows; ++nb)
        for (int kb = 0; kb < cols / 64; ++kb) {
            for (int r = 0; r < tile_rows; ++r)
                for (int c = 0; c < 64; ++c)
                    tile[static_cast<size_t>(r) * 64 + c] = std::ldexp(
                        bf16_bits_to_float(src[static_cast<size_t>(nb * tile_rows + r) * cols + kb * 64 + c]),
                        scale_exp);
            pack_q4_box(tile.data(), 64, tile_rows, fp16, dst + o);
            o += box;
        }
}

// Exponent s that puts the largest |w| of a bf16 plane in [2^14, 2^15).
int down_scale_exp(const uint16_t* w, size_t n) {
    float mx = 0.0f;
    for (size_t x = 0; x < n; ++x) mx = std::max(mx, std::fabs(bf16_bits_to_float(w[x])));
    if (!(mx > 0.0f) || !std::isfinite(mx)) return 0;
    int ex = 0;
    std::frexp(mx, &ex);  // mx = m * 2^ex, m in [0.5, 1)
    return 15 - ex;
}

// Offline repack of one expert's plane for the tensor-core path (section
// 3.3, "Offline NPU-Consumable Weight Layout", restated for TMA): the
// [rows][cols] row-major matrix (rows = output features, cols = the
// reduction) is stored tile-major as [rows/tile_rows][cols/64][tile_rows][64],
// so the TMA box of one (n-block, k-block) is a single contiguous run of
// tile_rows * 128 bytes instead of tile_rows strided 128-byte pieces.
template <typename Out, typename Conv>
void pack_tiles(const uint16_t* src, int rows, int cols, int tile_rows, Out* dst, Conv conv) {
    const int nkb = cols / 64;
    size_t o = 0;
    for (int nb = 0; nb < rows / tile_rows; ++nb)
        for (int kb = 0; kb < nkb; ++kb)
            for (int r = 0; r < tile_rows; ++r) {
                const uint16_t* row = src + static_cast<size_t>(nb * tile_rows + r) * cols + kb * 64;
                for (int c = 0; c < 64; ++c) dst[o++] = conv(row[c]);
            }
}

// Gate or up plane of one expert: bf16 copied into 128-row tiles; fp32 copied
// unchanged (the fp32 path reads row-major planes).
void pack_gate_up(const void* src, int F, int H, estream_dtype t, void* dst) {
    if (t == ESTREAM_Q4) {
        pack_q4_plane(static_cast<const uint16_t*>(src), F, H, 128, false, 0, static_cast<uint8_t*>(dst));
        return;
    }
    if (t == ESTREAM_F32) {
        std::memcpy(dst, src, sizeof(float) * static_cast<size_t>(F) * H);
        return;
    }
    pack_tiles(static_cast<const uint16_t*>(src), F, H, 128, static_cast<uint16_t*>(dst),
               [](uint16_t v) { return v; });
}

// Down plane of one expert ([H][F]). bf16: stored as fp16(w * 2^s) in
// 256-row tiles with the largest |w| scaled into [2^14, 2^15); returns 2^-s.
// fp32: copied unchanged, returns 1.
float pack_down(const void* src, int H, int F, estream_dtype t, void* dst) {
    const size_t n = static_cast<size_t>(H) * F;
    if (t == ESTREAM_F32) {
        std::memcpy(dst, src, n * sizeof(float));
        return 1.0f;
    }
    const uint16_t* w = static_cast<const uint16_t*>(src);
    const int s = down_scale_exp(w, n);
    if (t == ESTREAM_Q4) {
        pack_q4_plane(w, H, F, 256, true, s, static_cast<uint8_t*>(dst));
        return std::ldexp(1.0f, -s);
    }
    const float up = std::ldexp(1.0f, s);
    pack_tiles(w, H, F, 256, static_cast<__half*>(dst),
               [up](uint16_t v) { return __float2half_rn(bf16_bits_to_float(v) * up); });
    return std::ldexp(1.0f, -s);
}


estream_status desc_shape_ok(const estream_arena_desc* d) {
    if (!d) return ESTREAM_ERR_INVALID_ARG;
    if (d->wdtype != ESTREAM_F32 && d->wdtype != ESTREAM_BF16 && d->wdtype != ESTREAM_Q4)
        return ESTREAM_ERR_UNSUPPORTED;
    if (d->E < 1 || d->E > kMaxE || d->H < 256 || d->F < 128) return ESTREAM_ERR_INVALID_ARG;
    if (d->H % 256 != 0 || d->F % 128 != 0) return ESTREAM_ERR_INVALID_ARG;
    if (d->G < 1 || d->B < 1 || static_cast<long long>(d->G) * d->B > kMaxP)
        return ESTREAM_ERR_INVALID_ARG;
    return ESTREAM_OK;
}

}  // namespace

extern "C" {

const char* estream_status_string(estream_status s) {
    switch (s) {
        case ESTREAM_OK: return "ok";
        case ESTREAM_ERR_INVALID_ARG: return "invalid argument";
        case ESTREAM_ERR_CAPACITY: return "capacity exceeded";
        case ESTREAM_ERR_NOT_BOUND: return "context not bound";
        case ESTREAM_ERR_CUDA: return "CUDA error";
        case ESTREAM_ERR_PAGER: return "pager failure";
        case ESTREAM_ERR_TIMEOUT: return "device wait timed out";
        case ESTREAM_ERR_DEVICE: return "device-detected data error";
        case ESTREAM_ERR_UNSUPPORTED: return "unsupported device or type";
    }
    return "unknown status";
}

int estream_version(void) { return 10200; }

size_t estream_route_workspace_bytes(int T, int E, int k, int P) {
    if (T < 0 || E < 1 || k < 1 || P < 0 || P > kMaxP) return 0;
    (void)E;
    return route_workspace_layout(T, k, P).total;
}

estream_status estream_route_build(const float* logits, int T, int E, int k, int renorm,
                                   const int32_t* phi, int P, int32_t* topk_ids, float* alpha,
                                   int32_t* offsets, int32_t* rec_tok, int32_t* rec_route,
                                   void* workspace, size_t workspace_bytes, void* cuda_stream) {
    NvtxRange range(kNvRoute, -1);
    if (T < 0 || E < 1 || E > kMaxE || k < 1 || k > E || k > kMaxK || P < 0 || P > kMaxP)
        return ESTREAM_ERR_INVALID_ARG;
    if (!phi && P != E) return ESTREAM_ERR_INVALID_ARG;
    if (!offsets || !workspace || !aligned(workspace, 256)) return ESTREAM_ERR_INVALID_ARG;
    if (T > 0 && (!logits || !topk_ids || !alpha || !rec_tok || !rec_route))
        return ESTREAM_ERR_INVALID_ARG;
    if (static_cast<long long>(T) * k > (1ll << 30)) return ESTREAM_ERR_CAPACITY;
    if (workspace_bytes < route_workspace_layout(T, k, P).total) return ESTREAM_ERR_CAPACITY;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    cudaError_t rc = launch_route_build(logits, T, E, k, renorm, phi, P, topk_ids, alpha, offsets,
                                        rec_tok, rec_route, nullptr, nullptr, nullptr, 0, workspace,
                                        workspace_bytes, s, nullptr);
    return rc == cudaSuccess ? ESTREAM_OK : ESTREAM_ERR_CUDA;
}

// Router logits + route map from X and W_r. One cooperative launch where the
// fused kernel takes the shape; otherwise the router kernel, then the route
// build, on the same stream (the router's error goes to the same word, which
// the route build then keeps).
static cudaError_t route_from_x_any(const void* X, int T, int H, const void* W_r, int E, int k,
                                    int renorm, const int32_t* phi, int P, float* logits,
                                    int32_t* topk_ids, float* alpha, int32_t* offsets,
                                    int32_t* rec_tok, int32_t* rec_route, int32_t* rec_pos,
                                    int32_t* done, int32_t* tickets, int n_tickets, void* ws,
                                    size_t ws_bytes, cudaStream_t s, int* launches,
                                    const ResidualInit* resid, int withhold, int num_sms,
                                    bool* fused) {
    cudaError_t rc = launch_route_from_x(X, T, H, W_r, E, k, renorm, phi, P, logits, topk_ids, alpha,
                                         offsets, rec_tok, rec_route, rec_pos, done, tickets,
                                         n_tickets, ws, ws_bytes, s, launches, resid, withhold);
    if (fused) *fused = rc != cudaErrorNotSupported;
    if (rc != cudaErrorNotSupported) return rc;
    (void)cudaGetLastError();
    int* err = reinterpret_cast<int*>(static_cast<char*>(ws) + route_workspace_layout(T, k, P).err_off);
    rc = cudaMemsetAsync(err, 0, sizeof(int), s);
    if (rc != cudaSuccess) return rc;
    rc = launch_router_logits(X, T, H, W_r, E, logits, router_plan(T, H, E, num_sms), err, s);
    if (rc != cudaSuccess) return rc;
    if (launches && T > 0) *launches += 1;
    return launch_route_build(logits, T, E, k, renorm, phi, P, topk_ids, alpha, offsets, rec_tok,
                              rec_route, rec_pos, done, tickets, n_tickets, ws, ws_bytes, s, launches,
                              resid, withhold, /*clear_err=*/false);
}

estream_status estream_route_build_from_x(const void* X, int T, int H, const void* W_r, int E,
                                          int k, int renorm, const int32_t* phi, int P,
                                          float* logits, int32_t* topk_ids, float* alpha,
                                          int32_t* offsets, int32_t* rec_tok, int32_t* rec_route,
                                          void* workspace, size_t workspace_bytes,
                                          void* cuda_stream) {
    NvtxRange range(kNvRouteFromX, -1);
    if (T < 0 || E < 1 || E > kMaxE || k < 1 || k > E || k > kMaxK || P < 0 || P > kMaxP ||
        H < 64 || H % 64 != 0)
        return ESTREAM_ERR_INVALID_ARG;
    if (!phi && P != E) return ESTREAM_ERR_INVALID_ARG;
    if (!offsets || !workspace || !aligned(workspace, 256)) return ESTREAM_ERR_INVALID_ARG;
    if (T > 0 && (!X || !W_r || !logits || !topk_ids || !alpha || !rec_tok || !rec_route ||
                  !aligned(X, 16) || !aligned(W_r, 16)))
        return ESTREAM_ERR_INVALID_ARG;
    if (static_cast<long long>(T) * k > (1ll << 30)) return ESTREAM_ERR_CAPACITY;
    if (workspace_bytes < route_workspace_layout(T, k, P).total) return ESTREAM_ERR_CAPACITY;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return ESTREAM_ERR_CUDA;
    if (!device_supported(dev)) return ESTREAM_ERR_UNSUPPORTED;
    const cudaError_t rc = route_from_x_any(
        X, T, H, W_r, E, k, renorm, phi, P, logits, topk_ids, alpha, offsets, rec_tok, rec_route,
        nullptr, nullptr, nullptr, 0, workspace, workspace_bytes, static_cast<cudaStream_t>(cuda_stream),
        nullptr, nullptr, 0, sms, nullptr);
    return rc == cudaSuccess ? ESTREAM_OK : ESTREAM_ERR_CUDA;
}

int estream_route_build_from_x_fused(int T, int H, int E, int P) {
    return fused_route_plan(T, H, E, P).ok ? 1 : 0;
}

estream_status estream_workspace_error(void* workspace, void* cuda_stream) {
    if (!workspace) return ESTREAM_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    int* err = reinterpret_cast<int*>(static_cast<char*>(workspace) +
                                      route_workspace_layout(0, 1, 0).err_off);
    int host = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess) return ESTREAM_ERR_CUDA;
    if (cudaMemcpy(&host, err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return ESTREAM_ERR_CUDA;
    if (cudaMemset(err, 0, sizeof(int)) != cudaSuccess) return ESTREAM_ERR_CUDA;
    if (host == kDevErrNone) return ESTREAM_OK;
    return host == kDevErrTimeout ? ESTREAM_ERR_TIMEOUT : ESTREAM_ERR_DEVICE;
}

size_t estream_arena_bytes(int E, int H, int F, int G, int B, estream_dtype wdtype) {
    (void)E;
    if (H < 1 || F < 1 || G < 1 || B < 1) return 0;
    return static_cast<size_t>(B) * G * 3 * plane_slot_bytes(wdtype, F, H);
}

size_t estream_pool_bytes(int E, int H, int F, estream_dtype wdtype) {
    if (E < 1 || H < 1 || F < 1) return 0;
    return static_cast<size_t>(E) * 3 * plane_slot_bytes(wdtype, F, H) + align_up(sizeof(float) * E, 16);
}

size_t estream_shared_bytes(int n_shared, int H, int F_shared, estream_dtype wdtype) {
    if (n_shared < 1 || H < 1 || F_shared < 1) return 0;
    return static_cast<size_t>(n_shared) * 3 * plane_slot_bytes(wdtype, F_shared, H) +
           align_up(sizeof(float) * n_shared, 16);
}

estream_status estream_pack_experts(const estream_arena_desc* d, int layer, const void* wg,
                                    const void* wu, const void* wd, void* host_pool_out) {
    estream_status st = desc_shape_ok(d);
    if (st != ESTREAM_OK) return st;
    if (!wg || !wu || !wd || !host_pool_out || layer < 0 || layer >= std::max(1, d->L))
        return ESTREAM_ERR_INVALID_ARG;
    const size_t Sin = master_bytes(d->wdtype, d->F, d->H);    // one input matrix of one expert
    const size_t S = plane_slot_bytes(d->wdtype, d->F, d->H);  // one packed plane slice
    const size_t W = 3 * S;
    const int32_t* perm = d->perm ? d->perm + static_cast<size_t>(layer) * d->E : nullptr;
    std::vector<char> seen(d->E, 0);
    for (int e = 0; e < d->E; ++e) {
        const int pos = perm ? perm[e] : e;
        if (pos < 0 || pos >= d->E || seen[pos]) return ESTREAM_ERR_INVALID_ARG;
        seen[pos] = 1;
    }
    char* out = static_cast<char*>(host_pool_out);
    float* scales = reinterpret_cast<float*>(out + static_cast<size_t>(d->E) * W);
    for (int e = 0; e < d->E; ++e) {
        const int pos = perm ? perm[e] : e;
        const int q = pos / d->G, r = pos % d->G;
        const int n_q = std::min(d->G, d->E - q * d->G);
        char* grp = out + static_cast<size_t>(q) * d->G * W;
        pack_gate_up(static_cast<const char*>(wg) + e * Sin, d->F, d->H, d->wdtype,
                     grp + static_cast<size_t>(r) * S);
        pack_gate_up(static_cast<const char*>(wu) + e * Sin, d->F, d->H, d->wdtype,
                     grp + static_cast<size_t>(n_q) * S + static_cast<size_t>(r) * S);
        void* down = grp + 2 * static_cast<size_t>(n_q) * S + static_cast<size_t>(r) * S;
        scales[pos] = pack_down(static_cast<const char*>(wd) + e * Sin, d->H, d->F, d->wdtype, down);
    }
    return ESTREAM_OK;
}

estream_status estream_pack_shared(const estream_arena_desc* d, const void* sg, const void* su,
                                   const void* sd, void* out) {
    if (!d || !sg || !su || !sd || !out || d->n_shared < 1 || d->F_shared < 1 || d->H < 1)
        return ESTREAM_ERR_INVALID_ARG;
    if (d->wdtype != ESTREAM_F32 && d->wdtype != ESTREAM_BF16 && d->wdtype != ESTREAM_Q4)
        return ESTREAM_ERR_UNSUPPORTED;
    if (d->H % 256 != 0 || d->F_shared % 128 != 0) return ESTREAM_ERR_INVALID_ARG;
    const size_t Sin = master_bytes(d->wdtype, d->F_shared, d->H);
    const size_t S = plane_slot_bytes(d->wdtype, d->F_shared, d->H);
    const size_t ns = static_cast<size_t>(d->n_shared);
    char* o = static_cast<char*>(out);
    float* scales = reinterpret_cast<float*>(o + 3 * ns * S);
    for (size_t s = 0; s < ns; ++s) {
        pack_gate_up(static_cast<const char*>(sg) + s * Sin, d->F_shared, d->H, d->wdtype, o + s * S);
        pack_gate_up(static_cast<const char*>(su) + s * Sin, d->F_shared, d->H, d->wdtype,
                     o + ns * S + s * S);
        scales[s] = pack_down(static_cast<const char*>(sd) + s * Sin, d->H, d->F_shared, d->wdtype,
                              o + 2 * ns * S + s * S);
    }
    return ESTREAM_OK;
}

void estream_unbind(estream_ctx* c);

estream_status estream_bind_arena(estream_ctx** out, const estream_arena_desc* d) {
    if (!out) return ESTREAM_ERR_INVALID_ARG;
    *out = nullptr;
    estream_status st = desc_shape_ok(d);
    if (st != ESTREAM_OK) return st;
    if (d->L < 1 || d->T_max < 1 || d->k_max < 1 || d->k_max > d->E || d->k_max > kMaxK ||
        d->Q < 1 || !d->arena_dev || !aligned(d->arena_dev, 256) || !d->host_pool)
        return ESTREAM_ERR_INVALID_ARG;
    if (d->schedule != ESTREAM_SCHED_AFTER_ROUTING && d->schedule != ESTREAM_SCHED_PREFETCH)
        return ESTREAM_ERR_INVALID_ARG;
    if (d->ffn_form != ESTREAM_FFN_AUTO && d->ffn_form != ESTREAM_FFN_SINGLE &&
        d->ffn_form != ESTREAM_FFN_PAIR)
        return ESTREAM_ERR_INVALID_ARG;
    if (d->n_shared < 0 || (d->n_shared > 0 && (d->F_shared < 128 || d->F_shared % 128 != 0 ||
                                                 !d->shared_dev)))
        return ESTREAM_ERR_INVALID_ARG;
    if (d->arena_bytes < estream_arena_bytes(d->E, d->H, d->F, d->G, d->B, d->wdtype))
        return ESTREAM_ERR_CAPACITY;
    if (static_cast<long long>(d->T_max) * d->k_max > (1ll << 30)) return ESTREAM_ERR_CAPACITY;
    // tile row indices of the weight planes are 32-bit
    if (static_cast<long long>(d->B) * d->G * d->F * d->H / 64 >= (1ll << 31) ||
        static_cast<long long>(d->n_shared) * d->F_shared * d->H / 64 >= (1ll << 31))
        return ESTREAM_ERR_CAPACITY;
    for (int l = 0; l < d->L; ++l) {
        if (!d->host_pool[l]) return ESTREAM_ERR_INVALID_ARG;
        if (d->n_shared > 0 && (!d->shared_dev[l] || !aligned(d->shared_dev[l], 16)))
            return ESTREAM_ERR_INVALID_ARG;
        if (d->perm) {
            std::vector<char> seen(d->E, 0);
            for (int e = 0; e < d->E; ++e) {
                const int p = d->perm[static_cast<size_t>(l) * d->E + e];
                if (p < 0 || p >= d->E || seen[p]) return ESTREAM_ERR_INVALID_ARG;
                seen[p] = 1;
            }
        }
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return ESTREAM_ERR_CUDA;
    if (!device_supported(dev)) return ESTREAM_ERR_UNSUPPORTED;

    estream_ctx* c = new (std::nothrow) estream_ctx();
    if (!c) return ESTREAM_ERR_CUDA;
    c->d = *d;
    c->device = dev;
    c->P = d->B * d->G;
    c->n_groups = (d->E + d->G - 1) / d->G;
    c->es = static_cast<int>(elem_size(d->wdtype));
    c->S_gu = plane_slot_bytes(d->wdtype, d->F, d->H);
    c->S_d = plane_slot_bytes(d->wdtype, d->H, d->F);
    c->W_e = 2 * c->S_gu + c->S_d;
    c->host_pool.assign(d->host_pool, d->host_pool + d->L);
    c->perm.resize(static_cast<size_t>(d->L) * d->E);
    for (int l = 0; l < d->L; ++l)
        for (int e = 0; e < d->E; ++e)
            c->perm[static_cast<size_t>(l) * d->E + e] =
                d->perm ? d->perm[static_cast<size_t>(l) * d->E + e] : e;
    if (d->n_shared > 0) c->shared_dev.assign(d->shared_dev, d->shared_dev + d->L);
    c->d.host_pool = nullptr;
    c->d.perm = nullptr;
    c->d.shared_dev = nullptr;
    cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, dev);

    // Eq. 3: plane bases; slot s of plane j at base_j + s * S_j
    const size_t plane_bytes = static_cast<size_t>(c->P) * c->S_gu;
    c->plane_g = static_cast<char*>(d->arena_dev);
    c->plane_u = c->plane_g + plane_bytes;
    c->plane_d = c->plane_u + plane_bytes;

    const bool f32 = d->wdtype == ESTREAM_F32;
    const int R_cap = d->T_max * d->k_max;
    const int E = d->E;

    // workspace layout
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = align_up(off + (bytes ? bytes : 1), 1024);
        return o;
    };
    const size_t o_err = take(sizeof(int));
    const size_t o_perm = take(sizeof(int32_t) * c->perm.size());
    const size_t o_scale = take(sizeof(float) * c->perm.size());
    const size_t o_ids = take(sizeof(int32_t) * R_cap);
    const size_t o_alpha = take(sizeof(float) * R_cap);
    const size_t o_rtok = take(sizeof(int32_t) * R_cap);
    const size_t o_rroute = take(sizeof(int32_t) * R_cap);
    const size_t o_rpos = take(sizeof(int32_t) * R_cap);
    const size_t o_offs = take(sizeof(int32_t) * (E + 2));
    const size_t o_lg = take(f32 ? 0 : sizeof(float) * static_cast<size_t>(d->T_max) * E);
    const size_t o_rws = take(route_workspace_layout(d->T_max, d->k_max, E).total);
    const size_t o_done = take(sizeof(int32_t) * ((R_cap + kBM - 1) / kBM + E + 1));
    const size_t o_tick = take(sizeof(int32_t) * (E + 3));
    const size_t o_h = take(static_cast<size_t>(R_cap) * d->F * c->es);
    size_t o_sh_offs = 0, o_sh_mblk = 0, o_sh_tok = 0, o_hs = 0, o_outs = 0, o_out = 0;
    const int RS_cap = d->n_shared * d->T_max;
    size_t o_sh_done = 0;
    if (d->n_shared > 0) {
        o_sh_done = take(sizeof(int32_t) * (d->n_shared * ((d->T_max + kBM - 1) / kBM) + 1));
        o_sh_offs = take(sizeof(int32_t) * (d->n_shared + 2));
        o_sh_mblk = take(sizeof(int32_t) * (d->n_shared + 2));
        o_sh_tok = take(sizeof(int32_t) * RS_cap);
        o_hs = take(static_cast<size_t>(RS_cap) * d->F_shared * c->es);
    }
    if (d->deterministic) {
        o_out = take(static_cast<size_t>(R_cap) * d->H * sizeof(float));
        if (d->n_shared > 0) o_outs = take(static_cast<size_t>(RS_cap) * d->H * sizeof(float));
    }
    c->ws_bytes = off;
    st = ESTREAM_ERR_CUDA;
    do {
        if (cudaMalloc(&c->ws, c->ws_bytes) != cudaSuccess) break;
        c->dev_err = reinterpret_cast<int*>(c->ws + o_err);
        c->d_perm = reinterpret_cast<int32_t*>(c->ws + o_perm);
        c->d_scale = reinterpret_cast<float*>(c->ws + o_scale);
        c->topk_ids = reinterpret_cast<int32_t*>(c->ws + o_ids);
        c->alpha = reinterpret_cast<float*>(c->ws + o_alpha);
        c->rec_tok = reinterpret_cast<int32_t*>(c->ws + o_rtok);
        c->rec_route = reinterpret_cast<int32_t*>(c->ws + o_rroute);
        c->rec_pos = reinterpret_cast<int32_t*>(c->ws + o_rpos);
        c->offsets = reinterpret_cast<int32_t*>(c->ws + o_offs);
        c->logits_buf = f32 ? nullptr : reinterpret_cast<float*>(c->ws + o_lg);
        c->route_ws = c->ws + o_rws;
        c->route_ws_bytes = route_workspace_layout(d->T_max, d->k_max, E).total;
        c->done = reinterpret_cast<int32_t*>(c->ws + o_done);
        c->tickets = reinterpret_cast<int32_t*>(c->ws + o_tick);
        c->h = c->ws + o_h;
        c->ws_call_off = o_ids;
        c->n_done = (R_cap + kBM - 1) / kBM + E + 1;
        c->n_tickets = E + 3;
        if (d->n_shared > 0) {
            c->n_sh_done = d->n_shared * ((d->T_max + kBM - 1) / kBM) + 1;
            c->sh_done = reinterpret_cast<int32_t*>(c->ws + o_sh_done);
            c->sh_offsets = reinterpret_cast<int32_t*>(c->ws + o_sh_offs);
            c->sh_mblk = reinterpret_cast<int32_t*>(c->ws + o_sh_mblk);
            c->sh_rec_tok = reinterpret_cast<int32_t*>(c->ws + o_sh_tok);
            c->h_shared = c->ws + o_hs;
        }
        if (d->deterministic) {
            c->out_rows = reinterpret_cast<float*>(c->ws + o_out);
            if (d->n_shared > 0) c->out_shared = reinterpret_cast<float*>(c->ws + o_outs);
        }
        if (cudaMemset(c->ws, 0, o_perm) != cudaSuccess) break;
        // the route build's error word and grid-barrier counter
        if (cudaMemset(c->route_ws, 0, route_workspace_layout(0, 1, 0).hist_off) != cudaSuccess)
            break;
        if (cudaMemcpy(c->d_perm, c->perm.data(), sizeof(int32_t) * c->perm.size(),
                       cudaMemcpyHostToDevice) != cudaSuccess)
            break;
        bool sc_ok = true;
        for (int l = 0; l < d->L && sc_ok; ++l)
            sc_ok = cudaMemcpy(c->d_scale + static_cast<size_t>(l) * E,
                               static_cast<const char*>(c->host_pool[l]) + static_cast<size_t>(E) * c->W_e,
                               sizeof(float) * E, cudaMemcpyHostToDevice) == cudaSuccess;
        if (!sc_ok) break;
        if (cudaMallocHost(&c->h_offsets, sizeof(int32_t) * (E + 2)) != cudaSuccess) break;
        bool cs_ok = true;
        c->copy_streams.resize(d->Q, nullptr);
        for (int q = 0; q < d->Q && cs_ok; ++q)
            cs_ok = cudaStreamCreateWithFlags(&c->copy_streams[q], cudaStreamNonBlocking) == cudaSuccess;
        if (!cs_ok) break;
        c->copy_stream = c->copy_streams[0];
        if (cudaEventCreateWithFlags(&c->copy_done, cudaEventDisableTiming) != cudaSuccess) break;
        if (cudaEventCreateWithFlags(&c->preload_done, cudaEventDisableTiming) != cudaSuccess) break;
        c->banks.resize(d->B);
        bool ev_ok = true;
        for (auto& b : c->banks) {
            ev_ok = ev_ok && cudaEventCreateWithFlags(&b.ready, cudaEventDisableTiming) == cudaSuccess;
            ev_ok = ev_ok &&
                    cudaEventCreateWithFlags(&b.released, cudaEventDisableTiming) == cudaSuccess;
        }
        if (!ev_ok) break;
        // tensor maps (fixed bases, Eq. 3); the fp32 path reads the planes directly
        bool tm_ok = true;
        const CUtensorMapDataType BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
        const CUtensorMapDataType HF = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
        if (d->n_shared > 0) {
            c->shared_scale.resize(d->L);
            const size_t sp = static_cast<size_t>(d->n_shared) * plane_slot_bytes(d->wdtype, d->F_shared, d->H);
            for (int l = 0; l < d->L; ++l)
                c->shared_scale[l] = reinterpret_cast<const float*>(
                    static_cast<const char*>(c->shared_dev[l]) + 3 * sp);
        }
        const bool q4 = d->wdtype == ESTREAM_Q4;  // 4-bit planes are read with plain bulk copies
        if (!f32 && !q4) {
            // tile-major planes: one 128-byte row of 64 elements per tensor row
            const uint64_t plane_rows = static_cast<uint64_t>(c->P) * d->F * d->H / 64;
            tm_ok = tm_ok && encode_tmap_2d(&c->tm_wg, BF, c->plane_g, 64, plane_rows, 128, 64,
                                            128) == CUDA_SUCCESS;
            tm_ok = tm_ok && encode_tmap_2d(&c->tm_wu, BF, c->plane_u, 64, plane_rows, 128, 64,
                                            128) == CUDA_SUCCESS;
            tm_ok = tm_ok && encode_tmap_2d(&c->tm_wd, HF, c->plane_d, 64, plane_rows, 128, 64,
                                            256) == CUDA_SUCCESS;
            tm_ok = tm_ok && encode_tmap_2d(&c->tm_wd_half, HF, c->plane_d, 64, plane_rows, 128,
                                            64, 128) == CUDA_SUCCESS;
            tm_ok = tm_ok && encode_tmap_2d(&c->tm_wg64, BF, c->plane_g, 64, plane_rows, 128, 64,
                                            64) == CUDA_SUCCESS;
            tm_ok = tm_ok && encode_tmap_2d(&c->tm_wu64, BF, c->plane_u, 64, plane_rows, 128, 64,
                                            64) == CUDA_SUCCESS;
        }
        if (!f32) {
            tm_ok = tm_ok && encode_tmap_2d(&c->tm_h, HF, c->h, d->F, static_cast<uint64_t>(R_cap),
                                            static_cast<uint64_t>(d->F) * 2, 64, 128) == CUDA_SUCCESS;
            if (d->n_shared > 0)
                tm_ok = tm_ok && encode_tmap_2d(&c->tm_hs, HF, c->h_shared, d->F_shared,
                                                static_cast<uint64_t>(RS_cap),
                                                static_cast<uint64_t>(d->F_shared) * 2, 64, 128) ==
                                     CUDA_SUCCESS;
        }
        if (!f32 && !q4) {
            if (d->n_shared > 0) {
                const int Fs = d->F_shared;
                c->tm_sg.resize(d->L);
                c->tm_su.resize(d->L);
                c->tm_sd.resize(d->L);
                c->tm_sd_half.resize(d->L);
                c->tm_sg64.resize(d->L);
                c->tm_su64.resize(d->L);
                const size_t sp = static_cast<size_t>(d->n_shared) * Fs * d->H * 2;
                for (int l = 0; l < d->L && tm_ok; ++l) {
                    const char* base = static_cast<const char*>(c->shared_dev[l]);
                    const uint64_t srows = static_cast<uint64_t>(d->n_shared) * Fs * d->H / 64;
                    tm_ok = tm_ok && encode_tmap_2d(&c->tm_sg[l], BF, base, 64, srows, 128, 64,
                                                    128) == CUDA_SUCCESS;
                    tm_ok = tm_ok && encode_tmap_2d(&c->tm_su[l], BF, base + sp, 64, srows, 128,
                                                    64, 128) == CUDA_SUCCESS;
                    tm_ok = tm_ok && encode_tmap_2d(&c->tm_sd[l], HF, base + 2 * sp, 64, srows, 128,
                                                    64, 256) == CUDA_SUCCESS;
                    tm_ok = tm_ok && encode_tmap_2d(&c->tm_sd_half[l], HF, base + 2 * sp, 64,
                                                    srows, 128, 64, 128) == CUDA_SUCCESS;
                    tm_ok = tm_ok && encode_tmap_2d(&c->tm_sg64[l], BF, base, 64, srows, 128, 64,
                                                    64) == CUDA_SUCCESS;
                    tm_ok = tm_ok && encode_tmap_2d(&c->tm_su64[l], BF, base + sp, 64, srows, 128,
                                                    64, 64) == CUDA_SUCCESS;
                }
            }
        }
        if (!tm_ok) break;
        st = ESTREAM_OK;
    } while (false);
    if (st != ESTREAM_OK) {
        estream_unbind(c);
        return st;
    }
    *out = c;
    return ESTREAM_OK;
}

}  // extern "C"

namespace {

// Copies of storage group q of `layer` into bank b: three plane slices.
estream_status fill_bank(estream_ctx* c, int layer, int q, int b, size_t* bytes,
                         cudaStream_t cs, estream_ctx::GroupEvents* ev = nullptr) {
    const int G = c->d.G;
    const int n_q = std::min(G, c->d.E - q * G);
    const char* src = static_cast<const char*>(c->host_pool[layer]) +
                      static_cast<size_t>(q) * G * c->W_e;
    const size_t gbytes = static_cast<size_t>(n_q) * c->S_gu;
    const size_t dbytes = static_cast<size_t>(n_q) * c->S_d;
    Bank& bk = c->banks[b];
    if (bk.release_pending) {
        if (cudaStreamWaitEvent(cs, bk.released, 0) != cudaSuccess) return ESTREAM_ERR_CUDA;
        bk.release_pending = false;
    }
    if (ev) cudaEventRecord(ev->a, cs);
    trace_state(c, b, layer, q, kFilling);
    bk.layer = layer;
    bk.group = q;
    TimedScope io(c, cs, kTIo, static_cast<long long>(layer) * 65536 + q);
    const size_t slot0 = static_cast<size_t>(b) * G;
    if (cudaMemcpyAsync(c->plane_g + slot0 * c->S_gu, src, gbytes, cudaMemcpyHostToDevice, cs) !=
            cudaSuccess ||
        cudaMemcpyAsync(c->plane_u + slot0 * c->S_gu, src + gbytes, gbytes, cudaMemcpyHostToDevice,
                        cs) != cudaSuccess ||
        cudaMemcpyAsync(c->plane_d + slot0 * c->S_d, src + 2 * gbytes, dbytes,
                        cudaMemcpyHostToDevice, cs) != cudaSuccess)
        return ESTREAM_ERR_CUDA;
    io.end();
    if (ev) cudaEventRecord(ev->d, cs);
    if (cudaEventRecord(bk.ready, cs) != cudaSuccess) return ESTREAM_ERR_CUDA;
    trace_state(c, b, layer, q, kReady);
    *bytes += 2 * gbytes + dbytes;
    return ESTREAM_OK;
}

// Form of the bf16 fused expert kernel for `rows` records over `segments`
// expert segments: ESTREAM_FFN_AUTO takes the CTA-pair form (256-record
// tiles) when a segment holds on average at least ESTREAM_PAIR_MIN_ROWS.
bool pair_form(const estream_ctx* c, long long rows, int segments) {
    if (c->d.ffn_form == ESTREAM_FFN_PAIR) return true;
    if (c->d.ffn_form == ESTREAM_FFN_SINGLE) return false;
    return segments > 0 && rows >= static_cast<long long>(ESTREAM_PAIR_MIN_ROWS) * segments;
}

// Hands the call's pending residual rows to an expert launch over `seg`
// (which will launch: segments and m-blocks to cover).
void take_residual(estream_ctx* c, GemmSegments& seg) {
    if (!c->resid_pending || seg.seg_count <= 0 || seg.max_tiles_m <= 0) return;
    seg.resid_A = c->resid_A;
    seg.resid_Y = c->resid_Y;
    seg.resid_elem = c->es;
    seg.resid_T = c->resid_T;
    seg.resid_done = c->tickets + c->d.E + 2;
    c->resid_pending = false;
}

// K2 + K3 over segments [seg_begin, seg_begin + seg_count) of the routed
// route map, whose experts sit in consecutive arena slots from slot_base.
estream_status run_routed(estream_ctx* c, cudaStream_t s, const void* X, int layer,
                          const int32_t* mblk, int seg_begin, int seg_count, int slot_base,
                          int max_tiles_m, int max_rows, bool pair, float* Y) {
    GemmSegments seg{};
    seg.offsets = c->offsets;
    seg.mblk = mblk;
    seg.rec_tok = c->rec_tok;
    seg.rec_route = c->rec_route;
    seg.alpha = c->alpha;
    seg.seg_scale = c->d_scale + static_cast<size_t>(layer) * c->d.E;
    seg.seg_begin = seg_begin;
    seg.seg_count = seg_count;
    seg.slot_base = slot_base;
    seg.max_tiles_m = max_tiles_m;
    if (c->d.wdtype != ESTREAM_F32) take_residual(c, seg);
    TimedScope ts(c, s, kTFfn, layer);
    // this launch's dynamic tile counter, zeroed by the call's route build. The
    // 4-bit kernel takes its tiles dynamically (measured 5.5% faster on the
    // OLMoE shape); the bf16 kernel keeps the balanced static order (3% faster
    // than dynamic there).
    int* ticket = c->n_ffn_launch < c->d.E + 1 ? c->tickets + 1 + c->n_ffn_launch : nullptr;
    ++c->n_ffn_launch;
    cudaError_t rc;
    if (c->d.wdtype == ESTREAM_F32) {
        rc = launch_gateup_f32(static_cast<const float*>(X), reinterpret_cast<const float*>(c->plane_g),
                               reinterpret_cast<const float*>(c->plane_u), seg,
                               static_cast<float*>(c->h), c->d.H, c->d.F, max_rows, s);
        if (rc == cudaSuccess)
            rc = launch_down_f32(static_cast<const float*>(c->h),
                                 reinterpret_cast<const float*>(c->plane_d), seg, Y, c->out_rows,
                                 c->d.H, c->d.F, max_rows, s);
        c->stats.launches += 2;
    } else if (c->d.wdtype == ESTREAM_Q4) {
        rc = pair ? launch_expert_ffn_pair_q4(reinterpret_cast<const uint8_t*>(c->plane_g),
                                              reinterpret_cast<const uint8_t*>(c->plane_u),
                                              reinterpret_cast<const uint8_t*>(c->plane_d), c->S_gu,
                                              c->S_d, &c->tm_h, seg, X, c->h, Y, c->out_rows,
                                              c->done, c->d.H, c->d.F, c->ffn_phases, c->dev_err, s)
                  : launch_expert_ffn_q4(reinterpret_cast<const uint8_t*>(c->plane_g),
                                         reinterpret_cast<const uint8_t*>(c->plane_u),
                                         reinterpret_cast<const uint8_t*>(c->plane_d), c->S_gu,
                                         c->S_d, &c->tm_h, seg, X, c->h, Y, c->out_rows, c->done,
                                         ticket, c->d.H, c->d.F, c->ffn_phases, c->dev_err,
                                         c->num_sms, s);
        c->stats.launches += 1;
    } else {
        rc = pair
                 ? launch_expert_ffn_pair(&c->tm_wg, &c->tm_wu, &c->tm_wd_half, &c->tm_h, &c->tm_wg64,
                                          &c->tm_wu64, seg, X, c->h,
                                          Y, c->out_rows, c->done, c->d.H, c->d.F, c->ffn_phases, c->dev_err,
                                          false, s)
                 : launch_expert_ffn(&c->tm_wg, &c->tm_wu, &c->tm_wd, &c->tm_h, seg, X, c->h, Y,
                                     c->out_rows, c->done, nullptr, c->d.H, c->d.F, c->ffn_phases, c->dev_err,
                                     c->num_sms, s);
        c->stats.launches += 1;
    }
    if (rc != cudaSuccess) return ESTREAM_ERR_CUDA;
    c->stats.n_ffn += c->timing ? 1 : 0;
    return ESTREAM_OK;
}

// Shared experts: identity route map over all T tokens, weight 1.
estream_status run_shared(estream_ctx* c, cudaStream_t s, const void* X,
                          int layer, int T, float* Y) {
    TimedScope ts(c, s, kTShared, layer);
    const int ns = c->d.n_shared;
    if (launch_identity_map(T, ns, c->sh_offsets, c->sh_rec_tok, c->sh_mblk, c->sh_done, s) !=
        cudaSuccess)
        return ESTREAM_ERR_CUDA;
    GemmSegments seg{};
    seg.offsets = c->sh_offsets;
    seg.mblk = c->sh_mblk;
    seg.rec_tok = c->sh_rec_tok;
    seg.rec_route = nullptr;
    seg.alpha = nullptr;
    seg.seg_scale = c->shared_scale[layer];
    seg.seg_begin = 0;
    seg.seg_count = ns;
    seg.slot_base = 0;
    seg.max_tiles_m = ns * ((T + kBM - 1) / kBM);
    if (c->d.wdtype != ESTREAM_F32) take_residual(c, seg);
    const int Fs = c->d.F_shared;
    cudaError_t rc;
    if (c->d.wdtype == ESTREAM_F32) {
        const float* base = static_cast<const float*>(c->shared_dev[layer]);
        const size_t sp = static_cast<size_t>(ns) * Fs * c->d.H;
        rc = launch_gateup_f32(static_cast<const float*>(X), base, base + sp, seg,
                               static_cast<float*>(c->h_shared), c->d.H, Fs, ns * T, s);
        if (rc == cudaSuccess)
            rc = launch_down_f32(static_cast<const float*>(c->h_shared), base + 2 * sp, seg, Y,
                                 c->out_shared, c->d.H, Fs, ns * T, s);
    } else if (c->d.wdtype == ESTREAM_Q4) {
        const uint8_t* base = static_cast<const uint8_t*>(c->shared_dev[layer]);
        const size_t S1 = plane_slot_bytes(ESTREAM_Q4, Fs, c->d.H);  // one shared expert's plane
        const size_t sp = static_cast<size_t>(ns) * S1;
        rc = pair_form(c, T, 1)
                 ? launch_expert_ffn_pair_q4(base, base + sp, base + 2 * sp, S1, S1, &c->tm_hs, seg, X,
                                             c->h_shared, Y, c->out_shared, c->sh_done, c->d.H, Fs, 3,
                                             c->dev_err, s)
                 : launch_expert_ffn_q4(base, base + sp, base + 2 * sp, S1, S1, &c->tm_hs, seg, X,
                                        c->h_shared, Y, c->out_shared, c->sh_done, c->tickets, c->d.H,
                                        Fs, 3, c->dev_err, c->num_sms, s);
    } else {
        rc = pair_form(c, T, 1)
                 ? launch_expert_ffn_pair(&c->tm_sg[layer], &c->tm_su[layer], &c->tm_sd_half[layer],
                                          &c->tm_hs, &c->tm_sg64[layer], &c->tm_su64[layer],
                                          seg, X, c->h_shared, Y, c->out_shared,
                                          c->sh_done, c->d.H, Fs, 3, c->dev_err, true, s)
                 : launch_expert_ffn(&c->tm_sg[layer], &c->tm_su[layer], &c->tm_sd[layer], &c->tm_hs,
                                     seg, X, c->h_shared, Y, c->out_shared, c->sh_done, nullptr,
                                     c->d.H, Fs, 3, c->dev_err, c->num_sms, s);
    }
    if (rc != cudaSuccess) return ESTREAM_ERR_CUDA;
    c->stats.launches += c->d.wdtype == ESTREAM_F32 ? 3 : 2;
    return ESTREAM_OK;
}

bool layer_resident(const estream_ctx* c, int layer) {
    if (c->n_groups > c->d.B) return false;
    for (int q = 0; q < c->n_groups; ++q)
        if (c->banks[q].layer != layer || c->banks[q].group != q) return false;
    return true;
}

void drain(estream_ctx* c, cudaStream_t s) {
    for (cudaStream_t cs : c->copy_streams) cudaStreamSynchronize(cs);
    cudaStreamSynchronize(s);
}

estream_status sync_copies(estream_ctx* c) {
    for (cudaStream_t cs : c->copy_streams)
        if (cudaStreamSynchronize(cs) != cudaSuccess) return ESTREAM_ERR_CUDA;
    return ESTREAM_OK;
}

// The copy streams wait for all work enqueued so far on `s` (a bank may only
// be overwritten once earlier work on `s` no longer reads it).
estream_status copies_after(estream_ctx* c, cudaStream_t s) {
    if (cudaEventRecord(c->copy_done, s) != cudaSuccess) return ESTREAM_ERR_CUDA;
    for (cudaStream_t cs : c->copy_streams)
        if (cudaStreamWaitEvent(cs, c->copy_done, 0) != cudaSuccess) return ESTREAM_ERR_CUDA;
    return ESTREAM_OK;
}

// `s` waits for everything enqueued so far on the copy streams.
estream_status stream_after_copies(estream_ctx* c, cudaStream_t s) {
    for (cudaStream_t cs : c->copy_streams) {
        if (cudaEventRecord(c->copy_done, cs) != cudaSuccess ||
            cudaStreamWaitEvent(s, c->copy_done, 0) != cudaSuccess)
            return ESTREAM_ERR_CUDA;
    }
    return ESTREAM_OK;
}

void release_pipe_events(estream_ctx* c) {
    for (auto& g : c->pipe) {
        c->event_pool.push_back(g.a);
        c->event_pool.push_back(g.d);
        c->event_pool.push_back(g.s);
        c->event_pool.push_back(g.f);
    }
    c->pipe.clear();
    if (c->pipe_t0) c->event_pool.push_back(c->pipe_t0);
    if (c->pipe_tne) c->event_pool.push_back(c->pipe_tne);
    c->pipe_t0 = c->pipe_tne = nullptr;
}

}  // namespace

extern "C" {

estream_status estream_arena_preload(estream_ctx* c, int layer, void* cuda_stream) {
    NvtxRange range(kNvPreload, layer);
    if (!c) return ESTREAM_ERR_NOT_BOUND;
    if (layer < 0 || layer >= c->d.L || !on_bound_device(c)) return ESTREAM_ERR_INVALID_ARG;
    if (c->n_groups > c->d.B) return ESTREAM_ERR_CAPACITY;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    c->trace.clear();
    // the copies must not overwrite banks that earlier work on `s` reads
    estream_status st0 = copies_after(c, s);
    if (st0 != ESTREAM_OK) return st0;
    size_t bytes = 0;
    for (int q = 0; q < c->n_groups; ++q) {
        estream_status st = fill_bank(c, layer, q, q, &bytes, c->copy_streams[q % c->d.Q]);
        if (st != ESTREAM_OK) return st;
    }
    c->stats.h2d_bytes += static_cast<double>(bytes);
    c->stats.groups_loaded += c->n_groups;
    // preload_done covers every copy stream
    for (cudaStream_t cs : c->copy_streams) {
        if (cudaEventRecord(c->copy_done, cs) != cudaSuccess ||
            cudaStreamWaitEvent(c->copy_stream, c->copy_done, 0) != cudaSuccess)
            return ESTREAM_ERR_CUDA;
    }
    if (cudaEventRecord(c->preload_done, c->copy_stream) != cudaSuccess) return ESTREAM_ERR_CUDA;
    c->preload_pending = true;
    return ESTREAM_OK;
}

estream_status estream_arena_invalidate(estream_ctx* c) {
    if (!c) return ESTREAM_ERR_NOT_BOUND;
    if (sync_copies(c) != ESTREAM_OK) return ESTREAM_ERR_CUDA;
    for (auto& b : c->banks) {
        b.layer = -1;
        b.group = -1;
    }
    return ESTREAM_OK;
}

// One layer call; with A non-null the route build also initialises Y = A.
// One layer call; with A non-null the route build also initialises Y = A.
// Routing input: `logits`, or (logits null) the router weights W_r, whose
// logits go to logits_out when given.
static estream_status prefill_impl(estream_ctx* c, int layer, const void* X, const float* logits,
                                   const void* W_r, float* logits_out, int T, int k, int renorm,
                                   const void* A, float* Y, void* cuda_stream) {
    if (!c) return ESTREAM_ERR_NOT_BOUND;
    if (layer < 0 || layer >= c->d.L || !X || (!logits && !W_r) || !Y || T < 1 || k < 1 ||
        k > c->d.E)
        return ESTREAM_ERR_INVALID_ARG;
    if (!aligned(X, 16) || !aligned(Y, 16) || (A && !aligned(A, 16))) return ESTREAM_ERR_INVALID_ARG;
    if (W_r && (c->d.wdtype == ESTREAM_F32 || !aligned(W_r, 16) || !aligned(logits_out, 4)))
        return ESTREAM_ERR_INVALID_ARG;
    if (!on_bound_device(c)) return ESTREAM_ERR_INVALID_ARG;
    if (T > c->d.T_max || k > c->d.k_max) return ESTREAM_ERR_CAPACITY;
    // this call's routed expert kernels: both tile phases, or (a test of the
    // bounded waits) the down tiles alone, whose m-block counters then never fill
    c->ffn_phases = c->ffn_down_only_next ? 2 : 3;
    c->ffn_down_only_next = false;
    c->resid_pending = false;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    const int E = c->d.E, G = c->d.G, H = c->d.H;
    c->trace.clear();
    c->stats.calls += 1;
    c->n_ffn_launch = 0;
    TimedScope total(c, s, kTTotal, layer);
    release_pipe_events(c);
    const bool trace_pipe = c->timing;
    if (trace_pipe) {
        c->pipe_t0 = pool_event(c);
        if (c->pipe_t0) cudaEventRecord(c->pipe_t0, s);
    }
    std::vector<int> ev_of(c->n_groups, -1);  // group -> index into c->pipe (timing on)
    auto new_group_events = [&](int q) -> int {
        if (!trace_pipe) return -1;
        c->pipe.push_back({pool_event(c), pool_event(c), pool_event(c), pool_event(c)});
        ev_of[q] = static_cast<int>(c->pipe.size()) - 1;
        return ev_of[q];
    };
    auto events_of = [&](int q) -> estream_ctx::GroupEvents* {
        return ev_of[q] >= 0 ? &c->pipe[ev_of[q]] : nullptr;
    };
    int n_fills = 0;  // bank fills issued by this call: fill k uses copy stream k mod Q

    if (c->preload_pending) {
        if (cudaStreamWaitEvent(s, c->preload_done, 0) != cudaSuccess) return ESTREAM_ERR_CUDA;
        c->preload_pending = false;
    }
    const bool resident = layer_resident(c, layer);
    const int R = T * k;

    // optional early fill of free banks in storage order (section 3.4)
    std::deque<int> free_banks;
    for (int b = 0; b < c->d.B; ++b) free_banks.push_back(b);
    std::vector<int> prefetched(c->n_groups, -1);
    size_t bytes = 0;
    if (!resident && c->d.schedule == ESTREAM_SCHED_PREFETCH) {
        const int npre = std::min(c->d.B, c->n_groups);
        for (int q = 0; q < npre; ++q) {
            if (layer == c->fault_layer && q == c->fault_group) break;  // handled below
            const int b = free_banks.front();
            free_banks.pop_front();
            new_group_events(q);
            estream_status st = fill_bank(c, layer, q, b, &bytes,
                                          c->copy_streams[n_fills++ % c->d.Q], events_of(q));
            if (st != ESTREAM_OK) { drain(c, s); return st; }
            prefetched[q] = b;
        }
    }

    // K1: routing + route map over logical experts in storage order (Phi = pi, P = E)
    {
        TimedScope ts(c, s, kTRoute, layer);
        NvtxRange from_x(kNvRouteFromX, layer, W_r != nullptr);   // routing from the layer input
        int launches = 0;
        const ResidualInit ri{A, c->es, Y, H};
        // The residual rows: the route build copies them on CTAs it adds beside
        // the top-k (from X: on warps beside the router tile), but rows beyond
        // what those cover wait for the top-k and hold up the grid barriers
        // (T = 4096: 100 MB on the Mixtral shape, ~30 us). A bf16 or 4-bit
        // layer then has them written by its first expert launch instead (its
        // epilogue warps are idle until their first accumulator is ready, and
        // nothing adds into Y before the down tiles).
        const bool resid_in_ffn = A && c->d.wdtype != ESTREAM_F32 &&
                                  T > route_residual_overlap_rows(T);
        c->resid_pending = resid_in_ffn;
        c->resid_A = A;
        c->resid_Y = Y;
        c->resid_T = T;
        const ResidualInit* ri_route = A && !resid_in_ffn ? &ri : nullptr;
        const int32_t* phi = c->d_perm + static_cast<size_t>(layer) * E;
        int32_t* rec_pos = c->d.deterministic ? c->rec_pos : nullptr;
        const int withhold = c->route_withhold_next ? 1 : 0;
        const cudaError_t rc =
            W_r ? route_from_x_any(X, T, H, W_r, E, k, renorm, phi, E,
                                   logits_out ? logits_out : c->logits_buf, c->topk_ids, c->alpha,
                                   c->offsets, c->rec_tok, c->rec_route, rec_pos, c->done,
                                   c->tickets, E + 3, c->route_ws, c->route_ws_bytes, s, &launches,
                                   ri_route, withhold, c->num_sms, nullptr)
                : launch_route_build(logits, T, E, k, renorm, phi, E, c->topk_ids, c->alpha,
                                     c->offsets, c->rec_tok, c->rec_route, rec_pos, c->done,
                                     c->tickets, E + 3, c->route_ws, c->route_ws_bytes, s,
                                     &launches, ri_route, withhold);
        if (rc != cudaSuccess) {
            drain(c, s);
            return ESTREAM_ERR_CUDA;
        }
        c->route_withhold_next = false;
        c->stats.launches += launches;
    }
    if (trace_pipe) {
        c->pipe_tne = pool_event(c);
        if (c->pipe_tne) cudaEventRecord(c->pipe_tne, s);
    }
    const int32_t* mblk = reinterpret_cast<const int32_t*>(
        static_cast<char*>(c->route_ws) + route_workspace_layout(T, k, E).mblk_off);
    float* Y_routed = c->d.deterministic ? nullptr : Y;

    // shared experts need no arena: they run first and overlap the first fills
    if (c->d.n_shared > 0) {
        estream_status st = run_shared(c, s, X, layer, T, c->d.deterministic ? nullptr : Y);
        if (st != ESTREAM_OK) { drain(c, s); return st; }
    }

    estream_status st = ESTREAM_OK;
    if (resident) {
        // every group sits in bank q: one launch pair over all slots, no host sync
        for (int q = 0; q < c->n_groups; ++q) trace_state(c, q, layer, q, kInUse);
        st = run_routed(c, s, X, layer, mblk, 0, E, 0, (R + kBM - 1) / kBM + E, R,
                        pair_form(c, R, E), Y_routed);
        c->stats.groups_hit += c->n_groups;
        for (int q = 0; q < c->n_groups && st == ESTREAM_OK; ++q) {
            if (cudaEventRecord(c->banks[q].released, s) != cudaSuccess) st = ESTREAM_ERR_CUDA;
            c->banks[q].release_pending = true;
            trace_state(c, q, layer, q, kAvailable);
        }
    } else {
        // routes known -> per-group counts on the host (one D2H + sync)
        if (cudaMemcpyAsync(c->h_offsets, c->offsets, sizeof(int32_t) * (E + 2),
                            cudaMemcpyDeviceToHost, s) != cudaSuccess ||
            cudaStreamSynchronize(s) != cudaSuccess) {
            drain(c, s);
            return ESTREAM_ERR_CUDA;
        }
        for (int q = 0; q < c->n_groups && st == ESTREAM_OK; ++q) {
            const int s0 = q * G, s1 = std::min(E, s0 + G);
            const int cnt = c->h_offsets[s1] - c->h_offsets[s0];
            int b = prefetched[q];
            if (cnt == 0) {
                c->stats.groups_skipped += 1;
                if (b >= 0) {  // a Ready bank with no routed work is released directly
                    trace_state(c, b, layer, q, kAvailable);
                    free_banks.push_front(b);
                    if (auto* ev = events_of(q)) {  // retired: no execution
                        cudaEventRecord(ev->s, s);
                        cudaEventRecord(ev->f, s);
                    }
                }
                continue;
            }
            if (b < 0) {
                if (layer == c->fault_layer && q == c->fault_group) {
                    drain(c, s);
                    return ESTREAM_ERR_PAGER;
                }
                b = free_banks.front();
                free_banks.pop_front();
                new_group_events(q);
                st = fill_bank(c, layer, q, b, &bytes, c->copy_streams[n_fills++ % c->d.Q],
                               events_of(q));
                if (st != ESTREAM_OK) break;
            }
            estream_ctx::GroupEvents* ev = events_of(q);
            c->stats.groups_loaded += 1;
            if (cudaStreamWaitEvent(s, c->banks[b].ready, 0) != cudaSuccess) { st = ESTREAM_ERR_CUDA; break; }
            if (ev) cudaEventRecord(ev->s, s);
            trace_state(c, b, layer, q, kInUse);
            int mt = 0, active = 0;
            for (int e = s0; e < s1; ++e) {
                const int n = c->h_offsets[e + 1] - c->h_offsets[e];
                mt += (n + kBM - 1) / kBM;
                active += n > 0 ? 1 : 0;
            }
            st = run_routed(c, s, X, layer, mblk, s0, s1 - s0, b * G, mt, cnt,
                            pair_form(c, cnt, active), Y_routed);
            if (st != ESTREAM_OK) break;
            if (ev) cudaEventRecord(ev->f, s);
            if (cudaEventRecord(c->banks[b].released, s) != cudaSuccess) { st = ESTREAM_ERR_CUDA; break; }
            c->banks[b].release_pending = true;
            trace_state(c, b, layer, q, kAvailable);
            free_banks.push_back(b);
        }
        // the caller's stream also covers the copies of this call
        if (st == ESTREAM_OK) st = stream_after_copies(c, s);
    }
    if (st != ESTREAM_OK) {
        drain(c, s);
        return st;
    }
    c->stats.h2d_bytes += static_cast<double>(bytes);
    if (c->resid_pending) {
        // no expert launch took the residual rows (no routed group had work)
        c->resid_pending = false;
        if (launch_residual_rows(A, c->es, Y, T, H, s) != cudaSuccess) {
            drain(c, s);
            return ESTREAM_ERR_CUDA;
        }
        c->stats.launches += 1;
    }
    if (c->d.deterministic) {
        TimedScope ts(c, s, kTCombine, layer);
        if (launch_combine(c->out_rows, c->rec_pos, T, k, H, c->out_shared, c->d.n_shared, Y, s) !=
            cudaSuccess) {
            drain(c, s);
            return ESTREAM_ERR_CUDA;
        }
        c->stats.launches += 1;
    }
    return ESTREAM_OK;
}

estream_status estream_moe_layer_prefill(estream_ctx* c, int layer, const void* X,
                                         const float* logits, int T, int k, int renorm, float* Y,
                                         void* cuda_stream) {
    if (!logits) return c ? ESTREAM_ERR_INVALID_ARG : ESTREAM_ERR_NOT_BOUND;
    return prefill_impl(c, layer, X, logits, nullptr, nullptr, T, k, renorm, nullptr, Y, cuda_stream);
}

estream_status estream_moe_layer_prefill_residual(estream_ctx* c, int layer, const void* X,
                                                  const float* logits, int T, int k, int renorm,
                                                  const void* A, float* Y, void* cuda_stream) {
    if (!c) return ESTREAM_ERR_NOT_BOUND;
    if (!A) return ESTREAM_ERR_INVALID_ARG;
    if (!logits) return ESTREAM_ERR_INVALID_ARG;
    return prefill_impl(c, layer, X, logits, nullptr, nullptr, T, k, renorm, A, Y, cuda_stream);
}

estream_status estream_moe_layer_prefill_from_x(estream_ctx* c, int layer, const void* X,
                                                const void* W_r, int T, int k, int renorm,
                                                const void* A, float* Y, float* logits_out,
                                                void* cuda_stream) {
    if (!c) return ESTREAM_ERR_NOT_BOUND;
    if (!W_r) return ESTREAM_ERR_INVALID_ARG;
    return prefill_impl(c, layer, X, nullptr, W_r, logits_out, T, k, renorm, A, Y, cuda_stream);
}

estream_status estream_set_timing(estream_ctx* c, int on) {
    if (!c) return ESTREAM_ERR_NOT_BOUND;
    c->timing = on != 0;
    return ESTREAM_OK;
}

estream_status estream_reset_stats(estream_ctx* c) {
    if (!c) return ESTREAM_ERR_NOT_BOUND;
    if (sync_copies(c) != ESTREAM_OK) return ESTREAM_ERR_CUDA;
    for (auto& t : c->timed) {
        cudaEventSynchronize(t.b);
        c->event_pool.push_back(t.a);
        c->event_pool.push_back(t.b);
    }
    c->timed.clear();
    c->stats = estream_stats{};
    return ESTREAM_OK;
}

estream_status estream_last_stats(estream_ctx* c, estream_stats* out) {
    if (!c) return ESTREAM_ERR_NOT_BOUND;
    if (!out) return ESTREAM_ERR_INVALID_ARG;
    estream_status st = ESTREAM_OK;
    for (auto& t : c->timed) {
        float ms = 0.0f;
        if (cudaEventSynchronize(t.b) != cudaSuccess ||
            cudaEventElapsedTime(&ms, t.a, t.b) != cudaSuccess) {
            st = ESTREAM_ERR_CUDA;
            ms = 0.0f;
        }
        switch (t.kind) {
            case kTRoute: c->stats.ms_route += ms; break;
            case kTFfn: c->stats.ms_ffn += ms; break;
            case kTShared: c->stats.ms_shared += ms; break;
            case kTCombine: c->stats.ms_combine += ms; break;
            case kTTotal: c->stats.ms_total += ms; break;
            case kTIo: c->stats.ms_io_busy += ms; break;
        }
        c->event_pool.push_back(t.a);
        c->event_pool.push_back(t.b);
    }
    c->timed.clear();
    *out = c->stats;
    // overlap of loading and execution over the calls since the last reset
    const double t_io = out->ms_io_busy, t_total = out->ms_total;
    const double t_exec = out->ms_route + out->ms_ffn + out->ms_shared + out->ms_combine;
    auto clamp01 = [](double x) { return x < 0.0 ? 0.0 : (x > 1.0 ? 1.0 : x); };
    out->hidden_fraction = t_io > 0.0 ? clamp01((t_io + t_exec - t_total) / t_io) : 0.0;
    out->bubble_rate = t_total > 0.0 ? clamp01(1.0 - std::max(t_io, t_exec) / t_total) : 0.0;
    return st;
}

estream_status estream_poison_workspace(estream_ctx* c, void* cuda_stream) {
    if (!c) return ESTREAM_ERR_NOT_BOUND;
    if (!on_bound_device(c)) return ESTREAM_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    char* call = c->ws + c->ws_call_off;
    if (cudaMemsetAsync(call, 0xff, c->ws_bytes - c->ws_call_off, s) != cudaSuccess)
        return ESTREAM_ERR_CUDA;
    struct { int32_t* p; size_t n; } counters[3] = {
        {c->done, c->n_done}, {c->sh_done, c->n_sh_done}, {c->tickets, c->n_tickets}};
    for (const auto& r : counters)
        if (r.p && r.n && cudaMemsetAsync(r.p, 0x7f, sizeof(int32_t) * r.n, s) != cudaSuccess)
            return ESTREAM_ERR_CUDA;
    return ESTREAM_OK;
}

estream_status estream_get_device_error(estream_ctx* c) {
    if (!c) return ESTREAM_ERR_NOT_BOUND;
    if (sync_copies(c) != ESTREAM_OK) return ESTREAM_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return ESTREAM_ERR_CUDA;
    // the context's word (expert kernels, sticky until read) and the route
    // build's own word (the latest call's routing)
    int* words[2] = {c->dev_err, reinterpret_cast<int*>(static_cast<char*>(c->route_ws) +
                                                        route_workspace_layout(0, 1, 0).err_off)};
    int first = kDevErrNone;
    for (int* w : words) {
        int host = 0;
        if (cudaMemcpy(&host, w, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
            return ESTREAM_ERR_CUDA;
        if (host == kDevErrNone) continue;
        if (first == kDevErrNone) first = host;
        if (cudaMemset(w, 0, sizeof(int)) != cudaSuccess) return ESTREAM_ERR_CUDA;
    }
    if (first == kDevErrNone) return ESTREAM_OK;
    return first == kDevErrTimeout ? ESTREAM_ERR_TIMEOUT : ESTREAM_ERR_DEVICE;
}

estream_status estream_residency_trace(estream_ctx* c, int32_t* out, int cap, int* n) {
    if (!c) return ESTREAM_ERR_NOT_BOUND;
    if (!n || cap < 0 || (cap > 0 && !out)) return ESTREAM_ERR_INVALID_ARG;
    const int events = static_cast<int>(c->trace.size() / 4);
    const int m = std::min(events, cap);
    if (m > 0) std::memcpy(out, c->trace.data(), sizeof(int32_t) * 4 * m);
    *n = events;
    return ESTREAM_OK;
}

estream_status estream_pipeline_trace(estream_ctx* c, double* adsf, int cap, int* n, double* t_ne) {
    if (!c) return ESTREAM_ERR_NOT_BOUND;
    if (!n || cap < 0 || (cap > 0 && !adsf)) return ESTREAM_ERR_INVALID_ARG;
    *n = 0;
    if (!c->pipe_t0) return ESTREAM_OK;
    auto since = [&](cudaEvent_t e, double* out) {
        float ms = 0.0f;
        if (!e || cudaEventSynchronize(e) != cudaSuccess ||
            cudaEventElapsedTime(&ms, c->pipe_t0, e) != cudaSuccess)
            return false;
        *out = ms;
        return true;
    };
    if (t_ne && !since(c->pipe_tne, t_ne)) return ESTREAM_ERR_CUDA;
    const int m = std::min(cap, static_cast<int>(c->pipe.size()));
    for (int k = 0; k < m; ++k) {
        const auto& g = c->pipe[k];
        if (!since(g.a, adsf + 4 * k) || !since(g.d, adsf + 4 * k + 1) ||
            !since(g.s, adsf + 4 * k + 2) || !since(g.f, adsf + 4 * k + 3))
            return ESTREAM_ERR_CUDA;
    }
    *n = static_cast<int>(c->pipe.size());
    return ESTREAM_OK;
}

estream_status estream_inject_expert_timeout(estream_ctx* c) {
    if (!c) return ESTREAM_ERR_NOT_BOUND;
    c->ffn_down_only_next = true;
    return ESTREAM_OK;
}

estream_status estream_inject_route_timeout(estream_ctx* c) {
    if (!c) return ESTREAM_ERR_NOT_BOUND;
    c->route_withhold_next = true;
    return ESTREAM_OK;
}

estream_status estream_inject_pager_fault(estream_ctx* c, int layer, int group) {
    if (!c) return ESTREAM_ERR_NOT_BOUND;
    c->fault_layer = group < 0 ? -1 : layer;
    c->fault_group = group < 0 ? -1 : group;
    return ESTREAM_OK;
}

void estream_unbind(estream_ctx* c) {
    if (!c) return;
    for (cudaStream_t cs : c->copy_streams)
        if (cs) cudaStreamSynchronize(cs);
    release_pipe_events(c);
    for (auto& t : c->timed) {
        cudaEventSynchronize(t.b);
        cudaEventDestroy(t.a);
        cudaEventDestroy(t.b);
    }
    for (cudaEvent_t e : c->event_pool) cudaEventDestroy(e);
    for (auto& b : c->banks) {
        if (b.ready) cudaEventSynchronize(b.ready), cudaEventDestroy(b.ready);
        if (b.released) cudaEventSynchronize(b.released), cudaEventDestroy(b.released);
    }
    if (c->copy_done) cudaEventDestroy(c->copy_done);
    if (c->preload_done) cudaEventDestroy(c->preload_done);
    for (cudaStream_t cs : c->copy_streams)
        if (cs) cudaStreamDestroy(cs);
    if (c->h_offsets) cudaFreeHost(c->h_offsets);
    if (c->ws) {
        cudaDeviceSynchronize();
        cudaFree(c->ws);
    }
    delete c;
    // an error of the teardown itself (e.g. an event still referenced by a
    // caller's CUDA graph) must not surface in the caller's next CUDA call
    (void)cudaGetLastError();
}

estream_status estream_cast_f32_bf16(const float* src, void* dst, size_t n, void* cuda_stream) {
    if ((!src || !dst) && n > 0) return ESTREAM_ERR_INVALID_ARG;
    return launch_cast_f32_bf16(src, dst, n, static_cast<cudaStream_t>(cuda_stream)) == cudaSuccess
               ? ESTREAM_OK
               : ESTREAM_ERR_CUDA;
}

}  // extern "C"
