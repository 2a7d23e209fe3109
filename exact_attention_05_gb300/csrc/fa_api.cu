// fa_api.cu -- host side of the C ABI declared in include/fa.h: argument
// checks (all of them before any CUDA call), per-device state (architecture
// check, device status word, decode workspaces), TMA tensor-map encoding and
// the kernel launches.
//
// The status word that every kernel's bounded waits report to is static
// device memory (g_status_word below): each device that loads the module
// holds its own, zero at load, and finding its address allocates nothing, so
// the allocation-free decode shares it with every other entry point.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include <cuda.h>
#include <cuda_runtime.h>

#include "fa.h"
#include "fa_internal.h"

#define FA_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

constexpr unsigned long long kDefaultTimeoutNs = 2000000000ull;
std::atomic<unsigned long long> g_timeout_ns{kDefaultTimeoutNs};

// One status word per device: the low byte FA_DEV_TIMEOUT (or FA_DEV_LAYOUT),
// the next byte the wait site; zero when nothing went wrong.
static __device__ int g_status_word;

struct Workspace {
    void* ptr = nullptr;
    size_t bytes = 0;
    int* tickets = nullptr;  // zero between calls (the single-launch decode resets what it uses)
    size_t nticket = 0;
};

// Copy streams and events of fa_fwd_host for one caller stream: chunk c's
// inputs go in on `in` while chunk c-1 computes on the caller's stream and chunk
// c-2's outputs come back on `out`; slot c % 2 of the device staging is reused
// once chunk c-2's outputs are copied out.
struct HostPipe {
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t start = nullptr;
    cudaEvent_t landed[2] = {nullptr, nullptr}, computed[2] = {nullptr, nullptr},
                copied[2] = {nullptr, nullptr};
    bool ready = false;
};

struct DeviceState {
    bool checked = false;
    bool supported = false;
    int* status = nullptr;
    std::map<cudaStream_t, Workspace> workspaces;
    std::map<cudaStream_t, HostPipe> pipes;
};

std::mutex g_mu;
std::map<int, DeviceState> g_devices;

using fa::EncodeTiledFn;
EncodeTiledFn g_encode_driver = nullptr;  // cuTensorMapEncodeTiled

// Tensor maps already encoded, keyed by every argument of the encode call.
// A call's tensors are usually the previous call's (the same buffers, one
// step later), so each map is encoded once and then copied.  Bounded: the
// cache is emptied when it reaches kMaxCachedMaps entries.
struct MapKey {
    uint64_t v[24];
    bool operator<(const MapKey& o) const { return std::memcmp(v, o.v, sizeof(v)) < 0; }
};
constexpr size_t kMaxCachedMaps = 1024;
std::mutex g_map_mu;
std::map<MapKey, CUtensorMap> g_maps;

CUresult encode_tiled_cached(CUtensorMap* map, CUtensorMapDataType dtype, cuuint32_t rank,
                             void* base, const cuuint64_t* dims, const cuuint64_t* strides,
                             const cuuint32_t* box, const cuuint32_t* estr,
                             CUtensorMapInterleave il, CUtensorMapSwizzle sw,
                             CUtensorMapL2promotion l2, CUtensorMapFloatOOBfill oob) {
    if (rank < 1 || rank > 5) return g_encode_driver(map, dtype, rank, base, dims, strides, box,
                                                     estr, il, sw, l2, oob);
    MapKey key{};
    size_t n = 0;
    key.v[n++] = reinterpret_cast<uint64_t>(base);
    key.v[n++] = (uint64_t)dtype | ((uint64_t)rank << 8) | ((uint64_t)il << 16) |
                 ((uint64_t)sw << 24) | ((uint64_t)l2 << 32) | ((uint64_t)oob << 40);
    for (cuuint32_t i = 0; i < rank; ++i) key.v[n++] = dims[i];
    for (cuuint32_t i = 0; i + 1 < rank; ++i) key.v[n++] = strides[i];
    for (cuuint32_t i = 0; i < rank; ++i) key.v[n++] = ((uint64_t)box[i] << 32) | estr[i];
    {
        std::lock_guard<std::mutex> lock(g_map_mu);
        auto it = g_maps.find(key);
        if (it != g_maps.end()) {
            *map = it->second;
            return CUDA_SUCCESS;
        }
    }
    const CUresult r = g_encode_driver(map, dtype, rank, base, dims, strides, box, estr, il, sw,
                                       l2, oob);
    if (r == CUDA_SUCCESS) {
        std::lock_guard<std::mutex> lock(g_map_mu);
        if (g_maps.size() >= kMaxCachedMaps) g_maps.clear();
        g_maps.emplace(key, *map);
    }
    return r;
}

EncodeTiledFn g_encode = nullptr;  // encode_tiled_cached once the driver entry point is known

constexpr uint64_t kMaxElements = 1ull << 39;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Pure argument checks shared by both operations; no CUDA call.
fa_status check_args(const void* q, const void* k, const void* v, const void* o, const float* lse,
                     int B, int Hq, int Hkv, int N, int M, int d, float scale, int dtype) {
    if (!q || !k || !v || !o) return FA_ERR_INVALID_ARG;
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || N <= 0 || M <= 0 || d <= 0) return FA_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return FA_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !std::isfinite(scale)) return FA_ERR_INVALID_ARG;
    if (dtype != FA_FP16 && dtype != FA_BF16) return FA_ERR_UNSUPPORTED;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16))
        return FA_ERR_INVALID_ARG;
    if (lse && !aligned(lse, 4)) return FA_ERR_INVALID_ARG;
    if ((uint64_t)B * N * Hq * d >= kMaxElements) return FA_ERR_INVALID_ARG;
    if ((uint64_t)B * M * Hkv * d >= kMaxElements) return FA_ERR_INVALID_ARG;
    return FA_OK;
}

// Current device's state; checks the architecture and looks up the status word once.
fa_status device_state(DeviceState** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState& st = g_devices[dev];
    if (!st.checked) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return FA_ERR_CUDA;
        st.supported = (major == 10 && minor == 3);
        if (st.supported) {
            // the host-side name of the word is not its device address: look the
            // address up on this device (with it current)
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess || p == nullptr)
                return FA_ERR_CUDA;
            st.status = static_cast<int*>(p);
        }
        st.checked = true;
    }
    if (!st.supported) return FA_ERR_UNSUPPORTED;
    if (g_encode == nullptr) {
        cudaDriverEntryPointQueryResult q{};
        void* fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || fn == nullptr)
            return FA_ERR_CUDA;
        g_encode_driver = reinterpret_cast<EncodeTiledFn>(fn);
        g_encode = encode_tiled_cached;
    }
    *out = &st;
    return FA_OK;
}

// 4-D map over a [batch, seq, heads, d] tensor: dims innermost first
// {d, heads, seq, batch}; the box is box_d x 1 x box_rows x 1.
fa_status encode_map(CUtensorMap* map, const void* base, int dtype, int d, int heads, int seq,
                     int batch, int box_d, int box_rows, bool swizzle128) {
    const cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)seq,
                                (cuuint64_t)batch};
    const cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)heads * d * 2,
                                   (cuuint64_t)seq * heads * d * 2};
    const cuuint32_t box[4] = {(cuuint32_t)box_d, 1, (cuuint32_t)box_rows, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUresult r = g_encode(
        map, dtype == FA_FP16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
        4, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
        swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

// Workspace of at least `bytes` for (device, stream).
fa_status workspace(DeviceState* st, cudaStream_t stream, size_t bytes, void** out) {
    std::lock_guard<std::mutex> lock(g_mu);
    Workspace& w = st->workspaces[stream];
    if (w.bytes < bytes) {
        if (w.ptr != nullptr) {
            // the old buffer may still be read by work in flight on this stream
            if (cudaStreamSynchronize(stream) != cudaSuccess) return FA_ERR_CUDA;
            cudaFree(w.ptr);
            w.ptr = nullptr;
            w.bytes = 0;
        }
        size_t want = bytes + bytes / 4;
        want = (want + (1u << 20) - 1) & ~size_t((1u << 20) - 1);
        if (cudaMalloc(&w.ptr, want) != cudaSuccess) {
            (void)cudaGetLastError();
            w.ptr = nullptr;
            return FA_ERR_NO_MEMORY;
        }
        w.bytes = want;
    }
    *out = w.ptr;
    return FA_OK;
}

// Ticket counters of at least `count` ints for (device, stream), zero on return.
fa_status tickets(DeviceState* st, cudaStream_t stream, size_t count, int** out) {
    std::lock_guard<std::mutex> lock(g_mu);
    Workspace& w = st->workspaces[stream];
    if (w.nticket < count) {
        if (w.tickets != nullptr) {
            if (cudaStreamSynchronize(stream) != cudaSuccess) return FA_ERR_CUDA;
            cudaFree(w.tickets);
            w.tickets = nullptr;
            w.nticket = 0;
        }
        const size_t want = (count + 4095) & ~size_t(4095);
        if (cudaMalloc(&w.tickets, want * sizeof(int)) != cudaSuccess) {
            (void)cudaGetLastError();
            w.tickets = nullptr;
            return FA_ERR_NO_MEMORY;
        }
        if (cudaMemsetAsync(w.tickets, 0, want * sizeof(int), stream) != cudaSuccess)
            return FA_ERR_CUDA;
        w.nticket = want;
    }
    *out = w.tickets;
    return FA_OK;
}

fa_status from_cuda(cudaError_t e) { return e == cudaSuccess ? FA_OK : FA_ERR_CUDA; }

// Workspace and the common fields of a two-kernel decode launch over M keys.
fa_status decode_setup(DeviceState* st, cudaStream_t stream, const void* q, void* o, float* lse,
                       int B, int Hq, int Hkv, int M, int d, int chunk, float scale,
                       fa::DecodeArgs* a) {
    const int nc = (int)(((long long)M + chunk - 1) / chunk);
    const size_t part_elems = (size_t)B * Hq * nc * d;
    const size_t bytes = (part_elems + (size_t)B * Hq * nc) * sizeof(float);
    void* ws = nullptr;
    const fa_status s = workspace(st, stream, bytes, &ws);
    if (s != FA_OK) return s;
    *a = fa::DecodeArgs{};
    a->q = q;
    a->o = o;
    a->lse = lse;
    a->o_part = static_cast<float*>(ws);
    a->lse_part = static_cast<float*>(ws) + part_elems;
    a->B = B;
    a->Hq = Hq;
    a->Hkv = Hkv;
    a->M = M;
    a->chunk = chunk;
    a->nc = nc;
    a->scale_log2 = (float)((double)scale * 1.4426950408889634);
    a->status = st->status;
    a->timeout_ns = g_timeout_ns.load();
    return FA_OK;
}

}  // namespace

namespace fa {

int* status_word_current_device() {
    DeviceState* st = nullptr;
    return device_state(&st) == FA_OK ? st->status : nullptr;
}

unsigned long long wait_timeout_ns() { return g_timeout_ns.load(); }

EncodeTiledFn tensor_map_encoder() {
    DeviceState* st = nullptr;
    return device_state(&st) == FA_OK ? g_encode : nullptr;
}

}  // namespace fa

FA_EXPORT fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                           int Hq, int Hkv, int N, int M, int d, int causal, float scale,
                           fa_dtype dtype, fa_stream_t stream) {
    fa_status s = check_args(q, k, v, o, lse, B, Hq, Hkv, N, M, d, scale, (int)dtype);
    if (s != FA_OK) return s;
    if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
    const long long n_qtiles = (N + fa::kPrefillTile - 1) / fa::kPrefillTile;
    if (n_qtiles * B * Hq > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
    DeviceState* st = nullptr;
    if ((s = device_state(&st)) != FA_OK) return s;
    CUtensorMap tq, tk, tv, to;
    if ((s = encode_map(&tq, q, dtype, d, Hq, N, B, 64, fa::kPrefillTile, true)) != FA_OK) return s;
    if ((s = encode_map(&tk, k, dtype, d, Hkv, M, B, 64, fa::kPrefillTile, true)) != FA_OK) return s;
    if ((s = encode_map(&tv, v, dtype, d, Hkv, M, B, 64, fa::kPrefillTile, true)) != FA_OK) return s;
    if ((s = encode_map(&to, o, dtype, d, Hq, N, B, 64, fa::kPrefillTile, true)) != FA_OK) return s;
    fa::PrefillArgs a{};
    a.o = o;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.N = N;
    a.M = M;
    a.causal = causal;
    a.n_qtiles = (int)n_qtiles;
    a.scale_log2 = (float)((double)scale * 1.4426950408889634);
    a.lse = lse;
    a.status = st->status;
    a.timeout_ns = g_timeout_ns.load();
    return from_cuda(fa::launch_prefill(tq, tk, tv, to, a, d, (int)dtype, (cudaStream_t)stream));
}

namespace {

// The copy streams and events of fa_fwd_host for (current device, stream).
fa_status host_pipe(DeviceState* st, cudaStream_t stream, HostPipe** out) {
    std::lock_guard<std::mutex> lock(g_mu);
    HostPipe& p = st->pipes[stream];
    if (!p.ready) {
        if (cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking) != cudaSuccess ||
            cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&p.start, cudaEventDisableTiming) != cudaSuccess)
            return FA_ERR_CUDA;
        for (int i = 0; i < 2; ++i)
            if (cudaEventCreateWithFlags(&p.landed[i], cudaEventDisableTiming) != cudaSuccess ||
                cudaEventCreateWithFlags(&p.computed[i], cudaEventDisableTiming) != cudaSuccess ||
                cudaEventCreateWithFlags(&p.copied[i], cudaEventDisableTiming) != cudaSuccess)
                return FA_ERR_CUDA;
        p.ready = true;
    }
    *out = &p;
    return FA_OK;
}

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

FA_EXPORT fa_status fa_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse,
                                int B, int Hq, int Hkv, int N, int M, int d, int causal,
                                float scale, fa_dtype dtype, fa_stream_t stream) {
    fa_status s = check_args(q, k, v, o, lse, B, Hq, Hkv, N, M, d, scale, (int)dtype);
    if (s != FA_OK) return s;
    if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
    DeviceState* st = nullptr;
    if ((s = device_state(&st)) != FA_OK) return s;
    const cudaStream_t cs = (cudaStream_t)stream;
    HostPipe* p = nullptr;
    if ((s = host_pipe(st, cs, &p)) != FA_OK) return s;
    // Chunks of (b, group of kv heads with their query heads): one per batch entry
    // when B >= 4, else about four in all, so that each launch still fills the GPU
    // with CTAs while the copies of its neighbours run.
    const int g = Hq / Hkv;
    int per_b = B >= 4 ? 1 : (4 + B - 1) / B;
    if (per_b > Hkv) per_b = Hkv;
    const int hk_max = (Hkv + per_b - 1) / per_b;
    const int hq_max = hk_max * g;
    const size_t esz = 2;
    const size_t row_q = (size_t)Hq * d * esz, row_kv = (size_t)Hkv * d * esz;
    // device staging, two slots: q, o [N, hq, d]; k, v [M, hk, d]; lse [hq, N]
    const size_t bq = round256((size_t)N * hq_max * d * esz);
    const size_t bkv = round256((size_t)M * hk_max * d * esz);
    const size_t bl = round256((size_t)hq_max * N * sizeof(float));
    const size_t slot_bytes = 2 * bq + 2 * bkv + bl;
    void* ws = nullptr;
    if ((s = workspace(st, cs, 2 * slot_bytes, &ws)) != FA_OK) return s;
    auto err = [](cudaError_t e) { return e == cudaSuccess ? FA_OK : FA_ERR_CUDA; };
    if ((s = err(cudaEventRecord(p->start, cs))) != FA_OK) return s;
    if ((s = err(cudaStreamWaitEvent(p->in, p->start, 0))) != FA_OK) return s;
    if ((s = err(cudaStreamWaitEvent(p->out, p->start, 0))) != FA_OK) return s;
    int c = 0;
    for (int b = 0; b < B; ++b) {
        for (int kv0 = 0; kv0 < Hkv; kv0 += hk_max, ++c) {
            const int hk = Hkv - kv0 < hk_max ? Hkv - kv0 : hk_max;
            const int hq0 = kv0 * g, hq = hk * g;
            const int slot = c & 1;
            uint8_t* base = static_cast<uint8_t*>(ws) + slot * slot_bytes;
            uint8_t* qd = base;
            uint8_t* od = qd + bq;
            uint8_t* kd = od + bq;
            uint8_t* vd = kd + bkv;
            float* ld = reinterpret_cast<float*>(vd + bkv);
            // the slot's previous chunk must be copied out (it was computed before that)
            if (c >= 2 && (s = err(cudaStreamWaitEvent(p->in, p->copied[slot], 0))) != FA_OK)
                return s;
            const uint8_t* qh = static_cast<const uint8_t*>(q) + ((size_t)b * N * Hq + hq0) * d * esz;
            const uint8_t* kh = static_cast<const uint8_t*>(k) + ((size_t)b * M * Hkv + kv0) * d * esz;
            const uint8_t* vh = static_cast<const uint8_t*>(v) + ((size_t)b * M * Hkv + kv0) * d * esz;
            const size_t wq = (size_t)hq * d * esz, wkv = (size_t)hk * d * esz;
            if ((s = err(cudaMemcpy2DAsync(qd, wq, qh, row_q, wq, N, cudaMemcpyHostToDevice, p->in))) != FA_OK ||
                (s = err(cudaMemcpy2DAsync(kd, wkv, kh, row_kv, wkv, M, cudaMemcpyHostToDevice, p->in))) != FA_OK ||
                (s = err(cudaMemcpy2DAsync(vd, wkv, vh, row_kv, wkv, M, cudaMemcpyHostToDevice, p->in))) != FA_OK ||
                (s = err(cudaEventRecord(p->landed[slot], p->in))) != FA_OK ||
                (s = err(cudaStreamWaitEvent(cs, p->landed[slot], 0))) != FA_OK)
                return s;
            if ((s = fa_fwd(qd, kd, vd, od, lse ? ld : nullptr, 1, hq, hk, N, M, d, causal, scale,
                            dtype, stream)) != FA_OK)
                return s;
            if ((s = err(cudaEventRecord(p->computed[slot], cs))) != FA_OK ||
                (s = err(cudaStreamWaitEvent(p->out, p->computed[slot], 0))) != FA_OK)
                return s;
            uint8_t* oh = static_cast<uint8_t*>(o) + ((size_t)b * N * Hq + hq0) * d * esz;
            if ((s = err(cudaMemcpy2DAsync(oh, row_q, od, wq, wq, N, cudaMemcpyDeviceToHost, p->out))) != FA_OK)
                return s;
            if (lse && (s = err(cudaMemcpyAsync(lse + ((size_t)b * Hq + hq0) * N, ld,
                                                (size_t)hq * N * sizeof(float), cudaMemcpyDeviceToHost,
                                                p->out))) != FA_OK)
                return s;
            if ((s = err(cudaEventRecord(p->copied[slot], p->out))) != FA_OK) return s;
        }
    }
    // the caller's stream is ordered after every copy out
    for (int i = 0; i < 2 && i < c; ++i)
        if ((s = err(cudaStreamWaitEvent(cs, p->copied[i], 0))) != FA_OK) return s;
    return FA_OK;
}

FA_EXPORT fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o,
                           const float* lse, const void* dout, void* dq, void* dk, void* dv, int B,
                           int Hq, int Hkv, int N, int M, int d, int causal, float scale,
                           fa_dtype dtype, fa_stream_t stream) {
    fa_status s = check_args(q, k, v, o, lse, B, Hq, Hkv, N, M, d, scale, (int)dtype);
    if (s != FA_OK) return s;
    if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
    if (!lse || !dout || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
    if (!aligned(dout, 16) || !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16))
        return FA_ERR_INVALID_ARG;
    const long long nkt = ((long long)M + fa::kPrefillTile - 1) / fa::kPrefillTile;
    if (nkt * B * Hkv > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
    DeviceState* st = nullptr;
    if ((s = device_state(&st)) != FA_OK) return s;
    const size_t acc_elems = (size_t)B * N * Hq * d;
    const int n_qtiles = (N + fa::kPrefillTile - 1) / fa::kPrefillTile;
    const size_t pack_elems = (size_t)B * Hq * n_qtiles * 2 * fa::kPrefillTile;
    const size_t bytes = (acc_elems + pack_elems) * sizeof(float);
    void* ws = nullptr;
    if ((s = workspace(st, (cudaStream_t)stream, bytes, &ws)) != FA_OK) return s;
    CUtensorMap tq, tk, tv, tdo;
    if ((s = encode_map(&tq, q, dtype, d, Hq, N, B, 64, fa::kPrefillTile, true)) != FA_OK) return s;
    if ((s = encode_map(&tk, k, dtype, d, Hkv, M, B, 64, fa::kPrefillTile, true)) != FA_OK) return s;
    if ((s = encode_map(&tv, v, dtype, d, Hkv, M, B, 64, fa::kPrefillTile, true)) != FA_OK) return s;
    if ((s = encode_map(&tdo, dout, dtype, d, Hq, N, B, 64, fa::kPrefillTile, true)) != FA_OK)
        return s;
    // fp32 dQ accumulator [B, N, Hq, d], the target of the kernel's bulk reductions
    CUtensorMap tdq;
    {
        const cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)Hq, (cuuint64_t)N, (cuuint64_t)B};
        const cuuint64_t strides[3] = {(cuuint64_t)d * 4, (cuuint64_t)Hq * d * 4,
                                       (cuuint64_t)N * Hq * d * 4};
        const cuuint32_t box[4] = {32, 1, (cuuint32_t)fa::kPrefillTile, 1};
        const cuuint32_t estr[4] = {1, 1, 1, 1};
        if (g_encode(&tdq, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, ws, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return FA_ERR_CUDA;
    }
    fa::BackwardArgs a{};
    a.o = o;
    a.dout = dout;
    a.lse = lse;
    a.dq_acc = static_cast<float*>(ws);
    a.pack = static_cast<float*>(ws) + acc_elems;
    a.dq = dq;
    a.dk = dk;
    a.dv = dv;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.N = N;
    a.M = M;
    a.causal = causal;
    a.n_qtiles = n_qtiles;
    a.n_ktiles = (int)nkt;
    a.scale = scale;
    a.scale_log2 = (float)((double)scale * 1.4426950408889634);
    a.status = st->status;
    a.timeout_ns = g_timeout_ns.load();
    return from_cuda(
        fa::launch_backward(tq, tk, tv, tdo, tdq, a, d, (int)dtype, (cudaStream_t)stream));
}

FA_EXPORT fa_status fa_decode(const void* q, const void* k, const void* v, void* o, float* lse,
                              int B, int Hq, int Hkv, int M, int d, int chunk, float scale,
                              fa_dtype dtype, fa_stream_t stream) {
    fa_status s = check_args(q, k, v, o, lse, B, Hq, Hkv, 1, M, d, scale, (int)dtype);
    if (s != FA_OK) return s;
    if (chunk <= 0) return FA_ERR_INVALID_ARG;
    if (((long long)M + chunk - 1) / chunk * B * Hkv > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
    const int nc = (int)(((long long)M + chunk - 1) / chunk);
    DeviceState* st = nullptr;
    if ((s = device_state(&st)) != FA_OK) return s;
    const size_t part_elems = (size_t)B * Hq * nc * d;
    const size_t bytes = (part_elems + (size_t)B * Hq * nc) * sizeof(float);
    void* ws = nullptr;
    if ((s = workspace(st, (cudaStream_t)stream, bytes, &ws)) != FA_OK) return s;
    CUtensorMap tk, tv;
    if (!fa::encode_decode_maps(g_encode, k, v, dtype, d, Hkv, M, B, &tk, &tv)) return FA_ERR_CUDA;
    fa::DecodeArgs a{};
    a.q = q;
    a.o = o;
    a.lse = lse;
    a.o_part = static_cast<float*>(ws);
    a.lse_part = static_cast<float*>(ws) + part_elems;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.M = M;
    a.chunk = chunk;
    a.nc = nc;
    a.scale_log2 = (float)((double)scale * 1.4426950408889634);
    a.status = st->status;
    a.timeout_ns = g_timeout_ns.load();
    return from_cuda(fa::launch_decode(tk, tv, a, d, (int)dtype, (cudaStream_t)stream));
}

FA_EXPORT fa_status fa_decode_fused(const void* q, const void* k, const void* v, void* o,
                                    float* lse, int B, int Hq, int Hkv, int M, int d, int chunk,
                                    float scale, fa_dtype dtype, fa_stream_t stream) {
    fa_status s = check_args(q, k, v, o, lse, B, Hq, Hkv, 1, M, d, scale, (int)dtype);
    if (s != FA_OK) return s;
    if (chunk <= 0) return FA_ERR_INVALID_ARG;
    const long long nc = ((long long)M + chunk - 1) / chunk;
    if (nc * B * Hkv > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
    DeviceState* st = nullptr;
    if ((s = device_state(&st)) != FA_OK) return s;
    // chunk partials, then the stripe partials (at most one stripe per chunk);
    // the LSE blocks are padded to 64 floats so that every row block starts on
    // a 256-byte boundary (the kernel stores the rows as float4)
    const size_t part_elems = (size_t)B * Hq * nc * d;
    const size_t lse_elems = ((size_t)B * Hq * nc + 63) & ~size_t(63);
    const size_t floats = 2 * (part_elems + lse_elems);
    void* ws = nullptr;
    if ((s = workspace(st, (cudaStream_t)stream, floats * sizeof(float), &ws)) != FA_OK) return s;
    int* tk_counts = nullptr;
    if ((s = tickets(st, (cudaStream_t)stream, (size_t)B * Hkv, &tk_counts)) != FA_OK) return s;
    CUtensorMap tk, tv;
    if (!fa::encode_decode_maps(g_encode, k, v, dtype, d, Hkv, M, B, &tk, &tv)) return FA_ERR_CUDA;
    fa::DecodeArgs a{};
    float* f = static_cast<float*>(ws);
    a.q = q;
    a.o = o;
    a.lse = lse;
    a.o_part = f;
    a.lse_part = f + part_elems;
    a.g_o = a.lse_part + lse_elems;
    a.g_lse = a.g_o + part_elems;
    a.tickets = tk_counts;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.M = M;
    a.chunk = chunk;
    a.nc = (int)nc;
    a.scale_log2 = (float)((double)scale * 1.4426950408889634);
    a.status = st->status;
    a.timeout_ns = g_timeout_ns.load();
    return from_cuda(fa::launch_decode_fused(tk, tv, a, d, (int)dtype, (cudaStream_t)stream));
}

FA_EXPORT fa_status fa_decode_fp8(const void* q, const void* k8, const void* v8,
                                  const float* k_scale, const float* v_scale, void* o, float* lse,
                                  int B, int Hq, int Hkv, int M, int d, int chunk, float scale,
                                  fa_dtype dtype, fa_stream_t stream) {
    fa_status s = check_args(q, k8, v8, o, lse, B, Hq, Hkv, 1, M, d, scale, (int)dtype);
    if (s != FA_OK) return s;
    if (!k_scale || !v_scale || !aligned(k_scale, 4) || !aligned(v_scale, 4))
        return FA_ERR_INVALID_ARG;
    if (chunk <= 0) return FA_ERR_INVALID_ARG;
    if (((long long)M + chunk - 1) / chunk * B * Hkv > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
    DeviceState* st = nullptr;
    if ((s = device_state(&st)) != FA_OK) return s;
    fa::DecodeArgs a;
    if ((s = decode_setup(st, (cudaStream_t)stream, q, o, lse, B, Hq, Hkv, M, d, chunk, scale, &a)) !=
        FA_OK)
        return s;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    CUtensorMap tk, tv;
    if (!fa::encode_decode_maps_fp8(g_encode, k8, v8, d, Hkv, M, B, &tk, &tv)) return FA_ERR_CUDA;
    return from_cuda(fa::launch_decode_fp8(tk, tv, a, d, (int)dtype, (cudaStream_t)stream));
}

FA_EXPORT fa_status fa_decode_paged(const void* q, const void* k_cache, const void* v_cache,
                                    const int* block_table, const int* seq_lens, void* o,
                                    float* lse, int B, int Hq, int Hkv, int max_seq_len,
                                    int num_pages, int page_size, int max_pages_per_seq, int d,
                                    int chunk, float scale, fa_dtype dtype, fa_stream_t stream) {
    fa_status s = check_args(q, k_cache, v_cache, o, lse, B, Hq, Hkv, 1, max_seq_len, d, scale,
                             (int)dtype);
    if (s != FA_OK) return s;
    if (!block_table || !seq_lens || !aligned(block_table, 4) || !aligned(seq_lens, 4))
        return FA_ERR_INVALID_ARG;
    if (num_pages <= 0 || max_pages_per_seq <= 0) return FA_ERR_INVALID_ARG;
    if (page_size < 8 || page_size > 65536 || (page_size & (page_size - 1)) != 0)
        return FA_ERR_INVALID_ARG;
    const int rows = page_size < fa::kDecodeSubTile ? page_size : fa::kDecodeSubTile;
    if (chunk <= 0 || chunk % rows != 0) return FA_ERR_INVALID_ARG;
    if ((long long)max_pages_per_seq * page_size < max_seq_len) return FA_ERR_INVALID_ARG;
    if ((uint64_t)num_pages * page_size * Hkv * d >= kMaxElements) return FA_ERR_INVALID_ARG;
    if (((long long)max_seq_len + chunk - 1) / chunk * B * Hkv > 0x7fffffffLL)
        return FA_ERR_INVALID_ARG;
    DeviceState* st = nullptr;
    if ((s = device_state(&st)) != FA_OK) return s;
    fa::DecodeArgs a;
    if ((s = decode_setup(st, (cudaStream_t)stream, q, o, lse, B, Hq, Hkv, max_seq_len, d, chunk,
                          scale, &a)) != FA_OK)
        return s;
    a.block_table = block_table;
    a.seq_lens = seq_lens;
    a.page = page_size;
    a.max_pages = max_pages_per_seq;
    CUtensorMap tk, tv;
    if (!fa::encode_decode_maps_paged(g_encode, k_cache, v_cache, (int)dtype, d, Hkv, page_size,
                                      num_pages, &tk, &tv))
        return FA_ERR_CUDA;
    return from_cuda(fa::launch_decode_paged(tk, tv, a, d, (int)dtype, (cudaStream_t)stream));
}

FA_EXPORT const char* fa_status_string(fa_status status) {
    switch (status) {
        case FA_OK: return "FA_OK";
        case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG: invalid argument";
        case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED: unsupported head dim, dtype or device";
        case FA_ERR_CUDA: return "FA_ERR_CUDA: a CUDA call or launch failed";
        case FA_ERR_NO_MEMORY: return "FA_ERR_NO_MEMORY: workspace allocation failed";
        case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT: a device-side wait expired";
        case FA_ERR_SCRATCH_LIMIT:
            return "FA_ERR_SCRATCH_LIMIT: the problem needs more than the static decode scratch";
    }
    return "unknown fa_status";
}

FA_EXPORT fa_status fa_get_last_device_status(fa_stream_t stream) {
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return FA_ERR_CUDA;
    DeviceState* st = nullptr;
    const fa_status s = device_state(&st);
    if (s != FA_OK) return s == FA_ERR_UNSUPPORTED ? FA_OK : s;
    int word = 0;
    if (cudaMemcpy(&word, st->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return FA_ERR_CUDA;
    if (word == 0) return FA_OK;
    if (cudaMemset(st->status, 0, sizeof(int)) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess)
        return FA_ERR_CUDA;
    return (word & 0xff) == FA_DEV_TIMEOUT ? FA_ERR_TIMEOUT : FA_ERR_CUDA;
}

FA_EXPORT void fa_set_wait_timeout_ns(unsigned long long ns) {
    g_timeout_ns.store(ns == 0 ? kDefaultTimeoutNs : ns);
}

FA_EXPORT fa_status fa_selftest_wait_timeout(fa_stream_t stream) {
    DeviceState* st = nullptr;
    const fa_status s = device_state(&st);
    if (s != FA_OK) return s;
    return from_cuda(fa::launch_wait_selftest(st->status, g_timeout_ns.load(), (cudaStream_t)stream));
}

FA_EXPORT void fa_release_workspaces(void) {
    std::lock_guard<std::mutex> lock(g_mu);
    int cur = 0;
    const bool have_cur = cudaGetDevice(&cur) == cudaSuccess;
    for (auto& kv : g_devices) {
        if (kv.second.workspaces.empty() && kv.second.pipes.empty()) continue;
        if (cudaSetDevice(kv.first) != cudaSuccess) continue;
        cudaDeviceSynchronize();
        for (auto& w : kv.second.workspaces) {
            if (w.second.ptr) cudaFree(w.second.ptr);
            if (w.second.tickets) cudaFree(w.second.tickets);
        }
        kv.second.workspaces.clear();
        for (auto& pp : kv.second.pipes) {
            HostPipe& hp = pp.second;
            if (!hp.ready) continue;
            cudaStreamDestroy(hp.in);
            cudaStreamDestroy(hp.out);
            cudaEventDestroy(hp.start);
            for (int i = 0; i < 2; ++i) {
                cudaEventDestroy(hp.landed[i]);
                cudaEventDestroy(hp.computed[i]);
                cudaEventDestroy(hp.copied[i]);
            }
        }
        kv.second.pipes.clear();
    }
    if (have_cur) cudaSetDevice(cur);
}

FA_EXPORT int fa_abi_version(void) { return 1; }
