// fa_decode_noalloc.cu -- fa_decode_noalloc(): split-KV decode that allocates
// no device memory.
//
// fa_decode keeps its fp32 chunk partials in a workspace it allocates with
// cudaMalloc on first use.  Some callers cannot allow that: code running while
// a CUDA graph is being captured, processes whose device memory is handed out
// by a pool that must own every allocation, and hosts that forbid allocation
// after start-up.  For them this entry point runs the same two kernels
// (chunk partials, then the LSE-weighted merge) with the partials placed in a
// fixed array in static device memory, defined below.  The array exists on
// every GPU on which the library's module is loaded and lives until the
// process exits.
//
// Rules of use:
//   * the first call on a device resolves the array's device address with
//     cudaGetSymbolAddress (once per device, with that device current), looks
//     up the library's status word the same way and applies the launch
//     attributes of every decode kernel variant; make that first call before
//     any stream capture begins;
//   * problems that need more than FA_DECODE_NOALLOC_SCRATCH_BYTES of
//     partials are rejected with FA_ERR_SCRATCH_LIMIT before any launch;
//   * every call shares the one array and it keeps the previous call's
//     contents; the chunk kernel writes every partial before the merge reads
//     it, so nothing has to be cleared -- but calls that overlap on the GPU
//     (different streams, no ordering between them) race on the array;
//   * the kernels' bounded waits take the limit fa_set_wait_timeout_ns() set
//     (read at each call) and report an expiry in the library's status word,
//     the one fa_get_last_device_status() reads and clears; that word is
//     static device memory too.
#include <cmath>
#include <cstdint>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "fa.h"
#include "fa_internal.h"

#define FA_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

constexpr size_t kScratchFloats = FA_DECODE_NOALLOC_SCRATCH_BYTES / sizeof(float);

static __device__ __align__(256) float g_noalloc_scratch[kScratchFloats];

using fa::EncodeTiledFn;

struct DeviceSetup {
    bool done = false;
    fa_status result = FA_OK;
    float* scratch = nullptr;
    int* status = nullptr;
};

constexpr int kMaxDevices = 64;
DeviceSetup g_setup[kMaxDevices];
EncodeTiledFn g_encode = nullptr;
std::mutex g_mu;

constexpr uint64_t kMaxElements = 1ull << 39;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// One-time set-up of the current device: architecture check, the device
// addresses of the static array and of the status word, the library's
// tensor-map encoder (with its cache of encoded maps), the decode kernels'
// launch attributes.
fa_status setup_current_device(DeviceSetup** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceSetup& s = g_setup[dev];
    if (!s.done) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
            s.result = FA_ERR_CUDA;
        } else if (major != 10 || minor != 3) {
            s.result = FA_ERR_UNSUPPORTED;
        } else {
            void* p = nullptr;
            int* st = fa::status_word_current_device();
            if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr ||
                st == nullptr || fa::prepare_decode_kernels() != cudaSuccess) {
                s.result = FA_ERR_CUDA;
            } else {
                s.scratch = static_cast<float*>(p);
                s.status = st;
                s.result = FA_OK;
            }
        }
        if (s.result == FA_OK && g_encode == nullptr) {
            g_encode = fa::tensor_map_encoder();
            if (g_encode == nullptr) s.result = FA_ERR_CUDA;
        }
        s.done = true;
    }
    if (s.result != FA_OK) return s.result;
    *out = &s;
    return FA_OK;
}

}  // namespace

FA_EXPORT fa_status fa_decode_noalloc(const void* q, const void* k, const void* v, void* o,
                                      float* lse, int B, int Hq, int Hkv, int M, int d, int chunk,
                                      float scale, fa_dtype dtype, fa_stream_t stream) {
    // the same argument rules as fa_decode, checked before any CUDA call
    if (!q || !k || !v || !o) return FA_ERR_INVALID_ARG;
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || M <= 0 || d <= 0 || chunk <= 0) return FA_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return FA_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !std::isfinite(scale)) return FA_ERR_INVALID_ARG;
    if (dtype != FA_FP16 && dtype != FA_BF16) return FA_ERR_UNSUPPORTED;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16))
        return FA_ERR_INVALID_ARG;
    if (lse && !aligned(lse, 4)) return FA_ERR_INVALID_ARG;
    if ((uint64_t)B * Hq * d >= kMaxElements || (uint64_t)B * M * Hkv * d >= kMaxElements)
        return FA_ERR_INVALID_ARG;
    const long long nc = ((long long)M + chunk - 1) / chunk;
    if (nc * B * Hkv > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
    const unsigned long long part_elems = (unsigned long long)B * Hq * nc * d;
    const unsigned long long need = part_elems + (unsigned long long)B * Hq * nc;
    if (need > kScratchFloats) return FA_ERR_SCRATCH_LIMIT;

    DeviceSetup* s = nullptr;
    fa_status st = setup_current_device(&s);
    if (st != FA_OK) return st;
    CUtensorMap tk, tv;
    if (!fa::encode_decode_maps(g_encode, k, v, dtype, d, Hkv, M, B, &tk, &tv)) return FA_ERR_CUDA;
    fa::DecodeArgs a{};
    a.q = q;
    a.o = o;
    a.lse = lse;
    a.o_part = s->scratch;
    a.lse_part = s->scratch + part_elems;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.M = M;
    a.chunk = chunk;
    a.nc = (int)nc;
    a.scale_log2 = (float)((double)scale * 1.4426950408889634);
    a.status = s->status;
    a.timeout_ns = fa::wait_timeout_ns();
    return fa::launch_decode(tk, tv, a, d, (int)dtype, (cudaStream_t)stream) == cudaSuccess
               ? FA_OK
               : FA_ERR_CUDA;
}
