// fa_internal.h -- declarations shared by the translation units of libfa.so
// (host launchers and the argument blocks the kernels receive).  Not part of
// the public ABI; include/fa.h is.
#pragma once

#include <atomic>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

// Low byte of the device status word; the next byte says which wait expired.
#define FA_DEV_TIMEOUT 1
#define FA_DEV_LAYOUT 2   // a kernel found its shared-memory base misaligned

// Where a bounded wait sits (recorded in bits 8.. of the status word).
enum FaWaitSite {
    FA_SITE_PRODUCER_SLOT = 1,
    FA_SITE_MMA_Q = 2,
    FA_SITE_MMA_KV = 3,
    FA_SITE_MMA_P = 4,
    FA_SITE_SOFTMAX_S = 5,
    FA_SITE_SOFTMAX_O = 6,
    FA_SITE_DRAIN = 7,
    FA_SITE_DECODE_KV = 8,
    FA_SITE_SELFTEST = 9,
    FA_SITE_SMEM_ALIGN = 10,
    FA_SITE_WORK = 11,   // hand-over of the next work item between the roles of a CTA
};

namespace fa {

struct PrefillArgs {
    void* o;               // [B, N, Hq, d], 16-bit
    int B, Hq, Hkv, N, M;
    int causal;
    int n_qtiles;          // ceil(N / 128)
    float scale_log2;      // scale * log2(e)
    float* lse;            // [B, Hq, N] or nullptr
    int* status;           // device status word
    unsigned long long timeout_ns;
};

struct DecodeArgs {
    const void* q;         // [B, 1, Hq, d]
    void* o;               // [B, 1, Hq, d]
    float* lse;            // [B, Hq] or nullptr
    float* o_part;         // workspace [B, Hq, nc, d] fp32
    float* lse_part;       // workspace [B, Hq, nc] fp32, log2 domain
    int B, Hq, Hkv, M, chunk, nc;
    int nstripes;          // CTAs per (b, kv head); set by the launcher
    float scale_log2;
    int* status;
    unsigned long long timeout_ns;
    // e4m3 K/V only: per-kv-head dequantisation scales [Hkv] (K = k8 * k_scale)
    const float* k_scale;
    const float* v_scale;
    // paged K/V only: cache [num_pages, page, Hkv, d], block_table [B, max_pages]
    // (int32 page ids), seq_lens [B] (keys of each batch, <= M); M is the
    // largest sequence length and sets nc
    const int* block_table;
    const int* seq_lens;
    int page;
    int max_pages;
    // single-launch variant only: one merged partial per stripe (room for nc
    // stripes, the most there can be) and a self-resetting ticket per (b, kv head)
    float* g_o;            // [B, Hq, nstripes, d] fp32
    float* g_lse;          // [B, Hq, nstripes] fp32, log2 domain
    int* tickets;          // [B, Hkv]; all zero between calls
};

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// Encodes the K and V tensor maps the decode chunk kernel reads (their boxes
// and swizzle are the kernel's business).  Returns false if encoding failed.
bool encode_decode_maps(EncodeTiledFn enc, const void* k, const void* v, int dtype, int d,
                        int Hkv, int M, int B, CUtensorMap* tk, CUtensorMap* tv);

// dtype: 0 = fp16, 1 = bf16; d in {64, 128}.
cudaError_t launch_prefill(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const CUtensorMap& to, const PrefillArgs& a, int d, int dtype,
                           cudaStream_t stream);

// Backward (dQ, dK, dV).  Tensors as in the forward; lse [B, Hq, N] natural
// log (as fa_fwd writes it); pack and dq_acc [B, N, Hq, d] fp32 are workspace.
struct BackwardArgs {
    const void* o;         // [B, N, Hq, d] forward output
    const void* dout;      // [B, N, Hq, d]
    const float* lse;      // [B, Hq, N]
    float* pack;           // [B, Hq, n_qtiles, 2, 128]: LSE*log2(e) (+inf past N), then D_i = dO_i . O_i
    float* dq_acc;         // [B, N, Hq, d] fp32 accumulator of dQ / scale
    void* dq;              // [B, N, Hq, d]
    void* dk;              // [B, M, Hkv, d]
    void* dv;              // [B, M, Hkv, d]
    int B, Hq, Hkv, N, M;
    int causal;
    int n_qtiles, n_ktiles;
    float scale, scale_log2;
    int* status;
    unsigned long long timeout_ns;
};

// tq/tdo over [B, N, Hq, d], tk/tv over [B, M, Hkv, d]: 64 x 128-row boxes, 128-byte
// swizzle; tdq over the fp32 dQ accumulator [B, N, Hq, d]: 32 x 128-row boxes, 128-byte
// swizzle (the target of bulk reductions).
cudaError_t launch_backward(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const CUtensorMap& tdq, const BackwardArgs& a,
                            int d, int dtype, cudaStream_t stream);

cudaError_t launch_decode(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a, int d,
                          int dtype, cudaStream_t stream);

// e4m3 K/V with per-kv-head scales (q, o of `dtype`).
bool encode_decode_maps_fp8(EncodeTiledFn enc, const void* k8, const void* v8, int d, int Hkv,
                            int M, int B, CUtensorMap* tk, CUtensorMap* tv);
cudaError_t launch_decode_fp8(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a,
                              int d, int dtype, cudaStream_t stream);

// Paged K/V cache [num_pages, page, Hkv, d] addressed through a block table.
bool encode_decode_maps_paged(EncodeTiledFn enc, const void* kc, const void* vc, int dtype, int d,
                              int Hkv, int page, int num_pages, CUtensorMap* tk, CUtensorMap* tv);
cudaError_t launch_decode_paged(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a,
                                int d, int dtype, cudaStream_t stream);

// Single launch: the chunk kernel merges its own partials (two-level ticket merge).
cudaError_t launch_decode_fused(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a,
                                int d, int dtype, cudaStream_t stream);

cudaError_t launch_wait_selftest(int* status, unsigned long long timeout_ns, cudaStream_t stream);

// The library's status word on the current device: static device memory
// (every device that loads the module holds one, zero at load), so looking
// it up allocates nothing.  Resolved once per device with cudaGetSymbolAddress.
// Returns nullptr if the lookup failed.
int* status_word_current_device();

// The current limit of every device-side wait (fa_set_wait_timeout_ns).
unsigned long long wait_timeout_ns();

// cuTensorMapEncodeTiled behind the library's cache of encoded maps (a map
// whose arguments were seen before is copied, not encoded again), or nullptr
// if the current device is not usable.
EncodeTiledFn tensor_map_encoder();

// Sets a kernel's launch attributes once per device: the largest dynamic
// shared memory the device allows next to the kernel's static shared memory
// (so that a launch of any size up to that needs no further set-up), and the
// largest shared-memory carveout.  `configured` is the caller's per-kernel
// record of the devices done (bit i = device i; devices from 32 on are
// configured on every call).
template <typename Kernel>
cudaError_t configure_kernel_once(Kernel kern, std::atomic<unsigned>& configured) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    const unsigned bit = dev < 32 ? (1u << dev) : 0u;
    if (bit != 0u && (configured.load(std::memory_order_acquire) & bit) != 0u) return cudaSuccess;
    cudaFuncAttributes fattr{};
    int optin = 0;
    if ((err = cudaFuncGetAttributes(&fattr, kern)) != cudaSuccess) return err;
    if ((err = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) !=
        cudaSuccess)
        return err;
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               optin - int(fattr.sharedSizeBytes));
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                               int(cudaSharedmemCarveoutMaxShared));
    if (err != cudaSuccess) return err;
    configured.fetch_or(bit, std::memory_order_acq_rel);
    return cudaSuccess;
}

// Applies the launch attributes of every two-kernel 16-bit decode variant on
// the current device (all head dims, types and heads-per-pass), so that
// later calls configure nothing.
cudaError_t prepare_decode_kernels();

// Geometry the host needs to build tensor maps.
constexpr int kPrefillTile = 128;   // query rows per tile and keys per KV tile
constexpr int kDecodeSubTile = 128; // keys per decode sub-tile

}  // namespace fa
