// fa_decode.cu -- split-KV flash decoding over contiguous fp16/bf16 K/V: the
// chunk kernel plus the LSE-weighted merge kernel (two launches), the
// single-launch variant whose chunk kernel merges its own partials, and the
// bounded-wait self-test kernel.  The kernels themselves are in
// fa_decode_kernel.cuh ("CUDA 实现 Flash Decoding：解码阶段并行度重建与性能剖析",
// section 2.2, Steps 1 and 2).
#include "fa_decode_kernel.cuh"

namespace fa {
namespace {

template <int D, typename T>
cudaError_t launch_two(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a,
                       cudaStream_t stream) {
    return dec::launch<D, T, false, false, false>(tk, tv, a, stream);
}

template <int D, typename T>
cudaError_t launch_one(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a,
                       cudaStream_t stream) {
    return dec::launch<D, T, false, false, true>(tk, tv, a, stream);
}

__global__ void wait_selftest_kernel(int* status, unsigned long long timeout_ns) {
    __shared__ __align__(8) uint64_t bar_storage;
    __shared__ int abort_flag;
    const uint32_t bar = smem_addr(&bar_storage);
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const WaitCtl wc{&abort_flag, status, timeout_ns};
        // nobody arrives on this barrier: the wait must give up by itself
        (void)mbar_wait(bar, 0, wc, FA_SITE_SELFTEST);
    }
}

}  // namespace

bool encode_decode_maps(EncodeTiledFn enc, const void* k, const void* v, int dtype, int d,
                        int Hkv, int M, int B, CUtensorMap* tk, CUtensorMap* tv) {
    if (d == 128)
        return dtype == 0
                   ? dec::encode_kv_maps<128, __half, false>(enc, k, v, Hkv, M, B, kDecodeSubTile, tk, tv)
                   : dec::encode_kv_maps<128, __nv_bfloat16, false>(enc, k, v, Hkv, M, B,
                                                                   kDecodeSubTile, tk, tv);
    if (d == 64)
        return dtype == 0
                   ? dec::encode_kv_maps<64, __half, false>(enc, k, v, Hkv, M, B, kDecodeSubTile, tk, tv)
                   : dec::encode_kv_maps<64, __nv_bfloat16, false>(enc, k, v, Hkv, M, B,
                                                                  kDecodeSubTile, tk, tv);
    return false;
}

cudaError_t launch_decode(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a, int d,
                          int dtype, cudaStream_t stream) {
    if (d == 128)
        return dtype == 0 ? launch_two<128, __half>(tk, tv, a, stream)
                          : launch_two<128, __nv_bfloat16>(tk, tv, a, stream);
    if (d == 64)
        return dtype == 0 ? launch_two<64, __half>(tk, tv, a, stream)
                          : launch_two<64, __nv_bfloat16>(tk, tv, a, stream);
    return cudaErrorInvalidValue;
}

cudaError_t launch_decode_fused(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a,
                                int d, int dtype, cudaStream_t stream) {
    if (d == 128)
        return dtype == 0 ? launch_one<128, __half>(tk, tv, a, stream)
                          : launch_one<128, __nv_bfloat16>(tk, tv, a, stream);
    if (d == 64)
        return dtype == 0 ? launch_one<64, __half>(tk, tv, a, stream)
                          : launch_one<64, __nv_bfloat16>(tk, tv, a, stream);
    return cudaErrorInvalidValue;
}

cudaError_t prepare_decode_kernels() {
    cudaError_t err = cudaSuccess;
    auto one = [&](cudaError_t e) {
        if (err == cudaSuccess) err = e;
    };
    one(dec::configure_chunk<128, __half, false, false, 1, false>());
    one(dec::configure_chunk<128, __half, false, false, 2, false>());
    one(dec::configure_chunk<128, __half, false, false, 4, false>());
    one(dec::configure_chunk<128, __nv_bfloat16, false, false, 1, false>());
    one(dec::configure_chunk<128, __nv_bfloat16, false, false, 2, false>());
    one(dec::configure_chunk<128, __nv_bfloat16, false, false, 4, false>());
    one(dec::configure_chunk<64, __half, false, false, 1, false>());
    one(dec::configure_chunk<64, __half, false, false, 2, false>());
    one(dec::configure_chunk<64, __half, false, false, 4, false>());
    one(dec::configure_chunk<64, __nv_bfloat16, false, false, 1, false>());
    one(dec::configure_chunk<64, __nv_bfloat16, false, false, 2, false>());
    one(dec::configure_chunk<64, __nv_bfloat16, false, false, 4, false>());
    return err;
}

cudaError_t launch_wait_selftest(int* status, unsigned long long timeout_ns, cudaStream_t stream) {
    wait_selftest_kernel<<<1, 32, 0, stream>>>(status, timeout_ns);
    return cudaGetLastError();
}

}  // namespace fa
