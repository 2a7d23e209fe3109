// fa_decode_fp8.cu -- split-KV decode with e4m3 K/V and per-kv-head fp32
// scales (K = k8 * k_scale[h], V = v8 * v_scale[h]); q and o stay fp16/bf16.
// The kernels are in fa_decode_kernel.cuh; only the element format differs.
#include "fa_decode_kernel.cuh"

namespace fa {

bool encode_decode_maps_fp8(EncodeTiledFn enc, const void* k8, const void* v8, int d, int Hkv,
                            int M, int B, CUtensorMap* tk, CUtensorMap* tv) {
    if (d == 128)
        return dec::encode_kv_maps<128, __half, true>(enc, k8, v8, Hkv, M, B, kDecodeSubTile, tk, tv);
    if (d == 64)
        return dec::encode_kv_maps<64, __half, true>(enc, k8, v8, Hkv, M, B, kDecodeSubTile, tk, tv);
    return false;
}

cudaError_t launch_decode_fp8(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a,
                              int d, int dtype, cudaStream_t stream) {
    if (d == 128)
        return dtype == 0 ? dec::launch<128, __half, true, false, false>(tk, tv, a, stream)
                          : dec::launch<128, __nv_bfloat16, true, false, false>(tk, tv, a, stream);
    if (d == 64)
        return dtype == 0 ? dec::launch<64, __half, true, false, false>(tk, tv, a, stream)
                          : dec::launch<64, __nv_bfloat16, true, false, false>(tk, tv, a, stream);
    return cudaErrorInvalidValue;
}

}  // namespace fa
