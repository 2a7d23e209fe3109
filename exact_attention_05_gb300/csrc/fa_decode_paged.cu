// fa_decode_paged.cu -- split-KV decode over a paged K/V cache: key j of batch
// b lives at row j % page of page block_table[b][j / page] of a
// [num_pages, page, Hkv, d] cache, and batch b has seq_lens[b] keys.  The
// kernels are in fa_decode_kernel.cuh; only where the rows come from differs.
#include "fa_decode_kernel.cuh"

namespace fa {

bool encode_decode_maps_paged(EncodeTiledFn enc, const void* kc, const void* vc, int dtype, int d,
                              int Hkv, int page, int num_pages, CUtensorMap* tk, CUtensorMap* tv) {
    const int rows = page < kDecodeSubTile ? page : kDecodeSubTile;  // keys per copy
    if (d == 128)
        return dtype == 0 ? dec::encode_kv_maps<128, __half, false>(enc, kc, vc, Hkv, page,
                                                                    num_pages, rows, tk, tv)
                          : dec::encode_kv_maps<128, __nv_bfloat16, false>(enc, kc, vc, Hkv, page,
                                                                           num_pages, rows, tk, tv);
    if (d == 64)
        return dtype == 0 ? dec::encode_kv_maps<64, __half, false>(enc, kc, vc, Hkv, page,
                                                                   num_pages, rows, tk, tv)
                          : dec::encode_kv_maps<64, __nv_bfloat16, false>(enc, kc, vc, Hkv, page,
                                                                          num_pages, rows, tk, tv);
    return false;
}

cudaError_t launch_decode_paged(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a,
                                int d, int dtype, cudaStream_t stream) {
    if (d == 128)
        return dtype == 0 ? dec::launch<128, __half, false, true, false>(tk, tv, a, stream)
                          : dec::launch<128, __nv_bfloat16, false, true, false>(tk, tv, a, stream);
    if (d == 64)
        return dtype == 0 ? dec::launch<64, __half, false, true, false>(tk, tv, a, stream)
                          : dec::launch<64, __nv_bfloat16, false, true, false>(tk, tv, a, stream);
    return cudaErrorInvalidValue;
}

}  // namespace fa
