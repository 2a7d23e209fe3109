// fa_decode_kernel.cuh -- the split-KV decode chunk kernel and the LSE merge,
// shared by the decode entry points (contiguous 16-bit K/V, e4m3 K/V with
// per-kv-head scales, and K/V in a paged cache addressed through a block
// table).  Included by the translation units that instantiate it.
//
// What is computed follows "CUDA 实现 Flash Decoding：解码阶段并行度重建与性能剖析",
// section 2.2: for one query row per (b, h) the keys are cut into chunks of
// `chunk` keys; Step 1 gives every chunk its own partial
//     m_c = max s,  P_c = exp(s - m_c),  l_c = sum P_c,
//     O_c = P_c V_c / l_c,  lse_c = m_c + log l_c,
// and Step 2 merges them with global_lse = m + log sum_c exp(lse_c - m) and
// weights w_c = exp(lse_c - global_lse), O = sum_c w_c O_c.  Logits and LSEs
// are kept in base 2 (scale * log2 e folded in), which changes no result.
//
// Layout of the work on GB300:
//   * persistent CTAs of 128 threads, nstripes per (b, kv head) (one wave):
//     the CTA with stripe s walks chunks s, s + nstripes, ... and serves every
//     query head of the GQA group, so each K/V byte is read from HBM once; the
//     block index is ordered with (b, kv head) fastest so that CTAs running
//     together read whole contiguous key rows.  Warp 0 streams the K and V
//     sub-tiles (128 keys) through a ring of TMA slots in the order the chunks
//     consume them.
//   * scores: thread <-> key, the full dot product read from a swizzled K
//     tile (one 16-byte chunk per step, conflict-free); softmax in registers
//     with warp-shuffle reductions; P.V: thread <-> (4 columns, key group).
//   * the merge: each stripe CTA merges its own chunks on the fly when one
//     pass over a tile serves all its query heads (else it writes one partial
//     per chunk); then a second kernel (one CTA per (b, h) and 16 columns)
//     merges the stripes' partials, or, in the single launch, the last stripe
//     of a (b, kv head) does.
//   * e4m3 K/V: the same tiles at one byte per element; the per-kv-head scales
//     are applied once per score (s = k_scale * q.k8) and once per output
//     (o = v_scale * sum_j p_j v8_j), which is exact algebra.
//   * paged K/V: rows of key j of batch b live in page block_table[b][j / P]
//     at row j % P of a [num_pages, P, Hkv, d] cache; a 128-key sub-tile is
//     fetched by one TMA copy per page it spans, and batch b only has
//     seq_lens[b] keys (chunks past the end write an empty partial).
#pragma once

#include <atomic>
#include <cfloat>
#include <cmath>
#include <cuda_fp8.h>

#include "fa_device.cuh"
#include "fa_internal.h"

namespace fa {
namespace dec {

constexpr float kLn2 = 0.6931471805599453f;

// Element format of the K/V tiles.
template <typename T, bool FP8>
struct KvFmt {
    static constexpr int ESZ = FP8 ? 1 : 2;  // bytes per element
};

template <int D, typename T, bool FP8>
struct DecodeCfg {
    static constexpr int TK = kDecodeSubTile;           // keys per sub-tile
    static constexpr int THREADS = 128;                 // thread <-> key in the score step
    static constexpr int GMAX = 4;                      // query heads per pass (max)
    static constexpr int ESZ = KvFmt<T, FP8>::ESZ;
    static constexpr int ROW_BYTES = D * ESZ;           // one K or V row
    static constexpr int KBOX = ROW_BYTES < 128 ? ROW_BYTES : 128;  // swizzled K box row
    static constexpr int NSUBK = ROW_BYTES / KBOX;      // K boxes per row
    static constexpr int SUB_BYTES = TK * KBOX;         // one K sub-box
    static constexpr int TILE_BYTES = TK * ROW_BYTES;   // one K or one V sub-tile
    static constexpr bool IS_F16 = DTypeFmt<T>::value == 0;
    // Scores with a mixed-precision FMA (16-bit q times 16-bit k, fp32 sum)
    // unless the keys are e4m3 and q is bf16 (e4m3 widens exactly to f16 only).
    static constexpr bool QK_MIXED = !(FP8 && !IS_F16);
    // P.V with the mixed FMA on f16 values (fp16 V, or e4m3 V widened to f16;
    // P rounded to f16); bf16 V takes the fp32 route with fp32 P.
    static constexpr bool PV_MIXED = FP8 || IS_F16;
    static constexpr int QSZ = QK_MIXED ? 2 : 4;        // bytes per query element in smem
    // P.V mapping: thread <-> (group of 4 columns, key group)
    static constexpr int NCG = D / 4;
    static constexpr int KQ = THREADS / NCG;            // key groups
    static constexpr int KPG = TK / KQ;                 // keys per group
    // Ring of tile slots that K and V sub-tiles stream through, in load order
    // K0, V0, K1, V1, ...: 2 slots of 32 KB (16-bit, d = 128) up to 8 of 8 KB.
    static constexpr int RING_BYTES = FP8 ? 32768 : 65536;
    static constexpr int NSLOT = RING_BYTES / TILE_BYTES;
    static constexpr int SC_OFF = RING_BYTES;                      // float [GMAX][TK]
    static constexpr int PH_OFF = SC_OFF + GMAX * TK * 4;          // f16 P [GMAX][TK]
    static constexpr int RED_OFF = PH_OFF + GMAX * TK * 2;         // float4 [KQ-1][GMAX][NCG]
    static constexpr int HS_OFF = RED_OFF + (KQ - 1) * GMAX * D * 4;  // per warp max, sum [2][4][GMAX]
    static constexpr int BAR_OFF = HS_OFF + 2 * 4 * GMAX * 4;      // NSLOT full barriers
    static constexpr int MISC_OFF = BAR_OFF + 8 * NSLOT;
    static constexpr int QS_OFF = MISC_OFF + 16;                   // q [g][D], sized at launch
    static constexpr size_t smem_bytes(int g) {
        return size_t(QS_OFF) + size_t(g) * D * QSZ + 1024;        // + slack to align to 1 KB
    }
    static_assert(NSLOT >= 2 && RING_BYTES % TILE_BYTES == 0, "ring of whole tiles");
    static_assert(BAR_OFF % 8 == 0 && QS_OFF % 16 == 0, "alignment");
    // position of 16-byte chunk ch of K row i inside the swizzled box: the TMA
    // swizzle XORs the chunk index with address bits 7.. of the row start
    __device__ static int kchunk(int i, int ch) {
        return ch ^ (((i * KBOX) >> 7) & (KBOX / 16 - 1));
    }
};

// Eight consecutive elements of a 16-byte chunk -> fp32 (16-bit formats).
template <typename T>
__device__ __forceinline__ void unpack8(const uint4& w, float (&f)[8]) {
    const float2 a = unpack2<T>(w.x), b = unpack2<T>(w.y), c = unpack2<T>(w.z), d = unpack2<T>(w.w);
    f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
    f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
}

// Two e4m3 values (low byte first) -> fp32.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t v) {
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(v), __NV_E4M3);
    return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

// Mixed-precision FMAs (16-bit products, fp32 accumulators): c0 += a.lo * b.lo
// and c1 += a.hi * b.hi for two packed pairs, or c0 += a.lo * p, c1 += a.hi * p.
// The product of two 16-bit values is exact in fp32, so only the sum rounds.
template <typename T>
__device__ __forceinline__ void mfma2(float& c0, float& c1, uint32_t a, uint32_t b) {
    if constexpr (DTypeFmt<T>::value == 0)
        asm("{\n\t.reg .b16 a0, a1, b0, b1;\n\tmov.b32 {a0, a1}, %2;\n\tmov.b32 {b0, b1}, %3;\n\t"
            "fma.rn.f32.f16 %0, a0, b0, %0;\n\tfma.rn.f32.f16 %1, a1, b1, %1;\n\t}"
            : "+f"(c0), "+f"(c1) : "r"(a), "r"(b));
    else
        asm("{\n\t.reg .b16 a0, a1, b0, b1;\n\tmov.b32 {a0, a1}, %2;\n\tmov.b32 {b0, b1}, %3;\n\t"
            "fma.rn.f32.bf16 %0, a0, b0, %0;\n\tfma.rn.f32.bf16 %1, a1, b1, %1;\n\t}"
            : "+f"(c0), "+f"(c1) : "r"(a), "r"(b));
}
__device__ __forceinline__ void mfma2s_f16(float& c0, float& c1, uint32_t a, uint16_t p) {
    asm("{\n\t.reg .b16 a0, a1;\n\tmov.b32 {a0, a1}, %2;\n\t"
        "fma.rn.f32.f16 %0, a0, %3, %0;\n\tfma.rn.f32.f16 %1, a1, %3, %1;\n\t}"
        : "+f"(c0), "+f"(c1) : "r"(a), "h"(p));
}
// Two e4m3 values (low byte first) -> f16x2 (exact: every e4m3 value is an f16 value).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t v) {
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
    return r;
}

// Merges n partial results (fp32 rows of D at rows + i*stride*D, normalised,
// with log2-domain LSEs lse[i*stride]) into one with the LSE weights of the page's Step 2:
// w_i = 2^(lse_i - glse), glse = log2 sum_i 2^lse_i.  128 threads; thread t < D
// owns column t.  Returns glse; writes the row to out_f (fp32) or out_t.  If
// every partial is empty (lse = -inf) the row is zero and glse is -inf.
template <int D, typename T>
__device__ float merge_partials(const float* lse, const float* rows, int n, int stride, float* red,
                                float* out_f, T* out_t) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    float mx = -INFINITY;
    for (int i = tid; i < n; i += 128) mx = fmaxf(mx, __ldcg(lse + size_t(i) * stride));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if (lane == 0) red[warp] = mx;
    __syncthreads();
    mx = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
    __syncthreads();
    const float ref = mx == -INFINITY ? 0.f : mx;
    float sm = 0.f;
    for (int i = tid; i < n; i += 128) sm += fast_exp2(__ldcg(lse + size_t(i) * stride) - ref);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sm += __shfl_xor_sync(0xffffffffu, sm, off);
    if (lane == 0) red[warp] = sm;
    __syncthreads();
    sm = red[0] + red[1] + red[2] + red[3];
    __syncthreads();
    const float glse = mx == -INFINITY ? -INFINITY : mx + log2f(sm);
    if (tid < D) {
        float acc = 0.f;
        if (mx != -INFINITY) {
#pragma unroll 8
            for (int i = 0; i < n; ++i)
                acc = fmaf(fast_exp2(__ldcg(lse + size_t(i) * stride) - glse),
                           __ldcg(rows + size_t(i) * stride * D + tid), acc);
        }
        if (out_f != nullptr) out_f[tid] = acc;
        if (out_t != nullptr) out_t[tid] = static_cast<T>(acc);
    }
    return glse;
}

// Single launch (no merge kernel).  Every stripe CTA leaves one partial per
// query head: `merged` when the chunk loop already carried its running state
// across the stripe's chunks (one pass per tile), else it merges the chunk
// partials it wrote (rows stride nstripes apart, still in L2).  The last stripe
// CTA of a (b, kv head) to finish then merges the stripe partials into O and
// LSE.  The ticket is reset by whoever finishes it, so it is zero again when
// the kernel ends.
template <int D, typename T>
__device__ void fused_stripe_tail(const DecodeArgs& a, bool ok, int b, int kvh, int stripe,
                                  bool merged) {
    __shared__ int s_last;
    __shared__ float s_red[4];
    const int tid = threadIdx.x;
    const int g = a.Hq / a.Hkv;
    // The barrier orders every thread's partial stores before the merge reads
    // them back (and, through thread 0's cumulative fence, before the ticket).
    if (!__syncthreads_and(ok)) return;
    const int nmine = (a.nc - stripe + a.nstripes - 1) / a.nstripes;  // chunks stripe, stripe + nstripes, ...
    for (int gi = 0; gi < g && !merged; ++gi) {
        const size_t bh = size_t(b) * a.Hq + kvh * g + gi;
        const size_t src = bh * a.nc + stripe;
        const size_t dst = bh * a.nstripes + stripe;
        const float glse = merge_partials<D, T>(a.lse_part + src, a.o_part + src * D, nmine,
                                                a.nstripes, s_red, a.g_o + dst * D, nullptr);
        if (tid == 0) a.g_lse[dst] = glse;
        __syncthreads();
    }
    int* t = a.tickets + (size_t(b) * a.Hkv + kvh);
    if (tid == 0) {
        __threadfence();
        s_last = atomicAdd(t, 1) == a.nstripes - 1;
        if (s_last) __threadfence();  // acquire: the other stripes' partials are visible
    }
    __syncthreads();
    if (!s_last) return;
    for (int gi = 0; gi < g; ++gi) {
        const size_t bh = size_t(b) * a.Hq + kvh * g + gi;
        const float glse = merge_partials<D, T>(a.g_lse + bh * a.nstripes, a.g_o + bh * a.nstripes * D,
                                                a.nstripes, 1, s_red, nullptr,
                                                reinterpret_cast<T*>(a.o) + bh * D);
        if (tid == 0 && a.lse != nullptr) a.lse[bh] = glse * kLn2;
        __syncthreads();
    }
    if (tid == 0) *t = 0;
}

// The merge kernel.  One CTA of 128 threads per (b, h) and 16 output columns:
// thread t owns the float4 column group t % 4 and the chunks c = t / 4 (mod 32).
// A row whose partials are all empty (lse = -inf) gives O = 0, LSE = -inf.
template <int D, typename T>
__global__ void __launch_bounds__(128) merge_kernel(const DecodeArgs a) {
    // the chunk kernel's partials must be complete and visible (programmatic
    // dependent launch: this grid may start before the previous one ends)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    __shared__ float red[4];
    __shared__ float4 part[4][4];
    const int bh = blockIdx.x;
    const int col0 = blockIdx.y * 16;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const float* lse_row = a.lse_part + size_t(bh) * a.nc;
    const float* o_rows = a.o_part + size_t(bh) * a.nc * D;

    float mx = -INFINITY;
    for (int cc = tid; cc < a.nc; cc += 128) mx = fmaxf(mx, lse_row[cc]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if (lane == 0) red[warp] = mx;
    __syncthreads();
    mx = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
    __syncthreads();
    const bool empty = mx == -INFINITY;
    float sm = 0.f;
    for (int cc = tid; cc < a.nc; cc += 128) sm += fast_exp2(lse_row[cc] - (empty ? 0.f : mx));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sm += __shfl_xor_sync(0xffffffffu, sm, off);
    if (lane == 0) red[warp] = sm;
    __syncthreads();
    sm = red[0] + red[1] + red[2] + red[3];
    const float glse = empty ? -INFINITY : mx + log2f(sm);  // log2 domain

    const int cq = tid & 3;
    const float* src = o_rows + col0 + cq * 4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (!empty) {
#pragma unroll 8
        for (int cc = tid >> 2; cc < a.nc; cc += 32) {
            const float w = fast_exp2(lse_row[cc] - glse);
            const float4 v = *reinterpret_cast<const float4*>(src + size_t(cc) * D);
            acc.x = fmaf(w, v.x, acc.x);
            acc.y = fmaf(w, v.y, acc.y);
            acc.z = fmaf(w, v.z, acc.z);
            acc.w = fmaf(w, v.w, acc.w);
        }
    }
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        acc.x += __shfl_xor_sync(0xffffffffu, acc.x, off);
        acc.y += __shfl_xor_sync(0xffffffffu, acc.y, off);
        acc.z += __shfl_xor_sync(0xffffffffu, acc.z, off);
        acc.w += __shfl_xor_sync(0xffffffffu, acc.w, off);
    }
    if (lane < 4) part[warp][lane] = acc;
    __syncthreads();
    if (tid < 4) {
        float4 t = part[0][tid];
#pragma unroll
        for (int w = 1; w < 4; ++w) {
            t.x += part[w][tid].x;
            t.y += part[w][tid].y;
            t.z += part[w][tid].z;
            t.w += part[w][tid].w;
        }
        T* orow = reinterpret_cast<T*>(a.o) + size_t(bh) * D + col0 + tid * 4;
        *reinterpret_cast<uint2*>(orow) = make_uint2(pack2<T>(t.x, t.y), pack2<T>(t.z, t.w));
    }
    if (tid == 0 && blockIdx.y == 0 && a.lse != nullptr) a.lse[bh] = glse * kLn2;
}

// The chunk kernel.  FP8: K/V are e4m3 bytes with per-kv-head scales.  PAGED:
// K/V come from a paged cache through a block table (see the file header).
// GP query heads per pass over a tile (the host picks GP dividing the GQA
// group).  FUSED: the chunk kernel also merges (single launch); only for
// contiguous 16-bit K/V.
//
// Persistent over chunks: the grid is (b, kv head) x nstripes; the CTA with
// stripe s handles chunks s, s + nstripes, ... of its (b, kv head), so it loads
// its g query rows (and, paged, its sequence length) once.  Warp 0 issues the
// TMA copies of the K and V sub-tiles, in the order the chunks consume them,
// into a ring of tile slots, and refills a slot as soon as the last pass over
// it is done, so the next tiles stream in while the current one is computed.
// When one pass over a tile serves every query head of the group (g <= 4),
// a stripe's chunks are merged on the fly into one partial per stripe;
// otherwise (several passes per tile) each chunk yields its own partial
// (O_c, lse_c), as in Step 1.
template <int D, typename T, bool FP8, bool PAGED, int GP, bool FUSED>
__global__ void __launch_bounds__(128, (FP8 && GP == 1) ? 5 : 3)
    chunk_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                 const DecodeArgs a) {
    static_assert(!(FUSED && (FP8 || PAGED)), "the single launch is built for contiguous 16-bit K/V");
    using C = DecodeCfg<D, T, FP8>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const uint32_t sbase = smem_addr(smem);
    const uint32_t bar0 = sbase + C::BAR_OFF;  // full barrier of slot i at bar0 + 8 i
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF);
    float* qs = reinterpret_cast<float*>(smem + C::QS_OFF);
    float* sc = reinterpret_cast<float*>(smem + C::SC_OFF);
    float2* red = reinterpret_cast<float2*>(smem + C::RED_OFF);
    float* wmax = reinterpret_cast<float*>(smem + C::HS_OFF);  // [warp][head] max of a sub-tile
    float* wsum = wmax + 4 * C::GMAX;                             // [warp][head] sum of P

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    // Block index, (b, kv head) fastest: CTAs that run together read the
    // neighbouring heads of the same keys (whole contiguous key rows).
    const int nbh = a.B * a.Hkv;
    const int stripe = blockIdx.x / nbh;
    const int b = (blockIdx.x % nbh) / a.Hkv;
    const int kvh = blockIdx.x % a.Hkv;
    const int g = a.Hq / a.Hkv;
    const int npass = g / GP;
    const int mb = PAGED ? min(__ldg(a.seq_lens + b), a.M) : a.M;  // keys of this sequence
    constexpr int NCP = D / 2;

    if (tid == 0) {
        for (int i = 0; i < C::NSLOT; ++i) mbar_init(bar0 + 8 * i, 1);
        *abort_flag = 0;
        fence_barrier_init();
        prefetch_tensor_map(&tm_k);
        prefetch_tensor_map(&tm_v);
    }
    __syncthreads();
    const WaitCtl wc{abort_flag, a.status, a.timeout_ns};

    // ---- producer (warp 0): walks this CTA's loads in consumption order -------
    // Chunk c has nl loads: K, V of each sub-tile, once per pass if the chunk
    // spans several sub-tiles, else once (the tile stays for all passes).
    int p_c = stripe, p_li = 0, p_nl = 0, p_nsub = 1, p_key0 = 0, p_key1 = 0;
    int issued = 0;
    int pg_next = 0;  // paged: page id of this lane's copy of the next load
    auto p_setup = [&]() {
        // first chunk at or after p_c that has keys; p_c >= nc when none is left
        for (; p_c < a.nc; p_c += a.nstripes) {
            p_key0 = p_c * a.chunk;
            p_key1 = min(mb, p_key0 + a.chunk);
            if (p_key0 < p_key1) break;
        }
        if (p_c < a.nc) {
            p_nsub = (p_key1 - p_key0 + C::TK - 1) / C::TK;
            p_nl = 2 * (p_nsub > 1 ? p_nsub * npass : 1);
            p_li = 0;
        }
    };
    auto p_prefetch = [&]() {
        if constexpr (PAGED) {
            if (p_c < a.nc) {
                const int R = a.page < C::TK ? a.page : C::TK;
                const int row = p_key0 + ((p_li >> 1) % p_nsub) * C::TK;
                const int nrows = min(C::TK, p_key1 - row);
                if (lane * R < nrows)
                    pg_next = __ldg(a.block_table + size_t(b) * a.max_pages + (row + lane * R) / a.page);
            }
        }
    };
    auto p_issue = [&]() {
        const int slot = issued % C::NSLOT;
        const uint32_t bar = bar0 + 8 * slot;
        const uint32_t dst = sbase + slot * C::TILE_BYTES;
        const bool is_v = (p_li & 1) != 0;
        const int row = p_key0 + ((p_li >> 1) % p_nsub) * C::TK;
        if constexpr (!PAGED) {
            if (lane == 0) {
                mbar_arrive_expect_tx(bar, C::TILE_BYTES);
                if (!is_v) {
#pragma unroll
                    for (int s = 0; s < C::NSUBK; ++s)
                        tma_load_4d(dst + s * C::SUB_BYTES, &tm_k, s * (C::KBOX / C::ESZ), kvh, row,
                                    b, bar);
                } else {
                    tma_load_4d(dst, &tm_v, 0, kvh, row, b, bar);
                }
            }
        } else {
            // one copy of R rows per page spanned (only the rows the chunk needs);
            // lane r issues copy r
            const int R = a.page < C::TK ? a.page : C::TK;
            const int nrows = min(C::TK, p_key1 - row);
            const int ncopy = (nrows + R - 1) / R;
            if (lane == 0) mbar_arrive_expect_tx(bar, uint32_t(ncopy * R * C::ROW_BYTES));
            __syncwarp();
            if (lane < ncopy) {
                const int prow = (row + lane * R) % a.page;
                if (!is_v) {
#pragma unroll
                    for (int s = 0; s < C::NSUBK; ++s)
                        tma_load_4d(dst + s * C::SUB_BYTES + lane * R * C::KBOX, &tm_k,
                                    s * (C::KBOX / C::ESZ), kvh, prow, pg_next, bar);
                } else {
                    tma_load_4d(dst + lane * R * C::ROW_BYTES, &tm_v, 0, kvh, prow, pg_next, bar);
                }
            }
        }
        ++issued;
        if (++p_li >= p_nl) {
            p_c += a.nstripes;
            p_setup();
        }
        p_prefetch();
    };
    // keeps NSLOT loads ahead of the `released` loads the consumers are done with
    auto produce = [&](int released) {
        while (p_c < a.nc && issued < released + C::NSLOT) p_issue();
    };
    if (warp == 0) {
        p_setup();
        p_prefetch();
        produce(0);
    }

    // query rows of all g heads of this kv head (read as broadcasts): the raw
    // 16-bit values for the mixed-precision scores, else fp32
    {
        const T* qg = reinterpret_cast<const T*>(a.q) + (size_t(b) * a.Hq + kvh * g) * D;
        for (int e = tid; e < g * D; e += C::THREADS) {
            if constexpr (C::QK_MIXED)
                reinterpret_cast<T*>(qs)[e] = qg[e];
            else
                qs[e] = static_cast<float>(qg[e]);
        }
    }
    __syncthreads();

    const float kscale = FP8 ? __ldg(a.k_scale + kvh) : 1.f;
    const float vscale = FP8 ? __ldg(a.v_scale + kvh) : 1.f;
    const float sfac = kscale * a.scale_log2;
    bool ok = true;
    int cn = 0;  // loads consumed (and released) so far
    // P.V mapping: thread <-> (group of 4 columns cg, key group kq)
    const int cg = tid % C::NCG;
    const int kq = tid / C::NCG;
    uint16_t* ph = reinterpret_cast<uint16_t*>(smem + C::PH_OFF);

    // running max and sum of each head (kept identically by every thread) and two
    // accumulators per head (even and odd keys: independent FMA chains)
    float m_run[GP], l_run[GP], alpha[GP];
    float4 acc[GP], acc2[GP];
    auto reset = [&]() {
#pragma unroll
        for (int gi = 0; gi < GP; ++gi) {
            m_run[gi] = -INFINITY;
            l_run[gi] = 0.f;
            acc[gi] = acc2[gi] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    };
    // Adds up the key groups' accumulators of heads hg .. hg+GP-1 and writes the
    // normalised rows and log2-domain LSEs at o_dst + r*D, lse_dst[r], with
    // r = (b*Hq + h) * per_head + idx.  Collective (all 128 threads).
    auto write_partial = [&](int hg, float* o_dst, float* lse_dst, int per_head, int idx) {
        float4* red4 = reinterpret_cast<float4*>(red);
#pragma unroll
        for (int gi = 0; gi < GP; ++gi) {
            acc[gi].x += acc2[gi].x;
            acc[gi].y += acc2[gi].y;
            acc[gi].z += acc2[gi].z;
            acc[gi].w += acc2[gi].w;
        }
        if (kq > 0) {
#pragma unroll
            for (int gi = 0; gi < GP; ++gi) red4[((kq - 1) * C::GMAX + gi) * C::NCG + cg] = acc[gi];
        }
        __syncthreads();
        if (kq == 0) {
#pragma unroll
            for (int gi = 0; gi < GP; ++gi) {
                float4 t = acc[gi];
#pragma unroll
                for (int u = 1; u < C::KQ; ++u) {
                    const float4 o = red4[((u - 1) * C::GMAX + gi) * C::NCG + cg];
                    t.x += o.x;
                    t.y += o.y;
                    t.z += o.z;
                    t.w += o.w;
                }
                const int h = kvh * g + hg + gi;
                const size_t r = (size_t(b) * a.Hq + h) * per_head + idx;
                const bool empty = l_run[gi] == 0.f;  // no key reached this partial
                const float inv = empty ? 0.f : vscale / l_run[gi];
                reinterpret_cast<float4*>(o_dst + r * D)[cg] =
                    make_float4(t.x * inv, t.y * inv, t.z * inv, t.w * inv);
                if (cg == 0) lse_dst[r] = empty ? -INFINITY : m_run[gi] + log2f(l_run[gi]);
            }
        }
        __syncthreads();
    };
    // With one pass over each tile (all g heads at once) the stripe's chunks
    // are merged on the fly.  The running max, sum and accumulators carry on
    // from one chunk to the next (Step 2's merge, done online), and only the
    // stripe's own result is written: to the stripe partials of the single
    // launch, or as partial `stripe` of nstripes for the merge kernel.  A
    // paged stripe whose chunks all lie past its sequence's end leaves an
    // empty partial (O = 0, lse = -inf).
    const bool run_stripe = npass == 1;
    if (run_stripe) reset();

    for (int c = stripe; c < a.nc && ok; c += a.nstripes) {
        const int key0 = c * a.chunk;
        const int key1 = min(mb, key0 + a.chunk);
        if (key0 >= key1) {
            // a chunk past the end of a shorter (paged) sequence: an empty
            // partial, which the merge weighs with 2^-inf = 0 (nothing to add
            // when the stripe merges on the fly)
            for (int gi = 0; gi < g && !run_stripe; ++gi) {
                const size_t pr = (size_t(b) * a.Hq + kvh * g + gi) * a.nc + c;
                if (tid < NCP) reinterpret_cast<float2*>(a.o_part + pr * D)[tid] = make_float2(0.f, 0.f);
                if (tid == 0) a.lse_part[pr] = -INFINITY;
            }
            continue;
        }
        const int nsub = (key1 - key0 + C::TK - 1) / C::TK;
        for (int hg = 0; hg < g && ok; hg += GP) {
            // the tile is given back after its last use: after every pass when the
            // chunk spans several sub-tiles (each pass reloads them), else after the last
            const bool release = nsub > 1 || hg + GP >= g;
            if (!run_stripe) reset();

            for (int st = 0; st < nsub; ++st) {
                const int nk = min(C::TK, key1 - (key0 + st * C::TK));
                const int kslot = cn % C::NSLOT;
                const int vslot = (cn + 1) % C::NSLOT;
                const uint8_t* Ks = smem + kslot * C::TILE_BYTES;
                const uint8_t* Vs = smem + vslot * C::TILE_BYTES;
                bool got = mbar_wait(bar0 + 8 * kslot, uint32_t(cn / C::NSLOT) & 1u, wc,
                                     FA_SITE_DECODE_KV);
                if (!__syncthreads_and(got)) {
                    ok = false;
                    break;
                }
                // ---- scores: thread <-> key, full dot product from the swizzled K tile,
                // four partial sums per head (independent FMA chains); then the
                // max of each warp's 32 keys
                float tsc[GP];
                {
                    constexpr int CH = C::KBOX / 16;  // 16-byte chunks per K box row
                    constexpr int EPC = 16 / C::ESZ;  // elements per chunk
                    const int i = tid;
                    float s[GP][4];
#pragma unroll
                    for (int gi = 0; gi < GP; ++gi) s[gi][0] = s[gi][1] = s[gi][2] = s[gi][3] = 0.f;
#pragma unroll
                    for (int sub = 0; sub < C::NSUBK; ++sub) {
#pragma unroll
                        for (int ch = 0; ch < CH; ++ch) {
                            const uint4 w = *reinterpret_cast<const uint4*>(
                                Ks + sub * C::SUB_BYTES + i * C::KBOX + (C::kchunk(i, ch) << 4));
                            const int col = sub * (C::KBOX / C::ESZ) + ch * EPC;
                            if constexpr (C::QK_MIXED) {
                                // k as packed 16-bit pairs: kw[m] holds elements 2m, 2m+1
                                constexpr int NW = EPC / 2;
                                uint32_t kw[NW];
                                if constexpr (FP8) {
                                    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                                    for (int u = 0; u < 4; ++u) {
                                        kw[2 * u] = e4m3x2_to_f16x2(uint16_t(ww[u] & 0xffffu));
                                        kw[2 * u + 1] = e4m3x2_to_f16x2(uint16_t(ww[u] >> 16));
                                    }
                                } else {
                                    kw[0] = w.x;
                                    kw[1] = w.y;
                                    kw[2] = w.z;
                                    kw[3] = w.w;
                                }
                                const T* qb = reinterpret_cast<const T*>(qs) + (hg) * D + col;
#pragma unroll
                                for (int gi = 0; gi < GP; ++gi) {
#pragma unroll
                                    for (int m4 = 0; m4 < NW; m4 += 4) {
                                        const uint4 qw =
                                            *reinterpret_cast<const uint4*>(qb + gi * D + 2 * m4);
                                        mfma2<T>(s[gi][0], s[gi][1], kw[m4], qw.x);
                                        mfma2<T>(s[gi][2], s[gi][3], kw[m4 + 1], qw.y);
                                        mfma2<T>(s[gi][0], s[gi][1], kw[m4 + 2], qw.z);
                                        mfma2<T>(s[gi][2], s[gi][3], kw[m4 + 3], qw.w);
                                    }
                                }
                            } else {
                                float kf[EPC];
                                const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                                for (int u = 0; u < 4; ++u) {
                                    const float2 lo = e4m3x2_to_float2(uint16_t(ww[u] & 0xffffu));
                                    const float2 hi = e4m3x2_to_float2(uint16_t(ww[u] >> 16));
                                    kf[4 * u] = lo.x;
                                    kf[4 * u + 1] = lo.y;
                                    kf[4 * u + 2] = hi.x;
                                    kf[4 * u + 3] = hi.y;
                                }
                                const float* qb = qs + hg * D + col;
#pragma unroll
                                for (int gi = 0; gi < GP; ++gi) {
#pragma unroll
                                    for (int e4 = 0; e4 < EPC; e4 += 4) {
                                        const float4 qv =
                                            *reinterpret_cast<const float4*>(qb + gi * D + e4);
                                        s[gi][0] = fmaf(qv.x, kf[e4], s[gi][0]);
                                        s[gi][1] = fmaf(qv.y, kf[e4 + 1], s[gi][1]);
                                        s[gi][2] = fmaf(qv.z, kf[e4 + 2], s[gi][2]);
                                        s[gi][3] = fmaf(qv.w, kf[e4 + 3], s[gi][3]);
                                    }
                                }
                            }
                        }
                    }
#pragma unroll
                    for (int gi = 0; gi < GP; ++gi) {
                        const float t = (s[gi][0] + s[gi][1]) + (s[gi][2] + s[gi][3]);
                        tsc[gi] = i < nk ? t * sfac : -INFINITY;
                        float mx = tsc[gi];
#pragma unroll
                        for (int off = 16; off > 0; off >>= 1)
                            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
                        if (lane == 0) wmax[warp * C::GMAX + gi] = mx;
                    }
                }
                __syncthreads();
                // the K tile is consumed: refill its slot
                if (release && warp == 0) produce(cn + 1);
                // ---- softmax update: thread <-> key for every head (P of its own
                // score), the sub-tile max from the four warp maxima
#pragma unroll
                for (int gi = 0; gi < GP; ++gi) {
                    const float mx = fmaxf(fmaxf(wmax[gi], wmax[C::GMAX + gi]),
                                           fmaxf(wmax[2 * C::GMAX + gi], wmax[3 * C::GMAX + gi]));
                    const float m_new = fmaxf(m_run[gi], mx);
                    alpha[gi] = fast_exp2(m_run[gi] - m_new);  // 0 on the first sub-tile
                    m_run[gi] = m_new;
                    float p = fast_exp2(tsc[gi] - m_new);  // masked keys give exp2(-inf) = 0
                    if constexpr (C::PV_MIXED) {
                        // P.V takes P in f16; l sums the same rounded values
                        const __half hp = __float2half_rn(p);
                        ph[gi * C::TK + tid] = __half_as_ushort(hp);
                        p = __half2float(hp);
                    } else {
                        sc[gi * C::TK + tid] = p;
                    }
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) p += __shfl_xor_sync(0xffffffffu, p, off);
                    if (lane == 0) wsum[warp * C::GMAX + gi] = p;
                }
                got = mbar_wait(bar0 + 8 * vslot, uint32_t((cn + 1) / C::NSLOT) & 1u, wc,
                                FA_SITE_DECODE_KV);
                if (!__syncthreads_and(got)) {
                    ok = false;
                    break;
                }
                // ---- O_acc = alpha * O_acc + P V over this thread's key group and 4 columns
#pragma unroll
                for (int gi = 0; gi < GP; ++gi) {
                    const float al = alpha[gi];
                    l_run[gi] = l_run[gi] * al + ((wsum[gi] + wsum[C::GMAX + gi]) +
                                                  (wsum[2 * C::GMAX + gi] + wsum[3 * C::GMAX + gi]));
                    acc[gi].x *= al;
                    acc[gi].y *= al;
                    acc[gi].z *= al;
                    acc[gi].w *= al;
                    acc2[gi].x *= al;
                    acc2[gi].y *= al;
                    acc2[gi].z *= al;
                    acc2[gi].w *= al;
                }
                // columns 4cg .. 4cg+3 of V row j as two packed pairs (f16 on the mixed route)
                auto vquad = [&](int j) {
                    uint2 r;
                    if constexpr (FP8) {
                        const uint32_t w = *reinterpret_cast<const uint32_t*>(Vs + j * C::ROW_BYTES + cg * 4);
                        r.x = e4m3x2_to_f16x2(uint16_t(w & 0xffffu));
                        r.y = e4m3x2_to_f16x2(uint16_t(w >> 16));
                    } else {
                        r = *reinterpret_cast<const uint2*>(Vs + j * C::ROW_BYTES + cg * 8);
                    }
                    return r;
                };
                auto pv = [&](float4& o, uint2 vq, int gi, int j) {
                    if constexpr (C::PV_MIXED) {
                        const uint16_t pj = ph[gi * C::TK + j];
                        mfma2s_f16(o.x, o.y, vq.x, pj);
                        mfma2s_f16(o.z, o.w, vq.y, pj);
                    } else {
                        const float pj = sc[gi * C::TK + j];
                        const float2 a0 = unpack2<T>(vq.x), a1 = unpack2<T>(vq.y);
                        o.x = fmaf(pj, a0.x, o.x);
                        o.y = fmaf(pj, a0.y, o.y);
                        o.z = fmaf(pj, a1.x, o.z);
                        o.w = fmaf(pj, a1.y, o.w);
                    }
                };
                const int j0 = kq * C::KPG;
                const int j1 = min(j0 + C::KPG, nk);
                int j = j0;
#pragma unroll 2
                for (; j + 1 < j1; j += 2) {
                    const uint2 v0 = vquad(j), v1 = vquad(j + 1);
#pragma unroll
                    for (int gi = 0; gi < GP; ++gi) {
                        pv(acc[gi], v0, gi, j);
                        pv(acc2[gi], v1, gi, j + 1);
                    }
                }
                if (j < j1) {
                    const uint2 v0 = vquad(j);
#pragma unroll
                    for (int gi = 0; gi < GP; ++gi) pv(acc[gi], v0, gi, j);
                }
                __syncthreads();  // the V tile and the scores may be overwritten next
                if (release) {
                    if (warp == 0) produce(cn + 2);
                    cn += 2;
                }
            }
            if (!ok) break;
            // ---- the chunk partials of these heads (fp32, log2-domain lse)
            if (!run_stripe) write_partial(hg, a.o_part, a.lse_part, a.nc, c);
        }
    }
    if (run_stripe && ok)
        write_partial(0, FUSED ? a.g_o : a.o_part, FUSED ? a.g_lse : a.lse_part, a.nstripes, stripe);
    // every issued copy must have landed before the CTA exits (only a wait that
    // gave up leaves any outstanding)
    if (tid == 0) {
        for (int n = max(cn, issued - C::NSLOT); n < issued; ++n)
            mbar_drain_wait(bar0 + 8 * (n % C::NSLOT), uint32_t(n / C::NSLOT) & 1u, wc,
                            FA_SITE_DRAIN);
    }
    if constexpr (FUSED) {
        fused_stripe_tail<D, T>(a, ok, b, kvh, stripe, run_stripe);
    } else {
        // this CTA's partials are written: the merge grid may be scheduled
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    }
}

// Encodes the K and V maps the chunk kernel reads, over a 4-D view
// {d, Hkv, rows, outer} of the storage: [B, M, Hkv, d] (rows = M, outer = B)
// or a paged cache [num_pages, page, Hkv, d] (rows = page, outer = num_pages).
// K is read in swizzled boxes of KBOX bytes per row (so thread i reads key row
// i without bank conflicts), V as whole plain rows; box_rows keys per copy.
template <int D, typename T, bool FP8>
bool encode_kv_maps(EncodeTiledFn enc, const void* k, const void* v, int Hkv, int rows, int outer,
                    int box_rows, CUtensorMap* tk, CUtensorMap* tv) {
    using C = DecodeCfg<D, T, FP8>;
    const cuuint64_t esz = C::ESZ;
    const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)Hkv, (cuuint64_t)rows, (cuuint64_t)outer};
    const cuuint64_t strides[3] = {D * esz, (cuuint64_t)Hkv * D * esz,
                                   (cuuint64_t)rows * Hkv * D * esz};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUtensorMapDataType ty =
        FP8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
            : (DTypeFmt<T>::value == 0 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                       : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
    const cuuint32_t kbox[4] = {(cuuint32_t)(C::KBOX / C::ESZ), 1, (cuuint32_t)box_rows, 1};
    const cuuint32_t vbox[4] = {(cuuint32_t)D, 1, (cuuint32_t)box_rows, 1};
    const CUtensorMapSwizzle ksw =
        C::KBOX == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    if (enc(tk, ty, 4, const_cast<void*>(k), dims, strides, kbox, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, ksw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    return enc(tv, ty, 4, const_cast<void*>(v), dims, strides, vbox, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Dynamic shared memory a chunk kernel may need (227 KB, less its static
// shared memory, is what the device allows; a launch beyond it is refused).
constexpr size_t kMaxChunkSmem = size_t(227) * 1024;

// Launch attributes of one chunk-kernel variant, set once per device, so that
// a launch of any GQA group size needs no further set-up.
template <int D, typename T, bool FP8, bool PAGED, int GP, bool FUSED>
cudaError_t configure_chunk() {
    static std::atomic<unsigned> configured{0};
    return configure_kernel_once(chunk_kernel<D, T, FP8, PAGED, GP, FUSED>, configured);
}

template <int D, typename T, bool FP8, bool PAGED, int GP, bool FUSED>
cudaError_t launch_chunk(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a,
                         cudaStream_t stream, int* nstripes_out) {
    using C = DecodeCfg<D, T, FP8>;
    auto kern = chunk_kernel<D, T, FP8, PAGED, GP, FUSED>;
    const int g = a.Hq / a.Hkv;
    const size_t smem = C::smem_bytes(g);
    if (smem > kMaxChunkSmem) return cudaErrorInvalidConfiguration;
    cudaError_t err = configure_chunk<D, T, FP8, PAGED, GP, FUSED>();
    if (err != cudaSuccess) return err;
    // resident CTAs per SM for this shared-memory size (cached: it depends on g only)
    static std::atomic<long long> cached{-1};
    long long cv = cached.load(std::memory_order_relaxed);
    int occ = 0;
    if (cv >= 0 && (cv >> 8) == (long long)smem) {
        occ = int(cv & 0xff);
    } else {
        err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, C::THREADS, smem);
        if (err != cudaSuccess) return err;
        occ = occ < 1 ? 1 : (occ > 255 ? 255 : occ);
        cached.store(((long long)smem << 8) | occ, std::memory_order_relaxed);
    }
    int dev = 0, sms = 0;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
    if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return err;
    // one wave of persistent CTAs: every (b, kv head) gets the same number of
    // stripes, as many as fit (at least one)
    const long long nbh = (long long)a.B * a.Hkv;
    long long nstripes = (long long)occ * sms / nbh;
    nstripes = nstripes < 1 ? 1 : (nstripes > a.nc ? a.nc : nstripes);
    const long long nblocks = nbh * nstripes;
    if (nblocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    DecodeArgs la = a;
    la.nstripes = int(nstripes);
    *nstripes_out = la.nstripes;
    kern<<<dim3((unsigned)nblocks), dim3(C::THREADS), smem, stream>>>(tk, tv, la);
    return cudaGetLastError();
}

// The chunk kernel with GP dividing the GQA group, then (unless FUSED) the merge
// kernel as a programmatic dependent, so that its launch overlaps the chunk
// grid's tail; it waits for the data itself.  With one pass per tile (GP = g)
// the chunk kernel leaves one partial per stripe, so the merge kernel
// combines nstripes partials per (b, h) instead of nc.
template <int D, typename T, bool FP8, bool PAGED, bool FUSED>
cudaError_t launch(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a,
                   cudaStream_t stream) {
    const int g = a.Hq / a.Hkv;
    const int gp = (g % 4 == 0) ? 4 : (g % 2 == 0) ? 2 : 1;
    int nstripes = 0;
    cudaError_t err =
        gp == 4   ? launch_chunk<D, T, FP8, PAGED, 4, FUSED>(tk, tv, a, stream, &nstripes)
        : gp == 2 ? launch_chunk<D, T, FP8, PAGED, 2, FUSED>(tk, tv, a, stream, &nstripes)
                  : launch_chunk<D, T, FP8, PAGED, 1, FUSED>(tk, tv, a, stream, &nstripes);
    if (err != cudaSuccess || FUSED) return err;
    DecodeArgs ma = a;
    if (gp == g) ma.nc = nstripes;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(a.B * a.Hq, D / 16);
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, merge_kernel<D, T>, ma);
}

}  // namespace dec
}  // namespace fa

