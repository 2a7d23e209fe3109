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
//   * one CTA (128 threads) per (b, kv head, chunk) serves every query head of
//     the GQA group, so each K/V byte is read from HBM once; the block index is
//     ordered with (b, kv head) fastest so that CTAs running together read
//     whole contiguous key rows.  One thread issues TMA copies of the chunk's
//     K and V sub-tiles (128 keys) at CTA start; V streams in while the scores
//     are computed.
//   * scores: thread <-> key, the full dot product read from a swizzled K
//     tile (one 16-byte chunk per step, conflict-free); softmax per head by
//     one warp; P.V: thread <-> (column pair, key group).
//   * e4m3 K/V: the same tiles at one byte per element; the per-kv-head scales
//     are applied once per score (s = k_scale * q.k8) and once per output
//     (o = v_scale * sum_j p_j v8_j), which is exact algebra.
//   * paged K/V: rows of key j of batch b live in page block_table[b][j / P]
//     at row j % P of a [num_pages, P, Hkv, d] cache; a 128-key sub-tile is
//     fetched by one TMA copy per page it spans, and batch b only has
//     seq_lens[b] keys (chunks past the end write an empty partial).
#pragma once

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
    static constexpr int KQ = 256 / D;                  // key groups in the P.V step
    static constexpr int TILE_BYTES = TK * ROW_BYTES;
    static constexpr int K_OFF = 0;
    static constexpr int V_OFF = TILE_BYTES;
    static constexpr int QS_OFF = 2 * TILE_BYTES;                  // float [GMAX][D]
    static constexpr int SC_OFF = QS_OFF + GMAX * D * 4;           // float [GMAX][TK]
    static constexpr int RED_OFF = SC_OFF + GMAX * TK * 4;         // float2 [KQ-1][GMAX][D/2]
    static constexpr int HS_OFF = RED_OFF + (KQ - 1) * GMAX * D * 4;  // per head m, l, alpha
    static constexpr int BAR_OFF = HS_OFF + 3 * GMAX * 4;
    static constexpr int MISC_OFF = BAR_OFF + 16;
    static constexpr int SMEM_BYTES = MISC_OFF + 16 + 1024;        // + slack to align to 1 KB
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

// Merges n partial results (fp32 rows of D at rows + i*D, normalised, with
// log2-domain LSEs lse[i]) into one with the LSE weights of the page's Step 2:
// w_i = 2^(lse_i - glse), glse = log2 sum_i 2^lse_i.  128 threads; thread t < D
// owns column t.  Returns glse; writes the row to out_f (fp32) or out_t.  If
// every partial is empty (lse = -inf) the row is zero and glse is -inf.
template <int D, typename T>
__device__ float merge_partials(const float* lse, const float* rows, int n, float* red,
                                float* out_f, T* out_t) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    float mx = -INFINITY;
    for (int i = tid; i < n; i += 128) mx = fmaxf(mx, __ldcg(lse + i));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if (lane == 0) red[warp] = mx;
    __syncthreads();
    mx = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
    __syncthreads();
    const float ref = mx == -INFINITY ? 0.f : mx;
    float sm = 0.f;
    for (int i = tid; i < n; i += 128) sm += fast_exp2(__ldcg(lse + i) - ref);
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
                acc = fmaf(fast_exp2(__ldcg(lse + i) - glse), __ldcg(rows + size_t(i) * D + tid),
                           acc);
        }
        if (out_f != nullptr) out_f[tid] = acc;
        if (out_t != nullptr) out_t[tid] = static_cast<T>(acc);
    }
    return glse;
}

// Single launch (no merge kernel): the last CTA to finish a group of
// kDecodeMergeGroup chunks merges the group's partials; the last group merge of
// a (b, kv head) merges the group results into O and LSE.  Tickets are reset by
// whoever finishes them, so they are zero again when the kernel ends.
template <int D, typename T>
__device__ void fused_merge_tail(const DecodeArgs& a, bool ok, int b, int kvh, int c) {
    __shared__ int s_last;
    __shared__ float s_red[4];
    const int tid = threadIdx.x;
    const int g = a.Hq / a.Hkv;
    // The barrier orders every thread's partial stores before thread 0's
    // device-scope fence, which is cumulative; then the ticket.
    if (!__syncthreads_and(ok)) return;
    const int grp = c / kDecodeMergeGroup;
    const int c0 = grp * kDecodeMergeGroup;
    const int gsize = min(kDecodeMergeGroup, a.nc - c0);
    int* t1 = a.tickets + (size_t(b) * a.Hkv + kvh) * a.ngroups + grp;
    int* t2 = a.tickets + size_t(a.B) * a.Hkv * a.ngroups + (size_t(b) * a.Hkv + kvh);
    if (tid == 0) {
        __threadfence();
        s_last = atomicAdd(t1, 1) == gsize - 1;
        if (s_last) __threadfence();  // acquire: the others' partials are visible
    }
    __syncthreads();
    if (!s_last) return;
    for (int gi = 0; gi < g; ++gi) {
        const size_t bh = size_t(b) * a.Hq + kvh * g + gi;
        const size_t src = bh * a.nc + c0;
        const size_t dst = bh * a.ngroups + grp;
        const float glse = merge_partials<D, T>(a.lse_part + src, a.o_part + src * D, gsize, s_red,
                                                a.g_o + dst * D, nullptr);
        if (tid == 0) a.g_lse[dst] = glse;
        __syncthreads();
    }
    __syncthreads();
    if (tid == 0) {
        *t1 = 0;
        __threadfence();
        s_last = atomicAdd(t2, 1) == a.ngroups - 1;
        if (s_last) __threadfence();
    }
    __syncthreads();
    if (!s_last) return;
    for (int gi = 0; gi < g; ++gi) {
        const size_t bh = size_t(b) * a.Hq + kvh * g + gi;
        const float glse = merge_partials<D, T>(a.g_lse + bh * a.ngroups, a.g_o + bh * a.ngroups * D,
                                                a.ngroups, s_red, nullptr,
                                                reinterpret_cast<T*>(a.o) + bh * D);
        if (tid == 0 && a.lse != nullptr) a.lse[bh] = glse * kLn2;
        __syncthreads();
    }
    if (tid == 0) *t2 = 0;
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
// GP query heads per pass over the tile (the host picks GP dividing the GQA
// group).  FUSED: the chunk kernel also merges (single launch); only for
// contiguous 16-bit K/V.
template <int D, typename T, bool FP8, bool PAGED, int GP, bool FUSED>
__global__ void __launch_bounds__(128, 3)
    chunk_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                 const DecodeArgs a) {
    static_assert(!(FUSED && (FP8 || PAGED)), "the single launch is built for contiguous 16-bit K/V");
    using C = DecodeCfg<D, T, FP8>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const uint32_t sbase = smem_addr(smem);
    const uint32_t kbar = sbase + C::BAR_OFF;
    const uint32_t vbar = kbar + 8;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF);
    float* qs = reinterpret_cast<float*>(smem + C::QS_OFF);
    float* sc = reinterpret_cast<float*>(smem + C::SC_OFF);
    float2* red = reinterpret_cast<float2*>(smem + C::RED_OFF);
    float* hm = reinterpret_cast<float*>(smem + C::HS_OFF);
    float* hl = hm + C::GMAX;
    float* halpha = hl + C::GMAX;
    const uint8_t* Ks = smem + C::K_OFF;
    const uint8_t* Vs = smem + C::V_OFF;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    // Linear block index, (b, kv head) fastest: CTAs that run together read the
    // neighbouring heads of the same keys (whole contiguous key rows).
    const int nbh = a.B * a.Hkv;
    const int c = blockIdx.x / nbh;
    const int b = (blockIdx.x % nbh) / a.Hkv;
    const int kvh = blockIdx.x % a.Hkv;
    const int g = a.Hq / a.Hkv;
    const int mb = PAGED ? min(__ldg(a.seq_lens + b), a.M) : a.M;  // keys of this batch
    const int key0 = c * a.chunk;
    const int key1 = min(mb, key0 + a.chunk);
    constexpr int NCP = D / 2;

    if (key0 >= key1) {
        // a chunk past the end of a shorter (paged) sequence: an empty partial,
        // which the merge weighs with 2^-inf = 0
        for (int gi = 0; gi < g; ++gi) {
            const size_t pr = (size_t(b) * a.Hq + kvh * g + gi) * a.nc + c;
            if (tid < NCP) reinterpret_cast<float2*>(a.o_part + pr * D)[tid] = make_float2(0.f, 0.f);
            if (tid == 0) a.lse_part[pr] = -INFINITY;
        }
        return;
    }
    const int nsub = (key1 - key0 + C::TK - 1) / C::TK;

    if (tid == 0) {
        mbar_init(kbar, 1);
        mbar_init(vbar, 1);
        *abort_flag = 0;
        fence_barrier_init();
        prefetch_tensor_map(&tm_k);
        prefetch_tensor_map(&tm_v);
    }
    __syncthreads();
    const WaitCtl wc{abort_flag, a.status, a.timeout_ns};

    int loads = 0;  // sub-tiles loaded so far (the phase of both barriers)
    auto load_subtile = [&](int st) {
        if (tid == 0) {
            const int row = key0 + st * C::TK;
            if constexpr (!PAGED) {
                mbar_arrive_expect_tx(kbar, C::TILE_BYTES);
#pragma unroll
                for (int s = 0; s < C::NSUBK; ++s)
                    tma_load_4d(sbase + C::K_OFF + s * C::SUB_BYTES, &tm_k, s * (C::KBOX / C::ESZ),
                                kvh, row, b, kbar);
                mbar_arrive_expect_tx(vbar, C::TILE_BYTES);
                tma_load_4d(sbase + C::V_OFF, &tm_v, 0, kvh, row, b, vbar);
            } else {
                // one copy of R rows per page spanned; only the rows this chunk needs
                const int R = a.page < C::TK ? a.page : C::TK;
                const int nrows = min(C::TK, key1 - row);
                const int ncopy = (nrows + R - 1) / R;
                mbar_arrive_expect_tx(kbar, uint32_t(ncopy * R * C::ROW_BYTES));
                mbar_arrive_expect_tx(vbar, uint32_t(ncopy * R * C::ROW_BYTES));
                for (int r = 0; r < ncopy; ++r) {
                    const int key = row + r * R;
                    const int pg = __ldg(a.block_table + size_t(b) * a.max_pages + key / a.page);
                    const int prow = key % a.page;
#pragma unroll
                    for (int s = 0; s < C::NSUBK; ++s)
                        tma_load_4d(sbase + C::K_OFF + s * C::SUB_BYTES + r * R * C::KBOX, &tm_k,
                                    s * (C::KBOX / C::ESZ), kvh, prow, pg, kbar);
                    tma_load_4d(sbase + C::V_OFF + r * R * C::ROW_BYTES, &tm_v, 0, kvh, prow, pg,
                                vbar);
                }
            }
        }
        ++loads;
    };
    // The first sub-tile's copies go out before anything else.
    load_subtile(0);

    const float kscale = FP8 ? __ldg(a.k_scale + kvh) : 1.f;
    const float vscale = FP8 ? __ldg(a.v_scale + kvh) : 1.f;
    bool ok = true;
    // P.V mapping: thread <-> (column pair cp, key group kq)
    const int cp = tid % NCP;
    const int kq = tid / NCP;
    constexpr int KPG = C::TK / C::KQ;  // keys per group
    for (int hg = 0; hg < g && ok; hg += GP) {
        // this pass's query heads, as fp32 in shared memory (read as broadcasts)
        for (int e = tid; e < GP * D; e += C::THREADS) {
            const int gi = e / D, col = e % D;
            const int h = kvh * g + hg + gi;
            qs[e] = static_cast<float>(reinterpret_cast<const T*>(a.q)[(size_t(b) * a.Hq + h) * D + col]);
        }
        if (tid < C::GMAX) {
            hm[tid] = -INFINITY;
            hl[tid] = 0.f;
        }
        float2 acc[GP];
#pragma unroll
        for (int gi = 0; gi < GP; ++gi) acc[gi] = make_float2(0.f, 0.f);

        for (int st = 0; st < nsub; ++st) {
            const int ks = key0 + st * C::TK;
            const int nk = min(C::TK, key1 - ks);
            if (st > 0 || hg > 0) {
                // a chunk of one sub-tile keeps its tile resident across head groups
                if (nsub > 1) load_subtile(st);
            }
            const uint32_t ph = uint32_t(loads - 1) & 1u;
            bool got = mbar_wait(kbar, ph, wc, FA_SITE_DECODE_KV);
            if (!__syncthreads_and(got)) {
                ok = false;
                break;
            }
            // ---- scores: thread <-> key, full dot product from the swizzled K tile
            {
                constexpr int CH = C::KBOX / 16;  // 16-byte chunks per K box row
                constexpr int EPC = 16 / C::ESZ;  // elements per chunk
                const int i = tid;
                float s[GP];
#pragma unroll
                for (int gi = 0; gi < GP; ++gi) s[gi] = 0.f;
#pragma unroll
                for (int sub = 0; sub < C::NSUBK; ++sub) {
#pragma unroll
                    for (int ch = 0; ch < CH; ++ch) {
                        const uint4 w = *reinterpret_cast<const uint4*>(
                            Ks + sub * C::SUB_BYTES + i * C::KBOX + (C::kchunk(i, ch) << 4));
                        float kf[EPC];
                        if constexpr (FP8) {
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
                        } else {
                            unpack8<T>(w, kf);
                        }
                        const int col = sub * (C::KBOX / C::ESZ) + ch * EPC;
#pragma unroll
                        for (int gi = 0; gi < GP; ++gi) {
                            float t = s[gi];
#pragma unroll
                            for (int e4 = 0; e4 < EPC; e4 += 4) {
                                const float4 qv = *reinterpret_cast<const float4*>(qs + gi * D + col + e4);
                                t = fmaf(qv.x, kf[e4], t);
                                t = fmaf(qv.y, kf[e4 + 1], t);
                                t = fmaf(qv.z, kf[e4 + 2], t);
                                t = fmaf(qv.w, kf[e4 + 3], t);
                            }
                            s[gi] = t;
                        }
                    }
                }
                const float sfac = kscale * a.scale_log2;
#pragma unroll
                for (int gi = 0; gi < GP; ++gi) sc[gi * C::TK + i] = i < nk ? s[gi] * sfac : -INFINITY;
            }
            __syncthreads();
            // ---- softmax update of each head (one warp per head)
            for (int gi = warp; gi < GP; gi += 4) {
                float* srow = sc + gi * C::TK;
                float v[C::TK / 32];
                float mx = -INFINITY;
#pragma unroll
                for (int t = 0; t < C::TK / 32; ++t) {
                    v[t] = srow[lane + 32 * t];
                    mx = fmaxf(mx, v[t]);
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1)
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
                const float m_old = hm[gi];
                const float m_new = fmaxf(m_old, mx);
                const float alpha = fast_exp2(m_old - m_new);  // 0 on the first sub-tile
                float sum = 0.f;
#pragma unroll
                for (int t = 0; t < C::TK / 32; ++t) {
                    const float p = fast_exp2(v[t] - m_new);  // masked keys give exp2(-inf) = 0
                    srow[lane + 32 * t] = p;
                    sum += p;
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
                if (lane == 0) {
                    hm[gi] = m_new;
                    hl[gi] = hl[gi] * alpha + sum;
                    halpha[gi] = alpha;
                }
            }
            got = mbar_wait(vbar, ph, wc, FA_SITE_DECODE_KV);
            if (!__syncthreads_and(got)) {
                ok = false;
                break;
            }
            // ---- O_acc = alpha * O_acc + P V over this thread's key group and column pair
#pragma unroll
            for (int gi = 0; gi < GP; ++gi) {
                const float al = halpha[gi];
                acc[gi].x *= al;
                acc[gi].y *= al;
            }
            const int j0 = kq * KPG;
            const int j1 = min(j0 + KPG, nk);
#pragma unroll 4
            for (int j = j0; j < j1; ++j) {
                float2 vf;
                if constexpr (FP8)
                    vf = e4m3x2_to_float2(reinterpret_cast<const uint16_t*>(Vs)[j * NCP + cp]);
                else
                    vf = unpack2<T>(reinterpret_cast<const uint32_t*>(Vs)[j * NCP + cp]);
#pragma unroll
                for (int gi = 0; gi < GP; ++gi) {
                    const float p = sc[gi * C::TK + j];
                    acc[gi].x = fmaf(p, vf.x, acc[gi].x);
                    acc[gi].y = fmaf(p, vf.y, acc[gi].y);
                }
            }
            __syncthreads();  // the tile and the scores may be overwritten next
        }
        if (!ok) break;
        // ---- combine the key groups and write the chunk partials (fp32, log2-domain lse)
        if (kq > 0) {
#pragma unroll
            for (int gi = 0; gi < GP; ++gi) red[((kq - 1) * C::GMAX + gi) * NCP + cp] = acc[gi];
        }
        __syncthreads();
        if (kq == 0) {
#pragma unroll
            for (int gi = 0; gi < GP; ++gi) {
                float2 t = acc[gi];
#pragma unroll
                for (int u = 1; u < C::KQ; ++u) {
                    const float2 o = red[((u - 1) * C::GMAX + gi) * NCP + cp];
                    t.x += o.x;
                    t.y += o.y;
                }
                const int h = kvh * g + hg + gi;
                const size_t pr = (size_t(b) * a.Hq + h) * a.nc + c;
                const float inv = vscale / hl[gi];
                reinterpret_cast<float2*>(a.o_part + pr * D)[cp] = make_float2(t.x * inv, t.y * inv);
                if (cp == 0) a.lse_part[pr] = hm[gi] + log2f(hl[gi]);
            }
        }
        __syncthreads();
    }
    // every issued copy must have landed before the CTA exits
    if (tid == 0 && loads > 0) {
        mbar_drain_wait(kbar, uint32_t(loads - 1) & 1u, wc, FA_SITE_DRAIN);
        mbar_drain_wait(vbar, uint32_t(loads - 1) & 1u, wc, FA_SITE_DRAIN);
    }
    if constexpr (!FUSED) {
        // this CTA's partials are written: the merge grid may be scheduled
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    } else {
        fused_merge_tail<D, T>(a, ok, b, kvh, c);
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

template <int D, typename T, bool FP8, bool PAGED, int GP, bool FUSED>
cudaError_t launch_chunk(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a,
                         cudaStream_t stream) {
    using C = DecodeCfg<D, T, FP8>;
    auto kern = chunk_kernel<D, T, FP8, PAGED, GP, FUSED>;
    cudaError_t err =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (err != cudaSuccess) return err;
    const long long nblocks = (long long)a.nc * a.B * a.Hkv;
    if (nblocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    kern<<<dim3((unsigned)nblocks), dim3(C::THREADS), C::SMEM_BYTES, stream>>>(tk, tv, a);
    return cudaGetLastError();
}

// The chunk kernel with GP dividing the GQA group, then (unless FUSED) the merge
// kernel as a programmatic dependent, so that its launch overlaps the chunk
// grid's tail; it waits for the data itself.
template <int D, typename T, bool FP8, bool PAGED, bool FUSED>
cudaError_t launch(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a,
                   cudaStream_t stream) {
    const int g = a.Hq / a.Hkv;
    cudaError_t err = (g % 4 == 0)   ? launch_chunk<D, T, FP8, PAGED, 4, FUSED>(tk, tv, a, stream)
                      : (g % 2 == 0) ? launch_chunk<D, T, FP8, PAGED, 2, FUSED>(tk, tv, a, stream)
                                     : launch_chunk<D, T, FP8, PAGED, 1, FUSED>(tk, tv, a, stream);
    if (err != cudaSuccess || FUSED) return err;
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
    return cudaLaunchKernelEx(&cfg, merge_kernel<D, T>, a);
}

}  // namespace dec
}  // namespace fa

