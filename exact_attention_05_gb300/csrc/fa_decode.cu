// fa_decode.cu -- split-KV flash decoding for sm_103a: a chunk kernel and an
// LSE-weighted merge kernel.
//
// What is computed follows "CUDA 实现 Flash Decoding：解码阶段并行度重建与性能剖析",
// section 2.2: for one query row per (b, h) the M keys are cut into chunks
// of `chunk` keys; Step 1 gives every chunk its own partial
//     m_c = max s,  P_c = exp(s - m_c),  l_c = sum P_c,
//     O_c = P_c V_c / l_c,  lse_c = m_c + log l_c,
// and Step 2 merges them with global_lse = m + log sum_c exp(lse_c - m) and
// weights w_c = exp(lse_c - global_lse), O = sum_c w_c O_c.  Section 3 fixes
// the two-kernel structure (grid over chunks x heads, then one reduction per
// head).  Logits and LSEs are kept in base 2 (scale * log2 e folded in),
// which changes no result.
//
// GB300 layout of the work (not the page's sm_89 kernels):
//   * chunk kernel: one CTA (128 threads) per (b, kv head, chunk) serves every
//     query head of the GQA group, so each K/V byte is read from HBM once.
//     One thread issues TMA bulk-tensor copies of the chunk's K and V
//     sub-tiles (128 keys x d) into shared memory at CTA start; V streams in
//     while the scores are computed.  Scores: a warp per key, lanes split d
//     (8-byte shared loads, conflict-free), warp-shuffle reduction.  Softmax
//     per head by one warp.  P.V: thread <-> output column (d = 128) or
//     (column, key half) (d = 64).  Chunks longer than 128 keys are walked
//     in sub-tiles with the running max / sum rescaled between them.
//     Partials are fp32: O_c [B, Hq, nc, d], lse_c [B, Hq, nc].
//   * merge kernel: one CTA per (b, h, 32 output columns); the lse row is
//     reduced block-wide, the weighted sum is read as float4 rows.

#include <cfloat>
#include <cmath>

#include "fa_device.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

constexpr float kLn2 = 0.6931471805599453f;

template <int D>
struct DecodeCfg {
    static constexpr int TK = kDecodeSubTile;        // keys per sub-tile (TMA box rows)
    static constexpr int THREADS = 128;
    static constexpr int GMAX = 8;                   // query heads per pass over the tile
    static constexpr int EPL = D / 32;               // elements of a key row per lane
    static constexpr int KG = 128 / D;               // key groups in the P.V step
    static constexpr int TILE_BYTES = TK * D * 2;
    static constexpr int K_OFF = 0;
    static constexpr int V_OFF = TILE_BYTES;
    static constexpr int SC_OFF = 2 * TILE_BYTES;                 // float [GMAX][TK]
    static constexpr int RED_OFF = SC_OFF + GMAX * TK * 4;        // float [GMAX][KG][D]
    static constexpr int HS_OFF = RED_OFF + GMAX * KG * D * 4;    // per head m, l, alpha
    static constexpr int BAR_OFF = HS_OFF + 3 * GMAX * 4;
    static constexpr int MISC_OFF = BAR_OFF + 16;
    static constexpr int SMEM_BYTES = MISC_OFF + 16 + 128;        // + slack to align to 128 B
};

template <int D, typename T>
__global__ void __launch_bounds__(128)
    decode_chunk_kernel(const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const DecodeArgs a) {
    using C = DecodeCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                               ~uintptr_t(127));
    const uint32_t sbase = smem_addr(smem);
    const uint32_t kbar = sbase + C::BAR_OFF;
    const uint32_t vbar = kbar + 8;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF);
    float* sc = reinterpret_cast<float*>(smem + C::SC_OFF);
    float* red = reinterpret_cast<float*>(smem + C::RED_OFF);
    float* hm = reinterpret_cast<float*>(smem + C::HS_OFF);
    float* hl = hm + C::GMAX;
    float* halpha = hl + C::GMAX;
    const T* Ks = reinterpret_cast<const T*>(smem + C::K_OFF);
    const T* Vs = reinterpret_cast<const T*>(smem + C::V_OFF);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int c = blockIdx.x;
    const int b = blockIdx.y / a.Hkv;
    const int kvh = blockIdx.y % a.Hkv;
    const int g = a.Hq / a.Hkv;
    const int key0 = c * a.chunk;
    const int key1 = min(a.M, key0 + a.chunk);
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

    int loads = 0;  // sub-tiles loaded so far (phase of both barriers)
    auto load_subtile = [&](int st) {
        if (tid == 0) {
            mbar_arrive_expect_tx(kbar, C::TILE_BYTES);
            tma_load_4d(sbase + C::K_OFF, &tm_k, 0, kvh, key0 + st * C::TK, b, kbar);
            mbar_arrive_expect_tx(vbar, C::TILE_BYTES);
            tma_load_4d(sbase + C::V_OFF, &tm_v, 0, kvh, key0 + st * C::TK, b, vbar);
        }
        ++loads;
    };

    bool ok = true;
    const int col = tid % D;       // output column of this thread in the P.V step
    const int kg = tid / D;        // its key group
    for (int hg = 0; hg < g && ok; hg += C::GMAX) {
        const int G = min(C::GMAX, g - hg);
        // this pass's query heads, kept in fp32 registers: lane holds EPL elements
        float qf[C::GMAX][C::EPL];
#pragma unroll
        for (int gi = 0; gi < C::GMAX; ++gi) {
            if (gi < G) {
                const int h = kvh * g + hg + gi;
                const T* qrow = reinterpret_cast<const T*>(a.q) + (size_t(b) * a.Hq + h) * D;
#pragma unroll
                for (int e = 0; e < C::EPL; e += 2) {
                    const float2 f =
                        unpack2<T>(*reinterpret_cast<const uint32_t*>(qrow + lane * C::EPL + e));
                    qf[gi][e] = f.x;
                    qf[gi][e + 1] = f.y;
                }
            }
        }
        if (tid < C::GMAX) {
            hm[tid] = -INFINITY;
            hl[tid] = 0.f;
        }
        float acc[C::GMAX];
#pragma unroll
        for (int gi = 0; gi < C::GMAX; ++gi) acc[gi] = 0.f;

        for (int st = 0; st < nsub; ++st) {
            const int ks = key0 + st * C::TK;
            const int nk = min(C::TK, key1 - ks);
            // the tile of a single-sub-tile chunk stays resident across head groups
            const bool need_load = (hg == 0) || (nsub > 1);
            if (need_load) load_subtile(st);
            const uint32_t ph = uint32_t(loads - 1) & 1u;
            bool got = mbar_wait(kbar, ph, wc, FA_SITE_DECODE_KV);
            if (!__syncthreads_and(got)) {
                ok = false;
                break;
            }
            // ---- scores s = scale * log2(e) * q . k, one warp per key
            for (int i = warp; i < nk; i += 4) {
                const T* krow = Ks + i * D + lane * C::EPL;
                float kf[C::EPL];
                if constexpr (C::EPL == 4) {
                    const uint2 w = *reinterpret_cast<const uint2*>(krow);
                    const float2 f0 = unpack2<T>(w.x), f1 = unpack2<T>(w.y);
                    kf[0] = f0.x; kf[1] = f0.y; kf[2] = f1.x; kf[3] = f1.y;
                } else {
                    const float2 f0 = unpack2<T>(*reinterpret_cast<const uint32_t*>(krow));
                    kf[0] = f0.x; kf[1] = f0.y;
                }
#pragma unroll
                for (int gi = 0; gi < C::GMAX; ++gi) {
                    if (gi < G) {
                        float part = 0.f;
#pragma unroll
                        for (int e = 0; e < C::EPL; ++e) part = fmaf(qf[gi][e], kf[e], part);
#pragma unroll
                        for (int off = 16; off > 0; off >>= 1)
                            part += __shfl_xor_sync(0xffffffffu, part, off);
                        if (lane == 0) sc[gi * C::TK + i] = part * a.scale_log2;
                    }
                }
            }
            __syncthreads();
            // ---- softmax update of each head (one warp per head)
            for (int gi = warp; gi < G; gi += 4) {
                float* srow = sc + gi * C::TK;
                float v[C::TK / 32];
                float mx = -INFINITY;
#pragma unroll
                for (int t = 0; t < C::TK / 32; ++t) {
                    const int i = lane + 32 * t;
                    v[t] = i < nk ? srow[i] : -INFINITY;
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
                    const int i = lane + 32 * t;
                    const float p = i < nk ? fast_exp2(v[t] - m_new) : 0.f;
                    srow[i] = p;
                    sum += p;
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
                __syncwarp();
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
            // ---- O_acc = alpha * O_acc + P V
#pragma unroll
            for (int gi = 0; gi < C::GMAX; ++gi)
                if (gi < G) acc[gi] *= halpha[gi];
            for (int i = kg; i < nk; i += C::KG) {
                const float vf = static_cast<float>(Vs[i * D + col]);
#pragma unroll
                for (int gi = 0; gi < C::GMAX; ++gi)
                    if (gi < G) acc[gi] = fmaf(sc[gi * C::TK + i], vf, acc[gi]);
            }
            __syncthreads();  // the tile and scores may be overwritten next
        }
        if (!ok) break;
        // ---- combine key groups and write the chunk partials (fp32, log2-domain lse)
        if constexpr (C::KG > 1) {
#pragma unroll
            for (int gi = 0; gi < C::GMAX; ++gi)
                if (gi < G) red[(gi * C::KG + kg) * D + col] = acc[gi];
            __syncthreads();
            if (kg == 0) {
#pragma unroll
                for (int gi = 0; gi < C::GMAX; ++gi) {
                    if (gi < G) {
                        float t = 0.f;
#pragma unroll
                        for (int u = 0; u < C::KG; ++u) t += red[(gi * C::KG + u) * D + col];
                        acc[gi] = t;
                    }
                }
            }
        }
        if (kg == 0) {
#pragma unroll
            for (int gi = 0; gi < C::GMAX; ++gi) {
                if (gi < G) {
                    const int h = kvh * g + hg + gi;
                    const size_t pr = (size_t(b) * a.Hq + h) * a.nc + c;
                    a.o_part[pr * D + col] = acc[gi] / hl[gi];
                    if (col == 0) a.lse_part[pr] = hm[gi] + log2f(hl[gi]);
                }
            }
        }
        __syncthreads();
    }
    // every issued copy must have landed before the CTA exits
    if (tid == 0 && loads > 0) {
        mbar_drain_wait(kbar, uint32_t(loads - 1) & 1u, wc, FA_SITE_DRAIN);
        mbar_drain_wait(vbar, uint32_t(loads - 1) & 1u, wc, FA_SITE_DRAIN);
    }
}

// Block-wide max and sum over 256 threads (8 warps).
__device__ __forceinline__ float block_max_256(float v, float* red) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float r = red[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) r = fmaxf(r, red[w]);
    __syncthreads();
    return r;
}

__device__ __forceinline__ float block_sum_256(float v, float* red) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float r = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) r += red[w];
    __syncthreads();
    return r;
}

template <int D, typename T>
__global__ void __launch_bounds__(256) decode_merge_kernel(const DecodeArgs a) {
    __shared__ float red[8];
    __shared__ float4 part[8][32];
    const int bh = blockIdx.x;
    const int col0 = blockIdx.y * 32;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const float* lse_row = a.lse_part + size_t(bh) * a.nc;
    const float* o_rows = a.o_part + size_t(bh) * a.nc * D;

    float mx = -INFINITY;
    for (int cc = tid; cc < a.nc; cc += 256) mx = fmaxf(mx, lse_row[cc]);
    mx = block_max_256(mx, red);
    float sm = 0.f;
    for (int cc = tid; cc < a.nc; cc += 256) sm += fast_exp2(lse_row[cc] - mx);
    sm = block_sum_256(sm, red);
    const float glse = mx + log2f(sm);  // log2 domain

    // lane -> (4 columns, one of 4 chunks); warp -> chunk offset; 32 chunks per step
    const int cq = lane & 7;
    const int csub = lane >> 3;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
    for (int cc = warp * 4 + csub; cc < a.nc; cc += 32) {
        const float w = fast_exp2(lse_row[cc] - glse);
        const float4 v = *reinterpret_cast<const float4*>(o_rows + size_t(cc) * D + col0 + cq * 4);
        acc.x = fmaf(w, v.x, acc.x);
        acc.y = fmaf(w, v.y, acc.y);
        acc.z = fmaf(w, v.z, acc.z);
        acc.w = fmaf(w, v.w, acc.w);
    }
#pragma unroll
    for (int off = 8; off < 32; off <<= 1) {
        acc.x += __shfl_xor_sync(0xffffffffu, acc.x, off);
        acc.y += __shfl_xor_sync(0xffffffffu, acc.y, off);
        acc.z += __shfl_xor_sync(0xffffffffu, acc.z, off);
        acc.w += __shfl_xor_sync(0xffffffffu, acc.w, off);
    }
    if (csub == 0) part[warp][cq] = acc;
    __syncthreads();
    if (tid < 8) {
        float4 t = part[0][tid];
#pragma unroll
        for (int w = 1; w < 8; ++w) {
            t.x += part[w][tid].x;
            t.y += part[w][tid].y;
            t.z += part[w][tid].z;
            t.w += part[w][tid].w;
        }
        T* orow = reinterpret_cast<T*>(a.o) + size_t(bh) * D + col0 + tid * 4;
        const uint2 packed = make_uint2(pack2<T>(t.x, t.y), pack2<T>(t.z, t.w));
        *reinterpret_cast<uint2*>(orow) = packed;
    }
    if (tid == 0 && blockIdx.y == 0 && a.lse != nullptr) a.lse[bh] = glse * kLn2;
}

template <int D, typename T>
cudaError_t launch_decode_t(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a,
                            cudaStream_t stream) {
    using C = DecodeCfg<D>;
    auto chunk_kern = decode_chunk_kernel<D, T>;
    cudaError_t err = cudaFuncSetAttribute(chunk_kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           C::SMEM_BYTES);
    if (err != cudaSuccess) return err;
    chunk_kern<<<dim3(a.nc, a.B * a.Hkv), dim3(C::THREADS), C::SMEM_BYTES, stream>>>(tk, tv, a);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    decode_merge_kernel<D, T><<<dim3(a.B * a.Hq, D / 32), dim3(256), 0, stream>>>(a);
    return cudaGetLastError();
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

cudaError_t launch_decode(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a, int d,
                          int dtype, cudaStream_t stream) {
    if (d == 128)
        return dtype == 0 ? launch_decode_t<128, __half>(tk, tv, a, stream)
                          : launch_decode_t<128, __nv_bfloat16>(tk, tv, a, stream);
    if (d == 64)
        return dtype == 0 ? launch_decode_t<64, __half>(tk, tv, a, stream)
                          : launch_decode_t<64, __nv_bfloat16>(tk, tv, a, stream);
    return cudaErrorInvalidValue;
}

cudaError_t launch_wait_selftest(int* status, unsigned long long timeout_ns, cudaStream_t stream) {
    wait_selftest_kernel<<<1, 32, 0, stream>>>(status, timeout_ns);
    return cudaGetLastError();
}

}  // namespace fa
