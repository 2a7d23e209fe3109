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
    static constexpr int THREADS = 128;              // thread <-> key in the score step
    static constexpr int GMAX = 4;                   // query heads per pass over the tile
    static constexpr int NSUB = D / 64;              // 128-byte column halves of a K row
    static constexpr int SUB_BYTES = TK * 128;       // one swizzled K half-tile
    static constexpr int KQ = 256 / D;               // key groups in the P.V step
    static constexpr int TILE_BYTES = TK * D * 2;
    static constexpr int K_OFF = 0;                                // swizzled [NSUB][TK][64]
    static constexpr int V_OFF = TILE_BYTES;                       // plain [TK][D]
    static constexpr int QS_OFF = 2 * TILE_BYTES;                  // float [GMAX][D]
    static constexpr int SC_OFF = QS_OFF + GMAX * D * 4;           // float [GMAX][TK]
    static constexpr int RED_OFF = SC_OFF + GMAX * TK * 4;         // float2 [KQ-1][GMAX][D/2]
    static constexpr int HS_OFF = RED_OFF + (KQ - 1) * GMAX * D * 4;  // per head m, l, alpha
    static constexpr int BAR_OFF = HS_OFF + 3 * GMAX * 4;
    static constexpr int MISC_OFF = BAR_OFF + 16;
    static constexpr int SMEM_BYTES = MISC_OFF + 16 + 1024;        // + slack to align to 1 KB
};

template <typename T>
__device__ __forceinline__ void unpack8(const uint4& w, float (&f)[8]) {
    const float2 a = unpack2<T>(w.x), b = unpack2<T>(w.y), c = unpack2<T>(w.z), d = unpack2<T>(w.w);
    f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
    f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
}

// Merges n partial results (fp32 rows of D at rows + i*D, normalised, with
// log2-domain LSEs lse[i]) into one with the LSE weights of the page's Step 2:
// w_i = 2^(lse_i - glse), glse = log2 sum_i 2^lse_i.  128 threads; thread t < D
// owns column t.  Returns glse; writes the row to out_f (fp32) or out_t.
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
    float sm = 0.f;
    for (int i = tid; i < n; i += 128) sm += fast_exp2(__ldcg(lse + i) - mx);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sm += __shfl_xor_sync(0xffffffffu, sm, off);
    if (lane == 0) red[warp] = sm;
    __syncthreads();
    sm = red[0] + red[1] + red[2] + red[3];
    __syncthreads();
    const float glse = mx + log2f(sm);
    if (tid < D) {
        float acc = 0.f;
#pragma unroll 8
        for (int i = 0; i < n; ++i)
            acc = fmaf(fast_exp2(__ldcg(lse + i) - glse), __ldcg(rows + size_t(i) * D + tid), acc);
        if (out_f != nullptr) out_f[tid] = acc;
        if (out_t != nullptr) out_t[tid] = static_cast<T>(acc);
    }
    return glse;
}

template <int D, typename T, int GP, bool FUSED>
__global__ void __launch_bounds__(128, 3)
    decode_chunk_kernel(const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const DecodeArgs a) {
    using C = DecodeCfg<D>;
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
    const uint32_t* Vw = reinterpret_cast<const uint32_t*>(smem + C::V_OFF);  // pairs of T

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    // Linear block index, (b, kv head) fastest: CTAs that run together read the
    // neighbouring heads of the same keys, i.e. whole contiguous key rows of the
    // [B, M, Hkv, d] layout instead of one 2*d-byte slice every Hkv*d*2 bytes.
    const int nbh = a.B * a.Hkv;
    const int c = blockIdx.x / nbh;
    const int b = (blockIdx.x % nbh) / a.Hkv;
    const int kvh = blockIdx.x % a.Hkv;
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

    int loads = 0;  // sub-tiles loaded so far (the phase of both barriers)
    auto load_subtile = [&](int st) {
        if (tid == 0) {
            const int row = key0 + st * C::TK;
            mbar_arrive_expect_tx(kbar, C::TILE_BYTES);
#pragma unroll
            for (int s = 0; s < C::NSUB; ++s)
                tma_load_4d(sbase + C::K_OFF + s * C::SUB_BYTES, &tm_k, s * 64, kvh, row, b, kbar);
            mbar_arrive_expect_tx(vbar, C::TILE_BYTES);
            tma_load_4d(sbase + C::V_OFF, &tm_v, 0, kvh, row, b, vbar);
        }
        ++loads;
    };
    // The first sub-tile's copies go out before anything else.
    load_subtile(0);

    bool ok = true;
    // P.V mapping: thread <-> (column pair cp, key group kq)
    constexpr int NCP = D / 2;
    const int cp = tid % NCP;
    const int kq = tid / NCP;
    constexpr int KPG = C::TK / C::KQ;  // keys per group
    // GP query heads per pass; the host picks GP dividing the group size, so
    // every pass is full and no per-head predicate is needed
    for (int hg = 0; hg < g && ok; hg += GP) {
        constexpr int G = GP;
        // this pass's query heads, as fp32 in shared memory (read as broadcasts)
        for (int e = tid; e < GP * D; e += C::THREADS) {
            const int gi = e / D, col = e % D;
            float val = 0.f;
            if (gi < G) {
                const int h = kvh * g + hg + gi;
                val = static_cast<float>(
                    reinterpret_cast<const T*>(a.q)[(size_t(b) * a.Hq + h) * D + col]);
            }
            qs[e] = val;
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
                const int i = tid;
                float s[GP];
#pragma unroll
                for (int gi = 0; gi < GP; ++gi) s[gi] = 0.f;
#pragma unroll
                for (int half = 0; half < C::NSUB; ++half) {
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch) {
                        const uint4 w = *reinterpret_cast<const uint4*>(
                            Ks + half * C::SUB_BYTES + i * 128 + ((ch ^ (i & 7)) << 4));
                        float kf[8];
                        unpack8<T>(w, kf);
                        const int col = half * 64 + ch * 8;
#pragma unroll
                        for (int gi = 0; gi < GP; ++gi) {
                            if (gi < G) {
                                const float4 q0 = *reinterpret_cast<const float4*>(qs + gi * D + col);
                                const float4 q1 =
                                    *reinterpret_cast<const float4*>(qs + gi * D + col + 4);
                                float t = s[gi];
                                t = fmaf(q0.x, kf[0], t);
                                t = fmaf(q0.y, kf[1], t);
                                t = fmaf(q0.z, kf[2], t);
                                t = fmaf(q0.w, kf[3], t);
                                t = fmaf(q1.x, kf[4], t);
                                t = fmaf(q1.y, kf[5], t);
                                t = fmaf(q1.z, kf[6], t);
                                t = fmaf(q1.w, kf[7], t);
                                s[gi] = t;
                            }
                        }
                    }
                }
#pragma unroll
                for (int gi = 0; gi < GP; ++gi)
                    if (gi < G) sc[gi * C::TK + i] = i < nk ? s[gi] * a.scale_log2 : -INFINITY;
            }
            __syncthreads();
            // ---- softmax update of each head (one warp per head)
            for (int gi = warp; gi < G; gi += 4) {
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
                if (gi < G) {
                    const float al = halpha[gi];
                    acc[gi].x *= al;
                    acc[gi].y *= al;
                }
            }
            const int j0 = kq * KPG;
            const int j1 = min(j0 + KPG, nk);
#pragma unroll 4
            for (int j = j0; j < j1; ++j) {
                const float2 vf = unpack2<T>(Vw[j * NCP + cp]);
#pragma unroll
                for (int gi = 0; gi < GP; ++gi) {
                    if (gi < G) {
                        const float p = sc[gi * C::TK + j];
                        acc[gi].x = fmaf(p, vf.x, acc[gi].x);
                        acc[gi].y = fmaf(p, vf.y, acc[gi].y);
                    }
                }
            }
            __syncthreads();  // the tile and the scores may be overwritten next
        }
        if (!ok) break;
        // ---- combine the key groups and write the chunk partials (fp32, log2-domain lse)
        if (kq > 0) {
#pragma unroll
            for (int gi = 0; gi < GP; ++gi)
                if (gi < G) red[((kq - 1) * C::GMAX + gi) * NCP + cp] = acc[gi];
        }
        __syncthreads();
        if (kq == 0) {
#pragma unroll
            for (int gi = 0; gi < GP; ++gi) {
                if (gi < G) {
                    float2 t = acc[gi];
#pragma unroll
                    for (int u = 1; u < C::KQ; ++u) {
                        const float2 o = red[((u - 1) * C::GMAX + gi) * NCP + cp];
                        t.x += o.x;
                        t.y += o.y;
                    }
                    const int h = kvh * g + hg + gi;
                    const size_t pr = (size_t(b) * a.Hq + h) * a.nc + c;
                    const float inv = 1.f / hl[gi];
                    reinterpret_cast<float2*>(a.o_part + pr * D)[cp] = make_float2(t.x * inv, t.y * inv);
                    if (cp == 0) a.lse_part[pr] = hm[gi] + log2f(hl[gi]);
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
    if constexpr (!FUSED) {
        // this CTA's partials are written: the merge grid may be scheduled
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    } else {
        // Single launch (no merge kernel): the last CTA to finish a group of
        // kDecodeMergeGroup chunks merges the group's partials; the last group
        // merge of a (b, kv head) merges the group results into O and LSE.
        // Tickets are reset by whoever finishes them, so they are zero again
        // when the kernel ends.
        __shared__ int s_last;
        __shared__ float s_red[4];
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
            const float glse = merge_partials<D, T>(a.lse_part + src, a.o_part + src * D, gsize,
                                                    s_red, a.g_o + dst * D, nullptr);
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
            const float glse = merge_partials<D, T>(a.g_lse + bh * a.ngroups,
                                                    a.g_o + bh * a.ngroups * D, a.ngroups, s_red,
                                                    nullptr, reinterpret_cast<T*>(a.o) + bh * D);
            if (tid == 0 && a.lse != nullptr) a.lse[bh] = glse * kLn2;
            __syncthreads();
        }
        if (tid == 0) *t2 = 0;
    }
}

// One CTA of 128 threads per (b, h) and 16 output columns: thread t owns the
// float4 column group t % 4 and the chunks c = t / 4 (mod 32).
template <int D, typename T>
__global__ void __launch_bounds__(128) decode_merge_kernel(const DecodeArgs a) {
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
    float sm = 0.f;
    for (int cc = tid; cc < a.nc; cc += 128) sm += fast_exp2(lse_row[cc] - mx);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sm += __shfl_xor_sync(0xffffffffu, sm, off);
    if (lane == 0) red[warp] = sm;
    __syncthreads();
    sm = red[0] + red[1] + red[2] + red[3];
    const float glse = mx + log2f(sm);  // log2 domain

    const int cq = tid & 3;
    const float* src = o_rows + col0 + cq * 4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
    for (int cc = tid >> 2; cc < a.nc; cc += 32) {
        const float w = fast_exp2(lse_row[cc] - glse);
        const float4 v = *reinterpret_cast<const float4*>(src + size_t(cc) * D);
        acc.x = fmaf(w, v.x, acc.x);
        acc.y = fmaf(w, v.y, acc.y);
        acc.z = fmaf(w, v.z, acc.z);
        acc.w = fmaf(w, v.w, acc.w);
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

template <int D, typename T, int GP, bool FUSED = false>
cudaError_t launch_chunk(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a,
                         cudaStream_t stream) {
    using C = DecodeCfg<D>;
    auto kern = decode_chunk_kernel<D, T, GP, FUSED>;
    cudaError_t err =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (err != cudaSuccess) return err;
    const long long nblocks = (long long)a.nc * a.B * a.Hkv;
    if (nblocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    kern<<<dim3((unsigned)nblocks), dim3(C::THREADS), C::SMEM_BYTES, stream>>>(tk, tv, a);
    return cudaGetLastError();
}

template <int D, typename T>
cudaError_t launch_decode_t(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a,
                            cudaStream_t stream) {
    const int g = a.Hq / a.Hkv;
    cudaError_t err = (g % 4 == 0)   ? launch_chunk<D, T, 4>(tk, tv, a, stream)
                      : (g % 2 == 0) ? launch_chunk<D, T, 2>(tk, tv, a, stream)
                                     : launch_chunk<D, T, 1>(tk, tv, a, stream);
    if (err != cudaSuccess) return err;
    // the merge is launched as a programmatic dependent of the chunk grid so that
    // its launch overlaps the chunk grid's tail; it waits for the data itself
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
    return cudaLaunchKernelEx(&cfg, decode_merge_kernel<D, T>, a);
}

template <int D, typename T>
cudaError_t launch_decode_fused_t(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a,
                                  cudaStream_t stream) {
    const int g = a.Hq / a.Hkv;
    return (g % 4 == 0)   ? launch_chunk<D, T, 4, true>(tk, tv, a, stream)
           : (g % 2 == 0) ? launch_chunk<D, T, 2, true>(tk, tv, a, stream)
                          : launch_chunk<D, T, 1, true>(tk, tv, a, stream);
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
    // dims innermost first {d, heads, keys, batch}; K in 64-element (128-byte)
    // swizzled boxes so that thread i reads key row i without bank conflicts,
    // V as whole unswizzled rows (read row by row).
    const cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)Hkv, (cuuint64_t)M, (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)Hkv * d * 2,
                                   (cuuint64_t)M * Hkv * d * 2};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUtensorMapDataType ty =
        dtype == 0 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const cuuint32_t kbox[4] = {64, 1, (cuuint32_t)kDecodeSubTile, 1};
    const cuuint32_t vbox[4] = {(cuuint32_t)d, 1, (cuuint32_t)kDecodeSubTile, 1};
    if (enc(tk, ty, 4, const_cast<void*>(k), dims, strides, kbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    return enc(tv, ty, 4, const_cast<void*>(v), dims, strides, vbox, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

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

cudaError_t launch_decode_fused(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a,
                                int d, int dtype, cudaStream_t stream) {
    if (d == 128)
        return dtype == 0 ? launch_decode_fused_t<128, __half>(tk, tv, a, stream)
                          : launch_decode_fused_t<128, __nv_bfloat16>(tk, tv, a, stream);
    if (d == 64)
        return dtype == 0 ? launch_decode_fused_t<64, __half>(tk, tv, a, stream)
                          : launch_decode_fused_t<64, __nv_bfloat16>(tk, tv, a, stream);
    return cudaErrorInvalidValue;
}

cudaError_t launch_wait_selftest(int* status, unsigned long long timeout_ns, cudaStream_t stream) {
    wait_selftest_kernel<<<1, 32, 0, stream>>>(status, timeout_ns);
    return cudaGetLastError();
}

}  // namespace fa
