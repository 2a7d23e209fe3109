// fa_backward.cu -- backward of exact attention (dQ, dK, dV) for sm_103a.
//
// What is computed: the gradients of O = softmax(scale Q K^T [+ causal]) V
// for an upstream gradient dO.  "Tensor Core 迁移计划" (phase 2) names the
// backward's contractions: dV = P^T dO, dP = dO V^T, and dQ, dK from dS.  The
// softmax's Jacobian gives dS = P o (dP - D) with D_i = sum_j P_ij dP_ij, which
// equals dO_i . O_i (O_i = sum_j P_ij V_j); then dQ = scale dS K and
// dK = scale dS^T Q.  P is recomputed from the forward's per-row LSE:
// P_ij = exp(scale q_i . k_j - LSE_i), so nothing of size N x M is stored.
//
// How it runs on GB300 (three launches on the caller's stream):
//   1. dsum_kernel: D_i = dO_i . O_i in fp32 for every row, and zeroes the
//      fp32 dQ accumulator.
//   2. backward_kernel: one CTA per (b, kv head, 128-key tile j) keeps K_j
//      and V_j in shared memory and walks the 128-row Q tiles that see them
//      (from tile j on when causal), for every query head of the GQA group:
//        warp 4   TMA producer: K_j, V_j once; then Q_i and dO_i per tile;
//        warp 5   TMEM allocator and single-thread tcgen05 MMA issuer;
//        warps 0-3 thread r <-> TMEM lane r: query row r for S, dP and dQ,
//                 key row r for the final dK, dV.
//      Per Q tile:  S = Q K^T and dP = dO V^T (fp32 in TMEM); the compute
//      warps form P and dS in 16-bit, in 128-byte-swizzled shared-memory
//      tiles; then dV += P^T dO and dK += dS^T Q accumulate in TMEM (P and dS
//      read MN-major, i.e. transposed, by the tensor core), and dQ = dS K lands
//      in the columns of S, from where the compute warps add it to the fp32
//      accumulator in global memory with vector reductions.  TMEM (512
//      columns): S [0,128) (dQ over its first d), dP [128,256), dV [256,256+d),
//      dK [256+d, 256+2d).
//   3. dq_convert_kernel: dQ = scale * accumulator, rounded to the input type.
// Every wait is bounded; on expiry the CTA records the timeout, drains its own
// copies and MMAs, frees TMEM and returns.

#include <cfloat>
#include <cmath>

#include "fa_device.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

template <int D>
struct BwdCfg {
    static constexpr int BM = 128;                        // query rows per Q tile
    static constexpr int BN = 128;                        // keys per CTA
    static constexpr int NSUB = D / 64;                   // 64-element (128 B) column halves
    static constexpr int SUB_BYTES = 128 * 128;           // 128 rows x 128 B
    static constexpr int TILE_BYTES = NSUB * SUB_BYTES;   // a [128][D] tile
    static constexpr int PS_BYTES = 2 * SUB_BYTES;        // a [128][128] tile (P or dS)
    static constexpr int K_OFF = 0;
    static constexpr int V_OFF = K_OFF + TILE_BYTES;
    static constexpr int Q_OFF = V_OFF + TILE_BYTES;
    static constexpr int DO_OFF = Q_OFF + TILE_BYTES;
    static constexpr int P_OFF = DO_OFF + TILE_BYTES;
    static constexpr int DS_OFF = P_OFF + PS_BYTES;
    static constexpr int BAR_OFF = DS_OFF + PS_BYTES;
    // barriers
    static constexpr int B_KV = 0;      // K_j, V_j landed
    static constexpr int B_QFULL = 1;   // Q_i, dO_i landed
    static constexpr int B_QFREE = 2;   // the MMAs reading Q_i, dO_i are done
    static constexpr int B_S = 3;       // S in TMEM
    static constexpr int B_DP = 4;      // dP in TMEM
    static constexpr int B_P = 5;       // P, dS in shared memory (128 arrivals)
    static constexpr int B_DQ = 6;      // dQ in TMEM (and every earlier MMA done)
    static constexpr int B_SFREE = 7;   // dQ read out of TMEM (128 arrivals)
    static constexpr int B_FINAL = 8;   // every MMA done: dK, dV final
    static constexpr int NBAR = 9;
    static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
    static constexpr int SMEM_BYTES = MISC_OFF + 16 + 1024;  // + slack to align the base to 1 KB
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t TM_S = 0, TM_DQ = 0, TM_DP = 128, TM_DV = 256, TM_DK = 256 + D;
    static_assert(256 + 2 * D <= 512, "TMEM budget");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

constexpr int kBwdThreads = 192;
constexpr float kLog2e = 1.4426950408889634f;

// D_i = dO_i . O_i (fp32) for every (b, q, h) row, one warp per row; the same
// warp zeroes the row's fp32 dQ accumulator.
template <int D, typename T>
__global__ void __launch_bounds__(256) dsum_kernel(const BackwardArgs a) {
    constexpr int EPL = D / 32;  // elements per lane (2 or 4)
    const long long rows = (long long)a.B * a.N * a.Hq;
    const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const T* o = reinterpret_cast<const T*>(a.o) + row * D + lane * EPL;
    const T* g = reinterpret_cast<const T*>(a.dout) + row * D + lane * EPL;
    float acc = 0.f;
    if constexpr (EPL == 4) {
        const uint2 ov = *reinterpret_cast<const uint2*>(o);
        const uint2 gv = *reinterpret_cast<const uint2*>(g);
        const float2 o0 = unpack2<T>(ov.x), o1 = unpack2<T>(ov.y);
        const float2 g0 = unpack2<T>(gv.x), g1 = unpack2<T>(gv.y);
        acc = fmaf(o0.x, g0.x, fmaf(o0.y, g0.y, fmaf(o1.x, g1.x, o1.y * g1.y)));
    } else {
        const float2 o0 = unpack2<T>(*reinterpret_cast<const uint32_t*>(o));
        const float2 g0 = unpack2<T>(*reinterpret_cast<const uint32_t*>(g));
        acc = fmaf(o0.x, g0.x, o0.y * g0.y);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    // row = (b * N + q) * Hq + h  ->  dsum[(b * Hq + h) * N + q]
    const long long h = row % a.Hq;
    const long long bq = row / a.Hq;
    const long long q = bq % a.N, b = bq / a.N;
    if (lane == 0) a.dsum[(b * a.Hq + h) * a.N + q] = acc;
    float* acc_row = a.dq_acc + row * D + lane * EPL;
    if constexpr (EPL == 4)
        *reinterpret_cast<float4*>(acc_row) = make_float4(0.f, 0.f, 0.f, 0.f);
    else
        *reinterpret_cast<float2*>(acc_row) = make_float2(0.f, 0.f);
}

// dQ = scale * accumulator, rounded to T; four elements per thread.
template <typename T>
__global__ void __launch_bounds__(256) dq_convert_kernel(const BackwardArgs a, long long n4) {
    const long long i = (long long)blockIdx.x * 256 + threadIdx.x;
    if (i >= n4) return;
    const float4 v = reinterpret_cast<const float4*>(a.dq_acc)[i];
    const float s = a.scale;
    reinterpret_cast<uint2*>(a.dq)[i] = make_uint2(pack2<T>(v.x * s, v.y * s), pack2<T>(v.z * s, v.w * s));
}

__device__ __forceinline__ void red_add_v4(float* p, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c),
                 "f"(d)
                 : "memory");
}

template <int D, typename T>
__global__ void __launch_bounds__(kBwdThreads, 1)
    backward_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const BackwardArgs a) {
    using C = BwdCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const uint32_t sbase = smem_addr(smem);
    const uint32_t bars = sbase + C::BAR_OFF;
    volatile uint32_t* tmem_holder = reinterpret_cast<volatile uint32_t*>(smem + C::MISC_OFF);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 4);
    auto bar = [&](int i) -> uint32_t { return bars + 8u * uint32_t(i); };
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // block -> (key tile j, b, kv head); j = 0 (the most Q tiles when causal) first
    const int nbh = a.B * a.Hkv;
    const int j = blockIdx.x / nbh;
    const int b = (blockIdx.x % nbh) / a.Hkv;
    const int kvh = blockIdx.x % a.Hkv;
    const int g = a.Hq / a.Hkv;
    const int key0 = j * C::BN;
    // first Q tile with a row that sees key0 (top-left causal: key k visible to row q iff k <= q)
    const int i0 = a.causal ? key0 / C::BM : 0;
    const int nq = a.n_qtiles > i0 ? a.n_qtiles - i0 : 0;
    const int ntile = g * nq;  // (query head, Q tile) pairs this CTA walks
    auto tile_of = [&](int t, int& h, int& i) {
        h = kvh * g + t / nq;
        i = i0 + t % nq;
    };

    if (threadIdx.x == 0) {
        mbar_init(bar(C::B_KV), 1);
        mbar_init(bar(C::B_QFULL), 1);
        mbar_init(bar(C::B_QFREE), 1);
        mbar_init(bar(C::B_S), 1);
        mbar_init(bar(C::B_DP), 1);
        mbar_init(bar(C::B_P), 128);
        mbar_init(bar(C::B_DQ), 1);
        mbar_init(bar(C::B_SFREE), 128);
        mbar_init(bar(C::B_FINAL), 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 4 && lane == 0) {
        prefetch_tensor_map(&tm_q);
        prefetch_tensor_map(&tm_k);
        prefetch_tensor_map(&tm_v);
        prefetch_tensor_map(&tm_do);
    }
    if (warp == 5) {
        tmem_alloc(smem_addr(const_cast<uint32_t*>(tmem_holder)), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const WaitCtl wc{abort_flag, a.status, a.timeout_ns};

    if (warp == 4) {
        // ------------------------------------------------------------- producer
        if (lane == 0 && ntile > 0) {
            mbar_arrive_expect_tx(bar(C::B_KV), 2 * C::TILE_BYTES);
            for (int s = 0; s < C::NSUB; ++s) {
                tma_load_4d(sbase + C::K_OFF + s * C::SUB_BYTES, &tm_k, s * 64, kvh, key0, b, bar(C::B_KV));
                tma_load_4d(sbase + C::V_OFF + s * C::SUB_BYTES, &tm_v, s * 64, kvh, key0, b, bar(C::B_KV));
            }
            int t = 0;
            for (; t < ntile; ++t) {
                if (t > 0 && !mbar_wait(bar(C::B_QFREE), (t - 1) & 1, wc, FA_SITE_PRODUCER_SLOT)) break;
                int h, i;
                tile_of(t, h, i);
                mbar_arrive_expect_tx(bar(C::B_QFULL), 2 * C::TILE_BYTES);
                for (int s = 0; s < C::NSUB; ++s) {
                    tma_load_4d(sbase + C::Q_OFF + s * C::SUB_BYTES, &tm_q, s * 64, h, i * C::BM, b,
                                bar(C::B_QFULL));
                    tma_load_4d(sbase + C::DO_OFF + s * C::SUB_BYTES, &tm_do, s * 64, h, i * C::BM, b,
                                bar(C::B_QFULL));
                }
            }
            // every issued copy must have landed before the CTA may exit
            mbar_drain_wait(bar(C::B_KV), 0, wc, FA_SITE_DRAIN);
            if (t > 0) mbar_drain_wait(bar(C::B_QFULL), (t - 1) & 1, wc, FA_SITE_DRAIN);
        }
    } else if (warp == 5) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0 && ntile > 0) {
            constexpr uint32_t fmt = DTypeFmt<T>::value;
            constexpr uint32_t id_kk = instr_desc_f16(fmt, 128, 128, 0, 0);  // S, dP: both K-major
            constexpr uint32_t id_mn = instr_desc_f16(fmt, 128, D, 1, 1);    // dV, dK: P^T/dS^T, dO/Q MN-major
            constexpr uint32_t id_km = instr_desc_f16(fmt, 128, D, 0, 1);    // dQ: dS K-major, K MN-major
            // K-major (128-byte swizzle): a 16-element k-step advances 32 bytes inside a
            // 64-column half, halves are SUB_BYTES apart, 8-row groups 1024 bytes apart.
            // MN-major: a 16-row k-step advances 16 x 128 bytes; the 64-wide halves of the
            // M or N extent are SUB_BYTES apart (leading offset), 8-row groups 1024 bytes.
            auto koff = [](int kk) -> uint64_t {
                return uint64_t((kk / 4) * C::SUB_BYTES + (kk % 4) * 32) >> 4;
            };
            auto moff = [](int kk) -> uint64_t { return uint64_t(kk * 16 * 128) >> 4; };
            const uint64_t q_k = smem_desc(sbase + C::Q_OFF, 16, 1024);
            const uint64_t k_k = smem_desc(sbase + C::K_OFF, 16, 1024);
            const uint64_t do_k = smem_desc(sbase + C::DO_OFF, 16, 1024);
            const uint64_t v_k = smem_desc(sbase + C::V_OFF, 16, 1024);
            const uint64_t p_m = smem_desc(sbase + C::P_OFF, C::SUB_BYTES, 1024);
            const uint64_t ds_m = smem_desc(sbase + C::DS_OFF, C::SUB_BYTES, 1024);
            const uint64_t do_m = smem_desc(sbase + C::DO_OFF, C::SUB_BYTES, 1024);
            const uint64_t q_m = smem_desc(sbase + C::Q_OFF, C::SUB_BYTES, 1024);
            const uint64_t ds_k = smem_desc(sbase + C::DS_OFF, 16, 1024);
            const uint64_t k_m = smem_desc(sbase + C::K_OFF, C::SUB_BYTES, 1024);
            bool ok = mbar_wait_spin(bar(C::B_KV), 0, wc, FA_SITE_MMA_KV);
            for (int t = 0; ok && t < ntile; ++t) {
                if (!mbar_wait_spin(bar(C::B_QFULL), t & 1, wc, FA_SITE_MMA_Q) ||
                    (t > 0 && !mbar_wait_spin(bar(C::B_SFREE), (t - 1) & 1, wc, FA_SITE_MMA_P))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // S = Q K^T, dP = dO V^T  (M = query rows, N = keys, K = d)
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_ss(tmem + C::TM_S, q_k + koff(kk), k_k + koff(kk), id_kk, kk > 0 ? 1u : 0u);
                mma_commit(bar(C::B_S));
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_ss(tmem + C::TM_DP, do_k + koff(kk), v_k + koff(kk), id_kk, kk > 0 ? 1u : 0u);
                mma_commit(bar(C::B_DP));
                if (!mbar_wait_spin(bar(C::B_P), t & 1, wc, FA_SITE_MMA_P)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // dV += P^T dO, dK += dS^T Q  (M = keys, N = d, K = query rows)
#pragma unroll
                for (int kk = 0; kk < C::BM / 16; ++kk)
                    mma_ss(tmem + C::TM_DV, p_m + moff(kk), do_m + moff(kk), id_mn,
                           (t > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
                for (int kk = 0; kk < C::BM / 16; ++kk)
                    mma_ss(tmem + C::TM_DK, ds_m + moff(kk), q_m + moff(kk), id_mn,
                           (t > 0 || kk > 0) ? 1u : 0u);
                mma_commit(bar(C::B_QFREE));  // Q_i and dO_i are no longer read
                // dQ = dS K  (M = query rows, N = d, K = keys)
#pragma unroll
                for (int kk = 0; kk < C::BN / 16; ++kk)
                    mma_ss(tmem + C::TM_DQ, ds_k + koff(kk), k_m + moff(kk), id_km, kk > 0 ? 1u : 0u);
                mma_commit(bar(C::B_DQ));
            }
            // every MMA complete: dK, dV are final (and TMEM may be released)
            mma_commit(bar(C::B_FINAL));
            mbar_drain_wait(bar(C::B_FINAL), 0, wc, FA_SITE_DRAIN);
        }
    } else {
        // -------------------------------------------------------------- compute
        const int r = threadIdx.x;  // 0..127: TMEM lane
        const uint32_t lane_base = tmem + (uint32_t(warp * 32) << 16);
        const float sl2 = a.scale_log2;
        bool ok = true;
        for (int t = 0; ok && t < ntile; ++t) {
            int h, i;
            tile_of(t, h, i);
            const int q = i * C::BM + r;
            const bool valid = q < a.N;
            const size_t ridx = (size_t(b) * a.Hq + h) * a.N + q;
            const float lse2 = valid ? __ldg(a.lse + ridx) * kLog2e : 0.f;
            const float dr = valid ? __ldg(a.dsum + ridx) : 0.f;
            bool got = mbar_wait(bar(C::B_S), t & 1, wc, FA_SITE_SOFTMAX_S) &&
                       mbar_wait(bar(C::B_DP), t & 1, wc, FA_SITE_SOFTMAX_S);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // P = exp(scale S - LSE), dS = P (dP - D), 32 keys at a time -> 16-bit
            // [half][row][64] tiles with the 128-byte swizzle (chunk c of row r at c ^ (r & 7))
#pragma unroll 1
            for (int c = 0; c < C::BN / 32; ++c) {
                uint32_t sv[32], pv[32];
                tmem_ld32(lane_base + C::TM_S + c * 32, sv);
                tmem_ld32(lane_base + C::TM_DP + c * 32, pv);
                tmem_wait_ld();
                uint32_t pw[16], dw[16];
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    const int k = key0 + c * 32 + e;
                    const bool v0 = valid && k < a.M && (!a.causal || k <= q);
                    const bool v1 = valid && k + 1 < a.M && (!a.causal || k + 1 <= q);
                    const float p0 = v0 ? fast_exp2(fmaf(__uint_as_float(sv[e]), sl2, -lse2)) : 0.f;
                    const float p1 = v1 ? fast_exp2(fmaf(__uint_as_float(sv[e + 1]), sl2, -lse2)) : 0.f;
                    const float d0 = p0 * (__uint_as_float(pv[e]) - dr);
                    const float d1 = p1 * (__uint_as_float(pv[e + 1]) - dr);
                    pw[e / 2] = pack2<T>(p0, p1);
                    dw[e / 2] = pack2<T>(d0, d1);
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int cc = (c & 1) * 4 + u;
                    const int off = (c >> 1) * C::SUB_BYTES + r * 128 + ((cc ^ (r & 7)) << 4);
                    *reinterpret_cast<uint4*>(smem + C::P_OFF + off) =
                        make_uint4(pw[4 * u], pw[4 * u + 1], pw[4 * u + 2], pw[4 * u + 3]);
                    *reinterpret_cast<uint4*>(smem + C::DS_OFF + off) =
                        make_uint4(dw[4 * u], dw[4 * u + 1], dw[4 * u + 2], dw[4 * u + 3]);
                }
            }
            fence_async_shared();  // the tensor core reads P and dS through the async proxy
            tc_fence_before();
            mbar_arrive(bar(C::B_P));
            got = mbar_wait(bar(C::B_DQ), t & 1, wc, FA_SITE_SOFTMAX_O);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            tc_fence_after();
            float* dst = a.dq_acc + ((size_t(b) * a.N + q) * a.Hq + h) * D;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t v[32];
                tmem_ld32(lane_base + C::TM_DQ + c * 32, v);
                tmem_wait_ld();
                if (valid) {
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        red_add_v4(dst + c * 32 + 4 * u, __uint_as_float(v[4 * u]),
                                   __uint_as_float(v[4 * u + 1]), __uint_as_float(v[4 * u + 2]),
                                   __uint_as_float(v[4 * u + 3]));
                }
            }
            tc_fence_before();
            mbar_arrive(bar(C::B_SFREE));
        }
        // ---- dK (times scale) and dV of this CTA's keys
        if (ok && ntile > 0) {
            const bool got = mbar_wait(bar(C::B_FINAL), 0, wc, FA_SITE_DRAIN);
            ok = __all_sync(0xffffffffu, got);
            tc_fence_after();
        }
        // tcgen05.ld is warp-collective (.sync.aligned): every lane of the warp
        // loads, whether or not its key row exists; only the stores depend on it
        // (`ok` and `ntile` are the same for the whole warp).
        const int key = key0 + r;
        const bool store = key < a.M;
        if (ok) {
            T* dvrow = reinterpret_cast<T*>(a.dv) + ((size_t(b) * a.M + key) * a.Hkv + kvh) * D;
            T* dkrow = reinterpret_cast<T*>(a.dk) + ((size_t(b) * a.M + key) * a.Hkv + kvh) * D;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t vv[32], kv[32];
                if (ntile > 0) {
                    tmem_ld32(lane_base + C::TM_DV + c * 32, vv);
                    tmem_ld32(lane_base + C::TM_DK + c * 32, kv);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) vv[e] = kv[e] = 0u;
                }
                if (!store) continue;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    uint4 wv, wk;
                    wv.x = pack2<T>(__uint_as_float(vv[8 * u]), __uint_as_float(vv[8 * u + 1]));
                    wv.y = pack2<T>(__uint_as_float(vv[8 * u + 2]), __uint_as_float(vv[8 * u + 3]));
                    wv.z = pack2<T>(__uint_as_float(vv[8 * u + 4]), __uint_as_float(vv[8 * u + 5]));
                    wv.w = pack2<T>(__uint_as_float(vv[8 * u + 6]), __uint_as_float(vv[8 * u + 7]));
                    const float s = a.scale;
                    wk.x = pack2<T>(__uint_as_float(kv[8 * u]) * s, __uint_as_float(kv[8 * u + 1]) * s);
                    wk.y = pack2<T>(__uint_as_float(kv[8 * u + 2]) * s, __uint_as_float(kv[8 * u + 3]) * s);
                    wk.z = pack2<T>(__uint_as_float(kv[8 * u + 4]) * s, __uint_as_float(kv[8 * u + 5]) * s);
                    wk.w = pack2<T>(__uint_as_float(kv[8 * u + 6]) * s, __uint_as_float(kv[8 * u + 7]) * s);
                    *reinterpret_cast<uint4*>(dvrow + c * 32 + 8 * u) = wv;
                    *reinterpret_cast<uint4*>(dkrow + c * 32 + 8 * u) = wk;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

template <int D, typename T>
cudaError_t launch_all(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdo, const BackwardArgs& a, cudaStream_t stream) {
    using C = BwdCfg<D>;
    const long long rows = (long long)a.B * a.N * a.Hq;
    const long long nb0 = (rows + 7) / 8;
    if (nb0 > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    dsum_kernel<D, T><<<dim3((unsigned)nb0), dim3(256), 0, stream>>>(a);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    auto kern = backward_kernel<D, T>;
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (err != cudaSuccess) return err;
    const long long nblocks = (long long)a.n_ktiles * a.B * a.Hkv;
    if (nblocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    kern<<<dim3((unsigned)nblocks), dim3(kBwdThreads), C::SMEM_BYTES, stream>>>(tq, tk, tv, tdo, a);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    const long long n4 = rows * D / 4;
    dq_convert_kernel<T><<<dim3((unsigned)((n4 + 255) / 256)), dim3(256), 0, stream>>>(a, n4);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_backward(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const BackwardArgs& a, int d, int dtype,
                            cudaStream_t stream) {
    if (d == 128)
        return dtype == 0 ? launch_all<128, __half>(tq, tk, tv, tdo, a, stream)
                          : launch_all<128, __nv_bfloat16>(tq, tk, tv, tdo, a, stream);
    if (d == 64)
        return dtype == 0 ? launch_all<64, __half>(tq, tk, tv, tdo, a, stream)
                          : launch_all<64, __nv_bfloat16>(tq, tk, tv, tdo, a, stream);
    return cudaErrorInvalidValue;
}

}  // namespace fa
