// fa_prefill.cu -- fused exact-attention forward (prefill) for sm_103a.
//
// What is computed follows "[CUDA 优化实战] fmha sm120 : 超越 torch.sdpa
// (flash-attention-2)", sections 1 and 2: Q is cut into tiles of query rows,
// K/V tiles are streamed along the key axis, a running row max m and sum l
// are kept, O is rescaled when the max moves and normalised once at the end,
// only tiles on the causal diagonal are masked and tiles above it are never
// loaded, and query head h reads kv head h / (Hq / Hkv).  The exponentials are
// taken in base 2 with the softmax scale folded into one FMA, and the
// rescale of O is lazy: the exponent reference only moves when the row max
// has grown by more than 8 (a factor 2^8), as in the page's "lazy rescale"
// discussion, so that most tiles touch O not at all.
//
// How it runs on GB300 (not the page's design, which used ldmatrix + mma.sync):
//   * one CTA per 128-row Q tile, 6 warps with fixed roles:
//       warps 0-3  softmax: thread t owns query row t of the tile (TMEM lane t);
//                  it reads its S row from TMEM, masks, updates m/l, writes
//                  P (fp16/bf16) back into TMEM, rescales its O row when
//                  needed, and runs the epilogue (O / l -> smem -> TMA store,
//                  LSE -> global);
//       warp 4     TMA producer: Q once, then K/V tiles into a ring of
//                  shared-memory slots in the order the MMA consumes them;
//       warp 5     TMEM allocator and single-thread tcgen05 MMA issuer.
//   * S = Q K^T and O += P V run on the 5th-gen tensor core (tcgen05.mma,
//     M = 128) with fp32 accumulators in TMEM; S is double-buffered so the
//     MMA of tile j+1 overlaps the softmax of tile j, and P is read by the PV
//     MMA straight from TMEM (A operand in tensor memory), never from smem.
//   * K/V/Q tiles are 128-byte-swizzled 64-column halves written by TMA and
//     read by the MMA through shared-memory descriptors.
//   * TMEM map (512 columns): S0 [0,128), S1 [128,256), O [256,256+d),
//     P0 and P1 (64 columns each, two 16-bit values per column) after O.
//   * every wait is bounded; on expiry the CTA records the timeout, drains
//     its own copies and MMAs, frees TMEM and returns.

#include <cfloat>
#include <cmath>

#include "fa_device.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

template <int D>
struct PrefillCfg {
    static constexpr int BM = 128;
    static constexpr int BN = 128;
    static constexpr int NSUB = D / 64;                    // 64-element (128 B) column halves
    static constexpr int SUB_BYTES = 128 * 128;            // 128 rows x 128 B
    static constexpr int TILE_BYTES = NSUB * SUB_BYTES;    // one Q, K or V tile
    static constexpr int NSLOT = D == 128 ? 5 : 8;         // K/V ring depth
    static constexpr int Q_OFF = 0;
    static constexpr int SLOT_OFF = TILE_BYTES;
    static constexpr int BAR_OFF = SLOT_OFF + NSLOT * TILE_BYTES;
    // barrier indices
    static constexpr int B_QFULL = 0;
    static constexpr int B_FULL = 1;                       // NSLOT of them
    static constexpr int B_EMPTY = 1 + NSLOT;              // NSLOT of them
    static constexpr int B_SFULL = 1 + 2 * NSLOT;          // 2
    static constexpr int B_PFULL = 3 + 2 * NSLOT;          // 2
    static constexpr int B_ODONE = 5 + 2 * NSLOT;
    static constexpr int B_DRAIN = 6 + 2 * NSLOT;
    static constexpr int NBAR = 7 + 2 * NSLOT;
    static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
    static constexpr int SMEM_BYTES = MISC_OFF + 16 + 1024;  // + slack to align the base to 1 KB
    // TMEM columns
    static constexpr uint32_t TM_S0 = 0;
    static constexpr uint32_t TM_S1 = 128;
    static constexpr uint32_t TM_O = 256;
    static constexpr uint32_t TM_P0 = 256 + D;
    static constexpr uint32_t TM_P1 = 256 + D + 64;
    static constexpr uint32_t TMEM_COLS = 512;
    static_assert(TM_P1 + 64 <= TMEM_COLS, "TMEM budget");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

constexpr int kThreads = 192;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only when the max grows by > 2^8

template <int D, typename T>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                   const PrefillArgs a) {
    using C = PrefillCfg<D>;
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

    // Which tile: the latest (most expensive, when causal) query tiles go first.
    const int nbh = a.B * a.Hq;
    const int lin = blockIdx.x;
    const int qt = a.n_qtiles - 1 - lin / nbh;
    const int bh = lin % nbh;
    const int h = bh % a.Hq;
    const int b = bh / a.Hq;
    const int kvh = h / (a.Hq / a.Hkv);
    const int q0 = qt * C::BM;
    const int kv_end = a.causal ? min(a.M, q0 + C::BM) : a.M;
    const int nt = (kv_end + C::BN - 1) / C::BN;

    if (threadIdx.x == 0) {
        mbar_init(bar(C::B_QFULL), 1);
        for (int i = 0; i < C::NSLOT; ++i) {
            mbar_init(bar(C::B_FULL + i), 1);
            mbar_init(bar(C::B_EMPTY + i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(C::B_SFULL + i), 1);
            mbar_init(bar(C::B_PFULL + i), 128);
        }
        mbar_init(bar(C::B_ODONE), 1);
        mbar_init(bar(C::B_DRAIN), 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 4 && lane == 0) {
        prefetch_tensor_map(&tm_q);
        prefetch_tensor_map(&tm_k);
        prefetch_tensor_map(&tm_v);
        prefetch_tensor_map(&tm_o);
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
        if (lane == 0) {
            mbar_arrive_expect_tx(bar(C::B_QFULL), C::TILE_BYTES);
            for (int s = 0; s < C::NSUB; ++s)
                tma_load_4d(sbase + C::Q_OFF + s * C::SUB_BYTES, &tm_q, s * 64, h, q0, b,
                            bar(C::B_QFULL));
            int L = 0;  // loads issued, in consumption order K0, K1, V0, K2, V1, ...
            auto issue = [&](bool is_v, int j) -> bool {
                const int slot = L % C::NSLOT;
                const uint32_t parity = ((L / C::NSLOT) & 1) ^ 1;
                if (!mbar_wait(bar(C::B_EMPTY + slot), parity, wc, FA_SITE_PRODUCER_SLOT))
                    return false;
                mbar_arrive_expect_tx(bar(C::B_FULL + slot), C::TILE_BYTES);
                const uint32_t dst = sbase + C::SLOT_OFF + slot * C::TILE_BYTES;
                for (int s = 0; s < C::NSUB; ++s)
                    tma_load_4d(dst + s * C::SUB_BYTES, is_v ? &tm_v : &tm_k, s * 64, kvh, j * C::BN,
                                b, bar(C::B_FULL + slot));
                ++L;
                return true;
            };
            bool ok = issue(false, 0);
            if (ok && nt > 1) ok = issue(false, 1);
            for (int j = 0; ok && j < nt; ++j) {
                ok = issue(true, j);
                if (ok && j + 2 < nt) ok = issue(false, j + 2);
            }
            // Every issued copy must have landed before the CTA may exit.
            mbar_drain_wait(bar(C::B_QFULL), 0, wc, FA_SITE_DRAIN);
            for (int slot = 0; slot < C::NSLOT && slot < L; ++slot) {
                const int last = slot + ((L - 1 - slot) / C::NSLOT) * C::NSLOT;
                mbar_drain_wait(bar(C::B_FULL + slot), (last / C::NSLOT) & 1, wc, FA_SITE_DRAIN);
            }
        }
    } else if (warp == 5) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t fmt = DTypeFmt<T>::value;
            constexpr uint32_t idesc_qk = instr_desc_f16(fmt, 128, 128, 0, 0);  // Q, K both K-major
            constexpr uint32_t idesc_pv = instr_desc_f16(fmt, 128, D, 0, 1);    // V is MN-major
            const uint32_t qb = sbase + C::Q_OFF;
            int L = 0;
            auto qk = [&](int j) -> bool {
                const int slot = L % C::NSLOT;
                if (!mbar_wait(bar(C::B_FULL + slot), (L / C::NSLOT) & 1, wc, FA_SITE_MMA_KV))
                    return false;
                tc_fence_after();
                const uint32_t kb = sbase + C::SLOT_OFF + slot * C::TILE_BYTES;
                const uint32_t d_tmem = tmem + ((j & 1) ? C::TM_S1 : C::TM_S0);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    // K-major, 128-byte swizzle: k-steps of 16 elements advance 32 bytes
                    // inside a 64-column half; 8-row groups are 1024 bytes apart.
                    const uint32_t off = (kk / 4) * C::SUB_BYTES + (kk % 4) * 32;
                    mma_ss(d_tmem, smem_desc(qb + off, 16, 1024), smem_desc(kb + off, 16, 1024),
                           idesc_qk, kk > 0 ? 1u : 0u);
                }
                mma_commit(bar(C::B_EMPTY + slot));
                mma_commit(bar(C::B_SFULL + (j & 1)));
                ++L;
                return true;
            };
            bool ok = mbar_wait(bar(C::B_QFULL), 0, wc, FA_SITE_MMA_Q);
            if (ok) tc_fence_after();
            if (ok) ok = qk(0);
            if (ok && nt > 1) ok = qk(1);
            for (int j = 0; ok && j < nt; ++j) {
                if (!mbar_wait(bar(C::B_PFULL + (j & 1)), (j >> 1) & 1, wc, FA_SITE_MMA_P)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int slot = L % C::NSLOT;
                if (!mbar_wait(bar(C::B_FULL + slot), (L / C::NSLOT) & 1, wc, FA_SITE_MMA_KV)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t vb = sbase + C::SLOT_OFF + slot * C::TILE_BYTES;
                const uint32_t p_tmem = tmem + ((j & 1) ? C::TM_P1 : C::TM_P0);
#pragma unroll
                for (int kk = 0; kk < C::BN / 16; ++kk) {
                    // V is [key][d] = MN-major for B (N = d): 16 keys = 16 rows of 128 B;
                    // the two 64-column halves are SUB_BYTES apart (leading offset),
                    // 8-key groups 1024 bytes apart (stride offset).  P: 16 keys of
                    // 16-bit values = 8 TMEM columns.
                    mma_ts(tmem + C::TM_O, p_tmem + kk * 8,
                           smem_desc(vb + kk * 16 * 128, C::SUB_BYTES, 1024), idesc_pv,
                           (j > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(bar(C::B_EMPTY + slot));
                mma_commit(bar(C::B_ODONE));
                ++L;
                if (j + 2 < nt) ok = qk(j + 2);
            }
            // All MMAs must be complete before TMEM is released.
            mma_commit(bar(C::B_DRAIN));
            mbar_drain_wait(bar(C::B_DRAIN), 0, wc, FA_SITE_DRAIN);
        }
    } else {
        // ------------------------------------------------------------- softmax
        const int r = threadIdx.x;  // row in tile == TMEM lane
        const int row = q0 + r;
        const uint32_t lane_base = tmem + (uint32_t(warp * 32) << 16);
        const float sl2 = a.scale_log2;
        float m_ref = -INFINITY;  // exponent reference, log2 units of the scaled logits
        float l = 0.f;
        bool ok = true;
        for (int j = 0; j < nt; ++j) {
            bool got = mbar_wait(bar(C::B_SFULL + (j & 1)), (j >> 1) & 1, wc, FA_SITE_SOFTMAX_S);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            tc_fence_after();
            float s[C::BN];
            {
                const uint32_t s_addr = lane_base + ((j & 1) ? C::TM_S1 : C::TM_S0);
#pragma unroll
                for (int c = 0; c < C::BN / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld32(s_addr + c * 32, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) s[c * 32 + e] = __uint_as_float(v[e]);
                }
            }
            const int k0 = j * C::BN;
            if (k0 + C::BN > a.M || (a.causal && k0 + C::BN - 1 > q0)) {
                int lim = a.M - k0;
                if (a.causal) lim = min(lim, row - k0 + 1);
#pragma unroll
                for (int c = 0; c < C::BN; ++c)
                    if (c >= lim) s[c] = -INFINITY;
            }
            float mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < C::BN; ++c) mx = fmaxf(mx, s[c]);
            const float mt = mx * sl2;
            float alpha = 1.f;
            bool rescale = false;
            if (j == 0) {
                m_ref = mt;
            } else if (mt > m_ref + kRescaleThreshold) {
                alpha = fast_exp2(m_ref - mt);
                l *= alpha;
                m_ref = mt;
                rescale = true;
            }
            if (__any_sync(0xffffffffu, rescale)) {
                // O must hold every PV product so far before it is scaled.
                got = mbar_wait(bar(C::B_ODONE), (j - 1) & 1, wc, FA_SITE_SOFTMAX_O);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t o_addr = lane_base + C::TM_O;
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld32(o_addr + c * 32, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
                    tmem_st32(o_addr + c * 32, v);
                }
                tmem_wait_st();
            }
            const float neg = (m_ref == -INFINITY) ? 0.f : -m_ref;
            const uint32_t p_addr = lane_base + ((j & 1) ? C::TM_P1 : C::TM_P0);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t pk[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const float p0 = fast_exp2(fmaf(s[half * 64 + 2 * e], sl2, neg));
                    const float p1 = fast_exp2(fmaf(s[half * 64 + 2 * e + 1], sl2, neg));
                    l += p0 + p1;
                    pk[e] = pack2<T>(p0, p1);
                }
                tmem_st32(p_addr + half * 32, pk);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar(C::B_PFULL + (j & 1)));
        }
        // ------------------------------------------------------------ epilogue
        if (ok) {
            // The drain barrier completes once, after every MMA of the tile (the
            // per-PV barrier could alias phases here: the last two PVs may both
            // still be in flight).
            const bool got = mbar_wait(bar(C::B_DRAIN), 0, wc, FA_SITE_SOFTMAX_O);
            ok = __all_sync(0xffffffffu, got);
        }
        if (ok) {
            tc_fence_after();
            const float inv_l = 1.f / l;
            const uint32_t o_addr = lane_base + C::TM_O;
            uint8_t* stage = smem + C::Q_OFF;  // Q is dead once the last MMA has completed
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t v[32];
                tmem_ld32(o_addr + c * 32, v);
                tmem_wait_ld();
                uint32_t w[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    w[e] = pack2<T>(__uint_as_float(v[2 * e]) * inv_l,
                                    __uint_as_float(v[2 * e + 1]) * inv_l);
                const int col0 = c * 32;
                const int sub = col0 / 64;
                const int chunk0 = (col0 % 64) / 8;
#pragma unroll
                for (int qd = 0; qd < 4; ++qd) {
                    const int chunk = chunk0 + qd;
                    uint4* dst = reinterpret_cast<uint4*>(stage + sub * C::SUB_BYTES + r * 128 +
                                                          ((chunk ^ (r & 7)) << 4));
                    *dst = make_uint4(w[4 * qd], w[4 * qd + 1], w[4 * qd + 2], w[4 * qd + 3]);
                }
            }
            if (a.lse != nullptr && row < a.N)
                a.lse[(size_t(b) * a.Hq + h) * a.N + row] = (m_ref + log2f(l)) * kLn2;
        }
        fence_async_shared();
        named_barrier_sync(1, 128);
        if (threadIdx.x == 0 && *abort_flag == 0) {
            for (int s = 0; s < C::NSUB; ++s)
                tma_store_4d(&tm_o, sbase + C::Q_OFF + s * C::SUB_BYTES, s * 64, h, q0, b);
            tma_store_commit();
            tma_store_wait_all();
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

template <int D, typename T>
cudaError_t launch_prefill_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                             const CUtensorMap& to, const PrefillArgs& a, cudaStream_t stream) {
    using C = PrefillCfg<D>;
    auto kern = prefill_kernel<D, T>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           C::SMEM_BYTES);
    if (err != cudaSuccess) return err;
    const long long nblocks = (long long)a.n_qtiles * a.B * a.Hq;
    if (nblocks <= 0 || nblocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    kern<<<dim3((unsigned)nblocks), dim3(kThreads), C::SMEM_BYTES, stream>>>(tq, tk, tv, to, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const CUtensorMap& to, const PrefillArgs& a, int d, int dtype,
                           cudaStream_t stream) {
    if (d == 128)
        return dtype == 0 ? launch_prefill_t<128, __half>(tq, tk, tv, to, a, stream)
                          : launch_prefill_t<128, __nv_bfloat16>(tq, tk, tv, to, a, stream);
    if (d == 64)
        return dtype == 0 ? launch_prefill_t<64, __half>(tq, tk, tv, to, a, stream)
                          : launch_prefill_t<64, __nv_bfloat16>(tq, tk, tv, to, a, stream);
    return cudaErrorInvalidValue;
}

}  // namespace fa
