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
//   1. dsum_kernel: per (b, h, 128-row Q tile) a 1 KB record of LSE * log2(e)
//      (+inf for rows past N, so that their P is 0) and D_i = dO_i . O_i in
//      fp32; it also zeroes the fp32 dQ accumulator.
//   2. backward_kernel: one CTA per (b, kv head, 128-key tile j) keeps K_j
//      and V_j in shared memory and walks the 128-row Q tiles that see them
//      (from tile j on when causal), for every query head of the GQA group.
//      Everything is computed transposed, keys on the 128 TMEM lanes:
//        S^T = K Q^T and dP^T = V dO^T (fp32 in TMEM);
//        two compute warpgroups (one half of the 128 query columns each, key
//        row r on TMEM lane r) form P^T and dS^T = P^T o (dP^T - D) and write
//        them back into TMEM as 16-bit, over columns they have already read,
//        and dS into shared memory;
//        dV += P^T dO and dK += dS^T Q take P^T and dS^T straight from TMEM
//        (A operand in tensor memory); dQ = dS K reads dS from shared memory
//        (MN-major, i.e. transposed by the descriptor) and lands in the S^T
//        columns (P^T is dead by then), query rows on the lanes; the compute
//        warps stage it for the bulk reductions into the fp32 accumulator.
//      Q_i, dO_i and the tile's LSE/D record are double-buffered, so the next
//      tile streams in while the current one is computed.  The tensor core
//      runs dV(t), then dQ(t) and dK(t) back to back, then S^T(t+1) (which
//      waits for dQ(t) to be read out of TMEM) and dP^T(t+1).
//      TMEM (512 columns): S^T [0,128) (P^T over [0,32) and [64,96); later dQ
//      over [0,d)), dP^T [128,256) (dS^T over [128,160) and [192,224)), dV
//      [256,256+d), dK [256+d,256+2d).  dQ, dP^T(t+1) and S^T(t+1) overwrite
//      operands that earlier MMAs read: tcgen05 MMAs issued by one thread
//      execute in issue order.
//        warps 0-7 compute; warp 8 TMA producer; warp 9 TMEM allocator and
//        single-thread MMA issuer; warp 10 issues the dQ bulk reductions.
//      dQ is read out of TMEM, staged in this tile's Q and dO slots (dead once
//      dK and dV have read them) as 128-byte-swizzled fp32 boxes, and added to
//      the fp32 accumulator by TMA bulk reductions, which reduce whole lines in
//      L2; the slots are refilled once the reductions have read them.
//   3. dq_convert_kernel: dQ = scale * accumulator, rounded to the input type.
// Launches 2 and 3 are programmatic dependents of the launch before them: they
// may start (set-up, K/V loads) while it finishes, and the threads that read
// its results wait for it first (griddepcontrol.wait).
// Every wait is bounded; on expiry the CTA records the timeout, drains its own
// copies and MMAs, frees TMEM and returns.

#include <cfloat>
#include <cmath>

#include "fa_device.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start before the kernel ahead of it on the stream has
// finished.  grid_dep_wait() blocks the calling thread until that kernel has
// completed and its memory is visible (a no-op for a normal launch);
// grid_dep_launch_dependents() lets the next such kernel start once every CTA
// of this grid has called it or exited.
__device__ __forceinline__ void grid_dep_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void grid_dep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}


template <int D>
struct BwdCfg {
    static constexpr int BM = 128;                        // query rows per Q tile
    static constexpr int BN = 128;                        // keys per CTA
    static constexpr int NSUB = D / 64;                   // 64-element (128 B) column halves
    static constexpr int SUB_BYTES = 128 * 128;           // 128 rows x 128 B
    static constexpr int TILE_BYTES = NSUB * SUB_BYTES;   // a [128][D] tile
    static constexpr int DS_BYTES = 2 * SUB_BYTES;        // dS [128 keys][128 queries]
    static constexpr int LD_BYTES = 2 * BM * 4;           // LSE*log2e [128], D [128]
    static constexpr int K_OFF = 0;
    static constexpr int V_OFF = K_OFF + TILE_BYTES;
    static constexpr int Q_OFF = V_OFF + TILE_BYTES;      // two buffers
    static constexpr int DO_OFF = Q_OFF + 2 * TILE_BYTES; // two buffers
    static constexpr int DS_OFF = DO_OFF + 2 * TILE_BYTES;
    static constexpr int LD_OFF = DS_OFF + DS_BYTES;      // two buffers
    static constexpr int BAR_OFF = LD_OFF + 2 * LD_BYTES;
    // barriers
    static constexpr int B_KV = 0;       // K_j, V_j landed
    static constexpr int B_QFULL = 1;    // [2] Q_i and the LSE/D record of a buffer landed
    static constexpr int B_QFREE = 3;    // [2] the MMAs reading a buffer are done
    static constexpr int B_S = 5;        // S^T in TMEM
    static constexpr int B_DP = 6;       // dP^T in TMEM
    static constexpr int B_DS = 7;       // dS^T in TMEM and dS in smem (256 arrivals)
    static constexpr int B_DQ = 8;       // dQ in TMEM (and every earlier MMA done)
    static constexpr int B_DQFREE = 9;   // dQ read out of TMEM (256 arrivals)
    static constexpr int B_FINAL = 10;   // every MMA done: dK, dV final
    static constexpr int B_STAGEFULL = 11;  // dQ staged in the tile's Q/dO slots (256 arrivals)
    static constexpr int B_STAGED = 12;     // the dQ boxes staged in the dS buffer are read out
    static constexpr int B_PT = 14;         // P^T in TMEM (256 arrivals)
    static constexpr int B_DOFULL = 15;     // [2] dO_i of a buffer landed
    static constexpr int B_STAGED_DO = 17;  // [2] the dQ boxes staged in a buffer's dO slot are read out
    static constexpr int NBAR = 19;
    static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
    // The dynamic shared-memory base is 1 KB aligned (checked at run time), so
    // no alignment slack is allocated: the layout needs all but ~1 KB of the
    // 227 KB a CTA may have.
    static constexpr int SMEM_BYTES = MISC_OFF + 16;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t TM_S = 0, TM_DP = 128, TM_DQ = 0, TM_DV = 256, TM_DK = 256 + D;
    static_assert(256 + 2 * D <= 512, "TMEM budget");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

constexpr int kBwdThreads = 352;
constexpr int kComputeThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;

// One warp per padded query row (b, h, q < n_qtiles * 128): the tile record
// pack[((b * Hq + h) * n_qtiles + q / 128) * 256 + {q % 128, 128 + q % 128}] =
// {LSE * log2(e), D = dO . O}; rows past N get {+inf, 0}.  The same warp
// zeroes the row's fp32 dQ accumulator.
template <int D, typename T>
__global__ void __launch_bounds__(256) dsum_kernel(const BackwardArgs a) {
    // the backward kernel may start its set-up and K/V loads now; it waits for
    // this grid to finish before it reads the records or adds into dQ
    grid_dep_launch_dependents();
    constexpr int EPL = D / 32;  // elements per lane (2 or 4)
    const int nq_pad = a.n_qtiles * 128;
    const long long rows = (long long)a.B * a.Hq * nq_pad;
    const long long pr = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (pr >= rows) return;
    const long long bh = pr / nq_pad;
    const int q = int(pr % nq_pad);
    const long long b = bh / a.Hq, h = bh % a.Hq;
    float dsum = 0.f, lse2 = INFINITY;
    if (q < a.N) {
        const long long row = (b * a.N + q) * a.Hq + h;  // row of [B, N, Hq, d]
        const T* o = reinterpret_cast<const T*>(a.o) + row * D + lane * EPL;
        const T* g = reinterpret_cast<const T*>(a.dout) + row * D + lane * EPL;
        if constexpr (EPL == 4) {
            const uint2 ov = *reinterpret_cast<const uint2*>(o);
            const uint2 gv = *reinterpret_cast<const uint2*>(g);
            const float2 o0 = unpack2<T>(ov.x), o1 = unpack2<T>(ov.y);
            const float2 g0 = unpack2<T>(gv.x), g1 = unpack2<T>(gv.y);
            dsum = fmaf(o0.x, g0.x, fmaf(o0.y, g0.y, fmaf(o1.x, g1.x, o1.y * g1.y)));
        } else {
            const float2 o0 = unpack2<T>(*reinterpret_cast<const uint32_t*>(o));
            const float2 g0 = unpack2<T>(*reinterpret_cast<const uint32_t*>(g));
            dsum = fmaf(o0.x, g0.x, o0.y * g0.y);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) dsum += __shfl_xor_sync(0xffffffffu, dsum, off);
        lse2 = a.lse[bh * a.N + q] * kLog2e;
        float* acc_row = a.dq_acc + row * D + lane * EPL;
        if constexpr (EPL == 4)
            *reinterpret_cast<float4*>(acc_row) = make_float4(0.f, 0.f, 0.f, 0.f);
        else
            *reinterpret_cast<float2*>(acc_row) = make_float2(0.f, 0.f);
    }
    if (lane == 0) {
        float* rec = a.pack + (bh * a.n_qtiles + q / 128) * 256;
        rec[q % 128] = lse2;
        rec[128 + q % 128] = dsum;
    }
}

// dQ = scale * accumulator, rounded to T; four elements per thread.
template <typename T>
__global__ void __launch_bounds__(256) dq_convert_kernel(const BackwardArgs a, long long n4) {
    grid_dep_wait();  // every dQ reduction of the backward kernel has landed
    const long long i = (long long)blockIdx.x * 256 + threadIdx.x;
    if (i >= n4) return;
    const float4 v = reinterpret_cast<const float4*>(a.dq_acc)[i];
    const float s = a.scale;
    reinterpret_cast<uint2*>(a.dq)[i] = make_uint2(pack2<T>(v.x * s, v.y * s), pack2<T>(v.z * s, v.w * s));
}

// TMA bulk reduction: the box at `src` (shared) is added element-wise (fp32)
// into the tensor at the given coordinates; rows past the tensor's end are
// dropped.  Tracked by the issuing thread's bulk async-group.
__device__ __forceinline__ void tma_reduce_add_4d(const CUtensorMap* map, uint32_t src, int c0,
                                                  int c1, int c2, int c3) {
    asm volatile(
        "cp.reduce.async.bulk.tensor.4d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4, %5}], "
        "[%1];" ::"l"(reinterpret_cast<uint64_t>(map)),
        "r"(src), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

// Plain (non-tensor) bulk copy global -> shared, completing on `bar`.  Both
// addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

template <int D, typename T>
__global__ void __launch_bounds__(kBwdThreads, 1)
    backward_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_dq, const BackwardArgs a) {
    using C = BwdCfg<D>;
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sbase = smem_addr(smem);
    if (sbase & 1023u) {
        // the layout leaves no room to realign: report and do nothing
        if (threadIdx.x == 0) atomicCAS(a.status, 0, FA_DEV_LAYOUT | (FA_SITE_SMEM_ALIGN << 8));
        return;
    }
    const uint32_t bars = sbase + C::BAR_OFF;
    volatile uint32_t* tmem_holder = reinterpret_cast<volatile uint32_t*>(smem + C::MISC_OFF);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 4);
    auto bar = [&](int i) -> uint32_t { return bars + 8u * uint32_t(i); };
    // Where the fp32 dQ box k (columns [32k, 32k + 32), 128 rows) of a tile in
    // buffer buf is staged for its bulk reduction: the first NSUB boxes in the dS
    // buffer (free once the tile's dQ MMA has read dS), the rest in the tile's dO
    // slot (free once dV and dP have read dO).  The Q slot stays out of it, so
    // that the next loads of Q never wait for a reduction.
    auto stage_box = [](int k, int buf) -> uint32_t {
        return k < C::NSUB ? uint32_t(C::DS_OFF + k * C::SUB_BYTES)
                           : uint32_t(C::DO_OFF + buf * C::TILE_BYTES + (k - C::NSUB) * C::SUB_BYTES);
    };
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
        for (int x = 0; x < 2; ++x) {
            mbar_init(bar(C::B_QFULL + x), 1);
            mbar_init(bar(C::B_QFREE + x), 1);
            mbar_init(bar(C::B_DOFULL + x), 1);
            mbar_init(bar(C::B_STAGED_DO + x), 1);
        }
        mbar_init(bar(C::B_S), 1);
        mbar_init(bar(C::B_DP), 1);
        mbar_init(bar(C::B_DS), kComputeThreads);
        mbar_init(bar(C::B_PT), kComputeThreads);
        mbar_init(bar(C::B_DQ), 1);
        mbar_init(bar(C::B_DQFREE), kComputeThreads);
        mbar_init(bar(C::B_FINAL), 1);
        mbar_init(bar(C::B_STAGEFULL), kComputeThreads);
        mbar_init(bar(C::B_STAGED), 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 8 && lane == 0) {
        prefetch_tensor_map(&tm_q);
        prefetch_tensor_map(&tm_k);
        prefetch_tensor_map(&tm_v);
        prefetch_tensor_map(&tm_do);
        prefetch_tensor_map(&tm_dq);
    }
    if (warp == 9) {
        tmem_alloc(smem_addr(const_cast<uint32_t*>(tmem_holder)), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const WaitCtl wc{abort_flag, a.status, a.timeout_ns};

    if (warp == 8) {
        // ------------------------------------------------------------- producer
        if (lane == 0 && ntile > 0) {
            mbar_arrive_expect_tx(bar(C::B_KV), 2 * C::TILE_BYTES);
            for (int s = 0; s < C::NSUB; ++s) {
                tma_load_4d(sbase + C::K_OFF + s * C::SUB_BYTES, &tm_k, s * 64, kvh, key0, b, bar(C::B_KV));
                tma_load_4d(sbase + C::V_OFF + s * C::SUB_BYTES, &tm_v, s * 64, kvh, key0, b, bar(C::B_KV));
            }
            // the LSE/D records come from the preprocessing kernel
            grid_dep_wait();
            // Q_i (with its LSE/D record) and dO_i go into a buffer on barriers of
            // their own.  No dQ is staged in the Q slot, so Q_i loads as soon as the
            // MMAs of the tile two back are done; the dO slot also waits for the
            // reducer to have read the dQ boxes staged there.
            int t = 0, t_do = 0;  // tiles whose Q (resp. dO) copy was issued
            for (; t < ntile; ++t) {
                const int buf = t & 1;
                const uint32_t ph = ((t - 2) >> 1) & 1;
                // the tile two back used this buffer: its MMAs must be done with it
                if (t >= 2 && !mbar_wait(bar(C::B_QFREE + buf), ph, wc, FA_SITE_PRODUCER_SLOT))
                    break;
                int h, i;
                tile_of(t, h, i);
                const uint32_t full = bar(C::B_QFULL + buf);
                mbar_arrive_expect_tx(full, C::TILE_BYTES + C::LD_BYTES);
                for (int s = 0; s < C::NSUB; ++s)
                    tma_load_4d(sbase + C::Q_OFF + buf * C::TILE_BYTES + s * C::SUB_BYTES, &tm_q,
                                s * 64, h, i * C::BM, b, full);
                bulk_load(sbase + C::LD_OFF + buf * C::LD_BYTES,
                          a.pack + ((size_t(b) * a.Hq + h) * a.n_qtiles + i) * 256, C::LD_BYTES, full);
                // ... and the dQ staged in its dO slot
                if (t >= 2 && !mbar_wait(bar(C::B_STAGED_DO + buf), ph, wc, FA_SITE_PRODUCER_SLOT)) {
                    ++t;  // this tile's Q copy is in flight and must be drained
                    break;
                }
                const uint32_t dfull = bar(C::B_DOFULL + buf);
                mbar_arrive_expect_tx(dfull, C::TILE_BYTES);
                for (int s = 0; s < C::NSUB; ++s)
                    tma_load_4d(sbase + C::DO_OFF + buf * C::TILE_BYTES + s * C::SUB_BYTES, &tm_do,
                                s * 64, h, i * C::BM, b, dfull);
                t_do = t + 1;
            }
            // every issued copy must have landed before the CTA may exit
            mbar_drain_wait(bar(C::B_KV), 0, wc, FA_SITE_DRAIN);
            for (int u = t - 2 < 0 ? 0 : t - 2; u < t; ++u)
                mbar_drain_wait(bar(C::B_QFULL + (u & 1)), (u >> 1) & 1, wc, FA_SITE_DRAIN);
            for (int u = t_do - 2 < 0 ? 0 : t_do - 2; u < t_do; ++u)
                mbar_drain_wait(bar(C::B_DOFULL + (u & 1)), (u >> 1) & 1, wc, FA_SITE_DRAIN);
        }
    } else if (warp == 9) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0 && ntile > 0) {
            constexpr uint32_t fmt = DTypeFmt<T>::value;
            constexpr uint32_t id_kk = instr_desc_f16(fmt, 128, 128, 0, 0);  // S^T, dP^T: K-major A, B
            constexpr uint32_t id_ts = instr_desc_f16(fmt, 128, D, 0, 1);    // dV, dK: A in TMEM, B MN-major
            constexpr uint32_t id_mm = instr_desc_f16(fmt, 128, D, 1, 1);    // dQ: A = dS, B = K, both MN-major
            // K-major (128-byte swizzle): a 16-element k-step advances 32 bytes inside
            // a 64-column half, halves are SUB_BYTES apart, 8-row groups 1024 bytes.
            // MN-major: a 16-row k-step advances 16 x 128 bytes; the 64-wide halves of
            // the M or N extent are SUB_BYTES apart (leading offset), 8-row groups 1024 B.
            auto koff = [](int kk) -> uint64_t {
                return uint64_t((kk / 4) * C::SUB_BYTES + (kk % 4) * 32) >> 4;
            };
            auto moff = [](int kk) -> uint64_t { return uint64_t(kk * 16 * 128) >> 4; };
            // P^T / dS^T in TMEM: queries 16kk..16kk+15 are 8 packed columns, the
            // low 64 queries at [0,32), the high 64 at [64,96) of their region
            auto pcol = [](int kk) -> uint32_t { return uint32_t((kk < 4 ? 0 : 64) + (kk & 3) * 8); };
            constexpr uint64_t kBufStep = C::TILE_BYTES >> 4;
            const uint64_t k_k = smem_desc(sbase + C::K_OFF, 16, 1024);
            const uint64_t v_k = smem_desc(sbase + C::V_OFF, 16, 1024);
            const uint64_t q_k0 = smem_desc(sbase + C::Q_OFF, 16, 1024);
            const uint64_t do_k0 = smem_desc(sbase + C::DO_OFF, 16, 1024);
            const uint64_t q_m0 = smem_desc(sbase + C::Q_OFF, C::SUB_BYTES, 1024);
            const uint64_t do_m0 = smem_desc(sbase + C::DO_OFF, C::SUB_BYTES, 1024);
            const uint64_t ds_m = smem_desc(sbase + C::DS_OFF, C::SUB_BYTES, 1024);
            const uint64_t k_m = smem_desc(sbase + C::K_OFF, C::SUB_BYTES, 1024);
            // S^T(tt) = K Q(tt)^T  (M = keys, N = queries, K = d), once Q(tt) has landed
            auto issue_s = [&](int tt) -> bool {
                const int b2 = tt & 1;
                if (!mbar_wait_spin(bar(C::B_QFULL + b2), (tt >> 1) & 1, wc, FA_SITE_MMA_Q))
                    return false;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_ss(tmem + C::TM_S, k_k + koff(kk), q_k0 + (b2 ? kBufStep : 0) + koff(kk),
                           id_kk, kk > 0 ? 1u : 0u);
                mma_commit(bar(C::B_S));
                return true;
            };
            // dP^T(tt) = V dO(tt)^T, once dO(tt) has landed; it overwrites dS^T(tt-1),
            // which dK(tt-1), issued before it, has read by then
            auto issue_dp = [&](int tt) -> bool {
                const int b2 = tt & 1;
                if (!mbar_wait_spin(bar(C::B_DOFULL + b2), (tt >> 1) & 1, wc, FA_SITE_MMA_Q))
                    return false;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_ss(tmem + C::TM_DP, v_k + koff(kk), do_k0 + (b2 ? kBufStep : 0) + koff(kk),
                           id_kk, kk > 0 ? 1u : 0u);
                mma_commit(bar(C::B_DP));
                return true;
            };
            bool ok = mbar_wait_spin(bar(C::B_KV), 0, wc, FA_SITE_MMA_KV) && issue_s(0) &&
                      issue_dp(0);
            for (int t = 0; ok && t < ntile; ++t) {
                const int buf = t & 1;
                const uint64_t bstep = buf ? kBufStep : 0;
                // dV += P^T dO as soon as P^T is there (it overlaps the forming of dS)
                if (!mbar_wait_spin(bar(C::B_PT), t & 1, wc, FA_SITE_MMA_P)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < C::BM / 16; ++kk)
                    mma_ts(tmem + C::TM_DV, tmem + C::TM_S + pcol(kk), do_m0 + bstep + moff(kk), id_ts,
                           (t > 0 || kk > 0) ? 1u : 0u);
                if (!mbar_wait_spin(bar(C::B_DS), t & 1, wc, FA_SITE_MMA_P)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // dQ = dS K  (M = queries, N = d, K = keys) first, into the S^T columns
                // (P^T is dead once dV, issued before, has read it), signalled on its own
                // so that the compute warps read it out while dK runs
#pragma unroll
                for (int kk = 0; kk < C::BN / 16; ++kk)
                    mma_ss(tmem + C::TM_DQ, ds_m + moff(kk), k_m + moff(kk), id_mm, kk > 0 ? 1u : 0u);
                mma_commit(bar(C::B_DQ));
                // dK += dS^T Q  (M = keys, N = d, K = queries; A in TMEM)
#pragma unroll
                for (int kk = 0; kk < C::BM / 16; ++kk)
                    mma_ts(tmem + C::TM_DK, tmem + C::TM_DP + pcol(kk), q_m0 + bstep + moff(kk), id_ts,
                           (t > 0 || kk > 0) ? 1u : 0u);
                mma_commit(bar(C::B_QFREE + buf));  // Q_i, dO_i no longer read
                if (t + 1 < ntile) {
                    // S^T(t+1) once dQ(t) has left the S^T columns (the compute warps read
                    // it out while dK(t) runs), then dP^T(t+1) once dO(t+1) has landed
                    if (!mbar_wait_spin(bar(C::B_DQFREE), t & 1, wc, FA_SITE_MMA_P) ||
                        !issue_s(t + 1) || !issue_dp(t + 1)) {
                        ok = false;
                        break;
                    }
                }
            }
            // every MMA complete: dK, dV are final (and TMEM may be released)
            mma_commit(bar(C::B_FINAL));
            mbar_drain_wait(bar(C::B_FINAL), 0, wc, FA_SITE_DRAIN);
        }
    } else if (warp == 10) {
        // ------------------------------------------------------------- reducer
        if (lane == 0) {
            grid_dep_wait();  // the accumulator is zeroed by the preprocessing kernel
            for (int t = 0; t < ntile; ++t) {
                if (!mbar_wait(bar(C::B_STAGEFULL), t & 1, wc, FA_SITE_SOFTMAX_O)) break;
                const int buf = t & 1;
                int h, i;
                tile_of(t, h, i);
                // the boxes in the dS buffer first, as one bulk group, then those in
                // the dO slot; each may be overwritten (and the CTA may exit) once its
                // boxes have been read
                for (int k = 0; k < D / 32; ++k) {
                    tma_reduce_add_4d(&tm_dq, sbase + stage_box(k, buf), 32 * k, h, i * C::BM, b);
                    if (k == C::NSUB - 1) tma_store_commit();
                }
                tma_store_commit();
                tma_store_wait_read_1();
                mbar_arrive(bar(C::B_STAGED));
                tma_store_wait_all();
                mbar_arrive(bar(C::B_STAGED_DO + buf));
            }
        }
    } else {
        // ------------------------------------------------------------ compute
        // thread <-> TMEM lane r (key row for S^T, dP^T, dV, dK; query row for
        // dQ); warpgroup wg takes queries [64 wg, 64 wg + 64) of S^T / dP^T and
        // columns [wg d/2, wg d/2 + d/2) of dQ, dV and dK.
        const int wg = warp >> 2;
        const int r = (warp & 3) * 32 + lane;
        const uint32_t lane_base = tmem + (uint32_t((warp & 3) * 32) << 16);
        const int key = key0 + r;
        const bool kvalid = key < a.M;
        const float sl2 = a.scale_log2;
        constexpr int HD = D / 2;  // dQ / dV / dK columns per warpgroup
        bool ok = true;
        for (int t = 0; ok && t < ntile; ++t) {
            const int buf = t & 1;
            int h, i;
            tile_of(t, h, i);
            const float* lse2 = reinterpret_cast<const float*>(smem + C::LD_OFF + buf * C::LD_BYTES);
            const float* dsum = lse2 + C::BM;
            // the buffer's LSE/D record (the MMA issuer waited for it too; this
            // wait makes the copied data visible to these threads)
            bool got = mbar_wait(bar(C::B_QFULL + buf), (t >> 1) & 1, wc, FA_SITE_SOFTMAX_S) &&
                       mbar_wait(bar(C::B_S), t & 1, wc, FA_SITE_SOFTMAX_S);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // ---- P^T = exp2(scale log2e S^T - LSE log2e): 16-bit into TMEM [64 wg, 64 wg + 32).
            // Only a tile that straddles the diagonal needs the causal mask; keys
            // past M give P = 0 for the whole row; rows past N carry LSE = +inf.
            const bool diag = a.causal && key0 + C::BN - 1 > i * C::BM;
            float p[64];
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const int qb = 64 * wg + 32 * c;  // first query (in the tile) of this chunk
                uint32_t sv[32];
                tmem_ld32(lane_base + C::TM_S + qb, sv);
                tmem_wait_ld();
                uint32_t pw[16];
#pragma unroll
                for (int e = 0; e < 32; e += 4) {
                    const float4 l4 = *reinterpret_cast<const float4*>(lse2 + qb + e);
                    const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        p[32 * c + e + u] = fast_exp2(fmaf(__uint_as_float(sv[e + u]), sl2, -lv[u]));
                }
                if (diag || !kvalid) {
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int qg = i * C::BM + qb + e;  // global query row
                        if (!kvalid || key > qg) p[32 * c + e] = 0.f;
                    }
                }
#pragma unroll
                for (int e = 0; e < 32; e += 2) pw[e / 2] = pack2<T>(p[32 * c + e], p[32 * c + e + 1]);
                tmem_st16(lane_base + C::TM_S + 64 * wg + 16 * c, pw);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar(C::B_PT));
            got = mbar_wait(bar(C::B_DP), t & 1, wc, FA_SITE_SOFTMAX_S);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // ---- dS^T = P^T (dP^T - D): 16-bit into TMEM [128 + 64 wg, +32) and into
            // smem as dS [query half wg][key row r][64 queries], 128-byte swizzled.  The
            // smem copy is written last: the dS buffer holds the previous tile's staged
            // dQ boxes until the reducer has read them.
            uint32_t dws[2][16];
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const int qb = 64 * wg + 32 * c;
                uint32_t dv[32];
                tmem_ld32(lane_base + C::TM_DP + qb, dv);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; e += 4) {
                    const float4 d4 = *reinterpret_cast<const float4*>(dsum + qb + e);
                    const float d0 = p[32 * c + e] * (__uint_as_float(dv[e]) - d4.x);
                    const float d1 = p[32 * c + e + 1] * (__uint_as_float(dv[e + 1]) - d4.y);
                    const float d2 = p[32 * c + e + 2] * (__uint_as_float(dv[e + 2]) - d4.z);
                    const float d3 = p[32 * c + e + 3] * (__uint_as_float(dv[e + 3]) - d4.w);
                    dws[c][e / 2] = pack2<T>(d0, d1);
                    dws[c][e / 2 + 1] = pack2<T>(d2, d3);
                }
                tmem_st16(lane_base + C::TM_DP + 64 * wg + 16 * c, dws[c]);
            }
            if (t > 0) {
                got = mbar_wait(bar(C::B_STAGED), (t - 1) & 1, wc, FA_SITE_SOFTMAX_S);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
            }
#pragma unroll
            for (int c = 0; c < 2; ++c) {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int cc = 4 * c + u;  // 16-byte chunk (8 queries) within the half
                    const int off = wg * C::SUB_BYTES + r * 128 + ((cc ^ (r & 7)) << 4);
                    *reinterpret_cast<uint4*>(smem + C::DS_OFF + off) =
                        make_uint4(dws[c][4 * u], dws[c][4 * u + 1], dws[c][4 * u + 2], dws[c][4 * u + 3]);
                }
            }
            tmem_wait_st();
            fence_async_shared();  // the tensor core reads dS through the async proxy
            tc_fence_before();
            mbar_arrive(bar(C::B_DS));
            // ---- dQ (query row r) -> fp32 accumulator.  The row's columns of this
            // warpgroup are read out of TMEM first, so that dP^T(t+1) may overwrite
            // them at once, then staged as box k = columns [32k, 32k + 32) in the Q
            // slot (boxes 0 .. NSUB-1) and the dO slot (the rest) of this tile; the
            // reducer warp adds them to the accumulator.
            got = mbar_wait(bar(C::B_DQ), t & 1, wc, FA_SITE_SOFTMAX_O);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            tc_fence_after();
            constexpr int NB = HD / 32;  // boxes per warpgroup
            uint32_t v[NB][32];
#pragma unroll
            for (int x = 0; x < NB; ++x) tmem_ld32(lane_base + C::TM_DQ + 32 * (wg * NB + x), v[x]);
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(bar(C::B_DQFREE));
#pragma unroll
            for (int x = 0; x < NB; ++x) {
                const int k = wg * NB + x;
                uint8_t* box = smem + stage_box(k, buf);
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    *reinterpret_cast<uint4*>(box + r * 128 + ((u ^ (r & 7)) << 4)) =
                        make_uint4(v[x][4 * u], v[x][4 * u + 1], v[x][4 * u + 2], v[x][4 * u + 3]);
            }
            fence_async_shared();  // the reductions read the boxes through the async proxy
            mbar_arrive(bar(C::B_STAGEFULL));
        }
        // ---- dK (times scale) and dV of this CTA's keys: key row r, columns
        // [wg d/2, wg d/2 + d/2).  tcgen05.ld is warp-collective: every lane loads,
        // whether or not its key exists; only the stores depend on it.
        if (ok && ntile > 0) {
            const bool got = mbar_wait(bar(C::B_FINAL), 0, wc, FA_SITE_DRAIN);
            ok = __all_sync(0xffffffffu, got);
            tc_fence_after();
        }
        if (ok) {
            T* dvrow = reinterpret_cast<T*>(a.dv) + ((size_t(b) * a.M + key) * a.Hkv + kvh) * D + wg * HD;
            T* dkrow = reinterpret_cast<T*>(a.dk) + ((size_t(b) * a.M + key) * a.Hkv + kvh) * D + wg * HD;
#pragma unroll 1
            for (int c = 0; c < HD / 32; ++c) {
                uint32_t vv[32], kv[32];
                if (ntile > 0) {
                    tmem_ld32(lane_base + C::TM_DV + wg * HD + c * 32, vv);
                    tmem_ld32(lane_base + C::TM_DK + wg * HD + c * 32, kv);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) vv[e] = kv[e] = 0u;
                }
                if (!kvalid) continue;
                const float s = a.scale;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    uint4 wv, wk;
                    wv.x = pack2<T>(__uint_as_float(vv[8 * u]), __uint_as_float(vv[8 * u + 1]));
                    wv.y = pack2<T>(__uint_as_float(vv[8 * u + 2]), __uint_as_float(vv[8 * u + 3]));
                    wv.z = pack2<T>(__uint_as_float(vv[8 * u + 4]), __uint_as_float(vv[8 * u + 5]));
                    wv.w = pack2<T>(__uint_as_float(vv[8 * u + 6]), __uint_as_float(vv[8 * u + 7]));
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
    // all of this CTA's work is issued: the dQ conversion may launch once every
    // CTA got here (it waits for the grid to complete before reading dQ)
    if (threadIdx.x == 0) grid_dep_launch_dependents();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

template <int D, typename T>
cudaError_t launch_all(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdo, const CUtensorMap& tdq, const BackwardArgs& a,
                       cudaStream_t stream) {
    using C = BwdCfg<D>;
    const long long prow = (long long)a.B * a.Hq * a.n_qtiles * 128;
    const long long nb0 = (prow + 7) / 8;
    if (nb0 > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    dsum_kernel<D, T><<<dim3((unsigned)nb0), dim3(256), 0, stream>>>(a);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    auto kern = backward_kernel<D, T>;
    static std::atomic<unsigned> configured{0};
    err = configure_kernel_once(kern, configured);
    if (err != cudaSuccess) return err;
    const long long nblocks = (long long)a.n_ktiles * a.B * a.Hkv;
    if (nblocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    // The backward kernel and the dQ conversion are programmatic dependents of
    // the launch before them: their launch and set-up overlap its tail.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)nblocks);
    cfg.blockDim = dim3(kBwdThreads);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if ((err = cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, tdo, tdq, a)) != cudaSuccess) return err;
    const long long n4 = (long long)a.B * a.N * a.Hq * D / 4;
    const long long nb2 = (n4 + 255) / 256;
    if (nb2 > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    cfg.gridDim = dim3((unsigned)nb2);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    return cudaLaunchKernelEx(&cfg, dq_convert_kernel<T>, a, n4);
}

}  // namespace

cudaError_t launch_backward(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const CUtensorMap& tdq, const BackwardArgs& a,
                            int d, int dtype, cudaStream_t stream) {
    if (d == 128)
        return dtype == 0 ? launch_all<128, __half>(tq, tk, tv, tdo, tdq, a, stream)
                          : launch_all<128, __nv_bfloat16>(tq, tk, tv, tdo, tdq, a, stream);
    if (d == 64)
        return dtype == 0 ? launch_all<64, __half>(tq, tk, tv, tdo, tdq, a, stream)
                          : launch_all<64, __nv_bfloat16>(tq, tk, tv, tdo, tdq, a, stream);
    return cudaErrorInvalidValue;
}

}  // namespace fa
