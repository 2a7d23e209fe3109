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
//   * a work item is a pair of 128-row Q tiles sharing every K/V tile: rows r
//     and r + 128 of one (b, h), or -- causal with an even GQA group -- the
//     same 128 rows of query heads h and h + 1, which read the same kv head
//     and so walk the same causal key range.  The grid has one CTA per item,
//     in dispatch order (L2 groups of heads, heaviest rows first).  One CTA
//     fits per SM; when the grid has more CTAs than SMs, a CTA that is about
//     to finish its item cancels the launch of the next CTA that has not
//     started yet (cluster launch control) and takes over its item, so the
//     CTAs stay resident and one item's start
//     overlaps the previous one's end: the next item's Q tiles are brought
//     into L2 as soon as it is known and loaded as soon as the current Q
//     tiles are dead, its K/V follow the current ones in the same ring, and
//     its first QK runs during the current epilogue.
//   * 10 warps with fixed roles:
//       warps 0-3  softmax of Q tile 0, warps 4-7 softmax of Q tile 1: thread
//                  t of a warpgroup owns query row t of its tile (TMEM lane
//                  t); it reads its S row from TMEM, masks, updates m/l,
//                  writes P (fp16/bf16) back into TMEM over the upper half
//                  of its S row, rescales its O row when needed, and runs
//                  the epilogue (O / l -> a shared-memory staging buffer ->
//                  TMA store, LSE -> global); each warp signals its P with
//                  one arrive;
//       warp 8     TMA producer and work fetcher: per item Q0, Q1, then K0,
//                  V0, K1, V1, ... into a ring of shared-memory slots, and
//                  the request that takes over the next item;
//       warp 9     TMEM allocator and single-thread tcgen05 MMA issuer.
//   * the tensor core ping-pongs between the tiles:
//       ... PV0(j)  QK0(j+1)  PV1(j)  QK1(j+1)  PV0(j+1) ...
//     so the softmax of one tile (S -> P) runs while the other tile's two
//     GEMMs execute; after a tile's last PV of an item comes its first QK of
//     the next item.  S = Q K^T and O += P V accumulate in fp32 in TMEM, and
//     P is read by the PV MMA straight from TMEM (A operand in tensor memory).
//   * TMEM map (512 columns): S0 [0,128) with P0 in [64,128), S1 [128,256)
//     with P1 in [192,256), O0 [256,256+d), O1 [256+d,256+2d).  QKi(j+1)
//     overwrites the P_i that PVi(j) reads; tcgen05.mma operations issued by
//     one thread execute in issue order, and PVi(j) is issued first.  The
//     first PV of an item overwrites O_i only after the tile's softmax warps
//     have read it out: they signal that item's first P after their epilogue.
//   * K/V/Q tiles are 128-byte-swizzled 64-column halves written by TMA and
//     read by the MMA through shared-memory descriptors.
//   * few tcgen05.commit operations, each at the end of a group of MMAs: a
//     commit between two MMAs holds the tensor core until the MMAs before it
//     are done.  S_i(j) is signalled after QK_i(j); since it also covers every
//     earlier MMA of the single issuing thread, O-done is signalled only after
//     a tile's last PV of an item, and ring slots need no signal of their
//     own: the slot of K_m is free once tile 1's S(m) is signalled, that of
//     V_m once its next S is (the QK after PV1(m)); tile 0's QK reading a K
//     tile is always issued before tile 1's, across items too.  The producer
//     learns of each tile's S signals from a count that the tile's softmax
//     raises as it sees them, not from the barrier's phase parity: it may
//     fall behind while it fetches work, and a count cannot be mistaken two
//     phases on.
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
    static constexpr int BM = 128;                         // rows per Q tile
    static constexpr int BN = 128;                         // keys per KV tile
    static constexpr int NQ = 2;                           // Q tiles per CTA
    static constexpr int NSUB = D / 64;                    // 64-element (128 B) column halves
    static constexpr int SUB_BYTES = 128 * 128;            // 128 rows x 128 B
    static constexpr int TILE_BYTES = NSUB * SUB_BYTES;    // one Q, K or V tile
    static constexpr int NSLOT = D == 128 ? 4 : 8;         // K/V ring depth
    static constexpr int Q_OFF = 0;                        // Q0, Q1
    static constexpr int SLOT_OFF = NQ * TILE_BYTES;
    static constexpr int STG_OFF = SLOT_OFF + NSLOT * TILE_BYTES;  // O staging, 64 columns per tile
    static constexpr int BAR_OFF = STG_OFF + NQ * SUB_BYTES;
    // barrier indices
    static constexpr int B_QFULL = 0;                      // Q0 landed (one phase per item)
    static constexpr int B_QFULL1 = 1;                     // Q1 landed
    static constexpr int B_FULL = 2;                       // NSLOT of them
    static constexpr int B_SFULL = 2 + NSLOT;              // one per Q tile
    static constexpr int B_PFULL = 4 + NSLOT;              // one per Q tile
    static constexpr int B_ODONE = 6 + NSLOT;              // one per Q tile
    static constexpr int B_DRAIN = 8 + NSLOT;
    static constexpr int B_STEAL = 9 + NSLOT;              // answer of a work-stealing request
    static constexpr int B_ITEMF = 10 + NSLOT;             // two: next item posted
    static constexpr int B_ITEME = 12 + NSLOT;             // two: next item read by all
    static constexpr int B_STGF = 14 + NSLOT;              // one per tile: staging written
    static constexpr int B_STGE = 16 + NSLOT;              // one per tile: staging read by TMA
    static constexpr int NBAR = 18 + NSLOT;
    static constexpr int MISC_OFF = (BAR_OFF + NBAR * 8 + 15) & ~15;
    // MISC: +0 TMEM base, +4 abort flag, +8/+12 posted items, +16/+20 counts of
    // tile 0's / tile 1's S signals seen, +32 the 16-byte answer of a stealing request
    static constexpr int SMEM_BYTES = MISC_OFF + 48 + 1024;  // + slack to align the base to 1 KB
    static constexpr int ITEM_READERS = 1 + 8;             // MMA issuer + softmax warps
    // TMEM columns
    static constexpr uint32_t TMEM_COLS = 512;
    __host__ __device__ static constexpr uint32_t tm_s(int i) { return 128u * i; }
    __host__ __device__ static constexpr uint32_t tm_p(int i) { return 128u * i + 64u; }
    __host__ __device__ static constexpr uint32_t tm_o(int i) { return 256u + D * i; }
    static_assert(256 + 2 * D <= 512, "TMEM budget");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

constexpr int kThreads = 320;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only when the max grows by > 2^8
// K/V bytes of the heads whose items are dispatched together: half the 129 MB L2,
// leaving room for the Q and O tiles streaming through it.
constexpr double kL2GroupBytes = 64.0 * 1024 * 1024;

// One work item: a pair of Q tiles.  Tile i covers query head h + i*dh, rows
// q0 + i*dr.  Tile 1 always runs; when it would lie wholly below the last row
// (an odd number of row tiles, rows paired) it is computed over zero-filled Q
// rows and nothing of it is stored, so that every item signals both tiles.
struct PrefillItem {
    int b, h, kvh;
    int q0, dh, dr;
    int nt0, nt;  // KV tiles walked by tile 0 and by tile 1 (nt >= nt0)
};

// How work items map to (b, heads, rows), fixed per launch.  The head units
// (b, query head or head pair) are cut into `ngroups` consecutive groups of
// balanced size (the first `grem` hold gbase + 1 units, the others gbase)
// whose K/V fit in L2 together.  The groups are dispatched one after the other;
// inside a group the latest (most expensive, when causal) row positions go
// first, head units fastest, so that the items in flight at one time read the
// K/V of few heads.
struct PrefillSched {
    int pair_heads;  // causal with an even GQA group: tile 1 is the next query head
    int steal;       // the grid has more CTAs than fit at once: take over pending ones
    int nrow;        // row positions per head unit
    int gbase, grem;
    FastDiv div_nrow, div_g1, div_g0, div_nhu, div_group;  // by nrow, gbase + 1, gbase, units per b, Hq / Hkv
};

__device__ __forceinline__ PrefillItem prefill_item(int lin, const PrefillArgs& a, const PrefillSched& sc) {
    constexpr int BM = 128, BN = 128;
    PrefillItem it;
    it.dh = sc.pair_heads ? 1 : 0;
    it.dr = sc.pair_heads ? 0 : BM;
    const uint32_t u = fast_div(uint32_t(lin), sc.div_nrow);  // head unit of the item
    const uint32_t big = uint32_t(sc.gbase + 1) * uint32_t(sc.grem);
    const bool in_big = u < big;
    const uint32_t grp = in_big ? fast_div(u, sc.div_g1) : uint32_t(sc.grem) + fast_div(u - big, sc.div_g0);
    const int gstart = int(grp) * sc.gbase + min(int(grp), sc.grem);
    const int gr = lin - gstart * sc.nrow;  // position inside the group
    const FastDiv gsize = in_big ? sc.div_g1 : sc.div_g0;
    const int q = int(fast_div(uint32_t(gr), gsize));
    const int pt = sc.nrow - 1 - q;
    const int bh = gstart + (gr - q * int(gsize.d));
    const int b = int(fast_div(uint32_t(bh), sc.div_nhu));
    it.b = b;
    it.h = (bh - b * int(sc.div_nhu.d)) * (1 + it.dh);
    it.kvh = int(fast_div(uint32_t(it.h), sc.div_group));
    it.q0 = pt * (BM + it.dr);
    const bool t1 = sc.pair_heads || it.q0 + BM < a.N;
    auto ntiles = [&](int i) -> int {
        const int kv_end = a.causal ? min(a.M, it.q0 + i * it.dr + BM) : a.M;
        return (kv_end + BN - 1) / BN;
    };
    it.nt0 = ntiles(0);
    it.nt = t1 ? ntiles(1) : it.nt0;
    return it;
}

template <int D, typename T>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                   const PrefillArgs a, const PrefillSched sc) {
    using C = PrefillCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const uint32_t sbase = smem_addr(smem);
    const uint32_t bars = sbase + C::BAR_OFF;
    volatile uint32_t* tmem_holder = reinterpret_cast<volatile uint32_t*>(smem + C::MISC_OFF);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 4);
    volatile int* item_post = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 8);
    const uint32_t s0_seen = sbase + C::MISC_OFF + 16;
    const uint32_t s1_seen = sbase + C::MISC_OFF + 20;
    const uint32_t steal_resp = sbase + C::MISC_OFF + 32;
    auto bar = [&](int i) -> uint32_t { return bars + 8u * uint32_t(i); };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(bar(C::B_QFULL), 1);
        mbar_init(bar(C::B_QFULL1), 1);
        for (int i = 0; i < C::NSLOT; ++i) mbar_init(bar(C::B_FULL + i), 1);
        for (int i = 0; i < C::NQ; ++i) {
            mbar_init(bar(C::B_SFULL + i), 1);
            mbar_init(bar(C::B_PFULL + i), 4);  // one arrive per softmax warp
            mbar_init(bar(C::B_ODONE + i), 1);
        }
        mbar_init(bar(C::B_DRAIN), 1);
        mbar_init(bar(C::B_STEAL), 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(C::B_ITEMF + i), 1);
            mbar_init(bar(C::B_ITEME + i), C::ITEM_READERS);
            mbar_init(bar(C::B_STGF + i), 4);  // one arrive per softmax warp of the tile
            mbar_init(bar(C::B_STGE + i), 1);
        }
        *abort_flag = 0;
        st_release_shared(s0_seen, 0);
        st_release_shared(s1_seen, 0);
        fence_barrier_init();
    }
    if (warp == 8 && lane == 0) {
        prefetch_tensor_map(&tm_q);
        prefetch_tensor_map(&tm_k);
        prefetch_tensor_map(&tm_v);
        prefetch_tensor_map(&tm_o);
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
        // ------------------------------------------------- producer + work fetcher
        if (lane == 0) {
            // Q is read once: it leaves L2 before the K/V tiles other CTAs reuse
            const uint64_t once = l2_policy_evict_first();
            // Waits until a tile's softmax has seen `count` S signals in all.
            auto wait_seen = [&](uint32_t seen, int count) -> bool {
                if (ld_acquire_shared(seen) >= count) return true;
                const uint64_t t0 = global_timer_ns();
                for (uint32_t it = 1;; ++it) {
                    __nanosleep(32);
                    if (ld_acquire_shared(seen) >= count) return true;
                    if ((it & 15u) == 0) {
                        if (*abort_flag) return false;
                        if (global_timer_ns() - t0 > wc.timeout_ns) {
                            record_timeout(abort_flag, a.status, FA_SITE_PRODUCER_SLOT);
                            return false;
                        }
                    }
                }
            };
            int id = blockIdx.x;
            bool can_steal = sc.steal != 0;  // more CTAs than fit at once, and no request came back empty
            bool steal_pending = false;
            uint32_t steal_phase = 0;
            int next = -1;           // the next item, once a stealing request has brought one
            // Reads a landed stealing answer; on success brings the new item's Q tiles
            // into L2, so that their loads, which wait for the current Q tiles' last
            // QK, are short.
            auto take_steal = [&]() -> bool {
                steal_pending = false;
                steal_phase ^= 1u;
                next = clc_cancelled_x(steal_resp);
                if (next < 0) {
                    can_steal = false;
                    return true;
                }
                if (next >= (int)gridDim.x) {  // cannot happen; never index with it
                    record_timeout(abort_flag, a.status, FA_SITE_WORK);
                    next = -1;
                    return false;
                }
                const PrefillItem nx = prefill_item(next, a, sc);
                for (int i = 0; i < C::NQ; ++i) {
                    if (nx.q0 + i * nx.dr >= a.N) continue;  // a tile below the last row
                    for (int s = 0; s < C::NSUB; ++s)
                        tma_prefetch_4d(&tm_q, s * 64, nx.h + i * nx.dh, nx.q0 + i * nx.dr, nx.b);
                }
                return true;
            };
            int L = 0;               // K/V loads issued, all items
            int nq0 = 0, nq1 = 0;    // Q0 / Q1 loads issued (one of each per item)
            int s0 = 0, s1 = 0;      // S signals of tiles 0 / 1 in the items before this one
            bool ok = true;
            while (ok) {
                const PrefillItem it = prefill_item(id, a, sc);
                auto load_q = [&](int i, uint32_t full) {
                    mbar_arrive_expect_tx(full, C::TILE_BYTES);
                    for (int s = 0; s < C::NSUB; ++s)
                        tma_load_4d_hint(sbase + C::Q_OFF + i * C::TILE_BYTES + s * C::SUB_BYTES,
                                         &tm_q, s * 64, it.h + i * it.dh, it.q0 + i * it.dr, it.b, full,
                                         once);
                };
                // Q0's slot is free once the previous item's last QK0 is done
                if (nq0 > 0 && !wait_seen(s0_seen, s0)) {
                    ok = false;
                    break;
                }
                load_q(0, bar(C::B_QFULL));
                ++nq0;
                const int nload = 2 * it.nt;  // K0, V0, K1, V1, ...
                // ask for the next item two KV tiles before this one's last load
                const int steal_at = nload > 4 ? nload - 4 : 0;
                for (int l = 0; l < nload; ++l) {
                    if (l == 1) {
                        if (nq1 > 0 && !wait_seen(s1_seen, s1)) {  // the previous item's last QK1
                            ok = false;
                            break;
                        }
                        load_q(1, bar(C::B_QFULL1));
                        ++nq1;
                    }
                    const int slot = L % C::NSLOT;
                    if (L >= C::NSLOT) {
                        // The slot's previous load must be consumed: K_m's last reader is
                        // QK1(m), V_m's is PV1(m), which the next QK1 follows; the commit
                        // of that QK's S covers every MMA issued before it.  Loads come
                        // in pairs per S1 signal across items, so index arithmetic holds.
                        const int prev = L - C::NSLOT;
                        if (!wait_seen(s1_seen, (prev >> 1) + (prev & 1) + 1)) {
                            ok = false;
                            break;
                        }
                    }
                    mbar_arrive_expect_tx(bar(C::B_FULL + slot), C::TILE_BYTES);
                    const uint32_t dst = sbase + C::SLOT_OFF + slot * C::TILE_BYTES;
                    const CUtensorMap* map = (l & 1) ? &tm_v : &tm_k;
                    for (int s = 0; s < C::NSUB; ++s)
                        tma_load_4d(dst + s * C::SUB_BYTES, map, s * 64, it.kvh, (l >> 1) * C::BN, it.b,
                                    bar(C::B_FULL + slot));
                    ++L;
                    // after the load, so that the request never delays it
                    if (l == steal_at && can_steal) {
                        mbar_arrive_expect_tx(bar(C::B_STEAL), 16);
                        clc_try_cancel(steal_resp, bar(C::B_STEAL));
                        steal_pending = true;
                    } else if (steal_pending && mbar_test_wait(bar(C::B_STEAL), steal_phase)) {
                        if (!take_steal()) {
                            ok = false;
                            break;
                        }
                    }
                }
                if (!ok) break;
                s0 += it.nt0;
                s1 += it.nt;
                if (steal_pending) {
                    if (!mbar_wait(bar(C::B_STEAL), steal_phase, wc, FA_SITE_WORK) || !take_steal()) {
                        ok = false;
                        break;
                    }
                }
                // post item number nq0 (or the end) in slot nq0 & 1, its use (nq0 - 1) / 2
                const int ps = nq0 & 1, use = (nq0 - 1) >> 1;
                if (use > 0 &&
                    !mbar_wait(bar(C::B_ITEME + ps), uint32_t(use - 1) & 1u, wc, FA_SITE_WORK)) {
                    ok = false;
                    break;
                }
                item_post[ps] = next;
                mbar_arrive(bar(C::B_ITEMF + ps));
                if (next < 0) break;
                id = next;
                next = -1;
            }
            // Every issued copy and request must have landed before the CTA may exit.
            if (steal_pending) mbar_drain_wait(bar(C::B_STEAL), steal_phase, wc, FA_SITE_DRAIN);
            if (nq0 > 0) mbar_drain_wait(bar(C::B_QFULL), uint32_t(nq0 - 1) & 1u, wc, FA_SITE_DRAIN);
            if (nq1 > 0) mbar_drain_wait(bar(C::B_QFULL1), uint32_t(nq1 - 1) & 1u, wc, FA_SITE_DRAIN);
            for (int slot = 0; slot < C::NSLOT && slot < L; ++slot) {
                const int last = slot + ((L - 1 - slot) / C::NSLOT) * C::NSLOT;
                mbar_drain_wait(bar(C::B_FULL + slot), (last / C::NSLOT) & 1, wc, FA_SITE_DRAIN);
            }
        }
    } else if (warp == 9) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t fmt = DTypeFmt<T>::value;
            constexpr uint32_t idesc_qk = instr_desc_f16(fmt, 128, 128, 0, 0);  // Q, K both K-major
            constexpr uint32_t idesc_pv = instr_desc_f16(fmt, 128, D, 0, 1);    // V is MN-major
            // Issue must be cheap: the issuing thread shares its SMSP with two
            // softmax warps and the tensor core executes one 128x128x16 MMA every
            // 64 cycles, so descriptors are built once and advanced by constants
            // (the start address sits in the low 14 bits and never carries here:
            // shared addresses are below 256 KB).
            constexpr uint64_t kSlotStep = C::TILE_BYTES >> 4;
            const uint64_t dq0 = smem_desc(sbase + C::Q_OFF, 16, 1024);
            const uint64_t dq1 = dq0 + kSlotStep;
            const uint64_t dk0 = smem_desc(sbase + C::SLOT_OFF, 16, 1024);         // K-major view
            const uint64_t dv0 = smem_desc(sbase + C::SLOT_OFF, C::SUB_BYTES, 1024); // MN-major view
            const uint32_t bar_full0 = bar(C::B_FULL);
            // S_i = Q_i K^T from the K tile in ring slot ks
            auto qk = [&](int i, int ks) {
                const uint64_t da = i ? dq1 : dq0;
                const uint64_t db = dk0 + uint64_t(ks) * kSlotStep;
                const uint32_t d_tmem = tmem + C::tm_s(i);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    // K-major, 128-byte swizzle: k-steps of 16 elements advance 32 bytes
                    // inside a 64-column half; 8-row groups are 1024 bytes apart.
                    const uint64_t off = uint64_t((kk / 4) * C::SUB_BYTES + (kk % 4) * 32) >> 4;
                    mma_ss(d_tmem, da + off, db + off, idesc_qk, kk > 0 ? 1u : 0u);
                }
                mma_commit(bar(C::B_SFULL + i));
            };
            // O_i (+)= P_i V from the V tile in ring slot vs.  Only a tile's last PV
            // of an item signals O-done: otherwise the tile's next QK follows, and
            // the commit of its S (which covers every earlier MMA of this thread)
            // tells the softmax that O holds every product so far.
            auto pv = [&](int i, int vs, bool accumulate, bool last) {
                const uint64_t db = dv0 + uint64_t(vs) * kSlotStep;
                const uint32_t d_tmem = tmem + C::tm_o(i);
                const uint32_t a_tmem = tmem + C::tm_p(i);
#pragma unroll
                for (int kk = 0; kk < C::BN / 16; ++kk) {
                    // V is [key][d] = MN-major for B (N = d): 16 keys = 16 rows of 128 B;
                    // the two 64-column halves are SUB_BYTES apart (leading offset),
                    // 8-key groups 1024 bytes apart (stride offset).  P: 16 keys of
                    // 16-bit values = 8 TMEM columns.
                    mma_ts(d_tmem, a_tmem + kk * 8, db + uint64_t(kk * 16 * 128 >> 4), idesc_pv,
                           (accumulate || kk > 0) ? 1u : 0u);
                }
                if (last) mma_commit(bar(C::B_ODONE + i));
            };
            auto wait_slot = [&](int slot, uint32_t phase) -> bool {
                return mbar_wait_spin(bar_full0 + 8u * slot, phase, wc, FA_SITE_MMA_KV);
            };
            // ring positions of K_j (load 2j of the item) and V_j (load 2j+1), tracked
            // incrementally across items: an item's loads follow the previous one's
            int ks = 0, vs = 1 % C::NSLOT;
            uint32_t kph = 0, vph = (1 / C::NSLOT) & 1;
            auto advance2 = [](int& slot, uint32_t& ph) {
                slot += 2;
                if (slot >= C::NSLOT) {
                    slot -= C::NSLOT;
                    ph ^= 1u;
                }
            };

            // Only plain integers live across the loop: the issuing thread must not
            // wait on local memory between two groups.
            int nt0, nt;  // KV tiles of tiles 0 and 1 in the current item
            {
                const PrefillItem it0 = prefill_item(blockIdx.x, a, sc);
                nt0 = it0.nt0;
                nt = it0.nt;
            }
            uint32_t qph_next = 1;        // Q phase of the next item
            uint32_t pph0 = 0, pph1 = 0;  // P phases of tiles 0 / 1
            int post = 1;                 // number of the next item's post
            bool ok = mbar_wait_spin(bar(C::B_QFULL), 0, wc, FA_SITE_MMA_Q) && wait_slot(ks, kph);
            if (ok) {
                tc_fence_after();
                qk(0, ks);
                ok = mbar_wait_spin(bar(C::B_QFULL1), 0, wc, FA_SITE_MMA_Q);
                if (ok) {
                    tc_fence_after();
                    qk(1, ks);
                }
            }
            // Everything a tile's group of MMAs needs (its P, V_j, the K tile of its
            // next QK and, across items, the next Q tile) is complete before the
            // group is issued, so that the PV and the QK go to the tensor core back
            // to back.  The barriers are first tested all at once (a test takes ~100
            // cycles, and independent tests overlap) and only those not yet seen
            // complete this iteration; if one of them is not complete yet, the
            // bounded waits take over.
            auto ready_all = [&](uint32_t pbar, uint32_t pph, bool need_v, bool need_k, int kslot,
                                 uint32_t kphase, bool need_q, uint32_t qbar) -> bool {
                const bool p_ok = mbar_test_wait(pbar, pph);
                const bool v_ok = !need_v || mbar_test_wait(bar_full0 + 8u * vs, vph);
                const bool k_ok = !need_k || mbar_test_wait(bar_full0 + 8u * kslot, kphase);
                const bool q_ok = !need_q || mbar_test_wait(qbar, qph_next);
                if (p_ok && v_ok && k_ok && q_ok) return true;
                // a phase seen complete stays complete until this thread issues the
                // MMAs that read it, so only the others are waited for
                return (v_ok || wait_slot(vs, vph)) && (k_ok || wait_slot(kslot, kphase)) &&
                       (q_ok || mbar_wait_spin(qbar, qph_next, wc, FA_SITE_MMA_Q)) &&
                       (p_ok || mbar_wait_spin(pbar, pph, wc, FA_SITE_MMA_P));
            };
            while (ok) {
                // the next item (or the end), read from the producer's post when a
                // tile reaches its last group of this item
                int next_id = -2;  // -2: not read yet, -1: none
                int next_nt0 = 0, next_nt = 0;
                // Steady state: both tiles run and neither is at its last group.  This
                // loop is the whole per-group work of the issuer between two groups, so
                // it carries no item bookkeeping.
                int j = 0;
                for (; ok && j + 1 < nt0; ++j) {
                    int nks = ks;
                    uint32_t nkph = kph;
                    advance2(nks, nkph);  // K_{j+1}
                    if (!ready_all(bar(C::B_PFULL), pph0, true, true, nks, nkph, false, 0)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    pv(0, vs, j > 0, false);
                    qk(0, nks);
                    pph0 ^= 1u;
                    if (!ready_all(bar(C::B_PFULL + 1), pph1, false, false, nks, nkph, false, 0)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    pv(1, vs, j > 0, false);
                    qk(1, nks);
                    pph1 ^= 1u;
                    ks = nks;
                    kph = nkph;
                    advance2(vs, vph);
                }
                // The item's last one or two iterations.  A tile's last PV goes out as
                // soon as its P and V are there; the tile's first QK of the next item
                // follows once that item's Q tile has landed: right away, between later
                // groups, or at the latest before the next item begins.
                bool pend0 = false, pend1 = false;  // the next item's QK0(0) / QK1(0) not issued yet
                int k0s = 0;                        // ring position of the next item's K0
                uint32_t k0ph = 0;
                auto try_first_qk = [&](int i, uint32_t qbar) -> bool {
                    if (!mbar_test_wait(qbar, qph_next) || !mbar_test_wait(bar_full0 + 8u * k0s, k0ph))
                        return false;
                    tc_fence_after();
                    qk(i, k0s);
                    return true;
                };
                for (; ok && j < nt; ++j) {
                    int nks = ks;
                    uint32_t nkph = kph;
                    advance2(nks, nkph);  // K_{j+1}, or the next item's K0 after the last V
                    const bool last0 = j + 1 == nt0, last1 = j + 1 == nt;
                    if (next_id == -2) {
                        const int ps = post & 1;
                        if (!mbar_wait_spin(bar(C::B_ITEMF + ps), uint32_t((post - 1) >> 1) & 1u, wc,
                                            FA_SITE_WORK)) {
                            ok = false;
                            break;
                        }
                        next_id = item_post[ps];
                        mbar_arrive(bar(C::B_ITEME + ps));
                        if (next_id >= 0) {
                            const PrefillItem x = prefill_item(next_id, a, sc);
                            next_nt0 = x.nt0;
                            next_nt = x.nt;
                        }
                    }
                    bool v_seen = false, k_seen = false;
                    if (j < nt0) {
                        if (!ready_all(bar(C::B_PFULL), pph0, true, !last0, nks, nkph, false, 0)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        pv(0, vs, j > 0, last0);
                        if (!last0) {
                            qk(0, nks);
                            k_seen = true;
                        } else if (next_id >= 0) {
                            k0s = nks;
                            k0ph = nkph;
                            if (!last1) advance2(k0s, k0ph);
                            pend0 = !try_first_qk(0, bar(C::B_QFULL));
                        }
                        pph0 ^= 1u;
                        v_seen = true;
                    }
                    {
                        if (!ready_all(bar(C::B_PFULL + 1), pph1, !v_seen, !last1 && !k_seen, nks, nkph,
                                       false, 0)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        pv(1, vs, j > 0, last1);
                        if (!last1) {
                            qk(1, nks);
                        } else if (next_id >= 0) {
                            // QK0(0) of the next item goes first: the K0 slot is released
                            // by tile 1's S signal, which must cover both QKs that read it
                            k0s = nks;
                            k0ph = nkph;
                            pend1 = pend0 || !try_first_qk(1, bar(C::B_QFULL1));
                        }
                        pph1 ^= 1u;
                    }
                    if (pend0 && !last1) pend0 = !try_first_qk(0, bar(C::B_QFULL));
                    ks = nks;
                    kph = nkph;
                    advance2(vs, vph);
                }
                if (ok && pend0) {
                    ok = mbar_wait_spin(bar(C::B_QFULL), qph_next, wc, FA_SITE_MMA_Q) && wait_slot(k0s, k0ph);
                    if (ok) {
                        tc_fence_after();
                        qk(0, k0s);
                    }
                }
                if (ok && pend1) {
                    ok = mbar_wait_spin(bar(C::B_QFULL1), qph_next, wc, FA_SITE_MMA_Q) && wait_slot(k0s, k0ph);
                    if (ok) {
                        tc_fence_after();
                        qk(1, k0s);
                    }
                }
                if (!ok || next_id < 0) break;
                nt0 = next_nt0;
                nt = next_nt;
                qph_next ^= 1u;
                ++post;
            }
            // All MMAs must be complete before TMEM is released.
            mma_commit(bar(C::B_DRAIN));
            mbar_drain_wait(bar(C::B_DRAIN), 0, wc, FA_SITE_DRAIN);
        }
    } else {
        // ------------------------------------------------------------- softmax
        const int tile = warp >> 2;  // 0 or 1
        const int r = threadIdx.x & 127;  // row in tile == TMEM lane
        const uint32_t lane_base = tmem + (uint32_t((warp & 3) * 32) << 16);
        const bool poster = (warp & 3) == 0 && lane == 0;  // raises the tile's S count
        int stg_use = 0;                                     // uses of the tile's O staging
        const float sl2 = a.scale_log2;
        int id = blockIdx.x;
        int n = 0;              // items started
        int s_seen = 0;         // S signals of this tile seen, all items
        bool ok = true;
        while (ok) {
            const PrefillItem it = prefill_item(id, a, sc);
            const int row0 = it.q0 + tile * it.dr;
            const int ht = it.h + tile * it.dh;  // this tile's query head
            const int row = row0 + r;
            const int nti = tile == 0 ? it.nt0 : it.nt;
            // KV tiles [0, jfull) are visible to every row of the tile and lie inside M
            int jfull = a.M / C::BN;
            if (a.causal) jfull = min(jfull, row0 / C::BN);
            float m_ref = -INFINITY;  // exponent reference, log2 units of the scaled logits
            float l = 0.f;
            for (int j = 0; ok && j < nti; ++j) {
                bool got = mbar_wait(bar(C::B_SFULL + tile), uint32_t(s_seen) & 1u, wc,
                                     FA_SITE_SOFTMAX_S);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                ++s_seen;
                if (poster) st_release_shared(tile ? s1_seen : s0_seen, s_seen);
                tc_fence_after();
                float s[C::BN];
                {
                    const uint32_t s_addr = lane_base + C::tm_s(tile);
#pragma unroll
                    for (int c = 0; c < C::BN / 32; ++c) {
                        uint32_t v[32];
                        tmem_ld32(s_addr + c * 32, v);
#pragma unroll
                        for (int e = 0; e < 32; ++e) s[c * 32 + e] = __uint_as_float(v[e]);
                    }
                    tmem_wait_ld();
                }
                const int k0 = j * C::BN;
                if (j >= jfull) {
                    int lim = a.M - k0;
                    if (a.causal) lim = min(lim, row - k0 + 1);
#pragma unroll
                    for (int c = 0; c < C::BN; ++c)
                        if (c >= lim) s[c] = -INFINITY;
                }
                // row max: four independent chains of three-input max
                float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int c = 0; c < C::BN; c += 8) {
#pragma unroll
                    for (int u = 0; u < 4; ++u) mx[u] = fmax3(mx[u], s[c + 2 * u], s[c + 2 * u + 1]);
                }
                const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * sl2;
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
                    // O holds every PV product so far: PV(j-1) was issued before QK(j)
                    // by the same thread, and the commit of S(j), which we waited for,
                    // signals once every MMA issued before it is done.
                    const uint32_t o_addr = lane_base + C::tm_o(tile);
#pragma unroll 1
                    for (int c = 0; c < D / 16; ++c) {
                        uint32_t v[16];
                        tmem_ld16(o_addr + c * 16, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
                        tmem_st16(o_addr + c * 16, v);
                    }
                    tmem_wait_st();
                }
                const float neg = (m_ref == -INFINITY) ? 0.f : -m_ref;
                const uint32_t p_addr = lane_base + C::tm_p(tile);
                // p = exp2(s * scale * log2(e) - m_ref), two lanes per packed FMA/ADD
                const uint64_t sl2x2 = f2_pack(sl2, sl2);
                const uint64_t negx2 = f2_pack(neg, neg);
                uint64_t lsum[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int c = q4 * 32 + 2 * e;
                        float x0, x1;
                        f2_unpack(f2_fma(f2_pack(s[c], s[c + 1]), sl2x2, negx2), x0, x1);
                        const float p0 = fast_exp2(x0);
                        const float p1 = fast_exp2(x1);
                        lsum[e & 1] = f2_add(lsum[e & 1], f2_pack(p0, p1));
                        pk[e] = pack2<T>(p0, p1);
                    }
                    tmem_st16(p_addr + q4 * 16, pk);
                }
                {
                    float a0, a1, b0, b1;
                    f2_unpack(lsum[0], a0, a1);
                    f2_unpack(lsum[1], b0, b1);
                    l += (a0 + a1) + (b0 + b1);
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::B_PFULL + tile));
            }
            // ------------------------------------------- next item, then epilogue
            // The next item is read first: when there is none, O can be staged in
            // this tile's Q slot, which no load will refill.
            int next = -1;
            if (ok) {
                const int m = n + 1, ps = m & 1, use = (m - 1) >> 1;
                const bool got = mbar_wait(bar(C::B_ITEMF + ps), uint32_t(use) & 1u, wc, FA_SITE_WORK);
                ok = __all_sync(0xffffffffu, got);
                if (ok) {
                    next = item_post[ps];
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(C::B_ITEME + ps));
                }
            }
            if (ok) {
                // the tile's last PV of the item is the only one that signals O-done
                const bool got = mbar_wait(bar(C::B_ODONE + tile), uint32_t(n) & 1u, wc,
                                           FA_SITE_SOFTMAX_O);
                ok = __all_sync(0xffffffffu, got);
            }
            if (ok) {
                // O / l -> shared memory (128-byte swizzle, as the TMA store reads it)
                // -> global memory.  Staging is the tile's 64-column buffer, one half
                // at a time, or after the CTA's last item the tile's Q slot, all of O
                // at once.  Every warp writes its 32 rows and signals; the tile's
                // first thread stores and frees the buffer once the store has read
                // it.  mbarriers, not named barriers: every wait stays bounded even if
                // the tile's warps part ways on a timeout.
                tc_fence_after();
                const PrefillItem it = prefill_item(id, a, sc);
                const int ht = it.h + tile * it.dh;  // this tile's query head
                const int row0 = it.q0 + tile * it.dr;
                const float inv_l = 1.f / l;
                const uint32_t o_addr = lane_base + C::tm_o(tile);
                const int hpp = next < 0 ? C::NSUB : 1;  // 64-column halves per staging pass
                uint8_t* buf = next < 0 ? smem + C::Q_OFF + tile * C::TILE_BYTES
                                        : smem + C::STG_OFF + tile * C::SUB_BYTES;
#pragma unroll 1
                for (int h0 = 0; ok && h0 < C::NSUB; h0 += hpp, ++stg_use) {
                    if (stg_use > 0) {
                        const bool got = mbar_wait(bar(C::B_STGE + tile), uint32_t(stg_use - 1) & 1u, wc,
                                                   FA_SITE_SOFTMAX_O);
                        if (!__all_sync(0xffffffffu, got)) {
                            ok = false;
                            break;
                        }
                    }
#pragma unroll 1
                    for (int c = 2 * h0; c < 2 * (h0 + hpp); ++c) {  // 32-column chunks
                        uint32_t v[32];
                        tmem_ld32(o_addr + c * 32, v);
                        tmem_wait_ld();
                        uint8_t* sub = buf + (c / 2 - h0) * C::SUB_BYTES + r * 128;
#pragma unroll
                        for (int qd = 0; qd < 4; ++qd) {
                            uint32_t w[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int x = qd * 8 + 2 * e;
                                w[e] = pack2<T>(__uint_as_float(v[x]) * inv_l, __uint_as_float(v[x + 1]) * inv_l);
                            }
                            const int chunk = (c & 1) * 4 + qd;
                            *reinterpret_cast<uint4*>(sub + ((chunk ^ (r & 7)) << 4)) =
                                make_uint4(w[0], w[1], w[2], w[3]);
                        }
                    }
                    fence_async_shared();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(C::B_STGF + tile));
                    if (r == 0) {
                        if (!mbar_wait(bar(C::B_STGF + tile), uint32_t(stg_use) & 1u, wc, FA_SITE_SOFTMAX_O)) {
                            ok = false;
                        } else {
                            if (row0 < a.N && *abort_flag == 0) {
                                const uint64_t once = l2_policy_evict_first();  // O is not read again
                                for (int hh = 0; hh < hpp; ++hh)
                                    tma_store_4d_hint(&tm_o, smem_addr(buf) + hh * C::SUB_BYTES, (h0 + hh) * 64,
                                                      ht, row0, it.b, once);
                                tma_store_commit();
                            }
                            tma_store_wait_all();  // the store has read the buffer
                            mbar_arrive(bar(C::B_STGE + tile));
                        }
                    }
                    ok = __all_sync(0xffffffffu, ok);
                }
                if (ok && a.lse != nullptr && row < a.N)
                    a.lse[(size_t(it.b) * a.Hq + ht) * a.N + row] = (m_ref + log2f(l)) * kLn2;
                tc_fence_before();
            }
            if (!ok || next < 0) break;
            id = next;
            ++n;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// The multiplier and shift of fast_div for the divisor d >= 1.
FastDiv make_fast_div(uint32_t d) {
    uint32_t s = 0;
    while ((uint64_t(1) << s) < d) ++s;
    const uint64_t m = ((uint64_t(1) << 32) * ((uint64_t(1) << s) - d)) / d + 1;
    return FastDiv{d, uint32_t(m), s};
}

template <int D, typename T>
cudaError_t launch_prefill_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                             const CUtensorMap& to, const PrefillArgs& a, cudaStream_t stream) {
    using C = PrefillCfg<D>;
    auto kern = prefill_kernel<D, T>;
    static std::atomic<unsigned> configured{0};
    cudaError_t err = configure_kernel_once(kern, configured);
    if (err != cudaSuccess) return err;
    // causal with an even GQA group: pair the same rows of two query heads
    const int pair_heads = (a.causal && (a.Hq / a.Hkv) % 2 == 0) ? 1 : 0;
    const long long nbh = (long long)a.B * (pair_heads ? a.Hq / 2 : a.Hq);
    const long long nblocks = pair_heads ? (long long)a.n_qtiles * nbh
                                         : (long long)((a.n_qtiles + 1) / 2) * nbh;
    if (nblocks <= 0 || nblocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    // L2 groups: as many as it takes for each group's K/V to fit in kL2GroupBytes
    const double kv_bytes = 2.0 * a.M * D * sizeof(T) * (double)a.B * a.Hkv;
    long long ngroups = (long long)std::ceil(kv_bytes / kL2GroupBytes);
    ngroups = ngroups < 1 ? 1 : (ngroups > nbh ? nbh : ngroups);
    // one CTA fits per SM; a grid that fits at once has no pending CTAs to take over
    int dev = 0, sms = 0;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
    if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return err;
    PrefillSched sc;
    sc.pair_heads = pair_heads;
    sc.steal = nblocks > sms ? 1 : 0;
    sc.nrow = pair_heads ? a.n_qtiles : (a.n_qtiles + 1) / 2;
    sc.gbase = (int)(nbh / ngroups);
    sc.grem = (int)(nbh % ngroups);
    sc.div_nrow = make_fast_div((uint32_t)sc.nrow);
    sc.div_g1 = make_fast_div((uint32_t)sc.gbase + 1);
    sc.div_g0 = make_fast_div((uint32_t)sc.gbase);
    sc.div_nhu = make_fast_div((uint32_t)(pair_heads ? a.Hq / 2 : a.Hq));
    sc.div_group = make_fast_div((uint32_t)(a.Hq / a.Hkv));
    kern<<<dim3((unsigned)nblocks), dim3(kThreads), C::SMEM_BYTES, stream>>>(tq, tk, tv, to, a, sc);
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
