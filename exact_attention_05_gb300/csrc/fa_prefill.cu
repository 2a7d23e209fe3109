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
//   * one CTA per pair of 128-row Q tiles sharing every K/V tile: rows r and
//     r + 128 of one (b, h), or -- causal with an even GQA group -- the same
//     128 rows of query heads h and h + 1, which read the same kv head and
//     so walk the same causal key range (no lone last KV tile for tile 1);
//     10 warps with fixed roles:
//       warps 0-3  softmax of Q tile 0, warps 4-7 softmax of Q tile 1: thread
//                  t of a warpgroup owns query row t of its tile (TMEM lane
//                  t); it reads its S row from TMEM, masks, updates m/l,
//                  writes P (fp16/bf16) back into TMEM over the upper half
//                  of its S row, rescales its O row when needed, and runs
//                  the epilogue (O / l -> smem -> TMA store, LSE -> global);
//                  each warp signals its P with one arrive (after __syncwarp);
//       warp 8     TMA producer: Q0, Q1 once, then K0, V0, K1, V1, ... into a
//                  ring of shared-memory slots, reusing a slot once the S
//                  signal that covers its last reader has fired;
//       warp 9     TMEM allocator and single-thread tcgen05 MMA issuer.
//   * the tensor core ping-pongs between the tiles:
//       ... PV0(j)  QK0(j+1)  PV1(j)  QK1(j+1)  PV0(j+1) ...
//     so the softmax of one tile (S -> P) runs while the other tile's two
//     GEMMs execute; S = Q K^T and O += P V accumulate in fp32 in TMEM, and P
//     is read by the PV MMA straight from TMEM (A operand in tensor memory).
//   * TMEM map (512 columns): S0 [0,128) with P0 in [64,128), S1 [128,256)
//     with P1 in [192,256), O0 [256,256+d), O1 [256+d,256+2d).  QKi(j+1)
//     overwrites the P_i that PVi(j) reads; tcgen05.mma operations issued by
//     one thread execute in issue order, and PVi(j) is issued first.
//   * K/V/Q tiles are 128-byte-swizzled 64-column halves written by TMA and
//     read by the MMA through shared-memory descriptors.
//   * few tcgen05.commit operations, each at the end of a group of MMAs: a
//     commit between two MMAs holds the tensor core until the MMAs before it
//     are done.  S_i(j) is signalled after QK_i(j); since it also covers every
//     earlier MMA of the single issuing thread, O-done is signalled only after
//     a tile's last PV, and ring slots need no signal of their own: the
//     producer reuses the slot of K_m once the last tile's S(m) is signalled,
//     and that of V_m once its S(m+1) is (QK(m+1) follows PV(m)).
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
    static constexpr int NSLOT = D == 128 ? 5 : 8;         // K/V ring depth
    static constexpr int Q_OFF = 0;                        // Q0, Q1
    static constexpr int SLOT_OFF = NQ * TILE_BYTES;
    static constexpr int BAR_OFF = SLOT_OFF + NSLOT * TILE_BYTES;
    // barrier indices
    static constexpr int B_QFULL = 0;
    static constexpr int B_FULL = 1;                       // NSLOT of them
    static constexpr int B_SFULL = 1 + NSLOT;              // one per Q tile (also frees ring slots)
    static constexpr int B_PFULL = 3 + NSLOT;              // one per Q tile
    static constexpr int B_ODONE = 5 + NSLOT;              // one per Q tile
    static constexpr int B_DRAIN = 7 + NSLOT;
    static constexpr int B_QFULL1 = 8 + NSLOT;             // Q1 (B_QFULL covers Q0)
    static constexpr int NBAR = 9 + NSLOT;
    static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
    static constexpr int SMEM_BYTES = MISC_OFF + 16 + 1024;  // + slack to align the base to 1 KB
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
// K/V bytes of the heads whose CTAs are dispatched together: half the 129 MB L2,
// leaving room for the Q and O tiles streaming through it.
constexpr double kL2GroupBytes = 64.0 * 1024 * 1024;

template <int D, typename T>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                   const PrefillArgs a, const int pair_heads, const int ngroups) {
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

    // Which pair of Q tiles.  Tile i covers query head h + i*dh, rows q0 + i*dr:
    // consecutive rows of one head, or (pair_heads) the same rows of two heads.
    // The head units (b, query head or head pair) are cut into `ngroups`
    // consecutive groups of balanced size whose K/V fit in L2 together.  The
    // groups are dispatched one after the other; inside a group the latest
    // (most expensive, when causal) row positions go first, head units
    // fastest, so the CTAs resident at one time read the K/V of few heads.
    const int dh = pair_heads ? 1 : 0;
    const int dr = pair_heads ? 0 : C::BM;
    const int nrow = pair_heads ? a.n_qtiles : (a.n_qtiles + 1) / 2;  // row positions
    const int nhu = pair_heads ? a.Hq / 2 : a.Hq;                      // head units
    const int nbh = a.B * nhu;
    const int lin = blockIdx.x;
    const int gbase = nbh / ngroups, grem = nbh % ngroups;  // groups 0..grem-1 hold gbase + 1
    const int u = lin / nrow;
    const int grp = u < (gbase + 1) * grem ? u / (gbase + 1) : grem + (u - (gbase + 1) * grem) / gbase;
    const int gstart = grp * gbase + min(grp, grem);
    const int gsize = gbase + (grp < grem ? 1 : 0);
    const int gr = lin - gstart * nrow;
    const int pt = nrow - 1 - gr / gsize;
    const int bh = gstart + gr % gsize;
    const int h = (bh % nhu) * (1 + dh);  // query head of tile 0
    const int b = bh / nhu;
    const int kvh = h / (a.Hq / a.Hkv);
    const int q0 = pt * (C::BM + dr);
    const bool t1 = pair_heads || q0 + C::BM < a.N;  // does Q tile 1 exist?
    auto ntiles = [&](int i) -> int {
        const int kv_end = a.causal ? min(a.M, q0 + i * dr + C::BM) : a.M;
        return (kv_end + C::BN - 1) / C::BN;
    };
    const int nt0 = ntiles(0);
    const int nt = t1 ? ntiles(1) : nt0;  // KV tiles the CTA walks (nt >= nt0)

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
        *abort_flag = 0;
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
        // ------------------------------------------------------------- producer
        if (lane == 0) {
            // Q0 and K0 first: the first QK needs nothing else; Q1 follows on its own
            // barrier (the first wave's loads all go out at once, so order matters)
            // Q is read once: it leaves L2 before the K/V tiles other CTAs reuse
            const uint64_t once = l2_policy_evict_first();
            auto load_q = [&](int i, uint32_t full) {
                mbar_arrive_expect_tx(full, C::TILE_BYTES);
                for (int s = 0; s < C::NSUB; ++s)
                    tma_load_4d_hint(sbase + C::Q_OFF + i * C::TILE_BYTES + s * C::SUB_BYTES, &tm_q,
                                     s * 64, h + i * dh, q0 + i * dr, b, full, once);
            };
            load_q(0, bar(C::B_QFULL));
            bool q1_issued = false;
            int L = 0;  // loads issued: K0, V0, K1, V1, ...
            bool ok = true;
            for (; ok && L < 2 * nt; ++L) {
                if (L == 1 && t1) {
                    load_q(1, bar(C::B_QFULL1));
                    q1_issued = true;
                }
                const int slot = L % C::NSLOT;
                if (L >= C::NSLOT) {
                    // The slot's previous load must be consumed.  Its last reader is
                    // the last tile's QK(m) for K_m, or its PV(m) for V_m, which
                    // that tile's QK(m+1) follows; the commit of that QK's S covers
                    // every MMA issued before it.  (The MMA issuer cannot get two
                    // S phases ahead of this wait: it needs the loads that follow.)
                    const int prev = L - C::NSLOT;
                    const int phase = (prev >> 1) + (prev & 1);
                    if (!mbar_wait(bar(C::B_SFULL + (t1 ? 1 : 0)), uint32_t(phase) & 1u, wc,
                                   FA_SITE_PRODUCER_SLOT)) {
                        ok = false;
                        break;
                    }
                }
                mbar_arrive_expect_tx(bar(C::B_FULL + slot), C::TILE_BYTES);
                const uint32_t dst = sbase + C::SLOT_OFF + slot * C::TILE_BYTES;
                const CUtensorMap* map = (L & 1) ? &tm_v : &tm_k;
                for (int s = 0; s < C::NSUB; ++s)
                    tma_load_4d(dst + s * C::SUB_BYTES, map, s * 64, kvh, (L >> 1) * C::BN, b,
                                bar(C::B_FULL + slot));
            }
            // Every issued copy must have landed before the CTA may exit.
            mbar_drain_wait(bar(C::B_QFULL), 0, wc, FA_SITE_DRAIN);
            if (q1_issued) mbar_drain_wait(bar(C::B_QFULL1), 0, wc, FA_SITE_DRAIN);
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
            // shared addresses are below 256 KB), and ring slots and phases are
            // tracked incrementally.
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
            // O_i (+)= P_i V from the V tile in ring slot vs.  Only the tile's last
            // PV signals O-done: otherwise the tile's next QK follows, and the
            // commit of its S (which covers every earlier MMA of this thread) tells
            // the softmax that O holds every product so far.
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

            // ring positions of K_j (load 2j) and V_j (load 2j+1)
            int ks = 0, vs = 1 % C::NSLOT;
            uint32_t kph = 0, vph = (1 / C::NSLOT) & 1;
            auto advance2 = [](int& slot, uint32_t& ph) {
                slot += 2;
                if (slot >= C::NSLOT) {
                    slot -= C::NSLOT;
                    ph ^= 1u;
                }
            };

            bool ok = mbar_wait_spin(bar(C::B_QFULL), 0, wc, FA_SITE_MMA_Q) && wait_slot(ks, kph);
            if (ok) {
                tc_fence_after();
                qk(0, ks);
                if (t1) {
                    ok = mbar_wait_spin(bar(C::B_QFULL1), 0, wc, FA_SITE_MMA_Q);
                    if (ok) {
                        tc_fence_after();
                        qk(1, ks);
                    }
                }
            }
            // Everything a tile's group of MMAs needs (its P, V_j and the next K
            // tile) is complete before the group is issued, so that PV_i(j) and
            // QK_i(j+1) go to the tensor core back to back.  The group's barriers
            // are first tested all at once: a barrier test takes ~100 cycles here,
            // and three of them one after the other (each result deciding whether
            // to issue the next) left the tensor core idle for ~400 cycles between
            // two iterations; independent tests overlap.  If one of them is not
            // complete yet, the bounded waits take over.  V_j and K_{j+1} have
            // normally landed long before; P is the one on the critical path.
            auto ready_all = [&](int tile, int j, bool next_k, int nks, uint32_t nkph,
                                 bool need_vk) -> bool {
                const bool p_ok = mbar_test_wait(bar(C::B_PFULL + tile), uint32_t(j) & 1u);
                const bool v_ok = !need_vk || mbar_test_wait(bar_full0 + 8u * vs, vph);
                const bool k_ok = !need_vk || !next_k || mbar_test_wait(bar_full0 + 8u * nks, nkph);
                if (p_ok && v_ok && k_ok) return true;
                // a phase seen complete stays complete until this thread issues the
                // MMAs that read it, so only the others are waited for
                return (v_ok || wait_slot(vs, vph)) && (k_ok || wait_slot(nks, nkph)) &&
                       (p_ok || mbar_wait_spin(bar(C::B_PFULL + tile), uint32_t(j) & 1u, wc,
                                               FA_SITE_MMA_P));
            };
            for (int j = 0; ok && j < nt; ++j) {
                int nks = ks;
                uint32_t nkph = kph;
                advance2(nks, nkph);  // K_{j+1}
                const bool next_k = j + 1 < nt;  // some tile still needs K_{j+1}
                bool have_vk = false;
                if (j < nt0) {
                    if (!ready_all(0, j, next_k, nks, nkph, true)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    have_vk = true;
                    pv(0, vs, j > 0, j + 1 >= nt0);
                    if (j + 1 < nt0) qk(0, nks);
                }
                if (t1) {
                    if (!ready_all(1, j, next_k, nks, nkph, !have_vk)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    pv(1, vs, j > 0, !next_k);
                    if (next_k) qk(1, nks);
                }
                ks = nks;
                kph = nkph;
                advance2(vs, vph);
            }
            // All MMAs must be complete before TMEM is released.
            mma_commit(bar(C::B_DRAIN));
            mbar_drain_wait(bar(C::B_DRAIN), 0, wc, FA_SITE_DRAIN);
        }
    } else {
        // ------------------------------------------------------------- softmax
        const int tile = warp >> 2;  // 0 or 1
        const int r = threadIdx.x & 127;  // row in tile == TMEM lane
        const int row0 = q0 + tile * dr;
        const int ht = h + tile * dh;  // this tile's query head
        const int row = row0 + r;
        const uint32_t lane_base = tmem + (uint32_t((warp & 3) * 32) << 16);
        const int nti = tile == 0 ? nt0 : nt;
        const bool active = tile == 0 || t1;
        const float sl2 = a.scale_log2;
        // KV tiles [0, jfull) are visible to every row of the tile and lie inside M
        int jfull = a.M / C::BN;
        if (a.causal) jfull = min(jfull, row0 / C::BN);
        float m_ref = -INFINITY;  // exponent reference, log2 units of the scaled logits
        float l = 0.f;
        bool ok = active;
        for (int j = 0; ok && j < nti; ++j) {
            bool got = mbar_wait(bar(C::B_SFULL + tile), j & 1, wc, FA_SITE_SOFTMAX_S);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
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
                    for (int e = 0; e < 16; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
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
        // ------------------------------------------------------------ epilogue
        if (ok) {
            // the tile's last PV is the only one that signals O-done
            const bool got = mbar_wait(bar(C::B_ODONE + tile), 0, wc, FA_SITE_SOFTMAX_O);
            ok = __all_sync(0xffffffffu, got);
        }
        uint8_t* stage = smem + C::Q_OFF + tile * C::TILE_BYTES;  // Q_i is dead by now
        if (ok) {
            tc_fence_after();
            const float inv_l = 1.f / l;
            const uint32_t o_addr = lane_base + C::tm_o(tile);
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
                a.lse[(size_t(b) * a.Hq + ht) * a.N + row] = (m_ref + log2f(l)) * kLn2;
        }
        fence_async_shared();
        named_barrier_sync(1 + tile, 128);
        if (r == 0 && ok && *abort_flag == 0) {
            const uint64_t once = l2_policy_evict_first();  // O is not read again here
            for (int s = 0; s < C::NSUB; ++s)
                tma_store_4d_hint(&tm_o, smem_addr(stage) + s * C::SUB_BYTES, s * 64, ht, row0, b,
                                  once);
            tma_store_commit();
            tma_store_wait_all();
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
    kern<<<dim3((unsigned)nblocks), dim3(kThreads), C::SMEM_BYTES, stream>>>(tq, tk, tv, to, a,
                                                                           pair_heads, (int)ngroups);
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
