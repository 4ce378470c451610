// fa_fwd_pair.cu -- forward attention on CTA pairs (sm_103a, cluster of 2).
//
// Same result as the other forward kernels (O and LSE of exact attention,
// online softmax with the conditional rescale; FlashAttention-4 blog,
// "Forward pass"), with the tensor-core work of two SMs fused into one
// M = 256 product (tcgen05 .cta_group::2).  A pair of CTAs owns 256 query rows
// (128 per CTA) and streams keys in blocks of 256:
//
//   S = Q K_j^T   M = 256, N = 256 keys: each CTA holds its 128 query rows
//                 and 128 of the block's keys; each CTA's tensor memory gets
//                 its rows x all 256 keys.
//   O += P V_j    M = 256, N = 128 (head dim), K = 256 keys: P from each
//                 CTA's tensor memory, V split by head-dim columns (64 each).
//
// Per SM and key block this halves both the K/V bytes that TMA writes into
// shared memory and the operand bytes the tensor core reads from it, compared
// with one CTA running the same 128 x 256 product alone -- on GB300 the
// single-CTA form is bounded by shared-memory bandwidth, not by the tensor
// core.
//
// Tensor memory (512 columns, same layout in both CTAs): S cols 0-255 (fp32),
// P cols 256-383 (bf16 pairs), O cols 384-511 (fp32).
//
// Roles (384 threads per CTA): warps 0-3 and 4-7 are two softmax warpgroups
// splitting each row's 256 columns; warp 8 loads Q and K, warp 10 loads V
// (both CTAs, each its own halves); in the even CTA warp 9 issues the S
// products and warp 11 the P V products, committing to both CTAs' barriers.
// Barriers the issuers wait on live in the even CTA: the odd CTA's TMA loads
// and softmax arrivals count there.
//
// Fixed-length and packed varlen inputs.
#include "fa_exp2.cuh"
#include "fa_internal.h"
#include "fa_sched.cuh"

namespace fa {
namespace {

constexpr int kPThreads = 384;
constexpr int kBlockN = 256;                        // keys per block
constexpr uint32_t kQBytes = 32768;                 // 128 rows x 128 bf16 (this CTA's rows)
constexpr uint32_t kQBox = 16384;                   // 128 rows x 64 bf16
constexpr uint32_t kKHalf = 32768;                  // 128 keys x 128 bf16 (this CTA's keys)
constexpr uint32_t kKBox = 16384;
constexpr uint32_t kVHalf = 32768;                  // 256 keys x 64 bf16 (this CTA's head-dim half)
constexpr int kKS = 3, kVS = 2;                     // ring slots
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kQBytes;
constexpr uint32_t kOffV = kOffK + kKS * kKHalf;
constexpr uint32_t kOffRed = kOffV + kVS * kVHalf;  // row max / sum exchange [2][2][128] float
// Varlen unit tables (fa_sched.cuh); a fixed-length call has none and uses
// the region as the second O staging box.
constexpr uint32_t kOffTab = kOffRed + 2 * 2 * 128 * 4;
static_assert(kOffTab % 1024 == 0 && kTableInts * 4 <= 16384, "tables / second staging box");
constexpr uint32_t kOffBar = kOffTab + 16384;
constexpr uint32_t kOffStg = (kOffBar + 512 + 1023) & ~1023u;   // O staging: 128 rows x 64 bf16 (one TMA box)
constexpr uint32_t kPSmem = kOffStg + 16384;
static_assert(kPSmem <= 232448, "shared memory plan");

constexpr uint32_t kColS = 0, kColP = 256, kColO = 384;
constexpr uint16_t kBoth = 3;                       // CTA mask: both CTAs of the pair

enum : int { kPSiteQEmpty = 61, kPSiteKEmpty, kPSiteVEmpty, kPSiteQFull, kPSiteKFull, kPSiteVFull, kPSiteSFree,
             kPSiteP, kPSiteOFree, kPSiteS, kPSitePV, kPSiteO };

struct PairShared {
    uint64_t q_full, q_empty;
    uint64_t kfull[kKS], kempty[kKS], vfull[kVS], vempty[kVS];
    uint64_t s_full, s_free, p_ready, pv_done, o_done, o_free, drain;
    uint32_t tmem_base;
    int abort_flag;
    int total, maxm;
    Sched sched;
};
static_assert(sizeof(PairShared) <= 512, "barrier block");

// Unit order (fa_sched.cuh): fixed length non-causal head-major with query
// blocks minor; causal longest-first (query blocks from the last) inside L2
// sections of (batch, head) pairs; varlen sequences sorted by block count,
// longest first (FlashAttention-4 blog, "Scheduling").

// Key blocks the pair needs: causal stops at the block holding the last row.
__device__ __forceinline__ int pair_blocks(const Unit& U, int causal) {
    int keys = U.len;
    if (causal) {
        const int last = (U.m + 1) * kBlockN;
        keys = last < keys ? last : keys;
    }
    return (keys + kBlockN - 1) / kBlockN;
}

// S = Q K^T for the pair: M = 256, N = 256, K = d = 128; K-major, 128-B swizzle.
__device__ __forceinline__ void pair_qk(uint32_t d_tmem, uint32_t q_smem, uint32_t k_smem) {
    constexpr uint32_t idesc = idesc_bf16_f32(256, 256, 0, 0);
    const uint64_t qd = sdesc_sw128(q_smem, 16, 1024), kd = sdesc_sw128(k_smem, 16, 1024);
    static_for<8>([&](auto kc) {
        constexpr uint32_t k = kc;
        constexpr uint32_t off = ((k >> 2) * kQBox + (k & 3) * 32) >> 4;   // Q and K halves share the layout
        umma_ss_k<off, off, 2>(d_tmem, qd, kd, idesc, k > 0);
    });
}

// O (+)= P V for the pair: M = 256, N = 128, K = 256 keys; P from tensor
// memory (8 columns per 16 keys), V MN-major, one 64-wide head-dim chunk per CTA.
__device__ __forceinline__ void pair_pv(uint32_t d_tmem, uint32_t p_tmem, uint32_t v_smem, uint32_t acc) {
    constexpr uint32_t idesc = idesc_bf16_f32(256, 128, 0, 1);
    const uint64_t vd = sdesc_sw128(v_smem, kVHalf, 1024);
    static_for<16>([&](auto kc) {
        constexpr uint32_t k = kc;
        umma_ts_k<k * 8, ((k * 2048) >> 4), 2>(d_tmem, p_tmem, vd, idesc, (acc | k) != 0);
    });
}

__device__ __forceinline__ bool pnamed_bar_or(int id, int n, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r) : "r"((uint32_t)pred), "r"(id), "r"(n) : "memory");
    return r != 0;
}

// Bounded wait on a phase this thread cannot report through (end-of-kernel drains).
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(smem_u32(bar), parity) && globaltimer_ns() - t0 < kWaitLimitNs) {}
}

// kEmu16: of every 16 column pairs of a row half, how many take their exp2
// from the FMA-pipe polynomial (fa_exp2.cuh) instead of MUFU.EX2
// (FlashAttention-4 blog, "Faster exponential").  kDbg: the debug counters
// are armed (a separate build of the kernel: their tests in the softmax loop
// cost 1-4 % of the forward).
template <int kEmu16, bool kDbg>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kPThreads, 1)
fwd_pair_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap to, const FwdArgs a) {
    extern __shared__ __align__(1024) uint8_t dsm[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t base = smem_u32(dsm);
    // Both CTAs run the same code, so both see the same base and return together.
    if (base & 1023u) {
        if (tid == 0 && atomicCAS(&a.status->code, 0, -1) == 0) a.status->where = 600;
        return;
    }
    // With cluster dimensions (2, 1, 1) the rank in the pair is blockIdx.x & 1.
    const bool leader = cluster_rank() == 0;
    PairShared& sh = *reinterpret_cast<PairShared*>(dsm + kOffBar);
    float* red = reinterpret_cast<float*>(dsm + kOffRed);   // [2 parity][2 halves][128 rows]
    const uint32_t sQ = base + kOffQ, sK = base + kOffK, sV = base + kOffV;
    // Pair index and count, and this CTA's rank, are re-read from special
    // registers where used rather than held (the softmax has no registers to spare).
#define PAIR_ID ((int)(blockIdx.x >> 1))
#define NUM_PAIRS ((int)(gridDim.x >> 1))
#define RANK ((int)(blockIdx.x & 1))

    if (tid == 0) {
        mbar_init(&sh.q_full, 1);
        mbar_init(&sh.q_empty, 1);
        for (int i = 0; i < kKS; ++i) { mbar_init(&sh.kfull[i], 1); mbar_init(&sh.kempty[i], 1); }
        for (int i = 0; i < kVS; ++i) { mbar_init(&sh.vfull[i], 1); mbar_init(&sh.vempty[i], 1); }
        mbar_init(&sh.s_full, 1);
        mbar_init(&sh.s_free, 16);     // one arrival per softmax warp of both CTAs
        mbar_init(&sh.p_ready, 16);
        mbar_init(&sh.pv_done, 1);
        mbar_init(&sh.o_done, 1);
        mbar_init(&sh.o_free, 16);
        mbar_init(&sh.drain, 2);       // both issuers of the even CTA
        sh.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 8 && lane == 0) {
        tma_prefetch_desc(&tq);
        tma_prefetch_desc(&tk);
        tma_prefetch_desc(&tv);
    }
    if (warp == 0) {
        tmem_alloc_pair(&sh.tmem_base, 512);
        tmem_relinquish_pair();
    }
    {   // unit tables: both CTAs build the same ones
        int* s_cu = reinterpret_cast<int*>(dsm + kOffTab);
        int* s_order = s_cu + (kMaxVarlenSeqs + 1);
        int* s_pref = s_order + kMaxVarlenSeqs;
        build_sched_tables(a, s_cu, s_order, s_pref, &sh.maxm, &sh.total, tid, kPThreads);
        __syncthreads();
        if (tid == 0) {
            sh.sched.B = a.B; sh.sched.Hq = a.Hq; sh.sched.N = a.N; sh.sched.causal = a.causal;
            sh.sched.varlen = a.varlen; sh.sched.num_m = sh.maxm; sh.sched.maxm = sh.maxm;
            sh.sched.sec = a.l2_section; sh.sched.total = sh.total;
            sh.sched.zz = a.causal && !a.varlen && !a.naive && sh.maxm % 2 == 0;
            sh.sched.naive = a.naive;
            sh.sched.s_cu = s_cu; sh.sched.s_order = s_order; sh.sched.s_pref = s_pref;
        }
    }
    tc_fence_before();
    cluster_sync_all();   // barriers of both CTAs initialised before any remote arrival
    tc_fence_after();
    // Read through shared memory on every call (keeps the decode state out of
    // the registers of the lean warps).
    const Sched& sched = sh.sched;

    const WaitCtx wc{&sh.abort_flag, a.status};
    const uint32_t tmem = sh.tmem_base;
    const int group = a.Hq / a.Hkv;
    // Cluster address of the even CTA's copy of a barrier (computed where
    // used: the softmax threads have no registers to spare).
    auto lead = [](uint64_t* bar) { return mapa_rank(smem_u32(bar), 0); };

    // Register split: 2 * 128 * 224 + 128 * 56 == 384 * 168.
    if (warp >= 8) {
        regs_dec<56>();
        if (warp == 8) {
            // --------------------------------------------------- Q and K loader
            if (lane == 0) {
                uint32_t kit = 0, uc = 0;
                bool ok = true;
                for (int n = 0; ok; ++n) {
                    const int u = sched.nth(PAIR_ID, NUM_PAIRS, n);
                    Unit U;
                    if (!sched.get(u, U)) break;
                    const int hk = U.h / group, nb = pair_blocks(U, a.causal);
                    if (!(ok = mbar_wait(&sh.q_empty, (uc & 1) ^ 1, wc, kPSiteQEmpty))) break;
                    if (leader) mbar_arrive_expect_tx(&sh.q_full, 2 * kQBytes);
                    const int qrow = U.tok0 + U.m * kBlockN + RANK * kTileM;
                    for (int c = 0; c < 2; ++c) tma_load_3d_pair(sQ + c * kQBox, &tq, lead(&sh.q_full), c * 64, U.h, qrow);
                    for (int j = 0; j < nb; ++j) {
                        const uint32_t slot = kit % kKS;
                        if (!(ok = mbar_wait(&sh.kempty[slot], ((kit / kKS) & 1) ^ 1, wc, kPSiteKEmpty))) break;
                        if (leader) mbar_arrive_expect_tx(&sh.kfull[slot], 2 * kKHalf);
                        const uint32_t bar = lead(&sh.kfull[slot]);
                        const int krow = U.tok0 + j * kBlockN + RANK * kTileM;
                        for (int c = 0; c < 2; ++c)
                            tma_load_3d_pair(sK + slot * kKHalf + c * kKBox, &tk, bar, c * 64, hk, krow);
                        ++kit;
                    }
                    ++uc;
                }
                // The even CTA's full barriers count both CTAs' bytes: once the
                // last phases are complete nothing of ours is in flight.
                if (leader) {
                    for (uint32_t i = (kit > kKS ? kit - kKS : 0); i < kit; ++i)
                        drain_wait(&sh.kfull[i % kKS], (i / kKS) & 1);
                    if (uc > 0) drain_wait(&sh.q_full, (uc - 1) & 1);
                }
            }
            __syncwarp();
        } else if (warp == 10) {
            // --------------------------------------------------------- V loader
            if (lane == 0) {
                uint32_t vit = 0;
                bool ok = true;
                for (int n = 0; ok; ++n) {
                    const int u = sched.nth(PAIR_ID, NUM_PAIRS, n);
                    Unit U;
                    if (!sched.get(u, U)) break;
                    const int hk = U.h / group, nb = pair_blocks(U, a.causal);
                    for (int j = 0; j < nb; ++j) {
                        const uint32_t slot = vit % kVS;
                        if (!(ok = mbar_wait(&sh.vempty[slot], ((vit / kVS) & 1) ^ 1, wc, kPSiteVEmpty))) break;
                        if (leader) mbar_arrive_expect_tx(&sh.vfull[slot], 2 * kVHalf);
                        tma_load_3d_pair(sV + slot * kVHalf, &tv, lead(&sh.vfull[slot]),
                                         RANK * 64, hk, U.tok0 + j * kBlockN);
                        ++vit;
                    }
                }
                if (leader)
                    for (uint32_t i = (vit > kVS ? vit - kVS : 0); i < vit; ++i)
                        drain_wait(&sh.vfull[i % kVS], (i / kVS) & 1);
            }
            __syncwarp();
        } else if (warp == 9 && leader) {
            // ------------------------------------------------------- S issuer
            // S(j) for every j: K block loaded and the previous S (of this or
            // the previous unit) copied out by both CTAs.  Q is released after
            // the unit's last S, so the next unit's Q loads while this unit's
            // last block is still in softmax and P V.
            uint32_t kit = 0, uc = 0, gs = 0;
            bool ok = true;
            for (int n = 0; ok; ++n) {
                const int u = sched.nth(PAIR_ID, NUM_PAIRS, n);
                Unit U;
                if (!sched.get(u, U)) break;
                const int nb = pair_blocks(U, a.causal);
                if (!(ok = mbar_wait_w(&sh.q_full, uc & 1, wc, kPSiteQFull))) break;
                for (int j = 0; j < nb; ++j) {
                    const uint32_t kslot = kit % kKS;
                    if (!(ok = mbar_wait_w(&sh.kfull[kslot], (kit / kKS) & 1, wc, kPSiteKFull))) break;
                    ++kit;
                    if (gs > 0 && !(ok = mbar_wait_w(&sh.s_free, (gs - 1) & 1, wc, kPSiteSFree))) break;
                    tc_fence_after();
                    pair_qk(tmem + kColS, sQ, sK + kslot * kKHalf);
                    umma_commit_pair_w(&sh.s_full, kBoth);
                    umma_commit_pair_w(&sh.kempty[kslot], kBoth);
                    if (j + 1 == nb) umma_commit_pair_w(&sh.q_empty, kBoth);
                    ++gs;
                }
                ++uc;
            }
            umma_commit_pair_w(&sh.drain, 1);   // this CTA only
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(smem_u32(&sh.drain), 0) && globaltimer_ns() - t0 < kWaitLimitNs) {}
            __syncwarp();
        } else if (warp == 11 && leader) {
            // ----------------------------------------------------- P V issuer
            // A warp of its own, so that neither product kind waits behind the
            // other's issue (the tensor core's queue is short: issuing blocks
            // until earlier products drain).
            uint32_t vit = 0, uc = 0, gp = 0;
            bool ok = true;
            for (int n = 0; ok; ++n) {
                const int u = sched.nth(PAIR_ID, NUM_PAIRS, n);
                Unit U;
                if (!sched.get(u, U)) break;
                const int nb = pair_blocks(U, a.causal);
                for (int j = 0; j < nb; ++j) {
                    const uint32_t vslot = vit % kVS;
                    if (!(ok = mbar_wait_w(&sh.vfull[vslot], (vit / kVS) & 1, wc, kPSiteVFull))) break;
                    ++vit;
                    if (j == 0 && !(ok = mbar_wait_w(&sh.o_free, (uc & 1) ^ 1, wc, kPSiteOFree))) break;
                    if (!(ok = mbar_wait_w(&sh.p_ready, gp & 1, wc, kPSiteP))) break;
                    tc_fence_after();
                    pair_pv(tmem + kColO, tmem + kColP, sV + vslot * kVHalf, j > 0);
                    umma_commit_pair_w(&sh.pv_done, kBoth);
                    umma_commit_pair_w(&sh.vempty[vslot], kBoth);
                    ++gp;
                }
                if (!ok) break;
                umma_commit_pair_w(&sh.o_done, kBoth);
                ++uc;
            }
            umma_commit_pair_w(&sh.drain, 1);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(smem_u32(&sh.drain), 0) && globaltimer_ns() - t0 < kWaitLimitNs) {}
            __syncwarp();
        }
    } else {
        regs_inc<224>();
        // ------------------------------------------------------------ softmax
        const int x = warp >> 2;                      // which half of the 256 columns
        const int r = (warp & 3) * 32 + lane;         // row == TMEM lane
        const uint32_t lb = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + lb + kColS + x * 128;
        const uint32_t tP = tmem + lb + kColP + x * 64;
        const uint32_t tO = tmem + lb + kColO + x * 64;
        const float scale = a.scale_log2;
        uint32_t sc = 0, pc = 0, ucd = 0;   // S phases, P V phases, epilogues done
        uint32_t ep = 0;   // barrier epoch: exchange buffers alternate with it
        bool ok = true;
        bool first = true;                   // no P V precedes this CTA's first block
        int u_pend = -1;                     // unit whose output is still in TMEM
        float l_pend = 0.f, m_pend = 0.f;
        // Epilogue of unit up (run after the next unit's first P is out, so
        // the wait for the unit's last P V overlaps that block): whole-row sum
        // from the two halves, O / l, LSE; then O's columns are free for the
        // next unit's first P V.
        auto epilogue = [&](int up, float lp, float mp, bool okw) -> bool {
            Unit U;
            sched.get(up, U);
            const int m = U.m * 2 + RANK;
            const int qi = m * kTileM + r;
            okw = mbar_wait(&sh.o_done, ucd & 1, wc, kPSiteO) && okw;
            ++ucd;
            tc_fence_after();
            // Epilogue: whole-row sum from the two halves, O / l, LSE.
            float* rl = red + (ep & 1) * 256;
            rl[x * 128 + r] = lp;
            ++ep;
            // The previous unit's O stores have read the staging boxes before
            // anyone passes the barrier below and refills them.
            if (x == 0 && r == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
            if (pnamed_bar_or(2, 256, !okw)) return false;
            const float lt = rl[r] + rl[128 + r];
            const bool valid = qi < U.len;
            const float inv_l = lt > 0.f ? 1.f / lt : 0.f;
            uint4 ov[8];   // this thread's 64 output columns, bf16
#pragma unroll
            for (int c0 = 0; c0 < 64; c0 += 32) {
                uint32_t o[32];
                tmem_ld32(tO + c0, o);
                tmem_wait_ld();
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float* f = reinterpret_cast<const float*>(o + 8 * q);
                    ov[c0 / 8 + q] = make_uint4(pack_bf16x2(f[0] * inv_l, f[1] * inv_l),
                                                pack_bf16x2(f[2] * inv_l, f[3] * inv_l),
                                                pack_bf16x2(f[4] * inv_l, f[5] * inv_l),
                                                pack_bf16x2(f[6] * inv_l, f[7] * inv_l));
                }
            }
            if ((m + 1) * kTileM <= U.len && !a.varlen) {
                // A full tile, fixed length: the two halves into two 128-B-
                // swizzled staging boxes at once (the second in the unused
                // table region), then one thread sends both with TMA stores;
                // their reads of the boxes are waited for by the next epilogue
                // (scattered 16-byte row stores from every thread serialise in
                // the load/store unit).
                uint8_t* srow = dsm + (x ? kOffTab : kOffStg) + r * 128;
#pragma unroll
                for (int q = 0; q < 8; ++q) *reinterpret_cast<uint4*>(srow + ((q ^ (r & 7)) << 4)) = ov[q];
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                asm volatile("bar.sync 2, 256;" ::: "memory");
                if (x == 0 && r == 0) {
                    asm volatile(
                        "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];\n\t"
                        "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%5, %2, %3}], [%6];\n\t"
                        "cp.async.bulk.commit_group;"
                        ::"l"(reinterpret_cast<uint64_t>(&to)), "r"(0), "r"(U.h), "r"(U.tok0 + m * kTileM),
                          "r"(base + kOffStg), "r"(64), "r"(base + kOffTab) : "memory");
                }
            } else if ((m + 1) * kTileM <= U.len) {
                // A full tile, varlen (the tables hold the second box's
                // space): each half in turn through the one staging box.
                uint8_t* srow = dsm + kOffStg + r * 128;
#pragma unroll
                for (int xr = 0; xr < 2; ++xr) {
                    if (x == xr) {
#pragma unroll
                        for (int q = 0; q < 8; ++q) *reinterpret_cast<uint4*>(srow + ((q ^ (r & 7)) << 4)) = ov[q];
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    }
                    asm volatile("bar.sync 2, 256;" ::: "memory");
                    if (x == 0 && r == 0) {
                        asm volatile(
                            "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];\n\t"
                            "cp.async.bulk.commit_group;\n\t"
                            "cp.async.bulk.wait_group.read 0;"
                            ::"l"(reinterpret_cast<uint64_t>(&to)), "r"(xr * 64), "r"(U.h), "r"(U.tok0 + m * kTileM),
                              "r"(base + kOffStg) : "memory");
                    }
                    asm volatile("bar.sync 2, 256;" ::: "memory");
                }
            } else if (valid) {
                uint4* orow = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.o) +
                                                       ((size_t)(U.tok0 + qi) * a.Hq + U.h) * kHeadDim + x * 64);
#pragma unroll
                for (int q = 0; q < 8; ++q) orow[q] = ov[q];
            }
            if (valid && x == 0) {
                const size_t li = a.varlen ? (size_t)U.h * a.N + U.tok0 + qi : ((size_t)U.seq * a.Hq + U.h) * a.N + qi;
                a.lse[li] = lt > 0.f ? (mp + __log2f(lt)) * 0.69314718055994531f : -INFINITY;
            }
            if (kDbg && x == 0 && r == 0 && m * kTileM < U.len)
                dbg_count(a.dbg_visits, (long long)U.h * (a.varlen ? a.N : (long long)a.B * a.N) + U.tok0 + m * kTileM);
            tc_fence_before();
            mbar_arrive_remote_w(lead(&sh.o_free));
            return true;
        };
        for (int n = 0; ok; ++n) {
            const int u = sched.nth(PAIR_ID, NUM_PAIRS, n);
            Unit U;
            if (!sched.get(u, U)) break;
            const int nb = pair_blocks(U, a.causal);
            const int m = U.m * 2 + RANK;         // this CTA's 128-row query tile
            const int qi = m * kTileM + r;
            float m_ref = -INFINITY, l = 0.f;           // l: this half's partial row sum
            bool okw = true;
            for (int j = 0; j < nb; ++j) {
                okw = mbar_wait(&sh.s_full, sc & 1, wc, kPSiteS) && okw;
                ++sc;
                tc_fence_after();
                float s[128];
                {
                    uint32_t* su = reinterpret_cast<uint32_t*>(s);
                    tmem_ld32(tS + 0, *reinterpret_cast<uint32_t(*)[32]>(su + 0));
                    tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(su + 32));
                    tmem_ld32(tS + 64, *reinterpret_cast<uint32_t(*)[32]>(su + 64));
                    tmem_ld32(tS + 96, *reinterpret_cast<uint32_t(*)[32]>(su + 96));
                    tmem_wait_ld();
                }
                tc_fence_before();
                mbar_arrive_remote_w(lead(&sh.s_free));   // the next S may overwrite these columns
                const int k0 = j * kBlockN + x * 128;   // key of column 0 of this half
                if (k0 + 128 > U.len || (a.causal && k0 + 127 > m * kTileM)) {
                    const int lim_len = U.len - k0;
                    const int lim_causal = a.causal ? qi - k0 + 1 : 128;
                    const int lim = lim_len < lim_causal ? lim_len : lim_causal;
#pragma unroll
                    for (int c = 0; c < 128; ++c)
                        if (c >= lim) s[c] = -INFINITY;
                }
                // Row max of this half: three-input max, four chains.
                float mx0 = fmaxf(s[0], s[1]), mx1 = fmaxf(s[2], s[3]), mx2 = fmaxf(s[4], s[5]),
                      mx3 = fmaxf(s[6], s[7]);
#pragma unroll
                for (int c = 8; c < 128; c += 8) {
                    mx0 = fmax3(mx0, s[c], s[c + 1]);
                    mx1 = fmax3(mx1, s[c + 2], s[c + 3]);
                    mx2 = fmax3(mx2, s[c + 4], s[c + 5]);
                    mx3 = fmax3(mx3, s[c + 6], s[c + 7]);
                }
                float* rb = red + (ep & 1) * 256;
                rb[x * 128 + r] = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));
                ++ep;
                if (pnamed_bar_or(2, 256, !okw)) { ok = false; break; }
                const float m_blk = fmaxf(rb[r], rb[128 + r]) * scale;   // whole-row max, log2 units
                const float m_new = fmaxf(m_ref, m_blk);
                // Conditional rescale (FlashAttention-4 blog, "Forward pass"):
                // both halves see the same row maxima, so their warp votes agree.
                const bool jump = (m_ref == -INFINITY) ? (m_new != -INFINITY) : (m_new - m_ref > a.tau);
                const bool rescale = __any_sync(0xffffffffu, jump);
                if (kDbg && lane == 0 && x == 0) dbg_count_rescale(a.dbg_rescale, j > 0, rescale);
                float fac = 1.f;
                if (rescale) {
                    fac = (m_ref == -INFINITY) ? 0.f : ex2_mufu(m_ref - m_new);
                    l *= fac;
                    m_ref = m_new;
                }
                const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
                // Exponents two at a time (packed fp32 FMA), exp2 on MUFU
                // (kEmu16 of every 16 pairs on the FMA pipe), row sum in two
                // packed accumulators.
                uint32_t pk[64];
                const uint64_t sc2 = f2_pack(scale, scale), nm2 = f2_pack(-m_use, -m_use);
                uint64_t la = f2_pack(0.f, 0.f), lb = la;
#pragma unroll
                for (int i = 0; i < 64; ++i) {
                    float x0, x1;
                    f2_unpack(f2_fma(f2_pack(s[2 * i], s[2 * i + 1]), sc2, nm2), x0, x1);
                    float p0, p1;
                    if ((i & 15) < kEmu16) {
                        exp2_fma_x2(x0, x1, p0, p1);
                    } else {
                        p0 = ex2_mufu(x0);
                        p1 = ex2_mufu(x1);
                    }
                    if (i & 1) lb = f2_add(lb, f2_pack(p0, p1));
                    else la = f2_add(la, f2_pack(p0, p1));
                    pk[i] = pack_bf16x2(p0, p1);
                }
                {
                    float a0, a1, b0, b1;
                    f2_unpack(la, a0, a1);
                    f2_unpack(lb, b0, b1);
                    l += (a0 + a1) + (b0 + b1);
                }
                // P's columns (and, inside a unit, O) are free once the previous
                // P V is done -- also across units: the previous unit's last
                // P V still reads P.
                if (!first) {
                    okw = mbar_wait(&sh.pv_done, pc & 1, wc, kPSitePV) && okw;
                    ++pc;
                    tc_fence_after();
                    if (j > 0 && rescale) {
#pragma unroll
                        for (int c0 = 0; c0 < 64; c0 += 32) {
                            uint32_t o[32];
                            tmem_ld32(tO + c0, o);
                            tmem_wait_ld();
                            const uint64_t f2 = f2_pack(fac, fac);
#pragma unroll
                            for (int i = 0; i < 32; i += 2) {
                                float y0, y1;
                                f2_unpack(f2_mul(f2_pack(__uint_as_float(o[i]), __uint_as_float(o[i + 1])), f2), y0, y1);
                                o[i] = __float_as_uint(y0);
                                o[i + 1] = __float_as_uint(y1);
                            }
                            tmem_st32(tO + c0, o);
                        }
                    }
                }
#pragma unroll
                for (int st = 0; st < 4; ++st)
                    tmem_st16(tP + st * 16, *reinterpret_cast<const uint32_t(*)[16]>(pk + st * 16));
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive_remote_w(lead(&sh.p_ready));
                first = false;
                if (j == 0 && u_pend >= 0) {   // the previous unit's output
                    if (!epilogue(u_pend, l_pend, m_pend, okw)) { ok = false; break; }
                    u_pend = -1;
                }
            }
            if (!ok) break;
            u_pend = u;
            l_pend = l;
            m_pend = m_ref;
        }
        if (ok && u_pend >= 0) ok = epilogue(u_pend, l_pend, m_pend, true);
    }

    if (warp == 0 && lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");   // O stores complete

    // After an abort the odd CTA cannot observe its own last loads (they count
    // on the even CTA's barriers): give them time to land before its shared
    // memory is released.
    if (sh.abort_flag) {
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 200000ull) {}
    }
    tc_fence_before();
    cluster_sync_all();   // no product, load or remote arrival still targets either CTA
    tc_fence_after();
    if (warp == 0) tmem_dealloc_pair(tmem, 512);
}

#undef PAIR_ID
#undef NUM_PAIRS
#undef RANK

}  // namespace

int g_pairs_resident = 0;

namespace {

template <int E, bool kDbg>
cudaError_t launch_fwd_pair_t(const FwdLaunch& L, cudaStream_t stream) {
    auto kern = fwd_pair_kernel<E, kDbg>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPSmem);
    if (e != cudaSuccess) return e;
    // Persistent: as many pairs as can be resident at once (clusters must fit
    // inside one GPC, so this can be below half the SM count).
    int max_pairs = g_pairs_resident;
    if (max_pairs == 0) {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(2 * (unsigned)(L.num_sms / 2), 1, 1);
        cfg.blockDim = dim3(kPThreads, 1, 1);
        cfg.dynamicSmemBytes = kPSmem;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n < 1) n = L.num_sms / 2;
        max_pairs = g_pairs_resident = n;
    }
    // Upper bound on the unit count (varlen: the kernel computes the exact one).
    const long long units = L.a.varlen ? ((long long)L.a.N / kBlockN + L.a.B) * L.a.Hq
                                       : (long long)L.a.B * L.a.Hq * ((L.a.N + kBlockN - 1) / kBlockN);
    int pairs = (int)(units < max_pairs ? units : max_pairs);
    if (pairs < 1) pairs = 1;
    kern<<<2 * pairs, kPThreads, kPSmem, stream>>>(L.tq, L.tk, L.tv, L.to, L.a);
    return cudaGetLastError();
}

template <bool kDbg>
cudaError_t launch_fwd_pair_d(const FwdLaunch& L, cudaStream_t stream) {
    switch (L.emu16) {
        case 0: return launch_fwd_pair_t<0, kDbg>(L, stream);
        case 1: return launch_fwd_pair_t<1, kDbg>(L, stream);
        case 2: return launch_fwd_pair_t<2, kDbg>(L, stream);
        case 3: return launch_fwd_pair_t<3, kDbg>(L, stream);
        case 4: return launch_fwd_pair_t<4, kDbg>(L, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_fwd_pair(const FwdLaunch& L, cudaStream_t stream) {
    return (L.a.dbg_visits || L.a.dbg_rescale) ? launch_fwd_pair_d<true>(L, stream) : launch_fwd_pair_d<false>(L, stream);
}

}  // namespace fa
