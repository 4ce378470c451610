// fa_bwd256.cu -- backward main kernel for head dim d = 256 (sm_103a).
//
// The same gradients as fa_bwd.cu (FlashAttention-4 blog, "Backward pass":
// S, dP, dV, dK, dQ plus the elementwise P and dS), at the head dim where the
// products, not the exponentials, set the pace (paper summary, roofline
// remarks).  At d = 256 neither of the one-CTA kernel's resources fits:
//   * tensor memory: the dK and dV accumulators of a 128-key tile are
//     128 x 256 fp32 each, i.e. all 512 columns together;
//   * shared memory: a 128-row tile of K, V, Q or dO is 64 KB.
// So each work unit (one 128-key tile of one key/value head) runs twice, once
// per head-dim half h of the outputs: pass h keeps dK[:, h], dV[:, h] (128
// columns each) in tensor memory and produces dQ[:, h].  Both passes recompute
// S^T and dP^T over the full head dim (the price of the split: 14 instead of
// 10 product units per tile).
//
// V is only ever the A operand of dP^T = V dO^T, so it lives in tensor memory
// (128 columns of bf16 pairs, copied there once per unit through the dO ring);
// K stays in shared memory (64 KB: S^T reads it K-major, dQ^T head-dim-major).
// That leaves room for two full steps of Q and of dO (64 queries x 256, 32 KB
// each): the next step's copies land while the current step still reads its
// own, instead of waiting for the last product of the step (dK reads Q, dV
// reads dO) and then for a whole L2 round trip.  It also takes V's 64 KB per
// step off the shared-memory operand reads, the bound of these products.
//
// Per step (128 keys x 64 queries), keys on the tensor-memory lanes:
//   S^T  = K Q^T        M 128, N 64, K 256 (both K-major, shared memory)
//   dP^T = V dO^T       M 128, N 64, K 256 (A = V from tensor memory)
//   P^T  = 2^(alpha log2e S^T - LSE log2e)  -> bf16 into tensor memory
//   dS^T = P^T (dP^T - D)                   -> bf16 into shared memory
//   dV_h += P^T dO_h    M 128, N 128, K 64  (A = P^T from tensor memory)
//   dK_h += dS^T Q_h    M 128, N 128, K 64
//   dQ_h^T = K_h^T dS^T M 128 (head-dim half), N 64 (queries), K 128 (keys)
// Tensor memory: dK_h 0-127, dV_h 128-255, V 256-383, S^T / P^T 384-447, and
// dP^T 448-511, which dQ^T reuses once the key rows have read dP^T (the next
// dP^T waits until the dQ drain has read dQ^T out).
// dQ is produced transposed: each of the 128 drain threads owns one head-dim
// column, so each drain warp holds a 32-column strip -- exactly one 128-B
// box of the fp32 accumulator -- and adds it with its own TMA bulk tensor
// reductions, staged 32 query rows at a time (per-thread red.global
// additions of the same data measured far slower: L2 absorbs bulk
// reductions much faster).
//
// Warp roles (512 threads): warps 0-3 and 12-15 key rows (V into tensor
// memory, P^T, dS^T; 32 of the step's 64 queries each); warps 4-7 the dQ
// drain and the dK/dV epilogue; warp 8 loader; warp 9 issues every product
// (warps 10-11 idle).  Deterministic mode orders the dQ additions per
// (half, head, 64-row query step) by key tile with the semaphores of the
// one-CTA kernel.
#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kD6 = 256;
constexpr int kStep = 64;                        // query rows per step
constexpr int kThreads6 = 512;
constexpr uint32_t kKBox6 = 16384;               // 128 rows x 128 B (K, V staging, dS^T)
constexpr uint32_t kQBox6 = 8192;                // 64 rows x 128 B (Q, dO)
constexpr uint32_t kStage6 = 4 * kQBox6;         // one step of Q or dO, all 256 columns
constexpr uint32_t kStgBox6 = 4096;              // dQ staging: 32 query rows x 32 fp32 (128 B)
constexpr uint32_t kOffK6 = 0, kOffQ6 = 4 * kKBox6, kOffDO6 = kOffQ6 + 2 * kStage6,
                   kOffDS6 = kOffDO6 + 2 * kStage6, kOffStat6 = kOffDS6 + kKBox6,   // [2][LSE 64, D 64]
                   kOffStg6 = kOffStat6 + 1024,                                     // one box per drain warp
                   kOffBar6 = kOffStg6 + 4 * kStgBox6;
constexpr uint32_t kSmem6 = kOffBar6 + 1024;
static_assert(kSmem6 <= 232448, "shared memory plan");
static_assert(kOffStat6 % 1024 == 0 && kOffStg6 % 1024 == 0, "swizzled boxes need 1024-byte alignment");
static_assert(2 * kStage6 == 4 * kKBox6, "V is staged in the two dO stages");
constexpr uint32_t kColDK6 = 0, kColDV6 = 128, kColV6 = 256, kColS6 = 384, kColDP6 = 448;

enum : int { k6SiteKvEmpty = 81, k6SiteQEmpty, k6SiteDoEmpty, k6SiteKvFull, k6SiteAcc, k6SiteQFull, k6SiteDoFull,
             k6SiteP, k6SiteDs, k6SiteDqFree, k6SiteS, k6SiteDp, k6SiteDsFree, k6SiteDq, k6SiteDkdv, k6SiteSem,
             k6SiteUnit, k6SiteVFull, k6SiteVReady };

struct Shared6 {
    uint64_t kv_full, kv_empty;     // K (and V's staging) of a unit; empty once the unit's products are done
    uint64_t v_full, v_ready;       // V staged in the dO ring; V copied into tensor memory
    uint64_t q_full[2], q_empty[2], do_full[2], do_empty[2];   // two steps of Q (with LSE, D) and of dO
    uint64_t s_full, dp_full, p_ready, ds_ready, ds_free, dq_full, dq_free, dkdv_done, acc_free, drain;
    uint64_t unit_full[4], unit_empty[4];
    int unit_id[4];
    uint32_t tmem_base;
    int abort_flag;
    int total;
};
static_assert(sizeof(Shared6) <= 1024, "barrier block");

constexpr uint32_t kUnitReaders6 = 1 + 256 + 128;

struct Unit6 {
    int seq, hk, k, tok0, len, n, nq, i0, pass;
};

// Work unit u: base unit u / 2 (one 128-key tile of one key/value head, in
// the one-CTA kernel's order: head-major for non-causal atomic runs and in
// the naive order of fa_set_schedule_order, key-tile-major otherwise, the
// planned list for varlen), head-dim half u % 2.  The two halves of a tile are neighbours in the list, so the CTAs
// running them read the same K and V from L2 at about the same time.
__device__ __forceinline__ bool unit6(const BwdArgs& a, int total, int u, Unit6& U) {
    if (u < 0 || u >= total) return false;
    const int ub = u >> 1;
    U.pass = u & 1;
    if (!a.varlen) {
        const int bh = a.B * a.Hkv;
        int r;
        if ((a.deterministic || a.causal) && !a.naive) {
            U.k = ub / bh;
            r = ub - U.k * bh;
        } else {
            const int nk = (a.N + kTileN - 1) / kTileN;
            r = ub / nk;
            U.k = ub - r * nk;
        }
        U.seq = r / a.Hkv;
        U.hk = r - U.seq * a.Hkv;
        U.tok0 = U.seq * a.N;
        U.len = a.N;
    } else {
        const int4 e = a.units[ub];
        U.seq = e.x;
        U.hk = e.y;
        U.k = e.z;
        U.tok0 = a.cu_s[U.seq];           // sanitised by the plan kernel
        U.len = a.cu_s[U.seq + 1] - U.tok0;
    }
    U.nq = (U.len + kStep - 1) / kStep;
    U.i0 = a.causal ? 2 * U.k : 0;        // first 64-row step that sees key tile k
    if (U.i0 > U.nq) U.i0 = U.nq;
    U.n = (a.Hq / a.Hkv) * (U.nq - U.i0);
    return true;
}

// S^T = K Q^T: M = 128 keys, N = 64 queries, K = 256 in 16 steps over the
// four 64-column boxes of both operands (both K-major).
__device__ __forceinline__ void mma6_s(uint32_t d, uint32_t a_smem, uint32_t b_smem) {
    constexpr uint32_t idesc = idesc_bf16_f32(128, 64, 0, 0);
    const uint64_t ad = sdesc_sw128(a_smem, 16, 1024), bd = sdesc_sw128(b_smem, 16, 1024);
    static_for<16>([&](auto kc) {
        constexpr uint32_t k = kc;
        constexpr uint32_t ao = ((k >> 2) * kKBox6 + (k & 3) * 32) >> 4;
        constexpr uint32_t bo = ((k >> 2) * kQBox6 + (k & 3) * 32) >> 4;
        umma_ss_k<ao, bo>(d, ad, bd, idesc, k > 0 ? 1u : 0u);
    });
}

// dP^T = V dO^T: A = V from tensor memory (lane = key row; K-step k, head-dim
// columns 16k .. 16k+15, in tensor-memory columns 8k .. 8k+7 as bf16 pairs),
// B = dO K-major from shared memory.  M = 128, N = 64, K = 256.
__device__ __forceinline__ void mma6_dp(uint32_t d, uint32_t v_tmem, uint32_t b_smem) {
    constexpr uint32_t idesc = idesc_bf16_f32(128, 64, 0, 0);
    const uint64_t bd = sdesc_sw128(b_smem, 16, 1024);
    static_for<16>([&](auto kc) {
        constexpr uint32_t k = kc;
        constexpr uint32_t bo = ((k >> 2) * kQBox6 + (k & 3) * 32) >> 4;
        umma_ts_k<8 * k, bo>(d, v_tmem, bd, idesc, k > 0 ? 1u : 0u);
    });
}

// dV_h += P^T dO_h: M = 128 keys, N = 128 (the half's head-dim columns, two
// 64-wide boxes), K = 64 queries.  A is bf16 in tensor memory: queries 0-31
// in columns 0-15 of the S region, queries 32-63 in columns 32-47 (each key-
// row warpgroup packs over the first half of the 32 columns it read).
__device__ __forceinline__ void mma6_dv(uint32_t d, uint32_t p_tmem, uint32_t b_smem, uint32_t acc) {
    constexpr uint32_t idesc = idesc_bf16_f32(128, 128, 0, 1);
    const uint64_t bd = sdesc_sw128(b_smem, kQBox6, 1024);
    static_for<4>([&](auto kc) {
        constexpr uint32_t k = kc, col = k * 8 + (k >= 2 ? 16 : 0);
        umma_ts_k<col, ((k * 2048) >> 4)>(d, p_tmem, bd, idesc, (acc | k) != 0);
    });
}

// dK_h += dS^T Q_h: A = dS^T K-major ([key][query], one 128 x 64 box), B = the
// half's Q boxes MN-major.  M = 128, N = 128, K = 64.
__device__ __forceinline__ void mma6_dk(uint32_t d, uint32_t a_smem, uint32_t b_smem, uint32_t acc) {
    constexpr uint32_t idesc = idesc_bf16_f32(128, 128, 0, 1);
    const uint64_t ad = sdesc_sw128(a_smem, 16, 1024), bd = sdesc_sw128(b_smem, kQBox6, 1024);
    static_for<4>([&](auto kc) {
        constexpr uint32_t k = kc, ao = (k * 32) >> 4, bo = (k * 2048) >> 4;
        umma_ss_k<ao, bo>(d, ad, bd, idesc, (acc | k) != 0);
    });
}

// dQ_h^T = K_h^T dS^T: A = K's boxes of half h read MN-major (head dim
// contiguous, the two 64-wide boxes one box apart), B = dS^T MN-major (the
// queries contiguous in each key row).  M = 128, N = 64, K = 128 keys.
__device__ __forceinline__ void mma6_dqt(uint32_t d, uint32_t a_smem, uint32_t b_smem) {
    constexpr uint32_t idesc = idesc_bf16_f32(128, 64, 1, 1);
    const uint64_t ad = sdesc_sw128(a_smem, kKBox6, 1024), bd = sdesc_sw128(b_smem, kKBox6, 1024);
    static_for<8>([&](auto kc) {
        constexpr uint32_t k = kc, off = (k * 2048) >> 4;
        umma_ss_k<off, off>(d, ad, bd, idesc, k > 0);
    });
}

__device__ __forceinline__ void fence6_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void bar6(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }
__device__ __forceinline__ bool bar6_or(int id, int n, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r) : "r"((uint32_t)pred), "r"(id), "r"(n) : "memory");
    return r != 0;
}
__device__ __forceinline__ int ld6_acquire(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void red6_release_add(int* p, int v) {
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void tma6_reduce_add(const CUtensorMap* map, uint32_t src, int x, int y) {
    asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3}], [%1];"
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(src), "r"(x), "r"(y) : "memory");
}
__device__ __forceinline__ void bulk6_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk6_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk6_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence6_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }
__device__ __forceinline__ void drain6(uint64_t* bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(smem_u32(bar), parity) && globaltimer_ns() - t0 < kWaitLimitNs) {}
}

// kDbg: the debug counters are armed (a separate build of the kernel, so
// that their tests cost nothing otherwise).
template <bool kDbg>
__global__ void __launch_bounds__(kThreads6, 1)
bwd256_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
              const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
              const __grid_constant__ CUtensorMap tdq, const BwdArgs a) {
    extern __shared__ __align__(1024) uint8_t dsm[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t base = smem_u32(dsm);
    if (base & 1023u) {  // the swizzled tiles need a 1024-byte aligned window
        if (tid == 0 && atomicCAS(&a.hdr->status.code, 0, -1) == 0) a.hdr->status.where = 310;
        return;
    }
    Shared6& sh = *reinterpret_cast<Shared6*>(dsm + kOffBar6);
    float* s_stat = reinterpret_cast<float*>(dsm + kOffStat6);   // stage s: [LSE * log2(e) 64, D 64]
    const uint32_t sK = base + kOffK6, sQ = base + kOffQ6, sDO = base + kOffDO6, sDS = base + kOffDS6;

    if (tid == 0) {
        mbar_init(&sh.kv_full, 1);
        mbar_init(&sh.kv_empty, 1);
        mbar_init(&sh.v_full, 1);
        mbar_init(&sh.v_ready, 256);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&sh.q_full[s], 1);
            mbar_init(&sh.q_empty[s], 1);
            mbar_init(&sh.do_full[s], 1);
            mbar_init(&sh.do_empty[s], 1);
        }
        mbar_init(&sh.s_full, 1);
        mbar_init(&sh.dp_full, 1);
        mbar_init(&sh.p_ready, 256);
        mbar_init(&sh.ds_ready, 256);
        mbar_init(&sh.ds_free, 1);
        mbar_init(&sh.dq_full, 1);
        mbar_init(&sh.dq_free, 128);
        mbar_init(&sh.dkdv_done, 1);
        mbar_init(&sh.acc_free, 128);
        mbar_init(&sh.drain, 1);
        for (int s = 0; s < 4; ++s) { mbar_init(&sh.unit_full[s], 1); mbar_init(&sh.unit_empty[s], kUnitReaders6); }
        sh.abort_flag = 0;
        int total = 2 * (a.varlen ? a.hdr->total_units : a.B * a.Hkv * ((a.N + kTileN - 1) / kTileN));
        if (a.varlen && (a.hdr->unit_keys != kTileN || a.hdr->unit_heads != 0)) {   // a list planned for other units
            if (atomicCAS(&a.hdr->status.code, 0, -1) == 0) a.hdr->status.where = 202;
            total = 0;
        }
        sh.total = total;
        fence_mbar_init();
    }
    if (warp == 8 && lane == 0) {
        tma_prefetch_desc(&tq);
        tma_prefetch_desc(&tk);
        tma_prefetch_desc(&tv);
        tma_prefetch_desc(&tdo);
        tma_prefetch_desc(&tdq);
    }
    if (warp == 0) {
        tmem_alloc(&sh.tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const WaitCtx wc{&sh.abort_flag, &a.hdr->status};
    const uint32_t tmem = sh.tmem_base;
    const int total = sh.total;
    const int g = a.Hq / a.Hkv;
    const float scale = a.scale_log2;

    // Register split (launch 512 x 128 = 65536): key-row warpgroups 144 each,
    // dQ / epilogue warpgroup 168, loader / issuer warpgroup 56.
    if (warp >= 8 && warp < 12) {
        regs_dec<56>();
        if (warp == 8) {
            // ------------------------------------------------------------ loader
            uint32_t jj = 0, uc = 0;
            // Loads issued on each full barrier, for the drain at the end.
            uint32_t n_q0 = 0, n_q1 = 0, n_do0 = 0, n_do1 = 0, n_kv = 0;
            bool ok = true;
            for (uint32_t n = 0; ok; ++n) {
                int u = -1;
                if (lane == 0) {
                    ok = mbar_wait(&sh.unit_empty[n & 3], ((n >> 2) & 1) ^ 1, wc, k6SiteUnit);
                    if (ok) {
                        // The first unit by block index, later ones in list
                        // order from the workspace counter; the last CTA to
                        // find the list exhausted rewinds it.
                        u = n == 0 ? (int)blockIdx.x : (int)gridDim.x + atomicAdd(&a.hdr->next_unit, 1);
                        if (u >= total) {
                            u = -1;
                            if (atomicAdd(&a.hdr->done_ctas, 1) == (int)gridDim.x - 1) {
                                atomicExch(&a.hdr->next_unit, 0);
                                atomicExch(&a.hdr->done_ctas, 0);
                            }
                        }
                        sh.unit_id[n & 3] = u;
                        mbar_arrive(&sh.unit_full[n & 3]);
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                u = __shfl_sync(0xffffffffu, u, 0);
                if (!ok) break;
                Unit6 U;
                if (!unit6(a, total, u, U)) break;
                // K, and V into the dO ring, once the previous unit's products are done.
                if (lane == 0) ok = mbar_wait(&sh.kv_empty, (uc & 1) ^ 1, wc, k6SiteKvEmpty);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&sh.kv_full, 4 * kKBox6);
                    mbar_arrive_expect_tx(&sh.v_full, 4 * kKBox6);
                    for (int c = 0; c < 4; ++c) {
                        tma_load_3d(sK + c * kKBox6, &tk, &sh.kv_full, c * 64, U.hk, U.tok0 + U.k * kTileN);
                        tma_load_3d(sDO + c * kKBox6, &tv, &sh.v_full, c * 64, U.hk, U.tok0 + U.k * kTileN);
                    }
                }
                ++n_kv;
                const int span = U.nq - U.i0;
                // LSE and D of a step, loaded one step ahead into registers.
                float nl[2], nd[2];
                auto load_stats = [&](int t) {
                    const int h = U.hk * g + t / span, i = U.i0 + t % span;
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int q = i * kStep + 2 * lane + e;
                        nl[e] = 0.f;
                        nd[e] = 0.f;
                        if (q < U.len) {
                            const size_t li = a.varlen ? (size_t)h * a.T + U.tok0 + q
                                                       : ((size_t)U.seq * a.Hq + h) * a.N + q;
                            nl[e] = a.lse[li] * 1.4426950408889634f;
                            nd[e] = a.D[(size_t)h * a.T + U.tok0 + q];
                        }
                    }
                };
                load_stats(0);
                for (int t = 0; t < U.n; ++t, ++jj) {
                    const int h = U.hk * g + t / span, i = U.i0 + t % span, row = U.tok0 + i * kStep;
                    const uint32_t s = jj & 1, ep = ((jj >> 1) & 1) ^ 1;
                    const uint32_t sq = sQ + s * kStage6, sdo = sDO + s * kStage6;
                    // dO before Q: its slot frees first (dV reads dO, dK reads Q
                    // last) -- except on the unit's first step, where dO waits
                    // for V to leave the ring.
                    if (t > 0 && lane == 0) {
                        ok = mbar_wait(&sh.do_empty[s], ep, wc, k6SiteDoEmpty);
                        if (ok) {
                            mbar_arrive_expect_tx(&sh.do_full[s], kStage6);
                            for (int c = 0; c < 4; ++c) tma_load_3d(sdo + c * kQBox6, &tdo, &sh.do_full[s], c * 64, h, row);
                            if (s) ++n_do1; else ++n_do0;
                        }
                    }
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (!ok) break;
                    if (lane == 0) {
                        ok = mbar_wait(&sh.q_empty[s], ep, wc, k6SiteQEmpty);
                        if (ok) {
                            mbar_expect_tx(&sh.q_full[s], kStage6);
                            for (int c = 0; c < 4; ++c) tma_load_3d(sq + c * kQBox6, &tq, &sh.q_full[s], c * 64, h, row);
                        }
                    }
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (!ok) break;
                    if (s) ++n_q1; else ++n_q0;
                    // q_full's one arrival follows the LSE / D stores.
                    float* st = s_stat + s * 2 * kStep;
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        st[2 * lane + e] = nl[e];
                        st[kStep + 2 * lane + e] = nd[e];
                    }
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&sh.q_full[s]);
                        if (t == 0) {
                            ok = mbar_wait(&sh.v_ready, uc & 1, wc, k6SiteVReady);
                            if (ok) ok = mbar_wait(&sh.do_empty[s], ep, wc, k6SiteDoEmpty);
                            if (ok) {
                                mbar_arrive_expect_tx(&sh.do_full[s], kStage6);
                                for (int c = 0; c < 4; ++c)
                                    tma_load_3d(sdo + c * kQBox6, &tdo, &sh.do_full[s], c * 64, h, row);
                                if (s) ++n_do1; else ++n_do0;
                            }
                        }
                    }
                    if (t + 1 < U.n) load_stats(t + 1);
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (!ok) break;
                }
                ++uc;
            }
            if (lane == 0) {  // every copy this thread issued has landed before teardown
                if (n_q0) drain6(&sh.q_full[0], (n_q0 - 1) & 1);
                if (n_q1) drain6(&sh.q_full[1], (n_q1 - 1) & 1);
                if (n_do0) drain6(&sh.do_full[0], (n_do0 - 1) & 1);
                if (n_do1) drain6(&sh.do_full[1], (n_do1 - 1) & 1);
                if (n_kv) {
                    drain6(&sh.kv_full, (n_kv - 1) & 1);
                    drain6(&sh.v_full, (n_kv - 1) & 1);
                }
            }
            __syncwarp();
        } else if (warp == 9) {
            // ----------------------------------- S^T, dP^T, dV, dQ^T, dK issuer
            uint32_t jj = 0, uc = 0;
            bool ok = true;
            for (uint32_t n = 0; ok; ++n) {
                if (!(ok = mbar_wait_w(&sh.unit_full[n & 3], (n >> 2) & 1, wc, k6SiteUnit))) break;
                const int u = *(volatile int*)&sh.unit_id[n & 3];
                __syncwarp();
                if (lane == 0) mbar_arrive(&sh.unit_empty[n & 3]);
                Unit6 U;
                if (!unit6(a, total, u, U)) break;
                if (!(ok = mbar_wait_w(&sh.kv_full, uc & 1, wc, k6SiteKvFull))) break;
                if (!(ok = mbar_wait_w(&sh.v_ready, uc & 1, wc, k6SiteVReady))) break;
                const uint32_t oK = U.pass * 2 * kKBox6, oQ = U.pass * 2 * kQBox6;   // the pass's half
                // S^T of the unit's first step.  Every S^T overwrites the
                // columns the previous step's dV reads P^T from; this thread
                // issued that dV earlier, and the tensor core runs one
                // thread's products in issue order.
                if (!(ok = mbar_wait_w(&sh.q_full[jj & 1], (jj >> 1) & 1, wc, k6SiteQFull))) break;
                tc_fence_after();
                mma6_s(tmem + kColS6, sK, sQ + (jj & 1) * kStage6);
                umma_commit_w(&sh.s_full);
                for (int t = 0; t < U.n; ++t, ++jj) {
                    const uint32_t s = jj & 1, sq = sQ + s * kStage6, sdo = sDO + s * kStage6;
                    if (!(ok = mbar_wait_w(&sh.do_full[s], (jj >> 1) & 1, wc, k6SiteDoFull))) break;
                    // dQ^T of the previous step (in the dP^T columns) has been drained.
                    if (jj > 0 && !(ok = mbar_wait_w(&sh.dq_free, (jj - 1) & 1, wc, k6SiteDqFree))) break;
                    tc_fence_after();
                    mma6_dp(tmem + kColDP6, tmem + kColV6, sdo);
                    umma_commit_w(&sh.dp_full);
                    if (!(ok = mbar_wait_w(&sh.p_ready, jj & 1, wc, k6SiteP))) break;
                    // The previous unit's epilogue has read dK_h, dV_h out.
                    if (t == 0 && !(ok = mbar_wait_w(&sh.acc_free, (uc & 1) ^ 1, wc, k6SiteAcc))) break;
                    tc_fence_after();
                    mma6_dv(tmem + kColDV6, tmem + kColS6, sdo + oQ, t > 0);
                    umma_commit_w(&sh.do_empty[s]);  // dO read by dP^T and dV
                    if (t + 1 < U.n) {               // the next step's S^T, right behind dV (see above)
                        const uint32_t s1 = (jj + 1) & 1;
                        if (!(ok = mbar_wait_w(&sh.q_full[s1], ((jj + 1) >> 1) & 1, wc, k6SiteQFull))) break;
                        tc_fence_after();
                        mma6_s(tmem + kColS6, sK, sQ + s1 * kStage6);
                        umma_commit_w(&sh.s_full);
                    }
                    if (!(ok = mbar_wait_w(&sh.ds_ready, jj & 1, wc, k6SiteDs))) break;
                    tc_fence_after();
                    // dK before dQ^T: Q's slot is released, and the copy of
                    // the step after next queued, ahead of dQ's reductions
                    // (they share the copy engine).
                    mma6_dk(tmem + kColDK6, sDS, sq + oQ, t > 0);
                    umma_commit_w(&sh.q_empty[s]);   // Q (and the step's LSE / D) consumed
                    mma6_dqt(tmem + kColDP6, sK + oK, sDS);   // every key row has read dP^T
                    umma_commit_w(&sh.dq_full);
                    umma_commit_w(&sh.ds_free);      // dS^T read by dQ^T and dK
                }
                if (!ok) break;
                umma_commit_w(&sh.dkdv_done);
                umma_commit_w(&sh.kv_empty);
                ++uc;
            }
            umma_commit_w(&sh.drain);
            drain6(&sh.drain, 0);
            __syncwarp();
        }
    } else if (warp < 4 || warp >= 12) {
        regs_inc<144>();
        // ------------------------------------ V into tensor memory, P^T, dS^T (key rows)
        const int hc = warp >= 12 ? 1 : 0;                   // which 32 of the step's 64 queries (V: head-dim half)
        const int cb = hc * 32;
        const int r = (warp & 3) * 32 + lane;                // key row in the tile == TMEM lane
        const uint32_t lb = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + lb + kColS6 + cb, tDP = tmem + lb + kColDP6 + cb;
        uint8_t* ds_row = dsm + kOffDS6 + r * 128;
        const int sw = r & 7;
        uint32_t jj = 0, uc = 0;
        bool ok = true;
        for (uint32_t n = 0; ok; ++n) {
            if (!(ok = mbar_wait(&sh.unit_full[n & 3], (n >> 2) & 1, wc, k6SiteUnit))) break;
            const int u = *(volatile int*)&sh.unit_id[n & 3];
            mbar_arrive(&sh.unit_empty[n & 3]);
            Unit6 U;
            if (!unit6(a, total, u, U)) break;
            // V of the unit, staged by TMA in the dO ring (four 64-column
            // boxes, 128-B swizzled rows), into tensor memory: this thread's
            // key row, head-dim half hc.  Chunk q of box c (columns 64c+8q ..
            // +7) sits at position q ^ (row % 8) and becomes columns
            // 32c+4q .. +3 of the A operand (bf16 pairs).  The loader issued
            // these copies after every product of the previous unit had
            // completed, so V's old columns are no longer read.
            if (!(ok = mbar_wait(&sh.v_full, uc & 1, wc, k6SiteVFull))) break;
            tc_fence_after();
#pragma unroll 1   // one box at a time: 32 registers
            for (int b = 0; b < 2; ++b) {
                const int c = 2 * hc + b;
                const uint8_t* src = dsm + kOffDO6 + c * kKBox6 + r * 128;
                uint32_t w[32];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const uint4 x = *reinterpret_cast<const uint4*>(src + ((q ^ sw) << 4));
                    w[4 * q] = x.x;
                    w[4 * q + 1] = x.y;
                    w[4 * q + 2] = x.z;
                    w[4 * q + 3] = x.w;
                }
                tmem_st32(tmem + lb + kColV6 + 32 * c, w);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&sh.v_ready);
            ++uc;
            const int key = U.k * kTileN + r;
            const int span = U.nq - U.i0;
            for (int t = 0; t < U.n; ++t, ++jj) {
                const int i = U.i0 + t % span;
                const float* s_lse = s_stat + (jj & 1) * 2 * kStep;
                const float* s_D = s_lse + kStep;
                if (!(ok = mbar_wait(&sh.q_full[jj & 1], (jj >> 1) & 1, wc, k6SiteQFull))) break;   // LSE / D stored
                if (!(ok = mbar_wait(&sh.s_full, jj & 1, wc, k6SiteS))) break;
                tc_fence_after();
                float p[32];
                tmem_ld32(tS, *reinterpret_cast<uint32_t(*)[32]>(p));
                tmem_wait_ld();
                // visible columns c: query 64 i + cb + c < len, key < len, key <= query if causal
                const int c_lo = (a.causal ? key - i * kStep : 0) - cb;
                const int c_hi = (key >= U.len ? 0 : U.len - i * kStep) - cb;
                const float4* l4v = reinterpret_cast<const float4*>(s_lse + cb);
                if (c_lo <= 0 && c_hi >= 32) {
#pragma unroll
                    for (int c4 = 0; c4 < 8; ++c4) {
                        const float4 l4 = l4v[c4];
                        p[4 * c4] = ex2_mufu(fmaf(p[4 * c4], scale, -l4.x));
                        p[4 * c4 + 1] = ex2_mufu(fmaf(p[4 * c4 + 1], scale, -l4.y));
                        p[4 * c4 + 2] = ex2_mufu(fmaf(p[4 * c4 + 2], scale, -l4.z));
                        p[4 * c4 + 3] = ex2_mufu(fmaf(p[4 * c4 + 3], scale, -l4.w));
                    }
                } else {
#pragma unroll
                    for (int c4 = 0; c4 < 8; ++c4) {
                        const float4 l4 = l4v[c4];
                        const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int c = 4 * c4 + e;
                            const float pe = ex2_mufu(fmaf(p[c], scale, -lv[e]));
                            p[c] = (c >= c_lo && c < c_hi) ? pe : 0.f;
                        }
                    }
                }
                {
                    uint32_t pk[16];
#pragma unroll
                    for (int m = 0; m < 16; ++m) pk[m] = pack_bf16x2(p[2 * m], p[2 * m + 1]);
                    tmem_st16(tS, pk);   // P^T: two bf16 per column, over this half's first 16 columns
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&sh.p_ready);

                // dS^T from this half's dP^T columns, into shared memory.
                if (!(ok = mbar_wait(&sh.dp_full, jj & 1, wc, k6SiteDp))) break;
                if (!(ok = mbar_wait(&sh.ds_free, (jj & 1) ^ 1, wc, k6SiteDsFree))) break;
                tc_fence_after();
                uint32_t dp[32];
                tmem_ld32(tDP, dp);
                tmem_wait_ld();
                const float4* d4v = reinterpret_cast<const float4*>(s_D + cb);
                uint32_t pk[16];
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    const float4 d4 = d4v[m];
                    const int c = 4 * m;
                    pk[2 * m] = pack_bf16x2(p[c] * (__uint_as_float(dp[c]) - d4.x),
                                            p[c + 1] * (__uint_as_float(dp[c + 1]) - d4.y));
                    pk[2 * m + 1] = pack_bf16x2(p[c + 2] * (__uint_as_float(dp[c + 2]) - d4.z),
                                                p[c + 3] * (__uint_as_float(dp[c + 3]) - d4.w));
                }
                // 32 queries = four 16-byte chunks; chunk q of the row holds
                // queries 8q .. 8q+7 at position q ^ (row % 8) (128-B swizzle).
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int q = hc * 4 + m;
                    *reinterpret_cast<uint4*>(ds_row + ((q ^ sw) << 4)) =
                        make_uint4(pk[4 * m], pk[4 * m + 1], pk[4 * m + 2], pk[4 * m + 3]);
                }
                fence6_async_smem();   // dS^T is read by the dQ^T and dK products
                tc_fence_before();
                mbar_arrive(&sh.ds_ready);
            }
        }
    } else {
        regs_inc<168>();
        // -------------------------------------------- dQ drain, dK/dV epilogue
        const int r = tid - 128;                             // head-dim column (dQ^T) / key row (dK, dV)
        const uint32_t lb = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tDQ = tmem + lb + kColDP6;
        uint32_t jj = 0, uc = 0;
        bool ok = true;
        // Deterministic mode: a step's semaphore is released one step late,
        // once the group reaches the next step's semaphore (or the unit's
        // epilogue) -- by then its bulk reductions have long completed, so
        // waiting for them costs nothing, where waiting at once stalled the
        // drain every step.  Each warp's elected lane waits for its own
        // reductions; one thread then releases.  A release always comes
        // before the group's next wait, so no CTA holds one semaphore while
        // it waits on another.
        int* sem_pend = nullptr;
        auto release_pending6 = [&]() {
            if (sem_pend) {
                if (lane == 0) {
                    bulk6_wait0();          // this warp's additions are complete ...
                    fence6_async_global();  // ... and ordered before the release
                }
                bar6(1, 128);               // ... for every warp of the group
                if (r == 0) red6_release_add(sem_pend, 1);
            }
            sem_pend = nullptr;
        };
        for (uint32_t n = 0; ok; ++n) {
            ok = mbar_wait(&sh.unit_full[n & 3], (n >> 2) & 1, wc, k6SiteUnit);
            if (bar6_or(1, 128, !ok)) { ok = false; break; }
            const int u = *(volatile int*)&sh.unit_id[n & 3];
            mbar_arrive(&sh.unit_empty[n & 3]);
            Unit6 U;
            if (!unit6(a, total, u, U)) break;
            const int span = U.nq - U.i0;
            for (int t = 0; t < U.n; ++t, ++jj) {
                const int h = U.hk * g + t / span, i = U.i0 + t % span;
                ok = mbar_wait(&sh.dq_full, jj & 1, wc, k6SiteDq);
                ok = !bar6_or(1, 128, !ok);
                if (!ok) break;
                tc_fence_after();
                float v[64];
                tmem_ld32(tDQ, *reinterpret_cast<uint32_t(*)[32]>(v));
                tmem_ld32(tDQ + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
                tmem_wait_ld();
                tc_fence_before();
                mbar_arrive(&sh.dq_free);
                int* sem = a.deterministic
                               ? a.sem + ((size_t)U.pass * a.Hq + h) * a.sem_stride + U.seq + (U.tok0 + i * kStep) / kStep
                               : nullptr;
                if (sem) {
                    release_pending6();
                    // Key tiles add into this query step in ascending order.
                    bool gave_up = false;
                    if (r == 0) {
                        const uint64_t t0 = globaltimer_ns();
                        uint32_t spins = 0;
                        while (ld6_acquire(sem) != U.k) {
                            if ((++spins & 255u) == 0 &&
                                (*(volatile int*)&sh.abort_flag || globaltimer_ns() - t0 > kWaitLimitNs)) {
                                if (atomicCAS(&a.hdr->status.code, 0, kStatusTimeout) == 0) {
                                    a.hdr->status.where = k6SiteSem;
                                    a.hdr->status.block = blockIdx.x;
                                }
                                *(volatile int*)&sh.abort_flag = 1;
                                gave_up = true;
                                break;
                            }
                        }
                    }
                    if (bar6_or(1, 128, gave_up)) { ok = false; break; }
                    if (lane == 0) fence6_async_global();   // our bulk reductions follow the acquire
                }
                // This warp's strip (head-dim columns 32 (warp % 4) .. +31 of
                // the half) in two boxes of 32 query rows, staged in the
                // 128-B swizzled layout of the accumulator's tensor map (row e
                // of a box: 16-byte chunk c at position c ^ (e % 8)).  Rows
                // past the sequence hold exact zeros (their dS is zero), so
                // adding them to the neighbouring rows changes nothing.
                const int y0 = h * (int)a.T + U.tok0 + i * kStep, x0 = U.pass * 128 + (warp & 3) * 32;
                uint8_t* box = dsm + kOffStg6 + (warp & 3) * kStgBox6;
                const uint32_t box_s = base + kOffStg6 + (warp & 3) * kStgBox6;
#pragma unroll
                for (int qh = 0; qh < 2; ++qh) {
                    if (lane == 0) bulk6_wait_read0();   // the box's previous reduction has read it
                    __syncwarp();
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        *reinterpret_cast<float*>(box + e * 128 + ((((lane >> 2) ^ (e & 7)) << 4) | ((lane & 3) << 2))) =
                            v[qh * 32 + e];
                    fence6_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma6_reduce_add(&tdq, box_s, x0, y0 + qh * 32);
                        bulk6_commit();
                    }
                }
                if (sem) sem_pend = sem;
                if (kDbg && r == 0 && U.pass == 0) dbg_count(a.dbg_inner, (long long)h * a.T + U.tok0 + i * kStep);
            }
            if (!ok) break;
            release_pending6();   // the next key tile may be waiting for it
            ok = mbar_wait(&sh.dkdv_done, uc & 1, wc, k6SiteDkdv);
            if (bar6_or(1, 128, !ok)) { ok = false; break; }
            ++uc;
            tc_fence_after();
            const int key = U.k * kTileN + r;
            const bool kvalid = key < U.len;
            const size_t orow = ((size_t)(U.tok0 + key) * a.Hkv + U.hk) * kD6 + U.pass * 128;
#pragma unroll
            for (int which = 0; which < 2; ++which) {
                const uint32_t tacc = tmem + lb + (which ? kColDV6 : kColDK6);
                const float mul = which ? 1.f : a.alpha;
                uint4* out = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(which ? a.dv : a.dk) + orow);
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    uint32_t w[32];
                    tmem_ld32(tacc + cc * 32, w);
                    tmem_wait_ld();
                    if (kvalid) {
#pragma unroll
                        for (int m = 0; m < 4; ++m) {
                            const float* f = reinterpret_cast<const float*>(w + 8 * m);
                            out[cc * 4 + m] = make_uint4(pack_bf16x2(f[0] * mul, f[1] * mul), pack_bf16x2(f[2] * mul, f[3] * mul),
                                                         pack_bf16x2(f[4] * mul, f[5] * mul), pack_bf16x2(f[6] * mul, f[7] * mul));
                        }
                    }
                }
            }
            if (kDbg && r == 0 && U.pass == 0) dbg_count(a.dbg_visits, (long long)U.hk * a.T + U.tok0 + U.k * kTileN);
            tc_fence_before();
            mbar_arrive(&sh.acc_free);
        }
        if (lane == 0) bulk6_wait0();   // every bulk reduction this warp issued has completed
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

}  // namespace

cudaError_t launch_bwd256_main(const BwdLaunch& L, cudaStream_t stream) {
    const BwdArgs& a = L.a;
    auto kern = (a.dbg_visits || a.dbg_inner) ? bwd256_kernel<true> : bwd256_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem6);
    if (e != cudaSuccess) return e;
    const long long units = 2 * (a.varlen ? (long long)a.Hkv * ((a.T + kTileN - 1) / kTileN + a.B)
                                          : (long long)a.B * a.Hkv * ((a.N + kTileN - 1) / kTileN));
    int grid = (int)(units < L.num_sms ? units : L.num_sms);
    if (grid < 1) grid = 1;
    kern<<<grid, kThreads6, kSmem6, stream>>>(L.tq, L.tk, L.tv, L.tdo, L.tdq, a);
    return cudaGetLastError();
}

}  // namespace fa
