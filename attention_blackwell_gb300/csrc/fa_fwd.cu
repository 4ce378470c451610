// fa_fwd.cu -- forward attention kernel for sm_103a (tcgen05 / TMEM / TMA).
//
// Computes O = softmax(alpha Q K^T [+ causal]) V and LSE for d = 128 or 64
// (a template parameter D) with an online softmax (FlashAttention-4 blog, "Forward pass: a new softmax pipeline
// with conditional rescaling"; FlashAttention-4 paper summary §3.1.2-§3.1.4).
//
// One persistent CTA per SM walks a list of work units.  A unit is two query
// tiles of 128 rows (tile 0 and tile 1 -- the pages' Q^H and Q^L) of one
// (sequence, head); the CTA ping-pongs between them so the tensor core works
// on one tile while the softmax of the other runs.  Warp roles:
//
//   warps 0-3   softmax warpgroup for tile 0 (one thread per row)
//   warps 4-7   softmax warpgroup for tile 1
//   warp  8     TMA loader: Q tiles once per unit, then a K/V ring
//   warp  9     UMMA issuer (one thread): S = Q K^T and O += P V
//   warps 10-11 idle (complete the third warpgroup)
//
// Tensor memory (512 columns x 128 lanes, fp32 cells), per the paper
// summary's "2 x O + 2 x S, P overlapping S" layout:
//   cols   0-127  O of tile 0      cols 128-255  O of tile 1 (D columns used)
//   cols 256-383  S/P of tile 0    cols 384-511  S/P of tile 1
// P (bf16, two per 32-bit cell) overwrites the first 64 columns of its S.
//
// Per key tile j the softmax thread of row r: loads its 128 S values,
// masks, takes the row max in log2 units (scale alpha*log2 e), decides the
// conditional rescale per warp (any row's max jump > tau), rescales its O
// row and l in TMEM/registers when it must (the tensor core has finished the
// previous P V by then: the commit that signalled S_j covers every earlier
// MMA), forms P = 2^(x - m) with part of the exponentials on the FMA pipe,
// writes P as bf16 into TMEM in four 32-column stages and signals the UMMA
// warp.  After the last tile it normalises O by 1/l and stores O and LSE.
#include "fa_internal.h"
#include "fa_sched.cuh"
#include "fa_exp2.cuh"

namespace fa {
namespace {

constexpr int kStages = 4;                     // K/V ring depth (one tile per slot)
constexpr int kThreads = 384;
constexpr uint32_t kBoxBytes = 16384;          // 128 rows x 64 bf16 (one TMA box)
// Per head dim D: a 128-row tile of Q, K or V is D / 64 boxes.
template <int D> struct Geo {
    static_assert(D == 64 || D == 128, "head dim");
    static constexpr int kBoxes = D / 64;
    static constexpr uint32_t kTileBytes = 128u * D * 2u;
    static constexpr uint32_t kSmemTiles = 2 * kTileBytes + kStages * kTileBytes;
    static constexpr uint32_t kSmemBytes = 1024 + kSmemTiles + kTableInts * 4;
};

// TMEM column bases of O and S/P for tile x.
__device__ __forceinline__ uint32_t col_o(int x) { return (uint32_t)x * 128u; }
__device__ __forceinline__ uint32_t col_s(int x) { return 256u + (uint32_t)x * 128u; }

// Wait-site identifiers reported through the status word.
enum : int { kSiteQEmpty = 1, kSiteRingEmpty, kSiteQFull, kSiteRingFull, kSiteP0, kSiteP1, kSiteS, kSiteO,
             kSiteDrain, kSiteSelftest = 990 };

// Key tiles tile x (0/1) of a unit needs.
__device__ __forceinline__ int kv_tiles(const Unit& U, int x, int causal) {
    const int all = (U.len + kTileN - 1) / kTileN;
    if (!causal) return all;
    const int diag = (U.m * kUnitRows + x * kTileM) / kTileN + 1;
    return diag < all ? diag : all;
}

struct FwdShared {
    uint64_t q_full, q_empty;
    uint64_t full[kStages], empty[kStages];
    uint64_t s_full[2], p_ready[2], o_done[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
    int total, maxm;
    Sched sched;
};

// S = Q K^T for one 128x128 tile: D / 16 UMMAs of K = 16 over the head dim.
// Both operands K-major; k-step k reads 32 bytes at column (k % 4) * 16 of box k / 4.
template <int D>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint32_t q_smem, uint32_t k_smem) {
    constexpr uint32_t idesc = idesc_bf16_f32(128, 128, 0, 0);
    const uint64_t qd = sdesc_sw128(q_smem, 16, 1024), kd = sdesc_sw128(k_smem, 16, 1024);
    static_for<D / 16>([&](auto kc) {
        constexpr uint32_t k = kc, off = ((k >> 2) * kBoxBytes + (k & 3) * 32) >> 4;  // 16-byte units
        umma_ss_k<off, off>(d_tmem, qd, kd, idesc, k > 0);
    });
}

// O (+)= P V: A = P (bf16 in TMEM, 8 columns per k-step of 16 keys),
// B = V MN-major (k-step k = 16 key rows = 2048 bytes further; N = D, the
// 64-column boxes kBoxBytes apart).
template <int D>
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint32_t v_smem, uint32_t acc) {
    constexpr uint32_t idesc = idesc_bf16_f32(128, D, 0, 1);
    const uint64_t vd = sdesc_sw128(v_smem, kBoxBytes, 1024);
    static_for<8>([&](auto kc) {
        constexpr uint32_t k = kc;
        umma_ts_k<k * 8, ((k * 2048) >> 4)>(d_tmem, p_tmem, vd, idesc, (acc | k) != 0);
    });
}

template <int kEmu16, int D>
__global__ void __launch_bounds__(kThreads, 1)
fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
           const __grid_constant__ CUtensorMap tv, const FwdArgs a) {
    extern __shared__ uint8_t dsmem[];
    __shared__ FwdShared sh;

    using G = Geo<D>;
    constexpr uint32_t kTileBytes = G::kTileBytes;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t base = (smem_u32(dsmem) + 1023u) & ~1023u;
    uint8_t* gbase = dsmem + (base - smem_u32(dsmem));
    const uint32_t sQ = base;                        // 2 tiles
    const uint32_t sRing = base + 2 * kTileBytes;    // kStages tiles
    int* s_cu = reinterpret_cast<int*>(gbase + G::kSmemTiles);
    int* s_order = s_cu + (kMaxVarlenSeqs + 1);
    int* s_pref = s_order + kMaxVarlenSeqs;

    if (tid == 0) {
        mbar_init(&sh.q_full, 1);
        mbar_init(&sh.q_empty, 1);
        for (int i = 0; i < kStages; ++i) { mbar_init(&sh.full[i], 1); mbar_init(&sh.empty[i], 1); }
        for (int x = 0; x < 2; ++x) {
            mbar_init(&sh.s_full[x], 1);
            mbar_init(&sh.p_ready[x], 128);
            mbar_init(&sh.o_done[x], 1);
        }
        mbar_init(&sh.drain, 1);
        sh.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 8 && lane == 0) {
        tma_prefetch_desc(&tq);
        tma_prefetch_desc(&tk);
        tma_prefetch_desc(&tv);
    }
    if (warp == 0) {
        tmem_alloc(&sh.tmem_base, 512);
        tmem_relinquish();
    }

    build_sched_tables(a, s_cu, s_order, s_pref, &sh.maxm, &sh.total, tid, kThreads);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    if (tid == 0) {
        sh.sched.B = a.B; sh.sched.Hq = a.Hq; sh.sched.N = a.N; sh.sched.causal = a.causal;
        sh.sched.varlen = a.varlen; sh.sched.num_m = sh.maxm; sh.sched.maxm = sh.maxm;
        sh.sched.sec = a.l2_section; sh.sched.total = sh.total;
        sh.sched.zz = a.causal && !a.varlen && !a.naive && sh.maxm % 2 == 0;
        sh.sched.naive = a.naive;
        sh.sched.s_cu = s_cu; sh.sched.s_order = s_order; sh.sched.s_pref = s_pref;
    }
    __syncthreads();
    // Read through shared memory on every call: keeps the decode state out of
    // the registers of the lean loader/UMMA warps.
    const Sched& sched = sh.sched;

    const WaitCtx wc{&sh.abort_flag, a.status};
    const uint32_t tmem = sh.tmem_base;
    const int group = a.Hq / a.Hkv;

    // Register split (launch: 384 x 168): the two softmax warpgroups hold a
    // 128-float S row per thread and get 224; the loader/UMMA warpgroup 40.
    // 2*128*224 + 128*40 = 62464 <= 64512.
    if (warp >= 8) {
      regs_dec<40>();
      if (warp == 8) {
        // ------------------------------------------------------------ loader
        if (lane == 0) {
            uint32_t it = 0, uc = 0;
            bool ok = true;
            for (int un = 0; ok; ++un) {
                const int u = sched.nth((int)blockIdx.x, (int)gridDim.x, un);
                Unit U;
                if (!sched.get(u, U)) break;
                const int hk = U.h / group;
                if (!(ok = mbar_wait(&sh.q_empty, (uc & 1) ^ 1, wc, kSiteQEmpty))) break;
                mbar_arrive_expect_tx(&sh.q_full, 2 * kTileBytes);
                for (int x = 0; x < 2; ++x)
                    for (int c = 0; c < G::kBoxes; ++c)
                        tma_load_3d(sQ + x * kTileBytes + c * kBoxBytes, &tq, &sh.q_full, c * 64, U.h,
                                    U.tok0 + U.m * kUnitRows + x * kTileM);
                const int n = kv_tiles(U, 1, a.causal);
                for (int j = 0; j < n && ok; ++j) {
                    for (int kv = 0; kv < 2; ++kv) {
                        const uint32_t slot = it % kStages;
                        if (!(ok = mbar_wait(&sh.empty[slot], ((it / kStages) & 1) ^ 1, wc, kSiteRingEmpty))) break;
                        mbar_arrive_expect_tx(&sh.full[slot], kTileBytes);
                        const CUtensorMap* map = kv ? &tv : &tk;
                        for (int c = 0; c < G::kBoxes; ++c)
                            tma_load_3d(sRing + slot * kTileBytes + c * kBoxBytes, map, &sh.full[slot], c * 64,
                                        hk, U.tok0 + j * kTileN);
                        ++it;
                    }
                }
                ++uc;
            }
            // Drain: every copy this thread issued has landed before teardown.
            const uint32_t first = it > kStages ? it - kStages : 0;
            for (uint32_t i = first; i < it; ++i) {
                uint32_t bar = smem_u32(&sh.full[i % kStages]);
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(bar, (i / kStages) & 1) && globaltimer_ns() - t0 < kWaitLimitNs) {}
            }
            if (uc > 0) {
                uint32_t bar = smem_u32(&sh.q_full);
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(bar, (uc - 1) & 1) && globaltimer_ns() - t0 < kWaitLimitNs) {}
            }
        }
        __syncwarp();
      } else if (warp == 9) {
        // ------------------------------------------------------- UMMA issuer
        {   // the whole warp runs the issue loop (see umma_ss_w)
            uint32_t it = 0, uc = 0, pc[2] = {0, 0};
            bool ok = true;
            for (int un = 0; ok; ++un) {
                const int u = sched.nth((int)blockIdx.x, (int)gridDim.x, un);
                Unit U;
                if (!sched.get(u, U)) break;
                const int n0 = kv_tiles(U, 0, a.causal), n1 = kv_tiles(U, 1, a.causal);
                // Shared-memory operands land through TMA and are read by the
                // tensor core (both async proxy): the mbarrier completion is
                // the only ordering needed.  A tcgen05 fence is needed only
                // after waits that hand over TENSOR memory (P from softmax).
                if (!(ok = mbar_wait_w(&sh.q_full, uc & 1, wc, kSiteQFull))) break;
                uint32_t slot_k = it % kStages;
                if (!(ok = mbar_wait_w(&sh.full[slot_k], (it / kStages) & 1, wc, kSiteRingFull))) break;
                ++it;
                tc_fence_after();  // S of the previous unit's epilogue (O) is in order
                issue_qk<D>(tmem + col_s(0), sQ, sRing + slot_k * kTileBytes);
                umma_commit_w(&sh.s_full[0]);
                issue_qk<D>(tmem + col_s(1), sQ + kTileBytes, sRing + slot_k * kTileBytes);
                umma_commit_w(&sh.s_full[1]);
                umma_commit_w(&sh.empty[slot_k]);
                for (int j = 0; j < n1; ++j) {
                    const uint32_t slot_v = it % kStages;
                    if (!(ok = mbar_wait_w(&sh.full[slot_v], (it / kStages) & 1, wc, kSiteRingFull))) break;
                    ++it;
                    const bool more = j + 1 < n1;
                    if (more) {  // K of the next tile: waited here so PV and S issue back to back
                        slot_k = it % kStages;
                        if (!(ok = mbar_wait_w(&sh.full[slot_k], (it / kStages) & 1, wc, kSiteRingFull))) break;
                        ++it;
                    }
                    if (j < n0) {
                        if (!(ok = mbar_wait_w(&sh.p_ready[0], pc[0] & 1, wc, kSiteP0))) break;
                        ++pc[0];
                        tc_fence_after();
                        issue_pv<D>(tmem + col_o(0), tmem + col_s(0), sRing + slot_v * kTileBytes, j > 0);
                        if (j == n0 - 1) umma_commit_w(&sh.o_done[0]);
                        if (more && j + 1 < n0) {
                            issue_qk<D>(tmem + col_s(0), sQ, sRing + slot_k * kTileBytes);
                            umma_commit_w(&sh.s_full[0]);
                        }
                    }
                    if (!(ok = mbar_wait_w(&sh.p_ready[1], pc[1] & 1, wc, kSiteP1))) break;
                    ++pc[1];
                    tc_fence_after();
                    issue_pv<D>(tmem + col_o(1), tmem + col_s(1), sRing + slot_v * kTileBytes, j > 0);
                    umma_commit_w(&sh.empty[slot_v]);
                    if (j == n1 - 1) umma_commit_w(&sh.o_done[1]);
                    if (more) {
                        issue_qk<D>(tmem + col_s(1), sQ + kTileBytes, sRing + slot_k * kTileBytes);
                        umma_commit_w(&sh.s_full[1]);
                        umma_commit_w(&sh.empty[slot_k]);
                    }
                }
                umma_commit_w(&sh.q_empty);
                ++uc;
            }
            // Drain: all issued MMAs complete before tensor memory is freed.
            umma_commit_w(&sh.drain);
            const uint32_t bar = smem_u32(&sh.drain);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(bar, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {}
        }
        __syncwarp();
      }
    } else {
        regs_inc<224>();
        // ------------------------------------------------------------ softmax
        const int x = warp >> 2;                 // which Q tile
        const int r = (warp & 3) * 32 + lane;    // row within the tile == TMEM lane
        const uint32_t lane_bits = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + lane_bits + col_s(x);
        const uint32_t tO = tmem + lane_bits + col_o(x);
        const float scale = a.scale_log2;
        uint32_t sc = 0, uc = 0;
        bool ok = true;
        for (int un = 0; ok; ++un) {
            const int u = sched.nth((int)blockIdx.x, (int)gridDim.x, un);
            Unit U;
            if (!sched.get(u, U)) break;
            const int n = kv_tiles(U, x, a.causal);
            const int qi = U.m * kUnitRows + x * kTileM + r;       // row within the sequence
            const int q_first = U.m * kUnitRows + x * kTileM;     // first row of the tile
            float m_ref = -INFINITY, l = 0.f;
            for (int j = 0; j < n; ++j) {
                if (!(ok = mbar_wait(&sh.s_full[x], sc & 1, wc, kSiteS))) break;
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
                const int k0 = j * kTileN;
                const bool need_mask = (k0 + kTileN > U.len) || (a.causal && k0 + kTileN - 1 > q_first);
                if (need_mask) {
                    const int lim_len = U.len - k0;                          // keys c < lim_len valid
                    const int lim_causal = a.causal ? qi - k0 + 1 : kTileN;  // keys c < lim_causal valid
                    const int lim = lim_len < lim_causal ? lim_len : lim_causal;
#pragma unroll
                    for (int c = 0; c < 128; ++c)
                        if (c >= lim) s[c] = -INFINITY;
                }
                // Row max: three-input max, four chains; then the exponents two
                // at a time (packed fp32 FMA) and the row sum in two packed
                // accumulators, so that no long chain of dependent adds sits
                // between the exponentials (d = 64 forward 893 -> 957 TFLOP/s).
                float mx0 = fmaxf(s[0], s[1]), mx1 = fmaxf(s[2], s[3]), mx2 = fmaxf(s[4], s[5]),
                      mx3 = fmaxf(s[6], s[7]);
#pragma unroll
                for (int c = 8; c < 128; c += 8) {
                    mx0 = fmax3(mx0, s[c], s[c + 1]);
                    mx1 = fmax3(mx1, s[c + 2], s[c + 3]);
                    mx2 = fmax3(mx2, s[c + 4], s[c + 5]);
                    mx3 = fmax3(mx3, s[c + 6], s[c + 7]);
                }
                const float m_blk = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * scale;
                const float m_new = fmaxf(m_ref, m_blk);
                // Conditional rescale (paper summary §3.1.4, blog rescale
                // equation): move to the new max only if some row of this warp
                // jumped by more than tau; the first tile always initialises.
                const bool jump = (m_ref == -INFINITY) ? (m_new != -INFINITY) : (m_new - m_ref > a.tau);
                const bool rescale = __any_sync(0xffffffffu, jump);
                if (lane == 0) dbg_count_rescale(a.dbg_rescale, j > 0, rescale);
                if (rescale) {
                    const float fac = (m_ref == -INFINITY) ? 0.f : ex2_mufu(m_ref - m_new);
                    l *= fac;
                    if (j > 0) {
#pragma unroll
                        for (int c0 = 0; c0 < D; c0 += 32) {
                            uint32_t o[32];
                            tmem_ld32(tO + c0, o);
                            tmem_wait_ld();
#pragma unroll
                            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * fac);
                            tmem_st32(tO + c0, o);
                        }
                    }
                    m_ref = m_new;
                }
                const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
                const uint64_t sc2 = f2_pack(scale, scale), nm2 = f2_pack(-m_use, -m_use);
                uint64_t la = f2_pack(0.f, 0.f), lb = la;
#pragma unroll
                for (int st = 0; st < 4; ++st) {
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int c = st * 32 + 2 * i;
                        float x0, x1;
                        f2_unpack(f2_fma(f2_pack(s[c], s[c + 1]), sc2, nm2), x0, x1);
                        float p0, p1;
                        if (i < kEmu16) { p0 = exp2_fma(x0); p1 = exp2_fma(x1); }   // kEmu16 of 16 pairs
                        else { p0 = ex2_mufu(x0); p1 = ex2_mufu(x1); }
                        if (i & 1) lb = f2_add(lb, f2_pack(p0, p1));
                        else la = f2_add(la, f2_pack(p0, p1));
                        pk[i] = pack_bf16x2(p0, p1);
                    }
                    tmem_st16(tS + st * 16, pk);
                }
                {
                    float a0, a1, b0, b1;
                    f2_unpack(la, a0, a1);
                    f2_unpack(lb, b0, b1);
                    l += (a0 + a1) + (b0 + b1);
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&sh.p_ready[x]);
            }
            if (!ok) break;
            if (!(ok = mbar_wait(&sh.o_done[x], uc & 1, wc, kSiteO))) break;
            ++uc;
            tc_fence_after();
            // Epilogue: O / l -> bf16, LSE = (m + log2 l) ln 2.
            const bool valid = qi < U.len;
            const float inv_l = l > 0.f ? 1.f / l : 0.f;
            uint4* orow = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.o) +
                                                   ((size_t)(U.tok0 + qi) * a.Hq + U.h) * D);
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t o[32];
                tmem_ld32(tO + c0, o);
                tmem_wait_ld();
                if (valid) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint4 v;
                        v.x = pack_bf16x2(__uint_as_float(o[8 * q + 0]) * inv_l, __uint_as_float(o[8 * q + 1]) * inv_l);
                        v.y = pack_bf16x2(__uint_as_float(o[8 * q + 2]) * inv_l, __uint_as_float(o[8 * q + 3]) * inv_l);
                        v.z = pack_bf16x2(__uint_as_float(o[8 * q + 4]) * inv_l, __uint_as_float(o[8 * q + 5]) * inv_l);
                        v.w = pack_bf16x2(__uint_as_float(o[8 * q + 6]) * inv_l, __uint_as_float(o[8 * q + 7]) * inv_l);
                        orow[c0 / 8 + q] = v;
                    }
                }
            }
            if (valid) {
                const float lse = l > 0.f ? (m_ref + __log2f(l)) * 0.69314718055994531f : -INFINITY;
                const size_t li = a.varlen ? (size_t)U.h * a.N + U.tok0 + qi
                                           : ((size_t)U.seq * a.Hq + U.h) * a.N + qi;
                a.lse[li] = lse;
            }
            if (r == 0 && q_first < U.len)
                dbg_count(a.dbg_visits, (long long)U.h * (a.varlen ? a.N : (long long)a.B * a.N) + U.tok0 + q_first);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

// One warp waits, through the bounded wait of every pipeline here, on an
// mbarrier that no thread arrives at: the wait gives up after kWaitLimitNs,
// records the timeout in the status word and returns false.
__global__ void selftest_timeout_kernel(DevStatus* status) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const WaitCtx wc{&abort_flag, status};
    const bool ok = mbar_wait_w(&bar, 0, wc, kSiteSelftest);
    if (ok && threadIdx.x == 0) atomicCAS(&status->code, 0, -1);   // the phase cannot complete
}

// Both forms the forward kernels use: the scalar one (ping-pong kernel) and
// the packed pair (CTA-pair kernel).  They must agree bit for bit; an element
// where they do not is returned as NaN, so a test of y checks both.
__global__ void exp2_emu_kernel(const float* __restrict__ x, float* __restrict__ y, int64_t n) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        // The second lane gets the neighbouring element, so both lanes of
        // the packed form are checked.
        const int64_t nb = (i ^ 1) < n ? (i ^ 1) : i;
        const float xi = x[i], xn = x[nb];
        const float ys = exp2_fma(xi), yn = exp2_fma(xn);
        float yp, yq;
        exp2_fma_x2(xi, xn, yp, yq);
        const bool same = __float_as_uint(ys) == __float_as_uint(yp) && __float_as_uint(yn) == __float_as_uint(yq);
        y[i] = same ? ys : __int_as_float(0x7fc00000);
    }
}

template <int E, int D>
cudaError_t launch_fwd_t(const FwdLaunch& L, cudaStream_t stream, int grid) {
    auto kern = fwd_kernel<E, D>;
    constexpr uint32_t smem = Geo<D>::kSmemBytes;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, smem, stream>>>(L.tq, L.tk, L.tv, L.a);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_fwd_d(const FwdLaunch& L, cudaStream_t stream, int grid) {
    switch (L.emu16) {
        case 0: return launch_fwd_t<0, D>(L, stream, grid);
        case 1: return launch_fwd_t<1, D>(L, stream, grid);
        case 2: return launch_fwd_t<2, D>(L, stream, grid);
        case 3: return launch_fwd_t<3, D>(L, stream, grid);
        case 4: return launch_fwd_t<4, D>(L, stream, grid);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_fwd(const FwdLaunch& L, cudaStream_t stream) {
    // Upper bound on the unit count; the kernel computes the exact one.
    long long units;
    if (L.a.varlen)
        units = ((long long)L.a.N / kUnitRows + L.a.B) * L.a.Hq;
    else
        units = (long long)L.a.B * L.a.Hq * ((L.a.N + kUnitRows - 1) / kUnitRows);
    int grid = (int)(units < L.num_sms ? units : L.num_sms);
    if (grid < 1) grid = 1;
    if (L.d == 64) return launch_fwd_d<64>(L, stream, grid);
    if (L.d == 128) return launch_fwd_d<128>(L, stream, grid);
    return cudaErrorInvalidValue;
}

cudaError_t launch_selftest_timeout(DevStatus* status, cudaStream_t stream) {
    selftest_timeout_kernel<<<1, 32, 0, stream>>>(status);
    return cudaGetLastError();
}

cudaError_t launch_exp2_emu(const float* x, float* y, int64_t n, cudaStream_t stream) {
    if (n <= 0) return cudaSuccess;
    long long blocks = (n + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    exp2_emu_kernel<<<(int)blocks, 256, 0, stream>>>(x, y, n);
    return cudaGetLastError();
}

}  // namespace fa
