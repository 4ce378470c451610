// fa_bwd_pair.cu -- backward main kernel on CTA pairs (sm_103a, cluster of 2).
//
// The same gradients as fa_bwd.cu's main kernel (FlashAttention-4 blog,
// "Backward pass"), with the products of two SMs fused into tcgen05
// .cta_group::2 instructions ("2-CTA backward"): a pair owns one 256-key
// block of one (sequence, key/value head), CTA r the keys r*128 .. +127, and
// streams the query tiles (128 rows) of every query head of the group:
//
//   S^T  = K Q_i^T     M = 256 keys, N = 128 queries, K = d   (A: own K; B: Q_i,
//                      each CTA 64 of the queries)
//   dP^T = V dO_i^T    same shape (A: own V; B: dO_i, 64 queries per CTA)
//   dV  += P^T dO_i    M = 256 keys, N = d, K = 128 queries   (A: P^T in TMEM;
//                      B: dO_i, 64 head-dim columns per CTA)
//   dK  += dS^T Q_i    same shape (A: dS^T in TMEM; B: Q_i, 64 columns per CTA)
//   dQ_i = dS K        M = 128 queries (64 per CTA), N = d, K = 256 keys
//
// Each CTA therefore stages half of every B operand, and the dQ product,
// whose reduction axis (the keys) is split between the CTAs, becomes a pair
// product after an exchange of half of dS through distributed shared memory:
// CTA r ends up holding dS for queries r*64 .. +63 over all 256 keys, and adds
// a 64 x 128 slice of dQ_i into the fp32 accumulator -- half of what one CTA
// adds per tile in fa_bwd.cu (blog, "2-CTA backward": exchange of half of dS,
// halved atomic reductions).
//
// Fixed-length and packed varlen inputs; dQ accumulated atomically or, in
// deterministic mode, in ascending key-block order at every query tile
// (FlashAttention-4 blog, "Deterministic mode": semaphores).
//
// Roles (512 threads per CTA, both CTAs): warps 0-3 and 12-15 key-row
// warpgroups (P^T, dS^T; one thread per key row, each group half of the 128
// query columns); warps 4-7 dQ drain (one thread per TMEM lane: 64 columns of
// one dQ row) and the dK/dV epilogue; warp 8 loader; warp 11 relays "this
// CTA's dS buffer is complete" to the even CTA.  In the even CTA warp 9
// issues dP, dV, S and dK, and warp 10 issues dQ.  Barriers an issuer waits
// on live in the even CTA: the odd CTA's TMA bytes and warp arrivals count
// there; commits go to both CTAs.
//
// Order (blog, "2-CTA backward": the previous tile's dQ before the current
// dP, in the S columns next to P): the dQ product of tile j waits for the
// exchange of dS(j), which takes about as long as a tile.  So dQ(j) is not
// on the chain dS(j) -> dQ(j) -> dP(j+1): it is issued by a thread of its
// own once the key rows have read S^T(j+1) out of R0 (its columns 64-127
// hold dQ(j) from then until the drain has read it), and only S^T(j+2)
// waits for that drain.  dP^T then has R1 to itself, and the dS exchange of
// tile j overlaps the elementwise work of tile j+1.  Warp 9 issues, per tile
// j: dP^T(j), dV(j) (when P^T(j) is ready), S^T(j+1) right behind dV (the
// same thread's products run in order, so S^T(j+1) may overwrite the P^T
// columns dV reads), then dK(j) (when dS^T(j) is ready).
//
// The dS exchange: the key-row half whose queries belong to this CTA writes
// its rows into this CTA's dS buffer; the other half writes them into an
// outbox, and one bulk copy (shared memory to the peer's shared memory,
// completing on the peer's barrier) moves them -- async-proxy traffic end to
// end, so no thread waits for remote stores to drain.
//
// Tensor memory (512 columns, both CTAs): dK 0-127, dV 128-255,
//   R0 256-383: S^T(j), then P^T(j) in columns 0-63 (bf16; half 0 packs its
//               64 queries into columns 0-31, half 1 into 32-63 once half 0
//               has read them) and dQ(j-1) in columns 64-127 once half 1 has
//               read S^T(j) there (an M = 128 pair product leaves each CTA's
//               64 rows in 128 lanes x 64 columns: row m, column n at lane
//               m + 64 (n / 64), column n % 64);
//   R1 384-511: dP^T, then dS^T (bf16: half 0 in columns 0-31, half 1 in
//               96-127, each over dP^T columns it has read).
#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kPBThreads = 512;
constexpr int kKeyBlock = 256;                      // keys per pair
constexpr uint32_t kT16 = 16384, kT32 = 32768;
// Shared memory (232448 bytes, the per-CTA maximum).
constexpr uint32_t kOffK = 0;                       // own 128 keys x 128 d, K-major (2 boxes)
constexpr uint32_t kOffV = kOffK + kT32;            // own V
constexpr uint32_t kOffKdq = kOffV + kT32;          // 256 keys x this CTA's 64 d (2 boxes), MN-major B of dQ
constexpr uint32_t kOffQs = kOffKdq + kT32;         // 64 queries x 128 d (2 boxes of 8 KB), read by S^T only
constexpr uint32_t kOffOut = kOffQs + kT16;         // dS rows of this CTA's keys for the peer's query half
constexpr uint32_t kOffQd = kOffOut + kT16;         // 128 queries x this CTA's 64 d
constexpr uint32_t kOffDOs = kOffQd + kT16;         // dO: 64 queries x 128 d
constexpr uint32_t kOffDOd = kOffDOs + kT16;        // dO: 128 queries x 64 d
constexpr uint32_t kOffDS = kOffDOd + kT16;         // dS for this CTA's 64 queries x 256 keys, MN-major A of dQ
constexpr uint32_t kOffStage = kOffDS + kT32;       // dQ staging: 2 boxes of 64 rows x 32 fp32
constexpr uint32_t kOffStat = kOffStage + kT16;     // lse2[2][128], D[2][128]
constexpr uint32_t kOffBar = kOffStat + 4 * 128 * 4;
constexpr uint32_t kPBSmem = kOffBar + 1024;
static_assert(kPBSmem == 232448, "shared memory plan");

constexpr uint32_t kColDK = 0, kColDV = 128, kColR0 = 256, kColR1 = 384;
constexpr uint16_t kBoth = 3, kLead = 1;

enum : int { kPBSiteKv = 81, kPBSiteQ, kPBSiteDo, kPBSiteS, kPBSiteP, kPBSiteDp, kPBSiteDs, kPBSiteDsFree,
             kPBSiteDq, kPBSiteDqFree, kPBSiteDkdv, kPBSiteAcc, kPBSiteR0, kPBSiteSt, kPBSiteSem };

struct PBShared {
    uint64_t kv_full, kv_empty, qs_full, qs_empty, q_empty[2], qd_full, do_full, do_empty, st_full[2];
    uint64_t s_full, dp_full, p_ready, ds_ready, ds_free, dq_full, dkdv_done, acc_free, drain;
    // Per tile parity: the waiters below skip tiles (a unit's last dQ does not
    // wait for the next S^T), and a parity wait must never be more than one
    // phase behind its barrier.
    uint64_t s_read[2], dq_free[2];
    uint64_t dsx, dsx_ready;
    uint32_t tmem_base;
    int abort_flag;
    int total;   // work units of this call
};
static_assert(sizeof(PBShared) <= 1024, "barrier block");

struct PBUnit {
    int seq, hk, kb, tok0, len, nq, i0, n;
};

// Unit order as in fa_bwd.cu: non-causal atomic head-major (the live Q, dO
// and dQ accumulator of a few heads stay in L2), causal and deterministic
// key-block-major (longest first under the mask: a key block sees query
// tiles 2 kb .. nq-1).  In deterministic mode a unit waits at its
// semaphores only on units of smaller index (the same head's earlier key
// blocks); every pair takes its units in increasing index, so the earliest
// unfinished unit always runs.  The naive order (fa_set_schedule_order) is
// head-major in every mode.  Packed varlen batches: the plan kernel's list
// of (sequence, key/value head, 256-key block), most expensive first (its
// causal order lists each sequence's blocks in ascending order, as the
// semaphores need).

// Units of this call, read once per CTA; a varlen list planned for 128-key
// units or split by query-head group (the one-CTA kernel's) is refused: no
// units, FA_ERR_INVALID.
template <bool kVar>
__device__ __forceinline__ int pb_total(const BwdArgs& a) {
    if constexpr (!kVar) return a.B * a.Hkv * ((a.N + kKeyBlock - 1) / kKeyBlock);
    if (a.hdr->unit_keys != kKeyBlock || a.hdr->unit_heads != 0) {
        if (atomicCAS(&a.hdr->status.code, 0, -1) == 0) a.hdr->status.where = 202;
        return 0;
    }
    return a.hdr->total_units;
}

// Decode unit u (false past the end; total from pb_total).
template <bool kVar>
__device__ __forceinline__ bool pb_unit(const BwdArgs& a, int total, int u, PBUnit& U) {
    if (u < 0 || u >= total) return false;
    if constexpr (kVar) {
        const int4 e = a.units[u];
        U.seq = e.x;
        U.hk = e.y;
        U.kb = e.z;
        U.tok0 = a.cu_s[U.seq];            // sanitised by the plan kernel
        U.len = a.cu_s[U.seq + 1] - U.tok0;
    } else {
        const int nkb = (a.N + kKeyBlock - 1) / kKeyBlock, bh = a.B * a.Hkv;
        int r;
        if ((a.causal || a.deterministic) && !a.naive) {
            U.kb = u / bh;
            r = u - U.kb * bh;
        } else {
            r = u / nkb;
            U.kb = u - r * nkb;
        }
        U.seq = r / a.Hkv;
        U.hk = r - U.seq * a.Hkv;
        U.tok0 = U.seq * a.N;
        U.len = a.N;
    }
    U.nq = (U.len + kTileM - 1) / kTileM;
    U.i0 = a.causal ? 2 * U.kb : 0;
    if (U.i0 > U.nq) U.i0 = U.nq;
    U.n = (a.Hq / a.Hkv) * (U.nq - U.i0);
    return true;
}

// S^T / dP^T: M = 256 (keys), N = 128 (queries, 64 per CTA), K = d; both K-major.
__device__ __forceinline__ void pb_mma_kq(uint32_t d, uint32_t a_smem, uint32_t b_smem) {
    constexpr uint32_t idesc = idesc_bf16_f32(256, 128, 0, 0);
    const uint64_t ad = sdesc_sw128(a_smem, 16, 1024), bd = sdesc_sw128(b_smem, 16, 1024);
    static_for<8>([&](auto kc) {
        constexpr uint32_t k = kc;
        constexpr uint32_t ao = ((k >> 2) * kT16 + (k & 3) * 32) >> 4;   // A boxes: 128 rows x 128 B
        constexpr uint32_t bo = ((k >> 2) * 8192 + (k & 3) * 32) >> 4;   // B boxes: 64 rows x 128 B
        umma_ss_k<ao, bo, 2>(d, ad, bd, idesc, k > 0);
    });
}

// dV / dK: M = 256 (keys), N = d (64 per CTA, MN-major), K = 128 queries; A
// (bf16) from TMEM: queries 0-63 in columns 0-31 of the region, queries
// 64-127 kGap columns further than contiguous (P^T: 0, dS^T: 64).
template <uint32_t kGap>
__device__ __forceinline__ void pb_mma_tn(uint32_t d, uint32_t a_tmem, uint32_t b_smem, uint32_t acc) {
    constexpr uint32_t idesc = idesc_bf16_f32(256, 128, 0, 1);
    const uint64_t bd = sdesc_sw128(b_smem, kT16, 1024);
    static_for<8>([&](auto kc) {
        constexpr uint32_t k = kc, col = k * 8 + (k >= 4 ? kGap : 0);
        umma_ts_k<col, ((k * 2048) >> 4), 2>(d, a_tmem, bd, idesc, (acc | k) != 0);
    });
}

// dQ: M = 128 (queries, 64 per CTA), N = d (64 per CTA), K = 256 keys; A and B
// MN-major (a 16-key step is 2048 bytes further in both).
__device__ __forceinline__ void pb_mma_dq(uint32_t d, uint32_t a_smem, uint32_t b_smem) {
    constexpr uint32_t idesc = idesc_bf16_f32(128, 128, 1, 1);
    const uint64_t ad = sdesc_sw128(a_smem, kT32, 1024), bd = sdesc_sw128(b_smem, kT32, 1024);
    static_for<16>([&](auto kc) {
        constexpr uint32_t k = kc, off = (k * 2048) >> 4;
        umma_ss_k<off, off, 2>(d, ad, bd, idesc, k > 0);
    });
}

__device__ __forceinline__ void pb_fence_async_cta() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
// Per-warp arrival (elected lane) with cluster-scope release: the even CTA's
// tensor core reads shared memory this warp wrote (dS exchange).
__device__ __forceinline__ void pb_arrive_release_cluster_w(uint32_t cluster_addr) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];\n\t}"
        ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ void pb_tma_reduce_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
    asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3}], [%1];"
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(src), "r"(x), "r"(y) : "memory");
}
__device__ __forceinline__ void pb_bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void pb_bulk_wait_read0() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void pb_bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void pb_fence_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }
__device__ __forceinline__ int pb_ld_acquire(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void pb_red_release_add(int* p, int v) {
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void pb_named_bar(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void pb_named_arrive(int id, int n) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ bool pb_named_bar_or(int id, int n, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r) : "r"((uint32_t)pred), "r"(id), "r"(n) : "memory");
    return r != 0;
}
// Bounded whole-warp wait with cluster-scope acquire: the phase completes on
// arrivals released by both CTAs after writing shared memory the next
// product reads.
__device__ __forceinline__ bool pb_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool pb_wait_cluster_w(uint64_t* bar, uint32_t parity, const WaitCtx& w, int site) {
    const uint32_t a = smem_u32(bar);
    bool ok = pb_try_wait_cluster(a, parity) || mbar_wait(bar, parity, w, site);
    if (ok) ok = pb_try_wait_cluster(a, parity);   // the completed phase, observed with cluster acquire
    return __all_sync(0xffffffffu, ok);
}
__device__ __forceinline__ void pb_drain_wait(uint64_t* bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(smem_u32(bar), parity) && globaltimer_ns() - t0 < kWaitLimitNs) {}
}

#define PB_PAIR ((int)(blockIdx.x >> 1))
#define PB_NPAIRS ((int)(gridDim.x >> 1))
#define PB_RANK ((int)(blockIdx.x & 1))

// kDbg: the debug counters are armed (a separate build of the kernel, so
// that their tests cost nothing otherwise).  kVar: packed varlen batches (a
// separate build too: the fixed-length kernel measured 5 % slower with both
// decodes in one body).
template <bool kDbg, bool kVar>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kPBThreads, 1)
bwd_pair_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tq64,
                const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                const __grid_constant__ CUtensorMap tdo, const __grid_constant__ CUtensorMap tdo64,
                const __grid_constant__ CUtensorMap tdq64, const BwdArgs a) {
    extern __shared__ __align__(1024) uint8_t dsm[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t base = smem_u32(dsm);
    if (base & 1023u) {  // both CTAs see the same base and return together
        if (tid == 0 && atomicCAS(&a.hdr->status.code, 0, -1) == 0) a.hdr->status.where = 800;
        return;
    }
    const bool leader = cluster_rank() == 0;
    PBShared& sh = *reinterpret_cast<PBShared*>(dsm + kOffBar);
    float* s_lse = reinterpret_cast<float*>(dsm + kOffStat);  // [2][128], LSE * log2(e)
    float* s_D = s_lse + 256;                                 // [2][128]
    const uint32_t sK = base + kOffK, sV = base + kOffV, sKdq = base + kOffKdq, sDS = base + kOffDS;

    if (tid == 0) {
        mbar_init(&sh.kv_full, 1);
        mbar_init(&sh.kv_empty, 2);    // both issuers (dQ reads K too)
        mbar_init(&sh.qs_full, 1);
        mbar_init(&sh.qs_empty, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&sh.q_empty[s], 1);
            mbar_init(&sh.st_full[s], 1);
        }
        mbar_init(&sh.dsx, 4);         // the local half's warps (one carries the peer's bytes)
        mbar_init(&sh.dsx_ready, 2);   // one relay arrival from each CTA
        mbar_init(&sh.qd_full, 1);
        mbar_init(&sh.do_full, 1);
        mbar_init(&sh.do_empty, 1);
        mbar_init(&sh.s_full, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&sh.s_read[s], 16);    // key-row warps of both CTAs have loaded S^T
            mbar_init(&sh.dq_free[s], 8);    // drain warps of both CTAs
        }
        mbar_init(&sh.dp_full, 1);
        mbar_init(&sh.p_ready, 16);    // key-row warps of both CTAs
        mbar_init(&sh.ds_ready, 16);
        mbar_init(&sh.ds_free, 1);
        mbar_init(&sh.dq_full, 1);
        mbar_init(&sh.dkdv_done, 1);
        mbar_init(&sh.acc_free, 8);
        mbar_init(&sh.drain, 2);       // both issuers
        sh.abort_flag = 0;
        sh.total = pb_total<kVar>(a);
        fence_mbar_init();
    }
    if (warp == 8 && lane == 0) {
        tma_prefetch_desc(&tq);
        tma_prefetch_desc(&tq64);
        tma_prefetch_desc(&tk);
        tma_prefetch_desc(&tv);
        tma_prefetch_desc(&tdo);
        tma_prefetch_desc(&tdo64);
        tma_prefetch_desc(&tdq64);
    }
    if (warp == 0) {
        tmem_alloc_pair(&sh.tmem_base, 512);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync_all();   // barriers of both CTAs initialised before any remote arrival
    tc_fence_after();

    const WaitCtx wc{&sh.abort_flag, &a.hdr->status};
    const uint32_t tmem = sh.tmem_base;
    const int total = sh.total;
    const int g = a.Hq / a.Hkv;
    const float scale = a.scale_log2;
    auto lead = [](uint64_t* bar) { return mapa_rank(smem_u32(bar), 0); };

    // Register split as in fa_bwd.cu: 128 * (144 + 144 + 168 + 56) = 65536.
    if (warp >= 8 && warp < 12) {
        regs_dec<56>();
        if (warp == 8) {
            // ------------------------------------------------------------ loader
            // Lane 0 waits and issues the TMA loads; the whole warp loads LSE/D.
            uint32_t jj = 0, uc = 0;
            bool ok = true;
            for (int u = PB_PAIR; ok; u += PB_NPAIRS) {
                PBUnit U;
                if (!pb_unit<kVar>(a, total, u, U)) break;
                if (lane == 0) {
                    ok = mbar_wait(&sh.kv_empty, (uc & 1) ^ 1, wc, kPBSiteKv);
                    if (ok) {
                        if (leader) mbar_arrive_expect_tx(&sh.kv_full, 2 * 3 * kT32);
                        const uint32_t bar = lead(&sh.kv_full);
                        const int k0 = U.tok0 + U.kb * kKeyBlock;
                        for (int c = 0; c < 2; ++c) {
                            tma_load_3d_pair(sK + c * kT16, &tk, bar, c * 64, U.hk, k0 + PB_RANK * kTileM);
                            tma_load_3d_pair(sV + c * kT16, &tv, bar, c * 64, U.hk, k0 + PB_RANK * kTileM);
                            tma_load_3d_pair(sKdq + c * kT16, &tk, bar, PB_RANK * 64, U.hk, k0 + c * kTileM);
                        }
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                const int span = U.nq - U.i0;
                for (int t = 0; t < U.n; ++t, ++jj) {
                    const int st = jj & 1, h = U.hk * g + t / span, i = U.i0 + t % span;
                    const int q0 = U.tok0 + i * kTileM;
                    // Q rows of this CTA's query half (read by S^T only) once the
                    // previous S^T is done; LSE/D slot once dK two tiles back is.
                    if (lane == 0) {
                        ok = mbar_wait(&sh.qs_empty, (jj & 1) ^ 1, wc, kPBSiteQ);
                        if (ok) {
                            if (leader) mbar_arrive_expect_tx(&sh.qs_full, 2 * kT16);
                            for (int c = 0; c < 2; ++c)
                                tma_load_3d_pair(base + kOffQs + c * 8192, &tq64, lead(&sh.qs_full), c * 64, h,
                                                 q0 + PB_RANK * 64);
                            ok = mbar_wait(&sh.q_empty[st], ((jj >> 1) & 1) ^ 1, wc, kPBSiteQ);
                        }
                    }
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (!ok) break;
                    // LSE (log2 units) and D of all 128 queries, for this CTA's key rows.
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int row = 4 * lane + e, q = i * kTileM + row;
                        float l2 = 0.f, dd = 0.f;
                        if (q < U.len) {
                            const size_t li = kVar ? (size_t)h * a.T + U.tok0 + q
                                                   : ((size_t)U.seq * a.Hq + h) * a.N + q;
                            l2 = a.lse[li] * 1.4426950408889634f;
                            dd = a.D[(size_t)h * a.T + U.tok0 + q];
                        }
                        s_lse[st * 128 + row] = l2;
                        s_D[st * 128 + row] = dd;
                    }
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&sh.st_full[st]);
                        // dO, both halves, once dV of the previous tile is done:
                        // dP is the tile's first product after S, so its operand
                        // goes ahead of Q's dK half below, which waits for the
                        // previous tile's dK, a product later.
                        ok = mbar_wait(&sh.do_empty, (jj & 1) ^ 1, wc, kPBSiteDo);
                        if (ok) {
                            if (leader) mbar_arrive_expect_tx(&sh.do_full, 2 * 2 * kT16);
                            for (int c = 0; c < 2; ++c)
                                tma_load_3d_pair(base + kOffDOs + c * 8192, &tdo64, lead(&sh.do_full), c * 64, h,
                                                 q0 + PB_RANK * 64);
                            tma_load_3d_pair(base + kOffDOd, &tdo, lead(&sh.do_full), PB_RANK * 64, h, q0);
                            // Q columns of this CTA's head-dim half (dK) once dK of the previous tile is done.
                            if (jj > 0) ok = mbar_wait(&sh.q_empty[(jj - 1) & 1], ((jj - 1) >> 1) & 1, wc, kPBSiteQ);
                        }
                        if (ok) {
                            if (leader) mbar_arrive_expect_tx(&sh.qd_full, 2 * kT16);
                            tma_load_3d_pair(base + kOffQd, &tq, lead(&sh.qd_full), PB_RANK * 64, h, q0);
                        }
                    }
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (!ok) break;
                }
                ++uc;
            }
            // The even CTA's full barriers count both CTAs' bytes: once their
            // last phases are complete nothing is in flight.
            if (lane == 0 && leader) {
                if (jj > 0) {
                    pb_drain_wait(&sh.qs_full, (jj - 1) & 1);
                    pb_drain_wait(&sh.qd_full, (jj - 1) & 1);
                    pb_drain_wait(&sh.do_full, (jj - 1) & 1);
                }
                if (uc > 0) pb_drain_wait(&sh.kv_full, (uc - 1) & 1);
            }
            __syncwarp();
        } else if (warp == 10 && leader) {
            // ------------------------------------------------------ dQ issuer
            // dQ(j) = dS K into R0 columns 64-127 once both CTAs' dS buffers
            // are complete and those columns are free: the key rows have read
            // S^T(j+1) there, or, for the unit's last tile (whose dQ reads
            // this unit's K, so it cannot wait for the next unit's S^T), the
            // drain has read dQ(j-1) and the key rows S^T(j).
            uint32_t jj = 0;
            bool ok = true;
            for (int u = PB_PAIR; ok; u += PB_NPAIRS) {
                PBUnit U;
                if (!pb_unit<kVar>(a, total, u, U)) break;
                for (int t = 0; t < U.n; ++t, ++jj) {
                    if (t + 1 < U.n) {
                        const uint32_t n1 = jj + 1;
                        if (!(ok = mbar_wait_w(&sh.s_read[n1 & 1], (n1 >> 1) & 1, wc, kPBSiteR0))) break;
                    } else {
                        if (!(ok = mbar_wait_w(&sh.s_read[jj & 1], (jj >> 1) & 1, wc, kPBSiteR0))) break;
                        const uint32_t p1 = jj - 1;
                        if (jj > 0 && !(ok = mbar_wait_w(&sh.dq_free[p1 & 1], (p1 >> 1) & 1, wc, kPBSiteDqFree))) break;
                    }
                    if (!(ok = pb_wait_cluster_w(&sh.dsx_ready, jj & 1, wc, kPBSiteDs))) break;
                    tc_fence_after();
                    pb_mma_dq(tmem + kColR0 + 64, sDS, sKdq);
                    umma_commit_pair_w(&sh.dq_full, kBoth);
                    umma_commit_pair_w(&sh.ds_free, kBoth);      // both CTAs' dS buffers read
                }
                if (!ok) break;
                umma_commit_pair_w(&sh.kv_empty, kBoth);         // this unit's K (dQ's B) read
            }
            umma_commit_pair_w(&sh.drain, kLead);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(smem_u32(&sh.drain), 0) && globaltimer_ns() - t0 < kWaitLimitNs) {}
            __syncwarp();
        } else if (warp == 11) {
            // --------------------------------------------------- dS relay
            // This CTA's dS buffer is complete once its own half has written
            // its rows and the peer's rows have arrived (bulk copy, counted on
            // dsx): tell the even CTA's issuer, whose dQ product reads it.
            uint32_t jj = 0;
            bool ok = true;
            for (int u = PB_PAIR; ok; u += PB_NPAIRS) {
                PBUnit U;
                if (!pb_unit<kVar>(a, total, u, U)) break;
                for (int t = 0; t < U.n; ++t, ++jj) {
                    if (!(ok = mbar_wait_w(&sh.dsx, jj & 1, wc, kPBSiteDs))) break;
                    pb_arrive_release_cluster_w(lead(&sh.dsx_ready));
                }
            }
            __syncwarp();
        } else if (warp == 9 && leader) {
            // ---------------------------------------------- dP, dV, S, dK issuer
            uint32_t jj = 0, uc = 0;
            bool ok = true;
            for (int u = PB_PAIR; ok; u += PB_NPAIRS) {
                PBUnit U;
                if (!pb_unit<kVar>(a, total, u, U)) break;
                if (U.n == 0) {   // no visible query tile: only the zero epilogue
                    if (!(ok = mbar_wait_w(&sh.kv_full, uc & 1, wc, kPBSiteKv))) break;
                    if (!(ok = mbar_wait_w(&sh.acc_free, (uc & 1) ^ 1, wc, kPBSiteAcc))) break;
                    umma_commit_pair_w(&sh.dkdv_done, kBoth);
                    umma_commit_pair_w(&sh.kv_empty, kBoth);
                    ++uc;
                    continue;
                }
                if (!(ok = mbar_wait_w(&sh.kv_full, uc & 1, wc, kPBSiteKv))) break;
                if (!(ok = mbar_wait_w(&sh.acc_free, (uc & 1) ^ 1, wc, kPBSiteAcc))) break;
                // S^T(j) into R0: both 64-column halves must be free.  The P^T
                // half was read by dV(j-1), issued earlier by this thread.  The
                // dQ half holds dQ(j-2) (written once the key rows had read
                // S^T(j-1)) until the drain has read it -- or, for a unit's
                // first tile, dQ(j-1): the previous unit's last dQ did not wait
                // for this S^T.
                auto issue_s = [&](uint32_t j, bool first) -> bool {
                    const uint32_t lag = first ? 1u : 2u, jt = j - lag;
                    if (j >= lag && !mbar_wait_w(&sh.dq_free[jt & 1], (jt >> 1) & 1, wc, kPBSiteDqFree)) return false;
                    if (!mbar_wait_w(&sh.qs_full, j & 1, wc, kPBSiteQ)) return false;
                    tc_fence_after();
                    pb_mma_kq(tmem + kColR0, sK, base + kOffQs);
                    umma_commit_pair_w(&sh.s_full, kBoth);
                    umma_commit_pair_w(&sh.qs_empty, kBoth);   // the Q rows may reload
                    return true;
                };
                if (!(ok = issue_s(jj, true))) break;
                for (int t = 0; t < U.n; ++t, ++jj) {
                    const uint32_t st = jj & 1;
                    // dP^T(j) into R1, which dK(j-1) (issued earlier by this thread) has read.
                    if (!(ok = mbar_wait_w(&sh.do_full, jj & 1, wc, kPBSiteDo))) break;
                    pb_mma_kq(tmem + kColR1, sV, base + kOffDOs);
                    umma_commit_pair_w(&sh.dp_full, kBoth);
                    if (!(ok = mbar_wait_w(&sh.p_ready, jj & 1, wc, kPBSiteP))) break;
                    tc_fence_after();
                    pb_mma_tn<0>(tmem + kColDV, tmem + kColR0, base + kOffDOd, t > 0);
                    umma_commit_pair_w(&sh.do_empty, kBoth);   // dO read by dP and dV
                    if (t + 1 < U.n && !(ok = issue_s(jj + 1, false))) break;   // right behind dV
                    if (!(ok = mbar_wait_w(&sh.ds_ready, jj & 1, wc, kPBSiteDs))) break;
                    if (!(ok = mbar_wait_w(&sh.qd_full, jj & 1, wc, kPBSiteQ))) break;
                    tc_fence_after();
                    pb_mma_tn<64>(tmem + kColDK, tmem + kColR1, base + kOffQd, t > 0);
                    umma_commit_pair_w(&sh.q_empty[st], kBoth);  // Q columns and LSE/D of this tile consumed
                }
                if (!ok) break;
                umma_commit_pair_w(&sh.dkdv_done, kBoth);
                umma_commit_pair_w(&sh.kv_empty, kBoth);
                ++uc;
            }
            umma_commit_pair_w(&sh.drain, kLead);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(smem_u32(&sh.drain), 0) && globaltimer_ns() - t0 < kWaitLimitNs) {}
            __syncwarp();
        }
    } else if (warp < 4 || warp >= 12) {
        regs_inc<144>();
        // ------------------------------------------------ P^T and dS^T (key rows)
        const int hc = warp >= 12 ? 1 : 0;                   // query half: columns 64 hc .. +63
        const int cb = hc * 64;
        const int r = (warp & 3) * 32 + lane;                // key row of this CTA == TMEM lane
        const uint32_t lb = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tR0 = tmem + lb + kColR0, tR1 = tmem + lb + kColR1;
        // dS row of this key in the dQ A operand of CTA hc (queries 64 hc .. +63):
        // key row R = 128 rank + r of that CTA's 256-row buffer.  The half for
        // this CTA writes it in place; the other half writes it to the outbox
        // (same row layout: R % 8 == r % 8), which one bulk copy moves to the
        // peer.
        const bool local_half = hc == PB_RANK;
        uint8_t* ds_row = local_half ? dsm + kOffDS + (PB_RANK * 128 + r) * 128 : dsm + kOffOut + r * 128;
        const int sw = r & 7;
        uint32_t jj = 0;
        bool ok = true;
        for (int u = PB_PAIR; ok; u += PB_NPAIRS) {
            PBUnit U;
            if (!pb_unit<kVar>(a, total, u, U)) break;
            const int key = U.kb * kKeyBlock + PB_RANK * kTileM + r;
            const int span = U.nq - U.i0;
            for (int t = 0; t < U.n; ++t, ++jj) {
                const int st = jj & 1, i = U.i0 + t % span;
                bool okw = mbar_wait(&sh.st_full[st], (jj >> 1) & 1, wc, kPBSiteSt);
                okw = okw && mbar_wait(&sh.s_full, jj & 1, wc, kPBSiteS);
                float p[64];
                if (okw) {
                    tc_fence_after();
                    uint32_t* pu = reinterpret_cast<uint32_t*>(p);
                    tmem_ld32(tR0 + cb, *reinterpret_cast<uint32_t(*)[32]>(pu + 0));
                    tmem_ld32(tR0 + cb + 32, *reinterpret_cast<uint32_t(*)[32]>(pu + 32));
                    tmem_wait_ld();
                    tc_fence_before();
                    mbar_arrive_remote_w(lead(&sh.s_read[jj & 1]));   // R0 columns 64-127 may take dQ(j-1)
                    // Half 1 packs its P^T into columns 32-63, which half 0
                    // reads: half 0 signals its loads done on the lane
                    // quadrant's named barrier, half 1 waits there before its
                    // stores.  Both do so in every tile, whatever their waits
                    // returned (the else branch below).
                    if (hc == 0) pb_named_arrive(2 + (warp & 3), 64);
                    tc_fence_after();
                    const int c_lo = (a.causal ? key - i * kTileM : 0) - cb;
                    const int c_hi = (key >= U.len ? 0 : U.len - i * kTileM) - cb;
                    const float4* l2v = reinterpret_cast<const float4*>(s_lse + st * 128 + cb);
                    if (c_lo <= 0 && c_hi >= 64) {
#pragma unroll
                        for (int c4 = 0; c4 < 16; ++c4) {
                            const float4 l4 = l2v[c4];
                            p[4 * c4] = ex2_mufu(fmaf(p[4 * c4], scale, -l4.x));
                            p[4 * c4 + 1] = ex2_mufu(fmaf(p[4 * c4 + 1], scale, -l4.y));
                            p[4 * c4 + 2] = ex2_mufu(fmaf(p[4 * c4 + 2], scale, -l4.z));
                            p[4 * c4 + 3] = ex2_mufu(fmaf(p[4 * c4 + 3], scale, -l4.w));
                        }
                    } else {
#pragma unroll
                        for (int c4 = 0; c4 < 16; ++c4) {
                            const float4 l4 = l2v[c4];
                            const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int c = 4 * c4 + e;
                                const float pe = ex2_mufu(fmaf(p[c], scale, -lv[e]));
                                p[c] = (c >= c_lo && c < c_hi) ? pe : 0.f;
                            }
                        }
                    }
                    if (hc == 1) {
                        pb_named_bar(2 + (warp & 3), 64);
                        tc_fence_after();
                    }
#pragma unroll
                    for (int stg = 0; stg < 2; ++stg) {
                        uint32_t pk[16];
#pragma unroll
                        for (int m = 0; m < 16; ++m) pk[m] = pack_bf16x2(p[stg * 32 + 2 * m], p[stg * 32 + 2 * m + 1]);
                        tmem_st16(tR0 + hc * 32 + stg * 16, pk);   // P^T: columns 32 hc .. +31
                    }
                    tmem_wait_st();
                    tc_fence_before();
                    mbar_arrive_remote_w(lead(&sh.p_ready));
                    okw = mbar_wait(&sh.dp_full, jj & 1, wc, kPBSiteDp);
                    okw = okw && mbar_wait(&sh.ds_free, (jj & 1) ^ 1, wc, kPBSiteDsFree);
                } else if (hc == 0) {
                    pb_named_arrive(2 + (warp & 3), 64);
                } else {
                    pb_named_bar(2 + (warp & 3), 64);
                }
                // dS^T over the dP^T columns this thread has read: half 0 packs
                // into R1 columns 0-31, half 1 into 96-127 (taking its second
                // chunk first), which leaves columns 32-95 for dQ_i.
                if (okw) {
                    tc_fence_after();
                    const float4* dv4 = reinterpret_cast<const float4*>(s_D + st * 128 + cb);
                    auto chunk = [&](auto ccc) {
                        constexpr int cc = ccc;
                        uint32_t dp[32];
                        tmem_ld32(tR1 + cb + cc * 32, dp);
                        tmem_wait_ld();
                        uint32_t pk[16];
#pragma unroll
                        for (int m = 0; m < 8; ++m) {
                            const float4 d4 = dv4[cc * 8 + m];
                            const int c = cc * 32 + 4 * m;
                            pk[2 * m] = pack_bf16x2(p[c] * (__uint_as_float(dp[4 * m]) - d4.x),
                                                    p[c + 1] * (__uint_as_float(dp[4 * m + 1]) - d4.y));
                            pk[2 * m + 1] = pack_bf16x2(p[c + 2] * (__uint_as_float(dp[4 * m + 2]) - d4.z),
                                                        p[c + 3] * (__uint_as_float(dp[4 * m + 3]) - d4.w));
                        }
                        // 32 queries = four 16-byte chunks of the 128-byte row:
                        // chunk q (queries 64 hc + 8q .. +7) at position q ^ (R % 8)
                        // of the row in CTA hc's buffer.
#pragma unroll
                        for (int m = 0; m < 4; ++m) {
                            const int q = cc * 4 + m;
                            *reinterpret_cast<uint4*>(ds_row + ((q ^ sw) << 4)) =
                                make_uint4(pk[4 * m], pk[4 * m + 1], pk[4 * m + 2], pk[4 * m + 3]);
                        }
                        tmem_st16(tR1 + hc * 96 + cc * 16, pk);
                    };
                    if (hc == 0) {
                        chunk(std::integral_constant<int, 0>{});
                        chunk(std::integral_constant<int, 1>{});
                    } else {
                        chunk(std::integral_constant<int, 1>{});
                        chunk(std::integral_constant<int, 0>{});
                    }
                }
                // Both warps of the lane quadrant leave together (the P^T
                // hand-off above needs both in every tile).
                if (pb_named_bar_or(6 + (warp & 3), 64, !okw)) { ok = false; break; }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive_remote_w(lead(&sh.ds_ready));   // dS^T in TMEM: dK may start
                pb_fence_async_cta();                        // this thread's dS rows before the copy / product
                __syncwarp();
                if (lane == 0) {
                    if (local_half) {
                        if ((warp & 3) == 0) mbar_arrive_expect_tx(&sh.dsx, kT16);   // the peer's rows, by bulk copy
                        else mbar_arrive(&sh.dsx);
                    } else {
                        // This warp's 32 rows (keys of this CTA, the peer's
                        // queries) into the peer's buffer at rows 128 rank +
                        // 32 w .. +31, counted on the peer's dsx: four copies in
                        // flight per CTA.
                        const uint32_t rows = (uint32_t)(warp & 3) * 32 * 128;
                        const uint32_t dst = mapa_rank(sDS + PB_RANK * 128 * 128 + rows, hc);
                        const uint32_t bar = mapa_rank(smem_u32(&sh.dsx), hc);
                        asm volatile(
                            "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                            ::"r"(dst), "r"(base + kOffOut + rows), "r"(32 * 128), "r"(bar) : "memory");
                    }
                }
            }
        }
    } else {
        regs_inc<168>();
        // -------------------------------------------- dQ drain, dK/dV epilogue
        const int r = tid - 128;                             // TMEM lane
        const int wq = warp & 3;
        const uint32_t lb = (uint32_t)(wq * 32) << 16;
        const uint32_t tDQ = tmem + lb + kColR0 + 64;
        const int qrow = r & 63, dh = r >> 6;                // dQ row of this CTA's 64 and head-dim half
        uint32_t jj = 0, uc = 0;
        bool ok = true;
        // Deterministic mode: a query tile's semaphore counts the CTAs that
        // have added their 64-row slice of it; key block kb adds once the
        // count has reached 2 kb (both CTAs of every earlier block).  The
        // release of a tile's count waits for that tile's reductions to
        // complete; it is done at the next tile's semaphore wait (or before
        // the unit's dK/dV epilogue), so the drain does not stall on the
        // round trip to L2 every tile.
        int* sem_pend = nullptr;
        auto release_pending = [&]() {
            if (r == 0 && sem_pend) {
                pb_bulk_wait0();          // the tile's additions are complete
                pb_fence_async_global();  // ... and ordered before the release
                pb_red_release_add(sem_pend, 1);
            }
            sem_pend = nullptr;
        };
        for (int u = PB_PAIR; ok; u += PB_NPAIRS) {
            PBUnit U;
            if (!pb_unit<kVar>(a, total, u, U)) break;
            const int span = U.nq - U.i0;
            for (int t = 0; t < U.n; ++t, ++jj) {
                const int h = U.hk * g + t / span, i = U.i0 + t % span;
                ok = mbar_wait(&sh.dq_full, jj & 1, wc, kPBSiteDq);
                ok = !pb_named_bar_or(1, 128, !ok);
                if (!ok) break;
                tc_fence_after();
                uint32_t v[64];
                tmem_ld32(tDQ + 0, *reinterpret_cast<uint32_t(*)[32]>(v + 0));
                tmem_ld32(tDQ + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
                tmem_wait_ld();
                tc_fence_before();
                mbar_arrive_remote_w(lead(&sh.dq_free[jj & 1]));
                int* sem = a.deterministic ? a.sem + (size_t)h * a.sem_stride + U.seq + (U.tok0 + i * kTileM) / kTileN
                                           : nullptr;
                if (sem) {
                    release_pending();
                    // Wait (bounded) for the earlier key blocks' slices; the
                    // wait runs in another warp than the releasing thread, and
                    // the barrier below orders it before this tile's additions.
                    bool gave_up = false;
                    if (r == 32) {
                        const uint64_t t0 = globaltimer_ns();
                        uint32_t spins = 0;
                        while (pb_ld_acquire(sem) < 2 * U.kb) {
                            if ((++spins & 255u) == 0 &&
                                (*(volatile int*)&sh.abort_flag || globaltimer_ns() - t0 > kWaitLimitNs)) {
                                if (atomicCAS(&a.hdr->status.code, 0, kStatusTimeout) == 0) {
                                    a.hdr->status.where = kPBSiteSem;
                                    a.hdr->status.block = blockIdx.x;
                                }
                                *(volatile int*)&sh.abort_flag = 1;
                                gave_up = true;
                                break;
                            }
                        }
                    }
                    if (pb_named_bar_or(1, 128, gave_up)) { ok = false; break; }
                    if (r == 0) pb_fence_async_global();  // our bulk reduction follows the acquire
                }
                // Add this CTA's 64 x 128 slice of dQ_i into the fp32
                // accumulator: two rounds, each two 64-row x 32-column boxes
                // (one per head-dim half), staged like a 128-B TMA box.
                const int grow = h * (int)a.T + U.tok0 + i * kTileM + PB_RANK * 64;
                uint8_t* stage_row = dsm + kOffStage + dh * 8192 + qrow * 128;
#pragma unroll
                for (int rnd = 0; rnd < 2; ++rnd) {
                    if (r == 0) pb_bulk_wait_read0();
                    pb_named_bar(1, 128);
                    const uint32_t* src = v + rnd * 32;
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        *reinterpret_cast<uint4*>(stage_row + ((q ^ (qrow & 7)) << 4)) =
                            make_uint4(src[4 * q], src[4 * q + 1], src[4 * q + 2], src[4 * q + 3]);
                    pb_fence_async_cta();
                    pb_named_bar(1, 128);
                    if (r == 0) {
                        pb_tma_reduce_2d(&tdq64, base + kOffStage, rnd * 32, grow);
                        pb_tma_reduce_2d(&tdq64, base + kOffStage + 8192, 64 + rnd * 32, grow);
                        pb_bulk_commit();
                    }
                }
                sem_pend = sem;
                // This CTA's key tile contributed to query tile i unless it
                // lies past the sequence or (causal) after the tile's rows.
                const int kt = 2 * U.kb + PB_RANK;
                if (kDbg && r == 0 && kt * kTileN < U.len && (!a.causal || i >= kt))
                    dbg_count(a.dbg_inner, (long long)h * a.T + U.tok0 + i * kTileM);
            }
            if (!ok) break;
            release_pending();   // before the dK/dV epilogue: the next key block is waiting
            if (!(ok = mbar_wait(&sh.dkdv_done, uc & 1, wc, kPBSiteDkdv))) break;
            ++uc;
            tc_fence_after();
            const int key = U.kb * kKeyBlock + PB_RANK * kTileM + r;
            const bool kvalid = key < U.len;
            const size_t orow = ((size_t)(U.tok0 + key) * a.Hkv + U.hk) * kHeadDim;
#pragma unroll
            for (int which = 0; which < 2; ++which) {
                const uint32_t tacc = tmem + lb + (which ? kColDV : kColDK);
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
                            // Units that see no query tile leave the accumulators untouched: write zeros.
                            const float* f = reinterpret_cast<const float*>(w + 8 * m);
                            const float z = U.n > 0 ? 1.f : 0.f;
                            out[cc * 4 + m] = make_uint4(pack_bf16x2(f[0] * mul * z, f[1] * mul * z),
                                                         pack_bf16x2(f[2] * mul * z, f[3] * mul * z),
                                                         pack_bf16x2(f[4] * mul * z, f[5] * mul * z),
                                                         pack_bf16x2(f[6] * mul * z, f[7] * mul * z));
                        }
                    }
                }
            }
            if (kDbg && r == 0 && (2 * U.kb + PB_RANK) * kTileN < U.len)
                dbg_count(a.dbg_visits, (long long)U.hk * a.T + U.tok0 + (2 * U.kb + PB_RANK) * kTileN);
            tc_fence_before();
            mbar_arrive_remote_w(lead(&sh.acc_free));
        }
        if (r == 0) pb_bulk_wait0();   // every bulk reduction issued here has completed
    }

    if (sh.abort_flag) {   // the odd CTA cannot observe its own last loads (they count on the even CTA)
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 200000ull) {}
    }
    tc_fence_before();
    cluster_sync_all();   // no product, load or remote access still targets either CTA
    tc_fence_after();
    if (warp == 0) tmem_dealloc_pair(tmem, 512);
}

#undef PB_PAIR
#undef PB_NPAIRS
#undef PB_RANK

}  // namespace

int g_bwd_pairs_resident = 0;

bool bwd_pair_supported(const BwdArgs&) { return true; }

cudaError_t launch_bwd_pair_main(const BwdLaunch& L, cudaStream_t stream) {
    const bool dbg = L.a.dbg_visits || L.a.dbg_inner;
    auto kern = L.a.varlen ? (dbg ? bwd_pair_kernel<true, true> : bwd_pair_kernel<false, true>)
                           : (dbg ? bwd_pair_kernel<true, false> : bwd_pair_kernel<false, false>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPBSmem);
    if (e != cudaSuccess) return e;
    int max_pairs = g_bwd_pairs_resident;
    if (max_pairs == 0) {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(2 * (unsigned)(L.num_sms / 2), 1, 1);
        cfg.blockDim = dim3(kPBThreads, 1, 1);
        cfg.dynamicSmemBytes = kPBSmem;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n < 1) n = L.num_sms / 2;
        max_pairs = g_bwd_pairs_resident = n;
    }
    const BwdArgs& a = L.a;
    const long long units = a.varlen ? (long long)a.Hkv * ((a.T + kKeyBlock - 1) / kKeyBlock + a.B)
                                     : (long long)a.B * a.Hkv * ((a.N + kKeyBlock - 1) / kKeyBlock);
    int pairs = (int)(units < max_pairs ? units : max_pairs);
    if (pairs < 1) pairs = 1;
    kern<<<2 * pairs, kPBThreads, kPBSmem, stream>>>(L.tq, L.tq64, L.tk, L.tv, L.tdo, L.tdo64, L.tdq64, a);
    return cudaGetLastError();
}

}  // namespace fa
