// fa_fwd256.cu -- forward attention for head dim d = 256 (sm_103a).
//
// The same O = softmax(alpha Q K^T [+ causal]) V and LSE as fa_fwd.cu
// (FlashAttention-4 blog, "Forward pass"), for the head dim at which the
// products, not the exponentials, set the pace (FlashAttention-4 paper
// summary, roofline remarks: the balance point moves with d).  At d = 256 a
// 128-row tile of Q, K or V is 64 KB, so the layout differs from the d = 128
// kernels: one CTA per SM owns one 128-row query tile at a time and streams
// 64-key blocks of K and V.  Fixed-length and packed variable-length inputs.
//
//   warps 0-3  softmax: one thread per query row (TMEM lane), 64 scores per
//              block; conditional rescale of its O row (tau), P as bf16 into
//              tensor memory over the scores it read, the epilogue; between
//              units, the copy of the next query tile from shared into
//              tensor memory;
//   warp  4    TMA loader: K and V blocks through one ring in the order the
//              products read them (K0, K1, V0, K2, V1, K3, ...), so a K block
//              is requested ~2.5 blocks ahead; the next unit's Q after this
//              unit's K0 and K1;
//   warp  5    UMMA issuer: S = Q K^T (M 128, N 64, K 256: 16 steps, Q from
//              tensor memory) and O += P V (M 128, N 256, K 64: 4 steps, P
//              from tensor memory).
//
// Tensor memory (512 columns): O 0-255; S/P of block j in 256 + 64 (j % 2)
// (two regions, so S of block j+1 is computed while the softmax of block j
// runs; P of block j overwrites the first 32 columns of its region and is
// read by the P V of block j before S of block j+2 is written there -- the
// issuer emits both, in that order); the query tile, bf16 pairs, in 384-511.
// With Q in tensor memory an S step reads only its 2 KB of K from shared
// memory: a 128 x 64 x 16 product with both operands in shared memory reads
// 6 KB and runs at two thirds of the tensor rate, bound by shared-memory
// bandwidth (measured on GB300: 48 instead of 32 cycles).
//
// Shared memory: a 64 KB landing area for Q (four 128-row x 64-column boxes)
// and a ring of five 32 KB slots, each one 64-key block of K or V (four 64-row
// x 64-column boxes).
#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kD = 256;
constexpr int kBlk = 64;                         // keys per block
constexpr int kThreads256 = 192;
constexpr int kRing = 5;                         // K and V blocks in consumption order
constexpr uint32_t kQBox = 16384;                // 128 rows x 128 B
constexpr uint32_t kKVBox = 8192;                // 64 rows x 128 B
constexpr uint32_t kQBytes = 4 * kQBox, kKVBytes = 4 * kKVBox;
constexpr uint32_t kOffQ = 0, kOffR = kQBytes;
constexpr uint32_t kSmem256 = 1024 + kOffR + kRing * kKVBytes;   // + alignment slack
static_assert(kSmem256 <= 232448, "shared memory plan");
constexpr uint32_t kColO = 0, kColS = 256, kColQ = 384;

enum : int { k6QEmpty = 41, k6KEmpty, k6VEmpty, k6QFull, k6KFull, k6VFull, k6S, k6P, k6PV, k6O, k6OFree };

struct Shared256 {
    uint64_t q_full, q_empty, full[kRing], empty[kRing];
    uint64_t qt_full, s_full[2], p_ready[2], pv_done[2], o_done, o_free, drain;
    uint32_t tmem_base;
    int abort_flag;
};

struct Unit256 {
    int seq, h, m, tok0, len, nb;
};

// Blocks of 64 keys a query tile visits: all of its sequence's, or under the
// causal mask those holding keys up to the tile's last row.
__device__ __forceinline__ void set_blocks(const FwdArgs& a, Unit256& U) {
    const int all = (U.len + kBlk - 1) / kBlk;
    const int diag = (U.m * kTileM + kTileM - 1) / kBlk + 1;
    U.nb = a.causal && diag < all ? diag : all;
}

// Fixed length, unit u: one 128-row query tile of one (batch, head).
// Non-causal (and the naive order of fa_set_schedule_order): (batch, head)
// major; causal: query tiles from the last (longest first), (batch, head)
// minor.
__device__ __forceinline__ bool unit256(const FwdArgs& a, int u, Unit256& U) {
    const int nm = (a.N + kTileM - 1) / kTileM, bh_all = a.B * a.Hq;
    if (u < 0 || u >= bh_all * nm) return false;
    int bh;
    if (a.causal && !a.naive) {
        U.m = nm - 1 - u / bh_all;
        bh = u % bh_all;
    } else {
        bh = u / nm;
        U.m = u - bh * nm;
    }
    U.seq = bh / a.Hq;
    U.h = bh - U.seq * a.Hq;
    U.tok0 = U.seq * a.N;
    U.len = a.N;
    set_blocks(a, U);
    return true;
}

// Units of packed variable-length sequences (cu_seqlens).  Level k holds
// every sequence's k-th query tile counted from its last one (under the
// causal mask the last tile is the most expensive, so the costliest units
// come first); within a level, sequences in order, heads minor.  Each role
// asks for its units in non-decreasing order, so one cursor per thread walks
// the levels and sequences once: O(levels x B) reads of cu_seqlens per CTA.
// Offsets are sanitised by the rule every kernel here applies: each is
// clamped to [0, T] and raised to at least the one before it (a running
// maximum the cursor carries along), so malformed offsets give empty
// sequences, never rows outside the tensors or overlapping sequences.
struct Walk256 {
    int k = -1, lvl_start = 0, lvl_count = 0, b = 0, idx_b = 0;
    int c0 = 0, c1 = 0;   // sanitised offsets of sequence b

    __device__ __forceinline__ static int clamp_t(const FwdArgs& a, int c) {
        return c < 0 ? 0 : (c > a.N ? a.N : c);
    }
    __device__ __forceinline__ void first(const FwdArgs& a) {
        b = 0;
        c0 = clamp_t(a, a.cu_seqlens[0]);
        c1 = max(c0, clamp_t(a, a.cu_seqlens[1]));
    }
    __device__ __forceinline__ void next(const FwdArgs& a) {   // sequence b + 1 (b + 1 < B)
        ++b;
        c0 = c1;
        c1 = max(c1, clamp_t(a, a.cu_seqlens[b + 1]));
    }
    __device__ __forceinline__ int tiles() const { return (c1 - c0 + kTileM - 1) / kTileM; }

    // The naive order: (sequence, head) major, query tiles ascending.
    __device__ bool get_naive(const FwdArgs& a, int u, Unit256& U) {
        if (u < 0) return false;
        if (k < 0) {
            k = 0;
            lvl_start = 0;
            first(a);
        }
        while (u >= lvl_start + a.Hq * tiles()) {   // a later sequence
            if (b + 1 >= a.B) return false;           // past the last one
            lvl_start += a.Hq * tiles();
            next(a);
        }
        const int i = u - lvl_start, nt = tiles();
        U.seq = b;
        U.h = i / nt;
        U.m = i - U.h * nt;
        U.tok0 = c0;
        U.len = c1 - c0;
        set_blocks(a, U);
        return true;
    }

    __device__ bool get(const FwdArgs& a, int u, Unit256& U) {
        if (!a.varlen) return unit256(a, u, U);
        if (a.naive) return get_naive(a, u, U);
        if (u < 0) return false;
        while (k < 0 || u >= lvl_start + lvl_count) {
            lvl_start += lvl_count;
            ++k;
            int n = 0;
            first(a);
            for (int s = 0; s < a.B; ++s) {
                n += tiles() > k;
                if (s + 1 < a.B) next(a);
            }
            lvl_count = n * a.Hq;
            if (n == 0) return false;                    // past the last level
            for (first(a); tiles() <= k; next(a)) {}     // stops at a sequence of this level
            idx_b = 0;
        }
        const int i = u - lvl_start;
        while (i >= idx_b + a.Hq) {                      // a later sequence of this level
            idx_b += a.Hq;
            do next(a); while (tiles() <= k);
        }
        U.seq = b;
        U.h = i - idx_b;
        U.tok0 = c0;
        U.len = c1 - c0;
        U.m = (U.len + kTileM - 1) / kTileM - 1 - k;
        set_blocks(a, U);
        return true;
    }
};

// S = Q K^T: both K-major; k-step k (16 of the 256 head-dim columns) is box
// k / 4, bytes (k % 4) * 32 of each 128-byte row.
__device__ __forceinline__ void issue_s(uint32_t d_tmem, uint32_t q_tmem, uint32_t k_smem) {
    constexpr uint32_t idesc = idesc_bf16_f32(128, kBlk, 0, 0);
    const uint64_t kd = sdesc_sw128(k_smem, 16, 1024);
    static_for<16>([&](auto kc) {
        constexpr uint32_t k = kc;
        constexpr uint32_t bo = ((k >> 2) * kKVBox + (k & 3) * 32) >> 4;
        umma_ts_k<k * 8, bo>(d_tmem, q_tmem, kd, idesc, k > 0);
    });
}

// O (+)= P V: A = P (bf16 in tensor memory, 8 columns per 16 keys); B = V
// MN-major, N = 256 over four 64-column boxes kKVBox apart, a 16-key step
// 16 rows x 128 B = 2048 bytes further.
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint32_t v_smem, uint32_t acc) {
    constexpr uint32_t idesc = idesc_bf16_f32(128, kD, 0, 1);
    const uint64_t vd = sdesc_sw128(v_smem, kKVBox, 1024);
    static_for<kBlk / 16>([&](auto kc) {
        constexpr uint32_t k = kc;
        umma_ts_k<k * 8, ((k * 2048) >> 4)>(d_tmem, p_tmem, vd, idesc, (acc | k) != 0);
    });
}

// kDbg: the debug counters are armed (a separate build of the kernel, so
// that their tests cost nothing otherwise).
template <bool kDbg>
__global__ void __launch_bounds__(kThreads256, 1)
fwd256_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
              const __grid_constant__ CUtensorMap tv, const FwdArgs a) {
    extern __shared__ uint8_t dsmem[];
    __shared__ Shared256 sh;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t base = (smem_u32(dsmem) + 1023u) & ~1023u;
    const uint32_t sQ = base + kOffQ, sR = base + kOffR;

    if (tid == 0) {
        mbar_init(&sh.q_full, 1);
        mbar_init(&sh.q_empty, 128);
        mbar_init(&sh.qt_full, 128);
        for (int i = 0; i < kRing; ++i) { mbar_init(&sh.full[i], 1); mbar_init(&sh.empty[i], 1); }
        mbar_init(&sh.s_full[0], 1);
        mbar_init(&sh.s_full[1], 1);
        mbar_init(&sh.p_ready[0], 128);
        mbar_init(&sh.p_ready[1], 128);
        mbar_init(&sh.pv_done[0], 1);
        mbar_init(&sh.pv_done[1], 1);
        mbar_init(&sh.o_done, 1);
        mbar_init(&sh.o_free, 128);
        mbar_init(&sh.drain, 1);
        sh.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 4 && lane == 0) {
        tma_prefetch_desc(&tq);
        tma_prefetch_desc(&tk);
        tma_prefetch_desc(&tv);
    }
    if (warp == 0) {
        tmem_alloc(&sh.tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const WaitCtx wc{&sh.abort_flag, a.status};
    const uint32_t tmem = sh.tmem_base;
    const int group = a.Hq / a.Hkv;

    if (warp == 4) {
        // ---------------------------------------------------------------- loader
        if (lane == 0) {
            uint32_t it = 0, qc = 0;
            bool ok = true;
            // One block of K or V (64 keys x 256) into the next ring slot.
            auto load = [&](const CUtensorMap* m, int hk, int row) -> bool {
                const uint32_t rs = it % kRing;
                if (!mbar_wait(&sh.empty[rs], ((it / kRing) & 1) ^ 1, wc, k6KEmpty)) return false;
                mbar_arrive_expect_tx(&sh.full[rs], kKVBytes);
                for (int c = 0; c < 4; ++c)
                    tma_load_3d(sR + rs * kKVBytes + c * kKVBox, m, &sh.full[rs], c * 64, hk, row);
                ++it;
                return true;
            };
            auto load_q = [&](const Unit256& U) -> bool {
                if (!mbar_wait(&sh.q_empty, (qc & 1) ^ 1, wc, k6QEmpty)) return false;
                mbar_arrive_expect_tx(&sh.q_full, kQBytes);
                for (int c = 0; c < 4; ++c)
                    tma_load_3d(sQ + c * kQBox, &tq, &sh.q_full, c * 64, U.h, U.tok0 + U.m * kTileM);
                ++qc;
                return true;
            };
            Walk256 walk;
            {
                Unit256 U;
                if (walk.get(a, blockIdx.x, U)) ok = load_q(U);
            }
            for (int u = blockIdx.x; ok; u += gridDim.x) {
                Unit256 U, Un;
                if (!walk.get(a, u, U)) break;
                const int hk = U.h / group;
                // The issuer's order: K0, K1, then V j followed by K j+2; Q of
                // the next unit goes out early (its slot is free once this
                // unit's Q is in tensor memory).
                if (!(ok = load(&tk, hk, U.tok0))) break;
                if (U.nb > 1 && !(ok = load(&tk, hk, U.tok0 + kBlk))) break;
                if (walk.get(a, u + gridDim.x, Un) && !(ok = load_q(Un))) break;
                for (int j = 0; j < U.nb && ok; ++j) {
                    if (!(ok = load(&tv, hk, U.tok0 + j * kBlk))) break;
                    if (j + 2 < U.nb && !(ok = load(&tk, hk, U.tok0 + (j + 2) * kBlk))) break;
                }
            }
            // Every copy this thread issued lands before teardown.
            const uint64_t t0 = globaltimer_ns();
            for (uint32_t i = (it > kRing ? it - kRing : 0); i < it; ++i)
                while (!mbar_try_wait(smem_u32(&sh.full[i % kRing]), (i / kRing) & 1) && globaltimer_ns() - t0 < kWaitLimitNs) {}
            if (qc > 0)
                while (!mbar_try_wait(smem_u32(&sh.q_full), (qc - 1) & 1) && globaltimer_ns() - t0 < kWaitLimitNs) {}
        }
        __syncwarp();
    } else if (warp == 5) {
        // ---------------------------------------------------------- UMMA issuer
        uint32_t it = 0, uc = 0, gs = 0, gp = 0;   // ring slots taken; S and P V blocks so far
        bool ok = true;
        bool v_ready = false;   // the next V block's full wait already taken
        auto issue_s_block = [&](bool then_v) -> bool {
            const uint32_t ks = it % kRing;
            if (!mbar_wait_w(&sh.full[ks], (it / kRing) & 1, wc, k6KFull)) return false;
            ++it;
            if (then_v) {   // the next ring item is the V of the next P V
                if (!mbar_wait_w(&sh.full[it % kRing], (it / kRing) & 1, wc, k6VFull)) return false;
                v_ready = true;
            }
            tc_fence_after();
            issue_s(tmem + kColS + 64 * (gs & 1), tmem + kColQ, sR + ks * kKVBytes);
            umma_commit_w(&sh.s_full[gs & 1]);
            umma_commit_w(&sh.empty[ks]);
            ++gs;
            return true;
        };
        Walk256 walk;
        for (int u = blockIdx.x; ok; u += gridDim.x) {
            Unit256 U;
            if (!walk.get(a, u, U)) break;
            if (!(ok = mbar_wait_w(&sh.qt_full, uc & 1, wc, k6QFull))) break;
            tc_fence_after();
            if (!(ok = issue_s_block(false))) break;
            if (U.nb > 1 && !(ok = issue_s_block(false))) break;
            for (int j = 0; j < U.nb; ++j) {
                const uint32_t vs = it % kRing;
                if (!v_ready && !(ok = mbar_wait_w(&sh.full[vs], (it / kRing) & 1, wc, k6VFull))) break;
                v_ready = false;
                ++it;
                if (j == 0 && uc > 0 && !(ok = mbar_wait_w(&sh.o_free, (uc - 1) & 1, wc, k6OFree))) break;
                // P of block gp.  Two barriers, alternating: the softmax can
                // finish block gp + 1 (its S was issued above) before this
                // wait, never block gp + 2 (its S comes after this P V).
                if (!(ok = mbar_wait_w(&sh.p_ready[gp & 1], (gp >> 1) & 1, wc, k6P))) break;
                tc_fence_after();
                issue_pv(tmem + kColO, tmem + kColS + 64 * (gp & 1), sR + vs * kKVBytes, j > 0);
                umma_commit_w(&sh.empty[vs]);
                umma_commit_w(&sh.pv_done[gp & 1]);
                ++gp;
                // S of block j + 2 into the region P of block j was just read from.
                // V of block j + 1 directly follows K of block j + 2 in the ring.
                if (j + 2 < U.nb && !(ok = issue_s_block(true))) break;
            }
            if (!ok) break;
            umma_commit_w(&sh.o_done);
            ++uc;
        }
        umma_commit_w(&sh.drain);
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(smem_u32(&sh.drain), 0) && globaltimer_ns() - t0 < kWaitLimitNs) {}
        __syncwarp();
    } else {
        // ------------------------------------------------------------- softmax
        const int r = warp * 32 + lane;                       // query row in the tile == TMEM lane
        const uint32_t lane_bits = (uint32_t)(warp * 32) << 16;
        const uint32_t tO = tmem + lane_bits + kColO;
        const float scale = a.scale_log2;
        const bool o32 = (reinterpret_cast<uintptr_t>(a.o) & 31u) == 0;
        uint32_t gs = 0, uc = 0, qc = 0;
        bool ok = true;
        // This row of the next unit's Q tile, shared memory (128 B per row and
        // 64-column box, 16-byte chunks swizzled by row % 8) -> tensor memory
        // columns kColQ + 0..127 (bf16 pairs, the A operand of S).
        auto copy_q = [&]() -> bool {
            if (!mbar_wait(&sh.q_full, qc & 1, wc, k6QFull)) return false;
            ++qc;
#pragma unroll 1
            for (int b = 0; b < 4; ++b) {
                uint32_t v[32];
                const uint32_t row = sQ + b * kQBox + r * 128;
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(v[4 * c]), "=r"(v[4 * c + 1]), "=r"(v[4 * c + 2]), "=r"(v[4 * c + 3])
                                 : "r"(row + ((c ^ (r & 7)) << 4)) : "memory");
                tmem_st32(tmem + lane_bits + kColQ + 32 * b, v);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&sh.q_empty);
            mbar_arrive(&sh.qt_full);
            return true;
        };
        Walk256 walk;
        {
            Unit256 U;
            if (walk.get(a, blockIdx.x, U)) ok = copy_q();
        }
        for (int u = blockIdx.x; ok; u += gridDim.x) {
            Unit256 U, Un;
            if (!walk.get(a, u, U)) break;
            const int q_first = U.m * kTileM, qi = q_first + r;
            float m_ref = -INFINITY, l = 0.f;
            for (int j = 0; j < U.nb; ++j) {
                const uint32_t g = gs;   // this block's global index (S and P V alike)
                const uint32_t tS = tmem + lane_bits + kColS + 64 * (g & 1);
                if (!(ok = mbar_wait(&sh.s_full[g & 1], (g >> 1) & 1, wc, k6S))) break;
                ++gs;
                tc_fence_after();
                float s[kBlk];
                {
                    uint32_t* su = reinterpret_cast<uint32_t*>(s);
                    tmem_ld32(tS, *reinterpret_cast<uint32_t(*)[32]>(su));
                    tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(su + 32));
                    tmem_wait_ld();
                }
                const int k0 = j * kBlk;
                if (k0 + kBlk > U.len || (a.causal && k0 + kBlk - 1 > q_first)) {
                    const int lim_len = U.len - k0;
                    const int lim_causal = a.causal ? qi - k0 + 1 : kBlk;
                    const int lim = lim_len < lim_causal ? lim_len : lim_causal;
#pragma unroll
                    for (int c = 0; c < kBlk; ++c)
                        if (c >= lim) s[c] = -INFINITY;
                }
                // Row max: three-input max, four chains; exponents two at a
                // time (packed fp32 FMA) and the row sum in two packed
                // accumulators, as in the CTA-pair forward (large_d256 forward
                // 1587 -> 1655 TFLOP/s).
                float mx0 = fmaxf(s[0], s[1]), mx1 = fmaxf(s[2], s[3]), mx2 = fmaxf(s[4], s[5]),
                      mx3 = fmaxf(s[6], s[7]);
#pragma unroll
                for (int c = 8; c < kBlk; c += 8) {
                    mx0 = fmax3(mx0, s[c], s[c + 1]);
                    mx1 = fmax3(mx1, s[c + 2], s[c + 3]);
                    mx2 = fmax3(mx2, s[c + 4], s[c + 5]);
                    mx3 = fmax3(mx3, s[c + 6], s[c + 7]);
                }
                const float m_new = fmaxf(m_ref, fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * scale);
                // Conditional rescale (blog, "Forward pass"): move to the new
                // maximum only when some row of this warp jumped by more than tau.
                const bool jump = (m_ref == -INFINITY) ? (m_new != -INFINITY) : (m_new - m_ref > a.tau);
                const bool rescale = __any_sync(0xffffffffu, jump);
                if (kDbg && lane == 0) dbg_count_rescale(a.dbg_rescale, j > 0, rescale);
                if (rescale) {
                    const float fac = (m_ref == -INFINITY) ? 0.f : ex2_mufu(m_ref - m_new);
                    l *= fac;
                    if (j > 0) {
                        // O is touched only after the previous block's P V is
                        // done.  Its barrier (of two, alternating) has at that
                        // point completed every earlier phase -- S of block g-1,
                        // observed, was issued after P V g-3 -- and cannot have
                        // completed the next one (P V g+1 needs this block's P),
                        // so the parity identifies the phase.
                        if (!(ok = mbar_wait(&sh.pv_done[(g - 1) & 1], ((g - 1) >> 1) & 1, wc, k6PV))) break;
                        tc_fence_after();
#pragma unroll 1
                        for (int c0 = 0; c0 < kD; c0 += 32) {
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
                for (int st = 0; st < 2; ++st) {
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int c = st * 32 + 2 * i;
                        float x0, x1;
                        f2_unpack(f2_fma(f2_pack(s[c], s[c + 1]), sc2, nm2), x0, x1);
                        const float p0 = ex2_mufu(x0), p1 = ex2_mufu(x1);
                        if (i & 1) lb = f2_add(lb, f2_pack(p0, p1));
                        else la = f2_add(la, f2_pack(p0, p1));
                        pk[i] = pack_bf16x2(p0, p1);
                    }
                    tmem_st16(tS + st * 16, pk);   // P over the scores just read
                }
                {
                    float a0, a1, b0, b1;
                    f2_unpack(la, a0, a1);
                    f2_unpack(lb, b0, b1);
                    l += (a0 + a1) + (b0 + b1);
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&sh.p_ready[g & 1]);
            }
            if (!ok) break;
            // Every S of this unit has been read: its Q columns take the next tile.
            if (walk.get(a, u + gridDim.x, Un) && !(ok = copy_q())) break;
            // Epilogue: O / l -> bf16, LSE = (m + log2 l) ln 2.
            if (!(ok = mbar_wait(&sh.o_done, uc & 1, wc, k6O))) break;
            ++uc;
            tc_fence_after();
            const bool valid = qi < U.len;
            const float inv_l = l > 0.f ? 1.f / l : 0.f;
            uint4* orow = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.o) +
                                                   ((size_t)(U.tok0 + qi) * a.Hq + U.h) * kD);
#pragma unroll 1
            for (int c0 = 0; c0 < kD; c0 += 32) {
                uint32_t o[32];
                tmem_ld32(tO + c0, o);
                tmem_wait_ld();
                if (valid) {
                    if (o32) {   // whole 32-byte sectors
#pragma unroll
                        for (int q = 0; q < 2; ++q) {
                            const float* f = reinterpret_cast<const float*>(o + 16 * q);
                            uint32_t w[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) w[e] = pack_bf16x2(f[2 * e] * inv_l, f[2 * e + 1] * inv_l);
                            asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
                                         :: "l"(orow + c0 / 8 + 2 * q), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]),
                                            "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7]) : "memory");
                        }
                    } else {
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float* f = reinterpret_cast<const float*>(o + 8 * q);
                            orow[c0 / 8 + q] = make_uint4(pack_bf16x2(f[0] * inv_l, f[1] * inv_l), pack_bf16x2(f[2] * inv_l, f[3] * inv_l),
                                                          pack_bf16x2(f[4] * inv_l, f[5] * inv_l), pack_bf16x2(f[6] * inv_l, f[7] * inv_l));
                        }
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&sh.o_free);
            if (valid) {
                const size_t li = a.varlen ? (size_t)U.h * a.N + U.tok0 + qi     // [Hq, T]
                                           : ((size_t)U.seq * a.Hq + U.h) * a.N + qi;
                a.lse[li] = l > 0.f ? (m_ref + __log2f(l)) * 0.69314718055994531f : -INFINITY;
            }
            if (kDbg && r == 0 && q_first < U.len)
                dbg_count(a.dbg_visits, (long long)U.h * (a.varlen ? a.N : (long long)a.B * a.N) + U.tok0 + q_first);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

}  // namespace

cudaError_t launch_fwd256(const FwdLaunch& L, cudaStream_t stream) {
    const FwdArgs& a = L.a;
    // Varlen: sum over sequences of ceil(len / 128) <= ceil(T / 128) + B.
    const long long units = a.varlen ? (long long)a.Hq * ((a.N + kTileM - 1) / kTileM + a.B)
                                     : (long long)a.B * a.Hq * ((a.N + kTileM - 1) / kTileM);
    int grid = (int)(units < L.num_sms ? units : L.num_sms);
    if (grid < 1) grid = 1;
    auto kern = (a.dbg_visits || a.dbg_rescale) ? fwd256_kernel<true> : fwd256_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem256);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads256, kSmem256, stream>>>(L.tq, L.tk, L.tv, a);
    return cudaGetLastError();
}

}  // namespace fa
