// fa_fwd_wide.cu -- forward attention with 256-key S products (sm_103a).
//
// Same result as fa_fwd.cu's ping-pong kernel (O and LSE of exact attention,
// online softmax with the conditional rescale; FlashAttention-4 blog,
// "Forward pass"), shaped for GB300's tensor core: a 128x256x16 UMMA runs at
// the full rate while the 128x128x16 shape the ping-pong kernel's S product
// uses reaches about 60 % of it with shared-memory operands.  So each CTA
// works on one 128-row query tile and streams keys in blocks of 256:
//
//   S = Q K_j^T     128 x 256, operands in shared memory (N = 256)
//   O += P_j V_j    128 x 128, P read from tensor memory (K = 256)
//
// Tensor memory (512 columns): S cols 0-255 (fp32), P cols 256-383 (bf16,
// two per cell), O cols 384-511 (fp32).  P has its own columns, so the next
// S product starts as soon as the softmax has copied S_j into registers --
// it runs on the tensor core while the softmax exponentiates -- and P V
// follows when P is written.
//
// Warp roles (384 threads): warps 0-3 and 4-7 are two softmax warpgroups
// that split every row's 256 columns (one thread per row and half); they
// combine row maxima and sums through shared memory.  Warp 8 loads Q and K
// (TMA), warp 10 loads V, warp 9 issues the UMMAs, warp 11 idles.
//
// Fixed-length inputs only; packed variable-length batches use fa_fwd.cu.
#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kWThreads = 384;
constexpr int kBlockN = 256;                        // keys per block
constexpr uint32_t kQBytes = 32768;                 // 128 x 128 bf16
constexpr uint32_t kKVBytes = 65536;                // 256 x 128 bf16
constexpr uint32_t kQBox = 16384;                   // 128 rows x 64 bf16
constexpr uint32_t kKVBox = 32768;                  // 256 rows x 64 bf16
// K ring of two 64-KB slots (K(j+2) loads once S(j) is done, well before
// S(j+2)) and one V slot (V(j+1) loads once P V(j) is done).
constexpr int kKStages = 2;
constexpr uint32_t kOffQW = 0;
constexpr uint32_t kOffK = kQBytes;
constexpr uint32_t kOffVW = kOffK + kKStages * kKVBytes;
constexpr uint32_t kOffRed = kOffVW + kKVBytes;                // row max / sum exchange
constexpr uint32_t kOffWBar = kOffRed + 2 * 2 * 128 * 4;
constexpr uint32_t kWSmem = kOffWBar + 512;

constexpr uint32_t kColS = 0, kColP = 256, kColO = 384;

enum : int { kWSiteQEmpty = 41, kWSiteRingEmpty, kWSiteQFull, kWSiteRingFull, kWSiteSFree, kWSiteP, kWSiteOFree,
             kWSiteS, kWSitePV, kWSiteO };

struct WideShared {
    uint64_t q_full, q_empty;
    uint64_t kfull[kKStages], kempty[kKStages], vfull, vempty;
    uint64_t s_full, s_free, p_ready, pv_done, o_done, o_free, drain;
    uint32_t tmem_base;
    int abort_flag;
};
static_assert(sizeof(WideShared) <= 512, "barrier block");

struct WUnit {
    int seq, h, m, tok0, len;
};

// Unit order: non-causal (batch, head)-major with query tiles minor;
// causal longest-first (query tiles from the last) inside L2 sections of
// (batch, head) pairs (FlashAttention-4 blog, "Scheduling").
__device__ __forceinline__ bool wide_unit(const FwdArgs& a, int num_m, int u, WUnit& U) {
    const int BH = a.B * a.Hq;
    if (u >= BH * num_m) return false;
    int bh, m;
    if (!a.causal) {
        bh = u / num_m;
        m = u - bh * num_m;
    } else {
        const int sec = a.l2_section, per = sec * num_m, full = BH / sec;
        if (u < full * per) {
            const int s = u / per, r = u - s * per;
            m = num_m - 1 - r / sec;
            bh = s * sec + r % sec;
        } else {
            const int rem = BH - full * sec, r = u - full * per;
            m = num_m - 1 - r / rem;
            bh = full * sec + r % rem;
        }
    }
    U.seq = bh / a.Hq;
    U.h = bh - U.seq * a.Hq;
    U.m = m;
    U.tok0 = U.seq * a.N;
    U.len = a.N;
    return true;
}

// Key blocks a unit needs (causal: up to the tile's last row).
__device__ __forceinline__ int wide_blocks(const WUnit& U, int causal) {
    int keys = U.len;
    if (causal) {
        const int last = U.m * kTileM + kTileM;
        keys = last < keys ? last : keys;
    }
    return (keys + kBlockN - 1) / kBlockN;
}

// S = Q K^T: M = 128, N = 256, K = d = 128; both K-major, 128-B swizzle.
__device__ __forceinline__ void wide_qk(uint32_t d_tmem, uint32_t q_smem, uint32_t k_smem) {
    constexpr uint32_t idesc = idesc_bf16_f32(128, 256, 0, 0);
    const uint64_t qd = sdesc_sw128(q_smem, 16, 1024), kd = sdesc_sw128(k_smem, 16, 1024);
    static_for<8>([&](auto kc) {
        constexpr uint32_t k = kc;
        constexpr uint32_t qo = ((k >> 2) * kQBox + (k & 3) * 32) >> 4;
        constexpr uint32_t ko = ((k >> 2) * kKVBox + (k & 3) * 32) >> 4;
        umma_ss_k<qo, ko>(d_tmem, qd, kd, idesc, k > 0);
    });
}

// O (+)= P V: M = 128, N = d = 128, K = 256 keys; A = P from TMEM (8 columns
// per 16 keys), B = V MN-major (the second 64-wide d chunk 32 KB further).
__device__ __forceinline__ void wide_pv(uint32_t d_tmem, uint32_t p_tmem, uint32_t v_smem, uint32_t acc) {
    constexpr uint32_t idesc = idesc_bf16_f32(128, 128, 0, 1);
    const uint64_t vd = sdesc_sw128(v_smem, kKVBox, 1024);
    static_for<16>([&](auto kc) {
        constexpr uint32_t k = kc;
        umma_ts_k<k * 8, ((k * 2048) >> 4)>(d_tmem, p_tmem, vd, idesc, (acc | k) != 0);
    });
}

__device__ __forceinline__ bool wnamed_bar_or(int id, int n, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r) : "r"((uint32_t)pred), "r"(id), "r"(n) : "memory");
    return r != 0;
}

__global__ void __launch_bounds__(kWThreads, 1)
fwd_wide_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                const __grid_constant__ CUtensorMap tv, const FwdArgs a) {
    extern __shared__ __align__(1024) uint8_t dsm[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t base = smem_u32(dsm);
    if (base & 1023u) {  // the swizzled tiles need a 1024-byte aligned window
        if (tid == 0 && atomicCAS(&a.status->code, 0, -1) == 0) a.status->where = 400;
        return;
    }
    WideShared& sh = *reinterpret_cast<WideShared*>(dsm + kOffWBar);
    float* red = reinterpret_cast<float*>(dsm + kOffRed);   // [2 parity][2 halves][128 rows]
    const uint32_t sQ = base + kOffQW, sK = base + kOffK, sV = base + kOffVW;
    const int num_m = (a.N + kTileM - 1) / kTileM;

    if (tid == 0) {
        mbar_init(&sh.q_full, 1);
        mbar_init(&sh.q_empty, 1);
        for (int i = 0; i < kKStages; ++i) { mbar_init(&sh.kfull[i], 1); mbar_init(&sh.kempty[i], 1); }
        mbar_init(&sh.vfull, 1);
        mbar_init(&sh.vempty, 1);
        mbar_init(&sh.s_full, 1);
        mbar_init(&sh.s_free, 256);
        mbar_init(&sh.p_ready, 256);
        mbar_init(&sh.pv_done, 1);
        mbar_init(&sh.o_done, 1);
        mbar_init(&sh.o_free, 256);
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
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const WaitCtx wc{&sh.abort_flag, a.status};
    const uint32_t tmem = sh.tmem_base;
    const int group = a.Hq / a.Hkv;

    // Register split: 2 * 128 * 224 + 128 * 48 <= 384 * 168.
    if (warp >= 8) {
        regs_dec<48>();
        if (warp == 8) {
            // ------------------------------------------------------------ loader
            if (lane == 0) {
                uint32_t kit = 0, uc = 0;
                bool ok = true;
                auto load_k = [&](const WUnit& U, int hk, int j) -> bool {
                    const uint32_t slot = kit % kKStages;
                    if (!mbar_wait(&sh.kempty[slot], ((kit / kKStages) & 1) ^ 1, wc, kWSiteRingEmpty)) return false;
                    mbar_arrive_expect_tx(&sh.kfull[slot], kKVBytes);
                    for (int c = 0; c < 2; ++c)
                        tma_load_3d(sK + slot * kKVBytes + c * kKVBox, &tk, &sh.kfull[slot], c * 64, hk,
                                    U.tok0 + j * kBlockN);
                    ++kit;
                    return true;
                };
                for (int u = blockIdx.x; ok; u += gridDim.x) {
                    WUnit U;
                    if (!wide_unit(a, num_m, u, U)) break;
                    const int hk = U.h / group, nb = wide_blocks(U, a.causal);
                    if (!(ok = mbar_wait(&sh.q_empty, (uc & 1) ^ 1, wc, kWSiteQEmpty))) break;
                    mbar_arrive_expect_tx(&sh.q_full, kQBytes);
                    for (int c = 0; c < 2; ++c)
                        tma_load_3d(sQ + c * kQBox, &tq, &sh.q_full, c * 64, U.h, U.tok0 + U.m * kTileM);
                    for (int j = 0; j < nb && ok; ++j) ok = load_k(U, hk, j);
                    ++uc;
                }
                const uint64_t t0 = globaltimer_ns();  // drain this thread's copies
                for (uint32_t i2 = (kit > kKStages ? kit - kKStages : 0); i2 < kit; ++i2)
                    while (!mbar_try_wait(smem_u32(&sh.kfull[i2 % kKStages]), (i2 / kKStages) & 1) &&
                           globaltimer_ns() - t0 < kWaitLimitNs) {}
                if (uc > 0)
                    while (!mbar_try_wait(smem_u32(&sh.q_full), (uc - 1) & 1) && globaltimer_ns() - t0 < kWaitLimitNs) {}
            }
            __syncwarp();
        } else if (warp == 10) {
            // ---------------------------------------------------------- V loader
            // V(j+1) waits only for P V(j); K(j+2) (warp 8) only for S(j).
            if (lane == 0) {
                uint32_t vit = 0;
                bool ok = true;
                for (int u = blockIdx.x; ok; u += gridDim.x) {
                    WUnit U;
                    if (!wide_unit(a, num_m, u, U)) break;
                    const int hk = U.h / group, nb = wide_blocks(U, a.causal);
                    for (int j = 0; j < nb; ++j) {
                        if (!(ok = mbar_wait(&sh.vempty, (vit & 1) ^ 1, wc, kWSiteRingEmpty))) break;
                        mbar_arrive_expect_tx(&sh.vfull, kKVBytes);
                        for (int c = 0; c < 2; ++c)
                            tma_load_3d(sV + c * kKVBox, &tv, &sh.vfull, c * 64, hk, U.tok0 + j * kBlockN);
                        ++vit;
                    }
                }
                const uint64_t t0 = globaltimer_ns();
                if (vit > 0)
                    while (!mbar_try_wait(smem_u32(&sh.vfull), (vit - 1) & 1) && globaltimer_ns() - t0 < kWaitLimitNs) {}
            }
            __syncwarp();
        } else if (warp == 9) {
            // ------------------------------------------------------- UMMA issuer
            uint32_t kit = 0, vit = 0, uc = 0, gs = 0, gp = 0;   // K uses, V uses, units, S issued, PV issued
            bool ok = true;
            for (int u = blockIdx.x; ok; u += gridDim.x) {
                WUnit U;
                if (!wide_unit(a, num_m, u, U)) break;
                const int nb = wide_blocks(U, a.causal);
                if (!(ok = mbar_wait_w(&sh.q_full, uc & 1, wc, kWSiteQFull))) break;
                uint32_t kslot = kit % kKStages;
                if (!(ok = mbar_wait_w(&sh.kfull[kslot], (kit / kKStages) & 1, wc, kWSiteRingFull))) break;
                ++kit;
                tc_fence_after();
                wide_qk(tmem + kColS, sQ, sK + kslot * kKVBytes);
                umma_commit_w(&sh.s_full);
                umma_commit_w(&sh.kempty[kslot]);
                ++gs;
                for (int j = 0; j < nb; ++j) {
                    if (j + 1 < nb) {   // next S as soon as the softmax has copied this one out
                        kslot = kit % kKStages;
                        if (!(ok = mbar_wait_w(&sh.kfull[kslot], (kit / kKStages) & 1, wc, kWSiteRingFull))) break;
                        ++kit;
                        if (!(ok = mbar_wait_w(&sh.s_free, (gs - 1) & 1, wc, kWSiteSFree))) break;
                        tc_fence_after();
                        wide_qk(tmem + kColS, sQ, sK + kslot * kKVBytes);
                        umma_commit_w(&sh.s_full);
                        umma_commit_w(&sh.kempty[kslot]);
                        ++gs;
                    }
                    if (!(ok = mbar_wait_w(&sh.vfull, vit & 1, wc, kWSiteRingFull))) break;
                    ++vit;
                    if (j == 0 && !(ok = mbar_wait_w(&sh.o_free, (uc & 1) ^ 1, wc, kWSiteOFree))) break;
                    if (!(ok = mbar_wait_w(&sh.p_ready, gp & 1, wc, kWSiteP))) break;
                    tc_fence_after();
                    wide_pv(tmem + kColO, tmem + kColP, sV, j > 0);
                    umma_commit_w(&sh.pv_done);
                    umma_commit_w(&sh.vempty);
                    ++gp;
                }
                umma_commit_w(&sh.o_done);
                umma_commit_w(&sh.q_empty);
                ++uc;
            }
            umma_commit_w(&sh.drain);
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
        const uint32_t tS = tmem + lb + kColS + x * 128;     // this half's 128 S columns
        const uint32_t tP = tmem + lb + kColP + x * 64;      // its 64 P columns (bf16 pairs)
        const uint32_t tO = tmem + lb + kColO + x * 64;      // its 64 O columns
        const float scale = a.scale_log2;
        uint32_t sc = 0, pc = 0, uc = 0;
        uint32_t ep = 0;   // barrier epoch: exchange buffers alternate with it
        bool ok = true;
        for (int u = blockIdx.x; ok; u += gridDim.x) {
            WUnit U;
            if (!wide_unit(a, num_m, u, U)) break;
            const int nb = wide_blocks(U, a.causal);
            const int qi = U.m * kTileM + r;
            float m_ref = -INFINITY, l = 0.f;           // l: this half's partial row sum
            // The halves meet at named barriers: a wait that gives up does not
            // leave the loop on its own; both halves leave at the next barrier.
            bool okw = true;
            for (int j = 0; j < nb; ++j) {
                okw = mbar_wait(&sh.s_full, sc & 1, wc, kWSiteS) && okw;
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
                mbar_arrive(&sh.s_free);                // the next S may overwrite these columns
                const int k0 = j * kBlockN + x * 128;   // key of column 0 of this half
                if (k0 + 128 > U.len || (a.causal && k0 + 127 > U.m * kTileM)) {
                    const int lim_len = U.len - k0;
                    const int lim_causal = a.causal ? qi - k0 + 1 : 128;
                    const int lim = lim_len < lim_causal ? lim_len : lim_causal;
#pragma unroll
                    for (int c = 0; c < 128; ++c)
                        if (c >= lim) s[c] = -INFINITY;
                }
                float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
                for (int c = 4; c < 128; c += 4) {
                    mx0 = fmaxf(mx0, s[c]);
                    mx1 = fmaxf(mx1, s[c + 1]);
                    mx2 = fmaxf(mx2, s[c + 2]);
                    mx3 = fmaxf(mx3, s[c + 3]);
                }
                float* rb = red + (ep & 1) * 256;
                rb[x * 128 + r] = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));
                ++ep;
                if (wnamed_bar_or(2, 256, !okw)) { ok = false; break; }
                const float m_blk = fmaxf(rb[r], rb[128 + r]) * scale;   // whole-row max, log2 units
                const float m_new = fmaxf(m_ref, m_blk);
                // Conditional rescale (paper summary §3.1.4): both halves see
                // the same row maxima, so their warp votes agree.
                const bool jump = (m_ref == -INFINITY) ? (m_new != -INFINITY) : (m_new - m_ref > a.tau);
                const bool rescale = __any_sync(0xffffffffu, jump);
                float fac = 1.f;
                if (rescale) {
                    fac = (m_ref == -INFINITY) ? 0.f : ex2_mufu(m_ref - m_new);
                    l *= fac;
                    m_ref = m_new;
                }
                const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
                uint32_t pk[64];
                float l0 = 0.f, l1 = 0.f;
#pragma unroll
                for (int i = 0; i < 64; ++i) {
                    const float p0 = ex2_mufu(fmaf(s[2 * i], scale, -m_use));
                    const float p1 = ex2_mufu(fmaf(s[2 * i + 1], scale, -m_use));
                    l0 += p0;
                    l1 += p1;
                    pk[i] = pack_bf16x2(p0, p1);
                }
                l += l0 + l1;
                // P's columns and O are free once the previous P V is done.
                if (j > 0) {
                    okw = mbar_wait(&sh.pv_done, pc & 1, wc, kWSitePV) && okw;
                    ++pc;
                    tc_fence_after();
                    if (rescale) {
#pragma unroll
                        for (int c0 = 0; c0 < 64; c0 += 32) {
                            uint32_t o[32];
                            tmem_ld32(tO + c0, o);
                            tmem_wait_ld();
#pragma unroll
                            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * fac);
                            tmem_st32(tO + c0, o);
                        }
                    }
                }
#pragma unroll
                for (int st = 0; st < 4; ++st)
                    tmem_st16(tP + st * 16, *reinterpret_cast<const uint32_t(*)[16]>(pk + st * 16));
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&sh.p_ready);
            }
            if (!ok) break;
            okw = mbar_wait(&sh.o_done, uc & 1, wc, kWSiteO) && okw;
            ++uc;
            // The last P V of the unit is done: account for its pv_done phase.
            if (nb > 0) ++pc;
            tc_fence_after();
            // Epilogue: whole-row sum from the two halves, O / l, LSE.
            float* rl = red + (ep & 1) * 256;
            rl[x * 128 + r] = l;
            ++ep;
            if (wnamed_bar_or(2, 256, !okw)) { ok = false; break; }
            const float lt = rl[r] + rl[128 + r];
            const bool valid = qi < U.len;
            const float inv_l = lt > 0.f ? 1.f / lt : 0.f;
            uint4* orow = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.o) +
                                                   ((size_t)(U.tok0 + qi) * a.Hq + U.h) * kHeadDim + x * 64);
#pragma unroll
            for (int c0 = 0; c0 < 64; c0 += 32) {
                uint32_t o[32];
                tmem_ld32(tO + c0, o);
                tmem_wait_ld();
                if (valid) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float* f = reinterpret_cast<const float*>(o + 8 * q);
                        orow[c0 / 8 + q] = make_uint4(pack_bf16x2(f[0] * inv_l, f[1] * inv_l),
                                                      pack_bf16x2(f[2] * inv_l, f[3] * inv_l),
                                                      pack_bf16x2(f[4] * inv_l, f[5] * inv_l),
                                                      pack_bf16x2(f[6] * inv_l, f[7] * inv_l));
                    }
                }
            }
            if (valid && x == 0)
                a.lse[((size_t)U.seq * a.Hq + U.h) * a.N + qi] =
                    lt > 0.f ? (m_ref + __log2f(lt)) * 0.69314718055994531f : -INFINITY;
            tc_fence_before();
            mbar_arrive(&sh.o_free);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

}  // namespace

cudaError_t launch_fwd_wide(const FwdLaunch& L, cudaStream_t stream) {
    const long long units = (long long)L.a.B * L.a.Hq * ((L.a.N + kTileM - 1) / kTileM);
    int grid = (int)(units < L.num_sms ? units : L.num_sms);
    if (grid < 1) grid = 1;
    cudaError_t e = cudaFuncSetAttribute(fwd_wide_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kWSmem);
    if (e != cudaSuccess) return e;
    fwd_wide_kernel<<<grid, kWThreads, kWSmem, stream>>>(L.tq, L.tk, L.tv, L.a);
    return cudaGetLastError();
}

}  // namespace fa
