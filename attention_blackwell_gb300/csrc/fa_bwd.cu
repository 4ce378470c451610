// fa_bwd.cu -- backward attention for sm_103a (tcgen05 / TMEM / TMA).
//
// Gradients of O = softmax(alpha Q K^T [+ causal]) V for d = 128 or 64
// (FlashAttention-4 blog, "Backward pass" section): with upstream dO,
//   D_i = sum_d dO_id O_id,  P = exp(alpha Q K^T - LSE),
//   dV = P^T dO,  dP = dO V^T,  dS = P * (dP - D),
//   dK = alpha dS^T Q,  dQ = alpha dS K.
//
// Three stages on the caller's stream:
//   1. preprocess: D (one warp per query row and head), dQacc := 0,
//      semaphores := 0, and for varlen a work list in longest-first order;
//   2. main kernel: one persistent CTA per SM, claiming work units in list
//      order from a global counter as it frees up; a work unit is one 128-key
//      tile of one (sequence, key/value head); the CTA keeps K, V and the dK,
//      dV accumulators resident and streams the query tiles of every query
//      head of the group.  It recomputes S and P transposed (keys on the
//      TMEM lanes) so that P^T sits in TMEM exactly as operand A of the dV
//      product (FlashAttention-4 blog, "Backward pass": transposed
//      recompute, P^T/dS^T resident as operand A), runs the five UMMAs per
//      tile and adds dQ into an fp32 accumulator in global memory with
//      vector reductions -- in a fixed order behind per-tile semaphores in
//      deterministic mode (blog, "Deterministic mode");
//   3. postprocess: dq = bf16(alpha * dQacc).
#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kLevelsMax = 1024;  // key-tile levels of the varlen plan (max_seqlen <= 131072)

__device__ __forceinline__ float bf16lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

// ---------------------------------------------------------------- stage 1

// Per lane of a warp on one row of D elements: D / 32 consecutive elements.
template <int D> struct LaneVec;
struct float8v { float4 lo, hi; };
template <> struct LaneVec<256> { using bf = uint4; using f = float8v; };
template <> struct LaneVec<128> { using bf = uint2; using f = float4; };
template <> struct LaneVec<64> { using bf = uint32_t; using f = float2; };

__device__ __forceinline__ float dot_bf16(uint2 a, uint2 b) {
    return bf16lo(a.x) * bf16lo(b.x) + bf16hi(a.x) * bf16hi(b.x) + bf16lo(a.y) * bf16lo(b.y) + bf16hi(a.y) * bf16hi(b.y);
}
__device__ __forceinline__ float dot_bf16(uint32_t a, uint32_t b) {
    return bf16lo(a) * bf16lo(b) + bf16hi(a) * bf16hi(b);
}
__device__ __forceinline__ float dot_bf16(uint4 a, uint4 b) {
    return dot_bf16(make_uint2(a.x, a.y), make_uint2(b.x, b.y)) + dot_bf16(make_uint2(a.z, a.w), make_uint2(b.z, b.w));
}
__device__ __forceinline__ void zero_vec(float8v& v) {
    v.lo = make_float4(0.f, 0.f, 0.f, 0.f);
    v.hi = v.lo;
}
__device__ __forceinline__ void zero_vec(float4& v) { v = make_float4(0.f, 0.f, 0.f, 0.f); }
__device__ __forceinline__ void zero_vec(float2& v) { v = make_float2(0.f, 0.f); }
__device__ __forceinline__ uint2 pack_scaled(float4 g, float s) {
    return make_uint2(pack_bf16x2(g.x * s, g.y * s), pack_bf16x2(g.z * s, g.w * s));
}
__device__ __forceinline__ uint32_t pack_scaled(float2 g, float s) { return pack_bf16x2(g.x * s, g.y * s); }
__device__ __forceinline__ uint4 pack_scaled(float8v g, float s) {
    const uint2 a = pack_scaled(g.lo, s), b = pack_scaled(g.hi, s);
    return make_uint4(a.x, a.y, b.x, b.y);
}

template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const BwdArgs a) {
    // One warp per (token, head) row, four consecutive rows (4 D bf16 of O and
    // of dO) per step with all eight loads issued before any is used.
    using BV = typename LaneVec<D>::bf;
    using FV = typename LaneVec<D>::f;
    const int lane = threadIdx.x & 31;
    const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
    const long long rows = a.T * a.Hq;
    const BV* o2 = reinterpret_cast<const BV*>(a.o);
    const BV* d2 = reinterpret_cast<const BV*>(a.dO);
    for (long long w0 = (((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5) * 4; w0 < rows; w0 += nwarps * 4) {
        BV ov[4], dv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const long long w = w0 + e < rows ? w0 + e : rows - 1;
            ov[e] = o2[w * 32 + lane];
            dv[e] = d2[w * 32 + lane];
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const long long w = w0 + e;
            float s = dot_bf16(ov[e], dv[e]);
#pragma unroll
            for (int m = 16; m > 0; m >>= 1) s += __shfl_xor_sync(0xffffffffu, s, m);
            if (w < rows) {
                const long long tok = w / a.Hq;
                const int h = (int)(w - tok * a.Hq);
                const size_t r = (size_t)h * a.T + tok;
                if (lane == 0) a.D[r] = s;
                FV z;
                zero_vec(z);
                reinterpret_cast<FV*>(a.dqacc + r * D)[lane] = z;
            }
        }
    }
    if (a.kv_split) {        // the fp32 dK / dV partial sums of split units
        const long long n = 2LL * a.Hkv * a.T * D / 4;
        float4* z4 = reinterpret_cast<float4*>(a.dkvacc);
        for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
             i += (long long)gridDim.x * blockDim.x)
            z4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (a.deterministic) {   // d = 256: one set per head-dim half
        const long long n = (D == 256 ? 2LL : 1LL) * a.Hq * a.sem_stride;
        for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
             i += (long long)gridDim.x * blockDim.x)
            a.sem[i] = 0;
    }
}

// Varlen work list: units (sequence, key/value head, key tile k), the most
// expensive first, so that CTAs claiming them in list order finish close
// together (longest-processing-time-first).  A unit streams every query tile
// its key tile sees, times the group's query heads, so its cost is set by
// the number of those query tiles: nk - k under a causal mask, nk without
// (nk = the sequence's tile count).
//   causal: level L holds the units that see c = maxk - L query tiles: one
//     per sequence with at least c tiles and key/value head, the shortest
//     sequence first -- which lists each sequence's key tiles in ascending
//     order, the order the deterministic semaphores need;
//   non-causal: level L is sequence order[L] (longest first), key/value
//     head major, key tiles ascending (the heads' Q and dO stay in L2 while
//     their key tiles run).
// The naive order (fa_set_schedule_order) lists every call like the
// non-causal one, with the sequences in index order.
// Split units (kv_split query heads each, atomic mode, groups of at least
// kSplitMinGroup query heads): sequence-major (longest first), then
// key/value head, head group, key tiles ascending, so that the CTAs of a wave
// share one group's rows of Q, dO and the fp32 dQ accumulator and their
// reductions hit L2; each unit adds its partial dK and dV into fp32 sums.
// kt: keys per unit, 128
// (one CTA per key tile) or 256 (the CTA-pair kernel's key blocks); the
// header records it, so that a main kernel never reads a list built for the
// other.  One CTA of 1024 threads.
__global__ void __launch_bounds__(1024) bwd_plan_kernel(const BwdArgs a, int kt) {
    __shared__ int s_cu[kMaxVarlenSeqs + 1], s_order[kMaxVarlenSeqs], s_pref[kLevelsMax + 1], s_cnt[kLevelsMax];
    __shared__ int s_maxk, s_levels;
    const int tid = threadIdx.x, B = a.B;
    for (int i = tid; i <= B; i += blockDim.x) {
        const int c = a.cu_seqlens[i];
        s_cu[i] = c < 0 ? 0 : (c > a.N ? a.N : c);
    }
    __syncthreads();
    if (tid == 0)
        for (int i = 1; i <= B; ++i) s_cu[i] = s_cu[i] > s_cu[i - 1] ? s_cu[i] : s_cu[i - 1];
    __syncthreads();
    // The main kernel reads the units' bounds from this copy, so that plan
    // and main kernel agree on every sequence whatever the offsets were.
    for (int i = tid; i <= B; i += blockDim.x) a.cu_s[i] = s_cu[i];
    auto nkv = [&](int s) { return (s_cu[s + 1] - s_cu[s] + kt - 1) / kt; };
    for (int i = tid; i < B; i += blockDim.x) {
        const int ni = nkv(i);
        int rank = 0;
        if (!a.naive)
            for (int j = 0; j < B; ++j) {
                const int nj = nkv(j);
                rank += (nj > ni) || (nj == ni && j < i);
            }
        s_order[a.naive ? i : rank] = i;   // tile count descending, index ascending among equals
    }
    __syncthreads();
    const int gs = a.kv_split, ng = gs ? (a.Hq / a.Hkv) / gs : 1;   // query heads, groups per unit
    const bool levels_by_cost = a.causal && !a.naive && !gs;
    if (tid == 0) {
        int maxk = 0;
        for (int i = 0; i < B; ++i) maxk = nkv(i) > maxk ? nkv(i) : maxk;
        if (maxk > kLevelsMax) {
            if (atomicCAS(&a.hdr->status.code, 0, -1) == 0) a.hdr->status.where = 200;
            maxk = 0;
        }
        int acc = 0, levels;
        if (levels_by_cost) {
            int p = 0;
            for (int L = 0; L < maxk; ++L) {
                while (p < B && nkv(s_order[p]) >= maxk - L) ++p;   // sequences with >= c tiles
                s_cnt[L] = p;
                s_pref[L] = acc;
                acc += p * a.Hkv;
            }
            levels = maxk;
        } else {
            levels = maxk > 0 ? B : 0;
            for (int L = 0; L < levels; ++L) {
                s_pref[L] = acc;
                acc += nkv(s_order[L]) * a.Hkv * ng;
            }
        }
        s_pref[levels] = acc;
        s_maxk = maxk;
        s_levels = levels;
        a.hdr->total_units = acc;
        a.hdr->unit_keys = kt;
        a.hdr->unit_heads = gs;
    }
    __syncthreads();
    const int maxk = s_maxk, levels = s_levels, total = s_pref[levels];
    for (int u = tid; u < total; u += blockDim.x) {
        int lo = 0, hi = levels;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (s_pref[mid + 1] > u) hi = mid; else lo = mid + 1;
        }
        const int r = u - s_pref[lo];
        int seq, hk, k, grp = 0;
        if (levels_by_cost) {
            seq = s_order[s_cnt[lo] - 1 - r / a.Hkv];
            hk = r % a.Hkv;
            k = nkv(seq) - (maxk - lo);
        } else {
            seq = s_order[lo];
            const int nk = nkv(seq);
            hk = r / (nk * ng);
            const int r2 = r - hk * nk * ng;
            grp = r2 / nk;
            k = r2 - grp * nk;
        }
        a.units[u] = make_int4(seq, hk, k, grp);
    }
}

// ---------------------------------------------------------------- stage 3

template <int D>
__global__ void __launch_bounds__(256) bwd_post_kernel(const BwdArgs a) {
    using BV = typename LaneVec<D>::bf;
    using FV = typename LaneVec<D>::f;
    const int lane = threadIdx.x & 31;
    const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
    const long long rows = a.T * a.Hq;
    // Four rows per warp and step, all loads issued first.
    for (long long w0 = (((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5) * 4; w0 < rows; w0 += nwarps * 4) {
        FV g[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {   // rows of dQacc in its own (head, token) order
            const long long w = w0 + e < rows ? w0 + e : rows - 1;
            g[e] = reinterpret_cast<const FV*>(a.dqacc + (size_t)w * D)[lane];
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const long long w = w0 + e;
            if (w < rows) {
                const long long h = w / a.T, tok = w - h * a.T;
                reinterpret_cast<BV*>(a.dq)[(tok * a.Hq + h) * 32 + lane] = pack_scaled(g[e], a.alpha);
            }
        }
    }
    if (a.kv_split) {   // split units: dK = bf16(alpha sum), dV = bf16(sum) of the fp32 partial sums
        const long long kvrows = a.T * a.Hkv;   // rows per accumulator, (key/value head, token) order
        // Only the sequences' rows: the sanitised sequences tile [cu_s[0], cu_s[B]).
        const long long c_lo = a.cu_s[0], c_hi = a.cu_s[a.B];
        for (long long w0 = (((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5) * 4; w0 < 2 * kvrows;
             w0 += nwarps * 4) {
            FV g[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const long long w = w0 + e < 2 * kvrows ? w0 + e : 2 * kvrows - 1;
                g[e] = reinterpret_cast<const FV*>(a.dkvacc + (size_t)w * D)[lane];
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const long long w = w0 + e;
                if (w < 2 * kvrows) {
                    const int which = w >= kvrows;
                    const long long rem = w - which * kvrows, hk = rem / a.T, tok = rem - hk * a.T;
                    if (tok >= c_lo && tok < c_hi)
                        reinterpret_cast<BV*>(which ? a.dv : a.dk)[(tok * a.Hkv + hk) * 32 + lane] =
                            pack_scaled(g[e], which ? 1.f : a.alpha);
                }
            }
        }
    }
}

// ---------------------------------------------------------------- stage 2
//
// Warp roles (384 threads):
//   warps 0-3   "softmax" warpgroup, one thread per KEY row (TMEM lane):
//               P^T = 2^(alpha log2e S^T - LSE log2e) -> bf16 into TMEM
//               (operand A of dV += P^T dO); dS^T = P^T (dP^T - D) -> bf16
//               into shared memory in the 128-B swizzled key-major layout,
//               which the dQ UMMA reads as an MN-major A, and also into TMEM
//               as operand A of dK += dS^T Q (at d = 128 beside the dP^T it
//               was computed from, at d = 64 in columns 64-127, which the
//               64-column accumulators leave free);
//   warps 4-7   dQ warpgroup, one thread per QUERY row: drains dQ_i from TMEM
//               into the fp32 accumulator (vector reductions), then at the end
//               of a unit stores dK (x alpha) and dV in bf16;
//   warp  8     loader: K, V once per unit (TMA), then Q_i, dO_i (TMA) and
//               LSE_i, D_i (plain loads) into a two-stage ring;
//   warp  9     issues dV, dQ, dK, dP (and, at d = 128, S);  warp 10 issues S
//               at d = 64;  warp 11 idle.
//
// Tensor memory (512 columns): dK acc 0-127, dV acc 128-255 (d columns used;
//   at d = 64 columns 64-127 hold dS^T, bf16, queries 0-63 in 64-95 and
//   64-127 in 96-127),
//   R0 256-383: S^T, then P^T (bf16; each key-row half packs its 64 queries
//               into the first 32 of the 64 columns it read);
//   R1 384-511: dP^T, then at d = 128 dS^T (bf16, packed like P^T in R0),
//               then dQ_i (d columns) once dK has read dS^T (issued first by
//               the same thread) -- the paper's 1-CTA sharing of dP/dS/dQ
//               columns.  Taking dK's A operand from TMEM saves 32 KB of the
//               ~512 KB of shared-memory traffic per tile that bounds the
//               kernel (headline backward 1183 -> 1196 TFLOP/s, bitwise the
//               same gradients; at d = 64 large_d64 782 -> 787).
// The next tile's S^T is computed while this tile's dS is (FlashAttention-4
// blog, "Backward pass": the next tile's products overlap the elementwise
// work).  At d = 128 one thread issues every product: dV(j), then S^T(j+1)
// right behind it (S^T overwrites the R0 columns dV reads P^T from; one
// thread's products run in issue order, so it need not wait for dV to
// complete), then dK(j), so that Q's stage frees early for the copy two
// tiles ahead, then dQ(j) and the next dP.  At d = 64, where the products
// are short and the exponentials set the pace, warp 10 issues each S^T once
// its Q tile is loaded and dV has completed, and warp 9 issues dV, dQ, dK and
// the next dP, dQ before dK so that the hand-off of dQ out of R1 (which the
// next dP waits for) overlaps the dK product (each order measured faster for
// its head dim).
//
// Shared memory (dynamic, 1024-aligned; 232448 bytes at d = 128), a tile
// being 128 rows x d bf16 (32K at d = 128, 16K at d = 64):
//   K | V | Q[2] | dO | dS 32K | dQ staging 32K | lse2[2][128], D[2][128] | barriers
// dO is single-buffered: it is free once dV has read it and is next needed
// by dP of the next tile, after S, dQ, dK and the dQ hand-off.
constexpr int kBwdThreads = 512;
constexpr uint32_t kBox = 16384;                        // one TMA box: 128 rows x 128 bytes
template <int D> struct BGeo {
    static_assert(D == 64 || D == 128, "head dim");
    static constexpr int kBoxes = D / 64;               // boxes per Q, K, V or dO tile
    static constexpr uint32_t kTile = 256u * D;         // 128 rows x D bf16
    static constexpr uint32_t kOffK = 0, kOffV = kTile, kOffQ = 2 * kTile, kOffDO = 4 * kTile, kOffDS = 5 * kTile;
    static constexpr uint32_t kOffStage = kOffDS + 32768;   // dQ staging for the TMA reductions
    static constexpr uint32_t kOffStat = kOffStage + 32768; // lse2[2][128], D[2][128] floats
    static constexpr uint32_t kOffBar = kOffStat + 4 * 128 * 4;
    static constexpr uint32_t kSmem = kOffBar + 1024;
};
static_assert(BGeo<128>::kSmem == 232448, "shared memory plan");

struct BwdShared {
    uint64_t kv_full, kv_empty, q_full[2], q_empty[2], do_full, do_empty;
    uint64_t s_full, dp_full, p_ready, ds_ready, ds_free, dq_full, dq_free, dkdv_done, acc_free, drain, r0_free;
    uint64_t unit_full[4], unit_empty[4];   // ring of claimed unit indices
    int unit_id[4];
    uint32_t tmem_base;
    int abort_flag;
    int total;
};
static_assert(sizeof(BwdShared) <= 1024, "barrier block");

constexpr uint32_t kColDK = 0, kColDV = 128, kColR0 = 256, kColR1 = 384;
constexpr uint32_t kColDS64 = 64;   // dS^T at d = 64 (past the 64-column dK)

enum : int { kBSiteKvEmpty = 11, kBSiteQEmpty, kBSiteKvFull, kBSiteAcc, kBSiteQFull, kBSiteP, kBSiteDs,
             kBSiteDqFree, kBSiteS, kBSiteDp, kBSiteDsFree, kBSiteDq, kBSiteDkdv, kBSiteSem, kBSiteUnit };

// One thread issues every product at d = 128, two at d = 64 (see above).
template <int D> constexpr int kIssuers = D == 128 ? 1 : 2;

// Readers of each claimed unit index: the issuer warps (one arrival each),
// the 256 key-row threads and the 128 dQ threads.
template <int D> constexpr uint32_t kUnitReaders = kIssuers<D> + 256 + 128;

struct BUnit {
    int seq, hk, k, tok0, len, n, nq, i0;
    int h0;   // first query head of the unit within its key/value head's group
};

// Decode unit u.  Fixed length, non-causal, atomic mode: (sequence,
// key/value head) major, key tiles ascending within it, so the CTAs at work
// at any time share a few heads and those heads' Q, dO and fp32 dQ
// accumulator stay in L2 (FlashAttention-4 blog, "Scheduling": L2-sized
// batch-head sections).  Fixed length otherwise: key tile k = u / (B*Hkv),
// all first key tiles before any second one -- longest first under a causal
// mask, and in deterministic mode a key tile waits at its semaphores only on
// tiles that are already claimed.  Both orders put every unit after the
// ones it waits on, and CTAs claim units in list order, so the earliest
// unfinished unit always runs.  The naive order (fa_set_schedule_order) is
// head-major with key tiles ascending in every mode, which also lists a
// unit after those it waits on.  Varlen: the planned work list (a split
// unit covers kv_split query heads from its group's h0).  u < 0 is
// the end of the list.
__device__ __forceinline__ bool bwd_unit(const BwdArgs& a, int total, int u, BUnit& U) {
    if (u < 0 || u >= total) return false;
    if (!a.varlen) {
        const int bh = a.B * a.Hkv;
        int r;
        if ((a.deterministic || a.causal) && !a.naive) {
            U.k = u / bh;
            r = u - U.k * bh;
        } else {
            const int nk = (a.N + kTileN - 1) / kTileN;
            r = u / nk;
            U.k = u - r * nk;
        }
        U.seq = r / a.Hkv;
        U.hk = r - U.seq * a.Hkv;
        U.tok0 = U.seq * a.N;
        U.len = a.N;
        U.h0 = 0;
    } else {
        const int4 e = a.units[u];
        U.seq = e.x;
        U.hk = e.y;
        U.k = e.z;
        U.h0 = e.w * a.kv_split;        // head group (split units), else 0
        const int c0 = a.cu_s[U.seq];   // sanitised by the plan kernel
        U.tok0 = c0;
        U.len = a.cu_s[U.seq + 1] - c0;
    }
    U.nq = (U.len + kTileM - 1) / kTileM;
    U.i0 = a.causal ? U.k : 0;
    U.n = (a.varlen && a.kv_split ? a.kv_split : a.Hq / a.Hkv) * (U.nq - U.i0);
    return true;
}

// A 128x128 product over the head dim (D / 16 steps) with both operands
// K-major in shared memory (S^T = K Q^T and dP^T = V dO^T).
template <int D>
__device__ __forceinline__ void mma_kk(uint32_t d, uint32_t a_smem, uint32_t b_smem) {
    constexpr uint32_t idesc = idesc_bf16_f32(128, 128, 0, 0);
    const uint64_t ad = sdesc_sw128(a_smem, 16, 1024), bd = sdesc_sw128(b_smem, 16, 1024);
    static_for<D / 16>([&](auto kc) {
        constexpr uint32_t k = kc, off = ((k >> 2) * kBox + (k & 3) * 32) >> 4;
        umma_ss_k<off, off>(d, ad, bd, idesc, k > 0);
    });
}

// D (+)= A[tmem] B, B MN-major in shared memory (dV += P^T dO, and at
// d = 128 dK += dS^T Q).  A is bf16 in the region the two key-row halves
// wrote: queries 0-63 in columns 0-31 of the region, queries 64-127 in
// columns 64-95 (each half packs its 64 queries at the start of the 64
// columns it read).  N = D.
template <int D>
__device__ __forceinline__ void mma_tn(uint32_t d, uint32_t a_tmem, uint32_t b_smem, uint32_t acc) {
    constexpr uint32_t idesc = idesc_bf16_f32(128, D, 0, 1);
    const uint64_t bd = sdesc_sw128(b_smem, kBox, 1024);
    static_for<8>([&](auto kc) {
        constexpr uint32_t k = kc, col = k * 8 + (k >= 4 ? 32 : 0);
        umma_ts_k<col, ((k * 2048) >> 4)>(d, a_tmem, bd, idesc, (acc | k) != 0);
    });
}

// The same with A's queries in consecutive columns (dK += dS^T Q at d = 64,
// dS^T in the columns the 64-column accumulators leave free).
template <int D>
__device__ __forceinline__ void mma_tl(uint32_t d, uint32_t a_tmem, uint32_t b_smem, uint32_t acc) {
    constexpr uint32_t idesc = idesc_bf16_f32(128, D, 0, 1);
    const uint64_t bd = sdesc_sw128(b_smem, kBox, 1024);
    static_for<8>([&](auto kc) {
        constexpr uint32_t k = kc, col = k * 8;
        umma_ts_k<col, ((k * 2048) >> 4)>(d, a_tmem, bd, idesc, (acc | k) != 0);
    });
}

// D = A B with A and B both MN-major in shared memory (dQ = dS K: dS^T is
// stored key-major, i.e. queries contiguous = M contiguous).  N = D.
template <int D>
__device__ __forceinline__ void mma_nn(uint32_t d, uint32_t a_smem, uint32_t b_smem) {
    constexpr uint32_t idesc = idesc_bf16_f32(128, D, 1, 1);
    const uint64_t ad = sdesc_sw128(a_smem, kBox, 1024), bd = sdesc_sw128(b_smem, kBox, 1024);
    static_for<8>([&](auto kc) {
        constexpr uint32_t k = kc, off = (k * 2048) >> 4;
        umma_ss_k<off, off>(d, ad, bd, idesc, k > 0);
    });
}

__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// TMA bulk tensor reduction: global[tile at (x, y)] += shared tile (fp32 add).
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
    asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3}], [%1];"
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(src), "r"(x), "r"(y) : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ void named_bar(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Named barrier that also ORs a predicate over its threads (uniform result).
__device__ __forceinline__ bool named_bar_or(int id, int n, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r) : "r"((uint32_t)pred), "r"(id), "r"(n) : "memory");
    return r != 0;
}

__device__ __forceinline__ int ld_acquire(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void red_release_add(int* p, int v) {
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
bwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
           const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
           const __grid_constant__ CUtensorMap tdq, const __grid_constant__ CUtensorMap tdkv, const BwdArgs a) {
    extern __shared__ __align__(1024) uint8_t dsm[];
    using G = BGeo<D>;
    constexpr uint32_t kOffK = G::kOffK, kOffV = G::kOffV, kOffQ = G::kOffQ, kOffDO = G::kOffDO, kOffDS = G::kOffDS,
                       kOffStage = G::kOffStage, kOffStat = G::kOffStat, kOffBar = G::kOffBar, kT32 = G::kTile;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t base = smem_u32(dsm);
    if (base & 1023u) {  // the swizzled tiles need a 1024-byte aligned window
        if (tid == 0 && atomicCAS(&a.hdr->status.code, 0, -1) == 0) a.hdr->status.where = 300;
        return;
    }
    BwdShared& sh = *reinterpret_cast<BwdShared*>(dsm + kOffBar);
    float* s_lse = reinterpret_cast<float*>(dsm + kOffStat);  // [2][128], LSE * log2(e)
    float* s_D = s_lse + 256;                                 // [2][128]
    const uint32_t sK = base + kOffK, sV = base + kOffV, sDS = base + kOffDS;

    if (tid == 0) {
        mbar_init(&sh.kv_full, 1);
        mbar_init(&sh.kv_empty, 1);
        for (int s = 0; s < 2; ++s) { mbar_init(&sh.q_full[s], 1); mbar_init(&sh.q_empty[s], 1); }
        mbar_init(&sh.do_full, 1);
        mbar_init(&sh.do_empty, 1);
        mbar_init(&sh.s_full, 1);
        mbar_init(&sh.dp_full, 1);
        mbar_init(&sh.p_ready, 256);
        mbar_init(&sh.ds_ready, 256);
        mbar_init(&sh.ds_free, 1);
        mbar_init(&sh.dq_full, 1);
        mbar_init(&sh.dq_free, 128);
        mbar_init(&sh.dkdv_done, 1);
        mbar_init(&sh.acc_free, 128);
        mbar_init(&sh.drain, kIssuers<D>);
        mbar_init(&sh.r0_free, 1);
        for (int s = 0; s < 4; ++s) { mbar_init(&sh.unit_full[s], 1); mbar_init(&sh.unit_empty[s], kUnitReaders<D>); }
        sh.abort_flag = 0;
        int total = a.varlen ? a.hdr->total_units : a.B * a.Hkv * ((a.N + kTileN - 1) / kTileN);
        if (a.varlen && a.hdr->unit_keys != kTileN) {   // planned for the CTA-pair kernel
            if (atomicCAS(&a.hdr->status.code, 0, -1) == 0) a.hdr->status.where = 202;
            total = 0;
        }
        if (a.varlen && a.hdr->unit_heads != a.kv_split) {   // planned for the other mode
            if (atomicCAS(&a.hdr->status.code, 0, -1) == 0) a.hdr->status.where = 203;
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
        if (a.kv_split) tma_prefetch_desc(&tdkv);
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

    // Register split (launch 512 x 128 = 65536): the two key-row warpgroups
    // 144 each (a 64-float half row of P), the dQ warpgroup 168 (a whole dQ
    // row), the loader/UMMA warpgroup 56: 128 * (144 + 144 + 168 + 56) = 65536.
    if (warp >= 8 && warp < 12) {
        regs_dec<56>();
        if (warp == 8) {
            // ------------------------------------------------------------ loader
            uint32_t jj = 0, uc = 0;
            bool ok = true;
            for (uint32_t n = 0; ok; ++n) {
                // Claim the next unit: the first by block index, then in
                // list order from the global counter, so that a CTA that
                // finishes early takes more.  Exhausting the list counts the
                // CTA out; the last one out rewinds the counter for the next
                // launch.
                int u = -1;
                if (lane == 0) {
                    ok = mbar_wait(&sh.unit_empty[n & 3], ((n >> 2) & 1) ^ 1, wc, kBSiteUnit);
                    if (ok) {
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
                BUnit U;
                if (!bwd_unit(a, total, u, U)) break;
                if (lane == 0) ok = mbar_wait(&sh.kv_empty, (uc & 1) ^ 1, wc, kBSiteKvEmpty);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&sh.kv_full, 2 * kT32);
                    for (int c = 0; c < G::kBoxes; ++c) {
                        tma_load_3d(sK + c * kBox, &tk, &sh.kv_full, c * 64, U.hk, U.tok0 + U.k * kTileN);
                        tma_load_3d(sV + c * kBox, &tv, &sh.kv_full, c * 64, U.hk, U.tok0 + U.k * kTileN);
                    }
                }
                const int span = U.nq - U.i0;
                // LSE and D of a query tile are loaded one tile ahead, into
                // registers, so that their latency overlaps the waits for the
                // ring instead of delaying the tile's q_full.
                float nl[4], nd[4];
                auto load_stats = [&](int t) {
                    const int h = U.hk * g + U.h0 + t / span, i = U.i0 + t % span;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int q = i * kTileM + 4 * lane + e;
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
                    const int st = jj & 1, h = U.hk * g + U.h0 + t / span, i = U.i0 + t % span;
                    if (lane == 0) ok = mbar_wait(&sh.q_empty[st], ((jj >> 1) & 1) ^ 1, wc, kBSiteQEmpty);
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (!ok) break;
                    // Q first; the phase's one arrival follows the LSE/D stores.
                    if (lane == 0) {
                        mbar_expect_tx(&sh.q_full[st], kT32);
                        for (int c = 0; c < G::kBoxes; ++c)
                            tma_load_3d(base + kOffQ + st * kT32 + c * kBox, &tq, &sh.q_full[st], c * 64, h,
                                        U.tok0 + i * kTileM);
                    }
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        s_lse[st * 128 + 4 * lane + e] = nl[e];
                        s_D[st * 128 + 4 * lane + e] = nd[e];
                    }
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&sh.q_full[st]);
                        ok = mbar_wait(&sh.do_empty, (jj & 1) ^ 1, wc, kBSiteQEmpty);
                        if (ok) {
                            mbar_arrive_expect_tx(&sh.do_full, kT32);
                            for (int c = 0; c < G::kBoxes; ++c)
                                tma_load_3d(base + kOffDO + c * kBox, &tdo, &sh.do_full, c * 64, h, U.tok0 + i * kTileM);
                        }
                    }
                    if (t + 1 < U.n) load_stats(t + 1);
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (!ok) break;
                }
                ++uc;
            }
            if (lane == 0) {  // drain this thread's copies before teardown
                const uint64_t t0 = globaltimer_ns();
                for (uint32_t d = (jj > 2 ? jj - 2 : 0); d < jj; ++d)
                    while (!mbar_try_wait(smem_u32(&sh.q_full[d & 1]), (d >> 1) & 1) &&
                           globaltimer_ns() - t0 < kWaitLimitNs) {}
                if (uc > 0)
                    while (!mbar_try_wait(smem_u32(&sh.kv_full), (uc - 1) & 1) &&
                           globaltimer_ns() - t0 < kWaitLimitNs) {}
                if (jj > 0)
                    while (!mbar_try_wait(smem_u32(&sh.do_full), (jj - 1) & 1) &&
                           globaltimer_ns() - t0 < kWaitLimitNs) {}
            }
            __syncwarp();
        } else if (warp == 10 && kIssuers<D> == 2) {
            // ------------------------------------------------------- S issuer
            // S^T(j) = K Q_j^T into R0 as soon as Q_j is loaded and dV(j-1)
            // has finished reading P^T(j-1) there; a warp of its own, so the
            // wait for Q never holds back the other four products.
            uint32_t jj = 0, uc = 0;
            bool ok = true;
            for (uint32_t n = 0; ok; ++n) {
                if (!(ok = mbar_wait_w(&sh.unit_full[n & 3], (n >> 2) & 1, wc, kBSiteUnit))) break;
                const int u = *(volatile int*)&sh.unit_id[n & 3];
                __syncwarp();
                if (lane == 0) mbar_arrive(&sh.unit_empty[n & 3]);
                BUnit U;
                if (!bwd_unit(a, total, u, U)) break;
                if (!(ok = mbar_wait_w(&sh.kv_full, uc & 1, wc, kBSiteKvFull))) break;
                for (int t = 0; t < U.n; ++t, ++jj) {
                    if (!(ok = mbar_wait_w(&sh.q_full[jj & 1], (jj >> 1) & 1, wc, kBSiteQFull))) break;
                    if (jj > 0 && !(ok = mbar_wait_w(&sh.r0_free, (jj - 1) & 1, wc, kBSiteP))) break;
                    tc_fence_after();
                    mma_kk<D>(tmem + kColR0, sK, base + kOffQ + (jj & 1) * kT32);
                    umma_commit_w(&sh.s_full);
                }
                ++uc;
            }
            umma_commit_w(&sh.drain);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(smem_u32(&sh.drain), 0) && globaltimer_ns() - t0 < kWaitLimitNs) {}
            __syncwarp();
        } else if (warp == 9) {
            // ---------------------------------------- dV, dK, dQ, dP issuer
            uint32_t jj = 0, uc = 0;
            bool ok = true;
            for (uint32_t n = 0; ok; ++n) {
                if (!(ok = mbar_wait_w(&sh.unit_full[n & 3], (n >> 2) & 1, wc, kBSiteUnit))) break;
                const int u = *(volatile int*)&sh.unit_id[n & 3];
                __syncwarp();
                if (lane == 0) mbar_arrive(&sh.unit_empty[n & 3]);
                BUnit U;
                if (!bwd_unit(a, total, u, U)) break;
                if (!(ok = mbar_wait_w(&sh.kv_full, uc & 1, wc, kBSiteKvFull))) break;
                if (!(ok = mbar_wait_w(&sh.acc_free, (uc & 1) ^ 1, wc, kBSiteAcc))) break;
                if (jj > 0) {
                    if (!(ok = mbar_wait_w(&sh.dq_free, (jj - 1) & 1, wc, kBSiteDqFree))) break;
                    tc_fence_after();
                }
                if constexpr (kIssuers<D> == 1) {
                    // S^T of the unit's first tile (R0 was last read by the
                    // previous dV, which this thread issued earlier).
                    if (!(ok = mbar_wait_w(&sh.q_full[jj & 1], (jj >> 1) & 1, wc, kBSiteQFull))) break;
                    tc_fence_after();
                    mma_kk<D>(tmem + kColR0, sK, base + kOffQ + (jj & 1) * kT32);
                    umma_commit_w(&sh.s_full);
                }
                if (!(ok = mbar_wait_w(&sh.do_full, jj & 1, wc, kBSiteQFull))) break;
                mma_kk<D>(tmem + kColR1, sV, base + kOffDO);
                umma_commit_w(&sh.dp_full);
                for (int t = 0; t < U.n; ++t, ++jj) {
                    const uint32_t st = jj & 1;
                    const bool more = t + 1 < U.n;
                    if (!(ok = mbar_wait_w(&sh.p_ready, jj & 1, wc, kBSiteP))) break;
                    tc_fence_after();
                    mma_tn<D>(tmem + kColDV, tmem + kColR0, base + kOffDO, t > 0);
                    umma_commit_w(&sh.do_empty);     // dO read by dP and dV: the next may load
                    if constexpr (kIssuers<D> == 1) {
                        if (more) {                  // the next S^T, right behind dV
                            const uint32_t s1 = (jj + 1) & 1;
                            if (!(ok = mbar_wait_w(&sh.q_full[s1], ((jj + 1) >> 1) & 1, wc, kBSiteQFull))) break;
                            tc_fence_after();
                            mma_kk<D>(tmem + kColR0, sK, base + kOffQ + s1 * kT32);
                            umma_commit_w(&sh.s_full);
                        }
                    } else {
                        umma_commit_w(&sh.r0_free);  // P^T read: the next S^T may overwrite R0
                    }
                    if (!(ok = mbar_wait_w(&sh.ds_ready, jj & 1, wc, kBSiteDs))) break;
                    tc_fence_after();
                    // dQ goes over dP^T, which the dS step has read.  At
                    // d = 128 dK reads dS^T from R1 and dQ, issued after it
                    // by this thread, overwrites it; at d = 64 dK reads it
                    // from columns of its own.
                    if constexpr (kIssuers<D> == 1) {
                        mma_tn<D>(tmem + kColDK, tmem + kColR1, base + kOffQ + st * kT32, t > 0);
                        umma_commit_w(&sh.q_empty[st]);  // Q and LSE/D of this stage are consumed
                        mma_nn<D>(tmem + kColR1, sDS, sK);
                        umma_commit_w(&sh.dq_full);
                    } else {
                        mma_nn<D>(tmem + kColR1, sDS, sK);
                        umma_commit_w(&sh.dq_full);
                        mma_tl<D>(tmem + kColDK, tmem + kColDS64, base + kOffQ + st * kT32, t > 0);
                        umma_commit_w(&sh.q_empty[st]);  // Q and LSE/D of this stage are consumed
                    }
                    umma_commit_w(&sh.ds_free);      // dS read by dQ and dK
                    if (more) {
                        if (!(ok = mbar_wait_w(&sh.dq_free, jj & 1, wc, kBSiteDqFree))) break;
                        tc_fence_after();
                        if (!(ok = mbar_wait_w(&sh.do_full, (jj + 1) & 1, wc, kBSiteQFull))) break;
                        mma_kk<D>(tmem + kColR1, sV, base + kOffDO);
                        umma_commit_w(&sh.dp_full);
                    }
                }
                if (!ok) break;
                umma_commit_w(&sh.dkdv_done);
                umma_commit_w(&sh.kv_empty);
                ++uc;
            }
            umma_commit_w(&sh.drain);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(smem_u32(&sh.drain), 0) && globaltimer_ns() - t0 < kWaitLimitNs) {}
            __syncwarp();
        }
    } else if (warp < 4 || warp >= 12) {
        regs_inc<144>();
        // ------------------------------------------------ P^T and dS^T (key rows)
        // Two warpgroups share each key row: warps 0-3 take query columns
        // 0-63, warps 12-15 columns 64-127.
        const int hc = warp >= 12 ? 1 : 0;                   // which column half
        const int cb = hc * 64;
        const int r = (warp & 3) * 32 + lane;                // key row in the tile == TMEM lane
        const uint32_t lb = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tR0 = tmem + lb + kColR0, tR1 = tmem + lb + kColR1;
        uint8_t* ds_row = dsm + kOffDS + hc * kBox + r * 128;
        const int sw = r & 7;
        uint32_t jj = 0;
        bool ok = true;
        for (uint32_t n = 0; ok; ++n) {
            if (!(ok = mbar_wait(&sh.unit_full[n & 3], (n >> 2) & 1, wc, kBSiteUnit))) break;
            const int u = *(volatile int*)&sh.unit_id[n & 3];
            mbar_arrive(&sh.unit_empty[n & 3]);
            BUnit U;
            if (!bwd_unit(a, total, u, U)) break;
            const int key = U.k * kTileN + r;
            const int span = U.nq - U.i0;
            for (int t = 0; t < U.n; ++t, ++jj) {
                const int st = jj & 1, i = U.i0 + t % span;
                if (!(ok = mbar_wait(&sh.q_full[st], (jj >> 1) & 1, wc, kBSiteQFull))) break;
                if (!(ok = mbar_wait(&sh.s_full, jj & 1, wc, kBSiteS))) break;
                tc_fence_after();
                float p[64];
                {
                    uint32_t* pu = reinterpret_cast<uint32_t*>(p);
                    tmem_ld32(tR0 + cb, *reinterpret_cast<uint32_t(*)[32]>(pu + 0));
                    tmem_ld32(tR0 + cb + 32, *reinterpret_cast<uint32_t(*)[32]>(pu + 32));
                    tmem_wait_ld();
                }
                // visible columns c: query 128 i + c < len, key < len, and key <= query if causal
                const int c_lo = (a.causal ? key - i * kTileM : 0) - cb;
                const int c_hi = (key >= U.len ? 0 : U.len - i * kTileM) - cb;
                const float4* l2v = reinterpret_cast<const float4*>(s_lse + st * 128 + cb);
                // At d = 128 the exponent arguments here and p (dP - D) below are
                // computed two at a time on packed fp32 pairs (each lane rounds
                // as the scalar form does, so the results are the same bits):
                // headline backward 1175 -> 1185, causal_bwd 1127 -> 1147
                // TFLOP/s; at d = 64 the scalar form measured faster.
                const uint64_t sc2 = f2_pack(scale, scale);
                if (c_lo <= 0 && c_hi >= 64) {   // every column visible: no mask
#pragma unroll
                    for (int c4 = 0; c4 < 16; ++c4) {
                        const float4 l4 = l2v[c4];
                        if constexpr (D == 128) {
                            float x0, x1, x2, x3;
                            f2_unpack(f2_fma(f2_pack(p[4 * c4], p[4 * c4 + 1]), sc2, f2_pack(-l4.x, -l4.y)), x0, x1);
                            f2_unpack(f2_fma(f2_pack(p[4 * c4 + 2], p[4 * c4 + 3]), sc2, f2_pack(-l4.z, -l4.w)), x2, x3);
                            p[4 * c4] = ex2_mufu(x0);
                            p[4 * c4 + 1] = ex2_mufu(x1);
                            p[4 * c4 + 2] = ex2_mufu(x2);
                            p[4 * c4 + 3] = ex2_mufu(x3);
                        } else {
                            p[4 * c4] = ex2_mufu(fmaf(p[4 * c4], scale, -l4.x));
                            p[4 * c4 + 1] = ex2_mufu(fmaf(p[4 * c4 + 1], scale, -l4.y));
                            p[4 * c4 + 2] = ex2_mufu(fmaf(p[4 * c4 + 2], scale, -l4.z));
                            p[4 * c4 + 3] = ex2_mufu(fmaf(p[4 * c4 + 3], scale, -l4.w));
                        }
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
#pragma unroll
                for (int stg = 0; stg < 2; ++stg) {
                    uint32_t pk[16];
#pragma unroll
                    for (int m = 0; m < 16; ++m) pk[m] = pack_bf16x2(p[stg * 32 + 2 * m], p[stg * 32 + 2 * m + 1]);
                    tmem_st16(tR0 + cb + stg * 16, pk);   // P^T: two bf16 per column, in this half's own columns
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&sh.p_ready);

                // dS^T from this half's dP^T columns, into shared memory.
                if (!(ok = mbar_wait(&sh.dp_full, jj & 1, wc, kBSiteDp))) break;
                if (!(ok = mbar_wait(&sh.ds_free, (jj & 1) ^ 1, wc, kBSiteDsFree))) break;
                tc_fence_after();
                const float4* dv4 = reinterpret_cast<const float4*>(s_D + st * 128 + cb);
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    uint32_t dp[32];
                    tmem_ld32(tR1 + cb + cc * 32, dp);
                    tmem_wait_ld();
                    uint32_t pk[16];
#pragma unroll
                    for (int m = 0; m < 8; ++m) {
                        const float4 d4 = dv4[cc * 8 + m];
                        const int c = cc * 32 + 4 * m;
                        if constexpr (D == 128) {
                            float a0, a1, a2, a3;
                            f2_unpack(f2_mul(f2_pack(p[c], p[c + 1]),
                                             f2_add(f2_pack(__uint_as_float(dp[4 * m]), __uint_as_float(dp[4 * m + 1])),
                                                    f2_pack(-d4.x, -d4.y))), a0, a1);
                            f2_unpack(f2_mul(f2_pack(p[c + 2], p[c + 3]),
                                             f2_add(f2_pack(__uint_as_float(dp[4 * m + 2]), __uint_as_float(dp[4 * m + 3])),
                                                    f2_pack(-d4.z, -d4.w))), a2, a3);
                            pk[2 * m] = pack_bf16x2(a0, a1);
                            pk[2 * m + 1] = pack_bf16x2(a2, a3);
                        } else {
                            pk[2 * m] = pack_bf16x2(p[c] * (__uint_as_float(dp[4 * m]) - d4.x),
                                                    p[c + 1] * (__uint_as_float(dp[4 * m + 1]) - d4.y));
                            pk[2 * m + 1] = pack_bf16x2(p[c + 2] * (__uint_as_float(dp[4 * m + 2]) - d4.z),
                                                        p[c + 3] * (__uint_as_float(dp[4 * m + 3]) - d4.w));
                        }
                    }
                    // 32 queries = four 16-byte chunks; chunk q of this half's
                    // box holds queries cb + 8q .. +7 at position q ^ (row % 8).
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const int q = cc * 4 + m;
                        *reinterpret_cast<uint4*>(ds_row + ((q ^ sw) << 4)) =
                            make_uint4(pk[4 * m], pk[4 * m + 1], pk[4 * m + 2], pk[4 * m + 3]);
                    }
                    // And into TMEM as dK's A operand: at d = 128 into this
                    // half's own R1 columns, which this thread has read
                    // (packed as P^T is); at d = 64 into the free columns
                    // 64-127, which dK of the previous tile has read (ds_free).
                    if constexpr (D == 128) tmem_st16(tR1 + cb + cc * 16, pk);
                    else tmem_st16(tmem + lb + kColDS64 + hc * 32 + cc * 16, pk);
                }
                tmem_wait_st();
                fence_async_smem();   // dS is read by the dQ product
                tc_fence_before();    // dP^T read: dQ may overwrite it
                mbar_arrive(&sh.ds_ready);
            }
        }
    } else {
        regs_inc<168>();
        // -------------------------------------------- dQ drain, dK/dV epilogue
        const int r = tid - 128;                             // query row (dQ) / key row (dK, dV)
        const uint32_t lb = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tR1 = tmem + lb + kColR1;
        uint32_t jj = 0, uc = 0;
        bool ok = true;
        // Deterministic mode: the semaphore of the previous query tile, to be
        // released once that tile's reductions are complete -- checked at the
        // start of the next tile instead of waited for at the end of this one,
        // so the drain does not stall on the round trip to L2 every tile.
        int* sem_pend = nullptr;
        // Add a 128-row tile of fp32 rows (this thread's row in v) into an
        // accumulator with TMA bulk tensor reductions of whole 128-byte
        // lines, staged in shared memory in D / 32 rounds of one 32-column
        // box (128 rows x 128 B, swizzled like a 128-B TMA box) alternating
        // between two buffers, so each round's reduction reads one buffer
        // while the threads fill the other.
        auto stage_add = [&](const uint32_t (&v)[D], const CUtensorMap* map, int grow) {
            uint8_t* stage_row = dsm + kOffStage + r * 128;
#pragma unroll
            for (int rnd = 0; rnd < D / 32; ++rnd) {
                const int b = rnd & 1;
                // At most the latest group may still be reading: the one
                // before it used this buffer.
                if (r == 0) bulk_wait_read1();
                named_bar(1, 128);
                const uint32_t* src = v + rnd * 32;
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    *reinterpret_cast<uint4*>(stage_row + b * kBox + ((q ^ (r & 7)) << 4)) =
                        make_uint4(src[4 * q], src[4 * q + 1], src[4 * q + 2], src[4 * q + 3]);
                fence_async_smem();
                named_bar(1, 128);
                if (r == 0) {
                    tma_reduce_add_2d(map, base + kOffStage + b * kBox, rnd * 32, grow);
                    bulk_commit();
                }
            }
        };
        auto release_pending = [&]() {
            if (r == 0 && sem_pend) {
                bulk_wait0();          // the tile's additions are complete
                fence_async_global();  // ... and ordered before the release
                red_release_add(sem_pend, 1);
            }
            sem_pend = nullptr;
        };
        for (uint32_t n = 0; ok; ++n) {
            ok = mbar_wait(&sh.unit_full[n & 3], (n >> 2) & 1, wc, kBSiteUnit);
            // The warpgroup meets at named barriers below: it leaves together.
            if (named_bar_or(1, 128, !ok)) { ok = false; break; }
            const int u = *(volatile int*)&sh.unit_id[n & 3];
            mbar_arrive(&sh.unit_empty[n & 3]);
            BUnit U;
            if (!bwd_unit(a, total, u, U)) break;
            const int span = U.nq - U.i0;
            for (int t = 0; t < U.n; ++t, ++jj) {
                const int h = U.hk * g + U.h0 + t / span, i = U.i0 + t % span;
                ok = mbar_wait(&sh.dq_full, jj & 1, wc, kBSiteDq);
                // Named barriers follow: every thread of the warpgroup must
                // take the same path, so the warpgroup agrees on aborts.
                ok = !named_bar_or(1, 128, !ok);
                if (!ok) break;
                tc_fence_after();
                // dQ_i out of TMEM into registers; the columns are free for the
                // next dP at once.
                uint32_t v[D];
#pragma unroll
                for (int c0 = 0; c0 < D; c0 += 32)
                    tmem_ld32(tR1 + c0, *reinterpret_cast<uint32_t(*)[32]>(v + c0));
                tmem_wait_ld();
                tc_fence_before();
                mbar_arrive(&sh.dq_free);
                int* sem = a.deterministic ? a.sem + (size_t)h * a.sem_stride + U.seq + (U.tok0 + i * kTileM) / kTileN
                                           : nullptr;
                if (sem) {
                    release_pending();
                    // Key tiles add into this query tile in ascending order;
                    // wait (bounded) until the previous one has released it.
                    // The wait runs in another warp than the releasing thread,
                    // so the two round trips to L2 overlap; the barrier below
                    // then orders the acquire before this tile's reductions.
                    bool gave_up = false;
                    if (r == 32) {
                        const uint64_t t0 = globaltimer_ns();
                        uint32_t spins = 0;
                        while (ld_acquire(sem) != U.k) {
                            if ((++spins & 255u) == 0 &&
                                (*(volatile int*)&sh.abort_flag || globaltimer_ns() - t0 > kWaitLimitNs)) {
                                if (atomicCAS(&a.hdr->status.code, 0, kStatusTimeout) == 0) {
                                    a.hdr->status.where = kBSiteSem;
                                    a.hdr->status.block = blockIdx.x;
                                }
                                *(volatile int*)&sh.abort_flag = 1;
                                gave_up = true;
                                break;
                            }
                        }
                    }
                    if (named_bar_or(1, 128, gave_up)) { ok = false; break; }
                    if (r == 0) fence_async_global();  // our bulk reduction follows the acquire
                }
                // Add dQ_i into the fp32 accumulator.  Rows past the sequence
                // end hold exact zeros (their P, hence dS, is zero), so adding
                // them to the neighbouring rows changes nothing.
                stage_add(v, &tdq, h * (int)a.T + U.tok0 + i * kTileM);
                sem_pend = sem;
                if (r == 0) dbg_count(a.dbg_inner, (long long)h * a.T + U.tok0 + i * kTileM);
            }
            if (!ok) break;
            release_pending();   // before the dK/dV epilogue: the next key tile is waiting
            ok = mbar_wait(&sh.dkdv_done, uc & 1, wc, kBSiteDkdv);
            if (named_bar_or(1, 128, !ok)) { ok = false; break; }
            ++uc;
            tc_fence_after();
            if (a.kv_split) {
                // A split unit's dK and dV are partial (its head group's
                // share): added into the fp32 sums [2][Hkv][T][d], which the
                // last stage converts.  Key rows past the sequence end hold
                // exact zeros, as dQ's rows do.
#pragma unroll
                for (int which = 0; which < 2; ++which) {
                    uint32_t v[D];
                    const uint32_t tacc = tmem + lb + (which ? kColDV : kColDK);
#pragma unroll
                    for (int c0 = 0; c0 < D; c0 += 32)
                        tmem_ld32(tacc + c0, *reinterpret_cast<uint32_t(*)[32]>(v + c0));
                    tmem_wait_ld();
                    if (which == 1) {   // both accumulators read: the next unit may start
                        if (r == 0) dbg_count(a.dbg_visits, (long long)U.hk * a.T + U.tok0 + U.k * kTileN);
                        tc_fence_before();
                        mbar_arrive(&sh.acc_free);
                    }
                    stage_add(v, &tdkv, (which * a.Hkv + U.hk) * (int)a.T + U.tok0 + U.k * kTileN);
                }
                continue;
            }
            const int key = U.k * kTileN + r;
            const bool kvalid = key < U.len;
            const size_t orow = ((size_t)(U.tok0 + key) * a.Hkv + U.hk) * D;
#pragma unroll
            for (int which = 0; which < 2; ++which) {
                const uint32_t tacc = tmem + lb + (which ? kColDV : kColDK);
                const float mul = which ? 1.f : a.alpha;
                uint4* out = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(which ? a.dv : a.dk) + orow);
#pragma unroll
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t v[32];
                    tmem_ld32(tacc + cc * 32, v);
                    tmem_wait_ld();
                    if (kvalid) {
#pragma unroll
                        for (int m = 0; m < 4; ++m) {
                            const float* f = reinterpret_cast<const float*>(v + 8 * m);
                            out[cc * 4 + m] = make_uint4(pack_bf16x2(f[0] * mul, f[1] * mul), pack_bf16x2(f[2] * mul, f[3] * mul),
                                                         pack_bf16x2(f[4] * mul, f[5] * mul), pack_bf16x2(f[6] * mul, f[7] * mul));
                        }
                    }
                }
            }
            if (r == 0) dbg_count(a.dbg_visits, (long long)U.hk * a.T + U.tok0 + U.k * kTileN);
            tc_fence_before();
            mbar_arrive(&sh.acc_free);
        }
        if (r == 0) bulk_wait0();  // every bulk reduction issued here has completed
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

__global__ void bwd_reset_status_kernel(BwdHeader* hdr) {
    hdr->status.code = 0;
    hdr->status.where = 0;
    hdr->status.block = 0;
    hdr->next_unit = 0;
    hdr->done_ctas = 0;
}

}  // namespace

template <int D>
cudaError_t launch_bwd_d(const BwdLaunch& L, int stages, cudaStream_t stream) {
    const BwdArgs& a = L.a;
    const int ew_grid = L.num_sms * 8;
    if (stages & 1) {
        bwd_reset_status_kernel<<<1, 1, 0, stream>>>(a.hdr);
        bwd_pre_kernel<D><<<ew_grid, 256, 0, stream>>>(a);
        if (a.varlen) bwd_plan_kernel<<<1, 1024, 0, stream>>>(a, L.pair ? 2 * kTileN : kTileN);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if constexpr (D == 256) {
        if (stages & 2) {
            cudaError_t e = launch_bwd256_main(L, stream);
            if (e != cudaSuccess) return e;
        }
    } else if ((stages & 2) && L.pair) {
        cudaError_t e = launch_bwd_pair_main(L, stream);
        if (e != cudaSuccess) return e;
    } else if (stages & 2) {
        constexpr uint32_t smem = BGeo<D>::kSmem;
        cudaError_t e0 = cudaFuncSetAttribute(bwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e0 != cudaSuccess) return e0;
        long long units = a.varlen ? (long long)a.Hkv * ((a.T + kTileN - 1) / kTileN + a.B)
                                   : (long long)a.B * a.Hkv * ((a.N + kTileN - 1) / kTileN);
        if (a.kv_split) units *= (a.Hq / a.Hkv) / a.kv_split;
        int grid = (int)(units < L.num_sms ? units : L.num_sms);
        if (grid < 1) grid = 1;
        bwd_kernel<D><<<grid, kBwdThreads, smem, stream>>>(L.tq, L.tk, L.tv, L.tdo, L.tdq, L.tdkv, a);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (stages & 4) {
        bwd_post_kernel<D><<<ew_grid, 256, 0, stream>>>(a);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_bwd(const BwdLaunch& L, int stages, cudaStream_t stream) {
    if (L.d == 64) return launch_bwd_d<64>(L, stages, stream);
    if (L.d == 128) return launch_bwd_d<128>(L, stages, stream);
    if (L.d == 256) return launch_bwd_d<256>(L, stages, stream);
    return cudaErrorInvalidValue;
}

}  // namespace fa
