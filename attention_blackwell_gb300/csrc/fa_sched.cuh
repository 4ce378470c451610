// fa_sched.cuh -- forward work-unit order, shared by the forward kernels.
//
// A unit is one 256-row query block of one (sequence, head): the ping-pong
// kernel's two 128-row tiles, or the CTA pair's two halves.  Packed varlen
// batches are scheduled from tables each CTA builds in its shared memory from
// cu_seqlens (identical in every CTA, so the CTAs of a pair agree on them).
#pragma once
#include "fa_internal.h"

namespace fa {

constexpr uint32_t kTableInts = (kMaxVarlenSeqs + 1) + kMaxVarlenSeqs + (kMaxVarlenSeqs + 1);

struct Unit {
    int seq, m, h, tok0, len;
};

// Work-unit order.
//  fixed length, non-causal: (batch, head)-major, query block minor, so the
//    CTAs running at one time share the K/V of few heads in L2;
//  fixed length, causal: longest-processing-time first inside L2-sized
//    sections of (batch, head) pairs -- sections in order, query blocks in
//    reverse (longest first), then the pairs of the section (FlashAttention-4
//    blog, "Scheduling").  With an even block count the blocks go out in
//    zig-zag couples instead: block m and block num_m - 1 - m of one (batch,
//    head), one after the other to the same worker, so every couple costs
//    num_m + 1 key blocks and a static stride over the couples leaves no
//    worker with more than one couple of extra work;
//  varlen: sequences sorted by block count (descending); causal walks query
//    block levels from the top down over the sorted sequences (longest
//    first), non-causal walks the sorted sequences head-major.
// naive (fa_set_schedule_order(1), for testing): every call walks
//    (sequence, head) major, query blocks ascending, sequences in index order.
struct Sched {
    int B, Hq, N, causal, varlen, num_m, sec, total, maxm;
    int zz;   // fixed length, causal, even num_m: zig-zag couples
    int naive;
    const int* s_cu;
    const int* s_order;
    const int* s_pref;

    __device__ __forceinline__ int nblk(int s) const {
        return (s_cu[s + 1] - s_cu[s] + kUnitRows - 1) / kUnitRows;
    }

    // Index of worker p's n-th unit (of P workers); at least total past the end.
    __device__ __forceinline__ int nth(int p, int P, int n) const {
        if (zz) return 2 * (p + (n >> 1) * P) + (n & 1);
        return p + n * P;
    }

    __device__ __forceinline__ bool get(int u, Unit& U) const {
        if (u < 0 || u >= total) return false;
        if (!varlen) {
            const int BH = B * Hq;
            int bh, m;
            if (!causal || naive) {
                bh = u / num_m;
                m = u - bh * num_m;
            } else if (zz) {
                // couple c = u / 2 of the section order; its first unit is the
                // longer block
                const int c = u >> 1, hm = num_m >> 1, per_sec = sec * hm;
                const int full = BH / sec;
                int mm;
                if (c < full * per_sec) {
                    const int s = c / per_sec, r = c - s * per_sec;
                    mm = r / sec;
                    bh = s * sec + r % sec;
                } else {
                    const int rem = BH - full * sec, r = c - full * per_sec;
                    mm = r / rem;
                    bh = full * sec + r % rem;
                }
                m = (u & 1) ? mm : num_m - 1 - mm;
            } else {
                const int per_sec = sec * num_m;
                const int full = BH / sec;
                if (u < full * per_sec) {
                    const int s = u / per_sec, r = u - s * per_sec;
                    m = num_m - 1 - r / sec;
                    bh = s * sec + r % sec;
                } else {
                    const int rem = BH - full * sec, r = u - full * per_sec;
                    m = num_m - 1 - r / rem;
                    bh = full * sec + r % rem;
                }
            }
            U.seq = bh / Hq;
            U.h = bh - U.seq * Hq;
            U.m = m;
            U.tok0 = U.seq * N;
            U.len = N;
            return true;
        }
        const bool levels = causal && !naive;
        const int n = levels ? maxm : B;
        int lo = 0, hi = n;  // first index with pref > u, minus one
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (s_pref[mid + 1] > u) hi = mid; else lo = mid + 1;
        }
        const int r = u - s_pref[lo];
        if (levels) {
            U.seq = s_order[r / Hq];
            U.h = r % Hq;
            U.m = maxm - 1 - lo;
        } else {
            U.seq = s_order[lo];
            const int nb = nblk(U.seq);
            U.h = r / nb;
            U.m = r - U.h * nb;
        }
        U.tok0 = s_cu[U.seq];
        U.len = s_cu[U.seq + 1] - U.tok0;
        return true;
    }
};

// Unit tables in shared memory (s_cu[B+1], s_order[B], s_pref[levels+1]) and
// the unit count, for fixed-length and varlen calls.  Every thread of the CTA
// calls this; *sh_maxm and *sh_total are written by thread 0 and valid after
// the caller's next __syncthreads.
__device__ __forceinline__ void build_sched_tables(const FwdArgs& a, int* s_cu, int* s_order, int* s_pref,
                                                   int* sh_maxm, int* sh_total, int tid, int nthreads) {
    // Work-unit tables (varlen): sanitised offsets, sequences sorted by
    // block count, and the unit prefix used by Sched::get.
    if (a.varlen) {
        for (int i = tid; i <= a.B; i += nthreads) {
            int c = a.cu_seqlens[i];
            s_cu[i] = c < 0 ? 0 : (c > a.N ? a.N : c);
        }
        __syncthreads();
        if (tid == 0)
            for (int i = 1; i <= a.B; ++i) s_cu[i] = s_cu[i] > s_cu[i - 1] ? s_cu[i] : s_cu[i - 1];
        __syncthreads();
        for (int i = tid; i < a.B; i += nthreads) {
            const int ni = (s_cu[i + 1] - s_cu[i] + kUnitRows - 1) / kUnitRows;
            int rank = 0;
            if (!a.naive)
                for (int j = 0; j < a.B; ++j) {
                    const int nj = (s_cu[j + 1] - s_cu[j] + kUnitRows - 1) / kUnitRows;
                    rank += (nj > ni) || (nj == ni && j < i);
                }
            s_order[a.naive ? i : rank] = i;
        }
        __syncthreads();
        if (tid == 0) {
            auto nb = [&](int s) { return (s_cu[s + 1] - s_cu[s] + kUnitRows - 1) / kUnitRows; };
            int maxm = 0;
            for (int i = 0; i < a.B; ++i) maxm = nb(i) > maxm ? nb(i) : maxm;
            int acc = 0;
            if (maxm > kMaxUnitLevels) {
                if (atomicCAS(&a.status->code, 0, -1) == 0) { a.status->where = 100; a.status->block = blockIdx.x; }
                *sh_maxm = 0;
                *sh_total = 0;
            } else if (a.causal && !a.naive) {
                int p = 0;
                for (int l = 0; l < maxm; ++l) {
                    const int m = maxm - 1 - l;
                    while (p < a.B && nb(s_order[p]) > m) ++p;
                    s_pref[l] = acc;
                    acc += a.Hq * p;
                }
                s_pref[maxm] = acc;
                *sh_maxm = maxm;
                *sh_total = acc;
            } else {
                for (int i = 0; i < a.B; ++i) { s_pref[i] = acc; acc += a.Hq * nb(s_order[i]); }
                s_pref[a.B] = acc;
                *sh_maxm = maxm;
                *sh_total = acc;
            }
        }
    } else if (tid == 0) {
        *sh_maxm = (a.N + kUnitRows - 1) / kUnitRows;
        *sh_total = a.B * a.Hq * *sh_maxm;
    }
}

}  // namespace fa
