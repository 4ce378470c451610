// fa_internal.h -- host-side structures shared by the C-ABI layer and the
// kernel translation units of libfa.so (not installed, not part of the ABI).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "fa_prim.cuh"

namespace fa {

constexpr int kHeadDim = 128;
constexpr int kTileM = 128;             // query rows per Q tile (one TMEM lane per row)
constexpr int kTileN = 128;             // keys per K/V tile
constexpr int kUnitRows = 2 * kTileM;   // two Q tiles (ping-pong) per forward work unit
constexpr int kMaxVarlenSeqs = 1024;    // sequences a varlen call may pack
constexpr int kMaxUnitLevels = 512;     // ceil(max_seqlen / 256) limit (max_seqlen <= 131072)
// Varlen backward: units of kSplitHeads query heads when a key/value head's
// group has at least kSplitMinGroup of them (a multiple of kSplitHeads).
constexpr int kSplitHeads = 8;
constexpr int kSplitMinGroup = 16;

// Forward arguments that are not tensor maps.
struct FwdArgs {
    void* o;                 // bf16 [.., Hq, 128]
    float* lse;              // float32
    const int* cu_seqlens;   // device int32[B+1] or nullptr
    DevStatus* status;       // device status word
    int B, Hq, Hkv;
    int N;                   // fixed length: sequence length; varlen: total tokens T
    int causal, varlen;
    int max_seqlen;          // varlen: bound on sequence length; fixed: N
    int l2_section;          // causal fixed-length: (batch, head) pairs per L2 section
    float scale_log2;        // alpha * log2(e)
    float tau;               // conditional-rescale threshold (log2 units)
    int naive;               // 1: work units in plain enumeration order (fa_set_schedule_order)
    // Debug counters (nullptr unless fa_set_debug_counters armed them):
    // visits[h * T + first row of a 128-row query tile] += 1 per finished
    // tile; rescale[0] += 1 per warp that takes the rescale branch after a
    // row block's first key block, rescale[1] += 1 per such warp decision.
    int* dbg_visits;
    unsigned long long* dbg_rescale;
};

struct FwdLaunch {
    CUtensorMap tq, tk, tv;  // 3-D maps {128, H, T}, box {64, 1, 128}, 128-B swizzle
    CUtensorMap to;          // O, same shape as tq (pair kernel: TMA stores of full tiles)
    FwdArgs a;
    int emu16;               // 0..4: share of exp2 pairs on the FMA pipe, in sixteenths
    int num_sms;
    int d = 128;             // head dim (128; 64 on the ping-pong kernel; 256 on fa_fwd256.cu)
};

// ---------------------------------------------------------------- backward
//
// Workspace layout (caller-allocated, sized by fa_bwd_workspace_size):
//   [0, 256)           BwdHeader (status word, unit count)
//   D                  float [Hq][T]            rowsum(dO * O)
//   dQacc              float [Hq][T][d]         fp32 dQ accumulator
//   semaphores         int   [Hq][T/128 + B + 1] (deterministic mode;
//                                                d = 256: [2][Hq][T/64 + B + 1])
//   units              int4  [Hkv * (T/128 + B)] (varlen work list)
//   cu                 int   [B+1]              (varlen: sanitised offsets)
// T = B*N for fixed length, the packed token count for varlen.
//
// Sanitised offsets (the one rule every kernel applies to cu_seqlens):
// c'_0 = clamp(c_0, 0, T), c'_s = max(c'_{s-1}, clamp(c_s, 0, T)); sequence
// s owns rows [c'_s, c'_{s+1}).  Malformed offsets therefore give empty
// sequences, never rows outside the tensors or overlapping sequences.
struct BwdHeader {
    DevStatus status;
    int total_units;   // varlen: written by the plan kernel
    int next_unit;     // main kernel: units claimed past the first wave
    int done_ctas;     // main kernel: CTAs that found the list exhausted (follows next_unit)
    int unit_keys;     // varlen: keys per unit of the planned list (256 for the CTA-pair kernel, else 128)
    int unit_heads;    // varlen: query heads per unit of the planned list (0: the whole group)
    int pad[55];
};
static_assert(sizeof(BwdHeader) == 256, "backward workspace header");
static_assert(offsetof(BwdHeader, done_ctas) == offsetof(BwdHeader, next_unit) + sizeof(int), "claim counters");

struct WsLayout {
    size_t d_off, dq_off, sem_off, unit_off, cu_off, kv_off, total;
    long long sem_stride;  // semaphores per query head
};

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

inline WsLayout ws_layout(long long T, int B, int Hq, int deterministic, int varlen, int d = kHeadDim) {
    WsLayout w;
    const long long tiles = (T + kTileN - 1) / kTileN;
    // Semaphores per query head: one per 128-row query tile (d = 256: per
    // 64-row query step, and a set for each head-dim half).
    const long long steps = d == 256 ? (T + 63) / 64 : tiles;
    const size_t sem_sets = d == 256 ? 2 : 1;
    w.sem_stride = steps + B + 1;
    w.d_off = align256(sizeof(BwdHeader));
    w.dq_off = align256(w.d_off + (size_t)Hq * T * 4);
    w.sem_off = align256(w.dq_off + (size_t)Hq * T * d * 4);
    w.unit_off = align256(w.sem_off + (deterministic ? sem_sets * Hq * w.sem_stride * 4 : 0));
    w.cu_off = align256(w.unit_off + (varlen ? (size_t)Hq * (tiles + B) * 16 : 0));
    // Varlen at d = 64 / 128: fp32 dK and dV partial sums [2][Hkv][T][d] for
    // work units split by query-head group, which needs Hq >= kSplitMinGroup
    // * Hkv, so Hq * T * d / 2 bytes always hold them.
    w.kv_off = align256(w.cu_off + (varlen ? (size_t)(B + 1) * 4 : 0));
    w.total = align256(w.kv_off + (varlen && d != 256 ? (size_t)Hq * T * d / 2 : 0));
    return w;
}

struct BwdArgs {
    const void* o;           // bf16 [T, Hq, 128] (forward output)
    const void* dO;          // bf16 [T, Hq, 128]
    const float* lse;        // forward LSE: [B, Hq, N] or varlen [Hq, T]
    void* dq;                // bf16 [T, Hq, 128]
    void* dk;                // bf16 [T, Hkv, 128]
    void* dv;                // bf16 [T, Hkv, 128]
    const int* cu_seqlens;   // device int32[B+1] or nullptr
    BwdHeader* hdr;
    float* D;
    float* dqacc;
    int* sem;
    int4* units;
    int* cu_s;               // varlen: sanitised offsets [B+1], written by the plan kernel
    float* dkvacc;           // varlen: fp32 dK, dV partial sums [2][Hkv][T][d] (split units)
    int kv_split;            // varlen: query heads per work unit when a unit covers part of
                             // its key/value head's group (its dK, dV then partial), else 0
    long long sem_stride;
    int B, Hq, Hkv;
    int N;                   // fixed: sequence length; varlen: T
    long long T;
    int causal, varlen, deterministic, max_seqlen;
    float alpha, scale_log2;
    int naive;               // 1: work units in plain enumeration order (fa_set_schedule_order)
    // Debug counters (nullptr unless fa_set_debug_counters armed them):
    // visits[hk * T + first row of a 128-key tile] += 1 per finished work
    // unit (key tile of one key/value head, or of one query-head group of it
    // for split units); inner[h * T + first row of a
    // 128-row query tile] += 1 per (key tile, query tile) product chain.
    int* dbg_visits;
    int* dbg_inner;
};

struct BwdLaunch {
    CUtensorMap tq, tk, tv, tdo;
    CUtensorMap tdq;         // dQacc as fp32 [Hq*T, d], box {32, 128}, 128-B swizzle
    CUtensorMap tdkv;        // dkvacc as fp32 [2*Hkv*T, d], box {32, 128} (split units)
    // CTA-pair main kernel only: Q and dO with 64-row boxes, dQacc with 64-row boxes.
    CUtensorMap tq64, tdo64, tdq64;
    BwdArgs a;
    int num_sms;
    int pair;                // stage 2 runs the CTA-pair kernel (fa_bwd_pair.cu; d = 128 only)
    int d = 128;             // head dim (128, 64 or 256)
};

// Head-dim 256 backward main kernel (fa_bwd256.cu): Q and dO maps with 64-row
// boxes, K and V with 128-row boxes, the dQ accumulator with 32 x 32 boxes.
cudaError_t launch_bwd256_main(const BwdLaunch& L, cudaStream_t stream);

// CTA-pair backward main kernel (fa_bwd_pair.cu): fixed length, atomic mode.
bool bwd_pair_supported(const BwdArgs& a);
cudaError_t launch_bwd_pair_main(const BwdLaunch& L, cudaStream_t stream);
extern int g_bwd_pairs_resident;

// Backward stages (fa_bwd.cu): 1 = preprocess (D, zero dQacc/semaphores,
// varlen plan), 2 = main kernel (dK, dV, dQacc), 4 = dQ postprocess.
cudaError_t launch_bwd(const BwdLaunch& L, int stages, cudaStream_t stream);

// Launch the forward kernel (fa_fwd.cu).  Returns a cudaError_t.
cudaError_t launch_fwd(const FwdLaunch& L, cudaStream_t stream);

// CTA-pair kernel (clusters of two), fixed length, MUFU exp2.
cudaError_t launch_fwd_pair(const FwdLaunch& L, cudaStream_t stream);
// CTA pairs the pair kernel keeps resident (0 until its first launch).
extern int g_pairs_resident;

// Evaluate the FMA-pipe exp2 on n floats (fa_fwd.cu).
cudaError_t launch_exp2_emu(const float* x, float* y, int64_t n, cudaStream_t stream);
cudaError_t launch_selftest_timeout(DevStatus* status, cudaStream_t stream);
// Forward for head dim 256 (fa_fwd256.cu): fixed length; tq with 128-row
// boxes, tk and tv with 64-row boxes.
cudaError_t launch_fwd256(const FwdLaunch& L, cudaStream_t stream);

// The library's device status word on the current device.
DevStatus* device_status_ptr();

// Debug counter increment (no-op while the counters are off).
__device__ __forceinline__ void dbg_count(int* counts, long long idx) {
    if (counts) atomicAdd(counts + idx, 1);
}
__device__ __forceinline__ void dbg_count_rescale(unsigned long long* c, bool after_first, bool taken) {
    if (c && after_first) {
        atomicAdd(c + 1, 1ull);
        if (taken) atomicAdd(c, 1ull);
    }
}

// fa_bwd's host-side argument checks (everything but the workspace), in the
// order fa_bwd applies them; on FA_OK *T_out is the token count.  ptrs: q,
// k, v, o, lse, dout, dq, dk, dv.
int bwd_validate(const void* const ptrs[9], int B, int Hq, int Hkv, int N, int d, float alpha, int causal,
                 const int* cu_seqlens, int max_seqlen, int deterministic, long long* T_out);

// Header of fa_bwd_noalloc's scratch area on the current device, or nullptr
// while no call has set the area up there (fa_noalloc.cu).
BwdHeader* noalloc_header_current_device();

}  // namespace fa
