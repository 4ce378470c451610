// fa_prim.cuh -- sm_103a device primitives written as inline PTX:
// mbarriers with bounded waits, TMA tile loads, tensor-memory (TMEM)
// allocation, tcgen05.mma (UMMA) issue/commit, tcgen05.ld/st, and the shared
// memory / instruction descriptors the UMMA reads.
//
// Hardware features named by the FlashAttention-4 blog, "New hardware
// features on Blackwell": TMEM (256 KB per SM, a scratchpad wired to the
// tensor cores), fully asynchronous tcgen05.mma accumulating in TMEM and
// issued by a single thread, operand A optionally read from TMEM.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <type_traits>

namespace fa {

// ----------------------------------------------------------------------------
// Device status word and bounded waits.
//
// Every spin-wait is bounded: after kWaitLimitNs without progress the waiter
// records FA_ERR_TIMEOUT in the device status word, raises the CTA's abort
// flag and returns false; every later wait of any thread sees the flag and
// returns false at once, so each role leaves its loop and the CTA reaches its
// teardown (drain, TMEM free) instead of hanging the GPU.
// ----------------------------------------------------------------------------
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s
constexpr int kStatusTimeout = -5;                            // == FA_ERR_TIMEOUT

struct DevStatus {
    int code;     // 0 or kStatusTimeout
    int where;    // which wait gave up (site id)
    int block;    // blockIdx.x of the first CTA that gave up
    int pad;
};

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Per-wait context: the CTA abort flag in shared memory and the device status.
struct WaitCtx {
    volatile int* abort_flag;     // shared
    DevStatus* status;            // global
};

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}

static __device__ __forceinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, const WaitCtx& w, int site) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 0) {
            if (*w.abort_flag) return false;
            if (*(volatile int*)&w.status->code != 0) { *w.abort_flag = 1; return false; }
            if (globaltimer_ns() - t0 > kWaitLimitNs) {
                if (atomicCAS(&w.status->code, 0, kStatusTimeout) == 0) {
                    w.status->where = site;
                    w.status->block = blockIdx.x;
                }
                *w.abort_flag = 1;
                return false;
            }
        }
    }
}

// Wait for the phase of parity `parity` of mbarrier `bar`; false on abort.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const WaitCtx& w, int site) {
    const uint32_t a = smem_u32(bar);
    if (mbar_try_wait(a, parity)) return true;
    return mbar_wait_slow(a, parity, w, site);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Raise the phase's expected transaction bytes without arriving.
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

// ----------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor), tile mode, completion counted on an mbarrier.
// Every x coordinate passed here is a multiple of 64 bf16 elements (128 B).
// ----------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint64_t* bar,
                                            int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
        : "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ----------------------------------------------------------------------------
// Tensor memory.  Addresses: bits [31:16] lane, [15:0] column (32-bit cells).
// A warp may touch only its lane quarter: lanes 32*(warp%4) .. +31.
// ----------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {  // whole warp
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_u32(dst_smem)), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {  // whole warp
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {  // whole warp
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 32 lanes x 32 consecutive 32-bit columns; thread t gets lane (base+t).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
        ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
          "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
        ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
          "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
          "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
          "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

// ----------------------------------------------------------------------------
// UMMA descriptors.
//
// Shared-memory matrix descriptor (64 bit): start address >> 4 in [0,14),
// leading-dimension byte offset >> 4 in [16,30), stride-dimension byte offset
// >> 4 in [32,46), descriptor version 1 in [46,48), base offset 0 (tiles are
// 1024-byte aligned), layout type in [61,64) with 2 = 128-byte swizzle.
//
// Tiles are stored the way a TMA load with 128-byte swizzle writes a box of
// 64 bf16 (128 B) x R rows: row r at byte 128*r, 16-byte chunks XOR-permuted
// by (r % 8).  A 128 x 128 bf16 tile is two such boxes, 64 columns each.
//   K-major operand (K contiguous, e.g. Q and K rows): 8-row groups 1024 B
//     apart (SBO); one K=16 step = 32 B inside the 128-B row; the second
//     64-column box begins at +R*128 B.
//   MN-major operand (N contiguous, e.g. V as the B of P V): 8 K-rows of
//     128 B form an atom, 8-row groups 1024 B apart (SBO); the second 64-wide
//     N chunk (the second box) is LBO = R*128 B away.
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1u << 46;
    d |= (uint64_t)2u << 61;
    return d;
}

// Instruction descriptor for kind::f16: bf16 A and B, f32 accumulator.
// c_format [4,6)=1 (f32), a_format [7,10)=1 (bf16), b_format [10,13)=1,
// a_major bit 15, b_major bit 16 (0 = K-major, 1 = MN-major),
// N>>3 in [17,23), M>>4 in [24,29).
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, int a_mn_major, int b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn_major << 15) | ((uint32_t)b_mn_major << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T   (cta_group::1, kind::f16)
__device__ __forceinline__ void umma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]   (A read from tensor memory)
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
        ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}

// Warp-wide issue: the whole (converged) warp executes these with warp-uniform
// operands and elect.sync picks the one lane that issues.  Keeping the issue
// loop converged lets the compiler hold descriptors in uniform registers; an
// issue loop run by a single lane inside a divergent branch issues UMMAs
// markedly slower than the tensor core retires them.
__device__ __forceinline__ void umma_ss_w(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}

__device__ __forceinline__ void umma_ts_w(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
        ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}

__device__ __forceinline__ void umma_commit_w(uint64_t* bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}"
        ::"r"(smem_u32(bar)) : "memory");
}

// ----------------------------------------------------------------------------
// CTA pairs (a cluster of two CTAs sharing one tcgen05 product).
//
// With .cta_group::2 one thread of the even CTA issues an M = 256 product:
// each CTA supplies 128 rows of A (from its shared or tensor memory) and half
// of B's N extent (the even CTA the first N/2, the odd CTA the rest); each
// CTA's tensor memory receives its 128 rows x all N columns.  Allocation and
// release of tensor memory are collective: one warp of each CTA executes them
// and both receive the same column address.  Every tcgen05 instruction of a
// kernel uses the same CTA-group size.
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Address of the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_rank(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
// Every thread of both CTAs; orders earlier shared-memory effects cluster-wide.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// One arrival per warp (elected lane) on a cluster-addressed mbarrier.  The
// caller's lanes must be converged; a preceding tcgen05.wait::ld / ::st is
// warp-collective, so every lane's tensor-memory access is complete here.
// The arrival carries the default CTA-scope release: what the waiting CTA
// needs to observe is the barrier itself (tensor-memory effects are ordered by
// the tcgen05 fences), and a cluster-scope release costs hundreds of cycles
// because it first drains this thread's outstanding memory operations.
__device__ __forceinline__ void mbar_arrive_remote_w(uint32_t cluster_addr) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e mbarrier.arrive.shared::cluster.b64 _, [%0];\n\t}"
        ::"r"(cluster_addr) : "memory");
}
// TMA load into this CTA's shared memory whose completion is counted on an
// mbarrier of either CTA of the pair (cluster address).
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar_cluster,
                                                 int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y), "r"(z)
        : "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {  // one warp per CTA
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_u32(dst_smem)), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {  // one warp per CTA
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void umma_ss_pair_w(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                               uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}
__device__ __forceinline__ void umma_ts_pair_w(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                               uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
        ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}
// Arrive on the mbarrier at this offset in every CTA of `cta_mask` once all
// earlier pair products issued by this thread are complete.
__device__ __forceinline__ void umma_commit_pair_w(uint64_t* bar, uint16_t cta_mask) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n\t}"
        ::"r"(smem_u32(bar)), "h"(cta_mask) : "memory");
}

// ----------------------------------------------------------------------------
// Straight-line issue.  A 128x128x16 product occupies the tensor core for 64
// cycles; an issue loop that recomputes descriptors at run time costs the
// issuing warp more than that per instruction, so the core starves (measured
// on GB300: 8 K-steps from a rolled loop ~105 cycles each, from straight-line
// code 64.1).  These forms take each step's descriptor offset as an immediate
// and add it to the low word inside the instruction's own asm block: a shared
// address below 256 KB keeps the 14-bit start-address field from carrying,
// and nothing is hoisted into registers.
// ----------------------------------------------------------------------------
template <int... I>
struct int_seq {};
template <int N, int... I>
struct make_int_seq : make_int_seq<N - 1, N - 1, I...> {};
template <int... I>
struct make_int_seq<0, I...> {
    using type = int_seq<I...>;
};
template <typename F, int... I>
__device__ __forceinline__ void static_for_impl(F& f, int_seq<I...>) {
    (f(std::integral_constant<int, I>{}), ...);
}
// f(std::integral_constant<int, k>) for k = 0 .. N-1, unrolled at compile time.
template <int N, typename F>
__device__ __forceinline__ void static_for(F&& f) {
    static_for_impl(f, typename make_int_seq<N>::type{});
}

// D[tmem] (+)= A[smem] B[smem]; AO, BO: descriptor offsets (bytes >> 4).
template <uint32_t AO, uint32_t BO, int GROUP = 1>
__device__ __forceinline__ void umma_ss_k(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
    if constexpr (GROUP == 1)
        asm volatile(
            "{\n\t.reg .pred p, e;\n\t.reg .b32 al, ah, bl, bh;\n\t.reg .b64 ad, bd;\n\t"
            "mov.b64 {al, ah}, %1;\n\tmov.b64 {bl, bh}, %2;\n\t"
            "add.u32 al, al, %5;\n\tadd.u32 bl, bl, %6;\n\t"
            "mov.b64 ad, {al, ah};\n\tmov.b64 bd, {bl, bh};\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "elect.sync _|e, 0xffffffff;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %3, p;\n\t}"
            ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "n"(AO), "n"(BO) : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p, e;\n\t.reg .b32 al, ah, bl, bh;\n\t.reg .b64 ad, bd;\n\t"
            "mov.b64 {al, ah}, %1;\n\tmov.b64 {bl, bh}, %2;\n\t"
            "add.u32 al, al, %5;\n\tadd.u32 bl, bl, %6;\n\t"
            "mov.b64 ad, {al, ah};\n\tmov.b64 bd, {bl, bh};\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "elect.sync _|e, 0xffffffff;\n\t"
            "@e tcgen05.mma.cta_group::2.kind::f16 [%0], ad, bd, %3, p;\n\t}"
            ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "n"(AO), "n"(BO) : "memory");
}

// D[tmem] (+)= A[tmem + AC columns] B[smem]; BO: descriptor offset (bytes >> 4).
template <uint32_t AC, uint32_t BO, int GROUP = 1>
__device__ __forceinline__ void umma_ts_k(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
    if constexpr (GROUP == 1)
        asm volatile(
            "{\n\t.reg .pred p, e;\n\t.reg .b32 bl, bh, at;\n\t.reg .b64 bd;\n\t"
            "mov.b64 {bl, bh}, %2;\n\tadd.u32 bl, bl, %6;\n\tmov.b64 bd, {bl, bh};\n\t"
            "add.u32 at, %1, %5;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "elect.sync _|e, 0xffffffff;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], bd, %3, p;\n\t}"
            ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate), "n"(AC), "n"(BO) : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p, e;\n\t.reg .b32 bl, bh, at;\n\t.reg .b64 bd;\n\t"
            "mov.b64 {bl, bh}, %2;\n\tadd.u32 bl, bl, %6;\n\tmov.b64 bd, {bl, bh};\n\t"
            "add.u32 at, %1, %5;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "elect.sync _|e, 0xffffffff;\n\t"
            "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [at], bd, %3, p;\n\t}"
            ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate), "n"(AC), "n"(BO) : "memory");
}

// Bounded wait executed by a whole warp; the result is made warp-uniform.
__device__ __forceinline__ bool mbar_wait_w(uint64_t* bar, uint32_t parity, const WaitCtx& w, int site) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, w, site));
}

// Arrive once on `bar` when every previously issued tcgen05.mma of this
// thread has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(smem_u32(bar)) : "memory");
}

// ----------------------------------------------------------------------------
// Packed fp32 pairs (sm_100 family: one instruction applies to both halves of
// a 64-bit register pair) and the three-input max.
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// ----------------------------------------------------------------------------
// Small math helpers.
// ----------------------------------------------------------------------------
__device__ __forceinline__ float ex2_mufu(float x) {  // MUFU.EX2 path
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Warpgroup register re-balancing (all 128 threads of the warpgroup execute it).
template <int kRegs>
__device__ __forceinline__ void regs_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegs));
}
template <int kRegs>
__device__ __forceinline__ void regs_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegs));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

}  // namespace fa
