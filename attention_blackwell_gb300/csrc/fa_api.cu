// fa_api.cu -- the C ABI of libfa.so (declared in include/fa.h): argument
// validation, TMA tensor-map construction, persistent-grid sizing, the device
// status word, and the kernel launches.  No device memory is allocated here.
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <mutex>

#include "../../include/fa.h"
#include "fa_internal.h"

namespace fa {

// One status word per device the library runs on (static device storage).
__device__ DevStatus g_status;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    bool ready = false;
    int num_sms = 0;
    int l2_bytes = 0;
    DevStatus* status = nullptr;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

int g_emu16 = 0;               // share of exp2 pairs on the FMA pipe (sixteenths)
int g_bwd_kernel = 0;          // 0: one CTA per 128-key tile; 1: CTA pairs per 256-key block
int g_fwd_kernel = 2;          // 0: ping-pong of two 128-row query tiles; 2: CTA pairs
float g_tau = 8.0f;            // conditional-rescale threshold, log2(256)
int g_naive = 0;               // 1: work units in plain enumeration order
int* g_dbg_visits = nullptr;   // debug counters (fa_set_debug_counters)
int* g_dbg_inner = nullptr;
unsigned long long* g_dbg_rescale = nullptr;

int current_device_info(DeviceInfo** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_LAUNCH;
    std::lock_guard<std::mutex> lock(g_dev_mu);
    DeviceInfo& d = g_dev[dev];
    if (!d.ready) {
        if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return FA_ERR_LAUNCH;
        if (cudaDeviceGetAttribute(&d.l2_bytes, cudaDevAttrL2CacheSize, dev) != cudaSuccess) return FA_ERR_LAUNCH;
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return FA_ERR_LAUNCH;
        d.status = static_cast<DevStatus*>(p);
        d.ready = true;
    }
    *out = &d;
    return FA_OK;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// bf16 tensor [T, H, d] -> 3-D map {d, H, T}, box {64, 1, box_rows}, 128-B swizzle.
// Rows past T read as zero.
int make_map(CUtensorMap* map, const void* ptr, int H, long long T, int box_rows = kTileM, int d = kHeadDim) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return FA_ERR_LAUNCH;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)T};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FA_OK : FA_ERR_INVALID;
}

// fp32 accumulator [rows, d] -> 2-D map {d, rows}, box {32, 128}, 128-B swizzle.
int make_map_acc(CUtensorMap* map, const void* ptr, long long rows, int box_rows = kTileM, int d = kHeadDim) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return FA_ERR_LAUNCH;
    cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)d * 4};
    cuuint32_t box[2] = {32, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FA_OK : FA_ERR_INVALID;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

DevStatus* device_status_ptr() {
    DeviceInfo* d = nullptr;
    return current_device_info(&d) == FA_OK ? d->status : nullptr;
}

}  // namespace fa

using namespace fa;

extern "C" {

const char* fa_status_string(int status) {
    switch (status) {
        case FA_OK: return "FA_OK";
        case FA_ERR_INVALID: return "FA_ERR_INVALID: invalid argument";
        case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED: configuration not supported by this build";
        case FA_ERR_ALIGN: return "FA_ERR_ALIGN: tensor not 16-byte aligned";
        case FA_ERR_LAUNCH: return "FA_ERR_LAUNCH: CUDA launch error";
        case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT: a device-side wait gave up";
        case FA_ERR_WORKSPACE: return "FA_ERR_WORKSPACE: workspace missing or too small";
        default: return "FA_ERR_UNKNOWN";
    }
}

int fa_num_sms(void) {
    DeviceInfo* d = nullptr;
    int rc = current_device_info(&d);
    return rc == FA_OK ? d->num_sms : rc;
}

int fa_set_tuning(int exp2_emu_sixteenths, float tau) {
    if (exp2_emu_sixteenths < 0 || exp2_emu_sixteenths > 4) return FA_ERR_UNSUPPORTED;
    if (!(tau >= 0.0f) || !(tau <= 64.0f)) return FA_ERR_INVALID;
    g_emu16 = exp2_emu_sixteenths;
    g_tau = tau;
    return FA_OK;
}

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int N, int d,
           float alpha, int causal, const int* cu_seqlens, int max_seqlen, cudaStream_t stream) {
    if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID;
    if (B < 1 || N < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0) return FA_ERR_INVALID;
    if (!(alpha > 0.0f) || !isfinite(alpha)) return FA_ERR_INVALID;
    if (causal != 0 && causal != 1) return FA_ERR_INVALID;
    if (d != 128 && d != 64 && d != 256) return FA_ERR_UNSUPPORTED;
    const bool varlen = cu_seqlens != nullptr;
    if (varlen) {
        if (max_seqlen < 1) return FA_ERR_INVALID;
        if (B > kMaxVarlenSeqs || (max_seqlen + kUnitRows - 1) / kUnitRows > kMaxUnitLevels)
            return FA_ERR_UNSUPPORTED;
    }
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse)) return FA_ERR_ALIGN;
    if (varlen && (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u)) return FA_ERR_ALIGN;
    const long long T = varlen ? (long long)N : (long long)B * N;
    if (T == 0) return FA_OK;
    if (T > 0x7fffffffLL || (long long)Hq * T > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;

    DeviceInfo* dev = nullptr;
    int rc = current_device_info(&dev);
    if (rc != FA_OK) return rc;

    // d = 64 runs on the ping-pong kernel.
    const bool pair = d == 128 && g_fwd_kernel == 2;
    FwdLaunch L;
    L.d = d;
    if (d == 256) {
        // One 128-row query tile per CTA, 64-key blocks (fa_fwd256.cu).
        if ((rc = make_map(&L.tq, q, Hq, T, kTileM, d)) != FA_OK) return rc;
        if ((rc = make_map(&L.tk, k, Hkv, T, 64, d)) != FA_OK) return rc;
        if ((rc = make_map(&L.tv, v, Hkv, T, 64, d)) != FA_OK) return rc;
    }
    // K boxes: 128 rows (the pair kernel loads a block's half); V boxes: 256
    // rows for the pair kernel (it loads 64 columns of each block's 256 keys).
    if (d != 256) {
        if ((rc = make_map(&L.tq, q, Hq, T, kTileM, d)) != FA_OK) return rc;
        if ((rc = make_map(&L.tk, k, Hkv, T, kTileM, d)) != FA_OK) return rc;
        if ((rc = make_map(&L.tv, v, Hkv, T, pair ? 256 : kTileM, d)) != FA_OK) return rc;
    }
    if (pair && (rc = make_map(&L.to, o, Hq, T)) != FA_OK) return rc;
    L.a.o = o;
    L.a.lse = lse;
    L.a.cu_seqlens = cu_seqlens;
    L.a.status = dev->status;
    L.a.B = B;
    L.a.Hq = Hq;
    L.a.Hkv = Hkv;
    L.a.N = N;
    L.a.causal = causal;
    L.a.varlen = varlen ? 1 : 0;
    L.a.max_seqlen = varlen ? max_seqlen : N;
    // Causal fixed length: (batch, head) pairs per L2 section so that the K/V
    // of one section (2 * N * d * 2 bytes per key/value head) fill about
    // half of L2; pairs of one group share their K/V head.
    {
        const long long kv_bytes = 4LL * d * (N > 0 ? N : 1);
        long long sec = (long long)(Hq / Hkv) * ((long long)dev->l2_bytes / 2) / kv_bytes;
        if (sec < 1) sec = 1;
        if (sec > (long long)B * Hq) sec = (long long)B * Hq;
        L.a.l2_section = (int)sec;
    }
    L.a.scale_log2 = alpha * 1.4426950408889634f;
    L.a.tau = g_tau;
    L.a.naive = g_naive;
    L.a.dbg_visits = g_dbg_visits;
    L.a.dbg_rescale = g_dbg_rescale;
    L.emu16 = g_emu16;
    L.num_sms = dev->num_sms;
    cudaError_t e = d == 256 ? launch_fwd256(L, stream)
                    : pair    ? launch_fwd_pair(L, stream)
                              : launch_fwd(L, stream);
    return e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

int fa_fwd_pairs_resident(void) { return g_pairs_resident; }

int fa_set_debug_counters(int* visits, int* inner, unsigned long long* rescales) {
    if ((reinterpret_cast<uintptr_t>(visits) & 3u) || (reinterpret_cast<uintptr_t>(inner) & 3u) ||
        (reinterpret_cast<uintptr_t>(rescales) & 7u))
        return FA_ERR_ALIGN;
    g_dbg_visits = visits;
    g_dbg_inner = inner;
    g_dbg_rescale = rescales;
    return FA_OK;
}

int fa_set_bwd_kernel(int kernel) {
    if (kernel < 0 || kernel > 1) return FA_ERR_INVALID;
    g_bwd_kernel = kernel;
    return FA_OK;
}

int fa_bwd_pairs_resident(void) { return g_bwd_pairs_resident; }

int fa_set_schedule_order(int order) {
    if (order < 0 || order > 1) return FA_ERR_INVALID;
    g_naive = order;
    return FA_OK;
}

int fa_set_fwd_kernel(int kernel) {
    if (kernel != 0 && kernel != 2) return FA_ERR_INVALID;
    g_fwd_kernel = kernel;
    return FA_OK;
}

static int read_and_clear(DevStatus* where) {
    DevStatus s;
    if (cudaMemcpy(&s, where, sizeof s, cudaMemcpyDeviceToHost) != cudaSuccess) return FA_ERR_LAUNCH;
    if (s.code == 0) return FA_OK;
    if (getenv("FA_LOG"))
        fprintf(stderr, "fa: device status %d at wait site %d (block %d)\n", s.code, s.where, s.block);
    DevStatus z = {0, 0, 0, 0};
    if (cudaMemcpy(where, &z, sizeof z, cudaMemcpyHostToDevice) != cudaSuccess) return FA_ERR_LAUNCH;
    return s.code;
}

// A backward workspace's status word; after a reported failure the main
// stage's unit claim counter is rewound too (a main kernel that gave up may
// leave it mid-list), so that a later main stage run without the preprocess
// starts from the first unit.
static int read_and_clear_ws(BwdHeader* h) {
    const int b = read_and_clear(&h->status);
    if (b != FA_OK && b != FA_ERR_LAUNCH) {
        const int zero[2] = {0, 0};
        if (cudaMemcpy(&h->next_unit, zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
            return FA_ERR_LAUNCH;
    }
    return b;
}

int fa_get_device_status(const void* workspace, cudaStream_t stream) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) return FA_ERR_LAUNCH;
    DeviceInfo* dev = nullptr;
    int rc = current_device_info(&dev);
    if (rc != FA_OK) return rc;
    int a = read_and_clear(dev->status);
    int b = FA_OK, c = FA_OK;
    if (workspace) b = read_and_clear_ws(static_cast<BwdHeader*>(const_cast<void*>(workspace)));
    // fa_bwd_noalloc's scratch area on this device, once a call has set it up.
    BwdHeader* nh = noalloc_header_current_device();
    if (nh && nh != workspace) c = read_and_clear_ws(nh);
    return a != FA_OK ? a : (b != FA_OK ? b : c);
}

size_t fa_bwd_workspace_size(int B, int Hq, int N, int d, int deterministic, int varlen) {
    if (B < 1 || Hq < 1 || N < 0 || (d != 128 && d != 64 && d != 256)) return 0;
    const long long T = varlen ? (long long)N : (long long)B * N;
    return ws_layout(T, B, Hq, deterministic ? 1 : 0, varlen ? 1 : 0, d).total;
}

}  // extern "C"

namespace fa {

int bwd_validate(const void* const ptrs[9], int B, int Hq, int Hkv, int N, int d, float alpha, int causal,
                 const int* cu_seqlens, int max_seqlen, int deterministic, long long* T_out) {
    for (int i = 0; i < 9; ++i)
        if (!ptrs[i]) return FA_ERR_INVALID;
    if (B < 1 || N < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0) return FA_ERR_INVALID;
    if (!(alpha > 0.0f) || !isfinite(alpha)) return FA_ERR_INVALID;
    if ((causal != 0 && causal != 1) || (deterministic != 0 && deterministic != 1)) return FA_ERR_INVALID;
    if (d != 128 && d != 64 && d != 256) return FA_ERR_UNSUPPORTED;
    const bool varlen = cu_seqlens != nullptr;
    if (varlen) {
        if (max_seqlen < 1) return FA_ERR_INVALID;
        if (B > kMaxVarlenSeqs || max_seqlen > 131072) return FA_ERR_UNSUPPORTED;
    }
    for (int i = 0; i < 9; ++i)
        if (!aligned16(ptrs[i])) return FA_ERR_ALIGN;
    if (varlen && (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u)) return FA_ERR_ALIGN;
    const long long T = varlen ? (long long)N : (long long)B * N;
    if (T > 0x7fffffffLL || (long long)Hq * T > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
    *T_out = T;
    return FA_OK;
}

}  // namespace fa

extern "C" {

int fa_bwd_stages(int stages, const void* q, const void* k, const void* v, const void* o, const float* lse,
                  const void* dout, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int N, int d, float alpha,
                  int causal, const int* cu_seqlens, int max_seqlen, int deterministic, void* workspace,
                  size_t workspace_bytes, cudaStream_t stream) {
    if (stages < 1 || stages > 7) return FA_ERR_INVALID;
    const void* ptrs[9] = {q, k, v, o, lse, dout, dq, dk, dv};
    long long T = 0;
    int rc = bwd_validate(ptrs, B, Hq, Hkv, N, d, alpha, causal, cu_seqlens, max_seqlen, deterministic, &T);
    if (rc != FA_OK) return rc;
    if (T == 0) return FA_OK;
    const bool varlen = cu_seqlens != nullptr;
    const WsLayout w = ws_layout(T, B, Hq, deterministic, varlen ? 1 : 0, d);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < w.total)
        return FA_ERR_WORKSPACE;

    DeviceInfo* dev = nullptr;
    if ((rc = current_device_info(&dev)) != FA_OK) return rc;
    BwdLaunch L;
    L.d = d;
    // Q and dO boxes: 128 rows (d = 256: 64-row query steps).
    const int qbox = d == 256 ? 64 : kTileM;
    if ((rc = make_map(&L.tq, q, Hq, T, qbox, d)) != FA_OK) return rc;
    if ((rc = make_map(&L.tk, k, Hkv, T, kTileM, d)) != FA_OK) return rc;
    if ((rc = make_map(&L.tv, v, Hkv, T, kTileM, d)) != FA_OK) return rc;
    if ((rc = make_map(&L.tdo, dout, Hq, T, qbox, d)) != FA_OK) return rc;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    // The fp32 dQ accumulator's map for the TMA reductions: boxes of 32
    // columns x 128 rows (d = 256: 32 rows).
    if ((rc = make_map_acc(&L.tdq, ws + w.dq_off, (long long)Hq * T, d == 256 ? 32 : kTileM, d)) != FA_OK) return rc;
    BwdArgs& a = L.a;
    a.o = o;
    a.dO = dout;
    a.lse = lse;
    a.dq = dq;
    a.dk = dk;
    a.dv = dv;
    a.cu_seqlens = cu_seqlens;
    a.hdr = reinterpret_cast<BwdHeader*>(ws);
    a.D = reinterpret_cast<float*>(ws + w.d_off);
    a.dqacc = reinterpret_cast<float*>(ws + w.dq_off);
    a.sem = reinterpret_cast<int*>(ws + w.sem_off);
    a.units = reinterpret_cast<int4*>(ws + w.unit_off);
    a.cu_s = reinterpret_cast<int*>(ws + w.cu_off);
    a.sem_stride = w.sem_stride;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.N = N;
    a.T = T;
    a.causal = causal;
    a.varlen = varlen ? 1 : 0;
    a.deterministic = deterministic;
    a.max_seqlen = varlen ? max_seqlen : N;
    a.alpha = alpha;
    a.scale_log2 = alpha * 1.4426950408889634f;
    a.naive = g_naive;
    a.dbg_visits = g_dbg_visits;
    a.dbg_inner = g_dbg_inner;
    L.num_sms = dev->num_sms;
    L.pair = d == 128 && g_bwd_kernel == 1 && bwd_pair_supported(a) ? 1 : 0;
    // Packed batches whose key/value heads serve many query heads (MQA-like):
    // the one-CTA kernel's work units cover kSplitHeads query heads each and
    // add their dK, dV into fp32 partial sums (atomic mode only, so that
    // deterministic mode keeps one unit per key tile and its fixed order).
    const int G = Hq / Hkv;
    a.kv_split = varlen && !deterministic && d != 256 && !L.pair && G >= kSplitMinGroup && G % kSplitHeads == 0
                     ? kSplitHeads : 0;
    a.dkvacc = varlen && d != 256 ? reinterpret_cast<float*>(ws + w.kv_off) : nullptr;
    if (a.kv_split) {
        if ((rc = make_map_acc(&L.tdkv, ws + w.kv_off, 2LL * Hkv * T, kTileM, d)) != FA_OK) return rc;
    } else {
        L.tdkv = L.tdq;   // not read
    }
    if (L.pair) {
        if ((rc = make_map(&L.tq64, q, Hq, T, 64)) != FA_OK) return rc;
        if ((rc = make_map(&L.tdo64, dout, Hq, T, 64)) != FA_OK) return rc;
        if ((rc = make_map_acc(&L.tdq64, ws + w.dq_off, (long long)Hq * T, 64)) != FA_OK) return rc;
    }
    cudaError_t e = launch_bwd(L, stages, stream);
    return e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout, void* dq,
           void* dk, void* dv, int B, int Hq, int Hkv, int N, int d, float alpha, int causal, const int* cu_seqlens,
           int max_seqlen, int deterministic, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    return fa_bwd_stages(7, q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, N, d, alpha, causal, cu_seqlens,
                         max_seqlen, deterministic, workspace, workspace_bytes, stream);
}

int fa_selftest_timeout(cudaStream_t stream) {
    DeviceInfo* dev = nullptr;
    int rc = current_device_info(&dev);
    if (rc != FA_OK) return rc;
    return launch_selftest_timeout(dev->status, stream) == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

int fa_exp2_emu(const float* x, float* y, int64_t n, cudaStream_t stream) {
    if (n < 0 || (n > 0 && (!x || !y))) return FA_ERR_INVALID;
    return launch_exp2_emu(x, y, n, stream) == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

}  // extern "C"
