// fa_noalloc.cu -- fa_bwd_noalloc: the backward for callers that cannot
// allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they need the
// gradients: code running inside a CUDA-graph-building framework or a custom
// allocator's hooks, embedded runtimes that own every device allocation
// themselves, or plugins whose host application forbids allocation after
// start-up.  fa_bwd needs a caller-provided workspace for its fp32 dQ
// accumulator, the D rows and the varlen work list; this variant instead uses
// one fixed scratch area compiled into the library as a file-scope device
// array.  The caller still passes every input and output tensor.
//
// The scratch array is ordinary static device storage: every GPU that loads
// this library reserves kNoAllocScratchBytes for it until the process exits.
// Host code cannot use the array's name as a device address (in host code it
// names a host-side stand-in), so the device address is taken with
// cudaGetSymbolAddress once per device, with that device current, on the
// first call made on that device.
#include <mutex>

#include "../../include/fa.h"
#include "fa_internal.h"

namespace fa {
namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)64 << 20;  // 64 MiB per device

static __device__ __align__(256) uint8_t g_bwd_scratch[kNoAllocScratchBytes];

constexpr int kMaxScratchDevices = 64;
void* g_scratch_addr[kMaxScratchDevices];
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device (set-up on first use).
int scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxScratchDevices) return FA_ERR_LAUNCH;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress((void**)&p, g_bwd_scratch) != cudaSuccess || p == nullptr) return FA_ERR_LAUNCH;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return FA_OK;
}

}  // namespace

BwdHeader* noalloc_header_current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxScratchDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    return static_cast<BwdHeader*>(g_scratch_addr[dev]);
}

}  // namespace fa

extern "C" int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                              const void* dout, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int N, int d,
                              float alpha, int causal, const int* cu_seqlens, int max_seqlen, int deterministic,
                              cudaStream_t stream) {
    // fa_bwd's own checks first, so that both entry points return the same
    // code for the same arguments; then the size limit of the scratch area.
    const void* ptrs[9] = {q, k, v, o, lse, dout, dq, dk, dv};
    long long T = 0;
    const int vrc = fa::bwd_validate(ptrs, B, Hq, Hkv, N, d, alpha, causal, cu_seqlens, max_seqlen, deterministic, &T);
    if (vrc != FA_OK) return vrc;
    if (T == 0) return FA_OK;
    const size_t need = fa_bwd_workspace_size(B, Hq, N, d, deterministic, cu_seqlens ? 1 : 0);
    if (need == 0) return FA_ERR_INVALID;
    if (need > fa::kNoAllocScratchBytes) return FA_ERR_WORKSPACE;
    void* scratch = nullptr;
    const int rc = fa::scratch_address(&scratch);
    if (rc != FA_OK) return rc;
    // Every call reuses the same scratch; fa_bwd's first stage re-zeroes the
    // parts that must start at zero (status word, dQ accumulator, semaphores).
    return fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, N, d, alpha, causal, cu_seqlens, max_seqlen,
                  deterministic, scratch, fa::kNoAllocScratchBytes, stream);
}
