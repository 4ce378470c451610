// fa_internal.h -- host-side structures shared by the C-ABI layer and the
// kernel translation units of libfa.so (not installed, not part of the ABI).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "fa_prim.cuh"

namespace fa {

constexpr int kHeadDim = 128;
constexpr int kTileM = 128;             // query rows per Q tile (one TMEM lane per row)
constexpr int kTileN = 128;             // keys per K/V tile
constexpr int kUnitRows = 2 * kTileM;   // two Q tiles (ping-pong) per forward work unit
constexpr int kMaxVarlenSeqs = 1024;    // sequences a varlen call may pack
constexpr int kMaxUnitLevels = 512;     // ceil(max_seqlen / 256) limit (max_seqlen <= 131072)

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
};

struct FwdLaunch {
    CUtensorMap tq, tk, tv;  // 3-D maps {128, H, T}, box {64, 1, 128}, 128-B swizzle
    FwdArgs a;
    int emu_eighths;         // 0..4: share of exp2 pairs on the FMA pipe, in eighths
    int num_sms;
};

// Launch the forward kernel (fa_fwd.cu).  Returns a cudaError_t.
cudaError_t launch_fwd(const FwdLaunch& L, cudaStream_t stream);

// Evaluate the FMA-pipe exp2 on n floats (fa_fwd.cu).
cudaError_t launch_exp2_emu(const float* x, float* y, int64_t n, cudaStream_t stream);

// The library's device status word on the current device.
DevStatus* device_status_ptr();

}  // namespace fa
