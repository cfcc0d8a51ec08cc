// Internal (non-ABI) declarations shared by the C-ABI layer and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "fa_geom.h"

namespace fa {

// Status codes written by kernels into the device status word.
enum DeviceStatus { DEV_OK = 0, DEV_TIMEOUT = 1 };

// Parameters of the tensor-core kernel (passed as one __grid_constant__).
struct TcParams {
    CUtensorMap tm_q;   // 3-D maps over [B*H, N, D] 16-bit, box {64, 128, 1}, 128B swizzle
    CUtensorMap tm_k;
    CUtensorMap tm_v;
    void* o;            // [B*H, N, D], 16-bit or fp32 (o_f32)
    float* lse;         // [B*H, N] or null
    Geom g;
    int BH;
    int n_units;
    int order;
    float scale_log2;   // scale * log2(e)
    int o_f32;
    unsigned long long wait_limit_ns;
    int* status;        // device status word
};

struct SimtParams {
    const float* q;
    const float* k;
    const float* v;
    float* o;
    float* lse;
    Geom g;
    int BH;
    int D;
    float scale;
};

// Launchers (return the CUDA error of the launch, if any).
cudaError_t launch_tc(const TcParams& p, int D, bool bf16, bool pos_scale, int grid, cudaStream_t s);
cudaError_t launch_simt_f32(const SimtParams& p, cudaStream_t s);
cudaError_t launch_selftest_timeout(int* status, unsigned long long limit_ns, cudaStream_t s);

}  // namespace fa
