// hp_host_io_kernel.cu -- the copy-in of a cascade step whose queries are in
// page-locked host memory (hp_cascade_decode_host): the B x Hq query rows are
// read over the host link and stored, contiguous, in the workspace, where the
// step's persistent kernel reads them.
//
// Launched as a programmatic dependent of the kernel before it in the stream
// (the previous step's merge): each thread issues its host reads first, so
// their latency overlaps that kernel's tail, then waits for it to complete
// before it overwrites the staging rows (the previous step read them).  The
// step's persistent kernel may start setting up as soon as every CTA here has
// started, and waits for this grid to complete before it reads q.
#include <cuda_runtime.h>

#include "hp_internal.h"

namespace hp {

namespace {

constexpr int kStageThreads = 256;
constexpr int kStagePer = 2;  // 16-byte pieces per thread, loaded together

__global__ void __launch_bounds__(kStageThreads) hp_stage_kernel(const __grid_constant__ StageParams p)
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int per_row = p.d / 8;
    const int64_t n = (int64_t)p.B * p.Hq * per_row;
    uint4 v[kStagePer];
    int64_t idx[kStagePer];
#pragma unroll
    for (int u = 0; u < kStagePer; ++u) {
        idx[u] = ((int64_t)blockIdx.x * kStagePer + u) * kStageThreads + threadIdx.x;
        if (idx[u] < n) {
            const int64_t row = idx[u] / per_row;
            const int c = (int)(idx[u] - row * per_row);
            const int64_t b = row / p.Hq, h = row - b * p.Hq;
            v[u] = *reinterpret_cast<const uint4 *>(p.src + b * p.sb + h * p.sh + c * 8);
        }
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
#pragma unroll
    for (int u = 0; u < kStagePer; ++u)
        if (idx[u] < n)
            reinterpret_cast<uint4 *>(p.dst)[idx[u]] = v[u];
}

}  // namespace

cudaError_t launch_stage(const StageParams &p, cudaStream_t s)
{
    const int64_t n = (int64_t)p.B * p.Hq * (p.d / 8);
    if (n <= 0)
        return cudaSuccess;
    const int64_t per_cta = (int64_t)kStageThreads * kStagePer;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((n + per_cta - 1) / per_cta));
    cfg.blockDim = dim3(kStageThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, hp_stage_kernel, p);
}

}  // namespace hp
