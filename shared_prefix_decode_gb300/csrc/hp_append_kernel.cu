// hp_append_kernel.cu -- the decode loop's KV append: each sequence's new key
// and value rows go to the next free slot of its private suffix, then the
// suffix length moves on by one.
//
// During autoregressive decoding every step adds one token per sequence to
// that sequence's suffix, and the next step attends over it (Hydragen,
// "Inter-Sequence Batched Prefix Attention", on autoregressive decoding).  The
// suffix pages are reserved up to a fixed capacity when the loop plan is
// built, and the current length lives on the device, so the step is the same
// launch every time and a whole loop can be one CUDA graph (Hydragen,
// "Implementation Details", attention primitives).
//
// One CTA per sequence: thread 0 reads the length and the page of the free
// slot, the CTA copies Hkv x d bf16 of K and of V in 16-byte pieces, and
// thread 0 then stores the new length.  Each CTA owns its sequence's length,
// so no two CTAs touch the same word.
#include <cuda_runtime.h>

#include "hp_internal.h"

namespace hp {

namespace {

constexpr int kAppendThreads = 128;

__global__ void __launch_bounds__(kAppendThreads) hp_append_kernel(const __grid_constant__ AppendParams p)
{
    // Launched as a programmatic dependent of the kernel before it (the
    // previous step's merge).  The decode step that follows may start setting
    // up at once; it waits for this grid to complete before it reads the
    // lengths or the pools.  This grid waits for the one before it, and so
    // for everything earlier in the stream, before touching them.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    __shared__ int s_pos, s_page;
    const int b = blockIdx.x;
    if (threadIdx.x == 0) {
        const int pos = p.suffix_len[b];
        int page = -1;
        if (pos >= 0 && pos < p.capacity) {
            const int pid = p.leaf_tab[(int64_t)b * p.leaf_stride + pos / p.page_size];
            if (pid >= 0 && pid < p.num_pages)
                page = pid;
        }
        if (page < 0)
            atomicOr(p.status, kStBounds);
        s_pos = pos;
        s_page = page;
    }
    __syncthreads();
    const int page = s_page, pos = s_pos;
    if (page < 0)
        return;  // the whole CTA: nothing written, the length kept
    const int per_row = p.d / 8;  // 16-byte pieces of one head's row
    const int n = p.Hkv * per_row;
    const int64_t slot = pos % p.page_size;
    for (int i = threadIdx.x; i < 2 * n; i += kAppendThreads) {
        const bool is_v = i >= n;
        const int j = is_v ? i - n : i;
        const int h = j / per_row, c = j % per_row;
        const uint16_t *src = (is_v ? p.v_new : p.k_new) + (int64_t)b * p.kv_sb + (int64_t)h * p.kv_sh + c * 8;
        uint16_t *dst = (is_v ? p.v_pool : p.k_pool) +
                        (((int64_t)page * p.Hkv + h) * p.page_size + slot) * p.d + c * 8;
        *reinterpret_cast<uint4 *>(dst) = *reinterpret_cast<const uint4 *>(src);
    }
    __syncthreads();
    if (threadIdx.x == 0)
        p.suffix_len[b] = pos + 1;
}

}  // namespace

cudaError_t launch_append(const AppendParams &p, cudaStream_t s)
{
    if (p.B <= 0)
        return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.B);
    cfg.blockDim = dim3(kAppendThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, hp_append_kernel, p);
}

}  // namespace hp
