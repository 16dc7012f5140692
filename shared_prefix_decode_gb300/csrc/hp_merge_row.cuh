// hp_merge_row.cuh -- exact log-sum-exp merge of the partial attention
// states of one output row by one warp (the merge kernel's row body).
//
// Each output row (b, h) has a fixed, ordered list of partial states (O_i
// normalised over its own keys, LSE_i); the merge is Hydragen Eq. 5 applied
// to all of them in its max-subtracted form (combine_lse):
//   M = max_i LSE_i;  w_i = e^(LSE_i - M);  O = sum_i w_i O_i / sum_i w_i;
//   LSE = M + ln sum_i w_i.
// An empty part has LSE = -inf and weight exactly 0; a row with no parts, or
// only empty ones, gets O = 0 and LSE = -inf.  The parts are taken in their
// fixed order, so the result is deterministic.
//
// Partial rows are read through L2 only (ld.global.cg): other SMs wrote them,
// and an L1 line of the same workspace address could still hold an earlier
// step's row.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "hp_internal.h"
#include "hp_ptx.cuh"

namespace hp {
namespace mrg {

constexpr float kLog2e = 1.4426950408889634f;

// Where the merged row goes.
struct RowOut {
    void *out;        // bf16 or f32 row of d values
    int out_f32;
    float *lse;       // may be null
};

// One warp merges the n parts of a row.  Lane l holds the partial rows of
// parts l and l + 32 in pr_a / pr_b; far(e) gives the row of part e >= 64.
// Load instructions and round trips, not bytes, bound this code, so the
// first kFirst = kUnroll * 32 / (D / 8) parts are fetched in one round:
//   - lane e loads the LSE of part e (one instruction per 32 parts);
//   - the O rows are read 16 bytes (8 columns) per lane, 32 / (D / 8) parts
//     per instruction, each lane holding its own part's slice;
// then the max and the denominator are warp reductions and each lane weights
// its part; the part groups are summed by shuffles at the end.  Further
// parts (rows with more than kFirst) take further rounds.  The sums run over
// the parts in a fixed lane order, so the result is deterministic.
template <int D, int kUnroll, class Far>
__device__ __forceinline__ void merge_row(const uint16_t *part_o, const float *part_lse, int n, int pr_a, int pr_b,
                                          const Far &far, int lane, const RowOut &o)
{
    constexpr int kLpp = D / 8;      // lanes per part row (8 bf16 columns each)
    constexpr int kPpi = 32 / kLpp;  // parts per load instruction
    const int sub = lane / kLpp;     // which part of an instruction's group
    const int col = (lane % kLpp) * 8;
    // one round: every LSE of the first 64 parts and the O slices of the
    // first kUnroll * kPpi parts
    const float la = lane < n ? __ldcg(part_lse + pr_a) : -INFINITY;
    const float lb = lane + 32 < n ? __ldcg(part_lse + pr_b) : -INFINITY;
    uint4 x[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
        const int e = u * kPpi + sub;
        const int pr = __shfl_sync(0xffffffffu, e < 32 ? pr_a : pr_b, e & 31);
        x[u] = e < n ? __ldcg(reinterpret_cast<const uint4 *>(part_o + (size_t)pr * D + col))
                     : make_uint4(0u, 0u, 0u, 0u);
    }
    float M = fmaxf(la, lb);
    for (int e = lane + 64; e < n; e += 32)
        M = fmaxf(M, __ldcg(part_lse + far(e)));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    const float Ms = M == -INFINITY ? 0.f : M;  // no part has any weight
    const float wa = fast_exp2((la - Ms) * kLog2e), wb = fast_exp2((lb - Ms) * kLog2e);  // 0 for empty parts
    float den = wa + wb;
    for (int e = lane + 64; e < n; e += 32)
        den += fast_exp2((__ldcg(part_lse + far(e)) - Ms) * kLog2e);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        den += __shfl_xor_sync(0xffffffffu, den, off);
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        acc[i] = 0.f;
    auto add = [&](const uint4 &xv, float w) {
        acc[0] = fmaf(w, bf16lo_to_f32(xv.x), acc[0]);
        acc[1] = fmaf(w, bf16hi_to_f32(xv.x), acc[1]);
        acc[2] = fmaf(w, bf16lo_to_f32(xv.y), acc[2]);
        acc[3] = fmaf(w, bf16hi_to_f32(xv.y), acc[3]);
        acc[4] = fmaf(w, bf16lo_to_f32(xv.z), acc[4]);
        acc[5] = fmaf(w, bf16hi_to_f32(xv.z), acc[5]);
        acc[6] = fmaf(w, bf16lo_to_f32(xv.w), acc[6]);
        acc[7] = fmaf(w, bf16hi_to_f32(xv.w), acc[7]);
    };
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
        const int e = u * kPpi + sub;
        const float w = __shfl_sync(0xffffffffu, e < 32 ? wa : wb, e & 31);
        add(x[u], e < n ? w : 0.f);
    }
    // rows with more parts: one more round per kPpi parts
    for (int e0 = kUnroll * kPpi; e0 < n; e0 += kPpi) {
        const int e = e0 + sub;
        const int src = e & 31;
        int pr = __shfl_sync(0xffffffffu, e < 32 ? pr_a : pr_b, src);
        float w = __shfl_sync(0xffffffffu, e < 32 ? wa : wb, src);
        if (e < n) {
            if (e >= 64) {
                pr = far(e);
                w = fast_exp2((__ldcg(part_lse + pr) - Ms) * kLog2e);
            }
            add(__ldcg(reinterpret_cast<const uint4 *>(part_o + (size_t)pr * D + col)), w);
        }
    }
#pragma unroll
    for (int off = kLpp; off < 32; off <<= 1)
#pragma unroll
        for (int i = 0; i < 8; ++i)
            acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], off);
    const float inv = den > 0.f ? 1.f / den : 0.f;
    if (lane < kLpp) {
        if (o.out_f32) {
            float *dst = reinterpret_cast<float *>(o.out) + col;
#pragma unroll
            for (int i = 0; i < 8; i += 2)
                *reinterpret_cast<float2 *>(dst + i) = make_float2(acc[i] * inv, acc[i + 1] * inv);
        } else {
            __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(o.out) + col;
#pragma unroll
            for (int i = 0; i < 8; i += 2)
                *reinterpret_cast<__nv_bfloat162 *>(dst + i) = __floats2bfloat162_rn(acc[i] * inv, acc[i + 1] * inv);
        }
    }
    if (lane == 0 && o.lse != nullptr)
        *o.lse = den > 0.f ? M + __logf(den) : -INFINITY;
}

}  // namespace mrg
}  // namespace hp
