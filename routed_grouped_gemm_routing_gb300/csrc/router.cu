// Router top-k gating: logits [T, E] FP32 -> topk_idx [T, k], topk_w [T, k]
// (the step in front of the layer: the Primus-Turbo "Mega MoE" README takes
// topk_idx / topk_weights from the router, "Key points"; the ROCm Primus MoE
// training guide's router computes them from the router logits).
//
// Per token: the k largest logits in decreasing order, equal logits in
// increasing expert id, a NaN logit ranked as -infinity; the weights are the
// softmax over the k selected logits (limit weights 1/n on the selected
// logits equal to an infinite maximum).
//
// One warp per token.  Lane l holds logits e = l, l + 32, ... (E <= 1024, so
// at most 32 per lane, in registers).  k passes each take the warp-wide best
// (logit, lower id) not yet taken by a butterfly of shuffles; the selected
// logits wait in shared memory for the softmax, whose sum is a fixed-order
// warp reduction (deterministic).
#include <math.h>

#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kRouterWarps = 8;

__device__ __forceinline__ float router_key(float v) { return isnan(v) ? -INFINITY : v; }

// a precedes b: larger key, or equal key and lower id
__device__ __forceinline__ bool precedes(float ka, int ia, float kb, int ib) {
    return ka > kb || (ka == kb && ia < ib);
}

__global__ void __launch_bounds__(32 * kRouterWarps) router_topk_kernel(const float* __restrict__ logits, int T,
                                                                        int E, int k, int32_t* __restrict__ topk_idx,
                                                                        float* __restrict__ topk_w) {
    extern __shared__ float sel_keys[];  // [kRouterWarps][k]
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    float* keys = sel_keys + (size_t)warp * k;
    const int per_lane = (E + 31) >> 5;
    for (long long t = (long long)blockIdx.x * kRouterWarps + warp; t < T; t += (long long)gridDim.x * kRouterWarps) {
        const float* row = logits + (size_t)t * E;
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int e = lane + 32 * i;
            v[i] = (i < per_lane && e < E) ? router_key(__ldg(row + e)) : -INFINITY;
        }
        uint32_t taken = 0;  // bit i: expert lane + 32 i is already selected (or does not exist)
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (!(i < per_lane && lane + 32 * i < E)) taken |= 1u << i;
        for (int j = 0; j < k; ++j) {
            // this lane's best untaken expert
            float bk = -INFINITY;
            int bi = 0x7fffffff;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int e = lane + 32 * i;
                if (!(taken >> i & 1u) && precedes(v[i], e, bk, bi)) {
                    bk = v[i];
                    bi = e;
                }
            }
            // the warp's best
#pragma unroll
            for (int s = 16; s >= 1; s >>= 1) {
                const float ok = __shfl_xor_sync(0xffffffffu, bk, s);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, s);
                if (precedes(ok, oi, bk, bi)) {
                    bk = ok;
                    bi = oi;
                }
            }
            if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
            if (lane == 0) {
                topk_idx[(size_t)t * k + j] = bi;
                keys[j] = bk;
            }
        }
        __syncwarp();
        // softmax over the selected keys; keys[0] is the largest
        const float m = keys[0];
        float part = 0.0f;
        if (isinf(m)) {
            for (int j = lane; j < k; j += 32) part += keys[j] == m ? 1.0f : 0.0f;
        } else {
            for (int j = lane; j < k; j += 32) part += expf(keys[j] - m);
        }
#pragma unroll
        for (int s = 16; s >= 1; s >>= 1) part += __shfl_xor_sync(0xffffffffu, part, s);
        for (int j = lane; j < k; j += 32) {
            const float num = isinf(m) ? (keys[j] == m ? 1.0f : 0.0f) : expf(keys[j] - m);
            topk_w[(size_t)t * k + j] = num / part;
        }
        __syncwarp();
    }
}

}  // namespace

int launch_router_topk(const float* logits, int T, int E, int k, int32_t* topk_idx, float* topk_w, int num_sms,
                       cudaStream_t st) {
    if (T == 0) return 0;
    const long long need = ((long long)T + kRouterWarps - 1) / kRouterWarps;
    const long long cap = (long long)num_sms * 8;
    const int blocks = (int)(need < cap ? need : cap);
    const size_t smem = sizeof(float) * (size_t)kRouterWarps * (size_t)k;  // <= 32 KiB for k <= 1024
    router_topk_kernel<<<blocks, 32 * kRouterWarps, smem, st>>>(logits, T, E, k, topk_idx, topk_w);
    return (int)cudaGetLastError();
}

}  // namespace moe
