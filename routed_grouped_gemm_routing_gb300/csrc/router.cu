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
// One warp per token.  Lane l holds logits e = l, l + 32, ... in registers:
// P per lane, P the power of two with 32 (P / 2) < E <= 32 P (E <= 1024, so
// P <= 32), one instantiation per P so that a lane scans only its own
// logits.  k passes each take the warp-wide best (logit, lower id) not yet
// taken by two warp reductions; the selected logits wait in shared
// memory for the softmax, whose sum is a fixed-order warp reduction
// (deterministic).
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

// Order-preserving code of a key (never NaN): a larger key has a larger
// code; -0 and +0 share one code, being equal keys.  key_of inverts it (a
// zero comes back as +0).
__device__ __forceinline__ uint32_t key_code(float f) {
    const uint32_t u = __float_as_uint(f == 0.0f ? 0.0f : f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_of(uint32_t c) {
    return __uint_as_float((c & 0x80000000u) ? (c & 0x7fffffffu) : ~c);
}

template <int P>
__global__ void __launch_bounds__(32 * kRouterWarps)
    router_topk_kernel(const float* __restrict__ logits, int T, int E, int k, int32_t* __restrict__ topk_idx,
                       float* __restrict__ topk_w) {
    extern __shared__ float sel_keys[];  // [kRouterWarps][k]
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    float* keys = sel_keys + (size_t)warp * k;
    for (long long t = (long long)blockIdx.x * kRouterWarps + warp; t < T; t += (long long)gridDim.x * kRouterWarps) {
        const float* row = logits + (size_t)t * E;
        float v[P];
#pragma unroll
        for (int i = 0; i < P; ++i) {
            const int e = lane + 32 * i;
            v[i] = e < E ? router_key(__ldg(row + e)) : -INFINITY;
        }
        uint32_t taken = 0;  // bit i: expert lane + 32 i is already selected (or does not exist)
#pragma unroll
        for (int i = 0; i < P; ++i)
            if (lane + 32 * i >= E) taken |= 1u << i;
        for (int j = 0; j < k; ++j) {
            // this lane's best untaken expert
            float bk = -INFINITY;
            int bi = 0x7fffffff;
#pragma unroll
            for (int i = 0; i < P; ++i) {
                const int e = lane + 32 * i;
                if (!(taken >> i & 1u) && precedes(v[i], e, bk, bi)) {
                    bk = v[i];
                    bi = e;
                }
            }
            // the warp's best: the largest key, then the lowest id holding it
            // (a lane with nothing left offers -inf and an id above any expert)
            const uint32_t code = key_code(bk);
            const uint32_t wcode = __reduce_max_sync(0xffffffffu, code);
            const int wid = (int)__reduce_min_sync(0xffffffffu, code == wcode ? (uint32_t)bi : 0xffffffffu);
            if ((wid & 31) == lane) taken |= 1u << (wid >> 5);
            if (lane == 0) {
                topk_idx[(size_t)t * k + j] = wid;
                keys[j] = key_of(wcode);
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
    const int per_lane = (E + 31) >> 5;
    if (per_lane <= 1)
        router_topk_kernel<1><<<blocks, 32 * kRouterWarps, smem, st>>>(logits, T, E, k, topk_idx, topk_w);
    else if (per_lane <= 2)
        router_topk_kernel<2><<<blocks, 32 * kRouterWarps, smem, st>>>(logits, T, E, k, topk_idx, topk_w);
    else if (per_lane <= 4)
        router_topk_kernel<4><<<blocks, 32 * kRouterWarps, smem, st>>>(logits, T, E, k, topk_idx, topk_w);
    else if (per_lane <= 8)
        router_topk_kernel<8><<<blocks, 32 * kRouterWarps, smem, st>>>(logits, T, E, k, topk_idx, topk_w);
    else if (per_lane <= 16)
        router_topk_kernel<16><<<blocks, 32 * kRouterWarps, smem, st>>>(logits, T, E, k, topk_idx, topk_w);
    else if (per_lane <= 32)
        router_topk_kernel<32><<<blocks, 32 * kRouterWarps, smem, st>>>(logits, T, E, k, topk_idx, topk_w);
    else
        return (int)cudaErrorInvalidValue;
    return (int)cudaGetLastError();
}

}  // namespace moe
