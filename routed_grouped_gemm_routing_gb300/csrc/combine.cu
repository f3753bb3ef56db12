// Combine kernels: the per-token reduction over the k routed contributions
// (Primus-Turbo "Mega MoE" README, "Pipeline": the top-k reduce that sums the
// num_topk contributions per token; in backward the same reduction gathers
// the per-row gradients of the dispatched x back to tokens).  On one GPU the
// cross-rank push becomes a read of the token's k padded rows through the
// inverse permutation.  Sums are FP32 in slot order j = 0..k-1, rounded once
// to bf16: deterministic, no atomics.
#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {

namespace {

// dst[t, :] = sum_j rows[inv[t*k + j], :]   (dropped slots add nothing)
// One thread per 16-byte chunk (8 columns) of a token row; consecutive
// threads cover consecutive chunks, so every row read is coalesced.
__global__ void __launch_bounds__(256) combine_kernel(const __nv_bfloat16* __restrict__ rows,
                                                      const int32_t* __restrict__ inv, int T, int k, int H,
                                                      __nv_bfloat16* __restrict__ dst) {
    const int cpr = H / 8;
    const long long total = (long long)T * cpr;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int t = (int)(i / cpr);
        const int c = (int)(i - (long long)t * cpr);
        float acc[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
        const int32_t* iv = inv + (size_t)t * k;
        int j = 0;
        // four independent row loads in flight per step
        for (; j + 4 <= k; j += 4) {
            int r[4];
            uint4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) r[u] = __ldg(iv + j + u);
#pragma unroll
            for (int u = 0; u < 4; ++u)
                v[u] = r[u] >= 0 ? __ldg(reinterpret_cast<const uint4*>(rows + (size_t)r[u] * H) + c) : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                float f[8];
                unpack_bf16x8(v[u], f);
#pragma unroll
                for (int q = 0; q < 8; ++q) acc[q] += f[q];
            }
        }
        for (; j < k; ++j) {
            const int r = __ldg(iv + j);
            if (r >= 0) {
                float f[8];
                unpack_bf16x8(__ldg(reinterpret_cast<const uint4*>(rows + (size_t)r * H) + c), f);
#pragma unroll
                for (int q = 0; q < 8; ++q) acc[q] += f[q];
            }
        }
        uint4 o;
        o.x = pack_bf16x2(acc[0], acc[1]);
        o.y = pack_bf16x2(acc[2], acc[3]);
        o.z = pack_bf16x2(acc[4], acc[5]);
        o.w = pack_bf16x2(acc[6], acc[7]);
        reinterpret_cast<uint4*>(dst + (size_t)t * H)[c] = o;
    }
}

// out[s] = sum_n dw_part[inv[s], n]  in n order (0 for a dropped slot):
// the gradient of the layer output with respect to topk_weights[s].
__global__ void __launch_bounds__(256) dw_reduce_kernel(const float* __restrict__ dw_part, int cols,
                                                        const int32_t* __restrict__ inv, long long slots,
                                                        float* __restrict__ out) {
    for (long long s = (long long)blockIdx.x * blockDim.x + threadIdx.x; s < slots;
         s += (long long)gridDim.x * blockDim.x) {
        const int r = __ldg(inv + s);
        float v = 0.0f;
        if (r >= 0)
            for (int n = 0; n < cols; ++n) v += __ldg(dw_part + (size_t)r * cols + n);
        out[s] = v;
    }
}

}  // namespace

int launch_combine(const __nv_bfloat16* rows, const int32_t* inv, int T, int k, int H, __nv_bfloat16* out,
                   int num_sms, cudaStream_t st) {
    const long long total = (long long)T * (H / 8);
    if (total == 0) return 0;
    long long blocks = (total + 255) / 256;
    const long long cap = (long long)num_sms * 8;
    if (blocks > cap) blocks = cap;
    combine_kernel<<<(int)blocks, 256, 0, st>>>(rows, inv, T, k, H, out);
    return (int)cudaGetLastError();
}

int launch_dw_reduce(const float* dw_part, int cols, const int32_t* inv, long long slots, float* out, int num_sms,
                     cudaStream_t st) {
    if (slots == 0) return 0;
    long long blocks = (slots + 255) / 256;
    const long long cap = (long long)num_sms * 4;
    if (blocks > cap) blocks = cap;
    dw_reduce_kernel<<<(int)blocks, 256, 0, st>>>(dw_part, cols, inv, slots, out);
    return (int)cudaGetLastError();
}

}  // namespace moe
