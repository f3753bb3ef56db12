// FP8 forward of the layer (DeepGEMM Mega-MoE article, usage example:
// activations cast per token to FP8 with UE8M0 scale factors at a
// granularity of 32 elements before they are dispatched, and the weights
// transformed once for its low-precision kernel): the quantization kernels
// of the input and of the weights, and the instantiations of the two GEMMs
// on E4M3 operands.
#include "grouped_gemm_2sm.cuh"

namespace moe {
namespace {

// One warp per 256 consecutive elements of x (row-major [T, H], H a multiple
// of 32, so no 32-element group straddles two rows): lane l takes elements
// 8l..8l+7; the four lanes of a group combine their maxima by shuffles.
// Writes q[i] = E4M3(x[i] / 2^e) (round to nearest even, saturating) and
// sf[g] = e + 127.  HBM-bound: 2 bytes read and 33/32 bytes written per
// element.
__global__ void __launch_bounds__(256) quantize_fp8_kernel(const __nv_bfloat16* __restrict__ x, long long n,
                                                           uint8_t* __restrict__ q, uint8_t* __restrict__ sf) {
    const int lane = threadIdx.x & 31;
    const long long nchunk = (n + 255) / 256;
    const long long nwarps = (long long)gridDim.x * (blockDim.x >> 5);
    for (long long w = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); w < nchunk; w += nwarps) {
        const long long e0 = w * 256 + (long long)lane * 8;
        const bool ok = e0 < n;
        const uint4 raw = ok ? __ldg(reinterpret_cast<const uint4*>(x + e0)) : make_uint4(0u, 0u, 0u, 0u);
        float v[8];
        unpack_bf16x8(raw, v);
        float amax = 0.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(v[j]));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        const int e = fp8_group_exponent(amax);
        if (ok) {
            uint32_t word[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t acc = 0;
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const float2 f = make_float2(ldexpf(v[4 * h + 2 * j], -e), ldexpf(v[4 * h + 2 * j + 1], -e));
                    const __nv_fp8x2_storage_t two = __nv_cvt_float2_to_fp8x2(f, __NV_SATFINITE, __NV_E4M3);
                    acc |= (uint32_t)two << (16 * j);
                }
                word[h] = acc;
            }
            *reinterpret_cast<uint2*>(q + e0) = make_uint2(word[0], word[1]);
            if ((lane & 3) == 0) sf[e0 >> 5] = (uint8_t)(e + 127);
        }
    }
}

// The inverse: x_out[i] = decode(q[i]) * 2^(sf[g] - 127) as bf16 (exact), one
// thread per 8 elements.
__global__ void __launch_bounds__(256) dequantize_fp8_kernel(const uint8_t* __restrict__ q,
                                                             const uint8_t* __restrict__ sf, long long n,
                                                             __nv_bfloat16* __restrict__ out) {
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i * 8 < n; i += stride) {
        const long long e0 = i * 8;
        const uint2 raw = __ldg(reinterpret_cast<const uint2*>(q + e0));
        const float sc = fp8_scale(__ldg(sf + (e0 >> 5)));
        uint4 o;
        o.x = e4m3x2_to_bf16x2(raw.x & 0xffffu, sc);
        o.y = e4m3x2_to_bf16x2(raw.x >> 16, sc);
        o.z = e4m3x2_to_bf16x2(raw.y & 0xffffu, sc);
        o.w = e4m3x2_to_bf16x2(raw.y >> 16, sc);
        *reinterpret_cast<uint4*>(out + e0) = o;
    }
}

// A weight tensor W [E][K][C] bf16 (K the contraction index of its GEMM) to
// E4M3, one scale per 32 consecutive k of a column, written K-major as
// q[E][C][K] with the scale bytes in the GEMM's atom layout: for column c
// in atom group g at atom row r, K group j32 = k / 32, block kb = j32 / 4
// and step j = j32 % 4: byte ((e G + g) (K / 128) + kb) 512 + 16 (r % 32) +
// 4 (r / 32) + j, G groups per expert.
//   W1 [E][H][2I] (kW1): column f (gate f < I, up I + f') has g = (f mod I)
//     / 64, r = 64 (f >= I) + (f mod I) % 64, G = I / 64 (a CTA of the L1
//     GEMM holds 64 gate and the matching 64 up features);
//   W2 [E][I][H]: column h has g = h / 128, r = h % 128, G = H / 128.
// One block of 128 threads per 32 rows of k x 128 columns: the tile comes in
// coalesced through shared memory and each thread quantizes one column's
// group.  The same rule as the input (smallest power of two with 448 2^e >=
// max|group|, round to nearest even, saturate).
template <bool kW1>
__global__ void __launch_bounds__(128) quantize_w_fp8_kernel(const __nv_bfloat16* __restrict__ W, int E, int K, int C,
                                                             uint8_t* __restrict__ q, uint8_t* __restrict__ atoms) {
    __shared__ __align__(16) __nv_bfloat16 tile[32][128];
    const int ncol = C / 128, nrow = K / 32, nkb = K / 128;
    const int I = C / 2;  // kW1 only
    const long long ntiles = (long long)E * nrow * ncol;
    const int tid = threadIdx.x;
    for (long long ti = blockIdx.x; ti < ntiles; ti += gridDim.x) {
        const int cb = (int)(ti % ncol);
        const int kr = (int)((ti / ncol) % nrow);
        const int e = (int)(ti / ((long long)ncol * nrow));
        const int c0 = cb * 128, k0 = kr * 32;
        __syncthreads();  // the previous tile has been read
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int ch = tid + 128 * i;  // 16-byte chunk: row ch / 16, columns 8 (ch % 16)
            const int rr = ch >> 4, cc = (ch & 15) * 8;
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(W + ((size_t)e * K + k0 + rr) * (size_t)C + c0 + cc));
            *reinterpret_cast<uint4*>(&tile[rr][cc]) = v;
        }
        __syncthreads();
        float v[32];
        float amax = 0.0f;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            v[j] = __bfloat162float(tile[j][tid]);
            amax = fmaxf(amax, fabsf(v[j]));
        }
        const int ex = fp8_group_exponent(amax);
        uint32_t w[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            uint32_t acc = 0;
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                const float2 f = make_float2(ldexpf(v[4 * j + 2 * m], -ex), ldexpf(v[4 * j + 2 * m + 1], -ex));
                acc |= (uint32_t)__nv_cvt_float2_to_fp8x2(f, __NV_SATFINITE, __NV_E4M3) << (16 * m);
            }
            w[j] = acc;
        }
        const int c = c0 + tid;
        uint8_t* dst = q + ((size_t)e * (size_t)C + c) * (size_t)K + k0;
        reinterpret_cast<uint4*>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
        reinterpret_cast<uint4*>(dst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
        int g, r, G;
        if constexpr (kW1) {
            const int fi = c < I ? c : c - I;
            g = fi >> 6;
            r = (c < I ? 0 : 64) + (fi & 63);
            G = I / 64;
        } else {
            g = c >> 7;
            r = c & 127;
            G = C / 128;
        }
        const int kb = kr >> 2, js = kr & 3;
        atoms[(((size_t)e * G + g) * nkb + kb) * 512 + 16 * (r & 31) + 4 * (r >> 5) + js] = (uint8_t)(ex + 127);
    }
}

}  // namespace

int launch_quantize_w1_fp8(const __nv_bfloat16* W1, int E, int H, int I, uint8_t* q, uint8_t* atoms, int num_sms,
                           cudaStream_t st) {
    const long long ntiles = (long long)E * (H / 32) * (2 * I / 128);
    if (ntiles <= 0) return 0;
    const long long cap = (long long)num_sms * 16;
    quantize_w_fp8_kernel<true><<<(unsigned)(ntiles < cap ? ntiles : cap), 128, 0, st>>>(W1, E, H, 2 * I, q, atoms);
    return (int)cudaGetLastError();
}

int launch_quantize_w2_fp8(const __nv_bfloat16* W2, int E, int H, int I, uint8_t* q, uint8_t* atoms, int num_sms,
                           cudaStream_t st) {
    const long long ntiles = (long long)E * (I / 32) * (H / 128);
    if (ntiles <= 0) return 0;
    const long long cap = (long long)num_sms * 16;
    quantize_w_fp8_kernel<false><<<(unsigned)(ntiles < cap ? ntiles : cap), 128, 0, st>>>(W2, E, I, H, q, atoms);
    return (int)cudaGetLastError();
}

int launch_dequantize_fp8(const uint8_t* q, const uint8_t* sf, long long n, __nv_bfloat16* out, int num_sms,
                          cudaStream_t st) {
    if (n <= 0) return 0;
    long long blocks = (n / 8 + 255) / 256;
    const long long cap = (long long)num_sms * 8;
    if (blocks > cap) blocks = cap;
    dequantize_fp8_kernel<<<(unsigned)blocks, 256, 0, st>>>(q, sf, n, out);
    return (int)cudaGetLastError();
}

int launch_quantize_fp8(const __nv_bfloat16* x, long long n, uint8_t* q, uint8_t* sf, int num_sms, cudaStream_t st) {
    if (n <= 0) return 0;
    const long long nchunk = (n + 255) / 256;
    long long blocks = (nchunk + 7) / 8;
    const long long cap = (long long)num_sms * 8;
    if (blocks > cap) blocks = cap;
    quantize_fp8_kernel<<<(unsigned)blocks, 256, 0, st>>>(x, n, q, sf);
    return (int)cudaGetLastError();
}

// L1 GEMM + SwiGLU on E4M3 weights and gathered E4M3 rows (block-scaled MMA)
int launch_gemm_l1_fwd_mx(const GemmArgs& a, const GemmMaps& m, int max_units, cudaStream_t st) {
    return launch_gemm_pair<L1_FWD_MX>(a, m, max_units, st);
}

// L2 GEMM + top-k weights on E4M3 W2 and the E4M3 rows of a (block-scaled MMA)
int launch_gemm_l2_fwd_mx(const GemmArgs& a, const GemmMaps& m, int max_units, cudaStream_t st) {
    return launch_gemm_pair<L2_FWD_MX>(a, m, max_units, st);
}

}  // namespace moe
