// FP8 forward of the layer (DeepGEMM Mega-MoE article, usage example:
// activations cast per token to FP8 with UE8M0 scale factors at a
// granularity of 32 elements before they are dispatched, and the weights
// transformed once for its low-precision kernel): the quantization kernels
// of the input and of the weights, and the instantiations of the two GEMMs
// on E4M3 operands.
#include <climits>

#include "grouped_gemm_2sm.cuh"

namespace moe {
namespace {

// 2^-e for a group exponent e in [-127, 127] (the subnormal 2^-127 for e =
// 127): x times it is exact up to the one rounding of x / 2^e, the value
// ldexpf(x, -e) gives.
__device__ __forceinline__ float fp8_inv_scale(int e) {
    return e >= 127 ? __uint_as_float(0x00400000u) : __uint_as_float((uint32_t)(127 - e) << 23);
}

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
        const float inv = fp8_inv_scale(e);
        if (ok) {
            uint32_t word[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t acc = 0;
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const float2 f = make_float2(v[4 * h + 2 * j] * inv, v[4 * h + 2 * j + 1] * inv);
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
// One block of 256 threads per tile of 128 k x 64 columns: the tile comes in
// as 128-byte rows (16-byte loads, the next tile's already in flight while
// this one is quantized), each thread quantizes one column's 32-k group
// (column tid % 64, group tid / 64) into a shared-memory copy of the
// output tile, and the tile leaves as 64 rows of 128 K-major bytes, so
// that both the reads and the writes are whole 128-byte lines.  The same
// rule as the input (smallest power of two with 448 2^e >= max|group|,
// round to nearest even, saturate).  HBM-bound: 2 bytes read and 33/32
// bytes written per element.
constexpr int kQwK = 128, kQwC = 64, kQwThreads = 256, kQwBlocksPerSm = 4;
template <bool kW1>
__global__ void __launch_bounds__(kQwThreads, 4) quantize_w_fp8_kernel(const __nv_bfloat16* __restrict__ W, int E, int K,
                                                                    int C, uint8_t* __restrict__ q,
                                                                    uint8_t* __restrict__ atoms) {
    // rows padded by 16 bytes: the column reads and the 16-byte row writes
    // of a warp spread over all banks
    __shared__ __align__(16) __nv_bfloat16 tile[kQwK][kQwC + 8];
    __shared__ __align__(16) uint8_t out[kQwC][kQwK + 16];
    const int ncol = C / kQwC, nkt = K / kQwK;
    const int I = C / 2;  // kW1 only
    const int ntiles = E * nkt * ncol;  // below 2^31 (checked at launch)
    const int tid = threadIdx.x;
    // 16-byte chunk i of a tile: row tid / 8 + 32 i, columns 8 (tid % 8) ..
    const int lr = tid >> 3, lc = (tid & 7) * 8;
    auto load = [&](int ti, uint4 (&v)[4]) {
        const int cb = ti % ncol;
        const int kt = (ti / ncol) % nkt;
        const int e = ti / (ncol * nkt);
        const __nv_bfloat16* src = W + ((size_t)e * K + (size_t)kt * kQwK + lr) * (size_t)C + (size_t)cb * kQwC + lc;
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = __ldg(reinterpret_cast<const uint4*>(src + (size_t)(32 * i) * C));
    };
    uint4 nxt[4];
    if ((int)blockIdx.x < ntiles) load((int)blockIdx.x, nxt);
    for (int ti = (int)blockIdx.x; ti < ntiles; ti += (int)gridDim.x) {
        const int cb = ti % ncol;
        const int kt = (ti / ncol) % nkt;
        const int e = ti / (ncol * nkt);
        const int c0 = cb * kQwC, k0 = kt * kQwK;
        __syncthreads();  // the previous tile's shared memory has been read
#pragma unroll
        for (int i = 0; i < 4; ++i) *reinterpret_cast<uint4*>(&tile[lr + 32 * i][lc]) = nxt[i];
        __syncthreads();
        if (ti + (int)gridDim.x < ntiles) load(ti + (int)gridDim.x, nxt);
        const int c = tid & (kQwC - 1), g = tid / kQwC;
        // the group is read twice from shared memory (maximum, then codes)
        // rather than held in registers
        const __nv_bfloat16* col = &tile[32 * g][c];
        float amax = 0.0f;
#pragma unroll
        for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(__bfloat162float(col[j * (kQwC + 8)])));
        const int ex = fp8_group_exponent(amax);
        const float inv = fp8_inv_scale(ex);
        uint32_t w[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            uint32_t acc = 0;
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                const int r = 4 * j + 2 * m;
                const float2 f = make_float2(__bfloat162float(col[r * (kQwC + 8)]) * inv,
                                             __bfloat162float(col[(r + 1) * (kQwC + 8)]) * inv);
                acc |= (uint32_t)__nv_cvt_float2_to_fp8x2(f, __NV_SATFINITE, __NV_E4M3) << (16 * m);
            }
            w[j] = acc;
        }
        *reinterpret_cast<uint4*>(&out[c][32 * g]) = make_uint4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<uint4*>(&out[c][32 * g + 16]) = make_uint4(w[4], w[5], w[6], w[7]);
        const int cg = c0 + c;
        int ag, r, G;
        if constexpr (kW1) {
            const int fi = cg < I ? cg : cg - I;
            ag = fi >> 6;
            r = (cg < I ? 0 : 64) + (fi & 63);
            G = I / 64;
        } else {
            ag = cg >> 7;
            r = cg & 127;
            G = C / 128;
        }
        // 32-k group 4 kt + g: atom block kt, step g
        atoms[(((size_t)e * G + ag) * nkt + kt) * 512 + 16 * (r & 31) + 4 * (r >> 5) + g] = (uint8_t)(ex + 127);
        __syncthreads();
        // 64 rows of 128 bytes: q[e][c0 + row][k0 ..]
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int ch = tid + kQwThreads * i;
            const int row = ch >> 3, part = ch & 7;
            *reinterpret_cast<uint4*>(q + ((size_t)e * C + c0 + row) * (size_t)K + k0 + 16 * part) =
                *reinterpret_cast<const uint4*>(&out[row][16 * part]);
        }
    }
}

}  // namespace

int launch_quantize_w1_fp8(const __nv_bfloat16* W1, int E, int H, int I, uint8_t* q, uint8_t* atoms, int num_sms,
                           cudaStream_t st) {
    const long long ntiles = (long long)E * (H / kQwK) * (2 * I / kQwC);
    if (ntiles <= 0) return 0;
    if (ntiles > INT_MAX) return (int)cudaErrorInvalidValue;
    const long long cap = (long long)num_sms * kQwBlocksPerSm;  // resident blocks
    quantize_w_fp8_kernel<true><<<(unsigned)(ntiles < cap ? ntiles : cap), kQwThreads, 0, st>>>(W1, E, H, 2 * I, q,
                                                                                              atoms);
    return (int)cudaGetLastError();
}

int launch_quantize_w2_fp8(const __nv_bfloat16* W2, int E, int H, int I, uint8_t* q, uint8_t* atoms, int num_sms,
                           cudaStream_t st) {
    const long long ntiles = (long long)E * (I / kQwK) * (H / kQwC);
    if (ntiles <= 0) return 0;
    if (ntiles > INT_MAX) return (int)cudaErrorInvalidValue;
    const long long cap = (long long)num_sms * kQwBlocksPerSm;
    quantize_w_fp8_kernel<false><<<(unsigned)(ntiles < cap ? ntiles : cap), kQwThreads, 0, st>>>(W2, E, I, H, q,
                                                                                               atoms);
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
