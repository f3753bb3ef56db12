// Internal definitions shared by the library's host code and kernels.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_layer.h"

namespace moe {

// Tile sizes of the SM-pair GEMMs: 128 TMEM lanes (output rows or features)
// per CTA, accumulators of up to 256 columns, 64-deep K blocks.
constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 64;
constexpr int kGatherWarps = 8;  // warps issuing the cp.async row gathers
// warps 0-3 epilogue, 4 TMA producer, 5 MMA issuer, 6.. gather producers
constexpr int kWarpTma = 4;
constexpr int kWarpMma = 5;
constexpr int kWarpGather0 = 6;
constexpr int kGemmThreads = 32 * (kWarpGather0 + kGatherWarps);
constexpr int kMaxDevices = 64;
constexpr int kMaxExperts = 1024;  // E accepted by the entry points
constexpr int kEpiWarps = 4;
constexpr int kStageEpiBytes = 8192;  // per epilogue warp: TMA-store staging

// The six grouped GEMMs of the layer.
//   L1_FWD    h = gather(x) . W1[e]            + SwiGLU epilogue -> h, a
//   L2_FWD    o = w * (a . W2[e])              (weight epilogue)
//   L2_DGRAD  g = gather(dY) . W2[e]^T         + SwiGLU^T epilogue -> dh, aw, dw_part
//   L1_DGRAD  dxp = dh . W1[e]^T
//   DW1       dW1[e] = gather(x)^T . dh        (K = the expert's rows)
//   DW2       dW2[e] = aw^T . gather(dY)       (K = the expert's rows)
//   DW1_MG, DW2_MG  the same, added in FP32 to the caller's FP32 main gradient
//   L1_FWD_MX   L1_FWD on E4M3 weights and gathered E4M3 rows with UE8M0
//               scales per 32 elements of K (block-scaled MMA); a leaves as
//               E4M3 rows with a UE8M0 scale per 32 features (q_out, sf_out)
//   L2_FWD_MX   L2_FWD on E4M3 W2 and those E4M3 rows of a
enum Flavour : int {
    L1_FWD = 0, L2_FWD = 1, L2_DGRAD = 2, L1_DGRAD = 3, DW1 = 4, DW2 = 5, DW1_MG = 6, DW2_MG = 7, L1_FWD_MX = 8,
    L2_FWD_MX = 9
};

struct GemmArgs {
    int T, H, I, E, k;
    int K;          // contraction length (row-grouped flavours)
    int n_tiles;    // output column tiles
    int m_tiles;    // output row tiles per expert (weight-gradient flavours)
    int tiles_cap;  // bound on routed-row tiles (row-grouped flavours)
    int dw_cols;    // columns of dw_part
    float clamp;    // SwiGLU input clamp (INFINITY = none)
    uint32_t* cmask;  // clamp decisions [rows_cap][2I/32] (written by L1, read by L2 dgrad)
    const int32_t* perm;
    const int32_t* offs;
    const int32_t* counts;
    const int32_t* tiles;
    const int32_t* pair_offs;   // first tile pair of each expert in the walk (decreasing count)
    const int32_t* pair_owner;  // expert of each tile pair of the walk
    int32_t* status;
    const __nv_bfloat16* gsrc;  // gathered source rows [T, H] (x or dY)
    const float* topk_w;
    const __nv_bfloat16* h_in;  // saved h (L2_DGRAD epilogue)
    const __nv_bfloat16* a_in;  // saved a (L2_DGRAD epilogue)
    float* outf;                // dw_part (L2_DGRAD epilogue); bf16 outputs leave by TMA store
    const uint8_t* gsrc8;       // L1_FWD_MX: E4M3 rows [T, H]
    const uint8_t* gsf;         // UE8M0 scales of the E4M3 B rows: L1_FWD_MX [T, H / 32],
                                // L2_FWD_MX [rows_cap, I / 32] (those of a)
    uint8_t* q_out;             // L1_FWD_MX: a as E4M3 [rows_cap, I] (required)
    uint8_t* sf_out;            // L1_FWD_MX: the scales of q_out [rows_cap, I / 32]
};

// Tensor maps of one grouped-GEMM launch: operands A, B (loads), up to two
// outputs C0, C1 (TMA stores) and one more epilogue input D.  Unused maps
// are zero.
struct GemmMaps {
    CUtensorMap a, b, c0, c1, d;
};

// Layout of the three workspaces (host only).
int compute_layout(const moe_shape* s, moe_layout* L);

// The routing prologue cuts the T*k slots into at most kMaxRouteBlocks blocks
// of whole 1024-slot rounds: nblk blocks of per_blk slots (the last one
// shorter); nblk = 0 when there are no slots.
constexpr int kMaxRouteBlocks = 1024;
void route_block_split(long long tk, int* nblk, long long* per_blk);

// Kernel tracing hook (moe_trace_begin): events around every launch.
void trace_pre(cudaStream_t st);
void trace_post(cudaStream_t st, const char* name);

// Kernel launchers (return a cudaError_t as int).
int launch_route_prologue(const moe_shape& s, const moe_layout& L, const int32_t* topk_idx, uint8_t* route,
                          cudaStream_t st);
int launch_gemm(int flavour, const GemmArgs& a, const GemmMaps& maps, int grid, cudaStream_t st);
int launch_combine(const __nv_bfloat16* rows, const int32_t* inv, int T, int k, int H, __nv_bfloat16* out,
                   int num_sms, cudaStream_t st);
int launch_router_topk(const float* logits, int T, int E, int k, int32_t* topk_idx, float* topk_w, int num_sms,
                       cudaStream_t st);
int launch_quantize_fp8(const __nv_bfloat16* x, long long n, uint8_t* q, uint8_t* sf, int num_sms, cudaStream_t st);
int launch_quantize_w1_fp8(const __nv_bfloat16* W1, int E, int H, int I, uint8_t* q, uint8_t* atoms, int num_sms,
                           cudaStream_t st);
int launch_quantize_w2_fp8(const __nv_bfloat16* W2, int E, int H, int I, uint8_t* q, uint8_t* atoms, int num_sms,
                           cudaStream_t st);
int launch_dequantize_fp8(const uint8_t* q, const uint8_t* sf, long long n, __nv_bfloat16* out, int num_sms,
                          cudaStream_t st);
int launch_wait_selftest(int32_t* status, uint64_t limit_ns, long long* elapsed, cudaStream_t st);
int launch_dw_reduce(const float* dw_part, int cols, const int32_t* inv, long long slots, float* out, int num_sms,
                     cudaStream_t st);

}  // namespace moe
