// Routing prologue: builds every routing table from topk_idx on the device,
// with no host synchronisation (Primus-Turbo "Mega MoE" README,
// "Implementation Map": dispatch prologue building routing tables, and
// "No-Sync, CUDA Graph compatible"; DeepGEMM Mega-MoE article, "Block-M
// Alignment for Irregular Token Counts").
//
// One CTA of 1024 threads:
//   1. per-expert histogram (shared-memory integer atomics: order-free, exact)
//      and a count of ids that are neither -1 nor in [0, E);
//   2. block-M padded sizes, exclusive prefix sum over experts with a
//      warp-shuffle scan -> offs, Mpad, tile-owner table;
//   3. stable placement: slots are visited in chunks of 1024 in increasing
//      slot order; inside a chunk a slot's row is
//        offs[e] + (slots of e in earlier chunks) + (slots of e in earlier
//        warps of this chunk) + (lower lanes of its warp with the same e),
//      the last term from __match_any_sync, so every expert's rows hold its
//      slots in increasing slot order, bit-exactly reproducible.
// Two scheduling tables for the grouped GEMMs ride along: the M tiles of an
// expert are taken two at a time by a 2-CTA cluster, so pair_offs is the
// exclusive prefix sum of ceil(tiles_e / 2) and pair_owner[q] the expert of
// tile pair q (-1 past the last pair).
#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kPrologueThreads = 1024;
constexpr int kWarps = kPrologueThreads / 32;

__device__ __forceinline__ int warp_incl_scan(int v, int lane) {
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, v, d);
        if (lane >= d) v += n;
    }
    return v;
}

__global__ void __launch_bounds__(kPrologueThreads, 1)
    route_prologue_kernel(int T, int E, int k, int bm, const int32_t* __restrict__ idx, int32_t* __restrict__ counts,
                          int32_t* __restrict__ offs, int32_t* __restrict__ perm, int32_t* __restrict__ inv,
                          int32_t* __restrict__ tiles, int32_t* __restrict__ status,
                          int32_t* __restrict__ pair_offs, int32_t* __restrict__ pair_owner, long long rows_cap,
                          long long tiles_cap) {
    extern __shared__ int sm[];
    int* cnt = sm;                // [E]
    int* base = sm + E;           // [E]
    int* wcnt = sm + 2 * E;       // [kWarps][E]
    __shared__ int warp_tot[kWarps];
    __shared__ int warp_tot2[kWarps];
    __shared__ int s_invalid;
    __shared__ int s_mpad;
    __shared__ int s_pairs;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const long long tk = (long long)T * k;

    for (int e = tid; e < E; e += kPrologueThreads) cnt[e] = 0;
    for (int q = tid; q < kWarps * E; q += kPrologueThreads) wcnt[q] = 0;
    if (tid == 0) s_invalid = 0;
    __syncthreads();

    // 1. histogram
    int bad = 0;
    for (long long s = tid; s < tk; s += kPrologueThreads) {
        const int e = __ldg(idx + s);
        if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);
        else if (e != -1) ++bad;
    }
    for (int d = 16; d > 0; d >>= 1) bad += __shfl_xor_sync(0xffffffffu, bad, d);
    if (lane == 0 && bad) atomicAdd(&s_invalid, bad);
    __syncthreads();

    // 2. padded exclusive scan over experts; each thread owns a contiguous run
    // (and the same scan of the per-expert tile-pair counts)
    const int per = (E + kPrologueThreads - 1) / kPrologueThreads;
    const int e0 = tid * per;
    int run = 0, run2 = 0;
    for (int q = 0; q < per; ++q) {
        const int e = e0 + q;
        if (e < E) {
            const int t = (cnt[e] + bm - 1) / bm;
            run += t * bm;
            run2 += (t + 1) / 2;
        }
    }
    const int incl = warp_incl_scan(run, lane);
    const int incl2 = warp_incl_scan(run2, lane);
    if (lane == 31) {
        warp_tot[warp] = incl;
        warp_tot2[warp] = incl2;
    }
    __syncthreads();
    if (warp == 0) {
        const int v = warp_incl_scan(warp_tot[lane], lane);
        const int v2 = warp_incl_scan(warp_tot2[lane], lane);
        warp_tot[lane] = v;  // inclusive totals per warp
        warp_tot2[lane] = v2;
    }
    __syncthreads();
    int acc = incl - run + (warp > 0 ? warp_tot[warp - 1] : 0);
    int acc2 = incl2 - run2 + (warp > 0 ? warp_tot2[warp - 1] : 0);
    for (int q = 0; q < per; ++q) {
        const int e = e0 + q;
        if (e < E) {
            const int t = (cnt[e] + bm - 1) / bm;
            offs[e] = acc;
            base[e] = acc;
            counts[e] = cnt[e];
            pair_offs[e] = acc2;
            for (int pq = acc2; pq < acc2 + (t + 1) / 2; ++pq) pair_owner[pq] = e;
            acc += t * bm;
            acc2 += (t + 1) / 2;
        }
    }
    if (tid == kPrologueThreads - 1) {
        s_mpad = warp_tot[kWarps - 1];
        s_pairs = warp_tot2[kWarps - 1];
        offs[E] = s_mpad;
        pair_offs[E] = s_pairs;
        status[MOE_STATUS_MPAD] = s_mpad;
        status[MOE_STATUS_NUM_TILES] = s_mpad / bm;
        status[MOE_STATUS_N_INVALID] = s_invalid;
        status[MOE_STATUS_FLAGS] = 0;
        status[MOE_STATUS_NUM_PAIRS] = s_pairs;
        for (int q = MOE_STATUS_NUM_PAIRS + 1; q < MOE_STATUS_WORDS; ++q) status[q] = 0;
    }
    for (long long r = tid; r < rows_cap; r += kPrologueThreads) perm[r] = -1;
    __syncthreads();

    // tile owners (and no owner past the last tile pair)
    const int mpad = s_mpad;
    for (long long m = (long long)mpad / bm + tid; m < tiles_cap; m += kPrologueThreads) tiles[m] = -1;
    for (long long q = (long long)s_pairs + tid; q < tiles_cap; q += kPrologueThreads) pair_owner[q] = -1;
    for (int e = tid; e < E; e += kPrologueThreads) {
        const int m_end = (base[e] + ((cnt[e] + bm - 1) / bm) * bm) / bm;
        for (int m = base[e] / bm; m < m_end; ++m) tiles[m] = e;
    }

    // 3. stable placement, 1024 slots per round
    const unsigned lt_mask = (1u << lane) - 1u;
    for (long long c0 = 0; c0 < tk; c0 += kPrologueThreads) {
        const long long s = c0 + tid;
        const int e = s < tk ? __ldg(idx + s) : -1;
        const bool valid = e >= 0 && e < E;
        const int key = valid ? e : -1;
        const unsigned peers = __match_any_sync(0xffffffffu, key);
        const int rank = __popc(peers & lt_mask);
        if (valid && rank == 0) wcnt[warp * E + e] = __popc(peers);
        __syncthreads();
        if (valid) {
            int pre = 0;
            for (int w = 0; w < warp; ++w) pre += wcnt[w * E + e];
            const int row = base[e] + pre + rank;
            perm[row] = (int32_t)s;
            inv[s] = row;
        } else if (s < tk) {
            inv[s] = -1;
        }
        __syncthreads();
        for (int q = tid; q < E; q += kPrologueThreads) {
            int tot = 0;
            for (int w = 0; w < kWarps; ++w) {
                tot += wcnt[w * E + q];
                wcnt[w * E + q] = 0;
            }
            base[q] += tot;
        }
        __syncthreads();
    }
}

}  // namespace

int launch_route_prologue(const moe_shape& s, const moe_layout& L, const int32_t* topk_idx, uint8_t* route,
                          cudaStream_t st) {
    const size_t smem = sizeof(int) * (size_t)(2 + kWarps) * (size_t)s.E;
    // opt in once per device to the largest size any E <= 1024 needs
    static bool done[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return (int)e;
    if (dev < 0 || dev >= kMaxDevices) return (int)cudaErrorInvalidDevice;
    if (!done[dev]) {
        e = cudaFuncSetAttribute(route_prologue_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)(sizeof(int) * (2 + kWarps) * 1024));
        if (e != cudaSuccess) return (int)e;
        done[dev] = true;
    }
    route_prologue_kernel<<<1, kPrologueThreads, smem, st>>>(
        s.T, s.E, s.k, s.block_m, topk_idx, reinterpret_cast<int32_t*>(route + L.counts),
        reinterpret_cast<int32_t*>(route + L.offs), reinterpret_cast<int32_t*>(route + L.perm),
        reinterpret_cast<int32_t*>(route + L.inv), reinterpret_cast<int32_t*>(route + L.tiles),
        reinterpret_cast<int32_t*>(route + L.status), reinterpret_cast<int32_t*>(route + L.pair_offs),
        reinterpret_cast<int32_t*>(route + L.pair_owner), (long long)L.rows_cap, (long long)L.tiles_cap);
    return (int)cudaGetLastError();
}

}  // namespace moe
