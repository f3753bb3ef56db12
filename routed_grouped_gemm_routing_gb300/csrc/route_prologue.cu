// Routing prologue: builds every routing table from topk_idx on the device,
// with no host synchronisation (Primus-Turbo "Mega MoE" README,
// "Implementation Map": dispatch prologue building routing tables, and
// "No-Sync, CUDA Graph compatible"; DeepGEMM Mega-MoE article, "Block-M
// Alignment for Irregular Token Counts").
//
// Three kernels on the caller's stream, so that the work spreads over the
// whole GPU instead of one SM:
//   1. route_hist (one CTA per slot block, blocks of whole 1024-slot rounds
//      in increasing slot order): per-expert counts of the block, and for
//      every valid slot its rank among the block's earlier slots of the same
//      expert (warp ranks from __match_any_sync, then earlier warps of the
//      round, then earlier rounds), kept in inv[] until step 3; ids that are
//      neither -1 nor in [0, E) are counted per block.  Also sets every
//      perm entry to -1 (padding).
//   2. route_scan (one CTA): per expert, the exclusive prefix over blocks of
//      the block counts (in place) and the total count; block-M padded sizes
//      and their exclusive prefix sum (warp-shuffle scan) -> offs, Mpad, the
//      tile-owner table, the status words, and the two scheduling tables of
//      the SM-pair GEMMs, which walk the experts in decreasing order of
//      routed rows (ties: smaller id first; a bitonic sort of (count, id)):
//      pair_offs[e] = first tile pair of expert e in that walk (the
//      exclusive prefix sum of ceil(tiles / 2) over the experts before it),
//      pair_offs[E] = the number of pairs, pair_owner[q] = expert of tile
//      pair q of the walk (-1 past the last pair).
//   3. route_place (grid over slots): row = offs[e] + (slots of e in earlier
//      blocks) + (rank inside the block); perm[row] = s, inv[s] = row, and
//      inv[s] = -1 for a dropped slot.
// An expert's rows therefore hold its slots in increasing slot order: the
// tables are bit-exact and reproducible, and need no atomics on global
// memory (the block counts are plain per-block integer sums).
#include <atomic>
#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ int warp_incl_scan(int v, int lane) {
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, v, d);
        if (lane >= d) v += n;
    }
    return v;
}

// 1. block counts and in-block ranks
__global__ void __launch_bounds__(kThreads, 1)
    route_hist_kernel(long long tk, int E, long long per_blk, const int32_t* __restrict__ idx,
                      int32_t* __restrict__ inv, int32_t* __restrict__ bcnt, int32_t* __restrict__ bbad,
                      int32_t* __restrict__ perm, long long rows_cap) {
    extern __shared__ int sm[];
    int* run = sm;       // [E] slots of expert e in this block's earlier rounds
    int* wcnt = sm + E;  // [kWarps][E] slots of e per warp in the current round
    __shared__ int s_bad;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int e = tid; e < E; e += kThreads) run[e] = 0;
    for (int q = tid; q < kWarps * E; q += kThreads) wcnt[q] = 0;
    if (tid == 0) s_bad = 0;
    for (long long r = (long long)blockIdx.x * kThreads + tid; r < rows_cap; r += (long long)gridDim.x * kThreads)
        perm[r] = -1;
    __syncthreads();

    const long long s0 = (long long)blockIdx.x * per_blk;
    const long long s1 = s0 + per_blk < tk ? s0 + per_blk : tk;
    const unsigned lt_mask = (1u << lane) - 1u;
    int bad = 0;
    for (long long c0 = s0; c0 < s1; c0 += kThreads) {
        const long long s = c0 + tid;
        const int e = s < s1 ? __ldg(idx + s) : -1;
        const bool valid = e >= 0 && e < E;
        if (s < s1 && !valid && e != -1) ++bad;
        const int key = valid ? e : -1;
        const unsigned peers = __match_any_sync(0xffffffffu, key);
        const int rank = __popc(peers & lt_mask);
        if (valid && rank == 0) wcnt[warp * E + e] = __popc(peers);
        __syncthreads();
        if (valid) {
            int pre = run[e];
            for (int w = 0; w < warp; ++w) pre += wcnt[w * E + e];
            inv[s] = pre + rank;
        }
        __syncthreads();
        for (int q = tid; q < E; q += kThreads) {
            int tot = 0;
            for (int w = 0; w < kWarps; ++w) {
                tot += wcnt[w * E + q];
                wcnt[w * E + q] = 0;
            }
            run[q] += tot;
        }
        __syncthreads();
    }
    for (int d = 16; d > 0; d >>= 1) bad += __shfl_xor_sync(0xffffffffu, bad, d);
    if (lane == 0 && bad) atomicAdd(&s_bad, bad);
    __syncthreads();
    for (int e = tid; e < E; e += kThreads) bcnt[(size_t)blockIdx.x * E + e] = run[e];
    if (tid == 0) bbad[blockIdx.x] = s_bad;
}

// 2. totals, padded offsets, tile and pair tables, status words (one CTA)
__global__ void __launch_bounds__(kThreads, 1)
    route_scan_kernel(int E, int nblk, int bm, int32_t* __restrict__ bcnt, const int32_t* __restrict__ bbad,
                      int32_t* __restrict__ counts, int32_t* __restrict__ offs, int32_t* __restrict__ tiles,
                      int32_t* __restrict__ status, int32_t* __restrict__ pair_offs,
                      int32_t* __restrict__ pair_owner, long long tiles_cap) {
    extern __shared__ int sm[];
    int* cnt = sm;       // [E]
    int* base = sm + E;  // [E]
    __shared__ unsigned long long walk_key[kMaxExperts];  // (count descending, id) sort keys
    __shared__ int warp_tot[kWarps];
    __shared__ int warp_tot2[kWarps];
    __shared__ int s_invalid;
    __shared__ int s_mpad;
    __shared__ int s_pairs;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    // per expert: exclusive prefix over blocks (in place) and the total; the
    // counts of 8 blocks are loaded before any of them is rewritten, so that
    // their loads are in flight together
    for (int e = tid; e < E; e += kThreads) {
        int acc = 0;
        for (int b0 = 0; b0 < nblk; b0 += 8) {
            int v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = b0 + i < nblk ? bcnt[(size_t)(b0 + i) * E + e] : 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (b0 + i < nblk) bcnt[(size_t)(b0 + i) * E + e] = acc;
                acc += v[i];
            }
        }
        cnt[e] = acc;
    }
    int bad = 0;
    for (int b = tid; b < nblk; b += kThreads) bad += bbad[b];
    for (int d = 16; d > 0; d >>= 1) bad += __shfl_xor_sync(0xffffffffu, bad, d);
    if (tid == 0) s_invalid = 0;
    __syncthreads();
    if (lane == 0 && bad) atomicAdd(&s_invalid, bad);

    // the GEMMs' walk order: ascending bitonic sort of ((2^31-1 - count) << 32
    // | id) over the next power of two >= E (padding keys sort last), one key
    // per thread; partners closer than a warp are exchanged by shuffles,
    // farther ones through shared memory
    static_assert(kThreads >= kMaxExperts, "one sort key per thread");
    int np2 = 1;
    while (np2 < E) np2 <<= 1;
    unsigned long long key = tid < E ? ((unsigned long long)(0x7fffffff - cnt[tid]) << 32) | (unsigned)tid : ~0ull;
    for (int len = 2; len <= np2; len <<= 1) {
        for (int j = len >> 1; j > 0; j >>= 1) {
            unsigned long long other;
            if (j >= 32) {
                if (tid < np2) walk_key[tid] = key;
                __syncthreads();
                other = walk_key[(tid ^ j) & (kMaxExperts - 1)];
                __syncthreads();
            } else {
                other = __shfl_xor_sync(0xffffffffu, key, j);
            }
            // the lower index of a pair keeps the smaller key in an ascending run
            const bool keep_min = ((tid & j) == 0) == ((tid & len) == 0);
            key = keep_min ? (key < other ? key : other) : (key > other ? key : other);
        }
    }
    if (tid < np2) walk_key[tid] = key;
    __syncthreads();

    // padded exclusive scan over experts (by id) and the scan of the tile-pair
    // counts over the walk (by rank); each thread owns a contiguous run of both
    const int per = (E + kThreads - 1) / kThreads;
    const int e0 = tid * per;
    int run = 0, run2 = 0;
    for (int q = 0; q < per; ++q) {
        const int e = e0 + q;
        if (e < E) {
            run += ((cnt[e] + bm - 1) / bm) * bm;
            const int w = (int)(walk_key[e] & 0xffffffffu);
            run2 += ((cnt[w] + bm - 1) / bm + 1) / 2;
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
            acc += t * bm;
            const int w = (int)(walk_key[e] & 0xffffffffu);  // expert of rank e
            const int np = ((cnt[w] + bm - 1) / bm + 1) / 2;
            pair_offs[w] = acc2;
            for (int pq = acc2; pq < acc2 + np; ++pq) pair_owner[pq] = w;
            acc2 += np;
        }
    }
    if (tid == kThreads - 1) {
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
    __syncthreads();

    // tile owners (and no owner past the last tile pair)
    const int mpad = s_mpad;
    for (long long m = (long long)mpad / bm + tid; m < tiles_cap; m += kThreads) tiles[m] = -1;
    for (long long q = (long long)s_pairs + tid; q < tiles_cap; q += kThreads) pair_owner[q] = -1;
    for (int e = tid; e < E; e += kThreads) {
        const int m_end = (base[e] + ((cnt[e] + bm - 1) / bm) * bm) / bm;
        for (int m = base[e] / bm; m < m_end; ++m) tiles[m] = e;
    }
}

// 3. placement
__global__ void __launch_bounds__(256)
    route_place_kernel(long long tk, int E, long long per_blk, const int32_t* __restrict__ idx,
                       const int32_t* __restrict__ offs, const int32_t* __restrict__ bcnt,
                       int32_t* __restrict__ perm, int32_t* __restrict__ inv) {
    for (long long s = (long long)blockIdx.x * blockDim.x + threadIdx.x; s < tk;
         s += (long long)gridDim.x * blockDim.x) {
        const int e = __ldg(idx + s);
        if (e >= 0 && e < E) {
            const int row = __ldg(offs + e) + bcnt[(size_t)(s / per_blk) * E + e] + inv[s];
            perm[row] = (int32_t)s;
            inv[s] = row;
        } else {
            inv[s] = -1;
        }
    }
}

// Host threads may race through the first call; setting the attribute twice
// is harmless.
int set_smem_once(const void* fn, int bytes, std::atomic<bool>* done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return (int)e;
    if (dev < 0 || dev >= kMaxDevices) return (int)cudaErrorInvalidDevice;
    if (!done[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess) return (int)e;
        done[dev].store(true, std::memory_order_release);
    }
    return 0;
}

}  // namespace

void route_block_split(long long tk, int* nblk, long long* per_blk) {
    const long long rounds = (tk + kThreads - 1) / kThreads;
    long long rpb = (rounds + kMaxRouteBlocks - 1) / kMaxRouteBlocks;
    if (rpb < 1) rpb = 1;
    *per_blk = rpb * kThreads;
    *nblk = (int)((tk + *per_blk - 1) / *per_blk);
}

int launch_route_prologue(const moe_shape& s, const moe_layout& L, const int32_t* topk_idx, uint8_t* route,
                          cudaStream_t st) {
    // opt in once per device to the largest size any E <= kMaxExperts needs
    static std::atomic<bool> done_hist[kMaxDevices] = {};
    int e = set_smem_once((const void*)route_hist_kernel, (int)(sizeof(int) * (1 + kWarps) * kMaxExperts), done_hist);
    if (e) return e;
    const long long tk = (long long)s.T * s.k;
    int nblk = 0;
    long long per_blk = 0;
    route_block_split(tk, &nblk, &per_blk);
    auto* counts = reinterpret_cast<int32_t*>(route + L.counts);
    auto* offs = reinterpret_cast<int32_t*>(route + L.offs);
    auto* perm = reinterpret_cast<int32_t*>(route + L.perm);
    auto* inv = reinterpret_cast<int32_t*>(route + L.inv);
    auto* bcnt = reinterpret_cast<int32_t*>(route + L.blk_counts);
    int32_t* bbad = bcnt + (size_t)nblk * s.E;
    if (nblk > 0) {
        trace_pre(st);
        route_hist_kernel<<<nblk, kThreads, sizeof(int) * (size_t)(1 + kWarps) * s.E, st>>>(
            tk, s.E, per_blk, topk_idx, inv, bcnt, bbad, perm, (long long)L.rows_cap);
        trace_post(st, "route_hist");
        if ((e = (int)cudaGetLastError())) return e;
    }
    trace_pre(st);
    route_scan_kernel<<<1, kThreads, sizeof(int) * 2 * (size_t)s.E, st>>>(
        s.E, nblk, s.block_m, bcnt, bbad, counts, offs, reinterpret_cast<int32_t*>(route + L.tiles),
        reinterpret_cast<int32_t*>(route + L.status), reinterpret_cast<int32_t*>(route + L.pair_offs),
        reinterpret_cast<int32_t*>(route + L.pair_owner), (long long)L.tiles_cap);
    trace_post(st, "route_scan");
    if ((e = (int)cudaGetLastError())) return e;
    if (tk > 0) {
        long long blocks = (tk + 255) / 256;
        if (blocks > 16384) blocks = 16384;
        trace_pre(st);
        route_place_kernel<<<(unsigned)blocks, 256, 0, st>>>(tk, s.E, per_blk, topk_idx, offs, bcnt, perm, inv);
        trace_post(st, "route_place");
        if ((e = (int)cudaGetLastError())) return e;
    }
    return 0;
}

}  // namespace moe
