// Persistent variable-K grouped GEMM on the 5th-generation tensor cores
// (tcgen05, TMEM accumulators) for the two weight gradients of the routed MoE
// layer, dW1[e] = gather(x)_e^T . dh_e and dW2[e] = aw_e^T . gather(dY)_e
// (Primus-Turbo "Mega MoE" README, "Pipeline": the backward's variable-K
// weight-gradient GEMMs, with the dispatched x recomputed by gathering).
// It also holds the helpers shared with the SM-pair kernels of the
// row-grouped GEMMs (grouped_gemm_2sm.cuh).
//
//  * A tile is 128 rows x 256 columns of dW[e]; tiles are walked (expert,
//    M tile, N tile) and K runs over expert e's routed rows.
//  * The token-side operand (x for dW1, dY for dW2) is GATHERED straight from
//    x or dY by the permutation table (16-byte cp.async into the
//    128-byte-swizzled layout the MMA reads), so the dispatched activations
//    are never written to memory (README, "Recompute dispatched x").  The
//    other operand (dh or aw) arrives by TMA.
//  * Warp roles: warps 0-3 epilogue (TMEM -> registers -> shared memory ->
//    TMA store), warp 4 TMA producer, warp 5 MMA issuer and TMEM owner,
//    warps 6.. gather producers.  A 4-stage shared-memory ring (full/empty
//    mbarriers) feeds the MMA; two 256-column TMEM accumulators let the
//    epilogue of one tile overlap the main loop of the next.
//  * Every wait is bounded; on a timeout the CTA raises a status flag,
//    drains what it issued, frees TMEM and returns.
#pragma once

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {

template <int F>
struct GemmTraits;
// dW1: A = gathered x (MN-major, M along H), B = dh rows (MN-major)
template <>
struct GemmTraits<DW1> {
    static constexpr bool kAGather = true, kBGather = false, kAMN = true, kBMN = true;
};
// dW2: A = aw rows (MN-major, M along I), B = gathered dY (MN-major)
template <>
struct GemmTraits<DW2> {
    static constexpr bool kAGather = false, kBGather = true, kAMN = true, kBMN = true;
};

struct TileCoord {
    int e;      // expert
    int m0;     // first output row of dW[e]
    int n0;     // first output column of dW[e]
    int nt;     // column tile index
    int nkb;    // number of 64-wide K blocks
    int krow0;  // first routed row of the expert
    int krows;  // routed rows of the expert
};

// A tile's coordinates come from the routing tables in global memory.  Each
// role reads the next tile's entries right after starting the current tile
// (load_tile_raw), so that latency is hidden behind the current tile's work
// instead of stalling every role at every tile boundary.
struct TileRaw {
    int cnt;  // counts[e]
    int off;  // offs[e]
};

template <int F>
__device__ __forceinline__ TileRaw load_tile_raw(int tile, const GemmArgs& p) {
    const int e = tile / (p.m_tiles * p.n_tiles);
    return TileRaw{__ldg(p.counts + e), __ldg(p.offs + e)};
}

template <int F>
__device__ __forceinline__ TileCoord finish_tile(int tile, TileRaw r, const GemmArgs& p) {
    TileCoord t;
    const int per_e = p.m_tiles * p.n_tiles;
    t.e = tile / per_e;
    const int rem = tile - t.e * per_e;
    const int mt = rem / p.n_tiles;
    t.nt = rem - mt * p.n_tiles;
    t.m0 = mt * kBM;
    t.n0 = t.nt * kBN;
    t.nkb = (r.cnt + kBK - 1) / kBK;
    t.krow0 = r.off;
    t.krows = r.cnt;
    return t;
}

// Iterates this CTA's tiles blockIdx.x, blockIdx.x + gridDim.x, ... with the
// table reads of the next tile in flight.
template <int F>
struct TileWalk {
    const GemmArgs& p;
    int total;
    int tile;
    TileRaw raw;
    __device__ __forceinline__ TileWalk(const GemmArgs& p_, int total_) : p(p_), total(total_), tile(blockIdx.x) {
        raw = tile < total ? load_tile_raw<F>(tile, p) : TileRaw{0, 0};
    }
    __device__ __forceinline__ bool valid() const { return tile < total; }
    // Coordinates of the current tile; issues the reads of the next one.
    __device__ __forceinline__ TileCoord take() {
        const TileCoord t = finish_tile<F>(tile, raw, p);
        const int nxt = tile + (int)gridDim.x;
        if (nxt < total) raw = load_tile_raw<F>(nxt, p);
        return t;
    }
    __device__ __forceinline__ void next() { tile += (int)gridDim.x; }
};

template <int F>
__device__ __forceinline__ int total_tiles(const GemmArgs& p) {
    return p.E * p.m_tiles * p.n_tiles;
}

struct Bars {
    uint32_t base;
    __device__ __forceinline__ uint32_t full(int s) const { return base + 8u * s; }
    __device__ __forceinline__ uint32_t empty(int s) const { return base + 8u * (kStages + s); }
    __device__ __forceinline__ uint32_t tfull(int a) const { return base + 8u * (2 * kStages + a); }
    __device__ __forceinline__ uint32_t tempty(int a) const { return base + 8u * (2 * kStages + 2 + a); }
    __device__ __forceinline__ uint32_t drain() const { return base + 8u * (2 * kStages + 4); }
};
constexpr int kNumBars = 2 * kStages + 5;

// Every lane of the warp waits; the warp proceeds only if all lanes saw the
// phase complete, so warp-collective instructions never run diverged.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
    const bool ok = mbar_wait(bar, parity, abort);
    return __all_sync(0xffffffffu, ok);
}

// ------------------------------------------------------------ TMA producer
template <int F>
__device__ void role_tma(const CUtensorMap* mA, const CUtensorMap* mB, const GemmArgs& p, int total, uint32_t sA,
                         uint32_t sB, Bars bars, volatile int* abort) {
    using Tr = GemmTraits<F>;
    constexpr uint32_t kTx = (Tr::kAGather ? 0u : (uint32_t)kStageABytes) + (Tr::kBGather ? 0u : (uint32_t)kStageBBytes);
    int stage = 0;
    uint32_t phase = 0;
    for (TileWalk<F> w(p, total); w.valid(); w.next()) {
        const TileCoord t = w.take();
        for (int kb = 0; kb < t.nkb; ++kb) {
            if (!mbar_wait(bars.empty(stage), phase ^ 1u, abort)) return;
            const uint32_t fb = bars.full(stage);
            mbar_arrive_expect_tx(fb, kTx);
            const uint32_t a = sA + stage * kStageABytes;
            const uint32_t b = sB + stage * kStageBBytes;
            const int k0 = kb * kBK;
            if constexpr (F == DW1) {
#pragma unroll
                for (int j = 0; j < 4; ++j) tma_load_2d(b + j * 8192, mB, t.n0 + 64 * j, t.krow0 + k0, fb);
            } else {  // DW2
#pragma unroll
                for (int j = 0; j < 2; ++j) tma_load_2d(a + j * 8192, mA, t.m0 + 64 * j, t.krow0 + k0, fb);
            }
            if (++stage == kStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
}

// --------------------------------------------------------- gather producer
// kGatherWarps warps copy 16-byte chunks of token rows into the
// 128-byte-swizzled tile layout (chunk c of tile row r lands at
// r*128 + ((c ^ (r & 7)) * 16)); each warp owns an equal share of the 64 K
// rows of every stage, so several warps' copies are in flight at once.
template <int F>
__device__ void role_gather(const GemmArgs& p, int total, uint32_t sA, uint32_t sB, Bars bars, volatile int* abort,
                            int gw, int lane) {
    using Tr = GemmTraits<F>;
    const int c = lane & 7;
    const int rb = lane >> 3;
    const int H = p.H;
    const int k = p.k;
    const __nv_bfloat16* src = p.gsrc;
    int stage = 0;
    uint32_t phase = 0;
    for (TileWalk<F> w(p, total); w.valid(); w.next()) {
        const TileCoord t = w.take();
        {
            // MN-major token operand of a weight gradient: the 64 K rows of a
            // stage are routed rows of expert e; columns run along H.
            constexpr int kRegions = (F == DW1) ? 2 : 4;
            constexpr int kRowsPerWarp = kBK / kGatherWarps;  // 16
            constexpr int kPerLane = kRowsPerWarp / 4;        // 4
            const int col0 = (F == DW1) ? t.m0 : t.n0;
            const int rw0 = gw * kRowsPerWarp;
            // permutation entries of this warp's rows, one k block ahead
            int nxt = t.nkb > 0 ? __ldg(p.perm + t.krow0 + rw0 + (lane & (kRowsPerWarp - 1))) : -1;
            for (int kb = 0; kb < t.nkb; ++kb) {
                const int cur = nxt;
                if (kb + 1 < t.nkb) nxt = __ldg(p.perm + t.krow0 + (kb + 1) * kBK + rw0 + (lane & (kRowsPerWarp - 1)));
                if (!warp_wait(bars.empty(stage), phase ^ 1u, abort)) return;
                const uint32_t dst0 = (F == DW1) ? (sA + stage * kStageABytes) : (sB + stage * kStageBBytes);
                const int tcur = cur >= 0 ? cur / k : -1;
                int tq[kPerLane];
#pragma unroll
                for (int q = 0; q < kPerLane; ++q) tq[q] = __shfl_sync(0xffffffffu, tcur, rb + 4 * q);
#pragma unroll
                for (int g = 0; g < kRegions; ++g) {
                    const int colg = col0 + 64 * g + 8 * c;
                    const bool okc = colg < H;
#pragma unroll
                    for (int q = 0; q < kPerLane; ++q) {
                        const int r = rw0 + rb + 4 * q;
                        const bool ok = okc && tq[q] >= 0;
                        const __nv_bfloat16* gp = src + (ok ? (size_t)tq[q] * (size_t)H + colg : (size_t)0);
                        cp_async_16(dst0 + g * 8192 + r * 128 + ((c ^ (r & 7)) << 4), gp, ok ? 16u : 0u);
                    }
                }
                cp_async_arrive_noinc(bars.full(stage));
                if (++stage == kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
    }
}

// -------------------------------------------------------------- MMA issuer
template <int F>
__device__ void role_mma(const GemmArgs& p, int total, uint32_t sA, uint32_t sB, Bars bars, uint32_t tmem_base,
                         volatile int* abort) {
    using Tr = GemmTraits<F>;
    constexpr uint32_t idesc = make_idesc_bf16(kBM, kBN, Tr::kAMN, Tr::kBMN);
    int stage = 0;
    uint32_t phase = 0;
    int it = 0;
    for (TileWalk<F> w(p, total); w.valid(); w.next(), ++it) {
        const TileCoord t = w.take();
        const int acc = it & 1;
        const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
        if (!mbar_wait(bars.tempty(acc), acc_phase ^ 1u, abort)) return;
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(acc * kBN);
        for (int kb = 0; kb < t.nkb; ++kb) {
            if (!mbar_wait(bars.full(stage), phase, abort)) return;
            tc_fence_after();
            fence_proxy_async_smem();  // the gathered operand was written by cp.async
            const uint32_t a = sA + stage * kStageABytes;
            const uint32_t b = sB + stage * kStageBBytes;
            // Weight gradients contract over the expert's routed rows: the
            // last K block stops at the 16-row step that holds the last
            // routed row, so rows past it (never written by the row-grouped
            // kernels) are never read.
            const int ksteps = min(kBK / 16, (t.krows - kb * kBK + 15) / 16);
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk) {
                if (kk >= ksteps) break;
                // MN-major: 16 K rows = 2 KiB; LBO = stride of 64-wide MN slabs.
                const uint64_t ad = make_sdesc_sw128(a + kk * 2048, 8192, 1024);
                const uint64_t bd = make_sdesc_sw128(b + kk * 2048, 8192, 1024);
                tc_mma_bf16(d, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
            }
            tc_commit(bars.empty(stage));
            if (++stage == kStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
        tc_commit(bars.tfull(acc));
    }
}

// ---------------------------------------------------------------- epilogue
// Each epilogue warp owns 32 TMEM lanes = 32 rows of the tile.  Results are
// written into this warp's 8 KiB staging area in shared memory, in the
// 128-byte swizzle of the output tensor map, and leave through TMA bulk
// stores of whole 32-row x 64-column boxes while the warp goes on with the
// next chunk.
struct OutMaps {
    const CUtensorMap* c0;
    const CUtensorMap* c1;
};

__device__ __forceinline__ void pack32(const float (&v)[32], uint32_t (&p)[16]) {
#pragma unroll
    for (int j = 0; j < 16; ++j) p[j] = pack_bf16x2(v[2 * j], v[2 * j + 1]);
}

template <int F>
__device__ void role_epilogue(const GemmArgs& p, OutMaps om, int total, Bars bars, uint32_t tmem_base,
                              uint32_t stage, volatile int* abort, int warp, int lane) {
    int it = 0;
    uint32_t nstore = 0;  // 64-column boxes stored by this warp (picks the staging half)
    for (TileWalk<F> w(p, total); w.valid(); w.next(), ++it) {
        const TileCoord t = w.take();
        const int acc = it & 1;
        const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
        if (!warp_wait(bars.tfull(acc), acc_phase, abort)) break;
        tc_fence_after();
        const uint32_t tacc = tmem_base + (uint32_t)(acc * kBN) + ((uint32_t)(warp * 32) << 16);
        const int row0 = t.m0 + warp * 32;  // first row of this warp's box

        // The weight gradient of expert e; an expert without routed rows
        // gets zeros.
        const int N_out = (F == DW1) ? 2 * p.I : p.H;
        const bool have_acc = t.nkb > 0;
#pragma unroll 1
        for (int c64 = 0; c64 < 4; ++c64) {
            const int col = t.n0 + 64 * c64;
            if (col >= N_out) break;
            uint32_t pk[32];
            {
                uint32_t r0[32], r1[32];
                if (have_acc) {
                    tmem_ld32_nowait(tacc + 64 * c64, r0);
                    tmem_ld32_nowait(tacc + 64 * c64 + 32, r1);
                    tmem_ld_wait();
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) r0[j] = r1[j] = 0u;
                }
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    pk[j] = pack_bf16x2(__uint_as_float(r0[2 * j]), __uint_as_float(r0[2 * j + 1]));
                    pk[16 + j] = pack_bf16x2(__uint_as_float(r1[2 * j]), __uint_as_float(r1[2 * j + 1]));
                }
            }
            const uint32_t buf = stage + (nstore & 1u) * 4096u;
            if (lane == 0) bulk_wait_read<1>();
            __syncwarp();
            stage_row_sw128(buf, lane, pk);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                tma_store_3d(om.c0, col, row0, t.e, buf);
                bulk_commit();
            }
            ++nstore;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.tempty(acc));
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
}

template <int F>
__global__ void __launch_bounds__(kGemmThreads, 1)
    moe_gemm_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                    const __grid_constant__ CUtensorMap mapC0, const __grid_constant__ CUtensorMap mapC1,
                    const GemmArgs p) {
    using Tr = GemmTraits<F>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw);
    const uint32_t sA = base;
    const uint32_t sB = base + kStages * kStageABytes;
    const uint32_t sStage = sB + kStages * kStageBBytes;  // 4 x 8 KiB epilogue staging
    const uint32_t bar_base = sStage + kEpiWarps * kStageEpiBytes;
    uint8_t* tail = base_ptr + (bar_base - base);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tail + 8 * kNumBars);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const Bars bars{bar_base};

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        constexpr uint32_t kFullCount = 1u + 32u * kGatherWarps;
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bars.full(s), kFullCount);
            mbar_init(bars.empty(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(bars.tfull(a), 1);
            mbar_init(bars.tempty(a), kEpiWarps);
        }
        mbar_init(bars.drain(), 1);
        *abort = 0;
        fence_mbar_init();
    }
    if (warp == kWarpMma) {
        tmem_alloc(smem_addr(tmem_slot), 2 * kBN);
        tmem_relinquish();
    }
    if (warp == kWarpTma && lane == 0) {
        if constexpr (!Tr::kAGather) tma_prefetch_map(&mapA);
        if constexpr (!Tr::kBGather) tma_prefetch_map(&mapB);
        tma_prefetch_map(&mapC0);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int total = total_tiles<F>(p);

    if (warp == kWarpTma) {
        if (lane == 0) role_tma<F>(&mapA, &mapB, p, total, sA, sB, bars, abort);
    } else if (warp >= kWarpGather0) {
        role_gather<F>(p, total, sA, sB, bars, abort, warp - kWarpGather0, lane);
        cp_async_wait_all();
    } else if (warp == kWarpMma) {
        if (lane == 0) {
            role_mma<F>(p, total, sA, sB, bars, tmem_base, abort);
            if (*abort) {
                // let every MMA already issued finish before TMEM is released
                tc_commit(bars.drain());
                const uint64_t t0 = global_timer_ns();
                while (!mbar_try_wait(bars.drain(), 0) && global_timer_ns() - t0 < 100000000ull) {
                }
            }
        }
    } else {
        role_epilogue<F>(p, OutMaps{&mapC0, &mapC1}, total, bars, tmem_base, sStage + warp * kStageEpiBytes, abort,
                         warp, lane);
    }
    if (warp == kWarpTma && lane == 0 && *abort) {
        // bulk copies already issued land within microseconds; give them time
        const uint64_t t0 = global_timer_ns();
        while (global_timer_ns() - t0 < 2000000ull) {
        }
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 2 * kBN);
    }
    if (threadIdx.x == 0 && *abort) atomicOr(reinterpret_cast<int*>(p.status + MOE_STATUS_FLAGS), 1);
}

template <int F>
int launch_gemm_flavour(const GemmArgs& a, const GemmMaps& m, int grid, cudaStream_t st) {
    // The shared-memory opt-in is a per-device function attribute: set it
    // once per device (outside any stream capture, on the first call).
    static bool done[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return (int)e;
    if (dev < 0 || dev >= kMaxDevices) return (int)cudaErrorInvalidDevice;
    if (!done[dev]) {
        e = cudaFuncSetAttribute(moe_gemm_kernel<F>, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmemBytes);
        if (e != cudaSuccess) return (int)e;
        done[dev] = true;
    }
    moe_gemm_kernel<F><<<grid, kGemmThreads, kGemmSmemBytes, st>>>(m.a, m.b, m.c0, m.c1, a);
    return (int)cudaGetLastError();
}

}  // namespace moe
