// Persistent grouped GEMM on the 5th-generation tensor cores (tcgen05, TMEM
// accumulators) for the six GEMMs of the routed MoE layer.
//
// The pages' design (Primus-Turbo "Mega MoE" README, "Pipeline") runs each
// grouped GEMM tile by tile over the routed rows of every expert, with the
// token dispatch folded into the GEMM.  Here one launch covers every expert:
//
//  * Tiles are 128 routed rows x 256 output columns.  Row-grouped GEMMs walk
//    (M-tile, N-tile) with the M-tile's expert read from the routing tile
//    table; weight-gradient GEMMs walk (expert, M-tile, N-tile) with K running
//    over that expert's block-M padded rows ("variable-K").
//  * The A operand of L1 / L2-dgrad and the token-side operand of dW1 / dW2
//    are GATHERED straight from x or dY by the permutation table (16-byte
//    cp.async into the 128-byte-swizzled layout the MMA reads), so the
//    dispatched activations are never written to memory, in forward or when
//    backward recomputes them (README, "Recompute dispatched x").
//  * Dense operands (weights, saved activations) arrive by TMA.
//  * Warp roles: warps 0-3 epilogue (TMEM -> registers -> global), warp 4 TMA
//    producer, warp 5 MMA issuer and TMEM owner, warps 6.. gather producers.  A
//    4-stage shared-memory ring (full/empty mbarriers) feeds the MMA; two
//    256-column TMEM accumulators let the epilogue of one tile overlap the
//    main loop of the next.
//  * Epilogues fuse SwiGLU (L1), the top-k weight (L2), SwiGLU^T with the
//    routing-weight gradient partials (L2 dgrad).
//  * Every wait is bounded; on a timeout the CTA raises a status flag,
//    drains what it issued, frees TMEM and returns.
#pragma once

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {

template <int F>
struct GemmTraits;
template <>
struct GemmTraits<L1_FWD> {
    static constexpr bool kAGather = true, kBGather = false, kAMN = false, kBMN = true, kWgrad = false;
};
template <>
struct GemmTraits<L2_FWD> {
    static constexpr bool kAGather = false, kBGather = false, kAMN = false, kBMN = true, kWgrad = false;
};
template <>
struct GemmTraits<L2_DGRAD> {
    static constexpr bool kAGather = true, kBGather = false, kAMN = false, kBMN = false, kWgrad = false;
};
template <>
struct GemmTraits<L1_DGRAD> {
    static constexpr bool kAGather = false, kBGather = false, kAMN = false, kBMN = false, kWgrad = false;
};
template <>
struct GemmTraits<DW1> {
    static constexpr bool kAGather = true, kBGather = false, kAMN = true, kBMN = true, kWgrad = true;
};
template <>
struct GemmTraits<DW2> {
    static constexpr bool kAGather = false, kBGather = true, kAMN = true, kBMN = true, kWgrad = true;
};

struct TileCoord {
    int e;      // expert
    int m0;     // first routed row (row-grouped) / first output row (weight gradients)
    int n0;     // first output column (L1_FWD: first gate column)
    int nt;     // column tile index
    int nkb;    // number of 64-wide K blocks
    int krow0;  // first routed row of the expert (weight gradients)
};

// A tile's coordinates come from the routing tables in global memory.  Each
// role reads the next tile's entries right after starting the current tile
// (load_tile_raw), so that latency is hidden behind the current tile's work
// instead of stalling every role at every tile boundary.
//
// Row-grouped GEMMs number their tiles expert by expert, then N tile, then
// M tile: the 2-3 M tiles of one expert that read the same weight tile get
// consecutive numbers, run on neighbouring CTAs at the same time, and share
// that weight tile through L2 (a block of consecutive tiles that straddles
// two waves of the persistent grid splits at most one such group).  Tile t
// belongs to expert e = tiles[t / n_tiles], because expert e owns M tiles
// [offs[e]/128, offs[e+1]/128) and so tile numbers
// [offs[e]/128 * n_tiles, offs[e+1]/128 * n_tiles).
struct TileRaw {
    int a;  // row-grouped: owner expert; weight gradients: counts[e]
    int b;  // offs[e]
    int c;  // row-grouped: offs[e + 1]
};

template <int F>
__device__ __forceinline__ TileRaw load_tile_raw(int tile, const GemmArgs& p) {
    TileRaw r{0, 0, 0};
    if constexpr (GemmTraits<F>::kWgrad) {
        const int e = tile / (p.m_tiles * p.n_tiles);
        r.a = __ldg(p.counts + e);
        r.b = __ldg(p.offs + e);
    } else {
        r.a = __ldg(p.tiles + tile / p.n_tiles);
        r.b = __ldg(p.offs + r.a);
        r.c = __ldg(p.offs + r.a + 1);
    }
    return r;
}

template <int F>
__device__ __forceinline__ TileCoord finish_tile(int tile, TileRaw r, const GemmArgs& p) {
    TileCoord t;
    if constexpr (GemmTraits<F>::kWgrad) {
        const int per_e = p.m_tiles * p.n_tiles;
        t.e = tile / per_e;
        const int rem = tile - t.e * per_e;
        const int mt = rem / p.n_tiles;
        t.nt = rem - mt * p.n_tiles;
        t.m0 = mt * kBM;
        t.n0 = t.nt * kBN;
        t.nkb = (r.a + kBK - 1) / kBK;
        t.krow0 = r.b;
    } else {
        const int ts = r.b / kBM;        // first M tile of expert e
        const int tc = (r.c - r.b) / kBM;  // M tiles of expert e (>= 1 here)
        const int l = tile - ts * p.n_tiles;
        t.nt = l / tc;
        const int mt = ts + (l - t.nt * tc);
        t.e = r.a;
        t.m0 = mt * kBM;
        t.n0 = t.nt * (F == L1_FWD ? kBN / 2 : kBN);
        t.nkb = p.K / kBK;
        t.krow0 = 0;
    }
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
        raw = tile < total ? load_tile_raw<F>(tile, p) : TileRaw{0, 0, 0};
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
    if constexpr (GemmTraits<F>::kWgrad) {
        return p.E * p.m_tiles * p.n_tiles;
    } else {
        int nt = *reinterpret_cast<const volatile int32_t*>(p.status + MOE_STATUS_NUM_TILES);
        nt = nt < 0 ? 0 : (nt > p.tiles_cap ? p.tiles_cap : nt);
        return nt * p.n_tiles;
    }
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
            if constexpr (F == L1_FWD) {
                // W1 viewed as [E][H][2][I]: box = 64 columns of one half x 64 rows of H.
#pragma unroll
                for (int j = 0; j < 4; ++j) tma_load_4d(b + j * 8192, mB, t.n0 + 64 * (j & 1), j >> 1, k0, t.e, fb);
            } else if constexpr (F == L2_FWD) {
                tma_load_2d(a, mA, k0, t.m0, fb);
#pragma unroll
                for (int j = 0; j < 4; ++j) tma_load_3d(b + j * 8192, mB, t.n0 + 64 * j, k0, t.e, fb);
            } else if constexpr (F == L2_DGRAD) {
                tma_load_3d(b, mB, k0, t.n0, t.e, fb);
            } else if constexpr (F == L1_DGRAD) {
                tma_load_2d(a, mA, k0, t.m0, fb);
                tma_load_3d(b, mB, k0, t.n0, t.e, fb);
            } else if constexpr (F == DW1) {
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
// r*128 + ((c ^ (r & 7)) * 16)); each warp owns an equal share of the rows of
// every stage, so several warps' copies are in flight at once.
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
        if constexpr (!Tr::kAMN) {
            // K-major A: the tile's 128 routed rows are fixed; K runs along H.
            constexpr int kRowsPerWarp = kBM / kGatherWarps;
            constexpr int kPerLane = kRowsPerWarp / 4;
            const int rw0 = gw * kRowsPerWarp;
            int tok[kPerLane];
#pragma unroll
            for (int jj = 0; jj < kPerLane; ++jj) {
                const int s = __ldg(p.perm + t.m0 + rw0 + rb + 4 * jj);
                tok[jj] = s >= 0 ? s / k : -1;
            }
            for (int kb = 0; kb < t.nkb; ++kb) {
                if (!warp_wait(bars.empty(stage), phase ^ 1u, abort)) return;
                const uint32_t a = sA + stage * kStageABytes;
                const int col = kb * kBK + c * 8;
#pragma unroll
                for (int jj = 0; jj < kPerLane; ++jj) {
                    const int r = rw0 + rb + 4 * jj;
                    const int tk = tok[jj];
                    const __nv_bfloat16* g = src + (size_t)(tk < 0 ? 0 : tk) * (size_t)H + col;
                    cp_async_16(a + r * 128 + ((c ^ (r & 7)) << 4), g, tk < 0 ? 0u : 16u);
                }
                cp_async_arrive_noinc(bars.full(stage));
                if (++stage == kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        } else {
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
            if constexpr (Tr::kAGather || Tr::kBGather) fence_proxy_async_smem();
            const uint32_t a = sA + stage * kStageABytes;
            const uint32_t b = sB + stage * kStageBBytes;
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk) {
                // K-major: 16 elements = 32 bytes along the swizzled row.
                // MN-major: 16 K rows = 2 KiB; LBO = stride of 64-wide MN slabs.
                const uint64_t ad = Tr::kAMN ? make_sdesc_sw128(a + kk * 2048, 8192, 1024)
                                             : make_sdesc_sw128(a + kk * 32, 16, 1024);
                const uint64_t bd = Tr::kBMN ? make_sdesc_sw128(b + kk * 2048, 8192, 1024)
                                             : make_sdesc_sw128(b + kk * 32, 16, 1024);
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
// swizzled layout of the output tensor map, and leave through TMA bulk
// stores of whole 32-row boxes (full 64- or 128-byte row segments) while the
// warp goes on with the next chunk.
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
        const int row = row0 + lane;

        if constexpr (F == L1_FWD) {
            // SwiGLU: accumulator columns [0,128) are gate, [128,256) up.
            const int I = p.I;
#pragma unroll 1
            for (int cc = 0; cc < 4; ++cc) {
                const int col = t.n0 + 32 * cc;
                if (col >= I) break;
                float g[32], u[32];
                {
                    uint32_t rg[32], ru[32];
                    tmem_ld32_nowait(tacc + 32 * cc, rg);
                    tmem_ld32_nowait(tacc + 128 + 32 * cc, ru);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        g[j] = __uint_as_float(rg[j]);
                        u[j] = __uint_as_float(ru[j]);
                    }
                }
                uint32_t pg[16], pu[16], pa[16];
                pack32(g, pg);
                pack32(u, pu);
#pragma unroll
                for (int j = 0; j < 32; ++j) g[j] = g[j] / (1.0f + __expf(-g[j])) * u[j];
                pack32(g, pa);
                if (lane == 0) bulk_wait_read<0>();
                __syncwarp();
                stage_row_sw64(stage, lane, pg);
                stage_row_sw64(stage + 2048, lane, pu);
                stage_row_sw64(stage + 4096, lane, pa);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(om.c0, col, row0, stage);
                    tma_store_2d(om.c0, I + col, row0, stage + 2048);
                    tma_store_2d(om.c1, col, row0, stage + 4096);
                    bulk_commit();
                }
            }
        } else if constexpr (F == L2_DGRAD) {
            // g = dY . W2^T at this row; da = w * g; SwiGLU^T from the saved h.
            const int s = __ldg(p.perm + row);
            const float wv = s >= 0 ? __ldg(p.topk_w + s) : 0.0f;
            const int I = p.I;
            const size_t hoff = (size_t)row * (size_t)(2 * I);
            const size_t aoff = (size_t)row * (size_t)I;
            float dws = 0.0f;
#pragma unroll 1
            for (int cc = 0; cc < 8; ++cc) {
                const int col = t.n0 + 32 * cc;
                if (col >= I) break;
                float g[32];
                tmem_ld32(tacc + 32 * cc, g);
                uint32_t pg[16], pu[16], pa[16];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int c8 = col + 8 * q;
                    float hg[8], hu[8], av[8];
                    unpack_bf16x8(__ldg(reinterpret_cast<const uint4*>(p.h_in + hoff + c8)), hg);
                    unpack_bf16x8(__ldg(reinterpret_cast<const uint4*>(p.h_in + hoff + I + c8)), hu);
                    unpack_bf16x8(__ldg(reinterpret_cast<const uint4*>(p.a_in + aoff + c8)), av);
                    float dg[8], du[8], aw[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float gj = g[8 * q + j];
                        const float da = wv * gj;
                        const float sg = 1.0f / (1.0f + __expf(-hg[j]));
                        dg[j] = da * hu[j] * sg * (1.0f + hg[j] * (1.0f - sg));
                        du[j] = da * hg[j] * sg;
                        aw[j] = wv * av[j];
                        dws += gj * av[j];
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        pg[4 * q + j] = pack_bf16x2(dg[2 * j], dg[2 * j + 1]);
                        pu[4 * q + j] = pack_bf16x2(du[2 * j], du[2 * j + 1]);
                        pa[4 * q + j] = pack_bf16x2(aw[2 * j], aw[2 * j + 1]);
                    }
                }
                if (lane == 0) bulk_wait_read<0>();
                __syncwarp();
                stage_row_sw64(stage, lane, pg);
                stage_row_sw64(stage + 2048, lane, pu);
                stage_row_sw64(stage + 4096, lane, pa);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(om.c0, col, row0, stage);
                    tma_store_2d(om.c0, I + col, row0, stage + 2048);
                    tma_store_2d(om.c1, col, row0, stage + 4096);
                    bulk_commit();
                }
            }
            p.outf[(size_t)row * (size_t)p.dw_cols + t.nt] = dws;
        } else {
            // One output: o (L2 fwd, times the routing weight), dxp (L1 dgrad),
            // or the weight gradient of expert e (dW1, dW2).
            constexpr bool kW = GemmTraits<F>::kWgrad;
            const int N_out = (F == DW1) ? 2 * p.I : p.H;
            float wv = 1.0f;
            if constexpr (F == L2_FWD) {
                const int s = __ldg(p.perm + row);
                wv = s >= 0 ? __ldg(p.topk_w + s) : 0.0f;
            }
            const bool have_acc = !kW || t.nkb > 0;
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
                        pk[j] = pack_bf16x2(wv * __uint_as_float(r0[2 * j]), wv * __uint_as_float(r0[2 * j + 1]));
                        pk[16 + j] = pack_bf16x2(wv * __uint_as_float(r1[2 * j]), wv * __uint_as_float(r1[2 * j + 1]));
                    }
                }
                const uint32_t buf = stage + (nstore & 1u) * 4096u;
                if (lane == 0) bulk_wait_read<1>();
                __syncwarp();
                stage_row_sw128(buf, lane, pk);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    if constexpr (kW) tma_store_3d(om.c0, col, row0, t.e, buf);
                    else tma_store_2d(om.c0, col, row0, buf);
                    bulk_commit();
                }
                ++nstore;
            }
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
        constexpr uint32_t kFullCount = 1u + ((Tr::kAGather || Tr::kBGather) ? 32u * kGatherWarps : 0u);
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
        if constexpr (F == L1_FWD || F == L2_DGRAD) tma_prefetch_map(&mapC1);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int total = total_tiles<F>(p);

    if (warp == kWarpTma) {
        if (lane == 0) role_tma<F>(&mapA, &mapB, p, total, sA, sB, bars, abort);
    } else if (warp >= kWarpGather0) {
        if constexpr (Tr::kAGather || Tr::kBGather)
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
