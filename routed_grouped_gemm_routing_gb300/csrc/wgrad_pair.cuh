// Weight gradients of the routed MoE layer on SM pairs (tcgen05 cta_group::2)
// with the gathered token operand kept in shared memory:
//   dW1[e] = gather(x)_e^T . dh_e        dW2[e] = aw_e^T . gather(dY)_e
// (Primus-Turbo "Mega MoE" README, "Pipeline": the backward's variable-K
// weight-gradient GEMMs, K = the expert's routed rows; the dispatched x is
// recomputed by gathering it again, section "Recompute dispatched x in
// backward").
//
// A work unit is (expert e, stationary tile s): 256 features of H, 128 in
// each CTA of a 2-CTA cluster.  Each CTA gathers its 128 features of the
// token operand (x for dW1, dY for dW2) for all of the expert's routed rows
// ONCE into a shared-memory slab (up to S 64-row K blocks), and then
// streams the other operand (dh for dW1, aw for dW2) by TMA, 128 of its
// features per CTA at a time, through a ring of 6 (S = 5) or 5 (S = 7)
// stages.  For every streamed
// tile t the pair issues M=256 x N=256 MMAs over the expert's rows:
//   dW1: A = slab (M = H features), B = dh (N = 2I features)
//   dW2: A = aw   (M = I features), B = slab (N = H features)
// so each CTA's TMEM holds 128 output rows x 256 output columns of dW[e]
// and leaves through a TMA-store epilogue (32-row boxes of 64 columns).
// The token operand is gathered once per unit instead of once per output
// tile (16x fewer gathered bytes for dW1, 8x for dW2), and each SM streams
// 16 KiB per K block instead of 48 KiB.
//
// Experts with more rows than the slab holds run K in chunks of S blocks,
// the slab gathered again for every round of tiles (w_group).  An expert
// without routed rows gets zeros.
//
// The streamed tiles of a unit start at tile (s mod T) so that the clusters
// of one expert's stationary tiles read different rows at any moment, and
// the weight-gradient stores are marked evict-first in L2 so that the
// streamed rows, re-read by those clusters, stay there.
//
// Roles (per CTA, 14 warps): 0-3 epilogue, 4 TMA producer (streamed
// operand), 5 MMA issuer on the even CTA / relay on the odd CTA (forwards
// "this CTA's half of a slab block has landed"), 6-13 gather producers
// (slab).  Both CTAs' TMA loads of a stage complete one barrier in the even
// CTA, so the MMA thread waits once per stage: issuing a tcgen05.mma costs
// the thread about two thirds of the MMA's own pipe time, so every extra
// wait in its loop would leave the tensor pipe idle.  Every wait is
// bounded, as in the other GEMM kernels.
#pragma once

#include "grouped_gemm_2sm.cuh"

namespace moe {

// Eleven 16 KiB operand blocks per CTA (twelve with S = 7, below), S of
// them for the slab (S 64-row K blocks: 64 S routed rows) and the rest for
// the streamed ring.  S = 5 (320 rows, 6 ring stages) unless the shape's
// mean rows per expert, T k / E, exceed 320; then S = 7 (448 rows, 5
// stages), so that such experts fit the slab (a 4-stage ring starves the
// 256-row experts of the V3-shaped layer, measured: dW1 3.2 -> 4.0 ms; 7
// slab blocks cut the V2-Lite-shaped layer's dW1 0.30 -> 0.24 ms and dW2
// 0.17 -> 0.12 ms).
constexpr int kWBlocks = 11;
constexpr int kWBlockBytes = 128 * kBK * 2;  // 16 KiB: 128 features x 64 rows, MN-major, 128B swizzle
constexpr int kWSlabSmall = 5, kWSlabLarge = 7;
constexpr int kWTailBytes = 512;
static_assert(8 * (3 * kWSlabLarge + 2 * (kWBlocks + 1 - kWSlabLarge) + 5) + 8 <= kWTailBytes &&
                  8 * (3 * kWSlabSmall + 2 * (kWBlocks - kWSlabSmall) + 5) + 8 <= kWTailBytes,
              "barrier area");
constexpr int kWSmemBytes = 1024 + kWBlocks * kWBlockBytes + kEpiWarps * kStageEpiBytes + kWTailBytes;
static_assert(kWSmemBytes <= 232448, "shared memory per CTA");
// With the 7-block slab the ring gets a fifth stage in place of the second
// 4 KiB store buffer of each epilogue warp (the same shared memory): the
// streamed operand's latency, not the epilogue, held the MMAs back there
// (V2-Lite-shaped layer, per-role cycle counters: the MMA warp waited 35 %
// of its time for streamed blocks with four stages; dW1 0.240 -> 0.226 ms).
template <int S>
__host__ __device__ constexpr int w_blocks() {
    return S == kWSlabLarge ? kWBlocks + 1 : kWBlocks;
}
template <int S>
__host__ __device__ constexpr int w_store_bufs() {  // 4 KiB store buffers per epilogue warp
    return S == kWSlabLarge ? 1 : 2;
}
static_assert(1024 + w_blocks<kWSlabLarge>() * kWBlockBytes + kEpiWarps * 4096 * w_store_bufs<kWSlabLarge>() +
                      kWTailBytes == kWSmemBytes &&
                  4096 * w_store_bufs<kWSlabSmall>() == kStageEpiBytes,
              "both slab sizes lay out the same shared memory");

template <int S>
struct WBars {
    static constexpr int kSlab = S, kStages = w_blocks<S>() - S;
    static constexpr int kNum = 3 * kSlab + 2 * kStages + 5;  // barriers
    uint32_t base;
    __device__ __forceinline__ uint32_t slab_full(int i) const { return base + 8u * i; }
    __device__ __forceinline__ uint32_t peer_slab_full(int i) const { return base + 8u * (kSlab + i); }
    __device__ __forceinline__ uint32_t slab_empty(int i) const { return base + 8u * (2 * kSlab + i); }
    // full: the even CTA's barrier counts both CTAs' bytes of a stage
    __device__ __forceinline__ uint32_t full(int s) const { return base + 8u * (3 * kSlab + s); }
    __device__ __forceinline__ uint32_t empty(int s) const { return base + 8u * (3 * kSlab + kStages + s); }
    __device__ __forceinline__ uint32_t tfull(int a) const { return base + 8u * (3 * kSlab + 2 * kStages + a); }
    __device__ __forceinline__ uint32_t tempty(int a) const {
        return base + 8u * (3 * kSlab + 2 * kStages + 2 + a);
    }
    __device__ __forceinline__ uint32_t drain() const { return base + 8u * (3 * kSlab + 2 * kStages + 4); }
};

// Shape of one unit (an expert's stationary tile; its streamed tiles run over
// 2I for dW1, over I for dW2).
struct WUnit {
    int e, s;
    int off;  // first routed row of the expert
    int cnt;  // routed rows of the expert
    int nkb;  // 64-row K blocks
    int nch;  // K chunks of at most S blocks (the slab)
};

// Experts in decreasing order of routed rows (ties by id), built in shared
// memory at kernel start just past the kernel's fixed shared memory (8 bytes
// per expert): the units of the heaviest experts are dealt first.
static_assert(kWSmemBytes + 8 * kMaxExperts <= 232448, "shared memory per CTA with the expert order");
__device__ __forceinline__ const int32_t* w_order_smem() {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    return reinterpret_cast<const int32_t*>(smem_raw + (base - raw) + (kWSmemBytes - 1024));
}

// Static walk.  Units (expert, stationary tile) are numbered heaviest expert
// first and dealt to the clusters in rounds, serpentine (round r goes to
// clusters 0..n-1 when r is even, n-1..0 when odd), so that with skewed
// routing every cluster gets a similar share of the rows; all roles of a
// CTA walk the same sequence.  The next unit's count and offset are read
// while the current one runs.
template <int S>
struct WWalk {
    const GemmArgs& p;
    const int32_t* order;  // experts by decreasing count
    int total, n, ncl, c, unit;
    int cnt, off;
    __device__ __forceinline__ WWalk(const GemmArgs& p_)
        : p(p_),
          order(w_order_smem()),
          total(p_.E * p_.m_tiles),
          n(0),
          ncl((int)gridDim.x >> 1),
          c((int)blockIdx.x >> 1) {
        unit = map(0);
        if (unit < total) load(unit);
    }
    __device__ __forceinline__ int map(int r) const { return r * ncl + ((r & 1) ? ncl - 1 - c : c); }
    __device__ __forceinline__ int expert(int u) const { return order[u / p.m_tiles]; }
    __device__ __forceinline__ void load(int u) {
        const int e = expert(u);
        cnt = __ldg(p.counts + e);
        off = __ldg(p.offs + e);
    }
    __device__ __forceinline__ bool valid() const { return unit < total; }
    __device__ __forceinline__ WUnit take() {
        WUnit w;
        w.e = expert(unit);
        w.s = unit % p.m_tiles;
        w.cnt = cnt;
        w.off = off;
        w.nkb = (cnt + kBK - 1) / kBK;
        w.nch = (w.nkb + S - 1) / S;
        const int nxt = map(n + 1);
        if (nxt < total) load(nxt);
        return w;
    }
    __device__ __forceinline__ void next() {
        ++n;
        unit = map(n);
    }
};

// Streamed tiles per slab round.  An expert whose rows fit the slab gathers
// it once for all its tiles.  A longer one gathers each chunk of its rows
// again for every round: per tile when it has two chunks (groups of one
// tile keep the two TMEM accumulators double-buffered), per pair of tiles
// from three chunks on (the pair accumulates in both accumulators side by
// side, so the gathered bytes halve while the epilogue no longer overlaps
// the pair's MMAs, which then take long anyway).  Measured with skewed
// routing (top expert 5649 rows): dW1 4.75 -> 4.42 ms, dW2 2.34 -> 2.22 ms.
__device__ __forceinline__ int w_group(const WUnit& u) { return u.nch > 2 ? 2 : 1; }

// K blocks [kb0, kb1) of chunk c.
template <int S>
__device__ __forceinline__ int w_kb0(int c) { return c * S; }
template <int S>
__device__ __forceinline__ int w_kb1(const WUnit& u, int c) { return min(u.nkb, (c + 1) * S); }

// ------------------------------------------------------------ TMA producer
// Streamed operand: 128 features (this CTA's half of the tile's 256) x 64 rows
// per K block, two 64 x 64 boxes, completing the even CTA's full barrier
// (which the even CTA's producer arms with both CTAs' bytes).
template <int F, int S>
__device__ void w_role_tma(const CUtensorMap* mS, const GemmArgs& p, uint32_t sS, WBars<S> bars, volatile int* abort,
                           int rank) {
    int stage = 0;
    uint32_t phase = 0;
    const int T = p.n_tiles;
    for (WWalk<S> w(p); w.valid(); w.next()) {
        const WUnit u = w.take();
        const int G = w_group(u);
        if (G == 1) {
            for (int t = 0; t < T; ++t) {
                const int tt = (t + u.s) % T;  // streamed tiles rotated per stationary tile
                const int f0 = tt * 256 + 128 * rank;
                for (int kb = 0; kb < u.nkb; ++kb) {
                    if (!mbar_wait(bars.empty(stage), phase ^ 1u, abort)) return;
                    if (rank == 0) mbar_arrive_expect_tx(bars.full(stage), 2u * kWBlockBytes);
                    const uint32_t fb = cluster_addr_of(bars.full(stage), 0);
                    const uint32_t dst = sS + stage * kWBlockBytes;
                    // the expert's streamed rows are read again by the other
                    // stationary tiles' clusters: keep them in L2 against the
                    // stream of weight-gradient stores (stored evict-first)
                    const uint64_t pol = l2_policy_evict_last();
                    tma_load_2d_pair_hint(dst, mS, f0, u.off + kb * kBK, fb, pol);
                    tma_load_2d_pair_hint(dst + 8192, mS, f0 + 64, u.off + kb * kBK, fb, pol);
                    if (++stage == WBars<S>::kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            continue;
        }
        // paired tiles: for each K block, the block of both tiles in turn
        for (int t0 = 0; t0 < T; t0 += G) {
            const int nt = min(G, T - t0);
            for (int kb = 0; kb < u.nkb; ++kb) {
                for (int j = 0; j < nt; ++j) {
                    const int tt = (t0 + j + u.s) % T;
                    const int f0 = tt * 256 + 128 * rank;
                    if (!mbar_wait(bars.empty(stage), phase ^ 1u, abort)) return;
                    if (rank == 0) mbar_arrive_expect_tx(bars.full(stage), 2u * kWBlockBytes);
                    const uint32_t fb = cluster_addr_of(bars.full(stage), 0);
                    const uint32_t dst = sS + stage * kWBlockBytes;
                    const uint64_t pol = l2_policy_evict_last();
                    tma_load_2d_pair_hint(dst, mS, f0, u.off + kb * kBK, fb, pol);
                    tma_load_2d_pair_hint(dst + 8192, mS, f0 + 64, u.off + kb * kBK, fb, pol);
                    if (++stage == WBars<S>::kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
    }
}

// --------------------------------------------------------- gather producer
// The slab: this CTA's 128 features of the token operand over the rows of K
// blocks [kb0, kb1), block kb in slot kb - kb0; 16-byte cp.async chunks into
// the 128-byte-swizzled MN-major layout (row r of a 64-feature region at
// r*128, chunk c at (c ^ (r & 7)) * 16); padding rows (perm = -1) and
// features past H are zero-filled.
template <int S>
__device__ __forceinline__ void w_gather_round(const GemmArgs& p, const WUnit& u, int kb0, int kb1, uint32_t sL,
                                               WBars<S> bars, uint32_t& sphase, volatile int* abort, int gw, int lane,
                                               int rank, bool& ok) {
    constexpr int kRowsPerWarp = kBK / kGatherWarps;  // 8
    const int c = lane & 7;
    const int rb = lane >> 3;
    const int H = p.H, k = p.k;
    const int rw0 = gw * kRowsPerWarp;
    const int col0 = u.s * 256 + 128 * rank;
    // permutation entries of this warp's rows in every block of the round
    int ent[S];
#pragma unroll
    for (int i = 0; i < S; ++i)
        ent[i] = (kb0 + i < kb1) ? __ldg(p.perm + u.off + (kb0 + i) * kBK + rw0 + (lane & (kRowsPerWarp - 1))) : -1;
#pragma unroll
    for (int i = 0; i < S; ++i) {
        if (kb0 + i >= kb1) break;
        if (!warp_wait(bars.slab_empty(i), ((sphase >> i) & 1u) ^ 1u, abort)) {
            ok = false;
            return;
        }
        const int tcur = ent[i] >= 0 ? ent[i] / k : -1;
        const int tq0 = __shfl_sync(0xffffffffu, tcur, rb);
        const int tq1 = __shfl_sync(0xffffffffu, tcur, rb + 4);
        const uint32_t dst0 = sL + i * kWBlockBytes;
#pragma unroll
        for (int g = 0; g < 2; ++g) {
            const int colg = col0 + 64 * g + 8 * c;
            const bool okc = colg < H;
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int tq = q ? tq1 : tq0;
                const int r = rw0 + rb + 4 * q;
                const bool v = okc && tq >= 0;
                const __nv_bfloat16* gp = p.gsrc + (v ? (size_t)tq * (size_t)H + colg : (size_t)0);
                cp_async_16(dst0 + g * 8192 + r * 128 + ((c ^ (r & 7)) << 4), gp, v ? 16u : 0u);
            }
        }
        cp_async_arrive_noinc(bars.slab_full(i));
        sphase ^= 1u << i;
    }
}

template <int S>
__device__ void w_role_gather(const GemmArgs& p, uint32_t sL, WBars<S> bars, volatile int* abort, int gw, int lane,
                              int rank) {
    uint32_t sphase = 0;
    bool ok = true;
    const int T = p.n_tiles;
    for (WWalk<S> w(p); w.valid() && ok; w.next()) {
        const WUnit u = w.take();
        if (u.nch == 1) {
            w_gather_round<S>(p, u, 0, u.nkb, sL, bars, sphase, abort, gw, lane, rank, ok);
        } else {
            for (int t0 = 0; t0 < T && ok; t0 += w_group(u))
                for (int c = 0; c < u.nch && ok; ++c)
                    w_gather_round<S>(p, u, w_kb0<S>(c), w_kb1<S>(u, c), sL, bars, sphase, abort, gw, lane, rank, ok);
        }
    }
}

// -------------------------------------------------------------- MMA issuer
// The whole MMA warp runs this loop: it waits warp-uniformly and one elected
// lane issues the MMAs and their commits (see warp_wait_uniform).
template <int F, int S>
__device__ void w_role_mma(const GemmArgs& p, uint32_t sL, uint32_t sS, WBars<S> bars, uint32_t tmem_base,
                           volatile int* abort) {
    constexpr uint32_t idesc = make_idesc_bf16(2 * kBM, 256, true, true);
    int stage = 0;
    uint32_t phase = 0, sphase = 0;
    int it = 0;
    const int T = p.n_tiles;
    for (WWalk<S> w(p); w.valid(); w.next()) {
        const WUnit u = w.take();
        if (w_group(u) == 1) {
            for (int t = 0; t < T; ++t, ++it) {
                const int acc = it & 1;
                const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
                if (!warp_wait_uniform<true>(bars.tempty(acc), acc_phase ^ 1u, abort)) return;
                tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(acc * 256);
                for (int c = 0; c < u.nch; ++c) {
                    const int kb0 = w_kb0<S>(c), kb1 = w_kb1<S>(u, c);
                    // the slab blocks of this round are waited for on their first
                    // use and released after their last one
                    const bool first = u.nch > 1 || t == 0;
                    const bool last = u.nch > 1 || t == T - 1;
                    for (int kb = kb0; kb < kb1; ++kb) {
                        const int i = kb - kb0;
                        if (first) {
                            if (!warp_wait_uniform<false>(bars.slab_full(i), (sphase >> i) & 1u, abort)) return;
                            if (!warp_wait_uniform<true>(bars.peer_slab_full(i), (sphase >> i) & 1u, abort)) return;
                        }
                        if (!warp_wait_uniform<true>(bars.full(stage), phase, abort)) return;
                        tc_fence_after();
                        const uint32_t sl = sL + i * kWBlockBytes;
                        const uint32_t st = sS + stage * kWBlockBytes;
                        // descriptors of the block's first 16 rows; the next 16 rows
                        // start 2048 bytes (128 descriptor units) further on
                        const uint64_t ad = make_sdesc_sw128((F == DW1) ? sl : st, 8192, 1024);
                        const uint64_t bd = make_sdesc_sw128((F == DW1) ? st : sl, 8192, 1024);
                        // stop at the 16-row step that holds the expert's last row
                        const int ksteps = min(kBK / 16, (u.cnt - kb * kBK + 15) / 16);
                        if (elect_one()) {
                            if (first) fence_proxy_async_smem();  // a slab block freshly written by cp.async
    #pragma unroll
                            for (int kk = 0; kk < kBK / 16; ++kk) {
                                if (kk >= ksteps) break;
                                tc_mma_bf16_pair(d, ad + 128u * kk, bd + 128u * kk, idesc, (kb | kk) != 0 ? 1u : 0u);
                            }
                            tc_commit_pair(bars.empty(stage));
                            if (last) tc_commit_pair(bars.slab_empty(i));
                        }
                        __syncwarp();
                        if (last) sphase ^= 1u << i;
                        if (++stage == WBars<S>::kStages) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
                if (elect_one()) tc_commit_pair(bars.tfull(acc));
                __syncwarp();
            }
            continue;
        }
        // an expert of three or more slab chunks: its tiles go in pairs (see w_group)
        const int G = 2;
        for (int t0 = 0; t0 < T; t0 += G) {
            const int nt = min(G, T - t0);
            // tiles it .. it + nt - 1 accumulate side by side (acc = it & 1)
            for (int j = 0; j < nt; ++j)
                if (!warp_wait_uniform<true>(bars.tempty((it + j) & 1), ((uint32_t)((it + j) >> 1) & 1u) ^ 1u, abort))
                    return;
            tc_fence_after();
            for (int c = 0; c < u.nch; ++c) {
                const int kb0 = w_kb0<S>(c), kb1 = w_kb1<S>(u, c);
                // the slab blocks of this round are waited for on their first
                // use and released after their last one
                const bool first = u.nch > 1 || t0 == 0;
                const bool last = u.nch > 1 || t0 + nt == T;
                for (int kb = kb0; kb < kb1; ++kb) {
                    const int i = kb - kb0;
                    if (first) {
                        if (!warp_wait_uniform<false>(bars.slab_full(i), (sphase >> i) & 1u, abort)) return;
                        if (!warp_wait_uniform<true>(bars.peer_slab_full(i), (sphase >> i) & 1u, abort)) return;
                    }
                    // stop at the 16-row step that holds the expert's last row
                    const int ksteps = min(kBK / 16, (u.cnt - kb * kBK + 15) / 16);
                    const uint32_t sl = sL + i * kWBlockBytes;
                    for (int j = 0; j < nt; ++j) {
                        if (!warp_wait_uniform<true>(bars.full(stage), phase, abort)) return;
                        tc_fence_after();
                        const uint32_t st = sS + stage * kWBlockBytes;
                        const uint32_t d = tmem_base + (uint32_t)(((it + j) & 1) * 256);
                        // descriptors of the block's first 16 rows; the next 16 rows
                        // start 2048 bytes (128 descriptor units) further on
                        const uint64_t ad = make_sdesc_sw128((F == DW1) ? sl : st, 8192, 1024);
                        const uint64_t bd = make_sdesc_sw128((F == DW1) ? st : sl, 8192, 1024);
                        if (elect_one()) {
                            if (first && j == 0) fence_proxy_async_smem();  // a slab block freshly written by cp.async
#pragma unroll
                            for (int kk = 0; kk < kBK / 16; ++kk) {
                                if (kk >= ksteps) break;
                                tc_mma_bf16_pair(d, ad + 128u * kk, bd + 128u * kk, idesc, (kb | kk) != 0 ? 1u : 0u);
                            }
                            tc_commit_pair(bars.empty(stage));
                            if (last && j == nt - 1) tc_commit_pair(bars.slab_empty(i));
                        }
                        __syncwarp();
                        if (++stage == WBars<S>::kStages) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    if (last) sphase ^= 1u << i;
                }
            }
            for (int j = 0; j < nt; ++j)
                if (elect_one()) tc_commit_pair(bars.tfull((it + j) & 1));
            __syncwarp();
            it += nt;
        }
    }
}

// The odd CTA's MMA thread: tells the even CTA that this CTA's half of a
// slab block is in shared memory, in the order the MMA uses the blocks.
template <int S>
__device__ void w_role_relay(const GemmArgs& p, WBars<S> bars, volatile int* abort) {
    uint32_t sphase = 0;
    const int T = p.n_tiles;
    for (WWalk<S> w(p); w.valid(); w.next()) {
        const WUnit u = w.take();
        const int G = w_group(u);
        for (int t0 = 0; t0 < T; t0 += G) {
            const int nt = min(G, T - t0);
            for (int c = 0; c < u.nch; ++c) {
                const int kb0 = w_kb0<S>(c), kb1 = w_kb1<S>(u, c);
                const bool first = u.nch > 1 || t0 == 0;
                const bool last = u.nch > 1 || t0 + nt == T;
                for (int kb = kb0; kb < kb1; ++kb) {
                    const int i = kb - kb0;
                    if (first) {
                        if (!mbar_wait(bars.slab_full(i), (sphase >> i) & 1u, abort)) return;
                        fence_proxy_async_smem();
                        mbar_arrive_cluster(cluster_addr_of(bars.peer_slab_full(i), 0));
                    }
                    if (last) sphase ^= 1u << i;
                }
            }
        }
    }
}

// ---------------------------------------------------------------- epilogue
// Warp w drains TMEM lanes 32w..32w+31 (32 output rows) x 256 columns as four
// 32 x 64 bf16 boxes in the 128-byte swizzle, each leaving by TMA store.
// kMG (FP32 main-grad accumulation): eight 32 x 32 FP32 boxes instead, each
// added element-wise to the caller's FP32 gradient by a TMA reduce-add; an
// expert without routed rows adds nothing.
template <int F, bool kMG, int S>
__device__ void w_role_epilogue(const GemmArgs& p, const CUtensorMap* mC, WBars<S> bars, uint32_t tmem_base,
                                uint32_t stage, volatile int* abort, int warp, int lane, int rank) {
    const uint32_t tempty_leader[2] = {cluster_addr_of(bars.tempty(0), 0), cluster_addr_of(bars.tempty(1), 0)};
    const int T = p.n_tiles;
    // dW1 is [E][H][2I], dW2 is [E][I][H]
    const int rows_out = (F == DW1) ? p.H : p.I;
    const int cols_out = (F == DW1) ? 2 * p.I : p.H;
    int it = 0;
    uint32_t nstore = 0;
    for (WWalk<S> w(p); w.valid(); w.next()) {
        const WUnit u = w.take();
        for (int t = 0; t < T; ++t, ++it) {
            const int acc = it & 1;
            const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
            if (!warp_wait(bars.tfull(acc), acc_phase, abort)) {
                if (lane == 0) bulk_wait_all();
                return;
            }
            tc_fence_after();
            const uint32_t tacc = tmem_base + (uint32_t)(acc * 256) + ((uint32_t)(warp * 32) << 16);
            const int tt = (t + u.s) % T;
            const int row0 = ((F == DW1) ? u.s : tt) * 256 + 128 * rank + 32 * warp;
            const int colb = ((F == DW1) ? tt : u.s) * 256;
            const bool have_acc = u.nkb > 0;
            if constexpr (kMG) {
#pragma unroll 1
                for (int c32 = 0; c32 < 8 && have_acc; ++c32) {
                    const int col = colb + 32 * c32;
                    if (row0 >= rows_out || col >= cols_out) break;
                    uint32_t r0[32];
                    tmem_ld32_nowait(tacc + 32 * c32, r0);
                    tmem_ld_wait();
                    const uint32_t buf = stage + (nstore % (uint32_t)w_store_bufs<S>()) * 4096u;
                    if (lane == 0) {
                        if constexpr (w_store_bufs<S>() == 1)
                            bulk_wait_read<0>();
                        else
                            bulk_wait_read<1>();
                    }
                    __syncwarp();
                    stage_row_sw128(buf, lane, r0);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_reduce_add_3d(mC, col, row0, u.e, buf);
                        bulk_commit();
                    }
                    ++nstore;
                }
            } else {
#pragma unroll 1
                for (int c64 = 0; c64 < 4; ++c64) {
                    const int col = colb + 64 * c64;
                    if (row0 >= rows_out || col >= cols_out) break;
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
                    const uint32_t buf = stage + (nstore % (uint32_t)w_store_bufs<S>()) * 4096u;
                    if (lane == 0) {
                        if constexpr (w_store_bufs<S>() == 1)
                            bulk_wait_read<0>();
                        else
                            bulk_wait_read<1>();
                    }
                    __syncwarp();
                    stage_row_sw128(buf, lane, pk);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_3d_hint(mC, col, row0, u.e, buf, l2_policy_evict_first());
                        bulk_commit();
                    }
                    ++nstore;
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(tempty_leader[acc]);
        }
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
}

// mapS: the streamed operand (dh for dW1, aw for dW2), box 64 x 64;
// mapC: the weight gradient [E][rows][cols], bf16 box 64 x 32 (kMG: the FP32
// main gradient, box 32 x 32).
template <int F, bool kMG, int S>
__global__ void __launch_bounds__(kGemmThreads, 1)
    moe_wgrad_pair_kernel(const __grid_constant__ CUtensorMap mapS, const __grid_constant__ CUtensorMap mapC,
                          const GemmArgs p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw);
    const uint32_t sL = base;                               // slab: S blocks
    const uint32_t sS = sL + S * kWBlockBytes;              // streamed ring: w_blocks<S>() - S blocks
    const uint32_t sE = base + w_blocks<S>() * kWBlockBytes;     // epilogue staging
    const uint32_t bar_base = sE + kEpiWarps * 4096u * (uint32_t)w_store_bufs<S>();
    uint8_t* tail = base_ptr + (bar_base - base);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tail + 8 * WBars<S>::kNum);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const WBars<S> bars{bar_base};
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int rank = (int)cluster_ctarank();

    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(bars.slab_full(i), 32u * kGatherWarps);
            mbar_init(bars.peer_slab_full(i), 1);
            mbar_init(bars.slab_empty(i), 1);
        }
        for (int s = 0; s < WBars<S>::kStages; ++s) {
            mbar_init(bars.full(s), 1);
            mbar_init(bars.empty(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(bars.tfull(a), 1);
            mbar_init(bars.tempty(a), 2 * kEpiWarps);
        }
        mbar_init(bars.drain(), 1);
        *abort = 0;
        fence_mbar_init();
    }
    if (warp == kWarpMma) {
        tmem_alloc_pair(smem_addr(tmem_slot), 512);
        tmem_relinquish_pair();
    }
    if (warp == kWarpTma && lane == 0) {
        tma_prefetch_map(&mapS);
        tma_prefetch_map(&mapC);
    }
    {
        // rank of expert e = the experts with more routed rows, or as many
        // and a smaller id; order[rank] = e
        int32_t* ord = reinterpret_cast<int32_t*>(base_ptr + (kWSmemBytes - 1024));
        int32_t* cnt = ord + p.E;
        for (int e = threadIdx.x; e < p.E; e += blockDim.x) cnt[e] = __ldg(p.counts + e);
        __syncthreads();
        for (int e = threadIdx.x; e < p.E; e += blockDim.x) {
            const int ce = cnt[e];
            int r = 0;
            for (int f = 0; f < p.E; ++f) {
                const int cf = cnt[f];
                r += (cf > ce || (cf == ce && f < e)) ? 1 : 0;
            }
            ord[r] = e;
        }
        // visible to every role after the cluster barrier below
    }
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == kWarpTma) {
        if (lane == 0) w_role_tma<F, S>(&mapS, p, sS, bars, abort, rank);
    } else if (warp >= kWarpGather0) {
        w_role_gather<S>(p, sL, bars, abort, warp - kWarpGather0, lane, rank);
        cp_async_wait_all();
    } else if (warp == kWarpMma) {
        if (rank == 0) {
            w_role_mma<F, S>(p, sL, sS, bars, tmem_base, abort);
            const bool aborted = __any_sync(0xffffffffu, *abort != 0);
            if (elect_one() && aborted) {
                // let every MMA already issued (by this same elected lane)
                // finish before TMEM is released
                tc_commit_pair_local(bars.drain());
                const uint64_t t0 = global_timer_ns();
                while (!mbar_try_wait(bars.drain(), 0) && global_timer_ns() - t0 < 100000000ull) {
                }
            }
            __syncwarp();
        } else if (lane == 0) {
            w_role_relay<S>(p, bars, abort);
        }
    } else {
        w_role_epilogue<F, kMG, S>(p, &mapC, bars, tmem_base, sE + warp * 4096u * (uint32_t)w_store_bufs<S>(), abort,
                                   warp, lane, rank);
    }
    if (warp == kWarpTma && lane == 0 && *abort) {
        const uint64_t t0 = global_timer_ns();
        while (global_timer_ns() - t0 < 2000000ull) {
        }
    }
    __syncwarp();
    tc_fence_before();
    cluster_sync();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, 512);
    }
    if (threadIdx.x == 0 && *abort) atomicOr(reinterpret_cast<int*>(p.status + MOE_STATUS_FLAGS), 1);
}

// One 2-CTA cluster per unit up to the clusters that fit at once
// (persistent, static unit stride).  a.m_tiles = stationary tiles per expert
// (ceil(H / 256)), a.n_tiles = streamed tiles (ceil(2I / 256) for dW1,
// ceil(I / 256) for dW2).
template <int F, bool kMG, int S>
int launch_wgrad_pair_s(const GemmArgs& a, const CUtensorMap& mapS, const CUtensorMap& mapC, cudaStream_t st) {
    // filled on the first call per device; host threads may race to fill it
    // with the same value
    static std::atomic<int> clusters_fit[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return (int)e;
    if (dev < 0 || dev >= kMaxDevices) return (int)cudaErrorInvalidDevice;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(kGemmThreads, 1, 1);
    // the expert order (and the counts it is built from) follow the fixed part
    if (a.E < 1 || a.E > kMaxExperts) return (int)cudaErrorInvalidValue;
    cfg.dynamicSmemBytes = kWSmemBytes + 8 * (size_t)a.E;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int fit = clusters_fit[dev].load(std::memory_order_relaxed);
    if (fit == 0) {
        // set once per device, outside any stream capture (on the first call)
        e = cudaFuncSetAttribute(moe_wgrad_pair_kernel<F, kMG, S>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kWSmemBytes + 8 * kMaxExperts);
        if (e != cudaSuccess) return (int)e;
        int sms = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return (int)e;
        cfg.gridDim = dim3((unsigned)(sms & ~1), 1, 1);
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, moe_wgrad_pair_kernel<F, kMG, S>, &cfg);
        if (e != cudaSuccess) return (int)e;
        if (n < 1) return (int)cudaErrorInvalidConfiguration;
        fit = n;
        clusters_fit[dev].store(n, std::memory_order_relaxed);
    }
    const long long units = (long long)a.E * a.m_tiles;
    if (units <= 0) return 0;
    const int clusters = units < fit ? (int)units : fit;
    cfg.gridDim = dim3((unsigned)(2 * clusters), 1, 1);
    e = cudaLaunchKernelEx(&cfg, moe_wgrad_pair_kernel<F, kMG, S>, mapS, mapC, a);
    if (e != cudaSuccess) return (int)e;
    return (int)cudaGetLastError();
}

// The slab / ring split from the shape (no routing statistic is read on the
// host): the large slab when the mean rows per expert exceed the small one.
template <int F, bool kMG = false>
int launch_wgrad_pair(const GemmArgs& a, const CUtensorMap& mapS, const CUtensorMap& mapC, cudaStream_t st) {
    const long long mean_rows = a.E > 0 ? (long long)a.T * a.k / a.E : 0;
    if (mean_rows > (long long)kWSlabSmall * kBK) return launch_wgrad_pair_s<F, kMG, kWSlabLarge>(a, mapS, mapC, st);
    return launch_wgrad_pair_s<F, kMG, kWSlabSmall>(a, mapS, mapC, st);
}

}  // namespace moe
