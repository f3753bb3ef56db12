// Row-grouped GEMMs of the routed MoE layer on SM pairs (tcgen05 cta_group::2),
// computed transposed: out^T[features x rows] = W^T . X^T.
//
// The pages' kernels tile these GEMMs over the routed rows of each expert
// (Primus-Turbo "Mega MoE" README, "Pipeline").  Here the MMA's M is 256
// output features of one expert (128 in each CTA of a 2-CTA cluster, taken
// from that expert's weights) and its N is a chunk of up to 256 of the
// expert's routed rows, split 128 + 128 between the two CTAs.  Because N
// runs in steps of 16, an expert's rows are padded to 32 instead of to a
// whole 128-row tile, and because each CTA loads only its half of the
// activations and its own 128 weight columns, an SM needs 32 KiB of
// operands per 64-deep K block instead of the 48 KiB of a one-SM
// 128 x 256 tile, so the same tensor-core work needs two thirds of the
// L2-to-SM bandwidth.
//
// Work units: (expert e, feature tile ft, row chunk j).  Expert e's rows are
// cut into nsub = ceil(count / 256) chunks of equal size (rounded up to 32);
// the routing prologue's pair tables order the experts by decreasing count
// and give each expert's first chunk in that order (pair_offs) and the
// owner of every chunk (pair_owner).  Units are numbered expert by expert
// in that order, then feature tile, then chunk, and handed to the clusters
// at run time from both ends of the numbering (unit feed below), so the
// chunks that stream the same weight tile run at the same time on
// different clusters and share it in L2.
//
// Roles (per CTA, 15 warps): 0-3 epilogue (TMEM lanes = this CTA's 128
// features, columns = rows), 4 TMA producer (weights; non-gathered
// activations), 5 MMA warp on the even CTA (warp-uniform waits, one elected
// lane issues) / relay on the odd CTA, 6-13 gather producers (x or dY rows
// picked by the permutation table; in the flavours fed by TMA alone, warps
// 6-8 are three more TMA producers, K blocks dealt round-robin), 14 unit
// scheduler (even CTA).
//   * Producers of both CTAs fill their own stage.  Both CTAs' TMA loads
//     complete the even CTA's full[s] directly (.cta_group::2), armed there
//     with both halves' bytes.  Where a flavour gathers rows (cp.async, L1
//     fwd and L2 dgrad), each CTA's gather threads arrive on its own full[s]
//     and the odd CTA's relay thread forwards its half to the even CTA's
//     full[s], so the MMA thread waits on one barrier per stage (issuing a
//     tcgen05.mma costs the thread a good part of the MMA's pipe time, and
//     every extra wait in its loop shows up as idle tensor-pipe time).
//   * The even CTA waits for full[s], issues the four M=256
//     MMAs of the stage, and its commit arrives on empty[s] of both CTAs;
//     after a unit's last K block a commit arrives on tfull[acc] of both.
//   * Both CTAs' epilogue warps drain their own accumulator rows and arrive
//     on the even CTA's tempty[acc] (8 arrivals) before it is reused.
// Every wait is bounded; a timeout raises the CTA's abort flag and the
// status word, and both CTAs leave through the closing cluster barrier.
#pragma once

#include <atomic>

#include "gemm_common.cuh"

namespace moe {

constexpr int kT2Stages = 6;              // barrier slots (the L2 dgrad kernel uses 5 stages)
constexpr int kT2ABytes = 128 * kBK * 2;  // this CTA's 128 features x 64 of K
constexpr int kT2BBytes = 128 * kBK * 2;  // up to 128 routed rows x 64 of K
constexpr int kT2InBytes = 3 * 2048;      // L2 dgrad epilogue inputs per warp: h gate, h up, a boxes
constexpr int kUR = 4;                    // slots of the unit ring
constexpr int kT2NumBars = 2 * kT2Stages + 9 + 2 * kEpiWarps + 2 * kUR + 1 + 4;
constexpr int kT2TailBytes = 512;         // barriers, TMEM address, abort flag, unit ring
constexpr int kT2RingOff = (8 * kT2NumBars + 8 + 15) & ~15;
static_assert(kT2RingOff + 16 * kUR <= kT2TailBytes, "barrier area");
constexpr int kWarpSched = kWarpGather0 + kGatherWarps;  // unit scheduler (even CTA, lane 0)
constexpr int kT2Threads = kGemmThreads + 32;

struct T2Bars {
    uint32_t base;
    __device__ __forceinline__ uint32_t full(int s) const { return base + 8u * s; }
    __device__ __forceinline__ uint32_t empty(int s) const { return base + 8u * (kT2Stages + s); }
    __device__ __forceinline__ uint32_t tfull(int a) const { return base + 8u * (2 * kT2Stages + a); }
    __device__ __forceinline__ uint32_t tempty(int a) const { return base + 8u * (2 * kT2Stages + 2 + a); }
    __device__ __forceinline__ uint32_t drain() const { return base + 8u * (2 * kT2Stages + 4); }
    // L1 epilogue: up-projection values handed from warp 2 + i to warp i
    __device__ __forceinline__ uint32_t xfull(int i) const { return base + 8u * (2 * kT2Stages + 5 + i); }
    __device__ __forceinline__ uint32_t xempty(int i) const { return base + 8u * (2 * kT2Stages + 7 + i); }
    // L2 dgrad epilogue: the saved h and a boxes of epilogue warp w have landed
    __device__ __forceinline__ uint32_t ein(int w) const { return base + 8u * (2 * kT2Stages + 9 + w); }
    // unit ring: slot i published (both CTAs) / read by every consumer of
    // both CTAs (even CTA's barrier); the even CTA's TMA producer took a unit
    __device__ __forceinline__ uint32_t ufull(int i) const { return base + 8u * (2 * kT2Stages + 9 + kEpiWarps + i); }
    __device__ __forceinline__ uint32_t uempty(int i) const {
        return base + 8u * (2 * kT2Stages + 9 + kEpiWarps + kUR + i);
    }
    __device__ __forceinline__ uint32_t ustart() const { return base + 8u * (2 * kT2Stages + 9 + kEpiWarps + 2 * kUR); }
    // L2 dgrad epilogue: the input boxes of warp w's buffer b have landed
    __device__ __forceinline__ uint32_t ein(int w, uint32_t b) const {
        return b == 0 ? ein(w) : base + 8u * (2 * kT2Stages + 9 + kEpiWarps + 2 * kUR + 1 + w);
    }
    // FP8 L1 epilogue: gate values handed from warp i to warp 2 + i
    __device__ __forceinline__ uint32_t gfull(int i) const {
        return base + 8u * (2 * kT2Stages + 9 + 2 * kEpiWarps + 2 * kUR + 1 + i);
    }
    __device__ __forceinline__ uint32_t gempty(int i) const {
        return base + 8u * (2 * kT2Stages + 9 + 2 * kEpiWarps + 2 * kUR + 3 + i);
    }
};

// ------------------------------------------------------- cluster helpers
__device__ __forceinline__ uint32_t cluster_addr_of(uint32_t local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// Arrival that makes this thread's earlier shared::cluster stores visible to
// whoever observes the phase with acquire.cluster.
__device__ __forceinline__ void mbar_arrive_release_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// TMA loads into this CTA's shared memory whose completion is counted on the
// mbarrier at `bar_cluster` (a shared::cluster address that may lie in the
// peer CTA of the pair: .cta_group::2), so that both CTAs' halves of a stage
// complete one barrier of the MMA-issuing CTA.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* m, int c0, int c1,
                                                 uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(bar_cluster)
        : "memory");
}
__device__ __forceinline__ void tma_load_2d_pair_hint(uint32_t dst, const CUtensorMap* m, int c0, int c1,
                                                      uint32_t bar_cluster, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(bar_cluster), "l"(pol)
        : "memory");
}
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* m, int c0, int c1, int c2,
                                                 uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(bar_cluster)
        : "memory");
}
__device__ __forceinline__ void tma_load_4d_pair(uint32_t dst, const CUtensorMap* m, int c0, int c1, int c2, int c3,
                                                 uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar_cluster)
        : "memory");
}
__device__ __forceinline__ void st_cluster_v4(uint32_t cluster_addr, int4 v) {
    asm volatile("st.shared::cluster.v4.s32 [%0], {%1, %2, %3, %4};" ::"r"(cluster_addr), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}
__device__ __forceinline__ int4 ld_shared_v4s(uint32_t addr) {
    int4 v;
    asm volatile("ld.shared.v4.s32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
                 : "memory");
    return v;
}
__device__ __forceinline__ bool mbar_try_wait_acq_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait on a barrier that receives arrivals from the other CTA.
__device__ __forceinline__ bool mbar_wait_cl(uint32_t bar, uint32_t parity, volatile int* abort) {
    if (mbar_try_wait_acq_cluster(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait_acq_cluster(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (*abort) return false;
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                *abort = 1;
                return false;
            }
        }
    }
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_mma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                 uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrives on the mbarrier at offset `bar` of both CTAs of the pair once
// every MMA issued so far by this thread is complete.
__device__ __forceinline__ void tc_commit_pair(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
        "h"((uint16_t)0x3)
        : "memory");
}
__device__ __forceinline__ void tc_commit_pair_local(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// ---------------------------------------------- block-scaled FP8 (MX) MMA
// D[tmem] (+)= sum over one 32-deep K step of (A 2^sa) (B 2^sb): E4M3 A and
// B, one UE8M0 scale per operand row and K step, FP32 accumulation
// (kind::mxf8f6f4, block_scale, one scale per 32 elements).  The scales are
// read from TMEM at sfa / sfb; the instruction descriptor picks the byte of
// each lane's word (the K step).
__device__ __forceinline__ void tc_mma_mx_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                               uint32_t sfa, uint32_t sfb, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
        : "memory");
}
// Copies 32 rows x 16 bytes of shared memory (described by sdesc) into TMEM
// columns [taddr, taddr + 4) of each of the four 32-lane quadrants (row i to
// lane 32 q + i), in both CTAs of the pair from their own shared memory.
// Ordered before the MMAs the same thread issues after it.
__device__ __forceinline__ void tc_cp_rows16_x4_pair(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
// Shared-memory descriptor of 32 rows x 16 bytes, no swizzle (8-row core
// matrices 128 bytes apart).
__device__ __forceinline__ uint64_t make_sdesc_rows16(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(1) << 16;             // leading byte offset 16 (one column of 16 bytes)
    d |= static_cast<uint64_t>(128 >> 4) << 32;      // stride byte offset 128
    d |= static_cast<uint64_t>(1) << 46;             // version 1, no swizzle
    return d;
}
// Instruction descriptor for kind::mxf8f6f4 with E4M3 A and B (K-major), UE8M0
// scales, scale byte `sf` (the K step) of both A's and B's scale words.
__host__ __device__ constexpr uint32_t make_idesc_mx_e4m3(int M, int N, int sf) {
    return ((uint32_t)sf << 4)                       // B scale byte
           | (static_cast<uint32_t>(N >> 3) << 17)   // N / 8
           | (1u << 23)                              // scale type: UE8M0
           | (static_cast<uint32_t>(M >> 4) << 24)   // M / 16
           | ((uint32_t)sf << 29);                   // A scale byte
}

// Column l of a 32-row x 32-column bf16 box in the 64-byte swizzle (row j
// at byte 64 j, its 16-byte chunk q stored at chunk q ^ ((j / 2) % 4)):
// v[j] is the value of row j.
__device__ __forceinline__ void stage_col_sw64(uint32_t box, int l, const float (&v)[32]) {
    const uint32_t within = (uint32_t)(l & 7) << 1;
    const int q = l >> 3;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const __nv_bfloat16 b = __float2bfloat16_rn(v[j]);
        const uint16_t u = *reinterpret_cast<const uint16_t*>(&b);
        asm volatile("st.shared.u16 [%0], %1;" ::"r"(box + j * 64 + ((uint32_t)(q ^ ((j >> 1) & 3)) << 4) + within),
                     "h"(u)
                     : "memory");
    }
}

// Rows j0..j0+15 of column l of the same box.
__device__ __forceinline__ void stage_col16_sw64(uint32_t box, int l, int j0, const float (&v)[16]) {
    const uint32_t within = (uint32_t)(l & 7) << 1;
    const int q = l >> 3;
#pragma unroll
    for (int jj = 0; jj < 16; ++jj) {
        const int j = j0 + jj;
        const __nv_bfloat16 b = __float2bfloat16_rn(v[jj]);
        const uint16_t u = *reinterpret_cast<const uint16_t*>(&b);
        asm volatile("st.shared.u16 [%0], %1;" ::"r"(box + j * 64 + ((uint32_t)(q ^ ((j >> 1) & 3)) << 4) + within),
                     "h"(u)
                     : "memory");
    }
}

// SwiGLU activation clamp (c = INFINITY: none): the input clamped to
// [-c, c], and whether its gradient passes (-c <= z <= c).
__device__ __forceinline__ float clamp_in(float z, float c) { return c < INFINITY ? fminf(fmaxf(z, -c), c) : z; }
__device__ __forceinline__ float clamp_pass(float z, float c) {
    return (c == INFINITY || (z >= -c && z <= c)) ? 1.0f : 0.0f;
}

__device__ __forceinline__ float ldg_bf16(const __nv_bfloat16* p) {
    const uint16_t u = __ldg(reinterpret_cast<const unsigned short*>(p));
    return __uint_as_float((uint32_t)u << 16);
}

// ------------------------------------------------------------ work units
template <int F>
struct T2;
template <>
struct T2<L1_FWD> {
    static constexpr bool kGather = true, kAMN = true;
    static constexpr int kFeatPerCta = 64;  // 64 gate + 64 up features
    static constexpr int kStages = 6;
    static constexpr int kProducers = 1;  // TMA producer threads (one TMA issue stream each)
    static constexpr int kEpiHalves = 1;  // epilogue warps per TMEM lane quadrant
    static constexpr int kInBytes = 0;
};
// FP8 forward: the same GEMM on E4M3 weights (pre-quantized, K-major,
// [E][2][I][H]) and gathered E4M3 rows, each with one UE8M0 scale per 32
// elements of K, by the block-scaled tcgen05.mma (kind::mxf8f6f4).  A stage
// is 128 deep in K (128 bytes per row, like a 64-deep bf16 stage).  Its
// scales sit in 512-byte atoms of 128 operand rows x 4 K steps (row r, step
// j at byte 16 (r % 32) + 4 (r / 32) + j, the order in which TMEM holds
// them: lane r % 32 of every 32-lane quadrant, column r / 32, byte j): one
// atom for this CTA's weights (by TMA, stored in that layout) and two for
// the unit's up to 256 rows (gathered; both CTAs hold all of them, since
// each CTA's half of the MMA reads the B scales of every column from its
// own TMEM), copied into TMEM by the MMA thread before the stage's four
// MMAs.
template <>
struct T2<L1_FWD_MX> : T2<L1_FWD> {
    static constexpr bool kAMN = false;
    static constexpr int kStages = 5;
    static constexpr int kSfBytes = 512 + 1024;  // per stage: the weights' atom, the rows' two atoms
    static constexpr int kInBytes = kStages * kSfBytes;
};
template <int F>
__host__ __device__ constexpr bool t2_is_l1() {
    return F == L1_FWD || F == L1_FWD_MX;
}
// the block-scaled FP8 flavours
template <int F>
__host__ __device__ constexpr bool t2_is_mx() {
    return F == L1_FWD_MX || F == L2_FWD_MX;
}
// flavours whose B rows come by TMA and their scales by one warp's cp.async
template <int F>
__host__ __device__ constexpr bool t2_sf_rows() {
    return F == L2_FWD_MX;
}
// K per stage: 64 bf16 or 128 E4M3 elements (128 bytes per operand row)
template <int F>
__host__ __device__ constexpr int t2_kblock() {
    return t2_is_mx<F>() ? 128 : kBK;
}
// TMEM of the FP8 flavour: accumulator 0 at column 0 (up to 256 columns),
// accumulator 1 at column 256 (up to 224: a unit of more rows always takes
// accumulator 0), and two slots of scale factors, the rows' two atoms at
// columns 480 + 8 s, the weights' atom at 496 + 4 s.
constexpr uint32_t kMxAcc1MaxN = 224, kMxSfb = 480, kMxSfa = 496;
// Accumulator of each unit in turn (the MMA warp and the epilogue warps walk
// the same units): the other one than the previous unit's when the unit
// fits accumulator 1, so that the epilogue of one overlaps the next one's
// MMAs; the phase of an accumulator counts its own uses.
struct MxAcc {
    int prev = 1;
    uint32_t uses[2] = {0u, 0u};
    __device__ __forceinline__ int pick(int n, uint32_t* phase) {
        const int a = n > (int)kMxAcc1MaxN ? 0 : prev ^ 1;
        prev = a;
        *phase = uses[a]++ & 1u;
        return a;
    }
};

template <>
struct T2<L2_FWD> {
    static constexpr bool kGather = false, kAMN = true;
    static constexpr int kFeatPerCta = 128;
    static constexpr int kStages = 6;
    static constexpr int kProducers = 4;  // TMA producer threads (one TMA issue stream each)
    // its units are short (K = I): a second set of epilogue warps (free
    // gather warps) takes every other 32-row chunk
    static constexpr int kEpiHalves = 2;
    static constexpr int kInBytes = 0;
};
// FP8 L2 forward: E4M3 W2 (pre-quantized, K-major [E][H][I], its scale
// atoms [E][H / 128][I / 128]) and the E4M3 rows of a with one UE8M0 scale
// per 32 features (written by the FP8 L1's epilogue), by the block-scaled
// MMA, 128 deep per stage like the FP8 L1.  The weights and their atom come
// by TMA, this CTA's rows of a by TMA, and the 4 scale bytes per row and
// stage of every row of the unit (both CTAs' MMA columns) by one warp's
// cp.async into the rows' two atoms; the odd CTA's relay forwards that
// warp's arrival as in the gathering flavours.
template <>
struct T2<L2_FWD_MX> : T2<L2_FWD> {
    static constexpr bool kAMN = false;
    static constexpr int kStages = 5;
    static constexpr int kSfBytes = 512 + 1024;  // per stage: the weights' atom, the rows' two atoms
    static constexpr int kInBytes = kStages * kSfBytes;
};
template <>
struct T2<L2_DGRAD> {
    static constexpr bool kGather = true, kAMN = false;
    static constexpr int kFeatPerCta = 128;
    static constexpr int kStages = 5;
    static constexpr int kProducers = 1;  // TMA producer threads (one TMA issue stream each)
    static constexpr int kEpiHalves = 1;  // epilogue warps per TMEM lane quadrant
    static constexpr int kInBytes = kEpiWarps * kT2InBytes;
};
template <>
struct T2<L1_DGRAD> {
    static constexpr bool kGather = false, kAMN = false;
    static constexpr int kFeatPerCta = 128;
    static constexpr int kStages = 6;
    static constexpr int kProducers = 4;  // TMA producer threads (one TMA issue stream each)
    static constexpr int kEpiHalves = 1;
    static constexpr int kInBytes = 0;
};

template <int F>
constexpr int t2_smem_bytes() {
    return 1024 + T2<F>::kStages * (kT2ABytes + kT2BBytes) + kEpiWarps * kStageEpiBytes + T2<F>::kInBytes +
           kT2TailBytes;
}
static_assert(t2_smem_bytes<L1_FWD>() <= 232448 && t2_smem_bytes<L2_DGRAD>() <= 232448 &&
                  t2_smem_bytes<L1_FWD_MX>() <= 232448 && t2_smem_bytes<L2_FWD_MX>() <= 232448,
              "shared memory per CTA");
// the warp of a t2_sf_rows flavour that copies the rows' scales: the first
// gather warp after its extra producers and second epilogue warps
template <int F>
__host__ __device__ constexpr int t2_sf_rows_warp() {
    return kWarpGather0 + T2<F>::kProducers - 1 + kEpiWarps * (T2<F>::kEpiHalves - 1);
}
static_assert(t2_sf_rows_warp<L2_FWD_MX>() < kWarpGather0 + kGatherWarps, "free gather warp for the rows' scales");
static_assert(T2<L2_FWD>::kProducers - 1 + kEpiWarps * (T2<L2_FWD>::kEpiHalves - 1) <= kGatherWarps &&
                  T2<L1_DGRAD>::kEpiHalves == 1 && T2<L1_FWD>::kEpiHalves == 1 && T2<L2_DGRAD>::kEpiHalves == 1,
              "free gather warps");
// A producer waits on the empty barrier of its block's stage by parity; the
// wait is unambiguous only if that barrier is at most one phase behind, which
// the producer's own previous block (kProducers earlier) guarantees only
// when kProducers <= kStages.
template <int F>
constexpr bool t2_producers_ok() {
    return T2<F>::kProducers <= T2<F>::kStages;
}
static_assert(t2_producers_ok<L1_FWD>() && t2_producers_ok<L2_FWD>() && t2_producers_ok<L2_DGRAD>() &&
                  t2_producers_ok<L1_DGRAD>() && t2_producers_ok<L1_FWD_MX>() && t2_producers_ok<L2_FWD_MX>(),
              "round-robin producers within the ring depth");
static_assert(T2<L1_FWD>::kProducers == 1 && T2<L2_DGRAD>::kProducers == 1 && T2<L2_FWD>::kProducers <= 1 + kGatherWarps &&
                  T2<L1_DGRAD>::kProducers <= 1 + kGatherWarps,
              "producer warps");

// Element (row j, column l) of a 32-row x 32-column bf16 box in the 64-byte swizzle.
__device__ __forceinline__ float lds_sw64(uint32_t box, int j, int l) {
    uint16_t u;
    asm volatile("ld.shared.u16 %0, [%1];"
                 : "=h"(u)
                 : "r"(box + j * 64 + ((uint32_t)((l >> 3) ^ ((j >> 1) & 3)) << 4) + ((uint32_t)(l & 7) << 1))
                 : "memory");
    return __uint_as_float((uint32_t)u << 16);
}
// Stores v as element (row j, column l) of the same kind of box.
__device__ __forceinline__ void sts_sw64(uint32_t box, int j, int l, float v) {
    const __nv_bfloat16 b = __float2bfloat16_rn(v);
    const uint16_t u = *reinterpret_cast<const uint16_t*>(&b);
    asm volatile("st.shared.u16 [%0], %1;" ::"r"(box + j * 64 + ((uint32_t)((l >> 3) ^ ((j >> 1) & 3)) << 4) +
                                               ((uint32_t)(l & 7) << 1)),
                 "h"(u)
                 : "memory");
}

// One step of a warp-wide transposed reduction of 32 values per lane: after
// the steps for S = 16, 8, 4, 2, 1, lane j holds the sum over all lanes of
// their value j.  At step S a lane keeps the half of its S * 2 live values
// selected by bit S of its lane id and adds the partner's copy of that half.
template <int S>
__device__ __forceinline__ void transpose_reduce_step(float (&v)[32], int lane) {
    const bool upper = (lane & S) != 0;
#pragma unroll
    for (int i = 0; i < S; ++i) {
        const float send = upper ? v[i] : v[i + S];
        const float keep = upper ? v[i + S] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, S);
    }
}

// SwiGLU^T of one 32-row chunk of the L2 dgrad epilogue, element (row j,
// feature lane): from g = v[j], the saved h (gate, up) and a boxes in
// shared memory and the routing weight w (lane j of wl), stage
//   da = w g,  dgate = da * up * s(gate) * (1 + gate (1 - s(gate))),
//   dup = da * silu(gate),  aw = w a
// into the three output boxes.  kClamp: gate and up clamped to [-c, c] and
// the gradients masked by the forward's decisions (bit lane of row j's
// gmask / umask word, lane j holding row j's words).  s(z) = 1 / (1 + e^-z)
// with the hardware exponential and the fast divide (within 2 ulp, and 0
// once e^-z overflows, which is the limit): with a full-precision divide
// this arithmetic outlasted the MMAs of a unit when K is short.
template <bool kClamp>
__device__ __forceinline__ void swiglu_t_chunk(uint32_t stage, uint32_t in_box, bool colok, int lane, float wl,
                                               const float (&v)[32], float c, uint32_t gmask, uint32_t umask) {
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        float hg = 0.0f, hu = 0.0f, av = 0.0f;
        if (colok) {
            hg = lds_sw64(in_box, j, lane);
            hu = lds_sw64(in_box + 2048, j, lane);
            av = lds_sw64(in_box + 4096, j, lane);
        }
        const float wv = __shfl_sync(0xffffffffu, wl, j);
        const float da = wv * v[j];
        float gc = hg, uc = hu, pg = 1.0f, pu = 1.0f;
        if constexpr (kClamp) {
            gc = fminf(fmaxf(hg, -c), c);
            uc = fminf(fmaxf(hu, -c), c);
            pg = (float)((__shfl_sync(0xffffffffu, gmask, j) >> lane) & 1u);
            pu = (float)((__shfl_sync(0xffffffffu, umask, j) >> lane) & 1u);
        }
        const float sg = __fdividef(1.0f, 1.0f + __expf(-gc));
        sts_sw64(stage, j, lane, da * uc * sg * (1.0f + gc * (1.0f - sg)) * pg);
        sts_sw64(stage + 2048, j, lane, da * gc * sg * pu);
        sts_sw64(stage + 4096, j, lane, wv * av);
    }
}

struct T2Unit {
    int e;       // expert
    int f0;      // first feature of this CTA (L1: of its 64 gate and 64 up features)
    int fcol;    // this CTA's feature tile (of kFeatPerCta features)
    int r0;      // first routed row of the unit (index into perm and the row-ordered buffers)
    int n;       // rows of the unit rounded up to 32: the MMA's N
    int nvalid;  // routed rows of the unit
};
// ------------------------------------------------------------ unit feed
// Units are handed out at run time, so that the clusters that stream the
// same weight tile (the row chunks of one expert and feature tile, numbered
// next to each other) start them at nearly the same moment and share the
// tile in L2; a static stride lets the clusters drift apart over a launch.
// Cluster c starts with unit c; the even CTA's scheduler thread claims each
// further unit from a global counter (ncl + atomicAdd) as soon as the even
// CTA's TMA producer has started the cluster's previous unit, decodes it from
// the routing tables and publishes it in a kUR-slot ring in the shared
// memory of both CTAs (ufull[i]); every consumer of both CTAs reads the slot
// and arrives on the even CTA's uempty[i].  An expert of -1 ends the walk.
// Slot: {expert, feature tile, first row, n << 16 | routed rows}.
__device__ __forceinline__ int4 t2_decode(const GemmArgs& p, int u) {
    const int e = __ldg(p.pair_owner + u / p.n_tiles);
    const int po = __ldg(p.pair_offs + e);
    const int off = __ldg(p.offs + e);
    const int cnt = __ldg(p.counts + e);
    const int nsub = ((cnt + kBM - 1) / kBM + 1) / 2;  // the prologue's tile pairs of e
    const int l = u - po * p.n_tiles;
    const int ft = l / nsub;
    const int j = l - ft * nsub;
    const int nb = (((cnt + nsub - 1) / nsub) + 31) & ~31;
    const int rs = j * nb;
    const int nvalid = min(nb, cnt - rs);
    const int n = (nvalid + 31) & ~31;
    return make_int4(e, ft, off + rs, (n << 16) | nvalid);
}

template <int F>
struct T2Feed {
    uint32_t ring;  // this CTA's ring slots
    T2Bars bars;
    int rank;
    int n;  // units taken so far
    __device__ __forceinline__ T2Feed(uint32_t ring_, T2Bars bars_, int rank_)
        : ring(ring_), bars(bars_), rank(rank_), n(0) {}
    // Takes the next unit into t; false at the end of the walk or on abort.
    // kWarp: every lane of the warp calls (warp-collective wait), otherwise
    // one thread.  start: the even CTA's TMA producer, whose take lets the
    // scheduler claim the cluster's next unit.
    template <bool kWarp>
    __device__ __forceinline__ bool next(T2Unit& t, volatile int* abort, int lane, bool start = false) {
        const int i = n % kUR;
        const uint32_t ph = (uint32_t)(n / kUR) & 1u;
        bool ok;
        if constexpr (kWarp) {
            ok = rank == 0 ? warp_wait_uniform<false>(bars.ufull(i), ph, abort)
                           : warp_wait_uniform<true>(bars.ufull(i), ph, abort);
        } else {
            ok = rank == 0 ? mbar_wait(bars.ufull(i), ph, abort) : mbar_wait_cl(bars.ufull(i), ph, abort);
        }
        if (!ok) return false;
        const int4 v = ld_shared_v4s(ring + 16u * (uint32_t)i);
        if constexpr (kWarp) __syncwarp();
        if (!kWarp || lane == 0) {
            if (rank == 0)
                mbar_arrive(bars.uempty(i));
            else
                mbar_arrive_release_cluster(cluster_addr_of(bars.uempty(i), 0));
            if (start) mbar_arrive(bars.ustart());
        }
        ++n;
        if (v.x < 0) return false;
        t.e = v.x;
        t.fcol = 2 * v.y + rank;
        t.f0 = t.fcol * T2<F>::kFeatPerCta;
        t.r0 = v.z;
        t.n = v.w >> 16;
        t.nvalid = v.w & 0xffff;
        return true;
    }
};

__device__ __forceinline__ int t2_total_units(const GemmArgs& p) {
    int np = *reinterpret_cast<const volatile int32_t*>(p.status + MOE_STATUS_NUM_PAIRS);
    np = np < 0 ? 0 : (np > p.tiles_cap ? p.tiles_cap : np);
    return np * p.n_tiles;
}

// The pair of status words (work counter, clusters done) of a flavour's unit
// feed: words MOE_STATUS_SCHED + 2 slot, + 1 of the eight the prologue
// zeroes.  The FP8 L1 shares the bf16 L1's pair (the two are never in flight
// on one route_ws at once, like any two calls on it).
template <int F>
__host__ __device__ constexpr int t2_sched_slot() {
    return F == L1_FWD_MX ? (int)L1_FWD : (F == L2_FWD_MX ? (int)L2_FWD : F);
}
static_assert(t2_sched_slot<L1_FWD>() < 4 && t2_sched_slot<L2_FWD>() < 4 && t2_sched_slot<L2_DGRAD>() < 4 &&
                  t2_sched_slot<L1_DGRAD>() < 4 && t2_sched_slot<L1_FWD_MX>() < 4 && t2_sched_slot<L2_FWD_MX>() < 4 &&
                  MOE_STATUS_SCHED + 2 * 4 <= MOE_STATUS_WORDS,
              "unit-feed counters inside the status words the prologue zeroes");

// Claims are served from both ends of the walk in turn: claim 2i takes unit
// i (the heaviest experts first), claim 2i + 1 unit total - 1 - i (the
// lightest first), so that with uneven routing the units in flight at any
// moment mix experts whose weight tiles are re-read from L2 by many row
// chunks (tensor- and gather-bound) with experts of a few rows, whose
// units stream their weights from DRAM.  Measured against the experts
// walked by id from one end, skewed routing (V3 shape, top expert 5636
// rows): L1 fwd 3.44 -> 3.28 ms, L2 fwd 1.75 -> 1.58, L1 dgrad 3.43 ->
// 3.12, the step 17.6 -> 17.0 ms; V3-shaped routing (experts of 208-308
// rows): L2 dgrad 1.78 -> 1.81 ms, the rest within noise.
__device__ __forceinline__ int t2_claimed_unit(int c, int total) {
    return (c & 1) ? total - 1 - (c >> 1) : (c >> 1);
}

// The even CTA's unit scheduler (one thread).  The work counter and the
// count of clusters done are status words of route_ws (zeroed by the routing
// prologue); the last cluster to finish puts both back to zero for the next
// launch on the same tables.
template <int F>
__device__ void t2_role_sched(const GemmArgs& p, uint32_t ring, T2Bars bars, volatile int* abort) {
    const int total = t2_total_units(p);
    const int ncl = (int)gridDim.x >> 1;
    int* ctr = reinterpret_cast<int*>(p.status + MOE_STATUS_SCHED + 2 * t2_sched_slot<F>());
    int* fin = ctr + 1;
    const uint32_t ring1 = cluster_addr_of(ring, 1);
    int c = (int)blockIdx.x >> 1;  // claim number
    for (int n = 0;; ++n) {
        if (n > 0) {
            if (!mbar_wait(bars.ustart(), (uint32_t)(n - 1) & 1u, abort)) break;
            c = ncl + atomicAdd(ctr, 1);
        }
        const int4 v = c < total ? t2_decode(p, t2_claimed_unit(c, total)) : make_int4(-1, 0, 0, 0);
        const int i = n % kUR;
        if (!mbar_wait_cl(bars.uempty(i), ((uint32_t)(n / kUR) & 1u) ^ 1u, abort)) break;
        st_shared_v4(ring + 16u * (uint32_t)i, (uint32_t)v.x, (uint32_t)v.y, (uint32_t)v.z, (uint32_t)v.w);
        st_cluster_v4(ring1 + 16u * (uint32_t)i, v);
        mbar_arrive(bars.ufull(i));
        mbar_arrive_release_cluster(cluster_addr_of(bars.ufull(i), 1));
        if (v.x < 0) break;
    }
    __threadfence();
    if (atomicAdd(fin, 1) == ncl - 1) {
        atomicExch(ctr, 0);
        atomicExch(fin, 0);
    }
}

// ------------------------------------------------------------ TMA producer
// The K blocks are dealt round-robin to kProducers threads in different warps
// (block g to thread g % kProducers): one thread's bulk tensor copies are
// processed one after the other, at about 30 bytes per cycle for these boxes
// on this GPU, whatever the number in flight, while copies from separate
// threads proceed side by side.
template <int F>
__device__ void t2_role_tma(const CUtensorMap* mA, const CUtensorMap* mB, const CUtensorMap* mD, const GemmArgs& p,
                            uint32_t ring, uint32_t sA, uint32_t sB, uint32_t sIn, T2Bars bars, volatile int* abort,
                            int rank, int pid) {
    constexpr int NP = T2<F>::kProducers;
    const int nkb = p.K / t2_kblock<F>();
    int stage = 0;
    uint32_t phase = 0;
    uint32_t g = 0;
    T2Feed<F> feed(ring, bars, rank);
    for (T2Unit t; feed.template next<false>(t, abort, 0, rank == 0 && pid == 0);) {
        const int nh = t.n >> 1;           // this CTA's rows of the unit
        const int nbox = (nh + 31) >> 5;   // 32-row boxes of a non-gathered B
        const int rb = t.r0 + nh * rank;
        const uint32_t tx = (uint32_t)kT2ABytes + (T2<F>::kGather ? 0u : (uint32_t)nbox * 4096u) +
                            (t2_is_mx<F>() ? 512u : 0u);
        for (int kb = 0; kb < nkb; ++kb, ++g) {
            if (NP > 1 && (int)(g % (uint32_t)NP) != pid) {
                if (++stage == T2<F>::kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
                continue;
            }
            if (!mbar_wait(bars.empty(stage), phase ^ 1u, abort)) return;
            const uint32_t a = sA + stage * kT2ABytes;
            const uint32_t b = sB + stage * kT2BBytes;
            const int k0 = kb * t2_kblock<F>();
            // both CTAs' TMA loads complete the even CTA's full barrier, armed
            // there with both halves' bytes
            if (rank == 0) mbar_arrive_expect_tx(bars.full(stage), 2u * tx);
            const uint32_t fb = cluster_addr_of(bars.full(stage), 0);
            if constexpr (F == L1_FWD_MX) {
                // E4M3 W1 viewed as [E][2][I][H] (K-major): the 64 gate rows,
                // then the same 64 up rows, 128 bytes of K each; then their
                // scale atom, atoms stored [E][I / 64][H / 128] (512 bytes,
                // two 256-byte rows of the atoms' tensor map)
                tma_load_4d_pair(a, mA, k0, t.f0, 0, t.e, fb);
                tma_load_4d_pair(a + 8192, mA, k0, t.f0, 1, t.e, fb);
                const int atom = (t.e * (p.I / 64) + t.fcol) * nkb + kb;
                tma_load_2d_pair(sIn + (uint32_t)stage * (uint32_t)T2<F>::kSfBytes, mB, 0, 2 * atom, fb);
            } else if constexpr (F == L2_FWD_MX) {
                // E4M3 W2 viewed as [E][H][I] (K-major): this CTA's 128 rows
                // of H, 128 bytes of K each; their scale atom ([E][H / 128]
                // [I / 128], two 256-byte rows of the atoms' tensor map);
                // this CTA's rows of a (E4M3, 128 bytes of K per row)
                tma_load_3d_pair(a, mA, k0, t.f0, t.e, fb);
                const int atom = (t.e * (p.H / 128) + t.fcol) * nkb + kb;
                tma_load_2d_pair(sIn + (uint32_t)stage * (uint32_t)T2<F>::kSfBytes, mD, 0, 2 * atom, fb);
                for (int i = 0; i < nbox; ++i) tma_load_2d_pair(b + i * 4096, mB, k0, rb + 32 * i, fb);
            } else if constexpr (t2_is_l1<F>()) {
                // W1 viewed as [E][H][2][I]: 64 gate columns, then the same 64 up columns
                tma_load_4d_pair(a, mA, t.f0, 0, k0, t.e, fb);
                tma_load_4d_pair(a + 8192, mA, t.f0, 1, k0, t.e, fb);
            } else if constexpr (F == L2_DGRAD) {
                tma_load_3d_pair(a, mA, k0, t.f0, t.e, fb);
            } else {
                if constexpr (F == L2_FWD) {
                    tma_load_3d_pair(a, mA, t.f0, k0, t.e, fb);
                    tma_load_3d_pair(a + 8192, mA, t.f0 + 64, k0, t.e, fb);
                } else {  // L1_DGRAD
                    tma_load_3d_pair(a, mA, k0, t.f0, t.e, fb);
                }
                for (int i = 0; i < nbox; ++i) tma_load_2d_pair(b + i * 4096, mB, k0, rb + 32 * i, fb);
            }
            if (++stage == T2<F>::kStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
}

// ------------------------------------------------------- gather producers
// This CTA's rows of the unit, 16 per warp, 16-byte cp.async chunks into the
// 128-byte-swizzled K-major layout; rows past the unit's half are left alone
// (the MMA reads only n / 2 rows).  Padding rows (perm = -1) are zero-filled.
template <int F>
__device__ void t2_role_gather(const GemmArgs& p, uint32_t ring, uint32_t sB, uint32_t stg, T2Bars bars,
                               volatile int* abort, int gw, int lane, int rank) {
    const int c = lane & 7;
    const int rb = lane >> 3;
    const int H = p.H;
    const int k = p.k;
    const int nkb = p.K / t2_kblock<F>();
    const __nv_bfloat16* src = p.gsrc;
    int stage = 0;
    uint32_t phase = 0;
    T2Feed<F> feed(ring, bars, rank);
    for (T2Unit t; feed.template next<true>(t, abort, lane);) {
        const int nh = t.n >> 1;
        const int rbase = t.r0 + nh * rank;
        int tok[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int r = gw * 16 + rb + 4 * q;
            int s = -1;
            if (r < nh) s = __ldg(p.perm + rbase + r);
            tok[q] = r < nh ? (s >= 0 ? s / k : -1) : -2;  // -2: row not in this unit
        }
        if constexpr (F == L1_FWD_MX) {
            // This CTA's rows as E4M3 bytes (128 per row and K block, the same
            // 16-byte chunks as a bf16 block), and the 4 scale bytes of the
            // block of one unit row per thread (every row of the unit: both
            // CTAs' MMA columns) into the rows' atoms: unit row u at byte
            // 512 (u / 128) + 16 (u % 32) + 4 ((u % 128) / 32) of them.
            const int G = H >> 5;  // scale bytes per row of x_sf
            const int us = gw * 32 + lane;
            int stok = -2;  // -2: past the unit's N, not read by the MMA
            if (us < t.n) {
                const int sl = __ldg(p.perm + t.r0 + us);
                stok = sl >= 0 ? sl / k : -1;
            }
            const uint32_t soff =
                512u + (uint32_t)(us >> 7) * 512u + (uint32_t)(us & 31) * 16u + (uint32_t)((us >> 5) & 3) * 4u;
            for (int kb = 0; kb < nkb; ++kb) {
                if (!warp_wait(bars.empty(stage), phase ^ 1u, abort)) return;
                const uint32_t b = sB + stage * kT2BBytes;
                const int colb = kb * 128 + c * 16;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int tk = tok[q];
                    if (tk == -2) continue;
                    const int r = gw * 16 + rb + 4 * q;
                    const uint8_t* g = p.gsrc8 + (size_t)(tk < 0 ? 0 : tk) * (size_t)H + colb;
                    cp_async_16(b + r * 128 + ((c ^ (r & 7)) << 4), g, tk < 0 ? 0u : 16u);
                }
                if (stok != -2)
                    cp_async_4(stg + (uint32_t)stage * (uint32_t)T2<L1_FWD_MX>::kSfBytes + soff,
                               p.gsf + (size_t)(stok < 0 ? 0 : stok) * (size_t)G + (size_t)kb * 4, stok < 0 ? 0u : 4u);
                cp_async_arrive_noinc(bars.full(stage));
                if (++stage == T2<F>::kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        } else {
            for (int kb = 0; kb < nkb; ++kb) {
                if (!warp_wait(bars.empty(stage), phase ^ 1u, abort)) return;
                const uint32_t b = sB + stage * kT2BBytes;
                const int col = kb * kBK + c * 8;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int tk = tok[q];
                    if (tk == -2) continue;
                    const int r = gw * 16 + rb + 4 * q;
                    const __nv_bfloat16* g = src + (size_t)(tk < 0 ? 0 : tk) * (size_t)H + col;
                    cp_async_16(b + r * 128 + ((c ^ (r & 7)) << 4), g, tk < 0 ? 0u : 16u);
                }
                cp_async_arrive_noinc(bars.full(stage));
                if (++stage == T2<F>::kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
    }
}

// The rows' scales of a t2_sf_rows flavour (one warp in each CTA): for each
// 128-deep stage, the 4 scale bytes of every row of the unit (both CTAs'
// MMA columns, so both CTAs hold all of them) into the rows' two atoms:
// unit row u at byte 512 (u / 128) + 16 (u % 32) + 4 ((u % 128) / 32) past
// the weights' atom.  The lanes arrive on this CTA's full barrier when
// their copies land (the odd CTA's relay passes that on).
template <int F>
__device__ void t2_role_sf_rows(const GemmArgs& p, uint32_t ring, uint32_t sIn, T2Bars bars, volatile int* abort,
                                int lane, int rank) {
    const int nkb = p.K / t2_kblock<F>();
    const int G = p.K >> 5;  // scale bytes per row
    int stage = 0;
    uint32_t phase = 0;
    T2Feed<F> feed(ring, bars, rank);
    for (T2Unit t; feed.template next<true>(t, abort, lane);) {
        for (int kb = 0; kb < nkb; ++kb) {
            if (!warp_wait(bars.empty(stage), phase ^ 1u, abort)) return;
            const uint32_t sf = sIn + (uint32_t)stage * (uint32_t)T2<F>::kSfBytes + 512u;
            for (int us = lane; us < t.n; us += 32)
                cp_async_4(sf + (uint32_t)(us >> 7) * 512u + (uint32_t)(us & 31) * 16u + (uint32_t)((us >> 5) & 3) * 4u,
                           p.gsf + (size_t)(t.r0 + us) * (size_t)G + (size_t)kb * 4, 4u);
            cp_async_arrive_noinc(bars.full(stage));
            if (++stage == T2<F>::kStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
}

// -------------------------------------------- MMA issuer (even CTA) / relay
// The whole MMA warp runs this loop: it waits warp-uniformly and one elected
// lane issues the MMAs and their commits (see warp_wait_uniform).
template <int F>
__device__ void t2_role_mma(const GemmArgs& p, uint32_t ring, uint32_t sA, uint32_t sB, T2Bars bars,
                            uint32_t tmem_base, volatile int* abort, int lane) {
    const int nkb = p.K / t2_kblock<F>();
    int stage = 0;
    uint32_t phase = 0;
    int it = 0;
    T2Feed<F> feed(ring, bars, 0);
    for (T2Unit t; feed.template next<true>(t, abort, lane); ++it) {
        const int acc = it & 1;
        const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
        if (!warp_wait_uniform<true>(bars.tempty(acc), acc_phase ^ 1u, abort)) return;
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(acc * kBN);
        const uint32_t idesc = make_idesc_bf16(2 * kBM, t.n, T2<F>::kAMN, false);
        for (int kb = 0; kb < nkb; ++kb) {
            if (!warp_wait_uniform<true>(bars.full(stage), phase, abort)) return;
            tc_fence_after();
            const uint32_t a = sA + stage * kT2ABytes;
            const uint32_t b = sB + stage * kT2BBytes;
            if (elect_one()) {
                if constexpr (T2<F>::kGather) fence_proxy_async_smem();
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk) {
                    const uint64_t ad = T2<F>::kAMN ? make_sdesc_sw128(a + kk * 2048, 8192, 1024)
                                                    : make_sdesc_sw128(a + kk * 32, 16, 1024);
                    const uint64_t bd = make_sdesc_sw128(b + kk * 32, 16, 1024);
                    tc_mma_bf16_pair(d, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
                }
                tc_commit_pair(bars.empty(stage));
            }
            __syncwarp();
            if (++stage == T2<F>::kStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (elect_one()) tc_commit_pair(bars.tfull(acc));
        __syncwarp();
    }
}

// The MMA warp of the FP8 flavour: per stage, the elected lane copies the
// stage's three scale atoms into the next of the two TMEM scale slots and
// issues the four block-scaled MMAs of the 128-deep block (one per 32-deep
// K step, each reading byte kk of the scale words); a copy and the MMAs
// after it run in issue order, and the slot a copy overwrites was last read
// by MMAs issued before it.
template <int F>
__device__ void t2_role_mma_mx(const GemmArgs& p, uint32_t ring, uint32_t sA, uint32_t sB, uint32_t sIn, T2Bars bars,
                               uint32_t tmem_base, volatile int* abort, int lane) {
    const int nkb = p.K / t2_kblock<F>();
    int stage = 0;
    uint32_t phase = 0, nblk = 0;
    MxAcc accs;
    T2Feed<F> feed(ring, bars, 0);
    for (T2Unit t; feed.template next<true>(t, abort, lane);) {
        uint32_t acc_phase;
        const int acc = accs.pick(t.n, &acc_phase);
        if (!warp_wait_uniform<true>(bars.tempty(acc), acc_phase ^ 1u, abort)) return;
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(acc * kBN);
        for (int kb = 0; kb < nkb; ++kb, ++nblk) {
            if (!warp_wait_uniform<true>(bars.full(stage), phase, abort)) return;
            tc_fence_after();
            const uint32_t a = sA + stage * kT2ABytes;
            const uint32_t b = sB + stage * kT2BBytes;
            const uint32_t sf = sIn + (uint32_t)stage * (uint32_t)T2<F>::kSfBytes;
            const uint32_t tsfa = tmem_base + kMxSfa + 4u * (nblk & 1u);
            const uint32_t tsfb = tmem_base + kMxSfb + 8u * (nblk & 1u);
            if (elect_one()) {
                fence_proxy_async_smem();  // rows and row scales written by cp.async
                tc_cp_rows16_x4_pair(tsfa, make_sdesc_rows16(sf));
                tc_cp_rows16_x4_pair(tsfb, make_sdesc_rows16(sf + 512));
                tc_cp_rows16_x4_pair(tsfb + 4, make_sdesc_rows16(sf + 1024));
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t ad = make_sdesc_sw128(a + kk * 32, 16, 1024);
                    const uint64_t bd = make_sdesc_sw128(b + kk * 32, 16, 1024);
                    tc_mma_mx_pair(d, ad, bd, make_idesc_mx_e4m3(2 * kBM, t.n, kk), tsfa, tsfb,
                                   (kb | kk) != 0 ? 1u : 0u);
                }
                tc_commit_pair(bars.empty(stage));
            }
            __syncwarp();
            if (++stage == T2<F>::kStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (elect_one()) tc_commit_pair(bars.tfull(acc));
        __syncwarp();
    }
}

// The odd CTA's MMA thread: tells the even CTA that this CTA's half of a
// stage is in shared memory.
template <int F>
__device__ void t2_role_relay(const GemmArgs& p, uint32_t ring, T2Bars bars, volatile int* abort) {
    const int nkb = p.K / t2_kblock<F>();
    int stage = 0;
    uint32_t phase = 0;
    T2Feed<F> feed(ring, bars, 1);
    for (T2Unit t; feed.template next<false>(t, abort, 0);) {
        // flavours fed by TMA alone complete the even CTA's barrier directly;
        // the relay still takes every unit from the feed
        if constexpr (!T2<F>::kGather && !t2_sf_rows<F>()) continue;
        for (int kb = 0; kb < nkb; ++kb) {
            // this CTA's gathered rows of the stage have landed (its local
            // full barrier counts only the gather threads): make them visible
            // to the tensor core and arrive on the even CTA's full barrier
            if (!mbar_wait(bars.full(stage), phase, abort)) return;
            fence_proxy_async_smem();
            mbar_arrive_cluster(cluster_addr_of(bars.full(stage), 0));
            if (++stage == T2<F>::kStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
}

// fp8_group_exponent from the bits m of a finite, non-negative maximum:
// amax = 1.f 2^(E - 127) = r 2^p with p = E - 126 and r = 1.f / 2, and
// r <= 0.875 exactly when the fraction bits are at most 0x600000 (1.f <=
// 1.75), so e = E - 135 or E - 134; subnormal maxima clamp to -127.
__device__ __forceinline__ int fp8_group_exponent_bits(uint32_t m) {
    if (m == 0u) return 0;
    const int e = (int)(m >> 23) - 135 + ((m & 0x7fffffu) > 0x600000u ? 1 : 0);
    return e < -127 ? -127 : e;
}

// The FP8 L1's activations a of R (16 or 32) rows of one chunk (v[j] = a of
// row row0 + j at feature col + lane) as E4M3 rows with one UE8M0 scale per
// row and 32 features, the rule of the input's quantization: scale 2^e with
// the smallest e such that 448 2^e >= max |a| over the warp's 32 features
// (NaN left out of the maximum), codes rounded to nearest even and
// saturating (a times 2^-e is exact, as in ldexpf).  Lane l writes byte col
// + l of each row (32 consecutive bytes a row per warp) and lane j < R the
// scale byte of row row0 + j.
template <int R>
__device__ __forceinline__ void store_a_e4m3(const GemmArgs& p, const float (&v)[R], int row0, int col, int lane) {
    static_assert(R == 16 || R == 32, "16 or 32 rows");
    const int I = p.I;
    // the maximum of row j over the warp's features, kept by lane j (and
    // lane j + 16 when R = 16): a transposing reduction (at offset S the
    // lanes with bit S set keep rows i + S, the others rows i, each taking
    // the larger with its partner), R - 1 shuffles for the R rows (+ 1)
    uint32_t t[R];
#pragma unroll
    for (int j = 0; j < R; ++j) {
        const uint32_t b = __float_as_uint(fabsf(v[j]));
        t[j] = b > 0x7f800000u ? 0u : b;
    }
#pragma unroll
    for (int S = R / 2; S > 0; S >>= 1) {
        const bool upper = (lane & S) != 0;
#pragma unroll
        for (int i = 0; i < S; ++i) {
            const uint32_t send = upper ? t[i] : t[i + S];
            const uint32_t keep = upper ? t[i + S] : t[i];
            t[i] = max(keep, __shfl_xor_sync(0xffffffffu, send, S));
        }
    }
    uint32_t mine = t[0];
    if constexpr (R == 16) mine = max(mine, __shfl_xor_sync(0xffffffffu, mine, 16));
    // lane j: the exponent of row j; each row's 2^-e comes back by shuffle
    const int ex = fp8_group_exponent_bits(mine);
    const float inv = __uint_as_float((uint32_t)(127 - ex) << 23);
    uint8_t* q = p.q_out + (size_t)row0 * (size_t)I + (size_t)(col + lane);
#pragma unroll
    for (int j = 0; j < R; j += 2) {
        const float s0 = __shfl_sync(0xffffffffu, inv, j), s1 = __shfl_sync(0xffffffffu, inv, j + 1);
        const uint32_t two = __nv_cvt_float2_to_fp8x2(make_float2(v[j] * s0, v[j + 1] * s1), __NV_SATFINITE, __NV_E4M3);
        q[(size_t)j * (size_t)I] = (uint8_t)(two & 0xffu);
        q[(size_t)(j + 1) * (size_t)I] = (uint8_t)(two >> 8);
    }
    if (lane < R) p.sf_out[(size_t)(row0 + lane) * (size_t)(I >> 5) + (size_t)(col >> 5)] = (uint8_t)(ex + 127);
}

// ---------------------------------------------------------------- epilogue
// Warp w holds TMEM lanes 32w..32w+31 = 32 features of this CTA and every
// column (routed row) of the unit.  Each 32-row chunk is written as a
// 32-row x 32-feature box in the 64-byte swizzle and leaves by TMA store.
// The L2 dgrad epilogue also reads the saved h and a at its rows and
// features: a TMA load brings each 32 x 32 box into shared memory (mapH,
// mapA), the first one while the accumulator is still being computed.
template <int F>
__device__ void t2_role_epilogue(const GemmArgs& p, OutMaps om, const CUtensorMap* mapH, const CUtensorMap* mapAs,
                                 uint32_t ring, T2Bars bars, uint32_t tmem_base, uint32_t stage, uint32_t stage_of_warp0,
                                 uint32_t in_box, volatile int* abort, int warp, int lane, int rank, int half) {
    const uint32_t tempty_leader[2] = {cluster_addr_of(bars.tempty(0), 0), cluster_addr_of(bars.tempty(1), 0)};
    int it = 0;
    uint32_t nstore = 0;
    uint32_t xchunk = 0;  // L1: chunks handed over between warp i and warp 2 + i
    uint32_t nin = 0;     // L2 dgrad: input boxes waited for
    MxAcc accs;
    T2Feed<F> feed(ring, bars, rank);
    for (T2Unit t; feed.template next<true>(t, abort, lane); ++it) {
        int acc = it & 1;
        uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
        if constexpr (t2_is_mx<F>()) acc = accs.pick(t.n, &acc_phase);
        if constexpr (F == L2_DGRAD) {
            if (lane == 0 && t.f0 + 32 * warp < p.I) {
                // the unit's first chunk, into buffer nin & 1, whose last
                // stores (chunk nin - 2) must have read it
                bulk_wait_read<1>();
                const uint32_t cur = (nin & 1u) ? stage : in_box;
                const uint32_t eb = bars.ein(warp, nin & 1u);
                mbar_arrive_expect_tx(eb, (uint32_t)kT2InBytes);
                tma_load_2d(cur, mapH, t.f0 + 32 * warp, t.r0, eb);
                tma_load_2d(cur + 2048, mapH, p.I + t.f0 + 32 * warp, t.r0, eb);
                tma_load_2d(cur + 4096, mapAs, t.f0 + 32 * warp, t.r0, eb);
            }
        }
        if (!warp_wait(bars.tfull(acc), acc_phase, abort)) break;
        tc_fence_after();
        const uint32_t tacc = tmem_base + (uint32_t)(acc * kBN) + ((uint32_t)(warp * 32) << 16);
        bool ok = true;
#pragma unroll 1
        for (int c32 = half; c32 < (t.n >> 5) && ok; c32 += T2<F>::kEpiHalves) {
            const int row0 = t.r0 + 32 * c32;
            float v[32];
            tmem_ld32(tacc + 32 * c32, v);
            if constexpr (F == L1_FWD_MX) {
                // The FP8 L1: the gate warp pr and the up warp 2 + pr split the
                // chunk's rows for SwiGLU and the quantization of a: the up warp
                // hands the gate warp its values of rows 0-15 and takes the
                // gate values of rows 16-31 (through the upper half of the up
                // warp's staging buffer); each then computes and quantizes its
                // 16 rows.  (The FP8 forward has no activation clamp.)
                const int I = p.I;
                const int pr = warp & 1;
                const int col = t.f0 + 32 * pr;
                const uint32_t xa = stage_of_warp0 + (uint32_t)(2 + pr) * kStageEpiBytes + 4096u;  // up rows 0-15
                const uint32_t xb = xa + 2048u;                                                   // gate rows 16-31
                float o[16];  // the other warp's values of this warp's 16 rows
                if (warp >= 2) {
                    if (!warp_wait(bars.xempty(pr), (xchunk & 1u) ^ 1u, abort)) {
                        ok = false;
                        break;
                    }
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        asm volatile("st.shared.f32 [%0], %1;" ::"r"(xa + (uint32_t)(j * 32 + lane) * 4u), "f"(v[j])
                                     : "memory");
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bars.xfull(pr));
                } else {
                    if (!warp_wait(bars.gempty(pr), (xchunk & 1u) ^ 1u, abort)) {
                        ok = false;
                        break;
                    }
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        asm volatile("st.shared.f32 [%0], %1;" ::"r"(xb + (uint32_t)(j * 32 + lane) * 4u),
                                     "f"(v[16 + j])
                                     : "memory");
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bars.gfull(pr));
                }
                // h (this warp's half: gate or up) leaves by TMA store
                const uint32_t buf = stage + (nstore & 1u) * 2048u;
                if (lane == 0) bulk_wait_read<1>();
                __syncwarp();
                stage_col_sw64(buf, lane, v);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0 && col < I) {
                    tma_store_2d(om.c0, (warp >= 2 ? I : 0) + col, row0, buf);
                    bulk_commit();
                }
                const uint32_t from = warp >= 2 ? xb : xa;
                if (!warp_wait(warp >= 2 ? bars.gfull(pr) : bars.xfull(pr), xchunk & 1u, abort)) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(o[j]) : "r"(from + (uint32_t)(j * 32 + lane) * 4u)
                                 : "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive(warp >= 2 ? bars.gempty(pr) : bars.xempty(pr));
                float a16[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float g = warp >= 2 ? o[j] : v[j];
                    const float u = warp >= 2 ? v[16 + j] : o[j];
                    a16[j] = __fdividef(g, 1.0f + __expf(-g)) * u;
                }
                if (col < I) store_a_e4m3<16>(p, a16, row0 + (warp >= 2 ? 16 : 0), col, lane);
                ++xchunk;
            } else if constexpr (t2_is_l1<F>()) {
                // lanes 0-63: gate features f0..f0+63, lanes 64-127: up features f0..f0+63
                const int I = p.I;
                const int pr = warp & 1;
                const int col = t.f0 + 32 * pr;
                const uint32_t xch = stage_of_warp0 + (uint32_t)(2 + pr) * kStageEpiBytes + 4096u;
                if (warp >= 2) {
                    // up: hand the FP32 values to warp pr, store the h up half
                    if (!warp_wait(bars.xempty(pr), (xchunk & 1u) ^ 1u, abort)) {
                        ok = false;
                        break;
                    }
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        asm volatile("st.shared.f32 [%0], %1;" ::"r"(xch + (uint32_t)(j * 32 + lane) * 4u), "f"(v[j])
                                     : "memory");
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bars.xfull(pr));
                    const uint32_t buf = stage + (nstore & 1u) * 2048u;
                    if (lane == 0) bulk_wait_read<1>();
                    __syncwarp();
                    stage_col_sw64(buf, lane, v);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0 && col < I) {
                        tma_store_2d(om.c0, I + col, row0, buf);
                        bulk_commit();
                    }
                } else {
                    if (!warp_wait(bars.xfull(pr), xchunk & 1u, abort)) {
                        ok = false;
                        break;
                    }
                    float u[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        asm volatile("ld.shared.f32 %0, [%1];" : "=f"(u[j]) : "r"(xch + (uint32_t)(j * 32 + lane) * 4u)
                                     : "memory");
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bars.xempty(pr));
                    const uint32_t buf = stage + (nstore & 1u) * 4096u;
                    if (lane == 0) bulk_wait_read<1>();
                    __syncwarp();
                    stage_col_sw64(buf, lane, v);
                    if (p.clamp == INFINITY) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] = __fdividef(v[j], 1.0f + __expf(-v[j])) * u[j];
                    } else {
                        if (col < I) {
                        // record the FP32 clamp decisions for the backward:
                        // one 32-feature word per row for gate, one for up
                        uint32_t gw = 0, uw = 0;
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const uint32_t bg = __ballot_sync(0xffffffffu, clamp_pass(v[j], p.clamp) != 0.0f);
                            const uint32_t bu = __ballot_sync(0xffffffffu, clamp_pass(u[j], p.clamp) != 0.0f);
                            if (lane == j) {
                                gw = bg;
                                uw = bu;
                            }
                        }
                        const size_t words = (size_t)(2 * I / 32);
                        p.cmask[(size_t)(row0 + lane) * words + (size_t)(col / 32)] = gw;
                        p.cmask[(size_t)(row0 + lane) * words + (size_t)((I + col) / 32)] = uw;
                        }
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const float g = clamp_in(v[j], p.clamp);
                            v[j] = __fdividef(g, 1.0f + __expf(-g)) * clamp_in(u[j], p.clamp);
                        }
                    }
                    stage_col_sw64(buf + 2048, lane, v);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0 && col < I) {
                        tma_store_2d(om.c0, col, row0, buf);
                        tma_store_2d(om.c1, col, row0, buf + 2048);
                        bulk_commit();
                    }
                }
                ++xchunk;
            } else if constexpr (F == L2_DGRAD) {
                // g = dY . W2^T; da = w g; SwiGLU^T from the saved h; aw = w a;
                // d(topk weight) partial = sum over this warp's features of g a.
                // Chunk nin (counted over the launch) has its saved h and a
                // boxes in buffer nin & 1 (in_box or stage) and overwrites
                // them in place with its three output boxes; the next chunk's
                // inputs come into the other buffer meanwhile.
                const int I = p.I;
                const int col = t.f0 + 32 * warp;
                if (col < I) {
                    const int sl = __ldg(p.perm + row0 + lane);
                    const float wl = sl >= 0 ? __ldg(p.topk_w + sl) : 0.0f;
                    const uint32_t cur = (nin & 1u) ? stage : in_box;
                    if (lane == 0 && c32 + 1 < (t.n >> 5)) {
                        bulk_wait_read<0>();  // the other buffer's stores (previous chunk) have read it
                        const uint32_t nxt = (nin & 1u) ? in_box : stage;
                        const uint32_t eb = bars.ein(warp, (nin + 1u) & 1u);
                        mbar_arrive_expect_tx(eb, (uint32_t)kT2InBytes);
                        tma_load_2d(nxt, mapH, col, row0 + 32, eb);
                        tma_load_2d(nxt + 2048, mapH, I + col, row0 + 32, eb);
                        tma_load_2d(nxt + 4096, mapAs, col, row0 + 32, eb);
                    }
                    if (!warp_wait(bars.ein(warp, nin & 1u), (nin >> 1) & 1u, abort)) {
                        ok = false;
                        break;
                    }
                    {
                        float prod[32];
#pragma unroll
                        for (int j = 0; j < 32; ++j) prod[j] = v[j] * lds_sw64(cur + 4096, j, lane);
                        // lane j ends with the sum over the warp's 32 features of row j
                        transpose_reduce_step<16>(prod, lane);
                        transpose_reduce_step<8>(prod, lane);
                        transpose_reduce_step<4>(prod, lane);
                        transpose_reduce_step<2>(prod, lane);
                        transpose_reduce_step<1>(prod, lane);
                        p.outf[(size_t)(row0 + lane) * (size_t)p.dw_cols + (size_t)(col >> 5)] = prod[0];
                    }
                    // the forward's clamp decisions of this warp's features: lane
                    // l loads the words of row row0 + l, row j's are shuffled out
                    uint32_t gmask = 0xffffffffu, umask = 0xffffffffu;
                    if (p.clamp < INFINITY) {
                        const size_t words = (size_t)(2 * I / 32);
                        gmask = __ldg(p.cmask + (size_t)(row0 + lane) * words + (size_t)(col / 32));
                        umask = __ldg(p.cmask + (size_t)(row0 + lane) * words + (size_t)((I + col) / 32));
                    }
                    // element (row j, feature lane) of each box is read, then
                    // overwritten, by this lane only: in place is safe
                    if (p.clamp < INFINITY)
                        swiglu_t_chunk<true>(cur, cur, true, lane, wl, v, p.clamp, gmask, umask);
                    else
                        swiglu_t_chunk<false>(cur, cur, true, lane, wl, v, p.clamp, gmask, umask);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(om.c0, col, row0, cur);
                        tma_store_2d(om.c0, I + col, row0, cur + 2048);
                        tma_store_2d(om.c1, col, row0, cur + 4096);
                        bulk_commit();
                    }
                    ++nin;
                }
            } else {
                // one output: o = w (a . W2) (L2 forward) or dxp = dh . W1^T (L1 dgrad)
                if constexpr (F == L2_FWD || F == L2_FWD_MX) {
                    const int sl = __ldg(p.perm + row0 + lane);
                    const float wl = sl >= 0 ? __ldg(p.topk_w + sl) : 0.0f;
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] *= __shfl_sync(0xffffffffu, wl, j);
                }
                const uint32_t buf = stage + (nstore & 1u) * 2048u;
                if (lane == 0) bulk_wait_read<1>();
                __syncwarp();
                stage_col_sw64(buf, lane, v);
                fence_proxy_async_smem();
                __syncwarp();
                const int col = t.f0 + 32 * warp;
                if (lane == 0 && col < p.H) {
                    tma_store_2d(om.c0, col, row0, buf);
                    bulk_commit();
                }
            }
            ++nstore;
        }
        if (!ok) break;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(tempty_leader[acc]);
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
}

template <int F>
__global__ void __launch_bounds__(kT2Threads, 1)
    moe_gemm_pair_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                         const __grid_constant__ CUtensorMap mapC0, const __grid_constant__ CUtensorMap mapC1,
                         const __grid_constant__ CUtensorMap mapD, const GemmArgs p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw);
    const uint32_t sA = base;
    const uint32_t sB = base + T2<F>::kStages * kT2ABytes;
    const uint32_t sStage = sB + T2<F>::kStages * kT2BBytes;
    const uint32_t sIn = sStage + kEpiWarps * kStageEpiBytes;  // L2 dgrad epilogue inputs
    const uint32_t bar_base = sIn + T2<F>::kInBytes;
    const uint32_t ring = bar_base + kT2RingOff;
    uint8_t* tail = base_ptr + (bar_base - base);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tail + 8 * kT2NumBars);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const T2Bars bars{bar_base};
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int rank = (int)cluster_ctarank();

    if (threadIdx.x == 0) {
        // even CTA: its producer's arrive (both CTAs' TMA bytes), its gather
        // threads and the odd CTA's relay; odd CTA: its gather threads only
        // (t2_sf_rows flavours: the scale warp's lanes in place of the gather threads)
        const uint32_t row_thr = T2<F>::kGather ? 32u * kGatherWarps : (t2_sf_rows<F>() ? 32u : 0u);
        const uint32_t full_count = row_thr == 0u ? 1u : (rank == 0 ? 2u + row_thr : row_thr);
        for (int s = 0; s < kT2Stages; ++s) {
            mbar_init(bars.full(s), full_count);
            mbar_init(bars.empty(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(bars.tfull(a), 1);
            mbar_init(bars.tempty(a), 2 * kEpiWarps * T2<F>::kEpiHalves);
            mbar_init(bars.xfull(a), 1);
            mbar_init(bars.xempty(a), 1);
            mbar_init(bars.gfull(a), 1);
            mbar_init(bars.gempty(a), 1);
        }
        mbar_init(bars.drain(), 1);
        for (int w = 0; w < kEpiWarps; ++w) {
            mbar_init(bars.ein(w, 0), 1);
            mbar_init(bars.ein(w, 1), 1);
        }
        // consumers of a published unit: TMA producers, MMA or relay,
        // epilogue warps, (gathering flavours) gather warps and (t2_sf_rows
        // flavours) the scale warp, in both CTAs
        const uint32_t consumers =
            2u * (1u + (uint32_t)T2<F>::kProducers + kEpiWarps * (uint32_t)T2<F>::kEpiHalves +
                  (T2<F>::kGather ? (uint32_t)kGatherWarps : 0u) + (t2_sf_rows<F>() ? 1u : 0u));
        for (int i = 0; i < kUR; ++i) {
            mbar_init(bars.ufull(i), 1);
            mbar_init(bars.uempty(i), consumers);
        }
        mbar_init(bars.ustart(), 1);
        *abort = 0;
        fence_mbar_init();
    }
    if (warp == kWarpMma) {
        tmem_alloc_pair(smem_addr(tmem_slot), 2 * kBN);
        tmem_relinquish_pair();
    }
    if (warp == kWarpTma && lane == 0) {
        tma_prefetch_map(&mapA);
        if constexpr (!T2<F>::kGather || F == L2_DGRAD || F == L1_FWD_MX) tma_prefetch_map(&mapB);
        if constexpr (F == L2_DGRAD || F == L2_FWD_MX) tma_prefetch_map(&mapD);
        tma_prefetch_map(&mapC0);
        if constexpr (t2_is_l1<F>() || F == L2_DGRAD) tma_prefetch_map(&mapC1);
    }
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    // producer id of this warp's lane 0, or -1
    int pid = warp == kWarpTma ? 0 : -1;
    if constexpr (!T2<F>::kGather) {
        // the gather warps are free in the flavours fed by TMA alone
        if (warp >= kWarpGather0 && warp < kWarpGather0 + T2<F>::kProducers - 1) pid = 1 + warp - kWarpGather0;
    }
    if (pid >= 0) {
        if (lane == 0) t2_role_tma<F>(&mapA, &mapB, &mapD, p, ring, sA, sB, sIn, bars, abort, rank, pid);
    } else if (warp == kWarpSched) {
        if (lane == 0 && rank == 0) t2_role_sched<F>(p, ring, bars, abort);
    } else if (T2<F>::kEpiHalves > 1 && warp >= kWarpGather0 + T2<F>::kProducers - 1 &&
               warp < kWarpGather0 + T2<F>::kProducers - 1 + kEpiWarps) {
        // second epilogue warp of TMEM lane quadrant warp % 4: the odd
        // chunks, staged in the upper half of that quadrant's buffer
        const int q = warp & 3;
        t2_role_epilogue<F>(p, OutMaps{&mapC0, &mapC1}, &mapB, &mapD, ring, bars, tmem_base,
                            sStage + q * kStageEpiBytes + 4096, sStage, sIn + q * kT2InBytes, abort, q, lane, rank, 1);
    } else if (t2_sf_rows<F>() && warp == t2_sf_rows_warp<F>()) {
        if constexpr (t2_sf_rows<F>()) t2_role_sf_rows<F>(p, ring, sIn, bars, abort, lane, rank);
        cp_async_wait_all();
    } else if (warp >= kWarpGather0) {
        if constexpr (T2<F>::kGather) t2_role_gather<F>(p, ring, sB, sIn, bars, abort, warp - kWarpGather0, lane, rank);
        cp_async_wait_all();
    } else if (warp == kWarpMma) {
        if (rank == 0) {
            if constexpr (t2_is_mx<F>())
                t2_role_mma_mx<F>(p, ring, sA, sB, sIn, bars, tmem_base, abort, lane);
            else
                t2_role_mma<F>(p, ring, sA, sB, bars, tmem_base, abort, lane);
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
            t2_role_relay<F>(p, ring, bars, abort);
        }
    } else {
        t2_role_epilogue<F>(p, OutMaps{&mapC0, &mapC1}, &mapB, &mapD, ring, bars, tmem_base,
                            sStage + warp * kStageEpiBytes, sStage, sIn + warp * kT2InBytes, abort, warp, lane, rank,
                            0);
    }
    if (pid >= 0 && lane == 0 && *abort) {
        // bulk copies already issued land within microseconds; give them time
        const uint64_t t0 = global_timer_ns();
        while (global_timer_ns() - t0 < 2000000ull) {
        }
    }
    __syncwarp();
    tc_fence_before();
    cluster_sync();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, 2 * kBN);
    }
    if (threadIdx.x == 0 && *abort) atomicOr(reinterpret_cast<int*>(p.status + MOE_STATUS_FLAGS), 1);
}

// Launches one 2-CTA cluster per unit up to the number of clusters that fit
// on the device at once (persistent: each cluster takes units from the unit
// feed until none is left).
template <int F>
int launch_gemm_pair(const GemmArgs& a, const GemmMaps& m, int max_units, cudaStream_t st) {
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
    cfg.blockDim = dim3(kT2Threads, 1, 1);
    cfg.dynamicSmemBytes = t2_smem_bytes<F>();
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int fit = clusters_fit[dev].load(std::memory_order_relaxed);
    if (fit == 0) {
        // set once per device, outside any stream capture (on the first call)
        e = cudaFuncSetAttribute(moe_gemm_pair_kernel<F>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 t2_smem_bytes<F>());
        if (e != cudaSuccess) return (int)e;
        int sms = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return (int)e;
        cfg.gridDim = dim3((unsigned)(sms & ~1), 1, 1);
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, moe_gemm_pair_kernel<F>, &cfg);
        if (e != cudaSuccess) return (int)e;
        if (n < 1) return (int)cudaErrorInvalidConfiguration;
        fit = n;
        clusters_fit[dev].store(n, std::memory_order_relaxed);
    }
    if (max_units <= 0) return 0;
    const int clusters = max_units < fit ? max_units : fit;
    cfg.gridDim = dim3((unsigned)(2 * clusters), 1, 1);
    e = cudaLaunchKernelEx(&cfg, moe_gemm_pair_kernel<F>, m.a, m.b, m.c0, m.c1, m.d, a);
    if (e != cudaSuccess) return (int)e;
    return (int)cudaGetLastError();
}

}  // namespace moe
