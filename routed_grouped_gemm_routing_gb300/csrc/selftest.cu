// Diagnostic kernel: runs the bounded-wait helpers of the GEMM kernels out on
// purpose, on a barrier that no thread or copy ever arrives on, so that the
// give-up path (abort flag raised, roles leave their waits, status bit 0 set
// for the host) can be checked without a fault or a hang.  Nothing of the
// layer runs here.
#include "gemm_common.cuh"

namespace moe {
namespace {

// One CTA of three warps, each in the wait form one kind of GEMM role uses:
//   warp 0: warp_wait (every lane polls; epilogue warps), limit limit_ns;
//   warp 1: warp_wait_uniform (warp-vote poll; MMA warps), limit 4 * limit_ns;
//   warp 2: mbar_wait by lane 0 alone (TMA producer threads), limit 4 * limit_ns.
// Warp 0 gives up first and raises the abort flag; warps 1 and 2 must then
// leave on the flag, well before their own limits.  elapsed[w] = ns warp w
// spent waiting (-1 if its wait returned true, which cannot happen here).
__global__ void __launch_bounds__(96, 1)
    moe_wait_selftest_kernel(int32_t* status, uint64_t limit_ns, long long* elapsed) {
    __shared__ __align__(8) uint64_t bar_word;
    __shared__ int abort_word;
    const uint32_t bar = smem_addr(&bar_word);
    volatile int* abort = &abort_word;
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);  // phase 0 completes only after one arrival, and none comes
        *abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint64_t t0 = global_timer_ns();
    bool ok = true;
    if (warp == 0) {
        ok = warp_wait(bar, 0u, abort, limit_ns);
    } else if (warp == 1) {
        ok = warp_wait_uniform<false>(bar, 0u, abort, 4 * limit_ns);
    } else if (lane == 0) {
        ok = mbar_wait(bar, 0u, abort, 4 * limit_ns);
    }
    const uint64_t dt = global_timer_ns() - t0;
    if (lane == 0 && elapsed) elapsed[warp] = ok ? -1ll : (long long)dt;
    __syncthreads();
    if (threadIdx.x == 0 && *abort) atomicOr(reinterpret_cast<int*>(status + MOE_STATUS_FLAGS), 1);
}

}  // namespace

int launch_wait_selftest(int32_t* status, uint64_t limit_ns, long long* elapsed, cudaStream_t st) {
    trace_pre(st);
    moe_wait_selftest_kernel<<<1, 96, 0, st>>>(status, limit_ns, elapsed);
    trace_post(st, "wait_selftest");
    return (int)cudaGetLastError();
}

}  // namespace moe
