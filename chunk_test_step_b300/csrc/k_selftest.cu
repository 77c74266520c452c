// Self-test of the failure path of the library's bounded waits: one thread
// initialises an mbarrier that nothing will arrive on and waits on it with a
// short budget, exactly as every pipeline wait in the kernels does; when the
// budget runs out it sets ST_TIMEOUT in the state's status word and returns.
// The GPU stays usable (nothing traps or spins without a limit), and the host
// reads LACT_ERR_TIMEOUT from lact_sync_status.
#include "lact_internal.cuh"
#include "tc_ptx.cuh"

namespace lact {

namespace {

__global__ void k_wait_selftest(int* status, uint64_t budget_ns) {
    __shared__ __align__(8) uint64_t never;
    const uint32_t b = tc::smem_u32(&never);
    tc::mbar_init(b, 1);
    tc::fence_mbar_init();
    if (!tc::mbar_wait(b, 0, budget_ns)) atomicOr(status, ST_TIMEOUT);
}

}  // namespace

cudaError_t launch_wait_selftest(int* status, uint64_t budget_ns, cudaStream_t s) {
    k_wait_selftest<<<1, 1, 0, s>>>(status, budget_ns);
    g_launches++;
    return cudaGetLastError();
}

}  // namespace lact
