// lora_wait_selftest: runs the bounded mbarrier wait that every tensor-core kernel of this
// library uses, on one barrier, so that a test can watch a wait give up.
//
// Every pipeline wait of the library (TMA stage full/empty, accumulator ready, DSMEM exchange)
// is bounded: after its limit it raises the CTA's abort flag, the kernel records LORA_ETIMEOUT
// in the batch status word, skips its output and returns -- no trap, no endless spin.  Making
// a real pipeline stall would need a broken kernel, so this entry point instead waits on a
// barrier that nothing completes (arrive = 0) with a caller-given limit, through the same
// mbar_wait and report_timeout_status the kernels call.  With arrive = 1 the barrier completes
// before the wait and the output is written.
#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace lora {
namespace {

__global__ void __launch_bounds__(128) wait_selftest_kernel(int32_t* status, float* out, int n, int arrive,
                                                           unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        ptx::mbar_init(&bar, 1);
        abort_flag = 0;
        ptx::fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        if (arrive) ptx::mbar_arrive(&bar);
        if (!ptx::mbar_wait(&bar, 0, &abort_flag, limit_ns)) ptx::report_timeout_status(status);
    }
    __syncthreads();
    if (*(volatile int*)&abort_flag) return;  // the output of a call whose wait gave up stays untouched
    for (int i = threadIdx.x; i < n; i += blockDim.x) out[i] = 1.0f;
}

constexpr unsigned long long kSelftestMaxNs = 100000000ull;  // 0.1 s

}  // namespace
}  // namespace lora

using namespace lora;

extern "C" int lora_wait_selftest(int32_t* status_dev, float* out_dev, int n, int arrive, uint64_t limit_ns,
                                  void* stream) {
    if (!status_dev || (n > 0 && !out_dev)) return set_error(LORA_EINVAL, "status/out is NULL");
    if (n < 0 || n > (1 << 20)) return set_error(LORA_EINVAL, "n %d outside [0, 2^20]", n);
    if (limit_ns > kSelftestMaxNs)
        return set_error(LORA_EINVAL, "limit %llu ns above %llu ns", (unsigned long long)limit_ns, kSelftestMaxNs);
    wait_selftest_kernel<<<1, 128, 0, static_cast<cudaStream_t>(stream)>>>(status_dev, out_dev, n, arrive ? 1 : 0,
                                                                           (unsigned long long)limit_ns);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(LORA_ECUDA, "wait_selftest_kernel: %s", cudaGetErrorString(e));
    count_launch();
    return LORA_OK;
}
