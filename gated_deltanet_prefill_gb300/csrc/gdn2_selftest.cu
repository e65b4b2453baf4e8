// Self-test of the kernels' failure detection.  Every wait in the tensor-core
// kernels is an mbarrier wait bounded in wall time (tc::mbar_wait); when it
// gives up, the kernel records GDN2_ERR_TIMEOUT in the workspace status word
// and unwinds, so the CUDA context stays usable and the host reads the error
// with gdn2_device_status.  This entry point exercises that path on purpose:
// one CTA waits, through the same helper, on an mbarrier that nothing ever
// completes, with a short limit, records the timeout and returns.
#include "gdn2_internal.cuh"
#include "gdn2_tc.cuh"

namespace gdn2 {

namespace {

__global__ void gdn2_wait_selftest_kernel(int *status, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        tc::mbar_init(&bar, 1);  // expects one arrival that never comes
        tc::fence_mbar_init();
        status[0] = GDN2_OK;
        status[1] = 0;
        status[2] = GDN2_OK;
        status[3] = GDN2_OK;
        status[5] = 0;
    }
    __syncthreads();
    if (threadIdx.x == 0 && !tc::mbar_wait_ns(&bar, 0, limit_ns))
        atomicExch(status + 2, static_cast<int>(GDN2_ERR_TIMEOUT));
}

}  // namespace

}  // namespace gdn2

using namespace gdn2;

extern "C" {

gdn2_status gdn2_selftest_wait_timeout(void *workspace, size_t workspace_bytes, uint64_t limit_ns, void *stream) {
    if (!workspace) return GDN2_ERR_NULL;
    if (workspace_bytes < kRecurrentWorkspaceBytes) return GDN2_ERR_WORKSPACE;
    if (limit_ns < 1000u || limit_ns > 100000000u) return GDN2_ERR_SHAPE;  // 1 us .. 100 ms
    if (!device_is_sm103(nullptr)) return GDN2_ERR_ARCH;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaGetLastError();
    gdn2_wait_selftest_kernel<<<1, 32, 0, s>>>(static_cast<int *>(workspace), limit_ns);
    return cudaGetLastError() == cudaSuccess ? GDN2_OK : GDN2_ERR_LAUNCH;
}

}  // extern "C"
