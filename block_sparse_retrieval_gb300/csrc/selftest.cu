// selftest.cu -- the bounded on-chip waits give up and report, they never hang.
//
// Every wait of the decode kernels (stage barriers, cluster hand-offs) is bounded by
// kWaitLimitNs and, when it runs out, sets SRKV_EFLAG_TIMEOUT and lets the kernel finish.
// This kernel exercises exactly that path without any fault: a CTA-scope mbarrier and a
// cluster-scope mbarrier that nothing ever arrives on.  Both waits run to their limit,
// raise the flag and return; the CTAs then leave normally, so the context stays usable.
#include "select.cuh"

namespace srkv {
namespace {

__global__ void __cluster_dims__(2, 1, 1) wait_timeout_kernel(int32_t* error_flags) {
  __shared__ uint64_t local_bar, cluster_bar;
  if (threadIdx.x == 0) {
    mbar_init(&local_bar, 1);    // one arrival expected, none will come
    mbar_init(&cluster_bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before either waits
  if (threadIdx.x == 0) {
    uint32_t flags = 0;
    if (!mbar_wait(&local_bar, 0)) flags |= SRKV_EFLAG_TIMEOUT;
    if (!mbar_wait_cluster(&cluster_bar, 0)) flags |= SRKV_EFLAG_TIMEOUT;
    if (flags) raise_flags(error_flags, flags);
  }
  __syncthreads();
  cluster_sync();  // neither CTA leaves while the other may still touch the cluster
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(int32_t* error_flags, cudaStream_t stream) {
  wait_timeout_kernel<<<2, 32, 0, stream>>>(error_flags);
  return cudaGetLastError();
}

}  // namespace srkv
