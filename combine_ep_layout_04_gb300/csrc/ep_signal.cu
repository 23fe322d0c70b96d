// ep_signal.cu -- the bounded wait of ep_wait_signal: one thread polls one
// destination rank's arrival signal (GIN-style waitSignal, with a time limit)
// and writes EP_OK or EP_ERR_NOT_READY to the caller's status word.
#include "ep_internal.cuh"
#include "ep_signal.cuh"

namespace ep {
namespace {

__global__ void wait_signal_kernel(const unsigned long long *signal, unsigned long long expected,
                                   unsigned long long timeout_ns, int32_t *status) {
    if (threadIdx.x == 0) *status = ep_signal_wait(signal, expected, timeout_ns) ? EP_OK : EP_ERR_NOT_READY;
}

}  // namespace

ep_status launch_wait_signal(const unsigned long long *signal, unsigned long long expected,
                             unsigned long long timeout_ns, int32_t *status, cudaStream_t st) {
    wait_signal_kernel<<<1, 32, 0, st>>>(signal, expected, timeout_ns, status);
    return cudaGetLastError() == cudaSuccess ? EP_OK : EP_ERR_CUDA;
}

}  // namespace ep
