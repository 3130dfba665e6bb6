// wait_probe.cu -- a diagnostic of the bounded waits every libdsa kernel relies on.
//
// One CTA waits on an mbarrier that nothing ever completes, through the same mbar_wait
// the pipelines use: the first waiter gives up after the time limit, records
// ERR_WAIT_TIMEOUT in the device error word and raises the CTA's abort flag; a second
// waiter on the same barrier sees the flag and gives up too.  Nothing faults and nothing
// hangs: the kernel ends, the host reads the word, and the context stays usable.
#include "internal.h"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr unsigned int KID_PROBE = 8;  // kernel id in the device error word

// out[0..1]: whether each waiter saw its barrier complete (expected 0); out[2..3]: how
// long each waited, in nanoseconds.
__global__ void __launch_bounds__(64, 1) wait_probe_kernel(unsigned long long *out) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);  // one arrival completes the phase; none ever comes
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if ((threadIdx.x & 31) == 0) {
        const int w = threadIdx.x >> 5;
        const uint64_t t0 = globaltimer_ns();
        const bool ok = mbar_wait(&bar, 0, KID_PROBE, &abort_flag);
        out[w] = ok ? 1ull : 0ull;
        out[2 + w] = globaltimer_ns() - t0;
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_inval(&bar);
}

}  // namespace

cudaError_t launch_wait_probe(unsigned long long *out, cudaStream_t stream) {
    wait_probe_kernel<<<1, 64, 0, stream>>>(out);
    return cudaGetLastError();
}

DSA_DEFINE_ERROR_READER(take_error_probe)

}  // namespace dsa
