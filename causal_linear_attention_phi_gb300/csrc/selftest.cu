// selftest.cu -- exercises the bounded-wait path of the device code without a fault:
// one thread waits on an mbarrier phase that nothing completes.  The wait gives up
// after its cycle limit (about a second), records LA_ERR_TIMEOUT in the sticky error
// word and returns, and the kernel ends normally, so the context stays usable.
#include "la_internal.cuh"
#include "sm100.cuh"

namespace la {
la_status checked_device();
la_status failed(la_status st, const char* msg);
void clear_detail();

namespace {

__global__ void bounded_wait_selftest_kernel(int* err) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        sm100::mbar_init(&bar, 1);  // one arrival would complete phase 0; none is made
        sm100::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) (void)sm100::mbar_wait(&bar, 0, err, LA_ERR_TIMEOUT);
}

}  // namespace
}  // namespace la

extern "C" la_status la_selftest_bounded_wait(la_stream_t stream) {
    la::clear_detail();
    la_status st = la::checked_device();
    if (st != LA_OK) return st;
    int* err = la::device_error_word();
    if (!err) return la::failed(LA_ERR_CUDA, "cannot locate the device error word");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    la::launch_begin("bounded_wait_selftest", s);
    la::bounded_wait_selftest_kernel<<<1, 32, 0, s>>>(err);
    return la::launch_end("bounded_wait_selftest", s) == cudaSuccess
               ? LA_OK
               : la::failed(LA_ERR_CUDA, "la_selftest_bounded_wait: launch failed");
}
