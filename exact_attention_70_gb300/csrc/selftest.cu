// selftest.cu -- exercises the kernels' failure path on a live GPU without faulting it.
//
// Every wait in the attention kernels is bounded (Watchdog in ptx.cuh): when a barrier phase
// does not complete in time, the waiting thread raises the timeout bit of the device status
// word, sets its CTA's abort flag so the other roles leave their loops, and returns.  This
// kernel runs that same wait, with a 20 ms limit, on an mbarrier that nothing ever arrives on,
// so a test can check that the status word reports the timeout and that the context stays
// usable afterwards.
//
// It also evaluates, for a test, the softcap map of the modifier kernel (softcap.cuh) on given
// scores, through the same device function.
#include "kernels.h"
#include "ptx.cuh"
#include "softcap.cuh"

namespace attn {

namespace {

constexpr unsigned long long kSelfTestLimitNs = 20000000ull;

__global__ void __launch_bounds__(64, 1) watchdog_selftest_kernel(unsigned* status) {
    __shared__ uint64_t never;  // no thread and no copy ever arrives on it
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&never, 1);
        abort_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();
    const Watchdog wd{&abort_flag, status};
    // Two warps wait: the first to run out raises the status bit and the abort flag, the
    // other sees the flag and gives up as well.
    if ((threadIdx.x & 31) == 0) (void)wd.wait<kSelfTestLimitNs>(&never, 0);
    __syncthreads();
}

// out[i] = c tanh(scale s[i] / c) as the modifier kernel computes it (n even, one pair a thread)
__global__ void __launch_bounds__(256) softcap_selftest_kernel(const float* s, float* out, int n,
                                                               float scale, float softcap) {
    const int i = 2 * (blockIdx.x * blockDim.x + threadIdx.x);
    if (i + 1 >= n) return;
    float s0 = s[i], s1 = s[i + 1];
    const float ku = softcap_ku(scale, softcap);
    softcap_tanh2(s0, s1, f2_make(ku, ku));
    out[i] = softcap * s0;
    out[i + 1] = softcap * s1;
}

}  // namespace

cudaError_t launch_softcap_selftest(const float* s, float* out, int n, float scale, float softcap,
                                    cudaStream_t stream) {
    const int pairs = n / 2;
    if (pairs == 0) return cudaSuccess;
    softcap_selftest_kernel<<<(pairs + 255) / 256, 256, 0, stream>>>(s, out, n, scale, softcap);
    return cudaGetLastError();
}

cudaError_t launch_watchdog_selftest(unsigned* status, cudaStream_t stream) {
    watchdog_selftest_kernel<<<1, 64, 0, stream>>>(status);
    return cudaGetLastError();
}

}  // namespace attn
