// fa_common.cuh -- pieces shared by the forward and backward attention kernels:
// bounded mbarrier waits with a CTA-wide abort path, the device error codes, the
// 128-byte swizzle used by TMA tiles and tcgen05 operands, and dependent launches.
#pragma once

#include "sm100_ptx.cuh"

namespace fa {

// Device-side error codes written to the library's error word (first error wins).
enum DeviceError : int {
    kDevOk = 0,
    kDevTimeoutLoad = 1,     // a TMA load never completed
    kDevTimeoutMma = 2,      // an MMA completion never arrived
    kDevTimeoutConsumer = 3, // a consumer never released a buffer
    kDevTimeoutSoftmax = 4,  // softmax/epilogue warps never signalled
};

// A wait gives up after this long (the kernels' real waits last microseconds).
constexpr uint64_t kWaitLimitNs = 4000000000ull;

// Wait for phase `parity` of mbarrier `bar`. Returns false (and raises the CTA abort flag
// and the global error word) if `limit_ns` expires, or if another role already aborted.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                           int* err, int code, uint64_t limit_ns = kWaitLimitNs) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if ((it & 15u) == 0) {
            if (*abort_flag) return false;
            if (ptx::globaltimer_ns() - t0 > limit_ns) {
                *abort_flag = 1;
                atomicCAS(err, 0, code);
                return false;
            }
        }
    }
}

// wait_phase for a whole warp: every lane polls, and the outcome is made warp-uniform.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          int* err, int code, uint64_t limit_ns = kWaitLimitNs) {
    return __all_sync(0xffffffffu, wait_phase(bar, parity, abort_flag, err, code, limit_ns));
}

// Byte offset of the 16-byte unit `u` (0..7) of row `r` inside a 128-byte-swizzled tile whose
// rows are 128 bytes apart (the layout TMA writes with CU_TENSOR_MAP_SWIZZLE_128B and the
// tcgen05 descriptors read with layout type 2). The tile base must be 1024-byte aligned.
__device__ __forceinline__ uint32_t sw128_offset(uint32_t r, uint32_t u) {
    return r * 128u + ((u ^ (r & 7u)) << 4);
}

// Launch with programmatic stream serialization: the kernel may start while the one before it
// in the stream finishes; it calls griddep_wait before using that kernel's results (or any
// buffer that kernel may still read). Without a programmatic trigger in the kernel before it,
// the launch behaves like an ordinary one.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

}  // namespace fa
