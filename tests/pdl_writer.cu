// pdl_writer.cu -- test helper, not part of libmoe: a "foreign" kernel that
// writes a buffer between moe_plan and moe_dispatch on the same stream.
//
// It is launched with programmatic dependent launch and lets its dependents
// start at once (before it has written anything), then waits for the kernel
// before it, lingers for `delay_ns` nanoseconds of %globaltimer (a bounded
// wait on the clock, never on a flag), and copies src to dst.  A dependent
// that reads dst before its own griddepcontrol.wait can see the old
// contents; one that reads after the wait sees the copy.
#include <cstdint>
#include <cuda_runtime.h>

namespace {

__global__ void pdl_write_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, long long n16,
                                 long long delay_ns) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (delay_ns > 0) {
        unsigned long long t0, t;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
        do {
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
        } while (t - t0 < (unsigned long long)delay_ns);
    }
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n16;
         i += (long long)gridDim.x * blockDim.x)
        dst[i] = src[i];
}

}  // namespace

// Copy `bytes` (a multiple of 16; both pointers 16-byte aligned) from src to
// dst on `stream`, launched as described above.  delay_ns is capped at one
// millisecond.  Returns the cudaError_t of the launch.
extern "C" __attribute__((visibility("default"))) int pdl_write(const void* src, void* dst, long long bytes,
                                                                 long long delay_ns, void* stream) {
    if (bytes <= 0 || bytes % 16 != 0) return (int)cudaErrorInvalidValue;
    if (delay_ns > 1000000) delay_ns = 1000000;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(64);
    cfg.blockDim = dim3(256);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return (int)cudaLaunchKernelEx(&cfg, pdl_write_kernel, static_cast<const uint4*>(src), static_cast<uint4*>(dst),
                                   bytes / 16, delay_ns);
}
