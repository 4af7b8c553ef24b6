// Launch sequence of one chunkwise KDA forward: the intra-chunk kernel
// (chunk-parallel) then the state scan (serial over each sequence's chunks).
#include "kda_internal.h"

namespace kda {

const char* kernel_name(int i) {
    static const char* names[kNumKernels] = {"kda_intra", "kda_scan"};
    return (i >= 0 && i < kNumKernels) ? names[i] : nullptr;
}

static int num_sms() {
    static int cached[32] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev >= 32) return 148;
    if (!cached[dev]) {
        int v = 0;
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        cached[dev] = v > 0 ? v : 148;
    }
    return cached[dev];
}

cudaError_t launch_forward(const FwdParams& p, cudaStream_t s, cudaEvent_t* marks) {
    cudaError_t e;
    if (marks) cudaEventRecord(marks[0], s);
    e = launch_intra(p, s);
    if (e != cudaSuccess) return e;
    if (marks) cudaEventRecord(marks[1], s);
    e = launch_scan(p, scan_groups(p.N, p.H, num_sms()), s);
    if (e != cudaSuccess) return e;
    if (marks) cudaEventRecord(marks[2], s);
    return cudaSuccess;
}

}  // namespace kda
