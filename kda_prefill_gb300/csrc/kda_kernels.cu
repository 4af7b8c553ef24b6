// Launch sequence of one KDA forward: the intra-chunk kernel (chunk-parallel),
// the state scan (serial over each long sequence's chunks), then the
// token-by-token kernel for the short sequences.
#include "kda_internal.h"

namespace kda {

const char* kernel_name(int i) {
    static const char* names[kNumKernels] = {"kda_intra", "kda_scan", "kda_decode"};
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

unsigned launched_kernels(const FwdParams& p) {
    const int n_scan = p.long_list ? p.n_long : p.N;
    return (p.n_chunks > 0 ? 1u : 0u) | (n_scan > 0 ? 2u : 0u) |
           (p.n_short > 0 && p.short_list ? 4u : 0u);
}

cudaError_t launch_forward(const FwdParams& p, cudaStream_t s, cudaEvent_t* marks) {
    cudaError_t e;
    if (marks) cudaEventRecord(marks[0], s);
    e = launch_intra(p, s);
    if (e != cudaSuccess) return e;
    if (marks) cudaEventRecord(marks[1], s);
    const int n_scan = p.long_list ? p.n_long : p.N;
    e = launch_scan(p, scan_groups(n_scan, p.H, num_sms()), s);
    if (e != cudaSuccess) return e;
    if (marks) cudaEventRecord(marks[2], s);
    e = launch_decode(p, s);
    if (e != cudaSuccess) return e;
    if (marks) cudaEventRecord(marks[3], s);
    return cudaSuccess;
}

}  // namespace kda
