// Launch sequence of one KDA forward: the intra-chunk kernel (chunk-parallel)
// and the state scan (serial over each long sequence's chunks) -- or, when the
// scan's walks leave enough SMs free, both in one fused launch -- then the
// token-by-token kernel for the short sequences.
#include "kda_internal.h"

namespace kda {

const char* kernel_name(int i) {
    static const char* names[kNumKernels] = {"kda_intra", "kda_scan", "kda_fused", "kda_decode"};
    return (i >= 0 && i < kNumKernels) ? names[i] : nullptr;
}

int num_sms() {
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
    const unsigned decode = (p.n_short > 0 && p.short_list) ? 8u : 0u;
    if (fused_eligible(p)) return 4u | decode;
    return (p.n_chunks > 0 ? 1u : 0u) | (n_scan > 0 ? 2u : 0u) | decode;
}

static int n_scan_of(const FwdParams& p) { return p.long_list ? p.n_long : p.N; }

// The scan's value-row split for this call; it counts the token-by-token
// kernel's (sequence, head) pairs, which run beside the scan.  The split does
// not depend on whether the kernels are timed one by one.
static int groups_of(const FwdParams& p) {
    const int beside = p.short_list && p.n_short > 0 ? p.n_short * p.H : 0;
    return scan_groups(n_scan_of(p), p.H, num_sms(), beside);
}

cudaError_t launch_forward(const FwdParams& p, cudaStream_t s, cudaEvent_t* marks) {
    cudaError_t e;
    const bool fused = fused_eligible(p);
    FwdParams q = p;  // the separate kernels neither publish nor wait for ready flags
    q.ready = nullptr;
    q.queue = nullptr;
    if (marks) cudaEventRecord(marks[0], s);
    if (!fused) {
        e = launch_intra(q, s);
        if (e != cudaSuccess) return e;
    }
    if (marks) cudaEventRecord(marks[1], s);
    if (!fused) {
        // right behind the intra-chunk kernel (not when the kernels are timed
        // one by one)
        e = launch_scan(q, groups_of(q), s, !marks && q.n_chunks > 0);
        if (e != cudaSuccess) return e;
    }
    if (marks) cudaEventRecord(marks[2], s);
    if (fused) {
        e = launch_fused(p, s);
        if (e == cudaErrorCooperativeLaunchTooLarge) {
            // the device refused the cooperative launch (and is marked so for
            // later calls): run the two kernels instead, re-recording their
            // marks so the per-kernel times land on kda_intra and kda_scan
            (void)cudaGetLastError();
            if (marks) cudaEventRecord(marks[0], s);
            e = launch_intra(q, s);
            if (marks) cudaEventRecord(marks[1], s);
            if (e == cudaSuccess) e = launch_scan(q, groups_of(q), s);
            if (marks) cudaEventRecord(marks[2], s);
        }
        if (e != cudaSuccess) return e;
    }
    if (marks) cudaEventRecord(marks[3], s);
    // after the plain scan (not the fused launch, which fills the GPU, nor when
    // the kernels are timed one by one), the token-by-token kernel runs beside it
    const bool beside = !fused && !marks && n_scan_of(q) > 0 && q.n_chunks > 0;
    e = launch_decode(q, s, beside);
    if (e != cudaSuccess) return e;
    if (marks) cudaEventRecord(marks[4], s);
    return cudaSuccess;
}

}  // namespace kda
