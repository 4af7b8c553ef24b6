// State scan of the chunkwise KDA forward: one CTA per (long sequence, head, block of
// VS = 8*NT value rows of the state), walking the sequence's chunks in order.
//
// Per chunk, with the incoming state S (VS rows x K):
//   U = u - w S^T                 (C x VS)   new values of the chunk
//   S = S Diag(gamma) + U^T kg    (VS x K)   the state after the chunk
//   o = qg S^T + A_qk U           (C x VS)   written to `out`
// (ROCm/aiter PR #4741, "Summary": the state scan and the output matmul of the
// KDA block; "Optimizations Applied": the serial state walk split over value
// channels.  The pool row is loaded at the start and the final state written
// back to the same row: ROCm/aiter PR #5754, "Technical Details".)
//
// Only the first two products are on the serial path from one chunk to the
// next, so the CTA is split by role:
//   * 4 state warps keep S (fp32 master copy in registers, warp wr owning key
//     channels 32wr..32wr+31 of S^T), compute U and the update, and publish the
//     chunk's incoming S and its U (fp16) in a two-slot ring;
//   * 4 output warps compute o from the ring one step behind (warp wr: chunk
//     rows 16wr..16wr+15) and store it;
//   * 1 producer warp streams each chunk's intermediates (w, qg, kg, A_qk,
//     gamma and the CTA's u columns) by TMA bulk copies into a three-stage
//     ring, and asks L2 for the chunks further ahead (a bulk L2 prefetch, each
//     of the CTAs of a (sequence, head) taking its share of the shared part).
// Hand-offs use mbarriers (stage full/empty, ring ready/free); the state warps
// synchronise among themselves on a named barrier.  Products are warp-level
// tensor-core MMAs (m16n8k16, fp16 operands, fp32 accumulation); fp16 tiles
// are written with stmatrix (transposing) and read with ldmatrix.

#include "kda_scan_walk.cuh"

namespace kda {
namespace {

// One CTA per (long sequence, head, block of value rows).
template <int NT>
__global__ void __launch_bounds__(scan::kScanThreads, 1) kda_scan_mma(FwdParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int n = p.long_list ? p.long_list[blockIdx.x] : (int)blockIdx.x;
    scan::scan_walk<NT>(p, smem, n, (int)blockIdx.y, (int)blockIdx.z);
}

template <int NT>
cudaError_t launch_scan_nt(const FwdParams& p, cudaStream_t s) {
    using L = scan::ScanSmem<NT>;
    static unsigned configured = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 32 && !(configured & (1u << dev))) {
        e = cudaFuncSetAttribute(kda_scan_mma<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 L::kTotal);
        if (e != cudaSuccess) return e;
        configured |= 1u << dev;
    }
    const int n_seq = p.long_list ? p.n_long : p.N;
    if (n_seq <= 0) return cudaSuccess;
    dim3 grid((unsigned)n_seq, (unsigned)p.H, (unsigned)(kD / L::VS));
    kda_scan_mma<NT><<<grid, scan::kScanThreads, L::kTotal, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

int scan_groups(int N, int H, int num_sms) {
    // 16 value rows per CTA while (sequence, head) pairs are few enough for the
    // finer split to fill the GPU, 32 otherwise.
    const long pairs = (long)N * H;
    return pairs * 8 <= 2L * num_sms ? 1 : 2;
}

cudaError_t launch_scan(const FwdParams& p, int groups, cudaStream_t s) {
    if (p.N <= 0) return cudaSuccess;
    return groups <= 1 ? launch_scan_nt<2>(p, s) : launch_scan_nt<4>(p, s);
}

}  // namespace kda
