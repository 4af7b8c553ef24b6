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

// ---- segmented scan --------------------------------------------------------
// For a batch with few (sequence, head) pairs the walks above leave most SMs
// idle for the whole length of the sequence.  The segmented scan cuts each long
// sequence into P segments of L chunks; with M_c the chunk's state transition
// and the recurrence S <- S M_c + N_c, a segment maps its start state S to
// S Phi + N (Phi = product of its M_c, N = its state from a zero start):
//   pass A  per segment but the last, in parallel: N from a zero state, and Phi
//           as the walk of the K identity rows with u = 0;
//   combine per (pair, 16 value rows), in order: S_start(s + 1) = S_start(s) Phi_s + N_s
//           (fp32), S_start(0) the pool state;
//   pass B  per segment, in parallel: the walk from S_start(s), writing the
//           outputs and, for the last segment, the pool.
// (ROCm/aiter PR #4741, "Optimizations Applied": the sequence-parallel split of
// the state walk into segments composed afterwards; the composition through the
// segment transitions is this build's.)
constexpr size_t kPlane = kSegPlaneFloats;

__device__ __forceinline__ float* seg_planes(const FwdParams& p, int P, int pair) {
    return p.seg + (size_t)pair * 3 * (P - 1) * kPlane;  // Phi_0.., N_0.., S_start(1)..
}

__device__ __forceinline__ void seg_pair(const FwdParams& p, int pair, int L, int& n, int& h, int& Pn) {
    const int sq = pair / p.H;
    h = pair % p.H;
    n = p.long_list ? p.long_list[sq] : sq;
    Pn = (p.seq_off[n + 1] - p.seq_off[n] + L - 1) / L;
}

template <bool PASS_B>
__global__ void __launch_bounds__(scan::kScanThreads, 1) kda_scan_seg(FwdParams p, int P, int L) {
    extern __shared__ __align__(1024) uint8_t smem[];
    int u = blockIdx.x;
    const int z = u % (kD / 16);
    u /= kD / 16;
    int kind = 0;
    if (!PASS_B) {
        kind = u & 1;
        u >>= 1;
    }
    const int segs = PASS_B ? P : P - 1;
    const int sg = u % segs, pair = u / segs;
    int n, h, Pn;
    seg_pair(p, pair, L, n, h, Pn);
    float* base = seg_planes(p, P, pair);
    scan::WalkRange R;
    R.first = sg * L;
    R.count = L;
    if (!PASS_B) {
        if (sg >= Pn - 1) return;  // the last segment needs no pass A
        R.init = kind ? 2 : 1;     // Phi from identity rows, N from zero
        R.zero_u = kind == 1;
        R.outputs = false;
        R.final_buf = base + (size_t)(kind ? sg : (P - 1) + sg) * kPlane;
    } else {
        if (sg >= Pn) return;
        if (sg > 0) {
            R.init = 3;
            R.init_buf = base + (size_t)(2 * (P - 1) + sg - 1) * kPlane;
        }
        R.final_state = sg == Pn - 1;  // the last segment writes the pool
        if (sg == Pn - 1) R.count = -1;
    }
    scan::scan_walk<2>(p, smem, n, h, z, R);
}

// S_start(s + 1) = S_start(s) Phi_s + N_s for value rows 16 blockIdx.y .. of pair
// blockIdx.x; thread t: row t / 16, keys 8 (t % 16) .. + 7.
constexpr int kCombThreads = 256;
constexpr int kCombSmem = (128 * 128 + 16 * 129) * 4;
__global__ void __launch_bounds__(kCombThreads) kda_scan_combine(FwdParams p, int P, int L) {
    extern __shared__ float csm[];
    float* phi = csm;               // [128][128]
    float* S = csm + 128 * 128;     // [16][129]
    const int pair = blockIdx.x, z = blockIdx.y, t = threadIdx.x;
    int n, h, Pn;
    seg_pair(p, pair, L, n, h, Pn);
    if (Pn < 2) return;
    const int r = t >> 4, k0 = (t & 15) * 8, v = 16 * z + r;
    // S_start(0): the pool row (zero without an initial state or for a slot outside the pool)
    bool init = p.has_init ? (p.has_init[n] != 0) : (p.st_in != nullptr);
    const int64_t slot = p.st_in_idx ? p.st_in_idx[n] : n;
    if (p.num_slots > 0 && (slot < 0 || slot >= p.num_slots)) init = false;
    const size_t row = (size_t)slot * p.st_in_stride + ((size_t)h * kD + v) * kD;
#pragma unroll
    for (int e = 0; e < 8; ++e) S[r * 129 + k0 + e] = init ? scan::load_state(p.st_in, p.st_dtype, row + k0 + e) : 0.f;
    float* base = seg_planes(p, P, pair);
    for (int sg = 0; sg < Pn - 1; ++sg) {
        const float4* ph = reinterpret_cast<const float4*>(base + (size_t)sg * kPlane);
        for (int i = t; i < 128 * 128 / 4; i += kCombThreads) reinterpret_cast<float4*>(phi)[i] = ph[i];
        const float* nb = base + (size_t)(P - 1 + sg) * kPlane + (size_t)v * kD + k0;
        float acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = nb[e];
        __syncthreads();
        for (int j = 0; j < 128; ++j) {
            const float a = S[r * 129 + j];
            const float4 p0 = *reinterpret_cast<const float4*>(phi + j * 128 + k0);
            const float4 p1 = *reinterpret_cast<const float4*>(phi + j * 128 + k0 + 4);
            acc[0] = fmaf(a, p0.x, acc[0]);
            acc[1] = fmaf(a, p0.y, acc[1]);
            acc[2] = fmaf(a, p0.z, acc[2]);
            acc[3] = fmaf(a, p0.w, acc[3]);
            acc[4] = fmaf(a, p1.x, acc[4]);
            acc[5] = fmaf(a, p1.y, acc[5]);
            acc[6] = fmaf(a, p1.z, acc[6]);
            acc[7] = fmaf(a, p1.w, acc[7]);
        }
        __syncthreads();  // S and phi are read
        float* out = base + (size_t)(2 * (P - 1) + sg) * kPlane + (size_t)v * kD + k0;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            S[r * 129 + k0 + e] = acc[e];
            out[e] = acc[e];
        }
    }
}

cudaError_t launch_scan_segmented(const FwdParams& p, int P, int L, cudaStream_t s) {
    using Lyt = scan::ScanSmem<2>;
    static unsigned configured = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 32 && !(configured & (1u << dev))) {
        e = cudaFuncSetAttribute(kda_scan_seg<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Lyt::kTotal);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(kda_scan_seg<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     Lyt::kTotal);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(kda_scan_combine, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kCombSmem);
        if (e != cudaSuccess) return e;
        configured |= 1u << dev;
    }
    const int pairs = (p.long_list ? p.n_long : p.N) * p.H;
    const int walks = kD / 16;
    kda_scan_seg<false><<<pairs * (P - 1) * 2 * walks, scan::kScanThreads, Lyt::kTotal, s>>>(p, P, L);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    kda_scan_combine<<<dim3(pairs, walks), kCombThreads, kCombSmem, s>>>(p, P, L);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    kda_scan_seg<true><<<pairs * P * walks, scan::kScanThreads, Lyt::kTotal, s>>>(p, P, L);
    return cudaGetLastError();
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

int scan_segments(const FwdParams& p, int num_sms, int* L) {
    const int n_long = p.long_list ? p.n_long : p.N;
    const int pairs = n_long * p.H;
    if (!p.seg || n_long <= 0 || pairs > 4 || p.max_long_chunks < 12) return 0;
    // pass A runs 16 walks per pair and segment boundary: one wave of the GPU,
    // and three state planes per boundary in the workspace
    int bounds = num_sms / (16 * pairs);
    if (bounds * pairs * 3 > kSegPlanes) bounds = kSegPlanes / (3 * pairs);
    int P = bounds + 1;
    if (P > p.max_long_chunks / 4) P = p.max_long_chunks / 4;  // segments of 4 chunks at least
    if (P < 3) return 0;
    *L = (p.max_long_chunks + P - 1) / P;
    return (p.max_long_chunks + *L - 1) / *L;
}

cudaError_t launch_scan(const FwdParams& p, int groups, cudaStream_t s) {
    if (p.N <= 0) return cudaSuccess;
    int L = 0;
    const int P = scan_segments(p, num_sms(), &L);
    if (P > 0) return launch_scan_segmented(p, P, L, s);
    return groups <= 1 ? launch_scan_nt<2>(p, s) : launch_scan_nt<4>(p, s);
}

}  // namespace kda
