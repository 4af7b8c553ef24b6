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
//
// This role split serves 16 value rows per CTA, for batches with few (sequence,
// head) pairs.  Batches with more pairs take 64 or 128 value rows per CTA in the
// values-partitioned walk of kda_scan_vp.cuh, where each warp owns its value
// rows for all keys and no state crosses between warps.

#include "kda_scan_vp.cuh"

namespace kda {
namespace {

// One CTA per (long sequence, head, block of value rows), the sequence the
// slowest-varying index: CTAs start in launch order, so the walks of the list's
// first sequences (the host orders it longest first) start in the first wave.
template <int NT>
__global__ void __launch_bounds__(scan::kScanThreads, 1)
kda_scan_mma(FwdParams p) {
    // a token-by-token grid launched after this one may start now: it takes the
    // SMs the walks leave free (it waits for this grid before it completes)
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (call_aborted(p)) return;
    extern __shared__ __align__(1024) uint8_t smem[];
    constexpr int kGroups = kD / scan::ScanSmem<NT>::VS;
    const int b = (int)blockIdx.x;
    const int z = b % kGroups, h = (b / kGroups) % p.H, sq = b / (kGroups * p.H);
    const int n = p.long_list ? p.long_list[sq] : sq;
    scan::scan_walk<NT>(p, smem, n, h, z);
}

// ---- segmented scan --------------------------------------------------------
// For a batch with few (sequence, head) pairs the walks above leave most SMs
// idle for the whole length of the sequence.  The segmented scan cuts each long
// sequence into P segments of L chunks; with M_c the chunk's state transition
// and the recurrence S <- S M_c + N_c, a segment maps its start state S to
// S Phi + N (Phi = product of its M_c, N = its state from a zero start):
//   pass A  per segment but the last, in parallel: N from a zero state, and Phi
//           as the walk of the K identity rows with u = 0;
//   combine per (pair, 4 value rows), in order: S_start(s + 1) = S_start(s) Phi_s + N_s
//           (fp32), S_start(0) the pool state;
//   pass B  per segment, in parallel: the walk from S_start(s), writing the
//           outputs and, for the last segment, the pool.
// (ROCm/aiter PR #4741, "Optimizations Applied": the sequence-parallel split of
// the state walk into segments composed afterwards; the page does not give the
// composition, which follows from each chunk's affine map of the state.)
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
    if (call_aborted(p)) return;
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

// S_start(s + 1) = S_start(s) Phi_s + N_s for kCombRows value rows (blockIdx.y) of
// pair blockIdx.x, one key channel k per thread: acc_r += S_start[r][j] Phi_s[j][k]
// over j, the rows of S_start read as one broadcast float4 per j and Phi_s as one
// coalesced row.  The transitions arrive by bulk copies into two shared buffers,
// the next one copied while the current step computes (they depend only on pass A).
constexpr int kCombRows = 4;
constexpr int kCombThreads = kD;
constexpr uint32_t kPlaneBytes = (uint32_t)(kPlane * sizeof(float));
constexpr int kCombSmem = (int)(2 * kPlaneBytes + kD * kCombRows * sizeof(float) + 2 * sizeof(uint64_t));
static_assert(kCombRows == 4, "the rows of S_start are read as one float4");

__global__ void __launch_bounds__(kCombThreads) kda_scan_combine(FwdParams p, int P, int L) {
    using namespace dev;
    if (call_aborted(p)) return;
    extern __shared__ __align__(128) uint8_t csm[];
    float* phi = reinterpret_cast<float*>(csm);                        // [2][K][K]
    float* st = phi + 2 * kPlane;                                      // [K][kCombRows]: S_start^T
    uint64_t* bar = reinterpret_cast<uint64_t*>(st + kD * kCombRows);  // one per buffer
    const int pair = blockIdx.x, v0 = kCombRows * (int)blockIdx.y, k = threadIdx.x;
    int n, h, Pn;
    seg_pair(p, pair, L, n, h, Pn);
    const int steps = Pn - 1;
    if (steps < 1) return;
    float* base = seg_planes(p, P, pair);
    if (k == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        fence_mbar_init();
        for (int b = 0; b < 2 && b < steps; ++b) {
            mbar_arrive_expect_tx(&bar[b], kPlaneBytes);
            bulk_g2s(phi + b * kPlane, base + (size_t)b * kPlane, kPlaneBytes, &bar[b]);
        }
    }
    // S_start(0): the pool rows (zero without an initial state or for a slot outside the pool)
    bool init = p.has_init ? (p.has_init[n] != 0) : (p.st_in != nullptr);
    const int64_t slot = p.st_in_idx ? p.st_in_idx[n] : n;
    if (p.num_slots > 0 && (slot < 0 || slot >= p.num_slots)) init = false;
    float s0[kCombRows];
#pragma unroll
    for (int r = 0; r < kCombRows; ++r)
        s0[r] = init ? scan::load_state(p.st_in, p.st_dtype,
                                        (size_t)slot * p.st_in_stride +
                                            ((size_t)h * kD + v0 + r) * kD + k)
                     : 0.f;
    *reinterpret_cast<float4*>(st + k * kCombRows) = make_float4(s0[0], s0[1], s0[2], s0[3]);
    __syncthreads();  // barriers initialised, S_start(0) in place

    for (int sg = 0; sg < steps; ++sg) {
        const int b = sg & 1;
        const uint32_t par = (uint32_t)(sg >> 1) & 1;
        const float* nb = base + (size_t)(P - 1 + sg) * kPlane + (size_t)v0 * kD + k;
        float acc[kCombRows];
#pragma unroll
        for (int r = 0; r < kCombRows; ++r) acc[r] = nb[(size_t)r * kD];
        if (!__syncthreads_and(mbar_wait(&bar[b], par))) {
            // report, and let this CTA's copies in flight land before it leaves
            if (k == 0) {
                if (p.status) atomicOr(p.status, 1);
                mbar_wait(&bar[b], par);
                if (sg + 1 < steps) mbar_wait(&bar[b ^ 1], (uint32_t)((sg + 1) >> 1) & 1);
            }
            return;
        }
        const float* ph = phi + b * kPlane;
#pragma unroll 8
        for (int j = 0; j < kD; ++j) {
            const float4 s = *reinterpret_cast<const float4*>(st + j * kCombRows);
            const float f = ph[j * kD + k];
            acc[0] = fmaf(s.x, f, acc[0]);
            acc[1] = fmaf(s.y, f, acc[1]);
            acc[2] = fmaf(s.z, f, acc[2]);
            acc[3] = fmaf(s.w, f, acc[3]);
        }
        __syncthreads();  // every thread is done with st and with buffer b
        if (k == 0 && sg + 2 < steps) {
            fence_proxy_async();
            mbar_arrive_expect_tx(&bar[b], kPlaneBytes);
            bulk_g2s(phi + b * kPlane, base + (size_t)(sg + 2) * kPlane, kPlaneBytes, &bar[b]);
        }
        float* out = base + (size_t)(2 * (P - 1) + sg) * kPlane + (size_t)v0 * kD + k;
#pragma unroll
        for (int r = 0; r < kCombRows; ++r) out[(size_t)r * kD] = acc[r];
        *reinterpret_cast<float4*>(st + k * kCombRows) = make_float4(acc[0], acc[1], acc[2], acc[3]);
        __syncthreads();  // S_start(sg + 1) in place
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
    kda_scan_combine<<<dim3(pairs, kD / kCombRows), kCombThreads, kCombSmem, s>>>(p, P, L);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    kda_scan_seg<true><<<pairs * P * walks, scan::kScanThreads, Lyt::kTotal, s>>>(p, P, L);
    return cudaGetLastError();
}

// Kernel launch, with programmatic stream serialization when `pdl` is set (the
// grid may then start beside the kernel launched before it and waits for that
// kernel's completion inside the walks, before it reads the intermediates).
template <typename... Params, typename... Args>
cudaError_t launch_maybe_pdl(void (*kernel)(Params...), unsigned grid, unsigned block, size_t smem,
                             cudaStream_t s, bool pdl, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <int NT>
cudaError_t launch_scan_nt(const FwdParams& p, cudaStream_t s, bool pdl) {
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
    const long blocks = (long)n_seq * p.H * (kD / L::VS);
    return launch_maybe_pdl(kda_scan_mma<NT>, (unsigned)blocks, scan::kScanThreads, L::kTotal, s, pdl,
                            p);
}

// One CTA per (long sequence, head, 16 NW value rows), sequence-major like
// kda_scan_mma: the values-partitioned walk of kda_scan_vp.cuh.
template <int NW>
__global__ void __launch_bounds__(scan::vp_threads<NW>(), 1)
kda_scan_vp(FwdParams p, const __grid_constant__ CUtensorMap out_map, int has_out_map) {
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (call_aborted(p)) return;
    extern __shared__ __align__(1024) uint8_t smem[];
    constexpr int kGroups = kD / scan::ScanSmemVP<NW>::VS;
    const int b = (int)blockIdx.x;
    const int z = b % kGroups, h = (b / kGroups) % p.H, sq = b / (kGroups * p.H);
    const int n = p.long_list ? p.long_list[sq] : sq;
    scan::scan_walk_vp<NW>(p, smem, n, h, z, has_out_map ? &out_map : nullptr);
}

template <int NW>
cudaError_t launch_scan_vp(const FwdParams& p, cudaStream_t s, bool pdl) {
    using L = scan::ScanSmemVP<NW>;
    static unsigned configured = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 32 && !(configured & (1u << dev))) {
        e = cudaFuncSetAttribute(kda_scan_vp<NW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 L::kTotal);
        if (e != cudaSuccess) return e;
        configured |= 1u << dev;
    }
    const int n_seq = p.long_list ? p.n_long : p.N;
    if (n_seq <= 0) return cudaSuccess;
    const long blocks = (long)n_seq * p.H * (kD / L::VS);
    CUtensorMap out_map = {};
    const int has_out_map = make_out_map(&out_map, p, 16, kC) ? 1 : 0;
    return launch_maybe_pdl(kda_scan_vp<NW>, (unsigned)blocks, scan::vp_threads<NW>(), L::kTotal, s,
                            pdl, p, out_map, has_out_map);
}

// Diagnostic: one thread waits, with the bounded waits every kernel uses, for
// something that never happens (kind 0: an mbarrier phase nothing arrives on;
// kind 1: a ready flag nothing sets), so that the give-up path, the status word
// and the context's use afterwards can be tested without faulting or hanging.
__global__ void kda_wait_probe(int kind, int* status, const int* flag) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        dev::mbar_init(&bar, 1);
        dev::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x != 0) return;
    const bool ok = kind == 0 ? dev::mbar_wait(&bar, 0) : scan::wait_ready_run(flag, 1, 1) > 0;
    if (!ok) atomicOr(status, 1);
}

}  // namespace

cudaError_t launch_wait_probe(int kind, int* status, const int* flag, cudaStream_t s) {
    kda_wait_probe<<<1, 32, 0, s>>>(kind, status, flag);
    return cudaGetLastError();
}

int scan_groups(int N, int H, int num_sms, int beside_pairs) {
    // 16 value rows per CTA while (sequence, head) pairs are few enough for the
    // finer split to fill the GPU, else 64 or 128: the head-wide chunk operands
    // each CTA reads then serve four or eight times as many value rows (64 rows
    // against 32: mixed batch 70.3 against 76.6 us, varlen batch 620 against
    // 699 us).  Walks of 64 rows while they fit one wave; walks of 128 rows
    // past that, and also when a token-by-token kernel with at least a wave of
    // (sequence, head) pairs runs beside the scan: half as many scan CTAs leave
    // it the other SMs (mixed batch of 4 x 2048 prefill tokens and 512 decode
    // tokens: 198.5 against 203.4 us per call).
    const long pairs = (long)N * H;
    if (pairs * 8 <= 2L * num_sms) return 1;
    return pairs * 2 <= num_sms && beside_pairs < num_sms ? 4 : 8;
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

cudaError_t launch_scan(const FwdParams& p, int groups, cudaStream_t s, bool after_intra) {
    if (p.N <= 0) return cudaSuccess;
    int L = 0;
    const int P = scan_segments(p, num_sms(), &L);
    if (P > 0) return launch_scan_segmented(p, P, L, s);
    if (groups <= 1) return launch_scan_nt<2>(p, s, after_intra);
    return groups == 4 ? launch_scan_vp<4>(p, s, after_intra) : launch_scan_vp<8>(p, s, after_intra);
}

}  // namespace kda
