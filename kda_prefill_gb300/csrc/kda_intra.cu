// CUDA kernels of the chunkwise KDA forward (sm_103a).
//
// Chunkwise form of the gated delta rule used here (derived from the token
// recurrence S_t = S_{t-1} Diag(e^{g_t}) (I - b_t k_t k_t^T) + b_t v_t k_t^T,
// o_t = S_t q_t).  Inside a chunk of C tokens with in-chunk cumulative
// log-decay G_i = g_1 + ... + g_i (per channel) and incoming state S_0:
//
//   A_kk[i][j] = b_i sum_c k_ic k_jc e^{G_ic - G_jc}      (j < i)
//   A_qk[i][j] =     sum_c q_ic k_jc e^{G_ic - G_jc}      (j <= i)
//   T  = (I + A_kk)^{-1}                                   (unit lower triangular)
//   w  = T (b k e^{G}),   u = T (b v)
//   U  = u - w S_0^T                                       (the chunk's new values)
//   o  = (q e^{G}) S_0^T + A_qk U
//   S_C = S_0 Diag(e^{G_C}) + U^T (k e^{G_C - G})
//
// The steps follow ROCm/aiter PR #4741 ("Summary": q/k L2 norm, gate cumsum,
// beta sigmoid, the two intra-chunk kernels, the w/u recompute, the state scan
// and the output matmul; "Optimizations Applied": sequence-parallel split into
// a chunk-parallel prep and a serial scan, zero padding as an exact no-op, and
// tiles built so that no factor exceeds 1: here every decay factor is the
// exponential of a non-positive difference G_i - G_j with j <= i).
//
// This file holds the intra-chunk kernels: the tensor-core kernel used for
// lower_bound >= -5 (kda_intra_tc) and an exact SIMT fp32 kernel for stronger
// decay bounds (kda_intra_exact).

#include "kda_device.cuh"
#include "kda_internal.h"

namespace kda {
namespace {

constexpr int C = kC;
constexpr int D = kD;
constexpr int P = D + 1;   // padded smem row pitch (floats) against bank conflicts
constexpr int PA = C + 1;  // pitch of C x C tiles
constexpr int kIntraThreads = 256;

__device__ __forceinline__ float sigmoidf_(float x) { return 1.0f / (1.0f + expf(-x)); }

constexpr size_t kIntraSmem =
    sizeof(float) * (4 * C * P + 3 * C * PA + 3 * C);

// Exact fp32 variant used when lower_bound < -5: one CTA per (chunk, head);
// prep (L2 norm, gate, cumsum, beta) fused with the intra-chunk tiles, every
// decay factor evaluated directly as e^{G_i - G_j} <= 1, the triangular solve
// and the w/u recompute.  Slow but valid for any decay strength.
__global__ void __launch_bounds__(kIntraThreads)
kda_intra_exact(FwdParams p) {
    if (call_aborted(p)) return;
    extern __shared__ float sm[];
    float* sQ = sm;             // [C][P] q, then q^
    float* sK = sQ + C * P;     // [C][P] k, then k^
    float* sG = sK + C * P;     // [C][P] g, then G (inclusive cumsum)
    float* sV = sG + C * P;     // [C][P] v, then b v
    float* sAk = sV + C * P;    // [C][PA]
    float* sAq = sAk + C * PA;  // [C][PA]
    float* sT = sAq + C * PA;   // [C][PA]
    float* sB = sT + C * PA;    // [C] beta
    float* sRq = sB + C;        // [C] 1/|q| / sqrt(K)
    float* sRk = sRq + C;       // [C] 1/|k|

    const int j = blockIdx.x;
    const int h = blockIdx.y;
    const int tid = threadIdx.x;
    const int seq = p.chunk_seq[j];
    const int tok0 = p.chunk_tok[j];
    const int len = min(C, p.cu[seq + 1] - tok0);

    for (int e = tid; e < C * D; e += kIntraThreads) {
        const int r = e / D, c = e % D;
        float qv = 0.f, kv = 0.f, vv = 0.f, gv = 0.f;
        if (r < len) {
            const size_t off = ((size_t)(tok0 + r) * p.H + h) * D + c;
            qv = __bfloat162float(p.q[off]);
            kv = __bfloat162float(p.k[off]);
            vv = __bfloat162float(p.v[off]);
            gv = p.lower_bound * sigmoidf_(load_raw(p.g_raw, p.raw_bf16, off));
        }
        sQ[r * P + c] = qv;
        sK[r * P + c] = kv;
        sV[r * P + c] = vv;
        sG[r * P + c] = gv;
    }
    for (int r = tid; r < C; r += kIntraThreads)
        sB[r] = (r < len) ? sigmoidf_(load_raw(p.beta_raw, p.raw_bf16, (size_t)(tok0 + r) * p.H + h))
                          : 0.f;
    __syncthreads();

    const int warp = tid / 32, lane = tid % 32;
    for (int r = warp; r < C; r += kIntraThreads / 32) {
        float sq = 0.f, sk = 0.f;
        for (int c = lane; c < D; c += 32) {
            sq += sQ[r * P + c] * sQ[r * P + c];
            sk += sK[r * P + c] * sK[r * P + c];
        }
        for (int o = 16; o > 0; o >>= 1) {
            sq += __shfl_xor_sync(0xffffffffu, sq, o);
            sk += __shfl_xor_sync(0xffffffffu, sk, o);
        }
        if (lane == 0) {
            sRq[r] = 1.0f / sqrtf(sq + 1e-6f) / sqrtf((float)D);
            sRk[r] = 1.0f / sqrtf(sk + 1e-6f);
        }
    }
    __syncthreads();
    for (int e = tid; e < C * D; e += kIntraThreads) {
        const int r = e / D, c = e % D;
        sQ[r * P + c] *= sRq[r];
        sK[r * P + c] *= sRk[r];
    }
    if (tid < D) {
        float acc = 0.f;
        for (int r = 0; r < C; ++r) {
            acc += sG[r * P + tid];
            sG[r * P + tid] = acc;
        }
    }
    __syncthreads();

    // Decay-weighted tiles; every factor is e^{G_i - G_j} <= 1 (j <= i).
    for (int e = tid; e < C * C; e += kIntraThreads) {
        const int i = e / C, jj = e % C;
        float ak = 0.f, aq = 0.f;
        if (jj <= i) {
            for (int c = 0; c < D; ++c) {
                const float f = expf(sG[i * P + c] - sG[jj * P + c]) * sK[jj * P + c];
                ak += sK[i * P + c] * f;
                aq += sQ[i * P + c] * f;
            }
        }
        sAk[i * PA + jj] = (jj < i) ? sB[i] * ak : 0.f;
        sAq[i * PA + jj] = aq;
    }
    __syncthreads();

    // T = (I + A_kk)^{-1} by forward substitution: T[i,:] = e_i - sum_{j<i} A[i,j] T[j,:]
    for (int i = 0; i < C; ++i) {
        if (tid < C) {
            const int col = tid;
            float acc = (col == i) ? 1.f : 0.f;
            for (int jj = 0; jj < i; ++jj) acc -= sAk[i * PA + jj] * sT[jj * PA + col];
            sT[i * PA + col] = (col <= i) ? acc : 0.f;
        }
        __syncthreads();
    }

    const size_t ch = (size_t)j * p.H + h;
    uint8_t* blk = p.ws + ch * kWsBytes;
    float* ggam = reinterpret_cast<float*>(blk + kWsGammaOff);

    for (int e = tid; e < C * D; e += kIntraThreads) {
        const int r = e / D, c = e % D;
        const float G = sG[r * P + c];
        const float GC = sG[(C - 1) * P + c];
        const uint32_t o = dev::sw128_off(r, c, C);
        *reinterpret_cast<__half*>(blk + kWsQGOff + o) = __float2half_rn(sQ[r * P + c] * expf(G));
        *reinterpret_cast<__half*>(blk + kWsKGOff + o) = __float2half_rn(sK[r * P + c] * expf(GC - G));
    }
    if (tid < D) ggam[tid] = expf(sG[(C - 1) * P + tid]);
    for (int e = tid; e < C * C; e += kIntraThreads) {
        const int i = e / C, jj = e % C;
        *reinterpret_cast<__half*>(blk + kWsAqkOff + dev::sw64_off(i, jj)) =
            __float2half_rn(sAq[i * PA + jj]);
    }
    __syncthreads();
    // reuse sQ for b k^ e^G and sV for b v
    for (int e = tid; e < C * D; e += kIntraThreads) {
        const int r = e / D, c = e % D;
        sQ[r * P + c] = sB[r] * sK[r * P + c] * expf(sG[r * P + c]);
        sV[r * P + c] = sB[r] * sV[r * P + c];
    }
    __syncthreads();
    for (int e = tid; e < C * D; e += kIntraThreads) {
        const int i = e / D, c = e % D;
        float aw = 0.f, au = 0.f;
        for (int jj = 0; jj <= i; ++jj) {
            const float t = sT[i * PA + jj];
            aw += t * sQ[jj * P + c];
            au += t * sV[jj * P + c];
        }
        *reinterpret_cast<__half*>(blk + kWsWOff + dev::sw128_off(i, c, C)) = __float2half_rn(aw);
        *reinterpret_cast<__half*>(blk + kWsUOff + (c / 16) * kWsUSliceBytes + (i * 16 + c % 16) * 2) =
            __float2half_rn(au);
    }
}

}  // namespace

cudaError_t launch_intra_exact(const FwdParams& p, cudaStream_t s) {
    if (p.n_chunks <= 0) return cudaSuccess;
    static unsigned configured = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 32 && !(configured & (1u << dev))) {
        e = cudaFuncSetAttribute(kda_intra_exact, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kIntraSmem);
        if (e != cudaSuccess) return e;
        configured |= 1u << dev;
    }
    dim3 grid((unsigned)p.n_chunks, (unsigned)p.H);
    kda_intra_exact<<<grid, kIntraThreads, kIntraSmem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace kda
