// Token-by-token kernel for short sequences (at most kShortMax tokens; empty
// sequences too): two CTAs per (sequence, head), each of 4 warps holding 64
// value rows of the state in fp32 registers.  Warp w of CTA z owns value rows
// 64z + 16w .. 64z + 16w + 15, a half-warp one row at a time (rows
// 64z + 16w + 2j + half), lane l of the half keys 8l..8l+7.  For each token of
// the sequence, in order:
//   S <- S Diag(a),   u = S k^,   S <- S + b (v - u) k^T,   o = S q^
// with q^ = q / |q| / sqrt(K), k^ = k / |k|, a = e^{lb sigmoid(g_raw)} and
// b = sigmoid(beta_raw) formed in the kernel, exactly the recurrence the
// chunked path evaluates in blocks of 64 tokens.
//
// A one-token sequence needs the whole V x K state read and written once per
// head, and nothing else of that size, so this path is bound by state
// bandwidth; the state is accumulated in fp32 whatever the pool's element type
// (ROCm/aiter PR #5249, description of the state-dtype option: decode streams
// the recurrent state per token, the recurrence accumulates in fp32 and the
// pool's element type only sets the bytes moved).  The pool row is read
// (unless the sequence has no initial state) and the final state written back
// to the same row with round-to-nearest-even (ROCm/aiter PR #5754, "Technical
// Details").

#include "kda_device.cuh"
#include "kda_internal.h"

namespace kda {
namespace {

constexpr int D = kD;
constexpr int kDecThreads = 128;  // one thread per key for the per-token vectors
static_assert(kDecThreads == D, "the per-token prep maps threads to keys");

// 8 consecutive state elements at element offset `off` (a multiple of 8, so
// the access is 16- or 32-byte aligned for a 16-byte aligned pool).
__device__ __forceinline__ void load8(const void* base, int dtype, size_t off, float* x) {
    if (dtype == 0) {
        const float4* s = reinterpret_cast<const float4*>(static_cast<const float*>(base) + off);
        const float4 a = s[0], b = s[1];
        x[0] = a.x, x[1] = a.y, x[2] = a.z, x[3] = a.w;
        x[4] = b.x, x[5] = b.y, x[6] = b.z, x[7] = b.w;
        return;
    }
    const uint4 r = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + off);
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if (dtype == 1) {
            x[2 * i] = __uint_as_float(w[i] << 16);
            x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        } else {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
            x[2 * i] = f.x;
            x[2 * i + 1] = f.y;
        }
    }
}

__device__ __forceinline__ void store8(void* base, int dtype, size_t off, const float* x) {
    if (dtype == 0) {
        float4* d = reinterpret_cast<float4*>(static_cast<float*>(base) + off);
        d[0] = make_float4(x[0], x[1], x[2], x[3]);
        d[1] = make_float4(x[4], x[5], x[6], x[7]);
        return;
    }
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        w[i] = (dtype == 1) ? dev::pack_bf162(x[2 * i], x[2 * i + 1])
                            : dev::pack_half2(x[2 * i], x[2 * i + 1]);
    *reinterpret_cast<uint4*>(static_cast<uint16_t*>(base) + off) = make_uint4(w[0], w[1], w[2], w[3]);
}

// Sums of the 8 values x[0..7] over the 16 lanes of each half-warp: a halving
// butterfly leaves the sum of value (lane >> 1) & 7 in lanes 2j and 2j + 1 of
// the half (xor partners stay in the half).
__device__ __forceinline__ float half_sums8(float (&x)[8], int lane) {
#pragma unroll
    for (int w = 4; w >= 1; w >>= 1) {  // lane bit 8, 4, 2
        const bool up = (lane & (2 * w)) != 0;
#pragma unroll
        for (int j = 0; j < w; ++j) {
            const float send = up ? x[j] : x[j + w];
            const float keep = up ? x[j + w] : x[j];
            x[j] = keep + __shfl_xor_sync(0xffffffffu, send, 2 * w);
        }
    }
    return x[0] + __shfl_xor_sync(0xffffffffu, x[0], 1);
}

__global__ void __launch_bounds__(kDecThreads) kda_decode(FwdParams p) {
    __shared__ __align__(16) float s_q[D], s_k[D], s_a[D];  // q^, k^, a of the token
    __shared__ float s_red[2][4], s_beta;

    const int n = p.short_list[blockIdx.x];
    const int h = blockIdx.y;
    const int vb = 64 * blockIdx.z;  // first value row of this CTA
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int hw = lane >> 4, l16 = lane & 15;
    const int k0 = 8 * l16;  // this lane's keys
    const int H = p.H;
    const float lb = p.lower_bound;

    const int tok0 = p.cu[n];
    const int len = p.cu[n + 1] - tok0;
    const bool has_init = p.has_init ? (p.has_init[n] != 0) : (p.st_in != nullptr);
    const int64_t in_slot = p.st_in_idx ? p.st_in_idx[n] : n;
    const int64_t out_slot = p.st_out_idx ? p.st_out_idx[n] : n;
    const size_t in_base = (size_t)in_slot * p.st_in_stride + (size_t)h * D * D;
    const size_t out_base = (size_t)out_slot * p.st_out_stride + (size_t)h * D * D;

    float S[8][8];  // rows vb + 16 warp + 2j + hw, keys k0..k0+7
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int vr = vb + 16 * warp + 2 * j + hw;
        if (has_init) {
            load8(p.st_in, p.st_dtype, in_base + (size_t)vr * D + k0, S[j]);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) S[j][e] = 0.f;
        }
    }

    for (int t = 0; t < len; ++t) {
        const size_t row = ((size_t)(tok0 + t) * H + h) * D;
        // the token's q^, k^ and a, one key per thread
        float qv = 0.f, kv = 0.f;
        if (tid == 0)
            s_beta = __fdividef(
                1.f, 1.f + __expf(-load_raw(p.beta_raw, p.raw_bf16, (size_t)(tok0 + t) * H + h)));
        {
            qv = __bfloat162float(p.q[row + tid]);
            kv = __bfloat162float(p.k[row + tid]);
            const float gv = load_raw(p.g_raw, p.raw_bf16, row + tid);
            s_a[tid] = __expf(lb * __fdividef(1.f, 1.f + __expf(-gv)));
            float sq = qv * qv, sk = kv * kv;
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) {
                sq += __shfl_xor_sync(0xffffffffu, sq, o);
                sk += __shfl_xor_sync(0xffffffffu, sk, o);
            }
            if (lane == 0) {
                s_red[0][warp] = sq;
                s_red[1][warp] = sk;
            }
        }
        __syncthreads();
        {
            const float sq = s_red[0][0] + s_red[0][1] + s_red[0][2] + s_red[0][3];
            const float sk = s_red[1][0] + s_red[1][1] + s_red[1][2] + s_red[1][3];
            s_q[tid] = qv * rsqrtf(sq + 1e-6f) * 0.08838834764831845f;  // 1/sqrt(128)
            s_k[tid] = kv * rsqrtf(sk + 1e-6f);
        }
        __syncthreads();

        float a8[8], k8[8], q8[8], vv[8];
        *reinterpret_cast<float4*>(a8) = *reinterpret_cast<const float4*>(s_a + k0);
        *reinterpret_cast<float4*>(a8 + 4) = *reinterpret_cast<const float4*>(s_a + k0 + 4);
        *reinterpret_cast<float4*>(k8) = *reinterpret_cast<const float4*>(s_k + k0);
        *reinterpret_cast<float4*>(k8 + 4) = *reinterpret_cast<const float4*>(s_k + k0 + 4);
        *reinterpret_cast<float4*>(q8) = *reinterpret_cast<const float4*>(s_q + k0);
        *reinterpret_cast<float4*>(q8 + 4) = *reinterpret_cast<const float4*>(s_q + k0 + 4);
        const float b = s_beta;
#pragma unroll
        for (int j = 0; j < 8; ++j) vv[j] = __bfloat162float(p.v[row + vb + 16 * warp + 2 * j + hw]);

        // u = S Diag(a) k^ for the 8 rows, reduced over the half-warp
        float x[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float u = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                S[j][e] *= a8[e];
                u = fmaf(S[j][e], k8[e], u);
            }
            x[j] = u;
        }
        const float uj = half_sums8(x, lane);  // u of row (lane >> 1) & 7
        // S += b (v - u) k^T, then o = S q^
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float u = __shfl_sync(0xffffffffu, uj, 16 * hw + 2 * j);
            const float d = b * (vv[j] - u);
            float o = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                S[j][e] = fmaf(d, k8[e], S[j][e]);
                o = fmaf(S[j][e], q8[e], o);
            }
            x[j] = o;
        }
        const float oj = half_sums8(x, lane);  // o of row (lane >> 1) & 7
        if ((lane & 1) == 0)
            p.out[row + vb + 16 * warp + 2 * ((l16 >> 1) & 7) + hw] = __float2bfloat16_rn(oj);
        __syncthreads();  // the next token rewrites the shared vectors
    }

#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int vr = vb + 16 * warp + 2 * j + hw;
        store8(p.st_out, p.st_dtype, out_base + (size_t)vr * D + k0, S[j]);
    }
}

}  // namespace

cudaError_t launch_decode(const FwdParams& p, cudaStream_t s) {
    if (p.n_short <= 0 || !p.short_list) return cudaSuccess;
    dim3 grid((unsigned)p.n_short, (unsigned)p.H, 2);
    kda_decode<<<grid, kDecThreads, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace kda
