// State scan of the chunkwise KDA forward: one CTA per (sequence, head, group
// of 16*NG value rows of the state), walking the sequence's chunks in order.
//
// Per chunk, with the incoming state S (V rows x K, fp32 in registers):
//   U = u - w S^T                 (C x Vs)   new values of the chunk
//   o = qg S^T + A_qk U           (C x Vs)   written to `out`
//   S = S Diag(gamma) + U^T kg    (Vs x K)
// (ROCm/aiter PR #4741, "Summary": the state scan and the output matmul of the
// KDA block; "Optimizations Applied": the serial state walk split over value
// channels.  The pool row is loaded at the start and the final state written
// back to the same row: ROCm/aiter PR #5754, "Technical Details".)
//
// The products are warp-level tensor-core MMAs (m16n8k16, fp16 operands, fp32
// accumulation).  They are tiny (M = 64, N = 16 per group) and sit on the serial
// critical path, so operands stay in registers / shared memory between the two
// dependent products of a chunk.  The chunk's intermediates (w, qg, kg, A_qk,
// gamma and the group's u columns) arrive by TMA bulk copies into a
// double-buffered shared-memory stage, one chunk ahead.
//
// Warp layout: 4 warps per group of 16 value rows.  Warp wr of a group owns
// rows 16*wr.. of U and o, and key channels 32*wr.. of S^T (its fp32 master
// copy lives in that warp's registers).  One extra warp only issues the TMA
// copies (full/empty mbarrier pair per stage), so no compute warp spends time
// issuing copies on the serial path.

#include "kda_device.cuh"
#include "kda_internal.h"

namespace kda {
namespace {

using namespace dev;

constexpr int C = kC;
constexpr int D = kD;

template <int NG>
struct ScanSmem {
    static constexpr int kShared = kWsSharedBytes;                   // w, qg, kg, aqk, gamma
    static constexpr int kSharedPad = (kShared + 1023) / 1024 * 1024;
    static constexpr int kU = NG * kWsUSliceBytes;                   // NG u slices
    static constexpr int kStage = kSharedPad + (kU + 1023) / 1024 * 1024;
    static constexpr int kS16 = 2 * kStage;                          // NG x [16][128] fp16
    static constexpr int kUt = kS16 + NG * 4096;                     // NG x [16][64] fp16
    static constexpr int kBar = kUt + NG * 2048;                     // full[2], empty[2]
    static constexpr int kTotal = kBar + 64;
};

__device__ __forceinline__ float load_state(const void* base, int dtype, size_t off) {
    if (dtype == 0) return static_cast<const float*>(base)[off];
    if (dtype == 1) return __bfloat162float(static_cast<const __nv_bfloat16*>(base)[off]);
    return __half2float(static_cast<const __half*>(base)[off]);
}

__device__ __forceinline__ void store_state(void* base, int dtype, size_t off, float x) {
    if (dtype == 0) {
        static_cast<float*>(base)[off] = x;
    } else if (dtype == 1) {
        static_cast<__nv_bfloat16*>(base)[off] = __float2bfloat16_rn(x);
    } else {
        static_cast<__half*>(base)[off] = __float2half_rn(x);
    }
}

template <int NG>
__global__ void __launch_bounds__(128 * NG + 32, 1) kda_scan_mma(FwdParams p) {
    using L = ScanSmem<NG>;
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);

    const int n = blockIdx.x;
    const int h = blockIdx.y;
    const int vs0 = blockIdx.z * NG;  // first 16-row value slice of this CTA
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int gi = warp >> 2;   // group
    const int wr = warp & 3;    // row block / key block within the group
    const int g = lane >> 2, tq = lane & 3;
    const int mi = lane >> 3, rr = lane & 7;  // ldmatrix addressing

    const int tok0 = p.cu[n];
    const int len = p.cu[n + 1] - tok0;
    const int c0 = p.seq_off[n];
    const int nch = p.seq_off[n + 1] - c0;

    const uint32_t sm_base = smem_u32(smem);
    // barrier among the compute warps only (id 1; id 0 is __syncthreads)
    auto consumer_sync = [&]() {
        asm volatile("bar.sync 1, %0;" ::"r"(128 * NG) : "memory");
    };
    // same barrier, returning whether any compute thread passed `flag` set
    auto consumer_sync_or = [&](bool flag) -> bool {
        uint32_t any;
        asm volatile(
            "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
            "bar.red.or.pred q, 1, %2, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
            : "=r"(any)
            : "r"((uint32_t)flag), "r"(128 * NG)
            : "memory");
        return any != 0;
    };
    const uint32_t s16 = sm_base + L::kS16 + gi * 4096;  // this group's S (fp16, [16][128])
    const uint32_t ut = sm_base + L::kUt + gi * 2048;    // this group's U^T (fp16, [16][64])

    constexpr int kConsumerWarps = 4 * NG;
    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        mbar_init(&bars[2], kConsumerWarps);
        mbar_init(&bars[3], kConsumerWarps);
        fence_mbar_init();
    }
    if (warp == kConsumerWarps) {
        // ---- producer warp: TMA copies of each chunk, one stage ahead ----------
        __syncthreads();
        if (lane == 0) {
            for (int lc = 0; lc < nch; ++lc) {
                const int stage = lc & 1;
                if (lc >= 2 && !mbar_wait(&bars[2 + stage], ((lc >> 1) - 1) & 1)) {
                    if (p.status) atomicOr(p.status, 1);
                    break;
                }
                const size_t ch = (size_t)(c0 + lc) * p.H + h;
                const uint8_t* src = p.ws + ch * kWsBytes;
                uint8_t* dst = smem + stage * L::kStage;
                mbar_arrive_expect_tx(&bars[stage], (uint32_t)(L::kShared + L::kU));
                bulk_g2s(dst, src, (uint32_t)L::kShared, &bars[stage]);
                bulk_g2s(dst + L::kSharedPad, src + kWsUOff + vs0 * kWsUSliceBytes,
                         (uint32_t)L::kU, &bars[stage]);
            }
        }
        return;
    }

    // ---- initial state -> fp32 master copy in registers --------------------
    const bool has_init = p.has_init ? (p.has_init[n] != 0) : (p.st_in != nullptr);
    const int64_t in_slot = p.st_in_idx ? p.st_in_idx[n] : n;
    const int64_t out_slot = p.st_out_idx ? p.st_out_idx[n] : n;
    const size_t in_base = (size_t)in_slot * p.st_in_stride + (size_t)h * D * D;
    const size_t out_base = (size_t)out_slot * p.st_out_stride + (size_t)h * D * D;
    const int vcol0 = (vs0 + gi) * 16;  // first value row of this group

    float Sm[2][2][4];  // [mt][nt][e]: k = 32wr+16mt+g+8(e>>1), v = 8nt+2tq+(e&1)
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int kk = 32 * wr + 16 * mt + g + 8 * (e >> 1);
                const int vv = vcol0 + 8 * nt + 2 * tq + (e & 1);
                Sm[mt][nt][e] =
                    has_init ? load_state(p.st_in, p.st_dtype, in_base + (size_t)vv * D + kk) : 0.f;
            }

    auto write_s16 = [&]() {
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int kk = 32 * wr + 16 * mt + g + 8 * (e >> 1);
                    const int vv = 8 * nt + 2 * tq + (e & 1);
                    const __half hv = __float2half_rn(Sm[mt][nt][e]);
                    asm volatile("st.shared.b16 [%0], %1;" ::"r"(s16 + sw128_off(vv, kk, 16)),
                                 "h"(*reinterpret_cast<const unsigned short*>(&hv)));
                }
    };

    // B fragments of S for U = w S^T and qg S^T: [ks][4] = b0,b1 (nt 0), b0,b1 (nt 1)
    uint32_t Sf[8][4];
    auto load_sfrag = [&]() {
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const int row = rr + 8 * (mi >> 1);
            const int col = 16 * ks + 8 * (mi & 1);
            ldsm_x4(s16 + sw128_off(row, col, 16), Sf[ks][0], Sf[ks][1], Sf[ks][2], Sf[ks][3]);
        }
    };

    write_s16();
    __syncthreads();  // consumers and producer: mbarriers initialised, S16 written
    load_sfrag();

    bool failed = false;
    for (int lc = 0; lc < nch; ++lc) {
        const int stage = lc & 1;
        // Bounded wait; the outcome is voted at the next compute-warp barrier so
        // that every compute warp leaves the walk together (nothing is written
        // to global memory before that vote).
        const bool ok = mbar_wait(&bars[stage], (lc >> 1) & 1);
        const uint32_t st = sm_base + stage * L::kStage;
        const uint32_t tw = st + kWsWOff, tqg = st + kWsQGOff, tkg = st + kWsKGOff;
        const uint32_t taqk = st + kWsAqkOff;
        const float* gam = reinterpret_cast<const float*>(smem + stage * L::kStage + kWsGammaOff);
        const uint32_t tu = st + L::kSharedPad + gi * kWsUSliceBytes;  // [64][16] fp16

        // (1) accU = w S^T, accO = qg S^T for rows 16wr..16wr+15
        // two independent accumulation chains per product (key halves) for ILP
        float accU[2][4] = {}, accO[2][4] = {}, accU2[2][4] = {}, accO2[2][4] = {};
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            uint32_t aw[4], aq[4];
            const int row = 16 * wr + rr + 8 * (mi & 1);
            const int col = 16 * ks + 8 * (mi >> 1);
            ldsm_x4(tw + sw128_off(row, col, 64), aw[0], aw[1], aw[2], aw[3]);
            ldsm_x4(tqg + sw128_off(row, col, 64), aq[0], aq[1], aq[2], aq[3]);
            float (*u)[4] = (ks & 1) ? accU2 : accU;
            float (*o)[4] = (ks & 1) ? accO2 : accO;
            mma_f16(u[0], aw, Sf[ks][0], Sf[ks][1]);
            mma_f16(u[1], aw, Sf[ks][2], Sf[ks][3]);
            mma_f16(o[0], aq, Sf[ks][0], Sf[ks][1]);
            mma_f16(o[1], aq, Sf[ks][2], Sf[ks][3]);
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                accU[nt][e] += accU2[nt][e];
                accO[nt][e] += accO2[nt][e];
            }
        // (2) U = u - accU, (3) U^T -> shared (fp16)
        float U[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int i = 16 * wr + g + 8 * hh;
                const int vv = 8 * nt + 2 * tq;
                uint32_t uv;
                asm volatile("ld.shared.b32 %0, [%1];" : "=r"(uv) : "r"(tu + i * 32 + vv * 2));
                const float2 uf = __half22float2(*reinterpret_cast<__half2*>(&uv));
                U[nt][2 * hh] = uf.x - accU[nt][2 * hh];
                U[nt][2 * hh + 1] = uf.y - accU[nt][2 * hh + 1];
                const __half h0 = __float2half_rn(U[nt][2 * hh]);
                const __half h1 = __float2half_rn(U[nt][2 * hh + 1]);
                asm volatile("st.shared.b16 [%0], %1;" ::"r"(ut + sw64_off(vv, i)),
                             "h"(*reinterpret_cast<const unsigned short*>(&h0)));
                asm volatile("st.shared.b16 [%0], %1;" ::"r"(ut + sw64_off(vv + 1, i)),
                             "h"(*reinterpret_cast<const unsigned short*>(&h1)));
            }
        if (consumer_sync_or(!ok)) {  // a copy never landed: report, stop the walk
            failed = true;
            if (tid == 0 && p.status) atomicOr(p.status, 1);
            break;
        }

        // (5) o = accO + A_qk U (A_qk lower triangular: key blocks 0..wr)
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
            if (ks > wr) break;
            uint32_t a[4], b[4];
            const int row = 16 * wr + rr + 8 * (mi & 1);
            const int col = 16 * ks + 8 * (mi >> 1);
            ldsm_x4(taqk + sw64_off(row, col), a[0], a[1], a[2], a[3]);
            ldsm_x4(ut + sw64_off(rr + 8 * (mi >> 1), 16 * ks + 8 * (mi & 1)), b[0], b[1], b[2],
                    b[3]);
            mma_f16(accO[0], a, b[0], b[1]);
            mma_f16(accO[1], a, b[2], b[3]);
        }
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int i = 16 * wr + g + 8 * hh;
            if (lc * C + i < len) {
                const size_t t = (size_t)(tok0 + lc * C + i);
                __nv_bfloat16* orow = p.out + (t * p.H + h) * D + vcol0;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const uint32_t pv = pack_bf162(accO[nt][2 * hh], accO[nt][2 * hh + 1]);
                    *reinterpret_cast<uint32_t*>(orow + 8 * nt + 2 * tq) = pv;
                }
            }
        }

        // (6) dS^T = kg^T U for key channels 32wr..32wr+31, (7) S = gamma S + dS
        float accS[2][2][4] = {};
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
            uint32_t b[4];
            ldsm_x4(ut + sw64_off(rr + 8 * (mi >> 1), 16 * ks + 8 * (mi & 1)), b[0], b[1], b[2],
                    b[3]);
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
                uint32_t a[4];
                const int srow = 16 * ks + rr + 8 * (mi >> 1);       // chunk row c
                const int scol = 32 * wr + 16 * mt + 8 * (mi & 1);   // key channel
                ldsm_x4_t(tkg + sw128_off(srow, scol, 64), a[0], a[1], a[2], a[3]);
                mma_f16(accS[mt][0], a, b[0], b[1]);
                mma_f16(accS[mt][1], a, b[2], b[3]);
            }
        }
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const float gk = gam[32 * wr + 16 * mt + g + 8 * hh];
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    Sm[mt][nt][2 * hh] = gk * Sm[mt][nt][2 * hh] + accS[mt][nt][2 * hh];
                    Sm[mt][nt][2 * hh + 1] = gk * Sm[mt][nt][2 * hh + 1] + accS[mt][nt][2 * hh + 1];
                }
            }
        // stage data fully consumed by this warp: release it to the producer
        __syncwarp();
        if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&bars[2 + stage])) : "memory");
        write_s16();
        consumer_sync();
        load_sfrag();
    }

    if (failed) return;
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int kk = 32 * wr + 16 * mt + g + 8 * (e >> 1);
                const int vv = vcol0 + 8 * nt + 2 * tq + (e & 1);
                store_state(p.st_out, p.st_dtype, out_base + (size_t)vv * D + kk, Sm[mt][nt][e]);
            }
}

template <int NG>
cudaError_t launch_scan_ng(const FwdParams& p, cudaStream_t s) {
    using L = ScanSmem<NG>;
    static unsigned configured = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 32 && !(configured & (1u << dev))) {
        e = cudaFuncSetAttribute(kda_scan_mma<NG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 L::kTotal);
        if (e != cudaSuccess) return e;
        configured |= 1u << dev;
    }
    dim3 grid((unsigned)p.N, (unsigned)p.H, (unsigned)(8 / NG));
    kda_scan_mma<NG><<<grid, 128 * NG + 32, L::kTotal, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

int scan_groups(int N, int H, int num_sms) {
    // Finest value split that still leaves whole sequences x heads to fill the
    // GPU: fewer groups per CTA when there are few (sequence, head) pairs.
    const long pairs = (long)N * H;
    return pairs * 8 <= 2L * num_sms ? 1 : 2;
}

cudaError_t launch_scan(const FwdParams& p, int ng, cudaStream_t s) {
    if (p.N <= 0) return cudaSuccess;
    switch (ng) {
        case 1: return launch_scan_ng<1>(p, s);
        case 2: return launch_scan_ng<2>(p, s);
        default: return launch_scan_ng<2>(p, s);
    }
}

}  // namespace kda
