// The scan walk for large batches, partitioned by value rows: one CTA per
// (sequence, head, 64 or 128 value rows), four or eight compute warps that each
// own 16 value rows of the state for all 128 keys (with four, a producer warp).
//
// Per chunk, warp w (value rows v = v0 + 16w ..), with S its rows of the chunk's
// incoming state (fp32 accumulators, M = the 16 value rows, N = the 128 keys):
//   U^T = u^T - S w^T       (16 x 64)    A = S from the warp's own accumulators
//   o^T = S qg^T + U^T A_qk^T            A = S, then U^T, from its accumulators
//   S   = S Diag(gamma) + U^T kg          A = U^T from its accumulators
// (the chunk recurrence of kda_scan.cu, transposed so that the state's value
// rows are the MMAs' M dimension.)  An m16n8 accumulator pair is an m16k16 A
// fragment, so no product needs another warp's rows or a shared-memory round
// trip of S or U: the warps never synchronise with each other.  Each warp reads
// the chunk's w, qg, kg and A_qk tiles itself (the B operands), which the
// role-split walk (kda_scan_walk.cuh) spreads over eight warps at the price of
// moving S and U through shared memory twice per chunk; at 64 value rows per CTA
// this form took the varlen batch's scan from 566 to 495 us.  The output rows
// are staged (stmatrix, transposing) and stored with one TMA store per warp and
// chunk.
#pragma once

#include "kda_scan_walk.cuh"

namespace kda {
namespace scan {

// NW compute warps (4 or 8): 16 NW value rows per CTA.  With 4 a producer warp
// streams the chunks; with 8 there is none (the CTA's 256 threads then get the
// registers they need) and the last warp done with a stage refills it.
template <int NW>
struct ScanSmemVP {
    static constexpr int VS = 16 * NW;                       // value rows per CTA
    static constexpr int kStages = NW >= 8 ? 2 : 3;
    static constexpr int kShared = kWsSharedBytes;           // w, qg, kg, aqk, gamma
    static constexpr int kSharedPad = round1k(kShared);
    static constexpr int kU = (VS / 16) * kWsUSliceBytes;    // the CTA's u columns
    static constexpr int kStage = kSharedPad + round1k(kU);
    static constexpr int kOutBuf = 64 * 16 * 2;              // a warp's [64][16] bf16 rows
    static constexpr int kOut = kStages * kStage;            // [NW warps][2][kOutBuf]
    static constexpr int kBar = kOut + NW * 2 * kOutBuf;     // full, empty [kStages]
    static constexpr int kCnt = kBar + 16 * kStages;         // [kStages] warps done (NW = 8)
    static constexpr int kTotal = kCnt + 64;
};
template <int NW>
constexpr int vp_threads() { return 32 * (NW + (NW >= 8 ? 0 : 1)); }

// One walk over the whole sequence from its pool (or zero) state: outputs, and
// the final state back to the pool.  Runs on vp_threads<NW>() threads over
// ScanSmemVP<NW>::kTotal bytes of shared memory at `smem` (1 KB aligned).
// out_map: a tensor map of `out` ([T][H][128] bf16, box 16 values x 1 head x 64
// rows) for whole chunks, or nullptr (every output element stored directly).
template <int NW>
__device__ __forceinline__ void scan_walk_vp(const FwdParams& p, uint8_t* smem, int n, int h, int z,
                                             const CUtensorMap* out_map) {
    using L = ScanSmemVP<NW>;
    constexpr int kStages = L::kStages;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBar);  // [kStages]
    uint64_t* empty = full + kStages;                               // [kStages] (NW = 4)
    uint32_t* done = reinterpret_cast<uint32_t*>(smem + L::kCnt);   // [kStages] (NW = 8)

    const int v0 = z * L::VS;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, tq = lane & 3;
    const int mi = lane >> 3, rr = lane & 7;

    const int tok0 = p.cu[n];
    const int len = p.cu[n + 1] - tok0;
    const int c0 = p.seq_off[n];
    const int nch = p.seq_off[n + 1] - c0;
    const uint32_t sm_base = smem_u32(smem);

    // No L2 prefetch ahead of the stage copies: with a CTA per (sequence, head)
    // on every SM, lines asked for several chunks ahead were evicted before
    // their copy and read twice from DRAM (varlen batch: 2.48 GB read against
    // the 1.57 GB of intermediates, scan 503 us; without the prefetch 415 us).

    // chunk lc's shared part and the CTA's u columns into stage lc % kStages
    auto issue_chunk = [&](int lc) {
        const int stage = lc % kStages;
        const uint8_t* src = p.ws + ((size_t)(c0 + lc) * p.H + h) * kWsBytes;
        uint8_t* dst = smem + stage * L::kStage;
        mbar_arrive_expect_tx(&full[stage], (uint32_t)(L::kShared + L::kU));
        bulk_g2s(dst, src, (uint32_t)L::kShared, &full[stage]);
        bulk_g2s(dst + L::kSharedPad, src + kWsUOff + (v0 / 16) * kWsUSliceBytes, (uint32_t)L::kU,
                 &full[stage]);
    };

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], NW);
            done[i] = 0;
        }
        fence_mbar_init();
    }
    __syncthreads();

    if constexpr (NW >= 8) {
        // no producer warp: the first stages now, the others by the last warp done
        // with each stage (below)
        // launched right behind the intra-chunk kernel, the CTA may start while
        // that kernel's last items run: the intermediates are read after it is done
        if (tid == 0) {
            grid_dep_wait();
            for (int lc = 0; lc < kStages && lc < nch; ++lc) issue_chunk(lc);
        }
    } else if (warp == NW) {
        // ======================= producer warp ==============================
        if (lane == 0) {
            grid_dep_wait();  // the intermediates are read after the intra-chunk kernel
            int issued = 0;
            for (int lc = 0; lc < nch; ++lc) {
                const int stage = lc % kStages;
                if (lc >= kStages && !mbar_wait(&empty[stage], ((lc / kStages) - 1) & 1)) {
                    if (p.status) atomicOr(p.status, 1);
                    break;
                }
                issue_chunk(lc);
                issued = lc + 1;
            }
            // the copies still in flight land before the CTA may leave
            for (int lc = issued > kStages ? issued - kStages : 0; lc < issued; ++lc)
                mbar_wait(&full[lc % kStages], (lc / kStages) & 1);
        }
        return;
    }

    // ======================= compute warps ==================================
    const int w = warp;
    const int vw = v0 + 16 * w;  // this warp's first value row
    bool has_init = p.has_init ? (p.has_init[n] != 0) : (p.st_in != nullptr);
    const int64_t in_slot = p.st_in_idx ? p.st_in_idx[n] : n;
    const int64_t out_slot = p.st_out_idx ? p.st_out_idx[n] : n;
    bool store_ok = true;
    if (p.num_slots > 0) {  // a slot outside the pool: no access, reported
        const bool bad_in = has_init && (in_slot < 0 || in_slot >= p.num_slots);
        const bool bad_out = out_slot < 0 || out_slot >= p.num_slots;
        if ((bad_in || bad_out) && w == 0 && lane == 0 && p.status) atomicOr(p.status, 4);
        if (bad_in) has_init = false;
        if (bad_out) store_ok = false;
    }
    const size_t in_base = has_init ? (size_t)in_slot * p.st_in_stride + (size_t)h * D * D : 0;
    const size_t out_base = store_ok ? (size_t)out_slot * p.st_out_stride + (size_t)h * D * D : 0;

    // the warp's state rows: Sa[nt][e] = S[vw + g + 8 (e >> 1)][8 nt + 2 tq + (e & 1)]
    float Sa[16][4];
#pragma unroll
    for (int nt = 0; nt < 16; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e)
            Sa[nt][e] = has_init ? load_state(p.st_in, p.st_dtype,
                                              in_base + (size_t)(vw + g + 8 * (e >> 1)) * D + 8 * nt +
                                                  2 * tq + (e & 1))
                                 : 0.f;

    // B fragments of a row-major [64 rows][128 keys] tile (w or qg) for the K step
    // of keys 16 ks..: [row n-tile][b0, b1]
    auto load_rows_b = [&](uint32_t tile, int ks, uint32_t (&b)[8][2]) {
#pragma unroll
        for (int np = 0; np < 4; ++np)
            ldsm_x4(tile + sw128_off(16 * np + 8 * (mi >> 1) + rr, 16 * ks + 8 * (mi & 1), 64),
                    b[2 * np][0], b[2 * np][1], b[2 * np + 1][0], b[2 * np + 1][1]);
    };

    grid_dep_wait();  // the state came from the pool; the chunks come after
    bool failed = false;
    for (int lc = 0; lc < nch; ++lc) {
        const int sg = lc % kStages;
        if (!mbar_wait(&full[sg], (lc / kStages) & 1)) {
            failed = true;
            if (p.status) atomicOr(p.status, 1);
            break;
        }
        const uint32_t st = sm_base + sg * L::kStage;
        const uint32_t tw = st + kWsWOff, tqg = st + kWsQGOff, tkg = st + kWsKGOff;
        const uint32_t taqk = st + kWsAqkOff;
        const uint32_t tu = st + L::kSharedPad + w * kWsUSliceBytes;  // [64 rows][16 values] fp16
        const float* gam = reinterpret_cast<const float*>(smem + sg * L::kStage + kWsGammaOff);

        // S (fp16) as A fragments over the K steps of 16 keys
        uint32_t sa[8][4];
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            sa[ks][0] = pack_half2(Sa[2 * ks][0], Sa[2 * ks][1]);
            sa[ks][1] = pack_half2(Sa[2 * ks][2], Sa[2 * ks][3]);
            sa[ks][2] = pack_half2(Sa[2 * ks + 1][0], Sa[2 * ks + 1][1]);
            sa[ks][3] = pack_half2(Sa[2 * ks + 1][2], Sa[2 * ks + 1][3]);
        }

        // S w^T and o^T = S qg^T (the next K step's w fragments load while the
        // current ones are used)
        float ua[8][4] = {}, oa[8][4] = {};
        {
            uint32_t bw[8][2], bq[8][2];
            load_rows_b(tw, 0, bw);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                load_rows_b(tqg, ks, bq);
#pragma unroll
                for (int nt = 0; nt < 8; ++nt) mma_f16(ua[nt], sa[ks], bw[nt][0], bw[nt][1]);
                if (ks + 1 < 8) load_rows_b(tw, ks + 1, bw);
#pragma unroll
                for (int nt = 0; nt < 8; ++nt) mma_f16(oa[nt], sa[ks], bq[nt][0], bq[nt][1]);
            }
        }

        // U^T = u^T - S w^T: u of the warp's 16 value columns read transposed into
        // the accumulator layout (value rows g, g + 8; chunk rows 2 tq, 2 tq + 1)
#pragma unroll
        for (int np = 0; np < 4; ++np) {
            uint32_t r[4];
            ldsm_x4_t(tu + (16 * np + 8 * (mi >> 1) + rr) * 32 + (mi & 1) * 16, r[0], r[1], r[2], r[3]);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int nt = 2 * np + (q >> 1), o2 = 2 * (q & 1);
                const float2 u2 = __half22float2(*reinterpret_cast<const __half2*>(&r[q]));
                ua[nt][o2] = u2.x - ua[nt][o2];
                ua[nt][o2 + 1] = u2.y - ua[nt][o2 + 1];
            }
        }
        // U^T (fp16) as A fragments over the K steps of 16 chunk rows
        uint32_t uf[4][4];
#pragma unroll
        for (int kr = 0; kr < 4; ++kr) {
            uf[kr][0] = pack_half2(ua[2 * kr][0], ua[2 * kr][1]);
            uf[kr][1] = pack_half2(ua[2 * kr][2], ua[2 * kr][3]);
            uf[kr][2] = pack_half2(ua[2 * kr + 1][0], ua[2 * kr + 1][1]);
            uf[kr][3] = pack_half2(ua[2 * kr + 1][2], ua[2 * kr + 1][3]);
        }

        // o^T += U^T A_qk^T: A_qk is lower triangular, so row blocks pp take key
        // blocks kr <= pp (ten blocks); each block's fragments load one block ahead
        {
            constexpr int kBlocks = 10;
            auto blk = [](int i, int& pp, int& kr) {  // (0,0) (1,0) (1,1) (2,0) .. (3,3)
                pp = i < 1 ? 0 : (i < 3 ? 1 : (i < 6 ? 2 : 3));
                kr = i - pp * (pp + 1) / 2;
            };
            auto load_aqk = [&](int i, uint32_t (&b4)[4]) {
                int pp, kr;
                blk(i, pp, kr);
                ldsm_x4(taqk + sw64_off(16 * pp + 8 * (mi >> 1) + rr, 16 * kr + 8 * (mi & 1)), b4[0],
                        b4[1], b4[2], b4[3]);
            };
            uint32_t bq2[2][4];
            load_aqk(0, bq2[0]);
#pragma unroll
            for (int i = 0; i < kBlocks; ++i) {
                if (i + 1 < kBlocks) load_aqk(i + 1, bq2[(i + 1) & 1]);
                int pp, kr;
                blk(i, pp, kr);
                mma_f16(oa[2 * pp], uf[kr], bq2[i & 1][0], bq2[i & 1][1]);
                mma_f16(oa[2 * pp + 1], uf[kr], bq2[i & 1][2], bq2[i & 1][3]);
            }
        }

        // S = S Diag(gamma) + U^T kg (kg read transposed: K = chunk rows, N = keys;
        // each pair of key n-tiles' fragments loads two pairs ahead)
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
            const float2 gk = *reinterpret_cast<const float2*>(gam + 8 * nt + 2 * tq);
            Sa[nt][0] *= gk.x;
            Sa[nt][1] *= gk.y;
            Sa[nt][2] *= gk.x;
            Sa[nt][3] *= gk.y;
        }
        {
            auto load_kg = [&](int i, uint32_t (&b4)[4]) {  // i = 8 kr + np
                const int kr = i >> 3, np = i & 7;
                ldsm_x4_t(tkg + sw128_off(16 * kr + 8 * (mi & 1) + rr, 16 * np + 8 * (mi >> 1), 64), b4[0],
                          b4[1], b4[2], b4[3]);
            };
            uint32_t bk[3][4];
            load_kg(0, bk[0]);
            load_kg(1, bk[1]);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                if (i + 2 < 32) load_kg(i + 2, bk[(i + 2) % 3]);
                const int kr = i >> 3, np = i & 7;
                mma_f16(Sa[2 * np], uf[kr], bk[i % 3][0], bk[i % 3][1]);
                mma_f16(Sa[2 * np + 1], uf[kr], bk[i % 3][2], bk[i % 3][3]);
            }
        }
        __syncwarp();
        if (lane == 0) {  // this warp is done with the stage
            if constexpr (NW >= 8) {
                // the last warp done refills it with the chunk kStages ahead
                uint32_t old;
                asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], 1;"
                             : "=r"(old)
                             : "r"(smem_u32(&done[sg]))
                             : "memory");
                if (old == NW - 1) {
                    done[sg] = 0;
                    if (lc + kStages < nch) issue_chunk(lc + kStages);
                }
            } else {
                mbar_arrive(&empty[sg]);
            }
        }

        // the outputs: a whole chunk staged ([64 rows][16 values] bf16, stmatrix
        // transposing the value-row fragments) and stored by one TMA store; the
        // buffer was last read two chunks back.  A partial chunk row by row.
        if (out_map && lc * C + C <= len) {
            const uint32_t ob = sm_base + L::kOut + (2 * w + (lc & 1)) * L::kOutBuf;
            if (lane == 0) bulk_wait_read<1>();
            __syncwarp();
#pragma unroll
            for (int np = 0; np < 4; ++np)
                stsm_x4_t(ob + (16 * np + 8 * (mi >> 1) + rr) * 32 + (mi & 1) * 16,
                          pack_bf162(oa[2 * np][0], oa[2 * np][1]), pack_bf162(oa[2 * np][2], oa[2 * np][3]),
                          pack_bf162(oa[2 * np + 1][0], oa[2 * np + 1][1]),
                          pack_bf162(oa[2 * np + 1][2], oa[2 * np + 1][3]));
            fence_proxy_async();  // the staged rows are read by the TMA store
            __syncwarp();
            if (lane == 0) {
                tma_store_3d(out_map, smem + (ob - sm_base), vw, h, tok0 + lc * C);
                bulk_commit();
            }
        } else {
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int row = 8 * nt + 2 * tq + (e & 1);
                    if (lc * C + row < len)
                        p.out[((size_t)(tok0 + lc * C + row) * p.H + h) * D + vw + g + 8 * (e >> 1)] =
                            __float2bfloat16_rn(oa[nt][e]);
                }
        }
    }
    if (lane == 0) bulk_wait_all();  // the TMA stores complete before the CTA leaves
    if constexpr (NW >= 8) {
        // the copies possibly still in flight land before the CTA may leave
        // (they all have, unless a wait gave up)
        if (tid == 0)
            for (int lc = nch > kStages ? nch - kStages : 0; lc < nch; ++lc)
                mbar_wait(&full[lc % kStages], (lc / kStages) & 1);
    }
    if (failed || !store_ok) return;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e)
            store_state(p.st_out, p.st_dtype,
                        out_base + (size_t)(vw + g + 8 * (e >> 1)) * D + 8 * nt + 2 * tq + (e & 1),
                        Sa[nt][e]);
}

}  // namespace scan
}  // namespace kda
