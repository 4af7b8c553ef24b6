// State scan of the chunkwise KDA forward, as a device function shared by the
// standalone scan kernel (kda_scan.cu) and the fused intra + scan kernel
// (kda_intra_tc.cu).  The walk itself is described in kda_scan.cu.
#pragma once

#include "kda_device.cuh"
#include "kda_internal.h"

namespace kda {
namespace scan {

using namespace dev;

// Ready flags of a walk's next blocks (consecutive chunks of one head, `stride`
// ints apart): waits (bounded) until the first is set, reading up to kAhead of
// them per round trip, and returns how many consecutive ones are set from the
// first (0: the wait gave up).  The relaxed loads followed by an acquire fence
// pair with the writers' release stores; the proxy fence then orders the blocks'
// contents before this thread's later bulk copies (async proxy) of them.
constexpr int kAhead = 8;
constexpr uint32_t kFlagRounds = 1u << 22;  // about a second of rounds on GB300 (measured)
__device__ __forceinline__ int wait_ready_run(const int* flags, int stride, int count) {
    for (uint32_t i = 0; i < kFlagRounds; ++i) {
        int v[kAhead];
#pragma unroll
        for (int j = 0; j < kAhead; ++j) {
            v[j] = 0;
            if (j < count)
                asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];"
                             : "=r"(v[j])
                             : "l"(flags + (size_t)j * stride)
                             : "memory");
        }
        int run = 0;
#pragma unroll
        for (int j = 0; j < kAhead; ++j)
            if (run == j && v[j] != 0) ++run;
        if (run > 0) {
            asm volatile("fence.acq_rel.gpu;" ::: "memory");
            asm volatile("fence.proxy.async.global;" ::: "memory");
            return run;
        }
        __nanosleep(64);
    }
    return 0;
}

constexpr int C = kC;
constexpr int D = kD;

constexpr int round1k(int x) { return (x + 1023) / 1024 * 1024; }

constexpr int kPrefetch = 6;  // chunks ahead of the stage loads asked of L2
// Slots of the S and U rings shared by the state and output warps: with two,
// the state warps may run one chunk ahead of the output warps (three measured
// slower: 188 against 183 us for the 16K prefill's scan).
constexpr int kRing = 2;

// The role-split walk serves 16 or 32 value rows per CTA; larger blocks of
// value rows take the values-partitioned walk (kda_scan_vp.cuh).
template <int NT>
struct ScanSmem {
    static_assert(NT == 2 || NT == 4, "16 or 32 value rows per CTA");
    static constexpr int VS = 8 * NT;                        // value rows per CTA
    static constexpr int kStages = 3;                        // chunk intermediates in flight
    static constexpr int kShared = kWsSharedBytes;           // w, qg, kg, aqk, gamma
    static constexpr int kSharedPad = round1k(kShared);
    static constexpr int kU = (VS / 16) * kWsUSliceBytes;    // the CTA's u columns
    static constexpr int kStage = kSharedPad + round1k(kU);
    static constexpr int kS16 = kStages * kStage;            // kRing slots x [VS][128] fp16
    static constexpr int kS16Slot = VS * 256;
    static constexpr int kUt = kS16 + kRing * kS16Slot;      // kRing slots x [VS][64] fp16
    static constexpr int kUtSlot = VS * 128;
    // The output rows are stored directly: staging them for TMA stores measured
    // slower here (the 16K prefill's scan 204 against 182 us).
    static constexpr int kBar = round1k(kUt + kRing * kUtSlot);  // mbarriers (2 kStages + 2 kRing)
    static constexpr int kAbort = kBar + 8 * (2 * kStages + 2 * kRing);  // int: a state warp gave up
    static constexpr int kTotal = kBar + 128;
    static_assert(kAbort + 4 <= kTotal, "mbarriers and the abort flag fit");
};

constexpr int kStateWarps = 4, kOutWarps = 4;
constexpr int kScanThreads = 32 * (kStateWarps + kOutWarps + 1);

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

// One walk: the CTA's value rows v0 = z * VS.. of head h of long sequence n.  Runs
// on threads 0..kScanThreads-1 of the CTA (others must not call it) over the
// shared memory at `smem` (1 KB aligned, ScanSmem<NT>::kTotal bytes).  With
// p.ready set, each chunk's operands are fetched only once their block is
// marked written (the fused launch, where the intra-chunk work runs alongside).
// What a walk covers, where its state starts and where it ends.  The default
// walks the whole sequence from its pool (or zero) state, writes the outputs
// and writes the final state back to the pool.  The segmented scan walks a
// range of chunks from a zero state, from identity rows with u = 0 (the range's
// transition), or from a given fp32 state.
struct WalkRange {
    int first = 0;                // first chunk of the sequence
    int count = -1;               // chunks to walk; -1: to the end
    int init = 0;                 // 0: pool per has_initial_state, 1: zero, 2: identity rows, 3: init_buf
    const float* init_buf = nullptr;  // init 3: [128][128] fp32, rows = value rows
    bool zero_u = false;          // u taken as 0
    bool outputs = true;          // write o
    bool final_state = true;      // write the final state
    float* final_buf = nullptr;   // ... into this [128][128] fp32 plane instead of the pool
};

template <int NT>
__device__ __forceinline__ void scan_walk(const FwdParams& p, uint8_t* smem, int n, int h, int z,
                                          const WalkRange& R = WalkRange()) {
    using L = ScanSmem<NT>;
    constexpr int VS = L::VS;
    constexpr int kStages = L::kStages;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBar);  // [kStages]
    uint64_t* empty = full + kStages;                               // [kStages]
    uint64_t* sready = full + 2 * kStages;                          // [kRing]
    uint64_t* sfree = sready + kRing;                               // [kRing]
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);

    const int v0 = z * VS;  // first value row of this CTA
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, tq = lane & 3;
    const int mi = lane >> 3, rr = lane & 7;  // ldmatrix / stmatrix addressing

    const int tok0 = p.cu[n] + R.first * C;  // token of the walk's first chunk
    const int len = p.cu[n + 1] - tok0;         // tokens from there to the sequence end
    const int c0 = p.seq_off[n] + R.first;
    const int left = p.seq_off[n + 1] - c0;
    const int nch = R.count < 0 || R.count > left ? left : R.count;

    const uint32_t sm_base = smem_u32(smem);
    auto stage_base = [&](int s) { return sm_base + s * L::kStage; };
    auto s16_slot = [&](int b) { return sm_base + L::kS16 + b * L::kS16Slot; };
    auto ut_slot = [&](int b) { return sm_base + L::kUt + b * L::kUtSlot; };

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kStateWarps + kOutWarps);
        }
        for (int i = 0; i < kRing; ++i) {
            mbar_init(&sready[i], 1);
            mbar_init(&sfree[i], kOutWarps);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    asm volatile("bar.sync 2, %0;" ::"n"(kScanThreads) : "memory");

    // ======================= producer warp ==================================
    // Launched right behind the intra-chunk kernel, the CTA may start while that
    // kernel's last items run: the intermediates are read only after it is done.
    if (warp == kStateWarps + kOutWarps) {
        grid_dep_wait();
        if (lane == 0) {
            // this CTA's share of the shared part for the L2 prefetch (16-byte units)
            constexpr int kGroups = D / VS;
            constexpr int kUnits = kWsSharedBytes / 16;
            const uint32_t pf_off = 16u * (uint32_t)(kUnits * z / kGroups);
            const uint32_t pf_len = 16u * (uint32_t)(kUnits * (z + 1) / kGroups) - pf_off;
            auto prefetch = [&](int lc) {
                const size_t ch = (size_t)(c0 + lc) * p.H + h;
                const uint8_t* src = p.ws + ch * kWsBytes;
                asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src + pf_off),
                             "r"(pf_len)
                             : "memory");
                asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(
                                 src + kWsUOff + (v0 / 16) * kWsUSliceBytes),
                             "r"((uint32_t)L::kU)
                             : "memory");
            };
            for (int lc = 0; lc < kPrefetch && lc < nch; ++lc) prefetch(lc);
            int ready_upto = 0;  // chunks known written (fused launch)
            for (int lc = 0; lc < nch; ++lc) {
                const int stage = lc % kStages;
                if (lc >= kStages && !mbar_wait(&empty[stage], ((lc / kStages) - 1) & 1)) {
                    if (p.status) atomicOr(p.status, 1);
                    break;
                }
                if (lc + kPrefetch < nch) prefetch(lc + kPrefetch);
                const size_t ch = (size_t)(c0 + lc) * p.H + h;
                if (p.ready && lc >= ready_upto) {
                    const int run = wait_ready_run(p.ready + ch, p.H, nch - lc);
                    if (run == 0) {
                        if (p.status) atomicOr(p.status, 1);
                        break;
                    }
                    ready_upto = lc + run;
                }
                const uint8_t* src = p.ws + ch * kWsBytes;
                uint8_t* dst = smem + stage * L::kStage;
                mbar_arrive_expect_tx(&full[stage], (uint32_t)(L::kShared + L::kU));
                bulk_g2s(dst, src, (uint32_t)L::kShared, &full[stage]);
                bulk_g2s(dst + L::kSharedPad, src + kWsUOff + (v0 / 16) * kWsUSliceBytes,
                         (uint32_t)L::kU, &full[stage]);
            }
        }
        return;
    }

    // ======================= output warps ===================================
    if (warp >= kStateWarps) {
        grid_dep_wait();
        const int wr = warp - kStateWarps;  // chunk rows 16wr..16wr+15
        for (int lc = 0; lc < nch; ++lc) {
            const int b = lc % kRing, sg = lc % kStages;
            const uint32_t par = (lc / kRing) & 1;
            if (!mbar_wait(&full[sg], (lc / kStages) & 1) || !mbar_wait(&sready[b], par)) {
                if (p.status) atomicOr(p.status, 1);
                break;
            }
            const uint32_t st = stage_base(sg);
            const uint32_t tqg = st + kWsQGOff, taqk = st + kWsAqkOff;
            const uint32_t s16 = s16_slot(b), ut = ut_slot(b);
            // qg S^T (two accumulation chains over the key halves) + A_qk U
            float acc[NT][4] = {}, acc2[NT][4] = {};
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                uint32_t a[4];
                ldsm_x4(tqg + sw128_off(16 * wr + rr + 8 * (mi & 1), 16 * ks + 8 * (mi >> 1), 64),
                        a[0], a[1], a[2], a[3]);
                float (*d)[4] = (ks & 1) ? acc2 : acc;  // two chains over the key halves
#pragma unroll
                for (int np = 0; np < NT / 2; ++np) {
                    uint32_t bb[4];
                    ldsm_x4(s16 + sw128_off(16 * np + rr + 8 * (mi >> 1), 16 * ks + 8 * (mi & 1), VS),
                            bb[0], bb[1], bb[2], bb[3]);
                    mma_f16(d[2 * np], a, bb[0], bb[1]);
                    mma_f16(d[2 * np + 1], a, bb[2], bb[3]);
                }
            }
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {  // A_qk lower triangular: key blocks 0..wr
                if (ks > wr) break;
                uint32_t a[4];
                ldsm_x4(taqk + sw64_off(16 * wr + rr + 8 * (mi & 1), 16 * ks + 8 * (mi >> 1)), a[0],
                        a[1], a[2], a[3]);
#pragma unroll
                for (int np = 0; np < NT / 2; ++np) {
                    uint32_t bb[4];
                    ldsm_x4(ut + sw64_off(16 * np + rr + 8 * (mi >> 1), 16 * ks + 8 * (mi & 1)), bb[0],
                            bb[1], bb[2], bb[3]);
                    mma_f16(acc2[2 * np], a, bb[0], bb[1]);
                    mma_f16(acc2[2 * np + 1], a, bb[2], bb[3]);
                }
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&sfree[b]);
                mbar_arrive(&empty[sg]);
            }
            // each row of `out` directly (within the sequence)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int i = 16 * wr + g + 8 * hh;
                if (R.outputs && lc * C + i < len) {
                    const size_t t = (size_t)(tok0 + lc * C + i);
                    __nv_bfloat16* orow = p.out + (t * p.H + h) * D + v0;
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        const uint32_t pv = pack_bf162(acc[nt][2 * hh] + acc2[nt][2 * hh],
                                                       acc[nt][2 * hh + 1] + acc2[nt][2 * hh + 1]);
                        *reinterpret_cast<uint32_t*>(orow + 8 * nt + 2 * tq) = pv;
                    }
                }
            }
        }
        return;
    }

    // ======================= state warps ====================================
    const int wr = warp;  // key channels 32wr..32wr+31 of S^T
    // The state warps meet on a named barrier twice per chunk.  A warp whose
    // wait gave up raises the shared abort flag before the barrier; all of them
    // read it after the same barrier, so they leave the walk together (the
    // read's latency is hidden behind the next products, the test comes after).
    auto state_sync = [&]() { asm volatile("bar.sync 1, 128;" ::: "memory"); };
    auto state_sync_flag = [&](bool failed_here) -> int {
        if (failed_here) *abort_flag = 1;
        state_sync();
        return *abort_flag;
    };

    bool has_init = R.init == 0 && (p.has_init ? (p.has_init[n] != 0) : (p.st_in != nullptr));
    const int64_t in_slot = p.st_in_idx ? p.st_in_idx[n] : n;
    const int64_t out_slot = p.st_out_idx ? p.st_out_idx[n] : n;
    bool store_ok = R.final_state;
    if (p.num_slots > 0) {  // a slot outside the pool: no access, reported
        const bool bad_in = has_init && (in_slot < 0 || in_slot >= p.num_slots);
        const bool bad_out = R.final_state && !R.final_buf && (out_slot < 0 || out_slot >= p.num_slots);
        if ((bad_in || bad_out) && wr == 0 && lane == 0 && p.status) atomicOr(p.status, 4);
        if (bad_in) has_init = false;
        if (bad_out) store_ok = false;
    }
    const size_t in_base = has_init ? (size_t)in_slot * p.st_in_stride + (size_t)h * D * D : 0;
    const size_t out_base = store_ok ? (size_t)out_slot * p.st_out_stride + (size_t)h * D * D : 0;

    float Sm[2][NT][4];  // [mt][nt][e]: k = 32wr+16mt+g+8(e>>1), v = 8nt+2tq+(e&1)
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int kk = 32 * wr + 16 * mt + g + 8 * (e >> 1);
                const int vv = v0 + 8 * nt + 2 * tq + (e & 1);
                Sm[mt][nt][e] =
                    has_init     ? load_state(p.st_in, p.st_dtype, in_base + (size_t)vv * D + kk)
                    : R.init == 2 ? (kk == vv ? 1.f : 0.f)
                    : R.init == 3 ? R.init_buf[(size_t)vv * D + kk]
                                  : 0.f;
            }

    // S (fp16) into ring slot b: S^T fragments stored transposed as S[v][k].
    auto write_s16 = [&](int b) {
        const uint32_t s16 = s16_slot(b);
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int np = 0; np < NT / 2; ++np) {
                // matrices (n-tile 2np + (mi >> 1), key half mi & 1): rows v, columns k
                const int vrow = 16 * np + 8 * (mi >> 1) + rr;
                const int kcol = 32 * wr + 16 * mt + 8 * (mi & 1);
                stsm_x4_t(s16 + sw128_off(vrow, kcol, VS),
                          pack_half2(Sm[mt][2 * np][0], Sm[mt][2 * np][1]),
                          pack_half2(Sm[mt][2 * np][2], Sm[mt][2 * np][3]),
                          pack_half2(Sm[mt][2 * np + 1][0], Sm[mt][2 * np + 1][1]),
                          pack_half2(Sm[mt][2 * np + 1][2], Sm[mt][2 * np + 1][3]));
            }
    };
    // S as the B operand of U = w S^T, [ks][nt][b0, b1]: loaded once after S is
    // published
    uint32_t Sf[8][NT][2];
    auto load_sfrag = [&](int b) {
        const uint32_t s16 = s16_slot(b);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
#pragma unroll
            for (int np = 0; np < NT / 2; ++np)
                ldsm_x4(s16 + sw128_off(16 * np + rr + 8 * (mi >> 1), 16 * ks + 8 * (mi & 1), VS),
                        Sf[ks][2 * np][0], Sf[ks][2 * np][1], Sf[ks][2 * np + 1][0],
                        Sf[ks][2 * np + 1][1]);
    };

    grid_dep_wait();  // the state came from the pool; the chunks come after
    write_s16(0);
    state_sync();
    load_sfrag(0);

    bool failed = false;
    for (int lc = 0; lc < nch; ++lc) {
        const int b = lc % kRing, sg = lc % kStages;
        const bool ok = mbar_wait(&full[sg], (lc / kStages) & 1);  // voted below, before any write
        const uint32_t st = stage_base(sg);
        const uint32_t tw = st + kWsWOff, tkg = st + kWsKGOff;
        const float* gam = reinterpret_cast<const float*>(smem + sg * L::kStage + kWsGammaOff);
        const uint32_t tu = st + L::kSharedPad;  // [VS/16][64][16] fp16
        const uint32_t ut = ut_slot(b);

        // U = u - w S^T for chunk rows 16wr..16wr+15 (two chains over the key halves)
        float accU[NT][4] = {}, accU2[NT][4] = {};
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            uint32_t a[4];
            ldsm_x4(tw + sw128_off(16 * wr + rr + 8 * (mi & 1), 16 * ks + 8 * (mi >> 1), 64), a[0],
                    a[1], a[2], a[3]);
            float (*d)[4] = (ks & 1) ? accU2 : accU;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma_f16(d[nt], a, Sf[ks][nt][0], Sf[ks][nt][1]);
        }
        uint32_t uf[NT][2];  // U as fp16 pairs: [nt][rows g, g + 8]
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int i = 16 * wr + g + 8 * hh;
                const int vv = 8 * nt + 2 * tq;
                uint32_t uv;
                asm volatile("ld.shared.b32 %0, [%1];"
                             : "=r"(uv)
                             : "r"(tu + (vv >> 4) * kWsUSliceBytes + (i * 16 + (vv & 15)) * 2));
                const float2 u2 = R.zero_u ? make_float2(0.f, 0.f)
                                           : __half22float2(*reinterpret_cast<__half2*>(&uv));
                const float x0 = u2.x - accU[nt][2 * hh] - accU2[nt][2 * hh];
                const float x1 = u2.y - accU[nt][2 * hh + 1] - accU2[nt][2 * hh + 1];
                uf[nt][hh] = pack_half2(x0, x1);
            }
        // U^T into ring slot b (rows v, columns c): stmatrix transposes 8x8 blocks
#pragma unroll
        for (int np = 0; np < NT / 2; ++np) {
            const int vrow = 16 * np + 8 * (mi >> 1) + rr;
            const int ccol = 16 * wr + 8 * (mi & 1);
            stsm_x4_t(ut + sw64_off(vrow, ccol), uf[2 * np][0], uf[2 * np][1], uf[2 * np + 1][0],
                      uf[2 * np + 1][1]);
        }
        // kg^T fragments of the update, loaded before the barrier (they do not
        // depend on U) so that their latency overlaps the wait
        uint32_t kga[4][2][4];
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
                ldsm_x4_t(tkg + sw128_off(16 * ks + rr + 8 * (mi >> 1), 32 * wr + 16 * mt + 8 * (mi & 1), 64),
                          kga[ks][mt][0], kga[ks][mt][1], kga[ks][mt][2], kga[ks][mt][3]);
        const int abort1 = state_sync_flag(!ok);  // a copy never landed (tested below)
        if (tid == 0) mbar_arrive(&sready[b]);  // S (published last step) and U of this chunk

        // dS^T = kg^T U for key channels 32wr..32wr+31; S = gamma S + dS
        {
            float accS[2][NT][4] = {};
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                uint32_t bb[NT][2];
#pragma unroll
                for (int np = 0; np < NT / 2; ++np)
                    ldsm_x4(ut + sw64_off(16 * np + rr + 8 * (mi >> 1), 16 * ks + 8 * (mi & 1)),
                            bb[2 * np][0], bb[2 * np][1], bb[2 * np + 1][0], bb[2 * np + 1][1]);
#pragma unroll
                for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) mma_f16(accS[mt][nt], kga[ks][mt], bb[nt][0], bb[nt][1]);
            }
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const float gk = gam[32 * wr + 16 * mt + g + 8 * hh];
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        Sm[mt][nt][2 * hh] = gk * Sm[mt][nt][2 * hh] + accS[mt][nt][2 * hh];
                        Sm[mt][nt][2 * hh + 1] = gk * Sm[mt][nt][2 * hh + 1] + accS[mt][nt][2 * hh + 1];
                    }
                }
        }
        if (abort1) {  // report, stop the walk
            failed = true;
            if (tid == 0 && p.status) atomicOr(p.status, 1);
            break;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[sg]);  // w, kg, gamma and u of this stage are read

        // publish the next chunk's incoming S in the next slot once the output
        // warps are done with the chunk that used it (kRing - 1 chunks back;
        // that also frees the slot the next chunk's U goes to)
        const int nb = (lc + 1) % kRing;
        bool ok2 = true;
        if (lc >= kRing - 1) ok2 = mbar_wait(&sfree[nb], ((lc + 1 - kRing) / kRing) & 1);
        if (ok2) write_s16(nb);
        const int abort2 = state_sync_flag(!ok2);
        load_sfrag(nb);
        if (abort2) {
            failed = true;
            if (tid == 0 && p.status) atomicOr(p.status, 1);
            break;
        }
    }
    if (failed || !store_ok) return;

#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int kk = 32 * wr + 16 * mt + g + 8 * (e >> 1);
                const int vv = v0 + 8 * nt + 2 * tq + (e & 1);
                if (R.final_buf)
                    R.final_buf[(size_t)vv * D + kk] = Sm[mt][nt][e];
                else
                    store_state(p.st_out, p.st_dtype, out_base + (size_t)vv * D + kk, Sm[mt][nt][e]);
            }
}

}  // namespace scan
}  // namespace kda
