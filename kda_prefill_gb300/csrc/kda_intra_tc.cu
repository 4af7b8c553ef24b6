// Intra-chunk kernel on tensor cores: one persistent CTA per SM (512 threads),
// each taking (chunk, head) items in chunk-major order.
//
// Per item (C = 64 tokens of one head), fused:
//   prep   q^ = q / |q| / sqrt(K),  k^ = k / |k|,  a = e^{lb*sigmoid(g_raw)},
//          b = sigmoid(beta_raw); rows past the sequence end get q^ = k^ = 0,
//          a = 1, b = 0 (an exact no-op).
//   tiles  A_qk[i][j] = sum_c q^_ic k^_jc e^{G_ic - G_jc} (j <= i),
//          A_kk[i][j] = b_i sum_c k^_ic k^_jc e^{G_ic - G_jc} (j < i).
//   solve  w = (I + A_kk)^{-1} (b k^ e^G),  u = (I + A_kk)^{-1} (b v),
//          plus qg = q^ e^G, kg = k^ e^{G_C - G}, gamma = e^{G_C}.
// (ROCm/aiter PR #4741, "Summary" and "Optimizations Applied": the prep pass
// with L2 norm, gate and beta folded in, the intra-chunk tiles built so that no
// decay factor overflows, the triangular solve and the w/u recompute.)
//
// Bounded tiles.  The chunk is cut into four 16-row blocks.  With P the
// cumulative decay product inside a block (P_r = product of a over the block up
// to row r) and E_B the total of block B, a pair (i in block I, j in block J < I)
// is  e^{G_i - G_j} = P_i * (E_{J+1} ... E_{I-1}) * (E_J / P_j): three factors
// that are all <= 1, so nothing overflows and an underflow only drops values
// below 1e-38.  Off-diagonal blocks run as fp16 MMAs (m16n8k16) on those
// factored operands.  Inside a diagonal block e^{G_i - G_j} = P_i / P_j; with
// lower_bound >= -5 a block holds at most 80 nats of decay, so P >= e^-80 and
// 1/P stay in fp32 range, and these blocks run as tf32 MMAs (m16n8k8) on fp32
// operand tiles for the extra mantissa the near-diagonal entries need.
//
// The decay pass runs on all warps, a thread taking 8 rows (half a block) of two
// channels; the halves exchange their products, and the rows' sums of squares
// (for the norms) are reduced in-warp and exchanged at the same barrier.
//
// The solve forms T = (I + A_kk)^{-1} in full: the 16x16 inverses T_II by
// forward substitution in registers (one warp per block), then the blocks below
// the diagonal column by column, T_IJ = T_II sum_{J<=m<I} (-A_Im) T_mJ, by three
// warps while the others form X = b k^ e^G; [w | u] = T [X | b v] is then one
// K = 64 product on the tensor cores (tcgen05, accumulators in tensor memory).
//
// Data movement: inputs by TMA tiled loads (3-D tensor maps over [T][H][128],
// 128-byte swizzle); the next item's q, k, g are loaded as soon as the decay
// pass has consumed the current ones, v one item ahead.  qg and kg go out from
// the decay pass as fp16 pairs (a warp writes 128 contiguous bytes of a row);
// w, u and A_qk are staged in shared memory in their workspace layout and
// written by TMA bulk stores.
//
// The item loop is a device function shared by this kernel (static item
// assignment) and the fused intra + scan launch at the end of the file, whose
// CTAs take items and scan walks from one queue.

#include <cuda.h>

#include <atomic>

#include "kda_device.cuh"
#include "kda_internal.h"
#include "kda_scan_walk.cuh"

namespace kda {

cudaError_t launch_intra_exact(const FwdParams& p, cudaStream_t s);

namespace {

using namespace dev;

constexpr int C = kC;
constexpr int kThreads = 512;

// Shared-memory layout (bytes).
constexpr int kQ = 0;          // q bf16 [64][128] (TMA, swizzled halves)
constexpr int kK = 16384;      // k bf16
constexpr int kG = 32768;      // g_raw fp32 [64][128] (TMA, swizzled quarters), or bf16 (halves, 16 KB)
constexpr int kV = 65536;      // v bf16 -> b v fp16 -> u (in place)
constexpr int kLq32 = 81920;   // q^ P fp32 [64][128]; later u for the store ([8][64][16])
constexpr int kLk32 = 114688;  // k^ P fp32 [64][128]
constexpr int kRd32 = 147456;  // k^ / P fp32 [64][128]; later A_qk, -A_kk, A_kk diag, T_II
constexpr int kLQ = 180224;    // q^ P fp16, rows 16..63 ([48][128]); later w ([64][128]) for the store
constexpr int kLK = 192512;    // k^ P fp16, rows 16..63 ([48][128])
constexpr int kRO = 204800;    // k^ E_B/P fp16, rows 0..63 ([64][128])
constexpr int kSc = 221184;    // beta[64] | NS [16][16] | F1 [4][128] | HT [4][2][128] (fp32) | E_1, E_2
constexpr int kMid = kSc + 256 + 1024 + 2048 + 4096;  // E_1, E_2 fp16 [2][128]
constexpr int kBar = kMid + 512;
constexpr int kSmemBytes = kBar + 64;
// the fused launch runs scan walks in the same shared memory
static_assert(scan::ScanSmem<2>::kTotal <= kSmemBytes, "a walk fits in the intra kernel's shared memory");
// Reuse of the k^/P area after the tile MMAs:
constexpr int kAqkStage = kRd32;          // A_qk fp16 [64][64] tile, to store (8 KB)
constexpr int kNAk = kRd32 + 8192;        // -A_kk off-diagonal blocks, fp16 [64][64] (8 KB)
constexpr int kAkd = kRd32 + 16384;       // A_kk diagonal blocks, fp32 [4][16][16] (4 KB)
constexpr int kT16 = kRd32 + 20480;       // T = (I + A_kk)^{-1}, fp16 [64][64] tile (8 KB)
// After the tile MMAs the k^ E_B / P area holds X = b k^ e^G (fp16 [64][128]).
constexpr int kX = kRO;

// Tensor memory of the w / u product: [w | u] = T [X | Y], an M = 64 product
// with fp32 accumulators: chunk rows 16 q .. 16 q + 15 sit in lanes 0..15 of
// lane quarter q (lanes 32 q ..), columns 0..127 w, 128..255 u.
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kIdescWU = mma_idesc(0, 0, 1, 64, 128);  // fp16; A K-major, B MN-major

struct IntraMaps {
    CUtensorMap q, k, v, g;
};


// Nearest tf32 value (ties away from zero) of x, as its fp32 bit pattern (the
// 13 bits below tf32 precision zero): one conversion instruction, which gives
// the same bits as adding half a tf32 unit in the last place to the magnitude
// and clearing those 13 bits (checked over 2^26 finite patterns on GB300).
__device__ __forceinline__ uint32_t tf32_bits(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ uint2 tf32_bits2(float2 x) { return make_uint2(tf32_bits(x.x), tf32_bits(x.y)); }

// 2^x by the special-function unit (approximate; subnormal results flushed)
__device__ __forceinline__ float ex2_approx(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// Channel pairs: the decay pass holds two channels of a row as a float2 and
// works on both with one packed fp32 instruction (sm_100 and later).
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 splat2(float x) { return make_float2(x, x); }
__device__ __forceinline__ uint32_t pack_half2v(float2 x) { return pack_half2(x.x, x.y); }

// Marks a (chunk, head) block as written for the fused launch's scan walks: the
// block's bulk stores have completed (cp.async.bulk.wait_group 0 by this
// thread) and the CTA's other stores to it came before a CTA barrier.
__device__ __forceinline__ void publish_ready(int* flag) {
    asm volatile("fence.proxy.async.global;" ::: "memory");
    __threadfence();
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(flag), "r"(1) : "memory");
}

// Item claims of the standalone launch: item blockIdx.x, then every
// gridDim.x-th.
struct StaticClaims {
    __device__ int first() { return blockIdx.x; }
    __device__ void claim() {}
    __device__ int next(int it) { return it + gridDim.x; }
};

// Off-diagonal block pairs in order (1,0) (2,0) (2,1) (3,0) (3,1) (3,2).
__device__ __forceinline__ void pair_of(int pi, int& I, int& J) {
    I = pi < 1 ? 1 : (pi < 3 ? 2 : 3);
    J = pi - I * (I - 1) / 2;
}

// Block column J of T = (I + A_kk)^{-1} below the diagonal, by one warp:
// T_IJ = T_II sum_{J<=m<I} (-A_Im) T_mJ for I = J+1..3, formed in transposed
// form (T_IJ^T = (sum_m T_mJ^T (-A_Im)^T) T_II^T) so that each result is
// already the A fragment of the next product; the warp also zeroes the blocks
// above the diagonal in row J.  Reads -A_kk (off-diagonal, fp16) and the T_II
// diagonal blocks from their tiles, writes T_IJ into the T tile.  Every operand
// fragment is loaded first and the products that need only T_JJ come before the
// dependent chain T_{J+1,J} -> T_{J+2,J} -> T_{J+3,J}.
template <int J>
__device__ __forceinline__ void t_column(uint8_t* smem, int lane) {
    const int mi = lane >> 3, rr = lane & 7;
    const uint32_t nak = smem_u32(smem + kNAk), t16 = smem_u32(smem + kT16);
    uint32_t tf[4][4];  // T_mJ^T as fp16 A fragments, m = J..3
    ldsm_x4_t(t16 + sw64_off(16 * J + 8 * (mi >> 1) + rr, 16 * J + 8 * (mi & 1)), tf[J][0], tf[J][1],
              tf[J][2], tf[J][3]);
    uint32_t nb[4][4][4];  // (-A_Im)^T B fragments, [I][m]
    uint32_t tb[4][4];     // T_II^T B fragments
#pragma unroll
    for (int I = J + 1; I < 4; ++I) {
#pragma unroll
        for (int m = J; m < I; ++m)
            ldsm_x4(nak + sw64_off(16 * I + 8 * (mi >> 1) + rr, 16 * m + 8 * (mi & 1)), nb[I][m][0],
                    nb[I][m][1], nb[I][m][2], nb[I][m][3]);
        ldsm_x4(t16 + sw64_off(16 * I + 8 * (mi >> 1) + rr, 16 * I + 8 * (mi & 1)), tb[I][0], tb[I][1],
                tb[I][2], tb[I][3]);
    }
    float acc[4][2][4];
#pragma unroll
    for (int I = J + 1; I < 4; ++I) {  // the terms with T_JJ (m = J)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[I][nt][e] = 0.f;
        mma_f16(acc[I][0], tf[J], nb[I][J][0], nb[I][J][1]);
        mma_f16(acc[I][1], tf[J], nb[I][J][2], nb[I][J][3]);
    }
#pragma unroll
    for (int I = J + 1; I < 4; ++I) {
        const uint32_t ra[4] = {pack_half2(acc[I][0][0], acc[I][0][1]), pack_half2(acc[I][0][2], acc[I][0][3]),
                                pack_half2(acc[I][1][0], acc[I][1][1]), pack_half2(acc[I][1][2], acc[I][1][3])};
        float tv[2][4] = {};
        mma_f16(tv[0], ra, tb[I][0], tb[I][1]);
        mma_f16(tv[1], ra, tb[I][2], tb[I][3]);
        tf[I][0] = pack_half2(tv[0][0], tv[0][1]);
        tf[I][1] = pack_half2(tv[0][2], tv[0][3]);
        tf[I][2] = pack_half2(tv[1][0], tv[1][1]);
        tf[I][3] = pack_half2(tv[1][2], tv[1][3]);
#pragma unroll
        for (int I2 = I + 1; I2 < 4; ++I2) {  // T_IJ's term in the later blocks
            mma_f16(acc[I2][0], tf[I], nb[I2][I][0], nb[I2][I][1]);
            mma_f16(acc[I2][1], tf[I], nb[I2][I][2], nb[I2][I][3]);
        }
        stsm_x4_t(t16 + sw64_off(16 * I + 8 * (mi >> 1) + rr, 16 * J + 8 * (mi & 1)), tf[I][0], tf[I][1],
                  tf[I][2], tf[I][3]);
        // block (J, I) above the diagonal is zero
        *reinterpret_cast<uint4*>(smem + kT16 + sw64_off(16 * J + (lane >> 1), 16 * I + 8 * (lane & 1))) =
            make_uint4(0u, 0u, 0u, 0u);
    }
}

// Hand-off of the solve's blocks from the warps that put or invert them (warps
// 3..9 arrive) to the warps that form T's block columns (warps 0..2 wait), on
// named barrier 1, so that T is formed while the other warps form X.  An arrive
// orders the arriving warp's earlier shared stores before the waiters' later
// loads, as a CTA barrier does.
constexpr int kSolveBarThreads = 320;
constexpr int kStoreTid = kThreads - 32;  // issues the bulk stores (lane 0 of warp 15)
__device__ __forceinline__ void solve_bar_wait() {
    asm volatile("bar.sync 1, %0;" ::"n"(kSolveBarThreads) : "memory");
}
__device__ __forceinline__ void solve_bar_arrive() {
    asm volatile("bar.arrive 1, %0;" ::"n"(kSolveBarThreads) : "memory");
}

// The intra-chunk items of one CTA, in the order `cl` hands them out (all
// threads call cl.first() once and, per item, cl.claim() before and cl.next()
// after a CTA barrier).  RAW16: raw gate and beta in bf16 (the gate tile then
// takes 16 KB of the g area, laid out like q and k) instead of fp32.
template <bool RAW16, class Claims>
__device__ __forceinline__ void intra_items(const IntraMaps& maps, const FwdParams& p, uint8_t* smem,
                                            Claims& cl) {
    float* beta = reinterpret_cast<float*>(smem + kSc);
    float* NS = beta + 64;  // [16 warps][16] row sums of squares over each warp's 64 channels
    float* F1 = NS + 256;   // [4][128] decay of the blocks before B (e^G at the block start)
    float* HT = F1 + 512;   // [4][2][128] decay product of each 8-row half block
    __half* MIDh = reinterpret_cast<__half*>(smem + kMid);     // [2][128] E_1, E_2 in fp16
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kBar);  // [0] q,k,g  [1] v  [2] w MMA
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + kBar + 24);  // tensor-memory base
    uint64_t* bar_u = reinterpret_cast<uint64_t*>(smem + kBar + 40);  // u MMA
    // raised before a CTA barrier by a thread whose bounded wait gave up, read by
    // every thread after it, so that all leave the item loop together
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kBar + 48);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int g8 = lane >> 2, tq = lane & 3;
    const int mi = lane >> 3, rr = lane & 7;
    const int H = p.H;
    const int n_items = p.n_chunks * H;
    const float lb = p.lower_bound;

    if ((smem_u32(smem) & 1023) != 0) {  // swizzled TMA tiles need 1 KB alignment
        if (tid == 0 && p.status) atomicOr(p.status, 2);
        return;
    }
    if (tid == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        mbar_init(&bar[2], 1);
        mbar_init(bar_u, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&maps.q);
        prefetch_tmap(&maps.k);
        prefetch_tmap(&maps.v);
        prefetch_tmap(&maps.g);
    }
    if (warp == 0) tmem_alloc(tslot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    // TMA issue (one thread).
    auto issue_inputs = [&](int it, int t0) {
        const int h = it % H;
        mbar_arrive_expect_tx(&bar[0], RAW16 ? 49152 : 65536);
        tma_load_3d(smem + kQ, &maps.q, &bar[0], 0, h, t0);
        tma_load_3d(smem + kQ + 8192, &maps.q, &bar[0], 64, h, t0);
        tma_load_3d(smem + kK, &maps.k, &bar[0], 0, h, t0);
        tma_load_3d(smem + kK + 8192, &maps.k, &bar[0], 64, h, t0);
        if (RAW16) {
            tma_load_3d(smem + kG, &maps.g, &bar[0], 0, h, t0);
            tma_load_3d(smem + kG + 8192, &maps.g, &bar[0], 64, h, t0);
        } else {
#pragma unroll
            for (int qt = 0; qt < 4; ++qt)
                tma_load_3d(smem + kG + qt * 8192, &maps.g, &bar[0], 32 * qt, h, t0);
        }
    };
    auto issue_v = [&](int it, int t0) {
        const int h = it % H;
        mbar_arrive_expect_tx(&bar[1], 16384);
        tma_load_3d(smem + kV, &maps.v, &bar[1], 0, h, t0);
        tma_load_3d(smem + kV + 8192, &maps.v, &bar[1], 64, h, t0);
    };
    // first token and valid length of an item's chunk
    auto item_tok = [&](int it) { return p.chunk_tok[it / H]; };
    auto item_len = [&](int it, int t0) { return min(C, p.cu[p.chunk_seq[it / H] + 1] - t0); };

    // A tile results of one warp into place: sel 0 = A_qk (to the staging tile,
    // j <= i), sel 1 = A_kk (diagonal block in fp32, column-major, with j < i;
    // off-diagonal blocks negated in fp16).
    auto put = [&](int sel, int tI, int tJ, const float (&acc)[2][4]) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int i = 16 * tI + g8 + 8 * hh;
                const int j = 16 * tJ + 8 * nt + 2 * tq;
                float x0 = acc[nt][2 * hh], x1 = acc[nt][2 * hh + 1];
                if (sel == 0) {
                    if (tI == tJ) {
                        if (j > i) x0 = 0.f;
                        if (j + 1 > i) x1 = 0.f;
                    }
                    *reinterpret_cast<uint32_t*>(smem + kAqkStage + sw64_off(i, j)) = pack_half2(x0, x1);
                } else if (tI == tJ) {  // column-major: d[j][i] = A_kk[i][j]
                    float* d = reinterpret_cast<float*>(smem + kAkd) + tI * 256;
                    const float bi = beta[i];
                    d[(j & 15) * 16 + (i & 15)] = (j >= i) ? 0.f : bi * x0;
                    d[((j + 1) & 15) * 16 + (i & 15)] = (j + 1 >= i) ? 0.f : bi * x1;
                } else {
                    const float bi = -beta[i];
                    *reinterpret_cast<uint32_t*>(smem + kNAk + sw64_off(i, j)) =
                        pack_half2(bi * x0, bi * x1);
                }
            }
    };

    const int first = cl.first();
    int tok_next = 0, len_next = 0;
    float braw_next = 0.f;
    if (first < n_items) {
        tok_next = item_tok(first);
        len_next = item_len(first, tok_next);
        if (tid == 0) {
            issue_inputs(first, tok_next);
            issue_v(first, tok_next);
        }
        if (tid < len_next) braw_next = load_raw(p.beta_raw, RAW16, (size_t)(tok_next + tid) * H + first % H);
    }

    int n_local = 0, prev = -1;
    for (int it = first; it < n_items; ++n_local) {
        const int len = len_next;
        const float braw = braw_next;
        uint8_t* blk = p.ws + (size_t)it * kWsBytes;
        int nxt = n_items;  // the next item, read after part 1's barrier
        cl.claim();

        // the inputs' wait gives up only if a copy never lands; part 1 then works
        // on stale data and the loop stops at part 1's barrier
        const bool ok_in = mbar_wait(&bar[0], n_local & 1);

        // ---- decay pass, all warps: thread (block B, row half hf, channels c0,
        //      c0 + 1) over 8 rows.  Part 1: a = e^{lb sigmoid(g)}, the half's
        //      product, q and k kept in registers, and the rows' sums of squares
        //      over the warp's 64 channels; the halves exchange their products
        //      and the two warps of a row their sums.  Part 2: row norms,
        //      forward P (q^ P and k^ P: tf32 for the
        //      diagonal tiles, fp16 for the off-diagonal left operands, qg =
        //      q^ e^G to the workspace), backward R = product of a after the row
        //      in the block (k^ R / E_B in tf32, k^ R in fp16, kg = k^ e^{G_C - G}
        //      to the workspace).
        {
            const int B = warp >> 2, hf = (warp >> 1) & 1;
            const int c0 = 64 * (warp & 1) + 2 * lane;
            const int rb = 16 * B + 8 * hf;
            float2 a[8], q[8], k[8];  // the two channels' gate factors and (normed) q, k
            float2 Lh = make_float2(1.f, 1.f);
            const float2 m_log2e = splat2(-1.4426950408889634f), lb_log2e = splat2(lb * 1.4426950408889634f);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int r = rb + i;
                float2 gr;
                if (RAW16) {
                    const uint32_t gw = *reinterpret_cast<const uint32_t*>(smem + kG + sw128_off(r, c0, 64));
                    gr = make_float2(__uint_as_float(gw << 16), __uint_as_float(gw & 0xffff0000u));
                } else {
                    gr = *reinterpret_cast<const float2*>(smem + kG + sw128f_off(r, c0, 64));
                }
                const bool valid = r < len;
                // sigmoid of both channels from one reciprocal: with d = 1 + e^{-g}
                // (g clamped to [-40, 40], where sigmoid is 0 or 1 to fp32 precision,
                // so d0 d1 stays finite), s0 = d1 / (d0 d1) and s1 = d0 / (d0 d1);
                // e^x is taken as 2^(x log2 e)
                const float2 t = mul2(make_float2(fminf(fmaxf(gr.x, -40.f), 40.f),
                                                  fminf(fmaxf(gr.y, -40.f), 40.f)), m_log2e);
                const float2 d = __fadd2_rn(make_float2(ex2_approx(t.x), ex2_approx(t.y)), splat2(1.f));
                const float rd = __fdividef(1.f, d.x * d.y);
                const float2 e = mul2(mul2(make_float2(d.y, d.x), splat2(rd)), lb_log2e);
                a[i] = valid ? make_float2(ex2_approx(e.x), ex2_approx(e.y)) : make_float2(1.f, 1.f);
                Lh = mul2(Lh, a[i]);
                const uint32_t o16 = sw128_off(r, c0, 64);
                const uint32_t qw = *reinterpret_cast<const uint32_t*>(smem + kQ + o16);
                const uint32_t kw = *reinterpret_cast<const uint32_t*>(smem + kK + o16);
                q[i] = make_float2(__uint_as_float(qw << 16), __uint_as_float(qw & 0xffff0000u));
                k[i] = make_float2(__uint_as_float(kw << 16), __uint_as_float(kw & 0xffff0000u));
            }
            *reinterpret_cast<float2*>(HT + (2 * B + hf) * 128 + c0) = Lh;
            {
                // sums of squares of the 8 rows (value 2i: q, 2i + 1: k) over the
                // warp's 64 channels: a halving butterfly leaves value lane / 2 in
                // lanes 2v and 2v + 1
                float x[16];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    x[2 * i] = fmaf(q[i].x, q[i].x, q[i].y * q[i].y);
                    x[2 * i + 1] = fmaf(k[i].x, k[i].x, k[i].y * k[i].y);
                }
#pragma unroll
                for (int w = 8; w >= 1; w >>= 1) {  // lane bit 16, 8, 4, 2
                    const bool up = (lane & (2 * w)) != 0;
#pragma unroll
                    for (int j = 0; j < w; ++j) {
                        const float send = up ? x[j] : x[j + w];
                        const float keep = up ? x[j + w] : x[j];
                        x[j] = keep + __shfl_xor_sync(0xffffffffu, send, 2 * w);
                    }
                }
                x[0] += __shfl_xor_sync(0xffffffffu, x[0], 1);
                if ((lane & 1) == 0) NS[warp * 16 + (lane >> 1)] = x[0];
            }
            if (tid < C) beta[tid] = (tid < len) ? __fdividef(1.f, 1.f + __expf(-braw)) : 0.f;
            // the previous item's bulk stores must have read the staging areas
            // (u in the q^P area, A_qk in the k^/P area, w in the LQ area) before
            // part 2 rewrites them (their completion, for the fused launch's ready
            // flag, is awaited during the tiles, off the CTA's barriers)
            if (tid == kStoreTid) bulk_wait_read_all();
            if (!ok_in) *abort_flag = 1;
            __syncthreads();
            if (*abort_flag) {  // uniform: every thread reads the flag after the barrier
                if (tid == 0 && p.status) atomicOr(p.status, 1);
                break;
            }
            // the claim made at the item's start is visible after the barrier
            nxt = cl.next(it);
            // the next item's chunk metadata, loaded while this one runs
            if (nxt < n_items) {
                tok_next = item_tok(nxt);
                len_next = item_len(nxt, tok_next);
            }
            {
                // row norms: lane 2v (v = 2i + s) forms the norm factor of value v
                // (row i, s = 0: q with 1/sqrt(K), 1: k), then all lanes take theirs
                const int v = lane >> 1;
                const float ssum = NS[warp * 16 + v] + NS[(warp ^ 1) * 16 + v];
                float nf = (rb + (v >> 1) < len) ? rsqrtf(ssum + 1e-6f) : 0.f;
                if ((v & 1) == 0) nf *= 0.08838834764831845f;  // 1/sqrt(128)
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float sq = __shfl_sync(0xffffffffu, nf, 4 * i);
                    const float sk = __shfl_sync(0xffffffffu, nf, 4 * i + 2);
                    q[i] = mul2(q[i], splat2(sq));
                    k[i] = mul2(k[i], splat2(sk));
                }
            }
            // block totals E_m = (first half) x (second half); F1 = product over
            // blocks before B, F2 = product over blocks after B
            float2 E[4];
#pragma unroll
            for (int m = 0; m < 4; ++m)
                E[m] = mul2(*reinterpret_cast<const float2*>(HT + (2 * m) * 128 + c0),
                            *reinterpret_cast<const float2*>(HT + (2 * m + 1) * 128 + c0));
            float2 f1 = make_float2(1.f, 1.f), f2 = make_float2(1.f, 1.f);
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                if (m < B) f1 = mul2(f1, E[m]);
                if (m > B) f2 = mul2(f2, E[m]);
            }
            const float2 own0 = *reinterpret_cast<const float2*>(HT + (2 * B) * 128 + c0);
            const float2 own1 = *reinterpret_cast<const float2*>(HT + (2 * B + 1) * 128 + c0);
            const float2 eb = mul2(own0, own1);
            if (hf == 0) {
                *reinterpret_cast<float2*>(F1 + B * 128 + c0) = f1;
                if (B == 1 || B == 2)
                    *reinterpret_cast<uint32_t*>(MIDh + (B - 1) * 128 + c0) = pack_half2v(eb);
                if (B == 0) *reinterpret_cast<float2*>(blk + kWsGammaOff + 4 * c0) = mul2(eb, f2);
            }
            // forward: P_i = (first-half product, for the second half) x prefix
            float2 P = hf ? own0 : make_float2(1.f, 1.f);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int r = rb + i;
                P = mul2(P, a[i]);
                const float2 x = mul2(q[i], P), l = mul2(k[i], P);
                const uint32_t o32 = sw128f_off(r, c0, 64);
                *reinterpret_cast<uint2*>(smem + kLq32 + o32) = tf32_bits2(x);
                *reinterpret_cast<uint2*>(smem + kLk32 + o32) = tf32_bits2(l);
                if (B >= 1) {
                    const uint32_t h16 = sw128_off(r - 16, c0, 48);
                    *reinterpret_cast<uint32_t*>(smem + kLQ + h16) = pack_half2v(x);
                    *reinterpret_cast<uint32_t*>(smem + kLK + h16) = pack_half2v(l);
                }
                *reinterpret_cast<uint32_t*>(blk + kWsQGOff + sw128_off(r, c0, 64)) = pack_half2v(mul2(x, f1));
            }
            // backward: R_i = product of a after row i in the block
            const float2 ie = make_float2(__fdividef(1.f, eb.x), __fdividef(1.f, eb.y));
            float2 R = hf ? make_float2(1.f, 1.f) : own1;
#pragma unroll
            for (int i = 7; i >= 0; --i) {
                const int r = rb + i;
                const float2 x = mul2(k[i], R);
                *reinterpret_cast<uint2*>(smem + kRd32 + sw128f_off(r, c0, 64)) = tf32_bits2(mul2(x, ie));
                const uint32_t o16 = sw128_off(r, c0, 64);
                *reinterpret_cast<uint32_t*>(smem + kRO + o16) = pack_half2v(x);
                *reinterpret_cast<uint32_t*>(blk + kWsKGOff + o16) = pack_half2v(mul2(x, f2));
                R = mul2(R, a[i]);
            }
        }
        __syncthreads();
        // q, k, g of this item are consumed: load the next item's now
        if (tid == kThreads - 32 && nxt < n_items) issue_inputs(nxt, tok_next);

        // ---- A tiles: diagonal blocks (warps 0-3, tf32: block I = warp, A_qk and
        //      A_kk sharing the right operand), off-diagonal block pairs (warps
        //      4-9, fp16, likewise), b v (warps 10-14) and the previous item's
        //      ready flag (warp 15) ----------------------------------------------
        float acc[2][2][4] = {};  // [0]: q-left (A_qk), [1]: k-left (A_kk)
        if (warp < 4) {
            const int I = warp;
            const uint32_t Lq = smem_u32(smem + kLq32), Lk = smem_u32(smem + kLk32);
            const uint32_t Rb = smem_u32(smem + kRd32);
#pragma unroll 8
            for (int ks = 0; ks < 16; ++ks) {
                uint32_t aq[4], ak[4], b4[4];
                const uint32_t ao = sw128f_off(16 * I + rr + 8 * (mi & 1), 8 * ks + 4 * (mi >> 1), 64);
                ldsm_x4(Lq + ao, aq[0], aq[1], aq[2], aq[3]);
                ldsm_x4(Lk + ao, ak[0], ak[1], ak[2], ak[3]);
                ldsm_x4(Rb + sw128f_off(16 * I + rr + 8 * (mi >> 1), 8 * ks + 4 * (mi & 1), 64), b4[0],
                        b4[1], b4[2], b4[3]);
                mma_tf32(acc[0][0], aq, b4[0], b4[1]);
                mma_tf32(acc[0][1], aq, b4[2], b4[3]);
                mma_tf32(acc[1][0], ak, b4[0], b4[1]);
                mma_tf32(acc[1][1], ak, b4[2], b4[3]);
            }
        } else if (warp < 10) {
            int tI, tJ;
            pair_of(warp - 4, tI, tJ);
            // decay of the blocks strictly between J and I (blocks 1 and/or 2)
            const bool use1 = tJ < 1 && 1 < tI, use2 = tJ < 2 && 2 < tI;
            const uint32_t lq = smem_u32(smem + kLQ), lk = smem_u32(smem + kLK);
            const uint32_t rt = smem_u32(smem + kRO);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                uint32_t aq[4], ak[4], b4[4];
                const uint32_t ao =
                    sw128_off(16 * (tI - 1) + rr + 8 * (mi & 1), 16 * ks + 8 * (mi >> 1), 48);
                ldsm_x4(lq + ao, aq[0], aq[1], aq[2], aq[3]);
                ldsm_x4(lk + ao, ak[0], ak[1], ak[2], ak[3]);
                ldsm_x4(rt + sw128_off(16 * tJ + rr + 8 * (mi >> 1), 16 * ks + 8 * (mi & 1), 64), b4[0],
                        b4[1], b4[2], b4[3]);
                if (use1 || use2) {
                    const int cc = 16 * ks + 2 * tq;
                    const __half2* m1 = reinterpret_cast<const __half2*>(MIDh);
                    const __half2* m2 = reinterpret_cast<const __half2*>(MIDh + 128);
                    __half2 mlo, mhi;
                    if (use1 && use2) {
                        mlo = __hmul2(m1[cc >> 1], m2[cc >> 1]);
                        mhi = __hmul2(m1[(cc + 8) >> 1], m2[(cc + 8) >> 1]);
                    } else {
                        const __half2* m = use1 ? m1 : m2;
                        mlo = m[cc >> 1];
                        mhi = m[(cc + 8) >> 1];
                    }
                    __half2* hq = reinterpret_cast<__half2*>(aq);
                    __half2* hk = reinterpret_cast<__half2*>(ak);
                    hq[0] = __hmul2(hq[0], mlo);
                    hq[1] = __hmul2(hq[1], mlo);
                    hq[2] = __hmul2(hq[2], mhi);
                    hq[3] = __hmul2(hq[3], mhi);
                    hk[0] = __hmul2(hk[0], mlo);
                    hk[1] = __hmul2(hk[1], mlo);
                    hk[2] = __hmul2(hk[2], mhi);
                    hk[3] = __hmul2(hk[3], mhi);
                }
                mma_f16(acc[0][0], aq, b4[0], b4[1]);
                mma_f16(acc[0][1], aq, b4[2], b4[3]);
                mma_f16(acc[1][0], ak, b4[0], b4[1]);
                mma_f16(acc[1][1], ak, b4[2], b4[3]);
            }
        } else if (warp == 15) {
            // the thread that issued the previous item's bulk stores waits for
            // them to complete and marks that item written (fused launch)
            if (lane == 0 && p.ready && prev >= 0) {
                bulk_wait_all();
                publish_ready(p.ready + prev);
            }
        } else {
            // warps 10..14, free during the tiles: b v in fp16, in place (the right
            // operand of the u product), 16-byte pieces of v (64 rows x 16)
            const bool ok_v = mbar_wait(&bar[1], n_local & 1);
            if (!ok_v && p.status) atomicOr(p.status, 1);
            constexpr int kBvThreads = kThreads - 320 - 32;
#pragma unroll
            for (int e = 0; e < (C * 16 + kBvThreads - 1) / kBvThreads; ++e) {
                const int pc = tid - 320 + kBvThreads * e;
                if (pc < C * 16) {
                    const int r = pc >> 4, c8 = (pc & 15) * 8;
                    uint4* vp = reinterpret_cast<uint4*>(smem + kV + sw128_off(r, c8, 64));
                    uint4 raw = *vp;
                    uint32_t* w4 = reinterpret_cast<uint32_t*>(&raw);
                    const float2 br = splat2(beta[r]);
#pragma unroll
                    for (int x = 0; x < 4; ++x)
                        w4[x] = pack_half2v(mul2(br, make_float2(__uint_as_float(w4[x] << 16),
                                                                __uint_as_float(w4[x] & 0xffff0000u))));
                    *vp = raw;
                }
            }
        }
        __syncthreads();  // the operand tiles are consumed (k^ P stays for the solve)

        // beta of the next item (its chunk metadata has landed by now; len_next <=
        // 64, so only the first 64 threads load)
        braw_next = (nxt < n_items && tid < len_next)
                        ? load_raw(p.beta_raw, RAW16, (size_t)(tok_next + tid) * H + nxt % H)
                        : 0.f;

        // ---- results into place; then the diagonal warps invert their 16x16
        //      block T_II = (I + A_II)^{-1} (registers, 16 lanes) and warps 0..2
        //      form T's block columns, beside the X rows --------------------------
        if (warp < 4) {
            const int I = warp;
            put(0, I, I, acc[0]);
            put(1, I, I, acc[1]);
            {
                __syncwarp();
                if (lane < 16) {
                    // column col of T by forward substitution, column by column of
                    // A: once t[j] is final, every later row takes its update from
                    // it (independent updates, so the dependent chain is 16 long)
                    const int col = lane;
                    const float* Ad = reinterpret_cast<const float*>(smem + kAkd) + I * 256;
                    float t[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) t[i] = (i == col) ? 1.f : 0.f;
#pragma unroll
                    for (int j = 0; j < 15; ++j) {
                        float acol[16];
#pragma unroll
                        for (int i4 = 0; i4 < 4; ++i4)
                            if (4 * i4 + 3 > j)
                                *reinterpret_cast<float4*>(acol + 4 * i4) =
                                    *reinterpret_cast<const float4*>(Ad + j * 16 + 4 * i4);
                        const float tj = t[j];
#pragma unroll
                        for (int i = j + 1; i < 16; ++i) t[i] = fmaf(-acol[i], tj, t[i]);
                    }
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        *reinterpret_cast<__half*>(smem + kT16 + sw64_off(16 * I + i, 16 * I + col)) =
                            __float2half_rn(t[i]);
                }
            }
            // ---- T = (I + A_kk)^{-1} in full, once every T_II and -A_Im is in
            //      place: warp J forms block column J below the diagonal,
            //      T_IJ = T_II sum_{J<=m<I} (-A_Im) T_mJ for I = J+1..3, in
            //      transposed form (T_IJ^T = (sum T_mJ^T (-A_Im)^T) T_II^T) so that
            //      each result is already the A fragment of the next product, and
            //      zeroes the blocks above the diagonal in row J (t_column)
            if (warp < 3) {
                solve_bar_wait();
                if (warp == 0) t_column<0>(smem, lane);
                if (warp == 1) t_column<1>(smem, lane);
                if (warp == 2) t_column<2>(smem, lane);
            } else {
                solve_bar_arrive();
            }
        } else if (warp < 10) {
            int tI, tJ;
            pair_of(warp - 4, tI, tJ);
            put(0, tI, tJ, acc[0]);
            put(1, tI, tJ, acc[1]);
            solve_bar_arrive();
        }
        // ---- X = b k^ e^G in fp16 for the w product, by the 12 warps that do not
        //      invert (beside the 16x16 inverses): k^ P from its fp32 tile (a lane
        //      reads one 16-byte chunk, four columns, a warp two whole rows, so a
        //      read takes the four wavefronts 512 bytes need) times b and the
        //      prefix F1 of the row's block, into the free k^ E_B / P area
        // the A_qk blocks above the diagonal are zero, so that the tile, which goes
        // out whole, is the full lower-triangular matrix and holds no stale shared
        // memory; warps 10..15 take one block each: (0,1) (0,2) (0,3) (1,2) (1,3) (2,3)
        if (warp >= 10) {
            const int b = warp - 10;
            const int I = b < 3 ? 0 : (b < 5 ? 1 : 2);
            const int J = b < 3 ? b + 1 : (b < 5 ? b - 1 : 3);
            *reinterpret_cast<uint4*>(smem + kAqkStage + sw64_off(16 * I + (lane >> 1), 16 * J + 8 * (lane & 1))) =
                make_uint4(0u, 0u, 0u, 0u);
        }
        if (warp >= 4) {
            // piece pc = row r (32 pieces of four columns each): lane = piece in
            // the row, row r = warp - 4 + 12 j; a fixed trip count, so that the
            // loads of all iterations can be in flight together
            const int qt = lane >> 3, cc = lane & 7, c = 32 * qt + 4 * cc;
#pragma unroll
            for (int j = 0; j < 6; ++j) {
                const int r = warp - 4 + 12 * j;
                if (r < C) {
                    const float4 kp = *reinterpret_cast<const float4*>(
                        smem + kLk32 + qt * 8192 + r * 128 + ((cc ^ (r & 7)) << 4));
                    const float4 f1 = *reinterpret_cast<const float4*>(F1 + (r >> 4) * 128 + c);
                    const float2 br = splat2(beta[r]);
                    *reinterpret_cast<uint2*>(smem + kX + sw128_off(r, c, 64)) = make_uint2(
                        pack_half2v(mul2(mul2(br, make_float2(f1.x, f1.y)), make_float2(kp.x, kp.y))),
                        pack_half2v(mul2(mul2(br, make_float2(f1.z, f1.w)), make_float2(kp.z, kp.w))));
                }
            }
        }
        // the A_qk staging tile is read by the bulk store, T's blocks and X by the
        // tensor cores
        fence_proxy_async();
        __syncthreads();
        if (tid == kStoreTid) {
            bulk_s2g(blk + kWsAqkOff, smem + kAqkStage, 8192);
            bulk_commit();
        }

        // ---- [w | u] = T [X | Y] on the tensor cores: A = T (K-major), B = X and
        //      Y read MN-major from their row-major tiles (K = the chunk's rows);
        //      w and u complete on mbarriers of their own, so that w is read back
        //      while the u product runs
        if (tid == 0) {
            tc_fence_after();
            const uint32_t sb = smem_u32(smem);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)  // K = 16 rows per MMA
                mma_f16_ss(tmem, sw128_desc(sb + kT16 + ks * 32, 16, 1024),
                           sw128_desc(sb + kX + ks * 2048, 8192, 1024), kIdescWU, ks > 0);
            mma_commit(&bar[2]);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                mma_f16_ss(tmem + 128, sw128_desc(sb + kT16 + ks * 32, 16, 1024),
                           sw128_desc(sb + kV + ks * 2048, 8192, 1024), kIdescWU, ks > 0);
            mma_commit(bar_u);
        }

        // ---- w, then u, out of tensor memory into their staging tiles: warp w
        //      reads lane quarter qd = w % 4, whose lanes 0..15 hold chunk rows
        //      16 qd + lane, and columns 32 cb .. 32 cb + 31 (cb = w / 4) of each.
        //      A wait that gives up is reported at the barrier that closes the
        //      read-back (the values read are then not stored).
        bool ok_wu = true;
        {
            const int qd = warp & 3, cb = warp >> 2;
            const int i = 16 * qd + (lane & 15);
            const uint32_t tcol = tmem + ((uint32_t)(32 * qd) << 16) + 32 * cb;
#pragma unroll
            for (int m = 0; m < 2; ++m) {  // 0: w, 1: u
                ok_wu = mbar_wait(m == 0 ? &bar[2] : bar_u, n_local & 1) && ok_wu;
                tc_fence_after();
                float x[2][16];
                tmem_ld16(tcol + 128 * m, x[0]);
                tmem_ld16(tcol + 128 * m + 16, x[1]);
                tmem_wait_ld();
                if (lane < 16) {
#pragma unroll
                    for (int g2 = 0; g2 < 2; ++g2) {
                        const float* xv = x[g2];
                        const uint4 lo = make_uint4(pack_half2(xv[0], xv[1]), pack_half2(xv[2], xv[3]),
                                                    pack_half2(xv[4], xv[5]), pack_half2(xv[6], xv[7]));
                        const uint4 hi = make_uint4(pack_half2(xv[8], xv[9]), pack_half2(xv[10], xv[11]),
                                                    pack_half2(xv[12], xv[13]), pack_half2(xv[14], xv[15]));
                        const int c = 32 * cb + 16 * g2;  // column of w or u
                        if (m == 0) {
                            *reinterpret_cast<uint4*>(smem + kLQ + sw128_off(i, c, 64)) = lo;
                            *reinterpret_cast<uint4*>(smem + kLQ + sw128_off(i, c + 8, 64)) = hi;
                        } else {
                            uint8_t* dst = smem + kLq32 + (c >> 4) * kWsUSliceBytes + i * 32;  // 16 value columns a slice
                            *reinterpret_cast<uint4*>(dst) = lo;
                            *reinterpret_cast<uint4*>(dst + 16) = hi;
                        }
                    }
                }
            }
        }
        tc_fence_before();
        fence_proxy_async();
        if (!ok_wu) *abort_flag = 1;
        __syncthreads();
        if (*abort_flag) {  // a product never completed: report and stop (uniform)
            if (tid == 0 && p.status) atomicOr(p.status, 1);
            break;
        }
        if (tid == kStoreTid) {
            bulk_s2g(blk + kWsWOff, smem + kLQ, 16384);
            bulk_s2g(blk + kWsUOff, smem + kLq32, 16384);
            bulk_commit();
            if (nxt < n_items) issue_v(nxt, tok_next);  // v of this item is consumed
        }
        prev = it;
        it = nxt;
    }
    if (tid == kStoreTid) {
        bulk_wait_all();  // stores complete before the CTA releases its smem
        if (p.ready && prev >= 0) publish_ready(p.ready + prev);
    }
    // every tensor-memory read has completed (tcgen05.wait::ld) before the release
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

template <bool RAW16>
__global__ void __launch_bounds__(kThreads, 1)
kda_intra_tc(const __grid_constant__ IntraMaps maps, FwdParams p) {
    // the scan launched after this grid may place its CTAs on the SMs this
    // grid's CTAs leave when their items are done (it waits for the whole grid
    // before it reads the intermediates)
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (call_aborted(p)) return;
    extern __shared__ __align__(1024) uint8_t smem[];
    StaticClaims cl;
    intra_items<RAW16>(maps, p, smem, cl);
}

// ---- fused intra + scan launch ---------------------------------------------
// One CTA per SM, all resident at once (cooperative launch).  The CTAs take
// work from one queue: positions [0, split) are intra items 0..split-1,
// [split, split + n_walks) are scan walks, the rest intra items split.. .  The
// CTAs that take a walk leave the intra work and run it; the others finish the
// intra items, which each walk waits for (ready flags) chunk by chunk.  With
// the split chosen so that the intra items stay ahead of the walks, the scan
// runs alongside the second part of the intra work instead of after it.
struct QueueClaims {
    int* queue;
    volatile int* slot;  // the claimed position, shared memory
    int split, n_walks, n_items;
    int last;  // the last claimed position
    __device__ int item(int q) const {
        return q < split ? q : (q < split + n_walks ? n_items : q - n_walks);
    }
    __device__ int first() {
        if (threadIdx.x == 0) *slot = atomicAdd(queue, 1);
        __syncthreads();
        last = *slot;
        __syncthreads();  // every thread has read it before the next claim
        return item(last);
    }
    __device__ void claim() {
        if (threadIdx.x == 0) *slot = atomicAdd(queue, 1);
    }
    __device__ int next(int) {
        last = *slot;
        return item(last);
    }
};

template <bool RAW16>
__global__ void __launch_bounds__(kThreads, 1)
kda_fused(const __grid_constant__ IntraMaps maps, FwdParams p, int split, int n_walks) {
    if (call_aborted(p)) return;  // every CTA leaves: no walk waits on an item
    extern __shared__ __align__(1024) uint8_t smem[];
    QueueClaims cl{p.queue, reinterpret_cast<volatile int*>(smem + kBar + 32), split, n_walks,
                   p.n_chunks * p.H, -1};
    intra_items<RAW16>(maps, p, smem, cl);
    const int w = cl.last - split;
    if (w < 0 || w >= n_walks || threadIdx.x >= scan::kScanThreads) return;
    // walk w: (long sequence, head) pair w / 8, value rows 16 (w % 8) ..
    const int pair = w >> 3;
    const int sq = pair / p.H, h = pair % p.H;
    const int n = p.long_list ? p.long_list[sq] : sq;
    scan::scan_walk<2>(p, smem, n, h, w & 7);
}

// ---- host side -------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    }
    return fn;
}

bool make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int elt, int box_x,
              int H, int64_t T, int box_rows = C,
              CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {128, (cuuint64_t)H, (cuuint64_t)T};
    cuuint64_t strides[2] = {(cuuint64_t)128 * elt, (cuuint64_t)H * 128 * elt};
    cuuint32_t box[3] = {(cuuint32_t)box_x, 1, (cuuint32_t)box_rows};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_maps(IntraMaps* maps, const FwdParams& p) {
    return make_map(&maps->q, p.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 64, p.H, p.T) &&
           make_map(&maps->k, p.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 64, p.H, p.T) &&
           make_map(&maps->v, p.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 64, p.H, p.T) &&
           (p.raw_bf16 ? make_map(&maps->g, p.g_raw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 64, p.H, p.T)
                       : make_map(&maps->g, p.g_raw, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, 32, p.H, p.T));
}

// SMs kept on intra-chunk items once the walks have started, at least.
constexpr int kFusedIntraSms = 32;
// How many intra items one SM finishes while a walk advances by one chunk (a
// walk step takes ~0.7 us and an item ~7.3 us on GB300), and a lead of whole
// walk steps' items done before the walks start (a CTA that claims a walk first
// finishes its item).  Fitted on the 1 x 4096 and 1 x 16384, H = 12 prefills
// (sweeps of the rate, 0.065 .. 0.16, and of the lead, 3 .. 9 steps): about 430
// of 768 and 1500 of 3072 items before the walks.
constexpr double kItemsPerWalkStep = 0.115;
constexpr int kWalkLeadSteps = 6;

// Per device: cooperative launch supported and one fused CTA fits on an SM.
int g_fused_state[32] = {0};  // per device: 0 unknown, 1 usable, 2 not

bool fused_device_ok() {
    int* state = g_fused_state;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev >= 32) return false;
    if (!state[dev]) {
        int coop = 0, per_sm = 0;
        bool ok = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) == cudaSuccess && coop;
        ok = ok && cudaFuncSetAttribute(kda_fused<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        kSmemBytes) == cudaSuccess;
        ok = ok && cudaFuncSetAttribute(kda_fused<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        kSmemBytes) == cudaSuccess;
        ok = ok && cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kda_fused<false>, kThreads,
                                                                 kSmemBytes) == cudaSuccess && per_sm >= 1;
        ok = ok && cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kda_fused<true>, kThreads,
                                                                 kSmemBytes) == cudaSuccess && per_sm >= 1;
        state[dev] = ok ? 1 : 2;
    }
    return state[dev] == 1;
}

}  // namespace

bool make_out_map(CUtensorMap* m, const FwdParams& p, int box_values, int box_rows) {
    // box_rows rows of box_values values of one head, dense in shared memory
    if (!p.out || (reinterpret_cast<uintptr_t>(p.out) & 15) != 0 || p.T <= 0) return false;
    return make_map(m, p.out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, box_values, p.H, p.T, box_rows,
                    CU_TENSOR_MAP_SWIZZLE_NONE);
}

static std::atomic<bool> g_fused_enabled{true};
void set_fused_enabled(bool on) { g_fused_enabled.store(on); }

bool fused_eligible(const FwdParams& p) {
    if (!g_fused_enabled.load()) return false;
    if (!p.ready || !p.queue || p.n_chunks <= 0 || p.lower_bound < -5.0f) return false;
    const int n_seq = p.long_list ? p.n_long : p.N;
    if (n_seq <= 0) return false;
    const int sms = num_sms();
    if (scan_groups(n_seq, p.H, sms) != 1) return false;  // walks of 16 value rows
    int seg_len = 0;
    if (scan_segments(p, sms, &seg_len) > 0) return false;  // the segmented scan does better
    const long n_walks = (long)n_seq * p.H * (kD / 16);
    return n_walks <= sms - kFusedIntraSms && fused_device_ok();
}

cudaError_t launch_fused(const FwdParams& p, cudaStream_t s) {
    IntraMaps maps;
    if (!make_maps(&maps, p)) return cudaErrorInvalidValue;
    const int sms = num_sms();
    const int n_seq = p.long_list ? p.n_long : p.N;
    const int pairs = n_seq * p.H;
    const int n_walks = pairs * (kD / 16);
    const int n_items = p.n_chunks * p.H;
    // Split: the walks start once the items done before them, plus what the
    // remaining SMs finish meanwhile, keep each walk's next chunk ready: per
    // chunk step the walks consume `pairs` items and the other SMs produce
    // (sms - n_walks) * kItemsPerWalkStep; the first chunk's items and a lead
    // of kWalkLeadSteps steps are done before.
    const double steps = (double)p.n_chunks / n_seq;  // chunks per sequence, on average
    const double deficit = pairs - (sms - n_walks) * kItemsPerWalkStep;
    double split = (double)pairs * (1 + kWalkLeadSteps) + (steps - 1.0) * (deficit > 0 ? deficit : 0.0);
    if (split > n_items) split = n_items;
    // (the work counter is cleared with the status word by the caller)
    cudaError_t e = cudaMemsetAsync(p.ready, 0, (size_t)n_items * sizeof(int), s);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)sms);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int sp = (int)split;
    e = p.raw_bf16 ? cudaLaunchKernelEx(&cfg, kda_fused<true>, maps, p, sp, n_walks)
                   : cudaLaunchKernelEx(&cfg, kda_fused<false>, maps, p, sp, n_walks);
    if (e == cudaErrorCooperativeLaunchTooLarge) {  // fewer SMs than expected are ours
        int dev = 0;
        if (cudaGetDevice(&dev) == cudaSuccess && dev < 32) g_fused_state[dev] = 2;
    }
    return e;
}

cudaError_t launch_intra(const FwdParams& p, cudaStream_t s) {
    if (p.n_chunks <= 0) return cudaSuccess;
    if (p.lower_bound < -5.0f) return launch_intra_exact(p, s);
    IntraMaps maps;
    if (!make_maps(&maps, p)) return cudaErrorInvalidValue;
    static unsigned configured = 0;
    static int sms[32] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 32 && !(configured & (1u << dev))) {
        e = cudaFuncSetAttribute(kda_intra_tc<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kSmemBytes);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(kda_intra_tc<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kSmemBytes);
        if (e != cudaSuccess) return e;
        cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev);
        configured |= 1u << dev;
    }
    const int n_items = p.n_chunks * p.H;
    const int grid = n_items < sms[dev < 32 ? dev : 0] ? n_items : sms[dev < 32 ? dev : 0];
    if (p.raw_bf16)
        kda_intra_tc<true><<<grid > 0 ? grid : 1, kThreads, kSmemBytes, s>>>(maps, p);
    else
        kda_intra_tc<false><<<grid > 0 ? grid : 1, kThreads, kSmemBytes, s>>>(maps, p);
    return cudaGetLastError();
}

}  // namespace kda
