// Token-by-token kernel for short sequences (at most kShortMax tokens; empty
// sequences too).  The work items are (sequence, head, half of the value rows):
// 64 value rows of the state, held in fp32 registers by a CTA of 4 warps.  Warp
// w owns value rows 16w .. 16w + 15 of the item's half, a half-warp one row at a
// time (rows 16w + 2j + half), lane l of the half keys 8l..8l+7.  For each token
// of the sequence, in order:
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
//
// The CTAs are persistent (as many as fit on the GPU at once, three per SM) and
// walk the items with a grid stride.  Besides the 4 compute warps each CTA has a
// producer warp: its lanes resolve the routing of 32 upcoming items at once
// (sequence, bounds, initial-state flag, slots, the first token's beta_raw),
// then lane 0 fills a ring of shared-memory stages, a few items ahead, by bulk
// copies: the item's 64 state rows (one contiguous block of the pool) and the
// first token's q, k and g_raw rows and half v row, plus a small header.  The
// compute warps read everything from the stage, so the state reads stay in
// flight while they reduce and store, and no global-load latency sits on their
// path (later tokens of a multi-token sequence are read directly).

#include "kda_device.cuh"
#include "kda_internal.h"

namespace kda {
namespace {

using namespace dev;

constexpr int D = kD;

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

// One stage of the ring: the item's 64 state rows (32 KB fp32, 16 KB otherwise),
// the first token's q, k and g_raw rows and the item's half of its v row, and a
// header the producer writes (the first token's beta_raw and the item's routing).
constexpr int kItemRows = 64;
constexpr int kConsumers = 128;                 // 4 compute warps, one thread per key
constexpr int kDecThreadsAll = kConsumers + 32;  // + the producer warp
static_assert(kConsumers == D, "the per-token prep maps compute threads to keys");
constexpr int kClaim = 8;    // items per claim from the shared counter (1 near the end)
constexpr int kEnd = -2;     // StageHeader::len of the end marker
struct StageHeader {
    int tok0, len, has_init, h, vb, pad;
    long long out_slot;
    float beta_raw;
};
constexpr int kTokQ = 0, kTokK = 256, kTokV = 512, kTokG = 640;  // bytes in the token area
constexpr int kTokBytes = kTokG + 512;                          // g_raw fp32 at most
constexpr int kHdrOff = kTokBytes;
constexpr int kStageExtra = 1280;  // token area + header, rounded
static_assert(kHdrOff + (int)sizeof(StageHeader) <= kStageExtra, "stage extra");

__host__ __device__ constexpr int dec_stages(int dtype) { return dtype == 0 ? 2 : 4; }
__host__ __device__ constexpr int dec_tile_bytes(int dtype) {
    return kItemRows * D * (dtype == 0 ? 4 : 2);
}
__host__ __device__ constexpr int dec_stage_bytes(int dtype) {
    return dec_tile_bytes(dtype) + kStageExtra;
}
__host__ __device__ constexpr int dec_smem(int dtype) {
    return dec_stages(dtype) * dec_stage_bytes(dtype) + 128;
}
constexpr int kDecSmemMax = dec_smem(1) > dec_smem(0) ? dec_smem(1) : dec_smem(0);

// The kernel's work; it may return early (an aborted call, a wait that gave up).
__device__ __forceinline__ void decode_items(const FwdParams& p, long long n_items) {
    if (call_aborted(p)) return;
    extern __shared__ __align__(128) uint8_t ring[];  // stages, then mbarriers
    __shared__ __align__(16) float s_q[D], s_k[D], s_a[D];  // q^, k^, a of the token
    __shared__ float s_red[2][4], s_beta;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int H = p.H;
    const int stages = dec_stages(p.st_dtype);
    const int tile = dec_tile_bytes(p.st_dtype);
    const int sbytes = dec_stage_bytes(p.st_dtype);
    const int elt = p.st_dtype == 0 ? 4 : 2;
    const int gbytes = p.raw_bf16 ? 256 : 512;
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + stages * sbytes);  // [stages]
    uint64_t* empty = full + stages;                                         // [stages]

    if (tid == 0) {
        for (int i = 0; i < stages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kConsumers / 32);
        }
        fence_mbar_init();
    }
    __syncthreads();

    // ======================= producer warp ==================================
    // The CTA's items: with p.dec_queue, batches of kClaim consecutive items taken
    // from the shared counter (CTAs that start late, e.g. beside the scan, take
    // what is left); without it, items blockIdx.x + i * gridDim.x.  After the
    // last item the next stage gets an end marker (len = kEnd, no copy).
    if (warp == kConsumers / 32) {
        const bool dyn = p.dec_queue != nullptr;
        int r = 0;  // stage sequence number
        int claim = kClaim;
        for (long long base = 0;;) {
            long long first = 0, stride = 1;
            int cnt = claim;
            if (dyn) {
                int b0 = 0;
                if (lane == 0) b0 = atomicAdd(p.dec_queue, claim);
                first = __shfl_sync(0xffffffffu, b0, 0);
                // near the end single items, so that the CTAs finish together
                if (n_items - (first + claim) < (long long)gridDim.x * kClaim) claim = 1;
            } else {
                first = blockIdx.x + base * gridDim.x;
                stride = gridDim.x;
                cnt = 32;
                base += 32;
            }
            // lane i resolves the routing of item first + i * stride
            const long long my_it = first + (long long)lane * stride;
            int n = 0, h = 0, vb = 0, tok0 = 0, len = 0, init = 0;
            long long in_slot = 0, out_slot = 0;
            float braw = 0.f;
            if (lane < cnt && my_it < n_items) {
                const long long sh = my_it >> 1;
                vb = kItemRows * (int)(my_it & 1);
                h = (int)(sh % H);
                n = p.short_list[sh / H];
                tok0 = p.cu[n];
                len = p.cu[n + 1] - tok0;
                init = p.has_init ? (p.has_init[n] != 0) : (p.st_in != nullptr);
                in_slot = p.st_in_idx ? p.st_in_idx[n] : n;
                out_slot = p.st_out_idx ? p.st_out_idx[n] : n;
                if (p.num_slots > 0) {  // a slot outside the pool: no access, reported
                    const bool bad_in = init && (in_slot < 0 || in_slot >= p.num_slots);
                    const bool bad_out = out_slot < 0 || out_slot >= p.num_slots;
                    if ((bad_in || bad_out) && p.status) atomicOr(p.status, 4);
                    if (bad_in) init = 0;
                    if (bad_out) out_slot = -1;  // no store
                }
                if (len > 0) braw = load_raw(p.beta_raw, p.raw_bf16, (size_t)tok0 * H + h);
            }
            bool stop = false;
            for (int j = 0; j < cnt; ++j, ++r) {
                const bool end = first + (long long)j * stride >= n_items;
                const int jh = __shfl_sync(0xffffffffu, h, j);
                const int jvb = __shfl_sync(0xffffffffu, vb, j);
                const int jtok0 = __shfl_sync(0xffffffffu, tok0, j);
                const int jlen = __shfl_sync(0xffffffffu, len, j);
                const int jinit = __shfl_sync(0xffffffffu, init, j);
                const long long jin = __shfl_sync(0xffffffffu, in_slot, j);
                const long long jout = __shfl_sync(0xffffffffu, out_slot, j);
                const float jb = __shfl_sync(0xffffffffu, braw, j);
                if (lane == 0) {
                    const int st = r % stages;
                    if (r >= stages && !mbar_wait(&empty[st], (uint32_t)(((r / stages) - 1) & 1))) {
                        if (p.status) atomicOr(p.status, 1);
                        stop = true;
                    } else if (end) {
                        uint8_t* stg = ring + st * sbytes;
                        reinterpret_cast<StageHeader*>(stg + tile + kHdrOff)->len = kEnd;
                        mbar_arrive(&full[st]);  // the end marker: nothing to copy
                        stop = true;
                    } else {
                        uint8_t* stg = ring + st * sbytes;
                        StageHeader* hd = reinterpret_cast<StageHeader*>(stg + tile + kHdrOff);
                        hd->tok0 = jtok0;
                        hd->len = jlen;
                        hd->has_init = jinit;
                        hd->h = jh;
                        hd->vb = jvb;
                        hd->out_slot = jout;
                        hd->beta_raw = jb;
                        const uint32_t bytes =
                            (jinit ? (uint32_t)tile : 0u) + (jlen > 0 ? 640u + (uint32_t)gbytes : 0u);
                        if (bytes == 0) {
                            mbar_arrive(&full[st]);  // nothing to copy: the phase completes now
                        } else {
                            mbar_arrive_expect_tx(&full[st], bytes);
                            if (jinit) {
                                const size_t off = (size_t)jin * p.st_in_stride +
                                                   (size_t)jh * D * D + (size_t)jvb * D;
                                bulk_g2s(stg, static_cast<const uint8_t*>(p.st_in) + off * elt,
                                         (uint32_t)tile, &full[st]);
                            }
                            if (jlen > 0) {
                                const size_t row = ((size_t)jtok0 * H + jh) * D;
                                uint8_t* tk = stg + tile;
                                bulk_g2s(tk + kTokQ, p.q + row, 256, &full[st]);
                                bulk_g2s(tk + kTokK, p.k + row, 256, &full[st]);
                                bulk_g2s(tk + kTokV, p.v + row + jvb, 128, &full[st]);
                                bulk_g2s(tk + kTokG,
                                         static_cast<const uint8_t*>(p.g_raw) + row * (gbytes / D),
                                         (uint32_t)gbytes, &full[st]);
                            }
                        }
                    }
                }
                if (__shfl_sync(0xffffffffu, (int)stop, 0)) {
                    stop = true;
                    break;
                }
            }
            if (stop) break;
        }
        return;
    }

    // ======================= compute warps ==================================
    const int hw = lane >> 4, l16 = lane & 15;
    const int k0 = 8 * l16;  // this lane's keys
    const float lb = p.lower_bound;
    auto csync = [&]() { asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory"); };
    auto csync_or = [&](bool flag) -> bool {
        uint32_t any;
        asm volatile(
            "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
            "bar.red.or.pred q, 1, %2, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
            : "=r"(any)
            : "r"((uint32_t)flag), "n"(kConsumers)
            : "memory");
        return any != 0;
    };

    for (int r = 0;; ++r) {
        const int st = r % stages;
        const bool ok = mbar_wait(&full[st], (uint32_t)((r / stages) & 1));
        if (csync_or(!ok)) {  // a copy never landed: report, leave together
            if (tid == 0) {
                if (p.status) atomicOr(p.status, 1);
                for (int rq = r; rq < r + stages; ++rq)  // copies possibly in flight, bounded
                    mbar_wait(&full[rq % stages], (uint32_t)((rq / stages) & 1));
            }
            return;
        }
        const uint8_t* stg = ring + st * sbytes;
        const StageHeader* hd = reinterpret_cast<const StageHeader*>(stg + tile + kHdrOff);
        if (hd->len == kEnd) break;  // the producer's end marker
        const int tok0 = hd->tok0, len = hd->len, h = hd->h, vb = hd->vb;
        const bool has_init = hd->has_init != 0;
        const bool store_ok = hd->out_slot >= 0;
        const size_t out_base =
            store_ok ? (size_t)hd->out_slot * p.st_out_stride + (size_t)h * D * D : 0;
        float braw = hd->beta_raw;

        float S[8][8];  // rows vb + 16 warp + 2j + hw, keys k0..k0+7
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (has_init) {
                load8(stg, p.st_dtype, (size_t)(16 * warp + 2 * j + hw) * D + k0, S[j]);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) S[j][e] = 0.f;
            }
        }
        // the first token's inputs from the stage; later tokens' from memory
        float qv = 0.f, kv = 0.f, gv = 0.f, vv[8];
        if (len > 0) {
            const uint8_t* tk = stg + tile;
            qv = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(tk + kTokQ)[tid]);
            kv = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(tk + kTokK)[tid]);
            gv = load_raw(tk + kTokG, p.raw_bf16, tid);
#pragma unroll
            for (int j = 0; j < 8; ++j)
                vv[j] = __bfloat162float(
                    reinterpret_cast<const __nv_bfloat16*>(tk + kTokV)[16 * warp + 2 * j + hw]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);  // this warp is done with the stage

        for (int t = 0; t < len; ++t) {
            const size_t row = ((size_t)(tok0 + t) * H + h) * D;
            if (t > 0) {
                qv = __bfloat162float(p.q[row + tid]);
                kv = __bfloat162float(p.k[row + tid]);
                gv = load_raw(p.g_raw, p.raw_bf16, row + tid);
                if (tid == 0) braw = load_raw(p.beta_raw, p.raw_bf16, (size_t)(tok0 + t) * H + h);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    vv[j] = __bfloat162float(p.v[row + vb + 16 * warp + 2 * j + hw]);
            }
            // the token's q^, k^ and a, one key per thread
            if (tid == 0) s_beta = __fdividef(1.f, 1.f + __expf(-braw));
            {
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
            csync();
            {
                const float sq = s_red[0][0] + s_red[0][1] + s_red[0][2] + s_red[0][3];
                const float sk = s_red[1][0] + s_red[1][1] + s_red[1][2] + s_red[1][3];
                s_q[tid] = qv * rsqrtf(sq + 1e-6f) * 0.08838834764831845f;  // 1/sqrt(128)
                s_k[tid] = kv * rsqrtf(sk + 1e-6f);
            }
            csync();

            float a8[8], k8[8], q8[8];
            *reinterpret_cast<float4*>(a8) = *reinterpret_cast<const float4*>(s_a + k0);
            *reinterpret_cast<float4*>(a8 + 4) = *reinterpret_cast<const float4*>(s_a + k0 + 4);
            *reinterpret_cast<float4*>(k8) = *reinterpret_cast<const float4*>(s_k + k0);
            *reinterpret_cast<float4*>(k8 + 4) = *reinterpret_cast<const float4*>(s_k + k0 + 4);
            *reinterpret_cast<float4*>(q8) = *reinterpret_cast<const float4*>(s_q + k0);
            *reinterpret_cast<float4*>(q8 + 4) = *reinterpret_cast<const float4*>(s_q + k0 + 4);
            const float b = s_beta;

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
            csync();  // the next token rewrites the shared vectors
        }

        if (store_ok) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int vr = vb + 16 * warp + 2 * j + hw;
                store8(p.st_out, p.st_dtype, out_base + (size_t)vr * D + k0, S[j]);
            }
        }
    }
}

__global__ void __launch_bounds__(kDecThreadsAll, 3) kda_decode(FwdParams p, long long n_items) {
    decode_items(p, n_items);
    // Launched beside the scan (programmatic stream serialization), this grid
    // completes only after the scan has, however its CTAs left: later work on
    // the stream sees both.  Without such a predecessor the wait returns at once.
    if (threadIdx.x == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace

cudaError_t launch_decode(const FwdParams& p, cudaStream_t s, bool beside_scan) {
    if (p.n_short <= 0 || !p.short_list) return cudaSuccess;
    // per device: the ring's shared memory allowance, and how many CTAs fit on
    // the GPU at once for each ring size (fp32 pool, 2-byte pool)
    static int fit[32][2] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const int cls = p.st_dtype == 0 ? 0 : 1;
    const size_t smem = (size_t)dec_smem(p.st_dtype);
    int ctas = dev < 32 ? fit[dev][cls] : 0;
    if (!ctas) {
        e = cudaFuncSetAttribute(kda_decode, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kDecSmemMax);
        if (e != cudaSuccess) return e;
        int per_sm = 0, sms = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kda_decode, kDecThreadsAll,
                                                          smem);
        if (e != cudaSuccess) return e;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        ctas = (per_sm > 0 ? per_sm : 1) * (sms > 0 ? sms : 1);
        if (dev < 32) fit[dev][cls] = ctas;
    }
    const long long n_items = 2LL * p.n_short * p.H;
    const unsigned grid = (unsigned)(n_items < ctas ? n_items : ctas);
    if (!beside_scan || !p.dec_queue) {
        kda_decode<<<grid, kDecThreadsAll, smem, s>>>(p, n_items);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kDecThreadsAll);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kda_decode, p, n_items);
}

}  // namespace kda
