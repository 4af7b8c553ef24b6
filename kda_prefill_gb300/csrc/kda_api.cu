// Host side of the C ABI declared in include/kda.h: argument validation, the
// per-bounds metadata cache with its single pinned non-blocking upload, and
// the kernel launches.
//
// Metadata (ROCm/aiter PR #6912, "Changes"): chunk indices are built from
// host bounds and numbered by the sequence's position in cu_seqlens; all
// tables share one int32 buffer whose blocks start 16-byte aligned, uploaded
// with one non-blocking copy from pinned memory and cached on the bounds'
// contents.  A hit from another stream waits on the uploading stream; a miss
// while the stream is being captured fails; entries a capture used are kept for
// the life of the process so eviction cannot free them under a graph.

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <list>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "kda.h"
#include "kda_internal.h"

namespace {

thread_local std::string g_err;

int fail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_err = buf;
    return code;
}

int cuda_fail(cudaError_t e, const char* what) {
    return fail(KDA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

constexpr int kChunk = kda::kC;
constexpr int kD = kda::kD;

inline int64_t chunks_of(int64_t len) { return (len + kChunk - 1) / kChunk; }
// Chunks a sequence gets in the chunked kernels: none when it is short enough
// for the token-by-token kernel.
inline bool is_short(int64_t len) { return len <= kda::kShortMax; }
inline int64_t routed_chunks(int64_t len) { return is_short(len) ? 0 : chunks_of(len); }

int64_t max_chunks(int64_t T, int32_t N) { return (T + kChunk - 1) / kChunk + N; }

size_t state_elt(int dtype) { return dtype == KDA_STATE_F32 ? 4 : 2; }

struct Range {
    const char* name;
    uintptr_t lo, hi;  // [lo, hi)
};

bool overlaps(const Range& a, const Range& b) {
    if (a.lo == a.hi || b.lo == b.hi) return false;
    return a.lo < b.hi && b.lo < a.hi;
}

Range rng(const char* name, const void* p, size_t bytes) {
    uintptr_t lo = reinterpret_cast<uintptr_t>(p);
    return Range{name, lo, p ? lo + bytes : lo};
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_host_bounds(const int32_t* cu, int32_t N, int64_t T) {
    if (cu[0] != 0) return fail(KDA_ERR_INVALID_ARG, "cu_seqlens_host[0] = %d, expected 0", cu[0]);
    for (int32_t n = 0; n < N; ++n)
        if (cu[n + 1] < cu[n])
            return fail(KDA_ERR_INVALID_ARG, "cu_seqlens_host decreases at %d (%d -> %d)", n,
                        cu[n], cu[n + 1]);
    if ((int64_t)cu[N] != T)
        return fail(KDA_ERR_INVALID_ARG, "cu_seqlens_host[%d] = %d, expected total_tokens = %lld",
                    N, cu[N], (long long)T);
    return KDA_OK;
}

// ---------------------------------------------------------------------------
// Metadata: layout of the single int32 buffer.
// ---------------------------------------------------------------------------
struct MetaLayout {
    int64_t n_chunks = 0;
    int32_t n_long = 0, n_short = 0;
    int32_t max_long_chunks = 0;  // chunks of the longest sequence the chunked kernels take
    size_t off_cu = 0, off_seq_off = 0, off_chunk_seq = 0, off_chunk_tok = 0;  // int32 units
    size_t off_long = 0, off_short = 0;
    size_t words = 0;
};

inline size_t align4(size_t w) { return (w + 3) & ~size_t(3); }  // 16-byte blocks

// Chunk count and routing of the sequences from host bounds.
MetaLayout meta_layout(const int32_t* cu, int32_t N) {
    MetaLayout L;
    for (int32_t n = 0; n < N; ++n) {
        const int64_t len = (int64_t)cu[n + 1] - cu[n];
        L.n_chunks += routed_chunks(len);
        if (is_short(len)) ++L.n_short; else ++L.n_long;
        L.max_long_chunks = std::max<int32_t>(L.max_long_chunks, (int32_t)routed_chunks(len));
    }
    size_t o = 0;
    L.off_cu = o;        o = align4(o + (size_t)N + 1);
    L.off_seq_off = o;   o = align4(o + (size_t)N + 1);
    L.off_chunk_seq = o; o = align4(o + (size_t)L.n_chunks);
    L.off_chunk_tok = o; o = align4(o + (size_t)L.n_chunks);
    L.off_long = o;      o = align4(o + (size_t)N);
    L.off_short = o;     o = align4(o + (size_t)N);
    L.words = std::max<size_t>(o, 4);
    return L;
}

void meta_fill(const int32_t* cu, int32_t N, const MetaLayout& L, int32_t* buf) {
    std::memset(buf, 0, L.words * sizeof(int32_t));
    int32_t* mcu = buf + L.off_cu;
    int32_t* off = buf + L.off_seq_off;
    int32_t* cseq = buf + L.off_chunk_seq;
    int32_t* ctok = buf + L.off_chunk_tok;
    int32_t* lng = buf + L.off_long;
    int32_t* sht = buf + L.off_short;
    int64_t j = 0;
    int32_t nl = 0, ns = 0;
    for (int32_t n = 0; n < N; ++n) {
        mcu[n] = cu[n];
        off[n] = (int32_t)j;
        const int64_t len = (int64_t)cu[n + 1] - cu[n];
        if (is_short(len)) sht[ns++] = n; else lng[nl++] = n;
        const int64_t nc = routed_chunks(len);
        for (int64_t c = 0; c < nc; ++c, ++j) {
            cseq[j] = n;
            ctok[j] = (int32_t)(cu[n] + c * kChunk);
        }
    }
    mcu[N] = cu[N];
    off[N] = (int32_t)j;
    // longest first: the scan launches its walks in this order, so that the long
    // walks start in the first wave and the short ones fill the last
    std::stable_sort(lng, lng + nl, [&](int32_t a, int32_t b) {
        return cu[a + 1] - cu[a] > cu[b + 1] - cu[b];
    });
}

// ---------------------------------------------------------------------------
// Pinned staging for the metadata uploads and the bounds read-back: a set of
// pinned host blocks, each used as a ring.  A region is handed out again only
// once the copy that last used it has completed, which is checked with
// cudaEventQuery: acquiring never waits for the GPU.  When the region the next
// copy needs is still in flight in every block (the GPU is behind by more than
// a block's worth of uploads), another block is allocated and kept for later
// calls; requests larger than a block get a block of their own size class,
// reused in the same way.  Only past kMaxBlocks blocks does a request wait, for
// the oldest copy of its block, so that a runaway producer cannot pin unbounded
// host memory.
// ---------------------------------------------------------------------------
class PinnedPool {
  public:
    static constexpr size_t kBlock = size_t(8) << 20;
    static constexpr int kMaxBlocks = 32;

    // Returns a staging area of `bytes` (256-aligned) or nullptr on failure.
    // The caller records `*done` on its stream after enqueueing the copy.
    void* acquire(size_t bytes, cudaEvent_t** done) {
        bytes = (bytes + 255) & ~size_t(255);
        const size_t cap = block_size(bytes);
        for (auto& b : blocks_) {
            if (b.cap != cap) continue;
            void* p = try_block(b, bytes, done);
            if (p) return p;
        }
        if ((int)blocks_.size() < kMaxBlocks) {
            Block b;
            if (cudaHostAlloc(&b.base, cap, cudaHostAllocDefault) != cudaSuccess) return nullptr;
            b.cap = cap;
            blocks_.push_back(std::move(b));
            return try_block(blocks_.back(), bytes, done);
        }
        // every block of this size is busy and no more may be added: wait for
        // the region of the first one (the only blocking case)
        for (auto& b : blocks_) {
            if (b.cap != cap) continue;
            void* p = take(b, bytes, done, /*wait=*/true);
            if (p) return p;
        }
        return nullptr;
    }

  private:
    struct Pending {
        size_t lo, hi;
        cudaEvent_t ev;
    };
    struct Block {
        void* base = nullptr;
        size_t cap = 0, head = 0;
        std::list<Pending> pending;
    };

    static size_t block_size(size_t bytes) {
        size_t cap = kBlock;
        while (cap < bytes) cap <<= 1;
        return cap;
    }

    static void* try_block(Block& b, size_t bytes, cudaEvent_t** done) {
        return take(b, bytes, done, /*wait=*/false);
    }

    // The region at the block's head (wrapping to the start when the tail is
    // too short), if every earlier copy into it has completed (or, with
    // `wait`, after waiting for them).
    static void* take(Block& b, size_t bytes, cudaEvent_t** done, bool wait) {
        const size_t lo = (b.head + bytes > b.cap) ? 0 : b.head, hi = lo + bytes;
        for (auto it = b.pending.begin(); it != b.pending.end();) {
            if (it->lo < hi && lo < it->hi) {
                cudaError_t q = wait ? cudaEventSynchronize(it->ev) : cudaEventQuery(it->ev);
                if (q == cudaErrorNotReady) return nullptr;
                cudaEventDestroy(it->ev);
                it = b.pending.erase(it);
            } else {
                ++it;
            }
        }
        b.pending.push_back(Pending{lo, hi, nullptr});
        if (cudaEventCreateWithFlags(&b.pending.back().ev, cudaEventDisableTiming) != cudaSuccess) {
            b.pending.pop_back();
            return nullptr;
        }
        *done = &b.pending.back().ev;
        b.head = hi;
        return static_cast<char*>(b.base) + lo;
    }

    std::vector<Block> blocks_;
};

struct MetaEntry {
    std::vector<int32_t> key;  // device, N, bounds
    int device = 0;
    MetaLayout layout;
    int32_t* dev = nullptr;
    cudaEvent_t ready = nullptr;
    cudaStream_t upload_stream = nullptr;
    bool captured = false;
    std::vector<std::pair<cudaStream_t, cudaEvent_t>> uses;  // last use per stream
    uint64_t stamp = 0;
};

class MetaCache {
  public:
    static constexpr size_t kMaxEntries = 256;

    std::mutex mu;
    std::map<std::vector<int32_t>, MetaEntry*> map;
    PinnedPool ring;
    uint64_t clock = 0;

    // Finds or builds the entry for these bounds; enqueues the upload on a miss
    // and the cross-stream wait on a hit.
    int get(const int32_t* cu, int32_t N, cudaStream_t stream, bool capturing, MetaEntry** out) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
        std::vector<int32_t> key;
        key.reserve((size_t)N + 3);
        key.push_back(dev);
        key.push_back(kChunk);
        key.push_back(N);
        key.insert(key.end(), cu, cu + N + 1);
        auto it = map.find(key);
        if (it != map.end()) {
            MetaEntry* m = it->second;
            m->stamp = ++clock;
            if (m->upload_stream != stream) {
                // A global-mode capture (on this thread or another) forbids
                // cudaEventQuery on this thread; the upload event is never part
                // of a capture, so the thread queries it in relaxed mode.
                cudaStreamCaptureMode mode = cudaStreamCaptureModeRelaxed;
                cudaThreadExchangeStreamCaptureMode(&mode);
                cudaError_t q = cudaEventQuery(m->ready);
                cudaThreadExchangeStreamCaptureMode(&mode);
                if (q == cudaErrorNotReady) {
                    if (capturing)
                        return fail(KDA_ERR_CAPTURE_MISS,
                                    "metadata upload still in flight on another stream while "
                                    "this stream is capturing; synchronize before capturing");
                    e = cudaStreamWaitEvent(stream, m->ready, 0);
                    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamWaitEvent");
                } else if (q != cudaSuccess) {
                    return cuda_fail(q, "cudaEventQuery");
                }
            }
            if (capturing) m->captured = true;
            *out = m;
            return KDA_OK;
        }
        if (capturing)
            return fail(KDA_ERR_CAPTURE_MISS,
                        "metadata for these bounds is not cached and the stream is capturing; "
                        "run the call once before capture");
        int rc = evict_if_full(stream);
        if (rc != KDA_OK) return rc;

        auto* m = new MetaEntry();
        m->key = std::move(key);
        m->device = dev;
        m->layout = meta_layout(cu, N);
        const size_t bytes = m->layout.words * sizeof(int32_t);
        cudaEvent_t* done = nullptr;
        void* host = ring.acquire(bytes, &done);
        if (!host) {
            delete m;
            return fail(KDA_ERR_CUDA, "pinned staging allocation failed");
        }
        meta_fill(cu, N, m->layout, static_cast<int32_t*>(host));
        e = cudaMallocAsync(reinterpret_cast<void**>(&m->dev), bytes, stream);
        if (e != cudaSuccess) {
            cudaEventRecord(*done, stream);  // the staging region is free again
            delete m;
            return cuda_fail(e, "cudaMallocAsync (metadata)");
        }
        e = cudaMemcpyAsync(m->dev, host, bytes, cudaMemcpyHostToDevice, stream);
        cudaEventRecord(*done, stream);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&m->ready, cudaEventDisableTiming);
        if (e != cudaSuccess) {  // nothing refers to the entry yet: release it
            cudaFreeAsync(m->dev, stream);
            delete m;
            return cuda_fail(e, "metadata upload");
        }
        cudaEventRecord(m->ready, stream);
        m->upload_stream = stream;
        m->stamp = ++clock;
        map[m->key] = m;
        *out = m;
        return KDA_OK;
    }

    // Records that `stream` used the entry (for safe eviction later).
    void mark_use(MetaEntry* m, cudaStream_t stream, bool capturing) {
        if (capturing) return;
        for (auto& u : m->uses) {
            if (u.first == stream) {
                cudaEventRecord(u.second, stream);
                return;
            }
        }
        cudaEvent_t ev;
        if (cudaEventCreateWithFlags(&ev, cudaEventDisableTiming) != cudaSuccess) return;
        cudaEventRecord(ev, stream);
        m->uses.emplace_back(stream, ev);
    }

    int evict_if_full(cudaStream_t stream) {
        while (map.size() >= kMaxEntries) {
            auto victim = map.end();
            for (auto it = map.begin(); it != map.end(); ++it) {
                if (it->second->captured) continue;
                if (victim == map.end() || it->second->stamp < victim->second->stamp) victim = it;
            }
            if (victim == map.end()) return KDA_OK;  // everything captured: keep growing
            MetaEntry* m = victim->second;
            int dev = 0;
            cudaGetDevice(&dev);
            if (m->device == dev) {
                // free stream-ordered after every recorded use
                for (auto& u : m->uses) cudaStreamWaitEvent(stream, u.second, 0);
                cudaStreamWaitEvent(stream, m->ready, 0);
                cudaFreeAsync(m->dev, stream);
            } else {
                leaked_.push_back(m->dev);  // other device: released by kda_release_cache
            }
            destroy_events(m);
            map.erase(victim);
            delete m;
        }
        return KDA_OK;
    }

    static void destroy_events(MetaEntry* m) {
        for (auto& u : m->uses) cudaEventDestroy(u.second);
        m->uses.clear();
        if (m->ready) cudaEventDestroy(m->ready);
        m->ready = nullptr;
    }

    int release() {
        int rc = KDA_OK;
        int cur = 0;
        cudaGetDevice(&cur);
        for (auto it = map.begin(); it != map.end();) {
            MetaEntry* m = it->second;
            if (m->captured) {
                ++it;
                continue;
            }
            cudaSetDevice(m->device);
            if (cudaDeviceSynchronize() != cudaSuccess) rc = KDA_ERR_CUDA;
            cudaFree(m->dev);
            destroy_events(m);
            delete m;
            it = map.erase(it);
        }
        for (void* p : leaked_) cudaFree(p);
        leaked_.clear();
        cudaSetDevice(cur);
        return rc;
    }

  private:
    std::vector<void*> leaked_;
};

MetaCache& cache() {
    static MetaCache* c = new MetaCache();  // never destroyed: outlives static teardown
    return *c;
}

// Per-kernel timing records (guarded by the cache mutex).
struct Timing {
    bool enabled = false;
    std::vector<std::vector<cudaEvent_t>> calls;  // kNumKernels + 1 marks per call
    std::vector<unsigned> launched;               // per call: kernels that had work
    std::vector<cudaEvent_t> free_events;

    cudaEvent_t take() {
        if (!free_events.empty()) {
            cudaEvent_t e = free_events.back();
            free_events.pop_back();
            return e;
        }
        cudaEvent_t e = nullptr;
        cudaEventCreate(&e);
        return e;
    }
};

Timing& timing() {
    static Timing* t = new Timing();
    return *t;
}

struct StateArgs {
    const void* in;
    void* out;
    int64_t in_stride, out_stride;
    const int32_t* in_idx;
    const int32_t* out_idx;
    const uint8_t* has_init;
    int32_t num_slots;  // paged calls: slots are checked against it on the device; 0 = dense
};

int run_forward(const void* q, const void* k, const void* v, const void* g_raw,
                const void* beta_raw, int raw_bf16, const int32_t* cu_dev,
                const int32_t* cu_host, int32_t N, int64_t T, int32_t H, const StateArgs& st,
                int state_dtype, void* out, float lower_bound, void* workspace,
                size_t workspace_bytes, cudaStream_t stream) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(stream, &cap);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
    const bool capturing = (cap != cudaStreamCaptureStatusNone);

    std::lock_guard<std::mutex> lock(cache().mu);
    std::vector<int32_t> readback;
    if (!cu_host) {
        if (capturing)
            return fail(KDA_ERR_CAPTURE_MISS,
                        "device bounds cannot be read back while the stream is capturing; "
                        "pass cu_seqlens_host");
        readback.resize((size_t)N + 1);
        cudaEvent_t* done = nullptr;
        void* host = cache().ring.acquire(readback.size() * sizeof(int32_t), &done);
        if (!host) return fail(KDA_ERR_CUDA, "pinned staging allocation failed");
        e = cudaMemcpyAsync(host, cu_dev, readback.size() * sizeof(int32_t),
                            cudaMemcpyDeviceToHost, stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
        if (e == cudaSuccess) std::memcpy(readback.data(), host, readback.size() * sizeof(int32_t));
        cudaEventRecord(*done, stream);
        if (e != cudaSuccess) return cuda_fail(e, "read-back of cu_seqlens");
        cu_host = readback.data();
        int rc = check_host_bounds(cu_host, N, T);
        if (rc != KDA_OK) return rc;
    }

    MetaEntry* m = nullptr;
    int rc = cache().get(cu_host, N, stream, capturing, &m);
    if (rc != KDA_OK) return rc;

    uint8_t* ws = static_cast<uint8_t*>(workspace);

    kda::FwdParams p{};
    p.q = static_cast<const __nv_bfloat16*>(q);
    p.k = static_cast<const __nv_bfloat16*>(k);
    p.v = static_cast<const __nv_bfloat16*>(v);
    p.g_raw = g_raw;
    p.beta_raw = beta_raw;
    p.raw_bf16 = raw_bf16;
    p.out = static_cast<__nv_bfloat16*>(out);
    p.H = H;
    p.N = N;
    p.n_chunks = (int)m->layout.n_chunks;
    p.T = T;
    p.lower_bound = lower_bound;
    p.cu = m->dev + m->layout.off_cu;
    p.seq_off = m->dev + m->layout.off_seq_off;
    p.chunk_seq = m->dev + m->layout.off_chunk_seq;
    p.chunk_tok = m->dev + m->layout.off_chunk_tok;
    p.long_list = m->dev + m->layout.off_long;
    p.short_list = m->dev + m->layout.off_short;
    p.n_long = m->layout.n_long;
    p.n_short = m->layout.n_short;
    p.ws = ws ? ws + kda::kWsHeader : nullptr;
    p.status = ws ? reinterpret_cast<int*>(ws) : nullptr;
    p.queue = ws ? reinterpret_cast<int*>(ws + kda::kWsQueueOff) : nullptr;
    p.dec_queue = ws ? reinterpret_cast<int*>(ws + kda::kWsDecodeOff) : nullptr;
    p.ready = ws ? reinterpret_cast<int*>(ws + kda::flags_offset(max_chunks(T, N), H)) : nullptr;
    p.seg = ws ? reinterpret_cast<float*>(ws + kda::seg_offset(max_chunks(T, N), H)) : nullptr;
    p.max_long_chunks = m->layout.max_long_chunks;
    p.st_in = st.in;
    p.st_out = st.out;
    p.st_in_stride = st.in_stride;
    p.st_out_stride = st.out_stride;
    p.st_in_idx = st.in_idx;
    p.st_out_idx = st.out_idx;
    p.has_init = st.has_init;
    p.num_slots = st.num_slots;
    p.st_dtype = state_dtype;
    (void)workspace_bytes;

    if (p.status) {
        // the status word and the two work counters, one memset
        e = cudaMemsetAsync(p.status, 0, kda::kWsClearBytes, stream);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync (status)");
    }
    cudaEvent_t* marks = nullptr;
    std::vector<cudaEvent_t> ev;
    if (timing().enabled && !capturing) {
        for (int i = 0; i <= kda::kNumKernels; ++i) ev.push_back(timing().take());
        marks = ev.data();
    }
    e = kda::launch_forward(p, stream, marks);
    if (marks) {
        timing().calls.push_back(ev);
        timing().launched.push_back(kda::launched_kernels(p));
    }
    if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
    cache().mark_use(m, stream, capturing);
    return KDA_OK;
}

// Checks of the activations, bounds, dtype and lower bound (everything but the
// state and the workspace).
int input_checks(const void* q, const void* k, const void* v, const void* g_raw,
                 const void* beta_raw, int raw_bf16, const int32_t* cu_dev,
                 const int32_t* cu_host, int32_t N, int64_t T, int32_t H, void* out,
                 float lower_bound, int state_dtype) {
    if (N < 0) return fail(KDA_ERR_INVALID_ARG, "num_seqs = %d < 0", N);
    if (T < 0) return fail(KDA_ERR_INVALID_ARG, "total_tokens = %lld < 0", (long long)T);
    if (T > INT32_MAX - kChunk)
        return fail(KDA_ERR_INVALID_ARG, "total_tokens = %lld exceeds the int32 token index",
                    (long long)T);
    if (H <= 0 || H > 65535) return fail(KDA_ERR_INVALID_ARG, "num_heads = %d out of range", H);
    if (N == 0 && T != 0) return fail(KDA_ERR_INVALID_ARG, "tokens without sequences");
    if (state_dtype < KDA_STATE_F32 || state_dtype > KDA_STATE_F16)
        return fail(KDA_ERR_UNSUPPORTED, "state_dtype %d not supported (0 fp32, 1 bf16, 2 fp16)",
                    state_dtype);
    if (!(lower_bound <= 0.0f && lower_bound >= -64.0f))
        return fail(KDA_ERR_UNSUPPORTED, "lower_bound %g outside [-64, 0]", (double)lower_bound);
    if (!cu_dev && !cu_host)
        return fail(KDA_ERR_INVALID_ARG, "cu_seqlens and cu_seqlens_host are both NULL");
    if (T > 0) {
        if (!q || !k || !v || !g_raw || !beta_raw || !out)
            return fail(KDA_ERR_INVALID_ARG, "a q/k/v/g_raw/beta_raw/out pointer is NULL");
        const void* p16[] = {q, k, v, g_raw, out};
        const char* n16[] = {"q", "k", "v", "g_raw", "out"};
        for (int i = 0; i < 5; ++i)
            if (!aligned(p16[i], 16))
                return fail(KDA_ERR_UNSUPPORTED, "%s is not 16-byte aligned", n16[i]);
        const size_t relt = raw_bf16 ? 2 : 4;  // bytes per raw gate / beta element
        if (!aligned(beta_raw, relt))
            return fail(KDA_ERR_UNSUPPORTED, "beta_raw is not %zu-byte aligned", relt);
        const size_t act = (size_t)T * H * kD * 2;
        Range ro = rng("out", out, act);
        Range ins[] = {rng("q", q, act), rng("k", k, act), rng("v", v, act),
                       rng("g_raw", g_raw, act / 2 * relt),
                       rng("beta_raw", beta_raw, (size_t)T * H * relt)};
        for (auto& r : ins)
            if (overlaps(ro, r)) return fail(KDA_ERR_INVALID_ARG, "out overlaps %s", r.name);
    }
    if (cu_host) {
        int rc = check_host_bounds(cu_host, N, T);
        if (rc != KDA_OK) return rc;
    }
    return KDA_OK;
}

int common_checks(const void* q, const void* k, const void* v, const void* g_raw,
                  const void* beta_raw, int raw_bf16, const int32_t* cu_dev,
                  const int32_t* cu_host, int32_t N, int64_t T, int32_t H, void* out,
                  float lower_bound, int state_dtype, void* workspace,
                  size_t workspace_bytes) {
    int rc = input_checks(q, k, v, g_raw, beta_raw, raw_bf16, cu_dev, cu_host, N, T, H, out,
                          lower_bound, state_dtype);
    if (rc != KDA_OK) return rc;
    const size_t need = kda_workspace_size(T, N, H);
    if (need > 0 && (!workspace || workspace_bytes < need))
        return fail(KDA_ERR_WORKSPACE, "workspace of %zu bytes given, %zu needed",
                    workspace ? workspace_bytes : (size_t)0, need);
    if (workspace && !aligned(workspace, 256))
        return fail(KDA_ERR_UNSUPPORTED, "workspace is not 256-byte aligned");
    return KDA_OK;
}

// The allocation-free entry point's built-in scratch (defined further down).
int noalloc_scratch(void** out);

}  // namespace

extern "C" {

int kda_chunk_size(void) { return kChunk; }

size_t kda_workspace_size(int64_t total_tokens, int32_t num_seqs, int32_t num_heads) {
    if (total_tokens < 0 || num_seqs < 0 || num_heads <= 0) return 0;
    if (num_seqs == 0) return 0;
    return kda::workspace_bytes(max_chunks(total_tokens, num_seqs), num_heads);
}

const char* kda_last_error(void) { return g_err.c_str(); }

int kda_plan_chunks(const int32_t* cu, int32_t N, int32_t chunk_size, int32_t* chunk_seq,
                    int32_t* chunk_in_seq, int32_t* seq_chunk_offset, int64_t capacity,
                    int64_t* n_chunks) {
    if (!cu || N < 0 || chunk_size <= 0 || !n_chunks)
        return fail(KDA_ERR_INVALID_ARG, "invalid arguments to kda_plan_chunks");
    if (cu[0] != 0) return fail(KDA_ERR_INVALID_ARG, "cu_seqlens_host[0] != 0");
    int64_t total = 0;
    for (int32_t n = 0; n < N; ++n) {
        if (cu[n + 1] < cu[n]) return fail(KDA_ERR_INVALID_ARG, "cu_seqlens_host decreases at %d", n);
        total += ((int64_t)cu[n + 1] - cu[n] + chunk_size - 1) / chunk_size;
    }
    *n_chunks = total;
    if (total > capacity) return fail(KDA_ERR_WORKSPACE, "capacity %lld < %lld chunks",
                                      (long long)capacity, (long long)total);
    int64_t j = 0;
    for (int32_t n = 0; n < N; ++n) {
        if (seq_chunk_offset) seq_chunk_offset[n] = (int32_t)j;
        const int64_t nc = ((int64_t)cu[n + 1] - cu[n] + chunk_size - 1) / chunk_size;
        for (int64_t c = 0; c < nc; ++c, ++j) {
            if (chunk_seq) chunk_seq[j] = n;
            if (chunk_in_seq) chunk_in_seq[j] = (int32_t)c;
        }
    }
    if (seq_chunk_offset) seq_chunk_offset[N] = (int32_t)j;
    return KDA_OK;
}

}  // extern "C"

namespace {
// Checks of the paged state pool: the pool, indices and flags are given, the
// slots can hold the sequences, the slot stride covers a plane and keeps 16-byte
// alignment, and the pool overlaps no activation.
int pool_checks(const void* q, const void* k, const void* v, const void* g_raw,
                const void* beta_raw, int raw_bf16, int32_t num_seqs, int64_t total_tokens,
                int32_t num_heads, const void* state_cache, int64_t state_stride0,
                int32_t num_slots, const int32_t* state_indices,
                const uint8_t* has_initial_state, const void* out, int state_dtype) {
    if (num_seqs <= 0) return KDA_OK;
    const int64_t plane = (int64_t)num_heads * kD * kD;
    if (!state_cache || !state_indices || !has_initial_state)
        return fail(KDA_ERR_INVALID_ARG,
                    "state_cache, state_indices and has_initial_state are required");
    if (num_slots <= 0) return fail(KDA_ERR_INVALID_ARG, "num_slots = %d", num_slots);
    if (num_slots < num_seqs)
        return fail(KDA_ERR_INVALID_ARG, "num_slots %d < num_seqs %d (slots are distinct)",
                    num_slots, num_seqs);
    if (state_stride0 < plane)
        return fail(KDA_ERR_INVALID_ARG,
                    "state_stride0 %lld is smaller than the slot plane H*V*K = %lld",
                    (long long)state_stride0, (long long)plane);
    const size_t elt = state_elt(state_dtype);
    if (!aligned(state_cache, 16) || ((size_t)state_stride0 * elt) % 16 != 0)
        return fail(KDA_ERR_UNSUPPORTED, "state_cache and its slot stride must be 16-byte aligned");
    const size_t pool_bytes = ((size_t)(num_slots - 1) * state_stride0 + plane) * elt;
    Range rp = rng("state_cache", state_cache, pool_bytes);
    const size_t act = (size_t)total_tokens * num_heads * kD * 2;
    const size_t relt = raw_bf16 ? 2 : 4;
    Range others[] = {rng("q", q, act), rng("k", k, act), rng("v", v, act),
                      rng("g_raw", g_raw, act / 2 * relt),
                      rng("beta_raw", beta_raw, (size_t)total_tokens * num_heads * relt),
                      rng("out", out, act)};
    for (auto& r : others)
        if (overlaps(rp, r)) return fail(KDA_ERR_INVALID_ARG, "state_cache overlaps %s", r.name);
    return KDA_OK;
}

// The paged forward for either raw gate / beta type (raw_bf16: bf16, else fp32).
int paged_forward(const void* q, const void* k, const void* v, const void* g_raw,
                  const void* beta_raw, int raw_bf16, const int32_t* cu_seqlens,
                  const int32_t* cu_seqlens_host, int32_t num_seqs, int64_t total_tokens,
                  int32_t num_heads, void* state_cache, int64_t state_stride0,
                  int32_t num_slots, const int32_t* state_indices,
                  const uint8_t* has_initial_state, void* out, float lower_bound,
                  int state_dtype, void* workspace, size_t workspace_bytes,
                  kda_stream_t stream) {
    int rc = common_checks(q, k, v, g_raw, beta_raw, raw_bf16, cu_seqlens, cu_seqlens_host,
                           num_seqs, total_tokens, num_heads, out, lower_bound, state_dtype,
                           workspace, workspace_bytes);
    if (rc == KDA_OK)
        rc = pool_checks(q, k, v, g_raw, beta_raw, raw_bf16, num_seqs, total_tokens, num_heads,
                         state_cache, state_stride0, num_slots, state_indices,
                         has_initial_state, out, state_dtype);
    if (rc != KDA_OK) return rc;
    StateArgs st{state_cache, state_cache, state_stride0, state_stride0,
                 state_indices, state_indices, has_initial_state, num_slots};
    return run_forward(q, k, v, g_raw, beta_raw, raw_bf16, cu_seqlens, cu_seqlens_host,
                       num_seqs, total_tokens, num_heads, st, state_dtype, out, lower_bound,
                       workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}
}  // namespace

extern "C" {

int kda_chunk_fwd(const void* q, const void* k, const void* v, const float* g_raw,
                  const float* beta_raw, const int32_t* cu_seqlens,
                  const int32_t* cu_seqlens_host, int32_t num_seqs, int64_t total_tokens,
                  int32_t num_heads, void* state_cache, int64_t state_stride0,
                  int32_t num_slots, const int32_t* state_indices,
                  const uint8_t* has_initial_state, void* out, float lower_bound,
                  int state_dtype, void* workspace, size_t workspace_bytes,
                  kda_stream_t stream) {
    return paged_forward(q, k, v, g_raw, beta_raw, 0, cu_seqlens, cu_seqlens_host, num_seqs,
                         total_tokens, num_heads, state_cache, state_stride0, num_slots,
                         state_indices, has_initial_state, out, lower_bound, state_dtype,
                         workspace, workspace_bytes, stream);
}

int kda_chunk_fwd_raw_bf16(const void* q, const void* k, const void* v, const void* g_raw,
                           const void* beta_raw, const int32_t* cu_seqlens,
                           const int32_t* cu_seqlens_host, int32_t num_seqs,
                           int64_t total_tokens, int32_t num_heads, void* state_cache,
                           int64_t state_stride0, int32_t num_slots,
                           const int32_t* state_indices, const uint8_t* has_initial_state,
                           void* out, float lower_bound, int state_dtype, void* workspace,
                           size_t workspace_bytes, kda_stream_t stream) {
    return paged_forward(q, k, v, g_raw, beta_raw, 1, cu_seqlens, cu_seqlens_host, num_seqs,
                         total_tokens, num_heads, state_cache, state_stride0, num_slots,
                         state_indices, has_initial_state, out, lower_bound, state_dtype,
                         workspace, workspace_bytes, stream);
}

int kda_chunk_fwd_dense(const void* q, const void* k, const void* v, const float* g_raw,
                        const float* beta_raw, const int32_t* cu_seqlens,
                        const int32_t* cu_seqlens_host, int32_t num_seqs,
                        int64_t total_tokens, int32_t num_heads, const void* initial_state,
                        const uint8_t* has_initial_state, void* final_state, int state_dtype,
                        void* out, float lower_bound, void* workspace,
                        size_t workspace_bytes, kda_stream_t stream) {
    int rc = common_checks(q, k, v, g_raw, beta_raw, 0, cu_seqlens, cu_seqlens_host, num_seqs,
                           total_tokens, num_heads, out, lower_bound, state_dtype, workspace,
                           workspace_bytes);
    if (rc != KDA_OK) return rc;
    const int64_t plane = (int64_t)num_heads * kD * kD;
    if (num_seqs > 0) {
        if (!final_state) return fail(KDA_ERR_INVALID_ARG, "final_state is NULL");
        if (has_initial_state && !initial_state)
            return fail(KDA_ERR_INVALID_ARG, "has_initial_state given without initial_state");
        if (!aligned(final_state, 16) || (initial_state && !aligned(initial_state, 16)))
            return fail(KDA_ERR_UNSUPPORTED, "state buffers must be 16-byte aligned");
        const size_t bytes = (size_t)num_seqs * plane * state_elt(state_dtype);
        Range rf = rng("final_state", final_state, bytes);
        const size_t act = (size_t)total_tokens * num_heads * kD * 2;
        Range others[] = {rng("q", q, act), rng("k", k, act), rng("v", v, act),
                          rng("g_raw", g_raw, act * 2),
                          rng("beta_raw", beta_raw, (size_t)total_tokens * num_heads * 4),
                          rng("out", out, act)};
        for (auto& r : others)
            if (overlaps(rf, r)) return fail(KDA_ERR_INVALID_ARG, "final_state overlaps %s", r.name);
        if (initial_state && initial_state != final_state &&
            overlaps(rf, rng("initial_state", initial_state, bytes)))
            return fail(KDA_ERR_INVALID_ARG, "final_state partially overlaps initial_state");
    }
    StateArgs st{initial_state, final_state, plane, plane, nullptr, nullptr, has_initial_state, 0};
    return run_forward(q, k, v, g_raw, beta_raw, 0, cu_seqlens, cu_seqlens_host, num_seqs,
                       total_tokens, num_heads, st, state_dtype, out, lower_bound, workspace,
                       workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

int kda_release_cache(void) {
    std::lock_guard<std::mutex> lock(cache().mu);
    int rc = cache().release();
    return rc == KDA_OK ? KDA_OK : fail(rc, "cudaDeviceSynchronize failed during release");
}

int kda_cache_entries(void) {
    std::lock_guard<std::mutex> lock(cache().mu);
    return (int)cache().map.size();
}

int kda_set_kernel_timing(int enable) {
    std::lock_guard<std::mutex> lock(cache().mu);
    timing().enabled = enable != 0;
    return KDA_OK;
}

int kda_check_status(const void* workspace, kda_stream_t stream, int* status) {
    if (!status) return fail(KDA_ERR_INVALID_ARG, "status is NULL");
    const void* word = workspace;
    if (!word) {  // the allocation-free entry point's built-in scratch
        void* scratch = nullptr;
        const int rc = noalloc_scratch(&scratch);
        if (rc != KDA_OK) return rc;
        word = scratch;
    }
    int v = 0;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(&v, word, sizeof(int), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "kda_check_status");
    *status = v;
    return KDA_OK;
}

int kda_debug_wait_timeout(int kind, void* workspace, kda_stream_t stream) {
    if (kind != 0 && kind != 1) return fail(KDA_ERR_INVALID_ARG, "kind %d is not 0 or 1", kind);
    if (!workspace) return fail(KDA_ERR_INVALID_ARG, "workspace is NULL");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // the header (status word at 0, a zero flag at byte 128) is cleared first
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    cudaError_t e = cudaMemsetAsync(ws, 0, kda::kWsHeader, s);
    if (e == cudaSuccess)
        e = kda::launch_wait_probe(kind, reinterpret_cast<int*>(ws), reinterpret_cast<const int*>(ws + 128), s);
    if (e != cudaSuccess) return cuda_fail(e, "kda_debug_wait_timeout");
    return KDA_OK;
}

int kda_set_fused_launch(int enable) {
    kda::set_fused_enabled(enable != 0);
    return KDA_OK;
}

int kda_kernel_times(float* ms, int capacity, int* count, int* calls) {
    std::lock_guard<std::mutex> lock(cache().mu);
    if (!ms || !count || !calls || capacity < kda::kNumKernels)
        return fail(KDA_ERR_INVALID_ARG, "kda_kernel_times needs room for %d kernels",
                    kda::kNumKernels);
    for (int i = 0; i < kda::kNumKernels; ++i) ms[i] = 0.f;
    Timing& t = timing();
    int rc = KDA_OK;
    for (size_t j = 0; j < t.calls.size(); ++j) {
        const auto& c = t.calls[j];
        const unsigned ran = t.launched[j];
        cudaError_t e = cudaSuccess;
        for (cudaEvent_t ev : c)  // the marks may sit on several streams
            if (e == cudaSuccess) e = cudaEventSynchronize(ev);
        if (e != cudaSuccess) rc = cuda_fail(e, "cudaEventSynchronize");
        for (int i = 0; i < kda::kNumKernels && rc == KDA_OK; ++i) {
            if (!(ran & (1u << i))) continue;  // not launched: no time
            float x = 0.f;
            e = cudaEventElapsedTime(&x, c[i], c[i + 1]);
            if (e != cudaSuccess) rc = cuda_fail(e, "cudaEventElapsedTime");
            ms[i] += x;
        }
        for (cudaEvent_t ev : c) t.free_events.push_back(ev);
    }
    *calls = (int)t.calls.size();
    *count = kda::kNumKernels;
    t.calls.clear();
    t.launched.clear();
    return rc;
}

const char* kda_kernel_name(int i) { return kda::kernel_name(i); }

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free entry point: the workspace and the chunk table live in a
// fixed array compiled into the library instead of caller- or cache-owned
// device memory.
// ---------------------------------------------------------------------------
namespace {

// Every device that loads the library holds this array until process exit.
static __device__ __align__(256) uint8_t g_noalloc_scratch[KDA_NOALLOC_SCRATCH_BYTES];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64] = {nullptr};

// Device address of the scratch array on the current device.  The array's
// name is only a host-side stand-in in host code, so the address is looked up
// once per device (with that device current) and cached.
int noalloc_scratch(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(KDA_ERR_UNSUPPORTED, "device ordinal %d", dev);
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress (scratch)");
        g_noalloc_ptr[dev] = ptr;
    }
    *out = g_noalloc_ptr[dev];
    return KDA_OK;
}

// Checksum of a bounds array, the same on the host and on the device: the sum
// of cu[n] (2n + 1) modulo 2^32.  Two arrays that pass the device checks below
// but differ anywhere give different sums except in contrived cases.
inline uint32_t bounds_sum(const int32_t* cu, int32_t N) {
    uint32_t s = 0;
    for (int32_t n = 0; n <= N; ++n) s += (uint32_t)cu[n] * (uint32_t)(2 * n + 1);
    return s;
}

// What the host derived from cu_seqlens_host, for the device to compare with.
struct HostPlan {
    int64_t T;
    int64_t cap_chunks;  // chunk-table capacity (entries)
    int64_t n_chunks;
    int32_t n_long, max_long;
    uint32_t sum;
};

// Chunk table and sequence routing from the device bounds, one CTA: per
// sequence its chunk count and whether it is long (short sequences, at most
// kShortMax tokens, get no chunk and go to the token-by-token kernel), two
// inclusive prefix sums in tiles of 1024 sequences, then each sequence's
// chunks and its place in the long or the short list.  Same numbering as the
// host planner (chunks follow the sequence's position in cu_seqlens).
//
// The device bounds are not trusted: they are first clamped into [0, T] and
// made non-decreasing (a running maximum), so every token index the kernels
// derive from them lies in [0, T), and every table write is bounded by the
// table's capacity.  The totals (chunks, long sequences, longest sequence),
// the first and last bound and the checksum are then compared with the host's;
// on any difference the status word gets kStatusBounds and every kernel of
// the call leaves on entry without reading the table.
__global__ void __launch_bounds__(1024) kda_noalloc_meta(const int32_t* cu, int N, int C,
                                                         HostPlan hp, int32_t* mcu,
                                                         int32_t* off, int32_t* cseq,
                                                         int32_t* ctok, int32_t* lng,
                                                         int32_t* sht, int* status) {
    __shared__ int32_t sbuf[1024];
    __shared__ int32_t lbuf[1024];
    __shared__ int32_t mbuf[1024];
    __shared__ int32_t carry, lcarry, bmax, lmax;
    __shared__ uint32_t csum;
    __shared__ volatile int bad;
    const int tid = threadIdx.x;
    const int T = (int)hp.T;
    if (tid == 0) {
        carry = 0;
        lcarry = 0;
        bmax = 0;  // running maximum of the clamped bounds before this tile
        lmax = 0;
        csum = 0;
        bad = (N >= 0 && cu[0] != 0) ? 1 : 0;
    }
    __syncthreads();
    for (int base = 0; base < N; base += 1024) {
        const int n = base + tid;
        // clamped bounds: b0 = bound n, b1 = bound n + 1, both in [0, T], then
        // the running maximum over the array makes them non-decreasing
        const int r1 = (n < N) ? cu[n + 1] : 0;
        if (n < N && (r1 < 0 || r1 > T)) bad = 1;
        mbuf[tid] = (n < N) ? min(max(r1, 0), T) : 0;
        if (n < N) atomicAdd(&csum, (uint32_t)r1 * (uint32_t)(2 * (n + 1) + 1));
        __syncthreads();
        for (int o = 1; o < 1024; o <<= 1) {  // inclusive running maximum
            const int x = (tid >= o) ? mbuf[tid - o] : 0;
            __syncthreads();
            mbuf[tid] = max(mbuf[tid], x);
            __syncthreads();
        }
        const int b1 = max(mbuf[tid], bmax);
        const int b0 = tid > 0 ? max(mbuf[tid - 1], bmax) : bmax;
        const int len = (n < N) ? b1 - b0 : 0;
        if (n < N && r1 < cu[n]) bad = 1;  // decreasing
        const int is_long = (n < N && len > kda::kShortMax) ? 1 : 0;
        const int nc = is_long ? (len + C - 1) / C : 0;
        sbuf[tid] = nc;
        lbuf[tid] = is_long;
        __syncthreads();
        for (int o = 1; o < 1024; o <<= 1) {
            const int x = (tid >= o) ? sbuf[tid - o] : 0;
            const int y = (tid >= o) ? lbuf[tid - o] : 0;
            __syncthreads();
            sbuf[tid] += x;
            lbuf[tid] += y;
            __syncthreads();
        }
        const int excl = carry + sbuf[tid] - nc;
        const int lpos = lcarry + lbuf[tid] - is_long;  // long sequences before n
        if (n < N) {
            mcu[n] = b0;
            off[n] = excl;
            for (int c = 0; c < nc && (int64_t)excl + c < hp.cap_chunks; ++c) {
                cseq[excl + c] = n;
                ctok[excl + c] = b0 + c * C;
            }
            if (is_long)
                lng[lpos] = n;
            else
                sht[n - lpos] = n;
            if (nc > 0) atomicMax(&lmax, nc);
        }
        __syncthreads();
        if (tid == 1023) {
            carry += sbuf[1023];
            lcarry += lbuf[1023];
            bmax = max(bmax, mbuf[1023]);
        }
        __syncthreads();
    }
    if (tid == 0) {
        mcu[N] = bmax;
        off[N] = carry;
        const uint32_t sum = csum + (N >= 0 ? (uint32_t)cu[0] : 0u);
        if (bad || bmax != T || carry != hp.n_chunks || lcarry != hp.n_long ||
            lmax != hp.max_long || sum != hp.sum)
            atomicOr(status, kda::kStatusBounds);
    }
}

}  // namespace

extern "C" int kda_chunk_fwd_noalloc(const void* q, const void* k, const void* v,
                                     const float* g_raw, const float* beta_raw,
                                     const int32_t* cu_seqlens, const int32_t* cu_seqlens_host,
                                     int32_t num_seqs, int64_t total_tokens, int32_t num_heads,
                                     void* state_cache, int64_t state_stride0, int32_t num_slots,
                                     const int32_t* state_indices,
                                     const uint8_t* has_initial_state, void* out,
                                     float lower_bound, int state_dtype, kda_stream_t stream_) {
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (!cu_seqlens || !cu_seqlens_host)
        return fail(KDA_ERR_INVALID_ARG,
                    "kda_chunk_fwd_noalloc needs both cu_seqlens and cu_seqlens_host");
    int rc = input_checks(q, k, v, g_raw, beta_raw, 0, cu_seqlens, cu_seqlens_host, num_seqs,
                          total_tokens, num_heads, out, lower_bound, state_dtype);
    if (rc == KDA_OK)
        rc = pool_checks(q, k, v, g_raw, beta_raw, 0, num_seqs, total_tokens, num_heads,
                         state_cache, state_stride0, num_slots, state_indices,
                         has_initial_state, out, state_dtype);
    if (rc != KDA_OK) return rc;
    // The host bounds give the exact chunk count, so the scratch is laid out for
    // it (not for kda_workspace_size's bound of total_tokens / C + num_seqs,
    // which counts a partial chunk for every sequence, short ones included).
    int64_t n_chunks = 0;
    int32_t n_long = 0, max_long = 0;
    for (int32_t n = 0; n < num_seqs; ++n) {
        const int64_t len = (int64_t)cu_seqlens_host[n + 1] - cu_seqlens_host[n];
        n_chunks += routed_chunks(len);
        n_long += is_short(len) ? 0 : 1;
        max_long = std::max<int32_t>(max_long, (int32_t)routed_chunks(len));
    }
    // scratch layout: [workspace][cu | seq_off | chunk_seq | chunk_tok | long | short]
    const int64_t bound = std::max<int64_t>(n_chunks, 1);  // chunk-table capacity
    const size_t ws_need = num_seqs > 0 ? kda::workspace_bytes(bound, num_heads) : 0;
    const size_t ws_part = (ws_need + 255) & ~size_t(255);
    const size_t meta_words = 2 * align4((size_t)num_seqs + 1) + 2 * align4((size_t)bound) +
                              2 * align4((size_t)num_seqs);
    const size_t need = ws_part + meta_words * sizeof(int32_t);
    if (need > (size_t)KDA_NOALLOC_SCRATCH_BYTES)
        return fail(KDA_ERR_WORKSPACE,
                    "kda_chunk_fwd_noalloc: these sizes need %zu bytes of scratch, the built-in "
                    "scratch holds %llu (KDA_NOALLOC_SCRATCH_BYTES)",
                    need, (unsigned long long)KDA_NOALLOC_SCRATCH_BYTES);
    void* scratch = nullptr;  // 256-byte aligned, and large enough by the check above
    rc = noalloc_scratch(&scratch);
    if (rc != KDA_OK) return rc;

    uint8_t* base = static_cast<uint8_t*>(scratch);
    int32_t* meta = reinterpret_cast<int32_t*>(base + ws_part);
    int32_t* mcu = meta;
    int32_t* off = mcu + align4((size_t)num_seqs + 1);
    int32_t* cseq = off + align4((size_t)num_seqs + 1);
    int32_t* ctok = cseq + align4((size_t)bound);
    int32_t* lng = ctok + align4((size_t)bound);
    int32_t* sht = lng + align4((size_t)num_seqs);

    // the status word and the fused launch's work counter
    cudaError_t e = cudaMemsetAsync(base, 0, kda::kWsClearBytes, stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync (status)");
    if (num_seqs > 0) {
        HostPlan hp{total_tokens, bound, n_chunks, n_long, max_long,
                    bounds_sum(cu_seqlens_host, num_seqs)};
        kda_noalloc_meta<<<1, 1024, 0, stream>>>(cu_seqlens, num_seqs, kChunk, hp, mcu, off,
                                                  cseq, ctok, lng, sht,
                                                  reinterpret_cast<int*>(base));
        e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e, "chunk table kernel launch");
    }
    kda::FwdParams p{};
    p.q = static_cast<const __nv_bfloat16*>(q);
    p.k = static_cast<const __nv_bfloat16*>(k);
    p.v = static_cast<const __nv_bfloat16*>(v);
    p.g_raw = g_raw;
    p.beta_raw = beta_raw;
    p.out = static_cast<__nv_bfloat16*>(out);
    p.H = num_heads;
    p.N = num_seqs;
    p.n_chunks = (int)n_chunks;
    p.T = total_tokens;
    p.lower_bound = lower_bound;
    p.cu = mcu;
    p.seq_off = off;
    p.chunk_seq = cseq;
    p.chunk_tok = ctok;
    p.long_list = lng;
    p.short_list = sht;
    p.n_long = n_long;
    p.n_short = num_seqs - n_long;
    p.ws = base + kda::kWsHeader;
    p.status = reinterpret_cast<int*>(base);
    p.queue = reinterpret_cast<int*>(base + kda::kWsQueueOff);
    p.dec_queue = reinterpret_cast<int*>(base + kda::kWsDecodeOff);
    p.ready = reinterpret_cast<int*>(base + kda::flags_offset(bound, num_heads));
    p.seg = reinterpret_cast<float*>(base + kda::seg_offset(bound, num_heads));
    p.max_long_chunks = max_long;
    p.st_in = state_cache;
    p.st_out = state_cache;
    p.st_in_stride = state_stride0;
    p.st_out_stride = state_stride0;
    p.st_in_idx = state_indices;
    p.st_out_idx = state_indices;
    p.has_init = has_initial_state;
    p.st_dtype = state_dtype;
    p.num_slots = num_slots;
    p.abort_word = p.status;  // the kernels skip a call whose device bounds disagree
    e = kda::launch_forward(p, stream, nullptr);
    if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
    return KDA_OK;
}
