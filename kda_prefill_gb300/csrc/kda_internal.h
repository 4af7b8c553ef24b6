// Internal interface between the host side of the C ABI (kda_api.cu) and the
// CUDA kernels.  Not installed; not part of the ABI.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace kda {

constexpr int kD = 128;  // K = V = head dimension
constexpr int kC = 64;   // tokens per chunk
// Sequences of at most kShortMax tokens (empty ones included) bypass the
// chunked kernels and run token by token in kda_decode.
constexpr int kShortMax = 8;

// Workspace: one block of kWsBytes per (chunk, head), chunk-major
// (block index = chunk * H + head).  Inside a block:
//   w    [64][128] fp16  T (b k^ e^G)            swizzled 16-bit tile (two halves)
//   qg   [64][128] fp16  q^ e^G                   swizzled
//   kg   [64][128] fp16  k^ e^{G_C - G}           swizzled
//   aqk  [64][64]  fp16  decay-weighted q^ k^T    swizzled, lower incl. diagonal
//   gamma [128]    fp32  e^{G_C}
//   u    [8][64][16] fp16  T (b v), one 2 KB slice per 16 value columns
// The first kWsSharedBytes (everything but u) are read by every value slice.
constexpr int kWsWOff = 0;
constexpr int kWsQGOff = 16384;
constexpr int kWsKGOff = 32768;
constexpr int kWsAqkOff = 49152;
constexpr int kWsGammaOff = 57344;
constexpr int kWsSharedBytes = 57856;
constexpr int kWsUOff = 57856;
constexpr int kWsUSliceBytes = 2048;
constexpr int kWsBytes = 74240;
// Workspace header: one int status word (bit 0: a bounded wait gave up), at
// byte kWsQueueOff the work counter of the fused launch and at kWsDecodeOff the
// token-by-token kernel's item counter (all three cleared by one memset per
// call); the chunk blocks start at kWsHeader.  After the blocks (bounded by
// max_chunks * H) come the fused launch's ready flags, one int per (chunk, head)
// block.
constexpr int kWsHeader = 256;
constexpr int kWsQueueOff = 64;
constexpr int kWsDecodeOff = 68;
constexpr int kWsClearBytes = kWsDecodeOff + 4;

// Everything one forward launch sequence needs.  Device pointers unless noted.
struct FwdParams {
    const __nv_bfloat16* q;
    const __nv_bfloat16* k;
    const __nv_bfloat16* v;
    const void* g_raw;      // [T][H][128], fp32, or bf16 when raw_bf16
    const void* beta_raw;   // [T][H], fp32, or bf16 when raw_bf16
    int raw_bf16;
    __nv_bfloat16* out;
    int H;
    int N;
    int n_chunks;
    int64_t T;
    float lower_bound;

    // metadata (one int32 buffer uploaded by the host, see kda_api.cu)
    const int32_t* cu;         // [N+1] sequence bounds
    const int32_t* seq_off;    // [N+1] first chunk of each sequence
    const int32_t* chunk_seq;  // [n_chunks] sequence of each chunk
    const int32_t* chunk_tok;  // [n_chunks] first token of each chunk
    // sequence routing: long_list (n_long) names the sequences the chunked
    // kernels process, short_list (n_short) those kda_decode processes.  With
    // long_list == nullptr every sequence goes through the chunked kernels.
    const int32_t* long_list;
    const int32_t* short_list;
    int n_long;
    int n_short;

    uint8_t* ws;   // chunk blocks (kWsBytes each)
    int* status;   // workspace header
    int* queue;    // fused launch: work counter (workspace header)
    int* dec_queue;  // token-by-token kernel: item counter (workspace header), or nullptr
    int* ready;    // fused launch: per (chunk, head) block, nonzero once it is written

    // state (paged: st_in == st_out == pool, idx = state_indices;
    //        dense: separate bases, idx == nullptr means identity)
    const void* st_in;
    void* st_out;
    int64_t st_in_stride;   // elements between slots
    int64_t st_out_stride;
    const int32_t* st_in_idx;
    const int32_t* st_out_idx;
    const uint8_t* has_init;  // nullptr: every sequence has one iff st_in != nullptr
    int st_dtype;             // 0 fp32, 1 bf16, 2 fp16
    // pool slots of a paged call: a slot outside [0, num_slots) is neither read
    // nor written, and the status word gets bit 2 (value 4); 0 = not checked
    int num_slots;

    // segmented scan (few long sequences): chunks of the longest long sequence,
    // and the workspace area of the segments' fp32 state planes (nullptr: none)
    int max_long_chunks;
    float* seg;

    // When set (the allocation-free entry point, whose chunk table is built on
    // the device from device bounds), every kernel reads this status word on
    // entry and does nothing if it carries kStatusBounds: the device bounds
    // disagreed with the host bounds that sized the launch.
    const int* abort_word;
};

// Status bit of a call whose device bounds disagree with its host bounds
// (KDA_STATUS_BOUNDS_MISMATCH in kda.h).
constexpr int kStatusBounds = 8;

// True when the call's chunk table must not be used (see FwdParams::abort_word).
// Every thread of a kernel calls it on entry and leaves when it is true, so a
// kernel either runs in full or not at all.
__device__ __forceinline__ bool call_aborted(const FwdParams& p) {
    if (!p.abort_word) return false;
    return (*reinterpret_cast<const volatile int*>(p.abort_word) & kStatusBounds) != 0;
}

// Element i of a raw gate / beta array (fp32, or bf16 when raw_bf16 is set).
__device__ __forceinline__ float load_raw(const void* p, int raw_bf16, size_t i) {
    return raw_bf16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i])
                    : static_cast<const float*>(p)[i];
}

inline size_t flags_offset(int64_t max_chunks, int H) {
    return (size_t)kWsHeader + (size_t)max_chunks * (size_t)H * (size_t)kWsBytes;
}
// The segmented scan's fp32 [128][128] state planes (at most kSegPlanes: three
// per segment boundary, with (pairs) x (segments - 1) <= 152 / 16) follow the flags.
constexpr int kSegPlaneFloats = 128 * 128;
constexpr int kSegPlanes = 32;
inline size_t seg_offset(int64_t max_chunks, int H) {
    return flags_offset(max_chunks, H) + (((size_t)max_chunks * (size_t)H * 4 + 255) & ~size_t(255));
}
inline size_t workspace_bytes(int64_t max_chunks, int H) {
    return seg_offset(max_chunks, H) + (size_t)kSegPlanes * kSegPlaneFloats * 4;
}

// Number of kernels one forward launches, and their names (launch order).
// Kernel 3 is the fused intra + scan launch, which replaces kernels 0 and 1
// when the scan's CTAs leave enough SMs free for the intra-chunk work.
constexpr int kNumKernels = 4;
const char* kernel_name(int i);

// Enqueues the kernels of one forward on `s`.  When `marks` is non-null it
// holds kNumKernels + 1 events: marks[0] is recorded before the first kernel
// and marks[i + 1] after kernel i.
cudaError_t launch_forward(const FwdParams& p, cudaStream_t s, cudaEvent_t* marks);
// Bit i set when kernel i (launch order) has work for these parameters; a
// kernel without work is not launched and its timing interval is empty.  Read
// after launch_forward: a fused launch the device refused then reads as the
// two kernels that ran instead.
unsigned launched_kernels(const FwdParams& p);

// Individual stages (kda_intra.cu, kda_scan.cu, kda_decode.cu).
cudaError_t launch_intra(const FwdParams& p, cudaStream_t s);
// after_intra: launched right behind the intra-chunk kernel with programmatic
// stream serialization, so that its CTAs take SMs as that kernel's CTAs finish;
// the walks read the intermediates only once it has completed.
cudaError_t launch_scan(const FwdParams& p, int groups, cudaStream_t s, bool after_intra = false);
// beside_scan: launched right after the scan with programmatic stream
// serialization, so that its CTAs take the SMs the scan's walks leave free (the
// decode's items are other sequences, independent of the scan's); the decode
// grid completes only after the scan has.
cudaError_t launch_decode(const FwdParams& p, cudaStream_t s, bool beside_scan = false);
// Fused intra + scan launch (kda_intra_tc.cu), used instead of the two when
// fused_eligible(p): the walks need few enough SMs, the device takes a
// cooperative launch of one CTA per SM, and p.ready / p.queue are set.
// The caller clears p.queue together with the status word before the launch.
// set_fused_enabled(false) makes every call use the separate kernels.  When the
// device refuses the cooperative launch, launch_fused returns
// cudaErrorCooperativeLaunchTooLarge having enqueued nothing but the flag reset,
// and the device is not offered the fused launch again.
bool fused_eligible(const FwdParams& p);
void set_fused_enabled(bool on);
cudaError_t launch_fused(const FwdParams& p, cudaStream_t s);
int num_sms();
int scan_groups(int N, int H, int num_sms, int beside_pairs = 0);
// One thread of one CTA runs a bounded wait that cannot complete (kind 0: an
// mbarrier; 1: the zero ready flag at `flag`) and, when it gives up, ORs 1 into
// *status.
cudaError_t launch_wait_probe(int kind, int* status, const int* flag, cudaStream_t s);
// A tensor map of `out` for a walk's TMA stores (box box_values values x 1 head
// x box_rows rows); false when it cannot be made (the walk then stores directly).
bool make_out_map(CUtensorMap* m, const FwdParams& p, int box_values, int box_rows);
// Segments per long sequence when the scan runs segmented (few (sequence, head)
// pairs, so that the segments' walks fill the GPU), else 0; *L = chunks per segment.
int scan_segments(const FwdParams& p, int num_sms, int* L);

}  // namespace kda
